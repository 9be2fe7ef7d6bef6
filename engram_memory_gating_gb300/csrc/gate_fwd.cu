// Saved-state gate, forward (cuDNN Frontend "Engram saved-state gate",
// semantics and saved-state paragraphs).
//
// Per token n and stream s < 4:
//   rstd_X = 1/sqrt(mean(x^2) + eps), rstd_key = 1/sqrt(mean(k^2) + eps)
//   dot    = sum_i (x_i rstd_X) w_i (k_i rstd_key) = rstd_X rstd_key sum_i x_i w_i k_i
//   gate   = sigmoid(sign(dot) sqrt(max(|dot|, 1e-6)))
//   out    = bf16_rn(x + gate v)            (false mask: out = x, gate saved as 0)
//
// Every per-token quantity of a (token, stream) row is a reduction over that
// row only.  Two designs:
//  * gate_fwd_kernel: one warp per row, no communication between warps.  The
//    warp streams the row's X and key with 16-byte loads (lane l takes the
//    chunks l, l+32, ...; two groups of chunks in flight), forms the three
//    sums with packed fp32x2 arithmetic, reduces them with a butterfly of
//    shuffles (every lane ends with the same totals), computes the gate, then
//    streams X again (an L2 hit: the row was read a few microseconds earlier)
//    and v, two groups in flight, and writes `out` with streaming stores.  The
//    four rows of a token go to four warps of the same CTA, so v is read from
//    HBM once and from L1/L2 after.
//  * gate_fwd_quad_kernel (4096 <= d <= 5120, any batch): the four warps of
//    a quad share a row, each owning a quarter of the columns (five chunks
//    per lane).  A warp's quarters of X and key arrive by bulk copies into
//    its own shared buffer a row ahead; it keeps its X chunks in registers
//    from the reduction to the output pass, issues its v loads before the
//    exchange, and the quad adds the four partial sums through shared memory
//    in a fixed order.  Splitting rows four ways evens out the work of short
//    batches, where a warp would otherwise own only a dozen rows.
// The fused weight (80 KB) stays resident in L1.  Warps (or quads) loop over
// rows persistently.
//
// sum x w k uses error-free transformations (TwoProd via FMA, TwoSum) so the
// dot product keeps its accuracy when the terms cancel; the squares are
// summed in plain fp32 (all terms positive).
#include "common.cuh"
#include "engram_internal.h"

namespace eg {
namespace {

constexpr int kS = 4;       // streams

// Programmatic dependent launch.  Launched with programmatic stream
// serialisation, a forward kernel first waits for the preceding kernel of the
// stream to complete (griddepcontrol.wait: its writes are then visible) and
// only then lets the next kernel be scheduled, so that early scheduling never
// runs ahead of a producer; only the launch latency overlaps.
EG_DEV void grid_dep_start() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
constexpr int kGroup = 4;   // 16-byte chunks per lane per load group

// 16-byte loads: read-only path; `_na` does not allocate in L1 (data used once).
EG_DEV uint4 ldg16(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
EG_DEV uint4 ldg16_na(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Butterfly sums across the warp; every lane ends with the same value.
EG_DEV void warp_sum(float& a) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) a = __fadd_rn(a, __shfl_xor_sync(kFullMask, a, off));
}
EG_DEV void warp_sum_pair(float& hi, float& lo) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        cacc_merge(hi, lo, __shfl_xor_sync(kFullMask, hi, off), __shfl_xor_sync(kFullMask, lo, off));
}

// kDFix = 5120: the packed layout (KV rows, saved state as (N, 4, 4) records)
// with hidden size and strides known at compile time; kDFix = 0: any hidden
// size d (a multiple of 8), key / value rows through runtime strides, saved
// state as four (N, 4) arrays.
template <int kDFix>
__global__ void __launch_bounds__(256, 2) gate_fwd_kernel(const GateFwdParams p) {
    grid_dep_start();
    const int lane = threadIdx.x & 31;
    const long long gwarp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const long long rows = p.N * kS;
    const int d = kDFix ? kDFix : p.d;
    const int nch = d >> 3;                         // 16-byte chunks per row
    const int ng = ((nch + 31) / 32 + kGroup - 1) / kGroup;  // load groups per lane
    const float inv_d = 1.0f / static_cast<float>(d);
    // chunk m of this lane (chunk index lane + 32 m) exists
    auto has = [&](int m) { return (kDFix != 0 && (kDFix / 8) % 32 == 0) || lane + 32 * m < nch; };

    for (long long row = gwarp; row < rows; row += nwarps) {
        const long long n = row >> 2;
        const int s = static_cast<int>(row & 3);
        const uint4* xr = reinterpret_cast<const uint4*>(p.x + (n * kS + s) * d) + lane;
        const long long key_ts = kDFix ? 5LL * kDFix : p.key_ts;
        const long long v_ts = kDFix ? 5LL * kDFix : p.v_ts;
        const uint4* kr = reinterpret_cast<const uint4*>(p.key + n * key_ts + static_cast<long long>(s) * d) + lane;
        const uint4* vr = reinterpret_cast<const uint4*>(p.v + n * v_ts) + lane;
        const float4* wr = reinterpret_cast<const float4*>(p.w + static_cast<long long>(s) * d) + 2 * lane;
        const bool on = (p.mask == nullptr) || (__ldg(p.mask + n) != 0);

        // ---- pass 1: sum x^2, sum k^2, sum x w k (compensated)
        float2 ssx = make_float2(0.f, 0.f), ssk = ssx, hi = ssx, lo = ssx;
        uint4 xa[kGroup], ka[kGroup], xb[kGroup], kb[kGroup];
        auto load = [&](int g, uint4 (&xq)[kGroup], uint4 (&kq)[kGroup]) {
#pragma unroll
            for (int c = 0; c < kGroup; ++c) {
                const int m = g * kGroup + c;
                if (has(m)) {
                    xq[c] = ldg16(xr + 32 * m);
                    kq[c] = ldg16_na(kr + 32 * m);
                } else {
                    xq[c] = kq[c] = make_uint4(0, 0, 0, 0);
                }
            }
        };
        auto accum = [&](int g, const uint4 (&xq)[kGroup], const uint4 (&kq)[kGroup]) {
#pragma unroll
            for (int c = 0; c < kGroup; ++c) {
                const int m = g * kGroup + c;
                if (!has(m)) continue;
                const float4 wa = __ldg(wr + 64 * m);
                const float4 wb = __ldg(wr + 64 * m + 1);
                const float2 w2[4] = {make_float2(wa.x, wa.y), make_float2(wa.z, wa.w),
                                      make_float2(wb.x, wb.y), make_float2(wb.z, wb.w)};
                const uint32_t xw[4] = {xq[c].x, xq[c].y, xq[c].z, xq[c].w};
                const uint32_t kw[4] = {kq[c].x, kq[c].y, kq[c].z, kq[c].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x2 = bf2(xw[e]);
                    const float2 k2 = bf2(kw[e]);
                    ssx = fma2(x2, x2, ssx);
                    ssk = fma2(k2, k2, ssk);
                    // x*k is exact in fp32 (two 8-bit significands)
                    cacc_prod_x2(hi, lo, mul2(x2, k2), w2[e]);
                }
            }
        };
        load(0, xa, ka);
#pragma unroll
        for (int g = 0; g < ng; g += 2) {
            if (g + 1 < ng) load(g + 1, xb, kb);
            accum(g, xa, ka);
            if (g + 1 < ng) {
                if (g + 2 < ng) load(g + 2, xa, ka);
                accum(g + 1, xb, kb);
            }
        }
        float sx = __fadd_rn(ssx.x, ssx.y);
        float sk = __fadd_rn(ssk.x, ssk.y);
        float h = hi.x, l = lo.x;
        cacc_merge(h, l, hi.y, lo.y);
        warp_sum(sx);
        warp_sum(sk);
        warp_sum_pair(h, l);

        // ---- gate (the same in every lane)
        const float rstd_x = rsqrtf(fmaf(sx, inv_d, p.eps));
        const float rstd_k = rsqrtf(fmaf(sk, inv_d, p.eps));
        const float dot = __fadd_rn(h, l) * rstd_x * rstd_k;
        const float ad = fmaxf(fabsf(dot), p.clamp);
        const float sqm = ad * rsqrtf(ad);
        const float sq = dot > 0.f ? sqm : (dot < 0.f ? -sqm : 0.f);
        const float gate = on ? __frcp_rn(1.0f + __expf(-sq)) : 0.f;
        if (lane == 0) {
            if (kDFix) {
                if (p.saved != nullptr) stg_f4(p.saved + row * 4, gate, dot, rstd_x, rstd_k);
            } else if (p.sv_gate != nullptr) {
                p.sv_gate[row] = gate;
                p.sv_dot[row] = dot;
                p.sv_rx[row] = rstd_x;
                p.sv_rk[row] = rstd_k;
            }
        }

        // ---- pass 2: out = x + gate * v, one rounding; a false mask copies X.
        // Two load groups in flight (the pass-1 buffers are free by now).
        uint4* o = reinterpret_cast<uint4*>(p.out + (n * kS + s) * d) + lane;
        const float2 g2 = splat2(gate);
        auto load2 = [&](int g, uint4 (&xq)[kGroup], uint4 (&vq)[kGroup]) {
#pragma unroll
            for (int c = 0; c < kGroup; ++c) {
                const int m = g * kGroup + c;
                xq[c] = has(m) ? ldg16(xr + 32 * m) : make_uint4(0, 0, 0, 0);
                vq[c] = (on && has(m)) ? ldg16(vr + 32 * m) : make_uint4(0, 0, 0, 0);
            }
        };
        auto store2 = [&](int g, const uint4 (&xq)[kGroup], const uint4 (&vq)[kGroup]) {
#pragma unroll
            for (int c = 0; c < kGroup; ++c) {
                const int m = g * kGroup + c;
                uint4 ov = xq[c];
                if (on) {
                    ov.x = pack2(fma2(g2, bf2(vq[c].x), bf2(xq[c].x)));
                    ov.y = pack2(fma2(g2, bf2(vq[c].y), bf2(xq[c].y)));
                    ov.z = pack2(fma2(g2, bf2(vq[c].z), bf2(xq[c].z)));
                    ov.w = pack2(fma2(g2, bf2(vq[c].w), bf2(xq[c].w)));
                }
                if (has(m)) stg_cs(o + 32 * m, ov);
            }
        };
        load2(0, xa, ka);
#pragma unroll
        for (int g = 0; g < ng; g += 2) {
            if (g + 1 < ng) load2(g + 1, xb, kb);
            store2(g, xa, ka);
            if (g + 1 < ng) {
                if (g + 2 < ng) load2(g + 2, xa, ka);
                store2(g + 1, xb, kb);
            }
        }
    }
}

// Named barrier of the four warps of quad `q` (ids 1 and 2, 128 threads; the
// ids must be immediates).
EG_DEV void quad_sync(int q) {
    if (q == 0)
        asm volatile("bar.sync 1, 128;" ::: "memory");
    else
        asm volatile("bar.sync 2, 128;" ::: "memory");
}

// The four warps of a quad share a row, warp 4q + j owning the j-th quarter of
// its 16-byte chunks (at most five per lane: d <= 5120; for the packed layout,
// d = 5120, exactly chunks 160j .. 160j + 159).  Each keeps its X chunks in
// registers from the reduction to the output pass, so that pass loads only v.
// The quad exchanges its partial sums through shared memory (two slots by row
// parity, one quad barrier per row) and every warp merges them in part order,
// so all four form the same gate.  kPacked: packed KV and saved records with
// d = 5120 at compile time; otherwise runtime d and strides, saved arrays.
// A warp's quarters of a row (up to 2560 contiguous bytes of X and as many of
// key; 16-byte multiples at 16-byte offsets, as d % 8 == 0) arrive by two 1-D
// bulk copies into the warp's own shared buffer, issued as soon as the warp
// has taken the previous row's quarters into registers, so the next row's
// loads are in flight for a whole row of work.
constexpr int kParts = 4;
constexpr int kPerLane = kGateHidden / 8 / kParts / 32;  // 5
constexpr int kQuadMaxHidden = kParts * kPerLane * 32 * 8;  // 5120
constexpr int kQuarter = kPerLane * 32;                   // 16-byte chunks of a packed quarter

template <bool kPacked>
__global__ void __launch_bounds__(256, 2) gate_fwd_quad_kernel(const GateFwdParams p) {
    grid_dep_start();
    __shared__ float4 xch[2][2][kParts];   // [quad][row parity][part]: sum x^2, sum k^2, hi, lo
    // each warp's (X, key) quarters of its next row, and the warp's mbarrier
    __shared__ __align__(128) uint4 stage[8][2][kQuarter];
    __shared__ uint64_t sbar[8];
    const int d = kPacked ? kGateHidden : p.d;
    const long long key_ts = kPacked ? 5LL * kGateHidden : p.key_ts;
    const long long v_ts = kPacked ? 5LL * kGateHidden : p.v_ts;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int quad = warp >> 2, part = warp & 3;
    const long long gq = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 7;
    const long long nq = (static_cast<long long>(gridDim.x) * blockDim.x) >> 7;
    const long long rows = p.N * kS;
    const float inv_d = 1.0f / static_cast<float>(d);
    const int nch = d >> 3;
    const int per = kPacked ? kGateHidden / 8 / kParts : (nch + kParts - 1) / kParts;  // chunks per part
    const int cbeg = part * per;
    const int cnt = kPacked ? per : max(0, min(per, nch - cbeg));       // this part's chunks
    const int ch0 = cbeg + lane;
    auto has = [&](int m) { return kPacked || lane + 32 * m < cnt; };
    uint4* const bx = stage[warp][0];
    uint4* const bk = stage[warp][1];
    const uint32_t qbytes = 16u * static_cast<uint32_t>(cnt);   // this part's quarter (0 if it has none)
    uint64_t* const bar = &sbar[warp];
    // lane 0: the quarters of row r into this warp's buffer (copy k of the
    // warp completes the barrier's phase k)
    uint32_t issued = 0;
    auto issue = [&](long long r) {
        ++issued;
        const long long nn = r >> 2;
        const int ss = static_cast<int>(r & 3);
        mbar_arrive_expect_tx(bar, 2 * qbytes);
        if (qbytes > 0) {
            bulk_g2s(bx, p.x + r * d + cbeg * 8, qbytes, bar);
            bulk_g2s(bk, p.key + nn * key_ts + static_cast<long long>(ss) * d + cbeg * 8, qbytes, bar);
        }
    };
    bool failed = false;
    uint32_t ph = 0;
    {
        if (lane == 0) {
            mbar_init(bar, 1);
            fence_mbar_init();
            if (gq < rows) issue(gq);
        }
        __syncwarp();
    }
    int par = 0;
    for (long long row = gq; row < rows; row += nq, par ^= 1) {
        const long long n = row >> 2;
        const int s = static_cast<int>(row & 3);
        const uint4* vr = reinterpret_cast<const uint4*>(p.v + n * v_ts) + ch0;
        const float4* wr = reinterpret_cast<const float4*>(p.w + static_cast<long long>(s) * d) + 2 * ch0;
        const bool on = (p.mask == nullptr) || (__ldg(p.mask + n) != 0);
        uint4 xq[kPerLane], kq[kPerLane];
        // this row's quarters have landed; take them into registers, then free
        // the buffer for the next row
        if (!failed && !mbar_wait(bar, ph)) failed = true;
        failed = __any_sync(kFullMask, failed);
        ph ^= 1u;
#pragma unroll
        for (int m = 0; m < kPerLane; ++m) {
            xq[m] = has(m) ? bx[lane + 32 * m] : make_uint4(0, 0, 0, 0);
            kq[m] = has(m) ? bk[lane + 32 * m] : make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
        if (lane == 0 && !failed && row + nq < rows) {
            fence_proxy_async();
            issue(row + nq);
        }

        // ---- pass 1 over this part: sum x^2, sum k^2, sum x w k (compensated)
        float2 ssx = make_float2(0.f, 0.f), ssk = ssx, hi = ssx, lo = ssx;
#pragma unroll
        for (int m = 0; m < kPerLane; ++m) {
            if (!has(m)) continue;
            const float4 wa = __ldg(wr + 64 * m);
            const float4 wb = __ldg(wr + 64 * m + 1);
            const float2 w2[4] = {make_float2(wa.x, wa.y), make_float2(wa.z, wa.w),
                                  make_float2(wb.x, wb.y), make_float2(wb.z, wb.w)};
            const uint32_t xw[4] = {xq[m].x, xq[m].y, xq[m].z, xq[m].w};
            const uint32_t kw[4] = {kq[m].x, kq[m].y, kq[m].z, kq[m].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x2 = bf2(xw[e]);
                const float2 k2 = bf2(kw[e]);
                ssx = fma2(x2, x2, ssx);
                ssk = fma2(k2, k2, ssk);
                // x*k is exact in fp32 (two 8-bit significands)
                cacc_prod_x2(hi, lo, mul2(x2, k2), w2[e]);
            }
        }
        // v for the output pass, in flight during the exchange
        uint4 vq[kPerLane];
#pragma unroll
        for (int m = 0; m < kPerLane; ++m) vq[m] = (on && has(m)) ? ldg16(vr + 32 * m) : make_uint4(0, 0, 0, 0);
        float sx = __fadd_rn(ssx.x, ssx.y);
        float sk = __fadd_rn(ssk.x, ssk.y);
        float h = hi.x, l = lo.x;
        cacc_merge(h, l, hi.y, lo.y);
        warp_sum(sx);
        warp_sum(sk);
        warp_sum_pair(h, l);
        if (lane == 0) xch[quad][par][part] = make_float4(sx, sk, h, l);
        quad_sync(quad);
        {
            const float4 a = xch[quad][par][0];
            sx = a.x;
            sk = a.y;
            h = a.z;
            l = a.w;
#pragma unroll
            for (int j = 1; j < kParts; ++j) {
                const float4 b = xch[quad][par][j];
                sx = __fadd_rn(sx, b.x);
                sk = __fadd_rn(sk, b.y);
                cacc_merge(h, l, b.z, b.w);
            }
        }

        // ---- gate (the same in every lane of the quad)
        const float rstd_x = rsqrtf(fmaf(sx, inv_d, p.eps));
        const float rstd_k = rsqrtf(fmaf(sk, inv_d, p.eps));
        const float dot = __fadd_rn(h, l) * rstd_x * rstd_k;
        const float ad = fmaxf(fabsf(dot), p.clamp);
        const float sqm = ad * rsqrtf(ad);
        const float sq = dot > 0.f ? sqm : (dot < 0.f ? -sqm : 0.f);
        const float gate = on ? __frcp_rn(1.0f + __expf(-sq)) : 0.f;
        if (lane == 0 && part == 0) {
            if (kPacked) {
                if (p.saved != nullptr) stg_f4(p.saved + row * 4, gate, dot, rstd_x, rstd_k);
            } else if (p.sv_gate != nullptr) {
                p.sv_gate[row] = gate;
                p.sv_dot[row] = dot;
                p.sv_rx[row] = rstd_x;
                p.sv_rk[row] = rstd_k;
            }
        }

        // ---- pass 2: out = x + gate * v, one rounding; a false mask copies X
        uint4* o = reinterpret_cast<uint4*>(p.out + row * d) + ch0;
        const float2 g2 = splat2(gate);
#pragma unroll
        for (int m = 0; m < kPerLane; ++m) {
            uint4 ov = xq[m];
            if (on) {
                ov.x = pack2(fma2(g2, bf2(vq[m].x), bf2(xq[m].x)));
                ov.y = pack2(fma2(g2, bf2(vq[m].y), bf2(xq[m].y)));
                ov.z = pack2(fma2(g2, bf2(vq[m].z), bf2(xq[m].z)));
                ov.w = pack2(fma2(g2, bf2(vq[m].w), bf2(xq[m].w)));
            }
            if (has(m)) stg_cs(o + 32 * m, ov);
        }
    }
    // the last copy, which may still be in flight only after a wait gave up
    // (no copy is issued after that), lands or times out before the CTA leaves
    if (failed && lane == 0) {
        atomicOr(p.err, kErrTimeout);
        if (issued > 0) (void)mbar_wait(bar, (issued - 1u) & 1u);
    }
}

}  // namespace

cudaError_t gate_fwd_prepare(int) {
    // the quad kernel's row buffers (41 KB a CTA, two CTAs an SM) in shared
    // memory, the rest of the unified cache as L1 for the 80 KB weight; the
    // row kernel uses no shared memory
    cudaError_t e = cudaFuncSetAttribute(gate_fwd_quad_kernel<true>, cudaFuncAttributePreferredSharedMemoryCarveout, 40);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gate_fwd_quad_kernel<false>, cudaFuncAttributePreferredSharedMemoryCarveout, 40);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gate_fwd_kernel<kGateHidden>, cudaFuncAttributePreferredSharedMemoryCarveout, 0);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gate_fwd_kernel<0>, cudaFuncAttributePreferredSharedMemoryCarveout, 0);
}

// Co-resident CTAs of the forward on this device (threads per CTA given): the
// smallest count of its kernels, so the grid suits each.
cudaError_t gate_fwd_max_clusters(int, int threads, int, int* out) {
    int m = 1 << 30, v = 0, dev = 0, sms = 0;
    cudaError_t e = cudaSuccess;
    const void* kernels[] = {reinterpret_cast<const void*>(gate_fwd_quad_kernel<true>),
                             reinterpret_cast<const void*>(gate_fwd_quad_kernel<false>),
                             reinterpret_cast<const void*>(gate_fwd_kernel<kGateHidden>),
                             reinterpret_cast<const void*>(gate_fwd_kernel<0>)};
    for (const void* k : kernels) {
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, k, threads, 0);
        if (e == cudaSuccess && v < m) m = v;
    }
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    *out = m * sms;
    return e;
}

// Four warps per row for 4096 <= d <= 5120, at every batch size: with its
// quarters prefetched a row ahead the quad kernel is faster than one warp per
// row from 2,048 to 262,144 tokens, masked or not (N = 65,536: 1.26 against
// 1.50 ms; 262,144: 5.29 against 5.99 ms); narrower and wider rows take one
// warp per row (narrower rows leave most lanes of a quarter idle).
cudaError_t gate_fwd_launch(const GateFwdParams& p, const LaunchCfg& c, cudaStream_t s) {
    const bool quad = p.d >= 4096 && p.d <= kQuadMaxHidden;
    // programmatic stream serialisation (each kernel waits for its predecessor first)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(c.clusters), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(c.threads), 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.packed && quad) return cudaLaunchKernelEx(&cfg, gate_fwd_quad_kernel<true>, p);
    if (p.packed) return cudaLaunchKernelEx(&cfg, gate_fwd_kernel<kGateHidden>, p);
    if (quad) return cudaLaunchKernelEx(&cfg, gate_fwd_quad_kernel<false>, p);
    return cudaLaunchKernelEx(&cfg, gate_fwd_kernel<0>, p);
}

}  // namespace eg
