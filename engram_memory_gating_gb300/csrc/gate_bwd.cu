// Saved-state gate, backward (cuDNN Frontend "Engram saved-state gate",
// layout, saved-state and workspace paragraphs; tile-kernels engram gate
// backward test, which reduces per-block grad_w partials with a sum).
//
// With the forward's saved (gate, dot, rstd_X, rstd_key) per (n, s) and
//   dgate = sum_i g_i v_i,   sq = sqrt(max(|dot|, 1e-6)),
//   ddot  = dgate * sigmoid(sq) * sigmoid(-sq) * 0.5/sqrt(|dot|)   (0 if |dot| < 1e-6
//           or the saved gate is 0, i.e. a masked token; sigmoid' is taken from
//           the saved dot because an fp32 gate near 1 has lost the bits of 1 - gate)
//   A = ddot rstd_X rstd_key,  B = ddot rstd_X^2 dot / d,  Ck = ddot rstd_key^2 dot / d:
//   grad_x_i   = g_i + A w_i k_i - B x_i
//   grad_key_i = A w_i x_i - Ck k_i
//   grad_v_i   = sum_{s=0..3} gate_s g_{s,i}      (fp32, one rounding)
//   grad_w_i  += A x_i k_i                         (= ddot * xh_i * kh_i)
// These are the chain rule through the RMS norms written with the saved dot
// (sum_i xh_i w_i kh_i): d dot/d x_i = rstd_X (w_i kh_i - xh_i dot/d).
//
// Three kernels, none of which communicates across CTAs:
//  1. coefficients: one warp per token reads the token's grad_out rows and v
//     (16-byte loads), reduces the four dgate sums with error-free
//     accumulation and shuffles, and lanes 0..3 turn them into the per-stream
//     scalars (A as a double-float pair, -B, -Ck) in fp64, written to the
//     workspace's 16 floats per token;
//  2. elementwise: a CTA owns a 1024-column slice of every stream over a
//     group of consecutive tokens; the slice rows of X, the keys and grad_out
//     plus the token's scalars and saved record stream through a ring of
//     shared-memory stages (1-D bulk copies); each thread writes its 8
//     columns of grad_x, grad_key and grad_v and accumulates grad_w for its
//     columns over the group as an unevaluated (hi, lo) pair, stored in the
//     workspace's block slots (group g: slots 2g and 2g+1);
//  3. the pairs are merged in ascending group order (bitwise reproducible).
// The per-token scalars are evaluated in fp64 because a relative error of a
// few fp32 ulps in A, summed over 8192 tokens, would exceed the 1e-6
// absolute accuracy asked of grad_w near zero.
#include "common.cuh"
#include "engram_internal.h"

namespace eg {
namespace {

constexpr int kS = 4;
constexpr int kD = 5120;
constexpr int kChunks = kD / 256;   // 16-byte chunks per lane per row
constexpr int kCG = 2;              // chunk indices per load group (kernel 1)
constexpr int kRows = 3 * kS;       // X rows, key rows, grad_out rows (kernel 2)
static_assert(kChunks % kCG == 0, "row must split into whole groups");

EG_DEV uint4 ldg16_na(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

EG_DEV void warp_sum_pair(float& hi, float& lo) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        cacc_merge(hi, lo, __shfl_xor_sync(kFullMask, hi, off), __shfl_xor_sync(kFullMask, lo, off));
}

// ---------------------------------------------------------------- kernel 1
__global__ void __launch_bounds__(256, 2) gate_bwd_coef_kernel(const GateBwdParams p) {
    const int lane = threadIdx.x & 31;
    const long long gwarp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long n = gwarp; n < p.N; n += nwarps) {
        const uint4* vr = reinterpret_cast<const uint4*>(p.kv + (n * (kS + 1) + kS) * kD) + lane;
        const uint4* gr = reinterpret_cast<const uint4*>(p.gout + n * kS * kD) + lane;
        float2 hi[kS], lo[kS];
#pragma unroll
        for (int s = 0; s < kS; ++s) hi[s] = lo[s] = make_float2(0.f, 0.f);
        uint4 vb[2][kCG], gb[2][kS][kCG];
#pragma unroll
        for (int c = 0; c < kCG; ++c) {
            vb[0][c] = ldg16_na(vr + 32 * c);
#pragma unroll
            for (int s = 0; s < kS; ++s) gb[0][s][c] = ldg16_na(gr + s * (kD / 8) + 32 * c);
        }
#pragma unroll
        for (int grp = 0; grp < kChunks / kCG; ++grp) {
            const int cur = grp & 1;
            if (grp + 1 < kChunks / kCG) {
#pragma unroll
                for (int c = 0; c < kCG; ++c) {
                    const int m = (grp + 1) * kCG + c;
                    vb[cur ^ 1][c] = ldg16_na(vr + 32 * m);
#pragma unroll
                    for (int s = 0; s < kS; ++s) gb[cur ^ 1][s][c] = ldg16_na(gr + s * (kD / 8) + 32 * m);
                }
            }
#pragma unroll
            for (int c = 0; c < kCG; ++c) {
                const float2 v2[4] = {bf2(vb[cur][c].x), bf2(vb[cur][c].y), bf2(vb[cur][c].z),
                                      bf2(vb[cur][c].w)};
#pragma unroll
                for (int s = 0; s < kS; ++s) {
                    const uint4 gq = gb[cur][s][c];
                    // g*v is exact in fp32 (two 8-bit significands)
                    cacc_add_x2(hi[s], lo[s], mul2(bf2(gq.x), v2[0]));
                    cacc_add_x2(hi[s], lo[s], mul2(bf2(gq.y), v2[1]));
                    cacc_add_x2(hi[s], lo[s], mul2(bf2(gq.z), v2[2]));
                    cacc_add_x2(hi[s], lo[s], mul2(bf2(gq.w), v2[3]));
                }
            }
        }
        float h[kS], l[kS];
#pragma unroll
        for (int s = 0; s < kS; ++s) {
            h[s] = hi[s].x;
            l[s] = lo[s].x;
            cacc_merge(h[s], l[s], hi[s].y, lo[s].y);
            warp_sum_pair(h[s], l[s]);
        }
        if (lane < kS) {
            // stream s = lane: fp64 scalars; rsqrt and the reciprocal start from
            // fp32 estimates refined by one Newton step, exp is the fp64 routine
            const float hs = lane == 0 ? h[0] : lane == 1 ? h[1] : lane == 2 ? h[2] : h[3];
            const float ls = lane == 0 ? l[0] : lane == 1 ? l[1] : lane == 2 ? l[2] : l[3];
            const float4 sv = __ldg(reinterpret_cast<const float4*>(p.saved + (n * kS + lane) * 4));
            const float gate = sv.x;
            const double dot = sv.y, rx = sv.z, rk = sv.w;
            const double ad = fabs(dot);
            double ddot = 0.0;
            if (ad >= 1e-6 && gate != 0.f) {
                double y = rsqrtf(fabsf(sv.y));
                y = y * (1.5 - 0.5 * ad * y * y);           // 1/sqrt(|dot|)
                const double sqm = ad * y;                  // |sq| = sqrt(|dot|)
                const double ex = exp(-sqm);
                const double den = 1.0 + ex;
                double rc = __frcp_rn(static_cast<float>(den));
                rc = rc * (2.0 - den * rc);                 // 1/(1 + e^-|sq|)
                const double dsig = ex * rc * rc;           // sigmoid(sq) sigmoid(-sq)
                const double dgate = static_cast<double>(hs) + static_cast<double>(ls);
                ddot = dgate * dsig * (0.5 * y);            // d sq/d dot = 0.5/sqrt(|dot|)
            }
            const double dd = dot / static_cast<double>(kD);
            const double av = ddot * rx * rk;
            const float a_hi = static_cast<float>(av);
            const float a_lo = static_cast<float>(av - static_cast<double>(a_hi));
            stg_f4(p.coef + (n * kS + lane) * 4, a_hi, a_lo, static_cast<float>(-(ddot * rx * rx * dd)),
                   static_cast<float>(-(ddot * rk * rk * dd)));
        }
    }
}

// ---------------------------------------------------------------- kernel 2
constexpr int kRing2Off = 256;  // after the stage mbarriers

__global__ void __launch_bounds__(128, 2) gate_bwd_main_kernel(const GateBwdParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    unsigned char* ring = smem + kRing2Off;

    const int tid = threadIdx.x;
    const int col0 = static_cast<int>(blockIdx.x) * p.ncols;
    const long long grp = blockIdx.y;
    const bool active = tid < p.ngroups;
    const uint32_t row_bytes = static_cast<uint32_t>(p.ncols) * 2u;
    const uint32_t stage_bytes = kRows * row_bytes + 128u;
    const int stages = p.stages;
    const long long t0 = grp * p.group_tokens;
    const long long t1 = (t0 + p.group_tokens < p.N) ? t0 + p.group_tokens : p.N;
    const long long ntok = t1 > t0 ? t1 - t0 : 0;

    float2 w2[kS][4];
#pragma unroll
    for (int s = 0; s < kS; ++s) {
        if (active) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(p.w + s * kD + col0 + 8 * tid));
            const float4 b = __ldg(reinterpret_cast<const float4*>(p.w + s * kD + col0 + 8 * tid + 4));
            w2[s][0] = make_float2(a.x, a.y);
            w2[s][1] = make_float2(a.z, a.w);
            w2[s][2] = make_float2(b.x, b.y);
            w2[s][3] = make_float2(b.z, b.w);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) w2[s][e] = make_float2(0.f, 0.f);
        }
    }

    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(&full[st], 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](long long j) {
        const long long n = t0 + j;
        const int st = static_cast<int>(j % stages);
        unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        mbar_arrive_expect_tx(&full[st], stage_bytes);
#pragma unroll
        for (int s = 0; s < kS; ++s) {
            bulk_g2s(b + s * row_bytes, p.x + (n * kS + s) * kD + col0, row_bytes, &full[st]);
            bulk_g2s(b + (kS + s) * row_bytes, p.kv + (n * (kS + 1) + s) * kD + col0, row_bytes, &full[st]);
            bulk_g2s(b + (2 * kS + s) * row_bytes, p.gout + (n * kS + s) * kD + col0, row_bytes, &full[st]);
        }
        bulk_g2s(b + kRows * row_bytes, p.coef + n * kS * 4, 64u, &full[st]);
        bulk_g2s(b + kRows * row_bytes + 64, p.saved + n * kS * 4, 64u, &full[st]);
    };
    if (tid == 0) {
        const long long pro = ntok < stages ? ntok : stages;
        for (long long j = 0; j < pro; ++j) issue(j);
    }

    float2 phi[kS][4], plo[kS][4];  // grad_w of this thread's columns, hi + lo
#pragma unroll
    for (int s = 0; s < kS; ++s)
#pragma unroll
        for (int e = 0; e < 4; ++e) phi[s][e] = plo[s][e] = make_float2(0.f, 0.f);

    bool failed = false;
    for (long long j = 0; j < ntok; ++j) {
        const long long n = t0 + j;
        const int st = static_cast<int>(j % stages);
        if (!failed && !mbar_wait(&full[st], static_cast<uint32_t>((j / stages) & 1))) failed = true;
        const unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        const float* cf = reinterpret_cast<const float*>(b + kRows * row_bytes);  // [s][4]
        const float* sv = cf + 16;                                                // [s][4]
        if (active) {
            float2 gv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) gv[e] = make_float2(0.f, 0.f);
            uint16_t* gxo = p.gx + n * kS * kD + col0 + 8 * tid;
            uint16_t* gko = p.gkv + n * (kS + 1) * kD + col0 + 8 * tid;
#pragma unroll
            for (int s = 0; s < kS; ++s) {
                const float4 c4 = *reinterpret_cast<const float4*>(cf + 4 * s);
                const float2 A2 = splat2(c4.x), Al2 = splat2(c4.y);
                const float2 nB2 = splat2(c4.z), nC2 = splat2(c4.w);
                const float2 G2 = splat2(sv[4 * s]);
                const uint4 xq = lds128(b + s * row_bytes + 16 * tid);
                const uint4 kq = lds128(b + (kS + s) * row_bytes + 16 * tid);
                const uint4 gq = lds128(b + (2 * kS + s) * row_bytes + 16 * tid);
                const uint32_t xw[4] = {xq.x, xq.y, xq.z, xq.w};
                const uint32_t kw[4] = {kq.x, kq.y, kq.z, kq.w};
                const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
                uint32_t ox[4], ok[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x2 = bf2(xw[e]), k2 = bf2(kw[e]), g2 = bf2(gw[e]);
                    const float2 aw = mul2(A2, w2[s][e]);
                    ox[e] = pack2(fma2(aw, k2, fma2(nB2, x2, g2)));
                    ok[e] = pack2(fma2(aw, x2, mul2(nC2, k2)));
                    gv[e] = fma2(G2, g2, gv[e]);
                    cacc_prod2_x2(phi[s][e], plo[s][e], A2, Al2, mul2(x2, k2));
                }
                stg_cs(gxo + s * kD, make_uint4(ox[0], ox[1], ox[2], ox[3]));
                stg_cs(gko + s * kD, make_uint4(ok[0], ok[1], ok[2], ok[3]));
            }
            stg_cs(gko + kS * kD, make_uint4(pack2(gv[0]), pack2(gv[1]), pack2(gv[2]), pack2(gv[3])));
        }
        // every thread is done with this stage: refill it
        __syncthreads();
        if (tid == 0 && j + stages < ntok) {
            fence_proxy_async();
            issue(j + stages);
        }
    }
    // this group's grad_w for the slice: (hi, lo) in slots 2g, 2g+1, or
    // hi + lo in slot 0 when a single group covers a single block
    if (active && ntok > 0) {
#pragma unroll
        for (int s = 0; s < kS; ++s) {
            float* o = p.partial + ((p.pair_slots ? 2 * grp : grp) * kS + s) * kD + col0 + 8 * tid;
            if (p.pair_slots) {
                float* ol = o + static_cast<long long>(kS) * kD;
                stg_f4(o, phi[s][0].x, phi[s][0].y, phi[s][1].x, phi[s][1].y);
                stg_f4(o + 4, phi[s][2].x, phi[s][2].y, phi[s][3].x, phi[s][3].y);
                stg_f4(ol, plo[s][0].x, plo[s][0].y, plo[s][1].x, plo[s][1].y);
                stg_f4(ol + 4, plo[s][2].x, plo[s][2].y, plo[s][3].x, plo[s][3].y);
            } else {
                float r[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    r[2 * e] = __fadd_rn(phi[s][e].x, plo[s][e].x);
                    r[2 * e + 1] = __fadd_rn(phi[s][e].y, plo[s][e].y);
                }
                stg_f4(o, r[0], r[1], r[2], r[3]);
                stg_f4(o + 4, r[4], r[5], r[6], r[7]);
            }
        }
    }
    if (failed) atomicOr(p.err, kErrTimeout);
}

// ---------------------------------------------------------------- kernel 3
// grad_weight[i] from the group partials, merged in ascending order with
// error-free additions (bitwise reproducible).  pairs: slot 2g = hi, 2g+1 = lo.
__global__ void __launch_bounds__(256) wreduce_kernel(const GateWReduceParams p) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    const float* src = p.partial + i;
    float hi = 0.f, lo = 0.f;
    if (!p.pairs) {
        for (int b = 0; b < p.nblocks; ++b) cacc_add(hi, lo, __ldg(src + static_cast<size_t>(b) * p.stride));
        p.out[i] = __fadd_rn(hi, lo);
        return;
    }
    const int np = p.nblocks / 2;
    int b = 0;
    for (; b + 4 <= np; b += 4) {
        float h[4], l[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            h[u] = __ldg(src + static_cast<size_t>(2 * (b + u)) * p.stride);
            l[u] = __ldg(src + static_cast<size_t>(2 * (b + u) + 1) * p.stride);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) cacc_merge(hi, lo, h[u], l[u]);
    }
    for (; b < np; ++b)
        cacc_merge(hi, lo, __ldg(src + static_cast<size_t>(2 * b) * p.stride),
                   __ldg(src + static_cast<size_t>(2 * b + 1) * p.stride));
    p.out[i] = __fadd_rn(hi, lo);
}

}  // namespace

cudaError_t gate_bwd_prepare(int smem_bytes) {
    cudaError_t e = cudaSuccess;
    if (smem_bytes > 0)  // 0: only the coefficient kernel is being set up
        e = cudaFuncSetAttribute(gate_bwd_main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem_bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gate_bwd_main_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gate_bwd_coef_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 0);
}

// Co-resident CTAs: of the coefficient kernel (threads = 256) when smem == 0,
// of the elementwise kernel otherwise.
cudaError_t gate_bwd_max_clusters(int, int threads, int smem, int* out) {
    int per_sm = 0, dev = 0, sms = 0;
    cudaError_t e = smem == 0
        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gate_bwd_coef_kernel, threads, 0)
        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gate_bwd_main_kernel, threads, smem);
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    *out = per_sm * sms;
    return e;
}

// kernel 1 then kernel 2 on the stream (kernel 3 is gate_wreduce_launch)
cudaError_t gate_bwd_launch(const GateBwdParams& p, const LaunchCfg& c, cudaStream_t s) {
    gate_bwd_coef_kernel<<<c.aux_blocks, 256, 0, s>>>(p);
    cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
    gate_bwd_main_kernel<<<dim3(c.clusters, c.grid_y, 1), c.threads, c.smem, s>>>(p);
    return cudaPeekAtLastError();
}

cudaError_t gate_wreduce_launch(const GateWReduceParams& p, cudaStream_t s) {
    const int threads = 128;
    const int blocks = (p.n + threads - 1) / threads;
    wreduce_kernel<<<blocks, threads, 0, s>>>(p);
    return cudaPeekAtLastError();
}

}  // namespace eg
