// Saved-state gate, backward (cuDNN Frontend "Engram saved-state gate",
// layout and saved-state paragraphs; tile-kernels engram gate backward test,
// which reduces per-block grad_w partials with a sum over blocks).
//
// With the forward's saved (gate, dot, rstd_X, rstd_key) per (n, s) and
//   dgate = sum_i g_i v_i,   sq = sqrt(max(|dot|, 1e-6)),
//   q = 0.5/sqrt(|dot|) if |dot| >= 1e-6 else 0,
//   ddot  = dgate * sigmoid(sq) * sigmoid(-sq) * q   (0 where the saved gate is 0,
//           i.e. a masked token; sigmoid' is taken from the saved dot because an
//           fp32 gate near 1 has lost the bits of 1 - gate),
//   A = ddot rstd_X rstd_key,  B = ddot rstd_X^2 dot / d,  Ck = ddot rstd_key^2 dot / d:
//   grad_x_i   = g_i + A w_i k_i - B x_i
//   grad_key_i = A w_i x_i - Ck k_i
//   grad_v_i   = sum_{s=0..3} gate_s g_{s,i}      (fp32, one rounding)
//   grad_w_i  += A x_i k_i                         (= ddot * xh_i * kh_i,
//                                                   error-free accumulation)
// The per-(token, stream) scalars are evaluated in fp64 (four per token, a
// negligible cost) and A is carried as a double-float pair into grad_w: a
// relative error of a few fp32 ulps in A would otherwise, summed over 8192
// tokens, exceed the 1e-6 absolute accuracy asked of grad_w near zero.
// These are the chain rule through the RMS norms written with the saved dot
// (sum_i xh_i w_i kh_i): d dot/d x_i = rstd_X (w_i kh_i - xh_i dot/d).
//
// Layout of the work: a cluster of C CTAs owns whole 64-token blocks; each CTA
// a column slice of every stream.  Per token the slice rows of X, the keys, v
// and grad_out plus the 64-byte saved record are bulk-copied into a ring of
// shared-memory stages; dgate (4 full-row reductions, compensated, packed
// fp32x2) is reduced across the warp and the CTA, and each CTA pushes its 4
// (hi, lo) pairs into every CTA of the cluster with st.async (mbarrier
// completion, no cluster barrier per token).  The loop is software-pipelined:
// token j+1's dgate pass runs while token j's partials travel, and one warp
// turns token j's totals into per-stream scalars (shared memory).  Each
// thread then writes its 8
// columns of grad_x, grad_key and grad_v and accumulates grad_w for its
// columns over all tokens of the cluster as an unevaluated (hi, lo) pair.
// With at least two 64-token blocks there are at most half as many clusters
// as blocks, so the pair fits the workspace's per-block partial slots: slot
// 2q holds cluster q's hi, slot 2q+1 its lo.  A second kernel merges the
// pairs in ascending cluster order (bitwise reproducible).
#include "common.cuh"
#include "engram_internal.h"

namespace eg {
namespace {

constexpr int kS = 4;
constexpr int kBlockTokens = 64;
constexpr int kRows = 3 * kS + 1;  // X rows, key rows, v, grad_out rows

// Warp reduce-scatter of 4 compensated (hi, lo) pairs.  On return lane l holds
// the warp total of stream s = 2*bit4(l) + bit3(l) in (v0, v1).
EG_DEV void warp_reduce_pairs4(const float (&acc)[8], int lane, float& v0, float& v1) {
    float a4[4], r4[4];
    const bool up16 = lane & 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = up16 ? acc[i] : acc[4 + i];
        a4[i] = up16 ? acc[4 + i] : acc[i];
        r4[i] = __shfl_xor_sync(kFullMask, send, 16);
    }
    cacc_merge(a4[0], a4[1], r4[0], r4[1]);
    cacc_merge(a4[2], a4[3], r4[2], r4[3]);
    const bool up8 = lane & 8;
    float p0 = up8 ? a4[2] : a4[0];
    float p1 = up8 ? a4[3] : a4[1];
    {
        const float s0 = up8 ? a4[0] : a4[2];
        const float s1 = up8 ? a4[1] : a4[3];
        const float q0 = __shfl_xor_sync(kFullMask, s0, 8);
        const float q1 = __shfl_xor_sync(kFullMask, s1, 8);
        cacc_merge(p0, p1, q0, q1);
    }
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) {
        const float q0 = __shfl_xor_sync(kFullMask, p0, off);
        const float q1 = __shfl_xor_sync(kFullMask, p1, off);
        cacc_merge(p0, p1, q0, q1);
    }
    v0 = p0;
    v1 = p1;
}

__global__ void __launch_bounds__(128, 2) gate_bwd_kernel(const GateBwdParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSmemBarOff);
    uint64_t* rxbar = reinterpret_cast<uint64_t*>(smem + kSmemRxBarOff);
    float* red = reinterpret_cast<float*>(smem + kSmemRedOff);  // [2][8 warps][8]
    float* rx = reinterpret_cast<float*>(smem + kSmemXchOff);   // [2][8 ranks][16]
    unsigned char* ring = smem + kSmemRingOff;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const long long q = cluster_index();
    const long long G = cluster_count();
    const int d = p.d;
    const int col0 = static_cast<int>(rank) * p.ncols;
    const bool active = tid < p.ngroups;
    const uint32_t row_bytes = static_cast<uint32_t>(p.ncols) * 2u;
    const uint32_t stage_bytes = kRows * row_bytes + 64u;
    const int stages = p.stages;
    const uint32_t xbytes = C * 8u * 4u;  // 4 streams x (hi, lo) from every CTA

    float2 w2[kS][4];
#pragma unroll
    for (int s = 0; s < kS; ++s) {
        if (active) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(p.w + s * d + col0 + 8 * tid));
            const float4 b = __ldg(reinterpret_cast<const float4*>(p.w + s * d + col0 + 8 * tid + 4));
            w2[s][0] = make_float2(a.x, a.y);
            w2[s][1] = make_float2(a.z, a.w);
            w2[s][2] = make_float2(b.x, b.y);
            w2[s][3] = make_float2(b.z, b.w);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) w2[s][e] = make_float2(0.f, 0.f);
        }
    }

    const long long nblocks = p.N / kBlockTokens;
    const long long myblocks = (nblocks > q) ? (nblocks - 1 - q) / G + 1 : 0;
    const long long ntok = myblocks * kBlockTokens;
    auto token_of = [&](long long j) {
        return (q + (j / kBlockTokens) * G) * kBlockTokens + (j % kBlockTokens);
    };

    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(&full[st], 1);
        mbar_init(&rxbar[0], 1);
        mbar_init(&rxbar[1], 1);
        fence_mbar_init();
        if (ntok > 0) mbar_arrive_expect_tx(&rxbar[0], xbytes);
        if (ntok > 1) mbar_arrive_expect_tx(&rxbar[1], xbytes);
    }
    cluster_sync();

    auto issue = [&](long long j) {
        const long long n = token_of(j);
        const int st = static_cast<int>(j % stages);
        unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        mbar_arrive_expect_tx(&full[st], stage_bytes);
        const uint16_t* xr = p.x + n * kS * d + col0;
        const uint16_t* kr = p.kv + n * (kS + 1) * d + col0;
        const uint16_t* gr = p.gout + n * kS * d + col0;
#pragma unroll
        for (int s = 0; s < kS; ++s) bulk_g2s(b + s * row_bytes, xr + s * d, row_bytes, &full[st]);
#pragma unroll
        for (int s = 0; s <= kS; ++s)
            bulk_g2s(b + (kS + s) * row_bytes, kr + s * d, row_bytes, &full[st]);
#pragma unroll
        for (int s = 0; s < kS; ++s)
            bulk_g2s(b + (2 * kS + 1 + s) * row_bytes, gr + s * d, row_bytes, &full[st]);
        bulk_g2s(b + kRows * row_bytes, p.saved + n * kS * 4, 64u, &full[st]);
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

    // dgate_s = sum_i g_{s,i} v_i (g*v exact in fp32; compensated sum); the
    // warp's 4 (hi, lo) pairs go to red[j & 1]
    auto reduce_pass = [&](long long j) {
        const int st = static_cast<int>(j % stages);
        if (!failed && !mbar_wait(&full[st], static_cast<uint32_t>((j / stages) & 1))) failed = true;
        const unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        if (active) {
            const uint4 vq = lds128(b + 2 * kS * row_bytes + 16 * tid);
            const float2 v2[4] = {bf2(vq.x), bf2(vq.y), bf2(vq.z), bf2(vq.w)};
#pragma unroll
            for (int s = 0; s < kS; ++s) {
                const uint4 gq = lds128(b + (2 * kS + 1 + s) * row_bytes + 16 * tid);
                const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
                float2 hi = make_float2(0.f, 0.f), lo = hi;
#pragma unroll
                for (int e = 0; e < 4; ++e) cacc_add_x2(hi, lo, mul2(bf2(gw[e]), v2[e]));
                float h = hi.x, l = lo.x;
                cacc_merge(h, l, hi.y, lo.y);
                acc[2 * s] = h;
                acc[2 * s + 1] = l;
            }
        }
        float v0, v1;
        warp_reduce_pairs4(acc, lane, v0, v1);
        if ((lane & 7) == 0) {
            const int sidx = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
            *reinterpret_cast<float2*>(red + (j & 1) * (kRedWarps * 8) + warp * 8 + sidx * 2) =
                make_float2(v0, v1);
        }
    };

    auto push = [&](long long j) {
        if (lane < kS) {
            const float* r = red + (j & 1) * (kRedWarps * 8);
            float a0 = r[2 * lane], a1 = r[2 * lane + 1];
            for (int wi = 1; wi < nwarps; ++wi)
                cacc_merge(a0, a1, r[wi * 8 + 2 * lane], r[wi * 8 + 2 * lane + 1]);
            const int slot = static_cast<int>(j & 1);
            const uint32_t dst = smem_addr(rx + (slot * 8 + rank) * 16 + 2 * lane);
            const uint32_t bar = smem_addr(&rxbar[slot]);
            for (uint32_t r2 = 0; r2 < C; ++r2)
                st_async_f2(map_to_rank(dst, r2), a0, a1, map_to_rank(bar, r2));
        }
    };

    // warp 0, lanes 0..3 (stream s = lane): per-stream scalars of token j in
    // fp64 from the cluster totals and the saved record, into cbuf[j & 1]:
    // A (hi, lo), -B, -Ck, gate.  rsqrt and the reciprocal start from fp32
    // estimates refined by one Newton step in fp64; exp is the fp64 routine.
    float* cbuf = reinterpret_cast<float*>(smem + kSmemCoefOff);  // [2][32]
    auto coefficients = [&](long long j, const unsigned char* b) {
        const int slot = static_cast<int>(j & 1);
        if (!failed && !mbar_wait_cluster(&rxbar[slot], static_cast<uint32_t>((j >> 1) & 1)))
            failed = true;
        if (lane < kS) {
            const float* r = rx + slot * 8 * 16 + 2 * lane;
            float hi = r[0], lo = r[1];
            for (uint32_t rr = 1; rr < C; ++rr) cacc_merge(hi, lo, r[rr * 16], r[rr * 16 + 1]);
            const float* sv = reinterpret_cast<const float*>(b + kRows * row_bytes);
            const float gate = sv[4 * lane + 0];
            const float dotf = sv[4 * lane + 1];
            const double rx_ = sv[4 * lane + 2];
            const double rk = sv[4 * lane + 3];
            const double dot = dotf;
            const double ad = fabs(dot);
            double ddot = 0.0;
            if (ad >= 1e-6 && gate != 0.f) {
                double y = rsqrtf(fabsf(dotf));
                y = y * (1.5 - 0.5 * ad * y * y);           // 1/sqrt(|dot|)
                const double sqm = ad * y;                  // sqrt(|dot|) = |sq|
                const double ex = exp(-sqm);
                const double den = 1.0 + ex;
                double rc = __frcp_rn(static_cast<float>(den));
                rc = rc * (2.0 - den * rc);                 // 1/(1 + e^-|sq|)
                const double dsig = ex * rc * rc;           // sigmoid(sq) sigmoid(-sq)
                const double dgate = static_cast<double>(hi) + static_cast<double>(lo);
                ddot = dgate * dsig * (0.5 * y);            // d sq / d dot = 0.5/sqrt(|dot|)
            }
            const double dd = dot / static_cast<double>(d);
            const double av = ddot * rx_ * rk;
            float* c = cbuf + slot * 32 + lane * 5;
            c[0] = static_cast<float>(av);
            c[1] = static_cast<float>(av - static_cast<double>(c[0]));
            c[2] = static_cast<float>(-(ddot * rx_ * rx_ * dd));
            c[3] = static_cast<float>(-(ddot * rk * rk * dd));
            c[4] = gate;
        }
    };

    if (ntok > 0) reduce_pass(0);
    __syncthreads();
    if (warp == 0 && ntok > 0) push(0);

    for (long long j = 0; j < ntok; ++j) {
        const long long n = token_of(j);
        const int slot = static_cast<int>(j & 1);
        const int st = static_cast<int>(j % stages);
        const unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        if (j + 1 < ntok) reduce_pass(j + 1);
        if (warp == 0) coefficients(j, b);
        // token j's scalars are published, red[(j+1)&1] is complete, and every
        // thread is done with token j-1 (its stage can be refilled)
        __syncthreads();
        if (tid == 0) {
            // re-arm this slot for token j + 2 before this CTA's push of token
            // j + 1, which every peer needs before it can push token j + 2
            if (j + 2 < ntok) mbar_arrive_expect_tx(&rxbar[slot], xbytes);
            if (j >= 1 && j - 1 + stages < ntok) {
                fence_proxy_async();
                issue(j - 1 + stages);
            }
        }
        if (warp == 0) {
            __syncwarp();
            if (j + 1 < ntok) push(j + 1);
        }

        // ---- elementwise: grad_x, grad_key, grad_v, grad_w (packed pairs)
        if (active) {
            float2 gv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) gv[e] = make_float2(0.f, 0.f);
            uint16_t* gxo = p.gx + n * kS * d + col0 + 8 * tid;
            uint16_t* gko = p.gkv + n * (kS + 1) * d + col0 + 8 * tid;
            const float* cb = cbuf + slot * 32;
#pragma unroll
            for (int s = 0; s < kS; ++s) {
                const float2 A2 = splat2(cb[s * 5 + 0]);
                const float2 Al2 = splat2(cb[s * 5 + 1]);
                const float2 nB2 = splat2(cb[s * 5 + 2]);
                const float2 nC2 = splat2(cb[s * 5 + 3]);
                const float2 G2 = splat2(cb[s * 5 + 4]);
                const uint4 xq = lds128(b + s * row_bytes + 16 * tid);
                const uint4 kq = lds128(b + (kS + s) * row_bytes + 16 * tid);
                const uint4 gq = lds128(b + (2 * kS + 1 + s) * row_bytes + 16 * tid);
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
                stg_cs(gxo + s * d, make_uint4(ox[0], ox[1], ox[2], ox[3]));
                stg_cs(gko + s * d, make_uint4(ok[0], ok[1], ok[2], ok[3]));
            }
            stg_cs(gko + kS * d, make_uint4(pack2(gv[0]), pack2(gv[1]), pack2(gv[2]), pack2(gv[3])));
        }
    }
    // ---- this cluster's grad_w for the slice: (hi, lo) in slots 2q, 2q+1, or
    // hi + lo in slot 0 when a single cluster covers a single block
    if (active) {
#pragma unroll
        for (int s = 0; s < kS; ++s) {
            float* o = p.partial + ((p.pair_slots ? 2 * q : q) * kS + s) * d + col0 + 8 * tid;
            if (p.pair_slots) {
                float* ol = o + static_cast<long long>(kS) * d;
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
    cluster_sync();
}

// grad_weight[i] from the cluster partials, merged in ascending order with
// error-free additions (bitwise reproducible).  pairs: slot 2q = hi, 2q+1 = lo.
__global__ void __launch_bounds__(256) wreduce_kernel(const GateWReduceParams p) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    const float* src = p.partial + i;
    if (!p.pairs) {
        float hi = 0.f, lo = 0.f;
        for (int b = 0; b < p.nblocks; ++b) cacc_add(hi, lo, __ldg(src + static_cast<size_t>(b) * p.stride));
        p.out[i] = __fadd_rn(hi, lo);
        return;
    }
    float hi = 0.f, lo = 0.f;
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
    cudaError_t e = cudaFuncSetAttribute(gate_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gate_bwd_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

cudaError_t gate_bwd_max_clusters(int cluster, int threads, int smem, int* out) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(cluster, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, gate_bwd_kernel, &cfg);
}

cudaError_t gate_bwd_launch(const GateBwdParams& p, const LaunchCfg& c, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(c.cluster * c.clusters, 1, 1);
    cfg.blockDim = dim3(c.threads, 1, 1);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gate_bwd_kernel, p);
}

cudaError_t gate_wreduce_launch(const GateWReduceParams& p, cudaStream_t s) {
    const int threads = 128;
    const int blocks = (p.n + threads - 1) / threads;
    wreduce_kernel<<<blocks, threads, 0, s>>>(p);
    return cudaPeekAtLastError();
}

}  // namespace eg
