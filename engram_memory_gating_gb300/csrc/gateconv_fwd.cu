// GateConv, forward (TileOPs "Engram Operators", GateConv section,
// EngramGateConvFwdOp: RMSNorm gating -> causal depthwise conv1d with 4 taps
// -> SiLU + residual; saves vhat, alpha, rrms_h, rrms_k, rrms_v).
//
// Per batch row m and token t (d columns, eps inside the root, mean over d):
//   rrms_h = 1/sqrt(mean H^2 + eps), rrms_k = 1/sqrt(mean k^2 + eps)
//   z      = rrms_h rrms_k sum_i H_i k_i w_h,i^2 / sqrt(d),  alpha = sigmoid(z)
//   vhat   = alpha v (fp32; stored as bf16)
//   rrms_v = 1/sqrt(alpha^2 mean v^2 + eps)   (= 1/sqrt(mean vhat^2 + eps))
//   u      = vhat rrms_v w_v
//   c_t    = sum_{j=0..3} conv_w[j] u_{t-3+j}   (zero before the row start)
//   Y      = c sigmoid(c) + vhat
//
// One cluster per range of consecutive tokens of one row; CTA `rank` owns a
// column slice and streams the H, k and v rows of its slice through a ring of
// shared-memory stages with bulk asynchronous copies.  Per chunk of tokens:
//   A  every warp forms sum H^2, sum k^2, sum H k w_h^2 and sum v^2 over its
//      lanes' columns and sends them to the cluster (gateconv_xch.cuh);
//   B  (one chunk behind) the totals give alpha and rrms_v; each thread runs
//      the causal conv over its 4 columns with the last three u values kept
//      in registers, and writes Y and vhat.
// A range that does not start at t = 0 first runs the 4 tokens before it
// (the halo) through A and B without writing them, to fill the window.
// Arithmetic on pairs of columns uses the packed fp32x2 instructions.
#include "common.cuh"
#include "engram_internal.h"
#include "gateconv_xch.cuh"

namespace eg {
namespace {

using gc::kChunk;

__global__ void __launch_bounds__(gc::kThreads, 2) gateconv_fwd_kernel(const GateConvFwdParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + gc::kOffFull);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + gc::kOffXbar);
    unsigned int* released = reinterpret_cast<unsigned int*>(smem + gc::kOffRel);
    float* xch = reinterpret_cast<float*>(smem + gc::kOffXch);
    unsigned char* ring = smem + p.ring_off;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nw = blockDim.x >> 5;
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int parts = static_cast<int>(C) * nw;
    const int part = static_cast<int>(rank) * nw + warp;
    const int q = static_cast<int>(cluster_index());
    const int d = p.d;
    const int col0 = static_cast<int>(rank) * p.ncols;
    const int cols = min(p.ncols, d - col0);
    const bool active = 4 * tid < cols;
    const int c0 = col0 + 4 * tid;
    const uint32_t row_bytes = 2u * static_cast<uint32_t>(cols);
    const uint32_t pitch = 2u * static_cast<uint32_t>(p.ncols);
    const uint32_t stage_bytes = 3u * pitch;
    constexpr int stages = gc::kStages;
    static_assert(stages % kChunk == 0, "a chunk must not wrap around the ring");

    // ranges start at multiples of kChunk, and so does the streamed halo, so
    // token t of the stream sits in window slot t % 4 = w for chunk position w
    const int m = q / p.ranges_per_row;
    const int t_out = (q - m * p.ranges_per_row) * p.range_len;
    const int t_end = min(p.T, t_out + p.range_len);
    const int t_first = t_out >= kChunk ? t_out - kChunk : 0;
    const int ntok = t_end - t_first;
    const int nchunks = (ntok + kChunk - 1) / kChunk;
    const long long row0 = static_cast<long long>(m) * p.T;
    const uint32_t xbytes = static_cast<uint32_t>(parts) * gc::kVals * 4u;

    float2 wh2[2], wv[2], cw[4][2];
    if (active) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p.wh + c0));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p.wv + c0));
        wh2[0] = make_float2(a.x * a.x, a.y * a.y);
        wh2[1] = make_float2(a.z * a.z, a.w * a.w);
        wv[0] = make_float2(b.x, b.y);
        wv[1] = make_float2(b.z, b.w);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 c = __ldg(reinterpret_cast<const float4*>(p.cw + static_cast<long long>(j) * d + c0));
            cw[j][0] = make_float2(c.x, c.y);
            cw[j][1] = make_float2(c.z, c.w);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            wh2[i] = wv[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 4; ++j) cw[j][i] = make_float2(0.f, 0.f);
        }
    }

    auto issue = [&](int j) {
        const int st = j % stages;
        const long long off = (row0 + t_first + j) * d + col0;
        unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        mbar_arrive_expect_tx(&full[st], 3u * row_bytes);
        bulk_g2s(b, p.H + off, row_bytes, &full[st]);
        bulk_g2s(b + pitch, p.k + off, row_bytes, &full[st]);
        bulk_g2s(b + 2 * pitch, p.v + off, row_bytes, &full[st]);
    };

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            released[s] = 0u;
        }
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        fence_mbar_init();
        // arm the exchange of chunks 0 and 1 (peers' bytes may land before or after)
        mbar_arrive_expect_tx(&xbar[0], xbytes);
        if (nchunks > 1) mbar_arrive_expect_tx(&xbar[1], xbytes);
        const int pro = ntok < stages ? ntok : stages;
        for (int j = 0; j < pro; ++j) issue(j);
    }
    // every CTA's barriers exist before any peer stores into its slots
    cluster_sync();

    float2 U[kChunk][2];  // u of the last four tokens, slot t % 4 (zero before the row start)
#pragma unroll
    for (int w = 0; w < kChunk; ++w) U[w][0] = U[w][1] = make_float2(0.f, 0.f);

    const float inv_d = 1.0f / static_cast<float>(d);
    bool failed = false;
    float alpha_l = 0.f, rv_l = 0.f;  // scalars of token (lane & 3) of chunk c - 1

    for (int c = 0; c <= nchunks; ++c) {
        // ---- A: partial sums of chunk c over this warp's columns (all waits
        // first, then branch-free arithmetic so the four tokens interleave)
        float val = 0.f;
        if (c < nchunks) {
            float sums[gc::kVals];
            const int j0 = c * kChunk;
            const unsigned char* b0 = ring + static_cast<size_t>(j0 % stages) * stage_bytes + 8 * tid;
            const uint32_t par = static_cast<uint32_t>((j0 / stages) & 1);
#pragma unroll
            for (int w = 0; w < kChunk; ++w)
                if (j0 + w < ntok && !failed && !mbar_wait(&full[j0 % stages + w], par)) failed = true;
#pragma unroll
            for (int w = 0; w < kChunk; ++w) {
                const unsigned char* b = b0 + static_cast<size_t>(w) * stage_bytes;
                const uint2 hq = lds64(b), kq = lds64(b + pitch), vq = lds64(b + 2 * pitch);
                const float2 h0 = bf2(hq.x), h1 = bf2(hq.y), k0 = bf2(kq.x), k1 = bf2(kq.y);
                const float2 v0 = bf2(vq.x), v1 = bf2(vq.y);
                const float2 hh = fma2(h1, h1, mul2(h0, h0));
                const float2 kk = fma2(k1, k1, mul2(k0, k0));
                const float2 hk = fma2(mul2(h1, k1), wh2[1], mul2(mul2(h0, k0), wh2[0]));
                const float2 vv = fma2(v1, v1, mul2(v0, v0));
                const bool ok = active && j0 + w < ntok;
                sums[4 * w + 0] = ok ? hh.x + hh.y : 0.f;
                sums[4 * w + 1] = ok ? kk.x + kk.y : 0.f;
                sums[4 * w + 2] = ok ? hk.x + hk.y : 0.f;
                sums[4 * w + 3] = ok ? vv.x + vv.y : 0.f;
            }
            val = gc::warp_reduce16(sums, lane);
        }
        // ---- totals of chunk c - 1 -> per-token scalars
        if (c >= 1) {
            const int buf = (c - 1) & 1;
            if (!failed && !mbar_wait_cluster(&xbar[buf], static_cast<uint32_t>(((c - 1) >> 1) & 1)))
                failed = true;
            if (tid == 0 && c + 1 < nchunks) mbar_arrive_expect_tx(&xbar[buf], xbytes);
            const float tot = gc::xch_total(xch, buf, parts, lane);
            const int tw = 4 * (lane & 3);
            const float sh = __shfl_sync(kFullMask, tot, tw + 0);
            const float sk = __shfl_sync(kFullMask, tot, tw + 1);
            const float shk = __shfl_sync(kFullMask, tot, tw + 2);
            const float sv = __shfl_sync(kFullMask, tot, tw + 3);
            const float rh = rsqrtf(fmaf(sh, inv_d, p.eps));
            const float rk = rsqrtf(fmaf(sk, inv_d, p.eps));
            const float z = rh * rk * shk * p.inv_sqrt_d;
            alpha_l = __fdividef(1.0f, 1.0f + __expf(-z));
            rv_l = rsqrtf(fmaf(alpha_l * alpha_l * sv, inv_d, p.eps));
            const int j = (c - 1) * kChunk + lane;
            if (rank == 0 && warp == 0 && lane < kChunk && j < ntok && t_first + j >= t_out) {
                const long long r = row0 + t_first + j;
                p.alpha[r] = alpha_l;
                p.rh[r] = rh;
                p.rk[r] = rk;
                p.rv[r] = rv_l;
            }
        }
        // ---- send chunk c (after this warp has read chunk c - 1)
        if (c < nchunks) gc::xch_send(xch, xbar, c & 1, parts, part, val, lane, C);
        // ---- B: conv, SiLU and outputs of chunk c - 1 (branch-free; stores
        // predicated)
        if (c >= 1) {
            const int j0 = (c - 1) * kChunk;
            const unsigned char* b0 =
                ring + static_cast<size_t>(j0 % stages) * stage_bytes + 2 * pitch + 8 * tid;
            const long long off0 = (row0 + t_first + j0) * d + c0;
#pragma unroll
            for (int w = 0; w < kChunk; ++w) {
                const float alpha = __shfl_sync(kFullMask, alpha_l, w);
                const float rv = __shfl_sync(kFullMask, rv_l, w);
                const uint2 vq = lds64(b0 + static_cast<size_t>(w) * stage_bytes);
                const float2 a2 = splat2(alpha), ar2 = splat2(alpha * rv);
                float2 vh[2], y[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float2 v2 = bf2(i == 0 ? vq.x : vq.y);
                    vh[i] = mul2(a2, v2);
                    const float2 u = mul2(mul2(ar2, v2), wv[i]);
                    const float2 cc =
                        fma2(cw[0][i], U[(w + 1) & 3][i],
                             fma2(cw[1][i], U[(w + 2) & 3][i], fma2(cw[2][i], U[(w + 3) & 3][i], mul2(cw[3][i], u))));
                    // SiLU(c) = c / (1 + e^-c)
                    const float2 rden = make_float2(gc::rcp_ftz(1.0f + gc::exp_neg_ftz(cc.x)), gc::rcp_ftz(1.0f + gc::exp_neg_ftz(cc.y)));
                    y[i] = fma2(cc, rden, vh[i]);
                    U[w][i] = u;
                }
                if (active && j0 + w < ntok && t_first + j0 + w >= t_out) {
                    const long long off = off0 + static_cast<long long>(w) * d;
                    stg_cs8(p.Y + off, make_uint2(pack2(y[0]), pack2(y[1])));
                    stg_cs8(p.vhat + off, make_uint2(pack2(vh[0]), pack2(vh[1])));
                }
            }
            // this warp is done with the chunk's stages; the last warp refills them
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                const int st0 = j0 % stages;
                if (atomicAdd(&released[st0], 1u) == static_cast<unsigned int>(nw - 1)) {
                    released[st0] = 0u;
                    fence_proxy_async();
                    for (int w = 0; w < kChunk && j0 + stages + w < ntok; ++w) issue(j0 + stages + w);
                }
            }
        }
    }
    if (failed) {
        atomicOr(p.err, kErrTimeout);
        // let copies issued by this CTA land before it leaves (bounded)
        if (tid == 0)
            for (int j = ntok > stages ? ntok - stages : 0; j < ntok; ++j)
                (void)mbar_wait(&full[j % stages], static_cast<uint32_t>((j / stages) & 1));
    }
    // no CTA leaves while a peer may still store into its slots
    cluster_sync();
}

}  // namespace

cudaError_t gateconv_fwd_prepare(int smem_bytes) {
    if (smem_bytes <= 0) return cudaSuccess;
    return cudaFuncSetAttribute(gateconv_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

cudaError_t gateconv_fwd_max_clusters(int cluster, int threads, int smem, int* out) {
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
    return cudaOccupancyMaxActiveClusters(out, gateconv_fwd_kernel, &cfg);
}

cudaError_t gateconv_fwd_launch(const GateConvFwdParams& p, const LaunchCfg& c, cudaStream_t s) {
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
    return cudaLaunchKernelEx(&cfg, gateconv_fwd_kernel, p);
}

}  // namespace eg
