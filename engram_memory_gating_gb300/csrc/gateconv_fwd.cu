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
// A range that does not start at t = 0 first runs the 3 tokens before it
// (the halo) through A and B without writing them, to fill the window.
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

    const int m = q / p.ranges_per_row;
    const int t_out = (q - m * p.ranges_per_row) * p.range_len;
    const int t_end = min(p.T, t_out + p.range_len);
    const int t_first = t_out - min(3, t_out);
    const int ntok = t_end - t_first;
    const int nchunks = (ntok + kChunk - 1) / kChunk;
    const long long row0 = static_cast<long long>(m) * p.T;
    const uint32_t xbytes = static_cast<uint32_t>(parts) * gc::kVals * 4u;

    float wh2[4], wv[4], cw[4][4];
    if (active) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p.wh + c0));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p.wv + c0));
        wh2[0] = a.x * a.x; wh2[1] = a.y * a.y; wh2[2] = a.z * a.z; wh2[3] = a.w * a.w;
        wv[0] = b.x; wv[1] = b.y; wv[2] = b.z; wv[3] = b.w;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 c = __ldg(reinterpret_cast<const float4*>(p.cw + static_cast<long long>(j) * d + c0));
            cw[j][0] = c.x; cw[j][1] = c.y; cw[j][2] = c.z; cw[j][3] = c.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            wh2[e] = wv[e] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) cw[j][e] = 0.f;
        }
    }

    auto issue = [&](int j, int st) {
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
        for (int j = 0; j < pro; ++j) issue(j, j);
    }
    // every CTA's barriers exist before any peer stores into its slots
    cluster_sync();

    float u1[4], u2[4], u3[4];  // u at t-1, t-2, t-3 (zero before the row start)
#pragma unroll
    for (int e = 0; e < 4; ++e) u1[e] = u2[e] = u3[e] = 0.f;

    const float inv_d = 1.0f / static_cast<float>(d);
    bool failed = false;
    int stA = 0, stB = 0;
    uint32_t phA = 0;
    float alpha_l = 0.f, rv_l = 0.f;  // scalars of token (lane & 3) of chunk c - 1

    for (int c = 0; c <= nchunks; ++c) {
        // ---- A: partial sums of chunk c over this warp's columns
        float val = 0.f;
        if (c < nchunks) {
            float sums[gc::kVals];
#pragma unroll
            for (int w = 0; w < kChunk; ++w) {
                float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
                if (c * kChunk + w < ntok) {
                    if (!failed && !mbar_wait(&full[stA], phA)) failed = true;
                    if (active) {
                        const unsigned char* b = ring + static_cast<size_t>(stA) * stage_bytes + 8 * tid;
                        float h[4], kk[4], vv[4];
                        unpack4(lds64(b), h);
                        unpack4(lds64(b + pitch), kk);
                        unpack4(lds64(b + 2 * pitch), vv);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            s0 = fmaf(h[e], h[e], s0);
                            s1 = fmaf(kk[e], kk[e], s1);
                            s2 = fmaf(h[e] * kk[e], wh2[e], s2);
                            s3 = fmaf(vv[e], vv[e], s3);
                        }
                    }
                    if (++stA == stages) {
                        stA = 0;
                        phA ^= 1u;
                    }
                }
                sums[4 * w + 0] = s0;
                sums[4 * w + 1] = s1;
                sums[4 * w + 2] = s2;
                sums[4 * w + 3] = s3;
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
            alpha_l = 1.0f / (1.0f + __expf(-z));
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
        // ---- B: conv, SiLU and outputs of chunk c - 1
        if (c >= 1) {
#pragma unroll
            for (int w = 0; w < kChunk; ++w) {
                const int j = (c - 1) * kChunk + w;
                if (j >= ntok) break;
                const float alpha = __shfl_sync(kFullMask, alpha_l, w);
                const float rv = __shfl_sync(kFullMask, rv_l, w);
                const int t = t_first + j;
                if (active) {
                    const unsigned char* b = ring + static_cast<size_t>(stB) * stage_bytes + 2 * pitch + 8 * tid;
                    float vv[4], y[4], vh[4];
                    unpack4(lds64(b), vv);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        vh[e] = alpha * vv[e];
                        const float u = vh[e] * rv * wv[e];
                        const float cc =
                            fmaf(cw[0][e], u3[e], fmaf(cw[1][e], u2[e], fmaf(cw[2][e], u1[e], cw[3][e] * u)));
                        y[e] = cc / (1.0f + __expf(-cc)) + vh[e];
                        u3[e] = u2[e];
                        u2[e] = u1[e];
                        u1[e] = u;
                    }
                    if (t >= t_out) {
                        const long long off = (row0 + t) * d + c0;
                        stg_cs8(p.Y + off, pack4(y));
                        stg_cs8(p.vhat + off, pack4(vh));
                    }
                }
                // this warp is done with the stage; the last warp refills it
                __syncwarp();
                if (lane == 0) {
                    __threadfence_block();
                    if (atomicAdd(&released[stB], 1u) == static_cast<unsigned int>(nw - 1)) {
                        released[stB] = 0u;
                        if (j + stages < ntok) {
                            fence_proxy_async();
                            issue(j + stages, stB);
                        }
                    }
                }
                if (++stB == stages) stB = 0;
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
