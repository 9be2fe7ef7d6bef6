// GateConv, backward (TileOPs "Engram Operators", GateConv section,
// EngramGateConvBwdOp: dH, dk, dv and fp32 drms_w_h, drms_w_v, dconv_w from
// dY and the forward's saved vhat, alpha, rrms_h, rrms_k, rrms_v).
//
// Chain rule through the forward (see gateconv_fwd.cu), at the saved values:
//   u_t   = vhat_t rrms_v w_v,  c_t = sum_j cw_j u_{t-3+j},  dc = dY SiLU'(c)
//   du_t  = sum_j cw_j dc_{t+3-j}                  (transposed causal conv)
//   m     = rrms_v S4 / d,  S4 = sum w_v du vhat
//   dvhat = dY + rrms_v w_v du - rrms_v^2 m vhat,   dv = alpha dvhat
//   dalpha = sum dvhat v = S1 - rrms_v^2 m S3,  S1 = sum (dY + rrms_v w_v du) v,
//                                                 S3 = sum vhat v
//   dz    = dalpha alpha (1 - alpha),  Ah = dz rrms_h rrms_k / sqrt(d)
//   dH    = Ah w_h^2 k - Ah rrms_h^2 (S5/d) H,   S5 = sum H k w_h^2
//   dk    = Ah w_h^2 H - Ah rrms_k^2 (S5/d) k
//   drms_w_h += 2 Ah w_h H k,  drms_w_v += du vhat rrms_v,
//   dconv_w[j] += dc_t u_{t-3+j}
//
// One cluster per range of consecutive output tokens of one row; CTA `rank`
// owns a column slice, each thread 4 columns, and the ring of shared-memory
// stages holds the dY, vhat, v, H and k rows of one token per stage.
// Stepping through the tokens, a thread forms u_tau, c_tau and dc_tau and
// keeps the last three u and dc in registers; du of token t is complete once
// dc_{t+3} is known.  Per chunk of output tokens:
//   1  du and the partial sums S1, S3, S4, S5 over the warp's columns, sent
//      to the cluster (gateconv_xch.cuh); du stays in registers;
//   2  (one chunk behind) the totals give the per-token coefficients, and the
//      thread writes dv, dH and dk from the rows still in the ring.
// Three tokens before the range (for u) and after it (for dc) are streamed as
// a halo.  Weight gradients accumulate per thread over the range and go to
// the workspace, one slot per range; a second kernel sums the slots in
// ascending order.
#include "common.cuh"
#include "engram_internal.h"
#include "gateconv_xch.cuh"

namespace eg {
namespace {

using gc::kChunk;
constexpr int kRows = 5;  // dY, vhat, v, H, k
constexpr int kMask = gc::kStages - 1;
static_assert((gc::kStages & kMask) == 0, "stage count must be a power of two");
static_assert(gc::kStages >= 3 * kChunk + 3, "ring too short for two chunks and the look-ahead");

__global__ void __launch_bounds__(gc::kThreads, 1) gateconv_bwd_kernel(const GateConvBwdParams p) {
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
    const uint32_t stage_bytes = kRows * pitch;
    constexpr int stages = gc::kStages;

    const int m = q / p.ranges_per_row;
    const int t_out = (q - m * p.ranges_per_row) * p.range_len;
    const int t_end = min(p.T, t_out + p.range_len);
    const int t_first = t_out - min(3, t_out);
    const int t_last = min(p.T, t_end + 3);
    const int ntok = t_last - t_first;             // streamed tokens (halo included)
    const int nchunks = (t_end - t_out + kChunk - 1) / kChunk;
    const long long row0 = static_cast<long long>(m) * p.T;
    const uint32_t xbytes = static_cast<uint32_t>(parts) * gc::kVals * 4u;

    float wh[4], wv[4], cw[4][4];
    if (active) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p.wh + c0));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p.wv + c0));
        wh[0] = a.x; wh[1] = a.y; wh[2] = a.z; wh[3] = a.w;
        wv[0] = b.x; wv[1] = b.y; wv[2] = b.z; wv[3] = b.w;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 c = __ldg(reinterpret_cast<const float4*>(p.cw + static_cast<long long>(j) * d + c0));
            cw[j][0] = c.x; cw[j][1] = c.y; cw[j][2] = c.z; cw[j][3] = c.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            wh[e] = wv[e] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) cw[j][e] = 0.f;
        }
    }

    auto issue = [&](int j) {
        const int st = j & kMask;
        const long long off = (row0 + t_first + j) * d + col0;
        unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        mbar_arrive_expect_tx(&full[st], kRows * row_bytes);
        bulk_g2s(b, p.dY + off, row_bytes, &full[st]);
        bulk_g2s(b + pitch, p.vhat + off, row_bytes, &full[st]);
        bulk_g2s(b + 2 * pitch, p.v + off, row_bytes, &full[st]);
        bulk_g2s(b + 3 * pitch, p.H + off, row_bytes, &full[st]);
        bulk_g2s(b + 4 * pitch, p.k + off, row_bytes, &full[st]);
    };
    auto stage_of = [&](int t) -> const unsigned char* {
        return ring + static_cast<size_t>((t - t_first) & kMask) * stage_bytes + 8 * tid;
    };
    // this warp is done with token t's stage; the last warp refills it
    auto release = [&](int t) {
        const int j = t - t_first;
        const int st = j & kMask;
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&released[st], 1u) == static_cast<unsigned int>(nw - 1)) {
                released[st] = 0u;
                if (j + stages < ntok) {
                    fence_proxy_async();
                    issue(j + stages);
                }
            }
        }
    };

    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            released[s] = 0u;
        }
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&xbar[0], xbytes);
        if (nchunks > 1) mbar_arrive_expect_tx(&xbar[1], xbytes);
        const int pro = ntok < stages ? ntok : stages;
        for (int j = 0; j < pro; ++j) issue(j);
    }
    cluster_sync();

    float u1[4], u2[4], u3[4];     // u at tau-1, tau-2, tau-3
    float dc1[4], dc2[4], dc3[4];  // dc at tau-1, tau-2, tau-3
    float gwh[4], gwv[4], gcw[4][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        u1[e] = u2[e] = u3[e] = dc1[e] = dc2[e] = dc3[e] = 0.f;
        gwh[e] = gwv[e] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) gcw[j][e] = 0.f;
    }
    bool failed = false;

    // Step to token tau: u_tau, c_tau, dc_tau (zero outside [t_out, t_last)),
    // the dconv_w contributions of tau inside the range; returns dc_tau.
    auto advance = [&](int tau, float (&dcv)[4]) {
#pragma unroll
        for (int e = 0; e < 4; ++e) dcv[e] = 0.f;
        if (tau >= t_last) return;
        const int j = tau - t_first;
        if (!failed && !mbar_wait(&full[j & kMask], static_cast<uint32_t>((j / stages) & 1))) failed = true;
        const float rv = __ldg(p.rv + row0 + tau);
        if (active) {
            const unsigned char* b = stage_of(tau);
            float vh[4], u[4];
            unpack4(lds64(b + pitch), vh);
#pragma unroll
            for (int e = 0; e < 4; ++e) u[e] = vh[e] * rv * wv[e];
            if (tau >= t_out) {
                float dy[4];
                unpack4(lds64(b), dy);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float cc =
                        fmaf(cw[0][e], u3[e], fmaf(cw[1][e], u2[e], fmaf(cw[2][e], u1[e], cw[3][e] * u[e])));
                    const float s = __frcp_rn(1.0f + __expf(-cc));
                    dcv[e] = dy[e] * s * fmaf(cc, 1.0f - s, 1.0f);
                    if (tau < t_end) {
                        gcw[0][e] = fmaf(dcv[e], u3[e], gcw[0][e]);
                        gcw[1][e] = fmaf(dcv[e], u2[e], gcw[1][e]);
                        gcw[2][e] = fmaf(dcv[e], u1[e], gcw[2][e]);
                        gcw[3][e] = fmaf(dcv[e], u[e], gcw[3][e]);
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                u3[e] = u2[e];
                u2[e] = u1[e];
                u1[e] = u[e];
            }
        }
        // halo tokens are not needed after this step
        if (tau < t_out || tau >= t_end) release(tau);
    };
    auto push_dc = [&](const float (&dcv)[4]) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            dc3[e] = dc2[e];
            dc2[e] = dc1[e];
            dc1[e] = dcv[e];
        }
    };

    // fill the windows: tokens before the range, and dc of its first 3 tokens
    for (int tau = t_first; tau < t_out + 3; ++tau) {
        float dcv[4];
        advance(tau, dcv);
        push_dc(dcv);
    }

    const float inv_d = 1.0f / static_cast<float>(d);
    float duA[kChunk][4], duB[kChunk][4];  // du of chunk c and of chunk c - 1
    float P_l = 0.f, Q_l = 0.f, a_l = 0.f, Ah_l = 0.f, Bh_l = 0.f, Bk_l = 0.f;

    for (int c = 0; c <= nchunks; ++c) {
        // ---- 1: du and partial sums of chunk c
        float val = 0.f;
        if (c < nchunks) {
            float sums[gc::kVals];
#pragma unroll
            for (int w = 0; w < kChunk; ++w) {
                const int t = t_out + c * kChunk + w;
                float s1 = 0.f, s3 = 0.f, s4 = 0.f, s5 = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) duA[w][e] = 0.f;
                if (t < t_end) {
                    float dcv[4];
                    advance(t + 3, dcv);
                    float du[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        du[e] = fmaf(cw[3][e], dc3[e], fmaf(cw[2][e], dc2[e], fmaf(cw[1][e], dc1[e], cw[0][e] * dcv[e])));
                    push_dc(dcv);
                    const float rv = __ldg(p.rv + row0 + t);
                    if (active) {
                        const unsigned char* b = stage_of(t);
                        float dy[4], vh[4], vv[4], h[4], kk[4];
                        unpack4(lds64(b), dy);
                        unpack4(lds64(b + pitch), vh);
                        unpack4(lds64(b + 2 * pitch), vv);
                        unpack4(lds64(b + 3 * pitch), h);
                        unpack4(lds64(b + 4 * pitch), kk);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float wdu = wv[e] * du[e];
                            s1 = fmaf(fmaf(rv, wdu, dy[e]), vv[e], s1);
                            s3 = fmaf(vh[e], vv[e], s3);
                            s4 = fmaf(wdu, vh[e], s4);
                            s5 = fmaf(h[e] * kk[e], wh[e] * wh[e], s5);
                            gwv[e] = fmaf(du[e], vh[e] * rv, gwv[e]);
                            duA[w][e] = du[e];
                        }
                    }
                }
                sums[4 * w + 0] = s1;
                sums[4 * w + 1] = s3;
                sums[4 * w + 2] = s4;
                sums[4 * w + 3] = s5;
            }
            val = gc::warp_reduce16(sums, lane);
        }
        // ---- totals of chunk c - 1 -> coefficients of token (lane & 3)
        if (c >= 1) {
            const int buf = (c - 1) & 1;
            if (!failed && !mbar_wait_cluster(&xbar[buf], static_cast<uint32_t>(((c - 1) >> 1) & 1)))
                failed = true;
            if (tid == 0 && c + 1 < nchunks) mbar_arrive_expect_tx(&xbar[buf], xbytes);
            const float tot = gc::xch_total(xch, buf, parts, lane);
            const int tw = 4 * (lane & 3);
            const float S1 = __shfl_sync(kFullMask, tot, tw + 0);
            const float S3 = __shfl_sync(kFullMask, tot, tw + 1);
            const float S4 = __shfl_sync(kFullMask, tot, tw + 2);
            const float S5 = __shfl_sync(kFullMask, tot, tw + 3);
            const int t = min(t_out + (c - 1) * kChunk + (lane & 3), t_end - 1);
            const long long r = row0 + t;
            const float rv = __ldg(p.rv + r), a = __ldg(p.alpha + r);
            const float rh = __ldg(p.rh + r), rk = __ldg(p.rk + r);
            const float mu = rv * S4 * inv_d;
            const float q2 = rv * rv * mu;
            const float dalpha = fmaf(-q2, S3, S1);
            const float dz = dalpha * a * (1.0f - a);
            const float Ah = dz * rh * rk * p.inv_sqrt_d;
            const float e5 = S5 * inv_d;
            P_l = rv;
            Q_l = q2;
            a_l = a;
            Ah_l = Ah;
            Bh_l = Ah * rh * rh * e5;
            Bk_l = Ah * rk * rk * e5;
        }
        // ---- send chunk c
        if (c < nchunks) gc::xch_send(xch, xbar, c & 1, parts, part, val, lane, C);
        // ---- 2: dv, dH, dk of chunk c - 1
        if (c >= 1) {
#pragma unroll
            for (int w = 0; w < kChunk; ++w) {
                const int t = t_out + (c - 1) * kChunk + w;
                if (t >= t_end) break;
                const float P = __shfl_sync(kFullMask, P_l, w);
                const float Q = __shfl_sync(kFullMask, Q_l, w);
                const float a = __shfl_sync(kFullMask, a_l, w);
                const float Ah = __shfl_sync(kFullMask, Ah_l, w);
                const float Bh = __shfl_sync(kFullMask, Bh_l, w);
                const float Bk = __shfl_sync(kFullMask, Bk_l, w);
                if (active) {
                    const unsigned char* b = stage_of(t);
                    float dy[4], vh[4], h[4], kk[4], oh[4], ok[4], ov[4];
                    unpack4(lds64(b), dy);
                    unpack4(lds64(b + pitch), vh);
                    unpack4(lds64(b + 3 * pitch), h);
                    unpack4(lds64(b + 4 * pitch), kk);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float dvh = fmaf(-Q, vh[e], fmaf(P * wv[e], duB[w][e], dy[e]));
                        ov[e] = a * dvh;
                        const float aw = Ah * wh[e] * wh[e];
                        oh[e] = fmaf(aw, kk[e], -Bh * h[e]);
                        ok[e] = fmaf(aw, h[e], -Bk * kk[e]);
                        gwh[e] = fmaf(2.0f * Ah * wh[e], h[e] * kk[e], gwh[e]);
                    }
                    const long long off = (row0 + t) * d + c0;
                    stg_cs8(p.dH + off, pack4(oh));
                    stg_cs8(p.dk + off, pack4(ok));
                    stg_cs8(p.dv + off, pack4(ov));
                }
                release(t);
            }
        }
#pragma unroll
        for (int w = 0; w < kChunk; ++w)
#pragma unroll
            for (int e = 0; e < 4; ++e) duB[w][e] = duA[w][e];
    }

    // per-range weight-gradient partial: [dwh | dwv | dcw0..3], each d wide
    if (active) {
        float* o = p.partial + static_cast<long long>(q) * 6 * d + c0;
        stg_f4(o, gwh[0], gwh[1], gwh[2], gwh[3]);
        stg_f4(o + d, gwv[0], gwv[1], gwv[2], gwv[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) stg_f4(o + (2 + j) * d, gcw[j][0], gcw[j][1], gcw[j][2], gcw[j][3]);
    }
    if (failed) {
        atomicOr(p.err, kErrTimeout);
        if (tid == 0)
            for (int j = ntok > stages ? ntok - stages : 0; j < ntok; ++j)
                (void)mbar_wait(&full[j & kMask], static_cast<uint32_t>((j / stages) & 1));
    }
    cluster_sync();
}

// out[i] = sum_b partial[b*stride + i], b ascending.
__global__ void __launch_bounds__(256) gc_wreduce_kernel(const GateWReduceParams p) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    const float* src = p.partial + i;
    float acc = 0.f;
    int b = 0;
    for (; b + 8 <= p.nblocks; b += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __ldg(src + static_cast<size_t>(b + u) * p.stride);
#pragma unroll
        for (int u = 0; u < 8; ++u) acc = __fadd_rn(acc, v[u]);
    }
    for (; b < p.nblocks; ++b) acc = __fadd_rn(acc, __ldg(src + static_cast<size_t>(b) * p.stride));
    p.out[i] = acc;
}

}  // namespace

cudaError_t gateconv_bwd_prepare(int smem_bytes) {
    if (smem_bytes <= 0) return cudaSuccess;
    return cudaFuncSetAttribute(gateconv_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

cudaError_t gateconv_bwd_max_clusters(int cluster, int threads, int smem, int* out) {
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
    return cudaOccupancyMaxActiveClusters(out, gateconv_bwd_kernel, &cfg);
}

cudaError_t gateconv_bwd_launch(const GateConvBwdParams& p, const LaunchCfg& c, cudaStream_t s) {
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
    return cudaLaunchKernelEx(&cfg, gateconv_bwd_kernel, p);
}

cudaError_t gateconv_wreduce_launch(const GateWReduceParams& p, cudaStream_t s) {
    const int threads = 128;
    const int blocks = (p.n + threads - 1) / threads;
    gc_wreduce_kernel<<<blocks, threads, 0, s>>>(p);
    return cudaPeekAtLastError();
}

}  // namespace eg
