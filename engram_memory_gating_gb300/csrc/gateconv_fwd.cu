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
// Work layout: the M*T tokens are cut into ranges of consecutive tokens of one
// batch row; one cluster of C CTAs walks a range in order, each CTA a column
// slice, each thread 8 columns.  The last three u values of a thread's
// columns stay in registers (a sliding window), so the conv costs no extra
// memory traffic; a range that does not start at t = 0 first recomputes u for
// the three tokens before it (the halo) without writing them.
#include "common.cuh"
#include "engram_internal.h"

namespace eg {
namespace {

// Warp reduce-scatter of 4 plain sums; lane l ends with the warp total of
// value 2*bit4(l) + bit3(l).
EG_DEV float warp_reduce4(const float (&v)[4], int lane) {
    const bool up16 = lane & 16;
    float a0 = up16 ? v[2] : v[0];
    float a1 = up16 ? v[3] : v[1];
    const float s0 = up16 ? v[0] : v[2];
    const float s1 = up16 ? v[1] : v[3];
    a0 += __shfl_xor_sync(kFullMask, s0, 16);
    a1 += __shfl_xor_sync(kFullMask, s1, 16);
    const bool up8 = lane & 8;
    float b = up8 ? a1 : a0;
    const float s = up8 ? a0 : a1;
    b += __shfl_xor_sync(kFullMask, s, 8);
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) b += __shfl_xor_sync(kFullMask, b, off);
    return b;
}

__global__ void __launch_bounds__(256) gateconv_fwd_kernel(const GateConvFwdParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSmemBarOff);
    float* red = reinterpret_cast<float*>(smem + kSmemRedOff);
    float* xch = reinterpret_cast<float*>(smem + kSmemXchOff);
    unsigned char* ring = smem + kSmemRingOff;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int q = static_cast<int>(cluster_index());
    const int d = p.d;
    const int col0 = static_cast<int>(rank) * p.ncols;
    const int c0 = col0 + 8 * tid;
    const bool active = tid < p.ngroups;
    const uint32_t row_bytes = static_cast<uint32_t>(p.ncols) * 2u;
    const uint32_t stage_bytes = 3u * row_bytes;
    const int stages = p.stages;

    const int m = q / p.ranges_per_row;
    const int t0 = (q % p.ranges_per_row) * p.range_len;
    const int t1 = min(p.T, t0 + p.range_len);
    const int first = t0 - min(3, t0);
    const long long ntok = (m < p.M && t0 < p.T) ? (t1 - first) : 0;

    float wh2[8], wv[8], cw[4][8];
    if (active) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(p.wh + c0 + 4 * h));
            const float4 b = __ldg(reinterpret_cast<const float4*>(p.wv + c0 + 4 * h));
            wh2[4 * h + 0] = a.x * a.x; wh2[4 * h + 1] = a.y * a.y;
            wh2[4 * h + 2] = a.z * a.z; wh2[4 * h + 3] = a.w * a.w;
            wv[4 * h + 0] = b.x; wv[4 * h + 1] = b.y; wv[4 * h + 2] = b.z; wv[4 * h + 3] = b.w;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 c = __ldg(reinterpret_cast<const float4*>(p.cw + j * d + c0 + 4 * h));
                cw[j][4 * h + 0] = c.x; cw[j][4 * h + 1] = c.y;
                cw[j][4 * h + 2] = c.z; cw[j][4 * h + 3] = c.w;
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            wh2[e] = 0.f;
            wv[e] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) cw[j][e] = 0.f;
        }
    }

    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(&full[st], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const long long row0 = static_cast<long long>(m) * p.T;
    auto issue = [&](long long j) {
        const long long r = row0 + first + j;
        const int st = static_cast<int>(j % stages);
        unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        mbar_arrive_expect_tx(&full[st], stage_bytes);
        bulk_g2s(b, p.H + r * d + col0, row_bytes, &full[st]);
        bulk_g2s(b + row_bytes, p.k + r * d + col0, row_bytes, &full[st]);
        bulk_g2s(b + 2 * row_bytes, p.v + r * d + col0, row_bytes, &full[st]);
    };
    if (tid == 0) {
        const long long pro = ntok < stages ? ntok : stages;
        for (long long j = 0; j < pro; ++j) issue(j);
    }

    float u1[8], u2[8], u3[8];  // u at t-1, t-2, t-3 (zero before the row start)
#pragma unroll
    for (int e = 0; e < 8; ++e) u1[e] = u2[e] = u3[e] = 0.f;

    bool failed = false;
    for (long long j = 0; j < ntok; ++j) {
        const int t = first + static_cast<int>(j);
        const long long r = row0 + t;
        const int st = static_cast<int>(j % stages);
        if (!failed && !mbar_wait(&full[st], static_cast<uint32_t>((j / stages) & 1))) failed = true;
        const unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;

        float part[4] = {0.f, 0.f, 0.f, 0.f};  // sum H^2, sum k^2, sum H k w_h^2, sum v^2
        uint4 vq = make_uint4(0, 0, 0, 0);
        if (active) {
            float hf[8], kf[8], vf[8];
            unpack8(lds128(b + 16 * tid), hf);
            unpack8(lds128(b + row_bytes + 16 * tid), kf);
            vq = lds128(b + 2 * row_bytes + 16 * tid);
            unpack8(vq, vf);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                part[0] = fmaf(hf[e], hf[e], part[0]);
                part[1] = fmaf(kf[e], kf[e], part[1]);
                part[2] = fmaf(hf[e] * kf[e], wh2[e], part[2]);
                part[3] = fmaf(vf[e], vf[e], part[3]);
            }
        }
        const float wsum = warp_reduce4(part, lane);
        if ((lane & 7) == 0) red[warp * 4 + ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1)] = wsum;
        __syncthreads();
        if (tid == 0 && j >= 1 && j - 1 + stages < ntok) {
            fence_proxy_async();
            issue(j - 1 + stages);
        }
        float* slot = xch + (j & 1) * 4;
        if (warp == 0 && lane < 4) {
            float a = red[lane];
            for (int wi = 1; wi < nwarps; ++wi) a += red[wi * 4 + lane];
            slot[lane] = a;
        }
        cluster_sync();
        float tot = 0.f;
        if (lane < 4) {
            const uint32_t a = smem_addr(slot + lane);
            tot = ld_cluster_f(map_to_rank(a, 0));
            for (uint32_t rr = 1; rr < C; ++rr) tot += ld_cluster_f(map_to_rank(a, rr));
        }
        const float sh = __shfl_sync(kFullMask, tot, 0);
        const float sk = __shfl_sync(kFullMask, tot, 1);
        const float shk = __shfl_sync(kFullMask, tot, 2);
        const float sv = __shfl_sync(kFullMask, tot, 3);
        const float inv_d = 1.0f / static_cast<float>(d);
        const float rh = 1.0f / sqrtf(fmaf(sh, inv_d, p.eps));
        const float rk = 1.0f / sqrtf(fmaf(sk, inv_d, p.eps));
        const float z = rh * rk * shk * p.inv_sqrt_d;
        const float alpha = 1.0f / (1.0f + expf(-z));
        const float rv = 1.0f / sqrtf(fmaf(alpha * alpha * sv, inv_d, p.eps));
        const bool out_tok = t >= t0;
        if (out_tok && rank == 0 && tid == 0) {
            p.alpha[r] = alpha;
            p.rh[r] = rh;
            p.rk[r] = rk;
            p.rv[r] = rv;
        }
        if (active) {
            float vf[8], y[8], vh[8];
            unpack8(vq, vf);
            const float s = alpha;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                vh[e] = s * vf[e];
                const float u = vh[e] * rv * wv[e];
                const float c = fmaf(cw[0][e], u3[e], fmaf(cw[1][e], u2[e], fmaf(cw[2][e], u1[e], cw[3][e] * u)));
                y[e] = c / (1.0f + __expf(-c)) + vh[e];
                u3[e] = u2[e];
                u2[e] = u1[e];
                u1[e] = u;
            }
            if (out_tok) {
                stg_cs(p.Y + r * d + c0, pack8(y));
                stg_cs(p.vhat + r * d + c0, pack8(vh));
            }
        }
    }
    if (failed) atomicOr(p.err, kErrTimeout);
    cluster_sync();
}

}  // namespace

cudaError_t gateconv_fwd_prepare(int smem_bytes) {
    return cudaFuncSetAttribute(gateconv_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_bytes);
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
