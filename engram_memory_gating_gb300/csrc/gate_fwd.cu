// Saved-state gate, forward (cuDNN Frontend "Engram saved-state gate",
// semantics and saved-state paragraphs).
//
// Per token n and stream s < 4:
//   rstd_X = 1/sqrt(mean(x^2) + eps), rstd_key = 1/sqrt(mean(k^2) + eps)
//   dot    = sum_i (x_i rstd_X) w_i (k_i rstd_key) = rstd_X rstd_key sum_i x_i w_i k_i
//   gate   = sigmoid(sign(dot) sqrt(max(|dot|, 1e-6)))
//   out    = bf16_rn(x + gate v)            (false mask: out = x, gate saved as 0)
//
// One pass over X and KV: a cluster of C CTAs owns a token row, each CTA a
// slice of ncols = d/C columns of every stream.  The slice rows of successive
// tokens (X: 4 rows, keys: 4 rows, v: 1 row) are bulk-copied into a ring of
// shared-memory stages.  The three per-stream reductions (sum x^2, sum k^2,
// sum x w k) are formed per thread, reduced across the warp, the CTA and the
// cluster (distributed shared memory), and every CTA then writes its slice of
// `out` from the X values still in registers.
//
// sum x w k is accumulated with error-free transformations (TwoProd via FMA,
// TwoSum) so that the dot product keeps its accuracy when the terms cancel;
// the squares are summed in plain fp32 (all terms positive).
#include "common.cuh"
#include "engram_internal.h"

namespace eg {
namespace {

constexpr int kS = 4;       // streams
constexpr int kVals = 16;   // per-thread partials: stream*4 + {ssx, ssk, hi, lo}

// Combine two (ssx, ssk, hi, lo) quads.
EG_DEV void quad_merge(float* a, const float* r) {
    a[0] = __fadd_rn(a[0], r[0]);
    a[1] = __fadd_rn(a[1], r[1]);
    cacc_merge(a[2], a[3], r[2], r[3]);
}

// Warp reduce-scatter of 16 partials.  On return lane l holds the warp total
// of stream s = 2*bit4(l) + bit3(l); kind = bit2(l) selects (ssx, ssk) [0] or
// (hi, lo) [1], returned in v0, v1.
EG_DEV void warp_reduce16(const float (&acc)[kVals], int lane, float& v0, float& v1) {
    float a8[8], r8[8];
    const bool up16 = lane & 16;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float send = up16 ? acc[i] : acc[8 + i];
        a8[i] = up16 ? acc[8 + i] : acc[i];
        r8[i] = __shfl_xor_sync(kFullMask, send, 16);
    }
    quad_merge(a8, r8);
    quad_merge(a8 + 4, r8 + 4);
    float a4[4], r4[4];
    const bool up8 = lane & 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = up8 ? a8[i] : a8[4 + i];
        a4[i] = up8 ? a8[4 + i] : a8[i];
        r4[i] = __shfl_xor_sync(kFullMask, send, 8);
    }
    quad_merge(a4, r4);
    const bool up4 = lane & 4;
    float p0 = up4 ? a4[2] : a4[0];
    float p1 = up4 ? a4[3] : a4[1];
    {
        const float s0 = up4 ? a4[0] : a4[2];
        const float s1 = up4 ? a4[1] : a4[3];
        const float q0 = __shfl_xor_sync(kFullMask, s0, 4);
        const float q1 = __shfl_xor_sync(kFullMask, s1, 4);
        if (up4) {
            cacc_merge(p0, p1, q0, q1);
        } else {
            p0 = __fadd_rn(p0, q0);
            p1 = __fadd_rn(p1, q1);
        }
    }
#pragma unroll
    for (int off = 2; off >= 1; off >>= 1) {
        const float q0 = __shfl_xor_sync(kFullMask, p0, off);
        const float q1 = __shfl_xor_sync(kFullMask, p1, off);
        if (up4) {
            cacc_merge(p0, p1, q0, q1);
        } else {
            p0 = __fadd_rn(p0, q0);
            p1 = __fadd_rn(p1, q1);
        }
    }
    v0 = p0;
    v1 = p1;
}

__global__ void __launch_bounds__(256) gate_fwd_kernel(const GateFwdParams p) {
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
    const long long q = cluster_index();
    const long long G = cluster_count();
    const int d = p.d;
    const int col0 = static_cast<int>(rank) * p.ncols;
    const bool active = tid < p.ngroups;
    const uint32_t row_bytes = static_cast<uint32_t>(p.ncols) * 2u;
    const uint32_t stage_bytes = 9u * row_bytes;
    const int stages = p.stages;

    // fused weight of this thread's 8 columns, all streams, kept in registers
    float w[kS][8];
#pragma unroll
    for (int s = 0; s < kS; ++s) {
        if (active) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(p.w + s * d + col0 + 8 * tid));
            const float4 b = __ldg(reinterpret_cast<const float4*>(p.w + s * d + col0 + 8 * tid + 4));
            w[s][0] = a.x; w[s][1] = a.y; w[s][2] = a.z; w[s][3] = a.w;
            w[s][4] = b.x; w[s][5] = b.y; w[s][6] = b.z; w[s][7] = b.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) w[s][e] = 0.f;
        }
    }

    const long long ntok = (p.N > q) ? (p.N - 1 - q) / G + 1 : 0;
    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(&full[st], 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](long long j) {
        const long long n = q + j * G;
        const int st = static_cast<int>(j % stages);
        unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        mbar_arrive_expect_tx(&full[st], stage_bytes);
        const uint16_t* xr = p.x + n * kS * d + col0;
        const uint16_t* kr = p.kv + n * (kS + 1) * d + col0;
#pragma unroll
        for (int s = 0; s < kS; ++s) bulk_g2s(b + s * row_bytes, xr + s * d, row_bytes, &full[st]);
#pragma unroll
        for (int s = 0; s <= kS; ++s)
            bulk_g2s(b + (kS + s) * row_bytes, kr + s * d, row_bytes, &full[st]);
    };
    if (tid == 0) {
        const long long pro = ntok < stages ? ntok : stages;
        for (long long j = 0; j < pro; ++j) issue(j);
    }

    bool failed = false;
    for (long long j = 0; j < ntok; ++j) {
        const long long n = q + j * G;
        const int st = static_cast<int>(j % stages);
        if (!failed && !mbar_wait(&full[st], static_cast<uint32_t>((j / stages) & 1))) failed = true;
        const unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;

        // ---- one pass: sum x^2, sum k^2, sum x w k (compensated) per stream
        float acc[kVals];
        uint4 xq[kS];
#pragma unroll
        for (int i = 0; i < kVals; ++i) acc[i] = 0.f;
        if (active) {
#pragma unroll
            for (int s = 0; s < kS; ++s) {
                xq[s] = lds128(b + s * row_bytes + 16 * tid);
                const uint4 kq = lds128(b + (kS + s) * row_bytes + 16 * tid);
                float xf[8], kf[8];
                unpack8(xq[s], xf);
                unpack8(kq, kf);
                float ssx = 0.f, ssk = 0.f, hi = 0.f, lo = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    ssx = fmaf(xf[e], xf[e], ssx);
                    ssk = fmaf(kf[e], kf[e], ssk);
                    // x*k is exact in fp32 (two 8-bit significands)
                    cacc_prod(hi, lo, __fmul_rn(xf[e], kf[e]), w[s][e]);
                }
                acc[4 * s + 0] = ssx;
                acc[4 * s + 1] = ssk;
                acc[4 * s + 2] = hi;
                acc[4 * s + 3] = lo;
            }
        } else {
#pragma unroll
            for (int s = 0; s < kS; ++s) xq[s] = make_uint4(0, 0, 0, 0);
        }
        float v0, v1;
        warp_reduce16(acc, lane, v0, v1);
        if ((lane & 3) == 0) {
            const int sidx = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
            const int kind = (lane >> 2) & 1;
            *reinterpret_cast<float2*>(red + warp * 16 + (sidx * 2 + kind) * 2) = make_float2(v0, v1);
        }
        __syncthreads();
        // every thread is past token j-1: its stage can be refilled
        if (tid == 0 && j >= 1 && j - 1 + stages < ntok) {
            fence_proxy_async();
            issue(j - 1 + stages);
        }
        float* slot = xch + (j & 1) * 16;
        if (warp == 0 && lane < 8) {
            const int kind = lane & 1;
            float a0 = red[2 * lane], a1 = red[2 * lane + 1];
            for (int wi = 1; wi < nwarps; ++wi) {
                const float b0 = red[wi * 16 + 2 * lane], b1 = red[wi * 16 + 2 * lane + 1];
                if (kind) {
                    cacc_merge(a0, a1, b0, b1);
                } else {
                    a0 = __fadd_rn(a0, b0);
                    a1 = __fadd_rn(a1, b1);
                }
            }
            *reinterpret_cast<float2*>(slot + 2 * lane) = make_float2(a0, a1);
        }
        cluster_sync();
        // ---- cluster totals, in rank order (identical in every CTA and warp)
        float t0 = 0.f, t1 = 0.f;
        if (lane < 8) {
            const int kind = lane & 1;
            const uint32_t a = smem_addr(slot + 2 * lane);
            const float2 r0 = ld_cluster_f2(map_to_rank(a, 0));
            t0 = r0.x;
            t1 = r0.y;
            for (uint32_t r = 1; r < C; ++r) {
                const float2 rr = ld_cluster_f2(map_to_rank(a, r));
                if (kind) {
                    cacc_merge(t0, t1, rr.x, rr.y);
                } else {
                    t0 = __fadd_rn(t0, rr.x);
                    t1 = __fadd_rn(t1, rr.y);
                }
            }
        }
        const float hi = __shfl_sync(kFullMask, t0, lane | 1);
        const float lo = __shfl_sync(kFullMask, t1, lane | 1);
        const bool on = (p.mask == nullptr) || (p.mask[n] != 0);
        float gate = 0.f;
        if (lane < 8 && (lane & 1) == 0) {
            const float inv_d = 1.0f / static_cast<float>(d);
            const float rstd_x = 1.0f / sqrtf(fmaf(t0, inv_d, p.eps));
            const float rstd_k = 1.0f / sqrtf(fmaf(t1, inv_d, p.eps));
            const float raw = __fadd_rn(hi, lo);
            const float dot = raw * rstd_x * rstd_k;
            float sq = sqrtf(fmaxf(fabsf(dot), 1e-6f));
            sq = dot > 0.f ? sq : (dot < 0.f ? -sq : 0.f);
            const float g = 1.0f / (1.0f + expf(-sq));
            gate = on ? g : 0.f;
            if (rank == 0 && warp == 0 && p.saved != nullptr)
                stg_f4(p.saved + (n * kS + (lane >> 1)) * 4, gate, dot, rstd_x, rstd_k);
        }
        float gs[kS];
#pragma unroll
        for (int s = 0; s < kS; ++s) gs[s] = __shfl_sync(kFullMask, gate, 2 * s);

        // ---- out = x + gate * v, one rounding; false mask copies X's bits
        if (active) {
            uint16_t* o = p.out + n * kS * d + col0 + 8 * tid;
            if (on) {
                float vf[8];
                unpack8(lds128(b + 2 * kS * row_bytes + 16 * tid), vf);
#pragma unroll
                for (int s = 0; s < kS; ++s) {
                    float xf[8];
                    unpack8(xq[s], xf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) xf[e] = fmaf(gs[s], vf[e], xf[e]);
                    stg_cs(o + s * d, pack8(xf));
                }
            } else {
#pragma unroll
                for (int s = 0; s < kS; ++s) stg_cs(o + s * d, xq[s]);
            }
        }
    }
    if (failed) atomicOr(p.err, kErrTimeout);
    // no CTA may leave while a peer can still read its exchange slots
    cluster_sync();
}

}  // namespace

cudaError_t gate_fwd_prepare(int smem_bytes) {
    return cudaFuncSetAttribute(gate_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_bytes);
}

cudaError_t gate_fwd_max_clusters(int cluster, int threads, int smem, int* out) {
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
    return cudaOccupancyMaxActiveClusters(out, gate_fwd_kernel, &cfg);
}

cudaError_t gate_fwd_launch(const GateFwdParams& p, const LaunchCfg& c, cudaStream_t s) {
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
    return cudaLaunchKernelEx(&cfg, gate_fwd_kernel, p);
}

}  // namespace eg
