// Saved-state gate, forward (cuDNN Frontend "Engram saved-state gate",
// semantics and saved-state paragraphs).
//
// Per token n and stream s < 4:
//   rstd_X = 1/sqrt(mean(x^2) + eps), rstd_key = 1/sqrt(mean(k^2) + eps)
//   dot    = sum_i (x_i rstd_X) w_i (k_i rstd_key) = rstd_X rstd_key sum_i x_i w_i k_i
//   gate   = sigmoid(sign(dot) sqrt(max(|dot|, 1e-6)))
//   out    = bf16_rn(x + gate v)            (false mask: out = x, gate saved as 0)
//
// One pass over X and KV.  A cluster of C CTAs owns a token row, each CTA a
// slice of d/C columns of every stream; each thread 8 columns.  The slice
// rows of successive tokens (X: 4 rows, keys: 4 rows, v: 1 row) arrive by
// 1-D bulk copies in a ring of shared-memory stages.  Per token the three
// per-stream sums (sum x^2, sum k^2, sum x w k) are formed per thread with
// packed fp32x2 arithmetic, reduced across the warp and the CTA, and every
// CTA pushes its 16 partials into the shared memory of every CTA of the
// cluster with st.async, completing on a per-slot mbarrier there: no cluster
// barrier per token.  The loop is software-pipelined: while the partials of
// token j travel, the CTA already reduces token j+1; one warp then turns the
// cluster totals of token j into gates (shared memory), and every thread
// writes its slice of token j's `out` from the X and v words it kept in
// registers, so a stage is refilled as soon as its reduction pass is done.
//
// sum x w k uses error-free transformations (TwoProd via FMA, TwoSum) so the
// dot product keeps its accuracy when the terms cancel; the squares are
// summed in plain fp32 (all terms positive).
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

__global__ void __launch_bounds__(128, 3) gate_fwd_kernel(const GateFwdParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSmemBarOff);
    uint64_t* rxbar = reinterpret_cast<uint64_t*>(smem + kSmemRxBarOff);
    float* red = reinterpret_cast<float*>(smem + kSmemRedOff);  // [2][warps][16]
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
    const uint32_t stage_bytes = 9u * row_bytes;
    const int stages = p.stages;
    const uint32_t xbytes = C * 16u * 4u;  // partial bytes arriving per token

    // fused weight of this thread's 8 columns, all streams, as 4 pairs each
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

    const long long ntok = (p.N > q) ? (p.N - 1 - q) / G + 1 : 0;
    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(&full[st], 1);
        mbar_init(&rxbar[0], 1);
        mbar_init(&rxbar[1], 1);
        fence_mbar_init();
        if (ntok > 0) mbar_arrive_expect_tx(&rxbar[0], xbytes);
        if (ntok > 1) mbar_arrive_expect_tx(&rxbar[1], xbytes);
    }
    // every CTA's exchange barriers are initialised and armed before any push
    cluster_sync();

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
    float* gbuf = reinterpret_cast<float*>(smem + kSmemCoefOff);  // [2][8]: 4 gates, on flag

    // reduction pass of token j: keeps its X and v words in registers (the
    // stage is free afterwards), leaves the warp's 16 partials in red[j & 1]
    auto reduce_pass = [&](long long j, uint4 (&xq)[kS], uint4& vq) {
        const int st = static_cast<int>(j % stages);
        if (!failed && !mbar_wait(&full[st], static_cast<uint32_t>((j / stages) & 1))) failed = true;
        const unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        float acc[kVals];
#pragma unroll
        for (int i = 0; i < kVals; ++i) acc[i] = 0.f;
        if (active) {
            vq = lds128(b + 2 * kS * row_bytes + 16 * tid);
#pragma unroll
            for (int s = 0; s < kS; ++s) {
                xq[s] = lds128(b + s * row_bytes + 16 * tid);
                const uint4 kq = lds128(b + (kS + s) * row_bytes + 16 * tid);
                const uint32_t xw[4] = {xq[s].x, xq[s].y, xq[s].z, xq[s].w};
                const uint32_t kw[4] = {kq.x, kq.y, kq.z, kq.w};
                float2 ssx = make_float2(0.f, 0.f), ssk = ssx, hi = ssx, lo = ssx;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x2 = bf2(xw[e]);
                    const float2 k2 = bf2(kw[e]);
                    ssx = fma2(x2, x2, ssx);
                    ssk = fma2(k2, k2, ssk);
                    // x*k is exact in fp32 (two 8-bit significands)
                    cacc_prod_x2(hi, lo, mul2(x2, k2), w2[s][e]);
                }
                float h = hi.x, l = lo.x;
                cacc_merge(h, l, hi.y, lo.y);
                acc[4 * s + 0] = __fadd_rn(ssx.x, ssx.y);
                acc[4 * s + 1] = __fadd_rn(ssk.x, ssk.y);
                acc[4 * s + 2] = h;
                acc[4 * s + 3] = l;
            }
        } else {
#pragma unroll
            for (int s = 0; s < kS; ++s) xq[s] = make_uint4(0, 0, 0, 0);
            vq = make_uint4(0, 0, 0, 0);
        }
        float v0, v1;
        warp_reduce16(acc, lane, v0, v1);
        if ((lane & 3) == 0) {
            const int sidx = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
            const int kind = (lane >> 2) & 1;
            float* r = red + (j & 1) * (32 * 16) + warp * 16 + (sidx * 2 + kind) * 2;
            *reinterpret_cast<float2*>(r) = make_float2(v0, v1);
        }
    };

    // warp 0: CTA total of token j's partials, pushed to every CTA's slot j&1
    auto push = [&](long long j) {
        if (lane < 8) {
            const int kind = lane & 1;
            const float* r = red + (j & 1) * (32 * 16);
            float a0 = r[2 * lane], a1 = r[2 * lane + 1];
            for (int wi = 1; wi < nwarps; ++wi) {
                const float b0 = r[wi * 16 + 2 * lane], b1 = r[wi * 16 + 2 * lane + 1];
                if (kind) {
                    cacc_merge(a0, a1, b0, b1);
                } else {
                    a0 = __fadd_rn(a0, b0);
                    a1 = __fadd_rn(a1, b1);
                }
            }
            const int slot = static_cast<int>(j & 1);
            const uint32_t dst = smem_addr(rx + (slot * 8 + rank) * 16 + 2 * lane);
            const uint32_t bar = smem_addr(&rxbar[slot]);
            for (uint32_t r2 = 0; r2 < C; ++r2)
                st_async_f2(map_to_rank(dst, r2), a0, a1, map_to_rank(bar, r2));
        }
    };

    // warp 0: gates of token j from the cluster totals (rank order) -> gbuf
    auto gates = [&](long long j, bool on) {
        const long long n = q + j * G;
        const int slot = static_cast<int>(j & 1);
        if (!failed && !mbar_wait_cluster(&rxbar[slot], static_cast<uint32_t>((j >> 1) & 1)))
            failed = true;
        float t0 = 0.f, t1 = 0.f;
        if (lane < 8) {
            const int kind = lane & 1;
            const float* r = rx + slot * 8 * 16 + 2 * lane;
            t0 = r[0];
            t1 = r[1];
            for (uint32_t rr = 1; rr < C; ++rr) {
                const float b0 = r[rr * 16], b1 = r[rr * 16 + 1];
                if (kind) {
                    cacc_merge(t0, t1, b0, b1);
                } else {
                    t0 = __fadd_rn(t0, b0);
                    t1 = __fadd_rn(t1, b1);
                }
            }
        }
        const float hi = __shfl_sync(kFullMask, t0, lane | 1);
        const float lo = __shfl_sync(kFullMask, t1, lane | 1);
        if (lane < 8 && (lane & 1) == 0) {
            const float inv_d = 1.0f / static_cast<float>(d);
            const float rstd_x = 1.0f / sqrtf(fmaf(t0, inv_d, p.eps));
            const float rstd_k = 1.0f / sqrtf(fmaf(t1, inv_d, p.eps));
            const float raw = __fadd_rn(hi, lo);
            const float dot = raw * rstd_x * rstd_k;
            float sq = sqrtf(fmaxf(fabsf(dot), 1e-6f));
            sq = dot > 0.f ? sq : (dot < 0.f ? -sq : 0.f);
            const float g = 1.0f / (1.0f + expf(-sq));
            const float gate = on ? g : 0.f;
            gbuf[slot * 8 + (lane >> 1)] = gate;
            if (rank == 0 && p.saved != nullptr)
                stg_f4(p.saved + (n * kS + (lane >> 1)) * 4, gate, dot, rstd_x, rstd_k);
        }
        if (lane == 0) gbuf[slot * 8 + 4] = on ? 1.f : 0.f;
    };

    uint4 xq_cur[kS], xq_nxt[kS], vq_cur, vq_nxt;
    uint8_t m_cur = 1, m_nxt = 1;
    if (ntok > 0) {
        if (p.mask != nullptr && warp == 0) m_cur = __ldg(p.mask + q);
        reduce_pass(0, xq_cur, vq_cur);
    }
    __syncthreads();
    if (tid == 0 && stages < ntok) {
        fence_proxy_async();
        issue(stages);
    }
    if (warp == 0 && ntok > 0) {
        __syncwarp();
        push(0);
    }

    for (long long j = 0; j < ntok; ++j) {
        const long long n = q + j * G;
        const int slot = static_cast<int>(j & 1);
        if (j + 1 < ntok) {
            if (p.mask != nullptr && warp == 0) m_nxt = __ldg(p.mask + n + G);
            reduce_pass(j + 1, xq_nxt, vq_nxt);
        }
        if (warp == 0) gates(j, m_cur != 0);
        // gates of token j are published; red[(j+1)&1] is complete; token
        // j+1's stage has been read by every thread
        __syncthreads();
        if (tid == 0) {
            // re-arm this slot for token j + 2 before this CTA's push of token
            // j + 1, which every peer needs before it can push token j + 2
            if (j + 2 < ntok) mbar_arrive_expect_tx(&rxbar[slot], xbytes);
            if (j + 1 + stages < ntok) {
                fence_proxy_async();
                issue(j + 1 + stages);
            }
        }
        if (warp == 0) {
            __syncwarp();
            if (j + 1 < ntok) push(j + 1);
        }

        // ---- out = x + gate * v, one rounding; a false mask copies X's bits
        if (active) {
            uint16_t* o = p.out + n * kS * d + col0 + 8 * tid;
            const float* gb = gbuf + slot * 8;
            if (gb[4] != 0.f) {
                const float2 v2[4] = {bf2(vq_cur.x), bf2(vq_cur.y), bf2(vq_cur.z), bf2(vq_cur.w)};
#pragma unroll
                for (int s = 0; s < kS; ++s) {
                    const float2 g2 = splat2(gb[s]);
                    const uint32_t xw[4] = {xq_cur[s].x, xq_cur[s].y, xq_cur[s].z, xq_cur[s].w};
                    uint4 ov;
                    ov.x = pack2(fma2(g2, v2[0], bf2(xw[0])));
                    ov.y = pack2(fma2(g2, v2[1], bf2(xw[1])));
                    ov.z = pack2(fma2(g2, v2[2], bf2(xw[2])));
                    ov.w = pack2(fma2(g2, v2[3], bf2(xw[3])));
                    stg_cs(o + s * d, ov);
                }
            } else {
#pragma unroll
                for (int s = 0; s < kS; ++s) stg_cs(o + s * d, xq_cur[s]);
            }
        }
#pragma unroll
        for (int s = 0; s < kS; ++s) xq_cur[s] = xq_nxt[s];
        vq_cur = vq_nxt;
        m_cur = m_nxt;
    }
    if (failed) atomicOr(p.err, kErrTimeout);
    // no CTA may leave while a peer can still push into its shared memory
    cluster_sync();
}

}  // namespace

cudaError_t gate_fwd_prepare(int smem_bytes) {
    cudaError_t e = cudaFuncSetAttribute(gate_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gate_fwd_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
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
