// GateConv, backward (TileOPs "Engram Operators", GateConv section,
// EngramGateConvBwdOp: dH, dk, dv and fp32 drms_w_h, drms_w_v, dconv_w from
// dY and the forward's saved vhat, alpha, rrms_h, rrms_k, rrms_v).
//
// Chain rule through the forward (see gateconv_fwd.cu), at the saved values:
//   u_t   = vhat_t rrms_v w_v,  c_t = sum_j cw_j u_{t-3+j},  dc = dY SiLU'(c)
//   du_t  = sum_j cw_j dc_{t+3-j}                  (transposed causal conv)
//   dvhat = dY + rrms_v w_v du - rrms_v^3 vhat R1/d,  R1 = sum w_v du vhat
//   dv    = alpha dvhat,  dalpha = sum dvhat v = A + rrms_v B - rrms_v^3 R1 Cs/d
//           with A = sum dY v, B = sum w_v du v, Cs = sum vhat v
//   dz    = dalpha alpha (1 - alpha),  z = rrms_h rrms_k sum H k w_h^2 / sqrt(d)
//   dH    = (dz rrms_h rrms_k/sqrt(d)) w_h^2 k - (dz rrms_h^2 z/d) H
//   dk    = (dz rrms_h rrms_k/sqrt(d)) w_h^2 H - (dz rrms_k^2 z/d) k
//   drms_w_h += 2 (dz rrms_h rrms_k/sqrt(d)) w_h H k
//   drms_w_v += du vhat rrms_v,   dconv_w[j] += dc_t u_{t-3+j}
//
// One in-order pass over a range of tokens of one batch row per cluster: at
// step tau the thread forms u_tau, c_tau and dc_tau for its columns, keeps the
// last four dc and three u in registers, and finalises token tau-3, whose du
// needs dc up to tau.  The ring of shared-memory stages keeps the rows of
// tokens tau-3 .. tau+2.  Three tokens before the range (for u) and three
// after it (for dc) are read as a halo; only their dY and vhat rows are
// loaded.  Per-range weight-gradient partials go to the workspace and a
// second kernel reduces them in ascending range order.
#include "common.cuh"
#include "engram_internal.h"

namespace eg {
namespace {

constexpr int kV = 4;  // columns per thread

EG_DEV void unpack4(const uint2& q, float (&f)[4]) {
    f[0] = bf_lo(q.x);
    f[1] = bf_hi(q.x);
    f[2] = bf_lo(q.y);
    f[3] = bf_hi(q.y);
}
EG_DEV uint2 pack4(const float (&f)[4]) {
    return make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
}
EG_DEV uint2 lds64(const void* p) { return *reinterpret_cast<const uint2*>(p); }
EG_DEV void stg_cs64(void* p, const uint2& v) {
    asm volatile("st.global.cs.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// Warp reduce-scatter of 8 plain sums; lane l ends with the warp total of
// value 4*bit4(l) + 2*bit3(l) + bit2(l).
EG_DEV float warp_reduce8(const float (&v)[8], int lane) {
    float a[4];
    const bool up16 = lane & 16;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = up16 ? v[i] : v[4 + i];
        a[i] = (up16 ? v[4 + i] : v[i]) + __shfl_xor_sync(kFullMask, send, 16);
    }
    const bool up8 = lane & 8;
    float b[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = up8 ? a[i] : a[2 + i];
        b[i] = (up8 ? a[2 + i] : a[i]) + __shfl_xor_sync(kFullMask, send, 8);
    }
    const bool up4 = lane & 4;
    float c = (up4 ? b[1] : b[0]) + __shfl_xor_sync(kFullMask, up4 ? b[0] : b[1], 4);
    c += __shfl_xor_sync(kFullMask, c, 2);
    c += __shfl_xor_sync(kFullMask, c, 1);
    return c;
}

// stage rows
constexpr int kRowDY = 0, kRowVhat = 1, kRowH = 2, kRowK = 3, kRowV = 4;

__global__ void __launch_bounds__(256) gateconv_bwd_kernel(const GateConvBwdParams p) {
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
    const int c0 = col0 + kV * tid;
    const bool active = tid < p.ngroups;
    const uint32_t row_bytes = static_cast<uint32_t>(p.ncols) * 2u;
    const uint32_t stage_bytes = 5u * row_bytes;
    const int stages = p.stages;

    const int m = q / p.ranges_per_row;
    const int t0 = (q % p.ranges_per_row) * p.range_len;
    const int t1 = min(p.T, t0 + p.range_len);
    const int first = t0 - min(3, t0);
    const int nstep = (t1 + 3) - first;                 // tau = first .. t1+2
    const int nload = min(t1 + 3, p.T) - first;         // tokens that exist

    float wh[kV], wv[kV], cw[4][kV];
    if (active) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p.wh + c0));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p.wv + c0));
        wh[0] = a.x; wh[1] = a.y; wh[2] = a.z; wh[3] = a.w;
        wv[0] = b.x; wv[1] = b.y; wv[2] = b.z; wv[3] = b.w;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 c = __ldg(reinterpret_cast<const float4*>(p.cw + j * d + c0));
            cw[j][0] = c.x; cw[j][1] = c.y; cw[j][2] = c.z; cw[j][3] = c.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < kV; ++e) {
            wh[e] = wv[e] = 0.f;
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
    auto issue = [&](int j) {
        const int tau = first + j;
        const long long r = row0 + tau;
        const int st = j % stages;
        unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        const bool own = tau >= t0 && tau < t1;
        mbar_arrive_expect_tx(&full[st], own ? 5u * row_bytes : 2u * row_bytes);
        bulk_g2s(b + kRowDY * row_bytes, p.dY + r * d + col0, row_bytes, &full[st]);
        bulk_g2s(b + kRowVhat * row_bytes, p.vhat + r * d + col0, row_bytes, &full[st]);
        if (own) {
            bulk_g2s(b + kRowH * row_bytes, p.H + r * d + col0, row_bytes, &full[st]);
            bulk_g2s(b + kRowK * row_bytes, p.k + r * d + col0, row_bytes, &full[st]);
            bulk_g2s(b + kRowV * row_bytes, p.v + r * d + col0, row_bytes, &full[st]);
        }
    };
    if (tid == 0) {
        const int pro = nload < stages ? nload : stages;
        for (int j = 0; j < pro; ++j) issue(j);
    }

    float u1[kV], u2[kV], u3[kV];          // u at tau-1, tau-2, tau-3
    float dc0[kV], dc1[kV], dc2[kV], dc3[kV];  // dc at tau, tau-1, tau-2, tau-3
    float gwh[kV], gwv[kV], gcw[4][kV];
#pragma unroll
    for (int e = 0; e < kV; ++e) {
        u1[e] = u2[e] = u3[e] = 0.f;
        dc0[e] = dc1[e] = dc2[e] = dc3[e] = 0.f;
        gwh[e] = gwv[e] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) gcw[j][e] = 0.f;
    }

    bool failed = false;
    for (int j = 0; j < nstep; ++j) {
        const int tau = first + j;
        // ---- early part for token tau: u, c, dc and the conv-weight grads
        float ut[kV], dct[kV];
#pragma unroll
        for (int e = 0; e < kV; ++e) ut[e] = dct[e] = 0.f;
        if (j < nload) {
            const int st = j % stages;
            if (!failed && !mbar_wait(&full[st], static_cast<uint32_t>((j / stages) & 1)))
                failed = true;
            if (active) {
                const unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
                const float rvt = __ldg(p.rv + row0 + tau);
                float vh[kV], dy[kV];
                unpack4(lds64(b + kRowVhat * row_bytes + 8 * tid), vh);
                unpack4(lds64(b + kRowDY * row_bytes + 8 * tid), dy);
#pragma unroll
                for (int e = 0; e < kV; ++e) {
                    ut[e] = vh[e] * rvt * wv[e];
                    if (tau >= t0) {
                        const float c = fmaf(cw[0][e], u3[e],
                                             fmaf(cw[1][e], u2[e], fmaf(cw[2][e], u1[e], cw[3][e] * ut[e])));
                        const float sg = 1.0f / (1.0f + __expf(-c));
                        dct[e] = dy[e] * sg * fmaf(c, 1.0f - sg, 1.0f);
                    }
                }
                if (tau >= t0 && tau < t1) {
#pragma unroll
                    for (int e = 0; e < kV; ++e) {
                        gcw[0][e] = fmaf(dct[e], u3[e], gcw[0][e]);
                        gcw[1][e] = fmaf(dct[e], u2[e], gcw[1][e]);
                        gcw[2][e] = fmaf(dct[e], u1[e], gcw[2][e]);
                        gcw[3][e] = fmaf(dct[e], ut[e], gcw[3][e]);
                    }
                }
            }
        }
#pragma unroll
        for (int e = 0; e < kV; ++e) {
            u3[e] = u2[e];
            u2[e] = u1[e];
            u1[e] = ut[e];
            dc3[e] = dc2[e];
            dc2[e] = dc1[e];
            dc1[e] = dc0[e];
            dc0[e] = dct[e];
        }

        // ---- finalise token sigma = tau - 3
        const int sigma = tau - 3;
        const bool fin = sigma >= t0 && sigma < t1;
        const long long rs = row0 + sigma;
        const unsigned char* bs = ring + static_cast<size_t>(((j - 3) % stages + stages) % stages) * stage_bytes;
        float du[kV];
        float sums[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint2 hq = make_uint2(0, 0), kq = make_uint2(0, 0), vq = make_uint2(0, 0);
        uint2 vhq = make_uint2(0, 0), dyq = make_uint2(0, 0);
#pragma unroll
        for (int e = 0; e < kV; ++e)
            du[e] = fmaf(cw[0][e], dc0[e], fmaf(cw[1][e], dc1[e], fmaf(cw[2][e], dc2[e], cw[3][e] * dc3[e])));
        if (fin && active) {
            dyq = lds64(bs + kRowDY * row_bytes + 8 * tid);
            vhq = lds64(bs + kRowVhat * row_bytes + 8 * tid);
            hq = lds64(bs + kRowH * row_bytes + 8 * tid);
            kq = lds64(bs + kRowK * row_bytes + 8 * tid);
            vq = lds64(bs + kRowV * row_bytes + 8 * tid);
            float dy[kV], vh[kV], hf[kV], kf[kV], vf[kV];
            unpack4(dyq, dy);
            unpack4(vhq, vh);
            unpack4(hq, hf);
            unpack4(kq, kf);
            unpack4(vq, vf);
#pragma unroll
            for (int e = 0; e < kV; ++e) {
                const float wdu = wv[e] * du[e];
                sums[0] = fmaf(wdu, vh[e], sums[0]);                 // R1
                sums[1] = fmaf(dy[e], vf[e], sums[1]);               // A
                sums[2] = fmaf(wdu, vf[e], sums[2]);                 // B
                sums[3] = fmaf(vh[e], vf[e], sums[3]);               // Cs
                sums[4] = fmaf(hf[e] * kf[e], wh[e] * wh[e], sums[4]);  // sum H k wh^2
            }
        }
        const float wsum = warp_reduce8(sums, lane);
        if ((lane & 3) == 0)
            red[warp * 8 + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1)] = wsum;
        __syncthreads();
        // token j-4 is finished by every thread: refill its stage
        if (tid == 0 && j >= 4 && j - 4 + stages < nload) {
            fence_proxy_async();
            issue(j - 4 + stages);
        }
        float* slot = xch + (j & 1) * 8;
        if (warp == 0 && lane < 8) {
            float a = red[lane];
            for (int wi = 1; wi < nwarps; ++wi) a += red[wi * 8 + lane];
            slot[lane] = a;
        }
        cluster_sync();
        float tot = 0.f;
        if (lane < 5) {
            const uint32_t a = smem_addr(slot + lane);
            tot = ld_cluster_f(map_to_rank(a, 0));
            for (uint32_t rr = 1; rr < C; ++rr) tot += ld_cluster_f(map_to_rank(a, rr));
        }
        const float R1 = __shfl_sync(kFullMask, tot, 0);
        const float sA = __shfl_sync(kFullMask, tot, 1);
        const float sB = __shfl_sync(kFullMask, tot, 2);
        const float sC = __shfl_sync(kFullMask, tot, 3);
        const float sHK = __shfl_sync(kFullMask, tot, 4);
        if (fin && active) {
            const float alpha = __ldg(p.alpha + rs);
            const float rh = __ldg(p.rh + rs);
            const float rk = __ldg(p.rk + rs);
            const float rv = __ldg(p.rv + rs);
            const float inv_d = 1.0f / static_cast<float>(d);
            const float rv3 = rv * rv * rv;
            const float K1 = rv3 * R1 * inv_d;
            const float dalpha = fmaf(rv, sB, sA) - K1 * sC;
            const float dz = dalpha * alpha * (1.0f - alpha);
            const float z = rh * rk * sHK * p.inv_sqrt_d;
            const float cH1 = dz * rh * rk * p.inv_sqrt_d;
            const float cH2 = dz * rh * rh * z * inv_d;
            const float cK2 = dz * rk * rk * z * inv_d;
            float dy[kV], vh[kV], hf[kV], kf[kV], oh[kV], ok[kV], ov[kV];
            unpack4(dyq, dy);
            unpack4(vhq, vh);
            unpack4(hq, hf);
            unpack4(kq, kf);
#pragma unroll
            for (int e = 0; e < kV; ++e) {
                const float dvh = fmaf(rv * wv[e], du[e], fmaf(-K1, vh[e], dy[e]));
                ov[e] = alpha * dvh;
                const float w2 = wh[e] * wh[e];
                oh[e] = fmaf(cH1 * w2, kf[e], -cH2 * hf[e]);
                ok[e] = fmaf(cH1 * w2, hf[e], -cK2 * kf[e]);
                gwh[e] = fmaf(2.0f * cH1 * wh[e], hf[e] * kf[e], gwh[e]);
                gwv[e] = fmaf(du[e] * rv, vh[e], gwv[e]);
            }
            stg_cs64(p.dH + rs * d + c0, pack4(oh));
            stg_cs64(p.dk + rs * d + c0, pack4(ok));
            stg_cs64(p.dv + rs * d + c0, pack4(ov));
        }
    }
    // per-range weight-gradient partial: [dwh | dwv | dcw0..3], each d wide
    if (active && nstep > 0) {
        float* o = p.partial + static_cast<long long>(q) * 6 * d + c0;
        stg_f4(o, gwh[0], gwh[1], gwh[2], gwh[3]);
        stg_f4(o + d, gwv[0], gwv[1], gwv[2], gwv[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) stg_f4(o + (2 + j) * d, gcw[j][0], gcw[j][1], gcw[j][2], gcw[j][3]);
    }
    if (failed) atomicOr(p.err, kErrTimeout);
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
    return cudaFuncSetAttribute(gateconv_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_bytes);
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
