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
#include <type_traits>

#include "common.cuh"
#include "engram_internal.h"
#include "gateconv_xch.cuh"

namespace eg {
namespace {

using gc::kChunk;

// Two CTA shapes: kW = 8 warps (at most 1024 columns, two CTAs per SM) and
// kW = 16 warps (at most 2048 columns, one CTA per SM, for rows that then
// split over fewer CTAs).  Shared memory: a fixed layout, so that every ring
// address of a token is a chunk base plus an immediate.  Each row slot holds
// the widest column slice of the shape (8 kW 32 bytes); a narrower slice
// leaves the slot's tail zero, which the threads without columns read.
constexpr int kRows = 3;                         // H, k, v
constexpr int kStages = gc::kStages;             // 16 one-token stages
constexpr int kSlots = kStages / kChunk;         // 4 chunk slots of the ring
constexpr int kOffFull = 0;                      // [kSlots] chunk-slot mbarriers
constexpr int kOffXbar = 128;                    // [2] cluster-exchange mbarriers
constexpr int kOffRel = 160;                     // [kStages] stage release counters
constexpr int kOffArr = 224;                     // [2] per-chunk arrival counters
constexpr int kOffLocal = 256;                   // [2][kW warps][16] warp totals
template <int kW>
struct FwdShape {
    static constexpr int kPitch = 256 * kW;      // bytes per row slot
    static constexpr int kStageBytes = kRows * kPitch;
    static constexpr int kOffTot = kOffLocal + 2 * kW * gc::kVals * 4;   // [2][8 ranks][16] CTA totals
    static constexpr int kRingOff = (kOffTot + 2 * 8 * gc::kVals * 4 + 127) / 128 * 128;
    static constexpr int kSmem = kRingOff + kStages * kStageBytes;
    static_assert(kSmem <= 232448 / (kW == 8 ? 2 : 1) - 1024, "shared memory of the CTAs an SM holds");
};
static_assert(kStages % kChunk == 0, "a chunk must not wrap around the ring");

template <int kW>
__global__ void __launch_bounds__(32 * kW, kW == 8 ? 2 : 1) gateconv_fwd_kernel(const GateConvFwdParams p) {
    constexpr int kPitch = FwdShape<kW>::kPitch;
    constexpr int kStageBytes = FwdShape<kW>::kStageBytes;
    constexpr int kOffTot = FwdShape<kW>::kOffTot;
    constexpr int kRingOff = FwdShape<kW>::kRingOff;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffFull);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + kOffXbar);
    unsigned int* released = reinterpret_cast<unsigned int*>(smem + kOffRel);
    unsigned int* arrived = reinterpret_cast<unsigned int*>(smem + kOffArr);
    float* local = reinterpret_cast<float*>(smem + kOffLocal);
    float* tot = reinterpret_cast<float*>(smem + kOffTot);
    unsigned char* ring = smem + kRingOff;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nw = blockDim.x >> 5;
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int q = static_cast<int>(cluster_index());
    const int d = p.d;
    const int col0 = static_cast<int>(rank) * p.ncols;
    const int cols = min(p.ncols, d - col0);
    const bool active = 4 * tid < cols;
    const int c0 = col0 + 4 * tid;
    const uint32_t row_bytes = 2u * static_cast<uint32_t>(cols);

    // ranges start at multiples of kChunk, and so does the streamed halo, so
    // token t of the stream sits in window slot t % 4 = w for chunk position w
    const int m = q / p.ranges_per_row;
    const int t_out = (q - m * p.ranges_per_row) * p.range_len;
    const int t_end = min(p.T, t_out + p.range_len);
    const int t_first = t_out >= kChunk ? t_out - kChunk : 0;
    const int ntok = t_end - t_first;
    const int j_out = t_out - t_first;               // first streamed token that is written
    const int nchunks = (ntok + kChunk - 1) / kChunk;
    const long long row0 = static_cast<long long>(m) * p.T;
    const uint32_t xbytes = C * gc::kVals * 4u;      // one 16-value total from each CTA

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

    const uint16_t* srcH = p.H + (row0 + t_first) * d + col0;
    const uint16_t* srcK = p.k + (row0 + t_first) * d + col0;
    const uint16_t* srcV = p.v + (row0 + t_first) * d + col0;
    // the tokens of chunk c (those of the stream) into chunk slot c % 4, all
    // completing on that slot's barrier
    auto issue = [&](int c) {
        const int slot = c & (kSlots - 1);
        const int j0 = c * kChunk;
        const int n = min(kChunk, ntok - j0);
        uint64_t* bar = &full[slot];
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n) * 3u * row_bytes);
        for (int w = 0; w < n; ++w) {
            const long long off = static_cast<long long>(j0 + w) * d;
            unsigned char* b = ring + (slot * kChunk + w) * kStageBytes;
            bulk_g2s(b, srcH + off, row_bytes, bar);
            bulk_g2s(b + kPitch, srcK + off, row_bytes, bar);
            bulk_g2s(b + 2 * kPitch, srcV + off, row_bytes, bar);
        }
    };

    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&full[s], 1);
            released[s] = 0u;
        }
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        arrived[0] = arrived[1] = 0u;
        fence_mbar_init();
        // arm the exchange of chunks 0 and 1 (peers' bytes may land before or after)
        mbar_arrive_expect_tx(&xbar[0], xbytes);
        if (nchunks > 1) mbar_arrive_expect_tx(&xbar[1], xbytes);
        for (int c = 0; c < kSlots && c < nchunks; ++c) issue(c);
    }
    // the tails of the row slots past this slice's columns, which no copy
    // writes, are zero (threads without columns read them)
    if (row_bytes < kPitch) {
        const int words = (kPitch - static_cast<int>(row_bytes)) / 4;
        for (int i = tid; i < kStages * kRows * words; i += blockDim.x) {
            const int slot = i / words;
            reinterpret_cast<uint32_t*>(ring + slot * kPitch + row_bytes)[i - slot * words] = 0u;
        }
    }
    // every CTA's barriers exist (and the tails are zero) before any peer
    // stores into its slots
    cluster_sync();

    float2 U[kChunk][2];  // u of the last four tokens, slot t % 4 (zero before the row start)
#pragma unroll
    for (int w = 0; w < kChunk; ++w) U[w][0] = U[w][1] = make_float2(0.f, 0.f);

    const float inv_d = 1.0f / static_cast<float>(d);
    bool failed = false;
    const unsigned char* bthread = ring + 8 * tid;
    uint16_t* outY = p.Y + (row0 + t_first) * d + c0;
    uint16_t* outV = p.vhat + (row0 + t_first) * d + c0;

    // One iteration per chunk c = 0 .. nchunks: A(c) forms the chunk's partial
    // sums, B(c - 1) turns the previous chunk's cluster totals into its
    // scalars and writes its outputs.  All waits of an iteration come first,
    // then one straight-line block with both halves (the scheduler overlaps
    // their latency chains), then the hand-in of chunk c and the release of
    // chunk c - 1's stages.  The first iteration has no B, the last no A.
    auto iteration = [&](auto has_a, auto has_b, int c) {
        constexpr bool kA = decltype(has_a)::value;
        constexpr bool kB = decltype(has_b)::value;
        const int buf = c & 1;
        const int ja = c * kChunk;             // first token of chunk c
        const int jb = ja - kChunk;            // first token of chunk c - 1
        const int sta = ja & (kStages - 1);
        const int stb = jb & (kStages - 1);
        if (kA) {
            if (!failed && !mbar_wait(&full[c & (kSlots - 1)], static_cast<uint32_t>((c / kSlots) & 1)))
                failed = true;
        }
        if (kB) {
            // every warp reads chunk c - 1's totals before it hands in chunk c
            if (!failed && !mbar_wait_cluster(&xbar[buf ^ 1], static_cast<uint32_t>(((c - 1) >> 1) & 1)))
                failed = true;
            if (tid == 0 && c + 1 < nchunks) mbar_arrive_expect_tx(&xbar[buf ^ 1], xbytes);
        }
        // ---------------- straight-line block
        float alpha_l = 0.f, ar_l = 0.f;       // scalars of token (lane & 3) of chunk c - 1
        if (kB) {
            const float* tp = tot + (buf ^ 1) * 8 * gc::kVals + (lane & 15);
            float tv = 0.f;
#pragma unroll
            for (int r = 0; r < 8; ++r)
                if (r < static_cast<int>(C)) tv += tp[r * gc::kVals];
            const int tw = 4 * (lane & 3);
            const float sh = __shfl_sync(kFullMask, tv, tw + 0);
            const float sk = __shfl_sync(kFullMask, tv, tw + 1);
            const float shk = __shfl_sync(kFullMask, tv, tw + 2);
            const float sv = __shfl_sync(kFullMask, tv, tw + 3);
            const float rh = rsqrtf(fmaf(sh, inv_d, p.eps));
            const float rk = rsqrtf(fmaf(sk, inv_d, p.eps));
            const float z = rh * rk * shk * p.inv_sqrt_d;
            alpha_l = __fdividef(1.0f, 1.0f + __expf(-z));
            const float rv = rsqrtf(fmaf(alpha_l * alpha_l * sv, inv_d, p.eps));
            ar_l = alpha_l * rv;
            const int j = jb + lane;
            if (rank == 0 && warp == 0 && lane < kChunk && j < ntok && j >= j_out) {
                const long long r = row0 + t_first + j;
                p.alpha[r] = alpha_l;
                p.rh[r] = rh;
                p.rk[r] = rk;
                p.rv[r] = rv;
            }
        }
        float val = 0.f;
        if (kA) {
            // a token past the range reads a stale stage; its sums are never used
            const unsigned char* b0 = bthread + sta * kStageBytes;
            float sums[gc::kVals];
#pragma unroll
            for (int w = 0; w < kChunk; ++w) {
                const unsigned char* b = b0 + w * kStageBytes;
                const uint2 hq = lds64(b), kq = lds64(b + kPitch), vq = lds64(b + 2 * kPitch);
                const float2 h0 = bf2(hq.x), h1 = bf2(hq.y), k0 = bf2(kq.x), k1 = bf2(kq.y);
                const float2 v0 = bf2(vq.x), v1 = bf2(vq.y);
                const float2 hh = fma2(h1, h1, mul2(h0, h0));
                const float2 kk = fma2(k1, k1, mul2(k0, k0));
                const float2 hk = fma2(mul2(h1, k1), wh2[1], mul2(mul2(h0, k0), wh2[0]));
                const float2 vv = fma2(v1, v1, mul2(v0, v0));
                sums[4 * w + 0] = hh.x + hh.y;
                sums[4 * w + 1] = kk.x + kk.y;
                sums[4 * w + 2] = hk.x + hk.y;
                sums[4 * w + 3] = vv.x + vv.y;
            }
            val = gc::warp_reduce16(sums, lane);
        }
        if (kB) {
            const unsigned char* b0 = bthread + stb * kStageBytes + 2 * kPitch;
#pragma unroll
            for (int w = 0; w < kChunk; ++w) {
                const float alpha = __shfl_sync(kFullMask, alpha_l, w);
                const float ar = __shfl_sync(kFullMask, ar_l, w);
                const uint2 vq = lds64(b0 + w * kStageBytes);
                const float2 a2 = splat2(alpha), ar2 = splat2(ar);
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
                    const float2 rden = make_float2(gc::rcp_ftz(1.0f + gc::exp_neg_ftz(cc.x)),
                                                    gc::rcp_ftz(1.0f + gc::exp_neg_ftz(cc.y)));
                    y[i] = fma2(cc, rden, vh[i]);
                    U[w][i] = u;
                }
                const int j = jb + w;
                const bool st_ok = active && j >= j_out && j < ntok;
                const long long off = static_cast<long long>(j) * d;
                stg_cs8_if(outY + off, make_uint2(pack2(y[0]), pack2(y[1])), st_ok);
                stg_cs8_if(outV + off, make_uint2(pack2(vh[0]), pack2(vh[1])), st_ok);
            }
        }
        // ---------------- hand in chunk c: the warp's 16 totals go to shared
        // memory; the last warp of the CTA to do so adds the warps' totals in
        // warp order and sends the CTA's total into slot `rank` of every CTA of
        // the cluster (st.async, completing on that CTA's exchange barrier)
        if (kA) {
            local[(buf * kW + warp) * gc::kVals + (lane >> 1)] = val;
            __syncwarp();
            unsigned int last = 0u;
            if (lane == 0) {
                __threadfence_block();
                if (atomicAdd(&arrived[buf], 1u) == static_cast<unsigned int>(nw - 1)) {
                    arrived[buf] = 0u;
                    __threadfence_block();
                    last = 1u;
                }
            }
            last = __shfl_sync(kFullMask, last, 0);
            if (last) {
                __syncwarp();   // the other warps' totals, seen by lane 0, to every lane
                const float* lp = local + buf * kW * gc::kVals + (lane & 15);
                float cta = 0.f;
                for (int w = 0; w < nw; ++w) cta += lp[w * gc::kVals];
                const uint32_t dst = smem_addr(tot + (buf * 8 + static_cast<int>(rank)) * gc::kVals + (lane & 15));
                const uint32_t bar = smem_addr(xbar + buf);
                for (uint32_t r = static_cast<uint32_t>(lane >> 4); r < C; r += 2)
                    st_async_f32(map_to_rank(dst, r), cta, map_to_rank(bar, r));
            }
        }
        // ---------------- chunk c - 1's stages are done; the last warp refills them
        if (kB) {
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                const int slot = (c - 1) & (kSlots - 1);
                if (atomicAdd(&released[slot], 1u) == static_cast<unsigned int>(nw - 1)) {
                    released[slot] = 0u;
                    fence_proxy_async();
                    if (c - 1 + kSlots < nchunks) issue(c - 1 + kSlots);
                }
            }
        }
    };
    iteration(std::true_type(), std::false_type(), 0);
    for (int c = 1; c < nchunks; ++c) iteration(std::true_type(), std::true_type(), c);
    iteration(std::false_type(), std::true_type(), nchunks);
    if (failed) {
        atomicOr(p.err, kErrTimeout);
        // let copies issued by this CTA land before it leaves (bounded)
        if (tid == 0)
            for (int c = nchunks > kSlots ? nchunks - kSlots : 0; c < nchunks; ++c)
                (void)mbar_wait(&full[c & (kSlots - 1)], static_cast<uint32_t>((c / kSlots) & 1));
    }
    // no CTA leaves while a peer may still store into its slots
    cluster_sync();
}

}  // namespace

int gateconv_fwd_smem(int threads) { return threads > 256 ? FwdShape<16>::kSmem : FwdShape<8>::kSmem; }

cudaError_t gateconv_fwd_prepare(int smem_bytes) {
    if (smem_bytes <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(gateconv_fwd_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gateconv_fwd_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
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
    return threads > 256 ? cudaOccupancyMaxActiveClusters(out, gateconv_fwd_kernel<16>, &cfg)
                         : cudaOccupancyMaxActiveClusters(out, gateconv_fwd_kernel<8>, &cfg);
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
    return c.threads > 256 ? cudaLaunchKernelEx(&cfg, gateconv_fwd_kernel<16>, p)
                           : cudaLaunchKernelEx(&cfg, gateconv_fwd_kernel<8>, p);
}

}  // namespace eg
