// Saved-state gate, backward, in one pass over the rows (cuDNN Frontend
// "Engram saved-state gate", layout, saved-state and workspace paragraphs):
// the same outputs as the coefficient + elementwise kernels of gate_bwd.cu,
// for the packed layout (d = 5120), without reading grad_out twice.
//
// Per token n and stream s (see gate_bwd.cu for the chain rule):
//   dgate = sum_i g_i v_i  ->  ddot  ->  A = ddot rstd_X rstd_key,
//   B = ddot rstd_X^2 dot / d,  Ck = ddot rstd_key^2 dot / d;
//   grad_x = g + A w k - B x,  grad_key = A w x - Ck k,
//   grad_v = (gate_0 g_0 + gate_1 g_1) + (gate_2 g_2 + gate_3 g_3),
//   grad_w += A x k.
// dgate is a sum over the whole row, the outputs need it: a thread-block
// cluster of two CTAs owns a range of consecutive tokens, CTA `rank` the
// column half [2560 rank, 2560 rank + 2560) of all four streams, so the two
// halves of a token's row are in the shared memory of two SMs of one TPC.
//
// Per CTA, 20 column warps (thread i: columns 4i .. 4i+3 of the half, all four
// streams) and four scalar warps.  In iteration t the column warps
//   A  form the partial dgate of each stream of token t + 2 over their columns
//      from the g and v rows in the ring (products exact in fp32, summed
//      without rounding loss as (hi, lo) pairs) and reduce them over the warp;
//      the last warp of the CTA to hand in adds the 20 warp totals in warp
//      order and sends the CTA's four pairs into slot `rank` of both CTAs of
//      the cluster (st.async, completing on that CTA's exchange mbarrier);
//   B  take token t's scalars from its scalar warp and write grad_x, grad_key
//      and grad_v from the x, key and g rows in the ring, accumulating grad_w
//      per thread as a (hi, lo) pair.
// Scalar warp k takes the tokens t = k (mod 4): it waits for a token's two
// halves, adds them in rank order (both CTAs form the same total), evaluates
// the scalars in fp64 (lane s = stream s, as the coefficient kernel does) and
// hands them to the column warps through shared memory.  One token's fp64
// chain on the narrow fp64 pipe takes about as long as a token's column work,
// hence four warps; the two-token lag between A and B covers the exchange and
// that chain.
//
// Rings (1-D bulk copies): g and v rows of 4 tokens, x and key rows of 2; the
// last column warp to finish B(t) refills them with tokens t + 4 and t + 2
// (no x and key rows for a token whose saved gates are all 0).
// The weights of the thread's columns wait in shared memory (each thread
// reads back only what it wrote), which keeps a thread within the 80
// registers that 24 warps (six per scheduler) allow.
// Slot reuse needs no acknowledgements.  A column warp hands in token j in
// iteration j - 2, after its B(j - 3); B(j) waits for the scalars of j, which
// are formed only after j's exchange has completed, i.e. after every column
// warp of both CTAs handed j in.  So when a column warp hands in t + 2 it has
// finished B(t - 2): the exchange of t - 2 is complete and its hand-in slot,
// which t + 2 reuses, has been read (4 hand-in slots).  A scalar warp writes
// the slot of token j only after every column warp's B(j - 3) (4 scalar
// slots, one per scalar warp).  And the peer's column warps, having handed in
// t - 1 (needed for our B(t - 1)), finished B(t - 4) and so B(t - 6): the peer
// has formed the scalars of t - 6 and read its exchange slot, which t + 2
// reuses (8 exchange slots).
// grad_w: cluster q writes the hi word of its (hi, lo) pair to fp32 slot q
// and the lo word, renormalised, as bf16 to row q of a second area (1.5 slots
// a cluster, so that one cluster per TPC fits the workspace); wreduce_kernel
// merges them in ascending q.
#include "common.cuh"
#include "engram_internal.h"

namespace eg {
namespace {

constexpr int kS = 4;
constexpr int kD = kGateHidden;           // 5120
constexpr int kHalf = kD / 2;             // columns per CTA
constexpr int kColWarps = kHalf / 4 / 32; // 20
constexpr int kScalarWarps = 4;           // warp k forms the scalars of tokens t = k (mod 4)
constexpr int kThreads = 32 * (kColWarps + kScalarWarps);
constexpr int kLag = 2;                   // A runs this many tokens ahead of B
constexpr int kRowB = kHalf * 2;          // bytes of a half row (5120)
constexpr int kGvStages = 4, kXkStages = 2;
constexpr int kGvStageB = 5 * kRowB;      // g rows 0-3, v
constexpr int kXkStageB = 8 * kRowB;      // x rows 0-3, key rows 0-3
constexpr int kXslots = 8, kHslots = 4, kSslots = 4, kRslots = 4;
// shared memory
constexpr int kOffGvFull = 0;                               // [4] mbarriers
constexpr int kOffXkFull = 32;                              // [2]
constexpr int kOffXbar = 64;                                // [8] exchange
constexpr int kOffReady = 128;                              // [4] scalars ready
constexpr int kOffRel = 160;                                // [4] release counters
constexpr int kOffArr = 176;                                // [4] hand-in counters
constexpr int kOffSz = 192;                                 // [4] all scalars zero
constexpr int kOffSkip = 208;                               // [4] all four gates zero (x, key rows not copied)
constexpr int kOffLocal = 256;                              // [4][20 warps][4] float2
constexpr int kOffXch = kOffLocal + kHslots * kColWarps * kS * 8;   // [8 slots][2 ranks][4] float2
constexpr int kOffSc = kOffXch + kXslots * 2 * kS * 8;               // [4][4] float4
constexpr int kOffSg = kOffSc + kSslots * kS * 16;                   // [4][4] float gate
constexpr int kOffW = 4096;                                 // [4 streams][2560] fp32 weights
constexpr int kOffGv = kOffW + kS * kHalf * 4;
constexpr int kOffXk = kOffGv + kGvStages * kGvStageB;
constexpr int kSmem = kOffXk + kXkStages * kXkStageB;
static_assert(kOffSg + kSslots * kS * 4 <= kOffW, "header");
static_assert(kSmem <= 232448, "shared memory");
static_assert(kColWarps * 32 * 4 == kHalf, "thread mapping");
static_assert(kGvStages >= kLag + 2 && kXkStages >= 2, "ring depths");
static_assert(kSslots == kScalarWarps && kXslots % kScalarWarps == 0, "a scalar warp owns its slots");

EG_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
EG_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// (hi, lo) pair merged with its partner lane `off` away (symmetric: both
// lanes end with the same pair)
EG_DEV void merge_xor(float& h, float& l, int off) {
    const float h2 = __shfl_xor_sync(kFullMask, h, off);
    const float l2 = __shfl_xor_sync(kFullMask, l, off);
    cacc_merge(h, l, h2, l2);
}

__global__ void __launch_bounds__(kThreads, 1) gate_bwd_fused_kernel(const GateBwdParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* gv_full = reinterpret_cast<uint64_t*>(smem + kOffGvFull);
    uint64_t* xk_full = reinterpret_cast<uint64_t*>(smem + kOffXkFull);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + kOffXbar);
    uint64_t* ready = reinterpret_cast<uint64_t*>(smem + kOffReady);
    unsigned int* rel = reinterpret_cast<unsigned int*>(smem + kOffRel);
    unsigned int* arrived = reinterpret_cast<unsigned int*>(smem + kOffArr);
    unsigned int* sz = reinterpret_cast<unsigned int*>(smem + kOffSz);
    unsigned int* skip = reinterpret_cast<unsigned int*>(smem + kOffSkip);
    float2* local = reinterpret_cast<float2*>(smem + kOffLocal);
    float2* xch = reinterpret_cast<float2*>(smem + kOffXch);
    float4* sc = reinterpret_cast<float4*>(smem + kOffSc);
    float* sg = reinterpret_cast<float*>(smem + kOffSg);
    float* wsm = reinterpret_cast<float*>(smem + kOffW);
    unsigned char* gv_ring = smem + kOffGv;
    unsigned char* xk_ring = smem + kOffXk;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t rank = cluster_rank();
    const long long q = static_cast<long long>(cluster_index());
    const long long G = static_cast<long long>(cluster_count());
    const long long n0 = p.N * q / G, n1 = p.N * (q + 1) / G;
    const int ntok = static_cast<int>(n1 - n0);
    const int col0 = static_cast<int>(rank) * kHalf;
    constexpr uint32_t kXchBytes = 2u * kS * 8u;    // 2 CTAs x 4 pairs

    if (tid == 0) {
        for (int i = 0; i < kGvStages; ++i) mbar_init(&gv_full[i], 1);
        for (int i = 0; i < kXkStages; ++i) mbar_init(&xk_full[i], 1);
        for (int i = 0; i < kXslots; ++i) mbar_init(&xbar[i], 1);
        for (int i = 0; i < kSslots; ++i) mbar_init(&ready[i], 1);
        for (int i = 0; i < 4; ++i) {
            rel[i] = 0u;
            arrived[i] = 0u;
        }
        fence_mbar_init();
        // the first phase of each exchange slot
        for (int i = 0; i < kXslots; ++i) mbar_arrive_expect_tx(&xbar[i], kXchBytes);
    }
    // both CTAs' barriers exist before either sends into the other
    cluster_sync();

    auto issue_gv = [&](int t) {
        const long long n = n0 + t;
        const int b = t % kGvStages;
        unsigned char* dst = gv_ring + b * kGvStageB;
        mbar_arrive_expect_tx(&gv_full[b], static_cast<uint32_t>(kGvStageB));
#pragma unroll
        for (int s = 0; s < kS; ++s)
            bulk_g2s(dst + s * kRowB, p.gout + (n * kS + s) * kD + col0, kRowB, &gv_full[b]);
        bulk_g2s(dst + kS * kRowB, p.v + n * (5LL * kD) + col0, kRowB, &gv_full[b]);
    };
    // x and key rows of token t; none for a token whose four saved gates are
    // 0 (a masked token needs only grad_out: its scalars are all zero)
    auto issue_xk = [&](int t, bool rows) {
        const long long n = n0 + t;
        const int b = t % kXkStages;
        unsigned char* dst = xk_ring + b * kXkStageB;
        if (!rows) {
            mbar_arrive(&xk_full[b]);
            return;
        }
        mbar_arrive_expect_tx(&xk_full[b], static_cast<uint32_t>(kXkStageB));
#pragma unroll
        for (int s = 0; s < kS; ++s) {
            bulk_g2s(dst + s * kRowB, p.x + (n * kS + s) * kD + col0, kRowB, &xk_full[b]);
            bulk_g2s(dst + (kS + s) * kRowB, p.key + n * (5LL * kD) + static_cast<long long>(s) * kD + col0, kRowB,
                     &xk_full[b]);
        }
    };
    // the inputs may have been written by the preceding kernel (the forward)
    grid_dep_wait();
    if (tid == 0) {
        for (int t = 0; t < kGvStages && t < ntok; ++t) issue_gv(t);
        for (int t = 0; t < kXkStages && t < ntok; ++t) issue_xk(t, true);
    }
    grid_dep_launch();
    bool failed = false;

    if (warp >= kColWarps) {
        // ------------------------------------------------ scalar warps
        const int k = warp - kColWarps;
        float4 sv = make_float4(0.f, 0.f, 0.f, 0.f);   // saved record of (token, lane), one token ahead
        if (lane < kS && k < ntok) sv = __ldg(reinterpret_cast<const float4*>(p.saved + ((n0 + k) * kS + lane) * 4));
        // saved gate of (token t + kXkStages, lane): whether that token's x and
        // key rows are copied is published with the scalars of token t, before
        // the refill that copies them (after every column warp's B(t))
        float gnext = 0.f;
        if (lane < kS && k + kXkStages < ntok) gnext = __ldg(p.saved + ((n0 + k + kXkStages) * kS + lane) * 4);
        for (int t = k; t < ntok; t += kScalarWarps) {
            const int xs = t % kXslots, ss = t % kSslots;
            bool zero = true;
            if (!failed && !mbar_wait(&xbar[xs], static_cast<uint32_t>((t / kXslots) & 1))) failed = true;
            if (lane < kS) {
                const float2 a = xch[(xs * 2 + 0) * kS + lane];
                const float2 b = xch[(xs * 2 + 1) * kS + lane];
                float hs = a.x, ls = a.y;
                cacc_merge(hs, ls, b.x, b.y);
                const float gate = sv.x;
                const double dot = sv.y, rx = sv.z, rk = sv.w;
                if (t + kScalarWarps < ntok)
                    sv = __ldg(reinterpret_cast<const float4*>(p.saved + ((n0 + t + kScalarWarps) * kS + lane) * 4));
                const double ad = fabs(dot);
                double ddot = 0.0;
                if (ad >= static_cast<double>(p.clamp) && gate != 0.f) {
                    double y = rsqrtf(static_cast<float>(ad));
                    y = y * (1.5 - 0.5 * ad * y * y);           // 1/sqrt(|dot|)
                    const double sqm = ad * y;                  // sqrt(|dot|)
                    const double ex = exp(-sqm);
                    const double den = 1.0 + ex;
                    double rc = __frcp_rn(static_cast<float>(den));
                    rc = rc * (2.0 - den * rc);                 // 1/(1 + e^-|sq|)
                    const double dsig = ex * rc * rc;           // sigmoid(sq) sigmoid(-sq)
                    const double dgate = static_cast<double>(hs) + static_cast<double>(ls);
                    ddot = dgate * dsig * (0.5 * y);
                }
                const double dd = dot / static_cast<double>(kD);
                const double av = ddot * rx * rk;
                const float a8 = __uint_as_float(__float_as_uint(static_cast<float>(av)) & 0xffff0000u);
                const float arest = static_cast<float>(av - static_cast<double>(a8));
                const float4 c = make_float4(a8, arest, static_cast<float>(-(ddot * rx * rx * dd)),
                                             static_cast<float>(-(ddot * rk * rk * dd)));
                sc[ss * kS + lane] = c;
                sg[ss * kS + lane] = gate;
                zero = c.x == 0.f && c.y == 0.f && c.z == 0.f && c.w == 0.f;
            }
            zero = __all_sync(kFullMask, zero);
            const bool masked = __all_sync(kFullMask, lane >= kS || gnext == 0.f);
            if (lane < kS && t + kXkStages + kScalarWarps < ntok)
                gnext = __ldg(p.saved + ((n0 + t + kXkStages + kScalarWarps) * kS + lane) * 4);
            if (lane == 0) {
                sz[ss] = zero ? 1u : 0u;
                skip[(t + kXkStages) & 3] = masked ? 1u : 0u;
            }
            __syncwarp();
            if (lane == 0) {
                // slot xs is read: arm it for token t + kXslots (whose data may already be arriving)
                if (t + kXslots < ntok) mbar_arrive_expect_tx(&xbar[xs], kXchBytes);
                mbar_arrive(&ready[ss]);
            }
        }
    } else {
        // ------------------------------------------------ column warps
        const int lc = 4 * tid;                     // first of this thread's 4 columns in the half
        const int col = col0 + lc;
#pragma unroll
        for (int s = 0; s < kS; ++s)
            *reinterpret_cast<float4*>(wsm + s * kHalf + lc) = __ldg(reinterpret_cast<const float4*>(p.w + s * kD + col));
        float2 phi[kS][2], plo[kS][2];
#pragma unroll
        for (int s = 0; s < kS; ++s) phi[s][0] = phi[s][1] = plo[s][0] = plo[s][1] = make_float2(0.f, 0.f);

        // A(t): partial dgate of token t over this CTA's columns, handed in
        auto phase_a = [&](int t) {
            const int b = t % kGvStages;
            if (!failed && !mbar_wait(&gv_full[b], static_cast<uint32_t>((t / kGvStages) & 1))) failed = true;
            const unsigned char* st = gv_ring + b * kGvStageB + 8 * tid;
            const uint2 vq = lds64(st + kS * kRowB);
            const float2 v0 = bf2(vq.x), v1 = bf2(vq.y);
            float h[kS], l[kS];
#pragma unroll
            for (int s = 0; s < kS; ++s) {
                const uint2 gq = lds64(st + s * kRowB);
                // g v is exact in fp32 (two 8-bit significands)
                float2 hi = mul2(bf2(gq.x), v0), lo = make_float2(0.f, 0.f);
                cacc_add_x2(hi, lo, mul2(bf2(gq.y), v1));
                h[s] = hi.x;
                l[s] = lo.x;
                cacc_merge(h[s], l[s], hi.y, lo.y);
            }
            // reduce-scatter over the warp: lanes with bit 4 keep streams 2, 3,
            // then bit 3 picks one of the two; lanes 8s hold stream s's total
            const bool b4 = lane & 16, b3 = lane & 8;
            float kh[2], kl[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                kh[k] = b4 ? h[2 + k] : h[k];
                kl[k] = b4 ? l[2 + k] : l[k];
                const float sh = b4 ? h[k] : h[2 + k];
                const float sl = b4 ? l[k] : l[2 + k];
                cacc_merge(kh[k], kl[k], __shfl_xor_sync(kFullMask, sh, 16), __shfl_xor_sync(kFullMask, sl, 16));
            }
            float rh = b3 ? kh[1] : kh[0], rl = b3 ? kl[1] : kl[0];
            {
                const float sh = b3 ? kh[0] : kh[1], sl = b3 ? kl[0] : kl[1];
                cacc_merge(rh, rl, __shfl_xor_sync(kFullMask, sh, 8), __shfl_xor_sync(kFullMask, sl, 8));
            }
            merge_xor(rh, rl, 4);
            merge_xor(rh, rl, 2);
            merge_xor(rh, rl, 1);
            const int hb = t % kHslots;
            if ((lane & 7) == 0) local[(hb * kColWarps + warp) * kS + (lane >> 3)] = make_float2(rh, rl);
            __syncwarp();
            unsigned int last = 0u;
            if (lane == 0) {
                __threadfence_block();
                if (atomicAdd(&arrived[hb], 1u) == static_cast<unsigned int>(kColWarps - 1)) {
                    arrived[hb] = 0u;
                    __threadfence_block();
                    last = 1u;
                }
            }
            last = __shfl_sync(kFullMask, last, 0);
            if (last) {
                __syncwarp();
                if (lane < 2 * kS) {
                    // lane = 4 * target rank + stream
                    const int s = lane & 3;
                    const float2* lp = local + hb * kColWarps * kS + s;
                    float th = lp[0].x, tl = lp[0].y;
                    for (int w = 1; w < kColWarps; ++w) cacc_merge(th, tl, lp[w * kS].x, lp[w * kS].y);
                    const int xs = t % kXslots;
                    const uint32_t dst = smem_addr(xch + (xs * 2 + static_cast<int>(rank)) * kS + s);
                    const uint32_t bar = smem_addr(xbar + xs);
                    const uint32_t r = static_cast<uint32_t>(lane >> 2);
                    st_async_f2(map_to_rank(dst, r), th, tl, map_to_rank(bar, r));
                }
            }
        };

        for (int t = 0; t < kLag && t < ntok; ++t) phase_a(t);
        for (int t = 0; t < ntok; ++t) {
            if (t + kLag < ntok) phase_a(t + kLag);
            // ---- B(t)
            const long long n = n0 + t;
            const int ss = t % kSslots;
            if (!failed && !mbar_wait(&ready[ss], static_cast<uint32_t>((t / kSslots) & 1))) failed = true;
            const int xb = t % kXkStages;
            if (!failed && !mbar_wait(&xk_full[xb], static_cast<uint32_t>((t / kXkStages) & 1))) failed = true;
            // all scalars zero (a masked token): grad_x = grad_out bit for bit,
            // grad_key = 0, no grad_w term
            const bool zt = sz[ss] != 0u;
            const unsigned char* gst = gv_ring + (t % kGvStages) * kGvStageB + 8 * tid;
            const unsigned char* xst = xk_ring + xb * kXkStageB + 8 * tid;
            float2 gsum[2][2];   // gate_s g_s summed in pairs (0 + 1), (2 + 3)
#pragma unroll
            for (int s = 0; s < kS; ++s) {
                const uint2 gq = lds64(gst + s * kRowB);
                const float2 g2[2] = {bf2(gq.x), bf2(gq.y)};
                const float2 G2 = splat2(sg[ss * kS + s]);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float2 tg = mul2(G2, g2[e]);
                    gsum[s >> 1][e] = (s & 1) ? add2(gsum[s >> 1][e], tg) : tg;
                }
                uint2 ox, ok;
                if (zt) {
                    ox = gq;
                    ok = make_uint2(0u, 0u);
                } else {
                    const float4 c4 = sc[ss * kS + s];
                    const float4 wq = *reinterpret_cast<const float4*>(wsm + s * kHalf + lc);
                    const float2 w2[2] = {make_float2(wq.x, wq.y), make_float2(wq.z, wq.w)};
                    const uint2 xq = lds64(xst + s * kRowB);
                    const uint2 kq = lds64(xst + (kS + s) * kRowB);
                    const float2 A82 = splat2(c4.x), Ar2 = splat2(c4.y);
                    const float2 A2 = splat2(__fadd_rn(c4.x, c4.y));
                    const float2 nB2 = splat2(c4.z), nC2 = splat2(c4.w);
                    uint32_t o1[2], o2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float2 x2 = bf2(e == 0 ? xq.x : xq.y), k2 = bf2(e == 0 ? kq.x : kq.y);
                        const float2 aw = mul2(A2, w2[e]);
                        o1[e] = pack2(fma2(aw, k2, fma2(nB2, x2, g2[e])));
                        o2[e] = pack2(fma2(aw, x2, mul2(nC2, k2)));
                        // grad_w += (a8 + arest) x k: a8 x k exact, error-free sum
                        const float2 xk = mul2(x2, k2);
                        float2 sum, err;
                        two_sum2(phi[s][e], mul2(A82, xk), sum, err);
                        phi[s][e] = sum;
                        plo[s][e] = fma2(Ar2, xk, add2(plo[s][e], err));
                    }
                    ox = make_uint2(o1[0], o1[1]);
                    ok = make_uint2(o2[0], o2[1]);
                }
                stg_cs8(p.gx + (n * kS + s) * kD + col, ox);
                stg_cs8(p.gkey + n * (5LL * kD) + static_cast<long long>(s) * kD + col, ok);
            }
            const float2 gv0 = add2(gsum[0][0], gsum[1][0]), gv1 = add2(gsum[0][1], gsum[1][1]);
            // this warp is done with the token's stages; the last one refills them
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                if (atomicAdd(&rel[t % kRslots], 1u) == static_cast<unsigned int>(kColWarps - 1)) {
                    rel[t % kRslots] = 0u;
                    fence_proxy_async();
                    if (t + kGvStages < ntok) issue_gv(t + kGvStages);
                    if (t + kXkStages < ntok) issue_xk(t + kXkStages, skip[(t + kXkStages) & 3] == 0u);
                }
            }
            stg_cs8(p.gv + n * (5LL * kD) + col, make_uint2(pack2(gv0), pack2(gv1)));
        }
        // this cluster's grad_w for the columns, renormalised (hi + lo exactly,
        // |lo| <= half an ulp of hi): hi to fp32 slot q, lo to row q of the bf16
        // low words (relative error of the pair 2^-9 of lo, at most 2^-34 of hi)
        if (ntok > 0) {
#pragma unroll
            for (int s = 0; s < kS; ++s) {
                float2 h[2], l[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) two_sum2(phi[s][e], plo[s][e], h[e], l[e]);
                stg_f4(p.partial + (q * kS + s) * kD + col, h[0].x, h[0].y, h[1].x, h[1].y);
                *reinterpret_cast<uint2*>(p.partial_lo + (q * kS + s) * kD + col) = make_uint2(pack2(l[0]), pack2(l[1]));
            }
        }
    }
    if (failed) atomicOr(p.err, kErrTimeout);
    // every copy issued into this CTA has landed before it leaves (bounded)
    __syncthreads();
    if (tid == 0) {
        for (int t = ntok > kGvStages ? ntok - kGvStages : 0; t < ntok; ++t)
            (void)mbar_wait(&gv_full[t % kGvStages], static_cast<uint32_t>((t / kGvStages) & 1));
        for (int t = ntok > kXkStages ? ntok - kXkStages : 0; t < ntok; ++t)
            (void)mbar_wait(&xk_full[t % kXkStages], static_cast<uint32_t>((t / kXkStages) & 1));
    }
}

}  // namespace

cudaError_t gate_bwd_fused_prepare() {
    cudaError_t e = cudaFuncSetAttribute(gate_bwd_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gate_bwd_fused_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

// Co-resident clusters of two CTAs of the fused kernel (0 if it cannot run).
cudaError_t gate_bwd_fused_max_clusters(int* out) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    *out = 0;
    return cudaOccupancyMaxActiveClusters(out, gate_bwd_fused_kernel, &cfg);
}

int gate_bwd_fused_threads() { return kThreads; }
int gate_bwd_fused_smem() { return kSmem; }

// G clusters of two CTAs; cluster q takes tokens [N q / G, N (q + 1) / G).
cudaError_t gate_bwd_fused_launch(const GateBwdParams& p, int G, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * G), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, gate_bwd_fused_kernel, p);
}

}  // namespace eg
