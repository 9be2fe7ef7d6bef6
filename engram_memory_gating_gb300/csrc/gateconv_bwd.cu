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
#include <type_traits>

#include "common.cuh"
#include "engram_internal.h"
#include "gateconv_xch.cuh"

namespace eg {
namespace {

using gc::kChunk;
constexpr int kRows = 5;  // dY, vhat, v, H, k
constexpr int kStages = gc::kStages;
static_assert(kStages % kChunk == 0, "a chunk must not wrap around the ring");
static_assert(kStages >= 3 * kChunk + 3, "ring too short for two chunks and the look-ahead");

// Per-thread sliding windows of the conv and its transpose: u and dc of the
// last four tokens, token tau in slot tau % 4 (each float2 = 2 columns).
struct Windows {
    float2 U[4][2];
    float2 D[4][2];
};

struct Weights {
    float2 wv[2], wh2[2], cw[4][2];
};

// Consumes token tau (S = tau % 4) from its stage row pointer `b` (this
// thread's 8 bytes of the dY row): u_tau = vhat rrms_v w_v and, for tokens
// of the range or after it (`dc`), c_tau and dc_tau = dY SiLU'(c_tau); `acc`
// adds the dconv_w contributions dc_tau u_{tau-3+j} of tokens inside the
// range.  A token that does not exist (`real` false: past the row end) gives
// u = dc = 0; values read for it are discarded by selection, never scaled by
// zero, so whatever the stage holds cannot leak in.
template <int S>
EG_DEV void consume(Windows& W, float2 (&gcw)[4][2], const Weights& P, const unsigned char* b,
                    uint32_t pitch, float rv, bool real, bool dc, bool acc) {
    const uint2 vq = lds64(b + pitch);
    const uint2 yq = lds64(b);
    const float2 rv2 = splat2(rv);
    const float2 zero = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        float2 u = mul2(mul2(bf2(i == 0 ? vq.x : vq.y), rv2), P.wv[i]);
        u = real ? u : zero;
        const float2 dy = bf2(i == 0 ? yq.x : yq.y);
        const float2 cc = fma2(P.cw[0][i], W.U[(S + 1) & 3][i],
                               fma2(P.cw[1][i], W.U[(S + 2) & 3][i],
                                    fma2(P.cw[2][i], W.U[(S + 3) & 3][i], mul2(P.cw[3][i], u))));
        const float2 sg = make_float2(gc::rcp_ftz(1.0f + gc::exp_neg_ftz(cc.x)), gc::rcp_ftz(1.0f + gc::exp_neg_ftz(cc.y)));
        // SiLU'(c) = s (1 + c (1 - s))
        const float2 one = splat2(1.0f);
        float2 d = mul2(mul2(dy, sg), fma2(cc, sub2(one, sg), one));
        d = (real && dc) ? d : zero;
        const float2 da = acc ? d : zero;
        gcw[0][i] = fma2(da, W.U[(S + 1) & 3][i], gcw[0][i]);
        gcw[1][i] = fma2(da, W.U[(S + 2) & 3][i], gcw[1][i]);
        gcw[2][i] = fma2(da, W.U[(S + 3) & 3][i], gcw[2][i]);
        gcw[3][i] = fma2(da, u, gcw[3][i]);
        W.D[S][i] = d;
        W.U[S][i] = u;
    }
}

// du_t = sum_j cw_j dc_{t+3-j} for t in slot S (dc_{t+3} already consumed)
template <int S>
EG_DEV void conv_t(const Windows& W, const Weights& P, float2 (&du)[2]) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
        du[i] = fma2(P.cw[3][i], W.D[S][i],
                     fma2(P.cw[2][i], W.D[(S + 1) & 3][i],
                          fma2(P.cw[1][i], W.D[(S + 2) & 3][i], mul2(P.cw[0][i], W.D[(S + 3) & 3][i]))));
}

// Warp-specialised kernel.  A CTA has two groups of eight warps over the same
// column slice, thread i of each group owning columns 4i .. 4i+3:
//  * phase-1 warps (warps 0-7) step through the tokens with the conv windows
//    (u, c, dc, du), form the partial sums S1, S3, S4, S5 of each chunk of
//    four output tokens and hand them to the cluster exchange, accumulate
//    dconv_w and drms_w_v, and leave t1 = dY + rrms_v w_v du of every column in
//    shared memory (three chunk slots);
//  * phase-2 warps (warps 8-15) take a chunk's cluster totals, form its
//    per-token coefficients and write dv = alpha (t1 - Q vhat), dH and dk from
//    t1 and the vhat, H and k rows still in the ring, accumulating drms_w_h.
// Splitting the two phases over different warps halves the state a thread
// holds, so a CTA of sixteen warps fits the register file (phase-1 warps take
// kP1Regs registers a thread, phase-2 warps kP2Regs, by setmaxnreg) where one
// warp doing both phases needed 236.
// Ordering: phase-1 warps hand in chunk c only after this CTA's phase-2 warps
// have read the totals of chunk c - 1 (barrier `tread`), so a peer's exchange
// buffer for chunk c (shared with chunk c - 2) has been read everywhere before
// it is written, and phase 1 never runs more than two chunks ahead, so three
// t1 slots suffice.  The ring completes per chunk of four streamed tokens
// (one mbarrier per chunk slot); phase-2 warps release a chunk's stages once
// they have written its outputs (phase-1 warps are done with them by then),
// and phase-1 warps release the halo chunk before the range.
constexpr int kPitch = 2048;
constexpr int kStageBytes = kRows * kPitch;
constexpr int kSlots = kStages / kChunk;         // 4 chunk slots of the ring
constexpr int kT1Slots = 3;
constexpr int kGroupWarps = 8;
constexpr int kWsThreads = 2 * 32 * kGroupWarps;  // 512
constexpr int kP1Regs = 152, kP2Regs = 104;
static_assert(kGroupWarps * 32 * (kP1Regs + kP2Regs) == 65536, "register split of a 512-thread CTA");
constexpr int kOffFull = 0;                      // [kSlots] chunk-slot mbarriers
constexpr int kOffXbar = 32;                     // [2] cluster-exchange mbarriers
constexpr int kOffTread = 48;                    // [2] phase-2 warps have read a chunk's totals
constexpr int kOffTready = 64;                   // [kT1Slots] phase-1 warps have written a chunk's t1
constexpr int kOffRel = 96;                      // [kSlots] release counters
constexpr int kOffArr = 112;                     // [2] hand-in counters
constexpr int kOffLocal = 256;                   // [2][8 warps][16] warp totals
constexpr int kOffTot = kOffLocal + 2 * 8 * gc::kVals * 4;   // [2][8 ranks][16] CTA totals
constexpr int kRingOff = kOffTot + 2 * 8 * gc::kVals * 4;
constexpr int kT1Off = kRingOff + kStages * kStageBytes;     // [kT1Slots][4 tokens][256 threads] float4
constexpr int kScOff = kT1Off + kT1Slots * kChunk * 256 * 16;   // saved scalars of the streamed tokens
constexpr int kSmem = kScOff + 16 * (kGcBwdMaxRange + 8);
static_assert(kRingOff % 128 == 0 && kT1Off % 16 == 0 && kScOff % 16 == 0, "alignment");
static_assert(kSmem <= 232448, "shared memory");

EG_DEV void reg_alloc_p1() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kP1Regs)); }
EG_DEV void reg_dealloc_p2() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kP2Regs)); }

__global__ void __launch_bounds__(kWsThreads, 1) gateconv_bwd_kernel(const GateConvBwdParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffFull);
    uint64_t* xbar = reinterpret_cast<uint64_t*>(smem + kOffXbar);
    uint64_t* tread = reinterpret_cast<uint64_t*>(smem + kOffTread);
    uint64_t* tready = reinterpret_cast<uint64_t*>(smem + kOffTready);
    unsigned int* released = reinterpret_cast<unsigned int*>(smem + kOffRel);
    unsigned int* arrived = reinterpret_cast<unsigned int*>(smem + kOffArr);
    float* local = reinterpret_cast<float*>(smem + kOffLocal);
    float* tot = reinterpret_cast<float*>(smem + kOffTot);
    unsigned char* ring = smem + kRingOff;
    float4* t1buf = reinterpret_cast<float4*>(smem + kT1Off);
    float4* sc = reinterpret_cast<float4*>(smem + kScOff);  // (rrms_v, alpha, rrms_h, rrms_k)

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const bool phase1 = warp < kGroupWarps;
    const int gt = tid & 255;                   // thread index within the group
    const int gw = warp & (kGroupWarps - 1);    // warp index within the group
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int q = static_cast<int>(cluster_index());
    const int d = p.d;
    const int col0 = static_cast<int>(rank) * p.ncols;
    const int cols = min(p.ncols, d - col0);
    const bool active = 4 * gt < cols;
    const int c0 = col0 + 4 * gt;
    const uint32_t row_bytes = 2u * static_cast<uint32_t>(cols);

    // ranges start at multiples of kChunk, and so does the streamed halo, so
    // token t sits in window slot t % 4 and the streamed chunks hold whole
    // output chunks
    const int m = q / p.ranges_per_row;
    const int t_out = (q - m * p.ranges_per_row) * p.range_len;
    const int t_end = min(p.T, t_out + p.range_len);
    const int t_first = t_out >= kChunk ? t_out - kChunk : 0;
    const int hc = (t_out - t_first) / kChunk;   // 1 if a halo chunk precedes the range
    const int t_last = min(p.T, t_end + 3);
    const int ntok = t_last - t_first;             // streamed tokens (halo included)
    const int nstream = (ntok + kChunk - 1) / kChunk;
    const int nchunks = (t_end - t_out + kChunk - 1) / kChunk;
    const long long row0 = static_cast<long long>(m) * p.T;
    const uint32_t xbytes = C * gc::kVals * 4u;     // one 16-value total from each CTA

    const long long base = (row0 + t_first) * d + col0;
    // streamed chunk k (tokens 4k .. 4k+3 of the stream) into ring slot k % 4
    auto issue = [&](int k) {
        const int slot = k & (kSlots - 1);
        const int j0 = k * kChunk;
        const int n = min(kChunk, ntok - j0);
        uint64_t* bar = &full[slot];
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n) * kRows * row_bytes);
        for (int w = 0; w < n; ++w) {
            const long long off = base + static_cast<long long>(j0 + w) * d;
            unsigned char* b = ring + (slot * kChunk + w) * kStageBytes;
            bulk_g2s(b, p.dY + off, row_bytes, bar);
            bulk_g2s(b + kPitch, p.vhat + off, row_bytes, bar);
            bulk_g2s(b + 2 * kPitch, p.v + off, row_bytes, bar);
            bulk_g2s(b + 3 * kPitch, p.H + off, row_bytes, bar);
            bulk_g2s(b + 4 * kPitch, p.k + off, row_bytes, bar);
        }
    };
    bool failed = false;
    auto wait_chunk = [&](int k) {   // streamed chunk k has landed
        if (!failed && !mbar_wait(&full[k & (kSlots - 1)], static_cast<uint32_t>((k / kSlots) & 1)))
            failed = true;
    };
    // this warp is done with streamed chunk k; the last of the group's eight
    // warps to say so refills its slot with chunk k + 4
    auto release = [&](int k) {
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const int slot = k & (kSlots - 1);
            if (atomicAdd(&released[slot], 1u) == static_cast<unsigned int>(kGroupWarps - 1)) {
                released[slot] = 0u;
                fence_proxy_async();
                if (k + kSlots < nstream) issue(k + kSlots);
            }
        }
    };
    const unsigned char* bthread = ring + 8 * gt;
    // this thread's 8 bytes of row 0 of streamed token t (t_first <= t < t_last)
    auto row_of = [&](int t) -> const unsigned char* {
        return bthread + ((t - t_first) & (kStages - 1)) * kStageBytes;
    };

    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&full[s], 1);
            released[s] = 0u;
        }
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        mbar_init(&tread[0], kGroupWarps);
        mbar_init(&tread[1], kGroupWarps);
        for (int s = 0; s < kT1Slots; ++s) mbar_init(&tready[s], kGroupWarps);
        arrived[0] = arrived[1] = 0u;
        fence_mbar_init();
        mbar_arrive_expect_tx(&xbar[0], xbytes);
        if (nchunks > 1) mbar_arrive_expect_tx(&xbar[1], xbytes);
        for (int k = 0; k < kSlots && k < nstream; ++k) issue(k);
    }
    // the saved per-token scalars of the streamed tokens, staged once
    for (int i = tid; i < ntok; i += blockDim.x) {
        const long long r = row0 + t_first + i;
        sc[i] = make_float4(__ldg(p.rv + r), __ldg(p.alpha + r), __ldg(p.rh + r), __ldg(p.rk + r));
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
    cluster_sync();

    const float inv_d = 1.0f / static_cast<float>(d);
    if (phase1) {
        reg_alloc_p1();
        Weights P;
        if (active) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(p.wh + c0));
            const float4 b = __ldg(reinterpret_cast<const float4*>(p.wv + c0));
            P.wh2[0] = make_float2(a.x * a.x, a.y * a.y);
            P.wh2[1] = make_float2(a.z * a.z, a.w * a.w);
            P.wv[0] = make_float2(b.x, b.y);
            P.wv[1] = make_float2(b.z, b.w);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 c = __ldg(reinterpret_cast<const float4*>(p.cw + static_cast<long long>(j) * d + c0));
                P.cw[j][0] = make_float2(c.x, c.y);
                P.cw[j][1] = make_float2(c.z, c.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                P.wh2[i] = P.wv[i] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < 4; ++j) P.cw[j][i] = make_float2(0.f, 0.f);
            }
        }
        Windows W;
        float2 gcw[4][2], gwv[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int s = 0; s < 4; ++s) W.U[s][i] = W.D[s][i] = gcw[s][i] = make_float2(0.f, 0.f);
            gwv[i] = make_float2(0.f, 0.f);
        }
        // Steps to token tau in slot S: real tokens are consumed (the halo
        // before the range for u only), tokens past the row end give dc = 0.
        auto step = [&](auto slot, int tau) {
            constexpr int S = decltype(slot)::value;
            if (tau < 0) return;
            if (tau >= t_last) {
                W.D[S][0] = W.D[S][1] = make_float2(0.f, 0.f);
                return;
            }
            wait_chunk((tau - t_first) / kChunk);
            const float rv = sc[tau - t_first].x;
            consume<S>(W, gcw, P, row_of(tau), kPitch, rv, true, tau >= t_out, active && tau >= t_out && tau < t_end);
        };
        // fill the windows: the 4 tokens before the range, and dc of its first 3
        step(std::integral_constant<int, 0>(), t_out - 4);
        step(std::integral_constant<int, 1>(), t_out - 3);
        step(std::integral_constant<int, 2>(), t_out - 2);
        step(std::integral_constant<int, 3>(), t_out - 1);
        step(std::integral_constant<int, 0>(), t_out);
        step(std::integral_constant<int, 1>(), t_out + 1);
        step(std::integral_constant<int, 2>(), t_out + 2);
        if (hc) release(0);   // the halo chunk before the range is not needed again

        for (int c = 0; c < nchunks; ++c) {
            const int tc = t_out + c * kChunk;      // first token of output chunk c
            const int buf = c & 1;
            // the streamed chunk of tokens tc .. tc + 3 (output chunk c; it also
            // holds token tc + 3) and the next one, which holds tokens tc + 4 ..
            // tc + 6, consumed while tc + 1 is in the range and tc + 4 streamed
            wait_chunk(c + hc);
            if (tc + 1 < t_end && tc + 4 < t_last) wait_chunk(c + hc + 1);
            float rvt[kChunk], rvc[kChunk];
#pragma unroll
            for (int w = 0; w < kChunk; ++w) {
                rvt[w] = sc[min(tc + w, t_end - 1) - t_first].x;
                rvc[w] = sc[min(tc + w + 3, t_last - 1) - t_first].x;
            }
            float4* t1w = t1buf + ((c % kT1Slots) * kChunk) * 256 + gt;
            float sums[gc::kVals];
            // output token t = tc + S: consume t + 3, then du_t, the partial
            // sums, drms_w_v and t1 (tokens past the range select 0)
            auto out1 = [&](auto slot) {
                constexpr int S = decltype(slot)::value;
                const int t = tc + S;
                const bool vt = active && t < t_end;
                consume<(S + 3) & 3>(W, gcw, P, row_of(t + 3), kPitch, rvc[S], t + 3 < t_last, true,
                                     active && t + 3 < t_end);
                float2 d2[2];
                conv_t<S>(W, P, d2);
                const unsigned char* b = row_of(t);
                const uint2 yq = lds64(b), hq = lds64(b + kPitch), vq = lds64(b + 2 * kPitch);
                const uint2 Hq = lds64(b + 3 * kPitch), kq = lds64(b + 4 * kPitch);
                const float2 rv2 = splat2(rvt[S]);
                const float2 zero = make_float2(0.f, 0.f);
                float2 s1 = zero, s3 = zero, s4 = zero, s5 = zero, t1[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float2 dy = bf2(i == 0 ? yq.x : yq.y), vh = bf2(i == 0 ? hq.x : hq.y);
                    const float2 vv = bf2(i == 0 ? vq.x : vq.y);
                    const float2 h = bf2(i == 0 ? Hq.x : Hq.y), kk = bf2(i == 0 ? kq.x : kq.y);
                    const float2 wdu = mul2(P.wv[i], d2[i]);
                    t1[i] = fma2(rv2, wdu, dy);             // dY + rrms_v w_v du
                    s1 = fma2(t1[i], vv, s1);
                    s3 = fma2(vh, vv, s3);
                    s4 = fma2(wdu, vh, s4);
                    s5 = fma2(mul2(h, kk), P.wh2[i], s5);
                    const float2 g = mul2(d2[i], mul2(vh, rv2));
                    gwv[i] = add2(gwv[i], vt ? g : zero);
                }
                t1w[S * 256] = make_float4(t1[0].x, t1[0].y, t1[1].x, t1[1].y);
                sums[4 * S + 0] = s1.x + s1.y;
                sums[4 * S + 1] = s3.x + s3.y;
                sums[4 * S + 2] = s4.x + s4.y;
                sums[4 * S + 3] = s5.x + s5.y;
            };
            out1(std::integral_constant<int, 0>());
            out1(std::integral_constant<int, 1>());
            out1(std::integral_constant<int, 2>());
            out1(std::integral_constant<int, 3>());
            const float val = gc::warp_reduce16(sums, lane);
            // this chunk's t1 is in shared memory (for the phase-2 warps)
            __syncwarp();
            if (lane == 0) mbar_arrive(&tready[c % kT1Slots]);
            // hand in chunk c once the phase-2 warps have read chunk c - 1's totals
            if (c >= 1 && lane == 0 && !failed &&
                !mbar_wait(&tread[buf ^ 1], static_cast<uint32_t>(((c - 1) >> 1) & 1)))
                failed = true;
            __syncwarp();
            local[(buf * 8 + gw) * gc::kVals + (lane >> 1)] = val;
            __syncwarp();
            unsigned int last = 0u;
            if (lane == 0) {
                __threadfence_block();
                if (atomicAdd(&arrived[buf], 1u) == static_cast<unsigned int>(kGroupWarps - 1)) {
                    arrived[buf] = 0u;
                    __threadfence_block();
                    last = 1u;
                }
            }
            last = __shfl_sync(kFullMask, last, 0);
            if (last) {
                __syncwarp();
                const float* lp = local + buf * 8 * gc::kVals + (lane & 15);
                float cta = 0.f;
#pragma unroll
                for (int w = 0; w < kGroupWarps; ++w) cta += lp[w * gc::kVals];
                const uint32_t dst = smem_addr(tot + (buf * 8 + static_cast<int>(rank)) * gc::kVals + (lane & 15));
                const uint32_t bar = smem_addr(xbar + buf);
                for (uint32_t r = static_cast<uint32_t>(lane >> 4); r < C; r += 2)
                    st_async_f32(map_to_rank(dst, r), cta, map_to_rank(bar, r));
            }
        }
        // per-range weight-gradient partial: [dwh | dwv | dcw0..3], each d wide
        if (active) {
            float* o = p.partial + static_cast<long long>(q) * 6 * d + c0;
            stg_f4(o + d, gwv[0].x, gwv[0].y, gwv[1].x, gwv[1].y);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                stg_f4(o + (2 + j) * d, gcw[j][0].x, gcw[j][0].y, gcw[j][1].x, gcw[j][1].y);
        }
    } else {
        reg_dealloc_p2();
        float2 wh2[2], wh[2], gwh[2];
        if (active) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(p.wh + c0));
            wh2[0] = make_float2(a.x * a.x, a.y * a.y);
            wh2[1] = make_float2(a.z * a.z, a.w * a.w);
            wh[0] = make_float2(a.x, a.y);
            wh[1] = make_float2(a.z, a.w);
        } else {
            wh2[0] = wh2[1] = wh[0] = wh[1] = make_float2(0.f, 0.f);
        }
        gwh[0] = gwh[1] = make_float2(0.f, 0.f);
        for (int c = 0; c < nchunks; ++c) {
            const int tp = t_out + c * kChunk;      // first token of output chunk c
            const int buf = c & 1;
            if (!failed && !mbar_wait_cluster(&xbar[buf], static_cast<uint32_t>((c >> 1) & 1))) failed = true;
            if (gt == 0 && c + 2 < nchunks) mbar_arrive_expect_tx(&xbar[buf], xbytes);
            const float* tq = tot + buf * 8 * gc::kVals + (lane & 15);
            float tv = 0.f;
#pragma unroll
            for (int r = 0; r < 8; ++r)
                if (r < static_cast<int>(C)) tv += tq[r * gc::kVals];
            // the totals are read: phase-1 warps may hand in chunk c + 1
            __syncwarp();
            if (lane == 0) mbar_arrive(&tread[buf]);
            const int tw = 4 * (lane & 3);
            const float S1 = __shfl_sync(kFullMask, tv, tw + 0);
            const float S3 = __shfl_sync(kFullMask, tv, tw + 1);
            const float S4 = __shfl_sync(kFullMask, tv, tw + 2);
            const float S5 = __shfl_sync(kFullMask, tv, tw + 3);
            const int tt = min(tp + (lane & 3), t_end - 1);
            const float4 s4 = sc[tt - t_first];
            const float rv = s4.x, a = s4.y, rh = s4.z, rk = s4.w;
            const float mu = rv * S4 * inv_d;
            const float q2 = rv * rv * mu;
            const float dalpha = fmaf(-q2, S3, S1);
            const float dz = dalpha * a * (1.0f - a);
            const float Ah = dz * rh * rk * p.inv_sqrt_d;
            const float e5 = S5 * inv_d;
            const float Q_l = q2, a_l = a, Ah_l = Ah;
            const float Bh_l = Ah * rh * rh * e5, Bk_l = Ah * rk * rk * e5;
            // t1 of the chunk, and its rows in the ring
            if (!failed && !mbar_wait(&tready[c % kT1Slots], static_cast<uint32_t>((c / kT1Slots) & 1))) failed = true;
            wait_chunk(c + hc);
            const float4* t1r = t1buf + ((c % kT1Slots) * kChunk) * 256 + gt;
            auto out2 = [&](auto slot) {
                constexpr int S = decltype(slot)::value;
                const int t = tp + S;
                const float Qv = __shfl_sync(kFullMask, Q_l, S);
                const float av = __shfl_sync(kFullMask, a_l, S);
                const float Ah = __shfl_sync(kFullMask, Ah_l, S);
                const float Bh = __shfl_sync(kFullMask, Bh_l, S);
                const float Bk = __shfl_sync(kFullMask, Bk_l, S);
                const bool vt = active && t < t_end;
                const unsigned char* b = row_of(t);
                const float4 t1 = t1r[S * 256];
                const uint2 hq = lds64(b + kPitch);
                const uint2 Hq = lds64(b + 3 * kPitch), kq = lds64(b + 4 * kPitch);
                const float2 nQ2 = splat2(-Qv), a2 = splat2(av);
                const float2 Ah2 = splat2(Ah), nBh2 = splat2(-Bh), nBk2 = splat2(-Bk), Ah22 = splat2(2.0f * Ah);
                const float2 zero = make_float2(0.f, 0.f);
                uint32_t oh[2], ok[2], ov[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const float2 vh = bf2(i == 0 ? hq.x : hq.y);
                    const float2 h = bf2(i == 0 ? Hq.x : Hq.y), kk = bf2(i == 0 ? kq.x : kq.y);
                    const float2 t12 = i == 0 ? make_float2(t1.x, t1.y) : make_float2(t1.z, t1.w);
                    const float2 dvh = fma2(nQ2, vh, t12);
                    ov[i] = pack2(mul2(a2, dvh));
                    const float2 aw = mul2(Ah2, wh2[i]);
                    oh[i] = pack2(fma2(aw, kk, mul2(nBh2, h)));
                    ok[i] = pack2(fma2(aw, h, mul2(nBk2, kk)));
                    const float2 g = mul2(mul2(Ah22, wh[i]), mul2(h, kk));
                    gwh[i] = add2(gwh[i], vt ? g : zero);
                }
                const long long off = (row0 + t) * d + c0;
                stg_cs8_if(p.dH + off, make_uint2(oh[0], oh[1]), vt);
                stg_cs8_if(p.dk + off, make_uint2(ok[0], ok[1]), vt);
                stg_cs8_if(p.dv + off, make_uint2(ov[0], ov[1]), vt);
            };
            out2(std::integral_constant<int, 0>());
            out2(std::integral_constant<int, 1>());
            out2(std::integral_constant<int, 2>());
            out2(std::integral_constant<int, 3>());
            release(c + hc);
        }
        if (active) {
            float* o = p.partial + static_cast<long long>(q) * 6 * d + c0;
            stg_f4(o, gwh[0].x, gwh[0].y, gwh[1].x, gwh[1].y);
        }
    }
    if (failed) {
        atomicOr(p.err, kErrTimeout);
        if (tid == 0)
            for (int k = nstream > kSlots ? nstream - kSlots : 0; k < nstream; ++k)
                (void)mbar_wait(&full[k & (kSlots - 1)], static_cast<uint32_t>((k / kSlots) & 1));
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

int gateconv_bwd_smem() { return kSmem; }

int gateconv_bwd_threads() { return kWsThreads; }

cudaError_t gateconv_bwd_prepare(int smem_bytes) {
    // The phase-1 warps raise their registers to kP1Regs and the phase-2 warps
    // lower theirs to kP2Regs (setmaxnreg).  That split must add up to what the
    // CTA is launched with, or the raise would wait forever: refuse to run a
    // build whose register count differs.
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, gateconv_bwd_kernel);
    if (e != cudaSuccess) return e;
    if (attr.numRegs * kWsThreads != kGroupWarps * 32 * (kP1Regs + kP2Regs)) return cudaErrorInvalidConfiguration;
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
