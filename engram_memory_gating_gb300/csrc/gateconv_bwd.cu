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
// A group of C CTAs per range of consecutive output tokens of one row (one
// CTA per SM, all resident at once); CTA `rank` of a group owns a column
// slice, each thread 4 columns, and the ring of shared-memory stages holds the
// dY, vhat, v, H and k rows of one token per stage.  Stepping through the
// tokens, a thread forms u_tau, c_tau and dc_tau and keeps the last three u
// and dc in registers; du of token t is complete once dc_{t+3} is known.  Per
// chunk of output tokens:
//   1  du and the partial sums S1, S3, S4, S5 over the CTA's columns, handed
//      to the group through exchange records in global memory; du stays in
//      registers;
//   2  (one chunk behind) the group's totals give the per-token coefficients,
//      and the thread writes dv, dH and dk from the rows still in the ring.
// Three tokens before the range (for u) and after it (for dc) are streamed as
// a halo.  Weight gradients accumulate per thread over the range and go to
// the workspace, one slot per range; a second kernel sums the slots in
// ascending order.
#include <type_traits>

#include "common.cuh"
#include "engram.h"
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
//    four output tokens and hand them to the exchange, accumulate dconv_w and
//    drms_w_v, and leave t1 = dY + rrms_v w_v du of every column in shared
//    memory (three chunk slots);
//  * phase-2 warps (warps 8-15) take a chunk's row totals, form its per-token
//    coefficients and write dv = alpha (t1 - Q vhat), dH and dk from t1 and
//    the vhat, H and k rows still in the ring, accumulating drms_w_h.
// Splitting the two phases over different warps halves the state a thread
// holds, so a CTA of sixteen warps fits the register file (phase-1 warps take
// kP1Regs registers a thread, phase-2 warps kP2Regs, by setmaxnreg) where one
// warp doing both phases needed 236.
//
// The exchange, two ways (kGroups).  A CTA's totals of a chunk's 16 row sums
// reach every CTA of its token row, and each adds the C values in rank order,
// so all form the same total.
//  * Clusters: CTA `rank` of a thread-block cluster owns column slice `rank`,
//    one cluster per token range; the last phase-1 warp to hand in stores the
//    CTA's totals into slot `rank` of every CTA's shared memory with
//    `st.async`, completing on that CTA's exchange mbarrier.
//  * Groups: the launch is cooperative (every CTA resident at once, one per
//    SM); CTAs g*C .. g*C + C - 1 form group g and take token ranges g, g + G,
//    g + 2G, ... one after another.  The totals go to the CTA's own exchange
//    record in global memory, slot s mod 2 for the chunk's running index s,
//    each value in one 64-bit word {sequence s + 1, value}; the first phase-2
//    warp of each CTA polls its group's C records until every word carries
//    the sequence it wants and leaves the totals in shared memory for the
//    others.  The host clears the records before the launch, and a word is
//    written and read whole, so a reader never pairs a stale value with a new
//    sequence.  Unlike a cluster the group need not sit in one GPC: at
//    d = 7168 21 groups of 7 CTAs fill 147 SMs where clusters of 8 packed
//    onto 120.
//
// Ordering: phase-1 warps hand in chunk s only after this CTA's phase-2 warps
// have read the totals of chunk s - 1 (barrier `tread`).  Those totals are
// complete only once every CTA of the row has handed in s - 1, which each
// did after its own phase-2 warps had read chunk s - 2; so an exchange slot
// (shared by chunks s and s - 2) has been read by the whole row before it is
// rewritten, and phase 1 never runs more than two chunks ahead, so three t1
// slots suffice.  The ring completes per chunk of four streamed tokens (one
// mbarrier per chunk slot); phase-2 warps release a chunk's stages once they
// have written its outputs (phase-1 warps are done with them by then), and
// phase-1 warps release the halo chunk before the range.  The chunk counts
// (streamed and output) run on across a CTA's ranges, so every mbarrier keeps
// one phase per chunk; between two ranges a barrier over the whole CTA, which
// both warp groups reach once per range, frees the ring, the t1 slots and the
// staged scalars for the next range.
constexpr int kPitch = 2048;
constexpr int kStageBytes = kRows * kPitch;
constexpr int kSlots = kStages / kChunk;         // 4 chunk slots of the ring
constexpr int kT1Slots = 3;
constexpr int kGroupWarps = 8;
constexpr int kWsThreads = 2 * 32 * kGroupWarps;  // 512
constexpr int kP1Regs = 152, kP2Regs = 104;
static_assert(kGroupWarps * 32 * (kP1Regs + kP2Regs) == 65536, "register split of a 512-thread CTA");
constexpr int kMaxGroup = 8;                     // CTAs of a group (d <= 8192, 1024 columns a CTA)
static_assert(kMaxGroup * 1024 >= ENGRAM_GATECONV_MAX_D, "a group must span the widest row");
constexpr int kOffFull = 0;                      // [kSlots] chunk-slot mbarriers
constexpr int kOffXready = 32;                   // [2] a chunk's totals (or the cluster's CTA totals) are in `tot`
constexpr int kOffTread = 48;                    // [2] phase-2 warps have read a chunk's totals
constexpr int kOffTready = 64;                   // [kT1Slots] phase-1 warps have written a chunk's t1
constexpr int kOffRel = 96;                      // [kSlots] release counters
constexpr int kOffArr = 112;                     // [2] hand-in counters
constexpr int kOffLocal = 256;                   // [2][8 warps][16] warp totals
constexpr int kOffTot = kOffLocal + 2 * 8 * gc::kVals * 4;   // [2][16] group totals, or [2][8 ranks][16] CTA totals
constexpr int kRingOff = kOffTot + 2 * kMaxGroup * gc::kVals * 4;
constexpr int kRecWords = gc::kVals;             // 64-bit words of a record slot
constexpr int kT1Off = kRingOff + kStages * kStageBytes;     // [kT1Slots][4 tokens][256 threads] float4
constexpr int kScOff = kT1Off + kT1Slots * kChunk * 256 * 16;   // saved scalars of the streamed tokens
constexpr int kSmem = kScOff + 16 * (kGcBwdMaxRange + 8);
static_assert(kRingOff % 128 == 0 && kT1Off % 16 == 0 && kScOff % 16 == 0, "alignment");
static_assert(kSmem <= 232448, "shared memory");

EG_DEV void reg_alloc_p1() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kP1Regs)); }
EG_DEV void reg_dealloc_p2() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kP2Regs)); }

// Named barrier 1 over all kWsThreads threads of the CTA.  The two warp
// groups reach it from their own branches; bar.sync counts the arriving
// warps, wherever they call it from.
EG_DEV void cta_barrier() { asm volatile("bar.sync 1, %0;" ::"n"(kWsThreads) : "memory"); }

// Exchange words: one 64-bit word {sequence, value} per value, stored and
// loaded whole with relaxed gpu-scope operations (coherent in L2, never
// served from a stale L1 line).  A reader accepts a word only when it carries
// the sequence the reader waits for, so it never takes a value from another
// chunk, and it needs no fence: the word is its own flag.
EG_DEV void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

EG_DEV unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// One value of a chunk's totals: word `rec` of the group's first record slot
// and the same word of the next C - 1 records (kRecWords * 2 words apart).
// group_load issues the C loads at once; group_total polls those that do
// not yet carry sequence `want` and adds the C values in rank order into `tv`.  It gives up after kWaitLimitNs (or
// kWaitMaxIters rounds of polls) and returns false.
EG_DEV void group_load(const unsigned long long* rec, uint32_t C, unsigned long long (&x)[kMaxGroup]) {
#pragma unroll
    for (int r = 0; r < kMaxGroup; ++r) {
        x[r] = 0ull;
        if (r < static_cast<int>(C)) x[r] = ld_relaxed_u64(rec + r * 2 * kRecWords);
    }
}

EG_DEV bool group_total(const unsigned long long* rec, uint32_t C, uint32_t want,
                        unsigned long long (&x)[kMaxGroup], float& tv) {
    uint32_t miss = 0u;
#pragma unroll
    for (int r = 0; r < kMaxGroup; ++r)
        if (r < static_cast<int>(C) && static_cast<uint32_t>(x[r] >> 32) != want) miss |= 1u << r;
    if (miss) {
        const unsigned long long t0 = globaltimer();
        for (uint32_t it = 0; miss && it < kWaitMaxIters; ++it) {
#pragma unroll
            for (int r = 0; r < kMaxGroup; ++r)
                if (miss & (1u << r)) x[r] = ld_relaxed_u64(rec + r * 2 * kRecWords);
#pragma unroll
            for (int r = 0; r < kMaxGroup; ++r)
                if ((miss & (1u << r)) && static_cast<uint32_t>(x[r] >> 32) == want) miss &= ~(1u << r);
            if (!miss) break;
            __nanosleep(32);
            if ((it & 63u) == 63u && globaltimer() - t0 > kWaitLimitNs) break;
        }
    }
    float t = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxGroup; ++r)
        if (r < static_cast<int>(C)) t += __uint_as_float(static_cast<uint32_t>(x[r]));
    tv = t;
    return miss == 0u;
}

// Token range q: output tokens [t_out, t_end) of batch row m, streamed tokens
// [t_first, t_last) around them (a chunk before, three after), and where this
// CTA's slice of the first streamed row starts.  Ranges start at multiples of
// kChunk, and so does the streamed halo, so token t sits in window slot t % 4
// and the streamed chunks hold whole output chunks.
struct RangeGeom {
    int t_out, t_end, t_first, t_last, hc, ntok, nstream, nchunks;
    long long row0, base;
};

EG_DEV RangeGeom range_geom(const GateConvBwdParams& p, int q, int col0) {
    RangeGeom g;
    const int m = q / p.ranges_per_row;
    g.t_out = (q - m * p.ranges_per_row) * p.range_len;
    g.t_end = min(p.T, g.t_out + p.range_len);
    g.t_first = g.t_out >= kChunk ? g.t_out - kChunk : 0;
    g.hc = (g.t_out - g.t_first) / kChunk;   // 1 if a halo chunk precedes the range
    g.t_last = min(p.T, g.t_end + 3);
    g.ntok = g.t_last - g.t_first;
    g.nstream = (g.ntok + kChunk - 1) / kChunk;
    g.nchunks = (g.t_end - g.t_out + kChunk - 1) / kChunk;
    g.row0 = static_cast<long long>(m) * p.T;
    g.base = (g.row0 + g.t_first) * p.d + col0;
    return g;
}

template <bool kGroups>
__global__ void __launch_bounds__(kWsThreads, 1) gateconv_bwd_kernel(const GateConvBwdParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffFull);
    uint64_t* xready = reinterpret_cast<uint64_t*>(smem + kOffXready);
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
    const int gt = tid & 255;                   // thread index within the warp group
    const int gw = warp & (kGroupWarps - 1);    // warp index within the warp group
    // a 1-D cluster of C CTAs is CTAs blockIdx.x / C * C .. + C - 1, rank
    // blockIdx.x % C, as a group is
    const uint32_t C = kGroups ? static_cast<uint32_t>(p.group) : cluster_size();
    const uint32_t rank = blockIdx.x % C;
    const int q0 = static_cast<int>(blockIdx.x / C);     // first range of this CTA's group
    const int qstep = static_cast<int>(gridDim.x / C);   // groups in the launch
    const int d = p.d;
    const int col0 = static_cast<int>(rank) * p.ncols;
    const int cols = min(p.ncols, d - col0);
    const bool active = 4 * gt < cols;
    const int c0 = col0 + 4 * gt;
    const uint32_t row_bytes = 2u * static_cast<uint32_t>(cols);
    const uint32_t xbytes = C * gc::kVals * 4u;     // a chunk's CTA totals from the cluster
    // this CTA's exchange record (two slots of kRecWords words), and word
    // lane & 15 of slot 0 of its group's first record
    unsigned long long* const myrec = p.xrec + static_cast<size_t>(blockIdx.x) * 2 * kRecWords;
    const unsigned long long* const grec =
        p.xrec + static_cast<size_t>(blockIdx.x - rank) * 2 * kRecWords + (lane & 15);

    // streamed chunk k of range R (its tokens 4k .. 4k+3) into ring slot
    // (kb + k) % 4, kb = the streamed chunks of this CTA's earlier ranges
    auto issue = [&](const RangeGeom& R, uint32_t kb, int k) {
        const int slot = static_cast<int>((kb + k) & (kSlots - 1));
        const int j0 = k * kChunk;
        const int n = min(kChunk, R.ntok - j0);
        uint64_t* bar = &full[slot];
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n) * kRows * row_bytes);
        for (int w = 0; w < n; ++w) {
            const long long off = R.base + static_cast<long long>(j0 + w) * d;
            unsigned char* b = ring + (slot * kChunk + w) * kStageBytes;
            bulk_g2s(b, p.dY + off, row_bytes, bar);
            bulk_g2s(b + kPitch, p.vhat + off, row_bytes, bar);
            bulk_g2s(b + 2 * kPitch, p.v + off, row_bytes, bar);
            bulk_g2s(b + 3 * kPitch, p.H + off, row_bytes, bar);
            bulk_g2s(b + 4 * kPitch, p.k + off, row_bytes, bar);
        }
    };
    bool failed = false;
    auto wait_chunk = [&](uint32_t kb, int k) {   // streamed chunk k has landed
        const uint32_t K = kb + static_cast<uint32_t>(k);
        if (!failed && !mbar_wait(&full[K & (kSlots - 1)], (K / kSlots) & 1u)) failed = true;
    };
    // this warp is done with streamed chunk k; the last of the warp group's
    // eight warps to say so refills its slot with chunk k + 4
    auto release = [&](const RangeGeom& R, uint32_t kb, int k) {
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            const int slot = static_cast<int>((kb + k) & (kSlots - 1));
            if (atomicAdd(&released[slot], 1u) == static_cast<unsigned int>(kGroupWarps - 1)) {
                released[slot] = 0u;
                fence_proxy_async();
                if (k + kSlots < R.nstream) issue(R, kb, k + kSlots);
            }
        }
    };
    const unsigned char* bthread = ring + 8 * gt;
    // this thread's 8 bytes of row 0 of streamed token t of range R
    auto row_of = [&](const RangeGeom& R, uint32_t kb, int t) -> const unsigned char* {
        return bthread + ((static_cast<int>(kb) * kChunk + t - R.t_first) & (kStages - 1)) * kStageBytes;
    };
    // the saved per-token scalars of a range's streamed tokens
    auto stage_scalars = [&](const RangeGeom& R) {
        for (int i = tid; i < R.ntok; i += kWsThreads) {
            const long long r = R.row0 + R.t_first + i;
            sc[i] = make_float4(__ldg(p.rv + r), __ldg(p.alpha + r), __ldg(p.rh + r), __ldg(p.rk + r));
        }
    };
    // a range after the first: once the whole CTA is done with the previous
    // one, refill the ring and restage the scalars
    auto next_range = [&](const RangeGeom& R, uint32_t kb) {
        cta_barrier();
        if (tid == 0) {
            fence_proxy_async();
            for (int k = 0; k < kSlots && k < R.nstream; ++k) issue(R, kb, k);
        }
        stage_scalars(R);
        cta_barrier();
    };

    const bool any = q0 < p.nranges;
    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&full[s], 1);
            released[s] = 0u;
        }
        mbar_init(&xready[0], 1);
        mbar_init(&xready[1], 1);
        mbar_init(&tread[0], kGroupWarps);
        mbar_init(&tread[1], kGroupWarps);
        for (int s = 0; s < kT1Slots; ++s) mbar_init(&tready[s], kGroupWarps);
        arrived[0] = arrived[1] = 0u;
        fence_mbar_init();
        if (any) {
            const RangeGeom R0 = range_geom(p, q0, col0);
            if (!kGroups) {
                // one range per cluster: the exchange of its first two chunks
                mbar_arrive_expect_tx(&xready[0], xbytes);
                if (R0.nchunks > 1) mbar_arrive_expect_tx(&xready[1], xbytes);
            }
            for (int k = 0; k < kSlots && k < R0.nstream; ++k) issue(R0, 0u, k);
        }
    }
    if (any) stage_scalars(range_geom(p, q0, col0));
    // the tails of the row slots past this slice's columns, which no copy
    // writes, are zero (threads without columns read them)
    if (row_bytes < kPitch) {
        const int words = (kPitch - static_cast<int>(row_bytes)) / 4;
        for (int i = tid; i < kStages * kRows * words; i += blockDim.x) {
            const int slot = i / words;
            reinterpret_cast<uint32_t*>(ring + slot * kPitch + row_bytes)[i - slot * words] = 0u;
        }
    }
    if (kGroups)
        __syncthreads();
    else
        cluster_sync();   // every CTA's barriers are initialised before a peer's st.async

    const float inv_d = 1.0f / static_cast<float>(d);
    uint32_t kb = 0u, cb = 0u;   // streamed and output chunks of the ranges done
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
        for (int q = q0; q < p.nranges; q += qstep) {
            const RangeGeom R = range_geom(p, q, col0);
            if (q != q0) next_range(R, kb);
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
                if (tau >= R.t_last) {
                    W.D[S][0] = W.D[S][1] = make_float2(0.f, 0.f);
                    return;
                }
                wait_chunk(kb, (tau - R.t_first) / kChunk);
                const float rv = sc[tau - R.t_first].x;
                consume<S>(W, gcw, P, row_of(R, kb, tau), kPitch, rv, true, tau >= R.t_out,
                           active && tau >= R.t_out && tau < R.t_end);
            };
            // fill the windows: the 4 tokens before the range, and dc of its first 3
            step(std::integral_constant<int, 0>(), R.t_out - 4);
            step(std::integral_constant<int, 1>(), R.t_out - 3);
            step(std::integral_constant<int, 2>(), R.t_out - 2);
            step(std::integral_constant<int, 3>(), R.t_out - 1);
            step(std::integral_constant<int, 0>(), R.t_out);
            step(std::integral_constant<int, 1>(), R.t_out + 1);
            step(std::integral_constant<int, 2>(), R.t_out + 2);
            if (R.hc) release(R, kb, 0);   // the halo chunk before the range is not needed again

            for (int c = 0; c < R.nchunks; ++c) {
                const uint32_t s = cb + static_cast<uint32_t>(c);   // running output chunk
                const int tc = R.t_out + c * kChunk;                // its first token
                const int buf = static_cast<int>(s & 1u);
                // the streamed chunk of tokens tc .. tc + 3 (output chunk c; it
                // also holds token tc + 3) and the next one, which holds tokens
                // tc + 4 .. tc + 6, consumed while tc + 1 is in the range and
                // tc + 4 streamed
                wait_chunk(kb, c + R.hc);
                if (tc + 1 < R.t_end && tc + 4 < R.t_last) wait_chunk(kb, c + R.hc + 1);
                float rvt[kChunk], rvc[kChunk];
#pragma unroll
                for (int w = 0; w < kChunk; ++w) {
                    rvt[w] = sc[min(tc + w, R.t_end - 1) - R.t_first].x;
                    rvc[w] = sc[min(tc + w + 3, R.t_last - 1) - R.t_first].x;
                }
                float4* t1w = t1buf + (static_cast<int>(s % kT1Slots) * kChunk) * 256 + gt;
                float sums[gc::kVals];
                // output token t = tc + S: consume t + 3, then du_t, the partial
                // sums, drms_w_v and t1 (tokens past the range select 0)
                auto out1 = [&](auto slot) {
                    constexpr int S = decltype(slot)::value;
                    const int t = tc + S;
                    const bool vt = active && t < R.t_end;
                    consume<(S + 3) & 3>(W, gcw, P, row_of(R, kb, t + 3), kPitch, rvc[S], t + 3 < R.t_last,
                                         true, active && t + 3 < R.t_end);
                    float2 d2[2];
                    conv_t<S>(W, P, d2);
                    const unsigned char* b = row_of(R, kb, t);
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
                if (lane == 0) mbar_arrive(&tready[s % kT1Slots]);
                // hand in chunk s once the phase-2 warps have read chunk s - 1's totals
                if (s >= 1u && lane == 0 && !failed && !mbar_wait(&tread[buf ^ 1], ((s - 1u) >> 1) & 1u))
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
                    if (kGroups) {
                        if (lane < 16)
                            st_relaxed_u64(myrec + buf * kRecWords + lane,
                                           (static_cast<unsigned long long>(s + 1u) << 32) | __float_as_uint(cta));
                    } else {
                        const uint32_t dst = smem_addr(tot + (buf * kMaxGroup + static_cast<int>(rank)) * gc::kVals + (lane & 15));
                        const uint32_t bar = smem_addr(xready + buf);
                        for (uint32_t r = static_cast<uint32_t>(lane >> 4); r < C; r += 2)
                            st_async_f32(map_to_rank(dst, r), cta, map_to_rank(bar, r));
                    }
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
            kb += static_cast<uint32_t>(R.nstream);
            cb += static_cast<uint32_t>(R.nchunks);
        }
    } else {
        reg_dealloc_p2();
        float2 wh2[2], wh[2];
        if (active) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(p.wh + c0));
            wh2[0] = make_float2(a.x * a.x, a.y * a.y);
            wh2[1] = make_float2(a.z * a.z, a.w * a.w);
            wh[0] = make_float2(a.x, a.y);
            wh[1] = make_float2(a.z, a.w);
        } else {
            wh2[0] = wh2[1] = wh[0] = wh[1] = make_float2(0.f, 0.f);
        }
        for (int q = q0; q < p.nranges; q += qstep) {
            const RangeGeom R = range_geom(p, q, col0);
            if (q != q0) next_range(R, kb);
            float2 gwh[2];
            gwh[0] = gwh[1] = make_float2(0.f, 0.f);
            for (int c = 0; c < R.nchunks; ++c) {
                const uint32_t s = cb + static_cast<uint32_t>(c);   // running output chunk
                const int tp = R.t_out + c * kChunk;                // its first token
                const int buf = static_cast<int>(s & 1u);
                float tv = 0.f;
                if (kGroups) {
                    // the first phase-2 warp waits for the group's records of
                    // the chunk, adds their values in rank order and leaves
                    // the totals in `tot`; the others wait for them there
                    if (gw == 0) {
                        if (lane < 16) {
                            unsigned long long x[kMaxGroup];
                            float t = 0.f;
                            group_load(grec + buf * kRecWords, C, x);
                            if (!failed && !group_total(grec + buf * kRecWords, C, s + 1u, x, t)) failed = true;
                            tot[buf * gc::kVals + lane] = t;
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&xready[buf]);
                    } else if (!failed && !mbar_wait(&xready[buf], (s >> 1) & 1u)) {
                        failed = true;
                    }
                    tv = tot[buf * gc::kVals + (lane & 15)];
                } else {
                    // the cluster's CTA totals, added in rank order
                    if (!failed && !mbar_wait_cluster(&xready[buf], (s >> 1) & 1u)) failed = true;
                    if (gt == 0 && c + 2 < R.nchunks) mbar_arrive_expect_tx(&xready[buf], xbytes);
                    const float* tq = tot + buf * kMaxGroup * gc::kVals + (lane & 15);
#pragma unroll
                    for (int r = 0; r < kMaxGroup; ++r)
                        if (r < static_cast<int>(C)) tv += tq[r * gc::kVals];
                }
                // the totals are read: phase-1 warps may hand in chunk s + 1
                __syncwarp();
                if (lane == 0) mbar_arrive(&tread[buf]);
                const int tw = 4 * (lane & 3);
                const float S1 = __shfl_sync(kFullMask, tv, tw + 0);
                const float S3 = __shfl_sync(kFullMask, tv, tw + 1);
                const float S4 = __shfl_sync(kFullMask, tv, tw + 2);
                const float S5 = __shfl_sync(kFullMask, tv, tw + 3);
                const int tt = min(tp + (lane & 3), R.t_end - 1);
                const float4 s4 = sc[tt - R.t_first];
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
                if (!failed && !mbar_wait(&tready[s % kT1Slots], (s / kT1Slots) & 1u)) failed = true;
                wait_chunk(kb, c + R.hc);
                const float4* t1r = t1buf + (static_cast<int>(s % kT1Slots) * kChunk) * 256 + gt;
                auto out2 = [&](auto slot) {
                    constexpr int S = decltype(slot)::value;
                    const int t = tp + S;
                    const float Qv = __shfl_sync(kFullMask, Q_l, S);
                    const float av = __shfl_sync(kFullMask, a_l, S);
                    const float Ahv = __shfl_sync(kFullMask, Ah_l, S);
                    const float Bh = __shfl_sync(kFullMask, Bh_l, S);
                    const float Bk = __shfl_sync(kFullMask, Bk_l, S);
                    const bool vt = active && t < R.t_end;
                    const unsigned char* b = row_of(R, kb, t);
                    const float4 t1 = t1r[S * 256];
                    const uint2 hq = lds64(b + kPitch);
                    const uint2 Hq = lds64(b + 3 * kPitch), kq = lds64(b + 4 * kPitch);
                    const float2 nQ2 = splat2(-Qv), a2 = splat2(av);
                    const float2 Ah2 = splat2(Ahv), nBh2 = splat2(-Bh), nBk2 = splat2(-Bk), Ah22 = splat2(2.0f * Ahv);
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
                    const long long off = (R.row0 + t) * d + c0;
                    stg_cs8_if(p.dH + off, make_uint2(oh[0], oh[1]), vt);
                    stg_cs8_if(p.dk + off, make_uint2(ok[0], ok[1]), vt);
                    stg_cs8_if(p.dv + off, make_uint2(ov[0], ov[1]), vt);
                };
                out2(std::integral_constant<int, 0>());
                out2(std::integral_constant<int, 1>());
                out2(std::integral_constant<int, 2>());
                out2(std::integral_constant<int, 3>());
                release(R, kb, c + R.hc);
            }
            if (active) {
                float* o = p.partial + static_cast<long long>(q) * 6 * d + c0;
                stg_f4(o, gwh[0].x, gwh[0].y, gwh[1].x, gwh[1].y);
            }
            kb += static_cast<uint32_t>(R.nstream);
            cb += static_cast<uint32_t>(R.nchunks);
        }
    }
    if (failed) {
        atomicOr(p.err, kErrTimeout);
        // before the CTA exits, the ring's copies still in flight (the last
        // streamed chunk of each slot) land or time out
        if (tid == 0)
            for (uint32_t K = kb > kSlots ? kb - kSlots : 0u; K < kb; ++K)
                (void)mbar_wait(&full[K & (kSlots - 1)], (K / kSlots) & 1u);
    }
    // no CTA of a cluster leaves while a peer may still store into its
    // shared memory
    if (!kGroups) cluster_sync();
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
    const void* kernels[2] = {reinterpret_cast<const void*>(gateconv_bwd_kernel<false>),
                              reinterpret_cast<const void*>(gateconv_bwd_kernel<true>)};
    for (const void* k : kernels) {
        cudaFuncAttributes attr;
        cudaError_t e = cudaFuncGetAttributes(&attr, k);
        if (e != cudaSuccess) return e;
        if (attr.numRegs * kWsThreads != kGroupWarps * 32 * (kP1Regs + kP2Regs))
            return cudaErrorInvalidConfiguration;
        if (smem_bytes > 0) {
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
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
    return cudaOccupancyMaxActiveClusters(out, gateconv_bwd_kernel<false>, &cfg);
}

cudaError_t gateconv_bwd_blocks_per_sm(int threads, int smem, int* out) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, gateconv_bwd_kernel<true>, threads, smem);
}

// groups == 0: one cluster of c.cluster CTAs per token range (c.clusters
// ranges).  groups > 0: `groups` groups of c.cluster CTAs, launched
// cooperatively; the launch fails (it does not wait) if they cannot all be
// resident at once, which the exchange between a group's CTAs relies on.
cudaError_t gateconv_bwd_launch(const GateConvBwdParams& p, const LaunchCfg& c, int groups, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    if (groups > 0) {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(c.cluster * groups), 1, 1);
    } else {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = c.cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(c.cluster * c.clusters), 1, 1);
    }
    cfg.blockDim = dim3(c.threads, 1, 1);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return groups > 0 ? cudaLaunchKernelEx(&cfg, gateconv_bwd_kernel<true>, p)
                      : cudaLaunchKernelEx(&cfg, gateconv_bwd_kernel<false>, p);
}

cudaError_t gateconv_wreduce_launch(const GateWReduceParams& p, cudaStream_t s) {
    const int threads = 128;
    const int blocks = (p.n + threads - 1) / threads;
    gc_wreduce_kernel<<<blocks, threads, 0, s>>>(p);
    return cudaPeekAtLastError();
}

}  // namespace eg
