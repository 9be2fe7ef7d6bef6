// Saved-state gate, backward (cuDNN Frontend "Engram saved-state gate",
// layout, saved-state and workspace paragraphs; tile-kernels engram gate
// backward test, which reduces per-block grad_w partials with a sum).
//
// With the forward's saved (gate, dot, rstd_X, rstd_key) per (n, s) and
//   dgate = sum_i g_i v_i,   sq = sqrt(max(|dot|, 1e-6)),
//   ddot  = dgate * sigmoid(sq) * sigmoid(-sq) * 0.5/sqrt(|dot|)   (0 if |dot| < 1e-6
//           or the saved gate is 0, i.e. a masked token; sigmoid' is taken from
//           the saved dot because an fp32 gate near 1 has lost the bits of 1 - gate)
//   A = ddot rstd_X rstd_key,  B = ddot rstd_X^2 dot / d,  Ck = ddot rstd_key^2 dot / d:
//   grad_x_i   = g_i + A w_i k_i - B x_i
//   grad_key_i = A w_i x_i - Ck k_i
//   grad_v_i   = (gate_0 g_0 + gate_1 g_1) + (gate_2 g_2 + gate_3 g_3)  (fp32, one rounding)
//   grad_w_i  += A x_i k_i                         (= ddot * xh_i * kh_i)
// These are the chain rule through the RMS norms written with the saved dot
// (sum_i xh_i w_i kh_i): d dot/d x_i = rstd_X (w_i kh_i - xh_i dot/d).
//
// Three kernels, none of which communicates across CTAs:
//  1. coefficients: a pair of warps per token (the packed layout; one warp
//     per token for a runtime hidden size) reads the token's grad_out rows
//     and v (16-byte loads), each warp one column half, and reduces the four
//     dgate sums with error-free accumulation and shuffles; the second warp
//     hands its sums to the first through shared memory.  Once eight tokens'
//     sums are waiting, one full-warp fp64 pass (lane = 4 token + stream)
//     turns them into the per-stream scalars (A split as an 8-significant-bit
//     head plus a float tail, -B, -Ck), written to the workspace's 16 floats
//     per token;
//  2. elementwise: a CTA owns a 512-column slice of every stream over a
//     group of consecutive tokens; the slice rows of X, the keys and grad_out
//     plus the token's scalars and saved record stream through a ring of
//     shared-memory stages (1-D bulk copies); each thread owns 8 columns of
//     one stream, writes grad_x and grad_key there, forms grad_v with two
//     shuffles across the four stream lanes, and accumulates grad_w for its
//     columns over the group as an unevaluated (hi, lo) pair, stored in the
//     workspace's block slots (group g: slots 2g and 2g+1).  The warps never
//     wait for one another: each counts itself out of a stage in shared
//     memory and the last one to leave it issues its refill;
//  3. the pairs are merged in ascending group order (bitwise reproducible);
//     for a fused weight w = wh * we the same pass also writes the product-rule
//     gradients grad_wh = grad_w * we and grad_we = grad_w * wh.
// The per-token scalars are evaluated in fp64 because a relative error of a
// few fp32 ulps in A, summed over thousands of tokens, would exceed the 1e-6
// absolute accuracy asked of grad_w near zero.
#include "common.cuh"
#include "engram_internal.h"

namespace eg {
namespace {

constexpr int kS = 4;
// chunk indices per load group (kernel 1): two for d = 5120, one for the
// runtime-d instantiation, whose two-chunk groups spilled registers
template <int kDFix>
constexpr int kCGOf = kDFix != 0 ? 2 : 1;
constexpr int kRows = 3 * kS;       // X rows, key rows, grad_out rows (kernel 2)

EG_DEV uint4 ldg16_na(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Programmatic dependent launch.  grid_dep_launch: this CTA lets the next
// kernel of the stream (launched with programmatic stream serialisation) be
// scheduled; grid_dep_wait: waits until the preceding kernel has completed
// and its memory operations are visible (a no-op without such a predecessor).
EG_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
EG_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

EG_DEV void warp_sum_pair(float& hi, float& lo) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        cacc_merge(hi, lo, __shfl_xor_sync(kFullMask, hi, off), __shfl_xor_sync(kFullMask, lo, off));
}

// Named barrier of the two warps of pair `pair` (ids 1..4, 64 threads; the
// ids must be immediates).
EG_DEV void pair_sync(int pair) {
    switch (pair) {
        case 0: asm volatile("bar.sync 1, 64;" ::: "memory"); break;
        case 1: asm volatile("bar.sync 2, 64;" ::: "memory"); break;
        case 2: asm volatile("bar.sync 3, 64;" ::: "memory"); break;
        default: asm volatile("bar.sync 4, 64;" ::: "memory"); break;
    }
}

// ---------------------------------------------------------------- kernel 1
// kDFix = 5120: hidden size known at compile time, packed saved records;
// kDFix = 0: any hidden size (a multiple of 8), separate saved arrays.
// With kDFix = 5120 two warps of a CTA share a token: warp 2q + h reduces
// column half h of its grad_out rows and v; the second hands its four (hi, lo)
// sums to the first through shared memory (two slots, by token parity, one
// pair barrier per token), which merges them after its own and evaluates the
// scalars.  The runtime-d instantiation keeps one warp per token and loads
// one chunk index per group (with two it spilled; a warp pair there gained
// nothing further).
template <int kDFix>
__global__ void __launch_bounds__(256, 2) gate_bwd_coef_kernel(const GateBwdParams p) {
    // launched with programmatic stream serialisation: first wait for the
    // preceding kernel (e.g. the forward that wrote the saved state), then let
    // the elementwise kernel be scheduled; it may copy its input rows while
    // this one runs and waits for this grid before it reads the scalars
    grid_dep_wait();
    grid_dep_launch();
    constexpr bool kPair = kDFix != 0;
    __shared__ float2 xfer[4][2][kS];   // [pair][token parity][stream]
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int pair = warp >> 1, half = kPair ? (warp & 1) : 0;
    constexpr int kUnitShift = kPair ? 6 : 5;  // threads per token: 64 or 32
    const long long gpair = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> kUnitShift;
    const long long npairs = (static_cast<long long>(gridDim.x) * blockDim.x) >> kUnitShift;
    const int d = kDFix ? kDFix : p.d;
    const int nch = d >> 3;                                   // 16-byte chunks per row
    // this warp's chunks [ch0, ch0 + nhalf) of each row
    const int nfirst = kDFix ? kDFix / 16 : nch;
    const int ch0 = half ? nfirst : 0;
    const int nhalf = kDFix ? kDFix / 16 : nch;
    constexpr int kCG = kCGOf<kDFix>;
    const int ng = (((nhalf + 31) / 32 + kCG - 1) / kCG + 1) & ~1;  // even number of load groups
    auto has = [&](int m) { return (kDFix != 0 && (kDFix / 16) % 32 == 0) ? (32 * m < kDFix / 16) : lane + 32 * m < nhalf; };
    uint4 v0[kCG], g0[kS][kCG], v1[kCG], g1[kS][kCG];
    auto load_group = [&](long long n, int grp, uint4 (&vb)[kCG], uint4 (&gb)[kS][kCG]) {
        const uint4* vr = reinterpret_cast<const uint4*>(p.v + n * (kDFix ? 5LL * kDFix : p.v_ts)) + ch0 + lane;
        const uint4* gr = reinterpret_cast<const uint4*>(p.gout + n * kS * d) + ch0 + lane;
#pragma unroll
        for (int c = 0; c < kCG; ++c) {
            const int m = grp * kCG + c;
            const bool ok = has(m);
            vb[c] = ok ? ldg16_na(vr + 32 * m) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int s = 0; s < kS; ++s) gb[s][c] = ok ? ldg16_na(gr + s * (d / 8) + 32 * m) : make_uint4(0, 0, 0, 0);
        }
    };
    float2 hi[kS], lo[kS];
    auto accumulate = [&](int grp, const uint4 (&vb)[kCG], const uint4 (&gb)[kS][kCG]) {
#pragma unroll
        for (int c = 0; c < kCG; ++c) {
            if (kDFix != 0 && !has(grp * kCG + c)) continue;   // compile-time empty group
            const float2 v2[4] = {bf2(vb[c].x), bf2(vb[c].y), bf2(vb[c].z), bf2(vb[c].w)};
#pragma unroll
            for (int s = 0; s < kS; ++s) {
                const uint4 gq = gb[s][c];
                // g*v is exact in fp32 (two 8-bit significands)
                cacc_add_x2(hi[s], lo[s], mul2(bf2(gq.x), v2[0]));
                cacc_add_x2(hi[s], lo[s], mul2(bf2(gq.y), v2[1]));
                cacc_add_x2(hi[s], lo[s], mul2(bf2(gq.z), v2[2]));
                cacc_add_x2(hi[s], lo[s], mul2(bf2(gq.w), v2[3]));
            }
        }
    };
    // The (hi, lo) dgate sums of a unit's tokens wait in shared memory until
    // kBatch of them are ready; one full-warp pass then evaluates their
    // scalars in fp64, lane = kS * token + stream.  An fp64 warp instruction
    // occupies the (narrow) fp64 pipe as long with 4 active lanes as with
    // 32, so this takes 8x fewer of them than a pass per token.
    constexpr int kBatch = 32 / kS;
    constexpr int kUnits = kPair ? 4 : 8;
    __shared__ float2 pend[kUnits][kBatch][kS];
    __shared__ long long pend_n[kUnits][kBatch];
    const int unit = kPair ? pair : warp;
    int npend = 0;
    auto flush = [&]() {
        __syncwarp();
        const int t = lane / kS, sl = lane % kS;
        if (t < npend) {
            // rsqrt and the reciprocal start from fp32 estimates refined by one
            // Newton step, exp is the fp64 routine
            const float2 hl = pend[unit][t][sl];
            const long long rs = pend_n[unit][t] * kS + sl;
            float4 sv;
            if (kDFix)
                sv = __ldg(reinterpret_cast<const float4*>(p.saved + rs * 4));
            else
                sv = make_float4(__ldg(p.sv_gate + rs), __ldg(p.sv_dot + rs), __ldg(p.sv_rx + rs), __ldg(p.sv_rk + rs));
            const float gate = sv.x;
            const double dot = sv.y, rx = sv.z, rk = sv.w;
            const double ad = fabs(dot);
            double ddot = 0.0;
            if (ad >= static_cast<double>(p.clamp) && gate != 0.f) {
                double y = rsqrtf(fabsf(sv.y));
                y = y * (1.5 - 0.5 * ad * y * y);           // 1/sqrt(|dot|)
                const double sqm = ad * y;                  // |sq| = sqrt(|dot|)
                const double ex = exp(-sqm);
                const double den = 1.0 + ex;
                double rc = __frcp_rn(static_cast<float>(den));
                rc = rc * (2.0 - den * rc);                 // 1/(1 + e^-|sq|)
                const double dsig = ex * rc * rc;           // sigmoid(sq) sigmoid(-sq)
                const double dgate = static_cast<double>(hl.x) + static_cast<double>(hl.y);
                ddot = dgate * dsig * (0.5 * y);            // d sq/d dot = 0.5/sqrt(|dot|)
            }
            const double dd = dot / static_cast<double>(d);
            const double av = ddot * rx * rk;
            // A = a8 + arest: a8 keeps 8 significant bits, so a8 * (x*k) is exact
            // in fp32 (8 + 16 bits); arest carries the next 24 bits
            const float a8 = __uint_as_float(__float_as_uint(static_cast<float>(av)) & 0xffff0000u);
            const float arest = static_cast<float>(av - static_cast<double>(a8));
            stg_f4(p.coef + rs * 4, a8, arest, static_cast<float>(-(ddot * rx * rx * dd)),
                   static_cast<float>(-(ddot * rk * rk * dd)));
        }
        __syncwarp();
        npend = 0;
    };
    // A masked token (its four saved gates 0) has ddot = 0 whatever dgate is,
    // so its grad_out and v rows are not read (its sums stay 0).  Lane s < 4
    // loads the saved gate of stream s one token ahead of its use.
    auto load_gate = [&](long long n) -> float {
        if (n >= p.N || lane >= kS) return 0.f;
        return kDFix ? __ldg(p.saved + (n * kS + lane) * 4) : __ldg(p.sv_gate + n * kS + lane);
    };
    bool skip = __all_sync(kFullMask, load_gate(gpair) == 0.f);
    if (gpair < p.N && !skip) load_group(gpair, 0, v0, g0);
    float gnext = load_gate(gpair + npairs);
    int par = 0;
    for (long long n = gpair; n < p.N; n += npairs, par ^= 1) {
        const bool has_next = n + npairs < p.N;
        const bool skip_next = __all_sync(kFullMask, gnext == 0.f);   // loaded one token ago
        gnext = load_gate(n + 2 * npairs);                            // in flight during this token
#pragma unroll
        for (int s = 0; s < kS; ++s) hi[s] = lo[s] = make_float2(0.f, 0.f);
        if (!skip) {
#pragma unroll
            for (int grp = 0; grp < ng; grp += 2) {
                // buffer 0 holds group grp; its successor goes to buffer 1, then
                // buffer 0 takes group grp + 2 or the first group of the next
                // token (whose loads then overlap this token's reduction and fp64 work)
                load_group(n, grp + 1, v1, g1);
                accumulate(grp, v0, g0);
                if (grp + 2 < ng)
                    load_group(n, grp + 2, v0, g0);
                else if (has_next && !skip_next)
                    load_group(n + npairs, 0, v0, g0);
                accumulate(grp + 1, v1, g1);
            }
        } else if (has_next && !skip_next) {
            load_group(n + npairs, 0, v0, g0);
        }
        skip = skip_next;
        float h[kS], l[kS];
#pragma unroll
        for (int s = 0; s < kS; ++s) {
            h[s] = hi[s].x;
            l[s] = lo[s].x;
            cacc_merge(h[s], l[s], hi[s].y, lo[s].y);
            warp_sum_pair(h[s], l[s]);
        }
        if (kPair) {
            // the second half's sums to the first warp of the pair
            if (half == 1 && lane < kS)
                xfer[pair][par][lane] = lane == 0 ? make_float2(h[0], l[0]) : lane == 1 ? make_float2(h[1], l[1])
                                      : lane == 2 ? make_float2(h[2], l[2]) : make_float2(h[3], l[3]);
            pair_sync(pair);
            if (half == 1) continue;
        }
        if (lane < kS) {
            float hs = lane == 0 ? h[0] : lane == 1 ? h[1] : lane == 2 ? h[2] : h[3];
            float ls = lane == 0 ? l[0] : lane == 1 ? l[1] : lane == 2 ? l[2] : l[3];
            if (kPair) {
                const float2 other = xfer[pair][par][lane];
                cacc_merge(hs, ls, other.x, other.y);
            }
            pend[unit][npend][lane] = make_float2(hs, ls);
            if (lane == 0) pend_n[unit][npend] = n;
        }
        if (++npend == kBatch) flush();
    }
    if (npend > 0) flush();
}

// ---------------------------------------------------------------- kernel 2
// Shared memory: stage mbarriers and release counters, the table's mbarrier,
// (packed layout) the token group's scalars and zero flags, then the ring.
constexpr int kTableBarOff = 192;
constexpr int kTableOff = 256;
constexpr int kZeroOff = kTableOff + kGateBwdTableTokens * 64;
template <bool kPacked>
constexpr int kRing2Off = kPacked ? kZeroOff + kGateBwdTableTokens : 256;
static_assert(kRing2Off<true> % 128 == 0, "ring alignment");

// Thread mapping: lane = 8 * stream + g, warp w; the thread owns the 8 columns
// col0 + 8 * (8w + g) of one stream.  The four streams of a column group sit
// in one warp, so grad_v (a sum over streams) is two shuffles.
// kPacked: d = 5120, packed KV / grad_kv rows and saved records, all strides
// known at compile time; otherwise runtime d and strides.  kTsplit: token
// mode (packed layout only; the host sets p.token_split to match).
template <bool kPacked, bool kTsplit>
__global__ void __launch_bounds__(256, 3) gate_bwd_main_kernel(const GateBwdParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);                            // [stages]
    unsigned int* released = reinterpret_cast<unsigned int*>(smem + kMaxStages * 8);  // [stages]
    uint64_t* tbar = reinterpret_cast<uint64_t*>(smem + kTableBarOff);
    unsigned char* ring = smem + kRing2Off<kPacked>;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int W = blockDim.x >> 5;
    const int s = lane >> 3;                               // stream
    // Column mode: warp w owns column groups 8w .. 8w+7 and every warp takes
    // every token of the group.  Token mode (p.token_split, a 64-column
    // slice): every warp owns the slice's 8 column groups and the warps split
    // the group's tokens (warp w: tokens w, w + W, ...), so that a short
    // group's tokens are not walked one after another by a single warp.
    constexpr bool tsplit = kTsplit;
    static_assert(kPacked || !kTsplit, "token mode serves the packed layout");
    const int warp = tid >> 5;
    const int cg = (tsplit ? 0 : warp * 8) + (lane & 7);  // column group in the slice
    const int d = kPacked ? kGateHidden : p.d;
    const long long key_ts = kPacked ? 5LL * kGateHidden : p.key_ts;
    const long long gkey_ts = kPacked ? 5LL * kGateHidden : p.gkey_ts;
    const long long gv_ts = kPacked ? 5LL * kGateHidden : p.gv_ts;
    const int col0 = static_cast<int>(blockIdx.x) * p.ncols;
    const int cols = min(p.ncols, d - col0);            // this slice (the last may be shorter)
    const int col = col0 + 8 * cg;
    const bool active = 8 * cg < cols;
    const long long grp = blockIdx.y;
    const uint32_t row_bytes = static_cast<uint32_t>(p.ncols) * 2u;   // stage row pitch
    const uint32_t copy_bytes = static_cast<uint32_t>(cols) * 2u;     // bytes copied per row
    // saved gate of (n, s): packed records (stride 4 floats) or a (N, 4) array
    const int gstride = (kPacked || p.saved != nullptr) ? 4 : 1;
    const uint32_t stage_bytes = kRows * row_bytes + 128u;
    const int stages = p.stages;
    const long long t0 = grp * p.group_tokens;
    const long long t1 = (t0 + p.group_tokens < p.N) ? t0 + p.group_tokens : p.N;
    const long long ntok = t1 > t0 ? t1 - t0 : 0;
    // Packed layout: the group's per-token scalars (16 floats a token), and a
    // flag per token whose scalars are all zero (a masked token: grad_x =
    // grad_out, grad_key = 0, no grad_w term, so its X and key rows are not
    // needed).  The separate-tensor gate has no mask; its stages carry their
    // token's scalars instead.
    float* table = reinterpret_cast<float*>(smem + kTableOff);
    unsigned char* zero_tok = smem + kZeroOff;

    float2 w2[4];
    if (active) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p.w + s * d + col));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p.w + s * d + col + 4));
        w2[0] = make_float2(a.x, a.y);
        w2[1] = make_float2(a.z, a.w);
        w2[2] = make_float2(b.x, b.y);
        w2[3] = make_float2(b.z, b.w);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) w2[e] = make_float2(0.f, 0.f);
    }

    if (tid == 0) {
        for (int st = 0; st < stages; ++st) {
            mbar_init(&full[st], 1);
            released[st] = 0u;
        }
        mbar_init(tbar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    const uint32_t gate_bytes = 16u * static_cast<uint32_t>(gstride);
    const uint32_t scalar_bytes = kPacked ? 0u : 64u;   // per-stage scalars (separate layout)
    // a stage: the token's input rows (grad_out only for a token whose scalars
    // are all zero), then (separate layout) its scalars and its saved gates
    // (the coefficient kernel's output and the state it read, copied only
    // after that grid has completed)
    auto issue_inputs = [&](int j, int st, bool rows_xk) {
        const long long n = t0 + j;
        unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        mbar_arrive_expect_tx(&full[st], (rows_xk ? kRows : kS) * copy_bytes + scalar_bytes + gate_bytes);
#pragma unroll
        for (int r = 0; r < kS; ++r) {
            if (rows_xk) {
                bulk_g2s(b + r * row_bytes, p.x + (n * kS + r) * d + col0, copy_bytes, &full[st]);
                bulk_g2s(b + (kS + r) * row_bytes, p.key + n * key_ts + static_cast<long long>(r) * d + col0,
                         copy_bytes, &full[st]);
            }
            bulk_g2s(b + (2 * kS + r) * row_bytes, p.gout + (n * kS + r) * d + col0, copy_bytes, &full[st]);
        }
    };
    auto issue_gates = [&](int j, int st) {
        const long long n = t0 + j;
        unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        if (!kPacked) bulk_g2s(b + kRows * row_bytes, p.coef + n * kS * 4, 64u, &full[st]);
        const float* gsrc = p.saved != nullptr ? p.saved + n * kS * 4 : p.sv_gate + n * kS;
        bulk_g2s(b + kRows * row_bytes + 64, gsrc, gate_bytes, &full[st]);
    };
    const int pro = ntok < stages ? static_cast<int>(ntok) : stages;
    if (tid == 0)
        for (int j = 0; j < pro; ++j) issue_inputs(j, j, true);
    // the inputs above were written before the coefficient kernel started;
    // the scalars are that kernel's output.  After the wait the merge kernel
    // may be scheduled (as this grid's CTAs leave; it waits for the whole grid
    // before it reads the partials)
    grid_dep_wait();
    grid_dep_launch();
    if (tid == 0) {
        if (kPacked) {
            // the group's scalars in one copy (ntok <= kGateBwdTableTokens)
            const uint32_t tb = static_cast<uint32_t>(ntok) * kS * 16u;
            mbar_arrive_expect_tx(tbar, tb);
            if (tb > 0) bulk_g2s(table, p.coef + t0 * kS * 4, tb, tbar);
        }
        for (int j = 0; j < pro; ++j) issue_gates(j, j);
    }
    bool failed = false;
    if (kPacked) {
        failed = !mbar_wait(tbar, 0u);
        for (int j = tid; j < ntok; j += blockDim.x) {
            const float4* c = reinterpret_cast<const float4*>(table + j * kS * 4);
            bool z = true;
#pragma unroll
            for (int q = 0; q < kS; ++q) {
                const float4 v = c[q];
                z = z && v.x == 0.f && v.y == 0.f && v.z == 0.f && v.w == 0.f;
            }
            zero_tok[j] = z ? 1 : 0;
        }
        __syncthreads();
    }

    float2 phi[4], plo[4];  // grad_w of this thread's columns, hi + lo
#pragma unroll
    for (int e = 0; e < 4; ++e) phi[e] = plo[e] = make_float2(0.f, 0.f);

    // token mode: a stage's tokens (j, j + stages, ...) all go to one warp,
    // as stages is a multiple of W; it refills the stage with its next token.
    // The stage and its phase parity follow j incrementally (no division).
    const int jstep = tsplit ? W : 1;
    int st = tsplit ? warp : 0;
    uint32_t phase = 0;
    for (int j = st; j < ntok; j += jstep) {
        const long long n = t0 + j;
        if (!failed && !mbar_wait(&full[st], phase)) failed = true;
        const unsigned char* b = ring + static_cast<size_t>(st) * stage_bytes;
        const float* cf = kPacked ? table + j * kS * 4 : reinterpret_cast<const float*>(b + kRows * row_bytes);
        const float4 c4 = *reinterpret_cast<const float4*>(cf + 4 * s);   // [s][4]
        const float2 A82 = splat2(c4.x), Ar2 = splat2(c4.y);
        const float2 A2 = splat2(__fadd_rn(c4.x, c4.y));
        const float2 nB2 = splat2(c4.z), nC2 = splat2(c4.w);
        // saved gate of stream s
        const float2 G2 = splat2(reinterpret_cast<const float*>(b + kRows * row_bytes + 64)[gstride * s]);
        const bool zt = kPacked && zero_tok[j] != 0;   // the same for the whole CTA
        float2 gv[4];
        uint32_t ox[4], ok[4];
        if (active && zt) {
            // all scalars zero: grad_x = grad_out bit for bit, grad_key = 0,
            // no grad_w term (X and key were not copied for this token)
            const uint4 gq = lds128(b + (2 * kS + s) * row_bytes + 16 * cg);
            const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ox[e] = gw[e];
                ok[e] = 0u;
                gv[e] = mul2(G2, bf2(gw[e]));
            }
        } else if (active) {
            const uint4 xq = lds128(b + s * row_bytes + 16 * cg);
            const uint4 kq = lds128(b + (kS + s) * row_bytes + 16 * cg);
            const uint4 gq = lds128(b + (2 * kS + s) * row_bytes + 16 * cg);
            const uint32_t xw[4] = {xq.x, xq.y, xq.z, xq.w};
            const uint32_t kw[4] = {kq.x, kq.y, kq.z, kq.w};
            const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x2 = bf2(xw[e]), k2 = bf2(kw[e]), g2 = bf2(gw[e]);
                const float2 aw = mul2(A2, w2[e]);
                ox[e] = pack2(fma2(aw, k2, fma2(nB2, x2, g2)));
                ok[e] = pack2(fma2(aw, x2, mul2(nC2, k2)));
                gv[e] = mul2(G2, g2);
                // grad_w += (a8 + arest) * (x*k): a8*(x*k) exact, error-free sum
                const float2 xk = mul2(x2, k2);
                float2 sum, err;
                two_sum2(phi[e], mul2(A82, xk), sum, err);
                phi[e] = sum;
                plo[e] = fma2(Ar2, xk, add2(plo[e], err));
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) gv[e] = make_float2(0.f, 0.f);
        }
        // this warp is done with the stage; the last warp to finish refills it
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&released[st], 1u) == static_cast<unsigned int>(tsplit ? 0 : W - 1)) {
                released[st] = 0u;
                if (j + stages < ntok) {
                    fence_proxy_async();
                    issue_inputs(j + stages, st, !kPacked || zero_tok[j + stages] == 0);
                    issue_gates(j + stages, st);
                }
            }
        }
        st += jstep;
        if (st >= stages) {
            st -= stages;
            phase ^= 1u;
        }
        // grad_v = (g0 + g1) + (g2 + g3) over the four streams' lanes
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            gv[e] = add2(gv[e], make_float2(__shfl_xor_sync(kFullMask, gv[e].x, 8),
                                            __shfl_xor_sync(kFullMask, gv[e].y, 8)));
            gv[e] = add2(gv[e], make_float2(__shfl_xor_sync(kFullMask, gv[e].x, 16),
                                            __shfl_xor_sync(kFullMask, gv[e].y, 16)));
        }
        if (active) {
            stg_cs(p.gx + (n * kS + s) * d + col, make_uint4(ox[0], ox[1], ox[2], ox[3]));
            stg_cs(p.gkey + n * gkey_ts + static_cast<long long>(s) * d + col,
                   make_uint4(ok[0], ok[1], ok[2], ok[3]));
            if (s == 0)
                stg_cs(p.gv + n * gv_ts + col,
                       make_uint4(pack2(gv[0]), pack2(gv[1]), pack2(gv[2]), pack2(gv[3])));
        }
    }
    // token mode: the warps' pairs for the same columns are merged in warp
    // order (every issued copy has been consumed, so the ring is free)
    if (tsplit) {
        __syncthreads();
        float* mine = reinterpret_cast<float*>(ring) + (warp * 32 + lane) * 16;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            mine[4 * e + 0] = phi[e].x;
            mine[4 * e + 1] = phi[e].y;
            mine[4 * e + 2] = plo[e].x;
            mine[4 * e + 3] = plo[e].y;
        }
        __syncthreads();
        if (warp == 0) {
            for (int w = 1; w < W; ++w) {
                const float* o = reinterpret_cast<const float*>(ring) + (w * 32 + lane) * 16;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    cacc_merge(phi[e].x, plo[e].x, o[4 * e + 0], o[4 * e + 2]);
                    cacc_merge(phi[e].y, plo[e].y, o[4 * e + 1], o[4 * e + 3]);
                }
            }
        }
    }
    // this group's grad_w for the columns: (hi, lo) in slots 2g, 2g+1, or
    // hi + lo in slot 0 when a single group covers a single block
    if (active && ntok > 0 && (!tsplit || warp == 0)) {
        float* o = p.partial + ((p.pair_slots ? 2 * grp : grp) * kS + s) * d + col;
        if (p.pair_slots) {
            float* ol = o + static_cast<long long>(kS) * d;
            stg_f4(o, phi[0].x, phi[0].y, phi[1].x, phi[1].y);
            stg_f4(o + 4, phi[2].x, phi[2].y, phi[3].x, phi[3].y);
            stg_f4(ol, plo[0].x, plo[0].y, plo[1].x, plo[1].y);
            stg_f4(ol + 4, plo[2].x, plo[2].y, plo[3].x, plo[3].y);
        } else {
            float r[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                r[2 * e] = __fadd_rn(phi[e].x, plo[e].x);
                r[2 * e + 1] = __fadd_rn(phi[e].y, plo[e].y);
            }
            stg_f4(o, r[0], r[1], r[2], r[3]);
            stg_f4(o + 4, r[4], r[5], r[6], r[7]);
        }
    }
    if (failed) {
        atomicOr(p.err, kErrTimeout);
        // let the copies this CTA issued land before it leaves (bounded)
        if (tid == 0) {
            if (kPacked) (void)mbar_wait(tbar, 0u);
            for (int t = ntok > stages ? static_cast<int>(ntok) - stages : 0; t < ntok; ++t)
                (void)mbar_wait(&full[t % stages], static_cast<uint32_t>((t / stages) & 1));
        }
    }
}

// ---------------------------------------------------------------- kernel 3
// grad_weight[i] from the group partials with error-free additions, in a fixed
// order (bitwise reproducible): warp g of a CTA merges the g-th eighth of the
// slots for 32 consecutive columns, then warp 0 merges the eight results in
// ascending g.  pairs 1: slot 2b = hi, 2b+1 = lo of group b; pairs 2 (the
// one-pass backward): slot b = hi, row b of lo16 = lo in bf16.
constexpr int kRedGroups = 8;

__global__ void __launch_bounds__(32 * kRedGroups) wreduce_kernel(const GateWReduceParams p) {
    // launched behind the elementwise kernel with programmatic stream
    // serialisation: the partials are complete and visible after this wait;
    // then the next kernel of the stream may be scheduled
    grid_dep_wait();
    grid_dep_launch();
    __shared__ float shi[kRedGroups][32], slo[kRedGroups][32];
    const int lane = threadIdx.x & 31;
    const int g = threadIdx.x >> 5;
    const int i = blockIdx.x * 32 + lane;
    const int nslot = p.pairs == 1 ? p.nblocks / 2 : p.nblocks;
    const int per = (nslot + kRedGroups - 1) / kRedGroups;
    const int b0 = min(nslot, g * per), b1 = min(nslot, b0 + per);
    float hi = 0.f, lo = 0.f;
    if (i < p.n) {
        const float* src = p.partial + i;
        if (p.pairs == 2) {
            // hi in fp32 slots, lo as bf16 (one-pass backward)
            for (int b = b0; b < b1; ++b)
                cacc_merge(hi, lo, __ldg(src + static_cast<size_t>(b) * p.stride),
                           __uint_as_float(static_cast<uint32_t>(__ldg(p.lo16 + static_cast<size_t>(b) * p.n + i)) << 16));
        } else if (p.pairs) {
            int b = b0;
            for (; b + 4 <= b1; b += 4) {
                float h[4], l[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    h[u] = __ldg(src + static_cast<size_t>(2 * (b + u)) * p.stride);
                    l[u] = __ldg(src + static_cast<size_t>(2 * (b + u) + 1) * p.stride);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) cacc_merge(hi, lo, h[u], l[u]);
            }
            for (; b < b1; ++b)
                cacc_merge(hi, lo, __ldg(src + static_cast<size_t>(2 * b) * p.stride),
                           __ldg(src + static_cast<size_t>(2 * b + 1) * p.stride));
        } else {
            for (int b = b0; b < b1; ++b) cacc_add(hi, lo, __ldg(src + static_cast<size_t>(b) * p.stride));
        }
    }
    shi[g][lane] = hi;
    slo[g][lane] = lo;
    __syncthreads();
    if (g == 0 && i < p.n) {
        float h = shi[0][lane], l = slo[0][lane];
#pragma unroll
        for (int k = 1; k < kRedGroups; ++k) cacc_merge(h, l, shi[k][lane], slo[k][lane]);
        const float gw = __fadd_rn(h, l);
        if (p.out != nullptr) p.out[i] = gw;
        if (p.grad_wh != nullptr) {
            // product rule of w = wh * we, in the same pass (one fp32 rounding each)
            p.grad_wh[i] = __fmul_rn(gw, __uint_as_float(static_cast<uint32_t>(p.we[i]) << 16));
            p.grad_we[i] = __fmul_rn(gw, __uint_as_float(static_cast<uint32_t>(p.wh[i]) << 16));
        }
    }
}

}  // namespace

cudaError_t gate_bwd_prepare(int smem_bytes) {
    const void* mains[3] = {reinterpret_cast<const void*>(gate_bwd_main_kernel<true, false>),
                            reinterpret_cast<const void*>(gate_bwd_main_kernel<true, true>),
                            reinterpret_cast<const void*>(gate_bwd_main_kernel<false, false>)};
    cudaError_t e = cudaSuccess;
    for (const void* k : mains) {
        if (smem_bytes > 0)  // 0: only the coefficient kernel is being set up
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(gate_bwd_coef_kernel<kGateHidden>, cudaFuncAttributePreferredSharedMemoryCarveout, 0);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gate_bwd_coef_kernel<0>, cudaFuncAttributePreferredSharedMemoryCarveout, 0);
}

// Co-resident CTAs: of the coefficient kernel (threads = 256) when smem == 0,
// of the elementwise kernel otherwise.
cudaError_t gate_bwd_max_clusters(int, int threads, int smem, int* out) {
    int per_sm = 0, dev = 0, sms = 0;
    cudaError_t e = smem == 0
        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gate_bwd_coef_kernel<kGateHidden>, threads, 0)
        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gate_bwd_main_kernel<true, false>, threads, smem);
    if (e == cudaSuccess) e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    *out = per_sm * sms;
    return e;
}

// kernel 1 then kernel 2 on the stream (kernel 3 is gate_wreduce_launch)
cudaError_t gate_bwd_launch(const GateBwdParams& p, const LaunchCfg& c, cudaStream_t s) {
    // programmatic stream serialisation for both: kernel 1 waits for its
    // predecessor first; kernel 2 may be scheduled while kernel 1 finishes
    // (it waits for kernel 1's grid before reading the scalars)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(c.aux_blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the compile-time specialisations serve the packed layout (d = 5120)
    cudaError_t e = p.packed ? cudaLaunchKernelEx(&cfg, gate_bwd_coef_kernel<kGateHidden>, p)
                             : cudaLaunchKernelEx(&cfg, gate_bwd_coef_kernel<0>, p);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(c.clusters, c.grid_y, 1);
    cfg.blockDim = dim3(c.threads, 1, 1);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (!p.packed) return cudaLaunchKernelEx(&cfg, gate_bwd_main_kernel<false, false>, p);
    return p.token_split ? cudaLaunchKernelEx(&cfg, gate_bwd_main_kernel<true, true>, p)
                         : cudaLaunchKernelEx(&cfg, gate_bwd_main_kernel<true, false>, p);
}

cudaError_t gate_wreduce_launch(const GateWReduceParams& p, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>((p.n + 31) / 32), 1, 1);
    cfg.blockDim = dim3(32 * kRedGroups, 1, 1);
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, wreduce_kernel, p);
}

}  // namespace eg
