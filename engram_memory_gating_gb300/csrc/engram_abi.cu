// C ABI of libengram.so: host-side argument validation, per-device one-time
// set-up and kernel launches.  No allocation, copy or synchronisation happens
// on the execute path (cuDNN Frontend "Engram saved-state gate": plan/execute
// paragraph -- execute does no allocation, conversion, compilation or sync).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "engram.h"
#include "engram_internal.h"

// Sticky device error word (bit 0: an asynchronous copy timed out).  Host code
// passes its device address, obtained with cudaGetSymbolAddress, to kernels.
__device__ unsigned int eg_error_word = 0u;

namespace eg {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kGateD = ENGRAM_GATE_HIDDEN;
constexpr int kGateBwdStages = 4;  // >= 3: a stage is refilled one token after its last use
static_assert(kGateBwdStages <= kMaxStages, "too many stages");
static_assert(kGateBwdStages >= 3, "ring too short");
// GateConv: CTAs of 256 threads, 4 columns each, 16 one-token ring stages
constexpr int kGcThreads = 256;
constexpr int kGcStages = 16;
constexpr int kGcMinRange = 16;    // tokens; bounds the 3-token halo overhead
constexpr int kGcRangeCost = 8;    // per-range set-up, in token-steps, for the range split
constexpr int64_t kGcBwdSlots = 256;  // backward weight-gradient slots (one per range)
// backward exchange records (two 128-byte slots per CTA) for up to
// kGcBwdMaxCtas CTAs, after the weight-gradient slots of the workspace
constexpr int kGcBwdMaxCtas = 1024;
constexpr size_t kGcXrecBytes = static_cast<size_t>(kGcBwdMaxCtas) * 2 * 128;

struct OccKey {
    int op, cluster, threads, smem;
};

// GateConv launch geometry for one (M, T, d).
struct GcGeom {
    LaunchCfg c;
    int ncols;
    int ring_off;
    int sc_off;  // backward: byte offset of the staged per-token scalars
    int range_len;
    int rpr;  // ranges per batch row
    int groups;  // backward: CTA groups launched (each takes ranges in turn)
};

struct GcCacheEntry {
    int64_t M = -1, T = -1, d = -1;
    GcGeom g;
};

struct DeviceState {
    bool init = false;
    bool ok = false;
    unsigned long long ctx = 0;  // unique ID of the context the set-up was done in
    int sm_count = 0;
    int smem_optin = 0;  // largest dynamic shared memory a CTA may opt in to
    unsigned int* err = nullptr;
    static constexpr int kCache = 64;
    OccKey keys[kCache];
    int vals[kCache];
    int n = 0;
    GcCacheEntry gc_last[2];  // forward, backward
    bool decode_ready = false;
    int fused_clusters = -1;  // co-resident clusters of the one-pass backward (-1: not asked yet)
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

int round_up(int a, int b) { return (a + b - 1) / b * b; }

// Occupancy-limited number of co-resident clusters for a kernel shape.
int max_clusters(DeviceState& st, int op, int cluster, int threads, int smem) {
    for (int i = 0; i < st.n; ++i)
        if (st.keys[i].op == op && st.keys[i].cluster == cluster &&
            st.keys[i].threads == threads && st.keys[i].smem == smem)
            return st.vals[i];
    int v = 0;
    cudaError_t e = cudaSuccess;
    // The dynamic shared-memory limit is an attribute of the kernel, shared by
    // every shape launched with it: set it once to the device's opt-in maximum
    // (the occupancy query below uses the shape's own size).
    const int lim = smem > 0 ? st.smem_optin : 0;
    if (smem > st.smem_optin) {
        e = cudaErrorInvalidValue;
    } else {
        switch (op) {
            case 0:
                e = gate_fwd_prepare(lim);
                if (e == cudaSuccess) e = gate_fwd_max_clusters(cluster, threads, smem, &v);
                break;
            case 1:
                e = gate_bwd_prepare(lim);
                if (e == cudaSuccess) e = gate_bwd_max_clusters(cluster, threads, smem, &v);
                break;
            case 2:
                e = gateconv_fwd_prepare(lim);
                if (e == cudaSuccess) e = gateconv_fwd_max_clusters(cluster, threads, smem, &v);
                break;
            case 3:
                e = gateconv_bwd_prepare(lim);
                if (e == cudaSuccess) e = gateconv_bwd_max_clusters(cluster, threads, smem, &v);
                break;
            default:
                // the backward's cooperative launch: groups of `cluster`
                // CTAs that fit the device at once
                e = gateconv_bwd_prepare(lim);
                if (e == cudaSuccess) e = gateconv_bwd_blocks_per_sm(threads, smem, &v);
                v = e == cudaSuccess ? v * st.sm_count / cluster : 0;
                break;
        }
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        v = 0;
    }
    if (st.n < DeviceState::kCache) {
        st.keys[st.n] = OccKey{op, cluster, threads, smem};
        st.vals[st.n] = v;
        ++st.n;
    }
    return v;
}

// Unique ID of the calling thread's current CUDA context (0 if none is
// current or the driver does not offer the query).  A device reset
// (cudaDeviceReset) replaces the primary context, and everything set up in the
// old one -- kernel attributes, device addresses of the library's __device__
// variables -- is void in the new one; comparing IDs tells the two apart (a
// context handle alone may be reused).  The driver functions are looked up
// through the runtime, so the library has no link-time dependence on libcuda.
unsigned long long current_ctx_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        looked_up = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
        (void)cudaGetLastError();
    }
    if (!get_current || !get_id) return 0;
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr || get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Per-device, per-context state (callers hold g_mu).  The context is
// identified by its ID; a call made after the device's context was replaced
// redoes the set-up instead of using the old context's addresses.
struct NoallocScratch {
    unsigned long long ctx = 0;
    void* ptr = nullptr;
};

// Returns the calling thread's current-device state, initialising it once per
// context of the device.
DeviceState* device_state() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return nullptr;
    }
    DeviceState& st = g_dev[dev];
    unsigned long long ctx = current_ctx_id();
    if (ctx == 0) {
        // no context current on this thread yet: make the device's primary
        // context current (cudaSetDevice initialises it) and ask again
        if (cudaSetDevice(dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        ctx = current_ctx_id();
    }
    if (st.init && ctx != st.ctx) st = DeviceState();  // a new context: set up again
    if (!st.init) {
        st.ctx = ctx;
        st.init = true;
        st.ok = false;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err), eg_error_word) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        // the library is built for sm_103a only
        if (!(major == 10 && minor == 3)) return nullptr;
        st.ok = true;
    }
    return st.ok ? &st : nullptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    const void* p;
    size_t n;
};

bool overlaps(const Range& a, const Range& b) {
    if (a.p == nullptr || b.p == nullptr || a.n == 0 || b.n == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.n && b0 < a0 + a.n;
}

// Every output range against every input and every other output range.
bool any_overlap(const Range* outs, int nout, const Range* ins, int nin) {
    for (int i = 0; i < nout; ++i) {
        for (int j = 0; j < nin; ++j)
            if (overlaps(outs[i], ins[j])) return true;
        for (int j = i + 1; j < nout; ++j)
            if (overlaps(outs[i], outs[j])) return true;
    }
    return false;
}

engram_status_t launch_status(cudaError_t e) {
    if (e == cudaSuccess) return ENGRAM_OK;
    (void)cudaGetLastError();
    return ENGRAM_ERR_LAUNCH;
}

// ---------------------------------------------------------------- geometry

// Forward: one warp per (token, stream) row, 8 warps per CTA, as many CTAs
// as fit on the device (persistent), fewer if there are fewer rows.
bool gate_fwd_cfg(DeviceState& st, int64_t N, LaunchCfg& c) {
    c.cluster = 1;
    c.threads = 256;
    c.stages = 0;
    c.smem = 0;
    const int mc = max_clusters(st, 0, 1, c.threads, 0);
    if (mc <= 0) return false;
    // rows per warp with every co-resident CTA busy, then the fewest CTAs that
    // keep that count, so the last round of rows leaves few warps idle
    const int64_t rows = N * 4;
    const int64_t rpw = (rows + 8LL * mc - 1) / (8LL * mc);
    const int64_t need = (rows + 8 * rpw - 1) / (8 * rpw);
    c.clusters = static_cast<int>(need < mc ? need : mc);
    return true;
}

// Backward: kernel 1 (per-token scalars) on a persistent grid of 256-thread
// CTAs; kernel 2 on a grid of (column slices of 512) x (token groups).  With
// `blocks` set, every 64-token block is its own group and writes one
// grad_weight partial (returned to the caller); otherwise a group covers at
// least two 64-token blocks, so its (hi, lo) grad_weight pair fits two of the
// workspace's block slots (a single-block problem uses one slot).
bool gate_bwd_cfg(DeviceState& st, int64_t N, int64_t d, bool blocks, LaunchCfg& c, int& ncols,
                  int& group_tokens) {
    // slices of 64 column groups: 8 warps x (8 groups x 4 streams); a warp
    // covers 64 columns of the four streams, a slice ncols / 64 warps
    ncols = 512;
    int C = static_cast<int>((d + ncols - 1) / ncols);
    c.cluster = 1;
    c.threads = 256;
    c.stages = kGateBwdStages;
    // barriers, (packed layout, blocks == false) the token group's scalars
    // (64 B a token) and zero flags, the ring
    auto smem_of = [&](int nc) {
        return 256 + (blocks ? 0 : kGateBwdTableTokens * (64 + 1)) + c.stages * (12 * nc * 2 + 128);
    };
    c.smem = smem_of(ncols);
    if (max_clusters(st, 1, 1, c.threads, c.smem) <= 0) return false;
    const int mc1 = max_clusters(st, 1, 1, 256, 0);
    if (mc1 <= 0) return false;
    const int64_t nb = (N + 63) / 64;
    if (blocks) {
        group_tokens = 64;
    } else {
        // A whole number of waves of token groups (a wave = the co-resident
        // CTAs / C groups), balanced to within a token.  A group spans at least
        // two 64-token blocks, so its (hi, lo) grad_weight pair fits two of the
        // workspace's block slots.  Many short groups keep the tokens in
        // flight contiguous in memory, which streams faster than a few long
        // ones (N = 65,536: 0.83 against 0.76 of the copy rate).
        const int resident = max_clusters(st, 1, 1, c.threads, c.smem);
        const int64_t wave = resident / C > 0 ? resident / C : 1;
        const int64_t most = nb >= 2 ? nb / 2 : 1;
        int64_t groups = most <= wave ? most : wave * (most / wave);
        // at most kGateBwdTableTokens tokens a group (its scalars are staged in
        // shared memory); ceil(N / 256) groups still fit the slots (<= nb / 2)
        const int64_t least = (N + kGateBwdTableTokens - 1) / kGateBwdTableTokens;
        if (groups < least) groups = least;
        group_tokens = static_cast<int>((N + groups - 1) / groups);
    }
    c.grid_y = static_cast<int>((N + group_tokens - 1) / group_tokens);
    c.token_split = 0;
    static_assert(kMaxStages % 8 == 0, "token mode: a stage's tokens go to one of 8 warps");
    if (!blocks && 10LL * c.grid_y < 8LL * st.sm_count) {
        // up to a few thousand tokens the groups (one per two 64-token blocks
        // of the workspace) are few and each is walked token by token: there
        // the CTAs take 64-column slices and their 8 warps split the group's
        // tokens, with a ring of 16 stages (a multiple of the warps, so each
        // stage has one consumer).  Measured (backward alone): N = 64 93.5 ->
        // 25.0 us, 320 217.7 -> 51.1, 1024 265.8 -> 87.4, 2048 277.3 -> 147.9,
        // 4096 292.5 -> 266.9.  From N = 3840 the one-pass kernel runs.  The
        // separate-tensor layout stays in column mode: its 64-token groups are
        // many already (N = 8192, H = 4096: 363.7 us, token mode 1495.5).
        ncols = 64;
        C = static_cast<int>((d + ncols - 1) / ncols);
        c.threads = 256;
        c.stages = kMaxStages;
        c.smem = smem_of(ncols);
        c.token_split = 1;
        if (max_clusters(st, 1, 1, c.threads, c.smem) <= 0) return false;
    }
    c.clusters = C;
    // coefficient kernel: a warp pair per token (packed, d = 5120) or a warp per
    // token (runtime d, the separate-tensor layout)
    const int64_t need1 = blocks ? (N + 7) / 8 : (N + 3) / 4;
    c.aux_blocks = static_cast<int>(need1 < mc1 ? need1 : mc1);
    return true;
}

// The one-pass gate backward (gate_bwd_fused.cu) runs G clusters of two
// CTAs, one per SM; each writes its grad_weight pair as 4 x 5120 fp32 hi
// words and 4 x 5120 bf16 lo words (122,880 bytes).  With the per-token
// scalars kept on chip the whole workspace is slot space: the hi slots, then
// the lo rows.  G is fixed by N and the device alone (not by the buffer a
// caller passes), and the call keeps the three-kernel backward when G would
// leave too many SMs idle (small N: its workspace is small).  The one-pass
// kernel's time is close to (N / G) x 2.64 us (measured at N = 3072 to 8192
// with G from 32 to 76).  Against the three kernels (token mode): N = 3712
// (G = 40) 238.3 against 236.5 us, 3840 (G = 42) 234.4 against 235.4, 3968
// (G = 43) 235.4 against 246.5, 4096 (G = 44) 241.7 against 249.1; so the one
// pass runs from 42 clusters (N = 3840) on.
constexpr int kFusedMinClusters = 42;
constexpr size_t kFusedSlotBytes = 4 * kGateD * (4 + 2);

int gate_bwd_fused_groups(DeviceState& st, int64_t N) {
    if (st.fused_clusters < 0) {
        int mc = 0;
        if (gate_bwd_fused_prepare() != cudaSuccess || gate_bwd_fused_max_clusters(&mc) != cudaSuccess) mc = 0;
        (void)cudaGetLastError();
        st.fused_clusters = mc;
    }
    const int64_t slots = static_cast<int64_t>(engram_gate_bwd_workspace_size(N) / kFusedSlotBytes);
    const int64_t G = std::min<int64_t>(st.fused_clusters, slots);
    return G >= kFusedMinClusters ? static_cast<int>(G) : 0;
}

bool gc_shape_ok(int64_t M, int64_t T, int64_t d) {
    if (M < 1 || T < 1 || d < 8 || d > ENGRAM_GATECONV_MAX_D || d % 8 != 0) return false;
    return M * T <= 2147483647LL;
}

// Weight-gradient slots of the backward's workspace: one per token range, at
// most max(M, kGcBwdSlots) ranges (fixed by M and T alone, so the workspace
// size does not depend on the device).
int64_t gc_bwd_slots(int64_t M, int64_t T) {
    const int64_t per_row = (T + kGcMinRange - 1) / kGcMinRange;
    int64_t s = M * per_row;
    if (s > kGcBwdSlots) s = kGcBwdSlots;
    const int64_t least = M * ((T + kGcBwdMaxRange - 1) / kGcBwdMaxRange);
    return s > least ? s : least;
}

// Column split over C CTAs per row, each of `threads` (a multiple of 32,
// at most 256) threads owning 4 columns; every slice is a whole number of
// 8-column groups, so every row slice is a multiple of 16 bytes (bulk-copy
// rule).
void gc_split(int64_t d, int rows, int C, GcGeom& g) {
    const int quads = static_cast<int>(d / 4);
    g.c.cluster = C;
    g.c.threads = round_up((quads + C - 1) / C, 32);
    g.ncols = 4 * g.c.threads;
    const int parts = C * (g.c.threads / 32);
    g.ring_off = round_up(256 + 2 * parts * 16 * 4, 128);
    g.c.stages = kGcStages;
    g.c.smem = g.ring_off + kGcStages * rows * g.ncols * 2;
}

// Token ranges: ranges_per_row r minimising (waves of clusters) x (tokens of
// the longest range + halo + set-up), with at most max_ranges ranges.  Range
// lengths are multiples of 4 tokens (the kernels' window slots rely on it).
void gc_ranges(int64_t M, int64_t T, int K, int64_t max_ranges, int64_t max_len, GcGeom& g) {
    const int64_t lo = (T + max_len - 1) / max_len;
    int64_t hi = (T + kGcMinRange - 1) / kGcMinRange;
    if (hi > max_ranges / M) hi = max_ranges / M;
    if (hi > lo + 4096) hi = lo + 4096;
    if (hi < lo) hi = lo;
    int64_t best_len = ((T + lo - 1) / lo + 3) / 4 * 4, best_cost = -1;
    for (int64_t r = lo; r <= hi; ++r) {
        const int64_t len = ((T + r - 1) / r + 3) / 4 * 4;
        const int64_t rr = (T + len - 1) / len;
        const int64_t waves = (M * rr + K - 1) / K;
        const int64_t cost = waves * (len + 4 + kGcRangeCost);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best_len = len;
        }
    }
    g.range_len = static_cast<int>(best_len);
    g.rpr = static_cast<int>((T + best_len - 1) / best_len);
    g.c.clusters = static_cast<int>(M * g.rpr);
}

// op 0: forward (3 rows per stage: H, k, v); op 1: backward (dY, vhat, v, H, k).
const GcGeom* gc_cfg(DeviceState& st, int op, int64_t M, int64_t T, int64_t d) {
    GcCacheEntry& e = st.gc_last[op];
    if (e.M == M && e.T == T && e.d == d) return &e.g;
    // C = ceil(d / 1024): measured on GB300, larger clusters (more, smaller
    // CTAs) did not run faster even where they packed onto more SMs.  The
    // backward also tries C rounded up to a power of two, where every CTA
    // still gets columns, and keeps it if more CTAs are co-resident: at
    // d = 7168 clusters of 7 fill 105 SMs and clusters of 8 fill 120 (1.8%
    // faster); at d = 5120 clusters of 5 fill more than 8 do.
    const int rows = op == 0 ? 3 : 5;
    auto shape = [&](int C, GcGeom& g) {
        g = {};
        gc_split(d, rows, C, g);
        // fixed layouts (2048-byte row slots; the backward's with the staged
        // saved scalars of up to kGcBwdMaxRange + 7 streamed tokens); a
        // backward CTA has two warp groups over its column slice
        g.c.smem = op == 0 ? gateconv_fwd_smem(g.c.threads) : gateconv_bwd_smem();
        if (op == 1) g.c.threads = gateconv_bwd_threads();
    };
    GcGeom g;
    const int C0 = static_cast<int>((d + 1023) / 1024);
    shape(C0, g);
    if (op == 0 && d > 1024) {
        // the forward also has 512-thread CTAs (one per SM, up to 2048
        // columns): half as many CTAs a row, kept when they cover more SMs
        // (d = 4096: clusters of four 256-thread CTAs fill 144 SMs, pairs
        // of 512-thread CTAs all 152)
        const int Cw = static_cast<int>((d + 2047) / 2048);
        GcGeom gw;
        shape(Cw, gw);
        if (gw.c.threads > 256) {
            const int kn = max_clusters(st, 2, g.c.cluster, g.c.threads, g.c.smem);
            const int kw = max_clusters(st, 2, gw.c.cluster, gw.c.threads, gw.c.smem);
            if (2 * kw * Cw > kn * C0) g = gw;
        }
    }
    if (op == 1) {
        const int p2 = C0 <= 1 ? 1 : C0 <= 2 ? 2 : C0 <= 4 ? 4 : 8;
        const int64_t cols = 4 * static_cast<int64_t>(round_up(static_cast<int>((d / 4 + p2 - 1) / p2), 32));
        if (p2 != C0 && cols <= 1024 && (p2 - 1) * cols < d) {
            GcGeom g2;
            shape(p2, g2);
            const int k0 = max_clusters(st, 3, g.c.cluster, g.c.threads, g.c.smem);
            const int k2 = max_clusters(st, 3, g2.c.cluster, g2.c.threads, g2.c.smem);
            if (k2 * p2 > k0 * C0) g = g2;
        }
    }
    int K = max_clusters(st, op == 0 ? 2 : 3, g.c.cluster, g.c.threads, g.c.smem);
    if (op == 1) {
        // Groups of C0 CTAs exchanging through global memory (a cooperative
        // launch) are not confined to a GPC as clusters are, and fill the
        // device where clusters pack poorly.  A CTA's time per token follows
        // its columns, and a group's exchange through L2 costs about 1/16 of
        // that (measured: 2.39 against 2.24 us a chunk of 1024 columns), so
        // the groups are taken when G * 15/16 / ncols beats K / ncols of the
        // clusters: d = 7168, 21 groups of 7 x 1024 columns against 15
        // clusters of 8 x 896 (2.26 -> 1.93 ms at M = 8, T = 8192); d = 4096
        // keeps 36 clusters of 4 (144 SMs) against 38 groups.
        GcGeom gg;
        shape(C0, gg);
        int G = max_clusters(st, 4, C0, gg.c.threads, gg.c.smem);
        if (G * C0 > kGcBwdMaxCtas) G = kGcBwdMaxCtas / C0;
        if (G > 0 && (K <= 0 || 15LL * G * g.ncols > 16LL * K * gg.ncols)) {
            g = gg;
            K = G;
            g.groups = G;
        }
    }
    if (K <= 0) return nullptr;
    if (op == 0) {
        gc_ranges(M, T, K, int64_t(1) << 31, int64_t(1) << 31, g);
    } else {
        gc_ranges(M, T, K, gc_bwd_slots(M, T), kGcBwdMaxRange, g);
        if (g.groups > 0 && g.c.clusters < g.groups) g.groups = g.c.clusters;
    }
    e.M = M;
    e.T = T;
    e.d = d;
    e.g = g;
    return &e.g;
}

// Tensor map of a (rows, cols) row-major bf16 matrix with 32-column x
// 256-row boxes (rows past the end read as zero; the 64-byte rows land in
// shared memory in the 64-byte swizzle), through the driver entry point (no
// link-time dependence on libcuda).
bool encode_weight_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    static bool looked_up = false;
    if (!looked_up) {
        looked_up = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        (void)cudaGetLastError();
    }
    if (!encode) return false;
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {32, 256};
    const cuuint32_t estride[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool decode_shape_ok(int64_t B, int64_t dmem, int64_t d) {
    return B >= 1 && B <= 1048560 && dmem >= 8 && dmem <= 65536 && dmem % 8 == 0 && d >= 64 &&
           d <= 65536 && d % 64 == 0;
}

}  // namespace
}  // namespace eg

using namespace eg;

extern "C" {

const char* engram_status_string(engram_status_t s) {
    switch (s) {
        case ENGRAM_OK: return "ok";
        case ENGRAM_ERR_NULL: return "null pointer";
        case ENGRAM_ERR_ALIGN: return "misaligned pointer (16 bytes required)";
        case ENGRAM_ERR_SHAPE: return "size out of range";
        case ENGRAM_ERR_OVERLAP: return "output overlaps another buffer";
        case ENGRAM_ERR_WORKSPACE: return "workspace too small";
        case ENGRAM_ERR_DEVICE: return "no usable sm_103 device";
        case ENGRAM_ERR_LAUNCH: return "kernel launch failed";
    }
    return "unknown status";
}

size_t engram_gate_bwd_workspace_size(int64_t N) {
    if (N < 64 || N > ENGRAM_GATE_BWD_MAX_TOKENS || N % 64 != 0) return 0;
    return static_cast<size_t>(4) *
           (16 * static_cast<size_t>(N) + 4 * static_cast<size_t>(kGateD) * static_cast<size_t>(N / 64));
}

engram_status_t engram_gate_fwd(const void* x, const void* kv, const float* weight,
                                const uint8_t* mask, void* out, float* saved, int64_t N,
                                float eps, cudaStream_t stream) {
    if (!x || !kv || !weight || !out) return ENGRAM_ERR_NULL;
    if (N < 1 || N > ENGRAM_GATE_MAX_TOKENS) return ENGRAM_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(kv) || !aligned16(weight) || !aligned16(out) ||
        (saved && !aligned16(saved)))
        return ENGRAM_ERR_ALIGN;
    const size_t n = static_cast<size_t>(N);
    const Range ins[] = {{x, n * 4 * kGateD * 2}, {kv, n * 5 * kGateD * 2},
                         {weight, 4 * kGateD * 4}, {mask, mask ? n : 0}};
    const Range outs[] = {{out, n * 4 * kGateD * 2}, {saved, saved ? n * 64 : 0}};
    if (any_overlap(outs, 2, ins, 4)) return ENGRAM_ERR_OVERLAP;

    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* st = device_state();
    if (!st) return ENGRAM_ERR_DEVICE;
    LaunchCfg c = {};
    if (!gate_fwd_cfg(*st, N, c)) return ENGRAM_ERR_DEVICE;
    GateFwdParams p = {};
    p.x = static_cast<const uint16_t*>(x);
    p.key = static_cast<const uint16_t*>(kv);
    p.v = static_cast<const uint16_t*>(kv) + 4 * kGateD;
    p.key_ts = p.v_ts = 5LL * kGateD;
    p.w = weight;
    p.mask = mask;
    p.out = static_cast<uint16_t*>(out);
    p.saved = saved;
    p.err = st->err;
    p.N = N;
    p.d = kGateD;
    p.packed = 1;
    p.eps = eps;
    p.clamp = ENGRAM_GATE_CLAMP;
    return launch_status(gate_fwd_launch(p, c, stream));
}

}  // extern "C"

namespace {

// The packed gate backward; with wh / we set (a fused weight w = wh * we) the
// grad_weight merge also writes grad_wh and grad_we, and grad_weight may be
// null.  Arguments are validated by the callers' shared checks below.
engram_status_t gate_bwd_impl(const void* x, const void* kv, const float* weight,
                              const float* saved, const void* grad_out, const void* wh,
                              const void* we, void* grad_x, void* grad_kv, float* grad_weight,
                              float* grad_wh, float* grad_we, void* workspace,
                              size_t workspace_bytes, int64_t N, cudaStream_t stream) {
    const bool prod = wh != nullptr;
    if (!x || !kv || !weight || !saved || !grad_out || !grad_x || !grad_kv || !workspace ||
        (!prod && !grad_weight) || (prod && (!we || !grad_wh || !grad_we)))
        return ENGRAM_ERR_NULL;
    if (N < 64 || N > ENGRAM_GATE_BWD_MAX_TOKENS || N % 64 != 0) return ENGRAM_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(kv) || !aligned16(weight) || !aligned16(saved) ||
        !aligned16(grad_out) || !aligned16(grad_x) || !aligned16(grad_kv) ||
        (grad_weight && !aligned16(grad_weight)) || !aligned16(workspace) ||
        (prod && (!aligned16(wh) || !aligned16(we) || !aligned16(grad_wh) || !aligned16(grad_we))))
        return ENGRAM_ERR_ALIGN;
    const size_t need = engram_gate_bwd_workspace_size(N);
    if (workspace_bytes < need) return ENGRAM_ERR_WORKSPACE;
    const size_t n = static_cast<size_t>(N);
    const size_t wn = 4 * kGateD;
    const Range ins[] = {{x, n * 4 * kGateD * 2}, {kv, n * 5 * kGateD * 2},
                         {weight, wn * 4}, {saved, n * 64}, {grad_out, n * 4 * kGateD * 2},
                         {wh, prod ? wn * 2 : 0}, {we, prod ? wn * 2 : 0}};
    const Range outs[] = {{grad_x, n * 4 * kGateD * 2}, {grad_kv, n * 5 * kGateD * 2},
                          {grad_weight, grad_weight ? wn * 4 : 0}, {workspace, need},
                          {grad_wh, prod ? wn * 4 : 0}, {grad_we, prod ? wn * 4 : 0}};
    if (any_overlap(outs, 6, ins, 7)) return ENGRAM_ERR_OVERLAP;

    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* st = device_state();
    if (!st) return ENGRAM_ERR_DEVICE;
    const int G = gate_bwd_fused_groups(*st, N);
    if (G > 0) {
        // one pass: the workspace holds only the grad_weight words (G fp32 hi
        // slots, then G bf16 lo rows)
        float* partial = static_cast<float*>(workspace);
        uint16_t* partial_lo = reinterpret_cast<uint16_t*>(partial + static_cast<size_t>(G) * 4 * kGateD);
        GateBwdParams p = {};
        p.x = static_cast<const uint16_t*>(x);
        p.key = static_cast<const uint16_t*>(kv);
        p.v = static_cast<const uint16_t*>(kv) + 4 * kGateD;
        p.key_ts = p.v_ts = 5LL * kGateD;
        p.w = weight;
        p.saved = saved;
        p.gout = static_cast<const uint16_t*>(grad_out);
        p.gx = static_cast<uint16_t*>(grad_x);
        p.gkey = static_cast<uint16_t*>(grad_kv);
        p.gv = static_cast<uint16_t*>(grad_kv) + 4 * kGateD;
        p.gkey_ts = p.gv_ts = 5LL * kGateD;
        p.partial = partial;
        p.partial_lo = partial_lo;
        p.err = st->err;
        p.N = N;
        p.d = kGateD;
        p.pair_slots = 1;
        p.packed = 1;
        p.clamp = ENGRAM_GATE_CLAMP;
        engram_status_t s = launch_status(gate_bwd_fused_launch(p, G, stream));
        if (s != ENGRAM_OK) return s;
        GateWReduceParams r = {};
        r.partial = partial;
        r.out = grad_weight;
        r.nblocks = G;
        r.n = 4 * kGateD;
        r.stride = 4 * kGateD;
        r.pairs = 2;
        r.lo16 = partial_lo;
        if (prod) {
            r.wh = static_cast<const uint16_t*>(wh);
            r.we = static_cast<const uint16_t*>(we);
            r.grad_wh = grad_wh;
            r.grad_we = grad_we;
        }
        return launch_status(gate_wreduce_launch(r, stream));
    }
    LaunchCfg c = {};
    int ncols;
    int group_tokens = 0;
    if (!gate_bwd_cfg(*st, N, kGateD, false, c, ncols, group_tokens)) return ENGRAM_ERR_DEVICE;
    // workspace: [(N, 4, 4) per-token scalars | (N/64, 4, 5120) fp32 partial slots]
    float* coef = static_cast<float*>(workspace);
    float* partial = reinterpret_cast<float*>(static_cast<char*>(workspace) + 64 * n);
    GateBwdParams p = {};
    p.x = static_cast<const uint16_t*>(x);
    p.key = static_cast<const uint16_t*>(kv);
    p.v = static_cast<const uint16_t*>(kv) + 4 * kGateD;
    p.key_ts = p.v_ts = 5LL * kGateD;
    p.w = weight;
    p.saved = saved;
    p.gout = static_cast<const uint16_t*>(grad_out);
    p.gx = static_cast<uint16_t*>(grad_x);
    p.gkey = static_cast<uint16_t*>(grad_kv);
    p.gv = static_cast<uint16_t*>(grad_kv) + 4 * kGateD;
    p.gkey_ts = p.gv_ts = 5LL * kGateD;
    p.coef = coef;
    p.partial = partial;
    p.err = st->err;
    p.N = N;
    p.d = kGateD;
    p.ncols = ncols;
    p.stages = c.stages;
    p.group_tokens = group_tokens;
    p.pair_slots = (N / 64) >= 2 ? 1 : 0;
    p.token_split = c.token_split;
    p.packed = 1;
    p.clamp = ENGRAM_GATE_CLAMP;
    engram_status_t s = launch_status(gate_bwd_launch(p, c, stream));
    if (s != ENGRAM_OK) return s;
    GateWReduceParams r = {};
    r.partial = partial;
    r.out = grad_weight;
    r.nblocks = p.pair_slots ? 2 * c.grid_y : c.grid_y;
    r.n = 4 * kGateD;
    r.stride = 4 * kGateD;
    r.pairs = p.pair_slots;
    if (prod) {
        r.wh = static_cast<const uint16_t*>(wh);
        r.we = static_cast<const uint16_t*>(we);
        r.grad_wh = grad_wh;
        r.grad_we = grad_we;
    }
    return launch_status(gate_wreduce_launch(r, stream));
}

}  // namespace

extern "C" {

engram_status_t engram_gate_bwd(const void* x, const void* kv, const float* weight,
                                const float* saved, const void* grad_out, void* grad_x,
                                void* grad_kv, float* grad_weight, void* workspace,
                                size_t workspace_bytes, int64_t N, cudaStream_t stream) {
    return gate_bwd_impl(x, kv, weight, saved, grad_out, nullptr, nullptr, grad_x, grad_kv,
                         grad_weight, nullptr, nullptr, workspace, workspace_bytes, N, stream);
}

engram_status_t engram_gate_bwd_fused_weight(const void* x, const void* kv, const float* weight,
                                             const float* saved, const void* grad_out,
                                             const void* wh, const void* we, void* grad_x,
                                             void* grad_kv, float* grad_weight, float* grad_wh,
                                             float* grad_we, void* workspace,
                                             size_t workspace_bytes, int64_t N,
                                             cudaStream_t stream) {
    if (!wh) return ENGRAM_ERR_NULL;
    return gate_bwd_impl(x, kv, weight, saved, grad_out, wh, we, grad_x, grad_kv, grad_weight,
                         grad_wh, grad_we, workspace, workspace_bytes, N, stream);
}

engram_status_t engram_gateconv_fwd(const void* H, const void* k, const void* v,
                                    const float* rms_w_h, const float* rms_w_v,
                                    const float* conv_w, void* Y, void* vhat, float* alpha,
                                    float* rrms_h, float* rrms_k, float* rrms_v, int64_t M,
                                    int64_t T, int64_t d, float eps, cudaStream_t stream) {
    if (!H || !k || !v || !rms_w_h || !rms_w_v || !conv_w || !Y || !vhat || !alpha || !rrms_h ||
        !rrms_k || !rrms_v)
        return ENGRAM_ERR_NULL;
    if (!gc_shape_ok(M, T, d)) return ENGRAM_ERR_SHAPE;
    const void* all[] = {H, k, v, rms_w_h, rms_w_v, conv_w, Y, vhat, alpha, rrms_h, rrms_k, rrms_v};
    for (const void* ptr : all)
        if (!aligned16(ptr)) return ENGRAM_ERR_ALIGN;
    const size_t t = static_cast<size_t>(M * T), dd = static_cast<size_t>(d);
    const Range ins[] = {{H, t * dd * 2}, {k, t * dd * 2}, {v, t * dd * 2},
                         {rms_w_h, dd * 4}, {rms_w_v, dd * 4}, {conv_w, 4 * dd * 4}};
    const Range outs[] = {{Y, t * dd * 2}, {vhat, t * dd * 2}, {alpha, t * 4},
                          {rrms_h, t * 4}, {rrms_k, t * 4}, {rrms_v, t * 4}};
    if (any_overlap(outs, 6, ins, 6)) return ENGRAM_ERR_OVERLAP;

    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* st = device_state();
    if (!st) return ENGRAM_ERR_DEVICE;
    const GcGeom* g = gc_cfg(*st, 0, M, T, d);
    if (!g) return ENGRAM_ERR_DEVICE;
    GateConvFwdParams p;
    p.H = static_cast<const uint16_t*>(H);
    p.k = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.wh = rms_w_h;
    p.wv = rms_w_v;
    p.cw = conv_w;
    p.Y = static_cast<uint16_t*>(Y);
    p.vhat = static_cast<uint16_t*>(vhat);
    p.alpha = alpha;
    p.rh = rrms_h;
    p.rk = rrms_k;
    p.rv = rrms_v;
    p.err = st->err;
    p.M = static_cast<int>(M);
    p.T = static_cast<int>(T);
    p.d = static_cast<int>(d);
    p.ncols = g->ncols;
    p.ring_off = g->ring_off;
    p.range_len = g->range_len;
    p.ranges_per_row = g->rpr;
    p.eps = eps;
    p.inv_sqrt_d = static_cast<float>(1.0 / sqrt(static_cast<double>(d)));
    return launch_status(gateconv_fwd_launch(p, g->c, stream));
}

engram_status_t engram_gate_sep_fwd(const void* x, const void* k, const void* v,
                                    const float* weight, void* out, float* dot, float* gate,
                                    float* rstd_x, float* rstd_k, int64_t N, int64_t H, float eps,
                                    float clamp, cudaStream_t stream) {
    if (!x || !k || !v || !weight || !out) return ENGRAM_ERR_NULL;
    const int nsaved = (dot != nullptr) + (gate != nullptr) + (rstd_x != nullptr) + (rstd_k != nullptr);
    if (nsaved != 0 && nsaved != 4) return ENGRAM_ERR_NULL;
    if (N < 1 || N > ENGRAM_GATE_MAX_TOKENS || H < 8 || H > ENGRAM_GATE_SEP_MAX_HIDDEN || H % 8 != 0)
        return ENGRAM_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(k) || !aligned16(v) || !aligned16(weight) || !aligned16(out) ||
        (nsaved && (!aligned16(dot) || !aligned16(gate) || !aligned16(rstd_x) || !aligned16(rstd_k))))
        return ENGRAM_ERR_ALIGN;
    const size_t n = static_cast<size_t>(N), h = static_cast<size_t>(H);
    const Range ins[] = {{x, n * 4 * h * 2}, {k, n * 4 * h * 2}, {v, n * h * 2}, {weight, 4 * h * 4}};
    const Range outs[] = {{out, n * 4 * h * 2}, {dot, dot ? n * 16 : 0}, {gate, gate ? n * 16 : 0},
                          {rstd_x, rstd_x ? n * 16 : 0}, {rstd_k, rstd_k ? n * 16 : 0}};
    if (any_overlap(outs, 5, ins, 4)) return ENGRAM_ERR_OVERLAP;

    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* st = device_state();
    if (!st) return ENGRAM_ERR_DEVICE;
    LaunchCfg c = {};
    if (!gate_fwd_cfg(*st, N, c)) return ENGRAM_ERR_DEVICE;
    GateFwdParams p = {};
    p.x = static_cast<const uint16_t*>(x);
    p.key = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.key_ts = 4LL * H;
    p.v_ts = H;
    p.w = weight;
    p.out = static_cast<uint16_t*>(out);
    p.sv_gate = gate;
    p.sv_dot = dot;
    p.sv_rx = rstd_x;
    p.sv_rk = rstd_k;
    p.err = st->err;
    p.N = N;
    p.d = static_cast<int>(H);
    p.eps = eps;
    p.clamp = clamp;
    return launch_status(gate_fwd_launch(p, c, stream));
}

size_t engram_gate_sep_bwd_workspace_size(int64_t N) {
    if (N < 1 || N > ENGRAM_GATE_MAX_TOKENS) return 0;
    return static_cast<size_t>(64) * static_cast<size_t>(N);
}

engram_status_t engram_gate_sep_bwd(const void* grad_out, const void* x, const void* k,
                                    const void* v, const float* weight, const float* dot,
                                    const float* gate, const float* rstd_x, const float* rstd_k,
                                    void* grad_x, void* grad_k, void* grad_v, float* grad_w_partial,
                                    void* workspace, size_t workspace_bytes, int64_t N, int64_t H,
                                    float clamp, cudaStream_t stream) {
    if (!grad_out || !x || !k || !v || !weight || !dot || !gate || !rstd_x || !rstd_k || !grad_x ||
        !grad_k || !grad_v || !grad_w_partial || !workspace)
        return ENGRAM_ERR_NULL;
    if (N < 1 || N > ENGRAM_GATE_MAX_TOKENS || H < 8 || H > ENGRAM_GATE_SEP_MAX_HIDDEN || H % 8 != 0)
        return ENGRAM_ERR_SHAPE;
    const void* all[] = {grad_out, x, k, v, weight, dot, gate, rstd_x, rstd_k,
                         grad_x, grad_k, grad_v, grad_w_partial, workspace};
    for (const void* ptr : all)
        if (!aligned16(ptr)) return ENGRAM_ERR_ALIGN;
    const size_t need = engram_gate_sep_bwd_workspace_size(N);
    if (workspace_bytes < need) return ENGRAM_ERR_WORKSPACE;
    const size_t n = static_cast<size_t>(N), h = static_cast<size_t>(H);
    const size_t nblk = (n + 63) / 64;
    const Range ins[] = {{grad_out, n * 4 * h * 2}, {x, n * 4 * h * 2}, {k, n * 4 * h * 2},
                         {v, n * h * 2}, {weight, 4 * h * 4}, {dot, n * 16}, {gate, n * 16},
                         {rstd_x, n * 16}, {rstd_k, n * 16}};
    const Range outs[] = {{grad_x, n * 4 * h * 2}, {grad_k, n * 4 * h * 2}, {grad_v, n * h * 2},
                          {grad_w_partial, nblk * 4 * h * 4}, {workspace, need}};
    if (any_overlap(outs, 5, ins, 9)) return ENGRAM_ERR_OVERLAP;

    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* st = device_state();
    if (!st) return ENGRAM_ERR_DEVICE;
    LaunchCfg c = {};
    int ncols;
    int group_tokens = 0;
    if (!gate_bwd_cfg(*st, N, H, true, c, ncols, group_tokens)) return ENGRAM_ERR_DEVICE;
    GateBwdParams p = {};
    p.x = static_cast<const uint16_t*>(x);
    p.key = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.key_ts = 4LL * H;
    p.v_ts = H;
    p.w = weight;
    p.sv_gate = gate;
    p.sv_dot = dot;
    p.sv_rx = rstd_x;
    p.sv_rk = rstd_k;
    p.gout = static_cast<const uint16_t*>(grad_out);
    p.gx = static_cast<uint16_t*>(grad_x);
    p.gkey = static_cast<uint16_t*>(grad_k);
    p.gv = static_cast<uint16_t*>(grad_v);
    p.gkey_ts = 4LL * H;
    p.gv_ts = H;
    p.coef = static_cast<float*>(workspace);
    p.partial = grad_w_partial;  // one slot per 64-token block, written directly
    p.err = st->err;
    p.N = N;
    p.d = static_cast<int>(H);
    p.ncols = ncols;
    p.stages = c.stages;
    p.group_tokens = group_tokens;
    p.pair_slots = 0;
    p.clamp = clamp;
    return launch_status(gate_bwd_launch(p, c, stream));
}

engram_status_t engram_fused_weight(const void* wh, const void* we, float* weight, int64_t n,
                                    cudaStream_t stream) {
    if (!wh || !we || !weight) return ENGRAM_ERR_NULL;
    if (n < 1 || n > (int64_t(1) << 40)) return ENGRAM_ERR_SHAPE;
    if (!aligned16(wh) || !aligned16(we) || !aligned16(weight)) return ENGRAM_ERR_ALIGN;
    const size_t m = static_cast<size_t>(n);
    const Range ins[] = {{wh, m * 2}, {we, m * 2}};
    const Range outs[] = {{weight, m * 4}};
    if (any_overlap(outs, 1, ins, 2)) return ENGRAM_ERR_OVERLAP;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!device_state()) return ENGRAM_ERR_DEVICE;
    FusedWeightParams p = {};
    p.wh = static_cast<const uint16_t*>(wh);
    p.we = static_cast<const uint16_t*>(we);
    p.weight = weight;
    p.n = n;
    return launch_status(fused_weight_launch(p, stream));
}

engram_status_t engram_fused_weight_bwd(const float* grad_w_partial, int64_t nblocks,
                                        const void* wh, const void* we, float* grad_w,
                                        float* grad_wh, float* grad_we, int64_t n,
                                        cudaStream_t stream) {
    if (!grad_w_partial || !wh || !we || !grad_wh || !grad_we) return ENGRAM_ERR_NULL;
    if (n < 1 || nblocks < 1 || n > (int64_t(1) << 40) / nblocks) return ENGRAM_ERR_SHAPE;
    if (!aligned16(grad_w_partial) || !aligned16(wh) || !aligned16(we) || !aligned16(grad_wh) ||
        !aligned16(grad_we) || (grad_w && !aligned16(grad_w)))
        return ENGRAM_ERR_ALIGN;
    const size_t m = static_cast<size_t>(n);
    const Range ins[] = {{grad_w_partial, m * static_cast<size_t>(nblocks) * 4}, {wh, m * 2}, {we, m * 2}};
    const Range outs[] = {{grad_w, grad_w ? m * 4 : 0}, {grad_wh, m * 4}, {grad_we, m * 4}};
    if (any_overlap(outs, 3, ins, 3)) return ENGRAM_ERR_OVERLAP;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!device_state()) return ENGRAM_ERR_DEVICE;
    FusedWeightParams p = {};
    p.wh = static_cast<const uint16_t*>(wh);
    p.we = static_cast<const uint16_t*>(we);
    p.partial = grad_w_partial;
    p.grad_w = grad_w;
    p.grad_wh = grad_wh;
    p.grad_we = grad_we;
    p.n = n;
    p.nblocks = nblocks;
    return launch_status(fused_weight_bwd_launch(p, stream));
}

size_t engram_decode_workspace_size(int64_t B, int64_t d_mem, int64_t d) {
    if (!decode_shape_ok(B, d_mem, d)) return 0;
    // [(B, d) fp32 v | (B, d / 32, 4) fp32 row sums of the 32-column tiles]
    return static_cast<size_t>(B) * static_cast<size_t>(d) * 4 + static_cast<size_t>(B) * (d / 32) * 16;
}

engram_status_t engram_decode_fwd(const void* e, const void* h, const void* state, int64_t L,
                                  const void* W_K, const void* W_V, const float* rms_w_h,
                                  const float* rms_w_v, const float* conv_w, void* y,
                                  void* new_state, void* workspace, size_t workspace_bytes,
                                  int64_t B, int64_t d_mem, int64_t d, int64_t max_len, int64_t w,
                                  int64_t dilation, float eps, cudaStream_t stream) {
    if (!e || !h || !W_K || !W_V || !rms_w_h || !rms_w_v || !conv_w || !y || !new_state || !workspace ||
        (L > 0 && !state))
        return ENGRAM_ERR_NULL;
    if (!decode_shape_ok(B, d_mem, d) || w < 1 || w > 64 || dilation < 1 || dilation > (1 << 20) ||
        max_len < 1 || max_len > 65536 || L < 0 || L > max_len)
        return ENGRAM_ERR_SHAPE;
    const void* all[] = {e, h, W_K, W_V, rms_w_h, rms_w_v, conv_w, y, new_state, workspace};
    for (const void* ptr : all)
        if (!aligned16(ptr)) return ENGRAM_ERR_ALIGN;
    if (L > 0 && !aligned16(state)) return ENGRAM_ERR_ALIGN;
    const size_t need = engram_decode_workspace_size(B, d_mem, d);
    if (workspace_bytes < need) return ENGRAM_ERR_WORKSPACE;
    const size_t b = static_cast<size_t>(B), dm = static_cast<size_t>(d_mem), dd = static_cast<size_t>(d);
    const Range ins[] = {{e, b * dm * 2}, {h, b * dd * 2}, {state, L > 0 ? b * L * dd * 2 : 0},
                         {W_K, dm * dd * 2}, {W_V, dm * dd * 2}, {rms_w_h, dd * 4}, {rms_w_v, dd * 4},
                         {conv_w, static_cast<size_t>(w) * dd * 4}};
    const Range outs[] = {{y, b * dd * 2}, {new_state, b * static_cast<size_t>(max_len) * dd * 2},
                          {workspace, need}};
    if (any_overlap(outs, 3, ins, 8)) return ENGRAM_ERR_OVERLAP;

    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* st = device_state();
    if (!st) return ENGRAM_ERR_DEVICE;
    if (!st->decode_ready) {
        if (decode_prepare() != cudaSuccess) {
            (void)cudaGetLastError();
            return ENGRAM_ERR_DEVICE;
        }
        st->decode_ready = true;
    }
    DecodeParams p = {};
    p.e = static_cast<const uint16_t*>(e);
    p.h = static_cast<const uint16_t*>(h);
    p.state = static_cast<const uint16_t*>(state);
    p.WK = static_cast<const uint16_t*>(W_K);
    p.WV = static_cast<const uint16_t*>(W_V);
    p.wh = rms_w_h;
    p.wv = rms_w_v;
    p.cw = conv_w;
    p.y = static_cast<uint16_t*>(y);
    p.new_state = static_cast<uint16_t*>(new_state);
    p.vbuf = static_cast<float*>(workspace);
    p.stats = reinterpret_cast<float*>(static_cast<char*>(workspace) + static_cast<size_t>(B) * d * 4);
    p.err = st->err;
    if (!encode_weight_map(&p.tmk, W_K, d_mem, d) || !encode_weight_map(&p.tmv, W_V, d_mem, d))
        return ENGRAM_ERR_DEVICE;
    p.B = static_cast<int>(B);
    p.dmem = static_cast<int>(d_mem);
    p.d = static_cast<int>(d);
    p.L = static_cast<int>(L);
    p.max_len = static_cast<int>(max_len);
    p.w = static_cast<int>(w);
    p.dil = static_cast<int>(dilation);
    p.eps = eps;
    p.inv_sqrt_d = static_cast<float>(1.0 / sqrt(static_cast<double>(d)));
    return launch_status(decode_launch(p, stream));
}

size_t engram_gateconv_bwd_workspace_size(int64_t M, int64_t T, int64_t d) {
    if (!gc_shape_ok(M, T, d)) return 0;
    return static_cast<size_t>(gc_bwd_slots(M, T)) * 6 * static_cast<size_t>(d) * 4 + kGcXrecBytes;
}

engram_status_t engram_gateconv_bwd(const void* dY, const void* H, const void* k,
                                    const void* v, const float* rms_w_h,
                                    const float* rms_w_v, const float* conv_w,
                                    const void* vhat, const float* alpha,
                                    const float* rrms_h, const float* rrms_k,
                                    const float* rrms_v, void* dH, void* dk, void* dv,
                                    float* drms_w_h, float* drms_w_v, float* dconv_w,
                                    void* workspace, size_t workspace_bytes, int64_t M,
                                    int64_t T, int64_t d, float eps, cudaStream_t stream) {
    if (!dY || !H || !k || !v || !rms_w_h || !rms_w_v || !conv_w || !vhat || !alpha || !rrms_h ||
        !rrms_k || !rrms_v || !dH || !dk || !dv || !drms_w_h || !drms_w_v || !dconv_w ||
        !workspace)
        return ENGRAM_ERR_NULL;
    if (!gc_shape_ok(M, T, d)) return ENGRAM_ERR_SHAPE;
    const void* all[] = {dY, H, k, v, rms_w_h, rms_w_v, conv_w, vhat, alpha, rrms_h, rrms_k,
                         rrms_v, dH, dk, dv, drms_w_h, drms_w_v, dconv_w, workspace};
    for (const void* ptr : all)
        if (!aligned16(ptr)) return ENGRAM_ERR_ALIGN;
    const size_t need = engram_gateconv_bwd_workspace_size(M, T, d);
    if (workspace_bytes < need) return ENGRAM_ERR_WORKSPACE;
    const size_t t = static_cast<size_t>(M * T), dd = static_cast<size_t>(d);
    const Range ins[] = {{dY, t * dd * 2}, {H, t * dd * 2}, {k, t * dd * 2}, {v, t * dd * 2},
                         {rms_w_h, dd * 4}, {rms_w_v, dd * 4}, {conv_w, 4 * dd * 4},
                         {vhat, t * dd * 2}, {alpha, t * 4}, {rrms_h, t * 4}, {rrms_k, t * 4},
                         {rrms_v, t * 4}};
    const Range outs[] = {{dH, t * dd * 2}, {dk, t * dd * 2}, {dv, t * dd * 2},
                          {drms_w_h, dd * 4}, {drms_w_v, dd * 4}, {dconv_w, 4 * dd * 4},
                          {workspace, need}};
    if (any_overlap(outs, 7, ins, 12)) return ENGRAM_ERR_OVERLAP;

    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* st = device_state();
    if (!st) return ENGRAM_ERR_DEVICE;
    const GcGeom* g = gc_cfg(*st, 1, M, T, d);
    if (!g) return ENGRAM_ERR_DEVICE;
    float* partial = static_cast<float*>(workspace);
    unsigned long long* xrec =
        reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) + (need - kGcXrecBytes));
    GateConvBwdParams p;
    p.dY = static_cast<const uint16_t*>(dY);
    p.H = static_cast<const uint16_t*>(H);
    p.k = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.wh = rms_w_h;
    p.wv = rms_w_v;
    p.cw = conv_w;
    p.vhat = static_cast<const uint16_t*>(vhat);
    p.alpha = alpha;
    p.rh = rrms_h;
    p.rk = rrms_k;
    p.rv = rrms_v;
    p.dH = static_cast<uint16_t*>(dH);
    p.dk = static_cast<uint16_t*>(dk);
    p.dv = static_cast<uint16_t*>(dv);
    p.partial = partial;
    p.xrec = xrec;
    p.err = st->err;
    p.M = static_cast<int>(M);
    p.T = static_cast<int>(T);
    p.d = static_cast<int>(d);
    p.group = g->c.cluster;
    p.nranges = g->c.clusters;
    p.ncols = g->ncols;
    p.ring_off = g->ring_off;
    p.sc_off = g->sc_off;
    p.range_len = g->range_len;
    p.ranges_per_row = g->rpr;
    p.eps = eps;
    p.inv_sqrt_d = static_cast<float>(1.0 / sqrt(static_cast<double>(d)));
    engram_status_t s = ENGRAM_OK;
    if (g->groups > 0) {
        // the exchange records start at zero (sequence 0 is never awaited)
        const size_t xbytes = static_cast<size_t>(g->groups) * g->c.cluster * 2 * 128;
        s = launch_status(cudaMemsetAsync(xrec, 0, xbytes, stream));
        if (s != ENGRAM_OK) return s;
    }
    s = launch_status(gateconv_bwd_launch(p, g->c, g->groups, stream));
    if (s != ENGRAM_OK) return s;
    const int R = g->c.clusters;
    float* outs3[3] = {drms_w_h, drms_w_v, dconv_w};
    const int offs[3] = {0, 1, 2};
    const int lens[3] = {1, 1, 4};
    for (int i = 0; i < 3; ++i) {
        GateWReduceParams r = {};
        r.partial = partial + static_cast<size_t>(offs[i]) * dd;
        r.out = outs3[i];
        r.nblocks = R;
        r.n = lens[i] * static_cast<int>(d);
        r.stride = 6 * static_cast<int>(d);
        r.pairs = 0;
        s = launch_status(gateconv_wreduce_launch(r, stream));
        if (s != ENGRAM_OK) return s;
    }
    return ENGRAM_OK;
}

}  // extern "C"

// Workspace of engram_gate_bwd_noalloc: a file-scope device array, so that
// callers without an allocator can run the backward.  Host code never uses
// the symbol itself as a pointer: its device address is looked up once per
// device, with that device current, and that address is what the kernels get.
static __device__ __align__(256) unsigned char g_gate_bwd_scratch[ENGRAM_GATE_BWD_NOALLOC_SCRATCH_BYTES];

namespace {
// the array's device address per device, with the ID of the context it was
// looked up in (a reset device gets a new context and a new address)
eg::NoallocScratch g_scratch[eg::kMaxDevices];
}  // namespace

extern "C" {

engram_status_t engram_gate_bwd_noalloc(const void* x, const void* kv, const float* weight,
                                        const float* saved, const void* grad_out, void* grad_x,
                                        void* grad_kv, float* grad_weight, int64_t N,
                                        cudaStream_t stream) {
    if (N < 64 || N > ENGRAM_GATE_BWD_NOALLOC_MAX_TOKENS || N % 64 != 0) return ENGRAM_ERR_SHAPE;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        int dev = 0;
        // device_state() makes the device's context current and identifies it
        if (!eg::device_state() || cudaGetDevice(&dev) != cudaSuccess || dev < 0 ||
            dev >= eg::kMaxDevices) {
            (void)cudaGetLastError();
            return ENGRAM_ERR_DEVICE;
        }
        eg::NoallocScratch& sc = g_scratch[dev];
        const unsigned long long ctx = eg::g_dev[dev].ctx;
        if (sc.ptr == nullptr || sc.ctx != ctx) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_gate_bwd_scratch) != cudaSuccess || ptr == nullptr) {
                (void)cudaGetLastError();
                return ENGRAM_ERR_DEVICE;
            }
            sc.ptr = ptr;
            sc.ctx = ctx;
        }
        scratch = sc.ptr;
    }
    // the regular backward, with the library's array as its workspace
    return engram_gate_bwd(x, kv, weight, saved, grad_out, grad_x, grad_kv, grad_weight, scratch,
                           ENGRAM_GATE_BWD_NOALLOC_SCRATCH_BYTES, N, stream);
}

engram_status_t engram_device_error(uint32_t* flags) {
    if (!flags) return ENGRAM_ERR_NULL;
    unsigned int v = 0u, zero = 0u;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(&v, eg_error_word, sizeof(v)) != cudaSuccess ||
        cudaMemcpyToSymbol(eg_error_word, &zero, sizeof(zero)) != cudaSuccess) {
        (void)cudaGetLastError();
        return ENGRAM_ERR_DEVICE;
    }
    *flags = v;
    return ENGRAM_OK;
}

engram_status_t engram_launch_info(int op, int64_t n0, int64_t n1, int64_t n2,
                                   engram_launch_info_t* info) {
    if (!info) return ENGRAM_ERR_NULL;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState* st = device_state();
    if (!st) return ENGRAM_ERR_DEVICE;
    LaunchCfg c = {};
    int ncols;
    bool ok = false;
    switch (op) {
        case 0:
            ok = n0 >= 1 && n0 <= ENGRAM_GATE_MAX_TOKENS && gate_fwd_cfg(*st, n0, c);
            break;
        case 1: {
            int gt = 0;
            ok = engram_gate_bwd_workspace_size(n0) > 0;
            const int G = ok ? gate_bwd_fused_groups(*st, n0) : 0;
            if (G > 0) {
                // one-pass backward: clusters of two CTAs (column halves) per
                // token range, plus the grad_weight merge
                info->cluster = 2;
                info->threads = gate_bwd_fused_threads();
                info->clusters = G;
                info->stages = 4;
                info->smem_bytes = gate_bwd_fused_smem();
                info->resident = st->fused_clusters;
                info->kernels = 2;
                return ENGRAM_OK;
            }
            ok = ok && gate_bwd_cfg(*st, n0, kGateD, false, c, ncols, gt);
            // CTAs sharing a token row = column slices; "clusters" = token groups
            if (ok) {
                c.cluster = c.clusters;
                c.clusters = c.grid_y;
            }
            break;
        }
        case 2:
        case 3: {
            const GcGeom* g = gc_shape_ok(n0, n1, n2) ? gc_cfg(*st, op - 2, n0, n1, n2) : nullptr;
            ok = g != nullptr;
            if (ok) c = g->c;
            if (ok && g->groups > 0) {
                // the backward's cooperative launch: groups of c.cluster CTAs,
                // each taking token ranges in turn
                info->cluster = c.cluster;
                info->threads = c.threads;
                info->clusters = c.clusters;
                info->stages = c.stages;
                info->smem_bytes = c.smem;
                info->resident = g->groups;
                info->kernels = 4;
                return ENGRAM_OK;
            }
            break;
        }
        default:
            return ENGRAM_ERR_SHAPE;
    }
    if (!ok) return ENGRAM_ERR_SHAPE;
    info->cluster = c.cluster;
    info->threads = c.threads;
    info->clusters = c.clusters;
    info->stages = c.stages;
    info->smem_bytes = c.smem;
    // co-resident CTA groups: CTAs for the gate kernels, clusters for GateConv
    info->resident = op == 1 ? max_clusters(*st, op, 1, c.threads, c.smem) / c.cluster
                             : max_clusters(*st, op, op >= 2 ? c.cluster : 1, c.threads, c.smem);
    // kernels a call launches: gate fwd 1; gate bwd coefficients, elementwise,
    // merge; GateConv fwd 1; GateConv bwd main + three merges
    info->kernels = op == 0 ? 1 : op == 1 ? 3 : op == 2 ? 1 : 4;
    return ENGRAM_OK;
}

}  // extern "C"
