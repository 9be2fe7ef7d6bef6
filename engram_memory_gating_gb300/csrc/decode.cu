// GateConv decode, one token (TileOPs "Engram Operators", Decode section,
// EngramDecodeFwdOp: GEMV projection + gating + dilated conv + SiLU, with a
// conv_state cache of at most max_conv_len tokens).  Per batch row b:
//   k = e W_K, v = e W_V                         (fp32 accumulation)
//   alpha = sigmoid(sum (h rrms_h w_h)(k rrms_k w_h) / sqrt(d)),  vhat = alpha v
//   u = vhat rrms_v w_v
//   c = sum_{j<w} conv_w[j] u_{t-(w-1-j) dil}    (u_t this token; older u from
//       the cache, most recent last; zero beyond its L rows)
//   y = SiLU(c) + vhat
//   new cache = the last max_len rows of [zeros, cache, bf16(u_t)]
//
// Kernel 1 (projection): a CTA owns 128 columns of d and a slice of the d_mem
// rows of both weight matrices, for up to 8 batch rows; each lane keeps two
// columns' running sums for every batch row (W read once from HBM per batch
// chunk, e staged in shared memory), the CTA's eight warps are summed in
// shared memory in a fixed order and the slice's partial k and v go to the
// workspace; the projection CTAs also shift the cache by one token (rows
// r + 1 -> r), which depends on nothing else.  Kernel 2 (a cluster of 8 CTAs
// per batch row, each owning an eighth of the columns): sums the slices in a
// fixed order, forms the row statistics (block reduction, then an exchange
// across the cluster through distributed shared memory), and writes y and the
// cache's new last row.
#include "common.cuh"
#include "engram_internal.h"

namespace eg {
namespace {

// Programmatic dependent launch: the row kernel is scheduled while the
// projection runs and waits for the projection grid only where it reads the
// partial sums.  The projection is itself launched that way: it waits for the
// preceding kernel (e.g. the previous decode step, which wrote the cache it
// shifts) before reading anything, so only its launch overlaps that kernel's
// tail.  Each kernel lets its successor be scheduled only after its own wait.
EG_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
EG_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// The two halves of a cluster barrier (every thread of every CTA; release on
// arrive, acquire on wait), so that work can run between them.
EG_DEV void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
EG_DEV void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Asynchronous 16-byte store into the shared memory of a CTA of this cluster,
// completing 16 bytes on that CTA's mbarrier.
EG_DEV void st_async_f4(uint32_t remote_addr, float4 v, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
            remote_addr),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(remote_bar)
        : "memory");
}

constexpr int kCols = 128;   // columns per projection CTA (32 lanes x 4 columns)
constexpr int kWarps1 = 8;   // warps of a projection CTA (interleaved 4-row groups)
constexpr int kBc = 8;       // batch rows per projection CTA
constexpr int kUnroll = 4;   // weight rows per warp iteration

// Kernel 1: CTA (x: 128-column tile, y: d_mem row split, z: batch chunk).
// Lane l owns columns tile + 4l .. 4l+3 of both matrices (8-byte loads; a
// warp reads 256 contiguous bytes of each weight row); warp w takes the row
// groups m0 + 4w + 32k; the next group's weights are loaded while the
// current one is used.  The eight warps' sums are added in warp order.
__global__ void __launch_bounds__(32 * kWarps1, 2) decode_proj_kernel(const DecodeParams p) {
    extern __shared__ __align__(16) float sm[];
    float* es = sm;                                   // [kBc][rows] e of this slice
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int col = blockIdx.x * kCols + 4 * lane;
    const int rows = p.rows_per_split;
    const int m0 = blockIdx.y * rows;
    const int m1 = min(p.dmem, m0 + rows);
    const int b0 = blockIdx.z * kBc;
    const int nb = min(kBc, p.B - b0);
    grid_dep_wait();
    grid_dep_launch();
    // the cache shift (independent of the projection), spread over all CTAs:
    // row r < max_len - 1 of the new cache is row r + 1 of the left-padded old one
    {
        const long long nq = static_cast<long long>(p.B) * (p.max_len - 1) * (p.d / 8);  // 16-byte chunks
        const long long ncta = static_cast<long long>(gridDim.x) * gridDim.y * gridDim.z;
        const long long cta = (static_cast<long long>(blockIdx.z) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        const long long q0 = nq * cta / ncta, q1 = nq * (cta + 1) / ncta;
        const int pad = p.max_len - p.L;
        const long long per_row = p.d / 8, per_b = static_cast<long long>(p.max_len - 1) * per_row;
        for (long long q = q0 + threadIdx.x; q < q1; q += blockDim.x) {
            const long long bb = q / per_b, rem = q - bb * per_b;
            const long long r = rem / per_row, i = (rem - r * per_row) * 8;
            const long long src = r + 1 - pad;
            uint4 val = make_uint4(0, 0, 0, 0);
            if (src >= 0 && src < p.L)
                val = __ldg(reinterpret_cast<const uint4*>(p.state + (bb * p.L + src) * p.d + i));
            *reinterpret_cast<uint4*>(p.new_state + (bb * p.max_len + r) * p.d + i) = val;
        }
    }
    for (int i = threadIdx.x; i < kBc * rows; i += blockDim.x) {
        const int b = i / rows, m = i - b * rows;
        es[i] = (b < nb && m0 + m < m1)
            ? __uint_as_float(static_cast<uint32_t>(__ldg(p.e + static_cast<long long>(b0 + b) * p.dmem + m0 + m)) << 16)
            : 0.f;
    }
    __syncthreads();

    float2 ak[kBc][2], av[kBc][2];
#pragma unroll
    for (int b = 0; b < kBc; ++b) ak[b][0] = ak[b][1] = av[b][0] = av[b][1] = make_float2(0.f, 0.f);
    const uint2* wk = reinterpret_cast<const uint2*>(p.WK + col);
    const uint2* wv = reinterpret_cast<const uint2*>(p.WV + col);
    const long long rs = p.d / 4;  // row stride in 4-column units
    uint2 qk[kUnroll], qv[kUnroll], nk[kUnroll], nv[kUnroll];
    const bool colok = col < p.d;  // the last tile may be partly outside d (d % 64 == 0)
    auto load = [&](int m, uint2 (&k4)[kUnroll], uint2 (&v4)[kUnroll]) {
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const bool ok = colok && m + r < m1;
            k4[r] = ok ? __ldg(wk + (m + r) * rs) : make_uint2(0u, 0u);
            v4[r] = ok ? __ldg(wv + (m + r) * rs) : make_uint2(0u, 0u);
        }
    };
    // the next row group is in flight while the current one is used
    constexpr int kStep = kWarps1 * kUnroll;
    int m = m0 + warp * kUnroll;
    if (m < m1) load(m, qk, qv);
    for (; m < m1; m += kStep) {
        if (m + kStep < m1) load(m + kStep, nk, nv);
#pragma unroll
        for (int b = 0; b < kBc; ++b) {
            const float4 e4 = *reinterpret_cast<const float4*>(es + b * rows + (m - m0));
            const float ev[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
            for (int r = 0; r < kUnroll; ++r) {
                const float2 e2 = splat2(ev[r]);
                ak[b][0] = fma2(e2, bf2(qk[r].x), ak[b][0]);
                ak[b][1] = fma2(e2, bf2(qk[r].y), ak[b][1]);
                av[b][0] = fma2(e2, bf2(qv[r].x), av[b][0]);
                av[b][1] = fma2(e2, bf2(qv[r].y), av[b][1]);
            }
        }
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            qk[r] = nk[r];
            qv[r] = nv[r];
        }
    }
    // the eight warps' sums, in warp order
    __syncthreads();
    float4* red = reinterpret_cast<float4*>(sm);      // [kWarps1][kBc][2][32]
#pragma unroll
    for (int b = 0; b < kBc; ++b) {
        red[((warp * kBc + b) * 2 + 0) * 32 + lane] = make_float4(ak[b][0].x, ak[b][0].y, ak[b][1].x, ak[b][1].y);
        red[((warp * kBc + b) * 2 + 1) * 32 + lane] = make_float4(av[b][0].x, av[b][0].y, av[b][1].x, av[b][1].y);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kBc * 2 * 32; i += blockDim.x) {
        const int b = i / 64, kvsel = (i >> 5) & 1, ln = i & 31;
        if (b >= nb || blockIdx.x * kCols + 4 * ln >= p.d) continue;
        float4 s = red[((0 * kBc + b) * 2 + kvsel) * 32 + ln];
        for (int w = 1; w < kWarps1; ++w) {
            const float4 q = red[((w * kBc + b) * 2 + kvsel) * 32 + ln];
            s.x += q.x;
            s.y += q.y;
            s.z += q.z;
            s.w += q.w;
        }
        float* dst = p.part + ((static_cast<long long>(kvsel) * p.splits + blockIdx.y) * p.B + b0 + b) * p.d +
                     blockIdx.x * kCols + 4 * ln;
        *reinterpret_cast<float4*>(dst) = s;
    }
}

constexpr int kThreads2 = 256;
constexpr int kCluster2 = 8;   // CTAs per batch row in kernel 2
constexpr int kCache = 4;      // columns per thread whose v is kept between the passes

// Kernel 2: a cluster of kCluster2 CTAs per batch row, CTA `rank` owning
// d / kCluster2 columns.  Each CTA sums its columns' row statistics and stores
// the four partial sums into slot `rank` of every CTA of the cluster
// (asynchronous remote stores completing on that CTA's mbarrier); each CTA
// adds the eight slots in rank order, so all form identical scalars, then
// writes y and the new cache for its columns.  Every CTA waits for all eight
// slots before it goes on, so none leaves while a store to it is in flight.
__global__ void __launch_bounds__(kThreads2) decode_row_kernel(const DecodeParams p) {
    __shared__ float4 sh[kThreads2 / 32];
    __shared__ float4 cta_sum;
    __shared__ float4 slots[kCluster2];
    __shared__ uint64_t xbar;
    if (threadIdx.x == 0) {
        mbar_init(&xbar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&xbar, kCluster2 * 16u);
    }
    // the barrier is initialised before any peer stores into this CTA (the
    // matching wait comes just before the stores)
    cluster_arrive();
    const uint32_t rank = cluster_rank();
    const int b = static_cast<int>(cluster_index());
    const int d = p.d;
    const int ncol = d / kCluster2;
    const int c0 = static_cast<int>(rank) * ncol;
    const long long pk = static_cast<long long>(p.splits) * p.B * d;  // offset of the v partials
    // k, v of column i: the splits summed in order (loads issued 8 at a time)
    auto kv_at = [&](int i, float& kk, float& vv) {
        kk = 0.f;
        vv = 0.f;
        const float* src = p.part + static_cast<long long>(b) * d + i;
        const long long ss = static_cast<long long>(p.B) * d;  // split stride
        for (int s0 = 0; s0 < p.splits; s0 += 8) {
            float a[8], c[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const bool ok = s0 + u < p.splits;
                a[u] = ok ? __ldg(src + (s0 + u) * ss) : 0.f;
                c[u] = ok ? __ldg(src + pk + (s0 + u) * ss) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                kk += a[u];
                vv += c[u];
            }
        }
    };
    auto bf = [](const uint16_t* q, long long i) { return __uint_as_float(static_cast<uint32_t>(__ldg(q + i)) << 16); };

    // ---- this CTA's share of the row statistics (v of the first kCache
    // columns of each thread kept for the second pass).  h and w_h of those
    // columns are inputs, read before waiting for the projection grid.
    float vc[kCache], hc[kCache], wc[kCache];
#pragma unroll
    for (int q = 0; q < kCache; ++q) {
        const int i = c0 + threadIdx.x + q * static_cast<int>(blockDim.x);
        const bool ok = i < c0 + ncol;
        hc[q] = ok ? bf(p.h, static_cast<long long>(b) * d + i) : 0.f;
        wc[q] = ok ? __ldg(p.wh + i) : 0.f;
    }
    grid_dep_wait();
    grid_dep_launch();   // the next decode step's projection may be scheduled (it waits for this grid)
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);   // sum h^2, k^2, h k w_h^2, v^2
    int it = 0;
    for (int i = c0 + threadIdx.x; i < c0 + ncol; i += blockDim.x, ++it) {
        float kk, vv;
        kv_at(i, kk, vv);
        float hh = 0.f, w = 0.f;
        if (it < kCache) {
#pragma unroll
            for (int q = 0; q < kCache; ++q)
                if (q == it) {
                    vc[q] = vv;
                    hh = hc[q];
                    w = wc[q];
                }
        } else {
            hh = bf(p.h, static_cast<long long>(b) * d + i);
            w = __ldg(p.wh + i);
        }
        acc.x = fmaf(hh, hh, acc.x);
        acc.y = fmaf(kk, kk, acc.y);
        acc.z = fmaf(hh * kk, w * w, acc.z);
        acc.w = fmaf(vv, vv, acc.w);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        acc.x += __shfl_xor_sync(kFullMask, acc.x, off);
        acc.y += __shfl_xor_sync(kFullMask, acc.y, off);
        acc.z += __shfl_xor_sync(kFullMask, acc.z, off);
        acc.w += __shfl_xor_sync(kFullMask, acc.w, off);
    }
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float4 t = sh[0];
        for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) {
            t.x += sh[w].x;
            t.y += sh[w].y;
            t.z += sh[w].z;
            t.w += sh[w].w;
        }
        cta_sum = t;
    }
    __syncthreads();
    cluster_wait();
    if (threadIdx.x < kCluster2) {
        const uint32_t dst = static_cast<uint32_t>(threadIdx.x);
        st_async_f4(map_to_rank(smem_addr(&slots[rank]), dst), cta_sum, map_to_rank(smem_addr(&xbar), dst));
    }
    if (!mbar_wait_cluster(&xbar, 0u) && threadIdx.x == 0) atomicOr(p.err, kErrTimeout);
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kCluster2; ++r) {
        const float4 q = slots[r];
        t.x += q.x;
        t.y += q.y;
        t.z += q.z;
        t.w += q.w;
    }
    const float inv_d = 1.0f / static_cast<float>(d);
    const float rh = rsqrtf(fmaf(t.x, inv_d, p.eps));
    const float rk = rsqrtf(fmaf(t.y, inv_d, p.eps));
    const float z = rh * rk * t.z * p.inv_sqrt_d;
    const float alpha = __fdividef(1.0f, 1.0f + __expf(-z));
    const float rv = rsqrtf(fmaf(alpha * alpha * t.w, inv_d, p.eps));

    // ---- conv, SiLU, output and the new cache row for this CTA's columns
    const uint16_t* st = p.state + static_cast<long long>(b) * p.L * d;
    uint16_t* ns = p.new_state + static_cast<long long>(b) * p.max_len * d;
    it = 0;
    for (int i = c0 + threadIdx.x; i < c0 + ncol; i += blockDim.x, ++it) {
        float vv = 0.f;
        if (it < kCache) {
#pragma unroll
            for (int q = 0; q < kCache; ++q)
                if (q == it) vv = vc[q];
        } else {
            float kk;
            kv_at(i, kk, vv);
        }
        const float vh = alpha * vv;
        const float u = vh * rv * __ldg(p.wv + i);
        float c = 0.f;
        for (int j = 0; j < p.w; ++j) {
            const int lag = (p.w - 1 - j) * p.dil;
            const float uj = lag == 0 ? u : (lag <= p.L ? bf(st, static_cast<long long>(p.L - lag) * d + i) : 0.f);
            c = fmaf(__ldg(p.cw + static_cast<long long>(j) * d + i), uj, c);
        }
        const float y = __fdividef(c, 1.0f + __expf(-c)) + vh;
        p.y[static_cast<long long>(b) * d + i] = static_cast<uint16_t>(pack_bf16x2(y, 0.f) & 0xffffu);
        ns[static_cast<long long>(p.max_len - 1) * d + i] = static_cast<uint16_t>(pack_bf16x2(u, 0.f) & 0xffffu);
    }
}

}  // namespace

int decode_proj_smem(int rows_per_split) {
    const int a = kBc * rows_per_split * 4;
    const int b = kWarps1 * kBc * 2 * 32 * 16;
    return a > b ? a : b;
}

cudaError_t decode_prepare() {
    return cudaFuncSetAttribute(decode_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
}

cudaError_t decode_launch(const DecodeParams& p, cudaStream_t s) {
    const dim3 g1(static_cast<unsigned>((p.d + kCols - 1) / kCols), static_cast<unsigned>(p.splits),
                  static_cast<unsigned>((p.B + kBc - 1) / kBc));
    cudaLaunchConfig_t cfg1 = {};
    cudaLaunchAttribute attr1[1];
    attr1[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr1[0].val.programmaticStreamSerializationAllowed = 1;
    cfg1.gridDim = g1;
    cfg1.blockDim = dim3(32 * kWarps1, 1, 1);
    cfg1.dynamicSmemBytes = static_cast<size_t>(decode_proj_smem(p.rows_per_split));
    cfg1.stream = s;
    cfg1.attrs = attr1;
    cfg1.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg1, decode_proj_kernel, p);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(p.B) * kCluster2, 1, 1);
    cfg.blockDim = dim3(kThreads2, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, decode_row_kernel, p);
}

}  // namespace eg
