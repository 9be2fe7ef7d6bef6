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
// Two kernels, each a single short chain of dependent memory round trips:
//  1 (projection): a CTA owns a 32-column tile of d and up to 8 batch rows,
//    over all d_mem rows, so its k and v are final (no split partials).  The
//    tile's weight rows arrive by 2-D TMA (16 KB boxes of 256 rows x 32
//    columns, which the copy engine gathers from the 64-byte row segments)
//    and the matching e values by cp.async, into a ring of four stages of 256
//    rows, all issued up front for d_mem <= 1024.  The sums run on mma.sync
//    (the batch of 8 is the n of an m16n8k16 product; the work is a pass over
//    the weights, so this only cuts the instruction count): eight warps each
//    take 32 rows of a stage, then add their sums in warp order.  The CTA
//    writes its v to the workspace together with the
//    tile's four row sums per batch row (sum h^2, sum k^2, sum h k w_h^2,
//    sum v^2; k is needed only there), and also shifts the cache by one token
//    (independent work).
//  2 (output): a CTA per (batch row, 256-column block).  It loads its inputs
//    that do not depend on kernel 1 (w_v, the conv taps, the cached u of each
//    tap) before it waits for kernel 1's grid, then adds the tiles' row sums
//    in a fixed tree (every thread loads some, warp butterflies, the warp
//    totals in warp order), forms the scalars and writes y and the new cache
//    row.
#include "common.cuh"
#include "engram_internal.h"

namespace eg {
namespace {

// Programmatic dependent launch: each kernel waits for the preceding kernel of
// the stream (griddepcontrol.wait) before it reads anything that kernel may
// write, and only then lets its successor be scheduled.
EG_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
EG_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

EG_DEV void cp_async16(void* smem_dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(src) : "memory");
}
EG_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
EG_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// waits until at most n (0 <= n <= 15) of this thread's most recent groups are pending
EG_DEV void cp_async_wait_n(int n) {
    switch (n) {
        case 0: cp_async_wait<0>(); break;
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        case 5: cp_async_wait<5>(); break;
        case 6: cp_async_wait<6>(); break;
        case 7: cp_async_wait<7>(); break;
        case 8: cp_async_wait<8>(); break;
        case 9: cp_async_wait<9>(); break;
        case 10: cp_async_wait<10>(); break;
        case 11: cp_async_wait<11>(); break;
        case 12: cp_async_wait<12>(); break;
        case 13: cp_async_wait<13>(); break;
        case 14: cp_async_wait<14>(); break;
        default: cp_async_wait<15>(); break;
    }
}

constexpr int kTile = 32;          // columns per projection CTA, of each of W_K and W_V
constexpr int kBc = 8;             // batch rows per projection CTA (the mma's n)
constexpr int kWarps1 = 8;         // one per batch row in the row sums
constexpr int kChunkRows = 256;    // weight rows per ring stage (the TMA box height)
constexpr int kRing = 4;           // ring stages
constexpr int kRowsPerWarp = kChunkRows / kWarps1;     // 32 rows: two k-steps of 16
// one stage: [2 matrices][256 rows][32 columns] bf16 (two TMA boxes, 64-byte
// rows in the 64-byte swizzle), then [8 batch][256 rows] bf16 of e at a row
// pitch of 528 bytes (the 8 rows of an ldmatrix land on distinct banks)
constexpr int kBoxBytes = kChunkRows * kTile * 2;     // 16 KB
constexpr int kWBytes = 2 * kBoxBytes;
constexpr int kEPitch = kChunkRows * 2 + 16;
constexpr int kEBytes = kBc * kEPitch;
constexpr int kStageB = (kWBytes + kEBytes + 1023) / 1024 * 1024;
constexpr int kOffBar = 0;                             // [kRing] stage mbarriers
constexpr int kOffRing = 1024;
constexpr int kOffRed = kOffRing + kRing * kStageB;    // [8 warps][2][8 batch][32] fp32
constexpr int kOffKv = kOffRed + kWarps1 * 2 * kBc * kTile * 4;  // [2][8 batch][32] final k, v of the tile
constexpr int kSmem1 = kOffKv + 2 * kBc * kTile * 4 + 1024;     // + the alignment of the base to 1024
static_assert(kSmem1 <= 227 * 1024, "projection shared memory");
static_assert(kRowsPerWarp == 32 && kWarps1 == kBc, "two k-steps per warp and stage; a warp per batch row");

// 2-D TMA load of box (x, y) of a tensor map into shared memory, completing on `bar`
EG_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// four 8x8 b16 matrices from shared memory (lanes 8i..8i+7 give the row
// addresses of matrix i); .trans hands each thread a column pair instead of a row pair
EG_DEV void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
EG_DEV void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
// D (16x8 fp32) += A (16x16 bf16, row) B (16x8 bf16, col)
EG_DEV void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// the cache shift for 16-byte chunks [q0, q1): row r < max_len - 1 of the new
// cache is row r + 1 of the left-padded old one (I: the index type, 32-bit
// whenever the chunk count fits)
template <typename I>
EG_DEV void shift_cache(const DecodeParams& p, I q0, I q1, I tid, I nthreads) {
    const I pad = p.max_len - p.L;
    const I per_row = p.d / 8, per_b = static_cast<I>(p.max_len - 1) * per_row;
    for (I q = q0 + tid; q < q1; q += nthreads) {
        const I bb = q / per_b, rem = q - bb * per_b;
        const I r = rem / per_row, i = (rem - r * per_row) * 8;
        const I src = r + 1 - pad;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (src >= 0 && src < p.L)
            val = __ldg(reinterpret_cast<const uint4*>(p.state + (static_cast<long long>(bb) * p.L + src) * p.d + i));
        *reinterpret_cast<uint4*>(p.new_state + (static_cast<long long>(bb) * p.max_len + r) * p.d + i) = val;
    }
}

// Kernel 1: CTA (x: chunk of 8 batch rows, y: 32-column tile).  The weight
// boxes come by TMA (the tensor maps cover (d_mem, d) row-major; rows past
// d_mem read as zero), e by cp.async.  The contraction runs on mma.sync
// m16n8k16: m = 16 output columns, n = the 8 batch rows, k = 16 rows of d_mem;
// warp w takes rows [32w, 32w + 32) of every stage for all four 16-column
// blocks (k and v, two each).
__global__ void __launch_bounds__(32 * kWarps1, 1) decode_proj_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ __align__(128) unsigned char sm_raw[];
    // the 64-byte swizzle is a function of the shared address: base at 1024
    unsigned char* sm = sm_raw + ((1024u - (smem_addr(sm_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile = blockIdx.y;
    const int ntiles = gridDim.y;
    const int c0 = tile * kTile;
    const int b0 = blockIdx.x * kBc;
    const int nb = min(kBc, p.B - b0);
    const int nchunk = (p.dmem + kChunkRows - 1) / kChunkRows;

    // inputs only: h and w_h of this warp's batch row and lane's column (row sums)
    const int hb = warp;
    const float hval = hb < nb ? __uint_as_float(static_cast<uint32_t>(__ldg(p.h + static_cast<long long>(b0 + hb) * p.d + c0 + lane)) << 16) : 0.f;
    const float whv = __ldg(p.wh + c0 + lane);
    if (tid == 0) {
        for (int i = 0; i < kRing; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    // chunk k of the weight rows (and of e) into ring stage k % kRing
    auto issue = [&](int k) {
        unsigned char* st = sm + kOffRing + (k % kRing) * kStageB;
        const int m0 = k * kChunkRows;
        if (tid == 0) {
            uint64_t* bar = &bars[k % kRing];
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kWBytes));
            tma_load_2d(st, &p.tmk, c0, m0, bar);
            tma_load_2d(st + kBoxBytes, &p.tmv, c0, m0, bar);
        }
        // e: 8 batch rows x 256 values as bf16, [batch][row] (a 16-byte copy
        // holds 8 consecutive values of one batch row); d_mem is a multiple of 8
        {
            const int b = tid >> 5, part = tid & 31;
            unsigned char* dst = st + kWBytes + b * kEPitch + part * 16;
            const int m = m0 + part * 8;
            if (b < nb && m < p.dmem)
                cp_async16(dst, p.e + static_cast<long long>(b0 + b) * p.dmem + m);
            else
                *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
        cp_async_commit();
    };
    __syncthreads();   // the barriers exist before any copy completes on them
    grid_dep_wait();
    grid_dep_launch();
    const int pro = nchunk < kRing ? nchunk : kRing;
    for (int k = 0; k < pro; ++k) issue(k);

    // the cache shift (independent of the projection), spread over all CTAs
    {
        const long long nq = static_cast<long long>(p.B) * (p.max_len - 1) * (p.d / 8);  // 16-byte chunks
        const long long ncta = static_cast<long long>(gridDim.x) * gridDim.y;
        const long long cta = static_cast<long long>(blockIdx.x) * gridDim.y + blockIdx.y;
        const long long q0 = nq * cta / ncta, q1 = nq * (cta + 1) / ncta;
        if (nq <= 0x7fffffffLL)
            shift_cache<int>(p, static_cast<int>(q0), static_cast<int>(q1), tid, blockDim.x);
        else
            shift_cache<long long>(p, q0, q1, tid, blockDim.x);
    }

    float acc[4][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[mt][j] = 0.f;
    // ldmatrix row of this lane: B (e, [n][k]) matrix lane >> 3 = k-step
    // half lane >> 4, k offset 8 (lane >> 3 & 1); A (weights, [k][m]) row k =
    // lane & 7 (+ 8 for lanes 16..31), 8-column chunk (lane >> 3) & 1
    const int kr = warp * kRowsPerWarp;
    const uint32_t e_off = static_cast<uint32_t>((lane & 7) * kEPitch + (kr + (lane >> 3) * 8) * 2);
    const int ka = (lane & 7) + ((lane >> 4) << 3);
    const int ca = (lane >> 3) & 1;
    bool failed = false;
    for (int k = 0; k < nchunk; ++k) {
        // chunk k's e has landed once no more than the groups committed after
        // it (chunks k + 1 .. min(nchunk, k + kRing) - 1) are pending; its
        // weights once its stage barrier completes
        cp_async_wait_n(min(nchunk - 1 - k, kRing - 1));
        if (!failed && !mbar_wait(&bars[k % kRing], static_cast<uint32_t>((k / kRing) & 1))) failed = true;
        __syncthreads();
        const uint32_t sA = smem_addr(sm + kOffRing + (k % kRing) * kStageB);
        uint32_t bf[4];
        ldsm_x4(bf, sA + kWBytes + e_off);
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const int kk = kr + ks * 16 + ka;                 // row of the stage
            const uint32_t row = sA + static_cast<uint32_t>(kk * (kTile * 2));
            const int sw = (kk >> 1) & 3;                     // 64-byte swizzle of this row
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const int c = ((mt & 1) << 1) + ca;           // 16-byte chunk of the 64-byte row
                uint32_t af[4];
                ldsm_x4_trans(af, row + (mt >> 1) * kBoxBytes + ((c ^ sw) << 4));
                mma_16816(acc[mt], af, bf[2 * ks], bf[2 * ks + 1]);
            }
        }
        if (k + kRing < nchunk) {
            __syncthreads();   // every warp is done with stage k % kRing
            fence_proxy_async();
            issue(k + kRing);
        }
    }
    if (failed) atomicOr(p.err, kErrTimeout);
    // the warps' sums, in warp order; accumulator (mt, j): column
    // 16 (mt & 1) + lane / 4 (+ 8 for j >= 2), batch row 2 (lane % 4) + (j & 1)
    float* red = reinterpret_cast<float*>(sm + kOffRed);    // [warp][mat][batch][32 columns]
    {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = ((mt & 1) << 4) + g + ((j >> 1) << 3);
                const int bb = 2 * t + (j & 1);
                red[((warp * 2 + (mt >> 1)) * kBc + bb) * kTile + col] = acc[mt][j];
            }
    }
    __syncthreads();
    float* kv = reinterpret_cast<float*>(sm + kOffKv);      // [mat][batch][32]
    for (int i = tid; i < 2 * kBc * kTile; i += blockDim.x) {
        float s = red[i];
#pragma unroll
        for (int w = 1; w < kWarps1; ++w) s += red[w * 2 * kBc * kTile + i];
        kv[i] = s;
        // v goes to the workspace for kernel 2 (k enters it only through the row sums)
        const int m2 = i / (kBc * kTile), b = (i / kTile) % kBc, col = i % kTile;
        if (m2 == 1 && b < nb) p.vbuf[static_cast<long long>(b0 + b) * p.d + c0 + col] = s;
    }
    __syncthreads();
    // the tile's row sums: warp = batch row, lane = column
    if (hb < nb) {
        const float kk = kv[hb * kTile + lane];
        const float vv = kv[(kBc + hb) * kTile + lane];
        float4 a = make_float4(hval * hval, kk * kk, hval * kk * (whv * whv), vv * vv);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            a.x += __shfl_xor_sync(kFullMask, a.x, off);
            a.y += __shfl_xor_sync(kFullMask, a.y, off);
            a.z += __shfl_xor_sync(kFullMask, a.z, off);
            a.w += __shfl_xor_sync(kFullMask, a.w, off);
        }
        if (lane == 0)
            *reinterpret_cast<float4*>(p.stats + (static_cast<long long>(b0 + hb) * ntiles + tile) * 4) = a;
    }
}

constexpr int kThreads2 = 256;
constexpr int kMaxTaps2 = 8;   // taps whose cached u is loaded before the grid wait

// Kernel 2: CTA (x: batch row, y: 256-column block).
__global__ void __launch_bounds__(kThreads2) decode_row_kernel(const __grid_constant__ DecodeParams p) {
    __shared__ float4 red[kThreads2 / 32];
    const int b = blockIdx.x;
    const int d = p.d;
    const int i = blockIdx.y * kThreads2 + threadIdx.x;
    const bool ok = i < d;
    const int ntiles = d / kTile;
    // inputs only, before the wait: w_v, the taps and the cached u of each tap
    const uint16_t* st = p.state + static_cast<long long>(b) * p.L * d;
    float wv = 0.f, cwv[kMaxTaps2], uj[kMaxTaps2];
#pragma unroll
    for (int j = 0; j < kMaxTaps2; ++j) {
        cwv[j] = 0.f;
        uj[j] = 0.f;
        if (ok && j < p.w) {
            const int lag = (p.w - 1 - j) * p.dil;
            cwv[j] = __ldg(p.cw + static_cast<long long>(j) * d + i);
            if (lag > 0 && lag <= p.L)
                uj[j] = __uint_as_float(static_cast<uint32_t>(__ldg(st + static_cast<long long>(p.L - lag) * d + i)) << 16);
        }
    }
    if (ok) wv = __ldg(p.wv + i);
    grid_dep_wait();
    grid_dep_launch();   // the next decode step's projection may be scheduled (it waits for this grid)
    const float vv = ok ? __ldcg(p.vbuf + static_cast<long long>(b) * d + i) : 0.f;
    // the row sums of batch row b: thread j loads the sums of tiles j, j + 256,
    // ... (one L2 round trip for d <= 8192), a butterfly adds them within each
    // warp, then every thread adds the eight warp totals in warp order
    {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int t = threadIdx.x; t < ntiles; t += kThreads2) {
            const float4 q = __ldcg(reinterpret_cast<const float4*>(p.stats + (static_cast<long long>(b) * ntiles + t) * 4));
            a.x += q.x;
            a.y += q.y;
            a.z += q.z;
            a.w += q.w;
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            a.x += __shfl_xor_sync(kFullMask, a.x, off);
            a.y += __shfl_xor_sync(kFullMask, a.y, off);
            a.z += __shfl_xor_sync(kFullMask, a.z, off);
            a.w += __shfl_xor_sync(kFullMask, a.w, off);
        }
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
    }
    __syncthreads();
    float4 tsum = red[0];
#pragma unroll
    for (int w = 1; w < kThreads2 / 32; ++w) {
        tsum.x += red[w].x;
        tsum.y += red[w].y;
        tsum.z += red[w].z;
        tsum.w += red[w].w;
    }
    const float inv_d = 1.0f / static_cast<float>(d);
    const float rh = rsqrtf(fmaf(tsum.x, inv_d, p.eps));
    const float rk = rsqrtf(fmaf(tsum.y, inv_d, p.eps));
    const float z = rh * rk * tsum.z * p.inv_sqrt_d;
    const float alpha = __fdividef(1.0f, 1.0f + __expf(-z));
    const float rv = rsqrtf(fmaf(alpha * alpha * tsum.w, inv_d, p.eps));
    if (!ok) return;
    const float vh = alpha * vv;
    const float u = vh * rv * wv;
    float c = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTaps2; ++j)
        if (j < p.w) c = fmaf(cwv[j], (p.w - 1 - j) * p.dil == 0 ? u : uj[j], c);
    for (int j = kMaxTaps2; j < p.w; ++j) {   // taps beyond those loaded early
        const int lag = (p.w - 1 - j) * p.dil;
        const float u2 = lag == 0 ? u
                                  : (lag <= p.L ? __uint_as_float(static_cast<uint32_t>(__ldg(st + static_cast<long long>(p.L - lag) * d + i)) << 16)
                                                : 0.f);
        c = fmaf(__ldg(p.cw + static_cast<long long>(j) * d + i), u2, c);
    }
    const float y = __fdividef(c, 1.0f + __expf(-c)) + vh;
    p.y[static_cast<long long>(b) * d + i] = static_cast<uint16_t>(pack_bf16x2(y, 0.f) & 0xffffu);
    p.new_state[(static_cast<long long>(b) * p.max_len + p.max_len - 1) * d + i] =
        static_cast<uint16_t>(pack_bf16x2(u, 0.f) & 0xffffu);
}

}  // namespace

cudaError_t decode_prepare() {
    return cudaFuncSetAttribute(decode_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem1);
}

cudaError_t decode_launch(const DecodeParams& p, cudaStream_t s) {
    cudaLaunchConfig_t cfg1 = {};
    cudaLaunchAttribute attr1[1];
    attr1[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr1[0].val.programmaticStreamSerializationAllowed = 1;
    cfg1.gridDim = dim3(static_cast<unsigned>((p.B + kBc - 1) / kBc), static_cast<unsigned>(p.d / kTile), 1);
    cfg1.blockDim = dim3(32 * kWarps1, 1, 1);
    cfg1.dynamicSmemBytes = kSmem1;
    cfg1.stream = s;
    cfg1.attrs = attr1;
    cfg1.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg1, decode_proj_kernel, p);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(p.B), static_cast<unsigned>((p.d + kThreads2 - 1) / kThreads2), 1);
    cfg.blockDim = dim3(kThreads2, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_row_kernel, p);
}

}  // namespace eg
