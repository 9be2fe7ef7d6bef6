// Constants and warp-level pieces shared by the GateConv kernels.
//
// A GateConv token row is cut into C column slices, one per CTA of a thread
// block cluster; each thread owns 4 consecutive columns of its CTA's slice.
// The per-token quantities both kernels need (RMS statistics, the gate logit,
// the gradient sums of the backward) are sums over the whole row, so each CTA
// forms partial sums over its slice and the cluster exchanges them, per chunk
// of kChunk tokens.  Every warp reduces the 4 x kChunk partial sums of a
// chunk across its lanes (warp_reduce16) and leaves them in shared memory;
// the last warp of the CTA to hand in adds the warps' totals in warp order
// and sends the CTA total into slot `rank` of every CTA of the cluster with
// asynchronous remote stores (st.async) that complete on that CTA's exchange
// mbarrier.  A receiver adds the C slots in rank order, so every CTA forms
// the same total.  The kernels read the totals of chunk c - 1 only after the
// row work of chunk c, so the exchange overlaps a chunk of work and no
// cluster-wide barrier runs inside the token loop.
#pragma once

#include "common.cuh"

namespace eg {
namespace gc {

// e^-x and 1/x on the special-function unit with the .ftz forms of the PTX
// approximate instructions (subnormal inputs and results flushed to zero,
// which spares the extra handling of the plain forms): e^-x = 2^(-x log2 e)
// by ex2.approx.ftz.f32, 1/x by rcp.approx.ftz.f32 (each about 2^-22
// relative error, PTX ISA).  Used only where a subnormal cannot matter: in
// 1 / (1 + e^-x) the denominator is at least 1, and an exponential that
// underflows only saturates the sigmoid.
EG_DEV float exp_neg_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x * -1.44269504f));
    return y;
}
EG_DEV float rcp_ftz(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr int kChunk = 4;         // tokens per exchange
constexpr int kVals = 4 * kChunk; // partial sums per warp and chunk
constexpr int kThreads = 256;     // threads per CTA (4 columns each)
constexpr int kStages = 16;       // ring stages (one token each)

// Sum of 16 values over the 32 lanes of a warp (reduce-scatter): lane l ends
// with the warp total of value l >> 1 (lanes l and l ^ 1 hold the same total).
EG_DEV float warp_reduce16(const float (&v)[16], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
    float a[8], b[4], c[2];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float keep = b4 ? v[8 + i] : v[i];
        const float send = b4 ? v[i] : v[8 + i];
        a[i] = keep + __shfl_xor_sync(kFullMask, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float keep = b3 ? a[4 + i] : a[i];
        const float send = b3 ? a[i] : a[4 + i];
        b[i] = keep + __shfl_xor_sync(kFullMask, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float keep = b2 ? b[2 + i] : b[i];
        const float send = b2 ? b[i] : b[2 + i];
        c[i] = keep + __shfl_xor_sync(kFullMask, send, 4);
    }
    const float e = (b1 ? c[1] : c[0]) + __shfl_xor_sync(kFullMask, b1 ? c[0] : c[1], 2);
    return e + __shfl_xor_sync(kFullMask, e, 1);
}

}  // namespace gc
}  // namespace eg
