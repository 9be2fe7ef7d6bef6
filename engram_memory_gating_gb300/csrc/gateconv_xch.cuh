// Shared-memory layout and cluster exchange of the GateConv kernels.
//
// A GateConv token row is cut into C column slices, one per CTA of a thread
// block cluster; each thread owns 4 consecutive columns of its CTA's slice.
// The per-token quantities both kernels need (RMS statistics, the gate logit,
// the gradient sums of the backward) are sums over the whole row, so each CTA
// forms partial sums over its slice and the cluster exchanges them.  Tokens go
// in chunks of kChunk: every warp reduces the 4 x kChunk partial sums of a
// chunk across its lanes and writes them into a slot of every CTA of the
// cluster with asynchronous remote stores (st.async) that complete on that
// CTA's exchange mbarrier.  A CTA reads the totals of chunk c - 1 only after
// it has finished the row work of chunk c, so the exchange latency overlaps a
// chunk of work and no cluster-wide barrier runs inside the token loop.
//
// Two slot buffers suffice: a CTA writes chunk c + 1 into a peer only after it
// has received chunk c from every warp of that peer, and every warp reads
// chunk c - 1 before it sends chunk c.
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

// Byte offsets in dynamic shared memory.
constexpr int kOffFull = 0;    // [kStages] stage mbarriers
constexpr int kOffXbar = 128;  // [2] exchange mbarriers
constexpr int kOffRel = 192;   // [kStages] per-stage release counters
constexpr int kOffXch = 256;   // [2][parts][kVals] fp32 exchange slots

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

// Sends this warp's chunk totals (value l >> 1 in lane l) into slot `part` of
// buffer `buf` of every CTA of the cluster; lanes l and l ^ 1 split the CTAs.
EG_DEV void xch_send(float* xch, uint64_t* xbar, int buf, int parts, int part, float val, int lane,
                     uint32_t C) {
    const uint32_t dst = smem_addr(xch + (buf * parts + part) * kVals + (lane >> 1));
    const uint32_t bar = smem_addr(xbar + buf);
    for (uint32_t rr = static_cast<uint32_t>(lane & 1); rr < C; rr += 2)
        st_async_f32(map_to_rank(dst, rr), val, map_to_rank(bar, rr));
}

// Total over all parts of value (lane & 15) of buffer `buf`, in a fixed order
// (even parts, odd parts, then their sum), the same in every warp.
EG_DEV float xch_total(const float* xch, int buf, int parts, int lane) {
    const float* s = xch + buf * parts * kVals + (lane & 15);
    float acc = 0.f;
    for (int p = lane >> 4; p < parts; p += 2) acc += s[p * kVals];
    return acc + __shfl_xor_sync(kFullMask, acc, 16);
}

}  // namespace gc
}  // namespace eg
