// Device-side building blocks shared by the Engram kernels (sm_103a).
//
// Every kernel here follows one pattern, "cluster row split": a token row of
// d columns is cut into C contiguous column slices, one per CTA of a thread
// block cluster.  Each CTA streams its slice of consecutive token rows into a
// ring of shared-memory stages with 1-D bulk asynchronous copies (TMA engine)
// completing on mbarriers, reduces its slice, and exchanges the per-token
// partial sums with the other CTAs of the cluster through distributed shared
// memory.  Each thread owns 8 consecutive columns (one 16-byte vector of bf16)
// of every stream of its slice for the whole kernel, so per-column weights
// live in registers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#define EG_DEV __device__ __forceinline__

namespace eg {

constexpr uint32_t kFullMask = 0xffffffffu;
constexpr uint32_t kErrTimeout = 1u;                  // sticky device error bit
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr uint32_t kWaitMaxIters = 1u << 30;

// ------------------------------------------------------------------ PTX glue

EG_DEV uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

EG_DEV unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

EG_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Makes mbarrier initialisation visible to the async proxy and the cluster.
EG_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Orders this thread's earlier generic-proxy shared accesses before later
// async-proxy (bulk copy) accesses.
EG_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

EG_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

// Same, with acquire at cluster scope: for phases completed by other CTAs'
// st.async writes into this CTA's shared memory.
EG_DEV bool mbar_try_wait_cluster(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

EG_DEV bool mbar_try_wait(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of a phase (acquire at CTA scope).
EG_DEV bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// One arrival (release at CTA scope), no transaction bytes.
EG_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Waits for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs of wall time (or kWaitMaxIters polls) and returns false; the
// caller records the failure and carries on without hanging the GPU.
EG_DEV bool mbar_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t addr = smem_addr(bar);
    if (mbar_try_wait(addr, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 0; it < kWaitMaxIters; ++it) {
        if (mbar_try_wait(addr, parity)) return true;
        if ((it & 63u) == 63u && globaltimer() - t0 > kWaitLimitNs) return false;
    }
    return false;
}

EG_DEV bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
    const uint32_t addr = smem_addr(bar);
    if (mbar_try_wait_cluster(addr, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 0; it < kWaitMaxIters; ++it) {
        if (mbar_try_wait_cluster(addr, parity)) return true;
        if ((it & 63u) == 63u && globaltimer() - t0 > kWaitLimitNs) return false;
    }
    return false;
}

// Asynchronous 8-byte store into the shared memory of a CTA of this cluster
// (addresses from map_to_rank), completing `bytes` on that CTA's mbarrier.
EG_DEV void st_async_f2(uint32_t remote_addr, float a, float b, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
            remote_addr),
        "f"(a), "f"(b), "r"(remote_bar)
        : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
EG_DEV void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst_smem)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

EG_DEV uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
EG_DEV uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
EG_DEV uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
EG_DEV uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Cluster-wide barrier with release/acquire semantics on shared memory.  Every
// thread of every CTA of the cluster must reach it (uniform control flow).
EG_DEV void cluster_sync() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::
            : "memory");
}

// Address of the same shared variable in CTA `rank` of this cluster.
EG_DEV uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

EG_DEV float2 ld_cluster_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr)
                 : "memory");
    return v;
}

EG_DEV float4 ld_cluster_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

EG_DEV float ld_cluster_f(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// Streaming 16-byte global store (evict-first in L1/L2).
EG_DEV void stg_cs(void* p, const uint4& v) {
    asm volatile("st.global.cs.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

EG_DEV void stg_f4(float* p, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}

EG_DEV uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }
EG_DEV uint2 lds64(const void* p) { return *reinterpret_cast<const uint2*>(p); }

// Streaming 8-byte global store.
EG_DEV void stg_cs8(void* p, const uint2& v) {
    asm volatile("st.global.cs.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// Streaming 8-byte global store done only where `pred` holds, as one
// predicated instruction (no branch), so that it can sit in straight-line code.
// No memory clobber: it only writes outputs that the kernel never reads.
EG_DEV void stg_cs8_if(void* p, const uint2& v, bool pred) {
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\t@q st.global.cs.v2.b32 [%0], {%1, %2};\n\t}" ::"l"(p),
        "r"(v.x), "r"(v.y), "r"(static_cast<uint32_t>(pred)));
}

// Asynchronous 4-byte store into the shared memory of a CTA of this cluster,
// completing 4 bytes on that CTA's mbarrier.
EG_DEV void st_async_f32(uint32_t remote_addr, float a, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(remote_addr),
        "f"(a), "r"(remote_bar)
        : "memory");
}

// ------------------------------------------------------------------ bf16

EG_DEV float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
EG_DEV float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

EG_DEV void unpack8(const uint4& q, float (&f)[8]) {
    f[0] = bf_lo(q.x);
    f[1] = bf_hi(q.x);
    f[2] = bf_lo(q.y);
    f[3] = bf_hi(q.y);
    f[4] = bf_lo(q.z);
    f[5] = bf_hi(q.z);
    f[6] = bf_lo(q.w);
    f[7] = bf_hi(q.w);
}

EG_DEV void unpack4(const uint2& q, float (&f)[4]) {
    f[0] = bf_lo(q.x);
    f[1] = bf_hi(q.x);
    f[2] = bf_lo(q.y);
    f[3] = bf_hi(q.y);
}

// Two fp32 values -> packed bf16x2, round-to-nearest-even (lo in the low half).
EG_DEV uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

EG_DEV uint2 pack4(const float (&f)[4]) {
    return make_uint2(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]));
}

EG_DEV uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// ------------------------------------------------------- packed fp32 pairs
// Blackwell executes two fp32 lanes per instruction on float2 operands.
EG_DEV float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
EG_DEV float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
EG_DEV float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
// a - b with one rounding (b * -1 + a)
EG_DEV float2 sub2(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.f, -1.f), a); }
EG_DEV float2 splat2(float a) { return make_float2(a, a); }
EG_DEV float2 bf2(uint32_t u) { return make_float2(bf_lo(u), bf_hi(u)); }
EG_DEV uint32_t pack2(float2 v) { return pack_bf16x2(v.x, v.y); }

// TwoSum on both lanes: s + e == a + b exactly, lane by lane.
EG_DEV void two_sum2(float2 a, float2 b, float2& s, float2& e) {
    s = add2(a, b);
    const float2 bb = sub2(s, a);
    const float2 aa = sub2(s, bb);
    e = add2(sub2(a, aa), sub2(b, bb));
}

// (hi, lo) += a * b on both lanes, product and sum errors kept in lo.
EG_DEV void cacc_prod_x2(float2& hi, float2& lo, float2 a, float2 b) {
    const float2 t = mul2(a, b);
    const float2 pe = fma2(a, b, make_float2(-t.x, -t.y));
    float2 s, e;
    two_sum2(hi, t, s, e);
    hi = s;
    lo = add2(lo, add2(e, pe));
}

// (hi, lo) += t on both lanes.
EG_DEV void cacc_add_x2(float2& hi, float2& lo, float2 t) {
    float2 s, e;
    two_sum2(hi, t, s, e);
    hi = s;
    lo = add2(lo, e);
}

// (hi, lo) += (ah + al) * b on both lanes, ah + al a double-float factor.
EG_DEV void cacc_prod2_x2(float2& hi, float2& lo, float2 ah, float2 al, float2 b) {
    const float2 t = mul2(ah, b);
    float2 pe = fma2(ah, b, make_float2(-t.x, -t.y));
    pe = fma2(al, b, pe);
    float2 s, e;
    two_sum2(hi, t, s, e);
    hi = s;
    lo = add2(lo, add2(e, pe));
}

// ------------------------------------------------- error-free transformations
// Knuth's TwoSum: s + e == a + b exactly.  Explicit _rn intrinsics keep the
// compiler from contracting or reassociating these operations.
EG_DEV void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float aa = __fsub_rn(s, bb);
    e = __fadd_rn(__fsub_rn(a, aa), __fsub_rn(b, bb));
}

// (hi, lo) += t with the rounding error of the addition kept in lo.
EG_DEV void cacc_add(float& hi, float& lo, float t) {
    float s, e;
    two_sum(hi, t, s, e);
    hi = s;
    lo = __fadd_rn(lo, e);
}

// (hi, lo) += a * b with both the product's and the sum's rounding errors
// kept in lo (the product error is exact via FMA).
EG_DEV void cacc_prod(float& hi, float& lo, float a, float b) {
    const float t = __fmul_rn(a, b);
    const float pe = __fmaf_rn(a, b, -t);
    float s, e;
    two_sum(hi, t, s, e);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(e, pe));
}

// (hi, lo) += (ah + al) * b, with ah + al an unevaluated double-float factor.
EG_DEV void cacc_prod2(float& hi, float& lo, float ah, float al, float b) {
    const float t = __fmul_rn(ah, b);
    float pe = __fmaf_rn(ah, b, -t);
    pe = __fmaf_rn(al, b, pe);
    float s, e;
    two_sum(hi, t, s, e);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(e, pe));
}

// (hi, lo) += (hi2, lo2)
EG_DEV void cacc_merge(float& hi, float& lo, float hi2, float lo2) {
    float s, e;
    two_sum(hi, hi2, s, e);
    hi = s;
    lo = __fadd_rn(__fadd_rn(lo, lo2), e);
}

}  // namespace eg
