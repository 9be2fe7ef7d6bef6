// Fused weight of the saved-state gate and its product rule (cuDNN Frontend
// "Engram saved-state gate", semantics paragraph: the weight is the FP32
// product of the query- and key-side normalisation weights; tile-kernels
// engram tests: fused_weight(wh, we) = wh * we in fp32, and after the
// backward grad_wh = grad_w * we, grad_we = grad_w * wh with grad_w the sum of
// the per-block partials).
//
// Forward: one thread per element; the product of two bf16 values is exact in
// fp32.  Backward: the block partials of each element are summed in a fixed
// order with error-free additions (8 warps each take a contiguous eighth of
// the blocks for 32 consecutive elements, then warp 0 merges the eight
// results in ascending order), and the product rule is applied to the total.
#include "common.cuh"
#include "engram_internal.h"

namespace eg {
namespace {

EG_DEV float bf16_at(const uint16_t* p, long long i) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(p + i)) << 16);
}

__global__ void fused_weight_kernel(const FusedWeightParams p) {
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < p.n) p.weight[i] = __fmul_rn(bf16_at(p.wh, i), bf16_at(p.we, i));
}

constexpr int kGroups = 8;

__global__ void __launch_bounds__(32 * kGroups) fused_weight_bwd_kernel(const FusedWeightParams p) {
    __shared__ float shi[kGroups][32], slo[kGroups][32];
    const int lane = threadIdx.x & 31;
    const int g = threadIdx.x >> 5;
    const long long i = static_cast<long long>(blockIdx.x) * 32 + lane;
    const long long per = (p.nblocks + kGroups - 1) / kGroups;
    const long long b0 = min(p.nblocks, g * per), b1 = min(p.nblocks, b0 + per);
    float hi = 0.f, lo = 0.f;
    if (i < p.n)
        for (long long b = b0; b < b1; ++b) cacc_add(hi, lo, __ldg(p.partial + b * p.n + i));
    shi[g][lane] = hi;
    slo[g][lane] = lo;
    __syncthreads();
    if (g == 0 && i < p.n) {
        float h = shi[0][lane], l = slo[0][lane];
#pragma unroll
        for (int k = 1; k < kGroups; ++k) cacc_merge(h, l, shi[k][lane], slo[k][lane]);
        const float gw = __fadd_rn(h, l);
        if (p.grad_w != nullptr) p.grad_w[i] = gw;
        p.grad_wh[i] = __fmul_rn(gw, bf16_at(p.we, i));
        p.grad_we[i] = __fmul_rn(gw, bf16_at(p.wh, i));
    }
}

}  // namespace

cudaError_t fused_weight_launch(const FusedWeightParams& p, cudaStream_t s) {
    fused_weight_kernel<<<static_cast<unsigned>((p.n + 255) / 256), 256, 0, s>>>(p);
    return cudaPeekAtLastError();
}

cudaError_t fused_weight_bwd_launch(const FusedWeightParams& p, cudaStream_t s) {
    fused_weight_bwd_kernel<<<static_cast<unsigned>((p.n + 31) / 32), 32 * kGroups, 0, s>>>(p);
    return cudaPeekAtLastError();
}

}  // namespace eg
