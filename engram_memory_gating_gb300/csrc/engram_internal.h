// Host-side interface between the C ABI layer (engram_abi.cu) and the kernel
// translation units.  Plain structs of device pointers and sizes.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace eg {

// Smallest cluster size C (1..8) that cuts the d/8 column groups of a row into
// equal slices of at most `max_groups` groups; 0 if none does.
int pick_cluster(int64_t d, int max_groups);

// Shared-memory layout common to the row-split kernels: mbarriers (ring
// stages, then the two exchange slots), per-warp partials (two buffers), the
// cluster exchange slots (2 x 8 ranks x 16 floats), then the ring of stages.
constexpr int kMaxStages = 16;
constexpr int kSmemBarOff = 0;                         // 16 stage ("full") mbarriers
constexpr int kSmemRxBarOff = kMaxStages * 8;          // 4 exchange mbarriers
constexpr int kSmemEmptyBarOff = kSmemRxBarOff + 4 * 8;  // 16 stage-release mbarriers
constexpr int kRedWarps = 8;                           // per-warp partial buffers
constexpr int kSmemRedOff = 512;                       // 2 x 8 warps x 16 floats
constexpr int kSmemXchOff = kSmemRedOff + 2 * kRedWarps * 16 * 4;  // exchange slots
constexpr int kXchSlots = 4;                           // tokens in flight per exchange
constexpr int kXchMaxParts = 20;                       // cluster CTAs x warps per token
constexpr int kSmemCoefOff = kSmemXchOff + kXchSlots * kXchMaxParts * 16 * 4;
constexpr int kSmemRingOff = kSmemCoefOff + 2 * 32 * 4;     // 128-byte aligned
static_assert(kSmemEmptyBarOff + kMaxStages * 8 <= kSmemRedOff, "barrier area");
static_assert(kSmemRingOff % 128 == 0, "ring alignment");

struct GateFwdParams {
    const uint16_t* x;
    const uint16_t* kv;
    const float* w;
    const uint8_t* mask;
    uint16_t* out;
    float* saved;
    unsigned int* err;
    long long N;
    int d;        // hidden size of one stream
    int ncols;    // columns per CTA slice
    int ngroups;  // 8-column groups per CTA slice (<= threads)
    int stages;
    float eps;
};

struct GateBwdParams {
    const uint16_t* x;
    const uint16_t* kv;
    const float* w;
    const float* saved;
    const uint16_t* gout;
    uint16_t* gx;
    uint16_t* gkv;
    float* coef;     // (N, 4, 4) fp32 per-token scalars: A hi, A lo, -B, -Ck
    float* partial;  // (N/64, 4, d) fp32 slots for per-group grad_weight
    unsigned int* err;
    long long N;
    int d;
    int ncols;        // columns per CTA slice
    int ngroups;      // 8-column groups per slice (<= threads)
    int stages;
    int group_tokens; // tokens per token group (one grad_weight partial each)
    int pair_slots;   // 1: group g writes (hi, lo) to slots 2g, 2g+1
};

struct GateWReduceParams {
    const float* partial;  // partial[b * stride + i], b < nblocks, i < n (fp32)
    float* out;            // (n)
    int nblocks;
    int n;
    int stride;
    int pairs;  // slots come as (hi, lo) pairs
};

struct GateConvFwdParams {
    const uint16_t* H;
    const uint16_t* k;
    const uint16_t* v;
    const float* wh;
    const float* wv;
    const float* cw;
    uint16_t* Y;
    uint16_t* vhat;
    float* alpha;
    float* rh;
    float* rk;
    float* rv;
    unsigned int* err;
    int M, T, d;
    int ncols, ngroups, stages;
    int range_len;       // tokens per range (last range of a row may be shorter)
    int ranges_per_row;
    float eps;
    float inv_sqrt_d;
};

struct GateConvBwdParams {
    const uint16_t* dY;
    const uint16_t* H;
    const uint16_t* k;
    const uint16_t* v;
    const float* wh;
    const float* wv;
    const float* cw;
    const uint16_t* vhat;
    const float* alpha;
    const float* rh;
    const float* rk;
    const float* rv;
    uint16_t* dH;
    uint16_t* dk;
    uint16_t* dv;
    float* partial;  // (ranges, 6, d): dwh, dwv, dcw[0..3]
    unsigned int* err;
    int M, T, d;
    int ncols, ngroups, stages;
    int range_len;
    int ranges_per_row;
    float eps;
    float inv_sqrt_d;
};

struct LaunchCfg {
    int cluster;
    int threads;
    int clusters;   // grid size in clusters (CTAs when cluster == 1)
    int stages;
    int smem;
    int grid_y;     // second grid dimension (1 unless stated)
    int aux_blocks; // CTAs of a preceding helper kernel, if any
};

// Kernel launchers (defined next to their kernels).  Each returns the launch
// status; none synchronises.
cudaError_t gate_fwd_prepare(int smem_bytes);
cudaError_t gate_fwd_max_clusters(int cluster, int threads, int smem, int* out);
cudaError_t gate_fwd_launch(const GateFwdParams& p, const LaunchCfg& c, cudaStream_t s);

cudaError_t gate_bwd_prepare(int smem_bytes);
cudaError_t gate_bwd_max_clusters(int cluster, int threads, int smem, int* out);
cudaError_t gate_bwd_launch(const GateBwdParams& p, const LaunchCfg& c, cudaStream_t s);
cudaError_t gate_wreduce_launch(const GateWReduceParams& p, cudaStream_t s);

cudaError_t gateconv_fwd_prepare(int smem_bytes);
cudaError_t gateconv_fwd_max_clusters(int cluster, int threads, int smem, int* out);
cudaError_t gateconv_fwd_launch(const GateConvFwdParams& p, const LaunchCfg& c, cudaStream_t s);

cudaError_t gateconv_bwd_prepare(int smem_bytes);
cudaError_t gateconv_bwd_max_clusters(int cluster, int threads, int smem, int* out);
cudaError_t gateconv_bwd_launch(const GateConvBwdParams& p, const LaunchCfg& c, cudaStream_t s);
cudaError_t gateconv_wreduce_launch(const GateWReduceParams& p, cudaStream_t s);

}  // namespace eg
