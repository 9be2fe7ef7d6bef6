// Host-side interface between the C ABI layer (engram_abi.cu) and the kernel
// translation units.  Plain structs of device pointers and sizes.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace eg {

// Hidden size of the saved-state gate's packed-KV entry points.
constexpr int kGateHidden = 5120;

// Largest number of ring stages any kernel uses (mbarrier area sizing).
constexpr int kMaxStages = 16;

// GateConv backward: longest token range (its saved scalars are staged in
// shared memory, 16 bytes a token, with up to 8 halo tokens).
constexpr int kGcBwdMaxRange = 1024;

// Largest token group of the backward's elementwise kernel: its per-token
// scalars (64 bytes a token) and zero flags are staged in shared memory.
constexpr int kGateBwdTableTokens = 256;

// Saved-state gate.  Row (n, s) of X is x + (n*4 + s)*d; the key row is
// key + n*key_ts + s*d and the shared value row v + n*v_ts (packed KV:
// key = kv, key_ts = 5d, v = kv + 4d, v_ts = 5d).  Saved state: packed
// (gate, dot, rstd_X, rstd_key) records `saved` (N, 4, 4), or four separate
// (N, 4) arrays sv_gate, sv_dot, sv_rx, sv_rk.
struct GateFwdParams {
    const uint16_t* x;
    const uint16_t* key;
    const uint16_t* v;
    long long key_ts, v_ts;
    const float* w;
    const uint8_t* mask;
    uint16_t* out;
    float* saved;
    float *sv_gate, *sv_dot, *sv_rx, *sv_rk;
    unsigned int* err;
    long long N;
    int d;
    int packed;   // 1: packed KV and saved records, d = 5120 (compile-time kernel)
    float eps;
    float clamp;
};

struct GateBwdParams {
    const uint16_t* x;
    const uint16_t* key;
    const uint16_t* v;
    long long key_ts, v_ts;
    const float* w;
    const float* saved;        // packed records, or null with the four arrays below
    const float *sv_gate, *sv_dot, *sv_rx, *sv_rk;
    const uint16_t* gout;
    uint16_t* gx;
    uint16_t* gkey;            // grad of key row (n, s) at gkey + n*gkey_ts + s*d
    uint16_t* gv;              // grad of the shared value row n at gv + n*gv_ts
    long long gkey_ts, gv_ts;
    float* coef;     // (N, 4, 4) fp32 per-token scalars: A hi, A lo, -B, -Ck
    float* partial;  // grad_weight slots (4, d) fp32 each
    uint16_t* partial_lo;  // one-pass backward: the low words of its (hi, lo) pairs, bf16 (4, d) each
    unsigned int* err;
    long long N;
    int d;
    int ncols;        // columns per CTA slice (the last slice may be shorter)
    int stages;
    int group_tokens; // tokens per token group (one grad_weight partial each)
    int pair_slots;   // 1: group g writes (hi, lo) to slots 2g, 2g+1
    int token_split;  // 1: a CTA's warps all cover its 64 columns and split its group's tokens
    int packed;       // 1: packed KV / grad_kv and saved records, d = 5120
    float clamp;
};

struct GateWReduceParams {
    const float* partial;  // partial[b * stride + i], b < nblocks, i < n (fp32)
    float* out;            // (n), may be null when grad_wh / grad_we are written
    int nblocks;
    int n;
    int stride;
    int pairs;  // 1: slots come as (hi, lo) pairs; 2: slot b holds hi, lo16 + b * n holds lo (bf16)
    const uint16_t* lo16;
    // product rule of a fused weight w = wh * we (null: not written):
    // grad_wh = grad_w * we, grad_we = grad_w * wh, wh and we bf16 (n)
    const uint16_t* wh;
    const uint16_t* we;
    float* grad_wh;
    float* grad_we;
};

// GateConv: one cluster per token range (consecutive tokens of one batch
// row); CTA `rank` of the cluster owns columns [rank * ncols, ...).
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
    int ncols;           // columns per CTA slice (4 per thread); the last may be shorter
    int ring_off;        // byte offset of the ring in shared memory
    int range_len;       // tokens per range (the last range of a row may be shorter)
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
    unsigned long long* xrec;  // exchange records, 2 slots x 16 words per CTA, zero at launch
    unsigned int* err;
    int M, T, d;
    int group;       // CTAs per token range (column slices), at most 8; cluster launch: unused
    int nranges;     // token ranges (M * ranges_per_row)
    int ncols;
    int ring_off;
    int sc_off;      // byte offset of the per-token saved scalars in shared memory
    int range_len;
    int ranges_per_row;
    float eps;
    float inv_sqrt_d;
};

// Fused weight of the gate (forward: weight = wh * we) and its backward
// (grad_w = sum over nblocks partials of n values each; grad_wh, grad_we).
struct FusedWeightParams {
    const uint16_t* wh;
    const uint16_t* we;
    float* weight;
    const float* partial;
    float* grad_w;
    float* grad_wh;
    float* grad_we;
    long long n;
    long long nblocks;
};

// GateConv decode step (one token per batch row).  The weight matrices are
// also described by 2-D tensor maps (box 32 columns x 256 rows), encoded on
// the host per call.
struct DecodeParams {
    CUtensorMap tmk;          // W_K as (d_mem, d) bf16
    CUtensorMap tmv;          // W_V
    const uint16_t* e;        // (B, dmem) bf16
    const uint16_t* h;        // (B, d) bf16
    const uint16_t* state;    // (B, L, d) bf16, may be null when L == 0
    const uint16_t* WK;       // (dmem, d) bf16
    const uint16_t* WV;
    const float* wh;          // (d)
    const float* wv;          // (d)
    const float* cw;          // (w, d)
    uint16_t* y;              // (B, d) bf16
    uint16_t* new_state;      // (B, max_len, d) bf16
    float* vbuf;              // workspace: (B, d) fp32 projected v
    float* stats;             // workspace: (B, d / 32, 4) fp32 row sums of each 32-column tile
    unsigned int* err;        // sticky device error word
    int B, dmem, d, L, max_len, w, dil;
    float eps, inv_sqrt_d;
};

struct LaunchCfg {
    int cluster;
    int threads;
    int clusters;   // grid size in clusters (CTAs when cluster == 1)
    int stages;
    int smem;
    int grid_y;     // second grid dimension (1 unless stated)
    int aux_blocks; // CTAs of a preceding helper kernel, if any
    int token_split;  // gate backward: the warps of a CTA split its tokens (see GateBwdParams)
};

// Kernel launchers (defined next to their kernels).  Each returns the launch
// status; none synchronises.
cudaError_t gate_fwd_prepare(int smem_bytes);
cudaError_t gate_fwd_max_clusters(int cluster, int threads, int smem, int* out);
cudaError_t gate_fwd_launch(const GateFwdParams& p, const LaunchCfg& c, cudaStream_t s);

cudaError_t gate_bwd_prepare(int smem_bytes);
cudaError_t gate_bwd_max_clusters(int cluster, int threads, int smem, int* out);
cudaError_t gate_bwd_launch(const GateBwdParams& p, const LaunchCfg& c, cudaStream_t s);
// the one-pass backward (packed layout): G clusters of two CTAs
cudaError_t gate_bwd_fused_prepare();
cudaError_t gate_bwd_fused_max_clusters(int* out);
int gate_bwd_fused_threads();
int gate_bwd_fused_smem();
cudaError_t gate_bwd_fused_launch(const GateBwdParams& p, int G, cudaStream_t s);
cudaError_t gate_wreduce_launch(const GateWReduceParams& p, cudaStream_t s);

cudaError_t fused_weight_launch(const FusedWeightParams& p, cudaStream_t s);
cudaError_t fused_weight_bwd_launch(const FusedWeightParams& p, cudaStream_t s);

cudaError_t decode_prepare();
cudaError_t decode_launch(const DecodeParams& p, cudaStream_t s);

int gateconv_fwd_smem(int threads);  // dynamic shared memory of the forward kernel of that CTA size (fixed layout)
int gateconv_bwd_smem();  // dynamic shared memory of the backward kernel (fixed layout)
int gateconv_bwd_threads();  // threads of a backward CTA (two warp groups over one column slice)
cudaError_t gateconv_fwd_prepare(int smem_bytes);
cudaError_t gateconv_fwd_max_clusters(int cluster, int threads, int smem, int* out);
cudaError_t gateconv_fwd_launch(const GateConvFwdParams& p, const LaunchCfg& c, cudaStream_t s);

cudaError_t gateconv_bwd_prepare(int smem_bytes);
cudaError_t gateconv_bwd_max_clusters(int cluster, int threads, int smem, int* out);
cudaError_t gateconv_bwd_blocks_per_sm(int threads, int smem, int* out);
cudaError_t gateconv_bwd_launch(const GateConvBwdParams& p, const LaunchCfg& c, int groups, cudaStream_t s);
cudaError_t gateconv_wreduce_launch(const GateWReduceParams& p, cudaStream_t s);

}  // namespace eg
