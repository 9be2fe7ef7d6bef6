/*
 * engram.h -- C ABI of the GB300 (sm_103a) Engram gate library, libengram.so.
 *
 * Two fused, memory-bound operators:
 *
 *  1. The four-stream saved-state gate (cuDNN Frontend, "Engram saved-state
 *     gate": semantics, layout and saved-state paragraphs, and its
 *     plan/execute example).  Per token n and stream s < 4, X[n,s,:] and its
 *     key KV[n, s*5120 : (s+1)*5120] are RMS-normalised separately
 *     (rstd = 1/sqrt(mean(x^2) + eps)); dot = sum_i xh_i * weight[s,i] * kh_i
 *     in FP32; sq = sign(dot) * sqrt(max(|dot|, 1e-6)); gate = sigmoid(sq);
 *     out = X + gate * v with v = KV[n, 20480:25600], rounded once to BF16.
 *     A false mask gives out == X bit for bit.
 *
 *  2. GateConv (TileOPs "Engram Operators", GateConv section,
 *     EngramGateConvFwdOp / EngramGateConvBwdOp): RMSNorm gating of H and k,
 *     a causal depthwise conv1d with 4 taps over the RMS-normalised gated
 *     value, then SiLU plus the gated value as residual.
 *
 * Conventions shared by every entry point
 *  - Pointers are DEVICE pointers to contiguous, row-major tensors.  BF16
 *    tensors are passed as `void*` holding IEEE bfloat16 values (the upper
 *    half of a binary32 word).  Floating tensors and workspaces must be
 *    16-byte aligned; the mask is a byte array with no alignment rule.
 *  - The caller allocates and owns every buffer.  The library keeps no
 *    pointer after the call returns.  Outputs and workspaces must not
 *    overlap any input or one another (checked on the host by address
 *    range; overlap returns ENGRAM_ERR_OVERLAP).
 *  - Every call is asynchronous on `stream` (0 = legacy default stream):
 *    it validates its arguments on the host, then enqueues kernels.  It
 *    performs no allocation, no host<->device copy and no synchronisation,
 *    so it may be captured in a CUDA graph.  The first call on a device also
 *    performs one-time, per-device set-up (kernel attributes and occupancy
 *    queries); make that first call before any stream capture.
 *  - Ordering is plain stream order.  Most kernels are launched with
 *    programmatic stream serialisation, so a kernel may be scheduled while
 *    the one before it on the stream finishes. Each waits for that kernel to
 *    complete (griddepcontrol.wait) before it reads anything the kernel may
 *    have written, and lets the next kernel be scheduled only after that
 *    wait.  A caller's kernel launched the same way after one of ours must
 *    likewise wait before it reads our outputs, as that launch mode requires.
 *  - A non-OK status means nothing was enqueued, except ENGRAM_ERR_LAUNCH
 *    (the launch itself failed; the stream state is then the CUDA runtime's).
 *    The library never prints, traps or aborts.
 *  - Kernels that wait on asynchronous copies give up after a bounded time
 *    and raise a sticky device flag instead of hanging; read it with
 *    engram_device_error().
 */
#ifndef ENGRAM_H_
#define ENGRAM_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ENGRAM_OK = 0,
    ENGRAM_ERR_NULL = 1,      /* a required pointer is NULL                  */
    ENGRAM_ERR_ALIGN = 2,     /* a floating tensor / workspace not 16-B aligned */
    ENGRAM_ERR_SHAPE = 3,     /* a size is out of the supported range        */
    ENGRAM_ERR_OVERLAP = 4,   /* an output or workspace overlaps another buffer */
    ENGRAM_ERR_WORKSPACE = 5, /* workspace_bytes below the required size     */
    ENGRAM_ERR_DEVICE = 6,    /* no usable sm_103 device / set-up failed     */
    ENGRAM_ERR_LAUNCH = 7     /* the kernel launch returned an error         */
} engram_status_t;

/* Human-readable name of a status code (static string). */
const char* engram_status_string(engram_status_t s);

/* Fixed layout of the saved-state gate (cuDNN "Engram saved-state gate",
 * layout paragraph): 4 streams of hidden size 5120; packed KV is 4 keys then
 * one shared value, 25600 columns. */
#define ENGRAM_GATE_STREAMS 4
#define ENGRAM_GATE_HIDDEN 5120
#define ENGRAM_GATE_KV_COLS 25600
#define ENGRAM_GATE_MAX_TOKENS 4194240   /* forward: 1 <= N <= 65535*64     */
#define ENGRAM_GATE_BWD_MAX_TOKENS 4194240 /* backward: N % 64 == 0, N <= 65535*64 */
#define ENGRAM_GATECONV_MAX_D 8192       /* GateConv: 8 <= d <= 8192, d % 8 == 0 */
#define ENGRAM_GATE_CLAMP 1e-6f          /* clamp of the signed square root         */
#define ENGRAM_GATE_SEP_MAX_HIDDEN 65536 /* separate-tensor gate: H % 8 == 0        */

/*
 * Saved-state gate, forward (cuDNN "Engram saved-state gate", semantics and
 * saved-state paragraphs).
 *   x      bf16 (N, 4, 5120)     input streams X
 *   kv     bf16 (N, 25600)       keys s = 0..3 in columns [s*5120, (s+1)*5120),
 *                                shared value in [20480, 25600)
 *   weight fp32 (4, 5120)        fused weight: product of the q/k norm weights
 *   mask   uint8 (N)             nonzero = true (torch.bool layout); a false
 *                                token gives out == X bit for bit; NULL = all true
 *   out    bf16 (N, 4, 5120)     X + gate * v, one round-to-nearest-even
 *   saved  fp32 (N, 4, 4) / NULL per (n, s): gate, dot, rstd_X, rstd_key.
 *                                A false token stores gate = 0 (dot and both
 *                                rstd as usual), which makes the backward the
 *                                derivative of out = X.  NULL skips the write;
 *                                `out` is bit-identical either way.
 *   N      1 <= N <= ENGRAM_GATE_MAX_TOKENS
 *   eps    RMS-norm epsilon (the pages' default is 1e-20)
 * Keep `saved` and the matching x / kv / weight alive and unmodified until the
 * backward that consumes them has run; each outstanding forward needs its
 * own `saved`.  The library cannot check that identity.
 * Workspace: none.
 */
engram_status_t engram_gate_fwd(const void* x, const void* kv, const float* weight,
                                const uint8_t* mask, void* out, float* saved,
                                int64_t N, float eps, cudaStream_t stream);

/* Bytes of workspace the backward needs: 4*(16*N + 4*5120*(N/64)) (cuDNN
 * "Engram saved-state gate", workspace paragraph).  0 for invalid N. */
size_t engram_gate_bwd_workspace_size(int64_t N);

/*
 * Saved-state gate, backward (cuDNN "Engram saved-state gate", layout and
 * saved-state paragraphs; tile-kernels test_engram_gate_bwd.py).
 *   x, kv, weight   the forward's inputs
 *   saved    fp32 (N, 4, 4)   the forward's saved state (gate, dot, rstd_X, rstd_key)
 *   grad_out bf16 (N, 4, 5120)
 *   grad_x   bf16 (N, 4, 5120)  out: grad_out + gate-path term, rounded once
 *   grad_kv  bf16 (N, 25600)    out: key grads in the key columns; the shared
 *                               value's grad = sum over the 4 streams of
 *                               gate_s * grad_out_s, summed in FP32 (stream
 *                               order 0..3) before its one BF16 rounding
 *   grad_weight fp32 (4, 5120)  out: sum over tokens of ddot * xh * kh, formed
 *                               as per-token-range partials in the workspace
 *                               and reduced in a fixed order (bitwise
 *                               reproducible run to run on a device)
 *   workspace  >= engram_gate_bwd_workspace_size(N) bytes, 16-B aligned,
 *              contents need no initialisation and are left undefined
 *   N        64 <= N <= ENGRAM_GATE_BWD_MAX_TOKENS, N % 64 == 0.  The cuDNN
 *            page caps N at 8192 (a limit of its workspace design); here the
 *            workspace grows by 1,344 bytes per token and the grad_weight
 *            merge reads N/64 slots per column, so any multiple of 64 up to
 *            the forward's maximum is accepted.
 * Two kernels on `stream` when the workspace holds 42 or more of the one-pass
 * kernel's clusters and the device runs them at once (N >= 3840 on GB300:
 * one pass over the rows, then the grad_weight merge), three otherwise
 * (per-token scalars, the elementwise pass, the merge), no host
 * synchronisation between them.
 */
engram_status_t engram_gate_bwd(const void* x, const void* kv, const float* weight,
                                const float* saved, const void* grad_out, void* grad_x,
                                void* grad_kv, float* grad_weight, void* workspace,
                                size_t workspace_bytes, int64_t N, cudaStream_t stream);

/*
 * Saved-state gate, backward, when the weight is a fused weight w = wh * we
 * (cuDNN "Engram saved-state gate", semantics paragraph: the weight is the
 * FP32 product of the query- and key-side normalisation weights and the
 * caller forms their product-rule gradients from grad_weight; tile-kernels
 * test_engram_gate_bwd.py checks grad_wh and grad_we formed that way).
 * engram_gate_bwd, plus the product rule in the same pass that merges
 * grad_weight (no further launch and no re-read of grad_weight):
 *   grad_wh[i] = grad_weight[i] * we[i],  grad_we[i] = grad_weight[i] * wh[i]
 * each one FP32 rounding of the FP32 grad_weight times the factor.
 *   wh, we      bf16 (4, 5120)  the factors of `weight` (weight[i] = wh[i] we[i],
 *                               as engram_fused_weight computes it), 16-B aligned
 *   grad_weight fp32 (4, 5120)  out, or NULL to skip it
 *   grad_wh, grad_we fp32 (4, 5120)  out
 * Every other argument, limit and error as engram_gate_bwd; outputs must not
 * overlap anything.  The kernels of engram_gate_bwd on `stream`.
 */
engram_status_t engram_gate_bwd_fused_weight(const void* x, const void* kv, const float* weight,
                                             const float* saved, const void* grad_out,
                                             const void* wh, const void* we, void* grad_x,
                                             void* grad_kv, float* grad_weight, float* grad_wh,
                                             float* grad_we, void* workspace,
                                             size_t workspace_bytes, int64_t N,
                                             cudaStream_t stream);

/*
 * Saved-state gate with separate key and value tensors and any hidden size
 * (tile-kernels 1.0.0 engram tests: engram_gate_fwd / engram_gate_bwd take x,
 * k (N, hc, H), v (N, H) and the fused weight, have no mask, return the saved
 * dot, gate score and both rstd only when asked, and return grad_w as
 * per-block partials that the caller sums).  Same arithmetic as
 * engram_gate_fwd / engram_gate_bwd, with hc = 4 streams.
 *   x, k       bf16 (N, 4, H)      streams and their keys
 *   v          bf16 (N, H)         shared value
 *   weight     fp32 (4, H)         fused weight
 *   out        bf16 (N, 4, H)      out: bf16(x + gate * v)
 *   dot, gate, rstd_x, rstd_k  fp32 (N, 4)  out, saved state: all four, or all
 *              four NULL to skip them (out is bit-identical either way)
 *   N: 1 <= N <= ENGRAM_GATE_MAX_TOKENS; H: 8 <= H <= ENGRAM_GATE_SEP_MAX_HIDDEN,
 *   H % 8 == 0; eps inside the root (1e-20 in the pages' tests); clamp of the
 *   signed square root (1e-6).  All pointers 16-byte aligned; outputs must
 *   not overlap anything.  Asynchronous on `stream`, no allocation.
 */
engram_status_t engram_gate_sep_fwd(const void* x, const void* k, const void* v,
                                    const float* weight, void* out, float* dot, float* gate,
                                    float* rstd_x, float* rstd_k, int64_t N, int64_t H, float eps,
                                    float clamp, cudaStream_t stream);

/* Bytes of workspace engram_gate_sep_bwd needs: 64 N (per-token scalars);
 * 0 if N is out of range. */
size_t engram_gate_sep_bwd_workspace_size(int64_t N);

/*
 * Backward of engram_gate_sep_fwd.
 *   grad_out   bf16 (N, 4, H)
 *   x, k, v, weight            as in the forward
 *   dot, gate, rstd_x, rstd_k  fp32 (N, 4), the forward's saved state
 *   grad_x, grad_k   bf16 (N, 4, H)   out
 *   grad_v           bf16 (N, H)      out: sum over the 4 streams of
 *                                     gate * grad_out before its BF16 cast
 *   grad_w_partial   fp32 (ceil(N/64), 4, H)  out: block b holds the grad_weight
 *                                     contribution of tokens 64b .. 64b+63
 *                                     (the caller sums over blocks)
 *   workspace  >= engram_gate_sep_bwd_workspace_size(N) bytes, 16-B aligned
 * Limits and errors as the forward.
 */
engram_status_t engram_gate_sep_bwd(const void* grad_out, const void* x, const void* k,
                                    const void* v, const float* weight, const float* dot,
                                    const float* gate, const float* rstd_x, const float* rstd_k,
                                    void* grad_x, void* grad_k, void* grad_v, float* grad_w_partial,
                                    void* workspace, size_t workspace_bytes, int64_t N, int64_t H,
                                    float clamp, cudaStream_t stream);

/*
 * Fused weight of the gate and its gradients (cuDNN "Engram saved-state
 * gate", semantics paragraph: the weight is the FP32 product of the query-
 * and key-side normalisation weights; tile-kernels engram tests).
 * engram_fused_weight: weight[i] = wh[i] * we[i] (exact in fp32).
 * engram_fused_weight_bwd: grad_w[i] = sum over b < nblocks of
 *   grad_w_partial[b * n + i] (fixed order, error-free additions), then
 *   grad_wh[i] = grad_w[i] * we[i] and grad_we[i] = grad_w[i] * wh[i].
 *   grad_w may be NULL.  grad_w_partial is the output of engram_gate_sep_bwd
 *   (nblocks = ceil(N/64), n = 4 H), or a single block (nblocks = 1) holding
 *   engram_gate_bwd's grad_weight.
 *   wh, we  bf16 (n); weight, grad_w, grad_wh, grad_we fp32 (n); all 16-byte
 *   aligned; 1 <= n, 1 <= nblocks, nblocks * n < 2^40; outputs must not
 *   overlap anything.  Asynchronous on `stream`, no allocation.
 */
engram_status_t engram_fused_weight(const void* wh, const void* we, float* weight, int64_t n,
                                    cudaStream_t stream);
engram_status_t engram_fused_weight_bwd(const float* grad_w_partial, int64_t nblocks,
                                        const void* wh, const void* we, float* grad_w,
                                        float* grad_wh, float* grad_we, int64_t n,
                                        cudaStream_t stream);

/*
 * GateConv, forward (TileOPs "Engram Operators", EngramGateConvFwdOp).
 *   H, k, v   bf16 (M, T, d)   hidden states, key and value projections
 *   rms_w_h   fp32 (d)         RMSNorm weight shared by H and k
 *   rms_w_v   fp32 (d)         RMSNorm weight of the gated value (conv input)
 *   conv_w    fp32 (4, d)      depthwise causal taps; tap 3 multiplies the
 *                              current token, tap j the token 3-j steps back
 *   Y         bf16 (M, T, d)   out: SiLU(conv(u)) + vhat (to be added to H
 *                              by the caller as a residual)
 *   vhat      bf16 (M, T, d)   out: alpha * v, saved for the backward
 *   alpha, rrms_h, rrms_k, rrms_v  fp32 (M, T)  out: scalar gate and the
 *                              reciprocal RMS of H, k and vhat
 * with rrms_x = 1/sqrt(mean(x^2) + eps), alpha = sigmoid(sum_i (H rrms_h w_h)_i
 * (k rrms_k w_h)_i / sqrt(d)), u = vhat * rrms_v * rms_w_v, conv zero-padded
 * at the start of each batch row.  Y and vhat are rounded once to BF16; the
 * forward uses the unrounded vhat for rrms_v, u and Y.
 *   1 <= M, 1 <= T, 8 <= d <= ENGRAM_GATECONV_MAX_D, d % 8 == 0,
 *   M*T <= 2^31 - 1; otherwise ENGRAM_ERR_SHAPE.
 * Workspace: none.
 */
engram_status_t engram_gateconv_fwd(const void* H, const void* k, const void* v,
                                    const float* rms_w_h, const float* rms_w_v,
                                    const float* conv_w, void* Y, void* vhat, float* alpha,
                                    float* rrms_h, float* rrms_k, float* rrms_v, int64_t M,
                                    int64_t T, int64_t d, float eps, cudaStream_t stream);

/* Bytes of workspace engram_gateconv_bwd needs for (M, T, d); 0 if invalid. */
size_t engram_gateconv_bwd_workspace_size(int64_t M, int64_t T, int64_t d);

/*
 * GateConv, backward (TileOPs "Engram Operators", EngramGateConvBwdOp).
 *   dY, H, k, v, rms_w_h, rms_w_v, conv_w   as in the forward
 *   vhat, alpha, rrms_h, rrms_k, rrms_v     the forward's saved tensors
 *   dH, dk, dv          bf16 (M, T, d)      out
 *   drms_w_h, drms_w_v  fp32 (d)            out, summed over all M*T tokens
 *   dconv_w             fp32 (4, d)         out, summed over all M*T tokens
 *   workspace  >= engram_gateconv_bwd_workspace_size(M, T, d) bytes, 16-B
 *              aligned: per-range fp32 weight-gradient partials (6 d floats
 *              per token range, at most max(M, 256) ranges), summed in a fixed
 *              order by a second kernel (bitwise reproducible), then 256 KiB
 *              of exchange records for the CTAs that share a token row, which
 *              the call clears on `stream` before its kernels when it uses
 *              them; nothing in it needs to start at zero
 * The CTAs of a token row (one 512-thread CTA per SM) exchange per-token sums
 * while they run: as a thread-block cluster, or, at widths where clusters
 * would leave SMs idle (d = 7168, for instance), as a cooperative launch of
 * CTA groups exchanging through the workspace's records; the call returns
 * ENGRAM_ERR_LAUNCH if the runtime refuses either launch.
 * The backward reads the saved bf16 vhat (not alpha * v) wherever the forward
 * used the gated value, and recomputes the gate's logit from H, k, rrms_h and
 * rrms_k.  Same size limits as the forward.
 */
engram_status_t engram_gateconv_bwd(const void* dY, const void* H, const void* k,
                                    const void* v, const float* rms_w_h,
                                    const float* rms_w_v, const float* conv_w,
                                    const void* vhat, const float* alpha,
                                    const float* rrms_h, const float* rrms_k,
                                    const float* rrms_v, void* dH, void* dk, void* dv,
                                    float* drms_w_h, float* drms_w_v, float* dconv_w,
                                    void* workspace, size_t workspace_bytes, int64_t M,
                                    int64_t T, int64_t d, float eps, cudaStream_t stream);

/*
 * GateConv decode, one token per batch row (TileOPs "Engram Operators",
 * Decode section, EngramDecodeFwdOp: GEMV projection + gating + dilated conv
 * + SiLU with a conv cache).
 *   e        bf16 (B, d_mem)    gathered N-gram embedding of the token
 *   h        bf16 (B, d)        hidden state of the token
 *   state    bf16 (B, L, d)     conv cache: conv inputs u of earlier tokens,
 *                               oldest first, most recent last; L <= max_len
 *                               (NULL allowed when L == 0)
 *   W_K, W_V bf16 (d_mem, d)    key and value projections (k = e W_K, v = e W_V)
 *   rms_w_h  fp32 (d)           RMSNorm weight of h and k
 *   rms_w_v  fp32 (d)           RMSNorm weight of the gated value
 *   conv_w   fp32 (w, d)        depthwise taps; tap j multiplies u at
 *                               (w-1-j)*dilation tokens back (tap w-1: this token)
 *   y        bf16 (B, d)        out: SiLU(c) + vhat (the residual to add to h)
 *   new_state bf16 (B, max_len, d)  out: the cache shifted by one token, this
 *                               token's u (rounded to bf16) in the last row
 * with alpha = sigmoid(sum (h rrms_h w_h)(k rrms_k w_h) / sqrt(d)), vhat =
 * alpha v, u = vhat rrms_v w_v, as in engram_gateconv_fwd; cache rows beyond L
 * read as zero.  workspace >= engram_decode_workspace_size(B, d_mem, d) bytes.
 *   1 <= B <= 1048560, 8 <= d_mem <= 65536 with d_mem % 8 == 0,
 *   64 <= d <= 65536 with d % 64 == 0, 1 <= w <= 64, dilation >= 1,
 *   1 <= max_len <= 65536, 0 <= L <= max_len.  All pointers 16-byte aligned;
 *   outputs and workspace must not overlap anything (the new cache is a
 *   separate buffer).  Asynchronous on `stream`, no allocation.
 */
size_t engram_decode_workspace_size(int64_t B, int64_t d_mem, int64_t d);
engram_status_t engram_decode_fwd(const void* e, const void* h, const void* state, int64_t L,
                                  const void* W_K, const void* W_V, const float* rms_w_h,
                                  const float* rms_w_v, const float* conv_w, void* y,
                                  void* new_state, void* workspace, size_t workspace_bytes,
                                  int64_t B, int64_t d_mem, int64_t d, int64_t max_len, int64_t w,
                                  int64_t dilation, float eps, cudaStream_t stream);

/*
 * Saved-state gate, backward, for callers that cannot allocate.  The pages
 * have no counterpart to this entry point.
 *
 * Some callers cannot call cudaMalloc (or any allocator, PyTorch's included)
 * at the point where they run the backward: plug-ins embedded in a host
 * framework that owns all device memory and forbids outside allocations, and
 * runtimes that work from a fixed, pre-planned memory budget.  They can pass inputs
 * and outputs they already own, but no workspace.  This call is
 * engram_gate_bwd with its workspace taken from a fixed array inside the
 * library (ENGRAM_GATE_BWD_NOALLOC_SCRATCH_BYTES, enough for N up to
 * ENGRAM_GATE_BWD_NOALLOC_MAX_TOKENS).  Every GPU that loads the library
 * holds that array until the process exits.
 *   Arguments: as engram_gate_bwd, without the workspace pair.
 *   N: 64 <= N <= ENGRAM_GATE_BWD_NOALLOC_MAX_TOKENS, N % 64 == 0; a larger N
 *      returns ENGRAM_ERR_SHAPE and enqueues nothing (use engram_gate_bwd
 *      with a caller-provided workspace instead).
 *   The first call on each device (and the first after the device's context
 *   was replaced) looks up the array's device address with that device
 *   current, a one-time set-up.  The call itself allocates nothing.
 *   All calls share the one array, which keeps the previous call's contents;
 *   nothing in it needs to start at zero (each call writes every slot it
 *   reads before reading it).  Calls whose kernels can overlap on the GPU
 *   (different streams without ordering between them) race on the array and
 *   give undefined results: serialise them.
 */
#define ENGRAM_GATE_BWD_NOALLOC_MAX_TOKENS 2048
#define ENGRAM_GATE_BWD_NOALLOC_SCRATCH_BYTES \
    (4 * (16 * ENGRAM_GATE_BWD_NOALLOC_MAX_TOKENS + 4 * 5120 * (ENGRAM_GATE_BWD_NOALLOC_MAX_TOKENS / 64)))
engram_status_t engram_gate_bwd_noalloc(const void* x, const void* kv, const float* weight,
                                        const float* saved, const void* grad_out, void* grad_x,
                                        void* grad_kv, float* grad_weight, int64_t N,
                                        cudaStream_t stream);

/*
 * Diagnostics (not part of the pages' API).
 * engram_device_error: synchronises the current device, copies the sticky
 * device error word into *flags (0 = none; bit 0 = an asynchronous copy did
 * not complete within its time limit) and clears it.  Returns ENGRAM_OK or
 * ENGRAM_ERR_DEVICE.  Not for use inside a stream capture.
 */
engram_status_t engram_device_error(uint32_t* flags);

/* Launch geometry chosen for a call, for tests and benchmarks: CTAs that
 * share one token row (thread-block cluster size, or column slices), threads
 * per CTA, number of such CTA groups, ring stages and dynamic shared memory
 * bytes of the main kernel, how many of those CTA groups the device runs at
 * once (occupancy), and how many kernels the call launches.  `op`: 0 gate
 * fwd, 1 gate bwd, 2 gateconv fwd, 3 gateconv bwd.  n0, n1, n2 = (N) for the
 * gate, (M, T, d) for GateConv. */
typedef struct {
    int cluster;
    int threads;
    int clusters;
    int stages;
    int smem_bytes;
    int resident;
    int kernels;
} engram_launch_info_t;
engram_status_t engram_launch_info(int op, int64_t n0, int64_t n1, int64_t n2,
                                   engram_launch_info_t* info);

#ifdef __cplusplus
}
#endif

#endif /* ENGRAM_H_ */
