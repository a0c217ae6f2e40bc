/*
 * upipe.h -- C ABI of the head-chunked GQA/RoPE causal attention layer
 * (UPipe, "Untied Ulysses") for one NVIDIA GB300 (sm_103a).
 *
 * What the library computes
 * -------------------------
 * One attention layer of a Llama-style transformer, computed one chunk of U
 * query heads at a time over the full sequence:
 *
 *   "Untied Ulysses: Memory-Efficient Context Parallelism via Headwise
 *   Chunking" (index page, Abstract): fine-grained chunking at the attention
 *   head level, reducing intermediate tensor memory of the attention layer.
 *   "Untied Ulysses Pushes Llama-3-8B Training to 5 Million Tokens" (talk
 *   write-up), paragraph on intermediate buffers: one group of heads is
 *   computed, attention is run and a partial result is stored; the next group
 *   reuses the buffers of the previous one; the attention formula itself is
 *   unchanged.
 *
 * For chunk c (query heads cU .. cU+U-1 and the KV heads they read):
 *   [Q_c|K_c|V_c] = x Wqkv[rows_c]^T, RoPE on Q_c and K_c,
 *   O_c = causal_softmax(Q_c K_c^T / sqrt(d)) V_c   (plus LSE per head),
 *   out32 += O_c Wo[:, cols_c]^T,                     out = bf16(out32).
 * The backward pass recomputes Q_c/K_c/V_c (and O_c unless it was kept, on
 * the device or in host memory), and produces the chunk's dQ/dK/dV, its rows
 * of dWqkv, its columns of dWo and its share of dx.  Every chunk reuses one
 * workspace region, so the intermediate activation memory is proportional to
 * U rather than H.
 *
 * Around the layer the library also computes, tiled along the sequence, the
 * block's SwiGLU MLP and the LM-head cross-entropy loss (upipe_mlp_*,
 * upipe_ce_*, below).
 *
 * Conventions (readings of points the pages leave open)
 * -----------------------------------------------------
 *  - Head dimension d = 128.  Query head h reads KV head h / g, g = H / Hkv.
 *  - Causal mask: key j is visible to query i iff j <= i.  Scale 1/sqrt(d).
 *  - RoPE pairs (i, i + d/2) of each head and rotates them by the angle
 *    p * theta^(-2i/d) (p = token position, angle evaluated in fp64).
 *  - Wqkv is [(H + 2 Hkv) d, D] row-major (rows: q heads, then k heads, then
 *    v heads, d rows each); Wo is [D, H d] row-major (nn.Linear layout).
 *  - LSE is the natural log of the row's sum of exp(scaled score), [H, L].
 *  - Reductions are deterministic and do not depend on U: a run with any
 *    valid U returns the same bits as a run with U = H.
 *
 * Memory, ownership, streams
 * --------------------------
 *  - Every pointer is a device pointer owned by the caller, including the
 *    workspace `ws`, whose size comes from upipe_workspace_bytes() (or the
 *    MLP / loss variants), except the host buffers the activation-offload
 *    calls name as such.  The library allocates no device memory.
 *  - bf16 tensors are passed as `uint16_t*` holding bfloat16 bit patterns.
 *  - Every pointer must be 16-byte aligned; tensors are dense row-major.
 *  - Work is enqueued on `stream` (a cudaStream_t, 0 = legacy default) and
 *    the call returns without waiting.  Calls that share a workspace must be
 *    ordered on the GPU (for example, issued on one stream).
 *  - The backward entry points also enqueue on one library-owned stream per
 *    device, created on the first backward call there with the device's
 *    greatest stream priority: each chunk's dK/dV kernel runs on it, forked
 *    from `stream` and joined back into it by events, while that chunk's dQ
 *    kernel runs on `stream`.  All of a call's work is still ordered after
 *    the work enqueued on `stream` before it, and work enqueued on `stream`
 *    after it waits for all of it.  Make the first backward call on each
 *    device outside stream capture.
 *  - The activation-offload calls below use two more library-owned streams
 *    per device (copies to and from the host), created on their first use.
 *  - Entry points may be called from several host threads (calls that share
 *    a workspace still need GPU ordering); the launch counter and the
 *    profiling hooks below are meant for one thread.
 *
 * Errors
 * ------
 * Every entry point returns 0 on success or a negative UPIPE_ERR_* code.
 * Argument errors are detected on the host before anything is enqueued.
 * Device-side waits are bounded (default 2 s, environment variable
 * UPIPE_SPIN_LIMIT_NS overrides; kernels count the limit in SM clock cycles
 * at 3 cycles per nanosecond, so at clocks below 3 GHz a wait lasts somewhat
 * longer than the limit, never shorter); a wait that runs out makes its
 * kernel unwind and sets a device status word, read by
 * upipe_last_device_status().
 */
#ifndef UPIPE_H_
#define UPIPE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define UPIPE_OK 0
#define UPIPE_ERR_INVALID_ARG (-1)        /* bad shape, null or misaligned pointer */
#define UPIPE_ERR_WS_TOO_SMALL (-2)       /* ws_bytes < upipe_workspace_bytes(...) */
#define UPIPE_ERR_CUDA (-3)               /* a CUDA runtime/driver call failed */
#define UPIPE_ERR_DEVICE_TIMEOUT (-4)     /* a bounded device wait ran out */
#define UPIPE_ERR_UNSUPPORTED_DEVICE (-5) /* current device is not sm_103 */
#define UPIPE_ERR_SCRATCH_LIMIT (-6)      /* needs more than UPIPE_NOALLOC_SCRATCH_BYTES */

/* Problem description.  All fields are read on every call.
 *   L          tokens (1 .. 2^31-1)
 *   D          hidden size; layer entries only, multiple of 128
 *   H, Hkv     query / KV heads; H % Hkv == 0, H + 2*Hkv <= 96
 *   d          head dimension; must be 128
 *   U          query heads per chunk; H % U == 0 and (U % g == 0 or g % U == 0)
 *   causal     must be 1
 *   rope_theta RoPE base (> 0); layer entries only                          */
typedef struct upipe_cfg {
  int64_t L;
  int32_t D;
  int32_t H;
  int32_t Hkv;
  int32_t d;
  int32_t U;
  int32_t causal;
  double rope_theta;
} upipe_cfg;

/* Where the layer entries keep the attention output O between the forward
 * and the backward (the o_mode argument below):
 *   UPIPE_O_RECOMPUTE  upipe_attn_fwd / _bwd with o_saved NULL: O lives in
 *                      the workspace one chunk at a time; the backward
 *                      recomputes it from the LSE
 *   UPIPE_O_DEVICE     upipe_attn_fwd / _bwd with o_saved given
 *   UPIPE_O_HOST       upipe_attn_fwd_host_o / _bwd_host_o: page-locked host
 *                      memory holds it; chunk buffers of O in the workspace
 *                      (three in the forward, two in the backward)         */
#define UPIPE_O_RECOMPUTE 0
#define UPIPE_O_DEVICE 1
#define UPIPE_O_HOST 2

/* Workspace bytes for one call.
 *   pass        0 = forward, 1 = backward
 *   core_only   1 = upipe_attn_core_fwd / _bwd, 0 = the layer entries
 *   o_mode      UPIPE_O_RECOMPUTE, UPIPE_O_DEVICE or UPIPE_O_HOST (layer
 *               entries; ignored with core_only)
 * Returns 0 for an invalid configuration, pass or o_mode (or a call that
 * needs none).                                                             */
size_t upipe_workspace_bytes(const upipe_cfg* cfg, int pass, int core_only, int o_mode);

/* Intermediate-activation accounting for one call (host arithmetic, no GPU):
 *   chunk_bytes  workspace that scales with U: the chunk's Q/K/V/O buffers
 *                and, in the backward pass, dO, Delta, dQ/dK/dV and the
 *                dK/dV carry (U < g);
 *   fixed_bytes  workspace that does not scale with U: the fp32 output carry
 *                (out32 or dx32) and the RoPE table.
 * Returns UPIPE_OK or UPIPE_ERR_INVALID_ARG.                                */
int upipe_activation_bytes(const upipe_cfg* cfg, int pass, int core_only, int o_mode,
                           size_t* chunk_bytes, size_t* fixed_bytes);

/* Largest chunk size U whose workspace fits a memory budget.  The talk
 * write-up's chunk-size ablation paragraph: larger chunks compute more heads
 * at once, use more memory and run somewhat faster, so a run picks the
 * headwise chunk size that fits its memory budget.
 *   cfg          every field but U is read (U is ignored)
 *   budget_bytes bytes the caller can give the workspace
 *   pass         0 = forward workspace, 1 = backward, 2 = the larger of the
 *                two (one workspace serving a whole training step)
 *   core_only, o_mode as for upipe_workspace_bytes
 * Considers every valid U (H % U == 0, and U % g == 0 or g % U == 0) and
 * returns the largest whose workspace is <= budget_bytes (the workspace is
 * not monotone in U: U = H drops the fp32 output carry).  Returns
 * UPIPE_ERR_INVALID_ARG for an invalid configuration or pass, and
 * UPIPE_ERR_WS_TOO_SMALL when no valid U fits.  Host arithmetic only.      */
int upipe_choose_u(const upipe_cfg* cfg, size_t budget_bytes, int pass, int core_only, int o_mode);

/* Layer forward (the write-up's paragraph on intermediate buffers).
 *   x        [L, D] bf16                 Wqkv [(H+2Hkv)*128, D] bf16
 *   Wo       [D, H*128] bf16             out  [L, D] bf16 (written)
 *   lse      [H, L] fp32 (written)
 *   o_saved  [L, H*128] bf16 or NULL: when given, the attention output O is
 *            written there (and may be passed to upipe_attn_bwd to skip the
 *            recomputation of O); when NULL, O lives only in the workspace.
 *            A kept O is computed from the final softmax probabilities
 *            (each row's LSE first, then O = sum_j exp(S_j - LSE) V_j), the
 *            same bits the backward's recomputation produces, so both
 *            backward variants return identical gradients; this costs the
 *            forward one more pass over the keys.
 *   ws       workspace of at least upipe_workspace_bytes(cfg, 0, 0, o_saved ?
 *            UPIPE_O_DEVICE : UPIPE_O_RECOMPUTE)                          */
int upipe_attn_fwd(const upipe_cfg* cfg, const uint16_t* x, const uint16_t* Wqkv, const uint16_t* Wo,
                   uint16_t* out, float* lse, uint16_t* o_saved, void* ws, size_t ws_bytes, void* stream);

/* Layer backward: gradients of sum(out * dout).
 *   dout     [L, D] bf16                 lse [H, L] fp32 from upipe_attn_fwd
 *   o_saved  NULL (recompute O per chunk) or the tensor upipe_attn_fwd wrote
 *   dx       [L, D] bf16 (written)
 *   dWqkv    [(H+2Hkv)*128, D] fp32 (written, not accumulated)
 *   dWo      [D, H*128] fp32 (written, not accumulated)
 *   ws       workspace of at least upipe_workspace_bytes(cfg, 1, 0, o_saved ?
 *            UPIPE_O_DEVICE : UPIPE_O_RECOMPUTE)                          */
int upipe_attn_bwd(const upipe_cfg* cfg, const uint16_t* x, const uint16_t* Wqkv, const uint16_t* Wo,
                   const uint16_t* dout, const float* lse, const uint16_t* o_saved, uint16_t* dx, float* dWqkv,
                   float* dWo, void* ws, size_t ws_bytes, void* stream);

/* Layer forward and backward with O kept in host memory: the talk
 * write-up's activation offloading (block activations that are expensive to
 * recompute go to CPU memory and are prefetched for the backward pass)
 * applied to the attention output, which the recomputing backward otherwise
 * rebuilds with a second pass over the keys.  Device memory still scales
 * with U: the workspace holds chunk buffers of O (three in the forward, two
 * in the backward), so that a chunk's copy runs while later chunks compute.
 *   o_host  L*H*128 bf16 (L*H*256 bytes) of page-locked host memory
 *           (cudaHostAlloc, or cudaHostRegister'ed); chunk c's O_c [L, U*128]
 *           sits at element offset c*L*U*128, so the layout depends on U and
 *           the backward must use the forward's cfg.  Not page-locked, or
 *           NULL: UPIPE_ERR_INVALID_ARG.
 *   upipe_attn_fwd_host_o writes out and lse as upipe_attn_fwd does; O_c is
 *     the online softmax's own output (not recomputed from the LSE), copied
 *     to o_host on the library's device-to-host copy stream while the next
 *     chunk runs.  Work enqueued on `stream` after the call sees o_host
 *     complete.
 *   upipe_attn_bwd_host_o returns the gradients of upipe_attn_bwd, with
 *     O_c brought back on the host-to-device copy stream during chunk
 *     c - 1 in place of the recomputation.  The gradients agree with the
 *     recomputing backward's within rounding (O from the online softmax
 *     differs from O recomputed from the LSE in its last bits), not bit for
 *     bit.
 *   ws  workspace of at least upipe_workspace_bytes(cfg, pass, 0,
 *       UPIPE_O_HOST).
 * Both hold the library's copy-stream lock for the duration of the host
 * call (calls from several threads serialise their enqueueing).            */
int upipe_attn_fwd_host_o(const upipe_cfg* cfg, const uint16_t* x, const uint16_t* Wqkv, const uint16_t* Wo,
                          uint16_t* out, float* lse, uint16_t* o_host, void* ws, size_t ws_bytes, void* stream);
int upipe_attn_bwd_host_o(const upipe_cfg* cfg, const uint16_t* x, const uint16_t* Wqkv, const uint16_t* Wo,
                          const uint16_t* dout, const float* lse, const uint16_t* o_host, uint16_t* dx, float* dWqkv,
                          float* dWo, void* ws, size_t ws_bytes, void* stream);

/* Attention core only (no projection, no RoPE), the per-rank slice that
 * head-sharded context parallelism leaves on one GPU ("Untied Ulysses Pushes
 * Llama-3-8B Training to 5 Million Tokens", paragraph on DeepSpeed Ulysses),
 * processed U query heads at a time.
 *   q, o     [L, H, 128] bf16            k, v [L, Hkv, 128] bf16
 *   lse      [H, L] fp32 (written)       cfg->D and rope_theta are ignored.
 *   ws       upipe_workspace_bytes(cfg, 0, 1, 0) bytes (0: may be NULL)      */
int upipe_attn_core_fwd(const upipe_cfg* cfg, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        uint16_t* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/* Core backward.  dout_o [L, H, 128] bf16 is the gradient of o; dq [L, H,
 * 128], dk, dv [L, Hkv, 128] bf16 are written.                              */
int upipe_attn_core_bwd(const upipe_cfg* cfg, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        const uint16_t* o, const float* lse, const uint16_t* dout_o, uint16_t* dq, uint16_t* dk,
                        uint16_t* dv, void* ws, size_t ws_bytes, void* stream);

/* Core backward that allocates nothing (no counterpart in the paper; a
 * convenience of this library).  Same arguments and results as
 * upipe_attn_core_bwd, minus the workspace.  It is meant for callers that may
 * not allocate device memory at the point of the call -- for example a
 * framework's allocator during its own out-of-memory or defragmentation
 * handling, or a runtime whose device memory budget is reserved up front and
 * fully claimed.  The scratch (the per-tile LSE/Delta records and, when
 * U < H/Hkv, the fp32 dK/dV carry) is a fixed array of
 * UPIPE_NOALLOC_SCRATCH_BYTES in the library's static device memory, which
 * every GPU that loads the library holds until the process exits.
 *  - Limit: problems whose upipe_workspace_bytes(cfg, 1, 1, 0) exceeds
 *    UPIPE_NOALLOC_SCRATCH_BYTES return UPIPE_ERR_SCRATCH_LIMIT before any
 *    GPU work (for example U = 1, Hkv = 1 fits up to about L = 32K tokens;
 *    U >= H/Hkv with U = 8 up to about L = 512K).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and creates the
 *    library's second stream and its events if no backward call has; make
 *    that first call before any stream capture.
 *  - All calls share the one array and it keeps the last call's contents:
 *    calls that overlap on the GPU (different streams, no ordering) race.
 *  - Calls no cudaMalloc, cudaFree or allocating library routine, and after
 *    the first call on a device creates no stream or event.  Its launches
 *    record no profiling events even while upipe_profile_enable(1) is on
 *    (recording may create events); they still count in
 *    upipe_launch_count().                                                  */
#define UPIPE_NOALLOC_SCRATCH_BYTES (32u << 20)
int upipe_attn_core_bwd_noalloc(const upipe_cfg* cfg, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const uint16_t* o, const float* lse, const uint16_t* dout_o, uint16_t* dq,
                                uint16_t* dk, uint16_t* dv, void* stream);

/* Activation offload ("Untied Ulysses Pushes Llama-3-8B Training to 5
 * Million Tokens", paragraph on activation offloading): a block input that
 * the backward pass needs and that cannot be cheaply recomputed -- for this
 * layer, x -- is moved to CPU memory while it is not needed and prefetched
 * before the backward pass reaches the layer, with the copies scheduled
 * around the computation.  On GB300 the host memory sits behind the
 * NVLink-C2C link.
 *   upipe_offload_async(host_dst, dev_src, bytes, stream)   device -> host
 *   upipe_prefetch_async(dev_dst, host_src, bytes, stream)  host -> device
 *     Each copy runs on a library-owned copy stream of the current device
 *     (one per direction, created on the first call there; make that first
 *     call outside stream capture), after all work enqueued on `stream`
 *     before the call, and returns without waiting.  Host buffers should be
 *     page-locked (cudaHostAlloc / pinned) for the copy to be asynchronous.
 *   upipe_copies_join(stream)
 *     Work enqueued on `stream` after this call waits for every copy issued
 *     so far on the current device (in both directions).  Join before
 *     overwriting or releasing an offloaded source, and before using a
 *     prefetched destination.
 * Return UPIPE_OK, UPIPE_ERR_INVALID_ARG (null pointer with bytes > 0) or
 * UPIPE_ERR_CUDA.  bytes == 0 is a no-op.  No counterpart of these calls
 * has its own device kernel: the copy engines move the bytes.             */
int upipe_offload_async(void* host_dst, const void* dev_src, size_t bytes, void* stream);
int upipe_prefetch_async(void* dev_dst, const void* host_src, size_t bytes, void* stream);
int upipe_copies_join(void* stream);

/* Sequence-tiled MLP and loss around the attention layer ("Untied Ulysses
 * Pushes Llama-3-8B Training to 5 Million Tokens", paragraph on Arctic Long
 * Sequence Training: the MLPs and the loss need no buffer that spans the
 * whole sequence; they are computed in tiles along the sequence axis).
 * Each call walks the L rows in tiles of T rows and keeps only one tile's
 * intermediates in the workspace, so their memory scales with T, not L.
 * Weight gradients are carried in place across tiles in a fixed fp32 order:
 * every T (a multiple of 128) returns the same bits as T >= L.
 *
 * SwiGLU MLP: y = (silu(x Wg^T) * (x Wu^T)) Wd^T, silu(g) = g sigmoid(g),
 * no biases (the MLP of the Llama-3 and Qwen models the pages train).
 *   L        rows (tokens)                 D  model width, multiple of 128
 *   F        hidden width, multiple of 128 T  rows per tile, multiple of 128 */
typedef struct upipe_mlp_cfg {
  int64_t L;
  int32_t D;
  int32_t F;
  int32_t T;
} upipe_mlp_cfg;

/* Workspace bytes (pass 0 forward: H [T, F] bf16; pass 1 backward: H, dH
 * [T, F] and [dG | dU] [T, 2F], bf16).  0 for an invalid configuration.   */
size_t upipe_mlp_workspace_bytes(const upipe_mlp_cfg* cfg, int pass);

/* Largest tile T (a multiple of 128, at most L rounded up to 128) whose MLP
 * workspace fits budget_bytes; pass 0 = forward, 1 = backward, 2 = both
 * (the backward's, the larger).  cfg->T is ignored.  Returns T, or
 * UPIPE_ERR_INVALID_ARG / UPIPE_ERR_WS_TOO_SMALL (not even T = 128 fits).
 * Host arithmetic only.                                                    */
int upipe_mlp_choose_t(const upipe_mlp_cfg* cfg, size_t budget_bytes, int pass);

/*   x    [L, D] bf16                Wgu [2F, D] bf16: the F gate rows, then the F up rows
 *   Wd   [D, F] bf16                y   [L, D] bf16 (written)             */
int upipe_mlp_fwd(const upipe_mlp_cfg* cfg, const uint16_t* x, const uint16_t* Wgu, const uint16_t* Wd, uint16_t* y,
                  void* ws, size_t ws_bytes, void* stream);

/* Gradients of sum(y * dy); the forward is recomputed per tile.
 *   dy   [L, D] bf16                dx [L, D] bf16 (written)
 *   dWgu [2F, D] fp32, dWd [D, F] fp32 (written, not accumulated)
 * Intermediates H, dH = dy Wd and [dG | dU] are stored as bf16.           */
int upipe_mlp_bwd(const upipe_mlp_cfg* cfg, const uint16_t* x, const uint16_t* Wgu, const uint16_t* Wd,
                  const uint16_t* dy, uint16_t* dx, float* dWgu, float* dWd, void* ws, size_t ws_bytes,
                  void* stream);

/* Cross-entropy of the LM head, loss and gradients in one call:
 * z = h W^T (fp32), loss_i = logsumexp(z_i) - z_i[label_i], and the
 * gradients of sum_i scale * loss_i.
 *   L, D (multiple of 128), V vocabulary (multiple of 128), T as above    */
typedef struct upipe_ce_cfg {
  int64_t L;
  int32_t D;
  int32_t V;
  int32_t T;
} upipe_ce_cfg;

/* Workspace bytes: the logits of one tile [T, V] fp32 and dZ [T, V] bf16. */
size_t upipe_ce_workspace_bytes(const upipe_ce_cfg* cfg);

/* Largest tile T for the loss whose workspace fits budget_bytes, as
 * upipe_mlp_choose_t.                                                      */
int upipe_ce_choose_t(const upipe_ce_cfg* cfg, size_t budget_bytes);

/*   h      [L, D] bf16              W [V, D] bf16
 *   labels [L] int32: a negative label ignores the token (loss 0, no
 *          gradient); a label >= V gives a NaN loss and no gradient
 *   scale  finite; e.g. 1 / (number of non-negative labels) for the mean
 *   loss   [L] fp32 (written)       dh [L, D] bf16 (written)
 *   dW     [V, D] fp32 (written, not accumulated)
 * dZ = scale (softmax(z) - onehot) enters dh = dZ W and dW = dZ^T h as bf16. */
int upipe_ce_fwd_bwd(const upipe_ce_cfg* cfg, const uint16_t* h, const uint16_t* W, const int32_t* labels,
                     float scale, float* loss, uint16_t* dh, float* dW, void* ws, size_t ws_bytes, void* stream);

/* Synchronizes `stream`, then reads and clears the device status word of
 * the current device.  Returns UPIPE_OK, UPIPE_ERR_DEVICE_TIMEOUT if a
 * bounded wait of any earlier call ran out, or UPIPE_ERR_CUDA.              */
int upipe_last_device_status(void* stream);

/* Test hook for the bounded-wait machinery: launches one CTA that waits on
 * an mbarrier nothing arrives on, with the given limit in nanoseconds, so
 * that the wait runs out and sets the status word.  Returns a launch code. */
int upipe_debug_wait_timeout(uint64_t limit_ns, void* stream);

/* Launch accounting and per-kernel timing.
 *   upipe_launch_count()  kernels this library has launched since load.
 *   upipe_profile_enable(1) makes every later launch record a CUDA event
 *   pair on the launching stream; upipe_profile_enable(0) stops recording.
 *   upipe_profile_read() synchronizes on the recorded events, writes for
 *   each kernel kind k < n its summed device time in ms (ms[k]) and launch
 *   count (launches[k]), clears the record and returns the number of kinds
 *   (UPIPE_KIND_COUNT).  Kinds are the UPIPE_KIND_* values below.          */
#define UPIPE_KIND_ROPE_TABLE 0
#define UPIPE_KIND_QKV_GEMM 1
#define UPIPE_KIND_ATTN_FWD 2
#define UPIPE_KIND_OPROJ_GEMM 3
#define UPIPE_KIND_DO_GEMM 4
#define UPIPE_KIND_DWO_GEMM 5
#define UPIPE_KIND_ATTN_BWD_DQ 6
#define UPIPE_KIND_ATTN_BWD_DKDV 7
#define UPIPE_KIND_DWQKV_GEMM 8
#define UPIPE_KIND_DX_GEMM 9
#define UPIPE_KIND_DELTA 10
#define UPIPE_KIND_ZERO_ROWS 11
#define UPIPE_KIND_ALST_GU 12     /* MLP gate/up GEMM with the SwiGLU epilogue (forward and backward) */
#define UPIPE_KIND_ALST_GEMM 13   /* MLP and loss GEMMs with one output per row: y, dH, dx, logits, dh */
#define UPIPE_KIND_ALST_WGRAD 14  /* MLP and loss weight gradients, carried across sequence tiles */
#define UPIPE_KIND_CE_ROWS 15     /* softmax rows of the loss */
#define UPIPE_KIND_COUNT 16
int64_t upipe_launch_count(void);
void upipe_profile_enable(int on);
int upipe_profile_read(double* ms, int64_t* launches, int n);

/* Static description of an error code. */
const char* upipe_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* UPIPE_H_ */
