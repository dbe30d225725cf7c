/*
 * tpmlp.h — C ABI of the GB300 (sm_103a) tensor-parallel / sequence-parallel
 * Transformer MLP block.
 *
 * The block (math convention A ∈ R^{h×f}, B ∈ R^{f×h}):
 *
 *     Z = act(X·A)·B
 *
 * with A split by columns into tp tensor shards and B split by rows
 * ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §2 column-parallel 与
 * row-parallel 的配合, and its f/g table).  On one GPU the tp shards are logical
 * partitions of one device's memory; the communication operators become
 * on-device kernels:
 *
 *   g  (forward all-reduce)     -> fixed-order float32 sum of the tp partial sums,
 *                                  rounded to the storage type;
 *   f  (backward all-reduce)    -> the same sum over the input-gradient partials;
 *   SP all-gather along dim 0   -> concatenation of the tp sequence chunks;
 *   SP reduce-scatter on dim 0  -> the shard sum, chunk i written to shard i.
 *
 * ("Sequence Parallel 与 Context Parallel", §SP：all-gather 进、reduce-scatter 出.)
 *
 * Layouts (all row-major, all in device memory unless stated otherwise):
 *   activations  [s, b, h], sequence-first; flattened to [M, h], M = s·b, row
 *                m = s_idx·b + b_idx ("Tensor Parallelism（TP）与 Sequence
 *                Parallelism（SP）", §1 sequence-first layout);
 *   W1 = Aᵀ      [f, h]   (SwiGLU: [2F, h], rows [0,F) gate, rows [F,2F) up);
 *                tensor shard i = rows [i·f/tp, (i+1)·f/tp) (SwiGLU: the gate rows
 *                and the matching up rows);
 *   W2 = Bᵀ      [h, f];  tensor shard i = columns [i·f/tp, (i+1)·f/tp);
 *   U, Y, dU     [M, f] saved pre-activation, activation output and its gradient
 *                (SwiGLU: U and dU are [M, 2F] laid out gate|up, Y is [M, F]);
 *                shard i = column block i;
 *   SP chunks    sequence chunk i = rows [i·s/tp, (i+1)·s/tp) of dim 0, each a
 *                separate contiguous [s/tp, b, h] buffer.
 *
 * Ownership and conventions:
 *   - The caller owns every buffer.  The library never allocates device memory;
 *     scratch space is the caller's workspace (tpmlp_workspace_size()).
 *   - Pointer arrays (x, z, dz, dx, shards, out) are HOST arrays of device
 *     pointers; the library copies the pointers before returning.
 *   - Every call enqueues work on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and returns without synchronising.
 *   - Arguments are validated on the host before anything is launched; a
 *     non-zero status means nothing was enqueued (except TPMLP_ERR_CUDA, which
 *     reports a failed launch).  tpmlp_last_error() then describes the problem.
 *   - No exceptions cross the ABI; no kernel traps.  Kernels that wait on an
 *     on-chip barrier give up after a bounded time and record
 *     TPMLP_ERR_TIMEOUT in a device status word (tpmlp_device_status()).
 *   - Outputs must not alias inputs or each other.
 *
 * Requirements of the tensor-core path (dtype TPMLP_F16 / TPMLP_BF16):
 *   h and f/tp multiples of 8, every pointer 16-byte aligned.  Otherwise the
 *   call returns TPMLP_ERR_UNSUPPORTED.  The TPMLP_F32 path (CUDA-core float32)
 *   has no shape or alignment requirement beyond 4-byte alignment.
 */
#ifndef TPMLP_H_
#define TPMLP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TPMLP_ABI_VERSION 4
#define TPMLP_MAX_TP 64

typedef enum tpmlp_status {
  TPMLP_OK = 0,
  TPMLP_ERR_INVALID_ARG = -1,   /* null pointer, negative size, bad enum, tp out of range */
  TPMLP_ERR_NOT_DIVISIBLE = -2, /* s % tp != 0 under SP, or f % tp != 0 */
  TPMLP_ERR_UNSUPPORTED = -3,   /* shape/alignment outside the tensor-core path */
  TPMLP_ERR_WORKSPACE = -4,     /* workspace smaller than tpmlp_workspace_size() */
  TPMLP_ERR_CUDA = -5,          /* a CUDA runtime call or launch failed */
  TPMLP_ERR_TIMEOUT = -6        /* a kernel's bounded on-chip wait expired */
} tpmlp_status;

typedef enum tpmlp_dtype { TPMLP_F32 = 0, TPMLP_F16 = 1, TPMLP_BF16 = 2 } tpmlp_dtype;

typedef enum tpmlp_act {
  TPMLP_ACT_GELU_TANH = 0, /* 0.5x(1 + tanh(√(2/π)(x + 0.044715x³))) */
  TPMLP_ACT_SWIGLU = 1,    /* silu(gate) ⊙ up, fc1 has 2F outputs */
  TPMLP_ACT_IDENTITY = 2,  /* for exact-arithmetic checks */
  TPMLP_ACT_RELU = 3       /* the two-layer example's activation */
} tpmlp_act;

typedef enum tpmlp_reduce {
  /* fc2 (and fc1's input gradient) write one float32 partial sum per tensor
   * shard into the workspace; a separate kernel sums them in shard order
   * 0..tp-1 in float32 and rounds once: the literal g / f-backward all-reduce. */
  TPMLP_REDUCE_PARTIALS = 0,
  /* the shard sum is folded into the GEMM: one float32 accumulator runs over
   * the K ranges of shards 0..tp-1 in order and the epilogue rounds once.
   * A different, equally valid summation order; no partial-sum traffic. */
  TPMLP_REDUCE_FUSED = 1
} tpmlp_reduce;

/* ---------------------------------------------------------------------------
 * tpmlp_workspace_size — bytes of device workspace that tpmlp_forward and
 * tpmlp_backward need for these arguments (the maximum of the two).
 *   SP on:   the gathered input [M,h] and, in backward, the gathered dZ [M,h]
 *            (neither when every SP chunk is a whole number of 128-row
 *            blocks: the tensor-core GEMMs then read the chunks in place);
 *   PARTIALS: tp float32 partial sums [tp, M, h].
 * tpmlp_forward_workspace_size gives the forward's own need (no dZ slot);
 * tpmlp_forward accepts a workspace of that size.
 * Both return 0 for invalid arguments (tpmlp_last_error() says why) or when no
 * workspace is needed.  The workspace must be 256-byte aligned.
 * ------------------------------------------------------------------------- */
size_t tpmlp_workspace_size(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp,
                            int dtype, int act, int mode);
size_t tpmlp_forward_workspace_size(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp,
                                    int dtype, int act, int mode);

/* ---------------------------------------------------------------------------
 * tpmlp_forward — forward pass of the block.
 *   Column-parallel fc1 + local activation: U_i = X·A_i, Y_i = act(U_i)
 *   ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §3 column 与 row 的切分
 *   选择: fc1 column-parallel, activation local); row-parallel fc2:
 *   P_i = Y_i·B_i; g: Z = Σ_i P_i (SP off) or reduce-scatter (SP on).
 *
 *   x    sp ? tp pointers to [s/tp,b,h] : 1 pointer to [s,b,h]      (input)
 *   w1   [f,h] (SwiGLU [2F,h])                                      (input)
 *   w2   [h,f]                                                      (input)
 *   u    [M,f] (SwiGLU [M,2F]) pre-activation, saved for backward  (output)
 *   y    [M,f] (SwiGLU [M,F]) activation output                    (output)
 *   z    sp ? tp pointers to [s/tp,b,h] : 1 pointer to [s,b,h]      (output)
 *   ws   workspace of ws_bytes >= tpmlp_workspace_size(...)
 * For SwiGLU, f is the ffn width F.
 * ------------------------------------------------------------------------- */
int tpmlp_forward(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype,
                  int act, int mode, const void* const* x, const void* w1, const void* w2,
                  void* u, void* y, void* const* z, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * tpmlp_backward — backward pass given dZ.
 *   g backward: identity (SP: all-gather dZ); fc2 input gradient
 *   dY_i = dZ·B_iᵀ with the activation derivative fused: dU_i = act'(U_i)⊙dY_i;
 *   fc2 weight gradient dB_i = Y_iᵀ·dZ (stored dW2 = dBᵀ, [h,f]);
 *   fc1 weight gradient dA_i = Xᵀ·dU_i (stored dW1 = dAᵀ, [f,h]; SP re-gathers X);
 *   f backward: dX = Σ_i dU_i·A_iᵀ (SP: reduce-scatter)
 *   ("tensor-parallelism-matrix-split", §Backward：为什么有些梯度需要求和 and
 *   §Backward 的通信; "Sequence Parallel 与 Context Parallel", §SP backward).
 *
 *   x, w1, w2     as in tpmlp_forward                                (input)
 *   u, y          the forward's saved U and Y                        (input)
 *   dz            sp ? tp pointers to [s/tp,b,h] : 1 pointer [s,b,h]  (input)
 *   dx            same layout as dz                                  (output)
 *   dw1 [f,h] (SwiGLU [2F,h]), dw2 [h,f]   weight gradients, overwritten (output)
 *   du  [M,f] (SwiGLU [M,2F])              pre-activation gradient   (output)
 * ------------------------------------------------------------------------- */
int tpmlp_backward(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype,
                   int act, int mode, const void* const* x, const void* w1, const void* w2,
                   const void* u, const void* y, const void* const* dz, void* const* dx,
                   void* dw1, void* dw2, void* du, void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * tpmlp_backward_main_grad — tpmlp_backward with the weight gradients
 * accumulated into float32 master-gradient buffers, Megatron's
 * gradient_accumulation_fusion ("Tensor Parallelism（TP）与 Sequence Parallelism
 * （SP）", §这组文档怎么读, the ColumnParallelLinear/RowParallelLinear row:
 * gradient_accumulation_fusion, main_grad):
 *   main_grad_w1 [f,h] (SwiGLU [2F,h]) float32  += dW1   (input and output)
 *   main_grad_w2 [h,f]                 float32  += dW2   (input and output)
 * Each weight-gradient GEMM keeps its float32 accumulator and adds it to
 * main_grad in its epilogue (one float32 add per element, no rounding to the
 * storage type first), so gradients of several micro-batches sum in float32.
 * Every other argument, output and rule is that of tpmlp_backward; the two
 * main_grad buffers must be 16-byte aligned.  s = 0 leaves them unchanged.
 * ------------------------------------------------------------------------- */
int tpmlp_backward_main_grad(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype,
                             int act, int mode, const void* const* x, const void* w1,
                             const void* w2, const void* u, const void* y, const void* const* dz,
                             void* const* dx, float* main_grad_w1, float* main_grad_w2, void* du,
                             void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * tpmlp_split_dim0 — shard i := full[i·s/tp : (i+1)·s/tp] (each [s/tp,b,h]);
 * an exact copy ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §1:
 * the split takes a contiguous slice of the outermost dimension).
 *   full    [s,b,h]                            (input)
 *   shards  host array of tp device pointers   (outputs)
 * s % tp != 0 -> TPMLP_ERR_NOT_DIVISIBLE (the page's divisibility assertion).
 * ------------------------------------------------------------------------- */
int tpmlp_split_dim0(const void* full, void* const* shards, int64_t s, int64_t b, int64_t h,
                     int tp, int dtype, void* stream);

/* ---------------------------------------------------------------------------
 * tpmlp_gather_dim0 — the SP all-gather: full = concat(shards) along dim 0;
 * an exact copy (same page, §1, gather along the first dimension).
 *   shards  host array of tp device pointers to [s/tp,b,h]   (inputs)
 *   full    [s,b,h]                                          (output)
 * ------------------------------------------------------------------------- */
int tpmlp_gather_dim0(const void* const* shards, void* full, int64_t s, int64_t b, int64_t h,
                      int tp, int dtype, void* stream);

/* ---------------------------------------------------------------------------
 * tpmlp_reduce_scatter_dim0 — g's all-reduce (scatter = 0) or the SP
 * reduce-scatter (scatter = 1) over float32 partial sums:
 *   R = ((P_0 + P_1) + P_2) + … + P_{tp-1}   in float32, round-to-nearest-even,
 * then rounded once to `dtype` (nearest-even).
 *   partials  float32 [tp, s, b, h] contiguous                       (input)
 *   out       scatter ? tp pointers to [s/tp,b,h] : 1 pointer to [s,b,h] (output)
 * ("Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §5 table: g forward
 * all-reduce, SP g forward reduce-scatter.)
 * ------------------------------------------------------------------------- */
int tpmlp_reduce_scatter_dim0(const float* partials, void* const* out, int64_t s, int64_t b,
                              int64_t h, int tp, int scatter, int dtype, void* stream);

/* ---------------------------------------------------------------------------
 * tpmlp_forward_noalloc — tpmlp_forward for callers that cannot supply a
 * device workspace.  (The pages have no counterpart; this is a library
 * convenience.)
 *
 * Who needs it: code whose GPU memory belongs to a memory manager that does not
 * let it allocate where it calls the block, and latency-critical loops that
 * must not pay cudaMalloc's implicit device-wide synchronisation.  Arguments
 * and results are those of tpmlp_forward without ws / ws_bytes; the caller
 * still passes every input and output buffer.
 *
 * Scratch: a fixed array of TPMLP_NOALLOC_SCRATCH_BYTES (64 MiB) compiled into
 * the library as device memory.  Every GPU that loads the library holds it
 * until the process exits.  The call allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine).
 *   - Sizes whose forward workspace (tpmlp_forward_workspace_size) exceeds
 *     the scratch are rejected with TPMLP_ERR_WORKSPACE and a message giving
 *     both sizes; use tpmlp_forward with a caller workspace for those.
 *   - The first call in each CUDA context of a device — the first call on the
 *     device, and the first after the caller replaced the context (e.g. by
 *     cudaDeviceReset) — looks up the scratch array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture on the device.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Nothing in it needs to start at zero (each call writes every scratch
 *     byte it reads).  Calls that can overlap on the GPU — on different
 *     streams, or from several host threads — race on the scratch; serialise
 *     them (one stream) or use tpmlp_forward with separate workspaces.
 * ------------------------------------------------------------------------- */
#define TPMLP_NOALLOC_SCRATCH_BYTES (64ull << 20)

int tpmlp_forward_noalloc(int64_t s, int64_t b, int64_t h, int64_t f, int tp, int sp, int dtype,
                          int act, int mode, const void* const* x, const void* w1,
                          const void* w2, void* u, void* y, void* const* z, void* stream);

/* ---------------------------------------------------------------------------
 * The sequence-parallel region around the block ("Sequence Parallel 与 Context
 * Parallel", §SP：all-gather 进、reduce-scatter 出: LayerNorm → fc1 → act → fc2 →
 * dropout, LayerNorm and dropout on the [s/tp, b, h] sequence chunks).  Every
 * tensor argument below is a HOST array of tp device pointers to the chunks
 * [s/tp, b, h] (row m of the full sequence is chunk m / (s/tp·b)); tp = 1 works
 * on an unsplit tensor.  s % tp != 0 -> TPMLP_ERR_NOT_DIVISIBLE.
 *
 * tpmlp_sp_layernorm_forward — y = (x − μ)/√(σ² + eps)·γ + β per token over h
 * (σ² without Bessel's correction).  gamma, beta [h] in dtype; mean, rstd [s·b]
 * float32 outputs kept for the backward.  The y chunks are what tpmlp_forward
 * takes as its x chunks: its fc1 reads them in place.
 * ------------------------------------------------------------------------- */
int tpmlp_sp_layernorm_forward(const void* const* x, const void* gamma, const void* beta, float eps,
                               void* const* y, float* mean, float* rstd, int64_t s, int64_t b,
                               int64_t h, int tp, int dtype, void* stream);

/* Bytes of float32 workspace tpmlp_sp_layernorm_backward needs (2·⌈s·b/8⌉·h·4). */
size_t tpmlp_sp_layernorm_backward_workspace(int64_t s, int64_t b, int64_t h);

/* ---------------------------------------------------------------------------
 * tpmlp_sp_layernorm_backward — given dy = ∂L/∂y:
 *   dx = rstd·(g − mean_h(g) − x̂·mean_h(g·x̂)),  g = dy·γ, x̂ = (x − μ)·rstd;
 *   written to dx (accumulate = 0) or added to it (accumulate = 1: dx holds the
 *   residual branch's gradient on entry);
 *   dgamma[h] = Σ_tokens dy·x̂, dbeta[h] = Σ_tokens dy (float32, overwritten;
 *   partial sums over fixed sets of tokens, added in a fixed order: the same
 *   bits on every call with the same shapes on the same device).
 * ws: tpmlp_sp_layernorm_backward_workspace() bytes, 16-byte aligned.
 * ------------------------------------------------------------------------- */
int tpmlp_sp_layernorm_backward(const void* const* x, const void* gamma, const float* mean,
                                const float* rstd, const void* const* dy, void* const* dx,
                                int accumulate, float* dgamma, float* dbeta, void* ws,
                                size_t ws_bytes, int64_t s, int64_t b, int64_t h, int tp, int dtype,
                                void* stream);

/* ---------------------------------------------------------------------------
 * tpmlp_sp_residual_dropout_forward — out = r + keep·z/(1 − p) on the chunks
 * after the reduce-scatter; keep: tp chunks of s/tp·b·h bytes, 0 = dropped,
 * nonzero = kept (the caller draws the mask); 0 <= p < 1.
 * tpmlp_sp_residual_dropout_backward — dz = keep·dout/(1 − p); the residual
 * branch's gradient is dout itself.
 * ------------------------------------------------------------------------- */
int tpmlp_sp_residual_dropout_forward(const void* const* r, const void* const* z,
                                      const uint8_t* const* keep, float p, void* const* out,
                                      int64_t s, int64_t b, int64_t h, int tp, int dtype, void* stream);
int tpmlp_sp_residual_dropout_backward(const void* const* dout, const uint8_t* const* keep, float p,
                                       void* const* dz, int64_t s, int64_t b, int64_t h, int tp,
                                       int dtype, void* stream);

/* Thread-local description of the last non-OK status returned on this thread. */
const char* tpmlp_last_error(void);

/* ---------------------------------------------------------------------------
 * tpmlp_device_status — synchronises `stream`, then returns the device status
 * word of the current device: TPMLP_OK, or TPMLP_ERR_TIMEOUT if a kernel's
 * bounded wait expired since the last reset.  reset != 0 clears it afterwards.
 * Returns TPMLP_ERR_CUDA if the synchronisation itself fails.
 * ------------------------------------------------------------------------- */
int tpmlp_device_status(void* stream, int reset);

/* Upper bound, in nanoseconds, of any single on-chip wait in the library's
 * kernels (default 2e9).  Values below 1e6 are raised to 1e6. */
void tpmlp_set_wait_timeout_ns(uint64_t ns);

/* ---------------------------------------------------------------------------
 * tpmlp_wait_timeout_selftest — enqueues one single-thread kernel that waits on
 * a shared-memory barrier no one ever arrives at, with a limit of timeout_ns.
 * The wait must expire: afterwards tpmlp_device_status() reports
 * TPMLP_ERR_TIMEOUT and the context stays usable.  Tests the bounded-wait
 * machinery without faulting or hanging the GPU.
 * ------------------------------------------------------------------------- */
int tpmlp_wait_timeout_selftest(uint64_t timeout_ns, void* stream);

/* ---------------------------------------------------------------------------
 * Tensor-parallel self-attention block ("tensor-parallel-megatron" reading,
 * attention section; "Tensor Parallelism（TP）与 Sequence Parallelism（SP）", §2
 * "attention 的道理是一样的"): the fused QKV projection is column-parallel with
 * whole heads per tensor shard, each head computes softmax(Q·Kᵀ/√d)·V on its
 * shard, and the output projection is row-parallel with one reduction at the
 * exit (g; the reduce-scatter under SP).  As in the MLP block the tp shards are
 * partitions of one device's buffers and the shard sums are folded into the
 * GEMM accumulators (the fused mode).
 *
 * Grouped-query attention ("tensor-parallel-megatron" reading, attention
 * section): kv_heads key/value heads (query groups) G, each shared by
 * r = heads/G query heads; kv_heads = heads is multi-head attention.  The fused
 * weight is [h + 2·h_kv, h] (h_kv = G·d), interleaved per group as the reading
 * prints it, [q₁ q₂ k₁ v₁ | q₃ q₄ k₂ v₂ | …]: group g holds rows
 * [g·(r+2)·d, (g+1)·(r+2)·d), its r query heads' q rows, then its k rows, then
 * its v rows.  Query head j belongs to group j / r.  Tensor shard i owns groups
 * [i·G/tp, (i+1)·G/tp) — contiguous rows of Wqkv, whole heads.
 *
 * Shapes: head width d = h/heads of 128 or 96 (else TPMLP_ERR_UNSUPPORTED);
 * heads % kv_heads == 0 and kv_heads % tp == 0 (else TPMLP_ERR_NOT_DIVISIBLE:
 * a shard must hold whole groups), s % tp == 0 under SP; float16 or bfloat16
 * storage (float32 -> TPMLP_ERR_UNSUPPORTED); b < 65536, s ≤ 65535·128.
 * Activations are sequence-first [s, b, ·] (row m = t·b + bi); every pointer
 * 16-byte aligned.  W = h + 2·h_kv below.
 *   x      sp ? tp chunk pointers [s/tp, b, h] : one pointer [s, b, h]
 *   wqkv   [W, h], rows in the group layout above
 *   wo     [h, h]: shard i owns the columns of its query heads
 *   qkv    [s·b, W] output of the forward, input of the backward (columns in
 *          the group layout)
 *   o      [s·b, h] attention output before the projection (query head j in
 *          columns d·j …); forward output, backward input
 *   lse    [b][heads][s_pad] float32, s_pad = s rounded up to a multiple of 128:
 *          log2 Σ_u 2^(x_tu) of each query row's scaled scores
 *          x = (q·k/√d)·log2(e); forward output, backward input
 *   z, dz, dx  like x
 *   dwqkv, dwo  weight gradients (overwritten), storage type
 *   dqkv   [s·b, W], dout [s·b, h]: backward scratch and outputs (dQKV, dO); a
 *          key/value head's gradient is the sum over its query heads
 * causal = 1 applies the decoder mask (key u visible to query t iff u ≤ t);
 * causal = 0 is the unmasked formula.  ws: tpmlp_attn_workspace_size() bytes
 * (same causal flag as the calls), 256-byte aligned: the gathered X and dZ when
 * SP chunks of s/tp·b rows are not whole multiples of 128 rows (the forward
 * needs only the gathered X), then Δ and −lse2, each [b][heads][s_pad] float32,
 * then the backward's 16-bit dSᵀ tiles: b·heads·T tiles of 16 KB (128 keys × 64
 * queries), T = nk·nq − nk·(nk−1) under the causal mask, else nk·nq, with
 * nk = ⌈s/128⌉ and nq = ⌈s/64⌉ (≈ b·heads·s²·2 bytes unmasked, half causal),
 * then with grouped-query attention (kv_heads < heads) the float32 dK/dV
 * partials of every group's r query heads, r·s·b·kv_heads·2·d·4 bytes, added in
 * query-head order by the backward (so results stay deterministic).
 * Every on-chip wait is bounded (tpmlp_set_wait_timeout_ns): an expired wait
 * is reported through tpmlp_device_status() as TPMLP_ERR_TIMEOUT.  Results
 * are deterministic (no atomics).
 * Environment: TPMLP_ATTN_FWD_PAIR=1 (read at every forward call) runs the
 * forward's core for head width 128 as CTA pairs (2-SM MMAs, 512 query rows a
 * pair) instead of one CTA per 256 query rows; same results within rounding,
 * measured slower, off by default.  With grouped-query attention the backward
 * splits each group's query heads over kv_split CTAs per key tile (the
 * smallest divisor of heads/kv_heads giving six waves of CTAs on the device)
 * and adds their float32 dK, dV partials in chunk order; TPMLP_ATTN_KV_SPLIT=n
 * (read at every backward call) sets the split when n divides heads/kv_heads.
 * tpmlp_attn_workspace_size covers the largest split.
 * ------------------------------------------------------------------------- */
size_t tpmlp_attn_workspace_size(int64_t s, int64_t b, int64_t h, int heads, int kv_heads, int tp, int sp,
                                 int dtype, int causal);
int tpmlp_attn_forward(int64_t s, int64_t b, int64_t h, int heads, int kv_heads, int tp, int sp, int dtype,
                       int causal, const void* const* x, const void* wqkv, const void* wo, void* qkv, void* o,
                       float* lse, void* const* z, void* ws, size_t ws_bytes, void* stream);
int tpmlp_attn_backward(int64_t s, int64_t b, int64_t h, int heads, int kv_heads, int tp, int sp, int dtype,
                        int causal, const void* const* x, const void* wqkv, const void* wo, const void* qkv,
                        const void* o, const float* lse, const void* const* dz, void* const* dx,
                        void* dwqkv, void* dwo, void* dqkv, void* dout, void* ws, size_t ws_bytes,
                        void* stream);

/* ---------------------------------------------------------------------------
 * Launch accounting (for benchmarks).  Between tpmlp_profile_start() and
 * tpmlp_profile_stop(), every kernel the library launches on this thread is
 * bracketed by two CUDA events recorded on its launching stream, and the
 * algorithmic work of the launch is added up per kernel kind:
 *   kind 0  tensor-core GEMM      work = 2·M·N·K FLOPs
 *   kind 1  float32 CUDA-core GEMM work = 2·M·N·K FLOPs
 *   kind 2  dim-0 chunk copy      work = bytes read + bytes written
 *   kind 3  shard sum             work = tp·n·4 bytes read + n·elem bytes written
 *   kind 4  SP-region kernels     work = bytes read + bytes written (LayerNorm,
 *                                 dropout + residual)
 *   kind 5  attention core        work = matmul FLOPs over the visible (query,
 *                                 key) pairs: 4·pairs·128·heads·b forward,
 *                                 8·pairs·128·heads·b backward (the recomputed
 *                                 scores are not counted)
 * tpmlp_profile_stop() synchronises the recorded events and fills `out`
 * (out may be NULL to discard).  Recording stays off unless started.
 * ------------------------------------------------------------------------- */
#define TPMLP_PROFILE_KINDS 6
typedef struct tpmlp_profile {
  int launches[TPMLP_PROFILE_KINDS];
  double ms[TPMLP_PROFILE_KINDS];
  double work[TPMLP_PROFILE_KINDS];
} tpmlp_profile;

int tpmlp_profile_start(void);
int tpmlp_profile_stop(tpmlp_profile* out);

/* TPMLP_ABI_VERSION of the built library. */
int tpmlp_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TPMLP_H_ */
