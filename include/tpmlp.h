/*
 * tpmlp: the column->row tensor-parallel MLP block and the vocab-parallel
 * cross-entropy, with T logical shards resident on one GPU.
 *
 * The method (page "一层 MLP 太宽而放不下时怎样切？列并行、行并行与块尾归约",
 * zwjcode.cn, §01-§06):
 *   Z^(r) = X W1^(r) + b1^(r),  H^(r) = act(Z^(r))      column shard r
 *   P^(r) = H^(r) W2^(r)                                 row shard r, [N, D]
 *   Y     = sum_r P^(r) + b2                             block-end SUM, b2 once
 * with W1^(r) = W1[:, r*F/T : (r+1)*F/T] and W2^(r) = W2[r*F/T : (r+1)*F/T, :].
 * Backward (§06): dH^(r) = dY W2^(r)^T, dZ^(r) = dH^(r) * act'(Z^(r)),
 *   dW2^(r) = H^(r)^T dY, dW1^(r) = X^T dZ^(r), dX = sum_r dZ^(r) W1^(r)^T.
 * Cross-entropy (page "unpurerationalist.github.io ... 3.4 TP for Embedding",
 * LM-head bullets; Megatron TP chapter §7.8): per vocab shard k the local max
 * m_k and sum s_k = sum exp(z - m_k); combined m = max_k m_k,
 * S = sum_k s_k exp(m_k - m); loss_n = m + ln S - z[n, t_n].
 *
 * Conventions for every entry point:
 * - All matrices are dense row-major. "[R, C]" means R rows of C elements,
 *   row pitch C elements.
 * - Tensor pointers are DEVICE pointers owned by the caller. Arrays of shard
 *   pointers ("const void* const* W1") are HOST arrays of T device pointers;
 *   the library reads them during the call only.
 * - Element type is `dt` for X, W1, b1, W2, b2, Y, H, Z, dY, dX, dW1, dW2,
 *   db1, db2. TPMLP_BF16 runs the tcgen05 tensor-core path (bf16 storage,
 *   fp32 accumulation, fp32 partial sums); TPMLP_F32 runs a CUDA-core fp32
 *   path (no TF32).
 * - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *   legacy default stream). The returned status reports argument errors and
 *   launch failures synchronously; nothing is launched when an argument is
 *   rejected. Errors found on the device (a bounded wait that expired, a
 *   target id out of range) set a per-device error word that
 *   tpmlp_check_device_error() reads.
 * - The library allocates no device memory. Scratch space is the caller's
 *   `workspace`; tpmlp_workspace_bytes() gives its size.
 * - Output buffers must not overlap input buffers, each other or the
 *   workspace (the one exception is tpmlp_vocab_ce_backward, which may run in
 *   place); overlapping buffers give undefined results.
 * - A workspace serves one call at a time: calls whose GPU work can overlap
 *   (other streams, other host threads without ordering) need separate
 *   workspaces; calls on one stream may share one.
 * - bf16 path alignment: every pointer 16-byte aligned and D % 8 == 0,
 *   (F/T) % 8 == 0 (tensor-memory-access row pitches are multiples of 16
 *   bytes); otherwise TPMLP_ERR_ALIGN.
 * - Two environment variables, read once per process, change how kernels are
 *   launched, never what they compute (results stay within the same
 *   tolerances; integer-valued inputs give the same bits):
 *   TPMLP_PDL=0 launches every kernel fully serialised after the previous
 *   one on its stream (default: programmatic dependent launch);
 *   TPMLP_ALT_ORDER=0 keeps every GEMM tile's K loop ascending and every band
 *   of tiles in one direction (default: odd waves walk K downwards and odd
 *   bands walk their tiles back, for L2 reuse).
 */
#ifndef TPMLP_H
#define TPMLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TPMLP_MAX_SHARDS 16

typedef enum {
    TPMLP_OK = 0,
    TPMLP_ERR_ARG = 1,        /* null pointer, bad enum, negative size; target id out of range (device) */
    TPMLP_ERR_SHAPE = 2,      /* F % T != 0, V % T != 0, T outside [1, TPMLP_MAX_SHARDS], zero width */
    TPMLP_ERR_ALIGN = 3,      /* bf16 path: pointer or row pitch not 16-byte aligned */
    TPMLP_ERR_DTYPE = 4,      /* unknown element type */
    TPMLP_ERR_CUDA = 5,       /* a CUDA runtime or driver call failed */
    TPMLP_ERR_TIMEOUT = 6,    /* a bounded device-side wait expired (device error word) */
    TPMLP_ERR_WORKSPACE = 7   /* workspace NULL or smaller than tpmlp_workspace_bytes() */
} tpmlp_status;

/* RELU: max(z, 0), act'(0) = 0. GELU_TANH: 0.5 z (1 + tanh(sqrt(2/pi)(z + 0.044715 z^3)))
 * (Hendrycks & Gimpel 2016). GELU_ERF: the exact form z Phi(z) = 0.5 z (1 + erf(z/sqrt(2)))
 * that the pages' code uses (nn.GELU(), F.gelu). GELU_SIGMOID: the interview page's
 * approximation z / (1 + exp(-1.702 z)). act' is the exact derivative of each. */
typedef enum {
    TPMLP_ACT_RELU = 0,
    TPMLP_ACT_GELU_TANH = 1,
    TPMLP_ACT_GELU_ERF = 2,
    TPMLP_ACT_GELU_SIGMOID = 3
} tpmlp_act;
typedef enum { TPMLP_F32 = 0, TPMLP_BF16 = 1 } tpmlp_dtype;

/* How the T full-shape partial sums are combined (§04 block-end reduction).
 * PARTIALS: each shard writes its fp32 partial P^(r) to the workspace, then a
 *   vectorised reduce kernel sums them in shard order r = 0..T-1, adds b2 once
 *   and casts (the single-GPU form of the all-reduce).
 * SPLITK: the row GEMM runs its K loop over (r, k) into one fp32 accumulator,
 *   so the shard sum never leaves the tensor-core accumulator; b2 is added
 *   once in the epilogue. No workspace. (For N <= 64 tokens the (r, k) loop
 *   of a tile may be split across a cluster of 2-4 CTAs whose partial
 *   accumulators are added in on-chip shared memory, or, given the optional
 *   scratch of tpmlp_workspace_bytes_balanced, dealt out evenly to all SMs;
 *   see tpmlp_gemm_plan.) */
typedef enum { TPMLP_REDUCE_PARTIALS = 0, TPMLP_REDUCE_SPLITK = 1 } tpmlp_reduce_mode;

typedef enum { TPMLP_OP_FORWARD = 0, TPMLP_OP_BACKWARD = 1 } tpmlp_op;

/* Forward of one block (§01-§05).
 *   X   [N, D]            input, replicated to every shard (read once)
 *   W1  T x [D, F/T]      column shards of W1
 *   b1  T x [F/T] or NULL column shards of b1 (NULL: no b1)
 *   W2  T x [F/T, D]      row shards of W2
 *   b2  [D] or NULL       added exactly once, after the shard sum
 *   Y   [N, D]            output
 *   H   T x [N, F/T]      output: act(Z^(r)) per shard (also the row GEMM's input)
 *   Z   T x [N, F/T] or NULL  output: pre-activation Z^(r), needed by backward
 * Workspace (PARTIALS only): partial P^(r), fp32 [N, D], starts at byte
 * r * round_up(N*D*4, 256); it keeps the partials after the call.
 * Errors: TPMLP_ERR_SHAPE if F % T != 0; TPMLP_ERR_WORKSPACE if mode is
 * PARTIALS and workspace_bytes < tpmlp_workspace_bytes(FORWARD, ...). N = 0
 * is valid and launches nothing. */
tpmlp_status tpmlp_forward(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T, tpmlp_act act,
                           const void* X, const void* const* W1, const void* const* b1,
                           const void* const* W2, const void* b2, void* Y,
                           void* const* H, void* const* Z, tpmlp_reduce_mode mode,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Gated (SwiGLU) form of the block (§08): gate and up projections split by
 * the SAME columns so every shard holds matching channels, the down
 * projection by the matching rows:
 *   G^(r) = X Wg^(r), U^(r) = X Wu^(r), H^(r) = SiLU(G^(r)) * U^(r),
 *   Y = sum_r H^(r) Wd^(r)        SiLU(z) = z / (1 + exp(-z))
 * The gate and up products of a shard run as ONE GEMM whose tiles carry both
 * accumulators, and the epilogue forms H directly.
 *   X   [N, D];  Wg, Wu  T x [D, F/T];  Wd  T x [F/T, D]
 *   Y   [N, D] out;  H  T x [N, F/T] out;  G, U  T x [N, F/T] out, or NULL
 * No biases. Block end, workspace and errors as tpmlp_forward. */
tpmlp_status tpmlp_swiglu_forward(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T,
                                  const void* X, const void* const* Wg, const void* const* Wu,
                                  const void* const* Wd, void* Y, void* const* H, void* const* G,
                                  void* const* U, tpmlp_reduce_mode mode, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Backward of one block (§06), for upstream gradient dY [N, D].
 *   inputs: X, W1 (T x [D, F/T]), W2 (T x [F/T, D]), H and Z (T x [N, F/T],
 *           as written by tpmlp_forward), dY [N, D]
 *   outputs: dX [N, D] (summed over the T column shards), dW1 T x [D, F/T],
 *            dW2 T x [F/T, D], db1 T x [F/T] or NULL, db2 [D] or NULL
 * The workspace holds dZ^(r) (T x [N, F/T] of dt, shard r at byte
 * r * round_up(N*(F/T)*sizeof(dt), 256)) and, in PARTIALS mode after those,
 * the T fp32 dX partials (stride round_up(N*D*4, 256)). N = 0 writes zeros to
 * dW1, dW2, db1, db2. */
tpmlp_status tpmlp_backward(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T, tpmlp_act act,
                            const void* X, const void* const* W1, const void* const* W2,
                            const void* const* H, const void* const* Z, const void* dY,
                            void* dX, void* const* dW1, void* const* dW2,
                            void* const* db1, void* db2, tpmlp_reduce_mode mode,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Block-end reduction alone (§04-§05): Y = sum_{r=0}^{T-1} P^(r) + b2, summed
 * in fp32 in shard order, b2 (element type dt, or NULL) added once, the result
 * stored as dt.
 *   partials  T x [N, D] fp32 (host array of T device pointers)
 *   b2        [D] or NULL
 *   Y         [N, D] */
tpmlp_status tpmlp_block_reduce(tpmlp_dtype dt, int64_t N, int64_t D, int T,
                                const float* const* partials, const void* b2, void* Y,
                                void* stream);

/* Reduce-scatter form of the block end (§04: the all-reduce may become a
 * reduce-scatter so that the output stays sharded by tokens): the same sum
 * Y = sum_r P^(r) + b2 as tpmlp_block_reduce, with rows [r N/T, (r+1) N/T)
 * written to Y_rows[r].
 *   partials  T x [N, D] fp32
 *   b2        [D] (element type dt) or NULL
 *   Y_rows    host array of T device pointers, each [N/T, D] of dt
 * Errors: TPMLP_ERR_SHAPE if N % T != 0. */
tpmlp_status tpmlp_block_reduce_scatter(tpmlp_dtype dt, int64_t N, int64_t D, int T,
                                        const float* const* partials, const void* b2,
                                        void* const* Y_rows, void* stream);

/* tpmlp_forward whose block end is the reduce-scatter: the same arguments,
 * with Y replaced by Y_rows (T device pointers, each [N/T, D]); rank r's row
 * block of Y lands in Y_rows[r]. In SPLITK mode the split-K row GEMM writes
 * each output row straight into its block; in PARTIALS mode the reduce kernel
 * scatters. Errors: those of tpmlp_forward, and TPMLP_ERR_SHAPE if N % T != 0. */
tpmlp_status tpmlp_forward_reduce_scatter(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T,
                                          tpmlp_act act, const void* X, const void* const* W1,
                                          const void* const* b1, const void* const* W2,
                                          const void* b2, void* const* Y_rows, void* const* H,
                                          void* const* Z, tpmlp_reduce_mode mode, void* workspace,
                                          size_t workspace_bytes, void* stream);

/* Vocab-parallel embedding lookup (textbook page §4.2.3 row-parallel
 * embedding; course notes §3.4 "TP for Embedding"): the table [V, Hd] is split
 * by rows into T shards of V/T rows; shard k returns its row for ids in
 * [k V/T, (k+1) V/T) and zeros otherwise, and the sum over shards (the
 * all-reduce) is the embedding. On one GPU every token's row is copied from
 * its owning shard, which is that sum exactly.
 *   ids    [N] int64
 *   table  host array of T device pointers, each [V/T, Hd] of dt
 *   out    [N, Hd] of dt
 * Errors: TPMLP_ERR_SHAPE if V % T != 0. An id outside [0, V) gets a zero row
 * (no shard owns it) and sets TPMLP_ERR_ARG in the device error word. */
tpmlp_status tpmlp_vocab_embedding(tpmlp_dtype dt, int64_t N, int64_t V, int64_t Hd, int T,
                                   const int64_t* ids, const void* const* table, void* out,
                                   void* stream);

/* Vocab-parallel cross-entropy forward (see the header comment).
 *   logits          [N, V] fp32; shard k owns columns [k*V/T, (k+1)*V/T)
 *   targets         [N] int64 in [0, V)
 *   loss_per_token  [N] fp32 out
 *   loss_mean       [1] fp32 out, or NULL: (1/N) sum_n loss_n (fixed order)
 *   argmax          [N] int32 out, or NULL: lowest index of the row maximum
 *   target_owner    [N] int32 out, or NULL: t_n / (V/T)
 * Errors: TPMLP_ERR_SHAPE if V % T != 0. A target outside [0, V) writes NaN
 * for that token and sets TPMLP_ERR_ARG in the device error word. */
tpmlp_status tpmlp_vocab_ce(int64_t N, int64_t V, int T, const float* logits,
                            const int64_t* targets, float* loss_per_token, float* loss_mean,
                            int32_t* argmax, int32_t* target_owner, void* stream);

/* Vocab-parallel cross-entropy backward (course notes §3.6.4, first step):
 *   dlogits[n, v] = grad_scale * (exp(z[n, v] - lse_n) - 1(v = t_n))
 * Every vocab shard's slice needs only the forward's per-token result, no
 * exchange of logits: lse_n = m_n + ln S_n is recovered as
 * loss_per_token[n] + z[n, t_n].
 *   logits          [N, V] fp32 (the forward's input)
 *   targets         [N] int64 in [0, V)
 *   loss_per_token  [N] fp32, as written by tpmlp_vocab_ce for these logits
 *   grad_scale      upstream gradient of each token's loss (1/N for the mean)
 *   dlogits         [N, V] fp32 out; may be the logits buffer itself (in place)
 * Errors: TPMLP_ERR_SHAPE if V % T != 0; a target outside [0, V) writes NaN
 * for that row and sets TPMLP_ERR_ARG in the device error word. */
tpmlp_status tpmlp_vocab_ce_backward(int64_t N, int64_t V, int T, const float* logits,
                                     const int64_t* targets, const float* loss_per_token,
                                     float grad_scale, float* dlogits, void* stream);

/* Size in bytes of the library's own scratch array (see tpmlp_forward_noalloc). */
#define TPMLP_NOALLOC_SCRATCH_BYTES (8u << 20)

/* tpmlp_forward in PARTIALS mode for callers that cannot allocate device
 * memory: the T fp32 partial sums live in a fixed array inside the library
 * instead of a caller workspace. The pages have no counterpart to this call;
 * it exists for callers such as a plug-in inside a host program that owns all
 * device memory, or a latency-bound loop that must not risk a cudaMalloc
 * (which can fail or synchronise the device).
 * - It allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 * - The array is static device memory of TPMLP_NOALLOC_SCRATCH_BYTES (8 MiB);
 *   every GPU that loads the library holds it until the process exits.
 * - Shapes must satisfy T * round_up(N*D*4, 256) <= TPMLP_NOALLOC_SCRATCH_BYTES
 *   (e.g. T = 8, N = 16, D = 12288); larger ones return TPMLP_ERR_WORKSPACE
 *   and launch nothing.
 * - The array serves as a workspace of TPMLP_NOALLOC_SCRATCH_BYTES, so the
 *   launch plans are those tpmlp_forward picks with a workspace of that size:
 *   the few-token GEMMs take the stream-K form only where its scratch fits
 *   behind the partials (small blocks such as N = 8, D = 2048, F/T = 128);
 *   wider few-token shapes such as T = 8, N = 16, D = 12288 run whole tiles
 *   or the cluster K split, which their plans prefer with or without the
 *   scratch.
 * - The first call on each device looks up the array's device address with
 *   that device current; make that first call before any stream capture.
 * - All calls share the one array. Calls whose GPU work can overlap (other
 *   streams, other host threads without ordering) race on it; calls on one
 *   stream are ordered. What an earlier call left in it is never read: the
 *   row GEMM overwrites every partial before the reduce reads it.
 * Arguments, outputs and the other errors are those of tpmlp_forward. */
tpmlp_status tpmlp_forward_noalloc(tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T,
                                   tpmlp_act act, const void* X, const void* const* W1,
                                   const void* const* b1, const void* const* W2, const void* b2,
                                   void* Y, void* const* H, void* const* Z, void* stream);

/* Workspace bytes tpmlp_forward / tpmlp_backward need for these arguments
 * (0 for a forward in SPLITK mode). Returns (size_t)-1 for invalid shapes. */
size_t tpmlp_workspace_bytes(tpmlp_op op, tpmlp_dtype dt, int64_t N, int64_t D, int64_t F, int T,
                             tpmlp_reduce_mode mode);

/* Workspace bytes that also hold the optional fp32 scratch of the bf16 path
 * (bf16 and N >= 1; for other arguments the same as tpmlp_workspace_bytes).
 * The scratch starts at round_up(required, 256) bytes: per-tile arrival
 * counters, then partial accumulators. Given a workspace of at least this
 * size (16-byte aligned; for a SPLITK forward this is the only use of the
 * workspace):
 * - with at most 64 tokens, the GEMMs whose M is the token count (the
 *   column GEMM, the row GEMM, dZ, dX) may run in the stream-K form: every
 *   SM streams the same number of k-blocks, and a tile whose K range two or
 *   more CTAs share is summed through the scratch, in CTA order, by the last
 *   CTA to finish it (no CTA waits for another);
 * - with more, a GEMM whose last wave of tiles would leave SMs idle cuts
 *   those tiles into equal K chunks run side by side and summed the same
 *   way;
 * - the backward's bias gradients (db1, db2), which run after its GEMMs,
 *   sum row chunks of contiguous column ranges into the scratch and then
 *   add the chunks in order.
 * Results do not depend on timing. A smaller workspace (down to the required
 * size) runs the same calls without the scratch, with a different order of
 * fp32 additions. The counters are reset on the call's stream before each
 * use; what the scratch held before is never read. Returns (size_t)-1 for
 * invalid shapes. Library extension; the source pages have no counterpart. */
size_t tpmlp_workspace_bytes_balanced(tpmlp_op op, tpmlp_dtype dt, int64_t N, int64_t D,
                                      int64_t F, int T, tpmlp_reduce_mode mode);

/* Human-readable name of a status code (static string). */
const char* tpmlp_status_str(tpmlp_status s);

/* Synchronizes `stream`, then reads and clears the current device's error
 * word. Returns TPMLP_OK, TPMLP_ERR_TIMEOUT or TPMLP_ERR_ARG (device-side
 * findings), or TPMLP_ERR_CUDA if the synchronization itself failed. */
tpmlp_status tpmlp_check_device_error(void* stream);

/* Upper bound, in nanoseconds, on every spin-wait inside the tensor-core
 * kernels (default 2e9). A wait that runs out sets TPMLP_ERR_TIMEOUT in the
 * device error word, the kernel drains its own copies, frees its tensor
 * memory and returns. */
void tpmlp_set_wait_timeout_ns(uint64_t ns);

/* Failure-detection self test: launches one kernel whose thread waits, with
 * the bounded wait above, on a barrier that nothing completes, so the wait
 * always runs out after `timeout_ns`. The caller then sees TPMLP_ERR_TIMEOUT
 * from tpmlp_check_device_error(). */
tpmlp_status tpmlp_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

/* Failure-detection self test of the tensor-core GEMM (page "一层 MLP 太宽而放
 * 不下时怎样切？", §11: a collective that waits forever, found by numbering
 * and timing the waits). While `role` is 1, 2 or 3, every bf16 GEMM launch
 * makes that role of each of its CTAs (1: the epilogue warps, 2: the
 * MMA-issuing thread, 3: the TMA-issuing thread) first wait, with the bounded
 * wait of tpmlp_set_wait_timeout_ns, on a barrier that nothing completes.
 * The wait runs out; the kernel records TPMLP_ERR_TIMEOUT in the device
 * error word, raises its abort flag, and every role leaves through the same
 * exit as after a real timeout: the copies and MMAs already issued are
 * waited for, tensor memory is freed, the CTAs of a cluster leave together.
 * The outputs of such a launch are undefined. 0 (the default) turns the stall
 * off; other values return TPMLP_ERR_ARG. Process-wide; set it only while no
 * other thread launches GEMMs. Library extension for tests. */
tpmlp_status tpmlp_selftest_gemm_stall(int role);

/* ---- instrumentation ---------------------------------------------------- */

/* Launch configuration the bf16 tensor-core GEMM chooses on the current
 * device for one GEMM of the block: M x N outputs per group, reduction
 * length K per group, G groups (shards), fold = 1 when the K loop runs over
 * all G groups into one output (the split-K shard sum), dual = 1 for the
 * gated GEMM (N counts outputs), balanced = 1 when the call's workspace holds
 * the few-token scratch (tpmlp_workspace_bytes_balanced). Writes the tile's
 * accumulator columns (128, 192 or 256), the CTAs that issue one MMA (1, or 2 for
 * a CTA pair) and the K split: the CTAs of a cluster that share one tile's
 * K range (1 = no split; 2-4 for folded GEMMs with M <= 64, where the weights
 * stream from HBM and the tiles are fewer than the SMs), or 0 for the
 * stream-K form (M <= 64 with the scratch). A query: launches nothing.
 * Returns TPMLP_ERR_ARG for a null output pointer, TPMLP_ERR_SHAPE for sizes
 * < 1 or above 2^31 - 1 or G outside [1, TPMLP_MAX_SHARDS], TPMLP_ERR_CUDA
 * when the device queries fail. Library introspection; the source pages
 * have no counterpart. */
tpmlp_status tpmlp_gemm_plan(int64_t M, int64_t N, int64_t K, int G, int fold, int dual,
                             int balanced, int* bn, int* mma_ctas, int* ksplit);

/* Number of kernels this library has launched in this process. */
int64_t tpmlp_launch_count(void);

typedef struct {
    char name[48];       /* kernel kind, e.g. "tc_gemm_col_act" */
    int64_t launches;
    double total_ms;     /* sum of per-launch CUDA-event durations */
} tpmlp_kernel_timing;

/* When on, every launch is bracketed by CUDA events recorded on the stream
 * the kernel is launched on. */
void tpmlp_timing_enable(int on);
/* Waits for the recorded events and writes up to max_entries aggregated
 * per-kernel records; returns the number written (-1 on a CUDA error). */
int tpmlp_timing_read(tpmlp_kernel_timing* out, int max_entries);
/* Drops all recorded events and aggregates. */
void tpmlp_timing_reset(void);

#ifdef __cplusplus
}
#endif

#endif /* TPMLP_H */
