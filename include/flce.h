/*
 * flce.h — fused LM-head projection + cross-entropy on GB300 (sm_103a).
 *
 * The operation is the last step of a language-model training step, as written
 * out in "What-Each-Parallelism-Actually-Shards" §1.4: hidden states X[N,H]
 * (N = B*S tokens) are projected by the LM head W[V,H] to logits
 * z[N,V] = X W^T, and the loss is the cross-entropy of those logits against
 * integer labels, with rows whose label equals ignore_index left out (the fused
 * call in §7.4 passes ignore_index = -100).  §7.4 describes the fused form this
 * library implements: keep a running log-sum-exp over the vocabulary, take only
 * the target token's logit, recompute logits in the backward pass, and never
 * write the [N,V] logits to global memory.
 *
 * Definitions (i = row, j = vocabulary id, y_i = label):
 *   lse_i  = log sum_j exp(z_ij)
 *   loss_i = (lse_i - z_{i,y_i}) * valid_i,   valid_i = [y_i != ignore_index]
 *   loss   = sum_i loss_i / n_valid  (FLCE_REDUCTION_MEAN; 0 when n_valid = 0)
 *          = sum_i loss_i            (FLCE_REDUCTION_SUM)
 *          = loss_i per row          (FLCE_REDUCTION_NONE; then `loss` points to N floats
 *                                     and the upstream gradient is one g_i per row)
 *   G_ij   = s * (exp(z_ij - lse_i) - [j = y_i]) * valid_i,
 *            s = g / n_valid (mean), g (sum) or g_i (none), g = upstream gradient of loss
 *   With shift = 1 (the causal next-token shift of §7.4's call), the label of
 *   row i is labels[i + 1], and the last row of each sequence of seq_len rows
 *   is ignored: position t of a sequence predicts the token at t + 1.
 *   dX = G W   (bf16 [N,H]),   dW = G^T X   (bf16 [V,H])
 *
 * Conventions for every call:
 *   - X, W, dX, dW are bf16, dense row-major, H contiguous.  labels is int32.
 *     loss, lse, grad_loss are fp32.  All data pointers are DEVICE pointers
 *     owned by the caller; the library never allocates or frees memory.
 *   - ws / ws_bytes: caller-owned device workspace, 256-byte aligned (the
 *     alignment of the regions the library lays out in it), of at least
 *     flce_workspace_bytes(p) bytes: O(N*(C + H)) for a fixed chunk width C,
 *     independent of V.  The row-chunk calls (flce_fwd_bwd_rowchunk,
 *     flce_soft_fwd_bwd_rowchunk) keep a chunk of the vocabulary gradient instead and
 *     take flce_workspace_bytes_rowchunk(p); the vocabulary-shard calls take
 *     flce_shard_workspace_bytes(p, shard).  The workspace is the only extra
 *     device memory the library touches.  Calls that share a workspace must be
 *     ordered on one stream.
 *   - Requirements: n >= 0, h >= 8, v >= 1, h % 8 == 0 (16-byte row pitch for
 *     the tensor-memory-access engine), X / W / dX / dW 16-byte aligned,
 *     labels / lse 4-byte aligned.  Violations return an error and launch
 *     nothing.
 *   - An empty batch (n = 0) has no valid row: the loss is 0 (mean and sum),
 *     dW is 0, nothing else has an element, and the pointers to per-row data
 *     (X, labels, lse, dX, per-row losses, top-k outputs, soft targets) may be
 *     NULL.  The workspace then needs 256 bytes (the status word).
 *   - stream: a cudaStream_t (NULL = legacy default stream).  Every call is
 *     asynchronous on it.  Host-detectable errors return immediately.
 *     Errors found on the device (a label outside [0,V) that is not
 *     ignore_index; a bounded wait inside a kernel that ran out) are recorded
 *     in the workspace's status word; read them with flce_read_device_status.
 *     After any error the outputs are unspecified.
 *   - Thread safety: calls on different workspaces may run concurrently.
 */
#ifndef FLCE_H
#define FLCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                       /* same type as cudaStream_t's target */
typedef struct CUstream_st* flce_stream_t;

typedef enum {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARGUMENT = 1,    /* null pointer, bad enum, n < 0, h/v < 1 */
  FLCE_ERR_UNSUPPORTED_SHAPE = 2,   /* h % 8 != 0, h < 8, or sizes beyond int32 tile coordinates */
  FLCE_ERR_MISALIGNED = 3,          /* a pointer breaks the alignment rules above */
  FLCE_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes below the call's workspace size (flce_workspace_bytes(p), or
                                       the row-chunk / shard / top-k / host-buffer size for those calls) */
  FLCE_ERR_LABEL_OUT_OF_RANGE = 5,  /* device: some label not in [0,V) and not ignore_index */
  FLCE_ERR_TIMEOUT = 6,             /* device: a bounded pipeline wait gave up (no hang, no trap) */
  FLCE_ERR_CUDA = 7,                /* a CUDA runtime/driver call failed, or no sm_100-family GPU */
  FLCE_ERR_NO_DEVICE_STATUS = 8,    /* flce_read_device_status could not read the word */
  FLCE_ERR_EXCEEDS_STATIC_SCRATCH = 9, /* flce_forward_noalloc: n above its fixed maximum */
  FLCE_ERR_BOUNDS = 10              /* device, debug build only: an index or TMA coordinate failed its check */
} flce_status_t;

typedef enum { FLCE_REDUCTION_MEAN = 0, FLCE_REDUCTION_SUM = 1, FLCE_REDUCTION_NONE = 2 } flce_reduction_t;

typedef struct {
  int64_t n;             /* rows (tokens), N = B*S */
  int64_t h;             /* hidden size */
  int64_t v;             /* vocabulary size */
  int32_t ignore_index;  /* label value that marks a row as ignored (commonly -100) */
  int32_t reduction;     /* flce_reduction_t */
  int32_t shift;         /* 0, or 1: row i is scored against labels[i + 1] (see above) */
  int32_t seq_len;       /* rows per sequence when shift = 1 (n must be a multiple); ignored otherwise */
} flce_problem_t;

/* Workspace of flce_forward, flce_backward and flce_fwd_bwd (0 if p is
 * invalid): the "extra HBM" of the fused operator, which
 * "What-Each-Parallelism-Actually-Shards" §7.4 asks to keep bounded inside the
 * operator instead of the [B,S,V] logits.  It holds the device status word,
 * per-row partial (max, sum) pairs and target logits (O(N)), one vocabulary
 * chunk of bf16 G (N x C, C = 8192 for N <= 16384 rows, else 4096) and an fp32
 * dX accumulator (N x H).  Independent of V: the logits are recomputed in the
 * backward pass, chunk by chunk, and never stored for a whole row. */
size_t flce_workspace_bytes(const flce_problem_t* p);

/* Workspace of the row-chunk calls (0 if p is invalid): a chunk of R rows of
 * the bf16 vocabulary gradient (R x V), one fp32 per (chunk row, 256-wide
 * vocabulary tile), with two or more chunks an fp32 dW accumulator (V x H),
 * the chunk's rows of X scaled by their per-row factor (R x H bf16) and O(N)
 * per-row words (§7.4's chunked cross-entropy, [B,C,V] per chunk).  Several
 * chunks have R = min(N/2, 1 GiB / 2V) rows; all N rows form one chunk (no
 * accumulator) whenever that takes no more memory than several — then the
 * chunk buffer has the [N,V] shape of the logits, in bf16. */
size_t flce_workspace_bytes_rowchunk(const flce_problem_t* p);

/* Forward ("What-Each-Parallelism-Actually-Shards" §7.4: online log-sum-exp over
 * vocabulary tiles, target logit only).  Writes the loss (device fp32 scalar,
 * or N per-row losses under FLCE_REDUCTION_NONE) and lse[N] (fp32).  Reads X,
 * W, labels.  Never stores logits. */
flce_status_t flce_forward(const flce_problem_t* p, const void* X, const void* W,
                           const int32_t* labels, float* loss, float* lse,
                           void* ws, size_t ws_bytes, flce_stream_t stream);

/* Backward (§7.4: recompute logits instead of saving them).  Given lse from
 * flce_forward on the same X, W, labels, writes dX [N,H] and dW [V,H] (bf16,
 * fp32 accumulation).  grad_loss: device fp32 scalar g, or NULL for g = 1;
 * under FLCE_REDUCTION_NONE, N per-row gradients g_i (required). */
flce_status_t flce_backward(const flce_problem_t* p, const void* X, const void* W,
                            const int32_t* labels, const float* lse, const float* grad_loss,
                            void* dX, void* dW, void* ws, size_t ws_bytes, flce_stream_t stream);

/* Forward then backward with g = 1 (under FLCE_REDUCTION_NONE: the gradients
 * of the sum of the per-row losses): loss, lse, dX, dW in one call, on the
 * bounded workspace of flce_workspace_bytes(p) ("What-Each-Parallelism-
 * Actually-Shards" §7.4: online log-sum-exp, target logit only, logits
 * recomputed in the backward pass).  Executes 8*N*H*V flops (the logits twice). */
flce_status_t flce_fwd_bwd(const flce_problem_t* p, const void* X, const void* W,
                           const int32_t* labels, float* loss, float* lse, void* dX, void* dW,
                           void* ws, size_t ws_bytes, flce_stream_t stream);

/* The same results, fused over row chunks (§7.4's chunked cross-entropy): the
 * logits are computed once (6*N*H*V flops).  The forward pass keeps each row
 * chunk's softmax, relative to each row's target logit, as bf16 in the
 * workspace, and once the chunk's lse is known dX and dW are contracted from it
 * with one factor per row.  Needs flce_workspace_bytes_rowchunk(p) bytes of
 * workspace, which grow with V (FLCE_ERR_WORKSPACE_TOO_SMALL below that). */
flce_status_t flce_fwd_bwd_rowchunk(const flce_problem_t* p, const void* X, const void* W,
                                    const int32_t* labels, float* loss, float* lse, void* dX, void* dW,
                                    void* ws, size_t ws_bytes, flce_stream_t stream);

/* End to end on host memory (no counterpart in the pages: the call for a caller
 * whose batch lives in host memory).  Reads X, W, labels from host memory and
 * writes loss, lse, dX, dW to host memory, with the shapes and layouts of
 * flce_fwd_bwd (the bounded path); page-locked host memory keeps the copies asynchronous.
 * Returns without waiting, having enqueued: one cudaMemcpyAsync per input to
 * the device on `in_stream`, the pass of flce_fwd_bwd on `stream` (after the
 * inputs), one cudaMemcpyAsync per result back to the host on `out_stream`
 * (after the pass).  Pass `stream` for all three to keep everything on one
 * stream; with separate copy streams, consecutive calls on two `dev` buffers
 * overlap one call's copies with the other's kernels while the kernels stay
 * in order on `stream`.
 *   - dev: a device buffer of at least flce_host_buffer_bytes(p) bytes,
 *     256-byte aligned, owned by the caller: the workspace of flce_fwd_bwd at
 *     its start (so flce_read_device_status(dev, stream) reads the call's device
 *     status), then the device copies of the inputs and results.
 *   - The host buffers and `dev` must not be touched, nor `dev` passed to
 *     another call, until `out_stream` has passed the call's result copies.
 *   - Errors: as flce_fwd_bwd; FLCE_ERR_WORKSPACE_TOO_SMALL if dev_bytes is
 *     below flce_host_buffer_bytes(p). */
size_t flce_host_buffer_bytes(const flce_problem_t* p);
flce_status_t flce_fwd_bwd_host(const flce_problem_t* p, const void* X, const void* W,
                                const int32_t* labels, float* loss, float* lse, void* dX, void* dW,
                                void* dev, size_t dev_bytes, flce_stream_t stream,
                                flce_stream_t in_stream, flce_stream_t out_stream);

/* dX *= g and dW *= g in place (bf16, g a device fp32 scalar): turns the
 * gradients flce_fwd_bwd computed for g = 1 into those of g * loss, so an
 * autograd wrapper can run the fused pass in its forward and apply the
 * upstream gradient in its backward. */
flce_status_t flce_scale_grads(const flce_problem_t* p, const float* grad_loss, void* dX, void* dW,
                               flce_stream_t stream);

/* Distillation without full logits ("What-Each-Parallelism-Actually-Shards"
 * §7.6: in distillation keep to top-k logits or chunked KL instead of returning
 * the [B,S,V] logits).
 *
 * flce_topk: for each row the k largest logits z_ij = x_i . w_j (1 <= k <= 16),
 * high to low (ties: lower id first), their vocabulary ids and the row's lse,
 * e.g. the teacher side of a distillation step.  topk_idx, topk_logit: [N, k];
 * lse: [N].  Needs flce_topk_workspace_bytes(p, k) of workspace.  Labels,
 * reduction and shift in p are not used. */
size_t flce_topk_workspace_bytes(const flce_problem_t* p, int32_t k);
flce_status_t flce_topk(const flce_problem_t* p, int32_t k, const void* X, const void* W, int32_t* topk_idx,
                        float* topk_logit, float* lse, void* ws, size_t ws_bytes, flce_stream_t stream);

/* flce_soft_fwd_bwd: loss and gradients against sparse soft targets, the student
 * side of a distillation step.  Row i has k target ids tgt_idx[i, :] with
 * probabilities q = tgt_prob[i, :] ([N, k], 1 <= k <= 16; entries with q <= 0
 * are unused; ids distinct).  With p = softmax(x_i W^T):
 *   loss_i = sum_k q_k log q_k - sum_k q_k log p_{id_k}      (KL(q || p) on the ids)
 *   G_ij   = s * (Q_i p_ij - sum_k q_k [j = id_k]),  Q_i = sum_k q_k
 * A row with Q_i = 0 is ignored; mean divides by the rows that are not.  k = 1,
 * q = 1 is the hard-label cross-entropy.  g = 1 as in flce_fwd_bwd.  shift must
 * be 0; labels unused.  Like flce_fwd_bwd it runs on the bounded workspace of
 * flce_workspace_bytes(p), the logits recomputed in the backward pass (each
 * chunk of G formed as s Q_i p_ij, then the targets' -s q_k entered in place);
 * flce_soft_fwd_bwd_rowchunk takes the row-chunk path and workspace instead. */
flce_status_t flce_soft_fwd_bwd(const flce_problem_t* p, int32_t k, const void* X, const void* W,
                                const int32_t* tgt_idx, const float* tgt_prob, float* loss, float* lse, void* dX,
                                void* dW, void* ws, size_t ws_bytes, flce_stream_t stream);
flce_status_t flce_soft_fwd_bwd_rowchunk(const flce_problem_t* p, int32_t k, const void* X, const void* W,
                                         const int32_t* tgt_idx, const float* tgt_prob, float* loss, float* lse,
                                         void* dX, void* dW, void* ws, size_t ws_bytes, flce_stream_t stream);

/* Synchronises `stream`, then returns the status word recorded in ws by the
 * kernels of earlier calls (FLCE_OK if none) and clears it.  The pages have no
 * counterpart: it is how a caller learns of the errors the kernels find
 * (labels outside [0,V), which the pages leave undefined; bounded waits that
 * ran out) without the kernels trapping. */
flce_status_t flce_read_device_status(void* ws, flce_stream_t stream);

/* Launches one kernel whose pipeline wait is on a barrier that nothing
 * completes, with the given limit in nanoseconds; the wait gives up, records
 * FLCE_ERR_TIMEOUT in ws and the kernel returns.  Exercises the error path of
 * the bounded waits used by every kernel. */
flce_status_t flce_selftest_timeout(void* ws, size_t ws_bytes, uint64_t limit_ns, flce_stream_t stream);

/* Debug build.  The library also builds as libflce_debug.so (compiled with
 * FLCE_DEBUG_CHECKS): every index the kernels compute into a workspace or
 * output buffer is tested against that buffer's size, and every TMA coordinate
 * against the 16-byte rule, before the access; a failed test records
 * FLCE_ERR_BOUNDS in the status word and skips the access (no trap; a skipped
 * load then ends in a bounded wait).  The pages have no counterpart.
 * flce_debug_checks returns 1 in that build, 0 in the release one.
 * flce_selftest_bounds launches one thread that tests an index one past a
 * one-element buffer: in the debug build the status word then reads
 * FLCE_ERR_BOUNDS, in the release build FLCE_OK; no memory is accessed. */
int flce_debug_checks(void);
flce_status_t flce_selftest_bounds(void* ws, size_t ws_bytes, flce_stream_t stream);

/* Diagnostics: per-launch device timing.  `mask` selects the kernel kinds to
 * time (bit k for kind k; 0 turns profiling off, -1 times every kind).  Each
 * launch of a selected kind is bracketed by two CUDA events on its stream; an
 * event between two launches keeps the second from starting its launch while
 * the first drains (the library's kernels otherwise overlap that way), so
 * select only the kinds to be measured.
 * flce_profile_read synchronises the recorded events and reports, for one
 * kernel kind, the launches recorded, their summed device time (ms) and their
 * summed algorithmic flops.  Kinds: 0 forward projection + online
 * log-sum-exp (2*N*V*H flops), 1 recomputed logits -> G for one vocabulary
 * chunk (2*N*C*H), 2 dX/dW contractions of one chunk (4*N*C*H), 3 small
 * kernels (label scan, finalize, reductions, dX cast; 0 flops).  Enabling or
 * disabling clears the totals.  Off by default.  Process-wide, not tied to a
 * workspace. */
flce_status_t flce_profile_enable(int mask);
flce_status_t flce_profile_read(int kind, int64_t* launches, double* total_ms, double* flops);

/* ----------------------------------------------------------------------------
 * Sharded loss ("What-Each-Parallelism-Actually-Shards" §3.2 vocab-parallel LM
 * head, §7.2 vocab-parallel cross-entropy, §7.3 sequence-sharded loss).  The
 * library holds no communicator: the caller runs the exchange (one all-gather
 * of [2,N] per rank for the vocabulary split, an all-reduce of dX partials; for
 * the sequence split, an all-reduce of the loss sum, the valid count and dW),
 * and the calls below do every step of arithmetic on either side of it.
 *
 * Vocabulary split: rank r holds rows [v_offset, v_offset + v_rows) of W (the
 * whole LM head has p->v rows; labels are global ids).  Steps:
 *   1. flce_shard_forward: the shard's per-row lse over its ids and the target
 *      logit where the shard holds the label (0 elsewhere);
 *   2. gather every rank's (lse_part, tgt_part) in rank order;
 *   3. flce_shard_combine: the global lse = log sum_r exp(lse_part_r), the
 *      target logit sum_r tgt_part_r, the loss (the same bits on every rank);
 *   4. flce_shard_backward with the global lse: the shard's dW rows (complete,
 *      bf16) and its fp32 part of dX = G_shard W_shard;
 *   5. sum the dX parts over ranks (fp32), flce_f32_to_bf16. */
typedef struct {
  int64_t v_offset;  /* first vocabulary id this shard holds */
  int64_t v_rows;    /* number of ids (rows of W_shard), >= 1, v_offset + v_rows <= p->v */
} flce_vocab_shard_t;

/* Workspace of the three shard calls (0 if p or sh is invalid): O(N*(C + 1)),
 * the bounded layout without the dX accumulator plus N shard-local labels.
 * Any workspace that serves a shard of p also serves flce_shard_combine and
 * flce_valid_count for p. */
size_t flce_shard_workspace_bytes(const flce_problem_t* p, const flce_vocab_shard_t* sh);

/* lse_part[N], tgt_part[N] (fp32 device): per row, log sum_{j in shard}
 * exp(z_ij) and z_{i,y_i} when y_i is in the shard, else 0 (also for ignored
 * rows).  Labels are checked against [0, p->v); reduction is not used. */
flce_status_t flce_shard_forward(const flce_problem_t* p, const flce_vocab_shard_t* sh, const void* X,
                                 const void* W_shard, const int32_t* labels, float* lse_part, float* tgt_part,
                                 void* ws, size_t ws_bytes, flce_stream_t stream);

/* lse_parts, tgt_parts: [parts, N] fp32 device, shard r in row r (1 <= parts <=
 * 65536, summed in that order).  Writes lse[N] (global) and the loss under
 * p->reduction (a scalar, or N per-row losses), as flce_forward would on the
 * whole vocabulary. */
flce_status_t flce_shard_combine(const flce_problem_t* p, int32_t parts, const float* lse_parts,
                                 const float* tgt_parts, const int32_t* labels, float* loss, float* lse,
                                 void* ws, size_t ws_bytes, flce_stream_t stream);

/* Given the global lse, G restricted to the shard's ids:
 * G_ij = s (exp(z_ij - lse_i) - [j = y_i]) valid_i, s from p->reduction, the
 * global valid count and grad_loss (NULL: g = 1; N per-row values under
 * FLCE_REDUCTION_NONE).  Writes dW_shard [v_rows, H] bf16 (= G_shard^T X) and
 * dX_part [N, H] fp32 (= G_shard W_shard, this shard's term of dX; 16-byte
 * aligned). */
flce_status_t flce_shard_backward(const flce_problem_t* p, const flce_vocab_shard_t* sh, const void* X,
                                  const void* W_shard, const int32_t* labels, const float* lse,
                                  const float* grad_loss, float* dX_part, void* dW_shard, void* ws,
                                  size_t ws_bytes, flce_stream_t stream);

/* *count (device int32) = the number of rows whose label is not ignore_index
 * (shift applied), with labels checked against [0, p->v).  The sequence split
 * all-reduces it to scale a mean loss by the global count. */
flce_status_t flce_valid_count(const flce_problem_t* p, const int32_t* labels, int32_t* count, void* ws,
                               size_t ws_bytes, flce_stream_t stream);

/* dst[i] = bf16(src[i]) (round to nearest even), i < count; both 16-byte
 * aligned device pointers.  Casts a summed fp32 dX to the bf16 output. */
flce_status_t flce_f32_to_bf16(const float* src, void* dst, int64_t count, flce_stream_t stream);

/* Forward pass that allocates nothing and takes no workspace.  The pages have
 * no counterpart; it exists for callers that cannot allocate device memory —
 * code embedded in another runtime that owns all device allocations and hands
 * over only input and output buffers, or latency-critical loops where a
 * cudaMalloc/cudaFree would synchronise the device.  Same arguments and
 * results as flce_forward, minus ws/ws_bytes.
 *   - Scratch: one fixed array of about 4.3 MiB in the library's own device
 *     memory, held by every GPU that loads the library until the process exits.
 *   - Limit: 1 <= n <= 32768 rows (FLCE_ERR_EXCEEDS_STATIC_SCRATCH above that);
 *     h and v as for the other calls.
 *   - The first call on each device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - All calls share the one array: calls whose work overlaps on the GPU
 *     (different streams, or different host threads without ordering) race
 *     and give wrong results.  Order them on one stream.
 *   - Errors found on the device (a label outside [0,V), a bounded wait that
 *     ran out, limited by FLCE_TIMEOUT_NS like every call) set the loss to NaN
 *     — the scalar, or every one of the N per-row losses under
 *     FLCE_REDUCTION_NONE; there is no status word to read.
 *   - The array's address is looked up once per device and kept: do not call
 *     this entry point on a device after cudaDeviceReset (or any reset of its
 *     primary context) in the same process. */
flce_status_t flce_forward_noalloc(const flce_problem_t* p, const void* X, const void* W,
                                   const int32_t* labels, float* loss, float* lse, flce_stream_t stream);

/* Static description of a status code. */
const char* flce_status_string(flce_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H */
