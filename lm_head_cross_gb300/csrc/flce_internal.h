// Internal interface between the C-ABI layer (flce_api.cu) and the kernels
// (flce_kernels.cu).  Not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define FLCE_HOST_DEVICE __host__ __device__
#else
#define FLCE_HOST_DEVICE
#endif

namespace flce {

// Tile shape of every tensor-core kernel: 128 rows (TMEM lanes) x 256 columns
// (TMEM columns of one accumulator), K staged 64 bf16 (one 128-byte swizzle row)
// at a time.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 6;    // 32 KiB per stage and CTA (own A rows + own half of B)
constexpr int kThreads = 192;  // warp 0: TMA producer, warp 1: MMA issuer, warps 2-5: epilogue
constexpr int kMaxSplit = 32;  // most vocabulary splits of the forward pass
constexpr int kPairRows = 2 * kBM;  // every launch runs on CTA pairs: a pair tile has 256 rows
constexpr int kBoxB = kBN / 2;      // rows of the B operand each CTA of a pair stages (K-major box)

// Grid of a tensor-core launch: CTA pairs, at most one CTA per SM.
inline int pair_grid(int sms, long long pair_work) {
  long long pairs = sms / 2;
  if (pair_work < pairs) pairs = pair_work;
  if (pairs < 1) pairs = 1;
  return static_cast<int>(2 * pairs);
}

// Vocabulary chunk width of the backward pass (a multiple of kBN).  The
// workspace holds one chunk of G, N x chunk bf16.
int chunk_width(int64_t n);

enum Mode : int { kModeForward = 0, kModeGrad = 1, kModeBwd = 2, kModeFwdStore = 3, kModeTopk = 4 };

// Forward-store: a row's p~ is stored relative to its reference logit (log2
// units) unless a tile's p~ sum exceeds 2^kRefSpan; then relative to the
// tile's max.
constexpr float kRefSpan = 64.f;

constexpr int kTopkMax = 16;     // largest k of flce_topk / of soft targets per row
constexpr int kTopkSplit = 16;   // most vocabulary splits of the top-k pass (bounds its partial buffer)

// Output format of the dX / dW tiles of a kModeBwd launch.
enum OutMode : int {
  kOutF32Store = 0,      // fp32 stored to dx_f32 / dw_f32
  kOutF32Add = 1,        // fp32 added at L2 to dx_f32 / dw_f32
  kOutBF16 = 2,          // bf16 through `out`/`out2`
  kOutF32AccToBF16 = 3,  // dW only: read the fp32 accumulator through `out2`, add, write bf16 through `out3`
};

// Everything a tensor-core launch needs besides its tensor maps.
struct TcParams {
  int n, h, v;
  int ignore_index;
  uint64_t timeout_ns;
  int* status;
  // forward: row pair tiles (256 rows) x vocabulary splits
  int row_tiles, vocab_tiles, vsplit;
  float* part_m;  // [vsplit][n] running max, log2 units
  float* part_l;  // [vsplit][n] running sum of 2^(t - m)
  float* tgt;     // [n] target logit z_{i, y_i}
  const int32_t* labels;
  int shift, seq_len;   // shift = 1: row i is scored against labels[i + 1]; each sequence's last row is ignored
  const float* grad_rows;  // grad (reduction none): per-row upstream gradient, or null
  // grad / bwd: one vocabulary chunk [c0, c0 + cw)
  int c0, cw;
  const float* lse;
  const float* scale;  // device scalar s
  int grad_n_tiles;    // grad: vocabulary tiles in the chunk
  // bwd: dX tiles then dW tiles
  int dx_tiles, dw_tiles;
  int h_tiles;          // ceil(h / kBN)
  int dw_m_tiles;       // ceil(cw / kPairRows)
  int dx_out, dw_out;   // OutMode of the dX and dW tiles
  float* dx_f32;        // bwd: the fp32 dX accumulator [n, h] for kOutF32Store / kOutF32Add dX tiles (else null)
  float* dw_f32;        // bwd: the fp32 dW accumulator [v, h] for kOutF32Store / kOutF32Add dW tiles (else null)
  int dx_k, dw_k;       // K extents: dX tiles run over dx_k vocabulary ids, dW tiles over dw_k rows
  int dx_first;         // 1: dX tiles are listed first (they are the long ones)
  int* tile_counter;    // bwd: global tile counter, zero at launch
  // row chunk of the forward-store pass: rows [r0, row_end) (row_end 0 means n)
  int r0, row_end;
  float* mtile;         // forward-store: per (chunk row, vocabulary tile) reference exponent, log2 units
  const float* mref;    // forward-store: per row of X its reference logit, log2 units
  const float* rowscale;  // bwd: per chunk row factor f_i of the stored G / (s f_i) (null: the buffer holds G)
  int b2_r0;            // bwd: first row of the dW B operand's tensor map
  int* zero_words;      // if set: two ints the launch sets to 0 once its predecessors are done
  // top-k pass: per (split, row) the best topk_k (logit, id) pairs, [vsplit][n][kTopkMax]
  float* topk_val;
  int32_t* topk_idx;
  int topk_k;
  unsigned* topk_thr;   // top-k: per row the best 16th-best value any range has reached (ordered key), zeroed
  int units_group;      // forward modes: row tiles per unit group (see units_group_rows)
  // element counts of the buffers above that are indexed by computed offsets (checked in
  // builds with FLCE_DEBUG_CHECKS): part_m / part_l, mtile, topk_val / topk_idx, rowscale
  int64_t part_count, mtile_count, topk_count, rowscale_count;
  int soft_grad;        // grad: soft targets (every row valid, no one-hot; grad_rows carries s Q_i)
};

// Unit order of the forward modes: units (row tile, vocabulary range) run row
// tile fastest within a group of this many row tiles, then range, then group.
// A group's X panels (256 rows x H bf16 each) fit in 48 MB, so they stay in
// L2 while the pairs of a wave share each W tile: W is read from memory about
// once per group instead of once per row tile.
inline int units_group_rows(int row_tiles, int64_t h) {
  const int64_t panel = static_cast<int64_t>(kPairRows) * h * 2;
  int64_t g = (int64_t{48} << 20) / panel;
  if (g < 1) g = 1;
  return static_cast<int>(g < row_tiles ? g : row_tiles);
}

// First vocabulary tile of range sp when vocab_tiles tiles are cut into vsplit
// ranges: the first (vocab_tiles % vsplit) ranges take one tile more than the
// rest, so the units handed out last (the highest ranges) are the smaller ones.
FLCE_HOST_DEVICE inline int range_begin(int sp, int vocab_tiles, int vsplit) {
  const int base = vocab_tiles / vsplit;
  const int rem = vocab_tiles % vsplit;
  return sp * base + (sp < rem ? sp : rem);
}

// The (row tile, range) of unit u in that order.
FLCE_HOST_DEVICE inline void unit_coords(int u, int row_tiles, int vsplit, int group, int* rt, int* sp) {
  const int per_group = group * vsplit;
  const int g = u / per_group;
  const int g0 = g * group;
  const int rows_g = row_tiles - g0 < group ? row_tiles - g0 : group;  // the last group may be short
  const int local = u - g * per_group;
  *rt = g0 + local % rows_g;
  *sp = local / rows_g;
}

struct TcMaps {
  CUtensorMap a;   // forward/grad: X (K-major, box 64x128); bwd: G K-major (dX)
  CUtensorMap b;   // forward/grad: W (K-major, box 64x256); bwd: W MN-major (dX)
  CUtensorMap out; // grad: G store (bf16 box 64x32); bwd: dX fp32 accumulator (box 32x32)
  CUtensorMap a2;  // bwd: G MN-major (dW A operand, box 64x64)
  CUtensorMap b2;  // bwd: X MN-major (dW B operand, box 64x64)
  CUtensorMap out2;// bwd: dW output (bf16 box 64x32, or the fp32 accumulator, box 32x32)
  CUtensorMap out3;// bwd, kOutF32AccToBF16: dW bf16 store (box 64x32)
};

// Launchers (asynchronous on `stream`; return the launch error, if any).
cudaError_t launch_tc(int mode, const TcMaps& maps, const TcParams& p, int grid, cudaStream_t stream);
// Labels as the kernels read them: with shift, row i takes labels[i + 1] and
// the last row of each sequence of seq_len rows is ignored.
struct LabelView {
  const int32_t* labels;   // hard labels (may be null when soft targets are given)
  int ignore_index;
  int shift, seq_len;
  // soft targets: per row soft_k (vocabulary id, probability) pairs; soft_k = 0 for hard labels
  const int32_t* soft_idx;
  const float* soft_prob;
  int soft_k;
};

cudaError_t launch_fwd_finalize_rows(int r0, int rows, int n, int v, int vsplit, LabelView lv, const float* part_m,
                                     const float* part_l, const float* tgt, float* lse, float* loss_rows,
                                     double* blk_loss, int* blk_valid, int* status, cudaStream_t stream);
// Fused path.  label_prep: label check, the rows' references (log2 units: the
// target logit, or for soft targets the q-weighted mean target logit, whose
// q-weighted sum goes to tgt; +inf for rows without a gradient) and, through
// the last block, n_valid and s.
cudaError_t launch_label_prep(int n, int h, int v, int reduction, LabelView lv, const void* X, const void* W,
                              float* mref, float* tgt, int* blk_cnt, int* ticket, int* n_valid, float* scale,
                              int* status, cudaStream_t stream);
// finalize_ref, rows [r0, r0 + rows) of one chunk: lse, losses and the loss
// partials (one per kRefRowsPerBlock rows, index r0 / kRefRowsPerBlock + b),
// the row factors f_i, the chunk buffer's target entries, xs = f x, and the
// list of rows a tile stored relative to its own max (fix_list / fix_count).
constexpr int kRefRowsPerBlock = 8;
cudaError_t launch_finalize_ref(int r0, int rows, int n, int h, int v, int vp, int vsplit, LabelView lv,
                                const float* part_m, const float* part_l, const float* tgt, const float* mref,
                                float* lse, float* loss_rows, double* blk_loss, int* blk_valid,
                                float* rowscale, const void* X, void* xs, void* P, int* fix_list, int* fix_count,
                                int* status, cudaStream_t stream);
// The listed rows' full fix-up (G / s in place), `grid` blocks.
cudaError_t launch_fixup_list(const int* fix_list, const int* fix_count, int r0, int v, int vp, int vtiles,
                              LabelView lv, const float* lse, const float* mtile, void* P, int grid,
                              cudaStream_t stream);
// nsub: the (max, sum) pairs and candidate lists per row, vocabulary sub-ranges.
cudaError_t launch_topk_finalize(int n, int nsub, int k, const float* part_m, const float* part_l,
                                 const float* cand_val, const int32_t* cand_idx, float* lse, float* out_val,
                                 int32_t* out_idx, cudaStream_t stream);
cudaError_t launch_label_scan_view(int n, int v, LabelView lv, double* blk_loss, int* blk_valid, int* status,
                                   cudaStream_t stream);
cudaError_t launch_reduce_final(int nblk, const double* blk_loss, const int* blk_valid, int reduction,
                                const float* grad_loss, float* loss_out, int* n_valid_out, float* scale_out,
                                cudaStream_t stream);
cudaError_t launch_convert_bf16(const float* src, void* dst, int64_t count, cudaStream_t stream);
// fp32 -> bf16 (round to nearest even) of any count; src and dst 16-byte aligned.
cudaError_t launch_f32_to_bf16(const float* src, void* dst, int64_t count, cudaStream_t stream);

// Soft targets on the bounded path: per row s Q_i (the grad launch's
// coefficient), and a vocabulary chunk's target entries G_ij -= s q_k in place.
cudaError_t launch_soft_rowcoef(int n, int k, const float* soft_prob, const float* scale, float* coef,
                               cudaStream_t stream);
cudaError_t launch_soft_chunk_targets(int n, int k, const int32_t* soft_idx, const float* soft_prob,
                                      const float* scale, int c0, int cw, int64_t pitch, void* G, int v, int* status,
                                      cudaStream_t stream);

// Vocabulary shards.  A shard's kernels read labels in shard-local form: -1 for an
// ignored row (the shard calls run with ignore_index -1), y - v0 for a label the
// shard holds, kNotOwned for a valid label held by another shard (it never equals
// a column index, so no tile gathers it and no one-hot entry is subtracted).
constexpr int kNotOwned = 0x7fffffff;
cudaError_t launch_shard_labels(int n, int64_t v_total, int64_t v0, int64_t vs, LabelView lv, int32_t* lab_local,
                                int* status, cudaStream_t stream);
// Per row: the shard's lse (natural log) from the split partials, and its target
// logit where the shard holds the label (0 elsewhere).
cudaError_t launch_shard_finalize(int n, int vsplit, const float* part_m, const float* part_l, const float* tgt,
                                  const int32_t* lab_local, float* lse_part, float* tgt_part, cudaStream_t stream);
// Per row: lse = log sum_r exp(lse_parts[r]), z = sum_r tgt_parts[r] (parts in index
// order), the loss row against the global labels, and per-block partials.
cudaError_t launch_shard_combine(int n, int parts, int64_t v_total, LabelView lv, const float* lse_parts,
                                 const float* tgt_parts, float* lse, float* loss_rows, double* blk_loss,
                                 int* blk_valid, int* status, cudaStream_t stream);
cudaError_t launch_scale_bf16(void* x, int64_t count, const float* g, cudaStream_t stream);
cudaError_t launch_timeout_selftest(int* status, uint64_t limit_ns, cudaStream_t stream);
// One thread tests index 1 against a buffer of one element: builds with
// FLCE_DEBUG_CHECKS record kErrBounds (and touch no memory), release builds nothing.
cudaError_t launch_bounds_selftest(int* status, cudaStream_t stream);

// Limit of every bounded wait in the kernels, in nanoseconds: FLCE_TIMEOUT_NS
// from the environment (read once), else 4 s.
uint64_t timeout_ns();

int tc_smem_bytes();
int tc_topk_subranges();  // vocabulary sub-ranges the top-k launch reports per range
constexpr int kFinalizeThreads = 256;

}  // namespace flce
