// C-ABI entry points declared in include/flce.h: argument validation, the
// workspace layout, TMA tensor maps, and the order of kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "../../include/flce.h"
#include "flce_internal.h"

namespace flce {
namespace {

constexpr size_t kAlign = 256;
constexpr int32_t kMaxShardParts = 1 << 16;  // most vocabulary shards flce_shard_combine takes
#ifdef FLCE_DEBUG_CHECKS
constexpr int kDebugChecksBuild = 1;
#else
constexpr int kDebugChecksBuild = 0;
#endif
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;  // 4 s; a healthy wait lasts microseconds

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Workspace layout (byte offsets from ws, each 256-byte aligned).
struct Layout {
  size_t status, n_valid, scale;  // header words
  size_t counter;                 // tile counter of the dynamically scheduled launches
  size_t fix_count;               // fused path: rows listed for the full fix-up in the current chunk
  size_t ticket;                  // fused path: blocks of the label pass done (its last block resets it)
  size_t fcount;                  // unit counters of the forward launches: one header word, or one per row
                                  // chunk of the fused path (zeroed at the start of every call)
  int nchunks;                    // fused path: row chunks
  size_t blk_loss, blk_valid;     // per-block partial sums of the finalize kernels
  size_t part_m, part_l, tgt;     // forward: per-split row state, target logits
  size_t g;                       // one chunk buffer: recompute path G [N, chunk]; fused path p~/G [rows, Vp]
  size_t dx_acc;                  // fp32 accumulator: recompute path dX [N, H]; fused path dW [V, H]
  size_t mtile;                   // fused path: per (chunk row, vocabulary tile) reference exponent
  size_t mref;                    // fused path: per row of X its target logit, log2 units
  size_t rowscale, fix_list;      // fused path: per chunk row factor f_i; rows listed for the full fix-up
  size_t xs;                      // fused path: f_i x_i for the chunk's rows, bf16 [rows, H]
  size_t lab;                     // vocabulary-shard calls: shard-local labels [N] int32
  size_t total;
  int nblk, chunk;
  int rows;                       // fused path: rows per chunk (0: layout without the fused path)
  int64_t vp;                     // fused path: row pitch of the chunk buffer (V rounded up to 8)
};

// Rows per chunk of the fused path, a multiple of 256 (the finalize block
// size).  Several chunks of R rows: R = min(half of N, the rows whose p~/G
// buffer [R, V] fits kFusedChunkBytes), and an fp32 dW accumulator (V x H)
// besides the buffer.  One chunk writes dW directly and needs no accumulator,
// so all rows form one chunk whenever its N x V buffer is no larger than the
// several-chunk buffer plus the accumulator (for R = N/2 that is N <= 4H).
constexpr size_t kFusedChunkBytes = size_t{1} << 30;

int fused_rows(int64_t n, int64_t v, int64_t h) {
  const int64_t vp = (v + 7) / 8 * 8;
  const int64_t cap = std::max<int64_t>(
      256, static_cast<int64_t>(kFusedChunkBytes / (2 * static_cast<size_t>(vp))) / 256 * 256);
  const int64_t half = ((n + 1) / 2 + 255) / 256 * 256;
  const int64_t rows = std::min(cap, std::max<int64_t>(256, half));
  const int64_t all = std::max<int64_t>(256, (n + 255) / 256 * 256);
  if (2 * all * vp <= 2 * rows * vp + 4 * v * h) return static_cast<int>(all);
  return static_cast<int>(rows);
}

// `shard`: the layout of the vocabulary-shard calls — no dX accumulator (the
// shard backward accumulates into the caller's fp32 buffer), plus the
// shard-local labels.
Layout make_layout(const flce_problem_t& p, bool fused, bool shard = false) {
  Layout L{};
  if (p.n == 0) {  // an empty batch needs the header (status word) only
    L.total = kAlign;
    return L;
  }
  const size_t n = static_cast<size_t>(p.n), h = static_cast<size_t>(p.h), v = static_cast<size_t>(p.v);
  L.nblk = static_cast<int>((p.n + kFinalizeThreads - 1) / kFinalizeThreads);
  L.chunk = chunk_width(p.n);
  L.rows = fused ? fused_rows(p.n, p.v, p.h) : 0;
  L.vp = (p.v + 7) / 8 * 8;
  const size_t vtiles = (v + kBN - 1) / kBN;
  size_t off = 0;
  L.status = off;
  L.n_valid = off + 4;
  L.scale = off + 8;
  L.counter = off + 16;
  L.fix_count = off + 20;
  L.ticket = off + 24;
  L.fcount = off + 28;
  off += kAlign;
  const size_t nblk_alloc = std::max<size_t>(L.nblk, (n + kRefRowsPerBlock - 1) / kRefRowsPerBlock);
  L.blk_loss = off;
  off = align_up(off + sizeof(double) * nblk_alloc);
  L.blk_valid = off;
  off = align_up(off + sizeof(int) * nblk_alloc);
  L.part_m = off;
  off = align_up(off + sizeof(float) * kMaxSplit * n);
  L.part_l = off;
  off = align_up(off + sizeof(float) * kMaxSplit * n);
  L.tgt = off;
  off = align_up(off + sizeof(float) * n);
  // the fused layout serves only the fused path (flce_fwd_bwd, flce_soft_fwd_bwd);
  // every other call lays out the workspace without it
  const bool one_chunk = fused && static_cast<int64_t>(L.rows) >= p.n;
  L.g = off;
  const size_t gbytes = fused ? 2 * static_cast<size_t>(L.rows) * static_cast<size_t>(L.vp)
                              : 2 * n * static_cast<size_t>(L.chunk);
  off = align_up(off + gbytes);
  L.dx_acc = off;
  const size_t accbytes = fused ? (one_chunk ? 0 : 4 * v * h) : (shard ? 0 : 4 * n * h);
  off = align_up(off + accbytes);
  L.mtile = off;
  if (fused) off = align_up(off + sizeof(float) * static_cast<size_t>(L.rows) * vtiles);
  L.mref = off;
  if (fused) off = align_up(off + sizeof(float) * n);
  L.rowscale = off;
  if (fused) off = align_up(off + sizeof(float) * static_cast<size_t>(L.rows));
  L.fix_list = off;
  if (fused) off = align_up(off + sizeof(int) * static_cast<size_t>(L.rows));
  L.xs = off;
  if (fused) off = align_up(off + 2 * static_cast<size_t>(L.rows) * h);
  L.lab = off;
  if (shard) off = align_up(off + sizeof(int32_t) * n);
  if (fused) {
    L.nchunks = static_cast<int>((p.n + L.rows - 1) / L.rows);
    L.fcount = off;
    off = align_up(off + sizeof(int) * static_cast<size_t>(L.nchunks));
  }
  L.total = off;
  return L;
}


PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D row-major tensor [outer, inner] with row pitch `pitch_bytes`, box
// {box_inner, box_outer}, 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint64_t inner, uint64_t outer,
              uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

uint64_t timeout_ns() {
  static uint64_t t = [] {
    const char* e = std::getenv("FLCE_TIMEOUT_NS");
    if (e && *e) {
      const unsigned long long v = std::strtoull(e, nullptr, 10);
      if (v > 0) return static_cast<uint64_t>(v);
    }
    return kDefaultTimeoutNs;
  }();
  return t;
}

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

flce_status_t check_problem(const flce_problem_t* p) {
  if (!p) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->n < 0 || p->h < 1 || p->v < 1) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->reduction != FLCE_REDUCTION_MEAN && p->reduction != FLCE_REDUCTION_SUM &&
      p->reduction != FLCE_REDUCTION_NONE)
    return FLCE_ERR_INVALID_ARGUMENT;
  if (p->shift != 0 && p->shift != 1) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->shift && (p->seq_len < 1 || p->n % p->seq_len != 0)) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->h < 8 || p->h % 8 != 0) return FLCE_ERR_UNSUPPORTED_SHAPE;
  // TMA coordinates and the kernels' tile indices are 32-bit.
  if (p->n > (int64_t{1} << 30) || p->v > (int64_t{1} << 30) || p->h > (int64_t{1} << 20))
    return FLCE_ERR_UNSUPPORTED_SHAPE;
  return FLCE_OK;
}

struct Device {
  int sms = 0;
  bool ok = false;
};

flce_status_t device_info(Device* d) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLCE_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return FLCE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return FLCE_ERR_CUDA;
  if (major != 10) return FLCE_ERR_CUDA;  // the binary carries sm_103a code only
  if (cudaDeviceGetAttribute(&d->sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FLCE_ERR_CUDA;
  d->ok = true;
  return FLCE_OK;
}

// Forward split count: the number of vocabulary ranges each row tile is cut
// into.  The forward modes hand out (row tile, range) units in the order
// unit_coords gives them (row tile fastest within groups of `group` row
// tiles), each pair taking the next unit when it finishes its current one; a
// pair's finishing time is the tiles of the units it took.  Picks the count
// (4..cap, at most the number of vocabulary tiles) whose list schedule over
// `grid` pairs ends earliest; among those, the one whose least loaded pair
// idles least (then the fewest ranges to merge).
int choose_vsplit_uncached(int row_tiles, int vocab_tiles, int grid, int cap, int group) {
  const int hi = std::min(cap, vocab_tiles);
  const int lo = std::min(4, hi);
  int best = lo;
  long long best_cost = -1, best_min = -1;
  for (int vs = lo; vs <= hi; ++vs) {
    const long long units = static_cast<long long>(row_tiles) * vs;
    const int g = static_cast<int>(std::min<long long>(grid, units));
    // min-heap of (busy until, pair): the pair that frees first takes the next unit
    std::vector<std::pair<long long, int>> heap;
    for (int b = 0; b < g; ++b) heap.emplace_back(0, b);
    auto cmp = [](const std::pair<long long, int>& a, const std::pair<long long, int>& b) { return a > b; };
    std::make_heap(heap.begin(), heap.end(), cmp);
    long long makespan = 0;
    for (long long u = 0; u < units; ++u) {
      int rt = 0, sp = 0;
      unit_coords(static_cast<int>(u), row_tiles, vs, group, &rt, &sp);
      const long long tiles = range_begin(sp + 1, vocab_tiles, vs) - range_begin(sp, vocab_tiles, vs);
      std::pop_heap(heap.begin(), heap.end(), cmp);
      heap.back().first += tiles;
      makespan = std::max(makespan, heap.back().first);
      std::push_heap(heap.begin(), heap.end(), cmp);
    }
    const long long least = heap.front().first;  // the heap's top: the least loaded pair
    if (best_cost < 0 || makespan < best_cost || (makespan == best_cost && least > best_min)) {
      best_cost = makespan;
      best_min = least;
      best = vs;
    }
  }
  return best;
}

int choose_vsplit(int row_tiles, int vocab_tiles, int grid, int cap, int group) {
  static std::mutex mu;
  static int key[5] = {-1, -1, -1, -1, -1};
  static int val = 1;
  std::lock_guard<std::mutex> lock(mu);
  if (key[0] != row_tiles || key[1] != vocab_tiles || key[2] != grid || key[3] != cap || key[4] != group) {
    val = choose_vsplit_uncached(row_tiles, vocab_tiles, grid, cap, group);
    key[0] = row_tiles;
    key[1] = vocab_tiles;
    key[2] = grid;
    key[3] = cap;
    key[4] = group;
  }
  return val;
}

struct Ctx {
  const flce_problem_t* p;
  Layout L;
  uint8_t* ws;
  cudaStream_t stream;
  Device dev;
  int* status() const { return reinterpret_cast<int*>(ws + L.status); }
  int* n_valid() const { return reinterpret_cast<int*>(ws + L.n_valid); }
  float* scale() const { return reinterpret_cast<float*>(ws + L.scale); }
  int* counter() const { return reinterpret_cast<int*>(ws + L.counter); }
  double* blk_loss() const { return reinterpret_cast<double*>(ws + L.blk_loss); }
  int* blk_valid() const { return reinterpret_cast<int*>(ws + L.blk_valid); }
  float* part_m() const { return reinterpret_cast<float*>(ws + L.part_m); }
  float* part_l() const { return reinterpret_cast<float*>(ws + L.part_l); }
  float* tgt() const { return reinterpret_cast<float*>(ws + L.tgt); }
  void* g() const { return ws + L.g; }
  float* dx_acc() const { return reinterpret_cast<float*>(ws + L.dx_acc); }
  float* mtile() const { return reinterpret_cast<float*>(ws + L.mtile); }
  int* ticket() const { return reinterpret_cast<int*>(ws + L.ticket); }
  int* fcount() const { return reinterpret_cast<int*>(ws + L.fcount); }
  int* fix_count() const { return reinterpret_cast<int*>(ws + L.fix_count); }
  int* fix_list() const { return reinterpret_cast<int*>(ws + L.fix_list); }
  float* mref() const { return reinterpret_cast<float*>(ws + L.mref); }
  float* rowscale() const { return reinterpret_cast<float*>(ws + L.rowscale); }
  void* xs() const { return ws + L.xs; }
  int32_t* lab() const { return reinterpret_cast<int32_t*>(ws + L.lab); }
  LabelView labels_of(const int32_t* labels) const {
    return LabelView{labels, p->ignore_index, p->shift, p->shift ? p->seq_len : 1, nullptr, nullptr, 0};
  }
  bool per_row() const { return p->reduction == FLCE_REDUCTION_NONE; }
};

flce_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA; }

// An empty batch (n = 0) has no valid row: the loss is 0 under mean (as for
// n_valid = 0) and under sum, dW = G^T X is 0, and no other output has an
// element.  Clears the workspace's status word like every call.
flce_status_t run_empty(const flce_problem_t* p, float* loss, void* dW, void* ws, size_t ws_bytes,
                        flce_stream_t stream) {
  if (!ws) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(ws, kAlign)) return FLCE_ERR_MISALIGNED;
  if (ws_bytes < kAlign) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, kAlign, s) != cudaSuccess) return FLCE_ERR_CUDA;
  if (loss && p->reduction != FLCE_REDUCTION_NONE && cudaMemsetAsync(loss, 0, sizeof(float), s) != cudaSuccess)
    return FLCE_ERR_CUDA;
  if (dW && cudaMemsetAsync(dW, 0, 2 * static_cast<size_t>(p->v) * static_cast<size_t>(p->h), s) != cudaSuccess)
    return FLCE_ERR_CUDA;
  return FLCE_OK;
}

// Row-indexed pointers (X, labels, lse, dX, per-row losses) may be null when the batch is empty.
bool rows_ok(const flce_problem_t* p, const void* ptr) { return ptr || (p && p->n == 0); }

// ----------------------------------------------------------------------------- diagnostics: per-launch timing

constexpr int kKinds = 4;  // forward, logits gradient, dX/dW contraction, small kernels

struct ProfRecord {
  int kind;
  cudaEvent_t start, stop;
  double flops;
};

struct Profiler {
  std::mutex mu;
  bool on = false;
  int mask = 0;  // bit k: bracket launches of kind k
  std::vector<ProfRecord> records;
  std::vector<cudaEvent_t> pool;
  int64_t launches[kKinds] = {};
  double ms[kKinds] = {};
  double flops[kKinds] = {};

  cudaEvent_t take() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }
  // Synchronise recorded events, fold them into the totals, recycle them.
  cudaError_t drain() {
    cudaError_t err = cudaSuccess;
    for (auto& r : records) {
      float t = 0.f;
      cudaError_t e = cudaEventSynchronize(r.stop);
      if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.start, r.stop);
      if (e != cudaSuccess) err = e;
      launches[r.kind] += 1;
      ms[r.kind] += t;
      flops[r.kind] += r.flops;
      pool.push_back(r.start);
      pool.push_back(r.stop);
    }
    records.clear();
    return err;
  }
  void clear() {
    drain();
    for (int k = 0; k < kKinds; ++k) {
      launches[k] = 0;
      ms[k] = 0.0;
      flops[k] = 0.0;
    }
  }
};

Profiler& profiler() {
  static Profiler p;
  return p;
}

// Runs `launch` (which enqueues one kernel on `stream`), bracketed by two
// events when profiling is on.
template <typename F>
cudaError_t timed(int kind, double flops, cudaStream_t stream, F&& launch) {
  Profiler& P = profiler();
  bool on;
  {
    std::lock_guard<std::mutex> lock(P.mu);
    on = P.on && ((P.mask >> kind) & 1);
  }
  if (!on) return launch();
  cudaEvent_t a, b;
  {
    std::lock_guard<std::mutex> lock(P.mu);
    a = P.take();
    b = P.take();
  }
  if (!a || !b) return launch();
  cudaEventRecord(a, stream);
  cudaError_t e = launch();
  cudaEventRecord(b, stream);
  std::lock_guard<std::mutex> lock(P.mu);
  P.records.push_back(ProfRecord{kind, a, b, flops});
  return e;
}

// Workspace layouts: the bounded one of every call (independent of V), the
// row-chunk one of the calls that keep a chunk of the vocabulary gradient
// (flce_fwd_bwd_rowchunk, flce_soft_fwd_bwd), the vocabulary-shard one.
enum class Lay { kBounded, kRowChunk, kShard };

flce_status_t prepare(Ctx* c, const flce_problem_t* p, void* ws, size_t ws_bytes, flce_stream_t stream,
                      Lay lay = Lay::kBounded) {
  flce_status_t st = check_problem(p);
  if (st != FLCE_OK) return st;
  if (!ws) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(ws, kAlign)) return FLCE_ERR_MISALIGNED;
  c->p = p;
  c->L = make_layout(*p, lay == Lay::kRowChunk, lay == Lay::kShard);
  if (ws_bytes < c->L.total) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  c->ws = static_cast<uint8_t*>(ws);
  c->stream = reinterpret_cast<cudaStream_t>(stream);
  st = device_info(&c->dev);
  if (st != FLCE_OK) return st;
  if (!encode_fn()) return FLCE_ERR_CUDA;
  // the header (status word, counters) starts every call cleared
  return cuda_status(cudaMemsetAsync(c->ws + c->L.status, 0, kAlign, c->stream));
}

// The forward projection with the online log-sum-exp: per (vocabulary range,
// row) partials in the workspace, target logits where a tile holds the label.
// Returns the split count through *vsplit.
flce_status_t run_forward_tc(const Ctx& c, const void* X, const void* W, const int32_t* labels, int* vsplit) {
  const flce_problem_t& p = *c.p;
  TcMaps maps;
  if (!make_map(&maps.a, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.n, p.h * 2, kBK, kBM)) return FLCE_ERR_CUDA;
  if (!make_map(&maps.b, W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.v, p.h * 2, kBK, kBoxB)) return FLCE_ERR_CUDA;
  maps.out = maps.a2 = maps.b2 = maps.out2 = maps.a;  // unused in this mode

  TcParams tp{};
  tp.n = static_cast<int>(p.n);
  tp.h = static_cast<int>(p.h);
  tp.v = static_cast<int>(p.v);
  tp.ignore_index = p.ignore_index;
  tp.timeout_ns = timeout_ns();
  tp.status = c.status();
  tp.row_tiles = static_cast<int>((p.n + kPairRows - 1) / kPairRows);
  tp.vocab_tiles = static_cast<int>((p.v + kBN - 1) / kBN);
  tp.units_group = units_group_rows(tp.row_tiles, p.h);
  tp.vsplit = choose_vsplit(tp.row_tiles, tp.vocab_tiles, c.dev.sms / 2, kMaxSplit, tp.units_group);
  tp.part_m = c.part_m();
  tp.part_l = c.part_l();
  tp.tgt = c.tgt();
  tp.labels = labels;
  tp.shift = p.shift;
  tp.seq_len = p.shift ? p.seq_len : 1;
  tp.r0 = 0;
  tp.row_end = tp.n;
  tp.tile_counter = c.fcount();  // a header word: zero since the call started
  tp.part_count = static_cast<int64_t>(kMaxSplit) * p.n;
  const long long units = static_cast<long long>(tp.row_tiles) * tp.vsplit;
  const int grid = pair_grid(c.dev.sms, units);
  const double flops = 2.0 * static_cast<double>(p.n) * static_cast<double>(p.v) * static_cast<double>(p.h);
  *vsplit = tp.vsplit;
  return cuda_status(timed(0, flops, c.stream, [&] { return launch_tc(kModeForward, maps, tp, grid, c.stream); }));
}

flce_status_t run_forward(const Ctx& c, const void* X, const void* W, const int32_t* labels, float* loss, float* lse,
                          const float* grad_loss) {
  const flce_problem_t& p = *c.p;
  int vsplit = 0;
  flce_status_t st = run_forward_tc(c, X, W, labels, &vsplit);
  if (st != FLCE_OK) return st;
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_fwd_finalize_rows(0, static_cast<int>(p.n), static_cast<int>(p.n), static_cast<int>(p.v), vsplit,
                                    c.labels_of(labels), c.part_m(), c.part_l(), c.tgt(), lse,
                                    c.per_row() ? loss : nullptr, c.blk_loss(), c.blk_valid(), c.status(), c.stream);
  }));
  if (st != FLCE_OK) return st;
  return cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_reduce_final(c.L.nblk, c.blk_loss(), c.blk_valid(), p.reduction, grad_loss,
                               c.per_row() ? nullptr : loss, c.n_valid(),
                               c.scale(), c.stream);
  }));
}

// Backward given lse and the scale already in the workspace.  dX accumulates
// in fp32 in `dx_acc` (the workspace's accumulator, or a caller buffer) and is
// written as bf16 to dX unless dX is null.
// With soft targets (`soft`), grad_rows holds s Q_i per row, the grad launches
// form s Q_i p_ij, and each chunk's target entries are subtracted in place before
// its dX/dW launch.
flce_status_t run_backward(const Ctx& c, const void* X, const void* W, const int32_t* labels, const float* lse,
                           const float* grad_rows, void* dX, void* dW, float* dx_acc,
                           const LabelView* soft = nullptr) {
  const flce_problem_t& p = *c.p;
  const int chunk = c.L.chunk;
  TcParams tp{};
  tp.n = static_cast<int>(p.n);
  tp.h = static_cast<int>(p.h);
  tp.v = static_cast<int>(p.v);
  tp.ignore_index = p.ignore_index;
  tp.timeout_ns = timeout_ns();
  tp.status = c.status();
  tp.labels = labels;
  tp.shift = p.shift;
  tp.seq_len = p.shift ? p.seq_len : 1;
  tp.grad_rows = grad_rows;
  tp.soft_grad = soft ? 1 : 0;
  tp.lse = lse;
  tp.scale = c.scale();
  tp.row_tiles = static_cast<int>((p.n + kPairRows - 1) / kPairRows);
  tp.h_tiles = static_cast<int>((p.h + kBN - 1) / kBN);

  TcMaps gm;  // grad: X, W K-major; G store
  if (!make_map(&gm.a, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.n, p.h * 2, kBK, kBM)) return FLCE_ERR_CUDA;
  if (!make_map(&gm.b, W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.v, p.h * 2, kBK, kBoxB)) return FLCE_ERR_CUDA;
  TcMaps bm;  // bwd: W MN-major (dX B operand), X MN-major (dW B operand), dW store; dX goes to dx_acc directly
  if (!make_map(&bm.b, W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.v, p.h * 2, 64, kBK)) return FLCE_ERR_CUDA;
  if (!make_map(&bm.b2, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.n, p.h * 2, 64, kBK)) return FLCE_ERR_CUDA;
  if (!make_map(&bm.out2, dW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.v, p.h * 2, 64, 32)) return FLCE_ERR_CUDA;
  bm.out = bm.out2;  // unused by these tiles (a valid map for the prologue's prefetch)

  for (int64_t c0 = 0; c0 < p.v; c0 += chunk) {
    const int cw = static_cast<int>(std::min<int64_t>(chunk, p.v - c0));
    tp.c0 = static_cast<int>(c0);
    tp.cw = cw;
    // G for this chunk: [N, cw] bf16 with row pitch `chunk`
    if (!make_map(&gm.out, c.g(), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cw, p.n, static_cast<uint64_t>(chunk) * 2, 64, 32))
      return FLCE_ERR_CUDA;
    gm.a2 = gm.b2 = gm.out2 = gm.a;  // unused in this mode
    tp.grad_n_tiles = (cw + kBN - 1) / kBN;
    const long long gtiles = static_cast<long long>(tp.row_tiles) * tp.grad_n_tiles;
    const double gflops = 2.0 * static_cast<double>(p.n) * cw * static_cast<double>(p.h);
    flce_status_t st = cuda_status(timed(1, gflops, c.stream, [&] {
      return launch_tc(kModeGrad, gm, tp, pair_grid(c.dev.sms, gtiles), c.stream);
    }));
    if (st != FLCE_OK) return st;
    if (soft) {
      st = cuda_status(timed(3, 0.0, c.stream, [&] {
        return launch_soft_chunk_targets(tp.n, soft->soft_k, soft->soft_idx, soft->soft_prob, c.scale(), tp.c0, cw,
                                         chunk, c.g(), tp.v, c.status(), c.stream);
      }));
      if (st != FLCE_OK) return st;
    }

    if (!make_map(&bm.a, c.g(), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cw, p.n, static_cast<uint64_t>(chunk) * 2, kBK, kBM))
      return FLCE_ERR_CUDA;
    if (!make_map(&bm.a2, c.g(), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cw, p.n, static_cast<uint64_t>(chunk) * 2, 64, kBK))
      return FLCE_ERR_CUDA;
    tp.dw_m_tiles = (cw + kPairRows - 1) / kPairRows;
    tp.dw_tiles = tp.dw_m_tiles * tp.h_tiles;
    tp.dx_tiles = tp.row_tiles * tp.h_tiles;
    tp.dx_out = c0 > 0 ? kOutF32Add : kOutF32Store;
    tp.dx_f32 = dx_acc;
    tp.dw_out = kOutBF16;
    tp.dx_k = cw;
    tp.dw_k = tp.n;
    tp.dx_first = 0;
    tp.tile_counter = c.counter();
    st = cuda_status(cudaMemsetAsync(c.counter(), 0, sizeof(int), c.stream));
    if (st != FLCE_OK) return st;
    const long long btiles = static_cast<long long>(tp.dw_tiles) + tp.dx_tiles;
    st = cuda_status(timed(2, 2.0 * gflops, c.stream, [&] {
      return launch_tc(kModeBwd, bm, tp, pair_grid(c.dev.sms, btiles), c.stream);
    }));
    if (st != FLCE_OK) return st;
  }
  if (!dX) return FLCE_OK;
  return cuda_status(timed(3, 0.0, c.stream, [&] { return launch_convert_bf16(dx_acc, dX, p.n * p.h, c.stream); }));
}

// Soft targets on the bounded workspace (8NHV executed): the targets' q-weighted
// logits and the valid count (label_prep_kernel, its row references and block
// counts going to the free chunk buffer), the forward's log-sum-exp, the KL
// rows and their reduction, then the recompute backward with the per-row
// coefficient s Q_i and each chunk's target entries subtracted in place.
flce_status_t run_soft_bounded(const Ctx& c, const void* X, const void* W, const LabelView lv, float* loss, float* lse,
                               void* dX, void* dW) {
  const flce_problem_t& p = *c.p;
  const int n = static_cast<int>(p.n);
  float* scratch = static_cast<float*>(c.g());  // free until the first grad launch
  flce_status_t st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_label_prep(n, static_cast<int>(p.h), static_cast<int>(p.v), p.reduction, lv, X, W, scratch,
                             c.tgt(), reinterpret_cast<int*>(scratch + p.n), c.ticket(), c.n_valid(), c.scale(),
                             c.status(), c.stream);
  }));
  if (st != FLCE_OK) return st;
  int vsplit = 0;
  st = run_forward_tc(c, X, W, nullptr, &vsplit);
  if (st != FLCE_OK) return st;
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_fwd_finalize_rows(0, n, n, static_cast<int>(p.v), vsplit, lv, c.part_m(), c.part_l(), c.tgt(), lse,
                                    c.per_row() ? loss : nullptr, c.blk_loss(), c.blk_valid(), c.status(), c.stream);
  }));
  if (st != FLCE_OK) return st;
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_reduce_final(c.L.nblk, c.blk_loss(), c.blk_valid(), p.reduction, nullptr,
                               c.per_row() ? nullptr : loss, c.n_valid(), c.scale(), c.stream);
  }));
  if (st != FLCE_OK) return st;
  // the target logits are consumed: their array now holds s Q_i
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_soft_rowcoef(n, lv.soft_k, lv.soft_prob, c.scale(), c.tgt(), c.stream);
  }));
  if (st != FLCE_OK) return st;
  return run_backward(c, X, W, nullptr, lse, c.tgt(), dX, dW, c.dx_acc(), &lv);
}

// Fused forward + backward over row chunks (6NHV executed, no recompute):
// per chunk, the forward-store pass writes p~ = 2^(S - ref_i) (relative to the
// row's reference logit) and the per-range row state; the finalize turns that
// into lse, the losses, the row factors f_i and f_i x_i, and patches each
// row's target entry; rows whose tiles outran the reference are rewritten by
// the list fix-up; one launch then computes dX for the chunk's rows (K = V,
// times s f_i, bf16 out) and adds s (f x)^T p~ into the fp32 dW accumulator
// (K = chunk rows).
flce_status_t run_fused(const Ctx& c, const void* X, const void* W, const LabelView lv, float* loss, float* lse,
                        void* dX, void* dW) {
  const flce_problem_t& p = *c.p;
  const int n = static_cast<int>(p.n), h = static_cast<int>(p.h), v = static_cast<int>(p.v);
  const int32_t* labels = lv.labels;
  const int vtiles = (v + kBN - 1) / kBN;
  const int h_tiles = (h + kBN - 1) / kBN;
  // The forward-store references each row to its target logit (soft targets:
  // their q-weighted mean logit); the row factor f_i then finishes G in the
  // dX/dW epilogues, and only rows whose tiles outrun that reference get the
  // full fix-up pass.
  const int nblk = (n + kRefRowsPerBlock - 1) / kRefRowsPerBlock;
  // every forward-store launch takes its units from its own counter, so no launch
  // resets a counter that a running one may still be drawing from
  flce_status_t st = cuda_status(
      cudaMemsetAsync(c.fcount(), 0, sizeof(int) * static_cast<size_t>(c.L.nchunks), c.stream));
  if (st != FLCE_OK) return st;
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_label_prep(n, h, v, p.reduction, lv, X, W, c.mref(), c.tgt(), reinterpret_cast<int*>(c.part_l()),
                             c.ticket(), c.n_valid(), c.scale(), c.status(), c.stream);
  }));
  if (st != FLCE_OK) return st;

  TcMaps fm;  // forward-store: X, W K-major; p~ store
  if (!make_map(&fm.a, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.n, p.h * 2, kBK, kBM)) return FLCE_ERR_CUDA;
  if (!make_map(&fm.b, W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.v, p.h * 2, kBK, kBoxB)) return FLCE_ERR_CUDA;
  TcMaps bm;  // bwd: G K-major (dX A), W MN-major (dX B), dX bf16 out; G MN-major (dW A), X MN-major (dW B), dW fp32
  if (!make_map(&bm.b, W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.v, p.h * 2, 64, kBK)) return FLCE_ERR_CUDA;
  if (!make_map(&bm.out, dX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.n, p.h * 2, 64, 32)) return FLCE_ERR_CUDA;
  const uint64_t pitch = static_cast<uint64_t>(c.L.vp) * 2;
  const int nchunks = (n + c.L.rows - 1) / c.L.rows;
  CUtensorMap dw_acc_map, dw_bf16_map;  // the fp32 accumulator exists only with several chunks
  if (nchunks > 1 &&
      !make_map(&dw_acc_map, c.dx_acc(), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.h, p.v, p.h * 4, 32, 32))
    return FLCE_ERR_CUDA;
  if (!make_map(&dw_bf16_map, dW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.v, p.h * 2, 64, 32)) return FLCE_ERR_CUDA;

  for (int r0 = 0; r0 < n; r0 += c.L.rows) {
    const int cr = std::min(c.L.rows, n - r0);
    if (!make_map(&fm.out, c.g(), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, cr, pitch, 64, 32)) return FLCE_ERR_CUDA;
    fm.a2 = fm.b2 = fm.out2 = fm.a;  // unused in this mode
    TcParams tp{};
    tp.n = n;
    tp.h = h;
    tp.v = v;
    tp.ignore_index = p.ignore_index;
    tp.timeout_ns = timeout_ns();
    tp.status = c.status();
    tp.labels = labels;
    tp.shift = p.shift;
    tp.seq_len = p.shift ? p.seq_len : 1;
    tp.r0 = r0;
    tp.row_end = r0 + cr;
    tp.row_tiles = (cr + kPairRows - 1) / kPairRows;
    tp.vocab_tiles = vtiles;
    tp.units_group = units_group_rows(tp.row_tiles, p.h);
    tp.vsplit = choose_vsplit(tp.row_tiles, vtiles, c.dev.sms / 2, kMaxSplit, tp.units_group);
    tp.part_m = c.part_m();
    tp.part_l = c.part_l();
    tp.tgt = c.tgt();
    tp.mtile = c.mtile();
    tp.mref = c.mref();
    tp.zero_words = c.counter();  // the backward launch's tile counter and the fix-up list count start at zero
    tp.tile_counter = c.fcount() + r0 / c.L.rows;
    tp.part_count = static_cast<int64_t>(kMaxSplit) * p.n;
    tp.mtile_count = static_cast<int64_t>(c.L.rows) * vtiles;
    const double fflops = 2.0 * cr * static_cast<double>(v) * h;
    const int fgrid = pair_grid(c.dev.sms, static_cast<long long>(tp.row_tiles) * tp.vsplit);
    st = cuda_status(timed(0, fflops, c.stream, [&] { return launch_tc(kModeFwdStore, fm, tp, fgrid, c.stream); }));
    if (st != FLCE_OK) return st;
    st = cuda_status(timed(3, 0.0, c.stream, [&] {
      return launch_finalize_ref(r0, cr, n, h, v, static_cast<int>(c.L.vp), tp.vsplit, lv, c.part_m(), c.part_l(),
                                 c.tgt(), c.mref(), lse, c.per_row() ? loss : nullptr,
                                 c.blk_loss(), c.blk_valid(), c.rowscale(), X, c.xs(), c.g(), c.fix_list(),
                                 c.fix_count(), c.status(), c.stream);
    }));
    if (st != FLCE_OK) return st;
    st = cuda_status(timed(3, 0.0, c.stream, [&] {
      return launch_fixup_list(c.fix_list(), c.fix_count(), r0, v, static_cast<int>(c.L.vp), vtiles, lv, lse,
                               c.mtile(), c.g(), 2 * c.dev.sms, c.stream);
    }));
    if (st != FLCE_OK) return st;

    if (!make_map(&bm.a, c.g(), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, cr, pitch, kBK, kBM)) return FLCE_ERR_CUDA;
    if (!make_map(&bm.a2, c.g(), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, cr, pitch, 64, kBK)) return FLCE_ERR_CUDA;
    if (!make_map(&bm.b2, c.xs(), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, cr, p.h * 2, 64, kBK)) return FLCE_ERR_CUDA;
    TcParams bp{};
    bp.n = n;
    bp.h = h;
    bp.v = v;
    bp.ignore_index = p.ignore_index;
    bp.timeout_ns = timeout_ns();
    bp.status = c.status();
    bp.r0 = r0;
    bp.row_end = r0 + cr;
    bp.b2_r0 = 0;
    bp.rowscale = c.rowscale();
    bp.rowscale_count = c.L.rows;
    bp.scale = c.scale();
    bp.c0 = 0;
    bp.cw = v;
    bp.h_tiles = h_tiles;
    bp.dx_tiles = ((cr + kPairRows - 1) / kPairRows) * h_tiles;
    bp.dw_tiles = ((v + kPairRows - 1) / kPairRows) * h_tiles;
    bp.dx_k = v;
    bp.dw_k = cr;
    bp.dx_first = 1;
    bp.dx_out = kOutBF16;
    // dW: the first chunk stores the fp32 accumulator, middle chunks add to it,
    // the last one adds it to its own part and writes bf16 (a single chunk writes bf16)
    const bool last = r0 + cr >= n;
    if (nchunks == 1) {
      bp.dw_out = kOutBF16;
      bm.out2 = dw_bf16_map;
    } else {
      bp.dw_out = last ? kOutF32AccToBF16 : (r0 == 0 ? kOutF32Store : kOutF32Add);
      bp.dw_f32 = last ? nullptr : c.dx_acc();
      bm.out2 = dw_acc_map;
      bm.out3 = dw_bf16_map;
    }
    bp.tile_counter = c.counter();
    const long long btiles = static_cast<long long>(bp.dx_tiles) + bp.dw_tiles;
    const int bgrid = pair_grid(c.dev.sms, btiles);
    st = cuda_status(
        timed(2, 2.0 * fflops, c.stream, [&] { return launch_tc(kModeBwd, bm, bp, bgrid, c.stream); }));
    if (st != FLCE_OK) return st;
  }
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_reduce_final(nblk, c.blk_loss(), c.blk_valid(), p.reduction, nullptr,
                               c.per_row() ? nullptr : loss, c.n_valid(), c.scale(), c.stream);
  }));
  return st;
}

// Top-k pass: the forward with a per-row best-k list, then the merge.
// Top-k candidates: per (vocabulary sub-range, row) the best kTopkMax.  A launch
// reports tc_topk_subranges() sub-ranges per range (one with four epilogue
// warps; two when two warps share a row, each on half of the columns); the
// buffer is sized for two.
constexpr int kTopkSubranges = 2 * kTopkSplit;
static_assert(kTopkSubranges <= kMaxSplit, "the sub-ranges' (max, sum) pairs fit the split partials");

size_t topk_cand_bytes(const flce_problem_t& p) {
  return align_up(static_cast<size_t>(kTopkSubranges) * static_cast<size_t>(p.n) * kTopkMax *
                  (sizeof(float) + sizeof(int32_t)));
}

size_t topk_extra_bytes(const flce_problem_t& p) {
  return topk_cand_bytes(p) + align_up(static_cast<size_t>(p.n) * sizeof(unsigned));  // + shared thresholds
}

flce_status_t run_topk(const Ctx& c, int k, const void* X, const void* W, int32_t* out_idx, float* out_val, float* lse) {
  const flce_problem_t& p = *c.p;
  const Layout base = make_layout(p, false);
  float* cand_val = reinterpret_cast<float*>(c.ws + base.total);
  int32_t* cand_idx = reinterpret_cast<int32_t*>(
      c.ws + base.total + static_cast<size_t>(kTopkSubranges) * static_cast<size_t>(p.n) * kTopkMax * sizeof(float));
  unsigned* thr = reinterpret_cast<unsigned*>(c.ws + base.total + topk_cand_bytes(p));
  if (cudaMemsetAsync(thr, 0, static_cast<size_t>(p.n) * sizeof(unsigned), c.stream) != cudaSuccess)
    return FLCE_ERR_CUDA;
  TcMaps maps;
  if (!make_map(&maps.a, X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.n, p.h * 2, kBK, kBM)) return FLCE_ERR_CUDA;
  if (!make_map(&maps.b, W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.h, p.v, p.h * 2, kBK, kBoxB)) return FLCE_ERR_CUDA;
  maps.out = maps.a2 = maps.b2 = maps.out2 = maps.a;
  TcParams tp{};
  tp.topk_thr = thr;
  tp.n = static_cast<int>(p.n);
  tp.h = static_cast<int>(p.h);
  tp.v = static_cast<int>(p.v);
  tp.ignore_index = p.ignore_index;
  tp.timeout_ns = timeout_ns();
  tp.status = c.status();
  tp.row_tiles = static_cast<int>((p.n + kPairRows - 1) / kPairRows);
  tp.vocab_tiles = static_cast<int>((p.v + kBN - 1) / kBN);
  tp.units_group = units_group_rows(tp.row_tiles, p.h);
  tp.vsplit = choose_vsplit(tp.row_tiles, tp.vocab_tiles, c.dev.sms / 2, kTopkSplit, tp.units_group);
  tp.part_m = c.part_m();
  tp.part_l = c.part_l();
  tp.tgt = c.tgt();
  tp.labels = nullptr;
  tp.r0 = 0;
  tp.row_end = tp.n;
  tp.topk_val = cand_val;
  tp.topk_idx = cand_idx;
  tp.topk_k = k;
  tp.tile_counter = c.fcount();  // a header word: zero since the call started
  tp.part_count = static_cast<int64_t>(kMaxSplit) * p.n;
  tp.topk_count = static_cast<int64_t>(kTopkSubranges) * p.n * kTopkMax;
  const double flops = 2.0 * static_cast<double>(p.n) * static_cast<double>(p.v) * static_cast<double>(p.h);
  const int grid = pair_grid(c.dev.sms, static_cast<long long>(tp.row_tiles) * tp.vsplit);
  flce_status_t st =
      cuda_status(timed(0, flops, c.stream, [&] { return launch_tc(kModeTopk, maps, tp, grid, c.stream); }));
  if (st != FLCE_OK) return st;
  return cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_topk_finalize(tp.n, tc_topk_subranges() * tp.vsplit, k, c.part_m(), c.part_l(), cand_val, cand_idx,
                                lse, out_val, out_idx, c.stream);
  }));
}

// Device buffer of flce_fwd_bwd_host: the workspace, then the device copies.
struct HostLayout {
  size_t ws, x, w, labels, loss, lse, dx, dw, total;
};

HostLayout host_layout(const flce_problem_t& p) {
  HostLayout L{};
  const size_t n = static_cast<size_t>(p.n), h = static_cast<size_t>(p.h), v = static_cast<size_t>(p.v);
  size_t off = align_up(make_layout(p, false).total);  // the workspace of flce_fwd_bwd
  L.ws = 0;
  L.x = off;
  off = align_up(off + 2 * n * h);
  L.w = off;
  off = align_up(off + 2 * v * h);
  L.labels = off;
  off = align_up(off + 4 * n);
  L.loss = off;
  off = align_up(off + 4 * (p.reduction == FLCE_REDUCTION_NONE ? n : 1));
  L.lse = off;
  off = align_up(off + 4 * n);
  L.dx = off;
  off = align_up(off + 2 * n * h);
  L.dw = off;
  off = align_up(off + 2 * v * h);
  L.total = off;
  return L;
}

// Events that order flce_fwd_bwd_host's copy streams around its pass, one pair
// per device and host thread.  Reusing them is safe: a stream wait takes the
// event's state at the time it is enqueued.
struct CopyEvents {
  cudaEvent_t in_done = nullptr, pass_done = nullptr;
};

flce_status_t copy_events(CopyEvents** out) {
  constexpr int kMaxDevices = 64;
  static thread_local CopyEvents ev[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FLCE_ERR_CUDA;
  CopyEvents& e = ev[dev];
  if (!e.in_done && cudaEventCreateWithFlags(&e.in_done, cudaEventDisableTiming) != cudaSuccess) return FLCE_ERR_CUDA;
  if (!e.pass_done && cudaEventCreateWithFlags(&e.pass_done, cudaEventDisableTiming) != cudaSuccess)
    return FLCE_ERR_CUDA;
  *out = &e;
  return FLCE_OK;
}

}  // namespace

int chunk_width(int64_t n) { return n <= 16384 ? 8192 : 4096; }

}  // namespace flce

using namespace flce;

extern "C" {

size_t flce_workspace_bytes(const flce_problem_t* p) {
  if (check_problem(p) != FLCE_OK) return 0;
  return make_layout(*p, false).total;
}

size_t flce_workspace_bytes_rowchunk(const flce_problem_t* p) {
  if (check_problem(p) != FLCE_OK) return 0;
  return make_layout(*p, true).total;
}

flce_status_t flce_forward(const flce_problem_t* p, const void* X, const void* W, const int32_t* labels, float* loss,
                           float* lse, void* ws, size_t ws_bytes, flce_stream_t stream) {
  if (!p || !W || !rows_ok(p, X) || !rows_ok(p, labels) || !rows_ok(p, lse) ||
      !(loss || (p->n == 0 && p->reduction == FLCE_REDUCTION_NONE)))
    return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(labels, 4) || !aligned(lse, 4) || !aligned(loss, 4))
    return FLCE_ERR_MISALIGNED;
  flce_status_t st = check_problem(p);
  if (st != FLCE_OK) return st;
  if (p->n == 0) return run_empty(p, loss, nullptr, ws, ws_bytes, stream);
  Ctx c;
  st = prepare(&c, p, ws, ws_bytes, stream);
  if (st != FLCE_OK) return st;
  return run_forward(c, X, W, labels, loss, lse, nullptr);
}

flce_status_t flce_backward(const flce_problem_t* p, const void* X, const void* W, const int32_t* labels,
                            const float* lse, const float* grad_loss, void* dX, void* dW, void* ws, size_t ws_bytes,
                            flce_stream_t stream) {
  if (!p || !W || !dW || !rows_ok(p, X) || !rows_ok(p, labels) || !rows_ok(p, lse) || !rows_ok(p, dX))
    return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(dX, 16) || !aligned(dW, 16) || !aligned(labels, 4) ||
      !aligned(lse, 4) || (grad_loss && !aligned(grad_loss, 4)))
    return FLCE_ERR_MISALIGNED;
  flce_status_t st = check_problem(p);
  if (st != FLCE_OK) return st;
  if (p->n == 0) return run_empty(p, nullptr, dW, ws, ws_bytes, stream);
  Ctx c;
  st = prepare(&c, p, ws, ws_bytes, stream);
  if (st != FLCE_OK) return st;
  if (c.per_row() && !grad_loss) return FLCE_ERR_INVALID_ARGUMENT;  // reduction none needs the per-row gradient
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_label_scan_view(static_cast<int>(p->n), static_cast<int>(p->v), c.labels_of(labels), c.blk_loss(),
                             c.blk_valid(), c.status(), c.stream);
  }));
  if (st != FLCE_OK) return st;
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_reduce_final(c.L.nblk, c.blk_loss(), c.blk_valid(), p->reduction, c.per_row() ? nullptr : grad_loss,
                               nullptr, c.n_valid(),
                               c.scale(), c.stream);
  }));
  if (st != FLCE_OK) return st;
  return run_backward(c, X, W, labels, lse, c.per_row() ? grad_loss : nullptr, dX, dW, c.dx_acc());
}

namespace {
flce_status_t fwd_bwd_args(const flce_problem_t* p, const void* X, const void* W, const int32_t* labels,
                           const float* loss, const float* lse, const void* dX, const void* dW) {
  if (!p || !W || !dW || !rows_ok(p, X) || !rows_ok(p, labels) || !rows_ok(p, lse) || !rows_ok(p, dX) ||
      !(loss || (p->n == 0 && p->reduction == FLCE_REDUCTION_NONE)))
    return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(dX, 16) || !aligned(dW, 16) || !aligned(labels, 4) ||
      !aligned(lse, 4) || !aligned(loss, 4))
    return FLCE_ERR_MISALIGNED;
  return check_problem(p);
}
}  // namespace

flce_status_t flce_fwd_bwd(const flce_problem_t* p, const void* X, const void* W, const int32_t* labels, float* loss,
                           float* lse, void* dX, void* dW, void* ws, size_t ws_bytes, flce_stream_t stream) {
  flce_status_t st = fwd_bwd_args(p, X, W, labels, loss, lse, dX, dW);
  if (st != FLCE_OK) return st;
  if (p->n == 0) return run_empty(p, loss, dW, ws, ws_bytes, stream);
  Ctx c;
  st = prepare(&c, p, ws, ws_bytes, stream);
  if (st != FLCE_OK) return st;
  st = run_forward(c, X, W, labels, loss, lse, nullptr);
  if (st != FLCE_OK) return st;
  return run_backward(c, X, W, labels, lse, nullptr, dX, dW, c.dx_acc());
}

flce_status_t flce_fwd_bwd_rowchunk(const flce_problem_t* p, const void* X, const void* W, const int32_t* labels,
                                    float* loss, float* lse, void* dX, void* dW, void* ws, size_t ws_bytes,
                                    flce_stream_t stream) {
  flce_status_t st = fwd_bwd_args(p, X, W, labels, loss, lse, dX, dW);
  if (st != FLCE_OK) return st;
  if (p->n == 0) return run_empty(p, loss, dW, ws, ws_bytes, stream);
  Ctx c;
  st = prepare(&c, p, ws, ws_bytes, stream, Lay::kRowChunk);
  if (st != FLCE_OK) return st;
  return run_fused(c, X, W, c.labels_of(labels), loss, lse, dX, dW);
}

size_t flce_host_buffer_bytes(const flce_problem_t* p) {
  if (check_problem(p) != FLCE_OK) return 0;
  return host_layout(*p).total;
}

flce_status_t flce_fwd_bwd_host(const flce_problem_t* p, const void* X, const void* W, const int32_t* labels,
                                float* loss, float* lse, void* dX, void* dW, void* dev, size_t dev_bytes,
                                flce_stream_t stream, flce_stream_t in_stream, flce_stream_t out_stream) {
  flce_status_t st = check_problem(p);
  if (st != FLCE_OK) return st;
  if (!W || !dW || !dev || !rows_ok(p, X) || !rows_ok(p, labels) || !rows_ok(p, lse) || !rows_ok(p, dX) ||
      !(loss || (p->n == 0 && p->reduction == FLCE_REDUCTION_NONE)))
    return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(dev, kAlign)) return FLCE_ERR_MISALIGNED;
  const HostLayout L = host_layout(*p);
  if (dev_bytes < L.total) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* d = static_cast<uint8_t*>(dev);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t si = reinterpret_cast<cudaStream_t>(in_stream);
  cudaStream_t so = reinterpret_cast<cudaStream_t>(out_stream);
  CopyEvents* ev = nullptr;
  if (si != s || so != s) {
    st = copy_events(&ev);
    if (st != FLCE_OK) return st;
  }
  const size_t n = static_cast<size_t>(p->n), h = static_cast<size_t>(p->h), v = static_cast<size_t>(p->v);
  const size_t loss_bytes = 4 * (p->reduction == FLCE_REDUCTION_NONE ? n : 1);
  // one copy per buffer; an empty one (n = 0) is skipped
  auto copy = [](void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, cudaStream_t cs) {
    return bytes == 0 ? cudaSuccess : cudaMemcpyAsync(dst, src, bytes, kind, cs);
  };
  if (copy(d + L.x, X, 2 * n * h, cudaMemcpyHostToDevice, si) != cudaSuccess ||
      copy(d + L.w, W, 2 * v * h, cudaMemcpyHostToDevice, si) != cudaSuccess ||
      copy(d + L.labels, labels, 4 * n, cudaMemcpyHostToDevice, si) != cudaSuccess)
    return FLCE_ERR_CUDA;
  if (si != s && (cudaEventRecord(ev->in_done, si) != cudaSuccess || cudaStreamWaitEvent(s, ev->in_done, 0) != cudaSuccess))
    return FLCE_ERR_CUDA;
  st = flce_fwd_bwd(p, d + L.x, d + L.w, reinterpret_cast<const int32_t*>(d + L.labels),
                    reinterpret_cast<float*>(d + L.loss), reinterpret_cast<float*>(d + L.lse), d + L.dx, d + L.dw,
                    d + L.ws, L.x - L.ws, stream);
  if (st != FLCE_OK) return st;
  if (so != s &&
      (cudaEventRecord(ev->pass_done, s) != cudaSuccess || cudaStreamWaitEvent(so, ev->pass_done, 0) != cudaSuccess))
    return FLCE_ERR_CUDA;
  if (copy(loss, d + L.loss, loss_bytes, cudaMemcpyDeviceToHost, so) != cudaSuccess ||
      copy(lse, d + L.lse, 4 * n, cudaMemcpyDeviceToHost, so) != cudaSuccess ||
      copy(dX, d + L.dx, 2 * n * h, cudaMemcpyDeviceToHost, so) != cudaSuccess ||
      copy(dW, d + L.dw, 2 * v * h, cudaMemcpyDeviceToHost, so) != cudaSuccess)
    return FLCE_ERR_CUDA;
  return FLCE_OK;
}

flce_status_t flce_scale_grads(const flce_problem_t* p, const float* grad_loss, void* dX, void* dW,
                               flce_stream_t stream) {
  flce_status_t st = check_problem(p);
  if (st != FLCE_OK) return st;
  if (!grad_loss || !rows_ok(p, dX) || !dW) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(dX, 16) || !aligned(dW, 16) || !aligned(grad_loss, 4)) return FLCE_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->n > 0) {
    st = cuda_status(timed(3, 0.0, s, [&] { return launch_scale_bf16(dX, p->n * p->h, grad_loss, s); }));
    if (st != FLCE_OK) return st;
  }
  return cuda_status(timed(3, 0.0, s, [&] { return launch_scale_bf16(dW, p->v * p->h, grad_loss, s); }));
}

flce_status_t flce_read_device_status(void* ws, flce_stream_t stream) {
  if (!ws || !aligned(ws, kAlign)) return FLCE_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FLCE_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FLCE_ERR_NO_DEVICE_STATUS;
  const int zero = 0;
  if (cudaMemcpy(ws, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FLCE_ERR_NO_DEVICE_STATUS;
  return static_cast<flce_status_t>(word);
}

int flce_debug_checks(void) { return kDebugChecksBuild; }

flce_status_t flce_selftest_bounds(void* ws, size_t ws_bytes, flce_stream_t stream) {
  if (!ws || ws_bytes < kAlign) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(ws, kAlign)) return FLCE_ERR_MISALIGNED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return FLCE_ERR_CUDA;
  return cuda_status(launch_bounds_selftest(static_cast<int*>(ws), s));
}

flce_status_t flce_selftest_timeout(void* ws, size_t ws_bytes, uint64_t limit_ns, flce_stream_t stream) {
  if (!ws || ws_bytes < kAlign) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(ws, kAlign)) return FLCE_ERR_MISALIGNED;
  if (limit_ns == 0 || limit_ns > 10000000000ull) return FLCE_ERR_INVALID_ARGUMENT;
  if (cudaMemsetAsync(ws, 0, sizeof(int), reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FLCE_ERR_CUDA;
  return cuda_status(launch_timeout_selftest(static_cast<int*>(ws), limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

size_t flce_topk_workspace_bytes(const flce_problem_t* p, int32_t k) {
  if (check_problem(p) != FLCE_OK || k < 1 || k > kTopkMax) return 0;
  return make_layout(*p, false).total + topk_extra_bytes(*p);
}

flce_status_t flce_topk(const flce_problem_t* p, int32_t k, const void* X, const void* W, int32_t* topk_idx,
                        float* topk_logit, float* lse, void* ws, size_t ws_bytes, flce_stream_t stream) {
  if (!p || !W || !rows_ok(p, X) || !rows_ok(p, topk_idx) || !rows_ok(p, topk_logit) || !rows_ok(p, lse))
    return FLCE_ERR_INVALID_ARGUMENT;
  if (k < 1 || k > kTopkMax) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(topk_idx, 4) || !aligned(topk_logit, 4) || !aligned(lse, 4))
    return FLCE_ERR_MISALIGNED;
  flce_status_t st = check_problem(p);
  if (st != FLCE_OK) return st;
  if (p->n == 0) return run_empty(p, nullptr, nullptr, ws, ws_bytes, stream);
  Ctx c;
  st = prepare(&c, p, ws, ws_bytes, stream);
  if (st != FLCE_OK) return st;
  if (ws_bytes < flce_topk_workspace_bytes(p, k)) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  c.L = make_layout(*p, false);
  return run_topk(c, k, X, W, topk_idx, topk_logit, lse);
}

namespace {
flce_status_t soft_fwd_bwd(const flce_problem_t* p, int32_t k, const void* X, const void* W,
                           const int32_t* tgt_idx, const float* tgt_prob, float* loss, float* lse, void* dX,
                           void* dW, void* ws, size_t ws_bytes, flce_stream_t stream, bool rowchunk) {
  if (!p || !W || !dW || !rows_ok(p, X) || !rows_ok(p, tgt_idx) || !rows_ok(p, tgt_prob) || !rows_ok(p, lse) ||
      !rows_ok(p, dX) || !(loss || (p->n == 0 && p->reduction == FLCE_REDUCTION_NONE)))
    return FLCE_ERR_INVALID_ARGUMENT;
  if (k < 1 || k > kTopkMax) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->shift) return FLCE_ERR_INVALID_ARGUMENT;  // targets are given per row
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(dX, 16) || !aligned(dW, 16) || !aligned(tgt_idx, 4) ||
      !aligned(tgt_prob, 4) || !aligned(lse, 4) || !aligned(loss, 4))
    return FLCE_ERR_MISALIGNED;
  flce_status_t st = check_problem(p);
  if (st != FLCE_OK) return st;
  if (p->n == 0) return run_empty(p, loss, dW, ws, ws_bytes, stream);
  Ctx c;
  st = prepare(&c, p, ws, ws_bytes, stream, rowchunk ? Lay::kRowChunk : Lay::kBounded);
  if (st != FLCE_OK) return st;
  const LabelView lv{nullptr, p->ignore_index, 0, 1, tgt_idx, tgt_prob, k};
  if (rowchunk) return run_fused(c, X, W, lv, loss, lse, dX, dW);
  return run_soft_bounded(c, X, W, lv, loss, lse, dX, dW);
}
}  // namespace

flce_status_t flce_soft_fwd_bwd(const flce_problem_t* p, int32_t k, const void* X, const void* W,
                                const int32_t* tgt_idx, const float* tgt_prob, float* loss, float* lse, void* dX,
                                void* dW, void* ws, size_t ws_bytes, flce_stream_t stream) {
  return soft_fwd_bwd(p, k, X, W, tgt_idx, tgt_prob, loss, lse, dX, dW, ws, ws_bytes, stream, false);
}

flce_status_t flce_soft_fwd_bwd_rowchunk(const flce_problem_t* p, int32_t k, const void* X, const void* W,
                                         const int32_t* tgt_idx, const float* tgt_prob, float* loss, float* lse,
                                         void* dX, void* dW, void* ws, size_t ws_bytes, flce_stream_t stream) {
  return soft_fwd_bwd(p, k, X, W, tgt_idx, tgt_prob, loss, lse, dX, dW, ws, ws_bytes, stream, true);
}

// ----------------------------------------------------------------------------- vocabulary / sequence shards

namespace {

// The shard of a problem as the kernels see it: v = the shard's rows of W,
// shard-local labels (ignore_index -1, no shift).
flce_status_t shard_problem(const flce_problem_t* p, const flce_vocab_shard_t* sh, flce_problem_t* q) {
  flce_status_t st = check_problem(p);
  if (st != FLCE_OK) return st;
  if (!sh || sh->v_offset < 0 || sh->v_rows < 1 || sh->v_offset > p->v - sh->v_rows) return FLCE_ERR_INVALID_ARGUMENT;
  *q = *p;
  q->v = sh->v_rows;
  q->ignore_index = -1;
  q->shift = 0;
  q->seq_len = 0;
  return check_problem(q);
}

LabelView global_labels(const flce_problem_t* p, const int32_t* labels) {
  return LabelView{labels, p->ignore_index, p->shift, p->shift ? p->seq_len : 1, nullptr, nullptr, 0};
}

}  // namespace

size_t flce_shard_workspace_bytes(const flce_problem_t* p, const flce_vocab_shard_t* sh) {
  flce_problem_t q;
  if (shard_problem(p, sh, &q) != FLCE_OK) return 0;
  return make_layout(q, false, true).total;
}

flce_status_t flce_shard_forward(const flce_problem_t* p, const flce_vocab_shard_t* sh, const void* X,
                                 const void* W_shard, const int32_t* labels, float* lse_part, float* tgt_part,
                                 void* ws, size_t ws_bytes, flce_stream_t stream) {
  if (!p || !W_shard || !rows_ok(p, X) || !rows_ok(p, labels) || !rows_ok(p, lse_part) || !rows_ok(p, tgt_part))
    return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(X, 16) || !aligned(W_shard, 16) || !aligned(labels, 4) || !aligned(lse_part, 4) ||
      !aligned(tgt_part, 4))
    return FLCE_ERR_MISALIGNED;
  flce_problem_t q;
  flce_status_t st = shard_problem(p, sh, &q);
  if (st != FLCE_OK) return st;
  if (p->n == 0) return run_empty(&q, nullptr, nullptr, ws, ws_bytes, stream);
  Ctx c;
  st = prepare(&c, &q, ws, ws_bytes, stream, Lay::kShard);
  if (st != FLCE_OK) return st;
  const int n = static_cast<int>(p->n);
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_shard_labels(n, p->v, sh->v_offset, sh->v_rows, global_labels(p, labels), c.lab(), c.status(),
                               c.stream);
  }));
  if (st != FLCE_OK) return st;
  int vsplit = 0;
  st = run_forward_tc(c, X, W_shard, c.lab(), &vsplit);
  if (st != FLCE_OK) return st;
  return cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_shard_finalize(n, vsplit, c.part_m(), c.part_l(), c.tgt(), c.lab(), lse_part, tgt_part, c.stream);
  }));
}

flce_status_t flce_shard_combine(const flce_problem_t* p, int32_t parts, const float* lse_parts,
                                 const float* tgt_parts, const int32_t* labels, float* loss, float* lse, void* ws,
                                 size_t ws_bytes, flce_stream_t stream) {
  if (!p || !rows_ok(p, lse_parts) || !rows_ok(p, tgt_parts) || !rows_ok(p, labels) || !rows_ok(p, lse) ||
      !(loss || (p->n == 0 && p->reduction == FLCE_REDUCTION_NONE)))
    return FLCE_ERR_INVALID_ARGUMENT;
  if (parts < 1 || parts > kMaxShardParts) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(lse_parts, 4) || !aligned(tgt_parts, 4) || !aligned(labels, 4) || !aligned(loss, 4) ||
      !aligned(lse, 4))
    return FLCE_ERR_MISALIGNED;
  flce_status_t st = check_problem(p);
  if (st != FLCE_OK) return st;
  if (p->n == 0) return run_empty(p, loss, nullptr, ws, ws_bytes, stream);
  if (!ws) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(ws, kAlign)) return FLCE_ERR_MISALIGNED;
  // the header and the block partials, which every layout places first
  Ctx c;
  c.p = p;
  c.L = make_layout(*p, false);
  if (ws_bytes < c.L.part_m) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  c.ws = static_cast<uint8_t*>(ws);
  c.stream = reinterpret_cast<cudaStream_t>(stream);
  st = device_info(&c.dev);
  if (st != FLCE_OK) return st;
  st = cuda_status(cudaMemsetAsync(c.ws + c.L.status, 0, kAlign, c.stream));
  if (st != FLCE_OK) return st;
  const int n = static_cast<int>(p->n);
  const int nblk = (n + kFinalizeThreads - 1) / kFinalizeThreads;
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_shard_combine(n, parts, p->v, global_labels(p, labels), lse_parts, tgt_parts, lse,
                                c.per_row() ? loss : nullptr, c.blk_loss(), c.blk_valid(), c.status(), c.stream);
  }));
  if (st != FLCE_OK) return st;
  return cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_reduce_final(nblk, c.blk_loss(), c.blk_valid(), p->reduction, nullptr,
                               c.per_row() ? nullptr : loss, c.n_valid(), c.scale(), c.stream);
  }));
}

flce_status_t flce_shard_backward(const flce_problem_t* p, const flce_vocab_shard_t* sh, const void* X,
                                  const void* W_shard, const int32_t* labels, const float* lse,
                                  const float* grad_loss, float* dX_part, void* dW_shard, void* ws, size_t ws_bytes,
                                  flce_stream_t stream) {
  if (!p || !W_shard || !dW_shard || !rows_ok(p, X) || !rows_ok(p, labels) || !rows_ok(p, lse) ||
      !rows_ok(p, dX_part))
    return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(X, 16) || !aligned(W_shard, 16) || !aligned(dX_part, 16) || !aligned(dW_shard, 16) ||
      !aligned(labels, 4) || !aligned(lse, 4) || (grad_loss && !aligned(grad_loss, 4)))
    return FLCE_ERR_MISALIGNED;
  flce_problem_t q;
  flce_status_t st = shard_problem(p, sh, &q);
  if (st != FLCE_OK) return st;
  if (p->n == 0) return run_empty(&q, nullptr, dW_shard, ws, ws_bytes, stream);
  Ctx c;
  st = prepare(&c, &q, ws, ws_bytes, stream, Lay::kShard);
  if (st != FLCE_OK) return st;
  if (c.per_row() && !grad_loss) return FLCE_ERR_INVALID_ARGUMENT;
  const int n = static_cast<int>(p->n);
  // the valid count and s from the global labels, then the shard-local labels
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_label_scan_view(n, static_cast<int>(p->v), global_labels(p, labels), c.blk_loss(), c.blk_valid(),
                                  c.status(), c.stream);
  }));
  if (st != FLCE_OK) return st;
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_reduce_final(c.L.nblk, c.blk_loss(), c.blk_valid(), p->reduction,
                               c.per_row() ? nullptr : grad_loss, nullptr, c.n_valid(), c.scale(), c.stream);
  }));
  if (st != FLCE_OK) return st;
  st = cuda_status(timed(3, 0.0, c.stream, [&] {
    return launch_shard_labels(n, p->v, sh->v_offset, sh->v_rows, global_labels(p, labels), c.lab(), c.status(),
                               c.stream);
  }));
  if (st != FLCE_OK) return st;
  return run_backward(c, X, W_shard, c.lab(), lse, c.per_row() ? grad_loss : nullptr, nullptr, dW_shard, dX_part);
}

flce_status_t flce_valid_count(const flce_problem_t* p, const int32_t* labels, int32_t* count, void* ws,
                               size_t ws_bytes, flce_stream_t stream) {
  if (!p || !count || !rows_ok(p, labels)) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(labels, 4) || !aligned(count, 4)) return FLCE_ERR_MISALIGNED;
  flce_status_t st = check_problem(p);
  if (st != FLCE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->n == 0) {
    st = run_empty(p, nullptr, nullptr, ws, ws_bytes, stream);
    if (st != FLCE_OK) return st;
    return cuda_status(cudaMemsetAsync(count, 0, sizeof(int32_t), s));
  }
  if (!ws) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(ws, kAlign)) return FLCE_ERR_MISALIGNED;
  Ctx c;
  c.p = p;
  c.L = make_layout(*p, false);
  if (ws_bytes < c.L.part_m) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  c.ws = static_cast<uint8_t*>(ws);
  c.stream = s;
  st = cuda_status(cudaMemsetAsync(c.ws + c.L.status, 0, kAlign, s));
  if (st != FLCE_OK) return st;
  st = cuda_status(timed(3, 0.0, s, [&] {
    return launch_label_scan_view(static_cast<int>(p->n), static_cast<int>(p->v), global_labels(p, labels),
                                  c.blk_loss(), c.blk_valid(), c.status(), s);
  }));
  if (st != FLCE_OK) return st;
  return cuda_status(timed(3, 0.0, s, [&] {
    return launch_reduce_final(c.L.nblk, c.blk_loss(), c.blk_valid(), FLCE_REDUCTION_SUM, nullptr, nullptr, count,
                               c.scale(), s);
  }));
}

flce_status_t flce_f32_to_bf16(const float* src, void* dst, int64_t count, flce_stream_t stream) {
  if (count < 0 || (count > 0 && (!src || !dst))) return FLCE_ERR_INVALID_ARGUMENT;
  if (!aligned(src, 16) || !aligned(dst, 16)) return FLCE_ERR_MISALIGNED;
  if (count == 0) return FLCE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return cuda_status(timed(3, 0.0, s, [&] { return launch_f32_to_bf16(src, dst, count, s); }));
}

flce_status_t flce_profile_enable(int mask) {
  Profiler& P = profiler();
  std::lock_guard<std::mutex> lock(P.mu);
  P.clear();
  P.on = mask != 0;
  P.mask = mask;
  // Create the events up front so that recording them costs no driver
  // allocation inside the region being timed.
  while (P.on && P.pool.size() < 4096) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) break;
    P.pool.push_back(e);
  }
  return FLCE_OK;
}

flce_status_t flce_profile_read(int kind, int64_t* launches, double* total_ms, double* flops) {
  if (kind < 0 || kind >= kKinds || !launches || !total_ms || !flops) return FLCE_ERR_INVALID_ARGUMENT;
  Profiler& P = profiler();
  std::lock_guard<std::mutex> lock(P.mu);
  const cudaError_t e = P.drain();
  *launches = P.launches[kind];
  *total_ms = P.ms[kind];
  *flops = P.flops[kind];
  return e == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA;
}

const char* flce_status_string(flce_status_t s) {
  switch (s) {
    case FLCE_OK: return "ok";
    case FLCE_ERR_INVALID_ARGUMENT: return "invalid argument";
    case FLCE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (h must be a multiple of 8, >= 8)";
    case FLCE_ERR_MISALIGNED: return "misaligned pointer";
    case FLCE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FLCE_ERR_LABEL_OUT_OF_RANGE: return "label outside [0, V) and not ignore_index";
    case FLCE_ERR_TIMEOUT: return "a bounded device wait timed out";
    case FLCE_ERR_CUDA: return "CUDA error or unsupported device";
    case FLCE_ERR_NO_DEVICE_STATUS: return "could not read the device status word";
    case FLCE_ERR_EXCEEDS_STATIC_SCRATCH: return "n exceeds the fixed scratch of flce_forward_noalloc (32768 rows)";
    case FLCE_ERR_BOUNDS: return "device: an index or TMA coordinate failed a check of the debug build";
    default: return "unknown status";
  }
}

}  // extern "C"
