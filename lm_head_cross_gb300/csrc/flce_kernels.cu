// Kernels of the fused LM-head projection + cross-entropy.
//
// One persistent, warp-specialised tcgen05 kernel template does all the dense
// work ("What-Each-Parallelism-Actually-Shards" §7.4: fuse the projection, the
// log-sum-exp, the target-logit read and the backward, so the [N,V] logits are
// never written to global memory).  Modes:
//
//   kModeForward   S = X W^T tile by tile (K = H) into TMEM; the epilogue keeps
//                  a running (max, sum-of-exp) per row over the vocabulary tiles
//                  of its split and picks out the target logit.
//   kModeFwdStore  the same, and it also writes p~ = 2^(S log2 e - r) as bf16
//                  for one row chunk (fused forward + backward), r the row's
//                  reference (its target logit) or, past a span, the tile max.
//   kModeTopk      the forward's log-sum-exp plus each row's best 16 logits
//                  and their ids per vocabulary range.
//   kModeGrad      recomputes S for one vocabulary chunk and writes
//                  G = s (exp(S - lse) - onehot) valid as bf16.
//   kModeBwd       dX and dW tiles of one chunk of G (or of p~ with per-row
//                  factors) in one launch, handed out longest-first by a
//                  global counter.
//
// CTA pairs: every launch is a grid of 2-CTA clusters.  A pair owns a 256 x 256
// output tile; each CTA stages its own 128 rows of A and its own half (128 rows)
// of B, and one thread of the even CTA issues tcgen05.mma.cta_group::2
// (256 x 256 x 16, bf16 -> fp32), which writes each CTA's 128 rows of D into
// that CTA's TMEM.  Per SM this halves the B operand traffic of a 128 x 256
// tile, so six 32 KiB stages fit in shared memory.
//
// Warp roles in each CTA: warp 0 lane 0 issues TMA loads (completion counted on
// the even CTA's barrier); warp 1 owns TMEM, and in the even CTA lane 0 issues
// the MMAs; warps 2-5 drain the other of two TMEM accumulators (2 x 256
// columns) with tcgen05.ld, one row per thread, so row reductions need no
// shuffles.  Every wait is bounded (see mbar_wait).
#include <algorithm>
#include <utility>

#include "flce_device.cuh"
#include "flce_internal.h"

namespace flce {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

constexpr int kPairM = 2 * kBM;                    // rows of a pair tile
constexpr int kHalfN = kBN / 2;                    // B rows staged by each CTA
constexpr int kAStage = kBM * kBK * 2;             // 16 KiB: this CTA's 128 rows of A
constexpr int kBStage = kHalfN * kBK * 2;          // 16 KiB: this CTA's half of B
constexpr int kStageBytes = kAStage + kBStage;     // 32 KiB
constexpr int kMnBlock = 64 * kBK * 2;             // one 64-wide MN block of 64 K rows: 8 KiB
constexpr int kStagingBuf = 32 * 128;              // 32 rows x 128 B
constexpr int kStagingPerWarp = 2 * kStagingBuf;
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr uint16_t kPairMask = 0x3;

// Per-mode shape of a CTA: epilogue warps (4, or 8 as two per TMEM lane
// quarter, each on half of a tile's columns, reported as two vocabulary
// sub-ranges) and ring stages.  Every mode runs 4 and the full ring: eight
// top-k epilogue warps with five stages were 5% faster at H = 2048 and 5%
// slower at H = 4096.
template <int MODE>
struct Cfg {
  static constexpr int kEpiWarps = 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static constexpr int kStages = flce::kStages;
  static constexpr int kSmemStagingOff = kStages * kStageBytes;
  static constexpr int kSmemBarOff = kSmemStagingOff + kEpiWarps * kStagingPerWarp;
  static constexpr int kSmemBytes = kSmemBarOff + 512 + 1024;  // barriers, ring, slot, flag; 1 KiB alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(2 * kStages + 6 + 2 * 8 + 4 + kEpiWarps <= 512 / 8, "barrier area");
};

struct Tile {
  int m0, n0;   // m0: this CTA's first row (pair base + 128 * rank); n0: first column of the 256-wide tile
  int kblocks;  // K steps of kBK
  int kind;     // 0 forward, 1 grad, 2 dX, 3 dW, 4 forward-store
  int first, last, split;
};

struct Sched {
  int unit, rt, sp, vt, ve;  // forward units
  int t;                     // grad / bwd tile index
  bool done;
  int ridx;                  // bwd: position in the tile ring
  uint32_t rphase;
};

constexpr int kRing = 8;
// Readers of each ring slot: the even CTA's MMA thread and 4 epilogue warps,
// the odd CTA's producer and 4 epilogue warps.
constexpr int kRingReaders = 10;

struct TileRing {
  volatile int* slot;  // [kRing]
  uint64_t* full;      // [kRing], one arrival (the even CTA's producer)
  uint64_t* empty;     // [kRing], kRingReaders arrivals, used in the even CTA
};

struct Pair {
  uint32_t rank;        // 0: even CTA (issues the MMAs), 1: odd CTA
  uint32_t peer;        // 1 - rank
  int id, count;        // pair index and number of pairs in the grid
};

template <int MODE>
constexpr bool kUnits = (MODE == kModeForward || MODE == kModeFwdStore || MODE == kModeTopk);

// Dynamic schedules hand out work through a global counter (p.tile_counter,
// zero at launch): the backward's tiles one by one, the forward modes' units
// (row tile, vocabulary range) one unit at a time.  A pair's first index is its
// pair index; the even CTA's producer takes every later one from the counter
// and publishes it to the pair through the tile ring.
template <int MODE>
constexpr bool kDynamic = (MODE == kModeBwd) || kUnits<MODE>;

enum Role : int { kRoleProducer = 0, kRoleMma = 1, kRoleEpilogue = 2 };

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ void fwd_unit_begin(const TcParams& p, Sched& s) {
  const int units = p.row_tiles * p.vsplit;
  if (s.unit >= units) {
    s.done = true;
    return;
  }
  unit_coords(s.unit, p.row_tiles, p.vsplit, p.units_group, &s.rt, &s.sp);
  s.vt = range_begin(s.sp, p.vocab_tiles, p.vsplit);
  s.ve = range_begin(s.sp + 1, p.vocab_tiles, p.vsplit);
}

template <int MODE>
__device__ __forceinline__ void sched_init(const TcParams& p, const Pair& pr, Sched& s) {
  s.done = false;
  s.ridx = 0;
  s.rphase = 0;
  s.t = pr.id;
  if (kUnits<MODE>) {
    s.unit = pr.id;
    fwd_unit_begin(p, s);
  }
}

// Tile of the current schedule position; m0 is this CTA's half of the pair tile.
template <int MODE>
__device__ __forceinline__ bool sched_get(const TcParams& p, const Pair& pr, const Sched& s, Tile& t) {
  const int half = static_cast<int>(pr.rank) * kBM;
  if (kUnits<MODE>) {
    if (s.done) return false;
    const int vb = range_begin(s.sp, p.vocab_tiles, p.vsplit);
    t.m0 = s.rt * kPairM + half;  // row inside the chunk [r0, row_end)
    t.n0 = s.vt * kBN;
    t.kblocks = ceil_div(p.h, kBK);
    t.kind = (MODE == kModeFwdStore) ? 4 : 0;
    t.first = (s.vt == vb);
    t.last = (s.vt == s.ve - 1);
    t.split = s.sp;
    return true;
  } else if (MODE == kModeGrad) {
    if (s.t >= p.row_tiles * p.grad_n_tiles) return false;
    t.m0 = (s.t / p.grad_n_tiles) * kPairM + half;
    t.n0 = (s.t % p.grad_n_tiles) * kBN;  // chunk-local vocabulary column
    t.kblocks = ceil_div(p.h, kBK);
    t.kind = 1;
    t.first = t.last = 0;
    t.split = 0;
    return true;
  } else {
    if (s.t >= p.dw_tiles + p.dx_tiles) return false;
    // the long tiles come first (dW when K = N, dX when K = V)
    const bool is_dx = p.dx_first ? (s.t < p.dx_tiles) : (s.t >= p.dw_tiles);
    const int u = p.dx_first ? (is_dx ? s.t : s.t - p.dx_tiles) : (is_dx ? s.t - p.dw_tiles : s.t);
    t.m0 = (u / p.h_tiles) * kPairM + half;  // dX: row of the G buffer; dW: column (vocabulary id) of the G buffer
    t.n0 = (u % p.h_tiles) * kBN;            // hidden column
    if (is_dx) {
      t.kblocks = ceil_div(p.dx_k, kBK);
      t.kind = 2;
    } else {
      t.kblocks = ceil_div(p.dw_k, kBK);
      t.kind = 3;
    }
    t.first = t.last = 0;
    t.split = 0;
    return true;
  }
}


// A wait gave up: record it, and stop both CTAs of the pair.
__device__ __forceinline__ void record_timeout(const TcParams& p, const Pair& pr, volatile int* abort_flag) {
  *abort_flag = 1;
  st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), pr.peer), 1u);
  atomicCAS(p.status, 0, kErrTimeout);
}

// Even CTA's producer: publish tile index `t` to both CTAs (a value past the
// last tile tells the readers to stop).
__device__ __forceinline__ bool ring_publish(const TcParams& p, const Pair& pr, TileRing& ring, Sched& s, int t,
                                             volatile int* abort_flag) {
  if (!mbar_wait(&ring.empty[s.ridx], s.rphase ^ 1u, p.timeout_ns, abort_flag)) return false;
  ring.slot[s.ridx] = t;
  st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(&ring.slot[s.ridx])), pr.peer), static_cast<uint32_t>(t));
  mbar_arrive(&ring.full[s.ridx]);
  mbar_arrive_cluster(mapa_shared(smem_u32(&ring.full[s.ridx]), pr.peer));
  if (++s.ridx == kRing) {
    s.ridx = 0;
    s.rphase ^= 1u;
  }
  return true;
}

// Reader side: the next published tile index.  `arrive` is true for the one
// thread per reader group that releases the slot (on the even CTA's barrier).
template <bool WHOLE_WARP>
__device__ __forceinline__ bool ring_read(const TcParams& p, TileRing& ring, Sched& s, bool arrive,
                                          volatile int* abort_flag) {
  if (!mbar_wait(&ring.full[s.ridx], s.rphase, p.timeout_ns, abort_flag)) return false;
  s.t = ring.slot[s.ridx];
  if (WHOLE_WARP) __syncwarp();  // every lane has read the slot before it is released
  if (arrive) mbar_arrive_cluster(mapa_shared(smem_u32(&ring.empty[s.ridx]), 0));
  if (++s.ridx == kRing) {
    s.ridx = 0;
    s.rphase ^= 1u;
  }
  return true;
}

// Next index of the dynamic schedule: a pair's first index is its pair index,
// the rest come from the global counter in the order the work is listed.
__device__ __forceinline__ int dynamic_next_index(const TcParams& p, const Pair& pr) {
  return pr.count + atomicAdd(p.tile_counter, 1);
}

// The pair's next index: the even CTA's producer draws and publishes it, every
// other reader (the MMA thread, the epilogue warps of both CTAs, the odd CTA's
// producer) reads it from the ring.  False if a ring wait gave up.
template <int MODE, int ROLE>
__device__ __forceinline__ bool sched_exchange(const TcParams& p, const Pair& pr, TileRing& ring, Sched& s, int lane,
                                               volatile int* abort_flag, bool first) {
  bool ok;
  if (ROLE == kRoleProducer && pr.rank == 0) {
    if (!first) s.t = dynamic_next_index(p, pr);
    ok = ring_publish(p, pr, ring, s, s.t, abort_flag);
  } else {
    ok = ring_read<ROLE == kRoleEpilogue>(p, ring, s, ROLE == kRoleEpilogue ? lane == 0 : true, abort_flag);
  }
  if (ok && kUnits<MODE>) {
    s.unit = s.t;
    fwd_unit_begin(p, s);
  }
  return ok;
}

// The first position of the schedule.
template <int MODE, int ROLE>
__device__ __forceinline__ bool sched_start(const TcParams& p, const Pair& pr, TileRing& ring, Sched& s, int lane,
                                            volatile int* abort_flag) {
  sched_init<MODE>(p, pr, s);
  if (!kDynamic<MODE>) return true;
  return sched_exchange<MODE, ROLE>(p, pr, ring, s, lane, abort_flag, true);
}

// After a tile: the next tile of the current forward unit, else the next index
// (static: pair-strided; dynamic: through the ring).
template <int MODE, int ROLE>
__device__ __forceinline__ bool sched_advance(const TcParams& p, const Pair& pr, TileRing& ring, Sched& s, int lane,
                                              volatile int* abort_flag) {
  if (kUnits<MODE> && ++s.vt < s.ve) return true;
  if (!kDynamic<MODE>) {
    s.t += pr.count;
    return true;
  }
  return sched_exchange<MODE, ROLE>(p, pr, ring, s, lane, abort_flag, false);
}

// ----------------------------------------------------------------------------- producer (TMA)

template <int MODE>
__device__ void run_producer(const TcMaps& maps, const TcParams& p, const Pair& pr, uint8_t* smem, uint64_t* full,
                             uint64_t* empty, TileRing ring, volatile int* abort_flag) {
  Sched s;
  if (!sched_start<MODE, kRoleProducer>(p, pr, ring, s, 0, abort_flag)) {
    record_timeout(p, pr, abort_flag);
    return;
  }
  const uint32_t full_even = mapa_shared(smem_u32(full), 0);  // completion is counted in the even CTA
  const int bhalf = static_cast<int>(pr.rank) * kHalfN;
  Tile t;
  int stage = 0;
  uint32_t phase = 0;
  while (sched_get<MODE>(p, pr, s, t)) {
    for (int kb = 0; kb < t.kblocks; ++kb) {
      if (!mbar_wait(&empty[stage], phase ^ 1u, p.timeout_ns, abort_flag)) {
        record_timeout(p, pr, abort_flag);
        return;
      }
      uint8_t* sa = smem + stage * kStageBytes;
      uint8_t* sb = sa + kAStage;
      const uint32_t bar = full_even + 8u * stage;
      if (pr.rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes);
      const int k0 = kb * kBK;
      // (debug builds: a load whose inner coordinate breaks the 16-byte rule is skipped and
      // recorded; the stage's transaction count then stays short and the bounded wait ends)
      if (t.kind <= 1 || t.kind == 4) {  // A = X [N,H] K-major, B = W [V,H] K-major
        const int vcol = (t.kind == 1) ? p.c0 + t.n0 : t.n0;
        if (tma_x_ok(k0, 2, p.status)) {
          tma_load_2d_pair(sa, &maps.a, bar, k0, p.r0 + t.m0);
          tma_load_2d_pair(sb, &maps.b, bar, k0, vcol + bhalf);
        }
      } else if (t.kind == 2) {  // dX: A = G K-major, B = W rows of the chunk, MN-major
        if (tma_x_ok(k0, 2, p.status)) tma_load_2d_pair(sa, &maps.a, bar, k0, t.m0);
#pragma unroll
        for (int j = 0; j < kHalfN / 64; ++j)
          if (tma_x_ok(t.n0 + bhalf + 64 * j, 2, p.status))
            tma_load_2d_pair(sb + j * kMnBlock, &maps.b, bar, t.n0 + bhalf + 64 * j, p.c0 + k0);
      } else {  // dW: A = G^T (G MN-major), B = X MN-major; K runs over token rows
#pragma unroll
        for (int j = 0; j < kBM / 64; ++j)
          if (tma_x_ok(t.m0 + 64 * j, 2, p.status))
            tma_load_2d_pair(sa + j * kMnBlock, &maps.a2, bar, t.m0 + 64 * j, k0);
#pragma unroll
        for (int j = 0; j < kHalfN / 64; ++j)
          if (tma_x_ok(t.n0 + bhalf + 64 * j, 2, p.status))
            tma_load_2d_pair(sb + j * kMnBlock, &maps.b2, bar, t.n0 + bhalf + 64 * j, p.b2_r0 + k0);
      }
      if (++stage == Cfg<MODE>::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!sched_advance<MODE, kRoleProducer>(p, pr, ring, s, 0, abort_flag)) {
      record_timeout(p, pr, abort_flag);
      return;
    }
  }
}

// ----------------------------------------------------------------------------- MMA issuer (even CTA)

template <int MODE>
__device__ void run_mma(const TcParams& p, const Pair& pr, uint8_t* smem, uint64_t* full, uint64_t* empty,
                        uint64_t* tfull, uint64_t* tempty, uint32_t tmem_base, TileRing ring,
                        volatile int* abort_flag) {
  Sched s;
  if (!sched_start<MODE, kRoleMma>(p, pr, ring, s, 0, abort_flag)) {
    record_timeout(p, pr, abort_flag);
    return;
  }
  Tile t;
  int stage = 0;
  uint32_t phase = 0;
  int acc = 0;
  uint32_t acc_phase = 0;
  while (sched_get<MODE>(p, pr, s, t)) {
    const bool a_mn = (t.kind == 3);
    const bool b_mn = (t.kind == 2 || t.kind == 3);
    const uint32_t idesc = instr_desc_bf16(kPairM, kBN, a_mn, b_mn);
    if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, p.timeout_ns, abort_flag)) {
      record_timeout(p, pr, abort_flag);
      return;
    }
    tc_fence_after_sync();
    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
    for (int kb = 0; kb < t.kblocks; ++kb) {
      if (!mbar_wait(&full[stage], phase, p.timeout_ns, abort_flag)) {
        record_timeout(p, pr, abort_flag);
        return;
      }
      tc_fence_after_sync();
      const uint32_t sa = smem_u32(smem + stage * kStageBytes);
      const uint32_t sb = sa + kAStage;
#pragma unroll
      for (int k = 0; k < kBK / 16; ++k) {
        const uint64_t ad = a_mn ? smem_desc_sw128(sa + k * 2048, kMnBlock, 1024) : smem_desc_sw128(sa + k * 32, 16, 1024);
        const uint64_t bd = b_mn ? smem_desc_sw128(sb + k * 2048, kMnBlock, 1024) : smem_desc_sw128(sb + k * 32, 16, 1024);
        umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
      }
      umma_commit_pair(&empty[stage], kPairMask);  // frees this stage in both CTAs once read
      if (++stage == Cfg<MODE>::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    umma_commit_pair(&tfull[acc], kPairMask);  // both CTAs' accumulators ready for their epilogues
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
    if (!sched_advance<MODE, kRoleMma>(p, pr, ring, s, 0, abort_flag)) {
      record_timeout(p, pr, abort_flag);
      return;
    }
  }
}

// ----------------------------------------------------------------------------- epilogue helpers

// Write one 128-byte row per lane into a 32-row staging buffer laid out the
// way a 128-byte-swizzled TMA box expects (16-byte chunk c of row r at c ^ (r & 7)).
__device__ __forceinline__ void stage_rows(uint8_t* buf, int lane, const uint32_t (&w)[32]) {
  uint8_t* row = buf + lane * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) << 4)) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

// Stage 32 rows x 128 B and hand them to a TMA store; two alternating buffers
// per warp so the next tile overlaps the previous copy.
__device__ __forceinline__ void stage_and_store(const CUtensorMap* map, uint8_t* stg, int& sbuf, int lane,
                                                const uint32_t (&w)[32], int x, int y, int* status) {
  if (!tma_x_ok(x, 4, status) || !in_bounds(y, INT32_MAX, status)) return;  // (y >= 0: no store starts above the tensor)
  uint8_t* buf = stg + sbuf * kStagingBuf;
  if (lane == 0) bulk_wait_group_read<1>();
  __syncwarp();
  stage_rows(buf, lane, w);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, buf, x, y);
    bulk_commit_group();
  }
  sbuf ^= 1;
}

// The even CTA's MMA waits for all 8 epilogue warps of the pair.
__device__ __forceinline__ void release_accumulator(uint64_t* tempty_acc, int lane) {
  tc_fence_before_sync();
  __syncwarp();
  if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(tempty_acc), 0));
}

// ----------------------------------------------------------------------------- top-k candidates
// Each epilogue thread (one row) appends (logit, id) candidates that beat its
// row's threshold to a buffer in the warp's shared-memory staging area (entry e
// of lane l at topk_slot(e, l)).  Whenever a lane holds more than
// kTopkCand - 8, the whole warp ranks that lane's entries (one per lane) and
// keeps the best k; the threshold becomes the smallest kept.

constexpr int kTopkCand = 32;

struct TopkBuf {
  float* val;    // [kTopkCand][32]
  int* idx;      // [kTopkCand][32]
  int count;
  float thr;
  unsigned* shared_thr;  // the row's threshold shared by all its vocabulary ranges (global memory), or null
};

// Word of entry e of lane l's buffer.  Rows of 32 words, the lane index XORed
// with the entry: a warp appending at equal counts, and a warp reading one
// lane's whole buffer (entry e by lane e), both touch 32 different banks.
__device__ __forceinline__ int topk_slot(int e, int l) { return e * 32 + (l ^ e); }

// Order-preserving map of a float to an unsigned (0 stands below every float).
__device__ __forceinline__ unsigned topk_key(float f) {
  const unsigned b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float topk_unkey(unsigned u) {
  if (u == 0u) return -INFINITY;
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

__device__ __forceinline__ bool topk_better(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && static_cast<unsigned>(ai) < static_cast<unsigned>(bi));
}

// Compact the buffers of every lane in `mask` (whole-warp call), keeping each
// row's best `keep` (= k, at most kTopkMax).  Lane e holds entry e of the
// buffer; its rank (how many entries beat it) comes from 32 independent shuffle
// rounds, and the best `keep` go to slots 0..keep-1 in rank order.  Entries are
// distinct (value, id) pairs, so the ranks of the filled slots are distinct.
__device__ __forceinline__ void topk_compact_lanes(TopkBuf& b, int lane, unsigned mask, int keep) {
  while (mask) {
    const int L = __ffs(mask) - 1;
    mask &= mask - 1;
    const int cnt = __shfl_sync(0xffffffffu, b.count, L);
    const bool filled = lane < cnt;
    const float v = filled ? b.val[topk_slot(lane, L)] : -INFINITY;
    const int i = filled ? b.idx[topk_slot(lane, L)] : -1;
    int rank = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float ov = __shfl_sync(0xffffffffu, v, j);
      const int oi = __shfl_sync(0xffffffffu, i, j);
      rank += topk_better(ov, oi, v, i) ? 1 : 0;
    }
    __syncwarp();  // every entry is in registers before the slots are rewritten
    if (filled && rank < keep) {
      b.val[topk_slot(rank, L)] = v;
      b.idx[topk_slot(rank, L)] = i;
    }
    const unsigned at_k = __ballot_sync(0xffffffffu, filled && rank == keep - 1);
    const float kth = __shfl_sync(0xffffffffu, v, at_k ? __ffs(at_k) - 1 : 0);
    __syncwarp();
    if (lane == L) {
      b.count = min(cnt, keep);
      if (cnt >= keep && at_k) {
        b.thr = kth;
        // `keep` values of this row are >= kth, so any value below it, in any range, is out
        if (b.shared_thr) atomicMax(b.shared_thr, topk_key(kth));
      }
    }
  }
}

// ----------------------------------------------------------------------------- epilogue

// Forward-store: a row's tile sum above this means some p~ may exceed 2^kRefSpan.
constexpr float kRefSumMax = 18446744073709551616.0f;  // 2^64
static_assert(kRefSpan == 64.f, "kRefSumMax is 2^kRefSpan");

// One 64-column group of a row: p~ = 2^(t log2 e - ref) packed as bf16 pairs
// into w, and their fp32 sum (columns at or past nv count as 0).
__device__ __forceinline__ float exp_pack_group(const uint32_t (&v)[64], uint32_t (&w)[32], int nv, float ref) {
  if (nv >= 64) {  // full group: no column test, four independent sums
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float a = fast_exp2(fmaf(__uint_as_float(v[2 * j]), kLog2e, -ref));
      const float b = fast_exp2(fmaf(__uint_as_float(v[2 * j + 1]), kLog2e, -ref));
      s4[j & 3] += a + b;
      w[j] = pack_bf16x2(a, b);
    }
    return (s4[0] + s4[1]) + (s4[2] + s4[3]);
  }
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float a = (2 * j < nv) ? fast_exp2(fmaf(__uint_as_float(v[2 * j]), kLog2e, -ref)) : 0.f;
    const float b = (2 * j + 1 < nv) ? fast_exp2(fmaf(__uint_as_float(v[2 * j + 1]), kLog2e, -ref)) : 0.f;
    sum += a + b;
    w[j] = pack_bf16x2(a, b);
  }
  return sum;
}

template <int MODE>
__device__ void run_epilogue(const TcMaps& maps, const TcParams& p, const Pair& pr, uint8_t* staging, uint64_t* tfull,
                             uint64_t* tempty, uint32_t tmem_base, TileRing ring, uint64_t* ebar,
                             volatile int* abort_flag) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int quarter = warp & 3;  // a warp may only touch TMEM lanes [32*(warp%4), +32)
  const int r = quarter * 32 + lane;
  // top-k: the second set of four warps takes the upper half of each tile's
  // columns and reports it as its own vocabulary sub-range (split 2s + 1)
  const int ehalf = (warp - 2) >> 2;
  constexpr int kChunkCols = kBN / 32 / (Cfg<MODE>::kEpiWarps / 4);  // 32-column chunks per warp and tile
  uint8_t* stg = staging + (warp - 2) * kStagingPerWarp;
  int sbuf = 0;
  uint64_t* my_ebar = &ebar[warp - 2];  // TMA loads into this warp's staging buffers
  uint32_t ephase = 0;

  Sched s;
  if (!sched_start<MODE, kRoleEpilogue>(p, pr, ring, s, lane, abort_flag)) {
    record_timeout(p, pr, abort_flag);
    return;
  }
  Tile t;
  int acc = 0;
  uint32_t acc_phase = 0;

  // forward state (one row per thread)
  TopkBuf tk;
  tk.val = reinterpret_cast<float*>(stg);
  tk.idx = reinterpret_cast<int*>(stg + kTopkCand * 32 * sizeof(float));
  tk.count = 0;
  tk.thr = -INFINITY;
  tk.shared_thr = nullptr;
  float gthr = -INFINITY;  // top-k: the row's shared threshold as last read
  static_assert(kTopkCand * 32 * 8 <= kStagingPerWarp, "top-k candidates fit the staging area");
  float run_m = -INFINITY, run_l = 0.f, z_tgt = 0.f;
  bool found = false;
  int y_fwd = p.ignore_index;
  float ref_row = 0.f;  // forward-store: the row's reference exponent, log2 units
  const float scale = (MODE == kModeGrad) ? *p.scale : 0.f;
  const int row_end = p.row_end > 0 ? p.row_end : p.n;

  while (sched_get<MODE>(p, pr, s, t)) {
    // top-k: the row's shared threshold, loaded before the wait so that the wait
    // hides its latency (an older value only keeps more candidates)
    unsigned thr_key = 0u;
    if (MODE == kModeTopk) {
      const int row = p.r0 + t.m0 + r;
      if (p.topk_thr && row < row_end) thr_key = *reinterpret_cast<volatile unsigned*>(p.topk_thr + row);
    }
    if (!mbar_wait(&tfull[acc], acc_phase, p.timeout_ns, abort_flag)) {
      record_timeout(p, pr, abort_flag);
      break;
    }
    __syncwarp();
    tc_fence_after_sync();
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * kBN);

    if (kUnits<MODE>) {
      const int lrow = t.m0 + r;   // row inside the chunk
      const int row = p.r0 + lrow;  // row of X
      if (t.first) {
        run_m = -INFINITY;
        run_l = 0.f;
        found = false;
        y_fwd = (row < row_end) ? label_at(p.labels, row, p.shift, p.seq_len, p.ignore_index) : p.ignore_index;
        if (MODE == kModeFwdStore) ref_row = (row < p.n) ? p.mref[row] : 0.f;
        if (MODE == kModeTopk) {
          tk.count = 0;
          tk.thr = -INFINITY;
          tk.shared_thr = (p.topk_thr && row < row_end) ? p.topk_thr + row : nullptr;
        }
      }
      if (MODE == kModeTopk && tk.shared_thr) gthr = topk_unkey(thr_key);
      if (MODE == kModeTopk && t.first) {
        // Before a range's first tile fills the candidate buffer from nothing: each of
        // the tile's 16 disjoint 16-column groups holds its max, so at least kTopkMax
        // values of the row are >= the smallest of those maxima, and nothing below it
        // can be among the row's best kTopkMax.  Raise the row's threshold to it.
        static_assert(kChunkCols * 2 >= kTopkMax, "one warp sees kTopkMax column groups of a tile");
        float t0 = INFINITY;
#pragma unroll 1
        for (int c = ehalf * kChunkCols; c < ehalf * kChunkCols + kTopkMax / 2; ++c) {
          const int col0 = t.n0 + c * 32;
          if (col0 >= p.v) {  // fewer than kTopkMax groups hold a value
            t0 = -INFINITY;
            break;
          }
          __syncwarp();
          uint32_t v[32];
          tmem_ld_32x32(tbase + c * 32, v);
          const int nv = min(32, p.v - col0);
          float g0 = -INFINITY, g1 = -INFINITY;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if (j < nv) g0 = fmaxf(g0, __uint_as_float(v[j]));
            if (j + 16 < nv) g1 = fmaxf(g1, __uint_as_float(v[j + 16]));
          }
          t0 = fminf(t0, fminf(g0, g1));
        }
        if (t0 > gthr) {
          gthr = t0;
          if (tk.shared_thr) atomicMax(tk.shared_thr, topk_key(t0));
        }
      }
      if (MODE == kModeForward || MODE == kModeTopk) {
        // 32 columns per TMEM load (64 measured the same for the forward and ran
        // slower for top-k, whose candidate code then unrolls over 64 columns)
        constexpr int kW = 32;
        constexpr int kGroups = kChunkCols;  // groups per warp and tile
#pragma unroll 1
        for (int c = ehalf * kGroups; c < (ehalf + 1) * kGroups; ++c) {
          const int col0 = t.n0 + c * kW;
          if (col0 >= p.v) break;  // same for the whole warp
          __syncwarp();
          uint32_t v[kW];
          tmem_ld_32x32(tbase + c * kW, v);
          const int yi = y_fwd - col0;
          if (static_cast<unsigned>(yi) < static_cast<unsigned>(kW)) {
#pragma unroll
            for (int j = 0; j < kW; ++j)
              if (j == yi) z_tgt = __uint_as_float(v[j]);
            found = true;
          }
          const int nv = min(kW, p.v - col0);
          if (nv < kW) {
#pragma unroll
            for (int j = 0; j < kW; ++j)
              if (j >= nv) v[j] = __float_as_uint(-INFINITY);
          }
          constexpr int kBlocks = kW / 8;
          float gmax[kBlocks];  // maxima of the group's 8-column blocks
#pragma unroll
          for (int hh = 0; hh < kBlocks; ++hh) {
            gmax[hh] = __uint_as_float(v[8 * hh]);
#pragma unroll
            for (int j = 8 * hh + 1; j < 8 * hh + 8; ++j) gmax[hh] = fmaxf(gmax[hh], __uint_as_float(v[j]));
          }
          float cmax = gmax[0];
#pragma unroll
          for (int hh = 1; hh < kBlocks; ++hh) cmax = fmaxf(cmax, gmax[hh]);
          const float new_m = fmaxf(run_m, cmax * kLog2e);
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < kW; ++j) s4[j & 3] += fast_exp2(fmaf(__uint_as_float(v[j]), kLog2e, -new_m));
          run_l = run_l * fast_exp2(run_m - new_m) + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
          run_m = new_m;
          if (MODE == kModeTopk) {
            // blocks of 8: a buffer holding at most kTopkCand - 8 never overflows, and a
            // lane is compacted only once it has gathered more than that
            // a value must beat this range's own 16th best (ids grow along the range, so an
            // equal later value ranks after it) and be no lower than the row's shared threshold
            // (a block whose max no lane keeps is skipped whole)
            if (__any_sync(0xffffffffu, cmax > tk.thr && cmax >= gthr)) {
#pragma unroll
              for (int hh = 0; hh < kBlocks; ++hh) {
                if (!__any_sync(0xffffffffu, gmax[hh] > tk.thr && gmax[hh] >= gthr)) continue;
#pragma unroll
                for (int j = 8 * hh; j < 8 * hh + 8; ++j) {
                  const float x = __uint_as_float(v[j]);
                  const bool keep = x > tk.thr && x >= gthr;
                  const int slot = topk_slot(tk.count, lane);
                  if (keep) {  // predicated stores, no branch
                    tk.val[slot] = x;
                    tk.idx[slot] = col0 + j;
                  }
                  tk.count += keep ? 1 : 0;
                }
                topk_compact_lanes(tk, lane, __ballot_sync(0xffffffffu, tk.count > kTopkCand - 8), p.topk_k);
              }
            }
          }
        }
        release_accumulator(&tempty[acc], lane);
      } else {
        // forward-store, one pass: p~ = 2^(t log2 e - r) as bf16 into the chunk
        // buffer (relative error 2^-9), its fp32 sum into the running log-sum-exp,
        // r the row's reference (its target logit; another of its logits for a
        // row without a gradient).  A tile whose sum exceeds 2^kRefSpan — so a
        // value may — is written again relative to its own max.
        float ref = ref_row;
        float sum = 0.f;
#pragma unroll 1
        for (int g = 0; g < kBN / 64; ++g) {
          const int col0 = t.n0 + g * 64;
          if (col0 >= p.v) break;  // same for the whole warp
          __syncwarp();
          uint32_t v[64];
          tmem_ld_32x64(tbase + g * 64, v);
          const int yi = y_fwd - col0;
          if (static_cast<unsigned>(yi) < 64u) {
#pragma unroll
            for (int j = 0; j < 64; ++j)
              if (j == yi) z_tgt = __uint_as_float(v[j]);
            found = true;
          }
          const int nv = p.v - col0;
          uint32_t w[32];
          sum += exp_pack_group(v, w, nv, ref);
          stage_and_store(&maps.out, stg, sbuf, lane, w, col0, t.m0 + quarter * 32, p.status);
        }
        const bool over = !(sum <= kRefSumMax);  // also true for a non-finite sum
        if (__any_sync(0xffffffffu, over)) {
          // again relative to the tile's max, for the rows that need it (the others
          // rewrite the same bytes); the first pass's stores land first
          if (lane == 0) bulk_wait_group_all();
          __syncwarp();
          float tmax = -INFINITY;
#pragma unroll 1
          for (int c = 0; c < kBN / 32; ++c) {
            const int col0 = t.n0 + c * 32;
            if (col0 >= p.v) break;
            __syncwarp();
            uint32_t v[32];
            tmem_ld_32x32(tbase + c * 32, v);
            const int nv = p.v - col0;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nv) tmax = fmaxf(tmax, __uint_as_float(v[j]));
          }
          if (over) {
            ref = tmax * kLog2e;
            sum = 0.f;
          }
#pragma unroll 1
          for (int g = 0; g < kBN / 64; ++g) {
            const int col0 = t.n0 + g * 64;
            if (col0 >= p.v) break;
            __syncwarp();
            uint32_t v[64];
            tmem_ld_32x64(tbase + g * 64, v);
            uint32_t w[32];
            const float gs = exp_pack_group(v, w, p.v - col0, ref);
            if (over) sum += gs;
            stage_and_store(&maps.out, stg, sbuf, lane, w, col0, t.m0 + quarter * 32, p.status);
          }
        }
        release_accumulator(&tempty[acc], lane);
        const int64_t mi = static_cast<int64_t>(lrow) * p.vocab_tiles + t.n0 / kBN;
        if (row < row_end && in_bounds(mi, p.mtile_count, p.status)) p.mtile[mi] = ref;
        const float new_m = fmaxf(run_m, ref);
        run_l = run_l * fast_exp2(run_m - new_m) + sum * fast_exp2(ref - new_m);
        run_m = new_m;
      }
      if (MODE == kModeTopk && t.last)
        topk_compact_lanes(tk, lane, __ballot_sync(0xffffffffu, tk.count > p.topk_k), p.topk_k);
      if (t.last && row < row_end) {
        const int osplit = (Cfg<MODE>::kEpiWarps == 8) ? 2 * t.split + ehalf : t.split;
        const int64_t pi = static_cast<int64_t>(osplit) * p.n + row;
        if (in_bounds(pi, p.part_count, p.status)) {
          p.part_m[pi] = run_m;
          p.part_l[pi] = run_l;
        }
        if (found && in_bounds(row, p.n, p.status)) p.tgt[row] = z_tgt;
        if (MODE == kModeTopk) {
          const int kept = tk.count;  // at most k (the merge does not need them sorted)
          const int64_t base = (static_cast<int64_t>(osplit) * p.n + row) * kTopkMax;
          for (int i = 0; i < kTopkMax; ++i) {
            if (!in_bounds(base + i, p.topk_count, p.status)) break;
            p.topk_val[base + i] = i < kept ? tk.val[topk_slot(i, lane)] : -INFINITY;
            p.topk_idx[base + i] = i < kept ? tk.idx[topk_slot(i, lane)] : -1;
          }
        }
      }
    } else if (MODE == kModeGrad) {
      const int row = t.m0 + r;
      // soft targets: G / s = Q p here (the per-row coefficient carries s Q_i), the
      // targets' -s q_k are subtracted from the stored chunk afterwards
      const int y = (row >= p.n) ? p.ignore_index
                                 : (p.soft_grad ? kNotOwned : label_at(p.labels, row, p.shift, p.seq_len, p.ignore_index));
      const bool valid = (row < p.n) && (p.soft_grad || y != p.ignore_index);
      const float coef = valid ? (p.grad_rows ? p.grad_rows[row] : scale) : 0.f;
      const float lse2 = (row < p.n) ? p.lse[row] * kLog2e : 0.f;
      const int ycol = y - (p.c0 + t.n0);  // label position inside this tile (if any)
#pragma unroll 1
      for (int g = 0; g < kBN / 64; ++g) {
        if (t.n0 + g * 64 >= p.cw) break;
        __syncwarp();
        uint32_t v[64];
        tmem_ld_32x64(tbase + g * 64, v);
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int c = g * 64 + 2 * j;
          float a = fast_exp2(fmaf(__uint_as_float(v[2 * j]), kLog2e, -lse2));
          float b = fast_exp2(fmaf(__uint_as_float(v[2 * j + 1]), kLog2e, -lse2));
          a = coef * (a - (c == ycol ? 1.f : 0.f));
          b = coef * (b - (c + 1 == ycol ? 1.f : 0.f));
          w[j] = pack_bf16x2(a, b);
        }
        // columns at or beyond the chunk width fall outside the store box's tensor and are dropped by TMA
        stage_and_store(&maps.out, stg, sbuf, lane, w, t.n0 + g * 64, t.m0 + quarter * 32, p.status);
      }
      release_accumulator(&tempty[acc], lane);
    } else {
      // dX tile: rows of X (offset r0), written to maps.out; dW tile: vocabulary
      // rows (offset c0), written to maps.out2.
      const bool is_dx = (t.kind == 2);
      const CUtensorMap* omap = is_dx ? &maps.out : &maps.out2;
      const int omode = is_dx ? p.dx_out : p.dw_out;
      const int y0 = (is_dx ? p.r0 : p.c0) + t.m0 + quarter * 32;
      // With per-row factors f the buffer holds G / (s f_i) row by row: a dX row
      // is scaled by s f_i, a dW tile (whose B operand rows are f_i x_i) by s.
      float osc = 1.f;
      if (p.rowscale) {
        osc = *p.scale;
        if (is_dx) {
          const int lr = t.m0 + quarter * 32 + lane;
          osc = (p.r0 + lr < p.row_end && in_bounds(lr, p.rowscale_count, p.status)) ? osc * p.rowscale[lr] : 0.f;
        }
      }
      if (omode == kOutF32AccToBF16) {
        // last row chunk: dW = accumulator (fp32, earlier chunks) + this chunk, written as bf16
#pragma unroll 1
        for (int g = 0; g < kBN / 64; ++g) {
          if (t.n0 + g * 64 >= p.h) break;
          if (lane == 0) {
            bulk_wait_group_read<0>();  // earlier stores are done with both staging buffers
            mbar_arrive_expect_tx(my_ebar, 2 * kStagingBuf);
            tma_load_2d(stg, &maps.out2, my_ebar, t.n0 + g * 64, y0);
            tma_load_2d(stg + kStagingBuf, &maps.out2, my_ebar, t.n0 + g * 64 + 32, y0);
          }
          __syncwarp();
          uint32_t v[64];
          tmem_ld_32x64(tbase + g * 64, v);
          if (!mbar_wait(my_ebar, ephase, p.timeout_ns, abort_flag)) {
            record_timeout(p, pr, abort_flag);
            break;
          }
          ephase ^= 1u;
          uint32_t w[32];
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const uint8_t* rowp = stg + hb * kStagingBuf + lane * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const float4 a = *reinterpret_cast<const float4*>(rowp + ((c ^ (lane & 7)) << 4));
              const int j = hb * 32 + 4 * c;
              w[j / 2] = pack_bf16x2(fmaf(__uint_as_float(v[j]), osc, a.x), fmaf(__uint_as_float(v[j + 1]), osc, a.y));
              w[j / 2 + 1] =
                  pack_bf16x2(fmaf(__uint_as_float(v[j + 2]), osc, a.z), fmaf(__uint_as_float(v[j + 3]), osc, a.w));
            }
          }
          __syncwarp();  // every lane has read the fp32 rows before buffer 0 is rewritten
          stage_rows(stg, lane, w);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&maps.out3, stg, t.n0 + g * 64, y0);
            bulk_commit_group();
          }
          sbuf = 1;  // a store may still read buffer 0
        }
      } else if (omode == kOutBF16) {
#pragma unroll 1
        for (int g = 0; g < kBN / 64; ++g) {
          if (t.n0 + g * 64 >= p.h) break;
          __syncwarp();
          uint32_t v[64];
          tmem_ld_32x64(tbase + g * 64, v);
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            w[j] = pack_bf16x2(__uint_as_float(v[2 * j]) * osc, __uint_as_float(v[2 * j + 1]) * osc);
          stage_and_store(omap, stg, sbuf, lane, w, t.n0 + g * 64, y0, p.status);
        }
      } else {
        // fp32 accumulator (the bounded path's dX, the row-chunk path's dW before its last
        // chunk): the staged rows are read back four rows per warp instruction and stored /
        // added at L2 with 16-byte accesses from the epilogue warps, which keeps this
        // traffic (a tile's 128 KiB per CTA, every 64 K steps for the bounded path's dX
        // tiles) off the TMA unit that feeds the operand stages
        float* const fbase = is_dx ? p.dx_f32 : p.dw_f32;
        const int frows = fbase ? (is_dx ? p.n : p.v) : 0;  // no address: nothing written, error recorded
        if (!fbase && lane == 0) atomicCAS(p.status, 0, kErrBounds);
        if (lane == 0) bulk_wait_group_read<0>();  // earlier TMA stores are done with the staging buffers
        __syncwarp();
#pragma unroll 1
        for (int c = 0; c < kBN / 32; ++c) {
          if (t.n0 + c * 32 >= p.h) break;
          __syncwarp();
          uint32_t v[32];
          tmem_ld_32x32(tbase + c * 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * osc);
          stage_rows(stg, lane, v);
          __syncwarp();
          const int x = t.n0 + c * 32 + (lane & 7) * 4;  // h is a multiple of 8: x < h means x + 4 <= h
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int rr = q * 4 + (lane >> 3);
            const int yy = y0 + rr;
            const uint4 val = *reinterpret_cast<const uint4*>(stg + rr * 128 + (((lane & 7) ^ (rr & 7)) << 4));
            const int64_t at = static_cast<int64_t>(yy) * p.h + x;
            if (yy < frows && x < p.h && in_bounds(at + 3, static_cast<int64_t>(frows) * p.h, p.status)) {
              if (omode == kOutF32Add)
                red_add_v4_f32(fbase + at, val);
              else
                *reinterpret_cast<uint4*>(fbase + at) = val;
            }
          }
          __syncwarp();  // every lane has read the staged rows before the next group rewrites them
        }
      }
      release_accumulator(&tempty[acc], lane);
    }
    acc ^= 1;
    if (acc == 0) acc_phase ^= 1u;
    if (!sched_advance<MODE, kRoleEpilogue>(p, pr, ring, s, lane, abort_flag)) {
      record_timeout(p, pr, abort_flag);
      break;
    }
  }
  if (lane == 0) bulk_wait_group_all();
  __syncwarp();
}

// ----------------------------------------------------------------------------- the kernel

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg<MODE>::kThreads, 1)
    tc_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
  // The prologue (barriers, TMEM, tensor-map prefetch) reads no global memory,
  // so it runs before the wait for the previous kernel (griddep_begin below).
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int kSt = Cfg<MODE>::kStages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg<MODE>::kSmemBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + kSt;
  uint64_t* tfull = bars + 2 * kSt;
  uint64_t* tempty = bars + 2 * kSt + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kSt + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kSt + 5);
  TileRing ring;
  ring.full = bars + 2 * kSt + 6;
  ring.empty = ring.full + kRing;
  ring.slot = reinterpret_cast<volatile int*>(ring.empty + kRing);
  uint64_t* ebar = ring.empty + kRing + kRing / 2;  // after the 8 slot ints: one per epilogue warp

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  Pair pr;
  pr.rank = cluster_ctarank();
  pr.peer = pr.rank ^ 1u;
  pr.id = static_cast<int>(blockIdx.x >> 1);
  pr.count = static_cast<int>(gridDim.x >> 1);

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < kSt; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 2 * Cfg<MODE>::kEpiWarps);  // one arrival per epilogue warp of the pair
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&ring.full[i], 1);
      mbar_init(&ring.empty[i], kRingReaders);
    }
    for (int i = 0; i < Cfg<MODE>::kEpiWarps; ++i) mbar_init(&ebar[i], 1);
    *abort_flag = 0;
    mbar_fence_init();
    fence_proxy_async_smem();
    tma_prefetch_map(&maps.a);
    tma_prefetch_map(&maps.b);
    if (MODE != kModeForward) tma_prefetch_map(&maps.out);  // grad / forward-store / bwd
    if (MODE == kModeBwd) {
      tma_prefetch_map(&maps.a2);
      tma_prefetch_map(&maps.b2);
      tma_prefetch_map(&maps.out2);
      if (p.dw_out == kOutF32AccToBF16) tma_prefetch_map(&maps.out3);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync_all();  // barriers of both CTAs initialised before any cross-CTA arrival
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // Wait for the previous kernel before touching memory it may write.  In the
  // forward modes the producer and MMA threads read only X and W, which no
  // kernel of the library writes, so they start the contraction at once and
  // only the epilogue (which reads the row state and writes the outputs) waits.
  if (!kUnits<MODE> || warp >= 2) griddep_wait();
  griddep_launch();
  if (p.zero_words && blockIdx.x == 0 && threadIdx.x == 64) {  // an epilogue thread: after the wait
    p.zero_words[0] = 0;
    p.zero_words[1] = 0;
  }

  if (warp == 0) {
    if (lane == 0) run_producer<MODE>(maps, p, pr, smem, full, empty, ring, abort_flag);
  } else if (warp == 1) {
    if (lane == 0 && pr.rank == 0) run_mma<MODE>(p, pr, smem, full, empty, tfull, tempty, tmem_base, ring, abort_flag);
  } else {
    run_epilogue<MODE>(maps, p, pr, smem + Cfg<MODE>::kSmemStagingOff, tfull, tempty, tmem_base, ring, ebar,
                       abort_flag);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (*abort_flag) {
    // A wait gave up: let copies and MMAs already in flight land before the
    // shared memory and TMEM are released (they finish in microseconds).
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 2000000ull) {
    }
  }
  cluster_sync_all();  // no CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ----------------------------------------------------------------------------- small kernels

// Merge a row's per-range (reference, sum) pairs: returns lse in log2 units
// and the largest reference in *m_out.  Loads are issued 16 ranges at a time
// before their first use, so a row costs one or two memory latencies rather
// than one per range.
__device__ __forceinline__ float merge_ranges(const float* __restrict__ part_m, const float* __restrict__ part_l,
                                              int vsplit, int n, int row, float* m_out) {
  constexpr int kBatch = 16;
  float m = -INFINITY, l = 0.f;
  for (int b = 0; b < vsplit; b += kBatch) {
    float pm[kBatch], pl[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int s = b + k;
      pm[k] = s < vsplit ? part_m[static_cast<int64_t>(s) * n + row] : -INFINITY;
      pl[k] = s < vsplit ? part_l[static_cast<int64_t>(s) * n + row] : 0.f;
    }
    float bm = -INFINITY;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) bm = fmaxf(bm, pm[k]);
    const float nm = fmaxf(m, bm);
    float bl = 0.f;
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      if (b + k < vsplit) bl += pl[k] * exp2f(pm[k] - nm);
    l = l * exp2f(m - nm) + bl;
    m = nm;
  }
  *m_out = m;
  return m + log2f(l);
}

// Merge the per-split (max, sum) pairs of each row into lse, check its label,
// and reduce the per-row losses of the block in a fixed order.
// Rows [r0, r0 + rows) of an n-row problem; r0 is a multiple of the block size,
// and block b writes partial r0 / kFinalizeThreads + b.
__global__ void __launch_bounds__(kFinalizeThreads) fwd_finalize_kernel(
    int r0, int rows, int n, int v, int vsplit, LabelView lv, const float* __restrict__ part_m,
    const float* __restrict__ part_l, const float* __restrict__ tgt, float* __restrict__ lse_out,
    float* __restrict__ loss_rows, double* __restrict__ blk_loss, int* __restrict__ blk_valid,
    int* __restrict__ status) {
  griddep_begin();
  const int ignore_index = lv.ignore_index;
  __shared__ double s_loss[kFinalizeThreads];
  __shared__ int s_valid[kFinalizeThreads];
  const int row = r0 + blockIdx.x * kFinalizeThreads + threadIdx.x;
  double li = 0.0;
  int valid = 0;
  if (row < r0 + rows) {
    float m;
    const float lse = merge_ranges(part_m, part_l, vsplit, n, row, &m) * kLn2;
    lse_out[row] = lse;
    if (lv.soft_k > 0) {
      // KL(q || p) over the row's targets: sum_t q_t log q_t + Q lse - sum_t q_t z_t, Q = sum_t q_t
      // (tgt holds sum_t q_t z_t; target ids were checked when it was gathered)
      double qd = 0.0, cd = 0.0;
      for (int t = 0; t < lv.soft_k; ++t) {
        const float q = lv.soft_prob[static_cast<int64_t>(row) * lv.soft_k + t];
        if (q > 0.f) {
          qd += static_cast<double>(q);
          cd += static_cast<double>(q) * log(static_cast<double>(q));
        }
      }
      if (qd > 0.0) {
        valid = 1;
        li = cd + qd * static_cast<double>(lse) - static_cast<double>(tgt[row]);
      }
    } else {
      const int y = label_at(lv.labels, row, lv.shift, lv.seq_len, ignore_index);
      if (y != ignore_index) {
        if (y >= 0 && y < v) {
          valid = 1;
          li = static_cast<double>(lse) - static_cast<double>(tgt[row]);
        } else {
          atomicCAS(status, 0, kErrLabel);
        }
      }
    }
    if (loss_rows) loss_rows[row] = static_cast<float>(li);
  }
  s_loss[threadIdx.x] = li;
  s_valid[threadIdx.x] = valid;
  __syncthreads();
  for (int w = kFinalizeThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      s_loss[threadIdx.x] += s_loss[threadIdx.x + w];
      s_valid[threadIdx.x] += s_valid[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    blk_loss[r0 / kFinalizeThreads + blockIdx.x] = s_loss[0];
    blk_valid[r0 / kFinalizeThreads + blockIdx.x] = s_valid[0];
  }
}

// One row of a chunk buffer: p~ 2^(ref_tile - lse2) times c, less c q at the
// target ids (q = 1 at y for a hard label), as bf16, in place.
__device__ __forceinline__ void fixup_row(uint4* __restrict__ prow, const float* __restrict__ mt, int v, float lse2,
                                          float coef, float mass, int y, int nsoft, const int* s_idx,
                                          const float* s_q, int q_begin = 0, int q_end = -1) {
  constexpr int kUnroll = 4;  // 16-byte loads in flight per thread
  const int nvec = q_end < 0 ? (v + 7) / 8 : q_end;  // 8-column groups [q_begin, nvec)
  for (int base = q_begin + threadIdx.x; base < nvec; base += blockDim.x * kUnroll) {
    uint4 u[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int q = base + k * blockDim.x;
      if (q < nvec) u[k] = prow[q];
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int q = base + k * blockDim.x;
      if (q >= nvec) break;
      const int j0 = q * 8;
      const float c = coef * mass * fast_exp2(mt[j0 / kBN] - lse2);
      const uint32_t in[4] = {u[k].x, u[k].y, u[k].z, u[k].w};
      float sub[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) sub[e] = (j0 + e == y) ? coef : 0.f;
      for (int t = 0; t < nsoft; ++t) {
        const int d = s_idx[t] - j0;
        if (static_cast<unsigned>(d) < 8u) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e == d) sub[e] += coef * s_q[t];
        }
      }
      uint32_t out[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = j0 + 2 * e;
        const float lo = __uint_as_float(in[e] << 16);
        const float hi = __uint_as_float(in[e] & 0xFFFF0000u);
        const float g0 = (j < v) ? fmaf(lo, c, -sub[2 * e]) : 0.f;
        const float g1 = (j + 1 < v) ? fmaf(hi, c, -sub[2 * e + 1]) : 0.f;
        out[e] = pack_bf16x2(g0, g1);
      }
      prow[q] = make_uint4(out[0], out[1], out[2], out[3]);
    }
  }
}

// x . w over h bf16 pairs, one warp: fp32 accumulation of the exact
// products, lanes over 16-byte pieces, then a butterfly sum (every lane holds it).
__device__ __forceinline__ float warp_dot_bf16(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w,
                                               int h, int lane) {
  const uint4* xr = reinterpret_cast<const uint4*>(x);
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  float dot = 0.f;
  for (int c = lane; c < h / 8; c += 32) {
    const uint4 a = xr[c], b = wr[c];
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      dot = fmaf(__uint_as_float(av[e] << 16), __uint_as_float(bv[e] << 16), dot);
      dot = fmaf(__uint_as_float(av[e] & 0xFFFF0000u), __uint_as_float(bv[e] & 0xFFFF0000u), dot);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
  return dot;
}

// Fused path, before the first row chunk.  One warp per row: the label check
// and the row's reference in log2 units — for a hard label its target logit
// x_i . w_{y_i}, for soft targets the q-weighted mean of the target logits
// (whose q-weighted sum, the KL's cross term, goes to tgt), for a row without
// a gradient its logit of vocabulary id 0; one valid count per block of 8 rows.  The last block to
// finish (ticket) adds the counts into n_valid and the gradient scale s, and
// resets the ticket.
__global__ void __launch_bounds__(256) label_prep_kernel(int n, int h, int v, int reduction, LabelView lv,
                                                         const __nv_bfloat16* __restrict__ X,
                                                         const __nv_bfloat16* __restrict__ W, float* __restrict__ mref,
                                                         float* __restrict__ tgt, int* __restrict__ blk_cnt,
                                                         int* __restrict__ ticket, int* __restrict__ n_valid_out,
                                                         float* __restrict__ scale_out, int* __restrict__ status) {
  griddep_begin();
  __shared__ int s_valid[8];
  __shared__ long long s_sum[256];
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 8 + warp;
  int valid = 0;
  if (row < n) {
    const __nv_bfloat16* xrow = X + static_cast<int64_t>(row) * h;
    float ref = INFINITY;
    if (lv.soft_k > 0) {
      float Q = 0.f, acc = 0.f;
      for (int t = 0; t < lv.soft_k; ++t) {
        const float q = lv.soft_prob[static_cast<int64_t>(row) * lv.soft_k + t];
        const int id = lv.soft_idx[static_cast<int64_t>(row) * lv.soft_k + t];
        if (!(q > 0.f)) continue;
        Q += q;
        if (id < 0 || id >= v) {
          if (lane == 0) atomicCAS(status, 0, kErrLabel);
          continue;
        }
        acc = fmaf(q, warp_dot_bf16(xrow, W + static_cast<int64_t>(id) * h, h, lane), acc);
      }
      if (lane == 0) tgt[row] = acc;
      if (Q > 0.f) {
        valid = 1;
        ref = acc / Q * kLog2e;
      }
    } else {
      const int y = label_at(lv.labels, row, lv.shift, lv.seq_len, lv.ignore_index);
      if (y != lv.ignore_index) {
        if (y >= 0 && y < v) {
          valid = 1;
          ref = warp_dot_bf16(xrow, W + static_cast<int64_t>(y) * h, h, lane) * kLog2e;
        } else if (lane == 0) {
          atomicCAS(status, 0, kErrLabel);
        }
      }
    }
    if (!valid) ref = warp_dot_bf16(xrow, W, h, lane) * kLog2e;
    if (lane == 0) mref[row] = ref;
  }
  if (lane == 0) s_valid[warp] = valid;
  __syncthreads();
  if (threadIdx.x == 0) {
    int c = 0;
    for (int w = 0; w < 8; ++w) c += s_valid[w];
    blk_cnt[blockIdx.x] = c;
    __threadfence();
    s_last = (atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  long long c = 0;
#pragma unroll 8
  for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += blockDim.x) c += __ldcg(blk_cnt + i);
  s_sum[threadIdx.x] = c;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) s_sum[threadIdx.x] += s_sum[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const long long nv = s_sum[0];
    *n_valid_out = static_cast<int>(nv);
    // as reduce_final_kernel with g = 1: mean 1 / n_valid (0 without valid rows), sum and none 1
    *scale_out = reduction == 0 ? (nv > 0 ? static_cast<float>(1.0 / static_cast<double>(nv)) : 0.f) : 1.f;
    *ticket = 0;
  }
}

static_assert(kMaxSplit <= 32, "finalize_ref_kernel merges one vocabulary range per lane");

// Fused path, one row chunk, kRefRowsPerBlock rows per block (one
// warp per row, one lane per vocabulary range).
//  - every thread first starts loading its share of the block's X rows;
//  - warp w, row w: lse from the per-range (reference, sum) pairs (butterfly
//    max and sum over the lanes), the row's loss; f_i = 2^(ref_i - lse_i log2 e)
//    and the target entry (p_iy - 1) / f_i of the chunk buffer, so that
//    G_i = s f_i p~_i; f_i = 0 for rows without a gradient; rows where some
//    tile used its own max (largest reference above ref_i) get f_i = 1 and go
//    on the list for the full fix-up;
//  - the block's loss partial, summed over its rows in order;
//  - all threads: xs_i = f_i x_i (bf16), the dW contraction's B operand.
__global__ void __launch_bounds__(kRefRowsPerBlock * 32) finalize_ref_kernel(
    int r0, int rows, int n, int h, int v, int vp, int vsplit, LabelView lv,
    const float* __restrict__ part_m, const float* __restrict__ part_l, const float* __restrict__ tgt,
    const float* __restrict__ mref, float* __restrict__ lse_out,
    float* __restrict__ loss_rows, double* __restrict__ blk_loss, int* __restrict__ blk_valid,
    float* __restrict__ rowscale, const __nv_bfloat16* __restrict__ X, __nv_bfloat16* __restrict__ xs,
    __nv_bfloat16* __restrict__ P, int* __restrict__ fix_list, int* __restrict__ fix_count,
    int* __restrict__ status) {
  griddep_begin();
  __shared__ float s_f[kRefRowsPerBlock];
  __shared__ double s_li[kRefRowsPerBlock];
  __shared__ int s_valid[kRefRowsPerBlock];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int lrow0 = blockIdx.x * kRefRowsPerBlock;
  const int nr = min(kRefRowsPerBlock, rows - lrow0);
  constexpr int kPre = 8;
  const int h8 = h / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(X + static_cast<int64_t>(r0 + lrow0) * h);
  uint4* xo = reinterpret_cast<uint4*>(xs + static_cast<int64_t>(lrow0) * h);
  const int total = nr * h8;
  uint4 xv[kPre];
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int q = threadIdx.x + k * blockDim.x;
    if (q < total) xv[k] = xr[q];
  }
  double li = 0.0;
  int valid = 0;
  float f = 0.f;
  if (warp < nr) {
    const int lrow = lrow0 + warp;
    const int row = r0 + lrow;
    const int k = lv.soft_k;
    const float pm = lane < vsplit ? part_m[static_cast<int64_t>(lane) * n + row] : -INFINITY;
    const float pl = lane < vsplit ? part_l[static_cast<int64_t>(lane) * n + row] : 0.f;
    const int y = k > 0 ? lv.ignore_index : label_at(lv.labels, row, lv.shift, lv.seq_len, lv.ignore_index);
    const float qv = lane < k ? lv.soft_prob[static_cast<int64_t>(row) * k + lane] : 0.f;
    const float z = tgt[row];
    const float ref = mref[row];
    float m = pm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = lane < vsplit ? pl * exp2f(pm - m) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    const float lse2 = m + log2f(l);
    const float lse = lse2 * kLn2;
    float Q = 0.f;
    if (k > 0) {
      // KL(q || p) over the row's targets: sum_t q_t log q_t + Q lse - sum_t q_t z_t, Q = sum_t q_t
      double qd = qv > 0.f ? static_cast<double>(qv) : 0.0;
      double cd = qv > 0.f ? qd * log(qd) : 0.0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        qd += __shfl_xor_sync(0xffffffffu, qd, o);
        cd += __shfl_xor_sync(0xffffffffu, cd, o);
      }
      Q = static_cast<float>(qd);
      if (qd > 0.0) {
        valid = 1;
        li = cd + qd * static_cast<double>(lse) - static_cast<double>(z);
      }
    } else if (y != lv.ignore_index) {
      if (y >= 0 && y < v) {
        valid = 1;
        Q = 1.f;
        li = static_cast<double>(lse) - static_cast<double>(z);
      } else if (lane == 0) {
        atomicCAS(status, 0, kErrLabel);
      }
    }
    // G_ij = s (Q p_ij - q_ij) = s f_i (p~_ij - q_ij / f_i), f_i = Q 2^(ref - lse2)
    if (valid) f = m > ref ? 1.f : Q * exp2f(ref - lse2);
    if (lane == 0) {
      lse_out[row] = lse;
      rowscale[lrow] = f;
      if (loss_rows) loss_rows[row] = static_cast<float>(li);
      if (valid) {
        __nv_bfloat16* prow = P + static_cast<int64_t>(lrow) * vp;
        if (m > ref) {
          const int slot = atomicAdd(fix_count, 1);
          if (in_bounds(slot, rows, status)) fix_list[slot] = lrow;
        } else if (k == 0) {
          // (p_iy - 1) 2^(lse2 - ref), p_iy = 2^(z_iy log2 e - lse2), from the fp32 logit
          prow[y] = __float2bfloat16_rn(exp2f(fmaf(z, kLog2e, -ref)) - exp2f(lse2 - ref));
        } else {
          for (int t = 0; t < k; ++t) {  // one lane, in order: repeated ids accumulate
            const float q = lv.soft_prob[static_cast<int64_t>(row) * k + t];
            const int id = lv.soft_idx[static_cast<int64_t>(row) * k + t];
            if (q > 0.f && id >= 0 && id < v) prow[id] = __float2bfloat16_rn(__bfloat162float(prow[id]) - q / f);
          }
        }
      }
      s_f[warp] = f;
      s_li[warp] = li;
      s_valid[warp] = valid;
    }
  } else if (lane == 0 && warp < kRefRowsPerBlock) {
    s_f[warp] = 0.f;
    s_li[warp] = 0.0;
    s_valid[warp] = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double bl = 0.0;
    int bv = 0;
    for (int w = 0; w < kRefRowsPerBlock; ++w) {
      bl += s_li[w];
      bv += s_valid[w];
    }
    blk_loss[r0 / kRefRowsPerBlock + blockIdx.x] = bl;
    blk_valid[r0 / kRefRowsPerBlock + blockIdx.x] = bv;
  }
  auto scale_store = [&](int q, const uint4& u) {
    const float c = s_f[q / h8];
    const uint32_t in[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[e] = pack_bf16x2(__uint_as_float(in[e] << 16) * c, __uint_as_float(in[e] & 0xFFFF0000u) * c);
    xo[q] = make_uint4(o[0], o[1], o[2], o[3]);
  };
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int q = threadIdx.x + k * blockDim.x;
    if (q < total) scale_store(q, xv[k]);
  }
#pragma unroll 4
  for (int q = threadIdx.x + kPre * blockDim.x; q < total; q += blockDim.x) scale_store(q, xr[q]);
}

// The rows finalize_ref listed (a tile of theirs was stored relative to its
// own max), in place: G / s = p~ 2^(r_tile - lse log2 e) - [j = y].  Work items
// are (listed row, segment of kFixSegment columns), taken round-robin by the
// blocks; an empty list costs one launch.
constexpr int kFixSegment = 8192;
__global__ void __launch_bounds__(256) fixup_list_kernel(const int* __restrict__ fix_list,
                                                         const int* __restrict__ fix_count, int r0, int v, int vp,
                                                         int vtiles, LabelView lv, const float* __restrict__ lse,
                                                         const float* __restrict__ mtile,
                                                         __nv_bfloat16* __restrict__ P) {
  griddep_begin();
  __shared__ int s_idx[kTopkMax];
  __shared__ float s_q[kTopkMax];
  const int nseg = (v + kFixSegment - 1) / kFixSegment;
  const int items = *fix_count * nseg;
  const int k = lv.soft_k;
  for (int e = blockIdx.x; e < items; e += gridDim.x) {  // the same count for the whole block
    const int lrow = fix_list[e / nseg];
    const int seg = e % nseg;
    const int row = r0 + lrow;
    int y = -1;
    float mass = 1.f;
    if (k > 0) {
      // soft targets: G / s = Q p - sum_t q_t [j = id_t]
      __syncthreads();  // the previous item's reads of s_q / s_idx are done
      if (threadIdx.x < k) {
        const float q = lv.soft_prob[static_cast<int64_t>(row) * k + threadIdx.x];
        s_q[threadIdx.x] = q > 0.f ? q : 0.f;
        s_idx[threadIdx.x] = lv.soft_idx[static_cast<int64_t>(row) * k + threadIdx.x];
      }
      __syncthreads();
      mass = 0.f;
      for (int t = 0; t < k; ++t) mass += s_q[t];
    } else {
      y = label_at(lv.labels, row, lv.shift, lv.seq_len, lv.ignore_index);
    }
    const int q0 = seg * (kFixSegment / 8);
    const int q1 = min((v + 7) / 8, q0 + kFixSegment / 8);
    fixup_row(reinterpret_cast<uint4*>(P + static_cast<int64_t>(lrow) * vp),
              mtile + static_cast<int64_t>(lrow) * vtiles, v, lse[row] * kLog2e, 1.f, mass, y, k, s_idx, s_q,
              q0, q1);
  }
}

// Label scan: range check and valid count, for a backward call on its own.
__global__ void __launch_bounds__(kFinalizeThreads) label_scan_kernel(int n, int v, LabelView lv,
                                                                       double* __restrict__ blk_loss,
                                                                       int* __restrict__ blk_valid,
                                                                       int* __restrict__ status) {
  griddep_begin();
  __shared__ int s_valid[kFinalizeThreads];
  const int ignore_index = lv.ignore_index;
  const int row = blockIdx.x * kFinalizeThreads + threadIdx.x;
  int valid = 0;
  if (row < n) {
    const int y = label_at(lv.labels, row, lv.shift, lv.seq_len, ignore_index);
    if (y != ignore_index) {
      if (y >= 0 && y < v)
        valid = 1;
      else
        atomicCAS(status, 0, kErrLabel);
    }
  }
  s_valid[threadIdx.x] = valid;
  __syncthreads();
  for (int w = kFinalizeThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) s_valid[threadIdx.x] += s_valid[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    blk_loss[blockIdx.x] = 0.0;
    blk_valid[blockIdx.x] = s_valid[0];
  }
}

// One block: fixed-order sum of the block partials; loss, valid count and the
// gradient scale s = g / n_valid (mean) or g (sum).
__global__ void __launch_bounds__(kFinalizeThreads) reduce_final_kernel(int nblk, const double* __restrict__ blk_loss,
                                                                         const int* __restrict__ blk_valid,
                                                                         int reduction, const float* grad_loss,
                                                                         float* loss_out, int* n_valid_out,
                                                                         float* scale_out) {
  griddep_begin();
  __shared__ double s_loss[kFinalizeThreads];
  __shared__ long long s_valid[kFinalizeThreads];
  double l = 0.0;
  long long c = 0;
#pragma unroll 8
  for (int i = threadIdx.x; i < nblk; i += kFinalizeThreads) {  // loads hoisted, sums kept in index order
    l += blk_loss[i];
    c += blk_valid[i];
  }
  s_loss[threadIdx.x] = l;
  s_valid[threadIdx.x] = c;
  __syncthreads();
  for (int w = kFinalizeThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      s_loss[threadIdx.x] += s_loss[threadIdx.x + w];
      s_valid[threadIdx.x] += s_valid[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double total = s_loss[0];
    const long long nv = s_valid[0];
    const double g = grad_loss ? static_cast<double>(*grad_loss) : 1.0;
    double loss, scale;
    if (reduction == 0) {  // mean over valid rows; no valid row gives 0 (sum / none: scale g)
      loss = nv > 0 ? total / static_cast<double>(nv) : 0.0;
      scale = nv > 0 ? g / static_cast<double>(nv) : 0.0;
    } else {
      loss = total;
      scale = g;
    }
    if (loss_out) *loss_out = static_cast<float>(loss);
    *n_valid_out = static_cast<int>(nv);
    *scale_out = static_cast<float>(scale);
  }
}

// Top-k pass: merge the per-sub-range candidates of each row into its best k
// (logit, id), high to low, and its log-sum-exp.  One warp per row: lane s
// merges sub-range s's (max, sum) pair; the candidates are spread over the
// lanes (coalesced loads) and the best k taken by k rounds of a warp-wide
// argmax (ties: the lower id first).
__global__ void __launch_bounds__(256) topk_finalize_kernel(int n, int nsub, int k, const float* __restrict__ part_m,
                                                            const float* __restrict__ part_l,
                                                            const float* __restrict__ cand_val,
                                                            const int32_t* __restrict__ cand_idx,
                                                            float* __restrict__ lse_out, float* __restrict__ out_val,
                                                            int32_t* __restrict__ out_idx) {
  griddep_begin();
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= n) return;  // whole warps
  const float pm = lane < nsub ? part_m[static_cast<int64_t>(lane) * n + row] : -INFINITY;
  const float pl = lane < nsub ? part_l[static_cast<int64_t>(lane) * n + row] : 0.f;
  constexpr int kPer = kMaxSplit * kTopkMax / 32;  // candidates per lane at most
  const int total = nsub * kTopkMax;
  float cv[kPer];
  int ci[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int c = lane + 32 * q;
    const bool ok = c < total;
    const int64_t at = (static_cast<int64_t>(c / kTopkMax) * n + row) * kTopkMax + c % kTopkMax;
    cv[q] = ok ? cand_val[at] : -INFINITY;
    ci[q] = ok ? cand_idx[at] : -1;
  }
  float m = pm;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = lane < nsub ? pl * exp2f(pm - m) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  if (lane == 0) lse_out[row] = (m + log2f(l)) * kLn2;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int bi = -1, bq = -1;
#pragma unroll
    for (int q = 0; q < kPer; ++q)
      if (topk_better(cv[q], ci[q], bv, bi)) {
        bv = cv[q];
        bi = ci[q];
        bq = q;
      }
    float wv = bv;
    int wi = bi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, wv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, wi, o);
      if (topk_better(ov, oi, wv, wi)) {
        wv = ov;
        wi = oi;
      }
    }
    if (bq >= 0 && wi >= 0 && bi == wi) {  // ids are unique within a row: one lane holds the winner
#pragma unroll
      for (int q = 0; q < kPer; ++q)
        if (q == bq) {
          cv[q] = -INFINITY;
          ci[q] = -1;
        }
    }
    if (lane == 0) {
      out_val[static_cast<int64_t>(row) * k + r] = wv;
      out_idx[static_cast<int64_t>(row) * k + r] = wi;
    }
  }
}

__global__ void convert_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, int64_t count8) {
  griddep_begin();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(src)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(src)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    o.z = pack_bf16x2(b.x, b.y);
    o.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4*>(dst)[i] = o;
  }
}

// fp32 -> bf16 of `count` values: 8 per thread-iteration through 16-byte
// accesses, then the tail of fewer than 8 one by one.
__global__ void f32_to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, int64_t count) {
  griddep_begin();
  const int64_t count8 = count / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  for (int64_t i = tid; i < count8; i += stride) {
    const float4 a = reinterpret_cast<const float4*>(src)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(src)[2 * i + 1];
    reinterpret_cast<uint4*>(dst)[i] =
        make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  }
  for (int64_t i = 8 * count8 + tid; i < count; i += stride) dst[i] = __float2bfloat16_rn(src[i]);
}

// ----------------------------------------------------------------------------- soft targets, bounded path

// Per row the gradient coefficient s Q_i (Q_i = the row's target mass; 0 for a
// row without targets), s the device scalar of the reduction.
__global__ void soft_rowcoef_kernel(int n, int k, const float* __restrict__ soft_prob, const float* __restrict__ scale,
                                    float* __restrict__ coef) {
  griddep_begin();
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= n) return;
  float Q = 0.f;
  for (int t = 0; t < k; ++t) {
    const float q = soft_prob[static_cast<int64_t>(row) * k + t];
    if (q > 0.f) Q += q;
  }
  coef[row] = *scale * Q;
}

// One vocabulary chunk of bf16 G, [n, pitch] with columns [c0, c0 + cw): the
// targets' term, G_ij -= s q_k at j = id_k, in place.  One thread per row takes
// the row's targets in order, so repeated ids add up.
__global__ void soft_chunk_targets_kernel(int n, int k, const int32_t* __restrict__ soft_idx,
                                          const float* __restrict__ soft_prob, const float* __restrict__ scale,
                                          int c0, int cw, int64_t pitch, __nv_bfloat16* __restrict__ G, int v,
                                          int* __restrict__ status) {
  griddep_begin();
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= n) return;
  const float s = *scale;
  for (int t = 0; t < k; ++t) {
    const float q = soft_prob[static_cast<int64_t>(row) * k + t];
    const int id = soft_idx[static_cast<int64_t>(row) * k + t];
    if (!(q > 0.f) || id < c0 || id >= c0 + cw || id >= v) continue;
    const int64_t at = static_cast<int64_t>(row) * pitch + (id - c0);
    if (!in_bounds(at, static_cast<int64_t>(n) * pitch, status)) continue;
    G[at] = __float2bfloat16_rn(__bfloat162float(G[at]) - s * q);
  }
}

// ----------------------------------------------------------------------------- vocabulary shards
// ("What-Each-Parallelism-Actually-Shards" §7.2: each rank covers one range of the
// vocabulary; ranks without the label still take part in the global max and
// sum-exp; the loss takes the target logit from the rank that holds it; the
// backward forms the local part of the logits gradient.)

// Shard-local labels (see kNotOwned): one thread per row, the global label read
// through the view (shift included), checked against the whole vocabulary.
__global__ void shard_labels_kernel(int n, int64_t v_total, int64_t v0, int64_t vs, LabelView lv,
                                    int32_t* __restrict__ lab_local, int* __restrict__ status) {
  griddep_begin();
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= n) return;
  const int y = label_at(lv.labels, row, lv.shift, lv.seq_len, lv.ignore_index);
  int out = -1;
  if (y != lv.ignore_index) {
    if (y >= 0 && y < v_total)
      out = (y >= v0 && y - v0 < vs) ? static_cast<int>(y - v0) : kNotOwned;
    else
      atomicCAS(status, 0, kErrLabel);
  }
  lab_local[row] = out;
}

__global__ void __launch_bounds__(kFinalizeThreads) shard_finalize_kernel(
    int n, int vsplit, const float* __restrict__ part_m, const float* __restrict__ part_l,
    const float* __restrict__ tgt, const int32_t* __restrict__ lab_local, float* __restrict__ lse_part,
    float* __restrict__ tgt_part) {
  griddep_begin();
  const int row = blockIdx.x * kFinalizeThreads + threadIdx.x;
  if (row >= n) return;
  float m;
  lse_part[row] = merge_ranges(part_m, part_l, vsplit, n, row, &m) * kLn2;
  const int y = lab_local[row];
  tgt_part[row] = (y >= 0 && y != kNotOwned) ? tgt[row] : 0.f;
}

// Combine the shards' per-row (lse, target logit) pairs, parts in index order
// (every rank that runs it on the same gathered parts gets the same bits), then
// the loss rows and the block partials of the fixed-order loss reduction.
__global__ void __launch_bounds__(kFinalizeThreads) shard_combine_kernel(
    int n, int parts, int64_t v_total, LabelView lv, const float* __restrict__ lse_parts,
    const float* __restrict__ tgt_parts, float* __restrict__ lse_out, float* __restrict__ loss_rows,
    double* __restrict__ blk_loss, int* __restrict__ blk_valid, int* __restrict__ status) {
  griddep_begin();
  __shared__ double s_loss[kFinalizeThreads];
  __shared__ int s_valid[kFinalizeThreads];
  const int row = blockIdx.x * kFinalizeThreads + threadIdx.x;
  double li = 0.0;
  int valid = 0;
  if (row < n) {
    float m = -INFINITY;
    for (int r = 0; r < parts; ++r) m = fmaxf(m, lse_parts[static_cast<int64_t>(r) * n + row]);
    float l = 0.f, z = 0.f;
    for (int r = 0; r < parts; ++r) {
      l += exp2f((lse_parts[static_cast<int64_t>(r) * n + row] - m) * kLog2e);
      z += tgt_parts[static_cast<int64_t>(r) * n + row];
    }
    const float lse = m + log2f(l) * kLn2;
    lse_out[row] = lse;
    const int y = label_at(lv.labels, row, lv.shift, lv.seq_len, lv.ignore_index);
    if (y != lv.ignore_index) {
      if (y >= 0 && y < v_total) {
        valid = 1;
        li = static_cast<double>(lse) - static_cast<double>(z);
      } else {
        atomicCAS(status, 0, kErrLabel);
      }
    }
    if (loss_rows) loss_rows[row] = static_cast<float>(li);
  }
  s_loss[threadIdx.x] = li;
  s_valid[threadIdx.x] = valid;
  __syncthreads();
  for (int w = kFinalizeThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      s_loss[threadIdx.x] += s_loss[threadIdx.x + w];
      s_valid[threadIdx.x] += s_valid[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    blk_loss[blockIdx.x] = s_loss[0];
    blk_valid[blockIdx.x] = s_valid[0];
  }
}

// x *= g for bf16 data (8 elements per thread-iteration), g a device scalar.
__global__ void scale_bf16_kernel(__nv_bfloat16* __restrict__ x, int64_t count8, const float* __restrict__ g) {
  griddep_begin();
  const float s = *g;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < count8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    uint4 u = reinterpret_cast<uint4*>(x)[i];
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = pack_bf16x2(__uint_as_float(w[e] << 16) * s, __uint_as_float(w[e] & 0xFFFF0000u) * s);
    reinterpret_cast<uint4*>(x)[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Waits on a barrier that nothing completes; the bounded wait gives up and the
// timeout lands in the status word.
__global__ void timeout_selftest_kernel(int* status, uint64_t limit_ns) {
  griddep_begin();
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&bar, 0, limit_ns, &abort_flag)) atomicCAS(status, 0, kErrTimeout);
  }
}

__global__ void bounds_selftest_kernel(int* status) {
  griddep_begin();
  if (threadIdx.x == 0) (void)in_bounds(1, 1, status);
}

}  // namespace

int tc_smem_bytes() { return Cfg<kModeForward>::kSmemBytes; }
int tc_topk_subranges() { return Cfg<kModeTopk>::kEpiWarps / 4; }

// Every launch carries the programmatic-stream-serialization attribute (see
// griddep_begin): a kernel may be scheduled while its predecessor drains.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int MODE>
static cudaError_t launch_mode(const TcMaps& maps, const TcParams& p, int grid, cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<MODE>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return launch_k(tc_kernel<MODE>, dim3(grid), dim3(Cfg<MODE>::kThreads), Cfg<MODE>::kSmemBytes, stream, maps, p);
}

cudaError_t launch_tc(int mode, const TcMaps& maps, const TcParams& p, int grid, cudaStream_t stream) {
  switch (mode) {
    case kModeForward: return launch_mode<kModeForward>(maps, p, grid, stream);
    case kModeGrad: return launch_mode<kModeGrad>(maps, p, grid, stream);
    case kModeBwd: return launch_mode<kModeBwd>(maps, p, grid, stream);
    case kModeFwdStore: return launch_mode<kModeFwdStore>(maps, p, grid, stream);
    case kModeTopk: return launch_mode<kModeTopk>(maps, p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd_finalize_rows(int r0, int rows, int n, int v, int vsplit, LabelView lv, const float* part_m,
                                     const float* part_l, const float* tgt, float* lse, float* loss_rows,
                                     double* blk_loss, int* blk_valid, int* status, cudaStream_t stream) {
  const int blocks = (rows + kFinalizeThreads - 1) / kFinalizeThreads;
  return launch_k(fwd_finalize_kernel, dim3(blocks), dim3(kFinalizeThreads), 0, stream,
                  r0, rows, n, v, vsplit, lv, part_m, part_l, tgt, lse, loss_rows, blk_loss, blk_valid, status);
}

cudaError_t launch_label_prep(int n, int h, int v, int reduction, LabelView lv, const void* X, const void* W,
                              float* mref, float* tgt, int* blk_cnt, int* ticket, int* n_valid, float* scale,
                              int* status, cudaStream_t stream) {
  const int blocks = (n + 7) / 8;  // 8 rows (warps) per block
  return launch_k(label_prep_kernel, dim3(blocks), dim3(256), 0, stream, n, h, v, reduction, lv,
                  static_cast<const __nv_bfloat16*>(X), static_cast<const __nv_bfloat16*>(W), mref, tgt, blk_cnt,
                  ticket, n_valid, scale, status);
}

cudaError_t launch_finalize_ref(int r0, int rows, int n, int h, int v, int vp, int vsplit, LabelView lv,
                                const float* part_m, const float* part_l, const float* tgt, const float* mref,
                                float* lse, float* loss_rows, double* blk_loss, int* blk_valid,
                                float* rowscale, const void* X, void* xs, void* P, int* fix_list, int* fix_count,
                                int* status, cudaStream_t stream) {
  const int blocks = (rows + kRefRowsPerBlock - 1) / kRefRowsPerBlock;
  return launch_k(finalize_ref_kernel, dim3(blocks), dim3(kRefRowsPerBlock * 32), 0, stream, r0, rows, n, h, v, vp,
                  vsplit, lv,
                  part_m, part_l, tgt, mref, lse, loss_rows, blk_loss, blk_valid, rowscale,
                  static_cast<const __nv_bfloat16*>(X), static_cast<__nv_bfloat16*>(xs),
                  static_cast<__nv_bfloat16*>(P), fix_list, fix_count, status);
}

cudaError_t launch_fixup_list(const int* fix_list, const int* fix_count, int r0, int v, int vp, int vtiles,
                              LabelView lv, const float* lse, const float* mtile, void* P, int grid,
                              cudaStream_t stream) {
  return launch_k(fixup_list_kernel, dim3(std::max(1, grid)), dim3(256), 0, stream, fix_list, fix_count, r0, v, vp,
                  vtiles, lv, lse, mtile, static_cast<__nv_bfloat16*>(P));
}

cudaError_t launch_label_scan_view(int n, int v, LabelView lv, double* blk_loss, int* blk_valid, int* status,
                                   cudaStream_t stream) {
  const int blocks = (n + kFinalizeThreads - 1) / kFinalizeThreads;
  return launch_k(label_scan_kernel, dim3(blocks), dim3(kFinalizeThreads), 0, stream,
                  n, v, lv, blk_loss, blk_valid, status);
}

cudaError_t launch_reduce_final(int nblk, const double* blk_loss, const int* blk_valid, int reduction,
                                const float* grad_loss, float* loss_out, int* n_valid_out, float* scale_out,
                                cudaStream_t stream) {
  return launch_k(reduce_final_kernel, dim3(1), dim3(kFinalizeThreads), 0, stream,
                  nblk, blk_loss, blk_valid, reduction, grad_loss, loss_out, n_valid_out, scale_out);
}

cudaError_t launch_convert_bf16(const float* src, void* dst, int64_t count, cudaStream_t stream) {
  const int64_t count8 = count / 8;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (count8 + 255) / 256;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  if (blocks < 1) blocks = 1;
  return launch_k(convert_bf16_kernel, dim3(static_cast<int>(blocks)), dim3(256), 0, stream, src,
                  static_cast<__nv_bfloat16*>(dst), count8);
}

cudaError_t launch_f32_to_bf16(const float* src, void* dst, int64_t count, cudaStream_t stream) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (count / 8 + 255) / 256;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  if (blocks < 1) blocks = 1;
  return launch_k(f32_to_bf16_kernel, dim3(static_cast<int>(blocks)), dim3(256), 0, stream, src,
                  static_cast<__nv_bfloat16*>(dst), count);
}

cudaError_t launch_soft_rowcoef(int n, int k, const float* soft_prob, const float* scale, float* coef,
                               cudaStream_t stream) {
  return launch_k(soft_rowcoef_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, n, k, soft_prob, scale, coef);
}

cudaError_t launch_soft_chunk_targets(int n, int k, const int32_t* soft_idx, const float* soft_prob,
                                      const float* scale, int c0, int cw, int64_t pitch, void* G, int v, int* status,
                                      cudaStream_t stream) {
  return launch_k(soft_chunk_targets_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, n, k, soft_idx, soft_prob,
                  scale, c0, cw, pitch, static_cast<__nv_bfloat16*>(G), v, status);
}

cudaError_t launch_shard_labels(int n, int64_t v_total, int64_t v0, int64_t vs, LabelView lv, int32_t* lab_local,
                                int* status, cudaStream_t stream) {
  return launch_k(shard_labels_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, n, v_total, v0, vs, lv,
                  lab_local, status);
}

cudaError_t launch_shard_finalize(int n, int vsplit, const float* part_m, const float* part_l, const float* tgt,
                                  const int32_t* lab_local, float* lse_part, float* tgt_part, cudaStream_t stream) {
  return launch_k(shard_finalize_kernel, dim3((n + kFinalizeThreads - 1) / kFinalizeThreads), dim3(kFinalizeThreads),
                  0, stream, n, vsplit, part_m, part_l, tgt, lab_local, lse_part, tgt_part);
}

cudaError_t launch_shard_combine(int n, int parts, int64_t v_total, LabelView lv, const float* lse_parts,
                                 const float* tgt_parts, float* lse, float* loss_rows, double* blk_loss,
                                 int* blk_valid, int* status, cudaStream_t stream) {
  return launch_k(shard_combine_kernel, dim3((n + kFinalizeThreads - 1) / kFinalizeThreads), dim3(kFinalizeThreads),
                  0, stream, n, parts, v_total, lv, lse_parts, tgt_parts, lse, loss_rows, blk_loss, blk_valid, status);
}

cudaError_t launch_topk_finalize(int n, int nsub, int k, const float* part_m, const float* part_l,
                                 const float* cand_val, const int32_t* cand_idx, float* lse, float* out_val,
                                 int32_t* out_idx, cudaStream_t stream) {
  return launch_k(topk_finalize_kernel, dim3((n + 7) / 8), dim3(256), 0, stream,
                  n, nsub, k, part_m, part_l, cand_val, cand_idx, lse, out_val, out_idx);
}

cudaError_t launch_scale_bf16(void* x, int64_t count, const float* g, cudaStream_t stream) {
  const int64_t count8 = count / 8;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (count8 + 255) / 256;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  if (blocks < 1) blocks = 1;
  return launch_k(scale_bf16_kernel, dim3(static_cast<int>(blocks)), dim3(256), 0, stream,
                  static_cast<__nv_bfloat16*>(x), count8, g);
}

cudaError_t launch_bounds_selftest(int* status, cudaStream_t stream) {
  return launch_k(bounds_selftest_kernel, dim3(1), dim3(32), 0, stream, status);
}

cudaError_t launch_timeout_selftest(int* status, uint64_t limit_ns, cudaStream_t stream) {
  return launch_k(timeout_selftest_kernel, dim3(1), dim3(32), 0, stream,
                  status, limit_ns);
}

}  // namespace flce
