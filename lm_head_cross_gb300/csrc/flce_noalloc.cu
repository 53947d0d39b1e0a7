// flce_forward_noalloc: the forward pass for callers that cannot allocate
// device memory — for example code running as a plugin or custom operator
// inside another runtime that owns every device allocation and hands it only
// its input and output buffers, or latency-critical loops where a cudaMalloc
// or cudaFree would synchronise the whole device.  Instead of a caller
// workspace, the scratch this pass needs lives in one fixed array in the
// library's own device memory, declared below.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/flce.h"
#include "flce_internal.h"

namespace flce {
namespace {

// Largest problem this entry point accepts (rows); any H and V the other calls accept.
constexpr int64_t kNoAllocMaxRows = 32768;
constexpr int kNoAllocSplit = 16;            // vocabulary ranges per row tile
constexpr int kMaxDevices = 64;

constexpr size_t round256(size_t x) { return (x + 255) / 256 * 256; }
constexpr size_t kMaxBlocks = (kNoAllocMaxRows + kFinalizeThreads - 1) / kFinalizeThreads;
// Scratch layout (byte offsets into the static array).
constexpr size_t kOffStatus = 0;             // int status, int n_valid, float scale, int unit counter
constexpr size_t kOffBlkLoss = 256;
constexpr size_t kOffBlkValid = kOffBlkLoss + round256(8 * kMaxBlocks);
constexpr size_t kOffPartM = kOffBlkValid + round256(4 * kMaxBlocks);
constexpr size_t kOffPartL = kOffPartM + round256(4 * kNoAllocSplit * kNoAllocMaxRows);
constexpr size_t kOffTgt = kOffPartL + round256(4 * kNoAllocSplit * kNoAllocMaxRows);
constexpr size_t kScratchBytes = kOffTgt + round256(4 * kNoAllocMaxRows);  // about 4.3 MiB

// The scratch itself.  In host code `g_scratch` only names a host-side stand-in
// for the symbol; its device address comes from cudaGetSymbolAddress below.
// Every device that loads this library keeps this array until the process ends.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device
// and kept for the life of the process.  A device reset (cudaDeviceReset, or a
// reset of the primary context) reloads the module elsewhere, so this entry
// point must not be called on a device after it has been reset.
flce_status_t scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLCE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FLCE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || !ptr) return FLCE_ERR_CUDA;
    g_scratch_dev[dev] = ptr;
  }
  *out = g_scratch_dev[dev];
  return FLCE_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// After the loss is reduced: if a label was out of range (or a wait timed out),
// every loss value — the scalar, or each of the n per-row losses — is set to
// NaN, so the error is visible without a workspace to read.
__global__ void poison_loss_on_error(const int* status, float* loss, int count) {
  if (*status == 0) return;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < count; i += gridDim.x * blockDim.x)
    loss[i] = __int_as_float(0x7fc00000);
}

bool aligned_to(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace
}  // namespace flce

using namespace flce;

extern "C" flce_status_t flce_forward_noalloc(const flce_problem_t* p, const void* X, const void* W,
                                              const int32_t* labels, float* loss, float* lse, flce_stream_t stream) {
  if (!p || !X || !W || !labels || !loss || !lse) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->n < 1 || p->h < 1 || p->v < 1) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->reduction != FLCE_REDUCTION_MEAN && p->reduction != FLCE_REDUCTION_SUM &&
      p->reduction != FLCE_REDUCTION_NONE)
    return FLCE_ERR_INVALID_ARGUMENT;
  if (p->shift != 0 && p->shift != 1) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->shift && (p->seq_len < 1 || p->n % p->seq_len != 0)) return FLCE_ERR_INVALID_ARGUMENT;
  if (p->h < 8 || p->h % 8 != 0 || p->h > (int64_t{1} << 20) || p->v > (int64_t{1} << 30))
    return FLCE_ERR_UNSUPPORTED_SHAPE;
  if (p->n > kNoAllocMaxRows) return FLCE_ERR_EXCEEDS_STATIC_SCRATCH;
  if (!aligned_to(X, 16) || !aligned_to(W, 16) || !aligned_to(labels, 4) || !aligned_to(loss, 4) ||
      !aligned_to(lse, 4))
    return FLCE_ERR_MISALIGNED;

  int dev = 0, major = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLCE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess || major != 10)
    return FLCE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FLCE_ERR_CUDA;

  void* base = nullptr;
  flce_status_t st = scratch_address(&base);
  if (st != FLCE_OK) return st;
  unsigned char* s = static_cast<unsigned char*>(base);
  int* status = reinterpret_cast<int*>(s + kOffStatus);
  int* n_valid = status + 1;
  float* scale = reinterpret_cast<float*>(s + kOffStatus + 8);
  double* blk_loss = reinterpret_cast<double*>(s + kOffBlkLoss);
  int* blk_valid = reinterpret_cast<int*>(s + kOffBlkValid);
  float* part_m = reinterpret_cast<float*>(s + kOffPartM);
  float* part_l = reinterpret_cast<float*>(s + kOffPartL);
  float* tgt = reinterpret_cast<float*>(s + kOffTgt);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

  TcMaps maps;
  if (!map_2d(&maps.a, X, p->h, p->n, kBK, kBM)) return FLCE_ERR_CUDA;
  if (!map_2d(&maps.b, W, p->h, p->v, kBK, kBoxB)) return FLCE_ERR_CUDA;
  maps.out = maps.a2 = maps.b2 = maps.out2 = maps.a;

  TcParams tp{};
  tp.n = static_cast<int>(p->n);
  tp.h = static_cast<int>(p->h);
  tp.v = static_cast<int>(p->v);
  tp.ignore_index = p->ignore_index;
  tp.timeout_ns = timeout_ns();
  tp.status = status;
  tp.row_tiles = static_cast<int>((p->n + kPairRows - 1) / kPairRows);
  tp.vocab_tiles = static_cast<int>((p->v + kBN - 1) / kBN);
  tp.vsplit = std::min(kNoAllocSplit, tp.vocab_tiles);
  tp.units_group = units_group_rows(tp.row_tiles, p->h);
  tp.part_m = part_m;
  tp.part_l = part_l;
  tp.tgt = tgt;
  tp.tile_counter = reinterpret_cast<int*>(s + kOffStatus + 12);
  tp.part_count = static_cast<int64_t>(kNoAllocSplit) * kNoAllocMaxRows;
  tp.labels = labels;
  tp.shift = p->shift;
  tp.seq_len = p->shift ? p->seq_len : 1;
  const long long units = static_cast<long long>(tp.row_tiles) * tp.vsplit;
  const int grid = pair_grid(sms, units);

  // Only the status word and the forward launch's unit counter must start at
  // zero; every other region the kernels read is written earlier in the same call.
  if (cudaMemsetAsync(status, 0, 16, cs) != cudaSuccess) return FLCE_ERR_CUDA;
  if (launch_tc(kModeForward, maps, tp, grid, cs) != cudaSuccess) return FLCE_ERR_CUDA;
  const bool per_row = p->reduction == FLCE_REDUCTION_NONE;
  const LabelView lv{labels, p->ignore_index, tp.shift, tp.seq_len};
  if (launch_fwd_finalize_rows(0, tp.n, tp.n, tp.v, tp.vsplit, lv, part_m, part_l, tgt, lse, per_row ? loss : nullptr,
                               blk_loss, blk_valid, status, cs) != cudaSuccess)
    return FLCE_ERR_CUDA;
  const int nblk = static_cast<int>((p->n + kFinalizeThreads - 1) / kFinalizeThreads);
  if (launch_reduce_final(nblk, blk_loss, blk_valid, p->reduction, nullptr, per_row ? nullptr : loss, n_valid, scale,
                          cs) != cudaSuccess)
    return FLCE_ERR_CUDA;
  const int nloss = per_row ? tp.n : 1;
  poison_loss_on_error<<<std::min(64, (nloss + 255) / 256), 256, 0, cs>>>(status, loss, nloss);
  return cudaGetLastError() == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA;
}
