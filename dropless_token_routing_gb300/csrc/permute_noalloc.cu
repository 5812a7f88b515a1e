// moe_permute_noalloc: the expert permutation for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: code running where cudaMalloc is not
// allowed or not wanted (an allocator-free runtime, a memory pool that is already carved up
// and must not grow, a process restricted to the buffers it was given). This entry point runs
// the same kernels as moe_permute, with their scratch (per-chunk expert histograms, their
// scans and the copies' local ranks) in one file-scope device array instead of a workspace.
//
// Limits: T*k <= kNoAllocMaxCopies and E * ceil(T / 64) <= kNoAllocMaxChunkCells; larger
// problems are rejected with MOE_ERR_WORKSPACE_TOO_SMALL before anything is launched.
// The array lives in every GPU that loads the library until the process exits (about 1.5 MB).
// The first call on a device looks up the array's device address (once per device, with that
// device current); make that first call before any stream capture.
// All calls share the one array: calls that overlap on the GPU (different streams without
// ordering between them) race on it. Each call overwrites every scratch word it reads, so
// nothing has to start at zero; the array keeps the last call's contents.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int64_t kNoAllocMaxCopies = int64_t(1) << 18;      // T*k token copies
constexpr int64_t kNoAllocMaxChunkCells = int64_t(1) << 16;  // E * ceil(T / 64)
constexpr int64_t kNoAllocScratchInts = 2 * kNoAllocMaxChunkCells + kNoAllocMaxCopies;

// [chunk histograms | chunk bases | local ranks], int32
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchInts];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_permute_noalloc(const void* x, const int32_t* topk_idx, const float* topk_w,
                                   const moe_dims* dims, void* x_perm, int32_t* dest,
                                   int32_t* row_src, int32_t* offsets, float* w_perm, int* dev_err,
                                   moe_stream_t stream) {
  if (dims == nullptr) return MOE_ERR_NULL_POINTER;
  if (dims->dtype != MOE_F32 && dims->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED_DTYPE;
  if (dims->k < 1 || dims->k > kMaxK || (dims->E >= 1 && dims->k > dims->E)) return MOE_ERR_BAD_TOPK;
  // the same row-width rule as moe_permute: d a multiple of 64 (bf16) or 8 (fp32)
  const int unit = dims->dtype == MOE_BF16 ? 64 : 8;
  if (dims->T < 0 || dims->E < 1 || dims->E > kMaxE || dims->d < 1 || dims->d % unit != 0)
    return MOE_ERR_BAD_DIMS;
  if (dims->capacity != 0) return MOE_ERR_BAD_DIMS;   // the dropless permutation only
  // bound T before any product of it is formed (k >= 1, so T <= T*k)
  if (dims->T > kNoAllocMaxCopies) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int64_t copies = dims->T * dims->k;
  const int64_t n_chunks = (dims->T + kChunk - 1) / kChunk;
  if (copies > kNoAllocMaxCopies || dims->E * n_chunks > kNoAllocMaxChunkCells)
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  const bool t0 = dims->T == 0;
  const void* ptrs[] = {x, topk_idx, x_perm, dest, row_src};
  for (const void* q : ptrs) {
    if (q == nullptr && !t0) return MOE_ERR_NULL_POINTER;
    if (q != nullptr && !aligned16(q)) return MOE_ERR_MISALIGNED;
  }
  if (offsets == nullptr) return MOE_ERR_NULL_POINTER;
  if (!aligned16(offsets) || (w_perm != nullptr && !aligned16(w_perm)) ||
      (topk_w != nullptr && !aligned16(topk_w)))
    return MOE_ERR_MISALIGNED;
  if (w_perm != nullptr && topk_w == nullptr && !t0) return MOE_ERR_NULL_POINTER;
  // the kernels update the error word with 32-bit atomics
  if (dev_err != nullptr && (reinterpret_cast<uintptr_t>(dev_err) & 3u) != 0) return MOE_ERR_MISALIGNED;
  const cudaStream_t st = (cudaStream_t)stream;
  if (t0)
    return cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (dims->E + 1), st) == cudaSuccess ? MOE_OK
                                                                                            : MOE_ERR_CUDA;
  void* scratch = nullptr;
  const int s = scratch_address(&scratch);
  if (s != MOE_OK) return s;
  // the permutation kernels address their scratch through a workspace layout: point the
  // three regions into the static array
  WsLayout L;
  memset(&L, 0, sizeof(L));
  L.n_chunks = n_chunks;
  L.chunk_hist = 0;
  L.chunk_base = sizeof(int32_t) * kNoAllocMaxChunkCells;
  L.local_rank = 2 * sizeof(int32_t) * kNoAllocMaxChunkCells;
  if (launch_permute(x, topk_idx, topk_w, *dims, x_perm, dest, row_src, offsets, w_perm, L,
                     static_cast<uint8_t*>(scratch), dev_err, st) != cudaSuccess)
    return MOE_ERR_LAUNCH;
  return MOE_OK;
}
