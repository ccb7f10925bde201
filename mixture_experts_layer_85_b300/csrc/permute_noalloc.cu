// moe_permute_noalloc: the dispatch step for callers that cannot allocate.
//
// moe_permute needs a caller-provided workspace for its per-chunk tables.  Some
// callers have no way to obtain one: a plug-in whose device memory belongs to
// the host framework's fixed arena, a process held to a hard memory budget, or
// a latency-critical loop that must never call cudaMalloc (it can block on the
// whole device and can fail when memory is fragmented).  This entry point runs
// the same permutation kernels with their scratch in a fixed-size array that
// lives in the library's own device image, so nothing is allocated per call.
#include "internal.h"

namespace moe {
namespace {

// Capacity: permute_chunks(T) * E entries for each of the two per-chunk tables
// (e.g. T <= 16384 tokens with E = 256 experts), plus a small header whose
// first int is the device status word.  About 256 KB on every device that
// loads the library, held until the process exits.
constexpr int kTableInts = 32768;
constexpr int kHeaderInts = 64;
static __device__ __align__(256) int32_t g_permute_scratch[kHeaderInts + 2 * kTableInts];

// Device address of g_permute_scratch on the current device, looked up once
// per device (in host code the array's name is only a host-side stand-in).
// After a context reset (cudaDeviceReset) the module is loaded again at
// another address, which this cache does not see: a process that resets a
// device must not call moe_permute_noalloc on it afterwards.
cudaError_t scratch_on_current_device(int32_t** out) {
  static PerDevice<int32_t*> addr;
  return addr.get(out, [](int32_t** p) {
    void* a = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&a, g_permute_scratch);
    *p = static_cast<int32_t*>(a);
    return e;
  });
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" MOE_API moe_status moe_permute_noalloc(const moe_config* cfg, const void* x, const int32_t* idx,
                                                  int32_t* counts, int32_t* offsets, int32_t* row2tok,
                                                  int32_t* tok2row, void* x_perm, int32_t* device_status,
                                                  void* stream) {
  size_t unused = 0;
  moe_status st = moe_workspace_size(cfg, &unused);   // the same configuration checks as every call
  if (st != MOE_OK) return st;
  const moe_config& c = *cfg;
  if (!x || !idx || !counts || !offsets || !row2tok || !tok2row || !x_perm) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(idx) || !aligned16(counts) || !aligned16(offsets) || !aligned16(row2tok) ||
      !aligned16(tok2row) || !aligned16(x_perm) || (device_status && !aligned16(device_status)))
    return MOE_ERR_INVALID_ARG;
  if ((long long)permute_chunks(c.T) * c.E > kTableInts) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c.T == 0) {
    // no tokens: every expert is empty, and nothing can go wrong on the device
    if (cudaMemsetAsync(offsets, 0, size_t(c.E + 1) * 4, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (device_status != nullptr && cudaMemsetAsync(device_status, 0, sizeof(int32_t), s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return cudaMemsetAsync(counts, 0, size_t(c.E) * 4, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  int32_t* base = nullptr;
  if (scratch_on_current_device(&base) != cudaSuccess) return MOE_ERR_CUDA;
  int* status = base;
  int32_t* chunk_counts = base + kHeaderInts;
  int32_t* chunk_base = chunk_counts + kTableInts;
  // The array keeps the previous call's contents.  The status word must start
  // at zero; both tables are fully written by the kernels before they are read.
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  int n = 0;
  cudaError_t e = launch_permute(c, x, idx, counts, offsets, row2tok, tok2row, x_perm, chunk_counts, chunk_base,
                                 status, s, &n);
  count_launches(n);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (device_status != nullptr &&
      cudaMemcpyAsync(device_status, status, sizeof(int), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
