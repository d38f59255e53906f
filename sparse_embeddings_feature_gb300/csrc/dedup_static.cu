// ctr_dedup_static: ctr_dedup for callers that cannot allocate device memory.
//
// Some callers of this library may not call cudaMalloc (or ask any allocator)
// on the path that runs the dedup: a plugin inside another runtime that owns
// every device allocation, a serving process whose memory budget is fixed at
// start-up, or a latency-critical loop where an allocation could stall the
// device.  For them this entry point runs the regular ctr_dedup with its
// scratch space taken from a fixed array in the library's own device memory
// instead of a caller workspace.  The caller still passes all inputs and
// outputs.
//
// Limits and sharing:
//   * The array holds the scratch of a call of up to kStaticMaxIds (2^20) IDs
//     whatever the tables' total row count: 48 MB, held on every GPU that
//     loads the library until the process exits.  The dedup's scratch depends
//     on the IDs and the row count; it peaks where the presence-bitmap path
//     meets its largest bitmap (total rows = 64 x IDs: 46 MB at 2^20 IDs), and
//     the sorted-key path needs 22 MB.  Larger calls return
//     CTR_ERR_UNSUPPORTED and launch nothing.
//   * Every call uses the same array, and the array keeps the previous call's
//     contents.  The error word at its head is cleared at the start of each
//     call; the sort's scratch is fully rewritten before it is read.  Two calls
//     that overlap on the GPU (different streams, or different host threads
//     without ordering) race on the array and must not be issued.
//   * The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make that
//     first call before any stream capture begins.  The cached address belongs
//     to the device's current context: do not call this entry point again on a
//     device after cudaDeviceReset in the same process.
#include <mutex>

#include "common.cuh"

namespace ctr {
namespace {

constexpr int64_t kStaticMaxIds = 1 << 20;
constexpr size_t kStaticScratchBytes = (size_t)48 << 20;

static __device__ __align__(256) unsigned char g_dedup_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once).
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CTR_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dedup_scratch) != cudaSuccess || !p) return CTR_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return CTR_OK;
}

}  // namespace
}  // namespace ctr

using namespace ctr;

extern "C" int ctr_dedup_static(const int64_t* ids, const int64_t* offsets, int32_t num_fields, int32_t batch,
                                const int32_t* bag_to_table, const int64_t* row_base, int32_t num_tables,
                                int64_t n_ids, int64_t* unique_rows, int64_t* n_unique, int32_t* inverse,
                                int32_t* sorted_pos, int32_t* sorted_bag, int32_t* run_offsets,
                                int64_t* unique_offsets, int32_t* device_status, ctr_stream_t stream) {
  if (n_ids < 0 || !row_base || num_tables <= 0) return CTR_ERR_INVALID_ARG;
  if (n_ids > kStaticMaxIds) return CTR_ERR_UNSUPPORTED;
  const size_t need = ctr_dedup_workspace_size(n_ids, num_fields, batch, row_base[num_tables]);
  if (need > kStaticScratchBytes) return CTR_ERR_UNSUPPORTED;
  void* ws = nullptr;
  if (int st = scratch_for_current_device(&ws)) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(ws, 0, kWsHeader, s) != cudaSuccess) return CTR_ERR_CUDA;
  const int st = ctr_dedup(ids, offsets, num_fields, batch, bag_to_table, row_base, num_tables, n_ids, unique_rows,
                           n_unique, inverse, sorted_pos, sorted_bag, run_offsets, unique_offsets, ws,
                           kStaticScratchBytes, stream);
  if (st) return st;
  if (device_status && cudaMemcpyAsync(device_status, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return CTR_ERR_CUDA;
  return CTR_OK;
}
