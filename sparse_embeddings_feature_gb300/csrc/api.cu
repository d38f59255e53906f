// Library-wide entry points: status handling, version, device info and the
// counter-based table generator used to build synthetic inputs.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace ctr {

int num_sms() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    cached[dev] = v;
  }
  return cached[dev];
}

namespace {
std::mutex g_timing_mu;
std::atomic<uint64_t> g_launches{0};
cudaEvent_t g_timing[CTR_KERNEL_COUNT][2] = {};
}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void timing_mark(int kernel, bool before, cudaStream_t s) {
  if (kernel <= 0 || kernel >= CTR_KERNEL_COUNT) return;
  cudaEvent_t e;
  {
    std::lock_guard<std::mutex> lock(g_timing_mu);
    e = g_timing[kernel][before ? 0 : 1];
  }
  if (!e) return;
  // inside a stream capture a plain record is only a dependency edge; an
  // external record becomes a node that records the event at every replay
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

namespace {


__global__ void fill_uniform_f32(float* __restrict__ t, int64_t count, uint64_t idx0, uint64_t seed, float scale) {
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < count; e += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t h = splitmix64(seed ^ (idx0 + (uint64_t)e));
    const int32_t c = (int32_t)(h >> 40) - (1 << 23);
    t[e] = __fmul_rn((float)c, scale);
  }
}

__global__ void fill_normal4_bf16(__nv_bfloat16* __restrict__ t, int64_t count, uint64_t idx0, uint64_t seed,
                                  float scale) {
  const uint64_t m22 = (1ull << 22) - 1;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < count; e += (int64_t)gridDim.x * blockDim.x) {
    const uint64_t idx = idx0 + (uint64_t)e;
    const uint64_t h1 = splitmix64(seed ^ (2 * idx));
    const uint64_t h2 = splitmix64(seed ^ (2 * idx + 1));
    const uint64_t s = (h1 >> 42) + ((h1 >> 20) & m22) + (h2 >> 42) + ((h2 >> 20) & m22);
    const int32_t c = (int32_t)s - ((1 << 23) - 2);
    t[e] = __float2bfloat16_rn(__fmul_rn((float)c, scale));
  }
}

__global__ void clear_word(int* w) { *w = 0; }

}  // namespace
}  // namespace ctr

using namespace ctr;

extern "C" const char* ctr_status_string(int status) {
  switch (status) {
    case CTR_OK: return "CTR_OK";
    case CTR_ERR_INVALID_ARG: return "CTR_ERR_INVALID_ARG";
    case CTR_ERR_UNSUPPORTED: return "CTR_ERR_UNSUPPORTED";
    case CTR_ERR_WORKSPACE: return "CTR_ERR_WORKSPACE";
    case CTR_ERR_INDEX_OUT_OF_RANGE: return "CTR_ERR_INDEX_OUT_OF_RANGE";
    case CTR_ERR_CUDA: return "CTR_ERR_CUDA";
    case CTR_ERR_TIMEOUT: return "CTR_ERR_TIMEOUT";
    case CTR_ERR_NOT_IMPLEMENTED: return "CTR_ERR_NOT_IMPLEMENTED";
    case CTR_ERR_BAD_OFFSETS: return "CTR_ERR_BAD_OFFSETS";
    default: return "CTR_ERR_UNKNOWN";
  }
}

extern "C" int ctr_version(void) { return 100; }

extern "C" uint64_t ctr_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" int ctr_set_timing_events(int kernel, void* before_event, void* after_event) {
  if (kernel <= 0 || kernel >= CTR_KERNEL_COUNT) return CTR_ERR_INVALID_ARG;
  if ((before_event == nullptr) != (after_event == nullptr)) return CTR_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_timing_mu);
  g_timing[kernel][0] = (cudaEvent_t)before_event;
  g_timing[kernel][1] = (cudaEvent_t)after_event;
  return CTR_OK;
}

extern "C" int ctr_status_reset(void* ws, ctr_stream_t stream) {
  if (!ws) return CTR_ERR_WORKSPACE;
  clear_word<<<1, 1, 0, (cudaStream_t)stream>>>((int*)ws); count_launch();
  return launch_status();
}

extern "C" int ctr_check_status(void* ws, ctr_stream_t stream) {
  if (!ws) return CTR_ERR_WORKSPACE;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CTR_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CTR_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(ws, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return CTR_ERR_CUDA;
  }
  return v;
}

extern "C" int ctr_fill_table(void* table, ctr_dtype dtype, int64_t rows, int32_t d, int64_t row0, int gen_kind,
                              uint64_t seed, float scale, ctr_stream_t stream) {
  if (!table || rows < 0 || d <= 0 || row0 < 0) return CTR_ERR_INVALID_ARG;
  if (rows == 0) return CTR_OK;
  const int64_t count = rows * d;
  const uint64_t idx0 = (uint64_t)row0 * (uint64_t)d;
  const int64_t blocks = imin64(ceil_div(count, 256), (int64_t)num_sms() * 32);
  cudaStream_t s = (cudaStream_t)stream;
  if (gen_kind == 0 && dtype == CTR_F32) {
    fill_uniform_f32<<<(unsigned)blocks, 256, 0, s>>>((float*)table, count, idx0, seed, scale); count_launch();
  } else if (gen_kind == 1 && dtype == CTR_BF16) {
    fill_normal4_bf16<<<(unsigned)blocks, 256, 0, s>>>((__nv_bfloat16*)table, count, idx0, seed, scale); count_launch();
  } else {
    return CTR_ERR_INVALID_ARG;
  }
  return launch_status();
}
