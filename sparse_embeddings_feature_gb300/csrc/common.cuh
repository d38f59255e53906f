// Shared device/host helpers of libctr (the CUDA path).  Nothing here is
// shared with the CPU oracle.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ctr.h"

namespace ctr {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr size_t kWsHeader = 256;  // sticky error word lives at the head of every workspace
constexpr size_t kWsCounterOffset = 64;  // a work counter some kernels keep in the header

// Next work unit for the calling warp, handed out in launch order from a
// global counter, so the warps in flight stay on a narrow window of
// consecutive units (their data shares L2) instead of drifting apart as a
// grid-stride loop does.
__device__ __forceinline__ int64_t next_unit(unsigned long long* counter) {
  unsigned long long u = 0;
  if ((threadIdx.x & 31) == 0) u = atomicAdd(counter, 1ull);
  return (int64_t)__shfl_sync(0xffffffffu, u, 0);
}

// Device-side error codes recorded in the workspace header (first one wins).
__device__ __forceinline__ void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__host__ __device__ __forceinline__ int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t imax64(int64_t a, int64_t b) { return a > b ? a : b; }
__host__ __device__ __forceinline__ size_t align_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

// Per-field table placement, passed by value as a kernel parameter.
struct FieldMap {
  int64_t base[CTR_MAX_FIELDS];  // row_base[bag_to_table[f]]
  int64_t rows[CTR_MAX_FIELDS];  // rows of that table
};

// Fill a FieldMap from the host arrays; returns a ctr_status.
inline int make_field_map(const int32_t* bag_to_table, const int64_t* row_base, int32_t F, int32_t T,
                          FieldMap* fm) {
  if (F <= 0 || T <= 0) return CTR_ERR_INVALID_ARG;
  if (F > CTR_MAX_FIELDS || T > CTR_MAX_TABLES) return CTR_ERR_UNSUPPORTED;
  if (row_base[0] != 0) return CTR_ERR_INVALID_ARG;
  for (int t = 0; t < T; ++t)
    if (row_base[t + 1] < row_base[t]) return CTR_ERR_INVALID_ARG;
  for (int f = 0; f < F; ++f) {
    int t = bag_to_table[f];
    if (t < 0 || t >= T) return CTR_ERR_INVALID_ARG;
    fm->base[f] = row_base[t];
    fm->rows[f] = row_base[t + 1] - row_base[t];
  }
  return CTR_OK;
}

// Timing hook (ctr_set_timing_events): record the caller's events around a launch.
void timing_mark(int kernel, bool before, cudaStream_t s);
// Counts one kernel launch (called right after each launch statement).
void count_launch();

// Number of SMs of the current device (cached per device).
int num_sms();

// Map the last CUDA error to a ctr_status.
inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CTR_OK : CTR_ERR_CUDA;
}

// Carves sub-buffers out of a caller workspace (after the header).
struct WsCarver {
  char* base;
  size_t cap;
  size_t used;
  explicit WsCarver(void* ws, size_t bytes) : base((char*)ws), cap(bytes), used(kWsHeader) {}
  template <typename T>
  T* take(size_t count) {
    size_t off = align_up(used, 256);
    used = off + align_up(count * sizeof(T), 256);
    return used <= cap ? (T*)(base + off) : nullptr;
  }
  bool ok() const { return used <= cap; }
};

// Same arithmetic without a buffer: used to size workspaces.
struct WsSizer {
  size_t used = kWsHeader;
  template <typename T>
  void take(size_t count) {
    size_t off = align_up(used, 256);
    used = off + align_up(count * sizeof(T), 256);
  }
};

inline bool ws_valid(void* ws, size_t ws_bytes, size_t need) {
  return ws != nullptr && ((uintptr_t)ws % 256) == 0 && ws_bytes >= need;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// L2 cache policies for data with known reuse: keep (evict_last) rows that are
// read many times within a kernel, let streamed data go first (evict_first).
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last_fraction(float f) {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, %1;" : "=l"(p) : "f"(f));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ float4 ldg_f4_policy(const float* p, uint64_t pol) {
  float4 r;
  asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p), "l"(pol));
  return r;
}
__device__ __forceinline__ void stg_f4_policy(float* p, float4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w), "l"(pol)
               : "memory");
}

// splitmix64 output function (Steele, Lea and Flood, OOPSLA 2014): a
// counter-based source of 64 random bits per index.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Four-lane accumulation with packed fp32 pairs (f32x2, sm_100+): two
// instructions instead of four; each half is the same IEEE operation as the
// scalar form, so the results are bit-identical.
__device__ __forceinline__ float4 add4_packed(float4 acc, float4 x) {
  uint64_t a0, a1, b0, b1;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a0) : "f"(acc.x), "f"(acc.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(a1) : "f"(acc.z), "f"(acc.w));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b0) : "f"(x.x), "f"(x.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(b1) : "f"(x.z), "f"(x.w));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a0) : "l"(b0));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a1) : "l"(b1));
  float4 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(a0));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.z), "=f"(r.w) : "l"(a1));
  return r;
}
}  // namespace ctr
