// Device-wide exclusive prefix sum (reduce-then-scan, Merrill and Grimshaw
// style): per-block partial sums, a scan of the partials (recursive when they
// do not fit one block), then a block-local scan seeded with its partial.
// No block waits on another, so no launch can hang.
#pragma once

#include "common.cuh"

namespace ctr {

template <typename T>
struct ScanTile {
  static constexpr int kThreads = 256;
  static constexpr int kItems = sizeof(T) >= 8 ? 8 : 16;
  static constexpr int kTile = kThreads * kItems;
};

__host__ __device__ constexpr int scan_pad(int a) { return a + (a >> 5); }

// Element count: the host bound, further limited by a device scalar if given.
__device__ __forceinline__ int64_t scan_count(int64_t n_host, const int64_t* n_dev) {
  if (!n_dev) return n_host;
  int64_t d = *n_dev;
  return d < n_host ? d : n_host;
}

// Exclusive scan of v[] (this thread's kItems consecutive values) across the
// block; returns the block total.  Uses warp_tot[kThreads / 32].
template <typename T, int kThreads, int kItems>
__device__ __forceinline__ T block_exclusive_scan(T (&v)[kItems], T* warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kThreads / 32;
  T sum = 0;
#pragma unroll
  for (int i = 0; i < kItems; ++i) {
    T x = v[i];
    v[i] = sum;
    sum += x;
  }
  T inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    T w = lane < kWarps ? warp_tot[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) warp_tot[lane] = w;
  }
  __syncthreads();
  T excl = (warp > 0 ? warp_tot[warp - 1] : T(0)) + inc - sum;
  T total = warp_tot[kWarps - 1];
#pragma unroll
  for (int i = 0; i < kItems; ++i) v[i] += excl;
  __syncthreads();
  return total;
}

template <typename T>
__global__ void __launch_bounds__(ScanTile<T>::kThreads)
    scan_reduce_kernel(const T* __restrict__ in, int64_t n_host, const int64_t* __restrict__ n_dev,
                       T* __restrict__ block_sums) {
  using S = ScanTile<T>;
  __shared__ T warp_tot[S::kThreads / 32];
  const int64_t n = scan_count(n_host, n_dev);
  const int64_t base = (int64_t)blockIdx.x * S::kTile;
  T sum = 0;
#pragma unroll 4
  for (int i = 0; i < S::kItems; ++i) {
    int64_t idx = base + (int64_t)i * S::kThreads + threadIdx.x;
    if (idx < n) sum += in[idx];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  if ((threadIdx.x & 31) == 0) warp_tot[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    T t = 0;
    for (int w = 0; w < S::kThreads / 32; ++w) t += warp_tot[w];
    block_sums[blockIdx.x] = t;
  }
}

// out[i] = offset(block) + exclusive prefix of in within the block.  In-place
// (out == in) is allowed: a block reads its whole tile before writing.
template <typename T>
__global__ void __launch_bounds__(ScanTile<T>::kThreads)
    scan_down_kernel(const T* in, T* out, int64_t n_host, const int64_t* __restrict__ n_dev,
                     const T* __restrict__ block_offsets, T* __restrict__ total_out) {
  using S = ScanTile<T>;
  __shared__ T tile[scan_pad(S::kTile) + 1];
  __shared__ T warp_tot[S::kThreads / 32];
  const int64_t n = scan_count(n_host, n_dev);
  const int64_t base = (int64_t)blockIdx.x * S::kTile;
#pragma unroll
  for (int i = 0; i < S::kItems; ++i) {
    int a = i * S::kThreads + threadIdx.x;
    int64_t idx = base + a;
    tile[scan_pad(a)] = idx < n ? in[idx] : T(0);
  }
  __syncthreads();
  T v[S::kItems];
#pragma unroll
  for (int i = 0; i < S::kItems; ++i) v[i] = tile[scan_pad(threadIdx.x * S::kItems + i)];
  __syncthreads();
  T total = block_exclusive_scan<T, S::kThreads, S::kItems>(v, warp_tot);
  T off = block_offsets ? block_offsets[blockIdx.x] : T(0);
#pragma unroll
  for (int i = 0; i < S::kItems; ++i) tile[scan_pad(threadIdx.x * S::kItems + i)] = v[i] + off;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < S::kItems; ++i) {
    int a = i * S::kThreads + threadIdx.x;
    int64_t idx = base + a;
    if (idx < n) out[idx] = tile[scan_pad(a)];
  }
  if (total_out && threadIdx.x == 0 && blockIdx.x == gridDim.x - 1) *total_out = off + total;
}

template <typename T, typename WS>
inline void scan_reserve(WS& ws, int64_t n_host) {
  using S = ScanTile<T>;
  while (n_host > S::kTile) {
    int64_t nb = ceil_div(n_host, S::kTile);
    ws.template take<T>((size_t)nb);
    n_host = nb;
  }
}

// Exclusive scan of in[0..n) into out (n = min(n_host, *n_dev) if n_dev).
// total_out (device, may be null) receives the sum of all n elements.
template <typename T>
inline int scan_exclusive(const T* in, T* out, int64_t n_host, const int64_t* n_dev, T* total_out, WsCarver& ws,
                          cudaStream_t s) {
  using S = ScanTile<T>;
  if (n_host <= S::kTile) {
    scan_down_kernel<T><<<1, S::kThreads, 0, s>>>(in, out, n_host, n_dev, nullptr, total_out); count_launch();
    return launch_status();
  }
  int64_t nb = ceil_div(n_host, S::kTile);
  T* sums = ws.take<T>((size_t)nb);
  if (!sums) return CTR_ERR_WORKSPACE;
  scan_reduce_kernel<T><<<(unsigned)nb, S::kThreads, 0, s>>>(in, n_host, n_dev, sums); count_launch();
  int st = launch_status();
  if (st) return st;
  st = scan_exclusive<T>(sums, sums, nb, nullptr, total_out, ws, s);
  if (st) return st;
  scan_down_kernel<T><<<(unsigned)nb, S::kThreads, 0, s>>>(in, out, n_host, n_dev, sums, nullptr); count_launch();
  return launch_status();
}

}  // namespace ctr
