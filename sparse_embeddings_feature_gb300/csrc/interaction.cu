// a3/a4. Pairwise dot interaction (CUDA-core kernels) and its derivative.
//
// Sources: "Meta DLRM", section 02 (dot products between all pairs of the
// embedding vectors and the processed dense features, cross terms only);
// "DHEN" notes, section 3.1, Eq. (3) (the pairwise products are concatenated
// with the dense features).  The derivative is not on the pages.
//
// Output layout per sample: [ x_0 (dense, d values) | <x_i, x_j> for
// 1 <= i < n, 0 <= j < i, row by row ].
//
// fp32, n = 27, d = 128 (the DLRM shapes): one warp per sample.  Lane l holds
// columns 4l..4l+3 of all n vectors in registers (one 16-byte load per vector,
// coalesced across the warp), forms the partial dots of 32 pairs at a time,
// and a transpose-reduction (five xor-shuffle stages, halving the live values
// each stage) leaves pair 32g + l fully summed in lane l, so the stores are
// coalesced too.  Everything is fp32 FMA in a fixed order.
// The backward keeps the same register layout: dX_i = sum_j dZ_ij x_j, with
// the 351 upstream pair gradients of the sample staged in shared memory and
// read as broadcasts.
// Other shapes (and bf16 shapes the tensor-core kernel does not cover) use a
// generic kernel: one block per sample, vectors staged in shared memory as
// fp32, one thread per pair.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"

namespace ctr {

int interaction_bf16_tc(const void* X, int32_t batch, int32_t n, int32_t d, int mode, void* out, int* err,
                        cudaStream_t s);
bool interaction_bf16_tc_supported(int32_t n, int32_t d);

namespace {


struct PairTable {
  unsigned char i[32 * 32];
  unsigned char j[32 * 32];
};

// Output modes (see ctr_interaction_mode): products (i, j) in output order.
//   0  i > j, row-major, after the dense vector
//   1  i >= j, row-major, after the dense vector
//   2  every (i, j), row-major, no dense vector
template <int N, int MODE>
constexpr PairTable make_pairs() {
  PairTable t{};
  int p = 0;
  for (int i = 0; i < N; ++i)
    for (int j = 0; j < N; ++j) {
      if ((MODE == 0 && j >= i) || (MODE == 1 && j > i)) continue;
      t.i[p] = (unsigned char)i;
      t.j[p] = (unsigned char)j;
      ++p;
    }
  return t;
}

__host__ __device__ constexpr int64_t mode_pairs(int64_t n, int mode) {
  return mode == 0 ? n * (n - 1) / 2 : (mode == 1 ? n * (n + 1) / 2 : n * n);
}
__host__ __device__ constexpr int64_t mode_width(int64_t n, int64_t d, int mode) {
  return (mode == 2 ? 0 : d) + mode_pairs(n, mode);
}

// Packed fp32 pairs (sm_100+ f32x2 arithmetic): each half is an ordinary
// IEEE fp32 operation with round-to-nearest, two per instruction.
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ float lo32(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi32(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

// Forward, n = 27, d = 128: one warp per sample, lane l holding columns
// 4l..4l+3 of every vector as two packed pairs.  For 32 pairs at a time each
// lane forms its 4-column partial dots ((x0 y0 + x2 y2) + (x1 y1 + x3 y3),
// packed), writes them as a row of a padded 32 x 32 block in shared memory,
// and sums one column: lane t then holds dot t of the group.  (Staging the
// next sample in shared memory was measured slower: it costs occupancy, and
// the kernel is bound by issue, not by DRAM latency.)
constexpr int kFwdWarps = 4;
constexpr int kRedStride = 36;  // padded row of the transposition block (16-byte rows, conflict-free columns)
template <int N, int D, int MODE>
__global__ void __launch_bounds__(kFwdWarps * 32) interaction_fwd_f32_regs(const float* __restrict__ X, int32_t batch,
                                                                          float* __restrict__ out) {
  static_assert(D == 128, "4 columns per lane");
  // the full Gram matrix is symmetric: compute i >= j once, store (i, j) and (j, i)
  constexpr int CM = MODE == 2 ? 1 : MODE;
  constexpr int P = (int)mode_pairs(N, CM);
  constexpr int G = (P + 31) / 32;
  constexpr int W = (int)mode_width(N, D, MODE);
  constexpr int OFF = MODE == 2 ? 0 : D;  // where the products start in an output row
  constexpr PairTable pt = make_pairs<N, CM>();
  __shared__ __align__(16) float sred[kFwdWarps][32 * kRedStride];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* red = sred[warp];
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < batch; b += nwarps) {
    uint64_t xl[N], xh[N];  // columns (4l, 4l+1) and (4l+2, 4l+3) of each vector
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const ulonglong2 v = __ldcs((const ulonglong2*)(X + b * (int64_t)N * D + i * D + lane * 4));
      xl[i] = v.x;
      xh[i] = v.y;
    }
    float* ob = out + b * (int64_t)W;
    if (MODE != 2) {
      __stcs(ob + lane * 4 + 0, lo32(xl[0]));
      __stcs(ob + lane * 4 + 1, hi32(xl[0]));
      __stcs(ob + lane * 4 + 2, lo32(xh[0]));
      __stcs(ob + lane * 4 + 3, hi32(xh[0]));
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float v[32];
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int p = g * 32 + t;
        if (p < P) {
          const int i = pt.i[p], j = pt.j[p];
          const uint64_t m = fma2(xh[i], xh[j], mul2(xl[i], xl[j]));
          v[t] = lo32(m) + hi32(m);
        } else {
          v[t] = 0.f;
        }
      }
      __syncwarp();  // the previous group's columns have been read
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *(float4*)(red + lane * kRedStride + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      __syncwarp();
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int r = 0; r < 32; ++r) acc[r & 3] += red[r * kRedStride + lane];
      const int p = g * 32 + lane;
      if (p < P) {
        const float dot = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        if (MODE == 2) {
          int i = (int)((1.f + sqrtf(1.f + 8.f * (float)p)) * 0.5f) - 1;  // pair p = i(i+1)/2 + j, j <= i
          if (i * (i + 1) / 2 > p) --i;
          if ((i + 1) * (i + 2) / 2 <= p) ++i;
          const int j = p - i * (i + 1) / 2;
          __stcs(ob + i * N + j, dot);
          if (i != j) __stcs(ob + j * N + i, dot);
        } else {
          __stcs(ob + OFF + p, dot);
        }
      }
    }
  }
}

constexpr int kBwdWarps = 4;

// Backward, n = 27, d = 128: one warp per sample.  The sample's upstream pair
// gradients are expanded into a symmetric matrix S (zero diagonal, rows padded
// to 28 floats) in the warp's shared memory; lane l holds columns 4l..4l+3 of
// every vector in registers, and row i of dX is the branch-free sweep
// dX_i = sum_j S[i][j] x_j: one 16-byte broadcast load of S per four j and
// sixteen FMAs.
template <int N, int D, int MODE>
__global__ void __launch_bounds__(kBwdWarps * 32) interaction_bwd_f32_regs(const float* __restrict__ dout,
                                                                          const float* __restrict__ X, int32_t batch,
                                                                          float* __restrict__ dX) {
  static_assert(D == 128, "4 columns per lane");
  constexpr int W = (int)mode_width(N, D, MODE);
  // S = G + G^T over the products the mode emits: built from the pairs i >= j
  // (i > j for mode 0, whose diagonal stays zero)
  constexpr int PS = MODE == 0 ? N * (N - 1) / 2 : N * (N + 1) / 2;
  constexpr int SH = MODE == 0 ? 0 : 1;  // pair (i, j) of the lower triangle is at i(i - 1 + 2 SH)/2 + j
  constexpr int NP = (N + 3) / 4 * 4;  // padded row length of S
  __shared__ __align__(16) float sS[kBwdWarps][N * NP];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  float* S = sS[warp];
  for (int e = lane; e < N * NP; e += 32) S[e] = 0.f;  // diagonal and padding stay zero
  __syncwarp();
  for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < batch; b += nwarps) {
    const float* xb = X + b * (int64_t)N * D + lane * 4;
    const float* gb = dout + b * (int64_t)W;
    float x[NP][4];
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float4 v = __ldcs((const float4*)(xb + i * D));
      x[i][0] = v.x;
      x[i][1] = v.y;
      x[i][2] = v.z;
      x[i][3] = v.w;
    }
#pragma unroll
    for (int i = N; i < NP; ++i) x[i][0] = x[i][1] = x[i][2] = x[i][3] = 0.f;
    float dense[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) dense[c] = MODE == 2 ? 0.f : __ldcs(gb + lane * 4 + c);
    __syncwarp();  // the previous sample's S is no longer read
    for (int p = lane; p < PS; p += 32) {
      int i = (int)((1.f + sqrtf(1.f + 8.f * (float)p)) * 0.5f) - SH;  // row of pair p
      if (i * (i - 1 + 2 * SH) / 2 > p) --i;
      if ((i + 1) * (i + 2 * SH) / 2 <= p) ++i;
      const int j = p - i * (i - 1 + 2 * SH) / 2;
      float g;
      if (MODE == 2) g = i == j ? 2.f * __ldcs(gb + i * N + i) : __ldcs(gb + i * N + j) + __ldcs(gb + j * N + i);
      else g = (i == j ? 2.f : 1.f) * __ldcs(gb + D + p);
      S[i * NP + j] = g;
      S[j * NP + i] = g;
    }
    __syncwarp();
    float* ob = dX + b * (int64_t)N * D + lane * 4;
#pragma unroll 1
    for (int i = 0; i < N; ++i) {
      float acc[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[c] = (i == 0) ? dense[c] : 0.f;
      const float4* Si = (const float4*)(S + i * NP);
#pragma unroll
      for (int q = 0; q < NP / 4; ++q) {
        const float4 s4 = Si[q];
        const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[c] = fmaf(sv[r], x[4 * q + r][c], acc[c]);
      }
      __stcs((float4*)(ob + i * D), make_float4(acc[0], acc[1], acc[2], acc[3]));
    }
  }
}

template <typename TT>
__device__ __forceinline__ float to_f(TT v);
template <>
__device__ __forceinline__ float to_f<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
__device__ __forceinline__ void put(float* o, float v) { *o = v; }
__device__ __forceinline__ void put(__nv_bfloat16* o, float v) { *o = __float2bfloat16_rn(v); }

constexpr int kGenThreads = 128;

// Generic: one block per sample (grid-stride), vectors in shared memory.
__device__ __forceinline__ void pair_of(int64_t p, int n, int mode, int& i, int& j) {
  if (mode == 2) {
    i = (int)(p / n);
    j = (int)(p - (int64_t)i * n);
    return;
  }
  // row i of slot p: the largest i with first(i) <= p, first(i) = i(i-1)/2 (mode 0) or i(i+1)/2 (mode 1)
  const int sh = mode == 1 ? 1 : 0;
  int r = (int)((1.0 + sqrt(1.0 + 8.0 * (double)p)) * 0.5) - sh;
  auto first = [&](int64_t x) { return mode == 1 ? x * (x + 1) / 2 : x * (x - 1) / 2; };
  while (r > 0 && first(r) > p) --r;
  while (first(r + 1) <= p) ++r;
  i = r;
  j = (int)(p - first(r));
}

template <typename TT>
__global__ void __launch_bounds__(kGenThreads) interaction_fwd_generic(const TT* __restrict__ X, int32_t batch,
                                                                      int32_t n, int32_t d, int mode,
                                                                      TT* __restrict__ out) {
  extern __shared__ float xs[];  // [n][d]
  const int64_t P = mode_pairs(n, mode);
  const int64_t W = mode_width(n, d, mode);
  const int64_t off = mode == 2 ? 0 : d;
  for (int64_t b = blockIdx.x; b < batch; b += gridDim.x) {
    const TT* xb = X + b * (int64_t)n * d;
    for (int e = threadIdx.x; e < n * d; e += blockDim.x) xs[e] = to_f(xb[e]);
    __syncthreads();
    TT* ob = out + b * W;
    if (mode != 2)
      for (int c = threadIdx.x; c < d; c += blockDim.x) ob[c] = xb[c];
    for (int64_t p = threadIdx.x; p < P; p += blockDim.x) {
      int i, j;
      pair_of(p, n, mode, i, j);
      const float* a = xs + i * d;
      const float* c = xs + j * d;
      float s = 0.f;
      for (int k = 0; k < d; ++k) s = fmaf(a[k], c[k], s);
      put(ob + off + p, s);
    }
    __syncthreads();
  }
}

// S_ij = G_ij + G_ji over the products the mode emits (the derivative of
// <x_i, x_j> adds x_j to dX_i and x_i to dX_j).
__device__ __forceinline__ float s_entry(const float* gb, int n, int d, int mode, int i, int j) {
  if (mode == 2) return gb[(int64_t)i * n + j] + gb[(int64_t)j * n + i];
  if (i == j) return mode == 1 ? 2.f * gb[d + (int64_t)i * (i + 1) / 2 + i] : 0.f;
  const int hi = i > j ? i : j, lo = i > j ? j : i;
  return gb[d + (mode == 1 ? (int64_t)hi * (hi + 1) / 2 : (int64_t)hi * (hi - 1) / 2) + lo];
}

__global__ void __launch_bounds__(kGenThreads) interaction_bwd_generic(const float* __restrict__ dout,
                                                                      const float* __restrict__ X, int32_t batch,
                                                                      int32_t n, int32_t d, int mode,
                                                                      float* __restrict__ dX) {
  extern __shared__ float sm[];  // xs [n][d], S [n][n]
  const int64_t W = mode_width(n, d, mode);
  float* xs = sm;
  float* S = sm + (int64_t)n * d;
  for (int64_t b = blockIdx.x; b < batch; b += gridDim.x) {
    const float* xb = X + b * (int64_t)n * d;
    const float* gb = dout + b * W;
    for (int e = threadIdx.x; e < n * d; e += blockDim.x) xs[e] = xb[e];
    for (int e = threadIdx.x; e < n * n; e += blockDim.x) S[e] = s_entry(gb, n, d, mode, e / n, e % n);
    __syncthreads();
    for (int e = threadIdx.x; e < n * d; e += blockDim.x) {
      const int i = e / d, c = e % d;
      float acc = (i == 0 && mode != 2) ? gb[c] : 0.f;
      for (int j = 0; j < n; ++j) acc = fmaf(S[i * n + j], xs[j * d + c], acc);
      dX[b * (int64_t)n * d + e] = acc;
    }
    __syncthreads();
  }
}

template <typename K>
int grid_blocks(K kernel, int threads, size_t smem, int64_t work_units) {
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
  int64_t cap = (int64_t)std::max(per_sm, 1) * num_sms();
  return (int)std::max<int64_t>(1, std::min(work_units, cap));
}

}  // namespace
}  // namespace ctr

using namespace ctr;

extern "C" size_t ctr_interaction_workspace_size(void) { return kWsHeader; }

extern "C" int64_t ctr_interaction_width(int32_t n, int32_t d, int mode) {
  if (n < 1 || d < 1 || mode < 0 || mode > 2) return -1;
  return mode_width(n, d, mode);
}

namespace {

template <int MODE>
void launch_fwd_fast(const float* X, int32_t batch, float* out, cudaStream_t s) {
  auto k = interaction_fwd_f32_regs<27, 128, MODE>;
  k<<<grid_blocks(k, kFwdWarps * 32, 0, ceil_div(batch, kFwdWarps)), kFwdWarps * 32, 0, s>>>(X, batch, out);
  count_launch();
}

template <int MODE>
void launch_bwd_fast(const float* dout, const float* X, int32_t batch, float* dX, cudaStream_t s) {
  auto k = interaction_bwd_f32_regs<27, 128, MODE>;
  k<<<grid_blocks(k, kBwdWarps * 32, 0, ceil_div(batch, kBwdWarps)), kBwdWarps * 32, 0, s>>>(dout, X, batch, dX);
  count_launch();
}

int dot_interaction_launch(const void* X, ctr_dtype dtype, int32_t batch, int32_t n, int32_t d, int mode, void* out,
                           void* ws, cudaStream_t s) {
  if (dtype == CTR_F32 && n == 27 && d == 128 && (uintptr_t)X % 16 == 0) {
    if (mode == 0) launch_fwd_fast<0>((const float*)X, batch, (float*)out, s);
    else if (mode == 1) launch_fwd_fast<1>((const float*)X, batch, (float*)out, s);
    else launch_fwd_fast<2>((const float*)X, batch, (float*)out, s);
    return launch_status();
  }
  if (dtype == CTR_BF16 && interaction_bf16_tc_supported(n, d) && (uintptr_t)X % 16 == 0 &&
      (uintptr_t)out % 16 == 0)
    return interaction_bf16_tc(X, batch, n, d, mode, out, (int*)ws, s);
  const size_t smem = (size_t)n * d * sizeof(float);
  if (smem > 48 * 1024) return CTR_ERR_UNSUPPORTED;
  if (dtype == CTR_F32) {
    auto k = interaction_fwd_generic<float>;
    k<<<grid_blocks(k, kGenThreads, smem, batch), kGenThreads, smem, s>>>((const float*)X, batch, n, d, mode,
                                                                           (float*)out);
    count_launch();
  } else {
    auto k = interaction_fwd_generic<__nv_bfloat16>;
    k<<<grid_blocks(k, kGenThreads, smem, batch), kGenThreads, smem, s>>>((const __nv_bfloat16*)X, batch, n, d, mode,
                                                                           (__nv_bfloat16*)out);
    count_launch();
  }
  return launch_status();
}

int dot_interaction_bwd_launch(const float* dout, const float* X, int32_t batch, int32_t n, int32_t d, int mode,
                               float* dX, cudaStream_t s) {
  if (n == 27 && d == 128 && (uintptr_t)X % 16 == 0 && (uintptr_t)dX % 16 == 0) {
    if (mode == 0) launch_bwd_fast<0>(dout, X, batch, dX, s);
    else if (mode == 1) launch_bwd_fast<1>(dout, X, batch, dX, s);
    else launch_bwd_fast<2>(dout, X, batch, dX, s);
    return launch_status();
  }
  const size_t smem = ((size_t)n * d + (size_t)n * n) * sizeof(float);
  if (smem > 48 * 1024) return CTR_ERR_UNSUPPORTED;
  auto k = interaction_bwd_generic;
  k<<<grid_blocks(k, kGenThreads, smem, batch), kGenThreads, smem, s>>>(dout, X, batch, n, d, mode, dX);
  count_launch();
  return launch_status();
}

int dot_interaction_entry(const void* X, ctr_dtype dtype, int32_t batch, int32_t n, int32_t d, int mode, void* out,
                          void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!X || !out || batch < 0 || n < 1 || d < 1) return CTR_ERR_INVALID_ARG;
  if (dtype != CTR_F32 && dtype != CTR_BF16) return CTR_ERR_INVALID_ARG;
  if (mode < 0 || mode > 2) return CTR_ERR_INVALID_ARG;
  if (!ws_valid(ws, ws_bytes, kWsHeader)) return CTR_ERR_WORKSPACE;
  if (batch == 0) return CTR_OK;
  timing_mark(CTR_KERNEL_INTERACTION, true, s);
  const int st = dot_interaction_launch(X, dtype, batch, n, d, mode, out, ws, s);
  timing_mark(CTR_KERNEL_INTERACTION, false, s);
  return st;
}

int dot_interaction_bwd_entry(const float* dout, const float* X, int32_t batch, int32_t n, int32_t d, int mode,
                              float* dX, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!dout || !X || !dX || batch < 0 || n < 1 || d < 1) return CTR_ERR_INVALID_ARG;
  if (mode < 0 || mode > 2) return CTR_ERR_INVALID_ARG;
  if (!ws_valid(ws, ws_bytes, kWsHeader)) return CTR_ERR_WORKSPACE;
  if (batch == 0) return CTR_OK;
  timing_mark(CTR_KERNEL_INTERACTION_BWD, true, s);
  const int st = dot_interaction_bwd_launch(dout, X, batch, n, d, mode, dX, s);
  timing_mark(CTR_KERNEL_INTERACTION_BWD, false, s);
  return st;
}

}  // namespace

extern "C" int ctr_dot_interaction(const void* X, ctr_dtype dtype, int32_t batch, int32_t n, int32_t d, void* out,
                                   void* ws, size_t ws_bytes, ctr_stream_t stream) {
  return dot_interaction_entry(X, dtype, batch, n, d, CTR_INTERACT_CROSS, out, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int ctr_dot_interaction_bwd(const float* dout, const float* X, int32_t batch, int32_t n, int32_t d,
                                       float* dX, void* ws, size_t ws_bytes, ctr_stream_t stream) {
  return dot_interaction_bwd_entry(dout, X, batch, n, d, CTR_INTERACT_CROSS, dX, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int ctr_dot_interaction_mode(const void* X, ctr_dtype dtype, int32_t batch, int32_t n, int32_t d, int mode,
                                        void* out, void* ws, size_t ws_bytes, ctr_stream_t stream) {
  return dot_interaction_entry(X, dtype, batch, n, d, mode, out, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int ctr_dot_interaction_bwd_mode(const float* dout, const float* X, int32_t batch, int32_t n, int32_t d,
                                            int mode, float* dX, void* ws, size_t ws_bytes, ctr_stream_t stream) {
  return dot_interaction_bwd_entry(dout, X, batch, n, d, mode, dX, ws, ws_bytes, (cudaStream_t)stream);
}
