// a5. Sparse backward: per-unique-row gradient reduce + SGD row update.
//
// Source: "How TensorNet Supercharges Sparse Feature Training on TensorFlow",
// Synchronous Architecture (only the sparse features present in the batch are
// synchronised) and Core Optimizations (the batch-sized matrix of unique rows).
//
// GPU design.  The occurrences of unique u are the sorted slots
// run_offsets[u] .. run_offsets[u+1]-1 (from the dedup); sorted_bag gives the
// bag whose pooled gradient each one contributes.  Runs are cut into pieces of
// at most kPiece occurrences:
//   1. count    pieces per run (and whether the run is long: > 1 piece)
//   2. scan     exclusive scans give each piece a slot and each long run a
//               slot in the list of long runs
//   3. expand   piece -> unique map, list of long runs
//   4. reduce   one warp per piece sums its rows in sorted order (fp32, fixed
//               order); a one-piece run is finished here (row update); a piece
//               of a long run stores a partial sum
//   5. combine  one CTA per long run sums its partials: each warp a fixed
//               contiguous segment, then a fixed tree over the warps, then the
//               row update.
// Every row is written by exactly one warp or CTA; there are no float atomics,
// and the summation order depends only on the run lengths, so the result is
// deterministic.  Because the unique rows are sorted table-major, the warps in
// flight all read pooled gradients of one field, whose slice stays in L2.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "scan.cuh"

namespace ctr {
namespace {

constexpr int kPiece = 128;        // occurrences per piece
constexpr int kRedThreads = 256;
constexpr int kCombThreads = 256;
constexpr int kUnrollB = 4;

struct BwdArgs {
  const float* G;
  int64_t sb, sf;
  const int64_t* offsets;
  int32_t B;
  int mean;
  const int64_t* unique_rows;
  const int64_t* n_unique;
  const int32_t* run_offsets;
  const int32_t* sorted_bag;
  float lr;
  void* table;
  int bf16;
  int32_t d;
  int64_t total_rows;
  float* grad_out;
  int* err;
  int64_t n_cap;         // occurrences (sorted_bag length)
  int64_t nbags;         // F * B
  // scratch
  uint64_t* pstart;      // [n] lo: first piece, hi: first long piece (exclusive scan)
  uint32_t* lstart;      // [n] slot in the long-run list (exclusive scan)
  uint64_t* ptotal;      // lo: pieces, hi: long pieces
  uint32_t* ltotal;      // long runs
  int32_t* piece_u;      // [pieces] unique of each piece
  int32_t* long_list;    // [long runs]
  float* partial;        // [long pieces, d]
};

__device__ __forceinline__ int64_t n_uniques(const BwdArgs& a, int64_t cap) {
  int64_t n = *a.n_unique;
  return n < cap ? n : cap;
}

// Run bounds of unique u; an inconsistent run is treated as empty (and flagged
// by piece_count_kernel), so no kernel indexes outside its buffers.
__device__ __forceinline__ void run_bounds(const BwdArgs& a, int64_t u, int64_t& r0, int64_t& r1) {
  r0 = a.run_offsets[u];
  r1 = a.run_offsets[u + 1];
  if (r0 < 0 || r1 < r0 || r1 > a.n_cap) r0 = r1 = 0;
}

__global__ void piece_count_kernel(const BwdArgs a, int64_t cap, uint64_t* __restrict__ cnt2,
                                   uint32_t* __restrict__ cnt1) {
  const int64_t n = n_uniques(a, cap);
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < n; u += (int64_t)gridDim.x * blockDim.x) {
    const int64_t q0 = a.run_offsets[u], q1 = a.run_offsets[u + 1];
    if (q0 < 0 || q1 < q0 || q1 > a.n_cap) set_error(a.err, CTR_ERR_BAD_OFFSETS);
    int64_t r0, r1;
    run_bounds(a, u, r0, r1);
    int64_t len = r1 - r0;
    uint64_t pcs = len > 0 ? (uint64_t)ceil_div(len, kPiece) : 1u;
    bool lng = pcs > 1;
    cnt2[u] = pcs | ((lng ? pcs : 0ull) << 32);
    cnt1[u] = lng ? 1u : 0u;
  }
}

__global__ void expand_kernel(const BwdArgs a, int64_t cap) {
  const int64_t n = n_uniques(a, cap);
  for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < n; u += (int64_t)gridDim.x * blockDim.x) {
    int64_t r0, r1;
    run_bounds(a, u, r0, r1);
    int64_t len = r1 - r0;
    int64_t pcs = len > 0 ? ceil_div(len, kPiece) : 1;
    uint64_t p0 = a.pstart[u] & 0xffffffffull;
    for (int64_t k = 0; k < pcs; ++k) a.piece_u[p0 + k] = (int32_t)u;
    if (pcs > 1) a.long_list[a.lstart[u]] = (int32_t)u;
  }
}

// Row update for unique u with its gradient chunk g (V floats at column c0).
template <int V>
__device__ __forceinline__ void finish_chunk(const BwdArgs& a, int64_t u, int c0, const float (&g)[V]) {
  const int64_t row = a.unique_rows[u];
  if (row < 0 || row >= a.total_rows) {
    set_error(a.err, CTR_ERR_INDEX_OUT_OF_RANGE);
    return;
  }
  if (a.grad_out) {
    float* go = a.grad_out + u * a.d + c0;
#pragma unroll
    for (int v = 0; v < V; ++v) go[v] = g[v];
  }
  if (!a.bf16) {
    float* w = (float*)a.table + row * a.d + c0;
    if (V == 4) {
      float4 x = *(float4*)w;
      x.x = fmaf(-a.lr, g[0], x.x);
      x.y = fmaf(-a.lr, g[1], x.y);
      x.z = fmaf(-a.lr, g[2], x.z);
      x.w = fmaf(-a.lr, g[3], x.w);
      *(float4*)w = x;
    } else {
#pragma unroll
      for (int v = 0; v < V; ++v) w[v] = fmaf(-a.lr, g[v], w[v]);
    }
  } else {
    __nv_bfloat16* w = (__nv_bfloat16*)a.table + row * a.d + c0;
#pragma unroll
    for (int v = 0; v < V; ++v) w[v] = __float2bfloat16_rn(fmaf(-a.lr, g[v], __bfloat162float(w[v])));
  }
}

__device__ __forceinline__ float4 ldg_f4(const float* p) {
  float4 r;
  asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p));
  return r;
}

// One warp per piece.  LPR lanes cover a row (4 floats each, CPL chunks per
// lane); 32/LPR occurrences are summed side by side and combined at the end.
template <int LPR, int CPL>
__global__ void __launch_bounds__(kRedThreads) reduce_pieces_kernel(const BwdArgs a) {
  constexpr int R = 32 / LPR;
  const int lane = threadIdx.x & 31;
  const int grp = lane / LPR, sub = lane % LPR;
  const int chunks = a.d / 4;
  const int64_t npieces = (int64_t)(*a.ptotal & 0xffffffffull);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t p = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < npieces; p += nwarps) {
    const int64_t u = a.piece_u[p];
    const uint64_t ps = a.pstart[u];
    const int64_t k = p - (int64_t)(ps & 0xffffffffull);
    int64_t r0, r1;
    run_bounds(a, u, r0, r1);
    const int64_t s0 = r0 + k * kPiece;
    const int64_t s1 = imin64(r1, s0 + kPiece);
    float acc[CPL][4];
#pragma unroll
    for (int c = 0; c < CPL; ++c)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[c][v] = 0.f;
    for (int64_t j0 = s0; j0 < s1; j0 += 32) {
      const int cnt = (int)imin64(32, s1 - j0);
      int64_t goff = -1;  // -1: this occurrence contributes nothing
      float scale = 1.f;
      if (lane < cnt) {
        const int32_t bag = a.sorted_bag[j0 + lane];
        if (bag < 0 || bag >= a.nbags) {
          set_error(a.err, CTR_ERR_BAD_OFFSETS);
        } else {
          const int32_t f = bag / a.B, b = bag - f * a.B;
          goff = (int64_t)b * a.sb + (int64_t)f * a.sf;
          if (a.mean) {
            int64_t len = a.offsets[bag + 1] - a.offsets[bag];
            scale = len > 0 ? 1.f / (float)len : 0.f;
          }
        }
      }
      for (int t0 = 0; t0 < cnt; t0 += R * kUnrollB) {
        float4 buf[kUnrollB][CPL];
        float sc[kUnrollB];
#pragma unroll
        for (int uu = 0; uu < kUnrollB; ++uu) {
          const int t = t0 + uu * R + grp;
          const int64_t go = __shfl_sync(kFull, goff, t & 31);
          sc[uu] = __shfl_sync(kFull, scale, t & 31);
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const int ch = sub + c * LPR;
            buf[uu][c] = (t < cnt && go >= 0 && ch < chunks) ? ldg_f4(a.G + go + ch * 4)
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
          }
          if (t >= cnt) sc[uu] = 0.f;
        }
#pragma unroll
        for (int uu = 0; uu < kUnrollB; ++uu)
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            if (a.mean) {
              acc[c][0] = fmaf(buf[uu][c].x, sc[uu], acc[c][0]);
              acc[c][1] = fmaf(buf[uu][c].y, sc[uu], acc[c][1]);
              acc[c][2] = fmaf(buf[uu][c].z, sc[uu], acc[c][2]);
              acc[c][3] = fmaf(buf[uu][c].w, sc[uu], acc[c][3]);
            } else {
              acc[c][0] += buf[uu][c].x;
              acc[c][1] += buf[uu][c].y;
              acc[c][2] += buf[uu][c].z;
              acc[c][3] += buf[uu][c].w;
            }
          }
      }
    }
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[c][v] += __shfl_xor_sync(kFull, acc[c][v], o);
    if (grp != 0) continue;
    const bool single = (r1 - r0) <= kPiece;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int ch = sub + c * LPR;
      if (ch >= chunks) continue;
      if (single) {
        finish_chunk<4>(a, u, ch * 4, acc[c]);
      } else {
        const int64_t lp = (int64_t)(ps >> 32) + k;
        *(float4*)(a.partial + lp * a.d + ch * 4) = make_float4(acc[c][0], acc[c][1], acc[c][2], acc[c][3]);
      }
    }
  }
}

// One CTA per long run: warps sum fixed contiguous segments of the run's
// partials, then a fixed tree over the warps.  Threads own 4-float chunks.
__global__ void __launch_bounds__(kCombThreads) combine_long_kernel(const BwdArgs a) {
  constexpr int W = kCombThreads / 32;
  extern __shared__ float sm[];  // [W][d]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int chunks = a.d / 4;
  const int64_t nlong = *a.ltotal;
  for (int64_t i = blockIdx.x; i < nlong; i += gridDim.x) {
    const int64_t u = a.long_list[i];
    int64_t r0, r1;
    run_bounds(a, u, r0, r1);
    const int64_t pcs = ceil_div(r1 - r0, kPiece);
    const int64_t lp0 = (int64_t)(a.pstart[u] >> 32);
    const int64_t seg = ceil_div(pcs, W);
    const int64_t q0 = imin64(pcs, warp * seg), q1 = imin64(pcs, q0 + seg);
    for (int ch = lane; ch < chunks; ch += 32) {
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      int64_t q = q0;
      for (; q + 4 <= q1; q += 4) {  // four loads in flight, summed in order
        float4 x0 = ldg_f4(a.partial + (lp0 + q) * a.d + ch * 4);
        float4 x1 = ldg_f4(a.partial + (lp0 + q + 1) * a.d + ch * 4);
        float4 x2 = ldg_f4(a.partial + (lp0 + q + 2) * a.d + ch * 4);
        float4 x3 = ldg_f4(a.partial + (lp0 + q + 3) * a.d + ch * 4);
        s.x += x0.x; s.y += x0.y; s.z += x0.z; s.w += x0.w;
        s.x += x1.x; s.y += x1.y; s.z += x1.z; s.w += x1.w;
        s.x += x2.x; s.y += x2.y; s.z += x2.z; s.w += x2.w;
        s.x += x3.x; s.y += x3.y; s.z += x3.z; s.w += x3.w;
      }
      for (; q < q1; ++q) {
        float4 x = ldg_f4(a.partial + (lp0 + q) * a.d + ch * 4);
        s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
      }
      *(float4*)(sm + warp * a.d + ch * 4) = s;
    }
    __syncthreads();
    for (int w = W / 2; w > 0; w >>= 1) {  // fixed pairwise tree over the warps
      if (warp < w)
        for (int ch = lane; ch < chunks; ch += 32) {
          float4 x = *(float4*)(sm + warp * a.d + ch * 4);
          float4 y = *(float4*)(sm + (warp + w) * a.d + ch * 4);
          *(float4*)(sm + warp * a.d + ch * 4) = make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
        }
      __syncthreads();
    }
    if (warp == 0)
      for (int ch = lane; ch < chunks; ch += 32) {
        float4 x = *(float4*)(sm + ch * 4);
        float g[4] = {x.x, x.y, x.z, x.w};
        finish_chunk<4>(a, u, ch * 4, g);
      }
    __syncthreads();
  }
}

template <typename WS>
void bwd_layout(WS& ws, int64_t n, int32_t d) {
  const int64_t max_pieces = n + ceil_div(n, kPiece) + 1;
  const int64_t max_long_pieces = 2 * ceil_div(n, kPiece) + 1;
  const int64_t max_long = ceil_div(n, kPiece) + 1;
  ws.template take<uint64_t>((size_t)n);                     // pstart
  ws.template take<uint32_t>((size_t)n);                     // lstart
  ws.template take<uint64_t>(1);                             // ptotal
  ws.template take<uint32_t>(1);                             // ltotal
  ws.template take<int32_t>((size_t)max_pieces);             // piece_u
  ws.template take<int32_t>((size_t)max_long);               // long_list
  ws.template take<float>((size_t)max_long_pieces * d);      // partial sums
  scan_reserve<uint64_t>(ws, n);
}

}  // namespace
}  // namespace ctr

using namespace ctr;

extern "C" size_t ctr_bwd_update_workspace_size(int64_t n_ids, int32_t d) {
  WsSizer s;
  bwd_layout(s, n_ids > 0 ? n_ids : 1, d > 0 ? d : 1);
  return s.used;
}

extern "C" int ctr_embedding_bag_bwd_update(const float* grad_pooled, int64_t g_stride_b, int64_t g_stride_f,
                                            const int64_t* offsets, int32_t num_fields, int32_t batch,
                                            ctr_pool pool, const int64_t* unique_rows, const int64_t* n_unique,
                                            const int32_t* run_offsets, const int32_t* sorted_bag, int64_t n_ids,
                                            float lr, void* table, ctr_dtype dtype, int32_t d, int64_t total_rows,
                                            float* grad_unique_out, void* ws, size_t ws_bytes,
                                            ctr_stream_t stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (!grad_pooled || !offsets || !unique_rows || !n_unique || !run_offsets || !table) return CTR_ERR_INVALID_ARG;
  if (num_fields <= 0 || batch <= 0 || d <= 0 || total_rows <= 0 || n_ids < 0) return CTR_ERR_INVALID_ARG;
  if (n_ids > 0 && !sorted_bag) return CTR_ERR_INVALID_ARG;
  if (dtype != CTR_F32 && dtype != CTR_BF16) return CTR_ERR_INVALID_ARG;
  if (pool != CTR_POOL_SUM && pool != CTR_POOL_MEAN) return CTR_ERR_INVALID_ARG;
  if (g_stride_b < 0 || g_stride_f < 0) return CTR_ERR_INVALID_ARG;
  if (n_ids >= ((int64_t)1 << 31)) return CTR_ERR_UNSUPPORTED;
  if (d % 4 != 0 || d > 512) return CTR_ERR_UNSUPPORTED;
  if (g_stride_b % 4 != 0 || g_stride_f % 4 != 0 || (uintptr_t)grad_pooled % 16 != 0) return CTR_ERR_UNSUPPORTED;
  if (dtype == CTR_F32 && (uintptr_t)table % 16 != 0) return CTR_ERR_UNSUPPORTED;
  if (grad_unique_out && (uintptr_t)grad_unique_out % 16 != 0) return CTR_ERR_UNSUPPORTED;
  if (!ws_valid(ws, ws_bytes, ctr_bwd_update_workspace_size(n_ids, d))) return CTR_ERR_WORKSPACE;
  if (n_ids == 0) return CTR_OK;

  WsCarver c(ws, ws_bytes);
  const int64_t n = n_ids;
  const int64_t max_pieces = n + ceil_div(n, kPiece) + 1;
  const int64_t max_long_pieces = 2 * ceil_div(n, kPiece) + 1;
  const int64_t max_long = ceil_div(n, kPiece) + 1;
  BwdArgs a;
  a.G = grad_pooled;
  a.sb = g_stride_b;
  a.sf = g_stride_f;
  a.offsets = offsets;
  a.B = batch;
  a.mean = pool == CTR_POOL_MEAN;
  a.unique_rows = unique_rows;
  a.n_unique = n_unique;
  a.run_offsets = run_offsets;
  a.sorted_bag = sorted_bag;
  a.lr = lr;
  a.table = table;
  a.bf16 = dtype == CTR_BF16;
  a.d = d;
  a.total_rows = total_rows;
  a.grad_out = grad_unique_out;
  a.err = (int*)ws;
  a.n_cap = n_ids;
  a.nbags = (int64_t)num_fields * batch;
  a.pstart = c.take<uint64_t>(n);
  a.lstart = c.take<uint32_t>(n);
  a.ptotal = c.take<uint64_t>(1);
  a.ltotal = c.take<uint32_t>(1);
  a.piece_u = c.take<int32_t>(max_pieces);
  a.long_list = c.take<int32_t>(max_long);
  a.partial = c.take<float>((size_t)max_long_pieces * d);
  if (!c.ok()) return CTR_ERR_WORKSPACE;
  (void)max_long_pieces;

  const int sms = num_sms();
  const int64_t tb = imin64(ceil_div(n, 256), (int64_t)sms * 8);
  piece_count_kernel<<<(unsigned)tb, 256, 0, s>>>(a, n, a.pstart, a.lstart);
  if (int st = launch_status()) return st;
  {
    WsCarver sc = c;
    if (int st = scan_exclusive<uint64_t>(a.pstart, a.pstart, n, n_unique, a.ptotal, sc, s)) return st;
    WsCarver sc2 = c;
    if (int st = scan_exclusive<uint32_t>(a.lstart, a.lstart, n, n_unique, a.ltotal, sc2, s)) return st;
  }
  expand_kernel<<<(unsigned)tb, 256, 0, s>>>(a, n);
  if (int st = launch_status()) return st;

  const int chunks = d / 4;
  {
    int per_sm = 0;
#define CTR_RED(LPR, CPL)                                                                   \
  {                                                                                         \
    auto k = reduce_pieces_kernel<LPR, CPL>;                                                \
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kRedThreads, 0);              \
    int64_t want = ceil_div(max_pieces, kRedThreads / 32);                                  \
    int64_t g = std::max<int64_t>(1, imin64(want, (int64_t)std::max(per_sm, 1) * sms)); \
    k<<<(unsigned)g, kRedThreads, 0, s>>>(a);                                               \
  }
    if (chunks <= 1) CTR_RED(1, 1)
    else if (chunks <= 2) CTR_RED(2, 1)
    else if (chunks <= 4) CTR_RED(4, 1)
    else if (chunks <= 8) CTR_RED(8, 1)
    else if (chunks <= 16) CTR_RED(16, 1)
    else if (chunks <= 32) CTR_RED(32, 1)
    else if (chunks <= 64) CTR_RED(32, 2)
    else CTR_RED(32, 4)
#undef CTR_RED
    if (int st = launch_status()) return st;
  }
  const size_t smem = (size_t)(kCombThreads / 32) * d * sizeof(float);
  combine_long_kernel<<<(unsigned)std::max(sms * 2, 1), kCombThreads, smem, s>>>(a);
  return launch_status();
}
