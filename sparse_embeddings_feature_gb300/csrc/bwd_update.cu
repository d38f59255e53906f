// a5. Sparse backward: per-unique-row gradient reduce + SGD row update.
//
// Source: "How TensorNet Supercharges Sparse Feature Training on TensorFlow",
// Synchronous Architecture (only the sparse features present in the batch are
// synchronised) and Core Optimizations (the batch-sized matrix of unique rows).
//
// The occurrences of unique u are the sorted slots run_offsets[u] ..
// run_offsets[u+1]-1 (from the dedup); sorted_bag names the bag whose pooled
// gradient each one contributes.  Under Zipf IDs most runs are 1-5 long and a
// few are very long, so the work is split by run length:
//
//   tiles     one warp per tile of TU consecutive uniques.  The tile's short
//             runs (<= kShort occurrences) are contiguous in sorted order; the
//             warp walks their occurrences with kU pooled-gradient rows in
//             flight, summing each run in sorted order into a shared-memory
//             accumulator (fp32).  Then it updates the tile's rows with
//             independent loads (8 rows in flight): the row read-modify-writes
//             do not wait on one another.  Long runs are appended to a list.
//   pieces    a long run is cut into pieces of kPiece occurrences; one warp
//             per piece sums it (same pipelined walk) into a partial row.
//   combine   one CTA per long run: each warp sums a fixed contiguous segment
//             of the run's partials, then a fixed tree over the warps, then
//             the row update.
// Every row is written by exactly one warp or CTA; there are no float atomics,
// and every summation order depends only on the run lengths, so the results
// are deterministic (the long-run list order may vary, but a run's result does
// not depend on where it sits in the list).  The unique rows are sorted
// table-major, so the warps in flight read pooled gradients of one field,
// whose slice stays in L2.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "common.cuh"
#include "scan.cuh"

namespace ctr {
namespace {

constexpr int kShort = 128;        // runs up to this length are summed by the tile kernel
constexpr int kPiece = 128;        // long runs are cut into pieces of this many occurrences
constexpr int kTileThreads = 256;
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kAccFloats = 2048;   // shared accumulator floats per warp (TU * d)
constexpr int kU = 8;              // pooled-gradient rows in flight per warp (for d <= 128)
constexpr int kCombThreads = 256;

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
  int32_t d;           // columns this launch processes
  int32_t ld;          // row stride (elements) of the table, the states and grad_out: d, or more when
                       // the short runs are processed in column slices
  int64_t total_rows;
  float* grad_out;
  int* err;
  // optimizer (CTR_OPT_*): Adagrad sum of squares or Adam m in s0 ([rows, d];
  // [rows] row-wise), Adam v in s1; bc1, bc2 = 1 - beta^step
  int opt;
  float eps, beta1, beta2, bc1, bc2;
  float* s0;
  float* s1;
  int sr;              // bf16 tables: stochastic rounding of the new rows
  uint64_t sr_seed;
  int64_t n_cap;       // occurrences (sorted_bag length)
  int64_t nbags;       // F * B
  int TU;              // uniques per tile
  int g4_ok;           // every pooled-gradient offset / 4 fits 32 bits
  // scratch
  int64_t* long_count;
  unsigned long long* work;  // [2] work counters: tiles, pieces
  int64_t max_long;
  int32_t* long_list;    // [max_long] unique of each long run
  uint32_t* long_pstart; // [max_long] pieces of each long run, then (scanned) its first piece
  uint32_t* pieces_total;
  int32_t* piece_owner;  // [pieces] long-run slot of each piece
  float* partial;        // [pieces, d]
};

__device__ __forceinline__ int64_t n_uniques(const BwdArgs& a) {
  const int64_t n = *a.n_unique;
  return n < a.n_cap ? n : a.n_cap;
}

// Run bounds of unique u; an inconsistent run is flagged and treated as empty,
// so no kernel indexes outside its buffers.
__device__ __forceinline__ void run_bounds(const BwdArgs& a, int64_t u, int64_t& r0, int64_t& r1) {
  r0 = a.run_offsets[u];
  r1 = a.run_offsets[u + 1];
  if (r0 < 0 || r1 < r0 || r1 > a.n_cap) {
    set_error(a.err, CTR_ERR_BAD_OFFSETS);
    r0 = r1 = 0;
  }
}

__device__ __forceinline__ float4 ldg_f4(const float* p) {
  float4 r;
  asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ float4 fma4(float4 x, float s, float4 acc) {
  return make_float4(fmaf(x.x, s, acc.x), fmaf(x.y, s, acc.y), fmaf(x.z, s, acc.z), fmaf(x.w, s, acc.w));
}

// Pooled-gradient offset and scale of sorted occurrence s (-1: contributes nothing).
__device__ __forceinline__ void occ_info(const BwdArgs& a, int64_t s, int64_t& goff, float& scale) {
  const int32_t bag = a.sorted_bag[s];
  if (bag < 0 || bag >= a.nbags) {
    set_error(a.err, CTR_ERR_BAD_OFFSETS);
    goff = -1;
    scale = 0.f;
    return;
  }
  const int32_t f = bag / a.B, b = bag - f * a.B;
  goff = (int64_t)b * a.sb + (int64_t)f * a.sf;
  scale = 1.f;
  if (a.mean) {
    const int64_t len = a.offsets[bag + 1] - a.offsets[bag];
    scale = len > 0 ? 1.f / (float)len : 0.f;
  }
}

// Row update of unique u with gradient chunk g at column 4*ch (w already loaded).
// The step of one value under optimizer OPT (state read-modify-written here):
//   Adagrad  s += g^2,                 step = lr g / (sqrt(s) + eps)
//   row-wise step = lr g * row_inv     (row_inv = 1 / (sqrt(s_row) + eps), from rowwise_inv)
//   Adam     m = b1 m + (1 - b1) g,  v = b2 v + (1 - b2) g^2,
//            step = lr (m / bc1) / (sqrt(v / bc2) + eps)
// The optimizer is a template argument so that the SGD kernels carry none of it.
template <int OPT>
__device__ __forceinline__ float opt_step1(const BwdArgs& a, float g, float& s, float& v, float row_inv) {
  if constexpr (OPT == CTR_OPT_ADAGRAD) {
    s = fmaf(g, g, s);
    return a.lr * g / (sqrtf(s) + a.eps);
  } else if constexpr (OPT == CTR_OPT_ROWWISE_ADAGRAD) {
    return a.lr * g * row_inv;
  } else {
    s = fmaf(1.f - a.beta1, g, a.beta1 * s);
    v = fmaf(1.f - a.beta2, g * g, a.beta2 * v);
    return a.lr * (s / a.bc1) / (sqrtf(v / a.bc2) + a.eps);
  }
}

template <int OPT>
__device__ __forceinline__ float4 opt_step(const BwdArgs& a, float4 g, float4& st, float4& sv, float row_inv) {
  float4 d;
  d.x = opt_step1<OPT>(a, g.x, st.x, sv.x, row_inv);
  d.y = opt_step1<OPT>(a, g.y, st.y, sv.y, row_inv);
  d.z = opt_step1<OPT>(a, g.z, st.z, sv.z, row_inv);
  d.w = opt_step1<OPT>(a, g.w, st.w, sv.w, row_inv);
  return d;
}

template <int OPT>
constexpr int kElemStates = OPT == CTR_OPT_ADAGRAD ? 1 : (OPT == CTR_OPT_ADAM ? 2 : 0);

// Row-wise Adagrad: s_row = s_prev + (sum over the row of g^2) / d and the
// row's 1 / (sqrt(s_row) + eps).  Called by all 32 lanes of a warp with their
// share of the sum of squares and the row's previous state; lane 0 writes it.
__device__ __forceinline__ float rowwise_inv(const BwdArgs& a, int64_t row, float ssq, float s_prev) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(kFull, ssq, o);
  const float s = s_prev + ssq / (float)a.d;
  __syncwarp();  // every lane has read the previous state before lane 0 replaces it
  if ((threadIdx.x & 31) == 0) a.s0[row] = s;
  return 1.f / (sqrtf(s) + a.eps);
}

__device__ __forceinline__ float sumsq4(float4 g) { return fmaf(g.w, g.w, fmaf(g.z, g.z, fmaf(g.y, g.y, g.x * g.x))); }

// Stochastic rounding of x to bf16 bits with 16 random bits u: u is added to
// the 16 bits bf16 drops, and the carry kept (rounds up in magnitude with
// probability equal to the dropped fraction).  Non-finite values and values at
// or beyond the largest finite bf16 round to nearest.
__device__ __forceinline__ uint32_t bf16_sr(float x, uint32_t u) {
  const uint32_t b = __float_as_uint(x);
  const uint32_t mag = b & 0x7fffffffu;
  if (mag >= 0x7f7f0000u) {
    const __nv_bfloat16 r = __float2bfloat16_rn(x);
    return (uint32_t)*(const uint16_t*)&r;
  }
  return ((b & 0x80000000u) | (mag + u)) >> 16;
}

// Store one 4-value chunk of a bf16 row with stochastic rounding: the chunk's
// 64 random bits are splitmix64(seed ^ (row d/4 + chunk)), 16 per value.  Out
// of line: the hash inlined into the unrolled tile loops bloats them.
__device__ __forceinline__ void store_bf16_sr_inl(const BwdArgs& a, int64_t row, int ch, float x0, float x1,
                                                  float x2, float x3) {
  const uint64_t h = splitmix64(a.sr_seed ^ (uint64_t)(row * (a.d / 4) + ch));
  uint2 out;
  out.x = bf16_sr(x0, (uint32_t)h & 0xffffu) | (bf16_sr(x1, (uint32_t)(h >> 16) & 0xffffu) << 16);
  out.y = bf16_sr(x2, (uint32_t)(h >> 32) & 0xffffu) | (bf16_sr(x3, (uint32_t)(h >> 48) & 0xffffu) << 16);
  *(uint2*)((__nv_bfloat16*)a.table + row * a.ld + ch * 4) = out;
}
__device__ __noinline__ void store_bf16_sr(const BwdArgs& a, int64_t row, int ch, float x0, float x1, float x2,
                                           float x3) {
  store_bf16_sr_inl(a, row, ch, x0, x1, x2, x3);
}

// Update one 4-value chunk of a row: w -= step, the elementwise states given
// (st, sv: their previous values) written back.  SR: the build that honours
// stochastic rounding (bf16 tables with a.sr set); without it the store has no
// out-of-line call and the tile loops keep their registers.  xdefer (SR
// builds): the new fp32 values go there, for the caller to round and store
// after its loop, instead of to the table.
template <int OPT, bool SR = false>
__device__ __forceinline__ void store_row_chunk_s(const BwdArgs& a, int64_t row, int64_t u, int ch, float4 g,
                                                  float4 w, uint2 wb, uint64_t pol, float row_inv, float4 st,
                                                  float4 sv, float* xdefer = nullptr) {
  if (a.grad_out) *(float4*)(a.grad_out + u * a.ld + ch * 4) = g;
  // SGD keeps its single fused multiply-add per value
  float4 step = g;
  float k = -a.lr;
  if constexpr (OPT != CTR_OPT_SGD) {
    step = opt_step<OPT>(a, g, st, sv, row_inv);
    k = -1.f;
    const int64_t e = row * a.ld + ch * 4;
    if constexpr (kElemStates<OPT> >= 1) *(float4*)(a.s0 + e) = st;
    if constexpr (kElemStates<OPT> >= 2) *(float4*)(a.s1 + e) = sv;
  }
  if (!a.bf16) {
    float4 x = make_float4(fmaf(k, step.x, w.x), fmaf(k, step.y, w.y), fmaf(k, step.z, w.z), fmaf(k, step.w, w.w));
    float* dst = (float*)a.table + row * a.ld + ch * 4;
    if (pol) stg_f4_policy(dst, x, pol);
    else *(float4*)dst = x;
  } else {
    const float w0 = __uint_as_float(wb.x << 16), w1 = __uint_as_float(wb.x & 0xffff0000u);
    const float w2 = __uint_as_float(wb.y << 16), w3 = __uint_as_float(wb.y & 0xffff0000u);
    const float x0 = fmaf(k, step.x, w0), x1 = fmaf(k, step.y, w1);
    const float x2 = fmaf(k, step.z, w2), x3 = fmaf(k, step.w, w3);
    if (SR && a.sr && xdefer) {
      *(float4*)xdefer = make_float4(x0, x1, x2, x3);
    } else if (SR && a.sr) {
      store_bf16_sr(a, row, ch, x0, x1, x2, x3);
    } else {
      __nv_bfloat162 p0 = __floats2bfloat162_rn(x0, x1);
      __nv_bfloat162 p1 = __floats2bfloat162_rn(x2, x3);
      *(uint2*)((__nv_bfloat16*)a.table + row * a.ld + ch * 4) = make_uint2(*(uint32_t*)&p0, *(uint32_t*)&p1);
    }
  }
}

// store_row_chunk_s as one out-of-line copy: the tile kernel's occurrence loop
// is unrolled 32 times, and an inlined optimizer update in each copy overflows
// the instruction cache.
template <int OPT, bool SR>
__device__ __noinline__ void store_row_chunk_call(const BwdArgs& a, int64_t row, int64_t u, int ch, float4 g,
                                                  float4 w, uint2 wb, uint64_t pol, float row_inv, float4 st,
                                                  float4 sv, float* xdefer) {
  store_row_chunk_s<OPT, SR>(a, row, u, ch, g, w, wb, pol, row_inv, st, sv, xdefer);
}

// The same, reading the elementwise states from global memory.
template <int OPT>
__device__ __forceinline__ void store_row_chunk_t(const BwdArgs& a, int64_t row, int64_t u, int ch, float4 g,
                                                  float4 w, uint2 wb, uint64_t pol, float row_inv) {
  float4 st = make_float4(0.f, 0.f, 0.f, 0.f), sv = make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t e = row * a.ld + ch * 4;
  if constexpr (kElemStates<OPT> >= 1) st = *(const float4*)(a.s0 + e);
  if constexpr (kElemStates<OPT> >= 2) sv = *(const float4*)(a.s1 + e);
  store_row_chunk_s<OPT, true>(a, row, u, ch, g, w, wb, pol, row_inv, st, sv);
}

// The same with the optimizer and the rounding chosen at run time (for the
// kernels off the hot path).
__device__ __forceinline__ void store_row_chunk(const BwdArgs& a, int64_t row, int64_t u, int ch, float4 g,
                                                float4 w, uint2 wb, uint64_t pol = 0, float row_inv = 0.f) {
  switch (a.opt) {
    case CTR_OPT_ADAGRAD: store_row_chunk_t<CTR_OPT_ADAGRAD>(a, row, u, ch, g, w, wb, pol, row_inv); break;
    case CTR_OPT_ROWWISE_ADAGRAD:
      store_row_chunk_t<CTR_OPT_ROWWISE_ADAGRAD>(a, row, u, ch, g, w, wb, pol, row_inv);
      break;
    case CTR_OPT_ADAM: store_row_chunk_t<CTR_OPT_ADAM>(a, row, u, ch, g, w, wb, pol, row_inv); break;
    default: store_row_chunk_t<CTR_OPT_SGD>(a, row, u, ch, g, w, wb, pol, row_inv); break;
  }
}

__device__ __forceinline__ void load_row_chunk(const BwdArgs& a, int64_t row, int ch, float4& w, uint2& wb) {
  if (!a.bf16) w = *(const float4*)((const float*)a.table + row * a.ld + ch * 4);
  else wb = *(const uint2*)((const __nv_bfloat16*)a.table + row * a.ld + ch * 4);
}

// Walk occurrences [s0, s1) of one run, kU rows in flight, summing in order.
template <int CPL>
__device__ __forceinline__ void sum_run(const BwdArgs& a, int64_t s0, int64_t s1, float4 (&acc)[CPL]) {
  constexpr int kU = ::ctr::kU / CPL;
  const int lane = threadIdx.x & 31;
  const int chunks = a.d / 4;
  for (int64_t j0 = s0; j0 < s1; j0 += 32) {
    const int cnt = (int)imin64(32, s1 - j0);
    int64_t goff = -1;
    float scale = 0.f;
    if (lane < cnt) occ_info(a, j0 + lane, goff, scale);
    for (int t0 = 0; t0 < cnt; t0 += kU) {
      float4 buf[kU][CPL];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int t = t0 + u;
        const int64_t go = __shfl_sync(kFull, goff, t & 31);
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const int ch = lane + c * 32;
          buf[u][c] = (t < cnt && go >= 0 && ch < chunks) ? ldg_f4(a.G + go + ch * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const float sc = __shfl_sync(kFull, scale, (t0 + u) & 31);
#pragma unroll
        for (int c = 0; c < CPL; ++c)
          if (t0 + u < cnt) acc[c] = fma4(buf[u][c], sc, acc[c]);
      }
    }
  }
}

template <int CPL>
__global__ void __launch_bounds__(kTileThreads, 2) bwd_tiles_kernel(const BwdArgs a) {
  constexpr int kU = ::ctr::kU / CPL;   // rows in flight in phase 1
  constexpr int kR = 8 / CPL;           // rows in flight in phase 2
  extern __shared__ float4 sacc[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int chunks = a.d / 4;
  const int TU = a.TU;
  float4* my = sacc + (size_t)warp * TU * chunks;
  const int64_t nu = n_uniques(a);
  const int64_t ntiles = ceil_div(nu, TU);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t tile = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; tile < ntiles; tile += nwarps) {
    const int64_t u = tile * TU + lane;
    const bool valid = lane < TU && u < nu;
    int64_t r0 = 0, r1 = 0;
    if (valid) run_bounds(a, u, r0, r1);
    const int64_t len = r1 - r0;
    const bool is_long = valid && len > kShort;
    const bool is_short = valid && !is_long && len > 0;
    int64_t row = -1;
    if (is_short) {
      row = a.unique_rows[u];
      if (row < 0 || row >= a.total_rows) {
        set_error(a.err, CTR_ERR_INDEX_OUT_OF_RANGE);
        row = -1;
      }
    }
    // exclusive scan of the short runs' lengths over the tile's lanes
    const int slen = is_short ? (int)len : 0;
    int inc = slen;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += y;
    }
    const int e = inc - slen;
    const int E = __shfl_sync(kFull, inc, 31);

    // phase 1: per-run sums of the tile's short runs into shared memory
    float4 acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < E; c0 += 32) {
      const int k = c0 + lane;
      int seg = 0;
#pragma unroll
      for (int step = 16; step > 0; step >>= 1) {  // largest lane i with e_i <= k
        const int cand = seg + step;
        const int ec = __shfl_sync(kFull, e, cand);
        if (ec <= k) seg = cand;
      }
      const int64_t r0s = __shfl_sync(kFull, r0, seg);
      const int es = __shfl_sync(kFull, e, seg);
      const int ls = __shfl_sync(kFull, slen, seg);
      int64_t goff = -1;
      float scale = 0.f;
      bool last = false;
      if (k < E) {
        occ_info(a, r0s + (k - es), goff, scale);
        last = (k + 1 == es + ls);
      }
      const int cnt = min(32, E - c0);
      for (int t0 = 0; t0 < cnt; t0 += kU) {
        float4 buf[kU][CPL];
#pragma unroll
        for (int uu = 0; uu < kU; ++uu) {
          const int t = t0 + uu;
          const int64_t go = __shfl_sync(kFull, goff, t & 31);
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const int ch = lane + c * 32;
            buf[uu][c] = (t < cnt && go >= 0 && ch < chunks) ? ldg_f4(a.G + go + ch * 4)
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int uu = 0; uu < kU; ++uu) {
          const int t = (t0 + uu) & 31;
          const float sc = __shfl_sync(kFull, scale, t);
          const bool lf = __shfl_sync(kFull, (int)last, t) != 0;
          const int sg = __shfl_sync(kFull, seg, t);
          if (t0 + uu < cnt) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] = fma4(buf[uu][c], sc, acc[c]);
            if (lf) {
#pragma unroll
              for (int c = 0; c < CPL; ++c) {
                const int ch = lane + c * 32;
                if (ch < chunks) my[sg * chunks + ch] = acc[c];
                acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
              }
            }
          }
        }
      }
    }
    __syncwarp();
    // phase 2: row updates, eight independent rows in flight
    for (int j0 = 0; j0 < TU; j0 += kR) {
      float4 w[kR][CPL];
      uint2 wb[kR][CPL];
      int64_t rj[kR];
#pragma unroll
      for (int jj = 0; jj < kR; ++jj) {
        const int j = (j0 + jj) & 31;
        rj[jj] = __shfl_sync(kFull, row, j);
        const int lj = __shfl_sync(kFull, slen, j);
        if (j0 + jj >= TU || lj == 0) rj[jj] = -1;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const int ch = lane + c * 32;
          if (rj[jj] >= 0 && ch < chunks) load_row_chunk(a, rj[jj], ch, w[jj][c], wb[jj][c]);
        }
      }
#pragma unroll
      for (int jj = 0; jj < kR; ++jj) {
        if (rj[jj] < 0) continue;
        float rinv = 0.f;
        if (a.opt == CTR_OPT_ROWWISE_ADAGRAD) {
          float q = 0.f;
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const int ch = lane + c * 32;
            if (ch < chunks) q += sumsq4(my[(j0 + jj) * chunks + ch]);
          }
          rinv = rowwise_inv(a, rj[jj], q, a.s0[rj[jj]]);
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const int ch = lane + c * 32;
          if (ch < chunks) store_row_chunk(a, rj[jj], tile * TU + j0 + jj, ch, my[(j0 + jj) * chunks + ch], w[jj][c],
                                           wb[jj][c], 0, rinv);
        }
      }
    }
    __syncwarp();
  }
}

// Clears the long-run count and the piece counter (the tile counter belongs
// to the short-run phase, which may run concurrently).
__global__ void clear_long_state(int64_t* long_count, unsigned long long* piece_counter) {
  *long_count = 0;
  *piece_counter = 0;
}

// The long runs (more than kShort occurrences) in ascending unique order (so
// the pieces of one table's runs are processed together and share its
// pooled-gradient rows in L2): per block of kLongChunk uniques a count, an
// exclusive scan of the counts, then each block writes its runs in order.
constexpr int kLongChunk = 2048;  // uniques per block (8 per thread)

__global__ void __launch_bounds__(256) long_count_kernel(const BwdArgs a, uint32_t* __restrict__ counts) {
  __shared__ uint32_t warp_tot[8];
  const int64_t nu = n_uniques(a);
  const int64_t u0 = (int64_t)blockIdx.x * kLongChunk;
  uint32_t c = 0;
#pragma unroll
  for (int q = 0; q < kLongChunk / 256; ++q) {
    const int64_t u = u0 + q * 256 + threadIdx.x;
    if (u < nu) {
      int64_t r0, r1;
      run_bounds(a, u, r0, r1);
      c += (r1 - r0 > kShort) ? 1u : 0u;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
  if ((threadIdx.x & 31) == 0) warp_tot[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int w = 0; w < 8; ++w) t += warp_tot[w];
    counts[blockIdx.x] = t;
  }
}

__global__ void __launch_bounds__(256) long_write_kernel(const BwdArgs a, const uint32_t* __restrict__ starts,
                                                         const uint32_t* __restrict__ total) {
  __shared__ uint32_t warp_tot[8];
  const int64_t nu = n_uniques(a);
  const int64_t u0 = (int64_t)blockIdx.x * kLongChunk + threadIdx.x * (kLongChunk / 256);
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.long_count = *total;
  uint32_t v[kLongChunk / 256];
  int64_t len[kLongChunk / 256];
#pragma unroll
  for (int q = 0; q < kLongChunk / 256; ++q) {  // this thread's consecutive uniques
    const int64_t u = u0 + q;
    len[q] = 0;
    if (u < nu) {
      int64_t r0, r1;
      run_bounds(a, u, r0, r1);
      len[q] = r1 - r0;
    }
    v[q] = len[q] > kShort ? 1u : 0u;
  }
  block_exclusive_scan<uint32_t, 256, kLongChunk / 256>(v, warp_tot);
  const uint32_t base = starts[blockIdx.x];
#pragma unroll
  for (int q = 0; q < kLongChunk / 256; ++q) {
    if (len[q] > kShort) {
      const int64_t slot = (int64_t)base + v[q];
      if (slot < a.max_long) {
        a.long_list[slot] = (int32_t)(u0 + q);
        a.long_pstart[slot] = (uint32_t)ceil_div(len[q], kPiece);
      }
    }
  }
}

__global__ void expand_long_kernel(const BwdArgs a) {
  const int64_t nl = imin64(*a.long_count, a.max_long);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nl; i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r0, r1;
    run_bounds(a, a.long_list[i], r0, r1);
    const int64_t pcs = ceil_div(r1 - r0, kPiece);
    const int64_t p0 = a.long_pstart[i];
    for (int64_t k = 0; k < pcs; ++k) a.piece_owner[p0 + k] = (int32_t)i;
  }
}

// One warp per piece of a long run: its sum goes to partial[piece].  For rows
// of at most 512 bytes the walk streams: sorted_bag is read two chunks ahead
// and the pooled-gradient rows run in a sliding window of kWin loads that
// continues across chunks.
constexpr int kWin = 8;
#ifndef CTR_TILE_ASYNC_MINB
#define CTR_TILE_ASYNC_MINB 3
#endif
// L2 policies of the backward: pooled-gradient rows are re-read by every
// unique of their bags (kept: evict_last on this fraction of their lines),
// table rows are read and written once (streamed: evict_first).
#ifndef CTR_BWD_G_KEEP_FRACTION
#define CTR_BWD_G_KEEP_FRACTION 1.0f
#endif
#ifndef CTR_BWD_ROW_STREAM
#define CTR_BWD_ROW_STREAM 1
#endif
__device__ __forceinline__ uint64_t g_policy() {
  return CTR_BWD_G_KEEP_FRACTION > 0.f ? l2_evict_last_fraction(CTR_BWD_G_KEEP_FRACTION) : l2_evict_normal();
}
__device__ __forceinline__ uint64_t row_policy() { return CTR_BWD_ROW_STREAM ? l2_evict_first() : l2_evict_normal(); }

#ifndef CTR_BWD_MINB
#define CTR_BWD_MINB 8  // piece kernel: resident blocks per SM (full occupancy, 32 registers)
#endif

// Rows wider than 512 bytes: one warp per piece, kU / CPL rows in flight.
template <int CPL>
__global__ void __launch_bounds__(256) long_pieces_kernel(const BwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int chunks = a.d / 4;
  const int64_t np = *a.pieces_total;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t p = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < np; p += nwarps) {
    const int64_t i = a.piece_owner[p];
    int64_t r0, r1;
    run_bounds(a, a.long_list[i], r0, r1);
    const int64_t k = p - (int64_t)a.long_pstart[i];
    const int64_t s0 = r0 + k * kPiece;
    const int64_t s1 = imin64(r1, s0 + kPiece);
    float4 acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    sum_run<CPL>(a, s0, s1, acc);
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int ch = lane + c * 32;
      if (ch < chunks) *(float4*)(a.partial + p * a.d + ch * 4) = acc[c];
    }
  }
}

// Pooled-gradient row of a bag in 16-byte units (kNoG: contributes nothing),
// and its MEAN scale.
constexpr uint32_t kNoG = 0xffffffffu;

__device__ __forceinline__ uint32_t bag_g4(const BwdArgs& a, int32_t bag, float& scale) {
  scale = 0.f;
  if (bag < 0) return kNoG;
  if (bag >= a.nbags) {
    set_error(a.err, CTR_ERR_BAD_OFFSETS);
    return kNoG;
  }
  const int32_t f = bag / a.B, b = bag - f * a.B;
  scale = 1.f;
  if (a.mean) {
    const int64_t len = a.offsets[bag + 1] - a.offsets[bag];
    scale = len > 0 ? 1.f / (float)len : 0.f;
  }
  return (uint32_t)(((int64_t)b * a.sb + (int64_t)f * a.sf) >> 2);
}

// Gradient-row loads in flight per lane in the piece kernel.  The kernel is
// latency-bound (ncu: L2 at half its throughput, 37% of warps active at 3
// blocks per SM with 8 loads each); 2 loads per lane at 8 blocks per SM keep
// more rows in flight per SM and cut it by 29% (4 at 4: 7%; 16 at 2: slower).
#ifndef CTR_PIECE_WIN
#define CTR_PIECE_WIN 2
#endif
constexpr int kPieceWin = CTR_PIECE_WIN;
static_assert(32 % kPieceWin == 0, "the load window must divide the chunk");

__global__ void __launch_bounds__(256, CTR_BWD_MINB) long_pieces_stream_kernel(const BwdArgs a) {
  const int lane = threadIdx.x & 31;
  const bool col = lane * 4 < a.d;  // this lane's 16-byte column exists
  const float* Gl = a.G + lane * 4;
  const uint64_t pol_keep = g_policy();
  const int64_t np = *a.pieces_total;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  (void)nwarps;
  for (int64_t p = next_unit(a.work + 1); p < np; p = next_unit(a.work + 1)) {
    const int64_t i = a.piece_owner[p];
    int64_t r0, r1;
    run_bounds(a, a.long_list[i], r0, r1);
    const int64_t k = p - (int64_t)a.long_pstart[i];
    const int32_t* sb = a.sorted_bag + r0 + k * kPiece;
    const int n = (int)imin64(kPiece, r1 - (r0 + k * kPiece));
    int32_t bag_b = (32 + lane < n) ? sb[32 + lane] : -1;
    float sc_cur;
    uint32_t cur = bag_g4(a, (lane < n) ? sb[lane] : -1, sc_cur);
    float4 buf[kPieceWin];
#pragma unroll
    for (int u = 0; u < kPieceWin; ++u) {
      const uint32_t r = __shfl_sync(kFull, cur, u);
      buf[u] = (r != kNoG && col) ? ldg_f4_policy(Gl + (uint64_t)r * 4, pol_keep) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < n; c0 += 32) {
      const int32_t bag_c = (c0 + 64 + lane < n) ? sb[c0 + 64 + lane] : -1;
      float sc_nxt;
      const uint32_t nxt = bag_g4(a, bag_b, sc_nxt);
      for (int g = 0; g < 32; g += kPieceWin) {
#pragma unroll
        for (int j = 0; j < kPieceWin; ++j) {
          const int t = g + j;
          const float4 x = buf[j];
          const int tn = t + kPieceWin;
          const uint32_t r = __shfl_sync(kFull, tn < 32 ? cur : nxt, tn & 31);
          buf[j] = (r != kNoG && col) ? ldg_f4_policy(Gl + (uint64_t)r * 4, pol_keep) : make_float4(0.f, 0.f, 0.f, 0.f);
          if (a.mean) acc = fma4(x, __shfl_sync(kFull, sc_cur, t), acc);
          else acc = make_float4(acc.x + x.x, acc.y + x.y, acc.z + x.z, acc.w + x.w);
        }
      }
      cur = nxt;
      sc_cur = sc_nxt;
      bag_b = bag_c;
    }
    if (col) *(float4*)(a.partial + p * a.d + lane * 4) = acc;
  }
}

// The same pieces for rows of at most 64 columns: a group of G lanes (one per
// 16-byte column, G = 4, 8 or 16) takes every (32 / G)-th occurrence of the
// piece, so narrow rows keep every lane and more loads busy; each group sums
// its occurrences in order and the groups' partials are added by a fixed
// butterfly (depth at most 128 / (32 / G) + log2(32 / G)).
template <int G>
__global__ void __launch_bounds__(256, CTR_BWD_MINB) long_pieces_grouped_kernel(const BwdArgs a) {
  constexpr int NG = 32 / G;     // occurrences per warp step
  constexpr int STEPS = 32 / NG;  // steps per chunk of 32 occurrences
  static_assert(STEPS % kPieceWin == 0, "the load window must divide a chunk's steps");
  const int lane = threadIdx.x & 31, grp = lane / G, sub = lane % G;
  const bool col = sub * 4 < a.d;
  const float* Gl = a.G + sub * 4;
  const uint64_t pol_keep = g_policy();
  const int64_t np = *a.pieces_total;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t p = next_unit(a.work + 1); p < np; p = next_unit(a.work + 1)) {
    const int64_t i = a.piece_owner[p];
    int64_t r0, r1;
    run_bounds(a, a.long_list[i], r0, r1);
    const int64_t k = p - (int64_t)a.long_pstart[i];
    const int32_t* sb = a.sorted_bag + r0 + k * kPiece;
    const int n = (int)imin64(kPiece, r1 - (r0 + k * kPiece));
    int32_t bag_b = (32 + lane < n) ? sb[32 + lane] : -1;
    float sc_cur;
    uint32_t cur = bag_g4(a, (lane < n) ? sb[lane] : -1, sc_cur);
    float4 buf[kPieceWin];
#pragma unroll
    for (int u = 0; u < kPieceWin; ++u) {
      const uint32_t r = __shfl_sync(kFull, cur, u * NG + grp);
      buf[u] = (r != kNoG && col) ? ldg_f4_policy(Gl + (uint64_t)r * 4, pol_keep) : zero;
    }
    float4 acc = zero;
    for (int c0 = 0; c0 < n; c0 += 32) {
      const int32_t bag_c = (c0 + 64 + lane < n) ? sb[c0 + 64 + lane] : -1;
      float sc_nxt;
      const uint32_t nxt = bag_g4(a, bag_b, sc_nxt);
      for (int g = 0; g < STEPS; g += kPieceWin) {
#pragma unroll
        for (int j = 0; j < kPieceWin; ++j) {
          const int t = (g + j) * NG + grp;  // this group's occurrence in the chunk
          const float4 x = buf[j];
          const int tn = t + kPieceWin * NG;
          const uint32_t r = __shfl_sync(kFull, tn < 32 ? cur : nxt, tn & 31);
          buf[j] = (r != kNoG && col) ? ldg_f4_policy(Gl + (uint64_t)r * 4, pol_keep) : zero;
          if (a.mean) acc = fma4(x, __shfl_sync(kFull, sc_cur, t), acc);
          else acc = make_float4(acc.x + x.x, acc.y + x.y, acc.z + x.z, acc.w + x.w);
        }
      }
      cur = nxt;
      sc_cur = sc_nxt;
      bag_b = bag_c;
    }
#pragma unroll
    for (int o = G; o < 32; o <<= 1) {
      acc.x += __shfl_xor_sync(kFull, acc.x, o);
      acc.y += __shfl_xor_sync(kFull, acc.y, o);
      acc.z += __shfl_xor_sync(kFull, acc.z, o);
      acc.w += __shfl_xor_sync(kFull, acc.w, o);
    }
    if (grp == 0 && col) *(float4*)(a.partial + p * a.d + sub * 4) = acc;
  }
}

// Streaming walk over a tile's short runs (rows of at most 512 bytes): the
// flattened occurrences are resolved 32 at a time (run by shuffle search,
// sorted_bag fetched ahead, one ballot for run ends).
struct TileChunk {
  int32_t bag;     // bag of this lane's occurrence (-1: none)
  int seg;         // run (lane) of the occurrence within the tile
  uint32_t lastm;  // ballot: occurrence t closes its run
};

__device__ __forceinline__ TileChunk tile_chunk(const BwdArgs& a, int kk, int E, int e, int r0, int slen) {
  TileChunk c;
  c.seg = 0;
#pragma unroll
  for (int step = 16; step > 0; step >>= 1) {  // largest lane i with e_i <= kk
    const int cand = c.seg + step;
    if (__shfl_sync(kFull, e, cand) <= kk) c.seg = cand;
  }
  const int es = __shfl_sync(kFull, e, c.seg);
  const int rs = __shfl_sync(kFull, r0, c.seg);
  const int ls = __shfl_sync(kFull, slen, c.seg);
  c.bag = kk < E ? a.sorted_bag[rs + (kk - es)] : -1;
  c.lastm = __ballot_sync(kFull, kk < E && kk + 1 == es + ls);
  return c;
}

// Tile kernel with the table rows staged by cp.async: when a tile starts, each
// lane issues asynchronous copies of its column of the tile's (at most TU)
// rows into the warp's shared memory, so the rows' DRAM reads overlap the
// pooled-gradient stream and hold no registers.  A run is updated at its last
// occurrence, straight from shared memory, and written back at once; there is
// no second phase and no accumulator staging.
__device__ __forceinline__ void cp_async_chunk(uint32_t dst, const void* src, int bytes, uint64_t pol) {
  if (bytes == 16)
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
  else
    asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Shared memory of one warp of the async tile kernel: the tile's TU table rows,
// then the elementwise optimizer states [ns][TU][d] fp32, then with stochastic
// rounding the rows' new values [TU][d] fp32; TU * row bytes is a multiple of
// 16 (the host keeps TU even for bf16 rows of d = 4 mod 8), so every section
// starts on a 16-byte boundary.
constexpr size_t tile_warp_bytes(int TU, int d, int esz, int ns, int xs) {
  return (size_t)TU * d * esz + (size_t)(ns + xs) * TU * d * 4;
}
constexpr int kSrDeferBytes = 4096;  // stochastic rounding: new values held per warp (caps TU)

// Short runs of fp32 rows under SGD, one column slice of every row per launch
// (the host runs one launch per slice).  Why slices: the tile kernel keeps the
// pooled-gradient rows of the table it is working on in L2 (they are re-read
// by every unique of their bags); at the full step's batch one table's
// gradient rows take 67 MB, more than the L2 holds next to the streamed table
// rows, and ncu counted 3.7 GB of re-fetched gradient rows per step.  A slice
// of half the columns halves that footprint.
//
// Each half-warp (16 lanes x 16 bytes = 64 columns) takes every other
// occurrence of the tile's flattened run list: a warp step consumes a pair of
// occurrences, so a slice costs no more instructions per byte than the whole
// row does in the plain kernel.  When a run closes, the two halves' partial
// sums are added (shuffle across the halves) and half 0 updates the row's
// slice, staged in shared memory by cp.async when the tile started.  Each run
// is summed in a fixed order (its even and odd positions in the flattened
// list separately, then the two partials), so the results are deterministic.
#ifndef CTR_PAIR_WIN
#define CTR_PAIR_WIN 4
#endif
#ifndef CTR_PAIR_TU
#define CTR_PAIR_TU 32
#endif
constexpr int kPairWin = CTR_PAIR_WIN;  // occurrence pairs in flight per warp
constexpr int kPairTU = CTR_PAIR_TU;    // uniques per tile
#ifndef CTR_TILE_PAIR_MINB
#define CTR_TILE_PAIR_MINB 3
#endif
#ifndef CTR_PAIR_FAST
#define CTR_PAIR_FAST 1  // a step in which neither occurrence closes its run only adds
#endif
template <bool MEAN>
__global__ void __launch_bounds__(kTileThreads, CTR_TILE_PAIR_MINB) bwd_tiles_pair_kernel(const BwdArgs a) {
  extern __shared__ __align__(16) unsigned char wsm_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = lane >> 4, sub = lane & 15;
  const bool col = sub * 4 < a.d;  // a.d <= 64 columns in this slice
  const int TU = a.TU;
  const int row_bytes = a.d * 4;
  unsigned char* wsm = wsm_raw + (size_t)warp * TU * row_bytes;
  const uint32_t wsm_s = (uint32_t)__cvta_generic_to_shared(wsm);
  const float* Gl = a.G + sub * 4;
  const uint64_t pol_keep = g_policy(), pol_stream = row_policy();
  const int64_t nu = n_uniques(a);
  const int64_t ntiles = ceil_div(nu, TU);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t tile = next_unit(a.work); tile < ntiles; tile = next_unit(a.work)) {
    const int64_t u = tile * TU + lane;
    const bool valid = lane < TU && u < nu;
    int64_t r0 = 0, r1 = 0;
    if (valid) run_bounds(a, u, r0, r1);
    const int64_t len = r1 - r0;
    const bool is_long = valid && len > kShort;
    const bool is_short = valid && !is_long && len > 0;
    int64_t row = -1;
    if (is_short) {
      row = a.unique_rows[u];
      if (row < 0 || row >= a.total_rows) {
        set_error(a.err, CTR_ERR_INDEX_OUT_OF_RANGE);
        row = -1;
      }
    }
    // stage the slices of the tile's rows: half h copies rows h, h + 2, ...
    for (int j0 = 0; j0 < TU; j0 += 2) {
      const int j = j0 + h;
      const int64_t rj = __shfl_sync(kFull, row, j & 31);
      if (j < TU && rj >= 0 && col)
        cp_async_chunk(wsm_s + j * row_bytes + sub * 16, (const float*)a.table + rj * a.ld + sub * 4, 16,
                       pol_stream);
    }
    cp_async_commit();
    const int slen = is_short ? (int)len : 0;
    int inc = slen;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += y;
    }
    const int e = inc - slen;
    const int E = __shfl_sync(kFull, inc, 31);
    const int r0i = (int)r0;

    TileChunk cur = tile_chunk(a, lane, E, e, r0i, slen);
    TileChunk pend = tile_chunk(a, 32 + lane, E, e, r0i, slen);
    float sc_cur;
    uint32_t gcur = bag_g4(a, cur.bag, sc_cur);
    float4 buf[kPairWin];
#pragma unroll
    for (int q = 0; q < kPairWin; ++q) {
      const uint32_t r = __shfl_sync(kFull, gcur, 2 * q + h);
      buf[q] = (r != kNoG && col) ? ldg_f4_policy(Gl + (uint64_t)r * 4, pol_keep) : zero;
    }
    float4 acc = zero;
    bool staged = false;
    // close run `sg` with this half's partial `part`: the halves' partials are
    // added, half 0 updates the slice of the row
    auto finish = [&](int sg, float4 part) {
      float4 tot;
      tot.x = part.x + __shfl_xor_sync(kFull, part.x, 16);
      tot.y = part.y + __shfl_xor_sync(kFull, part.y, 16);
      tot.z = part.z + __shfl_xor_sync(kFull, part.z, 16);
      tot.w = part.w + __shfl_xor_sync(kFull, part.w, 16);
      const int64_t rs = __shfl_sync(kFull, row, sg);
      if (!staged) {  // the slices were staged by both halves: wait for all of them
        cp_async_wait_all();
        __syncwarp();
        staged = true;
      }
      if (h == 0 && rs >= 0 && col) {
        if (a.grad_out) *(float4*)(a.grad_out + (tile * TU + sg) * a.ld + sub * 4) = tot;
        const float4 w = *(const float4*)(wsm + sg * row_bytes + sub * 16);
        const float k = -a.lr;
        stg_f4_policy((float*)a.table + rs * a.ld + sub * 4,
                      make_float4(fmaf(k, tot.x, w.x), fmaf(k, tot.y, w.y), fmaf(k, tot.z, w.z), fmaf(k, tot.w, w.w)),
                      pol_stream);
      }
    };
    for (int c0 = 0; c0 < E; c0 += 32) {
      const TileChunk ahead = tile_chunk(a, c0 + 64 + lane, E, e, r0i, slen);
      float sc_nxt;
      const uint32_t gnxt = bag_g4(a, pend.bag, sc_nxt);
      for (int g = 0; g < 16; g += kPairWin) {
#pragma unroll
        for (int j = 0; j < kPairWin; ++j) {
          const int q = g + j;
          const int t0 = 2 * q, t1 = 2 * q + 1;
          const float4 x = buf[j];
          const int tn = 2 * (q + kPairWin) + h;  // refill the slot with pair q + kPairWin
          const uint32_t r = __shfl_sync(kFull, tn < 32 ? gcur : gnxt, tn & 31);
          buf[j] = (r != kNoG && col) ? ldg_f4_policy(Gl + (uint64_t)r * 4, pol_keep) : zero;
          const bool v0 = c0 + t0 < E, v1 = c0 + t1 < E;
          if (!v0) continue;  // warp-uniform: the chunk's tail
          const float sc = MEAN ? __shfl_sync(kFull, sc_cur, 2 * q + h) : 1.f;
          if (CTR_PAIR_FAST && v1 && ((cur.lastm >> t0) & 3u) == 0u) {
            // neither occurrence closes its run, so both belong to the open one
            acc = MEAN ? fma4(x, sc, acc) : make_float4(acc.x + x.x, acc.y + x.y, acc.z + x.z, acc.w + x.w);
            continue;
          }
          const int seg0 = __shfl_sync(kFull, cur.seg, t0), seg1 = __shfl_sync(kFull, cur.seg, t1);
          const bool last1 = v1 && ((cur.lastm >> t1) & 1u);
          if (v1 && seg0 == seg1) {  // both occurrences belong to one run
            acc = MEAN ? fma4(x, sc, acc) : make_float4(acc.x + x.x, acc.y + x.y, acc.z + x.z, acc.w + x.w);
            if (last1) {
              finish(seg1, acc);
              acc = zero;
            }
          } else {  // occurrence t0 closes its run; t1 (if any) starts the next one
            float4 mine = acc;
            if (h == 0) mine = MEAN ? fma4(x, sc, acc) : make_float4(acc.x + x.x, acc.y + x.y, acc.z + x.z, acc.w + x.w);
            finish(seg0, mine);
            acc = zero;
            if (v1) {
              if (h == 1) acc = MEAN ? fma4(x, sc, zero) : x;
              if (last1) {
                finish(seg1, acc);
                acc = zero;
              }
            }
          }
        }
      }
      cur = pend;
      pend = ahead;
      gcur = gnxt;
      sc_cur = sc_nxt;
    }
    cp_async_wait_all();  // nothing may land in the buffer after the next tile reuses it
    __syncwarp();
  }
}

// Optimizers with state run at 2 blocks per SM: the state arithmetic needs the
// registers, and the staged states the shared memory.
#ifndef CTR_TILE_OPT_MINB
#define CTR_TILE_OPT_MINB 2
#endif
constexpr int kOptStageBytes = 12288;  // staged bytes per warp (rows and states) with an optimizer
template <int OPT, bool SR>
__global__ void __launch_bounds__(kTileThreads, OPT == CTR_OPT_SGD ? CTR_TILE_ASYNC_MINB : CTR_TILE_OPT_MINB)
    bwd_tiles_async_kernel(const BwdArgs a) {
  extern __shared__ __align__(16) unsigned char wsm_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool col = lane * 4 < a.d;
  const int TU = a.TU;
  const int esz = a.bf16 ? 2 : 4;
  const int row_bytes = a.d * esz;
  const int chunk = 4 * esz;  // this lane's 4 elements
  // per warp: the tile's table rows, then its elementwise optimizer states (fp32)
  constexpr int NS = kElemStates<OPT>;
  const int state_bytes = a.d * 4;
  constexpr int XS = SR ? 1 : 0;
  unsigned char* wsm = wsm_raw + (size_t)warp * TU * (row_bytes + (NS + XS) * state_bytes);
  const uint32_t wsm_s = (uint32_t)__cvta_generic_to_shared(wsm);
  unsigned char* ssm = wsm + (size_t)TU * row_bytes;  // state s of unique j: ssm + (s * TU + j) * state_bytes
  float* xsm = (float*)(ssm + NS * TU * state_bytes);  // new values of unique j: xsm + j * d
  const uint32_t ssm_s = (uint32_t)__cvta_generic_to_shared(ssm);
  const float* Gl = a.G + lane * 4;
  // pooled-gradient rows are re-read by every unique of their bags: keep them
  // in L2; the table rows are touched once: stream them
  const uint64_t pol_keep = g_policy(), pol_stream = row_policy();
  const int64_t nu = n_uniques(a);
  const int64_t ntiles = ceil_div(nu, TU);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  (void)nwarps;
  for (int64_t tile = next_unit(a.work); tile < ntiles; tile = next_unit(a.work)) {
    const int64_t u = tile * TU + lane;
    const bool valid = lane < TU && u < nu;
    int64_t r0 = 0, r1 = 0;
    if (valid) run_bounds(a, u, r0, r1);
    const int64_t len = r1 - r0;
    const bool is_long = valid && len > kShort;
    const bool is_short = valid && !is_long && len > 0;
    int64_t row = -1;
    if (is_short) {
      row = a.unique_rows[u];
      if (row < 0 || row >= a.total_rows) {
        set_error(a.err, CTR_ERR_INDEX_OUT_OF_RANGE);
        row = -1;
      }
    }
    // stage this tile's table rows and states (each lane its own column)
    for (int j = 0; j < TU; ++j) {
      const int64_t rj = __shfl_sync(kFull, row, j);
      if (rj >= 0 && col) {
        cp_async_chunk(wsm_s + j * row_bytes + lane * chunk,
                       (const char*)a.table + (rj * a.ld) * esz + lane * chunk, chunk, pol_stream);
        if constexpr (NS >= 1)
          cp_async_chunk(ssm_s + j * state_bytes + lane * 16, a.s0 + rj * a.ld + lane * 4, 16, pol_stream);
        if constexpr (NS >= 2)
          cp_async_chunk(ssm_s + (TU + j) * state_bytes + lane * 16, a.s1 + rj * a.ld + lane * 4, 16, pol_stream);
      }
    }
    cp_async_commit();
    float s_row = 0.f;  // row-wise Adagrad: the state of this lane's unique, fetched while the tile streams
    if constexpr (OPT == CTR_OPT_ROWWISE_ADAGRAD) {
      if (row >= 0) s_row = a.s0[row];
    }
    const int slen = is_short ? (int)len : 0;
    int inc = slen;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += y;
    }
    const int e = inc - slen;
    const int E = __shfl_sync(kFull, inc, 31);
    const int r0i = (int)r0;

    TileChunk cur = tile_chunk(a, lane, E, e, r0i, slen);
    TileChunk pend = tile_chunk(a, 32 + lane, E, e, r0i, slen);
    float sc_cur;
    uint32_t gcur = bag_g4(a, cur.bag, sc_cur);
    float4 buf[kWin];
#pragma unroll
    for (int q = 0; q < kWin; ++q) {
      const uint32_t r = __shfl_sync(kFull, gcur, q);
      buf[q] = (r != kNoG && col) ? ldg_f4_policy(Gl + (uint64_t)r * 4, pol_keep) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    bool staged = false;
    for (int c0 = 0; c0 < E; c0 += 32) {
      const TileChunk ahead = tile_chunk(a, c0 + 64 + lane, E, e, r0i, slen);
      float sc_nxt;
      const uint32_t gnxt = bag_g4(a, pend.bag, sc_nxt);
      for (int g = 0; g < 32; g += kWin) {
#pragma unroll
        for (int j = 0; j < kWin; ++j) {
          const int t = g + j;
          const float4 x = buf[j];
          const int tn = t + kWin;
          const uint32_t r = __shfl_sync(kFull, tn < 32 ? gcur : gnxt, tn & 31);
          buf[j] = (r != kNoG && col) ? ldg_f4_policy(Gl + (uint64_t)r * 4, pol_keep) : make_float4(0.f, 0.f, 0.f, 0.f);
          if (a.mean) acc = fma4(x, __shfl_sync(kFull, sc_cur, t), acc);
          else acc = make_float4(acc.x + x.x, acc.y + x.y, acc.z + x.z, acc.w + x.w);
          if ((cur.lastm >> t) & 1u) {
            const int sg = __shfl_sync(kFull, cur.seg, t);
            const int64_t rs = __shfl_sync(kFull, row, sg);
            float rinv = 0.f;
            if constexpr (OPT == CTR_OPT_ROWWISE_ADAGRAD) {
              const float sp = __shfl_sync(kFull, s_row, sg);
              if (rs >= 0) rinv = rowwise_inv(a, rs, col ? sumsq4(acc) : 0.f, sp);
            }
            if (rs >= 0 && col) {
              if (!staged) {
                cp_async_wait_all();  // this lane's own copies only: no warp barrier needed
                staged = true;
              }
              const unsigned char* wp = wsm + sg * row_bytes + lane * chunk;
              float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
              uint2 wb = make_uint2(0u, 0u);
              if (!a.bf16) w = *(const float4*)wp;
              else wb = *(const uint2*)wp;
              float4 st = make_float4(0.f, 0.f, 0.f, 0.f), sv = make_float4(0.f, 0.f, 0.f, 0.f);
              if constexpr (NS >= 1) st = *(const float4*)(ssm + sg * state_bytes + lane * 16);
              if constexpr (NS >= 2) sv = *(const float4*)(ssm + (TU + sg) * state_bytes + lane * 16);
              // the elementwise optimizers' updates (a divide and a square root per value) out of line
              if constexpr (OPT == CTR_OPT_ADAGRAD || OPT == CTR_OPT_ADAM)
                store_row_chunk_call<OPT, SR>(a, rs, tile * TU + sg, lane, acc, w, wb, pol_stream, rinv, st, sv,
                                              SR ? xsm + sg * a.d + lane * 4 : nullptr);
              else
                store_row_chunk_s<OPT, SR>(a, rs, tile * TU + sg, lane, acc, w, wb, pol_stream, rinv, st, sv,
                                           SR ? xsm + sg * a.d + lane * 4 : nullptr);
            }
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
      cur = pend;
      pend = ahead;
      gcur = gnxt;
      sc_cur = sc_nxt;
    }
    if constexpr (SR) {
      // the tile's new rows, rounded and stored outside the unrolled loop, with
      // every lane busy: 32 / (d/4) rows per round, one column chunk per lane
      __syncwarp();  // the chunks written above by other lanes
      const int chunks = a.d >> 2;
      const int rpi = 32 / chunks;
      const int jl = lane / chunks, ch = lane - jl * chunks;
      for (int j0 = 0; j0 < TU; j0 += rpi) {
        const int j = j0 + jl;
        const int64_t rj = __shfl_sync(kFull, row, j < 32 ? j : 0);
        if (jl < rpi && j < TU && rj >= 0) {
          const float4 x = *(const float4*)(xsm + j * a.d + ch * 4);
          store_bf16_sr_inl(a, rj, ch, x.x, x.y, x.z, x.w);
        }
      }
    }
    cp_async_wait_all();  // nothing may land in the buffer after the next tile reuses it
    __syncwarp();
  }
}

// Long runs of at most kCombWarpPieces pieces (most of them: a run of up to
// 4096 occurrences) are finished by one warp each, summing the run's partials
// in order with several loads in flight, then updating the row; no block
// barrier.  Longer runs (the Zipf head) take a CTA each (combine_long_kernel).
constexpr int kCombWarpPieces = 32;
__global__ void __launch_bounds__(256) combine_short_kernel(const BwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int chunks = a.d / 4;
  const int64_t nl = imin64(*a.long_count, a.max_long);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < nl; i += nwarps) {
    const int64_t u = a.long_list[i];
    int64_t r0, r1;
    run_bounds(a, u, r0, r1);
    const int64_t pcs = ceil_div(r1 - r0, kPiece);
    if (pcs > kCombWarpPieces) continue;  // warp-uniform: a CTA finishes it
    const int64_t p0 = a.long_pstart[i];
    const int64_t row = a.unique_rows[u];
    if (row < 0 || row >= a.total_rows) {
      if (lane == 0) set_error(a.err, CTR_ERR_INDEX_OUT_OF_RANGE);
      continue;
    }
    for (int ch = lane; ch < chunks; ch += 32) {
      float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
      int64_t q = 0;
      for (; q + 4 <= pcs; q += 4) {  // four loads in flight, summed in order
        const float4 x0 = ldg_f4(a.partial + (p0 + q) * a.d + ch * 4);
        const float4 x1 = ldg_f4(a.partial + (p0 + q + 1) * a.d + ch * 4);
        const float4 x2 = ldg_f4(a.partial + (p0 + q + 2) * a.d + ch * 4);
        const float4 x3 = ldg_f4(a.partial + (p0 + q + 3) * a.d + ch * 4);
        s4 = fma4(x0, 1.f, s4);
        s4 = fma4(x1, 1.f, s4);
        s4 = fma4(x2, 1.f, s4);
        s4 = fma4(x3, 1.f, s4);
      }
      for (; q < pcs; ++q) s4 = fma4(ldg_f4(a.partial + (p0 + q) * a.d + ch * 4), 1.f, s4);
      float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
      uint2 wb = make_uint2(0u, 0u);
      if (a.opt != CTR_OPT_ROWWISE_ADAGRAD) {
        load_row_chunk(a, row, ch, w, wb);
        store_row_chunk(a, row, u, ch, s4, w, wb, 0, 0.f);
      }
    }
  }
}

// One CTA per long run of more than kCombWarpPieces pieces (all long runs for
// row-wise Adagrad, whose row state needs the whole row): its 8 warps sum
// fixed contiguous segments of its partials, then a fixed pairwise tree over
// the warps (3 levels), then the row update.  (CTAs of 32 warps shorten the
// longest runs' chains but fit one per SM: 0.28 against 0.13 ms.)
__global__ void __launch_bounds__(kCombThreads) combine_long_kernel(const BwdArgs a) {
  constexpr int W = kCombThreads / 32;
  extern __shared__ float sm[];  // [W][d]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int chunks = a.d / 4;
  const int64_t nl = imin64(*a.long_count, a.max_long);
  for (int64_t i = blockIdx.x; i < nl; i += gridDim.x) {
    const int64_t u = a.long_list[i];
    int64_t r0, r1;
    run_bounds(a, u, r0, r1);
    const int64_t pcs = ceil_div(r1 - r0, kPiece);
    if (pcs <= kCombWarpPieces && a.opt != CTR_OPT_ROWWISE_ADAGRAD) continue;  // block-uniform: a warp finished it
    const int64_t p0 = a.long_pstart[i];
    const int64_t seg = ceil_div(pcs, W);
    const int64_t q0 = imin64(pcs, warp * seg), q1 = imin64(pcs, q0 + seg);
    for (int ch = lane; ch < chunks; ch += 32) {
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      int64_t q = q0;
      for (; q + 4 <= q1; q += 4) {  // four loads in flight, summed in order
        const float4 x0 = ldg_f4(a.partial + (p0 + q) * a.d + ch * 4);
        const float4 x1 = ldg_f4(a.partial + (p0 + q + 1) * a.d + ch * 4);
        const float4 x2 = ldg_f4(a.partial + (p0 + q + 2) * a.d + ch * 4);
        const float4 x3 = ldg_f4(a.partial + (p0 + q + 3) * a.d + ch * 4);
        s = fma4(x0, 1.f, s);
        s = fma4(x1, 1.f, s);
        s = fma4(x2, 1.f, s);
        s = fma4(x3, 1.f, s);
      }
      for (; q < q1; ++q) s = fma4(ldg_f4(a.partial + (p0 + q) * a.d + ch * 4), 1.f, s);
      *(float4*)(sm + warp * a.d + ch * 4) = s;
    }
    __syncthreads();
    for (int w = W / 2; w > 0; w >>= 1) {
      if (warp < w)
        for (int ch = lane; ch < chunks; ch += 32) {
          const float4 x = *(float4*)(sm + warp * a.d + ch * 4);
          const float4 y = *(float4*)(sm + (warp + w) * a.d + ch * 4);
          *(float4*)(sm + warp * a.d + ch * 4) = make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
        }
      __syncthreads();
    }
    if (warp == 0) {
      const int64_t row = a.unique_rows[u];
      if (row < 0 || row >= a.total_rows) {
        if (lane == 0) set_error(a.err, CTR_ERR_INDEX_OUT_OF_RANGE);
      } else {
        float rinv = 0.f;
        if (a.opt == CTR_OPT_ROWWISE_ADAGRAD) {
          float q = 0.f;
          for (int ch = lane; ch < chunks; ch += 32) q += sumsq4(*(float4*)(sm + ch * 4));
          rinv = rowwise_inv(a, row, q, a.s0[row]);
        }
        for (int ch = lane; ch < chunks; ch += 32) {
          float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
          uint2 wb = make_uint2(0u, 0u);
          load_row_chunk(a, row, ch, w, wb);
          store_row_chunk(a, row, u, ch, *(float4*)(sm + ch * 4), w, wb, 0, rinv);
        }
      }
    }
    __syncthreads();
  }
}

struct Sizes {
  int64_t max_long, max_pieces;
};

Sizes sizes(int64_t n) {
  Sizes z;
  z.max_long = n / (kShort + 1) + 1;
  z.max_pieces = n / kPiece + z.max_long + 1;
  return z;
}

template <typename WS>
void bwd_layout(WS& ws, int64_t n, int32_t d) {
  const Sizes z = sizes(n);
  ws.template take<int64_t>(1);                            // long_count
  ws.template take<unsigned long long>(2);                 // work counters
  ws.template take<uint32_t>(1);                           // pieces_total
  ws.template take<int32_t>((size_t)z.max_long);           // long_list
  ws.template take<uint32_t>((size_t)z.max_long);          // long_pstart
  ws.template take<int32_t>((size_t)z.max_pieces);         // piece_owner
  ws.template take<float>((size_t)z.max_pieces * d);       // partial sums
  const int64_t blocks = std::max<int64_t>(1, ceil_div(n, (int64_t)kLongChunk));
  ws.template take<uint32_t>((size_t)blocks);              // long runs per block of uniques, then their scan
  ws.template take<uint32_t>(1);                           // their total
  scan_reserve<uint32_t>(ws, blocks);
  scan_reserve<uint32_t>(ws, z.max_long);
}

template <typename K>
int grid_of(K kernel, int threads, size_t smem, int64_t want) {
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
  return (int)std::max<int64_t>(1, imin64(want, (int64_t)std::max(per_sm, 1) * num_sms()));
}

// Short runs of fp32 rows under SGD in column slices (bwd_tiles_pair_kernel):
// 0 = automatic (rows of at most 64 columns always; d = 128 when one table's
// pooled-gradient rows, batch x 512 bytes, exceed 32 MB and would not stay in
// L2), 1 = never, 2 = always where supported.  Process-wide
// (ctr_set_tile_slices).
std::atomic<int> g_tile_slices{0};
constexpr int64_t kSliceGradBytes = (int64_t)32 << 20;

bool use_pair_slices(const BwdArgs& a) {
  if (a.opt != CTR_OPT_SGD || a.sr || a.bf16 || !a.g4_ok) return false;
  if (a.d != 128 && !(a.d <= 64 && a.d % 4 == 0)) return false;
  const int mode = g_tile_slices.load();
  if (mode == 1) return false;
  if (mode == 2) return true;
  // rows of at most 64 columns are one slice: two occurrences per warp step
  // keep twice the lanes of the plain kernel busy
  return a.d <= 64 || (int64_t)a.B * a.d * 4 > kSliceGradBytes;
}

// The short-run pass: the tile kernel once, or the pair kernel once per
// 64-column slice.
template <typename K>
int launch_tiles(const BwdArgs& a, K tk, size_t tile_smem, cudaStream_t s, int64_t n) {
  if (use_pair_slices(a)) {
    auto pk = a.mean ? bwd_tiles_pair_kernel<true> : bwd_tiles_pair_kernel<false>;
    for (int c0 = 0; c0 < a.d; c0 += 64) {
      BwdArgs b = a;
      b.d = std::min(64, a.d - c0);
      b.ld = a.d;
      b.table = (float*)a.table + c0;
      b.G = a.G + c0;
      if (a.grad_out) b.grad_out = a.grad_out + c0;
      b.TU = kPairTU;
      const size_t smem = (size_t)kTileWarps * b.TU * b.d * 4;
      if (smem > 48 * 1024 &&
          cudaFuncSetAttribute(pk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return CTR_ERR_CUDA;
      if (cudaMemsetAsync(a.work, 0, sizeof(unsigned long long), s) != cudaSuccess) return CTR_ERR_CUDA;
      pk<<<grid_of(pk, kTileThreads, smem, ceil_div(n, (int64_t)b.TU * kTileWarps)), kTileThreads, smem, s>>>(b);
      count_launch();
      if (int st = launch_status()) return st;
    }
    return CTR_OK;
  }
  if (cudaMemsetAsync(a.work, 0, sizeof(unsigned long long), s) != cudaSuccess) return CTR_ERR_CUDA;
  tk<<<grid_of(tk, kTileThreads, tile_smem, ceil_div(n, (int64_t)a.TU * kTileWarps)), kTileThreads, tile_smem, s>>>(a);
  count_launch();
  return launch_status();
}

template <int CPL>
int launch_short(const BwdArgs& a, cudaStream_t s, int64_t n) {
  const int chunks = a.d / 4;
  const size_t acc_smem = (size_t)kTileWarps * a.TU * chunks * sizeof(float4);
  const bool use_async = CPL == 1 && a.g4_ok;
  auto async_k = a.sr ? (a.opt == CTR_OPT_ADAGRAD           ? bwd_tiles_async_kernel<CTR_OPT_ADAGRAD, true>
                         : a.opt == CTR_OPT_ROWWISE_ADAGRAD ? bwd_tiles_async_kernel<CTR_OPT_ROWWISE_ADAGRAD, true>
                         : a.opt == CTR_OPT_ADAM            ? bwd_tiles_async_kernel<CTR_OPT_ADAM, true>
                                                            : bwd_tiles_async_kernel<CTR_OPT_SGD, true>)
                      : (a.opt == CTR_OPT_ADAGRAD           ? bwd_tiles_async_kernel<CTR_OPT_ADAGRAD, false>
                         : a.opt == CTR_OPT_ROWWISE_ADAGRAD ? bwd_tiles_async_kernel<CTR_OPT_ROWWISE_ADAGRAD, false>
                         : a.opt == CTR_OPT_ADAM            ? bwd_tiles_async_kernel<CTR_OPT_ADAM, false>
                                                            : bwd_tiles_async_kernel<CTR_OPT_SGD, false>);
  auto tk = use_async ? async_k : bwd_tiles_kernel<CPL>;
  const int ns = a.opt == CTR_OPT_ADAGRAD ? 1 : (a.opt == CTR_OPT_ADAM ? 2 : 0);
  if (use_async && ((size_t)a.TU * a.d * (a.bf16 ? 2 : 4)) % 16 != 0) return CTR_ERR_UNSUPPORTED;  // layout rule
  const size_t tile_smem =
      use_async ? (size_t)kTileWarps * tile_warp_bytes(a.TU, a.d, a.bf16 ? 2 : 4, ns, a.sr ? 1 : 0) : acc_smem;
  if (tile_smem > 48 * 1024 &&
      cudaFuncSetAttribute(tk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tile_smem) != cudaSuccess)
    return CTR_ERR_CUDA;
  timing_mark(CTR_KERNEL_BWD_TILES, true, s);
  if (int st = launch_tiles(a, tk, tile_smem, s, n)) return st;
  timing_mark(CTR_KERNEL_BWD_TILES, false, s);
  return launch_status();
}

template <int CPL>
int launch_long(const BwdArgs& a, WsCarver& c, cudaStream_t s, int64_t n) {
  clear_long_state<<<1, 1, 0, s>>>(a.long_count, a.work + 1); count_launch();
  if (int st = launch_status()) return st;
  {
    // blocks cover the host bound on n_unique (the ID count); blocks past the
    // device count find no uniques
    const int64_t blocks = std::max<int64_t>(1, ceil_div(n, (int64_t)kLongChunk));
    WsCarver lc = c;
    uint32_t* counts = lc.take<uint32_t>((size_t)blocks);
    uint32_t* total = lc.take<uint32_t>(1);
    if (!lc.ok()) return CTR_ERR_WORKSPACE;
    long_count_kernel<<<(unsigned)blocks, 256, 0, s>>>(a, counts); count_launch();
    if (int st = launch_status()) return st;
    if (int st = scan_exclusive<uint32_t>(counts, counts, blocks, nullptr, total, lc, s)) return st;
    long_write_kernel<<<(unsigned)blocks, 256, 0, s>>>(a, counts, total); count_launch();
    if (int st = launch_status()) return st;
    c = lc;  // the scan below carves after these
  }
  {
    WsCarver sc = c;
    if (int st = scan_exclusive<uint32_t>(a.long_pstart, a.long_pstart, a.max_long, a.long_count, a.pieces_total,
                                          sc, s))
      return st;
  }
  expand_long_kernel<<<std::max(1, num_sms() * 2), 256, 0, s>>>(a); count_launch();
  if (int st = launch_status()) return st;
  timing_mark(CTR_KERNEL_BWD_PIECES, true, s);
  if (CPL == 1 && a.g4_ok && a.d <= 64) {
    auto pk = a.d <= 16 ? long_pieces_grouped_kernel<4>
              : a.d <= 32 ? long_pieces_grouped_kernel<8> : long_pieces_grouped_kernel<16>;
    pk<<<grid_of(pk, 256, 0, ceil_div(sizes(n).max_pieces, 8)), 256, 0, s>>>(a); count_launch();
  } else if (CPL == 1 && a.g4_ok) {
    auto pk = long_pieces_stream_kernel;
    pk<<<grid_of(pk, 256, 0, ceil_div(sizes(n).max_pieces, 8)), 256, 0, s>>>(a); count_launch();
  } else {
    auto pk = long_pieces_kernel<CPL>;
    pk<<<grid_of(pk, 256, 0, ceil_div(sizes(n).max_pieces, 8)), 256, 0, s>>>(a); count_launch();
  }
  timing_mark(CTR_KERNEL_BWD_PIECES, false, s);
  return launch_status();
}

int launch_finish(const BwdArgs& a, cudaStream_t s) {
  const size_t csmem = (size_t)(kCombThreads / 32) * a.d * sizeof(float);
  if (csmem > 48 * 1024 &&
      cudaFuncSetAttribute(combine_long_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem) != cudaSuccess)
    return CTR_ERR_CUDA;
  // one CTA per long run in flight, as many as fit (each run is a short latency chain)
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_long_kernel, kCombThreads, csmem) != cudaSuccess)
    per_sm = 2;
  const int64_t cgrid = imin64(std::max<int64_t>(a.max_long, 1), (int64_t)std::max(per_sm, 1) * num_sms());
  if (a.opt != CTR_OPT_ROWWISE_ADAGRAD) {
    int per_sm_w = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_w, combine_short_kernel, 256, 0) != cudaSuccess)
      per_sm_w = 4;
    const int64_t wgrid = imin64(std::max<int64_t>(ceil_div(a.max_long, (int64_t)8), 1),
                                 (int64_t)std::max(per_sm_w, 1) * num_sms());
    combine_short_kernel<<<(unsigned)wgrid, 256, 0, s>>>(a); count_launch();
    if (int st = launch_status()) return st;
  }
  combine_long_kernel<<<(unsigned)cgrid, kCombThreads, csmem, s>>>(a); count_launch();
  return launch_status();
}

}  // namespace
}  // namespace ctr

using namespace ctr;

extern "C" int ctr_set_tile_slices(int mode) { return g_tile_slices.exchange(mode < 0 || mode > 2 ? 0 : mode); }

extern "C" size_t ctr_bwd_update_workspace_size(int64_t n_ids, int32_t d) {
  WsSizer s;
  bwd_layout(s, n_ids > 0 ? n_ids : 1, d > 0 ? d : 1);
  return s.used;
}

namespace {

// Validates the arguments, fills the kernels' arguments and runs the phases
// in `phases` (CTR_BWD_SHORT_RUNS, CTR_BWD_LONG_RUNS, CTR_BWD_FINISH, in this
// order) on s.
int bwd_update_phases(const float* grad_pooled, int64_t g_stride_b, int64_t g_stride_f, const int64_t* offsets,
                      int32_t num_fields, int32_t batch, ctr_pool pool, const int64_t* unique_rows,
                      const int64_t* n_unique, const int32_t* run_offsets, const int32_t* sorted_bag, int64_t n_ids,
                      float lr, void* table, ctr_dtype dtype, int32_t d, int64_t total_rows, float* grad_unique_out,
                      int phases, const ctr_optimizer* opt, void* ws, size_t ws_bytes, cudaStream_t s) {
  const int kind = opt ? opt->kind : CTR_OPT_SGD;
  if (kind < CTR_OPT_SGD || kind > CTR_OPT_ADAM) return CTR_ERR_INVALID_ARG;
  if (kind != CTR_OPT_SGD && (!opt->state0 || (uintptr_t)opt->state0 % 16 != 0 || !(opt->eps > 0.f)))
    return CTR_ERR_INVALID_ARG;
  if (kind == CTR_OPT_ADAM &&
      (!opt->state1 || (uintptr_t)opt->state1 % 16 != 0 || opt->step < 1 || !(opt->beta1 >= 0.f && opt->beta1 < 1.f) ||
       !(opt->beta2 >= 0.f && opt->beta2 < 1.f)))
    return CTR_ERR_INVALID_ARG;
  if (!grad_pooled || !offsets || !unique_rows || !n_unique || !run_offsets || !table) return CTR_ERR_INVALID_ARG;
  if (num_fields <= 0 || batch <= 0 || d <= 0 || total_rows <= 0 || n_ids < 0) return CTR_ERR_INVALID_ARG;
  if (n_ids > 0 && !sorted_bag) return CTR_ERR_INVALID_ARG;
  if (dtype != CTR_F32 && dtype != CTR_BF16) return CTR_ERR_INVALID_ARG;
  if (pool != CTR_POOL_SUM && pool != CTR_POOL_MEAN) return CTR_ERR_INVALID_ARG;
  if (phases <= 0 || phases > (CTR_BWD_LONG_RUNS | CTR_BWD_SHORT_RUNS | CTR_BWD_FINISH)) return CTR_ERR_INVALID_ARG;
  if (g_stride_b < 0 || g_stride_f < 0) return CTR_ERR_INVALID_ARG;
  if (n_ids >= ((int64_t)1 << 31)) return CTR_ERR_UNSUPPORTED;
  if (d % 4 != 0 || d > 512) return CTR_ERR_UNSUPPORTED;
  if (g_stride_b % 4 != 0 || g_stride_f % 4 != 0 || (uintptr_t)grad_pooled % 16 != 0) return CTR_ERR_UNSUPPORTED;
  if ((uintptr_t)table % (dtype == CTR_F32 ? 16 : 8) != 0) return CTR_ERR_UNSUPPORTED;
  if (grad_unique_out && (uintptr_t)grad_unique_out % 16 != 0) return CTR_ERR_UNSUPPORTED;
  if (!ws_valid(ws, ws_bytes, ctr_bwd_update_workspace_size(n_ids, d))) return CTR_ERR_WORKSPACE;
  if (n_ids == 0) return CTR_OK;

  WsCarver c(ws, ws_bytes);
  const Sizes z = sizes(n_ids);
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
  a.ld = d;
  a.total_rows = total_rows;
  a.grad_out = grad_unique_out;
  a.err = (int*)ws;
  a.opt = kind;
  a.eps = opt ? opt->eps : 0.f;
  a.beta1 = opt ? opt->beta1 : 0.f;
  a.beta2 = opt ? opt->beta2 : 0.f;
  a.bc1 = kind == CTR_OPT_ADAM ? (float)(1.0 - std::pow((double)opt->beta1, (double)opt->step)) : 1.f;
  a.bc2 = kind == CTR_OPT_ADAM ? (float)(1.0 - std::pow((double)opt->beta2, (double)opt->step)) : 1.f;
  a.s0 = kind != CTR_OPT_SGD ? opt->state0 : nullptr;
  a.s1 = kind == CTR_OPT_ADAM ? opt->state1 : nullptr;
  a.sr = (opt && opt->stochastic_rounding && dtype == CTR_BF16) ? 1 : 0;
  a.sr_seed = opt ? opt->sr_seed : 0;
  a.n_cap = n_ids;
  a.nbags = (int64_t)num_fields * batch;
  {
    // uniques per tile: the tile kernel stages the tile's rows and elementwise
    // states in kAccFloats * 4 bytes of shared memory per warp
    const int ns = kind == CTR_OPT_ADAGRAD ? 1 : (kind == CTR_OPT_ADAM ? 2 : 0);
    const int staged = d * (dtype == CTR_BF16 ? 2 : 4) + ns * d * 4;
    const int budget = kind == CTR_OPT_SGD ? kAccFloats * 4 : kOptStageBytes;
    a.TU = std::max(1, std::min({32, kAccFloats / d, budget / staged}));
    if (a.sr) a.TU = std::max(1, std::min(a.TU, kSrDeferBytes / (d * 4)));
    // the async tile kernel's per-warp sections start on 16-byte boundaries:
    // TU rows of bf16 with d = 4 (mod 8) take an even TU
    if (dtype == CTR_BF16 && d % 8 != 0 && a.TU > 1) a.TU &= ~1;
  }
  {
    const int64_t max_off = (int64_t)(batch - 1) * g_stride_b + (int64_t)(num_fields - 1) * g_stride_f + d;
    a.g4_ok = (max_off >> 2) < (int64_t)0xffffffffll && n_ids < ((int64_t)1 << 31);
  }
  a.long_count = c.take<int64_t>(1);
  a.work = c.take<unsigned long long>(2);
  a.pieces_total = c.take<uint32_t>(1);
  a.max_long = z.max_long;
  a.long_list = c.take<int32_t>(z.max_long);
  a.long_pstart = c.take<uint32_t>(z.max_long);
  a.piece_owner = c.take<int32_t>(z.max_pieces);
  a.partial = c.take<float>((size_t)z.max_pieces * d);
  if (!c.ok()) return CTR_ERR_WORKSPACE;
  const int cpl = (int)ceil_div(d / 4, 32);
  // short runs first: the long runs' pieces then find many pooled-gradient rows in L2
  if (phases & CTR_BWD_SHORT_RUNS) {
    const int st = cpl <= 1 ? launch_short<1>(a, s, n_ids)
                 : cpl <= 2 ? launch_short<2>(a, s, n_ids) : launch_short<4>(a, s, n_ids);
    if (st) return st;
  }
  if (phases & CTR_BWD_LONG_RUNS) {
    const int st = cpl <= 1 ? launch_long<1>(a, c, s, n_ids)
                 : cpl <= 2 ? launch_long<2>(a, c, s, n_ids) : launch_long<4>(a, c, s, n_ids);
    if (st) return st;
  }
  if (phases & CTR_BWD_FINISH) return launch_finish(a, s);
  return CTR_OK;
}

}  // namespace

extern "C" int ctr_embedding_bag_bwd_update(const float* grad_pooled, int64_t g_stride_b, int64_t g_stride_f,
                                            const int64_t* offsets, int32_t num_fields, int32_t batch,
                                            ctr_pool pool, const int64_t* unique_rows, const int64_t* n_unique,
                                            const int32_t* run_offsets, const int32_t* sorted_bag, int64_t n_ids,
                                            float lr, void* table, ctr_dtype dtype, int32_t d, int64_t total_rows,
                                            float* grad_unique_out, void* ws, size_t ws_bytes,
                                            ctr_stream_t stream) {
  return bwd_update_phases(grad_pooled, g_stride_b, g_stride_f, offsets, num_fields, batch, pool, unique_rows,
                           n_unique, run_offsets, sorted_bag, n_ids, lr, table, dtype, d, total_rows, grad_unique_out,
                           CTR_BWD_SHORT_RUNS | CTR_BWD_LONG_RUNS | CTR_BWD_FINISH, nullptr, ws, ws_bytes,
                           (cudaStream_t)stream);
}

extern "C" int ctr_embedding_bag_bwd_update_phases(const float* grad_pooled, int64_t g_stride_b, int64_t g_stride_f,
                                                   const int64_t* offsets, int32_t num_fields, int32_t batch,
                                                   ctr_pool pool, const int64_t* unique_rows,
                                                   const int64_t* n_unique, const int32_t* run_offsets,
                                                   const int32_t* sorted_bag, int64_t n_ids, float lr, void* table,
                                                   ctr_dtype dtype, int32_t d, int64_t total_rows,
                                                   float* grad_unique_out, int phases, void* ws, size_t ws_bytes,
                                                   ctr_stream_t stream) {
  return bwd_update_phases(grad_pooled, g_stride_b, g_stride_f, offsets, num_fields, batch, pool, unique_rows,
                           n_unique, run_offsets, sorted_bag, n_ids, lr, table, dtype, d, total_rows, grad_unique_out,
                           phases, nullptr, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int ctr_embedding_bag_bwd_update_opt(const float* grad_pooled, int64_t g_stride_b, int64_t g_stride_f,
                                                const int64_t* offsets, int32_t num_fields, int32_t batch,
                                                ctr_pool pool, const int64_t* unique_rows, const int64_t* n_unique,
                                                const int32_t* run_offsets, const int32_t* sorted_bag, int64_t n_ids,
                                                float lr, void* table, ctr_dtype dtype, int32_t d, int64_t total_rows,
                                                float* grad_unique_out, int phases, const ctr_optimizer* opt, void* ws,
                                                size_t ws_bytes, ctr_stream_t stream) {
  if (!opt) return CTR_ERR_INVALID_ARG;
  return bwd_update_phases(grad_pooled, g_stride_b, g_stride_f, offsets, num_fields, batch, pool, unique_rows,
                           n_unique, run_offsets, sorted_bag, n_ids, lr, table, dtype, d, total_rows, grad_unique_out,
                           phases, opt, ws, ws_bytes, (cudaStream_t)stream);
}
