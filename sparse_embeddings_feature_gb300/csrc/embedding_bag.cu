// a2. Pooled embedding-bag forward, and the unique-row gather.
//
// Sources: "DHEN" notes, section 2.1 (a trainable d-vector per categorical
// term) and section 3.1, Solution 2 (sum the active embeddings); "Meta DLRM",
// section 02; "How TensorNet ...", Core Optimizations (the batch-sized matrix of
// unique rows).
//
// GPU design: one warp per bag (grid-stride over field-major bags, so the
// warps in flight all read one table and its Zipf-hot rows stay in L2).  A row
// is read as 16-byte vectors by LPR lanes (LPR = row bytes / 16, rounded up to a
// power of two); a warp therefore has 32/LPR rows in flight per step, and the
// loop is unrolled kUnroll steps deep so each lane keeps several independent
// loads outstanding.  Indices are fetched 32 at a time with one coalesced load
// and broadcast by shuffle.  Accumulation is fp32 in a fixed order (each lane
// group sums its rows in index order; groups combine by a fixed butterfly).
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "tma.cuh"

namespace ctr {
namespace {

constexpr int kBagThreads = 256;
constexpr int kUnroll = 4;

template <typename TT>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int kN = 4;
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
};

__device__ __forceinline__ uint4 ldg16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ void unpack(const uint4& v, float (&f)[4], float) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[8], __nv_bfloat16) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Store n consecutive fp32 values as fp32 or bf16 (round to nearest even).
__device__ __forceinline__ void store_out(void* out, int64_t off, const float* v, int n, bool bf16, bool vec_ok) {
  if (!bf16) {
    float* o = (float*)out + off;
    if (vec_ok && n == 4) {
      *(float4*)o = make_float4(v[0], v[1], v[2], v[3]);
    } else if (vec_ok && n == 2) {
      *(float2*)o = make_float2(v[0], v[1]);
    } else if (vec_ok && n == 8) {
      ((float4*)o)[0] = make_float4(v[0], v[1], v[2], v[3]);
      ((float4*)o)[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      for (int i = 0; i < n; ++i) o[i] = v[i];
    }
  } else {
    __nv_bfloat16* o = (__nv_bfloat16*)out + off;
    if (vec_ok && n == 8) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 p = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        w[i] = *(uint32_t*)&p;
      }
      *(uint4*)o = make_uint4(w[0], w[1], w[2], w[3]);
    } else if (vec_ok && n == 4) {
      __nv_bfloat162 p0 = __floats2bfloat162_rn(v[0], v[1]);
      __nv_bfloat162 p1 = __floats2bfloat162_rn(v[2], v[3]);
      *(uint2*)o = make_uint2(*(uint32_t*)&p0, *(uint32_t*)&p1);
    } else if (vec_ok && n == 2) {
      *(__nv_bfloat162*)o = __floats2bfloat162_rn(v[0], v[1]);
    } else {
      for (int i = 0; i < n; ++i) o[i] = __float2bfloat16_rn(v[i]);
    }
  }
}

struct BagArgs {
  const void* table;
  int32_t d;
  int32_t ld;      // row stride of the table in elements (d, or more for a column slice)
  int64_t total_rows;
  const void* idx;
  int64_t n_idx;
  const int64_t* offsets;
  int32_t F, B;
  int mapped;      // indices are table-local IDs of the field's table
  int mean;
  void* out;
  int out_bf16;
  int vec_out;     // output vectors are 16-byte aligned
  int64_t sb, sf;
  int* err;
  float* fm_out;   // optional: FM second-order term per bag (bag-major), or null
};

// LPR lanes per row, CPL 16-byte chunks per lane (rows wider than 32 chunks).
// Resident blocks per SM the register budget of the one-chunk-per-lane
// instantiations is sized for (more warps hide more row-load latency: bf16
// d = 64 gathers 7% faster at 5 than unbounded at 4); wider rows keep their
// registers, which at that budget would spill.
#ifndef CTR_BAG_MINB
#define CTR_BAG_MINB 5
#endif
template <typename TT, int LPR, int CPL, typename IT>
__global__ void __launch_bounds__(kBagThreads, CPL == 1 ? CTR_BAG_MINB : 1) bag_fwd_kernel(
    const BagArgs a, const __grid_constant__ FieldMap fm) {
  constexpr int V = Vec<TT>::kN;
  constexpr int R = 32 / LPR;  // rows per warp step
  const int lane = threadIdx.x & 31;
  const int grp = lane / LPR, sub = lane % LPR;
  const int chunks = a.d / V;  // 16-byte chunks per row
  const int64_t nbags = (int64_t)a.F * a.B;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const TT* table = (const TT*)a.table;
  const IT* idx = (const IT*)a.idx;
  for (int64_t bag = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; bag < nbags; bag += nwarps) {
    const int f = (int)(bag / a.B);
    const int b = (int)(bag - (int64_t)f * a.B);
    int64_t o0 = a.offsets[bag], o1 = a.offsets[bag + 1];
    const int64_t base = a.mapped ? fm.base[f] : 0;
    const int64_t nrows = a.mapped ? fm.rows[f] : a.total_rows;
    float acc[CPL][V];
    float sq = 0.f;  // this lane's share of the sum of squared row entries (FM term)
#pragma unroll
    for (int c = 0; c < CPL; ++c)
#pragma unroll
      for (int v = 0; v < V; ++v) acc[c][v] = 0.f;
    if (o0 < 0 || o1 < o0 || o1 > a.n_idx) {
      if (lane == 0) set_error(a.err, CTR_ERR_BAD_OFFSETS);
      o0 = o1 = 0;
    }
    for (int64_t j0 = o0; j0 < o1; j0 += 32) {
      const int cnt = (int)imin64(32, o1 - j0);
      int64_t row = -1;
      if (lane < cnt) {
        int64_t id = (int64_t)idx[j0 + lane];
        if (id < 0 || id >= nrows) set_error(a.err, CTR_ERR_INDEX_OUT_OF_RANGE);
        else row = base + id;
      }
      for (int t0 = 0; t0 < cnt; t0 += R * kUnroll) {
        uint4 buf[kUnroll][CPL];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int t = t0 + u * R + grp;
          const int64_t r = __shfl_sync(kFull, row, t & 31);
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const int ch = sub + c * LPR;
            if (t < cnt && r >= 0 && ch < chunks) buf[u][c] = ldg16(table + r * a.d + (int64_t)ch * V);
            else buf[u][c] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            float x[V];
            unpack(buf[u][c], x, TT());
#pragma unroll
            for (int v = 0; v < V; ++v) acc[c][v] += x[v];
            if (a.fm_out) {
#pragma unroll
              for (int v = 0; v < V; ++v) sq = fmaf(x[v], x[v], sq);
            }
          }
      }
    }
    // combine the R lane groups (fixed butterfly order)
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
      for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int v = 0; v < V; ++v) acc[c][v] += __shfl_xor_sync(kFull, acc[c][v], o);
    if (a.fm_out) {  // 1/2 (|sum v|^2 - sum |v|^2), from the bag's raw sum
      float s2 = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int v = 0; v < V; ++v) s2 = fmaf(acc[c][v], acc[c][v], s2);
      if (grp != 0) s2 = 0.f;  // every lane group holds the whole sum: count one
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        s2 += __shfl_xor_sync(kFull, s2, o);
        sq += __shfl_xor_sync(kFull, sq, o);
      }
      if (lane == 0) a.fm_out[bag] = 0.5f * (s2 - sq);
    }
    if (a.mean) {
      const int64_t len = o1 - o0;
#pragma unroll
      for (int c = 0; c < CPL; ++c)
#pragma unroll
        for (int v = 0; v < V; ++v) acc[c][v] = len > 0 ? acc[c][v] / (float)len : 0.f;
    }
    if (grp == 0) {
      const int64_t ob = (int64_t)b * a.sb + (int64_t)f * a.sf;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int ch = sub + c * LPR;
        if (ch < chunks) store_out(a.out, ob + (int64_t)ch * V, acc[c], V, a.out_bf16, a.vec_out);
      }
    }
  }
}

// 512-byte fp32 rows (d = 128): one warp walks 32 consecutive bags as one
// flattened list of occurrences (their index ranges are contiguous in CSR).
// Per chunk of 32 occurrences the lanes resolve, in parallel, the bag of each
// occurrence (binary search over the bags' first offsets by shuffle) and its
// 32-bit row; one ballot marks the occurrences that close a bag.  Indices are
// fetched two chunks ahead, and the row loads run in a sliding window kWinF
// deep that continues across bag and chunk boundaries, so a bag boundary never
// drains the pipeline.  Per occurrence the warp spends one shuffle (the row),
// one 16-byte load per lane and four adds.  Each bag is summed in the order of
// its indices; at its last occurrence the warp stores the row.
// Table-row loads in flight per lane, and resident blocks per SM the register
// budget is sized for: 2 loads at 8 blocks per SM (32 registers).  Alone the
// kernel is within 2% of 8 loads at 4 blocks, and in the full training step,
// where the dedup runs beside it on a side stream, the step is 0.9% faster
// (measured twice); 8 loads at 3 blocks was 10% slower alone.  A small batch
// gives too few 32-bag blocks to fill the GPU (DLRM's 2048 samples: 1664
// warps): there each warp's chain of row loads is the bound, and 8 loads at 2
// blocks per SM gathered 0.140 -> 0.097 ms (4 at 4: 0.116 ms).
constexpr int kWinSmall = 8, kMinbSmall = 2;
constexpr int64_t kSmallGridBlocks = 64;  // 32-bag blocks per SM below which the deeper window is used
#ifndef CTR_FLAT_WIN
#define CTR_FLAT_WIN 2
#endif
constexpr int kWinF = CTR_FLAT_WIN;
// The TMA gather variant is off unless selected (ctr_set_tma_gather): measured
// slower than the register window on GB300.
std::atomic<int> g_tma_gather{0};
constexpr uint32_t kNoRow = 0xffffffffu;
#ifndef CTR_FLAT_MINB
#define CTR_FLAT_MINB 8
#endif

// Cache handling of the flat gather's loads (a build-time choice; full-step
// gather times in the same sessions):
//   0  IDs and table rows with the default policy (3.30 ms);
//   1  IDs streamed (L1 no-allocate, L2 evict-first), table rows L2
//      evict-last (3.24 ms, twice);
//   2  IDs streamed, table rows with the default policy (3.28 ms);
//   3  as 1, and table rows not allocated in L1 (the default: 3.21 ms against
//      3.25 for 1): the Zipf head's L1 hits save nothing, so keeping hot rows
//      on chip (L1 or shared memory) does not pay for this gather;
//   4  as 1, with table rows L1 evict-last (3.27 ms).
#ifndef CTR_FLAT_POLICY
#define CTR_FLAT_POLICY 3
#endif
template <typename IT>
__device__ __forceinline__ IT ld_id(const IT* p, uint64_t pol) {
  if constexpr (CTR_FLAT_POLICY == 0) {
    (void)pol;
    return *p;
  } else if constexpr (sizeof(IT) == 8) {
    unsigned long long v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u64 %0, [%1], %2;" : "=l"(v) : "l"(p), "l"(pol));
    return (IT)v;
  } else {
    unsigned v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
    return (IT)v;
  }
}
__device__ __forceinline__ float4 ld_row16(const float* p, uint64_t pol) {
  if constexpr (CTR_FLAT_POLICY == 1 || CTR_FLAT_POLICY == 2) {
    if constexpr (CTR_FLAT_POLICY == 1) return ldg_f4_policy(p, pol);
    return *(const float4*)p;
  }
  if constexpr (CTR_FLAT_POLICY == 3) {  // rows not kept in L1
    float4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p), "l"(pol));
    return r;
  }
  if constexpr (CTR_FLAT_POLICY == 4) {  // rows kept in L1 as long as possible
    float4 r;
    asm volatile("ld.global.nc.L1::evict_last.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p), "l"(pol));
    return r;
  }
  (void)pol;
  return *(const float4*)p;
}

struct FlatChunk {
  uint32_t row;    // global row of this lane's occurrence, kNoRow if none
  uint32_t lastm;  // ballot: occurrence t closes its bag
  int seg;         // bag (lane) of this lane's occurrence within the block
};

template <typename IT>
__device__ __forceinline__ FlatChunk flat_chunk(const BagArgs& a, int kr, IT id, int rel0, int rel1, uint32_t base,
                                                uint32_t nrows) {
  FlatChunk m;
  m.seg = 0;
#pragma unroll
  for (int step = 16; step > 0; step >>= 1) {  // largest lane j with rel0_j <= kr
    const int cand = m.seg + step;
    if (__shfl_sync(kFull, rel0, cand) <= kr) m.seg = cand;
  }
  const uint32_t bs = __shfl_sync(kFull, base, m.seg);
  const uint32_t nr = __shfl_sync(kFull, nrows, m.seg);
  const int r1 = __shfl_sync(kFull, rel1, m.seg);
  m.row = kNoRow;
  bool last = false;
  if (kr < r1) {
    const int64_t v = (int64_t)id;
    if (v < 0 || v >= (int64_t)nr) set_error(a.err, CTR_ERR_INDEX_OUT_OF_RANGE);
    else m.row = bs + (uint32_t)v;
    last = (kr + 1 == r1);
  }
  m.lastm = __ballot_sync(kFull, last);
  return m;
}

// With FM, each lane also sums the squares of its columns of the rows, and at a
// bag's last occurrence the warp reduces |sum v|^2 and sum |v|^2 of the bag
// and stores 1/2 (|sum v|^2 - sum |v|^2).
template <typename IT, bool FM, int WIN = kWinF, int MINB = CTR_FLAT_MINB>
__global__ void __launch_bounds__(kBagThreads, MINB) bag_fwd_flat_kernel(const BagArgs a,
                                                                      const __grid_constant__ FieldMap fm) {
  static_assert(32 % WIN == 0, "the load window must divide the chunk");
  const int lane = threadIdx.x & 31;
  const int64_t nbags = (int64_t)a.F * a.B;
  const int64_t nblk = ceil_div(nbags, 32);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const IT* idx = (const IT*)a.idx;
  const float* table = (const float*)a.table + lane * 4;
  const int64_t end_all = a.offsets[nbags];
  const uint64_t pol_stream = l2_evict_first();  // pooled outputs are written once
  const uint64_t pol_rows = l2_evict_last();
  unsigned long long* counter = (unsigned long long*)((char*)a.err + kWsCounterOffset);
  (void)nwarps;
  for (int64_t blk = next_unit(counter); blk < nblk; blk = next_unit(counter)) {
    const int64_t bag = blk * 32 + lane;
    const bool bvalid = bag < nbags;
    int64_t o0 = bvalid ? a.offsets[bag] : end_all;
    int64_t o1 = bvalid ? a.offsets[bag + 1] : end_all;
    const bool bad = o0 < 0 || o1 < o0 || o1 > a.n_idx;
    const int f = bvalid ? (int)(bag / a.B) : 0;
    const int b = bvalid ? (int)(bag - (int64_t)f * a.B) : 0;
    const int64_t ooff = (int64_t)b * a.sb + (int64_t)f * a.sf + lane * 4;
    const float lenf = (float)(o1 - o0);
    const int64_t S0 = __shfl_sync(kFull, o0, 0);
    const int64_t S1 = __shfl_sync(kFull, o1, 31);
    if (__any_sync(kFull, bad) || S1 - S0 >= ((int64_t)1 << 30)) {
      if (lane == 0) set_error(a.err, CTR_ERR_BAD_OFFSETS);
      o0 = o1 = S0;  // write this block as zeros
    }
    unsigned empty = __ballot_sync(kFull, bvalid && o1 == o0);  // empty bags produce zero rows
    while (empty) {
      const int j = __ffs(empty) - 1;
      empty &= empty - 1;
      const float z[4] = {0.f, 0.f, 0.f, 0.f};
      store_out(a.out, __shfl_sync(kFull, ooff, j) - j * 4 + lane * 4, z, 4, a.out_bf16, a.vec_out);
    }
    if (FM && bvalid && o1 == o0) a.fm_out[bag] = 0.f;
    if (__all_sync(kFull, o1 == o0)) continue;
    const int rel0 = (int)(o0 - S0), rel1 = (int)(o1 - S0);
    const uint32_t base = a.mapped ? (uint32_t)fm.base[f] : 0u;
    const uint32_t nrows = a.mapped ? (uint32_t)fm.rows[f] : (uint32_t)a.total_rows;
    const int total = (int)(S1 - S0);

    const IT* ib = idx + S0;
    IT id_b = (32 + lane < total) ? ld_id(ib + 32 + lane, pol_stream) : IT(0);
    FlatChunk cur = flat_chunk(a, lane, (lane < total) ? ld_id(ib + lane, pol_stream) : IT(0), rel0, rel1, base, nrows);
    float4 buf[WIN];
#pragma unroll
    for (int u = 0; u < WIN; ++u) {
      const uint32_t r = __shfl_sync(kFull, cur.row, u);
      buf[u] = (r != kNoRow) ? ld_row16(table + (uint64_t)r * 128, pol_rows) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float sq = 0.f;
    for (int c0 = 0; c0 < total; c0 += 32) {
      const IT id_c = (c0 + 64 + lane < total) ? ld_id(ib + c0 + 64 + lane, pol_stream) : IT(0);
      const FlatChunk nxt = flat_chunk(a, c0 + 32 + lane, id_b, rel0, rel1, base, nrows);
      for (int g = 0; g < 32; g += WIN) {
#pragma unroll
        for (int j = 0; j < WIN; ++j) {
          const int t = g + j;
          const float4 x = buf[j];
          const int tn = t + WIN;  // refill the slot with occurrence tn
          const uint32_t r = __shfl_sync(kFull, tn < 32 ? cur.row : nxt.row, tn & 31);
          buf[j] = (r != kNoRow) ? ld_row16(table + (uint64_t)r * 128, pol_rows) : make_float4(0.f, 0.f, 0.f, 0.f);
          acc = add4_packed(acc, x);
          if (FM) sq = fmaf(x.w, x.w, fmaf(x.z, x.z, fmaf(x.y, x.y, fmaf(x.x, x.x, sq))));
          if ((cur.lastm >> t) & 1u) {
            const int jb = __shfl_sync(kFull, cur.seg, t);
            if (FM) {
              float s2 = fmaf(acc.w, acc.w, fmaf(acc.z, acc.z, fmaf(acc.y, acc.y, acc.x * acc.x)));
              float q = sq;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) {
                s2 += __shfl_xor_sync(kFull, s2, o);
                q += __shfl_xor_sync(kFull, q, o);
              }
              if (lane == 0) a.fm_out[blk * 32 + jb] = 0.5f * (s2 - q);
              sq = 0.f;
            }
            const int64_t oj = __shfl_sync(kFull, ooff, jb) - jb * 4 + lane * 4;
            float v[4] = {acc.x, acc.y, acc.z, acc.w};
            if (a.mean) {  // a closed bag is never empty
              const float lj = __shfl_sync(kFull, lenf, jb);
              v[0] /= lj;
              v[1] /= lj;
              v[2] /= lj;
              v[3] /= lj;
            }
            if (!a.out_bf16 && a.vec_out) stg_f4_policy((float*)a.out + oj, make_float4(v[0], v[1], v[2], v[3]), pol_stream);
            else store_out(a.out, oj, v, 4, a.out_bf16, a.vec_out);
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
      cur = nxt;
      id_b = id_c;
    }
  }
}

// Narrow rows (2 to 16 chunks of 16 bytes: bf16 d = 16..128, fp32 d = 8..64):
// the flattened walk of bag_fwd_flat_kernel with several rows per warp step.
// A lane group of G = chunks lanes holds one row; the NG = 32 / G groups of a
// warp take NG consecutive occurrences of the block's flattened list per step,
// with a window of kNarrowWin steps of row loads in flight that continues
// across bag and chunk boundaries (so a bag end never drains the pipeline, and
// short bags cost no more than long ones).  Each group sums the occurrences it
// takes of the open bag; when the bag closes, the groups' partials are added
// in a fixed tree: a reduce-scatter where each lane's V columns split evenly
// over the groups (each group then divides, for a mean, and stores its share
// of the row: fewer shuffles, adds and divisions than a butterfly), else a
// butterfly after which group 0 stores the row.  A step in which no bag closes
// (told by the chunk's bag-end mask, the same for the whole warp) only adds
// its rows.  Every bag's summation order depends only on the bag lengths, so
// results are deterministic.  With
// FM, each lane also sums the squares of its columns of the rows it takes; at
// a bag's close both sums are reduced the same way and lane 0 stores
// 1/2 (|sum v|^2 - sum |v|^2) (exactly 0 for a one-ID bag: both terms then
// round identically).
// Repeated IDs (a build-time option, off): within each chunk of 32
// occurrences, the occurrences of one bag that name the same row can be merged
// (match.any on bag and row; the first loads the row and adds it times the
// count, the others load nothing).  Under Zipf IDs a bag often repeats its
// hottest rows (about 28% of the lookups of the bf16 workload's bags of ~30
// IDs at alpha = 1.2), but those are L1/L2 hits, and the match costs more than
// they do: bf16 workload 1.26 -> 1.34 ms, TensorNet pooling 0.258 -> 0.301 ms.
#ifndef CTR_NARROW_WIN
#define CTR_NARROW_WIN 4
#endif
#ifndef CTR_NARROW_MINB
#define CTR_NARROW_MINB 4
#endif
constexpr int kNarrowWin = CTR_NARROW_WIN;
#ifndef CTR_USE_NARROW
#define CTR_USE_NARROW 1
#endif
#ifndef CTR_NARROW_MERGE
#define CTR_NARROW_MERGE 0
#endif
#ifndef CTR_NARROW_FAST
#define CTR_NARROW_FAST 1
#endif
#ifndef CTR_NARROW_SCATTER
#define CTR_NARROW_SCATTER 1
#endif
constexpr bool kNarrowFast = CTR_NARROW_FAST;

// Merge the repeats of (bag, row) among a chunk's occurrences: returns this
// occurrence's weight (the group's size for its first occurrence, 0 for the
// others, whose row becomes kNoRow so they load nothing).
__device__ __forceinline__ float merge_repeats(FlatChunk& m) {
  if (!CTR_NARROW_MERGE) return 1.f;
  const unsigned long long key =
      m.row == kNoRow ? ~0ull : (((unsigned long long)(unsigned)m.seg << 32) | (unsigned long long)m.row);
  const unsigned peers = __match_any_sync(kFull, key);
  const int lane = threadIdx.x & 31;
  if (m.row == kNoRow) return 0.f;
  if (__ffs(peers) - 1 != lane) {
    m.row = kNoRow;
    return 0.f;
  }
  return (float)__popc(peers);
}

template <typename TT, int G, typename IT, bool FM>
__global__ void __launch_bounds__(kBagThreads, CTR_NARROW_MINB) bag_fwd_narrow_kernel(
    const BagArgs a, const __grid_constant__ FieldMap fm) {
  constexpr int V = Vec<TT>::kN;  // elements per 16-byte chunk
  constexpr int NG = 32 / G;      // rows per warp step
  constexpr int STEPS = 32 / NG;  // steps per chunk of 32 occurrences
  constexpr unsigned kStepMask = (1u << NG) - 1u;  // a step's occurrences in a chunk's masks
  static_assert(STEPS % kNarrowWin == 0, "the load window must divide a chunk's steps");
  // without FM, a closing bag's sums are reduce-scattered over the groups (each group divides and
  // stores V / NG of each lane's columns) where the columns split evenly; else summed by a
  // butterfly into every group and stored by group 0
  constexpr bool kScatter = !FM && (V % NG == 0) && CTR_NARROW_SCATTER;
  constexpr int VG = kScatter ? V / NG : V;
  const int lane = threadIdx.x & 31;
  const int grp = lane / G, sub = lane % G;
  const int64_t nbags = (int64_t)a.F * a.B;
  const int64_t nblk = ceil_div(nbags, 32);
  const IT* idx = (const IT*)a.idx;
  const TT* table = (const TT*)a.table + sub * V;
  const int64_t end_all = a.offsets[nbags];
  const uint64_t pol_stream = l2_evict_first();
  const uint64_t pol_rows = l2_evict_last();
  unsigned long long* counter = (unsigned long long*)((char*)a.err + kWsCounterOffset);
  for (int64_t blk = next_unit(counter); blk < nblk; blk = next_unit(counter)) {
    const int64_t bag = blk * 32 + lane;
    const bool bvalid = bag < nbags;
    int64_t o0 = bvalid ? a.offsets[bag] : end_all;
    int64_t o1 = bvalid ? a.offsets[bag + 1] : end_all;
    const bool bad = o0 < 0 || o1 < o0 || o1 > a.n_idx;
    const int f = bvalid ? (int)(bag / a.B) : 0;
    const int b = bvalid ? (int)(bag - (int64_t)f * a.B) : 0;
    const int64_t ooff = (int64_t)b * a.sb + (int64_t)f * a.sf;  // this lane's bag's output row
    const float lenf = (float)(o1 - o0);
    const int64_t S0 = __shfl_sync(kFull, o0, 0);
    const int64_t S1 = __shfl_sync(kFull, o1, 31);
    if (__any_sync(kFull, bad) || S1 - S0 >= ((int64_t)1 << 30)) {
      if (lane == 0) set_error(a.err, CTR_ERR_BAD_OFFSETS);
      o0 = o1 = S0;  // write this block as zeros
    }
    unsigned empty = __ballot_sync(kFull, bvalid && o1 == o0);  // empty bags produce zero rows
    while (empty) {
      const int j = __ffs(empty) - 1;
      empty &= empty - 1;
      const float z[V] = {};
      const int64_t oj = __shfl_sync(kFull, ooff, j);
      if (lane < G) store_out(a.out, oj + (int64_t)lane * V, z, V, a.out_bf16, a.vec_out);
    }
    if (FM && bvalid && o1 == o0) a.fm_out[bag] = 0.f;
    if (__all_sync(kFull, o1 == o0)) continue;
    const int rel0 = (int)(o0 - S0), rel1 = (int)(o1 - S0);
    const uint32_t base = a.mapped ? (uint32_t)fm.base[f] : 0u;
    const uint32_t nrows = a.mapped ? (uint32_t)fm.rows[f] : (uint32_t)a.total_rows;
    const int total = (int)(S1 - S0);

    const IT* ib = idx + S0;
    IT id_b = (32 + lane < total) ? ld_id(ib + 32 + lane, pol_stream) : IT(0);
    FlatChunk cur = flat_chunk(a, lane, (lane < total) ? ld_id(ib + lane, pol_stream) : IT(0), rel0, rel1, base, nrows);
    float cur_w = merge_repeats(cur);
    float sq = 0.f;  // FM: this lane's sum of squares of the open bag's rows
    uint4 buf[kNarrowWin];
#pragma unroll
    for (int u = 0; u < kNarrowWin; ++u) {
      const int t = u * NG + grp;  // the first steps stay inside the first chunk (kNarrowWin * NG <= 32)
      const uint32_t r = __shfl_sync(kFull, cur.row, t);
      buf[u] = (r != kNoRow) ? ldg16(table + (uint64_t)r * a.ld) : make_uint4(0u, 0u, 0u, 0u);
    }
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = 0.f;
    for (int c0 = 0; c0 < total; c0 += 32) {
      const IT id_c = (c0 + 64 + lane < total) ? ld_id(ib + c0 + 64 + lane, pol_stream) : IT(0);
      FlatChunk nxt = flat_chunk(a, c0 + 32 + lane, id_b, rel0, rel1, base, nrows);
      const float nxt_w = merge_repeats(nxt);
      for (int q0 = 0; q0 < STEPS; q0 += kNarrowWin) {
#pragma unroll
        for (int j = 0; j < kNarrowWin; ++j) {
          const int q = q0 + j;
          const int t = q * NG + grp;  // this group's occurrence in this step
          float x[V];
          unpack(buf[j], x, TT());
          const int tn = t + kNarrowWin * NG;  // refill the slot (tn < 32 is the same for every group)
          const uint32_t r = __shfl_sync(kFull, tn < 32 ? cur.row : nxt.row, tn & 31);
          buf[j] = (r != kNoRow) ? ldg16(table + (uint64_t)r * a.ld) : make_uint4(0u, 0u, 0u, 0u);
          if (c0 + q * NG >= total) continue;  // warp-uniform: past the block's last occurrence
          const float wt = CTR_NARROW_MERGE ? __shfl_sync(kFull, cur_w, t) : 1.f;  // 0: a merged repeat
          if (kNarrowFast && ((cur.lastm >> (q * NG)) & kStepMask) == 0 && c0 + (q + 1) * NG <= total) {
            // no bag closes in this step and all its occurrences exist: they all belong to the open bag
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] = CTR_NARROW_MERGE ? fmaf(x[v], wt, acc[v]) : acc[v] + x[v];
            if (FM) {
#pragma unroll
              for (int v = 0; v < V; ++v) sq = fmaf(x[v], x[v] * wt, sq);
            }
            continue;
          }
          const bool valid = c0 + t < total;
          const int sg = __shfl_sync(kFull, cur.seg, t);
          const bool last = valid && ((cur.lastm >> t) & 1u);
          // the open bag is group 0's (occurrences are in bag order); close every bag that
          // ends in this step, in order, then keep the one that continues
          int open = __shfl_sync(kFull, cur.seg, q * NG);
          while (true) {
            if (valid && sg == open) {
#pragma unroll
              for (int v = 0; v < V; ++v) acc[v] = CTR_NARROW_MERGE ? fmaf(x[v], wt, acc[v]) : acc[v] + x[v];
              if (FM) {
#pragma unroll
                for (int v = 0; v < V; ++v) sq = fmaf(x[v], x[v] * wt, sq);
              }
            }
            if (!__any_sync(kFull, valid && sg == open && last)) break;  // the open bag continues
            const float lj = __shfl_sync(kFull, lenf, open);
            const int64_t oj = __shfl_sync(kFull, ooff, open);
            if constexpr (kScatter) {
              // reduce-scatter over the groups, lowest group bit first (the pairs the
              // butterfly below adds, in the same order, so both give the same bits): at each
              // level a lane sends the half of its live columns that its partner keeps and
              // adds the partner's copy of the half it keeps; each group ends with VG of each
              // lane's V columns, starting at column `coff`
              int coff = 0;
#pragma unroll
              for (int o = G, h = V / 2; o < 32; o <<= 1, h >>= 1) {
                const bool hi = (grp & (o / G)) != 0;
#pragma unroll
                for (int i = 0; i < h; ++i) {
                  const float send = hi ? acc[i] : acc[h + i];
                  const float keep = hi ? acc[h + i] : acc[i];
                  acc[i] = keep + __shfl_xor_sync(kFull, send, o);
                }
                if (hi) coff += h;
              }
              float out[VG];
#pragma unroll
              for (int v = 0; v < VG; ++v) out[v] = a.mean ? acc[v] / lj : acc[v];
              store_out(a.out, oj + (int64_t)sub * V + coff, out, VG, a.out_bf16, a.vec_out);
#pragma unroll
              for (int v = 0; v < V; ++v) acc[v] = 0.f;
              const unsigned later = __ballot_sync(kFull, valid && sg > open);
              if (!later) break;  // the bag closed at this step's last occurrence
              open = __shfl_sync(kFull, sg, __ffs(later) - 1);
              continue;
            }
#pragma unroll
            for (int o = G; o < 32; o <<= 1) {
#pragma unroll
              for (int v = 0; v < V; ++v) acc[v] += __shfl_xor_sync(kFull, acc[v], o);
              if (FM) sq += __shfl_xor_sync(kFull, sq, o);
            }
            if (FM) {  // every group now holds the bag's sums; reduce over the G lanes of a row
              float s2 = acc[0] * acc[0];
#pragma unroll
              for (int v = 1; v < V; ++v) s2 = fmaf(acc[v], acc[v], s2);
#pragma unroll
              for (int o = 1; o < G; o <<= 1) {
                s2 += __shfl_xor_sync(kFull, s2, o);
                sq += __shfl_xor_sync(kFull, sq, o);
              }
              if (lane == 0) a.fm_out[blk * 32 + open] = 0.5f * (s2 - sq);
              sq = 0.f;
            }
            if (grp == 0) {  // a closed bag is never empty
              float out[V];
#pragma unroll
              for (int v = 0; v < V; ++v) out[v] = a.mean ? acc[v] / lj : acc[v];
              store_out(a.out, oj + (int64_t)sub * V, out, V, a.out_bf16, a.vec_out);
            }
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] = 0.f;
            const unsigned later = __ballot_sync(kFull, valid && sg > open);
            if (!later) break;  // the bag closed at this step's last occurrence
            open = __shfl_sync(kFull, sg, __ffs(later) - 1);
          }
        }
      }
      cur = nxt;
      cur_w = nxt_w;
      id_b = id_c;
    }
  }
}

// The same flattened walk as bag_fwd_flat_kernel, with the rows staged by TMA
// instead of loaded into registers: for every four occurrences one lane issues
// a tile::gather4 (four 512-byte rows by row index, one mbarrier) into a ring
// of kTmaStages shared-memory stages owned by its warp, one chunk (32 rows)
// ahead of the lanes that sum them.  In flight per warp: 32 rows, held in
// shared memory, so registers no longer cap the loads in flight.  Each warp is
// an independent pipeline; every mbarrier wait is bounded and a warp that
// times out records CTR_ERR_TIMEOUT, waits (bounded) for its own copies and
// stops.
constexpr int kTmaWarps = 4;
constexpr int kTmaStages = 8;                 // 8 stages x 4 rows = one chunk ahead
constexpr int kTmaStageBytes = 4 * 512;

struct TmaRing {
  uint32_t data;     // shared address of stage 0 of this warp
  uint32_t bar;      // shared address of this warp's first mbarrier
  uint32_t issued;   // groups issued (stage = n % kTmaStages, parity = (n / kTmaStages) & 1)
  uint32_t consumed;
};

// Issue the gather of occurrences 4q .. 4q+3 of a chunk whose rows the lanes hold.
__device__ __forceinline__ void tma_issue(TmaRing& r, const CUtensorMap* map, uint32_t rows, int q) {
  const int lane = threadIdx.x & 31;
  int32_t rr[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t v = __shfl_sync(kFull, rows, 4 * q + i);
    rr[i] = v == kNoRow ? 0 : (int32_t)v;  // an unused slot still needs a valid row
  }
  const uint32_t st = r.issued % kTmaStages;
  if (lane == 0) {
    const uint32_t bar = r.bar + 8 * st;
    mbar_expect_tx(bar, kTmaStageBytes);
    tma_gather4(r.data + st * kTmaStageBytes, map, 0, rr[0], rr[1], rr[2], rr[3], bar);
  }
  ++r.issued;
}

template <typename IT>
__global__ void __launch_bounds__(kTmaWarps * 32) bag_fwd_tma_kernel(const BagArgs a,
                                                                     const __grid_constant__ FieldMap fm,
                                                                     const __grid_constant__ CUtensorMap map) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kTmaWarps][kTmaStages];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t aligned = (raw + 1023u) & ~1023u;
  const uint8_t* gen_base = smem_raw + (aligned - raw);
  TmaRing ring;
  ring.data = aligned + (uint32_t)warp * kTmaStages * kTmaStageBytes;
  ring.bar = smem_u32(&bars[warp][0]);
  ring.issued = ring.consumed = 0;
  const uint8_t* my = gen_base + (size_t)warp * kTmaStages * kTmaStageBytes + lane * 16;
  if (lane == 0) {
    for (int st = 0; st < kTmaStages; ++st) mbar_init(ring.bar + 8 * st, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int64_t nbags = (int64_t)a.F * a.B;
  const int64_t nblk = ceil_div(nbags, 32);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const IT* idx = (const IT*)a.idx;
  const int64_t end_all = a.offsets[nbags];
  bool ok = true;
  for (int64_t blk = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; ok && blk < nblk; blk += nwarps) {
    const int64_t bag = blk * 32 + lane;
    const bool bvalid = bag < nbags;
    int64_t o0 = bvalid ? a.offsets[bag] : end_all;
    int64_t o1 = bvalid ? a.offsets[bag + 1] : end_all;
    const bool bad = o0 < 0 || o1 < o0 || o1 > a.n_idx;
    const int f = bvalid ? (int)(bag / a.B) : 0;
    const int b = bvalid ? (int)(bag - (int64_t)f * a.B) : 0;
    const int64_t ooff = (int64_t)b * a.sb + (int64_t)f * a.sf + lane * 4;
    const float lenf = (float)(o1 - o0);
    const int64_t S0 = __shfl_sync(kFull, o0, 0);
    const int64_t S1 = __shfl_sync(kFull, o1, 31);
    if (__any_sync(kFull, bad) || S1 - S0 >= ((int64_t)1 << 30)) {
      if (lane == 0) set_error(a.err, CTR_ERR_BAD_OFFSETS);
      o0 = o1 = S0;
    }
    unsigned empty = __ballot_sync(kFull, bvalid && o1 == o0);
    while (empty) {
      const int j = __ffs(empty) - 1;
      empty &= empty - 1;
      const float z[4] = {0.f, 0.f, 0.f, 0.f};
      store_out(a.out, __shfl_sync(kFull, ooff, j) - j * 4 + lane * 4, z, 4, a.out_bf16, a.vec_out);
    }
    if (__all_sync(kFull, o1 == o0)) continue;
    const int rel0 = (int)(o0 - S0), rel1 = (int)(o1 - S0);
    const uint32_t base = a.mapped ? (uint32_t)fm.base[f] : 0u;
    const uint32_t nrows = a.mapped ? (uint32_t)fm.rows[f] : (uint32_t)a.total_rows;
    const int total = (int)(S1 - S0);
    const IT* ib = idx + S0;

    IT id_b = (32 + lane < total) ? ib[32 + lane] : IT(0);
    FlatChunk cur = flat_chunk(a, lane, (lane < total) ? ib[lane] : IT(0), rel0, rel1, base, nrows);
    uint32_t curv = __ballot_sync(kFull, cur.row != kNoRow);
    for (int q = 0; q < kTmaStages && 4 * q < total; ++q) tma_issue(ring, &map, cur.row, q);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; ok && c0 < total; c0 += 32) {
      const IT id_c = (c0 + 64 + lane < total) ? ib[c0 + 64 + lane] : IT(0);
      const FlatChunk nxt = flat_chunk(a, c0 + 32 + lane, id_b, rel0, rel1, base, nrows);
      const uint32_t nxtv = __ballot_sync(kFull, nxt.row != kNoRow);
      for (int q = 0; q < kTmaStages; ++q) {
        if (c0 + 4 * q >= total) break;
        const uint32_t st = ring.consumed % kTmaStages;
        if (!mbar_wait(ring.bar + 8 * st, (ring.consumed / kTmaStages) & 1)) {
          set_error(a.err, CTR_ERR_TIMEOUT);
          ok = false;
        }
        if (!__all_sync(kFull, ok)) {
          ok = false;
          break;
        }
        const uint8_t* sp = my + st * kTmaStageBytes;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = 4 * q + i;
          const float4 x = *(const float4*)(sp + i * 512);
          if ((curv >> t) & 1u) {
            acc.x += x.x;
            acc.y += x.y;
            acc.z += x.z;
            acc.w += x.w;
          }
          if ((cur.lastm >> t) & 1u) {
            const int jb = __shfl_sync(kFull, cur.seg, t);
            const int64_t oj = __shfl_sync(kFull, ooff, jb) - jb * 4 + lane * 4;
            float v[4] = {acc.x, acc.y, acc.z, acc.w};
            if (a.mean) {
              const float lj = __shfl_sync(kFull, lenf, jb);
              v[0] /= lj;
              v[1] /= lj;
              v[2] /= lj;
              v[3] /= lj;
            }
            store_out(a.out, oj, v, 4, a.out_bf16, a.vec_out);
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        ++ring.consumed;
        __syncwarp();  // every lane has read the stage before it is refilled
        if (c0 + 32 + 4 * q < total) tma_issue(ring, &map, nxt.row, q);
      }
      cur = nxt;
      curv = nxtv;
      id_b = id_c;
    }
  }
  // copies still in flight (only after a timeout) must land before the warp exits
  while (ring.consumed != ring.issued) {
    const uint32_t st = ring.consumed % kTmaStages;
    mbar_wait(ring.bar + 8 * st, (ring.consumed / kTmaStages) & 1);
    ++ring.consumed;
  }
}

// Tensor map of the table viewed as [total_rows, 128] fp32, one-row boxes.
bool make_row_map(const BagArgs& a, CUtensorMap* map) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || a.total_rows >= ((int64_t)1 << 31)) return false;
  cuuint64_t gdim[2] = {128, (cuuint64_t)a.total_rows};
  cuuint64_t gstride[1] = {512};
  cuuint32_t box[2] = {128, 1};
  cuuint32_t estride[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(a.table), gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows whose width is not a multiple of 16 bytes: one element per lane.
template <typename TT, typename IT>
__global__ void __launch_bounds__(kBagThreads) bag_fwd_scalar_kernel(const BagArgs a,
                                                                     const __grid_constant__ FieldMap fm) {
  const int lane = threadIdx.x & 31;
  const int64_t nbags = (int64_t)a.F * a.B;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const TT* table = (const TT*)a.table;
  const IT* idx = (const IT*)a.idx;
  for (int64_t bag = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; bag < nbags; bag += nwarps) {
    const int f = (int)(bag / a.B);
    const int b = (int)(bag - (int64_t)f * a.B);
    int64_t o0 = a.offsets[bag], o1 = a.offsets[bag + 1];
    const int64_t base = a.mapped ? fm.base[f] : 0;
    const int64_t nrows = a.mapped ? fm.rows[f] : a.total_rows;
    if (o0 < 0 || o1 < o0 || o1 > a.n_idx) {
      if (lane == 0) set_error(a.err, CTR_ERR_BAD_OFFSETS);
      o0 = o1 = 0;
    }
    for (int c0 = 0; c0 < a.d; c0 += 32) {
      const int c = c0 + lane;
      float acc = 0.f;
      for (int64_t i = o0; i < o1; ++i) {
        int64_t id = (int64_t)idx[i];
        if (id < 0 || id >= nrows) {
          if (lane == 0) set_error(a.err, CTR_ERR_INDEX_OUT_OF_RANGE);
          continue;
        }
        if (c < a.d) acc += (float)table[(base + id) * a.d + c];
      }
      if (a.mean) acc = (o1 > o0) ? acc / (float)(o1 - o0) : 0.f;
      if (c < a.d) store_out(a.out, (int64_t)b * a.sb + (int64_t)f * a.sf + c, &acc, 1, a.out_bf16, false);
    }
  }
}

template <typename K>
int grid_for(K kernel, int64_t nbags) {
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBagThreads, 0);
  int64_t want = ceil_div(nbags, kBagThreads / 32);
  int64_t cap = (int64_t)std::max(per_sm, 1) * num_sms();
  return (int)std::max<int64_t>(1, std::min(want, cap));
}

template <typename TT, typename IT>
int launch_bag_fwd(const BagArgs& a, const FieldMap& fm, cudaStream_t s) {
  constexpr int V = Vec<TT>::kN;
  const int64_t nbags = (int64_t)a.F * a.B;
  if (a.d % V != 0) {
    if (a.fm_out) return CTR_ERR_UNSUPPORTED;
    auto k = bag_fwd_scalar_kernel<TT, IT>;
    k<<<grid_for(k, nbags), kBagThreads, 0, s>>>(a, fm); count_launch();
    return launch_status();
  }
  const int chunks = a.d / V;
  CUtensorMap map;
  if (std::is_same<TT, float>::value && a.d == 128 && g_tma_gather.load(std::memory_order_relaxed) && !a.fm_out && make_row_map(a, &map)) {
    auto k = bag_fwd_tma_kernel<IT>;
    const size_t smem = 1024 + (size_t)kTmaWarps * kTmaStages * kTmaStageBytes;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return CTR_ERR_CUDA;
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kTmaWarps * 32, smem);
    const int64_t want = ceil_div(ceil_div(nbags, 32), kTmaWarps);
    const int grid = (int)std::max<int64_t>(1, imin64(want, (int64_t)std::max(per_sm, 1) * num_sms()));
    k<<<grid, kTmaWarps * 32, smem, s>>>(a, fm, map); count_launch();
    return launch_status();
  }
  if (std::is_same<TT, float>::value && a.d == 128 && a.total_rows < 0xffffffffll) {
    if (cudaMemsetAsync((char*)a.err + kWsCounterOffset, 0, sizeof(unsigned long long), s) != cudaSuccess)
      return CTR_ERR_CUDA;
    const bool small = ceil_div(nbags, 32) < kSmallGridBlocks * num_sms();
    auto k = a.fm_out ? (small ? bag_fwd_flat_kernel<IT, true, kWinSmall, kMinbSmall> : bag_fwd_flat_kernel<IT, true>)
                      : (small ? bag_fwd_flat_kernel<IT, false, kWinSmall, kMinbSmall> : bag_fwd_flat_kernel<IT, false>);
    k<<<grid_for(k, ceil_div(nbags, 32)), kBagThreads, 0, s>>>(a, fm); count_launch();
    return launch_status();
  }
  // narrow rows: the flattened walk with several rows per warp step (CTR_USE_NARROW=0 builds the
  // one-bag-per-warp kernel below instead, for comparison)
  if (CTR_USE_NARROW && (chunks == 4 || chunks == 8 || chunks == 16) && a.total_rows < 0xffffffffll) {
    if (cudaMemsetAsync((char*)a.err + kWsCounterOffset, 0, sizeof(unsigned long long), s) != cudaSuccess)
      return CTR_ERR_CUDA;
#define CTR_NARROW(G)                                                                       \
  {                                                                                         \
    auto k = a.fm_out ? bag_fwd_narrow_kernel<TT, G, IT, true> : bag_fwd_narrow_kernel<TT, G, IT, false>; \
    k<<<grid_for(k, ceil_div(nbags, 32)), kBagThreads, 0, s>>>(a, fm);                      \
    count_launch();                                                                         \
    return launch_status();                                                                 \
  }
    if (chunks == 4) CTR_NARROW(4)
    if (chunks == 8) CTR_NARROW(8)
    CTR_NARROW(16)
#undef CTR_NARROW
  }
#define CTR_LAUNCH(LPR, CPL)                                 \
  {                                                          \
    auto k = bag_fwd_kernel<TT, LPR, CPL, IT>;               \
    k<<<grid_for(k, nbags), kBagThreads, 0, s>>>(a, fm);     \
    count_launch();                                          \
    return launch_status();                                  \
  }
  if (chunks <= 1) CTR_LAUNCH(1, 1)
  if (chunks <= 2) CTR_LAUNCH(2, 1)
  if (chunks <= 4) CTR_LAUNCH(4, 1)
  if (chunks <= 8) CTR_LAUNCH(8, 1)
  if (chunks <= 16) CTR_LAUNCH(16, 1)
  if (chunks <= 32) CTR_LAUNCH(32, 1)
  if (chunks <= 64) CTR_LAUNCH(32, 2)
  if (chunks <= 128) CTR_LAUNCH(32, 4)
#undef CTR_LAUNCH
  return CTR_ERR_UNSUPPORTED;
}

// U[u] = table[unique_rows[u]]: one warp per row, 16-byte lanes.
__global__ void __launch_bounds__(256) gather_rows_kernel(const char* __restrict__ table, int64_t row_bytes,
                                                          int64_t total_rows, const int64_t* __restrict__ unique_rows,
                                                          const int64_t* __restrict__ n_unique, int64_t capacity,
                                                          char* __restrict__ U, int* err) {
  const int lane = threadIdx.x & 31;
  const int64_t n = imin64(*n_unique, capacity);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const bool vec = (row_bytes % 16) == 0;
  for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < n; u += nwarps) {
    const int64_t r = unique_rows[u];
    if (r < 0 || r >= total_rows) {
      if (lane == 0) set_error(err, CTR_ERR_INDEX_OUT_OF_RANGE);
      continue;
    }
    const char* src = table + r * row_bytes;
    char* dst = U + u * row_bytes;
    if (vec) {
      for (int64_t o = (int64_t)lane * 16; o < row_bytes; o += 32 * 16) *(uint4*)(dst + o) = ldg16(src + o);
    } else {
      for (int64_t o = lane; o < row_bytes; o += 32) dst[o] = src[o];
    }
  }
}

// Rows of G 16-byte chunks (G = 1..32, a power of two): a group of G lanes
// copies one row and the 32 / G groups of a warp take consecutive uniques, with
// kRowSteps such steps in flight per warp (their row indices, then their rows,
// are loaded before any is stored), so short rows keep every lane and many
// loads busy instead of one row per warp at a time.
constexpr int kRowSteps = 4;
template <int G>
__global__ void __launch_bounds__(256) gather_rows_grouped_kernel(const char* __restrict__ table, int64_t row_bytes,
                                                                  int64_t total_rows,
                                                                  const int64_t* __restrict__ unique_rows,
                                                                  const int64_t* __restrict__ n_unique,
                                                                  int64_t capacity, char* __restrict__ U, int* err) {
  constexpr int RPW = 32 / G;  // rows per warp step
  const int lane = threadIdx.x & 31, grp = lane / G, sub = lane % G;
  const int64_t n = imin64(*n_unique, capacity);
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  for (int64_t u0 = w0 * (RPW * kRowSteps); u0 < n; u0 += nwarps * (RPW * kRowSteps)) {
    int64_t r[kRowSteps];
#pragma unroll
    for (int k = 0; k < kRowSteps; ++k) {
      const int64_t u = u0 + k * RPW + grp;
      r[k] = u < n ? unique_rows[u] : -1;
      if (u < n && (r[k] < 0 || r[k] >= total_rows)) {
        set_error(err, CTR_ERR_INDEX_OUT_OF_RANGE);
        r[k] = -1;
      }
    }
    uint4 v[kRowSteps];
#pragma unroll
    for (int k = 0; k < kRowSteps; ++k)
      v[k] = r[k] >= 0 ? ldg16(table + r[k] * row_bytes + sub * 16) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < kRowSteps; ++k)
      if (r[k] >= 0) *(uint4*)(U + (u0 + k * RPW + grp) * row_bytes + sub * 16) = v[k];
  }
}

}  // namespace
}  // namespace ctr

using namespace ctr;

extern "C" size_t ctr_embedding_bag_workspace_size(void) { return kWsHeader; }

extern "C" int ctr_set_tma_gather(int on) { return g_tma_gather.exchange(on ? 1 : 0); }

namespace {

int embedding_bag_fwd(const void* table, ctr_dtype dtype, int32_t d, int64_t total_rows, const void* indices,
                      int indices_are_int32, int64_t n_indices, const int64_t* offsets, int32_t num_fields,
                      int32_t batch, const int32_t* bag_to_table, const int64_t* row_base, int32_t num_tables,
                      ctr_pool pool, void* out, ctr_dtype out_dtype, int64_t out_stride_b, int64_t out_stride_f,
                      float* fm_out, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!table || !offsets || !out || d <= 0 || total_rows <= 0) return CTR_ERR_INVALID_ARG;
  if (num_fields <= 0 || batch <= 0) return CTR_ERR_INVALID_ARG;
  if ((dtype != CTR_F32 && dtype != CTR_BF16) || (out_dtype != CTR_F32 && out_dtype != CTR_BF16))
    return CTR_ERR_INVALID_ARG;
  if (pool != CTR_POOL_SUM && pool != CTR_POOL_MEAN) return CTR_ERR_INVALID_ARG;
  if (out_stride_b < 0 || out_stride_f < 0) return CTR_ERR_INVALID_ARG;
  if (!ws_valid(ws, ws_bytes, ctr_embedding_bag_workspace_size())) return CTR_ERR_WORKSPACE;
  FieldMap fm;
  int mapped = bag_to_table != nullptr;
  if (mapped) {
    if (!row_base) return CTR_ERR_INVALID_ARG;
    if (int st = make_field_map(bag_to_table, row_base, num_fields, num_tables, &fm)) return st;
    if (row_base[num_tables] > total_rows) return CTR_ERR_INVALID_ARG;
  } else if (num_fields > CTR_MAX_FIELDS) {
    return CTR_ERR_UNSUPPORTED;
  }
  if (n_indices < 0 || (n_indices > 0 && !indices)) return CTR_ERR_INVALID_ARG;
  BagArgs a;
  a.table = table;
  a.d = d;
  a.ld = d;
  a.total_rows = total_rows;
  a.idx = indices;
  a.n_idx = n_indices;
  a.offsets = offsets;
  a.F = num_fields;
  a.B = batch;
  a.mapped = mapped;
  a.mean = pool == CTR_POOL_MEAN;
  a.out = out;
  a.out_bf16 = out_dtype == CTR_BF16;
  const int vout = out_dtype == CTR_BF16 ? 8 : 4;
  a.vec_out = ((uintptr_t)out % 16 == 0) && (out_stride_b % vout == 0) && (out_stride_f % vout == 0) && (d % vout == 0);
  a.sb = out_stride_b;
  a.sf = out_stride_f;
  a.err = (int*)ws;
  a.fm_out = fm_out;
  if ((uintptr_t)table % 16 != 0) return CTR_ERR_INVALID_ARG;
  timing_mark(CTR_KERNEL_GATHER, true, s);
  int st;
  if (dtype == CTR_F32)
    st = indices_are_int32 ? launch_bag_fwd<float, int32_t>(a, fm, s) : launch_bag_fwd<float, int64_t>(a, fm, s);
  else
    st = indices_are_int32 ? launch_bag_fwd<__nv_bfloat16, int32_t>(a, fm, s)
                           : launch_bag_fwd<__nv_bfloat16, int64_t>(a, fm, s);
  timing_mark(CTR_KERNEL_GATHER, false, s);
  return st;
}

}  // namespace

extern "C" int ctr_embedding_bag_fwd(const void* table, ctr_dtype dtype, int32_t d, int64_t total_rows,
                                     const void* indices, int indices_are_int32, int64_t n_indices,
                                     const int64_t* offsets,
                                     int32_t num_fields, int32_t batch, const int32_t* bag_to_table,
                                     const int64_t* row_base, int32_t num_tables, ctr_pool pool, void* out,
                                     ctr_dtype out_dtype, int64_t out_stride_b, int64_t out_stride_f, void* ws,
                                     size_t ws_bytes, ctr_stream_t stream) {
  return embedding_bag_fwd(table, dtype, d, total_rows, indices, indices_are_int32, n_indices, offsets, num_fields,
                           batch, bag_to_table, row_base, num_tables, pool, out, out_dtype, out_stride_b,
                           out_stride_f, nullptr, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int ctr_embedding_bag_fwd_fm(const void* table, ctr_dtype dtype, int32_t d, int64_t total_rows,
                                        const void* indices, int indices_are_int32, int64_t n_indices,
                                        const int64_t* offsets, int32_t num_fields, int32_t batch,
                                        const int32_t* bag_to_table, const int64_t* row_base, int32_t num_tables,
                                        ctr_pool pool, void* out, ctr_dtype out_dtype, int64_t out_stride_b,
                                        int64_t out_stride_f, float* fm_out, void* ws, size_t ws_bytes,
                                        ctr_stream_t stream) {
  if (!fm_out) return CTR_ERR_INVALID_ARG;
  return embedding_bag_fwd(table, dtype, d, total_rows, indices, indices_are_int32, n_indices, offsets, num_fields,
                           batch, bag_to_table, row_base, num_tables, pool, out, out_dtype, out_stride_b,
                           out_stride_f, fm_out, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int ctr_gather_rows(const void* table, ctr_dtype dtype, int32_t d, int64_t total_rows,
                               const int64_t* unique_rows, const int64_t* n_unique, int64_t capacity, void* U,
                               void* ws, size_t ws_bytes, ctr_stream_t stream) {
  if (!table || !unique_rows || !n_unique || !U || d <= 0 || total_rows <= 0 || capacity < 0)
    return CTR_ERR_INVALID_ARG;
  if (dtype != CTR_F32 && dtype != CTR_BF16) return CTR_ERR_INVALID_ARG;
  if (!ws_valid(ws, ws_bytes, kWsHeader)) return CTR_ERR_WORKSPACE;
  if (capacity == 0) return CTR_OK;
  const int64_t row_bytes = (int64_t)d * (dtype == CTR_F32 ? 4 : 2);
  if (row_bytes % 16 == 0 && (((uintptr_t)table | (uintptr_t)U) % 16) != 0) return CTR_ERR_INVALID_ARG;
  const int64_t chunks = row_bytes / 16;
  const bool grouped = row_bytes % 16 == 0 && chunks <= 32 && (chunks & (chunks - 1)) == 0;
  timing_mark(CTR_KERNEL_GATHER_ROWS, true, (cudaStream_t)stream);
  if (grouped) {
    // a full wave of 8 blocks per SM; each warp step covers 32 / chunks uniques
    const int64_t per_block = (int64_t)8 * (32 / chunks) * kRowSteps;
    const int64_t blocks = std::max<int64_t>(1, imin64(ceil_div(capacity, per_block), (int64_t)num_sms() * 8));
    auto k = chunks == 1    ? gather_rows_grouped_kernel<1>
             : chunks == 2  ? gather_rows_grouped_kernel<2>
             : chunks == 4  ? gather_rows_grouped_kernel<4>
             : chunks == 8  ? gather_rows_grouped_kernel<8>
             : chunks == 16 ? gather_rows_grouped_kernel<16>
                            : gather_rows_grouped_kernel<32>;
    k<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>((const char*)table, row_bytes, total_rows, unique_rows,
                                                         n_unique, capacity, (char*)U, (int*)ws);
  } else {
    const int64_t blocks = imin64(ceil_div(capacity, 8), (int64_t)num_sms() * 16);
    gather_rows_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
        (const char*)table, row_bytes, total_rows, unique_rows, n_unique, capacity, (char*)U, (int*)ws);
  }
  count_launch();
  timing_mark(CTR_KERNEL_GATHER_ROWS, false, (cudaStream_t)stream);
  return launch_status();
}
