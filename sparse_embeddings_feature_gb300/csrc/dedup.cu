// a1. Batch ID dedup into the "virtual sparse feature" index.
//
// Source: "How TensorNet Supercharges Sparse Feature Training on TensorFlow",
// Core Optimizations, embedding_lookup: collect the batch's IDs, sort them and
// give each distinct ID a continuous index.
//
// GPU design (sm_103a, one GPU).  Keys are 32-bit global rows
// (row_base[table(f)] + id).  Two paths, chosen from the sizes alone:
//
// Presence bitmap (total_rows <= 64 * n_ids, the common case):
//   mark       warp per bag: set bit key of a bitmap over all table rows
//              (L2-resident: 26 MB for 208M rows).
//   prefix     set bits per 1024-word block, a scan, then per word its bits
//              and the count of set bits before it; the unique rows are the
//              set bits in order, n_unique the total.
//   rank       warp per bag again: rank(key) = prefix(word) + popc(bits below),
//              which is the inverse map (written in ID order); sort keys =
//              ranks, values = bags (or positions when the caller wants the
//              permutation), digit histograms of every pass.
//   sort       LSD radix passes over the ranks only: ceil(bits(n_unique) / 8)
//              passes, planned on the device (24-bit ranks: 3 passes).
//   runs       ranks are dense, so the first slot holding rank r starts run r.
// Sorted keys (larger tables than the batch can fill):
//   keygen     warp per bag: keys, bag of each position, digit histograms.
//   sort       ceil(bits(total_rows) / 8) passes over the keys.
//   unique     head flags, per-tile head counts, a scan, then ranks:
//              unique_rows, run_offsets, inverse (scatter), sorted_bag
//              (gather of the bag of each sorted position), unique_offsets.
// Each radix pass is one kernel (Onesweep-style decoupled look-back, below).
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "scan.cuh"

namespace ctr {
namespace {

constexpr int kRsThreads = 256;
constexpr int kRsWarps = kRsThreads / 32;
// Keys per lane per tile, and resident blocks per SM the registers are capped
// for: 12 keys at 4 blocks (64 registers, 3072-key tiles) against 16 at 3 (80
// registers): the full step 13.61 -> 13.44 ms in one session (20 keys at 2
// blocks: 13.45; 8 at 5: slower).
#ifndef CTR_RS_ITEMS
#define CTR_RS_ITEMS 12
#endif
#ifndef CTR_RS_MINB
#define CTR_RS_MINB 4
#endif
constexpr int kRsItems = CTR_RS_ITEMS;            // keys per lane per tile
constexpr int kRsTile = kRsThreads * kRsItems;    // 3072 keys
constexpr int kRsWarpKeys = 32 * kRsItems;        // 384 keys per warp
constexpr int kMaxBits = 8;                       // digit width limit (256 buckets)
constexpr int kMaxDigits = 1 << kMaxBits;
constexpr int kMaxPasses = 4;                     // 32-bit keys
constexpr uint64_t kFlagAggregate = 1ull << 32;   // look-back word: tile's own digit count
constexpr uint64_t kFlagInclusive = 2ull << 32;   // look-back word: count of this and all earlier tiles

struct TableBases {
  int64_t row_base[CTR_MAX_TABLES + 1];
  int32_t num_tables;
};

struct PassPlan {
  int passes;
  int shift[kMaxPasses];
  int bits[kMaxPasses];
};

// Keys, bags, and the digit histograms of every radix pass (one read of the IDs).
__global__ void __launch_bounds__(256) keygen_kernel(const int64_t* __restrict__ ids,
                                                     const int64_t* __restrict__ offsets, int32_t F, int32_t B,
                                                     int64_t n_ids, const __grid_constant__ FieldMap fm,
                                                     uint32_t* __restrict__ keys, int32_t* __restrict__ bag_of,
                                                     const PassPlan plan, uint32_t* __restrict__ g_hist, int* err) {
  __shared__ uint32_t sh[kMaxPasses][kMaxDigits];
  for (int i = threadIdx.x; i < kMaxPasses * kMaxDigits; i += blockDim.x) (&sh[0][0])[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t nbags = (int64_t)F * B;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (offsets[0] != 0 || offsets[nbags] != n_ids) set_error(err, CTR_ERR_BAD_OFFSETS);
  }
  for (int64_t bag = warp0; bag < nbags; bag += nwarps) {
    const int f = (int)(bag / B);
    const int64_t o0 = offsets[bag], o1 = offsets[bag + 1];
    if (o0 < 0 || o1 < o0 || o1 > n_ids) {
      if (lane == 0) set_error(err, CTR_ERR_BAD_OFFSETS);
      continue;
    }
    const int64_t base = fm.base[f], rows = fm.rows[f];
    for (int64_t i = o0 + lane; i < o1; i += 32) {
      int64_t id = ids[i];
      if (id < 0 || id >= rows) {
        set_error(err, CTR_ERR_INDEX_OUT_OF_RANGE);
        id = rows - 1;
      }
      const uint32_t k = (uint32_t)(base + id);
      keys[i] = k;
      bag_of[i] = (int32_t)bag;
      for (int p = 0; p < plan.passes; ++p)
        atomicAdd(&sh[p][(k >> plan.shift[p]) & ((1u << plan.bits[p]) - 1)], 1u);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < plan.passes * kMaxDigits; i += blockDim.x) {
    const uint32_t c = (&sh[0][0])[i];
    if (c) atomicAdd(&g_hist[i], c);
  }
}

__device__ __forceinline__ uint32_t digit_of(uint32_t k, int shift, uint32_t mask) { return (k >> shift) & mask; }

// Look-back words carry their flag and count in one 64-bit access, so relaxed
// gpu-scope loads and stores suffice (nothing else is published through them).
static __device__ __forceinline__ void st_relaxed(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
static __device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
constexpr int kLbWindow = 4;  // predecessors read per look-back round trip
static __device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wall-clock limit of one look-back wait: 1 s, or what ctr_set_wait_limit_ns
// set (a diagnostic: a short limit makes ordinary waits run out, which tests
// the timeout path without faulting or hanging anything).
std::atomic<uint64_t> g_lookback_limit_ns{1000000000ull};

// One radix pass in one kernel (single-pass, after Adinets and Merrill's
// Onesweep): a block takes the next tile in launch order, ranks its keys
// stably (per 32 keys __match_any_sync groups equal digits; per-warp digit
// counters order the rows and warps), publishes its per-digit counts, and finds the
// counts of all earlier tiles by decoupled look-back: a predecessor's word
// holds either its own count or its inclusive prefix, so the walk stops at
// the first inclusive prefix; each thread reads kLbWindow predecessors per
// round trip.  Tiles are taken in order, so a block only
// ever waits on blocks that started before it; each wait is bounded by a
// wall-clock limit, after which the block records CTR_ERR_TIMEOUT and keeps
// its writes inside the output.  vals_in == nullptr means the values are
// the positions 0..n-1 (first pass).
__global__ void __launch_bounds__(kRsThreads, CTR_RS_MINB) onesweep_kernel(
    const uint32_t* __restrict__ keys_in, const int32_t* __restrict__ vals_in, uint32_t* __restrict__ keys_out,
    int32_t* __restrict__ vals_out, int64_t n, int shift, int nbits, const PassPlan* __restrict__ dplan, int pass,
    int32_t* __restrict__ vals_final, const uint32_t* __restrict__ g_hist, uint64_t* __restrict__ lookback,
    uint32_t* __restrict__ tile_counter, int* err, uint64_t limit_ns, int32_t* __restrict__ run_offsets,
    const int64_t* __restrict__ n_unique) {
  bool runs = false;  // this pass also writes the run starts (and not the sorted keys)
  if (dplan) {  // digit plan decided on the device (rank keys): passes beyond it do nothing
    if (pass >= dplan->passes) return;
    shift = dplan->shift[pass];
    nbits = dplan->bits[pass];
    if (pass == dplan->passes - 1 && vals_final) vals_out = vals_final;
    runs = run_offsets != nullptr && pass == dplan->passes - 1;
  }
  __shared__ uint32_t wcnt[kRsWarps][kMaxDigits];
  __shared__ uint32_t tile_start[kMaxDigits];
  __shared__ uint32_t glob_start[kMaxDigits];
  __shared__ uint32_t skeys[kRsTile];
  __shared__ int32_t svals[kRsTile];
  __shared__ uint32_t warp_tot[kRsWarps];
  __shared__ uint32_t tile_sh;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ndig = 1 << nbits;
  const uint32_t mask = (uint32_t)ndig - 1;
  for (int i = threadIdx.x; i < kRsWarps * kMaxDigits; i += kRsThreads) (&wcnt[0][0])[i] = 0;
  if (threadIdx.x == 0) tile_sh = atomicAdd(tile_counter, 1u);
  __syncthreads();
  // all offsets fit 32 bits: the entry point admits fewer than 2^31 keys
  const int n32 = (int)n;
  const int tile = (int)tile_sh;
  const int tile_base = tile * kRsTile;
  const int base = tile_base + warp * kRsWarpKeys;
  const unsigned lt = lanemask_lt();
  uint32_t key[kRsItems];
  int32_t val[kRsItems];
  uint32_t rank[kRsItems];
#pragma unroll
  for (int r = 0; r < kRsItems; ++r) {
    const int idx = base + r * 32 + lane;
    const bool valid = idx < n32;
    key[r] = valid ? keys_in[idx] : 0u;
    val[r] = valid ? (vals_in ? vals_in[idx] : idx) : 0;
  }
#pragma unroll
  for (int r = 0; r < kRsItems; ++r) {
    const bool valid = base + r * 32 + lane < n32;
    const uint32_t dg = digit_of(key[r], shift, mask);
    // lanes of this row holding the same digit (invalid lanes share a value no digit takes)
    const unsigned peers = __match_any_sync(kFull, valid ? dg : 0xffffffffu);
    const uint32_t prior = valid ? wcnt[warp][dg] : 0u;
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) wcnt[warp][dg] = prior + __popc(peers);
    __syncwarp();
    rank[r] = valid ? prior + __popc(peers & lt) : 0xffffffffu;
  }
  __syncthreads();
  // thread t owns digit t: exclusive over warps (in place), tile count, bucket start
  const int dg = threadIdx.x;  // kRsThreads == kMaxDigits
  uint32_t cnt = 0;
  if (dg < ndig) {
#pragma unroll
    for (int w = 0; w < kRsWarps; ++w) {
      const uint32_t c = wcnt[w][dg];
      wcnt[w][dg] = cnt;
      cnt += c;
    }
  }
  uint64_t* my_word = lookback + (int64_t)tile * kMaxDigits + dg;
  if (dg < ndig) st_relaxed(my_word, (tile == 0 ? kFlagInclusive : kFlagAggregate) | cnt);
  uint32_t gh[1] = {dg < ndig ? g_hist[dg] : 0u};
  uint32_t tc[1] = {cnt};
  block_exclusive_scan<uint32_t, kRsThreads, 1>(gh, warp_tot);  // bucket start of digit dg
  block_exclusive_scan<uint32_t, kRsThreads, 1>(tc, warp_tot);  // digit dg's start inside the tile
  bool timed_out = false;
  uint32_t excl = 0;
  if (dg < ndig && tile > 0) {
    // walk back kLbWindow predecessors per round trip; stop at the first
    // inclusive prefix, wait (bounded) where a predecessor has not published
    int j = tile - 1;
    uint64_t t0 = 0;
    while (j >= 0) {
      uint64_t w[kLbWindow];
#pragma unroll
      for (int q = 0; q < kLbWindow; ++q)
        w[q] = (j - q >= 0) ? ld_relaxed(lookback + (int64_t)(j - q) * kMaxDigits + dg) : kFlagInclusive;
      int used = 0;
      bool done = false, stalled = false;
#pragma unroll
      for (int q = 0; q < kLbWindow; ++q) {
        if (done || stalled) continue;
        const uint64_t flag = w[q] & ~0xffffffffull;
        if (flag == 0) {
          stalled = true;
        } else {
          excl += (uint32_t)w[q];
          ++used;
          if (flag == kFlagInclusive) done = true;
        }
      }
      if (done) break;
      j -= used;
      if (stalled) {
        const uint64_t t = now_ns();
        if (t0 == 0) t0 = t;
        else if (t - t0 > limit_ns) {
          timed_out = true;
          break;
        }
      } else {
        t0 = 0;
      }
    }
    st_relaxed(my_word, kFlagInclusive | (excl + cnt));
  }
  if (timed_out) set_error(err, CTR_ERR_TIMEOUT);
  if (dg < ndig) {
    tile_start[dg] = tc[0];
    glob_start[dg] = gh[0] + excl;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kRsItems; ++r) {
    if (rank[r] != 0xffffffffu) {
      const uint32_t d = digit_of(key[r], shift, mask);
      const uint32_t local = tile_start[d] + wcnt[warp][d] + rank[r];
      skeys[local] = key[r];
      svals[local] = val[r];
    }
  }
  __syncthreads();
  const int count = min(kRsTile, n32 - tile_base);
  const int64_t nu = runs ? *n_unique : 0;
  for (int i = threadIdx.x; i < count; i += kRsThreads) {
    const uint32_t k = skeys[i];
    const uint32_t d = digit_of(k, shift, mask);
    const uint32_t dest = glob_start[d] + (uint32_t)i - tile_start[d];
    if (dest < (uint32_t)n32) {  // always true unless a look-back timed out
      vals_out[dest] = svals[i];
      if (!runs) {
        keys_out[dest] = k;
      } else if ((int64_t)k >= nu) {  // only after an error that left key slots unwritten
        set_error(err, CTR_ERR_BAD_OFFSETS);
      } else if (i > (int)tile_start[d]) {
        // the element before it in the output is the one before it in this tile's
        // digit group: a run starts here iff the keys differ
        if (skeys[i - 1] != k) run_offsets[k] = (int32_t)dest;
      } else {
        // first of its digit group in this tile: the element before it was written by
        // an earlier tile, so every such candidate is offered and the smallest kept (the
        // starts were set to 0xffffffff before the passes)
        atomicMin((unsigned int*)(run_offsets + k), dest);
      }
      if (runs && dest == (uint32_t)n32 - 1) run_offsets[nu] = n32;
    }
  }
}

__global__ void clear_u64_kernel(uint64_t* __restrict__ p, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = 0;
}

// Heads per tile of the sorted keys.
__global__ void __launch_bounds__(kRsThreads) unique_count_kernel(const uint32_t* __restrict__ skeys, int64_t n,
                                                                  uint32_t* __restrict__ tile_heads) {
  __shared__ uint32_t warp_tot[kRsWarps];
  const int64_t base = (int64_t)blockIdx.x * kRsTile;
  uint32_t c = 0;
#pragma unroll 4
  for (int i = 0; i < kRsItems; ++i) {
    int64_t s = base + (int64_t)i * kRsThreads + threadIdx.x;
    if (s < n) c += (s == 0 || skeys[s] != skeys[s - 1]) ? 1u : 0u;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
  if ((threadIdx.x & 31) == 0) warp_tot[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int w = 0; w < kRsWarps; ++w) t += warp_tot[w];
    tile_heads[blockIdx.x] = t;
  }
}

__device__ __forceinline__ int table_of(const int64_t* rb, int T, int64_t k) {
  // largest t in [0, T) with rb[t] <= k
  int lo = 0, hi = T - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (rb[mid] <= k) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Ranks and outputs of one tile of sorted keys.  The tile's slots are read as
// kRsItems coalesced rows of 256 (slot = row * 256 + thread): head flags come
// from one ballot per warp and row, and a scan of the kRsItems x 8 per-warp
// head counts gives every slot its rank.
__global__ void __launch_bounds__(kRsThreads) unique_write_kernel(
    const uint32_t* __restrict__ skeys, const int32_t* __restrict__ spos, int64_t n,
    const uint32_t* __restrict__ tile_base_scan, const __grid_constant__ TableBases tb,
    const int32_t* __restrict__ bag_of, int64_t* __restrict__ unique_rows, int64_t* __restrict__ n_unique,
    int32_t* __restrict__ inverse, int32_t* __restrict__ sorted_bag, int32_t* __restrict__ run_offsets,
    int64_t* __restrict__ unique_offsets) {
  constexpr int kRows = kRsTile / kRsThreads;  // keys per thread
  __shared__ uint32_t cnt[kRows * kRsWarps];     // heads per (row, warp), then exclusive offsets
  __shared__ int64_t rb[CTR_MAX_TABLES + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int T = tb.num_tables;
  for (int i = threadIdx.x; i <= T; i += kRsThreads) rb[i] = tb.row_base[i];
  const int64_t tile0 = (int64_t)blockIdx.x * kRsTile;
  const unsigned lt = lanemask_lt();
  uint32_t key[kRows];
  unsigned mask[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int64_t sl = tile0 + r * kRsThreads + threadIdx.x;
    const bool valid = sl < n;
    key[r] = valid ? skeys[sl] : 0u;
    const uint32_t prevk = (valid && sl > 0) ? skeys[sl - 1] : ~key[r];
    mask[r] = __ballot_sync(kFull, valid && (sl == 0 || key[r] != prevk));
    if (lane == 0) cnt[r * kRsWarps + warp] = __popc(mask[r]);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the kRows x kRsWarps counts, kPer per lane, in slot order
    constexpr int kCounts = kRows * kRsWarps;
    constexpr int kPer = (kCounts + 31) / 32;
    uint32_t v[kPer], sum = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int i = lane * kPer + q;
      v[q] = i < kCounts ? cnt[i] : 0u;
      sum += v[q];
    }
    uint32_t inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += y;
    }
    uint32_t run = inc - sum;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int i = lane * kPer + q;
      if (i < kCounts) cnt[i] = run;
      run += v[q];
    }
  }
  __syncthreads();
  const uint32_t tbase = tile_base_scan[blockIdx.x];
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int64_t sl = tile0 + r * kRsThreads + threadIdx.x;
    if (sl >= n) break;
    const bool head = (mask[r] >> lane) & 1u;
    // rank of this key = heads in [0, sl] - 1
    const uint32_t rank = tbase + cnt[r * kRsWarps + warp] + __popc(mask[r] & lt) + (head ? 1u : 0u) - 1u;
    if (head) {
      unique_rows[rank] = (int64_t)key[r];
      if (run_offsets) run_offsets[rank] = (int32_t)sl;
      if (unique_offsets) {
        const int t = table_of(rb, T, (int64_t)key[r]);
        const int t0 = sl > 0 ? table_of(rb, T, (int64_t)skeys[sl - 1]) + 1 : 0;
        for (int tt = t0; tt <= t; ++tt) unique_offsets[tt] = rank;
      }
    }
    const int32_t p = spos[sl];
    if (inverse) inverse[p] = (int32_t)rank;
    if (sorted_bag) sorted_bag[sl] = bag_of[p];
    if (sl == n - 1) {
      const uint32_t nu = rank + 1;
      *n_unique = nu;
      if (run_offsets) run_offsets[nu] = (int32_t)n;
      if (unique_offsets) {
        const int t = table_of(rb, T, (int64_t)key[r]);
        for (int tt = t + 1; tt <= T; ++tt) unique_offsets[tt] = nu;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Presence-bitmap path (tables not much larger than the batch): the rank of a
// key among the batch's distinct keys is the number of set bits below it in a
// bitmap over all table rows, so the inverse map and the unique rows come from
// the bitmap directly; the radix sort only groups the occurrences by rank
// (ceil(bits(n_unique) / 8) passes instead of ceil(bits(total_rows) / 8)) and
// carries each occurrence's bag, so the grouped bags, and the run starts, come
// out of its last pass.
// ---------------------------------------------------------------------------
constexpr int64_t kBitmapRowsPerId = 64;  // bitmap path iff total_rows <= 64 * n_ids
constexpr int kBmWords = 1024;            // bitmap words per prefix block (4 per thread)

__device__ __forceinline__ uint32_t ld_l1(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.global.ca.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

constexpr int kKeyChunks = 4;  // chunks of 32 IDs a warp has in flight

// Keys (32-bit global rows), the sort's first values, and the presence bitmap,
// in one flat walk over the IDs: a warp takes 32 consecutive bags and its
// lanes take their IDs 32 at a time, kKeyChunks chunks at once (every lane
// busy whatever the bag lengths, several loads in flight); a lane finds its
// bag by a shuffle binary search over the lanes' bag starts.  IDs get the key
// generator's validation and clamping; a block of bags with inconsistent
// offsets is flagged and skipped.  A key whose bit is already set is not set
// again, so the hot rows of a skewed batch cost L1-cached loads, not atomics
// (bits only go from 0 to 1, so a stale word only costs a redundant atomic).
__global__ void __launch_bounds__(256) bitmap_keys_kernel(const int64_t* __restrict__ ids,
                                                          const int64_t* __restrict__ offsets, int32_t F, int32_t B,
                                                          int64_t n_ids, const __grid_constant__ FieldMap fm,
                                                          uint32_t* __restrict__ keys, int32_t* __restrict__ vals,
                                                          int vals_are_pos, int32_t* __restrict__ bag_of,
                                                          uint32_t* __restrict__ bitmap, int* err) {
  const int lane = threadIdx.x & 31;
  const int64_t nbags = (int64_t)F * B;
  const int64_t nblk = ceil_div(nbags, (int64_t)32);
  const int64_t end_all = offsets[nbags];
  if (blockIdx.x == 0 && threadIdx.x == 0 && (offsets[0] != 0 || end_all != n_ids))
    set_error(err, CTR_ERR_BAD_OFFSETS);
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t blk = warp0; blk < nblk; blk += nwarps) {
    const int64_t bag = blk * 32 + lane;
    const bool bvalid = bag < nbags;
    const int64_t o0 = bvalid ? offsets[bag] : end_all;
    const int64_t o1 = bvalid ? offsets[bag + 1] : end_all;
    const bool bad = o0 < 0 || o1 < o0 || o1 > n_ids;
    const int64_t S0 = __shfl_sync(kFull, o0, 0);
    const int64_t S1 = __shfl_sync(kFull, o1, 31);
    if (__any_sync(kFull, bad) || S1 < S0 || S1 - S0 >= ((int64_t)1 << 30)) {
      if (lane == 0) set_error(err, CTR_ERR_BAD_OFFSETS);
      continue;
    }
    const int rel0 = (int)(o0 - S0);
    const int total = (int)(S1 - S0);
    const int fld = bvalid ? (int)(bag / B) : 0;  // this lane's bag's field, once per block
    const uint32_t base_l = (uint32_t)fm.base[fld];
    const uint32_t rows_l = (uint32_t)fm.rows[fld];
    for (int c0 = 0; c0 < total; c0 += 32 * kKeyChunks) {
      int64_t id[kKeyChunks];
#pragma unroll
      for (int q = 0; q < kKeyChunks; ++q) {
        const int kr = c0 + q * 32 + lane;
        id[q] = kr < total ? ids[S0 + kr] : 0;
      }
      uint32_t key[kKeyChunks];
      bool ok[kKeyChunks];
#pragma unroll
      for (int q = 0; q < kKeyChunks; ++q) {
        const int kr = c0 + q * 32 + lane;
        int seg = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {  // largest lane j with rel0_j <= kr
          const int cand = seg + step;
          if (__shfl_sync(kFull, rel0, cand) <= kr) seg = cand;
        }
        const uint32_t base = __shfl_sync(kFull, base_l, seg);
        const uint32_t rows = __shfl_sync(kFull, rows_l, seg);
        ok[q] = kr < total;
        if (ok[q] && (id[q] < 0 || id[q] >= (int64_t)rows)) {
          set_error(err, CTR_ERR_INDEX_OUT_OF_RANGE);
          id[q] = (int64_t)rows - 1;
          ok[q] = rows > 0;  // an ID of an empty table has no row to stand in for it
        }
        key[q] = base + (uint32_t)id[q];
        if (ok[q]) {
          const int64_t i = S0 + kr;
          const int64_t bg = blk * 32 + seg;
          keys[i] = key[q];
          vals[i] = vals_are_pos ? (int32_t)i : (int32_t)bg;
          if (bag_of) bag_of[i] = (int32_t)bg;
        }
      }
      uint32_t word[kKeyChunks];
#pragma unroll
      for (int q = 0; q < kKeyChunks; ++q) word[q] = ok[q] ? ld_l1(bitmap + (key[q] >> 5)) : ~0u;
#pragma unroll
      for (int q = 0; q < kKeyChunks; ++q) {
        const uint32_t bit = 1u << (key[q] & 31);
        if (ok[q] && !(word[q] & bit)) atomicOr(bitmap + (key[q] >> 5), bit);
      }
    }
  }
}

// Set bits per block of kBmWords words.
__global__ void __launch_bounds__(256) bitmap_count_kernel(const uint32_t* __restrict__ bitmap, int64_t W,
                                                           uint32_t* __restrict__ bsum) {
  __shared__ uint32_t warp_tot[8];
  const int64_t w0 = (int64_t)blockIdx.x * kBmWords;
  uint32_t c = 0;
#pragma unroll
  for (int j = 0; j < kBmWords / 256; ++j) {
    const int64_t w = w0 + j * 256 + threadIdx.x;
    if (w < W) c += __popc(bitmap[w]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(kFull, c, o);
  if ((threadIdx.x & 31) == 0) warp_tot[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int q = 0; q < 8; ++q) t += warp_tot[q];
    bsum[blockIdx.x] = t;
  }
}

// pk[w] = (bits of word w, set bits in all earlier words); the unique rows are
// the set bits in order.
__global__ void __launch_bounds__(256) bitmap_pack_kernel(const uint32_t* __restrict__ bitmap, int64_t W,
                                                          const uint32_t* __restrict__ bscan,
                                                          uint2* __restrict__ pk, int64_t* __restrict__ unique_rows) {
  __shared__ uint32_t warp_tot[8];
  constexpr int kPer = kBmWords / 256;
  const int64_t w0 = (int64_t)blockIdx.x * kBmWords + threadIdx.x * kPer;
  uint32_t b[kPer], v[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    b[j] = (w0 + j < W) ? bitmap[w0 + j] : 0u;
    v[j] = __popc(b[j]);
  }
  block_exclusive_scan<uint32_t, 256, kPer>(v, warp_tot);
  const uint32_t base = bscan[blockIdx.x];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int64_t w = w0 + j;
    if (w >= W) break;
    uint32_t r = base + v[j];
    pk[w] = make_uint2(b[j], r);
    for (uint32_t bits = b[j]; bits; bits &= bits - 1) unique_rows[r++] = w * 32 + (__ffs(bits) - 1);
  }
}

// Read-only lookups through L1: under skewed IDs thousands of warps look up
// the same few words at once, which L2 would serve from one slice.
__device__ __forceinline__ uint32_t bitmap_rank(const uint2* __restrict__ pk, uint32_t k) {
  const uint2 e = __ldg(pk + (k >> 5));
  return e.y + __popc(e.x & ((1u << (k & 31)) - 1u));
}

// n_unique, the digit plan of the rank keys, and the per-table unique offsets.
__global__ void bitmap_plan_kernel(const uint32_t* __restrict__ total, int64_t* __restrict__ n_unique,
                                   const __grid_constant__ TableBases tb, int64_t total_rows,
                                   const uint2* __restrict__ pk, int64_t* __restrict__ unique_offsets,
                                   PassPlan* __restrict__ plan) {
  const uint32_t nu = *total;
  if (threadIdx.x == 0) {
    *n_unique = nu;
    int bits = 1;
    while (bits < 32 && (1ull << bits) < (unsigned long long)nu) ++bits;
    const int passes = (bits + kMaxBits - 1) / kMaxBits;
    const int nb = (bits + passes - 1) / passes;
    PassPlan p;
    p.passes = passes;
    for (int q = 0, sh = 0; q < kMaxPasses; ++q) {
      const int pb = q < passes ? (nb < bits - sh ? nb : bits - sh) : 0;
      p.shift[q] = sh;
      p.bits[q] = pb;
      sh += pb;
    }
    *plan = p;
  }
  if (unique_offsets)
    for (int t = threadIdx.x; t <= tb.num_tables; t += blockDim.x) {
      const int64_t k = tb.row_base[t];
      unique_offsets[t] = k >= total_rows ? (int64_t)nu : (int64_t)bitmap_rank(pk, (uint32_t)k);
    }
}

// Run starts of the n_unique ranks set to all ones (coalesced, n_unique read on the device).
__global__ void fill_starts_kernel(int32_t* __restrict__ run_offsets, const int64_t* __restrict__ n_unique) {
  const int64_t nu = *n_unique;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nu; i += (int64_t)gridDim.x * blockDim.x)
    run_offsets[i] = -1;
}

// Rank of every key among the distinct keys (the inverse map, which is also
// the sort's first keys) and the digit histograms of every pass of the device
// plan (per-warp shared histograms, then one global add per block and digit).
// A key outside the tables (a slot an invalid bag left unwritten) is flagged
// and ranked 0.
__device__ __forceinline__ uint32_t rank_or_flag(const uint2* __restrict__ pk, uint32_t k, int64_t total_rows,
                                                 int* err) {
  if ((int64_t)k < total_rows) return bitmap_rank(pk, k);
  set_error(err, CTR_ERR_BAD_OFFSETS);
  return 0u;
}

// 8 keys per thread and round: in the full step, beside the gather and the
// interaction, the sort took 2.86 ms live against 2.92 with 16 and 3.03 with 32
// (and 4 keys: 3.14), one session.
#ifndef CTR_RANK_VEC
#define CTR_RANK_VEC 2
#endif
constexpr int kRankVec = CTR_RANK_VEC;      // uint4 loads per thread and round
constexpr int kRankPer = 4 * kRankVec;      // keys per thread and round

// kRankPer consecutive keys per thread and round: their bitmap lookups are
// independent, so kRankPer are in flight per thread.  `vec` says both arrays
// are 16-byte aligned.
__global__ void __launch_bounds__(256) bitmap_rank_kernel(const uint32_t* __restrict__ keys, int64_t n,
                                                          int64_t total_rows, const uint2* __restrict__ pk,
                                                          const PassPlan* __restrict__ dplan,
                                                          uint32_t* __restrict__ ranks, int vec,
                                                          uint32_t* __restrict__ g_hist, int* err) {
  constexpr int kWarps = 256 / 32;
  __shared__ uint32_t sh[kWarps][kMaxPasses][kMaxDigits];
  for (int i = threadIdx.x; i < kWarps * kMaxPasses * kMaxDigits; i += blockDim.x) (&sh[0][0][0])[i] = 0;
  __syncthreads();
  const PassPlan plan = *dplan;
  const int warp = threadIdx.x >> 5;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t done = 0;
  if (vec) {
    const int64_t nu = n / kRankPer;
    uint4 nxt[kRankVec];  // the next round's keys, loaded while this round's lookups run
    if (t0 < nu) {
#pragma unroll
      for (int v = 0; v < kRankVec; ++v) nxt[v] = ((const uint4*)keys)[t0 * kRankVec + v];
    }
    for (int64_t u = t0; u < nu; u += stride) {
      uint4 k[kRankVec];
#pragma unroll
      for (int v = 0; v < kRankVec; ++v) k[v] = nxt[v];
      if (u + stride < nu) {
#pragma unroll
        for (int v = 0; v < kRankVec; ++v) nxt[v] = ((const uint4*)keys)[(u + stride) * kRankVec + v];
      }
      uint4 r[kRankVec];
#pragma unroll
      for (int v = 0; v < kRankVec; ++v) {
        r[v].x = rank_or_flag(pk, k[v].x, total_rows, err);
        r[v].y = rank_or_flag(pk, k[v].y, total_rows, err);
        r[v].z = rank_or_flag(pk, k[v].z, total_rows, err);
        r[v].w = rank_or_flag(pk, k[v].w, total_rows, err);
      }
      uint4* dst = (uint4*)ranks + u * kRankVec;
#pragma unroll
      for (int v = 0; v < kRankVec; ++v) dst[v] = r[v];
#pragma unroll
      for (int v = 0; v < kRankVec; ++v) {
        const uint32_t rr[4] = {r[v].x, r[v].y, r[v].z, r[v].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int p = 0; p < kMaxPasses; ++p)
            if (p < plan.passes) atomicAdd(&sh[warp][p][(rr[e] >> plan.shift[p]) & ((1u << plan.bits[p]) - 1)], 1u);
      }
    }
    done = nu * kRankPer;
  }
  for (int64_t i = done + t0; i < n; i += stride) {
    const uint32_t r = rank_or_flag(pk, keys[i], total_rows, err);
    ranks[i] = r;
#pragma unroll
    for (int p = 0; p < kMaxPasses; ++p)
      if (p < plan.passes) atomicAdd(&sh[warp][p][(r >> plan.shift[p]) & ((1u << plan.bits[p]) - 1)], 1u);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < plan.passes * kMaxDigits; i += blockDim.x) {
    uint32_t c = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) c += (&sh[w][0][0])[i];
    if (c) atomicAdd(&g_hist[i], c);
  }
}

// Run starts from the sorted ranks (ranks are dense, so the first slot of rank
// r starts run r), and the bag of each sorted position when the sort carried
// positions.
__device__ __forceinline__ void run_slot(const uint32_t* __restrict__ keys, int64_t p, uint32_t k, uint32_t prev,
                                         int64_t n, int64_t nu, int32_t* __restrict__ run_offsets,
                                         const int32_t* __restrict__ sorted_pos, const int32_t* __restrict__ bag_of,
                                         int32_t* __restrict__ sorted_bag, int* err) {
  if ((int64_t)k >= nu) {  // only after an error that left slots unwritten
    set_error(err, CTR_ERR_BAD_OFFSETS);
    return;
  }
  if (run_offsets) {
    if (p == 0 || prev != k) run_offsets[k] = (int32_t)p;
    if (p == n - 1) run_offsets[nu] = (int32_t)n;
  }
  if (sorted_bag) {
    const int32_t q = sorted_pos[p];
    sorted_bag[p] = (q >= 0 && q < n) ? bag_of[q] : -1;
  }
}

// Four consecutive sorted slots per thread (one 16-byte load of their ranks).
__global__ void __launch_bounds__(256) runs_kernel(const uint32_t* __restrict__ keys0,
                                                   const uint32_t* __restrict__ keys1,
                                                   const PassPlan* __restrict__ dplan, int64_t n,
                                                   const int64_t* __restrict__ n_unique,
                                                   int32_t* __restrict__ run_offsets,
                                                   const int32_t* __restrict__ sorted_pos,
                                                   const int32_t* __restrict__ bag_of,
                                                   int32_t* __restrict__ sorted_bag, int* err) {
  const uint32_t* keys = (dplan->passes & 1) ? keys1 : keys0;  // pass p writes buffer (p + 1) & 1
  const int64_t nu = *n_unique;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t n4 = n / 4;
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += stride) {
    const uint4 k = ((const uint4*)keys)[q];
    const int64_t p = q * 4;
    const uint32_t prev = p > 0 ? keys[p - 1] : 0u;
    run_slot(keys, p, k.x, prev, n, nu, run_offsets, sorted_pos, bag_of, sorted_bag, err);
    run_slot(keys, p + 1, k.y, k.x, n, nu, run_offsets, sorted_pos, bag_of, sorted_bag, err);
    run_slot(keys, p + 2, k.z, k.y, n, nu, run_offsets, sorted_pos, bag_of, sorted_bag, err);
    run_slot(keys, p + 3, k.w, k.z, n, nu, run_offsets, sorted_pos, bag_of, sorted_bag, err);
  }
  for (int64_t p = n4 * 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n; p += stride)
    run_slot(keys, p, keys[p], p > 0 ? keys[p - 1] : 0u, n, nu, run_offsets, sorted_pos, bag_of, sorted_bag, err);
}

__global__ void dedup_empty_kernel(int64_t* n_unique, int32_t* run_offsets, int64_t* unique_offsets, int T) {
  *n_unique = 0;
  if (run_offsets) run_offsets[0] = 0;
  if (unique_offsets)
    for (int t = 0; t <= T; ++t) unique_offsets[t] = 0;
}

int key_bits(int64_t total_rows) {
  int b = 1;
  while (b < 32 && ((int64_t)1 << b) < total_rows) ++b;
  return b;
}

// Sort state: per pass, one look-back word per (tile, digit); then the
// per-pass digit histograms and tile counters (uint32, packed two per word).
int64_t state_words(int64_t tiles) {
  return (int64_t)kMaxPasses * tiles * kMaxDigits + (kMaxPasses * kMaxDigits) / 2 + kMaxPasses;
}

bool use_bitmap(int64_t n_ids, int64_t total_rows) { return total_rows <= kBitmapRowsPerId * n_ids; }

int64_t bitmap_words(int64_t total_rows) { return ceil_div(total_rows, (int64_t)32); }

// Workspace of each path (the path follows from the sizes alone).
template <typename WS>
void dedup_layout(WS& ws, int64_t n_ids, int64_t total_rows) {
  const int64_t tiles = ceil_div(n_ids, kRsTile);
  if (use_bitmap(n_ids, total_rows)) {
    const int64_t W = bitmap_words(total_rows);
    const int64_t nblk = ceil_div(W, (int64_t)kBmWords);
    ws.template take<uint32_t>((size_t)n_ids);  // keys A
    ws.template take<uint32_t>((size_t)n_ids);  // keys B
    ws.template take<int32_t>((size_t)n_ids);   // values A
    ws.template take<int32_t>((size_t)n_ids);   // values B
    ws.template take<int32_t>((size_t)n_ids);   // bag of each position (when positions are sorted)
    ws.template take<uint64_t>((size_t)(state_words(tiles) + ceil_div(W, (int64_t)2)));  // sort state + bitmap
    ws.template take<uint2>((size_t)W);         // bitmap words with their prefix counts
    ws.template take<uint32_t>((size_t)nblk);   // set bits per block, then their exclusive scan
    ws.template take<uint32_t>(1);              // n_unique
    ws.template take<PassPlan>(1);
    scan_reserve<uint32_t>(ws, nblk);
    return;
  }
  ws.template take<uint32_t>((size_t)n_ids);           // keys A
  ws.template take<uint32_t>((size_t)n_ids);           // keys B
  ws.template take<int32_t>((size_t)n_ids);            // values scratch
  ws.template take<int32_t>((size_t)n_ids);            // sorted positions if the caller gives none
  ws.template take<int32_t>((size_t)n_ids);            // bag of each position
  ws.template take<uint64_t>((size_t)state_words(tiles));  // look-back words, histograms, tile counters
  ws.template take<uint32_t>((size_t)tiles);           // heads per tile
  scan_reserve<uint32_t>(ws, tiles);
}

void clear_words(uint64_t* p, int64_t words, cudaStream_t s) {
  const int64_t blocks = std::max<int64_t>(1, imin64(ceil_div(words, 256), (int64_t)num_sms() * 8));
  clear_u64_kernel<<<(unsigned)blocks, 256, 0, s>>>(p, words); count_launch();
}

int dedup_bitmap(const int64_t* ids, const int64_t* offsets, int32_t F, int32_t B, const FieldMap& fm,
                 const TableBases& tb, int64_t total_rows, int64_t n_ids, int64_t* unique_rows, int64_t* n_unique,
                 int32_t* inverse, int32_t* sorted_pos, int32_t* sorted_bag, int32_t* run_offsets,
                 int64_t* unique_offsets, int phases, void* ws, size_t ws_bytes, cudaStream_t s) {
  int* err = (int*)ws;
  WsCarver c(ws, ws_bytes);
  const int64_t tiles = ceil_div(n_ids, kRsTile);
  const int64_t W = bitmap_words(total_rows);
  const int64_t nblk = ceil_div(W, (int64_t)kBmWords);
  uint32_t* keys[2] = {c.take<uint32_t>(n_ids), c.take<uint32_t>(n_ids)};
  int32_t* vals[2] = {c.take<int32_t>(n_ids), c.take<int32_t>(n_ids)};
  int32_t* bag_of = c.take<int32_t>(n_ids);
  const int64_t sw = state_words(tiles);
  uint64_t* state = c.take<uint64_t>((size_t)(sw + ceil_div(W, (int64_t)2)));
  uint2* pk = c.take<uint2>((size_t)W);
  uint32_t* bsum = c.take<uint32_t>((size_t)nblk);
  uint32_t* total = c.take<uint32_t>(1);
  PassPlan* dplan = c.take<PassPlan>(1);
  if (!c.ok()) return CTR_ERR_WORKSPACE;
  uint64_t* lookback = state;
  uint32_t* g_hist = (uint32_t*)(state + (int64_t)kMaxPasses * tiles * kMaxDigits);
  uint32_t* tile_counter = g_hist + kMaxPasses * kMaxDigits;
  uint32_t* bitmap = (uint32_t*)(state + sw);
  const int sms = num_sms();
  const int64_t nbags = (int64_t)F * B;
  const int64_t key_blocks = std::max<int64_t>(1, imin64(ceil_div(nbags, 8), (int64_t)sms * 16));

  // the sort carries positions only when the caller asks for them; otherwise
  // it carries bags, and its last pass writes the grouped bags in place
  const bool pos = sorted_pos != nullptr;
  // without positions to carry, the last radix pass writes the run starts itself
  const bool fused_runs = run_offsets != nullptr && !pos;
  if (phases & CTR_DEDUP_PREPARE) {
  clear_words(state, sw + ceil_div(W, (int64_t)2), s);
  if (int st = launch_status()) return st;
  bitmap_keys_kernel<<<(unsigned)key_blocks, 256, 0, s>>>(ids, offsets, F, B, n_ids, fm, keys[1], vals[0],
                                                          pos ? 1 : 0, (pos && sorted_bag) ? bag_of : nullptr,
                                                          bitmap, err); count_launch();
  if (int st = launch_status()) return st;
  bitmap_count_kernel<<<(unsigned)nblk, 256, 0, s>>>(bitmap, W, bsum); count_launch();
  if (int st = launch_status()) return st;
  {
    WsCarver scan_ws = c;
    if (int st = scan_exclusive<uint32_t>(bsum, bsum, nblk, nullptr, total, scan_ws, s)) return st;
  }
  bitmap_pack_kernel<<<(unsigned)nblk, 256, 0, s>>>(bitmap, W, bsum, pk, unique_rows); count_launch();
  if (int st = launch_status()) return st;
  bitmap_plan_kernel<<<1, 256, 0, s>>>(total, n_unique, tb, total_rows, pk, unique_offsets, dplan); count_launch();
  if (int st = launch_status()) return st;
  if (fused_runs) {  // the last radix pass keeps the smallest start offered for each rank
    fill_starts_kernel<<<(unsigned)std::max<int64_t>(1, imin64(ceil_div(n_ids, 1024), (int64_t)sms * 4)), 256, 0, s>>>(
        run_offsets, n_unique); count_launch();
    if (int st = launch_status()) return st;
  }
  // ranks go straight into the caller's inverse map, which the first pass reads
  uint32_t* ranks = inverse ? (uint32_t*)inverse : keys[0];
  {
    // one full wave: the grid-stride rounds split evenly over the resident blocks
    // (a grid of more than the resident blocks ran a second, partly empty wave)
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bitmap_rank_kernel, 256, 0) != cudaSuccess)
      return CTR_ERR_CUDA;
    const int64_t blocks =
        std::max<int64_t>(1, imin64(ceil_div(n_ids, 256 * kRankPer), (int64_t)std::max(per_sm, 1) * sms));
    const int vec = ((uintptr_t)ranks % 16) == 0;
    bitmap_rank_kernel<<<(unsigned)blocks, 256, 0, s>>>(keys[1], n_ids, total_rows, pk, dplan, ranks, vec, g_hist,
                                                        err);
    count_launch();
    if (int st = launch_status()) return st;
  }
  }  // prepare
  if (!(phases & CTR_DEDUP_SORT)) return CTR_OK;
  uint32_t* ranks = inverse ? (uint32_t*)inverse : keys[0];
  int32_t* vals_final = pos ? sorted_pos : sorted_bag;
  const int max_passes = (key_bits(imin64(n_ids, total_rows)) + kMaxBits - 1) / kMaxBits;
  timing_mark(CTR_KERNEL_SORT, true, s);
  for (int p = 0; p < max_passes; ++p) {
    onesweep_kernel<<<(unsigned)tiles, kRsThreads, 0, s>>>(p == 0 ? ranks : keys[p & 1], vals[p & 1], keys[(p + 1) & 1],
                                                           vals[(p + 1) & 1], n_ids, 0, 0, dplan, p, vals_final,
                                                           g_hist + p * kMaxDigits,
                                                           lookback + (int64_t)p * tiles * kMaxDigits,
                                                           tile_counter + p, err, g_lookback_limit_ns.load(),
                                                           fused_runs ? run_offsets : nullptr, n_unique);
    count_launch();
    if (int st = launch_status()) return st;
  }
  timing_mark(CTR_KERNEL_SORT, false, s);
  if ((run_offsets && !fused_runs) || (pos && sorted_bag)) {
    const int64_t blocks = std::max<int64_t>(1, imin64(ceil_div(n_ids, 1024), (int64_t)sms * 8));
    runs_kernel<<<(unsigned)blocks, 256, 0, s>>>(keys[0], keys[1], dplan, n_ids, n_unique, run_offsets, sorted_pos,
                                                 bag_of, pos ? sorted_bag : nullptr, err); count_launch();
  }
  return launch_status();
}

}  // namespace
}  // namespace ctr

using namespace ctr;

extern "C" uint64_t ctr_set_wait_limit_ns(uint64_t ns) { return g_lookback_limit_ns.exchange(ns); }

extern "C" size_t ctr_dedup_workspace_size(int64_t n_ids, int32_t num_fields, int32_t batch, int64_t total_rows) {
  (void)num_fields;
  (void)batch;
  WsSizer s;
  dedup_layout(s, n_ids > 0 ? n_ids : 1, total_rows > 1 ? total_rows : 2);
  return s.used;
}

extern "C" int ctr_dedup(const int64_t* ids, const int64_t* offsets, int32_t num_fields, int32_t batch,
                         const int32_t* bag_to_table, const int64_t* row_base, int32_t num_tables, int64_t n_ids,
                         int64_t* unique_rows, int64_t* n_unique, int32_t* inverse, int32_t* sorted_pos,
                         int32_t* sorted_bag, int32_t* run_offsets, int64_t* unique_offsets, void* ws,
                         size_t ws_bytes, ctr_stream_t stream) {
  return ctr_dedup_phases(ids, offsets, num_fields, batch, bag_to_table, row_base, num_tables, n_ids, unique_rows,
                          n_unique, inverse, sorted_pos, sorted_bag, run_offsets, unique_offsets, CTR_DEDUP_ALL, ws,
                          ws_bytes, stream);
}

extern "C" int ctr_dedup_phases(const int64_t* ids, const int64_t* offsets, int32_t num_fields, int32_t batch,
                                const int32_t* bag_to_table, const int64_t* row_base, int32_t num_tables,
                                int64_t n_ids, int64_t* unique_rows, int64_t* n_unique, int32_t* inverse,
                                int32_t* sorted_pos, int32_t* sorted_bag, int32_t* run_offsets,
                                int64_t* unique_offsets, int32_t phases, void* ws, size_t ws_bytes,
                                ctr_stream_t stream) {
  cudaStream_t s = (cudaStream_t)stream;
  if (phases < CTR_DEDUP_PREPARE || phases > CTR_DEDUP_ALL) return CTR_ERR_INVALID_ARG;
  if (!offsets || !bag_to_table || !row_base || !unique_rows || !n_unique) return CTR_ERR_INVALID_ARG;
  if (num_fields <= 0 || batch <= 0 || num_tables <= 0) return CTR_ERR_INVALID_ARG;
  if (num_fields > CTR_MAX_FIELDS || num_tables > CTR_MAX_TABLES) return CTR_ERR_UNSUPPORTED;
  if (n_ids < 0 || (n_ids > 0 && !ids)) return CTR_ERR_INVALID_ARG;
  if (n_ids >= ((int64_t)1 << 31)) return CTR_ERR_UNSUPPORTED;
  if (row_base[0] != 0) return CTR_ERR_INVALID_ARG;
  for (int t = 0; t < num_tables; ++t)
    if (row_base[t + 1] < row_base[t]) return CTR_ERR_INVALID_ARG;
  const int64_t total_rows = row_base[num_tables];
  if (total_rows > ((int64_t)1 << 32)) return CTR_ERR_UNSUPPORTED;
  FieldMap fm;
  for (int f = 0; f < num_fields; ++f) {
    int t = bag_to_table[f];
    if (t < 0 || t >= num_tables) return CTR_ERR_INVALID_ARG;
    fm.base[f] = row_base[t];
    fm.rows[f] = row_base[t + 1] - row_base[t];
  }
  if (!ws_valid(ws, ws_bytes, ctr_dedup_workspace_size(n_ids, num_fields, batch, total_rows)))
    return CTR_ERR_WORKSPACE;
  int* err = (int*)ws;
  TableBases tb;
  tb.num_tables = num_tables;
  for (int t = 0; t <= num_tables; ++t) tb.row_base[t] = row_base[t];

  if (n_ids == 0) {
    if (phases & CTR_DEDUP_PREPARE) {
      dedup_empty_kernel<<<1, 1, 0, s>>>(n_unique, run_offsets, unique_offsets, num_tables); count_launch();
    }
    return launch_status();
  }

  if (use_bitmap(n_ids, total_rows))
    return dedup_bitmap(ids, offsets, num_fields, batch, fm, tb, total_rows, n_ids, unique_rows, n_unique, inverse,
                        sorted_pos, sorted_bag, run_offsets, unique_offsets, phases, ws, ws_bytes, s);

  WsCarver c(ws, ws_bytes);
  const int64_t tiles = ceil_div(n_ids, kRsTile);
  const int bits = key_bits(total_rows);
  const int passes = (bits + kMaxBits - 1) / kMaxBits;
  const int nb = (bits + passes - 1) / passes;
  uint32_t* keys[2] = {c.take<uint32_t>(n_ids), c.take<uint32_t>(n_ids)};
  int32_t* vscratch = c.take<int32_t>(n_ids);
  int32_t* vfinal_ws = c.take<int32_t>(n_ids);
  int32_t* bag_of = c.take<int32_t>(n_ids);
  uint64_t* state = c.take<uint64_t>((size_t)state_words(tiles));
  uint32_t* tile_heads = c.take<uint32_t>(tiles);
  if (!c.ok()) return CTR_ERR_WORKSPACE;
  int32_t* vfinal = sorted_pos ? sorted_pos : vfinal_ws;
  uint64_t* lookback = state;
  uint32_t* g_hist = (uint32_t*)(state + (int64_t)kMaxPasses * tiles * kMaxDigits);
  uint32_t* tile_counter = g_hist + kMaxPasses * kMaxDigits;

  PassPlan plan;
  plan.passes = passes;
  for (int p = 0, sh = 0; p < kMaxPasses; ++p) {
    const int pb = p < passes ? std::min(nb, bits - sh) : 0;
    plan.shift[p] = sh;
    plan.bits[p] = pb;
    sh += pb;
  }
  const int sms = num_sms();
  if (phases & CTR_DEDUP_PREPARE) {
    clear_words(state, state_words(tiles), s);
    if (int st = launch_status()) return st;
    const int64_t nbags = (int64_t)num_fields * batch;
    int64_t blocks = imin64(ceil_div(nbags, 8), (int64_t)sms * 16);
    keygen_kernel<<<(unsigned)std::max<int64_t>(blocks, 1), 256, 0, s>>>(ids, offsets, num_fields, batch, n_ids, fm,
                                                                        keys[0], bag_of, plan, g_hist, err); count_launch();
    if (int st = launch_status()) return st;
  }
  if (!(phases & CTR_DEDUP_SORT)) return CTR_OK;
  const int32_t* vin = nullptr;
  timing_mark(CTR_KERNEL_SORT, true, s);
  for (int p = 0; p < passes; ++p) {
    int32_t* vout = ((passes - 1 - p) % 2 == 0) ? vfinal : vscratch;
    onesweep_kernel<<<(unsigned)tiles, kRsThreads, 0, s>>>(keys[p & 1], vin, keys[(p + 1) & 1], vout, n_ids,
                                                           plan.shift[p], plan.bits[p], nullptr, p, nullptr,
                                                           g_hist + p * kMaxDigits,
                                                           lookback + (int64_t)p * tiles * kMaxDigits,
                                                           tile_counter + p, err, g_lookback_limit_ns.load(),
                                                           nullptr, nullptr);
    count_launch();
    if (int st = launch_status()) return st;
    vin = vout;
  }
  timing_mark(CTR_KERNEL_SORT, false, s);
  const uint32_t* skeys = keys[passes & 1];
  unique_count_kernel<<<(unsigned)tiles, kRsThreads, 0, s>>>(skeys, n_ids, tile_heads); count_launch();
  if (int st = launch_status()) return st;
  {
    WsCarver scan_ws = c;
    if (int st = scan_exclusive<uint32_t>(tile_heads, tile_heads, tiles, nullptr, nullptr, scan_ws, s)) return st;
  }
  unique_write_kernel<<<(unsigned)tiles, kRsThreads, 0, s>>>(skeys, vfinal, n_ids, tile_heads, tb, bag_of,
                                                             unique_rows, n_unique, inverse, sorted_bag, run_offsets,
                                                             unique_offsets); count_launch();
  return launch_status();
}
