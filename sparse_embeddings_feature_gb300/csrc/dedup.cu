// a1. Batch ID dedup into the "virtual sparse feature" index.
//
// Source: "How TensorNet Supercharges Sparse Feature Training on TensorFlow",
// Core Optimizations, embedding_lookup: collect the batch's IDs, sort them and
// give each distinct ID a continuous index.
//
// GPU design (sm_103a, one GPU):
//   keygen     warp per bag: key = row_base[table(f)] + id (32-bit global row),
//              bag id per position; IDs outside their table are flagged.
//   LSD radix  ceil(bits(total_rows) / 8) passes of <= 8 bits.  Each pass is
//              reduce-then-scan: per-tile digit histograms (digit-major), one
//              device-wide exclusive scan over them, then a stable scatter.
//              Stable ranking inside a tile uses __match_any_sync per 32 keys
//              and per-warp digit counters; the tile is reordered in shared
//              memory first so the global writes are coalesced runs.  No
//              block waits on another block.
//   unique     head flags, per-tile head counts, exclusive scan, then ranks:
//              unique_rows, run_offsets, inverse (scatter), sorted_bag
//              (gather of the bag of each sorted position), unique_offsets.
#include <algorithm>

#include "common.cuh"
#include "scan.cuh"

namespace ctr {
namespace {

constexpr int kRsThreads = 256;
constexpr int kRsWarps = kRsThreads / 32;
constexpr int kRsItems = 16;                      // keys per lane per tile
constexpr int kRsTile = kRsThreads * kRsItems;    // 4096 keys
constexpr int kRsWarpKeys = 32 * kRsItems;        // 512 keys per warp
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
constexpr uint64_t kLookbackLimitNs = 1000000000ull;  // 1 s

// One radix pass in one kernel (single-pass, after Adinets and Merrill's
// Onesweep): a block takes the next tile in launch order, ranks its keys
// stably (per 32 keys __match_any_sync groups equal digits; per-warp digit
// counters order the warps), publishes its per-digit counts, and finds the
// counts of all earlier tiles by decoupled look-back: a predecessor's word
// holds either its own count or its inclusive prefix, so the walk stops at
// the first inclusive prefix; each thread reads kLbWindow predecessors per
// round trip.  Lanes holding equal digits are found with one ballot per digit
// bit (votes, not the match unit).  Tiles are taken in order, so a block only
// ever waits on blocks that started before it; each wait is bounded by a
// wall-clock limit, after which the block records CTR_ERR_TIMEOUT and keeps
// its writes inside the output.  vals_in == nullptr means the values are
// the positions 0..n-1 (first pass).
__global__ void __launch_bounds__(kRsThreads) onesweep_kernel(
    const uint32_t* __restrict__ keys_in, const int32_t* __restrict__ vals_in, uint32_t* __restrict__ keys_out,
    int32_t* __restrict__ vals_out, int64_t n, int shift, int nbits, const uint32_t* __restrict__ g_hist,
    uint64_t* __restrict__ lookback, uint32_t* __restrict__ tile_counter, int* err) {
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
  const int64_t tile = tile_sh;

  const int64_t tile_base = tile * kRsTile;
  const int64_t base = tile_base + (int64_t)warp * kRsWarpKeys;
  const unsigned lt = lanemask_lt();
  uint32_t key[kRsItems];
  int32_t val[kRsItems];
  uint32_t rank[kRsItems];
#pragma unroll
  for (int r = 0; r < kRsItems; ++r) {
    const int64_t idx = base + r * 32 + lane;
    const bool valid = idx < n;
    key[r] = valid ? keys_in[idx] : 0u;
    val[r] = valid ? (vals_in ? vals_in[idx] : (int32_t)idx) : 0;
    const uint32_t dg = valid ? digit_of(key[r], shift, mask) : 0u;
    unsigned peers = __ballot_sync(kFull, valid);
#pragma unroll
    for (int b = 0; b < kMaxBits; ++b) {
      if (b < nbits) {
        const unsigned m = __ballot_sync(kFull, (dg >> b) & 1u);
        peers &= ((dg >> b) & 1u) ? m : ~m;
      }
    }
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
  uint64_t* my_word = lookback + tile * kMaxDigits + dg;
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
    int64_t j = tile - 1;
    uint64_t t0 = 0;
    while (j >= 0) {
      uint64_t w[kLbWindow];
#pragma unroll
      for (int q = 0; q < kLbWindow; ++q) w[q] = (j - q >= 0) ? ld_relaxed(lookback + (j - q) * kMaxDigits + dg)
                                                             : kFlagInclusive;
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
        else if (t - t0 > kLookbackLimitNs) {
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
  const int count = (int)imin64(kRsTile, n - tile_base);
  for (int i = threadIdx.x; i < count; i += kRsThreads) {
    const uint32_t k = skeys[i];
    const uint32_t d = digit_of(k, shift, mask);
    const int64_t dest = (int64_t)glob_start[d] + (i - (int64_t)tile_start[d]);
    if (dest >= 0 && dest < n) {  // always true unless a look-back timed out
      keys_out[dest] = k;
      vals_out[dest] = svals[i];
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

// Ranks and outputs of one tile of sorted keys.  The tile's 4096 slots are read
// as 16 coalesced rows of 256 (slot = row * 256 + thread): head flags come from
// one ballot per warp and row, and a scan of the 16 x 8 per-warp head counts
// gives every slot its rank.
__global__ void __launch_bounds__(kRsThreads) unique_write_kernel(
    const uint32_t* __restrict__ skeys, const int32_t* __restrict__ spos, int64_t n,
    const uint32_t* __restrict__ tile_base_scan, const __grid_constant__ TableBases tb,
    const int32_t* __restrict__ bag_of, int64_t* __restrict__ unique_rows, int64_t* __restrict__ n_unique,
    int32_t* __restrict__ inverse, int32_t* __restrict__ sorted_bag, int32_t* __restrict__ run_offsets,
    int64_t* __restrict__ unique_offsets) {
  constexpr int kRows = kRsTile / kRsThreads;  // 16
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
  if (warp == 0) {  // exclusive scan of the 128 counts, 4 per lane, in slot order
    uint32_t v[4], sum = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[q] = cnt[lane * 4 + q];
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
    for (int q = 0; q < 4; ++q) {
      cnt[lane * 4 + q] = run;
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

template <typename WS>
void dedup_layout(WS& ws, int64_t n_ids, int64_t total_rows) {
  const int64_t tiles = ceil_div(n_ids, kRsTile);
  const int bits = key_bits(total_rows);
  const int passes = (bits + kMaxBits - 1) / kMaxBits;
  const int nb = (bits + passes - 1) / passes;
  ws.template take<uint32_t>((size_t)n_ids);           // keys A
  ws.template take<uint32_t>((size_t)n_ids);           // keys B
  ws.template take<int32_t>((size_t)n_ids);            // values scratch
  ws.template take<int32_t>((size_t)n_ids);            // sorted positions if the caller gives none
  ws.template take<int32_t>((size_t)n_ids);            // bag of each position
  ws.template take<uint64_t>((size_t)state_words(tiles));  // look-back words, histograms, tile counters
  ws.template take<uint32_t>((size_t)tiles);           // heads per tile
  scan_reserve<uint32_t>(ws, tiles);
  (void)nb;
}

}  // namespace
}  // namespace ctr

using namespace ctr;

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
  cudaStream_t s = (cudaStream_t)stream;
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
    dedup_empty_kernel<<<1, 1, 0, s>>>(n_unique, run_offsets, unique_offsets, num_tables); count_launch();
    return launch_status();
  }

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
  clear_u64_kernel<<<(unsigned)std::max<int64_t>(1, imin64(ceil_div(state_words(tiles), 256), (int64_t)sms * 8)),
                     256, 0, s>>>(state, state_words(tiles)); count_launch();
  if (int st = launch_status()) return st;
  const int64_t nbags = (int64_t)num_fields * batch;
  {
    int64_t blocks = imin64(ceil_div(nbags, 8), (int64_t)sms * 16);
    keygen_kernel<<<(unsigned)std::max<int64_t>(blocks, 1), 256, 0, s>>>(ids, offsets, num_fields, batch, n_ids, fm,
                                                                        keys[0], bag_of, plan, g_hist, err); count_launch();
    if (int st = launch_status()) return st;
  }
  const int32_t* vin = nullptr;
  timing_mark(CTR_KERNEL_SORT, true, s);
  for (int p = 0; p < passes; ++p) {
    int32_t* vout = ((passes - 1 - p) % 2 == 0) ? vfinal : vscratch;
    onesweep_kernel<<<(unsigned)tiles, kRsThreads, 0, s>>>(keys[p & 1], vin, keys[(p + 1) & 1], vout, n_ids,
                                                           plan.shift[p], plan.bits[p], g_hist + p * kMaxDigits,
                                                           lookback + (int64_t)p * tiles * kMaxDigits,
                                                           tile_counter + p, err); count_launch();
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
