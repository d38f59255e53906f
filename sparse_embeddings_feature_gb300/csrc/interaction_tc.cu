// a3 (bf16). Pairwise dot interaction on the 5th-generation tensor cores.
//
// Sources: "Meta DLRM", section 02 (dot products between all pairs of the
// embedding vectors and the processed dense features, cross terms only);
// "DHEN" notes, section 3.1, Eq. (3) (concatenated with the dense features).
// The DHEN notes place this module on A100-class hardware; this kernel is a
// new design for sm_103a.
//
// Per sample the interaction is the Gram matrix X X^T of n <= 32 vectors.  S =
// floor(128 / n) samples are stacked into one 128-row tile, so one
// tcgen05.mma (M = 128, N = round_up(S n, 16), K = 16 per instruction) computes
// the tile's Gram matrix, whose S diagonal n x n blocks are the samples' own.
// A and B are the same shared-memory tile (both K-major, 128-byte swizzle),
// loaded by TMA straight from X viewed as [B*n, d].  The accumulator lives in
// TMEM (fp32, double-buffered); the epilogue reads the columns of each warp's
// diagonal blocks with tcgen05.ld, rounds the samples' own n x n blocks to
// bf16 into shared memory (only the diagonal blocks: S n x n values), and
// writes the samples' output rows from them in output order with coalesced
// stores: the dense pass-through first (first two modes), then the products
// the mode emits from each diagonal block (the strict lower triangle; or with
// the diagonal, "DHEN" notes section 3.1; or the whole block, the Gram matrix
// of "DHEN" notes section 3.3, Eq. (7)).
//
// Roles (persistent CTAs, two per SM where shared memory allows): warp 0
// issues TMA loads, warp 1 owns TMEM and issues the MMAs, and two epilogue
// groups of four warps (warps 2..5 and 6..9) take alternate tiles, each with
// its own TMEM accumulator and shared-memory blocks, so one group's output
// writes overlap the other's accumulator read-back (with one group the
// epilogue, about 1.7 us per tile, bounded the kernel).  Every mbarrier wait
// is bounded by a wall-clock limit; on expiry the kernel records
// CTR_ERR_TIMEOUT, waits (bounded) for its own copies and MMAs, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "tma.cuh"

namespace ctr {
namespace {

constexpr int kTcEpiWarps = 4;                        // warps per epilogue group
constexpr int kTcEpiGroups = 2;                       // groups, one per TMEM accumulator
constexpr int kTcThreads = 64 + 32 * kTcEpiWarps * kTcEpiGroups;
constexpr uint32_t kTmemCols = 256;
// Shared memory asked for per CTA, at least: more than a third of the SM's
// 228 KB, so no more than two CTAs (2 x 256 TMEM columns) are ever resident.
constexpr int kTcSmemFloor = 80 * 1024;
constexpr int kDensePre = 2;  // dense-vector pieces per epilogue thread loaded early

struct TcParams {
  int32_t batch, n, d, S, rows, N, kb, stages, W, mode, GS;
  int32_t aligned;  // 1: every sample at a 32-row boundary of the tile (17 <= n <= 32)
  uint32_t stage_bytes, tx_bytes, epi_bytes;
  const __nv_bfloat16* X;
  __nv_bfloat16* out;
  int* err;
};

// K-major operand, 128-byte swizzle: 8-row core groups 1024 B apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);     // start address
  d |= (uint64_t)1 << 16;                     // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset
  d |= (uint64_t)1 << 46;                     // descriptor version
  d |= (uint64_t)2 << 61;                     // SWIZZLE_128B
  return d;
}

// kind::f16 instruction descriptor: bf16 x bf16 -> fp32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive accumulator columns of this warp's 32 lanes, then the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Named barrier 1 over the 128 epilogue threads, returning the OR of `pred`.
// Named barrier `id` over one epilogue group's 128 threads, returning the OR of `pred`.
__device__ __forceinline__ bool epi_any(uint32_t id, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void epi_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__global__ void __launch_bounds__(kTcThreads, 1) interaction_bf16_tc_kernel(const TcParams p,
                                                                           const __grid_constant__ CUtensorMap map) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[2 * 8 + 4];
  __shared__ uint32_t tmem_base_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzled tiles need 1024-byte alignment
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t full0 = smem_u32(&bars[0]);
  const uint32_t empty0 = smem_u32(&bars[8]);
  const uint32_t tfull0 = smem_u32(&bars[16]);
  const uint32_t tempty0 = smem_u32(&bars[18]);
  const int64_t ntiles = ceil_div(p.batch, p.S);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, kTcEpiWarps);
    }
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int64_t it = 0;
      for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int s = (int)(it % p.stages);
        const uint32_t ph = (uint32_t)((it / p.stages) & 1);
        if (!mbar_wait(empty0 + 8 * s, ph ^ 1)) {
          set_error(p.err, CTR_ERR_TIMEOUT);
          atomicExch(&abort_flag, 1);
          break;
        }
        if (*(volatile int*)&abort_flag) break;
        mbar_expect_tx(full0 + 8 * s, p.tx_bytes);
        const uint32_t dst = base + (uint32_t)s * p.stage_bytes;
        const int32_t row0 = (int32_t)(t * p.S * p.n);
        for (int kb = 0; kb < p.kb; ++kb) {
          if (p.aligned) {  // one 32-row box per sample (rows past the sample's n are never read back)
            for (int q = 0; q < 4; ++q)
              tma_load_2d(dst + kb * 16384u + q * 4096u, &map, kb * 64, row0 + q * p.n, full0 + 8 * s);
          } else {
            tma_load_2d(dst + kb * 16384u, &map, kb * 64, row0, full0 + 8 * s);
          }
        }
      }
      // drain: every issued load must have landed before the CTA can exit
      const int64_t issued = it;
      for (int s = 0; s < p.stages && s < issued; ++s) {
        const int64_t last = issued - 1 - ((issued - 1 - s) % p.stages);  // last iteration using stage s
        if (!mbar_wait(full0 + 8 * s, (uint32_t)((last / p.stages) & 1))) set_error(p.err, CTR_ERR_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, p.N);
      int64_t it = 0;
      for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int s = (int)(it % p.stages);
        const uint32_t ph = (uint32_t)((it / p.stages) & 1);
        const int acc = (int)(it & 1);
        const uint32_t aph = (uint32_t)((it >> 1) & 1);
        if (!mbar_wait(tempty0 + 8 * acc, aph ^ 1) || !mbar_wait(full0 + 8 * s, ph)) {
          set_error(p.err, CTR_ERR_TIMEOUT);
          atomicExch(&abort_flag, 1);
          break;
        }
        if (*(volatile int*)&abort_flag) break;
        fence_after();
        const uint32_t a0 = base + (uint32_t)s * p.stage_bytes;
        const uint32_t d_tmem = tmem + (uint32_t)acc * 128u;
        uint32_t accumulate = 0;
        for (int kb = 0; kb < p.kb; ++kb)
          for (int k = 0; k < 4; ++k) {
            const uint64_t desc = smem_desc_sw128(a0 + kb * 16384u + k * 32u);
            mma_bf16(d_tmem, desc, desc, idesc, accumulate);
            accumulate = 1;
          }
        mma_commit(empty0 + 8 * s);
        mma_commit(tfull0 + 8 * acc);
      }
      // drain: the last commits must have arrived before TMEM is freed
      const int64_t issued = it;
      for (int a = 0; a < 2 && a < issued; ++a) {
        const int64_t last = issued - 1 - ((issued - 1 - a) % 2);
        if (!mbar_wait(tfull0 + 8 * a, (uint32_t)((last >> 1) & 1))) set_error(p.err, CTR_ERR_TIMEOUT);
      }
    }
  } else {
    // ---------------- epilogue (two groups of warps 2..5 and 6..9) ----------------
    // Phase A: each thread (one tile row = one TMEM lane) converts the
    // accumulator columns of its own sample's diagonal block to bf16 into the
    // group's shared blocks; the tile's dense vectors go to shared memory.
    // Phase B: the group's 128 threads write the tile's output rows in output
    // order, each product read from the blocks through the mode's source table.
    const int g = (warp - 2) / kTcEpiWarps;  // epilogue group: tiles it = g, g + 2, ...
    const uint32_t gbar = 1u + (uint32_t)g;  // the group's named barrier
    const int q = warp & 3;                  // TMEM lane quarter this warp may read
    const int row = q * 32 + lane;           // tile row = TMEM lane
    const int tid = threadIdx.x - 64 - g * 32 * kTcEpiWarps;  // 0..127 within the group
    // the accumulator columns this warp's rows need: the diagonal blocks of the
    // samples its 32 rows belong to, read 32 columns at a time (columns past N
    // lie inside the accumulator's 128 and are never read back)
    const int c_lo = ((q * 32) / p.n * p.n) & ~31;
    const int c_hi = min(p.N, ((q * 32 + 31) / p.n + 1) * p.n);
    const int dd = p.mode != 2 ? p.d : 0;  // dense pass-through width of an output row
    const int dchunks = dd / 8;            // its 16-byte pieces
    const int nn = p.aligned ? 32 * 32 : p.n * p.n;  // a sample's block in shared memory
    int16_t* ptab = (int16_t*)(base_ptr + (size_t)p.stages * p.stage_bytes);
    uint8_t* gsm = base_ptr + (size_t)p.stages * p.stage_bytes + align_up((size_t)(p.W - dd) * 2, 16) +
                   (size_t)g * p.epi_bytes;
    // [S][n][n] bf16 (sample s, row i, column j); aligned: [S][32][32], the
    // 16-byte pieces of row i rotated by (i / 2) mod 4 so the rows' vector
    // stores spread over the banks
    uint16_t* blocks = (uint16_t*)gsm;
    uint16_t* dsm = blocks + align_up((size_t)p.S * nn, 8);  // [S][dd] bf16
    // source of product slot u of a sample, relative to its block:
    //   mode 0: pair (r, j), j < r, at u = r(r-1)/2 + j;  mode 1: j <= r at
    //   u = r(r+1)/2 + j;  mode 2: (u / n, u mod n)
    for (int u = threadIdx.x - 64; u < p.W - dd; u += 32 * kTcEpiWarps * kTcEpiGroups) {
      int r = 0, j = 0;
      if (p.mode == 2) {
        r = u / p.n;
        j = u - r * p.n;
      } else {
        const int sh = p.mode == 0 ? -1 : 1;  // row r starts at r(r + sh)/2
        while ((r + 1) * (r + 1 + sh) / 2 <= u) ++r;
        j = u - r * (r + sh) / 2;
      }
      ptab[u] = (int16_t)(p.aligned ? r * 32 + ((((j >> 3) ^ (r >> 1)) & 3) << 3) + (j & 7) : r * p.n + j);
    }
    epi_sync(3, 32 * kTcEpiWarps * kTcEpiGroups);  // the table is complete for both groups
    // this thread's sample and row within it (rows past S n hold no sample)
    const int my_s = row / p.n, my_i = row - my_s * p.n;
    const bool my_row = row < p.S * p.n;
    for (int64_t it = g;; it += kTcEpiGroups) {
      const int64_t t = blockIdx.x + it * (int64_t)gridDim.x;
      if (t >= ntiles) break;
      const int acc = (int)(it & 1);  // = g: each group owns one accumulator
      const uint32_t aph = (uint32_t)((it >> 1) & 1);
      const int nvalid = (int)imin64(p.S, p.batch - t * p.S);
      // the tile's dense vectors: the first kDensePre pieces per thread are
      // loaded before the wait for the accumulator, so their latency overlaps it
      const int dense_n = nvalid * dchunks;
      uint4 dpre[kDensePre];
#pragma unroll
      for (int m = 0; m < kDensePre; ++m) {
        const int idx = tid + m * 128;
        if (idx < dense_n) {
          const int ks = idx / dchunks, c = idx - ks * dchunks;
          dpre[m] = *(const uint4*)(p.X + ((t * p.S + ks) * (int64_t)p.n) * p.d + c * 8);
        }
      }
      const bool ok = mbar_wait(tfull0 + 8 * acc, aph);
      if (!ok) {
        set_error(p.err, CTR_ERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
      }
      // one decision for the group's 128 threads (also: the blocks and the
      // dense vectors of its previous tile have been written out)
      if (epi_any(gbar, !ok || *(volatile int*)&abort_flag)) break;
      fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * 128u;
      if (p.aligned) {
        // warp q holds sample q's rows, and its block is accumulator columns 32q .. 32q + 31:
        // one read, then the row as four 16-byte stores
        uint32_t v[32];
        tmem_ld32(tbase + (uint32_t)(q * 32), v);
        if (q < nvalid && lane < p.n) {
          uint4* brow4 = (uint4*)(blocks + (size_t)q * nn + (size_t)lane * 32);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __nv_bfloat162 h2 =
                  __floats2bfloat162_rn(__uint_as_float(v[8 * c + 2 * k]), __uint_as_float(v[8 * c + 2 * k + 1]));
              w[k] = *(const uint32_t*)&h2;
            }
            brow4[c ^ ((lane >> 1) & 3)] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      uint16_t* brow = blocks + (size_t)my_s * nn + (size_t)my_i * p.n;  // this row of its sample's block
      const int b0 = my_s * p.n;                                       // the block's first column
      for (int c0 = c_lo; c0 < (p.aligned ? c_lo : c_hi); c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tbase + (uint32_t)c0, v);
        if (my_row) {
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const int j = c0 + cc - b0;
            if (j >= 0 && j < p.n) {
              const __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(v[cc]));
              brow[j] = *(const uint16_t*)&h;
            }
          }
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);  // the accumulator is free for the MMA two tiles on
      for (int idx = tid; idx < dense_n; idx += 128) {
        const int m = idx / 128;
        const int ks = idx / dchunks, c = idx - ks * dchunks;
        uint4 w;
        if (m < kDensePre) {
#pragma unroll
          for (int mm = 0; mm < kDensePre; ++mm)
            if (mm == m) w = dpre[mm];
        } else {
          w = *(const uint4*)(p.X + ((t * p.S + ks) * (int64_t)p.n) * p.d + c * 8);
        }
        *(uint4*)(dsm + (size_t)ks * dd + c * 8) = w;
      }
      epi_sync(gbar, 128);  // the blocks and the dense vectors are complete
      // Phase B: output element e of the tile is slot e mod W of sample e / W
      const int elems = nvalid * p.W;
      __nv_bfloat16* dst = p.out + t * p.S * (int64_t)p.W;
      if (((uintptr_t)dst % 8) == 0 && (elems % 4) == 0) {
        for (int e = 4 * tid; e < elems; e += 4 * 128) {
          int ks = e / p.W, u = e - ks * p.W;
          uint32_t h[4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            h[x] = u < dd ? dsm[ks * dd + u] : blocks[ks * nn + ptab[u - dd]];
            if (++u == p.W) {
              u = 0;
              ++ks;
            }
          }
          *(uint2*)(dst + e) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        }
      } else {
        uint16_t* dst16 = (uint16_t*)dst;
        for (int e = tid; e < elems; e += 128) {
          const int ks = e / p.W, u = e - ks * p.W;
          dst16[e] = u < dd ? dsm[ks * dd + u] : blocks[ks * nn + ptab[u - dd]];
        }
      }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

}  // namespace

bool interaction_bf16_tc_supported(int32_t n, int32_t d) { return n >= 2 && n <= 32 && d % 64 == 0 && d <= 256; }

int interaction_bf16_tc(const void* X, int32_t batch, int32_t n, int32_t d, int mode, void* out, int* err,
                        cudaStream_t s) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return CTR_ERR_CUDA;
  TcParams p;
  p.batch = batch;
  p.n = n;
  p.d = d;
  // 17 <= n <= 32: four samples per tile, each at a 32-row boundary, so each
  // epilogue warp's TMEM lanes are one sample and its block one aligned
  // 32-column read; else S = floor(128 / n) samples packed back to back
  p.aligned = n >= 17 ? 1 : 0;
  p.S = p.aligned ? 4 : 128 / n;
  p.rows = p.aligned ? 128 : p.S * n;
  p.N = (p.rows + 15) / 16 * 16;
  p.kb = d / 64;
  p.stage_bytes = 16384u * p.kb;
  p.tx_bytes = (uint32_t)(128 * p.rows * p.kb);
  p.stages = std::max(2, std::min(4, (int)((160 * 1024) / p.stage_bytes)));
  p.mode = mode;
  p.W = mode == 0 ? d + n * (n - 1) / 2 : (mode == 1 ? d + n * (n + 1) / 2 : n * n);
  // epilogue shared memory: the product source table (shared), then per group
  // the samples' diagonal blocks (S n x n bf16) and dense vectors (S x d bf16)
  p.GS = n;
  const int dd = mode != 2 ? d : 0;
  const size_t block_elems = p.aligned ? (size_t)32 * 32 : (size_t)n * n;
  p.epi_bytes = (uint32_t)align_up((align_up((size_t)p.S * block_elems, 8) + (size_t)p.S * dd) * 2, 16);
  p.X = (const __nv_bfloat16*)X;
  p.out = (__nv_bfloat16*)out;
  p.err = err;

  CUtensorMap map;
  cuuint64_t gdim[2] = {(cuuint64_t)d, (cuuint64_t)batch * n};
  cuuint64_t gstride[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)(p.aligned ? 32 : p.rows)};
  cuuint32_t estride[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), gdim, gstride, box, estride,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CTR_ERR_CUDA;
  // Two CTAs per SM where they fit: each holds kTmemCols of the SM's 512 TMEM
  // columns, and the shared memory asked for keeps a third off the SM (its
  // allocation would wait for one of the two to exit).
  const size_t need = 1024 + (size_t)p.stages * p.stage_bytes + align_up((size_t)(p.W - dd) * 2, 16) +
                      (size_t)kTcEpiGroups * p.epi_bytes;
  const size_t smem = std::max(need, (size_t)kTcSmemFloor);
  auto kern = interaction_bf16_tc_kernel;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return CTR_ERR_CUDA;
  // resident CTAs per SM from the SM's shared memory and registers (the
  // occupancy query reports one for this kernel where both allow two)
  int per_sm = 1;
  {
    int dev = 0, smem_sm = 0, reserved = 0, regs_sm = 0;
    cudaFuncAttributes fa;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, kern) != cudaSuccess)
      return CTR_ERR_CUDA;
    const size_t per_cta_smem = smem + fa.sharedSizeBytes + (size_t)reserved;
    const int regs_cta = kTcThreads * ((fa.numRegs + 7) / 8 * 8);
    per_sm = (int)std::min<size_t>(smem_sm / per_cta_smem, (size_t)(regs_sm / std::max(regs_cta, 1)));
    per_sm = std::max(1, std::min(per_sm, (int)(512 / kTmemCols)));
  }
  const int64_t ntiles = ceil_div(batch, p.S);
  const int grid = (int)std::max<int64_t>(1, imin64(ntiles, (int64_t)per_sm * num_sms()));
  kern<<<grid, kTcThreads, smem, s>>>(p, map); count_launch();
  return launch_status();
}

}  // namespace ctr
