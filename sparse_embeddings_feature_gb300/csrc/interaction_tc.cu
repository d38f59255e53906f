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
// TMEM (fp32, double-buffered); the epilogue reads it with tcgen05.ld, keeps
// the products its mode emits from each diagonal block (the strict lower
// triangle; or with the diagonal, "DHEN" notes section 3.1; or the whole
// block, the Gram matrix of "DHEN" notes section 3.3, Eq. (7)), rounds to
// bf16, adds the dense pass-through (first two modes) and writes the samples'
// output rows with coalesced stores through a shared-memory staging buffer.
//
// Roles (persistent CTA, one per SM): warp 0 issues TMA loads, warp 1 owns
// TMEM and issues the MMAs, warps 2..5 run the epilogue.  Every mbarrier wait
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

constexpr int kTcThreads = 192;
constexpr int kTcEpiWarps = 4;
constexpr uint32_t kTmemCols = 256;

struct TcParams {
  int32_t batch, n, d, S, rows, N, kb, stages, W, mode;
  uint32_t stage_bytes, tx_bytes, staging_bytes;
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

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Named barrier 1 over the 128 epilogue threads, returning the OR of `pred`.
__device__ __forceinline__ bool epi_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
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
  __nv_bfloat16* staging = (__nv_bfloat16*)(base_ptr + (size_t)p.stages * p.stage_bytes);
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
        for (int kb = 0; kb < p.kb; ++kb) tma_load_2d(dst + kb * 16384u, &map, kb * 64, row0, full0 + 8 * s);
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
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int row = q * 32 + lane;       // tile row = TMEM lane
    const int k = row / p.n;             // sample within the tile
    const int r = row - k * p.n;         // vector index within the sample
    // this row's products: columns j < jend of its sample's block, written from slot base
    //   mode 0: j < r at d + r(r-1)/2;  mode 1: j <= r at d + r(r+1)/2;  mode 2: all j at r n
    const int jend = p.mode == 0 ? r : (p.mode == 1 ? r + 1 : p.n);
    const int base = p.mode == 0 ? p.d + r * (r - 1) / 2 : (p.mode == 1 ? p.d + r * (r + 1) / 2 : r * p.n);
    int64_t it = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
      const int acc = (int)(it & 1);
      const uint32_t aph = (uint32_t)((it >> 1) & 1);
      const bool ok = mbar_wait(tfull0 + 8 * acc, aph);
      if (!ok) {
        set_error(p.err, CTR_ERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
      }
      // one decision for all 128 epilogue threads (also: the staging buffer is free again)
      if (epi_any(!ok || *(volatile int*)&abort_flag)) break;
      fence_after();
      const int64_t b = t * p.S + k;
      const bool valid = k < p.S && b < p.batch;
      __nv_bfloat16* st = staging + (size_t)k * p.W;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)acc * 128u;
      for (int c0 = 0; c0 < p.N; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(tbase + (uint32_t)c0, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int j = c0 + e - k * p.n;
          if (valid && j >= 0 && j < jend) st[base + j] = __float2bfloat16_rn(__uint_as_float(v[e]));
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      if (valid && p.mode != 2) {
        const __nv_bfloat16* xd = p.X + b * (int64_t)p.n * p.d;  // dense vector of sample b
        for (int c = r; c < p.d / 8; c += p.n) {
          uint4 w = *(const uint4*)(xd + c * 8);
          const __nv_bfloat16* h = (const __nv_bfloat16*)&w;
#pragma unroll
          for (int e = 0; e < 8; ++e) st[c * 8 + e] = h[e];
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");  // staging complete
      const int64_t nvalid = imin64(p.S, p.batch - t * p.S);
      const int64_t elems = nvalid * p.W;
      __nv_bfloat16* dst = p.out + t * p.S * (int64_t)p.W;
      const int tid = threadIdx.x - 64;
      if (((uintptr_t)dst % 8) == 0 && (elems % 4) == 0) {
        const uint2* src2 = (const uint2*)staging;
        uint2* dst2 = (uint2*)dst;
        for (int64_t e = tid; e < elems / 4; e += 128) dst2[e] = src2[e];
      } else {
        for (int64_t e = tid; e < elems; e += 128) dst[e] = staging[e];
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
  p.S = 128 / n;
  p.rows = p.S * n;
  p.N = (p.rows + 15) / 16 * 16;
  p.kb = d / 64;
  p.stage_bytes = 16384u * p.kb;
  p.tx_bytes = (uint32_t)(128 * p.rows * p.kb);
  p.stages = std::max(2, std::min(4, (int)((160 * 1024) / p.stage_bytes)));
  p.mode = mode;
  p.W = mode == 0 ? d + n * (n - 1) / 2 : (mode == 1 ? d + n * (n + 1) / 2 : n * n);
  p.staging_bytes = (uint32_t)align_up((size_t)p.S * p.W * 2, 16);
  p.X = (const __nv_bfloat16*)X;
  p.out = (__nv_bfloat16*)out;
  p.err = err;

  CUtensorMap map;
  cuuint64_t gdim[2] = {(cuuint64_t)d, (cuuint64_t)batch * n};
  cuuint64_t gstride[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)p.rows};
  cuuint32_t estride[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), gdim, gstride, box, estride,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CTR_ERR_CUDA;
  const size_t smem = 1024 + (size_t)p.stages * p.stage_bytes + p.staging_bytes;
  auto kern = interaction_bf16_tc_kernel;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return CTR_ERR_CUDA;
  const int64_t ntiles = ceil_div(batch, p.S);
  const int grid = (int)std::max<int64_t>(1, imin64(ntiles, num_sms()));
  kern<<<grid, kTcThreads, smem, s>>>(p, map); count_launch();
  return launch_status();
}

}  // namespace ctr
