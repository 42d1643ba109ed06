// Diagnostic single-tile tcgen05 product (see include/sparsp_diag.h).
#include "sparsp_diag.h"
#include "tc_helpers.cuh"

namespace sparsp {
namespace {

using namespace tc;

constexpr uint32_t kTile = 128 * 128 * 2, kHalf = 128 * 64 * 2;
// A tile, B tile, then 64 KB of slack so that any lbo/sbo <= 32 KB stays inside
constexpr uint32_t kSmem = 4 * kTile + 64 + 1024;
constexpr uint64_t kWaitNs = 1000000000ull, kDrainNs = 200000000ull;

__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit) return false;
  return true;
}

__global__ void __launch_bounds__(128, 1)
diag_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
            const __nv_bfloat16* __restrict__ a, float* __restrict__ d, int mode, uint32_t lbo, uint32_t sbo,
            int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base, sB = base + kTile, bar_ld = base + 4 * kTile, bar_mma = bar_ld + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + 4 * kTile + 16);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  if (mode == 1) {
    // row r of A into TMEM lane r, columns 256..319 as packed bf16 pairs
    const uint32_t* arow = reinterpret_cast<const uint32_t*>(a + threadIdx.x * 128);
    uint32_t v[32];
    for (int h = 0; h < 2; ++h) {
      for (int x = 0; x < 32; ++x) v[x] = arow[h * 32 + x];
      tmem_st32(tmem + lane_base + 256u + h * 32u, v);
    }
    wait_st();
  }
  fence_before();
  __syncthreads();
  fence_after();
  // thread 0 loads and multiplies; every wait is bounded. On a time-out the
  // copies or MMAs still in flight are drained (with a second bounded wait)
  // before TMEM is read or freed, and TMEM is then not read at all.
  volatile int32_t* ok_flag = reinterpret_cast<volatile int32_t*>(gbase + 4 * kTile + 20);
  if (threadIdx.x == 0) {
    const uint32_t bytes = mode == 1 ? kTile : 2 * kTile;
    mbar_arrive_expect_tx(bar_ld, bytes);
    if (mode != 1) {
      tma_load_2d(sA, &ta, bar_ld, 0, 0);
      tma_load_2d(sA + kHalf, &ta, bar_ld, 64, 0);
    }
    tma_load_2d(sB, &tb, bar_ld, 0, 0);
    tma_load_2d(sB + kHalf, &tb, bar_ld, 64, 0);
    bool ok = bounded_wait(bar_ld, 0, kWaitNs);
    if (!ok) {
      bounded_wait(bar_ld, 0, kDrainNs);   // the copies may still land
    } else {
      fence_after();
      const uint32_t id = idesc_bf16(128, 128, 0, mode == 0 ? 0 : 1);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t koff = (uint32_t)(kk >> 2) * kHalf + (uint32_t)(kk & 3) * 32u;
        const uint64_t bdesc = mode == 0 ? smem_desc(sB + koff, 16, 1024, kSwizzle128B)
                                         : smem_desc(sB + (uint32_t)kk * 2048u, lbo, sbo, kSwizzle128B);
        if (mode == 1)
          mma_ts(tmem, tmem + 256u + (uint32_t)kk * 8u, bdesc, id, kk > 0);
        else
          mma_ss(tmem, smem_desc(sA + koff, 16, 1024, kSwizzle128B), bdesc, id, kk > 0);
      }
      commit(bar_mma);
      ok = bounded_wait(bar_mma, 0, kWaitNs);
      if (!ok) bounded_wait(bar_mma, 0, kDrainNs);   // let the MMAs finish before TMEM is freed
    }
    if (!ok) report(err, SPARSP_ERR_TIMEOUT);
    *ok_flag = ok ? 1 : 0;
  }
  __syncthreads();
  fence_after();
  if (*ok_flag) {
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_base + c * 32u, r);
      wait_ld();
      for (int x = 0; x < 32; ++x) d[threadIdx.x * 128 + c * 32 + x] = __uint_as_float(r[x]);
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// One warp waits, with the attention kernels' bounded wait, on phase 0 of a
// barrier that expects one arrival nobody makes.
__global__ void __launch_bounds__(32, 1) wait_timeout_kernel(uint64_t limit_ns, int32_t* d_status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const Guard g{&abort_flag, d_status, limit_ns};
  wait_warp(smem_u32(&bar), 0u, g);
}

}  // namespace
}  // namespace sparsp

extern "C" sparsp_status_t sparsp_diag_wait_timeout(uint64_t limit_ns, int32_t* d_status, sparsp_stream_t stream) {
  using namespace sparsp;
  if (d_status == nullptr || ((uintptr_t)d_status & 3u)) return SPARSP_ERR_INVALID_ARG;
  if (limit_ns < 1000000ull || limit_ns > 5000000000ull) return SPARSP_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit_ns, d_status);
  return cudaGetLastError() == cudaSuccess ? SPARSP_OK : SPARSP_ERR_CUDA;
}

extern "C" sparsp_status_t sparsp_diag_umma_tile(const void* a, const void* b, float* d, int32_t mode,
                                                 int32_t lbo, int32_t sbo, int32_t* d_status,
                                                 sparsp_stream_t stream) {
  using namespace sparsp;
  if (a == nullptr || b == nullptr || d == nullptr) return SPARSP_ERR_INVALID_ARG;
  if (((uintptr_t)a | (uintptr_t)b | (uintptr_t)d) & 15u) return SPARSP_ERR_ALIGN;
  if (mode < 0 || mode > 2) return SPARSP_ERR_INVALID_ARG;
  if (d_status == nullptr || ((uintptr_t)d_status & 3u)) return SPARSP_ERR_INVALID_ARG;
  if (lbo < 16 || sbo < 16 || lbo > 32768 || sbo > 32768 || (lbo & 15) || (sbo & 15))
    return SPARSP_ERR_INVALID_ARG;
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return SPARSP_ERR_CUDA;
  if (major != 10) return SPARSP_ERR_UNSUPPORTED;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_rows(&ta, a, 128, 128, 128) || !make_tmap_bf16_rows(&tb, b, 128, 128, 128))
    return SPARSP_ERR_CUDA;
  if (cudaFuncSetAttribute(diag_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem) != cudaSuccess)
    return SPARSP_ERR_CUDA;
  diag_kernel<<<1, 128, kSmem, (cudaStream_t)stream>>>(ta, tb, (const __nv_bfloat16*)a, d, mode, (uint32_t)lbo,
                                                       (uint32_t)sbo, d_status);
  return cudaGetLastError() == cudaSuccess ? SPARSP_OK : SPARSP_ERR_CUDA;
}
