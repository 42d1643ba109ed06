// Small shared pieces: exclusive scan of counts, device SM count cache.
#include "common.cuh"

#include <atomic>

namespace sparsp {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanWarps = kScanThreads / 32;
constexpr int kScanPer = 16;

// One CTA scans a[0..n) in place into exclusive offsets and writes a[n] = total.
// Chunks of 4096 entries are processed in order with a running carry.
__global__ void __launch_bounds__(kScanThreads) scan_kernel(int32_t* a, int64_t n) {
  __shared__ int32_t warp_tot[kScanWarps];
  __shared__ int32_t carry_s;
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t c0 = 0; c0 < n; c0 += (int64_t)kScanThreads * kScanPer) {
    int32_t v[kScanPer];
    int32_t local = 0;
    const int64_t base = c0 + (int64_t)threadIdx.x * kScanPer;
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      v[u] = (base + u < n) ? a[base + u] : 0;
      local += v[u];
    }
    int32_t incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int32_t t = lane < kScanWarps ? warp_tot[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int32_t o = __shfl_up_sync(0xffffffffu, t, off);
        if (lane >= off) t += o;
      }
      if (lane < kScanWarps) warp_tot[lane] = t;   // inclusive over warps
    }
    __syncthreads();
    const int32_t carry = carry_s;
    int32_t run = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + (incl - local);
#pragma unroll
    for (int u = 0; u < kScanPer; ++u) {
      if (base + u < n) a[base + u] = run;
      run += v[u];
    }
    __syncthreads();
    if (threadIdx.x == 0) carry_s = carry + warp_tot[kScanWarps - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) a[n] = carry_s;
}

std::atomic<int> g_sm_count[64];

}  // namespace

sparsp_status_t launch_scan_counts(int32_t* a, int64_t n, cudaStream_t st) {
  scan_kernel<<<1, kScanThreads, 0, st>>>(a, n);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  int c = g_sm_count[dev].load(std::memory_order_relaxed);
  if (c > 0) return c;
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  g_sm_count[dev].store(v, std::memory_order_relaxed);
  return v;
}

}  // namespace sparsp
