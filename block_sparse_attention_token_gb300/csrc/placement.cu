// Dependency-aware placement of blocks on P virtual partitions (the one-GPU
// counterpart of placing sequence blocks on ranks by the sparse attention
// pattern): one assignment per batch element, shared by all heads, with the
// partition sizes of the contiguous split.
//
//  1. affinity_kernel - W[b][i][j] = number of heads in which block i selected
//     block j plus the same with i, j swapped (i != j); integer atomics, so the
//     counts are exact whatever the order.
//  2. greedy_kernel   - one CTA per batch element: blocks in order of total
//     affinity (descending; ties: lower index), each placed on the partition
//     with spare capacity whose blocks have the largest affinity to it (ties:
//     more spare capacity, then lower index). Scores are integer sums, so the
//     assignment is deterministic.
#include "common.cuh"

namespace sparsp {
namespace {

__global__ void __launch_bounds__(256)
affinity_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col_idx, int H, int nb,
                int64_t rows, int32_t* __restrict__ W, int32_t* d_status) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int64_t b = row / ((int64_t)H * nb);
  const int i = (int)(row % nb);
  const int32_t a = row_ptr[row], e1 = row_ptr[row + 1];
  if (e1 < a || e1 - a > nb) {
    if (lane == 0) report(d_status, SPARSP_ERR_DATA);
    return;
  }
  int32_t* Wb = W + b * nb * nb;
  for (int32_t e = a + lane; e < e1; e += 32) {
    const int32_t j = col_idx[e];
    if (j < 0 || j >= nb) {
      report(d_status, SPARSP_ERR_DATA);
      continue;
    }
    if (j == i) continue;
    atomicAdd(&Wb[(int64_t)i * nb + j], 1);
    atomicAdd(&Wb[(int64_t)j * nb + i], 1);
  }
}

constexpr int kThreads = 1024;

__device__ __forceinline__ unsigned long long max_key(unsigned long long v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
    v = o > v ? o : v;
  }
  return v;
}

__global__ void __launch_bounds__(kThreads)
greedy_kernel(const int32_t* __restrict__ W, int nb, int P, int32_t* __restrict__ owner) {
  __shared__ int32_t total[1024], order[1024], own[1024], caps[1024];
  __shared__ unsigned long long score[1024];
  __shared__ unsigned long long warp_best[32];
  const int b = blockIdx.x;
  const int32_t* Wb = W + (int64_t)b * nb * nb;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  // W is symmetric: the row sum of i is its column sum, read coalesced
  for (int i = t; i < nb; i += kThreads) {
    int32_t s = 0;
    for (int j = 0; j < nb; ++j) s += Wb[(int64_t)j * nb + i];
    total[i] = s;
    own[i] = -1;
  }
  for (int r = t; r < P; r += kThreads)
    caps[r] = (int)(((int64_t)(r + 1) * nb) / P - ((int64_t)r * nb) / P);
  __syncthreads();
  for (int i = t; i < nb; i += kThreads) {
    int rank = 0;
    for (int k = 0; k < nb; ++k) rank += (total[k] > total[i]) || (total[k] == total[i] && k < i);
    order[rank] = i;
  }
  __syncthreads();
  for (int step = 0; step < nb; ++step) {
    const int i = order[step];
    for (int r = t; r < P; r += kThreads) score[r] = 0ull;
    __syncthreads();
    for (int j = t; j < nb; j += kThreads) {
      const int r = own[j];
      if (r >= 0) atomicAdd(&score[r], (unsigned long long)Wb[(int64_t)i * nb + j]);
    }
    __syncthreads();
    // key = (score, spare capacity, -r): larger is better; full partitions are out
    unsigned long long best = 0ull;
    for (int r = t; r < P; r += kThreads)
      if (caps[r] > 0) {
        const unsigned long long key = (score[r] << 22) | ((unsigned long long)caps[r] << 11) |
                                       (unsigned long long)(1023 - r);
        best = key > best ? key : best;
      }
    best = max_key(best);
    if (lane == 0) warp_best[warp] = best;
    __syncthreads();
    if (warp == 0) {
      unsigned long long v = warp_best[lane];
      v = max_key(v);
      if (lane == 0) {
        const int r = 1023 - (int)(v & 1023ull);
        own[i] = r;
        caps[r] -= 1;
      }
    }
    __syncthreads();
  }
  for (int i = t; i < nb; i += kThreads) owner[(int64_t)b * nb + i] = own[i];
}

}  // namespace

size_t placement_ws(const Dims& s) { return (size_t)s.B * s.nb * s.nb * sizeof(int32_t); }

sparsp_status_t launch_placement(const Dims& s, const int32_t* row_ptr, const int32_t* col_idx, int P,
                                 int32_t* owner, void* ws, int32_t* d_status, cudaStream_t st) {
  int32_t* W = (int32_t*)ws;
  if (cudaMemsetAsync(W, 0, placement_ws(s), st) != cudaSuccess) return SPARSP_ERR_CUDA;
  const int64_t rows = s.rows();
  affinity_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(row_ptr, col_idx, s.H, s.nb, rows, W, d_status);
  SPARSP_LAUNCH_CHECK();
  greedy_kernel<<<s.B, kThreads, 0, st>>>(W, s.nb, P, owner);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace sparsp
