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
//     assignment is deterministic. The steps are sequential: each costs two
//     barriers, with the affinity rows read two steps ahead.
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
constexpr int kSmallP = 32;   // up to this many partitions one warp picks the winner

__device__ __forceinline__ unsigned long long max_key(unsigned long long v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
    v = o > v ? o : v;
  }
  return v;
}

// key = (score, spare capacity, -r): larger is better; full partitions are out
__device__ __forceinline__ unsigned long long place_key(uint32_t score, int cap, int r) {
  return cap > 0 ? ((unsigned long long)score << 22) | ((unsigned long long)cap << 11) |
                       (unsigned long long)(1023 - r)
                 : 0ull;
}

// One CTA of ceil(nb/32) warps per batch element; thread t owns block t. The
// affinity rows of the next two blocks in order are loaded ahead.
//
// Few partitions (kFew): shared memory keeps, for every block u and partition
// r, A[u][r] = the affinity of u to the blocks placed on r so far. A step
// adds the last placed block's row into its partition's column (one add per
// thread), then warp 0 reads the next block's A row and picks the partition
// with two warp reductions (score, then spare capacity and index).
// Otherwise the scores are summed with shared-memory atomics and the pick is a
// block-wide maximum.
template <bool kFew>
__global__ void __launch_bounds__(kThreads)
greedy_kernel(const int32_t* __restrict__ W, int nb, int P, int32_t* __restrict__ owner) {
  __shared__ int32_t total[1024], order[1024], caps[1024];
  __shared__ uint32_t score[kFew ? 1 : 1024];
  __shared__ unsigned long long warp_best[32];
  __shared__ int s_pick;
  extern __shared__ uint32_t aff[];   // kFew: [nb][stride]
  const int stride = P | 1;           // odd: the column updates and the row reads are conflict-free
  const int b = blockIdx.x;
  const int32_t* Wb = W + (int64_t)b * nb * nb;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nt = blockDim.x, nw = nt >> 5;
  // W is symmetric: the row sum of i is its column sum, read coalesced
  if (t < nb) {
    int32_t s = 0;
    for (int j = 0; j < nb; ++j) s += Wb[(int64_t)j * nb + t];
    total[t] = s;
    if (kFew)
      for (int r = 0; r < P; ++r) aff[t * stride + r] = 0u;
  }
  for (int r = t; r < P; r += nt)
    caps[r] = (int)(((int64_t)(r + 1) * nb) / P - ((int64_t)r * nb) / P);
  __syncthreads();
  if (t < nb) {
    int rank = 0;
    for (int k = 0; k < nb; ++k) rank += (total[k] > total[t]) || (total[k] == total[t] && k < t);
    order[rank] = t;
  }
  __syncthreads();
  int my_own = -1;   // partition of block t
  uint32_t w0 = t < nb ? (uint32_t)Wb[(int64_t)order[0] * nb + t] : 0u;
  uint32_t w1 = t < nb && nb > 1 ? (uint32_t)Wb[(int64_t)order[1] * nb + t] : 0u;
  uint32_t w_last = 0u;   // row of the block placed in the previous step (kFew)
  int r_last = -1;
  for (int step = 0; step < nb; ++step) {
    const int i = order[step];
    const uint32_t w = w0;
    w0 = w1;
    if (t < nb && step + 2 < nb) w1 = (uint32_t)Wb[(int64_t)order[step + 2] * nb + t];
    if (kFew) {
      if (r_last >= 0 && t < nb) aff[t * stride + r_last] += w_last;   // W[u][i_last] = W[i_last][u]
      __syncthreads();
      if (warp == 0) {
        const bool open = lane < P && caps[lane] > 0;
        const uint32_t sc = open ? aff[i * stride + lane] : 0u;
        const uint32_t top = __reduce_max_sync(0xffffffffu, sc);
        const uint32_t tie = open && sc == top ? ((uint32_t)caps[lane] << 11) | (uint32_t)(1023 - lane) : 0u;
        const uint32_t best = __reduce_max_sync(0xffffffffu, tie);
        if (lane == 0) {
          const int r = 1023 - (int)(best & 1023u);
          caps[r] -= 1;
          s_pick = r;
        }
      }
    } else {
      for (int r = t; r < P; r += nt) score[r] = 0u;
      __syncthreads();
      if (my_own >= 0) atomicAdd(&score[my_own], w);
      __syncthreads();
      unsigned long long best = 0ull;
      for (int r = t; r < P; r += nt) {
        const unsigned long long key = place_key(score[r], caps[r], r);
        best = key > best ? key : best;
      }
      best = max_key(best);
      if (lane == 0) warp_best[warp] = best;
      __syncthreads();
      if (warp == 0) {
        unsigned long long v = lane < nw ? warp_best[lane] : 0ull;
        v = max_key(v);
        if (lane == 0) {
          const int r = 1023 - (int)(v & 1023ull);
          caps[r] -= 1;
          s_pick = r;
        }
      }
    }
    __syncthreads();
    r_last = s_pick;
    w_last = w;
    if (t == i) my_own = r_last;
  }
  if (t < nb) owner[(int64_t)b * nb + t] = my_own;
}

size_t placement_few_smem(int nb, int P) { return (size_t)nb * (size_t)(P | 1) * sizeof(uint32_t); }

}  // namespace

size_t placement_ws(const Dims& s) { return (size_t)s.B * s.nb * s.nb * sizeof(int32_t); }

sparsp_status_t launch_placement(const Dims& s, const int32_t* row_ptr, const int32_t* col_idx, int P,
                                 int32_t* owner, void* ws, int32_t* d_status, cudaStream_t st) {
  int32_t* W = (int32_t*)ws;
  if (cudaMemsetAsync(W, 0, placement_ws(s), st) != cudaSuccess) return SPARSP_ERR_CUDA;
  const int64_t rows = s.rows();
  affinity_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(row_ptr, col_idx, s.H, s.nb, rows, W, d_status);
  SPARSP_LAUNCH_CHECK();
  const unsigned threads = (unsigned)((s.nb + 31) / 32 * 32);
  if (P <= kSmallP) {
    const size_t smem = placement_few_smem(s.nb, P);
    if (cudaFuncSetAttribute(greedy_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return SPARSP_ERR_CUDA;
    greedy_kernel<true><<<s.B, threads, smem, st>>>(W, s.nb, P, owner);
  } else {
    greedy_kernel<false><<<s.B, threads, 0, st>>>(W, s.nb, P, owner);
  }
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace sparsp
