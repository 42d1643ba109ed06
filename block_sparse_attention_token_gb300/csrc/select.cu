// Step 3: Top-p routing with a Top-k floor, compacted into a per-head CSR.
//
// Three launches, no atomics on data, deterministic:
//  1. count_kernel  - one warp per row (one CTA per row beyond 1,024 blocks,
//     count_row_kernel): bitonic sort of 64-bit keys
//     (score descending as an order-preserving integer, then block index) held
//     in registers and exchanged with shuffles; e_j = exp(S_j - max) rounded
//     to fp32 (expf, or the correctly rounded value for rows whose Top-p
//     crossing lies within 1e-6 of p); Z and the prefix masses in fp64;
//     m = min(nb, max(m_p, k_floor, 1)).
//     Writes m into row_ptr[row] and the key of the m-th kept block into ws.
//  2. scan          - exclusive scan of the counts -> row_ptr.
//  3. fill_kernel   - one warp per row: block j is kept iff its key <= the
//     stored threshold key; kept indices are compacted in ascending j order
//     with ballots.
#include "common.cuh"

namespace sparsp {

// Scratch of sparsp_select_noalloc: one 64-bit threshold key per CSR row, for
// at most kSelectNoAllocMaxRows rows (512 KB). It lives in the library's own
// device memory, so every device that loads the library holds it until exit.
static __device__ __align__(256) uint64_t g_select_scratch[kSelectNoAllocMaxRows];

namespace {

constexpr int kWarpsPerCta = 8;

// Order-preserving map of a finite float to uint32 (ascending), with -0 == +0.
__device__ __forceinline__ uint32_t ordered_bits(float s) {
  uint32_t u = __float_as_uint(s + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float from_ordered(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
  return __uint_as_float(u);
}

// key: smaller = kept earlier. High word: descending score; low word: index.
__device__ __forceinline__ uint64_t make_key(float s, int j) {
  return ((uint64_t)(~ordered_bits(s)) << 32) | (uint32_t)j;
}

__device__ __forceinline__ float key_score(uint64_t key) {
  return from_ordered(~(uint32_t)(key >> 32));
}

// m_p of one row held sorted in the warp's registers (positions lane*E + e):
// the smallest m whose leading prefix of e_j = exp(S_j - max) holds mass
// >= top_p * Z, with Z and the prefixes summed in float64. exact: e_j is the
// correctly rounded float32 of the exponential (evaluated in float64);
// otherwise expf. *near: some prefix lies within 1e-6 of Z of the target.
template <int E>
__device__ __forceinline__ int topp_count(const uint64_t (&key)[E], float smax, int lane, int nb, double top_p,
                                          bool exact, bool* near) {
  double ev[E];
  double lane_sum = 0.0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int p = lane * E + e;
    ev[e] = 0.0;
    if (p < nb) {
      const float x = key_score(key[e]) - smax;
      ev[e] = exact ? (double)__double2float_rn(exp((double)x)) : (double)expf(x);
    }
    lane_sum += ev[e];
  }
  // inclusive scan of lane sums
  double incl = lane_sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  const double Z = __shfl_sync(0xffffffffu, incl, 31);
  const double target = top_p * Z, band = 1e-6 * Z;
  double c = incl - lane_sum;   // exclusive prefix of this lane
  int below = 0;
  bool close = false;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int p = lane * E + e;
    c += ev[e];
    if (p < nb) {
      if (c < target) ++below;
      if (fabs(c - target) < band) close = true;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) below += __shfl_xor_sync(0xffffffffu, below, off);
  *near = __any_sync(0xffffffffu, close);
  return min(nb, below + 1);
}

template <int E>   // elements per lane; padded row length = 32*E
__global__ void __launch_bounds__(kWarpsPerCta * 32)
count_kernel(const float* __restrict__ S, int64_t rows, int nb, double top_p, int k_floor,
             int32_t* __restrict__ counts, uint64_t* __restrict__ thr, int32_t* d_status) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* srow = S + row * nb;
  uint64_t key[E];
  bool bad = false;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int p = lane * E + e;
    if (p < nb) {
      const float s = srow[p];
      if (!isfinite(s)) bad = true;
      key[e] = make_key(s, p);
    } else {
      key[e] = ~0ull;
    }
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) {
      report(d_status, SPARSP_ERR_DATA);
      counts[row] = 0;
      thr[row] = 0;
    }
    return;
  }
  // bitonic sort, ascending key, positions p = lane*E + e
  constexpr int NP = 32 * E;
#pragma unroll
  for (int size = 2; size <= NP; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride < E) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int e2 = e ^ stride;
          if (e2 > e) {
            const int p = lane * E + e;
            const bool asc = (p & size) == 0;
            const uint64_t a = key[e], b = key[e2];
            const bool swap = asc ? (a > b) : (a < b);
            key[e] = swap ? b : a;
            key[e2] = swap ? a : b;
          }
        }
      } else {
        const int lmask = stride / E;
        const bool lo = (lane & lmask) == 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int p = lane * E + e;
          const bool asc = (p & size) == 0;
          const uint64_t other = __shfl_xor_sync(0xffffffffu, key[e], lmask);
          const uint64_t mn = key[e] < other ? key[e] : other;
          const uint64_t mx = key[e] < other ? other : key[e];
          key[e] = (lo == asc) ? mn : mx;
        }
      }
    }
  }
  // Top-p cutoff from the softmax mass in sorted order (no exponentials are
  // needed for p <= 0 or p >= 1)
  int m_p;
  if (top_p <= 0.0) {
    m_p = 0;
  } else if (top_p >= 1.0) {
    m_p = nb;
  } else {
    const float smax = __shfl_sync(0xffffffffu, key_score(key[0]), 0);
    bool near = false;
    m_p = topp_count<E>(key, smax, lane, nb, top_p, false, &near);
    // e_j is defined as the float32 rounding of exp(S_j - max). expf is within
    // 2 ulp of the exact value, which moves any prefix sum (and Z) by at most
    // 3e-7 of Z; only a row whose crossing lies that close to p can decide
    // differently, and it is recomputed with the correctly rounded e_j.
    if (near) m_p = topp_count<E>(key, smax, lane, nb, top_p, true, &near);
  }
  const int m = min(nb, max(m_p, max(k_floor, 1)));
  // threshold key = key at sorted position m-1
  const int pos = m - 1;
  const int src_lane = pos / E, src_e = pos % E;
  uint64_t mine = 0;
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (e == src_e) mine = key[e];
  const uint64_t tk = __shfl_sync(0xffffffffu, mine, src_lane);
  if (lane == 0) {
    counts[row] = m;
    thr[row] = tk;
  }
}

// Rows longer than 1,024 blocks: one CTA of kRowThreads threads per row. The
// keys are sorted ascending with a bitonic network in shared memory (NP = the
// next power of two >= nb, at most 4,096); thread t then owns sorted positions
// [t*E, t*E + E) for the prefix masses, summed with a block-wide float64 scan.
// Same keys, same e_j (expf, or correctly rounded near the crossing), same
// cutoff rule as the warp-per-row kernel.
constexpr int kRowThreads = 512;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowMaxE = 8;   // 4,096 / 512

struct RowScratch {
  double wsum[kRowWarps];
  int32_t wcnt[kRowWarps];
  int32_t flag;
};

// Exclusive prefix (in sorted order) of this thread's chunk and the row total
// Z, from the chunk sums: a block-wide float64 scan.
__device__ __forceinline__ double block_excl_scan(double v, double* total, RowScratch& sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  __syncthreads();   // sc.wsum may still be read from a previous call
  if (lane == 31) sc.wsum[warp] = incl;
  __syncthreads();
  double before = 0.0, all = 0.0;
  for (int w = 0; w < kRowWarps; ++w) {
    if (w < warp) before += sc.wsum[w];
    all += sc.wsum[w];
  }
  *total = all;
  return before + incl - v;
}

__device__ __forceinline__ int block_topp_count(const uint64_t* keys, int nb, int E, float smax, double top_p,
                                                bool exact, bool* near, RowScratch& sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double ev[kRowMaxE];
  double sum = 0.0;
#pragma unroll
  for (int e = 0; e < kRowMaxE; ++e) {
    const int p = (int)threadIdx.x * E + e;
    ev[e] = 0.0;
    if (e < E && p < nb) {
      const float x = key_score(keys[p]) - smax;
      ev[e] = exact ? (double)__double2float_rn(exp((double)x)) : (double)expf(x);
    }
    sum += ev[e];
  }
  double Z;
  double c = block_excl_scan(sum, &Z, sc);
  const double target = top_p * Z, band = 1e-6 * Z;
  int below = 0;
  bool close = false;
#pragma unroll
  for (int e = 0; e < kRowMaxE; ++e) {
    const int p = (int)threadIdx.x * E + e;
    c += ev[e];
    if (e < E && p < nb) {
      if (c < target) ++below;
      if (fabs(c - target) < band) close = true;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) below += __shfl_xor_sync(0xffffffffu, below, off);
  if (lane == 0) sc.wcnt[warp] = below;
  *near = __syncthreads_or(close) != 0;
  int tot = 0;
  for (int w = 0; w < kRowWarps; ++w) tot += sc.wcnt[w];
  return min(nb, tot + 1);
}

__global__ void __launch_bounds__(kRowThreads)
count_row_kernel(const float* __restrict__ S, int nb, int NP, double top_p, int k_floor,
                 int32_t* __restrict__ counts, uint64_t* __restrict__ thr, int32_t* d_status) {
  extern __shared__ uint64_t keys[];   // [NP]
  __shared__ RowScratch sc;
  const int64_t row = blockIdx.x;
  const float* srow = S + row * nb;
  bool bad = false;
  for (int p = threadIdx.x; p < NP; p += kRowThreads) {
    if (p < nb) {
      const float v = srow[p];
      if (!isfinite(v)) bad = true;
      keys[p] = make_key(v, p);
    } else {
      keys[p] = ~0ull;
    }
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) {
      report(d_status, SPARSP_ERR_DATA);
      counts[row] = 0;
      thr[row] = 0;
    }
    return;
  }
  // bitonic sort, ascending
  for (int size = 2; size <= NP; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int q = threadIdx.x; q < NP / 2; q += kRowThreads) {
        const int i = (q / stride) * 2 * stride + (q % stride), j = i + stride;
        const bool asc = (i & size) == 0;
        const uint64_t a = keys[i], b = keys[j];
        if (asc ? a > b : a < b) {
          keys[i] = b;
          keys[j] = a;
        }
      }
      __syncthreads();
    }
  int m_p;
  if (top_p <= 0.0) {
    m_p = 0;
  } else if (top_p >= 1.0) {
    m_p = nb;
  } else {
    const float smax = key_score(keys[0]);
    const int E = (nb + kRowThreads - 1) / kRowThreads;
    bool near = false;
    m_p = block_topp_count(keys, nb, E, smax, top_p, false, &near, sc);
    if (near) m_p = block_topp_count(keys, nb, E, smax, top_p, true, &near, sc);
  }
  const int m = min(nb, max(m_p, max(k_floor, 1)));
  if (threadIdx.x == 0) {
    counts[row] = m;
    thr[row] = keys[m - 1];
  }
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
fill_kernel(const float* __restrict__ S, int64_t rows, int nb, const int32_t* __restrict__ row_ptr,
            const uint64_t* __restrict__ thr, int32_t* __restrict__ col_idx) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int32_t base = row_ptr[row];
  const int32_t cnt = row_ptr[row + 1] - base;
  if (cnt <= 0) return;
  const uint64_t tk = thr[row];
  const float* srow = S + row * nb;
  int written = 0;
  for (int j0 = 0; j0 < nb; j0 += 32) {
    const int j = j0 + lane;
    bool keep = false;
    if (j < nb) keep = make_key(srow[j], j) <= tk;
    const uint32_t ball = __ballot_sync(0xffffffffu, keep);
    if (keep) col_idx[base + written + __popc(ball & ((1u << lane) - 1u))] = j;
    written += __popc(ball);
  }
}

template <int E>
void count_go(const float* S, int64_t rows, int nb, double p, int kf, int32_t* counts,
              uint64_t* thr, int32_t* st_word, cudaStream_t st) {
  const int64_t ctas = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
  count_kernel<E><<<(unsigned)ctas, kWarpsPerCta * 32, 0, st>>>(S, rows, nb, p, kf, counts, thr,
                                                               st_word);
}

}  // namespace

size_t select_ws(const Dims& s) { return (size_t)s.rows() * sizeof(uint64_t); }

sparsp_status_t launch_select(const Dims& s, const float* scores, float top_p, int k_floor,
                              int32_t* row_ptr, int32_t* col_idx, void* ws, int32_t* d_status,
                              cudaStream_t st) {
  const int64_t rows = s.rows();
  uint64_t* thr = (uint64_t*)ws;
  const double p = (double)top_p;
  const int nb = s.nb;
  if (nb <= 32) count_go<1>(scores, rows, nb, p, k_floor, row_ptr, thr, d_status, st);
  else if (nb <= 64) count_go<2>(scores, rows, nb, p, k_floor, row_ptr, thr, d_status, st);
  else if (nb <= 128) count_go<4>(scores, rows, nb, p, k_floor, row_ptr, thr, d_status, st);
  else if (nb <= 256) count_go<8>(scores, rows, nb, p, k_floor, row_ptr, thr, d_status, st);
  else if (nb <= 512) count_go<16>(scores, rows, nb, p, k_floor, row_ptr, thr, d_status, st);
  else if (nb <= 1024) count_go<32>(scores, rows, nb, p, k_floor, row_ptr, thr, d_status, st);
  else {
    if (nb > kRowThreads * kRowMaxE) return SPARSP_ERR_UNSUPPORTED;
    int NP = 1;
    while (NP < nb) NP <<= 1;
    const size_t smem = (size_t)NP * sizeof(uint64_t);
    if (cudaFuncSetAttribute(count_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return SPARSP_ERR_CUDA;
    count_row_kernel<<<(unsigned)rows, kRowThreads, smem, st>>>(scores, nb, NP, p, k_floor, row_ptr, thr, d_status);
  }
  SPARSP_LAUNCH_CHECK();
  sparsp_status_t r = launch_scan_counts(row_ptr, rows, st);
  if (r != SPARSP_OK) return r;
  const int64_t ctas = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
  fill_kernel<<<(unsigned)ctas, kWarpsPerCta * 32, 0, st>>>(scores, rows, nb, row_ptr, thr, col_idx);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

sparsp_status_t launch_select_noalloc(const Dims& s, const float* scores, float top_p, int k_floor,
                                      int32_t* row_ptr, int32_t* col_idx, int32_t* d_status,
                                      cudaStream_t st) {
  if (s.rows() > kSelectNoAllocMaxRows) return SPARSP_ERR_WORKSPACE;
  // The host-side name of the array is not a device address: ask the runtime,
  // for the device and context current now, on every call. The answer is not
  // cached, because the array moves when the caller resets the device or
  // switches to another context on it. The query allocates nothing.
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_select_scratch) != cudaSuccess || ptr == nullptr) return SPARSP_ERR_CUDA;
  // Every row's threshold is written by the count pass before the fill pass
  // reads it, so nothing in the array has to start at zero.
  return launch_select(s, scores, top_p, k_floor, row_ptr, col_idx, ptr, d_status, st);
}

}  // namespace sparsp
