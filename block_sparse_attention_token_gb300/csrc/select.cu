// Step 3: Top-p routing with a Top-k floor, compacted into a per-head CSR.
//
// Three launches, no atomics on data, deterministic:
//  1. count_kernel  - one warp per row, without sorting: bitwise searches over
//     the order-preserving score bits find the Top-p cutoff and the m-th
//     block in the order (score descending, block index ascending); beyond
//     1,024 blocks one CTA per row (count_row_kernel) sorts the 64-bit keys
//     (score bits, then index) with a bitonic network in shared memory.
//     e_j = exp(S_j - max) rounded to fp32 (expf, or the correctly rounded
//     value for rows whose Top-p crossing lies within 1e-6 of p); Z and the
//     prefix masses as exact 64-bit fixed-point sums (float64 in the
//     CTA-per-row kernel); m = min(nb, max(m_p, k_floor, 1)).
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

// One warp per row of nb <= 32*E blocks, without sorting. Block j of the row
// has the order-preserving score bits u_j (larger score = larger u) and sits
// at position p = e*32 + lane. The kept set is the first m blocks in the order
// (score descending, index ascending); it is described by its last member,
// whose key (score bits, index) becomes the row's threshold for the fill
// pass. Two searches over the bits of u find it:
//  - Top-p: t* = the largest t whose mass M(t) = sum of e_j over u_j >= t
//    still reaches top_p * Z; the blocks with u > t* hold less than that, so
//    the crossing lies among the blocks tied at t*, which follow in index
//    order: m_p = #(u > t*) + the fewest of those ties that reach the target.
//  - the m-th block (m = min(nb, max(m_p, k_floor, 1))): the largest t with
//    #(u >= t) >= m, then the (m - #(u > t))-th of its ties by index.
// e_j = expf(s_j - max) in fp32 (correctly rounded instead for a row whose
// crossing lies within 1e-6 of p). The t* search runs on coarse integer sums
// (e_j truncated to 21-24 fraction bits, one warp reduction per step); t* and
// the tie count are then decided on exact sums of e_j in 64-bit fixed point
// (resolution 2^-52, each term truncated by less than that: for nb <= 1024
// the sums lie within 4e-13 of Z of float64 sums of the same values in any
// order, inside the 1e-12 band in which the two may disagree at all),
// stepping to a neighbouring score if the fp32 search landed off the crossing.
constexpr double kFix = 4503599627370496.0;   // 2^52

// e (0 <= e <= 1, fp32) in units of 2^-52, truncated: exact for e >= 2^-29
__device__ __forceinline__ uint64_t to_fix(float e) {
  const uint32_t b = __float_as_uint(e);
  const int ex = (int)((b >> 23) & 0xffu);
  if (ex == 0) return 0ull;   // zero or subnormal: below 2^-126
  const uint64_t mant = (uint64_t)((b & 0x7fffffu) | 0x800000u);
  const int sh = ex - 98;     // e * 2^52 = mant * 2^(ex - 127 - 23 + 52)
  return sh >= 0 ? mant << sh : (sh > -64 ? mant >> (-sh) : 0ull);
}

template <int E>
struct WarpRow {
  // the steering sums: e_j (<= 1) in units of 2^-kSteerBits, truncated, so that
  // the sum of all 32*E of them fits 31 bits and one integer warp reduction adds them
  static constexpr int kSteerBits = E <= 2 ? 24 : (E <= 8 ? 23 : (E <= 16 ? 22 : 21));
  uint32_t u[E];
  float ev[E];
  uint32_t es[E];   // e_j * 2^kSteerBits, truncated
  int nb, lane;

  __device__ __forceinline__ bool valid(int e) const { return e * 32 + lane < nb; }

  // number of blocks with u >= t (warp total)
  __device__ __forceinline__ int count_ge(uint32_t t) const {
    int c = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) c += (valid(e) && u[e] >= t) ? 1 : 0;
    return (int)__reduce_add_sync(0xffffffffu, (unsigned)c);
  }
  // coarse mass of the blocks with u >= t (warp total, in units of 2^-kSteerBits;
  // only steers the search)
  __device__ __forceinline__ uint32_t mass_steer(uint32_t t) const {
    uint32_t m = 0u;
#pragma unroll
    for (int e = 0; e < E; ++e) m += u[e] >= t ? es[e] : 0u;   // es = 0 past nb
    return __reduce_add_sync(0xffffffffu, m);
  }
  __device__ __forceinline__ void set_steer() {
#pragma unroll
    for (int e = 0; e < E; ++e) es[e] = valid(e) ? (uint32_t)(ev[e] * (float)(1u << kSteerBits)) : 0u;
  }
  // exact fixed-point mass of the blocks with u >= t (ge) or u > t (!ge)
  __device__ __forceinline__ uint64_t massq(uint32_t t, bool ge) const {
    uint64_t m = 0ull;
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (valid(e) && (ge ? u[e] >= t : u[e] > t)) m += to_fix(ev[e]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m += __shfl_xor_sync(0xffffffffu, m, off);
    return m;
  }
  // the largest u below t / the smallest u above t (warp-wide)
  __device__ __forceinline__ uint32_t below(uint32_t t) const {
    uint32_t b = 0u;
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (valid(e) && u[e] < t) b = max(b, u[e]);
    return __reduce_max_sync(0xffffffffu, b);
  }
  __device__ __forceinline__ uint32_t above(uint32_t t) const {
    uint32_t a = 0xffffffffu;
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (valid(e) && u[e] > t) a = min(a, u[e]);
    return __reduce_min_sync(0xffffffffu, a);
  }
  // index of the k-th (1-based) block with u == t, in index order
  __device__ __forceinline__ int kth_tie(uint32_t t, int k) const {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint32_t ball = __ballot_sync(0xffffffffu, valid(e) && u[e] == t);
      const int c = __popc(ball);
      if (k <= c) {
        uint32_t b = ball;
        for (int r = 1; r < k; ++r) b &= b - 1u;
        return e * 32 + __ffs(b) - 1;
      }
      k -= c;
    }
    return -1;   // not reached for 1 <= k <= #ties
  }
};

// Bits of the search: every t below the common prefix of umin and umax counts
// every block, so only the bits from the highest differing one need trying.
__device__ __forceinline__ int search_top_bit(uint32_t umin, uint32_t umax) {
  return umin == umax ? -1 : 31 - __clz(umin ^ umax);
}

__device__ __forceinline__ uint32_t search_start(uint32_t umin, int hb) {
  return hb < 0 ? umin : (umin & ~((2u << hb) - 1u));   // hb = 31: 2u << 31 == 0, start at 0
}

// Top-p cutoff m_p from e_j held in row.ev; *near when a prefix sum around the
// crossing lies within 1e-6 of Z of the target. *tstar: the score bits of the
// m_p-th block; *gt_out: the number of blocks above them.
template <int E>
__device__ __forceinline__ int topp_count(const WarpRow<E>& row, uint32_t umin, uint32_t umax, double top_p,
                                          bool* near, uint32_t* tstar, int* gt_out) {
  const uint64_t Zq = row.massq(0u, true);
  // the target p*Z and its 1e-6*Z band in the same fixed point, once per row
  // (float64 is slow on this GPU: every comparison below is on integers). For
  // an integer sum x, x >= p*Z exactly when x >= ceil(p*Z).
  const double Z = (double)Zq, target = top_p * Z, band = 1e-6 * Z;
  const uint64_t Tq = (uint64_t)ceil(target);
  const uint64_t near_lo = (uint64_t)fmax(floor(target - band), 0.0), near_hi = (uint64_t)ceil(target + band);
  const uint32_t target_s = (uint32_t)((float)top_p * (float)row.mass_steer(0u));
  const int hb = search_top_bit(umin, umax);
  uint32_t t = search_start(umin, hb);
  for (int bit = hb; bit >= 0; --bit) {
    const uint32_t cand = t | (1u << bit);
    if (row.mass_steer(cand) >= target_s) t = cand;
  }
  // exact: M(t) >= target > M(> t), with t a score of the row
  uint64_t ge = 0ull, gt = 0ull;
  for (int step = 0; step <= 2 * row.nb; ++step) {
    ge = row.massq(t, true);
    gt = row.massq(t, false);
    if (ge < Tq) {
      t = row.below(t);          // exists: M(umin) = Z >= target
    } else if (gt >= Tq) {
      t = row.above(t);          // exists: M(> umax) = 0 < target
    } else {
      break;
    }
  }
  const int gtc = t == 0xffffffffu ? 0 : row.count_ge(t + 1u);
  const int eq = row.count_ge(t) - gtc;
  // the ties all hold the same e_j: that of any of them
  float et = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (row.valid(e) && row.u[e] == t) et = row.ev[e];
  et = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(et)));   // et >= 0: bits order as values
  const uint64_t etq = to_fix(et);
  uint64_t cq = gt + etq, cq_prev = gt;
  int k = 1;
  while (cq < Tq && k < eq) {
    cq_prev = cq;
    cq += etq;
    ++k;
  }
  *near = (cq > near_lo && cq < near_hi) || (cq_prev > near_lo && cq_prev < near_hi);
  *tstar = t;
  *gt_out = gtc;
  return min(row.nb, gtc + k);
}

// Up to 512 blocks a row: registers capped for four CTAs (32 warps) per SM,
// so that a whole wave of rows hides the search's reduction latencies
// (measured faster than 80-128 registers at two or three CTAs).
template <int E>   // blocks per lane; nb <= 32*E
__global__ void __launch_bounds__(kWarpsPerCta * 32, E <= 16 ? 4 : 1)
count_kernel(const float* __restrict__ S, int64_t rows, int nb, double top_p, int k_floor,
             int32_t* __restrict__ counts, uint64_t* __restrict__ thr, int32_t* d_status) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (r >= rows) return;
  const float* srow = S + r * nb;
  WarpRow<E> row;
  row.nb = nb;
  row.lane = lane;
  bool bad = false;
  uint32_t umin = 0xffffffffu, umax = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    row.u[e] = 0u;
    row.ev[e] = 0.f;
    if (row.valid(e)) {
      const float sv = srow[e * 32 + lane];
      if (!isfinite(sv)) bad = true;
      row.u[e] = ordered_bits(sv);
      umin = min(umin, row.u[e]);
      umax = max(umax, row.u[e]);
    }
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) {
      report(d_status, SPARSP_ERR_DATA);
      counts[r] = 0;
      thr[r] = 0;
    }
    return;
  }
  umin = __reduce_min_sync(0xffffffffu, umin);
  umax = __reduce_max_sync(0xffffffffu, umax);
  int m_p;
  uint32_t tp = 0u;   // Top-p: score bits of the m_p-th block and the count above them
  int gtp = 0;
  if (top_p <= 0.0) {
    m_p = 0;
  } else if (top_p >= 1.0) {
    m_p = nb;
  } else {
    const float smax = from_ordered(umax);
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (row.valid(e)) row.ev[e] = expf(from_ordered(row.u[e]) - smax);
    row.set_steer();
    bool near = false;
    m_p = topp_count<E>(row, umin, umax, top_p, &near, &tp, &gtp);
    // e_j is defined as the float32 rounding of exp(S_j - max). expf is within
    // 2 ulp of the exact value, which moves any of these sums (and Z) by at
    // most 3e-7 of Z; only a row whose crossing lies that close to p can decide
    // differently, and it is recomputed with the correctly rounded e_j.
    if (near) {
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (row.valid(e)) row.ev[e] = __double2float_rn(exp((double)(from_ordered(row.u[e]) - smax)));
      row.set_steer();
      m_p = topp_count<E>(row, umin, umax, top_p, &near, &tp, &gtp);
    }
  }
  const int m = min(nb, max(m_p, max(k_floor, 1)));
  // the m-th block in (score descending, index ascending) order: the Top-p
  // search has found it already unless the floor raised the count
  uint32_t t = tp;
  int gt = gtp;
  if (m != m_p) {
    const int hb = search_top_bit(umin, umax);
    t = search_start(umin, hb);
    for (int bit = hb; bit >= 0; --bit) {
      const uint32_t cand = t | (1u << bit);
      if (row.count_ge(cand) >= m) t = cand;
    }
    gt = t == 0xffffffffu ? 0 : row.count_ge(t + 1u);
  }
  const int j = row.kth_tie(t, m - gt);
  if (lane == 0) {
    counts[r] = m;
    thr[r] = ((uint64_t)(~t) << 32) | (uint32_t)j;   // = make_key(score of t, j)
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
            const uint64_t* __restrict__ thr, int32_t* __restrict__ col_idx, int32_t* d_status) {
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
    if (keep) {
      const int32_t pos = written + __popc(ball & ((1u << lane) - 1u));
      if (dcheck(pos < cnt, d_status)) col_idx[base + pos] = j;
    }
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
  fill_kernel<<<(unsigned)ctas, kWarpsPerCta * 32, 0, st>>>(scores, rows, nb, row_ptr, thr, col_idx, d_status);
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
