// Virtual-rank load balancing and slack-aware sparse augmentation.
//
// Head costs are selected block pairs (equal attention work each). P virtual
// ranks hold the heads of one batch element; the critical rank sets the step.
//
//  balance_kernel  - one CTA per batch element: contiguous head split, then at
//                    most M greedy migrations from the most to the least loaded
//                    rank (the head whose move gives the smallest pair maximum;
//                    only moves that lower the critical rank's load).
//  aug_keys_kernel - one warp per CSR row: each unselected block's value
//                    v = fl32(e_j / Z) (e_j = expf(S_j - max) in fp32, Z summed
//                    in fp64), stored as the orderable key bits(v) + 1; selected
//                    blocks get key 0. Also writes the row's base count.
//  aug_rank_kernel - one CTA per (batch element, rank): slack = L* - L_r; a
//                    4-pass radix select finds the key T of the slack-th best
//                    candidate; keys above T are taken, and of the keys equal to
//                    T the first ones in (row, block) order. Writes each row's
//                    new count and its share of the ties.
//  scan            - counts -> row offsets.
//  aug_fill_kernel - one warp per row merges the selected and the added blocks
//                    in ascending order.
#include "common.cuh"

namespace sparsp {
namespace {

constexpr int kMaxHeads = 2048;
constexpr unsigned long long kNone = ~0ull;

__device__ __forceinline__ unsigned long long warp_min(unsigned long long v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, v, off);
    v = o < v ? o : v;
  }
  return v;
}

// Block-wide minimum (all threads get the result). `red` holds 32 entries.
__device__ unsigned long long block_min(unsigned long long v, unsigned long long* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_min(v);
  __syncthreads();              // earlier readers of red are done
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = lane < nw ? red[lane] : kNone;
  return warp_min(v);
}

__device__ __forceinline__ int64_t head_cost(const int32_t* row_ptr, int64_t bh, int nb) {
  return (int64_t)row_ptr[(bh + 1) * nb] - (int64_t)row_ptr[bh * nb];
}

__global__ void __launch_bounds__(1024)
balance_kernel(const int32_t* __restrict__ row_ptr, int H, int nb, int P, int max_moves,
               int32_t* __restrict__ head_rank, int64_t* __restrict__ loads_out,
               int32_t* __restrict__ moves_out) {
  __shared__ int64_t cost[kMaxHeads];
  __shared__ int32_t rank_of[kMaxHeads];
  __shared__ unsigned long long load[kMaxHeads];
  __shared__ unsigned long long red[32];
  const int b = blockIdx.x;
  for (int r = threadIdx.x; r < P; r += blockDim.x) load[r] = 0ull;
  __syncthreads();
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    int r = 0;   // contiguous split: the r with floor(r*H/P) <= h < floor((r+1)*H/P)
    while (r + 1 < P && ((int64_t)(r + 1) * H) / P <= h) ++r;
    cost[h] = head_cost(row_ptr, (int64_t)b * H + h, nb);
    rank_of[h] = r;
    atomicAdd(&load[r], (unsigned long long)cost[h]);
  }
  __syncthreads();
  int64_t* before = loads_out + (int64_t)b * 2 * P;
  for (int r = threadIdx.x; r < P; r += blockDim.x) before[r] = (int64_t)load[r];
  int moves = 0;
  for (int it = 0; it < max_moves; ++it) {
    // loads < 2^32 and ranks < 2^12: (load, index) packed into one ordered key
    unsigned long long kmax = kNone, kmin = kNone;
    for (int r = threadIdx.x; r < P; r += blockDim.x) {
      const unsigned long long up = ((load[r] ^ 0xffffffffull) << 12) | (unsigned long long)r;
      const unsigned long long dn = (load[r] << 12) | (unsigned long long)r;
      kmax = up < kmax ? up : kmax;
      kmin = dn < kmin ? dn : kmin;
    }
    kmax = block_min(kmax, red);
    kmin = block_min(kmin, red);
    const int c = (int)(kmax & 4095ull), t = (int)(kmin & 4095ull);
    const long long Lc = (long long)load[c], Lt = (long long)load[t];
    unsigned long long kh = kNone;
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
      if (rank_of[h] != c) continue;
      const long long a = Lc - cost[h], z = Lt + cost[h];
      const unsigned long long nm = (unsigned long long)(a > z ? a : z);
      const unsigned long long key = (nm << 12) | (unsigned long long)h;
      kh = key < kh ? key : kh;
    }
    kh = block_min(kh, red);
    if (kh == kNone || (long long)(kh >> 12) >= Lc) break;   // uniform: every thread has kh
    const int h = (int)(kh & 4095ull);
    __syncthreads();
    if (threadIdx.x == 0) {
      rank_of[h] = t;
      load[c] -= (unsigned long long)cost[h];
      load[t] += (unsigned long long)cost[h];
    }
    ++moves;
    __syncthreads();
  }
  __syncthreads();
  for (int r = threadIdx.x; r < P; r += blockDim.x) before[P + r] = (int64_t)load[r];
  for (int h = threadIdx.x; h < H; h += blockDim.x) head_rank[(int64_t)b * H + h] = rank_of[h];
  if (threadIdx.x == 0 && moves_out != nullptr) moves_out[b] = moves;
}

// --------------------------------------------------------------- augmentation

constexpr int kMaxWords = 32;   // nb <= 1024

__global__ void __launch_bounds__(256)
aug_keys_kernel(const float* __restrict__ scores, const int32_t* __restrict__ row_ptr,
                const int32_t* __restrict__ col_idx, int nb, int64_t rows, uint32_t* __restrict__ keys,
                int32_t* __restrict__ counts, int32_t* d_status) {
  __shared__ uint32_t bits_all[8][kMaxWords];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + warp;
  if (row >= rows) return;
  uint32_t* bits = bits_all[warp];
  bits[lane] = 0u;
  __syncwarp();
  const int32_t e0 = row_ptr[row], e1 = row_ptr[row + 1];
  if (e1 < e0 || e1 - e0 > nb) {
    if (lane == 0) report(d_status, SPARSP_ERR_DATA);
  } else {
    for (int32_t e = e0 + lane; e < e1; e += 32) {
      const int32_t j = col_idx[e];
      if (j < 0 || j >= nb) {
        report(d_status, SPARSP_ERR_DATA);
        continue;
      }
      atomicOr(&bits[j >> 5], 1u << (j & 31));
    }
  }
  __syncwarp();
  int sel = __popc(bits[lane]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sel += __shfl_xor_sync(0xffffffffu, sel, off);
  if (lane == 0) counts[row] = sel;
  const float* S = scores + row * nb;
  uint32_t* K = keys + row * nb;
  float m = -INFINITY;
  bool finite = true;
  for (int j = lane; j < nb; j += 32) {
    const float s = S[j];
    finite &= isfinite(s);
    m = fmaxf(m, s);
  }
  finite = __all_sync(0xffffffffu, finite);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (!finite) {
    if (lane == 0) report(d_status, SPARSP_ERR_DATA);
    for (int j = lane; j < nb; j += 32) K[j] = 0u;   // no candidates in this row
    return;
  }
  double Z = 0.0;
  for (int j = lane; j < nb; j += 32) Z += (double)expf(S[j] - m);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, off);
  for (int j = lane; j < nb; j += 32) {
    const bool selected = (bits[j >> 5] >> (j & 31)) & 1u;
    const float v = (float)((double)expf(S[j] - m) / Z);
    K[j] = selected ? 0u : __float_as_uint(v) + 1u;
  }
}

constexpr int kRankThreads = 1024;
constexpr int kRankWarps = kRankThreads / 32;
constexpr int kHist = 16;        // histogram copies (two warps share one)

struct RankOut {
  uint32_t T;        // keys > T are taken
  int32_t need_eq;   // and this many keys == T, first in (row, block) order
};

__global__ void __launch_bounds__(kRankThreads)
aug_rank_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ head_rank, int H, int nb,
                int P, const uint32_t* __restrict__ keys, int32_t* __restrict__ counts,
                int32_t* __restrict__ taken, RankOut* __restrict__ rank_out, int64_t* __restrict__ added,
                int32_t* d_status) {
  __shared__ unsigned long long load[kMaxHeads];
  __shared__ int32_t heads[kMaxHeads];
  __shared__ int32_t hist[kHist][256];
  __shared__ int32_t eqs[kRankWarps];
  __shared__ unsigned long long red[32];
  __shared__ int n_heads, s_digit, s_rem;
  __shared__ unsigned long long s_ncand;
  const int b = blockIdx.x / P, r = blockIdx.x % P;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int q = tid; q < P; q += kRankThreads) load[q] = 0ull;
  if (tid == 0) s_ncand = 0ull;
  __syncthreads();
  for (int h = tid; h < H; h += kRankThreads) {
    const int q = head_rank[(int64_t)b * H + h];
    if (q < 0 || q >= P) {
      if (r == 0) report(d_status, SPARSP_ERR_DATA);
      continue;
    }
    atomicAdd(&load[q], (unsigned long long)head_cost(row_ptr, (int64_t)b * H + h, nb));
  }
  if (tid == 0) {   // this rank's heads, ascending
    int n = 0;
    for (int h = 0; h < H; ++h)
      if (head_rank[(int64_t)b * H + h] == r) heads[n++] = h;
    n_heads = n;
  }
  __syncthreads();
  unsigned long long top = 0ull;
  for (int q = tid; q < P; q += kRankThreads) top = load[q] > top ? load[q] : top;
  top = ~block_min(~top, red);
  const unsigned long long slack = top - load[r];
  const int nh = n_heads;
  const int per_head = nb * nb;
  // candidates
  unsigned long long nc = 0ull;
  for (int hh = 0; hh < nh; ++hh) {
    const uint32_t* K = keys + ((int64_t)b * H + heads[hh]) * per_head;
    for (int e = tid; e < per_head; e += kRankThreads) nc += K[e] != 0u;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) nc += __shfl_xor_sync(0xffffffffu, nc, off);
  if (lane == 0) atomicAdd(&s_ncand, nc);
  __syncthreads();
  const unsigned long long ncand = s_ncand;
  const unsigned long long s = slack < ncand ? slack : ncand;
  uint32_t T;
  int need_eq;
  if (s == 0ull) {
    T = 0xffffffffu;
    need_eq = 0;
  } else if (s == ncand) {
    T = 0u;
    need_eq = 0;
  } else {
    uint32_t prefix = 0u, mask = 0u;
    int rem = (int)s;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int d = tid; d < kHist * 256; d += kRankThreads) hist[d >> 8][d & 255] = 0;
      __syncthreads();
      int32_t* my_hist = hist[warp % kHist];
      for (int hh = 0; hh < nh; ++hh) {
        const uint32_t* K = keys + ((int64_t)b * H + heads[hh]) * per_head;
        for (int e = tid; e < per_head; e += kRankThreads) {
          const uint32_t k = K[e];
          if (k != 0u && (k & mask) == prefix) atomicAdd(&my_hist[(k >> shift) & 255u], 1);
        }
      }
      __syncthreads();
      if (tid < 256) {
        int c = 0;
        for (int w = 0; w < kHist; ++w) c += hist[w][tid];
        hist[0][tid] = c;
      }
      __syncthreads();
      if (tid == 0) {
        int d = 255;
        for (; d > 0; --d) {
          if (hist[0][d] >= rem) break;
          rem -= hist[0][d];
        }
        s_digit = d;
        s_rem = rem;
      }
      __syncthreads();
      prefix |= (uint32_t)s_digit << shift;
      mask |= 255u << shift;
      rem = s_rem;
      __syncthreads();
    }
    T = prefix;
    need_eq = rem;
  }
  // per-row counts; ties go to rows in (head, row) order
  int tie_base = 0;
  const int nrows = nh * nb;
  for (int k0 = 0; k0 < nrows; k0 += kRankWarps) {
    const int k = k0 + warp;
    int gt = 0, eq = 0;
    int64_t row = -1;
    if (k < nrows) {
      row = ((int64_t)b * H + heads[k / nb]) * nb + k % nb;
      const uint32_t* K = keys + row * nb;
      for (int j = lane; j < nb; j += 32) {
        const uint32_t key = K[j];
        gt += key > T && key != 0u;
        eq += key == T && key != 0u;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        gt += __shfl_xor_sync(0xffffffffu, gt, off);
        eq += __shfl_xor_sync(0xffffffffu, eq, off);
      }
    }
    if (lane == 0) eqs[warp] = eq;
    __syncthreads();
    if (k < nrows && lane == 0) {
      int before = tie_base;
      for (int w = 0; w < warp; ++w) before += eqs[w];
      int t = need_eq - before;
      t = t < 0 ? 0 : (t > eq ? eq : t);
      taken[row] = t;
      counts[row] += gt + t;
    }
    int sum = 0;
    for (int w = 0; w < kRankWarps; ++w) sum += eqs[w];
    tie_base += sum;
    __syncthreads();
  }
  if (tid == 0) {
    rank_out[blockIdx.x] = RankOut{T, need_eq};
    if (added != nullptr) added[blockIdx.x] = (int64_t)s;
  }
}

__global__ void __launch_bounds__(256)
aug_fill_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col_idx,
                const int32_t* __restrict__ head_rank, int H, int nb, int P, int64_t rows,
                const uint32_t* __restrict__ keys, const int32_t* __restrict__ taken,
                const RankOut* __restrict__ rank_out, const int32_t* __restrict__ out_ptr,
                int32_t* __restrict__ out_idx, int64_t cap, int32_t* d_status) {
  __shared__ uint32_t bits_all[8][kMaxWords];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + warp;
  if (row >= rows) return;
  uint32_t* bits = bits_all[warp];
  bits[lane] = 0u;
  __syncwarp();
  const int32_t e0 = row_ptr[row], e1 = row_ptr[row + 1];
  if (e1 >= e0 && e1 - e0 <= nb)
    for (int32_t e = e0 + lane; e < e1; e += 32) {
      const int32_t j = col_idx[e];
      if (j >= 0 && j < nb) atomicOr(&bits[j >> 5], 1u << (j & 31));
    }
  __syncwarp();
  const int64_t bh = row / nb;
  const int q = head_rank[bh];
  const bool valid = q >= 0 && q < P;
  const RankOut ro = valid ? rank_out[(bh / H) * P + q] : RankOut{0xffffffffu, 0};
  const int my_ties = valid ? taken[row] : 0;
  const uint32_t* K = keys + row * nb;
  int64_t pos = out_ptr[row];
  const int64_t end = out_ptr[row + 1];
  int ties_seen = 0;
  for (int j0 = 0; j0 < nb; j0 += 32) {
    const int j = j0 + lane;
    bool keep = false, tie = false;
    if (j < nb) {
      const bool sel = (bits[j >> 5] >> (j & 31)) & 1u;
      const uint32_t key = K[j];
      tie = !sel && key != 0u && key == ro.T;
      keep = sel || (key != 0u && key > ro.T);
    }
    const unsigned tmask = __ballot_sync(0xffffffffu, tie);
    const int tie_rank = ties_seen + __popc(tmask & ((1u << lane) - 1u));
    keep = keep || (tie && tie_rank < my_ties);
    ties_seen += __popc(tmask);
    const unsigned kmask = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int64_t p = pos + __popc(kmask & ((1u << lane) - 1u));
      if (p < end && p < cap) out_idx[p] = j;
      else report(d_status, p >= cap ? SPARSP_ERR_CAPACITY : SPARSP_ERR_DATA);
    }
    pos += __popc(kmask);
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

sparsp_status_t launch_balance(const Dims& s, const int32_t* row_ptr, int P, int max_moves,
                               int32_t* head_rank, int64_t* loads, int32_t* moves, cudaStream_t st) {
  balance_kernel<<<s.B, 1024, 0, st>>>(row_ptr, s.H, s.nb, P, max_moves, head_rank, loads, moves);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

size_t augment_ws(const Dims& s, int P) {
  const int64_t rows = s.rows();
  return align256((size_t)rows * s.nb * sizeof(uint32_t)) + align256((size_t)rows * sizeof(int32_t)) +
         align256((size_t)s.B * P * sizeof(RankOut));
}

sparsp_status_t launch_augment(const Dims& s, int P, const float* scores, const int32_t* row_ptr,
                               const int32_t* col_idx, const int32_t* head_rank, int32_t* out_ptr,
                               int32_t* out_idx, int64_t cap, int64_t* added, void* ws, int32_t* d_status,
                               cudaStream_t st) {
  const int64_t rows = s.rows();
  char* w = (char*)ws;
  uint32_t* keys = (uint32_t*)w;
  w += align256((size_t)rows * s.nb * sizeof(uint32_t));
  int32_t* taken = (int32_t*)w;
  w += align256((size_t)rows * sizeof(int32_t));
  RankOut* ro = (RankOut*)w;
  const unsigned grid = (unsigned)((rows + 7) / 8);
  aug_keys_kernel<<<grid, 256, 0, st>>>(scores, row_ptr, col_idx, s.nb, rows, keys, out_ptr, d_status);
  SPARSP_LAUNCH_CHECK();
  aug_rank_kernel<<<s.B * P, kRankThreads, 0, st>>>(row_ptr, head_rank, s.H, s.nb, P, keys, out_ptr, taken, ro,
                                                    added, d_status);
  SPARSP_LAUNCH_CHECK();
  sparsp_status_t r = launch_scan_counts(out_ptr, rows, st);
  if (r != SPARSP_OK) return r;
  aug_fill_kernel<<<grid, 256, 0, st>>>(row_ptr, col_idx, head_rank, s.H, s.nb, P, rows, keys, taken, ro, out_ptr,
                                        out_idx, cap, d_status);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace sparsp
