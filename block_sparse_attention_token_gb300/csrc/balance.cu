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
//                    blocks get key 0. Also writes the row's base count. Rows
//                    of ranks without slack get no keys (nothing is read there).
//  aug_slack/count/hist/digit kernels - per (batch element, rank): slack =
//                    L* - L_r; candidates and the 8-bit digit histograms of a
//                    4-pass radix select are accumulated over all the rank's
//                    heads by CTAs of (head, key range); one CTA per rank fixes
//                    each digit. The result is the key T of the slack-th best
//                    candidate: keys above T are taken, and of the keys equal to
//                    T the first ones in (row, block) order.
//  aug_rowcount/tie kernels - each row's keys above T (one warp per row), and
//                    the ties shared out in (head, row) order where there are any.
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

constexpr int kRankThreads = 1024;
constexpr int kRankWarps = kRankThreads / 32;
constexpr int kKeysPerCta = 8192;   // key range of one CTA of a histogram pass

struct RankOut {
  uint32_t T;        // keys > T are taken
  uint32_t pad;
  int64_t need_eq;   // and this many keys == T, first in (head, row, block) order
};

// Selection state of one (batch element, rank), in the workspace.
struct RankState {
  unsigned long long slack;   // L* - L_r
  unsigned long long rem;     // rank of the cut among the keys matching prefix
  uint32_t prefix, mask;      // digits fixed so far
  int32_t done, pad;
};

constexpr int kMaxWords = 32;   // nb <= 1024

__global__ void __launch_bounds__(256)
aug_keys_kernel(const float* __restrict__ scores, const int32_t* __restrict__ row_ptr,
                const int32_t* __restrict__ col_idx, const int32_t* __restrict__ head_rank,
                const RankState* __restrict__ state, int H, int nb, int P, int64_t rows,
                uint32_t* __restrict__ keys, int32_t* __restrict__ counts, int32_t* d_status) {
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
  // rows of a rank without slack (or of no rank) take nothing: no keys
  const int64_t bh = row / nb;
  const int q = head_rank[bh];
  if (q < 0 || q >= P || state[(bh / H) * P + q].slack == 0ull) return;
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
  // Selected blocks get key 0. The candidates are compacted first, so that
  // the slow double-precision division runs on full warps of them.
  for (int j = lane; j < nb; j += 32)
    if ((bits[j >> 5] >> (j & 31)) & 1u) K[j] = 0u;
  const int words = (nb + 31) >> 5;
  uint32_t cw = 0u;
  if (lane < words) {
    const int tail = nb - lane * 32;
    cw = ~bits[lane] & (tail >= 32 ? 0xffffffffu : (1u << tail) - 1u);
  }
  const int pc = __popc(cw);
  int incl = pc;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  const int n_cand = __shfl_sync(0xffffffffu, incl, 31);
  __shared__ int32_t cpre_all[8][32];
  __shared__ uint32_t cword_all[8][32];
  int32_t* cpre = cpre_all[warp];
  uint32_t* cword = cword_all[warp];
  cpre[lane] = incl - pc;
  cword[lane] = cw;
  __syncwarp();
  for (int c = lane; c < n_cand; c += 32) {
    int w = 0;   // the last word that starts at or before candidate c
#pragma unroll
    for (int step = 16; step > 0; step >>= 1)   // w + step stays <= 31
      if (cpre[w + step] <= c) w += step;
    uint32_t x = cword[w];
    for (int n = c - cpre[w]; n > 0; --n) x &= x - 1u;   // drop the lower candidates of the word
    const int j = w * 32 + __ffs(x) - 1;
    const float v = (float)((double)expf(S[j] - m) / Z);
    K[j] = __float_as_uint(v) + 1u;
  }
}

// One CTA per batch element: rank loads, slack, fresh selection state and
// cleared histograms. A rank without slack is finished here.
__global__ void __launch_bounds__(kRankThreads)
aug_slack_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ head_rank, int H, int nb, int P,
                 RankState* __restrict__ state, RankOut* __restrict__ rank_out, int64_t* __restrict__ added,
                 unsigned long long* __restrict__ hist, int32_t* d_status) {
  __shared__ unsigned long long load[kMaxHeads];
  __shared__ unsigned long long red[32];
  const int b = blockIdx.x;
  for (int q = threadIdx.x; q < P; q += kRankThreads) load[q] = 0ull;
  for (int i = threadIdx.x; i < P * 256; i += kRankThreads) hist[(int64_t)b * P * 256 + i] = 0ull;
  __syncthreads();
  for (int h = threadIdx.x; h < H; h += kRankThreads) {
    const int q = head_rank[(int64_t)b * H + h];
    if (q < 0 || q >= P) {
      report(d_status, SPARSP_ERR_DATA);
      continue;
    }
    atomicAdd(&load[q], (unsigned long long)head_cost(row_ptr, (int64_t)b * H + h, nb));
  }
  __syncthreads();
  unsigned long long top = 0ull;
  for (int q = threadIdx.x; q < P; q += kRankThreads) top = load[q] > top ? load[q] : top;
  top = ~block_min(~top, red);
  for (int q = threadIdx.x; q < P; q += kRankThreads) {
    const int64_t br = (int64_t)b * P + q;
    const unsigned long long slack = top - load[q];
    state[br] = RankState{slack, 0ull, 0u, 0u, slack == 0ull, 0};
    if (slack == 0ull) {
      rank_out[br] = RankOut{0xffffffffu, 0u, 0};
      if (added != nullptr) added[br] = 0;
    }
  }
}

// grid (b*H + h, key range): histogram of the 8-bit digit at `shift` of the
// head's nonzero keys that match its rank's prefix, added into the rank's
// global histogram.
__global__ void __launch_bounds__(256)
aug_hist_kernel(const int32_t* __restrict__ head_rank, int H, int P, int nb, const uint32_t* __restrict__ keys,
                const RankState* __restrict__ state, unsigned long long* __restrict__ hist, int shift) {
  __shared__ int32_t h2[2][256];
  const int64_t bh = blockIdx.x;
  const int q = head_rank[bh];
  if (q < 0 || q >= P) return;
  const int64_t br = (bh / H) * P + q;
  const RankState st = state[br];
  if (st.done) return;
  h2[0][threadIdx.x] = 0;
  h2[1][threadIdx.x] = 0;
  __syncthreads();
  const int64_t per_head = (int64_t)nb * nb;
  const int64_t e0 = (int64_t)blockIdx.y * kKeysPerCta;
  const int64_t e1 = e0 + kKeysPerCta < per_head ? e0 + kKeysPerCta : per_head;
  const uint32_t* K = keys + bh * per_head;
  int32_t* mine = h2[(threadIdx.x >> 5) & 1];
  for (int64_t e = e0 + threadIdx.x; e < e1; e += 256) {
    const uint32_t k = K[e];
    if (k != 0u && (k & st.mask) == st.prefix) atomicAdd(&mine[(k >> shift) & 255u], 1);
  }
  __syncthreads();
  const int c = h2[0][threadIdx.x] + h2[1][threadIdx.x];
  if (c) atomicAdd(&hist[br * 256 + threadIdx.x], (unsigned long long)c);
}

// One CTA of 256 threads per (batch element, rank): fixes the digit at
// `shift` from the pass's histogram and clears it. The first pass (shift 24,
// empty prefix) also counts the candidates: a rank whose slack covers them
// all takes every one (T = 0), one without any takes none.
__global__ void __launch_bounds__(256)
aug_digit_kernel(RankState* __restrict__ state, unsigned long long* __restrict__ hist,
                 RankOut* __restrict__ rank_out, int64_t* __restrict__ added, int shift) {
  __shared__ unsigned long long warp_sum[8];
  __shared__ unsigned long long s_rem;
  __shared__ int s_stop;
  const int64_t br = blockIdx.x;
  RankState* st = state + br;
  const int done0 = st->done;
  const unsigned long long slack = st->slack;
  unsigned long long rem = st->rem;
  __syncthreads();   // every thread has read the state before thread 0 updates it
  if (done0) return;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  unsigned long long* hh = hist + br * 256;
  const int d = 255 - t;   // thread t holds digit 255 - t: an inclusive scan gives suffix sums
  const unsigned long long c = hh[d];
  unsigned long long incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  unsigned long long total = 0ull;
  for (int w = 0; w < 8; ++w) {
    if (w < warp) incl += warp_sum[w];
    total += warp_sum[w];
  }
  hh[d] = 0ull;   // every thread has read its digit
  if (t == 0) s_stop = 0;
  if (shift == 24) {
    const unsigned long long sel = slack < total ? slack : total;
    if (t == 0) {
      if (added != nullptr) added[br] = (int64_t)sel;
      if (sel == 0ull || sel == total) {
        rank_out[br] = RankOut{sel == 0ull ? 0xffffffffu : 0u, 0u, 0};
        st->done = 1;
        s_stop = 1;
      }
    }
    rem = sel;
  }
  __syncthreads();
  if (s_stop) return;
  // The cut's digit is the largest d whose suffix sum reaches rem (the suffix
  // sums grow as d falls, and the one at d = 0 is the total, at least rem).
  const int reach = __syncthreads_count(incl >= rem);
  const int dstar = reach - 1;
  if (d == dstar) s_rem = rem - (incl - c);
  __syncthreads();
  if (t == 0) {
    st->prefix |= (uint32_t)dstar << shift;
    st->mask |= 255u << shift;
    st->rem = s_rem;
    if (shift == 0) {
      rank_out[br] = RankOut{st->prefix, 0u, (int64_t)s_rem};
      st->done = 1;
    }
  }
}

// One warp per CSR row: blocks above the rank's cut, and keys equal to it.
// Without ties to share (need_eq = 0) the row's count is final here.
__global__ void __launch_bounds__(256)
aug_rowcount_kernel(const int32_t* __restrict__ head_rank, int H, int P, int nb, int64_t rows,
                    const uint32_t* __restrict__ keys, const RankOut* __restrict__ rank_out,
                    int32_t* __restrict__ counts, int32_t* __restrict__ taken, int32_t* __restrict__ gtrow,
                    int32_t* __restrict__ eqrow) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int64_t bh = row / nb;
  const int q = head_rank[bh];
  if (q < 0 || q >= P) {
    if (lane == 0) taken[row] = 0;
    return;
  }
  const RankOut ro = rank_out[(bh / H) * P + q];
  const uint32_t* K = keys + row * nb;
  int gt = 0, eq = 0;
  if (ro.T != 0xffffffffu) {   // else the rank takes nothing and may have no keys
    for (int j = lane; j < nb; j += 32) {
      const uint32_t key = K[j];
      gt += key > ro.T && key != 0u;
      eq += key == ro.T && key != 0u;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, off);
    eq += __shfl_xor_sync(0xffffffffu, eq, off);
  }
  if (lane == 0) {
    if (ro.need_eq == 0) {
      counts[row] += gt;
      taken[row] = 0;
    } else {
      gtrow[row] = gt;
      eqrow[row] = eq;
    }
  }
}

// Exclusive prefix sum over the CTA (kRankThreads threads); `total` gets the
// sum of all. `warp_sum` holds kRankWarps entries.
__device__ int64_t block_excl_scan(int64_t v, int64_t* warp_sum, int64_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  __syncthreads();   // earlier readers of warp_sum are done
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  int64_t before = 0, all = 0;
  for (int w = 0; w < kRankWarps; ++w) {
    const int64_t x = warp_sum[w];
    before += w < warp ? x : 0;
    all += x;
  }
  total = all;
  return before + incl - v;
}

// One CTA per (batch element, rank) with ties to share: the first need_eq
// keys equal to the cut, in (head, row, block) order, go to their rows. The
// rank's heads are compacted in ascending order, then its rows are taken
// kRankThreads at a time with a prefix sum of their tie counts.
__global__ void __launch_bounds__(kRankThreads)
aug_tie_kernel(const int32_t* __restrict__ head_rank, int H, int nb, int P, const RankOut* __restrict__ rank_out,
               const int32_t* __restrict__ gtrow, const int32_t* __restrict__ eqrow, int32_t* __restrict__ counts,
               int32_t* __restrict__ taken) {
  __shared__ int32_t heads[kMaxHeads];
  __shared__ int64_t warp_sum[kRankWarps];
  const int b = blockIdx.x / P, r = blockIdx.x % P;
  const int64_t need_eq = rank_out[blockIdx.x].need_eq;
  if (need_eq == 0) return;
  const int tid = threadIdx.x;
  int64_t n_heads = 0;
  for (int h0 = 0; h0 < H; h0 += kRankThreads) {
    const int h = h0 + tid;
    const bool mine = h < H && head_rank[(int64_t)b * H + h] == r;
    int64_t n;
    const int64_t pos = n_heads + block_excl_scan(mine ? 1 : 0, warp_sum, n);
    if (mine) heads[pos] = h;
    n_heads += n;
  }
  __syncthreads();
  const int64_t nrows = n_heads * nb;
  int64_t tie_base = 0;
  for (int64_t k0 = 0; k0 < nrows; k0 += kRankThreads) {
    const int64_t k = k0 + tid;
    int64_t row = -1;
    int eq = 0;
    if (k < nrows) {
      row = ((int64_t)b * H + heads[k / nb]) * nb + k % nb;
      eq = eqrow[row];
    }
    int64_t sum;
    const int64_t before = tie_base + block_excl_scan(eq, warp_sum, sum);
    if (row >= 0) {
      int64_t tk = need_eq - before;
      tk = tk < 0 ? 0 : (tk > eq ? eq : tk);
      taken[row] = (int32_t)tk;
      counts[row] += gtrow[row] + (int32_t)tk;
    }
    tie_base += sum;
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
  const RankOut ro = valid ? rank_out[(bh / H) * P + q] : RankOut{0xffffffffu, 0u, 0};
  const bool takes = ro.T != 0xffffffffu;   // else the row may have no keys
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
      const uint32_t key = takes ? K[j] : 0u;
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
  const size_t br = (size_t)s.B * P;
  return align256((size_t)rows * s.nb * sizeof(uint32_t)) + 3 * align256((size_t)rows * sizeof(int32_t)) +
         align256(br * sizeof(RankOut)) + align256(br * sizeof(RankState)) +
         align256(br * 256 * sizeof(unsigned long long));
}

sparsp_status_t launch_augment(const Dims& s, int P, const float* scores, const int32_t* row_ptr,
                               const int32_t* col_idx, const int32_t* head_rank, int32_t* out_ptr,
                               int32_t* out_idx, int64_t cap, int64_t* added, void* ws, int32_t* d_status,
                               cudaStream_t st) {
  const int64_t rows = s.rows();
  const size_t br = (size_t)s.B * P;
  char* w = (char*)ws;
  uint32_t* keys = (uint32_t*)w;
  w += align256((size_t)rows * s.nb * sizeof(uint32_t));
  int32_t* taken = (int32_t*)w;
  w += align256((size_t)rows * sizeof(int32_t));
  int32_t* gtrow = (int32_t*)w;
  w += align256((size_t)rows * sizeof(int32_t));
  int32_t* eqrow = (int32_t*)w;
  w += align256((size_t)rows * sizeof(int32_t));
  RankOut* ro = (RankOut*)w;
  w += align256(br * sizeof(RankOut));
  RankState* state = (RankState*)w;
  w += align256(br * sizeof(RankState));
  unsigned long long* hist = (unsigned long long*)w;

  const unsigned grid = (unsigned)((rows + 7) / 8);
  aug_slack_kernel<<<s.B, kRankThreads, 0, st>>>(row_ptr, head_rank, s.H, s.nb, P, state, ro, added, hist,
                                                 d_status);
  SPARSP_LAUNCH_CHECK();
  aug_keys_kernel<<<grid, 256, 0, st>>>(scores, row_ptr, col_idx, head_rank, state, s.H, s.nb, P, rows, keys,
                                        out_ptr, d_status);
  SPARSP_LAUNCH_CHECK();
  const int64_t per_head = (int64_t)s.nb * s.nb;
  const dim3 hgrid((unsigned)(s.B * s.H), (unsigned)((per_head + kKeysPerCta - 1) / kKeysPerCta));
  for (int shift = 24; shift >= 0; shift -= 8) {
    aug_hist_kernel<<<hgrid, 256, 0, st>>>(head_rank, s.H, P, s.nb, keys, state, hist, shift);
    SPARSP_LAUNCH_CHECK();
    aug_digit_kernel<<<(unsigned)br, 256, 0, st>>>(state, hist, ro, added, shift);
    SPARSP_LAUNCH_CHECK();
  }
  aug_rowcount_kernel<<<grid, 256, 0, st>>>(head_rank, s.H, P, s.nb, rows, keys, ro, out_ptr, taken, gtrow, eqrow);
  SPARSP_LAUNCH_CHECK();
  aug_tie_kernel<<<(unsigned)br, kRankThreads, 0, st>>>(head_rank, s.H, s.nb, P, ro, gtrow, eqrow, out_ptr, taken);
  SPARSP_LAUNCH_CHECK();
  sparsp_status_t r = launch_scan_counts(out_ptr, rows, st);
  if (r != SPARSP_OK) return r;
  aug_fill_kernel<<<grid, 256, 0, st>>>(row_ptr, col_idx, head_rank, s.H, s.nb, P, rows, keys, taken, ro, out_ptr,
                                        out_idx, cap, d_status);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace sparsp
