// Step 5c: longest-first work order, and the CSR transpose used by the backward.
//
// Grouped order (default): heads by total cost descending, then each head's
// query blocks by row cost descending, so that concurrently running CTAs work
// on few heads and their K/V stays L2-resident. Flat order: every item by row
// cost descending. Both break ties by index, so the order is deterministic.
// Ranks are computed by counting (no sort, no atomics on the output).
#include "common.cuh"

namespace sparsp {
namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads)
lpt_grouped_kernel(const int32_t* __restrict__ row_ptr, int BH, int nb, int32_t* __restrict__ items,
                   int32_t* __restrict__ counter) {
  __shared__ int32_t cost[kMaxBlocks];
  __shared__ int32_t head_rank;
  const int bh = blockIdx.x;
  if (threadIdx.x == 0) head_rank = 0;
  const int64_t r0 = (int64_t)bh * nb;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) cost[i] = row_ptr[r0 + i + 1] - row_ptr[r0 + i];
  __syncthreads();
  const int32_t mine = row_ptr[r0 + nb] - row_ptr[r0];
  int cnt = 0;
  for (int g = threadIdx.x; g < BH; g += blockDim.x) {
    const int32_t c = row_ptr[(int64_t)(g + 1) * nb] - row_ptr[(int64_t)g * nb];
    if (c > mine || (c == mine && g < bh)) ++cnt;
  }
  if (cnt) atomicAdd(&head_rank, cnt);
  __syncthreads();
  const int64_t slot0 = (int64_t)head_rank * nb;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) {
    const int32_t c = cost[i];
    int rank = 0;
    for (int i2 = 0; i2 < nb; ++i2) {
      const int32_t c2 = cost[i2];
      rank += (c2 > c) || (c2 == c && i2 < i);
    }
    items[slot0 + rank] = (int32_t)(r0 + i);
  }
  if (bh == 0 && threadIdx.x == 0 && counter != nullptr) *counter = 0;
}

constexpr int kMaxCost = kMaxBlocks;   // item costs are clamped to [0, cmax], cmax <= kMaxCost

// Flat order, pass 1: per-head histogram of item costs (0..cmax).
__global__ void __launch_bounds__(kThreads)
lpt_hist_kernel(const int32_t* __restrict__ row_ptr, int nb, int cmax, int32_t* __restrict__ hist) {
  __shared__ int32_t h[kMaxCost + 1];
  const int bh = blockIdx.x;
  for (int c = threadIdx.x; c <= cmax; c += blockDim.x) h[c] = 0;
  __syncthreads();
  const int64_t r0 = (int64_t)bh * nb;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) {
    int32_t c = row_ptr[r0 + i + 1] - row_ptr[r0 + i];
    c = c < 0 ? 0 : (c > cmax ? cmax : c);
    atomicAdd(&h[c], 1);
  }
  __syncthreads();
  for (int c = threadIdx.x; c <= cmax; c += blockDim.x) hist[(int64_t)bh * (cmax + 1) + c] = h[c];
}

// Flat order, pass 2: slot = #items with larger cost + #items of equal cost in
// earlier heads + #rows of equal cost earlier in this head.
__global__ void __launch_bounds__(kThreads)
lpt_place_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ hist, int BH,
                 int nb, int cmax, int32_t* __restrict__ items, int32_t* __restrict__ counter) {
  __shared__ int32_t greater[kMaxCost + 2];
  __shared__ int32_t before[kMaxCost + 1];
  __shared__ int16_t cost[kMaxBlocks];   // clamped to [0, cmax], cmax <= kMaxCost
  const int bh = blockIdx.x;
  const int64_t r0 = (int64_t)bh * nb;
  for (int c = threadIdx.x; c <= cmax; c += blockDim.x) {
    int32_t tot = 0, bef = 0;
    for (int g = 0; g < BH; ++g) {
      const int32_t v = hist[(int64_t)g * (cmax + 1) + c];
      tot += v;
      if (g < bh) bef += v;
    }
    greater[c] = tot;     // column totals for now
    before[c] = bef;
  }
  for (int i = threadIdx.x; i < nb; i += blockDim.x) {
    int32_t c = row_ptr[r0 + i + 1] - row_ptr[r0 + i];
    cost[i] = (int16_t)(c < 0 ? 0 : (c > cmax ? cmax : c));
  }
  __syncthreads();
  if (threadIdx.x == 0) {   // suffix sums: greater[c] = #items with cost > c
    int32_t run = 0;
    for (int c = cmax; c >= 0; --c) {
      const int32_t t = greater[c];
      greater[c] = run;
      run += t;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nb; i += blockDim.x) {
    const int32_t c = cost[i];
    int rank = 0;
    for (int i2 = 0; i2 < i; ++i2) rank += cost[i2] == c;
    items[(int64_t)greater[c] + before[c] + rank] = (int32_t)(r0 + i);
  }
  if (bh == 0 && threadIdx.x == 0 && counter != nullptr) *counter = 0;
}

constexpr int kBitmapMaxBlocks = 1024;

// CSR -> CSC per head beyond kBitmapMaxBlocks blocks. Rows are visited in
// order, one row per step, so each key block's list of query blocks comes out
// ascending.
__global__ void __launch_bounds__(kThreads)
csr_transpose_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col_idx,
                     int BH, int nb, int32_t* __restrict__ col_ptr, int32_t* __restrict__ row_idx,
                     int32_t* d_status) {
  __shared__ int32_t cnt[kMaxBlocks];
  __shared__ int32_t cursor[kMaxBlocks];
  __shared__ int32_t warp_tot[32];
  const int bh = blockIdx.x;
  const int64_t r0 = (int64_t)bh * nb;
  for (int j = threadIdx.x; j < nb; j += blockDim.x) cnt[j] = 0;
  __syncthreads();
  const int32_t e0 = row_ptr[r0], e1 = row_ptr[r0 + nb];
  for (int32_t e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
    const int32_t j = col_idx[e];
    if (j >= 0 && j < nb) atomicAdd(&cnt[j], 1);
    else report(d_status, SPARSP_ERR_DATA);
  }
  __syncthreads();
  // exclusive scan of cnt[0..nb): thread t takes the kPer entries from kPer*t
  // (nb <= kMaxBlocks = kPer * blockDim)
  constexpr int kPer = kMaxBlocks / kThreads;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j0 = threadIdx.x * kPer;
  int32_t v = 0;
#pragma unroll
  for (int u = 0; u < kPer; ++u) v += j0 + u < nb ? cnt[j0 + u] : 0;
  int32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t t = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += o;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  int32_t excl = (warp > 0 ? warp_tot[warp - 1] : 0) + incl - v;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int j = j0 + u;
    if (j < nb) {
      col_ptr[r0 + j] = e0 + excl;
      cursor[j] = e0 + excl;
      excl += cnt[j];
    }
  }
  if (bh == BH - 1 && threadIdx.x == 0) col_ptr[(int64_t)BH * nb] = row_ptr[(int64_t)BH * nb];
  __syncthreads();
  for (int i = 0; i < nb; ++i) {
    const int32_t a = row_ptr[r0 + i], b = row_ptr[r0 + i + 1];
    for (int32_t e = a + threadIdx.x; e < b; e += blockDim.x) {
      const int32_t jj = col_idx[e];
      if (jj >= 0 && jj < nb) {
        const int32_t pos = atomicAdd(&cursor[jj], 1);   // distinct jj within a row
        if (dcheck(pos >= e0 && pos < e1, d_status)) row_idx[pos] = i;
      }
    }
    __syncthreads();
  }
}

// Up to kBitmapMaxBlocks blocks: the head's CSR as a row-major bitmap in
// shared memory ([nb][ceil(nb/32)] words); thread j then walks column j down
// the rows and writes its list in ascending row order. A row listing an index
// twice, or one outside [0, nb), sets SPARSP_ERR_DATA.

__global__ void __launch_bounds__(kThreads)
csr_transpose_bitmap_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col_idx,
                            int BH, int nb, int32_t* __restrict__ col_ptr, int32_t* __restrict__ row_idx,
                            int32_t* d_status) {
  extern __shared__ uint32_t bm[];   // [nb][W]
  __shared__ int32_t cnt[kBitmapMaxBlocks];
  __shared__ int32_t warp_tot[32];
  const int bh = blockIdx.x;
  const int64_t r0 = (int64_t)bh * nb;
  const int W = (nb + 31) >> 5;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int w = threadIdx.x; w < nb * W; w += blockDim.x) bm[w] = 0u;
  for (int j = threadIdx.x; j < nb; j += blockDim.x) cnt[j] = 0;
  __syncthreads();
  // one warp per row: its bits and the column counts
  for (int i = warp; i < nb; i += nwarps) {
    const int32_t a = row_ptr[r0 + i], b = row_ptr[r0 + i + 1];
    bool bad = b < a;
    for (int32_t e = a + lane; e < b && !bad; e += 32) {
      const int32_t j = col_idx[e];
      if (j < 0 || j >= nb) {
        bad = true;
      } else {
        atomicOr(&bm[i * W + (j >> 5)], 1u << (j & 31));
        atomicAdd(&cnt[j], 1);
      }
    }
    __syncwarp();
    int c = 0;
    for (int w = lane; w < W; w += 32) c += __popc(bm[i * W + w]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
    if (__any_sync(0xffffffffu, bad) || (b >= a && c != b - a)) {
      if (lane == 0) report(d_status, SPARSP_ERR_DATA);
    }
  }
  __syncthreads();
  // exclusive scan of the counts (one entry per thread: nb <= blockDim)
  const int32_t e0 = row_ptr[r0];
  const int j = threadIdx.x;
  const int32_t v = j < nb ? cnt[j] : 0;
  int32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t t = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, t, off);
      if (lane >= off) t += o;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  int32_t pos = e0 + (warp > 0 ? warp_tot[warp - 1] : 0) + incl - v;
  if (j < nb) col_ptr[r0 + j] = pos;
  if (bh == BH - 1 && threadIdx.x == 0) col_ptr[(int64_t)BH * nb] = row_ptr[(int64_t)BH * nb];
  // column j, down the rows
  if (j < nb) {
    const int32_t end = pos + v;
    const uint32_t bit = 1u << (j & 31);
    const uint32_t* col = bm + (j >> 5);
    for (int i = 0; i < nb; ++i)
      if (col[i * W] & bit) {
        if (dcheck(pos < end, d_status)) row_idx[pos] = i;
        ++pos;
      }
  }
}

}  // namespace

// Histogram space for costs up to 2*nb (the pair items of 64-token blocks cost
// the sum of two rows).
size_t lpt_ws(const Dims& s) { return (size_t)s.B * s.H * (2 * s.nb + 1) * sizeof(int32_t); }

sparsp_status_t launch_lpt(const Dims& s, const int32_t* row_ptr, bool flat, int32_t* items,
                           int32_t* counter, void* ws, cudaStream_t st, int cmax) {
  const int BH = s.B * s.H;
  if (cmax <= 0) cmax = s.nb;
  if (cmax > kMaxCost) cmax = kMaxCost;   // the flat order then ties the costliest items
  if (!flat) {
    lpt_grouped_kernel<<<BH, kThreads, 0, st>>>(row_ptr, BH, s.nb, items, counter);
    SPARSP_LAUNCH_CHECK();
  } else {
    int32_t* hist = (int32_t*)ws;
    lpt_hist_kernel<<<BH, kThreads, 0, st>>>(row_ptr, s.nb, cmax, hist);
    SPARSP_LAUNCH_CHECK();
    lpt_place_kernel<<<BH, kThreads, 0, st>>>(row_ptr, hist, BH, s.nb, cmax, items, counter);
    SPARSP_LAUNCH_CHECK();
  }
  return SPARSP_OK;
}

namespace {

// Pair rows of 64-token blocks: pair p of head bh covers query blocks 2p and
// 2p + 1 (2p alone when nb is odd and 2p = nb - 1), so its "row" in a CSR of
// B*H*ceil(nb/2) rows starts where row 2p starts.
__global__ void pair_ptr_kernel(const int32_t* __restrict__ row_ptr, int64_t BH, int nb, int nbp,
                                int32_t* __restrict__ pair_ptr) {
  const int64_t n = BH * nbp;
  for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x <= n; x += (int64_t)gridDim.x * blockDim.x)
    pair_ptr[x] = x == n ? row_ptr[BH * nb] : row_ptr[(x / nbp) * nb + 2 * (x % nbp)];
}

}  // namespace

sparsp_status_t launch_pair_ptr(const Dims& s, const int32_t* row_ptr, int32_t* pair_ptr, cudaStream_t st) {
  const int64_t BH = (int64_t)s.B * s.H;
  const int nbp = (s.nb + 1) / 2;
  const int64_t n = BH * nbp + 1;
  const int threads = 256;
  int64_t blocks = (n + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  pair_ptr_kernel<<<(unsigned)blocks, threads, 0, st>>>(row_ptr, BH, s.nb, nbp, pair_ptr);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

sparsp_status_t launch_csr_transpose(const Dims& s, const int32_t* row_ptr, const int32_t* col_idx,
                                     int32_t* col_ptr, int32_t* row_idx, int32_t* d_status,
                                     cudaStream_t st) {
  const int BH = s.B * s.H;
  if (s.nb <= kBitmapMaxBlocks) {
    const size_t smem = (size_t)s.nb * ((s.nb + 31) / 32) * sizeof(uint32_t);   // up to 128 KB
    if (cudaFuncSetAttribute(csr_transpose_bitmap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return SPARSP_ERR_CUDA;
    csr_transpose_bitmap_kernel<<<BH, kThreads, smem, st>>>(row_ptr, col_idx, BH, s.nb, col_ptr, row_idx,
                                                            d_status);
    SPARSP_LAUNCH_CHECK();
    return SPARSP_OK;
  }
  csr_transpose_kernel<<<BH, kThreads, 0, st>>>(row_ptr, col_idx, BH, s.nb, col_ptr, row_idx,
                                                d_status);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace sparsp
