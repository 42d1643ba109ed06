// Step 2: block-score estimation.
//
// pool_kernel: one CTA per (tile, b*H+h, tensor) reads the tile's Bt x d
// block-ordered rows with 16-byte loads and writes the fp32 column means; for
// the low-rank predictor it then projects the mean through W[h] (d x rank).
// Summation order is fixed: 16 row lanes each sum a strided set of rows in
// order, then the 16 partial sums are added in lane order.
//
// product_kernel: S = A . B^T per head with A, B = pooled [nb, dd] fp32,
// dd = d (mean) or rank (low-rank); a 64x64 output tile per CTA (4x4 per
// thread), the dd reduction in index order with fmaf.
#include "common.cuh"

namespace sparsp {
namespace {

constexpr int kPoolThreads = 256;

__device__ __forceinline__ void add_vec(float* acc, const uint4& v, bool bf16) {
  if (bf16) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 f = __bfloat1622float2(p[e]);
      acc[2 * e] += f.x;
      acc[2 * e + 1] += f.y;
    }
  } else {
    const float* p = reinterpret_cast<const float*>(&v);
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] += p[e];
  }
}

// blockIdx.x = tile, blockIdx.y = b*H + h, blockIdx.z = 0 for Q, 1 for K.
__global__ void __launch_bounds__(kPoolThreads)
pool_kernel(const uint4* __restrict__ q, const uint4* __restrict__ k, int H, int64_t N, int Bt,
            int d, int bf16, const float* __restrict__ wq, const float* __restrict__ wk, int rank,
            float* __restrict__ out_q, float* __restrict__ out_k, int out_dim) {
  __shared__ float part[kPoolThreads][9];     // per thread: up to 8 column sums (+1 pad)
  __shared__ float mean[128];
  const int j = blockIdx.x;
  const int bh = blockIdx.y;
  const bool is_k = blockIdx.z != 0;
  const uint4* src = is_k ? k : q;
  const int elems_per_vec = bf16 ? 8 : 4;
  const int vec_per_row = d / elems_per_vec;           // 8 or 16 (bf16), 16 or 32 (fp32)
  const int lanes_per_row = vec_per_row;                // one 16-byte vector per thread per row
  const int row_groups = kPoolThreads / lanes_per_row;  // rows processed concurrently
  const int vcol = threadIdx.x % lanes_per_row;
  const int rg = threadIdx.x / lanes_per_row;
  const int64_t row0 = (int64_t)bh * N + (int64_t)j * Bt;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  if (rg < row_groups) {
    for (int r = rg; r < Bt; r += row_groups) {
      uint4 v = __ldcs(src + (row0 + r) * vec_per_row + vcol);
      add_vec(acc, v, bf16 != 0);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) part[threadIdx.x][e] = acc[e];
  __syncthreads();
  // column c = vcol*elems_per_vec + e; reduce over row groups in order
  const float inv = 1.0f / (float)Bt;   // Bt is a power of two: exact
  if (threadIdx.x < d) {
    const int c = threadIdx.x;
    const int vc = c / elems_per_vec, e = c % elems_per_vec;
    float s = 0.f;
    for (int g = 0; g < row_groups; ++g) s += part[g * lanes_per_row + vc][e];
    mean[c] = s * inv;
  }
  __syncthreads();
  const int64_t blk = (int64_t)bh * (N / Bt) + j;
  float* dst = (is_k ? out_k : out_q) + blk * out_dim;
  if (wq == nullptr) {
    if (threadIdx.x < d) dst[threadIdx.x] = mean[threadIdx.x];
  } else {
    const int h = bh % H;
    const float* W = (is_k ? wk : wq) + (int64_t)h * d * rank;
    if (threadIdx.x < rank) {
      const int r = threadIdx.x;
      float s = 0.f;
      for (int c = 0; c < d; ++c) s = fmaf(mean[c], W[(int64_t)c * rank + r], s);
      dst[r] = s;
    }
  }
}

constexpr int kTile = 64;        // output tile kTile x kTile per CTA

// S = A B^T for one head, A, B: [nb, dd] fp32. 256 threads, each owning a 4x4
// block of outputs (rows 4*ty.., columns 4*tx..); the whole dd extent of both
// input tiles is staged in shared memory (rows padded by one word). Every
// output is one fmaf chain over c = 0..dd-1 in order.
// blockIdx.x = column tile, blockIdx.y = row tile, blockIdx.z = b*H + h.
__global__ void __launch_bounds__(256)
product_kernel(const float* __restrict__ A, const float* __restrict__ Bm, int nb, int dd,
               float* __restrict__ S) {
  extern __shared__ float sm[];
  const int ld = dd + 1;
  float* sa = sm;                  // [kTile][ld]
  float* sb = sm + kTile * ld;     // [kTile][ld]
  const int bh = blockIdx.z;
  const int i0 = blockIdx.y * kTile, j0 = blockIdx.x * kTile;
  const float* a = A + (int64_t)bh * nb * dd;
  const float* bm = Bm + (int64_t)bh * nb * dd;
  for (int e = threadIdx.x; e < kTile * dd; e += 256) {
    const int r = e / dd, c = e % dd;
    sa[r * ld + c] = i0 + r < nb ? a[(int64_t)(i0 + r) * dd + c] : 0.f;
    sb[r * ld + c] = j0 + r < nb ? bm[(int64_t)(j0 + r) * dd + c] : 0.f;
  }
  __syncthreads();
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) acc[u][v] = 0.f;
  for (int c = 0; c < dd; ++c) {
    float av[4], bv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) av[u] = sa[(4 * ty + u) * ld + c];
#pragma unroll
    for (int v = 0; v < 4; ++v) bv[v] = sb[(4 * tx + v) * ld + c];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
  }
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int i = i0 + 4 * ty + u, jj = j0 + 4 * tx + v;
      if (i < nb && jj < nb) S[((int64_t)bh * nb + i) * nb + jj] = acc[u][v];
    }
}

sparsp_status_t launch_product(const float* a, const float* b, int nb, int dd, int BH, float* S,
                               cudaStream_t st) {
  const size_t smem = 2 * (size_t)kTile * (dd + 1) * sizeof(float);
  if (cudaFuncSetAttribute(product_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SPARSP_ERR_CUDA;
  dim3 grid((nb + kTile - 1) / kTile, (nb + kTile - 1) / kTile, BH);
  product_kernel<<<grid, 256, smem, st>>>(a, b, nb, dd, S);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

// Low-rank projection of pooled means: out[blk, r] = sum_c mean[blk, c] W[h, c, r]
// (c in order, fmaf). blockIdx.x = tile, blockIdx.y = b*H + h, blockIdx.z = Q (0) or K (1).
__global__ void __launch_bounds__(64)
project_kernel(const float* __restrict__ qm, const float* __restrict__ km, const float* __restrict__ wq,
               const float* __restrict__ wk, int H, int nb, int d, int rank, float* __restrict__ pq,
               float* __restrict__ pk) {
  const int r = threadIdx.x;
  if (r >= rank) return;
  const bool is_k = blockIdx.z != 0;
  const int bh = blockIdx.y, h = bh % H;
  const int64_t blk = (int64_t)bh * nb + blockIdx.x;
  const float* mean = (is_k ? km : qm) + blk * d;
  const float* W = (is_k ? wk : wq) + (int64_t)h * d * rank;
  float acc = 0.f;
  for (int c = 0; c < d; ++c) acc = fmaf(mean[c], W[(int64_t)c * rank + r], acc);
  (is_k ? pk : pq)[blk * rank + r] = acc;
}

}  // namespace

size_t scores_from_means_ws(const Dims& s, int estimator, int rank) {
  return estimator == SPARSP_EST_LOWRANK ? 2 * (size_t)s.B * s.H * s.nb * rank * sizeof(float) : 0;
}

sparsp_status_t launch_scores_from_means(const Dims& s, int estimator, const float* qm,
                                         const float* km, const float* wq, const float* wk,
                                         int rank, float* scores, void* ws, cudaStream_t st) {
  const float* a = qm;
  const float* bm = km;
  int dd = s.d;
  if (estimator == SPARSP_EST_LOWRANK) {
    float* pq = (float*)ws;
    float* pk = pq + (size_t)s.B * s.H * s.nb * rank;
    project_kernel<<<dim3(s.nb, s.B * s.H, 2), 64, 0, st>>>(qm, km, wq, wk, s.H, s.nb, s.d, rank, pq, pk);
    SPARSP_LAUNCH_CHECK();
    a = pq;
    bm = pk;
    dd = rank;
  }
  return launch_product(a, bm, s.nb, dd, s.B * s.H, scores, st);
}

size_t block_scores_ws(const Dims& s, int estimator, int rank) {
  const int dd = estimator == SPARSP_EST_LOWRANK ? rank : s.d;
  return 2 * (size_t)s.B * s.H * s.nb * dd * sizeof(float);
}

sparsp_status_t launch_block_scores(const Dims& s, int estimator, const void* q, const void* k,
                                    const float* wq, const float* wk, int rank, float* scores,
                                    void* ws, cudaStream_t st) {
  const bool low = estimator == SPARSP_EST_LOWRANK;
  const int dd = low ? rank : s.d;
  float* pq = (float*)ws;
  float* pk = pq + (size_t)s.B * s.H * s.nb * dd;
  dim3 g1(s.nb, s.B * s.H, 2);
  pool_kernel<<<g1, kPoolThreads, 0, st>>>((const uint4*)q, (const uint4*)k, s.H, s.N, s.Bt, s.d,
                                           s.dtype == SPARSP_BF16, low ? wq : nullptr,
                                           low ? wk : nullptr, rank, pq, pk, dd);
  SPARSP_LAUNCH_CHECK();
  return launch_product(pq, pk, s.nb, dd, s.B * s.H, scores, st);
}

}  // namespace sparsp
