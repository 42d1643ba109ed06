// Fitting the per-head low-rank predictor to the real block scores.
//
// Loss per head h (the mean squared error of the predicted block scores):
//   E[b,h,i,j] = (qm_i Wq[h]) . (km_j Wk[h]) - qm_i . km_j
//   L[h] = sum_{b,i,j} E^2 / (B nb^2)
// with gradients
//   dL/dWq[h] = 2/(B nb^2) sum_b qm^T (E (km Wk)),  dL/dWk[h] = 2/(B nb^2) sum_b km^T (E^T (qm Wq)).
//
//  1. scores of both kinds from the pooled means (the projections qm Wq and
//     km Wk come out of the low-rank pass, in the workspace);
//  2. ge_kernel   - grid (b*H + h, block of 32 rows): GA = E (km Wk),
//     GB = E^T (qm Wq), with E's row and column tiles staged in shared memory;
//  3. loss_part_kernel - grid (h, chunk): fp64 partial sums of the squared
//     errors (fixed strided subsets, a fixed tree); loss_final_kernel adds
//     each head's partials in chunk order;
//  4. gw_kernel   - grid (h, dd): the weight gradients (row slices summed in a
//     fixed tree) and, when lr != 0, the step W -= lr dL/dW in place (the
//     projections were taken before it).
// Every sum has a fixed order, so results are bitwise reproducible.
#include "common.cuh"

namespace sparsp {
namespace {

constexpr int kThreads = 256;

constexpr int kGeRows = 32;   // rows i of GA and GB per CTA
constexpr int kGeJ = 32;      // j per shared-memory stage
constexpr int kGeOut = 8;     // outputs per thread: 32 * rank / kThreads, rank <= 64

// grid (b*H + h, block of kGeRows rows): GA[i,c] = sum_j E[i,j] B[j,c] and
// GB[i,c] = sum_j E[j,i] A[j,c] with E = Sp - St. E's row and column tiles
// and the matching rows of A and B are staged in shared memory kGeJ at a time;
// every output is one sequential fmaf chain over j.
__global__ void __launch_bounds__(kThreads)
ge_kernel(const float* __restrict__ sp, const float* __restrict__ st, const float* __restrict__ pq,
          const float* __restrict__ pk, int nb, int rank, float* __restrict__ ga, float* __restrict__ gb) {
  __shared__ float er[kGeRows][kGeJ + 1];   // E[i0 + ii][j0 + jj]
  __shared__ float ec[kGeJ][kGeRows + 1];   // E[j0 + jj][i0 + ii]
  __shared__ float as[kGeJ * 64], bs[kGeJ * 64];
  const int64_t bh = blockIdx.x;
  const int i0 = blockIdx.y * kGeRows;
  const float* P = sp + bh * nb * nb;
  const float* T = st + bh * nb * nb;
  const float* A = pq + bh * nb * rank;
  const float* Bk = pk + bh * nb * rank;
  const int nout = kGeRows * rank;
  float a[kGeOut], b[kGeOut];
#pragma unroll
  for (int k = 0; k < kGeOut; ++k) a[k] = b[k] = 0.f;
  for (int j0 = 0; j0 < nb; j0 += kGeJ) {
    for (int x = threadIdx.x; x < kGeRows * kGeJ; x += kThreads) {
      const int r = x / kGeJ, c = x % kGeJ;   // consecutive threads: consecutive columns
      const int i = i0 + r, j = j0 + c;
      er[r][c] = i < nb && j < nb ? P[(int64_t)i * nb + j] - T[(int64_t)i * nb + j] : 0.f;
      const int jr = j0 + r, ic = i0 + c;
      ec[r][c] = jr < nb && ic < nb ? P[(int64_t)jr * nb + ic] - T[(int64_t)jr * nb + ic] : 0.f;
    }
    const int jn = nb - j0 < kGeJ ? nb - j0 : kGeJ;
    for (int x = threadIdx.x; x < jn * rank; x += kThreads) {
      as[x] = A[(int64_t)j0 * rank + x];
      bs[x] = Bk[(int64_t)j0 * rank + x];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kGeOut; ++k) {
      const int o = threadIdx.x + k * kThreads;
      if (o < nout) {
        const int ii = o / rank, c = o % rank;
        for (int jj = 0; jj < jn; ++jj) {
          a[k] = fmaf(er[ii][jj], bs[jj * rank + c], a[k]);
          b[k] = fmaf(ec[jj][ii], as[jj * rank + c], b[k]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int k = 0; k < kGeOut; ++k) {
    const int o = threadIdx.x + k * kThreads;
    const int i = i0 + o / rank;
    if (o < nout && i < nb) {
      ga[bh * nb * rank + (int64_t)i * rank + o % rank] = a[k];
      gb[bh * nb * rank + (int64_t)i * rank + o % rank] = b[k];
    }
  }
}

// One CTA per (h, dd): thread (slice, c) sums column c over its slice of the
// B*nb rows; the slices are then added in a fixed tree.
__global__ void __launch_bounds__(kThreads)
gw_kernel(const float* __restrict__ qm, const float* __restrict__ km, const float* __restrict__ ga,
          const float* __restrict__ gb, int B, int H, int nb, int d, int rank, float lr, float* __restrict__ wq,
          float* __restrict__ wk, float* __restrict__ gwq, float* __restrict__ gwk) {
  __shared__ float part[2][kThreads];
  const int h = blockIdx.x, dd = blockIdx.y;
  const int nslices = kThreads / rank;
  const int c = threadIdx.x % rank, slice = threadIdx.x / rank;
  float q = 0.f, k = 0.f;
  if (slice < nslices) {
    for (int b = 0; b < B; ++b) {
      const int64_t bh = (int64_t)b * H + h;
      for (int i = slice; i < nb; i += nslices) {
        const int64_t row = bh * nb + i;
        q = fmaf(qm[row * d + dd], ga[row * rank + c], q);
        k = fmaf(km[row * d + dd], gb[row * rank + c], k);
      }
    }
  }
  part[0][threadIdx.x] = q;
  part[1][threadIdx.x] = k;
  __syncthreads();
  if (threadIdx.x < rank) {
    float sq = 0.f, sk = 0.f;
    for (int sl = 0; sl < nslices; ++sl) {
      sq += part[0][sl * rank + threadIdx.x];
      sk += part[1][sl * rank + threadIdx.x];
    }
    const float scale = (float)(2.0 / ((double)B * nb * nb));
    const float g1 = sq * scale, g2 = sk * scale;
    const int64_t w = ((int64_t)h * d + dd) * rank + threadIdx.x;
    if (gwq != nullptr) gwq[w] = g1;
    if (gwk != nullptr) gwk[w] = g2;
    if (lr != 0.f) {
      wq[w] -= lr * g1;
      wk[w] -= lr * g2;
    }
  }
}

constexpr int kLossChunks = 64;        // most partial sums per head
constexpr int kLossPerChunk = 4096;    // fewest elements per partial sum

__host__ __device__ inline int loss_chunks(int64_t n) {
  const int64_t c = (n + kLossPerChunk - 1) / kLossPerChunk;
  return c < 1 ? 1 : (c > kLossChunks ? kLossChunks : (int)c);
}

// grid (h, chunk): chunk c of head h's B*nb^2 squared errors, summed in fp64
// (each thread a fixed strided subset, then a fixed tree).
__global__ void __launch_bounds__(kThreads)
loss_part_kernel(const float* __restrict__ sp, const float* __restrict__ st, int B, int H, int nb,
                 double* __restrict__ part) {
  __shared__ double red[kThreads];
  const int h = blockIdx.x, chunk = blockIdx.y, nchunks = gridDim.y;
  const int64_t per_b = (int64_t)nb * nb, n = (int64_t)B * per_b;
  const int64_t len = (n + nchunks - 1) / nchunks;
  const int64_t e0 = (int64_t)chunk * len;
  const int64_t e1 = e0 + len < n ? e0 + len : n;
  double acc = 0.0;
  for (int64_t e = e0 + threadIdx.x; e < e1; e += kThreads) {
    const int64_t b = e / per_b;
    const int64_t at = ((int64_t)b * H + h) * per_b + (e - b * per_b);
    const double x = (double)sp[at] - (double)st[at];
    acc += x * x;
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = kThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) part[(int64_t)h * nchunks + chunk] = red[0];
}

// One thread per head: its partial sums in chunk order.
__global__ void loss_final_kernel(const double* __restrict__ part, int B, int H, int nb, int nchunks,
                                  float* __restrict__ loss) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= H) return;
  double s = 0.0;
  for (int c = 0; c < nchunks; ++c) s += part[(int64_t)h * nchunks + c];
  loss[h] = (float)(s / ((double)B * nb * nb));
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t predictor_ws(const Dims& s, int rank) {
  const size_t bh = (size_t)s.B * s.H;
  return align256(scores_from_means_ws(s, SPARSP_EST_LOWRANK, rank)) +
         2 * align256(bh * s.nb * s.nb * sizeof(float)) + 2 * align256(bh * s.nb * rank * sizeof(float)) +
         align256((size_t)s.H * kLossChunks * sizeof(double)) +
         align256(scores_from_means_ws(s, SPARSP_EST_MEAN, rank));
}

sparsp_status_t launch_predictor_fit(const Dims& s, int rank, const float* qm, const float* km, float* wq,
                                     float* wk, float lr, float* loss, float* gwq, float* gwk, void* ws,
                                     cudaStream_t st) {
  const size_t bh = (size_t)s.B * s.H;
  char* w = (char*)ws;
  // the low-rank pass leaves the projections qm Wq, km Wk at the start of its workspace
  float* proj = (float*)w;
  w += align256(scores_from_means_ws(s, SPARSP_EST_LOWRANK, rank));
  float* sp = (float*)w;
  w += align256(bh * s.nb * s.nb * sizeof(float));
  float* strue = (float*)w;
  w += align256(bh * s.nb * s.nb * sizeof(float));
  float* ga = (float*)w;
  w += align256(bh * s.nb * rank * sizeof(float));
  float* gb = (float*)w;
  w += align256(bh * s.nb * rank * sizeof(float));
  double* part = (double*)w;
  w += align256((size_t)s.H * kLossChunks * sizeof(double));
  void* ws_mean = w;
  sparsp_status_t r = launch_scores_from_means(s, SPARSP_EST_LOWRANK, qm, km, wq, wk, rank, sp, proj, st);
  if (r != SPARSP_OK) return r;
  r = launch_scores_from_means(s, SPARSP_EST_MEAN, qm, km, nullptr, nullptr, rank, strue, ws_mean, st);
  if (r != SPARSP_OK) return r;
  const float* pq = proj;
  const float* pk = proj + bh * s.nb * rank;
  ge_kernel<<<dim3((unsigned)bh, (unsigned)((s.nb + kGeRows - 1) / kGeRows)), kThreads, 0, st>>>(
      sp, strue, pq, pk, s.nb, rank, ga, gb);
  SPARSP_LAUNCH_CHECK();
  if (loss != nullptr) {
    const int nchunks = loss_chunks((int64_t)s.B * s.nb * s.nb);
    loss_part_kernel<<<dim3((unsigned)s.H, (unsigned)nchunks), kThreads, 0, st>>>(sp, strue, s.B, s.H, s.nb, part);
    SPARSP_LAUNCH_CHECK();
    loss_final_kernel<<<(s.H + 127) / 128, 128, 0, st>>>(part, s.B, s.H, s.nb, nchunks, loss);
    SPARSP_LAUNCH_CHECK();
  }
  gw_kernel<<<dim3((unsigned)s.H, (unsigned)s.d), kThreads, 0, st>>>(qm, km, ga, gb, s.B, s.H, s.nb, s.d, rank, lr,
                                                                    wq, wk, gwq, gwk);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace sparsp
