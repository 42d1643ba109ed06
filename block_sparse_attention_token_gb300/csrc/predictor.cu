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
//  2. ge_kernel   - grid (b*H + h, chunk of 256 outputs): GA = E (km Wk),
//     GB = E^T (qm Wq), one output element per thread;
//  3. loss_kernel - one CTA per head: the loss (fp64 partials, a fixed tree);
//  4. gw_kernel   - grid (h, dd): the weight gradients (row slices summed in a
//     fixed tree) and, when lr != 0, the step W -= lr dL/dW in place (the
//     projections were taken before it).
// Every sum has a fixed order, so results are bitwise reproducible.
#include "common.cuh"

namespace sparsp {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
ge_kernel(const float* __restrict__ sp, const float* __restrict__ st, const float* __restrict__ pq,
          const float* __restrict__ pk, int nb, int rank, float* __restrict__ ga, float* __restrict__ gb) {
  const int64_t bh = blockIdx.x;
  const int idx = blockIdx.y * kThreads + threadIdx.x;
  if (idx >= nb * rank) return;
  const float* P = sp + bh * nb * nb;
  const float* T = st + bh * nb * nb;
  const float* A = pq + bh * nb * rank;
  const float* Bk = pk + bh * nb * rank;
  float* GA = ga + bh * nb * rank;
  float* GB = gb + bh * nb * rank;
  const int i = idx / rank, c = idx % rank;
  float a = 0.f, bsum = 0.f;
  for (int j = 0; j < nb; ++j) {
    a = fmaf(P[(int64_t)i * nb + j] - T[(int64_t)i * nb + j], Bk[(int64_t)j * rank + c], a);
    bsum = fmaf(P[(int64_t)j * nb + i] - T[(int64_t)j * nb + i], A[(int64_t)j * rank + c], bsum);
  }
  GA[idx] = a;
  GB[idx] = bsum;
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

// One CTA per head: every thread sums a fixed strided subset in fp64, then a
// fixed tree.
__global__ void __launch_bounds__(kThreads)
loss_kernel(const float* __restrict__ sp, const float* __restrict__ st, int B, int H, int nb,
            float* __restrict__ loss) {
  __shared__ double red[kThreads];
  const int h = blockIdx.x;
  double acc = 0.0;
  for (int b = 0; b < B; ++b) {
    const int64_t base = ((int64_t)b * H + h) * nb * nb;
    for (int64_t e = threadIdx.x; e < (int64_t)nb * nb; e += kThreads) {
      const double x = (double)sp[base + e] - (double)st[base + e];
      acc += x * x;
    }
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = kThreads / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) loss[h] = (float)(red[0] / ((double)B * nb * nb));
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t predictor_ws(const Dims& s, int rank) {
  const size_t bh = (size_t)s.B * s.H;
  return align256(scores_from_means_ws(s, SPARSP_EST_LOWRANK, rank)) +
         2 * align256(bh * s.nb * s.nb * sizeof(float)) + 2 * align256(bh * s.nb * rank * sizeof(float)) +
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
  void* ws_mean = w;
  sparsp_status_t r = launch_scores_from_means(s, SPARSP_EST_LOWRANK, qm, km, wq, wk, rank, sp, proj, st);
  if (r != SPARSP_OK) return r;
  r = launch_scores_from_means(s, SPARSP_EST_MEAN, qm, km, nullptr, nullptr, rank, strue, ws_mean, st);
  if (r != SPARSP_OK) return r;
  const float* pq = proj;
  const float* pk = proj + bh * s.nb * rank;
  ge_kernel<<<dim3((unsigned)bh, (unsigned)((s.nb * rank + kThreads - 1) / kThreads)), kThreads, 0, st>>>(
      sp, strue, pq, pk, s.nb, rank, ga, gb);
  SPARSP_LAUNCH_CHECK();
  if (loss != nullptr) {
    loss_kernel<<<s.H, kThreads, 0, st>>>(sp, strue, s.B, s.H, s.nb, loss);
    SPARSP_LAUNCH_CHECK();
  }
  gw_kernel<<<dim3((unsigned)s.H, (unsigned)s.d), kThreads, 0, st>>>(qm, km, ga, gb, s.B, s.H, s.nb, s.d, rank, lr,
                                                                    wq, wk, gwq, gwk);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace sparsp
