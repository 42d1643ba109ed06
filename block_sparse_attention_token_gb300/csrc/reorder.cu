// Step 1: video-aware block organisation - a permutation copy between the
// raster layout [B,N,H,d] and the tile-ordered layout [B,H,N,d]; optionally
// fused with the block pooling of step 2 (the tile means come out of the same
// pass, so the scores need no second read of Q and K).
//
// One CTA per (b, h, tile j) copies the tile's Bt rows of d elements with
// 16-byte vectors. Each thread issues all of its loads before its stores so
// that several 16-byte requests are in flight; data is touched once, so the
// loads and stores use the streaming cache policy.
#include "common.cuh"

namespace sparsp {
namespace {

constexpr int kThreads = 256;

// POOL (forward direction only): the same pass also writes the tile's fp32
// column means to `means` [B, H, nb, d]. Thread t always handles vector column
// t % VEC_PER_ROW; its tokens are summed in order, then the thread groups in
// group order: a fixed summation order.
template <int VEC_PER_ROW, int BT, bool POOL>
__global__ void __launch_bounds__(kThreads)
reorder_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, int H, int64_t N, int Y,
               int X, int tb, int tc, int ta, int nY, int nX, int inverse, int bf16,
               float* __restrict__ means) {
  const int j = blockIdx.x;      // tile
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int bx = j % nX;
  const int by = (j / nX) % nY;
  const int bt = j / (nX * nY);
  constexpr int kVecs = BT * VEC_PER_ROW;
  constexpr int kPer = (kVecs + kThreads - 1) / kThreads;
  uint4 buf[kPer];
  int64_t dst_off[kPer];
  const int tbc = tb * tc;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int idx = threadIdx.x + u * kThreads;
    dst_off[u] = -1;
    if (idx < kVecs) {
      const int o = idx / VEC_PER_ROW;      // token within tile
      const int vcol = idx % VEC_PER_ROW;
      const int it = o / tbc;
      const int rem = o - it * tbc;
      const int iy = rem / tc;
      const int ix = rem - iy * tc;
      const int64_t t = (int64_t)bt * ta + it;
      const int64_t y = (int64_t)by * tb + iy;
      const int64_t x = (int64_t)bx * tc + ix;
      const int64_t n = (t * Y + y) * X + x;                            // raster token
      const int64_t raster = (((int64_t)b * N + n) * H + h) * VEC_PER_ROW + vcol;
      const int64_t blocked = (((int64_t)b * H + h) * N + (int64_t)j * BT + o) * VEC_PER_ROW + vcol;
      const int64_t src = inverse ? blocked : raster;
      dst_off[u] = inverse ? raster : blocked;
      buf[u] = __ldcs(in + src);
    }
  }
  if (out != nullptr)   // null: the tile means alone (a pooling read of raster input)
#pragma unroll
    for (int u = 0; u < kPer; ++u)
      if (dst_off[u] >= 0) __stcs(out + dst_off[u], buf[u]);
  if (POOL) {
    __shared__ float part[kThreads][9];
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      if (dst_off[u] < 0) continue;
      if (bf16) {
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&buf[u]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h2[e]);
          acc[2 * e] += f.x;
          acc[2 * e + 1] += f.y;
        }
      } else {
        const float* f = reinterpret_cast<const float*>(&buf[u]);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] += f[e];
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) part[threadIdx.x][e] = acc[e];
    __syncthreads();
    const int epv = bf16 ? 8 : 4;                 // elements per 16-byte vector
    const int d = VEC_PER_ROW * epv;
    constexpr int kGroups = kThreads / VEC_PER_ROW;
    if (threadIdx.x < d) {
      const int c = threadIdx.x, vc = c / epv, e = c % epv;
      float sum = 0.f;
      for (int g2 = 0; g2 < kGroups; ++g2) sum += part[g2 * VEC_PER_ROW + vc][e];
      const int64_t nb = N / BT;
      means[(((int64_t)b * H + h) * nb + j) * d + c] = sum * (1.0f / (float)BT);
    }
  }
}

template <int VEC, int BT>
void go(const Dims& s, const void* in, void* out, bool inverse, float* means, cudaStream_t st) {
  dim3 grid(s.nb, s.H, s.B);
  const int bf16 = s.dtype == SPARSP_BF16;
  if (means != nullptr)
    reorder_kernel<VEC, BT, true><<<grid, kThreads, 0, st>>>(
        (const uint4*)in, (uint4*)out, s.H, s.N, s.Y, s.X, s.tb, s.tc, s.ta, s.nY, s.nX, 0, bf16, means);
  else
    reorder_kernel<VEC, BT, false><<<grid, kThreads, 0, st>>>(
        (const uint4*)in, (uint4*)out, s.H, s.N, s.Y, s.X, s.tb, s.tc, s.ta, s.nY, s.nX,
        inverse ? 1 : 0, bf16, nullptr);
}

}  // namespace

sparsp_status_t launch_reorder(const Dims& s, const void* in, void* out, bool inverse,
                               cudaStream_t st, float* means) {
  const int row_bytes = s.d * s.elem;  // 128, 256 or 512
  const int vec = row_bytes / 16;
  if (s.Bt == 64) {
    if (vec == 8) go<8, 64>(s, in, out, inverse, means, st);
    else if (vec == 16) go<16, 64>(s, in, out, inverse, means, st);
    else go<32, 64>(s, in, out, inverse, means, st);
  } else {
    if (vec == 8) go<8, 128>(s, in, out, inverse, means, st);
    else if (vec == 16) go<16, 128>(s, in, out, inverse, means, st);
    else go<32, 128>(s, in, out, inverse, means, st);
  }
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace sparsp
