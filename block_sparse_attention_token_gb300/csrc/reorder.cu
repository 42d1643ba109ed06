// Step 1: video-aware block organisation - a permutation copy between the
// raster layout [B,N,H,d] and the tile-ordered layout [B,H,N,d].
//
// One CTA per (b, h, tile j) copies the tile's Bt rows of d elements with
// 16-byte vectors. Each thread issues all of its loads before its stores so
// that several 16-byte requests are in flight; data is touched once, so the
// loads and stores use the streaming cache policy.
#include "common.cuh"

namespace sparsp {
namespace {

constexpr int kThreads = 256;

template <int VEC_PER_ROW, int BT>
__global__ void __launch_bounds__(kThreads)
reorder_kernel(const uint4* __restrict__ in, uint4* __restrict__ out, int H, int64_t N, int Y,
               int X, int tb, int tc, int ta, int nY, int nX, int inverse) {
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
#pragma unroll
  for (int u = 0; u < kPer; ++u)
    if (dst_off[u] >= 0) __stcs(out + dst_off[u], buf[u]);
}

template <int VEC, int BT>
void go(const Dims& s, const void* in, void* out, bool inverse, cudaStream_t st) {
  dim3 grid(s.nb, s.H, s.B);
  reorder_kernel<VEC, BT><<<grid, kThreads, 0, st>>>(
      (const uint4*)in, (uint4*)out, s.H, s.N, s.Y, s.X, s.tb, s.tc, s.ta, s.nY, s.nX,
      inverse ? 1 : 0);
}

}  // namespace

sparsp_status_t launch_reorder(const Dims& s, const void* in, void* out, bool inverse,
                               cudaStream_t st) {
  const int row_bytes = s.d * s.elem;  // 128, 256 or 512
  const int vec = row_bytes / 16;
  if (s.Bt == 64) {
    if (vec == 8) go<8, 64>(s, in, out, inverse, st);
    else if (vec == 16) go<16, 64>(s, in, out, inverse, st);
    else go<32, 64>(s, in, out, inverse, st);
  } else {
    if (vec == 8) go<8, 128>(s, in, out, inverse, st);
    else if (vec == 16) go<16, 128>(s, in, out, inverse, st);
    else go<32, 128>(s, in, out, inverse, st);
  }
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace sparsp
