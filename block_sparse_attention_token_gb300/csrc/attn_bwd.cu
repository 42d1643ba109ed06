// Step 5b: block-sparse attention backward (bf16 in, fp32 accumulate), with
// the selection held fixed.
//
//  rowdot_kernel - D = rowsum(dO * O) per query token (fp32; O read from block
//                  or raster order), and optionally LSE * log2(e) for the
//                  tcgen05 backward.
//  dq_kernel     - one work item per query block (CSR row): for each selected
//                  key block, recompute P = exp2(S*log2e*scale - LSE*log2e),
//                  dP = dO V^T, dS = P (dP - D), dQ += dS K. dQ stays in
//                  registers for the whole row.
//  dkdv_kernel   - one work item per key block (transposed CSR column): for
//                  each query block that selected it, recompute P^T and dS^T
//                  from K Q^T and V dO^T, then dV += P^T dO, dK += dS^T Q.
// Both are persistent, pull longest-first items through an atomic counter and
// run on mma.sync m16n8k16; each warp owns 16 rows of the item's block and
// walks the other side in halves of 64 tokens to bound register use. The sum
// order is fixed, so results are bitwise reproducible.
#include "mma_helpers.cuh"

namespace sparsp {
namespace {

using namespace mma;

constexpr float kLog2e = 1.4426950408889634f;

__global__ void __launch_bounds__(256)
rowdot_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
              int64_t rows, int d, float* __restrict__ delta, const float* __restrict__ lse,
              float* __restrict__ lse2, int Bt, int o_raster, RasterMap rm) {
  // 8 threads per row (d <= 128: 16 bf16 each) -> 32 rows per CTA
  const int64_t row = (int64_t)blockIdx.x * 32 + (threadIdx.x >> 3);
  const int sub = threadIdx.x & 7;
  // the block-order row's O row: the same, or its raster row (the index
  // arithmetic once per row, by the row's first thread)
  int64_t orow = row;
  if (o_raster) {
    int64_t r = 0;
    if (sub == 0 && row < rows) {
      const int64_t rem = row % rm.N;
      r = rm.row(row / rm.N, (int)(rem / Bt), (int)(rem % Bt));
    }
    orow = __shfl_sync(0xffffffffu, r, (threadIdx.x & 31) & ~7);
  }
  float acc = 0.f;
  if (row < rows) {
    const int per = d / 8;   // elements per thread: 8 or 16
    for (int c = sub * per; c < (sub + 1) * per; c += 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(o + orow * d + c);
      const uint4 b = *reinterpret_cast<const uint4*>(dout + row * d + c);
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(pa[e]), y = __bfloat1622float2(pb[e]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
  }
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sub == 0) {
    delta[row] = acc;
    if (lse2 != nullptr) lse2[row] = lse[row] * kLog2e;   // -inf stays -inf
  }
}

template <int BT, int D>
struct BwdCfg {
  static constexpr int kWarps = BT / 16;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kTileBytes = BT * D * 2;
  static constexpr int kHalf = 64;                 // other-side tokens per step
  static constexpr int kSmem = kTileBytes * 6 + 2 * 2 * BT * 4;
};

// Pull the next item; returns false when the list is exhausted.
__device__ __forceinline__ bool next_item(int32_t* counter, int64_t n_items, int32_t* item_s,
                                          const int32_t* items, int64_t* item) {
  if (threadIdx.x == 0) *item_s = atomicAdd(counter, 1);
  __syncthreads();
  const int32_t slot = *item_s;
  __syncthreads();
  if (slot >= n_items) return false;
  *item = items[slot];
  return true;
}

// Validates list [a, b) of block indices; returns length or -1.
__device__ __forceinline__ int checked_list(const int32_t* ptr, const int32_t* idx, int64_t r,
                                            int nb, int32_t* d_status, int threads) {
  const int32_t a = ptr[r], b = ptr[r + 1];
  int bad = (b < a || b - a > nb) ? 1 : 0;
  if (!bad)
    for (int32_t e = a + threadIdx.x; e < b; e += threads) {
      const int32_t j = idx[e];
      if (j < 0 || j >= nb) bad = 1;
    }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) report(d_status, SPARSP_ERR_DATA);
    return -1;
  }
  return b - a;
}

template <int BT, int D>
__global__ void __launch_bounds__(BwdCfg<BT, D>::kThreads, 1)
dq_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
          const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ dout,
          const float* __restrict__ lse, const float* __restrict__ delta,
          const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col_idx, int64_t N,
          int nb, int64_t n_items, float scale, __nv_bfloat16* __restrict__ dq,
          const int32_t* __restrict__ items, int32_t* __restrict__ counter, uint64_t* prof,
          int32_t* d_status) {
  using C = BwdCfg<BT, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int32_t item_s;
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sdO = sQ + C::kTileBytes;
  const uint32_t sK0 = sQ + 2 * C::kTileBytes;
  const uint32_t sV0 = sQ + 4 * C::kTileBytes;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const float sl2 = scale * kLog2e;
  const uint64_t t_start = globaltimer_ns();
  int64_t item;
  while (next_item(counter, n_items, &item_s, items, &item)) {
    const int64_t bh = item / nb;
    const int i = (int)(item % nb);
    const int len = checked_list(row_ptr, col_idx, item, nb, d_status, C::kThreads);
    if (len < 0) continue;
    const int32_t ea = row_ptr[item];
    const int64_t qrow0 = bh * N + (int64_t)i * BT;
    const int r0 = warp * 16 + g;
    if (len == 0) {
      for (int x = threadIdx.x; x < BT * D / 8; x += C::kThreads)
        reinterpret_cast<uint4*>(dq + qrow0 * D)[x] = make_uint4(0, 0, 0, 0);
      continue;
    }
    load_tile<BT, D, C::kThreads>(sQ, q + qrow0 * D);
    load_tile<BT, D, C::kThreads>(sdO, dout + qrow0 * D);
    {
      const int64_t key0 = bh * N + (int64_t)col_idx[ea] * BT;
      load_tile<BT, D, C::kThreads>(sK0, k + key0 * D);
      load_tile<BT, D, C::kThreads>(sV0, v + key0 * D);
    }
    cp_async_commit();
    const float lse2[2] = {lse[qrow0 + r0] * kLog2e, lse[qrow0 + r0 + 8] * kLog2e};
    const float dlt[2] = {delta[qrow0 + r0], delta[qrow0 + r0 + 8]};
    float acc[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
      for (int x = 0; x < 4; ++x) acc[n][x] = 0.f;
    for (int e = 0; e < len; ++e) {
      const int buf = e & 1;
      if (e + 1 < len) {
        const int64_t key0 = bh * N + (int64_t)col_idx[ea + e + 1] * BT;
        load_tile<BT, D, C::kThreads>(sK0 + (buf ^ 1) * C::kTileBytes, k + key0 * D);
        load_tile<BT, D, C::kThreads>(sV0 + (buf ^ 1) * C::kTileBytes, v + key0 * D);
        cp_async_commit();
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      const uint32_t sK = sK0 + buf * C::kTileBytes;
      const uint32_t sV = sV0 + buf * C::kTileBytes;
#pragma unroll 1
      for (int h0 = 0; h0 < BT; h0 += C::kHalf) {
        float s[C::kHalf / 8][4], dp[C::kHalf / 8][4];
#pragma unroll
        for (int n = 0; n < C::kHalf / 8; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x) s[n][x] = dp[n][x] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t a[4], ad[4];
          load_a<D>(sQ, warp * 16, kk * 16, a);
          load_a<D>(sdO, warp * 16, kk * 16, ad);
#pragma unroll
          for (int n2 = 0; n2 < C::kHalf / 16; ++n2) {
            uint32_t b[4], bv[4];
            load_b_nk<D>(sK, h0 + n2 * 16, kk * 16, b);
            load_b_nk<D>(sV, h0 + n2 * 16, kk * 16, bv);
            mma16816(s[2 * n2], a, b[0], b[1]);
            mma16816(s[2 * n2 + 1], a, b[2], b[3]);
            mma16816(dp[2 * n2], ad, bv[0], bv[1]);
            mma16816(dp[2 * n2 + 1], ad, bv[2], bv[3]);
          }
        }
        uint32_t ds[C::kHalf / 16][4];
#pragma unroll
        for (int n = 0; n < C::kHalf / 8; ++n) {
          const float p0 = ex2(s[n][0] * sl2 - lse2[0]), p1 = ex2(s[n][1] * sl2 - lse2[0]);
          const float p2 = ex2(s[n][2] * sl2 - lse2[1]), p3 = ex2(s[n][3] * sl2 - lse2[1]);
          ds[n >> 1][(n & 1) * 2 + 0] = pack_bf16(p0 * (dp[n][0] - dlt[0]), p1 * (dp[n][1] - dlt[0]));
          ds[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2 * (dp[n][2] - dlt[1]), p3 * (dp[n][3] - dlt[1]));
        }
        // dQ += dS K  (k = keys of this half, n = d)
#pragma unroll
        for (int kk = 0; kk < C::kHalf / 16; ++kk) {
#pragma unroll
          for (int n2 = 0; n2 < D / 16; ++n2) {
            uint32_t b[4];
            load_b_kn<D>(sK, h0 + kk * 16, n2 * 16, b);
            mma16816(acc[2 * n2], ds[kk], b[0], b[1]);
            mma16816(acc[2 * n2 + 1], ds[kk], b[2], b[3]);
          }
        }
      }
      __syncthreads();
    }
    // epilogue: scale, stage in the Q slot, coalesced store
    uint8_t* st = smem;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int col = n * 8 + tq * 2;
      *reinterpret_cast<uint32_t*>(st + swz<D>(r0, col >> 3) + (col & 7) * 2) =
          pack_bf16(acc[n][0] * scale, acc[n][1] * scale);
      *reinterpret_cast<uint32_t*>(st + swz<D>(r0 + 8, col >> 3) + (col & 7) * 2) =
          pack_bf16(acc[n][2] * scale, acc[n][3] * scale);
    }
    __syncthreads();
    for (int x = threadIdx.x; x < BT * D / 8; x += C::kThreads) {
      const int r = x / (D / 8), c = x % (D / 8);
      reinterpret_cast<uint4*>(dq + (qrow0 + r) * D)[c] =
          *reinterpret_cast<const uint4*>(st + swz<D>(r, c));
    }
    __syncthreads();
  }
  if (prof != nullptr && threadIdx.x == 0)
    atomicAdd((unsigned long long*)&prof[smid() % SPARSP_PROF_SLOTS],
              (unsigned long long)(globaltimer_ns() - t_start));
}

template <int BT, int D>
__global__ void __launch_bounds__(BwdCfg<BT, D>::kThreads, 1)
dkdv_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
            const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ dout,
            const float* __restrict__ lse, const float* __restrict__ delta,
            const int32_t* __restrict__ col_ptr, const int32_t* __restrict__ row_idx, int64_t N,
            int nb, int64_t n_items, float scale, __nv_bfloat16* __restrict__ dk,
            __nv_bfloat16* __restrict__ dv, const int32_t* __restrict__ items,
            int32_t* __restrict__ counter, uint64_t* prof, int32_t* d_status) {
  using C = BwdCfg<BT, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int32_t item_s;
  const uint32_t sK = smem_u32(smem);
  const uint32_t sV = sK + C::kTileBytes;
  const uint32_t sQ0 = sK + 2 * C::kTileBytes;
  const uint32_t sdO0 = sK + 4 * C::kTileBytes;
  float* sL = reinterpret_cast<float*>(smem + 6 * C::kTileBytes);   // [2][BT] lse*log2e
  float* sD = sL + 2 * BT;                                           // [2][BT] delta
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const float sl2 = scale * kLog2e;
  const uint64_t t_start = globaltimer_ns();
  int64_t item;
  while (next_item(counter, n_items, &item_s, items, &item)) {
    const int64_t bh = item / nb;
    const int j = (int)(item % nb);
    const int len = checked_list(col_ptr, row_idx, item, nb, d_status, C::kThreads);
    if (len < 0) continue;
    const int32_t ea = col_ptr[item];
    const int64_t krow0 = bh * N + (int64_t)j * BT;
    const int r0 = warp * 16 + g;      // key rows of this thread
    if (len == 0) {
      for (int x = threadIdx.x; x < BT * D / 8; x += C::kThreads) {
        reinterpret_cast<uint4*>(dk + krow0 * D)[x] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(dv + krow0 * D)[x] = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    load_tile<BT, D, C::kThreads>(sK, k + krow0 * D);
    load_tile<BT, D, C::kThreads>(sV, v + krow0 * D);
    {
      const int64_t qr = bh * N + (int64_t)row_idx[ea] * BT;
      load_tile<BT, D, C::kThreads>(sQ0, q + qr * D);
      load_tile<BT, D, C::kThreads>(sdO0, dout + qr * D);
      for (int x = threadIdx.x; x < BT; x += C::kThreads) {
        sL[x] = lse[qr + x] * kLog2e;
        sD[x] = delta[qr + x];
      }
    }
    cp_async_commit();
    float adk[D / 8][4], adv[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
      for (int x = 0; x < 4; ++x) adk[n][x] = adv[n][x] = 0.f;
    for (int e = 0; e < len; ++e) {
      const int buf = e & 1;
      if (e + 1 < len) {
        const int64_t qr = bh * N + (int64_t)row_idx[ea + e + 1] * BT;
        load_tile<BT, D, C::kThreads>(sQ0 + (buf ^ 1) * C::kTileBytes, q + qr * D);
        load_tile<BT, D, C::kThreads>(sdO0 + (buf ^ 1) * C::kTileBytes, dout + qr * D);
        for (int x = threadIdx.x; x < BT; x += C::kThreads) {
          sL[(buf ^ 1) * BT + x] = lse[qr + x] * kLog2e;
          sD[(buf ^ 1) * BT + x] = delta[qr + x];
        }
        cp_async_commit();
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      const uint32_t sQ = sQ0 + buf * C::kTileBytes;
      const uint32_t sdO = sdO0 + buf * C::kTileBytes;
      const float* L = sL + buf * BT;
      const float* Dl = sD + buf * BT;
#pragma unroll 1
      for (int h0 = 0; h0 < BT; h0 += C::kHalf) {
        float s[C::kHalf / 8][4], dp[C::kHalf / 8][4];
#pragma unroll
        for (int n = 0; n < C::kHalf / 8; ++n)
#pragma unroll
          for (int x = 0; x < 4; ++x) s[n][x] = dp[n][x] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t a[4], av[4];
          load_a<D>(sK, warp * 16, kk * 16, a);
          load_a<D>(sV, warp * 16, kk * 16, av);
#pragma unroll
          for (int n2 = 0; n2 < C::kHalf / 16; ++n2) {
            uint32_t b[4], bd[4];
            load_b_nk<D>(sQ, h0 + n2 * 16, kk * 16, b);
            load_b_nk<D>(sdO, h0 + n2 * 16, kk * 16, bd);
            mma16816(s[2 * n2], a, b[0], b[1]);
            mma16816(s[2 * n2 + 1], a, b[2], b[3]);
            mma16816(dp[2 * n2], av, bd[0], bd[1]);
            mma16816(dp[2 * n2 + 1], av, bd[2], bd[3]);
          }
        }
        uint32_t pt[C::kHalf / 16][4], dst[C::kHalf / 16][4];
#pragma unroll
        for (int n = 0; n < C::kHalf / 8; ++n) {
          const int qc = h0 + n * 8 + tq * 2;       // query columns qc, qc+1
          const float l0 = L[qc], l1 = L[qc + 1];
          const float d0 = Dl[qc], d1 = Dl[qc + 1];
          const float p0 = ex2(s[n][0] * sl2 - l0), p1 = ex2(s[n][1] * sl2 - l1);
          const float p2 = ex2(s[n][2] * sl2 - l0), p3 = ex2(s[n][3] * sl2 - l1);
          pt[n >> 1][(n & 1) * 2 + 0] = pack_bf16(p0, p1);
          pt[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2, p3);
          dst[n >> 1][(n & 1) * 2 + 0] = pack_bf16(p0 * (dp[n][0] - d0), p1 * (dp[n][1] - d1));
          dst[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2 * (dp[n][2] - d0), p3 * (dp[n][3] - d1));
        }
        // dV += P^T dO, dK += dS^T Q  (k = queries of this half, n = d)
#pragma unroll
        for (int kk = 0; kk < C::kHalf / 16; ++kk) {
#pragma unroll
          for (int n2 = 0; n2 < D / 16; ++n2) {
            uint32_t bd[4], bq[4];
            load_b_kn<D>(sdO, h0 + kk * 16, n2 * 16, bd);
            load_b_kn<D>(sQ, h0 + kk * 16, n2 * 16, bq);
            mma16816(adv[2 * n2], pt[kk], bd[0], bd[1]);
            mma16816(adv[2 * n2 + 1], pt[kk], bd[2], bd[3]);
            mma16816(adk[2 * n2], dst[kk], bq[0], bq[1]);
            mma16816(adk[2 * n2 + 1], dst[kk], bq[2], bq[3]);
          }
        }
      }
      __syncthreads();
    }
    // epilogue: dK (scaled) staged in the Q0 slot, dV in the Q1 slot
    uint8_t* stk = smem + 2 * C::kTileBytes;
    uint8_t* stv = smem + 3 * C::kTileBytes;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int col = n * 8 + tq * 2;
      const uint32_t o0 = swz<D>(r0, col >> 3) + (col & 7) * 2;
      const uint32_t o1 = swz<D>(r0 + 8, col >> 3) + (col & 7) * 2;
      *reinterpret_cast<uint32_t*>(stk + o0) = pack_bf16(adk[n][0] * scale, adk[n][1] * scale);
      *reinterpret_cast<uint32_t*>(stk + o1) = pack_bf16(adk[n][2] * scale, adk[n][3] * scale);
      *reinterpret_cast<uint32_t*>(stv + o0) = pack_bf16(adv[n][0], adv[n][1]);
      *reinterpret_cast<uint32_t*>(stv + o1) = pack_bf16(adv[n][2], adv[n][3]);
    }
    __syncthreads();
    for (int x = threadIdx.x; x < BT * D / 8; x += C::kThreads) {
      const int r = x / (D / 8), c = x % (D / 8);
      reinterpret_cast<uint4*>(dk + (krow0 + r) * D)[c] =
          *reinterpret_cast<const uint4*>(stk + swz<D>(r, c));
      reinterpret_cast<uint4*>(dv + (krow0 + r) * D)[c] =
          *reinterpret_cast<const uint4*>(stv + swz<D>(r, c));
    }
    __syncthreads();
  }
  if (prof != nullptr && threadIdx.x == 0)
    atomicAdd((unsigned long long*)&prof[smid() % SPARSP_PROF_SLOTS],
              (unsigned long long)(globaltimer_ns() - t_start));
}

template <typename K>
sparsp_status_t persistent_grid(const Dims& s, K kern, int threads, int smem, int64_t n_items, int64_t* grid) {
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return SPARSP_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return SPARSP_ERR_CUDA;
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
  if (per_sm < 1) per_sm = 1;
  *grid = cap_grid(s, (int64_t)sms * per_sm, n_items);
  return SPARSP_OK;
}

}  // namespace

sparsp_status_t launch_bwd_rowdot(const Dims& s, const __nv_bfloat16* o, const __nv_bfloat16* dout,
                                  float* delta, const float* lse, float* lse2, bool o_raster,
                                  cudaStream_t st) {
  const int64_t rows = (int64_t)s.B * s.H * s.N;
  rowdot_kernel<<<(unsigned)((rows + 31) / 32), 256, 0, st>>>(o, dout, rows, s.d, delta, lse, lse2, s.Bt,
                                                               o_raster ? 1 : 0, raster_map(s));
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

sparsp_status_t launch_attn_bwd_dq(const Dims& s, const __nv_bfloat16* q, const __nv_bfloat16* k,
                                   const __nv_bfloat16* v, const __nv_bfloat16* dout,
                                   const float* lse, const float* delta, const int32_t* row_ptr,
                                   const int32_t* col_idx, float scale, __nv_bfloat16* dq,
                                   const int32_t* items, int32_t* counter, uint64_t* prof,
                                   int32_t* d_status, cudaStream_t st) {
#define GO(BT, D)                                                                                 \
  do {                                                                                           \
    using C = BwdCfg<BT, D>;                                                                     \
    int64_t grid;                                                                                \
    auto kern = dq_kernel<BT, D>;                                                                \
    sparsp_status_t r = persistent_grid(s, kern, C::kThreads, C::kSmem, s.rows(), &grid);           \
    if (r != SPARSP_OK) return r;                                                                \
    kern<<<(unsigned)grid, C::kThreads, C::kSmem, st>>>(q, k, v, dout, lse, delta, row_ptr,     \
                                                        col_idx, s.N, s.nb, s.rows(), scale, dq, \
                                                        items, counter, prof, d_status);         \
  } while (0)
  if (s.Bt == 64) {
    if (s.d == 64) GO(64, 64); else GO(64, 128);
  } else {
    if (s.d == 64) GO(128, 64); else GO(128, 128);
  }
#undef GO
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

sparsp_status_t launch_attn_bwd_dkdv(const Dims& s, const __nv_bfloat16* q,
                                     const __nv_bfloat16* k, const __nv_bfloat16* v,
                                     const __nv_bfloat16* dout, const float* lse,
                                     const float* delta, const int32_t* col_ptr,
                                     const int32_t* row_idx, float scale, __nv_bfloat16* dk,
                                     __nv_bfloat16* dv, const int32_t* items, int32_t* counter,
                                     uint64_t* prof, int32_t* d_status, cudaStream_t st) {
#define GO(BT, D)                                                                                 \
  do {                                                                                           \
    using C = BwdCfg<BT, D>;                                                                     \
    int64_t grid;                                                                                \
    auto kern = dkdv_kernel<BT, D>;                                                              \
    sparsp_status_t r = persistent_grid(s, kern, C::kThreads, C::kSmem, s.rows(), &grid);           \
    if (r != SPARSP_OK) return r;                                                                \
    kern<<<(unsigned)grid, C::kThreads, C::kSmem, st>>>(q, k, v, dout, lse, delta, col_ptr,     \
                                                        row_idx, s.N, s.nb, s.rows(), scale, dk, \
                                                        dv, items, counter, prof, d_status);     \
  } while (0)
  if (s.Bt == 64) {
    if (s.d == 64) GO(64, 64); else GO(64, 128);
  } else {
    if (s.d == 64) GO(128, 64); else GO(128, 128);
  }
#undef GO
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace sparsp
