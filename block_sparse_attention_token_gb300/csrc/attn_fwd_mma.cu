// Step 5a, bf16, portable tensor-core path (mma.sync m16n8k16): block-sparse
// flash-attention forward over the CSR for any supported (Bt, d).
//
// Persistent CTAs of Bt/16 warps pull (b, h, query block) items from the
// longest-first list; warp w owns query rows 16w..16w+15 of the block. The
// selected K/V tiles are double-buffered in swizzled shared memory with
// cp.async; S = Q K^T and O += P V run on mma.sync with fp32 accumulators in
// registers and an online softmax in base 2. O is staged through shared
// memory for 16-byte coalesced stores.
#include "mma_helpers.cuh"

namespace sparsp {
namespace {

using namespace mma;

template <int BT, int D>
struct FwdCfg {
  static constexpr int kWarps = BT / 16;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kTileBytes = BT * D * 2;
  static constexpr int kSmem = kTileBytes * 5;   // Q, K[2], V[2]
};

template <int BT, int D>
__global__ void __launch_bounds__(FwdCfg<BT, D>::kThreads, 1)
attn_fwd_mma_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v, const int32_t* __restrict__ row_ptr,
                    const int32_t* __restrict__ col_idx, int64_t N, int nb, int64_t n_items,
                    float scale_log2, __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                    const int32_t* __restrict__ items, int32_t* __restrict__ counter,
                    uint64_t* prof, int32_t* d_status) {
  using C = FwdCfg<BT, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int32_t item_s;
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + C::kTileBytes;
  const uint32_t sV0 = sQ + 3 * C::kTileBytes;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const uint64_t t_start = globaltimer_ns();

  for (;;) {
    if (threadIdx.x == 0) item_s = atomicAdd(counter, 1);
    __syncthreads();
    const int32_t slot = item_s;
    __syncthreads();
    if (slot >= n_items) break;
    const int64_t item = items[slot];
    const int64_t bh = item / nb;
    const int i = (int)(item % nb);
    // validate the CSR row
    const int32_t ea = row_ptr[item], eb = row_ptr[item + 1];
    int bad = (eb < ea || eb - ea > nb) ? 1 : 0;
    if (!bad)
      for (int32_t e = ea + threadIdx.x; e < eb; e += C::kThreads) {
        const int32_t j = col_idx[e];
        if (j < 0 || j >= nb) bad = 1;
      }
    if (__syncthreads_or(bad)) {
      if (threadIdx.x == 0) report(d_status, SPARSP_ERR_DATA);
      continue;
    }
    const int len = eb - ea;
    const int64_t qrow0 = bh * N + (int64_t)i * BT;
    if (len == 0) {
      for (int x = threadIdx.x; x < BT * D / 8; x += C::kThreads)
        reinterpret_cast<uint4*>(o + qrow0 * D)[x] = make_uint4(0, 0, 0, 0);
      for (int x = threadIdx.x; x < BT; x += C::kThreads) lse[qrow0 + x] = -INFINITY;
      continue;
    }
    load_tile<BT, D, C::kThreads>(sQ, q + qrow0 * D);
    {
      const int64_t key0 = bh * N + (int64_t)col_idx[ea] * BT;
      load_tile<BT, D, C::kThreads>(sK0, k + key0 * D);
      load_tile<BT, D, C::kThreads>(sV0, v + key0 * D);
    }
    cp_async_commit();

    float acc_o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
      for (int x = 0; x < 4; ++x) acc_o[n][x] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY};
    float l_r[2] = {0.f, 0.f};
    uint32_t qa[D / 16][4];

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
      if (e == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) load_a<D>(sQ, warp * 16, kk * 16, qa[kk]);
      }
      const uint32_t sK = sK0 + buf * C::kTileBytes;
      const uint32_t sV = sV0 + buf * C::kTileBytes;
      // S = Q K^T for this warp's 16 rows x BT keys
      float s[BT / 8][4];
#pragma unroll
      for (int n = 0; n < BT / 8; ++n)
#pragma unroll
        for (int x = 0; x < 4; ++x) s[n][x] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int n2 = 0; n2 < BT / 16; ++n2) {
          uint32_t b[4];
          load_b_nk<D>(sK, n2 * 16, kk * 16, b);
          mma16816(s[2 * n2], qa[kk], b[0], b[1]);
          mma16816(s[2 * n2 + 1], qa[kk], b[2], b[3]);
        }
      }
      // online softmax (rows g and g+8 of the warp's slab)
      float mx[2] = {m_r[0], m_r[1]};
#pragma unroll
      for (int n = 0; n < BT / 8; ++n) {
        s[n][0] *= scale_log2; s[n][1] *= scale_log2;
        s[n][2] *= scale_log2; s[n][3] *= scale_log2;
        mx[0] = fmaxf(mx[0], fmaxf(s[n][0], s[n][1]));
        mx[1] = fmaxf(mx[1], fmaxf(s[n][2], s[n][3]));
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      }
      float alpha[2], rs[2] = {0.f, 0.f};
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        alpha[r] = ex2(m_r[r] - mx[r]);
        m_r[r] = mx[r];
      }
      uint32_t pa[BT / 16][4];
#pragma unroll
      for (int n = 0; n < BT / 8; ++n) {
        const float p0 = ex2(s[n][0] - mx[0]), p1 = ex2(s[n][1] - mx[0]);
        const float p2 = ex2(s[n][2] - mx[1]), p3 = ex2(s[n][3] - mx[1]);
        rs[0] += p0 + p1;
        rs[1] += p2 + p3;
        pa[n >> 1][(n & 1) * 2 + 0] = pack_bf16(p0, p1);
        pa[n >> 1][(n & 1) * 2 + 1] = pack_bf16(p2, p3);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) l_r[r] = l_r[r] * alpha[r] + rs[r];
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        acc_o[n][0] *= alpha[0]; acc_o[n][1] *= alpha[0];
        acc_o[n][2] *= alpha[1]; acc_o[n][3] *= alpha[1];
      }
      // O += P V
#pragma unroll
      for (int kk = 0; kk < BT / 16; ++kk) {
#pragma unroll
        for (int n2 = 0; n2 < D / 16; ++n2) {
          uint32_t b[4];
          load_b_kn<D>(sV, kk * 16, n2 * 16, b);
          mma16816(acc_o[2 * n2], pa[kk], b[0], b[1]);
          mma16816(acc_o[2 * n2 + 1], pa[kk], b[2], b[3]);
        }
      }
      __syncthreads();
    }
    // epilogue: row sums across the quad, normalise, stage O in smem (Q slot)
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
      l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
    }
    const float inv0 = 1.f / l_r[0], inv1 = 1.f / l_r[1];
    uint8_t* sQp = smem;
    const int r0 = warp * 16 + g;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int col = n * 8 + tq * 2;
      const uint32_t w0 = pack_bf16(acc_o[n][0] * inv0, acc_o[n][1] * inv0);
      const uint32_t w1 = pack_bf16(acc_o[n][2] * inv1, acc_o[n][3] * inv1);
      *reinterpret_cast<uint32_t*>(sQp + swz<D>(r0, col >> 3) + (col & 7) * 2) = w0;
      *reinterpret_cast<uint32_t*>(sQp + swz<D>(r0 + 8, col >> 3) + (col & 7) * 2) = w1;
    }
    if (tq == 0) {
      lse[qrow0 + r0] = (m_r[0] + log2f(l_r[0])) * 0.69314718055994531f;
      lse[qrow0 + r0 + 8] = (m_r[1] + log2f(l_r[1])) * 0.69314718055994531f;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < BT * D / 8; x += C::kThreads) {
      const int r = x / (D / 8), c = x % (D / 8);
      const uint4 val = *reinterpret_cast<const uint4*>(sQp + swz<D>(r, c));
      reinterpret_cast<uint4*>(o + (qrow0 + r) * D)[c] = val;
    }
    __syncthreads();
  }
  if (prof != nullptr && threadIdx.x == 0)
    atomicAdd((unsigned long long*)&prof[smid() % SPARSP_PROF_SLOTS],
              (unsigned long long)(globaltimer_ns() - t_start));
}

template <int BT, int D>
sparsp_status_t go(const Dims& s, const __nv_bfloat16* q, const __nv_bfloat16* k,
                   const __nv_bfloat16* v, const int32_t* row_ptr, const int32_t* col_idx,
                   float scale, __nv_bfloat16* o, float* lse, const int32_t* items,
                   int32_t* counter, uint64_t* prof, int32_t* d_status, cudaStream_t st) {
  using C = FwdCfg<BT, D>;
  auto kern = attn_fwd_mma_kernel<BT, D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) !=
      cudaSuccess)
    return SPARSP_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return SPARSP_ERR_CUDA;
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::kThreads, C::kSmem);
  if (per_sm < 1) per_sm = 1;
  const int64_t n_items = s.rows();
  const int64_t grid = cap_grid(s, (int64_t)sms * per_sm, n_items);
  kern<<<(unsigned)grid, C::kThreads, C::kSmem, st>>>(q, k, v, row_ptr, col_idx, s.N, s.nb,
                                                      n_items, scale * 1.4426950408889634f, o, lse,
                                                      items, counter, prof, d_status);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace

sparsp_status_t launch_attn_fwd_mma(const Dims& s, const __nv_bfloat16* q, const __nv_bfloat16* k,
                                    const __nv_bfloat16* v, const int32_t* row_ptr,
                                    const int32_t* col_idx, float scale, __nv_bfloat16* o,
                                    float* lse, const int32_t* items, int32_t* counter,
                                    uint64_t* prof, int32_t* d_status, cudaStream_t st) {
#define GO(BT, D) go<BT, D>(s, q, k, v, row_ptr, col_idx, scale, o, lse, items, counter, prof, d_status, st)
  if (s.Bt == 64) return s.d == 64 ? GO(64, 64) : GO(64, 128);
  return s.d == 64 ? GO(128, 64) : GO(128, 128);
#undef GO
}

}  // namespace sparsp
