// Step 5a, float32 inputs: block-sparse attention forward with true fp32 FFMA
// (no TF32), for workloads whose tolerance is 1e-4.
//
// Persistent CTAs of 256 threads pull work items from the longest-first list;
// an item is 16 query rows of a query block (the Bt/16 items of one block are
// consecutive, so their CTAs share the K and V tiles in L2). Thread (g, r)
// takes the keys [g Bt/16, (g+1) Bt/16) of every selected key block for
// query row r, with its own online softmax in base 2 (maximum, sum and a
// d-float accumulator in registers) up to eight keys at a time; every
// shared-memory read is 16 bytes, and a warp's K and V reads go to two
// addresses (its two key groups). The K and V tiles of a key block are one
// contiguous bulk copy each, completing on an mbarrier, two blocks in flight
// where both fit in shared memory. At the end of the item the sixteen partial
// states of each row are combined through shared memory (the usual merge of
// softmax partials: scale each by 2^(m_g - M) and add), each thread finishing
// d/16 of its row's columns.
#include "common.cuh"
#include "tc_helpers.cuh"

namespace sparsp {
namespace {

using tc::bulk_load;
using tc::fence_barrier_init;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_try_wait;

constexpr int kThreads = 256;
constexpr int kRows = 16;                        // query rows per item
constexpr int kGroups = kThreads / kRows;        // key groups, two per warp
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;

// Scans the CSR row; returns its length, or -1 (and reports) if malformed.
__device__ int checked_row(const int32_t* row_ptr, const int32_t* col_idx, int64_t r, int nb,
                           int32_t* d_status) {
  const int32_t a = row_ptr[r], b = row_ptr[r + 1];
  int bad = (b < a || b - a > nb) ? 1 : 0;
  if (!bad)
    for (int32_t e = a + threadIdx.x; e < b; e += blockDim.x) {
      const int32_t j = col_idx[e];
      if (j < 0 || j >= nb) bad = 1;
    }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (threadIdx.x == 0) report(d_status, SPARSP_ERR_DATA);
    return -1;
  }
  return b - a;
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, uint64_t limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit) return false;
  return true;
}

template <int D, int BT>
struct F32Cfg {
  static constexpr int KS = BT / kGroups;     // keys of a block per thread
  static constexpr int KC = KS < 8 ? KS : 8;  // keys per online-softmax update
  static constexpr int DP = D + 4;            // padded row stride (floats), 16-byte aligned
  static constexpr int kTile = BT * D;        // floats of one K (or V) tile
  static constexpr int NST = 2 * kTile <= 16384 ? 2 : 1;   // K+V stages in flight
  static constexpr int kTiles = NST * 2 * kTile;
  static constexpr int kMerge = kThreads * DP;
  static constexpr int kRegion = kTiles > kMerge ? kTiles : kMerge;   // tiles, then the merge
  static constexpr size_t kSmemBytes = (size_t)(kRegion + kRows * DP + 2 * kThreads) * sizeof(float);
  static_assert(KS % KC == 0 && D % (4 * kGroups) == 0 && BT % kRows == 0 && kRows * 2 == 32, "layout");
  static_assert(kSmemBytes <= 232448, "shared memory");
};

template <int D, int BT>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                    const float* __restrict__ v, const int32_t* __restrict__ row_ptr,
                    const int32_t* __restrict__ col_idx, int64_t N, int nb, int64_t n_items,
                    float scale_log2, float* __restrict__ o, float* __restrict__ lse,
                    const int32_t* __restrict__ items, int32_t* __restrict__ counter,
                    uint64_t* prof, int32_t* d_status) {
  using C = F32Cfg<D, BT>;
  constexpr int RG = BT / kRows;         // items per query block
  extern __shared__ __align__(16) float smem[];
  float* mrg = smem;                     // [16][16][DP] accumulators, over the tiles after the last block
  float* qs = smem + C::kRegion;         // [16][DP]
  float* ml = qs + kRows * C::DP;        // [16][16] maxima, then [16][16] sums
  __shared__ __align__(8) uint64_t full[2];
  __shared__ int32_t item_s;
  const uint64_t t_start = globaltimer_ns();
  const int t = threadIdx.x;
  const int g = t / kRows, r = t % kRows;   // warp w holds key groups 2w and 2w + 1
  if (t == 0) {
    mbar_init(tc::smem_u32(&full[0]), 1);
    mbar_init(tc::smem_u32(&full[1]), 1);
    fence_barrier_init();
  }
  __syncthreads();
  // stage of block b (counted over the CTA's items): b % NST, phase parity (b / NST) & 1
  uint32_t nblk = 0;
  // K and V tiles of key block j of head bh into the stage of block b (thread 0)
  auto load = [&](int64_t bh, int j, uint32_t b) {
    const uint32_t st = b % C::NST;
    float* ks = smem + st * 2 * C::kTile;
    const int64_t key0 = bh * N + (int64_t)j * BT;
    const uint32_t bar = tc::smem_u32(&full[st]);
    // earlier generic reads and writes of this stage come before the copy
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
    mbar_arrive_expect_tx(bar, 2u * C::kTile * 4u);
    bulk_load(tc::smem_u32(ks), k + key0 * D, C::kTile * 4u, bar);
    bulk_load(tc::smem_u32(ks + C::kTile), v + key0 * D, C::kTile * 4u, bar);
  };
  for (;;) {
    if (t == 0) item_s = atomicAdd(counter, 1);
    __syncthreads();      // also: the previous item's merge reads are done
    const int32_t slot = item_s;
    __syncthreads();
    if (slot >= n_items * RG) break;
    const int64_t item = items[slot / RG];
    const int rg = slot % RG;
    const int64_t bh = item / nb;
    const int i = (int)(item % nb);
    const int len = checked_row(row_ptr, col_idx, item, nb, d_status);
    if (len < 0) continue;
    const int32_t* cols = col_idx + row_ptr[item];
    const int64_t row0 = bh * N + (int64_t)i * BT + rg * kRows;   // first query row of the item
    if (C::NST == 2 && t == 0 && len > 0) load(bh, cols[0], nblk);
    for (int e = t; e < kRows * D / 4; e += kThreads) {
      const float4 x = reinterpret_cast<const float4*>(q + row0 * D)[e];
      const int rr = (e * 4) / D, c = (e * 4) % D;
      *reinterpret_cast<float4*>(qs + rr * C::DP + c) = x;
    }
    __syncthreads();
    float acc[D];
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] = 0.f;
    float m = -INFINITY, l = 0.f;
    const float4* qrow = reinterpret_cast<const float4*>(qs + r * C::DP);
    for (int e = 0; e < len; ++e) {
      const uint32_t b = nblk + (uint32_t)e;
      if (t == 0) {
        // the next block's tiles go to the other stage, whose last reader
        // (block b - 1) passed the block barrier at the end of its iteration
        if (C::NST == 1) load(bh, cols[e], b);
        else if (e + 1 < len) load(bh, cols[e + 1], b + 1);
      }
      const float* ks = smem + (b % C::NST) * 2 * C::kTile;
      const float* vs = ks + C::kTile;
      const bool ok = wait_phase(tc::smem_u32(&full[b % C::NST]), (b / C::NST) & 1u, kWaitNs);
      if (ok) {
        constexpr int kChunk = C::KC;
        for (int kb = g * C::KS; kb < (g + 1) * C::KS; kb += kChunk) {
          const float4* kr = reinterpret_cast<const float4*>(ks + kb * D);
          const float4* vr = reinterpret_cast<const float4*>(vs + kb * D);
          float s[kChunk];
#pragma unroll
          for (int u = 0; u < kChunk; ++u) s[u] = 0.f;
#pragma unroll 4
          for (int c4 = 0; c4 < D / 4; ++c4) {
            const float4 qc = qrow[c4];
#pragma unroll
            for (int u = 0; u < kChunk; ++u) {
              const float4 kc = kr[u * (D / 4) + c4];
              float a = fmaf(qc.x, kc.x, s[u]);
              a = fmaf(qc.y, kc.y, a);
              a = fmaf(qc.z, kc.z, a);
              s[u] = fmaf(qc.w, kc.w, a);
            }
          }
          float cmax = -INFINITY;
#pragma unroll
          for (int u = 0; u < kChunk; ++u) {
            s[u] *= scale_log2;
            cmax = fmaxf(cmax, s[u]);
          }
          const float m_new = fmaxf(m, cmax);
          const float alpha = exp2f(m - m_new);     // 0 on the first chunk (m = -inf)
          float p[kChunk];
          float psum = 0.f;
#pragma unroll
          for (int u = 0; u < kChunk; ++u) {
            p[u] = exp2f(s[u] - m_new);
            psum += p[u];
          }
          l = l * alpha + psum;
          m = m_new;
#pragma unroll
          for (int c4 = 0; c4 < D / 4; ++c4) {
            float a0 = acc[4 * c4] * alpha, a1 = acc[4 * c4 + 1] * alpha;
            float a2 = acc[4 * c4 + 2] * alpha, a3 = acc[4 * c4 + 3] * alpha;
#pragma unroll
            for (int u = 0; u < kChunk; ++u) {
              const float4 vc = vr[u * (D / 4) + c4];
              a0 = fmaf(p[u], vc.x, a0);
              a1 = fmaf(p[u], vc.y, a1);
              a2 = fmaf(p[u], vc.z, a2);
              a3 = fmaf(p[u], vc.w, a3);
            }
            acc[4 * c4] = a0;
            acc[4 * c4 + 1] = a1;
            acc[4 * c4 + 2] = a2;
            acc[4 * c4 + 3] = a3;
          }
        }
      }
      // every thread is done with this stage; all agree on whether to go on
      if (!__syncthreads_and(ok)) {
        if (t == 0) {
          report(d_status, SPARSP_ERR_TIMEOUT);
          // let the copies still in flight land before the CTA exits
          const uint32_t issued = C::NST == 1 ? b + 1 : (e + 1 < len ? b + 2 : b + 1);
          for (uint32_t x = b; x < issued; ++x)
            wait_phase(tc::smem_u32(&full[x % C::NST]), (x / C::NST) & 1u, kDrainNs);
        }
        __syncthreads();
        return;
      }
    }
    nblk += (uint32_t)len;
    // combine the sixteen partial states of each row; thread (g, r) then
    // finishes columns [g D/16, (g+1) D/16) of row r (no copy is in flight:
    // the tiles' last reads passed the block barrier above)
    {
      float* dst = mrg + (g * kRows + r) * C::DP;
#pragma unroll
      for (int c4 = 0; c4 < D / 4; ++c4)
        *reinterpret_cast<float4*>(dst + 4 * c4) =
            make_float4(acc[4 * c4], acc[4 * c4 + 1], acc[4 * c4 + 2], acc[4 * c4 + 3]);
      ml[g * kRows + r] = m;
      ml[kThreads + g * kRows + r] = l;
    }
    __syncthreads();
    const int64_t row = row0 + r;
    constexpr int DG = D / kGroups;
    if (len == 0) {
      for (int c = g * DG; c < (g + 1) * DG; c += 4)
        *reinterpret_cast<float4*>(o + row * D + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      if (g == 0) lse[row] = -INFINITY;
    } else {
      float M = -INFINITY;
#pragma unroll
      for (int h = 0; h < kGroups; ++h) M = fmaxf(M, ml[h * kRows + r]);
      float w[kGroups];
      float L = 0.f;
#pragma unroll
      for (int h = 0; h < kGroups; ++h) {
        w[h] = exp2f(ml[h * kRows + r] - M);
        L = fmaf(ml[kThreads + h * kRows + r], w[h], L);
      }
      const float inv = 1.0f / L;
      for (int c = g * DG; c < (g + 1) * DG; c += 4) {
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int h = 0; h < kGroups; ++h) {
          const float4 a = *reinterpret_cast<const float4*>(mrg + (h * kRows + r) * C::DP + c);
          sum.x = fmaf(a.x, w[h], sum.x);
          sum.y = fmaf(a.y, w[h], sum.y);
          sum.z = fmaf(a.z, w[h], sum.z);
          sum.w = fmaf(a.w, w[h], sum.w);
        }
        *reinterpret_cast<float4*>(o + row * D + c) =
            make_float4(sum.x * inv, sum.y * inv, sum.z * inv, sum.w * inv);
      }
      if (g == 0) lse[row] = (M + log2f(L)) * 0.69314718055994531f;
    }
  }
  if (prof != nullptr && t == 0)
    atomicAdd((unsigned long long*)&prof[smid() % SPARSP_PROF_SLOTS],
              (unsigned long long)(globaltimer_ns() - t_start));
}

template <int D, int BT>
sparsp_status_t go(const Dims& s, const float* q, const float* k, const float* v,
                   const int32_t* row_ptr, const int32_t* col_idx, float scale, float* o,
                   float* lse, const int32_t* items, int32_t* counter, uint64_t* prof,
                   int32_t* d_status, cudaStream_t st) {
  const size_t smem = F32Cfg<D, BT>::kSmemBytes;
  auto kern = attn_fwd_f32_kernel<D, BT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SPARSP_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return SPARSP_ERR_CUDA;
  const int64_t n_items = s.rows();   // query blocks; each is Bt / 16 work items
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (per_sm < 1) per_sm = 1;
  const int64_t grid = cap_grid(s, (int64_t)sms * per_sm, n_items * (BT / kRows));
  const float scale_log2 = scale * 1.4426950408889634f;
  kern<<<(unsigned)grid, kThreads, smem, st>>>(q, k, v, row_ptr, col_idx, s.N, s.nb, n_items, scale_log2,
                                               o, lse, items, counter, prof, d_status);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace

sparsp_status_t launch_attn_fwd_f32(const Dims& s, const float* q, const float* k, const float* v,
                                    const int32_t* row_ptr, const int32_t* col_idx, float scale,
                                    float* o, float* lse, const int32_t* items, int32_t* counter,
                                    uint64_t* prof, int32_t* d_status, cudaStream_t st) {
  if (s.d == 64 && s.Bt == 64)
    return go<64, 64>(s, q, k, v, row_ptr, col_idx, scale, o, lse, items, counter, prof, d_status, st);
  if (s.d == 64 && s.Bt == 128)
    return go<64, 128>(s, q, k, v, row_ptr, col_idx, scale, o, lse, items, counter, prof, d_status, st);
  if (s.d == 128 && s.Bt == 64)
    return go<128, 64>(s, q, k, v, row_ptr, col_idx, scale, o, lse, items, counter, prof, d_status, st);
  return go<128, 128>(s, q, k, v, row_ptr, col_idx, scale, o, lse, items, counter, prof, d_status, st);
}

}  // namespace sparsp
