// Step 5a, float32 inputs: block-sparse attention forward with true fp32 FFMA
// (no TF32), for workloads whose tolerance is 1e-4.
//
// Persistent CTAs of Bt threads pull work items (b, h, query block i) from
// the longest-first list. Thread t owns query row t: its O accumulator (d
// floats) lives in registers, its q row in padded shared memory. For each
// selected key block the K and V tiles are staged in shared memory; keys are
// consumed 8 at a time with an online softmax in base 2.
#include "common.cuh"

namespace sparsp {
namespace {

constexpr int kChunk = 8;

// Scans the CSR row; returns its length, or -1 (and reports) if malformed.
__device__ int checked_row(const int32_t* row_ptr, const int32_t* col_idx, int64_t r, int nb,
                           int32_t* d_status, int* flag_s) {
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

template <int D, int BT>
__global__ void __launch_bounds__(BT, 1)
attn_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                    const float* __restrict__ v, const int32_t* __restrict__ row_ptr,
                    const int32_t* __restrict__ col_idx, int64_t N, int nb, int64_t n_items,
                    float scale_log2, float* __restrict__ o, float* __restrict__ lse,
                    const int32_t* __restrict__ items, int32_t* __restrict__ counter,
                    uint64_t* prof, int32_t* d_status) {
  extern __shared__ float smem[];
  float* ks = smem;                      // [BT][D]
  float* vs = ks + BT * D;               // [BT][D]
  float* qs = vs + BT * D;               // [BT][D+1]
  __shared__ int32_t item_s;
  const uint64_t t_start = globaltimer_ns();
  const int t = threadIdx.x;
  for (;;) {
    if (t == 0) item_s = atomicAdd(counter, 1);
    __syncthreads();
    const int32_t slot = item_s;
    __syncthreads();
    if (slot >= n_items) break;
    const int64_t item = items[slot];
    const int64_t bh = item / nb;
    const int i = (int)(item % nb);
    const int len = checked_row(row_ptr, col_idx, item, nb, d_status, nullptr);
    if (len < 0) continue;
    const int32_t e0 = row_ptr[item];
    const int64_t row0 = bh * N + (int64_t)i * BT;       // first query row
    // stage q rows (padded) and zero the accumulator
    for (int e = t; e < BT * D / 4; e += BT) {
      const float4 x = reinterpret_cast<const float4*>(q + row0 * D)[e];
      const int r = (e * 4) / D, c = (e * 4) % D;
      float* dst = qs + r * (D + 1) + c;
      dst[0] = x.x; dst[1] = x.y; dst[2] = x.z; dst[3] = x.w;
    }
    float acc[D];
#pragma unroll
    for (int c = 0; c < D; ++c) acc[c] = 0.f;
    float m = -INFINITY, l = 0.f;
    const float* qrow = qs + t * (D + 1);
    for (int e = 0; e < len; ++e) {
      const int j = col_idx[e0 + e];
      const int64_t key0 = bh * N + (int64_t)j * BT;
      __syncthreads();      // previous tile fully consumed (and q staged)
      for (int x = t; x < BT * D / 4; x += BT) {
        reinterpret_cast<float4*>(ks)[x] = reinterpret_cast<const float4*>(k + key0 * D)[x];
        reinterpret_cast<float4*>(vs)[x] = reinterpret_cast<const float4*>(v + key0 * D)[x];
      }
      __syncthreads();
      for (int kb = 0; kb < BT; kb += kChunk) {
        float s[kChunk];
#pragma unroll
        for (int u = 0; u < kChunk; ++u) s[u] = 0.f;
        for (int c = 0; c < D; ++c) {
          const float qc = qrow[c];
#pragma unroll
          for (int u = 0; u < kChunk; ++u) s[u] = fmaf(qc, ks[(kb + u) * D + c], s[u]);
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
        for (int c = 0; c < D; ++c) {
          float a = acc[c] * alpha;
#pragma unroll
          for (int u = 0; u < kChunk; ++u) a = fmaf(p[u], vs[(kb + u) * D + c], a);
          acc[c] = a;
        }
      }
    }
    const int64_t row = row0 + t;
    if (len == 0) {
#pragma unroll
      for (int c = 0; c < D; ++c) o[row * D + c] = 0.f;
      lse[row] = -INFINITY;
    } else {
      const float inv = 1.0f / l;
#pragma unroll
      for (int c = 0; c < D; c += 4) {
        float4 w = make_float4(acc[c] * inv, acc[c + 1] * inv, acc[c + 2] * inv, acc[c + 3] * inv);
        reinterpret_cast<float4*>(o + row * D)[c / 4] = w;
      }
      lse[row] = (m + log2f(l)) * 0.69314718055994531f;
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
  const size_t smem = (size_t)(2 * BT * D + BT * (D + 1)) * sizeof(float);
  auto kern = attn_fwd_f32_kernel<D, BT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return SPARSP_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return SPARSP_ERR_CUDA;
  const int64_t n_items = s.rows();
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, BT, smem);
  if (per_sm < 1) per_sm = 1;
  const int64_t grid = cap_grid(s, (int64_t)sms * per_sm, n_items);
  const float scale_log2 = scale * 1.4426950408889634f;
  kern<<<(unsigned)grid, BT, smem, st>>>(q, k, v, row_ptr, col_idx, s.N, s.nb, n_items, scale_log2,
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
