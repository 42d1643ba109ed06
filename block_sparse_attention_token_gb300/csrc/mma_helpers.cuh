// Warp-level bf16 tensor-core helpers (mma.sync m16n8k16, ldmatrix, cp.async)
// and the XOR-swizzled shared-memory tile layout they read.
#pragma once

#include "common.cuh"

namespace sparsp {
namespace mma {

// Tile of R rows x D bf16 in shared memory; 16-byte chunk c of row r is stored
// at chunk position c ^ (r & 7), so that ldmatrix's 8 row addresses hit 8
// different bank groups.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c16) {
  return (uint32_t)(r * D * 2 + ((c16 ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Copy a [R x D] bf16 tile (row-major, contiguous) into swizzled smem.
template <int R, int D, int THREADS>
__device__ __forceinline__ void load_tile(uint32_t sbase, const __nv_bfloat16* g) {
  constexpr int kChunks = R * D / 8;
  constexpr int kPerRow = D / 8;
#pragma unroll
  for (int x = threadIdx.x; x < kChunks; x += THREADS) {
    const int r = x / kPerRow, c = x % kPerRow;
    cp_async16(sbase + swz<D>(r, c), g + (size_t)r * D + c * 8);
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A(16x16 row) * B(16x8 col), bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// A fragments (16 rows x 16 k) of a row-major [rows][D] swizzled tile.
template <int D>
__device__ __forceinline__ void load_a(uint32_t base, int row0, int k0, uint32_t* a) {
  const int lane = threadIdx.x & 31;
  const int r = row0 + (lane & 15);
  const int c = (k0 >> 3) + (lane >> 4);
  ldsm_x4(base + swz<D>(r, c), a[0], a[1], a[2], a[3]);
}

// B fragments for two n8 tiles (rows n0..n0+15 of a [n][k] tile) at k0: "col"
// operand from a row-major [n][D] tile (no transpose).
template <int D>
__device__ __forceinline__ void load_b_nk(uint32_t base, int n0, int k0, uint32_t* b) {
  const int lane = threadIdx.x & 31;
  const int r = n0 + (lane & 7) + ((lane >> 4) << 3);
  const int c = (k0 >> 3) + ((lane >> 3) & 1);
  ldsm_x4(base + swz<D>(r, c), b[0], b[1], b[2], b[3]);
}

// B fragments for two n8 tiles (columns n0..n0+15) at k rows k0..k0+15 of a
// row-major [k][D] tile (transposed load).
template <int D>
__device__ __forceinline__ void load_b_kn(uint32_t base, int k0, int n0, uint32_t* b) {
  const int lane = threadIdx.x & 31;
  const int r = k0 + (lane & 7) + (((lane >> 3) & 1) << 3);
  const int c = (n0 >> 3) + (lane >> 4);
  ldsm_x4_t(base + swz<D>(r, c), b[0], b[1], b[2], b[3]);
}

}  // namespace mma
}  // namespace sparsp
