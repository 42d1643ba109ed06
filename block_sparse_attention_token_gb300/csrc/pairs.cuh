// Pairs of neighbouring 64-token blocks as one 128-row tile (the tcgen05
// attention kernels): a pair's two CSR rows (or transposed-CSR columns) as
// bitmaps in shared memory, the ascending walk over their union, and the
// per-stage masks (which of the two rows selected each block of the union).
// Warp-collective where noted; all lanes run uniformly.
#pragma once

#include "common.cuh"

namespace sparsp {
namespace tc {

// Walk over the set bits of (a | b) in ascending order: the blocks of a pair
// item's stages, two at a time.
struct UnionWalk {
  const uint32_t* a;
  const uint32_t* b;
  int words, w;
  uint32_t cur;
  __device__ __forceinline__ UnionWalk(const uint32_t* a_, const uint32_t* b_, int words_)
      : a(a_), b(b_), words(words_), w(0), cur(words_ > 0 ? (a_[0] | b_[0]) : 0u) {}
  __device__ __forceinline__ int next() {
    while (cur == 0u) {
      if (++w >= words) return -1;
      cur = a[w] | b[w];
    }
    const int j = w * 32 + __ffs(cur) - 1;
    cur &= cur - 1u;
    return j;
  }
};

// Validates list r of a CSR-like structure (length <= nb, indices in [0, nb),
// no index twice) and writes its bitmap (words zeroed before). Warp-collective;
// returns false for a bad list, whose bitmap is then cleared.
__device__ __forceinline__ bool list_bitmap(const int32_t* ptr, const int32_t* idx, int nb, int64_t r,
                                            uint32_t* bm, int words, int lane) {
  const int32_t a = ptr[r], b = ptr[r + 1];
  bool bad = (b < a) || (b - a > nb);
  if (!bad)
    for (int32_t e = a + lane; e < b; e += 32) {
      const int32_t j = idx[e];
      if (j < 0 || j >= nb) bad = true;
      else atomicOr(&bm[j >> 5], 1u << (j & 31));
    }
  bad = __any_sync(0xffffffffu, bad);
  __syncwarp();
  if (!bad) {
    int cnt = 0;
    for (int w = lane; w < words; w += 32) cnt += __popc(bm[w]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
    bad = cnt != b - a;   // an index listed twice
  }
  if (bad) {
    for (int w = lane; w < words; w += 32) bm[w] = 0u;
    __syncwarp();
  }
  return !bad;
}

// The size u of the union of bitmaps a and b (warp-collective).
__device__ __forceinline__ int union_count(const uint32_t* a, const uint32_t* b, int words, int lane) {
  int u = 0;
  for (int w = lane; w < words; w += 32) u += __popc(a[w] | b[w]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) u += __shfl_xor_sync(0xffffffffu, u, off);
  return u;
}

// One byte per block of the union of a and b, in ascending order (byte 2s + t:
// block t of stage s; bit 0 = a has it, bit 1 = b has it), and a zero byte
// after an odd union (a lone last block has no partner). The union's set bits
// are ranked by a warp prefix sum over the words. Warp-collective; mk holds at
// least u + 1 bytes.
__device__ __forceinline__ void union_masks(const uint32_t* a, const uint32_t* b, int words, int u, int lane,
                                            uint8_t* mk) {
  int base_rank = 0;
  for (int w0 = 0; w0 < words; w0 += 32) {
    const int w = w0 + lane;
    const uint32_t x = w < words ? a[w] : 0u, y = w < words ? b[w] : 0u;
    uint32_t un = x | y;
    const int c = __popc(un);
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    int rk = base_rank + incl - c;
    while (un != 0u) {
      const int bit = __ffs(un) - 1;
      un &= un - 1u;
      mk[rk++] = (uint8_t)(((x >> bit) & 1u) | (((y >> bit) & 1u) << 1));
    }
    base_rank += __shfl_sync(0xffffffffu, incl, 31);
  }
  if ((u & 1) && lane == 0) mk[u] = 0;
}

// The same masks at two bits per union block (bit 2r: a has the block of
// rank r; bit 2r + 1: b has it), so that stage s (ranks 2s, 2s + 1) is nibble
// s of mk. Warp-collective; mk holds at least (2u + 31) / 32 + 1 words, which
// are cleared first (ranks of one word can come from different lanes).
__device__ __forceinline__ void union_masks2(const uint32_t* a, const uint32_t* b, int words, int u, int lane,
                                             uint32_t* mk) {
  const int nw = (2 * u + 31) / 32 + 1;
  for (int w = lane; w < nw; w += 32) mk[w] = 0u;
  __syncwarp();
  int base_rank = 0;
  for (int w0 = 0; w0 < words; w0 += 32) {
    const int w = w0 + lane;
    const uint32_t x = w < words ? a[w] : 0u, y = w < words ? b[w] : 0u;
    uint32_t un = x | y;
    const int c = __popc(un);
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += t;
    }
    // this word's c codes (ranks rk0 .. rk0 + c - 1) as 64 bits in registers,
    // then OR-ed into the at most three mask words they straddle
    const int rk0 = base_rank + incl - c;
    uint32_t lo = 0u, hi = 0u;
    for (int n = 0; un != 0u; ++n) {
      const int bit = __ffs(un) - 1;
      un &= un - 1u;
      const uint32_t code = ((x >> bit) & 1u) | (((y >> bit) & 1u) << 1);
      if (n < 16) lo |= code << (2 * n);
      else hi |= code << (2 * (n - 16));
    }
    if (c > 0) {
      const int wd = rk0 >> 4, sh = 2 * (rk0 & 15);
      atomicOr(&mk[wd], lo << sh);
      const uint32_t m1 = (sh ? lo >> (32 - sh) : 0u) | (hi << sh);
      const uint32_t m2 = sh ? hi >> (32 - sh) : 0u;
      if (m1) atomicOr(&mk[wd + 1], m1);
      if (m2) atomicOr(&mk[wd + 2], m2);
    }
    base_rank += __shfl_sync(0xffffffffu, incl, 31);
  }
  __syncwarp();
}

}  // namespace tc
}  // namespace sparsp
