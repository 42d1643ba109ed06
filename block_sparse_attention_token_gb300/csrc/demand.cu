// Step 4: KV demand of P virtual query partitions.
//
//  0. zero_bytes_kernel - clears the four byte counters.
//  1. bitmap_kernel - one CTA per partition (b, h, r). Contiguous split: the
//     partition's rows are consecutive CSR rows, so its entries are one
//     contiguous range of col_idx. With a block owner map: warps scan the
//     head's rows and take those whose owner is r. Each index is OR-ed into a
//     shared bitmap. Writes the bitmap, its population into dem_ptr[part] and
//     the byte counters.
//  2. scan          - dem_ptr counts -> offsets.
//  3. list_kernel   - one warp per partition writes the set bits ascending.
//  4. gather_kernel - one CTA per demanded slot copies the K and V tiles
//     (Bt x d, contiguous in the block-ordered layout) with 16-byte vectors;
//     stores are streaming (the gathered copy is not re-read here), loads keep
//     the default policy so the P-fold reuse of a source tile hits in L2. It
//     also runs alone (sparsp_kv_gather): with no shared memory and one warp of
//     at most 64 registers per SM sub-partition it fits beside the attention
//     kernel's CTA, on another stream.
#include "common.cuh"

namespace sparsp {
namespace {

constexpr int kMaxWords = kMaxBlocks / 32;   // bitmap words of nb <= kMaxBlocks blocks

__device__ __forceinline__ void or_row(const int32_t* __restrict__ col_idx, int32_t e0, int32_t e1,
                                       int step, int first, int nb, uint32_t* bits, int32_t* d_status) {
  for (int32_t e = e0 + first; e < e1; e += step) {
    const int32_t j = col_idx[e];
    if (j < 0 || j >= nb) {
      report(d_status, SPARSP_ERR_DATA);
      continue;
    }
    atomicOr(&bits[j >> 5], 1u << (j & 31));
  }
}

__global__ void __launch_bounds__(256)
bitmap_kernel(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ col_idx,
              const int32_t* __restrict__ owner, int H, int nb, int P, uint64_t tile2,
              uint32_t* __restrict__ bitmap, int32_t* __restrict__ counts,
              uint64_t* __restrict__ bytes, int32_t* d_status) {
  __shared__ uint32_t bits[kMaxWords], mine[kMaxWords];
  const int part = blockIdx.x;           // (b*H + h)*P + r
  const int bh = part / P, r = part % P;
  const int W = (nb + 31) / 32;
  for (int w = threadIdx.x; w < kMaxWords; w += blockDim.x) {
    bits[w] = 0u;
    mine[w] = 0u;
  }
  __syncthreads();
  if (owner == nullptr) {
    const int lo = (int)(((int64_t)r * nb) / P), hi = (int)(((int64_t)(r + 1) * nb) / P);
    for (int j = lo + (int)threadIdx.x; j < hi; j += blockDim.x) atomicOr(&mine[j >> 5], 1u << (j & 31));
    const int64_t row0 = (int64_t)bh * nb + lo, row1 = (int64_t)bh * nb + hi;
    const int32_t e0 = row_ptr[row0], e1 = row_ptr[row1];
    if (e1 < e0) {
      if (threadIdx.x == 0) report(d_status, SPARSP_ERR_DATA);
    } else {
      or_row(col_idx, e0, e1, blockDim.x, threadIdx.x, nb, bits, d_status);
    }
  } else {
    const int32_t* own_b = owner + (int64_t)(bh / H) * nb;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    for (int i = warp; i < nb; i += nwarps) {
      const int32_t oi = own_b[i];
      if (oi < 0 || oi >= P) {
        if (lane == 0 && r == 0) report(d_status, SPARSP_ERR_DATA);
        continue;
      }
      if (oi != r) continue;
      if (lane == 0) atomicOr(&mine[i >> 5], 1u << (i & 31));
      const int64_t row = (int64_t)bh * nb + i;
      const int32_t e0 = row_ptr[row], e1 = row_ptr[row + 1];
      if (e1 < e0) {
        if (lane == 0) report(d_status, SPARSP_ERR_DATA);
        continue;
      }
      or_row(col_idx, e0, e1, 32, lane, nb, bits, d_status);
    }
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    int total = 0, remote = 0, owned = 0;
    for (int w = threadIdx.x; w < W; w += 32) {
      const uint32_t word = bits[w], own = mine[w];
      bitmap[(int64_t)part * W + w] = word;
      total += __popc(word);
      remote += __popc(word & ~own);
      owned += __popc(own);
    }
    const int w = threadIdx.x;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      total += __shfl_xor_sync(0xffffffffu, total, off);
      remote += __shfl_xor_sync(0xffffffffu, remote, off);
      owned += __shfl_xor_sync(0xffffffffu, owned, off);
    }
    if (w == 0) {
      counts[part] = total;
      atomicAdd((unsigned long long*)&bytes[0], (unsigned long long)total * tile2);
      atomicAdd((unsigned long long*)&bytes[2], (unsigned long long)remote * tile2);
      atomicAdd((unsigned long long*)&bytes[3], (unsigned long long)(nb - owned) * tile2);
      atomicAdd((unsigned long long*)&bytes[1], (unsigned long long)nb * tile2);
    }
  }
}

__global__ void __launch_bounds__(256)
list_kernel(const uint32_t* __restrict__ bitmap, const int32_t* __restrict__ dem_ptr, int nparts,
            int W, int32_t* __restrict__ dem_idx, int32_t* d_status) {
  const int lane = threadIdx.x & 31;
  const int part = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (part >= nparts) return;
  // lane l takes words [l*per, l*per + per): the set bits come out ascending
  const int per = (W + 31) / 32, w0 = lane * per, w1 = min(W, w0 + per);
  const uint32_t* bm = bitmap + (int64_t)part * W;
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(bm[w]);
  int incl = cnt;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  int pos = dem_ptr[part] + incl - cnt;
  const int end = dem_ptr[part + 1];
  for (int w = w0; w < w1; ++w) {
    uint32_t word = bm[w];
    while (word) {
      const int bit = __ffs(word) - 1;
      if (dcheck(pos < end, d_status)) dem_idx[pos] = w * 32 + bit;
      ++pos;
      word &= word - 1;
    }
  }
}

__global__ void zero_bytes_kernel(uint64_t* bytes) {
  if (threadIdx.x < 4) bytes[threadIdx.x] = 0ull;
}

// One CTA per slot < min(total, cap). The owning partition is found by binary
// search in dem_ptr. Four warps of at most 64 registers: one warp per SM
// sub-partition, which is what the attention kernel's CTA leaves room for.
constexpr int kGatherThreads = 128;

__global__ void __launch_bounds__(kGatherThreads, 8)
gather_kernel(const int32_t* __restrict__ dem_ptr, const int32_t* __restrict__ dem_idx, int nparts,
              int P, int64_t N, int Bt, int nb, int vec_per_row, const uint4* __restrict__ k,
              const uint4* __restrict__ v, uint4* __restrict__ kg, uint4* __restrict__ vg,
              int64_t cap, int32_t* d_status) {
  // the lists may come from the caller (sparsp_kv_gather): a total beyond what
  // nparts partitions can demand, or an index outside [0, nb), is reported
  // and never used as an address
  int64_t total = dem_ptr[nparts];
  const int64_t slot = blockIdx.x;
  if (total < 0 || total > (int64_t)nparts * nb) {
    if (slot == 0 && threadIdx.x == 0) report(d_status, SPARSP_ERR_DATA);
    total = 0;
  }
  if (slot == 0 && total > cap && threadIdx.x == 0) report(d_status, SPARSP_ERR_CAPACITY);
  if (slot >= total || slot >= cap) return;
  int lo = 0, hi = nparts - 1;   // last part with dem_ptr[part] <= slot
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (dem_ptr[mid] <= slot) lo = mid; else hi = mid - 1;
  }
  const int bh = lo / P;
  const int j = dem_idx[slot];
  if (j < 0 || j >= nb) {
    if (threadIdx.x == 0) report(d_status, SPARSP_ERR_DATA);
    return;
  }
  const int64_t nvec = (int64_t)Bt * vec_per_row;
  const uint4* ks = k + ((int64_t)bh * N + (int64_t)j * Bt) * vec_per_row;
  const uint4* vs = v + ((int64_t)bh * N + (int64_t)j * Bt) * vec_per_row;
  uint4* kd = kg + slot * nvec;
  uint4* vd = vg + slot * nvec;
  constexpr int kUnroll = 4;
  if (nvec % (kUnroll * kGatherThreads) == 0) {   // whole rounds: no per-vector bounds checks
    const int t = threadIdx.x;
    for (int64_t e = 0; e < nvec; e += kUnroll * kGatherThreads) {
      uint4 a[kUnroll], b[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        a[u] = ks[e + u * kGatherThreads + t];
        b[u] = vs[e + u * kGatherThreads + t];
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        __stcs(kd + e + u * kGatherThreads + t, a[u]);
        __stcs(vd + e + u * kGatherThreads + t, b[u]);
      }
    }
    return;
  }
  for (int64_t e = threadIdx.x; e < nvec; e += 4 * blockDim.x) {
    uint4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t idx = e + u * blockDim.x;
      if (idx < nvec) {
        a[u] = ks[idx];
        b[u] = vs[idx];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t idx = e + u * blockDim.x;
      if (idx < nvec) {
        __stcs(kd + idx, a[u]);
        __stcs(vd + idx, b[u]);
      }
    }
  }
}

// The gather from raster K and V ([B, N, H, d]): the same slots and lists,
// each tile's token rows read at their raster addresses. Tile sides are powers
// of two (64- or 128-token tiles), so a token's offset inside its tile comes
// from shifts: token o = (it, iy, ix) sits (it*Y + iy)*X + ix raster tokens
// after the tile's first. Each thread copies 4 consecutive vectors (64 bytes)
// of one row per step, so that four threads cover a 256-byte row.
__global__ void __launch_bounds__(kGatherThreads, 8)
gather_raster_kernel(const int32_t* __restrict__ dem_ptr, const int32_t* __restrict__ dem_idx, int nparts,
                     int P, int64_t N, int H, int Y, int X, int ta, int tb, int tc, int nY, int nX, int Bt, int nb,
                     int vec_per_row, int l_tbc, int l_tc, const uint4* __restrict__ k,
                     const uint4* __restrict__ v, uint4* __restrict__ kg, uint4* __restrict__ vg, int64_t cap,
                     int32_t* d_status) {
  int64_t total = dem_ptr[nparts];
  const int64_t slot = blockIdx.x;
  if (total < 0 || total > (int64_t)nparts * nb) {
    if (slot == 0 && threadIdx.x == 0) report(d_status, SPARSP_ERR_DATA);
    total = 0;
  }
  if (slot == 0 && total > cap && threadIdx.x == 0) report(d_status, SPARSP_ERR_CAPACITY);
  if (slot >= total || slot >= cap) return;
  int lo = 0, hi = nparts - 1;   // last part with dem_ptr[part] <= slot
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (dem_ptr[mid] <= slot) lo = mid; else hi = mid - 1;
  }
  const int bh = lo / P;
  const int j = dem_idx[slot];
  if (j < 0 || j >= nb) {
    if (threadIdx.x == 0) report(d_status, SPARSP_ERR_DATA);
    return;
  }
  const int bx = j % nX, by = (j / nX) % nY, bt = j / (nX * nY);
  const int64_t n0 = ((int64_t)bt * ta * Y + (int64_t)by * tb) * X + (int64_t)bx * tc;   // the tile's first token
  const int64_t rowbase = ((int64_t)(bh / H) * N + n0) * H + bh % H;
  const int64_t yx = (int64_t)Y * X;
  const int64_t nvec = (int64_t)Bt * vec_per_row;
  uint4* kd = kg + slot * nvec;
  uint4* vd = vg + slot * nvec;
  for (int64_t e = 4 * (int64_t)threadIdx.x; e < nvec; e += 4 * kGatherThreads) {
    const int o = (int)(e / vec_per_row), col = (int)(e % vec_per_row);
    const int64_t off = (int64_t)(o >> l_tbc) * yx + (int64_t)((o >> l_tc) & (tb - 1)) * X + (o & (tc - 1));
    const int64_t src = (rowbase + off * H) * vec_per_row + col;
    uint4 a[4], b[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      a[u] = k[src + u];
      b[u] = v[src + u];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      __stcs(kd + e + u, a[u]);
      __stcs(vd + e + u, b[u]);
    }
  }
}

}  // namespace

sparsp_status_t launch_kv_demand(const Dims& s, int P, const int32_t* row_ptr,
                                 const int32_t* col_idx, const int32_t* owner, uint32_t* bitmap, int32_t* dem_ptr,
                                 int32_t* dem_idx, const void* k, const void* v, void* kg,
                                 void* vg, int64_t cap, uint64_t* bytes, int32_t* d_status,
                                 cudaStream_t st) {
  const int nparts = s.B * s.H * P;
  const int W = (s.nb + 31) / 32;
  const uint64_t tile2 = (uint64_t)s.Bt * s.d * s.elem * 2;
  zero_bytes_kernel<<<1, 32, 0, st>>>(bytes);
  SPARSP_LAUNCH_CHECK();
  bitmap_kernel<<<nparts, 256, 0, st>>>(row_ptr, col_idx, owner, s.H, s.nb, P, tile2, bitmap, dem_ptr,
                                        bytes, d_status);
  SPARSP_LAUNCH_CHECK();
  sparsp_status_t r = launch_scan_counts(dem_ptr, nparts, st);
  if (r != SPARSP_OK) return r;
  list_kernel<<<(nparts + 7) / 8, 256, 0, st>>>(bitmap, dem_ptr, nparts, W, dem_idx, d_status);
  SPARSP_LAUNCH_CHECK();
  if (kg != nullptr && vg != nullptr) return launch_kv_gather(s, P, dem_ptr, dem_idx, k, v, kg, vg, cap, d_status, st);
  return SPARSP_OK;
}

sparsp_status_t launch_kv_gather(const Dims& s, int P, const int32_t* dem_ptr, const int32_t* dem_idx,
                                 const void* k, const void* v, void* kg, void* vg, int64_t cap, int32_t* d_status,
                                 cudaStream_t st) {
  const int nparts = s.B * s.H * P;
  // grid >= 1 so that slot 0 can report a capacity shortfall even when cap == 0
  const int64_t upper = (int64_t)nparts * s.nb;
  int64_t grid = upper < cap ? upper : cap;
  if (grid < 1) grid = 1;
  const int vec_per_row = s.d * s.elem / 16;
  gather_kernel<<<(unsigned)grid, kGatherThreads, 0, st>>>(dem_ptr, dem_idx, nparts, P, s.N, s.Bt, s.nb, vec_per_row,
                                                 (const uint4*)k, (const uint4*)v, (uint4*)kg, (uint4*)vg, cap,
                                                 d_status);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

sparsp_status_t launch_kv_gather_raster(const Dims& s, int P, const int32_t* dem_ptr, const int32_t* dem_idx,
                                        const void* k, const void* v, void* kg, void* vg, int64_t cap,
                                        int32_t* d_status, cudaStream_t st) {
  const int nparts = s.B * s.H * P;
  const int64_t upper = (int64_t)nparts * s.nb;
  int64_t grid = upper < cap ? upper : cap;
  if (grid < 1) grid = 1;
  const int vec_per_row = s.d * s.elem / 16;
  // tile sides are powers of two (64 or 128 tokens)
  const int l_tc = __builtin_ctz((unsigned)s.tc), l_tbc = __builtin_ctz((unsigned)(s.tb * s.tc));
  gather_raster_kernel<<<(unsigned)grid, kGatherThreads, 0, st>>>(
      dem_ptr, dem_idx, nparts, P, s.N, s.H, s.Y, s.X, s.ta, s.tb, s.tc, s.nY, s.nX, s.Bt, s.nb, vec_per_row, l_tbc,
      l_tc, (const uint4*)k, (const uint4*)v, (uint4*)kg, (uint4*)vg, cap, d_status);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace sparsp
