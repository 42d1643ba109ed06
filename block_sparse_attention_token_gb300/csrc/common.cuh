// Shared internals of libsparsp: derived shape, status reporting, launchers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sparsp.h"

namespace sparsp {

// Largest number of blocks per (b, h) sequence: 4,096 (524,288 tokens in
// 128-token blocks). Dependency-aware placement and slack-aware augmentation
// keep shared-memory tables of one entry per block and take at most
// kMaxBlocksNext.
constexpr int kMaxBlocks = 4096;
constexpr int kMaxBlocksNext = 1024;

// Derived shape, validated by the API layer before any launcher sees it.
struct Dims {
  int B, H, T, Y, X, d, ta, tb, tc, dtype;
  int64_t N;      // tokens per (b, h)
  int Bt;         // tokens per tile
  int nb;         // tiles per (b, h)
  int nT, nY, nX; // tile lattice
  int elem;       // bytes per element
  int max_ctas = 0;   // attention kernels: persistent grid cap (0 = one per SM x occupancy)
  int64_t rows() const { return (int64_t)B * H * nb; }  // CSR rows = work items
};

// Where token o of tile i of head bh (b = bh / H, h = bh % H) sits in a
// raster [B, N, H, d] tensor: tile i = (bt, by, bx) in tile-raster order, token
// o = (it, iy, ix) in raster order inside the tile; the position is
// n = (bt*ta + it)*Y*X + (by*tb + iy)*X + bx*tc + ix and the row (b*N + n)*H + h.
// This is the map of sparsp_reorder, for kernels that read or write raster rows
// themselves.
struct RasterMap {
  int64_t N;
  int H, Y, X, ta, tb, tc, nY, nX;
  __device__ __forceinline__ int64_t row(int64_t bh, int i, int o) const {
    const int tbc = tb * tc;
    const int bx = i % nX, by = (i / nX) % nY, bt = i / (nX * nY);
    const int it = o / tbc, iy = (o - it * tbc) / tc, ix = o - it * tbc - iy * tc;
    const int64_t n = ((int64_t)bt * ta + it) * Y * X + ((int64_t)by * tb + iy) * X + (int64_t)bx * tc + ix;
    return ((bh / H) * N + n) * H + bh % H;
  }
};
inline RasterMap raster_map(const Dims& s) { return RasterMap{s.N, s.H, s.Y, s.X, s.ta, s.tb, s.tc, s.nY, s.nX}; }

// A persistent kernel's grid: `g` CTAs, at most one per work item and at most
// the caller's cap (SPARSP_GRID_CAP), never fewer than one.
inline int64_t cap_grid(const Dims& s, int64_t g, int64_t n_items) {
  if (s.max_ctas > 0 && g > s.max_ctas) g = s.max_ctas;
  if (g > n_items) g = n_items;
  return g < 1 ? 1 : g;
}

// First-error-wins device status word.
__device__ __forceinline__ void report(int32_t* st, int32_t code) {
  if (st != nullptr) atomicCAS(st, 0, code);
}

// Debug builds (compiled with -DSPARSP_DEBUG, see build.py) also check the
// addresses a kernel derives from its own arithmetic - TMA coordinates, output
// rows, list and CSR write positions - and report SPARSP_ERR_DATA instead of
// using one out of range. Release builds check what comes from the caller and
// compile these checks away.
#ifdef SPARSP_DEBUG
__device__ __forceinline__ bool dcheck(bool ok, int32_t* st) {
  if (!ok) report(st, SPARSP_ERR_DATA);
  return ok;
}
#else
__device__ __forceinline__ bool dcheck(bool, int32_t*) { return true; }
#endif

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smid() {
  uint32_t s;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
  return s;
}

// Launch-side helpers -------------------------------------------------------

int device_sm_count();   // cached per device; -1 on error


#define SPARSP_LAUNCH_CHECK()                                       \
  do {                                                              \
    cudaError_t e_ = cudaGetLastError();                            \
    if (e_ != cudaSuccess) return SPARSP_ERR_CUDA;                  \
  } while (0)

// Launchers (each returns SPARSP_OK or SPARSP_ERR_CUDA). -------------------

// means != nullptr: forward reorder that also writes the fp32 tile means [B,H,nb,d]
sparsp_status_t launch_reorder(const Dims& s, const void* in, void* out, bool inverse,
                               cudaStream_t st, float* means = nullptr);
// scores from pooled means (low-rank: projected through W first, into ws)
sparsp_status_t launch_scores_from_means(const Dims& s, int estimator, const float* qm,
                                         const float* km, const float* wq, const float* wk,
                                         int rank, float* scores, void* ws, cudaStream_t st);
size_t scores_from_means_ws(const Dims& s, int estimator, int rank);

sparsp_status_t launch_block_scores(const Dims& s, int estimator, const void* q, const void* k,
                                    const float* wq, const float* wk, int rank, float* scores,
                                    void* ws, cudaStream_t st);
size_t block_scores_ws(const Dims& s, int estimator, int rank);

sparsp_status_t launch_select(const Dims& s, const float* scores, float top_p, int k_floor,
                              int32_t* row_ptr, int32_t* col_idx, void* ws, int32_t* d_status,
                              cudaStream_t st);
size_t select_ws(const Dims& s);
constexpr int64_t kSelectNoAllocMaxRows = 65536;
sparsp_status_t launch_select_noalloc(const Dims& s, const float* scores, float top_p, int k_floor,
                                      int32_t* row_ptr, int32_t* col_idx, int32_t* d_status,
                                      cudaStream_t st);

sparsp_status_t launch_kv_demand(const Dims& s, int P, const int32_t* row_ptr,
                                 const int32_t* col_idx, const int32_t* owner, uint32_t* bitmap, int32_t* dem_ptr,
                                 int32_t* dem_idx, const void* k, const void* v, void* kg,
                                 void* vg, int64_t cap, uint64_t* bytes, int32_t* d_status,
                                 cudaStream_t st);
sparsp_status_t launch_kv_gather(const Dims& s, int P, const int32_t* dem_ptr, const int32_t* dem_idx,
                                 const void* k, const void* v, void* kg, void* vg, int64_t cap, int32_t* d_status,
                                 cudaStream_t st);
// the same gather from raster k, v [B, N, H, d]
sparsp_status_t launch_kv_gather_raster(const Dims& s, int P, const int32_t* dem_ptr, const int32_t* dem_idx,
                                        const void* k, const void* v, void* kg, void* vg, int64_t cap,
                                        int32_t* d_status, cudaStream_t st);

size_t placement_ws(const Dims& s);
sparsp_status_t launch_placement(const Dims& s, const int32_t* row_ptr, const int32_t* col_idx, int P,
                                 int32_t* owner, void* ws, int32_t* d_status, cudaStream_t st);

sparsp_status_t launch_balance(const Dims& s, const int32_t* row_ptr, int P, int max_moves,
                               int32_t* head_rank, int64_t* loads, int32_t* moves, cudaStream_t st);
size_t augment_ws(const Dims& s, int P);
sparsp_status_t launch_augment(const Dims& s, int P, const float* scores, const int32_t* row_ptr,
                               const int32_t* col_idx, const int32_t* head_rank, int32_t* out_ptr,
                               int32_t* out_idx, int64_t cap, int64_t* added, void* ws, int32_t* d_status,
                               cudaStream_t st);
constexpr int kBalanceMaxHeads = 2048;

size_t predictor_ws(const Dims& s, int rank);
sparsp_status_t launch_predictor_fit(const Dims& s, int rank, const float* qm, const float* km, float* wq,
                                     float* wk, float lr, float* loss, float* gwq, float* gwk, void* ws,
                                     cudaStream_t st);

size_t lpt_ws(const Dims& s);
// cmax: the largest item cost the flat order distinguishes (0 = nb).
sparsp_status_t launch_lpt(const Dims& s, const int32_t* row_ptr, bool flat, int32_t* items,
                           int32_t* counter, void* ws, cudaStream_t st, int cmax = 0);
// The CSR row offsets of the query-block pairs of 64-token blocks (pair p of
// head bh = blocks 2p and 2p+1): pair_ptr [B*H*ceil(nb/2) + 1].
sparsp_status_t launch_pair_ptr(const Dims& s, const int32_t* row_ptr, int32_t* pair_ptr, cudaStream_t st);

// Exclusive scan in place of n+1 int32 entries: a[0..n) counts -> offsets,
// a[n] = total. `base` (may be null) is added to every output.
sparsp_status_t launch_scan_counts(int32_t* a, int64_t n, cudaStream_t st);

sparsp_status_t launch_csr_transpose(const Dims& s, const int32_t* row_ptr, const int32_t* col_idx,
                                     int32_t* col_ptr, int32_t* row_idx, int32_t* d_status,
                                     cudaStream_t st);

// Attention forward variants. `items` is the work order, `counter` a zeroed
// int32 that persistent CTAs pull from.
sparsp_status_t launch_attn_fwd_f32(const Dims& s, const float* q, const float* k, const float* v,
                                    const int32_t* row_ptr, const int32_t* col_idx, float scale,
                                    float* o, float* lse, const int32_t* items, int32_t* counter,
                                    uint64_t* prof, int32_t* d_status, cudaStream_t st);
sparsp_status_t launch_attn_fwd_mma(const Dims& s, const __nv_bfloat16* q, const __nv_bfloat16* k,
                                    const __nv_bfloat16* v, const int32_t* row_ptr,
                                    const int32_t* col_idx, float scale, __nv_bfloat16* o,
                                    float* lse, const int32_t* items, int32_t* counter,
                                    uint64_t* prof, int32_t* d_status, cudaStream_t st);
bool attn_fwd_tc_supported(const Dims& s);
// Work items per head of the tcgen05 forward kernel: nb, or ceil(nb/2) pairs of
// query blocks with 64-token blocks. `items` must then order the pair items
// (b*H + h)*ceil(nb/2) + p (launch_pair_ptr + launch_lpt over the pairs).
int attn_fwd_tc_items_per_head(const Dims& s);
sparsp_status_t launch_attn_fwd_tc(const Dims& s, const __nv_bfloat16* q, const __nv_bfloat16* k,
                                   const __nv_bfloat16* v, const int32_t* row_ptr,
                                   const int32_t* col_idx, float scale, __nv_bfloat16* o,
                                   float* lse, bool raster, bool in_raster, const int32_t* items,
                                   int32_t* counter, uint64_t* prof, int32_t* d_status, cudaStream_t st);

// Attention backward pieces.
// D = rowsum(dO * O) per block-order row (o in raster order when o_raster)
sparsp_status_t launch_bwd_rowdot(const Dims& s, const __nv_bfloat16* o, const __nv_bfloat16* dout,
                                  float* delta, const float* lse, float* lse2, bool o_raster,
                                  cudaStream_t st);
// tcgen05 backward (bf16, Bt = d = 128). mode 0: dQ over the CSR rows;
// mode 1: dK, mode 2: dV, mode 3: dK (out) and dV (out2) over the transposed
// CSR. `lse2` = LSE * log2(e).
// Work items per head of the tcgen05 backward: nb, or ceil(nb/2) pairs of
// 64-token blocks (pair p = blocks 2p and 2p+1 of a CSR row / CSC column list).
int attn_bwd_tc_items_per_head(const Dims& s);
bool attn_bwd_tc_supported(const Dims& s);
sparsp_status_t launch_attn_bwd_tc(const Dims& s, int mode, const __nv_bfloat16* q,
                                   const __nv_bfloat16* k, const __nv_bfloat16* v,
                                   const __nv_bfloat16* dout, const float* lse2,
                                   const float* delta, const int32_t* ptr, const int32_t* idx,
                                   float scale, __nv_bfloat16* out, __nv_bfloat16* out2,
                                   const int32_t* items, int32_t* counter, uint64_t* prof, int32_t* d_status,
                                   bool raster, cudaStream_t st);
sparsp_status_t launch_attn_bwd_dq(const Dims& s, const __nv_bfloat16* q, const __nv_bfloat16* k,
                                   const __nv_bfloat16* v, const __nv_bfloat16* dout,
                                   const float* lse, const float* delta, const int32_t* row_ptr,
                                   const int32_t* col_idx, float scale, __nv_bfloat16* dq,
                                   const int32_t* items, int32_t* counter, uint64_t* prof,
                                   int32_t* d_status, cudaStream_t st);
sparsp_status_t launch_attn_bwd_dkdv(const Dims& s, const __nv_bfloat16* q,
                                     const __nv_bfloat16* k, const __nv_bfloat16* v,
                                     const __nv_bfloat16* dout, const float* lse,
                                     const float* delta, const int32_t* col_ptr,
                                     const int32_t* row_idx, float scale, __nv_bfloat16* dk,
                                     __nv_bfloat16* dv, const int32_t* items, int32_t* counter,
                                     uint64_t* prof, int32_t* d_status, cudaStream_t st);

}  // namespace sparsp
