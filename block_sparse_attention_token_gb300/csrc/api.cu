// extern "C" entry points of libsparsp: argument validation (before any CUDA
// call, so host errors leave outputs untouched) and dispatch to launchers.
#include <math.h>

#include "common.cuh"

using namespace sparsp;

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Validates the shape and fills Dims. Accepts d in {64,128}, Bt in {64,128},
// nb <= kMaxBlocks, B*H <= 65535.
sparsp_status_t check_shape(const sparsp_shape_t* sh, Dims* s) {
  if (sh == nullptr) return SPARSP_ERR_INVALID_ARG;
  if (sh->B <= 0 || sh->H <= 0 || sh->T <= 0 || sh->Y <= 0 || sh->X <= 0 || sh->d <= 0 ||
      sh->ta <= 0 || sh->tb <= 0 || sh->tc <= 0)
    return SPARSP_ERR_SHAPE;
  if (sh->dtype != SPARSP_F32 && sh->dtype != SPARSP_BF16) return SPARSP_ERR_UNSUPPORTED;
  if (sh->T % sh->ta || sh->Y % sh->tb || sh->X % sh->tc) return SPARSP_ERR_SHAPE;
  if (sh->d != 64 && sh->d != 128) return SPARSP_ERR_UNSUPPORTED;
  const int64_t Bt = (int64_t)sh->ta * sh->tb * sh->tc;
  if (Bt != 64 && Bt != 128) return SPARSP_ERR_UNSUPPORTED;
  const int64_t nT = sh->T / sh->ta, nY = sh->Y / sh->tb, nX = sh->X / sh->tc;
  const int64_t nb = nT * nY * nX;
  if (nb > kMaxBlocks) return SPARSP_ERR_UNSUPPORTED;
  if ((int64_t)sh->B * sh->H > 65535) return SPARSP_ERR_UNSUPPORTED;
  // int32 CSR offsets must hold B*H*nb*nb entries
  if ((int64_t)sh->B * sh->H * nb * nb > INT32_MAX) return SPARSP_ERR_UNSUPPORTED;
  s->B = sh->B; s->H = sh->H; s->T = sh->T; s->Y = sh->Y; s->X = sh->X; s->d = sh->d;
  s->ta = sh->ta; s->tb = sh->tb; s->tc = sh->tc; s->dtype = sh->dtype;
  s->N = (int64_t)sh->T * sh->Y * sh->X;
  s->Bt = (int)Bt;
  s->nb = (int)nb;
  s->nT = (int)nT; s->nY = (int)nY; s->nX = (int)nX;
  s->elem = sh->dtype == SPARSP_F32 ? 4 : 2;
  return SPARSP_OK;
}

#define CHECK_PTR(p)                                   \
  do {                                                 \
    if ((p) == nullptr) return SPARSP_ERR_INVALID_ARG; \
    if (!aligned16(p)) return SPARSP_ERR_ALIGN;        \
  } while (0)

#define CHECK_OPT_PTR(p)                                        \
  do {                                                          \
    if ((p) != nullptr && !aligned16(p)) return SPARSP_ERR_ALIGN; \
  } while (0)

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Every attention option bit; a call ignores the ones that do not concern it.
constexpr uint32_t kKnownFlags = SPARSP_SCHED_FLAT | SPARSP_KERNEL_PORTABLE | SPARSP_BWD_SPLIT_KV |
                                 SPARSP_OUT_RASTER | SPARSP_IN_RASTER | SPARSP_GRID_CAP_MASK;

// Attention workspace layout: items, counter(s), then backward extras.
struct AttnWs {
  int32_t* items;      // [rows]
  int32_t* counter;    // [4]
  int32_t* hist;       // [B*H*(2nb+1)] flat-order scratch
  int32_t* pair_ptr;   // [B*H*ceil(nb/2)+1] row offsets of query-block pairs (64-token blocks)
  // backward only
  int32_t* col_ptr;    // [rows+1]
  int32_t* row_idx;    // [B*H*nb*nb]
  int32_t* items2;     // [rows] order over CSC columns
  float* delta;        // [B*H*N]
  float* lse2;         // [B*H*N] LSE * log2(e)
  size_t bytes;
};

AttnWs attn_ws_layout(const Dims& s, bool backward, void* base) {
  AttnWs w{};
  uint8_t* p = (uint8_t*)base;
  size_t off = 0;
  auto take = [&](size_t n) {
    uint8_t* r = p ? p + off : nullptr;
    off += align256(n);
    return r;
  };
  const size_t rows = (size_t)s.rows();
  w.items = (int32_t*)take(rows * 4);
  w.counter = (int32_t*)take(16);
  w.hist = (int32_t*)take(lpt_ws(s));
  w.pair_ptr = (int32_t*)take(((size_t)s.B * s.H * ((s.nb + 1) / 2) + 1) * 4);
  if (backward) {
    w.col_ptr = (int32_t*)take((rows + 1) * 4);
    w.row_idx = (int32_t*)take(rows * (size_t)s.nb * 4);
    w.items2 = (int32_t*)take(rows * 4);
    w.delta = (float*)take((size_t)s.B * s.H * s.N * 4);
    w.lse2 = (float*)take((size_t)s.B * s.H * s.N * 4);
  }
  w.bytes = off;
  return w;
}

}  // namespace

extern "C" {

const char* sparsp_status_string(int32_t st) {
  switch (st) {
    case SPARSP_OK: return "SPARSP_OK";
    case SPARSP_ERR_INVALID_ARG: return "SPARSP_ERR_INVALID_ARG";
    case SPARSP_ERR_UNSUPPORTED: return "SPARSP_ERR_UNSUPPORTED";
    case SPARSP_ERR_SHAPE: return "SPARSP_ERR_SHAPE";
    case SPARSP_ERR_ALIGN: return "SPARSP_ERR_ALIGN";
    case SPARSP_ERR_WORKSPACE: return "SPARSP_ERR_WORKSPACE";
    case SPARSP_ERR_CAPACITY: return "SPARSP_ERR_CAPACITY";
    case SPARSP_ERR_DATA: return "SPARSP_ERR_DATA";
    case SPARSP_ERR_CUDA: return "SPARSP_ERR_CUDA";
    case SPARSP_ERR_TIMEOUT: return "SPARSP_ERR_TIMEOUT";
    default: return "SPARSP_ERR_UNKNOWN";
  }
}

int32_t sparsp_version(void) { return SPARSP_VERSION; }

int32_t sparsp_device_sm_count(void) { return device_sm_count(); }

sparsp_status_t sparsp_reorder(const sparsp_shape_t* shape, const void* in, void* out,
                               int32_t inverse, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  CHECK_PTR(in);
  CHECK_PTR(out);
  const size_t bytes = (size_t)s.B * s.H * s.N * s.d * s.elem;
  const uint8_t* a = (const uint8_t*)in;
  const uint8_t* b = (const uint8_t*)out;
  if (a < b + bytes && b < a + bytes) return SPARSP_ERR_INVALID_ARG;   // overlap
  return launch_reorder(s, in, out, inverse != 0, (cudaStream_t)stream);
}

sparsp_status_t sparsp_reorder_pool(const sparsp_shape_t* shape, const void* in, void* out,
                                    float* means, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  CHECK_PTR(in);
  CHECK_OPT_PTR(out);
  CHECK_PTR(means);
  const size_t bytes = (size_t)s.B * s.H * s.N * s.d * s.elem;
  const uint8_t* a = (const uint8_t*)in;
  const uint8_t* b = (const uint8_t*)out;
  if (b != nullptr && a < b + bytes && b < a + bytes) return SPARSP_ERR_INVALID_ARG;   // overlap
  return launch_reorder(s, in, out, false, (cudaStream_t)stream, means);
}

size_t sparsp_block_scores_pooled_workspace_size(const sparsp_shape_t* shape, int32_t estimator,
                                                 int32_t rank) {
  Dims s;
  if (check_shape(shape, &s) != SPARSP_OK) return 0;
  if (estimator == SPARSP_EST_LOWRANK && (rank < 1 || rank > 64)) return 0;
  return scores_from_means_ws(s, estimator, rank);
}

sparsp_status_t sparsp_block_scores_pooled(const sparsp_shape_t* shape, int32_t estimator,
                                           const float* qmeans, const float* kmeans,
                                           const float* wq, const float* wk, int32_t rank,
                                           float* scores, void* ws, size_t ws_bytes,
                                           sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (estimator != SPARSP_EST_MEAN && estimator != SPARSP_EST_LOWRANK)
    return SPARSP_ERR_INVALID_ARG;
  CHECK_PTR(qmeans);
  CHECK_PTR(kmeans);
  CHECK_PTR(scores);
  if (estimator == SPARSP_EST_LOWRANK) {
    if (rank < 1 || rank > 64) return SPARSP_ERR_UNSUPPORTED;
    CHECK_PTR(wq);
    CHECK_PTR(wk);
    CHECK_PTR(ws);
    if (ws_bytes < scores_from_means_ws(s, estimator, rank)) return SPARSP_ERR_WORKSPACE;
  }
  return launch_scores_from_means(s, estimator, qmeans, kmeans, wq, wk, rank, scores, ws,
                                  (cudaStream_t)stream);
}

size_t sparsp_block_scores_workspace_size(const sparsp_shape_t* shape, int32_t estimator,
                                          int32_t rank) {
  Dims s;
  if (check_shape(shape, &s) != SPARSP_OK) return 0;
  if (estimator == SPARSP_EST_LOWRANK && (rank < 1 || rank > 64)) return 0;
  return block_scores_ws(s, estimator, rank);
}

sparsp_status_t sparsp_block_scores(const sparsp_shape_t* shape, int32_t estimator,
                                    const void* q, const void* k, const float* wq,
                                    const float* wk, int32_t rank, float* scores, void* ws,
                                    size_t ws_bytes, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (estimator != SPARSP_EST_MEAN && estimator != SPARSP_EST_LOWRANK)
    return SPARSP_ERR_INVALID_ARG;
  CHECK_PTR(q);
  CHECK_PTR(k);
  CHECK_PTR(scores);
  CHECK_PTR(ws);
  if (estimator == SPARSP_EST_LOWRANK) {
    if (rank < 1 || rank > 64) return SPARSP_ERR_UNSUPPORTED;
    CHECK_PTR(wq);
    CHECK_PTR(wk);
  }
  if (ws_bytes < block_scores_ws(s, estimator, rank)) return SPARSP_ERR_WORKSPACE;
  return launch_block_scores(s, estimator, q, k, wq, wk, rank, scores, ws, (cudaStream_t)stream);
}

size_t sparsp_select_workspace_size(const sparsp_shape_t* shape) {
  Dims s;
  if (check_shape(shape, &s) != SPARSP_OK) return 0;
  return select_ws(s);
}

sparsp_status_t sparsp_select(const sparsp_shape_t* shape, const float* scores, float top_p,
                              int32_t k_floor, int32_t* row_ptr, int32_t* col_idx, void* ws,
                              size_t ws_bytes, int32_t* d_status, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (isnan(top_p)) return SPARSP_ERR_INVALID_ARG;
  if (k_floor < 0) return SPARSP_ERR_INVALID_ARG;
  CHECK_PTR(scores);
  CHECK_PTR(row_ptr);
  CHECK_PTR(col_idx);
  CHECK_PTR(ws);
  CHECK_OPT_PTR(d_status);
  if (ws_bytes < select_ws(s)) return SPARSP_ERR_WORKSPACE;
  return launch_select(s, scores, top_p, k_floor, row_ptr, col_idx, ws, d_status,
                       (cudaStream_t)stream);
}

sparsp_status_t sparsp_select_noalloc(const sparsp_shape_t* shape, const float* scores, float top_p,
                                      int32_t k_floor, int32_t* row_ptr, int32_t* col_idx,
                                      int32_t* d_status, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (isnan(top_p)) return SPARSP_ERR_INVALID_ARG;
  if (k_floor < 0) return SPARSP_ERR_INVALID_ARG;
  CHECK_PTR(scores);
  CHECK_PTR(row_ptr);
  CHECK_PTR(col_idx);
  CHECK_OPT_PTR(d_status);
  if (s.rows() > kSelectNoAllocMaxRows) return SPARSP_ERR_WORKSPACE;
  return launch_select_noalloc(s, scores, top_p, k_floor, row_ptr, col_idx, d_status,
                               (cudaStream_t)stream);
}

sparsp_status_t sparsp_kv_demand(const sparsp_shape_t* shape, int32_t P, const int32_t* row_ptr,
                                 const int32_t* col_idx, const int32_t* owner, uint32_t* bitmap,
                                 int32_t* dem_ptr, int32_t* dem_idx, const void* k, const void* v,
                                 void* kg, void* vg, int64_t gather_cap_blocks, uint64_t* bytes,
                                 int32_t* d_status, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (P < 1 || P > s.nb) return SPARSP_ERR_SHAPE;
  if ((int64_t)s.B * s.H * P * s.nb > INT32_MAX) return SPARSP_ERR_UNSUPPORTED;   // int32 list offsets
  CHECK_PTR(row_ptr);
  CHECK_PTR(col_idx);
  CHECK_OPT_PTR(owner);
  CHECK_PTR(bitmap);
  CHECK_PTR(dem_ptr);
  CHECK_PTR(dem_idx);
  CHECK_PTR(bytes);
  CHECK_OPT_PTR(d_status);
  if ((kg == nullptr) != (vg == nullptr)) return SPARSP_ERR_INVALID_ARG;
  if (kg != nullptr) {
    CHECK_PTR(kg);
    CHECK_PTR(vg);
    CHECK_PTR(k);
    CHECK_PTR(v);
    if (gather_cap_blocks < 0) return SPARSP_ERR_INVALID_ARG;
  }
  return launch_kv_demand(s, P, row_ptr, col_idx, owner, bitmap, dem_ptr, dem_idx, k, v, kg, vg,
                          gather_cap_blocks, bytes, d_status, (cudaStream_t)stream);
}

sparsp_status_t sparsp_kv_gather(const sparsp_shape_t* shape, int32_t P, const int32_t* dem_ptr,
                                 const int32_t* dem_idx, const void* k, const void* v, void* kg, void* vg,
                                 int64_t gather_cap_blocks, int32_t* d_status, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (P < 1 || P > s.nb) return SPARSP_ERR_SHAPE;
  if ((int64_t)s.B * s.H * P * s.nb > INT32_MAX) return SPARSP_ERR_UNSUPPORTED;   // int32 list offsets
  CHECK_PTR(dem_ptr);
  CHECK_PTR(dem_idx);
  CHECK_PTR(k);
  CHECK_PTR(v);
  CHECK_PTR(kg);
  CHECK_PTR(vg);
  CHECK_OPT_PTR(d_status);
  if (gather_cap_blocks < 0) return SPARSP_ERR_INVALID_ARG;
  return launch_kv_gather(s, P, dem_ptr, dem_idx, k, v, kg, vg, gather_cap_blocks, d_status,
                          (cudaStream_t)stream);
}

sparsp_status_t sparsp_kv_gather_raster(const sparsp_shape_t* shape, int32_t P, const int32_t* dem_ptr,
                                        const int32_t* dem_idx, const void* k, const void* v, void* kg, void* vg,
                                        int64_t gather_cap_blocks, int32_t* d_status, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (P < 1 || P > s.nb) return SPARSP_ERR_SHAPE;
  if ((int64_t)s.B * s.H * P * s.nb > INT32_MAX) return SPARSP_ERR_UNSUPPORTED;   // int32 list offsets
  CHECK_PTR(dem_ptr);
  CHECK_PTR(dem_idx);
  CHECK_PTR(k);
  CHECK_PTR(v);
  CHECK_PTR(kg);
  CHECK_PTR(vg);
  CHECK_OPT_PTR(d_status);
  if (gather_cap_blocks < 0) return SPARSP_ERR_INVALID_ARG;
  return launch_kv_gather_raster(s, P, dem_ptr, dem_idx, k, v, kg, vg, gather_cap_blocks, d_status,
                                 (cudaStream_t)stream);
}

size_t sparsp_placement_workspace_size(const sparsp_shape_t* shape) {
  Dims s;
  if (check_shape(shape, &s) != SPARSP_OK || s.nb > kMaxBlocksNext) return 0;
  return placement_ws(s);
}

sparsp_status_t sparsp_placement(const sparsp_shape_t* shape, int32_t P, const int32_t* row_ptr,
                                 const int32_t* col_idx, int32_t* owner, void* ws, size_t ws_bytes,
                                 int32_t* d_status, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (s.nb > kMaxBlocksNext) return SPARSP_ERR_UNSUPPORTED;
  if (P < 1 || P > s.nb) return SPARSP_ERR_SHAPE;
  CHECK_PTR(row_ptr);
  CHECK_PTR(col_idx);
  CHECK_PTR(owner);
  CHECK_PTR(ws);
  CHECK_OPT_PTR(d_status);
  if (ws_bytes < placement_ws(s)) return SPARSP_ERR_WORKSPACE;
  return launch_placement(s, row_ptr, col_idx, P, owner, ws, d_status, (cudaStream_t)stream);
}

sparsp_status_t sparsp_balance_heads(const sparsp_shape_t* shape, int32_t P, int32_t max_migrations,
                                     const int32_t* row_ptr, int32_t* head_rank, int64_t* loads,
                                     int32_t* migrations, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (s.H > kBalanceMaxHeads) return SPARSP_ERR_UNSUPPORTED;
  if (P < 1 || P > s.H) return SPARSP_ERR_SHAPE;
  if (max_migrations < 0) return SPARSP_ERR_INVALID_ARG;
  CHECK_PTR(row_ptr);
  CHECK_PTR(head_rank);
  CHECK_PTR(loads);
  CHECK_OPT_PTR(migrations);
  return launch_balance(s, row_ptr, P, max_migrations, head_rank, loads, migrations, (cudaStream_t)stream);
}

size_t sparsp_augment_workspace_size(const sparsp_shape_t* shape, int32_t P) {
  Dims s;
  if (check_shape(shape, &s) != SPARSP_OK || P < 1 || s.nb > kMaxBlocksNext) return 0;
  return augment_ws(s, P);
}

sparsp_status_t sparsp_augment(const sparsp_shape_t* shape, int32_t P, const float* scores,
                               const int32_t* row_ptr, const int32_t* col_idx, const int32_t* head_rank,
                               int32_t* row_ptr_out, int32_t* col_idx_out, int64_t col_cap, int64_t* added,
                               void* ws, size_t ws_bytes, int32_t* d_status, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (s.H > kBalanceMaxHeads || s.nb > kMaxBlocksNext) return SPARSP_ERR_UNSUPPORTED;
  if (P < 1 || P > s.H) return SPARSP_ERR_SHAPE;
  if (col_cap < 0) return SPARSP_ERR_INVALID_ARG;
  CHECK_PTR(scores);
  CHECK_PTR(row_ptr);
  CHECK_PTR(col_idx);
  CHECK_PTR(head_rank);
  CHECK_PTR(row_ptr_out);
  CHECK_PTR(col_idx_out);
  CHECK_OPT_PTR(added);
  CHECK_PTR(ws);
  CHECK_OPT_PTR(d_status);
  if (ws_bytes < augment_ws(s, P)) return SPARSP_ERR_WORKSPACE;
  return launch_augment(s, P, scores, row_ptr, col_idx, head_rank, row_ptr_out, col_idx_out, col_cap, added, ws,
                        d_status, (cudaStream_t)stream);
}

size_t sparsp_predictor_workspace_size(const sparsp_shape_t* shape, int32_t rank) {
  Dims s;
  if (check_shape(shape, &s) != SPARSP_OK || rank < 1 || rank > 64) return 0;
  return predictor_ws(s, rank);
}

sparsp_status_t sparsp_predictor_fit(const sparsp_shape_t* shape, int32_t rank, const float* qmeans,
                                     const float* kmeans, float* wq, float* wk, float lr, float* loss,
                                     float* gwq, float* gwk, void* ws, size_t ws_bytes,
                                     sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (rank < 1 || rank > 64) return SPARSP_ERR_UNSUPPORTED;
  if (!isfinite(lr)) return SPARSP_ERR_INVALID_ARG;
  CHECK_PTR(qmeans);
  CHECK_PTR(kmeans);
  CHECK_PTR(wq);
  CHECK_PTR(wk);
  CHECK_OPT_PTR(loss);
  CHECK_OPT_PTR(gwq);
  CHECK_OPT_PTR(gwk);
  CHECK_PTR(ws);
  if (ws_bytes < predictor_ws(s, rank)) return SPARSP_ERR_WORKSPACE;
  return launch_predictor_fit(s, rank, qmeans, kmeans, wq, wk, lr, loss, gwq, gwk, ws, (cudaStream_t)stream);
}

size_t sparsp_lpt_workspace_size(const sparsp_shape_t* shape) {
  Dims s;
  if (check_shape(shape, &s) != SPARSP_OK) return 0;
  return lpt_ws(s);
}

sparsp_status_t sparsp_lpt_schedule(const sparsp_shape_t* shape, const int32_t* row_ptr,
                                    uint32_t flags, int32_t* items, void* ws, size_t ws_bytes,
                                    sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (flags & ~kKnownFlags) return SPARSP_ERR_INVALID_ARG;
  CHECK_PTR(row_ptr);
  CHECK_PTR(items);
  const bool flat = (flags & SPARSP_SCHED_FLAT) != 0;
  if (flat) {
    CHECK_PTR(ws);
    if (ws_bytes < lpt_ws(s)) return SPARSP_ERR_WORKSPACE;
  }
  return launch_lpt(s, row_ptr, flat, items, nullptr, ws, (cudaStream_t)stream);
}

sparsp_status_t sparsp_csr_transpose(const sparsp_shape_t* shape, const int32_t* row_ptr,
                                     const int32_t* col_idx, int32_t* col_ptr, int32_t* row_idx,
                                     int32_t* d_status, sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  CHECK_PTR(row_ptr);
  CHECK_PTR(col_idx);
  CHECK_PTR(col_ptr);
  CHECK_PTR(row_idx);
  CHECK_OPT_PTR(d_status);
  return launch_csr_transpose(s, row_ptr, col_idx, col_ptr, row_idx, d_status,
                              (cudaStream_t)stream);
}

size_t sparsp_attn_workspace_size(const sparsp_shape_t* shape, int32_t backward) {
  Dims s;
  if (check_shape(shape, &s) != SPARSP_OK) return 0;
  return attn_ws_layout(s, backward != 0, nullptr).bytes;
}

sparsp_status_t sparsp_attn_fwd(const sparsp_shape_t* shape, const void* q, const void* k,
                                const void* v, const int32_t* row_ptr, const int32_t* col_idx,
                                float scale, void* o, float* lse, void* ws, size_t ws_bytes,
                                uint32_t flags, uint64_t* prof, int32_t* d_status,
                                sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (isnan(scale) || isinf(scale)) return SPARSP_ERR_INVALID_ARG;
  if (flags & ~kKnownFlags) return SPARSP_ERR_INVALID_ARG;
  s.max_ctas = (int)((flags & SPARSP_GRID_CAP_MASK) >> SPARSP_GRID_CAP_SHIFT);
  CHECK_PTR(q);
  CHECK_PTR(k);
  CHECK_PTR(v);
  CHECK_PTR(row_ptr);
  CHECK_PTR(col_idx);
  CHECK_PTR(o);
  CHECK_PTR(lse);
  CHECK_PTR(ws);
  CHECK_OPT_PTR(prof);
  CHECK_OPT_PTR(d_status);
  AttnWs w = attn_ws_layout(s, false, ws);
  if (ws_bytes < w.bytes) return SPARSP_ERR_WORKSPACE;
  if (scale <= 0.f) scale = 1.0f / sqrtf((float)s.d);
  const bool tc = s.dtype != SPARSP_F32 && !(flags & SPARSP_KERNEL_PORTABLE) && attn_fwd_tc_supported(s);
  const bool raster = (flags & SPARSP_OUT_RASTER) != 0;
  const bool in_raster = (flags & SPARSP_IN_RASTER) != 0;
  if ((raster || in_raster) && !tc) return SPARSP_ERR_UNSUPPORTED;   // only the tcgen05 kernel reads or writes raster rows
  cudaStream_t st = (cudaStream_t)stream;
  const bool flat = (flags & SPARSP_SCHED_FLAT) != 0;
  if (tc && attn_fwd_tc_items_per_head(s) != s.nb) {
    // the tcgen05 kernel's items are pairs of query blocks: order the pairs,
    // each costing the sum of its two rows
    r = launch_pair_ptr(s, row_ptr, w.pair_ptr, st);
    if (r != SPARSP_OK) return r;
    Dims sp = s;
    sp.nb = attn_fwd_tc_items_per_head(s);
    r = launch_lpt(sp, w.pair_ptr, flat, w.items, w.counter, w.hist, st, 2 * s.nb);
  } else {
    r = launch_lpt(s, row_ptr, flat, w.items, w.counter, w.hist, st);
  }
  if (r != SPARSP_OK) return r;
  if (s.dtype == SPARSP_F32)
    return launch_attn_fwd_f32(s, (const float*)q, (const float*)k, (const float*)v, row_ptr,
                               col_idx, scale, (float*)o, lse, w.items, w.counter, prof, d_status,
                               st);
  if (tc)
    return launch_attn_fwd_tc(s, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                              (const __nv_bfloat16*)v, row_ptr, col_idx, scale,
                              (__nv_bfloat16*)o, lse, raster, in_raster, w.items, w.counter, prof, d_status, st);
  return launch_attn_fwd_mma(s, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                             (const __nv_bfloat16*)v, row_ptr, col_idx, scale, (__nv_bfloat16*)o,
                             lse, w.items, w.counter, prof, d_status, st);
}

sparsp_status_t sparsp_attn_bwd(const sparsp_shape_t* shape, const void* q, const void* k,
                                const void* v, const void* o, const float* lse, const void* dout,
                                const int32_t* row_ptr, const int32_t* col_idx, float scale,
                                void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                                uint32_t flags, uint64_t* prof, int32_t* d_status,
                                sparsp_stream_t stream) {
  Dims s;
  sparsp_status_t r = check_shape(shape, &s);
  if (r != SPARSP_OK) return r;
  if (s.dtype != SPARSP_BF16) return SPARSP_ERR_UNSUPPORTED;
  if (isnan(scale) || isinf(scale)) return SPARSP_ERR_INVALID_ARG;
  if (flags & ~kKnownFlags) return SPARSP_ERR_INVALID_ARG;
  if (flags & SPARSP_IN_RASTER) return SPARSP_ERR_UNSUPPORTED;   // the backward reads block-ordered tiles
  s.max_ctas = (int)((flags & SPARSP_GRID_CAP_MASK) >> SPARSP_GRID_CAP_SHIFT);
  CHECK_PTR(q);
  CHECK_PTR(k);
  CHECK_PTR(v);
  CHECK_PTR(o);
  CHECK_PTR(lse);
  CHECK_PTR(dout);
  CHECK_PTR(row_ptr);
  CHECK_PTR(col_idx);
  CHECK_PTR(dq);
  CHECK_PTR(dk);
  CHECK_PTR(dv);
  CHECK_PTR(ws);
  CHECK_OPT_PTR(prof);
  CHECK_OPT_PTR(d_status);
  AttnWs w = attn_ws_layout(s, true, ws);
  if (ws_bytes < w.bytes) return SPARSP_ERR_WORKSPACE;
  if (scale <= 0.f) scale = 1.0f / sqrtf((float)s.d);
  cudaStream_t st = (cudaStream_t)stream;
  const bool flat = (flags & SPARSP_SCHED_FLAT) != 0;
  typedef const __nv_bfloat16* cb;
  const bool tc = !(flags & SPARSP_KERNEL_PORTABLE) && attn_bwd_tc_supported(s);
  const bool raster = (flags & SPARSP_OUT_RASTER) != 0;
  if (raster && !tc) return SPARSP_ERR_UNSUPPORTED;   // only the tcgen05 kernels write raster rows
  r = launch_bwd_rowdot(s, (cb)o, (cb)dout, w.delta, lse, tc ? w.lse2 : nullptr, raster, st);
  if (r != SPARSP_OK) return r;
  r = launch_csr_transpose(s, row_ptr, col_idx, w.col_ptr, w.row_idx, d_status, st);
  if (r != SPARSP_OK) return r;
  // the tcgen05 kernels' items with 64-token blocks are pairs of blocks, each
  // costing the sum of its two lists (CSR rows for dQ, CSC columns for dK/dV)
  const bool pairs = tc && attn_bwd_tc_items_per_head(s) != s.nb;
  Dims sp = s;
  sp.nb = pairs ? attn_bwd_tc_items_per_head(s) : s.nb;
  if (pairs) {
    r = launch_pair_ptr(s, row_ptr, w.pair_ptr, st);
    if (r != SPARSP_OK) return r;
    r = launch_lpt(sp, w.pair_ptr, flat, w.items, w.counter, w.hist, st, 2 * s.nb);
  } else {
    r = launch_lpt(s, row_ptr, flat, w.items, w.counter, w.hist, st);
  }
  if (r != SPARSP_OK) return r;
  if (tc) {
    r = launch_attn_bwd_tc(s, 0, (cb)q, (cb)k, (cb)v, (cb)dout, w.lse2, w.delta, row_ptr, col_idx, scale,
                           (__nv_bfloat16*)dq, nullptr, w.items, w.counter, prof, d_status, raster, st);
    if (r != SPARSP_OK) return r;
    if (pairs) {   // pair_ptr is free again: the dQ kernel reads only its item list
      r = launch_pair_ptr(s, w.col_ptr, w.pair_ptr, st);
      if (r != SPARSP_OK) return r;
      r = launch_lpt(sp, w.pair_ptr, flat, w.items2, w.counter + 1, w.hist, st, 2 * s.nb);
    } else {
      r = launch_lpt(s, w.col_ptr, flat, w.items2, w.counter + 1, w.hist, st);
    }
    if (r != SPARSP_OK) return r;
    if (!(flags & SPARSP_BWD_SPLIT_KV))
      return launch_attn_bwd_tc(s, 3, (cb)q, (cb)k, (cb)v, (cb)dout, w.lse2, w.delta, w.col_ptr, w.row_idx,
                                scale, (__nv_bfloat16*)dk, (__nv_bfloat16*)dv, w.items2, w.counter + 1, prof,
                                d_status, raster, st);
    r = launch_attn_bwd_tc(s, 1, (cb)q, (cb)k, (cb)v, (cb)dout, w.lse2, w.delta, w.col_ptr, w.row_idx,
                           scale, (__nv_bfloat16*)dk, nullptr, w.items2, w.counter + 1, prof, d_status, raster,
                           st);
    if (r != SPARSP_OK) return r;
    if (cudaMemsetAsync(w.counter + 2, 0, sizeof(int32_t), st) != cudaSuccess) return SPARSP_ERR_CUDA;
    return launch_attn_bwd_tc(s, 2, (cb)q, (cb)k, (cb)v, (cb)dout, w.lse2, w.delta, w.col_ptr, w.row_idx,
                              scale, (__nv_bfloat16*)dv, nullptr, w.items2, w.counter + 2, prof, d_status, raster,
                              st);
  }
  r = launch_attn_bwd_dq(s, (cb)q, (cb)k, (cb)v, (cb)dout, lse, w.delta, row_ptr, col_idx, scale,
                         (__nv_bfloat16*)dq, w.items, w.counter, prof, d_status, st);
  if (r != SPARSP_OK) return r;
  r = launch_lpt(s, w.col_ptr, flat, w.items2, w.counter + 1, w.hist, st);
  if (r != SPARSP_OK) return r;
  return launch_attn_bwd_dkdv(s, (cb)q, (cb)k, (cb)v, (cb)dout, lse, w.delta, w.col_ptr,
                              w.row_idx, scale, (__nv_bfloat16*)dk, (__nv_bfloat16*)dv, w.items2,
                              w.counter + 1, prof, d_status, st);
}

}  // extern "C"
