/*
 * sparsp.h - C ABI of libsparsp: dynamic, per-head block-sparse attention over
 * 3D video-DiT token sequences, on one NVIDIA GB300 (sm_103a).
 *
 * The method these calls implement is described, in words only, on the pages:
 *
 *  - "mlsift.com tag listing" (sequence parallelism), the Top-p video sparse-
 *    attention entry, abstract: video-aware block organisation, Top-p routing
 *    with a Top-k safety floor, per-head uneven workloads and their stragglers,
 *    and sparse attention compared against FlashAttention;
 *  - "Dynamic Sparsity in Large-Scale Video DiT Training", "How DSV works":
 *    the per-head rank-16 low-rank Q.K predictor, sparse attention computed
 *    only on the selected critical pairs without materialising the full score
 *    matrix, query grouping, and rebalancing of lopsided per-head work;
 *  - "SparSP: Exploiting Communication Sparsity for Sequence-Parallel Video
 *    DiTs", abstract: demand-directed KV routing, which the KV-demand call
 *    computes for P virtual query partitions on one GPU.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every call returns a sparsp_status_t. Errors that the host can see
 *    (null or misaligned pointers, bad shapes, small workspace) are returned
 *    synchronously BEFORE any work is enqueued; outputs are then untouched.
 *  - Errors that depend on device data (an out-of-range block index, a
 *    non-finite score, a full gather buffer, a wait that timed out) are
 *    written to the optional device word *d_status (int32, caller-owned,
 *    zero-initialised by the caller). The first error wins; the offending
 *    work item is skipped. Kernels never trap and never spin without a bound.
 *  - The caller owns every buffer. The library never allocates device
 *    memory, never synchronises, and keeps no state apart from a per-device
 *    cache of the SM count and of the tensor-map encoder entry point.
 *    Calls are thread-safe.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *  - All device pointers must be 16-byte aligned; tensors are contiguous.
 *  - Shapes: d in {64, 128}; Bt = ta*tb*tc in {64, 128}; nb = N/Bt <= 4096
 *    (524,288 tokens in 128-token blocks) and B*H*nb*nb < 2^31 (int32 CSR
 *    offsets); dtype SPARSP_F32 or SPARSP_BF16 (bf16 inputs accumulate in
 *    fp32). sparsp_placement and sparsp_augment take nb <= 1024 and return
 *    SPARSP_ERR_UNSUPPORTED beyond.
 *
 * Layouts
 * -------
 *  raster     [B, N, H, d]: N = T*Y*X tokens, t slowest, x fastest.
 *  blocked    [B, H, N, d]: row j*Bt + o is token o of tile j. Tiles are
 *             (ta, tb, tc) boxes numbered ((bt*nY)+by)*nX+bx (x tile fastest);
 *             inside a tile tokens are numbered ((it*tb)+iy)*tc+ix.
 *  scores     [B, H, nb, nb] float32; row (b, h, i) = query block i.
 *  CSR        row_ptr [B*H*nb + 1] int32 (row r = (b*H + h)*nb + i),
 *             col_idx [nnz] int32, key-block indices ascending within a row.
 *  LSE        [B, H, N] float32, natural log.
 */
#ifndef SPARSP_H
#define SPARSP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPARSP_VERSION 1

#if defined(__GNUC__)
#define SPARSP_API __attribute__((visibility("default")))
#else
#define SPARSP_API
#endif

/* A cudaStream_t, declared without CUDA headers. */
typedef struct CUstream_st* sparsp_stream_t;

typedef enum {
  SPARSP_OK = 0,
  SPARSP_ERR_INVALID_ARG = 1, /* null pointer, NaN parameter, bad enum      */
  SPARSP_ERR_UNSUPPORTED = 2, /* dtype, d, Bt, nb or rank outside support    */
  SPARSP_ERR_SHAPE = 3,       /* grid not divisible by tile, P out of range  */
  SPARSP_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned            */
  SPARSP_ERR_WORKSPACE = 5,   /* ws_bytes smaller than the size call returns */
  SPARSP_ERR_CAPACITY = 6,    /* device: gather buffer too small             */
  SPARSP_ERR_DATA = 7,        /* device: bad index, bad CSR row, NaN score   */
  SPARSP_ERR_CUDA = 8,        /* a CUDA launch or runtime call failed        */
  SPARSP_ERR_TIMEOUT = 9      /* device: a bounded wait expired              */
} sparsp_status_t;

typedef enum { SPARSP_F32 = 0, SPARSP_BF16 = 1 } sparsp_dtype_t;

typedef enum { SPARSP_EST_MEAN = 0, SPARSP_EST_LOWRANK = 1 } sparsp_estimator_t;

/* Attention options (bit flags). sparsp_lpt_schedule, sparsp_attn_fwd and
 * sparsp_attn_bwd accept any of them (each ignores the ones that do not
 * concern it) and return SPARSP_ERR_INVALID_ARG for any other bit. */
enum {
  /* Order work items purely by row cost across all heads instead of
   * head-grouped longest-first (see sparsp_lpt_schedule). */
  SPARSP_SCHED_FLAT = 1u << 0,
  /* Use the portable mma.sync kernel even where the tcgen05 kernel applies. */
  SPARSP_KERNEL_PORTABLE = 1u << 1,
  /* Backward on tcgen05: dK and dV by two kernels (each recomputing S^T)
   * instead of one kernel that accumulates both. */
  SPARSP_BWD_SPLIT_KV = 1u << 2,
  /* Forward: write O in raster order [B, N, H, d] (the layout of the inverse
   * sparsp_reorder) instead of block order; LSE stays [B, H, N] in block
   * order. Only the tcgen05 kernel (bf16 on sm_103a, Bt and d in {64, 128},
   * nb <= 1024 when Bt = 64 and d = 128, without SPARSP_KERNEL_PORTABLE) does
   * this; elsewhere the call returns SPARSP_ERR_UNSUPPORTED before enqueuing
   * anything.
   * Backward: o is read in raster order (as the forward wrote it with this
   * option) and dq, dk, dv are written in raster order; q, k, v, dout and lse
   * stay in block order (the kernels read them as tiles). Only the tcgen05
   * backward (the tcgen05 forward's shapes) does this; elsewhere
   * SPARSP_ERR_UNSUPPORTED. */
  SPARSP_OUT_RASTER = 1u << 3,
  /* Forward: q, k, v are read in raster order [B, N, H, d] (the layout
   * sparsp_reorder takes) instead of block order: the kernel loads each block
   * as one 5-D tile (column, head, x, y, frame), so no reorder pass is needed.
   * Results are bitwise those of the block-ordered inputs. Only the tcgen05
   * kernel does this; elsewhere SPARSP_ERR_UNSUPPORTED. */
  SPARSP_IN_RASTER = 1u << 4
};
/* Attention kernels: at most n persistent CTAs (1 <= n <= 4095) instead of
 * one per SM (times the kernel's occupancy), encoded in bits 16..27 of the
 * options as SPARSP_GRID_CAP(n); 0 there means no cap. Work items are pulled
 * from one counter in a fixed order and each item's sums run in a fixed
 * order inside its CTA, so the results are bitwise the same for every grid;
 * the cap exists to show that, and to leave SMs to other work. */
#define SPARSP_GRID_CAP_SHIFT 16
#define SPARSP_GRID_CAP_MASK (0xFFFu << SPARSP_GRID_CAP_SHIFT)
#define SPARSP_GRID_CAP(n) (((uint32_t)(n) << SPARSP_GRID_CAP_SHIFT) & SPARSP_GRID_CAP_MASK)

/* Per-SM profile slots that attention kernels accumulate into (see prof). */
#define SPARSP_PROF_SLOTS 1024

typedef struct {
  int32_t B, H;        /* batch, heads                         */
  int32_t T, Y, X;     /* latent grid (frames, height, width)  */
  int32_t d;           /* head dimension                       */
  int32_t ta, tb, tc;  /* tile (video-aware block) shape       */
  int32_t dtype;       /* sparsp_dtype_t of Q, K, V, O, dO...  */
} sparsp_shape_t;

/* Name of a status code (static string). */
SPARSP_API const char* sparsp_status_string(int32_t status);

/* SPARSP_VERSION of the loaded library. */
SPARSP_API int32_t sparsp_version(void);

/*
 * Step 1 - video-aware block organisation ("mlsift.com tag listing",
 * Top-p video sparse-attention entry, abstract).
 * inverse == 0: in = raster [B,N,H,d] -> out = blocked [B,H,N,d].
 * inverse != 0: in = blocked -> out = raster. A pure permutation (bit-exact).
 * in and out must not overlap. Element type = shape->dtype.
 */
SPARSP_API sparsp_status_t sparsp_reorder(const sparsp_shape_t* shape, const void* in, void* out,
                               int32_t inverse, sparsp_stream_t stream);

/*
 * Step 2 - cheap block-score estimation.
 * SPARSP_EST_MEAN:    S[b,h,i,j] = mean_{q in block i}(q) . mean_{k in block j}(k)
 *                     (plain pooled dot product, no 1/sqrt(d)).
 * SPARSP_EST_LOWRANK: S[b,h,i,j] = (mean_i(q) Wq[h]) . (mean_j(k) Wk[h]), which by
 *                     bilinearity equals the block-pair mean of the token-level
 *                     (q Wq)(k Wk)^T of the per-head low-rank predictor ("Dynamic
 *                     Sparsity in Large-Scale Video DiT Training", "How DSV works").
 * q, k: blocked [B,H,N,d] of shape->dtype. wq, wk: float32 [H, d, rank], NULL for
 * MEAN; rank in [1, 64]. scores: float32 [B,H,nb,nb]. Means and projections are
 * accumulated in float32 in a fixed order. ws: scratch of at least
 * sparsp_block_scores_workspace_size() bytes.
 */
SPARSP_API size_t sparsp_block_scores_workspace_size(const sparsp_shape_t* shape, int32_t estimator,
                                          int32_t rank);
SPARSP_API sparsp_status_t sparsp_block_scores(const sparsp_shape_t* shape, int32_t estimator,
                                    const void* q, const void* k, const float* wq,
                                    const float* wk, int32_t rank, float* scores, void* ws,
                                    size_t ws_bytes, sparsp_stream_t stream);

/*
 * Steps 1 + 2 fused ("Dynamic Sparsity in Large-Scale Video DiT Training",
 * "How DSV works" and "Why it works": critical-KV estimation fused into the
 * passes that already touch Q and K). sparsp_reorder_pool is the forward
 * sparsp_reorder of one tensor that also writes the fp32 mean of every tile
 * to `means` [B, H, nb, d] from the same read (a fixed summation order), so
 * the block scores need no second pass over Q and K. out may be NULL: the
 * means alone (for attention that reads raster input itself,
 * SPARSP_IN_RASTER).
 * sparsp_block_scores_pooled: the scores of sparsp_block_scores from those
 * means (estimator MEAN: q_mean . k_mean; LOWRANK: (q_mean Wq)(k_mean Wk)^T);
 * ws is used by LOWRANK only (sparsp_block_scores_pooled_workspace_size(),
 * 0 for MEAN, when ws may be NULL).
 */
SPARSP_API sparsp_status_t sparsp_reorder_pool(const sparsp_shape_t* shape, const void* in, void* out,
                                               float* means, sparsp_stream_t stream);
SPARSP_API size_t sparsp_block_scores_pooled_workspace_size(const sparsp_shape_t* shape,
                                                            int32_t estimator, int32_t rank);
SPARSP_API sparsp_status_t sparsp_block_scores_pooled(const sparsp_shape_t* shape, int32_t estimator,
                                                      const float* qmeans, const float* kmeans,
                                                      const float* wq, const float* wk, int32_t rank,
                                                      float* scores, void* ws, size_t ws_bytes,
                                                      sparsp_stream_t stream);

/*
 * Step 3 - Top-p routing with a Top-k safety floor ("mlsift.com tag listing",
 * Top-p video sparse-attention entry, abstract), per (b, h, i) row of scores:
 *   e_j = expf(S_j - max_j S_j) in float32; Z and prefix sums in float64;
 *   blocks ordered by (S_j descending, j ascending);
 *   m_p = smallest m whose prefix mass >= top_p * Z (0 if top_p <= 0, nb if >= 1);
 *   m = min(nb, max(m_p, k_floor, 1)); the first m blocks, stored ascending.
 * row_ptr [B*H*nb+1] and col_idx (capacity B*H*nb*nb) are written; nnz =
 * row_ptr[B*H*nb] stays on the device. A row holding a NaN or infinite score
 * sets SPARSP_ERR_DATA and is written as an empty row.
 * ws: at least sparsp_select_workspace_size() bytes.
 */
SPARSP_API size_t sparsp_select_workspace_size(const sparsp_shape_t* shape);
SPARSP_API sparsp_status_t sparsp_select(const sparsp_shape_t* shape, const float* scores, float top_p,
                              int32_t k_floor, int32_t* row_ptr, int32_t* col_idx, void* ws,
                              size_t ws_bytes, int32_t* d_status, sparsp_stream_t stream);

/*
 * sparsp_select without a workspace argument, for callers that cannot
 * allocate device memory when they call: for example an inference-engine
 * plug-in whose enqueue step must not allocate, or a service that reserves all
 * of its device memory at start-up and forbids allocation afterwards. The
 * pages have no counterpart to this call; it is an interface convenience.
 * Same arguments, results and errors as sparsp_select, except that its scratch
 * (one 64-bit key per row) lives in a fixed array inside the library:
 *  - at most SPARSP_SELECT_NOALLOC_MAX_ROWS rows (B*H*nb); a larger shape
 *    returns SPARSP_ERR_WORKSPACE before any work is enqueued;
 *  - the array costs 512 KB of device memory on every device that loads the
 *    library, held until the process exits;
 *  - every call asks the CUDA runtime for the array's address in the device
 *    and context current at the call (a query that allocates nothing; the
 *    address is not cached, so a device reset or another context on the same
 *    device is safe); the first call on a device may also load the library's
 *    device code there, so make that first call before any stream capture;
 *  - every call shares the one array, which keeps the last call's contents
 *    (nothing in it needs to start at zero): calls whose work can overlap on
 *    the GPU (different streams, or different host threads) race and must be
 *    serialised by the caller.
 * It never calls cudaMalloc, cudaFree or any allocating routine.
 */
#define SPARSP_SELECT_NOALLOC_MAX_ROWS 65536
SPARSP_API sparsp_status_t sparsp_select_noalloc(const sparsp_shape_t* shape, const float* scores,
                                                 float top_p, int32_t k_floor, int32_t* row_ptr,
                                                 int32_t* col_idx, int32_t* d_status,
                                                 sparsp_stream_t stream);

/*
 * Step 4 - KV demand of P virtual query partitions, the one-GPU analogue of
 * Demand-Directed KV Routing ("SparSP: Exploiting Communication Sparsity for
 * Sequence-Parallel Video DiTs", abstract). With owner == NULL partition r owns
 * the contiguous query blocks [floor(r*nb/P), floor((r+1)*nb/P)); otherwise
 * owner is int32 [B, nb] (device) and partition r of batch element b owns the
 * blocks i with owner[b*nb + i] == r, in every head (an entry outside [0, P)
 * sets SPARSP_ERR_DATA and its block belongs to no partition). A partition's
 * demand is the union of the CSR rows of the blocks it owns.
 *   bitmap  uint32 [B,H,P,ceil(nb/32)]: bit j of partition (b,h,r).
 *   dem_ptr int32 [B*H*P+1], dem_idx int32 (capacity B*H*P*nb): ascending set bits.
 *   kg, vg  [gather_cap_blocks, Bt, d] of shape->dtype: slot s holds the K/V tile
 *           of dem_idx[s] of its head, copied from blocked k, v. kg == vg == NULL
 *           skips the gather (k, v may then be NULL). Slots beyond
 *           gather_cap_blocks are not written and set SPARSP_ERR_CAPACITY.
 *   bytes   uint64 [4]: demanded, all (every partition receives all KV),
 *           remote_demanded, remote_all (blocks the partition does not own);
 *           K and V both counted.
 */
SPARSP_API sparsp_status_t sparsp_kv_demand(const sparsp_shape_t* shape, int32_t P, const int32_t* row_ptr,
                                 const int32_t* col_idx, const int32_t* owner, uint32_t* bitmap,
                                 int32_t* dem_ptr, int32_t* dem_idx, const void* k, const void* v,
                                 void* kg, void* vg, int64_t gather_cap_blocks, uint64_t* bytes,
                                 int32_t* d_status, sparsp_stream_t stream);

/*
 * Step 4, the copy alone: the gather of sparsp_kv_demand from the lists a
 * previous sparsp_kv_demand call (with kg == vg == NULL) wrote on the same
 * stream, or with the stream ordering made by the caller. Same P, dem_ptr,
 * dem_idx, k, v, kg, vg, gather_cap_blocks and results as the gather there:
 * slot s < min(dem_ptr[B*H*P], gather_cap_blocks) of kg / vg receives the K / V
 * tile dem_idx[s] of its partition's head; a total above gather_cap_blocks
 * sets SPARSP_ERR_CAPACITY. A total above B*H*P*nb or an index outside
 * [0, nb) sets SPARSP_ERR_DATA and is not used. It only reads k, v, dem_ptr and dem_idx and uses no
 * shared memory, so it can run on a second stream beside the attention kernel
 * (which holds almost all of each SM's shared memory); the lists need a small
 * amount of it and do not fit there.
 */
SPARSP_API sparsp_status_t sparsp_kv_gather(const sparsp_shape_t* shape, int32_t P, const int32_t* dem_ptr,
                                 const int32_t* dem_idx, const void* k, const void* v, void* kg, void* vg,
                                 int64_t gather_cap_blocks, int32_t* d_status, sparsp_stream_t stream);
/* The same gather with k and v in raster order [B, N, H, d] (the layout
 * sparsp_reorder takes): every tile's token rows are read at their raster
 * addresses; the results equal those of sparsp_kv_gather on the reordered
 * tensors. */
SPARSP_API sparsp_status_t sparsp_kv_gather_raster(const sparsp_shape_t* shape, int32_t P, const int32_t* dem_ptr,
                                        const int32_t* dem_idx, const void* k, const void* v, void* kg, void* vg,
                                        int64_t gather_cap_blocks, int32_t* d_status, sparsp_stream_t stream);

/*
 * Step 4b - Dependency-Aware Placement ("SparSP: Exploiting Communication
 * Sparsity for Sequence-Parallel Video DiTs", abstract: sequence blocks placed
 * on ranks according to the sparse attention pattern), over the P virtual
 * partitions of sparsp_kv_demand. The pages give no algorithm; this is a
 * deterministic greedy on the co-selection affinity of batch element b,
 *   A[i][j] = #heads whose row i holds j + #heads whose row j holds i (i != j),
 * with one assignment per batch element shared by all heads and the partition
 * sizes of the contiguous split (floor((r+1)*nb/P) - floor(r*nb/P)):
 *   blocks in order of sum_j A[i][j] descending (ties: lower i); each goes to
 *   the partition with spare capacity whose placed blocks have the largest
 *   summed affinity to it (ties: more spare capacity, then lower r).
 * owner: int32 [B, nb] (device), written with the partition of every block, to
 * pass to sparsp_kv_demand. ws: at least sparsp_placement_workspace_size()
 * bytes (B*nb*nb int32 affinity counts). A column index outside [0, nb) or a
 * row with more than nb entries sets SPARSP_ERR_DATA and is skipped.
 */
SPARSP_API size_t sparsp_placement_workspace_size(const sparsp_shape_t* shape);
SPARSP_API sparsp_status_t sparsp_placement(const sparsp_shape_t* shape, int32_t P, const int32_t* row_ptr,
                                 const int32_t* col_idx, int32_t* owner, void* ws, size_t ws_bytes,
                                 int32_t* d_status, sparsp_stream_t stream);

/*
 * Virtual-rank load balancing ("mlsift.com tag listing", Top-p video
 * sparse-attention entry, abstract: Runtime Load Balancing migrates a few heavy
 * heads to shorten the critical path of sequence-parallel ranks), modelled on
 * one GPU over P virtual ranks per batch element. The cost of head (b, h) is
 * its number of selected block pairs (row_ptr[(bh+1)*nb] - row_ptr[bh*nb]).
 * Start: the contiguous split, rank r holding heads [floor(r*H/P),
 * floor((r+1)*H/P)). Then at most max_migrations times: c = most loaded rank,
 * t = least loaded (ties: lower rank); among c's heads take the one whose move
 * to t gives the smallest max(L_c - cost, L_t + cost) (ties: lower head); move
 * it only if that is below L_c, else stop.
 *   head_rank  int32 [B, H] (device): the rank of every head.
 *   loads      int64 [B, 2, P] (device): rank loads before and after.
 *   migrations int32 [B] (device) or NULL: moves made.
 * Requires 1 <= P <= H <= 2048 (else SPARSP_ERR_SHAPE / SPARSP_ERR_UNSUPPORTED)
 * and max_migrations >= 0.
 */
SPARSP_API sparsp_status_t sparsp_balance_heads(const sparsp_shape_t* shape, int32_t P, int32_t max_migrations,
                                     const int32_t* row_ptr, int32_t* head_rank, int64_t* loads,
                                     int32_t* migrations, sparsp_stream_t stream);

/*
 * Slack-Aware Sparse Augmentation (same entry: slack on non-critical ranks is
 * filled with additional high-value blocks). With heads on ranks (head_rank
 * [B, H], e.g. from sparsp_balance_heads) and rank loads L_r, the critical load
 * is L* = max_r L_r. Rank r adds min(L* - L_r, #candidates) blocks: its heads'
 * unselected blocks (h, i, j) of largest value v = fl32(e_j / Z), where
 * e_j = exp(S_j - max_j S) in fp32 and Z = sum_j e_j in fp64 over the row of
 * scores (the mass selection assigns the block), ties by row (b*H + h)*nb + i
 * then j ascending. The critical load is unchanged.
 *   scores       float32 [B, H, nb, nb]: the block scores selection ran on.
 *   row_ptr/col_idx: the selection's CSR (ascending rows).
 *   row_ptr_out  int32 [B*H*nb + 1], col_idx_out int32 [col_cap]: the augmented
 *                CSR, ascending rows (col_cap >= B*H*nb*nb always suffices;
 *                overflow sets SPARSP_ERR_CAPACITY).
 *   added        int64 [B, P] (device) or NULL: blocks added per rank.
 *   ws           at least sparsp_augment_workspace_size() bytes.
 * A head_rank entry outside [0, P), a bad CSR row or a non-finite score row
 * sets SPARSP_ERR_DATA; such rows are copied without additions. Requires
 * 1 <= P <= H <= 2048.
 */
SPARSP_API size_t sparsp_augment_workspace_size(const sparsp_shape_t* shape, int32_t P);
SPARSP_API sparsp_status_t sparsp_augment(const sparsp_shape_t* shape, int32_t P, const float* scores,
                               const int32_t* row_ptr, const int32_t* col_idx, const int32_t* head_rank,
                               int32_t* row_ptr_out, int32_t* col_idx_out, int64_t col_cap, int64_t* added,
                               void* ws, size_t ws_bytes, int32_t* d_status, sparsp_stream_t stream);

/*
 * Predictor fitting ("Dynamic Sparsity in Large-Scale Video DiT Training",
 * "How DSV works / The idea": the two per-head matrices are trained so that
 * their product approximates the real query-key scores, beside the main graph
 * and during the forward pass). The pages call the loss magnitude-preserving
 * without defining it; here it is the mean squared error between the
 * predictor's block scores and the real block scores of the same pooled
 * means, per head:
 *   E[b,h,i,j] = (qm[b,h,i] Wq[h]) . (km[b,h,j] Wk[h]) - qm[b,h,i] . km[b,h,j]
 *   loss[h]    = sum_{b,i,j} E^2 / (B nb^2)
 * qmeans, kmeans: float32 [B,H,nb,d] tile means (sparsp_reorder_pool).
 * wq, wk: float32 [H,d,rank], 1 <= rank <= 64. Writes loss [H], gwq and gwk
 * [H,d,rank] = dloss/dWq, dloss/dWk (each may be NULL), all at the current
 * weights; then, if lr != 0, takes the step W -= lr * dloss/dW in place.
 * ws: at least sparsp_predictor_workspace_size() bytes. Sums run in a fixed
 * order: results are bitwise reproducible.
 */
SPARSP_API size_t sparsp_predictor_workspace_size(const sparsp_shape_t* shape, int32_t rank);
SPARSP_API sparsp_status_t sparsp_predictor_fit(const sparsp_shape_t* shape, int32_t rank, const float* qmeans,
                                     const float* kmeans, float* wq, float* wk, float lr, float* loss,
                                     float* gwq, float* gwk, void* ws, size_t ws_bytes,
                                     sparsp_stream_t stream);

/*
 * Step 5c - longest-first work order for the attention kernels (the per-head
 * straggler problem of the "mlsift.com tag listing" entry; the lopsided
 * per-head work of "Dynamic Sparsity in Large-Scale Video DiT Training",
 * "How DSV works"). Item (b,h,i) is encoded (b*H + h)*nb + i; its cost is its
 * CSR row length.
 *   flags & SPARSP_SCHED_FLAT == 0: heads by total cost descending (ties: lower
 *     head first), rows inside a head by cost descending (ties: lower i first).
 *   flags & SPARSP_SCHED_FLAT: all items by cost descending, ties by item.
 * items: int32 [B*H*nb]. ws: at least sparsp_lpt_workspace_size() bytes.
 */
SPARSP_API size_t sparsp_lpt_workspace_size(const sparsp_shape_t* shape);
SPARSP_API sparsp_status_t sparsp_lpt_schedule(const sparsp_shape_t* shape, const int32_t* row_ptr,
                                    uint32_t flags, int32_t* items, void* ws, size_t ws_bytes,
                                    sparsp_stream_t stream);

/*
 * Step 5a - block-sparse attention forward over the CSR ("Dynamic Sparsity in
 * Large-Scale Video DiT Training", "How DSV works": attention only on the
 * selected pairs, never materialising the full score matrix). For each query
 * token q of block i, over the key tokens of the blocks in row (b,h,i):
 *   O_q = sum_k softmax_k(scale q.k) v_k,   LSE_q = ln sum_k exp(scale q.k).
 * q, k, v, o: blocked [B,H,N,d] (o raster [B,N,H,d] with SPARSP_OUT_RASTER);
 * lse: float32 [B,H,N]. scale <= 0 means
 * 1/sqrt(d). An empty row gives O = 0, LSE = -inf. A row with an index outside
 * [0, nb) or more than nb entries sets SPARSP_ERR_DATA and is skipped. Rows
 * must list distinct blocks (sparsp_select writes them ascending); the
 * 64-token-block tcgen05 kernel also reports a repeated index as
 * SPARSP_ERR_DATA and skips that row, the other kernels do not check.
 * bf16 on sm_103a runs the tcgen05/TMEM/TMA kernel (Bt and d in {64, 128},
 * except 64-token blocks with d = 128 beyond 1,024 blocks;
 * with 64-token blocks each work item is a pair of neighbouring query blocks
 * over the union of their rows, so that every MMA has 128 query rows and 128
 * key columns); with SPARSP_KERNEL_PORTABLE an mma.sync kernel; float32 runs
 * an fp32 FFMA kernel. Work items are pulled longest-first by persistent CTAs.
 * prof: NULL or uint64 [SPARSP_PROF_SLOTS], caller-zeroed; receives per-SM busy
 * nanoseconds (index = SM id).
 * ws: at least sparsp_attn_workspace_size(shape, 0) bytes.
 */
SPARSP_API size_t sparsp_attn_workspace_size(const sparsp_shape_t* shape, int32_t backward);
SPARSP_API sparsp_status_t sparsp_attn_fwd(const sparsp_shape_t* shape, const void* q, const void* k,
                                const void* v, const int32_t* row_ptr, const int32_t* col_idx,
                                float scale, void* o, float* lse, void* ws, size_t ws_bytes,
                                uint32_t flags, uint64_t* prof, int32_t* d_status,
                                sparsp_stream_t stream);

/*
 * Step 5b - block-sparse attention backward with the selection held fixed.
 * Gradients of sum(dO * O) with O from sparsp_attn_fwd (its o and lse):
 *   D = rowsum(dO * O); P = exp(scale QK^T - LSE) on the selected blocks;
 *   dV = P^T dO; dS = P * (dO V^T - D); dQ = scale dS K; dK = scale dS^T Q.
 * bf16 only. dq, dk, dv: blocked [B,H,N,d] bf16 (raster [B,N,H,d], and o
 * raster too, with SPARSP_OUT_RASTER). dQ is accumulated per query
 * block over its CSR row and dK/dV per key block over the transposed CSR, so
 * the result is deterministic (no atomics on values). On tcgen05 (bf16, Bt
 * and d in {64, 128}, nb <= 1024 when Bt = 64 and d = 128, without
 * SPARSP_KERNEL_PORTABLE) one kernel computes dQ and one both dK and dV (two
 * with SPARSP_BWD_SPLIT_KV), 64-token blocks as pairs of neighbouring blocks
 * over the union of their two lists; other shapes run the portable mma.sync
 * kernels.
 * ws: at least sparsp_attn_workspace_size(shape, 1) bytes.
 */
SPARSP_API sparsp_status_t sparsp_attn_bwd(const sparsp_shape_t* shape, const void* q, const void* k,
                                const void* v, const void* o, const float* lse, const void* dout,
                                const int32_t* row_ptr, const int32_t* col_idx, float scale,
                                void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                                uint32_t flags, uint64_t* prof, int32_t* d_status,
                                sparsp_stream_t stream);

/*
 * Transpose of the per-head CSR (used by the backward): for each key block j
 * of head (b,h), the query blocks that selected it, ascending.
 * col_ptr int32 [B*H*nb+1]; row_idx int32 (capacity = nnz of the CSR).
 * An index outside [0, nb) sets SPARSP_ERR_DATA (the entry is left out); up
 * to 1,024 blocks so does a row that lists a block twice.
 */
SPARSP_API sparsp_status_t sparsp_csr_transpose(const sparsp_shape_t* shape, const int32_t* row_ptr,
                                     const int32_t* col_idx, int32_t* col_ptr, int32_t* row_idx,
                                     int32_t* d_status, sparsp_stream_t stream);

/* Number of SMs of the current device (cached), or -1 on error. */
SPARSP_API int32_t sparsp_device_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSP_H */
