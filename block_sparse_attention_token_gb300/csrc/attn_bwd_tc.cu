// Step 5b, bf16, Bt = 128 and d = 64 or 128 on sm_103a: block-sparse attention backward on
// the tcgen05 tensor cores, as persistent kernels of one template: mode 0 and
// mode 3 by default, modes 0, 1 and 2 when dK and dV are asked for apart.
//
//   mode 0 (dQ): item = query block i, blocks = its CSR row.
//                S = Q_i K_c^T, dP = dO_i V_c^T, dS = P (dP - D), dQ += dS K_c.
//   mode 1 (dK): item = key block j, blocks = the query blocks that selected it.
//                S^T = K_j Q_c^T, dP^T = V_j dO_c^T, dS^T = P^T (dP^T - D), dK += dS^T Q_c.
//   mode 2 (dV): item = key block j, as mode 1.  S^T = K_j Q_c^T, dV += P^T dO_c.
//   mode 3 (dK and dV): modes 1 and 2 in one pass, both accumulators in TMEM
//                (dK [256,256+d), dV [256+d,256+2d)); P^T is written over S^T and
//                dS^T over dP^T. With d = 128 the row tiles K_j, V_j stay in
//                shared memory (no TMEM left for them), so S^T and dP^T take
//                both operands from shared memory and the row tiles are
//                released by an MMA commit after the item's last S^T / dP^T;
//                with d = 64 they fit in TMEM as in the other modes.
// with P = exp2(S * scale*log2e - LSE*log2e) from the forward's LSE (no online
// maximum is needed), D = rowsum(dO * O), and dQ, dK scaled by `scale` at the
// end. Each column block is processed in two halves of 64 columns, double
// buffered in TMEM so that the softmax warps work on one half while the
// tensor pipe computes the next half's S and dP and the previous half's
// accumulate: half buffer b holds S_b [128b, 128b+64) and dP_b
// [128b+64, 128b+128), and the half's bf16 operand X (P or dS) is written over
// the first 32 columns of S_b; the fp32 accumulator is [256,256+d); the item's
// row tiles A1 [384,384+d/2) and A2 [384+d/2,384+d) sit in TMEM as packed bf16, so every
// MMA takes A from TMEM and only B from shared memory (a 128x64x16 MMA with
// both operands in shared memory is bound by shared-memory bandwidth at 62% of
// the tensor rate; with A in TMEM it runs at the full rate). A half buffer is
// free again once the accumulate MMA that read its X has completed. The dQ
// and the dK/dV kernels recompute S (and dP) instead of sharing it so that
// each fits TMEM. Modes 0-2 (and mode 3 with d = 64) are laid out as above;
// mode 3 with d = 128 as described with it. With d = 64 the column tiles are
// half the size and the ring holds 4 of them instead of 2.
// Sums are taken in a fixed order (no atomics), so results are bitwise
// reproducible. The gradient rows go to block order, or straight to their
// raster rows (the layout of the inverse reorder) when asked.
//
// One persistent CTA per SM, 7 warps (the forward kernel's structure):
//   warp 4     producer: pulls items longest-first, validates the block list,
//              TMA-loads the item's two row tiles (A1, A2) once (the softmax
//              warps copy them into TMEM) and, per block,
//              the two column tiles (B1, B2; two 64-column boxes each, 128-byte
//              swizzle) into a 2-stage ring; in modes 1-3 also the block's
//              LSE*log2e and D (512 bytes each) by 1-D bulk copy.
//   warp 5     S issuer: per half, S = A1 B1_h^T and (modes 0, 1, 3)
//              dP = A2 B2_h^T (N = 64), A from TMEM (from shared memory in
//              mode 3), B K-major from shared memory.
//   warp 6     accumulate issuer: per half, ACC += X B3_h (K = 64) with X from
//              TMEM and B3 (the column tile K_c, Q_c or dO_c) MN-major from
//              shared memory; mode 3 issues dV += P^T dO_c and dK += dS^T Q_c.
//   warps 0-3  thread t owns row t (TMEM lane t): copies its rows of A1, A2
//              into TMEM at the start of an item (modes 0-2); per half loads S and dP,
//              computes P and dS in fp32 from them and the statistics, packs
//              the operand to bf16 into X; epilogue ACC -> global, deferred
//              until the next item's row tiles are in TMEM so that its first
//              MMAs overlap the epilogue.
// Every mbarrier wait is bounded (2 s): on expiry the CTA reports
// SPARSP_ERR_TIMEOUT, all roles leave, in-flight copies and MMAs are drained
// with a second bounded wait and TMEM is released.
#include "pairs.cuh"
#include "tc_helpers.cuh"

namespace sparsp {
namespace {

using namespace tc;

constexpr int TR = 128;   // rows of a row or column tile (the MMA's M; one block, or a pair of 64-token blocks)
constexpr int kMaxNS = 4, kNI = 4;
constexpr uint32_t kBox = TR * 64 * 2;        // one 64-column swizzled box of a 128-row tile
constexpr uint32_t kStats = 1024;             // LSE*log2e [128] + D [128] of a column block
constexpr int kThreads = 224;
constexpr int HB = 64;   // columns of a half block
enum Bar {
  A_FULL = 0, A_EMPTY, AT_FULL, C_FULL, C_EMPTY = C_FULL + kMaxNS, SD_FULL = C_EMPTY + kMaxNS,
  X_FULL = SD_FULL + 2,
  X_DONE = X_FULL + 2, ACC_FULL = X_DONE + 2, ACC_EMPTY, I_FULL, I_EMPTY = I_FULL + kNI,
  TEAR = I_EMPTY + kNI, TEAR2, NBAR
};
// Tile geometry, shared-memory layout and TMEM map for head dimension D
// (64 or 128): row and column tiles are 128 x D (D / 64 boxes of 64 columns);
// TMEM holds the two half buffers [0,256), the accumulator(s) from 256
// (mode 3: dK [256, 256+D), dV [256+D, 256+2D)) and, where the row tiles live
// in TMEM, A1 [384, 384+D/2) and A2 [384+D/2, 384+D) as packed bf16.
//
// With 64-token blocks (PAIR) an item is a pair of neighbouring blocks (2p,
// 2p + 1: 128 contiguous rows) processed over the union of their two lists,
// two blocks per column stage (the two halves); each item slot holds the two
// lists as bitmaps and one byte per union block saying which of the two rows
// selected it, so that the row warps mask a half for a row block that did not.
template <int D_, int BTB_>
struct BCfg {
  static constexpr int D = D_, BTB = BTB_;
  static constexpr bool PAIR = BTB == 64;
  static constexpr int NBOX = D / 64;
  static constexpr uint32_t kTile = TR * D * 2;
  static constexpr int kNS = D == 64 ? 4 : 2;   // column-tile stages
  static constexpr uint32_t kColAcc = 256, kColAcc2 = 256 + D;
  static constexpr uint32_t kColA1 = 384, kColA2 = 384 + D / 2;
  static constexpr uint32_t kOffA2 = kTile, kOffStage = 2 * kTile;
  static constexpr uint32_t kStageBytes = 2 * kTile + kStats;   // a multiple of 1024: tiles stay aligned
  static constexpr uint32_t kOffBar = kOffStage + kNS * kStageBytes;
  static constexpr uint32_t kOffRing = kOffBar + 8 * NBAR;   // [kNI] int4: item, stages, bad-list bits
  // pairs: bitmap words of one list (up to 1,024 blocks with d = 128, kMaxBlocks with d = 64)
  static constexpr int MAXW = PAIR ? (D == 64 ? kMaxBlocks / 32 : 32) : 0;
  static constexpr uint32_t kOffBits = kOffRing + 16 * kNI;   // [kNI][2][MAXW]
  static constexpr uint32_t kMaskBytes = 32 * MAXW;           // per slot: one byte per union block (+1)
  static constexpr uint32_t kOffMask = kOffBits + kNI * 2 * MAXW * 4;
  static constexpr uint32_t kOffMisc = kOffMask + kNI * (kMaskBytes + (PAIR ? 16 : 0));
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
  static_assert(kNS <= kMaxNS && kSmemBytes <= 232448u, "shared memory");
};
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;

__device__ __forceinline__ bool wait_raw(uint32_t bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit) return false;
  return true;
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

struct Params {
  const int32_t* ptr;    // CSR row_ptr (mode 0) or CSC col_ptr (modes 1, 2)
  const int32_t* idx;    // CSR col_idx or CSC row_idx
  int64_t N;
  int nb;
  int nbp;               // items per head: nb, or ceil(nb / 2) pairs of 64-token blocks
  int64_t n_items;
  int64_t rows_total;    // B*H*N rows of every tensor
  float sl2;             // scale * log2(e)
  float out_scale;       // scale for dQ and dK, 1 for dV
  const float* lse2;     // LSE * log2(e), [B*H*N]
  const float* delta;    // rowsum(dO * O), [B*H*N]
  __nv_bfloat16* out;
  __nv_bfloat16* out2;   // mode 3: dV (out is dK)
  float out_scale2;      // mode 3: scale for dV
  const int32_t* items;
  int32_t* counter;
  uint64_t* prof;
  int32_t* d_status;
  int raster;            // outputs in raster order at rm.row(bh, block, token); else block order
  RasterMap rm;
};

template <int MODE, int D, int BTB>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap ta1, const __grid_constant__ CUtensorMap ta2,
                   const __grid_constant__ CUtensorMap tb1, const __grid_constant__ CUtensorMap tb2,
                   const Params p) {
  using C = BCfg<D, BTB>;
  constexpr bool PAIR = C::PAIR;
  constexpr bool kHasDP = MODE != 2;
  // the item's row tiles as the A operand in TMEM; mode 3 with d = 128 has no
  // TMEM left beside its two accumulators and reads them from shared memory
  constexpr bool kRowsInTmem = MODE != 3 || D == 64;
  constexpr uint32_t kTile = C::kTile, kStageBytes = C::kStageBytes;
  constexpr int kNS = C::kNS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA1 = base, sA2 = base + C::kOffA2;
  auto stage = [&](uint32_t st) -> uint32_t { return base + C::kOffStage + st * kStageBytes; };
  auto bar = [&](int idx) -> uint32_t { return base + C::kOffBar + 8u * (uint32_t)idx; };
  volatile int4* ring = reinterpret_cast<volatile int4*>(gbase + C::kOffRing);
  uint32_t* bits = reinterpret_cast<uint32_t*>(gbase + C::kOffBits);   // pairs: [kNI][2][MAXW]
  uint8_t* masks = gbase + C::kOffMask;                                 // pairs: [kNI][kMaskBytes + 16]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(gbase + C::kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t t_start = globaltimer_ns();

  if (threadIdx.x == 0) {
    mbar_init(bar(A_FULL), 1);
    mbar_init(bar(A_EMPTY), kRowsInTmem ? 128 : 1);   // else an MMA commit
    mbar_init(bar(AT_FULL), 128);
    for (int s = 0; s < kNS; ++s) {
      mbar_init(bar(C_FULL + s), 1);
      mbar_init(bar(C_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(SD_FULL + b), 1);
      mbar_init(bar(X_FULL + b), 128);
      mbar_init(bar(X_DONE + b), 1);
    }
    mbar_init(bar(ACC_FULL), 1);
    mbar_init(bar(ACC_EMPTY), 128);
    for (int r = 0; r < kNI; ++r) {
      mbar_init(bar(I_FULL + r), 1);
      mbar_init(bar(I_EMPTY + r), 6);
    }
    mbar_init(bar(TEAR), 1);
    mbar_init(bar(TEAR2), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&ta1);
    prefetch_tmap(&ta2);
    prefetch_tmap(&tb1);
    prefetch_tmap(&tb2);
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  const Guard g{abort_flag, p.d_status, kWaitNs};
  const int nb = p.nb, nbp = p.nbp;
  const int words = (nb + 31) >> 5;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    uint32_t it_fill = 0, a_fill = 0, c_fill = 0;
    for (;;) {
      int32_t slot = 0;
      if (lane == 0) slot = atomicAdd(p.counter, 1);
      slot = __shfl_sync(0xffffffffu, slot, 0);
      const int ri = (int)(it_fill % kNI);
      // the slot's bitmaps and masks stay in use until the row warps release it
      if (!wait_warp(bar(I_EMPTY + ri), ((it_fill / kNI) & 1u) ^ 1u, g)) break;
      uint32_t* bmA = bits + ri * 2 * C::MAXW;
      uint32_t* bmB = bmA + C::MAXW;
      int32_t item = -1, len = -2, badbits = 0;
      if (slot < p.n_items) {
        item = p.items[slot];
        if constexpr (PAIR) {
          // the pair's two lists as bitmaps; a bad list counts as empty
          const int64_t bh = item / nbp;
          const int iA = 2 * (item % nbp);
          for (int w = lane; w < 2 * C::MAXW; w += 32) bmA[w] = 0u;
          __syncwarp();
          const bool okA = list_bitmap(p.ptr, p.idx, nb, bh * nb + iA, bmA, words, lane);
          const bool okB = iA + 1 < nb ? list_bitmap(p.ptr, p.idx, nb, bh * nb + iA + 1, bmB, words, lane) : true;
          badbits = (okA ? 0 : 1) | (okB ? 0 : 2);
          if (badbits && lane == 0) report(p.d_status, SPARSP_ERR_DATA);
          const int u = union_count(bmA, bmB, words, lane);
          len = (badbits == 3) ? -1 : (u + 1) / 2;   // stages of two blocks
          union_masks(bmA, bmB, words, u, lane, masks + ri * (C::kMaskBytes + 16));
        } else {
          const int32_t a = p.ptr[item], b = p.ptr[item + 1];
          bool bad = (b < a) || (b - a > nb);
          if (!bad)
            for (int32_t e = a + lane; e < b; e += 32) {
              const int32_t j = p.idx[e];
              if (j < 0 || j >= nb) bad = true;
            }
          bad = __any_sync(0xffffffffu, bad);
          if (bad) {
            if (lane == 0) report(p.d_status, SPARSP_ERR_DATA);
            len = -1;
          } else {
            len = b - a;
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        ring[ri].x = item;
        ring[ri].y = len;
        ring[ri].z = badbits;
        mbar_arrive(bar(I_FULL + ri));
      }
      __syncwarp();
      ++it_fill;
      if (len == -2) break;
      if (len <= 0) continue;
      const int64_t bh = item / nbp;
      const int i0 = PAIR ? 2 * (item % nbp) : item % nb;   // the item's (first) row block
      int32_t ya = (int32_t)(bh * p.N + (int64_t)i0 * BTB);
      if (!dcheck(ya >= 0 && ya < p.rows_total, p.d_status)) ya = 0;
      if (!wait_warp(bar(A_EMPTY), (a_fill & 1u) ^ 1u, g)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(A_FULL), kHasDP ? 2 * kTile : kTile);
#pragma unroll
        for (int h = 0; h < C::NBOX; ++h) {
          tma_load_2d(sA1 + h * kBox, &ta1, bar(A_FULL), 64 * h, ya);
          if (kHasDP) tma_load_2d(sA2 + h * kBox, &ta2, bar(A_FULL), 64 * h, ya);
        }
      }
      ++a_fill;
      const int32_t e0 = PAIR ? 0 : p.ptr[item];
      UnionWalk walk(bmA, bmB, PAIR ? words : 0);
      bool ok = true;
      for (int e = 0; e < len; ++e) {
        // the stage's column block(s): one block, or the next two of the pair's union
        int32_t c1, c2 = 0;
        if constexpr (PAIR) {
          c1 = walk.next();
          c2 = walk.next();
          if (c2 < 0) c2 = c1;   // a lone last block: loaded twice, its second half masked
        } else {
          c1 = p.idx[e0 + e];
        }
        int64_t yc64 = bh * p.N + (int64_t)c1 * BTB, yc64b = bh * p.N + (int64_t)c2 * BTB;
        if (!dcheck(yc64 >= 0 && yc64 + BTB <= p.rows_total && yc64b >= 0 && yc64b + BTB <= p.rows_total,
                    p.d_status))
          yc64 = yc64b = 0;   // flagged; counts kept
        const int32_t yc = (int32_t)yc64, ycb = (int32_t)yc64b;
        const uint32_t st = c_fill % kNS;
        if (!(ok = wait_warp(bar(C_EMPTY + st), ((c_fill / kNS) & 1u) ^ 1u, g))) break;
        if (lane == 0) {
          const uint32_t sb = stage(st);
          mbar_arrive_expect_tx(bar(C_FULL + st), 2 * kTile + (MODE != 0 ? kStats : 0u));
#pragma unroll
          for (int h = 0; h < C::NBOX; ++h) {
            tma_load_2d(sb + h * kBox, &tb1, bar(C_FULL + st), 64 * h, yc);
            tma_load_2d(sb + kTile + h * kBox, &tb2, bar(C_FULL + st), 64 * h, yc);
            if (PAIR) {   // the second block's 64 rows, 8 KB into each box
              tma_load_2d(sb + h * kBox + kBox / 2, &tb1, bar(C_FULL + st), 64 * h, ycb);
              tma_load_2d(sb + kTile + h * kBox + kBox / 2, &tb2, bar(C_FULL + st), 64 * h, ycb);
            }
          }
          if (MODE != 0) {
            if (PAIR) {   // LSE*log2e and D of the two blocks' rows, side by side
              bulk_load(sb + 2 * kTile, p.lse2 + yc64, 256, bar(C_FULL + st));
              bulk_load(sb + 2 * kTile + 256, p.lse2 + yc64b, 256, bar(C_FULL + st));
              bulk_load(sb + 2 * kTile + 512, p.delta + yc64, 256, bar(C_FULL + st));
              bulk_load(sb + 2 * kTile + 768, p.delta + yc64b, 256, bar(C_FULL + st));
            } else {
              bulk_load(sb + 2 * kTile, p.lse2 + yc64, 512, bar(C_FULL + st));
              bulk_load(sb + 2 * kTile + 512, p.delta + yc64, 512, bar(C_FULL + st));
            }
          }
        }
        ++c_fill;
      }
      if (!ok) break;
    }
    if (*abort_flag && lane == 0) {
      if (a_fill) wait_raw(bar(A_FULL), (a_fill - 1) & 1u, kDrainNs);
      for (uint32_t s = 0; s < kNS; ++s)
        if (c_fill > s) wait_raw(bar(C_FULL + s), ((c_fill - 1 - s) / kNS) & 1u, kDrainNs);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ S (and dP) issuer
    constexpr uint32_t idS = idesc_bf16(128, HB, 0, 0);
    uint32_t it_use = 0, a_use = 0, c_use = 0, hg = 0;
    bool issued_any = false;
    for (;;) {
      const int ri = (int)(it_use % kNI);
      if (!wait_warp(bar(I_FULL + ri), (it_use / kNI) & 1u, g)) break;
      const int4 ent = make_int4(ring[ri].x, ring[ri].y, ring[ri].z, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(I_EMPTY + ri));
      ++it_use;
      if (ent.y == -2) break;
      if (ent.y <= 0) continue;
      const int len = ent.y;
      // the item's row tiles: in TMEM, or in shared memory (mode 3 with d = 128)
      if (!wait_warp(bar(kRowsInTmem ? AT_FULL : A_FULL), a_use & 1u, g)) break;
      ++a_use;
      fence_after();
      bool ok = true;
      for (int e = 0; e < len && ok; ++e) {
        const uint32_t st = c_use % kNS;
        if (!(ok = wait_warp(bar(C_FULL + st), (c_use / kNS) & 1u, g))) break;
        const uint32_t sb = stage(st);
        for (int h = 0; h < 2; ++h) {
          const uint32_t b = hg & 1u;
          // buffer b holds X of half hg - 2 until that half's accumulate MMA has completed
          if (!(ok = wait_warp(bar(X_DONE + b), ((hg >> 1) & 1u) ^ 1u, g))) break;
          fence_after();
          // rows [64h, 64h+64) of the column tile: 64 rows x 128 B = 8 KB into each box
          const uint32_t rows_h = (uint32_t)h * (HB * 128u);
          if constexpr (!kRowsInTmem) {
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (uint32_t)(kk >> 2) * kBox + (uint32_t)(kk & 3) * 32u;
                mma_ss(tmem + 128u * b, smem_desc(sA1 + off, 16, 1024, kSwizzle128B),
                       smem_desc(sb + rows_h + off, 16, 1024, kSwizzle128B), idS, kk > 0 ? 1u : 0u);
              }
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (uint32_t)(kk >> 2) * kBox + (uint32_t)(kk & 3) * 32u;
                mma_ss(tmem + 128u * b + HB, smem_desc(sA2 + off, 16, 1024, kSwizzle128B),
                       smem_desc(sb + kTile + rows_h + off, 16, 1024, kSwizzle128B), idS, kk > 0 ? 1u : 0u);
              }
              commit(bar(SD_FULL + b));
            }
          } else if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (uint32_t)(kk >> 2) * kBox + (uint32_t)(kk & 3) * 32u;
              mma_ts(tmem + 128u * b, tmem + C::kColA1 + (uint32_t)kk * 8u,
                     smem_desc(sb + rows_h + off, 16, 1024, kSwizzle128B), idS, kk > 0 ? 1u : 0u);
            }
            if (kHasDP) {
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (uint32_t)(kk >> 2) * kBox + (uint32_t)(kk & 3) * 32u;
                mma_ts(tmem + 128u * b + HB, tmem + C::kColA2 + (uint32_t)kk * 8u,
                       smem_desc(sb + kTile + rows_h + off, 16, 1024, kSwizzle128B), idS, kk > 0 ? 1u : 0u);
              }
            }
            commit(bar(SD_FULL + b));
          }
          __syncwarp();
          ++hg;
          issued_any = true;
        }
        ++c_use;
      }
      if (!ok) break;
      if (!kRowsInTmem) {   // the row tiles are free once this item's S^T and dP^T are done
        if (elect_one()) commit(bar(A_EMPTY));
        __syncwarp();
      }
    }
    if (*abort_flag && issued_any) {
      if (elect_one()) commit(bar(TEAR));
      __syncwarp();
      wait_raw(bar(TEAR), 0, kDrainNs);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ accumulate issuer
    constexpr uint32_t idAcc = idesc_bf16(128, D, 0, 1);
    // the column tile the accumulator multiplies: K_c / Q_c (B1) or dO_c (B2)
    constexpr uint32_t kB3 = MODE == 2 ? kTile : 0u;
    uint32_t it_use = 0, c_use = 0, hg = 0, acc_items = 0;
    bool issued_any = false;
    for (;;) {
      const int ri = (int)(it_use % kNI);
      if (!wait_warp(bar(I_FULL + ri), (it_use / kNI) & 1u, g)) break;
      const int4 ent = make_int4(ring[ri].x, ring[ri].y, ring[ri].z, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(I_EMPTY + ri));
      ++it_use;
      if (ent.y == -2) break;
      if (ent.y <= 0) continue;
      const int len = ent.y;
      bool ok = true;
      for (int e = 0; e < len && ok; ++e) {
        const uint32_t st = c_use % kNS;
        const uint32_t b3 = stage(st) + kB3;
        for (int h = 0; h < 2; ++h) {
          const uint32_t b = hg & 1u;
          if (!(ok = wait_warp(bar(X_FULL + b), (hg >> 1) & 1u, g))) break;
          if (e == 0 && h == 0 && !(ok = wait_warp(bar(ACC_EMPTY), (acc_items & 1u) ^ 1u, g))) break;
          fence_after();
          if (elect_one()) {
            // K = the half's 64 rows of the column tile: k-steps 4h .. 4h+3 of 16 rows (2 KB each)
            const uint32_t acc = (e > 0 || h > 0) ? 1u : 0u;
            if (MODE == 3) {
              const uint32_t bq = stage(st), bdo = stage(st) + kTile;
#pragma unroll
              for (int kk = 0; kk < HB / 16; ++kk)   // dV += P^T dO_c
                mma_ts(tmem + C::kColAcc2, tmem + 128u * b + (uint32_t)kk * 8u,
                       smem_desc(bdo + (uint32_t)(4 * h + kk) * 2048u, kBox, 1024, kSwizzle128B), idAcc,
                       acc | (kk > 0 ? 1u : 0u));
#pragma unroll
              for (int kk = 0; kk < HB / 16; ++kk)   // dK += dS^T Q_c
                mma_ts(tmem + C::kColAcc, tmem + 128u * b + HB + (uint32_t)kk * 8u,
                       smem_desc(bq + (uint32_t)(4 * h + kk) * 2048u, kBox, 1024, kSwizzle128B), idAcc,
                       acc | (kk > 0 ? 1u : 0u));
            } else {
#pragma unroll
              for (int kk = 0; kk < HB / 16; ++kk)
                mma_ts(tmem + C::kColAcc, tmem + 128u * b + (uint32_t)kk * 8u,
                       smem_desc(b3 + (uint32_t)(4 * h + kk) * 2048u, kBox, 1024, kSwizzle128B), idAcc,
                       acc | (kk > 0 ? 1u : 0u));
            }
            commit(bar(X_DONE + b));
            if (h == 1) commit(bar(C_EMPTY + st));   // last reader of this stage
            if (e + 1 == len && h == 1) commit(bar(ACC_FULL));
          }
          __syncwarp();
          ++hg;
          issued_any = true;
        }
        ++c_use;
      }
      if (!ok) break;
      ++acc_items;
    }
    if (*abort_flag && issued_any) {
      if (elect_one()) commit(bar(TEAR2));
      __syncwarp();
      wait_raw(bar(TEAR2), 0, kDrainNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ P / dS and epilogue
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
    const float sl2 = p.sl2;
    uint32_t it_use = 0, c_use = 0, hg = 0, acc_items = 0, a_use = 0;
    uint4* pending = nullptr;    // output row of the previous item, written once its accumulator is full
    uint4* pending2 = nullptr;   // mode 3: its dV row
    bool has_pending = false, pend_store = false;   // pairs: a row of a missing or bad block is not stored
    bool ok = true;
    // one accumulator (d columns at col) -> bf16 output row (the TMEM loads run in every lane)
    auto acc_out = [&](uint32_t col, float scale, uint4* orow, bool store) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(t_row + col + c * 32u, o);
        wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          w[x] = pack2(__uint_as_float(o[2 * x]) * scale, __uint_as_float(o[2 * x + 1]) * scale);
        if (store)
#pragma unroll
          for (int x = 0; x < 4; ++x) orow[c * 4 + x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
      }
    };
    // accumulator(s) -> output row(s); frees the accumulators for the next item
    auto epilogue = [&](uint4* orow, uint4* orow2, bool store) -> bool {
      if (!wait_warp(bar(ACC_FULL), acc_items & 1u, g)) return false;
      ++acc_items;
      fence_after();
      acc_out(C::kColAcc, p.out_scale, orow, store);
      if (MODE == 3) acc_out(C::kColAcc2, p.out_scale2, orow2, store);
      fence_before();
      mbar_arrive(bar(ACC_EMPTY));
      return true;
    };
    // this thread's row of a 128xD row tile (D/64 boxes of 64 columns, 128-byte
    // swizzle: 16-byte chunk c of row t sits at chunk c ^ (t & 7)) -> D/2 TMEM columns
    auto row_to_tmem = [&](uint32_t tile_off, uint32_t col) {
      const int t = threadIdx.x;
#pragma unroll
      for (int h = 0; h < C::NBOX; ++h) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(gbase + tile_off + (uint32_t)h * kBox +
                                                          (uint32_t)t * 128u + (uint32_t)((c ^ (t & 7)) * 16));
          w[4 * c] = v.x;
          w[4 * c + 1] = v.y;
          w[4 * c + 2] = v.z;
          w[4 * c + 3] = v.w;
        }
        tmem_st32(t_row + col + 32u * h, w);
      }
    };
    for (;;) {
      const int ri = (int)(it_use % kNI);
      if (!(ok = wait_warp(bar(I_FULL + ri), (it_use / kNI) & 1u, g))) break;
      const int4 ent = make_int4(ring[ri].x, ring[ri].y, ring[ri].z, 0);
      __syncwarp();
      // pairs read the slot's masks until the item ends; release it then
      auto release = [&]() {
        if (lane == 0) mbar_arrive(bar(I_EMPTY + ri));
      };
      if (!PAIR) release();
      ++it_use;
      if (ent.y == -2) {
        if (PAIR) release();
        break;
      }
      if (ent.y == -1) {
        if (PAIR) release();
        continue;
      }
      const int64_t item = ent.x;
      // with pairs, rows 0-63 are block 2p and rows 64-127 block 2p + 1
      const int half = PAIR ? (int)(threadIdx.x >> 6) : 0;
      const int64_t bh = item / nbp;
      const int i = PAIR ? 2 * (int)(item % nbp) + half : (int)(item % nb);   // this thread's row block
      const int o = PAIR ? (int)(threadIdx.x & 63) : (int)threadIdx.x;       // its token in the block
      const bool exists = !PAIR || (i < nb && !((ent.z >> half) & 1));      // warp-uniform
      int64_t row = bh * p.N + (int64_t)i * BTB + o;
      if (!exists || !dcheck(row >= 0 && row < p.rows_total, p.d_status)) row = 0;
      int64_t orow_idx = p.raster && exists ? p.rm.row(bh, i, o) : row;
      if (!dcheck(orow_idx >= 0 && orow_idx < p.rows_total, p.d_status)) orow_idx = 0;
      uint4* orow = reinterpret_cast<uint4*>(p.out + orow_idx * D);
      uint4* orow2 = MODE == 3 ? reinterpret_cast<uint4*>(p.out2 + orow_idx * D) : nullptr;
      const int len = ent.y;
      if (len == 0) {
        if (exists) {
#pragma unroll
          for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
          if (MODE == 3)
#pragma unroll
            for (int c = 0; c < D / 8; ++c) orow2[c] = make_uint4(0, 0, 0, 0);
        }
        if (PAIR) release();
        continue;
      }
      if (kRowsInTmem) {
        // the item's row tiles -> TMEM; the A region is free because every S/dP
        // MMA of the previous item has completed (this thread consumed their SD_FULL)
        if (!(ok = wait_warp(bar(A_FULL), a_use & 1u, g))) break;
        ++a_use;
        fence_after();
        row_to_tmem(0u, C::kColA1);
        if (kHasDP) row_to_tmem(C::kOffA2, C::kColA2);
        wait_st();
        fence_before();
        mbar_arrive(bar(A_EMPTY));   // the shared-memory tiles can take the next item's
        mbar_arrive(bar(AT_FULL));   // the S issuer may start this item
      }
      // the previous item's output, while this item's first S and dP run
      if (has_pending) {
        if (!(ok = epilogue(pending, pending2, pend_store))) break;
        has_pending = false;
      }
      // mode 0: this thread's query row has one LSE and one D
      const float own_l2 = MODE == 0 && exists ? p.lse2[row] : 0.f;
      const float own_d = MODE == 0 && exists ? p.delta[row] : 0.f;
      const uint16_t* mk = reinterpret_cast<const uint16_t*>(masks + ri * (C::kMaskBytes + 16));
      for (int e = 0; e < len && ok; ++e) {
        const uint32_t st = c_use % kNS;
        const float4* stats = reinterpret_cast<const float4*>(gbase + C::kOffStage + st * kStageBytes + 2 * kTile);
        const uint32_t msk = PAIR ? (uint32_t)mk[e] : 0xffffu;   // byte h: which rows selected block h
        for (int h = 0; h < 2; ++h) {
          const uint32_t b = hg & 1u;
          if (!(ok = wait_warp(bar(SD_FULL + b), (hg >> 1) & 1u, g))) break;
          fence_after();
          uint32_t sv[HB], dv[HB];
          tmem_ld32(t_row + 128u * b, sv);
          tmem_ld32(t_row + 128u * b + 32u, sv + 32);
          if (kHasDP) {
            tmem_ld32(t_row + 128u * b + HB, dv);
            tmem_ld32(t_row + 128u * b + HB + 32u, dv + 32);
          }
          wait_ld();
          // pairs: a row block that did not select this half's block (or does not
          // exist) gets X = 0 there (warp-uniform)
          const bool has = !PAIR || (exists && ((msk >> (8 * h + half)) & 1u));
          uint32_t xk[HB / 2];
          if constexpr (MODE == 3) {
            // P^T over S^T; dS^T = P^T (dP^T - D) over dP^T (both already in registers)
            uint32_t xd[HB / 2];
#pragma unroll
            for (int x = 0; x < HB / 2; ++x) xk[x] = xd[x] = 0u;
            if (has)
#pragma unroll
            for (int x4 = 0; x4 < HB / 4; ++x4) {
              const float4 L = stats[16 * h + x4];
              const float4 Dv = stats[32 + 16 * h + x4];
              const float l2[4] = {L.x, L.y, L.z, L.w}, dd[4] = {Dv.x, Dv.y, Dv.z, Dv.w};
              float pr[4], ds[4];
#pragma unroll
              for (int u = 0; u < 4; u += 2) {   // column pairs: each lane rounds as the scalar form
                const int x = 4 * x4 + u;
                float e0, e1, t0, t1;
                fma_x2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1]), sl2, -l2[u], -l2[u + 1], e0, e1);
                pr[u] = ex2f(e0);
                pr[u + 1] = ex2f(e1);
                sub_x2(__uint_as_float(dv[x]), __uint_as_float(dv[x + 1]), dd[u], dd[u + 1], t0, t1);
                mul_x2(pr[u], pr[u + 1], t0, t1, ds[u], ds[u + 1]);
              }
              xk[2 * x4] = pack2(pr[0], pr[1]);
              xk[2 * x4 + 1] = pack2(pr[2], pr[3]);
              xd[2 * x4] = pack2(ds[0], ds[1]);
              xd[2 * x4 + 1] = pack2(ds[2], ds[3]);
            }
            tmem_st32(t_row + 128u * b, xk);
            tmem_st32(t_row + 128u * b + HB, xd);
            wait_st();
            fence_before();
            mbar_arrive(bar(X_FULL + b));
          } else {
#pragma unroll
            for (int x = 0; x < HB / 2; ++x) xk[x] = 0u;
            if (has)
#pragma unroll
            for (int x4 = 0; x4 < HB / 4; ++x4) {
              float l2[4], dd[4];
              if (MODE == 0) {
#pragma unroll
                for (int u = 0; u < 4; ++u) { l2[u] = own_l2; dd[u] = own_d; }
              } else {
                const float4 L = stats[16 * h + x4];          // LSE*log2e of columns 64h+4x4 .. +3
                const float4 Dv = stats[32 + 16 * h + x4];    // D of the same columns
                l2[0] = L.x; l2[1] = L.y; l2[2] = L.z; l2[3] = L.w;
                dd[0] = Dv.x; dd[1] = Dv.y; dd[2] = Dv.z; dd[3] = Dv.w;
              }
              float v[4];
#pragma unroll
              for (int u = 0; u < 4; u += 2) {   // column pairs: each lane rounds as the scalar form
                const int x = 4 * x4 + u;
                float e0, e1;
                fma_x2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1]), sl2, -l2[u], -l2[u + 1], e0, e1);
                const float p0 = ex2f(e0), p1 = ex2f(e1);
                if (kHasDP) {
                  float t0, t1;
                  sub_x2(__uint_as_float(dv[x]), __uint_as_float(dv[x + 1]), dd[u], dd[u + 1], t0, t1);
                  mul_x2(p0, p1, t0, t1, v[u], v[u + 1]);
                } else {
                  v[u] = p0;
                  v[u + 1] = p1;
                }
              }
              xk[2 * x4] = pack2(v[0], v[1]);
              xk[2 * x4 + 1] = pack2(v[2], v[3]);
            }
            // X over the first 32 columns of this half's S (already in registers)
            tmem_st32(t_row + 128u * b, xk);
            wait_st();
            fence_before();
            mbar_arrive(bar(X_FULL + b));
          }
          ++hg;
        }
        ++c_use;
      }
      if (!ok) break;
      if (PAIR) release();
      pending = orow;
      pending2 = orow2;
      has_pending = true;
      pend_store = exists;
    }
    if (ok && has_pending) epilogue(pending, pending2, pend_store);
  }

  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
  if (p.prof != nullptr && threadIdx.x == 0)
    atomicAdd((unsigned long long*)&p.prof[smid() % SPARSP_PROF_SLOTS],
              (unsigned long long)(globaltimer_ns() - t_start));
}

template <int MODE, int D, int BTB>
sparsp_status_t go(const Dims& s, const CUtensorMap& a1, const CUtensorMap& a2, const CUtensorMap& b1,
                   const CUtensorMap& b2, const Params& prm, cudaStream_t st) {
  auto kern = attn_bwd_tc_kernel<MODE, D, BTB>;
  constexpr uint32_t kSmemBytes = BCfg<D, BTB>::kSmemBytes;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
    return SPARSP_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return SPARSP_ERR_CUDA;
  const int64_t grid = cap_grid(s, sms, prm.n_items);
  kern<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(a1, a2, b1, b2, prm);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace

bool attn_bwd_tc_supported(const Dims& s) {
  if (s.d != 128 && s.d != 64) return false;
  // 64-token blocks run as pairs; an item slot holds the pair's two lists as bitmaps
  if (s.Bt == 64 && s.nb > 32 * (s.d == 64 ? BCfg<64, 64>::MAXW : BCfg<128, 64>::MAXW)) return false;
  return (s.Bt == 128 || s.Bt == 64) && attn_fwd_tc_supported(s);
}

int attn_bwd_tc_items_per_head(const Dims& s) { return s.Bt == 64 ? (s.nb + 1) / 2 : s.nb; }

namespace {

// Tensor maps: the item's row tiles (A) are 128-row boxes, the column tiles
// (B) boxes of one block (two per stage with 64-token blocks).
struct Maps {
  CUtensorMap q, k, v, dout;   // 128-row boxes
  CUtensorMap qb, kb, vb, dob;  // one block per box
};

template <int D, int BTB>
sparsp_status_t launch_d(int mode, const Maps& m, const Dims& s, const Params& prm, cudaStream_t st) {
  if (mode == 0) return go<0, D, BTB>(s, m.q, m.dout, m.kb, m.vb, prm, st);
  if (mode == 1) return go<1, D, BTB>(s, m.k, m.v, m.qb, m.dob, prm, st);
  if (mode == 3) return go<3, D, BTB>(s, m.k, m.v, m.qb, m.dob, prm, st);
  return go<2, D, BTB>(s, m.k, m.k, m.qb, m.dob, prm, st);
}

}  // namespace

sparsp_status_t launch_attn_bwd_tc(const Dims& s, int mode, const __nv_bfloat16* q,
                                   const __nv_bfloat16* k, const __nv_bfloat16* v,
                                   const __nv_bfloat16* dout, const float* lse2,
                                   const float* delta, const int32_t* ptr, const int32_t* idx,
                                   float scale, __nv_bfloat16* out, __nv_bfloat16* out2,
                                   const int32_t* items, int32_t* counter, uint64_t* prof, int32_t* d_status,
                                   bool raster, cudaStream_t st) {
  const uint64_t rows = (uint64_t)s.B * s.H * s.N;
  const uint64_t d = (uint64_t)s.d;
  const uint32_t bt = (uint32_t)s.Bt;
  Maps m;
  if (!make_tmap_bf16_rows(&m.q, q, rows, d, TR) || !make_tmap_bf16_rows(&m.k, k, rows, d, TR) ||
      !make_tmap_bf16_rows(&m.v, v, rows, d, TR) || !make_tmap_bf16_rows(&m.dout, dout, rows, d, TR) ||
      !make_tmap_bf16_rows(&m.qb, q, rows, d, bt) || !make_tmap_bf16_rows(&m.kb, k, rows, d, bt) ||
      !make_tmap_bf16_rows(&m.vb, v, rows, d, bt) || !make_tmap_bf16_rows(&m.dob, dout, rows, d, bt))
    return SPARSP_ERR_CUDA;
  // 64-token blocks: items are pairs of blocks, ordered by the caller over the
  // pairs' lists (attn_bwd_tc_items_per_head per head)
  const int nbp = attn_bwd_tc_items_per_head(s);
  Params prm{ptr, idx, s.N, s.nb, nbp, (int64_t)s.B * s.H * nbp, (int64_t)rows, scale * 1.4426950408889634f,
             mode == 2 ? 1.0f : scale, lse2, delta, out, out2, 1.0f, items, counter, prof, d_status,
             raster ? 1 : 0, raster_map(s)};
  if (s.Bt == 64) {
    if (s.d == 64) return launch_d<64, 64>(mode, m, s, prm, st);
    return launch_d<128, 64>(mode, m, s, prm, st);
  }
  if (s.d == 64) return launch_d<64, 128>(mode, m, s, prm, st);
  return launch_d<128, 128>(mode, m, s, prm, st);
}

}  // namespace sparsp
