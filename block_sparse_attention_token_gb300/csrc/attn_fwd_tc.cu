// Step 5a, bf16, Bt and d in {64, 128} on sm_103a: block-sparse flash-attention
// forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Every MMA works on 128 query rows (M = 128, the 128 TMEM lanes) and on
// stages of 128 key tokens. With 128-token blocks a work item is one query
// block and a stage one key block. With 64-token blocks a work item is a PAIR
// of neighbouring query blocks of a head (2p and 2p + 1: 128 contiguous rows)
// processed over the union of their two CSR rows, and a stage holds two key
// blocks of that union (two 64-row TMA boxes side by side); each 64-column half
// of S is masked, for each of the two query blocks, when that block did not
// select the key block (its P is zero there and no exponential is evaluated).
// So no MMA row or column is computed for nothing except where the two rows'
// selections differ ("Dynamic Sparsity in Large-Scale Video DiT Training",
// "How DSV works": queries grouped so that one key set serves several).
//
// Persistent CTAs: one per SM with 7 warps (4 softmax warps, then the
// producer, the S issuer and the PV issuer) for d = 128; two per SM for d = 64,
// each with 8 warps (4 softmax warps, the producer, one warp issuing both GEMM
// streams, two idle warps that only give their registers to the softmax
// warpgroup) and half of the TMEM and shared memory (one S and one P buffer;
// see Cfg::DUO):
//   producer: pulls items longest-first through an atomic counter,
//              validates the CSR row(s), publishes the item in a shared-memory
//              ring (for pairs with the two rows as bitmaps), and TMA-loads the
//              query tile and the K / V tiles of each stage (64-column boxes
//              with 128-byte swizzle) into 3-stage K and V rings, addressed
//              through the CSR (row coordinate = bh*N + j*Bt).
//   S issuer: S = Q K^T into one of two TMEM S buffers (M=N=128,
//              K=16 per instruction, both operands K-major from shared memory).
//   PV issuer: O += P V (A = P read from TMEM as packed bf16,
//              B = V MN-major from shared memory).
//              With d = 128 the two GEMM streams are issued by different warps
//              so that a wait in one (for P, or for a free S buffer) never
//              holds back the other; each warp runs uniformly and one elected
//              lane issues tcgen05.mma / tcgen05.commit.
//   softmax and epilogue: thread t owns query row t = TMEM lane t.
//              It reads its S row from TMEM with the sm_103 load-with-maximum
//              (tcgen05.ld.red: each 32-column load also returns the maximum of
//              the 32 values, so the row max costs no extra instructions), keeps
//              a running max m and sum l in
//              base 2, writes P = exp2(S*scale*log2e - m) as bf16 into TMEM, and
//              rescales its O row in TMEM only when the row max grows by more
//              than 8 (a factor 256); otherwise the stale max is kept, which
//              leaves the result unchanged up to rounding because O and l use
//              the same reference. At the end of the row: O / l to global
//              memory, LSE = (m + log2 l) ln 2 (O = 0, LSE = -inf for a row
//              that attended to nothing). A warp's 32 rows belong to one query
//              block, so the masks of a pair are warp-uniform.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256,384), P0 [384,448),
// P1 [448,512); DUO (256 columns per CTA): S [0,128), O [128,192),
// P [192,256). Every mbarrier wait is bounded (2 s); on expiry the CTA sets
// SPARSP_ERR_TIMEOUT, all roles leave their loops, copies and MMAs in flight
// are drained with a second bounded wait, and TMEM is released.
#include "pairs.cuh"
#include "tc_helpers.cuh"

namespace sparsp {
namespace {

using namespace tc;

constexpr int kMaxStages = 6, kNI = 4;   // K / V ring depth <= kMaxStages (Cfg::NK); item ring <= kNI
enum Bar {
  Q_FULL = 0, Q_EMPTY, K_FULL, K_EMPTY = K_FULL + kMaxStages, V_FULL = K_EMPTY + kMaxStages,
  V_EMPTY = V_FULL + kMaxStages, S_FULL = V_EMPTY + kMaxStages, S_FREE = S_FULL + 2, P_FULL = S_FREE + 2, PV_DONE = P_FULL + 2, O_FULL = PV_DONE + 2,
  O_EMPTY,
  I_FULL, I_EMPTY = I_FULL + kNI, TEAR = I_EMPTY + kNI, TEAR_PV, NBAR
};
// Tile geometry for blocks of BT tokens and head dimension D. The query tile
// and a key/value stage are 128 rows each: one block, or two 64-token blocks
// (PAIR). Tiles are TMA'd as 64-column boxes of 128-byte rows with 128-byte
// swizzle; a stage of two blocks is two 64-row boxes per column box, the
// second 64 rows (8 KB, a whole number of 1 KB swizzle atoms) after the first.
template <int BT_, int D_>
struct Cfg {
  static constexpr int BT = BT_, D = D_, QR = 128, KR = 128;
  static constexpr bool PAIR = BT == 64;
  // d = 64 (64- or 128-token blocks): two CTAs per SM, each with half of the TMEM
  // (one S buffer [0,128), O [128,192), one P buffer [192,256)) and half of
  // the shared memory (3 K and 2 V stages), so that one CTA's softmax runs
  // while the other's MMAs keep the tensor pipe busy. The softmax warps hold
  // a whole 128-column S row in registers (one pass per stage, S released as
  // soon as it is loaded) with the 200 registers the register split below
  // gives them.
  static constexpr bool DUO = D == 64;
  static constexpr int NSM = 4;                           // softmax warps
  // MMA issuer warps: S and PV each get their own with d = 128; with DUO one
  // warp issues both streams (the softmax releases S(e-1) before it writes
  // P(e-1), so S(e) then PV(e-1) in one warp never wait on each other)
  static constexpr int NIS = DUO ? 1 : 2;
  // DUO: two idle warps complete the second warpgroup (producer, issuer), so
  // that the softmax warpgroup can take registers from it (setmaxnreg works
  // on whole warpgroups): two CTAs of 8 warps launch at 128 registers a
  // thread; the softmax warps rise to 200 and the other four drop to 56
  // (4 x 32 x 200 + 4 x 32 x 56 = 256 x 128)
  static constexpr int NIDLE = DUO ? 2 : 0;
  static constexpr int THREADS = 32 * (NSM + 1 + NIS + NIDLE);   // + producer, issuer(s), idle
  static constexpr int W_PROD = NSM, W_S = NSM + 1, W_PV = NSM + NIS;
  static constexpr uint32_t kRegSoftmax = 200, kRegAux = 56;
  static_assert(!DUO || (THREADS == 256 && NSM == 4 && 128 * (kRegSoftmax + kRegAux) == 256 * 128),
                "register split of the two warpgroups");
  // K and V ring stages: 3 of each fit beside a d = 128 query tile; a DUO CTA
  // has half of the SM's shared memory for tiles of half the size: 3 K and 2 V
  static constexpr int NK = 3, NV = DUO ? 2 : 3;
  static constexpr int NSB = DUO ? 1 : 2, NPB = DUO ? 1 : 2;   // S and P buffers in TMEM
  static constexpr int NI = DUO || PAIR ? 2 : kNI;              // item ring slots
  static constexpr int kMinCtas = DUO ? 2 : 1;                  // CTAs per SM
  static constexpr uint32_t kColS = 0, kColO = DUO ? 128 : 256, kColP = DUO ? 192 : 384;
  static constexpr uint32_t kTmemCols = DUO ? 256 : 512;
  // bitmap words of one CSR row in the item ring (pairs): up to kMaxBlocks
  // blocks, except for d = 128 whose tiles leave room for 1,024 blocks only
  // (larger shapes run the portable kernel, see attn_fwd_tc_supported)
  static constexpr int MAXW = D == 64 ? kMaxBlocks / 32 : 32;
  static constexpr int NBOX = D / 64;                     // 64-column boxes per row tile
  static constexpr uint32_t kQBox = QR * 128, kKBox = KR * 128, kHalfBox = 64 * 128;
  static constexpr uint32_t kQTile = kQBox * NBOX, kKTile = kKBox * NBOX;
  static constexpr uint32_t kOffK = kQTile, kOffV = kOffK + NK * kKTile, kOffBar = kOffV + NV * kKTile;
  static constexpr uint32_t kOffRing = kOffBar + 8 * NBAR;
  static constexpr uint32_t kOffBits = kOffRing + 16 * NI;
  static constexpr uint32_t kBitsBytes = PAIR ? NI * 2 * MAXW * 4 : 0;
  // pairs: per item slot, which of the pair's two rows selected each block of
  // the union of their rows (ascending), written by the producer with the item
  // so that the softmax warps read a stage's masks with one shared-memory load:
  // one byte per block with DUO (bytes 2s, 2s + 1: stage s; bit 0 = the first
  // row, bit 1 = the second), two bits per block where shared memory is short
  // (d = 128: stage s is nibble s)
  static constexpr bool MASK_BYTES = DUO;
  static constexpr uint32_t kMaskWords = !PAIR ? 0 : (MASK_BYTES ? 8 * MAXW + 4 : 2 * MAXW + 1);
  static constexpr uint32_t kOffMask = kOffBits + kBitsBytes;
  static constexpr uint32_t kOffMisc = kOffMask + NI * kMaskWords * 4;
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
  static_assert(kSmemBytes <= (DUO ? 115712u : 232448u), "shared memory");
};
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

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

// 32 columns of this thread's TMEM lane, and their maximum (sm_103 load with
// reduction)
__device__ __forceinline__ float tmem_ld32_max(uint32_t taddr, uint32_t* r) {
  float m;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=f"(m)
      : "r"(taddr));
  return m;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

struct Params {
  const int32_t* row_ptr;
  const int32_t* col_idx;
  int64_t N;
  int nb;
  int nbp;           // items per head: nb, or ceil(nb/2) pairs of 64-token blocks
  int64_t n_items;
  int64_t rows_total;   // B*H*N rows of Q, K, V, O and LSE
  float scale_log2;
  __nv_bfloat16* o;
  float* lse;
  // raster output: O rows at rm.row(bh, block, token) (the layout of the inverse
  // reorder); otherwise block order like Q
  int raster;
  RasterMap rm;
  // raster input: Q, K, V read from [B, N, H, d] through 5-D maps, one block per box
  int in_raster;
  RasterBox rbox;
  const int32_t* items;
  int32_t* counter;
  uint64_t* prof;
  int32_t* d_status;
};

template <int BT, int D>
__global__ void __launch_bounds__(Cfg<BT, D>::THREADS, Cfg<BT, D>::kMinCtas)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  using C = Cfg<BT, D>;
  constexpr bool PAIR = C::PAIR;
  const uint32_t sQ = base, sK = base + C::kOffK, sV = base + C::kOffV;
  auto bar = [&](int idx) -> uint32_t { return base + C::kOffBar + 8u * (uint32_t)idx; };
  // ring entry: x = item, y = stages (-1: skip, -2: end), z = bad-row bits (pairs)
  volatile int4* ring = reinterpret_cast<volatile int4*>(gbase + C::kOffRing);
  uint32_t* bits = reinterpret_cast<uint32_t*>(gbase + C::kOffBits);   // [C::NI][2][C::MAXW] (pairs)
  uint32_t* masks = reinterpret_cast<uint32_t*>(gbase + C::kOffMask);   // [C::NI][C::kMaskWords] (pairs)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(gbase + C::kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t t_start = globaltimer_ns();
  const int words = (p.nb + 31) >> 5;

  if (threadIdx.x == 0) {
    mbar_init(bar(Q_FULL), 1);
    mbar_init(bar(Q_EMPTY), 1);
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(bar(K_FULL + s), 1);
      mbar_init(bar(K_EMPTY + s), 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(bar(V_FULL + s), 1);
      mbar_init(bar(V_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(S_FULL + b), 1);
      mbar_init(bar(S_FREE + b), 32 * C::NSM);
      mbar_init(bar(P_FULL + b), 32 * C::NSM);
    }
    mbar_init(bar(PV_DONE), 1);
    mbar_init(bar(PV_DONE + 1), 1);
    mbar_init(bar(O_FULL), 1);
    mbar_init(bar(O_EMPTY), 32 * C::NSM);
    for (int r = 0; r < kNI; ++r) {
      mbar_init(bar(I_FULL + r), 1);
      mbar_init(bar(I_EMPTY + r), C::NSM + C::NIS);
    }
    mbar_init(bar(TEAR), 1);
    mbar_init(bar(TEAR_PV), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::W_PROD && lane == 0) {
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
  }
  if (warp == C::W_S) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  const Guard g{abort_flag, p.d_status, kWaitNs};
  const int nb = p.nb, nbp = p.nbp;

  if (warp >= C::NSM) {
  if constexpr (C::DUO) regs_decrease<C::kRegAux>();   // the whole second warpgroup
  if (warp == C::W_PROD) {
    // ------------------------------------------------------------ producer
    uint32_t it_fill = 0, q_fill = 0, k_fill = 0, v_fill = 0;
    for (;;) {
      int32_t slot = 0;
      if (lane == 0) slot = atomicAdd(p.counter, 1);
      slot = __shfl_sync(0xffffffffu, slot, 0);
      const int ri = (int)(it_fill % C::NI);
      if (!wait_warp(bar(I_EMPTY + ri), ((it_fill / C::NI) & 1u) ^ 1u, g)) break;
      uint32_t* bmA = bits + ri * 2 * C::MAXW;
      uint32_t* bmB = bmA + C::MAXW;
      int32_t item = -1, len = -2, badbits = 0;
      if (slot < p.n_items) {
        item = p.items[slot];
        if constexpr (PAIR) {
          // the two rows as bitmaps in the ring slot; a bad row counts as empty
          const int64_t bh = item / nbp;
          const int iA = 2 * (item % nbp);
          for (int w = lane; w < 2 * C::MAXW; w += 32) bmA[w] = 0u;
          __syncwarp();
          const bool okA = list_bitmap(p.row_ptr, p.col_idx, nb, bh * nb + iA, bmA, words, lane);
          const bool okB = iA + 1 < nb ? list_bitmap(p.row_ptr, p.col_idx, nb, bh * nb + iA + 1, bmB, words, lane)
                                       : true;
          badbits = (okA ? 0 : 1) | (okB ? 0 : 2);
          if (badbits && lane == 0) report(p.d_status, SPARSP_ERR_DATA);
          const int u = union_count(bmA, bmB, words, lane);
          len = (badbits == 3) ? -1 : (u + 1) / 2;   // stages of two key blocks
          if constexpr (C::MASK_BYTES)
            union_masks(bmA, bmB, words, u, lane, reinterpret_cast<uint8_t*>(masks + ri * C::kMaskWords));
          else
            union_masks2(bmA, bmB, words, u, lane, masks + ri * C::kMaskWords);
        } else {
          const int32_t a = p.row_ptr[item], b = p.row_ptr[item + 1];
          bool bad = (b < a) || (b - a > nb);
          if (!bad)
            for (int32_t e = a + lane; e < b; e += 32) {
              const int32_t j = p.col_idx[e];
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
      const int i0 = PAIR ? 2 * (item % nbp) : item % nb;   // first query block of the item
      int32_t yq = (int32_t)(bh * p.N + (int64_t)i0 * BT);
      if (!dcheck(yq >= 0 && yq < p.rows_total, p.d_status)) yq = 0;
      if (!wait_warp(bar(Q_EMPTY), (q_fill & 1u) ^ 1u, g)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(Q_FULL), C::kQTile);
#pragma unroll
        for (int h = 0; h < C::NBOX; ++h) {
          if (p.in_raster) {   // the item's block(s), one 5-D box each
            const int4 c = p.rbox.at(bh, i0);
            tma_load_5d(sQ + h * C::kQBox, &tq, bar(Q_FULL), 64 * h, c.x, c.y, c.z, c.w);
            if (PAIR) {   // a head's last pair of an odd nb loads its first block twice (never stored)
              const int4 c2 = p.rbox.at(bh, i0 + 1 < nb ? i0 + 1 : i0);
              tma_load_5d(sQ + h * C::kQBox + C::kHalfBox, &tq, bar(Q_FULL), 64 * h, c2.x, c2.y, c2.z, c2.w);
            }
          } else {
            tma_load_2d(sQ + h * C::kQBox, &tq, bar(Q_FULL), 64 * h, yq);
          }
        }
      }
      ++q_fill;
      const int32_t e0 = PAIR ? 0 : p.row_ptr[item];
      UnionWalk walk(bmA, bmB, PAIR ? words : 0);
      bool ok = true;
      for (int e = 0; e < len && ok; ++e) {
        int32_t j1, j2 = 0;
        if constexpr (PAIR) {
          j1 = walk.next();
          j2 = walk.next();
          if (j2 < 0) j2 = j1;   // a lone last block: loaded twice, its second half masked
        } else {
          j1 = p.col_idx[e0 + e];
        }
        int32_t yk1 = (int32_t)(bh * p.N + (int64_t)j1 * BT);
        int32_t yk2 = (int32_t)(bh * p.N + (int64_t)j2 * BT);
        if (!dcheck(yk1 >= 0 && yk1 + BT <= p.rows_total && yk2 >= 0 && yk2 + BT <= p.rows_total, p.d_status))
          yk1 = yk2 = 0;   // keep the transaction counts; the result is flagged
        const uint32_t ks = k_fill % C::NK;
        if (!(ok = wait_warp(bar(K_EMPTY + ks), ((k_fill / C::NK) & 1u) ^ 1u, g))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(K_FULL + ks), C::kKTile);
#pragma unroll
          for (int h = 0; h < C::NBOX; ++h) {
            const uint32_t dst = sK + ks * C::kKTile + h * C::kKBox;
            if (p.in_raster) {
              const int4 c1 = p.rbox.at(bh, j1);
              tma_load_5d(dst, &tk, bar(K_FULL + ks), 64 * h, c1.x, c1.y, c1.z, c1.w);
              if (PAIR) {
                const int4 c2 = p.rbox.at(bh, j2);
                tma_load_5d(dst + C::kHalfBox, &tk, bar(K_FULL + ks), 64 * h, c2.x, c2.y, c2.z, c2.w);
              }
            } else {
              tma_load_2d(dst, &tk, bar(K_FULL + ks), 64 * h, yk1);
              if (PAIR) tma_load_2d(dst + C::kHalfBox, &tk, bar(K_FULL + ks), 64 * h, yk2);
            }
          }
        }
        ++k_fill;
        const uint32_t vs = v_fill % C::NV;
        if (!(ok = wait_warp(bar(V_EMPTY + vs), ((v_fill / C::NV) & 1u) ^ 1u, g))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(V_FULL + vs), C::kKTile);
#pragma unroll
          for (int h = 0; h < C::NBOX; ++h) {
            const uint32_t dst = sV + vs * C::kKTile + h * C::kKBox;
            if (p.in_raster) {
              const int4 c1 = p.rbox.at(bh, j1);
              tma_load_5d(dst, &tv, bar(V_FULL + vs), 64 * h, c1.x, c1.y, c1.z, c1.w);
              if (PAIR) {
                const int4 c2 = p.rbox.at(bh, j2);
                tma_load_5d(dst + C::kHalfBox, &tv, bar(V_FULL + vs), 64 * h, c2.x, c2.y, c2.z, c2.w);
              }
            } else {
              tma_load_2d(dst, &tv, bar(V_FULL + vs), 64 * h, yk1);
              if (PAIR) tma_load_2d(dst + C::kHalfBox, &tv, bar(V_FULL + vs), 64 * h, yk2);
            }
          }
        }
        ++v_fill;
      }
      if (!ok) break;
    }
    if (*abort_flag && lane == 0) {
      // drain copies still in flight before the shared memory goes away
      if (q_fill) wait_raw(bar(Q_FULL), (q_fill - 1) & 1u, kDrainNs);
      for (uint32_t s = 0; s < C::NK; ++s)
        if (k_fill > s) wait_raw(bar(K_FULL + s), ((k_fill - 1 - s) / C::NK) & 1u, kDrainNs);
      for (uint32_t s = 0; s < C::NV; ++s)
        if (v_fill > s) wait_raw(bar(V_FULL + s), ((v_fill - 1 - s) / C::NV) & 1u, kDrainNs);
    }
  } else if (C::DUO && warp == C::W_S) {
    // ------------------------------------------------------------ S and PV from one warp (DUO)
    // Per item: S(0), then S(e) before PV(e-1) for e = 1 .. len-1, then PV(len-1).
    // S(e) waits for the softmax to have loaded S(e-1) (one S buffer) and PV(e-1)
    // for P(e-1); the softmax releases S(e-1) before it writes P(e-1), so neither
    // wait holds back the other stream, and S(e) runs under the softmax of e-1.
    constexpr uint32_t idS = idesc_bf16(128, C::KR, 0, 0);
    constexpr uint32_t idO = idesc_bf16(128, D, 0, 1);
    uint32_t it_use = 0, q_use = 0, k_use = 0, v_use = 0, s_issue = 0, pv = 0, o_items = 0;
    bool issued_any = false, ok = true;
    for (;;) {
      const int ri = (int)(it_use % C::NI);
      if (!(ok = wait_warp(bar(I_FULL + ri), (it_use / C::NI) & 1u, g))) break;
      const int len = ring[ri].y;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(I_EMPTY + ri));
      ++it_use;
      if (len == -2) break;
      if (len <= 0) continue;
      if (!(ok = wait_warp(bar(Q_FULL), q_use & 1u, g))) break;
      ++q_use;
      for (int e = 0; e <= len && ok; ++e) {
        if (e < len) {
          const uint32_t ks = k_use % C::NK;
          if (!(ok = wait_warp(bar(S_FREE), (s_issue & 1u) ^ 1u, g))) break;
          if (!(ok = wait_warp(bar(K_FULL + ks), (k_use / C::NK) & 1u, g))) break;
          fence_after();
          const uint32_t kb = sK + ks * C::kKTile;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t offq = (uint32_t)(kk >> 2) * C::kQBox + (uint32_t)(kk & 3) * 32u;
              const uint32_t offk = (uint32_t)(kk >> 2) * C::kKBox + (uint32_t)(kk & 3) * 32u;
              mma_ss(tmem + C::kColS, smem_desc(sQ + offq, 16, 1024, kSwizzle128B),
                     smem_desc(kb + offk, 16, 1024, kSwizzle128B), idS, kk > 0 ? 1u : 0u);
            }
            commit(bar(S_FULL));
            commit(bar(K_EMPTY + ks));
            if (e + 1 == len) commit(bar(Q_EMPTY));
          }
          __syncwarp();
          ++s_issue;
          ++k_use;
          issued_any = true;
        }
        if (e == 0) continue;
        // O += P(e-1) V(e-1)
        const uint32_t vs = v_use % C::NV;
        if (!(ok = wait_warp(bar(V_FULL + vs), (v_use / C::NV) & 1u, g))) break;
        if (!(ok = wait_warp(bar(P_FULL), pv & 1u, g))) break;
        if (e == 1 && !(ok = wait_warp(bar(O_EMPTY), (o_items & 1u) ^ 1u, g))) break;
        fence_after();
        const uint32_t vb = sV + vs * C::kKTile;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < C::KR / 16; ++kk)
            mma_ts(tmem + C::kColO, tmem + C::kColP + (uint32_t)kk * 8u,
                   smem_desc(vb + (uint32_t)kk * 2048u, C::kKBox, 1024, kSwizzle128B), idO,
                   (e > 1 || kk > 0) ? 1u : 0u);
          commit(bar(V_EMPTY + vs));
          commit(bar(PV_DONE));
          if (e == len) commit(bar(O_FULL));
        }
        __syncwarp();
        ++v_use;
        ++pv;
      }
      if (!ok) break;
      ++o_items;
    }
    if (*abort_flag && issued_any) {
      if (elect_one()) commit(bar(TEAR));
      __syncwarp();
      wait_raw(bar(TEAR), 0, kDrainNs);
    }
    __syncwarp();
  } else if (warp == C::W_S) {
    // ------------------------------------------------------------ S = Q K^T issuer
    constexpr uint32_t idS = idesc_bf16(128, C::KR, 0, 0);
    uint32_t it_use = 0, q_use = 0, k_use = 0, s_issue = 0;
    bool issued_any = false;
    for (;;) {
      const int ri = (int)(it_use % C::NI);
      if (!wait_warp(bar(I_FULL + ri), (it_use / C::NI) & 1u, g)) break;
      const int len = ring[ri].y;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(I_EMPTY + ri));
      ++it_use;
      if (len == -2) break;
      if (len <= 0) continue;
      if (!wait_warp(bar(Q_FULL), q_use & 1u, g)) break;
      ++q_use;
      bool ok = true;
      for (int e = 0; e < len; ++e) {
        const uint32_t b = s_issue % C::NSB, ks = k_use % C::NK;
        if (!(ok = wait_warp(bar(S_FREE + b), ((s_issue / C::NSB) & 1u) ^ 1u, g))) break;
        if (!(ok = wait_warp(bar(K_FULL + ks), (k_use / C::NK) & 1u, g))) break;
        fence_after();
        const uint32_t kb = sK + ks * C::kKTile;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // k-step kk: 16 columns = 32 bytes into the row, in box kk / 4
            const uint32_t offq = (uint32_t)(kk >> 2) * C::kQBox + (uint32_t)(kk & 3) * 32u;
            const uint32_t offk = (uint32_t)(kk >> 2) * C::kKBox + (uint32_t)(kk & 3) * 32u;
            mma_ss(tmem + C::kColS + b * 128u, smem_desc(sQ + offq, 16, 1024, kSwizzle128B),
                   smem_desc(kb + offk, 16, 1024, kSwizzle128B), idS, kk > 0 ? 1u : 0u);
          }
          commit(bar(S_FULL + b));
          commit(bar(K_EMPTY + ks));
          if (e + 1 == len) commit(bar(Q_EMPTY));   // every S of this item is issued
        }
        __syncwarp();
        ++s_issue;
        ++k_use;
        issued_any = true;
      }
      if (!ok) break;
    }
    if (*abort_flag && issued_any) {
      if (elect_one()) commit(bar(TEAR));
      __syncwarp();
      wait_raw(bar(TEAR), 0, kDrainNs);
    }
    __syncwarp();
  } else if (warp == C::W_PV) {
    // ------------------------------------------------------------ O += P V issuer
    constexpr uint32_t idO = idesc_bf16(128, D, 0, 1);
    uint32_t it_use = 0, v_use = 0, pv = 0, o_items = 0;
    bool issued_any = false;
    for (;;) {
      const int ri = (int)(it_use % C::NI);
      if (!wait_warp(bar(I_FULL + ri), (it_use / C::NI) & 1u, g)) break;
      const int len = ring[ri].y;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(I_EMPTY + ri));
      ++it_use;
      if (len == -2) break;
      if (len <= 0) continue;
      bool ok = true;
      for (int e = 0; e < len; ++e) {
        const uint32_t b = pv % C::NPB, vs = v_use % C::NV;
        if (!(ok = wait_warp(bar(V_FULL + vs), (v_use / C::NV) & 1u, g))) break;
        if (!(ok = wait_warp(bar(P_FULL + b), (pv / C::NPB) & 1u, g))) break;
        if (e == 0 && !(ok = wait_warp(bar(O_EMPTY), (o_items & 1u) ^ 1u, g))) break;
        fence_after();
        const uint32_t vb = sV + vs * C::kKTile;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < C::KR / 16; ++kk)
            mma_ts(tmem + C::kColO, tmem + C::kColP + b * 64u + (uint32_t)kk * 8u,
                   smem_desc(vb + (uint32_t)kk * 2048u, C::kKBox, 1024, kSwizzle128B), idO,
                   (e > 0 || kk > 0) ? 1u : 0u);
          commit(bar(V_EMPTY + vs));
          commit(bar(PV_DONE + b));
          if (e + 1 == len) commit(bar(O_FULL));
        }
        __syncwarp();
        ++v_use;
        ++pv;
        issued_any = true;
      }
      if (!ok) break;
      ++o_items;
    }
    if (*abort_flag && issued_any) {
      if (elect_one()) commit(bar(TEAR_PV));
      __syncwarp();
      wait_raw(bar(TEAR_PV), 0, kDrainNs);
    }
    __syncwarp();
  }
  } else {
    if constexpr (C::DUO) regs_increase<C::kRegSoftmax>();
    {
    // ------------------------------------------------------------ softmax + epilogue
      const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
      const uint32_t t_row = tmem + lane_base;
      uint32_t it_use = 0, s_use = 0, o_items = 0;
      uint64_t blocks_done = 0;
      const float sl2 = p.scale_log2;
      // with pairs, rows 0-63 are query block 2p and rows 64-127 block 2p + 1
      const int half = PAIR ? (int)(threadIdx.x >> 6) : 0;
      bool ok = true;
      for (;;) {
        const int ri = (int)(it_use % C::NI);
        if (!wait_warp(bar(I_FULL + ri), (it_use / C::NI) & 1u, g)) break;
        const int64_t item = ring[ri].x;
        const int len = ring[ri].y;
        const int badbits = ring[ri].z;
        __syncwarp();
        // pairs read the item's bitmaps until the item ends; release the slot then
        auto release = [&]() {
          if (lane == 0) mbar_arrive(bar(I_EMPTY + ri));
        };
        if (!PAIR) release();
        ++it_use;
        if (len == -2) {
          if (PAIR) release();
          break;
        }
        if (len == -1) {
          if (PAIR) release();
          continue;
        }
        const int64_t bh = item / nbp;
        const int i = PAIR ? 2 * (int)(item % nbp) + half : (int)(item % nb);   // this thread's query block
        const int o = PAIR ? (int)(threadIdx.x & 63) : (int)threadIdx.x;       // its token in the block
        const int64_t row = bh * p.N + (int64_t)i * BT + o;
        // rows past the block (or past the last block of a pair) are computed, never stored
        bool stores = o < BT && i < nb && !((badbits >> half) & 1);
        int64_t orow_idx = row;
        if (p.raster && stores) orow_idx = p.rm.row(bh, i, o);
        if (stores) stores = dcheck(row < p.rows_total && orow_idx >= 0 && orow_idx < p.rows_total, p.d_status);
        uint4* orow = reinterpret_cast<uint4*>(p.o + orow_idx * D);
        if (len == 0) {
          if (stores) {
  #pragma unroll
            for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
            p.lse[row] = -INFINITY;
          }
          if (PAIR) release();
          continue;
        }
        const uint32_t* mk = masks + ri * C::kMaskWords;
        float m = -INFINITY, l = 0.f;
        for (int e = 0; e < len; ++e) {
          // which halves of this stage's 128 columns this row attends to (warp-uniform)
          bool has1 = true, has2 = true;
          if constexpr (PAIR && C::MASK_BYTES) {
            const uint32_t st = reinterpret_cast<const uint16_t*>(mk)[e];   // bytes 2e, 2e + 1
            has1 = (st >> half) & 1u;
            has2 = (st >> (8 + half)) & 1u;
          } else if constexpr (PAIR) {
            const uint32_t nib = mk[e >> 3] >> (4 * (e & 7));   // stage e's two blocks, two rows
            has1 = (nib >> half) & 1u;
            has2 = (nib >> (2 + half)) & 1u;
          }
          const uint32_t b = s_use % C::NSB;
          if (!(ok = wait_warp(bar(S_FULL + b), (s_use / C::NSB) & 1u, g))) break;
          fence_after();
          {
          uint32_t s[C::KR];
          float cm[C::KR / 32];   // the maximum of each 32-column load (exact, as any order of max)
  #pragma unroll
          for (int c = 0; c < C::KR / 32; ++c)
            cm[c] = tmem_ld32_max(t_row + C::kColS + b * 128u + c * 32u, s + 32 * c);
          wait_ld();
          fence_before();
          mbar_arrive(bar(S_FREE + b));
          ++s_use;
          if (!has1) cm[0] = cm[1] = -INFINITY;
          if (!has2) cm[2] = cm[3] = -INFINITY;
          float mx = cm[0];
  #pragma unroll
          for (int c = 1; c < C::KR / 32; ++c) mx = fmaxf(mx, cm[c]);
          const float m_new = fmaxf(m, mx * sl2);
          // a rescale of O (by f) is applied after P is written, when the S row is
          // no longer held in registers
          bool resc = false;
          float f = 1.f;
          if (e == 0) {
            m = m_new;
          } else if (__any_sync(0xffffffffu, m_new > m + kRescaleThreshold)) {
            resc = true;
            f = ex2f(m - m_new);
            m = m_new;
          }
          uint32_t pk[C::KR / 2];
          float rs[8];
  #pragma unroll
          for (int u = 0; u < 8; ++u) rs[u] = 0.f;
  #pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            // columns [64*hh, 64*hh + 64): one key block of a pair (both halves of
            // one block otherwise)
            if (hh == 0 ? has1 : has2) {
              // two columns per instruction for the scale-and-subtract and the sums
              // (packed fp32 pairs: eight running sums, even and odd columns)
  #pragma unroll
              for (int c = 32 * hh; c < 32 * hh + 32; ++c) {
                float x0, x1;
                fma_x2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1]), sl2, -m, x0, x1);
                const float p0 = ex2f(x0), p1 = ex2f(x1);
                add_x2(rs[2 * (c & 3)], rs[2 * (c & 3) + 1], p0, p1);
                pk[c] = pack2(p0, p1);
              }
            } else {
  #pragma unroll
              for (int c = 32 * hh; c < 32 * hh + 32; ++c) pk[c] = 0u;
            }
          }
          // P buffer b was last read by the PV of block g - NPB
          const uint64_t gb = blocks_done + e;
          if (gb >= (uint64_t)C::NPB) {
            if (!(ok = wait_warp(bar(PV_DONE + b), (uint32_t)(((gb - C::NPB) / C::NPB) & 1u), g))) break;
            fence_after();
          }
  #pragma unroll
          for (int c = 0; c < C::KR / 64; ++c) tmem_st32(t_row + C::kColP + b * 64u + 32u * c, pk + 32 * c);
          if (resc) {
            // O must not change under the PV of block g-1 (g = global block index)
            const uint64_t gp = gb - 1;
            if (!(ok = wait_warp(bar(PV_DONE + (uint32_t)(gp % C::NPB)), (uint32_t)((gp / C::NPB) & 1u), g))) break;
            fence_after();
  #pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t ov[32];
              tmem_ld32(t_row + C::kColO + c * 32u, ov);
              wait_ld();
  #pragma unroll
              for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * f);
              tmem_st32(t_row + C::kColO + c * 32u, ov);
            }
            l *= f;
          }
          l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
          wait_st();
          fence_before();
          mbar_arrive(bar(P_FULL + b));
          }
        }
        if (PAIR) release();
        if (!ok) break;
        blocks_done += (uint64_t)len;
        if (!(ok = wait_warp(bar(O_FULL), o_items & 1u, g))) break;
        ++o_items;
        fence_after();
        // a row that attended to no key (its block's own row is empty in a pair) has l = 0
        const float inv = l > 0.f ? 1.0f / l : 0.f;
  #pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(t_row + C::kColO + c * 32u, ov);
          wait_ld();
          if (!stores) continue;
          uint32_t w[16];
  #pragma unroll
          for (int x = 0; x < 16; ++x)
            w[x] = pack2(__uint_as_float(ov[2 * x]) * inv, __uint_as_float(ov[2 * x + 1]) * inv);
  #pragma unroll
          for (int x = 0; x < 4; ++x) orow[c * 4 + x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
        }
        fence_before();
        mbar_arrive(bar(O_EMPTY));
        if (stores) p.lse[row] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
      }
    }
  }

  fence_before();
  __syncthreads();
  fence_after();
  if (warp == C::W_S) tmem_dealloc(tmem, C::kTmemCols);
  if (p.prof != nullptr && threadIdx.x == 0)
    atomicAdd((unsigned long long*)&p.prof[smid() % SPARSP_PROF_SLOTS],
              (unsigned long long)(globaltimer_ns() - t_start));
}

}  // namespace

int attn_fwd_tc_items_per_head(const Dims& s) { return s.Bt == 64 ? (s.nb + 1) / 2 : s.nb; }

bool attn_fwd_tc_supported(const Dims& s) {
  if (s.dtype != SPARSP_BF16 || (s.Bt != 64 && s.Bt != 128) || (s.d != 64 && s.d != 128)) return false;
  if (s.Bt == 64 && s.nb > 32 * (s.d == 64 ? Cfg<64, 64>::MAXW : Cfg<64, 128>::MAXW)) return false;
  if ((int64_t)s.B * s.H * s.N >= (int64_t)1 << 31) return false;
  int dev = 0, major = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  return major == 10;
}

namespace {

template <int BT, int D>
sparsp_status_t go_fwd(const Dims& s, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const Params& prm, cudaStream_t st) {
  using C = Cfg<BT, D>;
  auto kern = attn_fwd_tc_kernel<BT, D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes) != cudaSuccess)
    return SPARSP_ERR_CUDA;
  // all of the SM's memory as shared memory: one CTA of ~225 KB, or two of ~100 KB
  if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return SPARSP_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return SPARSP_ERR_CUDA;
  const int64_t grid = cap_grid(s, (int64_t)sms * C::kMinCtas, prm.n_items);
  kern<<<(unsigned)grid, C::THREADS, C::kSmemBytes, st>>>(tq, tk, tv, prm);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace

sparsp_status_t launch_attn_fwd_tc(const Dims& s, const __nv_bfloat16* q, const __nv_bfloat16* k,
                                   const __nv_bfloat16* v, const int32_t* row_ptr,
                                   const int32_t* col_idx, float scale, __nv_bfloat16* o,
                                   float* lse, bool raster, bool in_raster, const int32_t* items,
                                   int32_t* counter, uint64_t* prof, int32_t* d_status, cudaStream_t st) {
  const uint64_t rows = (uint64_t)s.B * s.H * s.N;
  CUtensorMap tq, tk, tv;
  if (in_raster) {
    // raster inputs: one block per 5-D box (two boxes for a pair's query tile)
    if (!make_tmap_bf16_raster(&tq, q, s) || !make_tmap_bf16_raster(&tk, k, s) || !make_tmap_bf16_raster(&tv, v, s))
      return SPARSP_ERR_CUDA;
  } else if (!make_tmap_bf16_rows(&tq, q, rows, (uint64_t)s.d, 128) ||   // Q boxes: the MMA's 128 rows
             !make_tmap_bf16_rows(&tk, k, rows, (uint64_t)s.d, (uint32_t)s.Bt) ||   // K, V: one block
             !make_tmap_bf16_rows(&tv, v, rows, (uint64_t)s.d, (uint32_t)s.Bt)) {
    return SPARSP_ERR_CUDA;
  }
  // 64-token blocks: items are pairs of query blocks, ordered by the caller
  // over the pair rows (attn_fwd_tc_items)
  const int nbp = attn_fwd_tc_items_per_head(s);
  Params prm{row_ptr, col_idx, s.N, s.nb, nbp, (int64_t)s.B * s.H * nbp, (int64_t)rows, scale * 1.4426950408889634f, o, lse,
             raster ? 1 : 0, raster_map(s), in_raster ? 1 : 0, raster_box(s), items, counter, prof, d_status};
  if (s.Bt == 128 && s.d == 128) return go_fwd<128, 128>(s, tq, tk, tv, prm, st);
  if (s.Bt == 128 && s.d == 64) return go_fwd<128, 64>(s, tq, tk, tv, prm, st);
  if (s.Bt == 64 && s.d == 128) return go_fwd<64, 128>(s, tq, tk, tv, prm, st);
  if (s.Bt == 64 && s.d == 64) return go_fwd<64, 64>(s, tq, tk, tv, prm, st);
  return SPARSP_ERR_UNSUPPORTED;
}

}  // namespace sparsp
