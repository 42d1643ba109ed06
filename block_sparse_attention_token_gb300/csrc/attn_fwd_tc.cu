// Step 5a, bf16, Bt and d in {64, 128} on sm_103a: block-sparse flash-attention
// forward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA). The query
// tile is always the MMA's 128 rows; with 64-token blocks its second half holds
// the next block's rows, computed and not stored.
//
// One persistent CTA per SM, 7 warps:
//   warp 4     producer: pulls (b, h, query block) items longest-first through
//              an atomic counter, validates the CSR row, publishes the item in
//              a shared-memory ring, and TMA-loads Q_i and the selected K_j / V_j
//              tiles (128 x 128 bf16, two 64-column boxes with 128-byte swizzle)
//              into 3-stage K and V rings, addressed through
//              the CSR (row coordinate = bh*N + j*128).
//   warp 5     S issuer: S_j = Q K_j^T into one of two TMEM S buffers (M=N=128,
//              K=16 per instruction, both operands K-major from shared memory).
//   warp 6     PV issuer: O += P_j V_j (A = P_j read from TMEM as packed bf16,
//              B = V_j MN-major from shared memory).
//              The two GEMM streams are issued by different warps so that a
//              wait in one (for P, or for a free S buffer) never holds back the
//              other; each warp runs uniformly and one elected lane issues
//              tcgen05.mma / tcgen05.commit.
//   warps 0-3  softmax and epilogue: thread t owns query row t = TMEM lane t.
//              It reads its S row from TMEM with the sm_103 load-with-maximum
//              (tcgen05.ld.red: each 32-column load also returns the maximum of
//              the 32 values, so the row max costs no extra instructions), keeps
//              a running max m and sum l in
//              base 2, writes P = exp2(S*scale*log2e - m) as bf16 into TMEM, and
//              rescales its O row in TMEM only when the row max grows by more
//              than 8 (a factor 256); otherwise the stale max is kept, which
//              leaves the result unchanged up to rounding because O and l use
//              the same reference. At the end of the row: O / l to global
//              memory, LSE = (m + log2 l) ln 2.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256,384), P0 [384,448),
// P1 [448,512). Every mbarrier wait is bounded (2 s); on expiry the CTA sets
// SPARSP_ERR_TIMEOUT, all roles leave their loops, copies and MMAs in flight
// are drained with a second bounded wait, and TMEM is released.
#include "tc_helpers.cuh"

namespace sparsp {
namespace {

using namespace tc;

constexpr int kNK = 3, kNV = 3, kNI = 4;
constexpr int kThreads = 224;   // 4 softmax warps, producer, S issuer, PV issuer
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;
enum Bar {
  Q_FULL = 0, Q_EMPTY, K_FULL, K_EMPTY = K_FULL + kNK, V_FULL = K_EMPTY + kNK, V_EMPTY = V_FULL + kNV,
  S_FULL = V_EMPTY + kNV, S_FREE = S_FULL + 2, P_FULL = S_FREE + 2, PV_DONE = P_FULL + 2, O_FULL = PV_DONE + 2,
  O_EMPTY,
  I_FULL, I_EMPTY = I_FULL + kNI, TEAR = I_EMPTY + kNI, TEAR_PV, NBAR
};
// Tile geometry for key blocks of BT tokens and head dimension D. The query
// tile is always 128 rows (the MMA's M; the 128 TMEM lanes): with BT = 64 the
// rows past the block belong to the next block (or are zero past the tensor's
// end), are computed and never stored. Tiles are TMA'd as 64-column boxes of
// 128-byte rows with 128-byte swizzle.
template <int BT_, int D_>
struct Cfg {
  static constexpr int BT = BT_, D = D_, QR = 128;
  static constexpr int NBOX = D / 64;                     // 64-column boxes per row tile
  static constexpr uint32_t kQBox = QR * 128, kKBox = BT * 128;
  static constexpr uint32_t kQTile = kQBox * NBOX, kKTile = kKBox * NBOX;
  static constexpr uint32_t kOffK = kQTile, kOffV = kOffK + kNK * kKTile, kOffBar = kOffV + kNV * kKTile;
  static constexpr uint32_t kOffRing = kOffBar + 8 * NBAR;
  static constexpr uint32_t kOffMisc = kOffRing + 8 * kNI;
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;   // + alignment slack
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
  int64_t n_items;
  float scale_log2;
  __nv_bfloat16* o;
  float* lse;
  // raster output: O row (b, h, token) at ((b*N + n)*H + h)*d with n the token's
  // raster index (t slowest, x fastest); otherwise block order like Q
  int raster, H, Y, X, ta, tb, tc, nY, nX;
  const int32_t* items;
  int32_t* counter;
  uint64_t* prof;
  int32_t* d_status;
};

template <int BT, int D>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  using C = Cfg<BT, D>;
  const uint32_t sQ = base, sK = base + C::kOffK, sV = base + C::kOffV;
  auto bar = [&](int idx) -> uint32_t { return base + C::kOffBar + 8u * (uint32_t)idx; };
  volatile int2* ring = reinterpret_cast<volatile int2*>(gbase + C::kOffRing);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffMisc);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(gbase + C::kOffMisc + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t t_start = globaltimer_ns();

  if (threadIdx.x == 0) {
    mbar_init(bar(Q_FULL), 1);
    mbar_init(bar(Q_EMPTY), 1);
    for (int s = 0; s < kNK; ++s) {
      mbar_init(bar(K_FULL + s), 1);
      mbar_init(bar(K_EMPTY + s), 1);
    }
    for (int s = 0; s < kNV; ++s) {
      mbar_init(bar(V_FULL + s), 1);
      mbar_init(bar(V_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(S_FULL + b), 1);
      mbar_init(bar(S_FREE + b), 128);
      mbar_init(bar(P_FULL + b), 128);
    }
    mbar_init(bar(PV_DONE), 1);
    mbar_init(bar(PV_DONE + 1), 1);
    mbar_init(bar(O_FULL), 1);
    mbar_init(bar(O_EMPTY), 128);
    for (int r = 0; r < kNI; ++r) {
      mbar_init(bar(I_FULL + r), 1);
      mbar_init(bar(I_EMPTY + r), 6);
    }
    mbar_init(bar(TEAR), 1);
    mbar_init(bar(TEAR_PV), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
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
  const int nb = p.nb;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    uint32_t it_fill = 0, q_fill = 0, k_fill = 0, v_fill = 0;
    for (;;) {
      int32_t slot = 0;
      if (lane == 0) slot = atomicAdd(p.counter, 1);
      slot = __shfl_sync(0xffffffffu, slot, 0);
      int32_t item = -1, len = -2;
      if (slot < p.n_items) {
        item = p.items[slot];
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
      const int ri = (int)(it_fill % kNI);
      if (!wait_warp(bar(I_EMPTY + ri), ((it_fill / kNI) & 1u) ^ 1u, g)) break;
      if (lane == 0) {
        ring[ri].x = item;
        ring[ri].y = len;
        mbar_arrive(bar(I_FULL + ri));
      }
      __syncwarp();
      ++it_fill;
      if (len == -2) break;
      if (len <= 0) continue;
      const int64_t bh = item / nb;
      const int i = item % nb;
      const int32_t yq = (int32_t)(bh * p.N + (int64_t)i * BT);
      if (!wait_warp(bar(Q_EMPTY), (q_fill & 1u) ^ 1u, g)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(Q_FULL), C::kQTile);
#pragma unroll
        for (int h = 0; h < C::NBOX; ++h) tma_load_2d(sQ + h * C::kQBox, &tq, bar(Q_FULL), 64 * h, yq);
      }
      ++q_fill;
      const int32_t e0 = p.row_ptr[item];
      bool ok = true;
      for (int e = 0; e < len && ok; ++e) {
        const int32_t j = p.col_idx[e0 + e];
        const int32_t yk = (int32_t)(bh * p.N + (int64_t)j * BT);
        const uint32_t ks = k_fill % kNK;
        if (!(ok = wait_warp(bar(K_EMPTY + ks), ((k_fill / kNK) & 1u) ^ 1u, g))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(K_FULL + ks), C::kKTile);
#pragma unroll
          for (int h = 0; h < C::NBOX; ++h)
            tma_load_2d(sK + ks * C::kKTile + h * C::kKBox, &tk, bar(K_FULL + ks), 64 * h, yk);
        }
        ++k_fill;
        const uint32_t vs = v_fill % kNV;
        if (!(ok = wait_warp(bar(V_EMPTY + vs), ((v_fill / kNV) & 1u) ^ 1u, g))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(V_FULL + vs), C::kKTile);
#pragma unroll
          for (int h = 0; h < C::NBOX; ++h)
            tma_load_2d(sV + vs * C::kKTile + h * C::kKBox, &tv, bar(V_FULL + vs), 64 * h, yk);
        }
        ++v_fill;
      }
      if (!ok) break;
    }
    if (*abort_flag && lane == 0) {
      // drain copies still in flight before the shared memory goes away
      if (q_fill) wait_raw(bar(Q_FULL), (q_fill - 1) & 1u, kDrainNs);
      for (uint32_t s = 0; s < kNK; ++s)
        if (k_fill > s) wait_raw(bar(K_FULL + s), ((k_fill - 1 - s) / kNK) & 1u, kDrainNs);
      for (uint32_t s = 0; s < kNV; ++s)
        if (v_fill > s) wait_raw(bar(V_FULL + s), ((v_fill - 1 - s) / kNV) & 1u, kDrainNs);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ S = Q K^T issuer
    constexpr uint32_t idS = idesc_bf16(128, BT, 0, 0);
    uint32_t it_use = 0, q_use = 0, k_use = 0, s_issue = 0;
    bool issued_any = false;
    for (;;) {
      const int ri = (int)(it_use % kNI);
      if (!wait_warp(bar(I_FULL + ri), (it_use / kNI) & 1u, g)) break;
      const int2 ent = make_int2(ring[ri].x, ring[ri].y);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(I_EMPTY + ri));
      ++it_use;
      if (ent.y == -2) break;
      if (ent.y <= 0) continue;
      const int len = ent.y;
      if (!wait_warp(bar(Q_FULL), q_use & 1u, g)) break;
      ++q_use;
      bool ok = true;
      for (int e = 0; e < len; ++e) {
        const uint32_t b = s_issue & 1u, ks = k_use % kNK;
        if (!(ok = wait_warp(bar(S_FREE + b), ((s_issue >> 1) & 1u) ^ 1u, g))) break;
        if (!(ok = wait_warp(bar(K_FULL + ks), (k_use / kNK) & 1u, g))) break;
        fence_after();
        const uint32_t kb = sK + ks * C::kKTile;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // k-step kk: 16 columns = 32 bytes into the row, in box kk / 4
            const uint32_t offq = (uint32_t)(kk >> 2) * C::kQBox + (uint32_t)(kk & 3) * 32u;
            const uint32_t offk = (uint32_t)(kk >> 2) * C::kKBox + (uint32_t)(kk & 3) * 32u;
            mma_ss(tmem + kColS + b * 128u, smem_desc(sQ + offq, 16, 1024, kSwizzle128B),
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
  } else if (warp == 6) {
    // ------------------------------------------------------------ O += P V issuer
    constexpr uint32_t idO = idesc_bf16(128, D, 0, 1);
    uint32_t it_use = 0, v_use = 0, pv = 0, o_items = 0;
    bool issued_any = false;
    for (;;) {
      const int ri = (int)(it_use % kNI);
      if (!wait_warp(bar(I_FULL + ri), (it_use / kNI) & 1u, g)) break;
      const int2 ent = make_int2(ring[ri].x, ring[ri].y);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(I_EMPTY + ri));
      ++it_use;
      if (ent.y == -2) break;
      if (ent.y <= 0) continue;
      const int len = ent.y;
      bool ok = true;
      for (int e = 0; e < len; ++e) {
        const uint32_t b = pv & 1u, vs = v_use % kNV;
        if (!(ok = wait_warp(bar(V_FULL + vs), (v_use / kNV) & 1u, g))) break;
        if (!(ok = wait_warp(bar(P_FULL + b), (pv >> 1) & 1u, g))) break;
        if (e == 0 && !(ok = wait_warp(bar(O_EMPTY), (o_items & 1u) ^ 1u, g))) break;
        fence_after();
        const uint32_t vb = sV + vs * C::kKTile;
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BT / 16; ++kk)
            mma_ts(tmem + kColO, tmem + kColP + b * 64u + (uint32_t)kk * 8u,
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
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t t_row = tmem + lane_base;
    uint32_t it_use = 0, s_use = 0, o_items = 0;
    uint64_t blocks_done = 0;
    const float sl2 = p.scale_log2;
    for (;;) {
      const int ri = (int)(it_use % kNI);
      if (!wait_warp(bar(I_FULL + ri), (it_use / kNI) & 1u, g)) break;
      const int2 ent = make_int2(ring[ri].x, ring[ri].y);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(I_EMPTY + ri));
      ++it_use;
      if (ent.y == -2) break;
      if (ent.y == -1) continue;
      const int64_t item = ent.x;
      const int64_t bh = item / nb;
      const int i = (int)(item % nb);
      const int64_t row = bh * p.N + (int64_t)i * BT + threadIdx.x;
      const bool stores = threadIdx.x < BT;   // rows past the block are computed, never stored
      int64_t orow_idx = row;
      if (p.raster && stores) {
        // tile i = (bt, by, bx) block-raster; token o = (it, iy, ix) raster inside the tile
        const int o = threadIdx.x, tbc = p.tb * p.tc;
        const int bx = i % p.nX, by = (i / p.nX) % p.nY, bt = i / (p.nX * p.nY);
        const int it = o / tbc, iy = (o - it * tbc) / p.tc, ix = o - it * tbc - iy * p.tc;
        const int64_t n = ((int64_t)bt * p.ta + it) * p.Y * p.X + ((int64_t)by * p.tb + iy) * p.X +
                          (int64_t)bx * p.tc + ix;
        orow_idx = ((bh / p.H) * p.N + n) * p.H + bh % p.H;
      }
      uint4* orow = reinterpret_cast<uint4*>(p.o + orow_idx * D);
      const int len = ent.y;
      if (len == 0) {
        if (stores) {
#pragma unroll
          for (int c = 0; c < D / 8; ++c) orow[c] = make_uint4(0, 0, 0, 0);
          p.lse[row] = -INFINITY;
        }
        continue;
      }
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int e = 0; e < len; ++e) {
        const uint32_t b = s_use & 1u;
        if (!(ok = wait_warp(bar(S_FULL + b), (s_use >> 1) & 1u, g))) break;
        fence_after();
        uint32_t s[BT];
        float cm[BT / 32];   // the maximum of each 32-column load (exact, as any order of max)
#pragma unroll
        for (int c = 0; c < BT / 32; ++c) cm[c] = tmem_ld32_max(t_row + kColS + b * 128u + c * 32u, s + 32 * c);
        wait_ld();
        fence_before();
        mbar_arrive(bar(S_FREE + b));
        ++s_use;
        float mx = cm[0];
#pragma unroll
        for (int c = 1; c < BT / 32; ++c) mx = fmaxf(mx, cm[c]);
        const float m_new = fmaxf(m, mx * sl2);
        if (e == 0) {
          m = m_new;
        } else if (__any_sync(0xffffffffu, m_new > m + kRescaleThreshold)) {
          // O must not change under the PV of block g-1 (g = global block index)
          const uint64_t gp = blocks_done + e - 1;
          if (!(ok = wait_warp(bar(PV_DONE + (uint32_t)(gp & 1u)), (uint32_t)((gp >> 1) & 1u), g))) break;
          fence_after();
          const float f = ex2f(m - m_new);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(t_row + kColO + c * 32u, o);
            wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
            tmem_st32(t_row + kColO + c * 32u, o);
          }
          wait_st();
          l *= f;
          m = m_new;
        }
        uint32_t pk[BT / 2];
        float rs[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) rs[u] = 0.f;
#pragma unroll
        for (int c = 0; c < BT / 2; ++c) {
          const float p0 = ex2f(fmaf(__uint_as_float(s[2 * c]), sl2, -m));
          const float p1 = ex2f(fmaf(__uint_as_float(s[2 * c + 1]), sl2, -m));
          rs[c & 7] += p0 + p1;
          pk[c] = pack2(p0, p1);
        }
        l += ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
        // P buffer b was last read by the PV of block g-2
        const uint64_t gb = blocks_done + e;
        if (gb >= 2) {
          if (!(ok = wait_warp(bar(PV_DONE + b), (uint32_t)(((gb - 2) >> 1) & 1u), g))) break;
          fence_after();
        }
#pragma unroll
        for (int c = 0; c < BT / 64; ++c) tmem_st32(t_row + kColP + b * 64u + 32u * c, pk + 32 * c);
        wait_st();
        fence_before();
        mbar_arrive(bar(P_FULL + b));
      }
      if (!ok) break;
      blocks_done += (uint64_t)len;
      if (!wait_warp(bar(O_FULL), o_items & 1u, g)) break;
      ++o_items;
      fence_after();
      const float inv = 1.0f / l;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(t_row + kColO + c * 32u, o);
        wait_ld();
        if (!stores) continue;
        uint32_t w[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          w[x] = pack2(__uint_as_float(o[2 * x]) * inv, __uint_as_float(o[2 * x + 1]) * inv);
#pragma unroll
        for (int x = 0; x < 4; ++x) orow[c * 4 + x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
      }
      fence_before();
      mbar_arrive(bar(O_EMPTY));
      if (stores) p.lse[row] = (m + log2f(l)) * 0.69314718055994531f;
    }
  }

  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
  if (p.prof != nullptr && threadIdx.x == 0)
    atomicAdd((unsigned long long*)&p.prof[smid() % SPARSP_PROF_SLOTS],
              (unsigned long long)(globaltimer_ns() - t_start));
}

}  // namespace

bool attn_fwd_tc_supported(const Dims& s) {
  if (s.dtype != SPARSP_BF16 || (s.Bt != 64 && s.Bt != 128) || (s.d != 64 && s.d != 128)) return false;
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
  const int sms = device_sm_count();
  if (sms <= 0) return SPARSP_ERR_CUDA;
  const int64_t grid = cap_grid(s, sms, s.rows());
  kern<<<(unsigned)grid, kThreads, C::kSmemBytes, st>>>(tq, tk, tv, prm);
  SPARSP_LAUNCH_CHECK();
  return SPARSP_OK;
}

}  // namespace

sparsp_status_t launch_attn_fwd_tc(const Dims& s, const __nv_bfloat16* q, const __nv_bfloat16* k,
                                   const __nv_bfloat16* v, const int32_t* row_ptr,
                                   const int32_t* col_idx, float scale, __nv_bfloat16* o,
                                   float* lse, bool raster, const int32_t* items, int32_t* counter,
                                   uint64_t* prof, int32_t* d_status, cudaStream_t st) {
  const uint64_t rows = (uint64_t)s.B * s.H * s.N;
  CUtensorMap tq, tk, tv;
  // Q boxes are 128 rows (the MMA's M) whatever the block size; K and V boxes one block
  if (!make_tmap_bf16_rows(&tq, q, rows, (uint64_t)s.d, 128) ||
      !make_tmap_bf16_rows(&tk, k, rows, (uint64_t)s.d, (uint32_t)s.Bt) ||
      !make_tmap_bf16_rows(&tv, v, rows, (uint64_t)s.d, (uint32_t)s.Bt))
    return SPARSP_ERR_CUDA;
  Params prm{row_ptr, col_idx, s.N, s.nb, s.rows(), scale * 1.4426950408889634f, o, lse,
             raster ? 1 : 0, s.H, s.Y, s.X, s.ta, s.tb, s.tc, s.nY, s.nX, items, counter, prof, d_status};
  if (s.Bt == 128 && s.d == 128) return go_fwd<128, 128>(s, tq, tk, tv, prm, st);
  if (s.Bt == 128 && s.d == 64) return go_fwd<128, 64>(s, tq, tk, tv, prm, st);
  if (s.Bt == 64 && s.d == 128) return go_fwd<64, 128>(s, tq, tk, tv, prm, st);
  if (s.Bt == 64 && s.d == 64) return go_fwd<64, 64>(s, tq, tk, tv, prm, st);
  return SPARSP_ERR_UNSUPPORTED;
}

}  // namespace sparsp
