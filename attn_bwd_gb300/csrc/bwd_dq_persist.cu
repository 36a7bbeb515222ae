// bwd_dq_persist.cu -- the deterministic dQ pass as a persistent kernel (the one
// used for every problem without an additive bias).
//
// The arithmetic, tiles, TMEM plan and warp roles are those of bwd_dq.cu (a
// 128-row query tile of one query head per work item, walking the KV tiles it
// can see in a fixed order with dQ kept in TMEM: the query-block grid of
// flash_attention_backward.cu, rustytorch rtx-flash-attention, block "Compute
// dQ"; three tcgen05 products per KV tile):
//   G1  S  [BQ x BK] = Q  . K^T      A = Q  (smem, K-major), B = K (K-major)
//   G2  dP [BQ x BK] = dO . V^T      A = dO (smem, K-major), B = V (K-major)
//   G5  dQ [BQ x d ] += dS . K       A = dS (TMEM, 16-bit),  B = K (MN-major)
// What differs is the schedule: one CTA per SM takes work items in the launch
// order of bwd_dq.cu (the longest query tiles first) from a counter in the
// workspace, one number each time its Q/dO producer starts an item, and the
// items flow through it back to back:
//   - K and V come through their rings on a tile counter of the CTA that runs
//     across items (warp 3), so the next item's first K/V tiles load while the
//     current item is computed; the S buffers, dP and every per-tile hand-off
//     follow the same counter;
//   - the next item's Q, dO, -L*log2e and D load as soon as the current item's
//     last S and dP products have read Q and dO;
//   - the softmax warps read dQ of an item out of TMEM and release it before
//     they store it, and the next item's first dQ product waits only for that.
// Each dQ element is still summed in the same fixed order (KV tile by KV tile,
// in one CTA), so the result is bit-identical from run to run and to bwd_dq.cu.
// No additive bias (bwd_dq.cu serves it).
#include <cstdint>
#include <climits>

#include "kernels.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace fa {
namespace {

constexpr int BQ = 128;    // query rows per work item (TMEM lanes)
constexpr int BK = 128;    // KV rows per step
constexpr int KST = 3;     // K ring depth: K is held until dQ += dS K of its tile
constexpr int VST = 2;     // V ring depth: V is free once dP = dO V^T of its tile completes
constexpr int kThreads = 384;
constexpr int kRing = 8;   // item-number slots

template <int D>
struct PLayout {
  static constexpr int NH = D / 64;
  static constexpr int HALF = 128 * 128;        // one 64-column half of a 128-row tile
  static constexpr int TILE = NH * HALF;        // one 128-row tile of Q, dO, K or V
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = TILE;
  static constexpr int OFF_K = 2 * TILE;        // K stage s at OFF_K + s*TILE
  static constexpr int OFF_V = OFF_K + KST * TILE;   // V stage s at OFF_V + s*TILE
  static constexpr int OFF_LD = OFF_V + VST * TILE;  // -L*log2e, then D, of the item's rows
  static constexpr int OFF_BAR = OFF_LD + 2 * BQ * 4;
  static constexpr int NBAR = 48;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // TMEM address, abort flag, then the item ring
  static constexpr int OFF_RING = OFF_MISC + 16;
  static constexpr int TOTAL = OFF_RING + kRing * 4;
  static constexpr int ALLOC = TOTAL + 1024;    // slack for 1024-byte alignment
  static constexpr int COL_S = 0;               // buffers at 0 and BK
  static constexpr int COL_DP = 2 * BK;
  static constexpr int COL_DQ = 3 * BK;
  static_assert(COL_DQ + D <= 512, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// barrier indices; S, DS, SFREE have one barrier per S buffer (tile g uses g & 1)
enum : int {
  QFULL = 0, QEMPTY, KFULL, KEMPTY = KFULL + KST, VFULL = KEMPTY + KST, VEMPTY = VFULL + VST,
  S = VEMPTY + VST, DS = S + 2, SFREE = DS + 2, DP = SFREE + 2, DPFREE, ACC, ACCFREE, AFIN1, AFIN2,
  ITEM_FULL, ITEM_EMPTY = ITEM_FULL + kRing, BAR_END = ITEM_EMPTY + kRing
};
static_assert(BAR_END <= PLayout<128>::NBAR, "barrier count");

struct Params {
  const float* nLg;
  const float* Dv;
  void* dq;
  unsigned int* status;       // device-wide report word
  unsigned int* call_abort;   // this call's abort word (in the workspace)
  SeqMap m;
  int B, Hq, Hkv, Nq, Nkv, NqPad;   // Nq, Nkv: the longest lengths of a packed batch
  float scale, scale_log2;
  int causal;
  int items;                  // (batch, query head, query tile) work items
  unsigned int* next_item;    // workspace: items handed out so far (zero between launches)
  unsigned int* done_ctas;    // workspace: CTAs that have finished (the last one resets both)
};

// One work item: query tile i of query head h of sequence b, and the T KV tiles it sees.
struct Item {
  int b, h, hk, q0, T;
  Seq sq;
};

__device__ __forceinline__ Item decode(int it, const Params& p) {
  Item w;
  const int BH = p.B * p.Hq;
  const int nQt = (p.Nq + BQ - 1) / BQ;
  const int i = nQt - 1 - it / BH;
  const int bh = it - (it / BH) * BH;
  w.b = bh / p.Hq;
  w.h = bh - w.b * p.Hq;
  w.sq = seq_of(p.m, w.b, p.status, 43);
  w.hk = w.h / (p.Hq / p.Hkv);
  w.q0 = i * BQ;
  const int nKt = (w.sq.nk + BK - 1) / BK;
  const int qmax = min(w.q0 + BQ, w.sq.nq) - 1;
  // causal: the last key any row of this tile sees is qmax + delta (none if negative)
  const int kmax = qmax + w.sq.delta;
  w.T = w.q0 >= w.sq.nq ? 0 : p.causal ? (kmax < 0 ? 0 : min(nKt, kmax / BK + 1)) : nKt;
  return w;
}

// Bounded wait that ignores the abort flags: used only to drain work already in
// flight before the CTA releases TMEM and exits.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const Params p) {
  using L = PLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sb + L::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::OFF_RING);

  if (threadIdx.x == 0) {
    mbar_init(bar(QFULL), 1);
    mbar_init(bar(QEMPTY), 9);         // the item's last S/dP products, and each softmax warp's L/D read
    for (int s = 0; s < KST; ++s) {
      mbar_init(bar(KFULL + s), 1);
      mbar_init(bar(KEMPTY + s), 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(bar(VFULL + s), 1);
      mbar_init(bar(VEMPTY + s), 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(bar(S + j), 1);
      mbar_init(bar(DS + j), 8);       // one arrival per softmax warp
      mbar_init(bar(SFREE + j), 1);
    }
    mbar_init(bar(DP), 1);
    mbar_init(bar(DPFREE), 8);
    mbar_init(bar(ACC), 1);
    mbar_init(bar(ACCFREE), 8);        // the item's dQ read out of TMEM: one arrival per softmax warp
    mbar_init(bar(AFIN1), 1);          // warp 1's products have completed (at exit)
    mbar_init(bar(AFIN2), 1);          // warp 2's
    for (int i = 0; i < kRing; ++i) {  // item ring: slot written / read by every other role's warp
      mbar_init(bar(ITEM_FULL + i), 1);
      mbar_init(bar(ITEM_EMPTY + i), 11);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{p.status, p.call_abort, abort_flag, 1u};   // the word is zeroed by the preprocess kernel
  // The k-th item of this CTA, as every role but the fetcher sees it: -1 past the last
  // item, -2 if the wait gave up.  A whole warp calls take_item, a single lane take_item1;
  // either releases the slot (one arrival per warp).
  auto take_item = [&](int k) -> int {
    const int slot = k % kRing;
    if (!__all_sync(0xffffffffu, mbar_wait(bar(ITEM_FULL + slot), (k / kRing) & 1, wc, 44))) return -2;
    const int it = ring[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(ITEM_EMPTY + slot));
    return it;
  };
  auto take_item1 = [&](int k) -> int {
    const int slot = k % kRing;
    if (!mbar_wait(bar(ITEM_FULL + slot), (k / kRing) & 1, wc, 45)) return -2;
    const int it = ring[slot];
    mbar_arrive(bar(ITEM_EMPTY + slot));
    return it;
  };

  if (warp == 0) {
    // ================================================================ TMA producer: Q, dO, L, D
    if (lane == 0) {
      const size_t ws_rows = static_cast<size_t>(p.B) * p.Hq * p.NqPad;
      int n = 0;                 // items with work loaded so far
      // The fetcher: item numbers from the workspace counter, each taken only when this
      // producer starts the item, into the ring.
      int fetched = 0;
      bool ended = false;
      auto fetch_until = [&](int k) -> bool {
        while (!ended && fetched <= k) {
          const int slot = fetched % kRing;
          if (fetched >= kRing && !mbar_wait(bar(ITEM_EMPTY + slot), ((fetched / kRing) - 1) & 1, wc, 46))
            return false;
          int v = static_cast<int>(atomicAdd(p.next_item, 1u));
          if (v >= p.items) {
            v = -1;
            ended = true;
          }
          ring[slot] = v;
          mbar_arrive(bar(ITEM_FULL + slot));
          ++fetched;
        }
        return true;
      };
      for (int k = 0;; ++k) {
        if (!fetch_until(k)) break;
        if (k >= fetched) break;                  // past the end marker
        const int it = ring[k % kRing];          // written by this thread
        if (it < 0) break;
        const Item w = decode(it, p);
        if (w.T == 0) continue;
        const int bc = bcoord(p.m, w.b);
        const int bh = w.b * p.Hq + w.h;
        // Q and dO once the previous item's products have read them, L and D once its
        // softmax warps have
        if (n >= 1 && !mbar_wait(bar(QEMPTY), (n - 1) & 1, wc, 47)) break;
        if (!FA_BOUNDS(w.h < p.Hq && bc < batch_extent(p.m) && w.sq.q_start + w.q0 < rows_q(p.m) &&
                           static_cast<size_t>(bh) * p.NqPad + w.q0 + BQ <= ws_rows,
                       wc, 73))
          break;
        mbar_arrive_expect_tx(bar(QFULL), 2 * L::TILE + 2 * BQ * 4);
#pragma unroll
        for (int hh = 0; hh < L::NH; ++hh) {
          tma_load_4d(sb + L::OFF_Q + hh * L::HALF, &tm_q, bar(QFULL), 64 * hh, w.sq.q_start + w.q0, w.h, bc);
          tma_load_4d(sb + L::OFF_DO + hh * L::HALF, &tm_do, bar(QFULL), 64 * hh, w.sq.q_start + w.q0, w.h, bc);
        }
        const size_t row = static_cast<size_t>(bh) * p.NqPad + w.q0;
        bulk_load(sb + L::OFF_LD, p.nLg + row, BQ * 4, bar(QFULL));
        bulk_load(sb + L::OFF_LD + BQ * 4, p.Dv + row, BQ * 4, bar(QFULL));
        ++n;
      }
      // never leave a copy in flight into shared memory this CTA is about to release
      if (n > 0) drain_wait(bar(QFULL), (n - 1) & 1);
    }
  } else if (warp == 3) {
    // ================================================================ TMA producer: K, V
    // K(g) once dQ(g - KST) has read its slot; V(g) once dP(g - VST) has read its slot
    // (dP(g - 2) completes before dQ(g - 2), so the V wait never holds back K(g + 1)).
    if (lane == 0) {
      int g = 0;                 // KV tiles issued so far, over all items
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int it = take_item1(k);
        if (it < 0) break;
        const Item w = decode(it, p);
        const int bc = bcoord(p.m, w.b);
        for (int t = 0; t < w.T; ++t, ++g) {
          const int ks = g % KST, vs = g % VST;
          if (!FA_BOUNDS(w.sq.k_start + t * BK < rows_k(p.m) && w.hk < p.Hkv && bc < batch_extent(p.m), wc, 74)) {
            ok = false;
            break;
          }
          if (g >= KST && !mbar_wait(bar(KEMPTY + ks), ((g / KST) & 1) ^ 1, wc, 31)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(KFULL + ks), L::TILE);
#pragma unroll
          for (int hh = 0; hh < L::NH; ++hh)
            tma_load_4d(sb + L::OFF_K + ks * L::TILE + hh * L::HALF, &tm_k, bar(KFULL + ks), 64 * hh,
                        w.sq.k_start + t * BK, w.hk, bc);
          if (g >= VST && !mbar_wait(bar(VEMPTY + vs), ((g / VST) & 1) ^ 1, wc, 32)) {
            ++g;                 // K(g) is in flight: drain it below
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(VFULL + vs), L::TILE);
#pragma unroll
          for (int hh = 0; hh < L::NH; ++hh)
            tma_load_4d(sb + L::OFF_V + vs * L::TILE + hh * L::HALF, &tm_v, bar(VFULL + vs), 64 * hh,
                        w.sq.k_start + t * BK, w.hk, bc);
        }
      }
      // every K and V fill this warp issued has landed before the CTA exits (a V fill
      // missing after an abort only makes the drain wait run out)
      for (int u = max(0, g - KST); u < g; ++u) drain_wait(bar(KFULL + u % KST), (u / KST) & 1);
      for (int u = max(0, g - VST); u < g; ++u) drain_wait(bar(VFULL + u % VST), (u / VST) & 1);
    }
  } else if (warp == 1 || warp == 2) {
    // ================================================================ MMA issuers
    constexpr uint32_t ID_S = make_idesc_f16(128, BK, BF16, false, false);
    constexpr uint32_t ID_Q = make_idesc_f16(128, D, BF16, false, true);
    const uint32_t tdP = tmem + L::COL_DP, tdQ = tmem + L::COL_DQ;
    const uint64_t dQ_k = sw128_desc(sb + L::OFF_Q, 16, 1024), dO_k = sw128_desc(sb + L::OFF_DO, 16, 1024);
    auto s_buf = [&](int g) -> uint32_t { return tmem + L::COL_S + (g & 1) * BK; };
    auto k_tile = [&](int g) -> uint32_t { return sb + L::OFF_K + (g % KST) * L::TILE; };
    auto v_tile = [&](int g) -> uint32_t { return sb + L::OFF_V + (g % VST) * L::TILE; };
    // K-major step ks (16 elements of d): 64-column half ks/4, 32 bytes per step inside it
    auto kstep = [](int ks) -> uint64_t {
      return static_cast<uint64_t>(((ks >> 2) * L::HALF + (ks & 3) * 32) >> 4);
    };
    auto wait = [&](uint32_t bb, uint32_t parity, uint32_t site) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bb, parity, wc, site));
    };
    int n = 0, g = 0;            // items with work, KV tiles (over all items)
    bool ok = true;
    if (warp == 1) {
      for (int k = 0; ok; ++k) {
        const int it = take_item(k);
        if (it < 0) break;
        const Item w = decode(it, p);
        if (w.T == 0) continue;
        if (!wait(bar(QFULL), n & 1, 33)) break;
        for (int t = 0; t < w.T; ++t, ++g) {
          if (!wait(bar(KFULL + g % KST), (g / KST) & 1, 34)) { ok = false; break; }
          if (g >= 2 && !wait(bar(SFREE + (g & 1)), ((g - 2) >> 1) & 1, 35)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dK_k = sw128_desc(k_tile(g), 16, 1024), dV_k = sw128_desc(v_tile(g), 16, 1024);
          // G1: S = Q K^T into buffer g & 1
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) umma_ss_warp(s_buf(g), dQ_k + kstep(ks), dK_k + kstep(ks), ID_S, ks > 0);
          umma_commit_warp(bar(S + (g & 1)));
          // G2: dP = dO V^T, once the softmax groups have loaded dP of the previous tile
          if (!wait(bar(VFULL + g % VST), (g / VST) & 1, 36)) { ok = false; break; }
          if (g >= 1 && !wait(bar(DPFREE), (g - 1) & 1, 37)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) umma_ss_warp(tdP, dO_k + kstep(ks), dV_k + kstep(ks), ID_S, ks > 0);
          umma_commit_warp(bar(DP));
          umma_commit_warp(bar(VEMPTY + g % VST));     // V(g) is read by G2(g) only
        }
        if (!ok) break;
        umma_commit_warp(bar(QEMPTY));   // the item's S and dP products have read Q and dO
        ++n;
      }
      umma_commit_warp(bar(AFIN1));      // this warp's MMAs complete before TMEM is released
      drain_wait(bar(AFIN1), 0);
    } else {
      for (int k = 0; ok; ++k) {
        const int it = take_item(k);
        if (it < 0) break;
        const Item w = decode(it, p);
        if (w.T == 0) continue;
        for (int t = 0; t < w.T; ++t, ++g) {
          // the item's first product starts a new dQ sum: the previous item's must have been read out
          if (t == 0 && n >= 1 && !wait(bar(ACCFREE), (n - 1) & 1, 38)) { ok = false; break; }
          // G5: dQ += dS K  (dS, 16-bit, packed into the first half of each group's
          // 64 columns of the S buffer; K read MN-major)
          if (!wait(bar(DS + (g & 1)), (g >> 1) & 1, 39)) { ok = false; break; }
          tc_fence_after();
          const uint64_t dK_mn = sw128_desc(k_tile(g), L::HALF, 1024);
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            umma_ts_warp(tdQ, s_buf(g) + 64 * (ks >> 2) + 8 * (ks & 3),
                         dK_mn + static_cast<uint64_t>((ks * 2048) >> 4), ID_Q, (t > 0 || ks > 0));
          umma_commit_warp(bar(SFREE + (g & 1)));
          // K(g): G1(g) has completed (dS(g) depends on it); G5(g) is tracked here
          umma_commit_warp(bar(KEMPTY + g % KST));
        }
        if (!ok) break;
        umma_commit_warp(bar(ACC));
        ++n;
      }
      umma_commit_warp(bar(AFIN2));
      drain_wait(bar(AFIN2), 0);
    }
  } else if (warp >= 4) {
    // ================================================================ softmax / dS groups, epilogue
    const int grp = (warp - 4) >> 2;                    // KV columns [64 grp, 64 grp + 64)
    const int r = threadIdx.x - 128 - 128 * grp;       // query row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tdP = tmem + lane_off + L::COL_DP + 64 * grp;
    const float* LD = reinterpret_cast<const float*>(smem + L::OFF_LD);
    const uint64_t sc2 = f2_bits(p.scale_log2, p.scale_log2);
    int n = 0, g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int it = take_item(k);
      if (it < 0) break;
      const Item w = decode(it, p);
      const Seq& sq = w.sq;
      const int q = w.q0 + r;
      uint8_t* out = reinterpret_cast<uint8_t*>(p.dq) + at(p.m.st.dq, p.m, w.b, w.h, sq.q_start + q) * 2;
      const bool row_ok = q < sq.nq && FA_BOUNDS(sq.q_start + q < rows_q(p.m), wc, 75);
      if (w.T == 0) {
        // rows that see no key: dQ = 0
        if (row_ok)
          for (int ch = 0; ch < D / 64; ++ch) {
            const int col = (D / 2) * grp + 32 * ch;
            uint4* d4 = reinterpret_cast<uint4*>(out + col * 2);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              if (col + 8 * k4 < p.m.d) d4[k4] = make_uint4(0u, 0u, 0u, 0u);
          }
        continue;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(QFULL), n & 1, wc, 48))) break;
      const uint64_t nl2 = f2_bits(LD[r], LD[r]);                  // -L*log2(e) of this query row
      const uint64_t dd2 = f2_bits(LD[BQ + r], LD[BQ + r]);        // D of this query row
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(QEMPTY));       // L and D are in registers
      for (int t = 0; t < w.T; ++t, ++g) {
        const int kv0 = t * BK;
        // columns c >= lim are masked: past the end of K/V, or (causal) after query q
        int lim = sq.nk - kv0 - 64 * grp;
        if (p.causal) lim = min(lim, q + sq.delta - kv0 - 64 * grp + 1);
        const bool need_mask = __any_sync(0xffffffffu, lim < 64);
        const uint32_t tS = tmem + lane_off + L::COL_S + (g & 1) * BK + 64 * grp;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(DP), g & 1, wc, 49))) { ok = false; break; }
        tc_fence_after();
        uint32_t dr[64];
        tmem_ld_x32(tdP, *reinterpret_cast<uint32_t(*)[32]>(dr));
        tmem_ld_x32(tdP + 32, *reinterpret_cast<uint32_t(*)[32]>(dr + 32));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(DPFREE));       // the dP buffer may take the next tile's G2
        if (!__all_sync(0xffffffffu, mbar_wait(bar(S + (g & 1)), (g >> 1) & 1, wc, 50))) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t sr[32], pk[16];
          tmem_ld_x32(tS + 32 * ch, sr);
          tmem_ld_wait();
#pragma unroll
          for (int c2 = 0; c2 < 16; ++c2) {
            const int c = 32 * ch + 2 * c2;
            const float2 x =
                f2_split(fma_f32x2(f2_bits(__uint_as_float(sr[2 * c2]), __uint_as_float(sr[2 * c2 + 1])), sc2, nl2));
            float p0 = ex2_approx(x.x);
            float p1 = ex2_approx(x.y);
            if (need_mask) {
              if (c >= lim) p0 = 0.f;
              if (c + 1 >= lim) p1 = 0.f;
            }
            const float2 ds = f2_split(mul_f32x2(f2_bits(p0, p1),
                sub_f32x2(f2_bits(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), dd2)));
            pk[c2] = pack2<BF16>(ds.x, ds.y);
          }
          // columns [16ch, 16ch+16) of this group's S columns were already read
          tmem_st_x16(tS + 16 * ch, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(DS + (g & 1)));
      }
      if (!ok) break;
      // ---- epilogue of the item: read dQ out of TMEM, release it, then store scale * dQ
      // (group grp writes columns [D/2 grp, D/2 (grp + 1)))
      if (!__all_sync(0xffffffffu, mbar_wait(bar(ACC), n & 1, wc, 11))) break;
      tc_fence_after();
      uint32_t v[D / 64][32];
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) tmem_ld_x32(tmem + lane_off + L::COL_DQ + (D / 2) * grp + 32 * ch, v[ch]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(ACCFREE));
      ++n;
      if (row_ok && *abort_flag == 0) {
#pragma unroll
        for (int ch = 0; ch < D / 64; ++ch) {
          const int col = (D / 2) * grp + 32 * ch;
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[c] = pack2<BF16>(__uint_as_float(v[ch][2 * c]) * p.scale, __uint_as_float(v[ch][2 * c + 1]) * p.scale);
          uint4* d4 = reinterpret_cast<uint4*>(out + col * 2);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            if (col + 8 * k4 < p.m.d) d4[k4] = make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // every CTA has stopped fetching when it gets here: the last one resets the counters
  // for the next launch on this workspace
  if (threadIdx.x == 0 && atomicAdd(p.done_ctas, 1u) == gridDim.x - 1) {
    atomicExch(p.next_item, 0u);
    atomicExch(p.done_ctas, 0u);
  }
}

template <int D, bool BF16>
cudaError_t launch_t(const DqArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk,
                     const CUtensorMap& tv, cudaStream_t stream) {
  using L = PLayout<D>;
  auto kern = bwd_dq_persist_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  Params p;
  p.nLg = a.ws.nLg;
  p.Dv = a.ws.Dv;
  p.dq = a.dq;
  p.status = a.status;
  p.call_abort = a.ws.abort;
  p.B = a.pb.B; p.Hq = a.pb.Hq; p.Hkv = a.pb.Hkv; p.Nq = a.pb.Nq; p.Nkv = a.pb.Nkv; p.NqPad = a.pb.NqPad;
  p.scale = a.pb.scale;
  p.scale_log2 = a.pb.scale * 1.4426950408889634f;
  p.causal = a.pb.causal;
  p.m = seq_map(a.pb);
  const long long items = static_cast<long long>((a.pb.Nq + BQ - 1) / BQ) * a.pb.B * a.pb.Hq;
  p.items = static_cast<int>(items);
  p.next_item = a.ws.abort + 3;
  p.done_ctas = a.ws.abort + 4;
  const long long grid = items < sm_count() ? items : sm_count();
  kern<<<static_cast<unsigned>(grid), kThreads, L::ALLOC, stream>>>(tq, tdo, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_persist(const DqArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                                  const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  if (a.pb.d > 64)
    return a.pb.bf16 ? launch_t<128, true>(a, tq, tdo, tk, tv, stream) : launch_t<128, false>(a, tq, tdo, tk, tv, stream);
  return a.pb.bf16 ? launch_t<64, true>(a, tq, tdo, tk, tv, stream) : launch_t<64, false>(a, tq, tdo, tk, tv, stream);
}

}  // namespace fa
