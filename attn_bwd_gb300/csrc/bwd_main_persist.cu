// bwd_main_persist.cu -- the main backward kernel as a persistent kernel (the one
// used for every problem without an additive bias).
//
// The arithmetic, tiles, TMEM plan and warp roles are those of bwd_main.cu (a
// 128-row KV tile of one key/value head per work item, walking the 64-row query
// tiles of every query head of its GQA group; five tcgen05 products per tile;
// the sequence-parallel scheme of triton #1806, "Minimal Repro", with the
// per-tile arithmetic of flash_attention_backward.cu).  What differs is the
// schedule: one CTA per SM takes work items c, c + grid, c + 2 grid, ... in the
// launch order of bwd_main.cu (chunks of (batch, kv-head) groups, tile-major,
// the longest first), fetching the next item number from a counter in the
// workspace as the hardware scheduler would start the next CTA, and the items
// flow through it back to back:
//   - the Q/dO ring, the two S^T buffers and every per-tile hand-off keep
//     running across items (their phases follow a tile counter of the CTA), so
//     the producer loads the next item's first Q/dO tiles while the current
//     item is computed;
//   - K and V of the next item are loaded (by a warp of their own) as soon as
//     the current item's last products have read them, or, for d <= 64, where
//     two K/V buffers fit next to the ring, while the current item is computed;
//   - the dQ warps (idle between their reductions, and in deterministic mode
//     altogether) read an item's dV, then dK, out of TMEM and store them,
//     while the softmax warps already work on the next item's first tiles;
//     the next item's first dV (dK) product waits only for the dV (dK)
//     read-out.
// With short items (a 256-token head walks 4 query tiles per KV tile) the
// set-up, load latency and epilogue of every item weigh on its time as much as
// its tiles.  The item numbers reach the CTA's roles through a ring of eight
// slots in shared memory, filled by the Q/dO producer as it starts each item.
// No additive bias (bwd_main.cu serves it).
#include <cstdint>
#include <climits>

#include "kernels.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace fa {
namespace {

constexpr int BN = kMainBN;   // KV rows per work item (TMEM lanes)
constexpr int BM = kMainBM;   // query rows per tile
constexpr int QST = 4;        // Q/dO ring depth
constexpr int kThreads = 512;
constexpr int kGroupChunk = 32;   // (batch, kv-head) groups per launch-order chunk

template <int D>
struct PLayout {
  static constexpr int NH = D / 64;               // 64-column halves of a row
  static constexpr int KHALF = BN * 128;          // bytes of one half of a K/V tile
  static constexpr int QHALF = BM * 128;          // bytes of one half of a Q/dO tile
  static constexpr int KV_BYTES = NH * KHALF;     // one K (or V) tile
  static constexpr int Q_BYTES = NH * QHALF;
  // K/V buffers: two where they fit next to a 4-stage Q/dO ring (d <= 64), so that the
  // next item's K and V load while the current item is computed; else one
  static constexpr int KVBUF = D <= 64 ? 2 : 1;
  static constexpr int OFF_KV = 0;                // buffer k: K at OFF_KV + 2k KV_BYTES, V after it
  static constexpr int OFF_Q = 2 * KVBUF * KV_BYTES;
  static constexpr int OFF_DO = OFF_Q + QST * Q_BYTES;
  static constexpr int OFF_DS = OFF_DO + QST * Q_BYTES;
  static constexpr int DS_BYTES = BN * BM * 2;    // dS^T, 128 rows x 128 B
  static constexpr int OFF_LD = OFF_DS + DS_BYTES;
  static constexpr int LD_BYTES = 2 * BM * 4;     // -L*log2e and D of one tile
  static constexpr int OFF_BAR = OFF_LD + QST * LD_BYTES;
  static constexpr int NBAR = 48;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // TMEM address, abort flag, then the item ring
  static constexpr int OFF_RING = OFF_MISC + 16;
  static constexpr int TOTAL = OFF_RING + 8 * 4;
  static constexpr int ALLOC = TOTAL + 1024;      // slack for 1024-byte alignment
  // TMEM columns, as in bwd_main.cu
  static constexpr int COL_DK = 0;
  static constexpr int COL_DV = D;
  static constexpr int COL_S = 2 * D;             // buffers at COL_S and COL_S + BM
  static constexpr int COL_DP = 2 * D + 2 * BM;
  static constexpr int COL_DQ = 2 * D + 3 * BM;
  static_assert(COL_DQ + BM <= 512, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// barrier indices; S, P, SFREE have one barrier per S^T buffer (tile g uses g & 1),
// KVFULL, KVEMPTY one per K/V buffer (item n uses n % KVBUF)
enum : int {
  KVFULL = 0, KVEMPTY = 2, QFULL = 4, QEMPTY = QFULL + QST, S = QEMPTY + QST, P = S + 2, SFREE = P + 2,
  DP = SFREE + 2, DPFREE, DS, DQFULL, DQEMPTY, DSFREE, ACC, ACCFREE_V, ACCFREE_K, AFIN1, AFIN2,
  ITEM_FULL, ITEM_EMPTY = ITEM_FULL + 8, BAR_END = ITEM_EMPTY + 8
};
static_assert(BAR_END <= PLayout<128>::NBAR, "barrier count");

struct Params {
  const float* nLg;
  const float* Dv;
  float* dq_acc;
  void* dk;
  void* dv;
  unsigned int* status;       // device-wide report word
  unsigned int* call_abort;   // this call's abort word (in the workspace)
  SeqMap m;
  int B, Hq, Hkv, Nq, Nkv, NqPad;   // Nq, Nkv: the longest lengths of a packed batch
  float scale, scale_log2;
  int causal;
  int items;                  // (batch, kv-head, KV tile) work items
  unsigned int* next_item;    // workspace: items handed out so far (zero between launches)
  unsigned int* done_ctas;    // workspace: CTAs that have finished (the last one resets both)
};

// One work item: KV tile j of key/value head hkv of sequence b, and the query
// tiles [i0, nQt) of each of the G query heads of its group (T tiles in all,
// head-major).  Decoded the same way by every warp.
struct Item {
  int j, b, hkv, kv0, i0, nQt, per_head, T;
  Seq sq;
};

__device__ __forceinline__ Item decode(int it, const Params& p, int G) {
  Item w;
  const int groups = p.B * p.Hkv;
  const int nKt = (p.Nkv + BN - 1) / BN;
  const int chunk = it / (kGroupChunk * nKt);
  const int rem = it - chunk * (kGroupChunk * nKt);
  const int cg = min(kGroupChunk, groups - chunk * kGroupChunk);
  w.j = rem / cg;
  const int gi = chunk * kGroupChunk + (rem - w.j * cg);
  w.b = gi / p.Hkv;
  w.hkv = gi - w.b * p.Hkv;
  w.sq = seq_of(p.m, w.b, p.status, 42);
  w.kv0 = w.j * BN;
  w.nQt = (w.sq.nq + BM - 1) / BM;
  const int qfirst = w.kv0 - w.sq.delta;
  w.i0 = p.causal ? (qfirst <= 0 ? 0 : min(qfirst / BM, w.nQt)) : 0;
  w.per_head = w.nQt - w.i0;
  w.T = w.kv0 < w.sq.nk ? G * w.per_head : 0;
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

template <bool BF16>
__device__ __forceinline__ void store_row_chunk(void* dst, const uint32_t (&pk)[16], int cols) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (8 * i < cols) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

template <int D, bool BF16, bool DET>
__global__ void __launch_bounds__(kThreads, 1)
bwd_main_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
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
  const int G = p.Hq / p.Hkv;
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::OFF_RING);

  if (threadIdx.x == 0) {
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(KVFULL + k), 1);
      mbar_init(bar(KVEMPTY + k), 1);
    }
    for (int s = 0; s < QST; ++s) {
      mbar_init(bar(QFULL + s), 1);
      mbar_init(bar(QEMPTY + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(S + i), 1);
      mbar_init(bar(P + i), 8);        // one arrival per softmax warp
      mbar_init(bar(SFREE + i), 1);
    }
    mbar_init(bar(DP), 1);
    mbar_init(bar(DPFREE), 8);
    mbar_init(bar(DS), 8);
    mbar_init(bar(DQFULL), 1);
    mbar_init(bar(DQEMPTY), 4);        // one arrival per dQ warp
    mbar_init(bar(DSFREE), 1);
    mbar_init(bar(ACC), 1);
    mbar_init(bar(ACCFREE_V), 4);      // the item's dV read out of TMEM: one arrival per epilogue warp
    mbar_init(bar(ACCFREE_K), 4);      // its dK
    mbar_init(bar(AFIN1), 1);          // warp 1's products have completed (at exit)
    mbar_init(bar(AFIN2), 1);          // warp 2's
    for (int i = 0; i < 8; ++i) {      // item ring: slot written / read by every other role's warp
      mbar_init(bar(ITEM_FULL + i), 1);
      mbar_init(bar(ITEM_EMPTY + i), 15);
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
    const int slot = k & 7;
    if (!__all_sync(0xffffffffu, mbar_wait(bar(ITEM_FULL + slot), (k >> 3) & 1, wc, 40))) return -2;
    const int it = ring[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(ITEM_EMPTY + slot));
    return it;
  };
  auto take_item1 = [&](int k) -> int {
    const int slot = k & 7;
    if (!mbar_wait(bar(ITEM_FULL + slot), (k >> 3) & 1, wc, 41)) return -2;
    const int it = ring[slot];
    mbar_arrive(bar(ITEM_EMPTY + slot));
    return it;
  };

  if (warp == 0) {
    // ================================================================ TMA producer: Q, dO, L, D
    if (lane == 0) {
      int g = 0;                 // tiles issued so far (ring stage g % QST)
      bool ok = true;
      // The fetcher: item numbers from the workspace counter, each taken only when this
      // producer starts the item (a number taken early would pin a long item to a CTA that
      // is still busy, as the hardware scheduler never does), into the ring.
      int fetched = 0;
      bool ended = false;
      auto fetch_until = [&](int k) -> bool {
        while (!ended && fetched <= k) {
          const int slot = fetched & 7;
          if (fetched >= 8 && !mbar_wait(bar(ITEM_EMPTY + slot), ((fetched >> 3) - 1) & 1, wc, 42)) return false;
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
      for (int k = 0; ok; ++k) {
        if (!fetch_until(k)) break;
        if (k >= fetched) break;                  // past the end marker
        const int it = ring[k & 7];              // written by this thread
        if (it < 0) break;
        const Item w = decode(it, p, G);
        const int bc = bcoord(p.m, w.b);
        for (int t = 0; t < w.T; ++t, ++g) {
          const int s = g % QST;
          if (g >= QST && !mbar_wait(bar(QEMPTY + s), ((g / QST) & 1) ^ 1, wc, 3)) { ok = false; break; }
          const int h = w.hkv * G + t / w.per_head;
          const int q0 = (w.i0 + t % w.per_head) * BM;
          const int bh = w.b * p.Hq + h;
          if (!FA_BOUNDS(h < p.Hq && q0 < w.sq.nq && w.sq.q_start + q0 < rows_q(p.m) &&
                             static_cast<size_t>(bh) * p.NqPad + q0 + BM <= static_cast<size_t>(p.B) * p.Hq * p.NqPad,
                         wc, 68)) {
            ok = false;
            break;
          }
          const uint32_t fb = bar(QFULL + s);
          mbar_arrive_expect_tx(fb, 2 * L::Q_BYTES + L::LD_BYTES);
#pragma unroll
          for (int hh = 0; hh < L::NH; ++hh) {
            tma_load_4d(sb + L::OFF_Q + s * L::Q_BYTES + hh * L::QHALF, &tm_q, fb, 64 * hh, w.sq.q_start + q0, h, bc);
            tma_load_4d(sb + L::OFF_DO + s * L::Q_BYTES + hh * L::QHALF, &tm_do, fb, 64 * hh, w.sq.q_start + q0, h,
                        bc);
          }
          const size_t row = static_cast<size_t>(bh) * p.NqPad + q0;
          bulk_load(sb + L::OFF_LD + s * L::LD_BYTES, p.nLg + row, BM * 4, fb);
          bulk_load(sb + L::OFF_LD + s * L::LD_BYTES + BM * 4, p.Dv + row, BM * 4, fb);
        }
      }
      // never leave a copy in flight into shared memory this CTA is about to release
      for (int u = max(0, g - QST); u < g; ++u) drain_wait(bar(QFULL + u % QST), (u / QST) & 1);
    }
  } else if (warp == 3) {
    // ================================================================ TMA producer: K, V
    // Item n's K and V go into buffer n % KVBUF once the item that used it before
    // (n - KVBUF) has had its last products read it; its Q/dO tiles are meanwhile
    // prefetched by warp 0.
    if (lane == 0) {
      constexpr int NB = L::KVBUF;
      int n = 0;                 // items with work so far
      for (int k = 0;; ++k) {
        const int it = take_item1(k);
        if (it < 0) break;
        const Item w = decode(it, p, G);
        if (w.T == 0) continue;
        const int bc = bcoord(p.m, w.b);
        const int kb = n % NB;
        if (n >= NB && !mbar_wait(bar(KVEMPTY + kb), ((n / NB) - 1) & 1, wc, 1)) break;
        if (!FA_BOUNDS(w.sq.k_start + w.kv0 < rows_k(p.m) && w.hkv < p.Hkv && bc < batch_extent(p.m), wc, 67)) break;
        const uint32_t fb = bar(KVFULL + kb);
        const uint32_t kdst = sb + L::OFF_KV + 2 * kb * L::KV_BYTES;
        mbar_arrive_expect_tx(fb, 2 * L::KV_BYTES);
#pragma unroll
        for (int hh = 0; hh < L::NH; ++hh) {
          tma_load_4d(kdst + hh * L::KHALF, &tm_k, fb, 64 * hh, w.sq.k_start + w.kv0, w.hkv, bc);
          tma_load_4d(kdst + L::KV_BYTES + hh * L::KHALF, &tm_v, fb, 64 * hh, w.sq.k_start + w.kv0, w.hkv, bc);
        }
        ++n;
      }
      for (int m = max(0, n - NB); m < n; ++m) drain_wait(bar(KVFULL + m % NB), (m / NB) & 1);
    }
  } else if (warp == 1 || warp == 2) {
    // ================================================================ MMA issuers
    constexpr uint32_t ID_S = make_idesc_f16(128, BM, BF16, false, false);
    constexpr uint32_t ID_KV = make_idesc_f16(128, D, BF16, false, true);
    constexpr uint32_t ID_Q = make_idesc_f16(128, BM, BF16, true, true);
    const uint32_t tdP = tmem + L::COL_DP;
    const uint32_t tdK = tmem + L::COL_DK, tdV = tmem + L::COL_DV, tdQ = tmem + L::COL_DQ;
    auto s_buf = [&](int g) -> uint32_t { return tmem + L::COL_S + (g & 1) * BM; };
    auto q_tile = [&](int g) -> uint32_t { return sb + L::OFF_Q + (g % QST) * L::Q_BYTES; };
    auto do_tile = [&](int g) -> uint32_t { return sb + L::OFF_DO + (g % QST) * L::Q_BYTES; };
    const uint64_t dS_mn = sw128_desc(sb + L::OFF_DS, L::DS_BYTES, 1024);
    const uint64_t dS_k = sw128_desc(sb + L::OFF_DS, 16, 1024);
    auto kstep = [](int ks, int half_bytes) -> uint64_t {
      return static_cast<uint64_t>(((ks >> 2) * half_bytes + (ks & 3) * 32) >> 4);
    };
    auto mnstep = [](int ks) -> uint64_t { return static_cast<uint64_t>((ks * 2048) >> 4); };
    auto a_col = [](int ks) -> uint32_t { return static_cast<uint32_t>(32 * (ks >> 1) + 8 * (ks & 1)); };
    auto wait = [&](uint32_t b_, uint32_t parity, uint32_t site) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b_, parity, wc, site));
    };
    int n = 0, g = 0;
    bool ok = true;
    if (warp == 1) {
      for (int k = 0; ok; ++k) {
        const int it = take_item(k);
        if (it < 0) break;
        const Item w = decode(it, p, G);
        if (w.T == 0) continue;
        const int kb = n % L::KVBUF;
        const uint32_t aK = sb + L::OFF_KV + 2 * kb * L::KV_BYTES;
        const uint64_t dK_k = sw128_desc(aK, 16, 1024), dV_k = sw128_desc(aK + L::KV_BYTES, 16, 1024);
        if (!wait(bar(KVFULL + kb), (n / L::KVBUF) & 1, 2)) break;
        ++n;
        for (int t = 0; t < w.T; ++t, ++g) {
          // G1: S^T(g) = K Q^T into buffer g & 1, once G3(g - 2) has read the P^T there
          if (!wait(bar(QFULL + g % QST), (g / QST) & 1, 3)) { ok = false; break; }
          if (g >= 2 && !wait(bar(SFREE + (g & 1)), ((g - 2) >> 1) & 1, 15)) { ok = false; break; }
          tc_fence_after();
          {
            const uint64_t dQ_k = sw128_desc(q_tile(g), 16, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              umma_ss_warp(s_buf(g), dK_k + kstep(ks, L::KHALF), dQ_k + kstep(ks, L::QHALF), ID_S, ks > 0);
            umma_commit_warp(bar(S + (g & 1)));
          }
          // G2: dP^T(g) = V dO^T, once the softmax groups have loaded dP^T(g - 1)
          if (g >= 1 && !wait(bar(DPFREE), (g - 1) & 1, 14)) { ok = false; break; }
          tc_fence_after();
          {
            const uint64_t dO_k = sw128_desc(do_tile(g), 16, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              umma_ss_warp(tdP, dV_k + kstep(ks, L::KHALF), dO_k + kstep(ks, L::QHALF), ID_S, ks > 0);
            umma_commit_warp(bar(DP));
          }
        }
      }
      // this warp's MMAs must have completed before TMEM is released
      umma_commit_warp(bar(AFIN1));
      drain_wait(bar(AFIN1), 0);
    } else {
      for (int k = 0; ok; ++k) {
        const int it = take_item(k);
        if (it < 0) break;
        const Item w = decode(it, p, G);
        if (w.T == 0) continue;
        const int kb = n % L::KVBUF;
        const uint64_t dK_mn = sw128_desc(sb + L::OFF_KV + 2 * kb * L::KV_BYTES, L::KHALF, 1024);
        for (int t = 0; t < w.T; ++t, ++g) {
          // the item's first products start new dV/dK sums: the previous item's must have been read out
          if (t == 0 && n >= 1 && !wait(bar(ACCFREE_V), (n - 1) & 1, 16)) { ok = false; break; }
          // G3: dV += P^T dO
          if (!wait(bar(P + (g & 1)), (g >> 1) & 1, 4)) { ok = false; break; }
          tc_fence_after();
          {
            const uint64_t dO_mn = sw128_desc(do_tile(g), L::QHALF, 1024);
#pragma unroll
            for (int ks = 0; ks < BM / 16; ++ks)
              umma_ts_warp(tdV, s_buf(g) + a_col(ks), dO_mn + mnstep(ks), ID_KV, (t > 0 || ks > 0));
            umma_commit_warp(bar(SFREE + (g & 1)));
          }
          // G4: dK += dS^T Q
          if (t == 0 && n >= 1 && !wait(bar(ACCFREE_K), (n - 1) & 1, 12)) { ok = false; break; }
          if (!wait(bar(DS), g & 1, 5)) { ok = false; break; }
          tc_fence_after();
          {
            const uint64_t dQ_mn = sw128_desc(q_tile(g), L::QHALF, 1024);
#pragma unroll
            for (int ks = 0; ks < BM / 16; ++ks)
              umma_ss_warp(tdK, dS_k + static_cast<uint64_t>((ks * 32) >> 4), dQ_mn + mnstep(ks), ID_KV,
                           (t > 0 || ks > 0));
          }
          if constexpr (!DET) {
            // G5: dQ^T = K^T dS^T
            if (g > 0 && !wait(bar(DQEMPTY), (g - 1) & 1, 6)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks)
              umma_ss_warp(tdQ, dK_mn + mnstep(ks), dS_mn + mnstep(ks), ID_Q, ks > 0);
            umma_commit_warp(bar(DQFULL));
          }
          umma_commit_warp(bar(DSFREE));
          umma_commit_warp(bar(QEMPTY + g % QST));
        }
        if (!ok) break;
        // every product of the item has been issued: K and V may be replaced once they
        // complete, and dK/dV are final
        umma_commit_warp(bar(KVEMPTY + kb));
        umma_commit_warp(bar(ACC));
        ++n;
      }
      umma_commit_warp(bar(AFIN2));
      drain_wait(bar(AFIN2), 0);
    }
  } else if (warp >= 4 && warp < 12) {
    // ================================================================ softmax / dS groups
    const int grp = (warp - 4) >> 2;                      // query columns [32 grp, 32 grp + 32)
    const int r = threadIdx.x - 128 - 128 * grp;          // KV row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tdP = tmem + lane_off + L::COL_DP + 32 * grp;
    uint8_t* ds_row = smem + L::OFF_DS + r * 128;
    const uint64_t sc2 = f2_bits(p.scale_log2, p.scale_log2);
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int it = take_item(k);
      if (it < 0) break;
      const Item w = decode(it, p, G);
      const int kv = w.kv0 + r;
      const bool row_ok = kv < w.sq.nk;
      if (w.T == 0) continue;
      int qi = w.i0, h = w.hkv * G;
      for (int t = 0; t < w.T; ++t, ++g, h += (qi + 1 == w.nQt), qi = (qi + 1 == w.nQt) ? w.i0 : qi + 1) {
        const int s = g % QST;
        const int q0 = qi * BM;
        const float* Ls = reinterpret_cast<const float*>(smem + L::OFF_LD + s * L::LD_BYTES) + 32 * grp;
        const float* Ds = Ls + BM;
        const uint32_t tS = tmem + lane_off + L::COL_S + (g & 1) * BM + 32 * grp;
        const int lim = p.causal ? (kv - w.sq.delta - q0 - 32 * grp) : INT_MIN;
        const bool need_mask = __any_sync(0xffffffffu, !row_ok || lim > 0);
        if (!__all_sync(0xffffffffu, mbar_wait(bar(S + (g & 1)), (g >> 1) & 1, wc, 7))) { ok = false; break; }
        tc_fence_after();
        uint32_t pk[16];
        {
          uint32_t sr[32];
          tmem_ld_x32(tS, sr);
          tmem_ld_wait();
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            // x = S * scale * log2(e) + (-L * log2(e)), two columns per instruction
            const ulonglong2 nl = *reinterpret_cast<const ulonglong2*>(Ls + 4 * c4);
            const int c = 4 * c4;
            const float2 xa = f2_split(fma_f32x2(f2_bits(__uint_as_float(sr[4 * c4 + 0]), __uint_as_float(sr[4 * c4 + 1])), sc2, nl.x));
            const float2 xb = f2_split(fma_f32x2(f2_bits(__uint_as_float(sr[4 * c4 + 2]), __uint_as_float(sr[4 * c4 + 3])), sc2, nl.y));
            float e0 = ex2_approx(xa.x);
            float e1 = ex2_approx(xa.y);
            float e2 = ex2_approx(xb.x);
            float e3 = ex2_approx(xb.y);
            if (need_mask) {
              if (!row_ok || c + 0 < lim) e0 = 0.f;
              if (!row_ok || c + 1 < lim) e1 = 0.f;
              if (!row_ok || c + 2 < lim) e2 = 0.f;
              if (!row_ok || c + 3 < lim) e3 = 0.f;
            }
            pk[2 * c4] = pack2<BF16>(e0, e1);
            pk[2 * c4 + 1] = pack2<BF16>(e2, e3);
          }
        }
        tmem_st_x16(tS, pk);                  // P^T, 16-bit, over the columns just read
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P + (g & 1)));
        if (!__all_sync(0xffffffffu, mbar_wait(bar(DP), g & 1, wc, 8))) { ok = false; break; }
        tc_fence_after();
        uint32_t dk[16];
        {
          uint32_t dr[32];
          tmem_ld_x32(tdP, dr);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(DPFREE));   // dP^T buffer may now take the next tile's G2
#pragma unroll
          for (int c4 = 0; c4 < 8; ++c4) {
            // dS = P * (dP - D), two columns per instruction
            const ulonglong2 d2 = *reinterpret_cast<const ulonglong2*>(Ds + 4 * c4);
            const float2 pa = unpack2<BF16>(pk[2 * c4]);
            const float2 pb = unpack2<BF16>(pk[2 * c4 + 1]);
            const float2 sa = f2_split(mul_f32x2(f2_bits(pa.x, pa.y),
                sub_f32x2(f2_bits(__uint_as_float(dr[4 * c4 + 0]), __uint_as_float(dr[4 * c4 + 1])), d2.x)));
            const float2 sbv = f2_split(mul_f32x2(f2_bits(pb.x, pb.y),
                sub_f32x2(f2_bits(__uint_as_float(dr[4 * c4 + 2]), __uint_as_float(dr[4 * c4 + 3])), d2.y)));
            dk[2 * c4] = pack2<BF16>(sa.x, sa.y);
            dk[2 * c4 + 1] = pack2<BF16>(sbv.x, sbv.y);
          }
        }
        {
          // dS^T row r into shared memory (128-byte swizzle), once G4/G5(g - 1) have read it
          if (g > 0 && !__all_sync(0xffffffffu, mbar_wait(bar(DSFREE), (g - 1) & 1, wc, 9))) { ok = false; break; }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = 4 * grp + i;
            *reinterpret_cast<uint4*>(ds_row + ((c ^ (r & 7)) << 4)) =
                make_uint4(dk[4 * i], dk[4 * i + 1], dk[4 * i + 2], dk[4 * i + 3]);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(DS));
      }
      if (!ok) break;
    }
  } else if (warp >= 12) {
    // ================================================================ dQ group, epilogue
    // Per tile (atomic mode): dQ^T from TMEM into the fp32 accumulator.  Per item: dK
    // (x scale) and dV of KV row r out of TMEM, release of the accumulators, then the
    // stores, while the softmax warps already work on the next item's first tiles.
    const int r = threadIdx.x - 384;                     // TMEM lane: dQ column, KV row of dK/dV
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tdQ = tmem + lane_off + L::COL_DQ;
    int n = 0, g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int it = take_item(k);
      if (it < 0) break;
      const Item w = decode(it, p, G);
      const int kv = w.kv0 + r;
      const bool row_ok = kv < w.sq.nk && FA_BOUNDS(w.sq.k_start + kv < rows_k(p.m), wc, 65);
      uint8_t* out_k = reinterpret_cast<uint8_t*>(p.dk) + at(p.m.st.dk, p.m, w.b, w.hkv, w.sq.k_start + kv) * 2;
      uint8_t* out_v = reinterpret_cast<uint8_t*>(p.dv) + at(p.m.st.dv, p.m, w.b, w.hkv, w.sq.k_start + kv) * 2;
      if (w.T == 0) {
        // keys no query sees: dK = dV = 0
        uint32_t zero[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) zero[c] = 0u;
        if (row_ok)
          for (int ch = 0; ch < D / 32; ++ch) {
            store_row_chunk<BF16>(out_k + ch * 64, zero, p.m.d - 32 * ch);
            store_row_chunk<BF16>(out_v + ch * 64, zero, p.m.d - 32 * ch);
          }
        continue;
      }
      if constexpr (!DET) {
        int h = w.hkv * G, qi = w.i0;
        for (int t = 0; t < w.T; ++t, ++g) {
          const int q0 = qi * BM;
          if (!__all_sync(0xffffffffu, mbar_wait(bar(DQFULL), g & 1, wc, 10))) { ok = false; break; }
          tc_fence_after();
          uint32_t v0[32], v1[32];
          tmem_ld_x32(tdQ, v0);
          tmem_ld_x32(tdQ + 32, v1);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(DQEMPTY));
          if (r < D && FA_BOUNDS(static_cast<size_t>(w.b * p.Hq + h) * p.NqPad + q0 + BM <=
                                     static_cast<size_t>(p.B) * p.Hq * p.NqPad,
                                 wc, 64)) {
            float* dst = p.dq_acc + (static_cast<size_t>(w.b * p.Hq + h) * p.NqPad + q0) * D + r;
#pragma unroll
            for (int c = 0; c < 32; ++c) red_add_f32(dst + c * D, __uint_as_float(v0[c]));
#pragma unroll
            for (int c = 0; c < 32; ++c) red_add_f32(dst + (32 + c) * D, __uint_as_float(v1[c]));
          }
          if (++qi == w.nQt) {
            qi = w.i0;
            ++h;
          }
        }
        if (!ok) break;
      }
      // ---- epilogue of the item: dV, then dK (x scale), of KV row r: each read out of TMEM
      // into 16-bit, released for the next item's first product into it, then stored
      if (!__all_sync(0xffffffffu, mbar_wait(bar(ACC), n & 1, wc, 13))) break;
      tc_fence_after();
      const bool store = row_ok && *abort_flag == 0;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const uint32_t tacc = tmem + lane_off + (which == 0 ? L::COL_DV : L::COL_DK);
        const float mul = which == 0 ? 1.0f : p.scale;
        uint32_t pk[D / 2];
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t a[32];
          tmem_ld_x32(tacc + ch * 32, a);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c)
            pk[16 * ch + c] = pack2<BF16>(__uint_as_float(a[2 * c]) * mul, __uint_as_float(a[2 * c + 1]) * mul);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(which == 0 ? ACCFREE_V : ACCFREE_K));
        if (store) {
          uint8_t* out = which == 0 ? out_v : out_k;
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch)
            store_row_chunk<BF16>(out + ch * 64, *reinterpret_cast<const uint32_t(*)[16]>(pk + 16 * ch),
                                  p.m.d - 32 * ch);
        }
      }
      ++n;
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

template <int D, bool BF16, bool DET>
cudaError_t launch_t(const MainArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo, const CUtensorMap& tk,
                     const CUtensorMap& tv, cudaStream_t stream) {
  using L = PLayout<D>;
  auto kern = bwd_main_persist_kernel<D, BF16, DET>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  Params p;
  p.nLg = a.ws.nLg;
  p.Dv = a.ws.Dv;
  p.dq_acc = a.ws.dq_acc;
  p.dk = a.dk;
  p.dv = a.dv;
  p.status = a.status;
  p.call_abort = a.ws.abort;
  p.B = a.pb.B; p.Hq = a.pb.Hq; p.Hkv = a.pb.Hkv; p.Nq = a.pb.Nq; p.Nkv = a.pb.Nkv; p.NqPad = a.pb.NqPad;
  p.scale = a.pb.scale;
  p.scale_log2 = a.pb.scale * 1.4426950408889634f;
  p.causal = a.pb.causal;
  p.m = seq_map(a.pb);
  const long long items = static_cast<long long>((a.pb.Nkv + BN - 1) / BN) * a.pb.B * a.pb.Hkv;
  p.items = static_cast<int>(items);
  p.next_item = a.ws.abort + 1;
  p.done_ctas = a.ws.abort + 2;
  const long long grid = items < sm_count() ? items : sm_count();
  kern<<<static_cast<unsigned>(grid), kThreads, L::ALLOC, stream>>>(tq, tdo, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_main_persist(const MainArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                                    const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  const bool det = a.pb.deterministic != 0;
  if (a.pb.d > 64) {
    if (a.pb.bf16) return det ? launch_t<128, true, true>(a, tq, tdo, tk, tv, stream)
                              : launch_t<128, true, false>(a, tq, tdo, tk, tv, stream);
    return det ? launch_t<128, false, true>(a, tq, tdo, tk, tv, stream)
               : launch_t<128, false, false>(a, tq, tdo, tk, tv, stream);
  }
  if (a.pb.bf16) return det ? launch_t<64, true, true>(a, tq, tdo, tk, tv, stream)
                            : launch_t<64, true, false>(a, tq, tdo, tk, tv, stream);
  return det ? launch_t<64, false, true>(a, tq, tdo, tk, tv, stream)
             : launch_t<64, false, false>(a, tq, tdo, tk, tv, stream);
}

}  // namespace fa
