// fwd_persist.cu -- the forward (O and the natural-log LSE L of the scaled,
// masked scores, the convention of flash_attention_backward.cu, rustytorch
// rtx-flash-attention, block "Compute softmax probabilities from scores and
// LSE") as a persistent kernel: the one used for every problem without an
// additive bias.
//
// The arithmetic, tiles, TMEM plan and warp roles are those of fwd.cu without a
// bias: a work item is a pair of 128-row query tiles of one query head, which
// walk the 64-key K/V tiles they see with two S buffers and O per query tile in
// TMEM and an online softmax with a lazily moved reference max:
//   G1  S [BQ x BK] = Q . K^T     A = Q (smem, K-major), B = K (K-major)
//   PV  O [BQ x d ] += P . V      A = P (TMEM, 16-bit),  B = V (MN-major)
// What differs is the schedule: one CTA per SM takes the work items of fwd.cu's
// launch order (the longest pairs first) in rounds of one item per CTA, every
// other round in reverse CTA order (a forward call has no workspace for a
// counter; a round holds pairs of about one length, and reversing the order
// every other round keeps any CTA from taking the longer item of every round),
// and the items flow through it back to back:
//   - the K/V ring runs across items on a tile counter of the CTA (warp 3 loads
//     it), so the next item's first K/V tiles load while the current item is
//     computed; the S buffers and every hand-off follow per-query-tile counters;
//   - the next item's query tiles load as soon as the current item's last S
//     products have read them;
//   - the softmax warpgroups read O of an item out of TMEM and release it before
//     they store it, so the next item's first P V waits only for that read-out.
#include <cstdint>
#include <climits>
#include <math_constants.h>

#include "kernels.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace fa {
namespace {

constexpr int BQ = 128;       // query rows per tile (TMEM lanes)
constexpr int NT = 2;         // query tiles per work item (one softmax warpgroup each; the softmax
                              // warpgroups select their tile's count between the two)
constexpr int BK = kFwdBK;    // keys per step
constexpr int STAGES = 4;     // K/V ring depth
constexpr int SB = 2;         // S buffers per query tile
constexpr int kThreads = 128 + NT * 128;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P stays <= 256

template <int D>
struct PLayout {
  static constexpr int NH = D / 64;
  static constexpr int HALF = 128 * 128;        // one 64-column half of a 128-row query tile
  static constexpr int TILE = NH * HALF;
  static constexpr int KHALF = BK * 128;        // one 64-column half of a K or V tile
  static constexpr int KV_TILE = NH * KHALF;
  static constexpr int OFF_Q = 0;               // query tile x at OFF_Q + x*TILE
  static constexpr int OFF_KV = NT * TILE;      // stage s: K at OFF_KV + 2*s*KV_TILE, V after it
  static constexpr int OFF_BAR = OFF_KV + STAGES * 2 * KV_TILE;
  static constexpr int NBAR = 40;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int TOTAL = OFF_MISC + 16;
  static constexpr int ALLOC = TOTAL + 1024;    // slack for 1024-byte alignment
  // TMEM of query tile x: its S buffers, then O
  static constexpr int TCOLS = SB * BK + 128;
  __host__ __device__ static constexpr int col_s(int x, int s) { return x * TCOLS + s * BK; }
  __host__ __device__ static constexpr int col_o(int x) { return x * TCOLS + SB * BK; }
  static_assert(NT * TCOLS <= 512 && D <= 128, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// Barriers.  Per query tile x and S buffer s (index 2x + s): S ready, P written, P read by
// P V.  Per query tile: P V complete, O read out of TMEM.
enum : int {
  QFULL = 0, QEMPTY, KVFULL, KVEMPTY = KVFULL + STAGES, S = KVEMPTY + STAGES, P = S + 4, SFREE = P + 4,
  PV = SFREE + 4, OFREE = PV + 2, AFIN1 = OFREE + 2, AFIN2, BAR_END
};
static_assert(BAR_END <= PLayout<128>::NBAR, "barrier count");

struct Params {
  void* o;
  float* lse;
  unsigned int* status;       // device-wide report word
  unsigned int* call_abort;   // this call's abort word (a slot of a ring)
  unsigned int call_tag;      // what this call stores there when it gives up
  SeqMap m;
  int B, Hq, Hkv, Nq, Nkv;    // Nq, Nkv: the longest lengths of a packed batch
  float scale_log2;
  int causal;
  int items;                  // (pair of query tiles, head, batch) work items
};

// One work item: query tiles 2i and 2i + 1 of head h of sequence b; each tile x walks
// the Tx[x] KV tiles it sees, and the item T = the larger of the two.
struct Item {
  int b, h, hk, q0, T;
  int Tx[NT];
  Seq sq;
};

__device__ __forceinline__ Item decode(int it, const Params& p) {
  Item w;
  const int BH = p.B * p.Hq;
  const int nPairs = ((p.Nq + BQ - 1) / BQ + NT - 1) / NT;
  const int i = nPairs - 1 - it / BH;
  const int bh = it - (it / BH) * BH;
  w.b = bh / p.Hq;
  w.h = bh - w.b * p.Hq;
  w.sq = seq_of(p.m, w.b, p.status, 53);
  w.hk = w.h / (p.Hq / p.Hkv);
  w.q0 = i * NT * BQ;
  const int nKt = (w.sq.nk + BK - 1) / BK;
  w.T = 0;
#pragma unroll
  for (int x = 0; x < NT; ++x) {
    // causal: up to the last key the tile's last row sees
    const int qx = w.q0 + x * BQ;
    const int kmax = min(qx + BQ, w.sq.nq) - 1 + w.sq.delta;
    w.Tx[x] = qx >= w.sq.nq ? 0 : p.causal ? (kmax < 0 ? 0 : min(nKt, kmax / BK + 1)) : nKt;
    w.T = max(w.T, w.Tx[x]);
  }
  return w;
}

__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
fwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using L = PLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sb + L::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  if (threadIdx.x == 0) {
    mbar_init(bar(QFULL), 1);
    mbar_init(bar(QEMPTY), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(KVFULL + s), 1);
      mbar_init(bar(KVEMPTY + s), 1);
    }
    for (int x = 0; x < NT; ++x) {
      for (int s = 0; s < SB; ++s) {
        mbar_init(bar(S + 2 * x + s), 1);
        mbar_init(bar(P + 2 * x + s), 4);       // one arrival per softmax warp
        mbar_init(bar(SFREE + 2 * x + s), 1);
      }
      mbar_init(bar(PV + x), 1);
      mbar_init(bar(OFREE + x), 4);             // one arrival per softmax warp
    }
    mbar_init(bar(AFIN1), 1);
    mbar_init(bar(AFIN2), 1);
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
  const WaitCtx wc{p.status, p.call_abort, abort_flag, p.call_tag};
  // The k-th item of this CTA: the items in launch order (the longest first), dealt in rounds
  // of one per CTA, every other round in reverse CTA order so that no CTA takes the longer item
  // of every round.
  const int step = static_cast<int>(gridDim.x);
  auto item_of = [&](int k) -> int {
    return k * step + ((k & 1) ? step - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
  };

  if (warp == 0) {
    // ================================================================ TMA producer: query tiles
    if (lane == 0) {
      int n = 0;                 // items with work loaded so far
      for (int k = 0, it = item_of(0); it < p.items; it = item_of(++k)) {
        const Item w = decode(it, p);
        if (w.T == 0) continue;
        const int bc = bcoord(p.m, w.b);
        // the previous item's S products have read its query tiles
        if (n >= 1 && !mbar_wait(bar(QEMPTY), (n - 1) & 1, wc, 84)) break;
        if (!FA_BOUNDS(w.h < p.Hq && bc < batch_extent(p.m) && w.sq.q_start + w.q0 < rows_q(p.m), wc, 85)) break;
        mbar_arrive_expect_tx(bar(QFULL), NT * L::TILE);
#pragma unroll
        for (int x = 0; x < NT; ++x)
#pragma unroll
          for (int hh = 0; hh < L::NH; ++hh)
            tma_load_4d(sb + L::OFF_Q + x * L::TILE + hh * L::HALF, &tm_q, bar(QFULL), 64 * hh,
                        w.sq.q_start + w.q0 + x * BQ, w.h, bc);
        ++n;
      }
      if (n > 0) drain_wait(bar(QFULL), (n - 1) & 1);
    }
  } else if (warp == 3) {
    // ================================================================ TMA producer: K, V
    if (lane == 0) {
      int g = 0;                 // K/V tiles issued so far, over all items
      bool ok = true;
      for (int k = 0, it = item_of(0); ok && it < p.items; it = item_of(++k)) {
        const Item w = decode(it, p);
        const int bc = bcoord(p.m, w.b);
        for (int t = 0; t < w.T; ++t, ++g) {
          const int s = g % STAGES;
          if (!FA_BOUNDS(w.sq.k_start + t * BK < rows_k(p.m) && w.hk < p.Hkv && bc < batch_extent(p.m), wc, 86)) {
            ok = false;
            break;
          }
          if (g >= STAGES && !mbar_wait(bar(KVEMPTY + s), ((g / STAGES) & 1) ^ 1, wc, 87)) { ok = false; break; }
          const uint32_t fb = bar(KVFULL + s);
          mbar_arrive_expect_tx(fb, 2 * L::KV_TILE);
          const uint32_t dst = sb + L::OFF_KV + s * 2 * L::KV_TILE;
#pragma unroll
          for (int hh = 0; hh < L::NH; ++hh) {
            tma_load_4d(dst + hh * L::KHALF, &tm_k, fb, 64 * hh, w.sq.k_start + t * BK, w.hk, bc);
            tma_load_4d(dst + L::KV_TILE + hh * L::KHALF, &tm_v, fb, 64 * hh, w.sq.k_start + t * BK, w.hk, bc);
          }
        }
      }
      for (int u = max(0, g - STAGES); u < g; ++u) drain_wait(bar(KVFULL + u % STAGES), (u / STAGES) & 1);
    }
  } else if (warp == 1 || warp == 2) {
    // ================================================================ MMA issuers
    constexpr uint32_t ID_S = make_idesc_f16(128, BK, BF16, false, false);
    constexpr uint32_t ID_O = make_idesc_f16(128, D, BF16, false, true);
    auto s_buf = [&](int x, int gx) -> uint32_t { return tmem + L::col_s(x, gx % SB); };
    auto o_buf = [&](int x) -> uint32_t { return tmem + L::col_o(x); };
    auto k_tile = [&](int g) -> uint32_t { return sb + L::OFF_KV + (g % STAGES) * 2 * L::KV_TILE; };
    // descriptor advance of k-step ks (16 columns of d) in a K-major tile of 64-column
    // halves of `half` bytes
    auto kstep = [](int ks, int half) -> uint64_t {
      return static_cast<uint64_t>(((ks >> 2) * half + (ks & 3) * 32) >> 4);
    };
    auto wait = [&](uint32_t bb, uint32_t parity, uint32_t site) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bb, parity, wc, site));
    };
    int n = 0, g = 0;            // items with work, K/V tiles
    int gx[NT] = {};             // S tiles of each query tile so far
    bool ok = true;
    if (warp == 1) {
      // G1: S_x = Q_x K^T into S buffer gx mod SB of tile x, once P V of its tile
      // gx - SB has read the P that sits in that buffer
      for (int k = 0, it = item_of(0); ok && it < p.items; it = item_of(++k)) {
        const Item w = decode(it, p);
        if (w.T == 0) continue;
        if (!wait(bar(QFULL), n & 1, 88)) break;
        for (int t = 0; t < w.T; ++t, ++g) {
          if (!wait(bar(KVFULL + g % STAGES), (g / STAGES) & 1, 89)) { ok = false; break; }
          const uint64_t dK_k = sw128_desc(k_tile(g), 16, 1024);
#pragma unroll
          for (int x = 0; x < NT; ++x) {
            if (t >= w.Tx[x]) continue;
            const int sbi = gx[x] % SB;
            if (gx[x] >= SB && !wait(bar(SFREE + 2 * x + sbi), ((gx[x] - SB) / SB) & 1, 90)) { ok = false; break; }
            tc_fence_after();
            const uint64_t dQ_k = sw128_desc(sb + L::OFF_Q + x * L::TILE, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              umma_ss_warp(s_buf(x, gx[x]), dQ_k + kstep(ks, L::HALF), dK_k + kstep(ks, L::KHALF), ID_S, ks > 0);
            umma_commit_warp(bar(S + 2 * x + sbi));
            ++gx[x];
          }
          if (!ok) break;
        }
        if (!ok) break;
        umma_commit_warp(bar(QEMPTY));   // the item's S products have read its query tiles
        ++n;
      }
      umma_commit_warp(bar(AFIN1));
      drain_wait(bar(AFIN1), 0);
    } else {
      // PV: O_x += P_x V (P, 16-bit, packed into the first half of its S buffer; V read
      // MN-major); the item's first P V of a tile waits for the previous item's O read-out
      int nx[NT] = {};           // items with work of each query tile so far
      for (int k = 0, it = item_of(0); ok && it < p.items; it = item_of(++k)) {
        const Item w = decode(it, p);
        if (w.T == 0) continue;
        for (int t = 0; t < w.T; ++t, ++g) {
          const uint64_t dV_mn = sw128_desc(k_tile(g) + L::KV_TILE, L::KHALF, 1024);
#pragma unroll
          for (int x = 0; x < NT; ++x) {
            if (t >= w.Tx[x]) continue;
            if (t == 0 && nx[x] >= 1 && !wait(bar(OFREE + x), (nx[x] - 1) & 1, 91)) { ok = false; break; }
            const int sbi = gx[x] % SB;
            if (!wait(bar(P + 2 * x + sbi), (gx[x] / SB) & 1, 92)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)
              umma_ts_warp(o_buf(x), s_buf(x, gx[x]) + 8 * ks, dV_mn + static_cast<uint64_t>((ks * 2048) >> 4),
                           ID_O, (t > 0 || ks > 0));
            umma_commit_warp(bar(SFREE + 2 * x + sbi));
            umma_commit_warp(bar(PV + x));
            ++gx[x];
          }
          if (!ok) break;
          umma_commit_warp(bar(KVEMPTY + g % STAGES));   // every G1 of this K/V tile completed before its P existed
        }
        if (!ok) break;
#pragma unroll
        for (int x = 0; x < NT; ++x) nx[x] += w.Tx[x] > 0;
        ++n;
      }
      umma_commit_warp(bar(AFIN2));
      drain_wait(bar(AFIN2), 0);
    }
  } else if (warp >= 4) {
    // ================================================================ softmax groups, epilogue
    const int qt = (warp - 4) >> 2;                     // query tile of this warpgroup
    const int r = threadIdx.x - 128 - 128 * qt;         // query row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + lane_off + L::col_o(qt);
    const uint64_t sc2 = f2_bits(p.scale_log2, p.scale_log2);
    int g = 0;                   // S tiles of this query tile so far (P V of this tile committed so far)
    bool ok = true;
    for (int k = 0, it = item_of(0); ok && it < p.items; it = item_of(++k)) {
      const Item w = decode(it, p);
      const Seq& sq = w.sq;
      const int q = w.q0 + qt * BQ + r;
      const int T = qt == 0 ? w.Tx[0] : w.Tx[1];   // no dynamic index: w stays in registers
      float m_ref = -CUDART_INF_F;                      // reference max (log2 units); -inf: no key seen yet
      float l = 0.f;                                    // sum of 2^(x - m_ref)
      for (int t = 0; t < T; ++t, ++g) {
        const int kv0 = t * BK;
        // columns c >= lim are masked: past the end of K/V, or (causal) after query q
        int lim = sq.nk - kv0;
        if (p.causal) lim = min(lim, q + sq.delta - kv0 + 1);
        const bool need_mask = __any_sync(0xffffffffu, lim < BK);
        const int sbi = g % SB;
        const uint32_t tS = tmem + lane_off + L::col_s(qt, sbi);
        if (!__all_sync(0xffffffffu, mbar_wait(bar(S + 2 * qt + sbi), (g / SB) & 1, wc, 93))) { ok = false; break; }
        tc_fence_after();
        float x[BK];
        {
          uint32_t sr[BK];
#pragma unroll
          for (int ch = 0; ch < BK / 32; ++ch) tmem_ld_x32(tS + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(sr + 32 * ch));
          tmem_ld_wait();
#pragma unroll
          for (int c2 = 0; c2 < BK / 2; ++c2) {   // two columns per instruction
            const float2 xx = f2_split(mul_f32x2(f2_bits(__uint_as_float(sr[2 * c2]), __uint_as_float(sr[2 * c2 + 1])), sc2));
            x[2 * c2] = xx.x;
            x[2 * c2 + 1] = xx.y;
          }
        }
        // row max over eight independent partial maxima
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < BK; ++c) {
          if (need_mask && c >= lim) x[c] = -CUDART_INF_F;
          mp[c & 7] = fmaxf(mp[c & 7], x[c]);
        }
        const float mt = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                               fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
        {
          // The first visible key sets the reference max (O and the sum are still 0).
          // After that it moves only when P would exceed 2^8; then O and the sum are
          // rescaled, which needs the previous P V (this item's, g - 1) to have completed.
          // P V of g - 2 has: S(g) waited for it.
          const bool first = m_ref == -CUDART_INF_F;
          const bool resc = !first && mt > m_ref + kRescaleThreshold;
          if (first) m_ref = mt;
          if (__any_sync(0xffffffffu, resc)) {
            if (!__all_sync(0xffffffffu, mbar_wait(bar(PV + qt), (g - 1) & 1, wc, 94))) { ok = false; break; }
            tc_fence_after();
            const float alpha = resc ? ex2_approx(m_ref - mt) : 1.f;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ++ch) {
              uint32_t ov[32];
              tmem_ld_x32(tO + 32 * ch, ov);
              tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
              tmem_st_x32(tO + 32 * ch, ov);
            }
            tmem_st_wait();
            if (resc) {
              l *= alpha;
              m_ref = mt;
            }
          }
        }
        const float m_use = m_ref == -CUDART_INF_F ? 0.f : m_ref;   // no key yet: every x is -inf
        const uint64_t m2 = f2_bits(m_use, m_use);
        float ls[8];                                   // partial row sums
#pragma unroll
        for (int i = 0; i < 8; ++i) ls[i] = 0.f;
#pragma unroll
        for (int ch = 0; ch < BK / 32; ++ch) {
          uint32_t pk[16];
#pragma unroll
          for (int c2 = 0; c2 < 16; ++c2) {
            const float2 xm = f2_split(sub_f32x2(f2_bits(x[32 * ch + 2 * c2], x[32 * ch + 2 * c2 + 1]), m2));
            const float p0 = ex2_approx(xm.x);
            const float p1 = ex2_approx(xm.y);
            ls[c2 & 7] += p0 + p1;
            pk[c2] = pack2<BF16>(p0, p1);
          }
          tmem_st_x16(tS + 16 * ch, pk);               // columns [16ch, 16ch+16) of S were already read
        }
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        tmem_st_wait();
        // Before the item's last P goes out, its previous P V must have completed: with two S
        // buffers the epilogue would otherwise have two P V to wait for, and once both have
        // completed, a parity wait for the older one would wait for a phase two ahead.  Here
        // at most that one P V is outstanding.
        if (t == T - 1 && T > 1 && !__all_sync(0xffffffffu, mbar_wait(bar(PV + qt), (g - 1) & 1, wc, 96))) {
          ok = false;
          break;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P + 2 * qt + sbi));
      }
      if (!ok) break;
      // ---- epilogue of the item: O = acc / l (16-bit), L = (m_ref + log2 l) * ln 2, once the
      // item's last P V (the only one still outstanding) has completed
      const bool row_ok = q < sq.nq && FA_BOUNDS(sq.q_start + q < rows_q(p.m), wc, 95);
      uint8_t* out = reinterpret_cast<uint8_t*>(p.o) + at(p.m.st.o, p.m, w.b, w.h, sq.q_start + q) * 2;
      if (T == 0) {
        // no key visible (or no row): O = 0, L = -inf
        if (row_ok) {
          for (int ch = 0; ch < D / 32; ++ch) {
            uint4* d4 = reinterpret_cast<uint4*>(out + ch * 64);
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4)
              if (32 * ch + 8 * k4 < p.m.d) d4[k4] = make_uint4(0u, 0u, 0u, 0u);
          }
          p.lse[at(p.m.st.lse, p.m, w.b, w.h, sq.q_start + q)] = -CUDART_INF_F;
        }
        continue;
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(PV + qt), (g - 1) & 1, wc, 97))) break;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;       // a row that saw no key: O = 0
      uint32_t pk[D / 2];
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        tmem_ld_x32(tO + 32 * ch, v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[16 * ch + c] = pack2<BF16>(__uint_as_float(v[2 * c]) * inv, __uint_as_float(v[2 * c + 1]) * inv);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(OFREE + qt));    // the next item's first P V may overwrite O
      if (row_ok && *abort_flag == 0) {
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint4* d4 = reinterpret_cast<uint4*>(out + ch * 64);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            if (32 * ch + 8 * k4 < p.m.d)
              d4[k4] = make_uint4(pk[16 * ch + 4 * k4], pk[16 * ch + 4 * k4 + 1], pk[16 * ch + 4 * k4 + 2],
                                  pk[16 * ch + 4 * k4 + 3]);
        }
        p.lse[at(p.m.st.lse, p.m, w.b, w.h, sq.q_start + q)] =
            l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16>
cudaError_t launch_t(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     unsigned int* status, unsigned int* call_abort, unsigned int call_tag, cudaStream_t stream) {
  using L = PLayout<D>;
  auto kern = fwd_persist_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  Params p;
  p.o = a.o;
  p.lse = a.lse;
  p.status = status;
  p.call_abort = call_abort;
  p.call_tag = call_tag;
  p.B = a.pb.B; p.Hq = a.pb.Hq; p.Hkv = a.pb.Hkv; p.Nq = a.pb.Nq; p.Nkv = a.pb.Nkv;
  p.scale_log2 = a.pb.scale * 1.4426950408889634f;
  p.causal = a.pb.causal;
  p.m = seq_map(a.pb);
  const long long items = static_cast<long long>(((a.pb.Nq + BQ - 1) / BQ + NT - 1) / NT) * a.pb.B * a.pb.Hq;
  p.items = static_cast<int>(items);
  const long long grid = items < sm_count() ? items : sm_count();
  kern<<<static_cast<unsigned>(grid), kThreads, L::ALLOC, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_persist(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               unsigned int* status, unsigned int* call_abort, unsigned int call_tag,
                               cudaStream_t stream) {
  if (a.pb.d > 64)
    return a.pb.bf16 ? launch_t<128, true>(a, tq, tk, tv, status, call_abort, call_tag, stream)
                     : launch_t<128, false>(a, tq, tk, tv, status, call_abort, call_tag, stream);
  return a.pb.bf16 ? launch_t<64, true>(a, tq, tk, tv, status, call_abort, call_tag, stream)
                   : launch_t<64, false>(a, tq, tk, tv, status, call_abort, call_tag, stream);
}

}  // namespace fa
