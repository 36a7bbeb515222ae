// fwd.cu -- exact attention forward on tcgen05 tensor cores, one CTA per work item
// (launched for problems with a bias; without one, fwd_persist.cu runs this kernel's
// no-bias configuration persistently), producing O and
// the log-sum-exp L that the backward consumes (L is the natural-log LSE of the
// scaled, masked scores: the convention of flash_attention_backward.cu,
// rustytorch rtx-flash-attention, block "Compute softmax probabilities from
// scores and LSE").
//
// One CTA owns a 128-row query tile of one query head and walks the KV tiles
// it can see (causal: up to the diagonal), keeping O in TMEM:
//   G1  S [BQ x BK] = Q . K^T     A = Q (smem, K-major), B = K (K-major)
//   PV  O [BQ x d ] += P . V      A = P (TMEM, 16-bit),  B = V (MN-major)
// Softmax runs in the log2 domain (x = S * scale * log2 e) with a running
// reference max m per row.  P = 2^(x - m) is accumulated unnormalised and O is
// divided by the row sum once at the end, so any reference max that is the
// same for O and the sum gives the exact result; m is therefore only moved
// (and O, sum rescaled by 2^(m_old - m_new)) when the row max exceeds it by
// more than 8, which keeps P <= 256 and makes rescaling rare after the first
// tiles.
//
// Warp roles (384 threads): warp 0 TMA producer (both query tiles once, a 4-stage ring
// of 64-key K/V tiles they share), warp 1 owns TMEM and issues G1, warp 2 issues PV,
// and one softmax warpgroup per query tile: thread r owns query row r (TMEM lane r)
// and all 64 columns of each S tile.  TMEM per query tile: two S buffers of 64
// columns and O (128 columns), so S of the next KV tile is computed while the
// softmax of the current one runs, and only S two tiles ahead waits for the P V
// that reads the P packed into its buffer.
// With an additive bias the CTA takes one query tile (256 threads) and steps over
// 128 keys with one S buffer, and the freed shared memory holds a 2-stage ring of
// [128 query x 128 key] bias tiles that the producer loads by TMA next to K and V
// (128-byte swizzle, so that each thread reads its own row in 16-byte pieces without
// bank conflicts).
#include <cstdint>
#include <climits>
#include <math_constants.h>

#include "kernels.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace fa {
namespace {

constexpr int BQ = 128;     // query rows per tile (TMEM lanes)
constexpr int BSTAGES = 2;  // bias ring depth
constexpr float kRescaleThreshold = 8.0f;   // log2 units: P stays <= 256

// Query tiles per CTA (one softmax warpgroup each), threads, keys per step, K/V ring
// depth (each K/V tile serves every query tile of the CTA) and S buffers per query tile.
template <bool BIAS>
struct Cfg {
  static constexpr int NT = BIAS ? 1 : 2;
  static constexpr int kThreads = 128 + NT * 128;
  static constexpr int BK = BIAS ? 128 : 64;
  static constexpr int STAGES = BIAS ? 2 : 4;
  static constexpr int SB = BIAS ? 1 : 2;
};

template <int D, bool BIAS>
struct Layout {
  static constexpr int NT = Cfg<BIAS>::NT;
  static constexpr int BK = Cfg<BIAS>::BK;
  static constexpr int STAGES = Cfg<BIAS>::STAGES;
  static constexpr int SB = Cfg<BIAS>::SB;
  static constexpr int NH = D / 64;
  static constexpr int HALF = 128 * 128;        // one 64-column half of a 128-row query tile
  static constexpr int TILE = NH * HALF;
  static constexpr int KHALF = BK * 128;        // one 64-column half of a K or V tile
  static constexpr int KV_TILE = NH * KHALF;
  static constexpr int OFF_Q = 0;               // query tile x at OFF_Q + x*TILE
  static constexpr int OFF_KV = NT * TILE;      // stage s: K at OFF_KV + 2*s*KV_TILE, V after it
  static constexpr int OFF_BIAS = OFF_KV + STAGES * 2 * KV_TILE;
  static constexpr int BIAS_TILE = 2 * HALF;    // [128 query x 128 key], two 64-key halves
  static constexpr int OFF_BAR = OFF_BIAS + (BIAS ? BSTAGES * BIAS_TILE : 0);
  static constexpr int NBAR = 32;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int TOTAL = OFF_MISC + 16;
  static constexpr int ALLOC = (TOTAL + 1024) > 120 * 1024 ? (TOTAL + 1024) : 120 * 1024;
  // TMEM of query tile x: its S buffers, then O
  static constexpr int TCOLS = SB * BK + 128;
  __host__ __device__ static constexpr int col_s(int x, int s) { return x * TCOLS + s * BK; }
  __host__ __device__ static constexpr int col_o(int x) { return x * TCOLS + SB * BK; }
  static_assert(NT * TCOLS <= 512 && D <= 128, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// Barriers.  Per query tile x and S buffer s (index 2x + s): S ready, P written, P read
// by P V (the buffer may take a new S).  Per query tile: P V complete.
template <bool BIAS>
struct Bars {
  static constexpr int ST = Cfg<BIAS>::STAGES;
  static constexpr int Q = 0, KVFULL = 1, KVEMPTY = 1 + ST, S = 1 + 2 * ST, P = S + 4, SFREE = P + 4,
                       PV = SFREE + 4, AFIN = PV + 2, BFULL = AFIN + 1, BEMPTY = BFULL + BSTAGES,
                       END = BEMPTY + BSTAGES;
};
static_assert(Bars<false>::END <= 32 && Bars<true>::END <= 32, "barrier count");

struct Params {
  void* o;
  float* lse;
  unsigned int* status;       // device-wide report word
  unsigned int* call_abort;   // this call's abort word (a slot of a ring)
  unsigned int call_tag;      // what this call stores there when it gives up
  SeqMap m;
  int B, Hq, Hkv, Nq, Nkv;   // Nq, Nkv: the longest lengths of a packed batch
  float scale_log2;
  int causal;
};

__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;
  }
}

template <int D, bool BF16, bool BIAS>
__global__ void __launch_bounds__(Cfg<BIAS>::kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_bias, const Params p) {
  using L = Layout<D, BIAS>;
  using Br = Bars<BIAS>;
  constexpr int NT = L::NT;
  constexpr int BK = L::BK;
  constexpr int STAGES = L::STAGES;
  constexpr int SB = L::SB;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base for the swizzled tiles.  Offsetting the array itself
  // (not a rounded integer) keeps the pointer in the shared address space, so
  // the compiler emits shared-memory loads instead of generic ones.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return sb + L::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  // ---- work item: query tiles 2i and 2i + 1 of head h of sequence b; largest i
  // first (longest under causal).  Both tiles take the same K/V tiles; a CTA
  // runs T = the larger of their KV tile counts, each tile only its own.
  const int BH = p.B * p.Hq;
  const int nPairs = ((p.Nq + BQ - 1) / BQ + NT - 1) / NT;
  const int i = nPairs - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const Seq sq = seq_of(p.m, b, p.status, 50);
  const int hk = h / (p.Hq / p.Hkv);                       // key/value head of the group
  const int bc = bcoord(p.m, b);                           // batch coordinate in the tensor maps
  const int q0 = i * NT * BQ;                               // first row of query tile 0
  const int nKt = (sq.nk + BK - 1) / BK;
  // KV tiles query tile x walks: causal, up to the last key its last row sees
  auto tiles_of = [&](int x) -> int {
    const int qx = q0 + x * BQ;
    const int kmax = min(qx + BQ, sq.nq) - 1 + sq.delta;
    return qx >= sq.nq ? 0 : p.causal ? (kmax < 0 ? 0 : min(nKt, kmax / BK + 1)) : nKt;
  };
  int Tx[NT];
#pragma unroll
  for (int x = 0; x < NT; ++x) Tx[x] = tiles_of(x);
  int T = 0;
#pragma unroll
  for (int x = 0; x < NT; ++x) T = max(T, Tx[x]);

  if (threadIdx.x == 0) {
    mbar_init(bar(Br::Q), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(Br::KVFULL + s), 1);
      mbar_init(bar(Br::KVEMPTY + s), 1);
    }
    for (int x = 0; x < NT; ++x) {        // per query tile
      for (int s = 0; s < SB; ++s) {      // and S buffer
        mbar_init(bar(Br::S + 2 * x + s), 1);
        mbar_init(bar(Br::P + 2 * x + s), 4);   // one arrival per softmax warp
        mbar_init(bar(Br::SFREE + 2 * x + s), 1);
      }
      mbar_init(bar(Br::PV + x), 1);
    }
    mbar_init(bar(Br::AFIN), 1);
    for (int i = 0; i < BSTAGES; ++i) {
      mbar_init(bar(Br::BFULL + i), 1);
      mbar_init(bar(Br::BEMPTY + i), 4);  // one arrival per softmax warp
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
  const WaitCtx wc{p.status, p.call_abort, abort_flag, p.call_tag};

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0 && T > 0 &&
        FA_BOUNDS(h < p.Hq && bc < batch_extent(p.m) && sq.q_start + q0 < rows_q(p.m), wc, 80)) {
      mbar_arrive_expect_tx(bar(Br::Q), NT * L::TILE);
#pragma unroll
      for (int x = 0; x < NT; ++x)
#pragma unroll
        for (int hh = 0; hh < L::NH; ++hh)
          tma_load_4d(sb + L::OFF_Q + x * L::TILE + hh * L::HALF, &tm_q, bar(Br::Q), 64 * hh,
                      sq.q_start + q0 + x * BQ, h, bc);
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % STAGES;
        const uint32_t ph = (t / STAGES) & 1;
        if (!FA_BOUNDS(sq.k_start + t * BK < rows_k(p.m) && hk < p.Hkv, wc, 81)) break;
        if constexpr (BIAS)
          if (!FA_BOUNDS(t * BK < p.Nkv && (p.m.bias_st.n == 0 || q0 < p.Nq) && h < p.Hq && b < p.B, wc, 82)) break;
        if (t >= STAGES && !mbar_wait(bar(Br::KVEMPTY + s), ph ^ 1, wc, 51)) break;
        const uint32_t fb = bar(Br::KVFULL + s);
        mbar_arrive_expect_tx(fb, 2 * L::KV_TILE);
        const uint32_t dst = sb + L::OFF_KV + s * 2 * L::KV_TILE;
#pragma unroll
        for (int hh = 0; hh < L::NH; ++hh) {
          tma_load_4d(dst + hh * L::KHALF, &tm_k, fb, 64 * hh, sq.k_start + t * BK, hk, bc);
          tma_load_4d(dst + L::KV_TILE + hh * L::KHALF, &tm_v, fb, 64 * hh, sq.k_start + t * BK, hk, bc);
        }
        if constexpr (BIAS) {
          // bias of (query rows q0.., keys t*BK..) of head h, sequence b; a broadcast
          // axis has extent 1 in the map and is addressed at 0
          const int bs = t & (BSTAGES - 1);
          if (t >= BSTAGES && !mbar_wait(bar(Br::BEMPTY + bs), ((t / BSTAGES) & 1) ^ 1, wc, 59)) break;
          const uint32_t bb = bar(Br::BFULL + bs);
          mbar_arrive_expect_tx(bb, L::BIAS_TILE);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            tma_load_4d(sb + L::OFF_BIAS + bs * L::BIAS_TILE + hh * L::HALF, &tm_bias, bb, t * BK + 64 * hh,
                        p.m.bias_st.n ? q0 : 0, p.m.bias_st.h ? h : 0, p.m.bias_st.b ? b : 0);
        }
        issued = t + 1;
      }
      drain_wait(bar(Br::Q), 0);
      for (int t = max(0, issued - STAGES); t < issued; ++t)
        drain_wait(bar(Br::KVFULL + t % STAGES), (t / STAGES) & 1);
      if constexpr (BIAS)
        for (int t = max(0, issued - BSTAGES); t < issued; ++t)
          drain_wait(bar(Br::BFULL + (t & (BSTAGES - 1))), (t / BSTAGES) & 1);
    }
  } else if (warp == 1 || warp == 2) {
    // ================================================================ MMA issuers
    if (T > 0) {
      constexpr uint32_t ID_S = make_idesc_f16(128, BK, BF16, false, false);
      constexpr uint32_t ID_O = make_idesc_f16(128, D, BF16, false, true);
      auto s_buf = [&](int x, int t) -> uint32_t { return tmem + L::col_s(x, t % SB); };
      auto o_buf = [&](int x) -> uint32_t { return tmem + L::col_o(x); };
      auto k_tile = [&](int t) -> uint32_t { return sb + L::OFF_KV + (t % STAGES) * 2 * L::KV_TILE; };
      // descriptor advance of k-step ks (16 columns of d) in a K-major tile of 64-column
      // halves of `half` bytes
      auto kstep = [](int ks, int half) -> uint64_t {
        return static_cast<uint64_t>(((ks >> 2) * half + (ks & 3) * 32) >> 4);
      };
      auto wait = [&](uint32_t bb, uint32_t parity, uint32_t site) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bb, parity, wc, site));
      };
      if (warp == 1) {
        // G1: S_x(t) = Q_x K(t)^T for both query tiles into S buffer t mod SB of tile x,
        // once P V of KV tile t - SB has read the P that sits in that buffer
        bool ok = wait(bar(Br::Q), 0, 52);
        for (int t = 0; ok && t < T; ++t) {
          if (!wait(bar(Br::KVFULL + t % STAGES), (t / STAGES) & 1, 53)) break;
          const uint64_t dK_k = sw128_desc(k_tile(t), 16, 1024);
          const int sbi = t % SB;
#pragma unroll
          for (int x = 0; x < NT; ++x) {
            if (t >= Tx[x]) continue;
            if (t >= SB && !wait(bar(Br::SFREE + 2 * x + sbi), ((t - SB) / SB) & 1, 54)) { ok = false; break; }
            tc_fence_after();
            const uint64_t dQ_k = sw128_desc(sb + L::OFF_Q + x * L::TILE, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              umma_ss_warp(s_buf(x, t), dQ_k + kstep(ks, L::HALF), dK_k + kstep(ks, L::KHALF), ID_S, ks > 0);
            umma_commit_warp(bar(Br::S + 2 * x + sbi));
          }
        }
        umma_commit_warp(bar(Br::AFIN));
        drain_wait(bar(Br::AFIN), 0);
      } else {
        // PV: O_x += P_x(t) V(t) (P, 16-bit, packed into the first half of its S buffer;
        // V read MN-major)
        bool ok = true;
        for (int t = 0; ok && t < T; ++t) {
          const uint64_t dV_mn = sw128_desc(k_tile(t) + L::KV_TILE, L::KHALF, 1024);
          const int sbi = t % SB;
#pragma unroll
          for (int x = 0; x < NT; ++x) {
            if (t >= Tx[x]) continue;
            if (!wait(bar(Br::P + 2 * x + sbi), (t / SB) & 1, 55)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)
              umma_ts_warp(o_buf(x), s_buf(x, t) + 8 * ks, dV_mn + static_cast<uint64_t>((ks * 2048) >> 4), ID_O,
                           (t > 0 || ks > 0));
            umma_commit_warp(bar(Br::SFREE + 2 * x + sbi));
            umma_commit_warp(bar(Br::PV + x));
          }
          if (!ok) break;
          umma_commit_warp(bar(Br::KVEMPTY + t % STAGES));   // every G1(t) completed before its P(t) existed
        }
        if (*abort_flag)
          for (int x = 0; x < NT; ++x)
            for (int t = max(0, min(Tx[x], T) - SB); t < Tx[x]; ++t) drain_wait(bar(Br::PV + x), t & 1);
      }
    }
  } else if (warp >= 4) {
    // ================================================================ softmax groups
    const int qt = (warp - 4) >> 2;                     // query tile of this warpgroup
    const int r = threadIdx.x - 128 - 128 * qt;         // query row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + lane_off + L::col_o(qt);
    const int q = q0 + qt * BQ + r;
    const int T = Tx[qt];
    // this thread's row of a staged bias tile (row 0 when the bias broadcasts over queries)
    const int brow = p.m.bias_st.n ? r : 0;
    float m_ref = -CUDART_INF_F;                        // reference max (log2 units); -inf: no key seen yet
    const uint64_t sc2 = f2_bits(p.scale_log2, p.scale_log2);
    float l = 0.f;                                      // sum of 2^(x - m_ref)
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int kv0 = t * BK;
      // columns c >= lim are masked: past the end of K/V, or (causal) after query q
      int lim = sq.nk - kv0;
      if (p.causal) lim = min(lim, q + sq.delta - kv0 + 1);
      const bool need_mask = __any_sync(0xffffffffu, lim < BK);
      const int sbi = t % SB;
      const uint32_t tS = tmem + lane_off + L::col_s(qt, sbi);
      if (!__all_sync(0xffffffffu, mbar_wait(bar(Br::S + 2 * qt + sbi), (t / SB) & 1, wc, 56))) { ok = false; break; }
      tc_fence_after();
      float x[BK];
      if constexpr (BIAS) {
        const int bs = t & (BSTAGES - 1);
        if (!__all_sync(0xffffffffu, mbar_wait(bar(Br::BFULL + bs), (t / BSTAGES) & 1, wc, 60))) { ok = false; break; }
        const uint8_t* btile = smem + L::OFF_BIAS + bs * L::BIAS_TILE + brow * 128;
#pragma unroll
        for (int ch = 0; ch < BK / 32; ++ch) {
          uint32_t sr[32];
          tmem_ld_x32(tS + 32 * ch, sr);
          // x = S * scale * log2(e) + bias * log2(e); keys 32 ch .. 32 ch + 31 are 16-byte
          // chunks 4 ch .. 4 ch + 3 of the row, chunk k of a 128-byte half stored at k ^ (row mod 8)
          float bv[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int k = 4 * ch + j;
            const uint4 u = *reinterpret_cast<const uint4*>(btile + (k >> 3) * L::HALF + (((k & 7) ^ (brow & 7)) << 4));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = unpack2<BF16>(w[e]);
              bv[8 * j + 2 * e] = q < sq.nq ? f.x : 0.f;
              bv[8 * j + 2 * e + 1] = q < sq.nq ? f.y : 0.f;
            }
          }
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c)
            x[32 * ch + c] = fmaf(bv[c], 1.4426950408889634f, __uint_as_float(sr[c]) * p.scale_log2);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Br::BEMPTY + bs));   // this warp's bias reads are done
      } else {
        // all four 32-column loads in flight at once, one wait
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
      // row max over eight independent partial maxima (a single running max is a
      // 128-long dependency chain)
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
        // rescaled, which needs the previous P V to have completed.
        const bool first = m_ref == -CUDART_INF_F;
        const bool resc = !first && mt > m_ref + kRescaleThreshold;
        if (first) m_ref = mt;
        if (__any_sync(0xffffffffu, resc)) {
          if (!__all_sync(0xffffffffu, mbar_wait(bar(Br::PV + qt), (t - 1) & 1, wc, 57))) { ok = false; break; }
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
      float ls[8];                                         // partial row sums
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
        // columns [16ch, 16ch+16) of S were already read
        tmem_st_x16(tS + 16 * ch, pk);
      }
      l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      tmem_st_wait();
      // With two S buffers, the previous P V must have completed before the last P goes out:
      // the epilogue would otherwise have two P V to wait for, and once both have completed, a
      // parity wait for the older one would wait for a phase two ahead.  Here at most that one
      // P V is outstanding.
      if (SB > 1 && t == T - 1 && T > 1 &&
          !__all_sync(0xffffffffu, mbar_wait(bar(Br::PV + qt), (t - 1) & 1, wc, 49))) {
        ok = false;
        break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(Br::P + 2 * qt + sbi));
    }
    // ---- epilogue: O = acc / l (16-bit), L = (m_ref + log2 l) * ln 2
    bool have = ok && T > 0;
    if (have) {
      // the last P V is the only one still outstanding (see the last tile's step above)
      have = __all_sync(0xffffffffu, mbar_wait(bar(Br::PV + qt), (T - 1) & 1, wc, 58));
      tc_fence_after();
    }
    const bool aborted = *abort_flag != 0 || !(q < sq.nq ? FA_BOUNDS(sq.q_start + q < rows_q(p.m), wc, 83) : true);
    const float inv = l > 0.f ? 1.f / l : 0.f;         // a row that saw no key: O = 0
    uint8_t* out = reinterpret_cast<uint8_t*>(p.o) + at(p.m.st.o, p.m, b, h, sq.q_start + q) * 2;
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t pk[16];
      if (have) {
        uint32_t v[32];
        tmem_ld_x32(tO + 32 * ch, v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack2<BF16>(__uint_as_float(v[2 * c]) * inv, __uint_as_float(v[2 * c + 1]) * inv);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = 0u;
      }
      if (q < sq.nq && !aborted) {
        uint4* d4 = reinterpret_cast<uint4*>(out + ch * 64);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          if (32 * ch + 8 * k4 < p.m.d) d4[k4] = make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
      }
    }
    if (q < sq.nq && !aborted)
      p.lse[at(p.m.st.lse, p.m, b, h, sq.q_start + q)] = l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : -CUDART_INF_F;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16, bool BIAS>
cudaError_t launch_t(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& tb, unsigned int* status, unsigned int* call_abort, unsigned int call_tag,
                     cudaStream_t stream) {
  using L = Layout<D, BIAS>;
  constexpr int NT = L::NT;
  auto kern = fwd_kernel<D, BF16, BIAS>;
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
  const long long grid = static_cast<long long>(((a.pb.Nq + BQ - 1) / BQ + NT - 1) / NT) * a.pb.B * a.pb.Hq;
  static_assert(Cfg<BIAS>::BK == (BIAS ? kFwdBKBias : kFwdBK), "K/V tensor-map box rows");
  kern<<<static_cast<unsigned>(grid), Cfg<BIAS>::kThreads, L::ALLOC, stream>>>(tq, tk, tv, tb, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tb, unsigned int* status, unsigned int* call_abort,
                       unsigned int call_tag, cudaStream_t stream) {
  // without a bias: the persistent form of this kernel's no-bias configuration
  if (a.pb.bias == nullptr) return launch_fwd_persist(a, tq, tk, tv, status, call_abort, call_tag, stream);
  if (a.pb.d > 64)
    return a.pb.bf16 ? launch_t<128, true, true>(a, tq, tk, tv, tb, status, call_abort, call_tag, stream)
                     : launch_t<128, false, true>(a, tq, tk, tv, tb, status, call_abort, call_tag, stream);
  return a.pb.bf16 ? launch_t<64, true, true>(a, tq, tk, tv, tb, status, call_abort, call_tag, stream)
                   : launch_t<64, false, true>(a, tq, tk, tv, tb, status, call_abort, call_tag, stream);
}

}  // namespace fa
