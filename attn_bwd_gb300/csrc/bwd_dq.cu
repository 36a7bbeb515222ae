// bwd_dq.cu -- deterministic dQ pass on tcgen05 tensor cores, one CTA per work
// item (the form that serves problems with an additive bias; bwd_dq_persist.cu
// runs the same products persistently for every other problem).
//
// One CTA owns a 128-row query tile of one query head and walks the KV tiles
// it can see in a fixed order, keeping dQ in TMEM, so the summation order of
// every dQ element is fixed and the result is bit-reproducible.  This is the
// query-block grid of flash_attention_backward.cu (rustytorch
// rtx-flash-attention; block "Compute dQ", dQ kept on chip across KV blocks
// and written once) mapped onto sm_103a:
//   G1  S  [BQ x BK] = Q  . K^T      A = Q  (smem, K-major), B = K (K-major)
//   G2  dP [BQ x BK] = dO . V^T      A = dO (smem, K-major), B = V (K-major)
//   G5  dQ [BQ x d ] += dS . K       A = dS (TMEM, 16-bit),  B = K (MN-major)
// and dQ = scale * dQ is written once in the 16-bit dtype.
//
// Warp roles (384 threads):
//   warp 0       TMA producer: Q, dO, -L*log2e, D once; K through a 3-stage ring and
//                V through a 2-stage ring (V is free after dP, K only after dQ)
//   warp 1       owns TMEM; issues G1 and G2 (the products the softmax groups consume)
//   warp 2       issues G5 (the product of what the softmax groups produce)
//   warps 4-11   two softmax groups: thread r of group g owns query row r (TMEM
//                lane r) and KV columns [64g, 64g+64) of each tile
// S is double-buffered in TMEM (S0, S1, dP, dQ = 4 x 128 columns); the dP
// buffer is released as soon as the softmax groups have loaded it, so G2 of
// the next tile overlaps their arithmetic; dS (16-bit) is packed into the S
// buffer it came from and read from there by G5.  The two issuing warps walk
// their loops with all lanes and elect.sync issues each MMA; every hand-off is
// an mbarrier with one arrival per warp.
#include <cstdint>
#include <climits>

#include "kernels.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace fa {
namespace {

constexpr int BQ = 128;    // query rows per CTA (TMEM lanes)
constexpr int BK = 128;    // KV rows per step
constexpr int KST = 3;     // K ring depth: K is held until dQ += dS K of its tile
constexpr int VST = 2;     // V ring depth: V is free once dP = dO V^T of its tile completes
constexpr int kThreads = 384;

template <int D>
struct Layout {
  static constexpr int NH = D / 64;
  static constexpr int HALF = 128 * 128;        // one 64-column half of a 128-row tile
  static constexpr int TILE = NH * HALF;        // one 128-row tile of Q, dO, K or V
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = TILE;
  static constexpr int OFF_K = 2 * TILE;        // K stage s at OFF_K + s*TILE
  static constexpr int OFF_V = OFF_K + KST * TILE;   // V stage s at OFF_V + s*TILE
  static constexpr int OFF_LD = OFF_V + VST * TILE;
  static constexpr int OFF_BAR = OFF_LD + 2 * BQ * 4;
  static constexpr int NBAR = 24;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int TOTAL = OFF_MISC + 16;
  static constexpr int ALLOC = (TOTAL + 1024) > 120 * 1024 ? (TOTAL + 1024) : 120 * 1024;
  static constexpr int COL_S = 0;               // buffers at 0 and BK
  static constexpr int COL_DP = 2 * BK;
  static constexpr int COL_DQ = 3 * BK;
  static_assert(COL_DQ + D <= 512, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

enum : int {
  B_Q = 0, B_KFULL = 1, B_KEMPTY = B_KFULL + KST, B_VFULL = B_KEMPTY + KST, B_VEMPTY = B_VFULL + VST,
  B_S = B_VEMPTY + VST, B_DS = B_S + 2, B_SFREE = B_DS + 2, B_DP = B_SFREE + 2, B_DPFREE, B_ACC, B_AFIN, B_END
};
static_assert(B_END <= 24, "barrier count");

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
};

__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;
  }
}

template <int D, bool BF16, bool BIAS>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const Params p) {
  using L = Layout<D>;
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

  // ---- work item: query tile i of head h of batch b; largest i first (longest under causal)
  const int BH = p.B * p.Hq;
  const int nQt = (p.Nq + BQ - 1) / BQ;
  const int i = nQt - 1 - static_cast<int>(blockIdx.x) / BH;
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int b = bh / p.Hq;
  const int h = bh - b * p.Hq;
  const Seq sq = seq_of(p.m, b, p.status, 20);
  const int hk = h / (p.Hq / p.Hkv);                       // key/value head of the group
  const int bc = bcoord(p.m, b);                           // batch coordinate in the tensor maps
  const int q0 = i * BQ;
  const int nKt = (sq.nk + BK - 1) / BK;
  const int qmax = min(q0 + BQ, sq.nq) - 1;
  // causal: the last key any row of this tile sees is qmax + delta (none if negative)
  const int kmax = qmax + sq.delta;
  const int T = q0 >= sq.nq ? 0 : p.causal ? (kmax < 0 ? 0 : min(nKt, kmax / BK + 1)) : nKt;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q), 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(bar(B_KFULL + s), 1);
      mbar_init(bar(B_KEMPTY + s), 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(bar(B_VFULL + s), 1);
      mbar_init(bar(B_VEMPTY + s), 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(bar(B_S + j), 1);
      mbar_init(bar(B_DS + j), 8);      // one arrival per softmax warp
      mbar_init(bar(B_SFREE + j), 1);
    }
    mbar_init(bar(B_DP), 1);
    mbar_init(bar(B_DPFREE), 8);
    mbar_init(bar(B_ACC), 1);
    mbar_init(bar(B_AFIN), 1);
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

  if (warp == 0) {
    // ================================================================ TMA producer
    const size_t ws_rows = static_cast<size_t>(p.B) * p.Hq * p.NqPad;
    // (a tile past its sequence's end, T == 0, is still loaded -- from the next sequence's
    // rows or as zero fill -- and never used)
    if (lane == 0 && FA_BOUNDS(h < p.Hq && bc < batch_extent(p.m) &&
                                   (q0 >= sq.nq || sq.q_start + q0 < rows_q(p.m)) &&
                                   static_cast<size_t>(bh) * p.NqPad + q0 + BQ <= ws_rows,
                               wc, 70)) {
      mbar_arrive_expect_tx(bar(B_Q), 2 * L::TILE + 2 * BQ * 4);
#pragma unroll
      for (int hh = 0; hh < L::NH; ++hh) {
        tma_load_4d(sb + L::OFF_Q + hh * L::HALF, &tm_q, bar(B_Q), 64 * hh, sq.q_start + q0, h, bc);
        tma_load_4d(sb + L::OFF_DO + hh * L::HALF, &tm_do, bar(B_Q), 64 * hh, sq.q_start + q0, h, bc);
      }
      const size_t row = static_cast<size_t>(bh) * p.NqPad + q0;
      bulk_load(sb + L::OFF_LD, p.nLg + row, BQ * 4, bar(B_Q));
      bulk_load(sb + L::OFF_LD + BQ * 4, p.Dv + row, BQ * 4, bar(B_Q));
      int k_issued = 0, v_issued = 0;
      for (int t = 0; t < T; ++t) {
        // K(t) once dQ(t - KST) has read its slot; V(t) once dP(t - VST) has read its slot
        // (dP(t - 2) completes before dQ(t - 2), so the V wait never holds back K(t + 1))
        const int ks = t % KST, vs = t % VST;
        if (!FA_BOUNDS(sq.k_start + t * BK < rows_k(p.m) && hk < p.Hkv, wc, 71)) break;
        if (t >= KST && !mbar_wait(bar(B_KEMPTY + ks), ((t / KST) & 1) ^ 1, wc, 21)) break;
        mbar_arrive_expect_tx(bar(B_KFULL + ks), L::TILE);
#pragma unroll
        for (int hh = 0; hh < L::NH; ++hh)
          tma_load_4d(sb + L::OFF_K + ks * L::TILE + hh * L::HALF, &tm_k, bar(B_KFULL + ks), 64 * hh,
                      sq.k_start + t * BK, hk, bc);
        k_issued = t + 1;
        if (t >= VST && !mbar_wait(bar(B_VEMPTY + vs), ((t / VST) & 1) ^ 1, wc, 20)) break;
        mbar_arrive_expect_tx(bar(B_VFULL + vs), L::TILE);
#pragma unroll
        for (int hh = 0; hh < L::NH; ++hh)
          tma_load_4d(sb + L::OFF_V + vs * L::TILE + hh * L::HALF, &tm_v, bar(B_VFULL + vs), 64 * hh,
                      sq.k_start + t * BK, hk, bc);
        v_issued = t + 1;
      }
      drain_wait(bar(B_Q), 0);
      for (int t = max(0, k_issued - KST); t < k_issued; ++t) drain_wait(bar(B_KFULL + t % KST), (t / KST) & 1);
      for (int t = max(0, v_issued - VST); t < v_issued; ++t) drain_wait(bar(B_VFULL + t % VST), (t / VST) & 1);
    }
  } else if (warp == 1 || warp == 2) {
    // ================================================================ MMA issuers
    if (T > 0) {
      constexpr uint32_t ID_S = make_idesc_f16(128, BK, BF16, false, false);
      constexpr uint32_t ID_Q = make_idesc_f16(128, D, BF16, false, true);
      const uint32_t tdP = tmem + L::COL_DP, tdQ = tmem + L::COL_DQ;
      const uint64_t dQ_k = sw128_desc(sb + L::OFF_Q, 16, 1024), dO_k = sw128_desc(sb + L::OFF_DO, 16, 1024);
      auto s_buf = [&](int t) -> uint32_t { return tmem + L::COL_S + (t & 1) * BK; };
      auto k_tile = [&](int t) -> uint32_t { return sb + L::OFF_K + (t % KST) * L::TILE; };
      auto v_tile = [&](int t) -> uint32_t { return sb + L::OFF_V + (t % VST) * L::TILE; };
      // K-major step ks (16 elements of d): 64-column half ks/4, 32 bytes per step inside it
      auto kstep = [](int ks) -> uint64_t {
        return static_cast<uint64_t>(((ks >> 2) * L::HALF + (ks & 3) * 32) >> 4);
      };
      auto wait = [&](uint32_t bb, uint32_t parity, uint32_t site) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(bb, parity, wc, site));
      };
      if (warp == 1) {
        bool ok = wait(bar(B_Q), 0, 22);
        for (int t = 0; ok && t < T; ++t) {
          if (!wait(bar(B_KFULL + t % KST), (t / KST) & 1, 23)) break;
          if (t >= 2 && !wait(bar(B_SFREE + (t & 1)), ((t - 2) >> 1) & 1, 24)) break;
          tc_fence_after();
          const uint64_t dK_k = sw128_desc(k_tile(t), 16, 1024), dV_k = sw128_desc(v_tile(t), 16, 1024);
          // G1: S = Q K^T into buffer t & 1
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) umma_ss_warp(s_buf(t), dQ_k + kstep(ks), dK_k + kstep(ks), ID_S, ks > 0);
          umma_commit_warp(bar(B_S + (t & 1)));
          // G2: dP = dO V^T, once the softmax groups have loaded dP of the previous tile
          if (!wait(bar(B_VFULL + t % VST), (t / VST) & 1, 19)) break;
          if (t >= 1 && !wait(bar(B_DPFREE), (t - 1) & 1, 25)) break;
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) umma_ss_warp(tdP, dO_k + kstep(ks), dV_k + kstep(ks), ID_S, ks > 0);
          umma_commit_warp(bar(B_DP));
          umma_commit_warp(bar(B_VEMPTY + t % VST));     // V(t) is read by G2(t) only
        }
        umma_commit_warp(bar(B_AFIN));   // this warp's MMAs complete before TMEM is released
        drain_wait(bar(B_AFIN), 0);
      } else {
        for (int t = 0; t < T; ++t) {
          // G5: dQ += dS K  (dS, 16-bit, packed into the first half of each group's
          // 64 columns of the S buffer; K read MN-major)
          if (!wait(bar(B_DS + (t & 1)), (t >> 1) & 1, 26)) break;
          tc_fence_after();
          const uint64_t dK_mn = sw128_desc(k_tile(t), L::HALF, 1024);
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            umma_ts_warp(tdQ, s_buf(t) + 64 * (ks >> 2) + 8 * (ks & 3),
                         dK_mn + static_cast<uint64_t>((ks * 2048) >> 4), ID_Q, (t > 0 || ks > 0));
          umma_commit_warp(bar(B_SFREE + (t & 1)));
          // K(t): G1(t) has completed (dS(t) depends on it); G5(t) is tracked here
          umma_commit_warp(bar(B_KEMPTY + t % KST));
        }
        umma_commit_warp(bar(B_ACC));
        if (*abort_flag) drain_wait(bar(B_ACC), 0);
      }
    }
  } else if (warp >= 4) {
    // ================================================================ softmax / dS groups
    const int grp = (warp - 4) >> 2;                    // KV columns [64 grp, 64 grp + 64)
    const int r = threadIdx.x - 128 - 128 * grp;       // query row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tdP = tmem + lane_off + L::COL_DP + 64 * grp;
    const int q = q0 + r;
    const uint16_t* brow = nullptr;                    // this row of the bias
    if constexpr (BIAS) brow = static_cast<const uint16_t*>(p.m.bias) + bias_row(p.m.bias_st, b, h, q);
    bool ok = __all_sync(0xffffffffu, mbar_wait(bar(B_Q), 0, wc, 27));
    const float* LD = reinterpret_cast<const float*>(smem + L::OFF_LD);
    const float nlq = ok ? LD[r] : 0.f;                // -L*log2(e) of this query row
    const float dq_ = ok ? LD[BQ + r] : 0.f;
    const uint64_t sc2 = f2_bits(p.scale_log2, p.scale_log2);
    const uint64_t nl2 = f2_bits(nlq, nlq);
    const uint64_t dd2 = f2_bits(dq_, dq_);
    for (int t = 0; ok && t < T; ++t) {
      const int kv0 = t * BK;
      // columns c >= lim are masked: past the end of K/V, or (causal) after query q
      int lim = sq.nk - kv0 - 64 * grp;
      if (p.causal) lim = min(lim, q + sq.delta - kv0 - 64 * grp + 1);
      const bool need_mask = __any_sync(0xffffffffu, lim < 64);
      const uint32_t tS = tmem + lane_off + L::COL_S + (t & 1) * BK + 64 * grp;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_DP), t & 1, wc, 28))) break;
      tc_fence_after();
      uint32_t dr[64];
      tmem_ld_x32(tdP, *reinterpret_cast<uint32_t(*)[32]>(dr));
      tmem_ld_x32(tdP + 32, *reinterpret_cast<uint32_t(*)[32]>(dr + 32));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DPFREE));       // the dP buffer may take the next tile's G2
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_S + (t & 1)), (t >> 1) & 1, wc, 29))) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t sr[32], pk[16];
        tmem_ld_x32(tS + 32 * ch, sr);
        float bv[32];                                  // bias of (query q, keys of this chunk)
        if constexpr (BIAS) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float v8[8];
            if (q < sq.nq) {
              bias8<BF16>(brow, kv0 + 64 * grp + 32 * ch + 8 * j, sq.nk, v8);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) v8[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) bv[8 * j + e] = v8[e];
          }
        }
        tmem_ld_wait();
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) {
          const int c = 32 * ch + 2 * c2;
          float2 x = f2_split(fma_f32x2(f2_bits(__uint_as_float(sr[2 * c2]), __uint_as_float(sr[2 * c2 + 1])), sc2, nl2));
          if constexpr (BIAS) {
            x.x = fmaf(bv[2 * c2], 1.4426950408889634f, x.x);
            x.y = fmaf(bv[2 * c2 + 1], 1.4426950408889634f, x.y);
          }
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
      if (lane == 0) mbar_arrive(bar(B_DS + (t & 1)));
    }
    // ---- epilogue: dQ = scale * acc, 16-bit; group g writes columns [D/2 g, D/2 (g+1))
    bool have = ok && T > 0;
    if (have) {
      have = __all_sync(0xffffffffu, mbar_wait(bar(B_ACC), 0, wc, 30));
      tc_fence_after();
    }
    const bool aborted = *abort_flag != 0;
    uint8_t* out = reinterpret_cast<uint8_t*>(p.dq) + at(p.m.st.dq, p.m, b, h, sq.q_start + q) * 2;
#pragma unroll 1
    for (int ch = 0; ch < D / 64; ++ch) {
      const int col = (D / 2) * grp + 32 * ch;
      uint32_t pk[16];
      if (have) {
        uint32_t v[32];
        tmem_ld_x32(tmem + lane_off + L::COL_DQ + col, v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack2<BF16>(__uint_as_float(v[2 * c]) * p.scale, __uint_as_float(v[2 * c + 1]) * p.scale);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = 0u;
      }
      if (q < sq.nq && !aborted && FA_BOUNDS(sq.q_start + q < rows_q(p.m), wc, 72)) {
        uint4* d4 = reinterpret_cast<uint4*>(out + col * 2);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          if (col + 8 * k4 < p.m.d) d4[k4] = make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
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

template <int D, bool BF16, bool BIAS>
cudaError_t launch_t(const DqArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                     const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  using L = Layout<D>;
  auto kern = bwd_dq_kernel<D, BF16, BIAS>;
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
  const long long grid = static_cast<long long>((a.pb.Nq + BQ - 1) / BQ) * a.pb.B * a.pb.Hq;
  kern<<<static_cast<unsigned>(grid), kThreads, L::ALLOC, stream>>>(tq, tdo, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_det(const DqArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                              const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  if (use_persistent(a.pb)) return launch_bwd_dq_persist(a, tq, tdo, tk, tv, stream);
  const bool bias = a.pb.bias != nullptr;
  if (a.pb.d > 64) {
    if (a.pb.bf16)
      return bias ? launch_t<128, true, true>(a, tq, tdo, tk, tv, stream)
                  : launch_t<128, true, false>(a, tq, tdo, tk, tv, stream);
    return bias ? launch_t<128, false, true>(a, tq, tdo, tk, tv, stream)
                : launch_t<128, false, false>(a, tq, tdo, tk, tv, stream);
  }
  if (a.pb.bf16)
    return bias ? launch_t<64, true, true>(a, tq, tdo, tk, tv, stream)
                : launch_t<64, true, false>(a, tq, tdo, tk, tv, stream);
  return bias ? launch_t<64, false, true>(a, tq, tdo, tk, tv, stream)
              : launch_t<64, false, false>(a, tq, tdo, tk, tv, stream);
}

}  // namespace fa
