// bwd_dq.cu -- deterministic dQ pass on tcgen05 tensor cores.
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
// Warp roles (256 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA
// issuer, warps 4-7 thread r owns query row r (TMEM lane r).
#include <cstdint>
#include <climits>

#include "kernels.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int BQ = 128;    // query rows per CTA (TMEM lanes)
constexpr int BK = 128;    // KV rows per step
constexpr int STAGES = 2;  // K/V ring depth
constexpr int kThreads = 256;

template <int D>
struct Layout {
  static constexpr int NH = D / 64;
  static constexpr int HALF = 128 * 128;        // one 64-column half of a 128-row tile
  static constexpr int TILE = NH * HALF;        // one 128-row tile of Q, dO, K or V
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = TILE;
  static constexpr int OFF_KV = 2 * TILE;       // stage s: K at OFF_KV + 2*s*TILE, V after it
  static constexpr int OFF_LD = OFF_KV + STAGES * 2 * TILE;
  static constexpr int OFF_BAR = OFF_LD + 2 * BQ * 4;
  static constexpr int NBAR = 12;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int TOTAL = OFF_MISC + 16;
  static constexpr int ALLOC = (TOTAL + 1024) > 120 * 1024 ? (TOTAL + 1024) : 120 * 1024;
  static constexpr int COL_S = 0;
  static constexpr int COL_DP = BK;
  static constexpr int COL_DQ = 2 * BK;
  static_assert(COL_DQ + D <= 512, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

enum : int { B_Q = 0, B_KVFULL = 1, B_KVEMPTY = 1 + STAGES, B_S = 1 + 2 * STAGES, B_DP, B_DS, B_ACC, B_END };

struct Params {
  const float* nLg;
  const float* Dv;
  void* dq;
  unsigned int* status;
  int B, Hq, Hkv, Nq, Nkv, NqPad;
  float scale, scale_log2;
  int causal;
};

__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const Params p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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
  const int kvh = b * p.Hkv + h / (p.Hq / p.Hkv);
  const int q0 = i * BQ;
  const int nKt = (p.Nkv + BK - 1) / BK;
  const int qmax = min(q0 + BQ, p.Nq) - 1;
  const int T = p.causal ? min(nKt, qmax / BK + 1) : nKt;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(B_KVFULL + s), 1);
      mbar_init(bar(B_KVEMPTY + s), 1);
    }
    mbar_init(bar(B_S), 1);
    mbar_init(bar(B_DP), 1);
    mbar_init(bar(B_DS), 128);
    mbar_init(bar(B_ACC), 1);
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
  const WaitCtx wc{p.status, abort_flag};

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(B_Q), 2 * L::TILE + 2 * BQ * 4);
#pragma unroll
      for (int hh = 0; hh < L::NH; ++hh) {
        tma_load_3d(sb + L::OFF_Q + hh * L::HALF, &tm_q, bar(B_Q), 64 * hh, q0, bh);
        tma_load_3d(sb + L::OFF_DO + hh * L::HALF, &tm_do, bar(B_Q), 64 * hh, q0, bh);
      }
      const size_t row = static_cast<size_t>(bh) * p.NqPad + q0;
      bulk_load(sb + L::OFF_LD, p.nLg + row, BQ * 4, bar(B_Q));
      bulk_load(sb + L::OFF_LD + BQ * 4, p.Dv + row, BQ * 4, bar(B_Q));
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = t % STAGES;
        const uint32_t ph = (t / STAGES) & 1;
        if (t >= STAGES && !mbar_wait(bar(B_KVEMPTY + s), ph ^ 1, wc, 21)) break;
        const uint32_t fb = bar(B_KVFULL + s);
        mbar_arrive_expect_tx(fb, 2 * L::TILE);
        const uint32_t dst = sb + L::OFF_KV + s * 2 * L::TILE;
#pragma unroll
        for (int hh = 0; hh < L::NH; ++hh) {
          tma_load_3d(dst + hh * L::HALF, &tm_k, fb, 64 * hh, t * BK, kvh);
          tma_load_3d(dst + L::TILE + hh * L::HALF, &tm_v, fb, 64 * hh, t * BK, kvh);
        }
        issued = t + 1;
      }
      drain_wait(bar(B_Q), 0);
      for (int t = max(0, issued - STAGES); t < issued; ++t)
        drain_wait(bar(B_KVFULL + t % STAGES), (t / STAGES) & 1);
    }
  } else if (warp == 1) {
    {   // the whole warp walks the loop; elect.sync issues each MMA
      constexpr uint32_t ID_S = make_idesc_f16(128, BK, BF16, false, false);
      constexpr uint32_t ID_Q = make_idesc_f16(128, D, BF16, false, true);
      const uint32_t tS = tmem + L::COL_S, tdP = tmem + L::COL_DP, tdQ = tmem + L::COL_DQ;
      const uint64_t dQ_k = sw128_desc(sb + L::OFF_Q, 16, 1024), dO_k = sw128_desc(sb + L::OFF_DO, 16, 1024);
      bool ok = __all_sync(0xffffffffu, mbar_wait(bar(B_Q), 0, wc, 22));
      for (int t = 0; ok && t < T; ++t) {
        const int s = t % STAGES;
        const uint32_t ph = (t / STAGES) & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_KVFULL + s), ph, wc, 23))) break;
        tc_fence_after();
        const uint32_t aK = sb + L::OFF_KV + s * 2 * L::TILE;
        const uint32_t aV = aK + L::TILE;
        // descriptors built once per tile, stepped by compile-time offsets >> 4
        const uint64_t dK_k = sw128_desc(aK, 16, 1024), dV_k = sw128_desc(aV, 16, 1024);
        const uint64_t dK_mn = sw128_desc(aK, L::HALF, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t o = static_cast<uint64_t>(((ks >> 2) * L::HALF + (ks & 3) * 32) >> 4);
          umma_ss_warp(tS, dQ_k + o, dK_k + o, ID_S, ks > 0);
        }
        umma_commit_warp(bar(B_S));
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t o = static_cast<uint64_t>(((ks >> 2) * L::HALF + (ks & 3) * 32) >> 4);
          umma_ss_warp(tdP, dO_k + o, dV_k + o, ID_S, ks > 0);
        }
        umma_commit_warp(bar(B_DP));
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_DS), t & 1, wc, 24))) break;
        tc_fence_after();
        // dQ += dS K: dS (16-bit) in the first BK/2 columns of S, K read MN-major
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks)
          umma_ts_warp(tdQ, tS + ks * 8, dK_mn + static_cast<uint64_t>((ks * 2048) >> 4), ID_Q, (t > 0 || ks > 0));
        umma_commit_warp(bar(B_KVEMPTY + s));
      }
      umma_commit_warp(bar(B_ACC));
      if (*abort_flag) drain_wait(bar(B_ACC), 0);
    }
  } else if (warp >= 4) {
    const int r = threadIdx.x - 128;                  // query row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + L::COL_S;
    const uint32_t tdP = tmem + lane_off + L::COL_DP;
    const int q = q0 + r;
    bool ok = __all_sync(0xffffffffu, mbar_wait(bar(B_Q), 0, wc, 25));
    const float* LD = reinterpret_cast<const float*>(smem + L::OFF_LD);
    const float nlq = ok ? LD[r] : 0.f;                // -L*log2(e) of this query row
    const float dq_ = ok ? LD[BQ + r] : 0.f;
    for (int t = 0; ok && t < T; ++t) {
      const int kv0 = t * BK;
      // columns c >= lim are masked: past the end of K/V, or (causal) after query q
      int lim = p.Nkv - kv0;
      if (p.causal) lim = min(lim, q - kv0 + 1);
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_S), t & 1, wc, 26))) break;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_DP), t & 1, wc, 27))) break;
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < BK / 32; ++ch) {
        uint32_t sr[32], dr[32], pk[16];
        tmem_ld_x32(tS + ch * 32, sr);
        tmem_ld_x32(tdP + ch * 32, dr);
        tmem_ld_wait();
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) {
          const int c = ch * 32 + 2 * c2;
          float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * c2]), p.scale_log2, nlq));
          float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * c2 + 1]), p.scale_log2, nlq));
          if (c >= lim) p0 = 0.f;
          if (c + 1 >= lim) p1 = 0.f;
          pk[c2] = pack2<BF16>(p0 * (__uint_as_float(dr[2 * c2]) - dq_),
                               p1 * (__uint_as_float(dr[2 * c2 + 1]) - dq_));
        }
        // columns [16ch, 16ch+16) of S were already read (chunk ch covers [32ch, 32ch+32))
        tmem_st_x16(tS + ch * 16, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(B_DS));
    }
    // ---- epilogue: dQ = scale * acc, 16-bit
    bool have = ok && T > 0;
    if (have) {
      have = __all_sync(0xffffffffu, mbar_wait(bar(B_ACC), 0, wc, 28));
      tc_fence_after();
    }
    const bool aborted = *abort_flag != 0;
    uint8_t* out = reinterpret_cast<uint8_t*>(p.dq) + (static_cast<size_t>(bh) * p.Nq + q) * D * 2;
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t pk[16];
      if (have) {
        uint32_t v[32];
        tmem_ld_x32(tmem + lane_off + L::COL_DQ + ch * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack2<BF16>(__uint_as_float(v[2 * c]) * p.scale, __uint_as_float(v[2 * c + 1]) * p.scale);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = 0u;
      }
      if (q < p.Nq && !aborted) {
        uint4* d4 = reinterpret_cast<uint4*>(out + ch * 64);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) d4[k4] = make_uint4(pk[4 * k4], pk[4 * k4 + 1], pk[4 * k4 + 2], pk[4 * k4 + 3]);
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
cudaError_t launch_t(const DqArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                     const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  using L = Layout<D>;
  auto kern = bwd_dq_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  Params p;
  p.nLg = a.ws.nLg;
  p.Dv = a.ws.Dv;
  p.dq = a.dq;
  p.status = a.status;
  p.B = a.pb.B; p.Hq = a.pb.Hq; p.Hkv = a.pb.Hkv; p.Nq = a.pb.Nq; p.Nkv = a.pb.Nkv; p.NqPad = a.pb.NqPad;
  p.scale = a.pb.scale;
  p.scale_log2 = a.pb.scale * 1.4426950408889634f;
  p.causal = a.pb.causal;
  const long long grid = static_cast<long long>((a.pb.Nq + BQ - 1) / BQ) * a.pb.B * a.pb.Hq;
  kern<<<static_cast<unsigned>(grid), kThreads, L::ALLOC, stream>>>(tq, tdo, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq_det(const DqArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                              const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
  if (a.pb.d == 128)
    return a.pb.bf16 ? launch_t<128, true>(a, tq, tdo, tk, tv, stream) : launch_t<128, false>(a, tq, tdo, tk, tv, stream);
  return a.pb.bf16 ? launch_t<64, true>(a, tq, tdo, tk, tv, stream) : launch_t<64, false>(a, tq, tdo, tk, tv, stream);
}

}  // namespace fa
