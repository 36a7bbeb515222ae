// bwd_main.cu -- KV-tile-parallel attention backward on tcgen05 tensor cores,
// one CTA per work item.  Problems without an additive bias run the same
// products in the persistent schedule of bwd_main_persist.cu; this kernel is
// launched for the bias path (it stages bias tiles and stores dBias).
//
// Decomposition: the sequence-parallel scheme of "Extra transposes cause 8x
// speedup for sequence-parallel Flash Attention backward" (triton #1806,
// "Minimal Repro"): one program per (batch, head, KV block) keeps its K and V
// block resident, walks every query block, accumulates dK and dV on chip and
// stores them once, while dQ contributions are added into an fp32 buffer.
// Here one CTA owns a 128-row KV tile of one key/value head and walks the
// query tiles of every query head of its GQA group ("[Kernel] Flash attention
// 2", Liger-Kernel #275, "Details"), so dK/dV are reduced over the group on
// chip.  The per-tile arithmetic is that of flash_attention_backward.cu
// (rustytorch rtx-flash-attention): recompute S, P = exp(S - L), dV += P^T dO,
// dP = dO V^T, dS = P o (dP - D), dK += dS^T Q, dQ += dS K.
//
// sm_103a mapping (BN = 128 KV rows on the TMEM lanes, BM = 64 query rows):
//   G1  S^T [BN x BM]  = K  . Q^T      A = K  (smem, K-major), B = Q  (K-major)
//   G2  dP^T[BN x BM]  = V  . dO^T     A = V  (smem, K-major), B = dO (K-major)
//   G3  dV  [BN x d ] += P^T . dO      A = P^T  (TMEM, 16-bit), B = dO (MN-major)
//   G4  dK  [BN x d ] += dS^T . Q      A = dS^T (smem, K-major), B = Q  (MN-major)
//   G5  dQ^T[d  x BM]  = K^T . dS^T    A = K  (smem, MN-major), B = dS^T (smem, MN-major)
// Every operand is read in place from the TMA-written tiles through
// descriptors of the right major-ness: no transposed copies exist.  That is
// the lesson of triton #1806, where the orientation of the dQ product alone
// made an 8x difference.
//
// Warp roles (512 threads):
//   warp 0       TMA producer: K, V once; Q, dO, L, D tiles through a 4-stage ring
//                (3 stages with an additive bias, whose [64 query x 128 key]
//                tiles then flow through a 2-stage ring of their own)
//   warp 1       owns TMEM; one lane issues every tcgen05.mma
//   warps 4-11   two "softmax" groups: thread r of group w owns KV row r (TMEM
//                lane r) and query columns [32w, 32w+32) of each tile; P, dS
//   warps 12-15  dQ group: TMEM -> registers -> red.global.add.f32 into the
//                workspace accumulator, one 128-byte row segment per warp
//                instruction (idle in deterministic mode)
//   epilogue     group 0 writes dK (x scale), group 1 writes dV
//
// Schedule.  S^T is double-buffered in TMEM and computed two tiles ahead:
//   G1(0) G2(0) G1(1) | per t: [P(t)] G3(t) G1(t+2) [dP(t) loaded] G2(t+1) [dS(t)] G4(t) G5(t)
// where [x] waits for the softmax groups.  When the softmax groups finish
// dS(t), S^T(t+1) is already in TMEM, so they go straight on to P(t+1) while
// the tensor core runs G4/G5 of tile t.  dS^T goes only to shared memory, so
// the single dP^T buffer is free as soon as the softmax groups have loaded it
// and G2(t+1) overlaps their dS(t) arithmetic.  The MMA unit executes one
// CTA's tcgen05.mma instructions in issue order, which is what lets G1(t+2)
// reuse the S^T buffer that G3(t) read without a further wait.  The ring keeps
// Q/dO loads about two tiles ahead of their first use (a load under full load
// takes ~1 us).
#include <cstdint>
#include <climits>

#include "kernels.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace fa {
namespace {

constexpr int BN = kMainBN;   // KV rows per CTA (TMEM lanes)
constexpr int BM = kMainBM;   // query rows per tile
constexpr int BSTAGES = 2;    // bias tiles in flight (with an additive bias)
constexpr int kThreads = 512;
constexpr int kGroupChunk = 32;   // (batch, kv-head) groups per launch-order chunk

template <int D, bool BIAS>
struct Layout {
  // Q/dO ring depth: loads run ~2 tiles ahead of use.  With a bias, one stage
  // makes room for the bias ring (two [BM query][BN key] tiles).
  static constexpr int STAGES = BIAS ? 3 : 4;
  static constexpr int NH = D / 64;               // 64-column halves of a row
  static constexpr int KHALF = BN * 128;          // bytes of one half of a K/V tile
  static constexpr int QHALF = BM * 128;          // bytes of one half of a Q/dO tile
  static constexpr int KV_BYTES = NH * KHALF;
  static constexpr int Q_BYTES = NH * QHALF;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KV_BYTES;
  static constexpr int OFF_Q = OFF_V + KV_BYTES;
  static constexpr int OFF_DO = OFF_Q + STAGES * Q_BYTES;
  static constexpr int OFF_DS = OFF_DO + STAGES * Q_BYTES;
  static constexpr int DS_BYTES = BN * BM * 2;    // dS^T, 128 rows x 128 B
  static constexpr int OFF_BIAS = OFF_DS + DS_BYTES;
  static constexpr int BIAS_BYTES = BM * BN * 2;  // bias of one tile: BM rows (queries) of BN keys, 256 B each
  static constexpr int OFF_DB = OFF_BIAS + (BIAS ? BSTAGES * BIAS_BYTES : 0);
  static constexpr int DB_HALF = 32 * BN * 2;     // dBias of one softmax group's 32 queries
  static constexpr int OFF_LD = OFF_DB + (BIAS ? 2 * DB_HALF : 0);
  static constexpr int LD_BYTES = 2 * BM * 4;     // -L*log2e and D of one tile
  static constexpr int OFF_BAR = OFF_LD + STAGES * LD_BYTES;
  static constexpr int NBAR = 32;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int TOTAL = OFF_MISC + 16;
  static constexpr int ALLOC = TOTAL + 1024;      // slack for 1024-byte alignment
  // TMEM columns (fp32 accumulators).  Two S^T buffers; the 16-bit P^T of
  // query columns [32w, 32w+32) is packed into columns [32w, 32w+16) of its
  // S^T buffer, i.e. into the half its own softmax group already read.
  static constexpr int COL_DK = 0;
  static constexpr int COL_DV = D;
  static constexpr int COL_S = 2 * D;               // buffers at COL_S and COL_S + BM
  static constexpr int COL_DP = 2 * D + 2 * BM;
  static constexpr int COL_DQ = 2 * D + 3 * BM;
  static_assert(COL_DQ + BM <= 512, "TMEM budget");
  static_assert(ALLOC <= 232448, "shared memory budget");
};
// barrier indices
// (S and P have one barrier per S^T buffer: tile t uses buffer t & 1)
template <int STAGES>
struct Bars {
  static constexpr int KV = 0, QFULL = 1, QEMPTY = 1 + STAGES, S = 1 + 2 * STAGES, P = S + 2, SFREE = P + 2,
                       DP = SFREE + 2, DPFREE = DP + 1, DS = DP + 2, DQFULL = DP + 3, DQEMPTY = DP + 4,
                       DSFREE = DP + 5, ACC = DP + 6, AFIN = DP + 7, BFULL = DP + 8, BEMPTY = BFULL + BSTAGES,
                       DBFULL = BEMPTY + BSTAGES, DBFREE = DBFULL + 2, END = DBFREE + 2;
};
static_assert(Bars<3>::END <= Layout<128, true>::NBAR, "barrier count");

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
};

// Bounded wait that ignores the abort flag: used only to drain work already
// in flight before the CTA releases TMEM and exits.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) return;
  }
}

// Stores the 16-byte pieces of a 32-column chunk that lie within the row's `cols` columns.
template <bool BF16>
__device__ __forceinline__ void store_row_chunk(void* dst, const uint32_t (&pk)[16], int cols) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (8 * i < cols) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

template <int D, bool BF16, bool DET, bool BIAS>
__global__ void __launch_bounds__(kThreads, 1)
bwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_bias, const __grid_constant__ CUtensorMap tm_dbias,
                const Params p) {
  using L = Layout<D, BIAS>;
  using BR = Bars<L::STAGES>;
  constexpr int STAGES = L::STAGES;
  // ring stage and phase of tile t
  auto stg = [](int t) -> int { return static_cast<int>(static_cast<unsigned>(t) % STAGES); };
  auto rph = [](int t) -> uint32_t { return (static_cast<unsigned>(t) / STAGES) & 1u; };
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

  // ---- work item: KV tile j of key/value head hkv of batch b.  The (batch,
  // kv-head) groups are taken in chunks of kGroupChunk, and inside a chunk the
  // order is tile-major, so that under causal masking the longest CTAs (small j)
  // start first and several KV tiles of each group run at the same time: they
  // sweep the same query tiles together, so their dQ reductions meet in L2.
  // (With more groups in flight than that, each group has about one CTA live
  // and nearly every reduction misses L2; a fully group-major order measured
  // slower on the dense headline, whose 32 groups fit one chunk.)
  const int groups = p.B * p.Hkv;
  const int nKt = (p.Nkv + BN - 1) / BN;
  const int chunk = static_cast<int>(blockIdx.x) / (kGroupChunk * nKt);
  const int rem = static_cast<int>(blockIdx.x) - chunk * (kGroupChunk * nKt);
  const int cg = min(kGroupChunk, groups - chunk * kGroupChunk);   // groups in this chunk
  const int j = rem / cg;
  const int gi = chunk * kGroupChunk + (rem - j * cg);
  const int b = gi / p.Hkv;
  const int hkv = gi - b * p.Hkv;
  const int G = p.Hq / p.Hkv;
  const Seq sq = seq_of(p.m, b, p.status, 40);
  const int kv0 = j * BN;
  const int nQt = (sq.nq + BM - 1) / BM;
  // first query tile that sees this KV tile: causal, query q sees key kv0 when q >= kv0 - delta
  const int qfirst = kv0 - sq.delta;
  const int i0 = p.causal ? (qfirst <= 0 ? 0 : min(qfirst / BM, nQt)) : 0;
  const int per_head = nQt - i0;
  const int T = kv0 < sq.nk ? G * per_head : 0;       // tiles this CTA processes

  if (threadIdx.x == 0) {
    mbar_init(bar(BR::KV), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(BR::QFULL + s), 1);
      mbar_init(bar(BR::QEMPTY + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(BR::S + i), 1);
      mbar_init(bar(BR::P + i), 8);        // one arrival per softmax warp
      mbar_init(bar(BR::SFREE + i), 1);
    }
    mbar_init(bar(BR::AFIN), 1);
    mbar_init(bar(BR::DP), 1);
    mbar_init(bar(BR::DPFREE), 8);
    mbar_init(bar(BR::DS), 8);
    mbar_init(bar(BR::DQFULL), 1);
    mbar_init(bar(BR::DQEMPTY), 4);      // one arrival per dQ warp
    mbar_init(bar(BR::DSFREE), 1);
    mbar_init(bar(BR::ACC), 1);
    for (int i = 0; i < BSTAGES; ++i) {
      mbar_init(bar(BR::BFULL + i), 1);
      mbar_init(bar(BR::BEMPTY + i), 8);   // one arrival per softmax warp
    }
    for (int g = 0; g < 2; ++g) {          // dBias block of softmax group g
      mbar_init(bar(BR::DBFULL + g), 4);   // written: one arrival per warp of the group
      mbar_init(bar(BR::DBFREE + g), 1);   // read out by the previous store
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

  if (warp == 0) {
    // ================================================================ TMA producer
    const int bc = bcoord(p.m, b);                        // batch coordinate in the tensor maps
    if (lane == 0 && T > 0 &&
        FA_BOUNDS(sq.k_start + kv0 < rows_k(p.m) && hkv < p.Hkv && bc < batch_extent(p.m), wc, 60)) {
      mbar_arrive_expect_tx(bar(BR::KV), 2 * L::KV_BYTES);
#pragma unroll
      for (int hh = 0; hh < L::NH; ++hh) {
        tma_load_4d(sb + L::OFF_K + hh * L::KHALF, &tm_k, bar(BR::KV), 64 * hh, sq.k_start + kv0, hkv, bc);
        tma_load_4d(sb + L::OFF_V + hh * L::KHALF, &tm_v, bar(BR::KV), 64 * hh, sq.k_start + kv0, hkv, bc);
      }
      int issued = 0;
      for (int t = 0; t < T; ++t) {
        const int s = stg(t);
        const uint32_t ph = rph(t);
        if (t >= STAGES && !mbar_wait(bar(BR::QEMPTY + s), ph ^ 1, wc, 1)) break;
        const int h = hkv * G + t / per_head;
        const int q0 = (i0 + t % per_head) * BM;
        const int bh = b * p.Hq + h;                      // workspace rows are (b, h, padded q)
        if (!FA_BOUNDS(h < p.Hq && q0 < sq.nq && sq.q_start + q0 < rows_q(p.m) &&
                           static_cast<size_t>(bh) * p.NqPad + q0 + BM <= static_cast<size_t>(p.B) * p.Hq * p.NqPad,
                       wc, 61))
          break;
        if constexpr (BIAS)
          if (!FA_BOUNDS(kv0 < p.Nkv && (p.m.bias_st.n == 0 || q0 < p.Nq) && h < p.Hq && b < p.B, wc, 63)) break;
        const uint32_t fb = bar(BR::QFULL + s);
        mbar_arrive_expect_tx(fb, 2 * L::Q_BYTES + L::LD_BYTES);
#pragma unroll
        for (int hh = 0; hh < L::NH; ++hh) {
          tma_load_4d(sb + L::OFF_Q + s * L::Q_BYTES + hh * L::QHALF, &tm_q, fb, 64 * hh, sq.q_start + q0, h, bc);
          tma_load_4d(sb + L::OFF_DO + s * L::Q_BYTES + hh * L::QHALF, &tm_do, fb, 64 * hh, sq.q_start + q0, h,
                      bc);
        }
        const size_t row = static_cast<size_t>(bh) * p.NqPad + q0;
        bulk_load(sb + L::OFF_LD + s * L::LD_BYTES, p.nLg + row, BM * 4, fb);
        bulk_load(sb + L::OFF_LD + s * L::LD_BYTES + BM * 4, p.Dv + row, BM * 4, fb);
        if constexpr (BIAS) {
          // bias of (query rows q0.., keys kv0..) of head h, sequence b: a broadcast axis
          // has extent 1 in the map and is addressed at 0
          const int bs = t & (BSTAGES - 1);
          if (t >= BSTAGES && !mbar_wait(bar(BR::BEMPTY + bs), ((t / BSTAGES) & 1) ^ 1, wc, 17)) break;
          const uint32_t bb = bar(BR::BFULL + bs);
          mbar_arrive_expect_tx(bb, L::BIAS_BYTES);
          tma_load_4d(sb + L::OFF_BIAS + bs * L::BIAS_BYTES, &tm_bias, bb, kv0, p.m.bias_st.n ? q0 : 0,
                      p.m.bias_st.h ? h : 0, p.m.bias_st.b ? b : 0);
        }
        issued = t + 1;
      }
      // Never leave a copy in flight into shared memory this CTA is about to release.
      drain_wait(bar(BR::KV), 0);
      for (int t = max(0, issued - STAGES); t < issued; ++t)
        drain_wait(bar(BR::QFULL + stg(t)), rph(t));
      if constexpr (BIAS)
        for (int t = max(0, issued - BSTAGES); t < issued; ++t)
          drain_wait(bar(BR::BFULL + (t & (BSTAGES - 1))), (t / BSTAGES) & 1);
    }
  } else if (warp == 1 || warp == 2) {
    // ================================================================ MMA issuers
    // Two warps issue tcgen05.mma, each walking its loop with all 32 lanes
    // (elect.sync picks the issuing lane):
    //   warp 1: G1 (S^T) and G2 (dP^T), the products the softmax groups consume;
    //   warp 2: G3, G4, G5, the products of what the softmax groups produce.
    // Each blocks only on its own inputs, so dK/dQ of tile t are issued as soon
    // as dS^T(t) exists instead of queueing behind later tiles' S^T and dP^T.
    // Every hand-off between the two streams is an mbarrier: G1 into an S^T
    // buffer waits for the G3 that read the P^T there (s_free).
    if (T > 0) {
      constexpr uint32_t ID_S = make_idesc_f16(128, BM, BF16, false, false);
      constexpr uint32_t ID_KV = make_idesc_f16(128, D, BF16, false, true);   // A K-major (TMEM or smem), B MN-major
      constexpr uint32_t ID_Q = make_idesc_f16(128, BM, BF16, true, true);
      const uint32_t tdP = tmem + L::COL_DP;
      const uint32_t tdK = tmem + L::COL_DK, tdV = tmem + L::COL_DV, tdQ = tmem + L::COL_DQ;
      const uint32_t aK = sb + L::OFF_K, aV = sb + L::OFF_V;
      auto s_buf = [&](int t) -> uint32_t { return tmem + L::COL_S + (t & 1) * BM; };
      auto q_tile = [&](int t) -> uint32_t { return sb + L::OFF_Q + stg(t) * L::Q_BYTES; };
      auto do_tile = [&](int t) -> uint32_t { return sb + L::OFF_DO + stg(t) * L::Q_BYTES; };
      // Each operand tile's descriptor is built once and stepped by
      // compile-time offsets (the start address is the descriptor's low field,
      // so adding offset >> 4 advances it).
      const uint64_t dK_k = sw128_desc(aK, 16, 1024), dV_k = sw128_desc(aV, 16, 1024);
      const uint64_t dK_mn = sw128_desc(aK, L::KHALF, 1024);
      const uint64_t dS_mn = sw128_desc(sb + L::OFF_DS, L::DS_BYTES, 1024);
      const uint64_t dS_k = sw128_desc(sb + L::OFF_DS, 16, 1024);
      // K-major step ks (16 elements of d): 64-column half ks/4, 32 bytes per step inside it
      auto kstep = [](int ks, int half_bytes) -> uint64_t {
        return static_cast<uint64_t>(((ks >> 2) * half_bytes + (ks & 3) * 32) >> 4);
      };
      // MN-major step ks: 16 rows of 128 bytes
      auto mnstep = [](int ks) -> uint64_t { return static_cast<uint64_t>((ks * 2048) >> 4); };
      // 16-bit A operand column for query rows [16ks, 16ks+16): group ks/2, second half if ks odd
      auto a_col = [](int ks) -> uint32_t { return static_cast<uint32_t>(32 * (ks >> 1) + 8 * (ks & 1)); };
      auto wait = [&](uint32_t b, uint32_t parity, uint32_t site) -> bool {
        return __all_sync(0xffffffffu, mbar_wait(b, parity, wc, site));
      };

      if (warp == 1) {
        bool ok = wait(bar(BR::KV), 0, 2);
        for (int t = 0; ok && t < T; ++t) {
          // G1: S^T(t) = K Q^T  (contraction over d, 16 per instruction), into buffer t & 1
          if (!wait(bar(BR::QFULL + stg(t)), rph(t), 3)) break;
          if (t >= 2 && !wait(bar(BR::SFREE + (t & 1)), ((t - 2) >> 1) & 1, 15)) break;
          tc_fence_after();
          {
            const uint64_t dQ_k = sw128_desc(q_tile(t), 16, 1024);
            const uint32_t tS = s_buf(t);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              umma_ss_warp(tS, dK_k + kstep(ks, L::KHALF), dQ_k + kstep(ks, L::QHALF), ID_S, ks > 0);
            umma_commit_warp(bar(BR::S + (t & 1)));
          }
          // G2: dP^T(t) = V dO^T, once the softmax groups have loaded dP^T(t-1)
          if (t >= 1 && !wait(bar(BR::DPFREE), (t - 1) & 1, 14)) break;
          tc_fence_after();
          {
            const uint64_t dO_k = sw128_desc(do_tile(t), 16, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              umma_ss_warp(tdP, dV_k + kstep(ks, L::KHALF), dO_k + kstep(ks, L::QHALF), ID_S, ks > 0);
            umma_commit_warp(bar(BR::DP));
          }
        }
        // this warp's MMAs must have completed before TMEM is released
        umma_commit_warp(bar(BR::AFIN));
        drain_wait(bar(BR::AFIN), 0);
      } else {
        for (int t = 0; t < T; ++t) {
          // G3: dV += P^T dO  (P^T from TMEM; contraction over the BM query rows)
          if (!wait(bar(BR::P + (t & 1)), (t >> 1) & 1, 4)) break;
          tc_fence_after();
          {
            const uint32_t tS = s_buf(t);
            const uint64_t dO_mn = sw128_desc(do_tile(t), L::QHALF, 1024);
#pragma unroll
            for (int ks = 0; ks < BM / 16; ++ks)
              umma_ts_warp(tdV, tS + a_col(ks), dO_mn + mnstep(ks), ID_KV, (t > 0 || ks > 0));
            umma_commit_warp(bar(BR::SFREE + (t & 1)));
          }
          // G4: dK += dS^T Q  (dS^T from its smem tile, K-major; contraction over the query rows)
          if (!wait(bar(BR::DS), t & 1, 5)) break;
          tc_fence_after();
          {
            const uint64_t dQ_mn = sw128_desc(q_tile(t), L::QHALF, 1024);
#pragma unroll
            for (int ks = 0; ks < BM / 16; ++ks)
              umma_ss_warp(tdK, dS_k + static_cast<uint64_t>((ks * 32) >> 4), dQ_mn + mnstep(ks), ID_KV,
                           (t > 0 || ks > 0));
          }
          if constexpr (!DET) {
            // G5: dQ^T = K^T dS^T  (contraction over the BN key rows); M = 128 covers d
            // (for d = 64 the upper 64 lanes are unused)
            if (t > 0 && !wait(bar(BR::DQEMPTY), (t - 1) & 1, 6)) break;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks)
              umma_ss_warp(tdQ, dK_mn + mnstep(ks), dS_mn + mnstep(ks), ID_Q, ks > 0);
            umma_commit_warp(bar(BR::DQFULL));
          }
          umma_commit_warp(bar(BR::DSFREE));
          // stage of tile t: G1/G2(t) have completed (P(t), dS(t) depend on them), G3/G4(t) are tracked here
          umma_commit_warp(bar(BR::QEMPTY + stg(t)));
        }
        umma_commit_warp(bar(BR::ACC));
        if (*abort_flag) drain_wait(bar(BR::ACC), 0);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ================================================================ softmax / dS groups
    const int grp = (warp - 4) >> 2;                      // query columns [32 grp, 32 grp + 32)
    const int r = threadIdx.x - 128 - 128 * grp;          // KV row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tdP = tmem + lane_off + L::COL_DP + 32 * grp;
    const int kv = kv0 + r;
    const bool row_ok = kv < sq.nk;
    uint8_t* ds_row = smem + L::OFF_DS + r * 128;
    const uint64_t sc2 = f2_bits(p.scale_log2, p.scale_log2);
    int qi = i0;                                          // query tile of tile t (walked, no division)
    int h = hkv * G;                                      // and its query head
    const bool db_lead = (threadIdx.x & 127) == 0;        // issues this group's dBias stores
    int n_db = 0;                                         // dBias blocks this group has stored by TMA
    for (int t = 0; t < T; ++t, h += (qi + 1 == nQt), qi = (qi + 1 == nQt) ? i0 : qi + 1) {
      const int s = stg(t);
      const int q0 = qi * BM;
      const int qc = q0 + 32 * grp;                       // query of this group's column 0
      // bias of (query qc + c, key kv): from the tile the producer staged (row = query,
      // 256-byte rows of keys, so a warp reads 64 contiguous bytes per query), read
      // four columns at a time where they are used; queries past the sequence read 0
      const uint16_t* bcol = nullptr;
      int bstep = 0, bvalid = 0;
      if constexpr (BIAS) {
        const int bs = t & (BSTAGES - 1);
        if (!__all_sync(0xffffffffu, mbar_wait(bar(BR::BFULL + bs), (t / BSTAGES) & 1, wc, 16))) break;
        const bool qbc = p.m.bias_st.n == 0;
        bcol = reinterpret_cast<const uint16_t*>(smem + L::OFF_BIAS + bs * L::BIAS_BYTES) + r +
               (qbc ? 0 : 32 * grp * BN);
        bstep = qbc ? 0 : BN;
        bvalid = sq.nq - qc;
      }
      const float* Ls = reinterpret_cast<const float*>(smem + L::OFF_LD + s * L::LD_BYTES) + 32 * grp;
      const float* Ds = Ls + BM;
      const uint32_t tS = tmem + lane_off + L::COL_S + (t & 1) * BM + 32 * grp;
      // columns c < lim are masked: key kv lies after query q0 + 32 grp + c.
      // Only KV-tail rows and the diagonal tiles need the per-element test;
      // the decision is made once per warp.
      const int lim = p.causal ? (kv - sq.delta - q0 - 32 * grp) : INT_MIN;
      const bool need_mask = __any_sync(0xffffffffu, !row_ok || lim > 0);
      if (!__all_sync(0xffffffffu, mbar_wait(bar(BR::S + (t & 1)), (t >> 1) & 1, wc, 7))) break;
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
          float2 xa = f2_split(fma_f32x2(f2_bits(__uint_as_float(sr[4 * c4 + 0]), __uint_as_float(sr[4 * c4 + 1])), sc2, nl.x));
          float2 xb = f2_split(fma_f32x2(f2_bits(__uint_as_float(sr[4 * c4 + 2]), __uint_as_float(sr[4 * c4 + 3])), sc2, nl.y));
          if constexpr (BIAS) {
            float bv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) bv[e] = c + e < bvalid ? half_to_float<BF16>(bcol[(c + e) * bstep]) : 0.f;
            const uint64_t l2e = f2_bits(1.4426950408889634f, 1.4426950408889634f);
            xa = f2_split(fma_f32x2(f2_bits(bv[0], bv[1]), l2e, f2_bits(xa.x, xa.y)));
            xb = f2_split(fma_f32x2(f2_bits(bv[2], bv[3]), l2e, f2_bits(xb.x, xb.y)));
          }
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
      if constexpr (BIAS) {
        __syncwarp();                       // this warp's bias reads are done: release the tile
        if (lane == 0) mbar_arrive(bar(BR::BEMPTY + (t & (BSTAGES - 1))));
      }
      tmem_st_x16(tS, pk);                  // P^T, 16-bit, over the columns just read
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BR::P + (t & 1)));
      if (!__all_sync(0xffffffffu, mbar_wait(bar(BR::DP), t & 1, wc, 8))) break;
      tc_fence_after();
      uint32_t dk[16];
      {
        uint32_t dr[32];
        tmem_ld_x32(tdP, dr);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BR::DPFREE));   // dP^T buffer may now take the next tile's G2
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
      if constexpr (BIAS) {
        // dBias = dS (the bias enters S with weight 1), the 16-bit values G4 and G5 use.
        // The group's [32 query x 128 key] block goes through shared memory and one
        // TMA store (which clips at the tensor's extent).  In a packed batch the
        // extent is the longest sequence, so a block that crosses this sequence's
        // end is stored element by element instead (the caller's dBias outside
        // the sequence is never written).
        if (p.m.dbias != nullptr && qc < sq.nq) {
          const bool by_tma = p.m.cu_q == nullptr || (qc + 32 <= sq.nq && kv0 + BN <= sq.nk);
          if (by_tma) {
            uint8_t* half = smem + L::OFF_DB + grp * L::DB_HALF;
            if (n_db > 0) {
              if (db_lead) {
                bulk_wait_group_read<0>();                  // the previous block has been read out
                mbar_arrive(bar(BR::DBFREE + grp));
              }
              if (!__all_sync(0xffffffffu, mbar_wait(bar(BR::DBFREE + grp), (n_db - 1) & 1, wc, 18))) break;
            }
#pragma unroll
            for (int c = 0; c < 32; ++c)
              *reinterpret_cast<uint16_t*>(half + c * (BN * 2) + r * 2) = static_cast<uint16_t>(dk[c >> 1] >> (16 * (c & 1)));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BR::DBFULL + grp));
            if ((warp & 3) == 0) {                          // the group's first warp issues the store
              if (!__all_sync(0xffffffffu, mbar_wait(bar(BR::DBFULL + grp), n_db & 1, wc, 19))) break;
              if (lane == 0 && FA_BOUNDS(kv0 < p.Nkv && qc < p.Nq && h < p.Hq && b < p.B, wc, 66)) {
                tma_store_4d(&tm_dbias, smem_u32(half), kv0, qc, h, b);
                bulk_commit_group();
              }
            }
            ++n_db;
          } else if (row_ok) {
            uint16_t* dcol = static_cast<uint16_t*>(p.m.dbias) + bias_row(p.m.dbias_st, b, h, qc) + kv;
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (qc + c < sq.nq) dcol[c * p.m.dbias_st.n] = static_cast<uint16_t>(dk[c >> 1] >> (16 * (c & 1)));
          }
        }
      }
      {
        // dS^T row r into shared memory, the operand of G4 (K-major A) and G5
        // (MN-major B): 128 B per row (this group's 64 B are 16-byte chunks
        // 4 grp .. 4 grp + 3), chunk c stored at chunk position c ^ (r mod 8)
        // (the 128-byte swizzle).
        if (t > 0 && !__all_sync(0xffffffffu, mbar_wait(bar(BR::DSFREE), (t - 1) & 1, wc, 9))) break;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = 4 * grp + i;
          *reinterpret_cast<uint4*>(ds_row + ((c ^ (r & 7)) << 4)) =
              make_uint4(dk[4 * i], dk[4 * i + 1], dk[4 * i + 2], dk[4 * i + 3]);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BR::DS));
    }
    if constexpr (BIAS)
      if (db_lead && n_db > 0) bulk_wait_group<0>();      // stores complete before the CTA exits
  } else if (warp >= 12) {
    // ================================================================ dQ group
    if constexpr (!DET) {
      const int r = threadIdx.x - 384;                     // TMEM lane == column of dQ
      const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t tdQ = tmem + lane_off + L::COL_DQ;
      int h = hkv * G, qi = i0;                          // head and query tile of tile t
      for (int t = 0; t < T; ++t) {
        const int q0 = qi * BM;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(BR::DQFULL), t & 1, wc, 10))) break;
        tc_fence_after();
        uint32_t v0[32], v1[32];
        tmem_ld_x32(tdQ, v0);
        tmem_ld_x32(tdQ + 32, v1);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BR::DQEMPTY));
        // Thread r holds column r of the 64 x d tile: for each query row, the 32
        // lanes of a warp add one contiguous 128-byte segment of the accumulator.
        if (r < D && FA_BOUNDS(static_cast<size_t>(b * p.Hq + h) * p.NqPad + q0 + BM <=
                                   static_cast<size_t>(p.B) * p.Hq * p.NqPad,
                               wc, 64)) {
          float* dst = p.dq_acc + (static_cast<size_t>(b * p.Hq + h) * p.NqPad + q0) * D + r;
#pragma unroll
          for (int c = 0; c < 32; ++c) red_add_f32(dst + c * D, __uint_as_float(v0[c]));
#pragma unroll
          for (int c = 0; c < 32; ++c) red_add_f32(dst + (32 + c) * D, __uint_as_float(v1[c]));
        }
        if (++qi == nQt) {
          qi = i0;
          ++h;
        }
      }
    }
  }

  // ================================================================ epilogue: dK, dV
  if (warp >= 4 && warp < 12) {
    const bool is_dk = warp < 8;
    const int r = threadIdx.x - (is_dk ? 128 : 256);
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tacc = tmem + lane_off + (is_dk ? L::COL_DK : L::COL_DV);
    const int kv = kv0 + r;
    const float mul = is_dk ? p.scale : 1.0f;
    uint8_t* out = reinterpret_cast<uint8_t*>(is_dk ? p.dk : p.dv) +
                   at(is_dk ? p.m.st.dk : p.m.st.dv, p.m, b, hkv, sq.k_start + kv) * 2;
    bool have = T > 0;
    if (have) {
      have = __all_sync(0xffffffffu, mbar_wait(bar(BR::ACC), 0, wc, 13));
      tc_fence_after();
    }
    const bool aborted = *abort_flag != 0;
#pragma unroll 1
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t pk[16];
      if (have) {
        uint32_t v[32];
        tmem_ld_x32(tacc + ch * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pk[c] = pack2<BF16>(__uint_as_float(v[2 * c]) * mul, __uint_as_float(v[2 * c + 1]) * mul);
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = 0u;
      }
      if (kv < sq.nk && !aborted && FA_BOUNDS(sq.k_start + kv < rows_k(p.m), wc, 65))
        store_row_chunk<BF16>(out + ch * 64, pk, p.m.d - 32 * ch);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16, bool DET, bool BIAS>
cudaError_t launch_t(const MainArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                     const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tb, const CUtensorMap& tdb,
                     cudaStream_t stream) {
  using L = Layout<D, BIAS>;
  auto kern = bwd_main_kernel<D, BF16, DET, BIAS>;
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
  const long long nkt = (a.pb.Nkv + BN - 1) / BN;
  const long long grid = nkt * a.pb.B * a.pb.Hkv;
  kern<<<static_cast<unsigned>(grid), kThreads, L::ALLOC, stream>>>(tq, tdo, tk, tv, tb, tdb, p);
  return cudaGetLastError();
}

}  // namespace

// Problems without a bias run the persistent form of this kernel (bwd_main_persist.cu);
// this one serves the bias path, so only its BIAS = true instantiations are launched.
cudaError_t launch_bwd_main(const MainArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                            const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tb,
                            const CUtensorMap& tdb, cudaStream_t stream) {
  if (use_persistent(a.pb)) return launch_bwd_main_persist(a, tq, tdo, tk, tv, stream);
  const bool det = a.pb.deterministic != 0;
  if (a.pb.d > 64) {
    if (a.pb.bf16) return det ? launch_t<128, true, true, true>(a, tq, tdo, tk, tv, tb, tdb, stream)
                              : launch_t<128, true, false, true>(a, tq, tdo, tk, tv, tb, tdb, stream);
    return det ? launch_t<128, false, true, true>(a, tq, tdo, tk, tv, tb, tdb, stream)
               : launch_t<128, false, false, true>(a, tq, tdo, tk, tv, tb, tdb, stream);
  }
  if (a.pb.bf16) return det ? launch_t<64, true, true, true>(a, tq, tdo, tk, tv, tb, tdb, stream)
                            : launch_t<64, true, false, true>(a, tq, tdo, tk, tv, tb, tdb, stream);
  return det ? launch_t<64, false, true, true>(a, tq, tdo, tk, tv, tb, tdb, stream)
             : launch_t<64, false, false, true>(a, tq, tdo, tk, tv, tb, tdb, stream);
}

}  // namespace fa
