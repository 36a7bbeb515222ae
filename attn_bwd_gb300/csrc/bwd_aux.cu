// bwd_aux.cu -- the HBM-bound kernels around the backward's main kernel.
//
// preprocess: D_i = sum_c dO_ic O_ic per query row in fp32 (the row-wise dot
//   product of flash_attention_backward.cu, rustytorch rtx-flash-attention,
//   block "Compute row-wise dot product: dO * O"; the D / delta input of the
//   Triton kernel in triton #1806), computed once per row instead of once per
//   CTA.  Fused with it: -L*log2(e) per row (the main kernel evaluates
//   exp(S - L) as exp2(S*scale*log2e + (-L*log2e)), one fused multiply-add),
//   -inf / 0 on the padding rows
//   so that padded query rows contribute exactly zero, and the zeroing of the
//   fp32 dQ accumulator (triton #1806 allocates it zero-filled).
// convert: dQ = scale * accumulator, rounded once to the 16-bit dtype.
// Both stream contiguous rows with 16-byte loads and stores; grids are sized
// in multiples of the SM count and walk the rows with a grid stride.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "kernels.h"
#include "ptx.cuh"
#include "seq.cuh"

namespace fa {
namespace {

template <bool BF16>
__device__ __forceinline__ void widen8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = unpack2<BF16>(w[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// One query row is handled by D/8 consecutive lanes (16 bytes of O and of dO each).
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
preprocess_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dO, const float* __restrict__ lse,
                  float* __restrict__ nLg, float* __restrict__ Dv, float4* __restrict__ dq_acc,
                  long long rows, int NqPad, SeqMap m, unsigned int* status, unsigned int* call_abort) {
  constexpr int TPR = D / 8;                 // lanes per row
  constexpr int RPB = 256 / TPR;             // rows per block per sweep
  const int sub = threadIdx.x % TPR;
  // the later kernels of this call start with a clear abort word (word 0 of the workspace
  // header) and item counters (words 1, 2: the persistent main kernel's; 3, 4: the
  // persistent deterministic dQ kernel's)
  if (blockIdx.x == 0 && threadIdx.x < 5) call_abort[threadIdx.x] = 0u;
  // The sweep base is block-uniform so every lane reaches the row shuffle below.
  for (long long base = static_cast<long long>(blockIdx.x) * RPB; base < rows;
       base += static_cast<long long>(gridDim.x) * RPB) {
    const long long row = base + threadIdx.x / TPR;
    const bool valid = row < rows;
    const long long bh = row / NqPad;
    const int r = static_cast<int>(row - bh * NqPad);
    const int b = static_cast<int>(bh / m.Hq);
    const int h = static_cast<int>(bh - static_cast<long long>(b) * m.Hq);
    const Seq sq = valid ? seq_of(m, b, status, 30) : Seq{0, 0, 0, 0, 0};
    const bool live = valid && r < sq.nq;
    const long long qrow = sq.q_start + r;
    float acc = 0.f;
    if (live && 8 * sub < m.d && FA_BOUNDS_S(qrow < rows_q(m), status, 90)) {
      float a[8], g[8];
      widen8<BF16>(__ldg(o + at(m.st.o, m, b, h, qrow) / 8 + sub), a);
      widen8<BF16>(__ldg(dO + at(m.st.dO, m, b, h, qrow) / 8 + sub), g);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(a[i], g[i], acc);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, TPR);
    if (!valid) continue;
    if (sub == 0) {
      Dv[row] = acc;
      // -L * log2(e); -inf on padding rows and on rows that see no key (L = -inf), so
      // that every exponent of such a row is -inf whatever the scores and bias are
      const float L = live ? lse[at(m.st.lse, m, b, h, qrow)] : -CUDART_INF_F;
      nLg[row] = L == -CUDART_INF_F ? -CUDART_INF_F : -L * 1.4426950408889634f;
    }
    if (dq_acc != nullptr) {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      dq_acc[row * (D / 4) + 2 * sub] = z;
      dq_acc[row * (D / 4) + 2 * sub + 1] = z;
    }
  }
}

// Each thread converts 8 consecutive fp32 of one accumulator row to 16-bit;
// accumulator rows are (b, h, padded q), and only rows of real queries are written.
template <int D, bool BF16>
__global__ void __launch_bounds__(256)
dq_convert_kernel(const float4* __restrict__ acc, uint4* __restrict__ dq, long long n8, int NqPad, float scale,
                  SeqMap m, unsigned int* status) {
  constexpr int C8 = D / 8;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n8;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = idx / C8;            // accumulator row: bh * NqPad + r
    const int c8 = static_cast<int>(idx - row * C8);
    const long long bh = row / NqPad;
    const int r = static_cast<int>(row - bh * NqPad);
    const int b = static_cast<int>(bh / m.Hq);
    const int h = static_cast<int>(bh - static_cast<long long>(b) * m.Hq);
    const Seq sq = seq_of(m, b, status, 31);
    if (r >= sq.nq || 8 * c8 >= m.d || !FA_BOUNDS_S(sq.q_start + r < rows_q(m), status, 91)) continue;
    const long long src = (row * D) / 4 + 2 * c8;
    const float4 a = __ldcs(acc + src);
    const float4 c = __ldcs(acc + src + 1);
    uint4 out;
    out.x = pack2<BF16>(a.x * scale, a.y * scale);
    out.y = pack2<BF16>(a.z * scale, a.w * scale);
    out.z = pack2<BF16>(c.x * scale, c.y * scale);
    out.w = pack2<BF16>(c.z * scale, c.w * scale);
    dq[at(m.st.dq, m, b, h, sq.q_start + r) / 8 + c8] = out;
  }
}

// Waits on a barrier nobody arrives on, bounded by timeout_ns; records the
// timeout in the status word and exits.
__global__ void wait_selftest_kernel(unsigned int* status, long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
      if (mbar_try_wait(b, 0)) break;  // never completes: nothing arrives
      if (globaltimer_ns() - t0 > static_cast<uint64_t>(timeout_ns)) {
        atomicCAS(status, 0u, (kStatusTimeout << 16) | 99u);
        break;
      }
    }
  }
  __syncthreads();
}

// dBias of a causal problem: the main kernel visits, for KV tile j, only the
// query tiles from i0(j) = max(0, j*BN - delta) / BM on and writes dS there;
// every key of the tiles it skips is masked for those queries, so dBias is 0.
// Query row q (tile qt = q / BM) is skipped exactly for the KV tiles j with
// i0(j) > qt, i.e. j*BN >= (qt + 1)*BM + delta: keys from
// jmin*BN = ceil(((qt + 1)*BM + delta) / BN) * BN to the end of the row.
// One warp per row, 16 bytes per lane and store.
template <bool BF16>
__global__ void __launch_bounds__(256)
dbias_zero_kernel(SeqMap m, long long rows, unsigned int* status) {
  const int lane = threadIdx.x & 31;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < rows;
       row += nwarps) {
    const long long bh = row / m.Nq;                       // rows are (b, h, q) with q < Nq (the longest)
    const int q = static_cast<int>(row - bh * m.Nq);
    const int b = static_cast<int>(bh / m.Hq);
    const int h = static_cast<int>(bh - static_cast<long long>(b) * m.Hq);
    const Seq sq = seq_of(m, b, status, 32);
    if (q >= sq.nq || !FA_BOUNDS_S(q < m.Nq && h < m.Hq && b < m.B, status, 92)) continue;
    const long long first = static_cast<long long>(q / kMainBM + 1) * kMainBM + sq.delta;
    const long long k0 = (first <= 0 ? 0 : (first + kMainBN - 1) / kMainBN) * kMainBN;
    uint16_t* dst = static_cast<uint16_t*>(m.dbias) + bias_row(m.dbias_st, b, h, q);
    for (long long kv = k0 + 8 * lane; kv < sq.nk; kv += 256) {
      if (kv + 8 <= sq.nk) {
        *reinterpret_cast<uint4*>(dst + kv) = make_uint4(0u, 0u, 0u, 0u);
      } else {
        for (long long e = kv; e < sq.nk; ++e) dst[e] = 0;
      }
    }
  }
}

// Grid of a grid-stride kernel: enough blocks for the work, at most 16 per SM.
long long grid_for(long long work_items, int per_block) {
  long long g = (work_items + per_block - 1) / per_block;
  const long long cap = static_cast<long long>(sm_count()) * 16;
  if (g > cap) g = cap;
  return g < 1 ? 1 : g;
}

template <int D, bool BF16>
cudaError_t pre_t(const Problem& pb, const void* o, const void* dO, const float* lse, const Workspace& ws,
                  unsigned int* status, cudaStream_t stream) {
  const long long rows = static_cast<long long>(pb.B) * pb.Hq * pb.NqPad;
  const long long grid = grid_for(rows, 256 / (D / 8));
  preprocess_kernel<D, BF16><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      static_cast<const uint4*>(o), static_cast<const uint4*>(dO), lse, ws.nLg, ws.Dv,
      pb.deterministic ? nullptr : reinterpret_cast<float4*>(ws.dq_acc), rows, pb.NqPad, seq_map(pb), status,
      ws.abort);
  return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t conv_t(const Problem& pb, const Workspace& ws, void* dq, unsigned int* status, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(pb.B) * pb.Hq * pb.NqPad * (D / 8);
  const long long grid = grid_for(n8, 256);
  dq_convert_kernel<D, BF16><<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(ws.dq_acc), static_cast<uint4*>(dq), n8, pb.NqPad, pb.scale, seq_map(pb),
      status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_preprocess(const Problem& pb, const void* o, const void* dO, const float* lse,
                              const Workspace& ws, unsigned int* status, cudaStream_t stream) {
  if (pb.d > 64)
    return pb.bf16 ? pre_t<128, true>(pb, o, dO, lse, ws, status, stream)
                   : pre_t<128, false>(pb, o, dO, lse, ws, status, stream);
  return pb.bf16 ? pre_t<64, true>(pb, o, dO, lse, ws, status, stream)
                 : pre_t<64, false>(pb, o, dO, lse, ws, status, stream);
}

cudaError_t launch_dq_convert(const Problem& pb, const Workspace& ws, void* dq, unsigned int* status,
                              cudaStream_t stream) {
  if (pb.d > 64)
    return pb.bf16 ? conv_t<128, true>(pb, ws, dq, status, stream) : conv_t<128, false>(pb, ws, dq, status, stream);
  return pb.bf16 ? conv_t<64, true>(pb, ws, dq, status, stream) : conv_t<64, false>(pb, ws, dq, status, stream);
}

cudaError_t launch_dbias_zero(const Problem& pb, unsigned int* status, cudaStream_t stream) {
  const long long rows = static_cast<long long>(pb.B) * pb.Hq * pb.Nq;
  const long long grid = grid_for(rows, 8);                 // 8 rows (warps) per block
  if (pb.bf16)
    dbias_zero_kernel<true><<<static_cast<unsigned>(grid), 256, 0, stream>>>(seq_map(pb), rows, status);
  else
    dbias_zero_kernel<false><<<static_cast<unsigned>(grid), 256, 0, stream>>>(seq_map(pb), rows, status);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(unsigned int* status, long long timeout_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fa
