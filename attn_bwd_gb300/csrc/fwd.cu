// fwd.cu -- exact attention forward producing O and the log-sum-exp L that
// the backward consumes (L is the natural-log LSE of the scaled, masked
// scores, the convention of flash_attention_backward.cu, rustytorch
// rtx-flash-attention, block "Compute softmax probabilities from scores and
// LSE").  This is a plain fp32 CUDA-core kernel with the usual running-max
// ("online") softmax over 64-row KV tiles; it exists to make inputs for the
// backward and is deliberately independent of the tensor-core machinery the
// backward uses.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "kernels.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int TQ = 64;     // query rows per CTA
constexpr int TK = 64;     // key rows per step
constexpr int kThreads = 256;

template <int D>
struct Smem {
  static constexpr int QS = D + 4;   // row strides (floats) chosen to spread banks
  static constexpr int KS = D + 1;
  static constexpr int SS = TK + 1;
  static constexpr int BYTES = 4 * (TQ * QS + TK * KS + TK * D + TQ * SS + 3 * TQ);
};

struct Params {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, Hq, Hkv, Nq, Nkv;
  float scale;
  int causal;
};

template <bool BF16>
__device__ __forceinline__ void load8(const void* base, long long elem, float* dst) {
  const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = unpack2<BF16>(w[i]);
    dst[2 * i] = f.x;
    dst[2 * i + 1] = f.y;
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kThreads)
fwd_kernel(const Params p) {
  using S = Smem<D>;
  extern __shared__ float sm[];
  float* Qs = sm;
  float* Ks = Qs + TQ * S::QS;
  float* Vs = Ks + TK * S::KS;
  float* Ss = Vs + TK * D;
  float* row_m = Ss + TQ * S::SS;
  float* row_l = row_m + TQ;
  float* row_a = row_l + TQ;

  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;
  const int q0 = blockIdx.x * TQ;
  const int h = blockIdx.y, b = blockIdx.z;
  const int hk = h / (p.Hq / p.Hkv);
  const long long qbase = (static_cast<long long>(b) * p.Hq + h) * p.Nq;
  const long long kbase = (static_cast<long long>(b) * p.Hkv + hk) * p.Nkv;

  for (int c = tid; c < TQ * D / 8; c += kThreads) {
    const int r = c / (D / 8), col = (c % (D / 8)) * 8;
    float tmp[8];
    if (q0 + r < p.Nq) load8<BF16>(p.q, (qbase + q0 + r) * D + col, tmp);
    else for (int i = 0; i < 8; ++i) tmp[i] = 0.f;
    for (int i = 0; i < 8; ++i) Qs[r * S::QS + col + i] = tmp[i];
  }
  if (tid < TQ) {
    row_m[tid] = -CUDART_INF_F;
    row_l[tid] = 0.f;
  }
  constexpr int OC = D / 16;
  float acc[4][OC];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < OC; ++c) acc[i][c] = 0.f;

  const int qlast = min(q0 + TQ, p.Nq) - 1;
  const int kv_end = p.causal ? min(p.Nkv, qlast + 1) : p.Nkv;
  for (int kv0 = 0; kv0 < kv_end; kv0 += TK) {
    __syncthreads();
    for (int c = tid; c < TK * D / 8; c += kThreads) {
      const int r = c / (D / 8), col = (c % (D / 8)) * 8;
      float kt[8], vt[8];
      if (kv0 + r < p.Nkv) {
        load8<BF16>(p.k, (kbase + kv0 + r) * D + col, kt);
        load8<BF16>(p.v, (kbase + kv0 + r) * D + col, vt);
      } else {
        for (int i = 0; i < 8; ++i) kt[i] = vt[i] = 0.f;
      }
      for (int i = 0; i < 8; ++i) {
        Ks[r * S::KS + col + i] = kt[i];
        Vs[r * D + col + i] = vt[i];
      }
    }
    __syncthreads();
    // scores: rows 4ty..4ty+3, columns tx + 16 jj
    float s[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) s[i][jj] = 0.f;
    for (int d = 0; d < D; ++d) {
      float kk[4];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) kk[jj] = Ks[(tx + 16 * jj) * S::KS + d];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float qv = Qs[(4 * ty + i) * S::QS + d];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) s[i][jj] = fmaf(qv, kk[jj], s[i][jj]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qi = q0 + 4 * ty + i;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int kj = kv0 + tx + 16 * jj;
        const bool masked = kj >= p.Nkv || (p.causal && kj > qi);
        Ss[(4 * ty + i) * S::SS + tx + 16 * jj] = masked ? -CUDART_INF_F : s[i][jj] * p.scale;
      }
    }
    __syncthreads();
    // running max / sum: 4 threads per row, 16 columns each
    {
      const int r = tid / 4, part = tid % 4;
      float* srow = Ss + r * S::SS + part * 16;
      float mx = -CUDART_INF_F;
      for (int c = 0; c < 16; ++c) mx = fmaxf(mx, srow[c]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_old = row_m[r];
      const float m_new = fmaxf(m_old, mx);
      float sum = 0.f;
      for (int c = 0; c < 16; ++c) {
        const float e = (m_new == -CUDART_INF_F) ? 0.f : expf(srow[c] - m_new);
        srow[c] = e;
        sum += e;
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      sum += __shfl_xor_sync(0xffffffffu, sum, 2);
      __syncwarp();
      if (part == 0) {
        const float alpha = (m_new == -CUDART_INF_F) ? 1.f : expf(m_old - m_new);
        row_a[r] = alpha;
        row_l[r] = row_l[r] * alpha + sum;
        row_m[r] = m_new;
      }
    }
    __syncthreads();
    // O = O * alpha + P V ; this thread: rows 4ty+i, columns tx + 16c
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float a = row_a[4 * ty + i];
#pragma unroll
      for (int c = 0; c < OC; ++c) acc[i][c] *= a;
    }
    for (int kk = 0; kk < TK; ++kk) {
      float pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pv[i] = Ss[(4 * ty + i) * S::SS + kk];
#pragma unroll
      for (int c = 0; c < OC; ++c) {
        const float vv = Vs[kk * D + tx + 16 * c];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][c] = fmaf(pv[i], vv, acc[i][c]);
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * ty + i;
    if (q0 + r >= p.Nq) continue;
    const float inv = 1.f / row_l[r];
    uint16_t* orow = static_cast<uint16_t*>(p.o) + (qbase + q0 + r) * D;
#pragma unroll
    for (int c = 0; c < OC; ++c) {
      const float val = acc[i][c] * inv;
      uint16_t bits;
      if constexpr (BF16) {
        const __nv_bfloat16 t = __float2bfloat16_rn(val);
        bits = *reinterpret_cast<const uint16_t*>(&t);
      } else {
        const __half t = __float2half_rn(val);
        bits = *reinterpret_cast<const uint16_t*>(&t);
      }
      orow[tx + 16 * c] = bits;
    }
  }
  if (tid < TQ && q0 + tid < p.Nq) p.lse[qbase + q0 + tid] = row_m[tid] + logf(row_l[tid]);
}

template <int D, bool BF16>
cudaError_t launch_t(const FwdArgs& a, cudaStream_t stream) {
  using S = Smem<D>;
  auto kern = fwd_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
  if (e != cudaSuccess) return e;
  Params p{a.q, a.k, a.v, a.o, a.lse, a.pb.B, a.pb.Hq, a.pb.Hkv, a.pb.Nq, a.pb.Nkv, a.pb.scale, a.pb.causal};
  dim3 grid((a.pb.Nq + TQ - 1) / TQ, a.pb.Hq, a.pb.B);
  kern<<<grid, kThreads, S::BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.pb.d == 128) return a.pb.bf16 ? launch_t<128, true>(a, stream) : launch_t<128, false>(a, stream);
  return a.pb.bf16 ? launch_t<64, true>(a, stream) : launch_t<64, false>(a, stream);
}

}  // namespace fa
