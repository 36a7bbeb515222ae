// seq.cuh -- where sequence b of a batch lives, for dense and packed batches.
//
// Dense batch:  Q-like tensors [B, Hq, Nq, d], K-like [B, Hkv, Nkv, d] (any
//               strides); every sequence has Nq queries and Nkv keys.
// Packed batch: Q-like tensors [Hq, total_q, d], K-like [Hkv, total_k, d];
//               sequence b owns rows [cu_q[b], cu_q[b+1]) of every query head
//               and [cu_k[b], cu_k[b+1]) of every key/value head, and attends
//               only within itself.  Nq / Nkv then hold the longest lengths,
//               which size the grids and the padded workspace rows.
// Every tensor is addressed through its own element strides for the batch,
// head and row axes (the d axis is contiguous), and through a 4-D tensor map
// (d, rows, heads, batch) built on the same strides.  A packed batch has a
// batch extent of 1; its sequence b starts at row cu[b] of every head.
#pragma once

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace fa {

struct Seq {
  int nq, nk;            // queries and keys of this sequence
  int q_start, k_start;  // first row of the sequence along its head's row axis
  int delta;             // causal: key j masked for query i when j > i + delta
};

// Status code for a packed-batch offset array that is out of range.
constexpr unsigned kStatusBadSeq = 10u;   // FA_ERR_ARG

// Reads and checks the offsets of sequence b.  An offset pair outside
// [0, total] or a length above the maximum is reported in the status word
// and the sequence is treated as empty (nothing is read or written for it).
__device__ __forceinline__ Seq seq_of(const SeqMap& m, int b, unsigned int* status, unsigned site) {
  Seq s;
  if (m.cu_q == nullptr) {
    s.nq = m.Nq;
    s.nk = m.Nkv;
    s.q_start = 0;
    s.k_start = 0;
  } else {
    const int q0 = __ldg(m.cu_q + b), q1 = __ldg(m.cu_q + b + 1);
    const int k0 = __ldg(m.cu_k + b), k1 = __ldg(m.cu_k + b + 1);
    const bool ok = q0 >= 0 && q0 <= q1 && q1 <= m.total_q && q1 - q0 <= m.Nq &&
                    k0 >= 0 && k0 <= k1 && k1 <= m.total_k && k1 - k0 <= m.Nkv;
    if (!ok) {
      atomicCAS(status, 0u, (kStatusBadSeq << 16) | site);
      s.nq = s.nk = s.q_start = s.k_start = 0;
    } else {
      s.nq = q1 - q0;
      s.nk = k1 - k0;
      s.q_start = q0;
      s.k_start = k0;
    }
  }
  s.delta = m.causal_mode == 2 ? s.nk - s.nq : 0;
  return s;
}

// Batch coordinate of sequence b in tensor maps and addresses (a packed batch
// has one: its sequences are told apart by their rows).
__device__ __forceinline__ int bcoord(const SeqMap& m, int b) { return m.cu_q ? 0 : b; }

// Extents of the tensors (those of their tensor maps): rows along each head's row
// axis of the Q-like and K-like tensors, and the batch extent.
__device__ __forceinline__ int rows_q(const SeqMap& m) { return m.cu_q ? m.total_q : m.Nq; }
__device__ __forceinline__ int rows_k(const SeqMap& m) { return m.cu_q ? m.total_k : m.Nkv; }
__device__ __forceinline__ int batch_extent(const SeqMap& m) { return m.cu_q ? 1 : m.B; }

// Element offset of row `row` of head h of sequence b in a tensor with strides s
// (row already includes the sequence's first row).
__device__ __forceinline__ long long at(const Str3& s, const SeqMap& m, int b, int h, long long row) {
  return static_cast<long long>(bcoord(m, b)) * s.b + static_cast<long long>(h) * s.h + row * s.n;
}

// Element offset of query row q (local to its sequence) of head h of sequence b
// in the bias or dBias tensor with strides s (the key index is added by the caller).
__device__ __forceinline__ long long bias_row(const Str3& s, int b, int h, int q) {
  return static_cast<long long>(b) * s.b + static_cast<long long>(h) * s.h + static_cast<long long>(q) * s.n;
}

template <bool BF16>
__device__ __forceinline__ float half_to_float(uint16_t u) {
  if constexpr (BF16) return __uint_as_float(static_cast<uint32_t>(u) << 16);
  else return __half2float(__ushort_as_half(u));
}

// Bias of keys col .. col + 7 of one row (16-byte aligned when col is a multiple
// of 8); keys at or past nk read as 0 without touching memory.
template <bool BF16>
__device__ __forceinline__ void bias8(const uint16_t* row, int col, int nk, float (&v)[8]) {
  if (col + 8 <= nk) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(row + col));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack2<BF16>(w[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = col + e < nk ? half_to_float<BF16>(__ldg(row + col + e)) : 0.f;
  }
}

}  // namespace fa
