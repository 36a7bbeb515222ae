// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Rows of every per-head query array in the workspace are padded to this.
constexpr int kRowPad = 128;

// Tile of the main backward kernel: KV rows per CTA and query rows per step.
// The dBias zeroing kernel reproduces which (query tile, KV tile) pairs it skips.
constexpr int kMainBN = 128;
constexpr int kMainBM = 64;

// Keys per step of the forward kernel: the box height of its K and V tensor maps.
constexpr int kFwdBK = 64;        // no bias
constexpr int kFwdBKBias = 128;   // with an additive bias

inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// SM count of the current device (1 if it cannot be read).
inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    return 1;
  return n;
}

// Workspace carve-up shared by every stage of the backward.
struct Workspace {
  unsigned int* abort;   // the call's abort word (first 256 bytes): zeroed by the preprocess
                         // kernel, set by the first CTA of the main or dQ kernel that gives up;
                         // words 1, 2 are the persistent main kernel's item counters, words 3, 4
                         // the persistent deterministic dQ kernel's
  float* nLg;     // [B*Hq*NqPad]   -L * log2(e); -inf on padding rows
  float* Dv;      // [B*Hq*NqPad]   rowsum(dO o O); 0 on padding rows
  float* dq_acc;  // [B*Hq*NqPad*d] fp32 dQ accumulator (atomic mode only)
};

// Element strides of a tensor's batch, head and row axes (its d axis is contiguous).
struct Str3 {
  long long b, h, n;
};

// Strides of every tensor of a problem.
struct Strides {
  Str3 q, k, v, o, dO, dq, dk, dv, lse;
};

// Geometry of the batch, passed to every kernel (see seq.cuh).
struct SeqMap {
  const int* cu_q;   // packed batch: [B + 1] query offsets (device); nullptr for a dense batch
  const int* cu_k;   // packed batch: [B + 1] key offsets (device)
  int B, Hq, Hkv;
  int d;             // head dimension of the tensors (<= the kernel's D; missing columns read as 0)
  int Nq, Nkv;       // dense: the lengths; packed: the longest lengths
  int total_q, total_k;  // packed: rows per head
  int causal_mode;   // 0 none, 1 top-left, 2 bottom-right
  Strides st;
  // Additive bias [B, Hq, Nq, Nkv] in the 16-bit dtype (key axis contiguous,
  // indices local to the sequence) and its gradient, or nullptr.
  const void* bias;
  Str3 bias_st;      // element strides of the batch, head and query axes (0 broadcasts)
  void* dbias;
  Str3 dbias_st;
};

struct Problem {
  int B, Hq, Hkv, Nq, Nkv, d;   // packed batch: Nq, Nkv are the longest lengths
  int NqPad;
  float scale;
  int causal;        // any causal mask (causal_mode != 0)
  int causal_mode;   // 0 none, 1 top-left, 2 bottom-right
  int bf16;
  int deterministic;
  const int* cu_q;   // packed batch offsets, or nullptr
  const int* cu_k;
  int total_q, total_k;
  Strides st;
  const void* bias;
  Str3 bias_st;
  void* dbias;
  Str3 dbias_st;
};

inline SeqMap seq_map(const Problem& pb) {
  SeqMap m;
  m.cu_q = pb.cu_q;
  m.cu_k = pb.cu_k;
  m.B = pb.B; m.Hq = pb.Hq; m.Hkv = pb.Hkv;
  m.d = pb.d;
  m.Nq = pb.Nq; m.Nkv = pb.Nkv;
  m.total_q = pb.total_q; m.total_k = pb.total_k;
  m.causal_mode = pb.causal_mode;
  m.st = pb.st;
  m.bias = pb.bias;
  m.bias_st = pb.bias_st;
  m.dbias = pb.dbias;
  m.dbias_st = pb.dbias_st;
  return m;
}

struct MainArgs {
  Problem pb;
  Workspace ws;
  void* dk;
  void* dv;
  unsigned int* status;
};

struct DqArgs {
  Problem pb;
  Workspace ws;
  void* dq;
  unsigned int* status;
};

struct FwdArgs {
  Problem pb;
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
};

// bwd_aux.cu
cudaError_t launch_preprocess(const Problem& pb, const void* o, const void* dO, const float* lse,
                              const Workspace& ws, unsigned int* status, cudaStream_t stream);
cudaError_t launch_dq_convert(const Problem& pb, const Workspace& ws, void* dq, unsigned int* status,
                              cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned int* status, long long timeout_ns, cudaStream_t stream);
// Writes dBias = 0 where the main kernel, under causal tile skipping, never visits.
cudaError_t launch_dbias_zero(const Problem& pb, unsigned int* status, cudaStream_t stream);

// bwd_main.cu: maps are Q, dO (box 64 x 64 rows), K, V (box 64 x 128 rows), the bias
// (box 128 keys x 64 queries) and dBias (box 128 keys x 32 queries); the last two are
// used only when the problem has a bias (and a dBias)
cudaError_t launch_bwd_main(const MainArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                            const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tb,
                            const CUtensorMap& tdb, cudaStream_t stream);

// bwd_main_persist.cu: the same products as a persistent kernel (one CTA per SM walking
// the work items back to back), which launch_bwd_main uses for every problem without an
// additive bias; maps as for bwd_main.cu
inline bool use_persistent(const Problem& pb) { return pb.bias == nullptr; }
cudaError_t launch_bwd_main_persist(const MainArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                                    const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream);

// bwd_dq.cu: maps are Q, dO (box 64 x 128 rows), K, V (box 64 x 128 rows)
// bwd_dq_persist.cu: the deterministic dQ pass as a persistent kernel (problems without a bias;
// launch_bwd_dq_det dispatches to it)
cudaError_t launch_bwd_dq_persist(const DqArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                                  const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream);
cudaError_t launch_bwd_dq_det(const DqArgs& a, const CUtensorMap& tq, const CUtensorMap& tdo,
                              const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream);

// fwd.cu: maps are Q (box 64 x 128 rows), K, V (box 64 x kFwdBK rows, or kFwdBKBias with a
// bias) and the bias (box 64 keys x 128 queries, 128-byte swizzle; used only when the
// problem has a bias)
// `call_abort` is the call's abort word (a slot of a ring) and `call_tag` the value the
// call stores there when it gives up; no earlier user of the slot had that tag.
cudaError_t launch_fwd(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tb, unsigned int* status, unsigned int* call_abort,
                       unsigned int call_tag, cudaStream_t stream);
// fwd_persist.cu: the forward as a persistent kernel (problems without a bias; launch_fwd
// dispatches to it)
cudaError_t launch_fwd_persist(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               unsigned int* status, unsigned int* call_abort, unsigned int call_tag,
                               cudaStream_t stream);

}  // namespace fa
