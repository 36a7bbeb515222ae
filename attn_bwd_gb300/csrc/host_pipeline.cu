// host_pipeline.cu -- fa_bwd_host: the backward for tensors that live in host
// memory, with the transfers overlapped with the computation.
//
// The (batch) sequences of a dense problem are independent, so the batch is
// cut into chunks of chunk_b sequences that flow through two device staging
// slots: while chunk c computes on the caller's stream, chunk c + 1 is copied
// in on one internal stream and chunk c - 1 is copied out on another.  Events
// order the three: a chunk computes once its inputs are in, its outputs are
// copied out once it has computed, and a slot is refilled once its outputs are
// out.  The caller owns the staging memory (fa_bwd_host_staging_size); the
// only state kept here is the two copy streams per device, created on first
// use.  Every copy is one cudaMemcpyAsync of a contiguous chunk.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace {

constexpr int kMaxDevices = 64;
struct CopyStreams {
  cudaStream_t in = nullptr;
  cudaStream_t out = nullptr;
};
CopyStreams g_copy[kMaxDevices];
std::mutex g_copy_mu;

int copy_streams(CopyStreams* cs) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_copy_mu);
  CopyStreams& c = g_copy[dev];
  if (c.in == nullptr) {
    if (cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking) != cudaSuccess) return FA_ERR_CUDA;
  }
  *cs = c;
  return FA_OK;
}

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Byte offsets of one staging slot holding a chunk of cb sequences.
struct Slot {
  size_t q, o, dO, dq, k, v, dk, dv, lse, ws, bytes;
  size_t q_bytes, k_bytes, lse_bytes, ws_bytes;
};

Slot slot_layout(int cb, int Hq, int Hkv, int Nq, int Nkv, int d, int deterministic) {
  Slot s;
  s.q_bytes = static_cast<size_t>(cb) * Hq * Nq * d * 2;
  s.k_bytes = static_cast<size_t>(cb) * Hkv * Nkv * d * 2;
  s.lse_bytes = static_cast<size_t>(cb) * Hq * Nq * 4;
  s.ws_bytes = fa_bwd_workspace_size(cb, Hq, Hkv, Nq, Nkv, d, deterministic);
  size_t off = 0;
  s.q = off; off += up(s.q_bytes);
  s.o = off; off += up(s.q_bytes);
  s.dO = off; off += up(s.q_bytes);
  s.dq = off; off += up(s.q_bytes);
  s.k = off; off += up(s.k_bytes);
  s.v = off; off += up(s.k_bytes);
  s.dk = off; off += up(s.k_bytes);
  s.dv = off; off += up(s.k_bytes);
  s.lse = off; off += up(s.lse_bytes);
  s.ws = off; off += up(s.ws_bytes);
  s.bytes = off;
  return s;
}

int slots_for(int B, int chunk_b) { return (B + chunk_b - 1) / chunk_b > 1 ? 2 : 1; }

struct Events {
  cudaEvent_t e[7] = {};
  ~Events() {
    for (cudaEvent_t x : e)
      if (x) cudaEventDestroy(x);   // released once the work that records it has completed
  }
  int create() {
    for (cudaEvent_t& x : e)
      if (cudaEventCreateWithFlags(&x, cudaEventDisableTiming) != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
  }
};

const uint8_t* at(const void* p, size_t off) { return static_cast<const uint8_t*>(p) + off; }
uint8_t* at(void* p, size_t off) { return static_cast<uint8_t*>(p) + off; }

}  // namespace

extern "C" {

size_t fa_bwd_host_staging_size(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int deterministic, int chunk_b) {
  if (chunk_b < 1 || chunk_b > B) return 0;
  if (fa_bwd_workspace_size(chunk_b, Hq, Hkv, Nq, Nkv, d, deterministic) == 0) return 0;
  return slots_for(B, chunk_b) * slot_layout(chunk_b, Hq, Hkv, Nq, Nkv, d, deterministic).bytes;
}

int fa_bwd_host(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int causal,
                int dtype, int deterministic, int chunk_b, void* staging, size_t staging_bytes,
                cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  if (B < 1 || chunk_b < 1 || chunk_b > B) return FA_ERR_SHAPE;
  const size_t need = fa_bwd_host_staging_size(B, Hq, Hkv, Nq, Nkv, d, deterministic, chunk_b);
  if (need == 0) {
    // invalid shape: fa_bwd's validation names the argument (it launches nothing)
    return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic,
                  nullptr, 0, stream);
  }
  if (staging == nullptr || staging_bytes < need) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(staging) & (kAlign - 1)) != 0) return FA_ERR_ALIGN;
  CopyStreams cs;
  int st = copy_streams(&cs);
  if (st) return st;
  Events ev;   // 0: entry; 1, 2: inputs of slot 0, 1 in; 3, 4: slot 0, 1 computed; 5, 6: slot 0, 1 free
  if ((st = ev.create())) return st;
  const Slot full = slot_layout(chunk_b, Hq, Hkv, Nq, Nkv, d, deterministic);
  const int nchunks = (B + chunk_b - 1) / chunk_b;
  const size_t q_seq = static_cast<size_t>(Hq) * Nq * d * 2;    // bytes of one sequence
  const size_t k_seq = static_cast<size_t>(Hkv) * Nkv * d * 2;
  const size_t l_seq = static_cast<size_t>(Hq) * Nq * 4;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // the copies start after whatever the caller queued before (e.g. an earlier use of the staging)
  if (!ok(cudaEventRecord(ev.e[0], stream)) || !ok(cudaStreamWaitEvent(cs.in, ev.e[0], 0))) return FA_ERR_CUDA;
  for (int c = 0; c < nchunks; ++c) {
    const int s = c & 1;
    const int b0 = c * chunk_b;
    const int cb = B - b0 < chunk_b ? B - b0 : chunk_b;
    uint8_t* base = at(staging, s * full.bytes);
    const size_t qn = cb * q_seq, kn = cb * k_seq, ln = cb * l_seq;
    // inputs of chunk c, once slot s has been emptied by chunk c - 2
    if (c >= 2 && !ok(cudaStreamWaitEvent(cs.in, ev.e[5 + s], 0))) return FA_ERR_CUDA;
    if (!ok(cudaMemcpyAsync(base + full.q, at(q, b0 * q_seq), qn, cudaMemcpyHostToDevice, cs.in)) ||
        !ok(cudaMemcpyAsync(base + full.k, at(k, b0 * k_seq), kn, cudaMemcpyHostToDevice, cs.in)) ||
        !ok(cudaMemcpyAsync(base + full.v, at(v, b0 * k_seq), kn, cudaMemcpyHostToDevice, cs.in)) ||
        !ok(cudaMemcpyAsync(base + full.o, at(o, b0 * q_seq), qn, cudaMemcpyHostToDevice, cs.in)) ||
        !ok(cudaMemcpyAsync(base + full.dO, at(dO, b0 * q_seq), qn, cudaMemcpyHostToDevice, cs.in)) ||
        !ok(cudaMemcpyAsync(base + full.lse, at(lse, b0 * l_seq), ln, cudaMemcpyHostToDevice, cs.in)) ||
        !ok(cudaEventRecord(ev.e[1 + s], cs.in)))
      return FA_ERR_CUDA;
    // compute chunk c on the caller's stream
    if (!ok(cudaStreamWaitEvent(stream, ev.e[1 + s], 0))) return FA_ERR_CUDA;
    st = fa_bwd(base + full.q, base + full.k, base + full.v, base + full.o, base + full.dO,
                reinterpret_cast<const float*>(base + full.lse), base + full.dq, base + full.dk, base + full.dv, cb,
                Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic, base + full.ws, full.ws_bytes, stream);
    if (st) return st;
    if (!ok(cudaEventRecord(ev.e[3 + s], stream))) return FA_ERR_CUDA;
    // outputs of chunk c
    if (!ok(cudaStreamWaitEvent(cs.out, ev.e[3 + s], 0)) ||
        !ok(cudaMemcpyAsync(at(dq, b0 * q_seq), base + full.dq, qn, cudaMemcpyDeviceToHost, cs.out)) ||
        !ok(cudaMemcpyAsync(at(dk, b0 * k_seq), base + full.dk, kn, cudaMemcpyDeviceToHost, cs.out)) ||
        !ok(cudaMemcpyAsync(at(dv, b0 * k_seq), base + full.dv, kn, cudaMemcpyDeviceToHost, cs.out)) ||
        !ok(cudaEventRecord(ev.e[5 + s], cs.out)))
      return FA_ERR_CUDA;
  }
  // the call completes on `stream` once the last outputs are in host memory
  for (int s = 0; s < (nchunks > 1 ? 2 : 1); ++s)
    if (!ok(cudaStreamWaitEvent(stream, ev.e[5 + s], 0))) return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"
