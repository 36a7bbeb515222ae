// host_pipeline.cu -- fa_bwd_host: the backward for tensors that live in host
// memory, with the transfers overlapped with the computation.
//
// The (batch, kv-head) groups of a dense problem are independent: group g owns
// query heads [g*G, g*G + G) of its sequence (G = Hq / Hkv) and key/value head
// g, and in the contiguous [B, H, N, d] layouts a run of consecutive groups is
// one contiguous range of every tensor.  So the problem is cut into chunks of
// chunk_groups groups, each computed as an fa_bwd of one "sequence" with
// G * chunk_groups query heads, and the chunks flow through a ring of `slots`
// device staging slots:
//   copy-in stream   inputs of chunk c into slot c % slots, once the slot's
//                    previous chunk has been copied out
//   slot stream s    fa_bwd of every chunk of slot s, once its inputs are in
//   copy-out stream  dQ, dK, dV of chunk c, once it has computed
// Each slot computes on a stream of its own, so the first CTAs of chunk c + 1
// fill the SMs that the tail of chunk c leaves idle (under causal masking the
// CTAs of one chunk are very unequal).  The host link is slower than the
// computation on large problems, so what this buys is that the copy-in stream
// never waits: the chunk size sets how long the first chunk's copy and the last
// chunk's copy-out stay exposed.  The caller owns the staging memory
// (fa_bwd_host_staging_size); the only state kept here is the copy and slot
// streams of each device, created on first use.  Every copy is one
// cudaMemcpyAsync of a contiguous range.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace {

constexpr int kMaxDevices = 64;
struct Streams {
  cudaStream_t in = nullptr;
  cudaStream_t out = nullptr;
  cudaStream_t slot[FA_HOST_MAX_SLOTS] = {};
};
Streams g_streams[kMaxDevices];
std::mutex g_streams_mu;

int device_streams(Streams* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_streams_mu);
  Streams& s = g_streams[dev];
  if (s.in == nullptr) {
    Streams n;
    bool ok = cudaStreamCreateWithFlags(&n.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&n.out, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < FA_HOST_MAX_SLOTS; ++i)
      ok = cudaStreamCreateWithFlags(&n.slot[i], cudaStreamNonBlocking) == cudaSuccess;
    if (!ok) {   // release what was created; the next call tries again
      for (cudaStream_t x : {n.in, n.out})
        if (x) cudaStreamDestroy(x);
      for (cudaStream_t x : n.slot)
        if (x) cudaStreamDestroy(x);
      return FA_ERR_CUDA;
    }
    s = n;
  }
  *out = s;
  return FA_OK;
}

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Byte offsets inside one staging slot holding a chunk of cg groups.
struct Slot {
  size_t q, o, dO, dq, k, v, dk, dv, lse, ws, bytes;
  size_t ws_bytes;
};

Slot slot_layout(int cg, int G, int Nq, int Nkv, int d, int deterministic) {
  Slot s;
  const size_t q_bytes = static_cast<size_t>(cg) * G * Nq * d * 2;
  const size_t k_bytes = static_cast<size_t>(cg) * Nkv * d * 2;
  const size_t lse_bytes = static_cast<size_t>(cg) * G * Nq * 4;
  s.ws_bytes = fa_bwd_workspace_size(1, cg * G, cg, Nq, Nkv, d, deterministic);
  size_t off = 0;
  s.q = off; off += up(q_bytes);
  s.o = off; off += up(q_bytes);
  s.dO = off; off += up(q_bytes);
  s.dq = off; off += up(q_bytes);
  s.k = off; off += up(k_bytes);
  s.v = off; off += up(k_bytes);
  s.dk = off; off += up(k_bytes);
  s.dv = off; off += up(k_bytes);
  s.lse = off; off += up(lse_bytes);
  s.ws = off; off += up(s.ws_bytes);
  s.bytes = off;
  return s;
}

// Slots in use: never more than there are chunks.
int slots_used(int groups, int chunk_groups, int slots) {
  const int nchunks = (groups + chunk_groups - 1) / chunk_groups;
  return nchunks < slots ? nchunks : slots;
}

struct Events {
  // per slot: 0 inputs in, 1 computed, 2 copied out (slot free); plus the entry event
  cudaEvent_t e[3 * FA_HOST_MAX_SLOTS + 1] = {};
  ~Events() {
    for (cudaEvent_t x : e)
      if (x) cudaEventDestroy(x);   // released once the work that records it has completed
  }
  int create(int slots) {
    for (int i = 0; i < 3 * slots; ++i)
      if (cudaEventCreateWithFlags(&e[i], cudaEventDisableTiming) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaEventCreateWithFlags(&e[3 * FA_HOST_MAX_SLOTS], cudaEventDisableTiming) != cudaSuccess)
      return FA_ERR_CUDA;
    return FA_OK;
  }
  cudaEvent_t entry() const { return e[3 * FA_HOST_MAX_SLOTS]; }
};

const uint8_t* at(const void* p, size_t off) { return static_cast<const uint8_t*>(p) + off; }
uint8_t* at(void* p, size_t off) { return static_cast<uint8_t*>(p) + off; }

bool shape_ok(int B, int Hq, int Hkv, int chunk_groups, int slots) {
  if (B < 1 || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0) return false;
  if (slots < 1 || slots > FA_HOST_MAX_SLOTS) return false;
  return chunk_groups >= 1 && static_cast<long long>(chunk_groups) <= static_cast<long long>(B) * Hkv;
}

}  // namespace

extern "C" {

size_t fa_bwd_host_staging_size(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int deterministic,
                                int chunk_groups, int slots) {
  if (!shape_ok(B, Hq, Hkv, chunk_groups, slots)) return 0;
  if (fa_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d, deterministic) == 0) return 0;
  const int G = Hq / Hkv;
  return slots_used(B * Hkv, chunk_groups, slots) * slot_layout(chunk_groups, G, Nq, Nkv, d, deterministic).bytes;
}

int fa_bwd_host(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int causal,
                int dtype, int deterministic, int chunk_groups, int slots, void* staging, size_t staging_bytes,
                cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  const size_t need = fa_bwd_host_staging_size(B, Hq, Hkv, Nq, Nkv, d, deterministic, chunk_groups, slots);
  if (need == 0) {
    if (fa_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d, deterministic) == 0) {
      // invalid problem: fa_bwd's validation names the argument (it launches nothing)
      return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic,
                    nullptr, 0, stream);
    }
    return FA_ERR_SHAPE;   // chunk_groups or slots out of range
  }
  if (staging == nullptr || staging_bytes < need) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(staging) & (kAlign - 1)) != 0) return FA_ERR_ALIGN;
  // the remaining arguments fa_bwd checks, checked before any copy is queued (so that a
  // rejected call leaves nothing in flight)
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || causal < FA_CAUSAL_NONE || causal > FA_CAUSAL_BOTTOM_RIGHT) return FA_ERR_ARG;
  Streams ss;
  int st = device_streams(&ss);
  if (st) return st;
  const int groups = B * Hkv;
  const int G = Hq / Hkv;
  const int nslots = slots_used(groups, chunk_groups, slots);
  Events ev;
  if ((st = ev.create(nslots))) return st;
  const Slot full = slot_layout(chunk_groups, G, Nq, Nkv, d, deterministic);
  const int nchunks = (groups + chunk_groups - 1) / chunk_groups;
  const size_t q_grp = static_cast<size_t>(G) * Nq * d * 2;    // bytes of one group
  const size_t k_grp = static_cast<size_t>(Nkv) * d * 2;
  const size_t l_grp = static_cast<size_t>(G) * Nq * 4;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  // After a failure, wait for whatever was queued on the internal streams, so that
  // no copy into or out of the caller's buffers outlives the call.
  auto fail = [&](int code) {
    cudaStreamSynchronize(ss.in);
    for (int i = 0; i < nslots; ++i) cudaStreamSynchronize(ss.slot[i]);
    cudaStreamSynchronize(ss.out);
    return code;
  };
  // everything starts after whatever the caller queued before (e.g. an earlier use of the staging)
  if (!ok(cudaEventRecord(ev.entry(), stream)) || !ok(cudaStreamWaitEvent(ss.in, ev.entry(), 0))) return FA_ERR_CUDA;
  for (int c = 0; c < nchunks; ++c) {
    const int s = c % nslots;
    cudaEvent_t in_done = ev.e[3 * s], computed = ev.e[3 * s + 1], freed = ev.e[3 * s + 2];
    const size_t g0 = static_cast<size_t>(c) * chunk_groups;
    const int cg = groups - static_cast<int>(g0) < chunk_groups ? groups - static_cast<int>(g0) : chunk_groups;
    uint8_t* base = at(staging, s * full.bytes);
    const size_t qn = cg * q_grp, kn = cg * k_grp, ln = cg * l_grp;
    // inputs of chunk c, once the slot's previous chunk has been copied out
    if (c >= nslots && !ok(cudaStreamWaitEvent(ss.in, freed, 0))) return fail(FA_ERR_CUDA);
    if (!ok(cudaMemcpyAsync(base + full.q, at(q, g0 * q_grp), qn, cudaMemcpyHostToDevice, ss.in)) ||
        !ok(cudaMemcpyAsync(base + full.k, at(k, g0 * k_grp), kn, cudaMemcpyHostToDevice, ss.in)) ||
        !ok(cudaMemcpyAsync(base + full.v, at(v, g0 * k_grp), kn, cudaMemcpyHostToDevice, ss.in)) ||
        !ok(cudaMemcpyAsync(base + full.o, at(o, g0 * q_grp), qn, cudaMemcpyHostToDevice, ss.in)) ||
        !ok(cudaMemcpyAsync(base + full.dO, at(dO, g0 * q_grp), qn, cudaMemcpyHostToDevice, ss.in)) ||
        !ok(cudaMemcpyAsync(base + full.lse, at(lse, g0 * l_grp), ln, cudaMemcpyHostToDevice, ss.in)) ||
        !ok(cudaEventRecord(in_done, ss.in)))
      return fail(FA_ERR_CUDA);
    // compute chunk c on its slot's stream
    cudaStream_t cs = ss.slot[s];
    if (!ok(cudaStreamWaitEvent(cs, in_done, 0))) return fail(FA_ERR_CUDA);
    st = fa_bwd(base + full.q, base + full.k, base + full.v, base + full.o, base + full.dO,
                reinterpret_cast<const float*>(base + full.lse), base + full.dq, base + full.dk, base + full.dv, 1,
                cg * G, cg, Nq, Nkv, d, scale, causal, dtype, deterministic, base + full.ws, full.ws_bytes, cs);
    if (st) return fail(st);
    if (!ok(cudaEventRecord(computed, cs))) return fail(FA_ERR_CUDA);
    // outputs of chunk c
    if (!ok(cudaStreamWaitEvent(ss.out, computed, 0)) ||
        !ok(cudaMemcpyAsync(at(dk, g0 * k_grp), base + full.dk, kn, cudaMemcpyDeviceToHost, ss.out)) ||
        !ok(cudaMemcpyAsync(at(dv, g0 * k_grp), base + full.dv, kn, cudaMemcpyDeviceToHost, ss.out)) ||
        !ok(cudaMemcpyAsync(at(dq, g0 * q_grp), base + full.dq, qn, cudaMemcpyDeviceToHost, ss.out)) ||
        !ok(cudaEventRecord(freed, ss.out)))
      return fail(FA_ERR_CUDA);
  }
  // the call completes on `stream` once the last outputs are in host memory (the copy-out
  // stream is in order, so its last event covers every chunk)
  if (!ok(cudaStreamWaitEvent(stream, ev.e[3 * ((nchunks - 1) % nslots) + 2], 0))) return fail(FA_ERR_CUDA);
  return FA_OK;
}

}  // extern "C"
