// noalloc.cu -- fa_bwd_noalloc: the backward for callers that cannot allocate
// device memory.
//
// fa_bwd needs a caller-provided workspace.  Some callers have no way to get
// one: a plugin running inside an inference engine whose host framework owns
// every device allocation and offers no scratch, or a serving loop that bans
// cudaMalloc after start-up because it synchronises the device and fragments
// the memory pool.  For them this entry point takes its scratch from one
// fixed array compiled into the library instead.  It allocates nothing itself:
// no cudaMalloc, no cudaFree, no allocating library routine.
//
// The array lives in every GPU's memory from the moment the library's device
// code is loaded on that GPU until the process exits.  Host code must not use
// the array's name as an address (on the host it names a stand-in, not device
// memory): the first call on each device asks the runtime for the device
// address with that device current, checks the result, and caches it.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[FA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_static_scratch on the current device (looked up once per device).
int static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                              const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Nq,
                              int Nkv, int d, float scale, int causal, int dtype, int deterministic,
                              cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  const size_t need = fa_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d, deterministic);
  if (need == 0) {
    // invalid shape: let fa_bwd's validation report which argument is wrong (it launches nothing)
    return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic,
                  nullptr, 0, stream);
  }
  // the checks fa_bwd makes before its workspace check come first here too
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  if (!std::isfinite(scale) || causal < FA_CAUSAL_NONE || causal > FA_CAUSAL_BOTTOM_RIGHT) return FA_ERR_ARG;
  if (need > FA_STATIC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  void* ws = nullptr;
  const int st = static_scratch(&ws);
  if (st != FA_OK) return st;
  // Every stage rewrites what it later reads (the abort word, -L*log2e, D and the
  // zeroed dQ accumulator), so whatever an earlier call left in the array is irrelevant.
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic, ws,
                FA_STATIC_SCRATCH_BYTES, stream);
}
