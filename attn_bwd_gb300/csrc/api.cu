// api.cu -- the C ABI declared in include/fa.h: argument validation, workspace
// carve-up, TMA descriptor encoding and the order of the backward's stages.
// No device memory is allocated here and nothing synchronises except
// fa_last_device_error().
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"
#include "kernels.h"

namespace fa {
namespace {

// Device status word shared by every kernel family (first failure wins).
__device__ unsigned int g_status;

constexpr int kMaxDevices = 64;
unsigned int* g_status_ptr[kMaxDevices] = {};
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int status_ptr(unsigned int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return FA_ERR_CUDA;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_status_ptr[dev];
  return FA_OK;
}

int get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return FA_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return FA_ERR_CUDA;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return FA_OK;
}

// 3-D view [heads][rows][d] of a contiguous 16-bit tensor; box = 64 columns x box_rows rows,
// 128-byte swizzle (one box row is exactly 128 bytes).  Rows past `rows` read as zero.
int make_map(CUtensorMap* m, const void* base, int bf16, int d, int rows, long long heads, int box_rows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(heads)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(rows) * d * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box_rows), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

int check_shape(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int dtype) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1) return FA_ERR_SHAPE;
  if (Nq > FA_MAX_SEQ || Nkv > FA_MAX_SEQ || B > 65535 || Hq > 65535) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEADDIM;
  if (Hq % Hkv != 0) return FA_ERR_GQA;
  if (dtype != FA_F16 && dtype != FA_BF16) return FA_ERR_DTYPE;
  // grid-size limits of the largest launch (one CTA per 64 query rows x head x batch)
  const long long bh = static_cast<long long>(B) * Hq;
  if (bh * ((Nq + 63) / 64) > 0x7fffffffLL || static_cast<long long>(B) * Hkv * ((Nkv + 127) / 128) > 0x7fffffffLL)
    return FA_ERR_SHAPE;
  return FA_OK;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

size_t ws_bytes(int B, int Hq, int Nq, int d, int deterministic) {
  const size_t rows = static_cast<size_t>(B) * Hq * round_up(Nq, kRowPad);
  size_t total = 2 * align_up(rows * sizeof(float));
  if (!deterministic) total += align_up(rows * d * sizeof(float));
  return total;
}

Workspace carve(void* ws, int B, int Hq, int Nq, int d, int deterministic) {
  const size_t rows = static_cast<size_t>(B) * Hq * round_up(Nq, kRowPad);
  uint8_t* p = static_cast<uint8_t*>(ws);
  Workspace w;
  w.nLg = reinterpret_cast<float*>(p);
  w.Dv = reinterpret_cast<float*>(p + align_up(rows * sizeof(float)));
  w.dq_acc = deterministic ? nullptr : reinterpret_cast<float*>(p + 2 * align_up(rows * sizeof(float)));
  (void)d;
  return w;
}

Problem make_problem(int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int causal, int dtype,
                     int deterministic) {
  Problem pb;
  pb.B = B; pb.Hq = Hq; pb.Hkv = Hkv; pb.Nq = Nq; pb.Nkv = Nkv; pb.d = d;
  pb.NqPad = round_up(Nq, kRowPad);
  pb.scale = scale;
  pb.causal = causal != FA_CAUSAL_NONE ? 1 : 0;
  pb.causal_off = causal == FA_CAUSAL_BOTTOM_RIGHT ? Nkv - Nq : 0;
  pb.bf16 = dtype == FA_BF16 ? 1 : 0;
  pb.deterministic = deterministic ? 1 : 0;
  return pb;
}

int check_ws(void* workspace, size_t bytes, int B, int Hq, int Nq, int d, int deterministic) {
  if (workspace == nullptr) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return FA_ERR_ALIGN;
  if (bytes < ws_bytes(B, Hq, Nq, d, deterministic)) return FA_ERR_WORKSPACE;
  return FA_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "invalid shape (a size < 1 or above the supported limit)";
    case FA_ERR_HEADDIM: return "head dimension must be 64 or 128";
    case FA_ERR_GQA: return "Hq must be a multiple of Hkv";
    case FA_ERR_ALIGN: return "a pointer is not 16-byte aligned (workspace: 256-byte)";
    case FA_ERR_WORKSPACE: return "workspace missing or smaller than fa_bwd_workspace_size()";
    case FA_ERR_DTYPE: return "dtype must be FA_F16 or FA_BF16";
    case FA_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    case FA_ERR_ARG: return "an argument is out of range";
    default: return "unknown fa_status";
  }
}

size_t fa_bwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int deterministic) {
  if (check_shape(B, Hq, Hkv, Nq, Nkv, d, FA_BF16) != FA_OK) return 0;
  return ws_bytes(B, Hq, Nq, d, deterministic);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
           int Nkv, int d, float scale, int causal, int dtype, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  int st = check_shape(B, Hq, Hkv, Nq, Nkv, d, dtype);
  if (st) return st;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o) || misaligned(lse)) return FA_ERR_ALIGN;
  if (!std::isfinite(scale) || causal < FA_CAUSAL_NONE || causal > FA_CAUSAL_BOTTOM_RIGHT) return FA_ERR_ARG;
  FwdArgs a;
  a.pb = make_problem(B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, 1);
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  if ((st = get_encoder())) return st;
  unsigned int* status = nullptr;
  if ((st = status_ptr(&status))) return st;
  CUtensorMap tq, tk, tv;
  const int bf = a.pb.bf16;
  if ((st = make_map(&tq, q, bf, d, Nq, static_cast<long long>(B) * Hq, 128))) return st;
  if ((st = make_map(&tk, k, bf, d, Nkv, static_cast<long long>(B) * Hkv, 128))) return st;
  if ((st = make_map(&tv, v, bf, d, Nkv, static_cast<long long>(B) * Hkv, 128))) return st;
  return cuda_status(launch_fwd(a, tq, tk, tv, status, stream));
}

int fa_bwd_preprocess(const void* o, const void* dO, const float* lse, int B, int Hq, int Hkv, int Nq, int Nkv,
                      int d, int dtype, int deterministic, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  if (!o || !dO || !lse) return FA_ERR_NULL;
  int st = check_shape(B, Hq, Hkv, Nq, Nkv, d, dtype);
  if (st) return st;
  if (misaligned(o) || misaligned(dO) || misaligned(lse)) return FA_ERR_ALIGN;
  if ((st = check_ws(workspace, workspace_bytes, B, Hq, Nq, d, deterministic))) return st;
  const Problem pb = make_problem(B, Hq, Hkv, Nq, Nkv, d, 1.0f, 0, dtype, deterministic);
  const Workspace w = carve(workspace, B, Hq, Nq, d, deterministic);
  return cuda_status(launch_preprocess(pb, o, dO, lse, w, stream));
}

int fa_bwd_main(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, int B, int Hq,
                int Hkv, int Nq, int Nkv, int d, float scale, int causal, int dtype, int deterministic,
                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !dO || !dk || !dv) return FA_ERR_NULL;
  int st = check_shape(B, Hq, Hkv, Nq, Nkv, d, dtype);
  if (st) return st;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(dO) || misaligned(dk) || misaligned(dv))
    return FA_ERR_ALIGN;
  if (!std::isfinite(scale) || causal < FA_CAUSAL_NONE || causal > FA_CAUSAL_BOTTOM_RIGHT) return FA_ERR_ARG;
  if ((st = check_ws(workspace, workspace_bytes, B, Hq, Nq, d, deterministic))) return st;
  if ((st = get_encoder())) return st;
  MainArgs a;
  a.pb = make_problem(B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic);
  a.ws = carve(workspace, B, Hq, Nq, d, deterministic);
  a.dk = dk;
  a.dv = dv;
  if ((st = status_ptr(&a.status))) return st;
  CUtensorMap tq, tdo, tk, tv;
  const int bf = a.pb.bf16;
  if ((st = make_map(&tq, q, bf, d, Nq, static_cast<long long>(B) * Hq, 64))) return st;
  if ((st = make_map(&tdo, dO, bf, d, Nq, static_cast<long long>(B) * Hq, 64))) return st;
  if ((st = make_map(&tk, k, bf, d, Nkv, static_cast<long long>(B) * Hkv, 128))) return st;
  if ((st = make_map(&tv, v, bf, d, Nkv, static_cast<long long>(B) * Hkv, 128))) return st;
  return cuda_status(launch_bwd_main(a, tq, tdo, tk, tv, stream));
}

int fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO, void* dq, int B, int Hq, int Hkv,
              int Nq, int Nkv, int d, float scale, int causal, int dtype, int deterministic, void* workspace,
              size_t workspace_bytes, cudaStream_t stream) {
  if (!dq) return FA_ERR_NULL;
  int st = check_shape(B, Hq, Hkv, Nq, Nkv, d, dtype);
  if (st) return st;
  if (misaligned(dq)) return FA_ERR_ALIGN;
  if (!std::isfinite(scale) || causal < FA_CAUSAL_NONE || causal > FA_CAUSAL_BOTTOM_RIGHT) return FA_ERR_ARG;
  if ((st = check_ws(workspace, workspace_bytes, B, Hq, Nq, d, deterministic))) return st;
  DqArgs a;
  a.pb = make_problem(B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic);
  a.ws = carve(workspace, B, Hq, Nq, d, deterministic);
  a.dq = dq;
  if (!deterministic) return cuda_status(launch_dq_convert(a.pb, a.ws, dq, stream));
  if (!q || !k || !v || !dO) return FA_ERR_NULL;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(dO)) return FA_ERR_ALIGN;
  if ((st = get_encoder())) return st;
  if ((st = status_ptr(&a.status))) return st;
  CUtensorMap tq, tdo, tk, tv;
  const int bf = a.pb.bf16;
  if ((st = make_map(&tq, q, bf, d, Nq, static_cast<long long>(B) * Hq, 128))) return st;
  if ((st = make_map(&tdo, dO, bf, d, Nq, static_cast<long long>(B) * Hq, 128))) return st;
  if ((st = make_map(&tk, k, bf, d, Nkv, static_cast<long long>(B) * Hkv, 128))) return st;
  if ((st = make_map(&tv, v, bf, d, Nkv, static_cast<long long>(B) * Hkv, 128))) return st;
  return cuda_status(launch_bwd_dq_det(a, tq, tdo, tk, tv, stream));
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dq,
           void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int causal, int dtype,
           int deterministic, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  int st = check_shape(B, Hq, Hkv, Nq, Nkv, d, dtype);
  if (st) return st;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o) || misaligned(dO) || misaligned(lse) ||
      misaligned(dq) || misaligned(dk) || misaligned(dv))
    return FA_ERR_ALIGN;
  if (!std::isfinite(scale) || causal < FA_CAUSAL_NONE || causal > FA_CAUSAL_BOTTOM_RIGHT) return FA_ERR_ARG;
  if ((st = check_ws(workspace, workspace_bytes, B, Hq, Nq, d, deterministic))) return st;
  if ((st = fa_bwd_preprocess(o, dO, lse, B, Hq, Hkv, Nq, Nkv, d, dtype, deterministic, workspace, workspace_bytes,
                              stream)))
    return st;
  if ((st = fa_bwd_main(q, k, v, dO, dk, dv, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic, workspace,
                        workspace_bytes, stream)))
    return st;
  return fa_bwd_dq(q, k, v, dO, dq, B, Hq, Hkv, Nq, Nkv, d, scale, causal, dtype, deterministic, workspace,
                   workspace_bytes, stream);
}

int fa_last_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
  unsigned int* p = nullptr;
  if (status_ptr(&p)) return FA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return FA_ERR_CUDA;
    return static_cast<int>(v >> 16) == FA_ERR_DEVICE_TIMEOUT ? FA_ERR_DEVICE_TIMEOUT : FA_ERR_CUDA;
  }
  return FA_OK;
}

int fa_selftest_wait_timeout(int timeout_us, cudaStream_t stream) {
  if (timeout_us < 1 || timeout_us > 5000000) return FA_ERR_ARG;
  unsigned int* p = nullptr;
  int st = status_ptr(&p);
  if (st) return st;
  return cuda_status(launch_wait_selftest(p, static_cast<long long>(timeout_us) * 1000, stream));
}

}  // extern "C"
