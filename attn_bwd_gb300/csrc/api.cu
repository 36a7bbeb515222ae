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

// Device-wide report word shared by every kernel (first failure since the last
// fa_last_device_error() wins).  Kernels only write it; none acts on it.
__device__ unsigned int g_status;

// Abort words of forward calls (a backward call keeps its own in its workspace).
// Call n of a device takes slot n mod kFwdSlots with tag n / kFwdSlots + 1: a tag
// that no earlier call on that slot had (for 2^32 - 1 rounds of the ring), so the
// word needs no zeroing before the launch and what an earlier call left in it is
// never read as this call's abort.  Calls in flight at the same time (up to
// kFwdSlots) never share a slot.
constexpr int kFwdSlots = 256;
__device__ unsigned int g_fwd_abort[kFwdSlots];

constexpr int kMaxDevices = 64;
unsigned int* g_status_ptr[kMaxDevices] = {};
unsigned int* g_fwd_abort_ptr[kMaxDevices] = {};
unsigned long long g_fwd_next[kMaxDevices] = {};
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

// Next forward abort slot of the current device and the call's tag for it.
int fwd_abort_slot(unsigned int** out, unsigned int* tag) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_fwd_abort_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fwd_abort) != cudaSuccess) return FA_ERR_CUDA;
    g_fwd_abort_ptr[dev] = static_cast<unsigned int*>(p);
  }
  const unsigned long long n = g_fwd_next[dev]++;
  *out = g_fwd_abort_ptr[dev] + n % kFwdSlots;
  *tag = static_cast<unsigned int>((n / kFwdSlots) % 0xFFFFFFFFull) + 1u;
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

// 4-D view (d, rows, heads, batch) of a 16-bit tensor with element strides s
// for the row, head and batch axes; box = 64 columns x box_rows rows of one
// head, 128-byte swizzle (one box row is exactly 128 bytes).  Columns past d
// and rows past `rows` read as zero.
int make_map(CUtensorMap* m, const void* base, int bf16, int d, int rows, int heads, int batch, Str3 s,
             int box_rows) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(s.n) * 2, static_cast<cuuint64_t>(s.h) * 2,
                                 static_cast<cuuint64_t>(s.b) * 2};
  const cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(box_rows), 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 4-D view (keys, queries, heads, batch) of a 16-bit bias (or dBias) with element strides s
// for the query, head and batch axes (0 broadcasts); box = box_k keys x box_q
// queries of one head and sequence: 128 keys unswizzled (256-byte rows in shared
// memory) or 64 keys with the 128-byte swizzle.  A broadcast axis gets extent 1
// (so it is addressed at coordinate 0) and a stride that is never used; keys
// past Nkv and queries past Nq read as zero (and are not written by a store).
int make_bias_map(CUtensorMap* m, const void* base, int bf16, int Nkv, int Nq, int Hq, int B, Str3 s, int box_k,
                  int box_q) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(Nkv), static_cast<cuuint64_t>(s.n ? Nq : 1),
                              static_cast<cuuint64_t>(s.h ? Hq : 1), static_cast<cuuint64_t>(s.b ? B : 1)};
  // a broadcast axis takes the stride of a dense layout (capped; it is never stepped)
  const cuuint64_t cap = 1ull << 39;
  const cuuint64_t rq = s.n ? static_cast<cuuint64_t>(s.n) * 2 : (static_cast<cuuint64_t>(Nkv) * 2 + 15) / 16 * 16;
  const cuuint64_t rh = s.h ? static_cast<cuuint64_t>(s.h) * 2 : (rq * dims[1] < cap ? rq * dims[1] : cap);
  const cuuint64_t rb = s.b ? static_cast<cuuint64_t>(s.b) * 2 : (rh * dims[2] < cap ? rh * dims[2] : cap);
  const cuuint64_t strides[3] = {rq, rh, rb};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(box_k), static_cast<cuuint32_t>(box_q), 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUresult r = g_encode(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                              const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              box_k == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

int check_shape(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int dtype) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1) return FA_ERR_SHAPE;
  if (Nq > FA_MAX_SEQ || Nkv > FA_MAX_SEQ || B > 65535 || Hq > 65535) return FA_ERR_SHAPE;
  if (d < 8 || d > 128 || d % 8 != 0) return FA_ERR_HEADDIM;   // served by the d = 64 / 128 kernels
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

// The fp32 dQ accumulator rows are as wide as the kernel that fills them (64 or 128).
int kernel_d(int d) { return d <= 64 ? 64 : 128; }

// Workspace: [256 B: the call's abort word][-L*log2e][D][fp32 dQ accumulator (atomic mode)].
size_t ws_bytes(int B, int Hq, int Nq, int d, int deterministic) {
  const size_t rows = static_cast<size_t>(B) * Hq * round_up(Nq, kRowPad);
  size_t total = kAlign + 2 * align_up(rows * sizeof(float));
  if (!deterministic) total += align_up(rows * kernel_d(d) * sizeof(float));
  return total;
}

Workspace carve(void* ws, int B, int Hq, int Nq, int d, int deterministic) {
  const size_t rows = static_cast<size_t>(B) * Hq * round_up(Nq, kRowPad);
  uint8_t* p = static_cast<uint8_t*>(ws);
  Workspace w;
  w.abort = reinterpret_cast<unsigned int*>(p);
  p += kAlign;
  w.nLg = reinterpret_cast<float*>(p);
  w.Dv = reinterpret_cast<float*>(p + align_up(rows * sizeof(float)));
  w.dq_acc = deterministic ? nullptr : reinterpret_cast<float*>(p + 2 * align_up(rows * sizeof(float)));
  (void)d;
  return w;
}

// Where the sequences of a batch live: a dense batch (cu_q == nullptr; Nq, Nkv
// are the lengths) or a packed one (Nq, Nkv are the longest lengths, total_q,
// total_k the rows of each head, cu_q / cu_k the device offsets).
struct Geo {
  int B, Hq, Hkv, Nq, Nkv, d;
  const int* cu_q;
  const int* cu_k;
  int total_q, total_k;
  Strides st;        // element strides of every tensor
  const void* bias = nullptr;   // optional additive bias and its gradient (see fa_bias)
  Str3 bias_st{0, 0, 0};
  void* dbias = nullptr;
  Str3 dbias_st{0, 0, 0};
  int batch() const { return cu_q ? 1 : B; }
  int rows_q() const { return cu_q ? total_q : Nq; }
  int rows_k() const { return cu_q ? total_k : Nkv; }
};

// Strides of contiguous [batch, heads, rows, d] tensors (and [batch, heads, rows] for L).
Str3 contiguous(int heads, long long rows, int d) {
  return Str3{heads * rows * d, rows * d, d};
}

Strides contiguous_all(int Hq, int Hkv, long long rows_q, long long rows_k, int d) {
  Strides s;
  s.q = s.o = s.dO = s.dq = contiguous(Hq, rows_q, d);
  s.k = s.v = s.dk = s.dv = contiguous(Hkv, rows_k, d);
  s.lse = contiguous(Hq, rows_q, 1);
  return s;
}

Geo dense(int B, int Hq, int Hkv, int Nq, int Nkv, int d) {
  return Geo{B, Hq, Hkv, Nq, Nkv, d, nullptr, nullptr, Nq, Nkv, contiguous_all(Hq, Hkv, Nq, Nkv, d)};
}

// Largest number of rows per head of a packed batch (keeps every TMA row
// coordinate, start of a sequence plus a tile, inside int32).
constexpr int kMaxTotal = 1 << 30;

// Strides must be positive, and those of 16-bit tensors multiples of 8 elements
// (16 bytes: TMA and the 16-byte loads and stores); a packed batch ignores the
// batch stride.
bool bad_str(const Str3& s, bool packed, int mult) {
  if (s.h < 1 || s.n < 1 || s.h % mult || s.n % mult) return true;
  if (!packed && (s.b < 1 || s.b % mult)) return true;
  return s.h > (1LL << 36) || s.n > (1LL << 36) || (!packed && s.b > (1LL << 36));
}

int check_geo(const Geo& g, int dtype) {
  int st = check_shape(g.B, g.Hq, g.Hkv, g.Nq, g.Nkv, g.d, dtype);
  if (st) return st;
  if (g.cu_q != nullptr || g.cu_k != nullptr) {
    if (g.cu_q == nullptr || g.cu_k == nullptr) return FA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(g.cu_q) & 3u) || (reinterpret_cast<uintptr_t>(g.cu_k) & 3u)) return FA_ERR_ALIGN;
    if (g.total_q < 1 || g.total_k < 1 || g.total_q > kMaxTotal || g.total_k > kMaxTotal) return FA_ERR_SHAPE;
  }
  const bool pk = g.cu_q != nullptr;
  const Strides& s = g.st;
  for (const Str3* t : {&s.q, &s.k, &s.v, &s.o, &s.dO, &s.dq, &s.dk, &s.dv})
    if (bad_str(*t, pk, 8)) return FA_ERR_ARG;
  if (bad_str(s.lse, pk, 1)) return FA_ERR_ARG;
  if (g.dbias != nullptr && g.bias == nullptr) return FA_ERR_NULL;
  if (g.bias != nullptr) {
    if (misaligned(g.bias)) return FA_ERR_ALIGN;
    const Str3& b = g.bias_st;        // 0 broadcasts; otherwise whole 16-byte pieces
    if (b.b < 0 || b.h < 0 || b.n < 0 || b.b % 8 || b.h % 8 || b.n % 8) return FA_ERR_ARG;
  }
  if (g.dbias != nullptr) {
    if (misaligned(g.dbias)) return FA_ERR_ALIGN;
    const Str3& b = g.dbias_st;       // every (b, h, q) row its own
    if (b.b < 1 || b.h < 1 || b.n < 1 || b.b % 8 || b.h % 8 || b.n % 8) return FA_ERR_ARG;
  }
  return FA_OK;
}

bool bad_args(float scale, int causal) {
  return !std::isfinite(scale) || causal < FA_CAUSAL_NONE || causal > FA_CAUSAL_BOTTOM_RIGHT;
}

Problem make_problem(const Geo& g, float scale, int causal, int dtype, int deterministic) {
  Problem pb;
  pb.B = g.B; pb.Hq = g.Hq; pb.Hkv = g.Hkv; pb.Nq = g.Nq; pb.Nkv = g.Nkv; pb.d = g.d;
  pb.NqPad = round_up(g.Nq, kRowPad);
  pb.scale = scale;
  pb.causal = causal != FA_CAUSAL_NONE ? 1 : 0;
  pb.causal_mode = causal;
  pb.cu_q = g.cu_q;
  pb.cu_k = g.cu_k;
  pb.total_q = g.rows_q();
  pb.total_k = g.rows_k();
  pb.st = g.st;
  pb.bias = g.bias;
  pb.bias_st = g.bias_st;
  pb.dbias = g.dbias;
  pb.dbias_st = g.dbias_st;
  pb.bf16 = dtype == FA_BF16 ? 1 : 0;
  pb.deterministic = deterministic ? 1 : 0;
  return pb;
}

int check_ws(void* workspace, size_t bytes, const Geo& g, int deterministic) {
  if (workspace == nullptr) return FA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return FA_ERR_ALIGN;
  if (bytes < ws_bytes(g.B, g.Hq, g.Nq, g.d, deterministic)) return FA_ERR_WORKSPACE;
  return FA_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

// Tensor maps of the Q-like and K-like tensors of a batch.
// A packed batch has one batch index; its (unused) batch stride is given a
// valid value for the tensor map.
Str3 map_strides(Str3 s, const Geo& g, int heads) {
  if (g.cu_q) s.b = s.h * heads;
  return s;
}
int map_q(CUtensorMap* m, const void* p, const Str3& s, int bf, const Geo& g, int box_rows) {
  return make_map(m, p, bf, g.d, g.rows_q(), g.Hq, g.batch(), map_strides(s, g, g.Hq), box_rows);
}
int map_k(CUtensorMap* m, const void* p, const Str3& s, int bf, const Geo& g, int box_rows) {
  return make_map(m, p, bf, g.d, g.rows_k(), g.Hkv, g.batch(), map_strides(s, g, g.Hkv), box_rows);
}

int run_fwd(const Geo& g, const void* q, const void* k, const void* v, void* o, float* lse, float scale, int causal,
            int dtype, cudaStream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  int st = check_geo(g, dtype);
  if (st) return st;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o) || misaligned(lse)) return FA_ERR_ALIGN;
  if (bad_args(scale, causal)) return FA_ERR_ARG;
  FwdArgs a;
  a.pb = make_problem(g, scale, causal, dtype, 1);
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  if ((st = get_encoder())) return st;
  unsigned int* status = nullptr;
  if ((st = status_ptr(&status))) return st;
  unsigned int* call_abort = nullptr;
  unsigned int call_tag = 0;
  if ((st = fwd_abort_slot(&call_abort, &call_tag))) return st;
  CUtensorMap tq, tk, tv;
  const int bf = a.pb.bf16;
  const int kv_rows = g.bias != nullptr ? kFwdBKBias : kFwdBK;
  if ((st = map_q(&tq, q, g.st.q, bf, g, 128))) return st;
  if ((st = map_k(&tk, k, g.st.k, bf, g, kv_rows))) return st;
  if ((st = map_k(&tv, v, g.st.v, bf, g, kv_rows))) return st;
  CUtensorMap tb{};
  if (g.bias != nullptr && (st = make_bias_map(&tb, g.bias, bf, g.Nkv, g.Nq, g.Hq, g.B, g.bias_st, 64, 128)))
    return st;
  return cuda_status(launch_fwd(a, tq, tk, tv, tb, status, call_abort, call_tag, stream));
}

int run_preprocess(const Geo& g, const void* o, const void* dO, const float* lse, int dtype, int deterministic,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!o || !dO || !lse) return FA_ERR_NULL;
  int st = check_geo(g, dtype);
  if (st) return st;
  if (misaligned(o) || misaligned(dO) || misaligned(lse)) return FA_ERR_ALIGN;
  if ((st = check_ws(workspace, workspace_bytes, g, deterministic))) return st;
  unsigned int* status = nullptr;
  if ((st = status_ptr(&status))) return st;
  const Problem pb = make_problem(g, 1.0f, 0, dtype, deterministic);
  const Workspace w = carve(workspace, g.B, g.Hq, g.Nq, g.d, deterministic);
  return cuda_status(launch_preprocess(pb, o, dO, lse, w, status, stream));
}

int run_main(const Geo& g, const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv,
             float scale, int causal, int dtype, int deterministic, void* workspace, size_t workspace_bytes,
             cudaStream_t stream) {
  if (!q || !k || !v || !dO || !dk || !dv) return FA_ERR_NULL;
  int st = check_geo(g, dtype);
  if (st) return st;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(dO) || misaligned(dk) || misaligned(dv))
    return FA_ERR_ALIGN;
  if (bad_args(scale, causal)) return FA_ERR_ARG;
  if ((st = check_ws(workspace, workspace_bytes, g, deterministic))) return st;
  if ((st = get_encoder())) return st;
  MainArgs a;
  a.pb = make_problem(g, scale, causal, dtype, deterministic);
  a.ws = carve(workspace, g.B, g.Hq, g.Nq, g.d, deterministic);
  a.dk = dk;
  a.dv = dv;
  if ((st = status_ptr(&a.status))) return st;
  CUtensorMap tq, tdo, tk, tv;
  const int bf = a.pb.bf16;
  if ((st = map_q(&tq, q, g.st.q, bf, g, 64))) return st;
  if ((st = map_q(&tdo, dO, g.st.dO, bf, g, 64))) return st;
  if ((st = map_k(&tk, k, g.st.k, bf, g, 128))) return st;
  if ((st = map_k(&tv, v, g.st.v, bf, g, 128))) return st;
  CUtensorMap tb{}, tdb{};
  if (g.bias != nullptr && (st = make_bias_map(&tb, g.bias, bf, g.Nkv, g.Nq, g.Hq, g.B, g.bias_st, 128, kMainBM)))
    return st;
  if (g.dbias != nullptr && (st = make_bias_map(&tdb, g.dbias, bf, g.Nkv, g.Nq, g.Hq, g.B, g.dbias_st, 128, 32)))
    return st;
  if (a.pb.dbias != nullptr && a.pb.causal)
    if ((st = cuda_status(launch_dbias_zero(a.pb, a.status, stream)))) return st;
  return cuda_status(launch_bwd_main(a, tq, tdo, tk, tv, tb, tdb, stream));
}

int run_dq(const Geo& g, const void* q, const void* k, const void* v, const void* dO, void* dq, float scale,
           int causal, int dtype, int deterministic, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!dq) return FA_ERR_NULL;
  int st = check_geo(g, dtype);
  if (st) return st;
  if (misaligned(dq)) return FA_ERR_ALIGN;
  if (bad_args(scale, causal)) return FA_ERR_ARG;
  if ((st = check_ws(workspace, workspace_bytes, g, deterministic))) return st;
  DqArgs a;
  a.pb = make_problem(g, scale, causal, dtype, deterministic);
  a.ws = carve(workspace, g.B, g.Hq, g.Nq, g.d, deterministic);
  a.dq = dq;
  if ((st = status_ptr(&a.status))) return st;
  if (!deterministic) return cuda_status(launch_dq_convert(a.pb, a.ws, dq, a.status, stream));
  if (!q || !k || !v || !dO) return FA_ERR_NULL;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(dO)) return FA_ERR_ALIGN;
  if ((st = get_encoder())) return st;
  CUtensorMap tq, tdo, tk, tv;
  const int bf = a.pb.bf16;
  if ((st = map_q(&tq, q, g.st.q, bf, g, 128))) return st;
  if ((st = map_q(&tdo, dO, g.st.dO, bf, g, 128))) return st;
  if ((st = map_k(&tk, k, g.st.k, bf, g, 128))) return st;
  if ((st = map_k(&tv, v, g.st.v, bf, g, 128))) return st;
  return cuda_status(launch_bwd_dq_det(a, tq, tdo, tk, tv, stream));
}

int run_bwd(const Geo& g, const void* q, const void* k, const void* v, const void* o, const void* dO,
            const float* lse, void* dq, void* dk, void* dv, float scale, int causal, int dtype, int deterministic,
            void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
  int st = check_geo(g, dtype);
  if (st) return st;
  if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(o) || misaligned(dO) || misaligned(lse) ||
      misaligned(dq) || misaligned(dk) || misaligned(dv))
    return FA_ERR_ALIGN;
  if (bad_args(scale, causal)) return FA_ERR_ARG;
  if ((st = check_ws(workspace, workspace_bytes, g, deterministic))) return st;
  if ((st = run_preprocess(g, o, dO, lse, dtype, deterministic, workspace, workspace_bytes, stream))) return st;
  if ((st = run_main(g, q, k, v, dO, dk, dv, scale, causal, dtype, deterministic, workspace, workspace_bytes,
                     stream)))
    return st;
  return run_dq(g, q, k, v, dO, dq, scale, causal, dtype, deterministic, workspace, workspace_bytes, stream);
}

Geo packed(int B, int Hq, int Hkv, int total_q, int total_k, int max_q, int max_k, int d, const int* cu_q,
           const int* cu_k) {
  return Geo{B, Hq, Hkv, max_q, max_k, d, cu_q, cu_k, total_q, total_k,
             contiguous_all(Hq, Hkv, total_q, total_k, d)};
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_strerror(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "invalid shape (a size < 1 or above the supported limit)";
    case FA_ERR_HEADDIM: return "head dimension must be a multiple of 8 from 8 to 128";
    case FA_ERR_GQA: return "Hq must be a multiple of Hkv";
    case FA_ERR_ALIGN: return "a pointer is not 16-byte aligned (workspace: 256-byte)";
    case FA_ERR_WORKSPACE: return "workspace missing or smaller than fa_bwd_workspace_size()";
    case FA_ERR_DTYPE: return "dtype must be FA_F16 or FA_BF16";
    case FA_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    case FA_ERR_ARG: return "an argument is out of range";
    case FA_ERR_BOUNDS: return "a kernel's bounds check failed (debug build)";
    default: return "unknown fa_status";
  }
}

size_t fa_bwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int deterministic) {
  if (check_shape(B, Hq, Hkv, Nq, Nkv, d, FA_BF16) != FA_OK) return 0;
  return ws_bytes(B, Hq, Nq, d, deterministic);
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
           int Nkv, int d, float scale, int causal, int dtype, cudaStream_t stream) {
  return run_fwd(dense(B, Hq, Hkv, Nq, Nkv, d), q, k, v, o, lse, scale, causal, dtype, stream);
}

int fa_bwd_preprocess(const void* o, const void* dO, const float* lse, int B, int Hq, int Hkv, int Nq, int Nkv,
                      int d, int dtype, int deterministic, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
  return run_preprocess(dense(B, Hq, Hkv, Nq, Nkv, d), o, dO, lse, dtype, deterministic, workspace, workspace_bytes,
                        stream);
}

int fa_bwd_main(const void* q, const void* k, const void* v, const void* dO, void* dk, void* dv, int B, int Hq,
                int Hkv, int Nq, int Nkv, int d, float scale, int causal, int dtype, int deterministic,
                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return run_main(dense(B, Hq, Hkv, Nq, Nkv, d), q, k, v, dO, dk, dv, scale, causal, dtype, deterministic, workspace,
                  workspace_bytes, stream);
}

int fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO, void* dq, int B, int Hq, int Hkv,
              int Nq, int Nkv, int d, float scale, int causal, int dtype, int deterministic, void* workspace,
              size_t workspace_bytes, cudaStream_t stream) {
  return run_dq(dense(B, Hq, Hkv, Nq, Nkv, d), q, k, v, dO, dq, scale, causal, dtype, deterministic, workspace,
                workspace_bytes, stream);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dq,
           void* dk, void* dv, int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int causal, int dtype,
           int deterministic, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return run_bwd(dense(B, Hq, Hkv, Nq, Nkv, d), q, k, v, o, dO, lse, dq, dk, dv, scale, causal, dtype,
                 deterministic, workspace, workspace_bytes, stream);
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int B, int Hq, int Hkv, int total_q, int total_k, int max_q, int max_k,
                  int d, float scale, int causal, int dtype, cudaStream_t stream) {
  if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_NULL;
  return run_fwd(packed(B, Hq, Hkv, total_q, total_k, max_q, max_k, d, cu_seqlens_q, cu_seqlens_k), q, k, v, o,
                 lse, scale, causal, dtype, stream);
}

size_t fa_bwd_varlen_workspace_size(int B, int Hq, int Hkv, int max_q, int max_k, int d, int deterministic) {
  return fa_bwd_workspace_size(B, Hq, Hkv, max_q, max_k, d, deterministic);
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                  void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq,
                  int Hkv, int total_q, int total_k, int max_q, int max_k, int d, float scale, int causal,
                  int dtype, int deterministic, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_NULL;
  return run_bwd(packed(B, Hq, Hkv, total_q, total_k, max_q, max_k, d, cu_seqlens_q, cu_seqlens_k), q, k, v, o,
                 dO, lse, dq, dk, dv, scale, causal, dtype, deterministic, workspace, workspace_bytes, stream);
}

namespace {
Str3 to_str3(const fa_stride3& s) { return Str3{s.b, s.h, s.n}; }

// Geometry of a strided call: dense (cu_q == NULL) or packed, with the given
// strides or the contiguous ones.
Geo strided_geo(const fa_strides* s, const int* cu_q, const int* cu_k, int B, int Hq, int Hkv, int Nq, int Nkv,
                int total_q, int total_k, int d) {
  Geo g = cu_q ? packed(B, Hq, Hkv, total_q, total_k, Nq, Nkv, d, cu_q, cu_k) : dense(B, Hq, Hkv, Nq, Nkv, d);
  if (cu_q == nullptr && cu_k != nullptr) g.cu_k = cu_k;   // rejected by check_geo
  if (s) {
    g.st.q = to_str3(s->q); g.st.k = to_str3(s->k); g.st.v = to_str3(s->v);
    g.st.o = to_str3(s->o); g.st.dO = to_str3(s->dO); g.st.dq = to_str3(s->dq);
    g.st.dk = to_str3(s->dk); g.st.dv = to_str3(s->dv); g.st.lse = to_str3(s->lse);
  }
  return g;
}

// Adds the bias of an fa_bias description to a geometry.
Geo with_bias(Geo g, const fa_bias* bias) {
  if (bias) {
    g.bias = bias->bias;
    g.bias_st = to_str3(bias->bias_strides);
    g.dbias = bias->dbias;
    g.dbias_st = to_str3(bias->dbias_strides);
  }
  return g;
}
}  // namespace

int fa_fwd_bias(const void* q, const void* k, const void* v, void* o, float* lse, const fa_bias* bias,
                const fa_strides* strides, const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq, int Hkv,
                int Nq, int Nkv, int total_q, int total_k, int d, float scale, int causal, int dtype,
                cudaStream_t stream) {
  if (bias != nullptr && bias->bias == nullptr) return FA_ERR_NULL;
  if (bias != nullptr && bias->dbias != nullptr) return FA_ERR_ARG;   // the forward writes no dBias
  return run_fwd(with_bias(strided_geo(strides, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, Nq, Nkv, total_q, total_k,
                                       d), bias),
                 q, k, v, o, lse, scale, causal, dtype, stream);
}

int fa_bwd_bias(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                void* dq, void* dk, void* dv, const fa_bias* bias, const fa_strides* strides,
                const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq, int Hkv, int Nq, int Nkv,
                int total_q, int total_k, int d, float scale, int causal, int dtype, int deterministic,
                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (bias != nullptr && bias->bias == nullptr) return FA_ERR_NULL;
  return run_bwd(with_bias(strided_geo(strides, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, Nq, Nkv, total_q, total_k,
                                       d), bias),
                 q, k, v, o, dO, lse, dq, dk, dv, scale, causal, dtype, deterministic, workspace, workspace_bytes,
                 stream);
}

int fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse, const fa_strides* strides,
                   const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int Hq, int Hkv, int Nq, int Nkv,
                   int total_q, int total_k, int d, float scale, int causal, int dtype, cudaStream_t stream) {
  return run_fwd(strided_geo(strides, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, Nq, Nkv, total_q, total_k, d), q, k,
                 v, o, lse, scale, causal, dtype, stream);
}

int fa_bwd_strided(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, const fa_strides* strides, const int* cu_seqlens_q,
                   const int* cu_seqlens_k, int B, int Hq, int Hkv, int Nq, int Nkv, int total_q, int total_k, int d,
                   float scale, int causal, int dtype, int deterministic, void* workspace, size_t workspace_bytes,
                   cudaStream_t stream) {
  return run_bwd(strided_geo(strides, cu_seqlens_q, cu_seqlens_k, B, Hq, Hkv, Nq, Nkv, total_q, total_k, d), q, k,
                 v, o, dO, lse, dq, dk, dv, scale, causal, dtype, deterministic, workspace, workspace_bytes, stream);
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
    const int code = static_cast<int>(v >> 16);
    return code == FA_ERR_DEVICE_TIMEOUT || code == FA_ERR_ARG || code == FA_ERR_BOUNDS ? code : FA_ERR_CUDA;
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
