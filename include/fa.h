/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention backward library.
 *
 * What is computed (per batch b and query head h; key/value head
 * h_kv = h / (Hq / Hkv), consecutive query heads share one key/value head):
 *
 *   S = scale * Q K^T, causal: S[i][j] = -inf when j > i + delta, where
 *       delta = 0 (causal = FA_CAUSAL_TOP_LEFT) or Nkv - Nq (FA_CAUSAL_BOTTOM_RIGHT)
 *   L = logsumexp_j S       (natural log of the scaled scores; -inf for a row
 *                            that sees no key, which bottom-right gives the
 *                            first Nq - Nkv rows when Nq > Nkv)
 *   P = exp(S - L) (0 where S = -inf),  O = P V
 *   dV = P^T dO,  dP = dO V^T,  D = rowsum(dO o O),  dS = P o (dP - D)
 *   dQ = scale * dS K,  dK = scale * dS^T Q
 *   dK, dV of a key/value head are summed over the query heads of its group.
 *
 * Sources: "flash_attention_backward.cu" (rustytorch rtx-flash-attention),
 * kernel flash_attention_backward_kernel, blocks "Recompute attention scores",
 * "Apply causal mask", "Compute softmax probabilities from scores and LSE",
 * "Compute dS", "Compute dQ", "Compute dK", "Compute dV" and "Compute row-wise
 * dot product: dO * O"; the sequence-parallel kernel in "Extra transposes cause
 * 8x speedup for sequence-parallel Flash Attention backward" (triton #1806,
 * "Minimal Repro"), which accumulates dQ in an fp32 buffer across KV tiles;
 * GQA as listed in "[Kernel] Flash attention 2" (Liger-Kernel #275, "Details").
 *
 * Layout: contiguous row-major tensors
 *   Q, O, dO, dQ : [B, Hq,  Nq,  d]   16-bit (fp16 or bf16, see fa_dtype)
 *   K, V, dK, dV : [B, Hkv, Nkv, d]   16-bit
 *   L (lse)      : [B, Hq,  Nq]       fp32, natural-log LSE of the scaled scores
 * for every entry point except the packed-batch ones (fa_*_varlen: [H, total,
 * d]), the strided ones (fa_*_strided, fa_*_bias: any batch, head and row
 * strides) and fa_bwd_host (host memory).
 * d: a multiple of 8 from 8 to 128 ("[Kernel] Flash attention 2", "Details":
 * no restriction on the head dimension; 8 keeps every row a whole number of
 * 16-byte pieces, and 128 is the most whose dK and dV accumulators, 128 rows x
 * d fp32 each, leave room in the 512 TMEM columns for the score, dP and dQ
 * tiles).  Other sizes run on the d = 64 or d = 128 kernels, which read the
 * missing columns as zeros: exact, since a zero column adds nothing to Q K^T
 * and produces a zero column of O, dQ, dK, dV, which is not written.
 * Every pointer is a DEVICE pointer on the current device (except for
 * fa_bwd_host), 16-byte aligned.  The caller owns every buffer (inputs,
 * outputs, workspace, staging) and the stream; the library allocates no
 * device memory, keeps no state besides small arrays compiled into it (one
 * status word per device, 256 forward abort words, fa_bwd_noalloc's scratch)
 * and fa_bwd_host's copy and slot streams, and never synchronises inside
 * fa_fwd* / fa_bwd*.  All work is enqueued on `stream` (fa_bwd_host forks
 * from it and joins back into it).
 *
 * Errors: each call validates its arguments first and, on failure, returns a
 * non-zero fa_status WITHOUT launching anything.  FA_ERR_CUDA reports a
 * failed launch (cudaGetLastError).  Device-side waits are bounded.  A wait
 * that runs out does two things:
 *   - it records FA_ERR_DEVICE_TIMEOUT in the device's status word, which
 *     fa_last_device_error() reads and clears; and
 *   - it sets the abort word of its own call, so that the other CTAs of that
 *     call stop waiting and skip their output stores.
 * Each call has its own abort word: fa_bwd* keeps it in the first 256 bytes
 * of its workspace (cleared by fa_bwd_preprocess); fa_fwd* takes the next of
 * 256 slots in the library together with a value that no earlier call on
 * that slot used, and a slot aborts a forward only when it holds that call's
 * value, so nothing is cleared before the kernel.  The status word only
 * reports: no kernel reads it.  A failure left unread
 * therefore never changes the results of later calls, on any stream.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_NULL = 1,            /* a required pointer is NULL                         */
  FA_ERR_SHAPE = 2,           /* B, Hq, Hkv, Nq or Nkv < 1, or above the size limit */
  FA_ERR_HEADDIM = 3,         /* d not a multiple of 8 in [8, 128]                  */
  FA_ERR_GQA = 4,             /* Hq not a multiple of Hkv                           */
  FA_ERR_ALIGN = 5,           /* a pointer is not 16-byte aligned                   */
  FA_ERR_WORKSPACE = 6,       /* workspace NULL or smaller than fa_bwd_workspace_size */
  FA_ERR_DTYPE = 7,           /* dtype not an fa_dtype value                        */
  FA_ERR_CUDA = 8,            /* a CUDA launch or driver call failed                */
  FA_ERR_DEVICE_TIMEOUT = 9,  /* a bounded device-side wait ran out (see fa_last_device_error) */
  FA_ERR_ARG = 10,            /* another argument is out of range (scale not finite, causal unknown, ...) */
  FA_ERR_BOUNDS = 11          /* a kernel's bounds check failed (debug builds with FA_DEBUG_BOUNDS only) */
} fa_status;

typedef enum { FA_F16 = 0, FA_BF16 = 1 } fa_dtype;

/*
 * Values of every entry point's `causal` argument.  The source kernel masks
 * key j for query i when j > i (top-left); "[Kernel] Flash attention 2"
 * (Liger-Kernel #275, "Details") lists causal masking together with different
 * Q and KV lengths without fixing the alignment, so both are offered.  With
 * Nq == Nkv they coincide.  Any other value is FA_ERR_ARG.
 */
typedef enum {
  FA_CAUSAL_NONE = 0,
  FA_CAUSAL_TOP_LEFT = 1,      /* key j masked for query i when j > i             */
  FA_CAUSAL_BOTTOM_RIGHT = 2   /* key j masked for query i when j > i + Nkv - Nq  */
} fa_causal;

/* Largest Nq / Nkv accepted (rows per head). */
#define FA_MAX_SEQ (1 << 24)

/*
 * fa_fwd -- exact attention forward: O = softmax(scale Q K^T [+ causal mask]) V
 * and L = logsumexp of the scaled (masked) scores, natural log.
 * Source: the forward that produces the O and LSE consumed by the backward in
 * flash_attention_backward.cu ("Compute softmax probabilities from scores and
 * LSE"); forward tables in "[Issue]: Backward performance" (ROCm #44).
 * q,k,v: inputs; o: output [B,Hq,Nq,d] (overwritten); lse: output [B,Hq,Nq] fp32.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int causal,
           int dtype, cudaStream_t stream);

/*
 * fa_bwd_workspace_size -- bytes of device workspace fa_bwd needs.
 * Holds the call's abort word (256 bytes), D = rowsum(dO o O) and
 * -L*log2(e) per query row (rows padded to a
 * multiple of 128), plus, when deterministic == 0, the fp32 dQ accumulator
 * [B, Hq, Nq padded, d] of the sequence-parallel scheme (triton #1806,
 * "Minimal Repro": dq is an fp32 buffer that every KV-tile program adds to).
 * Returns 0 when the shape is invalid.
 */
size_t fa_bwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int deterministic);

/*
 * fa_bwd -- full backward: dq, dk, dv (all OVERWRITTEN, not accumulated).
 * Runs fa_bwd_preprocess, fa_bwd_main and fa_bwd_dq in order on `stream`.
 * deterministic == 0: dQ is accumulated with fp32 reductions in the workspace
 *   (summation order not fixed; results may differ in the last bits between runs).
 * deterministic != 0: dQ comes from a separate query-tile-parallel pass with a
 *   fixed summation order; results are bit-identical from run to run.
 * workspace: device buffer of at least fa_bwd_workspace_size(...) bytes,
 *   256-byte aligned; its contents on entry do not matter.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
           const float* lse, void* dq, void* dk, void* dv,
           int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int causal,
           int dtype, int deterministic, void* workspace, size_t workspace_bytes,
           cudaStream_t stream);

/*
 * fa_bwd_preprocess -- step 1 of fa_bwd: D_i = sum_c dO_ic O_ic (fp32), the
 * row-wise dot product the pages precompute (flash_attention_backward.cu,
 * "Compute row-wise dot product: dO * O"; the D input of the Triton kernel in
 * triton #1806), -L*log2(e) per row, and (deterministic == 0) zeroes the fp32
 * dQ accumulator.  It also clears the workspace header: the call's abort word
 * and the work-item counters of the persistent main and deterministic dQ
 * kernels (each launch of those resets its counters when it completes; after a
 * device-side failure, start again from this step).  Writes only the workspace.
 */
int fa_bwd_preprocess(const void* o, const void* dO, const float* lse,
                      int B, int Hq, int Hkv, int Nq, int Nkv, int d, int dtype, int deterministic,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd_main -- step 2 of fa_bwd: the KV-tile-parallel kernel.  Each work
 * item, a (128-row KV tile, key/value head, batch), walks every query tile of
 * every query head of its GQA group (triton #1806, "Minimal Repro": grid over
 * (batch, head, KV block), loop over query blocks), recomputes S and P, and
 * accumulates dV += P^T dO and dK += dS^T Q on the tensor cores; dK, dV are
 * written once.  With deterministic == 0 it also forms dQ_tile = dS K and adds
 * it into the workspace accumulator.  Without a bias the items run on a
 * persistent grid (one CTA per SM, items taken from a counter in the
 * workspace); with one, one CTA per item.  Needs fa_bwd_preprocess first.
 */
int fa_bwd_main(const void* q, const void* k, const void* v, const void* dO,
                void* dk, void* dv,
                int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int causal,
                int dtype, int deterministic, void* workspace, size_t workspace_bytes,
                cudaStream_t stream);

/*
 * fa_bwd_dq -- step 3 of fa_bwd.  deterministic == 0: converts the fp32
 * accumulator to dq = scale * acc in the 16-bit dtype.  deterministic != 0:
 * runs the query-tile-parallel pass (flash_attention_backward.cu's
 * query-block grid with dQ kept on chip, "Compute dQ"; persistent like
 * fa_bwd_main when there is no bias) and writes dq directly.
 * Needs fa_bwd_preprocess (and, for deterministic == 0, fa_bwd_main) first.
 */
int fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO, void* dq,
              int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int causal,
              int dtype, int deterministic, void* workspace, size_t workspace_bytes,
              cudaStream_t stream);

/* Size of the scratch array compiled into the library for fa_bwd_noalloc (64 MiB per GPU). */
#define FA_STATIC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * fa_bwd_noalloc -- fa_bwd for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for callers of
 * this library that have no way to obtain a workspace: for example a plugin
 * inside an inference engine whose host framework owns every device
 * allocation and offers no scratch, or a serving loop that forbids cudaMalloc
 * after start-up because it synchronises the device and fragments the pool.
 * Same arguments and results as fa_bwd, minus the workspace: the scratch is a
 * fixed array of FA_STATIC_SCRATCH_BYTES compiled into the library, which
 * every GPU that loads the library holds until the process exits.  The call
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 * Limit: returns FA_ERR_WORKSPACE, launching nothing, when
 * fa_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d, deterministic) exceeds
 * FA_STATIC_SCRATCH_BYTES (deterministic mode needs 8 bytes per query row,
 * rows padded to 128 per head; atomic mode 8 + 4*64 (d <= 64) or 8 + 4*128 bytes
 * per padded row; plus 256 bytes).  Arguments are checked in fa_bwd's order,
 * so a call with, say, an unknown dtype gets FA_ERR_DTYPE whatever its size.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.  All calls share the one array, and each call rewrites
 * everything it reads from it, so earlier contents never matter; but calls
 * that overlap on the GPU (unordered streams or host threads) race on it.
 */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, void* dq, void* dk, void* dv,
                   int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int causal,
                   int dtype, int deterministic, cudaStream_t stream);

/*
 * Packed variable-length batches.  "[Kernel] Flash attention 2" (Liger-Kernel
 * #275, "Details") supports different Q and KV lengths with no restriction on
 * the sequence length; these entry points take a batch of sequences of
 * different lengths packed along the row axis of every head:
 *   Q, O, dO, dQ : [Hq,  total_q, d]   16-bit
 *   K, V, dK, dV : [Hkv, total_k, d]   16-bit
 *   L (lse)      : [Hq,  total_q]      fp32
 * Sequence b owns rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) of every query
 * head and rows [cu_seqlens_k[b], cu_seqlens_k[b+1]) of every key/value head,
 * and attends only to its own keys; causal alignment (fa_causal) is taken per
 * sequence.  A sequence may be empty; one with queries but no keys gets O = 0,
 * L = -inf, dQ = 0.  Rows not covered by any sequence are left untouched.
 * cu_seqlens_q / cu_seqlens_k: DEVICE int32 arrays of B + 1 offsets (4-byte
 * aligned), starting at 0, non-decreasing, ending at total_q / total_k, each
 * length at most max_q / max_k.  The host cannot read them without a
 * synchronisation, so the kernels check every sequence's offsets before using
 * them: a sequence whose offsets leave [0, total] or exceed the maximum is
 * skipped (nothing of it is read or written) and fa_last_device_error()
 * reports FA_ERR_ARG.  total_q, total_k: 1 .. 2^30; max_q, max_k: 1 .. FA_MAX_SEQ.
 * Workspace: fa_bwd_varlen_workspace_size(), rows padded per (sequence, query
 * head) to a multiple of 128 of max_q.  Other arguments as for fa_fwd / fa_bwd.
 */
int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens_q, const int* cu_seqlens_k,
                  int B, int Hq, int Hkv, int total_q, int total_k, int max_q, int max_k,
                  int d, float scale, int causal, int dtype, cudaStream_t stream);

size_t fa_bwd_varlen_workspace_size(int B, int Hq, int Hkv, int max_q, int max_k, int d, int deterministic);

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO,
                  const float* lse, void* dq, void* dk, void* dv,
                  const int* cu_seqlens_q, const int* cu_seqlens_k,
                  int B, int Hq, int Hkv, int total_q, int total_k, int max_q, int max_k,
                  int d, float scale, int causal, int dtype, int deterministic,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Strided tensors.  The Triton kernel of "Extra transposes cause 8x speedup for
 * sequence-parallel Flash Attention backward" (triton #1806, "Minimal Repro")
 * takes batch, head, row and column strides for every tensor; these entry
 * points take the batch, head and row strides, in ELEMENTS, of every tensor
 * (the d axis must be contiguous), so that e.g. [B, N, H, d] tensors or a
 * token-major packed batch [total, H, d] are used in place.
 * Strides must be positive; those of the 16-bit tensors multiples of 8 (16
 * bytes); a packed batch ignores the batch strides.  Tensors must not overlap.
 * Bad strides: FA_ERR_ARG.
 */
typedef struct {
  long long b, h, n;   /* element strides of the batch, head and row axes */
} fa_stride3;

typedef struct {
  fa_stride3 q, k, v, o, dO, dq, dk, dv;   /* 16-bit tensors */
  fa_stride3 lse;                          /* fp32 L */
} fa_strides;

/*
 * fa_fwd_strided / fa_bwd_strided -- the general forms of fa_fwd / fa_bwd and
 * of their packed-batch variants.  strides: NULL means contiguous ([B, H, N, d]
 * dense, [H, total, d] packed).  cu_seqlens_q == NULL (and cu_seqlens_k ==
 * NULL): a dense batch of B sequences of Nq queries and Nkv keys (total_q,
 * total_k ignored).  Otherwise a packed batch as for fa_fwd_varlen: Nq, Nkv
 * are the longest lengths and the row axes hold total_q / total_k rows.
 * Workspace: fa_bwd_workspace_size(B, Hq, Hkv, Nq, Nkv, d, deterministic).
 */
int fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                   const fa_strides* strides, const int* cu_seqlens_q, const int* cu_seqlens_k,
                   int B, int Hq, int Hkv, int Nq, int Nkv, int total_q, int total_k, int d,
                   float scale, int causal, int dtype, cudaStream_t stream);

int fa_bwd_strided(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, void* dq, void* dk, void* dv,
                   const fa_strides* strides, const int* cu_seqlens_q, const int* cu_seqlens_k,
                   int B, int Hq, int Hkv, int Nq, int Nkv, int total_q, int total_k, int d,
                   float scale, int causal, int dtype, int deterministic,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Additive attention bias.  "[Kernel] Flash attention 2" (Liger-Kernel #275,
 * "Details") supports attention bias and attention masking: the bias is added
 * to the scaled scores before the causal mask,
 *   S = scale * Q K^T + bias,
 * and a boolean mask is the bias -inf at the dropped keys (a row that keeps no
 * key gets O = 0, L = -inf).  The bias enters S with weight 1, so its gradient
 * is dBias = dS = P o (dP - D) of every query head.
 * bias: 16-bit (the dtype of Q), a [B, Hq, Nq, Nkv] view with the key axis
 *   contiguous and element strides bias_strides.b / .h / .n for the batch,
 *   head and query axes; a stride of 0 broadcasts that axis.  Indices are local
 *   to the sequence for packed batches.  Base 16-byte aligned, strides
 *   multiples of 8.
 * dbias (fa_bwd_bias only, may be NULL): 16-bit output [B, Hq, Nq, Nkv] with
 *   positive strides (every row its own), fully overwritten for every query
 *   and key of every sequence (0 where the causal mask drops the key).  A
 *   caller whose bias broadcasts sums dbias over the broadcast axes.
 */
typedef struct {
  const void* bias;
  fa_stride3 bias_strides;
  void* dbias;
  fa_stride3 dbias_strides;
} fa_bias;

/*
 * fa_fwd_bias / fa_bwd_bias -- fa_fwd_strided / fa_bwd_strided with an additive
 * bias (bias == NULL: none; fa_fwd_bias takes no dbias).
 */
int fa_fwd_bias(const void* q, const void* k, const void* v, void* o, float* lse,
                const fa_bias* bias, const fa_strides* strides,
                const int* cu_seqlens_q, const int* cu_seqlens_k,
                int B, int Hq, int Hkv, int Nq, int Nkv, int total_q, int total_k, int d,
                float scale, int causal, int dtype, cudaStream_t stream);

int fa_bwd_bias(const void* q, const void* k, const void* v, const void* o, const void* dO,
                const float* lse, void* dq, void* dk, void* dv,
                const fa_bias* bias, const fa_strides* strides,
                const int* cu_seqlens_q, const int* cu_seqlens_k,
                int B, int Hq, int Hkv, int Nq, int Nkv, int total_q, int total_k, int d,
                float scale, int causal, int dtype, int deterministic,
                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd_host -- fa_bwd for tensors in HOST memory (same layouts, contiguous),
 * with the transfers overlapped with the computation.  The pages have no
 * counterpart; it serves callers whose activations live in host memory (for
 * example offloaded between the forward and the backward).
 *
 * The problem is cut into chunks of `chunk_groups` (batch, kv-head) groups
 * (a group is one key/value head of one sequence with its Hq/Hkv query heads;
 * groups are numbered b*Hkv + hkv, and a run of them is contiguous in every
 * tensor).  Chunks flow through a ring of `slots` slots of the caller's DEVICE
 * staging memory: one copy stream brings chunk inputs in, chunk c computes on
 * the stream of slot c % slots once its inputs are in, and a second copy
 * stream takes dQ, dK, dV out; a slot is refilled once its previous chunk has
 * been copied out.  The copy streams and FA_HOST_MAX_SLOTS slot streams are
 * created by the library once per device.  Results equal fa_bwd's on the same
 * values (dK, dV and deterministic dQ bitwise).
 *
 * The call returns once everything is queued; the work is complete, dq/dk/dv
 * written in host memory, when `stream` reaches this point.  Host buffers
 * should be page-locked (cudaHostAlloc / cudaHostRegister); pageable memory
 * works but serialises the copies.  Small chunks shorten the exposed first
 * copy-in and last copy-out; enough slots keep the copy-in stream from waiting
 * (with the link slower than the computation, 3-4 slots suffice).
 *
 * chunk_groups in [1, B*Hkv], slots in [1, FA_HOST_MAX_SLOTS] (FA_ERR_SHAPE
 * otherwise).  staging: >= fa_bwd_host_staging_size(...) bytes (0 for invalid
 * arguments), 256-byte aligned (FA_ERR_ALIGN), not used by anything else until
 * `stream` passes the call (FA_ERR_WORKSPACE if NULL or too small).  Every
 * argument error (shape, dtype, scale, causal, staging) is returned before
 * anything is queued.  If a copy or launch fails after work has been queued
 * (FA_ERR_CUDA), the call first waits for everything it queued on its copy
 * and slot streams to finish, so no transfer into or out of the caller's
 * buffers is still running when it returns.
 */
#define FA_HOST_MAX_SLOTS 8

size_t fa_bwd_host_staging_size(int B, int Hq, int Hkv, int Nq, int Nkv, int d, int deterministic,
                                int chunk_groups, int slots);

int fa_bwd_host(const void* q, const void* k, const void* v, const void* o, const void* dO,
                const float* lse, void* dq, void* dk, void* dv,
                int B, int Hq, int Hkv, int Nq, int Nkv, int d, float scale, int causal,
                int dtype, int deterministic, int chunk_groups, int slots,
                void* staging, size_t staging_bytes, cudaStream_t stream);

/* Human-readable name of an fa_status value (static string, never NULL). */
const char* fa_strerror(int status);

/*
 * fa_last_device_error -- synchronises `stream`, then reads and clears the
 * current device's status word.  Returns FA_ERR_DEVICE_TIMEOUT if any bounded
 * wait in a kernel ran out since the word was last read, FA_ERR_ARG if a
 * kernel skipped a packed-batch sequence with out-of-range offsets,
 * FA_ERR_BOUNDS if a bounds check of the debug build failed,
 * FA_ERR_CUDA if the sync failed, FA_OK otherwise.
 * The word is one per device, not per stream: it holds the first failure of
 * any call on the device since the last read, and work on other streams that
 * has not finished yet may still set it after this returns.  Reading it is
 * optional; kernels never act on it (see "Errors" above).
 */
int fa_last_device_error(cudaStream_t stream);

/*
 * Debug build.  The library compiled with -DFA_DEBUG_BOUNDS (python -m
 * attn_bwd_gb300.build --debug-bounds: libattn_bwd_gb300_bounds.so) has the
 * same entry points; its kernels check every TMA tile coordinate, bulk copy
 * range and global store or reduction index against the extents of the
 * tensors they were given.  A failed check is recorded like a timeout
 * (fa_last_device_error() returns FA_ERR_BOUNDS), aborts the call, and the
 * access is skipped, so nothing outside a tensor is touched.  The normal
 * build compiles no checks.
 */

/*
 * fa_selftest_wait_timeout -- launches one CTA that waits on a barrier no one
 * arrives on, with a wait bound of `timeout_us` microseconds (1..5,000,000).
 * The kernel gives up, records FA_ERR_DEVICE_TIMEOUT and exits cleanly; the
 * caller then sees it through fa_last_device_error().  This exercises the
 * failure-detection path without faulting or hanging the GPU.
 */
int fa_selftest_wait_timeout(int timeout_us, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
