/*
 * fa.h -- C ABI of libfa: fused FlashAttention forward (plain, causal,
 * grouped-query, split-KV), its backward, and split-KV decode (per-head and
 * grouped-query) for one NVIDIA GB300 GPU (sm_103a).
 *
 * Sources (web pages, cited by title and section):
 *   [T1] "FlashAttention 简化版：Tiling + Online Softmax" (forceinjection.github.io)
 *   [T2] "Flash Attention 代码填空 (Level 2-3)" (boots-coder.github.io, LLM-101-CN)
 *   [T3] "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com)
 *   [T4] "从零手写 FlashAttention（PyTorch实现 + 原理推导）" (mokono.cn)
 *
 * Conventions shared by every entry point
 *   - Tensors are contiguous row-major [B, H, N, d] (d fastest).  Decode q and
 *     o are [B, H, d] (one query per head).  LSE is fp32 [B, H, Nq].
 *   - Every tensor pointer is a DEVICE pointer owned by the caller (except the
 *     tensors of fa_fwd_host, which are host pointers); device base addresses
 *     must be 16-byte aligned.  The library never frees caller memory and
 *     keeps no pointer after a call returns.
 *   - Calls are asynchronous: they validate, enqueue kernels on `stream`
 *     (NULL = the legacy default stream) and return.  A return of FA_OK means
 *     the work was enqueued; timeouts detected on the device are reported
 *     later by fa_check_device_error().
 *   - Arguments are validated before anything is launched; on any error
 *     nothing is enqueued.  No call prints or exits.
 *   - Calls are reentrant and may be made from several host threads.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared here so this header needs no CUDA header. */
struct CUstream_st;
typedef struct CUstream_st* fa_stream_t;

typedef enum { FA_FP32 = 0, FA_BF16 = 1 } fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* NULL or misaligned pointer, non-positive size, overflow, bad scale */
    FA_ERR_UNSUPPORTED = 2, /* valid but unsupported: head dim not 64/128, dtype, device not sm_103 */
    FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, allocation, tensor map) */
    FA_ERR_TIMEOUT = 4      /* a device-side wait ran past its limit (from fa_check_device_error) */
} fa_status;

/*
 * fa_fwd -- exact attention O = softmax(Q K^T * scale) V, computed tile by
 * tile with the online-softmax recurrence so the Nq x Nk score matrix never
 * reaches device memory ([T1] §2.3, §3.1; [T3] attn_row_1pass).  For each
 * query row the running maximum m, running sum l and unnormalised O are
 * updated per key tile with correction alpha = exp(m_old - m_new); O is
 * divided by l once at the end ([T3] demo 3, deferred normalisation).
 *
 *   q   [B, H, Nq, d]  in dtype       k, v [B, H, Nk, d] in dtype
 *   o   [B, H, Nq, d]  out, dtype     lse  [B, H, Nq] fp32 out, or NULL
 *   lse = m + ln(l) in natural log, in units of scaled scores ([T3] demo 2).
 *   dtype FA_BF16: bf16 operands, fp32 accumulation, P rounded to bf16 for P V.
 *   dtype FA_FP32: fp32 operands multiplied as TF32, P kept at TF32.  A prep
 *     pass first writes tf32-rounded (nearest) copies of Q and K and a
 *     key-major tf32 copy of V (tf32 tensor-core operands must be K-major).
 *   When the query tiles cannot fill the GPU (small B*H*Nq) the keys are also
 *   split across CTAs and merged (see fa_fwd_ex).  Any workspace these need
 *   (fa_fwd_workspace_bytes) is taken stream-ordered (cudaMallocAsync /
 *   cudaFreeAsync on `stream`).
 *   d must be 64 or 128; Nq, Nk >= 1 (ragged tails are masked); B, H >= 1;
 *   scale must be finite (1/sqrt(d) is the usual value; 1 reproduces [T4]-style
 *   unscaled scores).  Returns FA_OK or an fa_status code.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int Nq, int Nk, int d, float scale, int dtype,
           fa_stream_t stream);

/*
 * fa_fwd_ex -- fa_fwd with every option exposed.  fa_fwd(...) is
 * fa_fwd_ex(..., Hkv = H, causal = 0, kv_splits = 0, workspace = NULL, 0, stream).
 *   Hkv        key/value heads per batch (grouped-query attention): k and v are
 *              [B, Hkv, Nk, d]; query head h reads key/value head h / (H / Hkv).
 *              H must be a multiple of Hkv (Hkv = H: plain multi-head).
 *   causal     1 = causal mask aligned to the bottom-right corner: query row i
 *              sees keys 0 .. i + (Nk - Nq), so the last query sees every key
 *              and Nq == Nk gives the usual lower triangle ([T1] §7 names the
 *              extension).  Requires Nq <= Nk (FA_ERR_INVALID_ARG otherwise).
 *              Key tiles above the diagonal are skipped, not just masked.
 *   kv_splits  0 = automatic; 1 = one pass over all keys per query tile;
 *              n > 1 = the keys are cut into n ranges handled by separate CTAs,
 *              each writing an fp32 partial state (m, l, unnormalised O) that a
 *              merge kernel combines ([T3] demo 2, split-KV / flash-decoding
 *              applied to every query row).  Automatic splitting is used only
 *              when the query tiles alone cannot fill the GPU.  n may not exceed
 *              the number of key tiles (FA_ERR_INVALID_ARG).
 *              Automatic mode also shortens a short last wave (bf16, d = 64, no
 *              mask): when the CTAs of 256 query rows do not fill whole waves of
 *              two per SM and the rest is at most one per SM, the rows of that
 *              rest go to CTAs of 128 rows whose two halves of the keys run side
 *              by side and merge inside the CTA ([T3] demo 2).  No workspace; the
 *              result depends only on the shape and the GPU's SM count.
 *              kv_splits = 1 keeps every CTA on the whole key range.
 *   workspace  device buffer of at least fa_fwd_workspace_bytes(...) bytes,
 *              16-byte aligned, or NULL to allocate it stream-ordered.  Needed
 *              by the fp32 path (rounded / transposed operand copies) and by
 *              split runs; a bf16 call with one split needs none.
 */
int fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
              int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int dtype,
              int causal, int kv_splits, void* workspace, size_t workspace_bytes,
              fa_stream_t stream);

/* Bytes of workspace fa_fwd_ex needs for these arguments (kv_splits = 0 asks the
 * current device's SM count); 0 when none is needed or the arguments are invalid. */
size_t fa_fwd_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d, int dtype,
                              int causal, int kv_splits);

/*
 * fa_fwd_host -- fa_fwd_ex (kv_splits = 0) on HOST-resident tensors: the library
 * copies q, k, v to the device, computes, and copies o and lse back, in chunks
 * of whole key/value heads (about one wave of CTAs each) so that the
 * copies of one chunk overlap the compute of the previous one (copy-in and
 * copy-out on two internal streams, compute on `stream`, ordered by events).  The
 * exact attention computed is fa_fwd_ex's.
 *   q, k, v, o, lse   HOST pointers, same shapes and dtypes as fa_fwd_ex; lse may
 *                     be NULL.  Page-locked (pinned) memory is needed for the
 *                     copies to overlap; pageable memory works but serialises.
 *   workspace         device buffer of at least fa_fwd_host_workspace_bytes(...)
 *                     bytes (16-byte aligned) that receives the device copies, or
 *                     NULL to allocate it stream-ordered on `stream`.
 * Asynchronous: o and lse hold the result once `stream` has completed the work
 * enqueued up to this call (the call makes `stream` wait for the last copy out).
 * Calls on one device are serialised on the host while they enqueue.  Returns
 * FA_OK or an fa_status code.
 */
int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int dtype,
                int causal, void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Bytes of device workspace fa_fwd_host needs (0 for invalid arguments). */
size_t fa_fwd_host_workspace_bytes(int B, int H, int Hkv, int Nq, int Nk, int d, int dtype,
                                   int causal);

/*
 * fa_bwd -- gradients of exact attention (bf16 or fp32 tensors).
 * Given the forward's inputs, its output O and natural-log LSE, and dO (the
 * gradient of a loss with respect to O), writes
 *   dV = P^T dO, dQ = scale dS K, dK = scale dS^T Q, with P = exp(scale Q K^T - LSE)
 *   recomputed block by block from the saved LSE ("Flash Attention 代码填空
 *   (Level 2-3)", Exercise 5: the forward keeps O and the row statistics, the
 *   backward rebuilds P_ij and accumulates dV_j += P_ij^T dO_i), dP = dO V^T and
 *   dS = P * (dP - D), D_i = sum_c dO_ic O_ic (chain rule through the softmax).
 *   q, o, dout, dq  [B, H, Nq, d] in dtype   k, v, dk, dv [B, Hkv, Nk, d] in dtype
 *   lse             [B, H, Nq] fp32 in: as written by fa_fwd / fa_fwd_ex
 *   Hkv, causal     as in fa_fwd_ex; with Hkv < H, dk and dv sum over the query
 *                   heads that share a key/value head.
 *   dtype           FA_BF16: bf16 operands on the tensor cores, fp32 accumulation,
 *                   P and dS rounded to bf16 for their products.
 *                   FA_FP32: every product and sum in fp32 on the CUDA cores (the
 *                   tensor cores would round the operands to tf32).  d 64 or 128.
 *   workspace       device buffer of at least fa_bwd_workspace_bytes(B, H, Nq, d)
 *                   bytes (16-byte aligned) for D and the rescaled LSE, or NULL
 *                   to allocate it stream-ordered on `stream`.
 * No atomics: every gradient element is written once, by one CTA, so repeated
 * calls give bit-identical results.  Inputs are read only; outputs are fully
 * overwritten.  Returns FA_OK or an fa_status code; argument errors are
 * reported before anything is launched.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int Hkv,
           int Nq, int Nk, int d, float scale, int dtype, int causal,
           void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Bytes of workspace fa_bwd needs (0 for invalid arguments). */
size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int d);

/*
 * fa_decode_splitkv -- attention of one bf16 query per head over Nk keys,
 * split into `splits` chunks of ceil(Nk/splits) keys processed in parallel
 * (flash-decoding); each chunk yields a partial state (m, l, o) with o
 * unnormalised, and a second kernel merges the states ([T3] demo 2: the merge
 * is associative and commutative) and writes O = o / l as bf16.
 *
 *   q [B, H, d] bf16, k/v [B, H, Nk, d] bf16, o [B, H, d] bf16 out.
 *   scale is fixed at 1/sqrt(d).  1 <= splits <= Nk; d in {64, 128}.
 *   The fp32 workspace for the partial states is taken stream-ordered
 *   (cudaMallocAsync / cudaFreeAsync on `stream`).
 */
int fa_decode_splitkv(const void* q, const void* k, const void* v, void* o,
                      int B, int H, int Nk, int d, int splits,
                      fa_stream_t stream);

/*
 * fa_decode_splitkv_ex -- fa_decode_splitkv with every option exposed.
 *   scale        finite score scale.
 *   workspace    device buffer of at least fa_decode_workspace_bytes(B, H, d,
 *                splits) bytes, 16-byte aligned; NULL = allocate stream-ordered.
 *   merge_order  device int32 [splits], a permutation of 0..splits-1 giving the
 *                order in which chunk states are accumulated by the merge; NULL
 *                = index order.  The result is the same up to rounding for
 *                every order ([T3] demo 2).  Entries are validated on the
 *                device; a non-permutation makes the merge write NaN outputs.
 *   lse          fp32 [B, H] out (natural log, scaled-score units), or NULL.
 */
int fa_decode_splitkv_ex(const void* q, const void* k, const void* v, void* o,
                         int B, int H, int Nk, int d, int splits, float scale,
                         void* workspace, size_t workspace_bytes,
                         const int* merge_order, float* lse, fa_stream_t stream);

/* Bytes of fp32 partial-state workspace fa_decode_splitkv_ex (and _gqa) needs; 0 on bad arguments. */
size_t fa_decode_workspace_bytes(int B, int H, int d, int splits);

/*
 * fa_decode_splitkv_gqa -- split-KV decode where Hkv key/value heads serve H
 * query heads ("FlashAttention 简化版：Tiling + Online Softmax" §7 names
 * MQA/GQA): query head h reads key/value head h / (H / Hkv).  Each chunk of
 * each key/value head is read from device memory once for all the query heads
 * of its group; the chunk states and their merge are those of
 * fa_decode_splitkv_ex ([T3] demo 2), one state per (query head, chunk).
 *   q [B, H, d] bf16, k/v [B, Hkv, Nk, d] bf16, o [B, H, d] bf16 out.
 *   H / Hkv must be 1, 2, 4 or a multiple of 8 (FA_ERR_UNSUPPORTED otherwise);
 *   H % Hkv != 0 is FA_ERR_INVALID_ARG.  Other arguments as in
 *   fa_decode_splitkv_ex; the workspace size is fa_decode_workspace_bytes(B, H,
 *   d, splits).
 */
int fa_decode_splitkv_gqa(const void* q, const void* k, const void* v, void* o,
                          int B, int H, int Hkv, int Nk, int d, int splits, float scale,
                          void* workspace, size_t workspace_bytes,
                          const int* merge_order, float* lse, fa_stream_t stream);

/* Size of the fixed device scratch array behind fa_decode_splitkv_noalloc. */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/*
 * fa_decode_splitkv_noalloc -- fa_decode_splitkv for callers that cannot
 * allocate device memory during a call (for example serving processes that
 * reserve nearly all device memory up front and forbid later allocations, or
 * whose memory manager must own every allocation; cudaMalloc may also block
 * on the device).  The pages have no counterpart: this is a deployment
 * variant of the same split and merge kernels.
 *
 *   Arguments, layouts and results are those of fa_decode_splitkv (bf16,
 *   scale 1/sqrt(d)).  The partial states live in a fixed array of
 *   FA_DECODE_NOALLOC_SCRATCH_BYTES inside the library's device image, which
 *   every GPU that loads the library holds until the process exits.  The call
 *   allocates and frees nothing.
 *   - FA_ERR_UNSUPPORTED if fa_decode_workspace_bytes(B, H, d, splits) exceeds
 *     FA_DECODE_NOALLOC_SCRATCH_BYTES, or if the current device is not an
 *     sm_103 GPU (nothing is launched in either case).
 *   - All calls share the array: calls whose kernels may overlap on the GPU
 *     (unordered streams) race and must be ordered by the caller.  The array
 *     keeps the previous call's contents; nothing needs clearing, since every
 *     partial state is written before it is read.
 *   - The first call on each device looks up the array's address
 *     (cudaGetSymbolAddress, with that device current); make it before any
 *     stream capture.
 */
int fa_decode_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                              int B, int H, int Nk, int d, int splits,
                              fa_stream_t stream);

/*
 * fa_check_device_error -- reads and clears the library's device error word
 * on the current device (synchronises that device).  Returns FA_OK, or
 * FA_ERR_TIMEOUT if a kernel gave up on a wait since the last check (its
 * outputs are then undefined), or FA_ERR_CUDA if the read itself failed.
 */
int fa_check_device_error(void);

/* Static, human-readable name of a status code. */
const char* fa_status_string(int status);

/*
 * fa_last_cuda_error -- the CUDA error behind the calling host thread's last
 * FA_ERR_CUDA (a cudaError_t value, or 100000 + a CUresult from tensor-map
 * encoding); 0 if none.  fa_last_cuda_error_string gives its static text.
 */
int fa_last_cuda_error(void);
const char* fa_last_cuda_error_string(void);

/*
 * fa_debug_set_fault -- TEST ONLY.  Arms a host-side fault for the next
 * fa_fwd / fa_fwd_ex or fa_bwd call on this process (whichever comes first):
 * mode 1 makes the load warp of the forward kernel skip its first key-tile
 * copy, or the load warp of the backward's dK/dV kernel skip its key/value
 * copy (and the expected-byte count), so the consumers' bounded waits run
 * out, the kernel abandons its work, records FA_ERR_TIMEOUT and returns.
 * An fp32 fa_bwd call disarms it without effect (its kernels have no waits).
 * mode 0 disarms.  Returns FA_OK or FA_ERR_INVALID_ARG.
 */
int fa_debug_set_fault(int mode);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
