/*
 * fa_api.h -- libfa_b200: FlashAttention forward pass on one GB300 (sm_103a).
 *
 * C ABI (extern "C"), plain pointers and sizes.  The library computes
 *
 *     O   = softmax(scale * Q K^T  [+ causal mask]) V
 *     lse = log(sum_j exp(scale * Q K^T)_ij)            (natural log, per row)
 *
 * tile by tile with online-softmax rescaling: the S = QK^T and P = softmax(S)
 * matrices never reach device memory.  The operation is the reference
 * attention of "ops-transformer FlashAttention build and tuning" (section 4.3,
 * compute_reference_attention: scaled QK^T, triu(diagonal=1) filled with -inf
 * when causal, softmax, times V); the same page (section 1.2) describes the
 * FlashAttention-2 form used here -- Q blocks in the outer loop, K/V blocks
 * streamed in the inner loop, online normalisation of the softmax.  The
 * argument list mirrors the torch_npu entry point traced on the page
 * "npu_flash_attention, from ATen down to the Cube unit" (the
 * npu_flash_attention(q, k, v, head_num, input_layout, scale, keep_prob) call):
 * head count, layout string BNSD/BSND and scale become B, H, S_q, S_kv, D,
 * fa_layout_t and `scale`; keep_prob is fixed at 1.0 (no dropout).
 */
#ifndef FA_API_H
#define FA_API_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Tensor layouts.  Both are dense and contiguous, innermost dimension last:
 *   FA_LAYOUT_BNSD: [B, H, S, D]   (batch, heads, sequence, head dim)
 *   FA_LAYOUT_BSND: [B, S, H, D]   (the pages' [batch, seq, heads*head_dim])  */
typedef enum { FA_LAYOUT_BNSD = 0, FA_LAYOUT_BSND = 1 } fa_layout_t;

/* Element types of Q, K and V.
 *   FA_DTYPE_F16      IEEE binary16; O is binary16.
 *   FA_DTYPE_BF16     bfloat16; O is bfloat16.
 *   FA_DTYPE_FP8E4M3  OCP FP8 E4M3 ("fn": max 448, no inf) with one fp32 descale
 *                     per tensor (real value = code * descale); O is bfloat16.  */
typedef enum { FA_DTYPE_F16 = 0, FA_DTYPE_BF16 = 1, FA_DTYPE_FP8E4M3 = 2 } fa_dtype_t;

/* Status codes.  Errors are returned, never thrown or trapped. */
typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,    /* null pointer, size < 1, non-finite scale,
                                descale given for a 16-bit dtype, bad enum              */
  FA_ERR_UNSUPPORTED = 2,    /* D not in {64, 128}, or a size past the library's limits  */
  FA_ERR_MISALIGNED = 3,     /* a tensor pointer not 16-byte aligned (TMA requirement)   */
  FA_ERR_CUDA = 4,           /* a CUDA runtime/driver call or the launch failed          */
  FA_ERR_DEVICE_TIMEOUT = 5  /* a bounded device-side wait expired (kernel gave up)      */
} fa_status_t;

/*
 * fa_fwd -- one FlashAttention forward pass, asynchronous on `stream`.
 *
 * q    device, [B,H,S_q,D] or [B,S_q,H,D] per `layout`, element type `dtype`.
 * k, v device, same layout with S_kv rows, element type `dtype`.  K and V get
 *      separate descriptors (the Hygon retrospective, defect 13, is a backward
 *      kernel that read V with K's stride).
 * o    device, same layout and shape as q; element type: f16 for F16, bf16 for
 *      BF16 and FP8E4M3.  Only rows < S_q are written.
 * lse  device, fp32 [B, H, S_q] contiguous in every layout, natural log of the
 *      row's softmax denominator including `scale` (and the descales).
 * B, H, S_q, S_kv, D   sizes; all >= 1, D in {64, 128}.  Offsets are 64-bit:
 *      a single tensor may exceed 4 GB (the Hygon retrospective, defect 1).
 * scale  finite, of either sign (the reference attention of the Ascend page,
 *      section 4.3, holds for any real scale); multiplies Q K^T before the
 *      softmax (commonly D^-0.5).  For a negative scale the tensor cores
 *      compute -Q K^T (the products' negate-B bit) and the softmax works with
 *      |scale|, so that a row's maximum of the scores it sees is that of the
 *      scaled scores either way.
 * layout FA_LAYOUT_BNSD or FA_LAYOUT_BSND (o follows q's layout).
 * causal 0: every key visible.  Non-zero: query row i sees key j only if j <= i
 *      (top-left aligned, the verifier's triu(diagonal=1) mask; with S_q == S_kv
 *      this is the usual lower-triangular mask).
 * dtype  see fa_dtype_t.
 * descale_q/k/v  FP8 only: device pointers to one fp32 each, or NULL for 1.0.
 *      Must all be NULL for the 16-bit dtypes.
 * stream the CUDA stream to launch on (0 = legacy default stream).
 *
 * Pointers q, k, v, o must be 16-byte aligned; lse 4-byte aligned.  The caller
 * owns every buffer; the library allocates nothing per call and keeps no
 * per-call state.  Inputs may be NaN-poisoned past their last valid row: no
 * element outside [0, S) is read.  The checks above run on the host before
 * any launch and return an error without touching the device.
 * Returns FA_OK once the kernel is enqueued; FA_ERR_CUDA if a CUDA call or
 * the launch fails.  A bounded device-side wait that expires sets the
 * library's device error word; fa_last_device_error() reports it.
 * Stream order holds as for any launch.  The forward kernels are launched
 * with programmatic stream serialization: one may start its prologue on idle
 * SMs while the kernel before it on the stream still runs, but reads and
 * writes no global memory until that kernel has completed.
 */
fa_status_t fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                   int64_t B, int64_t H, int64_t S_q, int64_t S_kv, int64_t D, float scale,
                   fa_layout_t layout, int causal, fa_dtype_t dtype, const float* descale_q,
                   const float* descale_k, const float* descale_v, cudaStream_t stream);

/*
 * fa_fwd_gqa -- the same forward pass with grouped-query attention: q and o
 * have H heads, k and v have H_kv heads, H a multiple of H_kv.  With
 * ngroups = H / H_kv, query head h attends with key/value head h / ngroups:
 * the query heads are taken in their own flat order, i.e. q viewed as
 * [.., H_kv, ngroups, D] -- no regrouping or transposition of q by the
 * caller.  (The Hygon retrospective, defect 12, is a GQA bug caused by glue
 * code and kernel disagreeing on exactly this head order.)  lse is
 * [B, H, S_q].  Every other argument, check and status is as for fa_fwd;
 * additionally H_kv < 1 or H % H_kv != 0 gives FA_ERR_INVALID_ARG.
 * fa_fwd(...) is fa_fwd_gqa(...) with H_kv = H.
 */
fa_status_t fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                       int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv, int64_t D,
                       float scale, fa_layout_t layout, int causal, fa_dtype_t dtype,
                       const float* descale_q, const float* descale_k, const float* descale_v,
                       cudaStream_t stream);

/*
 * Split-KV ("flash-decoding") forward pass, for problems whose
 * batch x heads x query tiles cannot fill the GPU (few heads, short queries,
 * long keys).  Each query tile's keys are cut into n_splits chunks processed
 * in parallel; every chunk writes its normalised fp32 partial O and partial
 * log-sum-exp to `workspace`, and a second kernel merges them:
 *     lse = log sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s.
 * This is the partition-and-reduce of the paged-decode kernels in the Hygon
 * retrospective (defect 7: per-partition exp_sums / max_logits, then a reduce
 * kernel); the result is the same attention as fa_fwd_gqa.
 *
 * fa_fwd_splitkv_plan -- picks n_splits for the current device: the count
 *   (1..32, at least two 128-key blocks per split) that minimises waves of
 *   work items x (blocks per item + a fixed cost of about three blocks), so
 *   1 when the problem already fills the GPU; and the workspace it needs
 *   (0 when n_splits == 1).  Host only; FA_ERR_INVALID_ARG on bad sizes or
 *   NULL outputs, FA_ERR_CUDA if the device cannot be queried.
 *
 * fa_fwd_splitkv -- arguments as fa_fwd_gqa, plus n_splits (1..32; 1 runs
 *   fa_fwd_gqa and ignores the workspace) and a caller-owned device
 *   workspace of at least the planned bytes, 256-byte aligned (fp32 partial
 *   O [n_splits, B, H, S_q, D], then fp32 partial lse [n_splits, B, H, S_q]).
 *   FA_ERR_INVALID_ARG: n_splits < 1, workspace NULL or too small;
 *   FA_ERR_MISALIGNED: workspace not 256-byte aligned; FA_ERR_UNSUPPORTED:
 *   n_splits > 32.  Two launches on `stream`; the workspace is read and
 *   written by both, so calls sharing one workspace must not overlap.
 */
fa_status_t fa_fwd_splitkv_plan(int64_t B, int64_t H, int64_t S_q, int64_t S_kv, int64_t D,
                                int* n_splits, size_t* workspace_bytes);

fa_status_t fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                           int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv,
                           int64_t D, float scale, fa_layout_t layout, int causal,
                           fa_dtype_t dtype, const float* descale_q, const float* descale_k,
                           const float* descale_v, int n_splits, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv without a caller workspace.  The
 * attention pages have no counterpart to this call; it is a convenience of
 * this library.
 *
 * Who needs it: callers that may not allocate device memory where they run
 * attention and have no spare buffer to hand over -- code running under a
 * memory budget fixed up front, code called back from inside a memory
 * allocator, or a runtime whose hot path must not make the device-wide
 * synchronising calls that cudaMalloc / cudaFree can imply.  The library
 * itself never allocates here: the partials go to a fixed buffer of
 * FA_NOALLOC_SCRATCH_BYTES bytes that is part of the library's device image
 * (a file-scope __device__ array, one copy per device).
 *
 * Arguments, checks and statuses as fa_fwd_splitkv, without workspace and
 * workspace_bytes: its host checks run first, then the capacity check below.
 * n_splits = 1 uses no scratch at all.
 *   Limit: the workspace fa_fwd_splitkv would need for these B, H, S_q, D
 *   and n_splits (fp32 partial O and lse, 4 * n_splits * B * H * S_q *
 *   (D + 1) bytes plus alignment) must fit in FA_NOALLOC_SCRATCH_BYTES;
 *   otherwise FA_ERR_UNSUPPORTED, before any CUDA call (use fa_fwd_splitkv
 *   with your own workspace, or fewer splits).
 *   Zeroing: none needed; every partial the merge reads is written earlier
 *   in the same call.
 *   First call on a device: looks up the buffer's device address with that
 *   device current (cudaGetSymbolAddress) and caches it for the calling
 *   thread's current context; a call in another context (after a device
 *   reset, or from a caller that switched contexts) looks it up again.
 *   FA_ERR_CUDA if the lookup fails.  If the calls are to be made while a stream is being
 *   captured, make one call on each device before capture begins, so that
 *   this setup happens outside the capture.
 *   Overlap: all callers on a device share the one buffer.  Two calls whose
 *   execution can overlap on the same device (different streams, or host
 *   threads with no ordering between their launches) race on it and may
 *   return wrong results; order them on one stream or with events.
 */
#define FA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

fa_status_t fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                   float* lse, int64_t B, int64_t H, int64_t H_kv, int64_t S_q,
                                   int64_t S_kv, int64_t D, float scale, fa_layout_t layout,
                                   int causal, fa_dtype_t dtype, const float* descale_q,
                                   const float* descale_k, const float* descale_v, int n_splits,
                                   cudaStream_t stream);

/*
 * Variable-length sequences and paged K/V (forward).
 *
 * Packed queries: q and o are [total_q, H, D] (o in the output dtype), the
 * queries of sequence s are rows [cu_seqlens_q[s], cu_seqlens_q[s+1]); lse
 * is fp32 [H, total_q].  Each sequence is attended on its own, as the dense
 * call would on a [1, S_q, H, D] problem (query head h reads key/value head
 * h / (H / H_kv)).  cu_seqlens_q (and cu_seqlens_k, seqused_k,
 * block_table) are device int32 arrays read by the kernel; the host cannot
 * check them.  Offsets outside [0, total] or lengths that do not fit are
 * clamped so that nothing outside o and lse is ever written.
 *
 * causal: 0 none; FA_CAUSAL_TOP_LEFT (1): query i sees key j iff j <= i (the
 * dense call's mask); FA_CAUSAL_BOTTOM_RIGHT (2): iff j <= i + S_kv - S_q,
 * i.e. the queries are the last S_q positions of the key sequence (prefill
 * after a cached prefix, decode).  A query row that sees no key gets O = 0
 * and lse = -inf.
 *
 * max_seqlen_q: at least every sequence's query length (rows past it are not
 * computed); it sizes the launch.  total_q = 0 returns FA_OK at once.
 *
 * fa_fwd_varlen -- contiguous packed K/V: k and v are [total_k, H_kv, D], the
 *   keys of sequence s are rows [cu_seqlens_k[s], cu_seqlens_k[s+1]).
 *
 * fa_fwd_paged -- K/V in a paged cache (the PagedAttention scheme of the
 *   Hygon retrospective, defect 11): k_cache and v_cache are [num_pages,
 *   page_size, H_kv, D]; sequence s has seqused_k[s] keys and its key j is row
 *   j % page_size of page block_table[s * max_pages_per_seq + j / page_size].
 *   page_size: 16, 32, 64 or 128, or a multiple of 128 (else
 *   FA_ERR_UNSUPPORTED); a 128-key tile spanning several pages is fetched page
 *   by page, never as if the pages were adjacent.  Page ids outside
 *   [0, num_pages) read as zeros.
 *
 * Statuses as fa_fwd_gqa (dtype, D, alignment, descales), plus
 * FA_ERR_INVALID_ARG for NULL arrays, n_seqs < 1, total_q < 0,
 * max_seqlen_q < 1, causal outside {0, 1, 2} or paging sizes < 1;
 * FA_ERR_MISALIGNED for the int32 arrays off 4 bytes.  One launch on
 * `stream`; the library allocates nothing.
 */
#define FA_CAUSAL_NONE 0
#define FA_CAUSAL_TOP_LEFT 1
#define FA_CAUSAL_BOTTOM_RIGHT 2

fa_status_t fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                          int64_t n_seqs, int64_t total_q, int64_t total_k, int64_t max_seqlen_q,
                          int64_t H, int64_t H_kv, int64_t D, float scale, int causal,
                          fa_dtype_t dtype, const float* descale_q, const float* descale_k,
                          const float* descale_v, cudaStream_t stream);

fa_status_t fa_fwd_paged(const void* q, const void* k_cache, const void* v_cache, void* o,
                         float* lse, const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                         const int32_t* block_table, int64_t n_seqs, int64_t max_pages_per_seq,
                         int64_t page_size, int64_t num_pages, int64_t total_q,
                         int64_t max_seqlen_q, int64_t H, int64_t H_kv, int64_t D, float scale,
                         int causal, fa_dtype_t dtype, const float* descale_q,
                         const float* descale_k, const float* descale_v, cudaStream_t stream);

/*
 * fa_fwd_paged_split -- fa_fwd_paged with each (sequence, query tile)'s keys
 *   cut into n_splits chunks processed in parallel (fp32 partial O and lse
 *   in `workspace`, then the merge kernel: lse = log sum_s exp(lse_s),
 *   O = sum_s exp(lse_s - lse) O_s) -- the per-partition exp-sums and reduce
 *   of the paged-decode kernels in the Hygon retrospective (defect 7).  For
 *   decoding, where a few long sequences would otherwise leave most SMs
 *   idle.  Splits past a sequence's last key block are empty and get zero
 *   weight.  With a workspace the sequences are also taken longest first
 *   (a pre-pass ranks them by seqused_k; up to 16384 sequences, more keep
 *   their given order), so that the static hand-out of work items stays
 *   balanced when key lengths vary widely; the results do not depend on the
 *   order.  n_splits 1..32 (1: fa_fwd_paged, plus the ordering when a
 *   workspace is given); workspace: caller-owned device memory of at least
 *   fa_fwd_paged_split_workspace_size bytes (int32 [n_seqs] sequence order
 *   when n_seqs <= 16384, then for n_splits > 1 fp32 [n_splits, H, total_q,
 *   D] and fp32 [n_splits, H, total_q]; each part 256-byte aligned),
 *   256-byte aligned, contents on entry irrelevant; may be NULL only when
 *   n_splits is 1.  Statuses as fa_fwd_paged plus FA_ERR_INVALID_ARG
 *   (n_splits < 1, workspace missing or small), FA_ERR_MISALIGNED (workspace
 *   off 256 bytes), FA_ERR_UNSUPPORTED (n_splits > 32).  Up to three launches
 *   on `stream` (order, forward, merge); calls sharing a workspace must not
 *   overlap.
 *
 * fa_fwd_paged_split_workspace_size -- that workspace size for n_seqs
 *   sequences.  Host only; FA_ERR_INVALID_ARG on bad sizes or a NULL output.
 *
 * fa_fwd_paged_split_plan -- picks n_splits from sizes the host knows: the
 *   smallest count (1..32, at most half the longest sequence's 128-key
 *   blocks) at which the longest work item -- a split of the longest
 *   sequence, max_seqlen_k keys, plus about three blocks of fixed cost -- is
 *   at most half of one SM's share of all the work (total_k keys over the
 *   sequences, per group of query heads packed into a tile); and the
 *   workspace that count needs.  sm_count: the SMs to plan for, 0 for the
 *   current device's.  Host only; FA_ERR_INVALID_ARG on bad sizes
 *   (max_seqlen_k > total_k, H % H_kv != 0, ...) or NULL outputs, FA_ERR_CUDA
 *   if sm_count is 0 and the device cannot be queried.
 */
fa_status_t fa_fwd_paged_split_workspace_size(int64_t H, int64_t total_q, int64_t D, int n_splits,
                                              int64_t n_seqs, size_t* workspace_bytes);

fa_status_t fa_fwd_paged_split_plan(int64_t n_seqs, int64_t total_q, int64_t max_seqlen_q,
                                    int64_t total_k, int64_t max_seqlen_k, int64_t H,
                                    int64_t H_kv, int64_t D, int sm_count, int* n_splits,
                                    size_t* workspace_bytes);

fa_status_t fa_fwd_paged_split(const void* q, const void* k_cache, const void* v_cache, void* o,
                               float* lse, const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                               const int32_t* block_table, int64_t n_seqs,
                               int64_t max_pages_per_seq, int64_t page_size, int64_t num_pages,
                               int64_t total_q, int64_t max_seqlen_q, int64_t H, int64_t H_kv,
                               int64_t D, float scale, int causal, fa_dtype_t dtype,
                               const float* descale_q, const float* descale_k,
                               const float* descale_v, int n_splits, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream);

/*
 * Backward pass (fp16 / bf16): the gradients of the attention above with
 * respect to q, k and v, given the forward's o and lse and the upstream
 * gradient dout:
 *     P  = exp(scale * Q K^T - lse)   (masked entries 0; recomputed)
 *     dV = P^T dO,   dP = dO V^T,   dS = P * (dP - rowsum(dO * O))
 *     dQ = scale * dS K,   dK = scale * dS^T Q
 * -- the chain rule through the reference attention of "ops-transformer
 * FlashAttention build and tuning" (section 4.3); the pages train with this
 * operator (its mixed-precision training configuration) and describe the
 * backward dQ loop over key/value blocks (Hygon retrospective, defect 13).
 * With H_kv < H the gradient of a key/value head sums over the query heads
 * that read it.
 *
 * fa_bwd_workspace_size -- bytes of device workspace fa_bwd needs:
 *   2 * 4 * B * H * (S_q rounded up to 128), each half 256-byte aligned.
 *   Host only; FA_ERR_INVALID_ARG on bad sizes or a NULL output.
 *
 * fa_bwd -- q, k, v, o, dout, lse: as the forward's arguments and outputs
 *   (o and dout in q's layout and dtype, lse fp32 [B, H, S_q] natural log);
 *   dq (q's shape), dk and dv (k's shape): written, in the input dtype,
 *   round-to-nearest-even.  workspace: caller-owned device memory of at
 *   least fa_bwd_workspace_size bytes, 256-byte aligned; its contents on
 *   entry do not matter.  Checks and statuses as fa_fwd_gqa, plus:
 *   FA_ERR_INVALID_ARG for NULL dout / dq / dk / dv or a missing or small
 *   workspace; FA_ERR_MISALIGNED for those pointers off 16 bytes (workspace
 *   off 256); FA_ERR_UNSUPPORTED for FA_DTYPE_FP8E4M3.  Three launches on
 *   `stream` (a row-statistics pass, the dQ kernel, the dK/dV kernel); the
 *   workspace is written and read by them, so calls sharing one workspace
 *   must not overlap.  Deterministic: no atomics.
 */
fa_status_t fa_bwd_workspace_size(int64_t B, int64_t H, int64_t S_q, size_t* workspace_bytes);

fa_status_t fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H,
                   int64_t H_kv, int64_t S_q, int64_t S_kv, int64_t D, float scale,
                   fa_layout_t layout, int causal, fa_dtype_t dtype, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream);

/*
 * Strided tensors.  fa_strides_t gives a [B, H, S, D] tensor's element strides
 * along batch, head and sequence; D is contiguous.  Any layout follows: BNSD,
 * BSND, views of a fused QKV projection ([B, S, 3, H, D]: seq stride 3*H*D),
 * padded rows, or K and V with different strides -- the Hygon retrospective's
 * backward defect 13 came from stepping V by K's row stride, which passed
 * every test in which the two were equal.  Each stride * element size must
 * be a positive multiple of 16 bytes (a TMA requirement): FA_ERR_MISALIGNED
 * otherwise, FA_ERR_INVALID_ARG for a stride < 1 or a NULL array,
 * FA_ERR_UNSUPPORTED at or above 2^39 bytes.  lse stays dense [B, H, S_q].
 *
 * fa_fwd_strided -- fa_fwd_gqa with strides[0..3] = q, k, v, o.
 * fa_bwd_strided -- fa_bwd with strides[0..7] = q, k, v, o, dout, dq, dk, dv.
 */
typedef struct {
  int64_t batch, head, seq;
} fa_strides_t;

fa_status_t fa_fwd_strided(const void* q, const void* k, const void* v, void* o, float* lse,
                           int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv,
                           int64_t D, const fa_strides_t* strides, float scale, int causal,
                           fa_dtype_t dtype, const float* descale_q, const float* descale_k,
                           const float* descale_v, cudaStream_t stream);

fa_status_t fa_bwd_strided(const void* q, const void* k, const void* v, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_kv,
                           int64_t D, const fa_strides_t* strides, float scale, int causal,
                           fa_dtype_t dtype, void* workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/* A static, human-readable name for a status code (never NULL). */
const char* fa_status_string(fa_status_t s);

/*
 * fa_last_device_error -- synchronises `stream`, then reads and clears the
 * device error word of the current device.  Returns FA_OK if no kernel of this
 * library on that device has reported an error since the last call,
 * FA_ERR_DEVICE_TIMEOUT if a bounded wait expired, FA_ERR_CUDA if the
 * synchronisation or the read failed.
 */
fa_status_t fa_last_device_error(cudaStream_t stream);

/*
 * fa_set_wait_limit_ns -- the time limit, in nanoseconds of the device's
 * global timer, after which a device-side wait gives up and reports
 * FA_ERR_DEVICE_TIMEOUT (default 2e9 = 2 s).  0 restores the default.  A
 * process-wide host setting, read at each launch.
 */
void fa_set_wait_limit_ns(uint64_t ns);

/*
 * fa_probe_wait_timeout -- launches one block whose thread waits on a
 * shared-memory barrier that nothing ever arrives at, using the same bounded
 * wait as fa_fwd, with the given limit (ns).  The wait must expire, set the
 * device error word and return; the call then returns what
 * fa_last_device_error() reports (FA_ERR_DEVICE_TIMEOUT when the mechanism
 * works).  It exists so that the timeout path can be tested without a hang.
 */
fa_status_t fa_probe_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

/* Library version, "major.minor.patch". */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_API_H */
