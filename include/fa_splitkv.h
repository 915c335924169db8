/*
 * fa_splitkv.h -- C ABI of the split-KV flash-attention forward library
 * (libfa_splitkv.so) for NVIDIA GB300 (sm_103a).
 *
 * What it computes.  For every packed sequence b, query head h and query row
 * i < Lq_b, over the keys j the mask allows,
 *     s_j = scale * dq * dk * <Q[cu_q[b]+i, h, :], K[cu_k[b]+j, h/group, :]>
 *     LSE = ln(sum_j exp(s_j))
 *     O   = dv * sum_j exp(s_j - LSE) * V[cu_k[b]+j, h/group, :]
 * i.e. softmax(Q K^T * scale) V together with its natural-log log-sum-exp
 * (flash-attention PR "[Cute,Fwd,Sm100] Support q_stage=1 for inference",
 * description and "Benchmarks": split-KV forward; aiter PR "[FlyDSL] Enable
 * FP8 FMHA split-K for short cached-prefix queries": return_lse and FP8).
 * The key range of each (sequence, KV head, query tile) is cut into
 * num_splits parts processed by separate CTAs, each writing an fp32 partial
 * output and LSE to a caller-provided workspace; a combine kernel merges the
 * parts with LSE weights (aiter PR, timing note: "attention and split
 * combine").  Rows that see no key get O = 0 and LSE = -inf.
 *
 * Layout (cutlass "Adds variable sequence lengths to the Hopper CuTe DSL FMHA
 * example", section "Interface"): all tensors are packed along the token
 * axis, batch 1, innermost dimension contiguous:
 *     Q   [total_q, h_q,  d_qk]      K [total_k, h_kv, d_qk]
 *     V   [total_k, h_kv, d_v ]      O [total_q, h_q,  d_v ]
 *     LSE [h_q, total_q] float32 (natural log, includes the scale)
 *     cu_seqlens_q, cu_seqlens_k: int32 [batch+1], exclusive prefix sums;
 *     a fixed-length side is passed as uniform cu_seqlens.
 * GQA/MQA: h_q = group * h_kv, query head h reads KV head h / group.
 *
 * Masks (cutlass PR, section "Tests"): causal = 1 is bottom-right aligned
 * (query i sees keys j <= i + Lk - Lq); window_left >= 0 is a (window_left, 0)
 * sliding window (keys i+Lk-Lq-window_left .. i+Lk-Lq, inclusive), which
 * implies the causal right bound; window_left < 0 means no left bound.
 *
 * Memory and ownership.  Every pointer is caller-owned: q, k, v, cu_seqlens,
 * out, lse, workspace and descales are DEVICE pointers of the current CUDA
 * device.  The library allocates no device memory and never synchronises the
 * stream; all work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 * default stream), so calls can be captured in a CUDA graph.  Tensor-map
 * descriptors are encoded on the host per call.
 *
 * Alignment.  q, k, v, out and workspace must be 16-byte aligned and every
 * token stride (h * d * element size) a multiple of 16 bytes (TMA rule).
 *
 * Errors.  Invalid arguments are reported synchronously as a negative
 * fa_status before anything is launched.  Problems found on the device
 * (cu_seqlens inconsistent with batch / total_* / max_seqlen_q, or a
 * pipeline wait that timed out) skip the affected tiles and set a sticky
 * device error word, read with fa_get_device_error().
 */
#ifndef FA_SPLITKV_H
#define FA_SPLITKV_H

#include <stddef.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { FA_BF16 = 0, FA_FP16 = 1, FA_E4M3 = 2 } fa_dtype;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1,    /* bad pointer, size, alignment or value     */
  FA_ERR_UNSUPPORTED = -2,    /* valid but not implemented (dtype / dims)  */
  FA_ERR_WORKSPACE = -3,      /* workspace missing or too small            */
  FA_ERR_CUDA = -4,           /* a CUDA runtime call failed                */
  FA_ERR_DEVICE_TIMEOUT = -5, /* device: a pipeline wait ran out of time   */
  FA_ERR_DEVICE_ARG = -6,     /* device: cu_seqlens inconsistent with sizes */
  FA_ERR_DEVICE_BOUNDS = -7   /* device, debug build only: an index failed its
                                 bounds check and the access was skipped     */
} fa_status;

/* Kernel selection (flags argument of fa_fwd_splitkv_ex). */
#define FA_KERNEL_AUTO 0  /* by rows per KV head (see fa_fwd_splitkv_ex)            */
#define FA_KERNEL_SIMT 1  /* CUDA-core streaming kernel                            */
#define FA_KERNEL_UMMA 2  /* tcgen05 kernel, one 128-row query tile per CTA        */
#define FA_KERNEL_UMMA2 3 /* tcgen05 kernel, two 128-row tiles per CTA (16-bit)    */
#define FA_KERNEL_MASK 3
/* Stage selection (flags, OR-ed with the kernel choice).  By default a call
 * launches the partial kernel and, when the split count is > 1, the combine.
 * PARTIAL_ONLY launches only the partial kernel (which writes the workspace,
 * or O/LSE directly when the split count is 1); COMBINE_ONLY launches only the
 * combine over a workspace written by an earlier PARTIAL_ONLY call with the
 * same arguments.  Used to time the two kernels separately. */
#define FA_RUN_PARTIAL_ONLY 4
#define FA_RUN_COMBINE_ONLY 8

/*
 * fa_fwd_splitkv_ex -- split-KV attention forward (flash-decoding):
 * flash-attention PR "[Cute,Fwd,Sm100] Support q_stage=1 for inference"
 * (description: split KV over CTAs of one 128-row query tile), aiter PR
 * "[FlyDSL] Enable FP8 FMHA split-K for short cached-prefix queries"
 * (description: automatic and explicit splits, return_lse, FP8) and cutlass
 * "Adds variable sequence lengths to the Hopper CuTe DSL FMHA example"
 * ("Interface": cu_seqlens, packed varlen, GQA).
 *
 *  q, k, v        device inputs, layouts above, element type in_dtype.
 *  cu_seqlens_q/k device int32 [batch+1].
 *  batch          number of sequences (>= 0; 0 is a no-op).
 *  total_q/total_k rows of the packed Q/O and K/V buffers; cu_seqlens_q[batch]
 *                 must not exceed total_q, nor cu_seqlens_k[batch] total_k.
 *                 TMA reads never go past these rows (zero fill beyond).
 *  max_seqlen_q   largest Lq_b (sizes the tile grid and the workspace).
 *  h_q, h_kv      query and key/value heads, h_q % h_kv == 0, h_q/h_kv <= 128.
 *  d_qk, d_v      head dims: (64,64), (128,128) or (256,256) for bf16/fp16;
 *                 (128,128) or (192,128) for e4m3.
 *  scale          softmax scale; <= 0 selects 1/sqrt(d_qk) (cutlass PR,
 *                 "Implementation": the default scale uses the head dim).
 *  causal, window_left  masks, see above.
 *  num_splits     0 = automatic (fa_plan), else 1..128 splits of the key range.
 *  out            device [total_q, h_q, d_v] of out_dtype; rows of sequences
 *                 are written, other rows are untouched.
 *  lse            device float32 [h_q, total_q] or NULL.
 *  workspace      device scratch of >= fa_fwd_splitkv_workspace_size(...)
 *                 bytes, 16-byte aligned.  Required when the resolved split
 *                 count is > 1.  With one split it may be NULL: it then only
 *                 holds the persistent kernel's 16-byte tile counter, and
 *                 without it the non-persistent grid runs instead.  Contents
 *                 need no initialisation and are clobbered (in stream order).
 *  workspace_bytes size of workspace (checked).
 *  in_dtype, out_dtype  FA_BF16 / FA_FP16 / FA_E4M3 inputs.  Out is in_dtype
 *                 or FA_E4M3 for 16-bit inputs, and any of the three for e4m3
 *                 inputs.  An e4m3 O is the value itself rounded to nearest
 *                 even and saturated to +-448, with no output scale (the
 *                 pages define no fp8 output; this is the plainest form).
 *  descale_q/k/v  device float32 scalars, required for FA_E4M3 inputs
 *                 (per-tensor dequantisation factors), ignored otherwise.
 *  flags          FA_KERNEL_* selection, optionally OR FA_RUN_*_ONLY.  AUTO
 *                 picks the CUDA-core kernel for up to 2 rows (queries x
 *                 group) per KV head (up to 4 with head dim 64), the
 *                 one-tile tcgen05 kernel above that up to 128 rows and, for
 *                 e4m3 and head dim 256, beyond; and the two-tile tcgen05
 *                 kernel beyond 128
 *                 rows (16-bit, head dim <= 128; its persistent form for one
 *                 split over packed K/V with a workspace and a 32-byte
 *                 aligned out, at most 128 sequences and batch *
 *                 ceil(max_seqlen_q / (256 / group)) <= 4096 query pairs).
 *                 FA_KERNEL_UMMA2 always runs the non-persistent two-tile
 *                 kernel.
 *  stream         cudaStream_t.
 * Returns FA_OK or a negative fa_status.
 */
FA_API int fa_fwd_splitkv_ex(const void* q, const void* k, const void* v, const int* cu_seqlens_q,
                      const int* cu_seqlens_k, int batch, int total_q, int total_k,
                      int max_seqlen_q, int h_q, int h_kv, int d_qk, int d_v, float scale,
                      int causal, int window_left, int num_splits, void* out, float* lse,
                      void* workspace, size_t workspace_bytes, int in_dtype, int out_dtype,
                      const float* descale_q, const float* descale_k, const float* descale_v,
                      int flags, void* stream);

/*
 * fa_fwd_splitkv_paged -- the same forward pass over a paged K/V cache
 * (serving-style decode).  The pages this library follows do not describe a
 * paged layout; this one is the common serving convention:
 *   k_cache [num_pages, page_size, h_kv, d_qk], v_cache [num_pages, page_size,
 *   h_kv, d_v] (device, 16-byte aligned), block_table int32 [batch,
 *   max_pages_per_seq] (device): block_table[b][i] is the page holding keys
 *   i*page_size .. (i+1)*page_size-1 of sequence b; seqlens_k int32 [batch]
 *   (device): keys of sequence b.  page_size is a power of two >= 32.
 * Queries, outputs, masks, splits, dtypes, workspace and flags are as in
 * fa_fwd_splitkv_ex (fa_fwd_splitkv_workspace_size applies unchanged).  A
 * page index outside [0, num_pages) or a sequence longer than
 * max_pages_per_seq*page_size is skipped and reported as FA_ERR_DEVICE_ARG.
 */
FA_API int fa_fwd_splitkv_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int* cu_seqlens_q, const int* seqlens_k,
                                const int* block_table, int batch, int total_q, int num_pages,
                                int page_size, int max_pages_per_seq, int max_seqlen_q, int h_q,
                                int h_kv, int d_qk, int d_v, float scale, int causal,
                                int window_left, int num_splits, void* out, float* lse,
                                void* workspace, size_t workspace_bytes, int in_dtype,
                                int out_dtype, const float* descale_q, const float* descale_k,
                                const float* descale_v, int flags, void* stream);

/*
 * fa_fwd_splitkv -- bf16 in / bf16 out shorthand of fa_fwd_splitkv_ex with
 * automatic kernel selection: the split-KV forward of flash-attention PR
 * "[Cute,Fwd,Sm100] Support q_stage=1 for inference" (description: one
 * 128-row query tile per CTA, split KV on by default) with the automatic or
 * explicit split count of aiter PR "[FlyDSL] Enable FP8 FMHA split-K for
 * short cached-prefix queries" (description).  Arguments as in
 * fa_fwd_splitkv_ex; batch, total_q and total_k are needed because the host
 * cannot read cu_seqlens without synchronising and the tensor maps must know
 * where the buffers end.  The workspace is trusted to hold
 * fa_fwd_splitkv_workspace_size(...) bytes.
 */
FA_API int fa_fwd_splitkv(const void* q, const void* k, const void* v, const int* cu_seqlens_q,
                   const int* cu_seqlens_k, int batch, int total_q, int total_k,
                   int max_seqlen_q, int h_q, int h_kv, int d_qk, int d_v, float scale,
                   int causal, int window_left, int num_splits, void* out, float* lse,
                   void* workspace, void* stream);

/*
 * fa_fwd_splitkv_noalloc -- the same forward pass for callers that cannot
 * allocate device memory (no counterpart on the pages this library follows;
 * it is an addition for embedding).  Examples: code running under a runtime
 * or framework that owns all device allocations and gives the call site no
 * allocator, plugins without an allocator handle, and latency-critical paths
 * where cudaMalloc (which synchronises the device) is not allowed.  The
 * caller still passes inputs and outputs; the fp32 split workspace comes
 * from a fixed array of FA_NOALLOC_SCRATCH_BYTES in device global memory
 * defined by the library, which every device that loads it (at the latest on
 * the first call there) keeps until the process exits.
 *
 * Arguments are those of fa_fwd_splitkv_ex without workspace and
 * workspace_bytes.  The call allocates nothing and frees nothing.  Problems
 * whose workspace (fa_fwd_splitkv_workspace_size) exceeds
 * FA_NOALLOC_SCRATCH_BYTES are rejected with FA_ERR_WORKSPACE before any
 * launch.  The first call on each device looks up the array's device address
 * with that device current (make it before any stream capture).  All calls
 * on a device share the one array: calls that may overlap on the GPU (other
 * streams, other host threads) race on it and must be serialised by the
 * caller.  The array keeps the last call's contents.  Every partial a call
 * reads was written by that call, and the one word that must start at zero
 * (the persistent prefill kernel's tile counter) is zeroed in stream order by
 * each call before its launch.
 */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20) /* 8 MiB */
FA_API int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v,
                                  const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                                  int total_q, int total_k, int max_seqlen_q, int h_q, int h_kv,
                                  int d_qk, int d_v, float scale, int causal, int window_left,
                                  int num_splits, void* out, float* lse, int in_dtype,
                                  int out_dtype, const float* descale_q, const float* descale_k,
                                  const float* descale_v, int flags, void* stream);

/*
 * fa_fwd_splitkv_host -- the same forward pass on host buffers (no
 * counterpart on the pages this library follows; an addition for callers
 * whose inputs and outputs live in host memory, and the end-to-end call a
 * benchmark times).  q, k, v, cu_seqlens_q, cu_seqlens_k and, for FA_E4M3
 * inputs, descale_q/k/v (one float each) are read from HOST memory; out and
 * lse (may be NULL) are written to HOST memory.  Layouts are those of
 * fa_fwd_splitkv_ex.  Each transfer is one cudaMemcpyAsync on `stream` in
 * stream order: the inputs, then the forward pass, then O and LSE.  The
 * call returns once they are enqueued; synchronise the stream before
 * reading out/lse or reusing an input buffer.  Page-locked host buffers make
 * the copies asynchronous; pageable ones work, with each copy staged by the
 * driver.
 *
 * device_buffer (device, 256-byte aligned, caller-owned, device_buffer_bytes
 * at least fa_fwd_splitkv_host_buffer_size(...)) holds the device copies of
 * the inputs, O, LSE and the split workspace; the call allocates nothing.
 * Errors: FA_ERR_INVALID_ARG for invalid sizes or dtypes, a NULL or
 * misaligned device_buffer, or a NULL host buffer that has bytes to copy;
 * FA_ERR_WORKSPACE when device_buffer is too small (both before any copy);
 * FA_ERR_CUDA when a copy cannot be enqueued; otherwise whatever
 * fa_fwd_splitkv_ex returns for the device copies.
 */
FA_API int fa_fwd_splitkv_host(const void* q, const void* k, const void* v,
                               const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                               int total_q, int total_k, int max_seqlen_q, int h_q, int h_kv,
                               int d_qk, int d_v, float scale, int causal, int window_left,
                               int num_splits, void* out, float* lse, void* device_buffer,
                               size_t device_buffer_bytes, int in_dtype, int out_dtype,
                               const float* descale_q, const float* descale_k,
                               const float* descale_v, int flags, void* stream);

/*
 * fa_fwd_splitkv_host_buffer_size -- bytes of device buffer
 * fa_fwd_splitkv_host needs for these sizes (no counterpart on the pages
 * this library follows): 256-byte aligned regions for Q, K, V, the two
 * offset arrays, the descales, O, LSE and the split workspace of
 * fa_fwd_splitkv_workspace_size.  num_splits = 0 resolves the automatic
 * count on the current device.  Returns 0 for invalid sizes or dtypes.
 */
FA_API size_t fa_fwd_splitkv_host_buffer_size(int batch, int total_q, int total_k,
                                              int max_seqlen_q, int h_q, int h_kv, int d_qk,
                                              int d_v, int in_dtype, int out_dtype,
                                              int num_splits);

/*
 * fa_fwd_splitkv_workspace_size -- bytes of workspace fa_fwd_splitkv_ex needs
 * for these sizes.  aiter PR "[FlyDSL] Enable FP8 FMHA split-K for short
 * cached-prefix queries" (review: automatic split-K "plus a per-call fp32
 * workspace"; timing note: attention and split combine): the fp32 partial
 * outputs [ns, batch*max_seqlen_q, h_q, d_v] followed by the partial LSEs
 * [ns, batch*max_seqlen_q, h_q], indexed by (sequence, query) so that the
 * host can size them without reading cu_seqlens; 16 bytes (the persistent
 * kernel's tile counter) when the resolved split count is 1.  num_splits = 0
 * resolves the automatic count on the current device.  Returns 0 for
 * invalid sizes.
 */
FA_API size_t fa_fwd_splitkv_workspace_size(int batch, int max_seqlen_q, int h_q, int h_kv, int d_v,
                                     int num_splits);

/*
 * fa_plan -- the split planner (host only; no device work).  The pages give
 * its inputs, not its rule: aiter PR "[FlyDSL] Enable FP8 FMHA split-K for
 * short cached-prefix queries" (description: automatic and explicit split
 * selection; review: up to 16 splits) and flash-attention PR "[Cute,Fwd,
 * Sm100] Support q_stage=1 for inference" ("Benchmarks": the num_splits
 * sweep 1..128 at B=1, Q=1, K=131072, H=32, where too few splits leave SMs
 * idle).  The rule below is this library's reading.
 * units = batch * h_kv * ceil(max_seqlen_q * (h_q/h_kv) / 128) work units;
 * explicit num_splits > 0 is clipped to 128; with no work or with
 * units >= 2*num_sms the count is 1; otherwise it is the smallest ns in
 * 1..128 whose wave efficiency units*ns / (ceil(units*ns/num_sms)*num_sms)
 * reaches 0.9, else the first most efficient one.  num_sms <= 0 queries the
 * current device.  Writes the split count and the unit count (the kernels
 * decode a linear CTA index, so the launch shape is the unit count times the
 * split count, or one CTA per SM for the persistent kernel, not a 3-D grid).
 */
FA_API int fa_plan(int batch, int max_seqlen_q, int h_q, int h_kv, int num_splits, int num_sms,
            int* num_splits_out, int* units_out);

/*
 * fa_debug_split_ranges -- test hook (no counterpart on the pages; it exposes
 * the key split of flash-attention PR "[Cute,Fwd,Sm100] Support q_stage=1
 * for inference", description, as the kernels compute it on the device so
 * that it can be checked bit for bit): runs the device-side tile decode for a
 * tile of `tile_queries` queries and writes, for every (m_block, b, split),
 * the sequence-local key range [k0, k1) the kernels process (k1 <= k0 for an
 * empty split) to ranges_out: device int32 [ceil(max_seqlen_q/tile_queries),
 * batch, num_splits, 2].  Enqueued on stream.
 */
FA_API int fa_debug_split_ranges(const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                          int max_seqlen_q, int causal, int window_left, int num_splits,
                          int tile_queries, int* ranges_out, void* stream);

/* Test hook (no counterpart in the pages): enqueues one CTA whose single
 * thread waits, with the kernels' own bounded mbarrier wait, on a phase that
 * nothing completes.  After timeout_ms (1..10000) the wait gives up, records
 * FA_ERR_DEVICE_TIMEOUT in the device error word (if no error is recorded
 * yet) and the kernel returns; the context stays usable.  While the word
 * holds FA_ERR_DEVICE_TIMEOUT, the forward kernels skip their work.
 * Returns FA_ERR_INVALID_ARG for a timeout outside 1..10000 ms. */
FA_API int fa_debug_wait_timeout(unsigned int timeout_ms, void* stream);

/* Partial kernels a forward call can launch, as fa_debug_last_kernel reports
 * them (these are not flag values). */
typedef enum {
  FA_KID_NONE = 0,             /* no partial kernel launched                      */
  FA_KID_SIMT = 1,             /* CUDA-core streaming kernel                      */
  FA_KID_UMMA = 2,             /* tcgen05 kernel, one 128-row tile per CTA        */
  FA_KID_UMMA2 = 3,            /* tcgen05 kernel, two 128-row tiles per CTA       */
  FA_KID_UMMA2_PERSISTENT = 4  /* its persistent form (chosen by AUTO only)       */
} fa_kernel_id;

/* Test hook (no counterpart in the pages): the partial kernel that the calling
 * thread's most recent fa_fwd_splitkv* call enqueued, recorded on the host at
 * launch (fa_kernel_id); FA_KID_NONE if that call enqueued none (an argument
 * error, FA_RUN_COMBINE_ONLY, or no sequence). */
FA_API int fa_debug_last_kernel(void);

/* Sticky device error word of the current device (FA_OK if none); no
 * counterpart on the pages.  Waits for the device to finish its work.
 * clear != 0 resets the word. */
FA_API int fa_get_device_error(int clear);

/* Human-readable name of an fa_status value (static string); no counterpart
 * on the pages. */
FA_API const char* fa_status_string(int status);

/* Library version: major*10000 + minor*100 + patch; no counterpart on the
 * pages. */
FA_API int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_SPLITKV_H */
