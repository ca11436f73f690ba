/*
 * pfkv.h -- C ABI of libpfkv.so: decode attention over a paged FP8 (e4m3) or
 * BF16 KV cache with per-page integrity tags, for NVIDIA GB300 (sm_103a).
 *
 * What is computed comes from these web pages (cited by title and section):
 *  - "How we built the most efficient inference engine for Cloudflare's
 *    network", section "Batching to feed the Tensor Cores": the KV cache is
 *    split into small pages that are handed out only as a sequence grows.
 *  - "Workers AI targets the inference bottleneck", section "KV cache
 *    compression goes open source": a block table of integer page indices maps
 *    each sequence's logical pages onto physical pages, which lets every
 *    attention head keep a different number of tokens (per-head eviction).
 *  - "Cloudflare quantizes Kimi and GLM caches for 41% faster inference",
 *    2nd paragraph: the cache is stored as FP8 e4m3 instead of BF16, halving
 *    it, and decode (memory-bound) reads the FP8 cache; 4th paragraph: every
 *    physical page carries a tag that changes when the page is reallocated,
 *    each request's expected (page, tag) pairs are checked by a separate batch
 *    validation before decode reads the cache, a request with any mismatch is
 *    aborted, and with checking disabled a no-op tracker costs nothing.
 *
 * Conventions for every call:
 *  - Memory: every pointer argument not marked "host" is memory the GPU can
 *    address, owned by the caller: device memory, or host memory the device
 *    maps (pinned with cudaHostAlloc / cudaHostRegister, or any host memory on
 *    a system with a coherent CPU-GPU link such as Grace + NVLink-C2C).  The
 *    kernels read and write host memory directly, without a staging copy:
 *    per-step inputs and outputs (q, new K/V rows, positions, lengths, block
 *    tables, expected tags, out, flags) may live there; the pools, scales,
 *    tags and workspace belong in HBM, which the kernels stream.  The library
 *    never allocates device memory for data and keeps no state between calls,
 *    except the step-graph objects that a caller creates and destroys
 *    explicitly (CUDA graphs, a driver resource); calls on different streams
 *    are independent.
 *  - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  All
 *    work is enqueued asynchronously on it; no call synchronises the host.
 *  - Alignment: k_pages, v_pages, q, out, k_new and v_new 16-byte aligned;
 *    workspace 256-byte aligned; index, length, tag, scale and e4m3-utility
 *    arrays 4-byte aligned; flags 4-byte aligned and backed by at least
 *    round_up(batch, 4) bytes (bits are OR-ed through 32-bit words).
 *    Misalignment returns PFKV_ERR_ALIGNMENT.
 *  - Errors: argument errors the host can see are returned before anything is
 *    enqueued.  PFKV_ERR_CUDA means a launch failed (cudaGetLastError).  Errors
 *    in device-resident data (page ids, lengths, tags) never fault: they are
 *    reported per request in `flags` and that request's output is zero, which
 *    callers treat as "aborted".
 *  - Hardware: compiled for sm_103a only.  Calls return PFKV_ERR_UNSUPPORTED on
 *    other devices.
 */
#ifndef PFKV_H
#define PFKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PFKV_OK = 0,
    PFKV_ERR_INVALID_ARG = 1,  /* NULL pointer, bad size, stride or count      */
    PFKV_ERR_UNSUPPORTED = 2,  /* head_dim, group size, page size or device    */
    PFKV_ERR_ALIGNMENT = 3,    /* a pointer is not suitably aligned            */
    PFKV_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required   */
    PFKV_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed         */
    PFKV_ERR_DEVICE = 6        /* a device-side wait gave up: returned only by
                                  pfkv_flags_status (no call synchronises the
                                  host, so the call that met it cannot)       */
} pfkv_status;

typedef enum {
    PFKV_KV_BF16 = 0,          /* pages hold bf16 values                       */
    PFKV_KV_FP8_E4M3 = 1       /* pages hold OCP e4m3 bytes + fp32 unit scales */
} pfkv_kv_dtype;

/* Tokens per page. */
#define PFKV_PAGE_SIZE 16

/* Per-request flag bits (uint8 per request). */
#define PFKV_FLAG_TAG_MISMATCH 0x01u  /* a live page's tag != the expected tag  */
#define PFKV_FLAG_BAD_PAGE 0x02u      /* a live table entry is outside the pool  */
#define PFKV_FLAG_BAD_LENGTH 0x04u    /* length/position outside the table or
                                         above max_seq_len                       */
#define PFKV_FLAG_DEVICE_TIMEOUT 0x08u /* a bounded device-side wait gave up;
                                          the output of the request is invalid   */

/*
 * The page pool.  A "unit" is one (physical page, kv head) slab of
 * PFKV_PAGE_SIZE tokens x head_dim elements; a block-table entry `phys` read
 * for kv head h always names unit (phys, h).
 *   k_pages, v_pages : [num_pages][num_kv_heads][PFKV_PAGE_SIZE][head_dim],
 *                      bf16 (dtype BF16) or e4m3 bytes (dtype FP8_E4M3)
 *   k_scale, v_scale : fp32 [num_pages][num_kv_heads] for FP8 (value of an
 *                      element = e4m3 value x unit scale); ignored for BF16
 *   page_tags        : uint32 [num_pages][num_kv_heads], or NULL when tags are
 *                      not tracked (the no-op tracker: no check is run)
 */
typedef struct pfkv_cache {
    int32_t num_pages;
    int32_t num_kv_heads;
    int32_t page_size;     /* must be PFKV_PAGE_SIZE */
    int32_t head_dim;      /* 64 or 128 */
    int32_t dtype;         /* pfkv_kv_dtype */
    void *k_pages;
    void *v_pages;
    float *k_scale;
    float *v_scale;
    const uint32_t *page_tags;
} pfkv_cache;

/*
 * The batch's view of the pool.
 *   block_tables  : int32, entry (b, h, p) at
 *                   block_tables[b*bt_stride_b + h*bt_stride_h + p],
 *                   p < max_pages.  bt_stride_h = 0 shares one table across
 *                   kv heads; > 0 gives every kv head its own table.
 *   seq_lens      : int32 tokens of (b, h) at
 *                   seq_lens[b*len_stride_b + h*len_stride_h] (len_stride_h = 0:
 *                   one length per request).  Only entries p < ceil(len/16) are
 *                   live; the rest of a row is never read.
 *   expected_tags : uint32, indexed like block_tables: the tag the request
 *                   expects on each live page.  NULL iff page_tags is NULL.
 */
typedef struct pfkv_pages {
    int32_t batch;
    int32_t max_pages;
    const int32_t *block_tables;
    int64_t bt_stride_b;
    int64_t bt_stride_h;
    const int32_t *seq_lens;
    int64_t len_stride_b;
    int64_t len_stride_h;
    const uint32_t *expected_tags;
} pfkv_pages;

/*
 * pfkv_kv_append -- write new tokens' K and V into their page slots,
 * quantising to e4m3 for an FP8 pool ("Cloudflare quantizes Kimi and GLM
 * caches for 41% faster inference", 2nd paragraph).
 *
 *   positions    : int32, indexed with the length strides of `pages`: position
 *                  of the first new token of (b, h)
 *   new_lens     : int32 (same indexing) number of new tokens of (b, h), each
 *                  <= num_new_tokens; NULL means num_new_tokens for all
 *   num_new_tokens: T >= 1
 *   k_new, v_new : bf16 [batch][num_kv_heads][T][head_dim]
 *   flags        : uint8 [batch] or NULL; bits are OR-ed in, never cleared
 *
 * Token t of (b, h) goes to position pos = positions + t: unit
 * (block_tables[b,h,pos/16], h), slot pos % 16.  FP8: the call that writes
 * slot 0 of a unit sets that unit's K and V scales to absmax/448 (fp32 IEEE
 * division; 1 if absmax is 0) over the tokens it writes into the unit; other
 * calls keep the stored scales.  Each byte is the e4m3 encoding, round to
 * nearest even and saturating to +-448, of the fp32 quotient x / scale.  BF16:
 * values are copied.  seq_lens is not read or updated.
 * A destination whose logical page is >= max_pages (PFKV_FLAG_BAD_LENGTH),
 * whose page id is outside the pool (PFKV_FLAG_BAD_PAGE) or, when tags are
 * tracked, whose pool tag differs from the expected tag
 * (PFKV_FLAG_TAG_MISMATCH) is not written.  Two calls, or two (b, h), that
 * write the same unit concurrently race.
 */
pfkv_status pfkv_kv_append(const pfkv_cache *cache, const pfkv_pages *pages,
                           const int32_t *positions, const int32_t *new_lens,
                           int32_t num_new_tokens, const void *k_new,
                           const void *v_new, uint8_t *flags, void *stream);

/*
 * pfkv_decode_workspace_size -- bytes of device workspace that
 * pfkv_paged_decode_attn needs for these arguments (host call; reads no
 * device memory).  *bytes (host) receives the size.
 */
pfkv_status pfkv_decode_workspace_size(const pfkv_cache *cache, const pfkv_pages *pages,
                                       int32_t num_q_heads, int32_t split_tokens,
                                       int32_t max_seq_len, size_t *bytes);

/*
 * pfkv_paged_decode_attn -- one decode step of attention for every request
 * and query head, reading K/V through the block tables ("Workers AI targets
 * the inference bottleneck", KV cache compression section) from an FP8 or
 * BF16 pool ("Cloudflare quantizes Kimi and GLM caches ...", 2nd paragraph),
 * after the integrity check of the 4th paragraph of the same page.
 *
 *   q            : bf16 [batch][num_q_heads][head_dim]
 *   num_q_heads  : a multiple G of num_kv_heads with G in {1, 2, 4, 8}; query
 *                  head hq reads kv head hq / G
 *   sm_scale     : softmax scale (usually 1/sqrt(head_dim))
 *   split_tokens : tokens per split-KV chunk (a multiple of 16), or 0 to let
 *                  the library choose
 *   max_seq_len  : host-known upper bound of every seq_lens entry (sizes the
 *                  launch); a longer length is flagged PFKV_FLAG_BAD_LENGTH
 *   workspace    : >= pfkv_decode_workspace_size(...) bytes; contents on entry
 *                  are ignored; must not be used concurrently by another call
 *   out          : bf16 [batch][num_q_heads][head_dim]
 *   flags        : uint8 [batch], written (not OR-ed); may be NULL
 *
 * For each (b, hq) with h = hq / G and n = seq_lens(b, h):
 *   out = sum_j softmax_j(sm_scale * q . k_j) v_j over tokens j < n, where
 *   token j is slot j % 16 of unit (block_tables[b,h,j/16], h) and FP8 values
 *   are e4m3 value x unit scale, rounded to bf16.  Arithmetic: the two
 *   products run on the tensor cores with fp32 accumulation.  FP8 pools:
 *   e4m3 values are exact in f16; q enters as f16 after a power-of-two
 *   scaling (exact for every element within 2^14 of its largest); each
 *   softmax weight (times the unit's V scale over a power-of-two reference)
 *   enters as a pair of f16 values whose sum is within 2^-22 of it
 *   (relative; 2^-25 absolute where the low part is subnormal).  BF16 pools:
 *   K, V and q are exact in bf16 and each weight is a pair of bf16 values
 *   whose sum is within 2^-18 of it.  Scores, the running max and sums, and
 *   the merge of partial results are fp32.
 * out is zero for a zero-length head and for every head of a flagged request.
 * When page_tags is non-NULL every live entry's pool tag is compared with the
 * expected tag before any page of the batch is read (a separate validation
 * kernel, stream-ordered before attention); page ids and lengths are always
 * bounds-checked.
 */
pfkv_status pfkv_paged_decode_attn(const pfkv_cache *cache, const pfkv_pages *pages,
                                   const void *q, int32_t num_q_heads, float sm_scale,
                                   int32_t split_tokens, int32_t max_seq_len,
                                   void *workspace, size_t workspace_bytes, void *out,
                                   uint8_t *flags, void *stream);

/* Stages of one attention call, in stream order. */
#define PFKV_STAGE_VALIDATE 0x1u  /* tag/bounds check (runs only if tags tracked) */
#define PFKV_STAGE_SPLIT 0x2u     /* per-chunk attention into the workspace       */
#define PFKV_STAGE_COMBINE 0x4u   /* merge chunks, write out and flags            */
#define PFKV_STAGE_ALL 0x7u
/* Not a stage: an option bit of pfkv_paged_decode_attn_stages.  With it the
 * tag comparison runs inside the SPLIT stage's page loop, as in
 * pfkv_paged_decode_attn_fused_tags, and VALIDATE launches nothing. */
#define PFKV_STAGE_FUSED_TAGS 0x8u
/* Not a stage either: with it SPLIT and COMBINE run the per-chunk CUDA-core
 * kernels (e4m3 dequantised to fp32 in registers, fp32 FMAs, no tensor cores)
 * for every shape, instead of the persistent tensor-core kernel.  The result
 * is the same computation within the tolerance; the option exists to measure
 * the two designs against each other.  Its workspace can be larger than
 * pfkv_decode_workspace_size reports (PFKV_ERR_WORKSPACE if too small). */
#define PFKV_STAGE_CUDA_CORES 0x10u

/*
 * pfkv_paged_decode_attn_stages -- the same computation as
 * pfkv_paged_decode_attn, launching only the stages named in `stages` (a
 * PFKV_STAGE_* mask).  Calling VALIDATE, then SPLIT, then COMBINE with the
 * same arguments and workspace, in stream order, gives exactly the result of
 * one pfkv_paged_decode_attn call (which is this call with PFKV_STAGE_ALL).
 * The workspace carries the state between stages; calling a later stage
 * without the earlier ones of the same arguments gives unspecified (but
 * in-bounds) output.  Lets a caller time or interleave the kernels.
 * PFKV_STAGE_FUSED_TAGS may be added to any mask (see below).
 * No stage bit, or an unknown bit: PFKV_ERR_INVALID_ARG.
 */
pfkv_status pfkv_paged_decode_attn_stages(const pfkv_cache *cache, const pfkv_pages *pages,
                                          const void *q, int32_t num_q_heads, float sm_scale,
                                          int32_t split_tokens, int32_t max_seq_len,
                                          void *workspace, size_t workspace_bytes, void *out,
                                          uint8_t *flags, uint32_t stages, void *stream);

/*
 * pfkv_paged_decode_attn_fused_tags -- pfkv_paged_decode_attn with the
 * integrity check moved into the attention kernel.
 *
 * The tag-check page ("Cloudflare quantizes Kimi and GLM caches ...", 4th
 * paragraph) keeps the check in a separate batch pass because, fused into its
 * attention kernel, it would race with the use of the data.  Here no output
 * is written before the combine stage, and the combine is stream-ordered
 * after every attention CTA, so the check can run where the page ids are
 * loaded: each live entry's pool tag is compared with its expected tag, a
 * mismatching unit is not read, and the mismatch reaches the request's flags
 * through the per-segment status that the combine ORs.
 *
 * Same arguments, workspace size, out and flags as pfkv_paged_decode_attn:
 * the same bits for the same inputs, and all-zero output for a flagged
 * request.  One difference is visible only as memory traffic: the matching
 * pages of a request that has a mismatch elsewhere are still read.  Without
 * tags (page_tags NULL) the two calls are identical.
 */
pfkv_status pfkv_paged_decode_attn_fused_tags(const pfkv_cache *cache, const pfkv_pages *pages,
                                              const void *q, int32_t num_q_heads, float sm_scale,
                                              int32_t split_tokens, int32_t max_seq_len,
                                              void *workspace, size_t workspace_bytes, void *out,
                                              uint8_t *flags, void *stream);

/*
 * pfkv_decode_step -- one decode step of a layer: pfkv_kv_append of the new
 * tokens, then pfkv_paged_decode_attn over the same pages, in one call.
 *
 * Arguments are those of the two calls: positions .. append_flags as for
 * pfkv_kv_append (append_flags receives its bits), q .. flags as for
 * pfkv_paged_decode_attn (same workspace size).  options: 0, or
 * PFKV_STAGE_FUSED_TAGS for the check inside attention.
 *
 * The result is exactly that of the two calls in stream order: same pool
 * bytes, scales, outputs and flags.  The validation reads only tables, tags
 * and lengths, never the pool, so here it runs in the same launch as the
 * append, which saves one kernel's latency per step.  Every argument of both
 * parts is checked before anything is launched; on any error nothing runs.
 */
pfkv_status pfkv_decode_step(const pfkv_cache *cache, const pfkv_pages *pages,
                             const int32_t *positions, const int32_t *new_lens,
                             int32_t num_new_tokens, const void *k_new, const void *v_new,
                             uint8_t *append_flags, const void *q, int32_t num_q_heads,
                             float sm_scale, int32_t split_tokens, int32_t max_seq_len,
                             void *workspace, size_t workspace_bytes, void *out, uint8_t *flags,
                             uint32_t options, void *stream);

/*
 * pfkv_stage_copy -- copy `bytes` from `src` to `dst` with a kernel in which
 * every SM moves 16-byte words: for the per-step inputs a caller keeps in host
 * memory.  (The source pages have no counterpart; it exists for callers.)
 *
 * On a system with a coherent CPU-GPU link (Grace + NVLink-C2C) a kernel that
 * reads pinned host memory moves a few hundred KB sooner than a copy engine.
 * Staging the packed inputs of a decode step of the Llama-shaped layer
 * (q, new K/V rows, positions, lengths, block table, expected tags: 524 KB)
 * and then calling pfkv_decode_step on the device copy took 2.7 us more per
 * step than the call alone, against 12 us for a copy-engine node and 8 us for
 * the call's kernels reading those inputs from host memory in place.
 *
 * Like every kernel of this library it first waits for the previous kernel
 * in the stream, then lets the next one launch early (programmatic dependent
 * launch).  This library's kernels read dst only after the copy has
 * completed; a caller's kernel launched with programmatic dependent launch
 * must likewise wait (griddepcontrol.wait) before it reads dst.
 *
 *   dst, src : memory the GPU can address (device, or host memory the device
 *              maps), 16-byte aligned; the two ranges must not overlap
 *   bytes    : a multiple of 16; 0 enqueues nothing
 * Errors: NULL pointer or overlapping ranges -> PFKV_ERR_INVALID_ARG; a
 * misaligned pointer or size -> PFKV_ERR_ALIGNMENT; not an sm_103 device ->
 * PFKV_ERR_UNSUPPORTED.
 */
pfkv_status pfkv_stage_copy(void *dst, const void *src, size_t bytes, void *stream);

/*
 * pfkv_flags_status -- the library status that a finished call's per-request
 * flags amount to.  `flags` is HOST memory: the `flags` array of an attention
 * or decode-step call, copied back by the caller once that call's stream has
 * completed.  Returns PFKV_ERR_DEVICE if any of the first `batch` requests
 * carries PFKV_FLAG_DEVICE_TIMEOUT (a bounded device-side wait gave up, so
 * that request's output is not valid and the device may be unhealthy), else
 * PFKV_OK.  Tag, page and length flags describe the caller's data, not a
 * failure of the library, and give PFKV_OK.  No call of this library
 * synchronises the host, so none can return a device-side failure itself;
 * the flags carry it, and this query turns it into a status.  Requests
 * aborted by a mismatching tag are the pages' "aborted request" ("Cloudflare
 * quantizes Kimi and GLM caches ...", 4th paragraph); a timeout is this
 * library's own failure and is reported apart from them.  flags NULL with
 * batch > 0, or batch < 0: PFKV_ERR_INVALID_ARG.  Makes no CUDA call.
 */
pfkv_status pfkv_flags_status(const uint8_t *flags, int32_t batch);

/*
 * pfkv_paged_decode_attn_noalloc -- pfkv_paged_decode_attn without a
 * caller-provided workspace.  (The source pages have no counterpart to this
 * call; it exists for callers, not for the method.)
 *
 * For callers that cannot allocate device memory when they decode: an engine
 * that has already given all GPU memory to its weights and KV page pool, a
 * plugin whose host framework owns every device allocation, or a decode loop
 * that must not call cudaMalloc/cudaFree because they can synchronise the
 * device.  The workspace is instead a file-scope device array of
 * PFKV_NOALLOC_WORKSPACE_BYTES inside this library; every GPU that loads the
 * library holds it until the process exits.  This call allocates nothing.
 *
 * Arguments, results and errors are those of pfkv_paged_decode_attn, plus:
 *  - a call that would need more than PFKV_NOALLOC_WORKSPACE_BYTES of
 *    workspace (pfkv_decode_workspace_size) returns PFKV_ERR_WORKSPACE and
 *    enqueues nothing;
 *  - the first call with a given device (and CUDA context) current looks up
 *    the array's device address (cudaGetSymbolAddress) for it, and so does
 *    the first call after another context becomes current on that device
 *    (a plugin host's own context, or the primary context after a
 *    cudaDeviceReset); make that first call before capturing the stream into
 *    a CUDA graph;
 *  - all calls share the one array, which keeps the previous call's contents
 *    (this is harmless: the workspace's contents on entry are ignored).  Two
 *    calls whose work overlaps on the GPU (different streams, or different
 *    host threads without ordering) race on it and may return wrong results.
 */
#define PFKV_NOALLOC_WORKSPACE_BYTES (16u << 20)
pfkv_status pfkv_paged_decode_attn_noalloc(const pfkv_cache *cache, const pfkv_pages *pages,
                                           const void *q, int32_t num_q_heads, float sm_scale,
                                           int32_t split_tokens, int32_t max_seq_len, void *out,
                                           uint8_t *flags, void *stream);

/*
 * pfkv_paged_decode_attn_mass -- pfkv_paged_decode_attn that also adds each
 * live token's attention mass to a running total kept by the caller.
 *
 * Eviction ("Workers AI targets the inference bottleneck", section "KV cache
 * compression goes open source", 3rd paragraph) tracks how much attention
 * every KV entry has received over past steps and evicts the entries with
 * the lowest total.  For every (b, h) of a request that is not flagged, and
 * every token j < n = seq_lens(b, h):
 *   attn_mass[b*mass_stride_b + h*mass_stride_h + j] +=
 *       sum over the G query heads hq of kv head h of softmax_j(sm_scale q_hq . k_j)
 * (the weights the output uses, normalised over the head's n tokens, fp32).
 * Flagged requests and zero-length heads add nothing.  Rows of different
 * (b, h) must not overlap.
 *
 *   attn_mass     : float, 4-byte aligned; strides in elements (>= 0)
 *   options       : 0 or PFKV_STAGE_FUSED_TAGS (tag check inside attention)
 *   workspace     : >= pfkv_decode_mass_workspace_size(...) bytes, which adds
 *                   batch x num_q_heads x max_seq_len floats of final scores
 * out and flags are those of pfkv_paged_decode_attn.
 */
pfkv_status pfkv_decode_mass_workspace_size(const pfkv_cache *cache, const pfkv_pages *pages,
                                            int32_t num_q_heads, int32_t split_tokens,
                                            int32_t max_seq_len, size_t *bytes);
pfkv_status pfkv_paged_decode_attn_mass(const pfkv_cache *cache, const pfkv_pages *pages,
                                        const void *q, int32_t num_q_heads, float sm_scale,
                                        int32_t split_tokens, int32_t max_seq_len,
                                        void *workspace, size_t workspace_bytes, void *out,
                                        uint8_t *flags, float *attn_mass, int64_t mass_stride_b,
                                        int64_t mass_stride_h, uint32_t options, void *stream);

/*
 * pfkv_paged_decode_attn_multi -- attention of several query tokens per
 * request, causal among them: the verification pass of speculative
 * (prompt-lookup) decoding, which checks all candidate tokens in one forward
 * pass ("Workers AI targets the inference bottleneck", section "Speculative
 * decoding: predicting more than one token", 1st paragraph).
 *
 * The request's num_query_tokens = kq candidate tokens are the LAST kq tokens
 * of each of its heads (already written, e.g. by pfkv_kv_append with
 * num_new_tokens = kq).  Query token i (0-based) attends to the first
 * n - kq + 1 + i tokens of head h, n = seq_lens(b, h): the cached context, the
 * candidates before it and itself.  A query that would see no token (n < kq)
 * gives zero output.
 *
 *   q, out : bf16 [batch][kq][num_q_heads][head_dim]
 *   flags  : per request [batch], as in pfkv_paged_decode_attn; a flagged
 *            request gives zero output for all of its query tokens
 *   options: 0 or PFKV_STAGE_FUSED_TAGS
 *   workspace >= pfkv_decode_multi_workspace_size(...) bytes
 * kq = 1 is pfkv_paged_decode_attn.  The kq queries of a request read the
 * same pages; the kernels process them side by side so that repeated reads
 * of a page tend to hit L2.
 */
pfkv_status pfkv_decode_multi_workspace_size(const pfkv_cache *cache, const pfkv_pages *pages,
                                             int32_t num_q_heads, int32_t num_query_tokens,
                                             int32_t split_tokens, int32_t max_seq_len,
                                             size_t *bytes);
pfkv_status pfkv_paged_decode_attn_multi(const pfkv_cache *cache, const pfkv_pages *pages,
                                         const void *q, int32_t num_q_heads,
                                         int32_t num_query_tokens, float sm_scale,
                                         int32_t split_tokens, int32_t max_seq_len,
                                         void *workspace, size_t workspace_bytes, void *out,
                                         uint8_t *flags, uint32_t options, void *stream);

/*
 * Step graphs: one decode step of a stack of attention layers captured once
 * as a CUDA graph and replayed with a single launch.  The Infire page ("How
 * we built the most efficient inference engine for Cloudflare's network",
 * section "Rust-precise CUDA kernels", 2nd paragraph) keeps one graph per
 * batch size, built on first use and cached, because one graph launch costs
 * less than the kernel launches it replaces; a caller does the same with one
 * pfkv_step_graph per batch size.
 *
 * A graph records, for every layer in order, pfkv_kv_append (when the layer
 * has new tokens) followed by the attention call (with the separate or the
 * fused tag check), exactly as the direct calls would enqueue them, with the
 * pointers and sizes given at creation.  Replaying it reads the CURRENT
 * contents of every buffer (q, new rows, positions, lengths, tables, tags,
 * pools), so a caller rewrites those buffers in place between steps.  The
 * launch configuration is fixed at creation: lengths must stay within
 * max_seq_len (longer ones are flagged PFKV_FLAG_BAD_LENGTH), and a new batch
 * size or pool needs a new graph.  All layers share the tables, lengths,
 * positions and workspace; the workspace must not be used concurrently.
 */
typedef struct {
    pfkv_cache cache;            /* this layer's pool                               */
    const void *q;               /* bf16 [batch][num_q_heads][head_dim]             */
    const void *k_new, *v_new;   /* bf16 [batch][num_kv_heads][num_new_tokens][head_dim];
                                    both NULL: this layer appends nothing          */
    void *out;                   /* bf16 [batch][num_q_heads][head_dim]             */
    uint8_t *flags;              /* attention flags of this layer, or NULL          */
} pfkv_layer;

typedef struct pfkv_step_graph pfkv_step_graph;  /* opaque */

/*
 * pfkv_step_graph_create -- capture the step for `layers` (host array of
 * num_layers >= 1 entries) into *graph (host).  Arguments are those of
 * pfkv_kv_append (positions, new_lens, num_new_tokens, append_flags) and of
 * pfkv_paged_decode_attn (the rest), shared by every layer; `options` is 0 or
 * PFKV_STAGE_FUSED_TAGS.  Every argument check of the direct calls is made
 * here, for every layer, and its status returned (nothing is captured then).
 * The capture uses a private stream; nothing runs on the device.
 */
pfkv_status pfkv_step_graph_create(const pfkv_layer *layers, int32_t num_layers,
                                   const pfkv_pages *pages, const int32_t *positions,
                                   const int32_t *new_lens, int32_t num_new_tokens,
                                   uint8_t *append_flags, int32_t num_q_heads, float sm_scale,
                                   int32_t split_tokens, int32_t max_seq_len, void *workspace,
                                   size_t workspace_bytes, uint32_t options,
                                   pfkv_step_graph **graph);

/* pfkv_step_graph_launch -- enqueue one step (all layers) on `stream`. */
pfkv_status pfkv_step_graph_launch(pfkv_step_graph *graph, void *stream);

/* pfkv_step_graph_destroy -- free the graph (NULL is a no-op).  The caller
 * makes sure no launch of it is still running. */
pfkv_status pfkv_step_graph_destroy(pfkv_step_graph *graph);

/*
 * pfkv_selftest_bounded_wait -- runs the bounded device-side wait that every
 * kernel of the library uses on its shared-memory barriers, twice, in one
 * warp: first on a barrier phase that nothing completes, which must give up
 * after the library's wait limit (100 ms) instead of hanging; then on a phase
 * that completes, which must succeed.  *result (device, 4-byte aligned)
 * receives PFKV_FLAG_DEVICE_TIMEOUT if the first wait gave up, | 0x100 if the
 * second one succeeded: 0x108 on a working device.  The context stays usable.
 * (A check of the failure path, not part of the method.)
 */
pfkv_status pfkv_selftest_bounded_wait(uint32_t *result, void *stream);

/*
 * pfkv_e4m3_encode -- out[i] = e4m3 code of x[i] (fp32), round to nearest
 * even, saturating to +-448, NaN -> 0x7F: the conversion kv_append uses.
 * x: fp32 [n], out: uint8 [n] (device).  n >= 0.
 */
pfkv_status pfkv_e4m3_encode(const float *x, int64_t n, uint8_t *out, void *stream);

/*
 * pfkv_e4m3_decode -- out[i] = value of e4m3 code codes[i] (fp32, exact; NaN
 * for 0x7F/0xFF): the conversion the attention kernel uses.
 * codes: uint8 [n], out: fp32 [n] (device).  n >= 0.
 */
pfkv_status pfkv_e4m3_decode(const uint8_t *codes, int64_t n, float *out, void *stream);

/* Static, NUL-terminated description of a status code. */
const char *pfkv_status_string(pfkv_status status);

/* ABI version of this header (incremented on incompatible changes). */
#define PFKV_ABI_VERSION 1
int32_t pfkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PFKV_H */
