/*
 * bip.h -- batch-invariant paged prefill attention for GB300 (sm_103a).
 *
 * One operation: causal, GQA, paged-KV prefill attention whose output rows
 * are bit-identical however the batch is composed.  A request served from a
 * radix-cache prefix hit sends only its uncached tail rows
 * (q_len = seq_len - prefix_len; sglang PR 46351, "Root cause"); those rows
 * get `out` and `lse` bit-identical to the same rows of the full prefill of
 * the prompt, whatever the other requests, q_len, page placement or plan
 * policy.  The prior-art failure this removes: a tile size chosen from the
 * batch-average packed q length changes the softmax reduction order
 * (sglang PR 46351, "Root cause", and kahyunnam's review comment).
 *
 * Semantics (sglang PR 46351, jbymy2000's reply, "Tail alignment"): local q
 * row i of a request sits at sequence position i + kv_len - q_len and sees
 * keys 0..position (the diagonal is included).  Query head h reads KV head
 * h / (num_qo_heads / num_kv_heads).  Scores are q.k / sqrt(head_dim);
 * lse is the natural-log log-sum-exp of those scores.
 *
 * Numerics contract (fixed at compile time; no run-time knob changes bits):
 * keys are cut at absolute positions into blocks of BN (128 for head_dim
 * 128, 64 for head_dim 256) and segments of 4096 keys (the fixed 4096-token
 * KV split of the model-serving-minefield issue 73 correction, item 2).
 * Blocks are visited in ascending order inside a segment with an fp32 online
 * softmax; segments are merged in ascending order with one merge formula,
 * whether one CTA folds them or several CTAs write partials that a merge
 * kernel combines.  Each row's arithmetic depends only on its own q row and
 * on K/V at positions <= its own.
 *
 * Ownership: the caller owns every device buffer and the stream.  A plan
 * owns host copies of its work list (pinned and mapped into the device's
 * address space when a CUDA device is present: each call's upload reads it
 * from the GPU) and is immutable after creation; one plan may serve many
 * bip_prefill calls (one per layer) with the same lengths and shapes.
 *
 * Errors: every entry point returns a status and never aborts or exits the
 * process (the model-serving-minefield issue 73 correction: a fixed 2 GiB
 * workspace overflow killed the whole server).
 */
#ifndef BIP_H_
#define BIP_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bip_status {
  BIP_OK = 0,
  BIP_ERR_INVALID_ARG = 1,          /* malformed lengths, pointers, sizes */
  BIP_ERR_UNSUPPORTED = 2,          /* a valid request this library does not run */
  BIP_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below the plan's need */
  BIP_ERR_CUDA = 4,                 /* a CUDA runtime call failed */
  BIP_ERR_DEVICE_TIMEOUT = 5,       /* a bounded in-kernel wait gave up */
  BIP_ERR_OUT_OF_MEMORY = 6,        /* host allocation failed */
  BIP_ERR_BAD_PAGE_INDEX = 7        /* a kv_indices entry outside [0, num_pages) */
} bip_status;

typedef enum bip_kv_dtype {
  BIP_KV_BF16 = 0,
  BIP_KV_FP8_E4M3 = 1 /* OCP E4M3 pages, decoded to f16 operands in the kernel */
} bip_kv_dtype;

/* How multi-segment units are scheduled.  Numerically neutral: every policy
 * gives identical bits (tested). */
typedef enum bip_split_policy {
  BIP_SPLIT_AUTO = 0,   /* split long units into per-segment partials only when
                           there are too few units to fill the GPU */
  BIP_SPLIT_NEVER = 1,  /* every unit folds its segments in one CTA */
  BIP_SPLIT_ALWAYS = 2  /* split every multi-segment unit the budget allows */
} bip_split_policy;

typedef struct bip_plan_options {
  bip_split_policy split_policy; /* default BIP_SPLIT_AUTO */
  size_t split_budget_bytes;     /* cap on partial-state bytes; default 256 MiB */
  int32_t num_sms;               /* CTAs to fill; 0 = query the current device */
  uint64_t wait_limit_ns;        /* bound on every in-kernel wait; 0 = 4 s.  Counted in SM clock
                                    cycles at the device's peak clock, so at lower clocks a wait
                                    runs proportionally longer before it gives up */
  int32_t tiles_per_unit;        /* q tiles per CTA: 0 = auto, 1, or 2 (head_dim 128 only);
                                    numerically neutral (tested) */
  int32_t window_left;           /* sliding window: 0 = none (every earlier key is visible);
                                    W > 0: the row at position p sees keys p - W .. p only
                                    (sliding-window KV, a mask case of sglang PR 46351, "Fix") */
} bip_plan_options;

typedef struct bip_plan_info {
  int32_t batch, total_q, num_qo_heads, num_kv_heads, head_dim, page_size, kv_dtype;
  int32_t gqa_group;       /* num_qo_heads / num_kv_heads */
  int32_t tile_positions;  /* q positions per 128-row tile: floor(128 / gqa_group) */
  int32_t kv_block;        /* keys per block (BN) */
  int32_t split_len;       /* keys per segment (4096) */
  int32_t num_units;       /* (request, kv head, tiles_per_unit q tiles) units */
  int32_t num_items;       /* attention work items (units, or their segments) */
  int32_t num_split_units; /* units computed as per-segment partials + merge */
  int32_t grid;            /* CTAs of the persistent attention kernel */
  int32_t tiles_per_unit;  /* q tiles a unit (and a CTA) carries at once: 2 (d 128) or 1 */
  int64_t partial_rows;    /* rows of fp32 partial state (m, l, o[head_dim]) */
  int64_t kv_blocks;       /* KV blocks streamed, summed over items */
  uint64_t workspace_bytes;
  uint64_t partial_bytes;
  uint64_t scratch_bytes;  /* per-CTA fold state */
  uint64_t upload_bytes;   /* host->device bytes each bip_prefill copies */
} bip_plan_info;

typedef struct bip_plan_s* bip_plan_t;

/* Human-readable name of a status (static storage). */
const char* bip_status_string(bip_status s);

/* Upper bound of bip_plan's workspace_bytes for any batch with at most
 * max_batch requests and max_total_q q rows, any KV lengths, the given
 * heads/head_dim, and a split budget of at most split_budget_bytes.
 * Allocate this once and reuse it.  Returns 0 for unsupported shapes.
 * Host only; no device work. */
size_t bip_workspace_bound(int32_t max_batch, int32_t max_total_q, int32_t num_qo_heads,
                           int32_t num_kv_heads, int32_t head_dim, size_t split_budget_bytes);

/* Build a plan from HOST arrays (copied; the caller may free them after):
 *   qo_indptr[batch+1]      exclusive prefix sum of q rows, qo_indptr[0] = 0
 *   kv_indptr[batch+1]      exclusive prefix sum of pages,  kv_indptr[0] = 0
 *   kv_last_page_len[batch] valid slots of each request's last page,
 *                           1..page_size when it has pages
 * kv_len = (pages - 1) * page_size + last_page_len (0 with no pages);
 * 0 <= q_len <= kv_len is required; q_len = 0 is legal and yields no rows.
 * Supported now: head_dim 128 or 256, gqa_group <= 128, page_size a power of
 * two in [1, BN] (1 = a token-granular pool; below 8 the kernel gathers
 * token rows instead of whole pages, with the same bits), kv_dtype
 * BIP_KV_BF16 or BIP_KV_FP8_E4M3 (two q tiles per CTA exist at head_dim 128
 * with pages of 8 or more slots; tiles_per_unit = 2 elsewhere returns
 * BIP_ERR_UNSUPPORTED).
 * opts may be NULL (defaults).  On success *plan owns the result and
 * *workspace_bytes (if not NULL) receives the exact workspace size, never
 * above bip_workspace_bound for the same shapes.  No device work except a
 * pinned host allocation and an SM-count query when a device is present. */
bip_status bip_plan(bip_plan_t* plan, const int32_t* qo_indptr, const int32_t* kv_indptr,
                    const int32_t* kv_last_page_len, int32_t batch, int32_t num_qo_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                    bip_kv_dtype kv_dtype, const bip_plan_options* opts, size_t* workspace_bytes);

bip_status bip_plan_get_info(bip_plan_t plan, bip_plan_info* info);

/* Work items in launch order, 8 int32 each:
 *   request, kv_head, q_tile, seg_lo, seg_hi, split (0/1), kv_blocks, tile_mask
 * The item carries tiles q_tile + t for every bit t of tile_mask; tile u of
 * a request covers sequence positions kv_len - q_len + [u * tile_positions,
 * (u + 1) * tile_positions), clipped at kv_len (tiles count from the
 * request's first new row, so q_len rows take ceil(q_len / tile_positions)
 * tiles).
 * Writes at most capacity items; *count receives the total. */
bip_status bip_plan_get_items(bip_plan_t plan, int32_t* items, int32_t capacity, int32_t* count);

/* Release a plan.  Calls enqueued with it read its pinned host image when
 * they run, so this first waits (on the host) for every call that was
 * enqueued eagerly with the plan to complete.  A CUDA graph that captured a
 * call reads the image again at each replay: destroy the plan only after
 * the last replay of every such graph has completed. */
bip_status bip_plan_destroy(bip_plan_t plan);

/* Enqueue the attention on `stream`; never synchronizes.  DEVICE pointers:
 *   q        bf16 [num_q_rows, num_qo_heads, head_dim], rows contiguous;
 *            num_q_rows must equal qo_indptr[batch] (the shape check the
 *            paged wrapper of sglang PR 46351 raised, Woody-Hu's report)
 *   k_pages, v_pages  [num_pages, page_size, num_kv_heads, head_dim] (NHD),
 *            bf16 (or E4M3 bytes); page p starts at p * page_stride_elems
 *            elements, slots and heads contiguous inside a page
 *   kv_indices int32 [kv_indptr[batch]] page ids, each in [0, num_pages)
 *   out      bf16 [num_q_rows, num_qo_heads, head_dim]
 *   lse      fp32 [num_q_rows, num_qo_heads], natural log
 *   workspace  >= the plan's workspace_bytes, 256-byte aligned; its first
 *            bytes receive this call's work list and a status word, copied
 *            on `stream` by a small kernel that reads the plan's pinned,
 *            mapped host image (so the call never waits behind bulk copies
 *            that other streams have queued on the copy engines).
 * q, pages and out must be 16-byte aligned; page_stride_elems * element size
 * must be a multiple of 16 bytes (and, for page sizes below 8, below 2^31
 * bytes, else BIP_ERR_UNSUPPORTED).  k_scale multiplies the logits (folded
 * into the softmax scale) and v_scale the output; use 1.0 for bf16 pages.
 * Both must be finite, else BIP_ERR_INVALID_ARG.  Page slots at or beyond a
 * request's kv_len may hold anything (NaN too).  Calls sharing one workspace
 * must be ordered on the GPU. */
bip_status bip_prefill(bip_plan_t plan, const void* q, int64_t num_q_rows, const void* k_pages,
                       const void* v_pages, int64_t num_pages, int64_t page_stride_elems,
                       const int32_t* kv_indices, float k_scale, float v_scale, void* out,
                       float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* bip_prefill under a per-row custom mask: custom masks are one of the cases
 * the padding skipped (sglang PR 46351, "Fix").  The mask narrows the causal
 * rule (and the plan's sliding window): key j of a request is visible to one
 * of its q rows when j <= the row's position, the window allows it, and the
 * row's mask bit j is set.  Bits for keys past the row's position are never
 * read.  A row left with no visible key gets out = 0 and lse = -inf.
 *   mask     DEVICE uint32 words, 4-byte aligned: q row r (the row of q, over
 *            the whole batch) owns words [r * mask_row_words, (r + 1) *
 *            mask_row_words); bit j % 32 (least significant first) of word
 *            j / 32 is key j of the row's request
 *   mask_row_words  >= ceil(kv_len / 32) for every request with q rows, else
 *            BIP_ERR_INVALID_ARG
 * Every other argument, the contract and the errors as for bip_prefill.  A row
 * depends on its q row, its keys and its own mask row only: a radix-cache hit
 * whose tail rows carry the same mask rows as the full prefill gets the same
 * bits.  Blocks a mask leaves empty are still visited (the work list does not
 * depend on the mask). */
bip_status bip_prefill_masked(bip_plan_t plan, const void* q, int64_t num_q_rows, const void* k_pages,
                              const void* v_pages, int64_t num_pages, int64_t page_stride_elems,
                              const int32_t* kv_indices, const uint32_t* mask, int64_t mask_row_words,
                              float k_scale, float v_scale, void* out, float* lse, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/* Write each request's new K/V rows into its pages: the paged KV append that
 * precedes the attention of an extend: on a radix-cache prefix hit only the
 * uncached tail is computed and its K/V join the cached pages (sglang PR 46351,
 * "Motivation"); the FP8 E4M3 cache is the --kv-cache-dtype fp8_e4m3 setup of
 * the model-serving-minefield issue 73 report, "What were you serving".
 * The plan supplies the batch: request r's rows [qo_indptr[r], qo_indptr[r+1])
 * of k_new / v_new go to sequence positions kv_len_r - q_len_r .. kv_len_r - 1,
 * position p in page kv_indices[kv_indptr[r] + p / page_size], slot
 * p % page_size.  DEVICE pointers:
 *   k_new, v_new  bf16 [num_new_rows, num_kv_heads, head_dim], contiguous;
 *            num_new_rows must equal qo_indptr[batch]
 *   k_pages, v_pages  the pools bip_prefill reads (NHD, page stride as there),
 *            written in place; only the new rows' slots are touched
 *   kv_indices int32 page ids, each in [0, num_pages); others are counted
 *            (bip_read_device_status reports BIP_ERR_BAD_PAGE_INDEX) and skipped
 *   workspace  any buffer good for bip_prefill (only its first bytes are used);
 *            its first bytes receive the plan's tables and a status word.
 * bf16 pages receive the bits unchanged (k_scale and v_scale must be 1.0).
 * E4M3 pages receive e4m3(x / scale): x widened to float32, divided by the
 * scale with IEEE rounding, rounded to the nearest E4M3 value (ties to even)
 * and saturated at +-448; scales must be positive and finite.  Rows, pages
 * and the workspace must be 16-byte aligned.  Enqueued on `stream`; never
 * synchronizes.  Calls sharing a workspace must be ordered on the GPU. */
bip_status bip_append_kv(bip_plan_t plan, const void* k_new, const void* v_new, int64_t num_new_rows,
                         void* k_pages, void* v_pages, int64_t num_pages, int64_t page_stride_elems,
                         const int32_t* kv_indices, float k_scale, float v_scale, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/* ---- graph-replayable launches
 * A captured CUDA graph fixes its kernels' arguments, so the batch must come
 * from device memory and the work list must be built on the device (sglang
 * PR 46351: the full prefill CUDA graph keeps a static q buffer for the
 * captured token count, Woody-Hu's follow-up; a radix hit and the full
 * recompute of a prompt usually land in different captured buckets,
 * jbymy2000's correction).  A graph plan fixes only capacities and shapes;
 * bip_prefill_graph plans on the device from the indptr arrays each launch:
 * a batch of few units (fewer than 8 per CTA, e.g. short extends behind long
 * prefixes) has its multi-segment units split by segment, with partial
 * states and a merge launch, when they fit the plan's capacities; any other
 * batch folds every unit in one CTA.  Since no plan choice enters a row's
 * arithmetic, the results are the bits of bip_prefill for the same batch,
 * in any bucket. */
typedef struct bip_graph_plan_s* bip_graph_plan_t;

/* Capacities: batches of at most max_batch requests with at most
 * max_total_q q rows in all.  Heads, head_dim, page_size, kv_dtype as for
 * bip_plan; opts: num_sms, wait_limit_ns, tiles_per_unit and window_left
 * apply; split_policy BIP_SPLIT_AUTO (default) lets short batches split
 * within split_budget_bytes of partial states (default 64 MiB without
 * opts), BIP_SPLIT_NEVER folds every unit, BIP_SPLIT_ALWAYS is refused.
 * *workspace_bytes receives the fixed workspace size.  Host only; no device
 * work. */
bip_status bip_graph_plan(bip_graph_plan_t* plan, int32_t max_batch, int32_t max_total_q, int32_t num_qo_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t page_size, bip_kv_dtype kv_dtype,
                          const bip_plan_options* opts, size_t* workspace_bytes);

/* Enqueue a device-planned prefill on `stream` with no host-to-device copy
 * and no synchronisation: safe to capture in a CUDA graph and replay with
 * new contents in the same buffers.  DEVICE pointers:
 *   qo_indptr [batch + 1], kv_indptr [batch + 1], kv_last_page_len [batch]
 *            int32, read when the launch runs; batch <= max_batch is the
 *            launch's (host) request count, padding requests may have q_len 0
 *   q, out   [max_total_q, num_qo_heads, head_dim] bf16 buffers; rows past
 *            qo_indptr[batch] are not written
 *   lse      fp32 [max_total_q, num_qo_heads]
 *   pages, kv_indices, scales as for bip_prefill
 *   workspace >= the graph plan's workspace_bytes, 256-byte aligned.
 * Arguments checked on the device (indptr monotone from 0, last-page lengths,
 * q_len <= kv_len, qo_indptr[batch] <= max_total_q) set the status word to
 * BIP_ERR_INVALID_ARG and the launch computes nothing; read it with
 * bip_read_device_status.  The first launch per variant may set a kernel
 * attribute: make one before capturing. */
bip_status bip_prefill_graph(bip_graph_plan_t plan, int32_t batch, const int32_t* qo_indptr,
                             const int32_t* kv_indptr, const int32_t* kv_last_page_len, const void* q,
                             const void* k_pages, const void* v_pages, int64_t num_pages, int64_t page_stride_elems,
                             const int32_t* kv_indices, float k_scale, float v_scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* bip_prefill_graph under a custom mask (the bip_prefill_masked contract):
 * mask is a DEVICE array of mask_row_words 32-bit words per q buffer row,
 * read when the launch runs; a request with rows whose kv_len exceeds
 * 32 * mask_row_words sets the status word to BIP_ERR_INVALID_ARG and the
 * launch computes nothing. */
bip_status bip_prefill_graph_masked(bip_graph_plan_t plan, int32_t batch, const int32_t* qo_indptr,
                                    const int32_t* kv_indptr, const int32_t* kv_last_page_len, const void* q,
                                    const void* k_pages, const void* v_pages, int64_t num_pages,
                                    int64_t page_stride_elems, const int32_t* kv_indices, const uint32_t* mask,
                                    int64_t mask_row_words, float k_scale, float v_scale, void* out, float* lse,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Release a graph plan (host memory only). */
bip_status bip_graph_plan_destroy(bip_graph_plan_t plan);

/* Size of the device array that bip_prefill_no_alloc uses as its workspace. */
#define BIP_NO_ALLOC_WORKSPACE_BYTES ((size_t)32 << 20)

/* No counterpart on the pages: an entry point for callers that cannot allocate
 * device memory -- an engine plugin whose host framework owns the GPU's memory
 * through its own pool and gives the plugin no allocation hook, or a serving
 * loop that forbids allocation on the request path.  Same as bip_prefill, but
 * the workspace is a file-scope device array of BIP_NO_ALLOC_WORKSPACE_BYTES
 * inside this library, which every GPU that loads the library holds until
 * the process exits; the caller still passes inputs and outputs.  Allocates
 * nothing: no cudaMalloc, cudaFree or allocating library routine.
 *   - Plans whose workspace_bytes exceed the array return
 *     BIP_ERR_WORKSPACE_TOO_SMALL (a smaller split_budget_bytes makes a plan fit).
 *   - Uses the current device; the stream and buffers must belong to it.  The
 *     first call on a device looks up the array's device address with that
 *     device current (it may load the module): make it before any stream capture.
 *     The address is kept for the life of the process; calls after a
 *     cudaDeviceReset of that device are not supported.
 *   - Every call shares the one array, which keeps the last call's contents:
 *     calls whose work overlaps on the GPU race, so order them (one stream, or
 *     events).  Each call rewrites the status word at the head of the array
 *     before its kernels run, so nothing needs clearing between calls.  The
 *     array is private, so bip_read_device_status cannot read that word: a
 *     bounded wait that expires still returns early and leaves out/lse undefined. */
bip_status bip_prefill_no_alloc(bip_plan_t plan, const void* q, int64_t num_q_rows, const void* k_pages,
                                const void* v_pages, int64_t num_pages, int64_t page_stride_elems,
                                const int32_t* kv_indices, float k_scale, float v_scale, void* out,
                                float* lse, cudaStream_t stream);

/* Synchronize `stream` and read the status word the last bip_prefill on this
 * workspace left: BIP_OK, BIP_ERR_DEVICE_TIMEOUT (a bounded wait expired; the
 * kernel returned early and its outputs are undefined) or
 * BIP_ERR_BAD_PAGE_INDEX (an out-of-range page id was read as zeros). */
bip_status bip_read_device_status(const void* workspace, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BIP_H_ */
