/*
 * pie_attn.h -- C ABI of a paged-KV attention library for GB300 (sm_103a).
 *
 * The library keeps the KV state of many working sets in a pool of 16-token
 * pages and runs the per-layer attention step of a batched forward pass over
 * them: ops.attn.kv_append followed by attend / prefill ("Poem ops",
 * Operations table, row ops.attn).  Working sets follow "How Pie thinks",
 * section 4 "Working sets": a frozen prefix of committed tokens plus a
 * writable buffer of uncommitted (e.g. speculative) tokens; fork shares the
 * frozen prefix without copying it; frozen pages are deduplicated across
 * requests.  The runtime packs passes of many working sets into shared
 * kernel launches ("How Pie thinks", "Batching is still the engine's job"):
 * one pie_batch covers every segment of a pass, and one pie_kv_append /
 * pie_attend call per layer covers every row of it.
 *
 * Conventions
 *  - Every call returns a pie_status: 0 = PIE_OK, negative = error.  A
 *    failed call changes no host state (working sets, pages, reference
 *    counts, the open batch); pie_last_error() then describes it.  A CUDA
 *    failure part-way through enqueuing device work (PIE_ERR_CUDA) may
 *    leave the work enqueued before it on the stream.
 *  - Handles are opaque.  A context is not thread-safe: one host thread at a
 *    time.
 *  - Device pointers passed in are owned by the caller and only borrowed for
 *    stream-ordered use on the context's stream; no call synchronises that
 *    stream except where stated (pie_ctx_destroy, buffer growth in
 *    pie_batch_begin).
 *  - Device pools, K, V, Q and output arrays must be 16-byte aligned (any
 *    CUDA allocation is, and so is every row of a contiguous [rows][heads][d]
 *    array); LSE arrays, block tables and row lengths 4-byte aligned.  The
 *    kernels move them in 16-byte vectors and bulk copies; a call given a
 *    misaligned pointer returns PIE_ERR_INVALID and launches nothing.
 *  - All device work of a context is ordered on its stream, in call order
 *    (pie_attend may run part of a pass on a second stream the context owns,
 *    forked from and joined back into that stream within the call).  The
 *    caller must keep pools, inputs and outputs alive until that work ends.
 *
 * KV pool layout (device memory owned by the caller, borrowed by the
 * context; K and V have separate pools of identical layout):
 *    pool[layer][page][kv_head][block],
 *    block = 16 * head_dim * esize bytes (esize 2 for bf16, 1 for e4m3).
 *  A block is cut along the head dimension into panels of 128 bytes per key:
 *  panel p holds bytes [p*128, p*128+128) of every key's head vector and
 *  occupies block bytes [p*2048, p*2048+2048).  Within a panel, the 16-byte
 *  chunk c of key slot s (s = position % 16) is stored at byte
 *  s*128 + 16*(c ^ (s % 8)).  head_dim * esize must be a multiple of 128
 *  (bf16: head_dim 64 or 128; e4m3: head_dim 128).  bf16 elements are their
 *  little-endian bit patterns; e4m3 elements (OCP FP8 E4M3) are
 *  round-to-nearest-even, saturating encodings of float32(x) * float32(1 /
 *  scale[layer][kv_head]).
 *  The pools must be initialised (zeroed, say) before first use: the
 *  kernels read whole pages, and slots past a working set's length enter
 *  the tensor-core products with zero weight, so a non-finite value there
 *  would turn the result into NaN.  Slots the library writes always hold
 *  the appended (finite) values or copies of them.
 */
#ifndef PIE_ATTN_H
#define PIE_ATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t pie_status;
enum {
  PIE_OK = 0,
  PIE_ERR_INVALID = -1,    /* bad argument or configuration */
  PIE_ERR_BAD_HANDLE = -2, /* unknown working set or batch */
  PIE_ERR_NO_PAGES = -3,   /* the page pool cannot cover the pass */
  PIE_ERR_RANGE = -4,      /* freeze / rollback beyond the writable buffer */
  PIE_ERR_CUDA = -5,       /* a CUDA runtime call failed */
  PIE_ERR_STATE = -6       /* call not allowed in the current state */
};

enum { PIE_KV_BF16 = 0, PIE_KV_E4M3 = 1 };

typedef int32_t pie_ws;            /* working-set handle, > 0 */
typedef struct pie_ctx pie_ctx;
typedef struct pie_batch pie_batch;

typedef struct pie_config {
  int32_t num_layers;    /* layers sharing one page id space ("fold_layers") */
  int32_t num_q_heads;   /* Hq */
  int32_t num_kv_heads;  /* Hkv; Hq must be a multiple (grouped-query heads) */
  int32_t head_dim;      /* d */
  int32_t page_size;     /* must be 16 */
  int32_t kv_dtype;      /* PIE_KV_BF16 or PIE_KV_E4M3 */
  int32_t num_pages;     /* pages in each pool */
  int32_t num_sms;       /* SMs to plan for; 0 = query the device (152 when
                            k_pool is NULL) */
  const int32_t* free_list; /* host, nullable, copied: initial order of the
                               free-page stack, a permutation of
                               0..num_pages-1, first entry allocated first;
                               NULL = ascending */
  const float* k_scale;  /* host, copied, [num_layers*num_kv_heads]; e4m3 only:
                            dequantised K = code * k_scale[layer][kv_head] */
  const float* v_scale;  /* likewise for V */
  void* k_pool;          /* device, borrowed, layout above; NULL together with
                            v_pool = plan-only context (host state only, no
                            device work; pie_kv_append / pie_attend fail) */
  void* v_pool;
  void* stream;          /* cudaStream_t, borrowed; NULL = legacy default.
                            The context also creates one non-blocking stream
                            of its own: in a pass with both decode-kernel and
                            tensor-core items, pie_attend runs the decode
                            launch there, forked from and joined back into
                            `stream` by events within the call */
  float logit_softcap;   /* ops.attn.logit_softcap ("Poem ops"): c > 0 replaces
                            every scaled score s by c * tanh(s / c) before the
                            softmax (the LSE is over the capped scores);
                            0 = no cap; negative or non-finite is
                            PIE_ERR_INVALID */
  float rope_theta;      /* > 1: the context builds the rotary table of
                            pie_rope_table(rope_theta, head_dim,
                            rope_max_positions) on the device for
                            pie_kv_append_rope; 0 = none */
  int32_t rope_max_positions; /* positions the table covers (rope_theta > 0) */
} pie_config;

/* One segment of a pass: n_new new tokens of working set ws.  token_ids
 * (host, nullable, n_new entries) are recorded for prefix dedup; NULL means
 * unknown, and pages holding unknown tokens are never deduplicated. */
typedef struct pie_seg {
  pie_ws ws;
  int32_t n_new;
  const int32_t* token_ids;
} pie_seg;

/* Context: the KV space of one model's attention layers and the working
 * sets over it.  The per-layer, per-KV-head K and V caches follow "Write a
 * model in Poem", section 4 "State (caches)"; one page id space shared by
 * all layers follows fold_layers ("Write a model in Poem", section 5
 * "Forward pass"); grouped-query heads follow "Write a model in Poem",
 * "Shared building blocks"; the e4m3 cache follows the FP8 deployments of
 * "Write a model in Poem", section 2 "Deployments".
 * Copies the configuration; when k_pool is set, allocates its device
 * buffers (scales, the rotary table when rope_theta > 0, the plan, partial
 * results) with cudaMalloc and creates a second stream and two events of
 * its own.  PIE_ERR_INVALID for: a non-positive count, page_size != 16,
 * Hq not a multiple of Hkv, Hq/Hkv not a power of two <= 64, head_dim not
 * 64 or 128 (bf16) or 128 (e4m3), only one of k_pool / v_pool, missing or
 * non-positive e4m3 scales, a free_list that is not a permutation, a
 * negative or non-finite logit_softcap, or rope_theta in (0, 1].
 * PIE_ERR_CUDA if a device allocation fails (nothing is kept). */
pie_status pie_ctx_create(const pie_config* cfg, pie_ctx** out);
/* Synchronises the streams, frees everything the context allocated. */
pie_status pie_ctx_destroy(pie_ctx* ctx);
const char* pie_last_error(const pie_ctx* ctx);

/* ---- working sets ("How Pie thinks", section 4; host state only) ----
 * Not allowed while a batch is open (PIE_ERR_STATE). */

/* New empty working set; handles count up from 1 and are never reused. */
pie_status pie_ws_create(pie_ctx* ctx, pie_ws* out);
/* Releases every page reference, highest logical page first. */
pie_status pie_ws_destroy(pie_ctx* ctx, pie_ws ws);
/* New working set holding the parent's frozen tokens only, sharing their
 * pages (reference count + 1, no copy).  A shared partial page is copied
 * lazily by the first pass that writes into it. */
pie_status pie_ws_fork(pie_ctx* ctx, pie_ws parent, pie_ws* child);
/* Commits the first n writable tokens (all when n < 0).  Pages that become
 * fully frozen with known token ids are registered for dedup under
 * (previous page, token ids) when the previous page is registered or this is
 * page 0, unless that key is present.  n > writable: PIE_ERR_RANGE. */
pie_status pie_ws_freeze(pie_ctx* ctx, pie_ws ws, int32_t n);
/* Drops the last n writable tokens ("speculative drafts that you might roll
 * back") and releases emptied pages, highest first.  n > writable:
 * PIE_ERR_RANGE. */
pie_status pie_ws_rollback(pie_ctx* ctx, pie_ws ws, int32_t n);
/* Dedup lookup for an EMPTY working set: shares the registered pages whose
 * token ids match token_ids[0..n) page by page from the start; the matched
 * tokens become frozen.  *n_reused = matched tokens (a multiple of 16). */
pie_status pie_ws_match_prefix(pie_ctx* ctx, pie_ws ws, const int32_t* token_ids,
                               int32_t n, int32_t* n_reused);
/* Introspection of the working-set state of "How Pie thinks", section 4
 * (tokens, the frozen prefix, and the pages holding them; fork and dedup
 * share pages, so a page's reference count is the number of working sets
 * whose table holds it).  Host only; any output pointer may be NULL.
 * Unknown handle: PIE_ERR_BAD_HANDLE. */
pie_status pie_ws_info(const pie_ctx* ctx, pie_ws ws, int32_t* n_tokens,
                       int32_t* n_frozen, int32_t* n_pages);
/* Copies up to cap physical page ids (logical order) into out; *n = count. */
pie_status pie_ws_page_table(const pie_ctx* ctx, pie_ws ws, int32_t* out,
                             int32_t cap, int32_t* n);
/* Reference count of a page (0 = free); page out of range: PIE_ERR_INVALID. */
pie_status pie_page_refcount(const pie_ctx* ctx, int32_t page, int32_t* rc);
pie_status pie_free_pages(const pie_ctx* ctx, int32_t* n_free);

/* ---- one batched pass ----
 * The runtime packs the passes of many working sets into shared kernel
 * launches ("How Pie thinks", "Batching is still the engine's job"), and
 * the plan of a pass is built once for all layers (ops.attn.plan_prefill in
 * "Poem ops", Operations table; fold_layers in "Write a model in Poem",
 * section 5).  New tokens enter a working set's writable buffer ("How Pie
 * thinks", section 4).
 * Rows are the new tokens of all segments, in segment order, then token
 * order.  Each working set may appear once.  Reserves a slot for every row
 * (allocating pages segment by segment, token by token; a write into a
 * shared page first copies it), builds the attention plan (per-row page
 * tables and positions, fork/dedup groups, KV splits), uploads it with one
 * host-to-device copy and enqueues the copy-on-write page copies on the
 * stream.  The new tokens become writable tokens of their working sets.
 * Fails with PIE_ERR_NO_PAGES, changing nothing, if the pool cannot cover
 * the whole pass.  Fails with PIE_ERR_CUDA if a device buffer cannot grow
 * or the upload or the page-copy launch cannot be enqueued; the slots it
 * had reserved are released again and the host state is as before the
 * call.  One batch may be open per context. */
pie_status pie_batch_begin(pie_ctx* ctx, const pie_seg* segs, int32_t n_segs,
                           pie_batch** out);
/* Number of rows of the batch. */
pie_status pie_batch_rows(const pie_batch* b, int32_t* n_rows);
/* Host copies of the per-row position and slot (page * 16 + position % 16). */
pie_status pie_batch_slots(const pie_batch* b, int32_t* pos, int32_t* slot);
/* ops.attn.kv_append for one layer: k, v are device bf16 [n_rows][Hkv][d];
 * row r is written to its reserved slot in the pool (converted to e4m3 for
 * an e4m3 context). */
pie_status pie_kv_append(pie_ctx* ctx, pie_batch* b, int32_t layer,
                         const void* k, const void* v);
/* ops.elemwise.rope fused into ops.attn.kv_append ("Poem ops", Operations
 * table; the pages name the op without a formula, and the rotary embedding
 * of the Llama family is taken): for each row at position p, dimension i <
 * d/2 of a head pairs with i + d/2 and both turn by the angle p * w_i,
 * w_i = rope_theta^(-2i/d):
 *     y_i = x_i cos - x_{i+d/2} sin,   y_{i+d/2} = x_{i+d/2} cos + x_i sin,
 * with (cos, sin) from the context's table, each product and the sum in
 * float32 (no fused multiply-add), rounded to bf16.  K heads are rotated and
 * appended exactly as pie_kv_append would append the rotated bf16 rows (V is
 * appended unrotated); when q is non-NULL, q [n_rows][Hq][d] bf16 is rotated
 * into q_out (same layout; q_out may equal q) for the following pie_attend.
 * PIE_ERR_STATE if the context has no rotary table; PIE_ERR_RANGE, with
 * nothing launched, if a row position is >= rope_max_positions. */
pie_status pie_kv_append_rope(pie_ctx* ctx, pie_batch* b, int32_t layer, const void* k, const void* v,
                              const void* q, void* q_out);
/* Host: the rotary table, out [positions][head_dim/2][2] float = (cos, sin)
 * of p * theta^(-2i/head_dim), each computed in double and rounded to float.
 * theta > 1, head_dim even, positions > 0, else PIE_ERR_INVALID. */
pie_status pie_rope_table(float theta, int32_t head_dim, int32_t positions, float* out);

/* ops.attn.attend / prefill for one layer: q device bf16 [n_rows][Hq][d];
 * out device bf16 [n_rows][Hq][d]; lse device float [n_rows][Hq] (natural
 * log of the softmax denominator) or NULL.  Row r at position p of working
 * set w, query head h: softmax over keys 0..p of w, from KV head h / (Hq /
 * Hkv), of (q . k) / sqrt(d), applied to the values.  Requires that
 * pie_kv_append ran for this layer and batch first.
 * Precision: keys and values enter as stored (bf16, or the e4m3 code times
 * its scale); scores and sums are fp32; the softmax weights meet V as bf16
 * (bf16 pools) or f16 (e4m3 pools).  With an e4m3 pool, rows that take the
 * tensor-core path (prefill chunks, large fork groups) also round q to f16,
 * so |q| must stay below 65504 there.
 * Rows whose keys are split over several work items are combined from the
 * parts' (max, sum, partial output) as in "How Pie thinks", section 4 (the
 * shared prefix is attended once and its result combined with each
 * member's own pages): by the decode kernels themselves, the CTA that
 * stores a row's last part combining them (see pie_ctx_set_merge_mode),
 * or by a merge launch after the attention launches. */
pie_status pie_attend(pie_ctx* ctx, pie_batch* b, int32_t layer,
                      const void* q, void* out, float* lse);
/* How pie_attend combines split rows (the combination of partial results
 * under pie_attend, "How Pie thinks", section 4), for batches begun after
 * the call.  mode 0 (the default): a merge launch after the attention
 * launches.  mode 1: inside the decode launches, one launch per pie_attend,
 * when no tensor-core item of the batch is split (else a merge launch).
 * Merging inside holds each split CTA a few microseconds longer, to publish
 * its stores and count them; on one GB300, both modes in the same run, that
 * cost more than the merge launch: 2.1 % on a decode batch of 64 rows of
 * 32 q / 8 KV heads (2.9 MB of partials) and 1.4 % on one of 256 rows of
 * 64 q / 8 KV heads over e4m3 pages (23 MB).  PIE_ERR_INVALID for another
 * mode. */
pie_status pie_ctx_set_merge_mode(pie_ctx* ctx, int32_t mode);
/* Closes the batch.  Its device work stays enqueued on the stream. */
pie_status pie_batch_end(pie_ctx* ctx, pie_batch* b);

/* ---- decode attention that allocates nothing ----
 * The paper has no counterpart to this entry point; it is a convenience of
 * this library.  It serves callers that cannot call cudaMalloc: an engine
 * that reserved the GPU's memory for its own pool and allocator at start-up
 * (a library allocation would fail or fragment it), a serving loop that
 * cannot afford the device-wide synchronisation that cudaMalloc / cudaFree
 * may imply, or a plug-in whose host runtime forbids foreign allocations.
 * Such callers need no context (pie_ctx_create allocates): they pass the
 * pools, a per-row block table and the row lengths themselves.
 *
 * Decode attention for rows of one query token each, over bf16 pools in
 * the layout above: row r attends keys 0..seq_lens[r]-1 of its pages
 * block_table[r][0..], with the same softmax, head grouping and outputs as
 * pie_attend.  KV splits and their partial results live in one file-scope
 * device array of PIE_NOALLOC_SCRATCH_BYTES, which every GPU that loads the
 * library holds until the process exits.
 *  - Scratch needed, with R = num_rows and S = the KV splits the call picks
 *    (S >= 1): R*S*32 + 7*R*4 + (S > 1 ? R*S*Hq*(head_dim+2)*4 : 0) bytes
 *    plus alignment; the call lowers S to fit and returns PIE_ERR_RANGE,
 *    with nothing launched, when even S = 1 does not fit.
 *  - The splits are sized from max_pages_per_row, so keep it tight (the
 *    longest row's page count): a wider row stride gives every row more
 *    empty splits, which cost launch slots and merge reads but not accuracy.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address is kept for the process, so
 *    calls after a cudaDeviceReset (or any teardown of the device's primary
 *    context) are not supported.
 *  - Every call on a device shares the array and leaves its contents behind;
 *    nothing in it needs to start at zero, because each call writes every
 *    word it reads before reading it.  Calls that overlap on the GPU (other
 *    streams, other host threads) race on the array: order them.
 *  - No cudaMalloc, cudaFree or other allocating call is made.
 *  - Bounded waits inside the kernel end silently here (there is no context
 *    to carry an error word).
 *  - The caller guarantees 1 <= seq_lens[r] <= 16*max_pages_per_row and page
 *    ids < num_pages; they live on the device and are not checked. */
#define PIE_NOALLOC_SCRATCH_BYTES (16u << 20)
typedef struct pie_decode_args {
  int32_t num_rows;          /* rows (>= 0) */
  int32_t num_q_heads;       /* Hq */
  int32_t num_kv_heads;      /* Hkv; Hq/Hkv a power of two <= 64 */
  int32_t head_dim;          /* 64 or 128 */
  int32_t num_layers;        /* pool geometry */
  int32_t num_pages;
  int32_t layer;
  int32_t max_pages_per_row; /* row stride of block_table */
  const void* q;             /* device bf16 [num_rows][Hq][head_dim] */
  const void* k_pool;        /* device bf16 pools, layout above */
  const void* v_pool;
  const int32_t* block_table; /* device [num_rows][max_pages_per_row] */
  const int32_t* seq_lens;    /* device [num_rows] */
  void* out;                 /* device bf16 [num_rows][Hq][head_dim] */
  float* lse;                /* device [num_rows][Hq] or NULL */
  void* stream;              /* cudaStream_t, NULL = legacy default */
} pie_decode_args;
pie_status pie_attend_decode_noalloc(const pie_decode_args* args);

/* ---- introspection (tests, tools) ---- */
/* info[0..4] = decode-kernel items, tensor-core items, rows merged from
 * several partial results, copy-on-write page copies, and 1 when each
 * pie_attend of the batch ends with a merge launch, 0 when the decode
 * kernels merge the split rows themselves or no row is split. */
pie_status pie_batch_plan_info(const pie_batch* b, int32_t* info);
/* Copies work items (kind 0: decode kernel, 1: tensor-core kernel), 8 int32
 * each: first page index into the batch's page list, pages, first key
 * position, first row-list index, rows, part (-1 = direct output), keys,
 * and 1 when the item's rows are the consecutive batch rows starting at the
 * row-list index (the list is the identity there), else 0.  *n = total
 * items; at most cap are copied. */
pie_status pie_batch_items(const pie_batch* b, int32_t kind, int32_t* out, int32_t cap,
                           int32_t* n);
/* Synchronises the stream and returns (and clears) the kernels' error bits:
 * bit 0 = a bounded wait inside a kernel ran out (that launch's results are
 * invalid).  0 = no error. */
pie_status pie_ctx_check(pie_ctx* ctx, int32_t* flags);
/* Error-path self-test: enqueues one kernel whose mbarrier wait can never
 * complete, bounded at `polls` polls; it records bit 0 in the error word
 * (read it with pie_ctx_check) and ends.  The context stays usable. */
pie_status pie_selftest_wait_timeout(pie_ctx* ctx, int32_t polls);
/* Error-path self-test on the host: the next pie_batch_begin that passes
 * its argument and page-count checks fails with PIE_ERR_CUDA where it would
 * upload its plan -- after reserving its slots, as a real CUDA failure
 * there would -- so that tests can check that the reservation is undone.
 * Also works on plan-only contexts. */
pie_status pie_selftest_fail_next_begin(pie_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* PIE_ATTN_H */
