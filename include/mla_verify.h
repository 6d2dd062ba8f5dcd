/*
 * mla_verify.h -- C ABI of the GB300 (sm_103a) MLA tree-verify attention library.
 *
 * The operation ("verify attention" of tree speculative decoding, page "The
 * Shared Memory Ceiling", sections "The Broader Context" and "Technical Deep
 * Dive"): every draft-tree token of a request, in each of 64 heads, attends
 * to the request's latent KV cache.  A KV row is a 512-dim c_kv latent
 * followed by a 64-dim k_rope; all heads share it; V is the c_kv latent.  A
 * tree token sees the whole prefix and, among the tree's own latents, only
 * its ancestors and itself (given by a parent array).  The softmax is taken
 * online, tile by tile, so no full score row is ever held (same page,
 * "Technical Deep Dive", last paragraph).  Long prefixes with few requests
 * may be split along the KV axis and merged with log-sum-exp weights.
 *
 * Conventions of every call:
 *  - Pointers marked "device" are device memory owned by the caller; the
 *    library never frees, reallocates or retains them past the call.  bf16
 *    tensors are passed as raw 16-bit patterns (const void*).
 *  - Work is enqueued on the caller's stream; no call synchronises the host
 *    except mla_read_status().  mla_verify_attn and mla_split_combine
 *    allocate nothing; they are safe to capture in a CUDA graph once
 *    mla_init() has run on the device.
 *  - Every call returns an mla_status.  Errors detectable from the scalar
 *    arguments are returned before anything is launched.  Errors that depend
 *    on device data (an invalid tree, a block id outside the cache, a
 *    pipeline wait that timed out) are recorded in a status word inside the
 *    workspace; read it with mla_read_status().  Rows of a request with
 *    invalid data are written as out = 0, lse = -inf; no kernel traps.
 *  - Supported shapes: num_heads = 64, d_latent = 512, d_rope = 64,
 *    page_size a positive multiple of 64, 1 <= n_tree[b] <= 64 (or 0 for an
 *    empty request), bf16 inputs, fp32 outputs.  Anything else returns
 *    MLA_ERR_UNSUPPORTED.
 */
#ifndef MLA_VERIFY_H_
#define MLA_VERIFY_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, misaligned pointer  */
    MLA_ERR_UNSUPPORTED = 2,  /* shape outside the supported set above            */
    MLA_ERR_WORKSPACE = 3,    /* workspace null or smaller than required           */
    MLA_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed               */
    MLA_ERR_TIMEOUT = 5,      /* a bounded device-side wait expired (status word)  */
    MLA_ERR_BAD_TREE = 6,     /* parent outside [-1, i), n_tree > seq_len, sums    */
    MLA_ERR_BAD_BLOCK = 7,    /* block-table entry outside [0, num_pages)          */
    MLA_ERR_NOT_INITIALIZED = 8, /* mla_init() has not run on the current device   */
    MLA_ERR_BAD_INDEX = 9     /* sparse variant: a top-k slot outside {-1} u [0, prefix) */
} mla_status;

#define MLA_NUM_HEADS 64
#define MLA_D_LATENT 512
#define MLA_D_ROPE 64
#define MLA_MAX_TREE 64
#define MLA_MAX_SPLITS 64
/* num_splits value that asks for the persistent schedule (see mla_verify_num_splits) */
#define MLA_SPLITS_PERSISTENT (-1)
#define MLA_MAX_TOPK 2048

/* Library version (major * 10000 + minor * 100 + patch). */
int mla_version(void);

/* Human-readable text of a status code (static storage, never NULL). */
const char *mla_error_string(int status);

/*
 * Per-device set-up: checks that `device` is an sm_103 GPU, raises the
 * kernels' dynamic shared-memory limit, checks that the verify kernels were
 * compiled with the registers their warpgroups divide among themselves at run
 * time (MLA_ERR_UNSUPPORTED otherwise: such a build would wait forever) and
 * resolves the driver's tensor-map encoder.  Call once per device, outside
 * stream capture, before the first
 * verify call on that device.  Makes `device` current.  Idempotent.  After
 * cudaDeviceReset the device has a new context: call mla_init again before the
 * next call on it (it sets the kernels up again and forgets cached device
 * addresses of the old context).
 */
int mla_init(int device);

/*
 * Number of KV splits the verify call will use.  `requested` > 0 is honoured
 * (clamped to [1, MLA_MAX_SPLITS]); 0 picks a plan from the shape with a
 * model of the launch: (request, row-tile, split) work units in whole waves
 * over the SMs of the current device, at least 16 KV tiles of 64 keys per
 * split; when every unit fits in one wave three times over, as many splits as
 * still fit in that wave and shorten the chain of dependent tiles (three or
 * more, merged by the combine pass); or the persistent schedule below (0),
 * when every request has max_tree tree tokens and the model puts it ahead.
 * When 0 resolves to one split and a request has at least 12 KV tiles, the
 * verify call may also cut the work items of its last, partial round of CTA
 * pairs in two and merge them in the kernel (decided on the device from the
 * exact item count); an explicit request of 1 never does.
 * `requested` = MLA_SPLITS_PERSISTENT asks for the persistent schedule instead:
 * a fixed grid of 2-CTA clusters (as many as fit on the device at once), each
 * taking an equal, contiguous share of the sequence of all (row tile, KV tile)
 * pairs of the call and walking it with one pipeline across row tiles; a row
 * tile cut between clusters is merged inside the verify kernel by the last of
 * its pieces to finish, in piece order (the result does not depend on timing).
 * The shares are cut on the device from the exact work, so a graph captured
 * for a bucket computes exactly what the eager call computes.
 * Returns the count, 0 for the persistent schedule, or a negative mla_status
 * on invalid arguments.
 */
int mla_verify_num_splits(int batch, int total_q, int max_tree, int max_seq_len,
                          int num_heads, int requested);

/*
 * Bytes of device workspace mla_verify_attn needs for these sizes (with
 * `num_splits` resolved as by mla_verify_num_splits, including room for the
 * cut described there when `num_splits` is 0, and for the pieces' partials
 * when it is MLA_SPLITS_PERSISTENT: 2 x 128 rows x 512 fp32 per cluster).
 * Pass the same `num_splits` to mla_verify_attn.  0 on invalid input.
 */
size_t mla_verify_workspace_size(int batch, int total_q, int max_tree, int max_seq_len,
                                 int num_heads, int num_splits);

/*
 * Tree-verify attention over a paged latent KV cache.
 *
 *  q_lat       device bf16 [total_q, num_heads, 512]   query in the latent space
 *  q_rope      device bf16 [total_q, num_heads, 64]    rotary part of the query
 *  kv_cache    device bf16 [num_pages, page_size, 576] row = c_kv (512) | k_rope (64)
 *  block_table device int32 [batch, max_pages_per_seq]  page of KV position t of
 *              request b is block_table[b][t / page_size], row t % page_size
 *  seq_lens    device int32 [batch]  KV rows of request b = prefix_b + n_tree[b];
 *              the tree tokens' own latents occupy positions prefix_b .. seq_len-1
 *  tree_parent device int32 [total_q] request-local parent of each tree token,
 *              -1 for a root (child of the last prefix token); parent[i] < i
 *  n_tree      device int32 [batch]  tree tokens of each request; requests are
 *              laid out back to back in q_lat / tree_parent / out
 *  scale       softmax scale applied to q . k (latent and rope parts alike);
 *              finite and > 0, else MLA_ERR_INVALID_ARG
 *  out         device fp32 [total_q, num_heads, 512]  softmax-weighted c_kv
 *  lse         device fp32 [total_q, num_heads]  natural-log log-sum-exp of the
 *              scaled scores over the visible keys
 *  stream      stream the work is enqueued on
 *  batch, total_q      sizes of the arrays above (total_q = sum of n_tree)
 *  max_tree, max_seq_len  host-side upper bounds of n_tree[b] and seq_lens[b]
 *  num_heads   must be 64
 *  page_size   rows per page, a multiple of 64
 *  num_pages   pages in kv_cache (block ids must lie in [0, num_pages))
 *  max_pages_per_seq  row stride of block_table
 *  num_splits  KV splits (0 = choose, see mla_verify_num_splits).  With two
 *              splits the verify kernel merges them itself and the first split
 *              takes a shape-dependent share of each request's KV tiles (chosen
 *              so that the work units fill the SMs' rounds evenly); with more,
 *              a log-sum-exp combine pass follows the verify kernel.
 *              MLA_SPLITS_PERSISTENT: the persistent schedule (no combine pass).
 *  workspace   device scratch of at least mla_verify_workspace_size(...) bytes,
 *              256-byte aligned; it holds the status word, the per-call tree
 *              metadata and, when split, the partial outputs.  Its contents
 *              are owned by the library until the stream reaches the end of
 *              the call; do not share one workspace between calls that may run
 *              concurrently.
 *
 * Pointer alignment: bf16/fp32 tensors 16-byte aligned.  The result does not
 * depend on how pages are placed in the pool (only on the logical rows), and
 * repeated calls with the same inputs give bitwise-identical results.
 */
int mla_verify_attn(const void *q_lat, const void *q_rope, const void *kv_cache,
                    const int32_t *block_table, const int32_t *seq_lens,
                    const int32_t *tree_parent, const int32_t *n_tree, float scale,
                    float *out, float *lse, cudaStream_t stream,
                    int batch, int total_q, int max_tree, int max_seq_len, int num_heads,
                    int page_size, int num_pages, int max_pages_per_seq, int num_splits,
                    void *workspace, size_t workspace_bytes);

/*
 * Log-sum-exp merge of split-KV partials (flash-decoding combine).  A long
 * prefix with few requests is divided along the KV axis into splits, each
 * attended separately (the decode kernel of page "The SMEM Ceiling", section
 * "The Problem Space", is such a split kernel); their results are merged by
 * the rescale-and-add step of the online softmax (page "The Shared Memory
 * Ceiling", section "Technical Deep Dive": the softmax of the whole set is
 * reached incrementally, earlier partial sums rescaled by the change of the
 * running maximum), applied once per split with each split's log-sum-exp in
 * place of its running maximum and normaliser.
 *
 *  part_out  device fp32 [num_splits, rows, 512]  each split's normalised output
 *  part_lse  device fp32 [num_splits, rows]       each split's natural-log LSE;
 *            -inf marks a split that saw no key (weight 0)
 *  out       device fp32 [rows, 512]:  sum_s exp(lse_s - lse) * part_out[s]
 *  lse       device fp32 [rows]:       max_s lse_s + ln sum_s exp(lse_s - max_s lse_s)
 * A row whose partials are all -inf gets out = 0, lse = -inf.
 * 1 <= num_splits <= MLA_MAX_SPLITS; pointers 16-byte aligned.
 */
int mla_split_combine(const float *part_out, const float *part_lse, int num_splits, int rows,
                      float *out, float *lse, cudaStream_t stream);

/*
 * Splits split_begin .. split_begin + split_count - 1 of num_splits of every
 * request's KV, each one's normalised partial and log-sum-exp written to
 * part_out (device fp32 [split_count, total_q * 64, 512]) and part_lse (device
 * fp32 [split_count, total_q * 64]); nothing else is written.  Split s covers
 * KV tiles (64 keys) [n*s/S, n*(s+1)/S) of a request of n tiles (integer
 * division), so the tree's own keys fall in the last split.  For sharding one
 * long request's prefix across GPUs (the pages' serving setup runs on eight
 * cards: page "The 99KB Barrier", sections "Message Snapshot" and "The
 * Investigation Leading Up to This Message"): GPU r holds the KV pages
 * of its splits only -- the block table must still name a valid page for
 * every position, but pages outside the computed splits are never read --
 * computes its splits, the GPUs exchange the partials once (all-gather), and
 * mla_split_combine merges them.  Other arguments as for mla_verify_attn; the
 * workspace is sized by mla_verify_workspace_size(..., num_splits = 1).  No
 * sparse form.  Returns MLA_ERR_INVALID_ARG for an empty or out-of-range split
 * range.
 */
int mla_verify_attn_split_range(const void *q_lat, const void *q_rope, const void *kv_cache,
                                const int32_t *block_table, const int32_t *seq_lens,
                                const int32_t *tree_parent, const int32_t *n_tree, float scale,
                                float *part_out, float *part_lse, cudaStream_t stream,
                                int batch, int total_q, int max_tree, int max_seq_len, int num_heads,
                                int page_size, int num_pages, int max_pages_per_seq, int num_splits,
                                int split_begin, int split_count, void *workspace,
                                size_t workspace_bytes);

/*
 * Sparse (top-k) tree verification ("The SMEM Ceiling", section "The Problem
 * Space": during decode each token attends to a sparse set of previous tokens
 * chosen by a top-k index selection).  Arguments as for mla_verify_attn, plus
 *  topk_idx  device int32 [total_q, topk]: for each tree token, the prefix
 *            positions (0 <= t < seq_len - n_tree of its request) it attends
 *            to, in any order; -1 marks an unused slot.  Each listed slot is
 *            one key (a position listed twice counts twice).
 *  topk      1 <= topk <= MLA_MAX_TOPK (the pages' kernel uses 512).
 * Token i of request b then sees its listed prefix positions and its
 * ancestor-or-self tree tokens, in all heads: out / lse as for
 * mla_verify_attn over that key set.  A slot outside {-1} u [0, prefix) sets
 * status bit 1 << MLA_ERR_BAD_INDEX and the request's rows are written as
 * out = 0, lse = -inf.  The two tree tokens of a 128-row tile share one key
 * stream (their slot lists one after the other), so the tensor work per tile
 * is twice the visible work.
 * mla_verify_sparse_num_splits / mla_verify_sparse_workspace_size: as the
 * dense ones, for `topk` instead of max_seq_len.
 */
int mla_verify_sparse_num_splits(int batch, int total_q, int max_tree, int topk, int num_heads,
                                 int requested);
size_t mla_verify_sparse_workspace_size(int batch, int total_q, int max_tree, int topk,
                                        int num_heads, int num_splits);
int mla_verify_sparse_attn(const void *q_lat, const void *q_rope, const void *kv_cache,
                           const int32_t *block_table, const int32_t *seq_lens,
                           const int32_t *tree_parent, const int32_t *n_tree,
                           const int32_t *topk_idx, int topk, float scale, float *out, float *lse,
                           cudaStream_t stream, int batch, int total_q, int max_tree, int max_seq_len,
                           int num_heads, int page_size, int num_pages, int max_pages_per_seq,
                           int num_splits, void *workspace, size_t workspace_bytes);

/*
 * mla_verify_attn for callers that cannot allocate device memory: the page
 * text has no counterpart to this entry point.  Some callers cannot provide a
 * workspace -- e.g. a plugin inside a serving engine that owns all device
 * memory through its own pool and exposes no workspace hook, or a
 * latency-critical loop where cudaMalloc (which may synchronise the device)
 * is not acceptable.  This variant keeps the per-call scratch (status word,
 * query offsets, ancestor bit sets, work list) in a 1 MiB static device array
 * that every GPU loading the library holds until the process exits, and runs
 * with a single KV split.  The caller still passes inputs and outputs; the
 * arguments mean what they mean for mla_verify_attn.  It allocates nothing.
 *  - Sizes whose scratch would exceed 1 MiB (roughly 12 B per tree token plus
 *    20 B per request) return MLA_ERR_WORKSPACE before anything is launched.
 *  - The first call on a device looks up the array's device address; make that
 *    first call before any stream capture on that device.
 *  - All calls share the array.  The kernels clear what must start at zero and
 *    overwrite the rest before reading it, so a call never sees an earlier
 *    call's data, but calls whose work overlaps on the GPU (other streams,
 *    other host threads) race on it and must be serialised by the caller.
 *  - The device status word (as for mla_verify_attn) lives in the array; read
 *    it with mla_verify_noalloc_read_status once the call's stream has been
 *    synchronised and before the next call on the device.
 */
int mla_verify_attn_noalloc(const void *q_lat, const void *q_rope, const void *kv_cache,
                            const int32_t *block_table, const int32_t *seq_lens,
                            const int32_t *tree_parent, const int32_t *n_tree, float scale,
                            float *out, float *lse, cudaStream_t stream,
                            int batch, int total_q, int max_tree, int max_seq_len, int num_heads,
                            int page_size, int num_pages, int max_pages_per_seq);

/*
 * Copies the device status word of the last mla_verify_attn_noalloc call on the
 * current device (the bits of mla_read_status) to *device_status.  Synchronous
 * (a device-to-host copy); call it after synchronising the verify call's
 * stream.  No counterpart in the page text either.  MLA_ERR_INVALID_ARG for a
 * NULL pointer, MLA_ERR_CUDA if the copy fails.
 */
int mla_verify_noalloc_read_status(int *device_status);

/*
 * Paged-cache steps around verification ("The Shared Memory Ceiling", section
 * "The Broader Context": the draft tree's latents live in the same paged KV
 * cache that verification reads, and the step after it is a KV-cache defrag).
 * Rows are 576 bf16 values (c_kv then k_rope) moved as raw bits: exact.
 * Request b's tree region is KV positions P_b .. P_b + n_tree[b] - 1 with
 * P_b = seq_lens[b] - n_tree[b], mapped through block_table as for
 * mla_verify_attn; it must lie in pages no other request writes.
 *
 * mla_tree_kv_workspace_size: bytes of workspace both steps need (the device
 * status word, readable with mla_read_status).
 *
 * mla_tree_kv_append: writes tree_kv (device bf16 [total_q, 576], tokens back
 * to back in request order, as in q_lat) into each request's tree region of
 * kv_cache ([num_pages, page_size, 576], 16-byte aligned).  Request b's rows
 * start at the sum of n_tree[0..b), a negative count taken as 0.  A request
 * whose n_tree is outside [0, 64] or above its seq_len, or whose rows would
 * reach past total_q, sets status bit 1 << MLA_ERR_BAD_TREE; one whose tree
 * region maps to a block id outside [0, num_pages) sets 1 << MLA_ERR_BAD_BLOCK;
 * either request is left untouched (no row outside [0, total_q) is read).
 *
 * mla_tree_kv_accept: after verification, accept_len[b] (device int32 [batch])
 * tokens of request b are accepted; accept_idx (device int32 [total_q], same
 * layout as tree_parent) holds, at the start of each request's segment, their
 * node indices along a path from a root (the first one's parent is -1, each
 * next one is a child of the one before).  Accepted node k's row moves to
 * position P_b + k; rows after P_b + accept_len[b] keep their old contents,
 * and new_seq_lens[b] (device int32 [batch]) = P_b + accept_len[b].  All of a
 * request's accepted rows are read before any is written.  A malformed tree or
 * path, or accept_len outside [0, n_tree[b]], sets 1 << MLA_ERR_BAD_TREE; a bad
 * block id sets 1 << MLA_ERR_BAD_BLOCK; such a request is left untouched and
 * new_seq_lens[b] = seq_lens[b].
 *
 * Both: one thread block per request on `stream`; mla_init must have run on
 * the device; host-checkable errors return before any launch; the workspace
 * (caller-owned, >= mla_tree_kv_workspace_size() bytes) is cleared on the
 * stream first.  They allocate nothing and never synchronise.
 */
size_t mla_tree_kv_workspace_size(void);
int mla_tree_kv_append(const void *tree_kv, void *kv_cache, const int32_t *block_table,
                       const int32_t *seq_lens, const int32_t *n_tree, cudaStream_t stream,
                       int batch, int total_q, int page_size, int num_pages, int max_pages_per_seq,
                       void *workspace, size_t workspace_bytes);
int mla_tree_kv_accept(void *kv_cache, const int32_t *block_table, const int32_t *seq_lens,
                       const int32_t *n_tree, const int32_t *tree_parent, const int32_t *accept_len,
                       const int32_t *accept_idx, int32_t *new_seq_lens, cudaStream_t stream,
                       int batch, int total_q, int page_size, int num_pages, int max_pages_per_seq,
                       void *workspace, size_t workspace_bytes);

/*
 * Replayable verify step for a batch bucket (a CUDA graph of prep, slot check,
 * verify and combine, captured once).  Serving loops run the same step shape
 * every iteration at small batch, where launch overhead dominates.  A graph
 * replays its GPU work with no host involvement, so everything that
 * synchronises or chooses a configuration happens before the capture and the
 * captured shape is a batch bucket that smaller batches pad up to (page "SMEM
 * Ceiling", section "CUDA Graph Capture Safety: A Nuanced Understanding").
 *
 * mla_verify_graph_create: captures the step on `stream` (a private stream if
 * it is a default stream) for the bucket max_batch requests, max_total_q tree
 * tokens, with the arguments of mla_verify_attn (topk == 0) or
 * mla_verify_sparse_attn (topk > 0).  The buffers passed here are the ones
 * every replay reads and writes: the caller owns them, keeps them alive until
 * mla_verify_graph_destroy, and writes each step's inputs into them before a
 * launch.  Requires mla_init on the current device.  On success *graph holds
 * a host object; on error *graph is NULL and nothing was launched.
 *
 * mla_verify_graph_launch: replays the step for the first `batch` requests
 * (0 <= batch <= max_batch) on `stream`.  Requests batch .. max_batch - 1 are
 * padded: their n_tree and seq_lens entries are set to 0 on the stream
 * before the replay (so those entries of the caller's buffers are written).
 * The tree tokens of the real requests must number at most max_total_q; out
 * and lse rows past their total are not defined.  Errors are reported in the
 * workspace's status word as for mla_verify_attn.  Call it from the device the
 * graph was created on; it never synchronises.
 *
 * mla_verify_graph_destroy: releases the graph (NULL is accepted).
 */
typedef struct mla_verify_graph mla_verify_graph;
int mla_verify_graph_create(const void *q_lat, const void *q_rope, const void *kv_cache,
                            const int32_t *block_table, int32_t *seq_lens, const int32_t *tree_parent,
                            int32_t *n_tree, const int32_t *topk_idx, int topk, float scale, float *out,
                            float *lse, int max_batch, int max_total_q, int max_tree, int max_seq_len,
                            int num_heads, int page_size, int num_pages, int max_pages_per_seq,
                            int num_splits, void *workspace, size_t workspace_bytes, cudaStream_t stream,
                            mla_verify_graph **graph);
int mla_verify_graph_launch(mla_verify_graph *graph, int batch, cudaStream_t stream);
int mla_verify_graph_destroy(mla_verify_graph *graph);

/*
 * Measurement hook: while set, every mla_verify_attn call records `begin`
 * immediately before and `end` immediately after the launch of its fused
 * verify kernel, on the call's stream, so the kernel can be timed alone.
 * Pass NULL, NULL to stop.  Process-wide setting; not thread-safe.
 */
int mla_set_profile_events(cudaEvent_t begin, cudaEvent_t end);

/*
 * Synchronously read the device status word of the last call that used
 * `workspace` (waits for the device).  *device_status receives a bit mask:
 * bit k set means status code k was raised (e.g. 1 << MLA_ERR_BAD_TREE).
 * Returns MLA_OK if the word was read, MLA_ERR_CUDA otherwise.
 */
int mla_read_status(const void *workspace, int *device_status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_VERIFY_H_ */
