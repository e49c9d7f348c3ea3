/*
 * dhs.h -- C ABI of libdhs: speculative-verification sparse attention over a
 * two-tier KV cache, for one GB300 GPU (sm_103a).
 *
 * Source of every operation: "Adaptive DHiSparse: Speculative Decoding over a
 * Load-Adaptive KV Hierarchy" (arXiv 2610.13708), cited as [ADHS] with the
 * section, equation or figure that defines it.
 *
 * One dhs_ctx is one KV source (one payload layer, [ADHS] 2.2 "physical-source
 * sharing") serving n_slots request slots.  A verification round of request r
 * runs, all on one caller stream:
 *
 *   dhs_select   indexer scores + per-query top-k over the causal history
 *   dhs_resolve  union of the K_r selections, probe ring / optional map / hot
 *                cache, compact the misses, fetch each missing row once from
 *                pinned host memory into staging (a promoted row also into
 *                its hot-cache slot), emit one location per selected entry
 *   dhs_attend   write the block rows into the draft ring, attend every query
 *                over its own selection plus the block rows up to itself
 *   dhs_commit   keep the accepted prefix of the block, roll back the rest
 *
 * Conventions
 *   - Pointers marked "device" are CUDA device pointers; "host" pointers are
 *     read by the calling thread before the function returns; "pinned" host
 *     memory must stay allocated and page-locked (cudaHostAlloc or
 *     cudaHostRegister) while bound.
 *   - All calls that take a stream only enqueue work on it and return; argument
 *     errors are detected on the host before anything is launched.
 *   - The round's kernels are launched with programmatic stream serialization
 *     (each may be placed while the previous launch on the stream drains, and
 *     waits for it before touching its results).  Stream order is kept for
 *     ordinary caller work in between; a caller kernel placed between two
 *     calls that itself uses programmatic dependent launch must wait on its
 *     own grid dependency before it exits.
 *   - Kernels check the indices they read (selected rows, locations) and, on
 *     a bad one, skip the access and record DHS_ERR_DEVICE_CHECK in a device
 *     error word, which dhs_get_stats reports after synchronising the stream.
 *     No kernel ever traps or waits on a flag set by another launch; the one
 *     wait inside a kernel (on its own copies in flight) is bounded, and if
 *     it runs out the same error word is set and the kernel carries on.
 *   - Buffers passed by the caller stay owned by the caller.  Everything the
 *     context allocates (hot cache, staging, ring, optional pool, maps,
 *     scratch) is owned by it and freed by dhs_destroy.
 *   - bf16 values are passed as raw 16-bit storage (uint16_t).
 */
#ifndef DHS_H_
#define DHS_H_

#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dhs_ctx dhs_ctx;
typedef struct CUstream_st *dhs_stream; /* a cudaStream_t; NULL = legacy default stream */

/* Error codes. */
enum {
  DHS_OK = 0,
  DHS_ERR_INVALID = 1,      /* bad argument, shape or call order             */
  DHS_ERR_OOM = 2,          /* device or pinned allocation failed            */
  DHS_ERR_CAPACITY = 3,     /* request exceeds a configured capacity         */
  DHS_ERR_CUDA = 4,         /* a CUDA runtime call failed                    */
  DHS_ERR_DEVICE_CHECK = 5, /* a kernel found an out-of-range index          */
  DHS_ERR_TIMEOUT = 6       /* reserved: a bounded host wait ran out         */
};

/* Location tags, [ADHS] 3.5 eq. (12): each selected entry l_{r,j,i} names the
 * GPU tier that holds row s_{r,j,i} and its index within request r's part of
 * that tier: loc = (tier << 28) | index, or -1 for an empty entry.
 *   RING : draft-ring row (t mod R_d) of committed position t, eq. (10)
 *   OPT  : slot of the optional-history pool, [ADHS] 3.1
 *   HOT  : slot of the B-row hot cache, [ADHS] 2.2 / 3.2
 *   STAGE: row of the verification staging arena, [ADHS] 3.3-3.4 */
enum { DHS_LOC_RING = 0, DHS_LOC_OPT = 1, DHS_LOC_HOT = 2, DHS_LOC_STAGE = 3 };
#define DHS_LOC_TIER_SHIFT 28
#define DHS_LOC_INDEX_MASK ((1 << DHS_LOC_TIER_SHIFT) - 1)

/* Row layouts of the stored KV payload. */
enum {
  DHS_KV_SPLIT = 0, /* GQA: row = K of kv heads 0..Hkv-1 (qk_dim each), then V heads (v_dim each) */
  DHS_KV_LATENT = 1 /* MLA-like shared latent: row = qk_dim elements; K = row, V = row[0:v_dim]     */
};

/* Fixed at dhs_create.  Limits: n_slots <= 256, k_max <= 8, topk <= 2048 (a
 * multiple of 32), q_heads / kv_heads <= 16, qk_dim and v_dim multiples of 16,
 * idx_heads * idx_dim a multiple of 16 and <= 1024, budget <= 65535. */
typedef struct {
  int32_t n_slots;      /* N request slots                                      */
  int32_t k_max;        /* K_max: widest verification block, [ADHS] 3.3         */
  int32_t topk;         /* k: rows selected per query, [ADHS] eq. (1)           */
  int64_t s_max;        /* rows of history (plus room for commits) per request  */
  int32_t idx_heads;    /* H_idx: indexer heads, summed                         */
  int32_t idx_dim;      /* d_idx: int8 elements per indexer head                */
  int32_t q_heads;      /* Hq attention query heads                             */
  int32_t kv_heads;     /* Hkv kv heads (1 for DHS_KV_LATENT)                   */
  int32_t qk_dim;       /* key/query head dim (latent width for DHS_KV_LATENT)  */
  int32_t v_dim;        /* value head dim                                       */
  int32_t kv_layout;    /* DHS_KV_SPLIT or DHS_KV_LATENT                        */
  int32_t budget;       /* B: hot-cache rows per request, [ADHS] 2.2            */
  int32_t ring_window;  /* W: drafter window, [ADHS] eq. (9)                    */
  int32_t page_rows;    /* p: rows per page, [ADHS] eq. (9)                     */
  int64_t opt_rows_max; /* optional-pool rows per request (0 = no optional map) */
  float softmax_scale;  /* 0 = 1/sqrt(qk_dim)                                   */
  int32_t attn_pass;    /* attention kernel for shared retrieval, DHS_ATTN_*    */
  int32_t topk_pass;    /* top-k kernel of dhs_select, DHS_TOPK_*               */
  int32_t round_groups; /* dhs_round: request groups on internal streams (0/1 = one) */
  int32_t tokens_per_row; /* m of [ADHS] eq. (8): token positions packed into one
                             stored row of this source (0 or 1: uncompressed;
                             at most 64).  With m > 1 the history, the caches,
                             s_max and every selected index count stored rows,
                             n_committed and positions count tokens, and the
                             rows a round completes are committed with
                             dhs_commit_compressed. */
} dhs_config;

/* Top-k kernel of dhs_select.  Both return the same ordered lists:
 *   CLUSTER: a cluster of four CTAs per query, the query's scores staged in
 *            their shared memory; spreads few queries over many SMs.
 *   ROW    : one CTA per query with a small footprint, several per SM, the
 *            scores read from global memory; for rounds with many queries.
 *   AUTO   : ROW when the round's active queries (sum of K_r) are at least
 *            the device's SM count, else CLUSTER. */
enum { DHS_TOPK_AUTO = 0, DHS_TOPK_CLUSTER = 1, DHS_TOPK_ROW = 2 };

/* Attention kernel used after a shared dhs_resolve (per-query resolution
 * always uses the per-query pass).  Both compute eq. (5) for every query; they
 * differ in how rows reach the SMs:
 *   PER_QUERY: each (request, query) streams its own k + j + 1 rows; few
 *              dependent steps, best when the round is latency-bound.
 *   UNION    : each (request, kv head) streams the union U_r once and masks
 *              every score by the queries that selected the row; up to K_r
 *              times fewer row reads, best when the round is bound by HBM.
 *              For 128-dim heads with at most 128 (query, head) pairs per kv
 *              head it runs on the fifth-generation tensor cores (tcgen05
 *              MMAs with the scores and the output accumulated in tensor
 *              memory, one CTA per (request, kv head)); otherwise on mma.sync
 *              tiles.
 *   UNION_MMA: the union pass on mma.sync tiles whatever the shape (for
 *              comparison).
 *   AUTO     : UNION for 128-dim heads when the per-query pass would stream
 *              more than 128 MiB of rows per round (n_slots * k_max *
 *              (topk + k_max) rows), else PER_QUERY (always for latent rows). */
enum { DHS_ATTN_AUTO = 0, DHS_ATTN_PER_QUERY = 1, DHS_ATTN_UNION = 2, DHS_ATTN_UNION_MMA = 3 };

/* Cumulative counters since dhs_create (or dhs_reset_stats). */
typedef struct {
  int64_t resolve_calls;
  int64_t selections;        /* valid selected entries resolved               */
  int64_t union_rows;        /* sum over requests of |U_r|, eq. (6)           */
  int64_t ring_hits;         /* union rows served by the draft ring (tail)    */
  int64_t opt_hits;          /* union rows served by the optional map         */
  int64_t hot_hits;          /* union rows served by the hot cache            */
  int64_t misses;            /* distinct missing rows |D_r|, eq. (6)          */
  int64_t miss_selections;   /* selected entries whose row was missing        */
  int64_t host_rows_fetched; /* rows copied from host (shared: |D_r|)         */
  int64_t host_bytes;        /* bytes copied from host                        */
  int64_t installs;          /* rows promoted into the hot cache              */
  int64_t evictions;         /* promotions that replaced a cached row         */
  int64_t direct_only;       /* requests whose union resolved in step 1 only  */
  int32_t device_error;      /* first device check code (0 = none)           */
  int32_t device_error_site; /* kernel id that recorded it                    */
  int64_t topk_rescans;      /* long-domain queries whose sampled threshold
                                estimate missed, so top-k read the scores
                                again (an implementation counter; the result
                                is the same either way)                       */
} dhs_stats;

/* Create a context.  Allocates (cudaMalloc, on the current device) the hot
 * cache, staging arena (k_max * topk rows per slot, [ADHS] 3.4 with chi = 1),
 * draft ring (R_d = p * ceil((W + p - 1 + k_max) / p) rows per slot, [ADHS]
 * eq. (9)), optional pool, the row->slot maps and all scratch.  All slots start
 * unbound.  Returns DHS_ERR_INVALID on a bad config, DHS_ERR_OOM if an
 * allocation fails (nothing is leaked). */
int dhs_create(const dhs_config *cfg, dhs_ctx **out);

/* Free everything the context owns.  Synchronises the device first.  NULL is a no-op. */
void dhs_destroy(dhs_ctx *ctx);

/* Ring rows per slot, eq. (9), and staging bytes, M_stage of [ADHS] 3.4 with chi = 1. */
int64_t dhs_ring_rows(const dhs_ctx *ctx);
int64_t dhs_device_bytes(const dhs_ctx *ctx); /* total device memory the context holds */

/* Bind request slot `slot` to its history.
 *   host_kv  pinned host, bf16 [s_max][row_elems]: the full host backing H_r
 *            ([ADHS] 2.2 fixed-cache offloading).  Read by dhs_resolve and
 *            dhs_set_residency, written by dhs_commit.
 *   idx_keys device, int8 [s_max][idx_heads * idx_dim]: GPU index state
 *            ([ADHS] 2.2 "compact indexer state remains on the GPU").  Rows at
 *            or beyond n_committed may be filled later by the caller.
 *   n_committed  n_r, committed history rows (0 <= n_committed <= s_max).
 * Resets the slot's hot cache (empty), optional set (empty) and ring (no live
 * rows: positions before n_committed are served by the hierarchy). */
int dhs_bind_request(dhs_ctx *ctx, int32_t slot, const void *host_kv, const int8_t *idx_keys,
                     int64_t n_committed, dhs_stream stream);

/* Step 1, [ADHS] 2.1 eq. (1) with the causal domain of eq. (5).
 *   q_idx      device int8 [n_slots][k_max][idx_heads][idx_dim]
 *   k_per_req  host int32 [n_slots]: K_r queries of request r this round
 *              (0 = slot idle this round; bound slots only; <= k_max)
 *   pos        host int64 [n_slots][k_max] or NULL: position of query j; NULL
 *              means n_r + j.  Query j selects among rows [0, min(n_r, pos+1)).
 *   topk_out   device int32 [n_slots][k_max][topk]: rows ordered by score
 *              descending, ties to the lower row, padded with -1.  Entries of
 *              idle queries are left untouched.
 * Score I[s] = sum_h sum_d q[h][d] * K[s][h][d] in exact int32 arithmetic.
 * Called on an idle context (a new round), or after the round's dhs_attend
 * by a Reindex layer of the same source (see "Physical-source sharing"). */
int dhs_select(dhs_ctx *ctx, const int8_t *q_idx, const int32_t *k_per_req,
               const int64_t *pos, int32_t *topk_out, dhs_stream stream);

/* Steps 2-4, [ADHS] 3.2-3.3, eq. (6), Fig. 2, Fig. 3 callouts 2-3.
 *   topk     device int32 [n_slots][k_max][topk] (from dhs_select or the caller;
 *            entries must be -1 or rows < n_r, no row twice in one query's
 *            list -- a selection is a set; a repeat is reported as
 *            DHS_ERR_DEVICE_CHECK)
 *   loc_out  device int32 [n_slots][k_max][topk]: one location per entry
 *   shared   1: each distinct missing row of a request is fetched once and its
 *            staging location returned to every query that selected it;
 *            0: per-query baseline, every missing selection fetched on its own
 *            into staging row j*topk+i.  The cache state is the same in both.
 * Probe order per union row (ascending): live draft-ring rows
 * [max(first, n_r - W), n_r), then the ready optional map, then the hot cache
 * (a hit refreshes the slot's stamp to this call's tick).  Hot rows of the
 * union are protected; victims are the other slots ordered by (stamp, slot),
 * empty first; the first min(|D_r|, #victims) missing rows, ascending, take
 * them.  Their bytes are written to the slot as they arrive from host; no
 * location of this round names a victim slot, so attention is unaffected.
 * One tick of the LRU clock per call.  Must be followed by dhs_attend before
 * the next dhs_resolve or dhs_set_residency on this context. */
int dhs_resolve(dhs_ctx *ctx, const int32_t *topk, int32_t *loc_out, int32_t shared,
                dhs_stream stream);

/* Step 5, [ADHS] eq. (1), (5), (11): for every active (r, j < K_r) and query
 * head h (kv head h / (q_heads / kv_heads)):
 *   out = softmax(scale * K q) V over the rows at loc[r][j][*] (entries -1
 *   skipped) followed by block rows 0..j.
 *   q         device bf16 [n_slots][k_max][q_heads][qk_dim]
 *   block_kv  device bf16 [n_slots][k_max][row_elems]: rows the target computed
 *             for positions n_r .. n_r + K_r - 1; written to the draft ring
 *             at phi(r, n_r + u), eq. (10)
 *   loc       device int32 [n_slots][k_max][topk] from dhs_resolve
 *   out       device bf16 [n_slots][k_max][q_heads][v_dim]
 *   lse       device fp32 [n_slots][k_max][q_heads] natural-log sum-exp, or NULL
 * Follows the dhs_resolve of the same round on the stream.  The per-query
 * pass attends the rows held on the GPU (hot cache, optional pool, draft
 * ring) and the block rows while the resolve's host gather is still running,
 * and the staging rows after it; the union passes start once the gather has
 * finished.  q, block_kv and loc must therefore be complete when the call's
 * first kernel starts (in stream order, with no caller kernel in between that
 * releases its dependents before writing them). */
int dhs_attend(dhs_ctx *ctx, const void *q, const void *block_kv, const int32_t *loc,
               void *out, float *lse, dhs_stream stream);

/* Commit / rollback, [ADHS] eq. (7).
 *   accepted_len  host int32 [n_slots]: a_r rows kept, 0 <= a_r <= K_r (the
 *                 anchor plus accepted drafts, 1 + A_r; 0 rolls back all).
 * Kept rows become history: n_r += a_r, and the rows are written back to the
 * host backing (so every row not ready on the GPU has a host copy, eq. (6)).
 * Rejected rows are never published.  DHS_ERR_INVALID if a_r is out of range,
 * DHS_ERR_CAPACITY if n_r + a_r > s_max; nothing changes on error. */
int dhs_commit(dhs_ctx *ctx, const int32_t *accepted_len, dhs_stream stream);

/* Index keys of committed rows, [ADHS] 3.3 (kept rows join the immutable
 * history) with 2.2 (the compact indexer state of the history stays on the
 * GPU): the rows a commit keeps take their index keys with them.
 *   accepted_len    host int32 [n_slots]: a_r, the rows this round's commit
 *                   keeps (0 for idle or unbound slots)
 *   block_idx_keys  device int8 [n_slots][k_max][idx_heads * idx_dim], 16-byte
 *                   aligned: the index keys the target computed for positions
 *                   n_r .. n_r + K_r - 1
 * Copies block_idx_keys[r][u] to row n_r + u of the index-key buffer bound to
 * slot r (dhs_bind_request; it must be writable device memory), u < a_r, with
 * n_r the slot's committed history when the call is issued: issue it before
 * the round's dhs_commit, or before dhs_round.  The indexer reads rows below
 * n_r only, so later rounds see the keys and this round is unaffected.
 * DHS_ERR_INVALID if a_r < 0 or a_r > k_max, a_r > 0 on an unbound slot, or
 * the context is a follower (it holds no keys); DHS_ERR_CAPACITY if
 * n_r + a_r > s_max; nothing is copied on error. */
int dhs_append_keys(dhs_ctx *ctx, const int32_t *accepted_len, const int8_t *block_idx_keys,
                    dhs_stream stream);

/* Commit for a source that packs m = cfg.tokens_per_row token positions into
 * each stored row, [ADHS] eq. (8) and 3.3.  Keeping a_r of the block's
 * positions (0 <= a_r <= K_r, as dhs_commit) moves the slot's token count
 * from n_r to n_r + a_r, and the stored rows
 *     floor(n_r / m) <= s < floor((n_r + a_r) / m)
 * become complete (the page garbles the upper bound's bracket; the floor
 * keeps a partial group in the tail).  Their payload and index keys come
 * from the model's compressor:
 *   rows_kv        device bf16 [n_slots][ceil(k_max / m)][row_elems], 16-byte
 *                  aligned: row i of slot r is stored row floor(n_r / m) + i
 *   rows_idx_keys  device int8 [n_slots][ceil(k_max / m)][idx_heads*idx_dim],
 *                  16-byte aligned, or NULL when the caller writes the keys
 * They join the history: written to the host backing (its backup) and the
 * bound key buffer, and the history grows to floor((n_r + a_r) / m) rows.
 * The positions of a partial group stay counted in n_r with no row
 * published; the draft ring (the block's token rows) serves no history row
 * of such a source.  Follows dhs_attend like dhs_commit, which (with
 * dhs_append_keys and dhs_round) refuses contexts with m > 1; with m = 1 this
 * call commits the caller's rows in place of the ring's.  DHS_ERR_INVALID
 * as dhs_commit, DHS_ERR_CAPACITY if a history would pass s_max rows;
 * nothing changes on error. */
int dhs_commit_compressed(dhs_ctx *ctx, const int32_t *accepted_len, const void *rows_kv,
                          const int8_t *rows_idx_keys, dhs_stream stream);

/* Optional residency, [ADHS] 3.1: make `rows` (host int32 [n_rows], distinct,
 * each < n_r) the ready optional history of `slot`; rows[i] occupies pool slot
 * i.  Bytes are copied from the host backing first and the map entries
 * published after the copy, in stream order.  The previous optional set of the
 * slot stops being ready.  n_rows = 0 clears it.  DHS_ERR_CAPACITY if n_rows >
 * opt_rows_max.  `rows` is uploaded with an asynchronous copy on `stream`: a
 * pageable array is staged before the call returns and may be reused at once,
 * but a page-locked one (cudaHostAlloc / cudaHostRegister) is read when the
 * stream reaches the copy, so it must stay unchanged until then (for example
 * until an event recorded after this call has completed). */
int dhs_set_residency(dhs_ctx *ctx, int32_t slot, const int32_t *rows, int64_t n_rows,
                      dhs_stream stream);

/* Synchronise `stream` and copy out the counters; returns DHS_ERR_DEVICE_CHECK
 * if a kernel recorded a bad index (the counters are still filled). */
int dhs_get_stats(dhs_ctx *ctx, dhs_stats *out, dhs_stream stream);
int dhs_reset_stats(dhs_ctx *ctx, dhs_stream stream);

/* Internal buffers, readable for tests and tools (dhs_export copies `bytes`
 * bytes of buffer `which` into the caller's device buffer `dst`). */
enum {
  DHS_BUF_HOT_ROW = 0,   /* int32 [n_slots][budget], -1 = empty                */
  DHS_BUF_HOT_STAMP = 1, /* int32 [n_slots][budget], -1 = never used           */
  DHS_BUF_HOT_DATA = 2,  /* bf16 [n_slots][budget][row_elems]                  */
  DHS_BUF_RING = 3,      /* bf16 [n_slots][R_d][row_elems]                     */
  DHS_BUF_STAGE = 4,     /* bf16 [n_slots][k_max*topk][row_elems]              */
  DHS_BUF_OPT = 5,       /* bf16 [n_slots][opt_rows_max][row_elems]            */
  DHS_BUF_UNION = 6,     /* int32 [n_slots][k_max*topk], ascending             */
  DHS_BUF_MISS = 7,      /* int32 [n_slots][k_max*topk], ascending             */
  DHS_BUF_COUNTS = 8,    /* int32 [n_slots][4]: |U_r|, |D_r|, promoted, hits   */
  DHS_BUF_LRU = 9,       /* int32 [n_slots][budget]: slots by (stamp, slot)    */
  DHS_BUF_FRONTIER = 10, /* int64 [n_slots]: n_r                               */
  DHS_BUF_HOT_MAP = 11,  /* int32 [n_slots][s_max]: row -> hot slot or -1      */
  DHS_BUF_OPT_MAP = 12,  /* int32 [n_slots][s_max]: row -> pool slot or -1     */
  DHS_BUF_SCORES = 13,   /* int32 [n_slots][k_max][S]: indexer scores of the
                            last dhs_select, S = s_max rounded up to a
                            multiple of 32; valid for the rows below the
                            request's widest query domain                     */
  DHS_BUF_COUNT_ = 14
};
int64_t dhs_buffer_bytes(const dhs_ctx *ctx, int32_t which);
int dhs_export(dhs_ctx *ctx, int32_t which, void *dst, int64_t bytes, dhs_stream stream);

/* Per-kernel timing: when enabled, every kernel launch of the context is
 * bracketed by CUDA events on its stream; dhs_kernel_times synchronises and
 * returns, per kernel id, the number of launches and total milliseconds since
 * the last reset.  While it is enabled, dhs_round issues the round as one
 * request group on the caller's stream (no overlapping launches), so each
 * duration is that kernel's alone over the whole batch.  Kernel ids and
 * names: dhs_kernel_name(id). */
int dhs_set_timing(dhs_ctx *ctx, int32_t enable);
int dhs_kernel_times(dhs_ctx *ctx, int32_t max_ids, int64_t *launches, double *total_ms);

/* Calls made while `stream` is being captured into a CUDA graph (with timing
 * enabled) record their kernel events as event-record nodes of the graph.
 * After each launch of such a graph, this call waits for those events and
 * adds the kernel durations to the totals dhs_kernel_times reports. */
int dhs_timing_accumulate_graph(dhs_ctx *ctx);
const char *dhs_kernel_name(int32_t id);
int32_t dhs_kernel_count(void);

/* Snapshot of all mutable state (device buffers and host-side frontiers), for
 * benchmarks that repeat one round from the same state.  dhs_restore enqueues
 * device copies on `stream`. */
int dhs_snapshot(dhs_ctx *ctx, int32_t *snapshot_id, dhs_stream stream);
int dhs_restore(dhs_ctx *ctx, int32_t snapshot_id, dhs_stream stream);
/* Free a snapshot's device copies (synchronises the device first); its id is
 * not reused and restoring it afterwards is DHS_ERR_INVALID. */
int dhs_snapshot_free(dhs_ctx *ctx, int32_t snapshot_id);

/* Graph capture that keeps launch priorities (no counterpart in the paper).
 * dhs_round's request groups rely on the priorities of its internal streams,
 * which every kernel launch carries as an attribute; a CUDA graph ignores such
 * per-node priorities unless it is instantiated to use them.  dhs_graph_begin
 * starts capturing `stream` (relaxed mode); the caller then issues library
 * calls on it; dhs_graph_end stops the capture and instantiates the graph
 * with node priorities honoured.  dhs_graph_launch replays it on a stream;
 * dhs_graph_destroy frees it (NULL is a no-op).  DHS_ERR_CUDA if a CUDA call
 * fails (the capture is then ended and discarded). */
typedef struct dhs_graph dhs_graph;
int dhs_graph_begin(dhs_stream stream);
int dhs_graph_end(dhs_stream stream, dhs_graph **out);
int dhs_graph_launch(dhs_graph *graph, dhs_stream stream);
void dhs_graph_destroy(dhs_graph *graph);

/* One whole round on device buffers: select (causal domains at n_r + j),
 * resolve (shared retrieval), attend and commit, with the shapes of the
 * separate calls (topk_out and loc_out receive the selections and locations).
 * With cfg.round_groups = G > 1 the request slots are split into G contiguous
 * groups (the last one about 0.6 the size of the others, as nothing overlaps
 * its retrieval and attention) whose rounds are issued on G internal streams
 * forked from `stream`
 * and joined back into it before the call's work ends: requests are
 * independent ([ADHS] eq. (6): the union, misses and cache state are per
 * request), so one group's host gather (bound by the host link) can run while
 * another group's indexer (bound by HBM) runs -- the overlap of the copy path
 * with compute of [ADHS] 3.2 / 4.3.2.  The groups' selections run one
 * after another (group g's indexer starts when group g - 1's top-k has
 * finished), the internal streams have decreasing priorities in group order,
 * the rest of each group's round overlaps the next group's indexer, and a
 * group's attention starts once the next group's top-k has finished.
 * Results equal those of the separate
 * calls; the LRU clock advances once per call.  Forking and joining use CUDA
 * events, which stream capture turns into graph dependencies.  Not for
 * contexts on shared arenas or followers (DHS_ERR_INVALID).  Groups apply to
 * contexts whose attention is the tensor-core union pass; others (per-query
 * pass, union pass on mma.sync tiles) run the round as one group on `stream`. */
int dhs_round(dhs_ctx *ctx, const int8_t *q_idx, const int32_t *k_per_req, const void *q,
              const void *block_kv, const int32_t *accepted_len, int32_t *topk_out,
              int32_t *loc_out, void *out, float *lse, dhs_stream stream);

/* One whole round through host buffers: runs select, resolve (shared),
 * attend and commit on q_idx, q and block_kv in host memory and returns out
 * and lse (lse may be NULL) in host memory.  q_idx is copied to a device
 * buffer.  q, block_kv, out and lse are used in place when they are
 * page-locked (cudaHostAlloc / cudaHostRegister): the attention kernel reads
 * and writes them across the host link.  Pageable buffers are copied through
 * device buffers instead.  Synchronises `stream` before returning.  Shapes as
 * in the calls above.  With cfg.round_groups > 1 the round runs through
 * dhs_round (request groups on internal streams). */
int dhs_round_host(dhs_ctx *ctx, const int8_t *q_idx, const int32_t *k_per_req, const void *q,
                   const void *block_kv, const int32_t *accepted_len, void *out, float *lse,
                   dhs_stream stream);

const char *dhs_strerror(int code);

/* Indexer scores and ordered top-k without allocating anything.
 *
 * The paper has no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory at the moment they need a selection:
 * code recording a CUDA graph (cudaMalloc is not allowed during stream
 * capture), plug-ins inside an inference engine that owns every byte of
 * device memory, and decode loops where cudaMalloc or cudaFree would
 * synchronise the device.  It computes what dhs_select computes for one
 * request whose queries all see the whole key array, with no context:
 *   q_idx     device int8 [n_queries][idx_row_bytes], 16-byte aligned
 *   keys      device int8 [n_rows][idx_row_bytes], 16-byte aligned
 *   topk_out  device int32 [n_queries][topk]: rows by score descending,
 *             ties to the lower row, padded with -1 when n_rows < topk
 * Limits: 1 <= n_queries <= 8, 16 <= idx_row_bytes <= 1024 (a multiple of
 * 16), topk a multiple of 32 up to 4096, and n_queries * n_rows <= 2^21
 * (DHS_ERR_CAPACITY beyond it).  The intermediate scores live in one
 * fixed 8 MiB array inside the library image, which every GPU that loads
 * the library keeps until the process exits; no call allocates or frees
 * memory.  The first call on a device looks up that array's device address
 * (once per device, with the device current), so make the first call before
 * any stream capture.  All calls share the array and it keeps the last
 * call's contents: calls that overlap on the GPU race, so order them (for
 * example on one stream). */
int dhs_select_noalloc(const int8_t *q_idx, const int8_t *keys, int32_t n_queries,
                       int64_t n_rows, int32_t idx_row_bytes, int32_t topk, int32_t *topk_out,
                       dhs_stream stream);

/* ------------------------------------------------------------------------
 * Physical-source sharing and layer groups, [ADHS] 2.2 ("physical-source
 * sharing": Full, Reindex and Reuse layers), 3.2 (a Reuse consumer inherits
 * the preceding selected-location vector; a Reindex consumer re-selects over
 * the shared source, reusing the rows present; GLM-style index producers
 * announce positions for several follower payload layers) and 3.4 (staging
 * arenas reused across layer groups, M_stage = chi N K_max k d_KV).
 *
 * On one context (one physical source):
 *   - Reindex: after a round's dhs_attend and before its dhs_commit, another
 *     layer may call dhs_select (same K_r per request), dhs_resolve and
 *     dhs_attend again: the source's one cache state serves both selections,
 *     rows fetched for the earlier one stay available, and a fresh selection
 *     fetches only the rows absent from that state.
 *   - Reuse: dhs_attend may be called again after an attend of the same
 *     resolve, with another layer's queries and the same location vector:
 *     no resolution and no copy.  block_kv must be the same rows (the shared
 *     source's new rows; they are written to the draft ring again).
 *   - One dhs_commit ends the step for every layer of the source.
 * Across sources (layers with their own payload):
 *   - A follower layer (DHS_ROLE_FOLLOWER: no indexer scratch) takes the
 *     positions a producer's dhs_select returned: dhs_adopt(k_per_req, pos)
 *     sets the round's K_r and causal domains as dhs_select would, then
 *     dhs_resolve is given the producer's top-k list and fetches this
 *     source's own rows into this source's staging.
 *   - Layer groups: contexts created on shared arenas (dhs_create_on_arena)
 *     stage their misses in arena `arena` of the set instead of a staging
 *     buffer of their own; contexts of a layer group take distinct arenas,
 *     and the next group's contexts reuse them.  A resolve waits (on the GPU)
 *     for the attention readers of the arena's previous user; a resolve
 *     whose arena still holds another context's rows that no dhs_attend has
 *     read yet is refused (DHS_ERR_INVALID), as is an attend after another
 *     context took the arena.  Each call of such a context also waits for
 *     the work of that context's previous call, whatever stream it ran on,
 *     so a caller can issue the next group's resolves (with their host
 *     gathers) on a copy stream while this group attends on a compute
 *     stream.  These orderings use CUDA events recorded and waited on by the
 *     calls; issue them outside stream capture.  Not thread-safe: one host
 *     thread drives the contexts of a set of arenas.
 */
typedef struct dhs_arenas dhs_arenas;
enum { DHS_ROLE_FULL = 0, DHS_ROLE_FOLLOWER = 1 };

/* chi staging arenas, each n_slots * k_max * topk rows of row_elems bf16
 * (cudaMalloc on the current device).  DHS_ERR_INVALID for bad sizes,
 * DHS_ERR_OOM if the allocation fails. */
int dhs_arenas_create(int32_t chi, int32_t n_slots, int32_t k_max, int32_t topk,
                      int32_t row_elems, dhs_arenas **out);
/* Device bytes the arenas hold: M_stage = chi * n_slots * k_max * topk * row bytes. */
int64_t dhs_arenas_bytes(const dhs_arenas *arenas);
/* Frees the arenas (synchronises the device); DHS_ERR_INVALID while a
 * context created on them still exists.  NULL is a no-op. */
int dhs_arenas_destroy(dhs_arenas *arenas);

/* dhs_create for a source of a layer group: staging is arena `arena` (0 <=
 * arena < chi) of `arenas`, whose n_slots, k_max, topk and row width must
 * match the config.  role DHS_ROLE_FOLLOWER allocates no indexer scratch and
 * refuses dhs_select (it takes positions through dhs_adopt). */
int dhs_create_on_arena(const dhs_config *cfg, dhs_arenas *arenas, int32_t arena, int32_t role,
                        dhs_ctx **out);

/* A round whose positions another source's indexer chose ([ADHS] 3.2,
 * follower-layer copies): sets K_r (host int32 [n_slots]) and the causal
 * domains (pos as in dhs_select, NULL = n_r + j) exactly as dhs_select would,
 * without scoring; the caller then passes the producer's top-k list to
 * dhs_resolve (entries must be rows below this source's n_r).  Allowed where
 * dhs_select is. */
int dhs_adopt(dhs_ctx *ctx, const int32_t *k_per_req, const int64_t *pos, dhs_stream stream);

/* Text of the CUDA runtime error behind the context's last DHS_ERR_CUDA ("" if none). */
const char *dhs_last_error(const dhs_ctx *ctx);

/* ------------------------------------------------------------------------
 * Residency policy, [ADHS] 3.1, eq. (3) and (4): the host-side page accounting
 * that decides how much optional history each admitted request holds.  Pure
 * host logic (no CUDA call, no device); the caller carries its decisions out
 * with dhs_set_residency.  Units are pages (the workloads use 64-row pages).
 *
 * Budget, eq. (3): required pages (hot cache and tail, never lent) + optional
 * pages + reserve <= total, after every call.  The reclaim order is the
 * admission order, oldest first.  Not thread-safe: one caller per policy. */
typedef struct dhs_policy dhs_policy;

/* total_pages >= reserve_pages >= 0.  DHS_ERR_INVALID otherwise; DHS_ERR_OOM. */
int dhs_policy_create(int64_t total_pages, int64_t reserve_pages, dhs_policy **out);
void dhs_policy_destroy(dhs_policy *p); /* NULL is a no-op */

/* Admit `request` (an id not admitted now) with `required_pages` and
 * `history_pages` of imported history it could hold as optional pages.
 * When the free pages cover the required ones it is admitted and keeps
 * min(history, free - required) optional pages (resident-first admission).
 * Otherwise, with deficit D = required - free, the shortest prefix of the
 * reclaim order whose optional pages sum to at least D loses all of them,
 * eq. (4); those of its requests that held pages are written to reclaimed[]
 * (host int32, n_reclaimed of them), and the new request keeps
 * min(history, freed + free - required) optional pages.  If all optional
 * pages together cannot cover D, the admission waits: *admitted = 0 and
 * nothing changes.  The caller backs up a reclaimed request's history rows
 * and retires its optional rows (dhs_set_residency with no rows) before the
 * new request's pages are written.  DHS_ERR_INVALID for a bad argument or an
 * id already admitted; DHS_ERR_CAPACITY if required_pages exceeds total -
 * reserve (no reclaim or completion could ever admit it, so it is refused
 * instead of waiting) or if more than reclaimed_cap requests would lose
 * pages; nothing changes on an error. */
int dhs_policy_admit(dhs_policy *p, int32_t request, int64_t required_pages,
                     int64_t history_pages, int32_t *admitted, int64_t *optional_pages,
                     int32_t *reclaimed, int32_t reclaimed_cap, int32_t *n_reclaimed);

/* Completion releases the request's required and optional pages.
 * DHS_ERR_INVALID if it is not admitted. */
int dhs_policy_complete(dhs_policy *p, int32_t request);

/* One bounded round-robin repopulation attempt: starting after the request
 * the previous attempt served last, admitted requests (admission order,
 * cyclically, each visited once) get optional pages up to their history, in
 * total at most min(max_pages, free pages).  Writes (requests[i], pages[i]),
 * i < *n_out, the pages added per request; the caller copies those rows and
 * publishes them ready after the copy (dhs_set_residency).  cap must be at
 * least the number of admitted requests (DHS_ERR_CAPACITY, nothing changes). */
int dhs_policy_repopulate(dhs_policy *p, int64_t max_pages, int32_t *requests, int64_t *pages,
                          int32_t cap, int32_t *n_out);

/* The request's required, optional and history pages; DHS_ERR_INVALID if it
 * is not admitted. */
int dhs_policy_query(const dhs_policy *p, int32_t request, int64_t *required_pages,
                     int64_t *optional_pages, int64_t *history_pages);

/* total - reserve - required - optional pages; -1 for NULL. */
int64_t dhs_policy_free_pages(const dhs_policy *p);

#ifdef __cplusplus
}
#endif
#endif /* DHS_H_ */
