/*
 * forkkv.h -- C ABI of libforkkv: residual attention over a copy-on-write,
 * disaggregated KV cache, for one GB300 (sm_103a) GPU.
 *
 * Model (ForkKV guide, "Mathematical Decomposition of LoRA KV Activations"
 * and "The Disaggregated Memory Layout"; LRAgent summary, section 2
 * "BaseShared"):
 *   - many LoRA agents share one paged base cache (bCache) holding the
 *     post-RoPE keys Kb and values Vb computed with the frozen weights W0;
 *   - agent a keeps a rank-r_a residual cache (rCache) Lk_a = X A_k,a and
 *     Lv_a = X A_v,a ([T, r_a] per layer, shared by all kv heads) and its
 *     up-projections Bk_a, Bv_a ([r_a, H_kv*d] per layer);
 *   - for kv head h, agent a attends over
 *       K_a[t] = Kb[t] + s_a * RoPE_t(Lk_a[t] Bk_a[:, h*d:(h+1)*d])
 *       V_a[t] = Vb[t] + s_a * Lv_a[t] Bv_a[:, h*d:(h+1)*d]
 *     with rotate-half RoPE, theta_i = rope_base^(-2i/d), t the 0-based
 *     position in the agent's own sequence; query head hq reads kv head
 *     hq / (H_q/H_kv).
 *
 * Conventions shared by every call:
 *   - All tensors are row-major.  "bf16" is IEEE bfloat16 stored as uint16_t.
 *   - Device pointers ("dev") are CUDA global-memory addresses of the
 *     current device; host pointers ("host") are ordinary memory.  The
 *     caller owns every buffer it passes; the library keeps no pointer to a
 *     caller buffer after a call returns, except the pool carve-out given to
 *     fk_pool_create, which it uses until fk_pool_destroy.
 *   - Calls that take a stream enqueue work on it and return without
 *     synchronising; their device effects are ordered by that stream only.
 *     Calls on one pool must not run concurrently from several host threads,
 *     and kernels of two fk_residual_attention calls on one pool must not
 *     overlap on the GPU (they share the pool's workspace).
 *   - Every call returns an fk_status.  FK_OK is 0.  On failure nothing was
 *     enqueued, the pool's host state is unchanged, and fk_last_error()
 *     returns a message (thread-local, valid until the next call on that
 *     thread).  No call aborts, exits, or throws.
 */
#ifndef FORKKV_H
#define FORKKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int fk_status;
enum {
  FK_OK = 0,
  FK_ERR_INVALID_ARG = 1,   /* bad pointer, size, index, or state */
  FK_ERR_OUT_OF_PAGES = 2,  /* the page free list cannot satisfy the call */
  FK_ERR_OOM = 3,           /* a pool arena (rCache, workspace) is full */
  FK_ERR_UNSUPPORTED = 4,   /* shape the kernels do not implement */
  FK_ERR_CUDA = 5,          /* a CUDA runtime call failed */
  FK_ERR_DEVICE_CHECK = 6,  /* a kernel's own bounds check fired */
  FK_ERR_TIMEOUT = 7        /* a bounded device wait gave up */
};

/* Pool geometry.  All sizes are per layer unless stated. */
typedef struct fk_pool_config {
  int32_t n_layers;        /* >= 1 */
  int32_t n_q_heads;       /* H_q, a multiple of n_kv_heads */
  int32_t n_kv_heads;      /* H_kv */
  int32_t head_dim;        /* d: 64 or 128 */
  int32_t page_size;       /* P: must be 16 */
  int32_t num_pages;       /* physical bCache pages (page ids 0..num_pages-1,
                              the same ids name a page in every layer) */
  int32_t max_agents;      /* agent ids 0..max_agents-1 */
  int32_t max_rank;        /* largest r_a: a multiple of 8, <= 64 */
  int32_t max_tokens;      /* rCache capacity per agent (tokens) */
  int64_t rcache_rank_budget; /* sum of ranks of live agents the rCache
                              arena holds; 0 = max_agents * max_rank */
  int64_t workspace_bytes; /* device workspace for the cached work list and
                              split-K partials; 0 = 64 MiB */
  float   rope_base;       /* RoPE base (10000 for Llama-style layers) */
  int32_t compressed;      /* 1: also hold a compressed copy of the bCache
                              (int8 K, 3-bit V) for fk_pool_compress */
} fk_pool_config;

typedef struct fk_pool fk_pool;

/* Message of the last failed call on this thread ("" if none).  Library
 * plumbing: the pages define no error reporting; the convention is this
 * header's (see "Conventions shared by every call" above).  The pointer is
 * owned by the library and valid until the thread's next call. */
const char* fk_last_error(void);

/* Library version string. */
const char* fk_version(void);

/* Bytes of device memory the pool needs for `cfg` (0 and FK_ERR_* message
 * via fk_last_error if cfg is invalid).  The caller allocates them (e.g.
 * with torch) and hands them to fk_pool_create.  The carve-out holds the
 * two physically separate tiers of the ForkKV guide, "The Disaggregated
 * Memory Layout": the paged bCache (num_pages x n_layers x H_kv pages of
 * Kb and Vb) and the rCache arena (per agent, rank-r rows X A_k, X A_v of
 * max_tokens tokens per layer), plus each agent's Bk, Bv and the
 * workspace.  Host only; no device call. */
size_t fk_pool_bytes(const fk_pool_config* cfg);

/* Create a pool over the caller's device carve-out `dev_buf` (dev, 256-byte
 * aligned, >= fk_pool_bytes(cfg) bytes).  The buffer's contents need not be
 * initialised.  Host metadata (page free list and reference counts, agent
 * table) lives in the returned handle.  Uses the current CUDA device.  The
 * pool is the ForkKV guide's "DisaggregatedKVCache" ("Complete End-to-End
 * Implementation", item 2: it manages the physical bCache and rCache
 * memory pools) with the tiers of "The Disaggregated Memory Layout".
 * FK_ERR_INVALID_ARG on a bad config, a NULL or misaligned buffer, or too
 * few bytes (*out is then untouched); FK_ERR_CUDA if a device call fails.
 * Environment (read here, fixed for the pool's life):
 * FORKKV_DECODE_SLOTS=8 plans decode-shaped calls with d = 128 on the
 * uncompressed pool in tiles of eight agents (every base page read once
 * per kv head) instead of four. */
fk_status fk_pool_create(const fk_pool_config* cfg, void* dev_buf,
                         size_t bytes, fk_pool** out);
/* Free the handle and its host metadata (NULL: FK_ERR_INVALID_ARG).  The
 * caller must have synchronised every stream with work on the pool; the
 * carve-out stays the caller's to free.  Library plumbing (the pages
 * describe no teardown beyond reclaiming an agent's rCache, "Reference
 * Counting and Eviction"). */
fk_status fk_pool_destroy(fk_pool* pool);

/* Byte offset and size of a region of the pool carve-out, for reading the
 * pool back in tests and tools.  Regions and their element layouts:
 *   0 FK_REGION_KB   bf16 base keys:  [L][num_pages][H_kv][2][d/8][8][8]
 *                    (token-group of 8, d-chunk of 8, token, d: the
 *                    core-matrix order tensor cores read directly)
 *   1 FK_REGION_VB   bf16 base values: [L][num_pages][H_kv][2][d/8][8][8]
 *                    (token-chunk of 8, d-group of 8, d, token: values are
 *                    stored transposed inside each 8x8 core)
 *   2 FK_REGION_RC   rCache arena.  Per agent and layer: Lk as
 *                    [T_cap/8][rp/8][8][8] (token-group, r-chunk, token,
 *                    r), then Lv as [T_cap/8][rp/8][8][8] (token-chunk,
 *                    r-group, r, token); rp = rank rounded up to 16 (the
 *                    padding columns hold zeros), T_cap = max_tokens
 *                    rounded up to 128.  Rows never appended hold zeros.
 *   3 FK_REGION_KQ   int8 keys [L][num_pages][H_kv][16][d]
 *   4 FK_REGION_VC   3-bit value codes [L][num_pages][H_kv][16][3*d/8]
 *                    (three bit planes; code i at bit i%8 of byte i/8)
 *   5 FK_REGION_VN   fp32 value norms [L][num_pages][H_kv][16]
 *   6 FK_REGION_KS   fp32 key scale per layer [L]
 */
enum { FK_REGION_KB = 0, FK_REGION_VB = 1, FK_REGION_RC = 2,
       FK_REGION_KQ = 3, FK_REGION_VC = 4, FK_REGION_VN = 5,
       FK_REGION_KS = 6 };
fk_status fk_pool_region(const fk_pool* pool, int region, size_t* offset,
                         size_t* bytes);

/* ---- pages: reference-counted, copy-on-write (ForkKV guide, "The
 * Copy-on-Write Paradigm" and "Reference Counting and Eviction") ---- */

/* Take `n` free pages; their ids go to page_ids (host, n entries) with
 * reference count 1 and no tokens.  FK_ERR_OUT_OF_PAGES if fewer than n are
 * free (then none is taken). */
fk_status fk_pages_alloc(fk_pool* pool, int n, int32_t* page_ids);

/* Drop one reference to each page (host ids, n entries; -1 entries are
 * skipped).  A page whose count reaches 0 returns to the free list.
 * FK_ERR_INVALID_ARG (and no change) if any id is out of range or already
 * free. */
fk_status fk_pages_release(fk_pool* pool, int n, const int32_t* page_ids);

/* Fork: child_row[i] = parent_row[i] for i < n_pages and one more reference
 * to each named page (host arrays; -1 entries are copied as -1). */
fk_status fk_fork(fk_pool* pool, const int32_t* parent_row, int n_pages,
                  int32_t* child_row);

/* Current reference count of a page (0 = free), or -1 if out of range. */
int fk_page_refcount(const fk_pool* pool, int32_t page_id);

/* ---- agents ---- */

/* Register agent `agent` with rank `rank` (multiple of 8, <= max_rank) and
 * residual scale `s` (alpha/r of the adapter: ForkKV guide, "Mathematical
 * Decomposition of LoRA KV Activations", Delta K = (alpha/r) X A_k B_k and
 * likewise for V; the rCache keeps the factored X A, "The Disaggregated
 * Memory Layout", item 2), copying its up-projections
 * Bk, Bv (dev bf16 [n_layers][rank][H_kv*d]) into the pool and reserving
 * its rCache (n_layers x max_tokens x rank for Lk and for Lv).
 * FK_ERR_INVALID_ARG if the id is taken; FK_ERR_OOM if the rCache arena is
 * full.  Ranks that are not a multiple of 8 must be zero-padded by the
 * caller (padding columns of Lk/Lv and rows of Bk/Bv set to 0). */
fk_status fk_agent_register(fk_pool* pool, int agent, int rank, float s,
                            const uint16_t* Bk, const uint16_t* Bv,
                            void* stream);
fk_status fk_agent_release(fk_pool* pool, int agent);

/* Shared-A (LRAgent summary, "BaseLRShared"): register agent `agent` with
 * its own up-projections Bk, Bv and scale s but no rCache of its own: it
 * reads the low-rank rows of live agent `src` (same rank; with A shared by
 * the adapters, X A is the same for all of them), so those rows are stored
 * and streamed once.  Appends through either agent write the shared rows.
 * The rows are reclaimed when the last agent using them is released.
 * FK_ERR_INVALID_ARG if `agent` is taken or `src` is not live. */
fk_status fk_agent_register_shared(fk_pool* pool, int agent, int src, float s,
                                   const uint16_t* Bk, const uint16_t* Bv, void* stream);

/* Where agent `agent`'s residual cache lives: byte offset (from the pool
 * carve-out) of its layer-0 Lk block, the bytes one layer of Lk+Lv takes
 * (Lv follows Lk after half of them), and its padded rank (rank rounded up
 * to 16).  For reading the pool back in tests and tools. */
fk_status fk_agent_rcache(const fk_pool* pool, int agent, size_t* lk_offset,
                          size_t* layer_bytes, int* padded_rank);

/* ---- appends ---- */

/* Write base keys/values of tokens pos..pos+n-1 of one sequence into layer
 * `layer` of the bCache (ForkKV guide, "The Disaggregated Memory Layout",
 * item 1: base states, computed once, shared and immutable once shared;
 * "The Copy-on-Write Paradigm": a writer gets a private copy) pages named
 * by `block_table_row` (host, max_pages
 * entries, logical page -> page id, -1 = none).  Kb, Vb: dev bf16
 * [n][H_kv][d], post-RoPE.  Missing pages (-1) are allocated and written
 * into the row.  A named page whose reference count is above 1 is shared:
 * it is copied to a fresh page (all layers), the row entry is rewritten to
 * the copy and the shared page loses one reference (copy-on-write), so
 * shared pages are never written.  FK_ERR_OUT_OF_PAGES if pages run out
 * (the row may then hold pages allocated before the failure; they stay
 * valid). */
fk_status fk_base_append(fk_pool* pool, int layer, int32_t* block_table_row,
                         int max_pages, int pos, int n, const uint16_t* Kb,
                         const uint16_t* Vb, void* stream);

/* Write residual rows of tokens pos..pos+n-1 of agent `agent`, layer
 * `layer`: Lk, Lv dev bf16 [n][rank] (Lk = X A_k, Lv = X A_v of those
 * tokens: the factored rank-r activations the rCache stores, ForkKV guide,
 * "The Disaggregated Memory Layout", item 2).  pos + n <= max_tokens.
 * FK_ERR_INVALID_ARG for an agent that is not live or rows out of range
 * (nothing is launched); FK_ERR_CUDA if the copy kernel fails to launch. */
fk_status fk_residual_append(fk_pool* pool, int layer, int agent, int pos,
                             int n, const uint16_t* Lk, const uint16_t* Lv,
                             void* stream);

/* Low-rank prefill of agent `agent`, layer `layer`: computes Lk = X A_k and
 * Lv = X A_v for tokens pos..pos+n-1 on the device and writes them into the
 * agent's rCache (ForkKV guide, "Two-Tier Lookup Mechanics", case B: the
 * base cache already holds the prefix, so only the adapter's low-rank
 * projection of the hidden states is computed; LRAgent summary,
 * "BaseShared").  X: dev bf16 [n][d_model] row-major, the layer's input
 * hidden states (after its norm) of those tokens; Ak, Av: dev bf16
 * [d_model][rank] row-major (rank = the agent's registered rank).  The
 * product accumulates in fp32 over d_model and is rounded once to bf16
 * (nearest even).  d_model a positive multiple of 128; X, Ak, Av 16-byte
 * aligned; pos + n <= max_tokens.  The caller keeps ownership of X, Ak,
 * Av, which must stay valid until the stream reaches the call.  For a
 * Shared-A agent the rows land in the rCache it shares.
 * FK_ERR_INVALID_ARG on a bad argument (nothing is launched); a launch
 * failure is FK_ERR_CUDA; a kernel that timed out on a wait sets the
 * pool's error word (fk_check) and writes no rows. */
fk_status fk_residual_prefill(fk_pool* pool, int layer, int agent, int pos, int n,
                              const uint16_t* X, const uint16_t* Ak, const uint16_t* Av,
                              int d_model, void* stream);

/* ---- compressed shared pool (PolyKV summary, section 2B) ---- */

/* Encode layer `layer` of every live page (reference count > 0, rows that
 * hold tokens) into the compressed copy: keys as int8 with one fp32 scale
 * for the whole layer (scale = max|K|/127, codes = round-half-even(K/scale)
 * clamped to +-127); each value vector v (per token and kv head) as its
 * fp32 norm n and the 3-bit index of the nearest 8-level Lloyd-Max level
 * (unit normal) of each coordinate of z = H v / n, H the unnormalised
 * Sylvester Hadamard matrix (ties go to the upper level).  Needs
 * cfg.compressed = 1. */
fk_status fk_pool_compress(fk_pool* pool, int layer, void* stream);

/* Load an already-encoded layer: for the n_pages pages in page_ids (host),
 * kq (dev int8 [n_pages][16][H_kv][d]), vcodes (dev uint8
 * [n_pages][16][H_kv][3*d/8], bit planes as in FK_REGION_VC) and vnorm (dev
 * fp32 [n_pages][16][H_kv]) are copied into the compressed copy, and the
 * layer's key scale is set to k_scale. */
fk_status fk_pool_load_compressed(fk_pool* pool, int layer,
                                  const int32_t* page_ids, int n_pages,
                                  const int8_t* kq, const uint8_t* vcodes,
                                  const float* vnorm, float k_scale,
                                  void* stream);

/* ---- the hot path ---- */

/* Residual attention of A agents, C query rows each, at layer `layer`.
 *   q        dev bf16 [A][C][H_q][d], post-RoPE; row c of agent i sits at
 *            position seq_lens[i] - C + c.
 *   agents   host int32 [A], registered agent ids (distinct).
 *   block_table host int32 [A][max_pages], logical page -> page id.
 *   seq_lens host int32 [A], keys per agent (C <= seq_lens[i]); the agent's
 *            residual rows 0..seq_lens[i]-1 must have been appended.
 *   causal   1: row c sees keys t <= seq_lens[i] - C + c; 0: all keys.
 *   compressed 1: read the compressed copy of the bCache (keys dequantised
 *            in the kernel, values accumulated in the rotated domain and
 *            rotated back once per output row); 0: the bf16 bCache.
 *   out      dev bf16 [A][C][H_q][d], written with round-to-nearest-even.
 * Pages that several agents name at the same logical index are streamed
 * from HBM once per kv head for all of them.  The work list built from
 * (agents, block_table, seq_lens, A, C, causal) is cached in the pool and
 * reused while those inputs are unchanged.  Per-token residual keys are
 * rebuilt on chip (Lk Bk then RoPE) and the value residual is applied
 * factored as (P Lv) Bv after the split-K combine (LRAgent summary,
 * section 3 "Flash-LoRA-Attention"). */
fk_status fk_residual_attention(fk_pool* pool, int layer, const uint16_t* q,
                                const int32_t* agents,
                                const int32_t* block_table, int max_pages,
                                const int32_t* seq_lens, int A, int C,
                                int causal, int compressed, uint16_t* out,
                                void* stream);

/* Same computation and arguments as fk_residual_attention, for callers
 * that must not allocate device memory per call or share the pool's
 * workspace: for example a plug-in living inside a host program that owns
 * all of the GPU's memory through its own allocator (and has handed nearly
 * all of it to KV pages), so that any cudaMalloc from this library would
 * fail or would break that program's memory accounting.  No page of the
 * paper describes this call; it is a deployment aid.
 *
 * The per-call scratch (the work list and the split-K partials) lives in a
 * file-scope device array of FK_NOALLOC_SCRATCH_BYTES bytes inside the
 * library instead of the pool's workspace; every GPU that loads the library
 * keeps that array until the process exits.  The call allocates nothing: no
 * cudaMalloc, cudaFree, pinned-host or other allocating routine.  Calls
 * whose work list and partials need more than FK_NOALLOC_SCRATCH_BYTES
 * fail with FK_ERR_OOM and a message giving the size needed.  The first
 * call on a device looks up the array's device address (set-up done once
 * per device), so make that first call before any stream capture.  A call
 * whose work list differs from the last one on the device (other inputs,
 * another pool, agents registered or pages changed since) uploads it with
 * a copy from host memory the library keeps, which stream capture does
 * not take: make such calls outside capture; repeat calls with unchanged
 * inputs on the same pool enqueue only the kernels.  All calls share the
 * one array, which keeps the last call's contents; calls whose kernels
 * overlap on the GPU (other streams, other pools) race on it and must be
 * ordered by the caller.  FK_ERR_INVALID_ARG if the current CUDA device is
 * not the pool's (the array is per device). */
#define FK_NOALLOC_SCRATCH_BYTES (16u << 20)
fk_status fk_residual_attention_noalloc(fk_pool* pool, int layer,
                                        const uint16_t* q,
                                        const int32_t* agents,
                                        const int32_t* block_table,
                                        int max_pages,
                                        const int32_t* seq_lens, int A, int C,
                                        int causal, int compressed,
                                        uint16_t* out, void* stream);

/* Number of kernel launches the last fk_residual_attention enqueued. */
int fk_last_launch_count(const fk_pool* pool);

/* Measurement hook: if `event` (a cudaEvent_t, or NULL to clear) is set,
 * every later fk_residual_attention records it on its stream right after
 * the main attention kernel and before the split-K combine, so the main
 * kernel can be timed alone with CUDA events.  The event stays owned by the
 * caller. */
fk_status fk_pool_set_profile_event(fk_pool* pool, void* event);

/* Failure-detection test hook.  While `on` is nonzero, every later
 * fk_residual_attention call on the pool that runs the four-agent decode
 * kernel (decode-shaped calls, see fk_residual_attention) makes that
 * kernel's key-copy warp also wait on a barrier that nothing completes.
 * The wait gives up after its bound (about 2 s of GPU clock), the CTA takes
 * the same abort path as any timed-out wait (no further copy or MMA is
 * issued, MMAs in flight are drained, copies in flight get a grace period)
 * and the next fk_check returns FK_ERR_TIMEOUT.  The output of such a call
 * is undefined.  No GPU fault, trap or hang is involved; the pool and the
 * context stay usable.  Off by default.  Host only. */
fk_status fk_pool_set_test_stall(fk_pool* pool, int on);

/* Synchronise `stream` and read the pool's device error word: FK_OK, or
 * FK_ERR_DEVICE_CHECK if a kernel's bounds check fired since the last
 * fk_check (the word is then cleared). */
fk_status fk_check(fk_pool* pool, void* stream);

/* ---- work list (host only; exposed for inspection and tests) ---- */

/* One unit of GPU work: kv head `head`, rows [row_begin, row_begin+n_rows)
 * of the row table, consecutive logical pages lp_begin.. of page list
 * entries [page_begin, page_begin+n_pages), agents [agent_begin,
 * agent_begin+n_agents) of the tile agent list. */
typedef struct fk_work_item {
  int32_t head, row_begin, n_rows, page_begin, n_pages, lp_begin,
          agent_begin, n_agents, partial_begin, sum_rank;
} fk_work_item;

/* Build the work list for a call shape without a pool or GPU.  Outputs are
 * host arrays of the given capacities; counts go to *n_*.  row_agent[i] is
 * the call-local agent index of row i, row_cg[i] = c * G + g.  tile_agents
 * holds call-local agent indices.  page_ids holds physical page ids.
 * ranks: host int32 [A] ranks of the call's agents.  max_rows_per_tile,
 * max_rank_sum_per_tile: tile limits; target_items: desired work items
 * (e.g. 2 x SM count). */
fk_status fk_plan_host(int A, int C, int H_q, int H_kv, int page_size,
                       const int32_t* block_table, int max_pages,
                       const int32_t* seq_lens, const int32_t* ranks,
                       int max_rows_per_tile, int max_rank_sum_per_tile,
                       int target_items,
                       fk_work_item* items, int cap_items, int* n_items,
                       int32_t* row_agent, int32_t* row_cg, int cap_rows,
                       int* n_rows,
                       int32_t* page_ids, int cap_pages, int* n_pages,
                       int32_t* tile_agents, int cap_tile_agents,
                       int* n_tile_agents);

/* The work list of a decode-shaped call (four query rows per agent: G * C
 * == 4) in eight-slot tiles, as the eight-slot decode kernel runs it (pools
 * created with FORKKV_DECODE_SLOTS=8).  Same arguments and outputs as
 * fk_plan_host, with fixed tile limits: tile_agents holds 8 entries per
 * tile (-1: an empty slot); slot s owns the tile's rows 4 s .. 4 s + 3
 * (row_agent -1 on an empty slot's rows); each half of a tile (slots 0-3,
 * 4-7) holds at most 64 padded ranks.  FK_ERR_INVALID_ARG unless G * C ==
 * 4.  Host only. */
fk_status fk_plan_host_slots8(int A, int C, int H_q, int H_kv, int page_size,
                              const int32_t* block_table, int max_pages,
                              const int32_t* seq_lens, const int32_t* ranks,
                              int target_items, fk_work_item* items, int cap_items,
                              int* n_items, int32_t* row_agent, int32_t* row_cg,
                              int cap_rows, int* n_rows, int32_t* page_ids,
                              int cap_pages, int* n_pages, int32_t* tile_agents,
                              int cap_tile_agents, int* n_tile_agents);

/* Work list of the chunk kernel, the path of calls with at least 128 query
 * rows per agent and kv head (G * C >= 128, d = 128, uncompressed pool),
 * built without a pool or GPU.  Items: head, row_begin (first of the
 * item's rows among the agent's G*C rows, row index c * G + g), n_rows
 * (<= 128), page_begin (into page_ids), n_pages, lp_begin (first logical
 * page, a multiple of 8), agent_begin (the call agent), n_agents = 1,
 * partial_begin (the item's first split-partial slot; one slot per row).
 * CTA c runs items cta_begin[c] .. cta_begin[c+1]-1 (*n_cta entries).
 * csr_ptr (A * C * H_q + 1 entries) and csr_slots list the partial slots
 * of every output row (a, c, hq) in row order.  FK_ERR_OOM (with the
 * counts set) if a capacity is too small; FK_ERR_INVALID_ARG for a bad
 * shape or block table. */
fk_status fk_plan_chunk_host(int A, int C, int H_q, int H_kv, const int32_t* block_table,
                            int max_pages, const int32_t* seq_lens, int n_ctas,
                            fk_work_item* items, int cap_items, int* n_items, int32_t* cta_begin,
                            int cap_cta, int* n_cta, int32_t* page_ids, int cap_pages,
                            int* n_pages, int32_t* csr_ptr, int cap_ptr, int32_t* csr_slots,
                            int cap_slots, int* n_slots);

/* ------------------------------------------------ two-tier prefix index --
 * Host-only index above the page pool (ForkKV guide, "DualRadixTree:
 * Two-Tier Hierarchical Cache Indexing", "Two-Tier Lookup Mechanics" and
 * "Reference Counting and Eviction").  Tier 1 is a radix tree over prompt
 * token prefixes at page granularity: each node owns the physical bCache
 * page ids of its span.  Tier 2 is a set of adapter leaves per node: an
 * adapter id bound to the owner of its residual rows for that prefix (for
 * example the pool agent slot).  A node counts the adapter leaves at or
 * below it; only nodes with no such leaf and no children are evicted,
 * least recently used first.  Only whole pages of an exactly equal prefix
 * are indexed (a page's keys and values depend on every earlier token).
 *
 * A node handle (int64) names the end of a cached prefix; handles stay valid
 * until that node is evicted.  Handle 0 is the empty prefix.  The index
 * takes over one pool reference per page passed to fk_radix_insert and gives
 * it back through the ids that fk_radix_evict returns (release them with
 * fk_pages_release).  Not thread-safe: one host thread per index.
 * Errors: FK_ERR_INVALID_ARG with fk_last_error() set; nothing changes. */
typedef struct fk_radix fk_radix;

fk_status fk_radix_create(int page_size, fk_radix** out);
void fk_radix_destroy(fk_radix* index);

/* Tier-1 lookup: the longest cached page prefix of tokens[0, n_tokens).
 * *n_matched = whole pages matched; *node = handle of that prefix's end
 * (a node is split when the match ends inside its span).  If pages is not
 * NULL, the matched page ids are written there (cap_pages >= *n_matched).
 * Marks the prefix as used now. */
fk_status fk_radix_match(fk_radix* index, const int32_t* tokens, int n_tokens, int32_t* pages,
                         int cap_pages, int* n_matched, int64_t* node);

/* Caches the whole pages of tokens[0, n_tokens): new_pages[0, n_new) are the
 * ids of the pages after the currently cached prefix, which n_new must cover
 * exactly (floor(n_tokens / page_size) - cached pages).  *node = handle of
 * the prompt's last whole page. */
fk_status fk_radix_insert(fk_radix* index, const int32_t* tokens, int n_tokens,
                          const int32_t* new_pages, int n_new, int64_t* node);

/* Tier 2 at a node: *owner = the adapter's owner, or -1 if it has no leaf
 * (a full hit needs both tiers; base only is the partial hit). */
fk_status fk_radix_adapter_get(fk_radix* index, int64_t node, int32_t adapter, int32_t* owner);
/* Adds the adapter's leaf (counted by the node and all its ancestors). */
fk_status fk_radix_adapter_attach(fk_radix* index, int64_t node, int32_t adapter, int32_t owner);
/* Removes the leaf; *owner (if not NULL) = its owner, whose residual rows
 * the caller reclaims at once (fk_agent_release). */
fk_status fk_radix_adapter_detach(fk_radix* index, int64_t node, int32_t adapter, int32_t* owner);

/* Evicts unreferenced leaf nodes, least recently used first, until at least
 * want_pages page ids are written to pages_out (or no node is evictable, or
 * the next node's pages would not fit in cap_pages); *n_out = ids written. */
fk_status fk_radix_evict(fk_radix* index, int want_pages, int32_t* pages_out, int cap_pages,
                         int* n_out);

/* Cached nodes (not counting the empty prefix) and pages. */
fk_status fk_radix_stats(const fk_radix* index, int64_t* n_nodes, int64_t* n_pages);
/* Adapter leaves at or below a node. */
fk_status fk_radix_node_ref(const fk_radix* index, int64_t node, int64_t* ref);

/* ---------------------------------------------- workflow-aware eviction --
 * KVFlow review, "Agent Step Graph and Steps-to-Execution" and
 * "Workflow-aware eviction".  An agent's steps-to-execution is the number of
 * workflow steps before it runs again.  Each agent marks its fixed-prompt
 * prefix node (and every ancestor) with that value; a node's priority is the
 * smallest value marking it, so a prefix shared by several agents is kept
 * while any of them runs soon.  fk_radix_evict_workflow then evicts the
 * evictable leaf (no adapter leaf at or below it, no children) with the
 * largest priority first: unmarked nodes (dynamic suffixes) before every
 * marked node, equal priorities least recently used first; a parent becomes
 * a candidate once its last child is gone.  Evicting a node leaves the marks
 * its agents put on the ancestors (the agent still needs the shared prefix).
 * A split copies the marks of the split node to its new prefix node. */

/* One agent with steps-to-execution `step` (>= 0) whose fixed prompt ends
 * at `node` (not the root): +1 on that step's count at node and ancestors. */
fk_status fk_radix_priority_assign(fk_radix* index, int64_t node, int32_t step);
/* Undoes one such assignment (FK_ERR_INVALID_ARG, and no change, if a node
 * on the path holds no count for that step). */
fk_status fk_radix_priority_release(fk_radix* index, int64_t node, int32_t step);
/* Drops every assignment (before marking the next workflow step's values). */
fk_status fk_radix_priority_clear(fk_radix* index);
/* *priority = the node's priority, or -1 if no agent marks it. */
fk_status fk_radix_node_priority(const fk_radix* index, int64_t node, int32_t* priority);
/* Evicts as described above until at least want_pages page ids are written
 * to pages_out (or nothing is evictable, or the next node's pages would not
 * fit in cap_pages); *n_out = ids written, in eviction order. */
fk_status fk_radix_evict_workflow(fk_radix* index, int want_pages, int32_t* pages_out,
                                  int cap_pages, int* n_out);

/* Steps-to-execution of every agent of an agent step graph.  Agent i's
 * predecessors are preds[pred_offsets[i] .. pred_offsets[i+1]) (host, CSR,
 * pred_offsets[0] = 0, ids in [0, n_agents)); join[i] is FK_JOIN_AND (the
 * agent waits for all predecessors: max of their values + 1) or FK_JOIN_OR
 * (any predecessor triggers it: min + 1); fixed[i] >= 0 gives agent i's
 * value directly (e.g. 0 for agents that run in the current step), -1 lets
 * it be computed.  steps[i] (host, out) = the value, or -1 if the agent
 * never runs: no fixed value and no predecessor, an AND over a predecessor
 * that never runs, or an OR whose predecessors all never run.
 * FK_ERR_INVALID_ARG (steps untouched) on bad arguments or on a cycle whose
 * agents have no fixed value. */
enum { FK_JOIN_AND = 0, FK_JOIN_OR = 1 };
fk_status fk_workflow_steps(int n_agents, const int32_t* pred_offsets, const int32_t* preds,
                            const int32_t* join, const int32_t* fixed, int32_t* steps);

#ifdef __cplusplus
}
#endif
#endif /* FORKKV_H */
