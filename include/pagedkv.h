/*
 * pagedkv.h -- C ABI of the GB300 paged-KV decode-attention library.
 *
 * The library keeps the KV cache of a tree of decoding branches (the
 * trajectories of a reasoning search tree) in fixed 16-token blocks of a
 * caller-owned device pool.  Each branch has a block table; a fork points the
 * child at the parent's full blocks and adds a reference to each, so shared
 * prefixes are never copied; only a partial last block is copied
 * (copy-on-write); a block whose reference count drops to zero returns to the
 * free stack at once.  Decode attention reads every branch's keys/values
 * through its block table, and reads each shared-prefix block from HBM once
 * for all branches that share it.
 *
 * Sources ("page" = the web page, with its section):
 *   [TRM] "The Reasoning Engine Meltdown", §2.1 (attention, Memory_KV),
 *         §5 (paged tree, fork rules), §6 (TreePagedKVCacheManager).
 *   [DMW] "Dismantling the Memory Wall", PagedAttention section (16-token
 *         blocks, BlockTable.get_block_for_token), copy-on-write section.
 *   [RKSC] RKSC summary, §2.C RSBCM (eviction score omega).
 *
 * Conventions
 *   - Every function except kv_last_error / kv_bytes_per_token returns a
 *     kv_status.  On any error the call changes no state (pool metadata,
 *     device memory) and kv_last_error() describes the error.
 *   - A kv_pool is not thread-safe: the caller serialises calls on one pool.
 *   - The library never allocates device memory.  Pools, queries, outputs,
 *     tables, plans and workspaces are caller-owned device (or host, where
 *     stated) buffers.  The library owns only host metadata.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is asynchronous on that stream.
 *   - bf16 means IEEE bfloat16 (16-bit storage).
 *   - e4m3 means the 8-bit floating-point format with a sign bit, 4 exponent
 *     bits (bias 7) and 3 mantissa bits, no infinities, NaN = S.1111.111,
 *     largest finite magnitude 448 (exponent field 0: subnormals m/8 * 2^-6).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t kv_status;

#define KV_OK 0
#define KV_ERR_OOM 1          /* pool has too few free blocks ([TRM] §6 MemoryError) */
#define KV_ERR_INVALID_ARG 2  /* bad size, pointer, layout or plan */
#define KV_ERR_NOT_FOUND 3    /* unknown or already-freed branch ([TRM] §6 KeyError) */
#define KV_ERR_CUDA 4         /* a CUDA runtime call failed */
#define KV_ERR_DEVICE 5       /* a kernel recorded a bad block id / bad item */
#define KV_ERR_TIMEOUT 6      /* a kernel's bounded wait ran out */
#define KV_ERR_INTERNAL 7     /* an invariant of the library broke (a bug) */

/* Eviction stop rules for kv_evict. */
#define KV_STOP_FREE_BLOCKS 0     /* stop once >= target blocks are free */
#define KV_STOP_EVICTED_LEAVES 1  /* stop once >= target leaf nodes were freed */

/* Flags for paged_decode_plan. */
#define KV_PLAN_NO_TENSOR_CORES 1 /* route every segment through the per-row
                                     (mma.sync) kernel, never tcgen05 */
#define KV_PLAN_IGNORE_GROUPS 2   /* treat every branch as unshared (each
                                     branch re-reads its whole table) */
#define KV_PLAN_KV_E4M3 4         /* the step reads an e4m3 pool
                                     (paged_decode_attn_e4m3) */
#define KV_PLAN_NARROW_TILES 8    /* tcgen05 tiles of 128 rows only (no
                                     256-row items; used to compare the two
                                     tile kernels) */

/* Element type of a pool's K and V. */
#define KV_DTYPE_BF16 0
#define KV_DTYPE_E4M3 1

typedef struct kv_pool kv_pool; /* opaque */

typedef struct kv_pool_desc {
  int64_t num_blocks;   /* physical blocks in the pool, >= 1 */
  int32_t block_size;   /* tokens per block; must be 16 ([DMW]) */
  int32_t num_layers;   /* >= 1 */
  int32_t num_kv_heads; /* Hkv >= 1 */
  int32_t head_dim;     /* d: 64 or 128 */
  /* Device pools, caller-owned, each (bf16 pools)
   * [num_layers][num_blocks][num_kv_heads][block_size][head_dim] bf16,
   * 16-byte aligned.  Both NULL: a metadata-only pool (the allocator, tables
   * and eviction run; appends and forks move no data). */
  void* k_pool;
  void* v_pool;
  /* Host, nullable: a permutation of 0..num_blocks-1; element 0 is the first
   * block handed out.  NULL: ascending ids.  Copied; not retained. */
  const int32_t* initial_free_order;
  /* KV_DTYPE_BF16 (layout above) or KV_DTYPE_E4M3.  An e4m3 pool stores
   * each (layer, block, kv-head) K tile and V tile as 16 * head_dim e4m3
   * codes (k_pool, v_pool: [num_layers][num_blocks][num_kv_heads][16 *
   * head_dim] bytes) and one 16-byte scale record per (layer, block,
   * kv-head) in kv_scales ([num_layers][num_blocks][num_kv_heads] x
   * {float k_scale, float v_scale, 2 reserved words}, device, 16-byte
   * aligned).  Stored value = code value * scale; each scale is a power of
   * two 2^e, e in [-126, 120], the smallest with max|x| <= 448 * 2^e over
   * the tile's values (nothing saturates).  Byte order inside a tile, token
   * slot t, dimension c (0 <= c < head_dim):
   *   K: t * head_dim + c, except that for head_dim 128 the 16-byte chunk
   *      c / 16 of row t sits at chunk position (c / 16) ^ (t % 8);
   *   V: c * 16 + t (transposed: one 16-byte row of the 16 slots per
   *      dimension).
   * Writes quantise on the device: a write that starts a block (slot 0)
   * takes the scale of its own rows; a later write keeps the block's scale
   * unless its rows need a larger one, in which case the rows already
   * stored are re-encoded from their stored values under the new scale.
   * Each value is coded as the nearest e4m3 value of x / scale, ties to the
   * even mantissa.  Non-finite inputs give unspecified codes.  kv_scales
   * must be NULL for bf16 pools and for metadata-only pools. */
  int32_t kv_dtype;
  void* kv_scales;
} kv_pool_desc;

typedef struct kv_branch_info_t {
  int32_t live;       /* 1 until freed or evicted */
  int32_t parent;     /* -1 for a root */
  int32_t depth;      /* 0 for a root, parent's depth + 1 for a fork */
  int32_t seq_len;    /* cached tokens (0 once freed) */
  int32_t n_blocks;   /* entries in the block table = ceil(seq_len / 16) */
  int32_t n_children; /* forks ever made from this branch */
} kv_branch_info_t;

/* ---- pool lifetime ------------------------------------------------------ */

/* Create a pool over caller-owned device memory ([TRM] §6 __init__: a fixed
 * set of physical pages, all free).  The free stack starts in
 * initial_free_order (or ascending ids).  Errors: INVALID_ARG (sizes, a
 * non-permutation order, exactly one of k_pool / v_pool NULL).  *out is
 * released with kv_pool_destroy. */
kv_status kv_pool_create(const kv_pool_desc* desc, kv_pool** out);

/* Release the host metadata.  The device pools stay the caller's. */
kv_status kv_pool_destroy(kv_pool* pool);

/* ---- branches ----------------------------------------------------------- */

/* New empty root branch (depth 0, no blocks).  Handles are 0, 1, 2, ... in
 * creation order (roots and forks share the counter) and are never reused. */
kv_status kv_branch_create(kv_pool* pool, int32_t* out_id);

/* Append n_tokens tokens to a live branch ([TRM] §6 append_tokens; [DMW]
 * BlockTable: token t lives in block table[t / 16] at slot t % 16).
 * Allocates ceil((seq_len + n) / 16) - n_blocks new blocks, in logical order,
 * all or nothing; then copies the new rows into their slots on `stream`.
 * k_new, v_new: device, [num_layers][n_tokens][num_kv_heads][head_dim] bf16,
 * 16-byte aligned, read before the stream passes the copy; NULL for a
 * metadata-only pool.  An e4m3 pool quantises the rows on the device under
 * the block rule of kv_pool_desc (the appended rows of one block form one
 * write).  The partial last block being written is always owned
 * by this branch alone (forks copy it), so no other branch sees the write.
 * Errors: NOT_FOUND, OOM (state unchanged), INVALID_ARG, CUDA. */
kv_status kv_append(kv_pool* pool, int32_t id, int32_t n_tokens,
                    const void* k_new, const void* v_new, void* stream);

/* Batched append (tree expansion: one scatter launch for many branches).
 * Equivalent to kv_append(ids[i], n_tokens[i], ...) for i = 0..n-1 in order
 * (same blocks, same order), all or nothing over the whole batch.
 * k_new, v_new: device [num_layers][total][num_kv_heads][head_dim] bf16 with
 * total = sum(n_tokens); branch i's rows are rows sum(n_tokens[0..i)) + 0 ..
 * n_tokens[i]-1.  ids, n_tokens: host.  A branch may appear more than once
 * (an e4m3 pool applies the writes to one block in list order).
 * Errors: NOT_FOUND, OOM (no change), INVALID_ARG, CUDA. */
kv_status kv_append_batch(kv_pool* pool, int32_t n, const int32_t* ids,
                          const int32_t* n_tokens, const void* k_new,
                          const void* v_new, void* stream);

/* Reserve n_tokens[i] new token slots at the end of branch ids[i] (blocks
 * allocated exactly as kv_append_batch would, all or nothing) without
 * writing any data: the caller writes the rows, e.g. the decode step's new
 * token with paged_decode_append_attn.  Until written, the slots hold
 * whatever the blocks held.  Errors: NOT_FOUND, OOM (no change),
 * INVALID_ARG. */
kv_status kv_reserve(kv_pool* pool, int32_t n, const int32_t* ids,
                     const int32_t* n_tokens);

/* Fork a live branch ([TRM] §5 fork rules 1-2, §6 fork_node).  The child
 * shares the parent's full blocks (+1 reference each).  If the parent's last
 * block is partial, the child gets a fresh block holding a copy of that whole
 * block, all layers, K and V (copy-on-write at the divergence point, [DMW]
 * copy-on-write section), copied on `stream`; the parent keeps its own.
 * Child depth = parent depth + 1.  Errors: NOT_FOUND, OOM (no change), CUDA. */
kv_status kv_fork_branch(kv_pool* pool, int32_t parent, int32_t* out_child,
                         void* stream);

/* n forks of one parent in one call (one copy launch), identical in effect to
 * n kv_fork_branch calls.  out_children: host, n entries.  All or nothing. */
kv_status kv_fork_branches(kv_pool* pool, int32_t parent, int32_t n,
                           int32_t* out_children, void* stream);

/* Release one branch handle ([TRM] §5 rule 4, §6 free_node): -1 reference on
 * each block of its table, walked from index 0; a block reaching 0 is pushed
 * on the free stack at once.  Children keep their own references.
 * Errors: NOT_FOUND (unknown or already freed; the page's listing ignores
 * unknown ids silently, this library reports them). */
kv_status kv_free(kv_pool* pool, int32_t id);

/* Release every live branch of id's subtree, post-order, children in
 * creation order (id itself may already be freed).  out_freed_ids: host,
 * nullable, room for every branch ever created; *out_n_freed nullable. */
kv_status kv_free_subtree(kv_pool* pool, int32_t id, int32_t* out_n_freed,
                          int32_t* out_freed_ids);

/* Candidates sorted by ascending omega = score / (depth + 1) ([RKSC] §2.C),
 * computed in binary64, ties by ascending id.  ids, scores: host, n entries;
 * out_sorted: host, n entries.  Errors: NOT_FOUND, INVALID_ARG (NaN score). */
kv_status kv_evict_order(kv_pool* pool, int32_t n, const int32_t* ids,
                         const double* scores, int32_t* out_sorted);

/* Evict whole subtrees in kv_evict_order order until the stop rule holds
 * (checked before each candidate): KV_STOP_FREE_BLOCKS -- at least `target`
 * free blocks; KV_STOP_EVICTED_LEAVES -- at least `target` freed branches that
 * never had children.  A candidate whose subtree holds no live branch is
 * skipped.  out_evicted_ids: host, n entries, nullable. */
kv_status kv_evict(kv_pool* pool, int32_t n, const int32_t* ids,
                   const double* scores, int32_t stop_kind, int64_t target,
                   int32_t* out_n_evicted, int32_t* out_evicted_ids);

/* ---- host tier: spill and restore ([DMW] cross-tier memory offloading) ---- */

/* Attach a host tier: caller-owned pinned host pools host_k / host_v (and,
 * for an e4m3 pool, host_scales) with the device pools' layouts and
 * host_slots blocks each ([num_layers][host_slots][Hkv][...]), reachable
 * from the device (pinned memory under unified addressing), or all NULL for
 * a metadata-only pool.  host_scales must be NULL for a bf16 pool.  Free
 * slots form a LIFO stack, slot 0 handed out first.  Errors: INVALID_ARG
 * (sizes, a second tier, pointers not matching the pool's kind). */
kv_status kv_offload_attach(kv_pool* pool, void* host_k, void* host_v,
                            void* host_scales, int64_t host_slots);

/* Move the blocks that branches ids[0..n) own alone (reference count 1) to
 * host slots (taken in branch order, table order), copying every layer of K
 * and V on `stream`, and free them on the device (pushed on the free stack
 * in the same order); shared blocks stay on the device.  A spilled table
 * entry reads -(slot + 2) in kv_get_block_table.  A branch holding spilled
 * blocks cannot be appended to, forked, batched or indexed until
 * kv_restore; kv_free releases its host slots.  Later device work that
 * reuses the freed blocks must be ordered after `stream`.  *out_n_blocks
 * (nullable) = blocks moved.  All or nothing.  Errors: NOT_FOUND,
 * INVALID_ARG (no tier), OOM (host slots), CUDA. */
kv_status kv_spill(kv_pool* pool, int32_t n, const int32_t* ids, void* stream,
                   int32_t* out_n_blocks);

/* Bring every spilled block of branches ids[0..n) (each listed once) back
 * into device blocks popped from the free stack (branch order, table order),
 * copying on `stream`, and return their host slots to the host free stack.
 * All or nothing.  Errors: NOT_FOUND, INVALID_ARG, OOM (device blocks),
 * CUDA. */
kv_status kv_restore(kv_pool* pool, int32_t n, const int32_t* ids,
                     void* stream, int32_t* out_n_blocks);

/* Free host slots, next-to-be-handed-out first (host out[cap]). */
kv_status kv_get_host_free(kv_pool* pool, int32_t* out, int64_t cap,
                           int64_t* out_n);

/* ---- radix prefix index (host) ------------------------------------------- */

/* A token-keyed radix index over a pool ([DMW] RadixAttention section: a
 * compressed prefix tree whose nodes hold a token sequence and its KV, a
 * lock_ref pinning a node and all its ancestors while in use, and
 * least-recently-used eviction of leaves whose lock_ref is zero).  The
 * sharing unit is a full 16-token block: a node's key is a whole number of
 * blocks and its value the physical block of each.  The index holds one
 * reference on every block it stores.  Recency is a logical clock that ticks
 * once per kv_radix_match / kv_radix_insert; every node on the matched path
 * takes the current tick.  Node 0 is the root (empty key, never evicted).
 * Node ids are assigned in creation order and never reused; a node split
 * where a match ends inside it keeps its id for the deeper part and the new
 * id names the prefix part.  Host-only; not thread-safe with the pool. */
typedef struct kv_radix kv_radix;

typedef struct kv_radix_node_t {
  int32_t live;
  int32_t parent;      /* -1 for the root */
  int32_t n_blocks;    /* blocks (16 tokens each) of this node's key */
  int32_t lock_ref;
  int32_t n_children;
  int32_t reserved;
  int64_t last_access; /* logical clock of the last match / insert through it */
} kv_radix_node_t;

kv_status kv_radix_create(kv_pool* pool, kv_radix** out);
/* Releases every block reference the index holds, then the index. */
kv_status kv_radix_destroy(kv_radix* radix);

/* Longest cached prefix of tokens[0 .. n_tokens) in whole blocks.  *out_node
 * = deepest matched node (0 if none), *out_matched_tokens = 16 x matched
 * blocks.  A match ending inside a node splits it. */
kv_status kv_radix_match(kv_radix* radix, int32_t n_tokens,
                         const int32_t* tokens, int32_t* out_node,
                         int32_t* out_matched_tokens);

/* Index branch `branch`'s KV under its token sequence tokens[0 .. n_tokens)
 * (the caller's tokens of that branch, oldest first): the full blocks past
 * the longest cached prefix become a new leaf holding the branch's physical
 * blocks (+1 reference each).  *out_node = the node ending at the last full
 * block.  Errors: NOT_FOUND (branch), INVALID_ARG. */
kv_status kv_radix_insert(kv_radix* radix, int32_t branch, int32_t n_tokens,
                          const int32_t* tokens, int32_t* out_node);

/* New pool branch (a root: depth 0) whose table is the blocks on the path
 * from the root to `node` (+1 reference each): a request starting from a
 * cached prefix.  *out_branch = its handle. */
kv_status kv_radix_fork(kv_radix* radix, int32_t node, int32_t* out_branch);

/* lock_ref + 1 / - 1 on `node` and every ancestor (unlock: INVALID_ARG if any
 * would go below 0). */
kv_status kv_radix_lock(kv_radix* radix, int32_t node);
kv_status kv_radix_unlock(kv_radix* radix, int32_t node);

/* Evict leaves with lock_ref 0, least recently used first (ties: smaller
 * id), releasing their blocks, until the pool has at least
 * target_free_blocks free blocks or no leaf is evictable.  A parent left
 * without children becomes a leaf in turn.  out_evicted (nullable) gets the
 * ids in eviction order (room for kv_radix_num_nodes entries). */
kv_status kv_radix_evict(kv_radix* radix, int64_t target_free_blocks,
                         int32_t* out_n_evicted, int32_t* out_evicted);

kv_status kv_radix_node_info(kv_radix* radix, int32_t node,
                             kv_radix_node_t* out);
kv_status kv_radix_node_blocks(kv_radix* radix, int32_t node, int32_t* out,
                               int32_t cap, int32_t* out_n);
kv_status kv_radix_num_nodes(kv_radix* radix, int32_t* out_n);

/* ---- introspection (host) ----------------------------------------------- */

kv_status kv_branch_info(kv_pool* pool, int32_t id, kv_branch_info_t* out);

/* Copy a live branch's block table (physical ids, logical order) to host
 * `out` (cap entries).  *out_n = table length, *out_seq_len = its tokens. */
kv_status kv_get_block_table(kv_pool* pool, int32_t id, int32_t* out,
                             int32_t cap, int32_t* out_n,
                             int32_t* out_seq_len);

/* Reference count of every block: host out[num_blocks]. */
kv_status kv_get_refcounts(kv_pool* pool, int32_t* out);

/* Free stack, next-to-be-handed-out first: host out[cap]; *out_n = size. */
kv_status kv_get_free_stack(kv_pool* pool, int32_t* out, int64_t cap,
                            int64_t* out_n);

/* Branches ever created (live or not). */
kv_status kv_num_branches(kv_pool* pool, int32_t* out_n);

/* KV bytes per cached token: 2 x num_layers x num_heads x head_dim x
 * elem_bytes ([TRM] §2.1 Memory_KV with S = 1; 2,621,440 for 80/64/128/2). */
int64_t kv_bytes_per_token(int32_t num_layers, int32_t num_heads,
                           int32_t head_dim, int32_t elem_bytes);

/* ---- decode batch ----------------------------------------------------------- */

/* Largest table among the given live branches (the max_blocks a batch needs). */
kv_status kv_batch_max_blocks(kv_pool* pool, int32_t nb, const int32_t* ids,
                              int32_t* out_max_blocks);

/* Host arrays for one decode step over live branches ids[0..nb) (host), in
 * the caller's order (row b = ids[b]):
 *   tables:   int32 [nb][max_blocks], physical ids, padded with -1;
 *   seq_lens: int32 [nb];
 *   groups:   int32 [*out_n_groups][4] shared-prefix segments
 *             {branch_begin, branch_count, blk_begin, blk_count}: rows
 *             [branch_begin, +branch_count) hold the same physical block at
 *             every logical index in [blk_begin, +blk_count), all full.
 * Segments are the nested runs of consecutive rows with a common prefix of
 * full blocks; for each row they tile [0, end) with no gap.  Rows that are
 * not consecutive in `ids` share nothing (order the batch depth-first to get
 * every segment).  Errors: NOT_FOUND, INVALID_ARG (max_blocks too small,
 * groups_cap too small). */
kv_status kv_build_batch(kv_pool* pool, int32_t nb, const int32_t* ids,
                         int32_t max_blocks, int32_t* tables,
                         int32_t* seq_lens, int32_t groups_cap,
                         int32_t* out_n_groups, int32_t* groups);

/* ---- decode attention ---------------------------------------------------- */

typedef struct kv_decode_plan_info {
  int64_t plan_ints;       /* int32 entries of the plan */
  int64_t workspace_bytes; /* device workspace paged_decode_attn needs */
  int64_t partial_rows;    /* (o, m, l) partial rows in the workspace */
  int32_t n_row_items;     /* work items of the split-KV (mma.sync) kernel */
  int32_t n_tile_items;    /* work items of the tcgen05 kernels (the first
                              n_tile_wide_items of up to 256 rows, the rest
                              of up to 128) */
  int32_t n_merge_rows;    /* nb (one merge per branch and kv-head) */
  int32_t chunk_blocks;    /* blocks per split-KV item */
  int32_t n_tile_wide_items; /* tcgen05 items of up to 256 rows: segments of
                                more than 128 rows (bf16), two M-tiles per
                                item sharing every K/V load */
  int32_t flags;           /* the KV_PLAN_* flags the plan was made with */
  int32_t n_row_warp_items; /* the last n_row_warp_items of the split-KV
                               items are short (at most 16 blocks): the bf16
                               split-KV kernel runs them four to a CTA, one
                               per warp; the others take a whole CTA */
  int32_t reserved;        /* 0 */
} kv_decode_plan_info;

/* Host half of a decode step: split the step into work items.
 * seq_lens (host, nb), groups (host, n_groups x 4, the segments above) must
 * be the same arrays the device copies given to paged_decode_attn hold.
 * Validates: 1 <= seq_lens[b] <= max_blocks * 16; each segment's rows and
 * blocks in range and full; each row's segments tiling [0, end).  Writes
 * the plan to host `plan` (plan_cap int32 entries; pass plan = NULL to query
 * the size in info->plan_ints).  num_sms = the device's SM count (used to
 * size splits).  flags: KV_PLAN_*.  Errors: INVALID_ARG. */
kv_status paged_decode_plan(int32_t nb, int32_t Hq, int32_t Hkv,
                            int32_t head_dim, int32_t block_size,
                            int32_t max_blocks, const int32_t* seq_lens,
                            const int32_t* groups, int32_t n_groups,
                            int32_t num_sms, int32_t flags, int32_t* plan,
                            int64_t plan_cap, kv_decode_plan_info* info);

/* Device workspace bytes for a step (same number as info->workspace_bytes). */
kv_status paged_decode_attn_workspace_size(const kv_decode_plan_info* info,
                                           size_t* out_bytes);

/* Decode attention for one layer ([TRM] §2.1: softmax(q K^T * scale) V for
 * the one new query of each branch against all its cached tokens):
 *   out[b][h] = sum_t softmax_t(scale * q[b][h] . K_t) V_t,
 *   t over the seq_lens[b] tokens of branch b, token t read from block
 *   block_tables[b][t / 16] slot t % 16 of kv-head h / (Hq / Hkv).
 * Device inputs: q [nb][Hq][head_dim] bf16; k_pool, v_pool = this layer's
 * [num_blocks][Hkv][16][head_dim] bf16 pools; block_tables [nb][max_blocks]
 * int32; seq_lens [nb] int32; prefix_groups [n_groups][4] int32 (may be NULL
 * when n_groups == 0); plan = a device copy of paged_decode_plan's output for
 * these seq_lens/groups, with *info its host info.  Output: out
 * [nb][Hq][head_dim] bf16.  workspace: device, >= info->workspace_bytes,
 * 256-byte aligned, no initial contents needed.  Shared-prefix blocks are read
 * once per tile item (tensor cores for segments of >= 65 rows: one item per
 * 256 rows for segments of 129-256 rows, one per 128 rows otherwise).  When a
 * step has both tensor-core tiles and split-KV items (or both sizes of
 * tile items), the tile pass runs on one or two library-owned streams
 * (highest priority) forked from and joined back into `stream` (event
 * record / wait), so that the passes overlap; all work is still ordered
 * after earlier work on `stream` and before later work on it.
 * Error behaviour: argument errors return INVALID_ARG before any launch; a
 * block id outside [0, num_blocks) or a timed-out wait is recorded in the
 * workspace status word (the access is skipped, the output is then
 * unspecified) and reported by kv_check_device_status.  scale must be finite
 * and > 0.  Errors: INVALID_ARG, CUDA. */
kv_status paged_decode_attn(const void* q, const void* k_pool,
                            const void* v_pool, int64_t num_blocks,
                            const int32_t* block_tables,
                            const int32_t* seq_lens,
                            const int32_t* prefix_groups, int32_t n_groups,
                            int32_t nb, int32_t max_blocks, int32_t Hq,
                            int32_t Hkv, int32_t head_dim, int32_t block_size,
                            float scale, void* out, const int32_t* plan,
                            const kv_decode_plan_info* info, void* workspace,
                            size_t ws_bytes, void* stream);

/* The decode step fused with the append of each branch's newest token
 * ([TRM] §2.1: step t+1 caches the new key and value, then attends to all
 * of them).  Same arguments and result as paged_decode_attn, plus
 * k_step, v_step: device [nb][Hkv][head_dim] bf16, this layer's K and V of
 * token seq_lens[b] - 1 of each branch b (its slot reserved beforehand with
 * kv_reserve and included in block_tables / seq_lens).  In the same launch
 * the kernel writes those rows into their slots of k_pool / v_pool and
 * attends to them (it does not read the slot back from the pool).  The
 * newest token's block is owned by its branch alone (a partial last block is
 * copied at fork), so it is never inside a shared-prefix segment.
 * Errors: as paged_decode_attn. */
kv_status paged_decode_append_attn(
    const void* q, const void* k_step, const void* v_step, const void* k_pool,
    const void* v_pool, int64_t num_blocks, const int32_t* block_tables,
    const int32_t* seq_lens, const int32_t* prefix_groups, int32_t n_groups,
    int32_t nb, int32_t max_blocks, int32_t Hq, int32_t Hkv, int32_t head_dim,
    int32_t block_size, float scale, void* out, const int32_t* plan,
    const kv_decode_plan_info* info, void* workspace, size_t ws_bytes,
    void* stream);

/* Decode attention over an e4m3 pool (kv_pool_desc.kv_dtype =
 * KV_DTYPE_E4M3): the same result as paged_decode_attn computed from the
 * stored values (code value x the tile's scale), with q and out bf16 as
 * there.  k_pool, v_pool, kv_scales: this layer's base pointers of the
 * e4m3 pool (layouts under kv_pool_desc).  The plan must be made with
 * KV_PLAN_KV_E4M3 (and a bf16 step's plan without it).  Arithmetic: the
 * codes are widened to f16 exactly, q is carried in f16 after a per-row
 * power-of-two scaling (so nothing overflows), products accumulate in fp32.
 * Errors and status reporting: as paged_decode_attn. */
kv_status paged_decode_attn_e4m3(
    const void* q, const void* k_pool, const void* v_pool,
    const void* kv_scales, int64_t num_blocks, const int32_t* block_tables,
    const int32_t* seq_lens, const int32_t* prefix_groups, int32_t n_groups,
    int32_t nb, int32_t max_blocks, int32_t Hq, int32_t Hkv, int32_t head_dim,
    int32_t block_size, float scale, void* out, const int32_t* plan,
    const kv_decode_plan_info* info, void* workspace, size_t ws_bytes,
    void* stream);

/* paged_decode_append_attn for an e4m3 pool: first quantises each branch's
 * newest token (k_step, v_step bf16 [nb][Hkv][head_dim]) into its reserved
 * slot under the block rule above (one launch, writes to distinct blocks),
 * then runs paged_decode_attn_e4m3 over the pool, on `stream`.  Errors: as
 * paged_decode_attn. */
kv_status paged_decode_append_attn_e4m3(
    const void* q, const void* k_step, const void* v_step, const void* k_pool,
    const void* v_pool, void* kv_scales, int64_t num_blocks,
    const int32_t* block_tables, const int32_t* seq_lens,
    const int32_t* prefix_groups, int32_t n_groups, int32_t nb,
    int32_t max_blocks, int32_t Hq, int32_t Hkv, int32_t head_dim,
    int32_t block_size, float scale, void* out, const int32_t* plan,
    const kv_decode_plan_info* info, void* workspace, size_t ws_bytes,
    void* stream);

/* paged_decode_attn without a caller workspace.  The pages have no
 * counterpart: this exists for callers that cannot allocate device memory
 * (a plug-in whose host engine owns every device buffer and offers it no
 * allocator, a process that reserved the whole GPU at start-up, a
 * latency-critical path that cannot pay for cudaMalloc or its implicit
 * synchronisation).  Same arguments, meaning and errors as paged_decode_attn
 * minus workspace / ws_bytes: the step's scratch (status word and partial
 * results) lives in a library-owned __device__ array of 64 MiB that every GPU
 * loading the library holds until the process exits.  A step whose
 * info->workspace_bytes exceeds 64 MiB is rejected with INVALID_ARG.  The
 * first call on a device looks up the array's device address (with that
 * device current) and should come before any stream capture.  All calls share
 * the array and it keeps the last call's contents; each call clears the part
 * that must start at zero; calls whose work overlaps on the GPU race.  A bad
 * block id or a timed-out wait is recorded in the status word at the start of
 * the array; kv_check_noalloc_status reads it.  Calls no cudaMalloc, cudaFree
 * or other allocating routine. */
kv_status paged_decode_attn_noalloc(
    const void* q, const void* k_pool, const void* v_pool, int64_t num_blocks,
    const int32_t* block_tables, const int32_t* seq_lens,
    const int32_t* prefix_groups, int32_t n_groups, int32_t nb,
    int32_t max_blocks, int32_t Hq, int32_t Hkv, int32_t head_dim,
    int32_t block_size, float scale, void* out, const int32_t* plan,
    const kv_decode_plan_info* info, void* stream);

/* The status word of paged_decode_attn_noalloc's built-in scratch on the
 * current device, read (synchronising `stream`) and cleared, as
 * kv_check_device_status does for a caller workspace: *out_code 0,
 * KV_ERR_DEVICE or KV_ERR_TIMEOUT; *out_detail (nullable) the first bad value
 * recorded.  Like the entry point it serves, it has no counterpart in the
 * pages and allocates nothing.  Each paged_decode_attn_noalloc call clears
 * the word when it starts, so read it after the call whose errors are
 * wanted and before the next one.  Errors: INVALID_ARG, CUDA. */
kv_status kv_check_noalloc_status(void* stream, int32_t* out_code,
                                  int32_t* out_detail);

/* Read (synchronising `stream`) and clear the status word of a workspace used
 * by paged_decode_attn.  *out_code: 0, KV_ERR_DEVICE or KV_ERR_TIMEOUT;
 * *out_detail (nullable): the first bad value recorded.  Errors: CUDA. */
kv_status kv_check_device_status(void* workspace, void* stream,
                                 int32_t* out_code, int32_t* out_detail);

/* Diagnostic: launch one thread that waits, bounded by wait_cycles SM clock
 * cycles, on an mbarrier that nothing completes, then records KV_ERR_TIMEOUT
 * (detail 99) in the status word of `workspace` exactly as the attention
 * kernels do when one of their bounded waits runs out (their bound is 2^31
 * cycles, about a second); kv_check_device_status then reports it.  It lets
 * the timeout path be exercised without a fault or a hang.  workspace:
 * device, 256-byte aligned, >= 256 bytes.  wait_cycles in [1, 2^31].
 * Errors: INVALID_ARG, CUDA. */
kv_status kv_selftest_timeout(void* workspace, int64_t wait_cycles,
                              void* stream);

/* Optional per-kernel timing (measurement support, not part of the method).
 * While set, each paged_decode_attn call on this thread records, on its
 * stream, events[2*i] just before and events[2*i+1] just after its kernel i:
 * i = 0 the tcgen05 tile kernel, 1 the split-KV kernel, 2 the merge kernel;
 * a kernel that is not launched records nothing.  events: caller-created
 * cudaEvent_t handles (as void*), n_events entries (6 covers all three); the
 * array must stay valid while set.  Pass NULL / 0 to clear.  Errors: none. */
kv_status kv_set_launch_events(void* const* events, int32_t n_events);

/* Thread-local description of the last error on this thread ("" if none). */
const char* kv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
