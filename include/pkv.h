/*
 * pkv.h -- C ABI of the GB300 paged KV-cache decode-attention library (libpkv.so).
 *
 * Plain C: host integers and pointers only.  "device pointer" means memory the caller
 * allocated on the CUDA device the pool is attached to; "host pointer" means ordinary
 * process memory.  Every function returns a pkv_status (0 = PKV_OK) unless noted.
 * Kernels run asynchronously on the caller's stream (a cudaStream_t passed as void*,
 * NULL = the legacy default stream); argument errors are reported before anything is
 * launched, and violations found on the device (a block id or slot outside the pool, a
 * sequence length outside its table, a pipeline wait that gave up) set bits in the pool's
 * device error word, read with pkv_get_device_error().
 *
 * Sources (page title, section), cited per entry point below:
 *   [Slot]    "理解 KV Cache：Attention、P/D 分离与 vLLM 的页式显存管理" (steinslab.io),
 *             §3.3 slot addressing and the §3.4 example.
 *   [Layout]  same page, §3.2: a block holds block_size tokens of K and V per KV head,
 *             head-first ([num_kv_heads, block_size, head_dim]).
 *   [Life]    same page, §3.5: blocks are allocated from a free pool, used, and returned.
 *   [Decode]  same page, §1.2-§1.3 and §2.2: the new token's query attends over every
 *             cached position of its sequence (causal mask), computed as two fused GEMVs.
 *   [Attn]    "传统 Attention 的 KV Cache 问题" (pyllm.pages.dev), §1.1: scaled softmax
 *             attention sum_j softmax_j(q.K_j / sqrt(d_k)) V_j.
 *   [Paged]   "KV Cache 与推理优化" (note.yj-dis.top), section "PagedAttention：把 KV Cache
 *             当虚拟内存管": 16-token blocks, one block table per request mapping logical to
 *             physical blocks, shared prefix blocks, the kernel gathering K/V via the table.
 *   [GQA]     same page, section on MHA/GQA/MQA: query heads share KV heads in contiguous
 *             groups of g = Hq / Hkv.
 *   [Quant]   same page, section "KV 量化": K/V stored in FP8 (1 byte) with higher-precision
 *             arithmetic.
 *   [APC]     same page, section "APC：连计算都省了": a hash per full block; a request whose
 *             prefix matches a cached one reuses those physical blocks; the lookup stops at
 *             the first miss.  "一个请求为什么越生成越占内存?" (learning-field-guides), paging
 *             section: reuse must match the tokens, their positions and the model.
 *   [Bytes]   same page, section "KV Cache 有多大：一张显存账单": every layer keeps K and V
 *             for every token, 2 * layers * kv_heads * head_dim * element-bytes per token;
 *             "一个请求为什么越生成越占内存?" (learning-field-guides), capacity derivation:
 *             the same count summed over layers, positions and sequences.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID = 1,   /* bad argument; nothing was launched */
    PKV_ERR_OOM = 2,       /* the pool has fewer free blocks than requested */
    PKV_ERR_DEVICE = 3,    /* the device error word is non-zero (see PKV_DEVERR_*) */
    PKV_ERR_TIMEOUT = 4,   /* a kernel's bounded pipeline wait gave up */
    PKV_ERR_CUDA = 5       /* a CUDA runtime call failed (launch, copy, allocation) */
} pkv_status;

/* Bits of the device error word. */
#define PKV_DEVERR_SLOT     0x1u   /* kv_append: slot >= num_blocks * block_size (row skipped) */
#define PKV_DEVERR_BLOCK_ID 0x2u   /* decode: a needed table entry outside [0, num_blocks) */
#define PKV_DEVERR_SEQ_LEN  0x4u   /* decode: seq_len outside [1, max_blocks * block_size] */
#define PKV_DEVERR_TIMEOUT  0x8u   /* a pipeline wait exceeded its bound (about 1 s) */
#define PKV_DEVERR_PLAN     0x10u  /* prefill: the plan does not match the call (nothing ran) */

typedef enum { PKV_KV_BF16 = 0, PKV_KV_FP8E4M3 = 1 } pkv_kv_dtype;

/* Shape and element type of a paged K/V pool [Layout]: two caller-owned device tensors
 * key_cache and value_cache, each [num_layers, num_blocks, num_kv_heads, block_size,
 * head_dim], contiguous, 16-byte aligned.  block_size must be 16 [Paged]; head_dim 64 or
 * 128.  A block id names the same block_size positions in every layer, so one block table
 * per sequence serves all layers, and a token costs 2 * num_layers * num_kv_heads *
 * head_dim * element-bytes of cache [Bytes].  The single-layer entry points take the base
 * of one layer (cache + layer * pkv_pool_layer_bytes()); the *_layers entry points take the
 * base of layer 0 and cover all layers in one launch.  num_layers 0 means 1; at most 4096,
 * with num_layers * num_blocks * num_kv_heads < 2^31.  FP8 pools store OCP E4M3 codes of
 * x / scale with one scale per tensor [Quant]; k_scale and v_scale must be positive and
 * finite (ignored for bf16). */
typedef struct {
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t kv_dtype;      /* pkv_kv_dtype */
    float k_scale;
    float v_scale;
    int32_t num_layers;    /* layers stacked in each cache tensor (0 = 1) */
} pkv_pool_desc;

typedef struct pkv_pool pkv_pool;   /* host allocator state + the device error word */

/* Create a pool descriptor and its host block allocator [Life].  free_order (host,
 * optional) is a permutation of 0..num_blocks-1 giving the order in which free blocks are
 * handed out; NULL means ascending ids.  Touches no GPU.  *out receives the pool, owned by
 * the caller until pkv_pool_destroy.  INVALID on a bad descriptor or permutation. */
int pkv_pool_create(const pkv_pool_desc *desc, const int32_t *free_order, pkv_pool **out);

/* Free the pool, its allocator and (if attached) its device error word. */
int pkv_pool_destroy(pkv_pool *pool);

/* Copy the pool's descriptor to *out (num_layers >= 1). */
int pkv_pool_get_desc(const pkv_pool *pool, pkv_pool_desc *out);

/* Bytes of one layer of one cache tensor: num_blocks * num_kv_heads * block_size *
 * head_dim * element-bytes [Layout][Bytes].  Each of key_cache and value_cache holds
 * num_layers times this.  0 for a NULL pool. */
size_t pkv_pool_layer_bytes(const pkv_pool *pool);

/* Number of blocks currently free. */
int pkv_pool_num_free(const pkv_pool *pool, int32_t *out);

/* Reference count of one block (0 = free). */
int pkv_pool_refcount(const pkv_pool *pool, int32_t block_id, int32_t *out);

/* Take n blocks from the front of the free list [Life]; ids_out (host, n entries)
 * receives them, each with reference count 1.  OOM (nothing taken) if fewer than n free. */
int pkv_pool_alloc(pkv_pool *pool, int32_t n, int32_t *ids_out);

/* Add one reference to each listed block, which must be allocated: a shared prefix block
 * referenced by several block tables [Paged].  INVALID (nothing changed) otherwise. */
int pkv_pool_share(pkv_pool *pool, const int32_t *ids, int32_t n);

/* Drop one reference from each listed block; blocks reaching zero return to the back of
 * the free list [Life].  INVALID (nothing changed) on a free or out-of-range id. */
int pkv_pool_free(pkv_pool *pool, const int32_t *ids, int32_t n);

/* Build block tables for a batch [Paged][Life]: row b (tables_out is host int32
 * [batch, max_blocks], row-major) gets ceil(seq_lens[b] / block_size) entries -- first the
 * shared prefix ids (prefix_ids, host, num_prefix entries, already allocated; one more
 * reference each, as many as the row needs), then fresh blocks from the free list in
 * order -- and -1 in unused entries.  seq_lens counts the token appended this step.
 * INVALID if a length is < 1 or needs more than max_blocks entries; OOM if the pool runs
 * dry (then every block taken by this call is returned and tables_out is unspecified). */
int pkv_build_block_tables(pkv_pool *pool, const int32_t *seq_lens, int32_t batch,
                           int32_t max_blocks, const int32_t *prefix_ids, int32_t num_prefix,
                           int32_t *tables_out);

/* Copy-on-write before an append [Paged][Life]: sequence b (in batch order) is about to
 * write position L_b - 1 = seq_lens[b] - 1, in logical block (L_b - 1) / block_size.  If the
 * block that entry names is held by more than one reference, the sequence diverges from the
 * other holders: a fresh block is taken from the front of the free list, the shared block
 * loses one reference, the table entry (host int32 tables [batch, max_blocks], updated in
 * place) is pointed at the fresh block, and the pair is recorded -- src_out[i] = shared,
 * dst_out[i] = fresh (host int32, room for batch entries each), *num_copies = the count.
 * The last holder of a shared block writes it in place.  The content is not copied here:
 * run pkv_copy_blocks on the pairs before the append.  INVALID (nothing changed) on a
 * length outside [1, max_blocks * block_size] or an entry that is not an allocated block;
 * OOM (nothing changed, tables restored) if the free list runs dry. */
int pkv_cow_prepare(pkv_pool *pool, int32_t *tables, const int32_t *seq_lens, int32_t batch,
                    int32_t max_blocks, int32_t *src_out, int32_t *dst_out, int32_t *num_copies);

/* Copy whole blocks [Paged][Layout]: for each pair i and every layer of the pool, the K and
 * V content of block src[i] is copied to block dst[i] (device int32 arrays, num_pairs
 * entries; caches the whole stacked tensors).  The dst ids must be distinct and none may be
 * a src of this call.  An id outside [0, num_blocks) sets PKV_DEVERR_BLOCK_ID and that pair
 * is skipped. */
int pkv_copy_blocks(pkv_pool *pool, void *key_cache, void *value_cache, const int32_t *src,
                    const int32_t *dst, int32_t num_pairs, void *stream);

/* Slot of each sequence's newest token, at position seq_lens[b]-1 [Slot]:
 * slot = tables[b][(L-1) / block_size] * block_size + (L-1) % block_size.  Host arrays:
 * tables int32 [batch, max_blocks], seq_lens int32 [batch], slots_out int64 [batch].
 * INVALID on a length outside [1, max_blocks*block_size] or a negative table entry. */
int pkv_slot_mapping(const int32_t *tables, const int32_t *seq_lens, int32_t batch,
                     int32_t max_blocks, int32_t block_size, int64_t *slots_out);

/* Slots of every position 0 .. seq_lens[b]-1 of every sequence [Slot], sequence-major
 * (slots_out has sum(seq_lens) int64 entries): the slot mapping of a whole-prompt append.
 * Host arrays as in pkv_slot_mapping; same errors. */
int pkv_slot_mapping_all(const int32_t *tables, const int32_t *seq_lens, int32_t batch,
                         int32_t max_blocks, int32_t block_size, int64_t *slots_out);

/* Automatic prefix caching [APC] (host only).  A full block of block_size tokens is
 * identified by a chained hash: block i hashes, with 64-bit FNV-1a, the 8 little-endian
 * bytes of block i-1's hash (of `salt` for block 0) followed by its tokens as 4
 * little-endian bytes each.  Equal hashes thus stand for an equal salt (a model / adapter
 * identity: another model must never reuse the blocks) and equal tokens at every position
 * up to the end of the block.  A partial last block has no hash and is never shared.
 *
 * pkv_block_hashes: hashes_out (host, num_tokens / block_size entries) receives the hash of
 * every full block of tokens (host int32 token ids).  Needs no pool. */
int pkv_block_hashes(const int32_t *tokens, int32_t num_tokens, int32_t block_size, uint64_t salt,
                     uint64_t *hashes_out);

/* The physical blocks holding the longest cached prefix of a request [APC]: block i hits an
 * entry with its hash whose parent is the block hit for i-1 and whose stored salt and
 * tokens are the request's (so a hash collision never returns another prefix's block); the
 * walk stops at the first miss.  block_ids_out (host, room for num_tokens / block_size)
 * receives the hits in order, *num_hits their count.  Takes no references: pass the ids
 * as prefix_ids to pkv_build_block_tables, which does.  Marks the hits as recently used. */
int pkv_prefix_lookup(pkv_pool *pool, const int32_t *tokens, int32_t num_tokens, uint64_t salt,
                      int32_t *block_ids_out, int32_t *num_hits);

/* Cache every full block of a request whose block table row is table_row (host, row_len >=
 * num_tokens / block_size entries) [APC].  A block whose chain is cached already is only
 * marked as used; every other one is entered under its hash and gets one more reference,
 * held by the cache until it is evicted, so it outlives the request.  *num_added receives
 * the number of blocks entered.  INVALID (nothing changed) if a row block that would be
 * entered is not allocated, is cached under another chain, or appears twice. */
int pkv_prefix_insert(pkv_pool *pool, const int32_t *tokens, int32_t num_tokens, uint64_t salt,
                      const int32_t *table_row, int32_t row_len, int32_t *num_added);

/* Evict up to max_blocks cached blocks [APC][Life]: repeatedly the least recently used entry
 * that has no cached child and whose block only the cache holds (reference count 1) loses
 * its entry and the cache's reference, which returns the block to the back of the free
 * list.  evicted_out (host, room for max_blocks) receives their ids in order. */
int pkv_prefix_evict(pkv_pool *pool, int32_t max_blocks, int32_t *evicted_out, int32_t *num_evicted);

/* Drop every cache entry (least recently used leaves first), releasing the cache's
 * references; blocks still held by tables stay allocated. */
int pkv_prefix_clear(pkv_pool *pool);

/* Number of cached blocks. */
int pkv_prefix_cached_blocks(const pkv_pool *pool, int32_t *out);

/* Slots of each prompt chunk's positions [Slot]: sequence b's chunk is rows cu_q[b] ..
 * cu_q[b+1]-1 (host int32 [batch+1], cu_q[0] = 0), positions L_b - P_b .. L_b - 1 with
 * P_b = cu_q[b+1] - cu_q[b] and L_b = seq_lens[b] (the length including the chunk);
 * slots_out (host int64, cu_q[batch] entries) receives their slots in row order -- the
 * slot mapping of a prefill's kv_append.  INVALID as pkv_slot_mapping, or if P_b < 0 or
 * P_b > L_b. */
int pkv_slot_mapping_chunks(const int32_t *tables, const int32_t *seq_lens, const int32_t *cu_q,
                            int32_t batch, int32_t max_blocks, int32_t block_size, int64_t *slots_out);

/* Bind the pool to a CUDA device: allocates its 4-byte device error word (cudaMalloc) on
 * that device.  Required once before pkv_kv_append / pkv_paged_attention_decode. */
int pkv_pool_attach_device(pkv_pool *pool, int device);

/* Append K/V rows into their slots [Slot][Decode]: for each token t and KV head h with
 * slot = slot_mapping[t] >= 0, key_cache[slot/16][h][slot%16][:] = k[t][h][:] (bf16 bit
 * copy; FP8 pools store E4M3(fl32(k * fl32(1/k_scale))), round-to-nearest-even, saturated
 * to +-448), likewise V.  Device pointers: k, v bf16 [num_tokens, Hkv, D]; slot_mapping
 * int64 [num_tokens] (negative = padding, skipped); caches as in pkv_pool_desc.  A slot
 * beyond the pool sets PKV_DEVERR_SLOT and its row is skipped.  Slots must be distinct. */
int pkv_kv_append(pkv_pool *pool, const void *k, const void *v, const int64_t *slot_mapping,
                  int32_t num_tokens, void *key_cache, void *value_cache, void *stream);

/* pkv_kv_append for every layer of the pool in one launch [Slot][Bytes]: k, v are device
 * bf16 [num_layers, num_tokens, Hkv, D]; token t of layer l goes to slot slot_mapping[t] of
 * layer l (the same slot in every layer, since blocks span all layers).  key_cache and
 * value_cache are the whole stacked tensors.  Otherwise as pkv_kv_append. */
int pkv_kv_append_layers(pkv_pool *pool, const void *k, const void *v,
                         const int64_t *slot_mapping, int32_t num_tokens, void *key_cache,
                         void *value_cache, void *stream);

/* Tuning knobs for pkv_paged_attention_decode_ex; zero fields mean "choose". */
typedef struct {
    int32_t grid_ctas;        /* CTAs of the persistent grid (0 = SM count x CTAs per SM) */
    int32_t variant;          /* 0 = auto (3); 1 = CUDA-core dot products; 2 = tensor-core mma with
                                 the heads as rows; 3 = tensor-core mma with the tokens as rows */
    int32_t warps_per_cta;    /* 0 = auto (4); 4 or 8 */
    int32_t stages;           /* 0 = auto (16 KiB of tiles per warp: 2 bf16 / 4 FP8 at D 128); 2..4 */
    int32_t heads_per_copy;   /* variant 3: KV heads loaded by one copy (the block's tiles of
                                 consecutive heads are contiguous, so one copy brings several),
                                 which halves or quarters the units and their merges; must divide
                                 num_kv_heads and not exceed warps_per_cta; 0 = auto (1); 1, 2, 4 */
    int32_t shared_prefix_blocks;  /* variant 3 with heads_per_copy 1: blocks at the start of the
                                 tables that a shared-prefix pass may cover (0 = no pass).  Blocks
                                 that many sequences' tables share are stored once [Paged]; the
                                 pass reads each such block once per KV head for up to 64 query
                                 rows instead of once per sequence.  The reference is the longest
                                 sequence's table (the smallest index among equals); sequence b's
                                 covered blocks are its leading table entries -- at most this many,
                                 never the block that receives an appended token -- that equal the
                                 reference's.  The result is the same attention for any tables
                                 (only the order of the fp32 sums changes); the pass is one more
                                 launch on the stream before the decode, and the workspace grows
                                 by a partial state per query row. */
    int32_t unit_cost;        /* the persistent grid's split of the (block, KV head) tasks charges
                                 every unit (sequence, KV head group) this many tasks besides its
                                 blocks -- the fixed cost of a unit in a CTA -- so that a CTA
                                 given many short units gets fewer blocks; 0 = auto (16); -1 = none
                                 (an even split of the blocks); at most 4096 */
} pkv_decode_opts;

/* Device workspace bytes the decode needs for this shape and these opts (0 if the shape or
 * opts are invalid), for any of the decode entry points on this pool: the counters cover
 * all of the pool's layers.  Queries the current device. */
size_t pkv_decode_workspace_bytes(const pkv_pool *pool, int32_t batch, int32_t num_q_heads,
                                  int32_t max_blocks, const pkv_decode_opts *opts);

/* Paged decode attention, one query token per sequence [Decode][Attn][GQA][Paged]:
 *   out[b][hq][:] = sum_{j < L_b} softmax_j(scale * q[b][hq] . K_j) V_j,
 *   K_j, V_j = cache[block_tables[b][j / 16]][hq / (Hq/Hkv)][j % 16][:],  L_b = seq_lens[b].
 * Device pointers: q bf16 [batch, num_q_heads, D]; caches as in pkv_pool_desc;
 * block_tables int32 [batch, max_blocks]; seq_lens int32 [batch]; out bf16
 * [batch, num_q_heads, D] (fp32 accumulation, rounded to nearest even); workspace of at
 * least pkv_decode_workspace_bytes() bytes, 256-byte aligned, ZERO-FILLED before its first
 * use: it holds per-(sequence, KV head) counters that every call leaves at zero again
 * (re-zero it after a call that reported a device error), plus partial softmax states.
 * Calls sharing a workspace must not overlap on the GPU.
 * Positions j >= L_b are never used, whatever they hold.  The work -- every sequence's
 * blocks for every KV head -- is split evenly over a one-wave persistent grid; a
 * (sequence, head) cut by that split is finished by whichever of its CTAs ends last.  All
 * split points and merge orders depend only on seq_lens, the grid and logical positions,
 * so any physical placement of the blocks gives bit-identical output.  Requires
 * 1 <= batch <= 4096, num_q_heads a multiple of Hkv with group <= 16, an attached pool,
 * max_blocks >= 1, batch * max_blocks * Hkv < 2^31.  FP8 pools compute q.K with q rounded
 * to fp16 (|q| must stay below 65504).  An invalid seq_len sets PKV_DEVERR_SEQ_LEN and
 * zeroes that sequence's output. */
int pkv_paged_attention_decode(pkv_pool *pool, const void *q, const void *key_cache,
                               const void *value_cache, const int32_t *block_tables,
                               const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                               int32_t max_blocks, float scale, void *out, void *workspace,
                               size_t workspace_bytes, void *stream);

/* Same, with explicit tuning knobs (opts may be NULL). */
int pkv_paged_attention_decode_ex(pkv_pool *pool, const void *q, const void *key_cache,
                                  const void *value_cache, const int32_t *block_tables,
                                  const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                  int32_t max_blocks, float scale, void *out, void *workspace,
                                  size_t workspace_bytes, const pkv_decode_opts *opts,
                                  void *stream);

/* One whole decode step in one launch [Decode][Slot][Attn]: the new token of every sequence,
 * at position L_b - 1, has its K and V rows (k_new, v_new: device bf16 [batch, Hkv, D])
 * written into slot table[b][(L_b-1)/16]*16 + (L_b-1)%16 of the caches -- exactly what
 * pkv_slot_mapping + pkv_kv_append store (FP8 pools encode them the same way) -- and then
 * every sequence attends over positions 0 .. L_b-1 as in pkv_paged_attention_decode.  Each
 * row is written by the CTA that streams that block, just before it loads the block, so
 * no other launch and no slot mapping is needed.  The block holding the new token must not
 * be shared with another sequence (copy it first).  Other arguments, workspace rules and
 * errors as pkv_paged_attention_decode_ex. */
int pkv_decode_step(pkv_pool *pool, const void *q, const void *k_new, const void *v_new,
                    void *key_cache, void *value_cache, const int32_t *block_tables,
                    const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_blocks,
                    float scale, void *out, void *workspace, size_t workspace_bytes,
                    const pkv_decode_opts *opts, void *stream);

/* Decode every layer of the pool in one launch [Decode][Bytes]: the same computation as
 * pkv_decode_step (k_new and v_new given) or pkv_paged_attention_decode_ex (both NULL),
 * applied independently to each layer l of the stacked caches with layer l's queries and
 * new rows.  Device pointers: q, out bf16 [num_layers, batch, num_q_heads, D]; k_new,
 * v_new bf16 [num_layers, batch, Hkv, D] or both NULL; key_cache, value_cache the whole
 * stacked tensors; one block_tables / seq_lens for all layers.  Every (layer, sequence,
 * KV head) is a unit of the same persistent schedule, so one launch streams all layers.
 * Workspace, opts and errors as pkv_decode_step. */
int pkv_decode_step_layers(pkv_pool *pool, const void *q, const void *k_new, const void *v_new,
                           void *key_cache, void *value_cache, const int32_t *block_tables,
                           const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                           int32_t max_blocks, float scale, void *out, void *workspace,
                           size_t workspace_bytes, const pkv_decode_opts *opts, void *stream);

/* ---- Prefill and chunked prefill [Decode][Attn][GQA][Paged] ----
 * A batch packs, per sequence b, a chunk of P_b = cu_q[b+1] - cu_q[b] query rows (rows
 * cu_q[b] .. cu_q[b+1]-1 of q) whose K/V are already in the cache (pkv_kv_append with
 * pkv_slot_mapping_chunks), behind C_b = seq_lens[b] - P_b earlier positions.  Row
 * cu_q[b] + i is position C_b + i and attends causally over positions 0 .. C_b + i of its
 * own sequence:  out[row][hq] = sum_{j <= C_b + i} softmax_j(scale * q[row][hq] . K_j) V_j,
 * K_j, V_j gathered through block_tables[b] from KV head hq / (Hq / Hkv).  C_b = 0 is the
 * prefill of a whole prompt; C_b > 0 a later chunk of a long prompt.
 *
 * The work is planned on the host once per batch (every layer of a model can reuse the
 * plan) and run on the device per layer.  pkv_prefill_plan_bytes: an upper bound of the
 * plan's size for batch sequences and total_q packed rows (0 if the shape is invalid).
 * pkv_prefill_plan: cu_q (host int32 [batch+1], cu_q[0] = 0) and seq_lens (host int32
 * [batch], each >= its P_b, >= 1, needing at most max_blocks table entries) give the units
 * (sequence, KV head, tile of 256 / g query positions) and their assignment to a one-wave
 * persistent grid, heaviest unit first to the least-loaded CTA; plan_out (host,
 * plan_bytes) receives it and *grid_out the grid.  The caller copies the plan to device
 * memory (32-byte aligned) for pkv_paged_prefill.  Requires Hq a multiple of Hkv with
 * g <= 16.  Queries the current device's SM count. */
size_t pkv_prefill_plan_bytes(const pkv_pool *pool, int32_t batch, int32_t num_q_heads, int32_t total_q);
int pkv_prefill_plan(const pkv_pool *pool, const int32_t *cu_q, const int32_t *seq_lens, int32_t batch,
                     int32_t num_q_heads, int32_t max_blocks, void *plan_out, size_t plan_bytes,
                     int32_t *grid_out);

/* Run a plan: q bf16 [total_q, num_q_heads, D] (device); caches of one layer as in
 * pkv_pool_desc, bf16 or FP8 E4M3 ("KV Cache 与推理优化", KV 量化: the cache stored in FP8,
 * the arithmetic in higher precision: E4M3 tiles are converted to bf16 on the chip, exactly,
 * k_scale multiplies the scores and v_scale the output); block_tables int32
 * [batch, max_blocks] (device); plan the device copy of pkv_prefill_plan's output and grid
 * its grid; out bf16 [total_q, num_q_heads, D] (device, fp32 accumulation, rounded to
 * nearest even).  Rows are computed on the tcgen05 tensor cores: S = Q.K^T and O += P.V in
 * tensor memory, P in bf16.  Positions a row may not see are never used, whatever the
 * cache holds there.  A plan that does not match the call sets PKV_DEVERR_PLAN and
 * computes nothing; a table entry outside the pool sets PKV_DEVERR_BLOCK_ID (that
 * sequence's rows are then unspecified); a wait inside the kernel that runs out (about 1 s)
 * sets PKV_DEVERR_TIMEOUT and the launch ends. */
int pkv_paged_prefill(pkv_pool *pool, const void *q, const void *key_cache, const void *value_cache,
                      const int32_t *block_tables, int32_t batch, int32_t num_q_heads, int32_t max_blocks,
                      int32_t total_q, float scale, const void *plan, int32_t grid, void *out, void *stream);

/* Host side of one decode step, for pkv_decode_step_host: host memory, page-locked (pinned)
 * for the copies to be asynchronous.  block_tables and seq_lens may be NULL when the device
 * copies are already current (tables change only when a sequence gains a block).  With
 * k_new and v_new both NULL the step only decodes (pkv_paged_attention_decode_ex). */
typedef struct {
    const void *q;                  /* bf16 [batch, num_q_heads, D] */
    const void *k_new;              /* bf16 [batch, Hkv, D] */
    const void *v_new;              /* bf16 [batch, Hkv, D] */
    const int32_t *block_tables;    /* int32 [batch, max_blocks], or NULL */
    const int32_t *seq_lens;        /* int32 [batch], or NULL */
    void *out;                      /* bf16 [batch, num_q_heads, D], written */
    int32_t contiguous;             /* nonzero: the inputs lie back to back (see below) */
} pkv_host_step;

/* The device buffers of the same step (device memory, shapes as in pkv_host_step). */
typedef struct {
    void *q;
    void *k_new;
    void *v_new;
    int32_t *block_tables;
    int32_t *seq_lens;
    void *out;
} pkv_device_step;

/* One whole decode step from host memory in one call [Decode][Slot][Attn]: asynchronous
 * copies of the step's inputs host -> device on `stream`, pkv_decode_step on the device
 * buffers, and the copy of out back to host -- every operation issued by this call, in
 * stream order.  With host->contiguous set, the caller promises that the inputs present lie
 * back to back, in the order q, k_new, v_new, block_tables, seq_lens, within one host
 * allocation and likewise within one device allocation (dev->q first); they then travel in
 * one copy (INVALID if the pointers are not so laid out).  Otherwise each travels in its
 * own copy.  It returns once everything is issued: synchronise the stream before reading
 * host->out or reusing the host inputs.  Caches, workspace, opts and errors as
 * pkv_decode_step; INVALID if a needed pointer is NULL. */
int pkv_decode_step_host(pkv_pool *pool, const pkv_host_step *host, const pkv_device_step *dev,
                         void *key_cache, void *value_cache, int32_t batch, int32_t num_q_heads,
                         int32_t max_blocks, float scale, void *workspace, size_t workspace_bytes,
                         const pkv_decode_opts *opts, void *stream);

/* Bytes of the fixed device scratch behind pkv_paged_attention_decode_noalloc. */
#define PKV_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Paged decode attention that allocates nothing and takes no workspace.  The pages describe
 * no such call; it exists for hosts that cannot allocate device memory while they run (a
 * memory manager that owns every device byte, or a latency-bound loop that cannot afford an
 * allocation's synchronisation, cost or failure).  Same arguments, result and errors as
 * pkv_paged_attention_decode without the workspace: the scratch is a fixed array of
 * PKV_NOALLOC_SCRATCH_BYTES compiled into the library, held by every GPU that loads it
 * until the process exits.  Returns PKV_ERR_INVALID, launching nothing, if the shape needs
 * more scratch than that (pkv_decode_workspace_bytes() tells how much it needs).  The
 * pool's device must be the current device (INVALID otherwise).  The first call on a device
 * looks up the array's device address (once per device, with that device current); make
 * that first call before any stream capture.  The cached address does not survive
 * cudaDeviceReset(), which invalidates the pools' error words as well: create and attach
 * pools again and do not call this entry point across a reset.  Every argument check is
 * made before anything is queued; a call that passes them clears the array's counters with
 * an asynchronous memset on `stream`, then runs the same kernel with the same launch plan
 * as pkv_paged_attention_decode, so the two give bit-identical outputs.  All calls on a
 * device share the array, so calls that overlap on the GPU race and must not be issued.
 * The pool must be attached beforehand (pkv_pool_attach_device allocates its 4-byte error
 * word once). */
int pkv_paged_attention_decode_noalloc(pkv_pool *pool, const void *q, const void *key_cache,
                                       const void *value_cache, const int32_t *block_tables,
                                       const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                       int32_t max_blocks, float scale, void *out, void *stream);

/* Synchronise the stream, read the pool's device error word into *bits_out and clear it.
 * Returns PKV_OK if it was zero, PKV_ERR_TIMEOUT if the timeout bit was set, else
 * PKV_ERR_DEVICE. */
int pkv_get_device_error(pkv_pool *pool, void *stream, uint32_t *bits_out);

/* Test hook for the failure path of the kernels' bounded waits (the pages have no
 * counterpart; it exists so that a test can see that path run).  While `which` is
 * PKV_TEST_EXPIRE_DECODE (every decode entry point) or PKV_TEST_EXPIRE_PREFILL
 * (pkv_paged_prefill), every launch of that kernel makes one of its roles -- the decode's
 * streaming warps before their first block, the prefill's Q loader before its first load --
 * wait about 1 ms on an mbarrier that nothing completes.  The wait runs out, the kernel sets
 * PKV_DEVERR_TIMEOUT, and the roles that depend on the stalled one give up in turn (each
 * after its normal bound of about 1 s at most); copies already in flight are waited for
 * (bounded) before a CTA leaves, so the context stays usable and pkv_get_device_error()
 * returns PKV_ERR_TIMEOUT.  Outputs of such a launch are unspecified.  Decode workspace
 * counters still return to zero.  PKV_TEST_EXPIRE_NONE (the default) turns it off.  The
 * setting is process-wide and read when a call launches; INVALID for any other value. */
#define PKV_TEST_EXPIRE_NONE 0
#define PKV_TEST_EXPIRE_DECODE 1
#define PKV_TEST_EXPIRE_PREFILL 2
int pkv_test_expire_waits(int32_t which);

/* Device-to-device copy of `bytes` (a multiple of 16; both pointers 16-byte aligned) by a
 * plain streaming kernel: the bandwidth denominator measured in the same process. */
int pkv_probe_copy(void *dst, const void *src, size_t bytes, void *stream);

/* Number of SMs of a device (used by the partition planner). */
int pkv_device_sm_count(int device, int32_t *out);

/* Static description of a status code (never NULL). */
const char *pkv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
