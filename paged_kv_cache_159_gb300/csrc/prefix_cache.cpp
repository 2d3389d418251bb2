// prefix_cache.cpp -- automatic prefix caching on the host: a hash per full block, lookup of
// a request's longest cached prefix, insertion of a request's blocks, LRU eviction.
//
// "KV Cache 与推理优化" (note.yj-dis.top), section "APC：连计算都省了": every block gets a
// content hash; a new request whose prefix equals an earlier request's (a common system
// prompt) reuses those physical blocks and skips their prefill; the lookup walks the
// request's 16-token blocks and stops at the first miss, after which nothing can hit.
// "一个请求为什么越生成越占内存?" (learning-field-guides), paging section: reuse must match
// the tokens, their positions and the model.  So block i's hash covers the previous block's
// hash (a per-model salt for block 0) and its own tokens; equal hashes then stand for equal
// prefixes, and every hit is verified against the stored tokens, parent and salt, so a
// 64-bit collision can never hand out another prefix's block.  The hash is 64-bit FNV-1a
// (Fowler, Noll, Vo) over the 8 little-endian bytes of the previous hash followed by the
// block's tokens as 4 little-endian bytes each.
//
// A cached block holds one reference of its own (pkv_pool_share semantics), so it outlives
// the requests that computed it.  Eviction releases that reference for the least recently
// used entries that no table holds and that have no cached child (children go first, so a
// cached chain never has a hole).
#include <cstring>
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pkv_internal.h"

namespace {

constexpr uint64_t FNV_OFFSET = 0xCBF29CE484222325ull;
constexpr uint64_t FNV_PRIME = 0x100000001B3ull;

uint64_t fnv1a_step(uint64_t h, uint8_t byte) { return (h ^ byte) * FNV_PRIME; }

uint64_t block_hash(uint64_t prev, const int32_t *tok, int bs)
{
    uint64_t h = FNV_OFFSET;
    for (int i = 0; i < 8; ++i) h = fnv1a_step(h, (uint8_t)(prev >> (8 * i)));
    for (int t = 0; t < bs; ++t) {
        const uint32_t w = (uint32_t)tok[t];
        for (int i = 0; i < 4; ++i) h = fnv1a_step(h, (uint8_t)(w >> (8 * i)));
    }
    return h;
}

}  // namespace

struct pkv_prefix_entry {
    uint64_t hash, salt, stamp;
    int32_t block, parent, children;
    std::vector<int32_t> tokens;
};

struct pkv_prefix_cache {
    std::unordered_map<int32_t, pkv_prefix_entry> by_block;
    std::unordered_multimap<uint64_t, int32_t> by_hash;
    std::set<std::pair<uint64_t, int32_t>> leaves;        // (stamp, block), no cached child
    uint64_t clock = 0;

    void touch(pkv_prefix_entry &e)
    {
        const bool leaf = e.children == 0;
        if (leaf) leaves.erase({e.stamp, e.block});
        e.stamp = ++clock;
        if (leaf) leaves.insert({e.stamp, e.block});
    }

    pkv_prefix_entry *match(uint64_t h, int32_t parent, uint64_t salt, const int32_t *tok, int bs)
    {
        auto range = by_hash.equal_range(h);
        for (auto it = range.first; it != range.second; ++it) {
            pkv_prefix_entry &e = by_block.at(it->second);
            if (e.parent == parent && e.salt == salt &&
                std::memcmp(e.tokens.data(), tok, sizeof(int32_t) * bs) == 0)
                return &e;
        }
        return nullptr;
    }

    // Remove an entry and release the cache's reference on its block.
    void drop(pkv_pool *pool, int32_t block)
    {
        pkv_prefix_entry &e = by_block.at(block);
        leaves.erase({e.stamp, e.block});
        auto range = by_hash.equal_range(e.hash);
        for (auto it = range.first; it != range.second; ++it)
            if (it->second == block) {
                by_hash.erase(it);
                break;
            }
        if (e.parent >= 0) {
            pkv_prefix_entry &p = by_block.at(e.parent);
            if (--p.children == 0) leaves.insert({p.stamp, p.block});
        }
        by_block.erase(block);
        if (--pool->refcount[(size_t)block] == 0) pool->free_list.push_back(block);
    }
};

namespace pkv {

void destroy_prefix_cache(pkv_pool *pool)
{
    delete pool->prefix;
    pool->prefix = nullptr;
}

}  // namespace pkv

namespace {

pkv_prefix_cache *cache_of(pkv_pool *pool)
{
    if (!pool->prefix) pool->prefix = new (std::nothrow) pkv_prefix_cache();
    return pool->prefix;
}

}  // namespace

extern "C" {

int pkv_block_hashes(const int32_t *tokens, int32_t num_tokens, int32_t block_size, uint64_t salt,
                     uint64_t *hashes_out)
{
    if (num_tokens < 0 || block_size < 1) return PKV_ERR_INVALID;
    const int32_t n = num_tokens / block_size;
    if (n > 0 && (!tokens || !hashes_out)) return PKV_ERR_INVALID;
    uint64_t prev = salt;
    for (int32_t i = 0; i < n; ++i) {
        prev = block_hash(prev, tokens + (size_t)i * block_size, block_size);
        hashes_out[i] = prev;
    }
    return PKV_OK;
}

int pkv_prefix_lookup(pkv_pool *pool, const int32_t *tokens, int32_t num_tokens, uint64_t salt,
                      int32_t *block_ids_out, int32_t *num_hits)
{
    if (!pool || num_tokens < 0 || !num_hits) return PKV_ERR_INVALID;
    const int bs = pool->desc.block_size;
    const int32_t n = num_tokens / bs;
    if (n > 0 && (!tokens || !block_ids_out)) return PKV_ERR_INVALID;
    *num_hits = 0;
    pkv_prefix_cache *c = cache_of(pool);
    if (!c) return PKV_ERR_OOM;
    uint64_t prev = salt;
    int32_t parent = -1, hits = 0;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t *tok = tokens + (size_t)i * bs;
        prev = block_hash(prev, tok, bs);
        pkv_prefix_entry *e = c->match(prev, parent, salt, tok, bs);
        if (!e) break;                                  // the first miss ends the walk
        c->touch(*e);
        block_ids_out[hits++] = e->block;
        parent = e->block;
    }
    *num_hits = hits;
    return PKV_OK;
}

int pkv_prefix_insert(pkv_pool *pool, const int32_t *tokens, int32_t num_tokens, uint64_t salt,
                      const int32_t *table_row, int32_t row_len, int32_t *num_added)
{
    if (!pool || num_tokens < 0 || row_len < 0 || !num_added) return PKV_ERR_INVALID;
    const int bs = pool->desc.block_size;
    const int32_t n = num_tokens / bs;
    if (n > row_len) return PKV_ERR_INVALID;
    if (n > 0 && (!tokens || !table_row)) return PKV_ERR_INVALID;
    *num_added = 0;
    pkv_prefix_cache *c = cache_of(pool);
    if (!c) return PKV_ERR_OOM;
    // plan: per block, the entry it already matches, or the row block that will hold it
    struct Step { pkv_prefix_entry *hit; uint64_t hash; int32_t block, parent; };
    std::vector<Step> plan;
    plan.reserve((size_t)n);
    uint64_t prev = salt;
    int32_t parent = -1;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t *tok = tokens + (size_t)i * bs;
        prev = block_hash(prev, tok, bs);
        pkv_prefix_entry *e = c->match(prev, parent, salt, tok, bs);
        if (e) {
            plan.push_back({e, prev, e->block, parent});
            parent = e->block;
            continue;
        }
        const int32_t b = table_row[i];
        if (b < 0 || b >= pool->desc.num_blocks || pool->refcount[(size_t)b] < 1 || c->by_block.count(b))
            return PKV_ERR_INVALID;
        for (const Step &s : plan)
            if (!s.hit && s.block == b) return PKV_ERR_INVALID;      // the same block twice
        plan.push_back({nullptr, prev, b, parent});
        parent = b;
    }
    int32_t added = 0;
    for (int32_t i = 0; i < n; ++i) {
        const Step &s = plan[(size_t)i];
        if (s.hit) {
            c->touch(*s.hit);
            continue;
        }
        pkv_prefix_entry e;
        e.hash = s.hash;
        e.salt = salt;
        e.stamp = ++c->clock;
        e.block = s.block;
        e.parent = s.parent;
        e.children = 0;
        e.tokens.assign(tokens + (size_t)i * bs, tokens + (size_t)(i + 1) * bs);
        if (s.parent >= 0) {
            pkv_prefix_entry &p = c->by_block.at(s.parent);
            if (p.children++ == 0) c->leaves.erase({p.stamp, p.block});
        }
        c->leaves.insert({e.stamp, e.block});
        c->by_hash.emplace(e.hash, e.block);
        c->by_block.emplace(e.block, std::move(e));
        pool->refcount[(size_t)s.block] += 1;            // the cache's own reference
        ++added;
    }
    *num_added = added;
    return PKV_OK;
}

int pkv_prefix_evict(pkv_pool *pool, int32_t max_blocks, int32_t *evicted_out, int32_t *num_evicted)
{
    if (!pool || max_blocks < 0 || !num_evicted || (max_blocks > 0 && !evicted_out)) return PKV_ERR_INVALID;
    *num_evicted = 0;
    pkv_prefix_cache *c = pool->prefix;
    if (!c) return PKV_OK;
    int32_t n = 0;
    while (n < max_blocks) {
        int32_t victim = -1;
        for (const auto &leaf : c->leaves)                // least recently used first
            if (pool->refcount[(size_t)leaf.second] == 1) {
                victim = leaf.second;
                break;
            }
        if (victim < 0) break;
        c->drop(pool, victim);
        evicted_out[n++] = victim;
    }
    *num_evicted = n;
    return PKV_OK;
}

int pkv_prefix_clear(pkv_pool *pool)
{
    if (!pool) return PKV_ERR_INVALID;
    pkv_prefix_cache *c = pool->prefix;
    if (!c) return PKV_OK;
    while (!c->leaves.empty()) c->drop(pool, c->leaves.begin()->second);
    return PKV_OK;
}

int pkv_prefix_cached_blocks(const pkv_pool *pool, int32_t *out)
{
    if (!pool || !out) return PKV_ERR_INVALID;
    *out = pool->prefix ? (int32_t)pool->prefix->by_block.size() : 0;
    return PKV_OK;
}

}  // extern "C"
