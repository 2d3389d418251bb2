// pkv_internal.h -- definitions shared by the host allocator (pool.cpp) and the CUDA
// translation units of libpkv.so.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <deque>
#include <vector>

#include "../../include/pkv.h"

struct pkv_prefix_cache;               // prefix_cache.cpp

struct pkv_pool {
    pkv_pool_desc desc;
    std::deque<int32_t> free_list;     // front is handed out first
    std::vector<int32_t> refcount;     // per physical block, 0 = free
    int device = -1;                   // -1 until pkv_pool_attach_device
    uint32_t *d_err = nullptr;         // device error word (PKV_DEVERR_* bits)
    float inv_k_scale = 1.0f;          // fl32(1 / k_scale), computed once on the host
    float inv_v_scale = 1.0f;
    pkv_prefix_cache *prefix = nullptr;    // cached full blocks (created on first use)
};

namespace pkv {

// Free the pool's prefix cache, if any (its block references are not released).
void destroy_prefix_cache(pkv_pool *pool);

// Validation shared by the CUDA entry points.
int check_attached(const pkv_pool *pool);
inline int elem_bytes(const pkv_pool_desc &d) { return d.kv_dtype == PKV_KV_FP8E4M3 ? 1 : 2; }

}  // namespace pkv
