// pkv_internal.h -- definitions shared by the host allocator (pool.cpp) and the CUDA
// translation units of libpkv.so.  Not part of the public ABI.
#pragma once

#include <cuda.h>

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

// A tiled tensor map (TMA descriptor) of rank 3 or 4 over `ptr`: dims innermost first,
// strides in bytes of dims 1 .. rank-1, box in elements.  false if the driver's encoder is
// unavailable or refuses.
bool encode_tiled(CUtensorMap *map, const void *ptr, CUtensorMapDataType type, int rank, const uint64_t *dims,
                  const uint64_t *strides, const uint32_t *box, CUtensorMapSwizzle swizzle);
inline bool encode_tiled_3d(CUtensorMap *map, const void *ptr, CUtensorMapDataType type, const uint64_t (&dims)[3],
                            const uint64_t (&strides)[2], const uint32_t (&box)[3], CUtensorMapSwizzle swizzle)
{
    return encode_tiled(map, ptr, type, 3, dims, strides, box, swizzle);
}

// Which kernel (PKV_TEST_EXPIRE_*) the failure-path test hook currently targets.
int test_expire();

// Validation shared by the CUDA entry points.
int check_attached(const pkv_pool *pool);
inline int elem_bytes(const pkv_pool_desc &d) { return d.kv_dtype == PKV_KV_FP8E4M3 ? 1 : 2; }

namespace decode {
// Every host-side check of pkv_paged_attention_decode with batch >= 1 (arguments, alignment,
// launch plan, workspace size), without launching or queueing anything: PKV_OK, or the
// status that call would return.
int check_decode_call(const pkv_pool *pool, const void *q, const void *key_cache, const void *value_cache,
                      const int32_t *block_tables, const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                      int32_t max_blocks, float scale, const void *out, const void *workspace,
                      size_t workspace_bytes);
}  // namespace decode

}  // namespace pkv
