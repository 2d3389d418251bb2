// copy_blocks.cu -- copy whole physical blocks of the paged pool (every layer, K and V).
//
// "KV Cache 与推理优化" (note.yj-dis.top), PagedAttention section: a prefix block is stored
// once and shared by every request that references it; when a request diverges it gets its
// own copy before it writes (copy-on-write).  pkv_cow_prepare picks the (shared, fresh)
// pairs on the host; this kernel makes the fresh blocks byte-identical to the shared ones.
//
// Layout ("理解 KV Cache" §3.2): a cache is [layers, NB, Hkv, 16, D], so one block of one
// layer is a contiguous Hkv * 16 * D elements (32 KiB bf16 at Hkv 8, D 128).  One CTA copies
// one (pair, layer) for K and for V with 16-byte loads, 8 in flight per thread before the
// stores, streaming (evict-first) since the copied block is written again by the append.
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int CB_THREADS = 256;
constexpr int CB_UNROLL = 8;

__global__ void __launch_bounds__(CB_THREADS) copy_blocks_kernel(
    const int32_t *__restrict__ src, const int32_t *__restrict__ dst, int layers, int num_blocks,
    int64_t block_words, uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache,
    uint32_t *err)
{
    const int pair = blockIdx.x / layers, layer = blockIdx.x - pair * layers;
    const int s = __ldg(src + pair), d = __ldg(dst + pair);
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
        if (threadIdx.x == 0 && layer == 0) dev::flag_error(err, PKV_DEVERR_BLOCK_ID);
        return;
    }
    const int64_t base = (int64_t)layer * num_blocks * block_words;
    for (int kv = 0; kv < 2; ++kv) {
        uint4 *cache = kv ? value_cache : key_cache;
        const uint4 *from = cache + base + (int64_t)s * block_words;
        uint4 *to = cache + base + (int64_t)d * block_words;
        for (int64_t i0 = 0; i0 < block_words; i0 += (int64_t)CB_THREADS * CB_UNROLL) {
            uint4 w[CB_UNROLL];
#pragma unroll
            for (int u = 0; u < CB_UNROLL; ++u) {
                const int64_t i = i0 + (int64_t)u * CB_THREADS + threadIdx.x;
                if (i < block_words) w[u] = __ldcs(from + i);
            }
#pragma unroll
            for (int u = 0; u < CB_UNROLL; ++u) {
                const int64_t i = i0 + (int64_t)u * CB_THREADS + threadIdx.x;
                if (i < block_words) __stcs(to + i, w[u]);
            }
        }
    }
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_copy_blocks(pkv_pool *pool, void *key_cache, void *value_cache,
                               const int32_t *src, const int32_t *dst, int32_t num_pairs,
                               void *stream)
{
    int st = pkv::check_attached(pool);
    if (st != PKV_OK) return st;
    if (num_pairs < 0) return PKV_ERR_INVALID;
    if (num_pairs == 0) return PKV_OK;
    if (!key_cache || !value_cache || !src || !dst) return PKV_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(key_cache) & 15u) || (reinterpret_cast<uintptr_t>(value_cache) & 15u) ||
        (reinterpret_cast<uintptr_t>(src) & 3u) || (reinterpret_cast<uintptr_t>(dst) & 3u))
        return PKV_ERR_INVALID;
    const pkv_pool_desc &d = pool->desc;
    const int layers = d.num_layers;
    if ((int64_t)num_pairs * layers >= (int64_t)1 << 31) return PKV_ERR_INVALID;
    const int64_t block_words = (int64_t)d.num_kv_heads * d.block_size * d.head_dim * pkv::elem_bytes(d) / 16;
    pkv::copy_blocks_kernel<<<(unsigned)(num_pairs * layers), pkv::CB_THREADS, 0,
                              static_cast<cudaStream_t>(stream)>>>(
        src, dst, layers, d.num_blocks, block_words, static_cast<uint4 *>(key_cache),
        static_cast<uint4 *>(value_cache), pool->d_err);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
