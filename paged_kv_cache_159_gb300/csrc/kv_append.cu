// kv_append.cu -- scatter each new token's K/V rows into its slot of the paged pool.
//
// "理解 KV Cache：Attention、P/D 分离与 vLLM 的页式显存管理" (steinslab.io) §1.3 treats the
// KV cache as an append-only log: each decode step adds one K/V record per token and layer.
// §3.3 gives the address: physical block = slot / block_size, offset = slot % block_size,
// and §3.2 the per-block layout [num_kv_heads, block_size, head_dim].  FP8 pools follow the
// "KV 量化" section of "KV Cache 与推理优化" (note.yj-dis.top): 1-byte storage, scaled.
//
// Work split: one thread per 16-byte piece of a (layer, token, head) row, K and V handled by
// the same thread; consecutive threads cover consecutive bytes of a row, so reads of k/v are
// fully coalesced and each row lands as whole 16-byte stores.  The op moves a few hundred
// KB per step and layer and is launch-latency bound; it shares the decode's stream.  With
// several layers (k, v [layers, tokens, Hkv, D], caches stacked layer-major) one launch
// writes every layer: a token has the same slot in each, since a block spans all layers.
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

using dev::flag_error;

// Destination piece of source piece i, or -1 (padding slot) / -2 (slot beyond the pool).
// i runs over [layers, tokens, Hkv, chunks]; the cache is [layers, NB, Hkv, 16, chunks].
__device__ __forceinline__ int64_t dst_piece(int64_t i, const int64_t *__restrict__ slots,
                                             int64_t num_tokens, int num_kv_heads,
                                             int chunks_per_row, int64_t num_slots)
{
    const int64_t per_token = (int64_t)num_kv_heads * chunks_per_row;
    const int64_t lt = i / per_token;                  // layer * num_tokens + t
    const int64_t r = i - lt * per_token;              // = h * chunks_per_row + c
    const int64_t layer = lt / num_tokens, t = lt - layer * num_tokens;
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) return -1;
    if (slot >= num_slots) return -2;
    const int64_t blk = slot >> 4, off = slot & 15;
    const int64_t h = r / chunks_per_row, c = r - h * chunks_per_row;
    return (((layer * (num_slots >> 4) + blk) * num_kv_heads + h) * 16 + off) * chunks_per_row + c;
}

// bf16 pool: 16-byte bit copies.
__global__ void __launch_bounds__(256) kv_append_bf16_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, const int64_t *__restrict__ slots,
    int64_t num_tokens, int layers, int num_kv_heads, int chunks_per_row, int64_t num_slots,
    uint4 *__restrict__ key_cache, uint4 *__restrict__ value_cache, uint32_t *err)
{
    const int64_t total = layers * num_tokens * num_kv_heads * chunks_per_row;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t dst = dst_piece(i, slots, num_tokens, num_kv_heads, chunks_per_row, num_slots);
        if (dst == -2) flag_error(err, PKV_DEVERR_SLOT);
        if (dst < 0) continue;
        key_cache[dst] = __ldg(k + i);
        value_cache[dst] = __ldg(v + i);
    }
}

using dev::e4m3x2_satfinite;

// 8 bf16 values scaled by inv then encoded: 16 bytes in, 8 bytes out.
__device__ __forceinline__ uint2 encode8(uint4 x, float inv)
{
    uint2 o;
    o.x = e4m3x2_satfinite(dev::bf16_lo(x.x) * inv, dev::bf16_hi(x.x) * inv) |
          (e4m3x2_satfinite(dev::bf16_lo(x.y) * inv, dev::bf16_hi(x.y) * inv) << 16);
    o.y = e4m3x2_satfinite(dev::bf16_lo(x.z) * inv, dev::bf16_hi(x.z) * inv) |
          (e4m3x2_satfinite(dev::bf16_lo(x.w) * inv, dev::bf16_hi(x.w) * inv) << 16);
    return o;
}

// FP8 pool: read 8 bf16, write 8 codes.
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, const int64_t *__restrict__ slots,
    int64_t num_tokens, int layers, int num_kv_heads, int chunks_per_row, int64_t num_slots,
    float inv_k, float inv_v, uint2 *__restrict__ key_cache, uint2 *__restrict__ value_cache,
    uint32_t *err)
{
    const int64_t total = layers * num_tokens * num_kv_heads * chunks_per_row;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t dst = dst_piece(i, slots, num_tokens, num_kv_heads, chunks_per_row, num_slots);
        if (dst == -2) flag_error(err, PKV_DEVERR_SLOT);
        if (dst < 0) continue;
        key_cache[dst] = encode8(__ldg(k + i), inv_k);
        value_cache[dst] = encode8(__ldg(v + i), inv_v);
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int append_impl(pkv_pool *pool, int layers, const void *k, const void *v,
                const int64_t *slot_mapping, int32_t num_tokens, void *key_cache,
                void *value_cache, void *stream)
{
    int st = check_attached(pool);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !key_cache || !value_cache) return PKV_ERR_INVALID;
    if (!aligned16(k) || !aligned16(v) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PKV_ERR_INVALID;
    const pkv_pool_desc &d = pool->desc;
    const int chunks = d.head_dim / 8;                 // 8 bf16 source values per chunk
    const int64_t total = (int64_t)layers * num_tokens * d.num_kv_heads * chunks;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 65535LL * 32) blocks = 65535LL * 32;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t num_slots = (int64_t)d.num_blocks * d.block_size;
    if (d.kv_dtype == PKV_KV_BF16) {
        kv_append_bf16_kernel<<<(unsigned)blocks, threads, 0, s>>>(
            static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping,
            num_tokens, layers, d.num_kv_heads, chunks, num_slots, static_cast<uint4 *>(key_cache),
            static_cast<uint4 *>(value_cache), pool->d_err);
    } else {
        kv_append_fp8_kernel<<<(unsigned)blocks, threads, 0, s>>>(
            static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping,
            num_tokens, layers, d.num_kv_heads, chunks, num_slots, pool->inv_k_scale,
            pool->inv_v_scale, static_cast<uint2 *>(key_cache), static_cast<uint2 *>(value_cache),
            pool->d_err);
    }
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_kv_append(pkv_pool *pool, const void *k, const void *v,
                             const int64_t *slot_mapping, int32_t num_tokens, void *key_cache,
                             void *value_cache, void *stream)
{
    return pkv::append_impl(pool, 1, k, v, slot_mapping, num_tokens, key_cache, value_cache, stream);
}

extern "C" int pkv_kv_append_layers(pkv_pool *pool, const void *k, const void *v,
                                    const int64_t *slot_mapping, int32_t num_tokens,
                                    void *key_cache, void *value_cache, void *stream)
{
    if (!pool) return PKV_ERR_INVALID;
    return pkv::append_impl(pool, pool->desc.num_layers, k, v, slot_mapping, num_tokens, key_cache,
                            value_cache, stream);
}
