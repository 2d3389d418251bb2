// paged_decode.cu -- host entry points of paged decode attention (plan, validation,
// launch) and the split-KV combine kernel.  The decode kernels themselves are in
// decode_kernels.cuh, instantiated per (head_dim, pool dtype) by decode_inst_*.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "decode_kernels.cuh"

namespace pkv {
namespace decode {

// ------------------------------------------------------------------------------------
// Split-KV combine: out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p, p in logical order.
// One warp per (sequence, query head); lanes cover head_dim.
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const DecodeParams p)
{
    const int w = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (w >= p.B * p.Hq) return;
    const int b = w / p.Hq;
    const int L = __ldg(p.seq_lens + b);
    if (L < 1 || L > p.MB * BS) return;              // flagged by the decode kernel
    const int nblk = (L + BS - 1) / BS;
    const int nparts = (nblk + p.PB - 1) / p.PB;
    if (nparts <= 1) return;                         // written directly by the decode kernel
    const float *ml = p.part_ml + (size_t)w * p.P * 2;
    const float *po = p.part_o + (size_t)w * p.P * D;
    float M = -INFINITY;
    for (int q = 0; q < nparts; ++q) M = fmaxf(M, ml[2 * q]);
    constexpr int EPL = D / 32;
    float num[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) num[e] = 0.f;
    float den = 0.f;
    if (M != -INFINITY) {
        for (int q = 0; q < nparts; ++q) {
            const float mq = ml[2 * q];
            const float wt = mq == -INFINITY ? 0.f : dev::fast_exp2(mq - M);
            den += wt * ml[2 * q + 1];
#pragma unroll
            for (int e = 0; e < EPL; ++e) num[e] += wt * po[(size_t)q * D + e * 32 + lane];
        }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        const float o = den > 0.f ? num[e] / den : 0.f;
        const __nv_bfloat16 ob = __float2bfloat16_rn(o);
        p.out[(size_t)w * D + e * 32 + lane] = *reinterpret_cast<const uint16_t *>(&ob);
    }
}

// ------------------------------------------------------------------------------------
// Host side: plan, dispatch.
// ------------------------------------------------------------------------------------

int sm_count_cached()
{
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cached[dev] = v;
    }
    return cached[dev];
}

int make_plan(const pkv_pool_desc &d, int B, int Hq, int MB, const pkv_decode_opts *o, int sms,
              Plan &pl)
{
    if (B < 0 || Hq < 1 || MB < 1 || Hq % d.num_kv_heads != 0) return PKV_ERR_INVALID;
    const int group = Hq / d.num_kv_heads;
    if (group > 16) return PKV_ERR_INVALID;
    pkv_decode_opts z{};
    if (!o) o = &z;
    pl.variant = o->variant ? o->variant : 2;
    if (pl.variant != 1 && pl.variant != 2) return PKV_ERR_INVALID;
    if (pl.variant == 1 && group > 8) return PKV_ERR_INVALID;
    pl.nw = o->warps_per_cta ? o->warps_per_cta : 4;
    if (pl.nw != 1 && pl.nw != 2 && pl.nw != 4 && pl.nw != 8) return PKV_ERR_INVALID;
    pl.ns = o->stages ? o->stages : 2;
    if (pl.ns < 1 || pl.ns > 4) return PKV_ERR_INVALID;
    if (o->partition_blocks < 0) return PKV_ERR_INVALID;
    if (o->partition_blocks) {
        pl.pb = o->partition_blocks;
    } else {
        // Enough CTAs to cover every SM several times; split sequences only when the
        // (sequence, KV head) units alone are too few.
        const long units = (long)B * d.num_kv_heads;
        const long target = 3L * sms;
        if (units >= target || units == 0) {
            pl.pb = MB;
        } else {
            const long parts = (target + units - 1) / units;
            pl.pb = (int)((MB + parts - 1) / parts);
            pl.pb = std::max(pl.pb, 4 * pl.nw);      // at least 4 blocks per warp
        }
    }
    pl.pb = std::min(pl.pb, std::min(MB, PB_MAX));
    pl.parts = (MB + pl.pb - 1) / pl.pb;
    pl.ws_o = 0;
    pl.ws_ml = 0;
    pl.ws_bytes = 0;
    if (pl.parts > 1) {
        const size_t rows = (size_t)B * Hq * pl.parts;
        pl.ws_o = 0;
        pl.ws_ml = (rows * d.head_dim * 4 + 255) / 256 * 256;
        pl.ws_bytes = pl.ws_ml + (rows * 2 * 4 + 255) / 256 * 256;
    }
    return PKV_OK;
}

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

}  // namespace decode
}  // namespace pkv

extern template cudaError_t pkv::decode::dispatch_nw_ns<128, false>(const pkv::decode::Plan &, int, int, cudaStream_t, const pkv::decode::DecodeParams &);
extern template cudaError_t pkv::decode::dispatch_nw_ns<128, true>(const pkv::decode::Plan &, int, int, cudaStream_t, const pkv::decode::DecodeParams &);
extern template cudaError_t pkv::decode::dispatch_nw_ns<64, false>(const pkv::decode::Plan &, int, int, cudaStream_t, const pkv::decode::DecodeParams &);
extern template cudaError_t pkv::decode::dispatch_nw_ns<64, true>(const pkv::decode::Plan &, int, int, cudaStream_t, const pkv::decode::DecodeParams &);

extern "C" size_t pkv_decode_workspace_bytes(const pkv_pool *pool, int32_t batch, int32_t num_q_heads,
                                             int32_t max_blocks, const pkv_decode_opts *opts)
{
    if (!pool) return 0;
    pkv::decode::Plan pl;
    if (pkv::decode::make_plan(pool->desc, batch, num_q_heads, max_blocks, opts, pkv::decode::sm_count_cached(), pl) != PKV_OK)
        return 0;
    return pl.ws_bytes;
}

extern "C" int pkv_paged_attention_decode_ex(pkv_pool *pool, const void *q, const void *key_cache,
                                             const void *value_cache, const int32_t *block_tables,
                                             const int32_t *seq_lens, int32_t batch,
                                             int32_t num_q_heads, int32_t max_blocks, float scale,
                                             void *out, void *workspace, size_t workspace_bytes,
                                             const pkv_decode_opts *opts, void *stream)
{
    using namespace pkv;
    using namespace pkv::decode;
    int st = check_attached(pool);
    if (st != PKV_OK) return st;
    if (batch < 0 || !std::isfinite(scale)) return PKV_ERR_INVALID;
    if (batch == 0) return PKV_OK;
    if (!q || !key_cache || !value_cache || !block_tables || !seq_lens || !out) return PKV_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PKV_ERR_INVALID;
    const pkv_pool_desc &d = pool->desc;
    Plan pl;
    st = make_plan(d, batch, num_q_heads, max_blocks, opts, sm_count_cached(), pl);
    if (st != PKV_OK) return st;
    if (pl.ws_bytes > 0 && (!workspace || workspace_bytes < pl.ws_bytes || !aligned(workspace, 256)))
        return PKV_ERR_INVALID;
    const long long grid_ll = (long long)batch * d.num_kv_heads * pl.parts;
    if (grid_ll > 0x7fffffffLL) return PKV_ERR_INVALID;

    DecodeParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.key_cache = static_cast<const uint8_t *>(key_cache);
    p.value_cache = static_cast<const uint8_t *>(value_cache);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.out = static_cast<uint16_t *>(out);
    p.part_o = pl.ws_bytes ? reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + pl.ws_o) : nullptr;
    p.part_ml = pl.ws_bytes ? reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + pl.ws_ml) : nullptr;
    p.err = pool->d_err;
    p.B = batch;
    p.Hq = num_q_heads;
    p.Hkv = d.num_kv_heads;
    p.group = num_q_heads / d.num_kv_heads;
    p.MB = max_blocks;
    p.P = pl.parts;
    p.PB = pl.pb;
    p.num_blocks = d.num_blocks;
    p.score_scale = scale * d.k_scale * LOG2E;
    p.out_scale = d.v_scale;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int grid = (int)grid_ll;
    const bool fp8 = d.kv_dtype == PKV_KV_FP8E4M3;
    cudaError_t e;
    if (d.head_dim == 128)
        e = fp8 ? dispatch_nw_ns<128, true>(pl, p.group, grid, s, p) : dispatch_nw_ns<128, false>(pl, p.group, grid, s, p);
    else
        e = fp8 ? dispatch_nw_ns<64, true>(pl, p.group, grid, s, p) : dispatch_nw_ns<64, false>(pl, p.group, grid, s, p);
    if (e == cudaErrorInvalidConfiguration) return PKV_ERR_INVALID;
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    if (pl.parts > 1) {
        const int rows = batch * num_q_heads;
        const int cgrid = (rows + 3) / 4;
        if (d.head_dim == 128) combine_kernel<128><<<cgrid, 128, 0, s>>>(p);
        else combine_kernel<64><<<cgrid, 128, 0, s>>>(p);
        if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

extern "C" int pkv_paged_attention_decode(pkv_pool *pool, const void *q, const void *key_cache,
                                          const void *value_cache, const int32_t *block_tables,
                                          const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                          int32_t max_blocks, float scale, void *out, void *workspace,
                                          size_t workspace_bytes, void *stream)
{
    return pkv_paged_attention_decode_ex(pool, q, key_cache, value_cache, block_tables, seq_lens, batch,
                                         num_q_heads, max_blocks, scale, out, workspace, workspace_bytes,
                                         nullptr, stream);
}
