// paged_decode.cu -- host entry points of paged decode attention: launch plan, argument
// validation, launch.  The kernels are in decode_kernels.cuh, compiled per (head_dim, pool
// dtype) by decode_inst_*.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "decode_kernels.cuh"

extern template cudaError_t pkv::decode::dispatch_nw_ns<128, false>(const pkv::decode::Plan &, int, bool, int *,
                                                                    cudaStream_t, const pkv::decode::LaunchArgs *);
extern template cudaError_t pkv::decode::dispatch_nw_ns<128, true>(const pkv::decode::Plan &, int, bool, int *,
                                                                   cudaStream_t, const pkv::decode::LaunchArgs *);
extern template cudaError_t pkv::decode::dispatch_nw_ns<64, false>(const pkv::decode::Plan &, int, bool, int *,
                                                                   cudaStream_t, const pkv::decode::LaunchArgs *);
extern template cudaError_t pkv::decode::run_prefix<128, false>(const pkv::decode::LaunchArgs *, cudaStream_t);
extern template cudaError_t pkv::decode::run_prefix<128, true>(const pkv::decode::LaunchArgs *, cudaStream_t);
extern template cudaError_t pkv::decode::run_prefix<64, false>(const pkv::decode::LaunchArgs *, cudaStream_t);
extern template cudaError_t pkv::decode::run_prefix<64, true>(const pkv::decode::LaunchArgs *, cudaStream_t);
extern template cudaError_t pkv::decode::dispatch_nw_ns<64, true>(const pkv::decode::Plan &, int, bool, int *,
                                                                  cudaStream_t, const pkv::decode::LaunchArgs *);

namespace pkv {
namespace decode {
namespace {

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

cudaError_t dispatch(const pkv_pool_desc &d, const Plan &pl, int group, bool launch, int *per_sm,
                     cudaStream_t s, const LaunchArgs *p)
{
    const bool fp8 = d.kv_dtype == PKV_KV_FP8E4M3;
    if (d.head_dim == 128)
        return fp8 ? dispatch_nw_ns<128, true>(pl, group, launch, per_sm, s, p)
                   : dispatch_nw_ns<128, false>(pl, group, launch, per_sm, s, p);
    return fp8 ? dispatch_nw_ns<64, true>(pl, group, launch, per_sm, s, p)
               : dispatch_nw_ns<64, false>(pl, group, launch, per_sm, s, p);
}

// Choose variant, CTA shape and grid; size the workspace.  Queries the device (occupancy)
// unless opts fixes the grid.
int make_plan(const pkv_pool_desc &d, int B, int Hq, int MB, const pkv_decode_opts *o, Plan &pl)
{
    if (B < 1 || B > MAX_BATCH || Hq < 1 || MB < 1 || Hq % d.num_kv_heads != 0) return PKV_ERR_INVALID;
    const int group = Hq / d.num_kv_heads;
    if (group > 16) return PKV_ERR_INVALID;
    if ((long long)B * MB * d.num_kv_heads >= (1LL << 31)) return PKV_ERR_INVALID;
    if ((long long)d.num_layers * B * d.num_kv_heads >= (1LL << 31)) return PKV_ERR_INVALID;
    pkv_decode_opts z{};
    if (!o) o = &z;
    pl.variant = o->variant ? o->variant : 3;
    if (pl.variant < 1 || pl.variant > 3) return PKV_ERR_INVALID;
    if (pl.variant == 1 && group > 8) return PKV_ERR_INVALID;
    pl.nw = o->warps_per_cta ? o->warps_per_cta : 4;
    if (pl.variant == 3) {
        if (o->heads_per_copy) {
            pl.hp = o->heads_per_copy;
            if ((pl.hp != 1 && pl.hp != 2 && pl.hp != 4) || d.num_kv_heads % pl.hp) return PKV_ERR_INVALID;
        } else {
            pl.hp = 1;
        }
        if (pl.hp > pl.nw) return PKV_ERR_INVALID;
    } else {
        if (o->heads_per_copy > 1) return PKV_ERR_INVALID;
        pl.hp = 1;
    }
    // default ring: 16 KiB of tiles per warp (2 bf16 or 4 FP8 stages at head_dim 128)
    pl.ns = o->stages ? o->stages : (elem_bytes(d) == 1 && pl.variant >= 2 ? 4 : 2);
    if (o->grid_ctas < 0 || o->shared_prefix_blocks < 0) return PKV_ERR_INVALID;
    pl.sp = o->shared_prefix_blocks;
    if (pl.sp > 0 && (pl.variant != 3 || pl.hp != 1)) return PKV_ERR_INVALID;
    if (o->unit_cost < -1 || o->unit_cost > 4096) return PKV_ERR_INVALID;
    pl.uc = o->unit_cost == 0 ? 16 : (o->unit_cost < 0 ? 0 : o->unit_cost);
    const int tile = BS * d.head_dim * elem_bytes(d);
    pl.smem = Layout(pl.nw, pl.ns, tile, d.head_dim, group, B, pl.hp).total + 1024;   // + alignment slack
    if (pl.smem > 227 * 1024) return PKV_ERR_INVALID;
    if (o->grid_ctas) {
        pl.grid = o->grid_ctas;
    } else {
        int per_sm = 0;
        cudaError_t e = dispatch(d, pl, group, false, &per_sm, nullptr, nullptr);
        if (e == cudaErrorInvalidConfiguration) return PKV_ERR_INVALID;
        if (e != cudaSuccess || per_sm < 1) return PKV_ERR_CUDA;
        pl.grid = sm_count_cached() * per_sm;
    }
    const size_t rows = (size_t)pl.grid * 2 * group * pl.hp;
    pl.ws_counters = 0;
    pl.ws_o = ((size_t)d.num_layers * B * d.num_kv_heads * 4 + 255) / 256 * 256;   // counters
    pl.ws_ml = pl.ws_o + (rows * d.head_dim * 4 + 255) / 256 * 256;
    pl.ws_bytes = pl.ws_ml + (rows * 2 * 4 + 255) / 256 * 256;
    pl.ws_pre_n = pl.ws_pre_o = pl.ws_pre_ml = 0;
    if (pl.sp > 0) {
        // the shared-prefix pass: blocks covered per sequence, a partial state per query row
        const size_t prow = (size_t)d.num_layers * d.num_kv_heads * B * group;
        pl.ws_pre_n = pl.ws_bytes;
        pl.ws_pre_o = pl.ws_pre_n + ((size_t)B * 4 + 255) / 256 * 256;
        pl.ws_pre_ml = pl.ws_pre_o + (prow * d.head_dim * 4 + 255) / 256 * 256;
        pl.ws_bytes = pl.ws_pre_ml + (prow * 2 * 4 + 255) / 256 * 256;
    }
    return PKV_OK;
}

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

}  // namespace
}  // namespace decode
}  // namespace pkv

extern "C" size_t pkv_decode_workspace_bytes(const pkv_pool *pool, int32_t batch, int32_t num_q_heads,
                                             int32_t max_blocks, const pkv_decode_opts *opts)
{
    if (!pool) return 0;
    pkv::decode::Plan pl;
    if (pkv::decode::make_plan(pool->desc, batch, num_q_heads, max_blocks, opts, pl) != PKV_OK) return 0;
    return pl.ws_bytes;
}

namespace pkv {
namespace decode {
namespace {

// Every host-side check of a decode call with batch >= 1, and its launch plan; launches
// nothing and queues nothing.
int check_call(const pkv_pool *pool, const void *q, const void *k_new, const void *v_new,
               const void *key_cache, const void *value_cache, const int32_t *block_tables,
               const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_blocks,
               float scale, const void *out, const void *workspace, size_t workspace_bytes,
               const pkv_decode_opts *opts, Plan &pl)
{
    int st = check_attached(pool);
    if (st != PKV_OK) return st;
    if (batch < 1 || !std::isfinite(scale)) return PKV_ERR_INVALID;
    if (!q || !key_cache || !value_cache || !block_tables || !seq_lens || !out || !workspace)
        return PKV_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(workspace, 256))
        return PKV_ERR_INVALID;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID;
    if (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))) return PKV_ERR_INVALID;
    st = make_plan(pool->desc, batch, num_q_heads, max_blocks, opts, pl);
    if (st != PKV_OK) return st;
    if (workspace_bytes < pl.ws_bytes) return PKV_ERR_INVALID;
    return PKV_OK;
}

int decode_impl(pkv_pool *pool, int layers, const void *q, const void *k_new, const void *v_new,
                const void *key_cache, const void *value_cache, const int32_t *block_tables,
                const int32_t *seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_blocks,
                float scale, void *out, void *workspace, size_t workspace_bytes,
                const pkv_decode_opts *opts, void *stream)
{
    int st = check_attached(pool);
    if (st != PKV_OK) return st;
    if (batch < 0 || !std::isfinite(scale)) return PKV_ERR_INVALID;
    if (batch == 0) return PKV_OK;
    Plan pl;
    st = check_call(pool, q, k_new, v_new, key_cache, value_cache, block_tables, seq_lens, batch, num_q_heads,
                    max_blocks, scale, out, workspace, workspace_bytes, opts, pl);
    if (st != PKV_OK) return st;
    const pkv_pool_desc &d = pool->desc;

    LaunchArgs args;
    DecodeParams &p = args.p;
    if (pl.variant == 3) {
        // K and V tiles of every (layer, block, head) of the launch: [tiles][16 tokens][row]
        // with rows of D elements, copied per SEG-byte row segment with the matching swizzle
        const int eb = elem_bytes(d), rowb = d.head_dim * eb, seg = rowb < 128 ? rowb : 128;
        const uint64_t tiles = (uint64_t)layers * d.num_blocks * d.num_kv_heads;
        const CUtensorMapDataType type = eb == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const CUtensorMapSwizzle sw = seg == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        bool ok;
        if (rowb == 2 * seg) {
            // two row segments: [segment][token][seg] in shared memory from one 4-D copy whose
            // dimensions are (element in segment, token, segment, tile)
            const uint64_t dims[4] = {(uint64_t)(seg / eb), (uint64_t)BS, 2u, tiles};
            const uint64_t strides[3] = {(uint64_t)rowb, (uint64_t)seg, (uint64_t)rowb * BS};
            const uint32_t box[4] = {(uint32_t)(seg / eb), (uint32_t)BS, 2u, (uint32_t)pl.hp};
            ok = encode_tiled(&args.kmap, key_cache, type, 4, dims, strides, box, sw) &&
                 encode_tiled(&args.vmap, value_cache, type, 4, dims, strides, box, sw);
        } else {
            const uint64_t dims[3] = {(uint64_t)d.head_dim, (uint64_t)BS, tiles};
            const uint64_t strides[2] = {(uint64_t)rowb, (uint64_t)rowb * BS};
            const uint32_t box[3] = {(uint32_t)(seg / eb), (uint32_t)BS, (uint32_t)pl.hp};
            ok = encode_tiled_3d(&args.kmap, key_cache, type, dims, strides, box, sw) &&
                 encode_tiled_3d(&args.vmap, value_cache, type, dims, strides, box, sw);
        }
        if (!ok) return PKV_ERR_CUDA;
    }
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.q = static_cast<const uint16_t *>(q);
    p.key_cache = static_cast<const uint8_t *>(key_cache);
    p.value_cache = static_cast<const uint8_t *>(value_cache);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.out = static_cast<uint16_t *>(out);
    p.counters = reinterpret_cast<int32_t *>(ws + pl.ws_counters);
    p.part_o = reinterpret_cast<float *>(ws + pl.ws_o);
    p.part_ml = reinterpret_cast<float *>(ws + pl.ws_ml);
    p.err = pool->d_err;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.layers = layers;
    p.test_stall = test_expire() == PKV_TEST_EXPIRE_DECODE;
    p.shared_prefix = pl.sp;
    p.unit_cost = pl.uc;
    p.prefix_n = pl.sp ? reinterpret_cast<int32_t *>(ws + pl.ws_pre_n) : nullptr;
    p.pref_o = pl.sp ? reinterpret_cast<float *>(ws + pl.ws_pre_o) : nullptr;
    p.pref_ml = pl.sp ? reinterpret_cast<float *>(ws + pl.ws_pre_ml) : nullptr;
    p.B = batch;
    p.Hq = num_q_heads;
    p.Hkv = d.num_kv_heads;
    p.group = num_q_heads / d.num_kv_heads;
    p.MB = max_blocks;
    p.num_blocks = d.num_blocks;
    p.score_scale = scale * d.k_scale * LOG2E;
    p.out_scale = d.v_scale;
    p.inv_k_scale = pool->inv_k_scale;
    p.inv_v_scale = pool->inv_v_scale;

    if (pl.sp > 0) {
        const bool fp8 = d.kv_dtype == PKV_KV_FP8E4M3;
        const cudaStream_t cs = static_cast<cudaStream_t>(stream);
        const cudaError_t pe = d.head_dim == 128 ? (fp8 ? run_prefix<128, true>(&args, cs) : run_prefix<128, false>(&args, cs))
                                                 : (fp8 ? run_prefix<64, true>(&args, cs) : run_prefix<64, false>(&args, cs));
        if (pe != cudaSuccess) return PKV_ERR_CUDA;
    }
    cudaError_t e = dispatch(d, pl, p.group, true, nullptr, static_cast<cudaStream_t>(stream), &args);
    if (e == cudaErrorInvalidConfiguration) return PKV_ERR_INVALID;
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace

int check_decode_call(const pkv_pool *pool, const void *q, const void *key_cache, const void *value_cache,
                      const int32_t *block_tables, const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                      int32_t max_blocks, float scale, const void *out, const void *workspace,
                      size_t workspace_bytes)
{
    Plan pl;
    return check_call(pool, q, nullptr, nullptr, key_cache, value_cache, block_tables, seq_lens, batch,
                      num_q_heads, max_blocks, scale, out, workspace, workspace_bytes, nullptr, pl);
}

}  // namespace decode
}  // namespace pkv

extern "C" int pkv_paged_attention_decode_ex(pkv_pool *pool, const void *q, const void *key_cache,
                                             const void *value_cache, const int32_t *block_tables,
                                             const int32_t *seq_lens, int32_t batch,
                                             int32_t num_q_heads, int32_t max_blocks, float scale,
                                             void *out, void *workspace, size_t workspace_bytes,
                                             const pkv_decode_opts *opts, void *stream)
{
    return pkv::decode::decode_impl(pool, 1, q, nullptr, nullptr, key_cache, value_cache, block_tables,
                                    seq_lens, batch, num_q_heads, max_blocks, scale, out, workspace,
                                    workspace_bytes, opts, stream);
}

extern "C" int pkv_paged_attention_decode(pkv_pool *pool, const void *q, const void *key_cache,
                                          const void *value_cache, const int32_t *block_tables,
                                          const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                                          int32_t max_blocks, float scale, void *out, void *workspace,
                                          size_t workspace_bytes, void *stream)
{
    return pkv::decode::decode_impl(pool, 1, q, nullptr, nullptr, key_cache, value_cache, block_tables,
                                    seq_lens, batch, num_q_heads, max_blocks, scale, out, workspace,
                                    workspace_bytes, nullptr, stream);
}

extern "C" int pkv_decode_step(pkv_pool *pool, const void *q, const void *k_new, const void *v_new,
                               void *key_cache, void *value_cache, const int32_t *block_tables,
                               const int32_t *seq_lens, int32_t batch, int32_t num_q_heads,
                               int32_t max_blocks, float scale, void *out, void *workspace,
                               size_t workspace_bytes, const pkv_decode_opts *opts, void *stream)
{
    if (!k_new || !v_new) return PKV_ERR_INVALID;
    return pkv::decode::decode_impl(pool, 1, q, k_new, v_new, key_cache, value_cache, block_tables,
                                    seq_lens, batch, num_q_heads, max_blocks, scale, out, workspace,
                                    workspace_bytes, opts, stream);
}

extern "C" int pkv_decode_step_layers(pkv_pool *pool, const void *q, const void *k_new,
                                      const void *v_new, void *key_cache, void *value_cache,
                                      const int32_t *block_tables, const int32_t *seq_lens,
                                      int32_t batch, int32_t num_q_heads, int32_t max_blocks,
                                      float scale, void *out, void *workspace,
                                      size_t workspace_bytes, const pkv_decode_opts *opts,
                                      void *stream)
{
    if (!pool) return PKV_ERR_INVALID;
    return pkv::decode::decode_impl(pool, pool->desc.num_layers, q, k_new, v_new, key_cache,
                                    value_cache, block_tables, seq_lens, batch, num_q_heads,
                                    max_blocks, scale, out, workspace, workspace_bytes, opts, stream);
}

extern "C" int pkv_decode_step_host(pkv_pool *pool, const pkv_host_step *host, const pkv_device_step *dev,
                                    void *key_cache, void *value_cache, int32_t batch, int32_t num_q_heads,
                                    int32_t max_blocks, float scale, void *workspace, size_t workspace_bytes,
                                    const pkv_decode_opts *opts, void *stream)
{
    int st = pkv::check_attached(pool);
    if (st != PKV_OK) return st;
    if (!host || !dev || batch < 0 || num_q_heads < 1 || max_blocks < 1) return PKV_ERR_INVALID;
    if (batch == 0) return PKV_OK;
    const bool append = host->k_new || host->v_new;
    if (!host->q || !host->out || !dev->q || !dev->block_tables || !dev->seq_lens || !dev->out)
        return PKV_ERR_INVALID;
    if (append && (!host->k_new || !host->v_new || !dev->k_new || !dev->v_new)) return PKV_ERR_INVALID;
    const pkv_pool_desc &d = pool->desc;
    const size_t qb = (size_t)batch * num_q_heads * d.head_dim * 2;
    const size_t kb = (size_t)batch * d.num_kv_heads * d.head_dim * 2;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const struct { void *dst; const void *src; size_t n; } in[] = {
        {dev->q, host->q, qb},
        {dev->k_new, host->k_new, append ? kb : 0},
        {dev->v_new, host->v_new, append ? kb : 0},
        {dev->block_tables, host->block_tables, (size_t)batch * max_blocks * 4},
        {dev->seq_lens, host->seq_lens, (size_t)batch * 4},
    };
    if (host->contiguous) {
        // the caller lays the inputs out back to back in one host and one device allocation:
        // one copy (a copy may not span two allocations, so this is never inferred)
        const char *hs = static_cast<const char *>(host->q);
        char *ds = static_cast<char *>(dev->q);
        size_t n = 0;
        for (const auto &c : in) {
            if (!c.n) continue;
            if (c.src != hs + n || c.dst != ds + n) return PKV_ERR_INVALID;
            n += c.n;
        }
        if (cudaMemcpyAsync(ds, hs, n, cudaMemcpyHostToDevice, s) != cudaSuccess) return PKV_ERR_CUDA;
    } else {
        for (const auto &c : in)
            if (c.src && c.n && cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, s) != cudaSuccess)
                return PKV_ERR_CUDA;
    }
    st = append ? pkv_decode_step(pool, dev->q, dev->k_new, dev->v_new, key_cache, value_cache, dev->block_tables,
                                  dev->seq_lens, batch, num_q_heads, max_blocks, scale, dev->out, workspace,
                                  workspace_bytes, opts, stream)
                : pkv_paged_attention_decode_ex(pool, dev->q, key_cache, value_cache, dev->block_tables,
                                                dev->seq_lens, batch, num_q_heads, max_blocks, scale, dev->out,
                                                workspace, workspace_bytes, opts, stream);
    if (st != PKV_OK) return st;
    return cudaMemcpyAsync(host->out, dev->out, qb, cudaMemcpyDeviceToHost, s) == cudaSuccess ? PKV_OK
                                                                                              : PKV_ERR_CUDA;
}
