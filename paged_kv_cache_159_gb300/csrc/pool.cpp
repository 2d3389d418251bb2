// pool.cpp -- host side of the paged KV pool: block allocator, block-table builder, slot
// mapping, device binding and status strings.
//
// Block lifecycle follows "理解 KV Cache：Attention、P/D 分离与 vLLM 的页式显存管理"
// (steinslab.io) §3.5: the scheduler takes physical blocks from a free pool when a request
// arrives or grows, the attention kernels use them through the block table, and they go
// back to the pool when the request finishes or is preempted.  Shared prefix blocks are
// stored once and referenced by many tables ("KV Cache 与推理优化", PagedAttention
// section), which is why blocks carry reference counts.  Slot addressing is §3.3 of the
// steinslab.io page.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime_api.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>

#include "pkv_internal.h"

namespace {

bool valid_desc(const pkv_pool_desc *d)
{
    if (!d) return false;
    if (d->num_blocks < 1 || d->block_size != 16 || d->num_kv_heads < 1) return false;
    if (d->head_dim != 64 && d->head_dim != 128) return false;
    if (d->kv_dtype != PKV_KV_BF16 && d->kv_dtype != PKV_KV_FP8E4M3) return false;
    if (d->kv_dtype == PKV_KV_FP8E4M3) {
        if (!(d->k_scale > 0.0f) || !std::isfinite(d->k_scale)) return false;
        if (!(d->v_scale > 0.0f) || !std::isfinite(d->v_scale)) return false;
    }
    // the slot count must fit in int32, and so must the (layer, block, head) tile index the
    // kernels use
    if ((int64_t)d->num_blocks * d->block_size > INT32_MAX) return false;
    const int64_t layers = d->num_layers == 0 ? 1 : d->num_layers;
    if (layers < 1 || layers > 4096) return false;
    if (layers * d->num_blocks * d->num_kv_heads >= ((int64_t)1 << 31)) return false;
    return true;
}

}  // namespace

namespace pkv {

namespace {
std::atomic<int> g_test_expire{PKV_TEST_EXPIRE_NONE};
}

int test_expire() { return g_test_expire.load(std::memory_order_relaxed); }

bool encode_tiled(CUtensorMap *map, const void *ptr, CUtensorMapDataType type, int rank, const uint64_t *dims,
                  const uint64_t *strides, const uint32_t *box, CUtensorMapSwizzle swizzle)
{
    // the driver's encoder, looked up once through the runtime (no link against libcuda)
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    if (!enc || rank < 3 || rank > 4) return false;
    cuuint64_t d[4], st[3];
    cuuint32_t b[4], es[4];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    return enc(map, type, (cuuint32_t)rank, const_cast<void *>(ptr), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int check_attached(const pkv_pool *pool)
{
    if (!pool || !pool->d_err || pool->device < 0) return PKV_ERR_INVALID;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return PKV_ERR_CUDA;
    if (cur != pool->device) return PKV_ERR_INVALID;
    return PKV_OK;
}

}  // namespace pkv

extern "C" {

int pkv_pool_create(const pkv_pool_desc *desc, const int32_t *free_order, pkv_pool **out)
{
    if (!out || !valid_desc(desc)) return PKV_ERR_INVALID;
    *out = nullptr;
    pkv_pool *p = new (std::nothrow) pkv_pool();
    if (!p) return PKV_ERR_OOM;
    p->desc = *desc;
    if (p->desc.num_layers == 0) p->desc.num_layers = 1;
    const int32_t nb = desc->num_blocks;
    p->refcount.assign((size_t)nb, 0);
    if (free_order) {
        std::vector<char> seen((size_t)nb, 0);
        for (int32_t i = 0; i < nb; ++i) {
            int32_t id = free_order[i];
            if (id < 0 || id >= nb || seen[(size_t)id]) {
                delete p;
                return PKV_ERR_INVALID;
            }
            seen[(size_t)id] = 1;
            p->free_list.push_back(id);
        }
    } else {
        for (int32_t i = 0; i < nb; ++i) p->free_list.push_back(i);
    }
    if (desc->kv_dtype == PKV_KV_FP8E4M3) {
        p->inv_k_scale = 1.0f / desc->k_scale;
        p->inv_v_scale = 1.0f / desc->v_scale;
    } else {
        p->desc.k_scale = 1.0f;
        p->desc.v_scale = 1.0f;
    }
    *out = p;
    return PKV_OK;
}

int pkv_pool_destroy(pkv_pool *pool)
{
    if (!pool) return PKV_ERR_INVALID;
    int st = PKV_OK;
    if (pool->d_err) {
        int prev = -1;
        cudaGetDevice(&prev);
        if (prev != pool->device) cudaSetDevice(pool->device);
        if (cudaFree(pool->d_err) != cudaSuccess) st = PKV_ERR_CUDA;
        if (prev >= 0 && prev != pool->device) cudaSetDevice(prev);
    }
    pkv::destroy_prefix_cache(pool);
    delete pool;
    return st;
}

int pkv_pool_get_desc(const pkv_pool *pool, pkv_pool_desc *out)
{
    if (!pool || !out) return PKV_ERR_INVALID;
    *out = pool->desc;
    return PKV_OK;
}

size_t pkv_pool_layer_bytes(const pkv_pool *pool)
{
    if (!pool) return 0;
    const pkv_pool_desc &d = pool->desc;
    return (size_t)d.num_blocks * d.num_kv_heads * d.block_size * d.head_dim * pkv::elem_bytes(d);
}

int pkv_pool_num_free(const pkv_pool *pool, int32_t *out)
{
    if (!pool || !out) return PKV_ERR_INVALID;
    *out = (int32_t)pool->free_list.size();
    return PKV_OK;
}

int pkv_pool_refcount(const pkv_pool *pool, int32_t block_id, int32_t *out)
{
    if (!pool || !out || block_id < 0 || block_id >= pool->desc.num_blocks) return PKV_ERR_INVALID;
    *out = pool->refcount[(size_t)block_id];
    return PKV_OK;
}

int pkv_pool_alloc(pkv_pool *pool, int32_t n, int32_t *ids_out)
{
    if (!pool || n < 0 || (n > 0 && !ids_out)) return PKV_ERR_INVALID;
    if ((size_t)n > pool->free_list.size()) return PKV_ERR_OOM;
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = pool->free_list.front();
        pool->free_list.pop_front();
        pool->refcount[(size_t)id] = 1;
        ids_out[i] = id;
    }
    return PKV_OK;
}

int pkv_pool_share(pkv_pool *pool, const int32_t *ids, int32_t n)
{
    if (!pool || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID;
    for (int32_t i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= pool->desc.num_blocks || pool->refcount[(size_t)ids[i]] < 1)
            return PKV_ERR_INVALID;
    for (int32_t i = 0; i < n; ++i) pool->refcount[(size_t)ids[i]] += 1;
    return PKV_OK;
}

int pkv_pool_free(pkv_pool *pool, const int32_t *ids, int32_t n)
{
    if (!pool || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID;
    // validate first, counting repeats, so that a bad list changes nothing
    std::vector<int32_t> drop;
    drop.reserve((size_t)n);
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = ids[i];
        if (id < 0 || id >= pool->desc.num_blocks) return PKV_ERR_INVALID;
        int32_t repeats = 0;
        for (int32_t j = 0; j < i; ++j) repeats += (ids[j] == id);
        if (pool->refcount[(size_t)id] <= repeats) return PKV_ERR_INVALID;
    }
    for (int32_t i = 0; i < n; ++i) {
        int32_t id = ids[i];
        if (--pool->refcount[(size_t)id] == 0) pool->free_list.push_back(id);
    }
    return PKV_OK;
}

int pkv_build_block_tables(pkv_pool *pool, const int32_t *seq_lens, int32_t batch,
                           int32_t max_blocks, const int32_t *prefix_ids, int32_t num_prefix,
                           int32_t *tables_out)
{
    if (!pool || batch < 0 || max_blocks < 1 || num_prefix < 0) return PKV_ERR_INVALID;
    if ((batch > 0 && (!seq_lens || !tables_out)) || (num_prefix > 0 && !prefix_ids))
        return PKV_ERR_INVALID;
    const int32_t bs = pool->desc.block_size;
    for (int32_t p = 0; p < num_prefix; ++p)
        if (prefix_ids[p] < 0 || prefix_ids[p] >= pool->desc.num_blocks ||
            pool->refcount[(size_t)prefix_ids[p]] < 1)
            return PKV_ERR_INVALID;
    for (int32_t b = 0; b < batch; ++b) {
        if (seq_lens[b] < 1) return PKV_ERR_INVALID;
        int64_t nblk = ((int64_t)seq_lens[b] + bs - 1) / bs;
        if (nblk > max_blocks) return PKV_ERR_INVALID;
    }
    std::vector<int32_t> taken, shared;
    for (int32_t b = 0; b < batch; ++b) {
        int32_t nblk = (int32_t)(((int64_t)seq_lens[b] + bs - 1) / bs);
        int32_t nshared = nblk < num_prefix ? nblk : num_prefix;
        int32_t *row = tables_out + (int64_t)b * max_blocks;
        for (int32_t j = 0; j < nshared; ++j) {
            row[j] = prefix_ids[j];
            pool->refcount[(size_t)prefix_ids[j]] += 1;
            shared.push_back(prefix_ids[j]);
        }
        for (int32_t j = nshared; j < nblk; ++j) {
            if (pool->free_list.empty()) {   // undo this call and report OOM
                for (int32_t id : shared) pool->refcount[(size_t)id] -= 1;
                for (auto it = taken.rbegin(); it != taken.rend(); ++it) {
                    pool->refcount[(size_t)*it] = 0;
                    pool->free_list.push_front(*it);
                }
                return PKV_ERR_OOM;
            }
            int32_t id = pool->free_list.front();
            pool->free_list.pop_front();
            pool->refcount[(size_t)id] = 1;
            taken.push_back(id);
            row[j] = id;
        }
        for (int32_t j = nblk; j < max_blocks; ++j) row[j] = -1;
    }
    return PKV_OK;
}

// Copy-on-write before an append ("KV Cache 与推理优化", PagedAttention section: a shared
// prefix block is stored once; a request that diverges gets its own copy first).  Sequences
// are taken in batch order, so the holders of a shared block that write it get copies one
// after another until a single reference is left, and that last holder writes in place.
int pkv_cow_prepare(pkv_pool *pool, int32_t *tables, const int32_t *seq_lens, int32_t batch,
                    int32_t max_blocks, int32_t *src_out, int32_t *dst_out, int32_t *num_copies)
{
    if (!pool || batch < 0 || max_blocks < 1 || !num_copies) return PKV_ERR_INVALID;
    if (batch > 0 && (!tables || !seq_lens || !src_out || !dst_out)) return PKV_ERR_INVALID;
    const int32_t bs = pool->desc.block_size;
    // validate first: nothing changes on INVALID
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t L = seq_lens[b];
        if (L < 1 || (L - 1) / bs >= max_blocks) return PKV_ERR_INVALID;
        const int32_t e = tables[(size_t)b * max_blocks + (L - 1) / bs];
        if (e < 0 || e >= pool->desc.num_blocks || pool->refcount[(size_t)e] < 1) return PKV_ERR_INVALID;
    }
    int32_t n = 0;
    for (int32_t b = 0; b < batch; ++b) {
        int32_t &entry = tables[(size_t)b * max_blocks + (seq_lens[b] - 1) / bs];
        const int32_t shared = entry;
        if (pool->refcount[(size_t)shared] == 1) continue;    // private already
        if (pool->free_list.empty()) {
            // undo in reverse: fresh blocks go back to the front of the free list in the
            // order they were taken, references and table entries are restored
            for (int32_t i = n - 1; i >= 0; --i) {
                pool->refcount[(size_t)dst_out[i]] = 0;
                pool->free_list.push_front(dst_out[i]);
                pool->refcount[(size_t)src_out[i]] += 1;
            }
            for (int32_t bb = 0, i = 0; bb < b && i < n; ++bb) {
                int32_t &e2 = tables[(size_t)bb * max_blocks + (seq_lens[bb] - 1) / bs];
                if (e2 == dst_out[i]) e2 = src_out[i++];
            }
            *num_copies = 0;
            return PKV_ERR_OOM;
        }
        const int32_t fresh = pool->free_list.front();
        pool->free_list.pop_front();
        pool->refcount[(size_t)fresh] = 1;
        pool->refcount[(size_t)shared] -= 1;                  // still >= 1: others hold it
        entry = fresh;
        src_out[n] = shared;
        dst_out[n] = fresh;
        ++n;
    }
    *num_copies = n;
    return PKV_OK;
}

int pkv_slot_mapping_chunks(const int32_t *tables, const int32_t *seq_lens, const int32_t *cu_q,
                            int32_t batch, int32_t max_blocks, int32_t block_size, int64_t *slots_out)
{
    if (batch < 0 || max_blocks < 1 || block_size < 1) return PKV_ERR_INVALID;
    if (batch > 0 && (!tables || !seq_lens || !cu_q || !slots_out)) return PKV_ERR_INVALID;
    if (batch > 0 && cu_q[0] != 0) return PKV_ERR_INVALID;
    for (int32_t b = 0; b < batch; ++b) {           // validate first
        const int64_t P = (int64_t)cu_q[b + 1] - cu_q[b], L = seq_lens[b];
        if (P < 0 || P > L || L < 1 || L > (int64_t)max_blocks * block_size) return PKV_ERR_INVALID;
        for (int64_t pos = L - P; pos < L; ++pos)
            if (tables[(int64_t)b * max_blocks + pos / block_size] < 0) return PKV_ERR_INVALID;
    }
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t P = (int64_t)cu_q[b + 1] - cu_q[b], L = seq_lens[b];
        int64_t *out = slots_out + cu_q[b];
        for (int64_t i = 0; i < P; ++i) {
            const int64_t pos = L - P + i;
            out[i] = (int64_t)tables[(int64_t)b * max_blocks + pos / block_size] * block_size + pos % block_size;
        }
    }
    return PKV_OK;
}

int pkv_slot_mapping(const int32_t *tables, const int32_t *seq_lens, int32_t batch,
                     int32_t max_blocks, int32_t block_size, int64_t *slots_out)
{
    if (batch < 0 || max_blocks < 1 || block_size < 1) return PKV_ERR_INVALID;
    if (batch > 0 && (!tables || !seq_lens || !slots_out)) return PKV_ERR_INVALID;
    for (int32_t b = 0; b < batch; ++b) {
        int64_t pos = (int64_t)seq_lens[b] - 1;
        if (pos < 0 || pos >= (int64_t)max_blocks * block_size) return PKV_ERR_INVALID;
        int32_t phys = tables[(int64_t)b * max_blocks + pos / block_size];
        if (phys < 0) return PKV_ERR_INVALID;
        slots_out[b] = (int64_t)phys * block_size + pos % block_size;
    }
    return PKV_OK;
}

int pkv_slot_mapping_all(const int32_t *tables, const int32_t *seq_lens, int32_t batch,
                         int32_t max_blocks, int32_t block_size, int64_t *slots_out)
{
    if (batch < 0 || max_blocks < 1 || block_size < 1) return PKV_ERR_INVALID;
    if (batch > 0 && (!tables || !seq_lens || !slots_out)) return PKV_ERR_INVALID;
    for (int32_t b = 0; b < batch; ++b) {
        const int64_t L = seq_lens[b];
        if (L < 1 || L > (int64_t)max_blocks * block_size) return PKV_ERR_INVALID;
        const int32_t *row = tables + (int64_t)b * max_blocks;
        for (int64_t j = 0; j < (L + block_size - 1) / block_size; ++j)
            if (row[j] < 0) return PKV_ERR_INVALID;
    }
    int64_t k = 0;
    for (int32_t b = 0; b < batch; ++b) {
        const int32_t *row = tables + (int64_t)b * max_blocks;
        for (int64_t pos = 0; pos < seq_lens[b]; ++pos)
            slots_out[k++] = (int64_t)row[pos / block_size] * block_size + pos % block_size;
    }
    return PKV_OK;
}

int pkv_pool_attach_device(pkv_pool *pool, int device)
{
    if (!pool || device < 0) return PKV_ERR_INVALID;
    if (pool->d_err) return pool->device == device ? PKV_OK : PKV_ERR_INVALID;
    int n = 0;
    if (cudaGetDeviceCount(&n) != cudaSuccess || device >= n) return PKV_ERR_CUDA;
    int prev = -1;
    cudaGetDevice(&prev);
    if (cudaSetDevice(device) != cudaSuccess) return PKV_ERR_CUDA;
    void *w = nullptr;
    int st = PKV_OK;
    if (cudaMalloc(&w, 256) != cudaSuccess || cudaMemset(w, 0, 256) != cudaSuccess) {
        if (w) cudaFree(w);
        st = PKV_ERR_CUDA;
    } else {
        pool->d_err = static_cast<uint32_t *>(w);
        pool->device = device;
    }
    if (prev >= 0 && prev != device) cudaSetDevice(prev);
    return st;
}

int pkv_get_device_error(pkv_pool *pool, void *stream, uint32_t *bits_out)
{
    int st = pkv::check_attached(pool);
    if (st != PKV_OK) return st;
    if (!bits_out) return PKV_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t bits = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaMemcpy(&bits, pool->d_err, sizeof bits, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaMemset(pool->d_err, 0, sizeof bits) != cudaSuccess) return PKV_ERR_CUDA;
    *bits_out = bits;
    if (bits == 0) return PKV_OK;
    return (bits & PKV_DEVERR_TIMEOUT) ? PKV_ERR_TIMEOUT : PKV_ERR_DEVICE;
}

int pkv_device_sm_count(int device, int32_t *out)
{
    if (!out) return PKV_ERR_INVALID;
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return PKV_ERR_CUDA;
    *out = v;
    return PKV_OK;
}

int pkv_test_expire_waits(int32_t which)
{
    if (which != PKV_TEST_EXPIRE_NONE && which != PKV_TEST_EXPIRE_DECODE && which != PKV_TEST_EXPIRE_PREFILL)
        return PKV_ERR_INVALID;
    pkv::g_test_expire.store(which, std::memory_order_relaxed);
    return PKV_OK;
}

const char *pkv_status_string(int status)
{
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_INVALID: return "invalid argument";
    case PKV_ERR_OOM: return "pool out of free blocks";
    case PKV_ERR_DEVICE: return "device-side error flag set";
    case PKV_ERR_TIMEOUT: return "device pipeline wait timed out";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
    }
}

}  // extern "C"
