// decode_noalloc.cu -- paged decode attention for callers that must not allocate device
// memory while they run.
//
// Some hosts cannot call cudaMalloc on their hot path: a serving process whose memory
// manager owns every device byte and forbids allocations behind its back, or a latency-
// bound loop where an allocation's implicit device synchronisation, its unpredictable
// cost or its possible failure is unacceptable.  The regular decode entry point asks the
// caller for a workspace buffer; this one needs none.  Its scratch (the split counters and
// the partial softmax states) lives in a fixed array compiled into the library, so every
// GPU that loads libpkv.so holds PKV_NOALLOC_SCRATCH_BYTES of device memory for it until
// the process exits.
//
// The array is shared by every call on a device and keeps what the last call left there.
// Each call clears the counters that must start at zero (an asynchronous memset on the
// caller's stream, which allocates nothing).  Two calls that overlap on the GPU -- on
// different streams, or on one stream from two threads without ordering -- race on the
// array and must not be issued.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

// Host-side device address of g_decode_scratch, looked up once per device with that device
// current.  The symbol name in host code is only a stand-in; a kernel must be given this
// address instead.  A cudaDeviceReset() unloads the module, so the cached address (like every
// pool's error word) is not valid across one.
std::mutex g_mu;
void *g_scratch_addr[64] = {nullptr};

int scratch_address(int device, void **out)
{
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return PKV_ERR_CUDA;
    if (device < 0 || device >= 64 || cur != device) return PKV_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[device]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return PKV_ERR_CUDA;
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_paged_attention_decode_noalloc(pkv_pool *pool, const void *q, const void *key_cache,
                                                  const void *value_cache, const int32_t *block_tables,
                                                  const int32_t *seq_lens, int32_t batch,
                                                  int32_t num_q_heads, int32_t max_blocks, float scale,
                                                  void *out, void *stream)
{
    int st = pkv::check_attached(pool);            // also: the pool's device is the current one
    if (st != PKV_OK) return st;
    if (batch < 0) return PKV_ERR_INVALID;
    if (batch == 0) return PKV_OK;
    const size_t need = pkv_decode_workspace_bytes(pool, batch, num_q_heads, max_blocks, nullptr);
    if (need == 0 || need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_INVALID;
    void *scratch = nullptr;
    st = scratch_address(pool->device, &scratch);       // first call on a device: symbol lookup
    if (st != PKV_OK) return st;
    // every check the decode makes, before anything is queued on the shared array
    st = pkv::decode::check_decode_call(pool, q, key_cache, value_cache, block_tables, seq_lens, batch,
                                        num_q_heads, max_blocks, scale, out, scratch,
                                        (size_t)PKV_NOALLOC_SCRATCH_BYTES);
    if (st != PKV_OK) return st;
    // the per-(sequence, KV head) counters lead the scratch and must start at zero
    const size_t counters = ((size_t)batch * pool->desc.num_kv_heads * 4 + 255) / 256 * 256;
    if (cudaMemsetAsync(scratch, 0, counters, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return pkv_paged_attention_decode_ex(pool, q, key_cache, value_cache, block_tables, seq_lens, batch,
                                         num_q_heads, max_blocks, scale, out, scratch,
                                         (size_t)PKV_NOALLOC_SCRATCH_BYTES, nullptr, stream);
}
