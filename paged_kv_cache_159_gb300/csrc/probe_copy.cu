// probe_copy.cu -- a plain streaming device-to-device copy.  Its bandwidth, counted as
// bytes read plus bytes written, is the HBM roofline denominator the benchmark measures in
// the same process as the decode kernels.
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

// Grid-stride over 16-byte words, 4 independent loads in flight per thread.
__global__ void __launch_bounds__(512) copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                   size_t n)
{
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 a = __ldcs(src + i);
        const uint4 b = __ldcs(src + i + stride);
        const uint4 c = __ldcs(src + i + 2 * stride);
        const uint4 d = __ldcs(src + i + 3 * stride);
        __stcs(dst + i, a);
        __stcs(dst + i + stride, b);
        __stcs(dst + i + 2 * stride, c);
        __stcs(dst + i + 3 * stride, d);
    }
    for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_probe_copy(void *dst, const void *src, size_t bytes, void *stream)
{
    if (!dst || !src || (bytes & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u) ||
        (reinterpret_cast<uintptr_t>(src) & 15u))
        return PKV_ERR_INVALID;
    if (bytes == 0) return PKV_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PKV_ERR_CUDA;
    const size_t n = bytes / 16;
    size_t blocks = (size_t)sms * 4;
    const size_t need = (n + 512 * 4 - 1) / (512 * 4);
    if (need < blocks) blocks = need > 0 ? need : 1;
    pkv::copy_kernel<<<(unsigned)blocks, 512, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
