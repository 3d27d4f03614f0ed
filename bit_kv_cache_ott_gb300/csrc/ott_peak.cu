// ott_peak.cu -- a plain device-to-device copy kernel, used to measure the
// HBM bandwidth this GPU sustains in the same process as the decode timing
// (the denominator of the decode kernel's roofline fraction).
//
// Each thread moves 16-byte vectors, four in flight per iteration, with
// streaming cache hints (the data is touched once); the grid is a multiple
// of the SM count.
#include "ott_internal.cuh"

namespace {

__global__ void __launch_bounds__(512) k_copy(uint4 *__restrict__ dst, const uint4 *__restrict__ src, long long n) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = __ldcs(src + i + k * stride);
#pragma unroll
        for (int k = 0; k < 4; ++k) __stcs(dst + i + k * stride, v[k]);
    }
    for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

}  // namespace

extern "C" int ott_hbm_copy(void *dst, const void *src, long long bytes, void *stream) {
    if (!dst || !src || bytes < 0 || (bytes & 15) || (reinterpret_cast<uintptr_t>(dst) & 15) ||
        (reinterpret_cast<uintptr_t>(src) & 15))
        return OTT_ERR_INVALID;
    if (bytes == 0) return OTT_OK;
    const char *d = static_cast<const char *>(dst), *s = static_cast<const char *>(src);
    if (d < s + bytes && s < d + bytes) return OTT_ERR_INVALID;   // overlapping ranges
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return OTT_ERR_CUDA;
    k_copy<<<sms * 4, 512, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint4 *>(dst),
                                                                   static_cast<const uint4 *>(src), bytes / 16);
    return cudaGetLastError() == cudaSuccess ? OTT_OK : OTT_ERR_CUDA;
}
