// copy_bytes.cu -- byte copies between any two device-accessible buffers
// (device memory, or pinned host memory mapped into the device's address
// space) by the SMs: many 16-byte loads in flight at once, so a transfer of a
// few hundred KB between pinned host memory and the device is limited by the
// host link's bandwidth rather than by a copy engine's per-transfer latency.
#include <cuda_runtime.h>

#include <algorithm>

#include "pd_device.cuh"
#include "pd_internal.h"

namespace pd {
namespace {

constexpr int kCopyBytesThreads = 256;

int sms_of(int dev) {
    static int counts[64] = {};
    if (dev < 0 || dev >= 64) return 148;
    if (counts[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        counts[dev] = n;
    }
    return counts[dev];
}
constexpr int kCopyBytesUnroll = 4;     // 16-byte vectors per thread per pass

__global__ void __launch_bounds__(kCopyBytesThreads)
copy_bytes_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int64_t nvec) {
    const int64_t stride = int64_t(gridDim.x) * kCopyBytesThreads * kCopyBytesUnroll;
    for (int64_t base = int64_t(blockIdx.x) * kCopyBytesThreads * kCopyBytesUnroll + threadIdx.x;
         base < nvec; base += stride) {
        uint4 r[kCopyBytesUnroll];
#pragma unroll
        for (int k = 0; k < kCopyBytesUnroll; ++k) {
            const int64_t i = base + int64_t(k) * kCopyBytesThreads;
            if (i < nvec) r[k] = src[i];
        }
#pragma unroll
        for (int k = 0; k < kCopyBytesUnroll; ++k) {
            const int64_t i = base + int64_t(k) * kCopyBytesThreads;
            if (i < nvec) dst[i] = r[k];
        }
    }
}

}  // namespace

pd_status launch_copy_bytes(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
    const int64_t nvec = int64_t(bytes / 16);
    if (nvec == 0) return PD_OK;
    const int64_t per_cta = int64_t(kCopyBytesThreads) * kCopyBytesUnroll;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return launch_result(e);
    // enough CTAs for every vector in one pass, at most four per SM
    const int64_t cap = 4LL * sms_of(dev);
    const unsigned grid = unsigned(std::min<int64_t>((nvec + per_cta - 1) / per_cta, cap));
    copy_bytes_kernel<<<grid, kCopyBytesThreads, 0, stream>>>(static_cast<uint4*>(dst),
                                                             static_cast<const uint4*>(src), nvec);
    return launch_result(cudaGetLastError());
}

}  // namespace pd
