// decode_static.cu -- pd_paged_attention_decode_noalloc: decode attention
// whose partition scratch lives in a fixed array inside this library, so the
// caller never has to allocate device memory for it.
//
// Who needs this: callers that cannot allocate device memory on the call
// path -- engines that reserve all device memory when they start and forbid
// later allocations, or code that must not pay cudaMalloc's implicit
// synchronisation.  They still pass their own inputs and outputs.
//
// The scratch is a file-scope __device__ array of kStaticScratchBytes
// (32 MiB).  Every GPU that loads this library keeps it until the process
// exits.  Host code cannot use the array's name as a device address (on the
// host it names a stand-in object), so the address is looked up once per
// device with cudaGetSymbolAddress, with that device current, the first time
// the entry point runs on it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pd_attn.h"
#include "pd_internal.h"

namespace pd {
namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device).  nullptr with *err set on failure.
void* scratch_for_current_device(cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (*err != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace pd

using namespace pd;

extern "C" {

pd_status pd_paged_attention_decode_noalloc(void* out, const void* q, const void* key_cache,
                                            const void* value_cache,
                                            const int32_t* block_tables,
                                            int max_blocks_per_seq,
                                            const int32_t* context_lens, int B, int H, int Hk,
                                            int D, int S, int NB, int max_context_len,
                                            float scale, pd_dtype dt, int32_t* dev_err,
                                            cudaStream_t stream) {
    if (B < 0 || H < 1 || Hk < 1 || NB < 1 || max_blocks_per_seq < 1 || max_context_len < 0)
        return PD_ERR_INVALID_ARG;
    if (H % Hk != 0) return PD_ERR_INVALID_ARG;
    if (!supported_D(D) || !supported_S(S) || !supported_dt(dt)) return PD_ERR_UNSUPPORTED;
    if (B == 0) return PD_OK;
    if (!out || !q || !key_cache || !value_cache || !block_tables || !context_lens)
        return PD_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
        return PD_ERR_INVALID_ARG;
    if (B > 65535 || int64_t(max_blocks_per_seq) * S > (int64_t(1) << 30) ||
        decode_num_partitions(max_context_len) > 65535)
        return PD_ERR_UNSUPPORTED;
    // The batch's partition scratch must fit the fixed array.
    if (decode_workspace_bytes(B, H, D, max_context_len) > kStaticScratchBytes)
        return PD_ERR_WORKSPACE_TOO_SMALL;
    cudaError_t e = cudaSuccess;
    void* scratch = scratch_for_current_device(&e);
    if (scratch == nullptr) return launch_result(e);
    DecodeArgs a{out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                 B, H, Hk, D, S, NB, max_context_len, scale, scratch, dt, dev_err, stream};
    return launch_decode(a);
}

}  // extern "C"
