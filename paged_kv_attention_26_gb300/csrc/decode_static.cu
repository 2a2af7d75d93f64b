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
// host it names a stand-in object), so the address comes from
// cudaGetSymbolAddress with the calling device current.  Outside stream
// capture the lookup is repeated on every call (a host-side lookup, cheap),
// so an address that changed -- the module loaded again after
// cudaDeviceReset -- is never used stale; during capture the address found
// by the last call outside capture on that device is used, which is why the
// first call on a device must come before any capture.
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
void* g_scratch_ptr[kMaxDevices] = {};   // last address looked up per device

// Device address of the scratch array on the current device.  nullptr with
// *err set on failure.
void* scratch_for_current_device(cudaStream_t stream, cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    *err = cudaStreamIsCapturing(stream, &cap);
    if (*err != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (cap != cudaStreamCaptureStatusNone) {
        // no lookup while capturing: a device whose address was never looked
        // up outside capture is refused
        if (g_scratch_ptr[dev] == nullptr) *err = cudaErrorStreamCaptureUnsupported;
        return g_scratch_ptr[dev];
    }
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
    return p;
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
    // The checks of pd_paged_attention_decode, with the array's size as the
    // workspace size: a batch whose partition scratch does not fit gets
    // PD_ERR_WORKSPACE_TOO_SMALL.  The address is filled in afterwards.
    DecodeArgs a{};
    bool skip = false;
    const pd_status st = decode_prepare(out, q, key_cache, value_cache, nullptr, nullptr, false,
                                        block_tables, max_blocks_per_seq, context_lens, B, H, Hk,
                                        D, S, NB, max_context_len, scale, nullptr,
                                        kStaticScratchBytes, dt, dev_err, stream, &a, &skip, 1,
                                        /*check_workspace_ptr=*/false);
    if (st != PD_OK || skip) return st;
    cudaError_t e = cudaSuccess;
    void* scratch = scratch_for_current_device(stream, &e);
    if (scratch == nullptr) return launch_result(e);
    a.workspace = scratch;
    return launch_decode(a);
}

}  // extern "C"
