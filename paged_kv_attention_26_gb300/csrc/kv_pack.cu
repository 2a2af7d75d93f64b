// kv_pack.cu -- KV hand-over between a prefill worker and a decode worker
// (nanoPD page, "异步KV传输": the KV of a finished prefill moves to the decode
// side on a stream of its own; essay page "LLM推理PD分离架构深度工程实践",
// section 3.1: layer-by-layer transfer, so the receiver can start on the
// first layers while later ones are still in flight).
//
// pack gathers whole blocks of every layer into one contiguous staging buffer,
// layer-major:  staging[l][0 = K, 1 = V][i][Hk][S][D] = pool_l[block_ids[i]],
// so layer l is one run that a copy engine or a peer can move on its own;
// unpack scatters such a buffer into blocks of another pool.  A (block, layer,
// K or V) slab of Hk*S*D elements is contiguous on both sides, so each CTA
// streams one slab in 16-byte vectors.  Bit copies, HBM-bound.
#include <cuda_runtime.h>

#include "pd_device.cuh"
#include "pd_internal.h"

namespace pd {
namespace {

constexpr int kPackThreads = 256;
constexpr int kPackUnroll = 4;

// blockIdx.x = i (index into block_ids), blockIdx.y = layer, blockIdx.z = K / V.
template <bool kUnpack>
__global__ void __launch_bounds__(kPackThreads)
kv_pack_kernel(uint4* __restrict__ staging, void* const* __restrict__ key_caches,
               void* const* __restrict__ value_caches, const int32_t* __restrict__ block_ids,
               int nblk, int NB, int64_t slab_vecs, int32_t* dev_err) {
    const int blk = __ldg(block_ids + blockIdx.x);
    if (blk < 0 || blk >= NB) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
            flag_error(dev_err, PD_DEVERR_BLOCK_RANGE);
        return;
    }
    void* const* pools = blockIdx.z == 0 ? key_caches : value_caches;
    uint4* pool = static_cast<uint4*>(pools[blockIdx.y]);
    if (reinterpret_cast<uintptr_t>(pool) & 15u) {     // pointer table is device data
        if (threadIdx.x == 0) flag_error(dev_err, PD_DEVERR_BLOCK_RANGE);
        return;
    }
    uint4* p = pool + int64_t(blk) * slab_vecs;
    uint4* g = staging + ((int64_t(blockIdx.y) * 2 + blockIdx.z) * nblk + blockIdx.x) * slab_vecs;
    const uint4* src = kUnpack ? g : p;
    uint4* dst = kUnpack ? p : g;
    for (int64_t base = threadIdx.x; base < slab_vecs; base += kPackThreads * kPackUnroll) {
        uint4 r[kPackUnroll];
#pragma unroll
        for (int k = 0; k < kPackUnroll; ++k) {
            const int64_t i = base + int64_t(k) * kPackThreads;
            if (i < slab_vecs) r[k] = src[i];
        }
#pragma unroll
        for (int k = 0; k < kPackUnroll; ++k) {
            const int64_t i = base + int64_t(k) * kPackThreads;
            if (i < slab_vecs) dst[i] = r[k];
        }
    }
}

}  // namespace

pd_status launch_kv_pack(bool unpack, void* staging, void* const* key_caches,
                         void* const* value_caches, int L, const int32_t* block_ids, int nblk,
                         int Hk, int D, int S, int NB, int esize, int32_t* dev_err,
                         cudaStream_t stream) {
    if (nblk == 0 || L == 0) return PD_OK;
    const int64_t slab_vecs = int64_t(Hk) * S * D * esize / 16;
    dim3 grid(unsigned(nblk), unsigned(L), 2);
    if (unpack)
        kv_pack_kernel<true><<<grid, kPackThreads, 0, stream>>>(
            static_cast<uint4*>(staging), key_caches, value_caches, block_ids, nblk, NB,
            slab_vecs, dev_err);
    else
        kv_pack_kernel<false><<<grid, kPackThreads, 0, stream>>>(
            static_cast<uint4*>(staging), key_caches, value_caches, block_ids, nblk, NB,
            slab_vecs, dev_err);
    return launch_result(cudaGetLastError());
}

}  // namespace pd
