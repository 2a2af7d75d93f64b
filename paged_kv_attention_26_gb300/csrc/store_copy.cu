// store_copy.cu -- the two cache-maintenance kernels: storing new tokens into
// their slots (nanoPD page, "模块结构与代码组织": the paged KV store op) and
// copy-on-write block copies (tutorial page "LLM 推理服务引擎深度拆解",
// section 2.3, BlockManager.cow()).  Both are HBM-bound bit copies moved in
// 16-byte vectors; neither looks at the element type.
#include <cuda_runtime.h>

#include "pd_device.cuh"
#include "pd_internal.h"

namespace pd {
namespace {

constexpr int kStoreThreads = 256;

// One (token, kv head) row of D elements = D/8 16-byte vectors per row; each
// thread moves one vector of K and one of V.
__global__ void __launch_bounds__(kStoreThreads)
reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                         uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                         const int64_t* __restrict__ slot_mapping, int T, int Hk, int D,
                         int S, int NB, int64_t key_stride_vec, int64_t value_stride_vec,
                         int32_t* dev_err) {
    // a decode grid launched as our dependent may start its prologue now; it
    // waits for this grid's completion before reading the pools
    pdl_launch_dependents();
    const int vec_per_row = D / 8;
    const int64_t g = int64_t(blockIdx.x) * kStoreThreads + threadIdx.x;
    const int64_t row = g / vec_per_row;
    const int c = int(g % vec_per_row);
    if (row >= int64_t(T) * Hk) return;
    const int64_t n = row / Hk;
    const int h = int(row % Hk);
    // the token's vectors and its slot are independent loads: issue all three
    // before acting on the slot, so they overlap
    const uint4 kv = __ldg(key + n * key_stride_vec + int64_t(h) * vec_per_row + c);
    const uint4 vv = __ldg(value + n * value_stride_vec + int64_t(h) * vec_per_row + c);
    const int64_t slot = __ldg(slot_mapping + n);
    // Launched as a dependent of a block-copy grid, the writes wait for that
    // grid (the slot may lie in a block it is copying); returns at once for
    // an ordinary launch.
    pdl_wait_primary();
    if (slot < 0) return;                       // padding token
    if (slot >= int64_t(NB) * S) {
        if (c == 0) flag_error(dev_err, PD_DEVERR_SLOT_RANGE);
        return;
    }
    const int64_t blk = slot / S, off = slot % S;
    const int64_t dst = ((blk * Hk + h) * S + off) * vec_per_row + c;
    key_cache[dst] = kv;
    value_cache[dst] = vv;
}

// FP8 pools: one thread writes one 16-byte vector of K codes and one of V
// codes (16 values of a (token, kv head) row), reading 32 bytes of 16-bit
// input each.  code = e4m3_rn_satfinite(float(x) * (1 / scale[h])).
template <typename T>
__global__ void __launch_bounds__(kStoreThreads)
reshape_and_cache_fp8_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                             uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                             const int64_t* __restrict__ slot_mapping, int T_, int Hk, int D,
                             int S, int NB, int64_t key_stride_vec, int64_t value_stride_vec,
                             const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                             int32_t* dev_err) {
    using E = Elem<T>;
    pdl_launch_dependents();
    const int vec8 = D / 16;                    // 16-byte FP8 vectors per row
    const int64_t g = int64_t(blockIdx.x) * kStoreThreads + threadIdx.x;
    const int64_t row = g / vec8;
    const int c = int(g % vec8);
    if (row >= int64_t(T_) * Hk) return;
    const int64_t n = row / Hk;
    const int h = int(row % Hk);
    const int64_t src_k = n * key_stride_vec + int64_t(h) * (D / 8) + 2 * c;
    const int64_t src_v = n * value_stride_vec + int64_t(h) * (D / 8) + 2 * c;
    const uint4 k0 = __ldg(key + src_k), k1 = __ldg(key + src_k + 1);
    const uint4 v0 = __ldg(value + src_v), v1 = __ldg(value + src_v + 1);
    const int64_t slot = __ldg(slot_mapping + n);
    pdl_wait_primary();                         // as in the 16-bit store
    if (slot < 0) return;                       // padding token
    if (slot >= int64_t(NB) * S) {
        if (c == 0) flag_error(dev_err, PD_DEVERR_SLOT_RANGE);
        return;
    }
    const float kinv = __fdiv_rn(1.0f, __ldg(k_scale + h));
    const float vinv = __fdiv_rn(1.0f, __ldg(v_scale + h));
    auto quant = [](const uint4& a, const uint4& b, float inv) {
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 x0 = E::unpack2(w[2 * j]), x1 = E::unpack2(w[2 * j + 1]);
            uint16_t lo, hi;
            // cvt packs its first source into the upper byte
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
                : "=h"(lo) : "f"(__fmul_rn(x0.y, inv)), "f"(__fmul_rn(x0.x, inv)));
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
                : "=h"(hi) : "f"(__fmul_rn(x1.y, inv)), "f"(__fmul_rn(x1.x, inv)));
            o[j] = uint32_t(lo) | (uint32_t(hi) << 16);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    };
    const int64_t blk = slot / S, off = slot % S;
    const int64_t dst = ((blk * Hk + h) * S + off) * vec8 + c;
    key_cache[dst] = quant(k0, k1, kinv);
    value_cache[dst] = quant(v0, v1, vinv);
}

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

// blockIdx.x = pair, blockIdx.y = layer, blockIdx.z = 0 for K, 1 for V.
// The whole block (Hk * S * D elements) is contiguous in the pool.  The pools
// come from the device pointer arrays, or (key_caches == nullptr, one layer)
// are the pools k_pool / v_pool themselves.
__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(void* const* __restrict__ key_caches, void* const* __restrict__ value_caches,
                   void* k_pool, void* v_pool, const int64_t* __restrict__ block_mapping, int NB,
                   int64_t block_vecs, int32_t* dev_err) {
    // a store grid launched as our dependent may start now; it waits for
    // this grid before it writes
    pdl_launch_dependents();
    const int64_t src = __ldg(block_mapping + 2 * blockIdx.x);
    const int64_t dst = __ldg(block_mapping + 2 * blockIdx.x + 1);
    if (src < 0 || src >= NB || dst < 0 || dst >= NB) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
            flag_error(dev_err, PD_DEVERR_BLOCK_RANGE);
        return;
    }
    uint4* pool;
    if (key_caches != nullptr) {
        void* const* pools = blockIdx.z == 0 ? key_caches : value_caches;
        pool = static_cast<uint4*>(pools[blockIdx.y]);
    } else {
        pool = static_cast<uint4*>(blockIdx.z == 0 ? k_pool : v_pool);
    }
    if (reinterpret_cast<uintptr_t>(pool) & 15u) {     // pointer table is device data
        if (threadIdx.x == 0) flag_error(dev_err, PD_DEVERR_BLOCK_RANGE);
        return;
    }
    const uint4* s = pool + src * block_vecs;
    uint4* d = pool + dst * block_vecs;
    for (int64_t base = threadIdx.x; base < block_vecs; base += kCopyThreads * kCopyUnroll) {
        uint4 r[kCopyUnroll];
#pragma unroll
        for (int k = 0; k < kCopyUnroll; ++k) {
            const int64_t i = base + int64_t(k) * kCopyThreads;
            if (i < block_vecs) r[k] = s[i];
        }
#pragma unroll
        for (int k = 0; k < kCopyUnroll; ++k) {
            const int64_t i = base + int64_t(k) * kCopyThreads;
            if (i < block_vecs) d[i] = r[k];
        }
    }
}

}  // namespace

pd_status launch_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                   void* value_cache, const int64_t* slot_mapping, int T,
                                   int Hk, int D, int S, int NB, int64_t key_stride_tok,
                                   int64_t value_stride_tok, int32_t* dev_err,
                                   cudaStream_t stream, bool pdl) {
    if (T == 0) return PD_OK;
    const int64_t threads = int64_t(T) * Hk * (D / 8);
    const int64_t blocks = (threads + kStoreThreads - 1) / kStoreThreads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(kStoreThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return launch_result(cudaLaunchKernelEx(
        &cfg, reshape_and_cache_kernel, static_cast<const uint4*>(key),
        static_cast<const uint4*>(value), static_cast<uint4*>(key_cache),
        static_cast<uint4*>(value_cache), slot_mapping, T, Hk, D, S, NB, key_stride_tok / 8,
        value_stride_tok / 8, dev_err));
}

pd_status launch_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache,
                                       void* value_cache, const int64_t* slot_mapping, int T,
                                       int Hk, int D, int S, int NB, int64_t key_stride_tok,
                                       int64_t value_stride_tok, const float* k_scale,
                                       const float* v_scale, pd_dtype in_dt, int32_t* dev_err,
                                       cudaStream_t stream) {
    if (T == 0) return PD_OK;
    const int64_t threads = int64_t(T) * Hk * (D / 16);
    const int64_t blocks = (threads + kStoreThreads - 1) / kStoreThreads;
    auto k = in_dt == PD_BF16 ? reshape_and_cache_fp8_kernel<__nv_bfloat16>
                              : reshape_and_cache_fp8_kernel<__half>;
    k<<<unsigned(blocks), kStoreThreads, 0, stream>>>(
        static_cast<const uint4*>(key), static_cast<const uint4*>(value),
        static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache), slot_mapping, T, Hk, D,
        S, NB, key_stride_tok / 8, value_stride_tok / 8, k_scale, v_scale, dev_err);
    return launch_result(cudaGetLastError());
}

pd_status launch_copy_blocks(void* const* key_caches, void* const* value_caches, int L,
                             const int64_t* block_mapping, int npairs, int Hk, int D, int S,
                             int NB, int esize, int32_t* dev_err, cudaStream_t stream,
                             void* k_pool, void* v_pool) {
    if (npairs == 0 || L == 0) return PD_OK;
    const int64_t block_vecs = int64_t(Hk) * S * D * esize / 16;
    dim3 grid(unsigned(npairs), unsigned(L), 2);
    copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(key_caches, value_caches, k_pool,
                                                          v_pool, block_mapping, NB, block_vecs,
                                                          dev_err);
    return launch_result(cudaGetLastError());
}

}  // namespace pd
