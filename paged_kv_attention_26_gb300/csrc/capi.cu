// capi.cu -- the extern "C" entry points of pd_attn.h: argument validation,
// status codes and launch accounting around the per-op launchers.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "pd_attn.h"
#include "pd_internal.h"

namespace pd {
namespace {
thread_local int g_last_cuda_error = 0;
std::atomic<uint64_t> g_launches{0};
}  // namespace

pd_status launch_result(cudaError_t e) {
    if (e == cudaSuccess) {
        count_launch();
        return PD_OK;
    }
    g_last_cuda_error = int(e);
    return PD_ERR_CUDA;
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Checks the decode arguments and fills *a; *skip is set when there is
// nothing to launch (B == 0).  check_workspace_ptr == false skips the checks
// of the workspace pointer (not its size): the caller supplies the address
// after validation (the library's own scratch array).
pd_status decode_prepare(void* out, const void* q, const void* key_cache,
                         const void* value_cache, const float* k_scale, const float* v_scale,
                         bool fp8, const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int B, int H, int Hk, int D, int S, int NB,
                         int max_context_len, float scale, void* workspace,
                         size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                         cudaStream_t stream, DecodeArgs* a, bool* skip, int nq,
                         bool check_workspace_ptr, const SharedGroups* grp) {
    *skip = false;
    if (nq < 1 || nq > 8) return PD_ERR_UNSUPPORTED;
    if (grp && (grp->max_group < 1 || grp->max_group > 32 || grp->n_groups < 1 ||
                grp->n_groups > 65535 || nq != 1))
        return PD_ERR_UNSUPPORTED;
    if (B < 0 || H < 1 || Hk < 1 || NB < 1 || max_blocks_per_seq < 1 || max_context_len < 0)
        return PD_ERR_INVALID_ARG;
    if (H % Hk != 0) return PD_ERR_INVALID_ARG;
    if (!supported_D(D) || !supported_S(S) || !supported_dt(dt)) return PD_ERR_UNSUPPORTED;
    if (B == 0) {
        *skip = true;
        return PD_OK;
    }
    if (!out || !q || !key_cache || !value_cache || !block_tables || !context_lens)
        return PD_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
        return PD_ERR_INVALID_ARG;
    if (int64_t(B) * nq > 65535 || int64_t(max_blocks_per_seq) * S > (int64_t(1) << 30) ||
        decode_num_partitions(max_context_len) > 65535)
        return PD_ERR_UNSUPPORTED;
    if (grp && (!grp->start || !grp->shared)) return PD_ERR_INVALID_ARG;
    const size_t need = grp ? decode_shared_workspace_bytes(grp->n_groups, grp->max_group, H,
                                                            Hk, D)
                            : decode_workspace_bytes(B * nq, H, D, max_context_len);
    if (need > 0) {
        if (check_workspace_ptr &&
            (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
            return PD_ERR_INVALID_ARG;
        if (workspace_bytes < need) return PD_ERR_WORKSPACE_TOO_SMALL;
    }
    if (fp8 && (!k_scale || !v_scale)) return PD_ERR_INVALID_ARG;
    *a = DecodeArgs{out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                    context_lens, B, H, Hk, D, S, NB, max_context_len, scale, workspace, dt,
                    dev_err, stream};
    a->fp8 = fp8;
    a->k_scale = k_scale;
    a->v_scale = v_scale;
    a->nq = nq;
    if (grp) {
        a->grp_start = grp->start;
        a->grp_shared = grp->shared;
        a->n_groups = grp->n_groups;
        a->max_group = grp->max_group;
    }
    return PD_OK;
}

}  // namespace pd

using namespace pd;

extern "C" {

const char* pd_status_string(pd_status s) {
    switch (s) {
        case PD_OK: return "ok";
        case PD_ERR_INVALID_ARG: return "invalid argument";
        case PD_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PD_ERR_CUDA: return "CUDA launch error (see pd_last_cuda_error)";
        case PD_ERR_NO_FREE_BLOCK: return "no free block in the pool";
        case PD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case PD_ERR_NOT_FOUND: return "unknown sequence id";
    }
    return "unknown status";
}

int pd_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t pd_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

// Argument checks of the store (16-bit or FP8 pools); *skip when T == 0.
static pd_status store_check(const void* key, const void* value, const void* key_cache,
                             const void* value_cache, const int64_t* slot_mapping, int T, int Hk,
                             int D, int S, int NB, int64_t key_stride_tok,
                             int64_t value_stride_tok, bool fp8, const float* k_scale,
                             const float* v_scale, pd_dtype dt, bool* skip) {
    *skip = false;
    if (T < 0 || Hk < 1 || NB < 1) return PD_ERR_INVALID_ARG;
    if (!supported_D(D) || !supported_S(S) || !supported_dt(dt)) return PD_ERR_UNSUPPORTED;
    if (!key_cache || !value_cache || !aligned16(key_cache) || !aligned16(value_cache))
        return PD_ERR_INVALID_ARG;
    if (T == 0) {
        *skip = true;
        return PD_OK;
    }
    if (!key || !value || !slot_mapping || !aligned16(key) || !aligned16(value))
        return PD_ERR_INVALID_ARG;
    if (fp8 && (!k_scale || !v_scale)) return PD_ERR_INVALID_ARG;
    if (key_stride_tok < int64_t(Hk) * D || value_stride_tok < int64_t(Hk) * D ||
        key_stride_tok % 8 || value_stride_tok % 8)
        return PD_ERR_INVALID_ARG;
    return PD_OK;
}

pd_status pd_reshape_and_cache(const void* key, const void* value, void* key_cache,
                               void* value_cache, const int64_t* slot_mapping, int T, int Hk,
                               int D, int S, int NB, int64_t key_stride_tok,
                               int64_t value_stride_tok, pd_dtype dt, int32_t* dev_err,
                               cudaStream_t stream) {
    bool skip = false;
    const pd_status st = store_check(key, value, key_cache, value_cache, slot_mapping, T, Hk, D, S,
                                     NB, key_stride_tok, value_stride_tok, false, nullptr,
                                     nullptr, dt, &skip);
    if (st != PD_OK || skip) return st;
    return launch_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, T, Hk, D,
                                    S, NB, key_stride_tok, value_stride_tok, dev_err, stream);
}

size_t pd_decode_workspace_bytes(int B, int H, int D, int max_context_len) {
    if (B < 1 || H < 1 || !supported_D(D) || max_context_len < 0) return 0;
    return decode_workspace_bytes(B, H, D, max_context_len);
}

int pd_decode_partition_tokens(int max_context_len) {
    return decode_partition_tokens(max_context_len);
}

static pd_status decode_common(void* out, const void* q, const void* key_cache,
                               const void* value_cache, const float* k_scale,
                               const float* v_scale, bool fp8, const int32_t* block_tables,
                               int max_blocks_per_seq, const int32_t* context_lens, int B, int H,
                               int Hk, int D, int S, int NB, int max_context_len, float scale,
                               void* workspace, size_t workspace_bytes, pd_dtype dt,
                               int32_t* dev_err, cudaStream_t stream) {
    DecodeArgs a{};
    bool skip = false;
    const pd_status st = decode_prepare(out, q, key_cache, value_cache, k_scale, v_scale, fp8,
                                        block_tables, max_blocks_per_seq, context_lens, B, H, Hk,
                                        D, S, NB, max_context_len, scale, workspace,
                                        workspace_bytes, dt, dev_err, stream, &a, &skip);
    if (st != PD_OK || skip) return st;
    return launch_decode(a);
}

// Store then decode on one stream.  The decode grid is launched as a
// programmatic dependent of the store grid: its CTAs start while the store
// runs, do everything that does not read the pools (barriers, tensor-map
// prefetch, context lengths, work split, first block ids), and wait for the
// store grid's writes before their first K/V copy.  Both kernels follow
// ordinary stream order with respect to everything launched before the store.
static pd_status step_common(const void* key, const void* value, const int64_t* slot_mapping,
                             int T, int64_t key_stride_tok, int64_t value_stride_tok, void* out,
                             const void* q, void* key_cache, void* value_cache,
                             const float* k_scale, const float* v_scale, bool fp8,
                             const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* context_lens, int B, int H, int Hk, int D, int S,
                             int NB, int max_context_len, float scale, void* workspace,
                             size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                             cudaStream_t stream, int nq = 1) {
    DecodeArgs a{};
    bool skip_dec = false, skip_store = false;
    if (fp8 && nq > 1) return PD_ERR_UNSUPPORTED;
    pd_status st = decode_prepare(out, q, key_cache, value_cache, k_scale, v_scale, fp8,
                                  block_tables, max_blocks_per_seq, context_lens, B, H, Hk, D, S,
                                  NB, max_context_len, scale, workspace, workspace_bytes, dt,
                                  dev_err, stream, &a, &skip_dec, nq);
    if (st != PD_OK) return st;
    st = store_check(key, value, key_cache, value_cache, slot_mapping, T, Hk, D, S, NB,
                     key_stride_tok, value_stride_tok, fp8, k_scale, v_scale, dt, &skip_store);
    if (st != PD_OK) return st;
    if (!skip_store) {
        st = fp8 ? launch_reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping,
                                                T, Hk, D, S, NB, key_stride_tok, value_stride_tok,
                                                k_scale, v_scale, dt, dev_err, stream)
                 : launch_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, T,
                                            Hk, D, S, NB, key_stride_tok, value_stride_tok,
                                            dev_err, stream);
        if (st != PD_OK) return st;
    }
    if (skip_dec) return PD_OK;
    a.pdl = !skip_store;    // only ever dependent on our own store grid
    return launch_decode(a);
}

pd_status pd_paged_attention_decode(void* out, const void* q, const void* key_cache,
                                    const void* value_cache, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* context_lens, int B,
                                    int H, int Hk, int D, int S, int NB, int max_context_len,
                                    float scale, void* workspace, size_t workspace_bytes,
                                    pd_dtype dt, int32_t* dev_err, cudaStream_t stream) {
    return decode_common(out, q, key_cache, value_cache, nullptr, nullptr, false, block_tables,
                         max_blocks_per_seq, context_lens, B, H, Hk, D, S, NB, max_context_len,
                         scale, workspace, workspace_bytes, dt, dev_err, stream);
}

pd_status pd_paged_attention_decode_fp8(void* out, const void* q, const void* key_cache,
                                        const void* value_cache, const float* k_scale,
                                        const float* v_scale, const int32_t* block_tables,
                                        int max_blocks_per_seq, const int32_t* context_lens,
                                        int B, int H, int Hk, int D, int S, int NB,
                                        int max_context_len, float scale, void* workspace,
                                        size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                                        cudaStream_t stream) {
    return decode_common(out, q, key_cache, value_cache, k_scale, v_scale, true, block_tables,
                         max_blocks_per_seq, context_lens, B, H, Hk, D, S, NB, max_context_len,
                         scale, workspace, workspace_bytes, dt, dev_err, stream);
}

pd_status pd_decode_step(const void* key, const void* value, const int64_t* slot_mapping, int T,
                         int64_t key_stride_tok, int64_t value_stride_tok, void* out,
                         const void* q, void* key_cache, void* value_cache,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int B, int H, int Hk, int D, int S, int NB,
                         int max_context_len, float scale, void* workspace,
                         size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                         cudaStream_t stream) {
    return step_common(key, value, slot_mapping, T, key_stride_tok, value_stride_tok, out, q,
                       key_cache, value_cache, nullptr, nullptr, false, block_tables,
                       max_blocks_per_seq, context_lens, B, H, Hk, D, S, NB, max_context_len,
                       scale, workspace, workspace_bytes, dt, dev_err, stream);
}

pd_status pd_decode_step_fused(const void* key, const void* value, const int64_t* slot_mapping,
                               int T, int64_t key_stride_tok, int64_t value_stride_tok,
                               void* out, const void* q, void* key_cache, void* value_cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int B, int H, int Hk, int D, int S,
                               int NB, int max_context_len, float scale, void* workspace,
                               size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                               cudaStream_t stream) {
    DecodeArgs a{};
    bool skip_dec = false, skip_store = false;
    pd_status st = decode_prepare(out, q, key_cache, value_cache, nullptr, nullptr, false,
                                  block_tables, max_blocks_per_seq, context_lens, B, H, Hk, D, S,
                                  NB, max_context_len, scale, workspace, workspace_bytes, dt,
                                  dev_err, stream, &a, &skip_dec, 1);
    if (st != PD_OK) return st;
    st = store_check(key, value, key_cache, value_cache, slot_mapping, T, Hk, D, S, NB,
                     key_stride_tok, value_stride_tok, false, nullptr, nullptr, dt, &skip_store);
    if (st != PD_OK) return st;
    if (T != B) return PD_ERR_INVALID_ARG;              // one new row per sequence
    // every kv head must be read by one CTA group alone (G <= 8 query heads)
    if (H / Hk > 8) return PD_ERR_UNSUPPORTED;
    if (skip_dec) return PD_OK;
    if (!skip_store) {
        a.row_k = key;
        a.row_v = value;
        a.row_ks = key_stride_tok;
        a.row_vs = value_stride_tok;
        a.row_slots = slot_mapping;
    }
    return launch_decode(a);
}

pd_status pd_decode_step_fp8(const void* key, const void* value, const int64_t* slot_mapping,
                             int T, int64_t key_stride_tok, int64_t value_stride_tok, void* out,
                             const void* q, void* key_cache, void* value_cache,
                             const float* k_scale, const float* v_scale,
                             const int32_t* block_tables, int max_blocks_per_seq,
                             const int32_t* context_lens, int B, int H, int Hk, int D, int S,
                             int NB, int max_context_len, float scale, void* workspace,
                             size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                             cudaStream_t stream) {
    return step_common(key, value, slot_mapping, T, key_stride_tok, value_stride_tok, out, q,
                       key_cache, value_cache, k_scale, v_scale, true, block_tables,
                       max_blocks_per_seq, context_lens, B, H, Hk, D, S, NB, max_context_len,
                       scale, workspace, workspace_bytes, dt, dev_err, stream);
}

size_t pd_decode_shared_workspace_bytes(int n_groups, int max_group, int H, int Hk, int D) {
    if (n_groups < 1 || n_groups > 65535 || max_group < 1 || max_group > 32 || H < 1 ||
        Hk < 1 || H % Hk != 0 || !supported_D(D))
        return 0;
    return decode_shared_workspace_bytes(n_groups, max_group, H, Hk, D);
}

pd_status pd_paged_attention_decode_shared(void* out, const void* q, const void* key_cache,
                                           const void* value_cache, const int32_t* block_tables,
                                           int max_blocks_per_seq, const int32_t* context_lens,
                                           int B, int H, int Hk, int D, int S, int NB,
                                           int max_context_len, float scale,
                                           const int32_t* group_starts,
                                           const int32_t* shared_lens, int n_groups,
                                           int max_group, void* workspace,
                                           size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                                           cudaStream_t stream) {
    DecodeArgs a{};
    bool skip = false;
    const SharedGroups grp{group_starts, shared_lens, n_groups, max_group};
    const pd_status st = decode_prepare(out, q, key_cache, value_cache, nullptr, nullptr, false,
                                        block_tables, max_blocks_per_seq, context_lens, B, H, Hk,
                                        D, S, NB, max_context_len, scale, workspace,
                                        workspace_bytes, dt, dev_err, stream, &a, &skip, 1, true,
                                        &grp);
    if (st != PD_OK || skip) return st;
    return launch_decode(a);
}

pd_status pd_decode_step_shared(const int64_t* block_mapping, int npairs, const void* key,
                                const void* value, const int64_t* slot_mapping, int T,
                                int64_t key_stride_tok, int64_t value_stride_tok, void* out,
                                const void* q, void* key_cache, void* value_cache,
                                const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* context_lens, int B, int H, int Hk, int D, int S,
                                int NB, int max_context_len, float scale,
                                const int32_t* group_starts, const int32_t* shared_lens,
                                int n_groups, int max_group, void* workspace,
                                size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                                cudaStream_t stream) {
    DecodeArgs a{};
    bool skip_dec = false, skip_store = false;
    if (npairs < 0 || (npairs > 0 && !block_mapping)) return PD_ERR_INVALID_ARG;
    const SharedGroups grp{group_starts, shared_lens, n_groups, max_group};
    pd_status st = decode_prepare(out, q, key_cache, value_cache, nullptr, nullptr, false,
                                  block_tables, max_blocks_per_seq, context_lens, B, H, Hk, D, S,
                                  NB, max_context_len, scale, workspace, workspace_bytes, dt,
                                  dev_err, stream, &a, &skip_dec, 1, true, &grp);
    if (st != PD_OK) return st;
    st = store_check(key, value, key_cache, value_cache, slot_mapping, T, Hk, D, S, NB,
                     key_stride_tok, value_stride_tok, false, nullptr, nullptr, dt, &skip_store);
    if (st != PD_OK) return st;
    // copy -> store -> decode, each grid a programmatic dependent of the one
    // before it: the store waits for the copy before writing, the decode for
    // the store (and so for the copy) before reading the pools
    bool launched = false;
    if (npairs > 0) {
        st = launch_copy_blocks(nullptr, nullptr, 1, block_mapping, npairs, Hk, D, S, NB, 2,
                                dev_err, stream, key_cache, value_cache);
        if (st != PD_OK) return st;
        launched = true;
    }
    if (!skip_store) {
        st = launch_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, T, Hk, D,
                                      S, NB, key_stride_tok, value_stride_tok, dev_err, stream,
                                      launched);
        if (st != PD_OK) return st;
        launched = true;
    }
    if (skip_dec) return PD_OK;
    a.pdl = launched;
    return launch_decode(a);
}

pd_status pd_paged_attention_verify(void* out, const void* q, const void* key_cache,
                                    const void* value_cache, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* context_lens, int B,
                                    int nq, int H, int Hk, int D, int S, int NB,
                                    int max_context_len, float scale, void* workspace,
                                    size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                                    cudaStream_t stream) {
    DecodeArgs a{};
    bool skip = false;
    const pd_status st = decode_prepare(out, q, key_cache, value_cache, nullptr, nullptr, false,
                                        block_tables, max_blocks_per_seq, context_lens, B, H, Hk,
                                        D, S, NB, max_context_len, scale, workspace,
                                        workspace_bytes, dt, dev_err, stream, &a, &skip, nq);
    if (st != PD_OK || skip) return st;
    return launch_decode(a);
}

// Device address of p if the device can reach it (device or managed memory,
// or host memory registered / allocated pinned and mapped), else nullptr.
static const void* device_view(const void* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();                      // clear the sticky-free error
        return nullptr;
    }
    switch (at.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged:
            return p;
        case cudaMemoryTypeHost:
            return at.devicePointer;
        default:
            return nullptr;
    }
}

pd_status pd_copy_bytes(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
    if (bytes == 0) return PD_OK;
    if (!dst || !src || !aligned16(dst) || !aligned16(src) || (bytes & 15u))
        return PD_ERR_INVALID_ARG;
    const void* d = device_view(dst);
    const void* s = device_view(src);
    if (!d || !s || !aligned16(d) || !aligned16(s)) return PD_ERR_INVALID_ARG;
    return launch_copy_bytes(const_cast<void*>(d), s, bytes, stream);
}

pd_status pd_selftest_bounded_wait(int32_t* dev_err, uint64_t limit_ns, cudaStream_t stream) {
    if (!dev_err || limit_ns < 1000ull || limit_ns > 10000000000ull) return PD_ERR_INVALID_ARG;
    return launch_bounded_wait_selftest(dev_err, (unsigned long long)limit_ns, stream);
}

pd_status pd_verify_step(const void* key, const void* value, const int64_t* slot_mapping, int T,
                         int64_t key_stride_tok, int64_t value_stride_tok, void* out,
                         const void* q, void* key_cache, void* value_cache,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int B, int nq, int H, int Hk, int D, int S,
                         int NB, int max_context_len, float scale, void* workspace,
                         size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                         cudaStream_t stream) {
    return step_common(key, value, slot_mapping, T, key_stride_tok, value_stride_tok, out, q,
                       key_cache, value_cache, nullptr, nullptr, false, block_tables,
                       max_blocks_per_seq, context_lens, B, H, Hk, D, S, NB, max_context_len,
                       scale, workspace, workspace_bytes, dt, dev_err, stream, nq);
}

pd_status pd_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache,
                                   void* value_cache, const int64_t* slot_mapping, int T, int Hk,
                                   int D, int S, int NB, int64_t key_stride_tok,
                                   int64_t value_stride_tok, const float* k_scale,
                                   const float* v_scale, pd_dtype in_dt, int32_t* dev_err,
                                   cudaStream_t stream) {
    bool skip = false;
    const pd_status st = store_check(key, value, key_cache, value_cache, slot_mapping, T, Hk, D, S,
                                     NB, key_stride_tok, value_stride_tok, true, k_scale, v_scale,
                                     in_dt, &skip);
    if (st != PD_OK || skip) return st;
    return launch_reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping, T, Hk,
                                        D, S, NB, key_stride_tok, value_stride_tok, k_scale,
                                        v_scale, in_dt, dev_err, stream);
}

pd_status pd_copy_blocks(void* const* key_caches, void* const* value_caches, int L,
                         const int64_t* block_mapping, int npairs, int Hk, int D, int S, int NB,
                         pd_dtype dt, int32_t* dev_err, cudaStream_t stream) {
    if (L < 0 || npairs < 0 || Hk < 1 || NB < 1) return PD_ERR_INVALID_ARG;
    if (!supported_D(D) || !supported_S(S) || !supported_pool_dt(dt)) return PD_ERR_UNSUPPORTED;
    if (L == 0 || npairs == 0) return PD_OK;
    if (!key_caches || !value_caches || !block_mapping) return PD_ERR_INVALID_ARG;
    if (L > 65535) return PD_ERR_UNSUPPORTED;
    return launch_copy_blocks(key_caches, value_caches, L, block_mapping, npairs, Hk, D, S, NB,
                              elem_bytes(dt), dev_err, stream);
}

static pd_status kv_pack_common(bool unpack, void* staging, void* const* key_caches,
                                void* const* value_caches, int L, const int32_t* block_ids,
                                int nblk, int Hk, int D, int S, int NB, pd_dtype dt,
                                int32_t* dev_err, cudaStream_t stream) {
    if (L < 0 || nblk < 0 || Hk < 1 || NB < 1) return PD_ERR_INVALID_ARG;
    if (!supported_D(D) || !supported_S(S) || !supported_pool_dt(dt)) return PD_ERR_UNSUPPORTED;
    if (L == 0 || nblk == 0) return PD_OK;
    if (!staging || !key_caches || !value_caches || !block_ids || !aligned16(staging))
        return PD_ERR_INVALID_ARG;
    if (L > 65535) return PD_ERR_UNSUPPORTED;
    return launch_kv_pack(unpack, staging, key_caches, value_caches, L, block_ids, nblk, Hk, D,
                          S, NB, elem_bytes(dt), dev_err, stream);
}

pd_status pd_kv_pack(void* staging, void* const* key_caches, void* const* value_caches, int L,
                     const int32_t* block_ids, int nblk, int Hk, int D, int S, int NB,
                     pd_dtype dt, int32_t* dev_err, cudaStream_t stream) {
    return kv_pack_common(false, staging, key_caches, value_caches, L, block_ids, nblk, Hk, D, S,
                          NB, dt, dev_err, stream);
}

pd_status pd_kv_unpack(const void* staging, void* const* key_caches, void* const* value_caches,
                       int L, const int32_t* block_ids, int nblk, int Hk, int D, int S, int NB,
                       pd_dtype dt, int32_t* dev_err, cudaStream_t stream) {
    return kv_pack_common(true, const_cast<void*>(staging), key_caches, value_caches, L,
                          block_ids, nblk, Hk, D, S, NB, dt, dev_err, stream);
}

pd_status pd_paged_prefill_chunk(void* out, const void* q, int total_q,
                                 const int32_t* cu_q_lens, int max_q_len,
                                 const void* key_cache, const void* value_cache,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int B, int H, int Hk, int D, int S,
                                 int NB, float scale, pd_dtype dt, int32_t* dev_err,
                                 cudaStream_t stream) {
    if (B < 0 || H < 1 || Hk < 1 || NB < 1 || max_blocks_per_seq < 1 || max_q_len < 0 ||
        total_q < 0)
        return PD_ERR_INVALID_ARG;
    if (H % Hk != 0 || !(scale > 0.f) || !std::isfinite(scale)) return PD_ERR_INVALID_ARG;
    if (!supported_D(D) || !supported_S(S) || !supported_dt(dt)) return PD_ERR_UNSUPPORTED;
    if (B == 0 || max_q_len == 0 || total_q == 0) return PD_OK;
    if (!out || !q || !cu_q_lens || !key_cache || !value_cache || !block_tables || !context_lens)
        return PD_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache))
        return PD_ERR_INVALID_ARG;
    if (B > 65535 || int64_t(max_blocks_per_seq) * S > (int64_t(1) << 30))
        return PD_ERR_UNSUPPORTED;
    if (int64_t(max_q_len) > int64_t(65535) * 128 || int64_t(NB) * Hk * S > (int64_t(1) << 31))
        return PD_ERR_UNSUPPORTED;
    PrefillArgs a{out, q, total_q, cu_q_lens, max_q_len, key_cache, value_cache, block_tables,
                  max_blocks_per_seq, context_lens, B, H, Hk, D, S, NB, scale, dt, dev_err,
                  stream};
    return launch_prefill(a);
}

}  // extern "C"
