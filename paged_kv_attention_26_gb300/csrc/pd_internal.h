// pd_internal.h -- host-side declarations shared by the library's translation
// units (validation helpers, launch accounting, per-op launchers).
#pragma once

#include <cstddef>
#include <cstdint>

#include "pd_attn.h"

namespace pd {

// Record a kernel launch result; returns PD_OK or PD_ERR_CUDA (and keeps
// the cudaError_t for pd_last_cuda_error()).
pd_status launch_result(cudaError_t e);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool supported_D(int D) { return D == 64 || D == 128; }
inline bool supported_S(int S) { return S == 8 || S == 16 || S == 32 || S == 64; }
inline bool supported_dt(pd_dtype dt) { return dt == PD_F16 || dt == PD_BF16; }
inline bool supported_pool_dt(pd_dtype dt) { return supported_dt(dt) || dt == PD_FP8_E4M3; }
inline int elem_bytes(pd_dtype dt) { return dt == PD_FP8_E4M3 ? 1 : 2; }

// ---- decode ------------------------------------------------------------------
// Partition length chosen for a batch; a multiple of 64 tokens.
int decode_partition_tokens(int max_context_len);
int decode_num_partitions(int max_context_len);
size_t decode_workspace_bytes(int B, int H, int D, int max_context_len);
// Workspace of the shared-prefix mode (H % Hk == 0, 1 <= max_group <= 32).
size_t decode_shared_workspace_bytes(int n_groups, int max_group, int H, int Hk, int D);

struct DecodeArgs {
    void* out;
    const void* q;
    const void* key_cache;
    const void* value_cache;
    const int32_t* block_tables;
    int max_blocks_per_seq;
    const int32_t* context_lens;
    int B, H, Hk, D, S, NB;
    int max_context_len;
    float scale;
    void* workspace;
    pd_dtype dt;                 // q and out
    int32_t* dev_err;
    cudaStream_t stream;
    bool fp8 = false;            // pools hold E4M3 codes ...
    const float* k_scale = nullptr;   // ... standing for code * scale[kv head]
    const float* v_scale = nullptr;
    bool pdl = false;            // launch as a programmatic dependent of the previous grid
    // pd_decode_step_fused: row i of row_k / row_v (row_ks / row_vs elements
    // between rows) is stored at row_slots[i] by the decode itself (null: none)
    const void* row_k = nullptr;
    const void* row_v = nullptr;
    int64_t row_ks = 0, row_vs = 0;
    const int64_t* row_slots = nullptr;
    int nq = 1;                  // query tokens per sequence (> 1: speculative verification)
    // shared-prefix mode (n_groups > 0): groups of consecutive sequences whose
    // tables agree on their first blocks
    const int32_t* grp_start = nullptr;    // device [n_groups + 1]
    const int32_t* grp_shared = nullptr;   // device [n_groups], tokens
    int n_groups = 0;
    int max_group = 1;           // most members a group may have (<= 32)
};
pd_status launch_decode(const DecodeArgs& a);
// Groups of the shared-prefix decode (device arrays, see
// pd_paged_attention_decode_shared).
struct SharedGroups {
    const int32_t* start;
    const int32_t* shared;
    int n_groups;
    int max_group;
};
// Argument checks shared by every decode entry point (defined in capi.cu);
// fills *a, sets *skip when B == 0.  check_workspace_ptr == false leaves the
// workspace address to the caller (checked size only); grp != nullptr selects
// the shared-prefix mode and its workspace size.
pd_status decode_prepare(void* out, const void* q, const void* key_cache,
                         const void* value_cache, const float* k_scale, const float* v_scale,
                         bool fp8, const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* context_lens, int B, int H, int Hk, int D, int S, int NB,
                         int max_context_len, float scale, void* workspace,
                         size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                         cudaStream_t stream, DecodeArgs* a, bool* skip, int nq = 1,
                         bool check_workspace_ptr = true, const SharedGroups* grp = nullptr);
pd_status launch_bounded_wait_selftest(int32_t* dev_err, unsigned long long limit_ns,
                                       cudaStream_t stream);
pd_status launch_copy_bytes(void* dst, const void* src, size_t bytes, cudaStream_t stream);

// ---- store / copy ----------------------------------------------------------------
pd_status launch_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                   void* value_cache, const int64_t* slot_mapping, int T,
                                   int Hk, int D, int S, int NB, int64_t key_stride_tok,
                                   int64_t value_stride_tok, int32_t* dev_err,
                                   cudaStream_t stream, bool pdl = false);
pd_status launch_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache,
                                       void* value_cache, const int64_t* slot_mapping, int T,
                                       int Hk, int D, int S, int NB, int64_t key_stride_tok,
                                       int64_t value_stride_tok, const float* k_scale,
                                       const float* v_scale, pd_dtype in_dt, int32_t* dev_err,
                                       cudaStream_t stream);
// key_caches == nullptr: one layer whose pools are k_pool / v_pool.
pd_status launch_copy_blocks(void* const* key_caches, void* const* value_caches, int L,
                             const int64_t* block_mapping, int npairs, int Hk, int D, int S,
                             int NB, int esize, int32_t* dev_err, cudaStream_t stream,
                             void* k_pool = nullptr, void* v_pool = nullptr);

// ---- KV pack / unpack ------------------------------------------------------------------
pd_status launch_kv_pack(bool unpack, void* staging, void* const* key_caches,
                         void* const* value_caches, int L, const int32_t* block_ids, int nblk,
                         int Hk, int D, int S, int NB, int esize, int32_t* dev_err,
                         cudaStream_t stream);

// ---- prefill -------------------------------------------------------------------------
struct PrefillArgs {
    void* out;
    const void* q;
    int total_q;
    const int32_t* cu_q_lens;
    int max_q_len;
    const void* key_cache;
    const void* value_cache;
    const int32_t* block_tables;
    int max_blocks_per_seq;
    const int32_t* context_lens;
    int B, H, Hk, D, S, NB;
    float scale;
    pd_dtype dt;
    int32_t* dev_err;
    cudaStream_t stream;
};
pd_status launch_prefill(const PrefillArgs& a);

void count_launch();

}  // namespace pd
