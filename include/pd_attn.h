/*
 * pd_attn.h -- C ABI of the paged KV-cache attention library (GB300, sm_103a).
 *
 * The operations are those of a prefill/decode-disaggregated serving engine
 * whose KV cache is paged (nanoPD page "nanoPD：从零实现的LLM预填充/解码分离推
 * 理引擎", sections "分页KV缓存", "分块预填充", "自定义CUDA分页注意力内核" and
 * "模块结构与代码组织": paged KV store op and paged multi-head attention
 * kernel), with the paging scheme of the tutorial page "LLM 推理服务引擎深度拆
 * 解", section 2.2: fixed-size blocks of S tokens, a per-sequence block table
 * mapping logical block i to a physical block, and one indirection per KV read.
 *
 * Conventions shared by every device entry point
 * - Cache layout, one pool per layer and per K/V: [NB][Hk][S][D] elements,
 *   contiguous (block-major, then kv head, then token offset, then dim).
 *   Logical token t of sequence i lives in physical block
 *   block_tables[i * max_blocks_per_seq + t / S] at offset t % S; its slot
 *   number is block * S + t % S.
 * - All tensor pointers are CALLER-OWNED DEVICE memory, 16-byte aligned;
 *   the library allocates nothing on the device and never synchronises: work
 *   is enqueued on `stream` (NULL = legacy default stream) and returns.
 * - Element types: K, V, Q and outputs share one `pd_dtype` (fp16 or bf16).
 *   Attention accumulates in fp32 and rounds its output to the element type
 *   with round-to-nearest-even.
 * - Supported shapes: D in {64, 128}; S in {8, 16, 32, 64}; H % Hk == 0.
 *   Other values return PD_ERR_UNSUPPORTED; bad pointers, negative sizes or
 *   inconsistent arguments return PD_ERR_INVALID_ARG.  Nothing is launched
 *   when a call returns an error.
 * - Device-side faults are never trapped.  Kernels check every slot, block
 *   id and context length they read against the sizes given; an offender is
 *   skipped and a bit is OR-ed into *dev_err (caller-owned device int32,
 *   may be NULL to ignore).  Results touched by a flagged input are
 *   unspecified.  Every wait inside a kernel is bounded in time; a wait that
 *   runs out sets PD_DEVERR_TIMEOUT and the kernel returns.
 * - PD_ERR_CUDA means a launch failed; pd_last_cuda_error() returns the
 *   cudaError_t value of the last failure in this thread.
 */
#ifndef PD_ATTN_H
#define PD_ATTN_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

/* Exported symbols keep default visibility when the library is built with
 * -fvisibility=hidden. */
#if defined(__GNUC__)
#define PD_API __attribute__((visibility("default")))
#else
#define PD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pd_status {
    PD_OK = 0,
    PD_ERR_INVALID_ARG = 1,
    PD_ERR_UNSUPPORTED = 2,
    PD_ERR_CUDA = 3,
    PD_ERR_NO_FREE_BLOCK = 4,
    PD_ERR_WORKSPACE_TOO_SMALL = 5,
    PD_ERR_NOT_FOUND = 6
} pd_status;

typedef enum pd_dtype { PD_F16 = 0, PD_BF16 = 1, PD_FP8_E4M3 = 2 } pd_dtype;

/* Bits OR-ed into the caller's device error word. */
#define PD_DEVERR_SLOT_RANGE 0x1  /* slot >= NB * S in a store               */
#define PD_DEVERR_BLOCK_RANGE 0x2 /* block id outside [0, NB)                */
#define PD_DEVERR_CTX_RANGE 0x4   /* context longer than table / promise     */
#define PD_DEVERR_TIMEOUT 0x8     /* a bounded wait inside a kernel expired  */
#define PD_DEVERR_SHARED_PREFIX 0x10 /* shared-prefix groups malformed, or a
                                        member's table differs in the prefix */
#define PD_DEVERR_STEP_SLOT 0x20  /* fused step: a slot that is not the one of
                                     the sequence's last token (not stored) */

/* Text for a status code (static storage). */
PD_API const char* pd_status_string(pd_status s);
/* cudaError_t of the last PD_ERR_CUDA returned to this thread (0 if none). */
PD_API int pd_last_cuda_error(void);
/* Number of kernels this library has launched in this process (a counter
 * for accounting; every successful launch increments it by one). */
PD_API uint64_t pd_launch_count(void);

/* ---------------------------------------------------------------------- */
/* Store new tokens' K/V into their cache slots (nanoPD page, "模块结构与代码
 * 组织": the paged KV store op; slots come from the block manager, tutorial
 * page section 2.3, Sequence.append_token).
 *   key, value    [T][Hk][D] (token stride key_stride_tok / value_stride_tok
 *                 elements, heads contiguous at stride D)
 *   key_cache, value_cache   [NB][Hk][S][D], written in place
 *   slot_mapping  int64 [T]; slot < 0 skips the token (padding);
 *                 slot >= NB*S is skipped and flags PD_DEVERR_SLOT_RANGE.
 * A bit copy: no conversion.  Two tokens mapped to one slot race. */
PD_API pd_status pd_reshape_and_cache(const void* key, const void* value,
                               void* key_cache, void* value_cache,
                               const int64_t* slot_mapping, int T, int Hk,
                               int D, int S, int NB, int64_t key_stride_tok,
                               int64_t value_stride_tok, pd_dtype dt,
                               int32_t* dev_err, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Decode attention: one query token per sequence over its paged context
 * (nanoPD page, "自定义CUDA分页注意力内核": gather attention over
 * non-contiguous KV blocks; GQA as in the essay page "LLM推理PD分离架构深度
 * 工程实践", section 6.2: q head h reads kv head h / (H / Hk)).
 *   out[i][h][:] = sum_{t < ctx_i} softmax_t(scale * q[i][h] . k_t) v_t
 * with ctx_i = context_lens[i] (it counts any token stored this step) and
 * ctx_i == 0 giving zeros.
 *   out, q        [B][H][D]
 *   block_tables  int32 [B][max_blocks_per_seq]
 *   context_lens  int32 [B], each <= max_context_len (the caller's promise,
 *                 checked on device: PD_DEVERR_CTX_RANGE, the context is
 *                 then cut to max_context_len and to what the table holds)
 * One kernel launch.  The resident CTAs form one group per kv head (or
 * head group); each group cuts that head's work over the batch into equal
 * contiguous runs of 64-token stages, one per CTA, so a long context may be
 * split across CTAs (online softmax per piece, pieces kept in `workspace`);
 * the CTA that finishes a context's last outstanding piece merges the
 * pieces in fixed order.  A context that one CTA finishes is written
 * directly.
 *   workspace     device scratch of at least
 *                 pd_decode_workspace_bytes(B, H, D, max_context_len) bytes
 *                 (always > 0), 256-byte aligned.  Nothing in it needs to
 *                 start at zero: pieces are written before they are read in
 *                 the same launch, and the per-context arrival counters carry
 *                 a per-launch tag, so whatever an earlier launch (or other
 *                 data) left there counts as zero.  The arrival that
 *                 completes a context writes its counter back to zero, so a
 *                 launch captured in a CUDA graph (tag fixed at capture)
 *                 may be replayed any number of times; after a replay that
 *                 flagged PD_DEVERR_TIMEOUT, zero the workspace before the
 *                 next replay.  Overwritten; callers sharing one workspace
 *                 on two streams race.
 *                 PD_ERR_WORKSPACE_TOO_SMALL if short. */
PD_API size_t pd_decode_workspace_bytes(int B, int H, int D, int max_context_len);
/* Token granule of the work split: a CTA takes at least this many tokens
 * before another CTA shares a context, so one context is cut into at most
 * ceil(ctx / granule) + 1 pieces (exposed for accounting and tests). */
PD_API int pd_decode_partition_tokens(int max_context_len);
PD_API pd_status pd_paged_attention_decode(void* out, const void* q,
                                    const void* key_cache,
                                    const void* value_cache,
                                    const int32_t* block_tables,
                                    int max_blocks_per_seq,
                                    const int32_t* context_lens, int B, int H,
                                    int Hk, int D, int S, int NB,
                                    int max_context_len, float scale,
                                    void* workspace, size_t workspace_bytes,
                                    pd_dtype dt, int32_t* dev_err,
                                    cudaStream_t stream);

/* Decode attention without any device allocation by the caller: same
 * operation, arguments and results as pd_paged_attention_decode, minus the
 * workspace.  The pages describe no such call; it exists for callers that
 * cannot allocate device memory on the call path (engines that reserve all
 * device memory at start-up and forbid later allocations, or code that must
 * not pay cudaMalloc's implicit synchronisation).
 * - The partition scratch is a fixed 32 MiB array inside the library; every
 *   GPU that loads the library keeps it until the process exits.  A batch
 *   whose pd_decode_workspace_bytes(B, H, D, max_context_len) exceeds
 *   32 MiB (33554432 bytes) is rejected with PD_ERR_WORKSPACE_TOO_SMALL and
 *   nothing is launched.
 * - The array's device address is looked up (cudaGetSymbolAddress, with the
 *   calling device current) on every call made outside stream capture, so a
 *   module reloaded after cudaDeviceReset is never reached through a stale
 *   address.  A call made while `stream` is capturing uses the address found
 *   by the last call outside capture on that device: make the first call on
 *   a device before any stream capture on it (otherwise PD_ERR_CUDA).
 * - Nothing in the scratch needs to start at zero (as for the workspace of
 *   pd_paged_attention_decode): every call tags its arrival counters with a
 *   tag of its own, so counts left behind by an earlier call, including one
 *   that flagged PD_DEVERR_TIMEOUT, read as zero.  A launch repeated with an
 *   unchanged tag would meet them; the caller has no address for the array
 *   and cannot clear it.
 * - All calls share the one array and it keeps what the last call wrote:
 *   calls that may overlap on the GPU (other streams, other host threads)
 *   race and must be serialised by the caller.
 * - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
PD_API pd_status pd_paged_attention_decode_noalloc(void* out, const void* q,
                                           const void* key_cache,
                                           const void* value_cache,
                                           const int32_t* block_tables,
                                           int max_blocks_per_seq,
                                           const int32_t* context_lens, int B,
                                           int H, int Hk, int D, int S, int NB,
                                           int max_context_len, float scale,
                                           pd_dtype dt, int32_t* dev_err,
                                           cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Decode attention for forks that share a prompt's blocks (tutorial page "LLM
 * 推理服务引擎深度拆解", section 2.3: parallel sampling forks a sequence n ways,
 * every fork keeps the prompt's blocks, with zero copies, and only a written
 * shared block is copied; nanoPD page "分页KV缓存": CoW for beam search and
 * speculative branches).  Same operation and result as
 * pd_paged_attention_decode on the same arguments; the work is arranged so
 * that each shared block is read from memory once for all the forks that
 * hold it, instead of once per fork.
 *   group_starts  DEVICE int32 [n_groups + 1]: group g is sequences
 *                 group_starts[g] .. group_starts[g+1] - 1 (consecutive);
 *                 group_starts[0] == 0, non-decreasing, group_starts[n_groups]
 *                 == B, at most max_group members per group
 *   shared_lens   DEVICE int32 [n_groups]: the caller's promise that every
 *                 member's block table holds the first member's block ids
 *                 over its first shared_lens[g] tokens.  The kernel uses
 *                 sh = shared_lens[g] rounded down to a multiple of S and cut
 *                 to the shortest member's context, reads tokens [0, sh) of
 *                 every member through the FIRST member's table and the rest
 *                 through each member's own.  A group layout that breaks the
 *                 rules above, or a member whose table differs from the first
 *                 member's within [0, sh), flags PD_DEVERR_SHARED_PREFIX
 *                 (checked on the device; results of that group unspecified).
 *                 shared_lens[g] == 0 is allowed (no sharing).
 *   max_group     1 .. 32 (sizes the column layout; (H / Hk) heads of up to
 *                 32 / max_group forks go through one pass over a kv head)
 *   workspace     device scratch of at least
 *                 pd_decode_shared_workspace_bytes(n_groups, max_group, H, Hk,
 *                 D) bytes, 256-byte aligned, same rules as the workspace of
 *                 pd_paged_attention_decode (nothing needs to start at zero)
 * every other argument as for pd_paged_attention_decode (16-bit pools).
 * With fp16 elements, probabilities enter the P.V product as one fp16 value
 * (2^-11 relative rounding); with bf16 as a hi + lo pair as in decode.
 * PD_ERR_UNSUPPORTED: max_group outside 1 .. 32, n_groups < 1 or > 65535. */
PD_API size_t pd_decode_shared_workspace_bytes(int n_groups, int max_group, int H, int Hk,
                                               int D);
PD_API pd_status pd_paged_attention_decode_shared(void* out, const void* q,
                                                  const void* key_cache,
                                                  const void* value_cache,
                                                  const int32_t* block_tables,
                                                  int max_blocks_per_seq,
                                                  const int32_t* context_lens, int B, int H,
                                                  int Hk, int D, int S, int NB,
                                                  int max_context_len, float scale,
                                                  const int32_t* group_starts,
                                                  const int32_t* shared_lens, int n_groups,
                                                  int max_group, void* workspace,
                                                  size_t workspace_bytes, pd_dtype dt,
                                                  int32_t* dev_err, cudaStream_t stream);
/* pd_decode_step_shared: one copy-on-write decode step of one layer over
 * forks that share blocks (tutorial page "LLM 推理服务引擎深度拆解", section
 * 2.3: a fork about to write a shared block first gets a copy of it, then
 * appends its token): the block copies, then the store of the new tokens,
 * then pd_paged_attention_decode_shared.  The result is exactly that of
 * pd_copy_blocks (this layer's pools only), pd_reshape_and_cache and
 * pd_paged_attention_decode_shared on the same stream.
 *   block_mapping  DEVICE int64 [npairs][2] (src, dst) copied in key_cache
 *                  and value_cache as by pd_copy_blocks; npairs == 0: none
 * every other argument as for pd_reshape_and_cache (key, value,
 * slot_mapping, T, strides; T == 0 skips the store) and for
 * pd_paged_attention_decode_shared.  Each grid is launched as a programmatic
 * dependent of the one before it: the store waits for the copies before it
 * writes, the decode waits for the store (and so for the copies) before it
 * reads the pools; prologues overlap.  Reads of q, block_tables,
 * context_lens and the group arrays may happen while the copies and the
 * store run.  All checks are made before anything is launched. */
PD_API pd_status pd_decode_step_shared(const int64_t* block_mapping, int npairs,
                                       const void* key, const void* value,
                                       const int64_t* slot_mapping, int T,
                                       int64_t key_stride_tok, int64_t value_stride_tok,
                                       void* out, const void* q, void* key_cache,
                                       void* value_cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int B, int H, int Hk, int D, int S, int NB,
                                       int max_context_len, float scale,
                                       const int32_t* group_starts, const int32_t* shared_lens,
                                       int n_groups, int max_group, void* workspace,
                                       size_t workspace_bytes, pd_dtype dt, int32_t* dev_err,
                                       cudaStream_t stream);
/* Host helper for the shared-prefix calls (no CUDA calls): cut sequences 0 .. B-1 into
 * groups of consecutive sequences that share leading blocks.  block_tables and
 * context_lens are HOST arrays laid out as for the decode calls.  For each
 * sequence i, its shared prefix with the first member f of the current group
 * is n * S tokens, n = the number of leading entries with
 * block_tables[i][b] == block_tables[f][b], counting only blocks b that are
 * full in both (b < min(ctx_i, ctx_f) / S).  Sequence i joins the group when
 * the group has fewer than max_group members and that prefix is at least
 * max(min_shared_tokens, S) tokens and at least the group's current shared
 * length (a later member never shortens what the earlier ones share); else
 * it starts a new group.  A group's shared_lens entry is its members' common
 * prefix (0 for a group of one).
 *   group_starts_out  [B + 1] (n_groups + 1 entries written)
 *   shared_lens_out   [B]     (n_groups entries written)
 * PD_ERR_INVALID_ARG on NULL pointers (block_tables, context_lens and
 * shared_lens_out may be NULL when B == 0), B < 0, max_blocks_per_seq < 1,
 * S < 1, or max_group outside 1 .. 32. */
PD_API pd_status pd_find_shared_prefixes(const int32_t* block_tables, int max_blocks_per_seq,
                                         const int32_t* context_lens, int B, int S,
                                         int max_group, int min_shared_tokens,
                                         int32_t* group_starts_out, int32_t* shared_lens_out,
                                         int* n_groups_out);

/* ---------------------------------------------------------------------- */
/* FP8 (E4M3) KV cache (essay page "LLM推理PD分离架构深度工程实践", section
 * 6.2; tutorial page "LLM 推理服务引擎深度拆解", section 8.1): pools hold one
 * E4M3 byte per value (1 sign, 4 exponent bits with bias 7, 3 fraction bits;
 * largest 448), half the bytes of BF16.  Each kv head h has a K scale
 * k_scale[h] and a V scale v_scale[h] (DEVICE float32 [Hk], > 0 and finite):
 * a stored code c stands for e4m3(c) * scale.
 *
 * pd_reshape_and_cache_fp8: as pd_reshape_and_cache, with key/value of type
 * in_dt (fp16 or bf16) and pools of E4M3 bytes [NB][Hk][S][D]: the code
 * stored is y = float(x) * (1.0f / scale[h]) (float32 product) rounded to the
 * nearest E4M3 value, ties to even, magnitudes beyond 448 saturating to 448.
 * A NaN input stores a NaN code. */
PD_API pd_status pd_reshape_and_cache_fp8(const void* key, const void* value,
                                          void* key_cache, void* value_cache,
                                          const int64_t* slot_mapping, int T,
                                          int Hk, int D, int S, int NB,
                                          int64_t key_stride_tok,
                                          int64_t value_stride_tok,
                                          const float* k_scale,
                                          const float* v_scale, pd_dtype in_dt,
                                          int32_t* dev_err, cudaStream_t stream);
/* pd_paged_attention_decode_fp8: decode attention over E4M3 pools:
 *   out[i][h] = sum_t softmax_t(scale * q . (k_t * k_scale[g])) v_t * v_scale[g]
 * with g = h / (H / Hk); q and out are of type dt (fp16 or bf16), every other
 * argument as for pd_paged_attention_decode (same workspace size).  The
 * tensor-core products run on fp16 operands: K and V are widened exactly, q
 * is rounded to fp16 (|q| must stay below 65504); the scales are applied in
 * float32. */
PD_API pd_status pd_paged_attention_decode_fp8(void* out, const void* q,
                                               const void* key_cache,
                                               const void* value_cache,
                                               const float* k_scale,
                                               const float* v_scale,
                                               const int32_t* block_tables,
                                               int max_blocks_per_seq,
                                               const int32_t* context_lens,
                                               int B, int H, int Hk, int D, int S,
                                               int NB, int max_context_len,
                                               float scale, void* workspace,
                                               size_t workspace_bytes, pd_dtype dt,
                                               int32_t* dev_err, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Speculative verification (tutorial page "LLM 推理服务引擎深度拆解",
 * section 7.1, 投机解码: the k drafted tokens and the last accepted one go
 * through the large model in a single forward pass, so the weights and the
 * KV cache are read once for k + 1 positions).
 * nq query tokens per sequence, the last nq positions of its context (their
 * K/V already stored): query j of sequence i sits at position
 * context_lens[i] - nq + j and attends to positions 0 .. that position
 * (causal among the nq).
 *   out, q        [B][nq][H][D] of type dt, contiguous
 *   nq            1 .. 8 (1 is exactly pd_paged_attention_decode)
 *   workspace     pd_decode_workspace_bytes(B * nq, H, D, max_context_len)
 *                 bytes, same rules as for decode
 * every other argument as for pd_paged_attention_decode (16-bit pools only).
 * The decode kernel, with the 8 MMA columns of a stream holding (head, query
 * token) pairs: the K/V of a kv head is read once for up to 8 / nq of its
 * query heads.  A context shorter than nq (but not empty) flags
 * PD_DEVERR_CTX_RANGE; queries that see no key then read 0.
 * PD_ERR_UNSUPPORTED: nq outside 1..8, B * nq > 65535. */
PD_API pd_status pd_paged_attention_verify(void* out, const void* q,
                                           const void* key_cache,
                                           const void* value_cache,
                                           const int32_t* block_tables,
                                           int max_blocks_per_seq,
                                           const int32_t* context_lens, int B, int nq,
                                           int H, int Hk, int D, int S, int NB,
                                           int max_context_len, float scale,
                                           void* workspace, size_t workspace_bytes,
                                           pd_dtype dt, int32_t* dev_err,
                                           cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* pd_verify_step: store the step's drafted tokens (key/value/slot_mapping/T
 * as for pd_reshape_and_cache), then pd_paged_attention_verify over them
 * (out/q [B][nq][H][D], workspace as for that call), the verify grid
 * launched as a programmatic dependent of the store grid exactly as in
 * pd_decode_step.  16-bit pools; nq 1 .. 8. */
PD_API pd_status pd_verify_step(const void* key, const void* value,
                                const int64_t* slot_mapping, int T,
                                int64_t key_stride_tok, int64_t value_stride_tok,
                                void* out, const void* q, void* key_cache,
                                void* value_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens,
                                int B, int nq, int H, int Hk, int D, int S, int NB,
                                int max_context_len, float scale, void* workspace,
                                size_t workspace_bytes, pd_dtype dt,
                                int32_t* dev_err, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* pd_copy_bytes: copies `bytes` bytes from src to dst with an SM kernel on
 * `stream`.  Each side may be device memory, managed memory, or pinned host
 * memory mapped into the device's address space (cudaHostAlloc /
 * cudaHostRegister); pageable host memory is refused.  Used to move a step's
 * inputs and results between pinned host buffers and the device: many
 * 16-byte loads in flight make a few-hundred-KB transfer link-bound rather
 * than bound by a copy engine's per-transfer latency.
 * Both pointers 16-byte aligned, bytes a multiple of 16; the ranges must not
 * overlap.  PD_ERR_INVALID_ARG otherwise (nothing launched); bytes == 0
 * launches nothing. */
PD_API pd_status pd_copy_bytes(void* dst, const void* src, size_t bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* pd_selftest_bounded_wait: exercises the in-kernel wait limit that every
 * kernel of the library uses.  Launches one CTA that waits on a shared-memory
 * barrier nothing completes; after limit_ns nanoseconds (1e3 .. 1e10) the
 * wait gives up, PD_DEVERR_TIMEOUT is OR-ed into *dev_err (DEVICE int32,
 * required) and the kernel returns, leaving the context usable.  For tests
 * of failure detection; it faults, traps and hangs nothing. */
PD_API pd_status pd_selftest_bounded_wait(int32_t* dev_err, uint64_t limit_ns,
                                          cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* One decode step of one layer: store the step's new K/V rows, then decode
 * attention that already sees them (nanoPD page, "模块结构与代码组织": the
 * attention layer writes the new token into its slot, then attends over the
 * whole paged context).  The result is exactly that of pd_reshape_and_cache
 * (or pd_reshape_and_cache_fp8) followed by pd_paged_attention_decode (or
 * pd_paged_attention_decode_fp8) on the same stream; the arguments are the
 * union of theirs, with key/value/slot_mapping/T/strides those of the store
 * and dt the type of key, value, q and out.
 * Difference: the decode grid is launched as a programmatic dependent of the
 * store grid, so its prologue (work split, context lengths, first block ids)
 * overlaps the store; every read of the pools waits for the store grid.
 * Ordering with earlier work on the stream is ordinary stream order.  Reads
 * of q, block_tables and context_lens may happen while the store runs, so the
 * store's inputs must not alias them (they never do in a decode step).
 * All checks of both calls are made before anything is launched; on an error
 * nothing is launched.  T == 0 skips the store (the decode then launches
 * normally); B == 0 skips the decode.
 * Host-to-host steps: key, value, slot_mapping, q, block_tables,
 * context_lens and out may be pinned host memory mapped into the device's
 * address space (cudaHostAlloc, or cudaHostRegister with
 * cudaHostRegisterMapped), given by its device address (with unified
 * addressing, the host address): the store and the decode then read the
 * step's inputs and write its result over the host link, with no separate
 * copy.  Each CTA of the decode reads the context lengths and its streams'
 * table rows, so those cross the link more than once; measured on a batch
 * of 64 that costs no more than copying them to the device first. */
PD_API pd_status pd_decode_step(const void* key, const void* value,
                                const int64_t* slot_mapping, int T,
                                int64_t key_stride_tok, int64_t value_stride_tok,
                                void* out, const void* q, void* key_cache,
                                void* value_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens,
                                int B, int H, int Hk, int D, int S, int NB,
                                int max_context_len, float scale, void* workspace,
                                size_t workspace_bytes, pd_dtype dt,
                                int32_t* dev_err, cudaStream_t stream);
/* pd_decode_step_fused: the same step as pd_decode_step (same arguments, the
 * same result) in ONE kernel, for the usual shape of a decode step: T == B,
 * row i of key/value is the new token of sequence i, the last of its
 * context (position context_lens[i] - 1), and slot_mapping[i] is that
 * token's slot through the sequence's table (or < 0: nothing stored for it).
 * The decode CTA that copies a sequence's last 64-token stage for a kv head
 * writes the row into the pool right before that copy; no other CTA reads
 * the block.  So the block holding a sequence's new token must be read by
 * no other sequence of the batch (the copy-on-write rule of the tutorial
 * page, section 2.3, gives every appended-to block a single owner).
 * A slot that is not the one of the sequence's last token (or a context cut
 * short by the table or max_context_len) is not stored and flags
 * PD_DEVERR_STEP_SLOT.  16-bit pools, G = H / Hk <= 8 (else
 * PD_ERR_UNSUPPORTED); T != B is PD_ERR_INVALID_ARG; T == B == 0 does
 * nothing.  Inputs may be pinned host memory as for pd_decode_step. */
PD_API pd_status pd_decode_step_fused(const void* key, const void* value,
                                      const int64_t* slot_mapping, int T,
                                      int64_t key_stride_tok, int64_t value_stride_tok,
                                      void* out, const void* q, void* key_cache,
                                      void* value_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* context_lens,
                                      int B, int H, int Hk, int D, int S, int NB,
                                      int max_context_len, float scale, void* workspace,
                                      size_t workspace_bytes, pd_dtype dt,
                                      int32_t* dev_err, cudaStream_t stream);
/* pd_decode_step_fp8: the same over E4M3 pools with per-kv-head float32
 * k_scale / v_scale [Hk] (DEVICE), used by both the store and the decode. */
PD_API pd_status pd_decode_step_fp8(const void* key, const void* value,
                                    const int64_t* slot_mapping, int T,
                                    int64_t key_stride_tok, int64_t value_stride_tok,
                                    void* out, const void* q, void* key_cache,
                                    void* value_cache, const float* k_scale,
                                    const float* v_scale, const int32_t* block_tables,
                                    int max_blocks_per_seq,
                                    const int32_t* context_lens, int B, int H, int Hk,
                                    int D, int S, int NB, int max_context_len,
                                    float scale, void* workspace,
                                    size_t workspace_bytes, pd_dtype dt,
                                    int32_t* dev_err, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Copy-on-write block copies for fork (parallel sampling, beam search):
 * tutorial page section 2.3, BlockManager.cow(): a shared block that is about
 * to be written is duplicated into a fresh block first; nanoPD page "分页KV
 * 缓存": CoW for beam-search and speculative branches.
 *   key_caches, value_caches  DEVICE arrays of L device pointers, one pool
 *                             [NB][Hk][S][D] per layer
 *   block_mapping  DEVICE int64 [npairs][2] = (src, dst); for every pair and
 *                  every layer the whole block (all heads, all S offsets) of
 *                  K and of V is copied.  Ids outside [0, NB) skip the pair
 *                  and flag PD_DEVERR_BLOCK_RANGE.  A dst that is also a src
 *                  of another pair, or two pairs with one dst, race.
 * dt may also be PD_FP8_E4M3 (one-byte pools).
 * A bit copy.  npairs == 0 or L == 0 launches nothing. */
PD_API pd_status pd_copy_blocks(void* const* key_caches, void* const* value_caches,
                         int L, const int64_t* block_mapping, int npairs,
                         int Hk, int D, int S, int NB, pd_dtype dt,
                         int32_t* dev_err, cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* KV hand-over between a prefill worker and a decode worker (nanoPD page,
 * "异步KV传输": the KV of a finished prefill moves to the decode side on a
 * stream of its own; essay page "LLM推理PD分离架构深度工程实践", section 3.1:
 * layer-by-layer transfer, so the receiver can start on the first layers while
 * later ones are in flight).
 * pd_kv_pack gathers whole blocks of every layer into one contiguous staging
 * buffer, layer-major:
 *   staging[l][0 = K, 1 = V][i][Hk][S][D] = pool_l[block_ids[i]]
 * so layer l is the run of 2 * nblk * Hk*S*D elements that starts at element
 * l * 2 * nblk * Hk*S*D.  pd_kv_unpack is the inverse: it writes each staged
 * slab into block block_ids[i] of the (receiving) pools.
 *   staging       device, 16-byte aligned, L * 2 * nblk * Hk*S*D elements
 *   key_caches, value_caches  DEVICE arrays of L device pointers, one pool
 *                 [NB][Hk][S][D] per layer (as for pd_copy_blocks)
 *   block_ids     DEVICE int32 [nblk]; an id outside [0, NB) skips its slabs
 *                 (pack leaves them untouched, unpack does not read them) and
 *                 flags PD_DEVERR_BLOCK_RANGE.  For unpack, two equal ids race.
 * dt may also be PD_FP8_E4M3 (one-byte pools and staging).
 * Bit copies.  nblk == 0 or L == 0 launches nothing. */
PD_API pd_status pd_kv_pack(void* staging, void* const* key_caches,
                            void* const* value_caches, int L,
                            const int32_t* block_ids, int nblk, int Hk, int D,
                            int S, int NB, pd_dtype dt, int32_t* dev_err,
                            cudaStream_t stream);
PD_API pd_status pd_kv_unpack(const void* staging, void* const* key_caches,
                              void* const* value_caches, int L,
                              const int32_t* block_ids, int nblk, int Hk, int D,
                              int S, int NB, pd_dtype dt, int32_t* dev_err,
                              cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Chunked-prefill attention (nanoPD page "分块预填充": long prompts are cut
 * into chunks interleaved with decode; tutorial page section 5.2): sequence
 * i appends a chunk of C_i query tokens after P_i cached tokens; its chunk
 * K/V are stored beforehand (pd_reshape_and_cache), so the context holds
 * ctx_i = P_i + C_i tokens.  Query j of the chunk (position P_i + j) attends
 * causally to keys 0 .. P_i + j:
 *   out[tok][h][:] = sum_{t <= P_i + j} softmax_t(scale * q[tok][h] . k_t) v_t
 *   q, out        packed [total_q][H][D]; sequence i's tokens are rows
 *                 cu_q_lens[i] .. cu_q_lens[i+1]-1
 *   cu_q_lens     int32 [B + 1], non-decreasing, cu_q_lens[B] <= total_q
 *                 (checked on device: PD_DEVERR_CTX_RANGE, sequence skipped)
 *   max_q_len     >= every C_i (sizes the launch grid)
 *   context_lens  int32 [B] = P_i + C_i (>= C_i; checked on device)
 * QK^T and PV run on the tensor cores (tcgen05, fp32 accumulation in tensor
 * memory); probabilities are rounded to the element type before PV.
 * scale must be positive and finite. */
PD_API pd_status pd_paged_prefill_chunk(void* out, const void* q, int total_q,
                                 const int32_t* cu_q_lens, int max_q_len,
                                 const void* key_cache, const void* value_cache,
                                 const int32_t* block_tables,
                                 int max_blocks_per_seq,
                                 const int32_t* context_lens, int B, int H,
                                 int Hk, int D, int S, int NB, float scale,
                                 pd_dtype dt, int32_t* dev_err,
                                 cudaStream_t stream);

/* ---------------------------------------------------------------------- */
/* Host-side block manager (tutorial page section 2.3, BlockManager and
 * Sequence): ref-counted physical blocks, copy-on-write and fork.  Pure host
 * code, no CUDA calls; not thread-safe (one manager per thread).
 * Allocation order is part of the contract: the free list starts as
 * 0 .. num_blocks-1, allocation takes its last id, freeing appends. */
typedef struct pd_bm pd_bm;

/* NULL on bad sizes (num_blocks < 1, block_size < 1) or out of memory. */
PD_API pd_bm* pd_bm_create(int num_blocks, int block_size);
PD_API void pd_bm_destroy(pd_bm* bm);
/* New empty sequence.  PD_ERR_INVALID_ARG if seq_id is in use or < 0. */
PD_API pd_status pd_bm_add_seq(pd_bm* bm, int seq_id);
/* Reserve the slot of the sequence's next token: a new block at a block
 * boundary, else copy-on-write of a shared last block.  *slot_out gets
 * block*S + offset; *cow_src_out / *cow_dst_out get the block copy the
 * caller must apply on the device (pd_copy_blocks) before storing, or -1.
 * PD_ERR_NO_FREE_BLOCK leaves the sequence unchanged. */
PD_API pd_status pd_bm_append_slot(pd_bm* bm, int seq_id, int64_t* slot_out,
                            int32_t* cow_src_out, int32_t* cow_dst_out);
/* Child shares every block of the parent (ref count + 1), copying nothing. */
PD_API pd_status pd_bm_fork(pd_bm* bm, int parent_id, int child_id);
/* Drop the sequence, one reference from each of its blocks. */
PD_API pd_status pd_bm_release(pd_bm* bm, int seq_id);
/* Copy the sequence's block table into out[0 .. cap); *n_out = its length
 * (PD_ERR_INVALID_ARG if cap is too small; *n_out still set). */
PD_API pd_status pd_bm_block_table(const pd_bm* bm, int seq_id, int32_t* out,
                            int cap, int* n_out);
/* Number of tokens of a sequence (-1 if unknown). */
PD_API int64_t pd_bm_seq_len(const pd_bm* bm, int seq_id);
/* Blocks in use / pool size. */
PD_API double pd_bm_usage(const pd_bm* bm);
/* Ref count of a block (-1 if out of range). */
PD_API int pd_bm_ref_count(const pd_bm* bm, int block_id);
/* Free blocks left. */
PD_API int pd_bm_num_free(const pd_bm* bm);
/* A new sequence whose first nblocks blocks are existing blocks (a cached
 * prefix, tutorial page section 4): each gets one more reference, nothing is
 * copied; its length is `length` tokens (within the last given block).  The
 * blocks must be in use (ref count >= 1).  Later appends follow the usual
 * rules (a shared, partly filled last block is copied on write). */
PD_API pd_status pd_bm_add_seq_shared(pd_bm* bm, int seq_id,
                                      const int32_t* blocks, int nblocks,
                                      int64_t length);
/* One more / one fewer reference on a block in use, held by a holder that
 * is not a sequence (the prefix cache); the last drop frees the block. */
PD_API pd_status pd_bm_retain(pd_bm* bm, int block_id);
PD_API pd_status pd_bm_drop(pd_bm* bm, int block_id);

/* ---------------------------------------------------------------------- */
/* Prefix cache: the hash chain of the tutorial page "LLM 推理服务引擎深度拆
 * 解", section 4.2 / 4.3.  A prompt is cut into full blocks of block_size
 * tokens; block i's key is the first 32 hex digits of
 *   sha256(parent + tokens + extra)
 * with parent = key of block i-1 ("ROOT" for block 0), tokens = the block's
 * ids in decimal joined by ",", extra = caller string (NULL = "").  The table
 * maps key -> physical block id, holds at most capacity_blocks entries and
 * evicts the least recently used key.  Host only. */
typedef struct pd_pc pd_pc;
PD_API pd_pc* pd_pc_create(int capacity_blocks, int block_size);
PD_API void pd_pc_destroy(pd_pc* pc);
/* Keys of every full block of token_ids[0..n) and the longest cached prefix.
 *   hit_tokens      tokens of the longest cached prefix (multiple of
 *                   block_size): blocks up to the first key not in the table
 *   chain_out       [n / block_size][33]: all n / block_size keys,
 *                   NUL-terminated (*n_chain = n / block_size), so that one
 *                   pd_pc_insert can cache the whole prompt
 *   hit_blocks_out  [n / block_size] (may be NULL): block ids of the hits
 * Touches every hit key; counts one hit (hit_tokens > 0) or one miss. */
PD_API pd_status pd_pc_lookup(pd_pc* pc, const int32_t* token_ids, int n,
                              const char* extra, int* hit_tokens,
                              char* chain_out, int32_t* hit_blocks_out,
                              int* n_chain);
/* Map chain[i] -> block_ids[i] for keys not yet held (evicting the least
 * recently used key when full) and touch every key of the chain.  The ids
 * of evicted entries go to evicted_out ([n_chain], may be NULL), their count
 * to *n_evicted: the caller drops its references on them. */
PD_API pd_status pd_pc_insert(pd_pc* pc, const char* chain, int n_chain,
                              const int32_t* block_ids, int32_t* evicted_out,
                              int* n_evicted);
PD_API int pd_pc_size(const pd_pc* pc);
PD_API int64_t pd_pc_hits(const pd_pc* pc);
PD_API int64_t pd_pc_misses(const pd_pc* pc);

#ifdef __cplusplus
}
#endif

#endif /* PD_ATTN_H */
