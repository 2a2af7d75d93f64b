// decode.cu -- paged decode attention, split-context.
//
// Operation (nanoPD page, "自定义CUDA分页注意力内核"; paging per the tutorial
// page "LLM 推理服务引擎深度拆解", section 2.2; GQA per the essay page
// "LLM推理PD分离架构深度工程实践", section 6.2):
//   out[i][h] = sum_{t < ctx_i} softmax_t(scale * q[i][h] . k_t) v_t,
//   k_t, v_t read from kv head h / G through block_tables[i][t / S].
//
// Decode is HBM-bound (about one FLOP per byte per query head, tutorial page
// section 1.1): the design streams every K/V byte once and keeps the
// instruction count per byte low enough that issue never caps bandwidth.
//  * grid = (kv head x head group, sequence, partition); a partition is a
//    fixed run of kPart logical tokens, so long contexts spread over SMs;
//  * one producer warp gathers the partition's K and V blocks with 2-D TMA
//    boxes ([S tokens][64 dims], 128-byte swizzle) through the block table
//    into a 3-stage shared-memory ring of 64-token stages (two CTAs per SM);
//  * four consumer warps take 16 tokens of each stage.  The G query heads
//    that share the kv head form the N = 8 side of warp-level tensor-core
//    products (mma.sync m16n8k16, fp32 accumulation): S^T = K q^T for 16
//    tokens, then O^T += V^T P^T.  The fragment layouts line up so each lane
//    owns the same two heads in S and in O: the online softmax (log2 domain,
//    lazy rescaling when a max grows by more than 2^8) needs only three
//    shuffle steps per head pair and no broadcasts; P is transposed into
//    operand layout with movmatrix;
//  * P enters the product as an unevaluated pair of 16-bit values
//    (hi = rn(p), lo = rn(p - hi)), two MMAs per tile, so P carries about
//    2^-17 relative error instead of the 2^-9 of a single bf16;
//  * the four warps merge in shared memory; a batch that fits one partition
//    writes `out` directly, otherwise partial (max, sum, unnormalised o) go
//    to the workspace and a reduce kernel, launched programmatically
//    dependent, merges them in fixed partition order.  No atomics touch
//    results: outputs are bit-identical for any placement of blocks.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "pd_device.cuh"
#include "pd_internal.h"
#include "pd_mma.cuh"
#include "pd_tcgen05.cuh"
#include "pd_tmap.h"

namespace pd {
namespace {

constexpr int kPart = 256;          // tokens per partition (multiple of the stage)
constexpr int kStageTokens = 64;    // tokens per pipeline stage
constexpr int kStages = 3;          // ring depth
constexpr int kConsumerWarps = 4;   // 16 tokens of each stage per warp
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kHeadsN = 8;          // MMA N: query heads per CTA, padded
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when max grows > 2^8
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DecodeSmem {
    static constexpr int kAtom = kStageTokens * 128;   // [64 tokens][64 values], 8 KB
    static constexpr int kTile = (D / 64) * kAtom;     // one stage of K (or of V)
    static constexpr int kFrag = (D / 16) * 4 + 4;     // per-lane merge record: o, m[2], l[2]
    static constexpr int kK = 0;
    static constexpr int kV = kK + kStages * kTile;
    static constexpr int kX = kV + kStages * kTile;    // merge exchange float [2][kFrag][32]
    static constexpr int kBar = kX + 2 * kFrag * 32 * 4;
    static constexpr int kMisc = kBar + 2 * kStages * 8;   // abort flag, issued count
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;           // base aligned to 1 KB in-kernel
};

// Shared address of 16-byte chunk `chunk` (of D/8) of token row `tok` in a
// stage laid out as 64-value swizzle atoms ([64 rows][128 B], chunk c of row
// r stored at position c ^ (r % 8)).
template <int D>
__device__ __forceinline__ uint32_t swz(uint32_t base, int tok, int chunk) {
    return base + (chunk >> 3) * DecodeSmem<D>::kAtom + tok * 128 +
           (((chunk & 7) ^ (tok & 7)) << 4);
}

// A work item is (partition, sequence, unit) with unit = (kv head, head group);
// the same enumeration drives the producer and the consumers.
struct Item {
    int part, seq, unit, t_begin, t_end, n_stages;
};

__device__ __forceinline__ Item decode_item(long item, int units, int B,
                                            const int32_t* __restrict__ context_lens, int cap,
                                            int32_t* dev_err, bool flag) {
    Item it;
    it.unit = int(item % units);
    const long rest = item / units;
    it.seq = int(rest % B);
    it.part = int(rest / B);
    int ctx = __ldg(context_lens + it.seq);
    if (ctx > cap || ctx < 0) {
        // context longer than the table / workspace promise: cut to what they hold
        if (flag && it.part == 0 && it.unit == 0) flag_error(dev_err, PD_DEVERR_CTX_RANGE);
        ctx = ctx < 0 ? 0 : cap;
    }
    it.t_begin = it.part * kPart;
    it.t_end = min(ctx, it.t_begin + kPart);
    it.n_stages = it.t_end > it.t_begin ? (it.t_end - it.t_begin + kStageTokens - 1) / kStageTokens
                                        : 0;
    return it;
}

// OR of `pred` over the consumer warps (named barrier 1), uniform result.
__device__ __forceinline__ bool consumers_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"(uint32_t(pred)), "n"(kConsumerWarps * 32) : "memory");
    return r != 0;
}

// Persistent: each CTA walks items blockIdx.x, blockIdx.x + gridDim.x, ...
template <typename T, int D>
__global__ void __launch_bounds__(kDecodeThreads, 2)
paged_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, T* __restrict__ out,
                          const T* __restrict__ q, const int32_t* __restrict__ block_tables,
                          int max_blocks_per_seq, const int32_t* __restrict__ context_lens,
                          int B, int H, int Hk, int S, int NB, int GH, float scale_log2,
                          int num_parts_max, float* __restrict__ ws_o,
                          float* __restrict__ ws_m, float* __restrict__ ws_l,
                          int32_t* dev_err) {
    using L = DecodeSmem<D>;
    using E = Elem<T>;
    constexpr int kAtoms = D / 64;
    constexpr int KS = D / 16;      // k-steps of q.k, m-tiles of p.v
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* xchg = reinterpret_cast<float*>(smem + L::kX);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint64_t* empty = full + kStages;
    volatile int32_t* abort_flag = reinterpret_cast<int32_t*>(smem + L::kMisc);
    volatile int32_t* issued = reinterpret_cast<int32_t*>(smem + L::kMisc + 4);

    pdl_launch_dependents();

    const int G = H / Hk;
    const int groups = G / GH;
    const int units = Hk * groups;
    const long n_items = long(num_parts_max) * B * units;
    const int cap = min(max_blocks_per_seq * S, num_parts_max * kPart);
    const bool direct = (num_parts_max == 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        *issued = 0;
        fence_mbar_init();
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer warp: streams stages across items ----------------
        const uint32_t block_bytes = uint32_t(S) * D * 2;        // one [S][D] slab
        uint32_t gs = 0;                                         // stages issued so far
        bool stop = false;
        for (long item = blockIdx.x; item < n_items && !stop; item += gridDim.x) {
            const Item it = decode_item(item, units, B, context_lens, cap, dev_err, false);
            if (it.n_stages == 0) continue;
            const int kvh = it.unit / groups;
            const int32_t* bt_row = block_tables + (int64_t)it.seq * max_blocks_per_seq;
            for (int st = 0; st < it.n_stages; ++st, ++gs) {
                const int slot = gs % kStages;
                // every lane waits (acquire), then the warp agrees on the outcome
                const bool ok = __all_sync(0xffffffffu, gs < kStages ||
                                           mbar_wait(&empty[slot], ((gs / kStages) - 1) & 1));
                if (!ok || __any_sync(0xffffffffu, *abort_flag != 0)) {
                    if (lane == 0 && !ok) {
                        flag_error(dev_err, PD_DEVERR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    stop = true;
                    break;
                }
                const int t0 = it.t_begin + st * kStageTokens;
                const int nt = min(kStageTokens, it.t_end - t0);
                const int nblk = (nt + S - 1) / S;             // <= 64 / S <= 8
                int row = -1;
                if (lane < nblk) {
                    const int blk = __ldg(bt_row + t0 / S + lane);
                    if (blk >= 0 && blk < NB) {
                        row = (blk * Hk + kvh) * S;
                    } else {
                        flag_error(dev_err, PD_DEVERR_BLOCK_RANGE);
                    }
                }
                const uint32_t ok_mask = __ballot_sync(0xffffffffu, row >= 0);
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[slot], 2u * block_bytes * __popc(ok_mask));
                __syncwarp();
                if (row >= 0) {
#pragma unroll
                    for (int a = 0; a < kAtoms; ++a) {
                        const int off = slot * L::kTile + a * L::kAtom + lane * S * 128;
                        tc::tma_load_2d(smem + L::kK + off, &tm_k, a * 64, row, &full[slot]);
                        tc::tma_load_2d(smem + L::kV + off, &tm_v, a * 64, row, &full[slot]);
                    }
                }
                if (lane == 0) *issued = int(gs + 1);
            }
        }
        return;
    }

    // ---------------- consumer warps ----------------
    const int j8 = lane >> 3, r8 = lane & 7;     // ldmatrix: matrix index, row within it
    const int tb = warp * 16;                    // this warp's tokens within a stage
    const uint32_t k_base0 = smem_u32(smem + L::kK);
    const uint32_t v_base0 = smem_u32(smem + L::kV);
    const float2 neg1 = make_float2(-1.f, -1.f);
    uint32_t gs = 0;                             // stages consumed so far
    bool aborted = false;

    for (long item = blockIdx.x; item < n_items; item += gridDim.x) {
        const Item it = decode_item(item, units, B, context_lens, cap, dev_err, warp == 0);
        const int kvh = it.unit / groups;
        const int h0 = kvh * G + (it.unit % groups) * GH;     // first q head of this unit
        if (it.n_stages == 0) {
            // Nothing to attend to.  A zero-length context still owes zeros.
            if (it.part == 0 && warp == 0) {
                if (direct) {
                    for (int idx = lane; idx < GH * D / 2; idx += 32) {
                        const int h = idx / (D / 2), d2 = idx % (D / 2);
                        reinterpret_cast<uint32_t*>(out + ((int64_t)it.seq * H + h0 + h) * D)[d2] = 0u;
                    }
                } else if (lane < GH) {
                    const int64_t r = ((int64_t)it.seq * H + h0 + lane) * num_parts_max;
                    ws_m[r] = -INFINITY;     // the reduce kernel sees an empty row
                    ws_l[r] = 0.f;
                }
            }
            continue;
        }
        // q^T as the MMA B operand: lane holds head lane/4, dims 16ks + 2(lane%4) + {0,1}
        // (register 0) and the same + 8 (register 1); heads past GH are zero.
        uint32_t qb[KS][2];
        {
            const int n = lane >> 2;
            const T* qrow = q + ((int64_t)it.seq * H + h0 + n) * D + 2 * (lane & 3);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                qb[ks][0] = n < GH ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks)) : 0u;
                qb[ks][1] =
                    n < GH ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8)) : 0u;
            }
        }
        // O^T fragments: m-tile mt covers dims 16mt..16mt+15; lane holds dims
        // 16mt + lane/4 (regs 0,1) and + 8 (regs 2,3), heads 2(lane%4) and + 1.
        float o[KS][4];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};

        for (int st = 0; st < it.n_stages; ++st, ++gs) {
            const int slot = gs % kStages;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (gs / kStages) & 1))) {
                if (lane == 0) {
                    flag_error(dev_err, PD_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                aborted = true;
                break;                   // skip the item's other stages
            }
            const int nt = min(kStageTokens, it.t_end - (it.t_begin + st * kStageTokens));
            if (tb < nt) {
                const uint32_t kb = k_base0 + slot * L::kTile;
                const uint32_t vb = v_base0 + slot * L::kTile;
                const bool partial = tb + 16 > nt;
                if (partial) {
                    // V rows past the partition end hold other data or were never
                    // loaded this round: zero them so that 0 * v stays 0.
                    unsigned char* vrow = smem + L::kV + slot * L::kTile;
                    for (int i = lane; i < 16 * kAtoms * 8; i += 32) {
                        const int tok = tb + i / (kAtoms * 8);
                        if (tok >= nt) {
                            const int a = (i / 8) % kAtoms, c = i % 8;
                            *reinterpret_cast<uint4*>(vrow + a * L::kAtom + tok * 128 + c * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    __syncwarp();
                }
                // ---- S^T[16 tokens][8 heads] = K q^T (two accumulators for ILP)
                float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t a[4];
                    wmma16::ldsm_x4(a, swz<D>(kb, tb + r8 + 8 * (j8 & 1), 2 * ks + (j8 >> 1)));
                    wmma16::Mma<T>::run(acc[ks & 1], a, qb[ks][0], qb[ks][1]);
                }
                // lane holds tokens tb + lane/4 (0,1) and + 8 (2,3); heads 2(lane%4) + {0,1}
                const int tok0 = tb + (lane >> 2);
                float x[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int tok = tok0 + (i >> 1) * 8;
                    x[i] = tok < nt ? (acc[0][i] + acc[1][i]) * scale_log2 : -INFINITY;
                }
                // ---- online softmax per head (lane-local state, 3 shuffles per head)
                float mx[2] = {fmaxf(x[0], x[2]), fmaxf(x[1], x[3])};
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], off));
                    mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], off));
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (mx[h] > m_run[h] + kRescaleThreshold) {
                        const float alpha = ex2(m_run[h] - mx[h]);   // 0 the first time
                        m_run[h] = mx[h];
                        l_run[h] *= alpha;
#pragma unroll
                        for (int mt = 0; mt < KS; ++mt) {
                            o[mt][h] *= alpha;
                            o[mt][2 + h] *= alpha;
                        }
                    }
                }
                const float p0 = ex2(x[0] - m_run[0]), p1 = ex2(x[1] - m_run[1]);
                const float p2 = ex2(x[2] - m_run[0]), p3 = ex2(x[3] - m_run[1]);
                l_run[0] += p0 + p2;
                l_run[1] += p1 + p3;
                // P as hi + lo 16-bit pairs, transposed into B-operand layout
                const uint32_t hi0 = E::pack2(p0, p1), hi1 = E::pack2(p2, p3);
                const float2 lo0 = ffma2(E::unpack2(hi0), neg1, make_float2(p0, p1));
                const float2 lo1 = ffma2(E::unpack2(hi1), neg1, make_float2(p2, p3));
                const uint32_t bh0 = wmma16::movm_t(hi0), bh1 = wmma16::movm_t(hi1);
                const uint32_t bl0 = wmma16::movm_t(E::pack2(lo0.x, lo0.y));
                const uint32_t bl1 = wmma16::movm_t(E::pack2(lo1.x, lo1.y));
                // ---- O^T[dims][heads] += V^T P^T
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
                    uint32_t a[4];
                    wmma16::ldsm_x4_t(a, swz<D>(vb, tb + r8 + 8 * (j8 >> 1), 2 * mt + (j8 & 1)));
                    wmma16::Mma<T>::run(o[mt], a, bh0, bh1);
                    wmma16::Mma<T>::run(o[mt], a, bl0, bl1);
                }
                if (partial) tc::fence_proxy_async_smem();   // zeros before the next TMA write
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        // All four consumer warps decide together whether to go on: a warp
        // that gave up still arrives here, so named-barrier counts stay matched.
        if (consumers_any(aborted || *abort_flag != 0)) {
            aborted = true;
            break;
        }

        // ---- merge the four warps in registers through a fragment-order buffer:
        // warps 2, 3 hand over to 0, 1, then warp 1 to warp 0.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 4);
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 8);
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 16);
        }
        auto put = [&](int buf) {
            float* x = xchg + buf * L::kFrag * 32 + lane;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) x[(mt * 4 + e) * 32] = o[mt][e];
            x[(KS * 4 + 0) * 32] = m_run[0];
            x[(KS * 4 + 1) * 32] = m_run[1];
            x[(KS * 4 + 2) * 32] = l_run[0];
            x[(KS * 4 + 3) * 32] = l_run[1];
        };
        auto take = [&](int buf) {
            const float* x = xchg + buf * L::kFrag * 32 + lane;
            float c_mine[2], c_other[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float mo = x[(KS * 4 + h) * 32], lo = x[(KS * 4 + 2 + h) * 32];
                const float M = fmaxf(m_run[h], mo);
                c_mine[h] = m_run[h] == -INFINITY ? 0.f : ex2(m_run[h] - M);
                c_other[h] = mo == -INFINITY ? 0.f : ex2(mo - M);
                l_run[h] = l_run[h] * c_mine[h] + lo * c_other[h];
                m_run[h] = M;
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[mt][e] = o[mt][e] * c_mine[e & 1] + x[(mt * 4 + e) * 32] * c_other[e & 1];
        };
        if (warp >= 2) put(warp - 2);
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
        if (warp < 2) take(warp);
        if (warp == 1) {
            __syncwarp();
            put(1);                      // own partner slot, already read by this warp
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
        if (warp == 0) {
            take(1);
            // lane: heads ha, ha + 1; dims 16mt + lane/4 and + 8
            const int ha = 2 * (lane & 3), d0 = lane >> 2;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int hh = ha + h;
                if (hh >= GH) continue;
                const int hq = h0 + hh;
                if (direct) {
                    const float inv = 1.f / l_run[h];
                    T* orow = out + ((int64_t)it.seq * H + hq) * D + d0;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        orow[16 * mt] = T(o[mt][h] * inv);
                        orow[16 * mt + 8] = T(o[mt][2 + h] * inv);
                    }
                } else {
                    const int64_t r = ((int64_t)it.seq * H + hq) * num_parts_max + it.part;
                    float* wrow = ws_o + r * D + d0;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        wrow[16 * mt] = o[mt][h];
                        wrow[16 * mt + 8] = o[mt][2 + h];
                    }
                    if (d0 == 0) {
                        ws_m[r] = m_run[h];
                        ws_l[r] = l_run[h];
                    }
                }
            }
        }
        // the exchange buffer is rewritten by the next item's merge
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    }

    if (aborted) {
        // Let copies already issued into the ring land before the CTA exits.
        if (threadIdx.x == 0) {
            const int n_issued = *issued;
            for (int s2 = int(gs); s2 < n_issued; ++s2)
                if (!mbar_wait(&full[s2 % kStages], (s2 / kStages) & 1)) break;
        }
    }
}

// Merge the partitions of each (sequence, q head): one warp per row, fixed
// partition order.  M = max_p m_p; out = sum_p o_p 2^(m_p - M) / sum_p l_p 2^(m_p - M).
constexpr int kReduceWarps = 4;

template <typename T, int D>
__global__ void __launch_bounds__(kReduceWarps * 32)
paged_decode_reduce_kernel(T* __restrict__ out, const int32_t* __restrict__ context_lens,
                           int B, int H, int num_parts_max, int cap,
                           const float* __restrict__ ws_o, const float* __restrict__ ws_m,
                           const float* __restrict__ ws_l) {
    using E = Elem<T>;
    constexpr int DV = D / 32;
    pdl_wait_primary();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * kReduceWarps + warp;
    if (row >= int64_t(B) * H) return;
    const int seq = int(row / H);
    int ctx = __ldg(context_lens + seq);
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    const int np = (ctx + kPart - 1) / kPart;
    const float* m = ws_m + row * num_parts_max;
    const float* l = ws_l + row * num_parts_max;
    float M = -INFINITY;
    for (int p = lane; p < np; p += 32) M = fmaxf(M, m[p]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[DV];
#pragma unroll
    for (int e = 0; e < DV; ++e) acc[e] = 0.f;
    float lsum = 0.f;
    for (int p0 = 0; p0 < np; p0 += 32) {
        const int p = p0 + lane;
        const float w = p < np ? ex2(m[p] - M) : 0.f;
        lsum += p < np ? l[p] * w : 0.f;
        const int n = min(32, np - p0);
        for (int u = 0; u < n; ++u) {
            const float wu = __shfl_sync(0xffffffffu, w, u);
            const float* o = ws_o + (row * num_parts_max + p0 + u) * D + lane * DV;
            if constexpr (DV == 4) {
                const float4 v = *reinterpret_cast<const float4*>(o);
                acc[0] += v.x * wu; acc[1] += v.y * wu; acc[2] += v.z * wu; acc[3] += v.w * wu;
            } else {
                const float2 v = *reinterpret_cast<const float2*>(o);
                acc[0] += v.x * wu; acc[1] += v.y * wu;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    const float inv = np > 0 ? 1.f / lsum : 0.f;
    uint32_t* dst = reinterpret_cast<uint32_t*>(out + row * D + lane * DV);
#pragma unroll
    for (int e = 0; e < DV / 2; ++e) dst[e] = E::pack2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
    size_t o, m, l, total;
};

WsLayout ws_layout(int B, int H, int D, int P) {
    WsLayout w;
    const size_t rows = size_t(B) * H * P;
    w.o = 0;
    w.m = align256(rows * D * sizeof(float));
    w.l = w.m + align256(rows * sizeof(float));
    w.total = w.l + align256(rows * sizeof(float));
    return w;
}

int sm_count(int dev) {
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

template <typename T, int D>
pd_status launch_decode_t(const DecodeArgs& a) {
    using Lt = DecodeSmem<D>;
    const int P = decode_num_partitions(a.max_context_len);
    const int G = a.H / a.Hk;
    int GH = 1;                          // largest divisor of G that fits N = 8
    for (int g = std::min(G, kHeadsN); g >= 1; --g)
        if (G % g == 0) { GH = g; break; }
    const int groups = G / GH;
    CUtensorMap tm_k, tm_v;
    const unsigned long long rows = (unsigned long long)a.NB * a.Hk * a.S;
    if (rows > 0x7fffffffull) return PD_ERR_UNSUPPORTED;   // TMA row coordinate is int32
    if (!encode_pool_map(&tm_k, a.key_cache, D, rows, a.S, a.dt) ||
        !encode_pool_map(&tm_v, a.value_cache, D, rows, a.S, a.dt))
        return launch_result(cudaErrorInvalidValue);
    auto kern = paged_decode_split_kernel<T, D>;
    static uint64_t attr_set = 0;   // one bit per device; benign if raced
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return launch_result(e0);
    if (dev >= 64 || !((attr_set >> dev) & 1)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Lt::kAlloc);
        if (e != cudaSuccess) return launch_result(e);
        if (dev < 64) attr_set |= uint64_t(1) << dev;
    }
    float* ws_o = nullptr;
    float* ws_m = nullptr;
    float* ws_l = nullptr;
    if (P > 1) {
        const WsLayout w = ws_layout(a.B, a.H, a.D, P);
        char* base = static_cast<char*>(a.workspace);
        ws_o = reinterpret_cast<float*>(base + w.o);
        ws_m = reinterpret_cast<float*>(base + w.m);
        ws_l = reinterpret_cast<float*>(base + w.l);
    }
    const float scale_log2 = a.scale * kLog2e;
    // Persistent grid: two CTAs per SM (shared memory bound), never more CTAs
    // than work items.
    const long n_items = long(P) * a.B * a.Hk * groups;
    const long grid = std::min<long>(n_items, 2L * sm_count(dev));
    kern<<<unsigned(grid), kDecodeThreads, Lt::kAlloc, a.stream>>>(
        tm_k, tm_v, static_cast<T*>(a.out), static_cast<const T*>(a.q), a.block_tables,
        a.max_blocks_per_seq, a.context_lens, a.B, a.H, a.Hk, a.S, a.NB, GH, scale_log2, P,
        ws_o, ws_m, ws_l, a.dev_err);
    pd_status st = launch_result(cudaGetLastError());
    if (st != PD_OK || P == 1) return st;

    // Reduce, launched as a programmatic dependent of the split kernel so its
    // launch overlaps the split kernel's tail.
    const int cap = std::min(a.max_blocks_per_seq * a.S, P * kPart);
    cudaLaunchConfig_t cfg = {};
    const int64_t nrows = int64_t(a.B) * a.H;
    cfg.gridDim = dim3(unsigned((nrows + kReduceWarps - 1) / kReduceWarps));
    cfg.blockDim = dim3(kReduceWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, paged_decode_reduce_kernel<T, D>,
                                       static_cast<T*>(a.out), a.context_lens, a.B, a.H, P, cap,
                                       static_cast<const float*>(ws_o),
                                       static_cast<const float*>(ws_m),
                                       static_cast<const float*>(ws_l));
    return launch_result(e);
}

}  // namespace

int decode_partition_tokens(int max_context_len) {
    (void)max_context_len;
    return kPart;
}

int decode_num_partitions(int max_context_len) {
    if (max_context_len <= 0) return 1;
    return (max_context_len + kPart - 1) / kPart;
}

size_t decode_workspace_bytes(int B, int H, int D, int max_context_len) {
    const int P = decode_num_partitions(max_context_len);
    if (P <= 1) return 0;
    return ws_layout(B, H, D, P).total;
}

pd_status launch_decode(const DecodeArgs& a) {
    if (a.dt == PD_BF16) {
        return a.D == 128 ? launch_decode_t<__nv_bfloat16, 128>(a)
                          : launch_decode_t<__nv_bfloat16, 64>(a);
    }
    return a.D == 128 ? launch_decode_t<__half, 128>(a) : launch_decode_t<__half, 64>(a);
}

}  // namespace pd
