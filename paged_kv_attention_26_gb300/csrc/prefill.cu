// prefill.cu -- chunked-prefill attention over the paged cache on the 5th-gen
// tensor cores (tcgen05 MMA, accumulators in tensor memory, operands staged by
// TMA).
//
// Operation (nanoPD page "分块预填充"; tutorial page "LLM 推理服务引擎深度拆解"
// section 5.2): sequence i appends a chunk of C_i queries after P_i cached
// tokens; query j sees keys 0 .. P_i + j of its own paged context:
//   out = softmax(scale * q K^T) V, causal, GQA head h -> kv head h / G.
// Prefill is a dense contraction (tensor-core bound, essay page
// "LLM推理PD分离架构深度工程实践" section 1), so QK^T and PV run as
// tcgen05.mma with fp32 accumulation in tensor memory.
//
// Tiling.  A CTA owns two 128-row query tiles (A, B) of one kv head group and
// streams 128-key tiles shared by both:
//  * GQA packing: the G' = min(G, 16) query heads that share a kv head are
//    interleaved into each tile (rows = 128/G' tokens x G' heads), so every
//    K/V tile is loaded once for all of them and the causal band is narrow;
//  * warp 0 issues TMA loads: the two Q tiles once (3-D map over
//    [tokens][heads][D]), then per key tile one 2-D box [S rows][64 dims] per
//    K and per V block, gathered through the block table with 128-byte
//    swizzle.  K and V have rings of their own (3 and 2 stages) and K runs
//    one tile ahead of V, matching the order the tensor cores use them in
//    (K of tile t+1 is needed before V of tile t is done), so each load has
//    more than a key tile's worth of time to land;
//  * warp 1 allocates all 512 tensor-memory columns (S_A, O_A, S_B, O_B) and
//    issues every MMA from one thread, alternating the two tiles: PV_A(t),
//    QK_A(t+1), PV_B(t), QK_B(t+1).  While one softmax warpgroup works on
//    its tile, the tensor cores run the other tile's products;
//  * warps 4-7 (tile A) and 8-11 (tile B), one query row per thread, run the
//    online softmax in the log2 domain with lazy rescaling (the accumulator
//    O is rescaled only when a row max grows by more than 2^8), reading the
//    S row from tensor memory in 32-column chunks (a max pass, then an
//    exponential pass), and write P over S for the PV product;
//  * P is rounded to 16 bits for the tensor cores.  Where one key can carry a
//    large share of a row's softmax mass (its weight may exceed 1/8), the
//    16-bit rounding error (2^-9 relative for bf16) is not averaged away, so
//    that tile also gets the residual lo = rn(p - hi) as a second PV pass (a
//    key of weight w <= 1/8 moves the output by at most 2^-12 |v| without it,
//    an eighth of the output's own bf16 rounding);
//    rows vote per warp, and the MMA issuer runs the second pass only when
//    some row of the tile asked for it.
// Every wait is bounded; a wait that runs out flags PD_DEVERR_TIMEOUT and the
// CTA drains its in-flight copies and MMAs, frees tensor memory and leaves.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <type_traits>
#include <cmath>

#include "pd_device.cuh"
#include "pd_internal.h"
#include "pd_tcgen05.cuh"
#include "pd_tmap.h"

namespace pd {
namespace {

constexpr int kTileM = 128;            // query rows per tile (MMA M)
constexpr int kTileN = 128;            // keys per tile
constexpr int kKStages = 3;
constexpr int kVStages = 2;             // the MMA issuer indexes V stages as t & 1
constexpr int kPrefillThreads = 384;   // warp 0 TMA, 1 MMA, 2-3 spare, 4-7 / 8-11 softmax A / B
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 512;    // S_A [0,128) O_A [128,256) S_B [256,384) O_B [384,512)
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLoWeight = 1.0f / 8.0f;   // weight above which P's rounding is corrected
constexpr float kLog2e = 1.4426950408889634f;
// Register split (384 threads launched at 168 each = 64512): the TMA/MMA
// warpgroup keeps 80, the two softmax warpgroups take 208, which holds a
// whole 128-column S row in registers.  128*80 + 256*208 = 63488 <= 64512.
// (80 / 208 measured 1% faster than 64 / 216.)
constexpr uint32_t kRegsControl = 80;
constexpr uint32_t kRegsSoftmax = 208;
// setmaxnreg.inc waits until enough registers are free: the split must fit
// in what the CTA was launched with (168 per thread at 384 threads).
static_assert(kRegsControl * 128 + kRegsSoftmax * 256 <= 168 * kPrefillThreads,
              "register split exceeds the launch allocation");

template <int D>
struct PrefillSmem {
    static constexpr int kAtom = kTileM * 128;          // 128 rows x 128 B (64 16-bit values)
    static constexpr int kTile = (D / 64) * kAtom;      // a [128][D] tile
    static constexpr int kQ = 0;                         // Q_A, Q_B
    static constexpr int kK = kQ + 2 * kTile;            // kKStages tiles
    static constexpr int kV = kK + kKStages * kTile;     // kVStages tiles
    static constexpr int kBar = kV + kVStages * kTile;
    // barriers: q_full, k_full[3], k_empty[3], v_full[2], v_empty[2],
    // s_full[A,B], p_full[A,B], pv_done[A0,A1,B0,B1], drain
    static constexpr int kNumBars = 20;
    static constexpr int kFlags = kBar + kNumBars * 8;  // int lo_flag[2 tiles][2 parity][4 warps]
    static constexpr int kMisc = kFlags + 16 * 4;       // tmem base, abort flag, K / V issued
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kAlloc = kBytes + 1024 > 116 * 1024 ? kBytes + 1024 : 116 * 1024;
};

template <typename T, int D>
__global__ void __launch_bounds__(kPrefillThreads, 1)
paged_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, T* __restrict__ out, int total_q,
                     const int32_t* __restrict__ cu_q_lens,
                     const int32_t* __restrict__ block_tables, int max_blocks_per_seq,
                     const int32_t* __restrict__ context_lens, int H, int Hk, int S, int NB,
                     int GP, float scale_log2, int32_t* dev_err) {
    using L = PrefillSmem<D>;
    using E = Elem<T>;
    constexpr bool kBf16 = E::kDtype == PD_BF16;
    constexpr uint32_t kIdescQK = tc::idesc_f16(kBf16, kTileM, kTileN, false, false);
    constexpr uint32_t kIdescPV = tc::idesc_f16(kBf16, kTileM, D, false, true);
    constexpr int kAtoms = D / 64;

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;      // [K stage]
    uint64_t* k_empty = bars + 4;     // [K stage]
    uint64_t* v_full = bars + 7;      // [V stage]
    uint64_t* v_empty = bars + 9;     // [V stage]
    uint64_t* s_full = bars + 11;     // [tile]
    uint64_t* p_full = bars + 13;     // [tile]
    // pv_done[tile * 2 + (u & 1)] completes when PV of key tile u (and every
    // earlier MMA) is done.  One barrier per parity keeps each wait within one
    // phase of the barrier's state, which parity waits need.
    uint64_t* pv_done = bars + 15;    // [4]
    uint64_t* drain = bars + 19;
    volatile int32_t* lo_flag = reinterpret_cast<volatile int32_t*>(smem + L::kFlags);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::kMisc);
    volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + L::kMisc + 4);
    volatile int32_t* k_issued = reinterpret_cast<volatile int32_t*>(smem + L::kMisc + 8);
    volatile int32_t* v_issued = reinterpret_cast<volatile int32_t*>(smem + L::kMisc + 12);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Heaviest work first.  Blocks are dispatched in block-index order, so a
    // block reads its z index as a rank among the batch's sequences sorted by
    // causal work C (2P + C) (ties by index) and its x index from the last
    // tile pair down: the last wave then holds the lightest tiles instead of
    // whatever the batch order put there.  Every block ranks the batch
    // itself (the ranks form a permutation whatever the values); batches of
    // more than 256 sequences keep the launch order.
    int seq = blockIdx.z;
    if (gridDim.z > 1 && gridDim.z <= 256) {
        __shared__ int picked;
        auto work = [&](int j) -> long long {
            const int c = __ldg(cu_q_lens + j + 1) - __ldg(cu_q_lens + j);
            const int p = __ldg(context_lens + j) - c;
            return (long long)c * (2LL * p + c);
        };
        const int t = threadIdx.x;
        if (t < int(gridDim.z)) {
            const long long wt = work(t);
            int rank = 0;
            for (int j = 0; j < int(gridDim.z); ++j) {
                const long long wj = work(j);
                rank += (wj > wt || (wj == wt && j < t)) ? 1 : 0;
            }
            if (rank == int(blockIdx.z)) picked = t;
        }
        __syncthreads();
        seq = picked;
    }
    const int TQ = kTileM / GP;                       // query tokens per tile
    const int q_begin = __ldg(cu_q_lens + seq);
    const int C = __ldg(cu_q_lens + seq + 1) - q_begin;
    const int q0 = (gridDim.x - 1 - blockIdx.x) * 2 * TQ;   // first chunk token of tile A
    if (q0 >= C) return;
    const int ctx = __ldg(context_lens + seq);
    const int P = ctx - C;
    if (C < 0 || P < 0 || ctx > max_blocks_per_seq * S || q_begin < 0 ||
        q_begin + C > total_q) {
        if (threadIdx.x == 0) flag_error(dev_err, PD_DEVERR_CTX_RANGE);
        return;
    }
    const int G = H / Hk;
    const int sub = G / GP;
    const int kvh = blockIdx.y / sub;
    const int head0 = kvh * G + (blockIdx.y % sub) * GP;
    const bool has_b = q0 + TQ < C;
    const int n_a = (P + min(C, q0 + TQ) + kTileN - 1) / kTileN;            // key tiles of A
    const int n_b = has_b ? (P + min(C, q0 + 2 * TQ) + kTileN - 1) / kTileN : 0;
    const int n_tiles = max(n_a, n_b);
    const int n_blocks_ctx = (ctx + S - 1) / S;
    const int32_t* bt_row = block_tables + (int64_t)seq * max_blocks_per_seq;

    const uint32_t sQ = smem_u32(smem + L::kQ);
    const uint32_t sK = smem_u32(smem + L::kK);
    const uint32_t sV = smem_u32(smem + L::kV);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&p_full[s], kSoftmaxThreads);
        }
        for (int s = 0; s < 4; ++s) mbar_init(&pv_done[s], 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        *k_issued = 0;
        *v_issued = 0;
        fence_mbar_init();
        tc::prefetch_tmap(&tm_q);
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
    }
    if (warp == 1) {
        tc::tmem_alloc(const_cast<uint32_t*>(tmem_slot), kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4) {
    // One register release for the whole control warpgroup (setmaxnreg is
    // warpgroup-aligned), then the warps take their roles.
    tc::regs_dec<kRegsControl>();
    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, uint32_t(has_b ? 2 : 1) * kTileM * D * 2);
            for (int a = 0; a < kAtoms; ++a) {
                tc::tma_load_3d(smem + L::kQ + a * L::kAtom, &tm_q, a * 64, head0, q_begin + q0,
                                q_full);
                if (has_b)
                    tc::tma_load_3d(smem + L::kQ + L::kTile + a * L::kAtom, &tm_q, a * 64, head0,
                                    q_begin + q0 + TQ, q_full);
            }
        }
        const int blocks_per_tile = kTileN / S;            // 2 .. 16
        // Load key tile t of K (is_v false) or V into its ring stage once the
        // stage is free; false if the CTA must stop.
        auto load = [&](bool is_v, int t) -> bool {
            const int stages = is_v ? kVStages : kKStages;
            const int st = t % stages;
            uint64_t* empty = is_v ? &v_empty[st] : &k_empty[st];
            uint64_t* full = is_v ? &v_full[st] : &k_full[st];
            const bool ok = __all_sync(0xffffffffu,
                                       t < stages || mbar_wait(empty, ((t / stages) - 1) & 1));
            if (!ok || __any_sync(0xffffffffu, *abort_flag != 0)) {
                if (lane == 0 && !ok) {
                    flag_error(dev_err, PD_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                return false;
            }
            int64_t row = -1;
            if (lane < blocks_per_tile) {
                const int lb = t * blocks_per_tile + lane;
                if (lb < n_blocks_ctx) {
                    const int blk = __ldg(bt_row + lb);
                    if (blk >= 0 && blk < NB) {
                        row = ((int64_t)blk * Hk + kvh) * S;
                    } else if (!is_v) {
                        flag_error(dev_err, PD_DEVERR_BLOCK_RANGE);
                    }
                }
            }
            const uint32_t ok_mask = __ballot_sync(0xffffffffu, row >= 0);
            if (lane == 0) mbar_arrive_expect_tx(full, uint32_t(__popc(ok_mask)) * S * D * 2);
            __syncwarp();
            if (row >= 0) {
                unsigned char* dst = smem + (is_v ? L::kV : L::kK) + st * L::kTile + lane * S * 128;
                for (int a = 0; a < kAtoms; ++a)
                    tc::tma_load_2d(dst + a * L::kAtom, is_v ? &tm_v : &tm_k, a * 64,
                                    int32_t(row), full);
            }
            if (lane == 0) *(is_v ? v_issued : k_issued) = t + 1;
            return true;
        };
        // K runs one key tile ahead of V: K0, K1, V0, K2, V1, ...
        if (n_tiles > 0 && load(false, 0)) {
            for (int t = 0; t < n_tiles; ++t) {
                if (t + 1 < n_tiles && !load(false, t + 1)) break;
                if (!load(true, t)) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------ MMA issuer --------------------------------
        // The whole warp runs this loop in step (every decision warp-uniform);
        // one elected lane issues each MMA and commit.
        constexpr uint32_t kHi = tc::sw128_desc_hi(1024);
        constexpr uint32_t kTile16 = uint32_t(L::kTile) >> 4;
        // Descriptor low halves, built once: every operand below is one of
        // these bases plus a constant (byte offset >> 4).
        const uint32_t q_lo = tc::smem_desc_sw128_lo(sQ, 16);
        const uint32_t k_lo = tc::smem_desc_sw128_lo(sK, 16);
        // V as an MN-major operand: N = D contiguous in 64-wide atoms (LBO
        // between them), K = keys at 128 B (SBO per 8 keys)
        const uint32_t v_lo = tc::smem_desc_sw128_lo(sV, L::kAtom);
        auto qk = [&](int x, uint32_t kst) {
            const uint32_t d_s = tmem + uint32_t(x) * 256;
            const uint32_t a0 = q_lo + uint32_t(x) * kTile16;
            const uint32_t b0 = k_lo + kst * kTile16;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t koff = uint32_t((kk >> 2) * L::kAtom + (kk & 3) * 32) >> 4;
                if (kk == 0)
                    tc::mma_ss_warp<false>(d_s, a0 + koff, kHi, b0 + koff, kHi, kIdescQK);
                else
                    tc::mma_ss_warp<true>(d_s, a0 + koff, kHi, b0 + koff, kHi, kIdescQK);
            }
            tc::commit_warp(&s_full[x]);
        };
        auto pv = [&](int x, int t, uint32_t vst) {
            // second pass when any of the four softmax warps asked for it
            const int32_t* f = const_cast<const int32_t*>(lo_flag) + x * 8 + (t & 1) * 4;
            const bool lo = (f[0] | f[1] | f[2] | f[3]) != 0;
            const uint32_t d_o = tmem + uint32_t(x) * 256 + 128;
            const uint32_t p0 = tmem + uint32_t(x) * 256;
            const uint32_t b0 = v_lo + vst * kTile16;
            // P over S: chunk c (keys 32c..32c+31) holds hi in columns
            // 32c..32c+15 and lo in 32c+16..32c+31
            for (int pass = 0; pass < (lo ? 2 : 1); ++pass) {
#pragma unroll
                for (int kk = 0; kk < kTileN / 16; ++kk)
                    tc::mma_ts_warp(d_o, p0 + uint32_t(32 * (kk >> 1) + 8 * (kk & 1) + 16 * pass),
                                    b0 + uint32_t(kk * 16 * 128 / 16), kHi, kIdescPV,
                                    uint32_t(t > 0 || kk > 0 || pass > 0));
            }
            tc::commit_warp(&pv_done[x * 2 + (t & 1)]);
        };
        bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0));
        if (ok && n_tiles > 0 && (ok = __all_sync(0xffffffffu, mbar_wait(&k_full[0], 0)))) {
            tc::fence_after_sync();
            if (n_a > 0) qk(0, 0);
            if (n_b > 0) qk(1, 0);
            tc::commit_warp(&k_empty[0]);
        }
        // Ring positions tracked incrementally: K of tile u = t + 1 in stage
        // kst with phase parity kpar; V of tile t in stage t & 1, parity
        // (t >> 1) & 1.  Waiting twice on a phase that completed is harmless:
        // a stage is only refilled after this warp releases it.
        uint32_t kst = 1 % kKStages, kpar = kKStages == 1 ? 1u : 0u;
        for (int t = 0; ok && t < n_tiles; ++t) {
            if (__any_sync(0xffffffffu, *abort_flag != 0)) { ok = false; break; }
            const uint32_t vst = uint32_t(t) & 1u, vpar = (uint32_t(t) >> 1) & 1u;
            for (int x = 0; x < 2 && ok; ++x) {
                const int nx = x == 0 ? n_a : n_b;
                if (t >= nx) continue;
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&p_full[x], uint32_t(t) & 1u)))) break;
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&v_full[vst], vpar)))) break;
                tc::fence_after_sync();
                pv(x, t, vst);
                if (t + 1 < nx) {
                    if (!(ok = __all_sync(0xffffffffu, mbar_wait(&k_full[kst], kpar)))) break;
                    tc::fence_after_sync();
                    qk(x, kst);
                }
            }
            if (ok) {
                tc::commit_warp(&v_empty[vst]);
                if (t + 1 < n_tiles) tc::commit_warp(&k_empty[kst]);
            }
            if (++kst == kKStages) { kst = 0; kpar ^= 1u; }
        }
        if (!ok && lane == 0) {
            flag_error(dev_err, PD_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }                                                  // warps 2, 3: spare
    } else {
        // --------------------------- softmax + epilogue ---------------------------
        tc::regs_inc<kRegsSoftmax>();
        const int x = warp >= 8 ? 1 : 0;               // tile A or B
        const int nx = x == 0 ? n_a : n_b;
        const int quarter = warp & 3;                  // tensor-memory lane quarter
        const int r = quarter * 32 + lane;             // tile row
        const int tok = r / GP;                        // token within the tile
        const int g = r % GP;
        const int qx0 = q0 + x * TQ;                   // first chunk token of this tile
        const int pos = P + qx0 + tok;                 // position of this query
        const int lim = min(pos, ctx - 1);             // last visible key
        const bool row_valid = qx0 + tok < C;
        const uint32_t lane_base = uint32_t(quarter * 32) << 16;
        const uint32_t s_cols = tmem + lane_base + uint32_t(x) * 256;
        const uint32_t o_cols = s_cols + 128;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int t = 0; t < nx; ++t) {
            const int par = t & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[x], par));
            if (!ok || __any_sync(0xffffffffu, *abort_flag != 0)) break;
            const int kbase = t * kTileN;
            uint32_t sr[kTileN];
            float p_max;
            {
                tc::fence_after_sync();
                // ---- the whole S row into registers (one burst of loads)
#pragma unroll
                for (int c = 0; c < kTileN / 32; ++c)
                    tc::tmem_ld32(s_cols + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
                tc::tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < kTileN / 32; ++c)
                    tc::tmem_ld_fence(*reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
                if (kbase + kTileN - 1 > lim) {        // only tiles that cross the limit
#pragma unroll
                    for (int e = 0; e < kTileN; ++e)
                        if (kbase + e > lim) sr[e] = __float_as_uint(-INFINITY);
                }
                float mxs[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < kTileN; e += 8) {
                    mxs[0] = fmax3(mxs[0], __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
                    mxs[1] = fmax3(mxs[1], __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]));
                    mxs[2] = fmax3(mxs[2], __uint_as_float(sr[e + 4]), __uint_as_float(sr[e + 5]));
                    mxs[3] = fmax3(mxs[3], __uint_as_float(sr[e + 6]), __uint_as_float(sr[e + 7]));
                }
                const float m_tile = fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])) * scale_log2;
                // The tensor-memory loads and stores below are warp-collective,
                // so the warp rescales together when any of its rows needs it;
                // each row uses its own exact factor (1 when its max did not grow).
                if (__any_sync(0xffffffffu, m_tile > m_run + kRescaleThreshold)) {
                    const float m_new = fmaxf(m_run, m_tile);
                    const float alpha = ex2(m_run - m_new);    // 0 on the first tile
                    if (t > 0) {
                        // O holds PV of tiles < t (already complete: QK of tile t
                        // was issued after PV of tile t-1); wait anyway, cheaply.
                        ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[x * 2 + ((t - 1) & 1)],
                                                               ((t - 1) >> 1) & 1));
                        if (!ok) break;
                        {
                            tc::fence_after_sync();
#pragma unroll
                            for (int c = 0; c < D / 16; ++c) {
                                uint32_t o[16];
                                tc::tmem_ld16(o_cols + c * 16, o);
                                tc::tmem_ld_wait();
                                tc::tmem_ld_fence(o);
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                                tc::tmem_st16(o_cols + c * 16, o);
                            }
                            tc::tmem_st_wait();
                        }
                    }
                    l_run *= alpha;
                    m_run = m_new;
                }
                // Can some key of this tile carry a weight above kLoWeight?
                // max weight <= p_max / (l_before + p_max).
                p_max = m_tile == -INFINITY ? 0.f : ex2(m_tile - m_run);
            }
            // The warp stores residuals when one of its rows needs them, and
            // zeros otherwise, so the MMA issuer can run the lo pass for the
            // whole tile when any warp asks for it.
            const bool need_lo = __any_sync(0xffffffffu, p_max > kLoWeight * (l_run + p_max));
            // ---- p = 2^(s * scale_log2 - m) over S: keys 32c..32c+31 -> hi in
            // columns 32c..32c+15, lo (when taken) in 32c+16..32c+31
            const float2 sc2 = make_float2(scale_log2, scale_log2);
            const float2 nm2 = make_float2(-m_run, -m_run);
            float2 lsum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            auto exp_pass = [&](auto with_lo) {
                constexpr bool kLo = decltype(with_lo)::value;
#pragma unroll
                for (int c = 0; c < kTileN / 32; ++c) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float2 xv = ffma2(make_float2(__uint_as_float(sr[c * 32 + 2 * e]),
                                                            __uint_as_float(sr[c * 32 + 2 * e + 1])),
                                                sc2, nm2);
                        const float2 pv = make_float2(ex2(xv.x), ex2(xv.y));
                        lsum[e & 1] = fadd2(lsum[e & 1], pv);
                        hi[e] = E::pack2(pv.x, pv.y);
                        if (kLo) {
                            const float2 d = fsub2(pv, E::unpack2(hi[e]));   // exact
                            lo[e] = E::pack2(d.x, d.y);
                        }
                    }
                    tc::tmem_st16(s_cols + c * 32, hi);
                    if (kLo) tc::tmem_st16(s_cols + c * 32 + 16, lo);
                    else tc::tmem_st16_zero(s_cols + c * 32 + 16);
                }
            };
            if (need_lo) exp_pass(std::true_type{});
            else exp_pass(std::false_type{});
            l_run += (lsum[0].x + lsum[0].y) + (lsum[1].x + lsum[1].y);
            tc::tmem_st_wait();
            if (lane == 0) lo_flag[x * 8 + par * 4 + quarter] = need_lo ? 1 : 0;
            // Keys past the context in the last tile: their V rows hold other
            // data (or were never loaded); zero them so 0 * v stays 0.  The
            // first tile to use this stage does it.
            const bool zero_v = kbase + kTileN > ctx && (x == 0 || t >= n_a);
            if (zero_v) {
                const int vst = t % kVStages;
                ok = __all_sync(0xffffffffu, mbar_wait(&v_full[vst], (t / kVStages) & 1));
                if (!ok) break;
                if (kbase + r >= ctx) {
                    unsigned char* vrow = smem + L::kV + vst * L::kTile + r * 128;
#pragma unroll
                    for (int a = 0; a < kAtoms; ++a)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<uint4*>(vrow + a * L::kAtom + c * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                }
                tc::fence_proxy_async_smem();
            }
            tc::fence_before_sync();
            mbar_arrive(&p_full[x]);
        }
        if (ok && nx > 0 && !__any_sync(0xffffffffu, *abort_flag != 0)) {
            ok = __all_sync(0xffffffffu, mbar_wait(&pv_done[x * 2 + ((nx - 1) & 1)],
                                                   ((nx - 1) >> 1) & 1));
            if (ok) {
                tc::fence_after_sync();
                const float inv = 1.f / l_run;
                T* orow = out + ((int64_t)(q_begin + qx0 + tok) * H + head0 + g) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tc::tmem_ld32(o_cols + c * 32, o);
                    tc::tmem_ld_wait();
                    tc::tmem_ld_fence(o);
                    uint32_t pk2[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk2[e] = E::pack2(__uint_as_float(o[2 * e]) * inv,
                                          __uint_as_float(o[2 * e + 1]) * inv);
                    if (row_valid) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_uint4(pk2[4 * e], pk2[4 * e + 1], pk2[4 * e + 2],
                                                pk2[4 * e + 3]);
                    }
                }
            }
        }
        if (!ok && lane == 0) {
            flag_error(dev_err, PD_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    __syncthreads();
    if (*abort_flag) {
        // Drain: no MMA may still be writing tensor memory, no TMA shared memory.
        if (warp == 1 && lane == 0) {
            tc::commit(drain);
            mbar_wait(drain, 0);
        }
        if (warp == 0 && lane == 0) {
            const int nk = *k_issued, nv = *v_issued;
            for (int t = max(0, nk - kKStages); t < nk; ++t)
                if (!mbar_wait(&k_full[t % kKStages], (t / kKStages) & 1)) break;
            for (int t = max(0, nv - kVStages); t < nv; ++t)
                if (!mbar_wait(&v_full[t % kVStages], (t / kVStages) & 1)) break;
            mbar_wait(q_full, 0);
        }
        __syncthreads();
    }
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- host side --------------------------------------------------------------------------

template <typename T, int D>
pd_status launch_prefill_t(const PrefillArgs& a) {
    using L = PrefillSmem<D>;
    const int G = a.H / a.Hk;
    int GP = 1;
    while (GP * 2 <= 16 && G % (GP * 2) == 0) GP *= 2;
    const int TQ = kTileM / GP;
    CUtensorMap tm_q, tm_k, tm_v;
    const unsigned long long rows = (unsigned long long)a.NB * a.Hk * a.S;
    if (rows > 0x7fffffffull) return PD_ERR_UNSUPPORTED;   // TMA row coordinate is int32
    if (!encode_q_map(&tm_q, a.q, D, a.H, a.total_q, GP, TQ, a.dt) ||
        !encode_pool_map(&tm_k, a.key_cache, D, rows, a.S, a.dt) ||
        !encode_pool_map(&tm_v, a.value_cache, D, rows, a.S, a.dt))
        return launch_result(cudaErrorInvalidValue);
    auto kern = paged_prefill_kernel<T, D>;
    static uint64_t attr_set = 0;   // one bit per device
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return launch_result(e0);
    if (dev >= 64 || !((attr_set >> dev) & 1)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             L::kAlloc);
        if (e != cudaSuccess) return launch_result(e);
        if (dev < 64) attr_set |= uint64_t(1) << dev;
    }
    dim3 grid(unsigned((a.max_q_len + 2 * TQ - 1) / (2 * TQ)), unsigned(a.Hk * (G / GP)),
              unsigned(a.B));
    kern<<<grid, kPrefillThreads, L::kAlloc, a.stream>>>(
        tm_q, tm_k, tm_v, static_cast<T*>(a.out), a.total_q, a.cu_q_lens, a.block_tables,
        a.max_blocks_per_seq, a.context_lens, a.H, a.Hk, a.S, a.NB, GP, a.scale * kLog2e,
        a.dev_err);
    return launch_result(cudaGetLastError());
}

}  // namespace

pd_status launch_prefill(const PrefillArgs& a) {
    if (a.dt == PD_BF16)
        return a.D == 128 ? launch_prefill_t<__nv_bfloat16, 128>(a)
                          : launch_prefill_t<__nv_bfloat16, 64>(a);
    return a.D == 128 ? launch_prefill_t<__half, 128>(a) : launch_prefill_t<__half, 64>(a);
}

}  // namespace pd
