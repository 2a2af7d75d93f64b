// decode.cu -- paged decode attention, split-context.
//
// Operation (nanoPD page, "自定义CUDA分页注意力内核"; paging per the tutorial
// page "LLM 推理服务引擎深度拆解", section 2.2; GQA per the essay page
// "LLM推理PD分离架构深度工程实践", section 6.2):
//   out[i][h] = sum_{t < ctx_i} softmax_t(scale * q[i][h] . k_t) v_t,
//   k_t, v_t read from kv head h / G through block_tables[i][t / S].
//
// Decode is HBM-bound (arithmetic intensity ~1 FLOP/byte per query head,
// tutorial page section 1.1), so the design is about streaming every K/V
// byte exactly once at full bandwidth:
//   * grid = (kv head x head group, sequence, partition); a partition is a
//     fixed run of PART logical tokens, so long contexts spread over many SMs;
//   * one producer warp streams the partition's K and V block slabs (each a
//     contiguous [S][D] run of the pool) into a 4-stage shared-memory ring
//     with bulk copies (TMA engine, mbarrier completion): up to 64 KB in
//     flight per CTA, three CTAs per SM;
//   * four consumer warps share each stage: q . k with 8 lanes per token
//     (16-byte conflict-free shared loads), a 3-step shuffle reduction that
//     leaves each lane with one (token, head) score, online softmax in the
//     log2 domain with lazy rescaling, and p * v with 32 lanes across D;
//     all fp32 with packed two-wide FMAs;
//   * the G query heads that share a kv head are processed together, so K/V
//     are read once per kv head;
//   * the four warps' partial results are merged in shared memory; a batch
//     that fits one partition writes `out` directly, otherwise partial
//     (max, sum, unnormalised output) triples go to the workspace and a
//     reduce kernel (launched programmatically dependent) merges them in
//     fixed partition order.  No atomics touch results: outputs are
//     bit-identical for any placement of blocks in the pool.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "pd_device.cuh"
#include "pd_internal.h"

namespace pd {
namespace {

constexpr int kPart = 256;          // tokens per partition (multiple of 64)
constexpr int kStageTokens = 32;    // tokens per pipeline stage
constexpr int kStages = 4;          // ring depth
constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when max grows > 2^8
constexpr float kLog2e = 1.4426950408889634f;

template <int D, int GH>
struct DecodeSmem {
    static constexpr int kStageBytes = kStageTokens * D * 2;
    static constexpr int kQuadsPerWarp = kStageTokens / 4 / kConsumerWarps;
    static constexpr int kTokPerWarp = kQuadsPerWarp * 4;
    // layout (bytes)
    static constexpr int kK = 0;
    static constexpr int kV = kK + kStages * kStageBytes;
    static constexpr int kP = kV + kStages * kStageBytes;             // float2 [warps][tok][GH]
    static constexpr int kPBytes = kConsumerWarps * kTokPerWarp * GH * 8;
    static constexpr int kM = kP + kPBytes;                           // float [warps][GH]
    static constexpr int kL = kM + kConsumerWarps * GH * 4;           // float [warps][GH]
    static constexpr int kBar = (kL + kConsumerWarps * GH * 4 + 15) / 16 * 16;
    static constexpr int kMisc = kBar + 2 * kStages * 8;              // int32 flags
    static constexpr int kBytes = kMisc + 16;
    // merge buffer float [warps][GH][D] aliases the K ring after the loop
    static_assert(kConsumerWarps * GH * D * 4 <= kStages * kStageBytes, "merge alias");
};

template <typename T, int D, int GH>
__global__ void __launch_bounds__(kDecodeThreads, 3)
paged_decode_split_kernel(T* __restrict__ out, const T* __restrict__ q,
                          const T* __restrict__ key_cache, const T* __restrict__ value_cache,
                          const int32_t* __restrict__ block_tables, int max_blocks_per_seq,
                          const int32_t* __restrict__ context_lens, int H, int Hk, int S,
                          int NB, int max_context_len, float scale_log2, int num_parts_max,
                          float* __restrict__ ws_o, float* __restrict__ ws_m,
                          float* __restrict__ ws_l, int32_t* dev_err) {
    using L = DecodeSmem<D, GH>;
    using E = Elem<T>;
    extern __shared__ __align__(128) unsigned char smem[];
    T* k_ring = reinterpret_cast<T*>(smem + L::kK);
    T* v_ring = reinterpret_cast<T*>(smem + L::kV);
    float2* pbuf = reinterpret_cast<float2*>(smem + L::kP);
    float* red_m = reinterpret_cast<float*>(smem + L::kM);
    float* red_l = reinterpret_cast<float*>(smem + L::kL);
    float* red_o = reinterpret_cast<float*>(smem + L::kK);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint64_t* empty = full + kStages;
    volatile int32_t* abort_flag = reinterpret_cast<int32_t*>(smem + L::kMisc);
    int32_t* issued = reinterpret_cast<int32_t*>(smem + L::kMisc + 4);

    pdl_launch_dependents();

    const int G = H / Hk;
    const int groups = G / GH;
    const int kvh = blockIdx.x / groups;
    const int h0 = kvh * G + (blockIdx.x % groups) * GH;   // first q head of this CTA
    const int seq = blockIdx.y;
    const int part = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Context of this sequence, cut to what the table and the workspace hold.
    int ctx = __ldg(context_lens + seq);
    const int cap = min(max_blocks_per_seq * S, num_parts_max * kPart);
    if (ctx > cap || ctx < 0) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && part == 0) flag_error(dev_err, PD_DEVERR_CTX_RANGE);
        ctx = ctx < 0 ? 0 : cap;
    }
    const int t_begin = part * kPart;
    const bool direct = (num_parts_max == 1);
    if (t_begin >= ctx) {
        // Nothing to attend to.  A zero-length context still owes zeros.
        if (part == 0 && direct) {
            for (int idx = threadIdx.x; idx < GH * D / 2; idx += kDecodeThreads) {
                const int h = idx / (D / 2), d2 = idx % (D / 2);
                reinterpret_cast<uint32_t*>(out + ((int64_t)seq * H + h0 + h) * D)[d2] = 0u;
            }
        }
        if (part == 0 && !direct && threadIdx.x < GH) {
            const int64_t r = ((int64_t)seq * H + h0 + threadIdx.x) * num_parts_max;
            ws_m[r] = -INFINITY;   // the reduce kernel sees an empty row
            ws_l[r] = 0.f;
        }
        return;
    }
    const int t_end = min(ctx, t_begin + kPart);
    const int n_stages = (t_end - t_begin + kStageTokens - 1) / kStageTokens;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        *issued = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const int32_t* bt_row = block_tables + (int64_t)seq * max_blocks_per_seq;

    if (warp == kConsumerWarps) {
        // ---------------- producer warp ----------------
        const int chunk = S < kStageTokens ? S : kStageTokens;    // tokens per bulk copy
        const uint32_t chunk_bytes = uint32_t(chunk) * D * 2;
        for (int st = 0; st < n_stages; ++st) {
            const int slot = st % kStages;
            // every lane waits (acquire), then the warp agrees on the outcome
            const bool ok = __all_sync(0xffffffffu, st < kStages ||
                                       mbar_wait(&empty[slot], ((st / kStages) - 1) & 1));
            if (!ok) {
                if (lane == 0) {
                    flag_error(dev_err, PD_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            const int t0 = t_begin + st * kStageTokens;
            const int nt = min(kStageTokens, t_end - t0);
            const int nchunks = (nt + chunk - 1) / chunk;
            int64_t src = -1;
            if (lane < nchunks) {
                const int t = t0 + lane * chunk;
                const int blk = __ldg(bt_row + t / S);
                if (blk >= 0 && blk < NB) {
                    src = (((int64_t)blk * Hk + kvh) * S + (t % S)) * D;
                } else {
                    flag_error(dev_err, PD_DEVERR_BLOCK_RANGE);
                }
            }
            const uint32_t ok_mask = __ballot_sync(0xffffffffu, src >= 0);
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], 2u * chunk_bytes * __popc(ok_mask));
            __syncwarp();
            if (src >= 0) {
                bulk_g2s(k_ring + slot * kStageTokens * D + lane * chunk * D, key_cache + src,
                         chunk_bytes, &full[slot]);
                bulk_g2s(v_ring + slot * kStageTokens * D + lane * chunk * D, value_cache + src,
                         chunk_bytes, &full[slot]);
            }
            if (lane == 0) *issued = st + 1;
        }
        return;
    }

    // ---------------- consumer warps ----------------
    constexpr int DQ = D / 8;          // dims per lane for q . k
    constexpr int CHQ = DQ / 8;        // 16-byte chunks per lane (2 or 1)
    constexpr int DV = D / 32;         // dims per lane for p * v (4 or 2)
    const int tg = lane >> 3;          // token within a quad
    const int j = lane & 7;            // lane within the token group

    // q (scaled into the log2 domain) for this lane's dims: chunk c = j + 8k.
    float2 qr[GH][CHQ][4];
#pragma unroll
    for (int h = 0; h < GH; ++h) {
        const uint4* qrow = reinterpret_cast<const uint4*>(q + ((int64_t)seq * H + h0 + h) * D);
#pragma unroll
        for (int k = 0; k < CHQ; ++k) {
            const uint4 w = __ldg(qrow + j + 8 * k);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = E::unpack2(ww[e]);
                qr[h][k][e] = make_float2(f.x * scale_log2, f.y * scale_log2);
            }
        }
    }
    // head whose full score this lane holds after the shuffle reduction
    const int my_h = GH == 4 ? (((j >> 2) & 1) * 2 + ((j >> 1) & 1)) : (GH == 2 ? ((j >> 2) & 1) : 0);

    float m_run[GH];
    float2 acc[GH][DV / 2];
#pragma unroll
    for (int h = 0; h < GH; ++h) {
        m_run[h] = -INFINITY;
#pragma unroll
        for (int e = 0; e < DV / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);
    }
    float l_lane = 0.f;
    float2* my_pbuf = pbuf + warp * L::kTokPerWarp * GH;

    int st = 0;
    for (; st < n_stages; ++st) {
        const int slot = st % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (st / kStages) & 1))) {
            if (lane == 0) {
                flag_error(dev_err, PD_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            break;
        }
        const int nt = min(kStageTokens, t_end - (t_begin + st * kStageTokens));
        const T* ks = k_ring + slot * kStageTokens * D;
        const T* vs = v_ring + slot * kStageTokens * D;

        // ---- scores for this warp's tokens: quads warp, warp + 4, ...
        float s[L::kQuadsPerWarp];
#pragma unroll
        for (int qd = 0; qd < L::kQuadsPerWarp; ++qd) {
            const int tq = (warp + kConsumerWarps * qd) * 4 + tg;
            float part_s[GH];
            if ((warp + kConsumerWarps * qd) * 4 < nt) {
                float2 a[GH];
#pragma unroll
                for (int h = 0; h < GH; ++h) a[h] = make_float2(0.f, 0.f);
                const uint4* krow = reinterpret_cast<const uint4*>(ks + tq * D);
#pragma unroll
                for (int k = 0; k < CHQ; ++k) {
                    const uint4 w = krow[j + 8 * k];
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 kf = E::unpack2(ww[e]);
#pragma unroll
                        for (int h = 0; h < GH; ++h) a[h] = ffma2(qr[h][k][e], kf, a[h]);
                    }
                }
#pragma unroll
                for (int h = 0; h < GH; ++h) part_s[h] = a[h].x + a[h].y;
            } else {
#pragma unroll
                for (int h = 0; h < GH; ++h) part_s[h] = 0.f;
            }
            // reduce over the 8 lanes of the token group; lane keeps head my_h
            float r;
            if constexpr (GH == 4) {
                const bool b2 = (j >> 2) & 1, b1 = (j >> 1) & 1;
                const float send0 = b2 ? part_s[0] : part_s[2];
                const float send1 = b2 ? part_s[1] : part_s[3];
                const float keep0 = b2 ? part_s[2] : part_s[0];
                const float keep1 = b2 ? part_s[3] : part_s[1];
                const float t0 = keep0 + __shfl_xor_sync(0xffffffffu, send0, 4);
                const float t1 = keep1 + __shfl_xor_sync(0xffffffffu, send1, 4);
                const float send = b1 ? t0 : t1;
                const float keep = b1 ? t1 : t0;
                r = keep + __shfl_xor_sync(0xffffffffu, send, 2);
                r += __shfl_xor_sync(0xffffffffu, r, 1);
            } else if constexpr (GH == 2) {
                const bool b2 = (j >> 2) & 1;
                const float send = b2 ? part_s[0] : part_s[1];
                const float keep = b2 ? part_s[1] : part_s[0];
                r = keep + __shfl_xor_sync(0xffffffffu, send, 4);
                r += __shfl_xor_sync(0xffffffffu, r, 2);
                r += __shfl_xor_sync(0xffffffffu, r, 1);
            } else {
                r = part_s[0];
                r += __shfl_xor_sync(0xffffffffu, r, 4);
                r += __shfl_xor_sync(0xffffffffu, r, 2);
                r += __shfl_xor_sync(0xffffffffu, r, 1);
            }
            s[qd] = tq < nt ? r : -INFINITY;
        }

        // ---- online softmax (log2 domain), lazy rescale
        float mx = s[0];
#pragma unroll
        for (int qd = 1; qd < L::kQuadsPerWarp; ++qd) mx = fmaxf(mx, s[qd]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        bool grow = false;
        float m_new[GH];
#pragma unroll
        for (int h = 0; h < GH; ++h) {
            const int src_lane = GH == 4 ? ((h >> 1) * 4 + (h & 1) * 2) : (GH == 2 ? h * 4 : 0);
            const float mh = __shfl_sync(0xffffffffu, mx, src_lane);
            m_new[h] = mh > m_run[h] + kRescaleThreshold ? mh : m_run[h];
            grow |= m_new[h] != m_run[h];
        }
        if (grow) {   // warp-uniform: every lane holds the same m_run / m_new
            float alpha_mine = 1.f;
#pragma unroll
            for (int h = 0; h < GH; ++h) {
                const float alpha = ex2(m_run[h] - m_new[h]);
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                for (int e = 0; e < DV / 2; ++e) acc[h][e] = fmul2(acc[h][e], a2);
                if (h == my_h) alpha_mine = alpha;
                m_run[h] = m_new[h];
            }
            l_lane *= alpha_mine;
        }
        float m_mine = m_run[0];
#pragma unroll
        for (int h = 1; h < GH; ++h) if (h == my_h) m_mine = m_run[h];
        // A warp that has not seen a valid token yet keeps max -inf; its
        // scores are all -inf too and must give p = 0, not 2^(-inf + inf).
        if (m_mine == -INFINITY) m_mine = 0.f;
#pragma unroll
        for (int qd = 0; qd < L::kQuadsPerWarp; ++qd) {
            const float p = ex2(s[qd] - m_mine);   // 0 for masked tokens
            l_lane += p;
            if ((j & ((8 / GH) - 1)) == 0)
                my_pbuf[(qd * 4 + tg) * GH + my_h] = make_float2(p, p);
        }
        __syncwarp();

        // ---- p * v: lane owns dims [lane*DV, lane*DV + DV)
#pragma unroll
        for (int qd = 0; qd < L::kQuadsPerWarp; ++qd) {
            const int tbase = (warp + kConsumerWarps * qd) * 4;
            if (tbase >= nt) break;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (tbase + u < nt) {
                    float2 vf[DV / 2];
                    if constexpr (DV == 4) {
                        const uint2 w = reinterpret_cast<const uint2*>(vs + (tbase + u) * D)[lane];
                        vf[0] = E::unpack2(w.x);
                        vf[1] = E::unpack2(w.y);
                    } else {
                        const uint32_t w = reinterpret_cast<const uint32_t*>(vs + (tbase + u) * D)[lane];
                        vf[0] = E::unpack2(w);
                    }
                    const float2* pp = my_pbuf + (qd * 4 + u) * GH;
#pragma unroll
                    for (int h = 0; h < GH; ++h) {
                        const float2 p2 = pp[h];
#pragma unroll
                        for (int e = 0; e < DV / 2; ++e) acc[h][e] = ffma2(p2, vf[e], acc[h][e]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // Named barrier over the consumer warps only (the producer has left).
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    if (*abort_flag) {
        // Let copies already issued into the ring land before the CTA exits.
        if (threadIdx.x == 0) {
            const int n_issued = *issued;
            for (int s2 = st; s2 < n_issued; ++s2)
                if (!mbar_wait(&full[s2 % kStages], (s2 / kStages) & 1)) break;
        }
        return;
    }

    // ---- merge the four warps: m, l per head; o per (head, dim)
    // l over the token groups (lanes xor 8, 16) for this lane's head
    l_lane += __shfl_xor_sync(0xffffffffu, l_lane, 8);
    l_lane += __shfl_xor_sync(0xffffffffu, l_lane, 16);
    if (lane < 8 && (j & ((8 / GH) - 1)) == 0) red_l[warp * GH + my_h] = l_lane;
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < GH; ++h) red_m[warp * GH + h] = m_run[h];
    }
#pragma unroll
    for (int h = 0; h < GH; ++h) {
#pragma unroll
        for (int e = 0; e < DV / 2; ++e)
            reinterpret_cast<float2*>(red_o + (warp * GH + h) * D + lane * DV)[e] = acc[h][e];
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");

    for (int idx = threadIdx.x; idx < GH * D / 2; idx += kConsumerWarps * 32) {
        const int h = idx / (D / 2), d = (idx % (D / 2)) * 2;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_m[w * GH + h]);
        float lsum = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float mw = red_m[w * GH + h];
            const float c = mw == -INFINITY ? 0.f : ex2(mw - M);
            lsum += red_l[w * GH + h] * c;
            const float2 ow = *reinterpret_cast<const float2*>(red_o + (w * GH + h) * D + d);
            o0 += ow.x * c;
            o1 += ow.y * c;
        }
        const int hq = h0 + h;
        if (direct) {
            const float inv = 1.f / lsum;
            reinterpret_cast<uint32_t*>(out + ((int64_t)seq * H + hq) * D)[d / 2] =
                E::pack2(o0 * inv, o1 * inv);
        } else {
            const int64_t r = ((int64_t)seq * H + hq) * num_parts_max + part;
            *reinterpret_cast<float2*>(ws_o + r * D + d) = make_float2(o0, o1);
            if (d == 0) {
                ws_m[r] = M;
                ws_l[r] = lsum;
            }
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

template <typename T, int D, int GH>
pd_status launch_decode_t(const DecodeArgs& a) {
    using Lt = DecodeSmem<D, GH>;
    const int P = decode_num_partitions(a.max_context_len);
    const int groups = (a.H / a.Hk) / GH;
    auto kern = paged_decode_split_kernel<T, D, GH>;
    static uint64_t attr_set = 0;   // one bit per device; benign if raced
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return launch_result(e0);
    if (dev >= 64 || !((attr_set >> dev) & 1)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Lt::kBytes);
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
    dim3 grid(unsigned(a.Hk * groups), unsigned(a.B), unsigned(P));
    kern<<<grid, kDecodeThreads, Lt::kBytes, a.stream>>>(
        static_cast<T*>(a.out), static_cast<const T*>(a.q), static_cast<const T*>(a.key_cache),
        static_cast<const T*>(a.value_cache), a.block_tables, a.max_blocks_per_seq,
        a.context_lens, a.H, a.Hk, a.S, a.NB, a.max_context_len, scale_log2, P, ws_o, ws_m,
        ws_l, a.dev_err);
    pd_status st = launch_result(cudaGetLastError());
    if (st != PD_OK || P == 1) return st;

    // Reduce, launched as a programmatic dependent of the split kernel so its
    // launch overlaps the split kernel's tail.
    const int cap = std::min(a.max_blocks_per_seq * a.S, P * kPart);
    cudaLaunchConfig_t cfg = {};
    const int64_t rows = int64_t(a.B) * a.H;
    cfg.gridDim = dim3(unsigned((rows + kReduceWarps - 1) / kReduceWarps));
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

template <typename T, int D>
pd_status launch_decode_d(const DecodeArgs& a) {
    const int G = a.H / a.Hk;
    if (G % 4 == 0) return launch_decode_t<T, D, 4>(a);
    if (G % 2 == 0) return launch_decode_t<T, D, 2>(a);
    return launch_decode_t<T, D, 1>(a);
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
        return a.D == 128 ? launch_decode_d<__nv_bfloat16, 128>(a)
                          : launch_decode_d<__nv_bfloat16, 64>(a);
    }
    return a.D == 128 ? launch_decode_d<__half, 128>(a) : launch_decode_d<__half, 64>(a);
}

}  // namespace pd
