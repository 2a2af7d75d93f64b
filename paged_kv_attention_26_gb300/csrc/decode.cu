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
//  * work split (stream-K per unit group): a unit is a kv head (or a group
//    of its query heads); the persistent grid (two CTAs per SM) is split into
//    one group of CTAs per unit, and each group cuts its unit's streams --
//    one per sequence, 64-token stages, laid end to end -- into equal
//    contiguous ranges of at least 4 stages, so every CTA streams the same
//    number of bytes.  Members with the same index in every group walk the
//    same blocks together, one head slab each (a block's slabs are adjacent
//    in the pool).  A stream that fits inside one CTA's range is finished
//    there; one that crosses range boundaries leaves one partial result per
//    CTA for the merge;
//  * one producer warp gathers K and V blocks with 2-D TMA boxes
//    ([S tokens][64 dims], 128-byte swizzle) through the block table into a
//    3-stage shared-memory ring (FP8 pools: raw one-byte stages, 6 deep),
//    running ahead across stream boundaries; launched as a dependent of a
//    store grid, it waits for that grid before its first copy;
//  * four consumer warps take 16 tokens of each stage.  The G query heads
//    that share the kv head form the N = 8 side of warp-level tensor-core
//    products (mma.sync m16n8k16, fp32 accumulation): S^T = K q^T for 16
//    tokens, then O^T += V^T P^T.  In verification mode the columns are
//    (query head, query token) pairs with a causal limit per column, and
//    with more than 8 columns the warps split into two column tiles of two
//    warps, each warp taking 32 tokens of a stage.  The fragment layouts line up so each lane
//    owns the same two heads in S and in O: the online softmax (log2 domain,
//    lazy rescaling when a max grows by more than 2^8) needs only three
//    shuffle steps per head pair and no broadcasts; P is transposed into
//    operand layout with movmatrix;
//  * with bf16 operands P enters the product as an unevaluated pair of
//    16-bit values (hi = rn(p), lo = rn(p - hi)), two MMAs per tile, so P
//    carries about 2^-17 relative error instead of the 2^-9 of a single bf16;
//    fp16 operands (fp16 pools, FP8 pools widened to fp16) take one fp16 P
//    (2^-11, the size of q's own rounding in the FP8 path);
//  * shared-prefix mode (fork groups) runs its consumers on the 5th-generation
//    tensor cores instead: the group's (member, head) columns are the rows of
//    128-row tcgen05 products, S^T = q K^T and O^T += P V, with S, P and O in
//    tensor memory; one warp runs the softmax over the columns (one per lane),
//    one issues the products, one counts and merges pieces;
//  * at the end of each stream piece the four warps merge through a small
//    exchange buffer (after which all but the result warp go on to the next
//    piece); a whole stream is normalised and written to `out`.
//    A piece of a longer stream leaves (max, sum, unnormalised o) in the
//    workspace and counts itself on the stream's arrival counter; the CTA
//    that brings the count to the number of pieces merges them all, in
//    fixed piece order, and writes `out`.  No second kernel, and no atomics
//    touch results: outputs are bit-identical for any placement of blocks
//    in the pool and any order in which CTAs finish.
//  * arrival counters need no clearing between calls: each 64-bit counter
//    carries the tag of the launch that last counted on it (high 44 bits)
//    beside its count (low 20 bits), and a counter holding another launch's
//    tag reads as zero.  Tags are distinct per launch within a process and
//    salted per process.  The arrival that completes a stream writes the
//    counter back to zero, so a launch replayed with its tag unchanged (a
//    captured CUDA graph) also finds its counters at zero.
#include <cuda_runtime.h>

#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <chrono>
#include <cmath>

#include "pd_device.cuh"
#include "pd_internal.h"
#include "pd_mma.cuh"
#include "pd_tcgen05.cuh"
#include "pd_tmap.h"

namespace pd {
namespace {

constexpr int kMinStagesPerCta = 4; // a CTA's range never ends before 4 stages
constexpr int kSegTokens = kMinStagesPerCta * 64;   // bounds pieces per stream
constexpr int kStageTokens = 64;    // tokens per pipeline stage
constexpr int kConsumerWarps = 4;   // 16 tokens of each stage per warp
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kPublisherWarp = kConsumerWarps + 1;   // one query per sequence only
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;     // verify, shared prefix
constexpr int kDecodeThreadsPub = (kConsumerWarps + 2) * 32;  // single-query decode
constexpr int kHeadsN = 8;          // MMA N: query heads per CTA, padded
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when max grows > 2^8
constexpr float kLog2e = 1.4426950408889634f;

// 16-bit pools: TMA fills a 3-stage ring of 16-bit tiles that the consumers
// read.  FP8 pools: TMA fills a 4-stage ring of raw E4M3 tiles (half the
// bytes); each consumer warp widens its own 16 rows of a stage (exactly) to
// fp16 into one 16-bit tile of the same layout, releases the raw stage at
// once, and runs the 16-bit code on fp16 operands.
// kTc: shared-prefix mode, whose consumers run on the tensor cores: the
// piece's q rows lie ahead of the ring, and there is no warp exchange.
template <int D, bool kF8 = false, bool kTc = false>
struct DecodeSmem {
    // FP8 with D = 128: consumers take MMA fragments straight from the raw
    // (128-byte swizzled) tiles, so there is no 16-bit tile and the ring is deeper.
    static constexpr bool kNative = kF8 && D == 128;
    static constexpr int kRing = kNative ? 6 : (kF8 ? 4 : 3);   // stages TMA fills
    static constexpr int kTiles16 = kNative ? 0 : (kF8 ? 1 : kRing);   // 16-bit tiles read
    static constexpr int kAtom = kStageTokens * 128;   // [64 tokens][64 values], 8 KB
    static constexpr int kTile = (D / 64) * kAtom;     // one stage of K (or of V)
    static constexpr int kTile8 = kStageTokens * D;    // one FP8 stage of K (or of V)
    static constexpr int kFrag = (D / 16) * 4 + 4;     // per-lane merge record: o, m[2], l[2]
    // kTc: q of the piece's (up to 32) columns at offset 0, K-major in
    // 64-value swizzle atoms of 32 rows (4 KB); the MMA reads 128 rows from
    // each atom's start, so rows 32.. fall on the atoms and tiles behind it
    // and are never used
    static constexpr int kQAtom = 32 * 128;
    static constexpr int kK = kTc ? (D / 64) * kQAtom : 0;
    static constexpr int kV = kK + kTiles16 * kTile;
    static constexpr int kK8 = kV + kTiles16 * kTile;
    static constexpr int kV8 = kK8 + (kF8 ? kRing * kTile8 : 0);
    static constexpr int kX = kV8 + (kF8 ? kRing * kTile8 : 0);    // merge exchange [2][32][kFrag]
    // a finished piece's stream, unit, piece count and index, and whether it
    // is the range's last (single-query decode: read by the publisher warp)
    static constexpr int kMeta = kX + (kTc ? 0 : 2 * kFrag * 32 * 4);
    static constexpr int kBar = kMeta + 32;
    // ring barriers (full, empty), then the tail-merge and hand-off barriers
    // (kTc: the tensor-core and publisher hand-offs, fourteen)
    // abort flag, issued count, flags (kTc: and the tensor-memory address)
    static constexpr int kMisc = kBar + (2 * kRing + (kTc ? 14 : 4)) * 8;
    // tail merge: the other piece of the range's last stream, [8 rows][D] of
    // o, then m[8], l[8]; kTc: a ring of kWalks walk positions (128 bytes
    // each) and the pieces each reading warp is done with, instead
    static constexpr int kWalks = 4;
    static constexpr int kTl = kMisc + (kTc ? 32 : 16);
    static constexpr int kBytes =
        kTl + (kTc ? kWalks * 128 + 16 : (kHeadsN * D + 2 * kHeadsN) * 4);
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

// Stream walk shared by the producer and the consumers.  The grid is split
// into one group of CTAs per unit (kv head, head group): CTA b works on unit
// b % units as member b / units of that group.  Within a unit the streams are
// ordered by sequence; stream (s, u) has L_s = ceil(ctx_s / 64) stages and
// starts at stage (sum of L over earlier sequences) of the unit's order, and
// the group cuts that order into equal contiguous ranges.  Members with the
// same index in every group therefore walk the same blocks at the same time,
// one head slab each, and a block's slabs lie side by side in the pool, so
// DRAM sees its neighbouring slabs read together.
//
// Shared-prefix mode: a stream is a group of consecutive sequences (forks of
// one prompt) whose block tables agree on their first blocks.  Its stages are
// the shared prefix, read once through the first member's table, followed by
// each member's own remaining tokens ("tails"), read through that member's
// table; a tail stage is seen only by that member's columns.
struct Walk {
    int s, u, L, ctx;     // current stream and its stage count / tokens (decode, verify)
    long start;           // stage index (in the unit's order) of the stream's first stage
    int off;              // next stage within the stream
    long pos, end;        // next stage; end of this CTA's range
    long per_cta;
    int bi;               // this CTA's index within its unit group
    // shared-prefix mode: the group (first sequence, members, shared tokens)
    // and the part the next stage falls in (pj = -1: the shared prefix, else
    // member pj's tail; stage pk of the part's plen, tokens [pt0, pend))
    int lead, nmem, sh;
    int pj, pk, plen, pt0, pend;
};

// A decode step's new rows stored by the decode itself (one per sequence:
// row i is token context_lens[i] - 1 of sequence i, at slots[i]); k == null:
// nothing to store.  The pools are written through kc / vc and read through
// the tensor maps.
struct StepRows {
    const void* k;
    const void* v;
    int64_t ks, vs;          // elements between consecutive rows
    const int64_t* slots;
    void* kc;
    void* vc;
};

// the shared-prefix consumers park one in shared memory (128 bytes)
static_assert(sizeof(Walk) <= 128 && alignof(Walk) <= 8, "walk record");

// Groups of the shared-prefix mode: sequences start[k] .. start[k+1]-1 share
// their first shared[k] tokens' blocks (rounded down to whole blocks and to
// the shortest member's context); at most Mmax members.
struct ForkArgs {
    const int32_t* start;     // [n_groups + 1]
    const int32_t* shared;    // [n_groups]
    int nseq;                 // sequences (rows of q / out)
    int Mmax;                 // most members a group may have (column layout)
    int ppu;                  // workspace pieces per unit: n_groups + CTAs per unit
};

__device__ __forceinline__ int stream_ctx(const int32_t* __restrict__ context_lens, int s,
                                          int cap) {
    const int c = __ldg(context_lens + s);
    return c < 0 ? 0 : (c > cap ? cap : c);
}

// Group k: first sequence, member count (0 for a malformed group), shared
// tokens (a multiple of S, at most every member's context) and, if L is
// given, its stages.  The members' context lengths are loaded eight at a
// time, so a group costs about one load latency, not one per member.
__device__ __forceinline__ void group_info(const ForkArgs& f,
                                           const int32_t* __restrict__ context_lens, int k,
                                           int cap, int S, int& lead, int& n, int& sh,
                                           long* L = nullptr) {
    const int a = __ldg(f.start + k), b = __ldg(f.start + k + 1);
    const int want = __ldg(f.shared + k);
    const bool bad = a < 0 || b < a || b > f.nseq || b - a > f.Mmax;
    lead = a;
    n = bad ? 0 : b - a;
    int c[8];
    int mn = cap;
    long tail_sum = 0;                 // stages of the members' tails, once sh is known
    for (int j0 = 0; j0 < n; j0 += 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = j0 + i < n ? stream_ctx(context_lens, a + j0 + i, cap) : cap;
#pragma unroll
        for (int i = 0; i < 8; ++i) mn = min(mn, c[i]);
    }
    sh = n > 0 ? (max(0, min(want, mn)) & ~(S - 1)) : 0;
    if (L == nullptr) return;
    for (int j0 = 0; j0 < n; j0 += 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            c[i] = j0 + i < n ? stream_ctx(context_lens, a + j0 + i, cap) : sh;   // L1 hits
#pragma unroll
        for (int i = 0; i < 8; ++i) tail_sum += (c[i] - sh + 63) / 64;
    }
    *L = n > 0 ? (sh + 63) / 64 + tail_sum : 0;
}

__device__ __forceinline__ long group_stages(const ForkArgs& f,
                                             const int32_t* __restrict__ context_lens, int k,
                                             int cap, int S) {
    int lead, n, sh;
    long L;
    group_info(f, context_lens, k, cap, S, lead, n, sh, &L);
    return L;
}

// Stages of stream k: ceil(ctx / 64) for a sequence; shared prefix plus tails
// for a group.
template <bool kFork>
__device__ __forceinline__ long stream_stages(const int32_t* __restrict__ context_lens, int k,
                                              int cap, int S, const ForkArgs& f) {
    if constexpr (kFork) return group_stages(f, context_lens, k, cap, S);
    return long((stream_ctx(context_lens, k, cap) + 63) / 64);
}

// Shared-prefix mode: place the part walk at stage `off` of the group stream.
__device__ __forceinline__ void part_seek(Walk& w, const int32_t* __restrict__ context_lens,
                                          int cap, int off) {
    const int ls = (w.sh + 63) / 64;
    w.pj = -1;
    w.pk = off;
    w.plen = ls;
    w.pt0 = 0;
    w.pend = w.sh;
    if (off < ls) return;
    off -= ls;
    for (int j = 0; j < w.nmem; ++j) {
        const int c = stream_ctx(context_lens, w.lead + j, cap);
        const int l = (c - w.sh + 63) / 64;
        if (off < l) {
            w.pj = j;
            w.pk = off;
            w.plen = l;
            w.pt0 = w.sh;
            w.pend = c;
            return;
        }
        off -= l;
    }
}

// Shared-prefix mode: the next stage of the group stream (the next member
// with a non-empty tail once a part is used up; nothing past the stream).
__device__ __forceinline__ void part_next(Walk& w, const int32_t* __restrict__ context_lens,
                                          int cap) {
    if (++w.pk < w.plen) return;
    for (int j = w.pj + 1; j < w.nmem; ++j) {
        const int c = stream_ctx(context_lens, w.lead + j, cap);
        const int l = (c - w.sh + 63) / 64;
        if (l > 0) {
            w.pj = j;
            w.pk = 0;
            w.plen = l;
            w.pt0 = w.sh;
            w.pend = c;
            return;
        }
    }
}

// Load stream w.s's description (every lane) and place the part walk at w.off.
template <bool kFork>
__device__ __forceinline__ void stream_setup(Walk& w, const int32_t* __restrict__ context_lens,
                                             int cap, int S, const ForkArgs& f) {
    if constexpr (kFork) {
        long L;
        group_info(f, context_lens, w.s, cap, S, w.lead, w.nmem, w.sh, &L);
        w.L = int(L);
        part_seek(w, context_lens, cap, w.off);
    } else {
        w.ctx = stream_ctx(context_lens, w.s, cap);
        w.L = (w.ctx + 63) / 64;
    }
}

// Position the walk at the start of this CTA's range (every warp computes it).
// B is the number of streams: sequences, or groups in shared-prefix mode.
template <bool kFork>
__device__ __forceinline__ bool walk_begin(Walk& w, const int32_t* __restrict__ context_lens,
                                           int B, int units, int cap, int S, const ForkArgs& f) {
    const int lane = threadIdx.x & 31;
    const int members = gridDim.x / units;          // CTAs per unit group (>= 1)
    w.u = blockIdx.x % units;
    w.bi = blockIdx.x / units;
    // Up to 128 streams: every lane's context lengths are loaded at once (one
    // round trip to memory instead of one per 32 streams) and kept for the
    // search below.
    constexpr int kHeld = 4;
    const bool held = !kFork && B <= 32 * kHeld;
    long sv[kHeld];
    long total = 0;                                 // stages of one unit
    if (held) {
#pragma unroll
        for (int i = 0; i < kHeld; ++i) {
            const int s = 32 * i + lane;
            sv[i] = s < B ? stream_stages<kFork>(context_lens, s, cap, S, f) : 0;
        }
#pragma unroll
        for (int i = 0; i < kHeld; ++i) total += sv[i];
    } else {
        for (int base = 0; base < B; base += 32) {
            const int s = base + lane;
            total += s < B ? stream_stages<kFork>(context_lens, s, cap, S, f) : 0;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    const long even = (total + members - 1) / members;
    w.per_cta = even > kMinStagesPerCta ? even : long(kMinStagesPerCta);
    const long r0 = long(w.bi) * w.per_cta;
    w.end = total < r0 + w.per_cta ? total : r0 + w.per_cta;
    if (w.bi >= members || r0 >= total) return false;
    // find the stream that contains r0
    long prefix = 0;
    for (int base = 0; base < B; base += 32) {
        const int s = base + lane;
        long v = 0;
        if (held) {
#pragma unroll
            for (int i = 0; i < kHeld; ++i)
                if (32 * i == base) v = sv[i];
        } else {
            v = s < B ? stream_stages<kFork>(context_lens, s, cap, S, f) : 0;
        }
        long incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        const bool hit = s < B && v > 0 && prefix + incl > r0 && prefix + incl - v <= r0;
        const uint32_t m = __ballot_sync(0xffffffffu, hit);
        if (m) {
            const int src = __ffs(m) - 1;
            w.s = base + src;
            w.start = prefix + __shfl_sync(0xffffffffu, incl - v, src);
            w.off = int(r0 - w.start);
            w.pos = r0;
            stream_setup<kFork>(w, context_lens, cap, S, f);
            return true;
        }
        prefix += __shfl_sync(0xffffffffu, incl, 31);
    }
    return false;
}

// After the current stream is exhausted, move to the next non-empty one.
template <bool kFork>
__device__ __forceinline__ void walk_next_stream(Walk& w, const int32_t* __restrict__ context_lens,
                                                 int B, int cap, int S, const ForkArgs& f) {
    w.start += w.L;
    w.off = 0;
    if constexpr (kFork) {
        do {
            ++w.s;
            w.L = w.s < B ? int(group_stages(f, context_lens, w.s, cap, S)) : 0;
        } while (w.s < B && w.L == 0);
        if (w.s < B) stream_setup<kFork>(w, context_lens, cap, S, f);
    } else {
        do {
            ++w.s;
            w.ctx = w.s < B ? stream_ctx(context_lens, w.s, cap) : 0;
        } while (w.s < B && w.ctx == 0);
        w.L = (w.ctx + 63) / 64;
    }
}

// One stage forward (producer): within the stream, or on to the next stream
// when this one is used up and the range goes on.
template <bool kFork>
__device__ __forceinline__ void walk_step(Walk& w, const int32_t* __restrict__ context_lens,
                                          int B, int cap, int S, const ForkArgs& f) {
    ++w.off;
    ++w.pos;
    if (w.off == w.L) {
        if (w.pos < w.end) walk_next_stream<kFork>(w, context_lens, B, cap, S, f);
    } else if constexpr (kFork) {
        part_next(w, context_lens, cap);
    }
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

// Count one arrived piece on a stream's tagged counter; true for the piece
// that completes the stream, which leaves the counter at zero (no other
// piece of this launch touches it afterwards).  High 44 bits: launch tag;
// low 20: count.
constexpr unsigned long long kCountBits = 20;
constexpr unsigned long long kCountMask = (1ull << kCountBits) - 1;

__device__ __forceinline__ bool arrive_piece(unsigned long long* cnt, unsigned long long tag,
                                             int nseg, unsigned long long cur) {
    // cur: the counter as read earlier (a stale value only costs one more CAS)
    for (;;) {
        const unsigned long long next =
            (cur >> kCountBits) == tag ? cur + 1 : (tag << kCountBits) | 1ull;
        const bool done = int(next & kCountMask) == nseg;
        const unsigned long long seen = atomicCAS(cnt, cur, done ? 0ull : next);
        if (seen == cur) return done;
        cur = seen;
    }
}

// Merge the np pieces of a stream's rows (one warp, fixed piece order):
// M = max_k m_k; out = sum_k o_k 2^(m_k - M) / sum_k l_k 2^(m_k - M).
// Four lanes per row (a quarter of D each), so every row is merged at once.
// With kAhead = 2 the o loads of the first two pieces go out together with
// the pieces' (m, l), later pieces two at a time, so a two-piece stream (the
// usual case) costs one L2 round trip; kAhead = 1 (kernels with no registers
// to spare) loads one piece at a time once M is known.  The caller gives each lane its row's output index
// orow (< 0: nothing to write) and the workspace index of the row's first
// piece; later pieces follow at stride pstride.  Pieces of other CTAs are
// read through L2.
template <typename T, int D, int kAhead>
__device__ __forceinline__ void merge_rows(T* __restrict__ out, const float* ws_o,
                                           const float* ws_m, const float* ws_l, int64_t orow,
                                           int64_t base, int pstride, int np, int lane) {
    using E = Elem<T>;
    constexpr int kDpl = D / 4;          // values per lane
    constexpr int kV = kDpl / 4;         // float4 per lane and piece
    constexpr int kCache = kAhead > 1 ? 4 : 8;   // pieces whose (m, l) stay in registers
    if (orow < 0) return;
    const int64_t row = orow;
    const float* m = ws_m + base;
    const float* l = ws_l + base;
    const float4* o = reinterpret_cast<const float4*>(ws_o + base * D + (lane & 3) * kDpl);
    const int64_t ostep = int64_t(pstride) * (D / 4);     // float4 from one piece to the next
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    float mc[kCache], lc[kCache];
    float4 v[kAhead][kV];
    auto load_o = [&](int p0) {
#pragma unroll
        for (int a = 0; a < kAhead; ++a)
#pragma unroll
            for (int c = 0; c < kV; ++c)
                v[a][c] = p0 + a < np ? __ldcg(o + int64_t(p0 + a) * ostep + c) : z4;
    };
#pragma unroll
    for (int p = 0; p < kCache; ++p) {
        mc[p] = p < np ? __ldcg(m + int64_t(p) * pstride) : -INFINITY;
        lc[p] = p < np ? __ldcg(l + int64_t(p) * pstride) : 0.f;
    }
    if constexpr (kAhead > 1) load_o(0);
    float M = -INFINITY;
#pragma unroll
    for (int p = 0; p < kCache; ++p) M = fmaxf(M, mc[p]);
    for (int p = kCache; p < np; ++p) M = fmaxf(M, __ldcg(m + int64_t(p) * pstride));
    float acc[kDpl];
#pragma unroll
    for (int e = 0; e < kDpl; ++e) acc[e] = 0.f;
    float lsum = 0.f;
    for (int p0 = 0; p0 < np; p0 += kAhead) {
        if (kAhead == 1 || p0 > 0) load_o(p0);
#pragma unroll
        for (int a = 0; a < kAhead; ++a) {
            const int p = p0 + a;
            if (p >= np) break;
            float mp = 0.f, lp = 0.f;
            if (p < kCache) {
#pragma unroll
                for (int k = 0; k < kCache; ++k)
                    if (k == p) { mp = mc[k]; lp = lc[k]; }
            } else {
                mp = __ldcg(m + int64_t(p) * pstride);
                lp = __ldcg(l + int64_t(p) * pstride);
            }
            const float w = mp != -INFINITY ? ex2(mp - M) : 0.f;
            lsum += lp * w;
#pragma unroll
            for (int c = 0; c < kV; ++c) {
                acc[4 * c + 0] += v[a][c].x * w;
                acc[4 * c + 1] += v[a][c].y * w;
                acc[4 * c + 2] += v[a][c].z * w;
                acc[4 * c + 3] += v[a][c].w * w;
            }
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;      // a query that saw no key: 0
    uint4* dst = reinterpret_cast<uint4*>(out + row * D + (lane & 3) * kDpl);
#pragma unroll
    for (int c = 0; c < kDpl / 8; ++c)
        dst[c] = make_uint4(E::pack2(acc[8 * c + 0] * inv, acc[8 * c + 1] * inv),
                            E::pack2(acc[8 * c + 2] * inv, acc[8 * c + 3] * inv),
                            E::pack2(acc[8 * c + 4] * inv, acc[8 * c + 5] * inv),
                            E::pack2(acc[8 * c + 6] * inv, acc[8 * c + 7] * inv));
}

// Combine a lane's partial (o fragments, and m, l of its two columns) with
// another share of the same columns stored as a lane record (o fragments,
// then m[2], l[2]): M = max(m, m'); o = o 2^(m - M) + o' 2^(m' - M), and l
// likewise.
template <int KS>
__device__ __forceinline__ void frag_combine(float (&o)[KS][4], float (&m_run)[2],
                                             float (&l_run)[2], const float4* x) {
    const float4 ml = x[KS];
    const float mo2[2] = {ml.x, ml.y}, lo2[2] = {ml.z, ml.w};
    float c_mine[2], c_other[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float mo = mo2[h], lo = lo2[h];
        const float M = fmaxf(m_run[h], mo);
        c_mine[h] = m_run[h] == -INFINITY ? 0.f : ex2(m_run[h] - M);
        c_other[h] = mo == -INFINITY ? 0.f : ex2(mo - M);
        l_run[h] = l_run[h] * c_mine[h] + lo * c_other[h];
        m_run[h] = M;
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        const float4 v = x[mt];
        o[mt][0] = o[mt][0] * c_mine[0] + v.x * c_other[0];
        o[mt][1] = o[mt][1] * c_mine[1] + v.y * c_other[1];
        o[mt][2] = o[mt][2] * c_mine[0] + v.z * c_other[0];
        o[mt][3] = o[mt][3] * c_mine[1] + v.w * c_other[1];
    }
}

// Rows of empty contexts get zeros (no stream covers them); contexts outside
// [0, cap], and non-empty ones shorter than the nq query tokens they hold,
// are flagged (the walk cuts them to cap).  CTA b takes sequences b, b +
// grid, ...; called by one warp.
template <typename T, int D>
__device__ __forceinline__ void zero_empty_rows(T* __restrict__ out,
                                                const int32_t* __restrict__ context_lens, int B,
                                                int H, int nq, int cap, int32_t* dev_err,
                                                int lane) {
    for (int s = blockIdx.x; s < B; s += gridDim.x) {
        const int raw = __ldg(context_lens + s);
        if ((raw < 0 || raw > cap || (raw > 0 && raw < nq)) && lane == 0)
            flag_error(dev_err, PD_DEVERR_CTX_RANGE);
        if (raw <= 0) {
            uint4* dst = reinterpret_cast<uint4*>(out + (int64_t)s * nq * H * D);
            for (int i = lane; i < nq * H * D * 2 / 16; i += 32)
                dst[i] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// Shared-prefix mode: the groups must cover sequences 0 .. nseq - 1 in order
// and every member's table must hold the first member's block ids over the
// group's shared prefix; otherwise PD_DEVERR_SHARED_PREFIX (the results of
// such a group are unspecified).  CTA b checks groups b, b + grid, ...;
// called by one warp.
__device__ __forceinline__ void check_groups(const ForkArgs& f, int n_groups,
                                             const int32_t* __restrict__ block_tables,
                                             int max_blocks_per_seq,
                                             const int32_t* __restrict__ context_lens, int cap,
                                             int S, int32_t* dev_err, int lane) {
    if (blockIdx.x == 0 && lane == 0 &&
        (__ldg(f.start) != 0 || __ldg(f.start + n_groups) != f.nseq))
        flag_error(dev_err, PD_DEVERR_SHARED_PREFIX);
    const int log2S = __ffs(S) - 1;
    for (int k = blockIdx.x; k < n_groups; k += gridDim.x) {
        const int a = __ldg(f.start + k), b = __ldg(f.start + k + 1);
        if (a < 0 || b < a || b > f.nseq || b - a > f.Mmax) {
            if (lane == 0) flag_error(dev_err, PD_DEVERR_SHARED_PREFIX);
            continue;
        }
        int lead, n, sh;
        group_info(f, context_lens, k, cap, S, lead, n, sh);
        const int nb = sh >> log2S;
        const int32_t* first = block_tables + (int64_t)lead * max_blocks_per_seq;
        bool bad = false;
        for (int i = lane; i < (n - 1) * nb; i += 32) {
            const int j = 1 + i / nb, blk = i - (i / nb) * nb;
            bad |= __ldg(block_tables + (int64_t)(lead + j) * max_blocks_per_seq + blk) !=
                   __ldg(first + blk);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) flag_error(dev_err, PD_DEVERR_SHARED_PREFIX);
    }
}

// Two E4M3 codes (low byte = lower index) -> two fp16 values, exactly (every
// E4M3 value is an fp16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

// Two E4M3 codes at bytes (i, j) of w -> fp16x2 exactly (byte i low).
template <uint32_t kSel>
__device__ __forceinline__ uint32_t e4m3_pair_to_f16x2(uint32_t w) {
    uint32_t t;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(t) : "r"(w), "n"(kSel));
    return e4m3x2_to_f16x2(uint16_t(t));
}

// Address of 16-byte chunk c of row r in a stage of 128-byte rows written by
// TMA with 128-byte swizzle (chunk c of row r at position c ^ (r % 8)).
__device__ __forceinline__ uint32_t swz128(uint32_t base, int r, int c) {
    return base + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// T: type of q and out.  kF8: the pools hold E4M3 codes with a K and a V scale
// per kv head; the tensor-core products then run on fp16 (K and V widened
// exactly, q rounded to fp16), and the scales are applied in fp32.
// kMQ: several columns per kv-head unit beyond its query heads, in tiles of 8
// (MMA N): one tile is the decode layout (each consumer warp takes 16 tokens
// of a stage, the four warps merge per piece); with two tiles (verify, up to
// 16 columns), warp w takes tile w / 2 and tokens 32 (w % 2) .. + 31 of each
// stage, so K/V of a kv head is still read once.  Verification (nq_arg query
// tokens per sequence, the last nq_arg positions of its context, each
// attending causally): columns are (head, query token) pairs, head-major.
// kFork (with kMQ): shared-prefix mode, B = groups of sequences; columns are
// (member, head) pairs, member-major (member j of the group: columns
// j GH .. j GH + GH - 1), up to 32, the M rows of the tensor-core consumers.
template <typename T, int D, bool kF8, bool kMQ, bool kFork>
__global__ void __launch_bounds__(kMQ && !kFork ? kDecodeThreads : kDecodeThreadsPub, 2)
paged_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, T* __restrict__ out,
                          const T* __restrict__ q, const int32_t* __restrict__ block_tables,
                          int max_blocks_per_seq, const int32_t* __restrict__ context_lens,
                          int B, int H, int Hk, int S, int NB, int GH, int nq_arg,
                          float scale_log2,
                          int max_segs, int cap, float* __restrict__ ws_o,
                          float* __restrict__ ws_m, float* __restrict__ ws_l,
                          unsigned long long* __restrict__ ws_cnt, unsigned long long tag,
                          const float* __restrict__ k_scale, const float* __restrict__ v_scale,
                          ForkArgs fk, StepRows sr, int32_t* dev_err) {
    static_assert(!kFork || (kMQ && !kF8), "shared-prefix mode: 16-bit pools, column tiles");
    using L = DecodeSmem<D, kF8, kFork>;
    constexpr bool kNative = L::kNative;
    using TM = typename std::conditional<kF8, __half, T>::type;   // tensor-core operand type
    using E = Elem<TM>;
    constexpr int kStages = L::kRing;
    constexpr int kAtoms = D / 64;
    constexpr int KS = D / 16;      // k-steps of q.k, m-tiles of p.v
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* xchg = reinterpret_cast<float*>(smem + L::kX);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBar);
    uint64_t* empty = full + kStages;
    // tail merge: the producer's decision (tail_flag) is made / the other
    // piece is in shared memory
    uint64_t* tail_ready = full + 2 * kStages;
    uint64_t* tail_data = tail_ready + 1;
    // single-query decode: warps 0 and 1 have handed a piece over / the
    // publisher warp has taken it
    uint64_t* pub_full = tail_ready + 2;
    uint64_t* pub_free = tail_ready + 3;
    volatile int32_t* abort_flag = reinterpret_cast<int32_t*>(smem + L::kMisc);
    volatile int32_t* issued = reinterpret_cast<int32_t*>(smem + L::kMisc + 4);
    volatile int32_t* tail_flag = reinterpret_cast<int32_t*>(smem + L::kMisc + 12);

    const int G = H / Hk;
    const int groups = G / GH;
    const int units = Hk * groups;
    const int nq = kMQ && !kFork ? nq_arg : 1;
    const int nseq = kFork ? fk.nseq : B;          // rows of q / out are sequences
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            // shared-prefix mode: freed by the MMA commit after the stage's P V
            mbar_init(&empty[s], kFork ? 1 : kConsumerWarps);
        }
        if constexpr (kFork) {
            // the tensor-core and publisher hand-offs; the publishers' release
            // of a piece (the eleventh and twelfth) takes both publisher warps
            for (int i = 0; i < 14; ++i)
                mbar_init(full + 2 * kStages + i, (i == 10 || i == 11) ? 2 : 1);
            *reinterpret_cast<volatile int32_t*>(smem + L::kMisc + 28) = 0;   // walks ready
            for (int i = 0; i < 4; ++i)                                       // ... and read
                reinterpret_cast<volatile int32_t*>(smem + L::kTl + L::kWalks * 128)[i] = 0;
        } else {
            mbar_init(tail_ready, 1);
            mbar_init(tail_data, 1);
            mbar_init(pub_full, 2);
            mbar_init(pub_free, 1);
        }
        *abort_flag = 0;
        *issued = 0;
        fence_mbar_init();
        tc::prefetch_tmap(&tm_k);
        tc::prefetch_tmap(&tm_v);
    }
    __syncthreads();

    Walk w;
    if (!walk_begin<kFork>(w, context_lens, B, units, cap, S, fk)) {   // uniform: no range
        if (warp == 0) {
            zero_empty_rows<T, D>(out, context_lens, nseq, H, nq, cap, dev_err, lane);
            if constexpr (kFork)
                check_groups(fk, B, block_tables, max_blocks_per_seq, context_lens, cap, S,
                             dev_err, lane);
        }
        return;
    }

    if (warp == kProducerWarp) {
        // ---------------- producer warp: streams stages across stream pieces ----------------
        constexpr int kRingP = kStages;
        uint64_t* p_full = full;
        uint64_t* p_empty = empty;
        const uint32_t block_bytes = uint32_t(S) * D * (kF8 ? 1 : 2);   // one [S][D] slab
        // Block ids of one stage: lane i < (blocks in the stage) loads the id of
        // block i (unchecked), other lanes -2.  The ids of stage gs + 1 are
        // loaded while stage gs is issued, so the table's latency overlaps the
        // copies instead of sitting in front of every stage.
        const int log2S = __ffs(S) - 1;                    // S is a power of two
        auto stage_blk = [&](const Walk& x) -> int {
            // the stage's first token, its end, and whose table holds it
            // (shared-prefix mode: the group's first member for the shared
            // part, the member itself for its tail; both start on a block)
            const int t0 = kFork ? x.pt0 + x.pk * kStageTokens : x.off * kStageTokens;
            const int tend = kFork ? x.pend : x.ctx;
            const int seq = kFork ? (x.pj < 0 ? x.lead : x.lead + x.pj) : x.s;
            const int nt = min(kStageTokens, tend - t0);
            const int nblk = (nt + S - 1) >> log2S;        // <= 64 / S <= 8
            const int32_t* p = block_tables + (int64_t)seq * max_blocks_per_seq +
                               (t0 >> log2S) + lane;
            int v = -2;
            // issued here, consumed one stage later
            if (lane < nblk) asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
            return v;
        };
        Walk wn = w;                                       // one stage ahead of w
        int blk_cur = stage_blk(w);
        // Fused step (single-query decode on 16-bit pools, one unit per kv
        // head): the new row of a stream is stored by the CTA that copies the
        // stream's last stage, the only one that reads its block, right
        // before that copy.  The row and its slot are loaded one stage ahead.
        constexpr bool kRows = !kMQ && !kFork && !kF8;
        auto row_load = [&](const Walk& x, uint4& r, int64_t& sl) {
            r = make_uint4(0u, 0u, 0u, 0u);
            sl = -1;
            if constexpr (kRows) {
                if (sr.k == nullptr || x.pos >= x.end || x.off != x.L - 1) return;
                sl = __ldg(sr.slots + x.s);
                const int c = lane & 15;             // 16-byte chunk: lanes 0.. K, 16.. V
                if (c < D / 8) {
                    const int64_t kvh_x = x.u / groups;
                    const T* src = lane < 16
                                       ? static_cast<const T*>(sr.k) + x.s * sr.ks + kvh_x * D
                                       : static_cast<const T*>(sr.v) + x.s * sr.vs + kvh_x * D;
                    r = __ldg(reinterpret_cast<const uint4*>(src) + c);
                }
            }
        };
        uint4 row_cur, row_next;
        int64_t rs_cur, rs_next;
        row_load(w, row_cur, rs_cur);
        // the stream of the last stage issued (tail merge)
        int tl_s = -1, tl_u = 0, tl_L = 0;
        long tl_start = 0;
        // The first block ids of a stream come from a table row no other
        // stage has touched, a full memory round trip that the one-stage
        // lookahead does not cover: while a stream is walked, the next
        // stream's first table line is fetched into L1 ahead of time.
        auto prefetch_next_row = [&](int s_cur) {
            if constexpr (!kFork) {
                if (lane == 0 && s_cur + 1 < B)
                    asm volatile("prefetch.global.L1 [%0];" ::"l"(
                        block_tables + (int64_t)(s_cur + 1) * max_blocks_per_seq));
            }
        };
        prefetch_next_row(w.s);
        // Launched as a dependent of the store grid, the CTA got here while
        // the store may still run: wait for its writes before the first K/V
        // copy (returns at once for an ordinary launch).
        pdl_wait_primary();
        asm volatile("fence.proxy.async.global;" ::: "memory");
        for (uint32_t gs = 0; w.pos < w.end; ++gs) {
            const int slot = gs % kRingP;
            // every lane waits (acquire), then the warp agrees on the outcome
            const bool ok = __all_sync(0xffffffffu, gs < uint32_t(kRingP) ||
                                       mbar_wait(&p_empty[slot], ((gs / kRingP) - 1) & 1));
            if (!ok || __any_sync(0xffffffffu, *abort_flag != 0)) {
                if (lane == 0 && !ok) {
                    flag_error(dev_err, PD_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            // start loading the next stage's block ids
            const int s_before = wn.s;
            walk_step<kFork>(wn, context_lens, B, cap, S, fk);
            if (wn.s != s_before) prefetch_next_row(wn.s);
            const int blk_next = wn.pos < wn.end ? stage_blk(wn) : -2;
            row_load(wn, row_next, rs_next);
            const int kvh = w.u / groups;
            int row = -1;
            if (blk_cur != -2) {
                if (blk_cur >= 0 && blk_cur < NB) {
                    row = (blk_cur * Hk + kvh) * S;
                } else {
                    flag_error(dev_err, PD_DEVERR_BLOCK_RANGE);
                }
            }
            if (kRows && rs_cur >= 0) {          // uniform: every lane loaded the slot
                // the stream's new row goes into its last block (the stage's
                // last, lane nblk - 1) before the copy: only the slot of the
                // sequence's last token is taken
                const int nt_w = w.ctx - w.off * kStageTokens;   // <= 64: the last stage
                const int blast = __shfl_sync(0xffffffffu, blk_cur, ((nt_w + S - 1) >> log2S) - 1);
                const int off_new = (w.ctx - 1) & (S - 1);
                const bool whole = __ldg(context_lens + w.s) == w.ctx;   // not cut short
                if (whole && blast >= 0 && blast < NB &&
                    rs_cur == int64_t(blast) * S + off_new) {
                    if ((lane & 15) < D / 8) {
                        T* dst = (lane < 16 ? static_cast<T*>(sr.kc) : static_cast<T*>(sr.vc)) +
                                 ((int64_t(blast) * Hk + kvh) * S + off_new) * D;
                        reinterpret_cast<uint4*>(dst)[lane & 15] = row_cur;
                        // each writer orders its store before the async
                        // proxy's accesses (the tensor copy reads the block)
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                    }
                } else if (lane == 0) {
                    flag_error(dev_err, PD_DEVERR_STEP_SLOT);
                }
                // ... and the warp barrier orders the writers before the lanes
                // that issue the copies (a global membar here cost ~2 us a
                // launch, one per stream end on the producer's path)
                __syncwarp();
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            const uint32_t ok_mask = __ballot_sync(0xffffffffu, row >= 0);
            if (lane == 0) mbar_arrive_expect_tx(&p_full[slot], 2u * block_bytes * __popc(ok_mask));
            __syncwarp();
            if (row >= 0) {
                if constexpr (kF8) {
                    // one [S tokens][D bytes] box per block, rows packed
                    const int off = slot * L::kTile8 + lane * S * D;
                    tc::tma_load_2d(smem + L::kK8 + off, &tm_k, 0, row, &p_full[slot]);
                    tc::tma_load_2d(smem + L::kV8 + off, &tm_v, 0, row, &p_full[slot]);
                } else {
#pragma unroll
                    for (int a = 0; a < kAtoms; ++a) {
                        const int off = slot * L::kTile + a * L::kAtom + lane * S * 128;
                        tc::tma_load_2d(smem + L::kK + off, &tm_k, a * 64, row, &p_full[slot]);
                        tc::tma_load_2d(smem + L::kV + off, &tm_v, a * 64, row, &p_full[slot]);
                    }
                }
            }
            if (lane == 0) *issued = int(gs + 1);
            tl_s = w.s;
            tl_u = w.u;
            tl_L = w.L;
            tl_start = w.start;
            w = wn;
            blk_cur = blk_next;
            row_cur = row_next;
            rs_cur = rs_next;
        }
        // ---- tail merge (one query per sequence).  The range's last stream
        // usually goes on in the next CTA's range, whose first piece was
        // counted long ago.  If so (two pieces, the other one counted), this
        // warp loads the other piece into shared memory now, while the
        // consumers finish theirs, and the publisher warp merges the stream
        // from there instead of publishing the last piece.
        [[maybe_unused]] float* tl = reinterpret_cast<float*>(smem + L::kTl);
        int tail = 0;
        if constexpr (!kMQ) {
            // two pieces: the stream starts in this range and ends in the
            // next one (this is piece 0), or starts in the previous range and
            // ends in this one (piece 1); comparisons, no 64-bit division
            const long r0 = long(w.bi) * w.per_cta, s_end = tl_start + tl_L;
            const bool starts_here = tl_start >= r0;
            const bool starts_prev = !starts_here && tl_start >= r0 - w.per_cta;
            const bool ends_here = s_end <= w.end;
            const bool ends_next = !ends_here && s_end <= w.end + w.per_cta;
            const bool two = (starts_here && ends_next) || (starts_prev && ends_here);
            const int t_seg = starts_here ? 0 : 1;
            if (tl_s >= 0 && two && *abort_flag == 0) {
                const unsigned long long c =
                    ld_acquire_u64(ws_cnt + (int64_t)tl_s * units + tl_u);
                tail = __all_sync(0xffffffffu,
                                  (c >> kCountBits) == tag && int(c & kCountMask) == 1) ? 1 : 0;
            }
            // the publisher waits for this decision with the last piece
            if (lane == 0) *tail_flag = tail;
            __syncwarp();
            if (lane == 0) mbar_arrive(tail_ready);
            if (tail) {
                const int t_h0 = (tl_u / groups) * G + (tl_u % groups) * GH;
                // into shared memory by asynchronous copies, all in flight at
                // once (lane: D / 32 values of each row; lanes < GH: m and l
                // of row lane); ordered after the acquire load above
                for (int k = 0; k < GH; ++k) {
                    const int64_t r = ((int64_t)tl_s * H + t_h0 + k) * max_segs + (1 - t_seg);
                    cp_async<D / 8>(tl + k * D + lane * (D / 32), ws_o + r * D + lane * (D / 32));
                }
                if (lane < GH) {
                    const int64_t r = ((int64_t)tl_s * H + t_h0 + lane) * max_segs + (1 - t_seg);
                    cp_async<4>(tl + kHeadsN * D + lane, ws_m + r);
                    cp_async<4>(tl + kHeadsN * D + kHeadsN + lane, ws_l + r);
                }
            }
        }
        // all loads are issued: the producer has time for the empty rows
        zero_empty_rows<T, D>(out, context_lens, nseq, H, nq, cap, dev_err, lane);
        if constexpr (kFork)
            check_groups(fk, B, block_tables, max_blocks_per_seq, context_lens, cap, S, dev_err,
                         lane);
        if constexpr (!kMQ) {
            if (tail) {
                cp_async_wait_all();
                __syncwarp();
                if (lane == 0) mbar_arrive(tail_data);     // the other piece has landed
            }
        }
        return;
    }

    if (!kFork && warp == kPublisherWarp) {
        // ---------------- publisher warp (one query per sequence) ----------------
        // Warps 0 and 1 hand each finished piece over as two partial results
        // in the exchange buffer (the four consumer warps' shares combined in
        // pairs).  This warp combines the two and does what follows, so that
        // the consumers go straight on to the next piece: the normalised rows
        // of a whole stream; or the piece's partial, its fence and arrival
        // count, and the stream's merge when the piece completes it; or, for
        // the range's last piece when the producer has fetched the stream's
        // other piece, the merged rows (the tail merge, with merge_rows'
        // arithmetic and piece order).
        if constexpr (!kMQ) {
            constexpr int KS = D / 16;
            const int32_t* meta = reinterpret_cast<const int32_t*>(smem + L::kMeta);
            const float* tl = reinterpret_cast<const float*>(smem + L::kTl);
            // lane: columns ha, ha + 1; dims 16mt + d0 and + kDd (the
            // consumers' fragment layout; native FP8: the m-tile rows g, g + 8
            // are dims 2g, 2g + 1)
            const int ha = 2 * (lane & 3);
            const int d0 = kNative ? 2 * (lane >> 2) : (lane >> 2);
            constexpr int kDd = kNative ? 1 : 8;
            // bounded wait on a barrier phase that also gives up on an abort
            auto wait_phase = [&](uint64_t* bar, uint32_t parity) -> bool {
                bool got = false;
                const uint64_t t0 = globaltimer();
                for (uint32_t i = 0;; ++i) {
                    if (mbar_try_wait(bar, parity)) { got = true; break; }
                    if (*abort_flag != 0) break;
                    if ((i & 255u) == 0 && globaltimer() - t0 > kWaitLimitNs) break;
                }
                got = __all_sync(0xffffffffu, got);
                if (!got && lane == 0 && *abort_flag == 0) {
                    flag_error(dev_err, PD_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                return got;
            };
            for (uint32_t job = 0;; ++job) {
                if (!wait_phase(pub_full, job & 1)) return;
                const int js = meta[0], ju = meta[1], jn = meta[2], jseg = meta[3];
                const bool jfinal = meta[4] != 0;
                float o[KS][4], m_run[2], l_run[2];
                {
                    const float4* x = reinterpret_cast<const float4*>(xchg + lane * L::kFrag);
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        const float4 v = x[mt];
                        o[mt][0] = v.x; o[mt][1] = v.y; o[mt][2] = v.z; o[mt][3] = v.w;
                    }
                    const float4 ml = x[KS];
                    m_run[0] = ml.x; m_run[1] = ml.y; l_run[0] = ml.z; l_run[1] = ml.w;
                }
                frag_combine<KS>(o, m_run, l_run, reinterpret_cast<const float4*>(
                                                      xchg + (32 + lane) * L::kFrag));
                __syncwarp();
                if (lane == 0) mbar_arrive(pub_free);    // the buffer is free again
                const int jkvh = ju / groups;
                if constexpr (kF8) {
                    const float vs = __ldg(v_scale + jkvh);
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) o[mt][e] *= vs;
                }
                const int jh0 = jkvh * G + (ju % groups) * GH;
                const int64_t row0 = (int64_t)js * H + jh0;      // one query per sequence
                unsigned long long* cnt = ws_cnt + (int64_t)js * units + ju;
                bool merged = false;
                if (jfinal && jn == 2) {
                    // the producer decided after its last copy (long before
                    // this piece ended, as a rule)
                    if (!wait_phase(tail_ready, 0)) return;
                    if (*tail_flag != 0) {
                        if (!wait_phase(tail_data, 0)) return;
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int c = ha + h;
                            if (c >= GH) continue;
                            const float mo = tl[kHeadsN * D + c], lo = tl[kHeadsN * D + kHeadsN + c];
                            // pieces in order: 0, then 1 (this one is jseg)
                            const float m0 = jseg == 0 ? m_run[h] : mo, m1 = jseg == 0 ? mo : m_run[h];
                            const float l0 = jseg == 0 ? l_run[h] : lo, l1 = jseg == 0 ? lo : l_run[h];
                            const float M = fmaxf(fmaxf(-INFINITY, m0), m1);
                            const float w0 = m0 != -INFINITY ? ex2(m0 - M) : 0.f;
                            const float w1 = m1 != -INFINITY ? ex2(m1 - M) : 0.f;
                            float lsum = 0.f;
                            lsum += l0 * w0;
                            lsum += l1 * w1;
                            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                            T* orow = out + (row0 + c) * D;
                            const float* trow = tl + c * D;
#pragma unroll
                            for (int mt = 0; mt < KS; ++mt) {
#pragma unroll
                                for (int r = 0; r < 2; ++r) {
                                    const int d = 16 * mt + d0 + r * kDd;
                                    const float vm = o[mt][h + 2 * r], vt = trow[d];
                                    float acc = 0.f;
                                    acc += (jseg == 0 ? vm : vt) * w0;
                                    acc += (jseg == 0 ? vt : vm) * w1;
                                    orow[d] = T(acc * inv);
                                }
                            }
                        }
                        // the stream is complete: its counter back to zero
                        if (lane == 0) st_relaxed_u64(cnt, 0ull);
                        merged = true;
                    }
                }
                if (!merged) {
                    // read now, so that its latency overlaps the writes and fence
                    unsigned long long c0 = 0;
                    if (jn > 1 && lane == 0) c0 = *reinterpret_cast<volatile unsigned long long*>(cnt);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int c = ha + h;
                        if (c >= GH) continue;
                        const int64_t row = row0 + c;
                        if (jn == 1) {
                            // the whole stream was in this CTA: final, normalised rows
                            const float inv = 1.f / l_run[h];
                            T* orow = out + row * D + d0;
#pragma unroll
                            for (int mt = 0; mt < KS; ++mt) {
                                orow[16 * mt] = T(o[mt][h] * inv);
                                orow[16 * mt + kDd] = T(o[mt][2 + h] * inv);
                            }
                        } else {
                            const int64_t r = row * max_segs + jseg;
                            float* wrow = ws_o + r * D + d0;
#pragma unroll
                            for (int mt = 0; mt < KS; ++mt) {
                                wrow[16 * mt] = o[mt][h];
                                wrow[16 * mt + kDd] = o[mt][2 + h];
                            }
                            if (d0 == 0) {
                                ws_m[r] = m_run[h];
                                ws_l[r] = l_run[h];
                            }
                        }
                    }
                    if (jn > 1) {
                        // publish the piece, count it; the last of the stream's
                        // pieces to arrive merges them all
                        __threadfence();
                        __syncwarp();
                        uint32_t last = 0;
                        if (lane == 0) last = arrive_piece(cnt, tag, jn, c0) ? 1u : 0u;
                        last = __shfl_sync(0xffffffffu, last, 0);
                        if (last) {
                            __threadfence();
                            const int n = lane >> 2;
                            const int64_t orow = n < GH ? row0 + n : -1;
                            merge_rows<T, D, 2>(out, ws_o, ws_m, ws_l, orow,
                                                orow < 0 ? 0 : orow * max_segs, 1, jn, lane);
                        }
                    }
                }
                if (jfinal) return;
            }
        }
        return;
    }

    if constexpr (kFork) {
        // ---------------- shared-prefix mode: consumers on the tensor cores ----------------
        // A stream's (member, head) columns are the M rows 0..31 of 128-row
        // tcgen05 MMAs; rows 32.. read whatever lies behind the q rows and are
        // never looked at.  Per stage g:
        //   S^T = q K^T   [column][64 tokens], fp32 in tensor memory (two buffers)
        //   P = exp2(S^T - m), written over S as 16 bits (bf16: hi, then lo)
        //   O^T += P V    [column][D] in tensor memory, V the MN-major operand
        // Warp 0 owns tensor-memory lanes 0..31, one column per lane: it writes
        // each piece's q rows, runs the online softmax and writes the piece's
        // result (final rows, or partials to the workspace).  Warp 1 issues
        // the MMAs.  Warps 2 and 3 count finished pieces on the stream's
        // arrival counter and merge the stream when its last piece is in.
        // Warp 5 walks the CTA's pieces ahead of the others.
        uint64_t* s_full = full + 2 * kStages;    // S of stage g is in tensor memory
        uint64_t* p_full = s_full + 2;            // P of stage g (and any O rescale) written
        uint64_t* pv_done = p_full + 2;           // O += P V of stage g has finished
        uint64_t* q_ready = pv_done + 2;          // the piece's q rows are written
        uint64_t* drained = q_ready + 1;          // every MMA issued has finished
        // by job parity: a piece's partials are written / taken by both
        // publishers / counted by warp 2
        uint64_t* pub_full_f = drained + 1;
        uint64_t* pub_free_f = pub_full_f + 2;
        uint64_t* last_ready = pub_free_f + 2;
        uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc + 16);
        // whether the piece completed its stream, by job parity
        volatile int32_t* last_f = reinterpret_cast<int32_t*>(smem + L::kMisc + 20);
        constexpr uint32_t kTmemCols = 256;       // S: 2 x 64 columns, then O: D columns
        constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
        const int ncols = GH * fk.Mmax;
        const int cstride = (ncols <= kHeadsN ? 1 : ncols <= 2 * kHeadsN ? 2 : 4) * kHeadsN;
        // bounded wait that also gives up on an abort; warp-uniform result
        auto wait_tc = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool got = false;
            const uint64_t t0 = globaltimer();
            for (uint32_t i = 0;; ++i) {
                if (mbar_try_wait(bar, parity)) { got = true; break; }
                if (*abort_flag != 0) break;
                if ((i & 255u) == 0 && globaltimer() - t0 > kWaitLimitNs) break;
            }
            got = __all_sync(0xffffffffu, got);
            if (!got && lane == 0 && *abort_flag == 0) {
                flag_error(dev_err, PD_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            return got;
        };
        // the piece at a walk position: its unit's first head, its stages, and
        // its place among the stream's pieces (c_first: the CTA index where
        // the stream begins)
        struct Piece {
            int h0, stages, nseg, seg;
            long c_first;
        };
        auto piece_at = [&](const Walk& x) {
            Piece p;
            p.h0 = (x.u / groups) * G + (x.u % groups) * GH;
            const long left = x.end - x.pos;
            p.stages = int(left < long(x.L - x.off) ? left : long(x.L - x.off));
            p.c_first = x.start / x.per_cta;
            p.nseg = int((x.start + x.L - 1) / x.per_cta - p.c_first + 1);
            p.seg = int(long(x.bi) - p.c_first);
            return p;
        };
        auto next_piece = [&](Walk& x, int stages) {
            x.off += stages;
            x.pos += stages;
            if (x.off == x.L && x.pos < x.end) walk_next_stream<kFork>(x, context_lens, B, cap, S, fk);
        };
        const int mem = lane / GH, hh = lane - (lane / GH) * GH;   // lane's column (warp 0)
        // output row of column lane in the group at x (-1: padding, or a member
        // without context, whose rows the producer zeroes)
        auto out_row = [&](const Walk& x, int h0) -> int64_t {
            if (lane >= ncols || mem >= x.nmem || stream_ctx(context_lens, x.lead + mem, cap) == 0)
                return -1;
            return (int64_t)(x.lead + mem) * H + h0 + hh;
        };
        // partials per (unit, piece, column): piece k + c_first + seg of group k
        auto ws_base = [&](const Walk& x, const Piece& p) -> int64_t {
            return ((int64_t)x.u * fk.ppu + x.s + p.c_first) * cstride;
        };
        // The walk position after each of the CTA's pieces, found ahead by
        // warp 5 (each is a chain of dependent loads: the next group's bounds,
        // then its members' context lengths) into a ring of kWalks slots; the
        // other warps read it from shared memory when they move on, and mark
        // each piece they are done with, which frees its slot.
        volatile int32_t* walks_ready = reinterpret_cast<int32_t*>(smem + L::kMisc + 28);
        Walk* walks = reinterpret_cast<Walk*>(smem + L::kTl);
        volatile int32_t* walks_done = reinterpret_cast<int32_t*>(smem + L::kTl + L::kWalks * 128);
        // bounded wait until *v >= want; false (with the abort flag set) when
        // it runs out or another warp gave up
        auto wait_at_least = [&](auto probe, int32_t want) -> bool {
            bool got = probe() >= want;
            if (!got) {
                const uint64_t t0 = globaltimer();
                for (uint32_t i = 0;; ++i) {
                    if (probe() >= want) { got = true; break; }
                    if (*abort_flag != 0) break;
                    if ((i & 255u) == 0 && globaltimer() - t0 > kWaitLimitNs) break;
                }
            }
            got = __all_sync(0xffffffffu, got);
            if (!got && lane == 0 && *abort_flag == 0) {
                flag_error(dev_err, PD_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            return got;
        };
        // x = the walk after piece k; `last` marks piece k done for this warp
        auto piece_after = [&](Walk& x, uint32_t k, bool last) -> bool {
            if (!wait_at_least([&] { return *walks_ready; }, int32_t(k + 1))) return false;
            __threadfence_block();
            x = walks[k % L::kWalks];
            if (last) {
                __threadfence_block();
                __syncwarp();
                if (lane == 0) walks_done[warp] = int32_t(k + 1);
            }
            return true;
        };
        if (warp == kPublisherWarp) {
            // ------------------------------- walker -------------------------------
            Walk x = w;
            for (int k = 0; x.pos < x.end; ++k) {
                // the slot's previous walk has been read by warps 0-3
                if (k >= L::kWalks &&
                    !wait_at_least([&] {
                        return min(min(walks_done[0], walks_done[1]),
                                   min(walks_done[2], walks_done[3]));
                    }, int32_t(k - L::kWalks + 1)))
                    return;
                __threadfence_block();              // their reads before this write
                next_piece(x, piece_at(x).stages);
                if (lane == 0) {
                    walks[k % L::kWalks] = x;
                    __threadfence_block();
                    *walks_ready = k + 1;
                }
                __syncwarp();
            }
            return;
        }
        if (warp >= 2) {
            // ------------------------------ publishers ------------------------------
            // For each piece of several: take it once warp 0 has written its
            // partials, count it (warp 2), and if it was the stream's last,
            // merge the stream's pieces, columns split between the two warps.
            uint32_t job = 0;
            for (uint32_t k = 0; w.pos < w.end; ++k) {
                const Piece pc = piece_at(w);
                if (pc.nseg > 1) {
                    if (!wait_tc(&pub_full_f[job & 1], (job >> 1) & 1)) return;
                    uint32_t last = 0;
                    if (warp == 2) {
                        unsigned long long* cnt = ws_cnt + (int64_t)w.s * units + w.u;
                        if (lane == 0) {
                            const unsigned long long cnt0 =
                                *reinterpret_cast<volatile unsigned long long*>(cnt);
                            // warp 0's writes, seen through the barrier, go out
                            // before the count
                            __threadfence();
                            last = arrive_piece(cnt, tag, pc.nseg, cnt0) ? 1u : 0u;
                            last_f[job & 1] = int32_t(last);
                        }
                        last = __shfl_sync(0xffffffffu, last, 0);
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&last_ready[job & 1]);
                    } else {
                        if (!wait_tc(&last_ready[job & 1], (job >> 1) & 1)) return;
                        last = uint32_t(last_f[job & 1]);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&pub_free_f[job & 1]);
                    ++job;
                    if (last) {
                        __threadfence();
                        const int64_t wb = ws_base(w, pc);
                        for (int n0 = (warp - 2) * 8; n0 < ncols; n0 += 16) {
                            const int n = n0 + (lane >> 2);
                            int64_t rn = -1;
                            if (n < ncols && n / GH < w.nmem &&
                                stream_ctx(context_lens, w.lead + n / GH, cap) > 0)
                                rn = (int64_t)(w.lead + n / GH) * H + pc.h0 + (n - (n / GH) * GH);
                            merge_rows<T, D, 1>(out, ws_o, ws_m, ws_l, rn, wb + n, cstride, pc.nseg,
                                                lane);
                        }
                    }
                }
                if (!piece_after(w, k, true)) return;
            }
            return;
        }
        if (warp == 1) {
            tc::tmem_alloc(tmem_slot, kTmemCols);
            tc::tmem_relinquish();
        }
        tc::fence_before_sync();
        asm volatile("bar.sync 3, 64;" ::: "memory");
        tc::fence_after_sync();
        const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
        const uint32_t o_tm = tmem + 2 * kStageTokens;
        bool ok = true;
        uint32_t g = 0;         // stages consumed by this CTA: ring slot, buffer and phases
        uint32_t npc = 0;       // pieces begun
        if (warp == 1) {
            // ------------------------------ MMA issuer ------------------------------
            // The whole warp runs the loop in step; one elected lane issues.
            constexpr uint32_t kHi = tc::sw128_desc_hi(1024);
            constexpr uint32_t kTile16 = uint32_t(L::kTile) >> 4;
            constexpr uint32_t kIdQK = tc::idesc_f16(kBf, 128, kStageTokens, false, false);
            constexpr uint32_t kIdPV = tc::idesc_f16(kBf, 128, D, false, true);
            const uint32_t q_lo = tc::smem_desc_sw128_lo(smem_u32(smem), 16);   // q tile
            const uint32_t k_lo = tc::smem_desc_sw128_lo(smem_u32(smem + L::kK), 16);
            // V as the MN-major operand: N = D in 64-value atoms (LBO between
            // them), K = tokens at 128 B (SBO per 8 tokens)
            const uint32_t v_lo = tc::smem_desc_sw128_lo(smem_u32(smem + L::kV), L::kAtom);
            // O += P V of stage gg (nt tokens: only the 16-token steps holding
            // some); the piece's first product overwrites O.  P of tokens
            // 32c..32c+31 sits over S as 16 columns of hi, then 16 of lo.
            auto pv = [&](uint32_t gg, int nt, bool first) -> bool {
                if (!wait_tc(&p_full[gg & 1], (gg >> 1) & 1)) return false;
                tc::fence_after_sync();
                const uint32_t slot = gg % kStages;
                const uint32_t p0 = tmem + (gg & 1) * kStageTokens;
                const uint32_t b0 = v_lo + slot * kTile16;
                const int nk = (nt + 15) >> 4;
#pragma unroll
                for (int pass = 0; pass < (kBf ? 2 : 1); ++pass)
                    for (int kk = 0; kk < nk; ++kk)
                        tc::mma_ts_warp(o_tm, p0 + uint32_t(32 * (kk >> 1) + 8 * (kk & 1) + 16 * pass),
                                        b0 + uint32_t(kk * 16 * 128 / 16), kHi, kIdPV,
                                        uint32_t(!first || kk > 0 || pass > 0));
                tc::commit_warp(&pv_done[gg & 1]);
                tc::commit_warp(&empty[slot]);       // K and V of the stage are used up
                return true;
            };
            while (ok && w.pos < w.end) {
                const Piece pc = piece_at(w);
                Walk pw = w;
                if (!(ok = wait_tc(q_ready, npc & 1))) break;
                tc::fence_after_sync();
                int nt_prev = 0;
                for (int st = 0; st < pc.stages; ++st, ++g) {
                    const uint32_t slot = g % kStages;
                    if (!(ok = wait_tc(&full[slot], (g / kStages) & 1))) break;
                    tc::fence_after_sync();
                    const uint32_t d_s = tmem + (g & 1) * kStageTokens;
                    const uint32_t b0 = k_lo + slot * kTile16;
#pragma unroll
                    for (int kk = 0; kk < KS; ++kk) {
                        const uint32_t qo = uint32_t((kk >> 2) * L::kQAtom + (kk & 3) * 32) >> 4;
                        const uint32_t ko = uint32_t((kk >> 2) * L::kAtom + (kk & 3) * 32) >> 4;
                        if (kk == 0)
                            tc::mma_ss_warp<false>(d_s, q_lo + qo, kHi, b0 + ko, kHi, kIdQK);
                        else
                            tc::mma_ss_warp<true>(d_s, q_lo + qo, kHi, b0 + ko, kHi, kIdQK);
                    }
                    tc::commit_warp(&s_full[g & 1]);
                    const int nt = min(kStageTokens, pw.pend - (pw.pt0 + pw.pk * kStageTokens));
                    part_next(pw, context_lens, cap);
                    // the previous stage's P V goes in behind this stage's S
                    if (st > 0 && !(ok = pv(g - 1, nt_prev, st == 1))) break;
                    nt_prev = nt;
                }
                if (!ok || !(ok = pv(g - 1, nt_prev, pc.stages == 1))) break;
                if (!(ok = piece_after(w, npc, true))) break;
                ++npc;
            }
            // nothing may still write tensor memory when it is freed
            tc::commit_warp(drained);
            (void)__all_sync(0xffffffffu, mbar_wait(drained, 0));
        } else {
            // ------------------------- softmax and results -------------------------
            const uint32_t q_base = smem_u32(smem);      // q tile
            const uint32_t v_base = smem_u32(smem + L::kV);
            uint32_t njob = 0;      // pieces handed to the publishers
            // q rows of the piece at x into the q tile (K-major, 128-byte
            // swizzle, lane = row), then hand them to the issuer
            auto write_q = [&](const Walk& x, int h0) -> int64_t {
                const int64_t r = out_row(x, h0);
                const uint4* src = reinterpret_cast<const uint4*>(q + (r < 0 ? 0 : r) * D);
#pragma unroll
                for (int a = 0; a < kAtoms; ++a) {
                    uint4 v[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        v[c] = r >= 0 ? __ldg(src + 8 * a + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_shared_v4(q_base + a * L::kQAtom + lane * 128 + ((c ^ (lane & 7)) << 4),
                                     v[c].x, v[c].y, v[c].z, v[c].w);
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(q_ready);
                return r;
            };
            int64_t orow = w.pos < w.end ? write_q(w, piece_at(w).h0) : -1;
            while (ok && w.pos < w.end) {
                const Piece pc = piece_at(w);
                Walk pw = w;
                // the next piece, found now: its q rows go to L2 at once and
                // into the q tile during this piece's last stage (no product
                // reads q once that stage's S is in)
                bool has_next;
                int64_t rn;
                {
                    Walk wn = w;
                    if (!(ok = piece_after(wn, npc, false))) break;
                    has_next = wn.pos < wn.end;
                    rn = has_next ? out_row(wn, piece_at(wn).h0) : -1;
                }
                if (rn >= 0)
                    for (int b = 0; b < D * 2; b += 128)
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(
                            reinterpret_cast<const unsigned char*>(q + rn * D) + b));
                float m_run = -INFINITY, l_run = 0.f;
                for (int st = 0; st < pc.stages; ++st, ++g) {
                    const int nt = min(kStageTokens, pw.pend - (pw.pt0 + pw.pk * kStageTokens));
                    const int act = pw.pj;            // -1: shared prefix, else member act's tail
                    part_next(pw, context_lens, cap);
                    if (!(ok = wait_tc(&s_full[g & 1], (g >> 1) & 1))) break;
                    tc::fence_after_sync();
                    if (st == pc.stages - 1 && has_next) {
                        // the piece's last S is in: the next piece's q rows
                        // (zeros for a padding column) copy in behind it
                        const uint4* src = reinterpret_cast<const uint4*>(q + (rn < 0 ? 0 : rn) * D);
#pragma unroll
                        for (int c = 0; c < D / 8; ++c) {
                            const uint32_t dst = q_base + (c >> 3) * L::kQAtom + lane * 128 +
                                                 (((c & 7) ^ (lane & 7)) << 4);
                            if (rn >= 0)
                                asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst),
                                             "l"(src + c) : "memory");
                            else
                                st_shared_v4(dst, 0u, 0u, 0u, 0u);
                        }
                    }
                    const uint32_t s_tm = tmem + (g & 1) * kStageTokens;
                    // a member's tail is seen only by that member's columns
                    const int lim = (orow >= 0 && (act < 0 || act == mem)) ? nt : 0;
                    // S is read twice, 32 tokens at a time (the maximum, then
                    // P), which keeps the registers to one chunk; chunks past
                    // the stage's tokens are skipped (no product reads them).
                    // kDense: a full stage of the shared prefix, which every
                    // column sees whole (no per-token masks).
                    auto softmax = [&](auto dense_c) -> bool {
                        constexpr bool kDense = decltype(dense_c)::value;
                        float mx = -INFINITY;
#pragma unroll
                        for (int c = 0; c < kStageTokens / 32; ++c) {
                            if (!kDense && 32 * c >= nt) break;
                            uint32_t r[32];
                            tc::tmem_ld32(s_tm + 32 * c, r);
                            tc::tmem_ld_wait();
                            tc::tmem_ld_fence(r);
                            float m8[8];
#pragma unroll
                            for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (kDense || 32 * c + j < lim)
                                    m8[j & 7] = fmaxf(m8[j & 7], __uint_as_float(r[j]));
                            mx = fmaxf(mx, fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                                 fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))));
                        }
                        mx = mx == -INFINITY ? mx : mx * scale_log2;
                        // lazy rescale: only when the maximum grows by more than 2^8
                        const bool grow = mx > m_run + kRescaleThreshold;
                        float alpha = 1.f;
                        if (grow) {
                            alpha = ex2(m_run - mx);      // 0 the first time
                            m_run = mx;
                            l_run *= alpha;
                        }
                        if (st > 0 && __any_sync(0xffffffffu, grow)) {
                            // O holds the stages before g: let the last of them finish
                            if (!wait_tc(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1)) return false;
                            tc::fence_after_sync();
#pragma unroll
                            for (int c = 0; c < D / 32; ++c) {
                                uint32_t r[32];
                                tc::tmem_ld32(o_tm + 32 * c, r);
                                tc::tmem_ld_wait();
                                tc::tmem_ld_fence(r);
#pragma unroll
                                for (int e = 0; e < 32; ++e)
                                    r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                                tc::tmem_st32(o_tm + 32 * c, r);
                            }
                        }
                        const float mu = m_run == -INFINITY ? 0.f : m_run;
                        // P over S, per 32 tokens c: hi in columns 32c..32c+15
                        // and (bf16) lo in 32c+16..32c+31
                        const float2 sc2 = make_float2(scale_log2, scale_log2);
                        const float2 nm2 = make_float2(-mu, -mu);
                        float2 ls4[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) ls4[k] = make_float2(0.f, 0.f);
#pragma unroll
                        for (int c = 0; c < kStageTokens / 32; ++c) {
                            if (!kDense && 32 * c >= nt) break;
                            uint32_t r[32];
                            tc::tmem_ld32(s_tm + 32 * c, r);
                            tc::tmem_ld_wait();
                            tc::tmem_ld_fence(r);
                            uint32_t hi[16];
                            [[maybe_unused]] uint32_t lo[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float2 xv = ffma2(make_float2(__uint_as_float(r[2 * e]),
                                                                    __uint_as_float(r[2 * e + 1])),
                                                        sc2, nm2);
                                const float p0 = kDense || 32 * c + 2 * e < lim ? ex2(xv.x) : 0.f;
                                const float p1 = kDense || 32 * c + 2 * e + 1 < lim ? ex2(xv.y) : 0.f;
                                ls4[e & 3] = fadd2(ls4[e & 3], make_float2(p0, p1));
                                hi[e] = E::pack2(p0, p1);
                                if constexpr (kBf) {
                                    const float2 d = fsub2(make_float2(p0, p1), E::unpack2(hi[e]));
                                    lo[e] = E::pack2(d.x, d.y);
                                }
                            }
                            tc::tmem_st16(s_tm + 32 * c, hi);
                            if constexpr (kBf) tc::tmem_st16(s_tm + 32 * c + 16, lo);
                        }
                        const float2 l01 = fadd2(fadd2(ls4[0], ls4[1]), fadd2(ls4[2], ls4[3]));
                        l_run += l01.x + l01.y;
                        return true;
                    };
                    // uniform: a full stage of the shared prefix
                    const bool dense = act < 0 && nt == kStageTokens;
                    if (!(ok = dense ? softmax(std::true_type{}) : softmax(std::false_type{}))) break;
                    if (nt & 15) {
                        // V rows nt .. 16 ceil(nt / 16) - 1 hold other data (or
                        // none yet): zeroed, so that 0 * v stays 0 in the last step
                        const uint32_t vb = v_base + (g % kStages) * L::kTile;
                        const int zr = 16 - (nt & 15);
                        for (int i = lane; i < zr * kAtoms * 8; i += 32) {
                            const int r = nt + i / (kAtoms * 8);
                            const int a = (i >> 3) % kAtoms;
                            st_shared_v4(vb + a * L::kAtom + r * 128 + (i & 7) * 16, 0u, 0u, 0u, 0u);
                        }
                        tc::fence_proxy_async_smem();
                    }
                    const bool q_in = st == pc.stages - 1 && has_next;
                    if (q_in) {
                        // the next piece's q rows are in: its first S can be
                        // computed while this piece's O is read out
                        cp_async_wait_all();
                        tc::fence_proxy_async_smem();
                    }
                    tc::tmem_st_wait();
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&p_full[g & 1]);
                        if (q_in) mbar_arrive(q_ready);
                    }
                }
                if (!ok) break;
                // the piece's last product, then O out of tensor memory, 32
                // values at a time, straight to the output or the workspace
                if (!(ok = wait_tc(&pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1))) break;
                tc::fence_after_sync();
                const int64_t wr = ws_base(w, pc) + int64_t(pc.seg) * cstride + lane;
                // the whole stream was here: final, normalised output
                const float inv = l_run == 0.f ? 0.f : 1.f / l_run;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tc::tmem_ld32(o_tm + 32 * c, o);
                    tc::tmem_ld_wait();
                    tc::tmem_ld_fence(o);
                    if (orow >= 0 && pc.nseg == 1) {
                        uint4* dst = reinterpret_cast<uint4*>(out + orow * D + 32 * c);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float* f = reinterpret_cast<const float*>(&o[8 * j]);
                            dst[j] = make_uint4(E::pack2(f[0] * inv, f[1] * inv),
                                                E::pack2(f[2] * inv, f[3] * inv),
                                                E::pack2(f[4] * inv, f[5] * inv),
                                                E::pack2(f[6] * inv, f[7] * inv));
                        }
                    } else if (orow >= 0) {
                        float4* dst = reinterpret_cast<float4*>(ws_o + wr * D + 32 * c);
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                                                 __uint_as_float(o[4 * j + 2]),
                                                 __uint_as_float(o[4 * j + 3]));
                    }
                }
                if (orow >= 0 && pc.nseg > 1) {
                    ws_m[wr] = m_run;
                    ws_l[wr] = l_run;
                }
                tc::fence_before_sync();
                if (pc.nseg > 1) {
                    // hand the partials to the publishers (once they have
                    // taken the piece before last, which used the same barriers)
                    if (njob > 1 && !(ok = wait_tc(&pub_free_f[njob & 1], ((njob - 2) >> 1) & 1)))
                        break;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&pub_full_f[njob & 1]);
                    ++njob;
                }
                if (!(ok = piece_after(w, npc, true))) break;
                ++npc;
                orow = rn;
            }
            if (*abort_flag != 0 && lane == 0) {
                // let copies already issued into the ring land before the CTA exits
                const int n_issued = *issued;
                for (int s2 = int(g); s2 < n_issued; ++s2)
                    if (!mbar_wait(&full[s2 % kStages], (s2 / kStages) & 1)) break;
            }
        }
        tc::fence_before_sync();
        asm volatile("bar.sync 3, 64;" ::: "memory");
        if (warp == 1) {
            tc::fence_after_sync();
            tc::tmem_dealloc(tmem, kTmemCols);
        }
        return;
    }

    // ---------------- consumer warps ----------------
    const int j8 = lane >> 3, r8 = lane & 7;     // ldmatrix: matrix index, row within it
    // columns of a stream, in 1 or 2 tiles of 8; this warp's tokens within a
    // stage (16 or 32) and its first column
    const int ncols = GH * nq;
    const int ctiles = kMQ ? (ncols <= kHeadsN ? 1 : 2) : 1;
    const int wpc = kConsumerWarps / ctiles;     // warps per column tile
    const int tb = kMQ ? (warp % wpc) * 16 * ctiles : warp * 16;
    const int col0 = kMQ ? (warp / wpc) * kHeadsN : 0;
    const uint32_t k_base0 = smem_u32(smem + L::kK);
    const uint32_t v_base0 = smem_u32(smem + L::kV);
    const float2 neg1 = make_float2(-1.f, -1.f);
    uint32_t gs = 0;                             // stages consumed so far
    bool aborted = false;
    // P enters PV as one 16-bit value when the products run on fp16 (fp16
    // pools, FP8 pools, whose codes widen to fp16): 2^-11 relative rounding,
    // as small as q's own; with bf16 operands (2^-9) as the hi + lo pair
    constexpr bool kLoP = !std::is_same<TM, __half>::value;

    // output row of column n (head h0 + n / nq, query n % nq) of stream x
    // whose unit starts at head h0 (-1: a padding column)
    auto col_row = [&](const Walk& x, int h0, int n) -> int64_t {
        const int hh = n / nq, j = n - hh * nq;
        return hh < GH ? ((int64_t)x.s * nq + j) * H + h0 + hh : -1;
    };

    uint32_t npub = 0;                           // pieces handed to the publisher warp
    while (w.pos < w.end) {
        // ---- one stream piece: stages [w.off, min(w.L, w.off + w.end - w.pos)) of (s, u)
        const int kvh = w.u / groups;
        const int h0 = kvh * G + (w.u % groups) * GH;     // first q head of this unit
        const long left = w.end - w.pos;
        const int piece_stages = int(left < long(w.L - w.off) ? left : long(w.L - w.off));
        const long c_first = w.start / w.per_cta;
        const long c_last = (w.start + w.L - 1) / w.per_cta;
        const int nseg = int(c_last - c_first + 1);
        const int seg = int(long(w.bi) - c_first);
        // q^T as the MMA B operand: lane holds head lane/4, dims 16ks + 2(lane%4) + {0,1}
        // (register 0) and the same + 8 (register 1); heads past GH are zero.
        uint32_t qb[KS][2];
        {
            // column n: head h0 + n / nq, query token n % nq (verify); member
            // n / GH, head h0 + n % GH (shared-prefix mode)
            const int64_t qrow_c = col_row(w, h0, col0 + (lane >> 2));
            const bool qv = qrow_c >= 0;
            const int64_t qrow_i = qv ? qrow_c : 0;
            const T* qrow = q + qrow_i * D + 2 * (lane & 3);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                if constexpr (kNative) {
                    // native FP8 path: k step ks pairs dims 16ks + 4t, +1 (register 0)
                    // and 16ks + 4t + 2, +3 (register 1), t = lane % 4, the order in
                    // which K comes out of its byte fragments
                    const T* qr = q + qrow_i * D + 16 * ks + 4 * (lane & 3);
                    const uint2 v = qv ? __ldg(reinterpret_cast<const uint2*>(qr))
                                       : make_uint2(0u, 0u);
                    qb[ks][0] = v.x;
                    qb[ks][1] = v.y;
                } else {
                    qb[ks][0] =
                        qv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks)) : 0u;
                    qb[ks][1] =
                        qv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8)) : 0u;
                }
                if constexpr (kF8 && !std::is_same<T, __half>::value) {
                    // q rounded to the fp16 operand type of the FP8 path
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const float2 f = Elem<T>::unpack2(qb[ks][r]);
                        qb[ks][r] = Elem<__half>::pack2(f.x, f.y);
                    }
                }
            }
        }
        // The next piece's q rows into L1 now, so that its loads at the piece
        // switch hit instead of waiting on HBM: the next stream of the range is
        // (s + 1, u) (an empty sequence is skipped by the walk, so that prefetch
        // is merely wasted).
        if (piece_stages < w.end - w.pos) {
            const int nu = w.u;                         // same unit, next sequence
            const int ns = w.s + 1;
            if (ns < B) {
                const int n = col0 + (lane >> 2);
                const int qh = n / nq, qj = n - qh * nq;
                if (qh < GH) {
                    const int nh0 = (nu / groups) * G + (nu % groups) * GH;
                    const T* nrow = q + (((int64_t)ns * nq + qj) * H + nh0 + qh) * D;
                    // the column's four lanes cover its row (D / 4 values each)
                    asm volatile("prefetch.global.L1 [%0];" ::"l"(nrow + (lane & 3) * (D / 4)));
                }
            }
        }
        // FP8 pools: the K scale joins the softmax scale, the V scale the output
        const float sl2 = kF8 ? scale_log2 * __ldg(k_scale + kvh) : scale_log2;
        // O^T fragments: m-tile mt covers dims 16mt..16mt+15; lane holds dims
        // 16mt + lane/4 (regs 0,1) and + 8 (regs 2,3), heads 2(lane%4) and + 1.
        float o[KS][4];
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};
        // columns 2(lane%4) + h: query token j sits nq - 1 - j positions
        // before the context end and sees no key past itself
        int dj[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) dj[h] = kMQ ? nq - 1 - (col0 + 2 * (lane & 3) + h) % nq : 0;

        for (int st = 0; st < piece_stages;) {
            // the native FP8 path takes two stages of the piece at a time
            const int nst = (kNative && st + 1 < piece_stages) ? 2 : 1;
            const int slot = gs % kStages;
            bool got = mbar_wait(&full[slot], (gs / kStages) & 1);
            if (nst == 2) got = got && mbar_wait(&full[(gs + 1) % kStages], ((gs + 1) / kStages) & 1);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) {
                    flag_error(dev_err, PD_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                aborted = true;
                break;                   // skip the piece's other stages
            }
            // context from this stage on, and the stage's tokens
            const int rem = w.ctx - (w.off + st) * kStageTokens;
            const int nt = min(kStageTokens, rem);
            // FP8 pools: this warp widens its own 16 rows of K and V to fp16 in
            // the one 16-bit tile (no other warp reads them), then frees the raw
            // stage for the next copy right away.
            const int tslot = kF8 ? 0 : slot;
            if constexpr (kF8 && !kNative) {
                if (tb < nt) {
                    // K and V widened exactly by the E4M3 -> fp16 conversion
                    constexpr int kChunks = D / 16;          // 16-byte chunks per FP8 row
                    const unsigned char* srck = smem + L::kK8 + slot * L::kTile8 + tb * D;
                    const unsigned char* srcv = smem + L::kV8 + slot * L::kTile8 + tb * D;
                    // (16 rows x kChunks) chunks, 32 per pass: a fixed trip count, so
                    // every load of the stage is issued up front
                    uint4 rk[16 * kChunks / 32], rv[16 * kChunks / 32];
#pragma unroll
                    for (int it = 0; it < 16 * kChunks / 32; ++it) {
                        const int i = it * 32 + lane;
                        rk[it] = *reinterpret_cast<const uint4*>(srck + i * 16);
                        rv[it] = *reinterpret_cast<const uint4*>(srcv + i * 16);
                    }
#pragma unroll
                    for (int it = 0; it < 16 * kChunks / 32; ++it) {
                        const int i = it * 32 + lane;
                        const int row = i / kChunks, c8 = i % kChunks;
                        const uint32_t wk[4] = {rk[it].x, rk[it].y, rk[it].z, rk[it].w};
                        const uint32_t wv[4] = {rv[it].x, rv[it].y, rv[it].z, rv[it].w};
                        uint32_t hk[8], hv[8];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            hk[2 * j] = e4m3x2_to_f16x2(uint16_t(wk[j] & 0xffffu));
                            hk[2 * j + 1] = e4m3x2_to_f16x2(uint16_t(wk[j] >> 16));
                            hv[2 * j] = e4m3x2_to_f16x2(uint16_t(wv[j] & 0xffffu));
                            hv[2 * j + 1] = e4m3x2_to_f16x2(uint16_t(wv[j] >> 16));
                        }
                        st_shared_v4(swz<D>(k_base0, tb + row, 2 * c8), hk[0], hk[1], hk[2], hk[3]);
                        st_shared_v4(swz<D>(k_base0, tb + row, 2 * c8 + 1), hk[4], hk[5], hk[6],
                                     hk[7]);
                        st_shared_v4(swz<D>(v_base0, tb + row, 2 * c8), hv[0], hv[1], hv[2], hv[3]);
                        st_shared_v4(swz<D>(v_base0, tb + row, 2 * c8 + 1), hv[4], hv[5], hv[6],
                                     hv[7]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
            if constexpr (kNative) {
              // NS consecutive stages of the piece (their slots are consecutive
              // in the ring): this warp's 16 tokens of each, processed together
              auto nbody = [&](auto ns_c) {
                constexpr int NS = decltype(ns_c)::value;
                int nts[NS];
                uint32_t k8[NS], v8[NS];
#pragma unroll
                for (int sb = 0; sb < NS; ++sb) {
                    const int sl = (gs + sb) % kStages;
                    nts[sb] = min(kStageTokens, rem - sb * kStageTokens);
                    k8[sb] = smem_u32(smem + L::kK8 + sl * L::kTile8);
                    v8[sb] = smem_u32(smem + L::kV8 + sl * L::kTile8);
                }
                // a second stage exists only after a full first one, so a warp
                // without tokens in the first stage has none in the second
                if (tb >= nts[0]) {
                    __syncwarp();
                    if (lane == 0)
                        for (int sb = 0; sb < NS; ++sb) mbar_arrive(&empty[(gs + sb) % kStages]);
                    return;
                }
                // ---- fragments straight from the raw E4M3 stages (128-byte rows,
                // swizzled): ldmatrix moves bytes, the conversion happens in registers
                const int lrow = tb + r8 + 8 * (j8 & 1);
                uint32_t kr[NS][D / 32][4], vr[NS][D / 32][4];
#pragma unroll
                for (int sb = 0; sb < NS; ++sb)
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        wmma16::ldsm_x4(kr[sb][c], swz128(k8[sb], lrow, 2 * c + (j8 >> 1)));
                        wmma16::ldsm_x4_t(vr[sb][c], swz128(v8[sb], lrow, 2 * c + (j8 >> 1)));
                    }
                __syncwarp();
                if (lane == 0)                               // the raw stages are free
                    for (int sb = 0; sb < NS; ++sb) mbar_arrive(&empty[(gs + sb) % kStages]);
                // ---- S^T = K q^T: register j of block c holds row g (+8 for odd j),
                // bytes 4t..4t+3 of dims 32c + 16 (j / 2) ..; bytes 0, 1 and 2, 3
                // widen exactly to the two fp16 pairs of the A fragment (one
                // conversion each: fewer integer instructions than assembling the
                // fp16 bits by hand, which kept the ALU pipe the busiest)
                float acc[NS][2][4];
#pragma unroll
                for (int sb = 0; sb < NS; ++sb)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[sb][0][e] = acc[sb][1][e] = 0.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
                        for (int sb = 0; sb < NS; ++sb) {
                            uint32_t a[4];
                            a[0] = e4m3x2_to_f16x2(uint16_t(kr[sb][c][2 * h2] & 0xffffu));
                            a[1] = e4m3x2_to_f16x2(uint16_t(kr[sb][c][2 * h2 + 1] & 0xffffu));
                            a[2] = e4m3x2_to_f16x2(uint16_t(kr[sb][c][2 * h2] >> 16));
                            a[3] = e4m3x2_to_f16x2(uint16_t(kr[sb][c][2 * h2 + 1] >> 16));
                            const int ks = 2 * c + h2;
                            wmma16::Mma<TM>::run(acc[sb][ks & 1], a, qb[ks][0], qb[ks][1]);
                        }
                    }
                }
                const int tok0 = tb + (lane >> 2);
                float x[NS][4];
#pragma unroll
                for (int sb = 0; sb < NS; ++sb)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int tok = tok0 + (i >> 1) * 8;
                        x[sb][i] = tok < nts[sb] ? (acc[sb][0][i] + acc[sb][1][i]) * sl2
                                                 : -INFINITY;
                    }
                float mx[2] = {fmaxf(x[0][0], x[0][2]), fmaxf(x[0][1], x[0][3])};
#pragma unroll
                for (int sb = 1; sb < NS; ++sb) {
                    mx[0] = fmaxf(mx[0], fmaxf(x[sb][0], x[sb][2]));
                    mx[1] = fmaxf(mx[1], fmaxf(x[sb][1], x[sb][3]));
                }
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
                uint32_t bh0[NS], bh1[NS];
                [[maybe_unused]] uint32_t bl0[NS], bl1[NS];   // the lo half (kLoP only)
                float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                for (int sb = 0; sb < NS; ++sb) {
                    const float p0 = ex2(x[sb][0] - m_run[0]), p1 = ex2(x[sb][1] - m_run[1]);
                    const float p2 = ex2(x[sb][2] - m_run[0]), p3 = ex2(x[sb][3] - m_run[1]);
                    if (sb == 0) {
                        ls0 = p0 + p2;
                        ls1 = p1 + p3;
                    } else {
                        ls0 += p0 + p2;
                        ls1 += p1 + p3;
                    }
                    const uint32_t hi0 = E::pack2(p0, p1), hi1 = E::pack2(p2, p3);
                    bh0[sb] = wmma16::movm_t(hi0);
                    bh1[sb] = wmma16::movm_t(hi1);
                    if constexpr (kLoP) {
                        const float2 lo0 = ffma2(E::unpack2(hi0), neg1, make_float2(p0, p1));
                        const float2 lo1 = ffma2(E::unpack2(hi1), neg1, make_float2(p2, p3));
                        bl0[sb] = wmma16::movm_t(E::pack2(lo0.x, lo0.y));
                        bl1[sb] = wmma16::movm_t(E::pack2(lo1.x, lo1.y));
                    }
                }
                l_run[0] += ls0;
                l_run[1] += ls1;
                // ---- O^T += V^T P^T: register j of block c holds tokens 2t, 2t+1
                // (+8 for odd j) x dims 2g, 2g+1 of chunk 2c + j / 2; m-tile 2c + j/2
                // has rows g -> dim 2g and g + 8 -> dim 2g + 1 of that chunk
                const int tk = tb + 2 * (lane & 3);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
                        for (int sb = 0; sb < NS; ++sb) {
                            uint32_t a[4];
                            a[0] = e4m3_pair_to_f16x2<0x4420u>(vr[sb][c][2 * h2]);
                            a[1] = e4m3_pair_to_f16x2<0x4431u>(vr[sb][c][2 * h2]);
                            a[2] = e4m3_pair_to_f16x2<0x4420u>(vr[sb][c][2 * h2 + 1]);
                            a[3] = e4m3_pair_to_f16x2<0x4431u>(vr[sb][c][2 * h2 + 1]);
                            if (tb + 16 > nts[sb]) {
                                // tokens past the context: their V bytes are other data
                                const int n = nts[sb];
                                const uint32_t m01 = (tk < n ? 0xffffu : 0u) |
                                                     (tk + 1 < n ? 0xffff0000u : 0u);
                                const uint32_t m23 = (tk + 8 < n ? 0xffffu : 0u) |
                                                     (tk + 9 < n ? 0xffff0000u : 0u);
                                a[0] &= m01;
                                a[1] &= m01;
                                a[2] &= m23;
                                a[3] &= m23;
                            }
                            const int mt = 2 * c + h2;
                            wmma16::Mma<TM>::run(o[mt], a, bh0[sb], bh1[sb]);
                            if constexpr (kLoP) wmma16::Mma<TM>::run(o[mt], a, bl0[sb], bl1[sb]);
                        }
                    }
                }
              };
              if (nst == 2) nbody(std::integral_constant<int, 2>{});
              else nbody(std::integral_constant<int, 1>{});
            } else {
              // NS sub-tiles of 16 tokens (tb .. tb + 16 NS - 1) processed together:
              // their products interleave and share one max, rescale and shuffle
              // round; NS = 1 is the decode layout, NS = 2 the two-tile verify one
              auto body = [&](auto ns_c) {
                constexpr int NS = decltype(ns_c)::value;
                if (tb >= nt) return;
                const uint32_t kb = k_base0 + tslot * L::kTile;
                const uint32_t vb = v_base0 + tslot * L::kTile;
                const bool partial = tb + 16 * NS > nt;
                if (partial) {
                    // V rows past the context end hold other data or were never
                    // loaded this round: zero them so that 0 * v stays 0.
                    unsigned char* vrow = smem + L::kV + tslot * L::kTile;
                    for (int i = lane; i < 16 * NS * kAtoms * 8; i += 32) {
                        const int tok = tb + i / (kAtoms * 8);
                        if (tok >= nt) {
                            const int a = (i / 8) % kAtoms, c = i % 8;
                            *reinterpret_cast<uint4*>(vrow + a * L::kAtom + tok * 128 + c * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    __syncwarp();
                }
                // ---- S^T[16 tokens][8 columns] = K q^T per sub-tile (two accumulators each)
                float acc[NS][2][4];
#pragma unroll
                for (int sb = 0; sb < NS; ++sb)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[sb][0][e] = acc[sb][1][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
                    for (int sb = 0; sb < NS; ++sb) {
                        uint32_t a[4];
                        wmma16::ldsm_x4(a, swz<D>(kb, tb + 16 * sb + r8 + 8 * (j8 & 1),
                                                  2 * ks + (j8 >> 1)));
                        wmma16::Mma<TM>::run(acc[sb][ks & 1], a, qb[ks][0], qb[ks][1]);
                    }
                }
                // lane holds tokens tb + 16 sb + lane/4 (0,1) and + 8 (2,3); columns
                // 2(lane%4) + {0,1}.  Tokens past a column's limit are masked: the
                // stage's end (decode); the query's causal limit (verify).
                int lim[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) lim[h] = kMQ ? rem - dj[h] : nt;
                float x[NS][4];
#pragma unroll
                for (int sb = 0; sb < NS; ++sb)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int tok = tb + 16 * sb + (lane >> 2) + (i >> 1) * 8;
                        x[sb][i] = tok < lim[i & 1]
                                       ? (acc[sb][0][i] + acc[sb][1][i]) * sl2 : -INFINITY;
                    }
                // ---- online softmax per column (lane-local state, 3 shuffles per column)
                float mx[2] = {fmaxf(x[0][0], x[0][2]), fmaxf(x[0][1], x[0][3])};
#pragma unroll
                for (int sb = 1; sb < NS; ++sb) {
                    mx[0] = fmaxf(mx[0], fmaxf(x[sb][0], x[sb][2]));
                    mx[1] = fmaxf(mx[1], fmaxf(x[sb][1], x[sb][3]));
                }
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
                // a verify column may not have seen a key yet (m = -inf): its p are 0
                const float mu0 = kMQ && m_run[0] == -INFINITY ? 0.f : m_run[0];
                const float mu1 = kMQ && m_run[1] == -INFINITY ? 0.f : m_run[1];
                uint32_t bh0[NS], bh1[NS];
                [[maybe_unused]] uint32_t bl0[NS], bl1[NS];   // the lo half (kLoP only)
                float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                for (int sb = 0; sb < NS; ++sb) {
                    const float p0 = ex2(x[sb][0] - mu0), p1 = ex2(x[sb][1] - mu1);
                    const float p2 = ex2(x[sb][2] - mu0), p3 = ex2(x[sb][3] - mu1);
                    if (sb == 0) {
                        ls0 = p0 + p2;
                        ls1 = p1 + p3;
                    } else {
                        ls0 += p0 + p2;
                        ls1 += p1 + p3;
                    }
                    // P as hi + lo 16-bit pairs, transposed into B-operand layout
                    const uint32_t hi0 = E::pack2(p0, p1), hi1 = E::pack2(p2, p3);
                    bh0[sb] = wmma16::movm_t(hi0);
                    bh1[sb] = wmma16::movm_t(hi1);
                    if constexpr (kLoP) {
                        const float2 lo0 = ffma2(E::unpack2(hi0), neg1, make_float2(p0, p1));
                        const float2 lo1 = ffma2(E::unpack2(hi1), neg1, make_float2(p2, p3));
                        bl0[sb] = wmma16::movm_t(E::pack2(lo0.x, lo0.y));
                        bl1[sb] = wmma16::movm_t(E::pack2(lo1.x, lo1.y));
                    }
                }
                l_run[0] += ls0;
                l_run[1] += ls1;
                // ---- O^T[dims][columns] += V^T P^T
#pragma unroll
                for (int mt = 0; mt < KS; ++mt) {
#pragma unroll
                    for (int sb = 0; sb < NS; ++sb) {
                        uint32_t a[4];
                        wmma16::ldsm_x4_t(a, swz<D>(vb, tb + 16 * sb + r8 + 8 * (j8 >> 1),
                                                    2 * mt + (j8 & 1)));
                        wmma16::Mma<TM>::run(o[mt], a, bh0[sb], bh1[sb]);
                        if constexpr (kLoP) wmma16::Mma<TM>::run(o[mt], a, bl0[sb], bl1[sb]);
                    }
                }
                if (partial && !kF8) tc::fence_proxy_async_smem();   // zeros before the next TMA write
              };
              if constexpr (kMQ) {
                  if (ctiles == 2) body(std::integral_constant<int, 2>{});
                  else body(std::integral_constant<int, 1>{});
              } else {
                  body(std::integral_constant<int, 1>{});
              }
            }
            __syncwarp();
            if (!kF8 && lane == 0) mbar_arrive(&empty[slot]);
            st += nst;
            gs += nst;
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
        // lane-major records (o, then m and l), 16-byte accesses: a quarter-warp's
        // eight records start on distinct 4-bank groups, so no conflicts
        auto put = [&](int buf) {
            float4* x = reinterpret_cast<float4*>(xchg + (buf * 32 + lane) * L::kFrag);
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
                x[mt] = make_float4(o[mt][0], o[mt][1], o[mt][2], o[mt][3]);
            x[KS] = make_float4(m_run[0], m_run[1], l_run[0], l_run[1]);
        };
        auto take = [&](int buf) {
            frag_combine<KS>(o, m_run, l_run, reinterpret_cast<const float4*>(
                                                  xchg + (buf * 32 + lane) * L::kFrag));
        };
        if constexpr (!kMQ) {
            // Warps 2, 3 hand their shares to 0, 1, which combine them and hand
            // the two partials to the publisher warp with the piece's
            // description; then all four go straight on.  The buffer is the
            // only thing shared with the publisher, which frees it as soon as
            // it has read it.
            if (npub > 0 && warp >= 2) {
                const bool ok = __all_sync(0xffffffffu, mbar_wait(pub_free, (npub - 1) & 1));
                if (!ok && lane == 0) {
                    flag_error(dev_err, PD_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
            }
            if (warp >= 2) put(warp - 2);
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
            if (warp < 2) {
                take(warp);
                __syncwarp();
                put(warp);                     // own slot, already read by this lane
                if (warp == 0 && lane == 0) {
                    int32_t* meta = reinterpret_cast<int32_t*>(smem + L::kMeta);
                    meta[0] = w.s;
                    meta[1] = w.u;
                    meta[2] = nseg;
                    meta[3] = seg;
                    meta[4] = long(piece_stages) == left ? 1 : 0;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(pub_full);
            }
            ++npub;
        } else {
            // one tile: warps 2, 3 hand over to 0, 1, then warp 1 to 0; two
            // tiles: warp 1 hands over to 0 and warp 3 to 2 (same tile); four
            // tiles: each warp holds its own columns whole
            if (ctiles == 1) {
                if (warp >= 2) put(warp - 2);
                asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
                if (warp < 2) take(warp);
                if (warp == 1) {
                    __syncwarp();
                    put(1);                  // own partner slot, already read by this warp
                }
                asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
                if (warp == 0) take(1);
            } else if (ctiles == 2) {
                if (warp & 1) put(warp >> 1);
                asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
                if (!(warp & 1)) take(warp >> 1);
            }
            // The exchange buffer has been read: the other warps go on to the
            // next piece while the warp(s) holding the result write it, publish
            // it and perhaps merge the stream. They fall behind by that much and
            // catch up on stages already in the ring (consuming is faster than
            // streaming).
            asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
            const bool leader = (warp % wpc) == 0;   // holds its tile's result
            // workspace index of a column's partial for piece `p` of this
            // stream: per output row
            auto ws_index = [&](int64_t row, long p) -> int64_t { return row * max_segs + p; };
            auto merge_tile = [&]() {               // verify
                const int n = col0 + (lane >> 2);
                const int64_t orow = col_row(w, h0, n);
                merge_rows<T, D, 1>(out, ws_o, ws_m, ws_l, orow, orow < 0 ? 0 : ws_index(orow, 0), 1,
                                    nseg, lane);
            };
            // the arrival counter is read now, so that its latency overlaps the
            // piece's writes and fence; a value changed meanwhile costs one more CAS
            unsigned long long* cnt = ws_cnt + (int64_t)w.s * units + w.u;
            unsigned long long cnt0 = 0;
            if (nseg > 1 && warp == 0 && lane == 0)
                cnt0 = *reinterpret_cast<volatile unsigned long long*>(cnt);
            if (leader) {
                // lane: columns ha, ha + 1; dims 16mt + lane/4 and + 8
                const int ha = 2 * (lane & 3);
                const int d0 = lane >> 2;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int c = col0 + ha + h;
                    const int64_t row = col_row(w, h0, c);
                    if (row < 0) continue;
                    if (nseg == 1) {
                        // the whole stream was here: final, normalised output
                        // (0 for a query that saw no key)
                        const float inv = l_run[h] == 0.f ? 0.f : 1.f / l_run[h];
                        T* orow = out + row * D + d0;
#pragma unroll
                        for (int mt = 0; mt < KS; ++mt) {
                            orow[16 * mt] = T(o[mt][h] * inv);
                            orow[16 * mt + 8] = T(o[mt][2 + h] * inv);
                        }
                    } else {
                        const int64_t r = ws_index(row, seg);
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
                if (nseg > 1 && ctiles == 1) {
                    // publish this piece, count it; the last of the stream's
                    // pieces to arrive merges them all
                    __threadfence();
                    __syncwarp();
                    uint32_t last = 0;
                    if (lane == 0) last = arrive_piece(cnt, tag, nseg, cnt0) ? 1u : 0u;
                    last = __shfl_sync(0xffffffffu, last, 0);
                    if (last) {
                        __threadfence();
                        merge_tile();
                    }
                }
            }
            if (ctiles > 1 && nseg > 1 && leader) {
                // every tile's leader (named barrier 2) has written its rows of
                // the piece before it is counted; then each merges its own tile
                // if the piece was the last
                volatile int32_t* last_flag = reinterpret_cast<int32_t*>(smem + L::kMisc + 8);
                __threadfence();
                asm volatile("bar.sync 2, %0;" ::"r"(ctiles * 32) : "memory");
                if (warp == 0 && lane == 0) *last_flag = arrive_piece(cnt, tag, nseg, cnt0) ? 1 : 0;
                asm volatile("bar.sync 2, %0;" ::"r"(ctiles * 32) : "memory");
                if (*last_flag) {
                    __threadfence();
                    merge_tile();
                }
            }
        }
        w.off += piece_stages;
        w.pos += piece_stages;
        if (w.off == w.L && w.pos < w.end) walk_next_stream<kFork>(w, context_lens, B, cap, S, fk);
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

// Launch tags for the arrival counters: 44 bits, never 0, distinct for
// every launch of this process (a salted counter).
unsigned long long next_launch_tag() {
    static const unsigned long long salt = [] {
        unsigned long long x = uint64_t(std::chrono::steady_clock::now().time_since_epoch().count());
        x ^= uint64_t(reinterpret_cast<uintptr_t>(&salt)) << 17;
        x ^= uint64_t(getpid()) << 40;
        // splitmix64 finaliser to spread the bits
        x ^= x >> 30; x *= 0xbf58476d1ce4e5b9ull;
        x ^= x >> 27; x *= 0x94d049bb133111ebull;
        x ^= x >> 31;
        return x;
    }();
    static std::atomic<unsigned long long> counter{0};
    const unsigned long long t = (salt + counter.fetch_add(1, std::memory_order_relaxed)) &
                                 ((1ull << (64 - kCountBits)) - 1);
    return t == 0 ? 1 : t;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
    size_t o, m, l, cnt, total;
};

WsLayout ws_layout(int B, int H, int D, int P) {
    WsLayout w;
    const size_t rows = size_t(B) * H;
    w.o = 0;
    w.m = align256(rows * P * D * sizeof(float));
    w.l = w.m + align256(rows * P * sizeof(float));
    w.cnt = w.l + align256(rows * P * sizeof(float));
    w.total = w.cnt + align256(rows * sizeof(unsigned long long));   // streams <= rows
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

// Largest divisor of G whose columns fit max_cols: 8 heads for decode; 16
// (two tiles of N = 8) for verification, GH * nq; 32 (the tensor-core rows
// read) in shared-prefix mode, GH * Mmax.
int heads_per_unit(int G, int cols_per_head, int max_cols) {
    for (int g = std::min(G, max_cols / cols_per_head); g >= 1; --g)
        if (G % g == 0) return g;
    return 1;
}

// Most CTAs a decode launch uses: two per SM, at most kMaxGrid (so that the
// shared-prefix workspace can be sized without asking the device).
constexpr int kMaxGrid = 1024;

// Shared-prefix workspace: partials of (unit, piece, column) with at most
// n_groups + kMaxGrid / units pieces per unit, then per-(group, unit) counters.
WsLayout fork_ws_layout(int n_groups, int max_group, int H, int Hk, int D, int* units_out,
                        int* ppu_max_out) {
    const int G = H / Hk;
    const int GH = heads_per_unit(G, max_group, 4 * kHeadsN);
    const int units = Hk * (G / GH);
    const int ncols = GH * max_group;
    const int cstride = (ncols <= kHeadsN ? 1 : ncols <= 2 * kHeadsN ? 2 : 4) * kHeadsN;
    const int ppu = n_groups + std::max(1, kMaxGrid / units);
    const size_t rows = size_t(units) * ppu * cstride;
    WsLayout w;
    w.o = 0;
    w.m = align256(rows * D * sizeof(float));
    w.l = w.m + align256(rows * sizeof(float));
    w.cnt = w.l + align256(rows * sizeof(float));
    w.total = w.cnt + align256(size_t(n_groups) * units * sizeof(unsigned long long));
    if (units_out) *units_out = units;
    if (ppu_max_out) *ppu_max_out = ppu;
    return w;
}

template <typename T, int D, bool kF8, bool kMQ, bool kFork>
pd_status launch_decode_t(const DecodeArgs& a) {
    using Lt = DecodeSmem<D, kF8, kFork>;
    const int G = a.H / a.Hk;
    const int nq = kMQ && !kFork ? a.nq : 1;
    const int GH = kFork ? heads_per_unit(G, a.max_group, 4 * kHeadsN)
                         : heads_per_unit(G, nq, kMQ ? 2 * kHeadsN : kHeadsN);
    CUtensorMap tm_k, tm_v;
    const unsigned long long rows = (unsigned long long)a.NB * a.Hk * a.S;
    if (rows > 0x7fffffffull) return PD_ERR_UNSUPPORTED;   // TMA row coordinate is int32
    const bool maps_ok = kF8 ? (encode_pool_map_u8(&tm_k, a.key_cache, D, rows, a.S, Lt::kNative) &&
                                encode_pool_map_u8(&tm_v, a.value_cache, D, rows, a.S, Lt::kNative))
                             : (encode_pool_map(&tm_k, a.key_cache, D, rows, a.S, a.dt) &&
                                encode_pool_map(&tm_v, a.value_cache, D, rows, a.S, a.dt));
    if (!maps_ok) return launch_result(cudaErrorInvalidValue);
    auto kern = paged_decode_split_kernel<T, D, kF8, kMQ, kFork>;
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
    // persistent grid: two CTAs per SM (shared memory bound), at most
    // kMaxGrid, rounded down to a multiple of the units so that every unit
    // group has the same size
    const int units = a.Hk * (G / GH);
    const int slots = std::min(2 * sm_count(dev), kMaxGrid);
    const int members = std::max(1, slots / units);
    const unsigned grid = unsigned(units * members);
    char* base = static_cast<char*>(a.workspace);
    WsLayout w;
    int P = 1;
    ForkArgs fk{a.grp_start, a.grp_shared, a.B, a.max_group, 0};
    if constexpr (kFork) {
        w = fork_ws_layout(a.n_groups, a.max_group, a.H, a.Hk, a.D, nullptr, nullptr);
        fk.ppu = a.n_groups + members;
    } else {
        P = decode_num_partitions(a.max_context_len);   // pieces per stream, at most
        w = ws_layout(a.B * nq, a.H, a.D, P);
    }
    float* ws_o = reinterpret_cast<float*>(base + w.o);
    float* ws_m = reinterpret_cast<float*>(base + w.m);
    float* ws_l = reinterpret_cast<float*>(base + w.l);
    unsigned long long* ws_cnt = reinterpret_cast<unsigned long long*>(base + w.cnt);
    const float scale_log2 = a.scale * kLog2e;
    // contexts are cut to what the table holds and to the caller's promise
    const int cap = int(std::min<long>(long(a.max_blocks_per_seq) * a.S, a.max_context_len));
    const int streams = kFork ? a.n_groups : a.B;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kMQ && !kFork ? kDecodeThreads : kDecodeThreadsPub);
    cfg.dynamicSmemBytes = Lt::kAlloc;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return launch_result(cudaLaunchKernelEx(
        &cfg, kern, tm_k, tm_v, static_cast<T*>(a.out), static_cast<const T*>(a.q),
        a.block_tables, a.max_blocks_per_seq, a.context_lens, streams, a.H, a.Hk, a.S, a.NB, GH,
        nq, scale_log2, P, cap, ws_o, ws_m, ws_l, ws_cnt, next_launch_tag(), a.k_scale, a.v_scale,
        fk,
        StepRows{a.row_k, a.row_v, a.row_ks, a.row_vs, a.row_slots,
                 const_cast<void*>(a.key_cache), const_cast<void*>(a.value_cache)},
        a.dev_err));
}

template <bool kF8, bool kMQ, bool kFork>
pd_status launch_decode_dt(const DecodeArgs& a) {
    if (a.dt == PD_BF16)
        return a.D == 128 ? launch_decode_t<__nv_bfloat16, 128, kF8, kMQ, kFork>(a)
                          : launch_decode_t<__nv_bfloat16, 64, kF8, kMQ, kFork>(a);
    return a.D == 128 ? launch_decode_t<__half, 128, kF8, kMQ, kFork>(a)
                      : launch_decode_t<__half, 64, kF8, kMQ, kFork>(a);
}

}  // namespace

int decode_partition_tokens(int max_context_len) {
    (void)max_context_len;
    return kSegTokens;
}

// Most pieces one stream can be cut into: a CTA's range holds at least
// kMinStagesPerCta stages, so a stream of L stages meets at most
// ceil(L / kMinStagesPerCta) + 1 ranges.
int decode_num_partitions(int max_context_len) {
    if (max_context_len <= 0) return 1;
    return (max_context_len + kSegTokens - 1) / kSegTokens + 1;
}

size_t decode_workspace_bytes(int B, int H, int D, int max_context_len) {
    return ws_layout(B, H, D, decode_num_partitions(max_context_len)).total;
}

size_t decode_shared_workspace_bytes(int n_groups, int max_group, int H, int Hk, int D) {
    return fork_ws_layout(n_groups, max_group, H, Hk, D, nullptr, nullptr).total;
}

pd_status launch_decode(const DecodeArgs& a) {
    if (a.n_groups > 0)
        return a.fp8 || a.nq > 1 ? PD_ERR_UNSUPPORTED : launch_decode_dt<false, true, true>(a);
    if (a.nq > 1) return a.fp8 ? PD_ERR_UNSUPPORTED : launch_decode_dt<false, true, false>(a);
    return a.fp8 ? launch_decode_dt<true, false, false>(a) : launch_decode_dt<false, false, false>(a);
}

}  // namespace pd
