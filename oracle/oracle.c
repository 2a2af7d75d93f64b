/*
 * oracle.c -- float64 CPU oracle for paged KV-cache attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library includes,
 * links or calls this file; only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load it.  It shares no code, header or
 * constant with the CUDA path.
 *
 * Everything here is the plain definition of each operation, written for a
 * reader to check by eye, with no blocking, fusion or reordering:
 *
 *   - Paging (page "LLM 推理服务引擎深度拆解", section 2.2 "分页思想"):
 *     K/V live in fixed-size physical blocks of S tokens; a per-sequence
 *     block table maps logical block t/S to a physical block, and token t
 *     sits at offset t%S inside it.  Cache layout per layer:
 *     [num_blocks][num_kv_heads][S][D], K and V in separate pools.
 *   - Store ("nanoPD" page, "模块结构与代码组织": paged KV store op):
 *     new token n goes to slot slot_mapping[n] = block*S + offset.
 *   - Copy-on-write block copy (tutorial page, section 2.3, the block
 *     manager's cow(): a shared block about to be written is duplicated).
 *   - Attention: out = softmax(scale * q k^T) v over the tokens a query
 *     may see, GQA head h reading kv head h / (H/Hk) (essay page
 *     "LLM推理PD分离架构深度工程实践", section 6.2, 8 KV heads shared by 32
 *     Q heads).  Decode sees tokens [0, ctx); chunked prefill query j of a
 *     chunk appended after P cached tokens sees [0, P+j] (tutorial page,
 *     section 5.2 "Chunked Prefill").
 *
 * Arithmetic is IEEE float64 from exactly up-converted fp16/bf16 inputs.
 * Build with -ffp-contract=off so x86 and Arm hosts give identical bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F16 = 0, ORC_BF16 = 1 };

/* ---- 16-bit float decoding, from the formats' definitions ------------ */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/2^10) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
static double bf16_to_double(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133); /* f * 2^-126 * 2^-7 */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 134); /* (1 + f/2^7) * 2^(e-127) */
    }
    return sign ? -v : v;
}

double orc_to_double(uint16_t bits, int dtype) {
    return dtype == ORC_BF16 ? bf16_to_double(bits) : f16_to_double(bits);
}

void orc_to_double_array(const uint16_t* src, double* dst, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) dst[i] = orc_to_double(src[i], dtype);
}

/* ---- paging ----------------------------------------------------------- */

/* Physical slot of logical token t of a sequence: block_table[t/S]*S + t%S. */
int64_t orc_slot_of(const int32_t* block_table_row, int64_t t, int S) {
    return (int64_t)block_table_row[t / S] * S + (t % S);
}

/* Address of element 0 of token `offset` of kv head `h` in physical block `blk`. */
static int64_t cache_index(int64_t blk, int h, int64_t offset, int Hk, int S, int D) {
    return ((blk * Hk + h) * S + offset) * D;
}

/* ---- store: write new K/V tokens into their slots ---------------------- */
/* Returns the number of tokens skipped because their slot was out of range
 * (a negative slot is padding and is skipped silently). */
int orc_reshape_and_cache(const uint16_t* key, const uint16_t* value,
                          uint16_t* key_cache, uint16_t* value_cache,
                          const int64_t* slot_mapping, int T, int Hk, int D,
                          int S, int NB, int64_t key_stride_tok,
                          int64_t value_stride_tok) {
    int bad = 0;
    for (int n = 0; n < T; ++n) {
        int64_t slot = slot_mapping[n];
        if (slot < 0) continue;
        if (slot >= (int64_t)NB * S) { ++bad; continue; }
        int64_t blk = slot / S, off = slot % S;
        for (int h = 0; h < Hk; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t dst = cache_index(blk, h, off, Hk, S, D) + d;
                key_cache[dst] = key[n * key_stride_tok + (int64_t)h * D + d];
                value_cache[dst] = value[n * value_stride_tok + (int64_t)h * D + d];
            }
        }
    }
    return bad;
}

/* ---- copy-on-write block copy ----------------------------------------- */
/* For each (src, dst) pair and each layer, the whole block (all kv heads,
 * all S offsets) of K and of V is copied.  Returns the number of pairs
 * skipped because an id was out of range. */
int orc_copy_blocks(uint16_t* const* key_caches, uint16_t* const* value_caches,
                    int L, const int64_t* block_mapping, int npairs, int Hk,
                    int D, int S, int NB) {
    int bad = 0;
    int64_t block_elems = (int64_t)Hk * S * D;
    for (int p = 0; p < npairs; ++p) {
        int64_t src = block_mapping[2 * p], dst = block_mapping[2 * p + 1];
        if (src < 0 || src >= NB || dst < 0 || dst >= NB) { ++bad; continue; }
        for (int l = 0; l < L; ++l) {
            for (int64_t e = 0; e < block_elems; ++e) {
                key_caches[l][dst * block_elems + e] = key_caches[l][src * block_elems + e];
                value_caches[l][dst * block_elems + e] = value_caches[l][src * block_elems + e];
            }
        }
    }
    return bad;
}

/* ---- KV pack / unpack ----------------------------------------------------
 * nanoPD page, "异步KV传输"; essay page "LLM推理PD分离架构深度工程实践",
 * section 3.1 (layer-by-layer KV transfer).  Staging layout, layer-major:
 *   staging[l][kv][i][Hk][S][D] = pool_{l,kv}[block_ids[i]]   (kv 0 = K, 1 = V)
 * pack copies pool -> staging, unpack staging -> pool.  Ids outside [0, NB)
 * are skipped; the count of skipped ids is returned. */
int orc_kv_pack(int unpack, uint16_t* staging, uint16_t* const* key_caches,
                uint16_t* const* value_caches, int L, const int32_t* block_ids, int nblk,
                int Hk, int D, int S, int NB) {
    int bad = 0;
    int64_t slab = (int64_t)Hk * S * D;
    for (int i = 0; i < nblk; ++i) {
        int32_t b = block_ids[i];
        if (b < 0 || b >= NB) { ++bad; continue; }
        for (int l = 0; l < L; ++l) {
            for (int kv = 0; kv < 2; ++kv) {
                uint16_t* pool = kv == 0 ? key_caches[l] : value_caches[l];
                uint16_t* st = staging + (((int64_t)l * 2 + kv) * nblk + i) * slab;
                for (int64_t e = 0; e < slab; ++e) {
                    if (unpack) pool[(int64_t)b * slab + e] = st[e];
                    else st[e] = pool[(int64_t)b * slab + e];
                }
            }
        }
    }
    return bad;
}

/* ---- attention of one query row over keys [0, n_keys) ------------------ */
/* out[d] = sum_t softmax_t(scale * q.k_t) * v_t[d], in float64, two passes
 * (max, then exponentials) for a well-defined result.  n_keys <= 0 gives
 * zeros.  Returns 0, or -1 if the block table names a block outside the pool
 * (the row is then filled with NaN). */
static int attend_row(double* out, const uint16_t* qrow, int64_t n_keys,
                      const int32_t* bt_row, int kvh, const uint16_t* kc,
                      const uint16_t* vc, int Hk, int D, int S, int NB,
                      double scale, int dtype) {
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n_keys <= 0) return 0;
    double* q = (double*)malloc(sizeof(double) * D);
    double* s = (double*)malloc(sizeof(double) * n_keys);
    for (int d = 0; d < D; ++d) q[d] = orc_to_double(qrow[d], dtype);
    int err = 0;
    for (int64_t t = 0; t < n_keys; ++t) {
        int64_t blk = bt_row[t / S];
        if (blk < 0 || blk >= NB) { err = -1; break; }
        const uint16_t* k = kc + cache_index(blk, kvh, t % S, Hk, S, D);
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * orc_to_double(k[d], dtype);
        s[t] = scale * dot;
    }
    if (err) {
        for (int d = 0; d < D; ++d) out[d] = NAN;
        free(q); free(s);
        return err;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < n_keys; ++t) if (s[t] > m) m = s[t];
    double l = 0.0;
    for (int64_t t = 0; t < n_keys; ++t) {
        double w = exp(s[t] - m);
        l += w;
        const uint16_t* v = vc + cache_index(bt_row[t / S], kvh, t % S, Hk, S, D);
        for (int d = 0; d < D; ++d) out[d] += w * orc_to_double(v[d], dtype);
    }
    for (int d = 0; d < D; ++d) out[d] /= l;
    free(q); free(s);
    return 0;
}

/* ---- decode: one query token per sequence ------------------------------ */
/* Rows r in [row_begin, row_end) are (sequence i, q head h) = (r / H, r % H);
 * out is [B*H][D].  Sequence i sees tokens [0, context_lens[i]).  Returns the
 * number of rows whose block table named a block outside the pool. */
int orc_decode(double* out, const uint16_t* q, const uint16_t* key_cache,
               const uint16_t* value_cache, const int32_t* block_tables,
               int max_blocks_per_seq, const int32_t* context_lens, int B,
               int H, int Hk, int D, int S, int NB, double scale, int dtype,
               int64_t row_begin, int64_t row_end) {
    int G = H / Hk, bad = 0;
    (void)B;
    for (int64_t r = row_begin; r < row_end; ++r) {
        int64_t i = r / H;
        int h = (int)(r % H);
        const int32_t* bt_row = block_tables + i * (int64_t)max_blocks_per_seq;
        bad += attend_row(out + r * D, q + r * D, context_lens[i], bt_row,
                          h / G, key_cache, value_cache, Hk, D, S, NB, scale,
                          dtype) != 0;
    }
    return bad;
}

/* ---- FP8 (E4M3) KV cache ------------------------------------------------
 * Essay page "LLM推理PD分离架构深度工程实践", section 6.2 and tutorial page
 * "LLM 推理服务引擎深度拆解", section 8.1: the KV cache stored in FP8 E4M3
 * (one byte per value) instead of BF16 halves its memory and bandwidth.
 * E4M3: 1 sign, 4 exponent (bias 7) and 3 fraction bits; exponent field 0 is
 * subnormal (f * 2^-9); S.1111.111 is NaN; no infinities; largest 448.
 * Each (layer, kv head) has a scale for K and one for V: a stored code c
 * stands for e4m3(c) * scale.  Storing rounds y = x * (1 / scale), both
 * products formed in float32, to the nearest code (ties to the even code),
 * values beyond 448 in magnitude saturate to 448, NaN stays NaN. */
double orc_e4m3_to_double(uint8_t c) {
    int sign = c >> 7, e = (c >> 3) & 15, f = c & 7;
    if (e == 15 && f == 7) return NAN;
    double v = e == 0 ? ldexp((double)f, -9) : ldexp((double)(8 + f), e - 10);
    return sign ? -v : v;
}

uint8_t orc_e4m3_encode(float y) {
    if (isnan(y)) return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0;
    double a = fabs((double)y);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    /* nearest of the non-negative finite codes 0x00 .. 0x7E (values rise
     * with the code); ties go to the even code */
    uint8_t best = 0;
    double best_d = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(orc_e4m3_to_double((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = (uint8_t)c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* Store new tokens into FP8 pools: code = encode(x * (1 / scale[h])). */
int orc_reshape_and_cache_fp8(const uint16_t* key, const uint16_t* value, int dtype,
                              uint8_t* key_cache, uint8_t* value_cache,
                              const int64_t* slot_mapping, int T, int Hk, int D, int S,
                              int NB, const float* k_scale, const float* v_scale) {
    int bad = 0;
    for (int n = 0; n < T; ++n) {
        int64_t slot = slot_mapping[n];
        if (slot < 0) continue;
        if (slot >= (int64_t)NB * S) { ++bad; continue; }
        int64_t blk = slot / S, off = slot % S;
        for (int h = 0; h < Hk; ++h) {
            float kinv = 1.0f / k_scale[h], vinv = 1.0f / v_scale[h];
            for (int d = 0; d < D; ++d) {
                int64_t src = ((int64_t)n * Hk + h) * D + d;
                int64_t dst = ((blk * Hk + h) * S + off) * D + d;
                float kx = (float)orc_to_double(key[src], dtype);
                float vx = (float)orc_to_double(value[src], dtype);
                key_cache[dst] = orc_e4m3_encode(kx * kinv);
                value_cache[dst] = orc_e4m3_encode(vx * vinv);
            }
        }
    }
    return bad;
}

/* Decode attention over FP8 pools: k = e4m3(code) * k_scale[kv head], the
 * same for v; q and the result as for orc_decode. */
int orc_decode_fp8(double* out, const uint16_t* q, int qdtype, const uint8_t* key_cache,
                   const uint8_t* value_cache, const float* k_scale, const float* v_scale,
                   const int32_t* block_tables, int max_blocks_per_seq,
                   const int32_t* context_lens, int H, int Hk, int D, int S, int NB,
                   double scale, int64_t row_begin, int64_t row_end) {
    int G = H / Hk, bad = 0;
    double* qd = (double*)malloc(sizeof(double) * D);
    for (int64_t r = row_begin; r < row_end; ++r) {
        int64_t i = r / H;
        int h = (int)(r % H), kvh = h / G;
        const int32_t* bt = block_tables + i * (int64_t)max_blocks_per_seq;
        int64_t n = context_lens[i];
        double* o = out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (n <= 0) continue;
        for (int d = 0; d < D; ++d) qd[d] = orc_to_double(q[r * D + d], qdtype);
        double* sc = (double*)malloc(sizeof(double) * n);
        int err = 0;
        for (int64_t t = 0; t < n && !err; ++t) {
            int64_t blk = bt[t / S];
            if (blk < 0 || blk >= NB) { err = 1; break; }
            const uint8_t* k = key_cache + ((blk * Hk + kvh) * S + t % S) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += qd[d] * (orc_e4m3_to_double(k[d]) * k_scale[kvh]);
            sc[t] = scale * dot;
        }
        if (err) {
            for (int d = 0; d < D; ++d) o[d] = NAN;
            free(sc);
            ++bad;
            continue;
        }
        double m = -INFINITY, l = 0.0;
        for (int64_t t = 0; t < n; ++t) if (sc[t] > m) m = sc[t];
        for (int64_t t = 0; t < n; ++t) {
            double w = exp(sc[t] - m);
            l += w;
            const uint8_t* v = value_cache + ((bt[t / S] * (int64_t)Hk + kvh) * S + t % S) * D;
            for (int d = 0; d < D; ++d) o[d] += w * (orc_e4m3_to_double(v[d]) * v_scale[kvh]);
        }
        for (int d = 0; d < D; ++d) o[d] /= l;
        free(sc);
    }
    free(qd);
    return bad;
}

/* ---- decode written as split-context partitions plus a merge ----------- */
/* The same result as orc_decode, reached the way the split-context kernel
 * organises it: partition p covers tokens [p*part, min(ctx, (p+1)*part));
 * each partition keeps its own max m_p, sum l_p = sum exp(s - m_p) and
 * unnormalised o_p = sum exp(s - m_p) v; the merge takes M = max_p m_p,
 * L = sum_p l_p exp(m_p - M) and out = sum_p o_p exp(m_p - M) / L. */
int orc_decode_split(double* out, const uint16_t* q, const uint16_t* key_cache,
                     const uint16_t* value_cache, const int32_t* block_tables,
                     int max_blocks_per_seq, const int32_t* context_lens, int B,
                     int H, int Hk, int D, int S, int NB, double scale,
                     int dtype, int part, int64_t row_begin, int64_t row_end) {
    int G = H / Hk, bad = 0;
    (void)B;
    double* qd = (double*)malloc(sizeof(double) * D);
    double* o = (double*)malloc(sizeof(double) * D);
    double* acc = (double*)malloc(sizeof(double) * D);
    for (int64_t r = row_begin; r < row_end; ++r) {
        int64_t i = r / H;
        int h = (int)(r % H), kvh = h / G;
        int64_t ctx = context_lens[i];
        const int32_t* bt_row = block_tables + i * (int64_t)max_blocks_per_seq;
        double* dst = out + r * D;
        for (int d = 0; d < D; ++d) { dst[d] = 0.0; acc[d] = 0.0; }
        if (ctx <= 0) continue;
        for (int d = 0; d < D; ++d) qd[d] = orc_to_double(q[r * D + d], dtype);
        int64_t nparts = (ctx + part - 1) / part;
        double* mp = (double*)malloc(sizeof(double) * nparts);
        double* lp = (double*)malloc(sizeof(double) * nparts);
        double* op = (double*)malloc(sizeof(double) * nparts * D);
        int err = 0;
        for (int64_t p = 0; p < nparts && !err; ++p) {
            int64_t t0 = p * part, t1 = t0 + part < ctx ? t0 + part : ctx;
            double m = -INFINITY;
            for (int64_t t = t0; t < t1; ++t) {
                int64_t blk = bt_row[t / S];
                if (blk < 0 || blk >= NB) { err = 1; break; }
                const uint16_t* k = key_cache + cache_index(blk, kvh, t % S, Hk, S, D);
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += qd[d] * orc_to_double(k[d], dtype);
                if (scale * dot > m) m = scale * dot;
            }
            if (err) break;
            double l = 0.0;
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            for (int64_t t = t0; t < t1; ++t) {
                int64_t blk = bt_row[t / S];
                const uint16_t* k = key_cache + cache_index(blk, kvh, t % S, Hk, S, D);
                const uint16_t* v = value_cache + cache_index(blk, kvh, t % S, Hk, S, D);
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += qd[d] * orc_to_double(k[d], dtype);
                double w = exp(scale * dot - m);
                l += w;
                for (int d = 0; d < D; ++d) o[d] += w * orc_to_double(v[d], dtype);
            }
            mp[p] = m;
            lp[p] = l;
            for (int d = 0; d < D; ++d) op[p * D + d] = o[d];
        }
        if (err) {
            for (int d = 0; d < D; ++d) dst[d] = NAN;
            ++bad;
        } else {
            double M = -INFINITY, L = 0.0;
            for (int64_t p = 0; p < nparts; ++p) if (mp[p] > M) M = mp[p];
            for (int64_t p = 0; p < nparts; ++p) {
                double c = exp(mp[p] - M);
                L += lp[p] * c;
                for (int d = 0; d < D; ++d) acc[d] += op[p * D + d] * c;
            }
            for (int d = 0; d < D; ++d) dst[d] = acc[d] / L;
        }
        free(mp); free(lp); free(op);
    }
    free(qd); free(o); free(acc);
    return bad;
}

/* ---- chunked prefill ---------------------------------------------------- */
/* q is packed [sum_i C_i][H][D]; cu_q_lens[i]..cu_q_lens[i+1] are sequence
 * i's chunk tokens.  context_lens[i] = P_i + C_i counts the chunk itself
 * (its K/V already stored).  Chunk token j of sequence i sits at position
 * P_i + j and sees keys [0, P_i + j].  `rows` lists flattened
 * (packed token, head) = tok*H + h indices to evaluate (a sample or all);
 * out is [nrows][D].  Returns the number of rows with a bad block id or a
 * token outside every chunk. */
int orc_prefill(double* out, const uint16_t* q, const int32_t* cu_q_lens,
                const uint16_t* key_cache, const uint16_t* value_cache,
                const int32_t* block_tables, int max_blocks_per_seq,
                const int32_t* context_lens, int B, int H, int Hk, int D,
                int S, int NB, double scale, int dtype, const int64_t* rows,
                int64_t nrows) {
    int G = H / Hk, bad = 0;
    for (int64_t n = 0; n < nrows; ++n) {
        int64_t tok = rows[n] / H;
        int h = (int)(rows[n] % H);
        int i = -1;
        for (int s = 0; s < B; ++s)
            if (tok >= cu_q_lens[s] && tok < cu_q_lens[s + 1]) { i = s; break; }
        if (i < 0) {
            for (int d = 0; d < D; ++d) out[n * D + d] = NAN;
            ++bad;
            continue;
        }
        int64_t C = cu_q_lens[i + 1] - cu_q_lens[i];
        int64_t P = context_lens[i] - C;
        int64_t j = tok - cu_q_lens[i];
        const int32_t* bt_row = block_tables + (int64_t)i * max_blocks_per_seq;
        bad += attend_row(out + n * D, q + rows[n] * D, P + j + 1, bt_row,
                          h / G, key_cache, value_cache, Hk, D, S, NB, scale,
                          dtype) != 0;
    }
    return bad;
}
