/*
 * ep_oracle.c -- plain, slow, single-threaded CPU oracle for the MoE
 * expert-parallel hot path: route-top-K -> layout -> dispatch -> combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library; every function is the plain definition of its step,
 * written for a reader to check against the source pages by eye:
 *
 *   [P1] "Anatomy of a High-Performance EP Kernel" (euno.news Korean
 *        rendering), sections "What we have to do", "High throughput: ask
 *        first, then send", "Dispatch".
 *   [P2] "21K output tokens/s DeepSeek inference on AMD Instinct MI300X with
 *        Expert Parallelism" (Moreh technical report), sections
 *        "Parallelization method", "Load balancing across GPUs".
 *   [P3] "Expert Parallelism" (SGLang documentation, wiki copy), sections
 *        "Backends for MoE computation" (deep_gemm row: contiguous layout for
 *        prefill, masked layout for decode, FP8 block-wise quantisation) and
 *        "Framework overview" (TopK -> dispatch -> runner -> combine).
 *   [P4] Chinese rendering of [P1] (66bd.net), router-logits table t0..t3.
 *
 * Floating point: routing weights are computed in double and rounded once
 * to float; the FP8 scale and the scaled value use IEEE float division (the
 * precision the quantised code is decided in, on both sides); combine
 * accumulates in float with one fused multiply-add per pick in pick order
 * (the accumulation precision and order the workload definition fixes).
 * Build with -ffp-contract=off so the compiler adds no contractions.
 *
 * Conventions shared with the library's public contract (not its code):
 *   - bf16 values are passed as their 16-bit patterns (uint16_t);
 *   - FP8 codes are OCP E4M3FN bytes;
 *   - an expert id outside [0, E) in topk_idx is "no pick": it is not
 *     counted, gets pos = -1, is not dispatched and contributes nothing.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 <-> float                                                            */
/* ------------------------------------------------------------------------ */

/* bf16 is the top half of an IEEE binary32: widening is exact. */
static float bf16_bits_to_float(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to even; NaN stays a quiet NaN. */
uint16_t oracle_float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* Step 1: top-K expert selection and gate weights                           */
/* ------------------------------------------------------------------------ */

typedef struct {
    float v;
    int32_t e;
} logit_t;

/* Order: logit descending; equal logits -> lower expert id first. */
static int logit_order(const void* pa, const void* pb) {
    const logit_t* a = (const logit_t*)pa;
    const logit_t* b = (const logit_t*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->e < b->e) ? -1 : (a->e > b->e ? 1 : 0);
}

/*
 * [P1] "What we have to do" / [P4] router-logits table: the router gives
 * each token a length-E logit vector, shape (B_i, E); the top-K indices form
 * the (B_i, K) assignment (t0 -> [3, 13]).  Picks are listed in descending
 * logit order; ties go to the lower expert id.
 * Gate weights (the pages name a gating network but print no formula; the
 * workload fixes softmax-renormalised top-K weights): softmax over the K
 * selected logits, w_k = exp(l_k - l_0) / sum_j exp(l_j - l_0), in double.
 * [P2] "Load balancing across GPUs": after experts are renumbered, the gate
 * must emit the new ids, so an optional expert_map[old] = new is applied to
 * the chosen ids without changing their order.  A map entry outside [0,E)
 * gives "no pick" (-1), as an invalid id does everywhere on this path (the
 * pages give no map format; the weights are those of the chosen logits).
 */
void oracle_route_topk(const float* logits, int64_t N, int32_t E, int32_t K,
                       const int32_t* expert_map, int32_t* topk_idx, float* topk_w) {
    logit_t* row = (logit_t*)malloc(sizeof(logit_t) * (size_t)E);
    double* ex = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t t = 0; t < N; ++t) {
        for (int32_t e = 0; e < E; ++e) {
            row[e].v = logits[t * E + e];
            row[e].e = e;
        }
        qsort(row, (size_t)E, sizeof(logit_t), logit_order);
        double top = (double)row[0].v;
        double sum = 0.0;
        for (int32_t k = 0; k < K; ++k) {
            ex[k] = exp((double)row[k].v - top);
            sum += ex[k];
        }
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = row[k].e;
            int32_t id = expert_map ? expert_map[e] : e;
            topk_idx[t * K + k] = (id >= 0 && id < E) ? id : -1;
            topk_w[t * K + k] = (float)(ex[k] / sum);
        }
    }
    free(ex);
    free(row);
}

/* ------------------------------------------------------------------------ */
/* Step 1b: balanced expert renumbering                                      */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t f;
    int32_t e;
} freq_t;

static int freq_order(const void* pa, const void* pb) {
    const freq_t* a = (const freq_t*)pa;
    const freq_t* b = (const freq_t*)pb;
    if (a->f > b->f) return -1;
    if (a->f < b->f) return 1;
    return (a->e < b->e) ? -1 : (a->e > b->e ? 1 : 0);
}

/*
 * [P2] "Load balancing across GPUs": measure each expert's activation
 * frequency, group the E experts into R sets of E/R with sums as even as
 * possible (a balanced number-partitioning variant), and renumber so each
 * set is contiguous.  The page gives no algorithm; this is the plain greedy:
 * frequency = column sums of the per-(rank, expert) count matrix; visit
 * experts by frequency descending (ties: lower id); put each in the set with
 * the smallest load among sets that still have room (ties: lower set id);
 * its new id is set * (E/R) + its arrival order in that set.
 */
void oracle_balance_map(const int32_t* counts, int32_t R, int32_t E, int32_t* expert_map) {
    int32_t per_set = E / R;
    freq_t* order = (freq_t*)malloc(sizeof(freq_t) * (size_t)E);
    int64_t* load = (int64_t*)calloc((size_t)R, sizeof(int64_t));
    int32_t* size = (int32_t*)calloc((size_t)R, sizeof(int32_t));
    for (int32_t e = 0; e < E; ++e) {
        int64_t f = 0;
        for (int32_t r = 0; r < R; ++r) f += counts[(int64_t)r * E + e];
        order[e].f = f;
        order[e].e = e;
    }
    qsort(order, (size_t)E, sizeof(freq_t), freq_order);
    for (int32_t i = 0; i < E; ++i) {
        int32_t best = -1;
        for (int32_t s = 0; s < R; ++s) {
            if (size[s] >= per_set) continue;
            if (best < 0 || load[s] < load[best]) best = s;
        }
        expert_map[order[i].e] = best * per_set + size[best];
        size[best] += 1;
        load[best] += order[i].f;
    }
    free(size);
    free(load);
    free(order);
}

/* ------------------------------------------------------------------------ */
/* Step 2: layout ("ask first, then send")                                   */
/* ------------------------------------------------------------------------ */

static int32_t rank_of(const int32_t* rank_offsets, int32_t R, int64_t t) {
    for (int32_t r = 0; r < R; ++r)
        if (t >= rank_offsets[r] && t < rank_offsets[r + 1]) return r;
    return -1;
}

/*
 * [P1] "High throughput: ask first, then send" and "Dispatch": before any
 * payload moves, every (rank, expert) pair's token count is known, and each
 * rank gathers the tokens of an expert into one dense buffer for the grouped
 * GEMM; each expert receives a different, possibly zero, number of tokens.
 *   counts[r][e]              picks of expert e made by tokens of rank r
 *   expert_offsets[e]         exclusive prefix over e of sum_r counts[r][e]
 *                             (expert_offsets[E] = number of valid picks)
 *   rank_expert_offsets[r][e] expert_offsets[e] + sum_{r'<r} counts[r'][e]
 *   pos[t][k]                 row of pick (t, k) in the expert-major buffer:
 *                             within an expert, picks keep (t, k) order, which
 *                             is source-rank order because tokens are packed
 *                             rank-major; -1 for an invalid expert id
 *   row_src[p]                token whose pick fills row p (-1 if unused)
 * [P3] deep_gemm row, masked layout: with cap > 0, masked_m[e] =
 * min(total_e, cap) valid rows, and overflow = picks beyond cap (dropped).
 */
void oracle_layout(const int32_t* topk_idx, const int32_t* rank_offsets, int32_t R,
                   int64_t N, int32_t E, int32_t K, int32_t cap,
                   int32_t* counts, int32_t* expert_offsets, int32_t* rank_expert_offsets,
                   int32_t* pos, int32_t* row_src, int32_t* masked_m, int32_t* overflow) {
    memset(counts, 0, sizeof(int32_t) * (size_t)R * (size_t)E);
    for (int64_t t = 0; t < N; ++t) {
        int32_t r = rank_of(rank_offsets, R, t);
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = topk_idx[t * K + k];
            if (e >= 0 && e < E && r >= 0) counts[(int64_t)r * E + e] += 1;
        }
    }
    expert_offsets[0] = 0;
    for (int32_t e = 0; e < E; ++e) {
        int32_t total = 0;
        for (int32_t r = 0; r < R; ++r) total += counts[(int64_t)r * E + e];
        expert_offsets[e + 1] = expert_offsets[e] + total;
    }
    for (int32_t e = 0; e < E; ++e) {
        int32_t run = expert_offsets[e];
        for (int32_t r = 0; r < R; ++r) {
            rank_expert_offsets[(int64_t)r * E + e] = run;
            run += counts[(int64_t)r * E + e];
        }
    }
    for (int64_t i = 0; i < N * K; ++i) {
        pos[i] = -1;
        row_src[i] = -1;
    }
    for (int32_t e = 0; e < E; ++e) {
        int32_t next = expert_offsets[e];
        for (int64_t t = 0; t < N; ++t) {
            for (int32_t k = 0; k < K; ++k) {
                if (topk_idx[t * K + k] == e) {
                    pos[t * K + k] = next;
                    row_src[next] = (int32_t)t;
                    next += 1;
                }
            }
        }
    }
    if (cap > 0) {
        int32_t dropped = 0;
        for (int32_t e = 0; e < E; ++e) {
            int32_t total = expert_offsets[e + 1] - expert_offsets[e];
            if (masked_m) masked_m[e] = total < cap ? total : cap;
            if (total > cap) dropped += total - cap;
        }
        if (overflow) *overflow = dropped;
    }
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3FN encoding (OCP 8-bit floating point specification)             */
/* ------------------------------------------------------------------------ */

/*
 * E4M3FN: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no
 * infinities; S.1111.111 is NaN, so the largest finite magnitude is
 * 1.75 * 2^8 = 448.  Subnormals (exponent field 0) are m/8 * 2^-6.
 * Round to nearest, ties to even; a finite value whose rounding exceeds 448
 * saturates to 448 ("satfinite"); the sign bit of a zero result is kept.
 */
uint8_t oracle_fp8_e4m3_encode(float v) {
    uint8_t sign = signbit(v) ? 0x80u : 0x00u;
    if (isnan(v)) return (uint8_t)(sign | 0x7Fu);
    double a = fabs((double)v);
    if (isinf(v)) return (uint8_t)(sign | 0x7Eu);
    int code;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: integer multiples of 2^-9 */
        double n = a * ldexp(1.0, 9); /* exact: scaling by a power of two */
        double m = nearbyint(n);      /* default rounding mode: ties to even */
        code = (int)m;                /* m == 8 is the smallest normal 0x08 */
    } else {
        int ex;
        frexp(a, &ex);                /* a = f * 2^ex, f in [0.5, 1) */
        int unbiased = ex - 1;        /* a in [2^unbiased, 2^(unbiased+1)) */
        double n = a * ldexp(1.0, 3 - unbiased); /* in [8, 16), exact */
        double m = nearbyint(n);
        if (m >= 16.0) {
            m = 8.0;
            unbiased += 1;
        }
        int biased = unbiased + 7;
        if (biased > 15) code = 0x7F + 1;             /* beyond the format */
        else code = (biased << 3) | ((int)m - 8);
    }
    if (code > 0x7E) code = 0x7E; /* satfinite: 0x7F is NaN, 448 is the max */
    return (uint8_t)(sign | (uint8_t)code);
}

/* Value of an E4M3FN code (NaN codes decode to NaN). */
double oracle_fp8_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1;
    int ex = (c >> 3) & 0xF;
    int m = c & 7;
    double mag;
    if (ex == 0xF && m == 7) return NAN;
    if (ex == 0) mag = ldexp((double)m, -9);
    else mag = ldexp(8.0 + (double)m, ex - 7 - 3);
    return s ? -mag : mag;
}

/*
 * [P3] deep_gemm row, "FP8 block-wise quantisation" (block 1 x 128, E4M3
 * and float scales fixed by the workload definition): for each token and each
 * 128-column block, amax = max |x|; scale = amax / 448 (float division;
 * amax == 0 gives scale 1); code = E4M3(x / scale) (float division, then the
 * encoding above).
 */
static void quantize_row_fp8(const uint16_t* xrow, int32_t H, uint8_t* codes, float* scales) {
    for (int32_t b = 0; b < H / 128; ++b) {
        float amax = 0.0f;
        for (int32_t j = 0; j < 128; ++j) {
            float a = fabsf(bf16_bits_to_float(xrow[b * 128 + j]));
            if (a > amax) amax = a;
        }
        float scale = (amax == 0.0f) ? 1.0f : amax / 448.0f;
        scales[b] = scale;
        for (int32_t j = 0; j < 128; ++j) {
            float v = bf16_bits_to_float(xrow[b * 128 + j]) / scale;
            codes[b * 128 + j] = oracle_fp8_e4m3_encode(v);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Step 3: dispatch                                                          */
/* ------------------------------------------------------------------------ */

/*
 * Destination row of pick (t, k), or -1 when it is not delivered.
 *   contiguous layout ([P1] "Dispatch"; [P3] deep_gemm "contiguous layout
 *   for prefill"): row pos[t][k] of an [N*K, H] expert-major buffer.
 *   masked layout ([P3] "masked layout for decode", low-latency mode):
 *   slot = pos[t][k] - expert_offsets[e]; row e*cap + slot of an [E, cap, H]
 *   buffer when slot < cap, otherwise the pick is dropped.
 */
static int64_t dest_row(int32_t p, int32_t e, const int32_t* expert_offsets,
                        int32_t E, int layout, int32_t cap) {
    if (p < 0 || e < 0 || e >= E) return -1;
    if (layout == 0) return p;
    int32_t slot = p - expert_offsets[e];
    if (slot >= cap) return -1;
    return (int64_t)e * cap + slot;
}

/*
 * dtype 0: bf16 rows copied bit for bit.  dtype 1: FP8 E4M3 codes [rows, H]
 * plus float scales [rows, H/128]; the same codes go to every destination.
 */
void oracle_dispatch(const uint16_t* x, int64_t N, int32_t H, int32_t E, int32_t K,
                     const int32_t* topk_idx, const int32_t* pos, const int32_t* expert_offsets,
                     int layout, int32_t cap, int dtype, void* out, float* out_scales) {
    uint8_t* codes = NULL;
    float* scales = NULL;
    if (dtype == 1) {
        codes = (uint8_t*)malloc((size_t)H);
        scales = (float*)malloc(sizeof(float) * (size_t)(H / 128));
    }
    for (int64_t t = 0; t < N; ++t) {
        const uint16_t* xrow = x + t * H;
        if (dtype == 1) quantize_row_fp8(xrow, H, codes, scales);
        for (int32_t k = 0; k < K; ++k) {
            int64_t row = dest_row(pos[t * K + k], topk_idx[t * K + k], expert_offsets, E, layout, cap);
            if (row < 0) continue;
            if (dtype == 0) {
                memcpy((uint16_t*)out + row * H, xrow, sizeof(uint16_t) * (size_t)H);
            } else {
                memcpy((uint8_t*)out + row * H, codes, (size_t)H);
                memcpy(out_scales + row * (H / 128), scales, sizeof(float) * (size_t)(H / 128));
            }
        }
    }
    free(scales);
    free(codes);
}

/* ------------------------------------------------------------------------ */
/* Step 4: combine                                                           */
/* ------------------------------------------------------------------------ */

/*
 * [P1] "run the expert GEMM there, then bring the results home" and the
 * dispatch/experts/combine figure; [P3] framework overview, combine ->
 * final_hidden_states: out[t] = sum_k w[t][k] * y[row(t, k)], accumulated in
 * float with one fused multiply-add per pick in pick order k = 0..K-1, then
 * rounded to bf16 (nearest, ties to even).  Undelivered picks add nothing.
 */
void oracle_combine(const uint16_t* y, int64_t N, int32_t H, int32_t E, int32_t K,
                    const int32_t* topk_idx, const float* topk_w, const int32_t* pos,
                    const int32_t* expert_offsets, int layout, int32_t cap, uint16_t* out) {
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)K);
    for (int64_t t = 0; t < N; ++t) {
        for (int32_t k = 0; k < K; ++k)
            rows[k] = dest_row(pos[t * K + k], topk_idx[t * K + k], expert_offsets, E, layout, cap);
        for (int32_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int32_t k = 0; k < K; ++k) {
                if (rows[k] < 0) continue;
                acc = fmaf(topk_w[t * K + k], bf16_bits_to_float(y[rows[k] * H + h]), acc);
            }
            out[t * H + h] = oracle_float_to_bf16(acc);
        }
    }
    free(rows);
}

/* ------------------------------------------------------------------------ */
/* Array forms of the scalar conversions (for the tests' exhaustive sweeps)  */
/* ------------------------------------------------------------------------ */

void oracle_fp8_e4m3_encode_n(const float* v, int64_t n, uint8_t* codes) {
    for (int64_t i = 0; i < n; ++i) codes[i] = oracle_fp8_e4m3_encode(v[i]);
}

void oracle_float_to_bf16_n(const float* v, int64_t n, uint16_t* bits) {
    for (int64_t i = 0; i < n; ++i) bits[i] = oracle_float_to_bf16(v[i]);
}
