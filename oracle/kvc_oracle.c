/*
 * kvc_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of the autoregressive KV-cache append and
 * causal attention step, written from the page "Autoregressive KV-cache append
 * and causal attention" (biotorch, problems/kv_cache_attention_step), section
 * "Required behavior". Only tests/, the package smoke check and bench.py's CPU
 * baseline may load this library. It shares no code, header or constant with
 * the CUDA implementation.
 *
 * What each function follows:
 *   kvo_widen          exact widening of fp32 / bf16 / fp16 storage to double
 *                      (IEEE 754 binary16 and the bfloat16 truncated-binary32
 *                      formats, from their definitions).
 *   kvo_append_count   "append_mask[B,Q] is bool and each row must be a prefix
 *                      of True values followed by False. Its count n must
 *                      satisfy length+n <= M" (Required behavior, bullet 3).
 *                      A row outside that contract (non-prefix mask, length
 *                      outside [0, M], length+n > M) is treated as n = 0 and
 *                      flagged: this follows "Fixed-capacity KV cache"
 *                      (aiengineeringfromscratch), Task: when append raises,
 *                      the cache does not change.
 *   kvo_step           the whole step: copy caches byte-wise, write new rows at
 *                      slots length+t for the True slots (bullet 3), return the
 *                      updated lengths (bullet 4), then for every query row the
 *                      scaled scores, stable softmax over the allowed slots
 *                      j <= old_length+t and j < new_length, attention and
 *                      context = attention . updated_values (bullets 4-5);
 *                      invalid rows (mask False) are all zero (bullet 4).
 *   kvo_rows           the same attention/context for a list of (b,h,t) rows
 *                      only, reading the updated cache through its definition
 *                      (new row if length <= j < length+n, else old cache row).
 *   kvo_attend_cache   the read-only re-attention of "ClikaRT::ops::
 *                      attention_over_cache" (docs.clika.io): packed queries
 *                      attend a cache another call already appended, through
 *                      a per-sequence cache row (slot_ids) and total cached
 *                      length (cu_seqlens_k); the cache is never written.
 *   kvo_step_backward  the gradients of kvo_step's four outputs with respect
 *                      to query, new_key, new_value and both caches (the
 *                      contract's test suite grades gradients: "Starter
 *                      code"), by the chain rule through the same definition:
 *                      the returned caches pass their gradient to the input
 *                      cache slot or the new row each entry came from; the
 *                      attention row a = softmax(s) over the allowed slots
 *                      takes ds_j = a_j (g_j - sum_k a_k g_k) with g the
 *                      gradient reaching a (from attention and, through
 *                      context = a . V', from context); s = scale q.K' then
 *                      gives dq and dK', context gives dV' = a dcontext.
 *
 * Precision: every element is widened exactly to double, dot products, max,
 * exp, sums and the weighted value sum are taken in double, in slot order.
 * Nothing is blocked, fused or reordered.
 *
 * Parity pins live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { KVO_F32 = 0, KVO_BF16 = 1, KVO_F16 = 2 };

/* Per-batch-row flags written by kvo_step / kvo_append_count. */
enum {
    KVO_FLAG_OVERFLOW = 1, /* length < 0, length > M, or length + n > M */
    KVO_FLAG_MASK = 2      /* append_mask row is not a True-prefix */
};

static int64_t elem_size(int dtype) { return dtype == KVO_F32 ? 4 : 2; }

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

double kvo_widen(int dtype, const void *base, int64_t i) {
    if (dtype == KVO_F32) {
        float f;
        memcpy(&f, (const char *)base + 4 * i, 4);
        return (double)f;
    }
    uint16_t u;
    memcpy(&u, (const char *)base + 2 * i, 2);
    return dtype == KVO_BF16 ? bf16_bits_to_double(u) : half_bits_to_double(u);
}

/* Decode n elements into out (used by the pins on the widening itself). */
void kvo_widen_n(int dtype, const void *base, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = kvo_widen(dtype, base, i);
}

int64_t kvo_append_count(const uint8_t *mask_row, int64_t Q, int64_t length, int64_t M,
                         int32_t *flags) {
    int64_t n = 0;
    while (n < Q && mask_row[n]) ++n;
    int32_t f = 0;
    for (int64_t t = n; t < Q; ++t)
        if (mask_row[t]) f |= KVO_FLAG_MASK;
    if (length < 0 || length > M || length + n > M) f |= KVO_FLAG_OVERFLOW;
    if (flags) *flags = f;
    return f ? 0 : n;
}

int kvo_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Element (b, head, row, d) of a dense [B, H, R, W] tensor. */
static int64_t at4(int64_t H, int64_t R, int64_t W, int64_t b, int64_t h, int64_t r, int64_t d) {
    return ((b * H + h) * R + r) * W + d;
}

/*
 * Attention for query row (b, h, t).
 * valid: t < n (the row's append slot is True); an invalid row is all zero.
 * The cache row at slot j is new_key[b, kv, j - length] when
 * length <= j < length + n_src, else key_cache[b, kv, j] (same for values).
 * kvo_step passes the already-updated cache with n_src = 0; kvo_rows passes
 * the input cache with n_src = n, which is the same row by definition.
 * Allowed slots: j <= length + t, which is < length + n = new_length.
 */
static void attend_row(int dtype, int64_t Hq, int64_t Hk, int64_t Q, int64_t D, int64_t Dv,
                       int64_t M, const void *query, const void *new_key, const void *new_value,
                       const void *key_cache, const void *value_cache, int64_t length,
                       int64_t n_src, int valid, double scale, int64_t b, int64_t h, int64_t t,
                       double *att_row /* M */, double *ctx_row /* Dv */, double *scratch /* M */) {
    for (int64_t j = 0; j < M; ++j) att_row[j] = 0.0;
    for (int64_t e = 0; e < Dv; ++e) ctx_row[e] = 0.0;
    if (!valid) return; /* invalid query row: zero attention and context */

    const int64_t group = Hq / Hk;
    const int64_t kv = h / group; /* query head h uses KV head floor(h/(Hq/Hk)) */
    const int64_t last = length + t; /* allowed: j <= old_length + t (< new_length) */
    const int64_t n = n_src;

    double m = -INFINITY;
    for (int64_t j = 0; j <= last; ++j) {
        double s = 0.0;
        for (int64_t d = 0; d < D; ++d) {
            double qd = kvo_widen(dtype, query, at4(Hq, Q, D, b, h, t, d));
            double kd = (j >= length && j < length + n)
                            ? kvo_widen(dtype, new_key, at4(Hk, Q, D, b, kv, j - length, d))
                            : kvo_widen(dtype, key_cache, at4(Hk, M, D, b, kv, j, d));
            s += qd * kd;
        }
        s *= scale;
        scratch[j] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int64_t j = 0; j <= last; ++j) {
        scratch[j] = exp(scratch[j] - m);
        l += scratch[j];
    }
    for (int64_t j = 0; j <= last; ++j) att_row[j] = scratch[j] / l;
    for (int64_t j = 0; j <= last; ++j) {
        for (int64_t e = 0; e < Dv; ++e) {
            double ve = (j >= length && j < length + n)
                            ? kvo_widen(dtype, new_value, at4(Hk, Q, Dv, b, kv, j - length, e))
                            : kvo_widen(dtype, value_cache, at4(Hk, M, Dv, b, kv, j, e));
            ctx_row[e] += att_row[j] * ve;
        }
    }
}

/*
 * The whole step. Layouts are dense row-major:
 *   query [B,Hq,Q,D], new_key [B,Hk,Q,D], new_value [B,Hk,Q,Dv],
 *   key_cache [B,Hk,M,D], value_cache [B,Hk,M,Dv] in `dtype`;
 *   lengths [B] int64; append_mask [B,Q] bytes (0 = False);
 *   out caches in `dtype`, out_lengths [B] int64,
 *   out_attention [B,Hq,Q,M] and out_context [B,Hq,Q,Dv] in double,
 *   flags [B] (nullable). Returns the OR of all flags.
 * work: caller scratch of M doubles per OpenMP thread (kvo_threads()).
 */
int kvo_step(int dtype, int64_t B, int64_t Hq, int64_t Hk, int64_t Q, int64_t D, int64_t Dv,
             int64_t M, const void *query, const void *new_key, const void *new_value,
             const void *key_cache, const void *value_cache, const int64_t *lengths,
             const uint8_t *append_mask, double scale, void *out_key_cache,
             void *out_value_cache, int64_t *out_lengths, double *out_attention,
             double *out_context, int32_t *flags, double *work) {
    const int64_t es = elem_size(dtype);
    int any = 0;
    /* 1. copy both caches byte for byte (every unwritten entry preserved). */
    memcpy(out_key_cache, key_cache, (size_t)(B * Hk * M * D * es));
    memcpy(out_value_cache, value_cache, (size_t)(B * Hk * M * Dv * es));
    for (int64_t b = 0; b < B; ++b) {
        int32_t f = 0;
        const int64_t L = lengths[b];
        const int64_t n = kvo_append_count(append_mask + b * Q, Q, L, M, &f);
        if (flags) flags[b] = f;
        any |= f;
        /* 2. write new rows t < n at slot L + t, per KV head. */
        for (int64_t k = 0; k < Hk; ++k) {
            for (int64_t t = 0; t < n; ++t) {
                memcpy((char *)out_key_cache + at4(Hk, M, D, b, k, L + t, 0) * es,
                       (const char *)new_key + at4(Hk, Q, D, b, k, t, 0) * es, (size_t)(D * es));
                memcpy((char *)out_value_cache + at4(Hk, M, Dv, b, k, L + t, 0) * es,
                       (const char *)new_value + at4(Hk, Q, Dv, b, k, t, 0) * es,
                       (size_t)(Dv * es));
            }
        }
        out_lengths[b] = L + n;
    }
    /* 3. attention over the updated cache for every (b, h, t). */
    const int64_t rows = B * Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < rows; ++bh) {
        const int64_t b = bh / Hq, h = bh % Hq;
        const int64_t L = lengths[b];
        const int64_t n = kvo_append_count(append_mask + b * Q, Q, L, M, NULL);
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *scratch = work + (int64_t)tid * M;
        for (int64_t t = 0; t < Q; ++t) {
            /* Read the updated cache itself: the rows written above. */
            attend_row(dtype, Hq, Hk, Q, D, Dv, M, query, new_key, new_value, out_key_cache,
                       out_value_cache, L, 0, t < n, scale, b, h, t,
                       out_attention + at4(Hq, Q, M, b, h, t, 0),
                       out_context + at4(Hq, Q, Dv, b, h, t, 0), scratch);
        }
    }
    return any;
}

/*
 * Attention and context for selected rows only, without building the updated
 * cache: rows_bht holds n_rows triples (b, h, t). Outputs are
 * att [n_rows, M] and ctx [n_rows, Dv] in double. work: M doubles per thread.
 */
int kvo_rows(int dtype, int64_t B, int64_t Hq, int64_t Hk, int64_t Q, int64_t D, int64_t Dv,
             int64_t M, const void *query, const void *new_key, const void *new_value,
             const void *key_cache, const void *value_cache, const int64_t *lengths,
             const uint8_t *append_mask, double scale, const int64_t *rows_bht, int64_t n_rows,
             double *att, double *ctx, double *work) {
    (void)B;
    int any = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : any)
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t b = rows_bht[3 * i], h = rows_bht[3 * i + 1], t = rows_bht[3 * i + 2];
        int32_t f = 0;
        const int64_t L = lengths[b];
        const int64_t n = kvo_append_count(append_mask + b * Q, Q, L, M, &f);
        any |= f;
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        attend_row(dtype, Hq, Hk, Q, D, Dv, M, query, new_key, new_value, key_cache,
                   value_cache, L, n, t < n, scale, b, h, t, att + i * M, ctx + i * Dv,
                   work + (int64_t)tid * M);
    }
    return any;
}

/*
 * Read-only re-attention ("ClikaRT::ops::attention_over_cache", the
 * function's description). Sequence b owns the packed query rows
 * cu_q[b] .. cu_q[b+1]-1 of q [total_q, Hq, D] (S_b rows) and reads cache row
 * slot_b = slot_ids[b] (b when slot_ids is NULL) of cache_key
 * [num_slots, Hk, M, D] / cache_value [num_slots, Hk, M, Dv], which holds its
 * K_b = seqlens_k[b] cached positions (the total, q's own positions
 * included). "q's position derives from cu_seqlens_k": the S_b queries are
 * the sequence's last S_b positions, so query t sits at K_b - S_b + t and
 * attends the slots j <= K_b - S_b + t (the lower-right causal rule of the
 * append step). Query head h reads KV head floor(h / (Hq/Hk)).
 * out [total_q, Hq, Dv] in double. A sequence outside the contract
 * (S_b < 0, S_b > K_b, K_b > M, slot_b outside [0, num_slots)) gets zero
 * rows and flag KVO_FLAG_OVERFLOW in flags[b] (nullable). Returns the OR of
 * all flags.
 */
int kvo_attend_cache(int dtype, int64_t B, int64_t Hq, int64_t Hk, int64_t D, int64_t Dv,
                     int64_t M, int64_t num_slots, const void *q, const void *cache_key,
                     const void *cache_value, const int32_t *cu_q, const int32_t *seqlens_k,
                     const int32_t *slot_ids, double scale, double *out, int32_t *flags,
                     double *work) {
    const int64_t total_q = cu_q[B];
    for (int64_t i = 0; i < total_q * Hq * Dv; ++i) out[i] = 0.0;
    const int64_t group = Hq / Hk;
    int any = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : any)
    for (int64_t b = 0; b < B; ++b) {
        const int64_t S = (int64_t)cu_q[b + 1] - cu_q[b];
        const int64_t K = seqlens_k[b];
        const int64_t slot = slot_ids ? slot_ids[b] : b;
        const int bad = S < 0 || S > K || K > M || slot < 0 || slot >= num_slots;
        if (flags) flags[b] = bad ? KVO_FLAG_OVERFLOW : 0;
        if (bad) {
            any |= KVO_FLAG_OVERFLOW;
            continue;
        }
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *sc = work + (int64_t)tid * M;
        for (int64_t t = 0; t < S; ++t) {
            const int64_t row = cu_q[b] + t;
            const int64_t last = K - S + t; /* allowed: j <= K - S + t */
            for (int64_t h = 0; h < Hq; ++h) {
                const int64_t kv = h / group;
                double m = -INFINITY;
                for (int64_t j = 0; j <= last; ++j) {
                    double s = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        s += kvo_widen(dtype, q, (row * Hq + h) * D + d) *
                             kvo_widen(dtype, cache_key, ((slot * Hk + kv) * M + j) * D + d);
                    s *= scale;
                    sc[j] = s;
                    if (s > m) m = s;
                }
                double l = 0.0;
                for (int64_t j = 0; j <= last; ++j) {
                    sc[j] = exp(sc[j] - m);
                    l += sc[j];
                }
                double *o = out + (row * Hq + h) * Dv;
                for (int64_t j = 0; j <= last; ++j) {
                    const double a = sc[j] / l;
                    for (int64_t e = 0; e < Dv; ++e)
                        o[e] += a * kvo_widen(dtype, cache_value, ((slot * Hk + kv) * M + j) * Dv + e);
                }
            }
        }
    }
    return any;
}

/*
 * Gradients of the step. Inputs as kvo_step, plus the gradients reaching its
 * outputs, in `dtype`, each nullable (= zero):
 *   d_key_out [B,Hk,M,D], d_value_out [B,Hk,M,Dv] (the returned caches),
 *   d_attention [B,Hq,Q,M], d_context [B,Hq,Q,Dv].
 * Outputs in double: d_query [B,Hq,Q,D], d_new_key [B,Hk,Q,D],
 * d_new_value [B,Hk,Q,Dv], d_key_cache [B,Hk,M,D], d_value_cache [B,Hk,M,Dv];
 * flags [B] (nullable) as kvo_step. A row outside the contract appends
 * nothing (n = 0), as in the forward. work: 3 M doubles per OpenMP thread.
 *
 * The updated cache is K'[j] = new_key[j - L] for L <= j < L + n, else
 * key_cache[j] (same for V'). Invalid query rows (t >= n) and disallowed
 * slots are constant zeros of the forward: no gradient flows through them.
 */
int kvo_step_backward(int dtype, int64_t B, int64_t Hq, int64_t Hk, int64_t Q, int64_t D,
                      int64_t Dv, int64_t M, const void *query, const void *new_key,
                      const void *new_value, const void *key_cache, const void *value_cache,
                      const int64_t *lengths, const uint8_t *append_mask, double scale,
                      const void *d_key_out, const void *d_value_out, const void *d_attention,
                      const void *d_context, double *d_query, double *d_new_key,
                      double *d_new_value, double *d_key_cache, double *d_value_cache,
                      int32_t *flags, double *work) {
    const int64_t group = Hq / Hk;
    int any = 0;
    for (int64_t b = 0; b < B; ++b) {
        int32_t f = 0;
        kvo_append_count(append_mask + b * Q, Q, lengths[b], M, &f);
        if (flags) flags[b] = f;
        any |= f;
    }
    const int64_t units = B * Hk;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t unit = 0; unit < units; ++unit) {
        const int64_t b = unit / Hk, kv = unit % Hk;
        const int64_t L = lengths[b];
        const int64_t n = kvo_append_count(append_mask + b * Q, Q, L, M, NULL);
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *s = work + (int64_t)tid * 3 * M, *a = s + M, *g = a + M;

        /* 1. The returned caches: each entry's gradient goes to where it came from. */
        for (int64_t t = 0; t < Q; ++t) {
            for (int64_t d = 0; d < D; ++d) d_new_key[at4(Hk, Q, D, b, kv, t, d)] = 0.0;
            for (int64_t e = 0; e < Dv; ++e) d_new_value[at4(Hk, Q, Dv, b, kv, t, e)] = 0.0;
        }
        for (int64_t j = 0; j < M; ++j) {
            const int is_new = j >= L && j < L + n;
            for (int64_t d = 0; d < D; ++d) {
                const double gk =
                    d_key_out ? kvo_widen(dtype, d_key_out, at4(Hk, M, D, b, kv, j, d)) : 0.0;
                if (is_new) {
                    d_new_key[at4(Hk, Q, D, b, kv, j - L, d)] = gk;
                    d_key_cache[at4(Hk, M, D, b, kv, j, d)] = 0.0;
                } else {
                    d_key_cache[at4(Hk, M, D, b, kv, j, d)] = gk;
                }
            }
            for (int64_t e = 0; e < Dv; ++e) {
                const double gv =
                    d_value_out ? kvo_widen(dtype, d_value_out, at4(Hk, M, Dv, b, kv, j, e)) : 0.0;
                if (is_new) {
                    d_new_value[at4(Hk, Q, Dv, b, kv, j - L, e)] = gv;
                    d_value_cache[at4(Hk, M, Dv, b, kv, j, e)] = 0.0;
                } else {
                    d_value_cache[at4(Hk, M, Dv, b, kv, j, e)] = gv;
                }
            }
        }

        /* 2. The attention rows of the query heads that use this KV head. */
        for (int64_t h = kv * group; h < (kv + 1) * group; ++h) {
            for (int64_t t = 0; t < Q; ++t) {
                double *dq = d_query + at4(Hq, Q, D, b, h, t, 0);
                for (int64_t d = 0; d < D; ++d) dq[d] = 0.0;
                if (t >= n) continue; /* invalid row: zero outputs, no gradient */
                const int64_t last = L + t;
                /* forward again: scores, softmax over j <= last */
                double m = -INFINITY;
                for (int64_t j = 0; j <= last; ++j) {
                    double acc = 0.0;
                    for (int64_t d = 0; d < D; ++d) {
                        const double qd = kvo_widen(dtype, query, at4(Hq, Q, D, b, h, t, d));
                        const double kd =
                            (j >= L && j < L + n)
                                ? kvo_widen(dtype, new_key, at4(Hk, Q, D, b, kv, j - L, d))
                                : kvo_widen(dtype, key_cache, at4(Hk, M, D, b, kv, j, d));
                        acc += qd * kd;
                    }
                    s[j] = scale * acc;
                    if (s[j] > m) m = s[j];
                }
                double l = 0.0;
                for (int64_t j = 0; j <= last; ++j) {
                    a[j] = exp(s[j] - m);
                    l += a[j];
                }
                for (int64_t j = 0; j <= last; ++j) a[j] /= l;
                /* g_j: gradient reaching a_j, from attention and through context */
                double dot_ag = 0.0;
                for (int64_t j = 0; j <= last; ++j) {
                    double gj = d_attention
                                    ? kvo_widen(dtype, d_attention, at4(Hq, Q, M, b, h, t, j))
                                    : 0.0;
                    if (d_context) {
                        for (int64_t e = 0; e < Dv; ++e) {
                            const double ve =
                                (j >= L && j < L + n)
                                    ? kvo_widen(dtype, new_value, at4(Hk, Q, Dv, b, kv, j - L, e))
                                    : kvo_widen(dtype, value_cache, at4(Hk, M, Dv, b, kv, j, e));
                            gj += kvo_widen(dtype, d_context, at4(Hq, Q, Dv, b, h, t, e)) * ve;
                        }
                    }
                    g[j] = gj;
                    dot_ag += a[j] * gj;
                }
                /* softmax backward, then through s = scale q.K' and context = a.V' */
                for (int64_t j = 0; j <= last; ++j) {
                    const double ds = a[j] * (g[j] - dot_ag);
                    const int is_new = j >= L && j < L + n;
                    for (int64_t d = 0; d < D; ++d) {
                        const double qd = kvo_widen(dtype, query, at4(Hq, Q, D, b, h, t, d));
                        const double kd =
                            is_new ? kvo_widen(dtype, new_key, at4(Hk, Q, D, b, kv, j - L, d))
                                   : kvo_widen(dtype, key_cache, at4(Hk, M, D, b, kv, j, d));
                        dq[d] += scale * ds * kd;
                        if (is_new)
                            d_new_key[at4(Hk, Q, D, b, kv, j - L, d)] += scale * ds * qd;
                        else
                            d_key_cache[at4(Hk, M, D, b, kv, j, d)] += scale * ds * qd;
                    }
                    if (d_context) {
                        for (int64_t e = 0; e < Dv; ++e) {
                            const double dc =
                                kvo_widen(dtype, d_context, at4(Hq, Q, Dv, b, h, t, e));
                            if (is_new)
                                d_new_value[at4(Hk, Q, Dv, b, kv, j - L, e)] += a[j] * dc;
                            else
                                d_value_cache[at4(Hk, M, Dv, b, kv, j, e)] += a[j] * dc;
                        }
                    }
                }
            }
        }
    }
    return any;
}

