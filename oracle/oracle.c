/*
 * Reference oracle for attention over a paged KV cache -- TEST INFRASTRUCTURE.
 *
 * Plain, slow, fp64 CPU code that states what the hot path computes, one loop
 * per definition, with no blocking, fusion or reordering.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it;
 * the library under test never calls it and shares no code with it.
 *
 * Sources (page title, section):
 *   [TS]   vllm.v1.attention.backends.flashinfer_ts -- module docstring
 *          ("Layout", "Sliding window"), FlashInferTSImpl._kv_views,
 *          FlashInferTSImpl.forward, FlashInferTSMetadataBuilder.build,
 *          FlashInferTSMetadataBuilder._restrict_to_window, _kv_kernel_dtype.
 *   [DASH] vllm.v1.attention.ops.dash_attention -- flash_dash_attention
 *          (docstring, the varlen attention call, the combine at its end).
 *   [FA]   vllm.v1.attention.backends.fa_utils --
 *          FlashAttentionCuTeDSLCompileSpec (Split-KV, return_softmax_lse).
 *
 * Every entry point returns 0 on success and a negative code on an input the
 * definition does not cover (an out-of-range page, a length above capacity).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BF16 0
#define ORC_FP16 1
#define ORC_FP8_E4M3 2
#define ORC_FP32 3

/* ---------------------------------------------------------------------------
 * Element decoding.  Each storage type is decoded to fp64 exactly from its
 * bit-level definition.  An fp8 cache is uint8 storage read as e4m3 ("fn":
 * no infinities, one NaN code per sign) [TS _kv_kernel_dtype].
 * ------------------------------------------------------------------------- */
static double orc_bf16(uint16_t h) {
    /* bf16 is the top half of an IEEE binary32 */
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double orc_fp16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-14 / 2^10 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

static double orc_e4m3(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN; /* the only non-finite code of e4m3fn */
    else if (e == 0)
        v = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

static double orc_load(const void* base, size_t idx, int dt) {
    switch (dt) {
    case ORC_BF16: return orc_bf16(((const uint16_t*)base)[idx]);
    case ORC_FP16: return orc_fp16(((const uint16_t*)base)[idx]);
    case ORC_FP8_E4M3: return orc_e4m3(((const uint8_t*)base)[idx]);
    case ORC_FP32: return (double)((const float*)base)[idx];
    default: return NAN;
    }
}

/* Decode n elements (used by the tests to pin the decoders themselves). */
int orc_decode(const void* src, int dt, long n, double* dst) {
    if (dt < 0 || dt > 3) return -1;
    for (long i = 0; i < n; ++i) dst[i] = orc_load(src, (size_t)i, dt);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Sliding-window restriction [TS _restrict_to_window, module docstring
 * "Sliding window"].  The query block ends the sequence, so the symmetric
 * window around it is the suffix [L - w - sq + 1, L).  Its start is rounded
 * DOWN to a page boundary (floor division, then clamped at zero) and every
 * query token of the block shares that one start.
 * ------------------------------------------------------------------------- */
static long orc_floor_div(long a, long b) {
    long q = a / b;
    if ((a % b != 0) && ((a < 0) != (b < 0))) q -= 1;
    return q;
}

/* first visible page of a request: 0 when the layer has no window */
long orc_window_start_page(long L, long window, long sq, long P) {
    if (window <= 0) return 0;
    long span = window + sq - 1;
    long sp = orc_floor_div(L - span, P);
    return sp < 0 ? 0 : sp;
}

/*
 * The reference's table form of the restriction: a new table whose column c
 * is the old column start_page + c (clamped to the old table's last column)
 * and a length renumbered from the new first page.
 */
int orc_restrict_to_window(const int32_t* seq_lens, const int32_t* block_table,
                           int B, int width_in, int window, int sq, int P,
                           int width_out, int32_t* out_lens, int32_t* out_table) {
    if (window <= 0 || P <= 0 || width_in <= 0) return -1;
    for (int b = 0; b < B; ++b) {
        long sp = orc_window_start_page(seq_lens[b], window, sq, P);
        for (int c = 0; c < width_out; ++c) {
            long idx = sp + c;
            if (idx > width_in - 1) idx = width_in - 1;
            out_table[(long)b * width_out + c] = block_table[(long)b * width_in + idx];
        }
        out_lens[b] = (int32_t)(seq_lens[b] - sp * P);
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * softmax(s) V with its log-sum-exp, by definition:
 *   lse = m + ln sum_j exp(s_j - m),  m = max_j s_j
 *   o   = sum_j exp(s_j - lse) V_j
 * An empty key set gives o = 0 and lse = -inf.  The natural log is the one
 * the DASH page asks of its kernels (lse_base "ln").
 * ------------------------------------------------------------------------- */
static void orc_softmax_lse(const double* s, long n, double* m_out, double* lse_out) {
    if (n == 0) {
        *m_out = -INFINITY;
        *lse_out = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (long j = 0; j < n; ++j)
        if (s[j] > m) m = s[j];
    double sum = 0.0;
    for (long j = 0; j < n; ++j) sum += exp(s[j] - m);
    *m_out = m;
    *lse_out = m + log(sum);
}

/* ---------------------------------------------------------------------------
 * Paged decode [TS FlashInferTSImpl.forward / _kv_views, FlashInferTSMetadataBuilder.build].
 *
 *   q      [B, sq, Hq, D]            (dtype q_dt)
 *   cache  [num_pages, Hkv, P, 2*D]  K = cache[..., :D], V = cache[..., D:]
 *   block_table int32 [B, bt_stride]: token t of request b is in page
 *          block_table[b, t / P] at slot t % P
 *   seq_lens int32 [B]
 *   out    [B, sq, Hq, D] fp64, lse [B, sq, Hq] fp64 (natural log)
 *
 * Query head h reads kv head h / (Hq / Hkv) (contiguous GQA groups).
 * Logits are bmm1 * (q . k) with bmm1 = scale * q_scale * k_scale and the
 * output is scaled by bmm2 = v_scale [TS forward: bmm1_scale, bmm2_scale].
 *
 * mask 0 ("dense"): every query token of the block sees every visible key;
 *   with window > 0 the visible keys are those from the page-aligned start
 *   of the restriction above to L.
 * mask 1 ("causal"): query token i sits at position L - sq + i and sees keys
 *   j <= that position; with window > 0 also j >= position - (window - 1),
 *   the plan's window_left = window - 1 [TS FlashInferTSMetadataBuilder._get_plan].
 * ------------------------------------------------------------------------- */
int orc_paged_decode(const void* q, int q_dt, const void* cache, int kv_dt,
                     long num_pages, const int32_t* block_table, long bt_stride,
                     const int32_t* seq_lens, int B, int sq, int Hq, int Hkv, int D, int P,
                     double scale, double q_scale, double k_scale, double v_scale,
                     int window, int mask, double* out, double* lse, int nthreads) {
    if (B < 0 || sq <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || P <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int G = Hq / Hkv;
    const double bmm1 = scale * q_scale * k_scale;
    const double bmm2 = v_scale;
    int status = 0;
    if (nthreads < 1) nthreads = 1;

#pragma omp parallel for collapse(2) schedule(dynamic) num_threads(nthreads)
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hq; ++h) {
            const int hk = h / G;
            const long L = seq_lens[b];
            double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
            double* qd = (double*)malloc(sizeof(double) * (size_t)D);
            for (int i = 0; i < sq; ++i) {
                const long row = ((long)b * sq + i) * Hq + h;
                for (int d = 0; d < D; ++d) qd[d] = orc_load(q, (size_t)(row * D + d), q_dt);
                /* visible key range [lo, hi) */
                long lo, hi;
                if (mask == 0) {
                    lo = orc_window_start_page(L, window, sq, P) * P;
                    hi = L;
                } else {
                    long pos = L - sq + i;
                    hi = pos + 1;
                    lo = window > 0 ? pos - (window - 1) : 0;
                    if (lo < 0) lo = 0;
                }
                long n = hi > lo ? hi - lo : 0;
                for (long t = 0; t < n; ++t) {
                    long j = lo + t;
                    long page = block_table[(long)b * bt_stride + j / P];
                    if (page < 0 || page >= num_pages) {
#pragma omp atomic write
                        status = -2;
                        s[t] = 0.0;
                        continue;
                    }
                    size_t kbase = (size_t)(((page * Hkv + hk) * P + j % P) * 2L * D);
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += qd[d] * orc_load(cache, kbase + d, kv_dt);
                    s[t] = bmm1 * dot;
                }
                double m, l;
                orc_softmax_lse(s, n, &m, &l);
                lse[row] = l;
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (long t = 0; t < n; ++t) {
                        long j = lo + t;
                        long page = block_table[(long)b * bt_stride + j / P];
                        if (page < 0 || page >= num_pages) continue;
                        size_t vbase = (size_t)(((page * Hkv + hk) * P + j % P) * 2L * D + D);
                        acc += exp(s[t] - l) * orc_load(cache, vbase + d, kv_dt);
                    }
                    out[row * D + d] = n > 0 ? bmm2 * acc : 0.0;
                }
            }
            free(qd);
            free(s);
        }
    }
    return status;
}

/* ---------------------------------------------------------------------------
 * DASH segmented attention and its combine [DASH flash_dash_attention].
 *
 *   q     [n, Hq, D];  k, v [n * (topk*bs + local), Hkv, D] contiguous
 *   used  int32 [n * (topk+1)]: valid prefix length of each segment
 *   bias  [n, topk] (fp64 here; the prior of the local segment is 0)
 *
 * Query i owns rows i*(topk*bs+local) ...; its segment g < topk starts at
 * row offset g*bs with capacity bs, the local segment starts at topk*bs with
 * capacity local.  Each (query, segment, head) is one softmax attention over
 * the first used[i, g] rows with scale D^-0.5, giving (o_g, lse_g).  Then
 *   live_g   = used[i, g] > 0
 *   logit_g  = lse_g + prior_g          (prior = [bias, 0])
 *   w        = softmax over g of logit_g with dead groups at -inf;
 *              a query with no live group gets w = 0 (the NaN zeroed)
 *   out      = sum_g w_g * (live_g ? o_g : 0)
 * seg_out [n, topk+1, Hq, D] and seg_lse [n, topk+1, Hq] (nullable) receive
 * the per-segment results.
 * ------------------------------------------------------------------------- */
int orc_segmented_attention(const void* q, const void* k, const void* v, int dt,
                            const int32_t* used, const double* bias, int n, int Hq, int Hkv,
                            int D, int topk, int bs, int local, double* out,
                            double* seg_out, double* seg_lse, int nthreads) {
    if (n < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || topk < 0 || bs < 0 || local < 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int G = Hq / Hkv;
    const int groups = topk + 1;
    const long rows_per_query = (long)topk * bs + local;
    const double scale = 1.0 / sqrt((double)D);
    int status = 0;
    if (nthreads < 1) nthreads = 1;

    for (long i = 0; i < (long)n * groups; ++i) {
        int g = (int)(i % groups);
        int cap = g < topk ? bs : local;
        if (used[i] < 0 || used[i] > cap) return -3;
    }

#pragma omp parallel for collapse(2) schedule(dynamic) num_threads(nthreads)
    for (int i = 0; i < n; ++i) {
        for (int h = 0; h < Hq; ++h) {
            const int hk = h / G;
            const int cap_max = bs > local ? bs : local;
            double* s = (double*)malloc(sizeof(double) * (size_t)(cap_max > 0 ? cap_max : 1));
            double* o = (double*)malloc(sizeof(double) * (size_t)groups * D);
            double* l = (double*)malloc(sizeof(double) * (size_t)groups);
            double* qd = (double*)malloc(sizeof(double) * (size_t)D);
            for (int d = 0; d < D; ++d) qd[d] = orc_load(q, (size_t)(((long)i * Hq + h) * D + d), dt);

            for (int g = 0; g < groups; ++g) {
                long off = (long)i * rows_per_query + (g < topk ? (long)g * bs : (long)topk * bs);
                long u = used[(long)i * groups + g];
                for (long t = 0; t < u; ++t) {
                    size_t base = (size_t)(((off + t) * Hkv + hk) * D);
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += qd[d] * orc_load(k, base + d, dt);
                    s[t] = scale * dot;
                }
                double m;
                orc_softmax_lse(s, u, &m, &l[g]);
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (long t = 0; t < u; ++t) {
                        size_t base = (size_t)(((off + t) * Hkv + hk) * D);
                        acc += exp(s[t] - l[g]) * orc_load(v, base + d, dt);
                    }
                    o[(long)g * D + d] = u > 0 ? acc : 0.0;
                }
                if (seg_out)
                    for (int d = 0; d < D; ++d)
                        seg_out[(((long)i * groups + g) * Hq + h) * D + d] = o[(long)g * D + d];
                if (seg_lse) seg_lse[((long)i * groups + g) * Hq + h] = l[g];
            }

            /* combine: softmax over live groups of (lse + prior) */
            double mx = -INFINITY;
            for (int g = 0; g < groups; ++g) {
                if (used[(long)i * groups + g] <= 0) continue;
                double prior = g < topk ? bias[(long)i * topk + g] : 0.0;
                double lg = l[g] + prior;
                if (lg > mx) mx = lg;
            }
            double denom = 0.0;
            for (int g = 0; g < groups; ++g) {
                if (used[(long)i * groups + g] <= 0) continue;
                double prior = g < topk ? bias[(long)i * topk + g] : 0.0;
                denom += exp(l[g] + prior - mx);
            }
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int g = 0; g < groups; ++g) {
                    if (used[(long)i * groups + g] <= 0) continue;
                    double prior = g < topk ? bias[(long)i * topk + g] : 0.0;
                    acc += exp(l[g] + prior - mx) / denom * o[(long)g * D + d];
                }
                out[((long)i * Hq + h) * D + d] = acc; /* no live group: acc stays 0 */
            }
            free(qd);
            free(l);
            free(o);
            free(s);
        }
    }
    return status;
}

/* ---------------------------------------------------------------------------
 * Merge of partial attention results by their log-sum-exp: the Split-KV
 * merge [FA FlashAttentionCuTeDSLCompileSpec: num_splits, return_softmax_lse]
 * and, with a prior and a live mask, the DASH combine [DASH flash_dash_attention].
 *
 *   part_out [N, S, H, D], part_lse [N, S, H], prior [N, S] (nullable),
 *   live [N, S] int32 (nullable; part s of row n is dead when live <= 0)
 *   logit_s = part_lse + prior;  a part with logit -inf is empty
 *   lse     = ln sum_{s live} exp(logit_s)
 *   out     = sum_{s live} exp(logit_s - lse) * part_out_s
 * With no live part: out = 0, lse = -inf.
 * ------------------------------------------------------------------------- */
int orc_lse_merge(const double* part_out, const double* part_lse, const double* prior,
                  const int32_t* live, int N, int S, int H, int D, double* out, double* lse_out) {
    if (N < 0 || S < 0 || H <= 0 || D <= 0) return -1;
    for (long nn = 0; nn < N; ++nn) {
        for (int h = 0; h < H; ++h) {
            double mx = -INFINITY;
            for (int s = 0; s < S; ++s) {
                if (live && live[nn * S + s] <= 0) continue;
                double lg = part_lse[(nn * S + s) * H + h] + (prior ? prior[nn * S + s] : 0.0);
                if (lg > mx) mx = lg;
            }
            if (mx == -INFINITY) {
                for (int d = 0; d < D; ++d) out[(nn * H + h) * D + d] = 0.0;
                if (lse_out) lse_out[nn * H + h] = -INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int s = 0; s < S; ++s) {
                if (live && live[nn * S + s] <= 0) continue;
                double lg = part_lse[(nn * S + s) * H + h] + (prior ? prior[nn * S + s] : 0.0);
                if (lg == -INFINITY) continue;
                sum += exp(lg - mx);
            }
            double total = mx + log(sum);
            if (lse_out) lse_out[nn * H + h] = total;
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int s = 0; s < S; ++s) {
                    if (live && live[nn * S + s] <= 0) continue;
                    double lg = part_lse[(nn * S + s) * H + h] + (prior ? prior[nn * S + s] : 0.0);
                    if (lg == -INFINITY) continue;
                    acc += exp(lg - total) * part_out[((nn * S + s) * H + h) * D + d];
                }
                out[(nn * H + h) * D + d] = acc;
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * KV-cache write [TS FlashInferTSImpl.do_kv_cache_update: reshape_and_cache_flash].
 *
 * Token t's key and value rows [Hkv, D] go to slot s = slot_mapping[t] of the
 * paged cache: page s / P, offset s % P, K into [..., :D] and V into
 * [..., D:] (the layout _kv_views reads back).  A negative slot is a padding
 * token and writes nothing.  A 16-bit cache of the input's type stores the
 * input bits unchanged; an fp8 cache stores e4m3(x / scale) with the key
 * (value) scale, the quotient taken in fp32 and rounded to nearest even,
 * saturating to +-448 (the largest finite e4m3fn value).
 * ------------------------------------------------------------------------- */
uint8_t orc_encode_e4m3(float x) {
    if (isnan(x)) return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;        /* saturate (and +-inf) */
    if (a < ldexp(1.0, -6)) {
        /* subnormal step 2^-9; a result of 8 is the smallest normal, code 0x08 */
        double t = nearbyint(a * 512.0);
        return sign | (uint8_t)t;
    }
    int k;
    frexp(a, &k);                               /* a = f * 2^k, f in [0.5, 1) */
    int e = k - 1;                              /* a = s * 2^e, s in [1, 2) */
    double t = nearbyint((ldexp(a, -e) - 1.0) * 8.0);
    if (t >= 8.0) {
        t = 0.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && t > 6.0)) return sign | 0x7E;  /* 480 and up round to the NaN code: saturate */
    return sign | (uint8_t)(((e + 7) << 3) | (int)t);
}

int orc_cache_write(const void* key, const void* value, int in_dt, const int64_t* slot_mapping,
                    long num_tokens, int Hkv, int D, int P, long num_pages, void* cache, int kv_dt,
                    float k_scale, float v_scale) {
    if (Hkv <= 0 || D <= 0 || P <= 0 || num_pages <= 0) return -1;
    if (kv_dt != ORC_FP8_E4M3 && kv_dt != in_dt) return -1;
    for (long t = 0; t < num_tokens; ++t) {
        const int64_t s = slot_mapping[t];
        if (s < 0) continue;
        const long page = (long)(s / P), off = (long)(s % P);
        if (page >= num_pages) return -2;
        for (int h = 0; h < Hkv; ++h) {
            const size_t src = ((size_t)t * Hkv + h) * D;
            const size_t dst = (((size_t)page * Hkv + h) * P + off) * 2 * (size_t)D;
            for (int d = 0; d < D; ++d) {
                if (kv_dt == ORC_FP8_E4M3) {
                    const float kx = (float)orc_load(key, src + d, in_dt);
                    const float vx = (float)orc_load(value, src + d, in_dt);
                    ((uint8_t*)cache)[dst + d] = orc_encode_e4m3(kx / k_scale);
                    ((uint8_t*)cache)[dst + D + d] = orc_encode_e4m3(vx / v_scale);
                } else {
                    ((uint16_t*)cache)[dst + d] = ((const uint16_t*)key)[src + d];
                    ((uint16_t*)cache)[dst + D + d] = ((const uint16_t*)value)[src + d];
                }
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * DASH segmented attention read from the paged cache: segment g of query i is
 * the key range [seg_start[i, g], seg_start[i, g] + used[i, g]) of request row
 * i, each key gathered through the block table exactly as paged decode reads
 * it; attention per segment and the combine are those of
 * orc_segmented_attention (scale D^-0.5, prior [bias, 0], dead segments out).
 * ------------------------------------------------------------------------- */
int orc_segmented_paged(const void* q, int dt, const void* cache, long num_pages, const int32_t* block_table,
                        long bt_stride, const int32_t* seg_start, const int32_t* used, const double* bias,
                        int n, int Hq, int Hkv, int D, int P, int topk, int bs, int local, double* out,
                        double* seg_out, double* seg_lse, int nthreads) {
    if (n < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || P <= 0 || topk < 0) return -1;
    if (Hq % Hkv != 0) return -1;
    const int G = Hq / Hkv;
    const int groups = topk + 1;
    const double scale = 1.0 / sqrt((double)D);
    if (nthreads < 1) nthreads = 1;
    for (long i = 0; i < (long)n * groups; ++i) {
        const int cap = (int)(i % groups) < topk ? bs : local;
        if (used[i] < 0 || used[i] > cap || seg_start[i] < 0) return -3;
        for (long t = seg_start[i]; t < (long)seg_start[i] + used[i]; ++t) {
            const long page = block_table[(i / groups) * bt_stride + t / P];
            if (page < 0 || page >= num_pages) return -2;
        }
    }

#pragma omp parallel for collapse(2) schedule(dynamic) num_threads(nthreads)
    for (int i = 0; i < n; ++i) {
        for (int h = 0; h < Hq; ++h) {
            const int hk = h / G;
            const int cap_max = bs > local ? bs : local;
            double* s = (double*)malloc(sizeof(double) * (size_t)(cap_max > 0 ? cap_max : 1));
            double* o = (double*)malloc(sizeof(double) * (size_t)groups * D);
            double* l = (double*)malloc(sizeof(double) * (size_t)groups);
            double* qd = (double*)malloc(sizeof(double) * (size_t)D);
            for (int d = 0; d < D; ++d) qd[d] = orc_load(q, (size_t)(((long)i * Hq + h) * D + d), dt);
            for (int g = 0; g < groups; ++g) {
                const long st = seg_start[(long)i * groups + g];
                const long u = used[(long)i * groups + g];
                for (long t = 0; t < u; ++t) {
                    const long j = st + t;
                    const long page = block_table[(long)i * bt_stride + j / P];
                    const size_t kbase = (size_t)(((page * Hkv + hk) * P + j % P) * 2L * D);
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += qd[d] * orc_load(cache, kbase + d, dt);
                    s[t] = scale * dot;
                }
                double m;
                orc_softmax_lse(s, u, &m, &l[g]);
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (long t = 0; t < u; ++t) {
                        const long j = st + t;
                        const long page = block_table[(long)i * bt_stride + j / P];
                        const size_t vbase = (size_t)(((page * Hkv + hk) * P + j % P) * 2L * D + D);
                        acc += exp(s[t] - l[g]) * orc_load(cache, vbase + d, dt);
                    }
                    o[(long)g * D + d] = u > 0 ? acc : 0.0;
                }
                if (seg_out)
                    for (int d = 0; d < D; ++d)
                        seg_out[(((long)i * groups + g) * Hq + h) * D + d] = o[(long)g * D + d];
                if (seg_lse) seg_lse[((long)i * groups + g) * Hq + h] = l[g];
            }
            double mx = -INFINITY;
            for (int g = 0; g < groups; ++g) {
                if (used[(long)i * groups + g] <= 0) continue;
                const double lg = l[g] + (g < topk ? bias[(long)i * topk + g] : 0.0);
                if (lg > mx) mx = lg;
            }
            double denom = 0.0;
            for (int g = 0; g < groups; ++g) {
                if (used[(long)i * groups + g] <= 0) continue;
                denom += exp(l[g] + (g < topk ? bias[(long)i * topk + g] : 0.0) - mx);
            }
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int g = 0; g < groups; ++g) {
                    if (used[(long)i * groups + g] <= 0) continue;
                    acc += exp(l[g] + (g < topk ? bias[(long)i * topk + g] : 0.0) - mx) / denom *
                           o[(long)g * D + d];
                }
                out[((long)i * Hq + h) * D + d] = acc;
            }
            free(qd);
            free(l);
            free(o);
            free(s);
        }
    }
    return 0;
}
