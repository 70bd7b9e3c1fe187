/*
 * hattn_oracle.c -- plain fp64 CPU oracle for hybrid sliding-window / global
 * attention with a learnable per-head attention sink.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle_hattn.so and
 * is loaded by the tests, by __graft_entry__.smoke() and by bench.py's CPU
 * baseline leg.  The product path (the CUDA library) never links, loads or
 * calls it, and it shares no code, header or table with that path.
 *
 * What is computed (every step is the plain definition, no tiling, no online
 * softmax, no reordering):
 *
 *   MiMo-V2-Flash Technical Report (xllm-io paper review), section 3.1
 *   "overall structure": GQA with 64 query heads over 8 KV heads (SWA layers)
 *   or 4 KV heads (GA layers); Q/K head dim 192, V head dim 128; RoPE on the
 *   first 64 dims; window W = 128.
 *   Same page, section 4 "pre-training": RoPE base 10K for SWA, 5M for GA
 *   after context extension.
 *   Same page, section 3.2 "hybrid SWA architecture": a learnable sink bias
 *   s_sink is added to the softmax denominator of every head (gpt-oss style).
 *   plmsmile notes on the MiMo series, MiMo-V2-Flash "Learnable Attention
 *   Sink": the sink sits in the denominator only, carries no value, and the
 *   weights of real tokens may sum to less than one.
 *   Same notes, "local window": an SWA query reads only the neighbouring 128
 *   tokens.
 *
 * Readings taken where the pages are silent (all listed in the design notes):
 *   - window W > 0 admits keys j with j <= p and p - j < W (W keys including
 *     the query itself); W == 0 means global causal attention;
 *   - the sink is a raw logit (not multiplied by the softmax scale), one per
 *     query head, and the returned lse includes it;
 *   - query head h reads KV head floor(h / G), G = hq / hkv;
 *   - RoPE rotates pairs (i, i + R/2) for i < R/2 ("rotate-half"), with
 *     theta_i = base^(-2 i / R), R = rope_dim;
 *   - decode / verify queries are the last T tokens of each sequence, at
 *     positions L - T + t.
 *
 * Arithmetic: inputs arrive as bf16 bit patterns and are widened exactly to
 * double; everything after that is double precision.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_NO_MEM 2

/* bf16 bit pattern -> double, exact (bf16 is the top half of an IEEE float). */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* theta_i = base^(-2i/R) for i < R/2. */
static double* rope_thetas(int rope_dim, double base) {
    int half = rope_dim / 2;
    double* th = (double*)malloc(sizeof(double) * (size_t)(half + 1));
    if (!th) return NULL;
    for (int i = 0; i < half; ++i) th[i] = pow(base, -2.0 * (double)i / (double)rope_dim);
    return th;
}

/* cos/sin of pos * theta_i for i < R/2. */
static void rope_angles(long pos, int rope_dim, const double* theta, double* c, double* s) {
    int half = rope_dim / 2;
    for (int i = 0; i < half; ++i) {
        double a = (double)pos * theta[i];
        c[i] = cos(a);
        s[i] = sin(a);
    }
}

/* y = RoPE(x) at the angles (c, s): pairs (i, i + R/2) rotated, rest copied. */
static void rope_apply(const double* x, double* y, int dim, int rope_dim, const double* c,
                       const double* s) {
    int half = rope_dim / 2;
    for (int d = 0; d < dim; ++d) y[d] = x[d];
    for (int i = 0; i < half; ++i) {
        double a = x[i], b = x[i + half];
        y[i] = a * c[i] - b * s[i];
        y[i + half] = b * c[i] + a * s[i];
    }
}

/*
 * Finish one attention row from its logits z[0..n) (keys in position order):
 * m = max(z, sink), Z = sum exp(z - m) (+ exp(sink - m)),
 * out = sum exp(z_j - m) v_j / Z, lse = m + ln Z.  v_j is the bf16 value row
 * of key j, widened exactly.  sink_on selects whether exp(sink) joins the
 * denominator.  With no key and no sink the row is empty: out = 0, lse = -inf.
 */
static void softmax_row(const double* z, long n, const uint16_t* const* v_rows, int dv, double sink,
                        int sink_on, double* out, double* lse) {
    double m = -INFINITY;
    for (long j = 0; j < n; ++j)
        if (z[j] > m) m = z[j];
    if (sink_on && sink > m) m = sink;
    for (int e = 0; e < dv; ++e) out[e] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double Z = 0.0;
    for (long j = 0; j < n; ++j) {
        double w = exp(z[j] - m);
        Z += w;
        for (int e = 0; e < dv; ++e) out[e] += w * bf16_to_double(v_rows[j][e]);
    }
    if (sink_on) Z += exp(sink - m);
    for (int e = 0; e < dv; ++e) out[e] /= Z;
    *lse = m + log(Z);
}

static double dot(const double* a, const double* b, int n) {
    double acc = 0.0;
    for (int d = 0; d < n; ++d) acc += a[d] * b[d];
    return acc;
}

static int omp_threads_used(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

int hattn_oracle_num_threads(int nthreads) { return omp_threads_used(nthreads); }

/* Standalone RoPE of rows x[n, dim] at positions pos[n]; results in double. */
int hattn_oracle_rope(const uint16_t* x, const long* pos, double* y, long n, int dim, int rope_dim,
                      double base) {
    if (!x || !pos || !y || n < 0 || dim <= 0 || rope_dim < 0 || rope_dim > dim || (rope_dim & 1))
        return ORACLE_BAD_ARG;
    double* xd = (double*)malloc(sizeof(double) * (size_t)dim);
    double* c = (double*)malloc(sizeof(double) * (size_t)(rope_dim / 2 + 1));
    double* s = (double*)malloc(sizeof(double) * (size_t)(rope_dim / 2 + 1));
    double* th = rope_thetas(rope_dim, base);
    if (!xd || !c || !s || !th) {
        free(xd); free(c); free(s); free(th);
        return ORACLE_NO_MEM;
    }
    for (long r = 0; r < n; ++r) {
        for (int d = 0; d < dim; ++d) xd[d] = bf16_to_double(x[r * dim + d]);
        rope_angles(pos[r], rope_dim, th, c, s);
        rope_apply(xd, y + r * dim, dim, rope_dim, c, s);
    }
    free(xd); free(c); free(s); free(th);
    return ORACLE_OK;
}

/* Which sequence holds packed token n. */
static int seq_of_token(const int* cu, int batch, long n) {
    for (int b = 0; b < batch; ++b)
        if (n >= cu[b] && n < cu[b + 1]) return b;
    return -1;
}

/*
 * Prefill over packed variable-length sequences.
 *   q    bf16 [total, hq, dqk]   un-rotated
 *   k    bf16 [total, hkv, dqk]  un-rotated
 *   v    bf16 [total, hkv, dv]
 *   sink double [hq]
 *   cu_seqlens int [batch + 1], cu[0] = 0, cu[batch] = total
 *   rows: packed token indices to evaluate (n_rows of them); NULL = all tokens
 *   out  double [n_rows, hq, dv], lse double [n_rows, hq]
 * Positions restart at 0 in every sequence.
 */
int hattn_oracle_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v, const double* sink,
                         double* out, double* lse, int batch, const int* cu_seqlens, int hq, int hkv,
                         int dqk, int dv, int rope_dim, double rope_base, int window, double scale,
                         const long* rows, long n_rows, int nthreads) {
    if (!q || !k || !v || !sink || !out || !lse || !cu_seqlens || batch <= 0 || hq <= 0 ||
        hkv <= 0 || hq % hkv || dqk <= 0 || dv <= 0 || rope_dim < 0 || rope_dim > dqk ||
        (rope_dim & 1) || window < 0)
        return ORACLE_BAD_ARG;
    long total = cu_seqlens[batch];
    if (!rows) n_rows = total;
    int G = hq / hkv;
    int maxlen = 0;
    for (int b = 0; b < batch; ++b) {
        int L = cu_seqlens[b + 1] - cu_seqlens[b];
        if (L < 0) return ORACLE_BAD_ARG;
        if (L > maxlen) maxlen = L;
    }
    double* th = rope_thetas(rope_dim, rope_base);
    if (!th) return ORACLE_NO_MEM;
    int bad = 0;
    int nt = omp_threads_used(nthreads);
    long maxkeys = (window > 0 && window < maxlen) ? window : maxlen;
#pragma omp parallel num_threads(nt)
    {
        int half = rope_dim / 2 + 1;
        double* qd = (double*)malloc(sizeof(double) * (size_t)dqk);
        double* qr = (double*)malloc(sizeof(double) * (size_t)dqk * (size_t)G);
        double* c = (double*)malloc(sizeof(double) * (size_t)half);
        double* s = (double*)malloc(sizeof(double) * (size_t)half);
        double* kd = (double*)malloc(sizeof(double) * (size_t)dqk);
        double* kr = (double*)malloc(sizeof(double) * (size_t)dqk);
        double* z = (double*)malloc(sizeof(double) * (size_t)(maxkeys + 1) * (size_t)G);
        const uint16_t** vr = (const uint16_t**)malloc(sizeof(uint16_t*) * (size_t)(maxkeys + 1));
        if (!qd || !qr || !c || !s || !kd || !kr || !z || !vr) {
#pragma omp atomic write
            bad = ORACLE_NO_MEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long r = 0; r < n_rows; ++r) {
                long n = rows ? rows[r] : r;
                int b = seq_of_token(cu_seqlens, batch, n);
                if (b < 0) {
#pragma omp atomic write
                    bad = ORACLE_BAD_ARG;
                    continue;
                }
                long base_tok = cu_seqlens[b];
                long p = n - base_tok; /* position within its sequence */
                long lo = (window > 0 && p - window + 1 > 0) ? p - window + 1 : 0;
                long nk = p - lo + 1;
                for (int g = 0; g < hkv; ++g) {
                    /* the G query heads of this KV head, rotated at position p */
                    rope_angles(p, rope_dim, th, c, s);
                    for (int hh = 0; hh < G; ++hh) {
                        const uint16_t* qs = q + (n * hq + g * G + hh) * (long)dqk;
                        for (int d = 0; d < dqk; ++d) qd[d] = bf16_to_double(qs[d]);
                        rope_apply(qd, qr + (long)hh * dqk, dqk, rope_dim, c, s);
                    }
                    /* logits against every visible key, rotated at its own position */
                    for (long j = lo; j <= p; ++j) {
                        const uint16_t* ks = k + ((base_tok + j) * hkv + g) * (long)dqk;
                        for (int d = 0; d < dqk; ++d) kd[d] = bf16_to_double(ks[d]);
                        rope_angles(j, rope_dim, th, c, s);
                        rope_apply(kd, kr, dqk, rope_dim, c, s);
                        for (int hh = 0; hh < G; ++hh)
                            z[(long)hh * nk + (j - lo)] = scale * dot(qr + (long)hh * dqk, kr, dqk);
                        vr[j - lo] = v + ((base_tok + j) * hkv + g) * (long)dv;
                    }
                    for (int hh = 0; hh < G; ++hh) {
                        int h = g * G + hh;
                        softmax_row(z + (long)hh * nk, nk, vr, dv, sink[h], 1,
                                    out + (r * hq + h) * (long)dv, lse + r * hq + h);
                    }
                }
            }
        }
        free(qd); free(qr); free(c); free(s); free(kd); free(kr); free(z); free((void*)vr);
    }
    free(th);
    return bad;
}

/*
 * Decode / MTP-verify: the last T tokens of each sequence attend over that
 * sequence's whole history (plmsmile notes, MiMo-V2-Flash MTP: drafts are verified in one
 * parallel pass of the main model).
 *   q      bf16 [B, T, hq, dqk]  un-rotated, query t at position L_b - T + t
 *   k_hist bf16 [B, Lmax, hkv, dqk] un-rotated keys by absolute position
 *   v_hist bf16 [B, Lmax, hkv, dv]
 *   seqlens int [B], L_b >= T, L_b <= Lmax (tokens incl. the T queries)
 *   key_lo, key_hi: only keys with key_lo <= j < key_hi take part
 *                   (key_hi < 0: no upper limit); used to pin the split/merge
 *                   identity of the log-sum-exp.
 *   sink_on: 0 drops the sink term (partial results of a split).
 *   out double [B, T, hq, dv], lse double [B, T, hq]
 */
int hattn_oracle_decode(const uint16_t* q, const uint16_t* k_hist, const uint16_t* v_hist,
                        const int* seqlens, const double* sink, double* out, double* lse, int B,
                        int T, long Lmax, int hq, int hkv, int dqk, int dv, int rope_dim,
                        double rope_base, int window, double scale, long key_lo, long key_hi,
                        int sink_on, int nthreads) {
    if (!q || !k_hist || !v_hist || !seqlens || !sink || !out || !lse || B <= 0 || T <= 0 ||
        hq <= 0 || hkv <= 0 || hq % hkv || dqk <= 0 || dv <= 0 || rope_dim < 0 ||
        rope_dim > dqk || (rope_dim & 1) || window < 0)
        return ORACLE_BAD_ARG;
    for (int b = 0; b < B; ++b)
        if (seqlens[b] < T || seqlens[b] > Lmax) return ORACLE_BAD_ARG;
    int G = hq / hkv;
    double* th = rope_thetas(rope_dim, rope_base);
    if (!th) return ORACLE_NO_MEM;
    int bad = 0;
    int nt = omp_threads_used(nthreads);
    long nrows = (long)B * T;
    long maxkeys = (window > 0 && window < Lmax) ? window : Lmax;
#pragma omp parallel num_threads(nt)
    {
        int half = rope_dim / 2 + 1;
        double* qd = (double*)malloc(sizeof(double) * (size_t)dqk);
        double* qr = (double*)malloc(sizeof(double) * (size_t)dqk * (size_t)G);
        double* c = (double*)malloc(sizeof(double) * (size_t)half);
        double* s = (double*)malloc(sizeof(double) * (size_t)half);
        double* kd = (double*)malloc(sizeof(double) * (size_t)dqk);
        double* kr = (double*)malloc(sizeof(double) * (size_t)dqk);
        double* z = (double*)malloc(sizeof(double) * (size_t)(maxkeys + 1) * (size_t)G);
        const uint16_t** vr = (const uint16_t**)malloc(sizeof(uint16_t*) * (size_t)(maxkeys + 1));
        if (!qd || !qr || !c || !s || !kd || !kr || !z || !vr) {
#pragma omp atomic write
            bad = ORACLE_NO_MEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long r = 0; r < nrows; ++r) {
                int b = (int)(r / T);
                long L = seqlens[b];
                long p = L - T + (r % T);
                long lo = (window > 0 && p - window + 1 > 0) ? p - window + 1 : 0;
                if (lo < key_lo) lo = key_lo;
                long hi = p; /* inclusive */
                if (key_hi >= 0 && hi > key_hi - 1) hi = key_hi - 1;
                long nk = hi >= lo ? hi - lo + 1 : 0;
                for (int g = 0; g < hkv; ++g) {
                    rope_angles(p, rope_dim, th, c, s);
                    for (int hh = 0; hh < G; ++hh) {
                        const uint16_t* qs = q + ((r * hq) + g * G + hh) * (long)dqk;
                        for (int d = 0; d < dqk; ++d) qd[d] = bf16_to_double(qs[d]);
                        rope_apply(qd, qr + (long)hh * dqk, dqk, rope_dim, c, s);
                    }
                    for (long j = lo; j <= hi; ++j) {
                        const uint16_t* ks = k_hist + (((long)b * Lmax + j) * hkv + g) * (long)dqk;
                        for (int d = 0; d < dqk; ++d) kd[d] = bf16_to_double(ks[d]);
                        rope_angles(j, rope_dim, th, c, s);
                        rope_apply(kd, kr, dqk, rope_dim, c, s);
                        for (int hh = 0; hh < G; ++hh)
                            z[(long)hh * nk + (j - lo)] = scale * dot(qr + (long)hh * dqk, kr, dqk);
                        vr[j - lo] = v_hist + (((long)b * Lmax + j) * hkv + g) * (long)dv;
                    }
                    for (int hh = 0; hh < G; ++hh) {
                        int h = g * G + hh;
                        softmax_row(z + (long)hh * nk, nk, vr, dv, sink[h], sink_on,
                                    out + (r * hq + h) * (long)dv, lse + r * hq + h);
                    }
                }
            }
        }
        free(qd); free(qr); free(c); free(s); free(kd); free(kr); free(z); free((void*)vr);
    }
    free(th);
    return bad;
}

/*
 * Backward of the prefill: the gradients of the scalar sum(dout * out) with
 * respect to q, k, v and the sink logits, i.e. the chain rule through the
 * forward definition above (MiMo-V2-Flash paper review, section 3.2: the sink
 * is a learnable per-head parameter, so its gradient is part of the step; the
 * sink carries no value, so it enters only through the softmax denominator).
 * Written out per row, in the forward's notation:
 *   z_j = scale * q'.k'_j over the visible keys, p_j = exp(z_j - lse),
 *   p_sink = exp(sink - lse), o = sum_j p_j v_j;
 *   delta = dout . o;  dp_j = dout . v_j;  dz_j = p_j (dp_j - delta);
 *   dsink += -p_sink * delta;
 *   dq' += scale * sum_j dz_j k'_j;  dk'_j += scale * dz_j q';  dv_j += p_j dout;
 * then dq, dk = the transposed rotation of dq', dk' (pairs (i, i + R/2) turned
 * back by the same angle).  o and lse are recomputed here in double, not taken
 * from any forward output.
 *   dout bf16 [total, hq, dv];  dq double [total, hq, dqk], dk [total, hkv, dqk],
 *   dv double [total, hkv, dv], dsink double [hq]
 * Work is split by (sequence, KV head): each task owns its keys' dk, dv rows
 * and its queries' dq rows, so the tasks write disjoint outputs; the sink
 * gradient is summed over the tasks afterwards, in task order.
 */
static void rope_apply_transposed(double* g, int rope_dim, const double* c, const double* s) {
    int half = rope_dim / 2;
    for (int i = 0; i < half; ++i) {
        double a = g[i], b = g[i + half];
        g[i] = a * c[i] + b * s[i];
        g[i + half] = b * c[i] - a * s[i];
    }
}

int hattn_oracle_prefill_backward(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  const double* sink, const uint16_t* dout, double* dq, double* dk,
                                  double* dv_out, double* dsink, int batch, const int* cu_seqlens,
                                  int hq, int hkv, int dqk, int dv, int rope_dim, double rope_base,
                                  int window, double scale, int nthreads) {
    if (!q || !k || !v || !sink || !dout || !dq || !dk || !dv_out || !dsink || !cu_seqlens ||
        batch <= 0 || hq <= 0 || hkv <= 0 || hq % hkv || dqk <= 0 || dv <= 0 || rope_dim < 0 ||
        rope_dim > dqk || (rope_dim & 1) || window < 0)
        return ORACLE_BAD_ARG;
    int G = hq / hkv;
    int maxlen = 0;
    for (int b = 0; b < batch; ++b) {
        int L = cu_seqlens[b + 1] - cu_seqlens[b];
        if (L < 0) return ORACLE_BAD_ARG;
        if (L > maxlen) maxlen = L;
    }
    double* th = rope_thetas(rope_dim, rope_base);
    double* ds_task = (double*)calloc((size_t)batch * hkv * G, sizeof(double));
    if (!th || !ds_task) {
        free(th); free(ds_task);
        return ORACLE_NO_MEM;
    }
    int bad = 0;
    int nt = omp_threads_used(nthreads);
    long ntask = (long)batch * hkv;
    long ml = maxlen > 0 ? maxlen : 1;
#pragma omp parallel num_threads(nt)
    {
        int half = rope_dim / 2 + 1;
        double* c = (double*)malloc(sizeof(double) * (size_t)half);
        double* s = (double*)malloc(sizeof(double) * (size_t)half);
        double* xd = (double*)malloc(sizeof(double) * (size_t)dqk);
        double* kr = (double*)malloc(sizeof(double) * (size_t)ml * dqk);  /* rotated keys */
        double* vd = (double*)malloc(sizeof(double) * (size_t)ml * dv);
        double* gk = (double*)malloc(sizeof(double) * (size_t)ml * dqk);  /* dk' */
        double* gv = (double*)malloc(sizeof(double) * (size_t)ml * dv);
        double* qr = (double*)malloc(sizeof(double) * (size_t)dqk);
        double* gq = (double*)malloc(sizeof(double) * (size_t)dqk);       /* dq' */
        double* go = (double*)malloc(sizeof(double) * (size_t)dv);
        double* o = (double*)malloc(sizeof(double) * (size_t)dv);
        double* z = (double*)malloc(sizeof(double) * (size_t)ml);
        if (!c || !s || !xd || !kr || !vd || !gk || !gv || !qr || !gq || !go || !o || !z) {
#pragma omp atomic write
            bad = ORACLE_NO_MEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long task = 0; task < ntask; ++task) {
                int b = (int)(task / hkv), g = (int)(task % hkv);
                long tok0 = cu_seqlens[b];
                long L = cu_seqlens[b + 1] - tok0;
                for (long j = 0; j < L; ++j) {
                    const uint16_t* ks = k + ((tok0 + j) * hkv + g) * (long)dqk;
                    for (int d = 0; d < dqk; ++d) xd[d] = bf16_to_double(ks[d]);
                    rope_angles(j, rope_dim, th, c, s);
                    rope_apply(xd, kr + j * dqk, dqk, rope_dim, c, s);
                    const uint16_t* vs = v + ((tok0 + j) * hkv + g) * (long)dv;
                    for (int e = 0; e < dv; ++e) vd[j * dv + e] = bf16_to_double(vs[e]);
                }
                for (long j = 0; j < L * dqk; ++j) gk[j] = 0.0;
                for (long j = 0; j < L * dv; ++j) gv[j] = 0.0;
                for (int hh = 0; hh < G; ++hh) {
                    int h = g * G + hh;
                    double dsink_h = 0.0;
                    for (long p = 0; p < L; ++p) {
                        long n = tok0 + p;
                        long lo = (window > 0 && p - window + 1 > 0) ? p - window + 1 : 0;
                        const uint16_t* qs = q + (n * hq + h) * (long)dqk;
                        for (int d = 0; d < dqk; ++d) xd[d] = bf16_to_double(qs[d]);
                        rope_angles(p, rope_dim, th, c, s);
                        rope_apply(xd, qr, dqk, rope_dim, c, s);
                        const uint16_t* gs = dout + (n * hq + h) * (long)dv;
                        for (int e = 0; e < dv; ++e) go[e] = bf16_to_double(gs[e]);
                        /* forward again: logits, lse (with the sink), o */
                        double m = sink[h];
                        for (long j = lo; j <= p; ++j) {
                            z[j] = scale * dot(qr, kr + j * dqk, dqk);
                            if (z[j] > m) m = z[j];
                        }
                        double Z = exp(sink[h] - m);
                        for (long j = lo; j <= p; ++j) Z += exp(z[j] - m);
                        double lse = m + log(Z);
                        for (int e = 0; e < dv; ++e) o[e] = 0.0;
                        for (long j = lo; j <= p; ++j) {
                            double pj = exp(z[j] - lse);
                            for (int e = 0; e < dv; ++e) o[e] += pj * vd[j * dv + e];
                        }
                        double delta = dot(go, o, dv);
                        dsink_h += -exp(sink[h] - lse) * delta;
                        for (int d = 0; d < dqk; ++d) gq[d] = 0.0;
                        for (long j = lo; j <= p; ++j) {
                            double pj = exp(z[j] - lse);
                            double dz = pj * (dot(go, vd + j * dv, dv) - delta);
                            for (int d = 0; d < dqk; ++d) {
                                gq[d] += scale * dz * kr[j * dqk + d];
                                gk[j * dqk + d] += scale * dz * qr[d];
                            }
                            for (int e = 0; e < dv; ++e) gv[j * dv + e] += pj * go[e];
                        }
                        rope_apply_transposed(gq, rope_dim, c, s);
                        for (int d = 0; d < dqk; ++d) dq[(n * hq + h) * (long)dqk + d] = gq[d];
                    }
                    ds_task[task * G + hh] = dsink_h;
                }
                for (long j = 0; j < L; ++j) {
                    rope_angles(j, rope_dim, th, c, s);
                    rope_apply_transposed(gk + j * dqk, rope_dim, c, s);
                    for (int d = 0; d < dqk; ++d)
                        dk[((tok0 + j) * hkv + g) * (long)dqk + d] = gk[j * dqk + d];
                    for (int e = 0; e < dv; ++e)
                        dv_out[((tok0 + j) * hkv + g) * (long)dv + e] = gv[j * dv + e];
                }
            }
        }
        free(c); free(s); free(xd); free(kr); free(vd); free(gk); free(gv); free(qr); free(gq);
        free(go); free(o); free(z);
    }
    for (int h = 0; h < hq; ++h) dsink[h] = 0.0;
    for (long task = 0; task < ntask; ++task)
        for (int hh = 0; hh < G; ++hh) dsink[(task % hkv) * G + hh] += ds_task[task * G + hh];
    free(th);
    free(ds_task);
    return bad;
}
