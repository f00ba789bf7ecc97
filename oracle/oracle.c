/*
 * oracle.c -- float64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no source, header, table or helper with
 * the CUDA library and includes nothing from it.
 *
 * What it computes (the plain definition, written out, no tiling, no fusion):
 *
 *   "FlashAttention V3 实战: Hopper ... Paged KV Cache", section 一 (problem
 *   definition): Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V.
 *   "Capstone: CUDA Softmax 与 Attention 算子", section 1.1: the same
 *   definition, and section 2.1: the row softmax is the three-pass safe
 *   softmax -- pass 1 m = max_j x_j, pass 2 l = sum_j exp(x_j - m),
 *   pass 3 p_j = exp(x_j - m) / l.
 *
 * For every output row (b, h, i), in float64, on exactly widened inputs:
 *   s_j = scale * sum_c q_ic k_jc         for j in the row's valid key set
 *   m   = max_j s_j                        (pass 1)
 *   l   = sum_j exp(s_j - m)               (pass 2)
 *   p_j = exp(s_j - m) / l;  o_i = sum_j p_j v_j   (pass 3)
 *   lse = m + ln(l)
 *
 * Readings where the pages leave a step open (each is listed in the design
 * notes with its justification):
 *   - scale is the caller's value (1/sqrt(d) in every workload), applied to
 *     the dot product before the softmax;
 *   - causal masking is the lower-triangular mask, aligned bottom-right when
 *     Nq != Nk: key j is valid for query i iff j <= i + (Nk - Nq);
 *   - a row with no valid key has o = 0 and lse = -inf;
 *   - lse is the natural-log log-sum-exp of the scaled scores;
 *   - FP8 inputs are decoded e4m3fn codes multiplied by the per-tensor
 *     descale; no probability quantisation happens here.
 *
 * Paged decode ("FlashAttention V3 实战", section 3.2, paged KV cache) is the
 * same row computation with one query per request, where key t of request r
 * lives at cache[block_table[r][t / page_size]][t % page_size][h][:].
 *
 * Paged attention in general (oracle_paged_attention) extends that to
 *   - grouped KV heads: the cache holds H_kv heads, H_kv divides H, and query
 *     head h reads KV head h / (H / H_kv) (H_kv = H is plain multi-head
 *     attention, H_kv = 1 multi-query attention);
 *   - several new query tokens per request (a prefill chunk appended to a
 *     cached prefix): request r owns query tokens cu_q[r] .. cu_q[r+1]-1 of a
 *     token-major q [total_q, H, d]; its keys are the seq_lens[r] cache
 *     entries, the last q_len of which belong to the new tokens, so query i
 *     of the request sits at position seq_lens[r] - q_len + i and, under the
 *     causal mask, sees keys t <= that position (the bottom-right alignment
 *     used for dense attention).
 *
 * Backward (oracle_attention_bwd): the gradients of the same definition.
 * The pages keep only the row statistics of the forward pass and recompute
 * P from Q and K when gradients are needed ("Capstone", section 6.1, the
 * pitfalls table, and section 7.3, question 1); the gradient formulas are the
 * chain rule applied to the definition, written out for one row i with
 * upstream gradient dO_i:
 *   o_i   = sum_j p_ij v_j,   p_ij = exp(s_ij - lse_i),  s_ij = scale q_i.k_j
 *   dV_j += p_ij dO_i
 *   dP_ij = dO_i . v_j
 *   D_i   = dO_i . o_i        (= sum_j p_ij dP_ij)
 *   dS_ij = p_ij (dP_ij - D_i)   (the softmax Jacobian applied to dP)
 *   dQ_i  = scale sum_j dS_ij k_j,   dK_j += scale dS_ij q_i
 * Masked (invisible) keys have p_ij = 0 and contribute nothing.
 *
 * Input element types: float64, float32, bfloat16 bit patterns, e4m3fn bit
 * patterns.  bf16 and e4m3fn are decoded from their bit-level definitions.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F64 = 0, OR_F32 = 1, OR_BF16 = 2, OR_E4M3 = 3 };

enum { OR_OK = 0, OR_BAD_ARG = 1, OR_NO_MEM = 2, OR_BAD_PAGE = 3 };

/* ---- element decoding ------------------------------------------------- */

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 e4m3fn: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits,
 * subnormals when the exponent field is 0, no infinities, and the two codes
 * with all exponent and mantissa bits set (0x7f, 0xff) are NaN. */
static double e4m3_bits_to_double(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int mant = b & 7;
    double mag;
    if (e == 15 && mant == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)mant / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, e - 7);
    return sign ? -mag : mag;
}

static int dtype_ok(int dt) { return dt == OR_F64 || dt == OR_F32 || dt == OR_BF16 || dt == OR_E4M3; }

/* Widen n consecutive elements starting at element index `off` into out[]. */
static void load_row(const void* base, int dt, int64_t off, int n, double descale, double* out) {
    int c;
    switch (dt) {
    case OR_F64: {
        const double* p = (const double*)base + off;
        for (c = 0; c < n; ++c) out[c] = p[c] * descale;
    } break;
    case OR_F32: {
        const float* p = (const float*)base + off;
        for (c = 0; c < n; ++c) out[c] = (double)p[c] * descale;
    } break;
    case OR_BF16: {
        const uint16_t* p = (const uint16_t*)base + off;
        for (c = 0; c < n; ++c) out[c] = bf16_bits_to_double(p[c]) * descale;
    } break;
    default: {
        const uint8_t* p = (const uint8_t*)base + off;
        for (c = 0; c < n; ++c) out[c] = e4m3_bits_to_double(p[c]) * descale;
    } break;
    }
}

int oracle_decode(const void* src, int dt, int64_t n, double* out) {
    if (!src || !out || !dtype_ok(dt) || n < 0) return OR_BAD_ARG;
    for (int64_t i = 0; i < n; i += 4096) {
        int64_t cnt = n - i < 4096 ? n - i : 4096;
        load_row(src, dt, i, (int)cnt, 1.0, out + i);
    }
    return OR_OK;
}

/* ---- one output row: the three-pass safe softmax ---------------------- */

typedef struct {
    const void* k; int k_dt; double k_ds;
    const void* v; int v_dt; double v_ds;
    int d;
    double scale;
} kv_src;

/* key_off[j] = element offset of key j's row (same offset indexes K and V).
 * qrow: the widened query row.  s: scratch of n doubles; kr: scratch of d. */
static void attend_row(const kv_src* src, const double* qrow, const int64_t* key_off, int64_t n,
                       double* s, double* kr, double* o, double* lse, double* psum) {
    const int d = src->d;
    int64_t j;
    int c;
    for (c = 0; c < d; ++c) o[c] = 0.0;
    if (n <= 0) {
        *lse = -INFINITY;
        if (psum) *psum = 0.0;
        return;
    }
    /* scores */
    for (j = 0; j < n; ++j) {
        double acc = 0.0;
        load_row(src->k, src->k_dt, key_off[j], d, src->k_ds, kr);
        for (c = 0; c < d; ++c) acc += qrow[c] * kr[c];
        s[j] = src->scale * acc;
    }
    /* pass 1: the row maximum */
    double m = s[0];
    for (j = 1; j < n; ++j)
        if (s[j] > m) m = s[j];
    /* pass 2: the denominator */
    double l = 0.0;
    for (j = 0; j < n; ++j) l += exp(s[j] - m);
    /* pass 3: probabilities and the weighted sum of value rows */
    double ps = 0.0;
    for (j = 0; j < n; ++j) {
        double p = exp(s[j] - m) / l;
        ps += p;
        load_row(src->v, src->v_dt, key_off[j], d, src->v_ds, kr);
        for (c = 0; c < d; ++c) o[c] += p * kr[c];
    }
    *lse = m + log(l);
    if (psum) *psum = ps;
}

/* ---- threading: rows are handed out one at a time from a shared counter */

typedef struct {
    /* dense problem */
    const void* q; int q_dt; double q_ds;
    kv_src kv;
    int64_t BH, Nq, Nk;
    int causal;
    const int64_t* rows; int64_t n_rows;
    /* paged problem (used when paged != 0); cu_q == NULL means one query
     * token per request */
    int paged;
    const int32_t* block_table; const int32_t* seq_lens; const int32_t* cu_q;
    int B, H, H_kv, page_size, max_pages; int64_t num_pages;
    /* outputs */
    double* o; double* lse; double* psum;
    /* work distribution and error reporting */
    int64_t next;
    int err;
} job_t;

static void* worker(void* arg) {
    job_t* jb = (job_t*)arg;
    const int d = jb->kv.d;
    int64_t nk_max = jb->paged ? (int64_t)jb->max_pages * jb->page_size : jb->Nk;
    if (nk_max < 1) nk_max = 1;
    double* s = (double*)malloc(sizeof(double) * nk_max);
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * nk_max);
    double* kr = (double*)malloc(sizeof(double) * d);
    double* qr = (double*)malloc(sizeof(double) * d);
    if (!s || !off || !kr || !qr) {
        __atomic_store_n(&jb->err, OR_NO_MEM, __ATOMIC_RELAXED);
        free(s); free(off); free(kr); free(qr);
        return NULL;
    }
    for (;;) {
        int64_t r = __atomic_fetch_add(&jb->next, 1, __ATOMIC_RELAXED);
        if (r >= jb->n_rows) break;
        int64_t n = 0, j;
        if (!jb->paged) {
            int64_t row = jb->rows ? jb->rows[r] : r; /* flattened (bh, i) */
            int64_t bh = row / jb->Nq, i = row % jb->Nq;
            load_row(jb->q, jb->q_dt, row * d, d, jb->q_ds, qr);
            n = jb->Nk;
            if (jb->causal) {
                int64_t last = i + (jb->Nk - jb->Nq); /* bottom-right aligned */
                n = last + 1;
                if (n < 0) n = 0;
                if (n > jb->Nk) n = jb->Nk;
            }
            for (j = 0; j < n; ++j) off[j] = (bh * jb->Nk + j) * d;
        } else {
            /* row r = (query token tok, query head h) of a token-major q */
            int64_t tok = r / jb->H, h = r % jb->H;
            int64_t req = tok, q_len = 1, i = 0;
            if (jb->cu_q) { /* the request whose token range holds tok */
                for (req = 0; req < jb->B; ++req)
                    if (tok >= jb->cu_q[req] && tok < jb->cu_q[req + 1]) break;
                q_len = jb->cu_q[req + 1] - jb->cu_q[req];
                i = tok - jb->cu_q[req];
            }
            const int64_t kvh = h / (jb->H / jb->H_kv); /* grouped KV head */
            load_row(jb->q, jb->q_dt, r * d, d, jb->q_ds, qr);
            const int64_t len = jb->seq_lens[req];
            n = len;
            if (n < 0 || n > (int64_t)jb->max_pages * jb->page_size) {
                __atomic_store_n(&jb->err, OR_BAD_PAGE, __ATOMIC_RELAXED);
                n = 0;
            } else if (jb->causal) {
                n = len - q_len + i + 1; /* keys up to the query's own position */
                if (n < 0) n = 0;
                if (n > len) n = len;
            }
            for (j = 0; j < n; ++j) {
                int64_t page = jb->block_table[req * jb->max_pages + j / jb->page_size];
                if (page < 0 || page >= jb->num_pages) {
                    __atomic_store_n(&jb->err, OR_BAD_PAGE, __ATOMIC_RELAXED);
                    n = 0;
                    break;
                }
                off[j] = ((page * jb->page_size + j % jb->page_size) * jb->H_kv + kvh) * d;
            }
        }
        attend_row(&jb->kv, qr, off, n, s, kr, jb->o + r * d, jb->lse + r,
                   jb->psum ? jb->psum + r : NULL);
    }
    free(s); free(off); free(kr); free(qr);
    return NULL;
}

static int run_job(job_t* jb, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if ((int64_t)nthreads > jb->n_rows) nthreads = jb->n_rows > 0 ? (int)jb->n_rows : 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
    if (!th) return OR_NO_MEM;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker, jb) != 0) break;
        ++started;
    }
    if (started == 0) worker(jb); /* no thread could be created: run inline */
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    return jb->err;
}

/* Dense attention over BHSD-contiguous tensors.
 *   q: [BH, Nq, d], k and v: [BH, Nk, d], element types q_dt / k_dt / v_dt,
 *   each element multiplied by its tensor's descale (1.0 for bf16/f32/f64).
 *   rows: optional list of flattened row ids bh*Nq + i (NULL = all rows in
 *   order).  o: [n_rows, d], lse: [n_rows], psum (optional): [n_rows], the sum
 *   of the row's probabilities as computed in pass 3. */
int oracle_attention(const void* q, int q_dt, double q_ds,
                     const void* k, int k_dt, double k_ds,
                     const void* v, int v_dt, double v_ds,
                     int64_t BH, int64_t Nq, int64_t Nk, int d, double scale, int causal,
                     const int64_t* rows, int64_t n_rows,
                     double* o, double* lse, double* psum, int nthreads) {
    if (!q || !k || !v || !o || !lse) return OR_BAD_ARG;
    if (!dtype_ok(q_dt) || !dtype_ok(k_dt) || !dtype_ok(v_dt)) return OR_BAD_ARG;
    if (BH < 0 || Nq < 0 || Nk < 0 || d < 1 || d > 4096) return OR_BAD_ARG;
    if (!rows) n_rows = BH * Nq;
    if (n_rows < 0) return OR_BAD_ARG;
    if (rows)
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= BH * Nq) return OR_BAD_ARG;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.q_dt = q_dt; jb.q_ds = q_ds;
    jb.kv.k = k; jb.kv.k_dt = k_dt; jb.kv.k_ds = k_ds;
    jb.kv.v = v; jb.kv.v_dt = v_dt; jb.kv.v_ds = v_ds;
    jb.kv.d = d; jb.kv.scale = scale;
    jb.BH = BH; jb.Nq = Nq; jb.Nk = Nk; jb.causal = causal;
    jb.rows = rows; jb.n_rows = n_rows;
    jb.o = o; jb.lse = lse; jb.psum = psum;
    return run_job(&jb, nthreads);
}

/* Paged-KV decode: one query token per request.
 *   q: [B, H, d]; k_cache and v_cache: [num_pages, page_size, H, d];
 *   block_table: [B, max_pages] physical page ids; seq_lens: [B].
 *   o: [B*H, d], lse: [B*H], psum optional [B*H].  Returns OR_BAD_PAGE (and
 *   treats the row as empty) when a length or a page id needed by a row is
 *   out of range. */
int oracle_paged_decode(const void* q, int q_dt,
                        const void* k_cache, const void* v_cache, int kv_dt,
                        const int32_t* block_table, const int32_t* seq_lens,
                        int B, int H, int d, int page_size, int max_pages, int64_t num_pages,
                        double scale, double* o, double* lse, double* psum, int nthreads) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !lse) return OR_BAD_ARG;
    if (!dtype_ok(q_dt) || !dtype_ok(kv_dt)) return OR_BAD_ARG;
    if (B < 0 || H < 1 || d < 1 || d > 4096 || page_size < 1 || max_pages < 0 || num_pages < 0)
        return OR_BAD_ARG;
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.q_dt = q_dt; jb.q_ds = 1.0;
    jb.kv.k = k_cache; jb.kv.k_dt = kv_dt; jb.kv.k_ds = 1.0;
    jb.kv.v = v_cache; jb.kv.v_dt = kv_dt; jb.kv.v_ds = 1.0;
    jb.kv.d = d; jb.kv.scale = scale;
    jb.paged = 1;
    jb.block_table = block_table; jb.seq_lens = seq_lens; jb.cu_q = NULL;
    jb.B = B; jb.H = H; jb.H_kv = H;
    jb.page_size = page_size; jb.max_pages = max_pages; jb.num_pages = num_pages;
    jb.n_rows = (int64_t)B * H;
    jb.o = o; jb.lse = lse; jb.psum = psum;
    return run_job(&jb, nthreads);
}

/* Paged attention with grouped KV heads and several query tokens per request.
 *   q: [total_q, H, d] token-major; k_cache and v_cache: [num_pages,
 *   page_size, H_kv, d] with H % H_kv == 0; block_table: [B, max_pages];
 *   cu_q: [B + 1] non-decreasing token offsets with cu_q[0] = 0 and
 *   cu_q[B] = total_q, or NULL for one query token per request (total_q = B);
 *   seq_lens: [B] key counts, each >= the request's query count.
 *   causal: query i of request r sees keys t <= seq_lens[r] - q_len_r + i.
 *   o: [total_q*H, d], lse: [total_q*H], psum optional.  Errors as
 *   oracle_paged_decode. */
int oracle_paged_attention(const void* q, int q_dt,
                           const void* k_cache, const void* v_cache, int kv_dt,
                           const int32_t* block_table, const int32_t* cu_q, const int32_t* seq_lens,
                           int B, int64_t total_q, int H, int H_kv, int d, int page_size, int max_pages,
                           int64_t num_pages, double scale, int causal,
                           double* o, double* lse, double* psum, int nthreads) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !lse) return OR_BAD_ARG;
    if (!dtype_ok(q_dt) || !dtype_ok(kv_dt)) return OR_BAD_ARG;
    if (B < 0 || total_q < 0 || H < 1 || H_kv < 1 || H % H_kv != 0 || d < 1 || d > 4096 ||
        page_size < 1 || max_pages < 0 || num_pages < 0)
        return OR_BAD_ARG;
    if (cu_q) {
        if (cu_q[0] != 0 || cu_q[B] != total_q) return OR_BAD_ARG;
        for (int r = 0; r < B; ++r)
            if (cu_q[r + 1] < cu_q[r]) return OR_BAD_ARG;
    } else if (total_q != B) {
        return OR_BAD_ARG;
    }
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.q_dt = q_dt; jb.q_ds = 1.0;
    jb.kv.k = k_cache; jb.kv.k_dt = kv_dt; jb.kv.k_ds = 1.0;
    jb.kv.v = v_cache; jb.kv.v_dt = kv_dt; jb.kv.v_ds = 1.0;
    jb.kv.d = d; jb.kv.scale = scale;
    jb.paged = 1;
    jb.causal = causal;
    jb.block_table = block_table; jb.seq_lens = seq_lens; jb.cu_q = cu_q;
    jb.B = B; jb.H = H; jb.H_kv = H_kv;
    jb.page_size = page_size; jb.max_pages = max_pages; jb.num_pages = num_pages;
    jb.n_rows = total_q * H;
    jb.o = o; jb.lse = lse; jb.psum = psum;
    return run_job(&jb, nthreads);
}

/* ---- backward ---------------------------------------------------------- */

typedef struct {
    const void* q; const void* k; const void* v; const void* dout; int dt;
    int64_t BH, Nq, Nk; int d; double scale; int causal;
    double* dq; double* dk; double* dv;
    int64_t next;
    int err;
} bwd_job_t;

/* One (batch, head) per work item: its dK and dV accumulate over all rows. */
static void* bwd_worker(void* arg) {
    bwd_job_t* jb = (bwd_job_t*)arg;
    const int d = jb->d;
    const int64_t Nq = jb->Nq, Nk = jb->Nk;
    double* kk = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1) * d);
    double* vv = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1) * d);
    double* s = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    double* dp = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
    double* qr = (double*)malloc(sizeof(double) * d);
    double* gr = (double*)malloc(sizeof(double) * d);
    double* o = (double*)malloc(sizeof(double) * d);
    if (!kk || !vv || !s || !dp || !qr || !gr || !o) {
        __atomic_store_n(&jb->err, OR_NO_MEM, __ATOMIC_RELAXED);
        free(kk); free(vv); free(s); free(dp); free(qr); free(gr); free(o);
        return NULL;
    }
    for (;;) {
        int64_t bh = __atomic_fetch_add(&jb->next, 1, __ATOMIC_RELAXED);
        if (bh >= jb->BH) break;
        int64_t i, j;
        int c;
        load_row(jb->k, jb->dt, bh * Nk * d, (int)(Nk * d), 1.0, kk);
        load_row(jb->v, jb->dt, bh * Nk * d, (int)(Nk * d), 1.0, vv);
        double* dK = jb->dk + bh * Nk * d;
        double* dV = jb->dv + bh * Nk * d;
        for (j = 0; j < Nk * d; ++j) { dK[j] = 0.0; dV[j] = 0.0; }
        for (i = 0; i < Nq; ++i) {
            double* dQ = jb->dq + (bh * Nq + i) * d;
            for (c = 0; c < d; ++c) dQ[c] = 0.0;
            int64_t n = Nk;
            if (jb->causal) {
                n = i + (Nk - Nq) + 1; /* bottom-right aligned */
                if (n < 0) n = 0;
                if (n > Nk) n = Nk;
            }
            if (n == 0) continue;
            load_row(jb->q, jb->dt, (bh * Nq + i) * d, d, 1.0, qr);
            load_row(jb->dout, jb->dt, (bh * Nq + i) * d, d, 1.0, gr);
            /* forward for the row: scores, max, denominator, probabilities, o */
            double m = -INFINITY;
            for (j = 0; j < n; ++j) {
                double acc = 0.0;
                for (c = 0; c < d; ++c) acc += qr[c] * kk[j * d + c];
                s[j] = jb->scale * acc;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (j = 0; j < n; ++j) l += exp(s[j] - m);
            for (c = 0; c < d; ++c) o[c] = 0.0;
            for (j = 0; j < n; ++j) {
                s[j] = exp(s[j] - m) / l; /* s now holds p_ij */
                for (c = 0; c < d; ++c) o[c] += s[j] * vv[j * d + c];
            }
            /* D_i = dO_i . o_i, dP_ij = dO_i . v_j */
            double D = 0.0;
            for (c = 0; c < d; ++c) D += gr[c] * o[c];
            for (j = 0; j < n; ++j) {
                double acc = 0.0;
                for (c = 0; c < d; ++c) acc += gr[c] * vv[j * d + c];
                dp[j] = acc;
            }
            for (j = 0; j < n; ++j) {
                const double p = s[j];
                const double ds = p * (dp[j] - D);
                for (c = 0; c < d; ++c) {
                    dV[j * d + c] += p * gr[c];
                    dQ[c] += jb->scale * ds * kk[j * d + c];
                    dK[j * d + c] += jb->scale * ds * qr[c];
                }
            }
        }
    }
    free(kk); free(vv); free(s); free(dp); free(qr); free(gr); free(o);
    return NULL;
}

/* Gradients of dense attention with respect to q, k, v for the upstream
 * gradient dout.  q, dout: [BH, Nq, d]; k, v: [BH, Nk, d]; all of element
 * type dt.  dq: [BH, Nq, d], dk, dv: [BH, Nk, d] float64.  Rows with no
 * visible key have zero gradients. */
int oracle_attention_bwd(const void* q, const void* k, const void* v, const void* dout, int dt,
                         int64_t BH, int64_t Nq, int64_t Nk, int d, double scale, int causal,
                         double* dq, double* dk, double* dv, int nthreads) {
    if (!q || !k || !v || !dout || !dq || !dk || !dv || !dtype_ok(dt)) return OR_BAD_ARG;
    if (BH < 0 || Nq < 0 || Nk < 0 || d < 1 || d > 4096 || Nk * d > 0x7fffffffLL) return OR_BAD_ARG;
    bwd_job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.q = q; jb.k = k; jb.v = v; jb.dout = dout; jb.dt = dt;
    jb.BH = BH; jb.Nq = Nq; jb.Nk = Nk; jb.d = d; jb.scale = scale; jb.causal = causal;
    jb.dq = dq; jb.dk = dk; jb.dv = dv;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if ((int64_t)nthreads > BH) nthreads = BH > 0 ? (int)BH : 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
    if (!th) return OR_NO_MEM;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, bwd_worker, &jb) != 0) break;
        ++started;
    }
    if (started == 0) bwd_worker(&jb);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(th);
    return jb.err;
}
