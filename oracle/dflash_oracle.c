/*
 * dflash_oracle.c -- plain, slow, fp64 CPU reference for DFlash block attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or load
 * this file: only the tests, the package smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header or constant with the CUDA
 * library; it is written from the definition of the operation alone.
 *
 * What it computes (the plain definition of exact attention, no tiling):
 *
 *   Each request b contributes a block of T = 1 + num_speculative_tokens
 *   queries ("num_query_per_req = 1 + num_speculative_tokens",
 *   kenforever1 "dflash-gemma4-31b-notes", section "why non-causal attention").
 *   The block's own keys are the last T of the L_b = seq_lens[b] keys, so block
 *   query i sits at absolute position p_i = L_b - T + i.
 *
 *   For query head h the key/value head is g = h / (Hq / Hkv) (consecutive
 *   query heads share one KV head).
 *
 *   Visible keys of query i:
 *     causal = 0 (default, "DFlash verify/block attention needs causal=False",
 *                 same page, PR #52 table): every key up to L_b - 1, so every
 *                 block query sees every block key;
 *     causal = 1 ("query i only sees itself and its left", same page, section
 *                 "why non-causal attention"; switch of vLLM PR #43445
 *                 "Allow causal DFlash"): keys up to p_i;
 *     window W > 0 (sliding-window layers, "dflash-gemma4-31b-notes" section on
 *                 Gemma 4 hybrid attention): additionally keys >= p_i - W + 1.
 *
 *   Key j lives in physical page page_table[b][j / P_s], slot j % P_s.
 *
 *   s_j = scale * <q, k_j>;  m = max s_j;  Z = sum exp(s_j - m)
 *   out = sum exp(s_j - m) v_j / Z;  lse = m + log Z   (natural log)
 *
 *   Split-KV: the same loop restricted to a chunk [kb, ke) of key positions
 *   gives a partial (o_c, lse_c); a chunk with no visible key has lse_c = -inf
 *   and o_c = 0. The combine ("split-KV combine", prhub report on vLLM PR
 *   #52816 "DFlash2", review highlights) is
 *     m* = max_c lse_c, w_c = exp(lse_c - m*), out = sum w_c o_c / sum w_c,
 *     lse = m* + log sum w_c.
 *
 * Layouts (all row-major, element strides):
 *   q        [B*T, Hq, D]
 *   q, k_cache, v_cache hold either fp32 values (in_dtype 0) or raw bf16 bit
 *   patterns (in_dtype 1, uint16); a bf16 value is widened exactly to fp32 by
 *   placing its 16 bits in the high half of a 32-bit word.
 *   k_cache  element (page, slot, head, d) at page*sp + slot*ss + head*sh + d
 *   v_cache  same layout as k_cache
 *   page_table [B, max_pages] int32, seq_lens [B] int32
 *   out      [B*T, Hq, D] double, lse [B*T, Hq] double
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const void* q;
    const void* k;
    const void* v;
    int32_t in_dtype; /* 0 = fp32, 1 = bf16 bit patterns */
    const int32_t* page_table;
    const int32_t* seq_lens;
    int32_t B, T, Hq, Hkv, D, page_size, num_pages, max_pages;
    int64_t sp, ss, sh;
    int32_t causal, window;
    double scale;
    int32_t kb, ke; /* chunk of key positions; ke < 0 means no restriction */
    double* out;
    double* lse;
    /* optional row list: triples (b, h, i); NULL = all rows */
    const int32_t* rows;
    int64_t n_rows;
    int32_t status;
    /* work distribution */
    int64_t n_items;
    int64_t next;
    pthread_mutex_t lock;
} oracle_job;

/* Element idx of an input array, exactly widened to double. */
static double elem(const void* base, int64_t idx, int32_t in_dtype)
{
    if (in_dtype == 1) {
        const uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof(f));
        return (double)f;
    }
    return (double)((const float*)base)[idx];
}

/* Returns 0 on success, a negative code when a page id is out of range. */
static int one_row(oracle_job* J, int32_t b, int32_t h, int32_t i, double* o, double* lse_out)
{
    const int32_t T = J->T, D = J->D, G = J->Hq / J->Hkv;
    const int32_t g = h / G;
    const int32_t L = J->seq_lens[b];
    const int64_t p = (int64_t)L - T + i;
    int64_t hi = J->causal ? p : (int64_t)L - 1;
    int64_t lo = 0;
    if (J->window > 0) {
        lo = p - J->window + 1;
        if (lo < 0) lo = 0;
    }
    if (J->ke >= 0) {
        if (lo < J->kb) lo = J->kb;
        if (hi > (int64_t)J->ke - 1) hi = (int64_t)J->ke - 1;
    }
    const int64_t qoff = (((int64_t)b * T + i) * J->Hq + h) * D;
    for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
    if (hi < lo) {
        *lse_out = -INFINITY;
        return 0;
    }
    const int64_t n = hi - lo + 1;
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    int64_t* voffs = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
    if (!s || !voffs) {
        free(s);
        free(voffs);
        return -2;
    }
    /* pass 1: scores */
    double m = -INFINITY;
    for (int64_t j = lo; j <= hi; ++j) {
        const int32_t page = J->page_table[(int64_t)b * J->max_pages + j / J->page_size];
        if (page < 0 || page >= J->num_pages) {
            free(s);
            free(voffs);
            return -1;
        }
        const int64_t off = (int64_t)page * J->sp + (j % J->page_size) * J->ss + (int64_t)g * J->sh;
        double acc = 0.0;
        for (int32_t d = 0; d < D; ++d)
            acc += elem(J->q, qoff + d, J->in_dtype) * elem(J->k, off + d, J->in_dtype);
        acc *= J->scale;
        s[j - lo] = acc;
        voffs[j - lo] = off;
        if (acc > m) m = acc;
    }
    /* pass 2: normaliser and weighted sum of values */
    double Z = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        const double e = exp(s[t] - m);
        Z += e;
        for (int32_t d = 0; d < D; ++d) o[d] += e * elem(J->v, voffs[t] + d, J->in_dtype);
    }
    for (int32_t d = 0; d < D; ++d) o[d] /= Z;
    *lse_out = m + log(Z);
    free(s);
    free(voffs);
    return 0;
}

static void* worker(void* arg)
{
    oracle_job* J = (oracle_job*)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t item = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (item >= J->n_items) break;
        int32_t b, h, i;
        double *o, *l;
        if (J->rows) {
            b = J->rows[3 * item + 0];
            h = J->rows[3 * item + 1];
            i = J->rows[3 * item + 2];
            o = J->out + item * J->D;
            l = J->lse + item;
        } else {
            /* item enumerates (b, i, h) in output order */
            h = (int32_t)(item % J->Hq);
            const int64_t bi = item / J->Hq;
            i = (int32_t)(bi % J->T);
            b = (int32_t)(bi / J->T);
            o = J->out + item * J->D;
            l = J->lse + item;
        }
        const int rc = one_row(J, b, h, i, o, l);
        if (rc != 0) {
            pthread_mutex_lock(&J->lock);
            J->status = rc;
            pthread_mutex_unlock(&J->lock);
        }
    }
    return NULL;
}

static int run_job(oracle_job* J, int32_t num_threads)
{
    if (J->Hkv <= 0 || J->Hq % J->Hkv != 0 || J->T <= 0 || J->D <= 0 || J->page_size <= 0) return -3;
    for (int32_t b = 0; b < J->B; ++b) {
        const int32_t L = J->seq_lens[b];
        if (L < J->T || (int64_t)(L + J->page_size - 1) / J->page_size > J->max_pages) return -4;
    }
    J->status = 0;
    J->next = 0;
    pthread_mutex_init(&J->lock, NULL);
    if (num_threads < 1) num_threads = 1;
    if (num_threads > 256) num_threads = 256;
    pthread_t tids[256];
    int started = 0;
    for (int t = 1; t < num_threads; ++t) {
        if (pthread_create(&tids[started], NULL, worker, J) == 0) ++started;
    }
    worker(J);
    for (int t = 0; t < started; ++t) pthread_join(tids[t], NULL);
    pthread_mutex_destroy(&J->lock);
    return J->status;
}

/* Full block attention (or one key chunk of it when ke >= 0) for every output row. */
int oracle_block_attn(const void* q, const void* k_cache, const void* v_cache, int32_t in_dtype,
                      const int32_t* page_table, const int32_t* seq_lens,
                      int32_t B, int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                      int32_t page_size, int32_t num_pages, int32_t max_pages,
                      int64_t stride_page, int64_t stride_slot, int64_t stride_head,
                      int32_t causal, int32_t window, double scale,
                      int32_t kb, int32_t ke,
                      double* out, double* lse, int32_t num_threads)
{
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k_cache; J.v = v_cache; J.in_dtype = in_dtype;
    J.page_table = page_table; J.seq_lens = seq_lens;
    J.B = B; J.T = T; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.page_size = page_size; J.num_pages = num_pages; J.max_pages = max_pages;
    J.sp = stride_page; J.ss = stride_slot; J.sh = stride_head;
    J.causal = causal; J.window = window; J.scale = scale;
    J.kb = kb; J.ke = ke;
    J.out = out; J.lse = lse;
    J.rows = NULL;
    J.n_items = (int64_t)B * T * Hq;
    return run_job(&J, num_threads);
}

/* Same definition, evaluated only for the listed (b, h, i) rows; row r of out/lse
   holds the result for triple r. Used to check sampled outputs of large cases. */
int oracle_block_attn_rows(const void* q, const void* k_cache, const void* v_cache, int32_t in_dtype,
                           const int32_t* page_table, const int32_t* seq_lens,
                           int32_t B, int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                           int32_t page_size, int32_t num_pages, int32_t max_pages,
                           int64_t stride_page, int64_t stride_slot, int64_t stride_head,
                           int32_t causal, int32_t window, double scale,
                           const int32_t* rows, int64_t n_rows,
                           double* out, double* lse, int32_t num_threads)
{
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k_cache; J.v = v_cache; J.in_dtype = in_dtype;
    J.page_table = page_table; J.seq_lens = seq_lens;
    J.B = B; J.T = T; J.Hq = Hq; J.Hkv = Hkv; J.D = D;
    J.page_size = page_size; J.num_pages = num_pages; J.max_pages = max_pages;
    J.sp = stride_page; J.ss = stride_slot; J.sh = stride_head;
    J.causal = causal; J.window = window; J.scale = scale;
    J.kb = 0; J.ke = -1;
    J.out = out; J.lse = lse;
    for (int64_t r = 0; r < n_rows; ++r) {
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 || rows[3 * r + 1] >= Hq ||
            rows[3 * r + 2] < 0 || rows[3 * r + 2] >= T)
            return -5;
    }
    J.rows = rows;
    J.n_items = n_rows;
    return run_job(&J, num_threads);
}

/* Log-sum-exp combine of S partial results: partial_out [S, N, D], partial_lse [S, N]
   -> out [N, D], lse [N]. Chunks with lse = -inf carry weight zero. */
int oracle_split_combine(const double* partial_out, const double* partial_lse,
                         int32_t S, int64_t N, int32_t D, double* out, double* lse)
{
    for (int64_t n = 0; n < N; ++n) {
        double m = -INFINITY;
        for (int32_t c = 0; c < S; ++c) {
            const double l = partial_lse[(int64_t)c * N + n];
            if (l > m) m = l;
        }
        double* o = out + n * D;
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        if (m == -INFINITY) {
            lse[n] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int32_t c = 0; c < S; ++c) {
            const double l = partial_lse[(int64_t)c * N + n];
            if (l == -INFINITY) continue;
            const double w = exp(l - m);
            wsum += w;
            const double* po = partial_out + ((int64_t)c * N + n) * D;
            for (int32_t d = 0; d < D; ++d) o[d] += w * po[d];
        }
        for (int32_t d = 0; d < D; ++d) o[d] /= wsum;
        lse[n] = m + log(wsum);
    }
    return 0;
}
