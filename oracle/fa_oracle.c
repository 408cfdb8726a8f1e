/*
 * fa_oracle.c -- plain, slow, fp64 CPU oracle for decode-step attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this code:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (the plain definition the method converges to):
 *   for every sequence b and query head h, with kv = h / (Hq / Hkv),
 *   L = seq_lens[b], lo = (W > 0 && L > W) ? L - W : 0,
 *     s_t = scale * sum_d q[b,h,d] * K_b[kv,t,d]          for t in [lo, L)
 *     p_t = exp(s_t - max s) / sum_u exp(s_u - max s)
 *     out[b,h,:] = sum_t p_t * V_b[kv,t,:]
 *   and a zero row when the range is empty.
 *
 * Sources (the mlx-native page "flash_attn_vec_hybrid.metal"):
 *   - head map kv_head = head / (n_heads / n_kv_heads): "GQA: map query head
 *     to KV head" in flash_attn_vec_hybrid_impl;
 *   - the sliding-window rule (keys with logical index < kv_seq_len - window
 *     are masked, window 0 = global) and the length mask: the mask block of
 *     the same kernel;
 *   - softmax(q K^T * scale) V is what the kernel's online softmax (running
 *     M and S, "Online softmax" block) and its cross-simdgroup / cross-
 *     workgroup merge reach in exact arithmetic, so the oracle evaluates the
 *     definition instead of that algorithm;
 *   - an empty range gives 0 ("S == 0 ? 0" in the output write).
 *   The cache append (oracle_append_kv, at the end) writes one step's K and V
 *   rows at each sequence's position.
 *   A slot map (oracle_fa_decode_slots, oracle_append_kv_slots) lets row b
 *   use cache slot slot_ids[b] of a pool of per-slot caches, as the batched
 *   kernels of the same page read slot_id_arr per query row.
 *   The int8 V codec (int8 codes times one fp16 scale per 32 elements) follows
 *   ggml's block_q8_0 dequantisation (qs[i] * d) shown on the DS4Server page
 *   "dsv4_hc.metal"; the quantiser itself (amax / 127, round half to even,
 *   clamp to +-127) is not on the pages and is the plain symmetric reading.
 *
 * Everything is evaluated in double, in ascending key order, one (b, h) row
 * per work item; rows are spread over POSIX threads.  Build with
 * -ffp-contract=off so no fused multiply-add changes the rounding.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------- IEEE binary16 <-> double (exact decode, RN encode) ------ */

double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);   /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even. */
uint16_t oracle_double_to_half(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (isnan(x))
        return 0x7E00;
    if (ax >= 65520.0)                 /* 65504 + half an ulp rounds up to inf */
        return sign | 0x7C00;
    if (ax == 0.0)
        return sign;
    int e2;
    frexp(ax, &e2);                    /* ax = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;                    /* unbiased exponent of ax */
    if (E < -14)
        E = -14;                       /* subnormal range keeps spacing 2^-24 */
    double ulp = ldexp(1.0, E - 10);
    double r = rint(ax / ulp) * ulp;   /* ax/ulp is exact; rint = ties-to-even */
    if (r == 0.0)
        return sign;
    if (r < ldexp(1.0, -14))
        return sign | (uint16_t)(r / ldexp(1.0, -24));
    frexp(r, &e2);
    E = e2 - 1;
    uint16_t mant = (uint16_t)((r / ldexp(1.0, E) - 1.0) * 1024.0);
    return sign | (uint16_t)((E + 15) << 10) | mant;
}

/* ---------------- int8 V packer (block of 32 along head_dim) -------------- */

/* x: [n_rows][D] fp32, D % 32 == 0.  codes: [n_rows][D] int8,
 * scales: [n_rows][D/32] binary16 bits.  Returns 0, or -1 on bad D. */
int oracle_pack_v_int8(const float *x, long long n_rows, int D, int8_t *codes,
                       uint16_t *scales)
{
    if (D <= 0 || D % 32)
        return -1;
    for (long long r = 0; r < n_rows; ++r) {
        for (int blk = 0; blk < D / 32; ++blk) {
            const float *xb = x + r * D + blk * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs((double)xb[i]);
                if (a > amax)
                    amax = a;
            }
            uint16_t sh = oracle_double_to_half(amax / 127.0);
            double s = oracle_half_to_double(sh);
            scales[r * (D / 32) + blk] = sh;
            for (int i = 0; i < 32; ++i) {
                double qv = 0.0;
                if (s != 0.0) {
                    qv = rint((double)xb[i] / s);
                    if (qv > 127.0)
                        qv = 127.0;
                    if (qv < -127.0)
                        qv = -127.0;
                }
                codes[r * D + blk * 32 + i] = (int8_t)qv;
            }
        }
    }
    return 0;
}

/* ---------------- cache addressing -------------------------------------- */

typedef struct {
    const uint16_t *q;         /* [B][Hq][D] binary16 */
    const uint16_t *k;         /* cache, binary16 */
    const void *v;             /* cache, binary16 or int8 */
    const uint16_t *v_scales;  /* NULL => V is binary16 */
    const int32_t *block_table;/* NULL => contiguous [B][Hkv][cap][D] */
    const int32_t *seq_lens;
    const int32_t *window;     /* NULL => all global */
    int B, Hq, Hkv, D, page_size, max_blocks;
    double scale;
    int ring;                  /* contiguous ring cache: token t at row t % capacity */
    int tq;                    /* queries per sequence (q is [B][tq][Hq][D]); 0 or 1 = one */
    const int32_t *slot_ids;   /* contiguous only: row b's cache is slot slot_ids[b] of
                                  [n_slots][Hkv][cap][D]; NULL => slot b */
    int n_slots;
} oracle_problem;

/* Cache slot of row b, or -1 when its slot id names no slot. */
static long long slot_of(const oracle_problem *P, int b)
{
    if (!P->slot_ids)
        return b;
    long long s = P->slot_ids[b];
    return (s >= 0 && s < P->n_slots) ? s : -1;
}

/* Element offset of row (b, kv, t) in a cache whose rows hold `row_elems`. */
static long long row_offset(const oracle_problem *P, int b, int kv, int t,
                            int row_elems)
{
    if (P->block_table) {
        long long blk = P->block_table[(long long)b * P->max_blocks + t / P->page_size];
        int r = t % P->page_size;
        return ((blk * P->Hkv + kv) * P->page_size + r) * (long long)row_elems;
    }
    /* contiguous: capacity (tokens) = max_blocks; a ring cache keeps token t
     * at row t % capacity */
    long long r = P->ring ? t % P->max_blocks : t;
    return ((slot_of(P, b) * P->Hkv + kv) * P->max_blocks + r) * (long long)row_elems;
}

static double v_elem(const oracle_problem *P, int b, int kv, int t, int d)
{
    if (!P->v_scales) {
        const uint16_t *v = (const uint16_t *)P->v;
        return oracle_half_to_double(v[row_offset(P, b, kv, t, P->D) + d]);
    }
    const int8_t *v = (const int8_t *)P->v;
    double code = (double)v[row_offset(P, b, kv, t, P->D) + d];
    double s = oracle_half_to_double(
        P->v_scales[row_offset(P, b, kv, t, P->D / 32) + d / 32]);
    return code * s;
}

/* Attended keys [lo, hi) of query j of sequence b.  With tq queries the
 * sequence's last tq tokens are the queries; query j sits at position
 * L - tq + j and sees the keys up to and including itself (the causal rule
 * of the tessl page's flash_attn_rows; window 0 = global).  One query: the
 * whole length. */
static void attended_range(const oracle_problem *P, int b, int j, int *lo, int *hi)
{
    int L = P->seq_lens[b];
    int W = P->window ? P->window[b] : 0;
    int tq = P->tq > 1 ? P->tq : 1;
    int end = L - (tq - 1 - j);
    if (end < 0)
        end = 0;
    *hi = end;
    *lo = (W > 0 && end > W) ? end - W : 0;
    /* a ring cache holds only the last `capacity` tokens (the pages' live
     * length min(seq_pos + 1, capacity) of the ring storage mode) */
    if (P->ring && *hi - P->max_blocks > *lo)
        *lo = *hi - P->max_blocks;
    /* a slot id that names no slot: no cache, an empty range */
    if (slot_of(P, b) < 0)
        *lo = *hi = 0;
}

/* Softmax weights p_t, t in [lo, hi), of row (b, h).  p must hold hi-lo. */
static void row_weights(const oracle_problem *P, int b, int j, int h, int lo, int hi,
                        double *p)
{
    int kv = h / (P->Hq / P->Hkv);
    int tq = P->tq > 1 ? P->tq : 1;
    const uint16_t *qrow = P->q + (((long long)b * tq + j) * P->Hq + h) * P->D;
    double smax = -INFINITY;
    for (int t = lo; t < hi; ++t) {
        const uint16_t *krow = P->k + row_offset(P, b, kv, t, P->D);
        double dot = 0.0;
        for (int d = 0; d < P->D; ++d)
            dot += oracle_half_to_double(qrow[d]) * oracle_half_to_double(krow[d]);
        double s = P->scale * dot;
        p[t - lo] = s;
        if (s > smax)
            smax = s;
    }
    double z = 0.0;
    for (int t = lo; t < hi; ++t) {
        p[t - lo] = exp(p[t - lo] - smax);
        z += p[t - lo];
    }
    for (int t = lo; t < hi; ++t)
        p[t - lo] /= z;
}

static void row_output(const oracle_problem *P, int b, int j, int h, double *out)
{
    int lo, hi;
    attended_range(P, b, j, &lo, &hi);
    for (int d = 0; d < P->D; ++d)
        out[d] = 0.0;
    if (hi <= lo)
        return;
    int kv = h / (P->Hq / P->Hkv);
    double *p = (double *)malloc(sizeof(double) * (size_t)(hi - lo));
    row_weights(P, b, j, h, lo, hi, p);
    for (int t = lo; t < hi; ++t)
        for (int d = 0; d < P->D; ++d)
            out[d] += p[t - lo] * v_elem(P, b, kv, t, d);
    free(p);
}

/* ---------------- threaded driver --------------------------------------- */

typedef struct {
    const oracle_problem *P;
    const int32_t *rows;      /* NULL => rows 0..n_rows-1 */
    int n_rows;
    double *out;              /* [n_rows][D] */
    int next;                 /* shared work counter */
    pthread_mutex_t mu;
} oracle_job;

static void *worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int i = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (i >= J->n_rows)
            break;
        /* row = (b * tq + j) * Hq + h */
        int row = J->rows ? J->rows[i] : i;
        int tq = J->P->tq > 1 ? J->P->tq : 1;
        int bj = row / J->P->Hq;
        row_output(J->P, bj / tq, bj % tq, row % J->P->Hq, J->out + (long long)i * J->P->D);
    }
    return NULL;
}

static int validate(const oracle_problem *P)
{
    if (!P->q || !P->k || !P->v || !P->seq_lens)
        return -1;
    if (P->B < 0 || P->Hq <= 0 || P->Hkv <= 0 || P->Hq % P->Hkv || P->D <= 0)
        return -3;
    if (P->v_scales && P->D % 32)
        return -2;
    if (P->block_table && P->page_size <= 0)
        return -6;
    long long cap = P->block_table ? (long long)P->max_blocks * P->page_size
                                   : (long long)P->max_blocks;
    if (P->ring && (P->block_table || P->max_blocks <= 0))
        return -6;
    if (P->slot_ids && (P->block_table || P->n_slots <= 0 || P->max_blocks <= 0))
        return -6;
    for (int b = 0; b < P->B; ++b)
        if (P->seq_lens[b] < 0 || (!P->ring && P->seq_lens[b] > cap))
            return -6;
    return 0;
}

/*
 * Attention output for the (b, h) rows listed in `rows` (row = b*Hq + h), or
 * for all B*Hq rows when rows == NULL.  out: [n_rows][D] double.
 * n_threads <= 0 uses every online core.  Returns 0 or a negative code.
 */
static int decode_impl(const oracle_problem *Pin, const int32_t *rows, int n_rows, int n_threads,
                       double *out);

int oracle_fa_decode(const uint16_t *q, const uint16_t *k_cache, const void *v_cache,
                     const uint16_t *v_scales, const int32_t *block_table,
                     const int32_t *seq_lens, const int32_t *window, int B, int Hq,
                     int Hkv, int D, int page_size, int max_blocks, double scale,
                     const int32_t *rows, int n_rows, int n_threads, double *out)
{
    oracle_problem P = {q, k_cache, v_cache, v_scales, block_table, seq_lens, window,
                        B, Hq, Hkv, D, page_size, max_blocks, scale, 0, 1};
    return decode_impl(&P, rows, n_rows, n_threads, out);
}

/*
 * Multi-query decode (speculative verify): q [B][tq][Hq][D] holds the last
 * tq tokens of each sequence, all already in the cache; query j attends the
 * keys up to its own position L - tq + j (window counted back from there).
 * out: [B][tq][Hq][D] (or the listed rows, row = (b*tq + j)*Hq + h).
 * tq = 1 is oracle_fa_decode.
 */
int oracle_fa_decode_multi(const uint16_t *q, const uint16_t *k_cache, const void *v_cache,
                           const uint16_t *v_scales, const int32_t *block_table,
                           const int32_t *seq_lens, const int32_t *window, int B, int tq, int Hq,
                           int Hkv, int D, int page_size, int max_blocks, double scale,
                           const int32_t *rows, int n_rows, int n_threads, double *out)
{
    if (tq <= 0)
        return -6;
    oracle_problem P = {q, k_cache, v_cache, v_scales, block_table, seq_lens, window,
                        B, Hq, Hkv, D, page_size, max_blocks, scale, 0, tq};
    return decode_impl(&P, rows, n_rows, n_threads, out);
}

/*
 * Ring cache: contiguous [B][Hkv][capacity][D] storage in which token t of a
 * sequence lives at row t % capacity; seq_lens counts every token seen (it
 * may exceed capacity) and only the last `capacity` of them are attended
 * (the ring storage mode of flash_attn_vec_hybrid_batched on the mlx-native
 * page: live length min(seq_pos + 1, capacity), rows remapped by ring_start).
 * The window rule applies on top.
 */
int oracle_fa_decode_ring(const uint16_t *q, const uint16_t *k_cache, const void *v_cache,
                          const uint16_t *v_scales, const int32_t *seq_lens,
                          const int32_t *window, int B, int Hq, int Hkv, int D, int capacity,
                          double scale, const int32_t *rows, int n_rows, int n_threads,
                          double *out)
{
    oracle_problem P = {q, k_cache, v_cache, v_scales, NULL, seq_lens, window,
                        B, Hq, Hkv, D, 1, capacity, scale, 1, 1};
    return decode_impl(&P, rows, n_rows, n_threads, out);
}

/*
 * Decode over a pool of per-slot caches addressed through a slot map: the
 * batched kernels of the mlx-native page read, per query row, the row's cache
 * slot (slot_id_arr) and position (seq_pos_arr) on the device, and address
 * the K/V rows of that slot in a [slots][n_kv_heads][capacity][head_dim]
 * pool.  Here row b of q, seq_lens, window and out uses slot slot_ids[b] of
 * k_cache / v_cache / v_scales [n_slots][Hkv][capacity][...]; seq_lens[b] is
 * that slot's length (the page's seq_pos + 1).  ring = 0: plain contiguous
 * slots (seq_lens[b] <= capacity); ring = 1: each slot a ring as in
 * oracle_fa_decode_ring.  A slot id outside [0, n_slots) gives a zero row.
 */
int oracle_fa_decode_slots(const uint16_t *q, const uint16_t *k_cache, const void *v_cache,
                           const uint16_t *v_scales, const int32_t *slot_ids, int n_slots,
                           const int32_t *seq_lens, const int32_t *window, int B, int Hq,
                           int Hkv, int D, int capacity, int ring, double scale,
                           const int32_t *rows, int n_rows, int n_threads, double *out)
{
    if (!slot_ids)
        return -1;
    oracle_problem P = {q, k_cache, v_cache, v_scales, NULL, seq_lens, window,
                        B, Hq, Hkv, D, 1, capacity, scale, ring ? 1 : 0, 1, slot_ids, n_slots};
    return decode_impl(&P, rows, n_rows, n_threads, out);
}

static int decode_impl(const oracle_problem *Pin, const int32_t *rows, int n_rows, int n_threads,
                       double *out)
{
    oracle_problem P = *Pin;
    int rc = validate(&P);
    if (rc)
        return rc;
    if (!rows)
        n_rows = P.B * (P.tq > 1 ? P.tq : 1) * P.Hq;
    if (n_threads <= 0)
        n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads > n_rows)
        n_threads = n_rows > 0 ? n_rows : 1;
    oracle_job J;
    J.P = &P;
    J.rows = rows;
    J.n_rows = n_rows;
    J.out = out;
    J.next = 0;
    pthread_mutex_init(&J.mu, NULL);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int i = 0; i < n_threads; ++i)
        pthread_create(&th[i], NULL, worker, &J);
    for (int i = 0; i < n_threads; ++i)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
    return 0;
}

/* Softmax weights of one row over its attended range; p: [hi - lo].
 * Writes the range to *lo_out / *hi_out.  Returns 0 or a negative code. */
int oracle_fa_weights(const uint16_t *q, const uint16_t *k_cache,
                      const int32_t *block_table, const int32_t *seq_lens,
                      const int32_t *window, int B, int Hq, int Hkv, int D,
                      int page_size, int max_blocks, double scale, int b, int h,
                      double *p, int *lo_out, int *hi_out)
{
    oracle_problem P = {q, k_cache, k_cache, NULL, block_table, seq_lens, window,
                        B, Hq, Hkv, D, page_size, max_blocks, scale, 0, 1};
    int rc = validate(&P);
    if (rc)
        return rc;
    int lo, hi;
    attended_range(&P, b, 0, &lo, &hi);
    *lo_out = lo;
    *hi_out = hi;
    if (hi > lo)
        row_weights(&P, b, 0, h, lo, hi, p);
    return 0;
}

/*
 * Gather sequence b's cache rows through the block table into a dense
 * [Hkv][n_tokens][row_bytes] byte buffer (row_bytes = D*2 for K or fp16 V,
 * D for int8 V, (D/32)*2 for the scales).  block_table == NULL reads the
 * contiguous [B][Hkv][max_blocks][...] layout (capacity = max_blocks tokens).  A byte copy: the result is the
 * exact bytes the cache holds.  Returns 0 or -1 on a bad argument.
 */
int oracle_gather_rows(const void *cache, int row_bytes, const int32_t *block_table,
                       int b, int Hkv, int page_size, int max_blocks, int n_tokens,
                       void *dense)
{
    long long cap = block_table ? (long long)max_blocks * page_size : (long long)max_blocks;
    if (!cache || !dense || row_bytes <= 0 || (block_table && page_size <= 0) ||
        n_tokens < 0 || n_tokens > cap)
        return -1;
    const uint8_t *src = (const uint8_t *)cache;
    uint8_t *dst = (uint8_t *)dense;
    for (int kv = 0; kv < Hkv; ++kv)
        for (int t = 0; t < n_tokens; ++t) {
            long long blk = block_table ? block_table[(long long)b * max_blocks + t / page_size]
                                        : -1;
            long long off;
            if (block_table)
                off = ((blk * Hkv + kv) * page_size + t % page_size) * (long long)row_bytes;
            else
                off = (((long long)b * Hkv + kv) * max_blocks + t) * (long long)row_bytes;
            memcpy(dst + ((long long)kv * n_tokens + t) * row_bytes, src + off,
                   (size_t)row_bytes);
        }
    return 0;
}

/*
 * Cache append: write this step's K and V rows into the cache at each
 * sequence's device-side position (the per-step "copy K f32 -> f16 into the
 * cache at cache_pos" of the hf2q page "batched_body.rs", and tessl's
 * kv_store_timestep on the "nn.rs" page, whose out-of-range offset makes the
 * store a no-op).
 *   k_new, v_new: [B][Hkv][D] fp32.
 *   K row <- fp16 round-to-nearest-even of k_new; V row <- the same for an
 *   fp16 V cache, or the int8 codec above (codes + per-32 scales).
 *   A position outside [0, capacity) or a block id outside [0, num_blocks)
 *   leaves that row untouched.
 * Returns 0, or a negative code for a bad argument.
 */
static int append_impl(const float *k_new, const float *v_new, uint16_t *k_cache, void *v_cache,
                       uint16_t *v_scales, const int32_t *block_table, const int32_t *positions,
                       int B, int Hkv, int D, int page_size, int max_blocks, int num_blocks,
                       int ring, const int32_t *slot_ids, int n_slots);

int oracle_append_kv(const float *k_new, const float *v_new, uint16_t *k_cache, void *v_cache,
                     uint16_t *v_scales, const int32_t *block_table, const int32_t *positions,
                     int B, int Hkv, int D, int page_size, int max_blocks, int num_blocks)
{
    return append_impl(k_new, v_new, k_cache, v_cache, v_scales, block_table, positions, B, Hkv,
                       D, page_size, max_blocks, num_blocks, 0, NULL, 0);
}

/* Append into a ring cache: token t goes to row t % capacity (t >= 0). */
int oracle_append_kv_ring(const float *k_new, const float *v_new, uint16_t *k_cache,
                          void *v_cache, uint16_t *v_scales, const int32_t *positions, int B,
                          int Hkv, int D, int capacity)
{
    return append_impl(k_new, v_new, k_cache, v_cache, v_scales, NULL, positions, B, Hkv, D, 1,
                       capacity, 0, 1, NULL, 0);
}

/* Append into a pool of per-slot caches [n_slots][Hkv][capacity][...]: row b
 * of k_new / v_new / positions writes slot slot_ids[b] (the slot map of
 * oracle_fa_decode_slots), as a plain contiguous slot (ring = 0) or a ring
 * (ring = 1).  A slot id outside [0, n_slots) writes nothing.  Rows are
 * written in order b = 0, 1, ... */
int oracle_append_kv_slots(const float *k_new, const float *v_new, uint16_t *k_cache,
                           void *v_cache, uint16_t *v_scales, const int32_t *slot_ids,
                           int n_slots, const int32_t *positions, int B, int Hkv, int D,
                           int capacity, int ring)
{
    if (!slot_ids || n_slots <= 0 || capacity <= 0)
        return -6;
    return append_impl(k_new, v_new, k_cache, v_cache, v_scales, NULL, positions, B, Hkv, D, 1,
                       capacity, 0, ring ? 1 : 0, slot_ids, n_slots);
}

static int append_impl(const float *k_new, const float *v_new, uint16_t *k_cache, void *v_cache,
                       uint16_t *v_scales, const int32_t *block_table, const int32_t *positions,
                       int B, int Hkv, int D, int page_size, int max_blocks, int num_blocks,
                       int ring, const int32_t *slot_ids, int n_slots)
{
    if (!k_new || !v_new || !k_cache || !v_cache || !positions || B < 0 || Hkv <= 0 || D <= 0)
        return -1;
    if (v_scales && D % 32)
        return -2;
    if (block_table && page_size <= 0)
        return -6;
    long long cap = block_table ? (long long)max_blocks * page_size : (long long)max_blocks;
    for (int b = 0; b < B; ++b) {
        long long t = positions[b];
        if (t < 0 || (!ring && t >= cap))
            continue;
        if (ring)
            t %= cap;
        long long slot = b;
        if (slot_ids) {
            slot = slot_ids[b];
            if (slot < 0 || slot >= n_slots)
                continue;
        }
        for (int kv = 0; kv < Hkv; ++kv) {
            long long row;
            if (block_table) {
                long long blk = block_table[(long long)b * max_blocks + t / page_size];
                if (blk < 0 || blk >= num_blocks)
                    continue;
                row = (blk * Hkv + kv) * page_size + t % page_size;
            } else {
                row = (slot * Hkv + kv) * max_blocks + t;
            }
            const float *kr = k_new + ((long long)b * Hkv + kv) * D;
            const float *vr = v_new + ((long long)b * Hkv + kv) * D;
            for (int d = 0; d < D; ++d)
                k_cache[row * D + d] = oracle_double_to_half((double)kr[d]);
            if (v_scales) {
                oracle_pack_v_int8(vr, 1, D, (int8_t *)v_cache + row * D, v_scales + row * (D / 32));
            } else {
                uint16_t *vc = (uint16_t *)v_cache;
                for (int d = 0; d < D; ++d)
                    vc[row * D + d] = oracle_double_to_half((double)vr[d]);
            }
        }
    }
    return 0;
}
