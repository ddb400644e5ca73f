/*
 * oracle.c -- plain, slow, fp64 CPU reference for paged KV-cache attention
 * under continuous batching.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file; it shares no code, header or table with the CUDA path.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 *
 * What it computes, and where that comes from:
 *
 *  - The cached "past key values" of every running request
 *    (text-generation-inference Router/Webserver deep dive, xxmr.cn,
 *    section "Prefill, Decode and past key values"): the first pass over a
 *    prompt computes the complete (causal) attention matrix; every later pass
 *    computes attention only for the one new token, against the cached keys
 *    and values.
 *  - The cache is paged: the router's block allocator hands out fixed-size
 *    blocks (TGI architecture wiki, data-sketchers.com, section "The Router";
 *    the v3 call-flow schema adds "paged attention support", section
 *    "Call Flow").  Token p of a sequence lives in physical block
 *    block_table[s][p / B] at offset p % B.
 *  - The attention itself is never written down on the pages; the plainest
 *    reading, used here, is textbook scaled dot-product softmax attention:
 *        out = sum_j softmax_j(scale * <q, k_j>) v_j ,  scale = 1/sqrt(d)
 *    with query head h reading KV head h / (Hq / Hkv) (grouped heads).
 *
 * Every value is converted from bf16 to double exactly; all arithmetic is in
 * double, in the order of the definition (max, exponentials, sum, weighted
 * sum, one division).  Block tables are dereferenced explicitly, token by
 * token.  No blocking, splitting or online rescaling.
 *
 * Pool layout (the library's contract, mirrored here independently):
 *     k_pool[N][Hkv][B][d], v_pool[N][Hkv][B][d]   (bf16, row-major)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_SLOT_RANGE -1
#define OR_ERR_SLOT_DUP -2
#define OR_ERR_BLOCK_RANGE -3
#define OR_ERR_ARG -4
#define OR_ERR_NOMEM -5

static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* KV append: scatter the new tokens' K/V rows into the pool at their slots.  */
/* Pure bit copy.  slot < 0 means "padding, skip".  A slot outside the pool   */
/* or a slot written twice in one call is an error (nothing is written then). */
/* ------------------------------------------------------------------------ */
int oracle_kv_append(int num_tokens, int num_kv_heads, int head_dim,
                     int block_size, int num_blocks,
                     const uint16_t *k_new, const uint16_t *v_new,
                     const int32_t *slot_mapping,
                     uint16_t *k_pool, uint16_t *v_pool) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks <= 0)
        return OR_ERR_ARG;
    long long num_slots = (long long)num_blocks * block_size;
    unsigned char *seen = (unsigned char *)calloc((size_t)num_slots, 1);
    if (!seen) return OR_ERR_NOMEM;
    for (int i = 0; i < num_tokens; ++i) {
        int32_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if ((long long)slot >= num_slots) { free(seen); return OR_ERR_SLOT_RANGE; }
        if (seen[slot]) { free(seen); return OR_ERR_SLOT_DUP; }
        seen[slot] = 1;
    }
    free(seen);
    for (int i = 0; i < num_tokens; ++i) {
        int32_t slot = slot_mapping[i];
        if (slot < 0) continue;
        long long blk = slot / block_size;
        long long off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t dst = (size_t)(((blk * num_kv_heads + h) * block_size + off) * head_dim);
            size_t src = (size_t)(((long long)i * num_kv_heads + h) * head_dim);
            for (int e = 0; e < head_dim; ++e) {
                k_pool[dst + e] = k_new[src + e];
                v_pool[dst + e] = v_new[src + e];
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Expected slot of every new token of a step, from the block table.         */
/* Sequence s owns query rows [q_start[s], q_start[s+1]); after the append   */
/* it holds seq_lens[s] tokens, so its new tokens sit at absolute positions  */
/* seq_lens[s] - n_s + i.  slot = block_table[s][p / B] * B + p % B.         */
/* ------------------------------------------------------------------------ */
int oracle_expected_slots(int num_seqs, const int32_t *q_start,
                          const int32_t *seq_lens, const int32_t *block_table,
                          int max_blocks_per_seq, int block_size,
                          int32_t *slots_out) {
    for (int s = 0; s < num_seqs; ++s) {
        int n = q_start[s + 1] - q_start[s];
        int p0 = seq_lens[s] - n;
        if (n < 0 || p0 < 0) return OR_ERR_ARG;
        for (int i = 0; i < n; ++i) {
            int p = p0 + i;
            int bi = p / block_size;
            if (bi >= max_blocks_per_seq) return OR_ERR_BLOCK_RANGE;
            int32_t blk = block_table[(size_t)s * max_blocks_per_seq + bi];
            if (blk < 0) return OR_ERR_BLOCK_RANGE;
            slots_out[q_start[s] + i] = blk * block_size + p % block_size;
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* One query vector against keys 0..L-1 of one sequence and one KV head,     */
/* read through the block table.  The definition, term by term:              */
/*   x_j = scale * sum_e q_e k_{j,e};  M = max_j x_j;  w_j = exp(x_j - M);    */
/*   out_e = (sum_j w_j v_{j,e}) / (sum_j w_j).   L == 0 gives zeros.         */
/* ------------------------------------------------------------------------ */
typedef struct {
    int num_kv_heads, head_dim, block_size, num_blocks;
    const uint16_t *k_pool, *v_pool;  /* bf16 pools, or NULL with ... */
    const uint8_t *k8, *v8;           /* ... fp8 e4m3 code pools and */
    const float *k_scale, *v_scale;   /* one scale per KV head */
} pool_view;

static double e4m3_to_double(uint8_t c);

/* Element e of row (blk, g, off) of the K (which = 0) or V pool, as a double:
 * a bf16 value, or an fp8 code times its KV head's scale. */
static double pool_elem(const pool_view *pv, int which, size_t row, int g, int e) {
    const size_t at = row * (size_t)pv->head_dim + (size_t)e;
    if (pv->k8) {
        const uint8_t *p8 = which ? pv->v8 : pv->k8;
        const float *sc = which ? pv->v_scale : pv->k_scale;
        return e4m3_to_double(p8[at]) * (double)sc[g];
    }
    return bf16_to_double((which ? pv->v_pool : pv->k_pool)[at]);
}

static int attend_paged(const pool_view *pv, const double *q, int L,
                        const int32_t *bt_row, int g, double scale,
                        double *x, double *out) {
    const int d = pv->head_dim, B = pv->block_size, H = pv->num_kv_heads;
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    if (L <= 0) return OR_OK;
    double M = -INFINITY;
    for (int j = 0; j < L; ++j) {
        int32_t blk = bt_row[j / B];
        if (blk < 0 || blk >= pv->num_blocks) return OR_ERR_BLOCK_RANGE;
        const size_t krow = (size_t)(((long long)blk * H + g) * B + j % B);
        double dot = 0.0;
        for (int e = 0; e < d; ++e) dot += q[e] * pool_elem(pv, 0, krow, g, e);
        x[j] = scale * dot;
        if (x[j] > M) M = x[j];
    }
    double Z = 0.0;
    for (int j = 0; j < L; ++j) {
        double w = exp(x[j] - M);
        x[j] = w;
        Z += w;
    }
    for (int j = 0; j < L; ++j) {
        int32_t blk = bt_row[j / B];
        const size_t vrow = (size_t)(((long long)blk * H + g) * B + j % B);
        for (int e = 0; e < d; ++e) out[e] += x[j] * pool_elem(pv, 1, vrow, g, e);
    }
    for (int e = 0; e < d; ++e) out[e] /= Z;
    return OR_OK;
}

/* Same definition with keys/values stored densely: key j of the sequence is  */
/* row (key_row0 + j) of k[*][Hkv][d].                                        */
static void attend_dense(const uint16_t *k, const uint16_t *v, int num_kv_heads,
                         int d, const double *q, long long key_row0, int L,
                         int g, double scale, double *x, double *out) {
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    if (L <= 0) return;
    double M = -INFINITY;
    for (int j = 0; j < L; ++j) {
        const uint16_t *kr = k + (size_t)((key_row0 + j) * num_kv_heads + g) * d;
        double dot = 0.0;
        for (int e = 0; e < d; ++e) dot += q[e] * bf16_to_double(kr[e]);
        x[j] = scale * dot;
        if (x[j] > M) M = x[j];
    }
    double Z = 0.0;
    for (int j = 0; j < L; ++j) {
        double w = exp(x[j] - M);
        x[j] = w;
        Z += w;
    }
    for (int j = 0; j < L; ++j) {
        const uint16_t *vr = v + (size_t)((key_row0 + j) * num_kv_heads + g) * d;
        for (int e = 0; e < d; ++e) out[e] += x[j] * bf16_to_double(vr[e]);
    }
    for (int e = 0; e < d; ++e) out[e] /= Z;
}

/* ------------------------------------------------------------------------ */
/* A tiny thread pool: items [0, n) split round-robin over nthreads.         */
/* ------------------------------------------------------------------------ */
typedef int (*item_fn)(void *ctx, long long item, double *x, double *qbuf);

typedef struct {
    item_fn fn;
    void *ctx;
    long long n;
    int tid, nthreads;
    size_t scratch;
    int head_dim;
    int status;
} worker_arg;

static void *worker_main(void *p) {
    worker_arg *a = (worker_arg *)p;
    double *x = (double *)malloc(sizeof(double) * (a->scratch > 0 ? a->scratch : 1));
    double *qb = (double *)malloc(sizeof(double) * (size_t)a->head_dim);
    if (!x || !qb) { a->status = OR_ERR_NOMEM; free(x); free(qb); return NULL; }
    for (long long it = a->tid; it < a->n; it += a->nthreads) {
        int st = a->fn(a->ctx, it, x, qb);
        if (st != OR_OK) { a->status = st; break; }
    }
    free(x);
    free(qb);
    return NULL;
}

static int run_items(item_fn fn, void *ctx, long long n, int nthreads,
                     size_t scratch, int head_dim) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    worker_arg args[256];
    int started = 0, status = OR_OK;
    for (int t = 0; t < nthreads; ++t) {
        args[t].fn = fn; args[t].ctx = ctx; args[t].n = n;
        args[t].tid = t; args[t].nthreads = nthreads;
        args[t].scratch = scratch; args[t].head_dim = head_dim;
        args[t].status = OR_OK;
    }
    if (nthreads == 1) {
        worker_main(&args[0]);
        return args[0].status;
    }
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker_main, &args[t]) != 0) {
            args[t].status = OR_ERR_NOMEM;
            break;
        }
        started++;
    }
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    for (int t = 0; t < nthreads; ++t)
        if (args[t].status != OR_OK) status = args[t].status;
    if (started < nthreads) status = OR_ERR_NOMEM;
    return status;
}

static double effective_scale(double scale, int head_dim) {
    return scale > 0.0 ? scale : 1.0 / sqrt((double)head_dim);
}

/* ------------------------------------------------------------------------ */
/* Decode: one query token per running sequence, against its whole cached    */
/* context (seq_lens[s] tokens, counted after this step's append).           */
/* Optional sample list: only the listed (s, h) pairs are computed.          */
/* ------------------------------------------------------------------------ */
typedef struct {
    pool_view pv;
    int Hq, G, max_blocks;
    double scale;
    const uint16_t *q;
    const int32_t *block_table, *seq_lens;
    const int32_t *pairs; /* nullable: [n][2] (s, h) */
    double *out;
} decode_ctx;

static int decode_item(void *c, long long it, double *x, double *qb) {
    decode_ctx *dc = (decode_ctx *)c;
    const int d = dc->pv.head_dim;
    long long s, h;
    if (dc->pairs) { s = dc->pairs[2 * it]; h = dc->pairs[2 * it + 1]; }
    else { s = it / dc->Hq; h = it % dc->Hq; }
    const uint16_t *qr = dc->q + (size_t)((s * dc->Hq + h) * d);
    for (int e = 0; e < d; ++e) qb[e] = bf16_to_double(qr[e]);
    int g = (int)(h / dc->G);
    return attend_paged(&dc->pv, qb, dc->seq_lens[s],
                        dc->block_table + (size_t)s * dc->max_blocks, g,
                        dc->scale, x, dc->out + (size_t)it * d);
}

int oracle_decode(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                  int block_size, int num_blocks, double scale,
                  const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                  const int32_t *block_table, int max_blocks_per_seq,
                  const int32_t *seq_lens, const int32_t *pairs, int num_pairs,
                  double *out, int nthreads) {
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return OR_ERR_ARG;
    int max_len = 0;
    for (int s = 0; s < num_seqs; ++s) {
        if (seq_lens[s] < 0) return OR_ERR_ARG;
        if (seq_lens[s] > (long long)max_blocks_per_seq * block_size) return OR_ERR_BLOCK_RANGE;
        if (seq_lens[s] > max_len) max_len = seq_lens[s];
    }
    decode_ctx dc;
    dc.pv.num_kv_heads = num_kv_heads; dc.pv.head_dim = head_dim;
    dc.pv.block_size = block_size; dc.pv.num_blocks = num_blocks;
    dc.pv.k_pool = k_pool; dc.pv.v_pool = v_pool;
    dc.pv.k8 = dc.pv.v8 = NULL; dc.pv.k_scale = dc.pv.v_scale = NULL;
    dc.Hq = num_q_heads; dc.G = num_q_heads / num_kv_heads;
    dc.max_blocks = max_blocks_per_seq;
    dc.scale = effective_scale(scale, head_dim);
    dc.q = q; dc.block_table = block_table; dc.seq_lens = seq_lens;
    dc.pairs = pairs; dc.out = out;
    long long n = pairs ? num_pairs : (long long)num_seqs * num_q_heads;
    return run_items(decode_item, &dc, n, nthreads, (size_t)max_len + 1, head_dim);
}

/* ------------------------------------------------------------------------ */
/* Prefill: the prompts of newly admitted requests, packed (ragged) by      */
/* cu_seqlens_q.  Row i of sequence s sits at absolute position p0_s + i     */
/* (p0_s = prefix_lens[s], 0 for a fresh prompt) and attends causally to     */
/* keys 0..p0_s+i.                                                           */
/*  - paged form: every key is read through the block table (the new keys   */
/*    were appended before);                                                 */
/*  - dense form: no prefix; key j of sequence s is row cu_seqlens_q[s] + j  */
/*    of the packed k/v.                                                     */
/* Optional sample list of (row, h) pairs.                                   */
/* ------------------------------------------------------------------------ */
typedef struct {
    pool_view pv;           /* paged form */
    const uint16_t *k, *v;  /* dense form */
    int paged;
    int Hq, G, num_seqs, max_blocks, head_dim, num_kv_heads;
    double scale;
    const uint16_t *q;
    const int32_t *cu, *prefix, *block_table;
    const int32_t *pairs; /* nullable: [n][2] (row, h) */
    double *out;
} prefill_ctx;

static int seq_of_row(const int32_t *cu, int num_seqs, long long row) {
    for (int s = 0; s < num_seqs; ++s)
        if (row >= cu[s] && row < cu[s + 1]) return s;
    return -1;
}

static int prefill_item(void *c, long long it, double *x, double *qb) {
    prefill_ctx *pc = (prefill_ctx *)c;
    const int d = pc->head_dim;
    long long row, h;
    if (pc->pairs) { row = pc->pairs[2 * it]; h = pc->pairs[2 * it + 1]; }
    else { row = it / pc->Hq; h = it % pc->Hq; }
    int s = seq_of_row(pc->cu, pc->num_seqs, row);
    double *o = pc->out + (size_t)it * d;
    if (s < 0) return OR_ERR_ARG;
    long long i = row - pc->cu[s];
    int p0 = pc->prefix ? pc->prefix[s] : 0;
    int L = (int)(p0 + i + 1);
    const uint16_t *qr = pc->q + (size_t)((row * pc->Hq + h) * d);
    for (int e = 0; e < d; ++e) qb[e] = bf16_to_double(qr[e]);
    int g = (int)(h / pc->G);
    if (pc->paged)
        return attend_paged(&pc->pv, qb, L,
                            pc->block_table + (size_t)s * pc->max_blocks, g,
                            pc->scale, x, o);
    attend_dense(pc->k, pc->v, pc->num_kv_heads, d, qb, pc->cu[s], L, g,
                 pc->scale, x, o);
    return OR_OK;
}

int oracle_prefill(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                   int block_size, int num_blocks, double scale,
                   const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const int32_t *cu_seqlens_q, const int32_t *prefix_lens,
                   const int32_t *block_table, int max_blocks_per_seq,
                   const int32_t *pairs, int num_pairs,
                   double *out, int nthreads) {
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return OR_ERR_ARG;
    int paged = block_table != NULL;
    if (!paged && prefix_lens) {
        for (int s = 0; s < num_seqs; ++s)
            if (prefix_lens[s] != 0) return OR_ERR_ARG;
    }
    int max_len = 0;
    for (int s = 0; s < num_seqs; ++s) {
        int n = cu_seqlens_q[s + 1] - cu_seqlens_q[s];
        int p0 = prefix_lens ? prefix_lens[s] : 0;
        if (n < 0 || p0 < 0) return OR_ERR_ARG;
        if (paged && (long long)p0 + n > (long long)max_blocks_per_seq * block_size)
            return OR_ERR_BLOCK_RANGE;
        if (p0 + n > max_len) max_len = p0 + n;
    }
    prefill_ctx pc;
    memset(&pc, 0, sizeof pc);
    pc.pv.num_kv_heads = num_kv_heads; pc.pv.head_dim = head_dim;
    pc.pv.block_size = block_size; pc.pv.num_blocks = num_blocks;
    pc.pv.k_pool = k; pc.pv.v_pool = v;
    pc.pv.k8 = pc.pv.v8 = NULL; pc.pv.k_scale = pc.pv.v_scale = NULL;
    pc.k = k; pc.v = v; pc.paged = paged;
    pc.Hq = num_q_heads; pc.G = num_q_heads / num_kv_heads;
    pc.num_seqs = num_seqs; pc.max_blocks = max_blocks_per_seq;
    pc.head_dim = head_dim; pc.num_kv_heads = num_kv_heads;
    pc.scale = effective_scale(scale, head_dim);
    pc.q = q; pc.cu = cu_seqlens_q; pc.prefix = prefix_lens;
    pc.block_table = block_table; pc.pairs = pairs; pc.out = out;
    long long n = pairs ? num_pairs : (long long)cu_seqlens_q[num_seqs] * num_q_heads;
    return run_items(prefill_item, &pc, n, nthreads, (size_t)max_len + 1, head_dim);
}

/*
 * Rotary position embedding of the new tokens' queries and keys.  The pages
 * only name the flashinfer build option that compiles its position-encoding
 * modes in; the plainest reading of "the" rotary embedding there is the one
 * of Su et al. (RoFormer, 2021) with the pairing of its Llama / GPT-NeoX
 * implementations: for a head vector x of even length d at position p, and
 * i < d/2, with f_i = theta^(-2i/d),
 *     y[i]       = x[i] cos(p f_i) - x[i + d/2] sin(p f_i)
 *     y[i + d/2] = x[i + d/2] cos(p f_i) + x[i] sin(p f_i).
 * x: bf16 bits [T][H][d]; pos: [T]; out: double [T][H][d].
 */
int oracle_rope(int num_tokens, int num_heads, int head_dim, const uint16_t *x, const int32_t *pos,
                double theta, double *out) {
    if (num_tokens < 0 || num_heads <= 0 || head_dim <= 0 || (head_dim & 1) || !(theta > 0.0)) return OR_ERR_ARG;
    const int half = head_dim / 2;
    for (int t = 0; t < num_tokens; ++t) {
        if (pos[t] < 0) return OR_ERR_ARG;
        for (int i = 0; i < half; ++i) {
            const double f = pow(theta, -2.0 * (double)i / (double)head_dim);
            const double a = (double)pos[t] * f;
            const double c = cos(a), s = sin(a);
            for (int h = 0; h < num_heads; ++h) {
                const size_t base = ((size_t)t * num_heads + h) * head_dim;
                const double x0 = bf16_to_double(x[base + i]), x1 = bf16_to_double(x[base + i + half]);
                out[base + i] = x0 * c - x1 * s;
                out[base + i + half] = x1 * c + x0 * s;
            }
        }
    }
    return OR_OK;
}

/*
 * Round doubles to bf16 (8 significant bits, round to nearest, ties to even),
 * directly from double (no intermediate float rounding).  Values past the
 * bf16 range become infinities; NaN stays NaN.
 */
int oracle_to_bf16(long long n, const double *x, uint16_t *out) {
    for (long long j = 0; j < n; ++j) {
        const double v = x[j];
        uint16_t sign = signbit(v) ? 0x8000u : 0u;
        if (isnan(v)) {
            out[j] = 0x7fc0u;
            continue;
        }
        double a = fabs(v);
        if (a == 0.0) {
            out[j] = sign;
            continue;
        }
        int e;
        (void)frexp(a, &e);  /* a = m 2^e, m in [0.5, 1) */
        /* quantum: 2^(e - 8) for normals; bf16's smallest step is 2^-133 */
        int qexp = e - 8;
        if (qexp < -133) qexp = -133;
        double r = ldexp(nearbyint(ldexp(a, -qexp)), qexp);
        if (r >= 0x1p128) {
            out[j] = (uint16_t)(sign | 0x7f80u);
            continue;
        }
        float f = (float)r;  /* exact: r has at most 8 significant bits */
        uint32_t bits;
        memcpy(&bits, &f, 4);
        out[j] = (uint16_t)(sign | ((bits >> 16) & 0x7fffu));
    }
    return OR_OK;
}

/*
 * fp8 KV cache (e4m3, one scale per KV head and for K and V apart).  The
 * pages compile flashinfer with FP8 off and name quantisation only as a
 * serving option; the plainest reading of an "fp8 e4m3 cache with a per-head
 * scale": a value x of KV head h is stored as the e4m3 code of x / scale[h]
 * (the quotient in float, as the library computes it, then rounded to
 * nearest-even in e4m3 with saturation at +-448) and read back as
 * e4m3(code) * scale[h].
 *
 * e4m3 (OCP FP8, "fn" variant): 1 sign, 4 exponent bits (bias 7), 3
 * significand bits; no infinities; S.1111.111 is NaN; largest finite 448;
 * subnormals m * 2^-9.
 */
static double e4m3_to_double(uint8_t c) {
    const int sg = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return sg ? -v : v;
}

static uint8_t e4m3_from_double(double x) {
    if (isnan(x)) return 0x7f;
    const uint8_t sg = signbit(x) ? 0x80 : 0x00;
    const double a = fabs(x);
    if (a >= 448.0) return sg | 0x7e;        /* saturate */
    if (a < ldexp(1.0, -6)) {                 /* subnormal range: quantum 2^-9 */
        const double m = nearbyint(ldexp(a, 9));  /* 0..8; 8 is the smallest normal */
        return sg | (uint8_t)m;
    }
    int ex;
    (void)frexp(a, &ex);                      /* a in [2^(ex-1), 2^ex) */
    const int e = ex - 1;                     /* unbiased exponent */
    double q = nearbyint(ldexp(a, 3 - e));    /* significand in eighths: 8..16 */
    int eb = e + 7;
    if (q >= 16.0) { q = 8.0; ++eb; }
    const int code = (eb << 3) | ((int)q - 8);
    return sg | (uint8_t)(code > 0x7e ? 0x7e : code);
}

int oracle_e4m3_from_float(long long n, const float *x, uint8_t *out) {
    for (long long j = 0; j < n; ++j) out[j] = e4m3_from_double((double)x[j]);
    return OR_OK;
}

int oracle_e4m3_to_double(long long n, const uint8_t *c, double *out) {
    for (long long j = 0; j < n; ++j) out[j] = e4m3_to_double(c[j]);
    return OR_OK;
}

/* Append with quantisation: for token i with slot >= 0, element e of KV head
 * h goes to [slot / B][h][slot % B][e] as e4m3(float(x) / scale[h]).  The
 * same checks as oracle_kv_append (slot range, duplicates). */
int oracle_kv_append_fp8(int num_tokens, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         const uint16_t *k_new, const uint16_t *v_new, const int32_t *slot_mapping,
                         const float *k_scale, const float *v_scale, uint8_t *k_pool, uint8_t *v_pool) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return OR_ERR_ARG;
    const long long num_slots = (long long)num_blocks * block_size;
    char *seen = calloc((size_t)num_slots, 1);
    if (!seen) return OR_ERR_NOMEM;
    for (int i = 0; i < num_tokens; ++i) {
        const int32_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if ((long long)slot >= num_slots) { free(seen); return OR_ERR_SLOT_RANGE; }
        if (seen[slot]) { free(seen); return OR_ERR_SLOT_DUP; }
        seen[slot] = 1;
        const long long blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            const size_t src = ((size_t)i * num_kv_heads + h) * head_dim;
            const size_t dst = (size_t)(((blk * num_kv_heads + h) * block_size + off) * head_dim);
            for (int e = 0; e < head_dim; ++e) {
                const float kq = (float)bf16_to_double(k_new[src + e]) / k_scale[h];
                const float vq = (float)bf16_to_double(v_new[src + e]) / v_scale[h];
                k_pool[dst + e] = e4m3_from_double((double)kq);
                v_pool[dst + e] = e4m3_from_double((double)vq);
            }
        }
    }
    free(seen);
    return OR_OK;
}

/* Decode over fp8 pools: oracle_decode with every key and value element read
 * as e4m3(code) * scale of its KV head. */
int oracle_decode_fp8(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      int num_blocks, double scale, const uint16_t *q, const uint8_t *k_pool,
                      const uint8_t *v_pool, const float *k_scale, const float *v_scale,
                      const int32_t *block_table, int max_blocks_per_seq, const int32_t *seq_lens,
                      const int32_t *pairs, int num_pairs, double *out, int nthreads) {
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return OR_ERR_ARG;
    int max_len = 0;
    for (int s = 0; s < num_seqs; ++s) {
        if (seq_lens[s] < 0) return OR_ERR_ARG;
        if (seq_lens[s] > (long long)max_blocks_per_seq * block_size) return OR_ERR_BLOCK_RANGE;
        if (seq_lens[s] > max_len) max_len = seq_lens[s];
    }
    decode_ctx dc;
    dc.pv.num_kv_heads = num_kv_heads; dc.pv.head_dim = head_dim;
    dc.pv.block_size = block_size; dc.pv.num_blocks = num_blocks;
    dc.pv.k_pool = dc.pv.v_pool = NULL;
    dc.pv.k8 = k_pool; dc.pv.v8 = v_pool; dc.pv.k_scale = k_scale; dc.pv.v_scale = v_scale;
    dc.Hq = num_q_heads; dc.G = num_q_heads / num_kv_heads;
    dc.max_blocks = max_blocks_per_seq;
    dc.scale = effective_scale(scale, head_dim);
    dc.q = q; dc.block_table = block_table; dc.seq_lens = seq_lens;
    dc.pairs = pairs; dc.out = out;
    long long n = pairs ? num_pairs : (long long)num_seqs * num_q_heads;
    return run_items(decode_item, &dc, n, nthreads, (size_t)max_len + 1, head_dim);
}
