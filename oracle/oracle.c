/*
 * oracle.c -- plain, slow fp64 CPU oracle for ring / context-parallel attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's timed
 * CPU baseline do.  It shares no code, header, table or constant with the
 * CUDA library: it has its own shard mapper, its own schedule and its own
 * merge.
 *
 * Sources (page title, section):
 *  - "Sequence Parallelism in LLMs: Megatron-SP, Ulysses, RingAttention"
 *    (llms.blog): "Algorithmic Mechanics" (contiguous partition into P blocks
 *    of s/P; step k uses KV from (i-k) mod P; the m/l/O online-softmax
 *    rescaling equations), "Causal Masking and Load Balancing" (j <= i),
 *    "DeepSpeed Ulysses" (the [Batch, S/P, H, D] <-> [Batch, S, H/P, D]
 *    relayout).
 *  - the same page, "Causal Masking and Load Balancing" (striped
 *    partitioning: token t goes to rank t mod P);
 *  - "Context Parallelism" (aiwiki): "The causal imbalance" (zigzag: 2N
 *    chunks, rank i holds chunks i and 2N-1-i), the ring sketch (source rank
 *    = (rank - step) mod world, N compute steps).
 *  - "Sequence and Context Parallelism" (praveentn.live): "What it does not
 *    change" (the distributed result equals single-device attention).
 *
 * Conventions (readings of the pages where they are silent):
 *  - tensors are BSHD in global token order: q [B][S][Hq][D],
 *    k, v [B][S][Hkv][D]; lse is [B][Hq][rows], natural log;
 *  - query head h uses kv head h / (Hq / Hkv) (contiguous GQA groups);
 *  - striped: rank r keeps its tokens r, r+N, r+2N, ... in ascending order
 *    (local row t is position r + N t);
 *  - causal means key j is visible to query i iff j <= i (diagonal included);
 *  - the page's O_block in the rescaling equations is the block's
 *    unnormalised numerator sum_j e^{s_j - m_block} v_j, while O_prev is the
 *    running normalised output (the only reading that makes O_new
 *    normalised);
 *  - an empty block (no visible key) leaves the running state unchanged; an
 *    empty row has out = 0, lse = -inf.
 *
 * Every loop is the definition written out; OpenMP only spreads independent
 * rows over cores.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_CONTIGUOUS 0
#define OR_ZIGZAG 1
#define OR_STRIPED 2

/* ------------------------------------------------------------------------ */
/* Sequence sharding ("Algorithmic Mechanics" step 1; "The causal imbalance") */

/* Shapes each layout accepts: N ranks of S/N rows; zigzag also needs 2N
 * equal chunks. */
static int or_layout_ok(int64_t S, int N, int layout)
{
    if (N < 1 || S < 0 || S % N) return 0;
    if (layout != OR_CONTIGUOUS && layout != OR_ZIGZAG && layout != OR_STRIPED) return 0;
    if (layout == OR_ZIGZAG && S % (2 * (int64_t)N)) return 0;
    return 1;
}

/* Global position of local row t of rank r. */
static int64_t or_pos(int64_t S, int N, int layout, int r, int64_t t)
{
    if (layout == OR_CONTIGUOUS) {
        int64_t blk = S / N;                 /* B = s/P */
        return (int64_t)r * blk + t;
    }
    if (layout == OR_STRIPED)                /* round robin: position p on rank p mod N */
        return (int64_t)r + (int64_t)N * t;
    int64_t c = S / (2 * (int64_t)N);        /* 2N chunks */
    if (t < c)
        return (int64_t)r * c + t;           /* chunk r */
    return (int64_t)(2 * N - 1 - r) * c + (t - c);   /* chunk 2N-1-r */
}

/* Ring schedule: at step k device r holds the KV block of rank (r-k) mod N. */
static int or_source(int N, int r, int k)
{
    int s = (r - k) % N;
    return s < 0 ? s + N : s;
}

int or_shard_pos(int64_t S, int N, int layout, int64_t *pos)
{
    if (!or_layout_ok(S, N, layout)) return -1;
    int64_t L = S / N;
    for (int r = 0; r < N; ++r)
        for (int64_t t = 0; t < L; ++t)
            pos[(int64_t)r * L + t] = or_pos(S, N, layout, r, t);
    return 0;
}

int or_ring_source_table(int N, int *src /* [N steps][N ranks] */)
{
    for (int k = 0; k < N; ++k)
        for (int r = 0; r < N; ++r)
            src[k * N + r] = or_source(N, r, k);
    return 0;
}

/* Masked-in (query, key) pairs of rank r at ring step k, counts[r*N + k].
 * Counted per query row: for each query position p of rank r, the number of
 * key positions j of the source rank with j <= p (all of them if not causal). */
int or_pair_counts(int64_t S, int N, int layout, int causal, int64_t *counts)
{
    if (!or_layout_ok(S, N, layout)) return -1;
    int64_t L = S / N;
    memset(counts, 0, sizeof(int64_t) * (size_t)N * N);
    for (int r = 0; r < N; ++r) {
        for (int k = 0; k < N; ++k) {
            int src = or_source(N, r, k);
            int64_t acc = 0;
            for (int64_t t = 0; t < L; ++t) {
                int64_t p = or_pos(S, N, layout, r, t);
                for (int64_t u = 0; u < L; ++u) {
                    int64_t j = or_pos(S, N, layout, src, u);
                    if (!causal || j <= p) ++acc;
                }
            }
            counts[r * N + k] = acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O1: definitional attention.  For query row i of (b, h):
 *   s_ij = scale * <q_i, k_j>   over visible j in [klo, khi)
 *   lse_i = ln sum_j e^{s_ij}   (max-subtracted)
 *   out_i = sum_j e^{s_ij - lse_i} v_j
 * rows == NULL means every row 0..S-1 (nrows == S).
 * out is [B][nrows][Hq][D], lse is [B][Hq][nrows]. */
int or_attn_fwd(const double *q, const double *k, const double *v,
                int B, int Hq, int Hkv, int64_t S, int D, int causal, double scale,
                int64_t nrows, const int64_t *rows, int64_t klo, int64_t khi,
                double *out, double *lse)
{
    if (Hkv < 1 || Hq % Hkv) return -1;
    const int grp = Hq / Hkv;
    if (khi > S) khi = S;
    if (klo < 0) klo = 0;
    int64_t total = (int64_t)B * Hq * nrows;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
#pragma omp for schedule(dynamic, 16)
        for (int64_t idx = 0; idx < total; ++idx) {
            int64_t ri = idx % nrows;
            int h = (int)((idx / nrows) % Hq);
            int b = (int)(idx / (nrows * Hq));
            int g = h / grp;
            int64_t i = rows ? rows[ri] : ri;
            const double *qi = q + (((int64_t)b * S + i) * Hq + h) * D;
            int64_t jend = khi;
            if (causal && i + 1 < jend) jend = i + 1;
            double m = -INFINITY;
            for (int64_t j = klo; j < jend; ++j) {
                const double *kj = k + (((int64_t)b * S + j) * Hkv + g) * D;
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += qi[d] * kj[d];
                s[j] = scale * acc;
                if (s[j] > m) m = s[j];
            }
            double *oi = out + (((int64_t)b * nrows + ri) * Hq + h) * D;
            double *li = lse + ((int64_t)b * Hq + h) * nrows + ri;
            for (int d = 0; d < D; ++d) oi[d] = 0.0;
            if (jend <= klo) { *li = -INFINITY; continue; }
            double l = 0.0;
            for (int64_t j = klo; j < jend; ++j) l += exp(s[j] - m);
            double L = m + log(l);
            *li = L;
            for (int64_t j = klo; j < jend; ++j) {
                double p = exp(s[j] - L);
                const double *vj = v + (((int64_t)b * S + j) * Hkv + g) * D;
                for (int d = 0; d < D; ++d) oi[d] += p * vj[d];
            }
        }
        free(s);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* O2: explicit ring emulation.  Rank r keeps its queries; at step k it holds
 * the KV block of src = (r-k) mod N, computes the block's row statistics
 * (m_block, l_block, unnormalised O_block) under the global-position causal
 * mask, and folds them into (O, m, l) with the online-softmax rescaling
 * equations.  Results are written back in global order:
 * out [B][S][Hq][D], lse [B][Hq][S]. */
int or_ring_fwd(const double *q, const double *k, const double *v,
                int B, int Hq, int Hkv, int64_t S, int D, int N, int causal, int layout,
                double scale, double *out, double *lse)
{
    if (!or_layout_ok(S, N, layout) || Hkv < 1 || Hq % Hkv) return -1;
    const int grp = Hq / Hkv;
    const int64_t L = S / N;
    int64_t total = (int64_t)B * Hq * S;   /* (b, h, r, t) flattened */
#pragma omp parallel
    {
        double *sblk = (double *)malloc(sizeof(double) * (size_t)L);
        double *ob = (double *)malloc(sizeof(double) * (size_t)D);
        double *O = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 16)
        for (int64_t idx = 0; idx < total; ++idx) {
            int64_t t = idx % L;
            int r = (int)((idx / L) % N);
            int h = (int)((idx / S) % Hq);
            int b = (int)(idx / (S * Hq));
            int g = h / grp;
            int64_t p = or_pos(S, N, layout, r, t);
            const double *qi = q + (((int64_t)b * S + p) * Hq + h) * D;
            double m = -INFINITY, l = 0.0;
            for (int d = 0; d < D; ++d) O[d] = 0.0;
            for (int step = 0; step < N; ++step) {
                int src = or_source(N, r, step);
                /* block statistics */
                double mb = -INFINITY;
                for (int64_t u = 0; u < L; ++u) {
                    int64_t j = or_pos(S, N, layout, src, u);
                    if (causal && j > p) { sblk[u] = -INFINITY; continue; }
                    const double *kj = k + (((int64_t)b * S + j) * Hkv + g) * D;
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d) acc += qi[d] * kj[d];
                    sblk[u] = scale * acc;
                    if (sblk[u] > mb) mb = sblk[u];
                }
                if (mb == -INFINITY) continue;          /* empty block: identity */
                double lb = 0.0;
                for (int d = 0; d < D; ++d) ob[d] = 0.0;
                for (int64_t u = 0; u < L; ++u) {
                    if (sblk[u] == -INFINITY) continue;
                    double e = exp(sblk[u] - mb);
                    lb += e;
                    int64_t j = or_pos(S, N, layout, src, u);
                    const double *vj = v + (((int64_t)b * S + j) * Hkv + g) * D;
                    for (int d = 0; d < D; ++d) ob[d] += e * vj[d];
                }
                /* m_new = max(m_prev, m_block)
                 * l_new = l_prev e^{m_prev-m_new} + l_block e^{m_block-m_new}
                 * O_new = O_prev (l_prev e^{m_prev-m_new} / l_new)
                 *       + O_block (e^{m_block-m_new} / l_new)                */
                double mn = m > mb ? m : mb;
                double a = l * exp(m - mn);            /* exp(-inf) = 0 on the first block */
                double bb = exp(mb - mn);
                double ln = a + lb * bb;
                for (int d = 0; d < D; ++d) O[d] = O[d] * (a / ln) + ob[d] * (bb / ln);
                m = mn;
                l = ln;
            }
            double *oi = out + (((int64_t)b * S + p) * Hq + h) * D;
            for (int d = 0; d < D; ++d) oi[d] = O[d];
            lse[((int64_t)b * Hq + h) * S + p] = (l > 0.0) ? m + log(l) : -INFINITY;
        }
        free(sblk);
        free(ob);
        free(O);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* One ring step of one device, on shard-local buffers (the flash_block call of
 * the "Context Parallelism" ring sketch; one step k of "Algorithmic
 * Mechanics").  q holds the C = S/N queries of rank r, k and v the C keys and
 * values of rank src, each in that rank's local order (row t is global
 * position or_pos(r, t)).  The state is the running normalised result:
 * out [B][C][Hq][D], lse [B][Hq][C]; a normalised state is (O = out, m = lse,
 * l = 1), or empty (l = 0) when lse = -inf.  The block statistics
 * (m_block, l_block, unnormalised O_block) under the global-position causal
 * mask are folded in with the same rescaling equations as or_ring_fwd.
 * accumulate = 0 starts from the empty state. */
int or_block_step(const double *q, const double *k, const double *v,
                  int B, int Hq, int Hkv, int64_t S, int D, int N, int layout, int causal,
                  int r, int src, double scale, int accumulate, double *out, double *lse)
{
    if (!or_layout_ok(S, N, layout) || Hkv < 1 || Hq % Hkv) return -1;
    if (r < 0 || r >= N || src < 0 || src >= N) return -1;
    const int grp = Hq / Hkv;
    const int64_t C = S / N;
    int64_t total = (int64_t)B * Hq * C;
#pragma omp parallel
    {
        double *sblk = (double *)malloc(sizeof(double) * (size_t)(C > 0 ? C : 1));
        double *ob = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 16)
        for (int64_t idx = 0; idx < total; ++idx) {
            int64_t t = idx % C;
            int h = (int)((idx / C) % Hq);
            int b = (int)(idx / (C * Hq));
            int g = h / grp;
            int64_t p = or_pos(S, N, layout, r, t);
            const double *qi = q + (((int64_t)b * C + t) * Hq + h) * D;
            double *oi = out + (((int64_t)b * C + t) * Hq + h) * D;
            double *li = lse + ((int64_t)b * Hq + h) * C + t;
            /* the running state */
            double m = accumulate ? *li : -INFINITY;
            double l = (m == -INFINITY) ? 0.0 : 1.0;
            if (!accumulate)
                for (int d = 0; d < D; ++d) oi[d] = 0.0;
            /* block statistics */
            double mb = -INFINITY;
            for (int64_t u = 0; u < C; ++u) {
                int64_t j = or_pos(S, N, layout, src, u);
                if (causal && j > p) { sblk[u] = -INFINITY; continue; }
                const double *kj = k + (((int64_t)b * C + u) * Hkv + g) * D;
                double acc = 0.0;
                for (int d = 0; d < D; ++d) acc += qi[d] * kj[d];
                sblk[u] = scale * acc;
                if (sblk[u] > mb) mb = sblk[u];
            }
            if (mb == -INFINITY) {                      /* empty block: identity */
                if (!accumulate) *li = -INFINITY;
                continue;
            }
            double lb = 0.0;
            for (int d = 0; d < D; ++d) ob[d] = 0.0;
            for (int64_t u = 0; u < C; ++u) {
                if (sblk[u] == -INFINITY) continue;
                double e = exp(sblk[u] - mb);
                lb += e;
                const double *vj = v + (((int64_t)b * C + u) * Hkv + g) * D;
                for (int d = 0; d < D; ++d) ob[d] += e * vj[d];
            }
            /* m_new, l_new, O_new as in or_ring_fwd */
            double mn = m > mb ? m : mb;
            double a = l * exp(m - mn);
            double bb = exp(mb - mn);
            double ln = a + lb * bb;
            for (int d = 0; d < D; ++d) oi[d] = oi[d] * (a / ln) + ob[d] * (bb / ln);
            *li = mn + log(ln);
        }
        free(sblk);
        free(ob);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Merge of two normalised partial results (out_x, lse_x) over disjoint key
 * sets.  A normalised partial is the state (O = out_x, m = lse_x, l = 1), so
 * the rescaling equations give
 *   m = max(lse_a, lse_b),  l = e^{lse_a-m} + e^{lse_b-m},
 *   out = out_a e^{lse_a-m}/l + out_b e^{lse_b-m}/l,  lse = m + ln l.
 * Both empty (-inf) gives (0, -inf). */
int or_lse_merge(const double *out_a, const double *lse_a, const double *out_b,
                 const double *lse_b, int64_t rows, int D, double *out, double *lse)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double la = lse_a[r], lb = lse_b[r];
        double m = la > lb ? la : lb;
        const double *xa = out_a + r * D, *xb = out_b + r * D;
        double *o = out + r * D;
        if (m == -INFINITY) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        double wa = exp(la - m), wb = exp(lb - m);
        double l = wa + wb;
        for (int d = 0; d < D; ++d) o[d] = xa[d] * (wa / l) + xb[d] * (wb / l);
        lse[r] = m + log(l);
    }
    return 0;
}

/* n-way merge of normalised partials over disjoint key sets, the same
 * log-sum-exp combination taken over all n at once:
 *   lse = ln sum_i e^{lse_i},  out = sum_i e^{lse_i - lse} out_i.
 * out_parts [n][rows][D], lse_parts [n][rows]; partials with lse = -inf have
 * weight 0; all empty gives (0, -inf). */
int or_lse_merge_n(const double *out_parts, const double *lse_parts, int n, int64_t rows, int D,
                   double *out, double *lse)
{
    if (n < 1 || rows < 0 || D < 1) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (int i = 0; i < n; ++i) {
            double li = lse_parts[(int64_t)i * rows + r];
            if (li > m) m = li;
        }
        double *o = out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double l = 0.0;
        for (int i = 0; i < n; ++i) l += exp(lse_parts[(int64_t)i * rows + r] - m);
        for (int i = 0; i < n; ++i) {
            double w = exp(lse_parts[(int64_t)i * rows + r] - m) / l;
            const double *x = out_parts + ((int64_t)i * rows + r) * D;
            for (int d = 0; d < D; ++d) o[d] += w * x[d];
        }
        lse[r] = m + log(l);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Ulysses relayout ("DeepSpeed Ulysses" diagram): rank r's sequence shard
 * [B, S/N, H, D] goes to head-group layout [B, S, H/N, D] on rank g, which
 * receives heads [g*H/N, (g+1)*H/N) of every rank's shard, in global token
 * order.  x is the rank-major stack [N][B][S/N][H][D]; y is [N][B][S][H/N][D].
 * Element size is elem bytes; pure byte copies. */
static int or_ulysses(const unsigned char *x, unsigned char *y, int B, int64_t S, int H, int D,
                      int N, int layout, int elem, int to_head)
{
    if (!or_layout_ok(S, N, layout) || H % N) return -1;
    const int64_t L = S / N;
    const int hg = H / N;
    const size_t row = (size_t)D * elem;
    for (int r = 0; r < N; ++r)
        for (int b = 0; b < B; ++b)
            for (int64_t t = 0; t < L; ++t) {
                int64_t s = or_pos(S, N, layout, r, t);
                for (int h = 0; h < H; ++h) {
                    int g = h / hg, hh = h % hg;
                    size_t xo = ((((size_t)r * B + b) * L + t) * H + h) * row;
                    size_t yo = ((((size_t)g * B + b) * S + s) * hg + hh) * row;
                    if (to_head) memcpy(y + yo, x + xo, row);
                    else         memcpy((unsigned char *)x + xo, y + yo, row);
                }
            }
    return 0;
}

int or_ulysses_seq_to_head(const void *x, void *y, int B, int64_t S, int H, int D, int N,
                           int layout, int elem)
{
    return or_ulysses((const unsigned char *)x, (unsigned char *)y, B, S, H, D, N, layout, elem, 1);
}

int or_ulysses_head_to_seq(const void *y, void *x, int B, int64_t S, int H, int D, int N,
                           int layout, int elem)
{
    return or_ulysses((const unsigned char *)x, (unsigned char *)y, B, S, H, D, N, layout, elem, 0);
}

/* ------------------------------------------------------------------------ */
/* Backward of L = sum(dO * out) (textbook attention gradient; the pages only
 * state that gradients equal single-device ones).  With P_ij = e^{s_ij - lse_i}:
 *   dP_ij = <dO_i, v_j>,  Delta_i = <dO_i, out_i>,  dS_ij = P_ij (dP_ij - Delta_i)
 *   dQ_i = scale sum_j dS_ij k_j
 *   dK_j = scale sum_{h in group, i} dS_ij q_i,  dV_j = sum_{h in group, i} P_ij dO_i
 * dq is [B][nq][Hq][D] for the query positions qrows; dk, dv are
 * [B][nk][Hkv][D] for the key positions krows. */

/* lse_i and Delta_i of one query row, using the definitional forward. */
static void or_row_stats(const double *q, const double *k, const double *v, const double *dout,
                         int b, int h, int g, int64_t i, int64_t S, int Hq, int Hkv, int D,
                         int causal, double scale, double *s, double *o, double *lse_out,
                         double *delta_out)
{
    const double *qi = q + (((int64_t)b * S + i) * Hq + h) * D;
    int64_t jend = causal ? i + 1 : S;
    double m = -INFINITY;
    for (int64_t j = 0; j < jend; ++j) {
        const double *kj = k + (((int64_t)b * S + j) * Hkv + g) * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qi[d] * kj[d];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < jend; ++j) l += exp(s[j] - m);
    double L = m + log(l);
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < jend; ++j) {
        double p = exp(s[j] - L);
        const double *vj = v + (((int64_t)b * S + j) * Hkv + g) * D;
        for (int d = 0; d < D; ++d) o[d] += p * vj[d];
    }
    const double *di = dout + (((int64_t)b * S + i) * Hq + h) * D;
    double dl = 0.0;
    for (int d = 0; d < D; ++d) dl += di[d] * o[d];
    *lse_out = L;
    *delta_out = dl;
}

int or_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                int B, int Hq, int Hkv, int64_t S, int D, int causal, double scale,
                int64_t nq, const int64_t *qrows, int64_t nk, const int64_t *krows,
                double *dq, double *dk, double *dv)
{
    if (Hkv < 1 || Hq % Hkv) return -1;
    const int grp = Hq / Hkv;

    /* dQ for the requested query rows */
    int64_t totq = (int64_t)B * Hq * nq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)S);
        double *o = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 4)
        for (int64_t idx = 0; idx < totq; ++idx) {
            int64_t ri = idx % nq;
            int h = (int)((idx / nq) % Hq);
            int b = (int)(idx / (nq * Hq));
            int g = h / grp;
            int64_t i = qrows[ri];
            double L, dl;
            or_row_stats(q, k, v, dout, b, h, g, i, S, Hq, Hkv, D, causal, scale, s, o, &L, &dl);
            const double *di = dout + (((int64_t)b * S + i) * Hq + h) * D;
            double *dqi = dq + (((int64_t)b * nq + ri) * Hq + h) * D;
            for (int d = 0; d < D; ++d) dqi[d] = 0.0;
            int64_t jend = causal ? i + 1 : S;
            for (int64_t j = 0; j < jend; ++j) {
                const double *kj = k + (((int64_t)b * S + j) * Hkv + g) * D;
                const double *vj = v + (((int64_t)b * S + j) * Hkv + g) * D;
                double p = exp(s[j] - L);
                double dp = 0.0;
                for (int d = 0; d < D; ++d) dp += di[d] * vj[d];
                double ds = p * (dp - dl);
                for (int d = 0; d < D; ++d) dqi[d] += scale * ds * kj[d];
            }
        }
        free(s);
        free(o);
    }

    if (nk == 0) return 0;
    /* dK, dV for the requested key rows: first the row statistics of every
     * query that can see one of them. */
    int64_t kmin = S;
    for (int64_t t = 0; t < nk; ++t) if (krows[t] < kmin) kmin = krows[t];
    int64_t i0 = causal ? kmin : 0;
    int64_t nrow = S - i0;
    double *Lse = (double *)malloc(sizeof(double) * (size_t)B * Hq * (size_t)(nrow > 0 ? nrow : 1));
    double *Del = (double *)malloc(sizeof(double) * (size_t)B * Hq * (size_t)(nrow > 0 ? nrow : 1));
    int64_t totr = (int64_t)B * Hq * nrow;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)S);
        double *o = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 4)
        for (int64_t idx = 0; idx < totr; ++idx) {
            int64_t ii = idx % nrow;
            int h = (int)((idx / nrow) % Hq);
            int b = (int)(idx / (nrow * Hq));
            or_row_stats(q, k, v, dout, b, h, h / grp, i0 + ii, S, Hq, Hkv, D, causal, scale, s, o,
                         &Lse[idx], &Del[idx]);
        }
        free(s);
        free(o);
    }
    int64_t totk = (int64_t)B * Hkv * nk;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t idx = 0; idx < totk; ++idx) {
        int64_t rj = idx % nk;
        int g = (int)((idx / nk) % Hkv);
        int b = (int)(idx / (nk * Hkv));
        int64_t j = krows[rj];
        const double *kj = k + (((int64_t)b * S + j) * Hkv + g) * D;
        const double *vj = v + (((int64_t)b * S + j) * Hkv + g) * D;
        double *dkj = dk + (((int64_t)b * nk + rj) * Hkv + g) * D;
        double *dvj = dv + (((int64_t)b * nk + rj) * Hkv + g) * D;
        for (int d = 0; d < D; ++d) { dkj[d] = 0.0; dvj[d] = 0.0; }
        for (int h = g * grp; h < (g + 1) * grp; ++h) {
            for (int64_t i = causal ? j : 0; i < S; ++i) {
                if (i < i0) continue;
                int64_t si = ((int64_t)b * Hq + h) * nrow + (i - i0);
                const double *qi = q + (((int64_t)b * S + i) * Hq + h) * D;
                const double *di = dout + (((int64_t)b * S + i) * Hq + h) * D;
                double acc = 0.0, dp = 0.0;
                for (int d = 0; d < D; ++d) { acc += qi[d] * kj[d]; dp += di[d] * vj[d]; }
                double p = exp(scale * acc - Lse[si]);
                double ds = p * (dp - Del[si]);
                for (int d = 0; d < D; ++d) {
                    dvj[d] += p * di[d];
                    dkj[d] += scale * ds * qi[d];
                }
            }
        }
    }
    free(Lse);
    free(Del);
    return 0;
}

int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
