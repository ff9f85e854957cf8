/*
 * txl_oracle.c -- fp64 CPU oracle for Transformer-XL relative multi-head attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file; only the test suite, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Everything is evaluated literally, in double precision, in the order the pages state
 * it: an explicit sinusoid R_delta per distance, an explicit projection by W_R, the four
 * score terms summed one by one, the mask, the 1/sqrt(d_head) scale, a softmax over the
 * visible keys and the weighted sum of plain value vectors.  There is no relative-shift
 * trick, no blocking and no fusion.
 *
 * Sources (page title, section):
 *  [S]  "跨窗口的相对位置编码" (qidao123.com), §2: R_delta^(2k) = sin(delta/10000^(2k/d)),
 *       R_delta^(2k+1) = cos(same), with the worked example R_{-2} for d = 4.
 *  [S5] "Transformer-XL 和相对位置编码" (felixzhao.cn), §2.3.2: the same sinusoid written
 *       with d_model and k = 0..d_model/2-1; terms (a)-(d) of A^rel; W_{k,R} on R_{i-j}.
 *  [A]  "跨窗口的相对位置编码" §3: A^rel_ij = Q_i.K_j + Q_i.R_{i-j} + u.K_j + v.R_{i-j}.
 *  [U]  "TransformerXL 相对位置编码" (2kiu.com), §2.3: u and v are per-head [d_head]
 *       vectors shared by every query position; §3.1: u, v and r_proj (no bias).
 *  [C]  same page §2.4: distances beyond the window are treated as the window edge.
 *  [K]  same page §4.2: mask after summing all four terms, then softmax;
 *       §4.3: keys span [memory ++ current], queries are the current segment only.
 *  [R]  "Transformer-XL 和相对位置编码" §2.3.1: K and V come from SG(h_prev) ∘ h,
 *       Q from the current segment only.
 *  [V]  "跨窗口的相对位置编码" §3.2 (last paragraphs): no position term on V.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - Query i of the current segment sits at absolute position M+i, key j at position j
 *    of [memory ++ current]; delta = (M+i) - j.
 *  - Clamp: delta_c = min(delta, clamp_len).  Negative delta only occurs on masked pairs.
 *  - Visibility: key j is visible to query i iff (M - mem_valid) <= j <= M+i.
 *    Masked keys are excluded from the softmax (probability exactly 0).
 *  - The scale 1/sqrt(d_head) multiplies the sum of all four terms.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------ */
/* [S], [S5]: the sinusoid relative encoding, interleaved sin/cos.                       */
/* R[2k] = sin(delta * 10000^(-2k/d_model)), R[2k+1] = cos(same), k = 0..d_model/2-1.     */
/* ------------------------------------------------------------------------------------ */
void txlo_sinusoid(double delta, int d_model, double *R)
{
    for (int k = 0; k < d_model / 2; ++k) {
        double denom = pow(10000.0, (2.0 * k) / (double)d_model);
        double angle = delta / denom;
        R[2 * k] = sin(angle);
        R[2 * k + 1] = cos(angle);
    }
}

/* ------------------------------------------------------------------------------------ */
/* [S5] term (b)/(d): W_{k,R} R_{i-j}.  For head h the position key vector is            */
/*   r[d] = sum_m R_delta[m] * W_R[m][h*D + d]     (W_R is [d_model][ld_w], row-major).   */
/* ------------------------------------------------------------------------------------ */
void txlo_rel_vec(double delta, int d_model, int D, const double *W_R, int64_t ld_w,
                  int h, double *r_out)
{
    double *R = (double *)malloc(sizeof(double) * (size_t)d_model);
    txlo_sinusoid(delta, d_model, R);
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int m = 0; m < d_model; ++m)
            acc += R[m] * W_R[(int64_t)m * ld_w + (int64_t)h * D + d];
        r_out[d] = acc;
    }
    free(R);
}

/* Full table r[delta][h][d] for delta = 0..n_rows-1 (the quantity txl_rel_pos_gen makes). */
void txlo_rel_table(int n_rows, int d_model, int H, int D, const double *W_R, int64_t ld_w,
                    double *r_out /* [n_rows][H][D] */)
{
    for (int delta = 0; delta < n_rows; ++delta)
        for (int h = 0; h < H; ++h)
            txlo_rel_vec((double)delta, d_model, D, W_R, ld_w, h,
                         r_out + ((int64_t)delta * H + h) * D);
}

/* ------------------------------------------------------------------------------------ */
/* [A], [S5] (a)+(b)+(c)+(d): the four terms summed literally, unscaled.                  */
/* ------------------------------------------------------------------------------------ */
double txlo_score_terms(int D, const double *q, const double *k, const double *r,
                        const double *u, const double *v, double *terms_out /* [4] or NULL */)
{
    double a = 0.0, b = 0.0, c = 0.0, d4 = 0.0;
    for (int d = 0; d < D; ++d) a += q[d] * k[d];   /* (a) content-content  */
    for (int d = 0; d < D; ++d) b += q[d] * r[d];   /* (b) content-position */
    for (int d = 0; d < D; ++d) c += u[d] * k[d];   /* (c) global content bias   */
    for (int d = 0; d < D; ++d) d4 += v[d] * r[d];  /* (d) global position bias  */
    if (terms_out) { terms_out[0] = a; terms_out[1] = b; terms_out[2] = c; terms_out[3] = d4; }
    return a + b + c + d4;
}

/* ------------------------------------------------------------------------------------ */
/* One call of relative attention over [memory ++ current]:                              */
/*   q   [B][L][H][D]            current-segment queries                                 */
/*   k,v [B][M+L][H][D]          keys/values in logical order, memory first              */
/*   u,vb [H][D]                 global content / position biases                        */
/*   W_R [d_model][ld_w]         position projection                                     */
/*   out [B][L][H][D]                                                                     */
/* Rows to evaluate: sel (n_sel triples b,h,i) or all rows when sel == NULL.              */
/* memo != 0 caches r(delta_c) per head for the heads touched (same function, same code). */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    int B, L, H, D, M, mem_valid, clamp_len, d_model;
    int64_t ld_w;
    double scale;
    const double *q, *k, *v, *u, *vb, *W_R;
    double *out;
    int memo;
    const int *sel;
    int64_t n_sel;
    double **memo_tab; /* [H] -> [n_memo][D] or NULL */
    int n_memo;
    int64_t next;     /* work counter */
    pthread_mutex_t lock;
} txlo_job;

static const double *txlo_rvec(txlo_job *J, int h, int delta_c, double *scratch)
{
    if (J->memo && J->memo_tab[h]) return J->memo_tab[h] + (int64_t)delta_c * J->D;
    txlo_rel_vec((double)delta_c, J->d_model, J->D, J->W_R, J->ld_w, h, scratch);
    return scratch;
}

static void txlo_one_row(txlo_job *J, int b, int h, int i, double *s, double *rs, double *acc)
{
    const int D = J->D, H = J->H, M = J->M, L = J->L;
    const int K = M + L;
    const int lo = M - J->mem_valid;            /* first visible memory key            */
    const int qpos = M + i;                     /* absolute position of query i        */
    const double *qi = J->q + (((int64_t)b * L + i) * H + h) * D;
    const double *uh = J->u + (int64_t)h * D;
    const double *vh = J->vb + (int64_t)h * D;
    double mx = -INFINITY;
    for (int j = 0; j < K; ++j) {
        int visible = (j >= lo) && (j <= qpos);
        if (!visible) continue;
        int delta = qpos - j;
        int delta_c = delta < J->clamp_len ? delta : J->clamp_len;
        const double *kj = J->k + (((int64_t)b * K + j) * H + h) * D;
        const double *r = txlo_rvec(J, h, delta_c, rs);
        s[j] = J->scale * txlo_score_terms(D, qi, kj, r, uh, vh, NULL);
        if (s[j] > mx) mx = s[j];
    }
    double den = 0.0;
    for (int j = 0; j < K; ++j) {
        int visible = (j >= lo) && (j <= qpos);
        if (!visible) continue;
        s[j] = exp(s[j] - mx);
        den += s[j];
    }
    /* accumulate in the caller's private buffer, then store the finished row: a row listed
     * twice in a selection is then written twice with the same values, never raced on */
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int j = 0; j < K; ++j) {
        int visible = (j >= lo) && (j <= qpos);
        if (!visible) continue;
        double p = s[j] / den;
        const double *vj = J->v + (((int64_t)b * K + j) * H + h) * D;
        for (int d = 0; d < D; ++d) acc[d] += p * vj[d];
    }
    double *o = J->out + (((int64_t)b * L + i) * H + h) * D;
    for (int d = 0; d < D; ++d) o[d] = acc[d];
}

static void *txlo_worker(void *arg)
{
    txlo_job *J = (txlo_job *)arg;
    const int K = J->M + J->L;
    double *s = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    double *rs = (double *)malloc(sizeof(double) * (size_t)J->D);
    double *acc = (double *)malloc(sizeof(double) * (size_t)J->D);
    int64_t total = J->sel ? J->n_sel : (int64_t)J->B * J->H * J->L;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t w = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (w >= total) break;
        int b, h, i;
        if (J->sel) {
            b = J->sel[3 * w]; h = J->sel[3 * w + 1]; i = J->sel[3 * w + 2];
        } else {
            b = (int)(w / ((int64_t)J->H * J->L));
            h = (int)((w / J->L) % J->H);
            i = (int)(w % J->L);
        }
        txlo_one_row(J, b, h, i, s, rs, acc);
    }
    free(s);
    free(rs);
    free(acc);
    return NULL;
}

/* Memo of r(delta_c) for delta_c = 0..n_memo-1, one table per needed head.  Each entry is
 * produced by txlo_rel_vec, exactly as the un-memoised path would produce it. */
typedef struct {
    int d_model, D, n_memo, h;
    int64_t ld_w;
    const double *W_R;
    double *tab;
} txlo_memo_arg;

static void *txlo_memo_worker(void *arg)
{
    txlo_memo_arg *a = (txlo_memo_arg *)arg;
    for (int dc = 0; dc < a->n_memo; ++dc)
        txlo_rel_vec((double)dc, a->d_model, a->D, a->W_R, a->ld_w, a->h,
                     a->tab + (int64_t)dc * a->D);
    return NULL;
}

static double **txlo_build_memo(int n_memo, int d_model, int H, int D, const double *W_R,
                                int64_t ld_w, const char *need, int n_threads)
{
    double **tab = (double **)calloc((size_t)H, sizeof(double *));
    txlo_memo_arg *args = (txlo_memo_arg *)calloc((size_t)H, sizeof(txlo_memo_arg));
    pthread_t *th = (pthread_t *)calloc((size_t)H, sizeof(pthread_t));
    for (int h = 0; h < H; ++h) {
        if (!need[h]) continue;
        tab[h] = (double *)malloc(sizeof(double) * (size_t)n_memo * D);
        args[h].d_model = d_model; args[h].D = D; args[h].n_memo = n_memo; args[h].h = h;
        args[h].ld_w = ld_w; args[h].W_R = W_R; args[h].tab = tab[h];
    }
    if (n_threads < 1) n_threads = 1;
    for (int h0 = 0; h0 < H; h0 += n_threads) {
        for (int h = h0; h < H && h < h0 + n_threads; ++h)
            if (need[h]) pthread_create(&th[h], NULL, txlo_memo_worker, &args[h]);
        for (int h = h0; h < H && h < h0 + n_threads; ++h)
            if (need[h]) pthread_join(th[h], NULL);
    }
    free(args);
    free(th);
    return tab;
}

static void txlo_free_memo(double **tab, int H)
{
    if (!tab) return;
    for (int h = 0; h < H; ++h) free(tab[h]);
    free(tab);
}

static char *txlo_needed_heads(int H, const int *sel, int64_t n_sel)
{
    char *need = (char *)calloc((size_t)H, 1);
    if (sel) { for (int64_t w = 0; w < n_sel; ++w) need[sel[3 * w + 1]] = 1; }
    else memset(need, 1, (size_t)H);
    return need;
}

static void txlo_run(txlo_job *J, int n_threads)
{
    if (n_threads < 1) n_threads = 1;
    pthread_mutex_init(&J->lock, NULL);
    J->next = 0;
    J->memo_tab = NULL;
    if (J->memo) {
        /* distances that can occur: delta_c in [0, min(clamp_len, M+L-1)] */
        int maxd = J->M + J->L - 1;
        if (J->clamp_len < maxd) maxd = J->clamp_len;
        J->n_memo = maxd + 1;
        char *need = txlo_needed_heads(J->H, J->sel, J->n_sel);
        J->memo_tab = txlo_build_memo(J->n_memo, J->d_model, J->H, J->D, J->W_R, J->ld_w,
                                      need, n_threads);
        free(need);
    }
    pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    for (int t = 0; t < n_threads; ++t) pthread_create(&th[t], NULL, txlo_worker, J);
    for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
    free(th);
    txlo_free_memo(J->memo_tab, J->H);
    pthread_mutex_destroy(&J->lock);
}

int txlo_rel_attn(int B, int L, int H, int D, int M, int mem_valid, int clamp_len,
                  int d_model, const double *q, const double *k, const double *v,
                  const double *u, const double *vb, const double *W_R, int64_t ld_w,
                  double scale, double *out, int memo, int n_threads,
                  const int *sel, int64_t n_sel)
{
    if (B < 0 || L < 0 || H <= 0 || D <= 0 || M < 0 || mem_valid < 0 || mem_valid > M ||
        clamp_len < 0 || d_model <= 0 || (d_model & 1))
        return -1;
    txlo_job J;
    memset(&J, 0, sizeof(J));
    J.B = B; J.L = L; J.H = H; J.D = D; J.M = M; J.mem_valid = mem_valid;
    J.clamp_len = clamp_len; J.d_model = d_model; J.ld_w = ld_w; J.scale = scale;
    J.q = q; J.k = k; J.v = v; J.u = u; J.vb = vb; J.W_R = W_R; J.out = out;
    J.memo = memo; J.sel = sel; J.n_sel = n_sel;
    txlo_run(&J, n_threads);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Segment recurrence on the concatenated sequence ([R], [K] §4.3, FIFO of mem_len from  */
/* "Transformer-XL架构解析" §1.1): the stream is cut into n_seg segments of L positions;  */
/* a query at global position t = s*L + i sees keys g in [max(0, s*L - M), t], with       */
/* delta = t - g.  The memory of segment s is the last min(s*L, M) positions before it.   */
/*   q,k,v [B][n_seg*L][H][D] ; out [B][n_seg*L][H][D]                                   */
/* sel: triples (b, h, t) of global query rows, or NULL for all.                          */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    int B, H, D, L, M, n_seg, clamp_len, d_model;
    int64_t ld_w;
    double scale;
    const double *q, *k, *v, *u, *vb, *W_R;
    double *out;
    int memo;
    double **memo_tab;
    int n_memo;
    const int *sel;
    int64_t n_sel;
    int64_t next;
    pthread_mutex_t lock;
} txlo_sjob;

static void *txlo_stream_worker(void *arg)
{
    txlo_sjob *J = (txlo_sjob *)arg;
    const int T = J->n_seg * J->L, D = J->D, H = J->H;
    double *s = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double *rs = (double *)malloc(sizeof(double) * (size_t)D);
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    int64_t total = J->sel ? J->n_sel : (int64_t)J->B * H * T;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t w = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (w >= total) break;
        int b, h, t;
        if (J->sel) { b = J->sel[3 * w]; h = J->sel[3 * w + 1]; t = J->sel[3 * w + 2]; }
        else { b = (int)(w / ((int64_t)H * T)); h = (int)((w / T) % H); t = (int)(w % T); }
        int seg = t / J->L;
        int g_lo = seg * J->L - J->M;
        if (g_lo < 0) g_lo = 0;
        const double *qt = J->q + (((int64_t)b * T + t) * H + h) * D;
        const double *uh = J->u + (int64_t)h * D, *vh = J->vb + (int64_t)h * D;
        double mx = -INFINITY;
        for (int g = g_lo; g <= t; ++g) {
            int delta = t - g;
            int dc = delta < J->clamp_len ? delta : J->clamp_len;
            const double *r;
            if (J->memo) r = J->memo_tab[h] + (int64_t)dc * D;
            else { txlo_rel_vec((double)dc, J->d_model, D, J->W_R, J->ld_w, h, rs); r = rs; }
            const double *kg = J->k + (((int64_t)b * T + g) * H + h) * D;
            s[g] = J->scale * txlo_score_terms(D, qt, kg, r, uh, vh, NULL);
            if (s[g] > mx) mx = s[g];
        }
        double den = 0.0;
        for (int g = g_lo; g <= t; ++g) { s[g] = exp(s[g] - mx); den += s[g]; }
        for (int d = 0; d < D; ++d) acc[d] = 0.0;        /* private, see txlo_one_row */
        for (int g = g_lo; g <= t; ++g) {
            double p = s[g] / den;
            const double *vg = J->v + (((int64_t)b * T + g) * H + h) * D;
            for (int d = 0; d < D; ++d) acc[d] += p * vg[d];
        }
        double *o = J->out + (((int64_t)b * T + t) * H + h) * D;
        for (int d = 0; d < D; ++d) o[d] = acc[d];
    }
    free(s);
    free(rs);
    free(acc);
    return NULL;
}

int txlo_stream_attn(int B, int H, int D, int L, int M, int n_seg, int clamp_len, int d_model,
                     const double *q, const double *k, const double *v, const double *u,
                     const double *vb, const double *W_R, int64_t ld_w, double scale,
                     double *out, int memo, int n_threads, const int *sel, int64_t n_sel)
{
    if (B < 0 || H <= 0 || D <= 0 || L <= 0 || M < 0 || n_seg <= 0 || clamp_len < 0 ||
        d_model <= 0 || (d_model & 1))
        return -1;
    if (n_threads < 1) n_threads = 1;
    txlo_sjob J;
    memset(&J, 0, sizeof(J));
    J.B = B; J.H = H; J.D = D; J.L = L; J.M = M; J.n_seg = n_seg; J.clamp_len = clamp_len;
    J.d_model = d_model; J.ld_w = ld_w; J.scale = scale;
    J.q = q; J.k = k; J.v = v; J.u = u; J.vb = vb; J.W_R = W_R; J.out = out;
    J.memo = memo; J.sel = sel; J.n_sel = n_sel;
    pthread_mutex_init(&J.lock, NULL);
    if (memo) {
        int maxd = M + L - 1;
        if (clamp_len < maxd) maxd = clamp_len;
        J.n_memo = maxd + 1;
        char *need = txlo_needed_heads(H, sel, n_sel);
        J.memo_tab = txlo_build_memo(J.n_memo, d_model, H, D, W_R, ld_w, need, n_threads);
        free(need);
    }
    pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    for (int t = 0; t < n_threads; ++t) pthread_create(&th[t], NULL, txlo_stream_worker, &J);
    for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
    free(th);
    txlo_free_memo(J.memo_tab, H);
    pthread_mutex_destroy(&J.lock);
    return 0;
}
