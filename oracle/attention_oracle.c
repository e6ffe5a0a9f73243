/*
 * Oracle for multi-head scaled dot-product attention -- TEST INFRASTRUCTURE.
 *
 * Plain, slow, obviously correct fp64 CPU code. Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the library's CUDA
 * path never calls it and shares no code, header or table with it.
 *
 * What it computes, and where the pages define it:
 *   - eq. (1), Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V, in the element
 *     form alpha_ij = exp(q_i.k_j/sqrt(d_k)) / sum_l exp(q_i.k_l/sqrt(d_k)),
 *     y_i = sum_j alpha_ij v_j
 *     ("Attention Is All You Need를 지금 다시 읽는 법" (eightmm.github.io),
 *      section "Attention 수식");
 *   - masks set the logit to -inf BEFORE the softmax so the weight is exactly 0
 *     ("[논문 리뷰]Attention Is All You Need" (kimjiil.github.io), section 3.2.3;
 *      "Attention Is All You Need 해부" (sj-techlog), section "mask는 softmax
 *      **전**에 더해야 한다"); causal: query i sees keys j <= i; key padding:
 *      keys j >= kv_len[b] are padding and receive no attention
 *      ("Attention Is All You Need 해부", the three-uses table of attention);
 *   - the max-subtraction ("pivot") before exp, which changes nothing
 *     mathematically ("Attention Is All You Need 해부", section "직접 검증");
 *   - restricted self-attention: query i considers only the keys around its
 *     own position, j in [i - window_left, i + window_right] (O(r n d) work
 *     instead of O(n^2 d); "[논문 리뷰]Attention Is All You Need"
 *     (kimjiil.github.io), section "[4] Why Self-Attention", Table 1, row
 *     "Self-Attention (restricted)"); a negative bound means "no limit on
 *     that side", so (-1, -1) is eq. (1) itself;
 *   - incremental decoding with a key/value cache: the new tokens' queries
 *     only, against the cached keys and values of every earlier position
 *     plus their own ("Attention Is All You Need 해부" (sj-techlog), section
 *     "KV cache는 추론의 같은 계산을 반복하지 않게 한다"; "[논문 리뷰]Attention
 *     Is All You Need", section 3.7 "Inference — auto-regressive 디코딩"):
 *     with L valid cache rows the n_q new tokens sit at positions
 *     L - n_q .. L - 1, and the causal rule (key j <= query position) applies;
 *   - the encoder sub-layers: output = LayerNorm(x + Sublayer(x)) (post-LN),
 *     LayerNorm(x) = gamma (x - mu) / sqrt(sigma^2 + eps) + beta over one
 *     token's features ("[논문 리뷰]Attention Is All You Need", section 3.1;
 *     "Attention Is All You Need 해부", section "4. residual connection과
 *     LayerNorm은 깊은 층을 학습 가능하게 한다"), and
 *     FFN(x) = max(0, x W_1 + b_1) W_2 + b_2 ("[논문 리뷰]", section 3.3);
 *   - MultiHead(Q,K,V) = Concat(head_1..head_h) W^O,
 *     head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V), with the per-head matrices
 *     being column block i of one [d_model, h*d] matrix
 *     ("[논문 리뷰]Attention Is All You Need", section 3.2.2).
 *
 * Readings where the pages are silent (listed with the design notes):
 *   - a query row whose every key is masked (kv_len = 0) has output 0 and
 *     weights 0;
 *   - kv_len values are clamped to [0, n_k];
 *   - causal masking is defined for n_q == n_k (query i vs key i), and so is
 *     the restricted window (query i and key i share a position);
 *   - Table 1 sizes the neighbourhood by r; the bounds are taken per side, so
 *     a neighbourhood of size r centred on the query is
 *     window_left = window_right = (r - 1) / 2 and a radius-r window is
 *     window_left = window_right = r.
 *
 * Parity pins: every function here is checked by the CPU tests against the
 * pages' worked examples, closed forms and invariants, and against
 * torch's fp64 scaled_dot_product_attention on small cases.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MASK_CAUSAL 1
#define ORACLE_MASK_KEY_PADDING 2

/* Threads of a parallel region: the caller's count, or the default team. A
 * num_threads clause, unlike omp_set_num_threads, leaves later calls alone. */
static int team(int nthreads)
{
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

static int clamp_len(int len, int n_k)
{
    if (len < 0) return 0;
    if (len > n_k) return n_k;
    return len;
}

/*
 * One query row of eq. (1).
 *   q_i [d_k], K [n_k, d_k], V [n_k, d_v] (row-major); i is the query position.
 *   scores: scratch of n_k doubles. weights (nullable) receives alpha_i.
 *   y_i [d_v] receives the output row.
 */
static void attend_row(const double *q_i, const double *K, const double *V,
                       int n_k, int d_k, int d_v, int i, int causal, int kv_len,
                       int win_left, int win_right,
                       double scale, double *scores, double *weights, double *y_i)
{
    int j, c;
    int any_allowed = 0;
    double m = -INFINITY, total = 0.0;

    /* logits s_j = (q_i . k_j) * scale, -inf where the connection is illegal */
    for (j = 0; j < n_k; ++j) {
        int allowed = (j < kv_len) && !(causal && j > i) &&
                      !(win_left >= 0 && j < i - win_left) &&
                      !(win_right >= 0 && j > i + win_right);
        if (allowed) {
            double dot = 0.0;
            for (c = 0; c < d_k; ++c) dot += q_i[c] * K[(size_t)j * d_k + c];
            scores[j] = dot * scale;
            any_allowed = 1;
            if (scores[j] > m) m = scores[j];
        } else {
            scores[j] = -INFINITY;
        }
    }

    for (c = 0; c < d_v; ++c) y_i[c] = 0.0;
    if (!any_allowed) {
        if (weights)
            for (j = 0; j < n_k; ++j) weights[j] = 0.0;
        return;
    }

    /* softmax over keys: exp(s_j - m) / sum_l exp(s_l - m); exp(-inf) = 0 */
    for (j = 0; j < n_k; ++j) {
        scores[j] = (scores[j] == -INFINITY) ? 0.0 : exp(scores[j] - m);
        total += scores[j];
    }
    for (j = 0; j < n_k; ++j) scores[j] /= total;
    if (weights)
        for (j = 0; j < n_k; ++j) weights[j] = scores[j];

    /* y_i = sum_j alpha_ij v_j */
    for (j = 0; j < n_k; ++j) {
        double a = scores[j];
        if (a == 0.0) continue;
        for (c = 0; c < d_v; ++c) y_i[c] += a * V[(size_t)j * d_v + c];
    }
}

/*
 * Scaled dot-product attention for every (batch, head, query row), optionally
 * restricted to the keys j in [i - win_left, i + win_right] (a negative bound
 * is no bound).
 * Layouts (row-major, contiguous): q [B,h,n_q,d_k], k [B,h,n_k,d_k],
 * v [B,h,n_k,d_v], out [B,h,n_q,d_v], weights (nullable) [B,h,n_q,n_k].
 * kv_lens: int32[B] or NULL (used only with the key-padding mask bit).
 * Returns 0 on success, -1 on invalid arguments.
 */
int oracle_attention_window(const double *q, const double *k, const double *v, double *out,
                            double *weights, int B, int h, int n_q, int n_k, int d_k, int d_v,
                            int mask_kind, const int32_t *kv_lens, int win_left, int win_right,
                            double scale, int nthreads)
{
    int bh;
    int causal = (mask_kind & ORACLE_MASK_CAUSAL) != 0;
    int padding = (mask_kind & ORACLE_MASK_KEY_PADDING) != 0;
    int windowed = win_left >= 0 || win_right >= 0;
    if (B < 0 || h < 0 || n_q < 0 || n_k < 0 || d_k <= 0 || d_v <= 0) return -1;
    if (padding && !kv_lens) return -1;
    if ((causal || windowed) && n_q != n_k) return -1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic) num_threads(team(nthreads))
#endif
    for (bh = 0; bh < B * h; ++bh) {
        int b = bh / h, i;
        int kv_len = padding ? clamp_len(kv_lens[b], n_k) : n_k;
        const double *K = k + (size_t)bh * n_k * d_k;
        const double *V = v + (size_t)bh * n_k * d_v;
        double *scores = (double *)malloc(sizeof(double) * (size_t)(n_k > 0 ? n_k : 1));
        for (i = 0; i < n_q; ++i) {
            attend_row(q + ((size_t)bh * n_q + i) * d_k, K, V, n_k, d_k, d_v, i, causal,
                       kv_len, win_left, win_right, scale,
                       scores, weights ? weights + ((size_t)bh * n_q + i) * n_k : NULL,
                       out + ((size_t)bh * n_q + i) * d_v);
        }
        free(scores);
    }
    return 0;
}

/* eq. (1) with the optional masks and no window. */
int oracle_attention(const double *q, const double *k, const double *v, double *out,
                     double *weights, int B, int h, int n_q, int n_k, int d_k, int d_v,
                     int mask_kind, const int32_t *kv_lens, double scale, int nthreads)
{
    return oracle_attention_window(q, k, v, out, weights, B, h, n_q, n_k, d_k, d_v, mask_kind,
                                   kv_lens, -1, -1, scale, nthreads);
}

/*
 * Selected query rows of one (batch, head): rows q_rows [R, d_k] sit at query
 * positions row_pos[R]; K [n_k, d_k], V [n_k, d_v]; out [R, d_v].
 * kv_len < 0 means "no padding". Rows are independent, so this equals the
 * corresponding rows of oracle_attention.
 */
int oracle_attention_rows_window(const double *q_rows, const int32_t *row_pos, int R,
                                 const double *K, const double *V, int n_k, int d_k, int d_v,
                                 int causal, int kv_len, int win_left, int win_right,
                                 double scale, double *out, int nthreads)
{
    int r;
    int len = kv_len < 0 ? n_k : clamp_len(kv_len, n_k);
    if (R < 0 || n_k < 0 || d_k <= 0 || d_v <= 0) return -1;
#ifdef _OPENMP
#pragma omp parallel num_threads(team(nthreads))
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(n_k > 0 ? n_k : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
        for (r = 0; r < R; ++r)
            attend_row(q_rows + (size_t)r * d_k, K, V, n_k, d_k, d_v, row_pos[r], causal, len,
                       win_left, win_right, scale, scores, NULL, out + (size_t)r * d_v);
        free(scores);
    }
    return 0;
}

int oracle_attention_rows(const double *q_rows, const int32_t *row_pos, int R,
                          const double *K, const double *V, int n_k, int d_k, int d_v,
                          int causal, int kv_len, double scale, double *out, int nthreads)
{
    return oracle_attention_rows_window(q_rows, row_pos, R, K, V, n_k, d_k, d_v, causal, kv_len,
                                        -1, -1, scale, out, nthreads);
}

/*
 * Decoding step against a key/value cache. q [B,h,n_q,d_k] are the queries of
 * the n_q newest tokens; k_cache [B,h,n_max,d_k], v_cache [B,h,n_max,d_v]
 * hold every position so far (the new tokens' own keys and values included);
 * cache_lens int32[B] (NULL = n_max) gives the valid rows L of each batch
 * entry (clamped to [0, n_max]). Query t sits at position L - n_q + t and
 * sees the keys j <= that position (j < L); a query at a negative position
 * sees none and gets 0. out [B,h,n_q,d_v].
 */
int oracle_decode(const double *q, const double *k_cache, const double *v_cache, double *out,
                  int B, int h, int n_q, int n_max, int d_k, int d_v, const int32_t *cache_lens,
                  double scale, int nthreads)
{
    int bh;
    if (B < 0 || h < 0 || n_q < 0 || n_max < 0 || d_k <= 0 || d_v <= 0) return -1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic) num_threads(team(nthreads))
#endif
    for (bh = 0; bh < B * h; ++bh) {
        int b = bh / h, t;
        int L = cache_lens ? clamp_len(cache_lens[b], n_max) : n_max;
        const double *K = k_cache + (size_t)bh * n_max * d_k;
        const double *V = v_cache + (size_t)bh * n_max * d_v;
        double *scores = (double *)malloc(sizeof(double) * (size_t)(n_max > 0 ? n_max : 1));
        for (t = 0; t < n_q; ++t) {
            int pos = L - n_q + t;
            attend_row(q + ((size_t)bh * n_q + t) * d_k, K, V, n_max, d_k, d_v, pos, 1, L, -1, -1,
                       scale, scores, NULL, out + ((size_t)bh * n_q + t) * d_v);
        }
        free(scores);
    }
    return 0;
}

/* C[M,N] = A[M,K] B[K,N], plain triple loop (row-major). */
static void matmul(const double *A, const double *Bm, double *C, int M, int N, int K,
                   int nthreads)
{
    int i;
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(team(nthreads))
#endif
    for (i = 0; i < M; ++i) {
        int j, p;
        double *c = C + (size_t)i * N;
        for (j = 0; j < N; ++j) c[j] = 0.0;
        for (p = 0; p < K; ++p) {
            double a = A[(size_t)i * K + p];
            const double *b = Bm + (size_t)p * N;
            for (j = 0; j < N; ++j) c[j] += a * b[j];
        }
    }
}

/*
 * Multi-head attention, section 3.2.2 of "[논문 리뷰]Attention Is All You Need":
 *   Q = X_q W_Q, K = X_kv W_K, V = X_kv W_V            (x.W convention, no biases)
 *   head_i = Attention(Q[:, i*d_k:(i+1)*d_k], K[:, i*d_k:...], V[:, i*d_v:...])
 *   out = Concat(head_1..head_h) W_O
 * Layouts: x_q [B,n_q,d_model], x_kv [B,n_k,d_model], w_q/w_k [d_model,h*d_k],
 * w_v [d_model,h*d_v], w_o [h*d_v,d_model], out [B,n_q,d_model].
 * concat_out (nullable) receives Concat(head_1..head_h) [B,n_q,h*d_v].
 */
int oracle_mha(const double *x_q, const double *x_kv, const double *w_q, const double *w_k,
               const double *w_v, const double *w_o, double *out, double *concat_out,
               int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
               int mask_kind, const int32_t *kv_lens, double scale, int nthreads)
{
    int b, hh, i, c, rc = 0;
    size_t qsz = (size_t)B * n_q * h * d_k, ksz = (size_t)B * n_k * h * d_k;
    size_t vsz = (size_t)B * n_k * h * d_v, osz = (size_t)B * n_q * h * d_v;
    double *Q, *Kp, *Vp, *Qh, *Kh, *Vh, *Oh, *concat;
    if (B < 0 || n_q < 0 || n_k < 0 || d_model <= 0 || h <= 0 || d_k <= 0 || d_v <= 0) return -1;
    Q = (double *)malloc(sizeof(double) * (qsz ? qsz : 1));
    Kp = (double *)malloc(sizeof(double) * (ksz ? ksz : 1));
    Vp = (double *)malloc(sizeof(double) * (vsz ? vsz : 1));
    Qh = (double *)malloc(sizeof(double) * (qsz ? qsz : 1));
    Kh = (double *)malloc(sizeof(double) * (ksz ? ksz : 1));
    Vh = (double *)malloc(sizeof(double) * (vsz ? vsz : 1));
    Oh = (double *)malloc(sizeof(double) * (osz ? osz : 1));
    concat = (double *)malloc(sizeof(double) * (osz ? osz : 1));

    /* projections of all positions at once */
    matmul(x_q, w_q, Q, B * n_q, h * d_k, d_model, nthreads);
    matmul(x_kv, w_k, Kp, B * n_k, h * d_k, d_model, nthreads);
    matmul(x_kv, w_v, Vp, B * n_k, h * d_v, d_model, nthreads);

    /* head split: head hh takes column block hh of each projection */
    for (b = 0; b < B; ++b)
        for (hh = 0; hh < h; ++hh) {
            for (i = 0; i < n_q; ++i)
                for (c = 0; c < d_k; ++c)
                    Qh[(((size_t)b * h + hh) * n_q + i) * d_k + c] =
                        Q[((size_t)b * n_q + i) * h * d_k + (size_t)hh * d_k + c];
            for (i = 0; i < n_k; ++i) {
                for (c = 0; c < d_k; ++c)
                    Kh[(((size_t)b * h + hh) * n_k + i) * d_k + c] =
                        Kp[((size_t)b * n_k + i) * h * d_k + (size_t)hh * d_k + c];
                for (c = 0; c < d_v; ++c)
                    Vh[(((size_t)b * h + hh) * n_k + i) * d_v + c] =
                        Vp[((size_t)b * n_k + i) * h * d_v + (size_t)hh * d_v + c];
            }
        }

    rc = oracle_attention(Qh, Kh, Vh, Oh, NULL, B, h, n_q, n_k, d_k, d_v, mask_kind, kv_lens,
                          scale, nthreads);

    /* head merge: Concat(head_1..head_h) along the feature axis */
    if (rc == 0) {
        for (b = 0; b < B; ++b)
            for (hh = 0; hh < h; ++hh)
                for (i = 0; i < n_q; ++i)
                    for (c = 0; c < d_v; ++c)
                        concat[((size_t)b * n_q + i) * h * d_v + (size_t)hh * d_v + c] =
                            Oh[(((size_t)b * h + hh) * n_q + i) * d_v + c];
        if (concat_out)
            for (size_t t = 0; t < osz; ++t) concat_out[t] = concat[t];
        matmul(concat, w_o, out, B * n_q, d_model, h * d_v, nthreads);
    }

    free(Q); free(Kp); free(Vp); free(Qh); free(Kh); free(Vh); free(Oh); free(concat);
    return rc;
}

/*
 * LayerNorm over the last axis: out[r] = gamma * (x[r] - mu) / sqrt(var + eps)
 * + beta, mu and var (the population variance) over the d features of row r.
 * x may alias out.
 */
void oracle_layernorm(const double *x, const double *gamma, const double *beta, double *out,
                      int rows, int d, double eps)
{
    int r, c;
    for (r = 0; r < rows; ++r) {
        const double *xr = x + (size_t)r * d;
        double mu = 0.0, var = 0.0, inv;
        for (c = 0; c < d; ++c) mu += xr[c];
        mu /= d;
        for (c = 0; c < d; ++c) var += (xr[c] - mu) * (xr[c] - mu);
        var /= d;
        inv = 1.0 / sqrt(var + eps);
        for (c = 0; c < d; ++c) out[(size_t)r * d + c] = gamma[c] * (xr[c] - mu) * inv + beta[c];
    }
}

/* FFN(x) = max(0, x W_1 + b_1) W_2 + b_2 for rows x [rows, d_model];
 * w_1 [d_model, d_ff], w_2 [d_ff, d_model]; out [rows, d_model]. */
int oracle_ffn(const double *x, const double *w_1, const double *b_1, const double *w_2,
               const double *b_2, double *out, int rows, int d_model, int d_ff, int nthreads)
{
    int r, c;
    double *hid;
    if (rows < 0 || d_model <= 0 || d_ff <= 0) return -1;
    hid = (double *)malloc(sizeof(double) * ((size_t)rows * d_ff ? (size_t)rows * d_ff : 1));
    matmul(x, w_1, hid, rows, d_ff, d_model, nthreads);
    for (r = 0; r < rows; ++r)
        for (c = 0; c < d_ff; ++c) {
            double v = hid[(size_t)r * d_ff + c] + b_1[c];
            hid[(size_t)r * d_ff + c] = v > 0.0 ? v : 0.0;
        }
    matmul(hid, w_2, out, rows, d_model, d_ff, nthreads);
    for (r = 0; r < rows; ++r)
        for (c = 0; c < d_model; ++c) out[(size_t)r * d_model + c] += b_2[c];
    free(hid);
    return 0;
}

/*
 * One encoder layer (self-attention sub-layer, then the feed-forward one,
 * each wrapped as LayerNorm(x + Sublayer(x))):
 *   y   = LayerNorm_1(x + MultiHead(x, x))
 *   out = LayerNorm_2(y + FFN(y))
 * x [B, n, d_model]; the attention weights and mask as oracle_mha; LayerNorm
 * parameters [d_model]; FFN as oracle_ffn. y_out (nullable) receives y.
 */
int oracle_encoder_layer(const double *x, const double *w_q, const double *w_k,
                         const double *w_v, const double *w_o, const double *g_1,
                         const double *be_1, const double *w_1, const double *b_1,
                         const double *w_2, const double *b_2, const double *g_2,
                         const double *be_2, double *out, double *y_out, int B, int n,
                         int d_model, int h, int d_k, int d_ff, int mask_kind,
                         const int32_t *kv_lens, double scale, double eps, int nthreads)
{
    size_t rows = (size_t)B * n, t;
    size_t sz = rows * d_model;
    double *att, *y, *f;
    int rc;
    if (B < 0 || n < 0 || d_model <= 0 || h <= 0 || d_k <= 0 || d_ff <= 0) return -1;
    att = (double *)malloc(sizeof(double) * (sz ? sz : 1));
    y = (double *)malloc(sizeof(double) * (sz ? sz : 1));
    f = (double *)malloc(sizeof(double) * (sz ? sz : 1));
    rc = oracle_mha(x, x, w_q, w_k, w_v, w_o, att, NULL, B, n, n, d_model, h, d_k, d_k,
                    mask_kind, kv_lens, scale, nthreads);
    if (rc == 0) {
        for (t = 0; t < sz; ++t) y[t] = x[t] + att[t];
        oracle_layernorm(y, g_1, be_1, y, (int)rows, d_model, eps);
        if (y_out)
            for (t = 0; t < sz; ++t) y_out[t] = y[t];
        rc = oracle_ffn(y, w_1, b_1, w_2, b_2, f, (int)rows, d_model, d_ff, nthreads);
    }
    if (rc == 0) {
        for (t = 0; t < sz; ++t) f[t] += y[t];
        oracle_layernorm(f, g_2, be_2, out, (int)rows, d_model, eps);
    }
    free(att); free(y); free(f);
    return rc;
}

/* Number of threads an OpenMP parallel region would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
