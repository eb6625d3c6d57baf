/*
 * ORACLE — test infrastructure, not product code.
 *
 * A plain, slow, fp64 CPU restatement of multi-head scaled dot-product
 * attention and of the post-norm multi-head-attention sublayer, written from
 * the explanatory pages on "Attention Is All You Need". Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg call it. It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * Conventions (the pages' notation):
 *   - activations are [B, n, h, d] row-major: head i of token t of batch b is
 *     the d-vector at ((b*n + t)*h + i)*d, i.e. the heads are concatenated
 *     along the feature axis exactly as X.W^Q produces them;
 *   - W^Q, W^K are [d_model, h*d_k], W^V is [d_model, h*d_v] and W^O is
 *     [h*d_v, d_model], all row-major, column block i belongs to head i;
 *   - mask_kind bit 0 (CAUSAL): key j is invisible to query t when j > t;
 *     mask_kind bit 1 (KEY_PADDING): key j is invisible when j >= key_lens[b].
 *
 * Every function is pinned by the tests in tests/test_oracle_pins.py against
 * values the pages print, closed forms, invariants and brute force.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_EEMPTY (-2) /* a query row with no visible key */
#define ORACLE_ENOMEM (-3)

#define ORACLE_MASK_CAUSAL 1
#define ORACLE_MASK_KEY_PADDING 2

/*
 * Row softmax over the visible entries of s[0..n).
 *
 * [hex4c59 "读懂 Attention Is All You Need", §六步算完一行注意力, step 3]: the
 * j-th weight is e^{s_j} / sum_k e^{s_k}; the weights are non-negative and sum
 * to 1. [same page, §用几十行代码核对刚才的数值]: subtracting the row maximum
 * first gives the same result and keeps the exponentials bounded.
 * [same page, §掩码必须在 softmax 之前生效]: a masked score is -inf before the
 * softmax, so its weight is exactly 0 (never e^0 = 1).
 * Returns ORACLE_EEMPTY when no entry is visible.
 */
int oracle_softmax(const double* s, const unsigned char* visible, int n, double* w)
{
    double m = -INFINITY;
    int any = 0;
    for (int j = 0; j < n; ++j) {
        if (visible && !visible[j]) continue;
        if (!any || s[j] > m) m = s[j];
        any = 1;
    }
    if (!any) {
        for (int j = 0; j < n; ++j) w[j] = 0.0;
        return ORACLE_EEMPTY;
    }
    double denom = 0.0;
    for (int j = 0; j < n; ++j) {
        if (visible && !visible[j]) {
            w[j] = 0.0;
            continue;
        }
        w[j] = exp(s[j] - m);
        denom += w[j];
    }
    for (int j = 0; j < n; ++j) w[j] /= denom;
    return ORACLE_OK;
}

/*
 * One query row of one head: out = softmax(scale * q.K^T [masked]) V.
 *
 * [hex4c59, §六步算完一行注意力]: step 1 dot products of the query with every
 * key, step 2 division by sqrt(d_k) (here the general `scale`), step 3 row
 * softmax, step 4 weighted sum of the value rows.
 * [hex4c59, §把所有位置合并，就是那条核心公式]: rows of the score matrix are
 * "who queries", columns "whom"; the softmax runs along each row.
 * [hex4c59, §掩码必须在 softmax 之前生效]: key j > t is invisible under the
 * causal mask (the diagonal stays visible); padding keys are invisible too.
 *
 * k0/v0 point at key 0 of this (batch, head); consecutive keys are
 * k_stride/v_stride doubles apart. s and vis are n_k-long scratch.
 */
static int attend_row(const double* q_row, const double* k0, const double* v0,
                      ptrdiff_t k_stride, ptrdiff_t v_stride, int n_k, int d_k, int d_v,
                      double scale, int t, int causal, int kv_len,
                      double* s, unsigned char* vis, double* w, double* out_row)
{
    for (int j = 0; j < n_k; ++j) {
        const double* k_row = k0 + (ptrdiff_t)j * k_stride;
        double dot = 0.0;
        for (int c = 0; c < d_k; ++c) dot += q_row[c] * k_row[c];
        s[j] = scale * dot;
        vis[j] = (unsigned char)(!(causal && j > t) && j < kv_len);
    }
    int rc = oracle_softmax(s, vis, n_k, w);
    for (int c = 0; c < d_v; ++c) out_row[c] = 0.0;
    if (rc != ORACLE_OK) return rc;
    for (int j = 0; j < n_k; ++j) {
        if (w[j] == 0.0) continue;
        const double* v_row = v0 + (ptrdiff_t)j * v_stride;
        for (int c = 0; c < d_v; ++c) out_row[c] += w[j] * v_row[c];
    }
    return ORACLE_OK;
}

static int check_attn_args(int B, int h, int n_q, int n_k, int d_k, int d_v, int mask_kind,
                           const int32_t* key_lens)
{
    if (B <= 0 || h <= 0 || n_q <= 0 || n_k <= 0 || d_k <= 0 || d_v <= 0) return ORACLE_EINVAL;
    if (mask_kind & ~(ORACLE_MASK_CAUSAL | ORACLE_MASK_KEY_PADDING)) return ORACLE_EINVAL;
    if (mask_kind & ORACLE_MASK_KEY_PADDING) {
        if (!key_lens) return ORACLE_EINVAL;
        for (int b = 0; b < B; ++b)
            if (key_lens[b] < 1 || key_lens[b] > n_k) return ORACLE_EINVAL;
    }
    return ORACLE_OK;
}

/*
 * Selected rows of multi-head attention. sel holds n_sel triples (b, t, i):
 * batch, query position, head. out_rows is n_sel x d_v; w_rows (optional) is
 * n_sel x n_k and receives the attention weights of each selected row.
 * [hex4c59, §多头注意力让一次读取有多组投影]: every head runs the same
 * scaled dot-product attention on its own slice of Q, K and V.
 */
int oracle_attn_rows(const double* q, const double* k, const double* v, int B, int h, int n_q,
                     int n_k, int d_k, int d_v, double scale, int mask_kind,
                     const int32_t* key_lens, const int32_t* sel, int n_sel, double* out_rows,
                     double* w_rows, int nthreads)
{
    int rc = check_attn_args(B, h, n_q, n_k, d_k, d_v, mask_kind, key_lens);
    if (rc != ORACLE_OK) return rc;
    for (int r = 0; r < n_sel; ++r) {
        int b = sel[3 * r], t = sel[3 * r + 1], i = sel[3 * r + 2];
        if (b < 0 || b >= B || t < 0 || t >= n_q || i < 0 || i >= h) return ORACLE_EINVAL;
    }
    int err = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)n_k);
        double* w = (double*)malloc(sizeof(double) * (size_t)n_k);
        unsigned char* vis = (unsigned char*)malloc((size_t)n_k);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n_sel; ++r) {
            if (!s || !w || !vis) {
#pragma omp atomic write
                err = ORACLE_ENOMEM;
                continue;
            }
            {
                int b = sel[3 * r], t = sel[3 * r + 1], i = sel[3 * r + 2];
                const double* q_row = q + (((size_t)b * n_q + t) * h + i) * (size_t)d_k;
                const double* k0 = k + ((size_t)b * n_k * h + i) * (size_t)d_k;
                const double* v0 = v + ((size_t)b * n_k * h + i) * (size_t)d_v;
                int kv_len = (mask_kind & ORACLE_MASK_KEY_PADDING) ? key_lens[b] : n_k;
                int row_rc = attend_row(q_row, k0, v0, (ptrdiff_t)h * d_k, (ptrdiff_t)h * d_v, n_k,
                                        d_k, d_v, scale, t, mask_kind & ORACLE_MASK_CAUSAL, kv_len,
                                        s, vis, w, out_rows + (size_t)r * d_v);
                if (w_rows) memcpy(w_rows + (size_t)r * n_k, w, sizeof(double) * (size_t)n_k);
                if (row_rc != ORACLE_OK) {
#pragma omp atomic write
                    err = row_rc;
                }
            }
        }
        free(s);
        free(w);
        free(vis);
    }
    return err;
}

/*
 * Full multi-head attention: out[b,t,i,:] for every batch, query and head,
 * written in the same [B, n_q, h, d_v] layout (the concatenation of heads).
 * [hex4c59, §把所有位置合并，就是那条核心公式]: Attention(Q,K,V) =
 * softmax(Q K^T / sqrt(d_k)) V, applied to every query row at once.
 */
int oracle_attn(const double* q, const double* k, const double* v, double* out, int B, int h,
                int n_q, int n_k, int d_k, int d_v, double scale, int mask_kind,
                const int32_t* key_lens, int nthreads)
{
    int rc = check_attn_args(B, h, n_q, n_k, d_k, d_v, mask_kind, key_lens);
    if (rc != ORACLE_OK) return rc;
    size_t n_rows = (size_t)B * n_q * h;
    int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * 3 * n_rows);
    if (!sel) return ORACLE_ENOMEM;
    size_t r = 0;
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < n_q; ++t)
            for (int i = 0; i < h; ++i, ++r) {
                sel[3 * r] = b;
                sel[3 * r + 1] = t;
                sel[3 * r + 2] = i;
            }
    /* Row r of the selection is exactly row r of out in [B, n_q, h, d_v]. */
    rc = oracle_attn_rows(q, k, v, B, h, n_q, n_k, d_k, d_v, scale, mask_kind, key_lens, sel,
                          (int)n_rows, out, NULL, nthreads);
    free(sel);
    return rc;
}

/*
 * C[M,N] = A[M,K] . W[K,N], all row-major, fp64. A plain matrix product: the
 * linear projection Q = X W^Q of [hex4c59, §Q、K、V 是三种计算角色].
 */
void oracle_matmul(const double* A, const double* W, double* C, int M, int K, int N, int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m) {
        double* c_row = C + (size_t)m * N;
        for (int n = 0; n < N; ++n) c_row[n] = 0.0;
        for (int kk = 0; kk < K; ++kk) {
            double a = A[(size_t)m * K + kk];
            const double* w_row = W + (size_t)kk * N;
            for (int n = 0; n < N; ++n) c_row[n] += a * w_row[n];
        }
    }
}

/*
 * LayerNorm of one d-vector: y = gamma * (z - mu) / sqrt(sigma^2 + eps) + beta,
 * mu and sigma^2 the mean and the biased (divide by d) variance of z.
 * [hex4c59, §Add & Norm 里究竟发生了什么？]: normalisation runs over one
 * token's feature dimension with learnable gamma, beta and a small epsilon.
 */
void oracle_layernorm_row(const double* z, const double* gamma, const double* beta, double eps,
                          int d, double* y)
{
    double mu = 0.0;
    for (int c = 0; c < d; ++c) mu += z[c];
    mu /= d;
    double var = 0.0;
    for (int c = 0; c < d; ++c) var += (z[c] - mu) * (z[c] - mu);
    var /= d;
    double inv = 1.0 / sqrt(var + eps);
    for (int c = 0; c < d; ++c) y[c] = gamma[c] * (z[c] - mu) * inv + beta[c];
}

static int check_mha_args(int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                          int mask_kind, const int32_t* key_lens)
{
    if (d_model <= 0) return ORACLE_EINVAL;
    return check_attn_args(B, h, n_q, n_k, d_k, d_v, mask_kind, key_lens);
}

/*
 * The post-norm multi-head-attention sublayer:
 *   Q = X_q W^Q, K = X_kv W^K, V = X_kv W^V                 (no biases)
 *   A = Concat_i Attention(Q_i, K_i, V_i)                    (scale 1/sqrt(d_k))
 *   y = LayerNorm(X_q + A W^O)
 * [hex4c59, §多头注意力让一次读取有多组投影] for the heads and W^O;
 * [hex4c59, §Add & Norm 里究竟发生了什么？] for residual-then-normalise
 * (post-LN); [hex4c59, §解码器有两种读取] for X_kv != X_q (cross-attention).
 * Optional q_out/k_out/v_out/a_out receive the fp64 intermediates.
 */
int oracle_mha(const double* x_q, const double* x_kv, const double* Wq, const double* Wk,
               const double* Wv, const double* Wo, const double* gamma, const double* beta,
               double eps, double* y, int B, int n_q, int n_k, int d_model, int h, int d_k,
               int d_v, int mask_kind, const int32_t* key_lens, int nthreads, double* q_out,
               double* k_out, double* v_out, double* a_out)
{
    int rc = check_mha_args(B, n_q, n_k, d_model, h, d_k, d_v, mask_kind, key_lens);
    if (rc != ORACLE_OK) return rc;
    size_t Mq = (size_t)B * n_q, Mk = (size_t)B * n_k;
    int hdk = h * d_k, hdv = h * d_v;
    double* Q = q_out ? q_out : (double*)malloc(sizeof(double) * Mq * hdk);
    double* K = k_out ? k_out : (double*)malloc(sizeof(double) * Mk * hdk);
    double* V = v_out ? v_out : (double*)malloc(sizeof(double) * Mk * hdv);
    double* A = a_out ? a_out : (double*)malloc(sizeof(double) * Mq * hdv);
    double* Z = (double*)malloc(sizeof(double) * Mq * d_model);
    if (!Q || !K || !V || !A || !Z) {
        rc = ORACLE_ENOMEM;
        goto done;
    }
    oracle_matmul(x_q, Wq, Q, (int)Mq, d_model, hdk, nthreads);
    oracle_matmul(x_kv, Wk, K, (int)Mk, d_model, hdk, nthreads);
    oracle_matmul(x_kv, Wv, V, (int)Mk, d_model, hdv, nthreads);
    rc = oracle_attn(Q, K, V, A, B, h, n_q, n_k, d_k, d_v, 1.0 / sqrt((double)d_k), mask_kind,
                     key_lens, nthreads);
    if (rc != ORACLE_OK) goto done;
    oracle_matmul(A, Wo, Z, (int)Mq, hdv, d_model, nthreads);
    for (size_t r = 0; r < Mq; ++r) {
        double* z = Z + r * d_model;
        const double* x = x_q + r * d_model;
        for (int c = 0; c < d_model; ++c) z[c] += x[c];
        oracle_layernorm_row(z, gamma, beta, eps, d_model, y + r * d_model);
    }
done:
    if (!q_out) free(Q);
    if (!k_out) free(K);
    if (!v_out) free(V);
    if (!a_out) free(A);
    free(Z);
    return rc;
}

/*
 * Selected output rows of the sublayer, for problems too large to run whole.
 * sel holds n_sel pairs (b, t); y_rows is n_sel x d_model. Computes K and V
 * of each batch that a selected row belongs to, then the row's own Q, its
 * heads, A W^O, the residual and the LayerNorm (same steps as oracle_mha).
 */
int oracle_mha_rows(const double* x_q, const double* x_kv, const double* Wq, const double* Wk,
                    const double* Wv, const double* Wo, const double* gamma, const double* beta,
                    double eps, int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v,
                    int mask_kind, const int32_t* key_lens, const int32_t* sel, int n_sel,
                    double* y_rows, int nthreads)
{
    int rc = check_mha_args(B, n_q, n_k, d_model, h, d_k, d_v, mask_kind, key_lens);
    if (rc != ORACLE_OK) return rc;
    for (int r = 0; r < n_sel; ++r) {
        int b = sel[2 * r], t = sel[2 * r + 1];
        if (b < 0 || b >= B || t < 0 || t >= n_q) return ORACLE_EINVAL;
    }
    int hdk = h * d_k, hdv = h * d_v;
    double* K = (double*)malloc(sizeof(double) * (size_t)n_k * hdk);
    double* V = (double*)malloc(sizeof(double) * (size_t)n_k * hdv);
    double* q = (double*)malloc(sizeof(double) * hdk);
    double* a = (double*)malloc(sizeof(double) * hdv);
    double* z = (double*)malloc(sizeof(double) * d_model);
    double* s = (double*)malloc(sizeof(double) * (size_t)n_k);
    double* w = (double*)malloc(sizeof(double) * (size_t)n_k);
    unsigned char* vis = (unsigned char*)malloc((size_t)n_k);
    int cur_b = -1;
    if (!K || !V || !q || !a || !z || !s || !w || !vis) {
        rc = ORACLE_ENOMEM;
        goto done;
    }
    for (int r = 0; r < n_sel && rc == ORACLE_OK; ++r) {
        int b = sel[2 * r], t = sel[2 * r + 1];
        if (b != cur_b) {
            oracle_matmul(x_kv + (size_t)b * n_k * d_model, Wk, K, n_k, d_model, hdk, nthreads);
            oracle_matmul(x_kv + (size_t)b * n_k * d_model, Wv, V, n_k, d_model, hdv, nthreads);
            cur_b = b;
        }
        const double* x = x_q + ((size_t)b * n_q + t) * d_model;
        oracle_matmul(x, Wq, q, 1, d_model, hdk, 1);
        int kv_len = (mask_kind & ORACLE_MASK_KEY_PADDING) ? key_lens[b] : n_k;
        for (int i = 0; i < h && rc == ORACLE_OK; ++i)
            rc = attend_row(q + (size_t)i * d_k, K + (size_t)i * d_k, V + (size_t)i * d_v,
                            (ptrdiff_t)hdk, (ptrdiff_t)hdv, n_k, d_k, d_v,
                            1.0 / sqrt((double)d_k), t, mask_kind & ORACLE_MASK_CAUSAL, kv_len,
                            s, vis, w, a + (size_t)i * d_v);
        if (rc != ORACLE_OK) break;
        oracle_matmul(a, Wo, z, 1, hdv, d_model, 1);
        for (int c = 0; c < d_model; ++c) z[c] += x[c];
        oracle_layernorm_row(z, gamma, beta, eps, d_model, y_rows + (size_t)r * d_model);
    }
done:
    free(K);
    free(V);
    free(q);
    free(a);
    free(z);
    free(s);
    free(w);
    free(vis);
    return rc;
}

/*
 * Sinusoidal positional encoding added to scaled embeddings:
 *   out[b,t,2i]   = emb_scale * emb[b,t,2i]   + sin((pos0 + t) / 10000^(2i/d_model))
 *   out[b,t,2i+1] = emb_scale * emb[b,t,2i+1] + cos((pos0 + t) / 10000^(2i/d_model))
 * [research-heat "做法 · Attention Is All You Need", §去掉循环，因而须补回顺序]:
 * PE(pos, 2i) = sin(pos / 10000^(2i/d_model)), PE(pos, 2i+1) = cos(...);
 * [hex4c59, §没有循环，模型怎样知道词序？]: the embedding, multiplied by
 * sqrt(d_model), and the encoding are added. emb may be NULL (encoding only).
 * d_model must be even.
 */
int oracle_pos_encoding(const double* emb, double* out, int B, int n, int d_model,
                        double emb_scale, int pos0)
{
    if (B <= 0 || n <= 0 || d_model <= 0 || (d_model & 1)) return ORACLE_EINVAL;
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < n; ++t)
            for (int i = 0; i < d_model / 2; ++i) {
                const double angle = (double)(pos0 + t) / pow(10000.0, 2.0 * i / d_model);
                const size_t at = ((size_t)b * n + t) * d_model + 2 * i;
                const double e0 = emb ? emb_scale * emb[at] : 0.0;
                const double e1 = emb ? emb_scale * emb[at + 1] : 0.0;
                out[at] = e0 + sin(angle);
                out[at + 1] = e1 + cos(angle);
            }
    return ORACLE_OK;
}

/*
 * The post-norm position-wise feed-forward sublayer, row by row:
 *   h = max(0, x W1 + b1)          (d_model -> d_ff, ReLU)
 *   f = h W2 + b2                  (d_ff -> d_model)
 *   y = LayerNorm(x + f)
 * [devpress "【深度学习】Transformer（Attention Is All You Need）", §2.3]:
 * x + FFN(x) = x + max(0, x W1 + b1) W2 + b2, followed by norm2(x + FFN(x));
 * [hex4c59, §前馈网络为什么放在注意力后面？]: the same FFN is applied to every
 * position independently (a row never reads another row), ReLU zeroes
 * negatives, the base model widens 512 -> 2048 -> 512.
 * W1 is [d_model, d_ff], W2 [d_ff, d_model], row-major; x and y are
 * [rows, d_model]. Rows are independent, so any subset of rows may be passed.
 */
int oracle_ffn(const double* x, const double* W1, const double* b1, const double* W2,
               const double* b2, const double* gamma, const double* beta, double eps, double* y,
               int rows, int d_model, int d_ff, int nthreads)
{
    if (rows <= 0 || d_model <= 0 || d_ff <= 0) return ORACLE_EINVAL;
    int rc = ORACLE_OK;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double* hid = (double*)malloc(sizeof(double) * (size_t)d_ff);
        double* z = (double*)malloc(sizeof(double) * (size_t)d_model);
        if (!hid || !z) {
#pragma omp atomic write
            rc = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(static)
            for (int r = 0; r < rows; ++r) {
                const double* xr = x + (size_t)r * d_model;
                for (int j = 0; j < d_ff; ++j) {
                    double acc = b1[j];
                    for (int c = 0; c < d_model; ++c) acc += xr[c] * W1[(size_t)c * d_ff + j];
                    hid[j] = acc > 0.0 ? acc : 0.0;
                }
                for (int c = 0; c < d_model; ++c) {
                    double acc = b2[c];
                    for (int j = 0; j < d_ff; ++j) acc += hid[j] * W2[(size_t)j * d_model + c];
                    z[c] = xr[c] + acc;
                }
                oracle_layernorm_row(z, gamma, beta, eps, d_model, y + (size_t)r * d_model);
            }
        }
        free(hid);
        free(z);
    }
    return rc;
}

/*
 * Gradients of multi-head attention, and the per-row log-sum-exp of the
 * forward pass.
 *
 * Training sends the loss gradient back through the attention weights and the
 * projections ([hex4c59, §参数是怎样学出来的？]; all target positions are trained
 * at once under the causal mask, §训练能并行，不意味着一次生成整句话). The pages
 * print no backward formulas; these are the chain rule applied to the forward
 * definition above, per (batch, head) and query row i:
 *   s_ij  = scale * q_i . k_j            (visible keys only)
 *   P_ij  = softmax_j(s_ij)              (0 for invisible keys)
 *   O_i   = sum_j P_ij v_j
 * with upstream gradient dO:
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)      (softmax Jacobian)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_i dS_ij q_i
 * lse (optional, [B, h, n_q]) receives ln sum_j exp(s_ij) over visible keys.
 * Layouts as oracle_attn; dq/dk/dv have the shapes of q/k/v.
 */
int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                    int B, int h, int n_q, int n_k, int d_k, int d_v, double scale, int mask_kind,
                    const int32_t* key_lens, double* dq, double* dk, double* dv, double* lse)
{
    int rc = check_attn_args(B, h, n_q, n_k, d_k, d_v, mask_kind, key_lens);
    if (rc != ORACLE_OK) return rc;
    const int causal = (mask_kind & ORACLE_MASK_CAUSAL) != 0;
    memset(dq, 0, sizeof(double) * (size_t)B * n_q * h * d_k);
    memset(dk, 0, sizeof(double) * (size_t)B * n_k * h * d_k);
    memset(dv, 0, sizeof(double) * (size_t)B * n_k * h * d_v);
    double* s = (double*)malloc(sizeof(double) * (size_t)n_k);
    double* w = (double*)malloc(sizeof(double) * (size_t)n_k);
    double* dp = (double*)malloc(sizeof(double) * (size_t)n_k);
    unsigned char* vis = (unsigned char*)malloc((size_t)n_k);
    if (!s || !w || !dp || !vis) {
        rc = ORACLE_ENOMEM;
        goto done;
    }
    for (int b = 0; b < B; ++b) {
        const int kv_len = (mask_kind & ORACLE_MASK_KEY_PADDING) ? key_lens[b] : n_k;
        for (int i = 0; i < h; ++i) {
            for (int t = 0; t < n_q; ++t) {
                const double* q_row = q + (((size_t)b * n_q + t) * h + i) * d_k;
                const double* do_row = dout + (((size_t)b * n_q + t) * h + i) * d_v;
                for (int j = 0; j < n_k; ++j) {
                    const double* k_row = k + (((size_t)b * n_k + j) * h + i) * d_k;
                    double dot = 0.0;
                    for (int c = 0; c < d_k; ++c) dot += q_row[c] * k_row[c];
                    s[j] = scale * dot;
                    vis[j] = (unsigned char)(!(causal && j > t) && j < kv_len);
                }
                rc = oracle_softmax(s, vis, n_k, w);
                if (rc != ORACLE_OK) goto done;
                if (lse) {
                    double m = -INFINITY;
                    for (int j = 0; j < n_k; ++j)
                        if (vis[j] && s[j] > m) m = s[j];
                    double sum = 0.0;
                    for (int j = 0; j < n_k; ++j)
                        if (vis[j]) sum += exp(s[j] - m);
                    lse[((size_t)b * h + i) * n_q + t] = m + log(sum);
                }
                double pdp = 0.0;
                for (int j = 0; j < n_k; ++j) {
                    dp[j] = 0.0;
                    if (!vis[j]) continue;
                    const double* v_row = v + (((size_t)b * n_k + j) * h + i) * d_v;
                    for (int c = 0; c < d_v; ++c) dp[j] += do_row[c] * v_row[c];
                    pdp += w[j] * dp[j];
                }
                double* dq_row = dq + (((size_t)b * n_q + t) * h + i) * d_k;
                for (int j = 0; j < n_k; ++j) {
                    if (!vis[j]) continue;
                    const double ds = w[j] * (dp[j] - pdp);
                    const double* k_row = k + (((size_t)b * n_k + j) * h + i) * d_k;
                    double* dk_row = dk + (((size_t)b * n_k + j) * h + i) * d_k;
                    double* dv_row = dv + (((size_t)b * n_k + j) * h + i) * d_v;
                    for (int c = 0; c < d_k; ++c) {
                        dq_row[c] += scale * ds * k_row[c];
                        dk_row[c] += scale * ds * q_row[c];
                    }
                    for (int c = 0; c < d_v; ++c) dv_row[c] += w[j] * do_row[c];
                }
            }
        }
    }
done:
    free(s);
    free(w);
    free(dp);
    free(vis);
    return rc;
}
