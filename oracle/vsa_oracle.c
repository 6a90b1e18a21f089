/*
 * vsa_oracle.c -- plain, slow CPU definition of tile-top-k block-sparse
 * attention (VSA), forward and backward.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark load this library. It shares no code,
 * header, table or constant with the CUDA library it checks, and the CUDA
 * library never calls it.
 *
 * Sources, cited by page title and section:
 *   [VSA-test]  FastVideo fastvideo-kernel/tests/test_vsa256_backward.py
 *   [FA4-adapt] FastVideo fastvideo-kernel/python/fastvideo_kernel/
 *               block_sparse_attn_cute_fwd.py
 *   [NPU-test]  Ascend op-plugin test/test_custom_ops/
 *               test_npu_block_sparse_attention_backward.py
 *
 * Precision. The pooled tile means and the coarse scores decide an integer
 * (the top-k selection), so they are computed in fp32 in one fixed order
 * that the CUDA path must reproduce bit for bit: a sequential round-to-
 * nearest sum over tokens, an IEEE divide, then a fused multiply-add chain
 * over the head dimension. Everything else (softmax attention, the gated
 * compression branch and all gradients) is computed in fp64 and takes fp64
 * inputs (the exact image of the bf16/fp16 tensors, or any fp64 values for
 * finite-difference checks). Build with -ffp-contract=off and without
 * -ffast-math so that the compiler keeps the stated order.
 *
 * Parity status of each function is pinned by tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int layout;          /* 0 = [B,H,S,D], 1 = [B,S,H,D], 2 = varlen [T,H,D] */
    int B, Hq, Hkv, D;
    int Sq, Skv;         /* padded per-batch lengths (layouts 0/1) or totals (2) */
    int tile_q, tile_kv; /* tokens per Q tile and per KV tile */
    int nQ, nKV;         /* tiles per batch entry */
    const int *cu_q;     /* [B+1] token offsets, layout 2 only */
    const int *cu_kv;
    const int *q_var;    /* [nQ]  valid tokens per Q tile, layouts 0/1 only */
    const int *kv_var;   /* [nKV] valid tokens per KV tile, layouts 0/1 only */
    double scale;        /* softmax scale applied to q.k */
} orc_desc;

/* ---------------------------------------------------------------- indexing */

/* Element offset of (batch b, token s of that batch entry, head h, dim e). */
static long off(const orc_desc *d, int q_side, int b, int s, int h, int e)
{
    int H = q_side ? d->Hq : d->Hkv;
    int S = q_side ? d->Sq : d->Skv;
    if (d->layout == 0)
        return (((long)b * H + h) * S + s) * d->D + e;
    if (d->layout == 1)
        return (((long)b * S + s) * H + h) * d->D + e;
    {
        const int *cu = q_side ? d->cu_q : d->cu_kv;
        return ((long)(cu[b] + s) * H + h) * d->D + e;
    }
}

/* Valid tokens in tile t of batch entry b. Padded video tiles hold their
 * valid tokens first, then zero slots ([VSA-test] _zero_pad_tail); in the
 * varlen layout a tile is cut by the end of its sequence ([NPU-test]
 * _expand_block_sparse_mask truncates the block mask to (q_len, kv_len)). */
static int tile_var(const orc_desc *d, int q_side, int b, int t)
{
    int T = q_side ? d->tile_q : d->tile_kv;
    if (d->layout == 2) {
        const int *cu = q_side ? d->cu_q : d->cu_kv;
        int v = (cu[b + 1] - cu[b]) - t * T;
        return v < 0 ? 0 : (v > T ? T : v);
    }
    return q_side ? d->q_var[t] : d->kv_var[t];
}

/* Query rows of tile i that exist. The FA4 valid-length mask ignores the
 * query index ([FA4-adapt] _vbs_mask_mod deletes m_idx), so in the padded
 * video layouts every slot of a Q tile is a query row; in the varlen layout
 * only rows inside the sequence exist. */
static int q_rows(const orc_desc *d, int b, int i)
{
    return d->layout == 2 ? tile_var(d, 1, b, i) : d->tile_q;
}

/* --------------------------------------------------------- O1: tile pooling */

/* Mean of the first var tokens of every tile, per head and dim, in fp32:
 * s = 0; s = s + x[t] for t ascending; p = s / var (p = 0 when var == 0).
 * out is [B][H][nT][D]. The pages use the tile means for the coarse scores
 * and state that the Q fill only enters the compression divisor
 * ([VSA-test] test_vsa256_cute_backward_partial_q_blocks docstring). */
void orc_pool_f32(const orc_desc *d, int q_side, const float *x, float *out)
{
    int H = q_side ? d->Hq : d->Hkv;
    int nT = q_side ? d->nQ : d->nKV;
    int T = q_side ? d->tile_q : d->tile_kv;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < d->B; b++)
        for (int h = 0; h < H; h++)
            for (int t = 0; t < nT; t++) {
                int v = tile_var(d, q_side, b, t);
                float *o = out + (((long)b * H + h) * nT + t) * d->D;
                for (int e = 0; e < d->D; e++) {
                    float s = 0.0f;
                    for (int r = 0; r < v; r++)
                        s = s + x[off(d, q_side, b, t * T + r, h, e)];
                    o[e] = v > 0 ? s / (float)v : 0.0f;
                }
            }
}

/* ------------------------------------------------ O2 + O3: scores and top-k */

/* Coarse score r_ij = pq_i . pk_j as an fp32 fma chain over ascending d,
 * starting from +0; r_ij = -inf when KV tile j has no valid token. Top-k
 * keeps the k = min(topk, nKV) largest r under the strict order (r desc,
 * j asc), so ties go to the lowest tile index. map[b,h,i,j] = 1 iff
 * selected. q_idx[b,h,i,:] lists the selected tiles that hold at least one
 * valid token, ascending; q_cnt counts them; unused slots are -1 (empty
 * tiles are dropped as in [FA4-adapt] _build_sparse_tensors, where only
 * vbs > 0 tiles enter the full or partial lists). In the varlen layout a
 * Q tile with no rows selects nothing. The softmax scale is not applied:
 * a positive scale does not change the order.
 * pq is [B][Hq][nQ][D], pk is [B][Hkv][nKV][D]; scores (optional) is
 * [B][Hq][nQ][nKV]; q_idx is [B][Hq][nQ][cap]. */
void orc_select(const orc_desc *d, const float *pq, const float *pk, int topk,
                uint8_t *map, int *q_idx, int *q_cnt, int cap, float *scores)
{
    int g = d->Hq / d->Hkv;
    int k = topk < d->nKV ? topk : d->nKV;
#pragma omp parallel
    {
        float *r = (float *)malloc(sizeof(float) * d->nKV);
        uint8_t *sel = (uint8_t *)malloc(d->nKV);
#pragma omp for collapse(3) schedule(static)
        for (int b = 0; b < d->B; b++)
            for (int h = 0; h < d->Hq; h++)
                for (int i = 0; i < d->nQ; i++) {
                    long row = ((long)b * d->Hq + h) * d->nQ + i;
                    const float *a = pq + row * d->D;
                    int exists = q_rows(d, b, i) > 0;
                    for (int j = 0; j < d->nKV; j++) {
                        const float *c = pk + (((long)b * d->Hkv + h / g) * d->nKV + j) * d->D;
                        float acc = 0.0f;
                        for (int e = 0; e < d->D; e++)
                            acc = fmaf(a[e], c[e], acc);
                        r[j] = tile_var(d, 0, b, j) > 0 ? acc : -INFINITY;
                        if (scores)
                            scores[row * d->nKV + j] = r[j];
                        sel[j] = 0;
                    }
                    for (int n = 0; exists && n < k; n++) {
                        int best = -1;
                        for (int j = 0; j < d->nKV; j++) {
                            if (sel[j])
                                continue;
                            if (best < 0 || r[j] > r[best])
                                best = j;
                        }
                        sel[best] = 1;
                    }
                    int cnt = 0;
                    for (int j = 0; j < d->nKV; j++) {
                        map[row * d->nKV + j] = sel[j];
                        if (sel[j] && tile_var(d, 0, b, j) > 0)
                            q_idx[row * cap + cnt++] = j;
                    }
                    q_cnt[row] = cnt;
                    for (int n = cnt; n < cap; n++)
                        q_idx[row * cap + n] = -1;
                }
        free(r);
        free(sel);
    }
}

/* A caller-given block map [B][Hq][nQ][nKV] (nonzero = attend) turned into
 * the Q-owned index: per Q tile, the marked KV tiles that hold valid tokens,
 * ascending ([FA4-adapt] _map_to_index and the vbs > 0 split in
 * _build_sparse_tensors). Blocks past the end of a varlen sequence, on
 * either side, are ignored ([NPU-test] _expand_block_sparse_mask). */
void orc_mask_index(const orc_desc *d, const uint8_t *map, int *q_idx, int *q_cnt, int cap)
{
    for (int b = 0; b < d->B; b++)
        for (int h = 0; h < d->Hq; h++)
            for (int i = 0; i < d->nQ; i++) {
                long row = ((long)b * d->Hq + h) * d->nQ + i;
                int cnt = 0;
                if (q_rows(d, b, i) > 0)
                    for (int j = 0; j < d->nKV; j++)
                        if (map[row * d->nKV + j] && tile_var(d, 0, b, j) > 0)
                            q_idx[row * cap + cnt++] = j;
                q_cnt[row] = cnt;
                for (int n = cnt; n < cap; n++)
                    q_idx[row * cap + n] = -1;
            }
}

/* ------------------------------------------------------ O4: KV-owned index */

/* For every KV tile j, the Q tiles whose index lists j, ascending
 * ([FA4-adapt] _build_sparse_tensors: the backward is KV-owned, one list of
 * selecting query tiles per physical KV tile). kv_ptr is [B][Hq][nKV+1]
 * with offsets into kv_qidx's [B][Hq][nQ*cap] row for that (b, h). */
void orc_transpose(const orc_desc *d, const int *q_idx, const int *q_cnt, int cap,
                   int *kv_ptr, int *kv_qidx)
{
    for (int b = 0; b < d->B; b++)
        for (int h = 0; h < d->Hq; h++) {
            long bh = (long)b * d->Hq + h;
            int *ptr = kv_ptr + bh * (d->nKV + 1);
            int *lst = kv_qidx + bh * (long)d->nQ * cap;
            int p = 0;
            for (int j = 0; j < d->nKV; j++) {
                ptr[j] = p;
                for (int i = 0; i < d->nQ; i++) {
                    long row = bh * d->nQ + i;
                    for (int n = 0; n < q_cnt[row]; n++)
                        if (q_idx[row * cap + n] == j)
                            lst[p++] = i;
                }
            }
            ptr[d->nKV] = p;
            for (int n = p; n < d->nQ * cap; n++)
                lst[n] = -1;
        }
}

/* ------------------------------------------------- O5: sparse attention row */

static double dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int e = 0; e < n; e++)
        s += a[e] * b[e];
    return s;
}

/* Softmax attention of query row s (of batch b, head h) over the valid keys
 * of the KV tiles listed for its Q tile: s_u = scale * q.k_u, P = softmax,
 * O = sum P v, LSE = max + ln(sum exp(s - max)) ([NPU-test]
 * cpu_block_sparse_attention_tnd_gqa_with_lse, with the key mask of
 * [FA4-adapt] _vbs_mask_mod: key u of tile j is valid iff
 * u mod tile < vbs[j]). GQA reads KV head h / (Hq/Hkv) ([NPU-test] the
 * TND golden's kv_head = n // group_size). A row with no valid key gets
 * O = 0 and LSE = -inf. sc is scratch for cap*tile_kv doubles. */
static void attend_row(const orc_desc *d, int b, int h, int s, const double *q, const double *k,
                       const double *v, const int *q_idx, const int *q_cnt, int cap,
                       double *sc, double *o, double *lse)
{
    int g = d->Hq / d->Hkv, hk = h / g, i = s / d->tile_q;
    long row = ((long)b * d->Hq + h) * d->nQ + i;
    const double *qr = q + off(d, 1, b, s, h, 0);
    double m = -INFINITY;
    int n_keys = 0;
    for (int n = 0; n < q_cnt[row]; n++) {
        int j = q_idx[row * cap + n], vv = tile_var(d, 0, b, j);
        for (int u = 0; u < vv; u++) {
            double x = d->scale * dot(qr, k + off(d, 0, b, j * d->tile_kv + u, hk, 0), d->D);
            sc[n_keys++] = x;
            if (x > m)
                m = x;
        }
    }
    for (int e = 0; e < d->D; e++)
        o[e] = 0.0;
    if (n_keys == 0) {
        *lse = -INFINITY;
        return;
    }
    double l = 0.0;
    int c = 0;
    for (int n = 0; n < q_cnt[row]; n++) {
        int j = q_idx[row * cap + n], vv = tile_var(d, 0, b, j);
        for (int u = 0; u < vv; u++) {
            double p = exp(sc[c++] - m);
            const double *vr = v + off(d, 0, b, j * d->tile_kv + u, hk, 0);
            l += p;
            for (int e = 0; e < d->D; e++)
                o[e] += p * vr[e];
        }
    }
    for (int e = 0; e < d->D; e++)
        o[e] /= l;
    *lse = m + log(l);
}

/* ------------------------------------------- O6: gated compression branch */

/* Tile means in fp64 (the compression branch's pooled q, k, v; the same
 * definition as orc_pool_f32 without the fp32 rounding). */
static void pool_f64(const orc_desc *d, int q_side, const double *x, double *out)
{
    int H = q_side ? d->Hq : d->Hkv;
    int nT = q_side ? d->nQ : d->nKV;
    int T = q_side ? d->tile_q : d->tile_kv;
    for (int b = 0; b < d->B; b++)
        for (int h = 0; h < H; h++)
            for (int t = 0; t < nT; t++) {
                int vv = tile_var(d, q_side, b, t);
                double *o = out + (((long)b * H + h) * nT + t) * d->D;
                for (int e = 0; e < d->D; e++) {
                    double s = 0.0;
                    for (int r = 0; r < vv; r++)
                        s += x[off(d, q_side, b, t * T + r, h, e)];
                    o[e] = vv > 0 ? s / vv : 0.0;
                }
            }
}

/* Softmax weights of Q tile i over the non-empty KV tiles:
 * a_ij = scale * pq_i . pk_j, A_i = softmax_j(a_ij). Empty tiles get 0. */
static void compress_weights(const orc_desc *d, int b, int h, int i, const double *pq,
                             const double *pk, double *A)
{
    int g = d->Hq / d->Hkv;
    const double *a = pq + (((long)b * d->Hq + h) * d->nQ + i) * d->D;
    double m = -INFINITY, l = 0.0;
    for (int j = 0; j < d->nKV; j++) {
        if (tile_var(d, 0, b, j) == 0) {
            A[j] = -INFINITY;
            continue;
        }
        const double *c = pk + (((long)b * d->Hkv + h / g) * d->nKV + j) * d->D;
        double x = 0.0;
        for (int e = 0; e < d->D; e++)
            x += a[e] * c[e];
        A[j] = d->scale * x;
        if (A[j] > m)
            m = A[j];
    }
    for (int j = 0; j < d->nKV; j++) {
        A[j] = (A[j] == -INFINITY) ? 0.0 : exp(A[j] - m);
        l += A[j];
    }
    for (int j = 0; j < d->nKV; j++)
        A[j] = l > 0.0 ? A[j] / l : 0.0;
}

/* Compression output per Q tile: c_i = sum_j A_ij pv_j, [B][Hq][nQ][D].
 * The gated branch composes out = O_sparse + gate (*) c_tile(t) on every
 * query row of the tile ([VSA-test] test_vsa256_cute_backward_with_compress
 * _gate: the gate is q-shaped and elementwise, and the composition must not
 * overwrite the sparse output). */
void orc_compress_c(const orc_desc *d, const double *q, const double *k, const double *v, double *c)
{
    long nq = (long)d->B * d->Hq * d->nQ * d->D, nk = (long)d->B * d->Hkv * d->nKV * d->D;
    double *pq = (double *)malloc(sizeof(double) * nq);
    double *pk = (double *)malloc(sizeof(double) * nk);
    double *pv = (double *)malloc(sizeof(double) * nk);
    pool_f64(d, 1, q, pq);
    pool_f64(d, 0, k, pk);
    pool_f64(d, 0, v, pv);
    int g = d->Hq / d->Hkv;
#pragma omp parallel
    {
        double *A = (double *)malloc(sizeof(double) * d->nKV);
#pragma omp for collapse(3) schedule(static)
        for (int b = 0; b < d->B; b++)
            for (int h = 0; h < d->Hq; h++)
                for (int i = 0; i < d->nQ; i++) {
                    compress_weights(d, b, h, i, pq, pk, A);
                    double *ci = c + (((long)b * d->Hq + h) * d->nQ + i) * d->D;
                    for (int e = 0; e < d->D; e++)
                        ci[e] = 0.0;
                    for (int j = 0; j < d->nKV; j++) {
                        const double *vj = pv + (((long)b * d->Hkv + h / g) * d->nKV + j) * d->D;
                        for (int e = 0; e < d->D; e++)
                            ci[e] += A[j] * vj[e];
                    }
                }
        free(A);
    }
    free(pq);
    free(pk);
    free(pv);
}

/* ------------------------------------------------------------ forward (O5/O6) */

/* Forward of the listed query rows. rows is n_rows triples (b, h, s) with s
 * the token index within batch entry b. For each listed row writes
 * o_sparse[r][D], lse[r] and, when gate is given, out[r][D] = o_sparse +
 * gate * c (c from orc_compress_c); with no gate out = o_sparse. */
void orc_forward_rows(const orc_desc *d, const double *q, const double *k, const double *v,
                      const int *q_idx, const int *q_cnt, int cap, const double *gate,
                      const double *c, const int *rows, long n_rows, double *out,
                      double *o_sparse, double *lse)
{
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)cap * d->tile_kv + 1);
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < n_rows; r++) {
            int b = rows[3 * r], h = rows[3 * r + 1], s = rows[3 * r + 2];
            double *os = o_sparse + r * d->D, *ot = out + r * d->D;
            attend_row(d, b, h, s, q, k, v, q_idx, q_cnt, cap, sc, os, lse + r);
            const double *ci = c ? c + (((long)b * d->Hq + h) * d->nQ + s / d->tile_q) * d->D : 0;
            for (int e = 0; e < d->D; e++)
                ot[e] = gate ? os[e] + gate[off(d, 1, b, s, h, e)] * ci[e] : os[e];
        }
        free(sc);
    }
}

/* ----------------------------------------------------------- backward (O7) */

/* dQ of the listed query rows: with P_u = exp(s_u - LSE), dP_u = dO.v_u,
 * Dvec = dO.O and dS_u = P_u (dP_u - Dvec), dQ = scale * sum_u dS_u k_u
 * ([NPU-test] _softmax_backward_np and the TND/GQA backward golden). LSE
 * and O of the row are recomputed here by attend_row. dpq (optional,
 * [B][Hq][nQ][D], from orc_compress_grads) adds dpq_i / q_var_i on the
 * valid rows of tile i. dq is packed per listed row. */
void orc_backward_dq_rows(const orc_desc *d, const double *dout, const double *q, const double *k,
                          const double *v, const int *q_idx, const int *q_cnt, int cap,
                          const double *dpq, const int *rows, long n_rows, double *dq)
{
    int g = d->Hq / d->Hkv;
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)cap * d->tile_kv + 1);
        double *o = (double *)malloc(sizeof(double) * d->D);
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < n_rows; r++) {
            int b = rows[3 * r], h = rows[3 * r + 1], s = rows[3 * r + 2];
            int i = s / d->tile_q, hk = h / g;
            long row = ((long)b * d->Hq + h) * d->nQ + i;
            double lse, *dqr = dq + r * d->D;
            attend_row(d, b, h, s, q, k, v, q_idx, q_cnt, cap, sc, o, &lse);
            const double *dor = dout + off(d, 1, b, s, h, 0);
            double Dv = 0.0;
            for (int e = 0; e < d->D; e++) {
                Dv += dor[e] * o[e];
                dqr[e] = 0.0;
            }
            int c = 0;
            for (int n = 0; lse > -INFINITY && n < q_cnt[row]; n++) {
                int j = q_idx[row * cap + n], vv = tile_var(d, 0, b, j);
                for (int u = 0; u < vv; u++) {
                    const double *kr = k + off(d, 0, b, j * d->tile_kv + u, hk, 0);
                    const double *vr = v + off(d, 0, b, j * d->tile_kv + u, hk, 0);
                    double p = exp(sc[c++] - lse);
                    double ds = p * (dot(dor, vr, d->D) - Dv);
                    for (int e = 0; e < d->D; e++)
                        dqr[e] += d->scale * ds * kr[e];
                }
            }
            int qv = tile_var(d, 1, b, i);
            if (dpq && s - i * d->tile_q < qv)
                for (int e = 0; e < d->D; e++)
                    dqr[e] += dpq[row * d->D + e] / qv;
        }
        free(sc);
        free(o);
    }
}

/* dK and dV of the listed KV tiles. tiles is n_tiles triples (b, hk, j).
 * For every query head h of the KV head's group, every Q tile i whose index
 * lists j, and every query row t of tile i:
 *   dV_u += P_tu dO_t,   dK_u += scale * dS_tu q_t
 * over the valid keys u of tile j, with P, dS as in orc_backward_dq_rows
 * (dK, dV summed over the group, as the GQA golden's += does). dpk, dpv
 * (optional, [B][Hkv][nKV][D]) add dpk_j / kv_var_j and dpv_j / kv_var_j
 * on the valid keys. dk, dv are [n_tiles][tile_kv][D]; padded keys get 0. */
void orc_backward_dkdv_tiles(const orc_desc *d, const double *dout, const double *q, const double *k,
                             const double *v, const int *q_idx, const int *q_cnt, int cap,
                             const double *dpk, const double *dpv, const int *tiles, long n_tiles,
                             double *dk, double *dv)
{
    int g = d->Hq / d->Hkv;
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)cap * d->tile_kv + 1);
        double *o = (double *)malloc(sizeof(double) * d->D);
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < n_tiles; r++) {
            int b = tiles[3 * r], hk = tiles[3 * r + 1], j = tiles[3 * r + 2];
            int vv = tile_var(d, 0, b, j);
            double *dkt = dk + r * (long)d->tile_kv * d->D, *dvt = dv + r * (long)d->tile_kv * d->D;
            for (long e = 0; e < (long)d->tile_kv * d->D; e++)
                dkt[e] = dvt[e] = 0.0;
            for (int h = hk * g; h < (hk + 1) * g; h++)
                for (int i = 0; i < d->nQ; i++) {
                    long row = ((long)b * d->Hq + h) * d->nQ + i;
                    int listed = 0;
                    for (int n = 0; n < q_cnt[row]; n++)
                        listed |= q_idx[row * cap + n] == j;
                    if (!listed)
                        continue;
                    for (int t = 0; t < q_rows(d, b, i); t++) {
                        int s = i * d->tile_q + t;
                        double lse;
                        attend_row(d, b, h, s, q, k, v, q_idx, q_cnt, cap, sc, o, &lse);
                        const double *qr = q + off(d, 1, b, s, h, 0);
                        const double *dor = dout + off(d, 1, b, s, h, 0);
                        double Dv = 0.0;
                        for (int e = 0; e < d->D; e++)
                            Dv += dor[e] * o[e];
                        for (int u = 0; u < vv; u++) {
                            const double *kr = k + off(d, 0, b, j * d->tile_kv + u, hk, 0);
                            const double *vr = v + off(d, 0, b, j * d->tile_kv + u, hk, 0);
                            double p = exp(d->scale * dot(qr, kr, d->D) - lse);
                            double ds = p * (dot(dor, vr, d->D) - Dv);
                            for (int e = 0; e < d->D; e++) {
                                dvt[(long)u * d->D + e] += p * dor[e];
                                dkt[(long)u * d->D + e] += d->scale * ds * qr[e];
                            }
                        }
                    }
                }
            if (dpk)
                for (int u = 0; u < vv; u++)
                    for (int e = 0; e < d->D; e++) {
                        long p = (((long)b * d->Hkv + hk) * d->nKV + j) * d->D + e;
                        dkt[(long)u * d->D + e] += dpk[p] / vv;
                        dvt[(long)u * d->D + e] += dpv[p] / vv;
                    }
        }
        free(sc);
        free(o);
    }
}

/* --------------------------------------------- O8: compression branch grads */

/* Gradients of the compression branch with respect to the pooled q, k, v,
 * given the upstream gradient dO of out and the gate:
 *   dc_i   = sum over the query rows t of tile i of gate_t (*) dO_t
 *   dA_ij  = dc_i . pv_j,   dpv_j += A_ij dc_i
 *   ds_ij  = A_ij (dA_ij - sum_j' A_ij' dA_ij')          (softmax backward)
 *   dpq_i  = scale sum_j ds_ij pk_j,   dpk_j += scale ds_ij pq_i
 * summed over the query heads of a GQA group for dpk, dpv. The selection
 * is held fixed (no gradient flows through top-k) and the gate gets none.
 * dpq is [B][Hq][nQ][D]; dpk, dpv are [B][Hkv][nKV][D]. */
void orc_compress_grads(const orc_desc *d, const double *dout, const double *gate, const double *q,
                        const double *k, const double *v, double *dpq, double *dpk, double *dpv)
{
    long nq = (long)d->B * d->Hq * d->nQ * d->D, nk = (long)d->B * d->Hkv * d->nKV * d->D;
    int g = d->Hq / d->Hkv;
    double *pq = (double *)malloc(sizeof(double) * nq);
    double *pk = (double *)malloc(sizeof(double) * nk);
    double *pv = (double *)malloc(sizeof(double) * nk);
    pool_f64(d, 1, q, pq);
    pool_f64(d, 0, k, pk);
    pool_f64(d, 0, v, pv);
    memset(dpq, 0, sizeof(double) * nq);
    memset(dpk, 0, sizeof(double) * nk);
    memset(dpv, 0, sizeof(double) * nk);
    double *A = (double *)malloc(sizeof(double) * d->nKV);
    double *dA = (double *)malloc(sizeof(double) * d->nKV);
    double *dc = (double *)malloc(sizeof(double) * d->D);
    for (int b = 0; b < d->B; b++)
        for (int h = 0; h < d->Hq; h++)
            for (int i = 0; i < d->nQ; i++) {
                long row = ((long)b * d->Hq + h) * d->nQ + i;
                for (int e = 0; e < d->D; e++)
                    dc[e] = 0.0;
                for (int t = 0; t < q_rows(d, b, i); t++) {
                    int s = i * d->tile_q + t;
                    for (int e = 0; e < d->D; e++)
                        dc[e] += gate[off(d, 1, b, s, h, e)] * dout[off(d, 1, b, s, h, e)];
                }
                compress_weights(d, b, h, i, pq, pk, A);
                double sum = 0.0;
                for (int j = 0; j < d->nKV; j++) {
                    const double *vj = pv + (((long)b * d->Hkv + h / g) * d->nKV + j) * d->D;
                    double x = 0.0;
                    for (int e = 0; e < d->D; e++)
                        x += dc[e] * vj[e];
                    dA[j] = x;
                    sum += A[j] * x;
                }
                for (int j = 0; j < d->nKV; j++) {
                    long kj = (((long)b * d->Hkv + h / g) * d->nKV + j) * d->D;
                    double ds = A[j] * (dA[j] - sum);
                    for (int e = 0; e < d->D; e++) {
                        dpv[kj + e] += A[j] * dc[e];
                        dpq[row * d->D + e] += d->scale * ds * pk[kj + e];
                        dpk[kj + e] += d->scale * ds * pq[row * d->D + e];
                    }
                }
            }
    free(A);
    free(dA);
    free(dc);
    free(pq);
    free(pk);
    free(pv);
}
