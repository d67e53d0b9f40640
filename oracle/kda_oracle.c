/*
 * kda_oracle.c -- plain float64 CPU oracle for the Kimi Delta Attention (KDA)
 * operator.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark load this file's library.  The CUDA library
 * shares no code, header, table or helper with it, and never calls it.
 *
 * What it computes ("Kimi K3, explained", section "The math"; the same steps
 * are spelled out in "How Kimi Delta Attention works, step by step"):
 *
 *   the page writes, per head, with S of size d_v x d_k,
 *       S_t = S_{t-1} Diag(alpha_t) (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *       o_t = S_t q_t.
 *   This file keeps the transpose, S of size d_k x d_v (row i = key channel i,
 *   d_v contiguous), which gives the identical numbers:
 *       S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *       o_t = scale * S_t^T q_t.
 *
 * One token is three plain passes over the state, in the page's order
 * (decay, then erase-and-write on the decayed state, then read):
 *   1. decay        S[i][j] *= alpha[i]
 *   2. erase/write  x[j] = sum_i S[i][j] k[i];  S[i][j] += beta k[i] (v[j] - x[j])
 *                   (the page's S <- S - beta (S k - v) k^T, applied to the
 *                   decayed state, in this orientation)
 *   3. read         o[j] = scale * sum_i S[i][j] q[i]
 *
 * With erase == 0 the erase term is dropped and step 2 is the write
 * S += beta k v^T alone: gated linear attention, which the page names as the
 * rule one gets by dropping the erase factor.  It exists for the oracle's own
 * checks (two writes to one key return their sum).
 *
 * Inputs are read in their storage dtype (q, k, v as float32 or bfloat16 bits;
 * beta, alpha float32) and widened exactly to double; every operation is done
 * in double, in the order written, with no blocking, fusion or reordering.
 *
 * Layouts (row-major, contiguous):
 *   q, k [T, H, d_k]   v [T, H, d_v]   beta [T, H]   alpha [T, H, d_k]
 *   states [d_k, d_v] per (sequence, head)   o [T, d_v] per (sequence, head)
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -shared -fPIC (no fused
 * multiply-add, so the rounding order is exactly the one written).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef KDA_ORACLE_MUTANT
/* Planted mistakes, compiled only by the oracle's own mutation test, to show
 * that the pins catch each of them:
 *   1 drop the erase term         2 decay after erase-and-write
 *   3 read before the update      4 decay along d_v instead of d_k
 *   5 wrong sign of the erase     6 erase with the decayed key alpha*k */
#define MUTANT KDA_ORACLE_MUTANT
#else
#define MUTANT 0
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

static double load_elem(const void* base, int dtype, int64_t idx) {
    if (dtype == ORACLE_BF16) {
        uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[idx];
}

/* One token of the recurrence on one head's state S [dk][dv] (double).
 * q, k, v are the token's vectors already widened to double; x is scratch [dv].
 * o (may be NULL) receives scale * S_t^T q_t. */
static void token_update(double* S, int dk, int dv, const double* q, const double* k,
                         const double* v, double beta, const double* alpha, double scale,
                         int erase, double* x, double* o) {
    int i, j;
#if MUTANT == 3
    if (o) {
        for (j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (i = 0; i < dk; ++i) acc += S[(int64_t)i * dv + j] * q[i];
            o[j] = scale * acc;
        }
    }
#endif
    /* 1. decay: Diag(alpha_t) S_{t-1} */
#if MUTANT != 2
    for (i = 0; i < dk; ++i) {
        for (j = 0; j < dv; ++j) {
#if MUTANT == 4
            S[(int64_t)i * dv + j] *= alpha[j % dk];
#else
            S[(int64_t)i * dv + j] *= alpha[i];
#endif
        }
    }
#endif
    /* 2. erase and write on the decayed state */
    for (j = 0; j < dv; ++j) {
        double acc = 0.0;
        for (i = 0; i < dk; ++i) {
#if MUTANT == 6
            acc += S[(int64_t)i * dv + j] * (alpha[i] * k[i]);
#else
            acc += S[(int64_t)i * dv + j] * k[i];
#endif
        }
        x[j] = acc;
    }
    for (i = 0; i < dk; ++i) {
        for (j = 0; j < dv; ++j) {
            double delta;
#if MUTANT == 1
            delta = v[j];
#elif MUTANT == 5
            delta = erase ? (v[j] + x[j]) : v[j];
#else
            delta = erase ? (v[j] - x[j]) : v[j];
#endif
            S[(int64_t)i * dv + j] += beta * k[i] * delta;
        }
    }
#if MUTANT == 2
    for (i = 0; i < dk; ++i)
        for (j = 0; j < dv; ++j) S[(int64_t)i * dv + j] *= alpha[i];
#endif
    /* 3. read with the query: o_t = scale * S_t^T q_t */
#if MUTANT != 3
    if (o) {
        for (j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (i = 0; i < dk; ++i) acc += S[(int64_t)i * dv + j] * q[i];
            o[j] = scale * acc;
        }
    }
#endif
}

/*
 * One (sequence, head) unit over tokens [t0, t0 + T) of packed arrays with H
 * heads.  s_in: [dk*dv] double or NULL (zero state).  s_out: [dk*dv] double.
 * o: NULL, or row t of the unit's output at o + t * o_stride (t = 0 .. T-1).
 * Returns 0, or -1 on a bad argument or failed allocation.
 */
int kda_oracle_unit(const void* q, const void* k, const void* v, int dtype_qkv,
                    const float* beta, const float* alpha, int64_t t0, int64_t T, int32_t H,
                    int32_t h, int32_t dk, int32_t dv, double scale, int32_t erase,
                    const double* s_in, double* s_out, double* o, int64_t o_stride) {
    if (!q || !k || !v || !beta || !alpha || !s_out || T < 0 || H <= 0 || h < 0 || h >= H ||
        dk <= 0 || dv <= 0)
        return -1;
    double* qv = (double*)malloc(sizeof(double) * (size_t)(2 * dk + 2 * dv) + sizeof(double) * (size_t)dk);
    if (!qv) return -1;
    double* kv = qv + dk;
    double* vv = kv + dk;
    double* x = vv + dv;
    double* av = x + dv;
    int64_t n = (int64_t)dk * dv;
    if (s_in)
        memcpy(s_out, s_in, sizeof(double) * (size_t)n);
    else
        memset(s_out, 0, sizeof(double) * (size_t)n);
    for (int64_t t = 0; t < T; ++t) {
        int64_t row = (t0 + t) * H + h;
        for (int i = 0; i < dk; ++i) {
            qv[i] = load_elem(q, dtype_qkv, row * dk + i);
            kv[i] = load_elem(k, dtype_qkv, row * dk + i);
            av[i] = (double)alpha[row * dk + i];
        }
        for (int j = 0; j < dv; ++j) vv[j] = load_elem(v, dtype_qkv, row * dv + j);
        token_update(s_out, dk, dv, qv, kv, vv, (double)beta[row], av, scale, erase, x,
                     o ? o + t * o_stride : NULL);
    }
    free(qv);
    return 0;
}

/*
 * One decode step for batch rows [b0, b1): token b of every head updates the
 * resident state pool[slot[b], h] (double, [P, H, dk, dv]) in place, where
 * slot = state_idx ? state_idx[b] : b, and writes o[b, h, :] (double).
 * Inputs are laid out like a packed prefill with T = B tokens.
 */
int kda_oracle_decode(const void* q, const void* k, const void* v, int dtype_qkv,
                      const float* beta, const float* alpha, double* pool, const int32_t* state_idx,
                      int32_t P, int32_t B, int32_t H, int32_t dk, int32_t dv, double scale,
                      double* o, int32_t b0, int32_t b1) {
    if (!q || !k || !v || !beta || !alpha || !pool || !o || B < 0 || H <= 0 || dk <= 0 || dv <= 0 ||
        b0 < 0 || b1 > B || b0 > b1)
        return -1;
    double* qv = (double*)malloc(sizeof(double) * (size_t)(3 * dk + 2 * dv));
    if (!qv) return -1;
    double* kv = qv + dk;
    double* av = kv + dk;
    double* vv = av + dk;
    double* x = vv + dv;
    int rc = 0;
    for (int32_t b = b0; b < b1 && rc == 0; ++b) {
        int32_t slot = state_idx ? state_idx[b] : b;
        if (slot < 0 || slot >= P) { rc = -1; break; }
        for (int32_t h = 0; h < H; ++h) {
            int64_t row = (int64_t)b * H + h;
            for (int i = 0; i < dk; ++i) {
                qv[i] = load_elem(q, dtype_qkv, row * dk + i);
                kv[i] = load_elem(k, dtype_qkv, row * dk + i);
                av[i] = (double)alpha[row * dk + i];
            }
            for (int j = 0; j < dv; ++j) vv[j] = load_elem(v, dtype_qkv, row * dv + j);
            double* S = pool + ((int64_t)slot * H + h) * (int64_t)dk * dv;
            token_update(S, dk, dv, qv, kv, vv, (double)beta[row], av, scale, 1, x, o + row * dv);
        }
    }
    free(qv);
    return rc;
}
