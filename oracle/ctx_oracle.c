/*
 * CPU oracle for the context-parallel attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY. This file is compiled into liboracle_ctx.so and
 * is loaded by the tests, by the smoke check and by the benchmark's CPU
 * baseline leg. The product path (the CUDA library) never links, loads or
 * calls it, and it shares no code, header or helper with that library.
 *
 * Everything here is the plain definition written out with explicit index
 * loops, in the order the pages state it:
 *
 *   pack   (sglang PR #33667, "_usp_input_all_to_all_qkv" excerpt and the
 *           pack_qkv_destination_major description): destination rank r gets
 *           heads [r*H/U, (r+1)*H/U) of every local row of Q, K and V, one
 *           destination after the other, so chunk r of the flat send buffer
 *           is exactly what rank r must receive. Layout [U,3,B,S_l,H/U,D].
 *   unpack (same excerpt, receive side): chunk r of the received buffer
 *           holds source rank r's rows, which become global rows
 *           [r*S_l, (r+1)*S_l); batch stays outermost. Output [B,U*S_l,H/U,D].
 *   pack_out / unpack_out (the reverse Ulysses all-to-all of
 *           "_usp_output_all_to_all" on the sglang page and step 4 of the
 *           composed order on the vllm-omni PR #7641 page): the exact inverse
 *           of the input exchange, rows back to their source rank and heads
 *           back to their global position.
 *   attention (vllm-omni PR #7641, local-Q / global-KV attention; the
 *           ChituDiffusion "Fast CP" support matrix: non-causal MHA): for each
 *           (b, h, query i), over the unmasked keys j,
 *             s_j = scale * sum_d q[i,d] k[j,d]
 *             O   = sum_j exp(s_j) v_j / sum_j exp(s_j)
 *             LSE = ln sum_j exp(s_j)
 *           computed in fp64 (the max is subtracted before exp only to avoid
 *           overflow; it cancels exactly in the quotient). A row with no
 *           valid key gets O = 0 and LSE = -inf.
 *
 * Inputs are 16-bit floating point bit patterns (bf16 or fp16), widened
 * exactly to double. bf16 is the upper half of an IEEE binary32; fp16 is
 * decoded from its IEEE binary16 fields.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_FP16 = 1 };

static double orc_widen(uint16_t h, int dtype)
{
    if (dtype == ORC_BF16) {
        uint32_t u = (uint32_t)h << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    /* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits */
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);   /* (1 + m/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* staging[r][t][b][s][h][d] = X_t[b][s][r*h_l + h][d] */
int orc_pack_qkv(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                 uint16_t *staging, long long B, long long S_l, long long H,
                 long long D, long long U)
{
    if (U <= 0 || H <= 0 || H % U != 0)
        return 1;
    long long h_l = H / U;
    const uint16_t *src[3] = {q, k, v};
    for (long long r = 0; r < U; ++r)
        for (long long t = 0; t < 3; ++t)
            for (long long b = 0; b < B; ++b)
                for (long long s = 0; s < S_l; ++s)
                    for (long long h = 0; h < h_l; ++h)
                        for (long long d = 0; d < D; ++d) {
                            long long dst = ((((r * 3 + t) * B + b) * S_l + s) * h_l + h) * D + d;
                            long long from = ((b * S_l + s) * H + (r * h_l + h)) * D + d;
                            staging[dst] = src[t][from];
                        }
    return 0;
}

/* X'_t[b][r*S_l + s][h][d] = recv[r][t][b][s][h][d] */
int orc_unpack_qkv(const uint16_t *recv, uint16_t *q, uint16_t *k, uint16_t *v,
                   long long B, long long S_l, long long h_l, long long D,
                   long long U)
{
    if (U <= 0)
        return 1;
    uint16_t *dst[3] = {q, k, v};
    for (long long r = 0; r < U; ++r)
        for (long long t = 0; t < 3; ++t)
            for (long long b = 0; b < B; ++b)
                for (long long s = 0; s < S_l; ++s)
                    for (long long h = 0; h < h_l; ++h)
                        for (long long d = 0; d < D; ++d) {
                            long long from = ((((r * 3 + t) * B + b) * S_l + s) * h_l + h) * D + d;
                            long long to = ((b * (U * S_l) + (r * S_l + s)) * h_l + h) * D + d;
                            dst[t][to] = recv[from];
                        }
    return 0;
}

/* send[r][b][s][h][d] = O[b][r*S_l + s][h][d] */
int orc_pack_out(const uint16_t *o, uint16_t *send, long long B, long long S_l,
                 long long h_l, long long D, long long U)
{
    if (U <= 0)
        return 1;
    for (long long r = 0; r < U; ++r)
        for (long long b = 0; b < B; ++b)
            for (long long s = 0; s < S_l; ++s)
                for (long long h = 0; h < h_l; ++h)
                    for (long long d = 0; d < D; ++d) {
                        long long to = (((r * B + b) * S_l + s) * h_l + h) * D + d;
                        long long from = ((b * (U * S_l) + (r * S_l + s)) * h_l + h) * D + d;
                        send[to] = o[from];
                    }
    return 0;
}

/* Y[b][s][r*h_l + h][d] = recv[r][b][s][h][d] */
int orc_unpack_out(const uint16_t *recv, uint16_t *y, long long B, long long S_l,
                   long long h_l, long long D, long long U)
{
    if (U <= 0)
        return 1;
    long long H = U * h_l;
    for (long long r = 0; r < U; ++r)
        for (long long b = 0; b < B; ++b)
            for (long long s = 0; s < S_l; ++s)
                for (long long h = 0; h < h_l; ++h)
                    for (long long d = 0; d < D; ++d) {
                        long long from = (((r * B + b) * S_l + s) * h_l + h) * D + d;
                        long long to = ((b * S_l + s) * H + (r * h_l + h)) * D + d;
                        y[to] = recv[from];
                    }
    return 0;
}

/* Attention probabilities of one query row (b, h, i): p[j] for every key j,
 * 0 for masked keys. Returns 0, or 1 if the row has no valid key (p all 0). */
int orc_attention_probs(const uint16_t *q, const uint16_t *k, const uint8_t *mask,
                        int dtype, double scale, long long B, long long Sq,
                        long long Sk, long long H, long long D, long long b,
                        long long h, long long i, double *p)
{
    (void)B;
    double m = -INFINITY;
    for (long long j = 0; j < Sk; ++j) {
        p[j] = -INFINITY;
        if (mask && !mask[b * Sk + j])
            continue;
        double acc = 0.0;
        for (long long d = 0; d < D; ++d)
            acc += orc_widen(q[((b * Sq + i) * H + h) * D + d], dtype) *
                   orc_widen(k[((b * Sk + j) * H + h) * D + d], dtype);
        p[j] = scale * acc;
        if (p[j] > m)
            m = p[j];
    }
    if (m == -INFINITY) {
        for (long long j = 0; j < Sk; ++j)
            p[j] = 0.0;
        return 1;
    }
    double l = 0.0;
    for (long long j = 0; j < Sk; ++j) {
        p[j] = (p[j] == -INFINITY) ? 0.0 : exp(p[j] - m);
        l += p[j];
    }
    for (long long j = 0; j < Sk; ++j)
        p[j] /= l;
    return 0;
}

/* Attention output for a list of n query rows given as (b, h, i) triples
 * (bhi[3*n]). out[n*D] receives O, lse[n] receives the natural-log LSE.
 * Q is [B,Sq,H,D], K and V are [B,Sk,H,D], mask is NULL or [B,Sk] (nonzero =
 * attend). Rows are independent; they are spread over OpenMP threads. */
int orc_attention_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const uint8_t *mask, int dtype, double scale,
                       long long B, long long Sq, long long Sk, long long H,
                       long long D, long long n, const long long *bhi,
                       double *out, double *lse)
{
    if (B <= 0 || Sq <= 0 || Sk <= 0 || H <= 0 || D <= 0 || n < 0)
        return 1;
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Sk);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !qd) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long long r = 0; r < n; ++r) {
            if (!s || !qd)
                continue;
            long long b = bhi[3 * r], h = bhi[3 * r + 1], i = bhi[3 * r + 2];
            for (long long d = 0; d < D; ++d)
                qd[d] = orc_widen(q[((b * Sq + i) * H + h) * D + d], dtype);
            /* scores of the valid keys */
            double m = -INFINITY;
            for (long long j = 0; j < Sk; ++j) {
                s[j] = -INFINITY;
                if (mask && !mask[b * Sk + j])
                    continue;
                double acc = 0.0;
                const uint16_t *kr = k + ((b * Sk + j) * H + h) * D;
                for (long long d = 0; d < D; ++d)
                    acc += qd[d] * orc_widen(kr[d], dtype);
                s[j] = scale * acc;
                if (s[j] > m)
                    m = s[j];
            }
            double *o = out + r * D;
            for (long long d = 0; d < D; ++d)
                o[d] = 0.0;
            if (m == -INFINITY) {  /* no valid key */
                lse[r] = -INFINITY;
                continue;
            }
            /* softmax weights, then the weighted sum of V */
            double l = 0.0;
            for (long long j = 0; j < Sk; ++j) {
                if (s[j] == -INFINITY)
                    continue;
                double w = exp(s[j] - m);
                l += w;
                const uint16_t *vr = v + ((b * Sk + j) * H + h) * D;
                for (long long d = 0; d < D; ++d)
                    o[d] += w * orc_widen(vr[d], dtype);
            }
            for (long long d = 0; d < D; ++d)
                o[d] /= l;
            lse[r] = m + log(l);
        }
        free(s);
        free(qd);
    }
    return bad ? 2 : 0;
}

/* Combination of attention results over P disjoint key segments (the merge
 * that consumes the LSE): for every row,
 *   lse = ln sum_p exp(lse_p),   out = sum_p exp(lse_p - lse) * o_p
 * o_parts [P][rows][D] 16-bit, lse_parts [P][rows] (natural log, -inf for a
 * segment without valid keys), out [rows][D] and lse [rows] in fp64. A row
 * whose segments are all empty gets out = 0 and lse = -inf. */
int orc_lse_merge(const uint16_t *o_parts, const double *lse_parts, int dtype, long long P,
                  long long rows, long long D, double *out, double *lse)
{
    if (P <= 0 || rows < 0 || D <= 0)
        return 1;
    for (long long r = 0; r < rows; ++r) {
        double m = -INFINITY;
        for (long long p = 0; p < P; ++p)
            if (lse_parts[p * rows + r] > m)
                m = lse_parts[p * rows + r];
        double *o = out + r * D;
        for (long long d = 0; d < D; ++d)
            o[d] = 0.0;
        if (m == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double l = 0.0;
        for (long long p = 0; p < P; ++p)
            if (lse_parts[p * rows + r] != -INFINITY)
                l += exp(lse_parts[p * rows + r] - m);
        const double total = m + log(l);
        lse[r] = total;
        for (long long p = 0; p < P; ++p) {
            const double lp = lse_parts[p * rows + r];
            if (lp == -INFINITY)
                continue;
            const double w = exp(lp - total);
            for (long long d = 0; d < D; ++d)
                o[d] += w * orc_widen(o_parts[(p * rows + r) * D + d], dtype);
        }
    }
    return 0;
}

/* Ulysses pack with the general options of the pages:
 *  - uneven heads (vllm-omni PR #7641, "advanced_uaa" head padding): the H
 *    heads are padded with zero heads to U*h_l, h_l = ceil(H/U), and
 *    destination r gets padded heads [r*h_l, (r+1)*h_l);
 *  - layout 0 = [U][3][B][S_l][h_l][D] (Q, K, V one after the other),
 *    layout 1 = [U][B][S_l][h_l][3*D] (Q, K, V interleaved on the last
 *    dimension, the sglang PR #33667 excerpt's staging buffer).
 * Element (r, t, b, s, h, d) = X_t[b][s][r*h_l + h][d] if r*h_l + h < H, else 0. */
int orc_pack_qkv_ex(const uint16_t *q, const uint16_t *k, const uint16_t *v, uint16_t *staging,
                    long long B, long long S_l, long long H, long long D, long long U, int layout)
{
    if (U <= 0 || H <= 0 || (layout != 0 && layout != 1))
        return 1;
    long long h_l = (H + U - 1) / U;
    const uint16_t *src[3] = {q, k, v};
    for (long long r = 0; r < U; ++r)
        for (long long t = 0; t < 3; ++t)
            for (long long b = 0; b < B; ++b)
                for (long long s = 0; s < S_l; ++s)
                    for (long long h = 0; h < h_l; ++h)
                        for (long long d = 0; d < D; ++d) {
                            long long g = r * h_l + h;
                            uint16_t val = (g < H) ? src[t][((b * S_l + s) * H + g) * D + d] : 0;
                            long long dst = layout == 0
                                                ? ((((r * 3 + t) * B + b) * S_l + s) * h_l + h) * D + d
                                                : ((((r * B + b) * S_l + s) * h_l + h) * 3 + t) * D + d;
                            staging[dst] = val;
                        }
    return 0;
}

/* Receive side for either staging layout: X'_t[b][r*S_l + s][h][d]. */
int orc_unpack_qkv_ex(const uint16_t *recv, uint16_t *q, uint16_t *k, uint16_t *v, long long B,
                      long long S_l, long long h_l, long long D, long long U, int layout)
{
    if (U <= 0 || (layout != 0 && layout != 1))
        return 1;
    uint16_t *dst[3] = {q, k, v};
    for (long long r = 0; r < U; ++r)
        for (long long t = 0; t < 3; ++t)
            for (long long b = 0; b < B; ++b)
                for (long long s = 0; s < S_l; ++s)
                    for (long long h = 0; h < h_l; ++h)
                        for (long long d = 0; d < D; ++d) {
                            long long from = layout == 0
                                                 ? ((((r * 3 + t) * B + b) * S_l + s) * h_l + h) * D + d
                                                 : ((((r * B + b) * S_l + s) * h_l + h) * 3 + t) * D + d;
                            dst[t][((b * (U * S_l) + (r * S_l + s)) * h_l + h) * D + d] = recv[from];
                        }
    return 0;
}

/* Reverse exchange receive side that drops padded heads:
 * Y[b][s][r*h_l + h][d] = recv[r][b][s][h][d] for r*h_l + h < H. */
int orc_unpack_out_ex(const uint16_t *recv, uint16_t *y, long long B, long long S_l, long long h_l,
                      long long H, long long D, long long U)
{
    if (U <= 0 || H > U * h_l)
        return 1;
    for (long long r = 0; r < U; ++r)
        for (long long b = 0; b < B; ++b)
            for (long long s = 0; s < S_l; ++s)
                for (long long h = 0; h < h_l; ++h) {
                    long long g = r * h_l + h;
                    if (g >= H)
                        continue;
                    for (long long d = 0; d < D; ++d)
                        y[((b * S_l + s) * H + g) * D + d] = recv[(((r * B + b) * S_l + s) * h_l + h) * D + d];
                }
    return 0;
}
