/*
 * svdq_oracle.c -- ORACLE.  Test infrastructure, not part of the product.
 *
 * A plain, slow, CPU reference for the SVDQuant W4A4 linear operator
 *
 *     y = scaled_mma(act4, wgt4) * wcscale + bias + lora_act_in @ lora_up
 *
 * as defined in "SVDQuant W4A4 on Blackwell" §2 (the operator and its input
 * formats) and §3.1 (NVFP4: two E2M1 nibbles per byte, one FP8-E4M3 scale per
 * 16 K elements, single-level scaling).  Everything is evaluated in fp64 in
 * the order the definition states it; there is no blocking, fusion or
 * reordering.  Only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library; the CUDA path never
 * does, and the two share no code.
 *
 * Readings of points the page leaves open (each is listed in the design
 * notes):
 *   - element k of a packed row sits in the low nibble of byte k/2 when k is
 *     even and in the high nibble when k is odd;
 *   - ascales[g][m] (M contiguous) scales act[m][16g .. 16g+15], and
 *     wscales[g][n] likewise scales wgt[n][16g .. 16g+15];
 *   - wgt is [N, K/2] (K-major), i.e. the product is act . wgt^T;
 *   - the LoRA term is added after the wcscale multiply (it is not scaled);
 *   - lora_act_in is fp32 and used exactly; lora_up, wcscale and bias are
 *     bf16 (or, in the fp16 variant the page also measures, IEEE binary16)
 *     and used exactly; a NULL wcscale means 1, a NULL bias means 0.
 *
 * Parity pins (tests): the E2M1 table against the format's published value
 * set, E4M3 exhaustively against a library conversion, exact brute force in
 * rational arithmetic on tiny shapes, exact equality with dequantize-then-
 * matmul, closed forms (all ones, one-hot, identity) and invariants.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* E2M1 element format (1 sign bit, 2 exponent bits with bias 1, 1 mantissa
 * bit), written out as its 16-code value table: exponent field 0 is
 * subnormal (0 or 0.5), exponent field e >= 1 gives 2^(e-1) * (1 + m/2).
 * Codes 8..15 carry the sign bit. */
static const double E2M1_VALUES[16] = {
    0.0,  0.5,  1.0,  1.5,  2.0,  3.0,  4.0,  6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};

double svdq_oracle_e2m1(int code) { return E2M1_VALUES[code & 15]; }

/* FP8-E4M3 decoded bit by bit: sign = bit 7, exponent field e = bits 6..3
 * (bias 7), mantissa f = bits 2..0.  e == 15 with f == 7 is NaN (the format
 * has no infinities), e == 0 is subnormal 2^-6 * f/8, otherwise the value is
 * 2^(e-7) * (1 + f/8). */
double svdq_oracle_e4m3(int byte) {
    int s = (byte >> 7) & 1;
    int e = (byte >> 3) & 15;
    int f = byte & 7;
    double v;
    if (e == 15 && f == 7) return NAN;
    if (e == 0)
        v = ldexp((double)f / 8.0, -6);
    else
        v = ldexp(1.0 + (double)f / 8.0, e - 7);
    return s ? -v : v;
}

/* bf16 is the upper half of an IEEE binary32. */
double svdq_oracle_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16 decoded bit by bit: sign = bit 15, exponent field e = bits
 * 14..10 (bias 15), fraction f = bits 9..0.  e == 0 is subnormal
 * 2^-14 * f/1024, e == 31 is infinity (f == 0) or NaN, otherwise the value is
 * 2^(e-15) * (1 + f/1024). */
double svdq_oracle_f16(uint16_t bits) {
    int s = (bits >> 15) & 1;
    int e = (bits >> 10) & 31;
    int f = bits & 1023;
    double v;
    if (e == 31) return f ? NAN : (s ? -INFINITY : INFINITY);
    if (e == 0)
        v = ldexp((double)f / 1024.0, -14);
    else
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return s ? -v : v;
}

/* Round an fp64 value to the nearest bf16 (ties to even), returning its bits.
 * Used only to report y in the output dtype; parity is judged on fp64 y. */
uint16_t svdq_oracle_round_bf16(double x) {
    uint16_t sign;
    double a, f, q;
    int e, E;
    if (isnan(x)) return 0x7FC0;
    sign = signbit(x) ? 0x8000 : 0;
    a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    f = frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    E = e - 1 + 127;                  /* biased exponent of 2f * 2^(e-1) */
    if (E >= 1) {
        q = nearbyint(ldexp(f, 8));   /* 8 significant bits: 128 .. 256 */
        if (q == 256.0) {
            q = 128.0;
            E += 1;
        }
        if (E >= 255) return (uint16_t)(sign | 0x7F80);
        return (uint16_t)(sign | (E << 7) | ((int)q - 128));
    }
    q = nearbyint(ldexp(a, 133));     /* subnormal: m * 2^-133 */
    if (q >= 128.0) return (uint16_t)(sign | 0x0080);
    return (uint16_t)(sign | (int)q);
}

int svdq_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static int nibble(const uint8_t* rowp, int64_t k) {
    return (rowp[k >> 1] >> (4 * (k & 1))) & 15;
}

/*
 * y[i][n] for every requested row m = rows[i] (all rows 0..M-1 when rows is
 * NULL) and every column n < N (h16(x) below is bf16(x), or f16(x) when
 * half_io is 1):
 *
 *   main(m,n) = sum_{g < K/16} e4m3(ascales[g][m]) * e4m3(wscales[g][n])
 *                             * sum_{k = 16g}^{16g+15} e2m1(a(m,k)) * e2m1(w(n,k))
 *   lora(m,n) = sum_{r < R} lora_act_in[m][r] * h16(lora_up[n][r])
 *   y(m,n)    = h16(wcscale[n]) * main(m,n) + h16(bias[n]) + lora(m,n)
 *
 * main_out (nullable) receives main(m,n) in the same [nrows, N] layout.
 * Returns 0, or -1 for bad arguments / allocation failure.
 */
int svdq_oracle_forward_io(const uint8_t* act, const uint8_t* wgt,
                           const uint8_t* ascales, const uint8_t* wscales,
                           const float* lora_act_in, const uint16_t* lora_up,
                           const uint16_t* wcscale, const uint16_t* bias,
                           int64_t M, int64_t N, int64_t K, int64_t R,
                           const int64_t* rows, int64_t nrows,
                           double* y, double* main_out, int half_io) {
    double (*h16)(uint16_t) = half_io ? svdq_oracle_f16 : svdq_oracle_bf16;
    int64_t G, i, g, n;
    double* wsc;
    int bad = 0;
    if (!act || !wgt || !ascales || !wscales || !y) return -1;
    if (M < 0 || N < 0 || K < 0 || R < 0 || K % 16) return -1;
    if (R > 0 && (!lora_act_in || !lora_up)) return -1;
    if (!rows) nrows = M;
    for (i = 0; rows && i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= M) return -1;
    G = K / 16;

    /* Decoded weight scales, shared by all rows. */
    wsc = (double*)malloc(sizeof(double) * (size_t)(G * N > 0 ? G * N : 1));
    if (!wsc) return -1;
    for (g = 0; g < G; ++g)
        for (n = 0; n < N; ++n) wsc[g * N + n] = svdq_oracle_e4m3(wscales[g * N + n]);

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (i = 0; i < nrows; ++i) {
        const int64_t m = rows ? rows[i] : i;
        const uint8_t* arow = act + m * (K / 2);
        double* a = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        double* asc = (double*)malloc(sizeof(double) * (size_t)(G > 0 ? G : 1));
        int64_t k, gg, nn, r;
        if (!a || !asc) {
            free(a);
            free(asc);
            bad |= 1;
            continue;
        }
        for (k = 0; k < K; ++k) a[k] = svdq_oracle_e2m1(nibble(arow, k));
        for (gg = 0; gg < G; ++gg) asc[gg] = svdq_oracle_e4m3(ascales[gg * M + m]);
        for (nn = 0; nn < N; ++nn) {
            const uint8_t* wrow = wgt + nn * (K / 2);
            double mainv = 0.0, lora = 0.0, wc, b;
            for (gg = 0; gg < G; ++gg) {
                double s = 0.0;
                for (k = 16 * gg; k < 16 * gg + 16; ++k)
                    s += a[k] * svdq_oracle_e2m1(nibble(wrow, k));
                mainv += asc[gg] * wsc[gg * N + nn] * s;
            }
            for (r = 0; r < R; ++r)
                lora += (double)lora_act_in[m * R + r] * h16(lora_up[nn * R + r]);
            wc = wcscale ? h16(wcscale[nn]) : 1.0;
            b = bias ? h16(bias[nn]) : 0.0;
            y[i * N + nn] = wc * mainv + b + lora;
            if (main_out) main_out[i * N + nn] = mainv;
        }
        free(a);
        free(asc);
    }
    free(wsc);
    return bad ? -1 : 0;
}

/* The bf16 operator (lora_up, wcscale, bias in bf16). */
int svdq_oracle_forward(const uint8_t* act, const uint8_t* wgt,
                        const uint8_t* ascales, const uint8_t* wscales,
                        const float* lora_act_in, const uint16_t* lora_up,
                        const uint16_t* wcscale, const uint16_t* bias,
                        int64_t M, int64_t N, int64_t K, int64_t R,
                        const int64_t* rows, int64_t nrows,
                        double* y, double* main_out) {
    return svdq_oracle_forward_io(act, wgt, ascales, wscales, lora_act_in, lora_up, wcscale,
                                  bias, M, N, K, R, rows, nrows, y, main_out, 0);
}
