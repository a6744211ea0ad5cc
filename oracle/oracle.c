/*
 * TEST INFRASTRUCTURE -- the float64 CPU oracle for the MXFP4 routed expert
 * linear. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it. The CUDA library never links or calls it, and it shares
 * no code, header, table or constant with the CUDA library.
 *
 * What it computes (problem statement "MXFP4 Routed Expert Linear", Kimi K3,
 * sections "What is stored in one group", "Apply the shared group scale",
 * "Reconstruct the matrix in the right orientation", "Route, weight, and add
 * the shared path"; restated formally on the tensortonic page of the same
 * name):
 *
 *   W_e[o, 32 g + 2 j    ] = LUT[ b & 15 ] * 2^(s - 127)
 *   W_e[o, 32 g + 2 j + 1] = LUT[ b >> 4 ] * 2^(s - 127)
 *       with b = packed[e, o, g, j] and s = scales[e, o, g];
 *   y_t = y_shared_t + sum_k p[t, k] * W_{sel[t, k]} x_t.
 *
 * The steps follow the page's "Implementation order": start from a copy of
 * the shared output, split each byte into low then high nibble, look the code
 * up in the E2M1 table, scale the group by 2^(s-127), take the dot product of
 * the reconstructed row with the token, weight it and add it.
 *
 * Arithmetic is float64. bf16 and fp32 inputs convert to float64 exactly,
 * every decoded weight LUT * 2^(s-127) is an exact double for every byte s,
 * so the only rounding is in the float64 products and sums.
 *
 * Alongside the result it returns abs_terms[t, o] = |y_shared[t, o]| +
 * sum_k sum_i |p[t,k] * W[o,i] * x[t,i]|, the scale that the comparison
 * tolerance is measured against.
 *
 * Readings where the pages are silent: an expert index outside [0, E) breaks
 * the stated precondition; such a pair contributes nothing and is counted in
 * the return value. Duplicate picks within a token are summed slot by slot.
 *
 * Parity: pinned (see tests/oracle_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* The 16-entry E2M1 value table printed on the problem page (starter code). */
static const double E2M1_TABLE[16] = {
    0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};

/* One reconstructed weight: element i of row o of expert e. */
static double decoded_weight(const uint8_t* packed, const uint8_t* scales,
                             int64_t O, int64_t G, int64_t e, int64_t o,
                             int64_t i) {
    int64_t g = i / 32;                 /* group of 32 input positions      */
    int64_t within = i % 32;            /* position inside the group        */
    int64_t j = within / 2;             /* byte of the group holding it     */
    uint8_t b = packed[((e * O + o) * G + g) * 16 + j];
    int code = (within % 2 == 0) ? (b & 0x0F)        /* low nibble first   */
                                 : ((b >> 4) & 0x0F); /* then the high one  */
    int s = scales[(e * O + o) * G + g];
    return ldexp(E2M1_TABLE[code], s - 127);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * x:        (T, I) float64        packed: (E, O, G, 16) uint8
 * scales:   (E, O, G) uint8       sel:    (T, K) int64
 * p:        (T, K) float64        y_shared: (T, O) float64
 * rows:     token ids to compute (n_rows of them); NULL means 0..T-1
 * out, abs_terms: (n_rows, O) float64, row r belongs to token rows[r]
 * Returns the number of (t, k) pairs whose expert index was out of range,
 * or -1 on a malformed call.
 */
int64_t oracle_expert_linear(const double* x, const uint8_t* packed,
                             const uint8_t* scales, const int64_t* sel,
                             const double* p, const double* y_shared,
                             int64_t T, int64_t E, int64_t I, int64_t O,
                             int64_t K, const int64_t* rows, int64_t n_rows,
                             double* out, double* abs_terms) {
    if (I <= 0 || I % 32 != 0 || T < 0 || E < 0 || O < 0 || K < 0)
        return -1;
    if (rows == NULL) n_rows = T;
    const int64_t G = I / 32;

    /* Pairs whose expert index breaks the precondition are counted once. */
    int64_t bad = 0;
    for (int64_t r = 0; r < n_rows; ++r) {
        const int64_t t = rows ? rows[r] : r;
        for (int64_t k = 0; k < K; ++k)
            if (sel[t * K + k] < 0 || sel[t * K + k] >= E) ++bad;
    }

    /* Every (token, output row) is independent; spread them over threads. */
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int64_t o = 0; o < O; ++o) {
            const int64_t t = rows ? rows[r] : r;
            /* Start from a copy of the shared output. */
            double y = y_shared[t * O + o];
            double a = fabs(y_shared[t * O + o]);
            for (int64_t k = 0; k < K; ++k) {
                const int64_t e = sel[t * K + k];
                if (e < 0 || e >= E) continue;
                const double pk = p[t * K + k];
                double dot = 0.0, mag = 0.0;
                for (int64_t i = 0; i < I; ++i) {
                    const double w = decoded_weight(packed, scales, O, G, e, o, i);
                    const double term = w * x[t * I + i];
                    dot += term;
                    mag += fabs(pk * term);
                }
                y += pk * dot;
                a += mag;
            }
            out[r * O + o] = y;
            abs_terms[r * O + o] = a;
        }
    }
    return bad;
}

/* The reconstructed matrix W_e as float64, (O, I) row-major. */
int oracle_decode_expert(const uint8_t* packed, const uint8_t* scales,
                         int64_t E, int64_t O, int64_t I, int64_t e,
                         double* W) {
    if (I <= 0 || I % 32 != 0 || e < 0 || e >= E) return -1;
    const int64_t G = I / 32;
    for (int64_t o = 0; o < O; ++o)
        for (int64_t i = 0; i < I; ++i)
            W[o * I + i] = decoded_weight(packed, scales, O, G, e, o, i);
    return 0;
}
