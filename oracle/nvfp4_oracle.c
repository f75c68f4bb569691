/*
 * NVFP4 block-scaled GEMM oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the library computes.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header, table or constant with the CUDA path.
 *
 * What is computed (all three pages state the same product):
 *   "nvfp4_group_gemm, submission 498453", custom_kernel docstring and the MMA
 *   loop comment "tCtAcc += tCrA * tCrSFA * tCrB * tCrSFB";
 *   "nvfp4 gemm, submission 125598", same MMA loop comment:
 *
 *     C[m,n] = fp16( sum_k  e2m1(A[m,k]) * e4m3(SFA[m,k/16])
 *                          * e2m1(B[n,k]) * e4m3(SFB[n,k/16]) )
 *
 *   A is M x K and B is N x K, both K-major, two FP4 codes per byte (low nibble
 *   = even k); one E4M3 scale per 16 consecutive k (sf_vec_size = 16 in the
 *   configuration block of submissions 498453 and 125598); C is fp16 row-major
 *   (c_dtype = Float16, and the (m,n,l):(n,1,m*n) C layout of submission 498453,
 *   kernel, "Construct C Tensor for each CTA").
 *
 * Arithmetic: decode by table, accumulate in fp64 sequentially in k, round once
 * from fp64 to fp16 with round-to-nearest-even (the epilogue of submission
 * 407526 converts with __floats2half2_rn, i.e. RNE).  On the inputs this
 * library is measured on, every term is a multiple of 2^-20 and the running
 * sum stays far below 2^53 ulps, so the fp64 sum is exact and the only rounding
 * is the final one.
 *
 * Build: plain C99, -O2 -fopenmp -ffp-contract=off (no fused multiply-add, so
 * the arithmetic is the same on every host).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* Decode tables.                                                             */
/* ------------------------------------------------------------------------- */

static double g_e2m1[16];
static double g_e4m3[256];
static int g_tables_ready = 0;

/* E2M1 (Float4E2M1FN, the ab_dtype of submissions 498453 and 125598):
 * bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa.  Exponent field
 * 0 is subnormal (0.m x 2^0).  The format has no Inf and no NaN. */
static double decode_e2m1_bits(unsigned code) {
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag;
    if (e == 0)
        mag = ldexp((double)m, -1);                 /* m/2 * 2^(1-1) */
    else
        mag = ldexp(1.0 + (double)m / 2.0, (int)e - 1);
    return s ? -mag : mag;
}

/* E4M3 "FN" (Float8E4M3FN, the sf_dtype of submissions 498453 and 125598):
 * bit 7 sign, bits 6..3 exponent with bias 7, bits 2..0 mantissa.  Exponent
 * field 0 is subnormal (m/8 x 2^-6).  No Inf; only S.1111.111 is NaN, so the
 * largest finite magnitude is 1.75 x 2^8 = 448. */
static double decode_e4m3_bits(unsigned code) {
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

static void build_tables(void) {
    if (g_tables_ready) return;
    for (unsigned c = 0; c < 16; ++c) g_e2m1[c] = decode_e2m1_bits(c);
    for (unsigned c = 0; c < 256; ++c) g_e4m3[c] = decode_e4m3_bits(c);
    g_tables_ready = 1;
}

void oracle_e2m1_table(double out[16]) {
    build_tables();
    memcpy(out, g_e2m1, sizeof g_e2m1);
}

void oracle_e4m3_table(double out[256]) {
    build_tables();
    memcpy(out, g_e4m3, sizeof g_e4m3);
}

/* ------------------------------------------------------------------------- */
/* fp64 -> fp16, round to nearest, ties to even, in one step.                 */
/* Overflow goes to +-Inf, fp16 subnormals are kept, NaN -> quiet NaN.        */
/* ------------------------------------------------------------------------- */
uint16_t oracle_f64_to_f16(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0) return sign;

    int E;
    frexp(a, &E);               /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1;              /* floor(log2(a)) */
    /* spacing of fp16 values around a: 2^(e-10) for normals, 2^-24 below 2^-14 */
    int qexp = (e < -14) ? -24 : e - 10;
    double n = ldexp(a, -qexp);  /* exact: scaling by a power of two */
    double fl = floor(n);
    double frac = n - fl;        /* exact: n < 2^12 and has the same ulp as a */
    double r;
    if (frac > 0.5) r = fl + 1.0;
    else if (frac < 0.5) r = fl;
    else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double v = ldexp(r, qexp);   /* the rounded magnitude */

    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -14)) {   /* subnormal: v = mant * 2^-24 */
        return (uint16_t)(sign | (uint16_t)ldexp(v, 24));
    }
    frexp(v, &E);
    e = E - 1;
    if (e + 15 >= 31) return (uint16_t)(sign | 0x7C00u);   /* >= 65536: Inf */
    unsigned mant = (unsigned)(ldexp(v, 10 - e) - 1024.0);
    return (uint16_t)(sign | (uint16_t)((unsigned)(e + 15) << 10) | (uint16_t)mant);
}

void oracle_f64_to_f16_array(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_f16(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Operand decode: the k-th element of a packed K-major row.                  */
/* Byte k/2 of the row holds element k in its low nibble when k is even and   */
/* in its high nibble when k is odd (float4_e2m1fn_x2 packing).               */
/* ------------------------------------------------------------------------- */
static inline unsigned fp4_code(const uint8_t* row, int64_t k) {
    uint8_t byte = row[k >> 1];
    return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 0xF);
}

/* Decode one row of an operand into a_k * sf_{k/16} (the first factor of the
 * product above, exact in fp64). */
static void decode_scaled_row(const uint8_t* codes, const uint8_t* sf, int64_t K, double* out) {
    for (int64_t k = 0; k < K; ++k)
        out[k] = g_e2m1[fp4_code(codes, k)] * g_e4m3[sf[k / 16]];
}

/* Sequential-in-k fp64 sum of the products, plus the sum of their magnitudes
 * (the latter feeds the elementwise tolerance). */
static void dot_row(const double* a, const double* b, int64_t K, double* acc, double* absacc) {
    double s = 0.0, sa = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = a[k] * b[k];
        s += p;
        sa += fabs(p);
    }
    *acc = s;
    *absacc = sa;
}

/* ------------------------------------------------------------------------- */
/* Dense problem, batch of L.                                                 */
/* Layouts (submission 498453 kernel, (m,k,l):(k,1,m*k) operand and           */
/* (m,n,l):(n,1,m*n) C layouts): A [L][M][K/2], B [L][N][K/2],                */
/* SFA [L][M][K/16], SFB [L][N][K/16], C [L][M][N] fp16 bits.                 */
/* acc / absacc may be NULL.                                                  */
/* ------------------------------------------------------------------------- */
int oracle_gemm(const uint8_t* A, const uint8_t* B, const uint8_t* SFA, const uint8_t* SFB,
                int M, int N, int K, int L, uint16_t* C, double* acc, double* absacc,
                int nthreads) {
    if (M < 0 || N < 0 || K < 0 || L < 0 || (K % 16) != 0) return -1;
    build_tables();
    const int64_t kb = K / 2, ks = K / 16;
    double* da = (double*)malloc(sizeof(double) * (size_t)((int64_t)M * K + 1));
    if (!da) return -2;
    int rc = 0;
    for (int l = 0; l < L && rc == 0; ++l) {
        const uint8_t* Al = A + (int64_t)l * M * kb;
        const uint8_t* Bl = B + (int64_t)l * N * kb;
        const uint8_t* SFAl = SFA + (int64_t)l * M * ks;
        const uint8_t* SFBl = SFB + (int64_t)l * N * ks;
        for (int m = 0; m < M; ++m)
            decode_scaled_row(Al + (int64_t)m * kb, SFAl + (int64_t)m * ks, K, da + (int64_t)m * K);
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
        {
            double* db = (double*)malloc(sizeof(double) * (size_t)(K + 1));
            if (!db) {
#pragma omp atomic write
                rc = -2;
            }
#pragma omp for schedule(dynamic, 4)
            for (int n = 0; n < N; ++n) {
                if (!db) continue;
                decode_scaled_row(Bl + (int64_t)n * kb, SFBl + (int64_t)n * ks, K, db);
                for (int m = 0; m < M; ++m) {
                    double s, sa;
                    dot_row(da + (int64_t)m * K, db, K, &s, &sa);
                    int64_t o = ((int64_t)l * M + m) * N + n;
                    C[o] = oracle_f64_to_f16(s);
                    if (acc) acc[o] = s;
                    if (absacc) absacc[o] = sa;
                }
            }
            free(db);
        }
    }
    free(da);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Selected output elements only (used on problems too large to run whole).   */
/* Point i is (ls[i], ms[i], ns[i]); layouts as in oracle_gemm.               */
/* ------------------------------------------------------------------------- */
int oracle_gemm_points(const uint8_t* A, const uint8_t* B, const uint8_t* SFA, const uint8_t* SFB,
                       int M, int N, int K, int L, int64_t npts,
                       const int* ls, const int* ms, const int* ns,
                       uint16_t* C, double* acc, double* absacc, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || L < 0 || (K % 16) != 0) return -1;
    for (int64_t i = 0; i < npts; ++i)
        if (ls[i] < 0 || ls[i] >= L || ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return -1;
    build_tables();
    const int64_t kb = K / 2, ks = K / 16;
    int rc = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
    {
        double* da = (double*)malloc(sizeof(double) * (size_t)(2 * (int64_t)K + 2));
        double* db = da ? da + K + 1 : NULL;
        if (!da) {
#pragma omp atomic write
            rc = -2;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < npts; ++i) {
            if (!da) continue;
            int64_t l = ls[i], m = ms[i], n = ns[i];
            decode_scaled_row(A + (l * M + m) * kb, SFA + (l * M + m) * ks, K, da);
            decode_scaled_row(B + (l * N + n) * kb, SFB + (l * N + n) * ks, K, db);
            double s, sa;
            dot_row(da, db, K, &s, &sa);
            C[i] = oracle_f64_to_f16(s);
            if (acc) acc[i] = s;
            if (absacc) absacc[i] = sa;
        }
        free(da);
    }
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Grouped problem: G independent problems, each with its own pointers and    */
/* M/N/K/L (submission 407526, group_gemm; submission 498453, custom_kernel   */
/* docstring: "each group has its own a, b, c, sfa, sfb").  The work is one   */
/* flat parallel loop over every (group, l, n) output column, so that group   */
/* indexing is exercised independently of the single-problem routine.         */
/* ------------------------------------------------------------------------- */
int oracle_gemm_grouped(int G, const uint8_t* const* A, const uint8_t* const* B,
                        const uint8_t* const* SFA, const uint8_t* const* SFB,
                        const int* M, const int* N, const int* K, const int* L,
                        uint16_t* const* C, int nthreads) {
    if (G < 0) return -1;
    build_tables();
    int64_t* first = (int64_t*)malloc(sizeof(int64_t) * (size_t)(G + 1));
    if (!first) return -2;
    first[0] = 0;
    for (int g = 0; g < G; ++g) {
        if (M[g] < 0 || N[g] < 0 || K[g] < 0 || L[g] < 0 || (K[g] % 16) != 0) { free(first); return -1; }
        first[g + 1] = first[g] + (int64_t)L[g] * N[g];
    }
    int rc = 0;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : omp_get_max_threads())
    {
        int64_t kmax = 1;
        for (int g = 0; g < G; ++g) if (K[g] > kmax) kmax = K[g];
        double* da = (double*)malloc(sizeof(double) * (size_t)(2 * kmax + 2));
        double* db = da ? da + kmax + 1 : NULL;
        if (!da) {
#pragma omp atomic write
            rc = -2;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t col = 0; col < first[G]; ++col) {
            if (!da) continue;
            int g = 0;
            while (col >= first[g + 1]) ++g;
            int64_t r = col - first[g];
            int64_t l = r / N[g], n = r % N[g];
            int64_t Kg = K[g], kb = Kg / 2, ks = Kg / 16, Mg = M[g], Ng = N[g];
            decode_scaled_row(B[g] + (l * Ng + n) * kb, SFB[g] + (l * Ng + n) * ks, Kg, db);
            for (int64_t m = 0; m < Mg; ++m) {
                decode_scaled_row(A[g] + (l * Mg + m) * kb, SFA[g] + (l * Mg + m) * ks, Kg, da);
                double s, sa;
                dot_row(da, db, Kg, &s, &sa);
                C[g][(l * Mg + m) * Ng + n] = oracle_f64_to_f16(s);
            }
        }
        free(da);
    }
    free(first);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Scale-factor repack, the layout the tensor-core path consumes.             */
/*                                                                            */
/* Submission 125598's custom_kernel docstring gives the logical shape of the */
/* permuted scales as [32, 4, rest_m, 4, rest_k, l]: row r = r0 + 32*r1 +     */
/* 128*rm, scale column c = c0 + 4*ck.  Submission 407526's TMA producer      */
/* (grouped_kernel, "SFA_base"/"sf_byte") reads one contiguous 512-byte atom  */
/* per (rm, ck) at byte (rm*rest_k + ck)*512, with rest_k = K/64, and 2048    */
/* bytes (four atoms) per 256-wide k-tile.  Inside an atom, the 32x128b       */
/* tensor-memory copy moves 32 rows of 16 bytes, and the same producer's      */
/* sfb_lane offset of 2 columns for rows 64..127 of a 128-row atom places     */
/* r1 at a 4-byte stride: byte = r0*16 + r1*4 + c0.                           */
/*                                                                            */
/* rest_k is padded up to a multiple of 4 atoms (whole 256-wide k-tiles) and  */
/* rest_m to whole 128-row blocks; padding bytes are zero.  For K a multiple  */
/* of 256 the padding in k is empty.  Input [L][rows][K/16], output           */
/* [L][rest_m][rest_k_padded][512].                                           */
/* ------------------------------------------------------------------------- */
int64_t oracle_repacked_bytes(int rows, int K, int L) {
    if (rows < 0 || K < 0 || L < 0 || (K % 16) != 0) return -1;
    int64_t rest_m = ((int64_t)rows + 127) / 128;
    int64_t rest_k = (((int64_t)K + 255) / 256) * 4;
    return (int64_t)L * rest_m * rest_k * 512;
}

int oracle_repack_scales(const uint8_t* sf, int rows, int K, int L, uint8_t* out) {
    if (oracle_repacked_bytes(rows, K, L) < 0) return -1;
    const int64_t cols = K / 16;
    const int64_t rest_m = ((int64_t)rows + 127) / 128;
    const int64_t rest_k = (((int64_t)K + 255) / 256) * 4;
    int64_t o = 0;
    for (int64_t l = 0; l < L; ++l)
        for (int64_t rm = 0; rm < rest_m; ++rm)
            for (int64_t ck = 0; ck < rest_k; ++ck)
                for (int64_t r0 = 0; r0 < 32; ++r0)
                    for (int64_t r1 = 0; r1 < 4; ++r1)
                        for (int64_t c0 = 0; c0 < 4; ++c0) {
                            int64_t r = rm * 128 + r1 * 32 + r0;
                            int64_t c = ck * 4 + c0;
                            out[o++] = (r < rows && c < cols) ? sf[(l * rows + r) * cols + c] : 0;
                        }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Quantization to NVFP4: the step that produces A, B and their scales.       */
/*                                                                            */
/* The pages take A, B, SFA and SFB already quantized (the harness generates  */
/* them) and print no quantizer, so this is the plainest reading of the       */
/* formats they name (E2M1 codes, one E4M3 scale per 16 consecutive k),       */
/* stated in IEEE fp32 on both the oracle and the GPU side:                   */
/*   amax    = max |x_i| over the 16 values of a block                        */
/*   sf      = E4M3(amax / 6)    6 = largest E2M1 magnitude; round to nearest, */
/*                               ties to the even code; finite values above    */
/*                               448 give 448                                  */
/*   d       = the value of sf                                                 */
/*   code_i  = E2M1(x_i / d)     round to nearest on {0,.5,1,1.5,2,3,4,6},     */
/*                               ties to the even code, magnitudes above 6     */
/*                               give 6, sign bit = sign bit of x_i / d;       */
/*                               d = 0 gives code 0                            */
/* x / d and amax / 6 are single correctly rounded fp32 divisions.            */
/* ------------------------------------------------------------------------- */

/* Index of the table entry nearest to v >= 0 among codes 0..ncodes-1 (whose */
/* values increase with the code), by plain scan; a tie goes to the even     */
/* code.                                                                     */
static unsigned nearest_code(double v, const double* tab, unsigned ncodes) {
    unsigned best = 0;
    double bd = fabs(v - tab[0]);
    for (unsigned c = 1; c < ncodes; ++c) {
        double d = fabs(v - tab[c]);
        if (d < bd || (d == bd && (c & 1u) == 0 && (best & 1u) == 1)) {
            best = c;
            bd = d;
        }
    }
    return best;
}

uint8_t oracle_e4m3_encode(float v) {
    build_tables();
    if (isnan(v)) return 0x7F;
    double a = fabs((double)v);
    unsigned c = a >= 448.0 ? 0x7Eu : nearest_code(a, g_e4m3, 0x7F); /* finite codes 0x00..0x7E */
    return (uint8_t)(c | (signbit(v) ? 0x80u : 0u));
}

uint8_t oracle_e2m1_encode(float v) {
    build_tables();
    double a = fabs((double)v);
    unsigned c = a >= 6.0 ? 7u : nearest_code(a, g_e2m1, 8);
    return (uint8_t)(c | (signbit(v) ? 8u : 0u));
}

void oracle_e4m3_encode_array(const float* v, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(v[i]);
}

void oracle_e2m1_encode_array(const float* v, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_encode(v[i]);
}

/* x [L][rows][K] fp32 (the exact values of bf16 / fp16 inputs) -> codes      */
/* [L][rows][K/2] (low nibble = even k) and row-major scales [L][rows][K/16]. */
int oracle_quantize(const float* x, int rows, int K, int L, uint8_t* codes, uint8_t* sf) {
    if (rows < 0 || K < 0 || L < 0 || (K % 16) != 0) return -1;
    build_tables();
    const int64_t nrow = (int64_t)L * rows;
#pragma omp parallel for schedule(static)
    for (int64_t lr = 0; lr < nrow; ++lr) {
        const float* xr = x + lr * K;
        uint8_t* cr = codes + lr * (K / 2);
        uint8_t* sr = sf + lr * (K / 16);
        for (int64_t b = 0; b < K / 16; ++b) {
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float m = fabsf(xr[b * 16 + i]);
                if (m > amax) amax = m;
            }
            const uint8_t sc = oracle_e4m3_encode(amax / 6.0f);
            const float d = (float)g_e4m3[sc];
            sr[b] = sc;
            for (int i = 0; i < 16; i += 2) {
                const float x0 = xr[b * 16 + i], x1 = xr[b * 16 + i + 1];
                const uint8_t q0 = d == 0.0f ? 0 : oracle_e2m1_encode(x0 / d);
                const uint8_t q1 = d == 0.0f ? 0 : oracle_e2m1_encode(x1 / d);
                cr[(b * 16 + i) / 2] = (uint8_t)(q0 | (q1 << 4));
            }
        }
    }
    return 0;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
