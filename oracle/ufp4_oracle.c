/*
 * UFP4 oracle: a plain, single-threaded, deliberately slow C restatement of
 * the fused Random Hadamard Transform + block-scaled 4-bit quantizer.
 *
 * THIS IS TEST INFRASTRUCTURE.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header, table or
 * constant generator with the CUDA library; the two meet only through the
 * seeded input generators and the documented output layout.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC (no FTZ/DAZ),
 * so every float operation below is one IEEE-754 binary32 operation rounded
 * to nearest-even, in the order written.
 *
 * Sources (pages on the UFP4 recipe and on 2D block FP4 training):
 *  [UFP4-data]   UFP4 summary (hyper.ai, arXiv 2606.20381), section "数据集"
 *                (format codebooks G, block partition, s_B = block amax / max
 *                level, RTNE and SR rounding, Q_G(T) = dequantized value).
 *  [UFP4-method] same page, section "方法": Sylvester recursion H_2n,
 *                H_n^T H_n = I, H'_n = S_n H_n, Y = XW^T = (XH')(WH')^T, the
 *                quantized GEMM, the bin-bias law, SR on dY only.
 *  [2D-block]    "Stable FP4 Training via Transposition-Invariant Block
 *                Quantization" tutorial: section "2D 方块量化" (b x b blocks,
 *                S(B)=S(B^T)), truncation-free scale S = 2^ceil(log2(2M/(Qp-Qn))),
 *                stochastic rounding E[roundS(x)] = x.
 *
 * Conventions the pages leave open (each listed in the design notes):
 *  - signs eps_i come from Philox4x32-10 (Salmon et al., SC'11), key =
 *    sign_seed, counter (i/128, 0, 2, 0), bit i%128 of the 128-bit output;
 *  - the FWHT runs stride 1 first (the recursion builds H_2n from two H_n),
 *    the 1/sqrt(2) factors are gathered into one final multiply by
 *    fp32(1/sqrt(n));
 *  - the element scaling is t = z * fp32(1/s), s = fp32(M / qmax);
 *  - RTNE ties go to the even level index; SR rounds the magnitude up iff a
 *    16-bit Philox draw u satisfies u < p * 65536;
 *  - the code keeps the sign of t, except that a zero level is always +0
 *    (nibble 0), so an all-zero input gives all-zero bytes;
 *  - two codes per byte, the lower element index in the low nibble.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_E1M2 = 0, ORC_INT4 = 1, ORC_E2M1 = 2, ORC_E2M1_R2 = 3 };
enum { ORC_RTNE = 0, ORC_SR = 1 };
enum { ORC_SCALE_FP32 = 0, ORC_SCALE_UE8M0 = 1, ORC_SCALE_E4M3 = 2 };

/* ---------------------------------------------------------------- codebooks
 * [UFP4-data]: each format has a normalized codebook G of fixed levels.  The
 * tables hold the non-negative magnitudes; index i is the 3-bit magnitude code.
 *  E1M2: 1 exponent bit, 2 mantissa bits -> 0, 0.25, ..., 1.75 (uniform).
 *  INT4: integers 0..7 (symmetric range -7..7; -8 is not used).
 *  E2M1: 2 exponent bits, 1 mantissa bit -> 0,0.5,1,1.5,2,3,4,6 (non-uniform).
 *  E2M1_R2: the range-limited use of E2M1 -- only its levels up to 2, i.e. the
 *  uniform sub-grid 0, 0.5, 1, 1.5, 2 (blocks scaled so that amax maps to 2),
 *  so the codes stay native E2M1 codes.  A reading of the UFP4 summary,
 *  section "实验" (a uniform grid cannot simply be substituted on native FP4
 *  hardware): the uniform part of E2M1 is what such a substitution can use.
 * NLEV is the number of levels a grid rounds to; the last one is qmax.
 */
static const double LEVELS[4][8] = {
    {0.0, 0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75},
    {0.0, 1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0},
    {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0},
    {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0},
};
static const int NLEV[4] = {8, 8, 8, 5};

double orc_level(int grid, int idx) { return LEVELS[grid][idx]; }
double orc_qmax(int grid) { return LEVELS[grid][NLEV[grid] - 1]; }
int orc_num_levels(int grid) { return NLEV[grid]; }

/* ----------------------------------------------------------- Philox4x32-10
 * Counter-based generator of Salmon, Moraes, Dror, Shaw, "Parallel random
 * numbers: as easy as 1, 2, 3" (SC'11): ten rounds of two 32x32->64 bit
 * multiplications by the constants 0xD2511F53 and 0xCD9E8D57, the key bumped
 * by the Weyl constants 0x9E3779B9 / 0xBB67AE85 between rounds. */
void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* ------------------------------------------------------------ random signs
 * [UFP4-method]: S_n = diag(eps_1..eps_n), eps_i in {-1,+1}.  eps_i = 1 - 2*b_i
 * where b_i is bit (i % 32) of word (i % 128) / 32 of Philox(key = sign_seed,
 * counter = (i / 128, 0, 2, 0)). */
void orc_signs(uint64_t sign_seed, int n, int8_t* eps) {
    uint32_t key[2] = {(uint32_t)sign_seed, (uint32_t)(sign_seed >> 32)};
    for (int i = 0; i < n; ++i) {
        uint32_t ctr[4] = {(uint32_t)(i / 128), 0u, 2u, 0u};
        uint32_t w[4];
        orc_philox4x32_10(ctr, key, w);
        uint32_t bit = (w[(i % 128) / 32] >> (i % 32)) & 1u;
        eps[i] = bit ? (int8_t)-1 : (int8_t)1;
    }
}

/* ------------------------------------------------------------------ bf16 */
static float bf16_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static int is_pow2(int n) { return n >= 1 && (n & (n - 1)) == 0; }

/* fp32(1/sqrt(n)): exact for n = 4^j, correctly rounded otherwise (the double
 * value 1/sqrt(n) rounds to the same float as the exact real, because double
 * sqrt and division are correctly rounded and no tie can occur). */
static float inv_sqrt_n(int n) { return (float)(1.0 / sqrt((double)n)); }

/* ---------------------------------------------------------------- the RHT
 * [UFP4-method]: z = x H'_n = x S_n H_n on each length-n segment.  H_n is the
 * Sylvester matrix built by H_2n = (1/sqrt 2)[[H_n, H_n], [H_n, -H_n]]: the
 * recursion transforms the two halves first and combines them last, so the
 * butterfly runs strides 1, 2, ..., n/2 in that order, each stage mapping a
 * pair (a, b) at indices (i, i+h), bit h of i clear, to (a+b, a-b).  All
 * normalisation factors are gathered in one multiply by fp32(1/sqrt(n)). */
static void rht_segment(float* v, int n, const int8_t* eps, float inv_s) {
    if (n == 1) return; /* n = 1 switches the transform off (identity, no sign) */
    for (int i = 0; i < n; ++i) v[i] = v[i] * (float)eps[i];
    for (int h = 1; h < n; h *= 2) {
        for (int i = 0; i < n; ++i) {
            if (i & h) continue;
            float a = v[i], b = v[i + h];
            v[i] = a + b;
            v[i + h] = a - b;
        }
    }
    for (int i = 0; i < n; ++i) v[i] = v[i] * inv_s;
}

/* z[rows x cols] = RHT along each row of the bf16 matrix x (leading dim ld). */
int orc_rht_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int n,
                 uint64_t sign_seed, float* z) {
    if (!is_pow2(n) || n > 256 || cols % n != 0) return 1;
    int8_t eps[256];
    orc_signs(sign_seed, n, eps);
    float inv_s = inv_sqrt_n(n);
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c) z[r * cols + c] = bf16_to_float(x[r * ld + c]);
        for (int64_t c0 = 0; c0 < cols; c0 += n) rht_segment(&z[r * cols + c0], n, eps, inv_s);
    }
    return 0;
}

/* --------------------------------------------------------- block scale
 * [UFP4-data]: s_B = (block amax) / (largest codebook magnitude).
 * fp32 mode: s = fp32(M / qmax) and the elements are multiplied by
 * r = fp32(1 / s); an all-zero block has s = 0 and r = 0. */
static void scale_fp32(float M, int grid, float* s_out, float* r_out) {
    float qmax = (float)orc_qmax(grid);
    float s = M / qmax;
    *s_out = s;
    *r_out = (s == 0.0f) ? 0.0f : 1.0f / s;
}

/* [2D-block], truncation-free scaling: S = 2^ceil(log2(2M / (Qp - Qn))).  For
 * the symmetric grids here Qp = qmax and Qn = -qmax, so 2M/(Qp-Qn) = M/qmax and
 * the exponent is the smallest integer e with M <= qmax * 2^e.  The comparison
 * is done in double, where qmax * 2^e is exact.  e is kept in [-127, 127] so
 * that it fits an UE8M0 byte (e + 127); the lower clamp only widens the
 * interval, so it stays truncation-free. */
int orc_po2_exponent(float M, int grid) {
    double qmax = orc_qmax(grid);
    if (M == 0.0f) return -127;
    int e = (int)ceil(log2((double)M / qmax));
    while ((double)M > ldexp(qmax, e)) ++e;
    while (e > -1000 && (double)M <= ldexp(qmax, e - 1)) --e;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* ---------------------------------------------------- two-level scale
 * The "two-level" option of the scale hierarchy [UFP4-method: the scale
 * hierarchy is chosen for hardware efficiency]: a per-tensor fp32 scale g
 * times a per-block scale stored as an E4M3 byte.  E4M3 (the OCP FP8 format
 * without infinities): 1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
 * normal values (1 + m/8) 2^(e-7), e = 1..15 (e = 15 with m = 7 is NaN, so the
 * largest finite value is 448 = 1.75 * 2^8); subnormals m * 2^-9.
 * Reading of the definition:
 *   T = max |z| over the whole tensor (z = the RHT output),
 *   g = fp32(T / fp32(qmax * 448))  (the block scale of amax lands on 448),
 *   per block: b = fp32(fp32(M / qmax) / g), stored as the E4M3 byte of b
 *   rounded to nearest even and saturated at 448 (0 when g = 0),
 *   s = fp32(e4m3(b) * g), elements scaled by fp32(1 / s) (0 when s = 0). */
uint8_t orc_e4m3_encode(double a) {
    if (!(a > 0.0)) return 0;
    if (a >= 448.0) return 0x7E;
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;          /* a in [2^E, 2^(E+1)) */
    if (E < -6) E = -6;      /* subnormals share the step of the smallest binade */
    double step = ldexp(1.0, E - 3);
    double k = a / step;     /* exact: scaling by a power of two */
    double fl = floor(k), rem = k - fl;
    double m = (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) ? fl + 1.0 : fl;
    double v = m * step;
    if (v > 448.0) v = 448.0;
    if (v < ldexp(1.0, -6)) return (uint8_t)(v / ldexp(1.0, -9));  /* subnormal: m * 2^-9 */
    int f2;
    frexp(v, &f2);
    int VE = f2 - 1;
    int mant = (int)((v / ldexp(1.0, VE) - 1.0) * 8.0);
    return (uint8_t)(((VE + 7) << 3) | mant);
}

double orc_e4m3_decode(uint8_t b) {
    int e = (b >> 3) & 15, m = b & 7;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (b & 0x80) ? -v : v;
}

/* g from the tensor amax T (fp32 arithmetic as written above). */
float orc_tensor_scale(float T, int grid) {
    float d = (float)orc_qmax(grid) * 448.0f;
    return T / d;
}

/* ---------------------------------------------------------------- rounding
 * [UFP4-data]: RTNE maps a scaled magnitude to the nearest level of G; an exact
 * tie goes to the level with the even index (the even mantissa / integer LSB,
 * i.e. IEEE round-to-nearest-even in each 4-bit format).  a is in [0, qmax]. */
int orc_round_rtne(int grid, float a) {
    double x = (double)a;
    int best = 0;
    double best_d = fabs(x - LEVELS[grid][0]);
    for (int i = 1; i < NLEV[grid]; ++i) {
        double d = fabs(x - LEVELS[grid][i]);
        if (d < best_d || (d == best_d && (i % 2) == 0 && (best % 2) != 0)) {
            best = i;
            best_d = d;
        }
    }
    return best;
}

/* [UFP4-data] / [2D-block]: stochastic rounding picks one of the two
 * neighbouring levels lo <= a <= hi with probability set by the distance, so
 * that E[SR(a)] = a.  With p = (a - lo) / (hi - lo), the magnitude rounds up
 * iff the 16-bit draw u satisfies u < p * 65536 (so P(up) = ceil(65536 p)/65536). */
int orc_round_sr(int grid, float a, uint32_t u16) {
    double x = (double)a;
    int lo = 0;
    for (int i = 0; i < NLEV[grid]; ++i)
        if (LEVELS[grid][i] <= x) lo = i;
    if (lo == NLEV[grid] - 1) return lo;
    double p = (x - LEVELS[grid][lo]) / (LEVELS[grid][lo + 1] - LEVELS[grid][lo]);
    return ((double)u16 < p * 65536.0) ? lo + 1 : lo;
}

/* 4-bit encodings: E1M2 and E2M1 are sign-magnitude (sign << 3 | index),
 * with the zero level always written as +0; INT4 is two's complement of the
 * signed integer level. */
static uint8_t encode(int grid, int negative, int idx) {
    if (idx == 0) return 0;
    if (grid == ORC_INT4) {
        int k = negative ? -idx : idx;
        return (uint8_t)(k & 0xF);
    }
    return (uint8_t)((negative ? 8 : 0) | idx);
}

/* 16-bit SR draw for output element `lin` (row-major linear index in the
 * quantized tensor's own layout): Philox(key = sr_seed, counter = (g lo, g hi,
 * stream, group)), g = lin / 8; element j = lin % 8 takes the low half of word
 * j/2 when j is even and the high half when j is odd. */
static uint32_t sr_draw(uint64_t sr_seed, uint64_t lin, uint32_t stream, uint32_t group) {
    uint64_t g = lin / 8;
    uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), stream, group};
    uint32_t key[2] = {(uint32_t)sr_seed, (uint32_t)(sr_seed >> 32)};
    uint32_t w[4];
    orc_philox4x32_10(ctr, key, w);
    int j = (int)(lin % 8);
    uint32_t word = w[j / 2];
    return (j % 2 == 0) ? (word & 0xFFFFu) : (word >> 16);
}

/* [UFP4-data]: the element step of the quantizer.  The scaled value t = z * r
 * of an element is clamped to qmax in magnitude, rounded to a level index
 * (RTNE, or SR with the element's 16-bit draw u16) and encoded with t's sign
 * (a zero level is +0). */
static uint8_t element_code(int grid, int round, float t, uint32_t u16) {
    float qmax = (float)orc_qmax(grid);
    float a = fabsf(t);
    if (a > qmax) a = qmax;
    int idx = (round == ORC_RTNE) ? orc_round_rtne(grid, a) : orc_round_sr(grid, a, u16);
    return encode(grid, signbit(t) ? 1 : 0, idx);
}

/* Test entries of the SR rule above, over many draws at once.
 *  orc_round_sr_array:  idx[i] = orc_round_sr(grid, a[i], u16[i]);
 *  orc_round_sr_philox: idx[i] = orc_round_sr(grid, a, draw of output element
 *                       lin0 + i), with the quantizer's counter layout. */
void orc_round_sr_array(int grid, const float* a, const uint16_t* u16, int64_t count, uint8_t* idx) {
    for (int64_t i = 0; i < count; ++i) idx[i] = (uint8_t)orc_round_sr(grid, a[i], u16[i]);
}

void orc_round_sr_philox(int grid, float a, uint64_t sr_seed, uint64_t lin0, int64_t count, uint32_t stream,
                         uint32_t group, uint8_t* idx) {
    for (int64_t i = 0; i < count; ++i)
        idx[i] = (uint8_t)orc_round_sr(grid, a, sr_draw(sr_seed, lin0 + (uint64_t)i, stream, group));
}

/* Test entry: the element step above over given scaled values t[0..count),
 * packed two per byte as the quantizer packs them (element i in the low
 * nibble of byte i/2 when i is even, the high nibble when odd).  u16 holds
 * the draws for SR and may be NULL for RTNE; count is even. */
void orc_round_encode_array(int grid, int round, const float* t, const uint16_t* u16, int64_t count,
                            uint8_t* codes) {
    for (int64_t i = 0; i < count; i += 2) {
        uint8_t lo = element_code(grid, round, t[i], round == ORC_RTNE ? 0u : u16[i]);
        uint8_t hi = element_code(grid, round, t[i + 1], round == ORC_RTNE ? 0u : u16[i + 1]);
        codes[i / 2] = (uint8_t)(lo | (hi << 4));
    }
}

/* --------------------------------------------------------- the quantizer
 * Quantize the bf16 matrix x (rows x cols, leading dimension ld) along its
 * rows: RHT on each length-n segment of a row, then blocks of
 * block_rows x block_cols (1 x 16, 1 x 32, or b x b), then the scale, the
 * rounding and the packing.  Outputs (caller-allocated):
 *   codes  [rows x cols/2] bytes, row-major;
 *   scales [rows/block_rows x cols/block_cols], float (fp32 mode) or uint8
 *          UE8M0 bytes (e + 127).
 * row0 is the index of x's first row in the whole tensor; it only enters the
 * SR counters, so a band of rows can be checked on its own.
 * Returns 0, or 1 on an unsupported argument. */
static int quantize_rows_impl(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int grid,
                              int block_rows, int block_cols, int n, uint64_t sign_seed, int round,
                              uint64_t sr_seed, int scale_fmt, uint32_t stream, uint32_t group,
                              uint64_t row0, float tensor_amax, uint8_t* codes, void* scales,
                              float* tensor_amax_out) {
    if (grid < 0 || grid > 3 || block_rows < 1 || block_cols < 2 || cols % 2) return 1;
    if (scale_fmt < 0 || scale_fmt > 2) return 1;
    if (rows % block_rows || cols % block_cols) return 1;
    float* z = (float*)malloc(sizeof(float) * (size_t)(rows * cols > 0 ? rows * cols : 1));
    if (!z) return 1;
    if (orc_rht_rows(x, rows, cols, ld, n, sign_seed, z)) {
        free(z);
        return 1;
    }
    float qmax = (float)orc_qmax(grid);
    int64_t nbr = rows / block_rows, nbc = cols / block_cols;
    memset(codes, 0, (size_t)(rows * cols / 2));
    /* two-level: the tensor amax (of this call's rows unless given) and g */
    float T = tensor_amax, g = 0.0f;
    if (scale_fmt == ORC_SCALE_E4M3) {
        if (T < 0.0f) {
            T = 0.0f;
            for (int64_t i = 0; i < rows * cols; ++i)
                if (fabsf(z[i]) > T) T = fabsf(z[i]);
        }
        g = orc_tensor_scale(T, grid);
        if (tensor_amax_out) *tensor_amax_out = T;
    }
    for (int64_t bi = 0; bi < nbr; ++bi) {
        for (int64_t bj = 0; bj < nbc; ++bj) {
            /* block amax [UFP4-data] */
            float M = 0.0f;
            for (int64_t r = bi * block_rows; r < (bi + 1) * block_rows; ++r)
                for (int64_t c = bj * block_cols; c < (bj + 1) * block_cols; ++c) {
                    float a = fabsf(z[r * cols + c]);
                    if (a > M) M = a;
                }
            /* scale */
            float rcp;
            if (scale_fmt == ORC_SCALE_FP32) {
                float s;
                scale_fp32(M, grid, &s, &rcp);
                ((float*)scales)[bi * nbc + bj] = s;
            } else if (scale_fmt == ORC_SCALE_E4M3) {
                float sb = M / qmax;
                uint8_t b8 = (g == 0.0f) ? 0 : orc_e4m3_encode((double)(sb / g));
                float s = (float)orc_e4m3_decode(b8) * g;
                rcp = (s == 0.0f) ? 0.0f : 1.0f / s;
                ((uint8_t*)scales)[bi * nbc + bj] = b8;
            } else {
                int e = orc_po2_exponent(M, grid);
                ((uint8_t*)scales)[bi * nbc + bj] = (uint8_t)(e + 127);
                rcp = (float)ldexp(1.0, -e);
            }
            /* scale, clamp, round, encode, pack */
            for (int64_t r = bi * block_rows; r < (bi + 1) * block_rows; ++r)
                for (int64_t c = bj * block_cols; c < (bj + 1) * block_cols; ++c) {
                    float t = z[r * cols + c] * rcp;
                    uint32_t u = 0;
                    if (round != ORC_RTNE) {
                        uint64_t lin = (row0 + (uint64_t)r) * (uint64_t)cols + (uint64_t)c;
                        u = sr_draw(sr_seed, lin, stream, group);
                    }
                    uint8_t nib = element_code(grid, round, t, u);
                    codes[r * (cols / 2) + c / 2] |= (uint8_t)(nib << (4 * (c % 2)));
                }
        }
    }
    free(z);
    return 0;
}

int orc_quantize_rows(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int grid,
                      int block_rows, int block_cols, int n, uint64_t sign_seed, int round,
                      uint64_t sr_seed, int scale_fmt, uint32_t stream, uint32_t group,
                      uint64_t row0, uint8_t* codes, void* scales) {
    if (scale_fmt == ORC_SCALE_E4M3) return 1;  /* needs the tensor amax: orc_quantize_rows_2level */
    return quantize_rows_impl(x, rows, cols, ld, grid, block_rows, block_cols, n, sign_seed, round, sr_seed,
                              scale_fmt, stream, group, row0, -1.0f, codes, scales, NULL);
}

/* Two-level scale (E4M3 block scales x fp32 tensor scale).  tensor_amax < 0:
 * T is the amax of this call's z; else T is given (a band of a larger tensor).
 * T is written to *tensor_amax_out. */
int orc_quantize_rows_2level(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int grid,
                             int block_rows, int block_cols, int n, uint64_t sign_seed, int round,
                             uint64_t sr_seed, uint32_t group, uint64_t row0, float tensor_amax,
                             uint8_t* codes, uint8_t* scales, float* tensor_amax_out) {
    return quantize_rows_impl(x, rows, cols, ld, grid, block_rows, block_cols, n, sign_seed, round, sr_seed,
                              ORC_SCALE_E4M3, 0u, group, row0, tensor_amax, codes, scales, tensor_amax_out);
}

/* Column-wise quantization [2D-block, the transposition problem; UFP4-method,
 * RHT on all three GEMMs]: the quantization of X^T along its rows, i.e. the RHT
 * and the blocks run along X's first dimension.  The outputs are in X^T's
 * layout: codes [cols x rows/2], scales [cols/block_rows' ...].  The oracle
 * builds X^T explicitly and reuses the row-wise routine with SR stream 1. */
int orc_quantize_cols(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int grid,
                      int block_rows, int block_cols, int n, uint64_t sign_seed, int round,
                      uint64_t sr_seed, int scale_fmt, uint32_t group, uint8_t* codes,
                      void* scales) {
    uint16_t* xt = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(rows * cols > 0 ? rows * cols : 1));
    if (!xt) return 1;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) xt[c * rows + r] = x[r * ld + c];
    int rc = orc_quantize_rows(xt, cols, rows, rows, grid, block_rows, block_cols, n, sign_seed,
                               round, sr_seed, scale_fmt, 1u, group, 0u, codes, scales);
    free(xt);
    return rc;
}

/* ------------------------------------------------------------- dequantize
 * [UFP4-data]: inside arithmetic Q_G(T) stands for the dequantized tensor,
 * level(code) * s_B.  fp32 output: fp32(level * s).  With inverse_rht, the
 * rotation is undone: x = z H'^T = z H S (H symmetric), i.e. the same
 * butterfly and the final fp32(1/sqrt(n)) multiply, then the signs. */
static double decode(int grid, uint8_t nib) {
    if (grid == ORC_INT4) {
        int k = (nib & 8) ? (int)nib - 16 : (int)nib;
        return (double)k;
    }
    double v = LEVELS[grid][nib & 7];
    return (nib & 8) ? -v : v;
}

static int dequantize_impl(const uint8_t* codes, const void* scales, int64_t rows, int64_t cols, int grid,
                           int block_rows, int block_cols, int scale_fmt, float tensor_amax, int n,
                           uint64_t sign_seed, int inverse_rht, float* out) {
    if (rows % block_rows || cols % block_cols || cols % 2) return 1;
    const float g = scale_fmt == ORC_SCALE_E4M3 ? orc_tensor_scale(tensor_amax, grid) : 0.0f;
    int64_t nbc = cols / block_cols;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t nib = (uint8_t)((codes[r * (cols / 2) + c / 2] >> (4 * (c % 2))) & 0xF);
            int64_t b = (r / block_rows) * nbc + (c / block_cols);
            float lv = (float)decode(grid, nib);
            float s;
            if (scale_fmt == ORC_SCALE_FP32)
                s = ((const float*)scales)[b];
            else if (scale_fmt == ORC_SCALE_E4M3)
                s = (float)orc_e4m3_decode(((const uint8_t*)scales)[b]) * g;  /* the quantizer's s */
            else
                s = (float)ldexp(1.0, (int)((const uint8_t*)scales)[b] - 127);
            out[r * cols + c] = lv * s;
        }
    if (inverse_rht && n > 1) {
        if (!is_pow2(n) || n > 256 || cols % n) return 1;
        int8_t eps[256];
        orc_signs(sign_seed, n, eps);
        float inv_s = inv_sqrt_n(n);
        for (int64_t r = 0; r < rows; ++r)
            for (int64_t c0 = 0; c0 < cols; c0 += n) {
                float* v = &out[r * cols + c0];
                for (int h = 1; h < n; h *= 2)
                    for (int i = 0; i < n; ++i) {
                        if (i & h) continue;
                        float a = v[i], b = v[i + h];
                        v[i] = a + b;
                        v[i + h] = a - b;
                    }
                for (int i = 0; i < n; ++i) v[i] = (v[i] * inv_s) * (float)eps[i];
            }
    }
    return 0;
}

int orc_dequantize(const uint8_t* codes, const void* scales, int64_t rows, int64_t cols, int grid,
                   int block_rows, int block_cols, int scale_fmt, int n, uint64_t sign_seed,
                   int inverse_rht, float* out) {
    if (scale_fmt == ORC_SCALE_E4M3) return 1;  /* needs the tensor amax: orc_dequantize_2level */
    return dequantize_impl(codes, scales, rows, cols, grid, block_rows, block_cols, scale_fmt, 0.0f, n,
                           sign_seed, inverse_rht, out);
}

int orc_dequantize_2level(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols, int grid,
                          int block_rows, int block_cols, float tensor_amax, int n, uint64_t sign_seed,
                          int inverse_rht, float* out) {
    return dequantize_impl(codes, scales, rows, cols, grid, block_rows, block_cols, ORC_SCALE_E4M3, tensor_amax,
                           n, sign_seed, inverse_rht, out);
}

/* Two-level exact fp64 values for the GEMM reference: level * e4m3(b) * g,
 * the product the block-scaled MMA forms (level * e4m3 block scale) times the
 * tensor scales applied to its output. */
int orc_dequantize_f64_2level(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols, int grid,
                              int block_rows, int block_cols, float tensor_amax, double* out) {
    if (rows % block_rows || cols % block_cols || cols % 2) return 1;
    const double g = (double)orc_tensor_scale(tensor_amax, grid);
    int64_t nbc = cols / block_cols;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t nib = (uint8_t)((codes[r * (cols / 2) + c / 2] >> (4 * (c % 2))) & 0xF);
            int64_t b = (r / block_rows) * nbc + (c / block_cols);
            out[r * cols + c] = decode(grid, nib) * orc_e4m3_decode(scales[b]) * g;
        }
    return 0;
}

/* Exact fp64 dequantized values (level * scale), for the GEMM reference
 * [UFP4-method, quantized GEMM: Y^ = Q_G(X H') Q_G(W H')^T]. */
int orc_dequantize_f64(const uint8_t* codes, const void* scales, int64_t rows, int64_t cols,
                       int grid, int block_rows, int block_cols, int scale_fmt, double* out) {
    if (rows % block_rows || cols % block_cols || cols % 2) return 1;
    int64_t nbc = cols / block_cols;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t nib = (uint8_t)((codes[r * (cols / 2) + c / 2] >> (4 * (c % 2))) & 0xF);
            int64_t b = (r / block_rows) * nbc + (c / block_cols);
            double s = (scale_fmt == ORC_SCALE_FP32)
                           ? (double)((const float*)scales)[b]
                           : ldexp(1.0, (int)((const uint8_t*)scales)[b] - 127);
            out[r * cols + c] = decode(grid, nib) * s;
        }
    return 0;
}

/* ------------------------------------------------------------------ MXFP8
 * [2D-block, section on mixed precision]: the Query and Key projections keep
 * MXFP8, a format with more precision and a wider dynamic range than FP4.
 * The page names the format and nothing more, so its definition is read as
 * the OCP Microscaling format MXFP8 (E4M3): blocks of 32 consecutive
 * elements along a row share one power-of-two scale X = 2^e stored as the
 * E8M0 byte e + 127, with e = floor(log2(max |z|)) - 8 (8 = the exponent of
 * E4M3's largest normal, 448 = 1.75 * 2^8), clamped to [-127, 127]; each
 * element is z / X rounded to E4M3 to nearest even, saturated at 448.  A
 * zero block has byte 0 and codes 0, and a value that rounds to zero is
 * written as +0 (byte 0x00), as for the 4-bit formats.  z is the row-wise
 * RHT of x (n = 1: x itself).  Outputs: codes [rows x cols] E4M3 bytes,
 * scales [rows x cols/32] E8M0 bytes. */
int orc_quantize_rows_mxfp8(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int n,
                            uint64_t sign_seed, uint8_t* codes, uint8_t* scales) {
    if (cols % 32) return 1;
    float* z = (float*)malloc(sizeof(float) * (size_t)(rows * cols > 0 ? rows * cols : 1));
    if (!z) return 1;
    if (orc_rht_rows(x, rows, cols, ld, n, sign_seed, z)) {
        free(z);
        return 1;
    }
    const int64_t nbc = cols / 32;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t bj = 0; bj < nbc; ++bj) {
            const float* zb = &z[r * cols + bj * 32];
            float M = 0.0f;
            for (int i = 0; i < 32; ++i)
                if (fabsf(zb[i]) > M) M = fabsf(zb[i]);
            int e = -127;
            if (M > 0.0f) {
                int e2;
                frexp((double)M, &e2); /* M in [2^(e2-1), 2^e2) */
                e = (e2 - 1) - 8;
                if (e < -127) e = -127;
                if (e > 127) e = 127;
            }
            scales[r * nbc + bj] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i) {
                double t = ldexp((double)zb[i], -e); /* exact */
                uint8_t b = orc_e4m3_encode(fabs(t));
                if (b != 0 && t < 0.0) b |= 0x80;
                codes[r * cols + bj * 32 + i] = b;
            }
        }
    free(z);
    return 0;
}

/* Exact fp64 values e4m3(code) * 2^(byte - 127) of an MXFP8 tensor. */
int orc_dequantize_f64_mxfp8(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                             double* out) {
    if (cols % 32) return 1;
    const int64_t nbc = cols / 32;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = orc_e4m3_decode(codes[r * cols + c]) *
                                ldexp(1.0, (int)scales[r * nbc + c / 32] - 127);
    return 0;
}
