/*
 * fp4gemv_oracle.c -- FP64 CPU oracle for the NVFP4 small-M GEMV family.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent reference that the
 * CUDA library is checked against.  Only tests/, __graft_entry__.smoke() and
 * the cpu_baseline leg of bench.py may load it.  It shares no code, header,
 * table or constant with the CUDA path.
 *
 * Everything here is a plain, slow, direct transcription of what the pages
 * define (cited per function as "page / section"):
 *   [nvfp4_gemv]   vllm.models.flint.ops.nvfp4_gemv, module docstring and the
 *                  nvfp4_gemv / bf16_gemv / dequantize_rows sections.
 *   [linear]       vllm.models.flint.ops.linear, _dequant_gemm and
 *                  _swizzled_scale_buffer sections.
 *   [moe_gemv]     vllm.models.flint.ops.moe_gemv, module docstring and the
 *                  gate_up / down_combine sections.
 *   [flashinfer]   vllm.model_executor.kernels.linear.nvfp4.flashinfer, the
 *                  W4A4 kernels' apply_weights (activation quantisation; its
 *                  arithmetic is a reading, stated at orc_quantize_act).
 *
 * Arithmetic: products and sums in double (every product of a bf16 activation
 * and an exactly-dequantised weight has <= 14 significant bits, so products
 * are exact; sums carry at most K * 2^-53 relative error).  The final and
 * intermediate roundings the pages name (fp32 scale, bf16 outputs) are done
 * explicitly, each as ONE rounding from the double value (no double rounding
 * through float on the way to bf16).
 *
 * Alternatives at intermediate roundings: the pages round some intermediate
 * values to bf16 before the output is formed (the gate / up outputs before
 * silu_mul, y_j, y_shared and the top-k sum in down_combine).  An
 * fp32-accumulating implementation computes such a value with a tiny
 * relative error, so where the exact value lies next to a bf16 rounding
 * midpoint both neighbours are correct.  Each such intermediate carries the
 * other neighbour as an alternative (relative window 2^-16 for the long dot
 * products; the rigorous fp32 bound for the top-k sum), and each output
 * reports (nominal, lo, hi): nominal takes every intermediate at its own
 * rounding, [lo, hi] is the hull of the outputs over the alternatives.
 * Final roundings get no window: an output with no intermediate rounding
 * has lo == hi == nominal, and the acceptance rule compares it with the
 * nominal value under the stated per-element tolerance.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* E2M1 magnitudes indexed by the low three code bits (e1 e0 m): the FP4
 * format of the NVFP4 weight codes [nvfp4_gemv, module docstring].  Sign is
 * code bit 3. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1(int code)
{
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

/* float8_e4m3fn from its bit fields (the dtype the pages view the block
 * scales as [nvfp4_gemv, dequantize_rows]): 1 sign, 4 exponent (bias 7),
 * 3 mantissa bits, no infinities, S.1111.111 is NaN. */
double orc_e4m3(int b)
{
    int s = (b >> 7) & 1, E = (b >> 3) & 15, M = b & 7;
    double v;
    if (E == 15 && M == 7) return NAN;
    if (E == 0) v = ldexp((double)M / 8.0, -6);
    else        v = ldexp(1.0 + (double)M / 8.0, E - 7);
    return s ? -v : v;
}

static double bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double orc_bf16_value(int h) { return bf16_to_double((uint16_t)h); }

/* Round a double to bf16 (8 significant bits, 8-bit exponent) in ONE step,
 * round-to-nearest-even, with gradual underflow and overflow to infinity. */
uint16_t orc_bf16_rne(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v), q, n, r, res;
    int ex, lead;
    float f;
    uint32_t u;
    if (isnan(v)) return (uint16_t)(sign | 0x7FC0u);
    if (isinf(v)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;
    frexp(a, &ex);                 /* a = f * 2^ex, f in [0.5, 1) */
    lead = ex - 1;                 /* exponent of the leading bit */
    if (lead < -126) lead = -126;  /* subnormal binade shares the min quantum */
    q = ldexp(1.0, lead - 7);      /* one bf16 ulp in this binade */
    n = a / q;                     /* exact: power-of-two scaling */
    r = nearbyint(n);              /* default mode: ties to even */
    res = r * q;
    if (res >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
    f = (float)res;                /* exact: res is a bf16 value */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

/* Round a double to fp32 (one step, ties to even). */
static double f32(double v) { return (double)(float)v; }

/* ------------------------------------------------------------------------ */
/* 128x4-swizzled block-scale layout                                         */
/* ------------------------------------------------------------------------ */

static int64_t roundup(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

/* Bytes of the flat scale buffer for a [rows, K] weight: the size formula of
 * _swizzled_scale_buffer [linear]. */
int64_t orc_scale_bytes(int64_t rows, int64_t K)
{
    return roundup(rows, 128) * roundup(K / 16, 4);
}

/* Byte offset of the scale of (row r, 16-wide K block kb).  Reading of the
 * "128x4" layout (the pages give only its name and size): rows are padded to
 * 128 and K blocks to 4; each (128-row, 4-block) tile is one 512-byte chunk,
 * chunks ordered K-block-group fastest within a 128-row group; inside a chunk
 * the byte index is (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4. */
int64_t orc_swz(int64_t r, int64_t kb, int64_t K)
{
    int64_t kbp = roundup(K / 16, 4);
    return ((r / 128) * (kbp / 4) + kb / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + kb % 4;
}

/* Inverse of orc_swz for offsets inside the used region (row < roundup(rows,
 * 128), kb < roundup(K/16, 4)): writes r, kb. */
void orc_unswz(int64_t off, int64_t K, int64_t* r, int64_t* kb)
{
    int64_t kbp = roundup(K / 16, 4);
    int64_t chunk = off / 512, in = off % 512;
    int64_t rg = chunk / (kbp / 4), kg = chunk % (kbp / 4);
    *r = rg * 128 + ((in / 4) % 4) * 32 + in / 16;
    *kb = kg * 4 + in % 4;
}

/* ------------------------------------------------------------------------ */
/* Dequantisation                                                            */
/* ------------------------------------------------------------------------ */

/* code(W, n, k): element 2j is the LOW nibble of byte j [nvfp4_gemv, module
 * docstring: each byte packs two E2M1 codes, the lower-indexed one in the low
 * nibble]. */
static int fp4_code(const uint8_t* wrow, int64_t k)
{
    uint8_t b = wrow[k / 2];
    return (k & 1) ? (b >> 4) : (b & 0xF);
}

/* Wd[r, k] = e2m1(code) * e4m3(scale(r, k/16)), exact in double and in bf16
 * [nvfp4_gemv, module docstring: the product of the two is the weight, with
 * no rounding]. */
static void dequant_row(const uint8_t* w, const uint8_t* sf, int64_t r, int64_t K, double* out)
{
    const uint8_t* wrow = w + r * (K / 2);
    for (int64_t k = 0; k < K; ++k) {
        double s = orc_e4m3(sf[orc_swz(r, k / 16, K)]);
        out[k] = orc_e2m1(fp4_code(wrow, k)) * s;
    }
}

/* dequantize_rows [nvfp4_gemv, dequantize_rows]: bf16 [rows, K] of the exact
 * products, global scale not applied.  Rows r0..r1-1 are written. */
void orc_dequant_rows(const uint8_t* w, const uint8_t* sf, int64_t K, int64_t r0, int64_t r1,
                      double* tmp, uint16_t* out)
{
    for (int64_t r = r0; r < r1; ++r) {
        dequant_row(w, sf, r, K, tmp);
        for (int64_t k = 0; k < K; ++k) out[r * K + k] = orc_bf16_rne(tmp[k]);
    }
}

/* Dot products                                                              */
/* ------------------------------------------------------------------------ */

/* sum_k x[k] * wd[k] in double. */
static double dot(const uint16_t* x, const double* wd, int64_t K)
{
    double a = 0.0;
    for (int64_t k = 0; k < K; ++k) a += bf16_to_double(x[k]) * wd[k];
    return a;
}

/* Dense NVFP4 accumulators for rows in `rows[0..nrows)`: acc[m * nrows + i]
 * = sum_k x[m, k] * Wd[rows[i], k] [nvfp4_gemv, nvfp4_gemv]. */
void orc_gemv_acc(const uint16_t* x, int64_t ldx, int64_t M, const uint8_t* w, const uint8_t* sf,
                  int64_t K, const int64_t* rows, int64_t nrows, double* tmp, double* acc)
{
    for (int64_t i = 0; i < nrows; ++i) {
        dequant_row(w, sf, rows[i], K, tmp);
        for (int64_t m = 0; m < M; ++m) acc[m * nrows + i] = dot(x + m * ldx, tmp, K);
    }
}

/* Dense BF16-weight accumulators [nvfp4_gemv, bf16_gemv]: W is bf16 [N, K]. */
void orc_bf16_gemv_acc(const uint16_t* x, int64_t ldx, int64_t M, const uint16_t* w, int64_t K,
                       const int64_t* rows, int64_t nrows, double* tmp, double* acc)
{
    for (int64_t i = 0; i < nrows; ++i) {
        for (int64_t k = 0; k < K; ++k) tmp[k] = bf16_to_double(w[rows[i] * K + k]);
        for (int64_t m = 0; m < M; ++m) acc[m * nrows + i] = dot(x + m * ldx, tmp, K);
    }
}

/* ------------------------------------------------------------------------ */
/* Roundings                                                                 */
/* ------------------------------------------------------------------------ */

/* Next bf16 bit pattern in value order (finite, non-NaN). */
static uint16_t bf16_next_up(uint16_t h)
{
    if (h == 0x8000u) return 0x0000u;
    return (h & 0x8000u) ? (uint16_t)(h - 1) : (uint16_t)(h + 1);
}

/* Relative half-width of the window around an intermediate bf16 rounding of
 * a long fp32 dot product (G and U before silu_mul, y_j and y_shared in
 * down_combine).  An fp32-accumulating implementation reaches such a value
 * with a small relative error; when the exact value lies within this
 * distance of a bf16 rounding midpoint, both neighbours are correct roundings
 * of a correct fp32 result. */
#define INTERMEDIATE_REL_WINDOW 0x1p-16

/* Round an intermediate v to bf16: *nom is the rounding of v itself, *alt
 * the other neighbour when a rounding midpoint lies within eps of v (else
 * *alt = *nom).  eps must be well below half a bf16 ulp. */
void orc_round_intermediate(double v, double eps, uint16_t* nom, uint16_t* alt)
{
    uint16_t n = orc_bf16_rne(v), a = orc_bf16_rne(v - eps), b = orc_bf16_rne(v + eps);
    *nom = n;
    *alt = (a != n) ? a : b;
}

/* y = bf16(f32(f32(acc) * s)) as an intermediate: nominal and alternative. */
static void scaled_intermediate(double acc, double s, uint16_t* nom, uint16_t* alt)
{
    double v = f32(f32(acc) * s);
    orc_round_intermediate(v, INTERMEDIATE_REL_WINDOW * fabs(v), nom, alt);
}

/* SiLU evaluated exactly (double): x / (1 + exp(-x)). */
static double silu(double g) { return g / (1.0 + exp(-g)); }

static void hull_add(uint16_t v, uint16_t* lo, uint16_t* hi)
{
    if (bf16_to_double(v) < bf16_to_double(*lo)) *lo = v;
    if (bf16_to_double(v) > bf16_to_double(*hi)) *hi = v;
}

/* out = bf16(silu(G) * U) for G in {gn, ga}, U in {un, ua} (the bf16 outputs
 * of the gate and up rows, each with its alternative rounding): the nominal
 * value from (gn, un) and the hull of all four. */
static void silu_mul_out(uint16_t gn, uint16_t ga, uint16_t un, uint16_t ua, uint16_t* nom, uint16_t* lo,
                         uint16_t* hi)
{
    const uint16_t gs_[2] = {gn, ga}, us_[2] = {un, ua};
    *nom = orc_bf16_rne(silu(bf16_to_double(gn)) * bf16_to_double(un));
    *lo = *hi = *nom;
    for (int i = 0; i < 2; ++i)
        for (int j = 0; j < 2; ++j)
            hull_add(orc_bf16_rne(silu(bf16_to_double(gs_[i])) * bf16_to_double(us_[j])), lo, hi);
}

/* ------------------------------------------------------------------------ */
/* Epilogues                                                                 */
/* ------------------------------------------------------------------------ */

/* Dense epilogue [nvfp4_gemv, module docstring: the fp32 accumulator is
 * multiplied by the fp32 global scale and rounded to bf16 once; nvfp4_gemv,
 * the silu_mul flag]:
 *   silu == 0: out[m, i] = bf16(f32(f32(acc) * gs)), one rounding, no
 *   alternative (lo == hi == nom).
 *   silu != 0: the accumulators hold gate rows in columns [0, half) and the
 *   matching up rows in [half, 2 half); G, U are the bf16 outputs and
 *   out[m, i] = bf16(silu(G) * U) (exact SiLU, rounded once); [lo, hi]
 *   is the hull over the alternative roundings of G and U. */
void orc_dense_epilogue(const double* acc, int64_t M, int64_t ncols, double gs, int silu_mul, uint16_t* nom,
                        uint16_t* lo, uint16_t* hi)
{
    if (!silu_mul) {
        for (int64_t i = 0; i < M * ncols; ++i) nom[i] = lo[i] = hi[i] = orc_bf16_rne(f32(f32(acc[i]) * gs));
        return;
    }
    int64_t half = ncols / 2;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t i = 0; i < half; ++i) {
            uint16_t gn, ga, un, ua;
            scaled_intermediate(acc[m * ncols + i], gs, &gn, &ga);
            scaled_intermediate(acc[m * ncols + half + i], gs, &un, &ua);
            silu_mul_out(gn, ga, un, ua, &nom[m * half + i], &lo[m * half + i], &hi[m * half + i]);
        }
}

/* ------------------------------------------------------------------------ */
/* MoE pair                                                                  */
/* ------------------------------------------------------------------------ */

/* Stored W1 row holding logical row (up ? up : gate) i of an expert in the
 * "[up; gate] in 64-row groups" layout [moe_gemv, module docstring]: stored
 * rows 128 g + [0, 64) are up rows 64 g + [0, 64), stored rows 128 g +
 * [64, 128) the gate rows 64 g + [0, 64). */
int64_t orc_w1_row(int64_t i, int up)
{
    return 128 * (i / 64) + (up ? 0 : 64) + i % 64;
}

/* gate_up [moe_gemv, gate_up], pairs p in [p0, p1) (p = t * topk + j):
 *   e = ids[p]; g, u = f32(acc) * alpha[e] in fp32 (not rounded to bf16);
 *   act[p, i] = bf16(silu(g) * u), one rounding, no alternative (the pages
 *   use an approximate sigmoid; the oracle uses the exact one and the
 *   output tolerance covers the difference).
 * Out-of-range expert ids leave the row untouched and return nonzero. */
int orc_moe_gate_up_routed(const uint16_t* x, const int32_t* ids, int64_t topk, const uint8_t* w1,
                           const uint8_t* w1_sf, const float* alpha, int64_t E, int64_t H, int64_t I,
                           int64_t p0, int64_t p1, double* tmp_g, double* tmp_u, uint16_t* nom,
                           uint16_t* lo, uint16_t* hi)
{
    int bad = 0;
    int64_t sfe = orc_scale_bytes(2 * I, H);
    for (int64_t p = p0; p < p1; ++p) {
        int64_t t = p / topk, e = ids[p];
        if (e < 0 || e >= E) { bad = 1; continue; }
        const uint8_t* we = w1 + e * (2 * I) * (H / 2);
        const uint8_t* se = w1_sf + e * sfe;
        double a = (double)alpha[e];
        for (int64_t i = 0; i < I; ++i) {
            dequant_row(we, se, orc_w1_row(i, 0), H, tmp_g);
            dequant_row(we, se, orc_w1_row(i, 1), H, tmp_u);
            double g = f32(f32(dot(x + t * H, tmp_g, H)) * a);
            double u = f32(f32(dot(x + t * H, tmp_u, H)) * a);
            int64_t o = p * I + i;
            nom[o] = lo[o] = hi[o] = orc_bf16_rne(silu(g) * u);
        }
    }
    return bad;
}

/* Shared expert of gate_up [moe_gemv, gate_up]: ModelOpt [gate; up] weight
 * [2 SI, H/2] with flat 128x4 scales; sact[t, i] = bf16(silu(G) * U) with
 * G, U = bf16(f32(acc) * gssh) (exact SiLU) -- the dense silu_mul epilogue. */
void orc_moe_gate_up_shared(const uint16_t* x, int64_t t0, int64_t t1, const uint8_t* wsh,
                            const uint8_t* ssh, double gssh, int64_t H, int64_t SI, double* tmp_g,
                            double* tmp_u, uint16_t* nom, uint16_t* lo, uint16_t* hi)
{
    for (int64_t t = t0; t < t1; ++t)
        for (int64_t i = 0; i < SI; ++i) {
            uint16_t gn, ga, un, ua;
            dequant_row(wsh, ssh, i, H, tmp_g);
            dequant_row(wsh, ssh, SI + i, H, tmp_u);
            scaled_intermediate(dot(x + t * H, tmp_g, H), gssh, &gn, &ga);
            scaled_intermediate(dot(x + t * H, tmp_u, H), gssh, &un, &ua);
            silu_mul_out(gn, ga, un, ua, &nom[t * SI + i], &lo[t * SI + i], &hi[t * SI + i]);
        }
}

/* down_combine [moe_gemv, module docstring and down_combine], tokens t in
 * [t0, t1):
 *   y_j  = bf16(f32(act[t*topk+j] @ W2[e_j]^T) * alpha2[e_j])
 *   y_sh = bf16(f32(sact[t] @ Wsd^T) * gssd)
 *   s    = bf16(sum_j tw[t, j] * y_j)      (fp32 sum, j = 0 .. topk-1)
 *   out  = bf16(s + y_sh)
 * The nominal output takes every intermediate at its own rounding.  [lo, hi]
 * is the hull of the outputs over the alternatives: y_j and y_sh at their
 * alternative roundings, and every bf16 rounding of an fp32 sum of the
 * chosen tw_j * y_j (topk fused multiply-adds, each within 2^-24 of the
 * running sum).  tw may have any sign.  Tokens with an out-of-range id are
 * skipped; returns nonzero if any. */
int orc_moe_down_combine(const uint16_t* act, const int32_t* ids, const float* tw, int64_t topk,
                         const uint8_t* w2, const uint8_t* w2_sf, const float* alpha2, int64_t E,
                         int64_t H, int64_t I, const uint16_t* sact, const uint8_t* wsd,
                         const uint8_t* ssd, double gssd, int64_t SI, int64_t t0, int64_t t1,
                         double* tmp, uint16_t* nom, uint16_t* lo, uint16_t* hi)
{
    int bad = 0;
    int64_t sfe = orc_scale_bytes(H, I);
    for (int64_t t = t0; t < t1; ++t) {
        int ok = 1;
        for (int64_t j = 0; j < topk; ++j)
            if (ids[t * topk + j] < 0 || ids[t * topk + j] >= E) ok = 0;
        if (!ok) { bad = 1; continue; }
        for (int64_t h = 0; h < H; ++h) {
            double sn = 0.0, slo = 0.0, shi = 0.0, sabs = 0.0;
            for (int64_t j = 0; j < topk; ++j) {
                int64_t e = ids[t * topk + j];
                uint16_t yn, ya;
                dequant_row(w2 + e * H * (I / 2), w2_sf + e * sfe, h, I, tmp);
                scaled_intermediate(dot(act + (t * topk + j) * I, tmp, I), (double)alpha2[e], &yn, &ya);
                double wj = (double)tw[t * topk + j];
                double pn = wj * bf16_to_double(yn); /* exact in double */
                double pa = wj * bf16_to_double(ya);
                sn += pn;
                slo += fmin(pn, pa);
                shi += fmax(pn, pa);
                sabs += fmax(fabs(pn), fabs(pa));
            }
            double es = (double)(topk + 1) * ldexp(1.0, -24) * sabs;
            uint16_t s_n = orc_bf16_rne(sn), s_lo = orc_bf16_rne(slo - es), s_hi = orc_bf16_rne(shi + es);
            uint16_t zn, za;
            dequant_row(wsd, ssd, h, SI, tmp);
            scaled_intermediate(dot(sact + t * SI, tmp, SI), gssd, &zn, &za);
            uint16_t o_n = orc_bf16_rne(bf16_to_double(s_n) + bf16_to_double(zn)), o_lo = o_n, o_hi = o_n;
            int steps = 0;
            for (uint16_t b = s_lo;; b = bf16_next_up(b)) {
                hull_add(orc_bf16_rne(bf16_to_double(b) + bf16_to_double(zn)), &o_lo, &o_hi);
                hull_add(orc_bf16_rne(bf16_to_double(b) + bf16_to_double(za)), &o_lo, &o_hi);
                if (b == s_hi || ++steps > 64) break;
            }
            nom[t * H + h] = o_n;
            lo[t * H + h] = o_lo;
            hi[t * H + h] = o_hi;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Activation quantisation (the W4A4 path)                                   */
/* ------------------------------------------------------------------------ */

/* The flashinfer page's W4A4 kernels (FlashInferB12xNvFp4LinearKernel and
 * the other NvFp4LinearKernel backends, apply_weights) quantise x with
 * scaled_fp4_quant(x, input_global_scale_inv) into an NVFP4 tensor of the
 * weight's own format (E2M1 codes, 128x4-swizzled E4M3 block scales, one per
 * 16 values) and hand both NVFP4 tensors and alpha to the NVFP4 GEMM.  The
 * pages do not print the quantiser's arithmetic.  Reading (the plainest one
 * the rest supports): e2m1 x e4m3 approximates x * gsi, so that
 * out = bf16(fp32(sum_k xq_k * wq_k) * alpha) with alpha = the product of
 * the activation's (1 / gsi) and the weight's global scales.  Per row m and
 * block b of 16 values, in float (binary32), each operation rounded to
 * nearest even, no fused multiply-add:
 *   amax = max |x[m, 16b .. 16b + 15]|
 *   s    = (amax / 6) * gsi
 *   sf   = orc_e4m3_encode(s)
 *   r    = gsi / e4m3(sf)             (sf = 0: every code of the block is 0)
 *   code = orc_e2m1_encode(x * r)
 * gsi must be positive and finite, x finite. */

/* The finite E4M3 code nearest v >= 0 (ties to the even code), saturating at
 * 448 (code 0x7E): a plain search over the 127 non-negative finite codes. */
int orc_e4m3_encode(float v)
{
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs((double)v - orc_e4m3(c));
        if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) != 0)) {
            best = c;
            bd = d;
        }
    }
    return best;
}

/* The E2M1 code nearest v (ties to the even magnitude code), saturating at
 * magnitude 6; the sign bit is set for v < 0 unless the magnitude code is 0
 * (a value that rounds to zero is stored as +0). */
int orc_e2m1_encode(float v)
{
    double a = fabs((double)v);
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c < 8; ++c) {
        double d = fabs(a - E2M1_MAG[c]);
        if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) != 0)) {
            best = c;
            bd = d;
        }
    }
    if (a > 6.0) best = 7;
    return (v < 0.0f && best != 0) ? (best | 8) : best;
}

/* scaled_fp4_quant as read above: x bf16 [M, K] (row stride ldx), K % 16 ==
 * 0; writes q [M, K / 2] (element 2j in the low nibble of byte j, as the
 * weights) and sf, orc_scale_bytes(M, K) bytes in the 128x4 layout (bytes of
 * padding rows and blocks are 0). */
void orc_quantize_act(const uint16_t* x, int64_t ldx, int64_t M, int64_t K, float gsi, uint8_t* q, uint8_t* sf)
{
    memset(sf, 0, (size_t)orc_scale_bytes(M, K));
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t b = 0; b < K / 16; ++b) {
            const uint16_t* xb = x + m * ldx + 16 * b;
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = (float)fabs(bf16_to_double(xb[i]));
                if (a > amax) amax = a;
            }
            float s = (amax / 6.0f) * gsi;
            int sc = orc_e4m3_encode(s);
            sf[orc_swz(m, b, K)] = (uint8_t)sc;
            float e = (float)orc_e4m3(sc);
            float r = e > 0.0f ? gsi / e : 0.0f;
            for (int i = 0; i < 16; i += 2) {
                float v0 = (float)bf16_to_double(xb[i]) * r;
                float v1 = (float)bf16_to_double(xb[i + 1]) * r;
                int c0 = e > 0.0f ? orc_e2m1_encode(v0) : 0;
                int c1 = e > 0.0f ? orc_e2m1_encode(v1) : 0;
                q[m * (K / 2) + 8 * b + i / 2] = (uint8_t)(c0 | (c1 << 4));
            }
        }
    }
}
