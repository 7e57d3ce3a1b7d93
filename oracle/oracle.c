/*
 * CPU oracle for the TMA-fed bf16 GEMM and the TMA tile-copy path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header or table with the CUDA library: it is a plain,
 * slow restatement of what the path computes, written so that a reader can check it
 * against the pages line by line.
 *
 * Sources (page title, section):
 *  - "GEMM: la moltiplicazione di matrici sull'hardware", section "Il conto, e il
 *    problema della versione ingenua": C_ij = sum_k A_ik B_kj, 2MNK flops; section
 *    "I tensor core": the BLAS form C <- alpha*A*B + beta*C with 16-bit inputs and a
 *    32-bit accumulator.
 *  - "H100 . cuTensorMap (TMA descriptor)", section 11.3 (swizzle formula
 *    a' = a ^ ((a & Y_mask) >> 3) and the three bit maps), section 11.4 (16-byte
 *    units inside 128-byte shared-memory rows), section 14 (OOB fill happens in
 *    shared memory, the source is untouched, zero or NaN).
 *  - "2 . Le Tensor Memory Accelerator", section 2.5 "Remplissage des bords"
 *    (out-of-bounds parts of a tile are filled with zeros).
 *
 * Precision: every product and sum is formed in IEEE double.  A bf16 value has an
 * 8-bit significand, so each product of two bf16 values is exact in double, and the
 * double sum of K such products carries a relative error of at most K*2^-53 of the
 * absolute-value sum -- far below the bf16/fp32 tolerances the tests apply.
 *
 * Readings taken where the pages are silent, each stated in full below:
 *  - Y_mask = ((1<<b)-1) << 7 with b = 1, 2, 3 for the 32B, 64B, 128B modes.  The
 *    page prints Y_mask = 1<<7, which only yields the 32B map; the generalised mask
 *    reproduces all three printed bit maps.
 *  - The swizzled address a is the byte offset of an element inside the box image,
 *    counted from a 1024-byte-aligned base.
 *  - The box is packed densely: row pitch = inner box extent in bytes.  With a swizzle
 *    this reading is applied only where the inner extent equals the swizzle span (the
 *    benchmark's boxes); on the hardware a narrower swizzled row is placed at the span's
 *    pitch, so the library does not offer that case and the oracle is not used for it.
 *  - Boxes appear in the output image in row-major order of the box grid (outer box
 *    index slowest).
 *  - OOB "fill none" means zero; the NaN fill's exact bit pattern is not stated on the
 *    pages ("parity unpinned" for that pattern): this model writes all-ones bytes,
 *    which is a NaN in every floating-point format, and tests only check isnan.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------------
 * Element decoding.  A bf16 value is the upper half of an IEEE binary32 value.
 * ------------------------------------------------------------------------------- */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent 0
 * encodes zero and subnormals (fraction * 2^-24), exponent 31 infinities and NaNs. */
static double f16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1F, f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* 8-bit floats.  E4M3 (the "fn" variant): 1 sign, 4 exponent bits (bias 7), 3 fraction
 * bits, no infinities, S.1111.111 is NaN, largest finite 448.  E5M2: 1 sign, 5 exponent
 * bits (bias 15), 2 fraction bits, IEEE-style infinities and NaNs. */
static double e4m3_bits_to_double(uint8_t h)
{
    int sign = (h >> 7) & 1, e = (h >> 3) & 0xF, f = h & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9);
    else
        v = ldexp((double)(8 + f), e - 10);
    return sign ? -v : v;
}

static double e5m2_bits_to_double(uint8_t h)
{
    int sign = (h >> 7) & 1, e = (h >> 2) & 0x1F, f = h & 0x3;
    double v;
    if (e == 31)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -16);
    else
        v = ldexp((double)(4 + f), e - 17);
    return sign ? -v : v;
}

/* tf32 as the GEMM page defines it in its tensor-core section: a binary32 input with
 * its mantissa truncated to 10 bits, i.e. the 13 low mantissa bits cleared (a NaN whose
 * payload lies only in those bits would become an infinity; no input here has one). */
static double tf32_bits_to_double(uint32_t w)
{
    uint32_t t = w & 0xFFFFE000u;
    float f;
    memcpy(&f, &t, sizeof f);
    return (double)f;
}

/* Element t of an operand array of type `kind`: 0 = bf16, 1 = fp16 (16-bit patterns),
 * 2 = E4M3, 3 = E5M2 (8-bit patterns), 4 = tf32 (binary32 patterns, truncated). */
static double operand(const void *X, int64_t t, int kind)
{
    switch (kind) {
    case 4: return tf32_bits_to_double(((const uint32_t *)X)[t]);
    case 1: return f16_bits_to_double(((const uint16_t *)X)[t]);
    case 2: return e4m3_bits_to_double(((const uint8_t *)X)[t]);
    case 3: return e5m2_bits_to_double(((const uint8_t *)X)[t]);
    default: return bf16_bits_to_double(((const uint16_t *)X)[t]);
    }
}

/* Exposed for the decoders' pins (every pattern against a library conversion). */
double oracle_f8_to_double(uint8_t h, int e5m2)
{
    return e5m2 ? e5m2_bits_to_double(h) : e4m3_bits_to_double(h);
}

static double f32_bits_to_double(uint32_t w)
{
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* C0 element (row i, column j) of a row-major matrix with leading dimension ldc;
 * c_dtype 0 = fp32, 1 = bf16, 2 = fp16. */
static double load_c0(const void *C0, int c_dtype, int64_t ldc, int64_t i, int64_t j)
{
    if (c_dtype == 1)
        return bf16_bits_to_double(((const uint16_t *)C0)[i * ldc + j]);
    if (c_dtype == 2)
        return f16_bits_to_double(((const uint16_t *)C0)[i * ldc + j]);
    return f32_bits_to_double(((const uint32_t *)C0)[i * ldc + j]);
}

/* Exposed for the decoder's pin (all 65536 patterns against a library conversion). */
double oracle_f16_to_double(uint16_t h) { return f16_bits_to_double(h); }

/* Exposed for the truncation's pins. */
double oracle_tf32_to_double(uint32_t w) { return tf32_bits_to_double(w); }

/* Operand storage.  `layout` bit 0: A is stored M-major (element (i,k) at A[k*lda + i])
 * instead of K-major (A[i*lda + k]); bit 1: the K x N operand B is stored N-major
 * (element (k,j) at B[k*ldb + j]) instead of K-major (B[j*ldb + k]).  Only the index
 * arithmetic differs; the sum is the same.  Bits 4-6: the operands' element type, 0 =
 * bf16, 1 = fp16 (the GEMM page's tensor-core section: 16-bit inputs, float16 or
 * bfloat16), 2 = E4M3, 3 = E5M2 (the FP8 the same page names among the shorter
 * formats), 4 = tf32 (its third path: float32 inputs truncated to 10 mantissa bits). */
static int64_t a_index(int layout, int64_t lda, int64_t i, int64_t k)
{
    return (layout & 1) ? k * lda + i : i * lda + k;
}

static int64_t b_index(int layout, int64_t ldb, int64_t j, int64_t k)
{
    return (layout & 2) ? k * ldb + j : j * ldb + k;
}

/* One output element of C = alpha * A * B + beta * C0, C_ij = sum_k A_ik * B_kj.
 * When beta == 0, C0 is not read at all (BLAS convention: NaNs in C do not leak).
 * *absprod receives sum_k |A_ik| * |B_kj|, the scale of the accumulation error. */
static double gemm_entry(int64_t K, const void *A, int64_t lda, const void *B,
                         int64_t ldb, int layout, const void *C0, int c_dtype, int64_t ldc,
                         double alpha, double beta, int64_t i, int64_t j,
                         double *absprod)
{
    const int kind = (layout >> 4) & 7;
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double a = operand(A, a_index(layout, lda, i, k), kind);
        double b = operand(B, b_index(layout, ldb, j, k), kind);
        acc += a * b;
        mag += fabs(a) * fabs(b);
    }
    double c = alpha * acc;
    if (beta != 0.0)
        c += beta * load_c0(C0, c_dtype, ldc, i, j);
    if (absprod)
        *absprod = mag;
    return c;
}

/* Rows [row0, row1) of C, written densely to out[(i-row0)*N + j] (and absprod, if
 * non-NULL, with the same indexing).  Plain i-j-k loops; rows run in parallel. */
void oracle_gemm_rows(int64_t M, int64_t N, int64_t K,
                      const void *A, int64_t lda,
                      const void *B, int64_t ldb, int layout,
                      const void *C0, int c_dtype, int64_t ldc,
                      double alpha, double beta,
                      int64_t row0, int64_t row1,
                      double *out, double *absprod)
{
    if (row0 < 0)
        row0 = 0;
    if (row1 > M)
        row1 = M;
    int64_t i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = row0; i < row1; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double mag;
            double c = gemm_entry(K, A, lda, B, ldb, layout, C0, c_dtype, ldc, alpha, beta,
                                  i, j, &mag);
            out[(i - row0) * N + j] = c;
            if (absprod)
                absprod[(i - row0) * N + j] = mag;
        }
    }
}

/* The same definition evaluated at n sampled positions (ii[t], jj[t]). */
void oracle_gemm_entries(int64_t K,
                         const void *A, int64_t lda,
                         const void *B, int64_t ldb, int layout,
                         const void *C0, int c_dtype, int64_t ldc,
                         double alpha, double beta,
                         int64_t n, const int64_t *ii, const int64_t *jj,
                         double *out, double *absprod)
{
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < n; ++t) {
        double mag;
        out[t] = gemm_entry(K, A, lda, B, ldb, layout, C0, c_dtype, ldc, alpha, beta,
                            ii[t], jj[t], &mag);
        if (absprod)
            absprod[t] = mag;
    }
}

/* ---------------------------------------------------------------------------------
 * MX (microscaling) operands, as the OCP Microscaling Formats (MX) specification v1.0
 * defines them: a block is 32 consecutive elements along K of one element type (here
 * FP8 E4M3 or E5M2) sharing one scale X of type E8M0, an 8-bit biased exponent with no
 * sign and no mantissa: X encodes 2^(X - 127), and X = 255 encodes NaN.  The value of an
 * element is its own value times its block's scale.  The product of two MX operands is
 * then the ordinary matrix product of those values; here it is summed in IEEE double.
 *
 * Scale storage (the library's layout, restated here on its own): the scales of an
 * operand with `rows` rows (M for A, N for B) come in 512-byte atoms, one per (group of
 * 128 rows, group of four 32-element blocks, i.e. 128 elements of K).  The byte of row r
 * and block j lies at
 *     ((j / 4) * RB + r / 128) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4),
 * RB = ceil(rows / 128): atoms of one 128-element slice of K follow each other in row
 * order, and inside an atom row r sits in the 16-byte line r % 32, at the 4-byte group of
 * its 32-row quarter, one byte per block.
 * ------------------------------------------------------------------------------- */
static double e8m0_to_double(uint8_t x)
{
    return x == 255 ? NAN : ldexp(1.0, (int)x - 127);
}

/* Exposed for the decoder's pins. */
double oracle_e8m0_to_double(uint8_t x) { return e8m0_to_double(x); }

int64_t oracle_mx_scale_offset(int64_t rows, int64_t r, int64_t j)
{
    const int64_t rb = (rows + 127) / 128;
    return ((j / 4) * rb + r / 128) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4);
}

/* One output element of C = alpha * A * B + beta * C0 with MX operands: A (M x K) and B
 * (stored N x K) K-major with leading dimensions lda, ldb; SA and SB their scales;
 * kind 2 = E4M3 elements, 3 = E5M2.  *absprod receives sum_k |a_ik| |b_jk| of the scaled
 * values. */
static double gemm_mx_entry(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda,
                            const uint8_t *SA, const uint8_t *B, int64_t ldb,
                            const uint8_t *SB, int kind, const void *C0, int c_dtype,
                            int64_t ldc, double alpha, double beta, int64_t i, int64_t j,
                            double *absprod)
{
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double sa = e8m0_to_double(SA[oracle_mx_scale_offset(M, i, k / 32)]);
        const double sb = e8m0_to_double(SB[oracle_mx_scale_offset(N, j, k / 32)]);
        const double a = operand(A, i * lda + k, kind) * sa;
        const double b = operand(B, j * ldb + k, kind) * sb;
        acc += a * b;
        mag += fabs(a) * fabs(b);
    }
    double c = alpha * acc;
    if (beta != 0.0)
        c += beta * load_c0(C0, c_dtype, ldc, i, j);
    if (absprod)
        *absprod = mag;
    return c;
}

void oracle_gemm_mx_entries(int64_t M, int64_t N, int64_t K, const uint8_t *A, int64_t lda,
                            const uint8_t *SA, const uint8_t *B, int64_t ldb,
                            const uint8_t *SB, int kind, const void *C0, int c_dtype,
                            int64_t ldc, double alpha, double beta, int64_t n,
                            const int64_t *ii, const int64_t *jj, double *out,
                            double *absprod)
{
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < n; ++t) {
        double mag;
        out[t] = gemm_mx_entry(M, N, K, A, lda, SA, B, ldb, SB, kind, C0, c_dtype, ldc, alpha,
                               beta, ii[t], jj[t], &mag);
        if (absprod)
            absprod[t] = mag;
    }
}

/* ---------------------------------------------------------------------------------
 * Swizzle: a' = a ^ ((a & Y_mask) >> 3).
 * mode 0 = none (identity), 1 = 32B, 2 = 64B, 3 = 128B; b = mode bits of the shared
 * memory row index (address bits 7 and up) are XORed into the 16-byte unit index
 * (address bits 4 and up).  Bits [3:0] are never touched.
 * ------------------------------------------------------------------------------- */
uint64_t oracle_swizzle(uint64_t a, int mode)
{
    if (mode <= 0)
        return a;
    uint64_t y_mask = ((1ull << mode) - 1ull) << 7;
    return a ^ ((a & y_mask) >> 3);
}

int oracle_omp_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------------
 * TMA box extraction model.
 *
 * The tensor T is 2-D: H rows (outer dimension) of W elements (inner dimension),
 * element size es bytes, row stride `stride` bytes.  A box is box_h rows by box_w
 * elements; the box grid has nbi = ceil(H/box_h) rows and nbj = ceil(W/box_w)
 * columns.  For box (bi, bj) with box_index = bi*nbj + bj:
 *   1. the logical dense box L: row r, element c holds T[bi*box_h + r][bj*box_w + c]
 *      when that position lies inside the tensor, otherwise the fill value;
 *   2. logical byte a = r*(box_w*es) + c*es + byte lands at image byte swizzle(a);
 *   3. the box image occupies out[box_index*box_bytes, +box_bytes), with
 *      box_bytes = box_h*box_w*es.
 * Boxes [box_begin, box_end) are produced; `out` points at the image of box_begin.
 * oob_nan = 0 -> zero fill, 1 -> NaN fill (all-ones bytes, see the header).
 * ------------------------------------------------------------------------------- */
void oracle_tma_box_images(const uint8_t *T, int64_t H, int64_t W, int64_t stride,
                           int es, int64_t box_w, int64_t box_h, int mode,
                           int oob_nan, int64_t box_begin, int64_t box_end,
                           uint8_t *out)
{
    int64_t nbj = (W + box_w - 1) / box_w;
    int64_t row_bytes = box_w * es;
    int64_t box_bytes = box_h * row_bytes;
    uint8_t fill = oob_nan ? 0xFF : 0x00;
    int64_t bx;
#pragma omp parallel for schedule(static)
    for (bx = box_begin; bx < box_end; ++bx) {
        int64_t bi = bx / nbj, bj = bx % nbj;
        uint8_t *img = out + (bx - box_begin) * box_bytes;
        for (int64_t r = 0; r < box_h; ++r) {
            int64_t row = bi * box_h + r;
            for (int64_t c = 0; c < box_w; ++c) {
                int64_t col = bj * box_w + c;
                int inside = (row < H) && (col < W);
                for (int byte = 0; byte < es; ++byte) {
                    uint64_t a = (uint64_t)(r * row_bytes + c * es + byte);
                    uint8_t v = inside ? T[row * stride + col * es + byte] : fill;
                    img[oracle_swizzle(a, mode)] = v;
                }
            }
        }
    }
}

/* ---------------------------------------------------------------------------------
 * Rank 1..5 box extraction with element strides ("H100 . cuTensorMap (TMA descriptor)",
 * sections 8-9: up to 5 dimensions, innermost first, byte strides for the outer ones,
 * boxDim per dimension, elementStrides = traversal step per dimension).
 *
 * Dimension i has dims[i] elements, consecutive indices `stride[i]` bytes apart
 * (stride[0] = es).  A box has traversal extent ext[i] and step estr[i]; it holds
 * L_i = ceil(ext[i] / estr[i]) elements along dimension i, element j_i taken from index
 * origin_i + j_i * estr[i] with origin_i = b_i * ext[i] (box grid index b_i, nb_i =
 * ceil(dims[i] / ext[i]) boxes).  Readings taken: the box lands densely in shared
 * memory, dimension 0 fastest (row pitch L_0 * es bytes), the same byte-address swizzle
 * applies, indices beyond dims[i] read the fill value, and boxes appear in the image
 * row-major over the box grid (dimension 0 fastest, the outermost slowest), as the
 * 2-D model above.
 * ------------------------------------------------------------------------------- */
/* Region form: the box grid along dimension i starts at index origin[i] (which may be
 * negative) and has nb[i] boxes, box b_i covering indices origin[i] + b_i * ext[i] ..
 * + ext[i] - 1.  Reading taken where the pages are silent: an index below 0 is out of
 * bounds exactly like one at or past dims[i] (the TMA page's edge fill and the
 * cuTensorMap page's section 14 only speak of a tile passing the tensor's edge); such
 * elements read the fill value. */
void oracle_tma_box_images_region(const uint8_t *T, int rank, const int64_t *dims,
                                  const int64_t *stride, int es, const int64_t *ext,
                                  const int64_t *estr, const int64_t *origin,
                                  const int64_t *nb, int mode, int oob_nan,
                                  int64_t box_begin, int64_t box_end, uint8_t *out)
{
    int64_t L[5];
    int64_t box_elems = 1;
    for (int i = 0; i < rank; ++i) {
        L[i] = (ext[i] + estr[i] - 1) / estr[i];
        box_elems *= L[i];
    }
    const int64_t box_bytes = box_elems * es;
    const uint8_t fill = oob_nan ? 0xFF : 0x00;
    int64_t bx;
#pragma omp parallel for schedule(static)
    for (bx = box_begin; bx < box_end; ++bx) {
        int64_t b[5], q = bx;
        for (int i = 0; i < rank; ++i) {  /* dimension 0 fastest */
            b[i] = q % nb[i];
            q /= nb[i];
        }
        uint8_t *img = out + (bx - box_begin) * box_bytes;
        for (int64_t e = 0; e < box_elems; ++e) {
            int64_t r = e, offset = 0;
            int inside = 1;
            for (int i = 0; i < rank; ++i) {
                const int64_t j = r % L[i];
                r /= L[i];
                const int64_t idx = origin[i] + b[i] * ext[i] + j * estr[i];
                if (idx < 0 || idx >= dims[i])
                    inside = 0;
                else
                    offset += idx * stride[i];
            }
            for (int byte = 0; byte < es; ++byte) {
                const uint64_t a = (uint64_t)(e * es + byte);
                img[oracle_swizzle(a, mode)] = inside ? T[offset + byte] : fill;
            }
        }
    }
}

/* The whole tensor: origin 0 and nb_i = ceil(dims[i] / ext[i]) boxes per dimension. */
void oracle_tma_box_images_nd(const uint8_t *T, int rank, const int64_t *dims,
                              const int64_t *stride, int es, const int64_t *ext,
                              const int64_t *estr, int mode, int oob_nan,
                              int64_t box_begin, int64_t box_end, uint8_t *out)
{
    int64_t origin[5] = {0, 0, 0, 0, 0}, nb[5] = {1, 1, 1, 1, 1};
    for (int i = 0; i < rank; ++i)
        nb[i] = (dims[i] + ext[i] - 1) / ext[i];
    oracle_tma_box_images_region(T, rank, dims, stride, es, ext, estr, origin, nb, mode,
                                 oob_nan, box_begin, box_end, out);
}
