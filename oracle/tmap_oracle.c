/*
 * tmap_oracle.c -- plain, slow CPU oracle for descriptor-driven tiled tensor movement.
 *
 * TEST INFRASTRUCTURE ONLY: see tmap_oracle.h for who may use it, the page tags and the pin status
 * of every function (the 64-byte and 32-byte swizzle layouts, which the pages do not define, are
 * pinned by NVIDIA's published chunk patterns for those modes).
 *
 * Everything here walks one element (or one byte) at a time in the order the definitions state.
 * There is no blocking, vectorisation or reordering, so that each function can be checked against
 * the pages by eye.  Build with -ffp-contract=off and without -ffast-math: the one floating-point
 * operation of the path, the fp32 reduce-add, must be a single IEEE binary32 add rounded to nearest.
 */
#include "tmap_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------------------------------
 * Swizzle.  [MLSys-TMA] §"TMA 如何写入 swizzled layout": in a 128-byte swizzled image each row holds
 * eight 16-byte sectors and logical sector c of row r lands in physical sector c XOR r.
 * §"用 3D TMA 搬运多个 swizzle atoms": the permutation is confined to an atom of 8 rows x 128 bytes,
 * physical_sector = logical_sector XOR (row % 8), with `row` counted inside the image.
 *
 * Written on the byte offset `off` of an image with 128-byte rows: the sector is bits 4..6 of off
 * and the row's position inside its 8-row atom is bits 7..9, so the rule XORs bits 7..9 into bits
 * 4..6.  For the 64-byte and 32-byte modes, which the pages name but do not define, this library
 * reads the same rule with two and one XOR bits (bits 7..8 into 4..5, bit 7 into 4): an atom of
 * 8 x 64 bytes resp. 8 x 32 bytes whose 16-byte chunks are permuted by the row bits above the 128-byte
 * line.  That reading is the chunk pattern NVIDIA's public CUDA documentation draws for the two
 * modes (repeating after 512 and 256 bytes), against which the tests check it.
 * ------------------------------------------------------------------------------------------- */
uint64_t orc_swz(uint64_t off, uint32_t span)
{
    uint64_t xor_bits;
    if (span == 128) {
        xor_bits = 3;
    } else if (span == 64) {
        xor_bits = 2;
    } else if (span == 32) {
        xor_bits = 1;
    } else {
        return off; /* no swizzle */
    }
    uint64_t line = (off >> 7) & ((1u << xor_bits) - 1u); /* row inside the atom (its low bits) */
    return off ^ (line << 4);
}

int orc_map_check(const orc_map* m)
{
    if (m->rank < 1 || m->rank > 5) return 1;
    if (m->esize != 1 && m->esize != 2 && m->esize != 4 && m->esize != 8) return 2;
    for (uint32_t i = 0; i < m->rank; i++) {
        if (m->box[i] < 1) return 3;
        if (m->estride[i] < 1 || m->estride[i] > 8) return 6;
    }
    if (m->span != 0 && m->span != 32 && m->span != 64 && m->span != 128) return 4;
    /* [MLSys-TMA] §"用 3D TMA 搬运多个 swizzle atoms": the inner box row may not exceed the atom
     * width; §"128-byte swizzle 的分组要求": an N-byte atom needs a row of at least N bytes.
     * Together: with a swizzle the inner box row is exactly `span` bytes, and (so that the image
     * row is that row) the innermost element stride is 1. */
    if (m->span != 0 && ((uint64_t)m->box[0] * m->esize != m->span || m->estride[0] != 1)) return 5;
    if (m->fill > ORC_FILL_NAN_F64) return 7;
    if ((m->fill == ORC_FILL_NAN_F16 || m->fill == ORC_FILL_NAN_BF16) && m->esize != 2) return 7;
    if (m->fill == ORC_FILL_NAN_F32 && m->esize != 4) return 7;
    if (m->fill == ORC_FILL_NAN_F64 && m->esize != 8) return 7;
    return 0;
}

/* [Book-TMA] §"Tensor descriptor：CUtensorMap": elementStrides is the step, in elements, between
 * the elements taken along each dim when the box is written to shared memory.  Read here as: of
 * the box's box[i] elements along dim i, every estride[i]-th one starting at the box's first is
 * taken, so the image holds ceil(box[i] / estride[i]) of them, packed. */
uint32_t orc_extent(const orc_map* m, uint32_t i)
{
    return i < m->rank ? (m->box[i] + m->estride[i] - 1) / m->estride[i] : 1u;
}

static int64_t step_of(const orc_map* m, uint32_t i) { return i < m->rank ? m->estride[i] : 1; }

uint64_t orc_box_bytes(const orc_map* m)
{
    uint64_t n = m->esize;
    for (uint32_t i = 0; i < m->rank; i++) n *= orc_extent(m, i);
    return n;
}

/* Number of boxes along dim i: the smallest count whose boxes cover the whole dimension. */
static uint64_t boxes_along(const orc_map* m, uint32_t i)
{
    return (m->dim[i] + m->box[i] - 1) / m->box[i];
}

uint64_t orc_num_boxes(const orc_map* m)
{
    uint64_t n = 1;
    for (uint32_t i = 0; i < m->rank; i++) n *= boxes_along(m, i);
    return n;
}

void orc_box_start(const orc_map* m, uint64_t b, int32_t* s)
{
    for (uint32_t i = 0; i < m->rank; i++) {
        uint64_t nb = boxes_along(m, i);
        s[i] = (int32_t)((b % nb) * m->box[i]);
        b /= nb;
    }
}

/* Element at global coordinate g: in bounds iff 0 <= g[i] < dim[i] for every dim
 * ([H200-TMA] §02, the out-of-bounds row of the table: the hardware fills such elements). */
static int in_bounds(const orc_map* m, const int64_t* g)
{
    for (uint32_t i = 0; i < m->rank; i++) {
        if (g[i] < 0 || (uint64_t)g[i] >= m->dim[i]) return 0;
    }
    return 1;
}

static uint8_t* element_address(const orc_map* m, const int64_t* g)
{
    int64_t off = 0;
    for (uint32_t i = 0; i < m->rank; i++) off += g[i] * m->stride[i];
    return m->base + off;
}

/* Visits every element of the image of the box starting at s, dim 0 fastest.  For each, `g` is
 * the global coordinate it comes from and `lin` its element index inside the (unswizzled) image. */
typedef void (*element_fn)(const orc_map* m, const int64_t* g, uint64_t lin, void* ctx);

static void for_each_element(const orc_map* m, const int32_t* s, element_fn fn, void* ctx)
{
    int64_t g[5] = {0, 0, 0, 0, 0};
    uint64_t lin = 0;
    for (uint32_t e4 = 0; e4 < orc_extent(m, 4); e4++)
    for (uint32_t e3 = 0; e3 < orc_extent(m, 3); e3++)
    for (uint32_t e2 = 0; e2 < orc_extent(m, 2); e2++)
    for (uint32_t e1 = 0; e1 < orc_extent(m, 1); e1++)
    for (uint32_t e0 = 0; e0 < orc_extent(m, 0); e0++) {
        uint32_t e[5] = {e0, e1, e2, e3, e4};
        for (uint32_t i = 0; i < 5; i++)
            g[i] = (i < m->rank ? (int64_t)s[i] : 0) + (int64_t)e[i] * step_of(m, i);
        fn(m, g, lin, ctx);
        lin++;
    }
}

/* Byte k (little-endian) of the fill element. */
static uint8_t fill_byte(const orc_map* m, uint32_t k)
{
    uint64_t v;
    switch (m->fill) {
        case ORC_FILL_NAN_F16: v = 0x7E00u; break;
        case ORC_FILL_NAN_BF16: v = 0x7FC0u; break;
        case ORC_FILL_NAN_F32: v = 0x7FC00000u; break;
        case ORC_FILL_NAN_F64: v = 0x7FF8000000000000ull; break;
        default: v = 0; break;
    }
    return (uint8_t)(v >> (8 * k));
}

static void image_one(const orc_map* m, const int64_t* g, uint64_t lin, void* ctx)
{
    uint8_t* img = (uint8_t*)ctx;
    int inb = in_bounds(m, g);
    const uint8_t* src = inb ? element_address(m, g) : 0;
    for (uint32_t k = 0; k < m->esize; k++) {
        img[orc_swz(lin * m->esize + k, m->span)] = inb ? src[k] : fill_byte(m, k);
    }
}

void orc_image(const orc_map* m, const int32_t* s, uint8_t* img)
{
    for_each_element(m, s, image_one, img);
}

static void store_one(const orc_map* m, const int64_t* g, uint64_t lin, void* ctx)
{
    const uint8_t* img = (const uint8_t*)ctx;
    if (!in_bounds(m, g)) return;
    uint8_t* dst = element_address(m, g);
    for (uint32_t k = 0; k < m->esize; k++) dst[k] = img[orc_swz(lin * m->esize + k, m->span)];
}

void orc_store(const orc_map* m, const int32_t* s, const uint8_t* img)
{
    for_each_element(m, s, store_one, (void*)img);
}

/* [Book-TMA] §"TMA reduce，把“搬运”和“归约”合并": the write-back combines each element with the value
 * already in global memory.  For fp32 add that is one binary32 addition per element. */
static void reduce_one(const orc_map* m, const int64_t* g, uint64_t lin, void* ctx)
{
    const uint8_t* img = (const uint8_t*)ctx;
    if (!in_bounds(m, g)) return;
    uint8_t* dst = element_address(m, g);
    uint8_t add_bytes[4];
    for (uint32_t k = 0; k < 4; k++) add_bytes[k] = img[orc_swz(lin * 4 + k, m->span)];
    float d, a;
    memcpy(&d, dst, 4);
    memcpy(&a, add_bytes, 4);
    d = d + a;
    memcpy(dst, &d, 4);
}

void orc_reduce_add_f32(const orc_map* dst, const int32_t* s, const uint8_t* img)
{
    for_each_element(dst, s, reduce_one, (void*)img);
}

static void start_of(const orc_map* m, const int32_t* coords, uint64_t b, int32_t* s)
{
    if (coords) {
        for (uint32_t i = 0; i < m->rank; i++) s[i] = coords[b * m->rank + i];
    } else {
        orc_box_start(m, b, s);
    }
}

void orc_tiled_copy(const orc_map* m, const int32_t* coords, uint64_t b0, uint64_t b1,
                    uint8_t* images)
{
    uint64_t bb = orc_box_bytes(m);
    for (uint64_t b = b0; b < b1; b++) {
        int32_t s[5];
        start_of(m, coords, b, s);
        orc_image(m, s, images + b * bb);
    }
}

void orc_tiled_roundtrip(const orc_map* m, const int32_t* coords, uint64_t b0, uint64_t b1,
                         const uint8_t* images)
{
    uint64_t bb = orc_box_bytes(m);
    for (uint64_t b = b0; b < b1; b++) {
        int32_t s[5];
        start_of(m, coords, b, s);
        orc_store(m, s, images + b * bb);
    }
}

/* The reduce path: load the source box into its (swizzled) image, then reduce the image into the
 * destination through a map with the same box and swizzle. */
void orc_tile_reduce_add(const orc_map* dst, const orc_map* src, uint64_t b0, uint64_t b1)
{
    uint8_t* img = (uint8_t*)malloc(orc_box_bytes(src));
    if (!img) return;
    for (uint64_t b = b0; b < b1; b++) {
        int32_t s[5];
        orc_box_start(dst, b, s);
        orc_image(src, s, img);
        orc_reduce_add_f32(dst, s, img);
    }
    free(img);
}

/* ---------------------------------------------------------------------------------------------
 * General reduce: add / min / max over f32, f16, bf16, u32, s32.
 * ------------------------------------------------------------------------------------------- */
double orc_f16_to_double(uint16_t h)
{
    const double sign = (h & 0x8000u) ? -1.0 : 1.0;
    const unsigned e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
    if (e == 0) return sign * ldexp((double)m, -24);              /* zero or subnormal */
    if (e == 31) return m ? NAN : sign * INFINITY;
    return sign * ldexp((double)(1024u + m), (int)e - 25);
}

/* The value v rounded to nearest, ties to even, in a binary format with `mbits` stored
 * significand bits and `ebits` exponent bits (bias 2^(ebits-1) - 1, subnormals, overflow to
 * infinity); returns the bits.  An infinite v stays infinite; a NaN v gives the format's quiet NaN
 * with an empty payload (IEEE 754 leaves the payload of an operation's NaN open). */
static uint32_t round_to_format(double v, int mbits, int ebits)
{
    const int emax = (1 << (ebits - 1)) - 1, emin = 1 - emax;
    const uint32_t all_ones = ((1u << ebits) - 1u) << mbits;
    if (isnan(v)) return all_ones | (1u << (mbits - 1));
    const uint32_t sign_bit = (signbit(v) ? 1u : 0u) << (mbits + ebits);
    v = fabs(v);
    if (isinf(v)) return sign_bit | all_ones;
    if (v == 0.0) return sign_bit;
    int e2;
    frexp(v, &e2);
    int E = e2 - 1;                              /* v in [2^E, 2^(E+1)) */
    if (E < emin) E = emin;                      /* subnormal range: fixed quantum */
    const double q = ldexp(1.0, E - mbits);      /* one unit in the last place at E */
    double n = nearbyint(v / q);                 /* exact scaling, then round half to even */
    const double one = ldexp(1.0, mbits);
    if (n >= 2.0 * one) {                        /* rounded up into the next binade */
        n /= 2.0;
        E += 1;
    }
    if (E > emax) return sign_bit | (((1u << ebits) - 1u) << mbits);   /* infinity */
    if (n < one) return sign_bit | (uint32_t)n;                        /* subnormal */
    return sign_bit | ((uint32_t)(E + emax) << mbits) | (uint32_t)(n - one);
}

uint16_t orc_f16_from_double(double v) { return (uint16_t)round_to_format(v, 10, 5); }
uint16_t orc_bf16_from_double(double v) { return (uint16_t)round_to_format(v, 7, 8); }

static double bf16_to_double(uint16_t h)
{
    uint32_t w = (uint32_t)h << 16;
    float f;
    memcpy(&f, &w, 4);
    return (double)f;
}

static double as_double(uint32_t bits, int type)
{
    if (type == ORC_F16) return orc_f16_to_double((uint16_t)bits);
    if (type == ORC_BF16) return bf16_to_double((uint16_t)bits);
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

uint32_t orc_combine(uint32_t a, uint32_t b, int type, int op)
{
    if (type == ORC_U32) {
        if (op == ORC_ADD) return a + b;                    /* modulo 2^32 */
        if (op == ORC_MIN) return a < b ? a : b;
        return a > b ? a : b;
    }
    if (type == ORC_S32) {
        const int32_t x = (int32_t)a, y = (int32_t)b;
        if (op == ORC_ADD) return a + b;                    /* two's complement wrap */
        if (op == ORC_MIN) return (uint32_t)(x < y ? x : y);
        return (uint32_t)(x > y ? x : y);
    }
    const double x = as_double(a, type), y = as_double(b, type);
    if (op == ORC_MIN) return x < y ? a : (y < x ? b : a);
    if (op == ORC_MAX) return x > y ? a : (y > x ? b : a);
    if (type == ORC_F32) {
        float fx, fy;
        memcpy(&fx, &a, 4);
        memcpy(&fy, &b, 4);
        const float r = fx + fy;                            /* one binary32 add, to nearest */
        uint32_t out;
        memcpy(&out, &r, 4);
        return out;
    }
    /* f16 / bf16: round the exact sum.  For two f16 operands the double sum is exact (both are
     * multiples of 2^-24 below 2^16).  For two bf16 operands it is exact when their exponents
     * differ by at most 45; otherwise the smaller is below 2^-45 of the larger, the exact sum lies
     * far from any bf16 rounding midpoint, and the double sum rounds to the same bf16 value. */
    const double sum = x + y;
    return type == ORC_F16 ? orc_f16_from_double(sum) : orc_bf16_from_double(sum);
}

typedef struct {
    const uint8_t* img;
    int type, op;
} reduce_ctx;

static void reduce_op_one(const orc_map* m, const int64_t* g, uint64_t lin, void* ctx)
{
    const reduce_ctx* rc = (const reduce_ctx*)ctx;
    if (!in_bounds(m, g)) return;
    uint8_t* dst = element_address(m, g);
    uint32_t a = 0, b = 0;
    for (uint32_t k = 0; k < m->esize; k++) {
        a |= (uint32_t)dst[k] << (8 * k);
        b |= (uint32_t)rc->img[orc_swz(lin * m->esize + k, m->span)] << (8 * k);
    }
    const uint32_t r = orc_combine(a, b, rc->type, rc->op);
    for (uint32_t k = 0; k < m->esize; k++) dst[k] = (uint8_t)(r >> (8 * k));
}

void orc_reduce_op(const orc_map* dst, const int32_t* s, const uint8_t* img, int type, int op)
{
    reduce_ctx rc = {img, type, op};
    for_each_element(dst, s, reduce_op_one, &rc);
}

void orc_tile_reduce(const orc_map* dst, const orc_map* src, uint64_t b0, uint64_t b1, int type,
                     int op)
{
    uint8_t* img = (uint8_t*)malloc(orc_box_bytes(src));
    if (!img) return;
    for (uint64_t b = b0; b < b1; b++) {
        int32_t s[5];
        orc_box_start(dst, b, s);
        orc_image(src, s, img);
        orc_reduce_op(dst, s, img, type, op);
    }
    free(img);
}

/* ---------------------------------------------------------------------------------------------
 * GEMM consumer of the k-ordered ring: C = A * B^T, one output element at a time, k in order.
 * ------------------------------------------------------------------------------------------- */
double orc_gemm_dot(const uint16_t* a, uint64_t lda, const uint16_t* b, uint64_t ldb, uint64_t k,
                    uint64_t m, uint64_t n)
{
    double acc = 0.0;
    for (uint64_t i = 0; i < k; i++) {
        acc += bf16_to_double(a[m * lda + i]) * bf16_to_double(b[n * ldb + i]);
    }
    return acc;
}

double orc_gemm_dot_abs(const uint16_t* a, uint64_t lda, const uint16_t* b, uint64_t ldb,
                        uint64_t k, uint64_t m, uint64_t n)
{
    double acc = 0.0;
    for (uint64_t i = 0; i < k; i++) {
        acc += fabs(bf16_to_double(a[m * lda + i]) * bf16_to_double(b[n * ldb + i]));
    }
    return acc;
}

void orc_gemm_block(const uint16_t* a, uint64_t lda, const uint16_t* b, uint64_t ldb, uint64_t k,
                    uint64_t m0, uint64_t m1, uint64_t n0, uint64_t n1, double* out)
{
    for (uint64_t m = m0; m < m1; m++) {
        for (uint64_t n = n0; n < n1; n++) {
            out[(m - m0) * (n1 - n0) + (n - n0)] = orc_gemm_dot(a, lda, b, ldb, k, m, n);
        }
    }
}

/* ---------------------------------------------------------------------------------------------
 * Ring consumer checksum.  The pages' pipeline ([MLSys-TMA] §"把 TMA 放进 pipeline") hands each
 * stage to a consumer but leave what it computes open; this library's consumer reads every element
 * of the tile through the swizzle and reduces it to one fp32 value and one exact integer.
 * ------------------------------------------------------------------------------------------- */
static float bf16_to_f32(uint16_t h)
{
    uint32_t w = (uint32_t)h << 16; /* bf16 is the upper half of a binary32: exact */
    float f;
    memcpy(&f, &w, 4);
    return f;
}

void orc_tile_checksum(const uint8_t* img, uint32_t rows, uint32_t row_bytes, uint32_t span,
                       float* cs, uint64_t* bits)
{
    float sums[256];
    uint32_t cols = row_bytes / 2;
    uint64_t total_bits = 0;
    for (uint32_t r = 0; r < rows; r++) {
        float acc = 0.0f;
        for (uint32_t c = 0; c < cols; c++) {
            uint64_t off = (uint64_t)r * row_bytes + (uint64_t)c * 2;
            uint16_t h = (uint16_t)(img[orc_swz(off, span)] | (img[orc_swz(off + 1, span)] << 8));
            total_bits += h;
            if (c == 0) {
                acc = bf16_to_f32(h);
            } else {
                acc = acc + bf16_to_f32(h);
            }
        }
        sums[r] = acc;
    }
    /* pairwise-adjacent tree, level by level: s'[i] = s[2i] + s[2i+1] */
    for (uint32_t n = rows; n > 1; n /= 2) {
        for (uint32_t i = 0; i < n / 2; i++) sums[i] = sums[2 * i] + sums[2 * i + 1];
    }
    *cs = sums[0];
    *bits = total_bits;
}

void orc_stream_checksums(const orc_map* a, const orc_map* b, uint64_t t0, uint64_t t1,
                          float* cs_a, float* cs_b, uint64_t* bits_a, uint64_t* bits_b)
{
    uint64_t bb = orc_box_bytes(a) > orc_box_bytes(b) ? orc_box_bytes(a) : orc_box_bytes(b);
    uint8_t* img = (uint8_t*)malloc(bb);
    if (!img) return;
    const orc_map* maps[2] = {a, b};
    for (uint64_t t = t0; t < t1; t++) {
        for (int w = 0; w < 2; w++) {
            const orc_map* m = maps[w];
            int32_t s[5];
            orc_box_start(m, t, s);
            orc_image(m, s, img);
            float cs;
            uint64_t bits;
            orc_tile_checksum(img, orc_extent(m, 1), orc_extent(m, 0) * m->esize, m->span, &cs,
                              &bits);
            if (w == 0) {
                cs_a[t] = cs;
                bits_a[t] = bits;
            } else {
                cs_b[t] = cs;
                bits_b[t] = bits;
            }
        }
    }
    free(img);
}

/* ---------------------------------------------------------------------------------------------
 * mbarrier phase model, [MLSys-TMA] §"如何等待 TMA load 完成": a phase tracks an arrival count and
 * pending transaction bytes and completes only when both are zero.  arrive.expect_tx counts one
 * arrival and adds the expected bytes; each finished copy subtracts its bytes (complete-tx); a
 * waiter on parity p returns once the phase with parity p has completed.
 * ------------------------------------------------------------------------------------------- */
static void maybe_complete(orc_mbar* b)
{
    if (b->pending == 0 && b->tx == 0) {
        b->completed++;
        b->phase ^= 1u;
        b->pending = b->count;
    }
}

void orc_mbar_init(orc_mbar* b, uint32_t count)
{
    b->count = count;
    b->pending = count;
    b->tx = 0;
    b->phase = 0;
    b->completed = 0;
}

void orc_mbar_expect_tx(orc_mbar* b, uint32_t bytes) { b->tx += bytes; }

void orc_mbar_arrive(orc_mbar* b)
{
    b->pending -= 1;
    maybe_complete(b);
}

void orc_mbar_arrive_expect_tx(orc_mbar* b, uint32_t bytes)
{
    b->tx += bytes;
    b->pending -= 1;
    maybe_complete(b);
}

void orc_mbar_complete_tx(orc_mbar* b, uint32_t bytes)
{
    b->tx -= bytes;
    maybe_complete(b);
}

int orc_mbar_test_wait(const orc_mbar* b, uint32_t parity)
{
    /* The phase with parity p has completed once the current phase's parity differs from p. */
    return (b->phase & 1u) != (parity & 1u);
}

/* ---------------------------------------------------------------------------------------------
 * [MLSys-TMA] §"128-byte swizzle 的分组要求": eight rows read the same sector column of a 16 x 16
 * sector grid; each 16-byte read covers four neighbouring banks, one "bank sector" of eight.
 * ------------------------------------------------------------------------------------------- */
void orc_bank_sectors(uint32_t col, uint32_t row0, int grouped, uint32_t* out8)
{
    for (uint32_t k = 0; k < 8; k++) {
        uint32_t row = row0 + k;
        uint64_t off;
        if (grouped) {
            /* group col/8 is its own 16-row image of 128-byte rows */
            off = (uint64_t)(col / 8) * 16 * 128 + (uint64_t)row * 128 + (uint64_t)(col % 8) * 16;
        } else {
            off = (uint64_t)row * 256 + (uint64_t)col * 16;
        }
        out8[k] = (uint32_t)((orc_swz(off, 128) >> 4) & 7u);
    }
}
