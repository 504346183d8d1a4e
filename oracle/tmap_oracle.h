/*
 * tmap_oracle.h -- plain, slow CPU oracle for descriptor-driven tiled tensor movement.
 *
 * TEST INFRASTRUCTURE ONLY.  This file and tmap_oracle.c define what the GPU path must compute,
 * written from the pages' definitions one element (or one byte) at a time.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may build, load or call it; the product
 * library never includes, links or calls anything here, and this code includes no CUDA header
 * and shares no source with the GPU path.
 *
 * Sources (the three pages this library follows):
 *   [MLSys-TMA]  mlc.ai "Modern GPU Programming for MLSys", chapter "异步数据搬运：TMA"
 *   [H200-TMA]   coolgpu "H200 · TMA · Tensor Memory Accelerator" feature card
 *   [Book-TMA]   fangpin "gpu-hpc-book", chapter 08 "Cuda TMA （Tensor Memory Accelerator）"
 *
 * Conventions: every dimension list is innermost first (dim 0 is the contiguous one), as in the
 * tensor-map encoder of [H200-TMA] §04 ① and the launcher in [Book-TMA] §"单 block、单 lane、单
 * tile 的 TMA load".  Byte strides are given for every dim, stride[0] being the element size.
 *
 * Pin status (what each function is checked against, beyond itself):
 *   orc_swz span 128 ........ pinned: [MLSys-TMA] §"TMA 如何写入 swizzled layout" formula
 *                             physical_sector = col XOR row, §"用 3D TMA 搬运多个 swizzle atoms"
 *                             physical_sector = logical_sector XOR (row % 8), and the bank-sector
 *                             formulas of §"128-byte swizzle 的分组要求".
 *   orc_swz span 64 / 32 .... pinned outside the pages: the pages name these modes (§"128-byte
 *                             swizzle 的分组要求", last paragraph) but never define their layout.
 *                             Read here as the same address-bit rule with 2 / 1 XOR bits, and
 *                             checked byte by byte against the chunk patterns NVIDIA's public CUDA
 *                             documentation draws for the 32B / 64B / 128B modes (a table in the
 *                             tests' golden files, cited there); plus the invariants (bijection,
 *                             involution, 16-byte units kept whole, eight bank sectors per column).
 *   orc_image / orc_store ... pinned: NONE mode equals numpy strided slicing of a zero-padded
 *                             tensor; 128B mode equals the page's sector-XOR-row rule applied to
 *                             that slice; store(image(x)) restores x with sentinels intact.
 *   elementStrides .......... pinned: the image equals numpy slicing with step estride[i] of the
 *                             zero-padded tensor ([Book-TMA] §"Tensor descriptor：CUtensorMap":
 *                             the step between elements along each dim, counted in elements);
 *                             the store writes exactly those positions.  Reading: the image keeps
 *                             ceil(box / estride) elements along each dim, packed.
 *   NaN fill ................ pinned: out-of-bounds image elements are NaN in the element's float
 *                             format (numpy isnan), in-bounds ones unchanged, stores unaffected.
 *   orc_reduce_add_f32 ...... pinned: numpy float32 addition (IEEE binary32, round to nearest).
 *   orc_combine ............. pinned: f16 add against numpy float16 of the (exact) double sum;
 *                             bf16 add against an exact rational sum rounded half-to-even in
 *                             Python; min / max / integer ops against numpy.  Rounding of f16 /
 *                             bf16 adds is this library's reading (the pages do not state it).
 *   orc_gemm_* .............. pinned: small integer matrices against exact Python integer
 *                             arithmetic, one-hot rows (C picks entries of B), random bf16 values
 *                             against an exact rational sum, and C(A, B) = C(B, A) transposed.
 *   orc_tile_checksum ....... pinned: numpy sequential cumsum + pairwise tree, and an exact
 *                             integer bit-sum.  The checksum itself is this library's definition;
 *                             the pages are silent on what the ring's consumer computes.
 *   orc_mbar_* .............. pinned: the 2048 + 2048 = 4096 byte tally of [MLSys-TMA]
 *                             §"如何等待 TMA load 完成".
 *   orc_bank_sectors ........ pinned: 8 distinct sectors grouped, 4 distinct (2-way) ungrouped,
 *                             [MLSys-TMA] §"128-byte swizzle 的分组要求".
 */
#ifndef TMAP_ORACLE_H
#define TMAP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A tensor map as the oracle sees it: the global tensor lives in HOST memory at `base`. */
typedef struct orc_map {
    uint32_t esize;     /* element size in bytes (1, 2, 4 or 8)                              */
    uint32_t rank;      /* 1..5                                                              */
    uint32_t span;      /* swizzle span in bytes: 0 = none, 32, 64 or 128                    */
    uint32_t fill;      /* out-of-bounds fill: ORC_FILL_ZERO or the NaN of a float format    */
    uint8_t* base;      /* host address of element (0, ..., 0)                               */
    uint64_t dim[5];    /* globalDim, innermost first                                        */
    int64_t  stride[5]; /* byte distance between neighbours along dim i; stride[0] = esize   */
    uint32_t box[5];    /* boxDim, innermost first                                           */
    uint32_t estride[5];/* elementStrides, in elements (1..8)                                */
} orc_map;

/* Out-of-bounds fill ([H200-TMA] §02: the hardware fills out-of-bounds elements with 0 or NaN).
 * The pages name no NaN bit pattern; the oracle writes the quiet NaN with only the leading
 * fraction bit set (f16 0x7E00, bf16 0x7FC0, f32 0x7FC00000, f64 0x7FF8000000000000), and the
 * tests accept any NaN there. */
enum { ORC_FILL_ZERO = 0, ORC_FILL_NAN_F16 = 1, ORC_FILL_NAN_BF16 = 2, ORC_FILL_NAN_F32 = 3,
       ORC_FILL_NAN_F64 = 4 };

/* 0 if the map is one the oracle defines (rank 1..5, box >= 1, elementStrides 1..8, span in
 * {0,32,64,128}, with a span elementStrides[0] = 1 and the inner box row exactly `span` bytes, a
 * NaN fill only in the format of the element size), otherwise a nonzero code. */
int orc_map_check(const orc_map* m);

/* Swizzled position of byte offset `off` of an image whose rows are `span` bytes wide. */
uint64_t orc_swz(uint64_t off, uint32_t span);

/* Image extent along dim i: ceil(box[i] / estride[i]) elements.  Image bytes: esize * prod. */
uint32_t orc_extent(const orc_map* m, uint32_t i);
uint64_t orc_box_bytes(const orc_map* m);
uint64_t orc_num_boxes(const orc_map* m);
/* Start coordinates of box number `b` of the box grid (dim 0 fastest): s[i] = k[i] * box[i]. */
void orc_box_start(const orc_map* m, uint64_t b, int32_t* s);

/* Shared-memory image of the box starting at s[0..rank-1]: image element e (e[i] < extent i) is
 * the tensor element at global coordinate g[i] = s[i] + e[i] * estride[i], stored at byte
 * swz(lin(e) * esize); out-of-bounds elements are the fill (zero bytes or the NaN pattern). */
void orc_image(const orc_map* m, const int32_t* s, uint8_t* img);
/* Writes each in-bounds element of the box starting at s from the image back to global memory
 * (image element e to coordinate s + e * estride); out-of-bounds elements are not written. */
void orc_store(const orc_map* m, const int32_t* s, const uint8_t* img);
/* dst(element) = fl32(dst(element) + image(element)) for each in-bounds element of the box. */
void orc_reduce_add_f32(const orc_map* dst, const int32_t* s, const uint8_t* img);

/* Boxes b0..b1-1 of a copy.  coords == NULL walks the box grid, else coords holds rank int32 per
 * box.  Image of box b goes to images + b * box_bytes. */
void orc_tiled_copy(const orc_map* m, const int32_t* coords, uint64_t b0, uint64_t b1,
                    uint8_t* images);
/* Boxes b0..b1-1 of a round trip: image b is stored through the map at box b's coordinates. */
void orc_tiled_roundtrip(const orc_map* m, const int32_t* coords, uint64_t b0, uint64_t b1,
                         const uint8_t* images);
/* Boxes b0..b1-1 of the box grid of dst (src has the same dims and box): dst += src. */
void orc_tile_reduce_add(const orc_map* dst, const orc_map* src, uint64_t b0, uint64_t b1);

/* The general reduce ([Book-TMA] §"TMA reduce，把“搬运”和“归约”合并": the write-back combines each
 * element with the value in global memory, "add, min and the like").  Element types and ops: */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_U32 = 3, ORC_S32 = 4 };
enum { ORC_ADD = 0, ORC_MIN = 1, ORC_MAX = 2 };
/* One element: the bit pattern of op(a, b), a from dst and b from src, in the element type.
 *   float add: the exact sum rounded to nearest, ties to even, in the element format (subnormal
 *              results kept, overflow to infinity);  float min / max: the smaller / larger value;
 *   u32 / s32 add: the sum modulo 2^32;  u32 / s32 min / max: unsigned / signed comparison. */
uint32_t orc_combine(uint32_t a, uint32_t b, int type, int op);
/* dst(element) = op(dst(element), image(element)) for each in-bounds element of the box. */
void orc_reduce_op(const orc_map* dst, const int32_t* s, const uint8_t* img, int type, int op);
/* Boxes b0..b1-1 of the grid of dst: load the src box into its image, reduce it into dst. */
void orc_tile_reduce(const orc_map* dst, const orc_map* src, uint64_t b0, uint64_t b1, int type,
                     int op);
/* Exact conversions used by the above (exposed for the pins). */
double orc_f16_to_double(uint16_t h);
uint16_t orc_f16_from_double(double v);
uint16_t orc_bf16_from_double(double v);

/* The k-ordered ring's tensor-core consumer ([MLSys-TMA] overview and §"把 TMA 放进 pipeline": while
 * the tensor cores work on the A and B tiles of step k, TMA loads those of step k + 1): for bf16 A
 * (M x K, row m at a + m * lda elements) and B (N x K, row n at b + n * ldb), both with K
 * contiguous, C[m][n] = sum over k of A[m][k] * B[n][k].  orc_gemm_dot returns that sum in double
 * (each bf16 product is exact in double; the K-term sum is exact up to about K * 2^-53 relative),
 * orc_gemm_dot_abs the sum of |A[m][k] * B[n][k]| (the scale of the fp32 tolerance). */
double orc_gemm_dot(const uint16_t* a, uint64_t lda, const uint16_t* b, uint64_t ldb, uint64_t k,
                    uint64_t m, uint64_t n);
double orc_gemm_dot_abs(const uint16_t* a, uint64_t lda, const uint16_t* b, uint64_t ldb,
                        uint64_t k, uint64_t m, uint64_t n);
/* C[m][n] for m in [m0, m1), n in [n0, n1) into out (row-major, (n1 - n0) per row). */
void orc_gemm_block(const uint16_t* a, uint64_t lda, const uint16_t* b, uint64_t ldb, uint64_t k,
                    uint64_t m0, uint64_t m1, uint64_t n0, uint64_t n1, double* out);

/* Checksum of one bf16 tile image of `rows` rows of `row_bytes` bytes (rows a power of two):
 * rowsum_r is the sequential fp32 sum of the row's elements in logical order, the tile value is
 * the pairwise-adjacent tree over the row sums, and bits is the sum of the raw 16-bit patterns. */
void orc_tile_checksum(const uint8_t* img, uint32_t rows, uint32_t row_bytes, uint32_t span,
                       float* cs, uint64_t* bits);
/* Tiles t0..t1-1 of two rank-2 bf16 maps walked in box-grid order, tile t of A paired with tile t
 * of B. */
void orc_stream_checksums(const orc_map* a, const orc_map* b, uint64_t t0, uint64_t t1,
                          float* cs_a, float* cs_b, uint64_t* bits_a, uint64_t* bits_b);

/* mbarrier phase model: pending arrivals, pending transaction bytes and phase parity. */
typedef struct orc_mbar {
    int64_t  count;        /* expected arrivals per phase (from init)        */
    int64_t  pending;      /* arrivals still missing in the current phase    */
    int64_t  tx;           /* transaction bytes still missing                */
    uint32_t phase;        /* parity of the current (incomplete) phase       */
    uint32_t completed;    /* number of completed phases                     */
} orc_mbar;
void orc_mbar_init(orc_mbar* b, uint32_t count);
void orc_mbar_expect_tx(orc_mbar* b, uint32_t bytes);
void orc_mbar_arrive(orc_mbar* b);
void orc_mbar_arrive_expect_tx(orc_mbar* b, uint32_t bytes);
void orc_mbar_complete_tx(orc_mbar* b, uint32_t bytes);
/* 1 once the phase with the given parity has completed. */
int orc_mbar_test_wait(const orc_mbar* b, uint32_t parity);

/* Bank sectors (0..7, four 4-byte banks each) hit by eight 16-byte reads of sector column `col`
 * (0..15) of a 16 x 16 sector grid, rows row0..row0+7, under 128-byte swizzle.  grouped != 0 splits
 * every 256-byte row into two 128-byte groups stored as separate 16-row images; grouped == 0 keeps
 * the 256-byte row stride. */
void orc_bank_sectors(uint32_t col, uint32_t row0, int grouped, uint32_t* out8);

#ifdef __cplusplus
}
#endif
#endif
