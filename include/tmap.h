/*
 * tmap.h -- C ABI of the GB300 (sm_103a) tiled tensor movement library (libtmap_gb300.so).
 *
 * A tensor map describes how a global tensor is cut into boxes; each box is moved between global
 * memory and a (possibly swizzled) shared-memory image by the Tensor Memory Accelerator, then
 * written out, stored back through a map, reduce-added, or consumed from a multi-stage ring.
 *
 * Sources (cited below by tag and section):
 *   [MLSys-TMA]  mlc.ai "Modern GPU Programming for MLSys", chapter "异步数据搬运：TMA"
 *   [H200-TMA]   coolgpu "H200 · TMA · Tensor Memory Accelerator" feature card
 *   [Book-TMA]   fangpin "gpu-hpc-book", chapter 08 "Cuda TMA （Tensor Memory Accelerator）"
 *
 * Conventions shared by every call
 *   - Every call returns an int status (TM_OK = 0 or a TM_E* code); tm_last_error() returns a
 *     thread-local description of the last failure.  No C++ exception or abort crosses the ABI.
 *   - The caller owns all memory.  Tensor bases, image buffers and checksum arrays are DEVICE
 *     pointers on the current CUDA device; coordinate lists and dimension arrays are HOST pointers
 *     read before the call returns.  The library never frees a caller's buffer.
 *   - Dimension, stride, box and coordinate arrays are innermost first (index 0 is the contiguous
 *     dimension), as in the encoder of [H200-TMA] §04 ① and the launcher of [Book-TMA]
 *     §"单 block、单 lane、单 tile 的 TMA load".
 *   - Launching calls are asynchronous on `stream` (a cudaStream_t passed as void*, NULL = the
 *     legacy default stream).  Argument errors are reported synchronously.  A wait that gives up
 *     inside a kernel (every mbarrier wait is bounded, default 1 s, TM_WAIT_TIMEOUT_NS overrides)
 *     is recorded in a per-device status word and reported by tm_stream_check().
 *   - The first call that launches work on a device allocates that device's 64-byte status word
 *     and 32 KiB of work counters (cudaMalloc) and reads its attributes; make that first call
 *     before capturing a stream.  A call given an explicit list of more than 8 boxes stages the
 *     list in device memory with cudaMallocAsync/cudaFreeAsync on `stream`.
 *   - The tensor-map copies, round trips and reduces split their boxes between CTAs dynamically:
 *     a launch takes items from a work counter of its stream (one per stream, up to 256 streams a
 *     device; zero between launches, reset by the launch itself), so a stream's launches must not
 *     run on another stream's counter -- the library keys them by cudaStreamGetId.  A launch made
 *     while its stream is being captured, launches on streams beyond the 256th, maps whose
 *     images take shared-memory slots of at most 1 KiB (boxes far smaller than a stage, whose
 *     launches run several CTAs per SM), and TM_DYNAMIC=0 use a fixed split instead; the bytes
 *     written are the same either way.
 *   - Environment (read at each launch; none changes the bytes written, only the launch shape;
 *     the defaults are the shapes measured fastest on GB300):
 *       TM_WAIT_TIMEOUT_NS        limit of every bounded wait (1e9)
 *       TM_DYNAMIC                0: fixed split everywhere (1)
 *       TM_DYN_BATCH, TM_DYN_BATCH_REDUCE   items a fetch for copies, reductions (1, 4)
 *       TM_DYN_TAPER              last items per CTA handed out singly in batched launches (4)
 *       TM_GROUP_BYTES            stage size of the tensor-map streaming kernels (32768; 16384
 *                                 for image slots of at most 1 KiB)
 *       TM_CTAS_PER_SM            CTAs per SM of those kernels (1; 4 for small slots)
 *       TM_STAGES, TM_STAGES_REDUCE   stage cap for copies, reductions (none, 4)
 *       TM_FB_SEG                 vector path segment form: 0 never, 1 whenever possible (auto)
 *       TM_FB_SEG_CTAS_PER_SM, TM_FB_SEG_STAGES, TM_FB_SEG_WARPS   segment kernels' shape
 *                                 (3, fewer if the SM cannot hold them; 3; 8 consumer warps:
 *                                 8, 12 or 16)
 *       TM_FB_COPY_CTAS_PER_SM, TM_FB_STORE_CTAS_PER_SM   per-window vector kernels (8, 6)
 *       TM_RING_GROUPS, TM_RING_EVICT_FIRST, TM_RING_ROW_PAIRS, TM_RING_PREFETCH   stream_tiles
 *                                 (2 consumer groups, evict-first loads on, 0, 0)
 *       TM_GEMM_PAIR, TM_GEMM_TAIL_SPLIT   stream_gemm: CTA pairs, split last wave (1, 1)
 */
#ifndef TMAP_GB300_H
#define TMAP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes --------------------------------------------------------------------------- */
#define TM_OK 0
#define TM_EINVAL 1        /* malformed argument: NULL pointer, bad enum, rank, count mismatch   */
#define TM_EALIGN 2        /* an address, stride or inner box row breaks an alignment rule       */
#define TM_ERANGE 3        /* a size is out of range: dim, box, stride, or box too large for smem */
#define TM_EUNSUPPORTED 4  /* legal for the hardware but not supported by this library           */
#define TM_ECUDA 5         /* the CUDA runtime or driver reported an error                       */
#define TM_ETIMEOUT 6      /* a bounded wait inside a kernel gave up                             */

/* ---- element types (numerically equal to CUtensorMapDataType) ----------------------------- */
typedef enum tm_dtype {
    TM_U8 = 0, TM_U16 = 1, TM_U32 = 2, TM_S32 = 3, TM_U64 = 4, TM_S64 = 5,
    TM_F16 = 6, TM_F32 = 7, TM_F64 = 8, TM_BF16 = 9
} tm_dtype;

/* ---- swizzle modes (numerically equal to CUtensorMapSwizzle) -------------------------------
 * [MLSys-TMA] §"TMA 如何写入 swizzled layout" and §"用 3D TMA 搬运多个 swizzle atoms": with 128B,
 * inside each atom of 8 rows x 128 bytes the 16-byte sector c of image row r is written to sector
 * c XOR (r % 8).  64B / 32B are the narrower atoms of §"128-byte swizzle 的分组要求" (8 rows x 64 /
 * 32 bytes, XOR of the row bits 7..8 / 7 into the chunk bits 4..5 / 4).  With any swizzle the inner
 * box row must be exactly the atom width (boxDim[0] * element size == 32, 64 or 128 bytes). */
typedef enum tm_swizzle {
    TM_SWIZZLE_NONE = 0, TM_SWIZZLE_32B = 1, TM_SWIZZLE_64B = 2, TM_SWIZZLE_128B = 3
} tm_swizzle;

/* ---- out-of-bounds fill, [H200-TMA] §02 (out-of-bounds row: the hardware fills with 0 / NaN) -
 * TM_OOB_ZERO: out-of-bounds image elements are zero bytes.  TM_OOB_NAN (floating-point dtypes
 * only): they are a NaN of the element's format.  The pages name no NaN bit pattern; both paths
 * write the one GB300's NaN-request fill was measured to write, the 16-bit pattern 0x7FF7 repeated
 * over the element (f16 / bf16 0x7FF7, f32 0x7FF77FF7, f64 0x7FF77FF77FF77FF7).  Stores and
 * reduces never write out-of-bounds elements, so the fill only shows in images. */
typedef enum tm_oob { TM_OOB_ZERO = 0, TM_OOB_NAN = 1 } tm_oob;

/* ---- execution paths ------------------------------------------------------------------------ */
#define TM_PATH_TMA 1      /* cp.async.bulk.tensor with a driver-encoded tensor map               */
#define TM_PATH_FALLBACK 2 /* the vector path where TMA cannot go: aligned 16-byte windows or
                            * bulk-copied row segments staged in shared memory, realigned
                            * there, written with 16-byte vector stores                      */
/* why a descriptor is on the fallback path (bit set in tm_desc.why_fallback) */
#define TM_WHY_STRIDE 1u   /* a global stride is not a multiple of 16 bytes ([H200-TMA] §03)     */
#define TM_WHY_BASE 2u     /* the base address is not 16-byte aligned ([H200-TMA] §03)           */
#define TM_WHY_DRIVER 4u   /* the driver's encoder refused the map                               */
#define TM_WHY_FORCED 8u   /* tmap_force_fallback() was called                                   */
#define TM_WHY_STEP0 16u   /* elementStrides[0] > 1: the tensor-map hardware ignores the step of
                            * dim 0 in a non-interleaved map (NVIDIA's driver documentation of
                            * cuTensorMapEncodeTiled says so) and delivers boxDim[0] elements per
                            * row, not the ceil(boxDim[0] / elementStrides[0]) the image holds */

/* ---- the descriptor -------------------------------------------------------------------------
 * [MLSys-TMA] §"一个 thread 如何描述整个 tile": the descriptor says how the whole tensor is laid
 * out (type, shape, strides, box, swizzle); each copy only adds a start coordinate and a
 * shared-memory address.  [Book-TMA] §"Tensor descriptor：CUtensorMap" lists its fields.
 * A caller-allocated plain struct, 64-byte aligned ([H200-TMA] §03: the CUtensorMap object itself
 * is 64-byte aligned), filled by tmap_encode() or tmap_plan() and passed by pointer; the library
 * copies the embedded CUtensorMap into kernel parameter space (__grid_constant__, [H200-TMA] §03).
 * Field offsets are part of the ABI (static-asserted in the library). */
typedef struct __attribute__((aligned(64))) tm_desc {
    uint32_t magic;         /* TM_DESC_MAGIC once filled                                        */
    uint32_t dtype;         /* tm_dtype                                                         */
    uint32_t esize;         /* element size in bytes                                            */
    uint32_t rank;          /* 1..5                                                             */
    uint32_t swizzle;       /* tm_swizzle                                                       */
    uint32_t oob;           /* tm_oob                                                           */
    uint32_t path;          /* TM_PATH_TMA or TM_PATH_FALLBACK                                  */
    uint32_t why_fallback;  /* TM_WHY_* bits when path == TM_PATH_FALLBACK                      */
    uint64_t base;          /* device address of element (0, ..., 0)                           */
    uint64_t dim[5];        /* globalDim, innermost first (unused entries 1)                    */
    uint64_t stride[5];     /* byte stride of each dim; stride[0] = esize (unused entries 0)    */
    uint32_t box[5];        /* boxDim (unused entries 1)                                        */
    uint32_t estride[5];    /* elementStrides, 1..8 (unused entries 1)                          */
    uint64_t nbox[5];       /* boxes along each dim: ceil(dim / box)                           */
    uint64_t box_bytes;     /* bytes of one box image: esize * prod(ceil(box / estride))        */
    uint64_t num_boxes;     /* prod(nbox)                                                       */
    uint32_t l2_promotion;  /* tm_l2_promotion of the TMA loads (tmap_set_l2_promotion)          */
    uint8_t reserved[36];
    uint8_t tmap[128];      /* CUtensorMap (driver-encoded) when path == TM_PATH_TMA            */
} tm_desc;

#define TM_DESC_MAGIC 0x544d4150u /* "TMAP" */
#define TM_MAX_BOX_BYTES 229376u  /* 224 KiB: one image must fit a CTA's shared memory          */
#define TM_MAX_STAGES 16u

/* tmap_plan -- validate a tensor map and fill `out` without touching the GPU or the driver.
 *   [H200-TMA] §03 rules: 1 <= rank <= 5 (else TM_EINVAL); 1 <= globalDim[i] <= 2^32 and
 *   1 <= boxDim[i] <= 256 (else TM_ERANGE); boxDim[0] * esize a multiple of 16 bytes (else
 *   TM_EALIGN); globalStrides below 2^40 (else TM_ERANGE).  [MLSys-TMA] §"用 3D TMA 搬运多个
 *   swizzle atoms" and §"128-byte swizzle 的分组要求": with a swizzle, boxDim[0] * esize equals the
 *   atom width (else TM_EUNSUPPORTED).  box_bytes above TM_MAX_BOX_BYTES gives TM_ERANGE.
 *   elementStrides (NULL = all 1; [Book-TMA] §"Tensor descriptor：CUtensorMap": the step, in
 *   elements, between the elements taken along each dim): each 1..8 (else TM_EINVAL).  Along dim
 *   i the image takes the box's elements start, start + es, ... below start + boxDim[i], i.e.
 *   ceil(boxDim[i] / es) of them, packed; the box grid still steps by boxDim.  The image row,
 *   ceil(boxDim[0] / es[0]) * esize bytes, must be a multiple of 16 (else TM_EALIGN), and a
 *   swizzled map needs elementStrides[0] == 1 (else TM_EUNSUPPORTED).  A map with
 *   elementStrides[0] > 1 goes to the fallback path (TM_WHY_STEP0).  oob: TM_OOB_NAN needs a
 *   floating-point dtype (else TM_EINVAL).
 *   A base or stride that is a multiple of the element size but not of 16 bytes is NOT an error:
 *   the map goes to the fallback path (why_fallback says which).  A base or stride that is not a
 *   multiple of the element size gives TM_EALIGN.
 *   dtype, rank, base: element type, number of dims, device address of element (0,...,0).
 *   globalDim[rank]: elements per dim.  globalStrides[rank-1]: bytes between neighbours along dims
 *   1..rank-1 (any order, strides need not grow with the dim index: [MLSys-TMA] §"用 3D TMA 搬运多个
 *   swizzle atoms" regroups a row with a smaller outer stride).  boxDim[rank]: box shape. */
int tmap_plan(tm_desc* out, tm_dtype dtype, uint32_t rank, void* base, const uint64_t* globalDim,
              const uint64_t* globalStrides, const uint32_t* boxDim,
              const uint32_t* elementStrides, tm_swizzle swizzle, tm_oob oob);

/* tmap_encode -- tmap_plan(), then, for a TMA-path map, encode the CUtensorMap with the driver's
 *   cuTensorMapEncodeTiled ([H200-TMA] §04 ①, [Book-TMA] §"单 block、单 lane、单 tile 的 TMA load";
 *   the map is created on the host, [H200-TMA] §05).  If the driver refuses a map that passed
 *   validation, the map goes to the fallback path with TM_WHY_DRIVER.  TM_ECUDA if no driver is
 *   reachable.  Same arguments as tmap_plan(). */
int tmap_encode(tm_desc* out, tm_dtype dtype, uint32_t rank, void* base,
                const uint64_t* globalDim, const uint64_t* globalStrides, const uint32_t* boxDim,
                const uint32_t* elementStrides, tm_swizzle swizzle, tm_oob oob);

/* tmap_replace_address -- move an encoded map to another base address of the same layout
 *   ([H200-TMA] §03 and §05: rebase with cuTensorMapReplaceAddress rather than rebuilding on the
 *   device).  A new base that is not 16-byte aligned moves the map to the fallback path; one that
 *   is not a multiple of the element size gives TM_EALIGN. */
int tmap_replace_address(tm_desc* d, void* new_base);

/* tmap_set_l2_promotion -- the L2 promotion the tensor map asks of its loads, a field of the
 *   driver's tensor map ([H200-TMA] §04 ① and [Book-TMA] §"单 block、单 lane、单 tile 的 TMA
 *   load" pass CU_TENSOR_MAP_L2_PROMOTION_NONE to cuTensorMapEncodeTiled).  Performance only: no
 *   result depends on it, and the oracle has no counterpart.  Maps start at TM_L2_128B (or the
 *   value of the environment variable TM_L2_PROMOTION, 0..3, when it is set).  An encoded
 *   tensor-map-path map is re-encoded with the new value; a planned or fallback-path map keeps it
 *   for a later encode.  promo above TM_L2_256B, or an unfilled descriptor: TM_EINVAL. */
typedef enum tm_l2_promotion {
    TM_L2_NONE = 0, TM_L2_64B = 1, TM_L2_128B = 2, TM_L2_256B = 3
} tm_l2_promotion;
int tmap_set_l2_promotion(tm_desc* d, tm_l2_promotion promo);

/* tmap_force_fallback -- put a valid map on the fallback path (why_fallback |= TM_WHY_FORCED).
 *   Used to check that both paths produce identical bytes. */
int tmap_force_fallback(tm_desc* d);

/* tile_load_image -- one box to its shared-memory image, written to `image` (device, box_bytes,
 *   16-byte aligned).  [Book-TMA] §"单 block、单 lane、单 tile 的 TMA load" (one block, one lane,
 *   one tile) and [MLSys-TMA] §"TMA 如何写入 swizzled layout": image element e (box coordinates,
 *   dim 0 fastest) sits at swizzle(lin(e) * esize) and comes from tensor coordinate
 *   start + e * elementStrides; elements outside the tensor are the map's fill (tm_oob).
 *   coords[rank] (host): signed start of the box; may lie partly or wholly outside the tensor. */
int tile_load_image(const tm_desc* src, const int32_t* coords, void* image, void* stream);

/* tiled_copy -- images of many boxes, image b written at images + b * box_bytes (tile-major).
 *   coords == NULL: the whole box grid, box b = k0 + nbox0 * (k1 + nbox1 * (...)) starting at
 *   k[i] * box[i]; nbox must be 0 or num_boxes.  Otherwise coords holds nbox * rank int32 (host).
 *   Each box is one TMA load completed through an mbarrier byte count ([MLSys-TMA] §"如何等待 TMA
 *   load 完成") and one bulk store of the image completed through a bulk async group.  `images`:
 *   device, nbox * box_bytes, 16-byte aligned.  An empty list (coords != NULL, nbox == 0)
 *   returns TM_OK at once, launches nothing and may pass images == NULL. */
int tiled_copy(const tm_desc* src, const int32_t* coords, size_t nbox, void* images,
               void* stream);

/* tiled_roundtrip -- the reverse of tiled_copy: image b (device, tile-major as above) is stored
 *   through `dst` at box b's coordinates.  Only in-bounds elements are written; padding and
 *   everything else in dst keeps its bytes.  Completion of each store is tracked with
 *   commit_group / wait_group ([MLSys-TMA] §"如何等待 TMA store 完成", [Book-TMA] §"TMA store").
 *   The tensor store writes whole 16-byte units of the innermost dimension, so a map whose
 *   globalDim[0] * esize is not a multiple of 16 (or a box list starting off the 16-byte grid or
 *   outside the tensor) is stored by the vector path instead, which writes exactly the in-bounds
 *   bytes.  So is a map with an elementStride other than 1: image element e goes back to tensor
 *   coordinate start + e * elementStrides, and no other element is written.  An empty list
 *   (coords != NULL, nbox == 0) returns TM_OK at once and may pass images == NULL. */
int tiled_roundtrip(const tm_desc* dst, const int32_t* coords, size_t nbox, const void* images,
                    void* stream);

/* tile_reduce_add -- dst += src over the whole box grid, fp32, one IEEE binary32 add (round to
 *   nearest) per in-bounds element, performed by the bulk tensor reduce ([Book-TMA] §"TMA reduce，
 *   把“搬运”和“归约”合并").  Both maps TM_F32 with equal dims, box and swizzle (else TM_EINVAL /
 *   TM_EUNSUPPORTED); strides and bases may differ.  dst and src must not overlap.  As for
 *   tiled_roundtrip, a dst whose globalDim[0] * esize is not a multiple of 16 is reduced by the
 *   vector path (one IEEE add per element, same result). */
int tile_reduce_add(const tm_desc* dst, const tm_desc* src, void* stream);

/* tile_reduce -- dst = op(dst, src) over the whole box grid, one combine per in-bounds element
 *   ([Book-TMA] §"TMA reduce，把“搬运”和“归约”合并": the write-back combines each element with the
 *   value in global memory, "add, min and the like").  Types TM_F32, TM_F16, TM_BF16, TM_U32,
 *   TM_S32 (else TM_EUNSUPPORTED); dst and src of one type with equal dims, box and swizzle (else
 *   TM_EINVAL), elementStrides all 1 (else TM_EUNSUPPORTED); they must not overlap.  Semantics: float add = the exact sum rounded to nearest,
 *   ties to even, in the element type (a reading: the pages fix no rounding); min / max = the
 *   smaller / larger value (dst kept on a tie); u32 / s32 add wraps modulo 2^32.  Add on every type
 *   and min / max on u32 / s32 use the bulk tensor reduce; float min / max, and maps the tensor
 *   store cannot take, run element-wise on the vector path (same results). */
typedef enum tm_redop { TM_RED_ADD = 0, TM_RED_MIN = 1, TM_RED_MAX = 2 } tm_redop;
int tile_reduce(const tm_desc* dst, const tm_desc* src, tm_redop op, void* stream);

/* stream_tiles -- a `stages`-deep producer/consumer ring ([MLSys-TMA] §"把 TMA 放进 pipeline"):
 *   one elected producer thread fills stage s with tile t of A and tile t of B (one mbarrier,
 *   expect_tx = 2 * box_bytes), consumer warps read the stage through the swizzle and release it.
 *   A and B: TM_BF16, rank 2, box {64, R} with R in {32, 64, 128, 256}, swizzle 128B or NONE,
 *   TMA path, elementStrides all 1 and TM_OOB_ZERO (else TM_EUNSUPPORTED), equal num_boxes; tiles
 *   are walked in box-grid order.  Per tile t (device outputs,
 *   num_boxes entries each): cs = fp32 checksum (each row summed in order from its first element,
 *   then a pairwise-adjacent tree over the rows), bits = sum of the 16-bit patterns.
 *   stages: 2..8.  With an even stage count two consumer groups take the even and the odd tiles
 *   (TM_RING_GROUPS=1 keeps one); TM_RING_ROW_PAIRS=1 reads each 32-row block in the row order of
 *   an ungrouped 256-byte row (the 2-way bank-conflict control of [MLSys-TMA] §"128-byte swizzle
 *   的分组要求").  Each tile is read once, so the tile loads carry an L2 evict-first policy: the
 *   stream recycles its own L2 lines instead of evicting other data (TM_RING_EVICT_FIRST=0 drops
 *   the policy).  None of these changes the outputs. */
int stream_tiles(const tm_desc* a, const tm_desc* b, uint32_t stages, float* cs_a, float* cs_b,
                 uint64_t* bits_a, uint64_t* bits_b, void* stream);

/* stream_gemm -- the ring in GEMM order, feeding the tensor cores ([MLSys-TMA] overview: while the
 *   tensor cores work on the A and B tiles of step k, TMA brings those of step k + 1 into shared
 *   memory in the swizzled layout the MMA reads; §"把 TMA 放进 pipeline": barriers hand each stage
 *   between the TMA producer and the MMA consumer).  C = A * B^T: A is M x K and B is N x K, bf16
 *   with K contiguous, given as rank-2 TM_BF16 maps {K, M} with box {64, 128} and {K, N} with box
 *   {64, 256}, 128-byte swizzle, TMA path, unit steps, zero fill (else TM_EUNSUPPORTED), equal K
 *   (else TM_EINVAL); M, N, K below 2^31.  Persistent CTAs (one per SM) run a `stages`-deep ring
 *   (stages 2..7, else TM_ERANGE): tcgen05.mma (bf16 in, fp32 accumulated in two tensor-memory accumulators, so
 *   one tile's epilogue overlaps the next tile's MMAs), k in steps of 64.  When C has more than one
 *   128-row tile, clusters of two CTAs on two SMs compute 256 x 256 tiles with tcgen05
 *   cta_group::2: each CTA loads its 128-row halves of the A and B tiles into 32 KiB stages (all 7
 *   usable), the leader issues the MMAs over both; a last wave that would leave at least half the
 *   pairs idle is done as 256 x 128 half tiles (TM_GEMM_TAIL_SPLIT=0 keeps whole tiles); TM_GEMM_PAIR=0 gives instead one SM per
 *   128 x 256 tile (48 KiB stages, at most 4 used).  A C of one 128-row tile uses one-SM CTAs.  c: device, fp32, row-major M x N with ldc >= N elements between
 *   rows, 16-byte aligned, ldc a multiple of 4 (else TM_EALIGN).  Ragged M, N and K are zero-filled by the
 *   loads; only in-bounds elements of C are written.  Accuracy: the fp32 result differs from the
 *   exact sum of the K products by at most K * 2^-23 * sum |A[m][k] * B[n][k]| (any summation order,
 *   rounding to nearest or toward zero).  A wait that gives up is reported by tm_stream_check();
 *   C is then undefined. */
int stream_gemm(const tm_desc* a, const tm_desc* b, float* c, uint64_t ldc, uint32_t stages,
                void* stream);

/* tiled_copy_noalloc -- tiled_copy for callers that must not allocate device memory.  The pages
 *   have no counterpart: it exists because tiled_copy allocates (its first launching call on a
 *   device cudaMallocs the status word; a list of more than 8 boxes is staged with
 *   cudaMallocAsync), and some callers cannot allow an allocation -- code running while another
 *   allocator owns all device memory, processes under a hard device-memory cap where a late
 *   allocation may fail, latency-critical loops that cannot afford an allocator call.
 *   Same arguments, the same image bytes and the same launch shape as tiled_copy (one rule and
 *   the same tunables for both), with the fixed split of boxes between CTAs: the dynamic split
 *   of tiled_copy takes its items from work counters the library allocates.  All scratch (a status word and the
 *   box list, at most TM_NOALLOC_MAX_BOXES boxes; a longer list gives TM_ERANGE) lives in one
 *   fixed __device__ array of 327,936 bytes inside the library, held by every GPU that loads the
 *   library until the process exits.  The first call on a device looks up that array's device
 *   address (cudaGetSymbolAddress, with the device current); make that first call before any
 *   stream capture.  The call returns when the copy has finished: it synchronises `stream` and
 *   returns TM_ETIMEOUT itself if a wait inside the kernel gave up.  Every call shares the one
 *   array and clears its status word first: calls that overlap on the GPU (other host threads,
 *   other streams) race on it and must not be issued. */
#define TM_NOALLOC_MAX_BOXES 16384u
int tiled_copy_noalloc(const tm_desc* src, const int32_t* coords, size_t nbox, void* images,
                       void* stream);

/* tm_stream_check -- synchronise `stream`, then read and clear the current device's status word:
 *   TM_ETIMEOUT if a kernel's bounded wait gave up since the last check (tm_last_error() names the
 *   kernel, block, stage, phase and box), TM_ECUDA on a CUDA error, else TM_OK.  Kernels on
 *   different streams share the word: the first failure is kept. */
int tm_stream_check(void* stream);

/* tm_selftest_wait_timeout -- launch one block that waits, with the given limit, on an mbarrier
 *   nothing will complete; the wait gives up, records TM_ETIMEOUT and the kernel returns.  Lets a
 *   caller check that failure reporting works without faulting anything. */
int tm_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

const char* tm_last_error(void);
size_t tm_box_bytes(const tm_desc* d);   /* 0 for an unfilled descriptor */
size_t tm_num_boxes(const tm_desc* d);   /* 0 for an unfilled descriptor */
int tm_path(const tm_desc* d);           /* TM_PATH_* or 0 */
size_t tm_desc_size(void);               /* sizeof(tm_desc) == 384 */
/* The widest swizzle whose atom row fits `inner_bytes` exactly, [MLSys-TMA] §"128-byte swizzle 的
 * 分组要求" (choose the widest swizzle the tile allows, else 64 or 32 bytes): 128 -> 128B,
 * 64 -> 64B, 32 -> 32B, anything else -> NONE. */
int tm_pick_swizzle(uint32_t inner_bytes);

#ifdef __cplusplus
}
#endif
#endif /* TMAP_GB300_H */
