// tm_internal.h -- launch parameters shared by the host side (tmap_host.cpp) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <algorithm>

#include "tmap.h"

namespace tmk {

// A non-negative integer from the environment (library tunables), or dflt when unset or malformed.
inline uint64_t env_u64(const char* name, uint64_t dflt)
{
    const char* v = getenv(name);
    if (!v || !*v) return dflt;
    char* end = nullptr;
    const unsigned long long x = strtoull(v, &end, 10);
    return (end && *end == 0) ? (uint64_t)x : dflt;
}

constexpr uint32_t kInlineBoxes = 8;   // explicit box lists up to this size travel in parameters
constexpr uint32_t kStageAlign = 1024; // 128B swizzle is computed on smem address bits 4..9

// Kernel ids recorded with a timeout.
enum KernelId : uint32_t {
    K_COPY = 1, K_ROUNDTRIP = 2, K_REDUCE = 3, K_STREAM = 4, K_FB_COPY = 5, K_FB_STORE = 6,
    K_FB_REDUCE = 7, K_SELFTEST = 8, K_GEMM = 9, K_FB_SEG_COPY = 10, K_FB_SEG_STORE = 11
};

// Per-device status word written by a kernel whose bounded wait gave up.
struct StatusBlock {
    int code;          // 0 or TM_ETIMEOUT; first failure wins (atomicCAS)
    uint32_t kernel;   // KernelId
    uint32_t block;    // blockIdx.x
    uint32_t stage;    // ring stage
    uint64_t box;      // box (or tile) index
    uint32_t phase;    // parity waited for
    uint32_t pad[9];
};
static_assert(sizeof(StatusBlock) == 64, "status block is 64 bytes");

// How a launch enumerates its boxes: the whole grid, a device list, or a short inline list.
enum WalkMode : uint32_t { WALK_GRID = 0, WALK_LIST = 1, WALK_INLINE = 2 };

struct BoxWalk {
    uint64_t nbox;         // boxes handled by the launch
    uint64_t grid_nb[5];   // boxes along each dim (grid mode)
    uint32_t box[5];       // box shape (unused dims 1)
    uint32_t rank;
    uint32_t mode;         // WalkMode
    const int32_t* list;   // nbox * rank coordinates (WALK_LIST)
    int32_t inl[kInlineBoxes * 5];
};

#if defined(__CUDACC__)
#define TM_HD __host__ __device__
#else
#define TM_HD
#endif

// TMA-path streaming kernels (copy, round trip, reduce).
//
// Work split over a grid of `grid` CTAs: the boxes are taken in full waves of grid x G consecutive
// boxes (G = group, the boxes sharing one stage), CTA c taking boxes (j * grid + c) * G .. + G - 1
// of wave j; the R < grid x G boxes after the last full wave form the tail, dealt out at box
// granularity: CTA c takes q + (c < r ? 1 : 0) consecutive boxes of it (q = R / grid, r = R % grid;
// at most G, so they fit one stage).  No CTA has more than one box above the mean.
struct StreamArgs {
    BoxWalk walk;
    uint64_t images;       // copy: destination images; round trip: source images
    uint32_t box_bytes;
    uint32_t stage_bytes;  // group * box_bytes rounded up to kStageAlign
    uint32_t stages;
    uint32_t group;        // G: consecutive boxes per stage
    uint32_t slot_bytes;   // stage bytes per box: box_bytes rounded up to its swizzle period
    uint32_t pad0;
    uint64_t timeout_ns;
    StatusBlock* status;
    // The launch-wide schedule, computed once on the host (stream_schedule) so that no CTA runs
    // 64-bit divisions before its first load.
    uint64_t waves;        // full waves of grid x G boxes
    uint64_t tail0;        // first box of the tail: waves x grid x G
    uint32_t tail_q;       // tail boxes per CTA: tail_q, one more below tail_r
    uint32_t tail_r;
    uint32_t dstep[5];     // digits (radix: the grid's box counts) of grid x G boxes
    uint32_t pad;
    // Dynamic work split (when sched is set): items g = 0 .. nitems - 1 of G boxes (the last one
    // short); CTA c takes c, c + grid, ... for its first stages + 1 items, then fetches from
    // sched[0] (a counter of this launch's stream, zero at launch; sched[1] counts the CTAs that
    // are done, and the last one sets both back to zero).  Fetches 0 .. batched - 1 take `batch`
    // consecutive items each, later fetches one item: the last items of a launch go out singly.
    unsigned long long* sched;
    uint64_t nitems;
    uint32_t batch;        // items per fetch from the counter, for the first `batched` fetches
    uint32_t pad2;
    uint64_t batched;
};

// CTAs per SM of the streaming kernels (see stream_plan).  One, with as many 32 KiB stages as fit
// (seven): measured on GB300 with the dynamic work split, 2-3.5 % faster than two CTAs of three
// stages on the 128 MiB copies and round trips and 1 % on the 3.2 GB reduce-add.
constexpr uint64_t kStreamCtasPerSm = 1;

// Stages of the streaming reductions (tensor loads of src, bulk reduce-adds into dst).  They read
// two tensors and write one, and keep more DRAM traffic in flight per stage than a copy: measured
// on GB300, four stages run the 3.2 GB fp32 reduce-add 0.8 % faster than seven (6895-6906 against
// 6845-6849 GB/s, three interleaved runs each; bf16 add likewise), while the copies lose 1.5 % at four.
constexpr uint64_t kStreamReduceStages = 4;

// Launch shape for boxes far smaller than a stage (image slots of at most kSmallSlotBytes, 16 or
// more to a stage).  Their elected lane issues one copy instruction per box in each direction, and
// its issue rate, not the DRAM, bounds them: more CTAs per SM (more issuing lanes), smaller stages,
// and the static split, whose items need no index decomposition.  Measured on GB300 on W3 through
// 64 x 4 boxes (512-byte images, 1 KiB slots): 5497-5544 GB/s with 4 CTAs of 16 KiB stages and the
// static split, 5206 with the dynamic split, 4726-4794 with 2 CTAs of 32 KiB, 5133-5196 with 6-12
// CTAs, 2188 with the one CTA of 32 KiB stages that larger boxes take.
constexpr uint64_t kSmallSlotBytes = 1024;
constexpr uint64_t kSmallGroupBytes = 16384;
constexpr uint64_t kSmallCtasPerSm = 4;

inline bool stream_small(const StreamArgs& a)
{
    return a.group > 1 && a.slot_bytes <= kSmallSlotBytes;
}

// Fills the schedule fields of a streaming launch over `grid` CTAs (walk and group already set).
inline void stream_schedule(StreamArgs& a, uint32_t grid)
{
    const uint64_t wave = (uint64_t)grid * a.group;
    a.waves = a.walk.nbox / wave;
    a.tail0 = a.waves * wave;
    const uint64_t rest = a.walk.nbox - a.tail0;
    a.tail_q = (uint32_t)(rest / grid);
    a.tail_r = (uint32_t)(rest % grid);
    uint64_t b = wave;
    for (uint32_t i = 0; i < 5; i++) {
        if (i < a.walk.rank) {
            a.dstep[i] = (uint32_t)(b % a.walk.grid_nb[i]);
            b /= a.walk.grid_nb[i];
        } else {
            a.dstep[i] = 0;
        }
    }
}

// Items (stages' worth of boxes) CTA c handles: the full waves, plus one if it has tail boxes.
TM_HD inline uint64_t stream_items(const StreamArgs& a, uint32_t c)
{
    return a.waves + ((a.tail_q > 0 || c < a.tail_r) ? 1u : 0u);
}

// First box and box count of item i of CTA c in a grid of `grid` CTAs.
TM_HD inline void stream_item(const StreamArgs& a, uint32_t c, uint32_t grid, uint64_t i,
                              uint64_t& b0, uint32_t& cnt)
{
    if (i < a.waves) {
        b0 = (i * grid + c) * a.group;
        cnt = a.group;
    } else {
        b0 = a.tail0 + (uint64_t)c * a.tail_q + (c < a.tail_r ? c : a.tail_r);
        cnt = a.tail_q + (c < a.tail_r ? 1u : 0u);
    }
}

// Dynamic split (a.sched set): CTA c of `grid` first takes items c, c + grid, ... for its first
// stages + 1 items (the static prefix, `prefix` = (stages + 1) * grid items in all), then fetches
// p = 0, 1, ... from the counter: fetch p covers items first .. first + count - 1 (clipped to
// nitems; a fetch past the items ends the CTA's work).  The first `batched` fetches take `batch`
// items each, later ones a single item.
TM_HD inline void dyn_fetch(const StreamArgs& a, uint64_t prefix, uint64_t p, uint64_t& first,
                            uint64_t& count)
{
    const uint64_t B = a.batch ? a.batch : 1u;
    if (p < a.batched) {
        first = prefix + p * B;
        count = B;
    } else {
        first = prefix + a.batched * B + (p - a.batched);
        count = 1;
    }
}

// Fills `batched` for a launch of `grid` CTAs: whole batches until about taper_per_cta x grid items
// are left, then single items (with several items a fetch, a CTA could otherwise hold a whole batch
// more than another when the items run out).
inline void dyn_taper(StreamArgs& a, uint32_t grid, uint64_t taper_per_cta)
{
    const uint64_t prefix = (uint64_t)(a.stages + 1) * grid;
    const uint64_t rest = a.nitems > prefix ? a.nitems - prefix : 0;
    const uint64_t single = rest < (uint64_t)grid * taper_per_cta ? rest : (uint64_t)grid * taper_per_cta;
    a.batched = a.batch > 1 ? (rest - single) / a.batch : 0;
}

// Generic fallback kernels.
struct FbArgs {
    BoxWalk walk;
    uint64_t base;         // tensor (destination for store / reduce) base address
    uint64_t src_base;     // reduce: source tensor base
    uint64_t dim[5];
    int64_t stride[5];     // bytes, destination / tensor
    int64_t src_stride[5]; // bytes, reduce source
    uint64_t images;
    uint32_t esize;
    uint32_t span;         // swizzle span in bytes, 0 = none
    uint32_t inner_bytes;  // image row: ibox[0] * esize
    uint32_t box_bytes;
    uint32_t stage_bytes;
    uint32_t rows;         // image rows = box_bytes / inner_bytes
    uint32_t block_rows;   // image rows handled per block (shared-memory row table / staging)
    uint16_t red_type;     // reduce: 0 f32, 1 f16, 2 bf16, 3 u32, 4 s32
    uint16_t red_op;       // reduce: 0 add, 1 min, 2 max
    uint32_t gspan0;       // box[0] * esize: bytes of the tensor row under one image row
    uint32_t fill_nan;     // 1: out-of-bounds image elements are `fill`; 0: zero bytes
    uint64_t fill;         // out-of-bounds element bit pattern (low esize bytes)
    uint32_t ibox[5];      // image extents ceil(box[i] / estride[i]) (unused dims 1)
    uint32_t estride[5];   // elementStrides (unused dims 1)
    uint64_t timeout_ns;
    StatusBlock* status;
};

// Boxes per stage of the TMA streaming kernels and the stage bytes each takes: small boxes share a
// stage of about `target` bytes, each in a slot starting on its swizzle period (the hardware
// swizzles on shared-memory address bits 4..9: 1024 / 512 / 256 bytes for a 128 / 64 / 32-byte
// span; 128 bytes, the tensor copy's alignment, without), so that every image keeps the phase it
// has in its own image.  (One box per 1 KiB stage was measured on GB300 at 1 TB/s for 512-byte
// boxes, against 5.5 TB/s for packed 2 KiB boxes.)
inline uint64_t slot_of(uint64_t box_bytes, uint32_t span)
{
    const uint64_t period = span == 128 ? 1024 : span == 64 ? 512 : span == 32 ? 256 : 128;
    return (box_bytes + period - 1) / period * period;
}

inline void tma_group(uint64_t box_bytes, uint32_t span, uint64_t target, uint32_t& group,
                      uint32_t& slot)
{
    const uint64_t sl = slot_of(box_bytes, span);
    const uint64_t g = target / sl;
    group = (uint32_t)(g < 1 ? 1 : g > 64 ? 64 : g);
    slot = group > 1 ? (uint32_t)sl : (uint32_t)box_bytes;
}

// Launch plan of a TMA streaming kernel over the boxes of a.walk, shared by every entry point that
// launches one: boxes per stage (tma_group, stages of about TM_GROUP_BYTES = 32 KiB, 16 KiB for
// small slots), CTAs per SM (TM_CTAS_PER_SM, default kStreamCtasPerSm, kSmallCtasPerSm for small
// slots; fewer when two stages would not fit), as many stages as fit
// (at most TM_STAGES when set; a reduction at most TM_STAGES_REDUCE, default kStreamReduceStages),
// the grid, the schedule and the dynamic shared memory.  budget(n) is the shared memory one of n
// CTAs on an SM may use.
template <class Budget>
inline void stream_plan(StreamArgs& a, uint64_t box_bytes, uint32_t span, uint32_t sms,
                        Budget budget, uint32_t& grid, size_t& smem, bool reduce = false)
{
    a.box_bytes = (uint32_t)box_bytes;
    const bool small = slot_of(box_bytes, span) <= kSmallSlotBytes;
    tma_group(box_bytes, span,
              std::max<uint64_t>(env_u64("TM_GROUP_BYTES", small ? kSmallGroupBytes : 32768), 1024),
              a.group, a.slot_bytes);
    const uint64_t stage = (uint64_t)a.group * a.slot_bytes;
    a.stage_bytes = (uint32_t)((stage + kStageAlign - 1) / kStageAlign * kStageAlign);
    uint32_t per_sm = (uint32_t)std::min<uint64_t>(
        std::max<uint64_t>(env_u64("TM_CTAS_PER_SM", small ? kSmallCtasPerSm : kStreamCtasPerSm), 1), 16);
    size_t b = budget(per_sm);
    while (per_sm > 1 && b < 2ull * a.stage_bytes) b = budget(--per_sm);
    uint32_t stages = (uint32_t)std::min<size_t>(b / a.stage_bytes, TM_MAX_STAGES);
    const uint64_t cap = reduce ? env_u64("TM_STAGES_REDUCE", kStreamReduceStages) : env_u64("TM_STAGES", 0);
    if (cap > 0) stages = (uint32_t)std::min<uint64_t>(stages, cap);
    a.stages = std::max<uint32_t>(stages, 1);
    const uint64_t units = (a.walk.nbox + a.group - 1) / a.group;
    grid = (uint32_t)std::min<uint64_t>(units, (uint64_t)sms * per_sm);
    stream_schedule(a, grid);
    a.nitems = units;
    a.sched = nullptr;  // the static schedule unless the caller hands the launch a counter
    a.batch = 1;        // items per fetch of the dynamic split (the caller may raise it)
    a.batched = 0;
    smem = (size_t)a.stages * a.stage_bytes + kStageAlign;
}

// NaN written for out-of-bounds elements of a map with TM_OOB_NAN on the vector path: the pattern
// GB300's tensor-map NaN-request fill was measured to write, 0x7FF7 repeated over the element.
inline uint64_t nan_fill_bits(uint32_t dtype)
{
    switch (dtype) {
        case TM_F16: case TM_BF16: return 0x7ff7ull;
        case TM_F32: return 0x7ff77ff7ull;
        case TM_F64: return 0x7ff77ff77ff77ff7ull;
        default: return 0;
    }
}

// Whether every elementStride of the map is 1.
inline bool unit_steps(const tm_desc* d)
{
    for (uint32_t i = 0; i < d->rank; i++)
        if (d->estride[i] != 1) return false;
    return true;
}

// The map's part of the vector kernels' arguments (tensor, image shape, fill).
inline void fb_from_desc(FbArgs& a, const tm_desc* d)
{
    a.base = d->base;
    for (int i = 0; i < 5; i++) {
        a.dim[i] = d->dim[i];
        a.stride[i] = (int64_t)d->stride[i];
        a.estride[i] = d->estride[i] ? d->estride[i] : 1u;
        a.ibox[i] = (d->box[i] + a.estride[i] - 1) / a.estride[i];
    }
    a.esize = d->esize;
    a.span = d->swizzle == TM_SWIZZLE_128B ? 128u : d->swizzle == TM_SWIZZLE_64B ? 64u
             : d->swizzle == TM_SWIZZLE_32B ? 32u : 0u;
    a.inner_bytes = a.ibox[0] * d->esize;
    a.gspan0 = d->box[0] * d->esize;
    a.box_bytes = (uint32_t)d->box_bytes;
    a.rows = (uint32_t)(d->box_bytes / a.inner_bytes);
    a.fill_nan = d->oob == TM_OOB_NAN ? 1u : 0u;
    a.fill = d->oob == TM_OOB_NAN ? nan_fill_bits(d->dtype) : 0ull;
}

// Shared memory per image row: the staged copy keeps the aligned 16-byte windows under the
// tensor row segment of `gspan0` bytes (one more window than 16-byte units) and the row's offset;
// the store keeps the offset only.
inline size_t fb_copy_row_bytes(uint32_t gspan0) { return (size_t)(gspan0 / 16 + 1) * 16 + 8; }
constexpr size_t kFbStoreRowBytes = 8;

// Launch shape of a vector kernel that handles image rows in blocks: the most CTAs per SM up to
// `want` (fewer when a block of 32 rows, or the whole box, would not fit), the fewest row blocks
// per box that fit, rows spread evenly over them (320 rows in 146-row blocks become 3 x 107, not
// 146 + 146 + 28), grid and dynamic shared memory.  budget(n) is the shared memory one of n CTAs
// on an SM may use.  (Splitting boxes into more blocks than needed, to shorten the last round of
// items, measured slower on GB300: the DRAM stays busy through a partial last round, while every
// block costs barriers.)
template <class Budget>
inline void fb_shape(FbArgs& a, uint64_t nbox, uint32_t sms, uint32_t want, size_t row_bytes,
                     Budget budget, uint32_t& grid, size_t& smem)
{
    const uint32_t min_rows = a.rows < 32 ? a.rows : 32;
    uint32_t per_sm = want < 1 ? 1 : want;
    while (per_sm > 1 && budget(per_sm) / row_bytes < min_rows) per_sm--;
    size_t fit = budget(per_sm) / row_bytes;
    fit = fit < 1 ? 1 : fit;
    const size_t nblk = (a.rows + fit - 1) / fit;
    a.block_rows = (uint32_t)((a.rows + nblk - 1) / nblk);
    smem = (size_t)a.block_rows * row_bytes;
    const uint64_t ctas = (uint64_t)sms * per_sm;
    const uint64_t items = nbox * ((a.rows + a.block_rows - 1) / a.block_rows);
    grid = (uint32_t)(items < ctas ? items : ctas);
}

// Segment form of the vector path (grid walks with unit elementStrides): the boxes along dim 0
// of one block of image rows are handled together as a run, which covers whole tensor rows; when
// dim 1 is contiguous with dim 0 (stride[1] == dim[0] * esize) the ibox[1] image rows of a box
// lie back to back in memory and form one segment.  The copy stages each segment by one 1-D bulk
// copy; the store stages each box's block of image rows by one.
struct SegArgs {
    FbArgs f;
    uint64_t nrun;          // runs = boxes / run
    uint32_t run;           // boxes per run: the grid's boxes along dim 0
    uint32_t seg_rows;      // image rows per segment: ibox[1] (dims 0 and 1 contiguous) or 1
    uint32_t outer0;        // first dim indexed per segment: 2 or 1
    uint32_t groups;        // segments per box = rows / seg_rows
    uint32_t block_groups;  // segments per item (one row block of a run)
    uint32_t nblk;          // items per run
    uint32_t seg_stride;    // shared-memory bytes per staged segment
    uint32_t row_bytes;     // dim[0] * esize: tensor bytes of one row
    uint32_t img_stride;    // store: shared-memory bytes per box image block of an item
    uint32_t stages;        // staging buffers (items in flight per CTA)
    uint64_t per;           // items per CTA: items / grid (CTAs below `extra` take one more),
    uint32_t extra;         // computed on the host with the grid
    uint32_t cwarps;        // consumer warps per CTA: 8, 12 or 16 (TM_FB_SEG_WARPS, default kSegWarps)
    // Dynamic item split (when sched is set; see SegSource in k_fb_seg.cu): a counter of the
    // launch's stream, zero at launch, reset by the launch's last CTA; batch items per fetch.
    unsigned long long* sched;
    uint64_t nitems;        // items of the launch: nrun * nblk
    uint32_t batch;
    uint32_t pad;
};
constexpr uint32_t kSegMinBytes = 512;  // shorter segments: the per-window copy (request rate)
constexpr uint32_t kSegMaxGroups = 64;
constexpr uint32_t kSegMaxStages = 8;

// The segment form's plan for a copy (load direction) over the whole grid, or false when the
// map does not take it: segments of ibox[1] rows when dims 0 and 1 are contiguous and such a
// segment fits, else of one row.  force: 1 = whenever the layout allows (any segment length),
// 0 = never, other = when segments are at least kSegMinBytes.  budget(n) as for fb_shape.
// Copy: a stage holds an item's segments (seg_stride bytes each) and a 4-byte shared-memory
// offset per image row.  Store (store = true): a stage holds the item's image block of each box of
// the run (img_stride bytes each) and an 8-byte tensor address per image row.
// Launch shape of the segment kernels: CTAs per SM, staging buffers of the copy and of the store,
// consumer warps.  Measured on GB300 on the W4 rank-5 view with the dynamic item split: two CTAs
// of eight warps and two buffers gave copy 5349-5362, store 5235-5240 GB/s; three buffers for the
// copy and twelve warps, 5542-5618 and 5215-5405; three CTAs of eight warps with three buffers
// each, 5583-5725 and 5430-5565 (five rounds against the previous shape on two boxes).  One CTA
// per SM lost 7-25 %; more CTAs than the SM can hold (three of twelve warps: their registers allow
// two) lost a quarter, which seg_fit keeps from happening.
constexpr uint64_t kSegCtasPerSm = 3;
constexpr uint64_t kSegCopyStages = 3;
constexpr uint64_t kSegStoreStages = 3;
constexpr uint64_t kSegWarps = 8;

template <class Budget>
inline bool seg_plan_rows(const FbArgs& a, uint64_t g1, uint32_t sms, uint32_t want,
                          uint32_t stages, int force, bool store, Budget budget, SegArgs& s,
                          uint32_t& grid, size_t& smem)
{
    const uint64_t row_bytes = a.dim[0] * a.esize;
    const uint64_t seg_max = g1 * row_bytes;
    if (force != 1 && seg_max < kSegMinBytes) return false;
    if (seg_max > (1u << 20)) return false;
    const uint64_t nb0 = a.walk.grid_nb[0];
    const uint64_t seg_stride = (seg_max + 48 + 15) / 16 * 16;
    const uint64_t S = std::min<uint32_t>(std::max<uint32_t>(stages, 2), kSegMaxStages);
    const uint64_t per_group =
        store ? S * (nb0 * g1 * a.inner_bytes + 8 * g1) : S * (seg_stride + 4 * g1);
    const uint64_t fixed = 64;
    uint32_t per_sm = want < 1 ? 1 : want;
    while (per_sm > 1 && budget(per_sm) < fixed + per_group) per_sm--;
    if (budget(per_sm) < fixed + per_group) return false;
    const uint64_t groups = a.rows / g1;
    uint64_t e = (budget(per_sm) - fixed) / per_group;
    e = std::min<uint64_t>(std::min<uint64_t>(e, groups), kSegMaxGroups);
    s.stages = (uint32_t)S;
    s.f = a;
    s.run = (uint32_t)nb0;
    s.seg_rows = (uint32_t)g1;
    s.outer0 = g1 > 1 ? 2u : 1u;
    s.groups = (uint32_t)groups;
    s.row_bytes = (uint32_t)row_bytes;
    s.seg_stride = store ? 0u : (uint32_t)seg_stride;
    s.nblk = (uint32_t)((groups + e - 1) / e);
    s.block_groups = (s.groups + s.nblk - 1) / s.nblk;
    s.img_stride = store ? (uint32_t)((uint64_t)s.block_groups * g1 * a.inner_bytes) : 0u;
    s.nrun = a.walk.nbox / nb0;
    const uint64_t items = s.nrun * s.nblk;
    const uint64_t ctas = (uint64_t)sms * per_sm;
    grid = (uint32_t)(items < ctas ? items : ctas);
    s.per = items / grid;
    s.extra = (uint32_t)(items % grid);
    s.nitems = items;
    s.sched = nullptr;  // the static split unless the caller hands the launch a counter
    s.batch = 1;
    const uint64_t w = env_u64("TM_FB_SEG_WARPS", kSegWarps);
    s.cwarps = w >= 16 ? 16u : w >= 12 ? 12u : 8u;
    smem = store ? (size_t)S * ((size_t)nb0 * s.img_stride + 8ull * s.block_groups * g1) + 16
                 : (size_t)S * s.block_groups * (s.seg_stride + 4 * g1) + 16;
    return true;
}

template <class Budget>
inline bool seg_plan(const FbArgs& a, const tm_desc* d, uint32_t sms, uint32_t want,
                     uint32_t stages, int force, bool store, Budget budget, SegArgs& s,
                     uint32_t& grid, size_t& smem)
{
    if (force == 0 || a.walk.mode != WALK_GRID || d->rank < 2 || !unit_steps(d)) return false;
    if (store && force != 1) {
        // Rows that all start on 16 bytes store faster through the per-window kernel (its 16-byte
        // image loads go straight to aligned 16-byte stores; measured on GB300 with W3 on the
        // vector path: 49.8 against 53.9 us); the segment store pays off on unaligned rows.
        bool aligned = a.base % 16 == 0;
        for (uint32_t i = 1; i < d->rank; i++) aligned = aligned && a.stride[i] % 16 == 0;
        if (aligned) return false;
    }
    const bool fused = a.stride[1] == (int64_t)(a.dim[0] * a.esize);
    if (fused && a.ibox[1] > 1 &&
        seg_plan_rows(a, a.ibox[1], sms, want, stages, force, store, budget, s, grid, smem))
        return true;
    return seg_plan_rows(a, 1, sms, want, stages, force, store, budget, s, grid, smem);
}

// Launch shape of the vector path's copy (load direction), shared by every entry point that
// launches one: the segment form when the map takes it (TM_FB_SEG: 0 never, 1 whenever the layout
// allows, unset when its segments are long enough for bulk copies; TM_FB_SEG_CTAS_PER_SM and
// TM_FB_SEG_STAGES, defaults kSegCtasPerSm and kSegCopyStages, at most cap_per_sm CTAs per SM),
// else the per-window form (TM_FB_COPY_CTAS_PER_SM, default 8).  Returns true for the
// segment form (s filled), false for the per-window form (a.block_rows set).  budget(n) as for
// fb_shape.
template <class Budget>
inline bool fb_copy_plan(FbArgs& a, const tm_desc* d, uint64_t nbox, uint32_t sms, Budget budget,
                         SegArgs& s, uint32_t& grid, size_t& smem, uint64_t cap_per_sm = 8)
{
    const uint64_t want = std::min<uint64_t>(env_u64("TM_FB_SEG_CTAS_PER_SM", kSegCtasPerSm), cap_per_sm);
    if (seg_plan(a, d, sms, (uint32_t)std::max<uint64_t>(std::min<uint64_t>(want, 8), 1),
                 (uint32_t)std::min<uint64_t>(env_u64("TM_FB_SEG_STAGES", kSegCopyStages), kSegMaxStages),
                 (int)env_u64("TM_FB_SEG", 2), false, budget, s, grid, smem))
        return true;
    fb_shape(a, nbox, sms, (uint32_t)std::min<uint64_t>(env_u64("TM_FB_COPY_CTAS_PER_SM", 8), 16),
             fb_copy_row_bytes(a.gspan0), budget, grid, smem);
    return false;
}

// A segment launch whose CTAs the SMs hold all at once: plan(cap) plans it with at most cap CTAs
// per SM and returns false when the segment form does not apply.  seg_plan sizes a CTA's shared
// memory only, and the kernel's registers can allow fewer CTAs per SM than planned (three CTAs of
// twelve consumer warps: two); CTAs beyond what the SMs hold would run as a second, short wave.
// So the planned launch goes to the occupancy calculator and is planned again with its answer.
int seg_resident_ctas(bool store, uint32_t cwarps, size_t smem);  // k_fb_seg.cu

template <class Plan>
inline bool seg_fit(bool store, uint32_t sms, const SegArgs& s, const uint32_t& grid,
                    const size_t& smem, Plan plan)
{
    if (!plan(8)) return false;
    const int fit = seg_resident_ctas(store, s.cwarps, smem);
    if (fit > 0 && (uint64_t)grid > (uint64_t)sms * (uint64_t)fit) return plan((uint64_t)fit);
    return true;
}

// Ring consumer (stream_tiles).
struct RingArgs {
    uint64_t ntiles;
    uint64_t a_nb0, b_nb0;   // boxes along dim 0 of A and B
    uint32_t rows;           // tile rows R (box[1]); rows are 128 bytes
    uint32_t stages;
    uint32_t tile_bytes;     // R * 128
    uint32_t swizzled;       // 1 = 128B, 0 = none
    uint32_t prefetch;       // tiles ahead of the ring prefetched into L2 (0 = none)
    uint32_t groups;         // consumer groups (1, or 2 when stages is even)
    uint32_t row_pairs;      // 1: lanes read rows two apart (the ungrouped 256-byte-row control)
    uint32_t evict_first;    // 1: tile loads carry an L2 evict-first policy (each tile is read once)
    float* cs_a;
    float* cs_b;
    unsigned long long* bits_a;
    unsigned long long* bits_b;
    uint64_t timeout_ns;
    StatusBlock* status;
    // The launch-wide schedule over `grid` CTAs, computed once on the host (ring_schedule).
    uint64_t n_base;         // tiles per CTA: ntiles / grid (CTAs below n_rem take one more)
    uint64_t a_d1, b_d1;     // grid / a_nb0, grid / b_nb0: a CTA's step in rows of boxes ...
    uint32_t a_d0, b_d0;     // ... and grid % a_nb0, grid % b_nb0 in boxes along dim 0
    uint32_t n_rem;
    uint32_t pad2;
};

inline void ring_schedule(RingArgs& r, uint32_t grid)
{
    r.n_base = r.ntiles / grid;
    r.n_rem = (uint32_t)(r.ntiles % grid);
    r.a_d0 = (uint32_t)(grid % r.a_nb0);
    r.a_d1 = grid / r.a_nb0;
    r.b_d0 = (uint32_t)(grid % r.b_nb0);
    r.b_d1 = grid / r.b_nb0;
}

// Tensor-core consumer of the k-ordered ring (stream_gemm): C = A * B^T.
constexpr uint32_t kGemmMaxStages = 4;      // one-SM form: 48 KiB stages
constexpr uint32_t kGemmMaxPairStages = 7;  // CTA-pair form: 32 KiB stages per CTA
struct GemmArgs {
    uint32_t m, n, k;        // C is m x n; A is m x k, B is n x k (bf16, k contiguous)
    uint32_t mtiles, ntiles; // 128-row and 256-column tiles of C
    uint32_t kblocks;        // 64-wide steps along k
    uint32_t stages;         // 2..kGemmMaxStages
    uint32_t split_from;     // pair form: tiles from here on are done as two 256 x 128 halves
    float* c;                // fp32, row-major
    uint64_t ldc;            // elements between rows of C
    uint64_t timeout_ns;
    StatusBlock* status;
};

// Launchers (defined next to their kernels).  Return a cudaError_t.
// Reduce kinds: KIND_REDUCE + op, op 0 add, 1 min, 2 max.
enum StreamKind : int {
    KIND_COPY = 0, KIND_ROUNDTRIP = 1, KIND_REDUCE = 2, KIND_REDUCE_MIN = 3, KIND_REDUCE_MAX = 4
};
cudaError_t launch_tma_stream(int kind, uint32_t rank, const CUtensorMap* in_map,
                              const CUtensorMap* out_map, const StreamArgs& a, uint32_t grid,
                              size_t smem, cudaStream_t s);
cudaError_t launch_fb_copy(const FbArgs& a, uint32_t grid, size_t smem, cudaStream_t s);
cudaError_t launch_fb_store(const FbArgs& a, uint32_t grid, size_t smem, cudaStream_t s);
cudaError_t launch_fb_reduce(const FbArgs& a, uint32_t grid, cudaStream_t s);
cudaError_t launch_fb_seg_copy(const SegArgs& a, uint32_t grid, size_t smem, cudaStream_t s);
cudaError_t launch_fb_seg_store(const SegArgs& a, uint32_t grid, size_t smem, cudaStream_t s);
cudaError_t launch_ring(const CUtensorMap* a, const CUtensorMap* b, const RingArgs& r,
                        uint32_t grid, size_t smem, cudaStream_t s);
cudaError_t launch_selftest(uint64_t timeout_ns, StatusBlock* status, cudaStream_t s);
cudaError_t launch_gemm(const CUtensorMap* a, const CUtensorMap* b, const GemmArgs& g,
                        uint32_t grid, size_t smem, cudaStream_t s);
cudaError_t launch_gemm_pair(const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* b_quarter,
                             const GemmArgs& g,
                             uint32_t grid, size_t smem, cudaStream_t s);

// Sets the thread's tm_last_error() text; returns `code`.
int set_last_error(int code, const char* msg);

}  // namespace tmk
