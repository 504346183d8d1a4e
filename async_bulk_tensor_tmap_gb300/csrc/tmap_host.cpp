// tmap_host.cpp -- the C ABI of include/tmap.h: descriptor validation and encoding, path
// selection, launch geometry, coordinate staging and the per-device status word.
//
// [MLSys-TMA] mlc.ai "Modern GPU Programming for MLSys", chapter "异步数据搬运：TMA"
// [H200-TMA]  coolgpu "H200 · TMA · Tensor Memory Accelerator" feature card
// [Book-TMA]  fangpin "gpu-hpc-book", chapter 08 "Cuda TMA （Tensor Memory Accelerator）"
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tm_internal.h"
#include "tmap.h"

using namespace tmk;

static_assert(sizeof(tm_desc) == 384, "tm_desc is 384 bytes");
static_assert(alignof(tm_desc) == 64, "tm_desc is 64-byte aligned");
static_assert(offsetof(tm_desc, base) == 32, "tm_desc layout");
static_assert(offsetof(tm_desc, box) == 120, "tm_desc layout");
static_assert(offsetof(tm_desc, nbox) == 160, "tm_desc layout");
static_assert(offsetof(tm_desc, box_bytes) == 200, "tm_desc layout");
static_assert(offsetof(tm_desc, tmap) == 256, "tm_desc layout");
static_assert(offsetof(tm_desc, l2_promotion) == 216, "tm_desc layout");
static_assert(sizeof(CUtensorMap) == 128, "CUtensorMap is 128 bytes");

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what)
{
    return fail(TM_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

uint32_t esize_of(int dt)
{
    switch (dt) {
        case TM_U8: return 1;
        case TM_U16: case TM_F16: case TM_BF16: return 2;
        case TM_U32: case TM_S32: case TM_F32: return 4;
        case TM_U64: case TM_S64: case TM_F64: return 8;
        default: return 0;
    }
}

uint32_t span_of(uint32_t sw)
{
    return sw == TM_SWIZZLE_128B ? 128u : sw == TM_SWIZZLE_64B ? 64u : sw == TM_SWIZZLE_32B ? 32u : 0u;
}

bool valid_desc(const tm_desc* d) { return d && d->magic == TM_DESC_MAGIC; }

// ---- driver entry points (no link-time dependency on libcuda) ---------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
using ReplaceAddressFn = CUresult (*)(CUtensorMap*, void*);

void* driver_symbol(const char* name)
{
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return p;
}

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] { fn = (EncodeTiledFn)driver_symbol("cuTensorMapEncodeTiled"); });
    return fn;
}

ReplaceAddressFn replace_fn()
{
    static std::once_flag once;
    static ReplaceAddressFn fn = nullptr;
    std::call_once(once, [] { fn = (ReplaceAddressFn)driver_symbol("cuTensorMapReplaceAddress"); });
    return fn;
}

// ---- per-device state ---------------------------------------------------------------------------
// Counters of the streaming kernels' dynamic work split: one per stream, never reassigned to
// another stream (a stream's launches run in order, so they can share one; launches on different
// streams may overlap, so they must not).  Each slot has its own 128-byte line.
constexpr uint32_t kSchedSlots = 256;
constexpr uint64_t kReduceBatch = 4;
// Items per CTA handed out singly at the end of a batched launch.  Measured on GB300 (two runs):
// four took the fp32 reduce-add from 6894-6900 to 6925-6935 GB/s, bf16 add from 6740-6752 to
// 6786-6791 and s32 min from 6904-6905 to 6937-6938; two and eight gained 0.1-0.2 %.
constexpr uint64_t kTaperPerCta = 4;
constexpr size_t kSchedSlotBytes = 128;

struct DevState {
    bool ready = false;
    int sms = 0;
    int smem_per_sm = 0;
    int smem_optin = 0;
    StatusBlock* status = nullptr;
    unsigned char* sched = nullptr;          // kSchedSlots counter slots, zero between launches
    unsigned long long sched_stream[kSchedSlots] = {};  // stream id of each slot (0: free)
    uint32_t sched_used = 0;
};

std::mutex g_mu;
DevState g_dev[64];

int device_state(DevState** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(TM_EUNSUPPORTED, "device ordinal %d above 63", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DevState& d = g_dev[dev];
    if (!d.ready) {
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) ||
            (e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                        dev)) ||
            (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                        dev)))
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if ((e = cudaMalloc((void**)&d.status, sizeof(StatusBlock))) != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(status word)");
        if ((e = cudaMemset(d.status, 0, sizeof(StatusBlock))) != cudaSuccess)
            return cuda_fail(e, "cudaMemset(status word)");
        if ((e = cudaMalloc((void**)&d.sched, kSchedSlots * kSchedSlotBytes)) != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(work counters)");
        if ((e = cudaMemset(d.sched, 0, kSchedSlots * kSchedSlotBytes)) != cudaSuccess)
            return cuda_fail(e, "cudaMemset(work counters)");
        d.ready = true;
    }
    *out = &d;
    return TM_OK;
}

uint64_t wait_limit_ns() { return env_u64("TM_WAIT_TIMEOUT_NS", 1000000000ull); }

// The work counter of `stream` for a streaming launch, or nullptr for the static split: while the
// stream is being captured into a graph (a graph may later run beside direct launches on the
// stream), when every slot belongs to another stream, or with TM_DYNAMIC=0.
unsigned long long* sched_slot(DevState& ds, cudaStream_t stream)
{
    if (env_u64("TM_DYNAMIC", 1) == 0) return nullptr;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (cs != cudaStreamCaptureStatusNone) return nullptr;
    unsigned long long id = 0;
    if (cudaStreamGetId(stream, &id) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    id += 1;  // 0 marks a free slot
    std::lock_guard<std::mutex> lk(g_mu);
    for (uint32_t i = 0; i < ds.sched_used; i++)
        if (ds.sched_stream[i] == id)
            return reinterpret_cast<unsigned long long*>(ds.sched + (size_t)i * kSchedSlotBytes);
    if (ds.sched_used == kSchedSlots) return nullptr;
    const uint32_t i = ds.sched_used++;
    ds.sched_stream[i] = id;
    return reinterpret_cast<unsigned long long*>(ds.sched + (size_t)i * kSchedSlotBytes);
}

// ---- launch geometry ------------------------------------------------------------------------
// Shared memory a CTA may use when `per_sm` CTAs share an SM (1 KiB per CTA is reserved by the
// hardware; 1 KiB more lets the kernel align its stages to 1024 bytes; 256 bytes of barriers).
size_t cta_budget(const DevState& ds, uint32_t per_sm)
{
    const size_t share = (size_t)ds.smem_per_sm / per_sm;
    const size_t cap = std::min<size_t>((size_t)ds.smem_optin, share > 1024 ? share - 1024 : 0);
    return cap > 2048 + 256 ? cap - 1024 - 256 : 0;
}

uint32_t stage_bytes_of(uint64_t box_bytes)
{
    return (uint32_t)((box_bytes + kStageAlign - 1) / kStageAlign * kStageAlign);
}

// ---- box lists --------------------------------------------------------------------------------
// Whether the TMA path may be given every box of an explicit list.  The tensor-map copies need the
// box's innermost start coordinate times the element size to be a multiple of 16 bytes.  Loads
// accept starts outside the tensor as long as part of the box is inside; stores and reduces are
// only given boxes that start inside the tensor.  Anything else runs on the fallback path, which
// gives the same bytes.
bool list_fits_tma(const tm_desc* d, const int32_t* coords, size_t n, bool store)
{
    for (size_t b = 0; b < n; b++) {
        const int32_t* c = coords + b * d->rank;
        if (((int64_t)c[0] * d->esize) % 16 != 0) return false;
        for (uint32_t i = 0; i < d->rank; i++) {
            const int64_t s = c[i];
            if (store && s < 0) return false;
            if (s >= (int64_t)d->dim[i] || s + (int64_t)d->box[i] <= 0) return false;
        }
    }
    return true;
}

// Fills the walk; a list longer than the inline capacity is copied to device memory allocated on
// `st` (freed by release_walk after the launch).
int make_walk(const tm_desc* d, const int32_t* coords, size_t n, cudaStream_t st, BoxWalk& w)
{
    memset(&w, 0, sizeof(w));
    w.nbox = coords ? n : d->num_boxes;
    w.rank = d->rank;
    for (int i = 0; i < 5; i++) {
        w.box[i] = d->box[i];
        w.grid_nb[i] = d->nbox[i];
    }
    if (!coords) {
        w.mode = WALK_GRID;
    } else if (n <= kInlineBoxes) {
        w.mode = WALK_INLINE;
        memcpy(w.inl, coords, n * d->rank * sizeof(int32_t));
    } else {
        w.mode = WALK_LIST;
        int32_t* dev = nullptr;
        const size_t bytes = n * d->rank * sizeof(int32_t);
        cudaError_t e = cudaMallocAsync((void**)&dev, bytes, st);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(box list)");
        e = cudaMemcpyAsync(dev, coords, bytes, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) {
            cudaFreeAsync(dev, st);
            return cuda_fail(e, "cudaMemcpyAsync(box list)");
        }
        w.list = dev;
    }
    return TM_OK;
}

// The tensor store and the tensor reduce write whole 16-byte units of the innermost dimension
// (measured on GB300: with globalDim[0] * esize not a multiple of 16, the out-of-bounds tail of
// the last unit of every row is overwritten with the image's zero fill).  Such maps store on the
// vector path, which writes exactly the in-bounds bytes.  So do maps with element strides: the
// pages define the strides for the load into shared memory only, and the vector path writes the
// image back to exactly the positions the load took.
bool store_fits_tma(const tm_desc* d)
{
    return d->path == TM_PATH_TMA && (d->dim[0] * d->esize) % 16 == 0 && unit_steps(d);
}

void release_walk(const BoxWalk& w, cudaStream_t st)
{
    if (w.mode == WALK_LIST && w.list) cudaFreeAsync((void*)w.list, st);
}

FbArgs fb_args(const tm_desc* d, const BoxWalk& w, uint64_t images, const DevState& ds)
{
    FbArgs a;
    memset(&a, 0, sizeof(a));
    a.walk = w;
    fb_from_desc(a, d);
    a.images = images;
    a.stage_bytes = stage_bytes_of(d->box_bytes);
    a.timeout_ns = wait_limit_ns();
    a.status = ds.status;
    return a;
}

// Arguments and launch geometry of a TMA streaming kernel over the walk's boxes.
struct Geometry {
    uint32_t grid;
    size_t smem;
};

// Items per fetch of the dynamic split.  Copies and round trips take one (measured on GB300 on
// the 128 MiB W3 / W4 maps: 2-4 % faster than the static split, with 2 or 4 a fetch no better
// than static).  Reductions take several: their counter sits in the L2 that also performs the
// bulk reductions, and one fetch per item cost the W5a reduce-add 15 % (four: +3 % over static).
uint32_t fetch_batch(bool reduce)
{
    const uint64_t b = reduce ? env_u64("TM_DYN_BATCH_REDUCE", kReduceBatch) : env_u64("TM_DYN_BATCH", 1);
    return (uint32_t)std::min<uint64_t>(std::max<uint64_t>(b, 1), 64);
}

StreamArgs stream_args(const tm_desc* d, const BoxWalk& w, uint64_t images, DevState& ds,
                       Geometry& g, cudaStream_t stream, bool reduce)
{
    StreamArgs a;
    memset(&a, 0, sizeof(a));
    a.walk = w;
    a.images = images;
    stream_plan(a, d->box_bytes, span_of(d->swizzle), (uint32_t)ds.sms,
                [&](uint32_t per_sm) { return cta_budget(ds, per_sm); }, g.grid, g.smem, reduce);
    a.sched = stream_small(a) ? nullptr : sched_slot(ds, stream);  // small boxes: static split
    a.batch = fetch_batch(reduce);
    // the last grid x kTaperPerCta items (TM_DYN_TAPER per CTA) go out one a fetch
    dyn_taper(a, g.grid, env_u64("TM_DYN_TAPER", kTaperPerCta));
    a.timeout_ns = wait_limit_ns();
    a.status = ds.status;
    return a;
}

int check_launch(cudaError_t e, const char* what)
{
    return e == cudaSuccess ? TM_OK : cuda_fail(e, what);
}

// Box copy in the load direction (tile_load_image, tiled_copy).
int copy_boxes(const tm_desc* src, const int32_t* coords, size_t nbox, void* images, void* stream)
{
    if (!valid_desc(src)) return fail(TM_EINVAL, "source descriptor is not filled");
    if (!coords && nbox != 0 && nbox != src->num_boxes)
        return fail(TM_EINVAL, "nbox %zu is neither 0 nor the grid's %llu boxes", nbox,
                    (unsigned long long)src->num_boxes);
    const uint64_t n = coords ? nbox : src->num_boxes;
    if (n == 0) return TM_OK;  // an empty box list moves nothing and needs no image buffer
    if (!images) return fail(TM_EINVAL, "images is NULL");
    if ((uintptr_t)images % 16) return fail(TM_EALIGN, "images must be 16-byte aligned");
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const bool tma = src->path == TM_PATH_TMA && (!coords || list_fits_tma(src, coords, n, false));
    BoxWalk w;
    if ((rc = make_walk(src, coords, n, st, w))) return rc;
    if (tma) {
        Geometry g;
        const StreamArgs a = stream_args(src, w, (uint64_t)images, *ds, g, st, false);
        const CUtensorMap* m = (const CUtensorMap*)src->tmap;
        rc = check_launch(launch_tma_stream(KIND_COPY, src->rank, m, m, a, g.grid, g.smem, st),
                          "tensor copy launch");
    } else {
        FbArgs a = fb_args(src, w, (uint64_t)images, *ds);
        uint32_t grid = 0;
        size_t smem = 0;
        SegArgs sa;
        const uint32_t sms = (uint32_t)ds->sms;
        auto budget = [&](uint32_t per_sm) { return cta_budget(*ds, per_sm); };
        if (seg_fit(false, sms, sa, grid, smem, [&](uint64_t cap) {
                return fb_copy_plan(a, src, n, sms, budget, sa, grid, smem, cap);
            })) {
            sa.sched = sched_slot(*ds, st);
            rc = check_launch(launch_fb_seg_copy(sa, grid, smem, st), "fallback segment copy launch");
        } else {
            rc = check_launch(launch_fb_copy(a, grid, smem, st), "fallback copy launch");
        }
    }
    release_walk(w, st);
    return rc;
}

int plan_impl(tm_desc* out, int dtype, uint32_t rank, void* base, const uint64_t* gdim,
              const uint64_t* gstr, const uint32_t* box, const uint32_t* estr, int sw, int oob)
{
    if (!out) return fail(TM_EINVAL, "descriptor pointer is NULL");
    memset(out, 0, sizeof(*out));
    const uint32_t es = esize_of(dtype);
    if (!es) return fail(TM_EINVAL, "unknown dtype %d", dtype);
    if (rank < 1 || rank > 5) return fail(TM_EINVAL, "rank %u outside 1..5", rank);
    if (!base) return fail(TM_EINVAL, "base is NULL");
    if (!gdim || !box || (rank > 1 && !gstr)) return fail(TM_EINVAL, "dims / strides / box NULL");
    if (sw < TM_SWIZZLE_NONE || sw > TM_SWIZZLE_128B) return fail(TM_EINVAL, "bad swizzle %d", sw);
    if (oob != TM_OOB_ZERO && oob != TM_OOB_NAN) return fail(TM_EINVAL, "bad oob fill %d", oob);
    if (oob == TM_OOB_NAN && dtype != TM_F16 && dtype != TM_BF16 && dtype != TM_F32 &&
        dtype != TM_F64)
        return fail(TM_EINVAL, "NaN out-of-bounds fill needs a floating-point dtype");
    uint32_t step[5] = {1, 1, 1, 1, 1};
    for (uint32_t i = 0; i < rank; i++) {
        if (gdim[i] < 1 || gdim[i] > (1ull << 32))
            return fail(TM_ERANGE, "globalDim[%u] = %llu outside 1..2^32", i,
                        (unsigned long long)gdim[i]);
        if (box[i] < 1 || box[i] > 256)
            return fail(TM_ERANGE, "boxDim[%u] = %u outside 1..256", i, box[i]);
        if (estr) {
            if (estr[i] < 1 || estr[i] > 8)
                return fail(TM_EINVAL, "elementStrides[%u] = %u outside 1..8", i, estr[i]);
            step[i] = estr[i];
        }
    }
    const uint64_t inner = (uint64_t)box[0] * es;
    if (inner % 16)
        return fail(TM_EALIGN, "boxDim[0] * element size = %llu bytes is not a multiple of 16",
                    (unsigned long long)inner);
    const uint64_t image_row = (uint64_t)((box[0] + step[0] - 1) / step[0]) * es;
    if (image_row % 16)
        return fail(TM_EALIGN, "the image row ceil(boxDim[0] / elementStrides[0]) * element size = "
                    "%llu bytes is not a multiple of 16", (unsigned long long)image_row);
    const uint32_t span = span_of((uint32_t)sw);
    if (span && step[0] != 1)
        return fail(TM_EUNSUPPORTED, "a swizzled map needs elementStrides[0] = 1");
    if (span && inner != span)
        return fail(TM_EUNSUPPORTED, "swizzle %u B needs an inner box row of exactly %u bytes, got %llu",
                    span, span, (unsigned long long)inner);
    uint64_t bb = es;
    for (uint32_t i = 0; i < rank; i++) bb *= (box[i] + step[i] - 1) / step[i];
    if (bb > TM_MAX_BOX_BYTES)
        return fail(TM_ERANGE, "box of %llu bytes exceeds %u", (unsigned long long)bb,
                    TM_MAX_BOX_BYTES);
    const uint64_t b = (uint64_t)(uintptr_t)base;
    if (b % es) return fail(TM_EALIGN, "base is not a multiple of the element size");
    uint32_t why = (b % 16) ? TM_WHY_BASE : 0u;
    if (step[0] != 1) why |= TM_WHY_STEP0;
    for (uint32_t i = 1; i < rank; i++) {
        const uint64_t s = gstr[i - 1];
        if (s == 0 || s >= (1ull << 40))
            return fail(TM_ERANGE, "globalStrides[%u] = %llu outside 1..2^40-1", i - 1,
                        (unsigned long long)s);
        if (s % es) return fail(TM_EALIGN, "globalStrides[%u] is not a multiple of the element size", i - 1);
        if (s % 16) why |= TM_WHY_STRIDE;
    }
    out->dtype = (uint32_t)dtype;
    out->esize = es;
    out->rank = rank;
    out->swizzle = (uint32_t)sw;
    out->oob = (uint32_t)oob;
    out->l2_promotion = (uint32_t)std::min<uint64_t>(env_u64("TM_L2_PROMOTION", TM_L2_128B), TM_L2_256B);
    out->path = why ? TM_PATH_FALLBACK : TM_PATH_TMA;
    out->why_fallback = why;
    out->base = b;
    uint64_t nb_total = 1;
    for (uint32_t i = 0; i < 5; i++) {
        const bool used = i < rank;
        out->dim[i] = used ? gdim[i] : 1;
        out->stride[i] = !used ? 0 : (i == 0 ? es : gstr[i - 1]);
        out->box[i] = used ? box[i] : 1;
        out->estride[i] = used ? step[i] : 1;
        out->nbox[i] = used ? (gdim[i] + box[i] - 1) / box[i] : 1;
        if (__builtin_mul_overflow(nb_total, out->nbox[i], &nb_total))
            return fail(TM_ERANGE, "box count overflows 64 bits");
    }
    out->box_bytes = bb;
    out->num_boxes = nb_total;
    out->magic = TM_DESC_MAGIC;
    return TM_OK;
}

int encode_into(tm_desc* d)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) {
        d->magic = 0;
        return fail(TM_ECUDA, "the CUDA driver's cuTensorMapEncodeTiled is not reachable");
    }
    cuuint64_t dims[5], strides[4];
    cuuint32_t boxd[5], estr[5];
    for (uint32_t i = 0; i < d->rank; i++) {
        dims[i] = d->dim[i];
        boxd[i] = d->box[i];
        estr[i] = d->estride[i];
        if (i > 0) strides[i - 1] = d->stride[i];
    }
    const CUtensorMapL2promotion promo = (CUtensorMapL2promotion)std::min<uint32_t>(d->l2_promotion, 3);
    const CUresult r = enc((CUtensorMap*)d->tmap, (CUtensorMapDataType)d->dtype, d->rank,
                           (void*)(uintptr_t)d->base, dims, strides, boxd, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, (CUtensorMapSwizzle)d->swizzle, promo,
                           d->oob == TM_OOB_NAN ? CU_TENSOR_MAP_FLOAT_OOB_FILL_NAN_REQUEST_ZERO_FMA
                                                : CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        memset(d->tmap, 0, sizeof(d->tmap));
        d->path = TM_PATH_FALLBACK;
        d->why_fallback |= TM_WHY_DRIVER;
    }
    return TM_OK;
}

}  // namespace

int tmk::set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }

extern "C" {

int tmap_plan(tm_desc* out, tm_dtype dtype, uint32_t rank, void* base, const uint64_t* globalDim,
              const uint64_t* globalStrides, const uint32_t* boxDim,
              const uint32_t* elementStrides, tm_swizzle swizzle, tm_oob oob)
{
    return plan_impl(out, dtype, rank, base, globalDim, globalStrides, boxDim, elementStrides,
                     swizzle, oob);
}

int tmap_encode(tm_desc* out, tm_dtype dtype, uint32_t rank, void* base,
                const uint64_t* globalDim, const uint64_t* globalStrides, const uint32_t* boxDim,
                const uint32_t* elementStrides, tm_swizzle swizzle, tm_oob oob)
{
    int rc = plan_impl(out, dtype, rank, base, globalDim, globalStrides, boxDim, elementStrides,
                       swizzle, oob);
    if (rc) return rc;
    if (out->path != TM_PATH_TMA) return TM_OK;
    return encode_into(out);
}

int tmap_replace_address(tm_desc* d, void* new_base)
{
    if (!valid_desc(d)) return fail(TM_EINVAL, "descriptor is not filled");
    const uint64_t nb = (uint64_t)(uintptr_t)new_base;
    if (!nb) return fail(TM_EINVAL, "new base is NULL");
    if (nb % d->esize) return fail(TM_EALIGN, "new base is not a multiple of the element size");
    const bool forced = (d->why_fallback & TM_WHY_FORCED) != 0;
    if (d->path == TM_PATH_TMA && nb % 16 == 0) {
        ReplaceAddressFn rep = replace_fn();
        if (!rep) return fail(TM_ECUDA, "the CUDA driver's cuTensorMapReplaceAddress is not reachable");
        if (rep((CUtensorMap*)d->tmap, new_base) != CUDA_SUCCESS)
            return fail(TM_ECUDA, "cuTensorMapReplaceAddress refused the new base");
        d->base = nb;
        return TM_OK;
    }
    // The path may change: rebuild from the stored fields.
    uint64_t gdim[5], gstr[4];
    uint32_t box[5], estr[5];
    for (uint32_t i = 0; i < d->rank; i++) {
        gdim[i] = d->dim[i];
        box[i] = d->box[i];
        estr[i] = d->estride[i];
        if (i > 0) gstr[i - 1] = d->stride[i];
    }
    tm_desc t;
    int rc = tmap_encode(&t, (tm_dtype)d->dtype, d->rank, new_base, gdim, gstr, box, estr,
                         (tm_swizzle)d->swizzle, (tm_oob)d->oob);
    if (rc) return rc;
    if (t.l2_promotion != d->l2_promotion) {  // keep the map's own promotion
        t.l2_promotion = d->l2_promotion;
        if (t.path == TM_PATH_TMA && (rc = encode_into(&t))) return rc;
    }
    if (forced) {
        t.path = TM_PATH_FALLBACK;
        t.why_fallback |= TM_WHY_FORCED;
    }
    *d = t;
    return TM_OK;
}

int tmap_set_l2_promotion(tm_desc* d, tm_l2_promotion promo)
{
    if (!valid_desc(d)) return fail(TM_EINVAL, "descriptor is not filled");
    if ((uint32_t)promo > TM_L2_256B) return fail(TM_EINVAL, "bad L2 promotion %d", (int)promo);
    d->l2_promotion = (uint32_t)promo;
    bool encoded = false;  // a planned map has an all-zero tensor map
    for (size_t i = 0; i < sizeof(d->tmap); i++) encoded = encoded || d->tmap[i] != 0;
    if (d->path == TM_PATH_TMA && encoded) return encode_into(d);
    return TM_OK;
}

int tmap_force_fallback(tm_desc* d)
{
    if (!valid_desc(d)) return fail(TM_EINVAL, "descriptor is not filled");
    d->path = TM_PATH_FALLBACK;
    d->why_fallback |= TM_WHY_FORCED;
    return TM_OK;
}

int tile_load_image(const tm_desc* src, const int32_t* coords, void* image, void* stream)
{
    if (!coords) return fail(TM_EINVAL, "coords is NULL");
    return copy_boxes(src, coords, 1, image, stream);
}

int tiled_copy(const tm_desc* src, const int32_t* coords, size_t nbox, void* images, void* stream)
{
    return copy_boxes(src, coords, nbox, images, stream);
}

int tiled_roundtrip(const tm_desc* dst, const int32_t* coords, size_t nbox, const void* images,
                    void* stream)
{
    if (!valid_desc(dst)) return fail(TM_EINVAL, "destination descriptor is not filled");
    if (!coords && nbox != 0 && nbox != dst->num_boxes)
        return fail(TM_EINVAL, "nbox %zu is neither 0 nor the grid's %llu boxes", nbox,
                    (unsigned long long)dst->num_boxes);
    const uint64_t n = coords ? nbox : dst->num_boxes;
    if (n == 0) return TM_OK;  // an empty box list moves nothing and needs no image buffer
    if (!images) return fail(TM_EINVAL, "images is NULL");
    if ((uintptr_t)images % 16) return fail(TM_EALIGN, "images must be 16-byte aligned");
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const bool tma = store_fits_tma(dst) && (!coords || list_fits_tma(dst, coords, n, true));
    BoxWalk w;
    if ((rc = make_walk(dst, coords, n, st, w))) return rc;
    if (tma) {
        Geometry g;
        const StreamArgs a = stream_args(dst, w, (uint64_t)images, *ds, g, st, false);
        const CUtensorMap* m = (const CUtensorMap*)dst->tmap;
        rc = check_launch(launch_tma_stream(KIND_ROUNDTRIP, dst->rank, m, m, a, g.grid, g.smem, st),
                          "tensor store launch");
    } else {
        FbArgs a = fb_args(dst, w, (uint64_t)images, *ds);
        uint32_t grid = 0;
        size_t smem = 0;
        SegArgs sa;
        // The segment form of the store (TM_FB_SEG as for the copy): image blocks staged by bulk
        // copies, rows written by the consumer warps.
        const uint32_t sms = (uint32_t)ds->sms;
        auto budget = [&](uint32_t per_sm) { return cta_budget(*ds, per_sm); };
        auto plan = [&](uint64_t cap) {
            const uint64_t want = std::min<uint64_t>(env_u64("TM_FB_SEG_CTAS_PER_SM", kSegCtasPerSm), cap);
            return seg_plan(a, dst, sms, (uint32_t)std::max<uint64_t>(std::min<uint64_t>(want, 8), 1),
                            (uint32_t)std::min<uint64_t>(env_u64("TM_FB_SEG_STAGES", kSegStoreStages), kSegMaxStages),
                            (int)env_u64("TM_FB_SEG", 2), true, budget, sa, grid, smem);
        };
        if (seg_fit(true, sms, sa, grid, smem, plan)) {
            sa.sched = sched_slot(*ds, st);
            rc = check_launch(launch_fb_seg_store(sa, grid, smem, st), "fallback segment store launch");
        } else {
            fb_shape(a, n, (uint32_t)ds->sms,
                     (uint32_t)std::min<uint64_t>(env_u64("TM_FB_STORE_CTAS_PER_SM", 6), 16),
                     kFbStoreRowBytes, [&](uint32_t per_sm) { return cta_budget(*ds, per_sm); },
                     grid, smem);
            rc = check_launch(launch_fb_store(a, grid, smem, st), "fallback store launch");
        }
    }
    release_walk(w, st);
    return rc;
}

int tile_reduce(const tm_desc* dst, const tm_desc* src, tm_redop op, void* stream)
{
    if (!valid_desc(dst) || !valid_desc(src)) return fail(TM_EINVAL, "descriptor is not filled");
    if (op != TM_RED_ADD && op != TM_RED_MIN && op != TM_RED_MAX)
        return fail(TM_EINVAL, "bad reduce op %d", (int)op);
    int red_type = -1;
    switch (dst->dtype) {
        case TM_F32: red_type = 0; break;
        case TM_F16: red_type = 1; break;
        case TM_BF16: red_type = 2; break;
        case TM_U32: red_type = 3; break;
        case TM_S32: red_type = 4; break;
        default: break;
    }
    if (red_type < 0) return fail(TM_EUNSUPPORTED, "reduce supports f32, f16, bf16, u32 and s32");
    if (src->dtype != dst->dtype) return fail(TM_EINVAL, "dst and src differ in element type");
    if (dst->rank != src->rank || dst->swizzle != src->swizzle)
        return fail(TM_EINVAL, "dst and src differ in rank or swizzle");
    if (!unit_steps(dst) || !unit_steps(src))
        return fail(TM_EUNSUPPORTED, "reduce takes maps whose elementStrides are all 1");
    for (uint32_t i = 0; i < dst->rank; i++) {
        if (dst->dim[i] != src->dim[i] || dst->box[i] != src->box[i])
            return fail(TM_EINVAL, "dst and src differ in dims or box (dim %u)", i);
    }
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    BoxWalk w;
    if ((rc = make_walk(dst, nullptr, 0, st, w))) return rc;
    // The tensor reduce is given add on every supported type and min / max on the integer types;
    // float min / max run element-wise on the vector path.
    const bool tma_op = op == TM_RED_ADD || red_type >= 3;
    if (tma_op && store_fits_tma(dst) && src->path == TM_PATH_TMA) {
        Geometry g;
        const StreamArgs a = stream_args(dst, w, 0, *ds, g, st, true);
        rc = check_launch(launch_tma_stream(KIND_REDUCE + (int)op, dst->rank,
                                            (const CUtensorMap*)src->tmap,
                                            (const CUtensorMap*)dst->tmap, a, g.grid, g.smem, st),
                          "tensor reduce launch");
    } else {
        FbArgs a = fb_args(dst, w, 0, *ds);
        a.src_base = src->base;
        for (int i = 0; i < 5; i++) a.src_stride[i] = (int64_t)src->stride[i];
        a.red_type = (uint16_t)red_type;
        a.red_op = (uint16_t)op;
        // the element-wise kernel's warps take 8 KiB pieces of the tensor's rows, grid-strided;
        // 3 CTAs of 8 warps per SM (fewer CTAs for a small tensor)
        uint64_t pieces = (dst->dim[0] * dst->esize + 8191) / 8192;
        for (uint32_t i = 1; i < dst->rank; i++) pieces *= dst->dim[i];
        const uint32_t grid = (uint32_t)std::min<uint64_t>((pieces + 7) / 8, (uint64_t)ds->sms * 3);
        rc = check_launch(launch_fb_reduce(a, std::max<uint32_t>(grid, 1), st),
                          "fallback reduce launch");
    }
    return rc;
}

int tile_reduce_add(const tm_desc* dst, const tm_desc* src, void* stream)
{
    if (!valid_desc(dst) || !valid_desc(src)) return fail(TM_EINVAL, "descriptor is not filled");
    if (dst->dtype != TM_F32 || src->dtype != TM_F32)
        return fail(TM_EUNSUPPORTED, "reduce-add supports TM_F32 maps only");
    return tile_reduce(dst, src, TM_RED_ADD, stream);
}

int stream_tiles(const tm_desc* a, const tm_desc* b, uint32_t stages, float* cs_a, float* cs_b,
                 uint64_t* bits_a, uint64_t* bits_b, void* stream)
{
    if (!valid_desc(a) || !valid_desc(b)) return fail(TM_EINVAL, "descriptor is not filled");
    if (!cs_a || !cs_b || !bits_a || !bits_b) return fail(TM_EINVAL, "an output array is NULL");
    if ((uintptr_t)cs_a % 4 || (uintptr_t)cs_b % 4 || (uintptr_t)bits_a % 8 || (uintptr_t)bits_b % 8)
        return fail(TM_EALIGN, "output arrays must be naturally aligned");
    for (const tm_desc* d : {a, b}) {
        if (d->dtype != TM_BF16 || d->rank != 2)
            return fail(TM_EUNSUPPORTED, "stream_tiles needs rank-2 TM_BF16 maps");
        const uint32_t rows = d->box[1];
        if (d->box[0] != 64 || !(rows == 32 || rows == 64 || rows == 128 || rows == 256))
            return fail(TM_EUNSUPPORTED, "stream_tiles needs boxes {64, R}, R in 32/64/128/256");
        if (d->swizzle != TM_SWIZZLE_128B && d->swizzle != TM_SWIZZLE_NONE)
            return fail(TM_EUNSUPPORTED, "stream_tiles reads 128B-swizzled or unswizzled tiles");
        if (d->path != TM_PATH_TMA) return fail(TM_EUNSUPPORTED, "stream_tiles needs TMA-path maps");
        if (!unit_steps(d) || d->oob != TM_OOB_ZERO)
            return fail(TM_EUNSUPPORTED, "stream_tiles needs unit elementStrides and zero fill");
    }
    if (a->box[1] != b->box[1] || a->swizzle != b->swizzle)
        return fail(TM_EINVAL, "A and B differ in tile rows or swizzle");
    if (a->num_boxes != b->num_boxes)
        return fail(TM_EINVAL, "A has %llu tiles, B has %llu", (unsigned long long)a->num_boxes,
                    (unsigned long long)b->num_boxes);
    if (stages < 2 || stages > 8) return fail(TM_ERANGE, "stages %u outside 2..8", stages);
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    RingArgs r;
    memset(&r, 0, sizeof(r));
    r.ntiles = a->num_boxes;
    r.a_nb0 = a->nbox[0];
    r.b_nb0 = b->nbox[0];
    r.rows = a->box[1];
    r.stages = stages;
    r.tile_bytes = (uint32_t)a->box_bytes;
    r.swizzled = a->swizzle == TM_SWIZZLE_128B ? 1u : 0u;
    r.prefetch = (uint32_t)std::min<uint64_t>(env_u64("TM_RING_PREFETCH", 0), 64);
    // Two consumer groups (even and odd tiles) when the stages divide between them
    // (TM_RING_GROUPS=1 keeps one): a group's per-tile chain of reads, ordered sums and the
    // cross-warp reduction then overlaps the other group's.
    r.groups = (stages % 2 == 0 && env_u64("TM_RING_GROUPS", 2) >= 2) ? 2u : 1u;
    // Bank-conflict control (TM_RING_ROW_PAIRS=1): the consumers read the rows of each 32-row
    // block in the order an ungrouped 256-byte row stride would give; same results.
    r.row_pairs = env_u64("TM_RING_ROW_PAIRS", 0) ? 1u : 0u;
    // Each tile is read once: its loads carry an L2 evict-first policy, so the stream recycles its
    // own L2 lines rather than evicting (and forcing the write-back of) other data
    // (TM_RING_EVICT_FIRST=0 drops the policy).
    r.evict_first = env_u64("TM_RING_EVICT_FIRST", 1) ? 1u : 0u;
    r.cs_a = cs_a;
    r.cs_b = cs_b;
    r.bits_a = (unsigned long long*)bits_a;
    r.bits_b = (unsigned long long*)bits_b;
    r.timeout_ns = wait_limit_ns();
    r.status = ds->status;
    const size_t smem = (size_t)stages * 2 * r.tile_bytes + kStageAlign;
    if (smem > cta_budget(*ds, 1)) return fail(TM_ERANGE, "%u stages of two tiles exceed shared memory", stages);
    uint32_t per_sm = 1;
    while (per_sm < 4 && cta_budget(*ds, per_sm + 1) >= smem) per_sm++;
    const uint32_t grid = (uint32_t)std::min<uint64_t>(r.ntiles, (uint64_t)ds->sms * per_sm);
    ring_schedule(r, grid);
    return check_launch(launch_ring((const CUtensorMap*)a->tmap, (const CUtensorMap*)b->tmap, r, grid,
                                    smem, (cudaStream_t)stream),
                        "ring launch");
}

int stream_gemm(const tm_desc* a, const tm_desc* b, float* c, uint64_t ldc, uint32_t stages,
                void* stream)
{
    if (!valid_desc(a) || !valid_desc(b)) return fail(TM_EINVAL, "descriptor is not filled");
    if (!c) return fail(TM_EINVAL, "c is NULL");
    const uint32_t want_box[2][2] = {{64, 128}, {64, 256}};
    const tm_desc* ops[2] = {a, b};
    for (int i = 0; i < 2; i++) {
        const tm_desc* d = ops[i];
        if (d->dtype != TM_BF16 || d->rank != 2)
            return fail(TM_EUNSUPPORTED, "stream_gemm needs rank-2 TM_BF16 maps");
        if (d->box[0] != want_box[i][0] || d->box[1] != want_box[i][1])
            return fail(TM_EUNSUPPORTED, "stream_gemm needs boxes {64, 128} for A and {64, 256} for B");
        if (d->swizzle != TM_SWIZZLE_128B)
            return fail(TM_EUNSUPPORTED, "stream_gemm needs 128-byte swizzled maps");
        if (d->path != TM_PATH_TMA || !unit_steps(d) || d->oob != TM_OOB_ZERO)
            return fail(TM_EUNSUPPORTED, "stream_gemm needs TMA-path maps with unit steps and zero fill");
    }
    if (a->dim[0] != b->dim[0])
        return fail(TM_EINVAL, "A has K = %llu, B has K = %llu", (unsigned long long)a->dim[0],
                    (unsigned long long)b->dim[0]);
    const uint64_t M = a->dim[1], N = b->dim[1], K = a->dim[0];
    if (M >= (1ull << 31) || N >= (1ull << 31) || K >= (1ull << 31))
        return fail(TM_ERANGE, "M, N and K must be below 2^31");
    if (ldc < N) return fail(TM_EINVAL, "ldc %llu is below N = %llu", (unsigned long long)ldc,
                             (unsigned long long)N);
    if ((uintptr_t)c % 16 || ldc % 4)
        return fail(TM_EALIGN, "c must be 16-byte aligned and ldc a multiple of 4");
    if (stages < 2 || stages > kGemmMaxPairStages)
        return fail(TM_ERANGE, "stages %u outside 2..%u", stages, kGemmMaxPairStages);
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    // Forms: the CTA-pair form (256-row tiles over the two SMs of a cluster, tcgen05 cta_group::2,
    // 32 KiB stages, up to 7), the default when C has more than one 128-row tile (measured on
    // GB300 at 8192 x 8192 x 4096: 1738-1821 TFLOP/s with 7 stages); one SM per 128 x 256 tile
    // otherwise, or with TM_GEMM_PAIR=0 (1392-1405 TFLOP/s).
    const bool pair = env_u64("TM_GEMM_PAIR", 1) != 0 && M > 128 && ds->sms >= 2;
    const uint32_t rows = pair ? 256u : 128u;
    const uint32_t S = std::min<uint32_t>(stages, pair ? kGemmMaxPairStages : kGemmMaxStages);
    GemmArgs g;
    memset(&g, 0, sizeof(g));
    g.m = (uint32_t)M;
    g.n = (uint32_t)N;
    g.k = (uint32_t)K;
    g.mtiles = (uint32_t)((M + rows - 1) / rows);
    g.ntiles = (uint32_t)((N + 255) / 256);
    g.kblocks = (uint32_t)((K + 63) / 64);
    g.stages = S;
    g.split_from = 0;
    g.c = c;
    g.ldc = ldc;
    g.timeout_ns = wait_limit_ns();
    g.status = ds->status;
    const uint64_t tiles = (uint64_t)g.mtiles * g.ntiles;
    if (tiles >= (1ull << 31)) return fail(TM_ERANGE, "too many tiles");
    const size_t smem = (size_t)S * (pair ? 32768 : 49152) + kStageAlign;
    if (smem > cta_budget(*ds, 1) + 1024) return fail(TM_ERANGE, "%u stages exceed shared memory", S);
    const CUtensorMap* ma = (const CUtensorMap*)a->tmap;
    const CUtensorMap* mb = (const CUtensorMap*)b->tmap;
    if (pair) {
        // Each CTA of a pair loads a 128-row half of the B tile: a map of B with a 128-row box
        // (the caller's has 256 rows).  Every stage expects exactly 16 KiB per half and per A tile.
        tm_desc bh;
        const uint64_t dims[2] = {b->dim[0], b->dim[1]};
        const uint64_t strides[1] = {b->stride[1]};
        const uint32_t box[2] = {64, 128};
        if ((rc = plan_impl(&bh, TM_BF16, 2, (void*)(uintptr_t)b->base, dims, strides, box, nullptr,
                            TM_SWIZZLE_128B, TM_OOB_ZERO)))
            return rc;
        if ((rc = encode_into(&bh))) return rc;
        if (bh.path != TM_PATH_TMA || bh.box_bytes != 16384 || a->box_bytes != 16384)
            return fail(TM_EUNSUPPORTED, "stream_gemm could not encode the half-tile map of B");
        const CUtensorMap* mbh = (const CUtensorMap*)bh.tmap;
        // persistent: one cluster of two CTAs per pair of SMs.  A last wave of r < pairs tiles
        // would leave pairs idle; when 2r <= pairs its tiles are done as 256 x 128 halves (each
        // CTA loading 64 B rows through a 64-row map of B), so that the wave takes half a tile
        // (TM_GEMM_TAIL_SPLIT=0 keeps whole tiles).
        const uint64_t pairs = std::min<uint64_t>(tiles, (uint64_t)ds->sms / 2);
        const uint64_t rem = tiles % pairs;
        const bool split = env_u64("TM_GEMM_TAIL_SPLIT", 1) != 0 && tiles > pairs && rem > 0 &&
                           2 * rem <= pairs;
        g.split_from = (uint32_t)(split ? tiles - rem : tiles);
        tm_desc bq;
        const uint32_t qbox[2] = {64, 64};
        if ((rc = plan_impl(&bq, TM_BF16, 2, (void*)(uintptr_t)b->base, dims, strides, qbox,
                            nullptr, TM_SWIZZLE_128B, TM_OOB_ZERO)))
            return rc;
        if ((rc = encode_into(&bq))) return rc;
        if (bq.path != TM_PATH_TMA || bq.box_bytes != 8192)
            return fail(TM_EUNSUPPORTED, "stream_gemm could not encode the quarter-tile map of B");
        return check_launch(launch_gemm_pair(ma, mbh, (const CUtensorMap*)bq.tmap, g,
                                             (uint32_t)(2 * pairs), smem, (cudaStream_t)stream),
                            "gemm launch (CTA pairs)");
    }
    if (a->box_bytes != 16384 || b->box_bytes != 32768)
        return fail(TM_EUNSUPPORTED, "stream_gemm: A and B tiles must be 16 and 32 KiB");
    // persistent: one CTA per SM (the stages and the two 256-column accumulators fill an SM)
    const uint64_t grid = std::min<uint64_t>(tiles, (uint64_t)ds->sms);
    return check_launch(launch_gemm(ma, mb, g, (uint32_t)grid, smem, (cudaStream_t)stream),
                        "gemm launch");
}

int tm_stream_check(void* stream)
{
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    StatusBlock sb;
    if ((e = cudaMemcpy(&sb, ds->status, sizeof(sb), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "reading the status word");
    if (sb.code == 0) return TM_OK;
    if ((e = cudaMemset(ds->status, 0, sizeof(sb))) != cudaSuccess)
        return cuda_fail(e, "clearing the status word");
    static const char* names[] = {"?", "tiled copy", "round trip", "reduce-add", "ring",
                                  "fallback copy", "fallback store", "fallback reduce", "self-test",
                                  "gemm", "fallback segment copy", "fallback segment store"};
    const char* kn = sb.kernel < sizeof(names) / sizeof(names[0]) ? names[sb.kernel] : "?";
    return fail(sb.code, "%s kernel: wait gave up in block %u, stage %u, parity %u, box %llu", kn,
                sb.block, sb.stage, sb.phase, (unsigned long long)sb.box);
}

int tm_selftest_wait_timeout(uint64_t timeout_ns, void* stream)
{
    DevState* ds = nullptr;
    int rc = device_state(&ds);
    if (rc) return rc;
    return check_launch(launch_selftest(timeout_ns, ds->status, (cudaStream_t)stream),
                        "self-test launch");
}

const char* tm_last_error(void) { return g_err; }
size_t tm_box_bytes(const tm_desc* d) { return valid_desc(d) ? (size_t)d->box_bytes : 0; }
size_t tm_num_boxes(const tm_desc* d) { return valid_desc(d) ? (size_t)d->num_boxes : 0; }
int tm_path(const tm_desc* d) { return valid_desc(d) ? (int)d->path : 0; }
size_t tm_desc_size(void) { return sizeof(tm_desc); }

int tm_pick_swizzle(uint32_t inner_bytes)
{
    return inner_bytes == 128 ? TM_SWIZZLE_128B
           : inner_bytes == 64 ? TM_SWIZZLE_64B
           : inner_bytes == 32 ? TM_SWIZZLE_32B
                               : TM_SWIZZLE_NONE;
}

}  // extern "C"
