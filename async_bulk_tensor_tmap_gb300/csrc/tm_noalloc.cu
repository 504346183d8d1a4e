// tm_noalloc.cu -- tiled_copy_noalloc: the tiled copy for callers that must not allocate device
// memory.
//
// tiled_copy allocates: the first launching call on a device cudaMallocs the device's status
// word, and an explicit list of more than 8 boxes is staged in memory from cudaMallocAsync.  Some
// callers cannot allow that -- code that runs while another allocator owns all device memory,
// processes under a hard device-memory cap where a late allocation may fail, latency-critical
// loops that cannot afford an allocator call.  This variant keeps all of its scratch (a status word
// and the box list) in one file-scope __device__ array of fixed size, so it allocates nothing;
// the caller still passes the tensor map and the output images.
//
// The array is a module global: every GPU that loads the library holds its 327,936 bytes until
// the process exits.  Host code may not use the array's name as a device address (it names a
// host-side stand-in), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current, and every launch receives that pointer.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tm_internal.h"
#include "tmap.h"

namespace {

constexpr size_t kMaxBoxes = TM_NOALLOC_MAX_BOXES;
constexpr size_t kStatusBytes = 256;  // status word, padded so the list stays 256-byte aligned
constexpr size_t kScratchBytes = kStatusBytes + kMaxBoxes * 5 * sizeof(int32_t);
static_assert(kScratchBytes == 327936, "scratch size as documented");
static_assert(sizeof(tmk::StatusBlock) <= kStatusBytes, "status word fits its slot");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct Dev {
    bool ready = false;
    unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int sms = 0, smem_per_sm = 0, smem_optin = 0;
};

std::mutex g_mu;
Dev g_devs[64];

int cuda_err(cudaError_t e, const char* what)
{
    char msg[256];
    snprintf(msg, sizeof(msg), "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    return tmk::set_last_error(TM_ECUDA, msg);
}

// Once per device, with that device current: the scratch address and the launch attributes.
int setup(Dev** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return tmk::set_last_error(TM_EUNSUPPORTED, "device ordinal above 63");
    std::lock_guard<std::mutex> lk(g_mu);
    Dev& d = g_devs[dev];
    if (!d.ready) {
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_scratch)) != cudaSuccess)
            return cuda_err(e, "cudaGetSymbolAddress(scratch)");
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) ||
            (e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                        dev)) ||
            (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)))
            return cuda_err(e, "cudaDeviceGetAttribute");
        d.scratch = static_cast<unsigned char*>(p);
        d.ready = true;
    }
    *out = &d;
    return TM_OK;
}

size_t budget(const Dev& d, uint32_t per_sm)
{
    const size_t share = (size_t)d.smem_per_sm / per_sm;
    const size_t cap = std::min<size_t>((size_t)d.smem_optin, share > 1024 ? share - 1024 : 0);
    return cap > 2048 + 256 ? cap - 1024 - 256 : 0;
}

uint32_t stage_of(uint64_t box_bytes)
{
    return (uint32_t)((box_bytes + tmk::kStageAlign - 1) / tmk::kStageAlign * tmk::kStageAlign);
}

// Same rule as the allocating entry point: the tensor-map hardware is only given lists whose
// innermost starts sit on the 16-byte grid and whose boxes overlap the tensor.
bool list_on_tma(const tm_desc* d, const int32_t* c, size_t n)
{
    for (size_t b = 0; b < n; b++) {
        const int32_t* s = c + b * d->rank;
        if (((int64_t)s[0] * d->esize) % 16 != 0) return false;
        for (uint32_t i = 0; i < d->rank; i++) {
            if ((int64_t)s[i] >= (int64_t)d->dim[i] || (int64_t)s[i] + (int64_t)d->box[i] <= 0)
                return false;
        }
    }
    return true;
}

uint64_t limit_ns() { return tmk::env_u64("TM_WAIT_TIMEOUT_NS", 1000000000ull); }

}  // namespace

extern "C" int tiled_copy_noalloc(const tm_desc* src, const int32_t* coords, size_t nbox,
                                  void* images, void* stream)
{
    using namespace tmk;
    if (!src || src->magic != TM_DESC_MAGIC)
        return set_last_error(TM_EINVAL, "source descriptor is not filled");
    if (!coords && nbox != 0 && nbox != src->num_boxes)
        return set_last_error(TM_EINVAL, "nbox is neither 0 nor the grid's box count");
    if (coords && nbox > kMaxBoxes) {
        char msg[160];
        snprintf(msg, sizeof(msg), "tiled_copy_noalloc takes at most %zu listed boxes, got %zu "
                 "(its scratch is a fixed array)", kMaxBoxes, nbox);
        return set_last_error(TM_ERANGE, msg);
    }
    const uint64_t n = coords ? nbox : src->num_boxes;
    if (n == 0) return TM_OK;  // an empty box list moves nothing and needs no image buffer
    if (!images) return set_last_error(TM_EINVAL, "images is NULL");
    if ((uintptr_t)images % 16) return set_last_error(TM_EALIGN, "images must be 16-byte aligned");
    Dev* d = nullptr;
    int rc = setup(&d);
    if (rc) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    StatusBlock* status = reinterpret_cast<StatusBlock*>(d->scratch);
    int32_t* list = reinterpret_cast<int32_t*>(d->scratch + kStatusBytes);

    // The array keeps the previous call's bytes: the status word must start at zero.
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(StatusBlock), st);
    if (e != cudaSuccess) return cuda_err(e, "clearing the scratch status word");
    BoxWalk w;
    memset(&w, 0, sizeof(w));
    w.nbox = n;
    w.rank = src->rank;
    for (int i = 0; i < 5; i++) {
        w.box[i] = src->box[i];
        w.grid_nb[i] = src->nbox[i];
    }
    if (coords) {
        w.mode = WALK_LIST;
        w.list = list;
        e = cudaMemcpyAsync(list, coords, n * src->rank * sizeof(int32_t), cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return cuda_err(e, "copying the box list to the scratch");
    } else {
        w.mode = WALK_GRID;
    }
    const bool tma = src->path == TM_PATH_TMA && (!coords || list_on_tma(src, coords, n));
    if (tma) {
        StreamArgs a;
        memset(&a, 0, sizeof(a));
        const uint32_t span = src->swizzle == TM_SWIZZLE_128B ? 128u : src->swizzle == TM_SWIZZLE_64B ? 64u
                              : src->swizzle == TM_SWIZZLE_32B ? 32u : 0u;
        a.walk = w;
        a.images = (uint64_t)images;
        uint32_t grid = 0;
        size_t smem = 0;
        // the launch shape of tiled_copy (same rule, same tunables); stream_plan leaves the work
        // split static (no counter: the dynamic split's counters are allocated memory)
        stream_plan(a, src->box_bytes, span, (uint32_t)d->sms,
                    [&](uint32_t per_sm) { return budget(*d, per_sm); }, grid, smem);
        a.timeout_ns = limit_ns();
        a.status = status;
        const CUtensorMap* m = (const CUtensorMap*)src->tmap;
        e = launch_tma_stream(KIND_COPY, src->rank, m, m, a, grid, smem, st);
    } else {
        FbArgs a;
        memset(&a, 0, sizeof(a));
        a.walk = w;
        fb_from_desc(a, src);
        a.images = (uint64_t)images;
        a.stage_bytes = stage_of(src->box_bytes);
        a.timeout_ns = limit_ns();
        a.status = status;
        uint32_t grid = 0;
        size_t smem = 0;
        SegArgs sa;
        // the launch shape of tiled_copy's vector path (same rule, same tunables)
        const uint32_t sms = (uint32_t)d->sms;
        auto cta_bytes = [&](uint32_t per_sm) { return budget(*d, per_sm); };
        if (seg_fit(false, sms, sa, grid, smem, [&](uint64_t cap) {
                return fb_copy_plan(a, src, n, sms, cta_bytes, sa, grid, smem, cap);
            })) {
            e = launch_fb_seg_copy(sa, grid, smem, st);
        } else {
            e = launch_fb_copy(a, grid, smem, st);
        }
    }
    if (e != cudaSuccess) return cuda_err(e, "copy launch");
    // The status word is read back before returning, so the call completes the copy.
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return cuda_err(e, "cudaStreamSynchronize");
    StatusBlock sb;
    if ((e = cudaMemcpy(&sb, status, sizeof(sb), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_err(e, "reading the scratch status word");
    if (sb.code != 0) {
        char msg[200];
        snprintf(msg, sizeof(msg), "tiled_copy_noalloc: a wait gave up in block %u, stage %u, "
                 "parity %u, box %llu", sb.block, sb.stage, sb.phase, (unsigned long long)sb.box);
        return set_last_error(sb.code, msg);
    }
    return TM_OK;
}
