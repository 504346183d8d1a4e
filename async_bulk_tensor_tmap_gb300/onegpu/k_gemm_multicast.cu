// k_gemm_multicast.cu -- libtmap_gb300_onegpu.so: the one-SM tensor-core GEMM of tm_gemm.cuh with
// the B tile shared by the two CTAs of a cluster through TMA multicast.  One-GPU only: built on
// request, never part of libtmap_gb300.so, and every call refuses tensors that are not device
// memory of the current device (include/tmap_onegpu.h).
//
// [H200-TMA] coolgpu "H200 · TMA · Tensor Memory Accelerator" feature card, §01 是什么 and §04 ③:
// one multicast copy lands in the shared memory of every CTA in the mask; the launch must be a
// cluster launch.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "tm_gemm.cuh"
#include "tmap_onegpu.h"

namespace tmk {
namespace {

// TMA tensor load of a 2-D box into the same shared-memory offset of every CTA in `mask`,
// completing on the mbarrier at offset `bar` in each of them.
__device__ __forceinline__ void tma_load_2d_multicast(uint32_t dst, const CUtensorMap* m, int32_t c0,
                                                      int32_t c1, uint32_t bar, uint16_t mask)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar), "h"(mask)
        : "memory");
}

// Arrives on the mbarrier at offset bar_saddr in every CTA of `mask` once every tcgen05 operation
// this thread issued before has completed.
__device__ __forceinline__ void tc_commit_multicast(uint32_t bar_saddr, uint16_t mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar_saddr),
        "h"(mask)
        : "memory");
}

// The two CTAs of a cluster (tiles 2m and 2m + 1 of one column of tiles) share each B tile: CTA r
// loads rows r * 128 .. r * 128 + 127 of it (the map's box is a 128-row half) multicast into both
// CTAs' stages, and each CTA's MMA commits release the stage in both.
struct SharedB {
    static constexpr uint32_t kShare = 2;
    __device__ static void load_b(uint32_t dst, const CUtensorMap* mb_half, uint32_t kb, uint32_t nt,
                                  uint32_t rank, uint32_t bar)
    {
        tma_load_2d_multicast(dst + rank * (kTileB / 2), mb_half, (int32_t)(kb * kBK),
                              (int32_t)(nt * kBN + rank * (kBN / 2)), bar, (uint16_t)0x3);
    }
    __device__ static void release(uint32_t empty_bar) { tc_commit_multicast(empty_bar, (uint16_t)0x3); }
};

static __device__ StatusBlock g_status;  // per device: this library's timeout report

thread_local char g_err[400] = "";

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

struct Dev {
    bool ready = false;
    int sms = 0, smem_optin = 0;
    StatusBlock* status = nullptr;  // device address of g_status on this device
};
std::mutex g_mu;
Dev g_devs[64];

int device(int* ordinal, Dev** out)
{
    cudaError_t e = cudaGetDevice(ordinal);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (*ordinal < 0 || *ordinal >= 64) return fail(TM_EUNSUPPORTED, "device ordinal above 63");
    std::lock_guard<std::mutex> lk(g_mu);
    Dev& d = g_devs[*ordinal];
    if (!d.ready) {
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_status)) != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(status)");
        if ((e = cudaMemset(p, 0, sizeof(StatusBlock))) != cudaSuccess)
            return cuda_fail(e, "clearing the status word");
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, *ordinal)) ||
            (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                        *ordinal)))
            return cuda_fail(e, "cudaDeviceGetAttribute");
        d.status = static_cast<StatusBlock*>(p);
        d.ready = true;
    }
    *out = &d;
    return TM_OK;
}

// Whether `p` is device memory of device `dev` (not host, managed or another GPU's memory).
bool on_device(const void* p, int dev)
{
    cudaPointerAttributes at;
    memset(&at, 0, sizeof(at));
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // clear the error an unregistered host pointer leaves
        return false;
    }
    return at.type == cudaMemoryTypeDevice && at.device == dev;
}

int check_map(const tm_desc* d, const char* name)
{
    if (!d || d->magic != TM_DESC_MAGIC) return fail(TM_EINVAL, "%s: descriptor is not filled", name);
    if (d->dtype != TM_BF16 || d->rank != 2)
        return fail(TM_EUNSUPPORTED, "%s: stream_gemm_multicast needs a rank-2 TM_BF16 map", name);
    if (d->box[0] != 64 || d->box[1] != 128)
        return fail(TM_EUNSUPPORTED, "%s: stream_gemm_multicast needs a {64, 128} box", name);
    if (d->swizzle != TM_SWIZZLE_128B || d->path != TM_PATH_TMA || d->oob != TM_OOB_ZERO ||
        d->estride[0] != 1 || d->estride[1] != 1)
        return fail(TM_EUNSUPPORTED, "%s: needs a 128-byte swizzled tensor-map-path map with unit "
                    "steps and zero fill", name);
    return TM_OK;
}

}  // namespace
}  // namespace tmk

extern "C" {

int stream_gemm_multicast(const tm_desc* a, const tm_desc* b, float* c, uint64_t ldc,
                          uint32_t stages, void* stream)
{
    using namespace tmk;
    const char* ws = getenv("WORLD_SIZE");
    if (ws && atoi(ws) > 1)
        return fail(TM_EUNSUPPORTED, "stream_gemm_multicast runs in one-GPU processes only "
                    "(WORLD_SIZE=%s)", ws);
    int rc = check_map(a, "a");
    if (rc || (rc = check_map(b, "b_half"))) return rc;
    if (!c) return fail(TM_EINVAL, "c is NULL");
    if (a->dim[0] != b->dim[0]) return fail(TM_EINVAL, "A and B differ in K");
    const uint64_t M = a->dim[1], N = b->dim[1], K = a->dim[0];
    if (M >= (1ull << 31) || N >= (1ull << 31) || K >= (1ull << 31))
        return fail(TM_ERANGE, "M, N and K must be below 2^31");
    if (ldc < N) return fail(TM_EINVAL, "ldc is below N");
    if ((uintptr_t)c % 16 || ldc % 4) return fail(TM_EALIGN, "c must be 16-byte aligned, ldc % 4 == 0");
    if (stages < 2 || stages > kGemmMaxStages)
        return fail(TM_ERANGE, "stages %u outside 2..%u", stages, kGemmMaxStages);
    int dev = 0;
    Dev* d = nullptr;
    if ((rc = device(&dev, &d))) return rc;
    // one GPU's own memory only: the maps' tensors and C
    if (!on_device((const void*)(uintptr_t)a->base, dev) || !on_device((const void*)(uintptr_t)b->base, dev) ||
        !on_device(c, dev))
        return fail(TM_EINVAL, "A, B and C must be device memory of the current device %d", dev);
    GemmArgs g;
    memset(&g, 0, sizeof(g));
    g.m = (uint32_t)M;
    g.n = (uint32_t)N;
    g.k = (uint32_t)K;
    g.mtiles = (uint32_t)((M + kBM - 1) / kBM);
    g.ntiles = (uint32_t)((N + kBN - 1) / kBN);
    g.kblocks = (uint32_t)((K + kBK - 1) / kBK);
    g.stages = stages;
    g.c = c;
    g.ldc = ldc;
    const char* lim = getenv("TM_WAIT_TIMEOUT_NS");
    g.timeout_ns = lim && *lim ? strtoull(lim, nullptr, 10) : 1000000000ull;
    g.status = d->status;
    const size_t smem = (size_t)stages * kGemmStage + kStageAlign;
    if (smem > (size_t)d->smem_optin) return fail(TM_ERANGE, "%u stages exceed shared memory", stages);
    // persistent: one cluster of two CTAs (row tiles 2m and 2m + 1 of one column of tiles) per
    // pair of SMs
    const uint64_t units = (uint64_t)((g.mtiles + 1) / 2) * g.ntiles;
    const uint64_t clusters = units < (uint64_t)d->sms / 2 ? units : (uint64_t)d->sms / 2;
    if (clusters == 0) return fail(TM_EUNSUPPORTED, "needs at least two SMs");
    cudaError_t e = cudaFuncSetAttribute(k_gemm_one_sm<SharedB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = launch_cluster2(k_gemm_one_sm<SharedB>, (uint32_t)(2 * clusters), smem,
                            (cudaStream_t)stream, *(const CUtensorMap*)a->tmap,
                            *(const CUtensorMap*)b->tmap, g);
    return e == cudaSuccess ? TM_OK : cuda_fail(e, "gemm launch (B multicast)");
}

int tm_onegpu_check(void* stream)
{
    using namespace tmk;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int dev = 0;
    Dev* d = nullptr;
    int rc = device(&dev, &d);
    if (rc) return rc;
    StatusBlock sb;
    if ((e = cudaMemcpy(&sb, d->status, sizeof(sb), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "reading the status word");
    if (sb.code == 0) return TM_OK;
    if ((e = cudaMemset(d->status, 0, sizeof(sb))) != cudaSuccess)
        return cuda_fail(e, "clearing the status word");
    return fail(sb.code, "multicast gemm: a wait gave up in block %u, stage %u, parity %u, tile %llu",
                sb.block, sb.stage, sb.phase, (unsigned long long)sb.box);
}

const char* tm_onegpu_last_error(void) { return tmk::g_err; }

}  // extern "C"
