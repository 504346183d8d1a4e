// tm_ptx.cuh -- the asynchronous-copy primitives of the path, as inline PTX for sm_103a.
//
// Written from the PTX ISA semantics the pages describe:
//   [MLSys-TMA] mlc.ai "Modern GPU Programming for MLSys", chapter "异步数据搬运：TMA"
//   [Book-TMA]  fangpin "gpu-hpc-book", chapter 08 "Cuda TMA （Tensor Memory Accelerator）"
//   [H200-TMA]  coolgpu "H200 · TMA · Tensor Memory Accelerator" feature card
//
// Every wait on an mbarrier here is bounded by a %globaltimer deadline: a wait that runs out
// returns false and the caller records TM_ETIMEOUT instead of spinning forever.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "tm_internal.h"

namespace tmk {

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t gtimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- per-CTA timeline (only in the tracing build, libtmap_gb300_trace.so, compiled with
//      -DTM_TRACE; in the library itself the stamps compile to nothing) --------------------------
// A kernel file declares its buffer with TM_TRACE_BUFFER(name): kTraceSlots %globaltimer stamps
// per CTA for the first kTraceCtas CTAs, read and cleared from the host through
// tm_trace_fetch_<name>() and tm_trace_clear_<name>().  TM_STAMP(name, slot) writes one stamp,
// TM_TRACE_PUT(name, slot, value) a plain number (a CTA's item count, say).
#ifdef TM_TRACE
constexpr uint32_t kTraceCtas = 2048, kTraceSlots = 64;
#define TM_TRACE_BUFFER(NAME)                                                                     \
    static __device__ unsigned long long g_trace_##NAME[kTraceCtas * kTraceSlots];                \
    extern "C" int tm_trace_fetch_##NAME(void* host, size_t bytes)                                \
    {                                                                                             \
        const size_t n = bytes < sizeof(g_trace_##NAME) ? bytes : sizeof(g_trace_##NAME);         \
        return (int)cudaMemcpyFromSymbol(host, g_trace_##NAME, n);                                \
    }                                                                                             \
    extern "C" int tm_trace_clear_##NAME(void)                                                    \
    {                                                                                             \
        void* p = nullptr;                                                                        \
        cudaError_t e = cudaGetSymbolAddress(&p, g_trace_##NAME);                                 \
        return (int)(e != cudaSuccess ? e : cudaMemset(p, 0, sizeof(g_trace_##NAME)));            \
    }
#define TM_STAMP(NAME, SLOT) TM_TRACE_PUT(NAME, SLOT, gtimer_ns())
#define TM_TRACE_PUT(NAME, SLOT, VALUE)                                                           \
    do {                                                                                          \
        if (blockIdx.x < kTraceCtas) g_trace_##NAME[blockIdx.x * kTraceSlots + (SLOT)] = (VALUE); \
    } while (0)
#else
#define TM_TRACE_BUFFER(NAME)
#define TM_STAMP(NAME, SLOT) \
    do {                     \
    } while (0)
#define TM_TRACE_PUT(NAME, SLOT, VALUE) \
    do {                                \
    } while (0)
#endif

// One thread of a full warp is chosen to issue ([MLSys-TMA] §"一个 thread 如何描述整个 tile": the
// other lanes are masked while the request is submitted; [H200-TMA] §03: one issuing thread).
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// ---- mbarrier ([MLSys-TMA] §"如何等待 TMA load 完成", [Book-TMA] §"TMA 完成异步数据搬运") ------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes initialised barriers visible to the async proxy (the TMA engine) before first use.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy reads of them.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One arrival plus `bytes` expected transaction bytes for the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits until the phase with parity `parity` has completed or `limit_ns` has passed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = gtimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (gtimer_ns() - t0 > limit_ns) return false;
    }
}

// Records the first failure of the launch set in the device status word.
__device__ __forceinline__ void record_timeout(StatusBlock* st, uint32_t kernel, uint32_t stage,
                                               uint32_t phase, uint64_t box)
{
    if (atomicCAS(&st->code, 0, TM_ETIMEOUT) == 0) {
        st->kernel = kernel;
        st->block = blockIdx.x;
        st->stage = stage;
        st->phase = phase;
        st->box = box;
        __threadfence();
    }
}

// ---- tensor-map copies ([Book-TMA] §"单 block、单 lane、单 tile 的 TMA load", §"TMA store",
//      §"TMA reduce，把“搬运”和“归约”合并"; [H200-TMA] §04 ②) ----------------------------------
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// L2 cache policies (createpolicy; the 64-bit policy rides on the copy's .L2::cache_hint operand).
// kL2Keep: no hint; kL2EvictFirst: the lines are the first candidates for eviction (bytes touched
// once: a stream then recycles its own lines instead of evicting other data); kL2EvictLast: the
// last.  The ring's tile loads use evict-first.  The store, reduce and bulk forms below take a
// policy as well, but no kernel passes one: on the streaming copies evict-first and evict-last
// measured no gain on GB300.
enum L2Hint : uint32_t { kL2Keep = 0, kL2EvictFirst = 1, kL2EvictLast = 2 };

__device__ __forceinline__ uint64_t l2_policy(uint32_t hint)
{
    uint64_t p = 0;
    if (hint == kL2EvictFirst) {
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    } else if (hint == kL2EvictLast) {
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    }
    return p;
}

// Global -> shared box load completing `box_bytes` on mbarrier `bar`; with H, its global reads
// carry the L2 policy `pol`.
#define TMK_LOAD_ASM(RANK, COORDS, BAR, ...)                                                     \
    if constexpr (H) {                                                                           \
        asm volatile("cp.async.bulk.tensor." RANK ".shared::cluster.global.tile"                 \
                     ".mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {" COORDS "}], [" \
                     BAR "], %" BAR_NEXT ";" ::"r"(dst), "l"(mp), __VA_ARGS__, "r"(bar),         \
                     "l"(pol) : "memory");                                                       \
    } else {                                                                                     \
        asm volatile("cp.async.bulk.tensor." RANK ".shared::cluster.global.tile"                 \
                     ".mbarrier::complete_tx::bytes [%0], [%1, {" COORDS "}], [" BAR "];"       \
                     ::"r"(dst), "l"(mp), __VA_ARGS__, "r"(bar) : "memory");                     \
    }

template <int R, bool H = false>
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* m, const int32_t* c,
                                         uint32_t bar, uint64_t pol = 0)
{
    const uint64_t mp = reinterpret_cast<uint64_t>(m);
    if constexpr (R == 1) {
#define BAR_NEXT "4"
        TMK_LOAD_ASM("1d", "%2", "%3", "r"(c[0]))
#undef BAR_NEXT
    } else if constexpr (R == 2) {
#define BAR_NEXT "5"
        TMK_LOAD_ASM("2d", "%2, %3", "%4", "r"(c[0]), "r"(c[1]))
#undef BAR_NEXT
    } else if constexpr (R == 3) {
#define BAR_NEXT "6"
        TMK_LOAD_ASM("3d", "%2, %3, %4", "%5", "r"(c[0]), "r"(c[1]), "r"(c[2]))
#undef BAR_NEXT
    } else if constexpr (R == 4) {
#define BAR_NEXT "7"
        TMK_LOAD_ASM("4d", "%2, %3, %4, %5", "%6", "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]))
#undef BAR_NEXT
    } else {
#define BAR_NEXT "8"
        TMK_LOAD_ASM("5d", "%2, %3, %4, %5, %6", "%7", "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]),
                     "r"(c[4]))
#undef BAR_NEXT
    }
}
#undef TMK_LOAD_ASM

// Shared -> global box store (only in-bounds elements are written), tracked by a bulk group; with
// H, its global writes carry the L2 policy `pol`.
#define TMK_STORE_ASM(RANK, COORDS, POL, ...)                                                    \
    if constexpr (H) {                                                                           \
        asm volatile("cp.async.bulk.tensor." RANK ".global.shared::cta.tile.bulk_group"          \
                     ".L2::cache_hint [%0, {" COORDS "}], [%1], " POL ";"                        \
                     ::"l"(mp), "r"(src), __VA_ARGS__, "l"(pol) : "memory");                     \
    } else {                                                                                     \
        asm volatile("cp.async.bulk.tensor." RANK ".global.shared::cta.tile.bulk_group"          \
                     " [%0, {" COORDS "}], [%1];" ::"l"(mp), "r"(src), __VA_ARGS__ : "memory");  \
    }

template <int R, bool H = false>
__device__ __forceinline__ void tma_store(const CUtensorMap* m, const int32_t* c, uint32_t src,
                                          uint64_t pol = 0)
{
    const uint64_t mp = reinterpret_cast<uint64_t>(m);
    if constexpr (R == 1) {
        TMK_STORE_ASM("1d", "%2", "%3", "r"(c[0]))
    } else if constexpr (R == 2) {
        TMK_STORE_ASM("2d", "%2, %3", "%4", "r"(c[0]), "r"(c[1]))
    } else if constexpr (R == 3) {
        TMK_STORE_ASM("3d", "%2, %3, %4", "%5", "r"(c[0]), "r"(c[1]), "r"(c[2]))
    } else if constexpr (R == 4) {
        TMK_STORE_ASM("4d", "%2, %3, %4, %5", "%6", "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]))
    } else {
        TMK_STORE_ASM("5d", "%2, %3, %4, %5, %6", "%7", "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]),
                      "r"(c[4]))
    }
}
#undef TMK_STORE_ASM

// Shared -> global element-wise reduction into the tensor, op OP = 0 add, 1 min, 2 max; the map's
// element type decides the arithmetic.  With H the global accesses carry the L2 policy `pol`.
#define TMK_RED_ASM(RANK, OPS, COORDS, POL, ...)                                                 \
    if constexpr (H) {                                                                           \
        asm volatile("cp.reduce.async.bulk.tensor." RANK ".global.shared::cta." OPS             \
                     ".tile.bulk_group.L2::cache_hint [%0, {" COORDS "}], [%1], " POL ";"        \
                     ::"l"(mp), "r"(src), __VA_ARGS__, "l"(pol) : "memory");                     \
    } else {                                                                                     \
        asm volatile("cp.reduce.async.bulk.tensor." RANK ".global.shared::cta." OPS             \
                     ".tile.bulk_group [%0, {" COORDS "}], [%1];"                                \
                     ::"l"(mp), "r"(src), __VA_ARGS__ : "memory");                               \
    }

template <int R, int OP, bool H = false>
__device__ __forceinline__ void tma_reduce(const CUtensorMap* m, const int32_t* c, uint32_t src,
                                           uint64_t pol = 0)
{
    const uint64_t mp = reinterpret_cast<uint64_t>(m);
    constexpr bool add = OP == 0, mn = OP == 1;
#define TMK_RED_OP(RANK, COORDS, POL, ...)                                                       \
    if constexpr (add) {                                                                         \
        TMK_RED_ASM(RANK, "add", COORDS, POL, __VA_ARGS__)                                       \
    } else if constexpr (mn) {                                                                   \
        TMK_RED_ASM(RANK, "min", COORDS, POL, __VA_ARGS__)                                       \
    } else {                                                                                     \
        TMK_RED_ASM(RANK, "max", COORDS, POL, __VA_ARGS__)                                       \
    }
    if constexpr (R == 1) {
        TMK_RED_OP("1d", "%2", "%3", "r"(c[0]))
    } else if constexpr (R == 2) {
        TMK_RED_OP("2d", "%2, %3", "%4", "r"(c[0]), "r"(c[1]))
    } else if constexpr (R == 3) {
        TMK_RED_OP("3d", "%2, %3, %4", "%5", "r"(c[0]), "r"(c[1]), "r"(c[2]))
    } else if constexpr (R == 4) {
        TMK_RED_OP("4d", "%2, %3, %4, %5", "%6", "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]))
    } else {
        TMK_RED_OP("5d", "%2, %3, %4, %5, %6", "%7", "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]),
                   "r"(c[4]))
    }
#undef TMK_RED_OP
}
#undef TMK_RED_ASM

// L2 prefetch of a 2-D box (no shared memory, no completion tracking).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* m, int32_t c0, int32_t c1)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 ::"l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1) : "memory");
}

// ---- untiled bulk copies (contiguous bytes; both addresses 16-byte aligned, size % 16 == 0;
//      with H the global accesses carry the L2 policy `pol`) ---------------------------------------
template <bool H = false>
__device__ __forceinline__ void bulk_load(uint32_t dst, uint64_t src, uint32_t bytes, uint32_t bar,
                                          uint64_t pol = 0)
{
    if constexpr (H) {
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
            " [%0], [%1], %2, [%3], %4;"
            ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
    } else {
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
            ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
    }
}

template <bool H = false>
__device__ __forceinline__ void bulk_store(uint64_t dst, uint32_t src, uint32_t bytes,
                                           uint64_t pol = 0)
{
    if constexpr (H) {
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
                     ::"l"(dst), "r"(src), "r"(bytes), "l"(pol) : "memory");
    } else {
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                     ::"l"(dst), "r"(src), "r"(bytes) : "memory");
    }
}

// ---- bulk async groups ([MLSys-TMA] §"如何等待 TMA store 完成": commit, then wait until the
//      source buffer may be reused) ---------------------------------------------------------------
__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// At most N committed groups may still be READING their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// At most N committed groups may still be in flight (writes included).
template <int N>
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ---- swizzle of an image byte offset (the hardware's placement; stages are 1024-byte aligned
//      so the image offset and the shared-memory address agree on bits 4..9).
//      [MLSys-TMA] §"用 3D TMA 搬运多个 swizzle atoms": 16-byte sector XOR (row % 8) in 128-byte rows;
//      64B / 32B use two / one row bits. ----------------------------------------------------------
__device__ __forceinline__ uint32_t swizzle_offset(uint32_t off, uint32_t span)
{
    const uint32_t bits = span == 128 ? 7u : span == 64 ? 3u : span == 32 ? 1u : 0u;
    return off ^ (((off >> 7) & bits) << 4);
}

// ---- box addressing ------------------------------------------------------------------------
// Grid box index -> per-dim box counters k[i] (dim 0 fastest).
__device__ __forceinline__ void grid_counters(const BoxWalk& w, uint64_t b, uint32_t* k)
{
#pragma unroll
    for (int i = 0; i < 5; i++) {
        if (i < (int)w.rank) {
            const uint64_t nb = w.grid_nb[i];
            const uint64_t q = b / nb;
            k[i] = (uint32_t)(b - q * nb);
            b = q;
        } else {
            k[i] = 0;
        }
    }
}

// The next grid box (odometer step of the counters).
__device__ __forceinline__ void grid_next(const BoxWalk& w, uint32_t* k)
{
#pragma unroll
    for (int i = 0; i < 5; i++) {
        if (i < (int)w.rank) {
            if (++k[i] < w.grid_nb[i]) return;
            k[i] = 0;
        }
    }
}

// Counters k += digits d, with carries (mixed radix: the grid's box counts).
__device__ __forceinline__ void grid_add(const BoxWalk& w, uint32_t* k, const uint32_t* d)
{
    uint32_t carry = 0;
#pragma unroll
    for (int i = 0; i < 5; i++) {
        if (i < (int)w.rank) {
            const uint64_t v = (uint64_t)k[i] + d[i] + carry;
            carry = v >= w.grid_nb[i] ? 1u : 0u;
            k[i] = (uint32_t)(carry ? v - w.grid_nb[i] : v);
        }
    }
}

// Start coordinates of the launch's box `b` (grid: k[i] * box[i] with dim 0 fastest).
__device__ __forceinline__ void box_start(const BoxWalk& w, uint64_t b, int32_t* c)
{
    if (w.mode == WALK_GRID) {
#pragma unroll
        for (int i = 0; i < 5; i++) {
            if (i < (int)w.rank) {
                const uint64_t nb = w.grid_nb[i];
                const uint64_t q = b / nb;
                c[i] = (int32_t)((b - q * nb) * w.box[i]);
                b = q;
            } else {
                c[i] = 0;
            }
        }
    } else {
        const int32_t* src = (w.mode == WALK_LIST) ? (w.list + b * w.rank) : (w.inl + b * w.rank);
#pragma unroll
        for (int i = 0; i < 5; i++) c[i] = i < (int)w.rank ? src[i] : 0;
    }
}

}  // namespace tmk
