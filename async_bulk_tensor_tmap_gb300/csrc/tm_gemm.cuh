// tm_gemm.cuh -- the one-SM tensor-core consumer of the k-ordered ring (C = A * B^T), shared by the
// library's stream_gemm and any separately built form that loads B differently.
//
// [MLSys-TMA] = mlc.ai "Modern GPU Programming for MLSys", chapter "异步数据搬运：TMA".  Overview:
// while the tensor cores work on the A and B tiles of step k, the next tiles must already be on
// their way into shared memory, and TMA writes them in the swizzled layout the MMA reads.
// §"把 TMA 放进 pipeline": stages are handed between the TMA producer and the MMA consumer with
// barriers.
//
// k_gemm_one_sm<BLoad>: a persistent CTA computes 128 x 256 tiles of C (fp32) from bf16 A (M x K)
// and B (N x K), both with K contiguous, streaming each (tile, k step) through an S-stage ring of
// 48 KiB stages (A 128 x 64 and B 256 x 64, 128-byte swizzled, one mbarrier per stage counting
// both tiles' bytes); two accumulators of 256 tensor-memory columns alternate between tiles:
//   warp 0  elected lane: the A tile's TMA load and BLoad::load_b for the B tile of each step
//   warp 1  owns the tensor memory; its elected lane issues four tcgen05.mma (K = 16 each) per
//           stage into an empty accumulator and hands the stage back with BLoad::release;
//           after a tile's last step it commits to the accumulator's full barrier
//   warps 2-5 read an accumulator with tcgen05.ld (each warp its 32-lane quarter), store the
//           in-bounds part of C and arrive on the accumulator's empty barrier
// BLoad supplies kShare (CTAs of a cluster that share each B tile: 1, or 2 for tiles 2m and
// 2m + 1), load_b (how the B tile reaches the stage) and release (how the stage's empty barrier
// learns that the MMAs are done with it; with kShare CTAs it counts kShare arrivals).
// Every wait is bounded; after one gives up the CTA still drains what it issued, reaches the final
// barrier and frees its tensor memory.
#pragma once

#include "tm_ptx.cuh"

namespace tmk {

namespace {

constexpr uint32_t kBM = 128, kBN = 256, kBK = 64, kUK = 16;
constexpr uint32_t kTileA = kBM * kBK * 2;         // 16 KiB
constexpr uint32_t kTileB = kBN * kBK * 2;         // 32 KiB
constexpr uint32_t kGemmStage = kTileA + kTileB;   // 48 KiB, a multiple of 1024
constexpr uint32_t kGemmThreads = 192;
constexpr uint32_t kTmemCols = kBN;                // fp32 accumulator: one column per N

// Instruction descriptor of tcgen05.mma kind::f16: D f32 (bits 4-5 = 1), A and B bf16 (bits 7-9
// and 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((kBN >> 3) << 17) |
                            ((kBM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major tile of 128-byte rows written by TMA with the
// 128-byte swizzle: start address >> 4 in bits 0-13, leading-dimension offset (unused for this
// layout) 16 bytes, stride between 8-row groups 1024 bytes >> 4 in bits 32-45, descriptor version 1
// in bits 46-47, swizzle mode 2 (128-byte) in bits 61-63.  The tile base is 1024-byte aligned, so
// the K = 16 steps inside a 128-byte row advance the start address by 32 bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_saddr, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (tensor memory) = A * B^T (+ D when accumulate != 0), A and B from shared-memory descriptors.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on the mbarrier once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar_saddr)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar_saddr)
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane (warp-wide, .32x32b shape).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
        "%30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of both CTAs of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// The shared::cluster address of this CTA's shared-memory location `saddr` in cluster CTA `rank`.
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Arrival on an mbarrier given by its shared::cluster address (possibly in the other CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr)
                 : "memory");
}

}  // namespace

template <class BLoad>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm_one_sm(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb,
                  const __grid_constant__ GemmArgs g)
{
    constexpr uint32_t kShare = BLoad::kShare;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kGemmMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kGemmMaxStages];
    __shared__ __align__(8) uint64_t acc_full[2];   // accumulator b holds a finished tile
    __shared__ __align__(8) uint64_t acc_empty[2];  // accumulator b has been read out
    __shared__ uint32_t tmem_slot;

    const uint32_t base = (smem_u32(smem_raw) + (kStageAlign - 1)) & ~(kStageAlign - 1);
    const uint32_t S = g.stages;
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Work units: tiles, or with kShare = 2 pairs of tiles (2 m, 2 m + 1; n) taken by the two
    // CTAs of a cluster (rank r takes row tile 2 m + r).  Unit u, u + units, ...: unit t is
    // (t % mgroups, t / mgroups), so the CTAs running together share B tiles (through L2, and
    // within a cluster through BLoad).
    const uint32_t rank = kShare > 1 ? cluster_rank() : 0u;
    const uint32_t unit = blockIdx.x / kShare, units = gridDim.x / kShare;
    const uint32_t mgroups = (g.mtiles + kShare - 1) / kShare;
    const uint32_t nunits = mgroups * g.ntiles;
    const uint32_t my_tiles = unit < nunits ? (nunits - 1 - unit) / units + 1 : 0;
    auto tile_of = [&](uint32_t i, uint32_t& mt, uint32_t& nt) {
        const uint32_t t = unit + i * units;
        mt = kShare * (t % mgroups) + rank;
        nt = t / mgroups;
    };

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; s++) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), kShare);  // released by the MMAs of every sharer
        }
        for (uint32_t b = 0; b < 2; b++) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 4);  // one arrival per epilogue warp
        }
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(&tmem_slot), 2 * kTmemCols);
    tc_fence_before();
    if constexpr (kShare > 1) {
        cluster_sync();  // every sharer's barriers exist before a copy or a commit reaches them
    } else {
        __syncthreads();
    }
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ---------------- producer: every (tile, k step) of this CTA through the ring ----------------
        if (elect_one()) {
            prefetch_tmap(&ma);
            prefetch_tmap(&mb);
            uint32_t s = 0, wraps = 0;
            uint64_t issued = 0;
            bool failed = false;
            for (uint32_t i = 0; i < my_tiles && !failed; i++) {
                uint32_t mt, nt;
                tile_of(i, mt, nt);
                for (uint32_t kb = 0; kb < g.kblocks; kb++) {
                    if (wraps > 0) {
                        const uint32_t parity = (wraps - 1) & 1u;
                        if (!mbar_wait(smem_u32(&empty_bar[s]), parity, g.timeout_ns)) {
                            record_timeout(g.status, K_GEMM, s, parity, unit + i * units);
                            failed = true;
                            break;
                        }
                    }
                    const uint32_t bar = smem_u32(&full_bar[s]);
                    const int32_t ca[2] = {(int32_t)(kb * kBK), (int32_t)(mt * kBM)};
                    mbar_arrive_expect_tx(bar, kGemmStage);  // the A and (all of) the B tile
                    tma_load<2>(base + s * kGemmStage, &ma, ca, bar);
                    BLoad::load_b(base + s * kGemmStage + kTileA, &mb, kb, nt, rank, bar);
                    issued++;
                    if (++s == S) {
                        s = 0;
                        wraps++;
                    }
                }
            }
            // Drain before shared memory goes away (bounded): after a failure the last loads may
            // still be landing; otherwise the MMA warp's last releases of the stages must land.
            for (uint64_t j = issued > S ? issued - S : 0; j < issued; j++) {
                const uint32_t js = (uint32_t)(j % S), jp = (uint32_t)((j / S) & 1);
                mbar_wait(smem_u32(failed ? &full_bar[js] : &empty_bar[js]), jp, g.timeout_ns);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (elect_one()) {
            uint32_t s = 0, phase = 0;
            bool failed = false;
            for (uint32_t i = 0; i < my_tiles && !failed; i++) {
                const uint32_t b = i & 1u;
                const uint32_t d = tmem + b * kTmemCols;
                if (i >= 2) {  // the epilogue has read out accumulator b's previous tile
                    const uint32_t parity = ((i >> 1) - 1) & 1u;
                    if (!mbar_wait(smem_u32(&acc_empty[b]), parity, g.timeout_ns)) {
                        record_timeout(g.status, K_GEMM, 8 + b, parity, i);
                        break;
                    }
                    tc_fence_after();
                }
                for (uint32_t kb = 0; kb < g.kblocks; kb++) {
                    if (!mbar_wait(smem_u32(&full_bar[s]), phase, g.timeout_ns)) {
                        record_timeout(g.status, K_GEMM, s, phase, i);
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = base + s * kGemmStage, b0 = a0 + kTileA;
#pragma unroll
                    for (uint32_t ks = 0; ks < kBK / kUK; ks++) {
                        mma_bf16(d, sw128_desc(a0 + ks * kUK * 2), sw128_desc(b0 + ks * kUK * 2),
                                 kIdesc, (kb | ks) != 0 ? 1u : 0u);
                    }
                    // the stage is free once these MMAs (of every sharer) have read it
                    BLoad::release(smem_u32(&empty_bar[s]));
                    if (++s == S) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
                // accumulator b is complete once every MMA issued so far has (after a failure: the
                // epilogue still gets its arrival, and the MMAs issued have completed)
                tc_commit(smem_u32(&acc_full[b]));
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warps 2-5, tensor-memory lane quarter warp % 4 ----------------
        const uint32_t q = warp & 3u;
        for (uint32_t i = 0; i < my_tiles; i++) {
            const uint32_t b = i & 1u;
            uint32_t mt, nt;
            tile_of(i, mt, nt);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&acc_full[b]), (i >> 1) & 1u,
                                                              g.timeout_ns));
            tc_fence_after();
            if (!ok) {
                if (lane == 0) record_timeout(g.status, K_GEMM, 10 + b, (i >> 1) & 1u, i);
                break;
            }
            const uint32_t row = mt * kBM + q * 32 + lane;
            float* const crow = g.c + (uint64_t)row * g.ldc;
            const uint32_t n0 = nt * kBN;
            for (uint32_t c0 = 0; c0 < kBN; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + b * kTmemCols + ((q * 32) << 16) + c0, r);
                if (row < g.m) {
                    const uint32_t n = n0 + c0;
                    if (n + 32 <= g.n) {
#pragma unroll
                        for (int v = 0; v < 8; v++) {
                            *reinterpret_cast<float4*>(crow + n + 4 * v) =
                                make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                            __uint_as_float(r[4 * v + 2]),
                                            __uint_as_float(r[4 * v + 3]));
                        }
                    } else {
#pragma unroll
                        for (int v = 0; v < 32; v++) {
                            if (n + v < g.n) crow[n + v] = __uint_as_float(r[v]);
                        }
                    }
                }
            }
            // this warp's reads of accumulator b are complete (tcgen05.wait::ld): hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acc_empty[b]));
        }
    }

    // Every tensor-memory read and every MMA has completed (and no copy or commit of a sharer is
    // still to reach this CTA): free the accumulators.
    tc_fence_before();
    if constexpr (kShare > 1) {
        cluster_sync();
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * kTmemCols);
    }
}


namespace {
template <class Kernel, class... Args>
cudaError_t launch_cluster2(Kernel k, uint32_t grid, size_t smem, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k, args...);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}
}  // namespace

}  // namespace tmk
