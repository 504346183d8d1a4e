// k_gemm.cu -- the k-ordered ring feeding the 5th-generation tensor cores: C = A * B^T.
//
// [MLSys-TMA] = mlc.ai "Modern GPU Programming for MLSys", chapter "异步数据搬运：TMA".  Overview:
// while the tensor cores work on the A and B tiles of step k, the next tiles must already be on
// their way into shared memory, and TMA writes them in the swizzled layout the MMA reads.
// §"把 TMA 放进 pipeline": stages are handed between the TMA producer and the MMA consumer with
// barriers -- the consumer waits for a stage's bytes, the producer for the consumer to be done
// with a stage before refilling it.
//
// Two forms.  The one-SM form (k_gemm_one_sm in tm_gemm.cuh, instantiated here with each CTA
// loading its own B tile): a persistent CTA per SM computes 128 x 256 tiles through an S-stage ring
// of 48 KiB stages into two alternating tensor-memory accumulators.  The CTA-pair form below
// (k_gemm_pair): a cluster of two CTAs on two SMs computes 256 x 256 tiles with tcgen05
// cta_group::2, each CTA loading its 128-row halves of the A and B tiles.
// Every wait is bounded; after one gives up the CTA still drains what it issued, reaches the final
// barrier and frees its tensor memory.
#include "tm_gemm.cuh"

namespace tmk {

namespace {

// ---- the CTA-pair form (tcgen05 cta_group::2): M = 256 over two CTAs of a cluster ----------------
constexpr uint32_t kPairTileA = 128 * kBK * 2;     // each CTA's half of A: 128 rows, 16 KiB
constexpr uint32_t kPairTileB = 128 * kBK * 2;     // each CTA's half of B: 128 of the 256 rows
constexpr uint32_t kPairStage = kPairTileA + kPairTileB;  // 32 KiB per CTA
// M = 256 (>> 4 in bits 24-28), N = 256, the rest as kIdesc
constexpr uint32_t kPairIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((kBN >> 3) << 17) |
                                ((256u >> 4) << 24);
// the same with N = 128: a 256 x 128 half tile (each CTA holds 64 rows of B)
constexpr uint32_t kPairIdescHalf = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) |
                                    ((256u >> 4) << 24);

// TMA tensor load into this CTA's shared memory completing on an mbarrier of either CTA of the
// pair (given by its shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m, int32_t c0,
                                                 int32_t c1, uint32_t bar_caddr)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar_caddr)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_saddr, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D (both CTAs' tensor memory) = A * B^T (+ D), A's and B's halves at the same shared-memory
// offsets in the two CTAs.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on the mbarrier at offset bar_saddr in both CTAs of the pair once every tcgen05
// operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar_saddr)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar_saddr),
        "h"((uint16_t)0x3)
        : "memory");
}

}  // namespace

// The CTA-pair form: a cluster of two CTAs (ranks 0 and 1, two SMs) computes 256 x 256 tiles of C.
// Per k step each CTA loads its 128-row half of the A tile and its 128-row half of the B tile into
// its own 32 KiB stage (so 7 stages fit), both CTAs' loads completing on the leader's (rank 0) full
// barrier.  The leader's elected lane issues tcgen05.mma.cta_group::2 (M = 256: A rows 0-127 from
// the leader's shared memory, 128-255 from the peer's at the same offset, B split the same way;
// each CTA's 128 rows of the accumulator land in its own tensor memory), and its commits arrive
// on the empty and accumulator-full barriers of both CTAs.  Each CTA's epilogue reads its own half
// and hands the accumulator back with arrivals on the leader's accumulator-empty barrier.
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb,
                const __grid_constant__ CUtensorMap mbq, const __grid_constant__ GemmArgs g)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kGemmMaxPairStages];   // the leader's are used
    __shared__ __align__(8) uint64_t empty_bar[kGemmMaxPairStages];
    __shared__ __align__(8) uint64_t acc_full[2];
    __shared__ __align__(8) uint64_t acc_empty[2];                   // the leader's are used
    __shared__ uint32_t tmem_slot;

    const uint32_t base = (smem_u32(smem_raw) + (kStageAlign - 1)) & ~(kStageAlign - 1);
    const uint32_t S = g.stages;
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const uint32_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const uint32_t ntiles = g.mtiles * g.ntiles;  // 256 x 256 tiles; tile t = (t % mtiles, t / mtiles)
    // Tiles below split_from are done whole, round-robin over the pairs; the rest (a last wave that
    // would leave pairs idle) as two 256 x 128 halves each, round-robin too.
    const uint32_t split = g.split_from;
    const uint32_t halves = 2 * (ntiles - split);
    const uint32_t nfull = pair < split ? (split - 1 - pair) / npairs + 1 : 0;
    const uint32_t nhalf = pair < halves ? (halves - 1 - pair) / npairs + 1 : 0;
    const uint32_t my_tiles = nfull + nhalf;
    // work item i of this pair: its tile (mt, nt) and half (0 or 1: columns half * 128 .. + 127 of
    // the tile; 2: the whole tile)
    auto item = [&](uint32_t i, uint32_t& mt, uint32_t& nt, uint32_t& half) {
        uint32_t t;
        if (i < nfull) {
            t = pair + i * npairs;
            half = 2;
        } else {
            const uint32_t hh = pair + (i - nfull) * npairs;
            t = split + (hh >> 1);
            half = hh & 1u;
        }
        mt = t % g.mtiles;
        nt = t / g.mtiles;
    };

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; s++) {
            mbar_init(smem_u32(&full_bar[s]), 1);   // the leader's expect_tx (both CTAs' bytes)
            mbar_init(smem_u32(&empty_bar[s]), 1);
        }
        for (uint32_t b = 0; b < 2; b++) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 8);  // four epilogue warps in each CTA
        }
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(&tmem_slot), 2 * kTmemCols);
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers are initialised and their tensor memory allocated
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t leader_full = peer_addr(smem_u32(&full_bar[0]), 0);         // + 8 * stage
    const uint32_t leader_acc_empty = peer_addr(smem_u32(&acc_empty[0]), 0);   // + 8 * buffer

    if (warp == 0) {
        // ---------------- producer (both CTAs): this CTA's halves of every step ----------------
        if (elect_one()) {
            prefetch_tmap(&ma);
            prefetch_tmap(&mb);
            prefetch_tmap(&mbq);
            uint32_t s = 0, wraps = 0;
            uint64_t issued = 0;
            bool failed = false;
            for (uint32_t i = 0; i < my_tiles && !failed; i++) {
                uint32_t mt, nt, half;
                item(i, mt, nt, half);
                const uint32_t t = i;  // reported with a timeout
                const uint32_t bytes = half == 2 ? 2 * kPairStage : 2 * (kPairTileA + kPairTileB / 2);
                for (uint32_t kb = 0; kb < g.kblocks; kb++) {
                    if (wraps > 0) {
                        const uint32_t parity = (wraps - 1) & 1u;
                        if (!mbar_wait(smem_u32(&empty_bar[s]), parity, g.timeout_ns)) {
                            record_timeout(g.status, K_GEMM, s, parity, t);
                            failed = true;
                            break;
                        }
                    }
                    // Only the leader arms the stage, for both CTAs' bytes; the peer's loads
                    // complete on the leader's barrier.  They cannot land on an earlier phase:
                    // the peer refills stage s only after the MMAs of the previous round, which
                    // waited for that phase to complete, have released it.  (A peer arrival per
                    // stage, a cluster-scope release, halved the rate.)
                    const uint32_t fb = leader_full + 8 * s;
                    if (rank == 0) mbar_arrive_expect_tx(smem_u32(&full_bar[s]), bytes);
                    tma_load_2d_pair(base + s * kPairStage, &ma, (int32_t)(kb * kBK),
                                     (int32_t)(mt * 256 + rank * 128), fb);
                    if (half == 2) {
                        tma_load_2d_pair(base + s * kPairStage + kPairTileA, &mb, (int32_t)(kb * kBK),
                                         (int32_t)(nt * 256 + rank * 128), fb);
                    } else {  // this CTA's 64 of the half tile's 128 B rows
                        tma_load_2d_pair(base + s * kPairStage + kPairTileA, &mbq, (int32_t)(kb * kBK),
                                         (int32_t)(nt * 256 + half * 128 + rank * 64), fb);
                    }
                    issued++;
                    if (++s == S) {
                        s = 0;
                        wraps++;
                    }
                }
            }
            // Drain before shared memory goes away (bounded).  Normally: the leader's last releases
            // of the stages must land here.  After a failure: the loads still in flight complete on
            // the leader's full barriers, which the leader waits for.
            for (uint64_t j = issued > S ? issued - S : 0; j < issued; j++) {
                const uint32_t js = (uint32_t)(j % S), jp = (uint32_t)((j / S) & 1);
                if (!failed) mbar_wait(smem_u32(&empty_bar[js]), jp, g.timeout_ns);
                else if (rank == 0) mbar_wait(smem_u32(&full_bar[js]), jp, g.timeout_ns);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (the leader only) ----------------
        if (rank == 0 && elect_one()) {
            uint32_t s = 0, phase = 0;
            bool failed = false;
            for (uint32_t i = 0; i < my_tiles && !failed; i++) {
                const uint32_t b = i & 1u;
                const uint32_t d = tmem + b * kTmemCols;
                uint32_t mt, nt, half;
                item(i, mt, nt, half);
                const uint32_t idesc = half == 2 ? kPairIdesc : kPairIdescHalf;
                if (i >= 2) {  // both CTAs' epilogues have read out accumulator b's previous tile
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
                    const uint32_t a0 = base + s * kPairStage, b0 = a0 + kPairTileA;
#pragma unroll
                    for (uint32_t ks = 0; ks < kBK / kUK; ks++) {
                        mma_bf16_pair(d, sw128_desc(a0 + ks * kUK * 2), sw128_desc(b0 + ks * kUK * 2),
                                      idesc, (kb | ks) != 0 ? 1u : 0u);
                    }
                    tc_commit_pair(smem_u32(&empty_bar[s]));  // both CTAs' stage s is free once read
                    if (++s == S) {
                        s = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit_pair(smem_u32(&acc_full[b]));
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (both CTAs): this CTA's 128 rows of each tile ----------------
        const uint32_t q = warp & 3u;
        for (uint32_t i = 0; i < my_tiles; i++) {
            const uint32_t b = i & 1u;
            uint32_t mt, nt, half;
            item(i, mt, nt, half);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&acc_full[b]), (i >> 1) & 1u,
                                                              g.timeout_ns));
            tc_fence_after();
            if (!ok) {
                if (lane == 0) record_timeout(g.status, K_GEMM, 10 + b, (i >> 1) & 1u, i);
                break;
            }
            const uint32_t row = mt * 256 + rank * 128 + q * 32 + lane;
            float* const crow = g.c + (uint64_t)row * g.ldc;
            const uint32_t n0 = nt * kBN + (half == 2 ? 0u : half * 128u);
            const uint32_t ncols = half == 2 ? kBN : 128u;
            for (uint32_t c0 = 0; c0 < ncols; c0 += 32) {
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
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(leader_acc_empty + 8 * b);
        }
    }

    // Both CTAs are done: no MMA reads either CTA's shared memory any more, every arrival has been
    // made; free the accumulators (both CTAs, as they were allocated).
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 2 * kTmemCols);
    }
}

namespace {
// The library's one-SM form: each CTA loads its whole B tile itself (CTAs running together share
// B tiles through L2) and releases a stage with one commit of its MMAs.
struct OwnB {
    static constexpr uint32_t kShare = 1;
    __device__ static void load_b(uint32_t dst, const CUtensorMap* mb, uint32_t kb, uint32_t nt,
                                  uint32_t /*rank*/, uint32_t bar)
    {
        const int32_t cb[2] = {(int32_t)(kb * kBK), (int32_t)(nt * kBN)};
        tma_load<2>(dst, mb, cb, bar);
    }
    __device__ static void release(uint32_t empty_bar) { tc_commit(empty_bar); }
};
}  // namespace

cudaError_t launch_gemm(const CUtensorMap* a, const CUtensorMap* b, const GemmArgs& g,
                        uint32_t grid, size_t smem, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(k_gemm_one_sm<OwnB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_gemm_one_sm<OwnB><<<grid, kGemmThreads, smem, s>>>(*a, *b, g);
    return cudaGetLastError();
}

cudaError_t launch_gemm_pair(const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* b_quarter,
                             const GemmArgs& g, uint32_t grid, size_t smem, cudaStream_t s)
{
    cudaError_t e =
        cudaFuncSetAttribute(k_gemm_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_cluster2(k_gemm_pair, grid, smem, s, *a, *b, *b_quarter, g);
}

}  // namespace tmk
