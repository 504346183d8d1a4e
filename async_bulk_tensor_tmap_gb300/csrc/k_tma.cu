// k_tma.cu -- persistent TMA streaming kernels: tiled copy, round trip and fp32 reduce-add.
//
// One CTA is one warp; its elected lane issues everything ([MLSys-TMA] = mlc.ai "Modern GPU
// Programming for MLSys", chapter "异步数据搬运：TMA", §"一个 thread 如何描述整个 tile": a single
// thread submits the copy, the engine does the addressing).  Boxes are taken in groups of G
// consecutive boxes sharing a stage (G > 1 for boxes well under a stage), each in a slot that
// starts on its swizzle period (1024 / 512 / 256 bytes for 128B / 64B / 32B, 128 without), so that
// each image in a stage keeps the swizzle phase it has in its own image; the lane walks the
// groups blockIdx.x, blockIdx.x + gridDim.x, ... through an S-stage ring of 1024-byte aligned
// shared-memory stages:
//
//   load   group i into stage i % S     (one mbarrier, arrive.expect_tx of the group's bytes, one
//                                         complete_tx per box, §"如何等待 TMA load 完成")
//   wait   full[i % S] for parity (i / S) & 1           -- bounded
//   write  stage i % S out, commit a bulk group          (§"如何等待 TMA store 完成")
//   refill stage (i - 1) % S with group i - 1 + S once the bulk group of group i - 1 has finished
//          READING shared memory (wait_group.read 1): the write of group i stays in flight
//          (with a single stage, the stage of group i once its own write has read it).
//
// The lane keeps two cursors over its groups, one for loads (running up to S groups ahead) and
// one for writes: each holds the stage, its phase parity and, for a grid walk, the box counters of
// the group's first box, stepped by G * gridDim.x boxes with carries; the boxes inside a group are
// stepped with an odometer.  No 64-bit division is left on the issue path.
//
// The three kinds differ only in the two copy instructions:
//   copy       load = tensor load of the box;  write = 1-D bulk store of the image (tile-major)
//   round trip load = 1-D bulk load of image b; write = tensor store through the map
//   reduce     load = tensor load of src;      write = tensor reduce (add, min or max) into dst
// ([Book-TMA] = fangpin "gpu-hpc-book" ch. 08 "Cuda TMA", §"TMA store" and §"TMA reduce，把“搬运”
// 和“归约”合并" show the single-tile forms of the last two.)
#include "tm_ptx.cuh"

namespace tmk {

// Counters of box b of the grid (as grid_counters), with 32-bit divisions whenever b and the box
// counts fit in 32 bits: this runs before a CTA's first load.
__device__ __forceinline__ void first_counters(const BoxWalk& w, uint64_t b, uint32_t* k)
{
    bool narrow = b <= 0xffffffffull;
#pragma unroll
    for (int i = 0; i < 5; i++) narrow = narrow && w.grid_nb[i] <= 0xffffffffull;
    if (!narrow) {
        grid_counters(w, b, k);
        return;
    }
    uint32_t x = (uint32_t)b;
#pragma unroll
    for (int i = 0; i < 5; i++) {
        if (i < (int)w.rank) {
            const uint32_t nb = (uint32_t)w.grid_nb[i];
            const uint32_t q = x / nb;
            k[i] = x - q * nb;
            x = q;
        } else {
            k[i] = 0;
        }
    }
}

template <int R, int KIND>
__global__ void __launch_bounds__(32, 1)
    k_tma_stream(const __grid_constant__ CUtensorMap in_map,
                 const __grid_constant__ CUtensorMap out_map, const __grid_constant__ StreamArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[TM_MAX_STAGES];

    if (!elect_one()) return;

    // Work unit: a group of `a.group` consecutive boxes sharing one stage (their images are
    // consecutive in the tile-major buffer as well).
    const uint64_t G = a.group;
    const uint64_t first = blockIdx.x;
    if (a.ngroups <= first) return;
    const uint64_t n_local = a.n_base + (first < a.n_rem ? 1u : 0u);
    const uint32_t S = a.stages;
    const uint32_t base = (smem_u32(smem_raw) + (kStageAlign - 1)) & ~(kStageAlign - 1);

    if constexpr (KIND != KIND_ROUNDTRIP) prefetch_tmap(&in_map);
    if constexpr (KIND != KIND_COPY) prefetch_tmap(&out_map);
    for (uint32_t s = 0; s < S; s++) mbar_init(smem_u32(&full_bar[s]), 1);
    fence_barrier_init();

    const bool grid = a.walk.mode == WALK_GRID;
    auto group_of = [&](uint64_t i) -> uint64_t { return first + i * gridDim.x; };
    auto count_of = [&](uint64_t g) -> uint32_t {
        const uint64_t b0 = g * G;
        return (uint32_t)(a.walk.nbox - b0 < G ? a.walk.nbox - b0 : G);
    };

    // Group i of this CTA: its stage, the phase parity of that stage's barrier, and (grid walks)
    // the counters of its first box.
    struct Cursor {
        uint64_t i;
        uint32_t s, phase;
        uint32_t k[5];
    };
    const uint32_t* const dstep = a.dstep;  // digits of G * gridDim.x boxes (from the host)
    Cursor ld{0, 0, 0, {0, 0, 0, 0, 0}};
    if (grid) first_counters(a.walk, first * G, ld.k);
    Cursor wr = ld;
    auto advance = [&](Cursor& c) {
        c.i++;
        if (++c.s == S) {
            c.s = 0;
            c.phase ^= 1u;
        }
        if (grid) grid_add(a.walk, c.k, dstep);
    };

    // Calls fn(j, coords) for the boxes of the cursor's group, in order.
    auto for_boxes = [&](const Cursor& c, auto&& fn) {
        const uint64_t g = group_of(c.i);
        const uint32_t cnt = count_of(g);
        int32_t co[5];
        if (grid) {
            uint32_t k[5];
#pragma unroll
            for (int d = 0; d < 5; d++) k[d] = c.k[d];
            for (uint32_t j = 0; j < cnt; j++) {
#pragma unroll
                for (int d = 0; d < 5; d++) co[d] = (int32_t)(k[d] * a.walk.box[d]);
                fn(j, co);
                grid_next(a.walk, k);
            }
        } else {
            for (uint32_t j = 0; j < cnt; j++) {
                box_start(a.walk, g * G + j, co);
                fn(j, co);
            }
        }
    };

    // Box j of a stage sits at j * slot_bytes: boxes smaller than their swizzle period get padded
    // slots so that each image starts its own swizzle phase; then the images are not contiguous
    // in the stage and move one bulk copy per box.
    const uint32_t slot = a.slot_bytes;
    const bool dense = slot == a.box_bytes;
    auto issue = [&](const Cursor& c) {
        const uint32_t bar = smem_u32(&full_bar[c.s]);
        const uint32_t dst = base + c.s * a.stage_bytes;
        const uint64_t g = group_of(c.i);
        const uint32_t cnt = count_of(g);
        mbar_arrive_expect_tx(bar, cnt * a.box_bytes);
        if constexpr (KIND == KIND_ROUNDTRIP) {
            if (dense) {
                bulk_load(dst, a.images + g * G * a.box_bytes, cnt * a.box_bytes, bar);
            } else {
                for (uint32_t j = 0; j < cnt; j++)
                    bulk_load(dst + j * slot, a.images + (g * G + j) * a.box_bytes, a.box_bytes, bar);
            }
        } else {
            for_boxes(c, [&](uint32_t j, const int32_t* co) {
                tma_load<R>(dst + j * slot, &in_map, co, bar);
            });
        }
    };

    auto write_out = [&](const Cursor& c) {
        const uint32_t src = base + c.s * a.stage_bytes;
        const uint64_t g = group_of(c.i);
        if constexpr (KIND == KIND_COPY) {
            if (dense) {
                bulk_store(a.images + g * G * a.box_bytes, src, count_of(g) * a.box_bytes);
            } else {
                const uint32_t cnt = count_of(g);
                for (uint32_t j = 0; j < cnt; j++)
                    bulk_store(a.images + (g * G + j) * a.box_bytes, src + j * slot, a.box_bytes);
            }
        } else {
            for_boxes(c, [&](uint32_t j, const int32_t* co) {
                if constexpr (KIND == KIND_ROUNDTRIP) {
                    tma_store<R>(&out_map, co, src + j * slot);
                } else {
                    tma_reduce<R, KIND - KIND_REDUCE>(&out_map, co, src + j * slot);
                }
            });
        }
        bulk_commit();
    };

    while (ld.i < n_local && ld.i < S) {
        issue(ld);
        advance(ld);
    }
    // Stage refilled after writing group i: the one group i - 1 used (its write may still be
    // reading), or with a single stage the one just written.
    const uint64_t lag = S > 1 ? 1 : 0;

    for (; wr.i < n_local; advance(wr)) {
        if (!mbar_wait(smem_u32(&full_bar[wr.s]), wr.phase, a.timeout_ns)) {
            const uint32_t kid = KIND == KIND_COPY ? K_COPY : KIND == KIND_ROUNDTRIP ? K_ROUNDTRIP
                                                                                    : K_REDUCE;
            record_timeout(a.status, kid, wr.s, wr.phase, group_of(wr.i) * G);
            // Let every load still in flight land (bounded) before the stages go away.
            for (uint64_t j = wr.i + 1; j < ld.i; j++) {
                mbar_wait(smem_u32(&full_bar[j % S]), (uint32_t)((j / S) & 1), a.timeout_ns);
            }
            break;
        }
        write_out(wr);
        if (wr.i >= lag && ld.i < n_local) {
            if (lag) {
                bulk_wait_read<1>();  // group i - 1's write has read its stage
            } else {
                bulk_wait_read<0>();  // the only stage: group i's write has read it
            }
            issue(ld);
            advance(ld);
        }
    }
    bulk_wait_all<0>();
}

template <int R>
static cudaError_t launch_rank(int kind, const CUtensorMap* in_map, const CUtensorMap* out_map,
                               const StreamArgs& a, uint32_t grid, size_t smem, cudaStream_t s)
{
    void (*fn)(const CUtensorMap, const CUtensorMap, const StreamArgs) =
        kind == KIND_COPY         ? k_tma_stream<R, KIND_COPY>
        : kind == KIND_ROUNDTRIP  ? k_tma_stream<R, KIND_ROUNDTRIP>
        : kind == KIND_REDUCE_MIN ? k_tma_stream<R, KIND_REDUCE_MIN>
        : kind == KIND_REDUCE_MAX ? k_tma_stream<R, KIND_REDUCE_MAX>
                                  : k_tma_stream<R, KIND_REDUCE>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    fn<<<grid, 32, smem, s>>>(*in_map, *out_map, a);
    return cudaGetLastError();
}

cudaError_t launch_tma_stream(int kind, uint32_t rank, const CUtensorMap* in_map,
                              const CUtensorMap* out_map, const StreamArgs& a, uint32_t grid,
                              size_t smem, cudaStream_t s)
{
    switch (rank) {
        case 1: return launch_rank<1>(kind, in_map, out_map, a, grid, smem, s);
        case 2: return launch_rank<2>(kind, in_map, out_map, a, grid, smem, s);
        case 3: return launch_rank<3>(kind, in_map, out_map, a, grid, smem, s);
        case 4: return launch_rank<4>(kind, in_map, out_map, a, grid, smem, s);
        case 5: return launch_rank<5>(kind, in_map, out_map, a, grid, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tmk
