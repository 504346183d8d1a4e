// k_tma.cu -- persistent TMA streaming kernels: tiled copy, round trip and fp32 reduce-add.
//
// One CTA is one warp; its elected lane issues everything ([MLSys-TMA] = mlc.ai "Modern GPU
// Programming for MLSys", chapter "异步数据搬运：TMA", §"一个 thread 如何描述整个 tile": a single
// thread submits the copy, the engine does the addressing).  The lane walks the launch's boxes
// blockIdx.x, blockIdx.x + gridDim.x, ... through an S-stage ring of 1024-byte aligned shared-memory
// stages:
//
//   load   box i into stage i % S       (mbarrier arrive.expect_tx + complete_tx, §"如何等待 TMA
//                                         load 完成")
//   wait   full[i % S] for parity (i / S) & 1           -- bounded
//   write  stage i % S out, commit a bulk group          (§"如何等待 TMA store 完成")
//   refill stage (i - 1) % S with box i - 1 + S once the bulk group of box i - 1 has finished
//          READING shared memory (wait_group.read 1): the write of box i stays in flight.
//
// The three kinds differ only in the two copy instructions:
//   copy       load = tensor load of the box;  write = 1-D bulk store of the image (tile-major)
//   round trip load = 1-D bulk load of image b; write = tensor store through the map
//   reduce     load = tensor load of src;      write = tensor reduce-add into dst
// ([Book-TMA] = fangpin "gpu-hpc-book" ch. 08 "Cuda TMA", §"TMA store" and §"TMA reduce，把“搬运”
// 和“归约”合并" show the single-tile forms of the last two.)
#include "tm_ptx.cuh"

namespace tmk {

template <int R, int KIND>
__global__ void __launch_bounds__(32, 1)
    k_tma_stream(const __grid_constant__ CUtensorMap in_map,
                 const __grid_constant__ CUtensorMap out_map, const __grid_constant__ StreamArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[TM_MAX_STAGES];

    if (!elect_one()) return;

    const uint64_t first = blockIdx.x;
    if (a.walk.nbox <= first) return;
    const uint64_t n_local = (a.walk.nbox - 1 - first) / gridDim.x + 1;
    const uint32_t S = a.stages;
    const uint32_t base = (smem_u32(smem_raw) + (kStageAlign - 1)) & ~(kStageAlign - 1);

    if constexpr (KIND != KIND_ROUNDTRIP) prefetch_tmap(&in_map);
    if constexpr (KIND != KIND_COPY) prefetch_tmap(&out_map);
    for (uint32_t s = 0; s < S; s++) mbar_init(smem_u32(&full_bar[s]), 1);
    fence_barrier_init();

    auto box_of = [&](uint64_t i) -> uint64_t { return first + i * gridDim.x; };

    auto issue = [&](uint64_t i) {
        const uint32_t s = (uint32_t)(i % S);
        const uint32_t bar = smem_u32(&full_bar[s]);
        const uint32_t dst = base + s * a.stage_bytes;
        const uint64_t b = box_of(i);
        mbar_arrive_expect_tx(bar, a.box_bytes);
        if constexpr (KIND == KIND_ROUNDTRIP) {
            bulk_load(dst, a.images + b * a.box_bytes, a.box_bytes, bar);
        } else {
            int32_t c[5];
            box_start(a.walk, b, c);
            tma_load<R>(dst, &in_map, c, bar);
        }
    };

    auto write_out = [&](uint64_t i) {
        const uint32_t s = (uint32_t)(i % S);
        const uint32_t src = base + s * a.stage_bytes;
        const uint64_t b = box_of(i);
        if constexpr (KIND == KIND_COPY) {
            bulk_store(a.images + b * a.box_bytes, src, a.box_bytes);
        } else {
            int32_t c[5];
            box_start(a.walk, b, c);
            if constexpr (KIND == KIND_ROUNDTRIP) {
                tma_store<R>(&out_map, c, src);
            } else {
                tma_reduce_add<R>(&out_map, c, src);
            }
        }
        bulk_commit();
    };

    uint64_t issued = 0;
    while (issued < n_local && issued < S) issue(issued++);

    for (uint64_t i = 0; i < n_local; i++) {
        const uint32_t s = (uint32_t)(i % S);
        const uint32_t parity = (uint32_t)((i / S) & 1);
        if (!mbar_wait(smem_u32(&full_bar[s]), parity, a.timeout_ns)) {
            const uint32_t kid = KIND == KIND_COPY ? K_COPY : KIND == KIND_ROUNDTRIP ? K_ROUNDTRIP
                                                                                    : K_REDUCE;
            record_timeout(a.status, kid, s, parity, box_of(i));
            // Let every load still in flight land (bounded) before the stages go away.
            for (uint64_t j = i + 1; j < issued; j++) {
                mbar_wait(smem_u32(&full_bar[j % S]), (uint32_t)((j / S) & 1), a.timeout_ns);
            }
            break;
        }
        write_out(i);
        if (i >= 1 && issued < n_local) {
            bulk_wait_read<1>();  // box i - 1's write has read its stage
            issue(issued++);
        }
    }
    bulk_wait_all<0>();
}

template <int R>
static cudaError_t launch_rank(int kind, const CUtensorMap* in_map, const CUtensorMap* out_map,
                               const StreamArgs& a, uint32_t grid, size_t smem, cudaStream_t s)
{
    void (*fn)(const CUtensorMap, const CUtensorMap, const StreamArgs) =
        kind == KIND_COPY        ? k_tma_stream<R, KIND_COPY>
        : kind == KIND_ROUNDTRIP ? k_tma_stream<R, KIND_ROUNDTRIP>
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
