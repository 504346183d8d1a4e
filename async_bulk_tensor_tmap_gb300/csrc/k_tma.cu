// k_tma.cu -- persistent TMA streaming kernels: tiled copy, round trip and tensor reduce (add, min, max).
//
// One CTA is one warp; its elected lane issues everything ([MLSys-TMA] = mlc.ai "Modern GPU
// Programming for MLSys", chapter "异步数据搬运：TMA", §"一个 thread 如何描述整个 tile": a single
// thread submits the copy, the engine does the addressing).  Boxes are taken in items of up to G
// consecutive boxes sharing a stage (G > 1 for boxes well under a stage), each in a slot that
// starts on its swizzle period (1024 / 512 / 256 bytes for 128B / 64B / 32B, 128 without), so that
// each image in a stage keeps the swizzle phase it has in its own image.  The items come from one
// of two splits: static (CTA c takes item c of every full wave of gridDim.x x G boxes, then its
// share of the tail, dealt out box by box: stream_item) or dynamic (a static prefix, then items
// from a counter of the launch's stream, so that faster CTAs take more; see next_item).  They
// pass through an S-stage ring of 1024-byte aligned shared-memory stages:
//
//   load   item i into stage i % S     (one mbarrier, arrive.expect_tx of the item's bytes, one
//                                        complete_tx per box, §"如何等待 TMA load 完成")
//   wait   full[i % S] for parity (i / S) & 1           -- bounded
//   write  stage i % S out, commit a bulk group          (§"如何等待 TMA store 完成")
//   refill stage (i - 1) % S with item i - 1 + S once the bulk group of item i - 1 has finished
//          READING shared memory (wait_group.read 1): the write of item i stays in flight
//          (with a single stage, the stage of item i once its own write has read it).
//
// Each stage records the item it holds (its first box, box count and, for a grid walk, the box
// counters of its first box), written when the loads are issued and read when the stage is
// written out.  The static split steps those counters by G * gridDim.x boxes with carries (the
// tail item's are found once, before the first load); the dynamic split decomposes each item's
// first box index (32-bit divisions when it fits); the boxes inside an item are stepped with an
// odometer.  The copy instructions carry no L2 policy: evict-first or evict-last policies on the
// loads or the writes measured no gain on GB300, and choosing between the policy and plain forms
// box by box cost the 512-byte-box copy a quarter of its issue rate.
//
// The three kinds differ only in the two copy instructions:
//   copy       load = tensor load of the box;  write = 1-D bulk store of the image (tile-major)
//   round trip load = 1-D bulk load of image b; write = tensor store through the map
//   reduce     load = tensor load of src;      write = tensor reduce (add, min or max) into dst
// ([Book-TMA] = fangpin "gpu-hpc-book" ch. 08 "Cuda TMA", §"TMA store" and §"TMA reduce，把“搬运”
// 和“归约”合并" show the single-tile forms of the last two.)
#include "tm_ptx.cuh"

namespace tmk {

// Timeline of the tracing build (see TM_TRACE_BUFFER), per CTA: slot 0 entry, 1 the first S items
// issued, 2 + i item i's stage complete (i < 58), 61 the CTA's item count (a number), 62 the last
// write issued, 63 exit (every write done).
TM_TRACE_BUFFER(stream)

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
    TM_STAMP(stream, 0);

    // Work unit: an item of up to G consecutive boxes sharing one stage (their images are
    // consecutive in the tile-major buffer as well).
    const uint32_t cta = blockIdx.x, grid_ctas = gridDim.x;
    const bool dyn = a.sched != nullptr;
    const uint64_t n_local = dyn ? 0 : stream_items(a, cta);  // static schedule only
    if (!dyn && n_local == 0) return;
    const uint32_t S = a.stages;
    const uint32_t G = a.group;
    const uint32_t base = (smem_u32(smem_raw) + (kStageAlign - 1)) & ~(kStageAlign - 1);

    if constexpr (KIND != KIND_ROUNDTRIP) prefetch_tmap(&in_map);
    if constexpr (KIND != KIND_COPY) prefetch_tmap(&out_map);
    for (uint32_t s = 0; s < S; s++) mbar_init(smem_u32(&full_bar[s]), 1);
    fence_barrier_init();

    const bool grid = a.walk.mode == WALK_GRID;

    // An item: its first box, its box count and (grid walks) the counters of its first box.  rec[s]
    // is the item stage s holds, written when its loads are issued, read when it is written out.
    struct Item {
        uint64_t b0;
        uint32_t cnt;
        uint32_t k[5];
    };
    Item rec[TM_MAX_STAGES];

    // The loads' source of items.  Static: this CTA's items of the host's schedule (stream_item),
    // their counters stepped by G * gridDim.x boxes with carries (the tail item's found once).
    // Dynamic: items g = 0 .. nitems - 1 of G boxes each (the last one short); CTA c first takes
    // c, c + gridDim.x, ... for its first S + 1 items (its first stages and their first refill),
    // then the items of the counter's fetches (dyn_fetch: batches of a.batch consecutive items,
    // single items past the first a.batched fetches).  The first batch is fetched right after
    // that first refill is issued, not before the first loads (all CTAs fetching at once made
    // every first stage 1.5 us late), and each further batch one batch ahead, right after a
    // stage's loads are issued: the producer's next arrive (a release) then finds the atomic long
    // done.  A CTA that runs faster than others takes more items.
    uint64_t si = 0;                        // static: the next item index of this CTA
    uint32_t sk[5] = {0, 0, 0, 0, 0};       // static: counters of item si - 1
    uint32_t tail_k[5] = {0, 0, 0, 0, 0};   // static: counters of the tail item's first box
    uint64_t dj = 0;                        // dynamic: items of the static prefix taken
    unsigned long long pend = 0;            // dynamic: the batch fetched ahead
    uint64_t bg = 0, bend = 0;              // dynamic: items bg .. bend - 1 of the current batch
    bool refetch = false;                   // dynamic: the batch ahead was taken: fetch another
    const uint64_t npre = (uint64_t)S + 1;  // static items per CTA before the counter
    const uint64_t prefix = npre * grid_ctas;
    bool first_fetch = dyn && prefix < a.nitems;
    if (!dyn && grid && a.waves > 0 && a.waves < n_local) {
        uint64_t tb;
        uint32_t tc;
        stream_item(a, cta, grid_ctas, a.waves, tb, tc);
        first_counters(a.walk, tb, tail_k);
    }
    auto next_item = [&](Item& it) -> bool {
        if (dyn) {
            uint64_t g;
            if (dj < npre) {
                // the static prefix (if it ends early, so do the items: nitems < prefix)
                g = cta + dj * grid_ctas;
                dj++;
                if (g >= a.nitems) return false;
            } else {
                if (bg == bend) {  // the current batch is done: take the one fetched ahead
                    uint64_t n;
                    dyn_fetch(a, prefix, (uint64_t)pend, bg, n);
                    if (bg >= a.nitems) return false;
                    bend = bg + n < a.nitems ? bg + n : a.nitems;
                    refetch = true;
                }
                g = bg++;
            }
            it.b0 = g * G;
            const uint64_t left = a.walk.nbox - it.b0;
            it.cnt = left < G ? (uint32_t)left : G;
            if (grid) first_counters(a.walk, it.b0, it.k);
            return true;
        }
        if (si >= n_local) return false;
        stream_item(a, cta, grid_ctas, si, it.b0, it.cnt);
        if (grid) {
            if (si == 0) {
                first_counters(a.walk, it.b0, sk);
            } else if (si < a.waves) {
                grid_add(a.walk, sk, a.dstep);
            } else {
#pragma unroll
                for (int d = 0; d < 5; d++) sk[d] = tail_k[d];
            }
#pragma unroll
            for (int d = 0; d < 5; d++) it.k[d] = sk[d];
        }
        si++;
        return true;
    };

    // Calls fn(j, coords) for the boxes of an item, in order.
    auto for_boxes = [&](const Item& it, auto&& fn) {
        int32_t co[5];
        if (grid) {
            uint32_t k[5];
#pragma unroll
            for (int d = 0; d < 5; d++) k[d] = it.k[d];
            for (uint32_t j = 0; j < it.cnt; j++) {
#pragma unroll
                for (int d = 0; d < 5; d++) co[d] = (int32_t)(k[d] * a.walk.box[d]);
                fn(j, co);
                grid_next(a.walk, k);
            }
        } else {
            for (uint32_t j = 0; j < it.cnt; j++) {
                box_start(a.walk, it.b0 + j, co);
                fn(j, co);
            }
        }
    };

    // Box j of a stage sits at j * slot_bytes: boxes smaller than their swizzle period get padded
    // slots so that each image starts its own swizzle phase; then the images are not contiguous
    // in the stage and move one bulk copy per box.
    const uint32_t slot = a.slot_bytes;
    const bool dense = slot == a.box_bytes;
    auto issue = [&](const Item& it, uint32_t s) {
        const uint32_t bar = smem_u32(&full_bar[s]);
        const uint32_t dst = base + s * a.stage_bytes;
        mbar_arrive_expect_tx(bar, it.cnt * a.box_bytes);
        if constexpr (KIND == KIND_ROUNDTRIP) {
            const uint64_t src = a.images + it.b0 * a.box_bytes;
            if (dense) {
                bulk_load(dst, src, it.cnt * a.box_bytes, bar);
            } else {
                for (uint32_t j = 0; j < it.cnt; j++)
                    bulk_load(dst + j * slot, src + j * a.box_bytes, a.box_bytes, bar);
            }
        } else {
            for_boxes(it, [&](uint32_t j, const int32_t* co) { tma_load<R>(dst + j * slot, &in_map, co, bar); });
        }
    };

    auto write_out = [&](const Item& it, uint32_t s) {
        const uint32_t src = base + s * a.stage_bytes;
        if constexpr (KIND == KIND_COPY) {
            const uint64_t dst = a.images + it.b0 * a.box_bytes;
            if (dense) {
                bulk_store(dst, src, it.cnt * a.box_bytes);
            } else {
                for (uint32_t j = 0; j < it.cnt; j++)
                    bulk_store(dst + j * a.box_bytes, src + j * slot, a.box_bytes);
            }
        } else {
            for_boxes(it, [&](uint32_t j, const int32_t* co) {
                if constexpr (KIND == KIND_ROUNDTRIP) {
                    tma_store<R>(&out_map, co, src + j * slot);
                } else {
                    tma_reduce<R, KIND - KIND_REDUCE>(&out_map, co, src + j * slot);
                }
            });
        }
        bulk_commit();
    };

    // Loads run up to S items ahead of the writes; the stage refilled after writing item w is the
    // one item w - 1 used (its write may still be reading), or with a single stage the one just
    // written.
    uint64_t issued = 0;
    uint32_t ls = 0;  // stage of the next load
    Item nx;
    bool have = true;
    while (issued < S && (have = next_item(nx))) {
        issue(nx, ls);
        rec[ls] = nx;
        issued++;
        ls = ls + 1 == S ? 0 : ls + 1;
    }
    TM_STAMP(stream, 1);
    const uint64_t lag = S > 1 ? 1 : 0;

    uint32_t ws = 0, wphase = 0;  // stage and phase parity of item w
    for (uint64_t w = 0; w < issued; w++) {
        if (!mbar_wait(smem_u32(&full_bar[ws]), wphase, a.timeout_ns)) {
            const uint32_t kid = KIND == KIND_COPY ? K_COPY : KIND == KIND_ROUNDTRIP ? K_ROUNDTRIP
                                                                                    : K_REDUCE;
            record_timeout(a.status, kid, ws, wphase, rec[ws].b0);
            // Let every load still in flight land (bounded) before the stages go away.
            for (uint64_t j = w + 1; j < issued; j++) {
                mbar_wait(smem_u32(&full_bar[j % S]), (uint32_t)((j / S) & 1), a.timeout_ns);
            }
            break;
        }
        if (w < 58) TM_STAMP(stream, 2 + w);
        write_out(rec[ws], ws);
        if (w >= lag && have && (have = next_item(nx))) {
            if (lag) {
                bulk_wait_read<1>();  // item w - 1's write has read its stage
            } else {
                bulk_wait_read<0>();  // the only stage: item w's write has read it
            }
            issue(nx, ls);
            rec[ls] = nx;
            issued++;
            ls = ls + 1 == S ? 0 : ls + 1;
            if (first_fetch && dj == npre) {  // after the prefix's last issue: the first batch
                pend = atomicAdd(a.sched, 1ull);
                first_fetch = false;
            } else if (refetch) {  // after the issue: the next batch, fetched while this item loads
                pend = atomicAdd(a.sched, 1ull);
                refetch = false;
            }
        }
        if (++ws == S) {
            ws = 0;
            wphase ^= 1u;
        }
    }
    TM_STAMP(stream, 62);
    TM_TRACE_PUT(stream, 61, issued);
    bulk_wait_all<0>();
    if (dyn) {
        // The launch's counter goes back to zero for the next launch on this stream: the last CTA
        // to get here knows that every CTA has made its last fetch.
        __threadfence();
        if (atomicAdd(a.sched + 1, 1ull) == (unsigned long long)grid_ctas - 1) {
            atomicExch(a.sched, 0ull);
            atomicExch(a.sched + 1, 0ull);
            __threadfence();
        }
    }
    TM_STAMP(stream, 63);
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
