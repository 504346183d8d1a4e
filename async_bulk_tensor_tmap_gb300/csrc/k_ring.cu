// k_ring.cu -- the multi-stage producer/consumer ring that streams GEMM-operand-shaped tiles.
//
// [MLSys-TMA] = mlc.ai "Modern GPU Programming for MLSys", chapter "异步数据搬运：TMA".
// §"把 TMA 放进 pipeline": while the consumer reads stage s the TMA engine fills the next stage; the
// consumer waits for the load of a stage before reading it, and the producer waits until the
// consumer is done with a stage before overwriting it.  §"如何等待 TMA load 完成": the two operand
// tiles of a stage complete on ONE mbarrier whose expected byte count is their sum (2 x 2048 bytes
// there, 2 x 16 KiB for 128 x 64 bf16 tiles).
//
// The ring holds S stages of shared memory; to keep more bytes in flight than that, the producer
// also prefetches tiles a few iterations ahead into L2 (cp.async.bulk.prefetch.tensor), so that
// each stage's load finds its tiles in L2.
//
// CTA = 1 + G x 8 warps.  Warp 0: producer, one elected lane.  The consumers form G groups (G = 2
// when S is even, else 1); group g takes tiles g, g + G, g + 2G, ..., so it always meets the same
// S / G stages, and the per-tile chain of one group (reads, ordered sums, cross-warp combine)
// overlaps the other's.  In a group, 4 warps consume the A tile and 4 the B tile (fewer for tiles
// under 128 rows); each consumer warp takes whole 32-row blocks.  full[s] (count 1) completes
// when both tiles' bytes have landed; empty[s] (one arrival per warp of the stage's group) when
// that group has read the stage.  A group's per-warp partial sums meet in its own shared-memory
// slots guarded by one more mbarrier per slot (S / G + 1 slots: within a group no warp can be
// S / G of the group's iterations ahead of another, so a slot is never rewritten before it was
// read).  Every wait is bounded; no named barrier is used, so a warp that gives up cannot leave
// the others hanging.
//
// Consumer reads follow [MLSys-TMA] §"128-byte swizzle 的分组要求": lane l reads row l of a 32-row
// block; at any instant eight neighbouring lanes read the same logical sector c of eight
// consecutive rows, which the 128B swizzle has spread over physical sectors c XOR (row % 8): eight
// distinct bank sectors, no conflict.  With swizzle NONE the same reads all hit sector c (8-way
// conflict).  The same section's ungrouped control (a 256-byte row stride, so that consecutive
// rows sit two 128-byte swizzle rows apart) is reproduced by the row_pairs read order: lane l
// reads row 2 (l mod 16) + l / 16, so eight neighbouring lanes meet swizzle rows 0, 2, ..., 14
// and only four distinct sectors c XOR (2j mod 8) (2-way conflict).  A shuffle then hands each
// row's sum to lane (row), so the results do not depend on the read order.
//
// What the consumer computes (the pages leave it open): per tile, each row is summed in fp32 in
// logical element order starting from its first element; rows are combined by a pairwise-adjacent
// tree (xor-shuffles 1, 2, 4, 8, 16 inside each 32-row block, then pairs of blocks); plus the exact
// integer sum of the 16-bit patterns.  (The warps hold contiguous 32-row blocks in order, so the
// shuffle levels, the in-warp block pairs and the cross-warp pairs together form exactly the
// pairwise-adjacent tree over all rows.)
#include "tm_ptx.cuh"

namespace tmk {

// Timeline of the tracing build (see TM_TRACE_BUFFER), per CTA: slot 0 entry, 1 the producer's
// first tile pair issued, 2 + i the consumers done with tile i (its A checksum written; i < 56),
// 60 the producer's last tile issued, 61 the CTA's tile count (a number), 63 the CTA's last
// checksum written.
TM_TRACE_BUFFER(ring)

constexpr uint32_t kRingMaxStages = 8;
constexpr uint32_t kRingMaxWpt = 4;                 // consumer warps per tile
constexpr uint32_t kRingMaxGroups = 2;              // consumer groups (tiles i % groups)
constexpr uint32_t kRingSlots = kRingMaxStages + 1;  // reduction slots: one more than the stages
constexpr uint32_t kRingThreads = 32 * (1 + kRingMaxGroups * 2 * kRingMaxWpt);

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kRingThreads, 1)
    k_ring(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb,
           const __grid_constant__ RingArgs r)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kRingMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kRingMaxStages];
    __shared__ __align__(8) uint64_t red_bar[kRingMaxGroups][2][kRingSlots];
    __shared__ float red_cs[kRingMaxGroups][2][kRingSlots][kRingMaxWpt];
    __shared__ uint32_t red_bits[kRingMaxGroups][2][kRingSlots][kRingMaxWpt];

    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + (kStageAlign - 1)) & ~(kStageAlign - 1);
    const uint8_t* const stage0 = smem_raw + (base - raw);
    const uint32_t S = r.stages;
    const uint32_t G = r.groups;   // 1, or 2 when S is even
    const uint32_t NS = S / G + 1;  // reduction slots of a group: one more than its stages
    const uint32_t tile = r.tile_bytes;  // multiple of 1024
    const uint32_t wpt = r.rows >= 32 * kRingMaxWpt ? kRingMaxWpt : r.rows / 32;
    const uint32_t rpl = r.rows / (32 * wpt);  // rows per lane

    const uint64_t first = blockIdx.x;
    if (r.ntiles <= first) return;
    const uint64_t n_local = r.n_base + (first < r.n_rem ? 1u : 0u);
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        TM_STAMP(ring, 0);
        TM_TRACE_PUT(ring, 61, n_local);
    }

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; s++) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), 2 * wpt);
        }
        for (uint32_t g = 0; g < G; g++) {
            for (uint32_t s = 0; s < NS; s++) {
                mbar_init(smem_u32(&red_bar[g][0][s]), wpt);
                mbar_init(smem_u32(&red_bar[g][1][s]), wpt);
            }
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------- producer ----------------
        if (!elect_one()) return;
        prefetch_tmap(&ma);
        prefetch_tmap(&mb);
        // Tile counters of A and B (box along dim 0, box along dim 1) of tile `first + i * G`
        // (G = gridDim.x), stepped by G tiles with a carry: one cursor for the loads and one for the
        // optional L2 prefetch r.prefetch tiles ahead of them (no completion is tracked for those).
        struct TileCursor {
            uint64_t a0, a1, b0, b1;
        };
        const uint32_t a_d0 = r.a_d0, b_d0 = r.b_d0;  // the grid step, from the host
        const uint64_t a_d1 = r.a_d1, b_d1 = r.b_d1;
        auto cursor_at = [&](uint64_t i) {
            const uint64_t t = first + i * gridDim.x;
            return TileCursor{t % r.a_nb0, t / r.a_nb0, t % r.b_nb0, t / r.b_nb0};
        };
        auto advance = [&](TileCursor& c) {
            c.a0 += a_d0;
            c.a1 += a_d1;
            if (c.a0 >= r.a_nb0) {
                c.a0 -= r.a_nb0;
                c.a1++;
            }
            c.b0 += b_d0;
            c.b1 += b_d1;
            if (c.b0 >= r.b_nb0) {
                c.b0 -= r.b_nb0;
                c.b1++;
            }
        };
        // The first tile (t = blockIdx.x) in 32-bit divisions when the box counts fit: this runs
        // before the first load.
        TileCursor ld;
        if (r.a_nb0 <= 0xffffffffull && r.b_nb0 <= 0xffffffffull) {
            const uint32_t t = blockIdx.x, na = (uint32_t)r.a_nb0, nb = (uint32_t)r.b_nb0;
            ld = TileCursor{t % na, t / na, t % nb, t / nb};
        } else {
            ld = cursor_at(0);
        }
        TileCursor pf = ld;
        uint64_t pf_i = 0;
        auto prefetch_to = [&](uint64_t upto) {  // prefetch tiles pf_i .. min(upto, n_local) - 1
            for (; pf_i < upto && pf_i < n_local; pf_i++) {
                tma_prefetch_l2_2d(&ma, (int32_t)(pf.a0 * 64), (int32_t)(pf.a1 * r.rows));
                tma_prefetch_l2_2d(&mb, (int32_t)(pf.b0 * 64), (int32_t)(pf.b1 * r.rows));
                advance(pf);
            }
        };
        if (r.prefetch) {
            pf = cursor_at(S);
            pf_i = S;
            prefetch_to(r.prefetch);
        }
        // each tile is read once: an evict-first policy lets the stream recycle its own L2 lines
        // instead of pushing other data out of L2
        const uint64_t policy = l2_policy(kL2EvictFirst);
        uint32_t s = 0, wraps = 0;
        uint64_t i = 0;
        for (; i < n_local; i++) {
            if (wraps > 0) {
                const uint32_t parity = (wraps - 1) & 1u;
                if (!mbar_wait(smem_u32(&empty_bar[s]), parity, r.timeout_ns)) {
                    record_timeout(r.status, K_STREAM, s, parity, first + i * gridDim.x);
                    break;
                }
            }
            const uint32_t bar = smem_u32(&full_bar[s]);
            const int32_t ca[2] = {(int32_t)(ld.a0 * 64), (int32_t)(ld.a1 * r.rows)};
            const int32_t cb[2] = {(int32_t)(ld.b0 * 64), (int32_t)(ld.b1 * r.rows)};
            mbar_arrive_expect_tx(bar, 2 * tile);
            if (r.evict_first) {
                tma_load<2, true>(base + s * 2 * tile, &ma, ca, bar, policy);
                tma_load<2, true>(base + s * 2 * tile + tile, &mb, cb, bar, policy);
            } else {
                tma_load<2>(base + s * 2 * tile, &ma, ca, bar);
                tma_load<2>(base + s * 2 * tile + tile, &mb, cb, bar);
            }
            if (r.prefetch) prefetch_to(i + 1 + r.prefetch);
            if (i == 0) TM_STAMP(ring, 1);
            if (i + 1 == n_local) TM_STAMP(ring, 60);
            advance(ld);
            if (++s == S) {
                s = 0;
                wraps++;
            }
        }
        // Loads still landing (only after a failure): wait for them, bounded, before leaving.
        const uint64_t lo = i > S ? i - S : 0;
        for (uint64_t j = lo; j < i && i < n_local; j++) {
            mbar_wait(smem_u32(&full_bar[j % S]), (uint32_t)((j / S) & 1), r.timeout_ns);
        }
        return;
    }

    // ---------------- consumers: G groups of 2 * wpt warps; group g takes tiles g, g + G, ...;
    // in a group, wpt warps read A and the next wpt read B ----------------
    const uint32_t cw = warp - 1;
    if (cw >= G * 2 * wpt) return;  // launched but idle (small tiles)
    const uint32_t gidx = cw / (2 * wpt);
    const uint32_t cwg = cw % (2 * wpt);
    const uint32_t grp = cwg / wpt;  // 0 = A, 1 = B
    const uint32_t wi = cwg % wpt;   // warp index inside the tile
    float* const cs_out = grp == 0 ? r.cs_a : r.cs_b;
    unsigned long long* const bits_out = grp == 0 ? r.bits_a : r.bits_b;
    const uint32_t xr = r.swizzled ? 7u : 0u;
    const uint32_t lrow = r.row_pairs ? 2 * (lane & 15) + (lane >> 4) : lane;  // row read by this lane

    // Stage of tile i (i % S; S is a multiple of G, so the group cycles through S / G stages) and
    // its phase parity; the group's reduction slot (its own iteration count mod NS) and parity.
    uint32_t s = gidx, parity = 0;
    uint32_t slot = 0, slot_parity = 0;
    for (uint64_t i = gidx; i < n_local; i += G) {
        if (i != gidx) {
            s += G;
            if (s >= S) {
                s -= S;
                parity ^= 1u;
            }
            if (++slot == NS) {
                slot = 0;
                slot_parity ^= 1u;
            }
        }
        const bool ok = __all_sync(0xffffffffu,
                                   mbar_wait(smem_u32(&full_bar[s]), parity, r.timeout_ns));
        if (!ok) {
            if (lane == 0) record_timeout(r.status, K_STREAM, s, parity, first + i * gridDim.x);
            break;
        }
        const uint8_t* const t_img = stage0 + s * 2 * tile + grp * tile;

        // This warp's rows: 32-row blocks wi*rpl .. wi*rpl + rpl - 1, lane l row l of a block.
        // All of them are read into registers first; the stage is released as soon as the reads
        // are done (the arrive orders them before the producer's next write into the stage), and
        // the sums are formed afterwards.
        float blk[8];
        uint32_t bits = 0;
#pragma unroll
        for (uint32_t q0 = 0; q0 < 8; q0 += 2) {
            if (q0 < rpl) {
                uint4 v[2][8];
#pragma unroll
                for (uint32_t u = 0; u < 2; u++) {
                    const uint32_t row = 32 * (wi * rpl + q0 + u) + lrow;
                    const uint8_t* const rp = t_img + row * 128;
#pragma unroll
                    for (uint32_t c = 0; c < 8; c++) {
                        v[u][c] = (q0 + u < rpl)
                                      ? *reinterpret_cast<const uint4*>(rp + ((c ^ (row & xr)) << 4))
                                      : make_uint4(0, 0, 0, 0);
                    }
                }
                if (q0 + 2 >= rpl) {  // last rows of this warp read: release the stage
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
                }
#pragma unroll
                for (uint32_t u = 0; u < 2; u++) {
                    if (q0 + u < rpl) {
                        float acc = 0.f;
                        uint32_t lo16 = 0, hi16 = 0;
#pragma unroll
                        for (uint32_t c = 0; c < 8; c++) {
                            const uint32_t w[4] = {v[u][c].x, v[u][c].y, v[u][c].z, v[u][c].w};
#pragma unroll
                            for (int h = 0; h < 4; h++) {
                                acc = (c == 0 && h == 0) ? bf16lo(w[h])
                                                         : __fadd_rn(acc, bf16lo(w[h]));
                                acc = __fadd_rn(acc, bf16hi(w[h]));
                                lo16 += w[h] & 0xffffu;
                                hi16 += w[h] >> 16;
                            }
                        }
                        bits += lo16 + hi16;
                        blk[q0 + u] = acc;
                    }
                }
            }
        }

        // pairwise tree: inside each 32-row block by xor-shuffles, then across this warp's blocks
#pragma unroll
        for (uint32_t q = 0; q < 8; q++) {
            if (q < rpl) {
                float v = blk[q];
                // row_pairs: lane l held row 2 (l mod 16) + l / 16; hand lane l the sum of row l
                if (r.row_pairs) v = __shfl_sync(0xffffffffu, v, (lane & 1) * 16 + (lane >> 1));
#pragma unroll
                for (int m = 1; m < 32; m <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, m));
                blk[q] = v;
            }
        }
        for (uint32_t n = rpl; n > 1; n >>= 1) {
#pragma unroll
            for (uint32_t q = 0; q < 4; q++) {
                if (q < n / 2) blk[q] = __fadd_rn(blk[2 * q], blk[2 * q + 1]);
            }
        }
        bits = __reduce_add_sync(0xffffffffu, bits);  // exact integer sum: order-free

        // ... then across the tile's warps, in warp order (slots of iteration i % NS)
        if (lane == 0) {
            red_cs[gidx][grp][slot][wi] = blk[0];
            red_bits[gidx][grp][slot][wi] = bits;
            mbar_arrive(smem_u32(&red_bar[gidx][grp][slot]));
        }
        if (wi == 0 && lane == 0) {
            if (!mbar_wait(smem_u32(&red_bar[gidx][grp][slot]), slot_parity, r.timeout_ns)) {
                record_timeout(r.status, K_STREAM, slot, slot_parity, first + i * gridDim.x);
                break;
            }
            float part[kRingMaxWpt];
            unsigned long long total = 0;
            for (uint32_t w = 0; w < wpt; w++) {
                part[w] = red_cs[gidx][grp][slot][w];
                total += red_bits[gidx][grp][slot][w];
            }
            for (uint32_t n = wpt; n > 1; n >>= 1) {
                for (uint32_t q = 0; q < n / 2; q++) part[q] = __fadd_rn(part[2 * q], part[2 * q + 1]);
            }
            const uint64_t t = first + i * gridDim.x;
            cs_out[t] = part[0];
            bits_out[t] = total;
            if (grp == 0) {
                if (i < 56) TM_STAMP(ring, 2 + i);
                if (i + 1 == n_local) TM_STAMP(ring, 63);
            }
        }
    }
}

__global__ void k_selftest(uint64_t timeout_ns, StatusBlock* st)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    // Nothing ever arrives on `bar`: the wait must give up and report.
    if (!mbar_wait(smem_u32(&bar), 0, timeout_ns)) record_timeout(st, K_SELFTEST, 0, 0, 0);
}

cudaError_t launch_ring(const CUtensorMap* a, const CUtensorMap* b, const RingArgs& r,
                        uint32_t grid, size_t smem, cudaStream_t s)
{
    cudaError_t e =
        cudaFuncSetAttribute(k_ring, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const uint32_t wpt = r.rows >= 32 * kRingMaxWpt ? kRingMaxWpt : r.rows / 32;
    k_ring<<<grid, 32 * (1 + r.groups * 2 * wpt), smem, s>>>(*a, *b, r);
    return cudaGetLastError();
}

cudaError_t launch_selftest(uint64_t timeout_ns, StatusBlock* status, cudaStream_t s)
{
    k_selftest<<<1, 32, 0, s>>>(timeout_ns, status);
    return cudaGetLastError();
}

}  // namespace tmk
