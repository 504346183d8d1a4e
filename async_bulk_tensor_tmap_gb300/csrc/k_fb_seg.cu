// k_fb_seg.cu -- the segment form of the vector path: maps the tensor-map hardware cannot take (a
// stride or base that is not a multiple of 16 bytes), walked over their whole box grid with unit
// elementStrides; both directions (copy: tensor -> images; store: images -> tensor).
//
// What it computes is the same box image as the tensor-map load ([Book-TMA] §"Tensor descriptor：
// CUtensorMap": the box at the grid start, elements outside the tensor filled; [MLSys-TMA]
// §"用 3D TMA 搬运多个 swizzle atoms": 16-byte sectors placed at logical sector XOR (row % 8) in
// 128-byte rows), and for the store, only in-bounds elements written back.  How it moves the
// bytes follows the pages' asynchronous-copy design: contiguous bytes are staged by 1-D bulk
// copies completing on an mbarrier ([MLSys-TMA] §"如何等待 TMA load 完成") by one producer warp,
// and consumer warps realign them ([MLSys-TMA] §"把 TMA 放进 pipeline": full / empty barriers hand
// each stage between producer and consumers).
//
// Work unit (item): one block of image rows of a RUN, the run being all boxes along dim 0 of one
// position of the grid in dims 1 and up.  A run covers whole tensor rows, so no tensor byte is
// read twice; and when dim 1 is contiguous with dim 0 (stride[1] == dim[0] * esize, a reshaped
// view) the ibox[1] image rows of a box lie back to back in memory and form one SEGMENT of
// ibox[1] * dim[0] * esize bytes (one bulk copy instead of many 16-byte windows; the W4 rank-5
// view's segments are 2000 bytes).  Without that contiguity a segment is one tensor row.
//
// Copy: the producer stages item i's segments into buffer i % S once the consumers have released
// that buffer's previous item, and writes beside it each image row's offset in the buffer; the
// consumers read each 16-byte image chunk at its byte offset (the widest shared loads the offset
// allows), fill beyond the tensor, and store it with one 16-byte store to its swizzled place in
// the global image (a warp's 32 chunks are four whole 128-byte image rows).  Store: the producer
// stages the item's image blocks (contiguous in the images) and each row's tensor address; the
// consumers write each chunk's in-bounds bytes to the tensor.  Every mbarrier wait is bounded; a
// wait that gives up is reported and the CTA leaves after its copies in flight have landed.
//
// Measured on GB300 (W4 rank-5 view, 299 MB a call): copy 56.8 us against 79.3 for the per-window
// kernel (5.26 against 3.77 TB/s); store 64.9-66.2 against 71.4 us.  Two CTAs per SM with two
// staging buffers (the largest items) were best; CTA-wide barriers per item instead of the
// producer / consumer barriers, and bulk-stored image blocks, were slower.
#include "tm_ptx.cuh"

namespace tmk {

// Timeline of the tracing build (see TM_TRACE_BUFFER), per CTA: slot 0 entry, 62 the producer past
// the CTA's barrier initialisation, 60 its first item's row table written, 1 that item's bulk
// copies issued, 2 + n the first consumer warp done with item n (n < 58), 61 the CTA's item count
// (a number), 63 that warp done with its last item.  Shared by the copy and the store (one of
// them runs at a time).
TM_TRACE_BUFFER(seg)

// Consumer warps per CTA: W (SegArgs::cwarps picks 8, 12 or 16; kSegWarps unless TM_FB_SEG_WARPS
// says otherwise), plus one producer warp.
template <uint32_t W>
constexpr uint32_t seg_threads() { return 32 * (1 + W); }

namespace {

// Segment g of the run whose first box starts at c (c[0] = 0): its tensor address, the number of
// its image rows that lie in the tensor (0: none) and its length in bytes.
struct Segment {
    uint64_t src;
    uint32_t rows;
    uint32_t bytes;
};

__device__ __forceinline__ Segment segment_of(const SegArgs& s, const int32_t* c, uint32_t g)
{
    const FbArgs& a = s.f;
    int64_t off = 0;
    bool ok = true;
    uint32_t r = g;
#pragma unroll
    for (int i = 1; i < 5; i++) {
        if (i >= (int)s.outer0 && i < (int)a.walk.rank) {
            const uint32_t bi = a.ibox[i];
            const uint32_t q = bi == 1 ? r : r / bi;
            const int64_t x = (int64_t)c[i] + (int64_t)(r - q * bi);
            r = q;
            ok = ok && (uint64_t)x < a.dim[i];
            off += x * a.stride[i];
        }
    }
    Segment sg;
    sg.rows = 0;
    sg.bytes = 0;
    sg.src = 0;
    if (!ok) return sg;
    if (s.outer0 == 2) {  // dims 0 and 1 contiguous: the box's rows along dim 1 in the tensor
        const uint64_t left = a.dim[1] - (uint64_t)c[1];
        sg.rows = (uint32_t)(left < s.seg_rows ? left : s.seg_rows);
        off += (int64_t)c[1] * a.stride[1];
    } else {
        sg.rows = 1;
    }
    sg.bytes = sg.rows * s.row_bytes;
    sg.src = (uint64_t)((int64_t)a.base + off);
    return sg;
}

// Grid counters of box b (as grid_counters), in 32-bit divisions when b and the box counts fit:
// this runs before a CTA's first bulk copy.
__device__ __forceinline__ void item_counters(const BoxWalk& w, uint64_t b, uint32_t* k)
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

// The producer's walk over its CTA's items: run u, row block q and the grid counters k of the
// run's first box (k[0] = 0), stepped with carries (divisions only to start).
struct ItemCursor {
    uint64_t u;
    uint32_t q;
    uint32_t k[5];

    // item m: run u = m / nblk, row block q = m % nblk, and the counters of the run's first box
    __device__ __forceinline__ void init(const SegArgs& s, uint64_t m)
    {
        if (m <= 0xffffffffull) {
            u = (uint32_t)m / s.nblk;
        } else {
            u = m / s.nblk;
        }
        q = (uint32_t)(m - u * s.nblk);
        item_counters(s.f.walk, u * s.run, k);
    }
    // start coordinates of the run's first box
    __device__ __forceinline__ void start(const SegArgs& s, int32_t* c) const
    {
#pragma unroll
        for (int i = 0; i < 5; i++) c[i] = (int32_t)(k[i] * s.f.walk.box[i]);
    }
    // the next row block, else the next run (odometer over dims 1..)
    __device__ __forceinline__ void next(const SegArgs& s)
    {
        if (++q < s.nblk) return;
        q = 0;
        u++;
        uint32_t carry = 1;
#pragma unroll
        for (int i = 1; i < 5; i++) {
            if (i < (int)s.f.walk.rank && carry) {
                k[i]++;
                carry = k[i] == s.f.walk.grid_nb[i] ? 1u : 0u;
                if (carry) k[i] = 0;
            }
        }
    }
};

// The 16 shared-memory bytes at p, whose address is p_al (p = p_al + d, d = p & 15), read with
// the widest loads the offset allows; two aligned 16-byte loads and a funnel shift when d is not
// a multiple of 4.
__device__ __forceinline__ uint4 load16(const uint8_t* p, uint32_t d)
{
    if (d == 0) return *reinterpret_cast<const uint4*>(p);
    if ((d & 7) == 0) {
        const uint2 x = reinterpret_cast<const uint2*>(p)[0];
        const uint2 y = reinterpret_cast<const uint2*>(p)[1];
        return make_uint4(x.x, x.y, y.x, y.y);
    }
    if ((d & 3) == 0) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(p);
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    const uint4* al = reinterpret_cast<const uint4*>(p - d);
    const uint4 lo = al[0], hi = al[1];
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const uint32_t qd = d >> 2, sh = (d & 3u) * 8u;
    uint32_t o[4];
#pragma unroll
    for (int t = 0; t < 4; t++) {
        uint32_t x0 = w[t], y0 = w[t + 1];
#pragma unroll
        for (uint32_t k = 1; k < 4; k++) {
            if (qd == k) {
                x0 = w[t + k];
                y0 = w[t + k + 1];
            }
        }
        o[t] = __funnelshift_r(x0, y0, sh);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Keeps the first `n` bytes (0 < n < 16) of v and puts fill bytes in the rest.
__device__ __forceinline__ uint4 keep_head(uint4 v, const uint4& fill, int n)
{
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
    const uint32_t* f = reinterpret_cast<const uint32_t*>(&fill);
#pragma unroll
    for (int t = 0; t < 4; t++) {
        const int k = n - 4 * t;
        const uint32_t m = k >= 4 ? 0xffffffffu : k <= 0 ? 0u : ((1u << (8 * k)) - 1u);
        w[t] = (w[t] & m) | (f[t] & ~m);
    }
    return v;
}

// 16 bytes of the fill element (zero, or the NaN pattern of a TM_OOB_NAN map).
__device__ __forceinline__ uint4 seg_fill(const FbArgs& a)
{
    if (!a.fill_nan) return make_uint4(0, 0, 0, 0);
    uint32_t lo, hi;
    if (a.esize == 2) {
        lo = hi = (uint32_t)(a.fill & 0xffffu) * 0x10001u;
    } else if (a.esize == 4) {
        lo = hi = (uint32_t)a.fill;
    } else {
        lo = (uint32_t)a.fill;
        hi = (uint32_t)(a.fill >> 32);
    }
    return make_uint4(lo, hi, lo, hi);
}

// Word t (0..3) of v, selected without indexing memory.
__device__ __forceinline__ uint32_t word_of(const uint4& v, uint32_t t)
{
    return t == 0 ? v.x : t == 1 ? v.y : t == 2 ? v.z : v.w;
}

// Writes the first n bytes (0 < n <= 16) of v to global address p with the widest stores the
// address and the byte count allow (nothing past p + n is touched).
__device__ __forceinline__ void put_head(uint8_t* p, const uint4& v, int n)
{
    const uintptr_t at = reinterpret_cast<uintptr_t>(p);
    if (n == 16 && (at & 15) == 0) {
        *reinterpret_cast<uint4*>(p) = v;
        return;
    }
    if (n == 16 && (at & 7) == 0) {
        *reinterpret_cast<uint2*>(p) = make_uint2(v.x, v.y);
        *reinterpret_cast<uint2*>(p + 8) = make_uint2(v.z, v.w);
        return;
    }
    int pos = 0;
    while (pos < n) {
        const uintptr_t q = at + (uintptr_t)pos;
        const uint32_t t = (uint32_t)pos >> 2;
        if ((q & 7) == 0 && (pos & 7) == 0 && pos + 8 <= n) {
            *reinterpret_cast<uint2*>(p + pos) = make_uint2(word_of(v, t), word_of(v, t + 1));
            pos += 8;
        } else if ((q & 3) == 0 && (pos & 3) == 0 && pos + 4 <= n) {
            *reinterpret_cast<uint32_t*>(p + pos) = word_of(v, t);
            pos += 4;
        } else if ((q & 1) == 0 && (pos & 1) == 0 && pos + 2 <= n) {
            *reinterpret_cast<uint16_t*>(p + pos) = (uint16_t)(word_of(v, t) >> (8 * (pos & 3)));
            pos += 2;
        } else {
            p[pos] = (uint8_t)(word_of(v, t) >> (8 * (pos & 3)));
            pos += 1;
        }
    }
}

}  // namespace

// What the producer leaves beside each staging buffer for the item it staged.
struct SegItem {
    uint64_t run;  // run index u: boxes u * run .. u * run + run - 1; kEndOfItems: no more items
    uint32_t r0;   // first image row of the item in its boxes
    uint32_t nr;   // image rows of the item in each box
};
constexpr uint64_t kEndOfItems = ~0ull;

// Where the producer warp takes its items from (every lane runs it in step).  Static: the CTA's
// contiguous share m0 .. m0 + total - 1 of the host's split.  Dynamic (s.sched set): CTA c first
// takes items c, c + gridDim.x, ... for its S staging buffers, then batches of s.batch
// consecutive items from the stream's counter (item S * gridDim.x + s.batch * atomicAdd), each
// batch fetched one ahead, right after an item's bulk copies are issued (the next arrive is a
// release and would otherwise wait for the atomic); a CTA that runs faster takes more items.
struct SegSource {
    bool dyn, first_fetch, refetch;
    uint32_t S, B;
    uint64_t m0, total, si, dj, prefix, bg, bend;
    unsigned long long pend;  // lane 0: the batch fetched ahead

    __device__ __forceinline__ void init(const SegArgs& s, uint64_t m0_, uint64_t total_)
    {
        dyn = s.sched != nullptr;
        S = s.stages;
        B = s.batch ? s.batch : 1u;
        m0 = m0_;
        total = total_;
        si = dj = bg = bend = 0;
        pend = 0;
        prefix = (uint64_t)S * gridDim.x;
        first_fetch = dyn && prefix < s.nitems;
        refetch = false;
    }
    // The next item, or false when this CTA has none left.
    __device__ __forceinline__ bool next(const SegArgs& s, uint64_t& m)
    {
        if (!dyn) {
            if (si >= total) return false;
            m = m0 + si++;
            return true;
        }
        if (dj < S) {
            m = blockIdx.x + dj * gridDim.x;
            dj++;
            return m < s.nitems;  // past the end of the prefix there is nothing left either
        }
        if (bg == bend) {
            const unsigned long long p = __shfl_sync(0xffffffffu, pend, 0);
            bg = prefix + p * B;
            if (bg >= s.nitems) return false;
            bend = bg + B < s.nitems ? bg + B : s.nitems;
            refetch = true;
        }
        m = bg++;
        return true;
    }
    // After an item's bulk copies: the first batch once the prefix is issued, then the next batch
    // once the one fetched ahead has been taken.
    __device__ __forceinline__ void after_issue(const SegArgs& s, uint32_t lane)
    {
        if (first_fetch && dj == S) {
            if (lane == 0) pend = atomicAdd(s.sched, 1ull);
            first_fetch = false;
        } else if (refetch) {
            if (lane == 0) pend = atomicAdd(s.sched, 1ull);
            refetch = false;
        }
    }
    // The launch's counter back to zero for the next launch of the stream: the last CTA to finish
    // knows that every CTA has made its last fetch.
    __device__ __forceinline__ void finish(const SegArgs& s, uint32_t lane)
    {
        if (!dyn || lane != 0) return;
        __threadfence();
        if (atomicAdd(s.sched + 1, 1ull) == (unsigned long long)gridDim.x - 1) {
            atomicExch(s.sched, 0ull);
            atomicExch(s.sched + 1, 0ull);
            __threadfence();
        }
    }
};

template <uint32_t kSegConsumerWarps>
__global__ void __launch_bounds__(seg_threads<kSegConsumerWarps>(), 2)
    k_fb_seg_copy(const __grid_constant__ SegArgs s)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kSegMaxStages];   // segments landed (count 1 + bytes)
    __shared__ __align__(8) uint64_t empty_bar[kSegMaxStages];  // consumers done (one per warp)
    __shared__ SegItem info[kSegMaxStages];
    const FbArgs& a = s.f;
    const uint32_t E = s.block_groups;
    const uint32_t G1 = s.seg_rows;
    const uint32_t S = s.stages;
    uint8_t* const sbuf0 = smem_raw;  // S x E segments
    // per staging buffer, the shared-memory offset of each image row's tensor byte 0 (-1: the
    // row lies outside the tensor)
    int32_t* const tabs = reinterpret_cast<int32_t*>(smem_raw + (size_t)S * E * s.seg_stride);

    const uint64_t per = s.per, extra = s.extra;  // the static item split, from the host
    const uint64_t m0 = blockIdx.x * per + (blockIdx.x < extra ? blockIdx.x : extra);
    const uint64_t total = per + (blockIdx.x < extra ? 1 : 0);
    if (s.sched == nullptr && total == 0) return;
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) TM_STAMP(seg, 0);
    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < S; i++) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), kSegConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) TM_STAMP(seg, 62);
        // ---- producer: walks the CTA's items with a cursor (every lane keeps the same copy).
        // Item i goes to buffer i % S once the consumers have released that buffer's item i - S.
        SegSource src;
        src.init(s, m0, total);
        ItemCursor cur;
        if (!src.dyn) cur.init(s, m0);
        // item i: buffer b = i % S, lap = i / S; for i >= S it waits for the release of item
        // i - S, the buffer's completion number lap - 1.  After the last item, buffer b gets the
        // end marker.
        uint32_t b = 0, lap = 0;
        uint64_t i = 0, m = 0;
        bool failed = false;
        for (;; i++) {
            const bool more = src.next(s, m);
            if (lap > 0) {
                const uint32_t eparity = (lap - 1) & 1u;
                const bool ok = mbar_wait(smem_u32(&empty_bar[b]), eparity, a.timeout_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) record_timeout(a.status, K_FB_SEG_COPY, b, eparity, m0 + i);
                    failed = true;
                    break;
                }
            }
            if (!more) break;
            if (src.dyn) cur.init(s, m);
            int32_t c[5];
            cur.start(s, c);
            const uint32_t g0 = cur.q * E;
            const uint32_t ng = min(E, s.groups - g0);
            int32_t* const tab = tabs + (size_t)b * E * G1;
            const uint32_t sbase = b * E * s.seg_stride;
            // lane j takes segments j, j + 32, ...: their rows' table entries, then (after lane 0
            // has posted the item's total bytes) their bulk copies
            uint32_t bytes = 0;
            for (uint32_t j = lane; j < ng; j += 32) {
                const Segment sg = segment_of(s, c, g0 + j);
                const int32_t at = (int32_t)(sbase + j * s.seg_stride + (uint32_t)(sg.src & 15));
                for (uint32_t e = 0; e < G1; e++)
                    tab[j * G1 + e] = e < sg.rows ? at + (int32_t)(e * s.row_bytes) : -1;
                if (sg.rows) bytes += (uint32_t)(((sg.src & 15) + sg.bytes + 15) & ~15ull);
            }
            bytes = __reduce_add_sync(0xffffffffu, bytes);
            if (i == 0 && lane == 0) TM_STAMP(seg, 60);
            const uint32_t bar = smem_u32(&full_bar[b]);
            if (lane == 0) {
                info[b].run = cur.u;
                info[b].r0 = g0 * G1;
                info[b].nr = ng * G1;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(bar, bytes);  // publishes the table and info
            __syncwarp();
            const uint32_t dst0 = smem_u32(sbuf0 + sbase);
            for (uint32_t j = lane; j < ng; j += 32) {
                const Segment sg = segment_of(s, c, g0 + j);
                if (sg.rows) {
                    const uint32_t n = (uint32_t)(((sg.src & 15) + sg.bytes + 15) & ~15ull);
                    bulk_load(dst0 + j * s.seg_stride, sg.src & ~15ull, n, bar);
                }
            }
            src.after_issue(s, lane);
            if (!src.dyn) cur.next(s);
            if (i == 0 && lane == 0) TM_STAMP(seg, 1);
            if (++b == S) {
                b = 0;
                lap++;
            }
        }
        if (!failed) {  // the end marker in buffer b (released by the consumers, waited for above)
            if (lane == 0) info[b].run = kEndOfItems;
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&full_bar[b]));
        }
        // the copies issued last land before the CTA leaves (the consumers normally saw them)
        if (lane == 0) {
            TM_TRACE_PUT(seg, 61, i);
            // (item i - S shares buffer i % S with the end marker, whose phase followed its own;
            // the consumers released that buffer before the marker went in, so it has landed)
            const uint64_t lo = failed ? (i > S ? i - S : 0) : (i >= S ? i - S + 1 : 0);
            for (uint64_t k = lo; k < i; k++)
                mbar_wait(smem_u32(&full_bar[k % S]), (uint32_t)((k / S) & 1), a.timeout_ns);
        }
        src.finish(s, lane);
        return;
    }

    // ---- consumers: realign item n's chunks, stored straight to the global images (a warp's 32
    // chunks cover whole 128-byte image rows, permuted inside each by the swizzle).  Box-major
    // when each box's block has at least one chunk per consumer thread (its images are then
    // written in order; measured on GB300 4 % faster than the row-major walk on the W4 rank-5
    // view), else row-major: the chunks of one image row of every box of the run are the 16-byte
    // chunks of one tensor row, so the item is nr rows x (run x cpr) chunks and no thread idles
    // on a run of many boxes with few rows; each thread steps its (row, chunk) with carries.
    const uint32_t inner = a.inner_bytes;
    const uint32_t cpr = inner >> 4;  // 16-byte chunks per image row
    const uint32_t cpr_shift = (cpr & (cpr - 1)) == 0 ? (uint32_t)(__ffs(cpr) - 1) : 32u;
    const uint4 fillv = seg_fill(a);
    const uint32_t row_bytes = s.row_bytes;
    const uint32_t ct = threadIdx.x - 32;  // consumer thread index
    constexpr uint32_t kCT = 32 * kSegConsumerWarps;
    const uint32_t rc = s.run * cpr;  // chunks per tensor row of the run
    const uint32_t r_start = ct / rc, c_start = ct - r_start * rc;
    const uint32_t r_step = kCT / rc, c_step = kCT - r_step * rc;
    uint32_t sb = 0, sparity = 0;  // staging buffer of item n (n % S) and its phase parity
    for (uint64_t n = 0;; n++) {
        if (n) {
            if (++sb == S) {
                sb = 0;
                sparity ^= 1u;
            }
        }
        const bool ok = mbar_wait(smem_u32(&full_bar[sb]), sparity, a.timeout_ns);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) record_timeout(a.status, K_FB_SEG_COPY, sb, sparity, m0 + n);
            break;
        }
        if (info[sb].run == kEndOfItems) break;
        const int32_t* const tab = tabs + (size_t)sb * E * G1;
        const uint32_t r0 = info[sb].r0;
        const uint32_t nr = info[sb].nr;
        uint8_t* const img0 = reinterpret_cast<uint8_t*>(a.images + info[sb].run * s.run * a.box_bytes);
        const uint32_t per_box = nr * cpr;
        if (per_box >= kCT) {
            for (uint32_t k = 0; k < s.run; k++) {
                uint8_t* const img = img0 + (size_t)k * a.box_bytes;
                for (uint32_t q = ct; q < per_box; q += kCT) {
                    const uint32_t r = cpr_shift < 32 ? q >> cpr_shift : q / cpr;
                    const uint32_t j = q - r * cpr;
                    const int32_t at = tab[r];
                    const int x = (int)(k * inner + 16 * j);  // the chunk's first tensor-row byte
                    const int left = (int)row_bytes - x;
                    uint4 v = fillv;
                    if (at >= 0 && left > 0) {
                        const uint32_t p = (uint32_t)at + (uint32_t)x;
                        v = load16(smem_raw + p, p & 15u);
                        if (left < 16) v = keep_head(v, fillv, left);
                    }
                    *reinterpret_cast<uint4*>(img + swizzle_offset((r0 + r) * inner + 16 * j, a.span)) = v;
                }
            }
        } else {
            for (uint32_t r = r_start, c = c_start; r < nr;) {
                const uint32_t k = cpr_shift < 32 ? c >> cpr_shift : c / cpr;  // box of the run
                const uint32_t j = c - k * cpr;                                  // chunk of its row
                const int32_t at = tab[r];
                const int x = (int)(16 * c);  // the chunk's first byte in the tensor row
                const int left = (int)row_bytes - x;
                uint4 v = fillv;
                if (at >= 0 && left > 0) {
                    const uint32_t p = (uint32_t)at + (uint32_t)x;
                    v = load16(smem_raw + p, p & 15u);
                    if (left < 16) v = keep_head(v, fillv, left);
                }
                *reinterpret_cast<uint4*>(img0 + (size_t)k * a.box_bytes +
                                          swizzle_offset((r0 + r) * inner + 16 * j, a.span)) = v;
                r += r_step;
                c += c_step;
                if (c >= rc) {
                    c -= rc;
                    r++;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty_bar[sb]));  // this warp's reads are done
        if (warp == 1 && lane == 0 && n < 58) TM_STAMP(seg, 2 + n);
    }
    if (warp == 1 && lane == 0) TM_STAMP(seg, 63);
}

// Store direction (tiled_roundtrip): the inverse walk.  The producer warp bulk-loads, per item,
// the block of image rows of each box of the run (contiguous in the images) into a staging buffer
// and writes each row's tensor address beside it; the consumer warps read each 16-byte chunk at
// its swizzled place and write its in-bounds bytes to the tensor (the widest stores the address
// allows; nothing beyond a row's last element is written, so padding after a row survives).
// (Measured on GB300 and dropped: assembling each segment in shared memory and writing it back
// with one bulk store, 71.9 against 64.9 us on the W4 rank-5 view -- a stage can then only be
// reloaded after its write-back has read it, which serialises the pipeline.)
template <uint32_t kSegConsumerWarps>
__global__ void __launch_bounds__(seg_threads<kSegConsumerWarps>(), 2)
    k_fb_seg_store(const __grid_constant__ SegArgs s)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kSegMaxStages];
    __shared__ __align__(8) uint64_t empty_bar[kSegMaxStages];
    __shared__ SegItem info[kSegMaxStages];
    const FbArgs& a = s.f;
    const uint32_t E = s.block_groups;
    const uint32_t G1 = s.seg_rows;
    const uint32_t S = s.stages;
    const size_t stage_bytes = (size_t)s.run * s.img_stride;  // image blocks of one item
    uint8_t* const sbuf0 = smem_raw;
    // per staging buffer, the tensor address of each image row's element 0 (~0: outside)
    uint64_t* const tabs = reinterpret_cast<uint64_t*>(smem_raw + S * stage_bytes);

    const uint64_t per = s.per, extra = s.extra;  // the static item split, from the host
    const uint64_t m0 = blockIdx.x * per + (blockIdx.x < extra ? blockIdx.x : extra);
    const uint64_t total = per + (blockIdx.x < extra ? 1 : 0);
    if (s.sched == nullptr && total == 0) return;
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) TM_STAMP(seg, 0);
    const uint32_t inner = a.inner_bytes;
    if (threadIdx.x == 0) {
        for (uint32_t i = 0; i < S; i++) {
            mbar_init(smem_u32(&full_bar[i]), 1);
            mbar_init(smem_u32(&empty_bar[i]), kSegConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) TM_STAMP(seg, 62);
        // ---- producer (the same item source, cursor and end marker as the copy)
        SegSource src;
        src.init(s, m0, total);
        ItemCursor cur;
        if (!src.dyn) cur.init(s, m0);
        uint32_t b = 0, lap = 0;
        uint64_t i = 0, m = 0;
        bool failed = false;
        for (;; i++) {
            const bool more = src.next(s, m);
            if (lap > 0) {
                const uint32_t eparity = (lap - 1) & 1u;
                const bool ok = mbar_wait(smem_u32(&empty_bar[b]), eparity, a.timeout_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) record_timeout(a.status, K_FB_SEG_STORE, b, eparity, m0 + i);
                    failed = true;
                    break;
                }
            }
            if (!more) break;
            if (src.dyn) cur.init(s, m);
            int32_t c[5];
            cur.start(s, c);
            const uint32_t g0 = cur.q * E;
            const uint32_t ng = min(E, s.groups - g0);
            const uint32_t nr = ng * G1;
            uint64_t* const tab = tabs + (size_t)b * E * G1;
            for (uint32_t j = lane; j < ng; j += 32) {
                const Segment sg = segment_of(s, c, g0 + j);
                for (uint32_t e = 0; e < G1; e++)
                    tab[j * G1 + e] = e < sg.rows ? sg.src + (uint64_t)e * s.row_bytes : ~0ull;
            }
            if (i == 0 && lane == 0) TM_STAMP(seg, 60);
            const uint32_t bar = smem_u32(&full_bar[b]);
            if (lane == 0) {
                info[b].run = cur.u;
                info[b].r0 = g0 * G1;
                info[b].nr = nr;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(bar, s.run * nr * inner);  // publishes table, info
            __syncwarp();
            const uint32_t dst0 = smem_u32(sbuf0 + b * stage_bytes);
            for (uint32_t k = lane; k < s.run; k += 32) {
                const uint64_t box = cur.u * s.run + k;
                bulk_load(dst0 + k * s.img_stride, a.images + box * a.box_bytes + (uint64_t)g0 * G1 * inner,
                          nr * inner, bar);
            }
            src.after_issue(s, lane);
            if (!src.dyn) cur.next(s);
            if (i == 0 && lane == 0) TM_STAMP(seg, 1);
            if (++b == S) {
                b = 0;
                lap++;
            }
        }
        if (!failed) {  // the end marker in buffer b
            if (lane == 0) info[b].run = kEndOfItems;
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&full_bar[b]));
        }
        if (lane == 0) {
            TM_TRACE_PUT(seg, 61, i);
            // (item i - S shares buffer i % S with the end marker, whose phase followed its own;
            // the consumers released that buffer before the marker went in, so it has landed)
            const uint64_t lo = failed ? (i > S ? i - S : 0) : (i >= S ? i - S + 1 : 0);
            for (uint64_t k = lo; k < i; k++)
                mbar_wait(smem_u32(&full_bar[k % S]), (uint32_t)((k / S) & 1), a.timeout_ns);
        }
        src.finish(s, lane);
        return;
    }

    // ---- consumers: the copy's row-major chunk walk, always (the tensor's rows are then written
    // in order; measured on GB300 10 % faster than box-major on the W4 rank-5 view)
    const uint32_t cpr = inner >> 4;
    const uint32_t cpr_shift = (cpr & (cpr - 1)) == 0 ? (uint32_t)(__ffs(cpr) - 1) : 32u;
    const uint32_t row_bytes = s.row_bytes;
    const uint32_t ct = threadIdx.x - 32;
    constexpr uint32_t kCT = 32 * kSegConsumerWarps;
    // Chunks per tensor row of the run that hold tensor bytes: the run's images cover the whole
    // row and more (its last box may reach past the tensor), and a store writes only the row.
    const uint32_t rc = min(s.run * cpr, (row_bytes + 15) / 16);
    const uint32_t r_start = ct / rc, c_start = ct - r_start * rc;
    const uint32_t r_step = kCT / rc, c_step = kCT - r_step * rc;
    uint32_t sb = 0, sparity = 0;
    for (uint64_t n = 0;; n++) {
        if (n) {
            if (++sb == S) {
                sb = 0;
                sparity ^= 1u;
            }
        }
        const bool ok = mbar_wait(smem_u32(&full_bar[sb]), sparity, a.timeout_ns);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) record_timeout(a.status, K_FB_SEG_STORE, sb, sparity, m0 + n);
            break;
        }
        if (info[sb].run == kEndOfItems) break;
        const uint64_t* const tab = tabs + (size_t)sb * E * G1;
        const uint32_t r0 = info[sb].r0;
        const uint32_t nr = info[sb].nr;
        const uint8_t* const blk0 = sbuf0 + sb * stage_bytes;
        for (uint32_t r = r_start, c = c_start; r < nr;) {
            const uint32_t k = cpr_shift < 32 ? c >> cpr_shift : c / cpr;  // box of the run
            const uint32_t j = c - k * cpr;                                  // chunk of its row
            const uint64_t row = tab[r];
            const int x = (int)(16 * c);
            const int left = (int)row_bytes - x;
            if (row != ~0ull && left > 0) {
                // the block starts at image row r0; the swizzle permutes inside a row
                const uint4 v = *reinterpret_cast<const uint4*>(
                    blk0 + k * s.img_stride + swizzle_offset((r0 + r) * inner + 16 * j, a.span) -
                    r0 * inner);
                put_head(reinterpret_cast<uint8_t*>(row + (uint64_t)x), v, left < 16 ? left : 16);
            }
            r += r_step;
            c += c_step;
            if (c >= rc) {
                c -= rc;
                r++;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty_bar[sb]));
        if (warp == 1 && lane == 0 && n < 58) TM_STAMP(seg, 2 + n);
    }
    if (warp == 1 && lane == 0) TM_STAMP(seg, 63);
}

namespace {
template <uint32_t W>
cudaError_t launch_store_w(const SegArgs& a, uint32_t grid, size_t smem, cudaStream_t st)
{
    cudaError_t e = cudaFuncSetAttribute(k_fb_seg_store<W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    k_fb_seg_store<W><<<grid, seg_threads<W>(), smem, st>>>(a);
    return cudaGetLastError();
}

template <uint32_t W>
cudaError_t launch_copy_w(const SegArgs& a, uint32_t grid, size_t smem, cudaStream_t st)
{
    cudaError_t e = cudaFuncSetAttribute(k_fb_seg_copy<W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    k_fb_seg_copy<W><<<grid, seg_threads<W>(), smem, st>>>(a);
    return cudaGetLastError();
}
}  // namespace

// CTAs of the segment kernel (store or copy direction, cwarps consumer warps) that one SM holds with
// `smem` bytes of dynamic shared memory each: the occupancy calculator's answer for the instance
// that will run (its registers decide as much as its shared memory); 0 if it cannot say.
int seg_resident_ctas(bool store, uint32_t cwarps, size_t smem)
{
    int n = 0;
    auto ask = [&](auto k, uint32_t threads) {
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, (int)threads, smem) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
    };
    if (store) {
        if (cwarps == 16) ask(k_fb_seg_store<16>, seg_threads<16>());
        else if (cwarps == 12) ask(k_fb_seg_store<12>, seg_threads<12>());
        else ask(k_fb_seg_store<8>, seg_threads<8>());
    } else {
        if (cwarps == 16) ask(k_fb_seg_copy<16>, seg_threads<16>());
        else if (cwarps == 12) ask(k_fb_seg_copy<12>, seg_threads<12>());
        else ask(k_fb_seg_copy<8>, seg_threads<8>());
    }
    return n;
}

cudaError_t launch_fb_seg_store(const SegArgs& a, uint32_t grid, size_t smem, cudaStream_t st)
{
    return a.cwarps == 16 ? launch_store_w<16>(a, grid, smem, st)
           : a.cwarps == 12 ? launch_store_w<12>(a, grid, smem, st)
                            : launch_store_w<8>(a, grid, smem, st);
}

cudaError_t launch_fb_seg_copy(const SegArgs& a, uint32_t grid, size_t smem, cudaStream_t st)
{
    return a.cwarps == 16 ? launch_copy_w<16>(a, grid, smem, st)
           : a.cwarps == 12 ? launch_copy_w<12>(a, grid, smem, st)
                            : launch_copy_w<8>(a, grid, smem, st);
}

}  // namespace tmk
