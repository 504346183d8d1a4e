// k_fallback.cu -- generic path for maps the tensor-map hardware cannot take (a base or stride
// that is a multiple of the element size but not of 16 bytes, e.g. a 200-byte group stride), and
// for explicit box lists the hardware must not be given (see tmap_host.cpp).
//
// Both directions produce exactly the bytes of the tensor-map path -- same swizzle, zero fill
// outside the tensor, only in-bounds elements written -- with threads doing the addressing the
// engine would do ([H200-TMA] = coolgpu "H200 · TMA · Tensor Memory Accelerator" card, §02: the
// per-thread cp.async / LDGSTS style of copy that TMA replaces):
//
//   copy   16-byte cp.async copies of the aligned windows under each image row into shared
//          memory, then a realign of each 16-byte chunk from two staged windows, then one
//          16-byte global store of the chunk at its swizzled place in the image.  (A first
//          design realigned in registers with warp shuffles; it was instruction-bound on GB300 at
//          about 1.9 TB/s, and most of its time stayed even with its global loads removed.)
//   store  each thread reads its 16-byte chunks of the image straight from global memory
//          (coalesced: a swizzle only permutes chunks inside a 128-byte row) and writes their
//          in-bounds bytes with the widest stores the destination alignment allows.
//   reduce element-wise add / min / max (f32, f16, bf16, u32, s32) straight from global memory.
//
// A window is only loaded when it holds at least one in-bounds byte of the row; an aligned
// 16-byte window never crosses a page, so no load can touch an unmapped address.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "tm_ptx.cuh"

namespace tmk {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t sel4(uint32_t q, uint32_t a, uint32_t b, uint32_t c,
                                         uint32_t d)
{
    return q == 0 ? a : q == 1 ? b : q == 2 ? c : d;
}

// Byte mask of the bytes [lo, hi) that fall in word t (bytes 4t .. 4t+3) of a 16-byte chunk.
__device__ __forceinline__ uint32_t word_mask(int lo, int hi, int t)
{
    const int s = min(max(lo - 4 * t, 0), 4);
    const int e = min(max(hi - 4 * t, 0), 4);
    if (e <= s) return 0u;
    const uint32_t ones = (e - s) == 4 ? 0xffffffffu : ((1u << (8 * (e - s))) - 1u);
    return ones << (8 * s);
}

// Image row `row` of a box -> global byte address of its element 0 (relative to base, may be
// negative) and whether every outer coordinate (dims 1..) is inside the tensor.  Image row
// coordinate e[i] (0 <= e[i] < ibox[i]) comes from tensor coordinate c[i] + e[i] * estride[i].
struct RowPos {
    int64_t off;
    bool ok;
};

__device__ __forceinline__ RowPos row_position(const FbArgs& a, const int32_t* c, uint32_t row,
                                               const int64_t* stride)
{
    RowPos p{(int64_t)c[0] * stride[0], true};
    uint32_t r = row;
#pragma unroll
    for (int i = 1; i < 5; i++) {
        if (i < (int)a.walk.rank) {
            const uint32_t bi = a.ibox[i];
            const uint32_t q = bi == 1 ? r : r / bi;  // a unit extent needs no division
            const int64_t g = (int64_t)c[i] + (int64_t)(r - q * bi) * a.estride[i];
            r = q;
            p.ok = p.ok && g >= 0 && (uint64_t)g < a.dim[i];
            p.off += g * stride[i];
        }
    }
    return p;
}

// In-bounds part of an image row of a box whose dim-0 start is c0: image elements [i_lo, i_hi)
// (element k comes from tensor coordinate c0 + k * estride[0]), and the bytes [g_lo, g_hi) of
// the tensor row segment under the image row, counted from element c0, that hold them.
struct XRange {
    int i_lo, i_hi, g_lo, g_hi;
};

__device__ __forceinline__ XRange x_range(const FbArgs& a, int32_t c0)
{
    const int64_t step = a.estride[0], n0 = a.ibox[0];
    const int64_t lo = max(-(int64_t)c0, (int64_t)0);
    const int64_t hi = max((int64_t)a.dim[0] - (int64_t)c0, (int64_t)0);
    XRange x;
    if (step == 1) {  // no division for the common unit step
        x.i_lo = (int)min(lo, n0);
        x.i_hi = (int)min(hi, n0);
    } else {
        x.i_lo = (int)min((lo + step - 1) / step, n0);
        x.i_hi = (int)min((hi + step - 1) / step, n0);
    }
    const int es = (int)a.esize;
    x.g_lo = x.i_lo * (int)step * es;
    x.g_hi = x.i_hi > x.i_lo ? ((x.i_hi - 1) * (int)step + 1) * es : x.g_lo;
    return x;
}

// 16 bytes of the fill element, repeated (zero, or the NaN pattern of a TM_OOB_NAN map).
__device__ __forceinline__ uint4 fill_vector(const FbArgs& a)
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

// Chunk j (16 bytes, 16 / sizeof(E) elements) of an image row whose dim-0 elements lie `step`
// elements apart in the staged row segment `row`; elements outside [i_lo, i_hi) are the fill.
template <typename E>
__device__ __forceinline__ uint4 gather_chunk(const uint8_t* row, int j, const XRange& x, int step,
                                              const uint4& fill)
{
    constexpr int n = 16 / (int)sizeof(E);
    union {
        uint4 v;
        E e[n];
    } u;
    u.v = fill;
#pragma unroll
    for (int t = 0; t < n; t++) {
        const int k = j * n + t;
        if (k >= x.i_lo && k < x.i_hi)
            u.e[t] = *reinterpret_cast<const E*>(row + (size_t)k * step * sizeof(E));
    }
    return u.v;
}

}  // namespace

constexpr int64_t kRowOutside = INT64_MIN;  // table entry of a row outside the tensor

// Image row and chunk of item `item` (chunks of a row are consecutive items).
__device__ __forceinline__ void split_item(uint32_t item, uint32_t cpr, uint32_t cpr_shift,
                                           uint32_t& row, uint32_t& j)
{
    row = cpr_shift < 32 ? item >> cpr_shift : item / cpr;
    j = item - row * cpr;
}

// Round-robin walk of (row block, box) items (the store kernel), item m = q + nblk * b: CTA c takes
// items c, c + G, c + 2G, ... (G = gridDim.x), so the blocks of neighbouring boxes run on
// neighbouring CTAs at the same time.  Thread 0 keeps the item's digits (row block
// q, then the box's grid counters) in shared memory and adds the digits of G with carries; a box
// list divides instead.
struct ItemWalk {
    uint32_t k[6];  // q, then the grid counters of box b
    uint32_t d[6];  // digits of G
    uint64_t box;   // b
    uint64_t dbox;  // G / nblk
};

__device__ __forceinline__ void item_walk_init(const BoxWalk& w, uint32_t nblk, uint64_t m,
                                               ItemWalk& s)
{
    s.box = m / nblk;
    s.k[0] = (uint32_t)(m - s.box * nblk);
    s.dbox = gridDim.x / nblk;
    s.d[0] = gridDim.x - (uint32_t)(s.dbox * nblk);
    if (w.mode == WALK_GRID) {
        grid_counters(w, s.box, s.k + 1);
        grid_counters(w, s.dbox, s.d + 1);  // past the grid only once the walk has ended
    }
}

__device__ __forceinline__ void item_walk_next(const BoxWalk& w, uint32_t nblk, ItemWalk& s)
{
    uint32_t q = s.k[0] + s.d[0];
    uint32_t carry = q >= nblk ? 1u : 0u;
    s.k[0] = carry ? q - nblk : q;
    s.box += s.dbox + carry;
    if (w.mode == WALK_GRID) {
#pragma unroll
        for (int i = 0; i < 5; i++) {
            if (i < (int)w.rank) {
                const uint64_t v = (uint64_t)s.k[i + 1] + s.d[i + 1] + carry;
                carry = v >= w.grid_nb[i] ? 1u : 0u;
                s.k[i + 1] = (uint32_t)(carry ? v - w.grid_nb[i] : v);
            }
        }
    }
}

// Start of the item's box.
__device__ __forceinline__ void item_box_start(const BoxWalk& w, const ItemWalk& s, int32_t* c)
{
    if (w.mode == WALK_GRID) {
#pragma unroll
        for (int i = 0; i < 5; i++) c[i] = i < (int)w.rank ? (int32_t)(s.k[i + 1] * w.box[i]) : 0;
    } else {
        box_start(w, s.box, c);
    }
}

// The 16 bytes at offset d (1..15, not a multiple of 4) of the two staged windows at `win`: two
// aligned 16-byte shared loads and a funnel shift per word (element sizes of 1 or 2 bytes only).
__device__ __noinline__ uint4 unaligned_chunk(const uint8_t* win, uint32_t d)
{
    const uint4 lo = reinterpret_cast<const uint4*>(win)[0];
    const uint4 hi = reinterpret_cast<const uint4*>(win)[1];
    const uint32_t qd = d >> 2, sh = (d & 3u) * 8u;
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t o[4];
#pragma unroll
    for (int t = 0; t < 4; t++) {
        const uint32_t x0 = sel4(qd, w[t], w[t + 1], w[t + 2], w[t + 3]);
        const uint32_t y0 = sel4(qd, w[t + 1], w[t + 2], w[t + 3], w[t + 4]);
        o[t] = __funnelshift_r(x0, y0, sh);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// ---- load direction: staged copy ------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, uint64_t src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Image of each box, rows taken in blocks of a.block_rows.  Work items are (row block, box) pairs,
// box-major; CTA c takes a contiguous range of an even split (the same number of items +-1), and
// thread 0 steps the box counters with an odometer and publishes each box start in shared memory.
// (Measured on GB300 against the round-robin item walk of the store: 2-3 % faster on the rank-5 W4
// view and the strided W3 copy, although it reads more sectors twice.)  Per block: the row offsets go to a shared table; every thread issues 16-byte
// cp.async copies of the aligned windows under its share of the rows (only windows holding an
// in-bounds byte), so a whole block of loads is in flight without occupying registers; after one
// wait each thread reads its 16-byte chunks from the staged windows at their byte offset (the
// widest shared loads the offset allows), fills elements outside the tensor, and stores the chunk
// to its swizzled place in the global image with one 16-byte store (the swizzle only permutes
// chunks inside a 128-byte row, so a warp's stores stay coalesced).  An aligned 16-byte window never crosses a
// page, so no copy touches an unmapped address.  (Measured on GB300: one 1-D bulk copy per image
// row instead of the per-window cp.async, 80-144 bytes each, was limited by the TMA engine's rate
// of small requests, 2.2 TB/s against 3.3 on the rank-5 W4 view.)
//
// kStep0: the map's elementStrides[0] is not 1.  The staged windows then cover the box's whole
// tensor row segment (box[0] elements) and each chunk gathers its elements `estride[0]` apart.
template <bool kStep0>
__global__ void __launch_bounds__(kThreads, 8) k_fb_copy(const __grid_constant__ FbArgs a)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ ItemWalk s_w;      // the current item (k[0] = row block, k[1..] = box counters)
    __shared__ int32_t s_c[5];    // its box start
    __shared__ XRange s_x;        // the box's in-bounds part along dim 0
    const uint32_t cpr = a.inner_bytes >> 4;      // 16-byte chunks per image row
    const uint32_t cpr_shift = (cpr & (cpr - 1)) == 0 ? (uint32_t)(__ffs(cpr) - 1) : 32u;
    const uint32_t wpr = (a.gspan0 >> 4) + 1;     // staged windows per row
    const uint32_t RB = a.block_rows;
    uint8_t* const stg = smem_raw;
    const uint32_t stg_u32 = smem_u32(stg);
    int64_t* const tab = reinterpret_cast<int64_t*>(smem_raw + (size_t)RB * wpr * 16);

    const uint32_t nblk = (a.rows + RB - 1) / RB;  // row blocks per box
    const uint64_t T = a.walk.nbox * nblk;
    const uint64_t per = T / gridDim.x, extra = T % gridDim.x;
    const uint64_t m0 = blockIdx.x * per + (blockIdx.x < extra ? blockIdx.x : extra);
    const uint64_t total = per + (blockIdx.x < extra ? 1 : 0);
    if (total == 0) return;
    const int64_t gbase = (int64_t)a.base;
    const int es = (int)a.esize;
    const int inner = (int)a.inner_bytes;
    const uint4 fillv = fill_vector(a);

    for (uint64_t n = 0; n < total; n++) {
        if (threadIdx.x == 0) {
            if (n == 0) {
                s_w.box = m0 / nblk;
                s_w.k[0] = (uint32_t)(m0 - s_w.box * nblk);
                if (a.walk.mode == WALK_GRID) grid_counters(a.walk, s_w.box, s_w.k + 1);
            } else if (++s_w.k[0] == nblk) {
                s_w.k[0] = 0;
                s_w.box++;
                if (a.walk.mode == WALK_GRID) grid_next(a.walk, s_w.k + 1);
            }
            item_box_start(a.walk, s_w, s_c);
            s_x = x_range(a, s_c[0]);
        }
        // the item is published; the previous block's windows and table are no longer read
        __syncthreads();
        const XRange x = s_x;
        const int lo_byte = x.i_lo * es, hi_byte = x.i_hi * es;
        const bool whole_x = lo_byte == 0 && hi_byte == inner;
        uint8_t* const img = reinterpret_cast<uint8_t*>(a.images + s_w.box * a.box_bytes);
        const uint32_t r0 = s_w.k[0] * RB;
        const uint32_t nr = min(RB, a.rows - r0);
        for (uint32_t r = threadIdx.x; r < nr; r += kThreads) {
            const RowPos p = row_position(a, s_c, r0 + r, a.stride);
            tab[r] = (p.ok && x.i_lo < x.i_hi) ? p.off : kRowOutside;
        }
        __syncthreads();
        const uint32_t nwin = nr * wpr;
        // Window w = r * wpr + k; the (r, k) pair is stepped along instead of divided out.
        const uint32_t dr = kThreads / wpr, dk = kThreads - dr * wpr;
        uint32_t r = threadIdx.x / wpr, k = threadIdx.x - r * wpr;
        for (uint32_t w = threadIdx.x; w < nwin; w += kThreads) {
            const int64_t off = tab[r];
            if (off != kRowOutside) {
                const int64_t row_addr = gbase + off;
                const int d = (int)(row_addr & 15);
                const int wlo = 16 * (int)k - d;  // window k holds row bytes [wlo, wlo + 16)
                if (wlo + 16 > x.g_lo && wlo < x.g_hi)
                    cp_async16(stg_u32 + w * 16, (uint64_t)(row_addr - d + 16 * (int64_t)k));
            }
            r += dr;
            k += dk;
            if (k >= wpr) {
                k -= wpr;
                r++;
            }
        }
        cp_async_wait_all();
        __syncthreads();
        const uint32_t nch = nr * cpr;
        for (uint32_t it = threadIdx.x; it < nch; it += kThreads) {
            uint32_t r, j;
            split_item(it, cpr, cpr_shift, r, j);
            const int64_t off = tab[r];
            const int blo = lo_byte - 16 * (int)j, bhi = hi_byte - 16 * (int)j;
            uint4 out = fillv;
            if (off == kRowOutside || blo >= 16 || bhi <= 0) {
                // a row outside the tensor, or a chunk wholly outside it along dim 0
            } else if (kStep0 && a.estride[0] == 2 && (es == 2 || es == 4) && blo <= 0 && bhi >= 16 &&
                       ((gbase + off) & 15) == 0) {
                // Every other element, the whole chunk inside the tensor and the row segment on a
                // 16-byte boundary: the chunk's elements are the even ones of the 32 staged bytes
                // at 32 j -- two aligned 16-byte loads and a byte permute, instead of one shared
                // load per element 4 or 8 bytes apart (8-way bank conflicts).
                const uint4* w = reinterpret_cast<const uint4*>(stg + r * wpr * 16 + 32 * j);
                const uint4 p = w[0], q = w[1];
                out = es == 4 ? make_uint4(p.x, p.z, q.x, q.z)
                              : make_uint4(__byte_perm(p.x, p.y, 0x5410), __byte_perm(p.z, p.w, 0x5410),
                                           __byte_perm(q.x, q.y, 0x5410), __byte_perm(q.z, q.w, 0x5410));
            } else if (kStep0) {
                const uint8_t* row = stg + r * wpr * 16 + ((gbase + off) & 15);
                const int step = (int)a.estride[0];
                out = es == 1   ? gather_chunk<uint8_t>(row, (int)j, x, step, fillv)
                      : es == 2 ? gather_chunk<uint16_t>(row, (int)j, x, step, fillv)
                      : es == 4 ? gather_chunk<uint32_t>(row, (int)j, x, step, fillv)
                                : gather_chunk<unsigned long long>(row, (int)j, x, step, fillv);
            } else {
                // The chunk is the 16 staged bytes starting d bytes into window j: read them with
                // the widest shared loads that offset allows (no realignment arithmetic).
                const uint32_t d = (uint32_t)((gbase + off) & 15);
                const uint8_t* const src = stg + (r * wpr + j) * 16 + d;
                if (d == 0) {
                    out = *reinterpret_cast<const uint4*>(src);
                } else if ((d & 7) == 0) {
                    const uint2 a = reinterpret_cast<const uint2*>(src)[0];
                    const uint2 b = reinterpret_cast<const uint2*>(src)[1];
                    out = make_uint4(a.x, a.y, b.x, b.y);
                } else if ((d & 3) == 0) {
                    const uint32_t* w = reinterpret_cast<const uint32_t*>(src);
                    out = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
                    out = unaligned_chunk(stg + (r * wpr + j) * 16, d);
                }
                if (!whole_x && (blo > 0 || bhi < 16)) {  // the chunk holding a row edge
                    uint32_t m = word_mask(blo, bhi, 0);
                    out.x = (out.x & m) | (fillv.x & ~m);
                    m = word_mask(blo, bhi, 1);
                    out.y = (out.y & m) | (fillv.y & ~m);
                    m = word_mask(blo, bhi, 2);
                    out.z = (out.z & m) | (fillv.z & ~m);
                    m = word_mask(blo, bhi, 3);
                    out.w = (out.w & m) | (fillv.w & ~m);
                }
            }
            *reinterpret_cast<uint4*>(
                img + swizzle_offset((r0 + r) * a.inner_bytes + j * 16, a.span)) = out;
        }
    }
}

// Writes bytes [pos, end) of a 16-byte chunk `v` to `dst` (the chunk's global address) with the
// widest stores both addresses allow.
__device__ __forceinline__ void store_chunk_bytes(uint8_t* dst, const uint4& v, int pos, int end)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    while (pos < end) {
        const uintptr_t at = reinterpret_cast<uintptr_t>(dst + pos);
        int wd = 16;
        while ((at & (uintptr_t)(wd - 1)) || (pos & (wd - 1)) || pos + wd > end) wd >>= 1;
        if (wd == 16) {
            *reinterpret_cast<uint4*>(dst) = v;
        } else if (wd == 8) {
            const uint32_t h = (uint32_t)pos >> 3;
            *reinterpret_cast<uint2*>(dst + pos) = make_uint2(h ? w[2] : w[0], h ? w[3] : w[1]);
        } else {
            const uint32_t word = sel4((uint32_t)pos >> 2, w[0], w[1], w[2], w[3]);
            if (wd == 4) {
                *reinterpret_cast<uint32_t*>(dst + pos) = word;
            } else if (wd == 2) {
                *reinterpret_cast<uint16_t*>(dst + pos) = (uint16_t)(word >> (8 * (pos & 3)));
            } else {
                dst[pos] = (uint8_t)(word >> (8 * (pos & 3)));
            }
        }
        pos += wd;
    }
}

// Store direction.  Image b is read straight from global memory: a warp's 32 chunks are 4
// consecutive 128-byte image rows (a swizzle only permutes chunks inside a row), so the 16-byte
// loads are coalesced; each thread keeps 4 in flight, then writes each chunk's in-bounds bytes
// with the widest stores the destination alignment allows.  Only the row table lives in shared
// memory; no wait on another thread's copy is involved.
// kStep0: elementStrides[0] is not 1; each chunk's in-bounds elements are written one by one,
// `estride[0]` elements apart.
template <bool kStep0>
__global__ void __launch_bounds__(kThreads, 6) k_fb_store(const __grid_constant__ FbArgs a)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ ItemWalk s_w;    // the current (row block, box) item, walked round-robin
    __shared__ int32_t s_c[5];  // its box start
    __shared__ XRange s_x;      // the box's in-bounds part along dim 0
    int64_t* const tab = reinterpret_cast<int64_t*>(smem_raw);
    constexpr int kLoads = 4;

    const uint32_t cpr = a.inner_bytes >> 4;
    const uint32_t cpr_shift = (cpr & (cpr - 1)) == 0 ? (uint32_t)(__ffs(cpr) - 1) : 32u;
    const uint32_t RB = a.block_rows;
    const uint32_t nblk = (a.rows + RB - 1) / RB;
    const uint64_t T = a.walk.nbox * nblk;
    if (T <= blockIdx.x) return;
    const uint64_t total = (T - 1 - blockIdx.x) / gridDim.x + 1;
    const int es = (int)a.esize;
    const int inner = (int)a.inner_bytes;

    for (uint64_t n = 0; n < total; n++) {
        if (threadIdx.x == 0) {
            if (n == 0) item_walk_init(a.walk, nblk, blockIdx.x, s_w);
            else item_walk_next(a.walk, nblk, s_w);
            item_box_start(a.walk, s_w, s_c);
            s_x = x_range(a, s_c[0]);
        }
        __syncthreads();  // the item is published; the previous block's table is no longer read
        const XRange x = s_x;
        const int lo_byte = x.i_lo * es, hi_byte = x.i_hi * es;
        const bool whole_x = lo_byte == 0 && hi_byte == inner;
        const uint8_t* const img = reinterpret_cast<const uint8_t*>(a.images + s_w.box * a.box_bytes);
        const int32_t* const c = s_c;
        {
            const uint32_t r0 = s_w.k[0] * RB;
            const uint32_t nr = min(RB, a.rows - r0);
            for (uint32_t r = threadIdx.x; r < nr; r += kThreads) {
                const RowPos p = row_position(a, c, r0 + r, a.stride);
                tab[r] = (p.ok && x.i_lo < x.i_hi) ? p.off : kRowOutside;
            }
            __syncthreads();
            if constexpr (kStep0) {
                // Element by element, consecutive threads on consecutive image elements of a row,
                // so that a warp's stores land elementStrides[0] elements apart in one stretch of
                // the row rather than one element in each of 32 chunks.
                // Four elements per thread per pass, all loaded before any is stored (one image
                // load per element and thread in flight was latency-bound: 36 % DRAM throughput).
                const uint32_t n0 = a.ibox[0];
                const uint32_t n0_shift = (n0 & (n0 - 1)) == 0 ? (uint32_t)(__ffs(n0) - 1) : 32u;
                const int step = (int)a.estride[0];
                const uint32_t nel = nr * n0;
                constexpr int kEl = 4;
                for (uint32_t e0 = threadIdx.x; e0 < nel; e0 += kThreads * kEl) {
                    unsigned long long v[kEl];
                    uint8_t* dst[kEl];
#pragma unroll
                    for (int u = 0; u < kEl; u++) {
                        const uint32_t e = e0 + u * kThreads;
                        dst[u] = nullptr;
                        v[u] = 0;
                        if (e >= nel) continue;
                        const uint32_t r = n0_shift < 32 ? e >> n0_shift : e / n0;
                        const int k = (int)(e - r * n0);
                        const int64_t off = tab[r];
                        if (off == kRowOutside || k < x.i_lo || k >= x.i_hi) continue;
                        const uint8_t* src = img + (size_t)(r0 + r) * a.inner_bytes + (size_t)k * es;
                        dst[u] = reinterpret_cast<uint8_t*>(a.base + off) + (int64_t)k * step * es;
                        v[u] = es == 2   ? __ldg(reinterpret_cast<const uint16_t*>(src))
                               : es == 4 ? __ldg(reinterpret_cast<const uint32_t*>(src))
                               : es == 8 ? __ldg(reinterpret_cast<const unsigned long long*>(src))
                                         : __ldg(src);
                    }
#pragma unroll
                    for (int u = 0; u < kEl; u++) {
                        if (!dst[u]) continue;
                        if (es == 2) {
                            *reinterpret_cast<uint16_t*>(dst[u]) = (uint16_t)v[u];
                        } else if (es == 4) {
                            *reinterpret_cast<uint32_t*>(dst[u]) = (uint32_t)v[u];
                        } else if (es == 8) {
                            *reinterpret_cast<unsigned long long*>(dst[u]) = v[u];
                        } else {
                            *dst[u] = (uint8_t)v[u];
                        }
                    }
                }
                continue;  // next item (a strided map is never swizzled: image rows are plain)
            }
            const uint32_t nch = nr * cpr;
            for (uint32_t it = threadIdx.x; it < nch; it += kThreads * kLoads) {
                uint4 v[kLoads];
#pragma unroll
                for (int k = 0; k < kLoads; k++) {
                    const uint32_t item = it + k * kThreads;
                    v[k] = make_uint4(0, 0, 0, 0);
                    if (item < nch) {
                        uint32_t r, j;
                        split_item(item, cpr, cpr_shift, r, j);
                        if (tab[r] != kRowOutside) {
                            v[k] = __ldg(reinterpret_cast<const uint4*>(
                                img + swizzle_offset((r0 + r) * a.inner_bytes + j * 16, a.span)));
                        }
                    }
                }
#pragma unroll
                for (int k = 0; k < kLoads; k++) {
                    const uint32_t item = it + k * kThreads;
                    if (item >= nch) continue;
                    uint32_t r, j;
                    split_item(item, cpr, cpr_shift, r, j);
                    const int64_t off = tab[r];
                    if (off == kRowOutside) continue;
                    const int pos = whole_x ? 0 : max(lo_byte - 16 * (int)j, 0);
                    const int end = whole_x ? 16 : min(hi_byte - 16 * (int)j, 16);
                    if (pos >= end) continue;
                    uint8_t* const chunk = reinterpret_cast<uint8_t*>(a.base + off + (int64_t)j * 16);
                    const uintptr_t at = reinterpret_cast<uintptr_t>(chunk);
                    if (pos == 0 && end == 16 && (at & 7) == 0) {  // whole chunk, 8-byte aligned
                        if ((at & 15) == 0) {
                            *reinterpret_cast<uint4*>(chunk) = v[k];
                        } else {
                            *reinterpret_cast<uint2*>(chunk) = make_uint2(v[k].x, v[k].y);
                            *reinterpret_cast<uint2*>(chunk + 8) = make_uint2(v[k].z, v[k].w);
                        }
                    } else {
                        store_chunk_bytes(chunk, v[k], pos, end);
                    }
                }
            }
        }
    }
}

// ---- reduce direction -------------------------------------------------------------------------
// op(a, b) for one element, a from dst, b from src (op 0 add, 1 min, 2 max).  Float adds: for two
// f16 or bf16 operands the binary32 sum is exact, or else too far from any 16-bit rounding midpoint
// to change the result, so rounding it to the element format gives the correctly rounded sum.
// Min / max keep dst on a tie of equal values.
template <int T>
__device__ __forceinline__ float to_f32(uint32_t bits)
{
    if constexpr (T == 1) return __half2float(__ushort_as_half((unsigned short)bits));
    if constexpr (T == 2) return __uint_as_float(bits << 16);
    return __uint_as_float(bits);
}

template <int T>
__device__ __forceinline__ uint32_t from_f32(float v)
{
    if constexpr (T == 1) return __half_as_ushort(__float2half_rn(v));
    if constexpr (T == 2) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    return __float_as_uint(v);
}

template <int T, int OP>
__device__ __forceinline__ uint32_t combine(uint32_t a, uint32_t b)
{
    if constexpr (T == 3) {  // u32
        return OP == 0 ? a + b : OP == 1 ? (b < a ? b : a) : (b > a ? b : a);
    } else if constexpr (T == 4) {  // s32
        const int32_t x = (int32_t)a, y = (int32_t)b;
        return OP == 0 ? a + b : (uint32_t)(OP == 1 ? (y < x ? y : x) : (y > x ? y : x));
    } else {
        const float x = to_f32<T>(a), y = to_f32<T>(b);
        if constexpr (OP == 1) return y < x ? b : a;
        if constexpr (OP == 2) return y > x ? b : a;
        return from_f32<T>(__fadd_rn(x, y));
    }
}

// Applies op to the elements of a 16-byte vector pair (4 x 32-bit or 8 x 16-bit elements).
template <int T, int OP>
__device__ __forceinline__ uint4 combine_vec(uint4 d, const uint4& s)
{
    uint32_t* dw = reinterpret_cast<uint32_t*>(&d);
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(&s);
#pragma unroll
    for (int w = 0; w < 4; w++) {
        if constexpr (T == 1 || T == 2) {
            const uint32_t lo = combine<T, OP>(dw[w] & 0xffffu, sw[w] & 0xffffu);
            const uint32_t hi = combine<T, OP>(dw[w] >> 16, sw[w] >> 16);
            dw[w] = (lo & 0xffffu) | (hi << 16);
        } else {
            dw[w] = combine<T, OP>(dw[w], sw[w]);
        }
    }
    return d;
}

// dst = op(dst, src) over the whole box grid.  The grid covers every in-bounds element exactly
// once and the op is element-wise (the image's swizzle cancels between load and store), so the
// kernel walks the tensor's rows (dim 0 runs) directly: work items are 16 KiB segments of a row;
// rows whose dst and src start on the same 16-byte phase go with 16-byte vector loads and stores
// (elements before the first and after the last full vector one by one), other rows element by
// element.
template <int T, int OP>
__device__ void fb_reduce_rows(const FbArgs& a)
{
    using E = typename std::conditional<(T == 1 || T == 2), uint16_t, uint32_t>::type;
    constexpr int es = (int)sizeof(E);
    constexpr uint32_t kVecPerLane = 4;
    constexpr uint64_t kSegBytes = 8192;  // one warp's item: 8 KiB of a row (4 passes of vectors)
    // A row is dim 0 and every following dim that is contiguous with it in both tensors (a view
    // that splits a row, like the rank-5 W4 view's 10 x 100, is walked as its whole rows).
    uint32_t f = 1;
    uint64_t row_elems = a.dim[0];
    while (f < a.walk.rank && a.stride[f] == (int64_t)(row_elems * es) &&
           a.src_stride[f] == (int64_t)(row_elems * es)) {
        row_elems *= a.dim[f];
        f++;
    }
    const uint64_t row_bytes = row_elems * es;
    const uint64_t segs = (row_bytes + kSegBytes - 1) / kSegBytes;
    uint64_t nrows = 1;
    for (uint32_t i = f; i < a.walk.rank; i++) nrows *= a.dim[i];
    const uint64_t items = nrows * segs;
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t w0 = (uint64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const uint64_t nw = (uint64_t)gridDim.x * (kThreads / 32);
    // The warp's items are w0, w0 + nw, ...: item it is piece seg of row `row`, whose counters
    // over dims f.. are g[].  They are found by division once; each step then adds nw items as
    // (rows dr, pieces ds) and the row step's digits dg[], with carries.
    // (Loops run over the fixed 5 dims, guarded, so that g[] and dg[] stay in registers.)
    const int rank = (int)a.walk.rank, f0 = (int)f;
    uint64_t seg = w0 % segs;
    uint64_t g[5] = {0, 0, 0, 0, 0}, dg[5] = {0, 0, 0, 0, 0};
    {
        uint64_t q = w0 / segs, qs = nw / segs;
#pragma unroll
        for (int i = 1; i < 5; i++) {
            if (i >= f0 && i < rank) {
                if (i + 1 < rank) {
                    g[i] = q % a.dim[i];
                    q /= a.dim[i];
                    dg[i] = qs % a.dim[i];
                    qs /= a.dim[i];
                } else {  // the top digits take what is left (past the end: never used)
                    g[i] = q;
                    dg[i] = qs;
                }
            }
        }
    }
    const uint64_t ds = nw % segs;
    for (uint64_t it = w0; it < items; it += nw) {
        int64_t od = 0, os = 0;
#pragma unroll
        for (int i = 1; i < 5; i++) {
            if (i >= f0 && i < rank) {
                od += (int64_t)g[i] * a.stride[i];
                os += (int64_t)g[i] * a.src_stride[i];
            }
        }
        const uint64_t cur_seg = seg;
        // step to item it + nw
        seg += ds;
        uint64_t carry = 0;
        if (seg >= segs) {
            seg -= segs;
            carry = 1;
        }
#pragma unroll
        for (int i = 1; i < 5; i++) {
            if (i >= f0 && i < rank) {
                uint64_t v = g[i] + dg[i] + carry;
                carry = 0;
                if (i + 1 < rank && v >= a.dim[i]) {
                    v -= a.dim[i];
                    carry = 1;
                }
                g[i] = v;
            }
        }
        uint8_t* const d = reinterpret_cast<uint8_t*>(a.base + od);
        const uint8_t* const sp = reinterpret_cast<const uint8_t*>(a.src_base + os);
        const uint64_t b0 = cur_seg * kSegBytes;
        const uint64_t b1 = min(b0 + kSegBytes, row_bytes);
        const uint32_t phase = (uint32_t)((uintptr_t)d & 15);
        uint64_t vs = b1, ve = b1;  // whole 16-byte vectors in [vs, ve) when both phases agree
        if (phase == ((uintptr_t)sp & 15)) {
            const uint64_t first_vec = ((uint64_t)((uintptr_t)d + b0) + 15) / 16 * 16 - (uintptr_t)d;
            vs = min(first_vec, b1);
            ve = vs + (b1 - vs) / 16 * 16;
        }
        // head [b0, vs) and tail [ve, b1) element by element
        for (uint64_t x = b0 + lane * es; x < vs; x += 32 * es) {
            E* p = reinterpret_cast<E*>(d + x);
            *p = (E)combine<T, OP>((uint32_t)*p, (uint32_t)*reinterpret_cast<const E*>(sp + x));
        }
        const uint64_t nv = (ve - vs) / 16;
        for (uint64_t v = lane; v < nv; v += 32 * kVecPerLane) {
            uint4 dv[kVecPerLane], sv[kVecPerLane];
#pragma unroll
            for (uint32_t u = 0; u < kVecPerLane; u++) {
                const uint64_t vi = v + u * 32;
                if (vi < nv) {
                    dv[u] = *reinterpret_cast<const uint4*>(d + vs + vi * 16);
                    sv[u] = __ldg(reinterpret_cast<const uint4*>(sp + vs + vi * 16));
                }
            }
#pragma unroll
            for (uint32_t u = 0; u < kVecPerLane; u++) {
                const uint64_t vi = v + u * 32;
                if (vi < nv)
                    *reinterpret_cast<uint4*>(d + vs + vi * 16) = combine_vec<T, OP>(dv[u], sv[u]);
            }
        }
        for (uint64_t x = ve + lane * es; x < b1; x += 32 * es) {
            E* p = reinterpret_cast<E*>(d + x);
            *p = (E)combine<T, OP>((uint32_t)*p, (uint32_t)*reinterpret_cast<const E*>(sp + x));
        }
    }
}

template <int T, int OP>
__global__ void __launch_bounds__(kThreads, 3) k_fb_reduce(const __grid_constant__ FbArgs a)
{
    fb_reduce_rows<T, OP>(a);
}

namespace {
// The grid cut to the CTAs the device's SMs hold at once (the occupancy calculator's answer for
// this kernel, block size and shared memory): these kernels split their items by gridDim.x, so
// fewer CTAs only take more items each, while CTAs beyond what the SMs hold would run as a second,
// short wave (12 CTAs of 256 threads per SM asked for 3072 threads where an SM holds 2048).
uint32_t resident_grid(void (*k)(const FbArgs), uint32_t grid, size_t smem)
{
    int per_sm = 0, dev = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, smem) != cudaSuccess ||
        cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return grid;
    }
    const uint64_t hold = (uint64_t)per_sm * (uint64_t)sms;
    return hold > 0 && hold < grid ? (uint32_t)hold : grid;
}
}  // namespace

cudaError_t launch_fb_copy(const FbArgs& a, uint32_t grid, size_t smem, cudaStream_t s)
{
    void (*k)(const FbArgs) = a.estride[0] != 1 ? k_fb_copy<true> : k_fb_copy<false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<resident_grid(k, grid, smem), kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fb_store(const FbArgs& a, uint32_t grid, size_t smem, cudaStream_t s)
{
    void (*k)(const FbArgs) = a.estride[0] != 1 ? k_fb_store<true> : k_fb_store<false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<resident_grid(k, grid, smem), kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fb_reduce(const FbArgs& a, uint32_t grid, cudaStream_t s)
{
    using Fn = void (*)(const FbArgs);
    static const Fn table[5][3] = {
        {k_fb_reduce<0, 0>, k_fb_reduce<0, 1>, k_fb_reduce<0, 2>},
        {k_fb_reduce<1, 0>, k_fb_reduce<1, 1>, k_fb_reduce<1, 2>},
        {k_fb_reduce<2, 0>, k_fb_reduce<2, 1>, k_fb_reduce<2, 2>},
        {k_fb_reduce<3, 0>, k_fb_reduce<3, 1>, k_fb_reduce<3, 2>},
        {k_fb_reduce<4, 0>, k_fb_reduce<4, 1>, k_fb_reduce<4, 2>},
    };
    if (a.red_type > 4 || a.red_op > 2) return cudaErrorInvalidValue;
    table[a.red_type][a.red_op]<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace tmk
