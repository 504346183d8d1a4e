// k_fallback.cu -- generic path for maps the tensor-map hardware cannot take (a base or stride
// that is a multiple of the element size but not of 16 bytes, e.g. a 200-byte group stride), and
// for explicit box lists the hardware must not be given (see tmap_host.cpp).
//
// The image is built exactly as the TMA path builds it -- same swizzle, zero fill outside the
// tensor -- but by the CTA's threads: each thread owns one 16-byte chunk of an image row, loads
// the aligned 16-byte window under the chunk's first byte, takes the following window from its
// neighbour lane with a warp shuffle (loading it itself only where the neighbour does not hold
// it: the row's last chunk, the warp's last lane), realigns the 32 bytes with funnel shifts and
// stores the chunk to its swizzled place with a 16-byte shared store ([H200-TMA] = coolgpu "H200 · TMA · Tensor Memory Accelerator" card, §02:
// the per-thread cp.async style of addressing that TMA replaces).  A proxy fence then hands the
// image to the same 1-D bulk store the TMA path uses.
//
// A window is only loaded when it holds at least one in-bounds byte of the chunk; an aligned
// 16-byte window never crosses a page, so no load can touch an unmapped address.
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
// negative) and whether every outer coordinate (dims 1..) is inside the tensor.
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
            const uint32_t bi = a.walk.box[i];
            const uint32_t q = r / bi;
            const int64_t g = (int64_t)c[i] + (int64_t)(r - q * bi);
            r = q;
            p.ok = p.ok && g >= 0 && (uint64_t)g < a.dim[i];
            p.off += g * stride[i];
        }
    }
    return p;
}

// In-bounds element range [k0, k1) of chunk j of a row whose element 0 has dim-0 coordinate x0.
__device__ __forceinline__ void chunk_range(int64_t x0, uint32_t j, uint32_t epc, uint64_t dim0,
                                            int& k0, int& k1)
{
    const int64_t first = x0 + (int64_t)j * epc;
    if (first >= 0 && first + (int64_t)epc <= (int64_t)dim0) {  // the common case: all inside
        k0 = 0;
        k1 = (int)epc;
        return;
    }
    const int64_t lo = first < 0 ? -first : 0;
    const int64_t hi = (int64_t)dim0 - first;
    k0 = (int)(lo < (int64_t)epc ? lo : (int64_t)epc);
    k1 = (int)(hi < 0 ? 0 : hi < (int64_t)epc ? hi : (int64_t)epc);
}

}  // namespace

constexpr int64_t kRowOutside = INT64_MIN;  // table entry of a row outside the tensor
constexpr int kBatch = 4;                    // chunks per thread whose loads are in flight together

// Per-box table of image-row offsets (relative to the tensor base; kRowOutside when an outer
// coordinate is outside the tensor), shared by every chunk of the row.
__device__ __forceinline__ void fill_row_table(const FbArgs& a, const int32_t* c, int64_t* tab,
                                               const int64_t* stride)
{
    for (uint32_t r = threadIdx.x; r < a.table_rows; r += kThreads) {
        const RowPos p = row_position(a, c, r, stride);
        tab[r] = p.ok ? p.off : kRowOutside;
    }
}

__device__ __forceinline__ int64_t row_offset(const FbArgs& a, const int32_t* c, const int64_t* tab,
                                              uint32_t row, const int64_t* stride)
{
    if (a.table_rows) return tab[row];
    const RowPos p = row_position(a, c, row, stride);
    return p.ok ? p.off : kRowOutside;
}

// Image row and chunk of item `item` (chunks of a row are consecutive items).
__device__ __forceinline__ void split_item(uint32_t item, uint32_t cpr, uint32_t cpr_shift,
                                           uint32_t& row, uint32_t& j)
{
    row = cpr_shift < 32 ? item >> cpr_shift : item / cpr;
    j = item - row * cpr;
}

__global__ void __launch_bounds__(kThreads) k_fb_copy(const __grid_constant__ FbArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + (kStageAlign - 1)) & ~(kStageAlign - 1);
    uint8_t* const stage0 = smem_raw + (base - raw);
    const uint32_t SB = a.stages;
    int64_t* const tab = reinterpret_cast<int64_t*>(stage0 + SB * a.stage_bytes);

    const uint64_t first = blockIdx.x;
    if (a.walk.nbox <= first) return;
    const uint64_t n_local = (a.walk.nbox - 1 - first) / gridDim.x + 1;

    const uint32_t lane = threadIdx.x & 31;
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t cpr = a.inner_bytes >> 4;  // 16-byte chunks per row
    const uint32_t cpr_shift = (cpr & (cpr - 1)) == 0 ? (uint32_t)(__ffs(cpr) - 1) : 32u;
    const uint32_t nchunks = a.rows * cpr;
    const uint32_t es = a.esize;
    const uint32_t epc = 16 / es;             // elements per chunk
    const int64_t gbase = (int64_t)a.base;

    for (uint64_t i = 0; i < n_local; i++) {
        const uint64_t b = first + i * gridDim.x;
        const uint32_t st = (uint32_t)(i % SB);
        uint8_t* const stage = stage0 + st * a.stage_bytes;
        int32_t c[5];
        box_start(a.walk, b, c);
        if (threadIdx.x == 0) {  // the write that last used this stage has read it
            if (SB == 2 && i >= 2) bulk_wait_read<1>();
            if (SB == 1 && i >= 1) bulk_wait_read<0>();
        }
        __syncthreads();  // also: every thread is done with the previous box's row table
        fill_row_table(a, c, tab, a.stride);
        __syncthreads();

        // Each warp takes 32 consecutive chunks per slot, kBatch slots per pass (trip count is
        // warp-uniform); all of a pass's loads are issued before any is used.  Per slot the thread
        // keeps its first window, the second window when no neighbour lane will hold it (the row's
        // last chunk, the warp's last lane, or a neighbour whose chunk is outside the tensor), and
        // one packed word: bits 0..3 d (misalignment), 4 need_lo, 5 need_hi, 6 valid, 7 own hi,
        // 8..14 j, 15.. row.
        for (uint32_t it = warp * 32; it < nchunks; it += kThreads * kBatch) {
            uint4 lo[kBatch], own[kBatch];
            uint32_t meta[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; k++) {
                const uint32_t item = it + k * kThreads + lane;
                const bool valid = item < nchunks;
                uint32_t row = 0, j = 0;
                if (valid) split_item(item, cpr, cpr_shift, row, j);
                const int64_t off = valid ? row_offset(a, c, tab, row, a.stride) : kRowOutside;
                int k0 = 0, k1 = 0;
                chunk_range(c[0], j, epc, a.dim[0], k0, k1);
                const bool any = off != kRowOutside && k0 < k1;
                const int64_t addr = gbase + (any ? off : 0) + (int64_t)j * 16;
                const uint32_t d = (uint32_t)addr & 15u;
                const bool need_lo = any && k0 * (int)es < 16 - (int)d;
                const bool need_hi = any && d != 0 && k1 * (int)es > 16 - (int)d;
                // The neighbour (same row, next chunk) loads the second window exactly when its
                // first element is inside the tensor.
                const int64_t next_x = (int64_t)c[0] + (int64_t)(j + 1) * epc;
                const bool nb_loads = lane < 31 && j + 1 < cpr && next_x >= 0 &&
                                      next_x < (int64_t)a.dim[0];
                const bool own_hi = need_hi && !nb_loads;
                meta[k] = d | (need_lo ? 1u << 4 : 0u) | (need_hi ? 1u << 5 : 0u) |
                          (valid ? 1u << 6 : 0u) | (own_hi ? 1u << 7 : 0u) | (j << 8) | (row << 15);
                const uint4* w0 = reinterpret_cast<const uint4*>(addr - (int64_t)d);
                lo[k] = need_lo ? __ldg(w0) : make_uint4(0, 0, 0, 0);
                own[k] = own_hi ? __ldg(w0 + 1) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < kBatch; k++) {
                const uint32_t d = meta[k] & 15u;
                const bool need_lo = (meta[k] >> 4) & 1u, need_hi = (meta[k] >> 5) & 1u;
                const bool valid = (meta[k] >> 6) & 1u, own_hi = (meta[k] >> 7) & 1u;
                const uint32_t j = (meta[k] >> 8) & 127u, row = meta[k] >> 15;
                uint4 nb;
                nb.x = __shfl_down_sync(0xffffffffu, lo[k].x, 1);
                nb.y = __shfl_down_sync(0xffffffffu, lo[k].y, 1);
                nb.z = __shfl_down_sync(0xffffffffu, lo[k].z, 1);
                nb.w = __shfl_down_sync(0xffffffffu, lo[k].w, 1);
                if (!valid) continue;
                const uint4 hi = !need_hi ? make_uint4(0, 0, 0, 0) : own_hi ? own[k] : nb;
                uint4 out = make_uint4(0, 0, 0, 0);
                int k0 = 0, k1 = 0;
                chunk_range(c[0], j, epc, a.dim[0], k0, k1);
                const bool whole = k0 == 0 && k1 == (int)epc;
                if (whole && d == 0) {  // aligned and inside: the window is the chunk
                    out = lo[k];
                } else if (whole && d == 8) {  // inside, 8-byte aligned: two words from each window
                    out = make_uint4(lo[k].z, lo[k].w, hi.x, hi.y);
                } else if (need_lo || need_hi) {
                    const int lo_b = k0 * (int)es, hi_b = k1 * (int)es;
                    const uint32_t q = d >> 2, sh = (d & 3u) * 8u;
                    const uint32_t w[8] = {lo[k].x, lo[k].y, lo[k].z, lo[k].w,
                                           hi.x, hi.y, hi.z, hi.w};
                    uint32_t o[4];
#pragma unroll
                    for (int t = 0; t < 4; t++) {
                        const uint32_t x = sel4(q, w[t], w[t + 1], w[t + 2], w[t + 3]);
                        const uint32_t y = sel4(q, w[t + 1], w[t + 2], w[t + 3], w[t + 4]);
                        o[t] = __funnelshift_r(x, y, sh) & word_mask(lo_b, hi_b, t);
                    }
                    out = make_uint4(o[0], o[1], o[2], o[3]);
                }
                *reinterpret_cast<uint4*>(stage + swizzle_offset(row * a.inner_bytes + j * 16,
                                                                 a.span)) = out;
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            bulk_store(a.images + b * a.box_bytes, base + st * a.stage_bytes, a.box_bytes);
            bulk_commit();
        }
    }
    if (threadIdx.x == 0) bulk_wait_all<0>();
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

// Store direction: image b is bulk-loaded into a stage, then each thread writes the in-bounds
// bytes of its chunks with the widest stores the destination alignment allows.
__global__ void __launch_bounds__(kThreads) k_fb_store(const __grid_constant__ FbArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[2];
    __shared__ int wait_ok;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + (kStageAlign - 1)) & ~(kStageAlign - 1);
    uint8_t* const stage0 = smem_raw + (base - raw);
    const uint32_t SB = a.stages;
    int64_t* const tab = reinterpret_cast<int64_t*>(stage0 + SB * a.stage_bytes);

    const uint64_t first = blockIdx.x;
    if (a.walk.nbox <= first) return;
    const uint64_t n_local = (a.walk.nbox - 1 - first) / gridDim.x + 1;
    const uint32_t cpr = a.inner_bytes >> 4;
    const uint32_t cpr_shift = (cpr & (cpr - 1)) == 0 ? (uint32_t)(__ffs(cpr) - 1) : 32u;
    const uint32_t nchunks = a.rows * cpr;
    const uint32_t es = a.esize;
    const uint32_t epc = 16 / es;

    auto issue = [&](uint64_t i) {
        const uint32_t st = (uint32_t)(i % SB);
        const uint32_t bar = smem_u32(&full_bar[st]);
        mbar_arrive_expect_tx(bar, a.box_bytes);
        bulk_load(base + st * a.stage_bytes, a.images + (first + i * gridDim.x) * a.box_bytes,
                  a.box_bytes, bar);
    };

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&full_bar[0]), 1);
        mbar_init(smem_u32(&full_bar[1]), 1);
        fence_barrier_init();
        issue(0);
        if (SB == 2 && n_local > 1) issue(1);
    }

    for (uint64_t i = 0; i < n_local; i++) {
        const uint32_t st = (uint32_t)(i % SB);
        int32_t c[5];
        box_start(a.walk, first + i * gridDim.x, c);
        fill_row_table(a, c, tab, a.stride);  // the previous box's table is no longer read
        if (threadIdx.x == 0) {
            const uint32_t parity = (uint32_t)((i / SB) & 1);
            const bool ok = mbar_wait(smem_u32(&full_bar[st]), parity, a.timeout_ns);
            if (!ok) {
                record_timeout(a.status, K_FB_STORE, st, parity, first + i * gridDim.x);
                if (SB == 2 && i + 1 < n_local) {  // the other stage's load may still be landing
                    mbar_wait(smem_u32(&full_bar[st ^ 1]), (uint32_t)(((i + 1) >> 1) & 1),
                              a.timeout_ns);
                }
            }
            wait_ok = ok ? 1 : 0;
        }
        __syncthreads();
        if (!wait_ok) break;

        const uint8_t* const stage = stage0 + st * a.stage_bytes;
        for (uint32_t item = threadIdx.x; item < nchunks; item += kThreads) {
            uint32_t row, j;
            split_item(item, cpr, cpr_shift, row, j);
            const int64_t off = row_offset(a, c, tab, row, a.stride);
            int k0 = 0, k1 = 0;
            chunk_range(c[0], j, epc, a.dim[0], k0, k1);
            if (off == kRowOutside || k0 >= k1) continue;
            const uint4 v = *reinterpret_cast<const uint4*>(
                stage + swizzle_offset(row * a.inner_bytes + j * 16, a.span));
            uint8_t* const chunk = reinterpret_cast<uint8_t*>(a.base + off + (int64_t)j * 16);
            const uintptr_t at = reinterpret_cast<uintptr_t>(chunk);
            if (k0 == 0 && k1 == (int)epc && (at & 7) == 0) {  // whole chunk, 8-byte aligned
                if ((at & 15) == 0) {
                    *reinterpret_cast<uint4*>(chunk) = v;
                } else {
                    *reinterpret_cast<uint2*>(chunk) = make_uint2(v.x, v.y);
                    *reinterpret_cast<uint2*>(chunk + 8) = make_uint2(v.z, v.w);
                }
            } else {
                store_chunk_bytes(chunk, v, k0 * (int)es, k1 * (int)es);
            }
        }
        fence_proxy_async_smem();  // generic reads of the stage before the next async write to it
        __syncthreads();
        if (threadIdx.x == 0 && i + SB < n_local) issue(i + SB);
    }
}

// Reduce direction on the fallback path: dst += src element by element (the swizzle of the image
// in between cancels between load and store, so the element read is src at the same coordinate).
__global__ void __launch_bounds__(kThreads) k_fb_reduce(const __grid_constant__ FbArgs a)
{
    const uint32_t lane = threadIdx.x & 31;
    const uint64_t warps = (uint64_t)gridDim.x * (kThreads / 32);
    const uint64_t total = a.walk.nbox * a.rows;
    const uint32_t box0 = a.walk.box[0];
    for (uint64_t rr = (uint64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); rr < total;
         rr += warps) {
        const uint64_t b = rr / a.rows;
        const uint32_t row = (uint32_t)(rr - b * a.rows);
        int32_t c[5];
        box_start(a.walk, b, c);
        const RowPos pd = row_position(a, c, row, a.stride);
        if (!pd.ok) continue;
        const RowPos ps = row_position(a, c, row, a.src_stride);
        for (uint32_t k = lane; k < box0; k += 32) {
            const int64_t x = (int64_t)c[0] + k;
            if (x < 0 || (uint64_t)x >= a.dim[0]) continue;
            float* d = reinterpret_cast<float*>(a.base + pd.off + (int64_t)k * 4);
            const float* s = reinterpret_cast<const float*>(a.src_base + ps.off + (int64_t)k * 4);
            *d = __fadd_rn(*d, *s);
        }
    }
}

cudaError_t launch_fb_copy(const FbArgs& a, uint32_t grid, size_t smem, cudaStream_t s)
{
    cudaError_t e =
        cudaFuncSetAttribute(k_fb_copy, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_fb_copy<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fb_store(const FbArgs& a, uint32_t grid, size_t smem, cudaStream_t s)
{
    cudaError_t e =
        cudaFuncSetAttribute(k_fb_store, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_fb_store<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fb_reduce(const FbArgs& a, uint32_t grid, cudaStream_t s)
{
    k_fb_reduce<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace tmk
