// k_fallback.cu -- generic path for maps the tensor-map hardware cannot take (a base or stride
// that is a multiple of the element size but not of 16 bytes, e.g. a 200-byte group stride), and
// for explicit box lists the hardware must not be given (see tmap_host.cpp).
//
// The image is built exactly as the TMA path builds it -- same swizzle, zero fill outside the
// tensor -- but by the CTA's threads: each thread owns one 16-byte chunk of an image row, loads
// the aligned 16-byte window under the chunk's first byte, takes the following window from its
// neighbour lane with a warp shuffle (loading it itself only where the neighbour does not hold
// it), realigns the 32 bytes with funnel shifts and stores the chunk to its swizzled place with a
// 16-byte shared store ([H200-TMA] = coolgpu "H200 · TMA · Tensor Memory Accelerator" card, §02:
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
    const int64_t lo = first < 0 ? -first : 0;
    const int64_t hi = (int64_t)dim0 - first;
    k0 = (int)(lo < (int64_t)epc ? lo : (int64_t)epc);
    k1 = (int)(hi < 0 ? 0 : hi < (int64_t)epc ? hi : (int64_t)epc);
}

}  // namespace

__global__ void __launch_bounds__(kThreads) k_fb_copy(const __grid_constant__ FbArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + (kStageAlign - 1)) & ~(kStageAlign - 1);
    uint8_t* const stage0 = smem_raw + (base - raw);

    const uint64_t first = blockIdx.x;
    if (a.walk.nbox <= first) return;
    const uint64_t n_local = (a.walk.nbox - 1 - first) / gridDim.x + 1;

    const uint32_t lane = threadIdx.x & 31;
    const uint32_t warp = threadIdx.x >> 5;
    const uint32_t cpr = a.inner_bytes >> 4;   // 16-byte chunks per row
    const uint32_t nchunks = a.rows * cpr;
    const uint32_t es = a.esize;
    const uint32_t epc = 16 / es;              // elements per chunk
    const uint64_t gbase = a.base;

    for (uint64_t i = 0; i < n_local; i++) {
        const uint64_t b = first + i * gridDim.x;
        const uint32_t st = (uint32_t)(i & 1);
        uint8_t* const stage = stage0 + st * a.stage_bytes;
        if (threadIdx.x == 0 && i >= 2) bulk_wait_read<1>();  // box i - 2's write left this stage
        __syncthreads();

        int32_t c[5];
        box_start(a.walk, b, c);

        for (uint32_t it = warp * 32; it < nchunks; it += kThreads) {  // warp-uniform trip count
            const uint32_t item = it + lane;
            const bool valid = item < nchunks;
            const uint32_t row = valid ? item / cpr : 0;
            const uint32_t j = item - row * cpr;
            const RowPos rp = row_position(a, c, row, a.stride);
            int k0 = 0, k1 = 0;
            chunk_range(c[0], j, epc, a.dim[0], k0, k1);
            const bool any = valid && rp.ok && k0 < k1;
            const int64_t addr = (int64_t)gbase + rp.off + (int64_t)j * 16;
            const uint32_t d = (uint32_t)addr & 15u;
            const uint64_t w0 = (uint64_t)(addr - (int64_t)d);
            const int lo_b = k0 * (int)es, hi_b = k1 * (int)es;
            const bool need_lo = any && lo_b < 16 - (int)d;
            const bool need_hi = any && d != 0 && hi_b > 16 - (int)d;

            uint4 lo = make_uint4(0, 0, 0, 0);
            if (need_lo) lo = __ldg(reinterpret_cast<const uint4*>(w0));
            // The next lane's first window is this lane's second one when it holds the next
            // chunk of the same row and loaded it.
            const uint32_t nb_has = __shfl_down_sync(0xffffffffu, need_lo ? 1u : 0u, 1);
            uint4 nb;
            nb.x = __shfl_down_sync(0xffffffffu, lo.x, 1);
            nb.y = __shfl_down_sync(0xffffffffu, lo.y, 1);
            nb.z = __shfl_down_sync(0xffffffffu, lo.z, 1);
            nb.w = __shfl_down_sync(0xffffffffu, lo.w, 1);
            uint4 hi = make_uint4(0, 0, 0, 0);
            if (need_hi) {
                if (lane < 31 && j + 1 < cpr && nb_has) {
                    hi = nb;
                } else {
                    hi = __ldg(reinterpret_cast<const uint4*>(w0 + 16));
                }
            }
            if (!valid) continue;
            uint4 out = make_uint4(0, 0, 0, 0);
            if (any) {
                const uint32_t q = d >> 2, sh = (d & 3u) * 8u;
                const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                uint32_t o[4];
#pragma unroll
                for (int t = 0; t < 4; t++) {
                    const uint32_t x = sel4(q, w[t], w[t + 1], w[t + 2], w[t + 3]);
                    const uint32_t y = sel4(q, w[t + 1], w[t + 2], w[t + 3], w[t + 4]);
                    o[t] = __funnelshift_r(x, y, sh) & word_mask(lo_b, hi_b, t);
                }
                out = make_uint4(o[0], o[1], o[2], o[3]);
            }
            const uint32_t soff = swizzle_offset(row * a.inner_bytes + j * 16, a.span);
            *reinterpret_cast<uint4*>(stage + soff) = out;
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

// Store direction: image b is bulk-loaded into a stage, then each thread writes the in-bounds
// bytes of its chunk with the widest stores the destination alignment allows.
__global__ void __launch_bounds__(kThreads) k_fb_store(const __grid_constant__ FbArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[2];
    __shared__ int wait_ok;
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + (kStageAlign - 1)) & ~(kStageAlign - 1);
    uint8_t* const stage0 = smem_raw + (base - raw);

    const uint64_t first = blockIdx.x;
    if (a.walk.nbox <= first) return;
    const uint64_t n_local = (a.walk.nbox - 1 - first) / gridDim.x + 1;
    const uint32_t cpr = a.inner_bytes >> 4;
    const uint32_t nchunks = a.rows * cpr;
    const uint32_t es = a.esize;
    const uint32_t epc = 16 / es;

    auto issue = [&](uint64_t i) {
        const uint32_t st = (uint32_t)(i & 1);
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
        if (n_local > 1) issue(1);
    }

    for (uint64_t i = 0; i < n_local; i++) {
        const uint32_t st = (uint32_t)(i & 1);
        if (threadIdx.x == 0) {
            const uint32_t parity = (uint32_t)((i >> 1) & 1);
            const bool ok = mbar_wait(smem_u32(&full_bar[st]), parity, a.timeout_ns);
            if (!ok) {
                record_timeout(a.status, K_FB_STORE, st, parity, first + i * gridDim.x);
                if (i + 1 < n_local) {  // the other stage's load may still be landing
                    mbar_wait(smem_u32(&full_bar[st ^ 1]), (uint32_t)(((i + 1) >> 1) & 1),
                              a.timeout_ns);
                }
            }
            wait_ok = ok ? 1 : 0;
        }
        __syncthreads();
        if (!wait_ok) break;

        const uint8_t* const stage = stage0 + st * a.stage_bytes;
        int32_t c[5];
        box_start(a.walk, first + i * gridDim.x, c);
        for (uint32_t item = threadIdx.x; item < nchunks; item += kThreads) {
            const uint32_t row = item / cpr;
            const uint32_t j = item - row * cpr;
            const RowPos rp = row_position(a, c, row, a.stride);
            int k0 = 0, k1 = 0;
            chunk_range(c[0], j, epc, a.dim[0], k0, k1);
            if (!rp.ok || k0 >= k1) continue;
            const uint4 v = *reinterpret_cast<const uint4*>(
                stage + swizzle_offset(row * a.inner_bytes + j * 16, a.span));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint8_t* const chunk = reinterpret_cast<uint8_t*>(a.base + rp.off + (int64_t)j * 16);
            int pos = k0 * (int)es;
            const int end = k1 * (int)es;
            while (pos < end) {
                const uintptr_t at = reinterpret_cast<uintptr_t>(chunk + pos);
                int wd = 16;
                while ((at & (uintptr_t)(wd - 1)) || (pos & (wd - 1)) || pos + wd > end) wd >>= 1;
                if (wd == 16) {
                    *reinterpret_cast<uint4*>(chunk) = v;
                } else if (wd == 8) {
                    const uint32_t h = (uint32_t)pos >> 2;
                    *reinterpret_cast<uint2*>(chunk + pos) =
                        make_uint2(sel4(h >> 1, w[0], w[2], w[0], w[2]),
                                   sel4(h >> 1, w[1], w[3], w[1], w[3]));
                } else if (wd == 4) {
                    *reinterpret_cast<uint32_t*>(chunk + pos) =
                        sel4((uint32_t)pos >> 2, w[0], w[1], w[2], w[3]);
                } else if (wd == 2) {
                    const uint32_t word = sel4((uint32_t)pos >> 2, w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint16_t*>(chunk + pos) =
                        (uint16_t)(word >> (8 * (pos & 3)));
                } else {
                    const uint32_t word = sel4((uint32_t)pos >> 2, w[0], w[1], w[2], w[3]);
                    chunk[pos] = (uint8_t)(word >> (8 * (pos & 3)));
                }
                pos += wd;
            }
        }
        fence_proxy_async_smem();  // generic reads of the stage before the next async write to it
        __syncthreads();
        if (threadIdx.x == 0 && i + 2 < n_local) issue(i + 2);
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
