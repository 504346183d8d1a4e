/* tmap_onegpu.h -- C ABI of libtmap_gb300_onegpu.so, the separately built one-GPU-only companion
 * of libtmap_gb300.so (include/tmap.h).
 *
 * [H200-TMA] coolgpu "H200 · TMA · Tensor Memory Accelerator" feature card, §01 是什么 and §04 ③:
 * a TMA load with cluster multicast lands one copy of a box in the shared memory of several CTAs of
 * a cluster (a 16-bit CTA mask; the launch must be a cluster launch), which saves L2 and global
 * bandwidth when several CTAs need the same tile.
 *
 * Why a separate library: a multicast load is kept out of libtmap_gb300.so, which every rank of a
 * multi-GPU command loads.  This library is built only on request
 * (async_bulk_tensor_tmap_gb300/onegpu/build.py, never by the package's default build), loaded only
 * by async_bulk_tensor_tmap_gb300.onegpu, and used by no benchmark or multi-GPU command.  It reads
 * only memory of the GPU it runs on: every call checks, with cudaPointerGetAttributes, that each
 * tensor it is given is device memory of the current device, and returns TM_EINVAL otherwise; it
 * also refuses to run (TM_EUNSUPPORTED) in a process whose WORLD_SIZE says it is one rank of
 * several.
 *
 * Status codes are those of tmap.h (TM_OK, TM_EINVAL, ...).  Descriptors are tm_desc values filled
 * by tmap_encode() of libtmap_gb300.so; this library reads them and never writes them.
 */
#ifndef TMAP_GB300_ONEGPU_H
#define TMAP_GB300_ONEGPU_H

#include "tmap.h"

#ifdef __cplusplus
extern "C" {
#endif

/* stream_gemm_multicast -- C = A * B^T on the tensor cores, as stream_gemm() of tmap.h, with the B
 *   tile shared by the two CTAs of a cluster ([H200-TMA] §04 ③).  Clusters of two one-SM CTAs
 *   compute the 128 x 256 tiles (2m, n) and (2m + 1, n) of C; per k step each CTA loads its own A
 *   tile and ONE 128-row half of the B tile with cp.async.bulk.tensor ... .multicast::cluster (CTA
 *   mask 0b11), so both halves land at the same stage offset in both CTAs' shared memory and count
 *   on both CTAs' stage barriers (48 KiB each: A and both halves); each CTA's MMA commits arrive on
 *   both CTAs' empty barriers, so neither refills a stage the other still reads.  Each SM pulls
 *   32 KiB per k step from L2 instead of 48.
 *   a: rank-2 TM_BF16 map {K, M} with box {64, 128}; b_half: rank-2 TM_BF16 map {K, N} of B with box
 *   {64, 128} (a half tile); both 128-byte swizzle, tensor-map path, unit steps, zero fill, equal K
 *   (else TM_EUNSUPPORTED / TM_EINVAL); M, N, K below 2^31.  c: device fp32, row-major M x N, ldc
 *   >= N elements between rows, 16-byte aligned, ldc a multiple of 4 (else TM_EALIGN).  stages:
 *   2..4 (48 KiB stages; else TM_ERANGE).  A, B and C must be device memory of the current device
 *   (else TM_EINVAL).  Accuracy as stream_gemm.  Asynchronous on `stream`; a wait that gives up is
 *   reported by tm_onegpu_check(). */
int stream_gemm_multicast(const tm_desc* a, const tm_desc* b_half, float* c, uint64_t ldc,
                          uint32_t stages, void* stream);

/* tm_onegpu_check -- synchronise `stream`, then read and clear this library's status word for the
 *   current device: TM_ETIMEOUT if a bounded wait of its kernel gave up, TM_ECUDA on a CUDA error,
 *   else TM_OK. */
int tm_onegpu_check(void* stream);

/* The thread's last error text of this library. */
const char* tm_onegpu_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* TMAP_GB300_ONEGPU_H */
