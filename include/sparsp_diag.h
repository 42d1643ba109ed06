/*
 * sparsp_diag.h - diagnostic entry point of libsparsp (not part of the
 * attention path): one 128 x 128 x 128 bf16 tile product on the tcgen05 tensor
 * cores, built from exactly the TMA boxes, shared-memory descriptors and TMEM
 * operand layout that sparsp_attn_fwd uses. A test compares it with a plain
 * product to check those layouts on the device.
 */
#ifndef SPARSP_DIAG_H
#define SPARSP_DIAG_H

#include "sparsp.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * a, b: device bf16 [128, 128] row-major, 16-byte aligned; d: device float32
 * [128, 128] row-major (written). One CTA on `stream`; returns
 * SPARSP_ERR_UNSUPPORTED on devices other than compute capability 10.x.
 *   mode 0: D = A B^T, A and B staged by TMA, both K-major (the S = Q K^T form).
 *   mode 1: D = A B,   A written to TMEM as packed bf16 rows, B staged by TMA
 *           and read MN-major (the O += P V form).
 *   mode 2: D = A B,   A staged by TMA (K-major), B MN-major.
 * lbo, sbo: leading / stride byte offsets of the MN-major B descriptor
 * (multiples of 16, at most 32768; ignored in mode 0).
 * d_status: device int32 (required, caller-zeroed). Every wait of the kernel
 * is bounded (1 s); if the tile copies or the MMAs do not complete in time,
 * SPARSP_ERR_TIMEOUT is written there, the work still in flight is drained
 * with a second bounded wait, and d is left unwritten.
 */
SPARSP_API sparsp_status_t sparsp_diag_umma_tile(const void* a, const void* b, float* d, int32_t mode,
                                                 int32_t lbo, int32_t sbo, int32_t* d_status,
                                                 sparsp_stream_t stream);

/*
 * The bounded-wait path of the tensor-core kernels, exercised on purpose: one
 * CTA waits, through the same bounded mbarrier wait the attention kernels use,
 * on a barrier phase that nothing completes. After limit_ns nanoseconds
 * (1e6 <= limit_ns <= 5e9, else SPARSP_ERR_INVALID_ARG) the wait gives up,
 * SPARSP_ERR_TIMEOUT is written to *d_status (device int32, required) and the
 * kernel returns normally, so the context stays usable. No fault, trap or
 * unbounded wait is involved.
 */
SPARSP_API sparsp_status_t sparsp_diag_wait_timeout(uint64_t limit_ns, int32_t* d_status, sparsp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSP_DIAG_H */
