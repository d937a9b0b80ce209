/*
 * bf16delta_debug.h -- fault injection into libbf16delta, for tests of its error paths.
 *
 * The batched compress of version-1 payloads runs as one persistent kernel in which a warp
 * that is to emit a tensor waits until another warp has finished counting that tensor.  The
 * schedule guarantees that every such wait ends; each is bounded all the same (about one
 * second of idle polling), after which the kernel reports BD_ERR_CUDA and returns, leaving the
 * CUDA context usable.  The hook below makes one wait run out on purpose, on the host's say,
 * without any fault: nothing is ever left pending on the GPU beyond that bound.
 */
#ifndef BF16DELTA_DEBUG_H
#define BF16DELTA_DEBUG_H

#include "bf16delta.h"

#ifdef __cplusplus
extern "C" {
#endif

/* bd_compress_batch with tensor `stall` (0 <= stall < k) never published: its count of
 * encoded chunks starts at a value that never reaches the tensor's chunk count, so the warps
 * that claim its emit work wait until their bound runs out.  Arguments as bd_compress_batch.
 * The call must take the persistent compress (every tensor at most 4096 batches of chunks;
 * true for all tensors up to 2^24 elements), else BD_ERR_INVALID_ARG, with nothing enqueued,
 * as for stall >= k.  Outcome on the stream, about one second later: d_status and every
 * tensor's d_status hold BD_ERR_CUDA; payloads, sizes and checksums are unspecified.  The
 * workspace may be used again by the next call. */
BD_API int bd_debug_compress_stall(const bd_compress_item* h_items, uint32_t k, uint32_t stall,
                                   void* d_ws, uint64_t ws_bytes, int32_t* d_status,
                                   void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BF16DELTA_DEBUG_H */
