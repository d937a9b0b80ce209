/*
 * bf16delta.h -- C ABI of libbf16delta, lossless delta sync of BF16 weights on one GB300.
 *
 * The operations are the ones described in
 *   [ARCv3] "Every byte counts: ARCv3 and the case for cross-region RL"
 *     - the paragraph on encoding the mantissa/exponent asymmetry and the figure
 *       "How ARCv3 encodes a block of weights": each old/new BF16 pair is XORed and
 *       classified by the field that changed; unchanged values are omitted; mantissa-only
 *       changes contribute just their mantissa bits; the rarer exponent/sign changes are
 *       packed separately, all their changed fields as one block; on the rollout side both
 *       streams are applied to the previous checkpoint and the result is checksummed
 *       against the trainer's original;
 *     - the API listing: delta_compress(src, dst) -> (compressed_diff, checksum) and
 *       delta_decompress(src, compressed_diff, checksum) -> restored, bit-identical to dst.
 *   [WT] "GPU-accelerated Weight Teleportation", section "Delta update algebra":
 *       mask = old XOR new on the trainer; old XOR mask = new on the rollout side; the
 *       weights are plain bits (no floating-point arithmetic, no rounding).
 *
 * Payload format "BF16DLT1" version 1 (the pages fix only the field split; the rest is this
 * library's format).  x = old ^ new as u16.  A change is mantissa-only (M) when x != 0 and
 * (x & 0xFF80) == 0, rare (R) when (x & 0xFF80) != 0.  Tensors are cut into chunks of
 * 4096 elements (C = ceil(n/4096), the last chunk may be shorter, length L_c).
 * Little-endian, no padding between sections:
 *   [header 64 B] [count table: C x {u16 M_c, u16 R_c}] [R stream: u16 x per R element]
 *   [positions: per chunk, the M block then the R block] [M stream: 7 bits (x & 0x7F) per
 *   M element, element j in stream bits [7j, 7j+7), bit b = bit b%8 of byte b/8, pad 0]
 * A position block with k entries for a chunk of length L is a delta list of k u16
 * (d_0 = p_0, d_j = p_j - p_{j-1}) when 2k < ceil(L/8), else a ceil(L/8)-byte bitmap
 * (bit p = bit p%8 of byte p/8).  Elements inside every stream are in ascending position.
 * Header: "BF16DLT1", u32 version=1, u32 chunk_elems=4096, u64 n, u64 C, u64 sum M,
 * u64 sum R, u64 position bytes, u64 total size.
 * Version 2 (bd_compress_versioned, format 2): the same payload with an 80-byte header --
 * version 2, the 64 bytes above, then u64 base checksum (the checksum of the weights the
 * payload applies to) and u64 flags (0 for an XOR payload) -- so every section starts 16
 * bytes later.
 * Version 3 (format 3): the version-2 header with version 3, and compact position blocks
 * standing in for the entropy stage the ARCv3 page applies to the sparse positions (which it
 * does not specify).  Sections:
 *   [header 80 B] [count table: C x u32] [R stream] [X stream: u16 per escaped gap]
 *   [positions] [M stream]
 * A count entry with bit 31 set marks a compact chunk: M in bits 0..8, R in 9..17, E in
 * 18..26, bits 27..30 zero, 1 <= M + R <= 508, E <= M + R.  Its block merges the chunk's
 * changes into one ascending list: M + R gap bytes (gap_0 = p_0 + 1, gap_i = p_i - p_{i-1};
 * a gap above 255 is written as 0 and its value taken from the X stream, E of them in order)
 * then ceil((M+R)/8) class bytes (bit i set: change i is rare; pad bits 0).  An entry with
 * bit 31 clear has M in bits 0..14, R in 15..29, bit 30 zero, and version-1 blocks.  Compress
 * codes a chunk compactly exactly when it has 1..508 changes and M + R + ceil((M+R)/8) + 2E
 * is below the bytes of its two version-1 blocks, so a version-3 payload is never longer
 * than the version-2 payload of the same update.  The header's position-bytes field counts
 * the position section only; the X stream is what the other sections leave of the total.
 * Version 4 (format 4): version 3 with the compact blocks coded by a Golomb-Rice code of the
 * same gaps instead (a second stand-in for the unspecified entropy stage), and no X stream:
 *   [header 80 B] [count table: C x u32] [R stream] [positions] [M stream]
 * A compact count entry (bit 31 set) holds M in bits 0..8, R in 9..17, the Rice parameter K
 * in 18..20 and the block's length B in bytes in 21..30 (1 <= M + R <= 508, B >= 1); plain
 * entries are as in version 3.  The block is a bit stream, bit b = bit b%8 of byte b/8: the
 * indices of the R rare changes in the merged list (9 bits each, strictly ascending, below
 * M + R), then each gap's remainder gap mod 2^K (K bits), then each gap's quotient gap >> K
 * in unary (that many 1 bits, then a 0), then 0 bits up to the end of byte B - 1, which must
 * be the byte holding the last used bit.  Every gap is at least 1 and every position below L.
 * Compress takes the K in 0..7 giving the fewest bits (the smallest on a tie) and codes a
 * chunk compactly exactly when it has 1..508 changes and B is below the bytes of its two
 * version-1 blocks, so a version-4 payload is never longer than the version-2 payload of the
 * same update.
 * Every decompress call accepts all four versions.
 * Overwrite payloads (versions 2 to 4 with header flags bit 0 = BD_FLAG_OVERWRITE; the u64 at
 * byte 72, whose other bits are zero): the NeMo-DCR page's second form of update payload,
 * absolute overwrites, through which partial writes are retried.  Positions, classes and
 * sizes are those of the XOR payload of the same update; the R stream holds each rare
 * element's new value and the M stream each mantissa-only element's new mantissa.  Applying
 * one writes those fields into place -- the new value, or the new mantissa under the element's
 * own sign and exponent (which a mantissa-only change does not alter) -- so applying it again,
 * to weights it has already updated wholly or in part, gives the same result.  The XOR
 * payload's value rules (a nonzero mantissa mask, a rare mask with a sign or exponent bit) do
 * not apply to it.
 * Checksum (returned beside the payload, not stored in it): with word_j the little-endian
 * 64-bit word of elements 4j..4j+3 (zero past n),
 *   checksum = sum_j mix64(word_j ^ (j+1) * 0x9E3779B97F4A7C15)  mod 2^64,
 * mix64 being the SplitMix64 output function (Steele, Lea & Flood 2014).
 *
 * Conventions for every call:
 *   - "d_" pointers are device memory, "h_" pointers host memory, all owned by the caller.
 *     The library allocates nothing; scratch comes from a caller-provided workspace.
 *   - BF16 tensors are arrays of uint16_t bit patterns, 16-byte aligned.  Payload
 *     buffers are 16-byte aligned; workspaces 256-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream).  Results are written to device memory in stream order.
 *   - The return value reports argument and launch errors only (BD_ERR_INVALID_ARG,
 *     BD_ERR_CUDA); nothing has been enqueued when it is not BD_OK.  Errors found on the
 *     device (capacity, format, checksum) arrive in the int32 status words.
 *   - The same workspace must not be used by two calls that may overlap on the GPU.
 */
#ifndef BF16DELTA_H
#define BF16DELTA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols (the library is built with hidden visibility otherwise). */
#if defined(__GNUC__)
#define BD_API __attribute__((visibility("default")))
#else
#define BD_API
#endif

typedef enum bd_status {
  BD_OK = 0,
  BD_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment, overlap or workspace size */
  BD_ERR_CAPACITY = 2,    /* compress: payload larger than the capacity given */
  BD_ERR_FORMAT = 3,      /* decompress: not a canonical BF16DLT1 payload for n elements */
  BD_ERR_CHECKSUM = 4,    /* decompress: checksum of the result differs from the expected */
  BD_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed (as a device status:
                             a wait inside the compress gave up, which its design excludes;
                             then the call and every tensor of it report this code, see
                             bf16delta_debug.h) */
  BD_ERR_BASE = 6         /* incremental apply: a payload of version 2 or later whose base checksum
                             is not the checksum of the weights it is applied to */
} bd_status;

#define BD_CHUNK_ELEMS 4096u
#define BD_HEADER_BYTES 64u
/* Largest tensor accepted, in elements (2^40, i.e. 2 TiB of BF16). */
#define BD_MAX_ELEMS (1ull << 40)

/* One tensor of a batched compress.  All device pointers; d_status may be NULL. */
typedef struct bd_compress_item {
  const uint16_t* d_old;  /* trainer weights before the step (n elements) */
  const uint16_t* d_new;  /* trainer weights after the step (n elements) */
  uint64_t n;             /* elements */
  void* d_payload;        /* output buffer of cap bytes */
  uint64_t cap;           /* capacity of d_payload in bytes */
  uint64_t* d_size;       /* out: exact payload size (also when it exceeds cap) */
  uint64_t* d_checksum;   /* out: checksum of d_new */
  int32_t* d_status;      /* out (optional): BD_OK or BD_ERR_CAPACITY */
} bd_compress_item;

/* One tensor of a batched decompress.  All device pointers; d_status may be NULL. */
typedef struct bd_decompress_item {
  const uint16_t* d_old;         /* rollout weights before the step (n elements) */
  uint16_t* d_out;               /* result (n elements); == d_old for an in-place apply */
  uint64_t n;                    /* elements */
  const void* d_payload;         /* payload produced by compress for this tensor */
  uint64_t size;                 /* payload bytes */
  const uint64_t* d_expected;    /* expected checksum of the result (from compress) */
  int32_t* d_status;             /* out (optional): BD_OK, BD_ERR_FORMAT or BD_ERR_CHECKSUM */
} bd_decompress_item;

/* One tensor of a batched incremental apply (bd_decompress_incremental_batch).  All device
 * pointers; d_ck_out and d_status may be NULL. */
typedef struct bd_incremental_item {
  uint16_t* d_w;                 /* rollout weights, updated in place (n elements) */
  uint64_t n;                    /* elements */
  const void* d_payload;         /* payload produced by compress for this tensor */
  uint64_t size;                 /* payload bytes */
  const uint64_t* d_ck_old;      /* checksum of d_w before the call */
  const uint64_t* d_expected;    /* expected checksum of the result (from compress) */
  uint64_t* d_ck_out;            /* out (optional): the result's checksum, computed as below */
  int32_t* d_status;             /* out (optional): BD_OK, BD_ERR_FORMAT or BD_ERR_CHECKSUM */
} bd_incremental_item;

/* Parsed payload header (host side).  base_checksum is 0 for a version-1 payload;
 * n_escapes (X-stream values) is 0 except in version 3; flags is the header flags word of
 * versions 2 to 4 (BD_FLAG_OVERWRITE: an overwrite payload), 0 for version 1. */
typedef struct bd_payload_info_t {
  uint64_t n, chunks, n_mant, n_rare, position_bytes, total_size;
  uint32_t version, chunk_elems;
  uint64_t base_checksum;
  uint64_t n_escapes;
  uint64_t flags;
} bd_payload_info_t;

/* Header flag of an overwrite payload, and the bit of bd_compress_versioned's format argument
 * that asks for one. */
#define BD_FLAG_OVERWRITE 1u
#define BD_FORMAT_OVERWRITE 0x100u

/* Library utility: no passage on the pages.  Largest payload compress can produce for n
 * elements (every chunk at its worst split, with the version-2 header), so a caller can size
 * a payload buffer before the first call.  Returns 0 for n > BD_MAX_ELEMS. */
BD_API uint64_t bd_compress_bound(uint64_t n);

/* Library utility: no passage on the pages.  Workspace bytes needed by bd_compress_batch /
 * bd_decompress_batch for k tensors of h_n[0..k) elements (k = 1 for the single-tensor
 * calls); h_n is a host array read during the call.  Returns 0 on bad arguments. */
BD_API uint64_t bd_compress_workspace_size(const uint64_t* h_n, uint32_t k);
BD_API uint64_t bd_decompress_workspace_size(const uint64_t* h_n, uint32_t k);

/* [ARCv3] delta_compress: encodes old -> new into d_payload and returns the checksum of new.
 * Writes the exact payload size to *d_size and the checksum to *d_checksum.  If the payload
 * does not fit in cap bytes, the status is BD_ERR_CAPACITY, *d_size still holds the size
 * needed and the payload bytes are unspecified.  d_status (optional, may be NULL) receives
 * BD_OK or BD_ERR_CAPACITY.  d_old and d_new may not overlap d_payload or d_ws. */
BD_API int bd_compress(const uint16_t* d_old, const uint16_t* d_new, uint64_t n, void* d_payload,
                uint64_t cap, void* d_ws, uint64_t ws_bytes, uint64_t* d_size,
                uint64_t* d_checksum, int32_t* d_status, void* stream);

/* Batched compress: one launch per phase for k tensors; each tensor's payload, size and
 * checksum are byte-identical to a single-tensor call.  h_items is read during the call
 * only.  d_status (optional) receives the largest status code over the tensors. */
BD_API int bd_compress_batch(const bd_compress_item* h_items, uint32_t k, void* d_ws,
                      uint64_t ws_bytes, int32_t* d_status, void* stream);

/* bd_compress writing a payload bound to its base version: format 2 (the version-1 payload
 * with the 80-byte header), 3 (compact position blocks, see above) or 4 (Rice-coded compact
 * position blocks), each optionally OR-ed with BD_FORMAT_OVERWRITE for an overwrite payload;
 * any other format is BD_ERR_INVALID_ARG.  Not on the pages: the NeMo-DCR page binds the installed weights to
 * the baseline of the next delta so that mismatched versions cannot enter silently.
 * *d_base_checksum (device, required) is the checksum of d_old as the caller knows it -- in
 * a steady update loop, the checksum of the previous update's new weights; it is stored in
 * the header, not recomputed.  The incremental apply refuses the payload with BD_ERR_BASE
 * when the receiver's checksum of its weights differs; bd_payload_info exposes the base for
 * a check on the host before a full apply.  Sizes, capacity and workspace as bd_compress
 * (bd_compress_bound covers every format). */
BD_API int bd_compress_versioned(const uint16_t* d_old, const uint16_t* d_new, uint64_t n,
                                 void* d_payload, uint64_t cap, void* d_ws, uint64_t ws_bytes,
                                 uint64_t* d_size, uint64_t* d_checksum,
                                 const uint64_t* d_base_checksum, uint32_t format,
                                 int32_t* d_status, void* stream);

/* Batched bd_compress_versioned, every item in the same format: h_base_checksums[i] (host
 * array of k device pointers, each required) is the base checksum of item i. */
BD_API int bd_compress_versioned_batch(const bd_compress_item* h_items,
                                       const uint64_t* const* h_base_checksums, uint32_t k,
                                       uint32_t format, void* d_ws, uint64_t ws_bytes,
                                       int32_t* d_status, void* stream);

/* [ARCv3] delta_decompress, [WT] weights_updated = weights_old XOR mask: applies the payload
 * to d_old, writing the result to d_out (d_out == d_old applies in place; any other overlap
 * is BD_ERR_INVALID_ARG), then verifies checksum(result) == *d_expected.  *d_status receives
 * BD_OK, BD_ERR_FORMAT or BD_ERR_CHECKSUM.  Chunks found malformed are left unwritten; on
 * any error an in-place apply can be undone by applying the same payload again (XOR is an
 * involution and decoding depends on the payload only). */
BD_API int bd_decompress(const uint16_t* d_old, uint64_t n, const void* d_payload, uint64_t size,
                  const uint64_t* d_expected, uint16_t* d_out, void* d_ws,
                  uint64_t ws_bytes, int32_t* d_status, void* stream);

/* Batched decompress: one launch per phase for k tensors.  *d_status (required) receives
 * the largest status code over the tensors; per-tensor codes go to the items' d_status. */
BD_API int bd_decompress_batch(const bd_decompress_item* h_items, uint32_t k, void* d_ws,
                        uint64_t ws_bytes, int32_t* d_status, void* stream);

/* bd_decompress_batch with every payload in HOST memory, streamed through two device slots:
 * the SM-only analog of the double-buffered pipeline of [WT], section "Double compression with
 * heterogeneous decompression" (payloads staged in pinned host RAM; one of two layer-sized
 * buffers is filled while the GPU applies from the other, so no device copy of the whole
 * update is needed).  Here the copy engines fill a slot instead of the decompression engine.
 * The items are cut, in order, into groups whose payloads (each placed at a 256-byte
 * boundary) fit in slot_bytes; group g's payloads are copied into slot g % 2 of d_staging on
 * copy_stream while group g - 1 is applied on stream, and a slot is refilled only after the
 * apply that read it.  Each item's d_payload is a HOST address (page-locked memory, e.g.
 * cudaHostAlloc, for the copies to overlap; pageable memory works but each copy may block the
 * host); it must stay valid and unchanged until stream has passed the call.  Payloads that
 * lie in host memory at the distances they take in the slot are copied together, with the
 * bytes between them.
 * d_staging: device, 256-byte aligned, 2 * slot_bytes bytes, slot_bytes a multiple of 256
 * (at most 2^40) and at least the largest payload rounded up to 256; it may not overlap any
 * output or the workspace.  copy_stream: a stream other than stream (use non-blocking streams:
 * the legacy default stream would serialise the copies with the applies).  The workspace is
 * bd_decompress_workspace_size of all k tensors.  Results, per-tensor statuses and *d_status
 * (required; the largest status over all tensors) are those of bd_decompress_batch on the
 * same items with device payloads.  Every argument is checked before anything is enqueued:
 * BD_ERR_INVALID_ARG otherwise (also for a payload larger than a slot); BD_ERR_CUDA when the
 * runtime refuses an event, copy or launch, with earlier groups possibly enqueued.  The call
 * creates five CUDA events and destroys them before it returns (no memory is allocated). */
BD_API int bd_decompress_batch_streamed(const bd_decompress_item* h_items, uint32_t k,
                                        void* d_staging, uint64_t slot_bytes, void* d_ws,
                                        uint64_t ws_bytes, int32_t* d_status, void* stream,
                                        void* copy_stream);

/* In-place apply verified incrementally.  Not on the pages, which verify by checksumming the
 * restored weights: a rollout process that applies updates one after another already holds
 * a verified checksum of its current weights (the expected checksum of its previous update),
 * so the terms of the unchanged words are known and only the changed words need new terms:
 *   ck = *d_ck_old + sum over the words the payload changes of
 *          mix64(new_word_j ^ (j+1)*G) - mix64(old_word_j ^ (j+1)*G)     (mod 2^64)
 * which equals the checksum of the result whenever *d_ck_old is the checksum of d_w before
 * the call.  The status is BD_OK when ck == *d_expected, else BD_ERR_CHECKSUM (format errors
 * as bd_decompress); ck goes to *d_ck_out when given.  A payload of version 2 or later whose base
 * checksum differs from *d_ck_old is refused with BD_ERR_BASE and nothing is written.  Only the 32-byte sectors holding
 * changes are read and written (plus the payload), against a full read of the tensor for
 * bd_decompress.  What it does not verify: a word of d_w that differs from the trainer's
 * old copy but is not touched by the payload (bd_decompress's full read catches that).
 * The workspace is bd_decompress_workspace_size's for the same tensors.  Malformed chunks
 * are left unwritten; applying the same payload again (with the checksums swapped) undoes
 * the call. */
BD_API int bd_decompress_incremental(uint16_t* d_w, uint64_t n, const void* d_payload,
                                     uint64_t size, const uint64_t* d_ck_old,
                                     const uint64_t* d_expected, uint64_t* d_ck_out,
                                     void* d_ws, uint64_t ws_bytes, int32_t* d_status,
                                     void* stream);

/* Batched bd_decompress_incremental: one launch per phase for k tensors.  *d_status
 * (required) receives the largest status code over the tensors. */
BD_API int bd_decompress_incremental_batch(const bd_incremental_item* h_items, uint32_t k,
                                           void* d_ws, uint64_t ws_bytes, int32_t* d_status,
                                           void* stream);

/* Largest tensor bd_decompress_noalloc accepts, in elements (2^27 = 128 Mi elements,
 * 256 MiB of BF16), and the size of the device array it uses as scratch. */
#define BD_NOALLOC_MAX_ELEMS (1ull << 27)
#define BD_NOALLOC_SCRATCH_BYTES (1ull << 20)

/* bd_decompress for callers that cannot allocate device memory.  The pages have no
 * counterpart of this call; it exists for users of this library, not for the method.
 *
 * Who needs it: a rollout or inference engine whose allocator already holds almost all of
 * HBM (weights plus a pre-reserved KV cache) cannot hand out a workspace, and calling
 * cudaMalloc / cudaFree from such a process either fails, fragments the engine's pool or
 * stalls the device at the wrong moment.  This entry point needs no workspace argument: its
 * scratch is a fixed BD_NOALLOC_SCRATCH_BYTES array in the library's device memory, which
 * every GPU that loads the library holds until the process exits.
 *
 * Arguments, result and status are those of bd_decompress.  Differences:
 *   - n above BD_NOALLOC_MAX_ELEMS is rejected with BD_ERR_INVALID_ARG before anything is
 *     enqueued;
 *   - it decodes every chunk with the block-level decoder, so it is slower than
 *     bd_decompress with a workspace;
 *   - all calls share the one scratch array (it keeps the last call's contents; each call
 *     clears what must start at zero), so two calls that may overlap on the GPU race:
 *     issue them on one stream, or order them with events;
 *   - every call looks up the array's device address on the current device (a host call,
 *     no allocation; so a device reset leaves no stale address behind); the first call on a
 *     device also loads the library's module there, so make that first call before any
 *     stream capture begins;
 *   - d_expected must be 8-byte and d_status 4-byte aligned, as for bd_decompress.
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine. */
BD_API int bd_decompress_noalloc(const uint16_t* d_old, uint64_t n, const void* d_payload,
                                 uint64_t size, const uint64_t* d_expected, uint16_t* d_out,
                                 int32_t* d_status, void* stream);

/* [ARCv3], the paragraph on encoding the mantissa/exponent asymmetry: the rollout side
 * checksums the restored weights against the trainer's original.  The page names no formula;
 * this computes the one given at the top of this header (sum of position-keyed SplitMix64
 * word terms) over the n BF16 values at d_w and writes it to *d_out, asynchronously on
 * stream.  n = 0 gives 0.  Needs no workspace; d_w 16-byte aligned, d_out 8-byte aligned. */
BD_API int bd_checksum(const uint16_t* d_w, uint64_t n, uint64_t* d_out, void* stream);

/* Library utility: no passage on the pages (the header layout is this library's format).
 * Parses and checks a payload header held in host memory (bytes >= 64; >= 80 for versions 2
 * to 4).  Checks magic, version, chunk size and the internal consistency of the header
 * fields (for version 3 the total leaves an even number of bytes, at most 2 * 508 per chunk,
 * for the X stream); returns BD_OK, BD_ERR_FORMAT or BD_ERR_INVALID_ARG.  Does not touch the
 * GPU. */
BD_API int bd_payload_info(const void* h_header, uint64_t bytes, bd_payload_info_t* out);

/* Library utility: no passage on the pages.  Waits for `stream` (the host blocks) and
 * returns the int32 status word at d_status, which must be device-readable and 4-byte
 * aligned (or BD_ERR_CUDA when the wait or the read fails). */
BD_API int bd_status_sync(const int32_t* d_status, void* stream);

/* Library utility: no passage on the pages.  Static description of a status code (never
 * NULL; unknown codes give a generic string). */
BD_API const char* bd_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* BF16DELTA_H */
