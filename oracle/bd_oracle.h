/*
 * bd_oracle.h -- plain single-threaded CPU oracle of the BF16 field-split delta format.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the cpu_baseline /
 * reference arm of bench.py may call, link or execute this code.  The product path (the
 * CUDA library) never uses it and shares no code, header, table or constant with it.
 *
 * What it computes follows
 *   [ARCv3]  "Every byte counts: ARCv3 and the case for cross-region RL" -- the paragraph on
 *            how ARCv3 encodes the mantissa/exponent asymmetry and the figure "How ARCv3
 *            encodes a block of weights" (XOR each prev/next pair, classify by changed field,
 *            omit unchanged, keep only mantissa bits of mantissa-only changes, pack the rarer
 *            exponent/sign changes separately as one block, checksum the result);
 *            the API listing (delta_compress returns (compressed_diff, checksum);
 *            delta_decompress(src, compressed_diff, checksum) restores dst bit for bit).
 *   [WT]     "GPU-accelerated Weight Teleportation", section "Delta update algebra"
 *            (mask = old XOR new; old XOR mask = new; bits only, no floating point).
 * Everything below the field split (chunking, position coding, byte layout, checksum
 * formula) is not on the pages; it is this library's format "BF16DLT1" version 1, whose
 * written specification the oracle follows step by step.
 */
#ifndef BD_ORACLE_H
#define BD_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Oracle status codes (numerically equal to the library's, but defined independently). */
enum {
  ORC_OK = 0,
  ORC_ERR_ARG = 1,
  ORC_ERR_CAPACITY = 2,
  ORC_ERR_FORMAT = 3,
  ORC_ERR_CHECKSUM = 4,
  ORC_ERR_BASE = 6      /* a version-2 payload applied to weights of another base version */
};

/* 64-bit checksum of n BF16 words (see bd_oracle.c for the definition). */
uint64_t orc_checksum(const uint16_t* w, uint64_t n);

/* Encodes the delta old -> neu (n elements).  Always stores the exact payload size in
 * *size_out and the checksum of neu in *checksum_out.  Writes the payload into out only when
 * cap >= size; otherwise returns ORC_ERR_CAPACITY and leaves out untouched. */
int orc_encode(const uint16_t* old, const uint16_t* neu, uint64_t n, uint8_t* out,
               uint64_t cap, uint64_t* size_out, uint64_t* checksum_out);

/* orc_encode writing a version-2 payload bound to its base version: the 80-byte header
 * carries `base` (the checksum of old, as the caller knows it) and 8 reserved zero bytes;
 * everything after the header is as in version 1. */
int orc_encode_versioned(const uint16_t* old, const uint16_t* neu, uint64_t n, uint64_t base,
                         uint8_t* out, uint64_t cap, uint64_t* size_out, uint64_t* checksum_out);

/* orc_encode_versioned writing a version-3 payload (compact positions: a merged gap-byte
 * list with escapes and class bits per chunk, see bd_oracle.c). */
int orc_encode_compact(const uint16_t* old, const uint16_t* neu, uint64_t n, uint64_t base,
                       uint8_t* out, uint64_t cap, uint64_t* size_out, uint64_t* checksum_out);

/* orc_encode_versioned / orc_encode_compact writing an overwrite payload (header flags bit 0):
 * the same positions and classes, the streams holding new values instead of XOR masks. */
int orc_encode_overwrite(const uint16_t* old, const uint16_t* neu, uint64_t n, uint64_t base,
                         uint8_t* out, uint64_t cap, uint64_t* size_out, uint64_t* checksum_out);
int orc_encode_compact_overwrite(const uint16_t* old, const uint16_t* neu, uint64_t n,
                                 uint64_t base, uint8_t* out, uint64_t cap, uint64_t* size_out,
                                 uint64_t* checksum_out);

/* orc_encode_versioned writing a version-4 payload (Rice-coded compact position blocks, see
 * bd_oracle.c); overwrite != 0 gives an overwrite payload as above. */
int orc_encode_rice(const uint16_t* old, const uint16_t* neu, uint64_t n, uint64_t base,
                    int overwrite, uint8_t* out, uint64_t cap, uint64_t* size_out,
                    uint64_t* checksum_out);

/* Decodes payload[0..size) (version 1, 2, 3 or 4; the base of a bound payload is not checked
 * here) against old (n elements) into out (n elements, must not alias
 * old), then verifies checksum(out) == expected.  Returns ORC_OK, ORC_ERR_FORMAT (payload
 * is not a canonical BF16DLT1 payload for n elements) or ORC_ERR_CHECKSUM.  On an error
 * the contents of out are unspecified. */
int orc_decode(const uint16_t* old, uint64_t n, const uint8_t* payload, uint64_t size,
               uint64_t expected, uint16_t* out);

/* Incremental verification (not on the pages; the rollout side often knows the checksum of
 * the weights it holds from its previous verified update).  Decodes like orc_decode (same
 * format rules), then computes
 *   ck = ck_old + sum over the words j where out differs from old of
 *          mix64(out_word_j ^ (j+1)*GAMMA) - mix64(old_word_j ^ (j+1)*GAMMA)   (mod 2^64)
 * which equals checksum(out) whenever ck_old == checksum(old).  Stores ck in *ck_out (when
 * not NULL and the payload is well formed) and returns ORC_OK when ck == expected, else
 * ORC_ERR_CHECKSUM (or ORC_ERR_FORMAT / ORC_ERR_ARG as orc_decode).  A version-2 payload whose
 * base checksum differs from ck_old gives ORC_ERR_BASE (after the header and count table are
 * checked, before any chunk is decoded). */
int orc_decode_incremental(const uint16_t* old, uint64_t n, const uint8_t* payload,
                           uint64_t size, uint64_t ck_old, uint64_t expected, uint16_t* out,
                           uint64_t* ck_out);

#ifdef __cplusplus
}
#endif

#endif /* BD_ORACLE_H */
