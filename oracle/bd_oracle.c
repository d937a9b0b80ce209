/*
 * bd_oracle.c -- plain, slow, single-threaded CPU oracle of the BF16DLT1 delta format.
 *
 * TEST INFRASTRUCTURE ONLY (see bd_oracle.h): never part of the product path.
 *
 * The steps follow the pages in their order:
 *   1. XOR every old/new BF16 pair ([WT] "Delta update algebra"; [ARCv3] figure "How ARCv3
 *      encodes a block of weights": each prev/next pair is XORed).
 *   2. Classify each XOR by the field that changed ([ARCv3] same figure): zero (unchanged),
 *      mantissa-only, or exponent/sign ("rare").
 *   3. Omit unchanged elements: only the positions of changed elements are recorded, per
 *      4096-element chunk, as a delta list or a bitmap, whichever is smaller.
 *   4. Mantissa-only changes contribute just their 7 mantissa bits ([ARCv3] paragraph on
 *      encoding the asymmetry: "mantissa-only changes contribute just their mantissa bits").
 *   5. Rare changes are packed separately, each as one 16-bit block holding all changed
 *      fields (sign, exponent and mantissa XOR together).
 *   6. A checksum of the new weights is returned beside the payload ([ARCv3] API listing;
 *      "the result is checksummed against the trainer's original").
 * Decoding XORs both streams back into old ([WT]: old XOR mask = new) and verifies the
 * checksum.  Readings where the pages are silent are the library's written format spec.
 *
 * Payload layout (all integers little-endian, no padding between sections):
 *   header (64 bytes) | count table (C x {u16 M_c, u16 R_c}) | R stream (u16 per rare
 *   element) | position section (per chunk: M block then R block) | M stream (7 bits per
 *   mantissa-only element, LSB-first bit packing, pad bits zero)
 * Version 2 (a payload bound to its base version; not on the pages, which only say that a
 * joint commit binds the installed weights to the baseline of the next delta): the version-1
 * header with version 2, followed by u64 base checksum (the checksum of the weights the
 * payload applies to) and u64 flags, i.e. an 80-byte header; the sections after it are the
 * same.  Flags bit 0 (versions 2 and 3; every other bit zero) marks an overwrite payload
 * ("Two forms of update payload": changes carried as absolute overwrites; "Retry-safe
 * versioning": partial writes retried through overwrites): the R stream holds each rare
 * element's new value and the M stream each mantissa-only element's new mantissa, and the
 * decoder writes them into place instead of XORing, so applying the payload again to weights
 * it has already (partly) updated leaves the same result.  Positions and classes are those of
 * the XOR payload of the same update.
 * Version 3 (compact positions; a byte-aligned code of the position gaps standing in for the
 * entropy stage of the pages' codecs): the version-2 header with version 3, then
 *   count table (C x u32) | R stream | X stream (u16 per escaped gap, chunks in order) |
 *   position section | M stream
 * Count entry: bit 31 set -- a compact chunk, M in bits 0..8, R in bits 9..17, E (escaped
 * gaps) in bits 18..26, bits 27..30 zero; bit 31 clear -- M in bits 0..14, R in bits 15..29,
 * bit 30 zero, blocks exactly as in version 1.  A compact chunk (k = M + R <= 508) has one
 * merged list of all its changes in ascending position: k gap bytes (g_0 = p_0 + 1,
 * g_i = p_i - p_{i-1}; the byte is g when g <= 255, else 0 and g is the chunk's next X value)
 * then ceil(k/8) class bytes (bit i, LSB-first, is 1 when change i is rare; pad bits 0).  The
 * encoder makes a chunk compact when k <= 508 and k + ceil(k/8) + 2E is smaller than its
 * version-1 blocks; decoders accept either coding of a chunk.
 * Version 4 (a Golomb-Rice code of the same gaps, the second stand-in for the entropy stage):
 * the version-3 layout without the X stream.  Compact count entry: bit 31 set, M in bits
 * 0..8, R in bits 9..17, the Rice parameter K in bits 18..20 and the block's bytes B in bits
 * 21..30 (M + R between 1 and 508, B at least 1); plain entries as in version 3.  A compact
 * block is a bit stream, LSB-first from its first byte: the R indices (within the merged
 * list, ascending, 9 bits each) of the rare changes; then for each gap g_i its remainder
 * g_i mod 2^K (K bits); then for each gap its quotient g_i >> K in unary (that many 1 bits,
 * then a 0); then zero pad bits up to B = ceil(bits / 8).  The encoder takes the K in 0..7
 * giving the fewest bits (the smallest such K) and makes a chunk compact when k <= 508 and B
 * is smaller than its version-1 blocks.
 */
#include "bd_oracle.h"

#include <stdlib.h>
#include <string.h>

#define ORC_CHUNK 4096u
#define ORC_HEADER 64u      /* version 1 */
#define ORC_HEADER_V2 80u   /* version 2 and 3: + base checksum + reserved */
#define ORC_COMPACT_MAX 508u /* version 3: most changes of a compact chunk */
/* Header flags (versions 2 and 3, the u64 at byte 72): bit 0 = the streams carry new field
 * values to overwrite instead of XOR masks.  Every other bit is zero. */
#define ORC_FLAG_OVERWRITE 1u

/* Field masks of a BF16 word: sign bit 15, exponent bits 14..7, mantissa bits 6..0. */
#define ORC_SIGN_EXP_BITS 0xFF80u
#define ORC_MANT_BITS 0x007Fu

/* Class of one XOR value. */
enum { CLASS_ZERO = 0, CLASS_MANT = 1, CLASS_RARE = 2 };

static int classify(uint16_t x) {
  if (x == 0) return CLASS_ZERO;
  if ((x & ORC_SIGN_EXP_BITS) == 0) return CLASS_MANT;
  return CLASS_RARE;
}

/* ---- little-endian helpers ---------------------------------------------------------- */

static void put_u16(uint8_t* p, uint16_t v) {
  p[0] = (uint8_t)(v & 0xFF);
  p[1] = (uint8_t)(v >> 8);
}
static void put_u32(uint8_t* p, uint32_t v) {
  for (int b = 0; b < 4; b++) p[b] = (uint8_t)(v >> (8 * b));
}
static void put_u64(uint8_t* p, uint64_t v) {
  for (int b = 0; b < 8; b++) p[b] = (uint8_t)(v >> (8 * b));
}
static uint16_t get_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t get_u32(const uint8_t* p) {
  uint32_t v = 0;
  for (int b = 0; b < 4; b++) v |= (uint32_t)p[b] << (8 * b);
  return v;
}
static uint64_t get_u64(const uint8_t* p) {
  uint64_t v = 0;
  for (int b = 0; b < 8; b++) v |= (uint64_t)p[b] << (8 * b);
  return v;
}

/* ---- checksum ----------------------------------------------------------------------- */
/*
 * The pages only say the result is "checksummed".  Definition used here: view the n BF16
 * values as W = ceil(n/4) little-endian 64-bit words (word j holds elements 4j..4j+3,
 * element 4j+e in bits 16e..16e+15, zero past n).  Each word is keyed by its position and
 * mixed with the SplitMix64 output function (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014):
 *   checksum = sum over j of  mix64( word_j XOR (j+1)*GAMMA )   (mod 2^64)
 * For an all-zero tensor the terms are exactly the SplitMix64 outputs for seed 0.
 */
static const uint64_t GAMMA = 0x9E3779B97F4A7C15ull;

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

uint64_t orc_checksum(const uint16_t* w, uint64_t n) {
  uint64_t sum = 0;
  uint64_t words = (n + 3) / 4;
  for (uint64_t j = 0; j < words; j++) {
    uint64_t word = 0;
    for (uint64_t e = 0; e < 4; e++) {
      uint64_t i = 4 * j + e;
      if (i < n) word |= (uint64_t)w[i] << (16 * e);
    }
    sum += mix64(word ^ ((j + 1) * GAMMA));
  }
  return sum;
}

/* ---- position blocks ---------------------------------------------------------------- */

/* Length of chunk c of an n-element tensor. */
static uint64_t chunk_len(uint64_t n, uint64_t c) {
  uint64_t start = c * ORC_CHUNK;
  uint64_t left = n - start;
  return left < ORC_CHUNK ? left : ORC_CHUNK;
}

/* Bytes of a position block holding k positions of a chunk of length L:
 * a delta list of k u16 values when 2k < ceil(L/8), otherwise a ceil(L/8)-byte bitmap. */
static uint64_t block_bytes(uint64_t k, uint64_t L) {
  uint64_t bitmap = (L + 7) / 8;
  if (2 * k < bitmap) return 2 * k;
  return bitmap;
}

/* Writes the block for the k ascending positions pos[0..k) of a chunk of length L at dst. */
static void write_block(uint8_t* dst, const uint16_t* pos, uint64_t k, uint64_t L) {
  uint64_t bitmap = (L + 7) / 8;
  if (2 * k < bitmap) {
    for (uint64_t j = 0; j < k; j++) {
      uint16_t d = (uint16_t)(j == 0 ? pos[0] : pos[j] - pos[j - 1]);
      put_u16(dst + 2 * j, d);
    }
  } else {
    memset(dst, 0, bitmap);
    for (uint64_t j = 0; j < k; j++) dst[pos[j] / 8] |= (uint8_t)(1u << (pos[j] % 8));
  }
}

/* Reads a block with k positions of a chunk of length L from src into pos[0..k).
 * Returns 0 when the block is canonical, -1 otherwise. */
static int read_block(const uint8_t* src, uint16_t* pos, uint64_t k, uint64_t L) {
  uint64_t bitmap = (L + 7) / 8;
  if (2 * k < bitmap) {
    uint64_t p = 0;
    for (uint64_t j = 0; j < k; j++) {
      uint64_t d = get_u16(src + 2 * j);
      if (j > 0 && d == 0) return -1; /* positions must be strictly increasing */
      p = (j == 0) ? d : p + d;
      if (p >= L) return -1;
      pos[j] = (uint16_t)p;
    }
    return 0;
  }
  uint64_t found = 0;
  for (uint64_t p = 0; p < bitmap * 8; p++) {
    if ((src[p / 8] >> (p % 8)) & 1) {
      if (p >= L) return -1; /* unused tail bits must be zero */
      if (found == k) return -1;
      pos[found++] = (uint16_t)p;
    }
  }
  return found == k ? 0 : -1;
}

/* ---- encode ------------------------------------------------------------------------- */

/* bound: write the 80-byte header (version 2) with base; overwrite (version 2 only): the
 * streams carry the new field values instead of XOR masks and the header flags say so. */
static int encode_impl(const uint16_t* old, const uint16_t* neu, uint64_t n, int bound,
                       uint64_t base, int overwrite, uint8_t* out, uint64_t cap,
                       uint64_t* size_out, uint64_t* checksum_out) {
  if ((n > 0 && (old == NULL || neu == NULL)) || size_out == NULL || checksum_out == NULL)
    return ORC_ERR_ARG;
  const uint64_t hdr = bound ? ORC_HEADER_V2 : ORC_HEADER;
  uint64_t C = (n + ORC_CHUNK - 1) / ORC_CHUNK;

  /* Steps 1-2: XOR and classify; count each class per chunk. */
  uint64_t* mcount = (uint64_t*)calloc(C ? C : 1, sizeof(uint64_t));
  uint64_t* rcount = (uint64_t*)calloc(C ? C : 1, sizeof(uint64_t));
  if (!mcount || !rcount) { free(mcount); free(rcount); return ORC_ERR_ARG; }
  for (uint64_t i = 0; i < n; i++) {
    int cls = classify((uint16_t)(old[i] ^ neu[i]));
    if (cls == CLASS_MANT) mcount[i / ORC_CHUNK]++;
    if (cls == CLASS_RARE) rcount[i / ORC_CHUNK]++;
  }

  /* Section sizes. */
  uint64_t sum_m = 0, sum_r = 0, pos_bytes = 0;
  for (uint64_t c = 0; c < C; c++) {
    uint64_t L = chunk_len(n, c);
    sum_m += mcount[c];
    sum_r += rcount[c];
    pos_bytes += block_bytes(mcount[c], L) + block_bytes(rcount[c], L);
  }
  uint64_t m_bytes = (7 * sum_m + 7) / 8;
  uint64_t size = hdr + 4 * C + 2 * sum_r + pos_bytes + m_bytes;

  /* Step 6: checksum of the new weights. */
  *size_out = size;
  *checksum_out = orc_checksum(neu, n);
  if (out == NULL || cap < size) { free(mcount); free(rcount); return ORC_ERR_CAPACITY; }

  memset(out, 0, size);
  /* Header. */
  memcpy(out, "BF16DLT1", 8);
  put_u32(out + 8, bound ? 2 : 1);   /* version */
  put_u32(out + 12, ORC_CHUNK);  /* chunk_elems */
  put_u64(out + 16, n);
  put_u64(out + 24, C);
  put_u64(out + 32, sum_m);
  put_u64(out + 40, sum_r);
  put_u64(out + 48, pos_bytes);
  put_u64(out + 56, size);
  if (bound) {
    put_u64(out + 64, base);                      /* base checksum */
    put_u64(out + 72, overwrite ? ORC_FLAG_OVERWRITE : 0);   /* flags */
  }

  /* Count table. */
  for (uint64_t c = 0; c < C; c++) {
    put_u16(out + hdr + 4 * c, (uint16_t)mcount[c]);
    put_u16(out + hdr + 4 * c + 2, (uint16_t)rcount[c]);
  }

  uint64_t r_off = hdr + 4 * C;
  uint64_t p_off = r_off + 2 * sum_r;
  uint64_t m_off = p_off + pos_bytes;

  /* Step 5: the rare stream -- the full 16-bit XOR of every exponent/sign change (with
   * overwrite: the full new value). */
  for (uint64_t i = 0; i < n; i++) {
    uint16_t x = (uint16_t)(old[i] ^ neu[i]);
    if (classify(x) == CLASS_RARE) {
      put_u16(out + r_off, overwrite ? neu[i] : x);
      r_off += 2;
    }
  }

  /* Step 3: positions of the changed elements, chunk by chunk (M block, then R block). */
  uint16_t* mpos = (uint16_t*)malloc(ORC_CHUNK * sizeof(uint16_t));
  uint16_t* rpos = (uint16_t*)malloc(ORC_CHUNK * sizeof(uint16_t));
  for (uint64_t c = 0; c < C; c++) {
    uint64_t L = chunk_len(n, c);
    uint64_t km = 0, kr = 0;
    for (uint64_t p = 0; p < L; p++) {
      uint64_t i = c * ORC_CHUNK + p;
      int cls = classify((uint16_t)(old[i] ^ neu[i]));
      if (cls == CLASS_MANT) mpos[km++] = (uint16_t)p;
      if (cls == CLASS_RARE) rpos[kr++] = (uint16_t)p;
    }
    write_block(out + p_off, mpos, km, L);
    p_off += block_bytes(km, L);
    write_block(out + p_off, rpos, kr, L);
    p_off += block_bytes(kr, L);
  }
  free(mpos);
  free(rpos);

  /* Step 4: the mantissa stream -- 7 bits (x & 0x7F; with overwrite: the new mantissa) per
   * mantissa-only change, element j of the stream in bits [7j, 7j+7), stream bit b = bit
   * (b % 8) of byte (b / 8). */
  uint64_t j = 0;
  for (uint64_t i = 0; i < n; i++) {
    uint16_t x = (uint16_t)(old[i] ^ neu[i]);
    if (classify(x) != CLASS_MANT) continue;
    uint16_t v = (uint16_t)((overwrite ? neu[i] : x) & ORC_MANT_BITS);
    for (uint64_t b = 0; b < 7; b++) {
      uint64_t bit = 7 * j + b;
      if ((v >> b) & 1) out[m_off + bit / 8] |= (uint8_t)(1u << (bit % 8));
    }
    j++;
  }

  free(mcount);
  free(rcount);
  return ORC_OK;
}

int orc_encode(const uint16_t* old, const uint16_t* neu, uint64_t n, uint8_t* out,
               uint64_t cap, uint64_t* size_out, uint64_t* checksum_out) {
  return encode_impl(old, neu, n, 0, 0, 0, out, cap, size_out, checksum_out);
}

int orc_encode_versioned(const uint16_t* old, const uint16_t* neu, uint64_t n, uint64_t base,
                         uint8_t* out, uint64_t cap, uint64_t* size_out,
                         uint64_t* checksum_out) {
  return encode_impl(old, neu, n, 1, base, 0, out, cap, size_out, checksum_out);
}

int orc_encode_overwrite(const uint16_t* old, const uint16_t* neu, uint64_t n, uint64_t base,
                         uint8_t* out, uint64_t cap, uint64_t* size_out,
                         uint64_t* checksum_out) {
  return encode_impl(old, neu, n, 1, base, 1, out, cap, size_out, checksum_out);
}

/* ---- version 3: compact positions ---------------------------------------------------- */

#define ORC_COMPACT_FLAG 0x80000000u

/* Escaped gaps of a chunk's merged list (gaps above 255). */
static uint64_t chunk_escapes(const uint16_t* old, const uint16_t* neu, uint64_t c, uint64_t L) {
  int64_t prev = -1;
  uint64_t e = 0;
  for (uint64_t p = 0; p < L; p++) {
    uint64_t i = c * ORC_CHUNK + p;
    if (classify((uint16_t)(old[i] ^ neu[i])) == CLASS_ZERO) continue;
    if ((int64_t)p - prev > 255) e++;
    prev = (int64_t)p;
  }
  return e;
}

static int compact_impl(const uint16_t* old, const uint16_t* neu, uint64_t n, uint64_t base,
                        int overwrite, uint8_t* out, uint64_t cap, uint64_t* size_out,
                        uint64_t* checksum_out) {
  if ((n > 0 && (old == NULL || neu == NULL)) || size_out == NULL || checksum_out == NULL)
    return ORC_ERR_ARG;
  uint64_t C = (n + ORC_CHUNK - 1) / ORC_CHUNK;

  /* XOR and classify: per-chunk counts; the coding of each chunk (compact when smaller). */
  uint64_t* mcount = (uint64_t*)calloc(C ? C : 1, sizeof(uint64_t));
  uint64_t* rcount = (uint64_t*)calloc(C ? C : 1, sizeof(uint64_t));
  uint64_t* ecount = (uint64_t*)calloc(C ? C : 1, sizeof(uint64_t));
  uint8_t* compact = (uint8_t*)calloc(C ? C : 1, 1);
  if (!mcount || !rcount || !ecount || !compact) {
    free(mcount); free(rcount); free(ecount); free(compact);
    return ORC_ERR_ARG;
  }
  for (uint64_t i = 0; i < n; i++) {
    int cls = classify((uint16_t)(old[i] ^ neu[i]));
    if (cls == CLASS_MANT) mcount[i / ORC_CHUNK]++;
    if (cls == CLASS_RARE) rcount[i / ORC_CHUNK]++;
  }
  uint64_t sum_m = 0, sum_r = 0, sum_e = 0, pos_bytes = 0;
  for (uint64_t c = 0; c < C; c++) {
    uint64_t L = chunk_len(n, c), k = mcount[c] + rcount[c];
    uint64_t plain = block_bytes(mcount[c], L) + block_bytes(rcount[c], L);
    if (k > 0 && k <= ORC_COMPACT_MAX) {
      uint64_t e = chunk_escapes(old, neu, c, L);
      if (k + (k + 7) / 8 + 2 * e < plain) {
        compact[c] = 1;
        ecount[c] = e;
      }
    }
    sum_m += mcount[c];
    sum_r += rcount[c];
    sum_e += ecount[c];
    pos_bytes += compact[c] ? k + (k + 7) / 8 : plain;
  }
  uint64_t m_bytes = (7 * sum_m + 7) / 8;
  uint64_t size = ORC_HEADER_V2 + 4 * C + 2 * sum_r + 2 * sum_e + pos_bytes + m_bytes;
  *size_out = size;
  *checksum_out = orc_checksum(neu, n);
  if (out == NULL || cap < size) {
    free(mcount); free(rcount); free(ecount); free(compact);
    return ORC_ERR_CAPACITY;
  }

  memset(out, 0, size);
  memcpy(out, "BF16DLT1", 8);
  put_u32(out + 8, 3);
  put_u32(out + 12, ORC_CHUNK);
  put_u64(out + 16, n);
  put_u64(out + 24, C);
  put_u64(out + 32, sum_m);
  put_u64(out + 40, sum_r);
  put_u64(out + 48, pos_bytes);
  put_u64(out + 56, size);
  put_u64(out + 64, base);
  put_u64(out + 72, overwrite ? ORC_FLAG_OVERWRITE : 0);
  for (uint64_t c = 0; c < C; c++) {
    uint32_t v = compact[c] ? ORC_COMPACT_FLAG | (uint32_t)mcount[c] | ((uint32_t)rcount[c] << 9) |
                                  ((uint32_t)ecount[c] << 18)
                            : (uint32_t)mcount[c] | ((uint32_t)rcount[c] << 15);
    put_u32(out + ORC_HEADER_V2 + 4 * c, v);
  }
  uint64_t r_off = ORC_HEADER_V2 + 4 * C;
  uint64_t x_off = r_off + 2 * sum_r;
  uint64_t p_off = x_off + 2 * sum_e;
  uint64_t m_off = p_off + pos_bytes;

  /* R stream: every rare change's 16-bit XOR, in position order. */
  for (uint64_t i = 0; i < n; i++) {
    uint16_t x = (uint16_t)(old[i] ^ neu[i]);
    if (classify(x) == CLASS_RARE) { put_u16(out + r_off, overwrite ? neu[i] : x); r_off += 2; }
  }
  /* X stream and position blocks, chunk by chunk. */
  uint16_t* mpos = (uint16_t*)malloc(ORC_CHUNK * sizeof(uint16_t));
  uint16_t* rpos = (uint16_t*)malloc(ORC_CHUNK * sizeof(uint16_t));
  for (uint64_t c = 0; c < C; c++) {
    uint64_t L = chunk_len(n, c), k = mcount[c] + rcount[c];
    if (compact[c]) {
      int64_t prev = -1;
      uint64_t j = 0;
      for (uint64_t p = 0; p < L; p++) {
        uint64_t i = c * ORC_CHUNK + p;
        int cls = classify((uint16_t)(old[i] ^ neu[i]));
        if (cls == CLASS_ZERO) continue;
        uint64_t g = (uint64_t)((int64_t)p - prev);
        if (g > 255) {
          out[p_off + j] = 0;
          put_u16(out + x_off, (uint16_t)g);
          x_off += 2;
        } else {
          out[p_off + j] = (uint8_t)g;
        }
        if (cls == CLASS_RARE) out[p_off + k + j / 8] |= (uint8_t)(1u << (j % 8));
        prev = (int64_t)p;
        j++;
      }
      p_off += k + (k + 7) / 8;
    } else {
      uint64_t km = 0, kr = 0;
      for (uint64_t p = 0; p < L; p++) {
        uint64_t i = c * ORC_CHUNK + p;
        int cls = classify((uint16_t)(old[i] ^ neu[i]));
        if (cls == CLASS_MANT) mpos[km++] = (uint16_t)p;
        if (cls == CLASS_RARE) rpos[kr++] = (uint16_t)p;
      }
      write_block(out + p_off, mpos, km, L);
      p_off += block_bytes(km, L);
      write_block(out + p_off, rpos, kr, L);
      p_off += block_bytes(kr, L);
    }
  }
  free(mpos);
  free(rpos);
  /* M stream: as in version 1. */
  uint64_t j = 0;
  for (uint64_t i = 0; i < n; i++) {
    uint16_t x = (uint16_t)(old[i] ^ neu[i]);
    if (classify(x) != CLASS_MANT) continue;
    for (uint64_t b = 0; b < 7; b++) {
      uint64_t bit = 7 * j + b;
      if ((((overwrite ? neu[i] : x) & ORC_MANT_BITS) >> b) & 1)
        out[m_off + bit / 8] |= (uint8_t)(1u << (bit % 8));
    }
    j++;
  }
  free(mcount); free(rcount); free(ecount); free(compact);
  return ORC_OK;
}

int orc_encode_compact(const uint16_t* old, const uint16_t* neu, uint64_t n, uint64_t base,
                       uint8_t* out, uint64_t cap, uint64_t* size_out, uint64_t* checksum_out) {
  return compact_impl(old, neu, n, base, 0, out, cap, size_out, checksum_out);
}

int orc_encode_compact_overwrite(const uint16_t* old, const uint16_t* neu, uint64_t n,
                                 uint64_t base, uint8_t* out, uint64_t cap, uint64_t* size_out,
                                 uint64_t* checksum_out) {
  return compact_impl(old, neu, n, base, 1, out, cap, size_out, checksum_out);
}

/* ---- version 4: Rice-coded positions --------------------------------------------------- */

#define ORC_RICE_IDX_BITS 9u   /* bits of a rare change's index in its chunk's merged list */

/* Changes of chunk c (length L) in ascending position: pos[i] and rare[i] (1: rare). */
static uint64_t chunk_changes(const uint16_t* old, const uint16_t* neu, uint64_t c, uint64_t L,
                              uint16_t* pos, uint8_t* rare) {
  uint64_t k = 0;
  for (uint64_t p = 0; p < L; p++) {
    uint64_t i = c * ORC_CHUNK + p;
    int cls = classify((uint16_t)(old[i] ^ neu[i]));
    if (cls == CLASS_ZERO) continue;
    pos[k] = (uint16_t)p;
    rare[k] = cls == CLASS_RARE;
    k++;
  }
  return k;
}

/* Bits of a Rice-coded block: R rare indices, k remainders of K bits, and for each gap its
 * quotient (gap >> K) in unary, ones then a zero.  Gaps: pos[0] + 1, then pos[i] - pos[i-1]. */
static uint64_t rice_bits(const uint16_t* pos, uint64_t k, uint64_t R, unsigned K) {
  uint64_t bits = ORC_RICE_IDX_BITS * R + k * K + k;
  int64_t prev = -1;
  for (uint64_t i = 0; i < k; i++) {
    bits += (uint64_t)((int64_t)pos[i] - prev) >> K;
    prev = pos[i];
  }
  return bits;
}

/* The encoder's Rice parameter: the K in 0..7 giving the fewest bits, the smallest on a tie. */
static unsigned rice_param(const uint16_t* pos, uint64_t k, uint64_t R) {
  unsigned best = 0;
  for (unsigned K = 1; K < 8; K++)
    if (rice_bits(pos, k, R, K) < rice_bits(pos, k, R, best)) best = K;
  return best;
}

static void put_bits(uint8_t* blk, uint64_t bit, uint32_t v, unsigned nbits) {
  for (unsigned b = 0; b < nbits; b++)
    if ((v >> b) & 1) blk[(bit + b) / 8] |= (uint8_t)(1u << ((bit + b) % 8));
}
static uint32_t get_bits(const uint8_t* blk, uint64_t bit, unsigned nbits) {
  uint32_t v = 0;
  for (unsigned b = 0; b < nbits; b++) v |= (uint32_t)((blk[(bit + b) / 8] >> ((bit + b) % 8)) & 1) << b;
  return v;
}

/* Writes the block of k changes (R of them rare) with parameter K at blk (zeroed): the rare
 * indices, ascending, 9 bits each; then the remainders gap mod 2^K, K bits each; then the
 * quotients in unary. */
static void write_rice(uint8_t* blk, const uint16_t* pos, const uint8_t* rare, uint64_t k,
                       uint64_t R, unsigned K) {
  uint64_t j = 0;
  for (uint64_t i = 0; i < k; i++)
    if (rare[i]) put_bits(blk, ORC_RICE_IDX_BITS * j++, (uint32_t)i, ORC_RICE_IDX_BITS);
  uint64_t u = ORC_RICE_IDX_BITS * R + k * K;
  int64_t prev = -1;
  for (uint64_t i = 0; i < k; i++) {
    uint64_t g = (uint64_t)((int64_t)pos[i] - prev);
    put_bits(blk, ORC_RICE_IDX_BITS * R + K * i, (uint32_t)(g & ((1u << K) - 1)), K);
    for (uint64_t q = g >> K; q > 0; q--) put_bits(blk, u++, 1, 1);
    u++;   /* the zero that ends the quotient */
    prev = pos[i];
  }
}

static int rice_impl(const uint16_t* old, const uint16_t* neu, uint64_t n, uint64_t base,
                     int overwrite, uint8_t* out, uint64_t cap, uint64_t* size_out,
                     uint64_t* checksum_out) {
  if ((n > 0 && (old == NULL || neu == NULL)) || size_out == NULL || checksum_out == NULL)
    return ORC_ERR_ARG;
  uint64_t C = (n + ORC_CHUNK - 1) / ORC_CHUNK;

  /* XOR and classify per chunk; a chunk is compact when its Rice block is smaller than its
   * two version-1 blocks. */
  uint64_t* mcount = (uint64_t*)calloc(C ? C : 1, sizeof(uint64_t));
  uint64_t* rcount = (uint64_t*)calloc(C ? C : 1, sizeof(uint64_t));
  uint32_t* kparam = (uint32_t*)calloc(C ? C : 1, sizeof(uint32_t));
  uint32_t* bbytes = (uint32_t*)calloc(C ? C : 1, sizeof(uint32_t));
  uint16_t* pos = (uint16_t*)malloc(ORC_CHUNK * sizeof(uint16_t));
  uint8_t* rare = (uint8_t*)malloc(ORC_CHUNK);
  if (!mcount || !rcount || !kparam || !bbytes || !pos || !rare) {
    free(mcount); free(rcount); free(kparam); free(bbytes); free(pos); free(rare);
    return ORC_ERR_ARG;
  }
  uint64_t sum_m = 0, sum_r = 0, pos_bytes = 0;
  for (uint64_t c = 0; c < C; c++) {
    uint64_t L = chunk_len(n, c);
    uint64_t k = chunk_changes(old, neu, c, L, pos, rare);
    uint64_t R = 0;
    for (uint64_t i = 0; i < k; i++) R += rare[i];
    mcount[c] = k - R;
    rcount[c] = R;
    uint64_t plain = block_bytes(k - R, L) + block_bytes(R, L);
    if (k > 0 && k <= ORC_COMPACT_MAX) {
      unsigned K = rice_param(pos, k, R);
      uint64_t B = (rice_bits(pos, k, R, K) + 7) / 8;
      if (B < plain) {
        kparam[c] = K;
        bbytes[c] = (uint32_t)B;
      }
    }
    sum_m += mcount[c];
    sum_r += rcount[c];
    pos_bytes += bbytes[c] ? bbytes[c] : plain;
  }
  uint64_t m_bytes = (7 * sum_m + 7) / 8;
  uint64_t size = ORC_HEADER_V2 + 4 * C + 2 * sum_r + pos_bytes + m_bytes;
  *size_out = size;
  *checksum_out = orc_checksum(neu, n);
  if (out == NULL || cap < size) {
    free(mcount); free(rcount); free(kparam); free(bbytes); free(pos); free(rare);
    return ORC_ERR_CAPACITY;
  }

  memset(out, 0, size);
  memcpy(out, "BF16DLT1", 8);
  put_u32(out + 8, 4);
  put_u32(out + 12, ORC_CHUNK);
  put_u64(out + 16, n);
  put_u64(out + 24, C);
  put_u64(out + 32, sum_m);
  put_u64(out + 40, sum_r);
  put_u64(out + 48, pos_bytes);
  put_u64(out + 56, size);
  put_u64(out + 64, base);
  put_u64(out + 72, overwrite ? ORC_FLAG_OVERWRITE : 0);
  for (uint64_t c = 0; c < C; c++) {
    uint32_t v = bbytes[c] ? ORC_COMPACT_FLAG | (uint32_t)mcount[c] | ((uint32_t)rcount[c] << 9) |
                                 (kparam[c] << 18) | (bbytes[c] << 21)
                           : (uint32_t)mcount[c] | ((uint32_t)rcount[c] << 15);
    put_u32(out + ORC_HEADER_V2 + 4 * c, v);
  }
  uint64_t r_off = ORC_HEADER_V2 + 4 * C;
  uint64_t p_off = r_off + 2 * sum_r;
  uint64_t m_off = p_off + pos_bytes;

  /* R stream: every rare change's XOR (overwrite: its new value), in position order. */
  for (uint64_t i = 0; i < n; i++) {
    uint16_t x = (uint16_t)(old[i] ^ neu[i]);
    if (classify(x) == CLASS_RARE) { put_u16(out + r_off, overwrite ? neu[i] : x); r_off += 2; }
  }
  /* Position blocks, chunk by chunk. */
  uint16_t* mpos = (uint16_t*)malloc(ORC_CHUNK * sizeof(uint16_t));
  uint16_t* rpos = (uint16_t*)malloc(ORC_CHUNK * sizeof(uint16_t));
  for (uint64_t c = 0; c < C; c++) {
    uint64_t L = chunk_len(n, c);
    uint64_t k = chunk_changes(old, neu, c, L, pos, rare);
    if (bbytes[c]) {
      write_rice(out + p_off, pos, rare, k, rcount[c], kparam[c]);
      p_off += bbytes[c];
    } else {
      uint64_t km = 0, kr = 0;
      for (uint64_t i = 0; i < k; i++) {
        if (rare[i]) rpos[kr++] = pos[i];
        else mpos[km++] = pos[i];
      }
      write_block(out + p_off, mpos, km, L);
      p_off += block_bytes(km, L);
      write_block(out + p_off, rpos, kr, L);
      p_off += block_bytes(kr, L);
    }
  }
  free(mpos);
  free(rpos);
  /* M stream: as in version 1 (overwrite: the new mantissas). */
  uint64_t j = 0;
  for (uint64_t i = 0; i < n; i++) {
    uint16_t x = (uint16_t)(old[i] ^ neu[i]);
    if (classify(x) != CLASS_MANT) continue;
    put_bits(out + m_off, 7 * j, (uint32_t)((overwrite ? neu[i] : x) & ORC_MANT_BITS), 7);
    j++;
  }
  free(mcount); free(rcount); free(kparam); free(bbytes); free(pos); free(rare);
  return ORC_OK;
}

int orc_encode_rice(const uint16_t* old, const uint16_t* neu, uint64_t n, uint64_t base,
                    int overwrite, uint8_t* out, uint64_t cap, uint64_t* size_out,
                    uint64_t* checksum_out) {
  return rice_impl(old, neu, n, base, overwrite != 0, out, cap, size_out, checksum_out);
}

/* Splits a version-3 count entry; returns -1 when its unused bits are not zero. */
static int v3_entry(uint32_t v, uint64_t* km, uint64_t* kr, uint64_t* ke, int* is_compact) {
  *is_compact = (v & ORC_COMPACT_FLAG) != 0;
  if (*is_compact) {
    if (v & 0x78000000u) return -1;
    *km = v & 0x1FF;
    *kr = (v >> 9) & 0x1FF;
    *ke = (v >> 18) & 0x1FF;
    if (*km + *kr == 0 || *km + *kr > ORC_COMPACT_MAX || *ke > *km + *kr) return -1;
  } else {
    if (v & 0x40000000u) return -1;
    *km = v & 0x7FFF;
    *kr = (v >> 15) & 0x7FFF;
    *ke = 0;
  }
  return 0;
}

/* Applying one change to the element at w.  An XOR payload flips the bits its value holds
 * ("Delta update algebra": old XOR mask = new).  An overwrite payload carries the new
 * field instead ("Two forms of update payload": absolute overwrites): a mantissa-only change
 * replaces the mantissa and keeps the sign and exponent, which it did not change; a rare
 * change replaces the whole value.  Applying an overwrite twice leaves the same result. */
static void apply_mant(uint16_t* w, uint16_t v, int overwrite) {
  if (overwrite) *w = (uint16_t)((*w & ORC_SIGN_EXP_BITS) | v);
  else *w ^= v;
}
static void apply_rare(uint16_t* w, uint16_t v, int overwrite) {
  if (overwrite) *w = v;
  else *w ^= v;
}

/* The 7-bit value j of the M stream starting at m. */
static uint16_t mant_at(const uint8_t* m, uint64_t j) {
  uint16_t v = 0;
  for (uint64_t b = 0; b < 7; b++) {
    uint64_t bit = 7 * j + b;
    v |= (uint16_t)(((m[bit / 8] >> (bit % 8)) & 1) << b);
  }
  return v;
}

/* Splits a version-4 count entry: a compact entry gives M, R, the Rice parameter K and the
 * block's bytes B; a plain entry M and R as in version 3.  Returns -1 on a malformed entry. */
static int v4_entry(uint32_t v, uint64_t* km, uint64_t* kr, unsigned* K, uint64_t* B,
                    int* is_compact) {
  *is_compact = (v & ORC_COMPACT_FLAG) != 0;
  *K = 0;
  *B = 0;
  if (*is_compact) {
    *km = v & 0x1FF;
    *kr = (v >> 9) & 0x1FF;
    *K = (v >> 18) & 0x7;
    *B = (v >> 21) & 0x3FF;
    if (*km + *kr == 0 || *km + *kr > ORC_COMPACT_MAX || *B == 0) return -1;
  } else {
    if (v & 0x40000000u) return -1;
    *km = v & 0x7FFF;
    *kr = (v >> 15) & 0x7FFF;
  }
  return 0;
}

/* Reads the B-byte Rice block of a compact version-4 chunk of length L with k changes, R of
 * them rare, parameter K: the merged list's positions into pos[0..k) and classes into
 * rare[0..k).  Returns 0 when the block is the canonical coding of such a list: rare indices
 * strictly ascending and below k; every gap (quotient << K | remainder) at least 1 and every
 * position below L; the k-th unary zero inside the block; B = ceil(bits used / 8), the pad
 * bits after them zero.  Otherwise -1. */
static int read_rice(const uint8_t* blk, uint64_t B, uint64_t k, uint64_t R, unsigned K,
                     uint64_t L, uint16_t* pos, uint8_t* rare) {
  uint64_t fixed = ORC_RICE_IDX_BITS * R + k * K;
  if (fixed > 8 * B) return -1;
  memset(rare, 0, k);
  for (uint64_t j = 0; j < R; j++) {
    uint64_t idx = get_bits(blk, ORC_RICE_IDX_BITS * j, ORC_RICE_IDX_BITS);
    uint64_t prev = j == 0 ? 0 : get_bits(blk, ORC_RICE_IDX_BITS * (j - 1), ORC_RICE_IDX_BITS);
    if (idx >= k || (j > 0 && idx <= prev)) return -1;
    rare[idx] = 1;
  }
  uint64_t u = fixed, p = 0;
  for (uint64_t i = 0; i < k; i++) {
    uint64_t q = 0;
    for (;;) {
      if (u >= 8 * B) return -1;           /* the quotient runs past the block */
      uint32_t bit = get_bits(blk, u++, 1);
      if (bit == 0) break;
      q++;
    }
    uint64_t g = (q << K) | get_bits(blk, ORC_RICE_IDX_BITS * R + K * i, K);
    if (g == 0) return -1;
    p = i == 0 ? g - 1 : p + g;
    if (p >= L) return -1;
    pos[i] = (uint16_t)p;
  }
  if ((u + 7) / 8 != B) return -1;
  for (uint64_t bit = u; bit < 8 * B; bit++)
    if (get_bits(blk, bit, 1)) return -1;
  return 0;
}

/* Decodes a version-3 or version-4 payload (header fields n, C, version and flags already
 * checked, size >= 80) into out; the base is checked against required_base as in
 * decode_into.  The two versions differ in the count entry of a compact chunk, the X stream
 * (version 3 only) and the coding of a compact chunk's merged list. */
static int decode_v3_v4(const uint16_t* old, uint64_t n, const uint8_t* payload, uint64_t size,
                     uint16_t* out, const uint64_t* required_base, int overwrite,
                     uint32_t version) {
  uint64_t C = (n + ORC_CHUNK - 1) / ORC_CHUNK;
  uint64_t hdr_m = get_u64(payload + 32), hdr_r = get_u64(payload + 40);
  uint64_t hdr_pos = get_u64(payload + 48), hdr_size = get_u64(payload + 56);
  if (hdr_size != size) return ORC_ERR_FORMAT;
  if ((size - ORC_HEADER_V2) / 4 < C) return ORC_ERR_FORMAT;
  uint64_t sum_m = 0, sum_r = 0, sum_e = 0, pos_bytes = 0;
  for (uint64_t c = 0; c < C; c++) {
    uint64_t L = chunk_len(n, c), km, kr, ke = 0, B = 0;
    unsigned K;
    int cmp;
    uint32_t v = get_u32(payload + ORC_HEADER_V2 + 4 * c);
    if (version == 3 ? v3_entry(v, &km, &kr, &ke, &cmp) : v4_entry(v, &km, &kr, &K, &B, &cmp))
      return ORC_ERR_FORMAT;
    if (km + kr > L) return ORC_ERR_FORMAT;
    sum_m += km;
    sum_r += kr;
    sum_e += ke;
    if (!cmp) pos_bytes += block_bytes(km, L) + block_bytes(kr, L);
    else pos_bytes += version == 3 ? km + kr + (km + kr + 7) / 8 : B;
  }
  if (sum_m != hdr_m || sum_r != hdr_r || pos_bytes != hdr_pos) return ORC_ERR_FORMAT;
  uint64_t m_bytes = (7 * sum_m + 7) / 8;
  if (ORC_HEADER_V2 + 4 * C + 2 * sum_r + 2 * sum_e + pos_bytes + m_bytes != size)
    return ORC_ERR_FORMAT;
  if (required_base != NULL && get_u64(payload + 64) != *required_base) return ORC_ERR_BASE;

  uint64_t r_off = ORC_HEADER_V2 + 4 * C;
  uint64_t x_off = r_off + 2 * sum_r;
  uint64_t p_off = x_off + 2 * sum_e;
  uint64_t m_off = p_off + pos_bytes;
  if (n > 0) memcpy(out, old, n * sizeof(uint16_t));
  uint16_t* mpos = (uint16_t*)malloc(ORC_CHUNK * sizeof(uint16_t));
  uint16_t* rpos = (uint16_t*)malloc(ORC_CHUNK * sizeof(uint16_t));
  uint16_t* kpos = (uint16_t*)malloc(ORC_COMPACT_MAX * sizeof(uint16_t));
  uint8_t* krare = (uint8_t*)malloc(ORC_COMPACT_MAX);
  uint64_t mj = 0, rj = 0, xj = 0;
  int status = ORC_OK;
  for (uint64_t c = 0; c < C && status == ORC_OK; c++) {
    uint64_t L = chunk_len(n, c), km, kr, ke = 0, B = 0;
    unsigned K = 0;
    int cmp;
    uint32_t v = get_u32(payload + ORC_HEADER_V2 + 4 * c);
    if (version == 3) v3_entry(v, &km, &kr, &ke, &cmp);
    else v4_entry(v, &km, &kr, &K, &B, &cmp);
    const uint8_t* blk = payload + p_off;
    uint64_t nm = 0, nr = 0;
    if (cmp && version == 4) {
      /* the merged list from the Rice block, split by class */
      if (read_rice(blk, B, km + kr, kr, K, L, kpos, krare) != 0) { status = ORC_ERR_FORMAT; break; }
      for (uint64_t i = 0; i < km + kr; i++) {
        if (krare[i]) rpos[nr++] = kpos[i];
        else mpos[nm++] = kpos[i];
      }
      if (nm != km) { status = ORC_ERR_FORMAT; break; }   /* cannot differ: R indices distinct */
      p_off += B;
    } else if (cmp) {
      /* the merged list: positions from the gaps, classes from the class bits */
      uint64_t k = km + kr, p = 0, esc = 0;
      for (uint64_t i = 0; i < k && status == ORC_OK; i++) {
        uint64_t g = blk[i];
        if (g == 0) {
          if (esc == ke) { status = ORC_ERR_FORMAT; break; }
          g = get_u16(payload + x_off + 2 * (xj + esc));
          esc++;
          if (g <= 255) { status = ORC_ERR_FORMAT; break; }   /* only gaps above 255 */
        }
        p = (i == 0) ? g - 1 : p + g;
        if (p >= L) { status = ORC_ERR_FORMAT; break; }
        if ((blk[k + i / 8] >> (i % 8)) & 1) {
          if (nr == kr) { status = ORC_ERR_FORMAT; break; }
          rpos[nr++] = (uint16_t)p;
        } else {
          if (nm == km) { status = ORC_ERR_FORMAT; break; }
          mpos[nm++] = (uint16_t)p;
        }
      }
      if (status == ORC_OK && (esc != ke || nm != km || nr != kr)) status = ORC_ERR_FORMAT;
      for (uint64_t i = k; status == ORC_OK && i < 8 * ((k + 7) / 8); i++)
        if ((blk[k + i / 8] >> (i % 8)) & 1) status = ORC_ERR_FORMAT;   /* class pad bits */
      p_off += k + (k + 7) / 8;
    } else {
      /* version-1 blocks; a position may not be in both */
      if (read_block(blk, mpos, km, L) != 0) status = ORC_ERR_FORMAT;
      blk += block_bytes(km, L);
      if (status == ORC_OK && read_block(blk, rpos, kr, L) != 0) status = ORC_ERR_FORMAT;
      for (uint64_t a = 0, b = 0; status == ORC_OK && a < km && b < kr;) {
        if (mpos[a] == rpos[b]) status = ORC_ERR_FORMAT;
        else if (mpos[a] < rpos[b]) a++;
        else b++;
      }
      nm = km;
      nr = kr;
      p_off += block_bytes(km, L) + block_bytes(kr, L);
    }
    if (status != ORC_OK) break;
    for (uint64_t i = 0; i < nm; i++) {
      uint16_t v = mant_at(payload + m_off, mj + i);
      if (!overwrite && v == 0) { status = ORC_ERR_FORMAT; break; }
      apply_mant(&out[c * ORC_CHUNK + mpos[i]], v, overwrite);
    }
    for (uint64_t i = 0; status == ORC_OK && i < nr; i++) {
      uint16_t v = get_u16(payload + r_off + 2 * (rj + i));
      if (!overwrite && (v & ORC_SIGN_EXP_BITS) == 0) { status = ORC_ERR_FORMAT; break; }
      apply_rare(&out[c * ORC_CHUNK + rpos[i]], v, overwrite);
    }
    mj += km;
    rj += kr;
    xj += ke;
  }
  free(mpos);
  free(rpos);
  free(kpos);
  free(krare);
  if (status != ORC_OK) return status;
  for (uint64_t bit = 7 * sum_m; bit < 8 * m_bytes; bit++)
    if ((payload[m_off + bit / 8] >> (bit % 8)) & 1) return ORC_ERR_FORMAT;
  return ORC_OK;
}

/* ---- decode ------------------------------------------------------------------------- */

/* Applies payload[0..size) to old into out and checks every format rule; no checksum.  When
 * required_base is not NULL and the payload is version 2, its base checksum must equal
 * *required_base (checked after the header and count table, before any chunk is decoded). */
static int decode_into(const uint16_t* old, uint64_t n, const uint8_t* payload, uint64_t size,
                       uint16_t* out, const uint64_t* required_base) {
  if ((n > 0 && (old == NULL || out == NULL)) || (size > 0 && payload == NULL))
    return ORC_ERR_ARG;
  if (size < ORC_HEADER) return ORC_ERR_FORMAT;
  if (memcmp(payload, "BF16DLT1", 8) != 0) return ORC_ERR_FORMAT;
  uint32_t version = get_u32(payload + 8);
  if (version < 1 || version > 4) return ORC_ERR_FORMAT;
  const uint64_t hdr = version >= 2 ? ORC_HEADER_V2 : ORC_HEADER;
  if (size < hdr) return ORC_ERR_FORMAT;
  const uint64_t flags = version >= 2 ? get_u64(payload + 72) : 0;
  if ((flags & ~(uint64_t)ORC_FLAG_OVERWRITE) != 0) return ORC_ERR_FORMAT;
  const int overwrite = (flags & ORC_FLAG_OVERWRITE) != 0;
  if (get_u32(payload + 12) != ORC_CHUNK) return ORC_ERR_FORMAT;
  uint64_t C = (n + ORC_CHUNK - 1) / ORC_CHUNK;
  if (get_u64(payload + 16) != n) return ORC_ERR_FORMAT;
  if (get_u64(payload + 24) != C) return ORC_ERR_FORMAT;
  if (version >= 3)
    return decode_v3_v4(old, n, payload, size, out, required_base, overwrite, version);
  uint64_t hdr_m = get_u64(payload + 32), hdr_r = get_u64(payload + 40);
  uint64_t hdr_pos = get_u64(payload + 48), hdr_size = get_u64(payload + 56);
  if (hdr_size != size) return ORC_ERR_FORMAT;
  if ((size - hdr) / 4 < C) return ORC_ERR_FORMAT; /* count table must fit */

  /* Count table: per-chunk counts, their totals and the closed-form size. */
  uint64_t sum_m = 0, sum_r = 0, pos_bytes = 0;
  for (uint64_t c = 0; c < C; c++) {
    uint64_t L = chunk_len(n, c);
    uint64_t km = get_u16(payload + hdr + 4 * c);
    uint64_t kr = get_u16(payload + hdr + 4 * c + 2);
    if (km + kr > L) return ORC_ERR_FORMAT;
    sum_m += km;
    sum_r += kr;
    pos_bytes += block_bytes(km, L) + block_bytes(kr, L);
  }
  if (sum_m != hdr_m || sum_r != hdr_r || pos_bytes != hdr_pos) return ORC_ERR_FORMAT;
  uint64_t m_bytes = (7 * sum_m + 7) / 8;
  if (hdr + 4 * C + 2 * sum_r + pos_bytes + m_bytes != size) return ORC_ERR_FORMAT;

  /* A payload bound to a base version is applied to that version only. */
  if (version == 2 && required_base != NULL && get_u64(payload + 64) != *required_base)
    return ORC_ERR_BASE;

  uint64_t r_off = hdr + 4 * C;
  uint64_t p_off = r_off + 2 * sum_r;
  uint64_t m_off = p_off + pos_bytes;

  if (n > 0) memcpy(out, old, n * sizeof(uint16_t));
  uint16_t* mpos = (uint16_t*)malloc(ORC_CHUNK * sizeof(uint16_t));
  uint16_t* rpos = (uint16_t*)malloc(ORC_CHUNK * sizeof(uint16_t));
  uint8_t* seen = (uint8_t*)malloc(ORC_CHUNK);
  int status = ORC_OK;
  uint64_t mj = 0, rj = 0;
  for (uint64_t c = 0; c < C && status == ORC_OK; c++) {
    uint64_t L = chunk_len(n, c);
    uint64_t km = get_u16(payload + hdr + 4 * c);
    uint64_t kr = get_u16(payload + hdr + 4 * c + 2);
    if (read_block(payload + p_off, mpos, km, L) != 0) { status = ORC_ERR_FORMAT; break; }
    p_off += block_bytes(km, L);
    if (read_block(payload + p_off, rpos, kr, L) != 0) { status = ORC_ERR_FORMAT; break; }
    p_off += block_bytes(kr, L);

    /* A position belongs to at most one class. */
    memset(seen, 0, ORC_CHUNK);
    for (uint64_t j = 0; j < km; j++) seen[mpos[j]] = 1;
    for (uint64_t j = 0; j < kr; j++) {
      if (seen[rpos[j]]) { status = ORC_ERR_FORMAT; break; }
    }
    if (status != ORC_OK) break;

    /* Mantissa-only changes: XOR the next 7-bit value into the mantissa (overwrite: the
     * value replaces the mantissa). */
    for (uint64_t j = 0; j < km; j++, mj++) {
      uint16_t v = 0;
      for (uint64_t b = 0; b < 7; b++) {
        uint64_t bit = 7 * mj + b;
        v |= (uint16_t)(((payload[m_off + bit / 8] >> (bit % 8)) & 1) << b);
      }
      if (!overwrite && v == 0) { status = ORC_ERR_FORMAT; break; }
      apply_mant(&out[c * ORC_CHUNK + mpos[j]], v, overwrite);
    }
    if (status != ORC_OK) break;

    /* Rare changes: XOR the next full 16-bit block (overwrite: the block replaces the
     * value). */
    for (uint64_t j = 0; j < kr; j++, rj++) {
      uint16_t v = get_u16(payload + r_off + 2 * rj);
      if (!overwrite && (v & ORC_SIGN_EXP_BITS) == 0) { status = ORC_ERR_FORMAT; break; }
      apply_rare(&out[c * ORC_CHUNK + rpos[j]], v, overwrite);
    }
  }
  free(mpos);
  free(rpos);
  free(seen);
  if (status != ORC_OK) return status;

  /* Pad bits after the last mantissa value must be zero. */
  for (uint64_t bit = 7 * sum_m; bit < 8 * m_bytes; bit++) {
    if ((payload[m_off + bit / 8] >> (bit % 8)) & 1) return ORC_ERR_FORMAT;
  }
  return ORC_OK;
}

int orc_decode(const uint16_t* old, uint64_t n, const uint8_t* payload, uint64_t size,
               uint64_t expected, uint16_t* out) {
  int status = decode_into(old, n, payload, size, out, NULL);
  if (status != ORC_OK) return status;
  if (orc_checksum(out, n) != expected) return ORC_ERR_CHECKSUM;
  return ORC_OK;
}

/* ---- incremental verification -------------------------------------------------------- */

/* Word j of w (elements 4j..4j+3, zero past n), as in the checksum definition. */
static uint64_t word_of(const uint16_t* w, uint64_t n, uint64_t j) {
  uint64_t word = 0;
  for (uint64_t e = 0; e < 4; e++) {
    uint64_t i = 4 * j + e;
    if (i < n) word |= (uint64_t)w[i] << (16 * e);
  }
  return word;
}

int orc_decode_incremental(const uint16_t* old, uint64_t n, const uint8_t* payload,
                           uint64_t size, uint64_t ck_old, uint64_t expected, uint16_t* out,
                           uint64_t* ck_out) {
  int status = decode_into(old, n, payload, size, out, &ck_old);
  if (status != ORC_OK) return status;
  /* ck_old plus, for every word the payload changed, its new term minus its old term */
  uint64_t ck = ck_old;
  uint64_t words = (n + 3) / 4;
  for (uint64_t j = 0; j < words; j++) {
    uint64_t wo = word_of(old, n, j), wn = word_of(out, n, j);
    if (wo != wn) ck += mix64(wn ^ ((j + 1) * GAMMA)) - mix64(wo ^ ((j + 1) * GAMMA));
  }
  if (ck_out) *ck_out = ck;
  return ck == expected ? ORC_OK : ORC_ERR_CHECKSUM;
}
