// bd_internal.cuh -- device-side definitions shared by the kernels of libbf16delta.
//
// Everything here follows the BF16DLT1 format (versions 1 to 4) described in include/bf16delta.h.
// The field split comes from "Every byte counts: ARCv3 and the case for cross-region RL"
// (figure "How ARCv3 encodes a block of weights"); the XOR algebra from "GPU-accelerated
// Weight Teleportation", section "Delta update algebra".
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "bf16delta.h"

namespace bd {

// ---------------------------------------------------------------------------- format
constexpr uint32_t kChunk = 4096;          // elements per chunk
constexpr uint32_t kChunkBitmap = 512;     // bitmap bytes of a full chunk
constexpr uint32_t kHeader = 64;           // header bytes, version 1
constexpr uint32_t kHeaderV2 = 80;         // version 2: + base checksum + reserved u64

// Count table of a tensor's payload: it ends where the R stream starts (r_start, known once
// the scan has run), so its place does not depend on the header version.
__host__ __device__ __forceinline__ uint64_t count_table_offset(uint64_t r_start,
                                                                uint64_t nchunks) {
  return r_start - 4 * nchunks;
}
constexpr uint16_t kSignExp = 0xFF80;      // sign + exponent field of a BF16 word
constexpr uint16_t kMant = 0x007F;         // mantissa field
constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

// Bytes of a position block holding k positions of a chunk whose bitmap has B bytes:
// a delta list (2k bytes) when 2k < B, otherwise the B-byte bitmap.
__host__ __device__ __forceinline__ uint32_t block_bytes(uint32_t k, uint32_t B) {
  return (2 * k < B) ? 2 * k : B;
}

// Version 3: compact position blocks.  A compact block holds the chunk's k = M + R changes as
// one ascending list -- k gap bytes (first gap = position + 1; a gap above 255 is written as a
// zero byte and its u16 value goes to the X stream) then ceil(k/8) class bytes (bit i set:
// change i is rare).  A count-table entry is a u32: compact (bit 31) with M in bits 0..8, R in
// 9..17 and E (escaped gaps) in 18..26, or plain (bit 31 clear) with M in bits 0..14 and R in
// 15..29 and version-1 blocks.  Positions of a chunk are below 4096 and every escaped gap is
// above 255, so a well-formed chunk has E <= 16.
constexpr uint32_t kCompactMax = 508;          // most changes of a compact chunk
constexpr uint32_t kCompactFlag = 0x80000000u;
__host__ __device__ __forceinline__ uint32_t compact_bytes(uint32_t k) { return k + (k + 7) / 8; }

// The encoder's choice: compact when the chunk has changes, at most kCompactMax of them, and
// the compact block plus its X-stream values is smaller than the two version-1 blocks.
__host__ __device__ __forceinline__ bool choose_compact(uint32_t M, uint32_t R, uint32_t E,
                                                        uint32_t B) {
  const uint32_t k = M + R;
  return k > 0 && k <= kCompactMax &&
         compact_bytes(k) + 2 * E < block_bytes(M, B) + block_bytes(R, B);
}

// Version 4: compact blocks coded with a Golomb-Rice code instead (no X stream).  A compact
// entry holds M in bits 0..8, R in 9..17, the Rice parameter K in 18..20 and the block's bytes
// in 21..30 (M + R in 1..508, at least one byte).  The block is a bit stream read LSB-first
// from its first byte: the merged-list indices of the R rare changes (9 bits each, strictly
// ascending, below M + R), the K-bit remainders g mod 2^K of the gaps, then the quotients
// g >> K in unary (ones closed by a zero), then zero pad bits up to the block's last byte.
constexpr uint32_t kRiceIdxBits = 9;

// One count-table entry, decoded for the payload's version.
struct ChunkCount {
  uint32_t M, R, E;   // mantissa-only and rare changes, escaped gaps (version-3 compact only)
  uint32_t K, nb;     // version-4 compact only: Rice parameter, block bytes
  bool compact;
  bool rice;          // a compact chunk of version 4
  bool bad;           // unused bits set, or a compact entry out of range
};
__host__ __device__ __forceinline__ ChunkCount parse_count(uint32_t v, uint32_t version) {
  ChunkCount c{0, 0, 0, 0, 0, false, false, false};
  if (version < 3) {
    c.M = v & 0xFFFFu;
    c.R = v >> 16;
  } else if ((v & kCompactFlag) && version == 4) {
    c.compact = true;
    c.rice = true;
    c.M = v & 0x1FFu;
    c.R = (v >> 9) & 0x1FFu;
    c.K = (v >> 18) & 0x7u;
    c.nb = (v >> 21) & 0x3FFu;
    c.bad = c.M + c.R == 0 || c.M + c.R > kCompactMax || c.nb == 0;
  } else if (v & kCompactFlag) {
    c.compact = true;
    c.M = v & 0x1FFu;
    c.R = (v >> 9) & 0x1FFu;
    c.E = (v >> 18) & 0x1FFu;
    c.bad = (v & 0x78000000u) != 0 || c.M + c.R == 0 || c.M + c.R > kCompactMax ||
            c.E > c.M + c.R;
  } else {
    c.M = v & 0x7FFFu;
    c.R = (v >> 15) & 0x7FFFu;
    c.bad = (v & 0x40000000u) != 0;
  }
  return c;
}
// Position-section bytes of a chunk whose bitmap has B bytes.
__host__ __device__ __forceinline__ uint32_t chunk_pos_bytes(const ChunkCount& c, uint32_t B) {
  if (c.rice) return c.nb;
  return c.compact ? compact_bytes(c.M + c.R) : block_bytes(c.M, B) + block_bytes(c.R, B);
}
// The count-table entry written by compress.
__host__ __device__ __forceinline__ uint32_t count_entry(uint32_t version, uint32_t M,
                                                         uint32_t R, uint32_t E, bool compact) {
  if (version < 3) return M | (R << 16);
  if (compact) return kCompactFlag | M | (R << 9) | (E << 18);
  return M | (R << 15);
}

// Header flags (the u64 at byte 72 of a header of version 2 or later).  kFlagOverwrite: the streams
// carry new field values (the whole value of a rare change, the mantissa of a mantissa-only
// change) that overwrite the weights instead of XOR masks; every other bit is zero.
constexpr uint32_t kFlagOverwrite = 1;

// Entries of the general layout -- compress slots of overwrite payloads, decoded changes in the
// general apply builds: bit 31 set for a rare change, the chunk-local position in bits 16..27,
// the value to emit or apply in bits 0..15.  XOR slots use pos << 16 | x (the class follows
// from x); ent_pos reads the position of either.
constexpr uint32_t kEntRare = 0x80000000u;
__host__ __device__ __forceinline__ uint32_t ent_pos(uint32_t e) { return (e >> 16) & 0xFFFu; }

// Compress workspace word of a chunk's counts: M in bits 0..12, R in 13..25, E (gaps above 255
// in the merged position list, counted only for version 3) in 26..30, bit 31 clear.  Version 4
// writes a chunk of 1..508 changes whose Rice block fits in 1023 bytes as the compact count
// entry it would have (bit 31 set, M, R, K, block bytes); the scan keeps it compact when the
// block is smaller than the version-1 blocks.  The wcount_* readers take the first layout
// only; the v4count_* readers take both.
__host__ __device__ __forceinline__ uint32_t wcount(uint32_t M, uint32_t R, uint32_t E) {
  return M | (R << 13) | (E << 26);
}
__host__ __device__ __forceinline__ uint32_t wcount_m(uint32_t v) { return v & 0x1FFFu; }
__host__ __device__ __forceinline__ uint32_t wcount_r(uint32_t v) { return (v >> 13) & 0x1FFFu; }
__host__ __device__ __forceinline__ uint32_t wcount_e(uint32_t v) { return (v >> 26) & 0x1Fu; }
__host__ __device__ __forceinline__ uint32_t v4count_m(uint32_t v) {
  return (v & kCompactFlag) ? v & 0x1FFu : v & 0x1FFFu;
}
__host__ __device__ __forceinline__ uint32_t v4count_r(uint32_t v) {
  return (v & kCompactFlag) ? (v >> 9) & 0x1FFu : (v >> 13) & 0x1FFFu;
}
// Version 4: whether the chunk (bitmap bytes B) is coded compactly.
__host__ __device__ __forceinline__ bool rice_compact(uint32_t v, uint32_t B) {
  if ((v & kCompactFlag) == 0) return false;
  const uint32_t M = v & 0x1FFu, R = (v >> 9) & 0x1FFu;
  return ((v >> 21) & 0x3FFu) < block_bytes(M, B) + block_bytes(R, B);
}

// How compress lays out a chunk of length L in a payload of `version`, from the chunk's count
// word w in the compress workspace: its counts, whether its positions take a compact block and
// the X-stream values E that block needs (version 3); its position bytes are chunk_pos_bytes.
// The count scan and the fused compress take the same decisions through this.
__host__ __device__ __forceinline__ ChunkCount chunk_layout(uint32_t w, uint32_t L,
                                                            uint32_t version) {
  const uint32_t B = (L + 7) >> 3;
  ChunkCount cc{};
  if (version == 4) {
    cc.M = v4count_m(w);
    cc.R = v4count_r(w);
    cc.compact = cc.rice = rice_compact(w, B);
    cc.nb = (w >> 21) & 0x3FFu;
  } else {
    cc.M = wcount_m(w);
    cc.R = wcount_r(w);
    cc.compact = version == 3 && choose_compact(cc.M, cc.R, wcount_e(w), B);
    cc.E = cc.compact ? wcount_e(w) : 0;
  }
  return cc;
}

// Sums over a chunk's gaps of g >> K for K = 1..7, packed in two words: a holds the sums for
// K = 1, 2 and 4 in fields of 12, 11 and 9 bits at bits 0, 12 and 23; b those for K = 3, 5, 6
// and 7 in fields of 10, 8, 7 and 6 bits at bits 0, 10, 18 and 25.  The gaps of a chunk add
// up to its last position + 1 <= 4096, so the sum for K is at most 4096 >> K and no field
// carries into the next, in a lane's partial sums or in the warp's total.
struct RiceSums {
  uint32_t a, b;
};
__device__ __forceinline__ void rice_add(RiceSums& s, uint32_t g) {
  s.a += (g >> 1) | ((g >> 2) << 12) | ((g >> 4) << 23);
  s.b += (g >> 3) | ((g >> 5) << 10) | ((g >> 6) << 18) | ((g >> 7) << 25);
}
__device__ __forceinline__ uint32_t rice_sum(const RiceSums& s, uint32_t K) {
  switch (K) {
    case 1: return s.a & 0xFFFu;
    case 2: return (s.a >> 12) & 0x7FFu;
    case 3: return s.b & 0x3FFu;
    case 4: return s.a >> 23;
    case 5: return (s.b >> 10) & 0xFFu;
    case 6: return (s.b >> 18) & 0x7Fu;
    default: return s.b >> 25;
  }
}
// The compress workspace word of a version-4 chunk with M + R changes: sum0 = the sum of the
// gaps (last position + 1), s = their sums for K = 1..7.  K takes the fewest bits
// (9R + K(M+R) + (M+R) + sum of g >> K), the smallest K on a tie.
__device__ __forceinline__ uint32_t rice_word(uint32_t M, uint32_t R, uint32_t sum0,
                                              const RiceSums& s) {
  const uint32_t k = M + R;
  if (k == 0 || k > kCompactMax) return wcount(M, R, 0);
  uint32_t bestK = 0, best = k + sum0;
#pragma unroll
  for (uint32_t K = 1; K < 8; K++) {
    const uint32_t bits = K * k + k + rice_sum(s, K);
    if (bits < best) { best = bits; bestK = K; }
  }
  const uint32_t nb = (9 * R + best + 7) / 8;
  if (nb > 1023) return wcount(M, R, 0);
  return kCompactFlag | M | (R << 9) | (bestK << 18) | (nb << 21);
}

// SplitMix64 output function (Steele, Lea & Flood 2014) applied to a position-keyed word.
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Checksum terms of the 8 BF16 values in v, whose first element is element 8*q of the
// tensor (q = group index) -- words 2q and 2q+1; `words` is the number of words of the
// tensor (ceil(n/4)), so a group straddling the end contributes only its real words.
__device__ __forceinline__ uint64_t group_hash(uint4 v, uint64_t q, uint64_t words) {
  uint64_t j0 = 2 * q;
  uint64_t w0 = (uint64_t)v.x | ((uint64_t)v.y << 32);
  uint64_t w1 = (uint64_t)v.z | ((uint64_t)v.w << 32);
  uint64_t k0 = (j0 + 1) * kGamma;
  uint64_t h = 0;
  if (j0 < words) h += mix64(w0 ^ k0);
  if (j0 + 1 < words) h += mix64(w1 ^ (k0 + kGamma));
  return h;
}

// ---------------------------------------------------------------------------- byte permutes
// The dense kernels move a group's 7-bit mantissa values between their packed stream order and
// their element positions with byte permutes driven by small tables indexed by the group's
// 8-bit class mask, instead of a loop over the set bits.

// PTX prmt in its default mode: byte n of the result is byte (s >> 4n) & 7 of the pair b:a;
// when bit 3 of that selector nibble is set, the selected byte's top bit is replicated instead
// (0x00 for a byte below 0x80, as every 7-bit value byte is).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
  return d;
}
// The four 7-bit fields at bits 0..27 of v spread to bytes 0..3, and back.
__device__ __forceinline__ uint32_t unpack7x4(uint32_t v) {
  return (v & 0x7Fu) | ((v << 1) & 0x7F00u) | ((v << 2) & 0x7F0000u) | ((v << 3) & 0x7F000000u);
}
__device__ __forceinline__ uint32_t pack7x4(uint32_t v) {
  return (v & 0x7Fu) | ((v >> 1) & 0x3F80u) | ((v >> 2) & 0x1FC000u) | ((v >> 3) & 0xFE00000u);
}
// Expand selectors of an 8-element group with class mask m: for word w (elements 2w, 2w+1),
// the selector that takes, from the bytes of the group's values in stream order, the value
// of element 2w into byte 0 and that of element 2w+1 into byte 2 (their ranks among the set
// bits of m), and 0x00 into the other bytes and for elements not in m.
__host__ __device__ __forceinline__ uint32_t expand_sel(uint32_t m, uint32_t w) {
  uint32_t sel = 0x8080u;
  for (uint32_t h = 0; h < 2; h++) {
    const uint32_t e = 2 * w + h;
    uint32_t nib = 8;
    if ((m >> e) & 1u) {
      nib = 0;
      for (uint32_t i = 0; i < e; i++) nib += (m >> i) & 1u;
    }
    sel |= nib << (8 * h);
  }
  return sel;
}
// Compress selectors of an 8-element group with class mask m: for half h, the selector that
// puts into byte k of the result (k = 0..3) the byte of the group's (4h + k)-th element in m,
// and 0x00 past the last one.
__host__ __device__ __forceinline__ uint32_t compress_sel(uint32_t m, uint32_t h) {
  uint32_t sel = 0, k = 0;
  for (uint32_t e = 0; e < 8; e++) {
    if ((m >> e) & 1u) {
      if (k >= 4 * h && k < 4 * h + 4) sel |= e << (4 * (k - 4 * h));
      k++;
    }
  }
  for (; k < 4 * h + 4; k++)
    if (k >= 4 * h) sel |= 8u << (4 * (k - 4 * h));
  return sel;
}

// Per-element class masks of the 8 XOR values in x (bit e <-> element e of the group).
__device__ __forceinline__ void classify8(uint4 x, uint32_t& mmask, uint32_t& rmask) {
  mmask = 0;
  rmask = 0;
  if ((x.x | x.y | x.z | x.w) == 0) return;
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; i++) {
    uint32_t lo = w[i] & 0xFFFFu, hi = w[i] >> 16;
    if (lo) { if (lo & kSignExp) rmask |= 1u << (2 * i); else mmask |= 1u << (2 * i); }
    if (hi) { if (hi & kSignExp) rmask |= 2u << (2 * i); else mmask |= 2u << (2 * i); }
  }
}

__device__ __forceinline__ uint32_t elem_of(uint4 v, int e) {
  uint32_t w = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
  return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// Loads 8 BF16 values starting at element e of p (16-byte aligned when e % 8 == 0);
// elements at or past n read as zero.
__device__ __forceinline__ uint4 load8(const uint16_t* __restrict__ p, uint64_t e, uint64_t n) {
  if (e + 8 <= n) return __ldg(reinterpret_cast<const uint4*>(p + e));
  uint32_t w[4] = {0, 0, 0, 0};
  for (int i = 0; i < 8; i++)
    if (e + i < n) w[i >> 1] |= (uint32_t)p[e + i] << (16 * (i & 1));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Little-endian u16 at a possibly odd address (position blocks after an odd-length bitmap).
__device__ __forceinline__ void store_u16(uint8_t* p, uint16_t v) {
  if ((reinterpret_cast<uintptr_t>(p) & 1) == 0) {
    *reinterpret_cast<uint16_t*>(p) = v;
  } else {
    p[0] = (uint8_t)(v & 0xFF);
    p[1] = (uint8_t)(v >> 8);
  }
}
__device__ __forceinline__ uint32_t load_u16(const uint8_t* p) {
  if ((reinterpret_cast<uintptr_t>(p) & 1) == 0) return *reinterpret_cast<const uint16_t*>(p);
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8);
}

// Streaming variant (data read once): bypasses L1.
__device__ __forceinline__ uint4 load8_stream(const uint16_t* __restrict__ p, uint64_t e,
                                              uint64_t n) {
  if (e + 8 <= n) return __ldcs(reinterpret_cast<const uint4*>(p + e));
  return load8(p, e, n);
}

// Asks L2 to fetch the 8 KiB at p (one full 4096-element chunk of BF16 values), one 128-byte
// line per lane and half, so that the loads of the chunk that follow find it in L2 while the
// warp is still busy with the chunk's other work.  A hint only: nothing waits for it.
__device__ __forceinline__ void prefetch_chunk_l2(const uint16_t* p) {
  const char* c = reinterpret_cast<const char*>(p);
  const int lane = threadIdx.x & 31;
  asm volatile("prefetch.global.L2 [%0];" ::"l"(c + 128 * lane));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(c + 128 * (lane + 32)));
}

// ---------------------------------------------------------------------------- jobs

// One tensor of a compress call, as the kernels see it (written into the workspace).
struct CJob {
  const uint16_t* old;
  const uint16_t* neu;
  uint8_t* payload;
  uint64_t n;
  uint64_t cap;
  uint64_t* d_size;
  uint64_t* d_checksum;
  int32_t* d_status;
  uint64_t chunk_base;  // global index of this tensor's chunk 0
  uint64_t nchunks;     // C = ceil(n / 4096)
  uint64_t tile_base;   // global index of this tensor's first scan tile
  const uint64_t* d_base;   // versions 2 to 4: the base checksum to bind to (NULL: version 1)
  uint32_t version;         // payload version written: 1, 2 or 3 (compact position blocks)
  uint32_t flags;           // header flags written (versions 2 to 4): kFlagOverwrite
  uint64_t pad[3];
};
static_assert(sizeof(CJob) == 128, "CJob layout");

// One tensor of a decompress call.
struct DJob {
  const uint16_t* old;
  uint16_t* out;
  const uint8_t* payload;
  uint64_t n;
  uint64_t size;
  const uint64_t* d_expected;
  int32_t* d_status;
  uint64_t chunk_base;
  uint64_t nchunks;
  uint64_t tile_base;
  const uint64_t* d_ck_old;   // incremental verification: checksum of out before the call
  uint64_t* d_ck_out;         // incremental verification (optional): the computed checksum
  uint64_t pad[4];
};
static_assert(sizeof(DJob) == 128, "DJob layout");

// Per-tensor results of the scan phase (workspace).
struct JobInfo {
  uint64_t sum_m, sum_r, sum_p, sum_e;   // totals
  uint64_t r_start, x_start, p_start, m_start, total;   // section offsets, payload size
  int32_t status;      // set by the scan phase; constant while later kernels run
  int32_t chunk_err;   // set by the apply kernel when a chunk is malformed
  uint32_t version;    // payload version (set by the scan phase)
  uint32_t flags;      // header flags (versions 2 to 4; set by the scan phase)
  uint64_t pad;
};
static_assert(sizeof(JobInfo) == 96, "JobInfo layout");

// Checksum accumulators per tensor: kCkSlots u64 spaced one 64-byte line apart so that
// atomics from different warps spread over L2.
constexpr int kCkSlots = 8;
constexpr int kCkStride = 8;  // u64 per slot
constexpr int kCkBytes = kCkSlots * kCkStride * 8;

constexpr uint64_t kMagic = 0x31544C4436314642ull;  // "BF16DLT1" little-endian
__host__ __device__ __forceinline__ uint64_t header_bytes(uint32_t version) {
  return version >= 2 ? kHeaderV2 : kHeader;
}

// The end of a compress for tensor j, one thread, once its totals are in I (sum_p, sum_m,
// sum_r, sum_e) and its checksum terms in its accumulators: section offsets, size and status
// (capacity), the checksum, the header (only when the payload fits), the per-tensor outputs,
// info[j] and the call's largest status.
__device__ __forceinline__ void finish_compress_job(const CJob& J, uint32_t j, JobInfo& I,
                                                    const uint8_t* ck_base, JobInfo* info,
                                                    int32_t* status_all) {
  I.version = J.version;
  I.flags = J.flags;
  I.r_start = header_bytes(J.version) + 4 * J.nchunks;
  I.x_start = I.r_start + 2 * I.sum_r;
  I.p_start = I.x_start + 2 * I.sum_e;
  I.m_start = I.p_start + I.sum_p;
  I.total = I.m_start + (7 * I.sum_m + 7) / 8;
  I.status = I.total > J.cap ? BD_ERR_CAPACITY : BD_OK;
  const uint64_t* ck = reinterpret_cast<const uint64_t*>(ck_base + (uint64_t)j * kCkBytes);
  uint64_t sum = 0;
  for (int s = 0; s < kCkSlots; s++) sum += ck[s * kCkStride];
  *J.d_size = I.total;
  *J.d_checksum = sum;
  if (I.status == BD_OK) {
    uint64_t* h = reinterpret_cast<uint64_t*>(J.payload);
    h[0] = kMagic;
    h[1] = (uint64_t)J.version | ((uint64_t)kChunk << 32);
    h[2] = J.n;
    h[3] = J.nchunks;
    h[4] = I.sum_m;
    h[5] = I.sum_r;
    h[6] = I.sum_p;
    h[7] = I.total;
    if (J.version >= 2) {   // the base this payload applies to, and the flags
      h[8] = *J.d_base;
      h[9] = J.flags;
    }
  }
  if (J.d_status) *J.d_status = I.status;
  info[j] = I;
  if (status_all) atomicMax(reinterpret_cast<int*>(status_all), I.status);
}

// Scan tiles: chunks per tile of the count scan.
constexpr uint32_t kTileChunks = 1024;

// Fused compress (every payload kind): batches of up to `bchunks` consecutive
// chunks of one tensor (chosen per call, at most kMaxBatchChunks; an empty tensor has one
// empty batch, so that its header is written), and control words in the zeroed state: [0] the
// next encode batch to hand out, [1] the next emit batch, [kCtlAbort] set when a wait gave up
// (emit_dense then fails every tensor of the call), then per tensor j [kCtlTensors + 2j] its
// chunks encoded so far and [kCtlTensors + 2j + 1] its flag "scanned, emit may start".
constexpr uint32_t kMaxBatchChunks = 32;
// The fused compress serves calls whose tensors have at most this many batches each: the warp
// finishing a tensor scans its batch totals alone, so a tensor of many small batches (a single
// large tensor, whose batches are kept small for parallelism) would hold every warp waiting on
// that one scan; such calls take the separate kernels.
constexpr uint64_t kMaxFusedBatches = 4096;
constexpr uint32_t kCtlAbort = 2;
constexpr uint32_t kCtlTensors = 4;
__host__ __device__ __forceinline__ uint64_t tensor_batches(uint64_t nchunks, uint32_t bchunks) {
  return nchunks ? (nchunks + bchunks - 1) / bchunks : 1;
}

struct TileSum {   // totals of one scan tile (or their exclusive prefix)
  uint64_t p, m, r, e;   // position bytes, M, R, escaped gaps (X-stream values)
};

// Per-chunk slot (workspace).  Entries are pos << 16 | x.
//   u32 info   bits 0..11 mantissa-only count M, bits 12..23 rare count R, bit 30 malformed
//              chunk, bit 31 overflow (more changes than kSlotEntries: entries incomplete)
//   u32 aux    compress: first mantissa-only XOR value of the chunk (bits 0..6), bit 7 set
//              when the chunk has one (valid even on overflow)
//   u32 pad[2]
//   u32 entry[kSlotEntries]
// Compress (encode_slots -> emit): one list of all changes in ascending position at [0, M+R).
// Decompress (decode -> apply_stream): mantissa-only entries at [0, M), then rare entries at
// [M, M+R), each class in ascending position.
constexpr uint32_t kSlotBytes = 1024;
constexpr uint32_t kSlotHeader = 16;
constexpr uint32_t kSlotEntries = (kSlotBytes - kSlotHeader) / 4;
constexpr uint32_t kSlotOverflow = 0x80000000u;
constexpr uint32_t kSlotBad = 0x40000000u;
constexpr uint32_t kAuxHasM = 0x80u;
__host__ __device__ __forceinline__ uint32_t slot_info(uint32_t M, uint32_t R) {
  return (M & 0xFFFu) | ((R & 0xFFFu) << 12);
}

// Branch-free field flags of the two BF16 values in a 32-bit word: bit 15 (low value) and
// bit 31 (high value) are set when the value is nonzero (nz) / has a sign or exponent bit set
// (rare).  The add carries a nonzero masked field into bit 15 without crossing into bit 16.
__device__ __forceinline__ uint32_t nz_flags(uint32_t w) {
  return (((w & 0x7FFF7FFFu) + 0x7FFF7FFFu) | w) & 0x80008000u;
}
__device__ __forceinline__ uint32_t rare_flags(uint32_t w) {
  return (((w & 0x7F807F80u) + 0x7F807F80u) | w) & 0x80008000u;
}
// 8-bit element-order mask (bit e <-> element e) from the flags of the 4 words of a group.
__device__ __forceinline__ uint32_t flags_to_mask8(uint32_t f0, uint32_t f1, uint32_t f2,
                                                   uint32_t f3) {
  const uint32_t t = (f0 >> 15) | (f1 >> 13) | (f2 >> 11) | (f3 >> 9);  // even at 0,2,4,6; odd at 16..22
  return (t | (t >> 15)) & 0xFFu;
}

// Workspace layout of one call (byte offsets from the workspace base, 256-aligned).
struct WsLayout {
  uint64_t state;        // memset to zero at the start of a call: ck slots, job info
  uint64_t state_bytes;
  uint64_t ck;           // k * kCkBytes
  uint64_t info;         // k * JobInfo
  uint64_t jobs;         // k * CJob / DJob
  uint64_t chunk_start;  // (k+1) u64: global chunk index where job j starts
  uint64_t tile_start;   // (k+1) u64
  uint64_t counts;       // Ctot u32 (compress only)
  uint64_t slots;        // Ctot * kSlotBytes
  uint64_t loc;          // Ctot uint4: chunk exclusive prefix inside its tile (p, m, r, e)
  uint64_t tile_tot;     // Utot TileSum
  uint64_t tile_pre;     // Utot TileSum
  uint64_t overflow;     // decompress: u32 words in the zeroed state -- the count of listed
                         // chunks, then kFlagV3Word ...
  uint64_t ovf_list;     // ... and Ctot u32 chunk indices handled by the block-level apply
  uint64_t ovf_job;      // Ctot u32: the tensor of each listed chunk (not in the no-workspace
                         // layout, whose one tensor needs none)
  uint64_t fused_ctl;    // compress: fused-compress control words (zeroed state)
  uint64_t batch_start;  // compress: (k+1) u64, global index of tensor j's first batch
  uint64_t batch_tot;    // compress: per batch uint4 (position bytes, M, R, 0)
  uint64_t batch_pre;    // compress: per batch TileSum, exclusive prefix inside its tensor
  uint64_t total;
};

// Decompress: word of the zeroed `overflow` state that the scan sets when a payload of the
// call is version 3 or an overwrite payload.  The thread-level apply kernels come in two
// builds, one for XOR payloads of versions 1 and 2 only (no compact blocks, no overwrites:
// fewer registers, aligned list loads) and a general one; both are launched and the one that
// does not match this word returns at once.
constexpr uint32_t kFlagV3Word = 1;
// ... and the word it sets when a payload of the call is an overwrite payload: the
// incremental apply has a third build, the general one with the overwrite code, selected by it.
constexpr uint32_t kFlagOwWord = 2;

// Index of the job containing global index g, given starts[0..k] (starts[k] = total).
__device__ __forceinline__ uint32_t find_job(const uint64_t* __restrict__ starts, uint32_t k,
                                             uint64_t g) {
  uint32_t lo = 0, hi = k;  // invariant: starts[lo] <= g < starts[hi]
  while (hi - lo > 1) {
    uint32_t mid = (lo + hi) >> 1;
    if (__ldg(starts + mid) <= g) lo = mid; else hi = mid;
  }
  return lo;
}

// Job of global index g when the previous index of this thread was in job j (g only grows).
__device__ __forceinline__ uint32_t advance_job(const uint64_t* __restrict__ starts, uint32_t k,
                                                uint32_t j, uint64_t g) {
  if (j >= k) return find_job(starts, k, g);
  if (__ldg(starts + j + 1) > g) return j;
  if (j + 2 <= k && __ldg(starts + j + 2) > g) return j + 1;
  return find_job(starts, k, g);
}

// The contiguous range [begin, end) of `total` items that warp `gwarp` of `nwarps` takes:
// consecutive chunks of one warp read consecutive memory, and its job index and count-table
// reads advance by one step at a time.
__device__ __forceinline__ void warp_range(uint64_t total, uint64_t gwarp, uint64_t nwarps,
                                           uint64_t& begin, uint64_t& end) {
  const uint64_t per = (total + nwarps - 1) / nwarps;
  begin = gwarp * per;
  end = begin + per < total ? begin + per : total;
}

// Warp-level inclusive scan (sum) of a 32-bit value.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    uint32_t o = __shfl_up_sync(0xFFFFFFFFu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

__device__ __forceinline__ int32_t warp_incl_max(int32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int32_t o = __shfl_up_sync(0xFFFFFFFFu, v, d);
    if (lane >= d) v = max(v, o);
  }
  return v;
}

__device__ __forceinline__ uint64_t warp_sum64(uint64_t v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, d);
  return v;
}

__device__ __forceinline__ void record_status(int32_t* info_status, int32_t code) {
  atomicMax(reinterpret_cast<int*>(info_status), code);
}

}  // namespace bd

// ---------------------------------------------------------------------------- launchers
// Host-side launch functions of each translation unit (internal linkage to the library).
namespace bd {
struct LaunchCtx {
  cudaStream_t stream;
  int sms;             // multiprocessors of the current device
  uint8_t* ws;         // workspace base
  WsLayout lay;
  uint32_t k;          // jobs
  uint64_t chunks;     // total chunks
  uint64_t tiles;      // total scan tiles
  uint64_t batches;    // total fused-compress batches
  uint32_t bchunks;    // chunks per fused-compress batch
};

// fmt: 0 (XOR payloads of versions 1 and 2), 3 (version 3, and overwrite payloads of version
// 2), 4 (version 4); overwrite: the payloads carry new values.
cudaError_t launch_encode_slots(const LaunchCtx& c, uint32_t fmt, bool overwrite);
cudaError_t launch_scan_tiles(const LaunchCtx& c, bool decompress);
cudaError_t launch_scan_jobs(const LaunchCtx& c, bool decompress, int32_t* d_status_all);
cudaError_t launch_emit(const LaunchCtx& c, uint32_t fmt, bool overwrite);
cudaError_t launch_emit_dense(const LaunchCtx& c, bool fused = false);
// The fused compress (encode, scan and emit in one persistent kernel; emit_dense follows it),
// in the same builds as encode_slots and emit.
cudaError_t launch_compress_fused(const LaunchCtx& c, uint32_t fmt, bool overwrite,
                                  int32_t* d_status_all);
cudaError_t launch_apply_chunks(const LaunchCtx& c);
cudaError_t launch_apply_incremental(const LaunchCtx& c);
cudaError_t launch_copy_jobs(const LaunchCtx& c);
cudaError_t launch_apply(const LaunchCtx& c, bool incremental = false);
// The listed chunks (those with a bitmap block) of a call with a workspace, one warp each.
cudaError_t launch_apply_bitmap(const LaunchCtx& c, bool incremental);
cudaError_t launch_apply_finish(const LaunchCtx& c, int32_t* d_status_all);
cudaError_t launch_checksum(const uint16_t* w, uint64_t n, uint64_t* out, cudaStream_t s,
                            int sms);
}  // namespace bd
