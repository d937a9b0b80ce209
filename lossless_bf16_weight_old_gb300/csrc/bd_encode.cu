// bd_encode.cu -- compress kernels of libbf16delta.
//
// "Every byte counts: ARCv3 and the case for cross-region RL", figure "How ARCv3 encodes a
// block of weights": XOR each old/new pair, classify by the changed field, omit unchanged
// values, keep only the mantissa bits of mantissa-only changes and pack exponent/sign changes
// separately as one block; the API returns a checksum beside the payload.
//
// A call goes through one persistent kernel, the fused compress at the end of this file (its
// parts are the kernels below), in one build per payload kind.  A call with a tensor too large
// for it takes two passes around the count scan (bd_scan.cu), neither of which waits on
// another CTA:
//   encode_slots  the only full-size read of old and new.  One warp per 4096-element chunk
//                 (each warp a contiguous range of chunks, each chunk prefetched into L2 as
//                 the warp starts it): branch-free classification, per-chunk class counts,
//                 the checksum of new, and the chunk's nonzero XORs (position, value) in a
//                 fixed 1 KiB workspace slot (a chunk with more changes than a slot holds is
//                 marked overflow and is read again by emit_dense).  The slot also records the
//                 chunk's first mantissa value.
//   emit          one warp per chunk, after the scan: writes the count-table entry, the rare
//                 stream, the position blocks and the chunk's share of the 7-bit mantissa
//                 stream, all at their final payload offsets, 32 slot entries at a time with
//                 the classes split by ballots.  A mantissa-stream byte is written by the
//                 chunk holding the element its first bit belongs to; when the byte reaches
//                 into the next chunk that has mantissa values, the first of them comes from
//                 that chunk's slot.
//   emit_dense    the same for the chunks listed by encode_slots as too dense for a slot:
//                 their changes are derived again from old and new.
#include "bd_internal.cuh"

namespace bd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ unsigned long long* ck_slot(uint8_t* ck_base, uint32_t job,
                                                       uint64_t salt) {
  return reinterpret_cast<unsigned long long*>(ck_base + (uint64_t)job * kCkBytes) +
         (salt & (kCkSlots - 1)) * kCkStride;
}

__device__ __forceinline__ uint4 xor4(uint4 a, uint4 b) {
  return make_uint4(a.x ^ b.x, a.y ^ b.y, a.z ^ b.z, a.w ^ b.w);
}

// 16-bit element-order mask of the nonzero values among the 16 of (x0, x1).
__device__ __forceinline__ uint32_t nz_mask16(uint4 x0, uint4 x1) {
  // per group: low values' flags at even bits 0..6, high values' at 16..22; the second group's
  // at 8..14 and 24..30; one fold moves every high value's flag next to its low neighbour
  const uint32_t ta = (nz_flags(x0.x) >> 15) | (nz_flags(x0.y) >> 13) | (nz_flags(x0.z) >> 11) |
                      (nz_flags(x0.w) >> 9);
  const uint32_t tb = (nz_flags(x1.x) >> 7) | (nz_flags(x1.y) >> 5) | (nz_flags(x1.z) >> 3) |
                      (nz_flags(x1.w) >> 1);
  const uint32_t u = ta | tb;
  return (u | (u >> 15)) & 0xFFFFu;
}

__device__ __forceinline__ uint32_t rare_mask16(uint4 x0, uint4 x1) {
  const uint32_t a = flags_to_mask8(rare_flags(x0.x), rare_flags(x0.y), rare_flags(x0.z),
                                    rare_flags(x0.w));
  const uint32_t b = flags_to_mask8(rare_flags(x1.x), rare_flags(x1.y), rare_flags(x1.z),
                                    rare_flags(x1.w));
  return a | (b << 8);
}

// Checksum terms of a full group of 8 values; key = (index of its first word + 1) * gamma.
__device__ __forceinline__ uint64_t hash_group_full(uint4 v, uint64_t key) {
  const uint64_t w0 = (uint64_t)v.x | ((uint64_t)v.y << 32);
  const uint64_t w1 = (uint64_t)v.z | ((uint64_t)v.w << 32);
  return mix64(w0 ^ key) + mix64(w1 ^ (key + kGamma));
}

// ------------------------------------------------------------------------ encode_slots

// Gaps above 255 in a chunk's merged position list, counted from its k slot entries (position
// order, either layout): the first gap is p_0 + 1, then p_i - p_{i-1}.
__device__ __forceinline__ uint32_t slot_escapes(const uint32_t* __restrict__ entries,
                                                 uint32_t k) {
  const int lane = threadIdx.x & 31;
  int32_t carry = -1;
  uint32_t esc = 0;
  for (uint32_t i0 = 0; i0 < k; i0 += 32) {
    const uint32_t i = i0 + lane;
    const int32_t pos = i < k ? (int32_t)ent_pos(entries[i]) : 0;
    int32_t prev = __shfl_up_sync(0xFFFFFFFFu, pos, 1);
    if (lane == 0) prev = carry;
    esc += __popc(__ballot_sync(0xFFFFFFFFu, i < k && pos - prev > 255));
    carry = __shfl_sync(0xFFFFFFFFu, pos, 31);
  }
  return esc;
}

// The same count for a chunk whose changes did not fit its slot, from old and new again (512
// elements per step, 16 per lane).  Only a lane's first change can follow a gap above 255 --
// its others are under 16 apart -- and its predecessor is the last change of the nearest lower
// lane that has one, or of the steps before.
template <bool FULL>
__device__ __noinline__ uint32_t chunk_escapes(const uint16_t* __restrict__ old,
                                               const uint16_t* __restrict__ neu, uint64_t n,
                                               uint64_t e0) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1;
  int32_t lastp = -1;
  uint32_t esc = 0;
  for (int s = 0; s < 8; s++) {
    const uint32_t eloc = s * 512 + lane * 16;
    const uint64_t e = e0 + eloc;
    uint4 o0, o1, n0, n1;
    if (FULL) {
      o0 = __ldg(reinterpret_cast<const uint4*>(old + e));
      o1 = __ldg(reinterpret_cast<const uint4*>(old + e + 8));
      n0 = __ldg(reinterpret_cast<const uint4*>(neu + e));
      n1 = __ldg(reinterpret_cast<const uint4*>(neu + e + 8));
    } else {
      o0 = load8(old, e, n); o1 = load8(old, e + 8, n);
      n0 = load8(neu, e, n); n1 = load8(neu, e + 8, n);
    }
    const uint32_t nz = nz_mask16(xor4(o0, n0), xor4(o1, n1));
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, nz != 0);
    if (bal == 0) continue;
    const int32_t last = (int32_t)(eloc + 31 - __clz(nz));   // meaningful where nz != 0
    const uint32_t lower = bal & lt;
    const int32_t below = __shfl_sync(0xFFFFFFFFu, last, lower ? 31 - __clz(lower) : 0);
    const int32_t prev = lower ? below : lastp;
    const bool big = nz != 0 && (int32_t)(eloc + __ffs(nz) - 1) - prev > 255;
    esc += __popc(__ballot_sync(0xFFFFFFFFu, big));
    lastp = __shfl_sync(0xFFFFFFFFu, last, 31 - __clz(bal));
  }
  return esc;
}

// Version 4: the Rice statistics of a chunk from its k >= 1 slot entries (position order, either
// layout): the sums of g >> K over its gaps (the warp's totals), and in sum0 the sum of the
// gaps (its last position + 1).
__device__ __forceinline__ RiceSums slot_rice(const uint32_t* __restrict__ entries, uint32_t k,
                                              uint32_t* sum0) {
  const int lane = threadIdx.x & 31;
  int32_t carry = -1;
  RiceSums acc{0, 0};
  for (uint32_t i0 = 0; i0 < k; i0 += 32) {
    const uint32_t i = i0 + lane;
    const int32_t pos = i < k ? (int32_t)ent_pos(entries[i]) : 0;
    int32_t prev = __shfl_up_sync(0xFFFFFFFFu, pos, 1);
    if (lane == 0) prev = carry;
    if (i < k) rice_add(acc, (uint32_t)(pos - prev));
    carry = __shfl_sync(0xFFFFFFFFu, pos, 31);
  }
  *sum0 = ent_pos(entries[k - 1]) + 1;
  return RiceSums{__reduce_add_sync(0xFFFFFFFFu, acc.a), __reduce_add_sync(0xFFFFFFFFu, acc.b)};
}

// The same statistics for a chunk whose changes did not fit its slot, from old and new again
// (512 elements per step, 16 per lane): a lane's first change follows the last change of the
// nearest lower lane that has one, or of the steps before; its others follow one another.
template <bool FULL>
__device__ __noinline__ RiceSums chunk_rice(const uint16_t* __restrict__ old,
                                            const uint16_t* __restrict__ neu, uint64_t n,
                                            uint64_t e0, uint32_t* sum0) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1;
  int32_t lastp = -1;
  RiceSums acc{0, 0};
  for (int s = 0; s < 8; s++) {
    const uint32_t eloc = s * 512 + lane * 16;
    const uint64_t e = e0 + eloc;
    uint4 o0, o1, n0, n1;
    if (FULL) {
      o0 = __ldg(reinterpret_cast<const uint4*>(old + e));
      o1 = __ldg(reinterpret_cast<const uint4*>(old + e + 8));
      n0 = __ldg(reinterpret_cast<const uint4*>(neu + e));
      n1 = __ldg(reinterpret_cast<const uint4*>(neu + e + 8));
    } else {
      o0 = load8(old, e, n); o1 = load8(old, e + 8, n);
      n0 = load8(neu, e, n); n1 = load8(neu, e + 8, n);
    }
    const uint32_t nz = nz_mask16(xor4(o0, n0), xor4(o1, n1));
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, nz != 0);
    if (bal == 0) continue;
    const int32_t last = (int32_t)(eloc + 31 - __clz(nz));   // meaningful where nz != 0
    const uint32_t lower = bal & lt;
    const int32_t below = __shfl_sync(0xFFFFFFFFu, last, lower ? 31 - __clz(lower) : 0);
    int32_t prev = lower ? below : lastp;
    for (uint32_t bits = nz; bits; bits &= bits - 1) {
      const int32_t p = (int32_t)(eloc + __ffs(bits) - 1);
      rice_add(acc, (uint32_t)(p - prev));
      prev = p;
    }
    lastp = __shfl_sync(0xFFFFFFFFu, last, 31 - __clz(bal));
  }
  *sum0 = (uint32_t)(lastp + 1);
  return RiceSums{__reduce_add_sync(0xFFFFFFFFu, acc.a), __reduce_add_sync(0xFFFFFFFFu, acc.b)};
}

// The compress workspace word of a version-4 chunk with M + R (1..508) changes, from its slot
// entries or, when they did not fit, from old and new.  One call for both (two calls from the
// encode loop spilled there).
template <bool FULL>
__device__ __noinline__ uint32_t rice_count(const uint32_t* entries, bool overflow,
                                            const uint16_t* old, const uint16_t* neu, uint64_t n,
                                            uint64_t e0, uint32_t M, uint32_t R) {
  uint32_t sum0;
  const RiceSums sums = !overflow ? slot_rice(entries, M + R, &sum0)
                                  : chunk_rice<FULL>(old, neu, n, e0, &sum0);
  return rice_word(M, R, sum0, sums);
}

// FMT: the payload kinds of the build -- 0: XOR payloads of versions 1 and 2; 3: version 3 (the
// chunk's escaped gaps counted) and overwrite payloads of version 2; 4: version 4 (the chunk's
// Rice statistics gathered, its K and block bytes chosen).
// OW: slot entries in the general layout (kEntRare | pos << 16 | value) with the new field
// values (the new value of a rare change, the new mantissa of a mantissa-only one), read back
// from a per-lane shared copy of the step's new values; otherwise pos << 16 | x (the class
// follows from x).
template <bool FULL, int FMT, bool OW>
__device__ __forceinline__ uint32_t encode_chunk(const uint16_t* __restrict__ old,
                                             const uint16_t* __restrict__ neu, uint64_t n,
                                             uint64_t e0, uint32_t* __restrict__ slot,
                                             uint64_t& ck, uint64_t g,
                                             uint32_t* __restrict__ counts,
                                             uint32_t* __restrict__ list_count,
                                             uint32_t* __restrict__ list,
                                             uint32_t* __restrict__ list_job, uint32_t j,
                                             uint4* __restrict__ xs, uint4* __restrict__ ns) {
  const int lane = threadIdx.x & 31;
  const uint16_t* xs16 = reinterpret_cast<const uint16_t*>(xs);
  const uint16_t* ns16 = reinterpret_cast<const uint16_t*>(ns);
  const uint64_t words = (n + 3) >> 2;
  uint32_t* __restrict__ entries = slot + kSlotHeader / 4;
  uint32_t running = 0;        // changes in the steps done so far
  uint32_t nl = 0, rl = 0;     // this lane's changes, and its rare ones
  uint32_t fm = 0;             // first mantissa value | kAuxHasM once found
  uint64_t e = e0 + lane * 16;
  uint4 o0, o1, n0, n1;
  if (FULL) {
    o0 = __ldcs(reinterpret_cast<const uint4*>(old + e));
    o1 = __ldcs(reinterpret_cast<const uint4*>(old + e + 8));
    n0 = __ldcs(reinterpret_cast<const uint4*>(neu + e));
    n1 = __ldcs(reinterpret_cast<const uint4*>(neu + e + 8));
  } else {
    o0 = load8(old, e, n); o1 = load8(old, e + 8, n);
    n0 = load8(neu, e, n); n1 = load8(neu, e + 8, n);
  }
  uint64_t key = ((e >> 2) + 1) * kGamma;  // key of this lane's first word
#pragma unroll 1
  for (int s = 0; s < 8; s++) {
    const uint4 po0 = o0, po1 = o1, pn0 = n0, pn1 = n1;
    if (s < 7) {
      const uint64_t en = e + 512;
      if (FULL) {
        o0 = __ldcs(reinterpret_cast<const uint4*>(old + en));
        o1 = __ldcs(reinterpret_cast<const uint4*>(old + en + 8));
        n0 = __ldcs(reinterpret_cast<const uint4*>(neu + en));
        n1 = __ldcs(reinterpret_cast<const uint4*>(neu + en + 8));
      } else {
        o0 = load8(old, en, n); o1 = load8(old, en + 8, n);
        n0 = load8(neu, en, n); n1 = load8(neu, en + 8, n);
      }
    }
    const uint32_t eloc = (uint32_t)(e - e0);
    if (FULL) {
      ck += hash_group_full(pn0, key) + hash_group_full(pn1, key + 2 * kGamma);
    } else {
      ck += group_hash(pn0, e >> 3, words) + group_hash(pn1, (e >> 3) + 1, words);
    }
    const uint4 x0 = xor4(po0, pn0), x1 = xor4(po1, pn1);
    const uint32_t nz = nz_mask16(x0, x1);
    if (nz) {   // the lane's 16 XOR values, read back by position in the loop below
      xs[0] = x0;
      xs[1] = x1;
      if (OW) {
        ns[0] = pn0;
        ns[1] = pn1;
      }
    }
    const uint32_t cnt = __popc(nz);
    const uint32_t incl = warp_incl_scan(cnt);
    uint32_t idx = running + incl - cnt;
    uint32_t lane_fm = 0;
    for (uint32_t bits = nz; bits; bits &= bits - 1) {
      const int b = __ffs(bits) - 1;
      const uint32_t xv = xs16[b];
      const bool rare = (xv & kSignExp) != 0;
      uint32_t val = xv;
      if (OW) val = rare ? (uint32_t)ns16[b] : (uint32_t)(ns16[b] & kMant);
      if (rare) {
        rl++;
      } else if (lane_fm == 0) {
        lane_fm = val | kAuxHasM;
      }
      if (idx < kSlotEntries)
        entries[idx] = OW ? ((rare ? kEntRare : 0u) | ((eloc + b) << 16) | val)
                          : (((eloc + b) << 16) | xv);
      idx++;
    }
    nl += cnt;
    if (fm == 0) {
      const uint32_t has = __ballot_sync(0xFFFFFFFFu, lane_fm != 0);
      if (has) fm = __shfl_sync(0xFFFFFFFFu, lane_fm, __ffs(has) - 1);
    }
    running += __shfl_sync(0xFFFFFFFFu, incl, 31);
    e += 512;
    key += 128 * kGamma;  // 512 elements = 128 words per step
  }
  // per-chunk class counts
  nl = warp_incl_scan(nl);
  rl = warp_incl_scan(rl);
  const uint32_t runR = __shfl_sync(0xFFFFFFFFu, rl, 31);
  const uint32_t runM = __shfl_sync(0xFFFFFFFFu, nl, 31) - runR;
  const bool overflow = runM + runR > kSlotEntries;
  uint32_t word = wcount(runM, runR, 0);
  if (FMT == 3 && runM + runR <= kCompactMax) {   // gaps above 255 in the merged list
    uint32_t esc;
    if (!overflow) {
      __syncwarp();   // the slot entries written by every lane are visible to the warp
      esc = slot_escapes(entries, runM + runR);
    } else {
      esc = chunk_escapes<FULL>(old, neu, n, e0);
    }
    word = wcount(runM, runR, esc);
  }
  if (FMT == 4 && runM + runR > 0 && runM + runR <= kCompactMax) {
    __syncwarp();   // the slot entries written by every lane are visible to the warp
    word = rice_count<FULL>(entries, overflow, old, neu, n, e0, runM, runR);
  }
  if (lane == 0) {
    slot[0] = overflow ? kSlotOverflow : slot_info(runM, runR);
    slot[1] = fm;
    counts[g] = word;
    if (overflow) {   // listed for emit_dense, with its tensor
      const uint32_t at = atomicAdd(list_count, 1u);
      list[at] = (uint32_t)g;
      list_job[at] = j;
    }
  }
  return word;   // the same on every lane
}

template <int FMT, bool OW>
__global__ void __launch_bounds__(kThreads, 4)
k_encode_slots(const CJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
               uint32_t k, uint64_t total_chunks, uint32_t* __restrict__ counts,
               uint8_t* __restrict__ slots, uint8_t* __restrict__ ck_base,
               uint32_t* __restrict__ list_count, uint32_t* __restrict__ list,
               uint32_t* __restrict__ list_job) {
  __shared__ uint4 s_xs[kThreads][2];   // per thread: the 16 XOR values of its current step
  __shared__ uint4 s_ns[OW ? kThreads : 1][2];   // OW: its 16 new values
  const int lane = threadIdx.x & 31;
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;

  uint32_t j = 0xFFFFFFFFu, cur = 0xFFFFFFFFu;
  uint64_t ck = 0;
  uint64_t g_begin, g_end;
  warp_range(total_chunks, gwarp, nwarps, g_begin, g_end);
  for (uint64_t g = g_begin; g < g_end; g++) {
    j = advance_job(chunk_start, k, j, g);
    if (j != cur) {
      if (cur != 0xFFFFFFFFu) {
        const uint64_t s = warp_sum64(ck);
        if (lane == 0) atomicAdd(ck_slot(ck_base, cur, gwarp), (unsigned long long)s);
      }
      cur = j;
      ck = 0;
    }
    const uint64_t n = jobs[j].n;
    const uint64_t e0 = (g - chunk_start[j]) * kChunk;
    uint32_t* slot = reinterpret_cast<uint32_t*>(slots + g * kSlotBytes);
    if (e0 + kChunk <= n) {   // the chunk of old and new into L2 ahead of the step loads
      prefetch_chunk_l2(jobs[j].old + e0);
      prefetch_chunk_l2(jobs[j].neu + e0);
    }
    uint4* ns = s_ns[OW ? threadIdx.x : 0];
    if (e0 + kChunk <= n)
      encode_chunk<true, FMT, OW>(jobs[j].old, jobs[j].neu, n, e0, slot, ck, g, counts,
                                  list_count, list, list_job, j, s_xs[threadIdx.x], ns);
    else
      encode_chunk<false, FMT, OW>(jobs[j].old, jobs[j].neu, n, e0, slot, ck, g, counts,
                                   list_count, list, list_job, j, s_xs[threadIdx.x], ns);
  }
  if (cur != 0xFFFFFFFFu) {
    const uint64_t s = warp_sum64(ck);
    if (lane == 0) atomicAdd(ck_slot(ck_base, cur, gwarp), (unsigned long long)s);
  }
}

// ------------------------------------------------------------------------ emit

// Per-warp shared scratch of emit.
struct EmitSmem {
  uint32_t bm[256];   // bitmaps: [0..128) mantissa-only, [128..256) rare
  uint8_t mv[528];    // window of the chunk's 7-bit mantissa values, by chunk-local rank
};

// Where one chunk's output goes.
struct EmitCtx {
  uint8_t* mblk;       // M position block
  uint8_t* rblk;       // R position block
  uint16_t* rstream;   // R stream at this chunk's first R element
  EmitSmem* sm;
  uint32_t M, R;       // the chunk's counts: no write goes past them
  uint32_t wbase;      // chunk-local rank of the value held in sm->mv[0]
  bool listM, listR;
};

struct EmitState {
  uint32_t rankM, rankR;   // elements of each class already emitted in this chunk
  int32_t lastM, lastR;    // position of the last emitted element of each class (0 at start)
};

// Emits one batch: lane holds the elements at positions p0 + b for the set bits b of
// mmask (mantissa-only) and rmask (rare), in ascending position across lanes.
template <typename XF>
__device__ __forceinline__ void emit_batch(uint32_t p0, uint32_t mmask, uint32_t rmask, XF xf,
                                           EmitState& st, const EmitCtx& cx) {
  const int lane = threadIdx.x & 31;
  const uint32_t cm = __popc(mmask), cr = __popc(rmask);
  const uint32_t packed = cm | (cr << 16);
  const uint32_t incl = warp_incl_scan(packed);
  const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
  const uint32_t excl = incl - packed;
  uint32_t rm = st.rankM + (excl & 0xFFFFu);
  uint32_t rr = st.rankR + (excl >> 16);
  // position of the last element of each class in lanes below (or the carry)
  const int32_t myLastM = mmask ? (int32_t)(p0 + 31 - __clz(mmask)) : -1;
  const int32_t myLastR = rmask ? (int32_t)(p0 + 31 - __clz(rmask)) : -1;
  const int32_t inclM = warp_incl_max(myLastM), inclR = warp_incl_max(myLastR);
  int32_t prevM = __shfl_up_sync(0xFFFFFFFFu, inclM, 1);
  int32_t prevR = __shfl_up_sync(0xFFFFFFFFu, inclR, 1);
  if (lane == 0) { prevM = -1; prevR = -1; }
  prevM = max(prevM, st.lastM);
  prevR = max(prevR, st.lastR);

  uint32_t bits = mmask | rmask;
  while (bits) {
    const int b = __ffs(bits) - 1;
    bits &= bits - 1;
    const uint32_t pos = p0 + b;
    const uint32_t x = xf(b);
    if ((mmask >> b) & 1) {
      if (rm >= cx.M) continue;  // never taken when counts and data agree
      if (cx.listM) store_u16(cx.mblk + 2 * rm, (uint16_t)(pos - (uint32_t)prevM));
      else atomicOr(&cx.sm->bm[pos >> 5], 1u << (pos & 31));
      cx.sm->mv[rm - cx.wbase] = (uint8_t)(x & kMant);
      prevM = (int32_t)pos;
      rm++;
    } else {
      if (rr >= cx.R) continue;
      if (cx.listR) store_u16(cx.rblk + 2 * rr, (uint16_t)(pos - (uint32_t)prevR));
      else atomicOr(&cx.sm->bm[128 + (pos >> 5)], 1u << (pos & 31));
      cx.rstream[rr] = (uint16_t)x;
      prevR = (int32_t)pos;
      rr++;
    }
  }
  st.rankM += tot & 0xFFFFu;
  st.rankR += tot >> 16;
  st.lastM = max(st.lastM, __shfl_sync(0xFFFFFFFFu, inclM, 31));
  st.lastR = max(st.lastR, __shfl_sync(0xFFFFFFFFu, inclR, 31));
}

// Writes the mantissa-stream bytes b in [b_lo, b_hi) owned by this chunk.  Byte b starts in
// global element floor(8b/7) (chunk-local jl) at bit s = 8b - 7*floor(8b/7); it takes the top
// 7-s bits of value jl and the low s+1 bits of value jl+1 (`after` when jl+1 == M).
__device__ __forceinline__ void put_mant_bytes(uint8_t* __restrict__ mout, uint64_t b_lo,
                                               uint64_t b_hi, uint64_t Mex, uint32_t M,
                                               uint32_t after, const EmitCtx& cx) {
  const int lane = threadIdx.x & 31;
  // bit offsets relative to the chunk's first mantissa bit 7*Mex fit in 32 bits
  const uint32_t nb = (uint32_t)(b_hi - b_lo);
  const uint32_t rel0 = (uint32_t)(8 * b_lo - 7 * Mex);
  for (uint32_t t = lane; t < nb; t += 32) {
    const uint32_t rel = rel0 + 8 * t;
    const uint32_t jl = rel / 7, s = rel - 7 * jl;
    const uint32_t v0 = cx.sm->mv[jl - cx.wbase];
    const uint32_t v1 = (jl + 1 < M) ? cx.sm->mv[jl + 1 - cx.wbase] : after;
    mout[b_lo + t] = (uint8_t)((v0 >> s) | (v1 << (7 - s)));
  }
}

// Copies a shared bitmap of B bytes to dst.  Every block of a tensor starts at an even
// offset except the R block after an odd-length M bitmap of a ragged last chunk.
__device__ __forceinline__ void store_bitmap(uint8_t* dst, const uint32_t* bm, uint32_t B) {
  const int lane = threadIdx.x & 31;
  const uint8_t* src = reinterpret_cast<const uint8_t*>(bm);
  if ((reinterpret_cast<uintptr_t>(dst) & 1) == 0) {
    for (uint32_t i = lane; i < B / 2; i += 32)
      reinterpret_cast<uint16_t*>(dst)[i] = reinterpret_cast<const uint16_t*>(src)[i];
    if ((B & 1) && lane == 0) dst[B - 1] = src[B - 1];
  } else {
    for (uint32_t i = lane; i < B; i += 32) dst[i] = src[i];
  }
}

// Position of the first mantissa value after chunk g (in g's tensor, ending at g_end) and
// its value, for the last owned byte of g that reaches past g's own values.  `cnt_next` and
// `aux_next` are the counts and slot aux word of chunk g + 1, already loaded.
template <bool V4>
__device__ __forceinline__ uint32_t next_mant_value(uint64_t g, uint64_t g_end, uint32_t cnt_next,
                                                    uint32_t aux_next,
                                                    const uint32_t* __restrict__ counts,
                                                    const uint8_t* __restrict__ slots) {
  const int lane = threadIdx.x & 31;
  if (g + 1 < g_end && (V4 ? v4count_m(cnt_next) : wcount_m(cnt_next)) != 0)
    return aux_next & kMant;
  for (uint64_t gg = g + 2; gg < g_end; gg += 32) {  // rare: chunks without mantissa values
    const uint64_t q = gg + lane;
    const bool has = q < g_end && (V4 ? v4count_m(counts[q]) : wcount_m(counts[q])) != 0;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, has);
    if (bal) {
      const uint64_t gn = gg + __ffs(bal) - 1;
      return reinterpret_cast<const uint32_t*>(slots + gn * kSlotBytes)[1] & kMant;
    }
  }
  return 0;
}

// Output of a version-3 compact chunk.
struct CompactOut {
  uint8_t* blk;        // the chunk's k gap bytes; its class bytes follow at blk + k
  uint16_t* xs;        // X stream at the chunk's first escaped gap
  uint16_t* rstream;   // R stream at the chunk's first rare value
  uint8_t* mv;         // shared: the chunk's 7-bit mantissa values by chunk-local rank
  uint32_t k;          // changes of the chunk
};
struct CompactState {
  uint32_t prev;           // position of the last change emitted (0xFFFFFFFF before the first)
  uint32_t i, m, r, x;     // changes, mantissa-only values, rare values, escapes emitted
};

// Emits the 32 changes cs.i .. cs.i+31 of a compact chunk in position order, lane l holding
// change cs.i + l as a slot entry (OW: the general layout; else pos << 16 | x) when `valid`
// (the valid lanes are a prefix; cs.i is a multiple of 32).  Gap g = pos - previous position (pos + 1 for the first change) goes to
// byte cs.i + l, or 0 there and g to the X stream when g > 255; the class bits of the batch
// are 4 whole bytes of the class section, written by lanes 0..3.
template <bool OW>
__device__ __forceinline__ void compact_batch(uint32_t e, bool valid, CompactState& cs,
                                              const CompactOut& o) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1;
  const uint32_t pos = ent_pos(e), x = e & 0xFFFFu;
  uint32_t prev = __shfl_up_sync(0xFFFFFFFFu, pos, 1);
  if (lane == 0) prev = cs.prev;
  const uint32_t gap = pos - prev;
  const bool rare = OW ? (e & kEntRare) != 0 : (x & kSignExp) != 0;
  const bool isR = valid && rare;
  const bool isM = valid && !rare;
  const bool esc = valid && gap > 255;
  const uint32_t bM = __ballot_sync(0xFFFFFFFFu, isM), bR = __ballot_sync(0xFFFFFFFFu, isR),
                 bE = __ballot_sync(0xFFFFFFFFu, esc);
  if (valid) {
    o.blk[cs.i + lane] = esc ? (uint8_t)0 : (uint8_t)gap;
    if (esc) o.xs[cs.x + __popc(bE & lt)] = (uint16_t)gap;
    if (isM) o.mv[cs.m + __popc(bM & lt)] = (uint8_t)(x & kMant);
    else o.rstream[cs.r + __popc(bR & lt)] = (uint16_t)x;
  }
  const uint32_t b0 = cs.i >> 3, nbytes = (o.k + 7) >> 3;
  if (lane < 4 && b0 + lane < nbytes) o.blk[o.k + b0 + lane] = (uint8_t)(bR >> (8 * lane));
  cs.prev = __shfl_sync(0xFFFFFFFFu, pos, 31);
  cs.i += 32;
  cs.m += __popc(bM);
  cs.r += __popc(bR);
  cs.x += __popc(bE);
}

// Sets the bits of v (below 2^9) at stream bit `at`: one word, or two when v straddles them.
__device__ __forceinline__ void or_bits(uint32_t* bits, uint32_t at, uint32_t v) {
  if (v == 0) return;
  const uint64_t t = (uint64_t)v << (at & 31);
  atomicOr(&bits[at >> 5], (uint32_t)t);
  if (t >> 32) atomicOr(&bits[(at >> 5) + 1], (uint32_t)(t >> 32));
}
// Sets the bits of the n-bit value v (n <= 64, no bits above them) at stream bit `at`: up to
// three words.
__device__ __forceinline__ void or_bits64(uint32_t* bits, uint32_t at, uint64_t v, uint32_t n) {
  const uint32_t w = at >> 5, s = at & 31;
  const uint32_t lo = (uint32_t)(v << s), mid = (uint32_t)(v >> (32 - s));
  if (lo) atomicOr(&bits[w], lo);
  if (n + s > 32 && mid) atomicOr(&bits[w + 1], mid);
  if (n + s > 64) {   // then s > 0
    const uint32_t hi = (uint32_t)(v >> (64 - s));
    if (hi) atomicOr(&bits[w + 2], hi);
  }
}
// Sets the q bits [at, at + q).
__device__ __forceinline__ void ones_run(uint32_t* bits, uint32_t at, uint32_t q) {
  while (q > 0) {
    const uint32_t off = at & 31, take = min(q, 32 - off);
    atomicOr(&bits[at >> 5], (take == 32 ? 0xFFFFFFFFu : (1u << take) - 1u) << off);
    at += take;
    q -= take;
  }
}

// Emits a version-4 compact chunk: its k = M + R changes in position order in list (OW: the
// general layout; else pos << 16 | x), Rice parameter K.  The block is assembled in `bits`
// (shared, zeroed words; stream bit b = bit b%32 of word b/32); the rare values go to rstream
// and the 7-bit mantissa values to mv by class rank.  Each lane takes a contiguous range of
// ceil(k/32) changes: a first pass counts its unary bits and its changes of each class, one
// warp scan places every lane's fields, and a second pass writes them -- the remainder g mod
// 2^K of change i at bit 9R + K*i, the quotient g >> K as that many ones ending before the
// change's unary zero, and for a rare change its index i at bit 9*(its rare rank).  A lane
// gathers its unary codes and its remainders in two 64-bit registers and writes each run with
// one to three atomic ORs (a quotient that does not fit is written on its own); lanes write
// disjoint bit ranges, so their ORs meet only on the words two ranges share.
template <bool OW>
__device__ __forceinline__ void rice_write(const uint32_t* list, uint32_t k, uint32_t R,
                                           uint32_t K, uint32_t* bits, uint16_t* rstream,
                                           uint8_t* mv) {
  const int lane = threadIdx.x & 31;
  const uint32_t per = (k + 31) >> 5;
  const uint32_t i0 = min(lane * per, k), i1 = min(i0 + per, k);
  const uint32_t last = i1 > i0 ? ent_pos(list[i1 - 1]) : 0u;
  uint32_t prev0 = __shfl_up_sync(0xFFFFFFFFu, last, 1);
  if (lane == 0) prev0 = 0xFFFFFFFFu;   // the first gap is the position + 1
  uint32_t U = 0, nr = 0, p = prev0;
  for (uint32_t i = i0; i < i1; i++) {
    const uint32_t e = list[i], pos = ent_pos(e);
    U += ((pos - p) >> K) + 1;
    nr += OW ? (e >> 31) : ((e & kSignExp) != 0);
    p = pos;
  }
  // unary bits (at most 8184), rare and mantissa-only counts (at most 508 each) in one scan
  const uint32_t mine = U | (nr << 14) | ((i1 - i0 - nr) << 23);
  const uint32_t excl = warp_incl_scan(mine) - mine;
  uint32_t ubit = kRiceIdxBits * R + K * k + (excl & 0x3FFFu);
  uint32_t rr = (excl >> 14) & 0x1FFu, mm = excl >> 23;
  const uint32_t rmask = (1u << K) - 1u;
  uint32_t rbit = kRiceIdxBits * R + K * i0;
  uint64_t ua = 0, ra = 0;   // pending unary bits (un of them) and remainder bits (rn)
  uint32_t un = 0, rn = 0;
  p = prev0;
  for (uint32_t i = i0; i < i1; i++) {
    const uint32_t e = list[i], pos = ent_pos(e), g = pos - p, x = e & 0xFFFFu;
    p = pos;
    const uint32_t q = g >> K;
    if (un + q + 1 <= 64) {
      ua |= ((1ull << q) - 1ull) << un;
      un += q + 1;
    } else {
      or_bits64(bits, ubit, ua, un);
      ubit += un;
      ua = 0;
      un = 0;
      ones_run(bits, ubit, q);
      ubit += q + 1;
    }
    if (rn + K > 64) {
      or_bits64(bits, rbit, ra, rn);
      rbit += rn;
      ra = 0;
      rn = 0;
    }
    ra |= (uint64_t)(g & rmask) << rn;
    rn += K;
    if (OW ? (e >> 31) != 0 : (x & kSignExp) != 0) {
      or_bits(bits, kRiceIdxBits * rr, i);
      rstream[rr++] = (uint16_t)x;
    } else {
      mv[mm++] = (uint8_t)(x & kMant);
    }
  }
  or_bits64(bits, ubit, ua, un);
  or_bits64(bits, rbit, ra, rn);
}

// Sets up the output pointers of chunk c (counts M, R, exclusive prefixes Pex / Rex).
__device__ __forceinline__ void emit_ctx(EmitCtx& cx, uint8_t* payload, const JobInfo& I,
                                         uint32_t M, uint32_t R, uint32_t B, uint64_t Pex,
                                         uint64_t Rex, EmitSmem* sm) {
  cx.listM = 2 * M < B;
  cx.listR = 2 * R < B;
  cx.mblk = payload + I.p_start + Pex;
  cx.rblk = cx.mblk + block_bytes(M, B);
  cx.rstream = reinterpret_cast<uint16_t*>(payload + I.r_start) + Rex;
  cx.sm = sm;
  cx.M = M;
  cx.R = R;
  cx.wbase = 0;
}

// The emit work of chunk g (chunk c of tensor j, whose chunks end at g_job_end) once the offsets
// of its tensor's sections (I) and the chunk's exclusive prefixes are known: Pex, Mex, Rex, Xex
// = position bytes, mantissa-only values, rare values and escaped gaps of the chunks before it
// in its tensor.  The slot's single position-ordered list is split by class 32 entries at a
// time with ballots (rank = set lanes below; the previous element of the same class, for the
// delta, is the nearest such lane below or the carry).  FMT as in encode_slots: 3 writes
// version-3 compact blocks, 4 version-4 ones; OW: slot entries in the general layout.
// prefetch_next: ask L2 for the next chunk's slot header and first 96 entries meanwhile.
template <int FMT, bool OW>
__device__ __forceinline__ void emit_chunk(const CJob* __restrict__ jobs, uint64_t g, uint32_t j,
                                           uint64_t c, uint64_t g_job_end, bool prefetch_next,
                                           const JobInfo& I, uint64_t Pex, uint64_t Mex,
                                           uint64_t Rex, uint64_t Xex,
                                           const uint32_t* __restrict__ counts,
                                           const uint8_t* __restrict__ slots, EmitSmem* sm) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1;
  // level 1: everything addressed by g and j alone, requested together
  const uint8_t* slot = slots + g * kSlotBytes;
  if (prefetch_next && lane < 4)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(slot + kSlotBytes + 128 * lane));
  const uint32_t* E = reinterpret_cast<const uint32_t*>(slot + kSlotHeader);
  const uint32_t hdr = *reinterpret_cast<const uint32_t*>(slot);
  uint32_t ent[8];
  // the first 96 entries are read with the header (a slot always has room for them); they
  // cover the whole list of most sparse chunks
  ent[0] = E[lane];
  ent[1] = E[32 + lane];
  ent[2] = E[64 + lane];
  constexpr bool GEN = FMT != 0;
  const uint32_t cnt_here = GEN ? counts[g] : 0u;
  const uint32_t cnt_next = g + 1 < g_job_end ? counts[g + 1] : 0u;
  const uint32_t aux_next =
      g + 1 < g_job_end ? reinterpret_cast<const uint32_t*>(slot + kSlotBytes)[1] : 0u;
  uint8_t* payload = jobs[j].payload;
  const uint64_t n = jobs[j].n;
  if (I.status != BD_OK || (hdr & kSlotOverflow)) return;

  // level 2: the rest of the list
  const uint32_t M = hdr & 0xFFFu, R = (hdr >> 12) & 0xFFFu, kk = M + R;
#pragma unroll
  for (int q = 3; q < 8; q++) ent[q] = 0u;
  if (kk > 96) {
#pragma unroll
    for (int q = 3; q < 8; q++) {
      const uint32_t i = 32 * q + lane;
      if (i < kk) ent[q] = E[i];
    }
  }

  const uint64_t e0 = c * kChunk;
  const uint32_t L = (n - e0) < kChunk ? (uint32_t)(n - e0) : kChunk;
  const uint32_t B = (L + 7) >> 3;
  const uint32_t nesc = wcount_e(cnt_here);
  const bool rice = FMT == 4 && I.version == 4 && rice_compact(cnt_here, B);
  const bool compact = rice || (FMT == 3 && I.version == 3 && choose_compact(M, R, nesc, B));
  if (lane == 0)
    reinterpret_cast<uint32_t*>(payload + count_table_offset(I.r_start, jobs[j].nchunks))[c] =
        rice ? cnt_here : count_entry(GEN ? I.version : 1u, M, R, nesc, compact);
  EmitCtx cx;
  emit_ctx(cx, payload, I, M, R, B, Pex, Rex, sm);
  if constexpr (FMT == 4) {
    if (rice) {
      cx.listM = cx.listR = true;   // no bitmap
      const uint32_t nb = (cnt_here >> 21) & 0x3FFu, K = (cnt_here >> 18) & 0x7u;
      for (uint32_t i = lane; i < (nb + 3) / 4; i += 32) sm->bm[i] = 0;
      __syncwarp();
      rice_write<OW>(E, kk, R, K, sm->bm, cx.rstream, sm->mv);
      __syncwarp();
      store_bitmap(payload + I.p_start + Pex, sm->bm, nb);
    }
  }
  if (FMT == 3 && compact) {
    cx.listM = cx.listR = true;   // no bitmap
    const CompactOut o{payload + I.p_start + Pex,
                       reinterpret_cast<uint16_t*>(payload + I.x_start) + Xex,
                       cx.rstream, sm->mv, kk};
    CompactState cs{0xFFFFFFFFu, 0, 0, 0, 0};
#pragma unroll
    for (int q = 0; q < 8; q++) {
      if (32u * q >= kk) break;
      compact_batch<OW>(ent[q], 32u * q + lane < kk, cs, o);
    }
  }
  if (!cx.listM || !cx.listR) {
    for (int i = lane; i < 256; i += 32) sm->bm[i] = 0;
    __syncwarp();
  }
  uint32_t baseM = 0, baseR = 0, carryM = 0, carryR = 0;
#pragma unroll
  for (int q = 0; q < 8; q++) {
    if (compact || 32u * q >= kk) break;
    const uint32_t e = ent[q], pos = OW ? ent_pos(e) : e >> 16, x = e & 0xFFFFu;
    const bool valid = 32u * q + lane < kk;
    const bool rare = OW ? (e & kEntRare) != 0 : (x & kSignExp) != 0;
    const bool isR = valid && rare;
    const bool isM = valid && !rare;
    const uint32_t bM = __ballot_sync(0xFFFFFFFFu, isM), bR = __ballot_sync(0xFFFFFFFFu, isR);
    // (In versions 1 and 2 every M block starts at an even offset; after an odd-length
    // compact block of version 3 it may not, hence the alignment-checking stores there.)
    if (bR == 0 && cx.listM) {
      // no rare entry in this batch: the mantissa-only entries are the first lanes in order
      const uint32_t prevL = __shfl_up_sync(0xFFFFFFFFu, pos, 1);
      if (isM) {
        const uint32_t r = baseM + lane;
        const uint32_t prev = lane ? prevL : carryM;
        if (GEN) store_u16(cx.mblk + 2 * r, (uint16_t)(pos - prev));
        else reinterpret_cast<uint16_t*>(cx.mblk)[r] = (uint16_t)(pos - prev);
        sm->mv[r] = (uint8_t)(x & kMant);
      }
      const uint32_t cntM = __popc(bM);
      carryM = __shfl_sync(0xFFFFFFFFu, pos, cntM - 1);
      baseM += cntM;
      continue;
    }
    const uint32_t lowM = bM & lt, lowR = bR & lt;
    const uint32_t pM = __shfl_sync(0xFFFFFFFFu, pos, lowM ? 31 - __clz(lowM) : lane);
    const uint32_t pR = __shfl_sync(0xFFFFFFFFu, pos, lowR ? 31 - __clz(lowR) : lane);
    if (isM) {
      const uint32_t r = baseM + __popc(lowM);
      const uint32_t prev = lowM ? pM : carryM;
      if (cx.listM && GEN) store_u16(cx.mblk + 2 * r, (uint16_t)(pos - prev));
      else if (cx.listM) reinterpret_cast<uint16_t*>(cx.mblk)[r] = (uint16_t)(pos - prev);
      else atomicOr(&sm->bm[pos >> 5], 1u << (pos & 31));
      sm->mv[r] = (uint8_t)(x & kMant);
    }
    if (isR) {
      const uint32_t r = baseR + __popc(lowR);
      const uint32_t prev = lowR ? pR : carryR;
      if (cx.listR) store_u16(cx.rblk + 2 * r, (uint16_t)(pos - prev));
      else atomicOr(&sm->bm[128 + (pos >> 5)], 1u << (pos & 31));
      cx.rstream[r] = (uint16_t)x;
    }
    // carries: position of the last element of each class so far
    const uint32_t topM = __shfl_sync(0xFFFFFFFFu, pos, bM ? 31 - __clz(bM) : 0);
    const uint32_t topR = __shfl_sync(0xFFFFFFFFu, pos, bR ? 31 - __clz(bR) : 0);
    if (bM) carryM = topM;
    if (bR) carryR = topR;
    baseM += __popc(bM);
    baseR += __popc(bR);
  }
  __syncwarp();
  // the mantissa-stream bytes owned by this chunk (first bit in one of its values)
  const uint64_t b_lo = (7 * Mex + 7) >> 3, b_hi = (7 * (Mex + M) + 7) >> 3;
  if (b_hi > b_lo) {
    uint32_t after = 0;
    // chunk-local value holding the first bit of the last owned byte (32-bit: the offset
    // from the chunk's first mantissa bit is below 7*M + 8)
    const uint32_t jl_last = (uint32_t)(8 * (b_hi - 1) - 7 * Mex) / 7;
    if (jl_last + 1 == M && Mex + M < I.sum_m)
      after = next_mant_value<FMT == 4>(g, g_job_end, cnt_next, aux_next, counts, slots);
    put_mant_bytes(payload + I.m_start, b_lo, b_hi, Mex, M, after, cx);
  }
  if (!cx.listM || !cx.listR) {
    __syncwarp();
    if (!cx.listM) store_bitmap(cx.mblk, sm->bm, B);
    if (!cx.listR) store_bitmap(cx.rblk, sm->bm + 128, B);
  }
  __syncwarp();
}

// Chunks whose changes fit their slot, each warp a contiguous range; the prefixes come from the
// count scan (tile prefix + chunk prefix inside the tile).
template <int FMT, bool OW>
__global__ void __launch_bounds__(kThreads, 4)
k_emit(const CJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
       const uint64_t* __restrict__ tile_start, uint32_t k, uint64_t total_chunks,
       const uint32_t* __restrict__ counts, const uint8_t* __restrict__ slots,
       const uint4* __restrict__ loc, const TileSum* __restrict__ tile_pre,
       const JobInfo* __restrict__ info) {
  __shared__ EmitSmem s_em[kWarps];
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  EmitSmem* sm = &s_em[threadIdx.x >> 5];
  uint32_t j = 0xFFFFFFFFu;
  uint64_t g_begin, g_end;
  warp_range(total_chunks, gwarp, nwarps, g_begin, g_end);
  for (uint64_t g = g_begin; g < g_end; g++) {
    j = advance_job(chunk_start, k, j, g);
    const uint4 lc = loc[g];
    const uint64_t c = g - chunk_start[j];
    const TileSum pre = tile_pre[tile_start[j] + c / kTileChunks];
    const JobInfo I = info[j];
    emit_chunk<FMT, OW>(jobs, g, j, c, chunk_start[j + 1], g + 1 < g_end, I, pre.p + lc.x,
                        pre.m + lc.y, pre.r + lc.z, pre.e + lc.w, counts, slots, sm);
  }
}

// Emits a version-4 compact chunk from its position-ordered list of changes lst (count word
// cnt; ow: entries in the general layout) and copies its block to dst.  Called, not inlined:
// inlined, emit_dense spilled.
__device__ __noinline__ void emit_rice_list(const uint32_t* lst, uint32_t cnt, bool ow,
                                            uint16_t* rstream, EmitSmem* sm, uint8_t* dst) {
  const int lane = threadIdx.x & 31;
  const uint32_t M = cnt & 0x1FFu, R = (cnt >> 9) & 0x1FFu, kk = M + R;
  const uint32_t nb = (cnt >> 21) & 0x3FFu, K = (cnt >> 18) & 0x7u;
  for (uint32_t i = lane; i < (nb + 3) / 4; i += 32) sm->bm[i] = 0;
  __syncwarp();
  if (ow) rice_write<true>(lst, kk, R, K, sm->bm, rstream, sm->mv);
  else rice_write<false>(lst, kk, R, K, sm->bm, rstream, sm->mv);
  __syncwarp();
  store_bitmap(dst, sm->bm, nb);
}

// Positions of one class in a delta list: lane holds the changes at p0 + b for the set bits b of
// mask, the class's first rank `rank` of them; `last` is the class's last position before this
// step (0 at the start of the chunk, so that the first delta is the position itself).
__device__ __forceinline__ void list_deltas(uint8_t* blk, uint32_t mask, uint32_t p0,
                                            uint32_t rank, uint32_t k, int32_t& last) {
  const int lane = threadIdx.x & 31;
  const int32_t mine = mask ? (int32_t)(p0 + 31 - __clz(mask)) : -1;
  const int32_t incl = warp_incl_max(mine);
  int32_t prev = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
  if (lane == 0) prev = -1;
  prev = max(prev, last);
  for (uint32_t b = mask; b; b &= b - 1, rank++) {
    const uint32_t pos = p0 + __ffs(b) - 1;
    if (rank < k) store_u16(blk + 2 * rank, (uint16_t)(pos - (uint32_t)prev));
    prev = (int32_t)pos;
  }
  last = max(last, __shfl_sync(0xFFFFFFFFu, incl, 31));
}

// A chunk too dense for a slot, with plain (version-1) blocks, one warp: 8 steps of 512 elements
// (lane l: elements 512s + 16l .. +15, the next step's loads in flight).  A bitmap block is
// written straight from the lane's 16-bit class mask (two bytes per lane and step), a delta
// list from the positions; rare values go to the R stream by rank.  The lane's mantissa-only
// values (moved to the front of each 8-element half by byte permutes chosen by the half's
// mask) are packed 7 bits each and ORed into a shared bit buffer at their stream offset
// (buffer bit 0 = stream bit 8 * b_next); after each step the complete bytes are written to the
// M stream and the buffer keeps the bits of the last, incomplete byte.  Only the bytes
// [b_lo, b_hi) belong to the chunk: the bits of its first value that fall in byte b_lo - 1 are
// the previous chunk's to write, and its last byte takes the low bits of the next mantissa
// value of the tensor, `after`.
template <bool FULL>
__device__ __forceinline__ void emit_dense_plain(const uint16_t* __restrict__ old,
                                                 const uint16_t* __restrict__ neu, uint64_t n,
                                                 uint64_t e0, uint32_t B, uint32_t M, uint32_t R,
                                                 uint64_t Mex, const EmitCtx& cx, bool ow,
                                                 uint8_t* __restrict__ mout, uint64_t b_lo,
                                                 uint64_t b_hi, uint32_t* __restrict__ sb,
                                                 uint64_t g, uint64_t g_job_end, uint64_t sum_m,
                                                 const uint32_t* __restrict__ counts,
                                                 const uint8_t* __restrict__ slots,
                                                 const uint2* __restrict__ csel) {
  const int lane = threadIdx.x & 31;
  uint8_t* sbb = reinterpret_cast<uint8_t*>(sb);
  for (int i = lane; i < 256; i += 32) sb[i] = 0;
  __syncwarp();
  uint64_t b_next = b_lo;
  uint32_t rM = 0, rR = 0;
  int32_t lastM = 0, lastR = 0;
  uint64_t e = e0 + 16 * (uint64_t)lane;
  // FULL: the chunk lies below n (no bounds on loads, every bitmap byte exists)
  auto ld = [n](const uint16_t* p, uint64_t at) {
    return FULL ? __ldg(reinterpret_cast<const uint4*>(p + at)) : load8(p, at, n);
  };
  uint4 o0 = ld(old, e), o1 = ld(old, e + 8);
  uint4 n0 = ld(neu, e), n1 = ld(neu, e + 8);
#pragma unroll 1
  for (uint32_t s = 0; s < 8; s++, e += 512) {
    const uint4 x0 = xor4(o0, n0), x1 = xor4(o1, n1);
    const uint4 w0 = ow ? n0 : x0, w1 = ow ? n1 : x1;   // the values written
    if (s < 7) {
      o0 = ld(old, e + 512);
      o1 = ld(old, e + 520);
      n0 = ld(neu, e + 512);
      n1 = ld(neu, e + 520);
    }
    const uint32_t rm = rare_mask16(x0, x1);
    const uint32_t mm = nz_mask16(x0, x1) & ~rm;
    const uint32_t packed = __popc(mm) | (__popc(rm) << 16);
    const uint32_t incl = warp_incl_scan(packed), excl = incl - packed;
    const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const uint32_t p0 = 512 * s + 16 * lane;
    const uint32_t q = 64 * s + 2 * lane;   // the lane's first bitmap byte
    // positions
    if (!cx.listM) {
      if (FULL || q + 1 < B) store_u16(cx.mblk + q, (uint16_t)mm);
      else if (q < B) cx.mblk[q] = (uint8_t)mm;
    } else {
      list_deltas(cx.mblk, mm, p0, rM + (excl & 0xFFFFu), M, lastM);
    }
    if (!cx.listR) {
      if (FULL || q + 1 < B) store_u16(cx.rblk + q, (uint16_t)rm);
      else if (q < B) cx.rblk[q] = (uint8_t)rm;
    } else {
      list_deltas(cx.rblk, rm, p0, rR + (excl >> 16), R, lastR);
    }
    // rare values
    {
      uint32_t r = rR + (excl >> 16);
      for (uint32_t b = rm; b; b &= b - 1, r++) {
        const int i = __ffs(b) - 1;
        if (r < R) cx.rstream[r] = (uint16_t)elem_of(i < 8 ? w0 : w1, i & 7);
      }
    }
    // mantissa-only values into the bit buffer: the 16 mantissas as bytes, the ones in mm
    // moved to the front of each half by byte permutes chosen by its 8-bit mask, then packed
    // 7 bits each
    if (mm) {
      const uint32_t lo8 = mm & 0xFFu, hi8 = mm >> 8;
      const uint32_t m0 = prmt(w0.x, w0.y, 0x6420u) & 0x7F7F7F7Fu;
      const uint32_t m1 = prmt(w0.z, w0.w, 0x6420u) & 0x7F7F7F7Fu;
      const uint32_t m2 = prmt(w1.x, w1.y, 0x6420u) & 0x7F7F7F7Fu;
      const uint32_t m3 = prmt(w1.z, w1.w, 0x6420u) & 0x7F7F7F7Fu;
      const uint2 sl = csel[lo8], sh8 = csel[hi8];
      const uint64_t lo = pack7x4(prmt(m0, m1, sl.x)) | ((uint64_t)pack7x4(prmt(m0, m1, sl.y)) << 28);
      const uint64_t hi = pack7x4(prmt(m2, m3, sh8.x)) | ((uint64_t)pack7x4(prmt(m2, m3, sh8.y)) << 28);
      // 128-bit value (Bh:A) of the lane's 7 * popc(mm) bits
      const uint32_t s0 = 7 * __popc(lo8);   // 0..56
      uint64_t A = lo | (hi << s0), Bh = s0 ? hi >> (64 - s0) : 0;
      int64_t rel = (int64_t)(7 * (Mex + rM + (excl & 0xFFFFu))) - (int64_t)(8 * b_next);
      if (rel < 0) {   // the chunk's first value: its bits below byte b_lo are not ours
        const uint32_t d = (uint32_t)(-rel);
        A = (A >> d) | (Bh << (64 - d));
        Bh >>= d;
        rel = 0;
      }
      const uint32_t wd = (uint32_t)rel >> 5, sh = (uint32_t)rel & 31;
      const uint32_t a0 = (uint32_t)A, a1 = (uint32_t)(A >> 32), a2 = (uint32_t)Bh,
                     a3 = (uint32_t)(Bh >> 32);
      const uint32_t o[5] = {a0 << sh, __funnelshift_l(a0, a1, sh), __funnelshift_l(a1, a2, sh),
                             __funnelshift_l(a2, a3, sh), __funnelshift_l(a3, 0u, sh)};
#pragma unroll
      for (int i = 0; i < 5; i++)
        if (o[i]) atomicOr(&sb[wd + i], o[i]);
    }
    rM += tot & 0xFFFFu;
    rR += tot >> 16;
    __syncwarp();
    // write the complete bytes, keep the incomplete one (the buffer holds `avail` bits; before
    // the chunk's first value it can be up to 7 short of byte b_lo)
    const int64_t avail = (int64_t)(7 * (Mex + rM)) - (int64_t)(8 * b_next);
    uint64_t nbytes = avail > 0 ? (uint64_t)avail >> 3 : 0;
    if (nbytes > b_hi - b_next) nbytes = b_hi - b_next;
    for (uint32_t t = lane; t < (uint32_t)nbytes; t += 32) mout[b_next + t] = sbb[t];
    const uint32_t keep = avail > (int64_t)(8 * nbytes) ? sbb[nbytes] : 0u;
    __syncwarp();
    const uint32_t used = avail > 0 ? (uint32_t)((avail + 31) >> 5) + 1 : 1u;
    for (uint32_t i = lane; i < used && i < 256; i += 32) sb[i] = 0;
    __syncwarp();
    if (lane == 0) sb[0] = keep;
    __syncwarp();
    b_next += nbytes;
  }
  if (b_hi > b_next) {   // the last byte: its high bits start the next value of the tensor
    uint32_t after = 0;
    if (Mex + M < sum_m) {   // (warp-uniform: every lane takes part in the search)
      const uint32_t cnt_next = g + 1 < g_job_end ? counts[g + 1] : 0u;
      const uint32_t aux_next =
          g + 1 < g_job_end ? reinterpret_cast<const uint32_t*>(slots + (g + 1) * kSlotBytes)[1] : 0u;
      after = next_mant_value<true>(g, g_job_end, cnt_next, aux_next, counts, slots);
    }
    const uint32_t bits = (uint32_t)(7 * (Mex + M) - 8 * b_next);   // 1..7
    if (lane == 0) mout[b_next] = (uint8_t)(sbb[0] | (after << bits));
  }
  __syncwarp();
}

// Chunks with more changes than a slot holds (listed by encode_slots): the changes are derived
// again from old and new, 512 elements per step, the whole chunk requested into L2 first.  A
// chunk with version-1 blocks goes through emit_dense_plain; a compact chunk (at most
// kCompactMax changes) first gathers its changes in position order into a shared list, then
// emits them 32 at a time as emit does.
// FUSED: after the fused compress, which leaves per-batch prefixes (batch_pre, batches of
// bchunks chunks from batch_start) instead of the count scan's tile and chunk prefixes; if a
// wait of the fused compress gave up (*abort), it emits nothing and fails every tensor.
template <bool FUSED>
__global__ void __launch_bounds__(kThreads, 3)
k_emit_dense(const CJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
             const uint64_t* __restrict__ tile_start, uint32_t k,
             const uint32_t* __restrict__ list_count, const uint32_t* __restrict__ list,
             const uint32_t* __restrict__ list_job,
             const uint32_t* __restrict__ counts, const uint8_t* __restrict__ slots,
             const uint4* __restrict__ loc, const TileSum* __restrict__ tile_pre,
             const JobInfo* __restrict__ info, const uint64_t* __restrict__ batch_start,
             const TileSum* __restrict__ batch_pre, uint32_t bchunks,
             const uint32_t* __restrict__ abort) {
  if (FUSED && *abort) {
    if (blockIdx.x == 0)
      for (uint32_t j = threadIdx.x; j < k; j += blockDim.x)
        if (jobs[j].d_status) *jobs[j].d_status = BD_ERR_CUDA;
    return;
  }
  __shared__ EmitSmem s_em[kWarps];
  __shared__ uint32_t s_list[kWarps][kCompactMax];   // compact chunks: pos << 16 | x
  __shared__ uint2 s_csel[256];                      // compress selectors by class mask
  static_assert(kThreads == 256, "one selector entry per thread");
  s_csel[threadIdx.x] = make_uint2(compress_sel(threadIdx.x, 0), compress_sel(threadIdx.x, 1));
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  EmitSmem* sm = &s_em[threadIdx.x >> 5];
  uint32_t* lst = s_list[threadIdx.x >> 5];
  const uint32_t listed = *list_count;
  for (uint64_t li = gwarp; li < listed; li += nwarps) {
    const uint64_t g = list[li];
    const uint32_t j = list_job[li];
    const JobInfo I = info[j];
    if (I.status != BD_OK) continue;
    const CJob& J = jobs[j];
    const uint64_t n = J.n;
    const uint64_t c = g - chunk_start[j];
    const uint64_t g_job_end = chunk_start[j + 1];
    const uint64_t e0 = c * kChunk;
    const uint32_t L = (n - e0) < kChunk ? (uint32_t)(n - e0) : kChunk;
    const uint32_t B = (L + 7) >> 3;
    const uint32_t cnt = counts[g];
    const uint32_t M = v4count_m(cnt), R = v4count_r(cnt);
    const uint32_t E = I.version == 3 ? wcount_e(cnt) : 0u;
    uint64_t Pex, Mex, Rex, Xex;
    if (FUSED) {   // the batch's prefix plus the full chunks before this one in its batch
      const uint64_t cb = c - c % bchunks;
      const TileSum pre = batch_pre[batch_start[j] + c / bchunks];
      Pex = pre.p;
      Mex = pre.m;
      Rex = pre.r;
      Xex = pre.e;
      for (uint64_t c2 = cb; c2 < c; c2++) {
        const ChunkCount cc = chunk_layout(counts[chunk_start[j] + c2], kChunk, I.version);
        Pex += chunk_pos_bytes(cc, kChunkBitmap);
        Mex += cc.M;
        Rex += cc.R;
        Xex += cc.E;
      }
    } else {
      const TileSum pre = tile_pre[tile_start[j] + c / kTileChunks];
      const uint4 lc = loc[g];
      Pex = pre.p + lc.x;
      Mex = pre.m + lc.y;
      Rex = pre.r + lc.z;
      Xex = pre.e + lc.w;
    }
    const bool rice = I.version == 4 && rice_compact(cnt, B);
    const bool compact = rice || (I.version == 3 && choose_compact(M, R, E, B));
    const bool ow = (J.flags & kFlagOverwrite) != 0;
    uint8_t* payload = J.payload;
    if (lane == 0)
      reinterpret_cast<uint32_t*>(payload + count_table_offset(I.r_start, jobs[j].nchunks))[c] =
          rice ? cnt : count_entry(I.version, M, R, E, compact);
    EmitCtx cx;
    emit_ctx(cx, payload, I, M, R, B, Pex, Rex, sm);
    if (compact) cx.listM = cx.listR = true;   // no bitmap
    uint8_t* mout = payload + I.m_start;
    const uint64_t b_lo = (7 * Mex + 7) >> 3, b_hi = (7 * (Mex + M) + 7) >> 3;
    const uint64_t b_next = b_lo;
    const uint16_t* __restrict__ old = J.old;
    const uint16_t* __restrict__ neu = J.neu;
    // the whole chunk of old and new requested from DRAM at once (16 KiB); the steps below
    // then find it in L2 instead of waiting for one step's 2 KiB at a time
    if (e0 + kChunk <= n) {
      prefetch_chunk_l2(old + e0);
      prefetch_chunk_l2(neu + e0);
    }
    if (compact) {
      // the chunk's changes in position order (M + R <= kCompactMax of them)
      uint32_t base = 0;
      for (int s = 0; s < 8; s++) {
        const uint32_t eloc = s * 512 + lane * 16;
        const uint64_t e = e0 + eloc;
        const uint4 x0 = xor4(load8(old, e, n), load8(neu, e, n));
        const uint4 x1 = xor4(load8(old, e + 8, n), load8(neu, e + 8, n));
        const uint32_t nz = nz_mask16(x0, x1);
        const uint32_t cntl = __popc(nz), incl = warp_incl_scan(cntl);
        uint32_t idx = base + incl - cntl;
        for (uint32_t bits = nz; bits; bits &= bits - 1, idx++) {
          const int b = __ffs(bits) - 1;
          const uint32_t xv = elem_of(b < 8 ? x0 : x1, b & 7);
          const bool rare = (xv & kSignExp) != 0;
          uint32_t val = xv;
          if (ow) {
            const uint32_t nv = elem_of(load8(neu, e + (b & 8), n), b & 7);
            val = rare ? nv : (nv & kMant);
          }
          if (idx < kCompactMax)
            lst[idx] = ow ? ((rare ? kEntRare : 0u) | ((eloc + b) << 16) | val)
                          : (((eloc + b) << 16) | xv);
        }
        base += __shfl_sync(0xFFFFFFFFu, incl, 31);
      }
      __syncwarp();
      const uint32_t kk = M + R;
      if (rice) {
        emit_rice_list(lst, cnt, ow, cx.rstream, sm, payload + I.p_start + Pex);
      } else {
        const CompactOut o{payload + I.p_start + Pex,
                           reinterpret_cast<uint16_t*>(payload + I.x_start) + Xex,
                           cx.rstream, sm->mv, kk};
        CompactState cs{0xFFFFFFFFu, 0, 0, 0, 0};
        for (uint32_t i0 = 0; i0 < kk; i0 += 32) {
          const bool valid = i0 + lane < kk;
          if (ow) compact_batch<true>(valid ? lst[i0 + lane] : 0u, valid, cs, o);
          else compact_batch<false>(valid ? lst[i0 + lane] : 0u, valid, cs, o);
        }
      }
    }
    if (!compact) {
      if (e0 + kChunk <= n)
        emit_dense_plain<true>(old, neu, n, e0, B, M, R, Mex, cx, ow, mout, b_lo, b_hi, sm->bm,
                               g, g_job_end, I.sum_m, counts, slots, s_csel);
      else
        emit_dense_plain<false>(old, neu, n, e0, B, M, R, Mex, cx, ow, mout, b_lo, b_hi, sm->bm,
                                g, g_job_end, I.sum_m, counts, slots, s_csel);
      continue;
    }
    // a compact chunk: the mantissa-stream bytes it owns, from its values in sm->mv
    __syncwarp();
    if (b_hi > b_next) {
      uint32_t after = 0;
      const uint64_t jg_last = (8 * (b_hi - 1)) / 7;
      if (jg_last + 1 == Mex + M && Mex + M < I.sum_m) {
        const uint32_t cnt_next = g + 1 < g_job_end ? counts[g + 1] : 0u;
        const uint32_t aux_next =
            g + 1 < g_job_end ? reinterpret_cast<const uint32_t*>(slots + (g + 1) * kSlotBytes)[1] : 0u;
        // (the reader of both count-word layouts: versions 1 to 3 never set bit 31)
        after = next_mant_value<true>(g, g_job_end, cnt_next, aux_next, counts, slots);
      }
      put_mant_bytes(mout, b_next, b_hi, Mex, M, after, cx);
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------------ fused compress
//
// Every payload kind (one build per kind, as encode_slots and emit have) in one persistent
// kernel instead of encode_slots, the count scan and emit.  Warps claim batches of consecutive chunks of one tensor (up to 32, per call) in
// order and encode them (encode_chunk, as encode_slots does); the warp that completes the last
// batch of a tensor scans the tensor's batch totals, finishes it (offsets, size, checksum,
// header) and publishes it.  Every batch is claimed a second time, in the same order, as emit
// work, which writes it into the payload (emit_chunk, as emit does): one warp in
// kEmitterEvery takes emit work whenever the next emit batch belongs to a published tensor,
// the others encode until no encode batch is left, then all emit.  A warp that has claimed an
// emit batch of a tensor not yet published encodes further batches while it waits.  Against
// the separate kernels this saves the count-scan launches and the gaps between kernels (a
// schedule that emits only after all encoding measured almost the same as this one).  Every
// claimed encode batch is held by a warp that is running it, and encoding and finishing never wait, so every wait ends, whether or not all
// blocks are resident; the waits are bounded all the same (kWaitLimit idle polls of 256 ns,
// about a second; the longest wait the schedule allows is one batch being encoded plus one
// tensor's scan, well under a millisecond), after which the warp reports BD_ERR_CUDA for the
// tensor and the call, raises the abort word and stops; emit_dense, next on the stream, then
// reports BD_ERR_CUDA for every tensor of the call, whose payloads may be incomplete.
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr uint32_t kEmitterEvery = 4;   // two warps of each block of eight

struct FusedArgs {
  const CJob* jobs;
  const uint64_t* chunk_start;
  const uint64_t* batch_start;
  uint32_t* counts;
  uint8_t* slots;
  uint8_t* ck_base;
  uint32_t* list_count;
  uint32_t* list;
  uint32_t* list_job;
  uint4* batch_tot;
  TileSum* batch_pre;
  JobInfo* info;
  uint32_t* ctl;
  int32_t* status_all;
  uint64_t batches;
  uint32_t k;
  uint32_t bchunks;   // chunks per batch
};

// A u32 that other warps change, read by lane 0 and given to the whole warp.
__device__ __forceinline__ uint32_t warp_read(const uint32_t* p) {
  uint32_t v = 0;
  if ((threadIdx.x & 31) == 0) v = *reinterpret_cast<const volatile uint32_t*>(p);
  return __shfl_sync(0xFFFFFFFFu, v, 0);
}
// The next value of a work counter, claimed for the whole warp.
__device__ __forceinline__ uint32_t warp_claim(uint32_t* ctr) {
  uint32_t v = 0;
  if ((threadIdx.x & 31) == 0) v = atomicAdd(ctr, 1u);
  return __shfl_sync(0xFFFFFFFFu, v, 0);
}

// Scans the batch totals of tensor j (all of its batches encoded) into exclusive prefixes,
// finishes the tensor and publishes it.  Each lane sums a contiguous segment of the batches
// (independent loads, in flight together), one warp scan places the segments, and each lane
// writes its segment's prefixes.  The host takes this path only for tensors of at most
// kMaxFusedBatches batches of at most kMaxBatchChunks chunks, so every sum fits in 32 bits
// (4096 batches x 32 chunks x 4096 values < 2^32).  X: the payloads have an X stream
// (version 3), whose values are scanned too.
template <bool X>
__device__ __noinline__ void fused_finish(const FusedArgs& a, uint32_t j) {
  const int lane = threadIdx.x & 31;
  __threadfence();   // the totals, counts, slots and checksum terms of the other batches
  const uint64_t b0 = a.batch_start[j], nb = a.batch_start[j + 1] - b0;
  const uint64_t per = (nb + 31) / 32;
  const uint64_t s0 = min((uint64_t)lane * per, nb), s1 = min(s0 + per, nb);
  uint32_t sP = 0, sM = 0, sR = 0, sE = 0;
#pragma unroll 4
  for (uint64_t i = s0; i < s1; i++) {
    const uint4 t = __ldcg(&a.batch_tot[b0 + i]);
    sP += t.x;
    sM += t.y;
    sR += t.z;
    if (X) sE += t.w;
  }
  const uint32_t iP = warp_incl_scan(sP), iM = warp_incl_scan(sM), iR = warp_incl_scan(sR),
                 iE = X ? warp_incl_scan(sE) : 0u;
  uint64_t p = iP - sP, m = iM - sM, r = iR - sR, x = iE - sE;
  for (uint64_t i = s0; i < s1; i++) {
    const uint4 t = __ldcg(&a.batch_tot[b0 + i]);
    a.batch_pre[b0 + i] = TileSum{p, m, r, x};
    p += t.x;
    m += t.y;
    r += t.z;
    if (X) x += t.w;
  }
  const uint64_t rP = __shfl_sync(0xFFFFFFFFu, iP, 31), rM = __shfl_sync(0xFFFFFFFFu, iM, 31),
                 rR = __shfl_sync(0xFFFFFFFFu, iR, 31),
                 rE = X ? __shfl_sync(0xFFFFFFFFu, iE, 31) : 0u;
  __threadfence();
  __syncwarp();
  if (lane == 0) {
    JobInfo I{};
    I.sum_p = rP;
    I.sum_m = rM;
    I.sum_r = rR;
    I.sum_e = rE;
    I.chunk_err = 0;
    finish_compress_job(a.jobs[j], j, I, a.ck_base, a.info, a.status_all);
    __threadfence();   // the prefixes, the tensor's info and header before the flag
    *reinterpret_cast<volatile uint32_t*>(&a.ctl[kCtlTensors + 2 * j + 1]) = 1u;
  }
  __syncwarp();
}

// chunk_layout for the build FMT, which fixes the version (FMT 3 also serves the overwrite
// payloads of version 2, so there the tensor's version decides).  The version-1 build keeps its
// own plain sums in fused_encode and fused_emit: through this helper it measured 0.6% slower.
template <int FMT>
__device__ __forceinline__ ChunkCount layout_of(uint32_t w, uint32_t L, uint32_t version) {
  return chunk_layout(w, L, FMT == 0 ? 1u : FMT == 4 ? 4u : version);
}

// Encodes batch b; the warp completing its tensor finishes it.
template <int FMT, bool OW>
__device__ __forceinline__ void fused_encode(const FusedArgs& a, uint32_t b, uint4* xs) {
  uint4* ns = OW ? xs + 2 : xs;   // OW: the step's new values after its XOR values
  const int lane = threadIdx.x & 31;
  const uint32_t j = find_job(a.batch_start, a.k, b);
  const CJob& J = a.jobs[j];
  const uint64_t n = J.n;
  const uint64_t c0 = (b - a.batch_start[j]) * a.bchunks;
  const uint64_t c1 = min(c0 + a.bchunks, J.nchunks);
  uint64_t ck = 0;
  uint32_t sP = 0, sM = 0, sR = 0, sE = 0;
  for (uint64_t c = c0; c < c1; c++) {
    const uint64_t g = J.chunk_base + c, e0 = c * kChunk;
    uint32_t* slot = reinterpret_cast<uint32_t*>(a.slots + g * kSlotBytes);
    uint32_t word;
    if (e0 + kChunk <= n) {   // the chunk of old and new into L2 ahead of the step loads
      prefetch_chunk_l2(J.old + e0);
      prefetch_chunk_l2(J.neu + e0);
      word = encode_chunk<true, FMT, OW>(J.old, J.neu, n, e0, slot, ck, g, a.counts,
                                         a.list_count, a.list, a.list_job, j, xs, ns);
    } else {
      word = encode_chunk<false, FMT, OW>(J.old, J.neu, n, e0, slot, ck, g, a.counts,
                                          a.list_count, a.list, a.list_job, j, xs, ns);
    }
    const uint32_t L = (n - e0) < kChunk ? (uint32_t)(n - e0) : kChunk;
    if constexpr (FMT == 0) {
      const uint32_t M = wcount_m(word), R = wcount_r(word), B = (L + 7) >> 3;
      sP += block_bytes(M, B) + block_bytes(R, B);
      sM += M;
      sR += R;
    } else {
      const ChunkCount cc = layout_of<FMT>(word, L, J.version);
      sP += chunk_pos_bytes(cc, (L + 7) >> 3);
      sM += cc.M;
      sR += cc.R;
      sE += cc.E;
    }
  }
  const uint64_t s = warp_sum64(ck);
  if (lane == 0) {
    if (c1 > c0) atomicAdd(ck_slot(a.ck_base, j, b), (unsigned long long)s);
    a.batch_tot[b] = make_uint4(sP, sM, sR, sE);
  }
  __threadfence();   // this batch's slots, counts, total and checksum terms before its count
  __syncwarp();
  uint32_t fin = 0;
  if (lane == 0) {
    const uint32_t cnt = (uint32_t)(c1 - c0);
    fin = atomicAdd(&a.ctl[kCtlTensors + 2 * j], cnt) + cnt == (uint32_t)J.nchunks;
  }
  if (__shfl_sync(0xFFFFFFFFu, fin, 0)) fused_finish<FMT != 0>(a, j);
}

// Emits batch e of a published tensor.
template <int FMT, bool OW>
__device__ __forceinline__ void fused_emit(const FusedArgs& a, uint32_t e, EmitSmem* sm) {
  const uint32_t j = find_job(a.batch_start, a.k, e);
  const CJob& J = a.jobs[j];
  const uint64_t c0 = (e - a.batch_start[j]) * a.bchunks;
  const uint64_t c1 = min(c0 + a.bchunks, J.nchunks);
  const JobInfo I = a.info[j];
  if (c1 <= c0 || I.status != BD_OK) return;
  const TileSum pre = a.batch_pre[e];
  uint64_t Pex = pre.p, Mex = pre.m, Rex = pre.r, Xex = FMT == 0 ? 0 : pre.e;
  const uint64_t g_job_end = J.chunk_base + J.nchunks;
  for (uint64_t c = c0; c < c1; c++) {
    const uint64_t g = J.chunk_base + c;
    const uint32_t w = a.counts[g];
    emit_chunk<FMT, OW>(a.jobs, g, j, c, g_job_end, c + 1 < c1, I, Pex, Mex, Rex, Xex, a.counts,
                        a.slots, sm);
    const uint64_t e0 = c * kChunk;
    const uint32_t L = (J.n - e0) < kChunk ? (uint32_t)(J.n - e0) : kChunk;
    if constexpr (FMT == 0) {
      const uint32_t B = (L + 7) >> 3;
      Pex += block_bytes(wcount_m(w), B) + block_bytes(wcount_r(w), B);
      Mex += wcount_m(w);
      Rex += wcount_r(w);
    } else {
      const ChunkCount cc = layout_of<FMT>(w, L, I.version);
      Pex += chunk_pos_bytes(cc, (L + 7) >> 3);
      Mex += cc.M;
      Rex += cc.R;
      Xex += cc.E;
    }
  }
}

// Waits until the tensor of emit batch e is published, encoding unclaimed batches meanwhile.
// Returns false when it gave up (reported as BD_ERR_CUDA).
template <int FMT, bool OW>
__device__ __noinline__ bool fused_wait(const FusedArgs& a, uint32_t e, uint4* xs) {
  const uint32_t j = find_job(a.batch_start, a.k, e);
  const uint32_t nbatches = (uint32_t)a.batches;
  uint32_t idle = 0;
  while (warp_read(&a.ctl[kCtlTensors + 2 * j + 1]) == 0) {
    if (warp_read(&a.ctl[0]) < nbatches) {
      const uint32_t b = warp_claim(&a.ctl[0]);
      if (b < nbatches) {
        fused_encode<FMT, OW>(a, b, xs);
        continue;
      }
    }
    if (++idle > kWaitLimit) {
      if ((threadIdx.x & 31) == 0) {
        if (a.jobs[j].d_status) *a.jobs[j].d_status = BD_ERR_CUDA;
        if (a.status_all) atomicMax(reinterpret_cast<int*>(a.status_all), (int)BD_ERR_CUDA);
        atomicExch(&a.ctl[kCtlAbort], 1u);
      }
      return false;
    }
    __nanosleep(256);
  }
  __threadfence();   // the tensor's prefixes, info, counts and slots after its flag
  return true;
}

// Three blocks per SM (80 registers, at most 24 bytes of spills in any build): at four (64
// registers) the inlined encoder and emitter spilled 130-250 bytes a thread; the version-1
// build was 1.2% slower there, and the other builds slower than the separate kernels.
template <int FMT, bool OW>
__global__ void __launch_bounds__(kThreads, 3) k_compress_fused(const FusedArgs a) {
  __shared__ uint4 s_xs[kThreads][OW ? 4 : 2];   // encode: a thread's step (OW: + new values)
  __shared__ EmitSmem s_em[kWarps];               // emit: per-warp bitmaps and mantissa values
  uint4* xs = s_xs[threadIdx.x];
  EmitSmem* sm = &s_em[threadIdx.x >> 5];
  const uint32_t nbatches = (uint32_t)a.batches;
  // While batches remain to be encoded, one warp in kEmitterEvery takes emit work: all warps
  // switching to emit as soon as a tensor is published drained the DRAM stream of the encoding
  // (slower than the separate kernels); a few emitters keep it flowing.  The same number in
  // every block measured best (one in four: 4.97 ms on dense7b; one in eight 4.99; one in
  // three, five or six, which give blocks one or two, 5.03-5.10; one in two 5.10).
  const bool emitter = ((((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5) % kEmitterEvery) == 0;
  for (;;) {
    // emit work first, when the next emit batch belongs to a published tensor
    const uint32_t peek = emitter ? warp_read(&a.ctl[1]) : nbatches;
    bool emit = false;
    if (peek < nbatches) {
      const uint32_t jp = find_job(a.batch_start, a.k, peek);
      emit = warp_read(&a.ctl[kCtlTensors + 2 * jp + 1]) != 0;
    }
    if (!emit) {
      const uint32_t b = warp_claim(&a.ctl[0]);
      if (b < nbatches) {
        fused_encode<FMT, OW>(a, b, xs);
        continue;
      }
    }
    const uint32_t e = warp_claim(&a.ctl[1]);   // (once encoding is all handed out, only this)
    if (e >= nbatches) break;
    if (!fused_wait<FMT, OW>(a, e, xs)) return;
    fused_emit<FMT, OW>(a, e, sm);
  }
}

template <typename K>
int blocks_per_sm(K kernel, int threads) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return per_sm;
}

uint64_t cap_grid(uint64_t want, uint64_t work_items_per_block, uint64_t items) {
  const uint64_t need = (items + work_items_per_block - 1) / work_items_per_block;
  return need < want ? (need ? need : 1) : want;
}

}  // namespace

// The build of a compress kernel for the payload kind (fmt 0, 3 or 4 and overwrite), with its
// blocks per SM.
template <typename K>
struct Builds {
  K k[5];   // <0,false> <3,false> <3,true> <4,false> <4,true>
  int per_sm[5];
  int pick(uint32_t fmt, bool overwrite) const {
    return fmt == 4 ? (overwrite ? 4 : 3) : (overwrite ? 2 : fmt == 3 ? 1 : 0);
  }
};

cudaError_t launch_encode_slots(const LaunchCtx& c, uint32_t fmt, bool overwrite) {
  if (c.chunks == 0) return cudaSuccess;
  using KT = decltype(&k_encode_slots<0, false>);
  static const Builds<KT> b = [] {
    Builds<KT> r{{k_encode_slots<0, false>, k_encode_slots<3, false>, k_encode_slots<3, true>,
                  k_encode_slots<4, false>, k_encode_slots<4, true>}, {}};
    for (int i = 0; i < 5; i++) r.per_sm[i] = blocks_per_sm(r.k[i], kThreads);
    return r;
  }();
  const int w = b.pick(fmt, overwrite);
  const uint64_t grid = cap_grid((uint64_t)b.per_sm[w] * c.sms, kWarps, c.chunks);
  auto kernel = b.k[w];
  kernel<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const CJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start), c.k, c.chunks,
      reinterpret_cast<uint32_t*>(c.ws + c.lay.counts), c.ws + c.lay.slots, c.ws + c.lay.ck,
      reinterpret_cast<uint32_t*>(c.ws + c.lay.overflow),
      reinterpret_cast<uint32_t*>(c.ws + c.lay.ovf_list),
      reinterpret_cast<uint32_t*>(c.ws + c.lay.ovf_job));
  return cudaGetLastError();
}

cudaError_t launch_emit_dense(const LaunchCtx& c, bool fused) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm = blocks_per_sm(k_emit_dense<false>, kThreads);
  const uint64_t grid = cap_grid((uint64_t)per_sm * c.sms, kWarps, c.chunks);
  (fused ? k_emit_dense<true> : k_emit_dense<false>)<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const CJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.tile_start), c.k,
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.overflow),
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.ovf_list),
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.ovf_job),
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.counts), c.ws + c.lay.slots,
      reinterpret_cast<const uint4*>(c.ws + c.lay.loc),
      reinterpret_cast<const TileSum*>(c.ws + c.lay.tile_pre),
      reinterpret_cast<const JobInfo*>(c.ws + c.lay.info),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.batch_start),
      reinterpret_cast<const TileSum*>(c.ws + c.lay.batch_pre), c.bchunks,
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.fused_ctl) + kCtlAbort);
  return cudaGetLastError();
}

cudaError_t launch_compress_fused(const LaunchCtx& c, uint32_t fmt, bool overwrite,
                                  int32_t* d_status_all) {
  if (c.batches == 0) return cudaSuccess;
  using KT = decltype(&k_compress_fused<0, false>);
  static const Builds<KT> bl = [] {
    Builds<KT> r{{k_compress_fused<0, false>, k_compress_fused<3, false>,
                  k_compress_fused<3, true>, k_compress_fused<4, false>,
                  k_compress_fused<4, true>}, {}};
    for (int i = 0; i < 5; i++) r.per_sm[i] = blocks_per_sm(r.k[i], kThreads);
    return r;
  }();
  const int wsel = bl.pick(fmt, overwrite);
  const int per_sm = bl.per_sm[wsel];
  // persistent: one wave of resident blocks (fewer when there is little work)
  const uint64_t grid = cap_grid((uint64_t)per_sm * c.sms, kWarps, c.batches);
  FusedArgs a;
  a.jobs = reinterpret_cast<const CJob*>(c.ws + c.lay.jobs);
  a.chunk_start = reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start);
  a.batch_start = reinterpret_cast<const uint64_t*>(c.ws + c.lay.batch_start);
  a.counts = reinterpret_cast<uint32_t*>(c.ws + c.lay.counts);
  a.slots = c.ws + c.lay.slots;
  a.ck_base = c.ws + c.lay.ck;
  a.list_count = reinterpret_cast<uint32_t*>(c.ws + c.lay.overflow);
  a.list = reinterpret_cast<uint32_t*>(c.ws + c.lay.ovf_list);
  a.list_job = reinterpret_cast<uint32_t*>(c.ws + c.lay.ovf_job);
  a.batch_tot = reinterpret_cast<uint4*>(c.ws + c.lay.batch_tot);
  a.batch_pre = reinterpret_cast<TileSum*>(c.ws + c.lay.batch_pre);
  a.info = reinterpret_cast<JobInfo*>(c.ws + c.lay.info);
  a.ctl = reinterpret_cast<uint32_t*>(c.ws + c.lay.fused_ctl);
  a.status_all = d_status_all;
  a.batches = c.batches;
  a.k = c.k;
  a.bchunks = c.bchunks;
  auto kernel = bl.k[wsel];
  kernel<<<(unsigned)grid, kThreads, 0, c.stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_emit(const LaunchCtx& c, uint32_t fmt, bool overwrite) {
  if (c.chunks == 0) return cudaSuccess;
  using KT = decltype(&k_emit<0, false>);
  static const Builds<KT> b = [] {
    Builds<KT> r{{k_emit<0, false>, k_emit<3, false>, k_emit<3, true>, k_emit<4, false>,
                  k_emit<4, true>}, {}};
    for (int i = 0; i < 5; i++) r.per_sm[i] = blocks_per_sm(r.k[i], kThreads);
    return r;
  }();
  const int w = b.pick(fmt, overwrite);
  const uint64_t grid = cap_grid((uint64_t)b.per_sm[w] * c.sms, kWarps, c.chunks);
  auto kernel = b.k[w];
  kernel<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const CJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.tile_start), c.k, c.chunks,
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.counts), c.ws + c.lay.slots,
      reinterpret_cast<const uint4*>(c.ws + c.lay.loc),
      reinterpret_cast<const TileSum*>(c.ws + c.lay.tile_pre),
      reinterpret_cast<const JobInfo*>(c.ws + c.lay.info));
  return cudaGetLastError();
}

}  // namespace bd
