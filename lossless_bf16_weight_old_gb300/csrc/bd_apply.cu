// bd_apply.cu -- decompress (apply) kernels of libbf16delta.
//
// "GPU-accelerated Weight Teleportation", section "Delta update algebra": the rollout side
// XORs the mask into its old weights to obtain the new ones.  "Every byte counts: ARCv3 and
// the case for cross-region RL": both streams are applied to the previous checkpoint and the
// result is checksummed against the trainer's original.
//
// After the count scan (bd_scan.cu):
//   copy_jobs      out-of-place only: out = old (warp per chunk), so the passes below work on
//                  out in place.
//   apply_chunks   one warp per chunk whose two position blocks are delta lists (the common
//                  case for sparse deltas) or whose block is a compact block (one ascending
//                  list of changes: gap bytes with class bits in version 3, a Rice code of the
//                  gaps with the rare indices in version 4): decodes and checks the whole
//                  chunk into shared memory, XORs each change into out with a 32-bit atomic
//                  XOR performed in L2, then reads the chunk back through L2 for its checksum
//                  terms.  The atomics
//                  bring the touched sectors into L2 where the read-back finds them, so each
//                  sector of out crosses HBM at most once each way.  Chunks with a bitmap
//                  block are listed.
//   apply_dense    one CTA per listed chunk: decodes into an 8 KiB shared mask, XORs the
//                  chunk, writes the changed 16-byte groups and adds their checksum terms.
//   apply_finish   one thread per tensor: checks the mantissa-stream pad bits, compares the
//                  checksum with the expected value and publishes the status.
// A malformed chunk is checked in full before anything is written and is left unwritten, so on
// any error applying the same payload again undoes the other chunks (XOR involution; decoding
// depends on the payload only).
#include <algorithm>

#include "bd_internal.cuh"

namespace bd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xFFFFFFFFu;

// Words of a warp's staging area for a version-4 block: the block (at most 1023 bytes, 256
// words) and a zero guard word, the 512-bit class bitmap of the merged list, then the chunk's
// first values as u16: mantissa-only values 0..127 at [0, 128), rare values 0..31 at
// [128, 160).
constexpr uint32_t kRiceCls = 260;
constexpr uint32_t kRiceVals = kRiceCls + 16;
constexpr uint32_t kRiceWords = kRiceVals + 80;

template <int PRE>
__device__ __forceinline__ bool decode_rice(const uint8_t* __restrict__ blk, uint32_t nb,
                                            uint32_t K, const uint8_t* __restrict__ mbytes,
                                            uint32_t s0, const uint16_t* __restrict__ rvals,
                                            uint32_t M, uint32_t R, uint32_t L, bool ow,
                                            uint32_t* __restrict__ sw,
                                            uint32_t* __restrict__ ent);
// The same as a called function: the block-level kernel holds more registers of its own
// across the decode (inlined there, it needed 128 registers and spilled; the warp-level
// kernels inline it).
__device__ __noinline__ bool decode_rice_call(const uint8_t* blk, uint32_t nb, uint32_t K,
                                              const uint8_t* mbytes, uint32_t s0,
                                              const uint16_t* rvals, uint32_t M, uint32_t R,
                                              uint32_t L, bool ow, uint32_t* sw, uint32_t* ent) {
  return decode_rice<4>(blk, nb, K, mbytes, s0, rvals, M, R, L, ow, sw, ent);
}

// 7-bit value j of an M stream.  The caller guarantees j < number of M values, so the
// second byte is read only when the value crosses into it (and then it exists).
__device__ __forceinline__ uint32_t mant_value(const uint8_t* __restrict__ ms, uint64_t j) {
  const uint64_t bit = 7 * j;
  const uint32_t s = (uint32_t)(bit & 7);
  uint32_t v = ms[bit >> 3] >> s;
  if (s > 1) v |= (uint32_t)ms[(bit >> 3) + 1] << (8 - s);
  return v & kMant;
}

// Adds a warp's checksum partial sum to tensor j's accumulators (one slot per warp parity
// class, so that the atomics of different warps spread over L2 lines).
__device__ __forceinline__ void flush_ck(uint8_t* ck_base, uint32_t j, uint64_t gwarp,
                                         uint64_t ck) {
  const uint64_t s = warp_sum64(ck);
  if ((threadIdx.x & 31) == 0)
    atomicAdd(reinterpret_cast<unsigned long long*>(ck_base + (uint64_t)j * kCkBytes) +
                  (gwarp & (kCkSlots - 1)) * kCkStride,
              (unsigned long long)s);
}

// Records the value of one change at chunk position pos in the shared mask (and, for an
// overwrite payload, the position in the record bitmap of its class).
__device__ __forceinline__ void put_record(uint16_t* s_mask, uint32_t* rec, uint32_t pos,
                                           uint32_t v, bool ow) {
  s_mask[pos] = (uint16_t)v;
  if (ow) atomicOr(&rec[pos >> 5], 1u << (pos & 31));
}

// Whether a rare change with value v may go to pos: not a position of a mantissa-only change,
// and for an XOR payload a value with a sign or exponent bit.  (An XOR payload's mantissa masks
// are nonzero, so a nonzero mask at pos marks one; an overwrite payload's may be zero, so
// its record bitmap does.)
__device__ __forceinline__ bool rare_ok(const uint16_t* s_mask, const uint32_t* rec_m,
                                        uint32_t pos, uint32_t v, bool ow) {
  if (ow) return ((rec_m[pos >> 5] >> (pos & 31)) & 1u) == 0;
  return (v & kSignExp) != 0 && s_mask[pos] == 0;
}

// Overwrite payloads: the XOR mask that takes the 8 current values o of a group to their
// targets -- a rare record's target is the new value, a mantissa-only record's the new
// mantissa under the current sign and exponent -- from the targets t and the group's record
// bits (bit i: element i); elements without a record keep their value.
__device__ __forceinline__ uint4 overwrite_mask(uint4 t, uint4 o, uint32_t rec_m, uint32_t rec_r) {
  uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 8; i++) {
    const uint32_t now = elem_of(o, i), to = elem_of(t, i);
    uint32_t x = 0;
    if ((rec_r >> i) & 1u) x = now ^ to;
    else if ((rec_m >> i) & 1u) x = (now & kMant) ^ to;
    w[i >> 1] |= x << (16 * (i & 1));
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Block-wide exclusive prefix sums of two quantities (0 and 1), each held in two slots per
// thread and ordered slot a of threads 0..255, then slot b of threads 0..255; tot0 / tot1 are
// the totals.  Starts and ends with a barrier, so s_tot may be reused by the next call.
__device__ __forceinline__ void block_scan_ab(uint32_t a0, uint32_t b0, uint32_t a1, uint32_t b1,
                                              uint32_t (*s_tot)[4], uint32_t& xa0,
                                              uint32_t& xb0, uint32_t& xa1, uint32_t& xb1,
                                              uint32_t& tot0, uint32_t& tot1) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t ia0 = warp_incl_scan(a0), ib0 = warp_incl_scan(b0);
  const uint32_t ia1 = warp_incl_scan(a1), ib1 = warp_incl_scan(b1);
  __syncthreads();
  if (lane == 31) { s_tot[w][0] = ia0; s_tot[w][1] = ib0; s_tot[w][2] = ia1; s_tot[w][3] = ib1; }
  __syncthreads();
  uint32_t pa0 = 0, pb0 = 0, pa1 = 0, pb1 = 0, ta0 = 0, tb0 = 0, ta1 = 0, tb1 = 0;
  for (int q = 0; q < kWarps; q++) {
    if (q < w) { pa0 += s_tot[q][0]; pb0 += s_tot[q][1]; pa1 += s_tot[q][2]; pb1 += s_tot[q][3]; }
    ta0 += s_tot[q][0]; tb0 += s_tot[q][1]; ta1 += s_tot[q][2]; tb1 += s_tot[q][3];
  }
  xa0 = pa0 + ia0 - a0;
  xb0 = ta0 + pb0 + ib0 - b0;
  xa1 = pa1 + ia1 - a1;
  xb1 = ta1 + pb1 + ib1 - b1;
  tot0 = ta0 + tb0;
  tot1 = ta1 + tb1;
  __syncthreads();
}

// One CTA per listed chunk (a chunk with a bitmap block, or any chunk on the path without a
// workspace, including version-3 compact chunks): decodes the chunk into an 8 KiB shared XOR
// mask, applies it, writes the changed 16-byte groups and adds the checksum terms of the
// result (INCR: the new-minus-old terms of the changed groups only).
template <bool INCR>
__global__ void __launch_bounds__(kThreads)
k_apply_dense(const DJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
              const uint64_t* __restrict__ tile_start, uint32_t k,
              const uint32_t* __restrict__ list_count, const uint32_t* __restrict__ list,
              const uint4* __restrict__ loc, const TileSum* __restrict__ tile_pre,
              JobInfo* __restrict__ info, uint8_t* __restrict__ ck_base) {
  __shared__ uint4 s_mask4[kChunk / 8];       // the chunk's XOR mask (overwrite: targets), 8 KiB
  __shared__ uint32_t s_rec[2][kChunk / 32];  // overwrite: positions with M / R records
  __shared__ uint32_t s_tot[kWarps][4];
  __shared__ uint32_t s_rice[kRiceWords];     // version 4: warp 0's staging area ...
  __shared__ uint32_t s_rent[kCompactMax];    // ... and the decoded changes
  __shared__ int s_bad;
  uint16_t* s_mask = reinterpret_cast<uint16_t*>(s_mask4);
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;

  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + t) >> 5;
  uint32_t cur = 0xFFFFFFFFu;
  uint64_t ck = 0;
  if (t == 0) s_bad = 0;
  __syncthreads();

  const uint32_t listed = *list_count;
  for (uint32_t li = blockIdx.x; li < listed; li += gridDim.x) {
    const uint64_t g = list[li];
    const uint32_t j = find_job(chunk_start, k, g);
    if (info[j].status != BD_OK) continue;
    if (j != cur) {   // block-uniform
      if (cur != 0xFFFFFFFFu) flush_ck(ck_base, cur, gwarp, ck);
      cur = j;
      ck = 0;
    }

    const DJob& J = jobs[j];
    const uint64_t n = J.n;
    const uint64_t c = g - chunk_start[j];
    const uint64_t e0 = c * kChunk;
    const uint32_t L = (n - e0) < kChunk ? (uint32_t)(n - e0) : kChunk;
    const uint32_t B = (L + 7) >> 3;
    const uint8_t* __restrict__ payload = J.payload;
    const ChunkCount cc = parse_count(reinterpret_cast<const uint32_t*>(
        payload + count_table_offset(info[j].r_start, J.nchunks))[c], info[j].version);
    const uint32_t M = cc.M, R = cc.R;
    const TileSum pre = tile_pre[tile_start[j] + c / kTileChunks];
    const uint4 lc = loc[g];
    const uint64_t Pex = pre.p + lc.x, Mex = pre.m + lc.y, Rex = pre.r + lc.z;
    const uint64_t p_start = info[j].p_start, r_start = info[j].r_start,
                   m_start = info[j].m_start;
    const bool listM = 2 * M < B, listR = 2 * R < B;
    const uint8_t* mblk = payload + p_start + Pex;
    const uint8_t* rblk = mblk + block_bytes(M, B);
    const uint8_t* mstream = payload + m_start;
    const uint8_t* rstream = payload + r_start + 2 * Rex;

    // the chunk of `out` (which holds old at this point): groups t and t + 256
    const uint64_t ea = e0 + 8 * (uint64_t)t, eb = ea + 2048;
    const uint4 oa = load8(J.out, ea, n), ob = load8(J.out, eb, n);
    s_mask4[t] = make_uint4(0, 0, 0, 0);
    s_mask4[t + 256] = make_uint4(0, 0, 0, 0);
    const bool ow = (info[j].flags & kFlagOverwrite) != 0;   // block-uniform
    if (ow && t < 128) {
      s_rec[0][t] = 0;
      s_rec[1][t] = 0;
    }
    // (the first block scan below orders these stores before every scatter)

    bool bad = false;
    if (cc.rice) {
      // warp 0 decodes and checks the Rice block, then every thread records two changes
      if (w == 0) {
        const uint64_t mbit0 = 7 * Mex;
        const bool b = decode_rice_call(mblk, cc.nb, cc.K, mstream + (mbit0 >> 3),
                                   (uint32_t)(mbit0 & 7),
                                   reinterpret_cast<const uint16_t*>(rstream), M, R, L, ow,
                                   s_rice, s_rent);
        if (lane == 0 && b) s_bad = 1;
      }
      __syncthreads();
      if (s_bad == 0) {
        for (uint32_t i = t; i < M + R; i += kThreads) {
          const uint32_t e = s_rent[i];
          put_record(s_mask, s_rec[e >> 31], ent_pos(e), e & 0xFFFFu, ow);
        }
      }
    } else if (cc.compact) {
      // changes t (slot a) and t + 256 (slot b) of the merged list; first the escapes and the
      // rare flags, then the gaps with the escaped values in place
      const uint32_t k = M + R, ia = t, ib = t + 256;
      const uint8_t* blk = mblk;
      const uint8_t* cls = blk + k;
      const uint16_t* xs =
          reinterpret_cast<const uint16_t*>(payload + info[j].x_start) + pre.e + lc.w;
      uint32_t ga = ia < k ? blk[ia] : 0u, gb = ib < k ? blk[ib] : 0u;
      const uint32_t escA = ia < k && ga == 0, escB = ib < k && gb == 0;
      const uint32_t rA = ia < k ? (cls[ia >> 3] >> (ia & 7)) & 1u : 0u;
      const uint32_t rB = ib < k ? (cls[ib >> 3] >> (ib & 7)) & 1u : 0u;
      uint32_t xEa, xEb, xRa, xRb, totE, totR;
      block_scan_ab(escA, escB, rA, rB, s_tot, xEa, xEb, xRa, xRb, totE, totR);
      if (escA) {
        if (xEa < cc.E) ga = xs[xEa];
        if (ga <= 255) bad = true;
      }
      if (escB) {
        if (xEb < cc.E) gb = xs[xEb];
        if (gb <= 255) bad = true;
      }
      if (totE != cc.E || totR != R) bad = true;
      if (t == 0 && (k & 7) != 0 && (cls[(k - 1) >> 3] >> (k & 7)) != 0) bad = true;
      uint32_t pa, pb, unused0, unused1, tg, unused2;
      block_scan_ab(ga, gb, 0u, 0u, s_tot, pa, pb, unused0, unused1, tg, unused2);
      pa += ga - 1;   // inclusive prefix of the gaps, minus one
      pb += gb - 1;
      if (ia < k) {
        uint32_t v = 0;
        if (rA) { if (xRa < R) v = load_u16(rstream + 2 * xRa); else bad = true; }
        else { if (ia - xRa < M) v = mant_value(mstream, Mex + ia - xRa); else bad = true; }
        if (!ow && (rA ? (v & kSignExp) == 0 : v == 0)) bad = true;
        if (pa >= L) bad = true;
        if (!bad) {
          s_mask[pa] = (uint16_t)v;
          if (ow) atomicOr(&s_rec[rA][pa >> 5], 1u << (pa & 31));
        }
      }
      if (ib < k) {
        uint32_t v = 0;
        if (rB) { if (xRb < R) v = load_u16(rstream + 2 * xRb); else bad = true; }
        else { if (ib - xRb < M) v = mant_value(mstream, Mex + ib - xRb); else bad = true; }
        if (!ow && (rB ? (v & kSignExp) == 0 : v == 0)) bad = true;
        if (pb >= L) bad = true;
        if (!bad) {
          s_mask[pb] = (uint16_t)v;
          if (ow) atomicOr(&s_rec[rB][pb >> 5], 1u << (pb & 31));
        }
      }
    } else {
      // per-thread scan inputs: list entry t (slot a) or bitmap bytes t, t+256 (slots a, b)
      uint32_t aM = 0, bM = 0, aR = 0, bR = 0;
      uint32_t byteMa = 0, byteMb = 0, byteRa = 0, byteRb = 0;
      if (listM) {
        if ((uint32_t)t < M) {
          aM = load_u16(mblk + 2 * t);
          if (t > 0 && aM == 0) bad = true;
        }
      } else {
        if ((uint32_t)t < B) byteMa = mblk[t];
        if ((uint32_t)t + 256 < B) byteMb = mblk[t + 256];
        aM = __popc(byteMa);
        bM = __popc(byteMb);
      }
      if (listR) {
        if ((uint32_t)t < R) {
          aR = load_u16(rblk + 2 * t);
          if (t > 0 && aR == 0) bad = true;
        }
      } else {
        if ((uint32_t)t < B) byteRa = rblk[t];
        if ((uint32_t)t + 256 < B) byteRb = rblk[t + 256];
        aR = __popc(byteRa);
        bR = __popc(byteRb);
      }
      // bitmap bits for positions >= L must be zero (only the byte holding position L-1 and
      // later ones can have them)
      if ((L & 7) != 0) {
        const uint32_t lastb = B - 1, keep = (1u << (L & 7)) - 1;
        if (!listM && (((uint32_t)t == lastb && (byteMa & ~keep)) ||
                       ((uint32_t)t + 256 == lastb && (byteMb & ~keep)))) bad = true;
        if (!listR && (((uint32_t)t == lastb && (byteRa & ~keep)) ||
                       ((uint32_t)t + 256 == lastb && (byteRb & ~keep)))) bad = true;
      }

      // block scan over slots in order [a: t = 0..255][b: t = 0..255]
      const uint32_t iaM = warp_incl_scan(aM), ibM = warp_incl_scan(bM);
      const uint32_t iaR = warp_incl_scan(aR), ibR = warp_incl_scan(bR);
      if (lane == 31) { s_tot[w][0] = iaM; s_tot[w][1] = ibM; s_tot[w][2] = iaR; s_tot[w][3] = ibR; }
      __syncthreads();
      uint32_t xaM = 0, xbM = 0, xaR = 0, xbR = 0, totaM = 0, totaR = 0, totbM = 0, totbR = 0;
      for (int q = 0; q < kWarps; q++) {
        if (q < w) { xaM += s_tot[q][0]; xbM += s_tot[q][1]; xaR += s_tot[q][2]; xbR += s_tot[q][3]; }
        totaM += s_tot[q][0]; totbM += s_tot[q][1]; totaR += s_tot[q][2]; totbR += s_tot[q][3];
      }
      xaM += iaM - aM;
      xbM += totaM + ibM - bM;
      xaR += iaR - aR;
      xbR += totaR + ibR - bR;

      // scatter the mantissa-only values
      if (listM) {
        if ((uint32_t)t < M) {
          const uint32_t pos = xaM + aM;   // inclusive prefix of the deltas
          const uint32_t v = mant_value(mstream, Mex + t);
          if (pos >= L || (!ow && v == 0)) bad = true;
          else put_record(s_mask, s_rec[0], pos, v, ow);
        }
      } else {
        if (totaM + totbM != M) bad = true;
        uint32_t r = xaM;
        for (uint32_t bits = byteMa; bits; bits &= bits - 1, r++) {
          const uint32_t pos = 8 * t + __ffs(bits) - 1;
          if (r >= M || pos >= L) { bad = true; break; }
          const uint32_t v = mant_value(mstream, Mex + r);
          if (!ow && v == 0) bad = true; else put_record(s_mask, s_rec[0], pos, v, ow);
        }
        r = xbM;
        for (uint32_t bits = byteMb; bits; bits &= bits - 1, r++) {
          const uint32_t pos = 8 * (t + 256) + __ffs(bits) - 1;
          if (r >= M || pos >= L) { bad = true; break; }
          const uint32_t v = mant_value(mstream, Mex + r);
          if (!ow && v == 0) bad = true; else put_record(s_mask, s_rec[0], pos, v, ow);
        }
      }
      __syncthreads();
      // scatter the rare values; a position already holding a mantissa value is malformed
      if (listR) {
        if ((uint32_t)t < R) {
          const uint32_t pos = xaR + aR;
          const uint32_t v = load_u16(rstream + 2 * t);
          if (pos >= L || !rare_ok(s_mask, s_rec[0], pos, v, ow)) bad = true;
          else put_record(s_mask, s_rec[1], pos, v, ow);
        }
      } else {
        if (totaR + totbR != R) bad = true;
        uint32_t r = xaR;
        for (uint32_t bits = byteRa; bits; bits &= bits - 1, r++) {
          const uint32_t pos = 8 * t + __ffs(bits) - 1;
          if (r >= R || pos >= L) { bad = true; break; }
          const uint32_t v = load_u16(rstream + 2 * r);
          if (!rare_ok(s_mask, s_rec[0], pos, v, ow)) bad = true;
          else put_record(s_mask, s_rec[1], pos, v, ow);
        }
        r = xbR;
        for (uint32_t bits = byteRb; bits; bits &= bits - 1, r++) {
          const uint32_t pos = 8 * (t + 256) + __ffs(bits) - 1;
          if (r >= R || pos >= L) { bad = true; break; }
          const uint32_t v = load_u16(rstream + 2 * r);
          if (!rare_ok(s_mask, s_rec[0], pos, v, ow)) bad = true;
          else put_record(s_mask, s_rec[1], pos, v, ow);
        }
      }
    }
    if (bad) s_bad = 1;
    __syncthreads();
    const bool chunk_bad = s_bad != 0;
    if (!chunk_bad) {
      uint4 ma = s_mask4[t], mb = s_mask4[t + 256];
      if (ow) {   // targets -> XOR masks against the current values of groups t and t + 256
        const uint32_t sh = (8 * t) & 31;
        ma = overwrite_mask(ma, oa, (s_rec[0][t >> 2] >> sh) & 0xFFu, (s_rec[1][t >> 2] >> sh) & 0xFFu);
        mb = overwrite_mask(mb, ob, (s_rec[0][(t + 256) >> 2] >> sh) & 0xFFu,
                            (s_rec[1][(t + 256) >> 2] >> sh) & 0xFFu);
      }
      const uint4 ra = make_uint4(oa.x ^ ma.x, oa.y ^ ma.y, oa.z ^ ma.z, oa.w ^ ma.w);
      const uint4 rb = make_uint4(ob.x ^ mb.x, ob.y ^ mb.y, ob.z ^ mb.z, ob.w ^ mb.w);
      const bool cha = (ma.x | ma.y | ma.z | ma.w) != 0, chb = (mb.x | mb.y | mb.z | mb.w) != 0;
      uint16_t* out = J.out;
      if (ea < n && cha) {
        if (ea + 8 <= n) *reinterpret_cast<uint4*>(out + ea) = ra;
        else for (int i = 0; ea + i < n; i++) out[ea + i] = (uint16_t)elem_of(ra, i);
      }
      if (eb < n && chb) {
        if (eb + 8 <= n) *reinterpret_cast<uint4*>(out + eb) = rb;
        else for (int i = 0; eb + i < n; i++) out[eb + i] = (uint16_t)elem_of(rb, i);
      }
      const uint64_t words = (n + 3) >> 2;
      if (INCR) {
        if (cha) ck += group_hash(ra, ea >> 3, words) - group_hash(oa, ea >> 3, words);
        if (chb) ck += group_hash(rb, eb >> 3, words) - group_hash(ob, eb >> 3, words);
      } else {
        ck += group_hash(ra, ea >> 3, words) + group_hash(rb, eb >> 3, words);
      }
    }
    __syncthreads();
    if (t == 0 && chunk_bad) {
      record_status(&info[j].chunk_err, BD_ERR_FORMAT);
      s_bad = 0;
    }
    __syncthreads();
  }
  if (cur != 0xFFFFFFFFu) flush_ck(ck_base, cur, gwarp, ck);
}

// ------------------------------------------------------------------------ apply_chunks

// Longest delta list of a chunk: a block is a list only while 2k < 512 bytes.
constexpr uint32_t kListMax = 255;
constexpr uint32_t kEntMax = 2 * kListMax + 2;
constexpr uint32_t kNone = 0xFFFFFFFFu;

// Loads served by L2 only (never by L1): `out` is changed by L2 atomics while the kernel runs.
// Volatile so that the compiler keeps them after the atomics and the fence that precede them.
__device__ __forceinline__ uint4 ld_l2(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_l2_u16(const uint16_t* p) {
  unsigned short v;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 load8_l2(const uint16_t* p, uint64_t e, uint64_t n) {
  if (e + 8 <= n) return ld_l2(p + e);
  uint32_t w[4] = {0, 0, 0, 0};
  for (int i = 0; i < 8; i++)
    if (e + i < n) w[i >> 1] |= ld_l2_u16(p + e + i) << (16 * (i & 1));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Checksum terms of one chunk of w (elements e0 .. e0+4095, clipped at n; used for the last,
// partial chunk of a tensor), one warp: two 512-element steps at a time per lane, with the
// next two steps' loads in flight.
template <bool FULL>
__device__ __forceinline__ uint64_t hash_chunk_r(const uint16_t* w, uint64_t n, uint64_t e0) {
  const int lane = threadIdx.x & 31;
  const uint64_t words = (n + 3) >> 2;
  uint64_t ck = 0;
  uint64_t e = e0 + 16 * lane;
  uint4 a0, a1, b0, b1;
  if (FULL) {
    a0 = ld_l2(w + e); a1 = ld_l2(w + e + 8);
    b0 = ld_l2(w + e + 512); b1 = ld_l2(w + e + 520);
  } else {
    a0 = load8_l2(w, e, n); a1 = load8_l2(w, e + 8, n);
    b0 = load8_l2(w, e + 512, n); b1 = load8_l2(w, e + 520, n);
  }
  uint64_t key = ((e >> 2) + 1) * kGamma;
#pragma unroll 1
  for (int s = 0; s < 8; s += 2) {
    const uint4 c0 = a0, c1 = a1, d0 = b0, d1 = b1;
    if (s < 6) {
      const uint64_t en = e + 1024;
      if (FULL) {
        a0 = ld_l2(w + en); a1 = ld_l2(w + en + 8);
        b0 = ld_l2(w + en + 512); b1 = ld_l2(w + en + 520);
      } else {
        a0 = load8_l2(w, en, n); a1 = load8_l2(w, en + 8, n);
        b0 = load8_l2(w, en + 512, n); b1 = load8_l2(w, en + 520, n);
      }
    }
    if (FULL) {
      const uint64_t kb = key + 128 * kGamma;
      ck += mix64(((uint64_t)c0.x | ((uint64_t)c0.y << 32)) ^ key) +
            mix64(((uint64_t)c0.z | ((uint64_t)c0.w << 32)) ^ (key + kGamma)) +
            mix64(((uint64_t)c1.x | ((uint64_t)c1.y << 32)) ^ (key + 2 * kGamma)) +
            mix64(((uint64_t)c1.z | ((uint64_t)c1.w << 32)) ^ (key + 3 * kGamma)) +
            mix64(((uint64_t)d0.x | ((uint64_t)d0.y << 32)) ^ kb) +
            mix64(((uint64_t)d0.z | ((uint64_t)d0.w << 32)) ^ (kb + kGamma)) +
            mix64(((uint64_t)d1.x | ((uint64_t)d1.y << 32)) ^ (kb + 2 * kGamma)) +
            mix64(((uint64_t)d1.z | ((uint64_t)d1.w << 32)) ^ (kb + 3 * kGamma));
    } else {
      ck += group_hash(c0, e >> 3, words) + group_hash(c1, (e >> 3) + 1, words) +
            group_hash(d0, (e + 512) >> 3, words) + group_hash(d1, ((e + 512) >> 3) + 1, words);
    }
    e += 1024;
    key += 256 * kGamma;
  }
  return ck;
}

// Checksum terms of one full chunk, one warp: the lane's 16 loads (its 8 KiB share of the
// chunk, 256 bytes) are all issued before the first term is formed.  The chunk was prefetched
// into L2, so the whole read-back costs one L2 round trip; this needs 76 registers, i.e. three
// blocks per SM, which measured faster than four blocks with two steps in flight.
template <bool FULL>
__device__ __forceinline__ uint64_t hash_chunk(const uint16_t* w, uint64_t n, uint64_t e0) {
  if (!FULL) return hash_chunk_r<false>(w, n, e0);
  const int lane = threadIdx.x & 31;
  const uint64_t e = e0 + 16 * lane;
  uint4 v[16];
#pragma unroll
  for (int s = 0; s < 8; s++) {
    v[2 * s] = ld_l2(w + e + 512 * s);
    v[2 * s + 1] = ld_l2(w + e + 512 * s + 8);
  }
  uint64_t key = ((e >> 2) + 1) * kGamma, ck = 0;
#pragma unroll
  for (int s = 0; s < 8; s++) {
    const uint4 c0 = v[2 * s], c1 = v[2 * s + 1];
    ck += mix64(((uint64_t)c0.x | ((uint64_t)c0.y << 32)) ^ key) +
          mix64(((uint64_t)c0.z | ((uint64_t)c0.w << 32)) ^ (key + kGamma)) +
          mix64(((uint64_t)c1.x | ((uint64_t)c1.y << 32)) ^ (key + 2 * kGamma)) +
          mix64(((uint64_t)c1.z | ((uint64_t)c1.w << 32)) ^ (key + 3 * kGamma));
    key += 128 * kGamma;
  }
  return ck;
}

// 7-bit value m of the M stream whose first value starts at bit s0 of mbytes; the caller
// guarantees m < the chunk's M, so the second byte is read only when the value crosses into it.
__device__ __forceinline__ uint32_t mant_at(const uint8_t* __restrict__ mbytes, uint32_t s0,
                                            uint32_t m) {
  const uint32_t bit = s0 + 7 * m, sh = bit & 7;
  uint32_t v = (uint32_t)mbytes[bit >> 3] >> sh;
  if (sh > 1) v |= (uint32_t)mbytes[(bit >> 3) + 1] << (8 - sh);
  return v & kMant;
}

// Decodes a version-3 compact chunk (one warp) into ent[0..M+R) in the general entry layout,
// in ascending position, 32 changes at a time: gap bytes from blk (a zero byte takes the next
// X-stream value, which must exceed 255; at most E of them, and exactly E), positions from
// the prefix sums of the gaps (first position = first gap - 1, all below L), classes from the
// class bits at blk + M + R (exactly R set, pad bits zero), mantissa-only values from the M
// stream, rare values from the R stream (XOR payloads: a mantissa mask is nonzero, a rare mask
// has a sign or exponent bit; an overwrite payload's values are unrestricted).  Returns
// whether the chunk is malformed (the same on every lane).
template <int PRE>
__device__ __forceinline__ bool decode_compact(const uint8_t* __restrict__ blk,
                                               const uint16_t* __restrict__ xs, uint32_t E,
                                               const uint8_t* __restrict__ mbytes, uint32_t s0,
                                               const uint16_t* __restrict__ rvals, uint32_t M,
                                               uint32_t R, uint32_t L, bool ow,
                                               uint32_t* __restrict__ ent) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1;
  const uint32_t k = M + R;
  const uint8_t* __restrict__ cls = blk + k;
  bool bad = false;
  uint32_t carry = 0xFFFFFFFFu, xr = 0, mr = 0, rr = 0;
  // the checks and the entry of change i, gap g (escaped values in place), class isR, value v
  auto finish = [&](uint32_t i, bool in, uint32_t g, bool isR, uint32_t v) {
    const uint32_t p = carry + warp_incl_scan(g);
    carry = __shfl_sync(kFull, p, 31);
    if (in) {
      if (!ow && (isR ? (v & kSignExp) == 0 : v == 0)) bad = true;
      if (p >= L) bad = true;
      if (!bad) ent[i] = (isR ? kEntRare : 0u) | (p << 16) | v;
    }
  };
  if constexpr (PRE > 0) {
    // the first PRE batches: gap bytes and class bits requested together, then -- their ranks
    // known from ballots -- every escaped gap and value, before the first is used
    constexpr int NQ = PRE > 0 ? PRE : 1;   // (arrays of size 0 are not allowed)
    uint32_t gq[NQ], cq[NQ], vq[NQ];
#pragma unroll
    for (int q = 0; q < PRE; q++) {
      const uint32_t i = 32 * q + lane;
      gq[q] = i < k ? (uint32_t)blk[i] : 0u;
      cq[q] = i < k ? (uint32_t)(cls[i >> 3] >> (i & 7)) & 1u : 0u;
    }
#pragma unroll
    for (int q = 0; q < PRE; q++) {
      const uint32_t i = 32 * q + lane;
      const bool in = i < k;
      const bool esc = in && gq[q] == 0;
      const bool isR = in && cq[q] != 0;
      const uint32_t bE = __ballot_sync(kFull, esc), bR = __ballot_sync(kFull, isR),
                     bM = __ballot_sync(kFull, in && !isR);
      if (esc) {
        const uint32_t xi = xr + __popc(bE & lt);
        if (xi < E) gq[q] = xs[xi];   // stays 0 past E: flagged below
        cq[q] |= 2u;
      }
      vq[q] = 0;
      if (isR) {
        const uint32_t r = rr + __popc(bR & lt);
        if (r < R) vq[q] = rvals[r];
        else cq[q] |= 4u;
      } else if (in) {
        const uint32_t m = mr + __popc(bM & lt);
        if (m < M) vq[q] = mant_at(mbytes, s0, m);
        else cq[q] |= 4u;
      }
      xr += __popc(bE);
      rr += __popc(bR);
      mr += __popc(bM);
    }
#pragma unroll
    for (int q = 0; q < PRE; q++) {
      if (32u * q >= k) break;
      const uint32_t i = 32 * q + lane;
      if (((cq[q] & 2u) && gq[q] <= 255) || (cq[q] & 4u)) bad = true;
      finish(i, i < k, gq[q], (cq[q] & 1u) != 0, vq[q]);
    }
  }
  for (uint32_t b0 = 32 * PRE; b0 < k; b0 += 32) {
    const uint32_t i = b0 + lane;
    const bool in = i < k;
    uint32_t g = in ? (uint32_t)blk[i] : 0u;
    const bool esc = in && g == 0;
    const uint32_t bE = __ballot_sync(kFull, esc);
    if (esc) {
      const uint32_t xi = xr + __popc(bE & lt);
      if (xi < E) g = xs[xi];
      if (g <= 255) bad = true;
    }
    xr += __popc(bE);
    const bool isR = in && ((cls[i >> 3] >> (i & 7)) & 1u);
    const uint32_t bR = __ballot_sync(kFull, isR), bM = __ballot_sync(kFull, in && !isR);
    uint32_t v = 0;
    if (isR) {
      const uint32_t r = rr + __popc(bR & lt);
      if (r < R) v = rvals[r];
      else bad = true;
    } else if (in) {
      const uint32_t m = mr + __popc(bM & lt);
      if (m < M) v = mant_at(mbytes, s0, m);
      else bad = true;
    }
    mr += __popc(bM);
    rr += __popc(bR);
    finish(i, in, g, isR, v);
  }
  if (xr != E || rr != R) bad = true;
  if (lane == 0 && (k & 7) != 0 && (cls[(k - 1) >> 3] >> (k & 7)) != 0) bad = true;
  return __any_sync(kFull, bad);
}

// Decodes a version-4 compact chunk (one warp) into ent[0..M+R) in the general entry layout,
// in ascending position: the nb-byte Rice block at blk with parameter K is staged as words in
// sw (kRiceWords, per warp), the rare indices set the class bitmap, each lane finds the zeros
// of one 32-bit window of the unary section (their offsets go to ent[rank] for rank < k), and
// the changes are then formed 32 at a time -- gap (quotient << K | remainder, quotient from
// two consecutive zeros), position from the prefix sums of the gaps, value from the M or R
// stream by class.  Checks, as the format requires: the fixed fields fit in the block; the
// rare indices strictly ascend below k; k zeros in the unary section; the bits used end in
// the block's last byte and the pad bits after them are zero (the ones of the section are
// exactly the quotients' ones); every gap is at least 1 and every position below L; the value
// rules of apply_chunks.  The first 32*PRE mantissa-only values and, when PRE > 0, the first
// 32 rare values are requested with the block (PRE <= 4).  Returns whether the chunk is
// malformed (the same on every lane).
template <int PRE>
__device__ __forceinline__ bool decode_rice(const uint8_t* __restrict__ blk, uint32_t nb,
                                            uint32_t K, const uint8_t* __restrict__ mbytes,
                                            uint32_t s0, const uint16_t* __restrict__ rvals,
                                            uint32_t M, uint32_t R, uint32_t L, bool ow,
                                            uint32_t* __restrict__ sw,
                                            uint32_t* __restrict__ ent) {
  const int lane = threadIdx.x & 31;
  const uint32_t lt = (1u << lane) - 1;
  const uint32_t k = M + R, nbits = 8 * nb, nw = (nb + 3) >> 2;   // nw <= 256
  uint32_t* __restrict__ cls = sw + kRiceCls;
  uint16_t* __restrict__ sv = reinterpret_cast<uint16_t*>(sw + kRiceVals);
  // the first 128 mantissa-only and 32 rare values are requested with the block, so that the
  // whole decode waits for one round of loads
  constexpr int NQ = PRE > 0 ? PRE : 1;   // (arrays of size 0 are not allowed)
  uint32_t mraw[NQ];
#pragma unroll
  for (int q = 0; q < PRE; q++) {
    const uint32_t m = 32 * q + lane;
    mraw[q] = 0;
    if (m < M) {
      const uint32_t bit = s0 + 7 * m;
      mraw[q] = mbytes[bit >> 3];
      if ((bit & 7) > 1) mraw[q] |= (uint32_t)mbytes[(bit >> 3) + 1] << 8;
    }
  }
  const uint32_t rv0 = PRE > 0 && (uint32_t)lane < R ? (uint32_t)rvals[lane] : 0u;
  // the block as little-endian words, bytes past it zero, and the guard word
  for (uint32_t i = lane; i <= nw; i += 32) {
    uint32_t v = 0;
#pragma unroll
    for (int b = 0; b < 4; b++)
      if (4 * i + b < nb) v |= (uint32_t)blk[4 * i + b] << (8 * b);
    sw[i] = v;
  }
  if (lane < 16) cls[lane] = 0;
#pragma unroll
  for (int q = 0; q < PRE; q++)
    sv[32 * q + lane] = (uint16_t)((mraw[q] >> ((s0 + 7 * (32 * q + lane)) & 7)) & kMant);
  if (PRE > 0) sv[128 + lane] = (uint16_t)rv0;
  __syncwarp();
  // nbits-bit field at bit `at` of the block (at < 32 * nw, so the second word exists)
  auto field = [&](uint32_t at, uint32_t bits) -> uint32_t {
    const uint32_t wd = at >> 5;
    return __funnelshift_r(sw[wd], sw[wd + 1], at & 31) & ((1u << bits) - 1u);
  };
  const uint32_t fixed = kRiceIdxBits * R + K * k;
  if (fixed >= nbits) return true;   // no room for the k unary zeros (the same on every lane)
  bool bad = false;
  // rare indices: strictly ascending, below k
  uint32_t last = 0;
  for (uint32_t j0 = 0; j0 < R; j0 += 32) {
    const uint32_t jj = j0 + lane;
    const bool in = jj < R;
    const uint32_t idx = in ? field(kRiceIdxBits * jj, kRiceIdxBits) : 0u;
    uint32_t before = __shfl_up_sync(kFull, idx, 1);
    if (lane == 0) before = last;
    if (in) {
      if (idx >= k || (jj > 0 && idx <= before)) bad = true;
      else atomicOr(&cls[idx >> 5], 1u << (idx & 31));
    }
    last = __shfl_sync(kFull, idx, 31);
  }
  // the unary section [fixed, nbits): the offsets of its zeros by rank into ent, and the count
  // of its ones.  A short section is read 32 bits at a time, the same word on every lane (lane
  // l ranks bit l); a long one (over 12 words, only in dense chunks) one word per lane, each
  // lane listing the zeros of its word.
  const uint32_t nwin = (nbits - fixed + 31) >> 5;
  uint32_t zeros = 0, ones = 0;
  if (nwin <= 12) {
    for (uint32_t at = fixed; at < nbits; at += 32) {
      const uint32_t avail = nbits - at;
      const uint32_t valid = avail >= 32 ? 0xFFFFFFFFu : (1u << avail) - 1u;
      const uint32_t wd = at >> 5;
      const uint32_t win = __funnelshift_r(sw[wd], sw[wd + 1], at & 31);
      const uint32_t zm = ~win & valid;
      ones += __popc(win & valid);
      const uint32_t r = zeros + __popc(zm & lt);
      if (((zm >> lane) & 1u) && r < k) ent[r] = at - fixed + lane;
      zeros += __popc(zm);
    }
  } else {
    for (uint32_t t0 = 0; t0 < nwin; t0 += 32) {
      const uint32_t t = t0 + lane;
      uint32_t zm = 0;
      if (t < nwin) {
        const uint32_t at = fixed + 32 * t, avail = nbits - at;
        const uint32_t valid = avail >= 32 ? 0xFFFFFFFFu : (1u << avail) - 1u;
        const uint32_t wd = at >> 5;
        const uint32_t win = __funnelshift_r(sw[wd], sw[wd + 1], at & 31);
        zm = ~win & valid;
        ones += __popc(win & valid);
      }
      const uint32_t cz = __popc(zm), incl = warp_incl_scan(cz);
      uint32_t r = zeros + incl - cz;
      for (; zm != 0 && r < k; zm &= zm - 1, r++) ent[r] = 32 * t + __ffs(zm) - 1;
      zeros += __shfl_sync(kFull, incl, 31);
    }
    ones = __reduce_add_sync(kFull, ones);
  }
  __syncwarp();
  if (__any_sync(kFull, bad) || zeros < k) return true;
  const uint32_t zlast = ent[k - 1];                  // offset of the k-th zero
  const uint32_t used = fixed + zlast + 1;
  if ((used + 7) / 8 != nb || ones != zlast + 1 - k) return true;
  // the changes, 32 at a time
  uint32_t carry = 0xFFFFFFFFu, zprev = 0xFFFFFFFFu, mr = 0, rr = 0;
  const uint32_t rem0 = kRiceIdxBits * R;
  // every value staged (the same on every lane): one shared load per change, no range checks
  // (the rare indices checked above make exactly R changes rare)
  const bool staged = PRE > 0 && M <= 32u * PRE && R <= 32;
  for (uint32_t b0 = 0; b0 < k; b0 += 32) {
    const uint32_t i = b0 + lane;
    const bool in = i < k;
    const uint32_t z = in ? ent[i] : 0u;
    uint32_t zp = __shfl_up_sync(kFull, z, 1);
    if (lane == 0) zp = zprev;
    zprev = __shfl_sync(kFull, z, 31);
    const uint32_t g = in ? ((z - zp - 1) << K) | field(rem0 + K * i, K) : 0u;
    const bool isR = in && ((cls[i >> 5] >> (i & 31)) & 1u);
    const uint32_t bR = __ballot_sync(kFull, isR), bM = __ballot_sync(kFull, in && !isR);
    uint32_t v = 0;
    if (staged) {
      if (in) v = sv[isR ? 128u + rr + __popc(bR & lt) : mr + __popc(bM & lt)];
    } else if (isR) {
      const uint32_t r = rr + __popc(bR & lt);
      if (PRE > 0 && r < 32) v = sv[128 + r];
      else if (r < R) v = rvals[r];
      else bad = true;
    } else if (in) {
      const uint32_t m = mr + __popc(bM & lt);
      if (PRE > 0 && m < 32u * PRE) v = sv[m];
      else if (m < M) v = mant_at(mbytes, s0, m);
      else bad = true;
    }
    rr += __popc(bR);
    mr += __popc(bM);
    if (in && g == 0) bad = true;
    __syncwarp();   // every lane has read its zero offset before the entries replace them
    const uint32_t p = carry + warp_incl_scan(g);
    carry = __shfl_sync(kFull, p, 31);
    if (in) {
      if (!ow && (isR ? (v & kSignExp) == 0 : v == 0)) bad = true;
      if (p >= L) bad = true;
      if (!bad) ent[i] = (isR ? kEntRare : 0u) | (p << 16) | v;
    }
  }
  return __any_sync(kFull, bad);
}

// Asks L2 for the 128-byte line holding p when p lies before end (a hint: nothing waits for
// it, and nothing is asked past the end of the payload).
__device__ __forceinline__ void prefetch_l2_before(const uint8_t* p, const uint8_t* end) {
  if (p < end) asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// The payload bytes of the chunk after this one in a warp's range follow this chunk's bytes in
// each section: ask L2 for their first lines (4 of the position section, 2 of the M stream, 1
// each of the R and X streams) while this chunk is decoded.
__device__ __forceinline__ void prefetch_next_payload(const uint8_t* pos_next,
                                                      const uint8_t* m_next,
                                                      const uint8_t* r_next,
                                                      const uint8_t* x_next, const uint8_t* end) {
  const int lane = threadIdx.x & 31;
  if (lane < 4) prefetch_l2_before(pos_next + 128 * lane, end);
  else if (lane < 6) prefetch_l2_before(m_next + 128 * (lane - 4), end);
  else if (lane == 6) prefetch_l2_before(r_next, end);
  else if (lane == 7) prefetch_l2_before(x_next, end);
}

// Listing a chunk for the bitmap kernel through a per-warp buffer of 32 entries in shared
// memory: every 32 entries (and at the end) the warp reserves their places with one atomic
// instead of one per chunk (all chunks of a call meet on the one counter).  Entry i is the
// chunk's global index in list[i] and its tensor in list_job[i], so that the bitmap kernel,
// whose warps take scattered entries, needs no search of the tensor table.  Both are called by
// the whole warp.
__device__ __forceinline__ void list_flush(uint2* wbuf, uint32_t& nbuf,
                                           uint32_t* __restrict__ list_count,
                                           uint32_t* __restrict__ list,
                                           uint32_t* __restrict__ list_job) {
  const int lane = threadIdx.x & 31;
  if (nbuf == 0) return;
  __syncwarp();
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(list_count, nbuf);
  base = __shfl_sync(kFull, base, 0);
  if ((uint32_t)lane < nbuf) {
    const uint2 e = wbuf[lane];
    list[base + lane] = e.x;
    list_job[base + lane] = e.y;
  }
  __syncwarp();
  nbuf = 0;
}
__device__ __forceinline__ void list_append(uint2* wbuf, uint32_t& nbuf, uint64_t g, uint32_t j,
                                            uint32_t* __restrict__ list_count,
                                            uint32_t* __restrict__ list,
                                            uint32_t* __restrict__ list_job) {
  if ((threadIdx.x & 31) == 0) wbuf[nbuf] = make_uint2((uint32_t)g, j);
  if (++nbuf == 32) list_flush(wbuf, nbuf, list_count, list, list_job);
}

// Entry i of a u16 delta list.  Versions 1 and 2 place every list at an even offset; after an
// odd-length compact block of version 3 one may start at an odd offset.
template <bool V3>
__device__ __forceinline__ uint32_t list_entry(const uint8_t* __restrict__ list, uint32_t i) {
  if (V3) return load_u16(list + 2 * i);
  return reinterpret_cast<const uint16_t*>(list)[i];
}

// One warp per chunk of every tensor whose scan status is BD_OK, each warp taking a contiguous
// range of chunks.  A chunk whose two position blocks are delta lists is decoded and checked
// in full into shared memory (positions from the prefix sums of the deltas, 7-bit values from
// the mantissa stream at bit 7*(M prefix + i), 16-bit values from the rare stream; a position
// in both classes, a zero delta after the first, a position past the chunk, a zero mantissa
// value or a rare value without a sign or exponent bit marks the chunk malformed).  A
// well-formed chunk is then XORed into `out` by one 32-bit atomic XOR per change, performed
// in L2 without a reply, and read back through L2 for its checksum terms.  The chunk is
// prefetched into L2 before the decode starts, so that the atomics and the read-back find it
// there (prefetching a later chunk instead thrashes L2 and was much slower).  Chunks with a
// bitmap block are listed for apply_dense, which also adds their checksum terms.
// The version-1/2 build runs at three blocks per SM (75 registers; four measured no better), the
// general build at four (64 registers, no spills: 6% faster on overwrite payloads, whose apply
// waits on a read of each changed element; version 3 the same or up to 3% faster, version 4
// the same -- its decode is bound by instruction issue).
template <bool V3>
__global__ void __launch_bounds__(kThreads, V3 ? 4 : 3)
k_apply_chunks(const DJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
               const uint64_t* __restrict__ tile_start, uint32_t k, uint64_t total_chunks,
               const uint4* __restrict__ loc, const TileSum* __restrict__ tile_pre,
               JobInfo* __restrict__ info, uint32_t* __restrict__ list_count,
               uint32_t* __restrict__ list, uint32_t* __restrict__ list_job,
               uint8_t* __restrict__ ck_base) {
  if ((list_count[kFlagV3Word] != 0) != V3) return;   // the other build runs this call
  __shared__ uint32_t s_ent[kWarps][kEntMax];       // pos << 16 | XOR value
  // mantissa-only positions (512 B); in the general build also a version-4 staging area
  __shared__ uint4 s_bits[kWarps][V3 ? kRiceWords / 4 : kChunk / 128];
  __shared__ uint2 s_lbuf[kWarps][32];   // chunks to list (index, tensor), not yet appended
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t* ent = s_ent[w];
  uint32_t* bits = reinterpret_cast<uint32_t*>(s_bits[w]);
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  uint32_t j = kNone, cur = kNone, nbuf = 0;
  uint64_t ck = 0;
  uint64_t g_begin, g_end;
  warp_range(total_chunks, gwarp, nwarps, g_begin, g_end);
  for (uint64_t g = g_begin; g < g_end; g++) {
    j = advance_job(chunk_start, k, j, g);
    const JobInfo& I = info[j];
    if (I.status != BD_OK) continue;
    if (j != cur) {
      if (cur != kNone) flush_ck(ck_base, cur, gwarp, ck);
      cur = j;
      ck = 0;
    }
    const DJob& J = jobs[j];
    const uint64_t n = J.n, c = g - chunk_start[j], e0 = c * kChunk;
    const uint32_t L = (n - e0) < kChunk ? (uint32_t)(n - e0) : kChunk;
    const uint32_t B = (L + 7) >> 3;
    const uint8_t* __restrict__ payload = J.payload;
    // the chunk's prefix sums are requested with its count word, not after it (one dependent
    // round trip fewer: 0.5-1% on the dense apply)
    const TileSum pre = tile_pre[tile_start[j] + c / kTileChunks];
    const uint4 lc = loc[g];
    const ChunkCount cc = parse_count(reinterpret_cast<const uint32_t*>(
        payload + count_table_offset(info[j].r_start, J.nchunks))[c], V3 ? I.version : 1u);
    const uint32_t M = cc.M, R = cc.R;
    if (!cc.compact && (2 * M >= B || 2 * R >= B)) {
      list_append(s_lbuf[w], nbuf, g, j, list_count, list, list_job);
      continue;
    }
    if (e0 + kChunk <= n) prefetch_chunk_l2(J.out + e0);   // in L2 by the time it is read

    if (M + R > 0) {
      const uint64_t Pex = pre.p + lc.x, Mex = pre.m + lc.y, Rex = pre.r + lc.z;
      // The rare values are 2-byte aligned (the R stream starts at the even offset
      // header + 4C); the delta lists are too in versions 1 and 2, but may start at an odd
      // offset after a compact block of version 3, hence the alignment-checking loads.
      const uint8_t* mlist = payload + I.p_start + Pex;
      const uint8_t* rlist = mlist + 2 * M;
      const uint16_t* rvals = reinterpret_cast<const uint16_t*>(payload + I.r_start) + Rex;
      const uint64_t mbit0 = 7 * Mex;
      const uint8_t* mbytes = payload + I.m_start + (mbit0 >> 3);
      const uint32_t s0 = (uint32_t)(mbit0 & 7);
      const bool both = M > 0 && R > 0;
      const bool ow = V3 && (I.flags & kFlagOverwrite) != 0;
      bool bad = false;
      if (V3 && cc.rice) {
        bad = decode_rice<4>(mlist, cc.nb, cc.K, mbytes, s0, rvals, M, R, L, ow, bits, ent);
      } else if (V3 && cc.compact) {
        bad = decode_compact<4>(mlist,
                             reinterpret_cast<const uint16_t*>(payload + I.x_start) + pre.e + lc.w,
                             cc.E, mbytes, s0, rvals, M, R, L, ow, ent);
      } else {
        if (both) s_bits[w][lane] = make_uint4(0, 0, 0, 0);
        // the payload of the first 128 mantissa-only and 32 rare changes, all requested before
        // the first is used (one round trip for most chunks instead of one per 32 changes:
        // -3% on the dense apply; in apply_incr, at 64 registers, the same spilled and was
        // much slower)
        uint32_t pd[4], pv[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
          const uint32_t i = 32 * q + lane;
          pd[q] = 0;
          pv[q] = 0;
          if (i < M) {
            pd[q] = list_entry<V3>(mlist, i);
            const uint32_t bit = s0 + 7 * i;
            pv[q] = mbytes[bit >> 3];
            if ((bit & 7) > 1) pv[q] |= (uint32_t)mbytes[(bit >> 3) + 1] << 8;
          }
        }
        uint32_t rd0 = 0, rv0 = 0;
        if ((uint32_t)lane < R) {
          rd0 = list_entry<V3>(rlist, lane);
          rv0 = rvals[lane];
        }
        __syncwarp();
        uint32_t carry = 0;
        auto m_batch = [&](uint32_t i, uint32_t d, uint32_t raw) {
          const bool in = i < M;
          if (in && i > 0 && d == 0) bad = true;
          const uint32_t p = carry + warp_incl_scan(d);
          carry = __shfl_sync(kFull, p, 31);
          if (in) {
            const uint32_t v = (raw >> ((s0 + 7 * i) & 7)) & kMant;
            if (p >= L || (!ow && v == 0)) {
              bad = true;
            } else {
              ent[i] = (p << 16) | v;
              if (both) atomicOr(&bits[p >> 5], 1u << (p & 31));
            }
          }
        };
#pragma unroll
        for (int q = 0; q < 4; q++) {
          if (32u * q >= M) break;
          m_batch(32 * q + lane, pd[q], pv[q]);
        }
        for (uint32_t b0 = 128; b0 < M; b0 += 32) {
          const uint32_t i = b0 + lane;
          uint32_t d = 0, raw = 0;
          if (i < M) {
            d = list_entry<V3>(mlist, i);
            const uint32_t bit = s0 + 7 * i;
            raw = mbytes[bit >> 3];
            if ((bit & 7) > 1) raw |= (uint32_t)mbytes[(bit >> 3) + 1] << 8;
          }
          m_batch(i, d, raw);
        }
        __syncwarp();
        carry = 0;
        for (uint32_t b0 = 0; b0 < R; b0 += 32) {
          const uint32_t i = b0 + lane;
          const bool in = i < R;
          uint32_t d = rd0, v = rv0;
          if (b0 > 0) {
            d = in ? list_entry<V3>(rlist, i) : 0u;
            v = in ? (uint32_t)rvals[i] : 0u;
          }
          if (in && i > 0 && d == 0) bad = true;
          const uint32_t p = carry + warp_incl_scan(d);
          carry = __shfl_sync(kFull, p, 31);
          if (in) {
            if (p >= L || (!ow && (v & kSignExp) == 0)) bad = true;
            else if (both && ((bits[p >> 5] >> (p & 31)) & 1u)) bad = true;
            else ent[M + i] = (V3 ? kEntRare : 0u) | (p << 16) | v;
          }
        }
      }
      if (__any_sync(kFull, bad)) {
        if (lane == 0) record_status(&info[j].chunk_err, BD_ERR_FORMAT);
        __syncwarp();
        continue;
      }
      __syncwarp();
      uint16_t* base = J.out + e0;   // 4-byte aligned: out is 16-byte aligned, e0 % 4096 == 0
      for (uint32_t i = lane; i < M + R; i += 32) {
        const uint32_t e = ent[i], p = V3 ? ent_pos(e) : e >> 16;
        uint32_t x = e & 0xFFFFu;
        if (ow) {   // the new value or mantissa, XORed in against the element's current bits
          const uint32_t now = ld_l2_u16(base + p);
          x = (e & kEntRare) ? (now ^ x) : ((now & kMant) ^ x);
        }
        if (x) atomicXor(reinterpret_cast<unsigned int*>(base + (p & ~1u)), x << (16 * (p & 1)));
      }
      // every lane's atomics are performed before any lane reads the chunk back
      __threadfence_block();
      __syncwarp();
    }
    if (e0 + kChunk <= n) ck += hash_chunk<true>(J.out, n, e0);
    else ck += hash_chunk<false>(J.out, n, e0);
  }
  list_flush(s_lbuf[w], nbuf, list_count, list, list_job);
  if (cur != kNone) flush_ck(ck_base, cur, gwarp, ck);
}

// Incremental verification, one warp per chunk (each warp a contiguous range of chunks) of
// every tensor whose scan status is BD_OK.  A chunk whose two position blocks are delta lists
// is decoded and checked exactly as in apply_chunks; a well-formed chunk then applies each
// change with a 64-bit atomic XOR that returns the word before it, and adds the word's
// checksum term after the change minus its term before (elements past n count as zero).
// Changes to the same word are serialised by the atomics, so their terms telescope to the
// word's final term minus its original one.  Nothing else of the chunk is read.  Chunks with
// a bitmap block are listed for apply_dense<true>.
template <bool V3, bool OW>
__global__ void __launch_bounds__(kThreads, 4)
k_apply_incr(const DJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
             const uint64_t* __restrict__ tile_start, uint32_t k, uint64_t total_chunks,
             const uint4* __restrict__ loc, const TileSum* __restrict__ tile_pre,
             JobInfo* __restrict__ info, uint32_t* __restrict__ list_count,
             uint32_t* __restrict__ list, uint32_t* __restrict__ list_job,
             uint8_t* __restrict__ ck_base) {
  // another build runs this call
  if ((list_count[kFlagV3Word] != 0) != V3 || (list_count[kFlagOwWord] != 0) != OW) return;
  __shared__ uint32_t s_ent[kWarps][kEntMax];       // pos << 16 | XOR value
  // mantissa-only positions (512 B); in the general build also a version-4 staging area
  __shared__ uint4 s_bits[kWarps][V3 ? kRiceWords / 4 : kChunk / 128];
  __shared__ uint2 s_lbuf[kWarps][32];   // chunks to list (index, tensor), not yet appended
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t* ent = s_ent[w];
  uint32_t* bits = reinterpret_cast<uint32_t*>(s_bits[w]);
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  uint32_t j = kNone, cur = kNone, nbuf = 0;
  uint64_t ck = 0;
  uint64_t g_begin, g_end;
  warp_range(total_chunks, gwarp, nwarps, g_begin, g_end);
  for (uint64_t g = g_begin; g < g_end; g++) {
    j = advance_job(chunk_start, k, j, g);
    const JobInfo& I = info[j];
    if (I.status != BD_OK) continue;
    if (j != cur) {
      if (cur != kNone) flush_ck(ck_base, cur, gwarp, ck);
      cur = j;
      ck = 0;
    }
    const DJob& J = jobs[j];
    const uint64_t n = J.n, c = g - chunk_start[j], e0 = c * kChunk;
    const uint32_t L = (n - e0) < kChunk ? (uint32_t)(n - e0) : kChunk;
    const uint32_t B = (L + 7) >> 3;
    const uint8_t* __restrict__ payload = J.payload;
    const ChunkCount cc = parse_count(reinterpret_cast<const uint32_t*>(
        payload + count_table_offset(info[j].r_start, J.nchunks))[c], V3 ? I.version : 1u);
    const uint32_t M = cc.M, R = cc.R;
    if (!cc.compact && (2 * M >= B || 2 * R >= B)) {
      list_append(s_lbuf[w], nbuf, g, j, list_count, list, list_job);
      continue;
    }
    if (M + R == 0) continue;
    const TileSum pre = tile_pre[tile_start[j] + c / kTileChunks];
    const uint4 lc = loc[g];
    const uint64_t Pex = pre.p + lc.x, Mex = pre.m + lc.y, Rex = pre.r + lc.z;
    // the rare values are 2-byte aligned, the delta lists not always (see apply_chunks)
    const uint8_t* mlist = payload + I.p_start + Pex;
    const uint8_t* rlist = mlist + 2 * M;
    const uint16_t* rvals = reinterpret_cast<const uint16_t*>(payload + I.r_start) + Rex;
    const uint64_t mbit0 = 7 * Mex;
    const uint8_t* mbytes = payload + I.m_start + (mbit0 >> 3);
    const uint32_t s0 = (uint32_t)(mbit0 & 7);
    prefetch_next_payload(mlist + chunk_pos_bytes(cc, B),
                          payload + I.m_start + ((7 * (Mex + M)) >> 3),
                          reinterpret_cast<const uint8_t*>(rvals + R),
                          payload + I.x_start + 2 * (pre.e + lc.w + cc.E), payload + J.size);
    const bool both = M > 0 && R > 0;
    const bool ow = OW && (I.flags & kFlagOverwrite) != 0;
    bool bad = false;
    if (V3 && cc.rice) {
      bad = decode_rice<0>(mlist, cc.nb, cc.K, mbytes, s0, rvals, M, R, L, ow, bits,
                                    ent);
    } else if (V3 && cc.compact) {
      bad = decode_compact<0>(mlist,
                           reinterpret_cast<const uint16_t*>(payload + I.x_start) + pre.e + lc.w,
                           cc.E, mbytes, s0, rvals, M, R, L, ow, ent);
    } else {
      if (both) s_bits[w][lane] = make_uint4(0, 0, 0, 0);
      __syncwarp();
      uint32_t carry = 0;
      for (uint32_t b0 = 0; b0 < M; b0 += 32) {
        const uint32_t i = b0 + lane;
        const bool in = i < M;
        const uint32_t d = in ? list_entry<V3>(mlist, i) : 0u;
        if (in && i > 0 && d == 0) bad = true;
        const uint32_t p = carry + warp_incl_scan(d);
        carry = __shfl_sync(kFull, p, 31);
        if (in) {
          const uint32_t bit = s0 + 7 * i, sh = bit & 7;
          uint32_t v = (uint32_t)mbytes[bit >> 3] >> sh;
          if (sh > 1) v |= (uint32_t)mbytes[(bit >> 3) + 1] << (8 - sh);
          v &= kMant;
          if (p >= L || (!ow && v == 0)) {
            bad = true;
          } else {
            ent[i] = (p << 16) | v;
            if (both) atomicOr(&bits[p >> 5], 1u << (p & 31));
          }
        }
      }
      __syncwarp();
      carry = 0;
      for (uint32_t b0 = 0; b0 < R; b0 += 32) {
        const uint32_t i = b0 + lane;
        const bool in = i < R;
        const uint32_t d = in ? list_entry<V3>(rlist, i) : 0u;
        if (in && i > 0 && d == 0) bad = true;
        const uint32_t p = carry + warp_incl_scan(d);
        carry = __shfl_sync(kFull, p, 31);
        if (in) {
          const uint32_t v = rvals[i];
          if (p >= L || (!ow && (v & kSignExp) == 0)) bad = true;
          else if (both && ((bits[p >> 5] >> (p & 31)) & 1u)) bad = true;
          else ent[M + i] = (V3 ? kEntRare : 0u) | (p << 16) | v;
        }
      }
    }
    if (__any_sync(kFull, bad)) {
      if (lane == 0) record_status(&info[j].chunk_err, BD_ERR_FORMAT);
      __syncwarp();
      continue;
    }
    __syncwarp();
    // 8-byte aligned: out is 16-byte aligned and e0 % 4096 == 0.  The last word of a tensor
    // whose n is not a multiple of 4 also covers up to 3 values past n: they are XORed with
    // zero (the atomic leaves them as they are) and count as zero in the checksum terms.
    unsigned long long* base = reinterpret_cast<unsigned long long*>(J.out + e0);
    const uint64_t wlast = (n - 1) >> 2;
    const uint32_t in_last = (uint32_t)(n - 4 * wlast);   // values of the last word, 1..4
    const uint64_t last_mask = in_last == 4 ? ~0ull : ((1ull << (16 * in_last)) - 1);
    // kB entries per lane per round: their atomics are issued back to back, then the terms
    // (3 in the general build, whose compact decoder leaves fewer registers: with 4 it
    // spilled at 64 registers, and 3 blocks per SM instead was slower; 2 in the build that
    // also applies overwrites, which spilled with 3)
    constexpr int kB = V3 ? (OW ? 2 : 3) : 4;
    for (uint32_t r0 = 0; r0 < M + R; r0 += 32 * kB) {
      uint64_t before[kB], dd[kB];
      uint32_t pp[kB];
      if (!ow) {
#pragma unroll
        for (int u = 0; u < kB; u++) {
          const uint32_t i = r0 + 32 * u + lane;
          pp[u] = 0xFFFFFFFFu;
          if (i < M + R) {
            const uint32_t e = ent[i], p = V3 ? ent_pos(e) : e >> 16;
            pp[u] = p;
            dd[u] = (uint64_t)(e & 0xFFFFu) << (16 * (p & 3));
            before[u] = atomicXor(base + (p >> 2), (unsigned long long)dd[u]);
          }
        }
      } else {
        // overwrite: the new value or mantissa, XORed in against the element's current bits
        // (the round's reads are issued before the first is used); an element that already
        // holds its new bits is left alone.  The word after the change is formed below from
        // the word before it, which holds this element's bits as read.
        uint32_t now[kB];
#pragma unroll
        for (int u = 0; u < kB; u++) {
          const uint32_t i = r0 + 32 * u + lane;
          pp[u] = 0xFFFFFFFFu;
          if (i < M + R) {
            pp[u] = ent_pos(ent[i]);
            now[u] = ld_l2_u16(J.out + e0 + pp[u]);
          }
        }
#pragma unroll
        for (int u = 0; u < kB; u++) {
          if (pp[u] != 0xFFFFFFFFu) {
            const uint32_t e = ent[r0 + 32 * u + lane], t = e & 0xFFFFu;
            const uint32_t x = (e & kEntRare) ? (now[u] ^ t) : ((now[u] & kMant) ^ t);
            if (x == 0) pp[u] = 0xFFFFFFFFu;
            else before[u] = atomicXor(base + (pp[u] >> 2),
                                       (unsigned long long)x << (16 * (pp[u] & 3)));
          }
        }
#pragma unroll
        for (int u = 0; u < kB; u++) {
          if (pp[u] != 0xFFFFFFFFu) {
            const uint32_t e = ent[r0 + 32 * u + lane], t = e & 0xFFFFu, sh = 16 * (pp[u] & 3);
            const uint32_t was = (uint32_t)(before[u] >> sh) & 0xFFFFu;
            const uint32_t to = (e & kEntRare) ? t : ((was & kSignExp) | t);
            dd[u] = (uint64_t)(was ^ to) << sh;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kB; u++) {
        if (pp[u] != 0xFFFFFFFFu) {
          uint64_t b = before[u], a = before[u] ^ dd[u];
          const uint64_t wj = (e0 >> 2) + (pp[u] >> 2);
          if (wj == wlast) {
            b &= last_mask;
            a &= last_mask;
          }
          const uint64_t key = (wj + 1) * kGamma;
          ck += mix64(a ^ key) - mix64(b ^ key);
        }
      }
    }
    __syncwarp();
  }
  list_flush(s_lbuf[w], nbuf, list_count, list, list_job);
  if (cur != kNone) flush_ck(ck_base, cur, gwarp, ck);
}

// ------------------------------------------------------------------------ apply_bitmap

// Little-endian u32 at the 4-byte aligned address p; bytes at or past `end` read as zero
// (nothing past the payload is read).
__device__ __forceinline__ uint32_t ld_u32_upto(const uint8_t* p, const uint8_t* end) {
  if (p + 4 <= end) return __ldg(reinterpret_cast<const uint32_t*>(p));
  uint32_t v = 0;
  for (int i = 0; i < 4; i++)
    if (p + i < end) v |= (uint32_t)p[i] << (8 * i);
  return v;
}

// The value v repeated in each of nine 7-bit fields (bits 7f .. 7f+6, f = 0..8).
constexpr uint64_t fields9(uint64_t v) {
  uint64_t r = 0;
  for (int f = 0; f < 9; f++) r |= v << (7 * f);
  return r;
}
constexpr uint64_t kField6 = fields9(0x3F), kField7 = fields9(0x40);

// 8 BF16 values at the 16-byte aligned p (a plain load: p is written by this kernel).
__device__ __forceinline__ uint4 ld_plain(const uint16_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}
// Checksum terms of a group of 8 values whose first word has key `key` (both words below n).
__device__ __forceinline__ uint64_t hash_pair(uint4 v, uint64_t key) {
  return mix64(((uint64_t)v.x | ((uint64_t)v.y << 32)) ^ key) +
         mix64(((uint64_t)v.z | ((uint64_t)v.w << 32)) ^ (key + kGamma));
}

// Per-warp shared state of apply_bitmap: the chunk's two position blocks as bitmaps (a block
// that is a bitmap in the payload is copied as the aligned words covering it, read from byte
// offset `off`; a delta list is decoded into a bitmap at offset 0).
struct BitmapSmem {
  uint32_t w[2][130];   // [0]: mantissa-only, [1]: rare
  uint32_t mw[902];     // the chunk's M-stream bytes, as the aligned words covering them
};

// Copies the M-stream bits of a chunk's M values (7 bits each, stream bit 7*Mex on) into
// sm->mw; returns the buffer bit of the chunk's first value bit.
__device__ __forceinline__ uint32_t stage_mstream(BitmapSmem* sm, const uint8_t* mstream,
                                                  uint64_t Mex, uint32_t M, const uint8_t* end) {
  const int lane = threadIdx.x & 31;
  const uint8_t* p = mstream + ((7 * Mex) >> 3);
  const uint8_t* a = reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(p) & ~(uintptr_t)3);
  const uint32_t first = (uint32_t)(p - a) * 8 + (uint32_t)((7 * Mex) & 7);
  const uint32_t nw = (first + 7 * M + 31) / 32;   // <= 898
  for (uint32_t i = lane; i < nw + 2; i += 32) sm->mw[i] = i < nw ? ld_u32_upto(a + 4 * i, end) : 0u;
  return first;
}

// The 64 buffer bits from buffer bit `bit` on.
__device__ __forceinline__ uint64_t mw_bits64(const BitmapSmem* sm, uint32_t bit) {
  const uint32_t w = bit >> 5, sh = bit & 31;
  const uint64_t lo = (uint64_t)sm->mw[w] | ((uint64_t)sm->mw[w + 1] << 32);
  return sh ? (lo >> sh) | ((uint64_t)sm->mw[w + 2] << (64 - sh)) : lo;
}

// Byte q (0 <= q < 512) of the class-c bitmap; bytes past the chunk's B read as zero.
__device__ __forceinline__ uint32_t bm_byte(const BitmapSmem* sm, int c, uint32_t off,
                                            uint32_t q, uint32_t B) {
  return q < B ? reinterpret_cast<const uint8_t*>(sm->w[c])[off + q] : 0u;
}
// The same for a full chunk (B = 512).
__device__ __forceinline__ uint32_t bm_byte_full(const BitmapSmem* sm, int c, uint32_t off,
                                                 uint32_t q) {
  return reinterpret_cast<const uint8_t*>(sm->w[c])[off + q];
}
// Word i of the class-c bitmap (positions 32i .. 32i+31), bytes past B as zero.
__device__ __forceinline__ uint32_t bm_word(const BitmapSmem* sm, int c, uint32_t off,
                                            uint32_t i, uint32_t B) {
  const uint32_t a = sm->w[c][(off >> 2) + i], b = sm->w[c][(off >> 2) + i + 1];
  uint32_t v = (off & 3) ? __funnelshift_r(a, b, 8 * (off & 3)) : a;
  if (4 * i + 4 > B) v &= 4 * i >= B ? 0u : (0xFFFFFFFFu >> (8 * (4 * i + 4 - B)));
  return v;
}

// Reads one position block of a chunk into a bitmap of sm: a delta list of k entries at blk
// (deltas of at least 1 after the first, positions below L) or a B-byte bitmap at blk.
// Returns the byte offset to read it from; sets bad for a malformed list.
__device__ __forceinline__ uint32_t load_block(BitmapSmem* sm, int c, const uint8_t* blk,
                                               uint32_t k, uint32_t B, uint32_t L, bool list,
                                               const uint8_t* end, bool& bad) {
  const int lane = threadIdx.x & 31;
  uint32_t* w = sm->w[c];
  if (!list) {
    const uint8_t* a = reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(blk) & ~(uintptr_t)3);
    const uint32_t off = (uint32_t)(blk - a);
    const uint32_t nw = (off + B + 3) / 4;
    for (uint32_t i = lane; i < nw; i += 32) w[i] = ld_u32_upto(a + 4 * i, end);
    if ((uint32_t)lane < 130 - nw && nw + lane < 130) w[nw + lane] = 0;   // guard words
    return off;
  }
  for (uint32_t i = lane; i < 130; i += 32) w[i] = 0;
  __syncwarp();
  uint32_t carry = 0;
  for (uint32_t b0 = 0; b0 < k; b0 += 32) {
    const uint32_t i = b0 + lane;
    const bool in = i < k;
    const uint32_t d = in ? load_u16(blk + 2 * i) : 0u;
    if (in && i > 0 && d == 0) bad = true;
    const uint32_t p = carry + warp_incl_scan(d);
    carry = __shfl_sync(kFull, p, 31);
    if (in) {
      if (p >= L) bad = true;
      else atomicOr(&w[p >> 5], 1u << (p & 31));
    }
  }
  return 0;
}

// The values of one 8-element group (XOR masks or overwrite targets) with class masks bm, br:
// its mantissa-only values are the next popc(bm) of the M stream (from buffer bit `mbit`),
// spread to bytes and permuted into their elements' places by the selectors of bm; its rare
// values are the next popc(br) of the R stream from rank r.
__device__ __forceinline__ uint4 group_values(const BitmapSmem* sm, const uint4* s_esel,
                                              uint32_t bm, uint32_t br, uint32_t mbit,
                                              const uint16_t* __restrict__ rstream, uint32_t r) {
  uint4 m = make_uint4(0, 0, 0, 0);
  if (bm) {
    const uint64_t win = mw_bits64(sm, mbit);
    const uint32_t a = unpack7x4((uint32_t)win), b = unpack7x4((uint32_t)(win >> 28));
    const uint4 sel = s_esel[bm];
    m = make_uint4(prmt(a, b, sel.x), prmt(a, b, sel.y), prmt(a, b, sel.z), prmt(a, b, sel.w));
  }
  if (br) {
    for (uint32_t b = br; b; b &= b - 1, r++) {   // mostly a single rare change
      const uint32_t i = __ffs(b) - 1;
      const uint32_t v = (uint32_t)rstream[r] << (16 * (i & 1));
      if (i < 2) m.x |= v;
      else if (i < 4) m.y |= v;
      else if (i < 6) m.z |= v;
      else m.w |= v;
    }
  }
  return m;
}

// The apply steps of one checked chunk (elements e0 .. e0 + 4095 of w, clipped at n): step s,
// lane l takes group 32s + l; returns the checksum terms (INCR: new minus old terms of the
// changed groups).  FULL: the whole chunk lies below n -- no bounds on loads, stores and terms,
// and the checksum keys advance by a constant per step.
template <bool FULL, bool INCR>
__device__ __forceinline__ uint64_t bitmap_steps(const BitmapSmem* sm, const uint4* s_esel,
                                                 uint16_t* __restrict__ w, uint64_t e0, uint64_t n,
                                                 uint32_t offM, uint32_t offR, uint32_t B,
                                                 uint32_t mbit0,
                                                 const uint16_t* __restrict__ rstream, bool ow) {
  const int lane = threadIdx.x & 31;
  const uint64_t words = (n + 3) >> 2;
  uint64_t ck = 0;
  uint32_t rM = 0, rR = 0;   // ranks of the values before this step
  uint32_t el = 8 * lane;    // chunk-local element of the lane's group
  uint64_t key = (((e0 + el) >> 2) + 1) * kGamma;   // FULL: key of the group's first word
  uint4 nxt = FULL ? ld_plain(w + el) : load8(w - e0, e0 + el, n);
#pragma unroll 1
  for (uint32_t s = 0; s < 16; s++, el += 256) {
    const uint4 now = nxt;
    if (s < 15) nxt = FULL ? ld_plain(w + el + 256) : load8(w - e0, e0 + el + 256, n);
    const uint32_t q = 32 * s + lane;
    const uint32_t bm = FULL ? bm_byte_full(sm, 0, offM, q) : bm_byte(sm, 0, offM, q, B);
    const uint32_t br = FULL ? bm_byte_full(sm, 1, offR, q) : bm_byte(sm, 1, offR, q, B);
    const uint32_t packed = __popc(bm) | (__popc(br) << 16);
    const uint32_t incl = warp_incl_scan(packed), excl = incl - packed;
    const uint32_t tot = __shfl_sync(kFull, incl, 31);
    uint4 m = group_values(sm, s_esel, bm, br, mbit0 + 7 * (rM + (excl & 0xFFFFu)), rstream,
                           rR + (excl >> 16));
    rM += tot & 0xFFFFu;
    rR += tot >> 16;
    if (ow) m = overwrite_mask(m, now, bm, br);
    const bool ch = (m.x | m.y | m.z | m.w) != 0;
    const uint4 res = make_uint4(now.x ^ m.x, now.y ^ m.y, now.z ^ m.z, now.w ^ m.w);
    const uint64_t e = e0 + el;
    if (FULL) {
      if (ch) *reinterpret_cast<uint4*>(w + el) = res;
      if (!INCR) ck += hash_pair(res, key);
      else if (ch) ck += hash_pair(res, key) - hash_pair(now, key);
      key += 64 * kGamma;
    } else {
      if (ch && e < n) {
        if (e + 8 <= n) *reinterpret_cast<uint4*>(w + el) = res;
        else for (int i = 0; e + i < n; i++) w[el + i] = (uint16_t)elem_of(res, i);
      }
      if (!INCR) ck += group_hash(res, e >> 3, words);
      else if (ch) ck += group_hash(res, e >> 3, words) - group_hash(now, e >> 3, words);
    }
  }
  return ck;
}

// One warp per listed chunk (a chunk with at least one bitmap block; compact chunks never have
// one), each warp taking every nwarps-th entry of the list.  The chunk is checked in full
// first -- the blocks (list deltas, positions below L, bitmap counts equal to M and R, no bit at
// or past L, no position in both classes) and, for an XOR payload, every value (a nonzero
// mantissa mask, a rare mask with a sign or exponent bit) -- and left unwritten when
// malformed.  Then 16 steps of 256 elements, lane l taking the 8-element group 32s + l: the
// ranks of the group's first values come from one warp scan of the two classes' bit counts,
// its mantissa-only values from one 64-bit window of the M stream (spread to bytes and put in
// place by four byte permutes chosen by the group's class mask), its rare values from the R
// stream; the group is XORed (an overwrite payload: its records written in place of the
// fields), stored when it changed, and its checksum terms added (INCR: new minus old terms of
// the changed groups).  The chunk is prefetched into L2 while its payload is checked, and
// each step's group loads are issued one step ahead; the chunk's M-stream bytes are staged in
// shared memory with its blocks.
template <bool INCR>
__global__ void __launch_bounds__(kThreads, 4)
k_apply_bitmap(const DJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
               const uint64_t* __restrict__ tile_start, uint32_t k,
               const uint32_t* __restrict__ list_count, const uint32_t* __restrict__ list,
               const uint32_t* __restrict__ list_job, const uint4* __restrict__ loc,
               const TileSum* __restrict__ tile_pre, JobInfo* __restrict__ info,
               uint8_t* __restrict__ ck_base) {
  __shared__ BitmapSmem s_bm[kWarps];
  __shared__ uint4 s_esel[256];   // expand selectors by class mask
  const int lane = threadIdx.x & 31;
  BitmapSmem* sm = &s_bm[threadIdx.x >> 5];
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  static_assert(kThreads == 256, "one selector entry per thread");
  s_esel[threadIdx.x] = make_uint4(expand_sel(threadIdx.x, 0), expand_sel(threadIdx.x, 1),
                                   expand_sel(threadIdx.x, 2), expand_sel(threadIdx.x, 3));
  __syncthreads();
  const uint32_t listed = *list_count;
  uint32_t cur = kNone;
  uint64_t ck = 0;
  for (uint64_t li = gwarp; li < listed; li += nwarps) {
    const uint64_t g = list[li];
    const uint32_t j = list_job[li];
    const JobInfo& I = info[j];
    if (I.status != BD_OK) continue;
    if (j != cur) {
      if (cur != kNone) flush_ck(ck_base, cur, gwarp, ck);
      cur = j;
      ck = 0;
    }
    const DJob& J = jobs[j];
    const uint64_t n = J.n, c = g - chunk_start[j], e0 = c * kChunk;
    uint16_t* __restrict__ out = J.out;
    if (e0 + kChunk <= n) prefetch_chunk_l2(out + e0);   // in L2 by the time it is read
    const uint32_t L = (n - e0) < kChunk ? (uint32_t)(n - e0) : kChunk;
    const uint32_t B = (L + 7) >> 3;
    const uint8_t* __restrict__ payload = J.payload;
    const uint8_t* end = payload + J.size;
    const TileSum pre = tile_pre[tile_start[j] + c / kTileChunks];
    const uint4 lc = loc[g];
    const ChunkCount cc = parse_count(reinterpret_cast<const uint32_t*>(
        payload + count_table_offset(I.r_start, J.nchunks))[c], I.version);
    const uint32_t M = cc.M, R = cc.R;
    const uint64_t Pex = pre.p + lc.x, Mex = pre.m + lc.y, Rex = pre.r + lc.z;
    const bool listM = 2 * M < B, listR = 2 * R < B;
    const uint8_t* mblk = payload + I.p_start + Pex;
    const uint8_t* rblk = mblk + block_bytes(M, B);
    const uint8_t* mstream = payload + I.m_start;
    const uint16_t* rstream = reinterpret_cast<const uint16_t*>(payload + I.r_start) + Rex;
    const bool ow = (I.flags & kFlagOverwrite) != 0;

    // ---- check the whole chunk before anything is written
    bool bad = cc.compact;   // (never listed)
    const uint32_t offM = load_block(sm, 0, mblk, M, B, L, listM, end, bad);
    const uint32_t offR = load_block(sm, 1, rblk, R, B, L, listR, end, bad);
    const uint32_t mbit0 = stage_mstream(sm, mstream, Mex, M, end);
    __syncwarp();
    uint32_t cM = 0, cR = 0;
    for (uint32_t i = lane; 4 * i < B; i += 32) {
      const uint32_t wM = bm_word(sm, 0, offM, i, B), wR = bm_word(sm, 1, offR, i, B);
      const uint32_t valid = 32 * i + 32 <= L ? 0xFFFFFFFFu : (0xFFFFFFFFu >> (32 * i + 32 - L));
      if ((wM & wR) != 0 || ((wM | wR) & ~valid) != 0) bad = true;
      cM += __popc(wM);
      cR += __popc(wR);
    }
    cM = __reduce_add_sync(kFull, cM);
    cR = __reduce_add_sync(kFull, cR);
    if (cM != M || cR != R) bad = true;
    if (!ow) {
      // every 7-bit mantissa mask nonzero: nine fields per 63-bit window, field f nonzero
      // exactly when bit 6 of ((f & 0x3F) + 0x3F) | f is set (the add cannot carry out of it)
      for (uint32_t v0 = 9 * lane; v0 < M; v0 += 9 * 32) {
        const uint32_t nf = M - v0 < 9 ? M - v0 : 9;
        const uint64_t x = mw_bits64(sm, mbit0 + 7 * v0);
        const uint64_t keep = kField7 & ((1ull << (7 * nf)) - 1);
        if (((((x & kField6) + kField6) | x) & keep) != keep) bad = true;
      }
      for (uint32_t i = lane; i < R; i += 32)
        if ((rstream[i] & kSignExp) == 0) bad = true;
    }
    if (__any_sync(kFull, bad)) {
      if (lane == 0) record_status(&info[j].chunk_err, BD_ERR_FORMAT);
      __syncwarp();
      continue;
    }

    // ---- apply, 16 steps of 256 elements
    if (e0 + kChunk <= n)
      ck += bitmap_steps<true, INCR>(sm, s_esel, out + e0, e0, n, offM, offR, B, mbit0, rstream, ow);
    else
      ck += bitmap_steps<false, INCR>(sm, s_esel, out + e0, e0, n, offM, offR, B, mbit0, rstream, ow);
  }
  if (cur != kNone) flush_ck(ck_base, cur, gwarp, ck);
}

// Out-of-place apply: copies old to out (warp per chunk) for the tensors with out != old.
__global__ void __launch_bounds__(kThreads)
k_copy_jobs(const DJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start, uint32_t k,
            uint64_t total_chunks, const JobInfo* __restrict__ info) {
  const int lane = threadIdx.x & 31;
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  uint32_t j = 0xFFFFFFFFu;
  for (uint64_t g = gwarp; g < total_chunks; g += nwarps) {
    j = advance_job(chunk_start, k, j, g);
    const DJob& J = jobs[j];
    if (J.out == J.old || info[j].status != BD_OK) continue;
    const uint64_t n = J.n, e0 = (g - chunk_start[j]) * kChunk;
    for (uint64_t e = e0 + 8 * lane; e < e0 + kChunk && e < n; e += 256) {
      if (e + 8 <= n) *reinterpret_cast<uint4*>(J.out + e) = __ldcs(reinterpret_cast<const uint4*>(J.old + e));
      else for (uint64_t i = e; i < n; i++) J.out[i] = J.old[i];
    }
  }
}

__global__ void k_apply_finish(const DJob* __restrict__ jobs, uint32_t k,
                               JobInfo* __restrict__ info, const uint8_t* __restrict__ ck_base,
                               int32_t* __restrict__ status_all) {
  const uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= k) return;
  const DJob& J = jobs[j];
  const JobInfo I = info[j];
  int32_t st = I.status;
  if (st == BD_OK && I.chunk_err != 0) st = BD_ERR_FORMAT;
  if (st == BD_OK) {
    const uint64_t mb = (7 * I.sum_m + 7) / 8;
    if (mb > 0) {
      const uint32_t used = (uint32_t)(7 * I.sum_m - 8 * (mb - 1));  // 1..8 bits
      const uint32_t last = J.payload[I.m_start + mb - 1];
      if (used < 8 && (last >> used) != 0) st = BD_ERR_FORMAT;
    }
  }
  if (st == BD_OK) {
    // incremental verification starts from the checksum of out before the call; the slots
    // then hold the new-minus-old terms of the changed words
    const uint64_t* ck = reinterpret_cast<const uint64_t*>(ck_base + j * kCkBytes);
    uint64_t sum = J.d_ck_old ? *J.d_ck_old : 0;
    for (int s = 0; s < kCkSlots; s++) sum += ck[s * kCkStride];
    if (J.d_ck_out) *J.d_ck_out = sum;
    if (sum != *J.d_expected) st = BD_ERR_CHECKSUM;
  }
  info[j].status = st;
  if (J.d_status) *J.d_status = st;
  if (status_all) atomicMax(reinterpret_cast<int*>(status_all), st);
}

template <typename K>
int blocks_per_sm(K kernel) {
  int v = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, kThreads, 0) != cudaSuccess || v < 1)
    v = 1;
  return v;
}

}  // namespace

// Launches the builds of a thread-level apply kernel (XOR payloads of versions 1-2 only, the
// general one; from `first`); the scan's selection words decide on the device which works.
template <typename K>
cudaError_t launch_both(const LaunchCtx& c, K k12, int per_sm12, K k3, int per_sm3,
                        int first = 0) {
  const uint64_t want = (c.chunks + kWarps - 1) / kWarps;
  for (int b = first; b < 2; b++) {
    const uint64_t grid = std::min<uint64_t>(want, (uint64_t)(b ? per_sm3 : per_sm12) * c.sms);
    (b ? k3 : k12)<<<(unsigned)grid, kThreads, 0, c.stream>>>(
        reinterpret_cast<const DJob*>(c.ws + c.lay.jobs),
        reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start),
        reinterpret_cast<const uint64_t*>(c.ws + c.lay.tile_start), c.k, c.chunks,
        reinterpret_cast<const uint4*>(c.ws + c.lay.loc),
        reinterpret_cast<const TileSum*>(c.ws + c.lay.tile_pre),
        reinterpret_cast<JobInfo*>(c.ws + c.lay.info),
        reinterpret_cast<uint32_t*>(c.ws + c.lay.overflow),
        reinterpret_cast<uint32_t*>(c.ws + c.lay.ovf_list),
        reinterpret_cast<uint32_t*>(c.ws + c.lay.ovf_job), c.ws + c.lay.ck);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_apply_chunks(const LaunchCtx& c) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm12 = blocks_per_sm(k_apply_chunks<false>);
  static const int per_sm3 = blocks_per_sm(k_apply_chunks<true>);
  return launch_both(c, k_apply_chunks<false>, per_sm12, k_apply_chunks<true>, per_sm3);
}

cudaError_t launch_copy_jobs(const LaunchCtx& c) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm = blocks_per_sm(k_copy_jobs);
  const uint64_t grid = std::min<uint64_t>((c.chunks + kWarps - 1) / kWarps, (uint64_t)per_sm * c.sms);
  k_copy_jobs<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const DJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start), c.k, c.chunks,
      reinterpret_cast<const JobInfo*>(c.ws + c.lay.info));
  return cudaGetLastError();
}

cudaError_t launch_apply_incremental(const LaunchCtx& c) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm12 = blocks_per_sm(k_apply_incr<false, false>);
  static const int per_sm3 = blocks_per_sm(k_apply_incr<true, false>);
  static const int per_smo = blocks_per_sm(k_apply_incr<true, true>);
  cudaError_t e = launch_both(c, k_apply_incr<false, false>, per_sm12, k_apply_incr<true, false>,
                              per_sm3);
  if (e != cudaSuccess) return e;
  return launch_both(c, k_apply_incr<true, true>, per_smo, k_apply_incr<true, true>, per_smo, 1);
}

cudaError_t launch_apply(const LaunchCtx& c, bool incremental) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm = blocks_per_sm(k_apply_dense<false>);
  const uint64_t grid = std::min<uint64_t>(c.chunks, (uint64_t)per_sm * c.sms);
  auto kernel = incremental ? k_apply_dense<true> : k_apply_dense<false>;
  kernel<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const DJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.tile_start), c.k,
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.overflow),
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.ovf_list),
      reinterpret_cast<const uint4*>(c.ws + c.lay.loc),
      reinterpret_cast<const TileSum*>(c.ws + c.lay.tile_pre),
      reinterpret_cast<JobInfo*>(c.ws + c.lay.info), c.ws + c.lay.ck);
  return cudaGetLastError();
}

cudaError_t launch_apply_bitmap(const LaunchCtx& c, bool incremental) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm = blocks_per_sm(k_apply_bitmap<false>);
  static const int per_sm_i = blocks_per_sm(k_apply_bitmap<true>);
  const uint64_t grid = std::min<uint64_t>((c.chunks + kWarps - 1) / kWarps,
                                           (uint64_t)(incremental ? per_sm_i : per_sm) * c.sms);
  auto kernel = incremental ? k_apply_bitmap<true> : k_apply_bitmap<false>;
  kernel<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const DJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.tile_start), c.k,
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.overflow),
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.ovf_list),
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.ovf_job),
      reinterpret_cast<const uint4*>(c.ws + c.lay.loc),
      reinterpret_cast<const TileSum*>(c.ws + c.lay.tile_pre),
      reinterpret_cast<JobInfo*>(c.ws + c.lay.info), c.ws + c.lay.ck);
  return cudaGetLastError();
}

cudaError_t launch_apply_finish(const LaunchCtx& c, int32_t* d_status_all) {
  const unsigned threads = 128;
  const unsigned grid = (unsigned)((c.k + threads - 1) / threads);
  k_apply_finish<<<grid, threads, 0, c.stream>>>(
      reinterpret_cast<const DJob*>(c.ws + c.lay.jobs), c.k,
      reinterpret_cast<JobInfo*>(c.ws + c.lay.info), c.ws + c.lay.ck, d_status_all);
  return cudaGetLastError();
}

}  // namespace bd
