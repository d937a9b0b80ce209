// bd_apply.cu -- decompress (apply) kernels of libbf16delta.
//
// "GPU-accelerated Weight Teleportation", section "Delta update algebra": the rollout side
// XORs the mask into its old weights to obtain the new ones.  "Every byte counts: ARCv3 and
// the case for cross-region RL": both streams are applied to the previous checkpoint and the
// result is checksummed against the trainer's original.
//
// After the count scan (bd_scan.cu):
//   decode        one warp per chunk: decodes the chunk's position blocks (delta list -> prefix
//                 sum, or bitmap -> popcount rank) and gathers its 7-bit and 16-bit XOR values
//                 into a position-sorted entry list in the chunk's workspace slot, checking
//                 every rule of the format.  Chunks with more changes than a slot holds are
//                 listed for apply_dense.
//   apply_stream  one warp per chunk, the streaming pass over old: per 512-element step it
//                 scatters the step's entries into a 1 KiB shared mask, XORs, checksums the
//                 result and writes back only the 16-byte groups that changed (in place) or
//                 every group (out of place).
//   apply_dense   one CTA per listed chunk: decodes straight from the payload into an 8 KiB
//                 shared mask (dense chunks, bitmap positions).
//   apply_finish  one thread per tensor: checks the mantissa-stream pad bits, compares the
//                 checksum with the expected value and publishes the status.
// Malformed chunks are detected before any write to them and are left unwritten.
#include <algorithm>

#include "bd_internal.cuh"

namespace bd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// 7-bit value j of an M stream.  The caller guarantees j < number of M values, so the
// second byte is read only when the value crosses into it (and then it exists).
__device__ __forceinline__ uint32_t mant_value(const uint8_t* __restrict__ ms, uint64_t j) {
  const uint64_t bit = 7 * j;
  const uint32_t s = (uint32_t)(bit & 7);
  uint32_t v = ms[bit >> 3] >> s;
  if (s > 1) v |= (uint32_t)ms[(bit >> 3) + 1] << (8 - s);
  return v & kMant;
}

__global__ void __launch_bounds__(kThreads)
k_apply_dense(const DJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
              const uint64_t* __restrict__ tile_start, uint32_t k,
              const uint32_t* __restrict__ list_count, const uint32_t* __restrict__ list,
              const uint4* __restrict__ loc, const TileSum* __restrict__ tile_pre,
              JobInfo* __restrict__ info, uint8_t* __restrict__ ck_base) {
  __shared__ uint4 s_mask4[kChunk / 8];       // the chunk's XOR mask, 8 KiB
  __shared__ uint32_t s_tot[kWarps][4];
  __shared__ int s_bad;
  __shared__ uint64_t s_ck[kWarps];
  uint16_t* s_mask = reinterpret_cast<uint16_t*>(s_mask4);
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;

  if (t == 0) s_bad = 0;
  uint32_t cur_job = 0xFFFFFFFFu;
  uint64_t ck = 0;
  __syncthreads();

  const uint32_t listed = *list_count;
  for (uint32_t li = blockIdx.x; li < listed; li += gridDim.x) {
    const uint64_t g = list[li];
    const uint32_t j = find_job(chunk_start, k, g);
    if (j != cur_job) {
      if (cur_job != 0xFFFFFFFFu) {
        const uint64_t s = warp_sum64(ck);
        if (lane == 0) s_ck[w] = s;
        __syncthreads();
        if (t == 0) {
          uint64_t tot = 0;
          for (int q = 0; q < kWarps; q++) tot += s_ck[q];
          atomicAdd(reinterpret_cast<unsigned long long*>(ck_base + (uint64_t)cur_job * kCkBytes) +
                        (blockIdx.x & (kCkSlots - 1)) * kCkStride,
                    (unsigned long long)tot);
        }
        __syncthreads();
      }
      cur_job = j;
      ck = 0;
    }
    if (info[j].status != BD_OK) continue;

    const DJob& J = jobs[j];
    const uint64_t n = J.n;
    const uint64_t c = g - chunk_start[j];
    const uint64_t e0 = c * kChunk;
    const uint32_t L = (n - e0) < kChunk ? (uint32_t)(n - e0) : kChunk;
    const uint32_t B = (L + 7) >> 3;
    const uint8_t* __restrict__ payload = J.payload;
    const uint32_t cnt = reinterpret_cast<const uint32_t*>(payload + kHeader)[c];
    const uint32_t M = cnt & 0xFFFFu, R = cnt >> 16;
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

    // the old chunk: groups t and t + 256 (8 elements each)
    const uint64_t ea = e0 + 8 * (uint64_t)t, eb = ea + 2048;
    const uint4 oa = load8(J.old, ea, n), ob = load8(J.old, eb, n);
    s_mask4[t] = make_uint4(0, 0, 0, 0);
    s_mask4[t + 256] = make_uint4(0, 0, 0, 0);

    // per-thread scan inputs: list entry t (slot a) or bitmap bytes t, t+256 (slots a, b)
    bool bad = false;
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
        if (pos >= L || v == 0) bad = true;
        else s_mask[pos] = (uint16_t)v;
      }
    } else {
      if (totaM + totbM != M) bad = true;
      uint32_t r = xaM;
      for (uint32_t bits = byteMa; bits; bits &= bits - 1, r++) {
        const uint32_t pos = 8 * t + __ffs(bits) - 1;
        if (r >= M || pos >= L) { bad = true; break; }
        const uint32_t v = mant_value(mstream, Mex + r);
        if (v == 0) bad = true; else s_mask[pos] = (uint16_t)v;
      }
      r = xbM;
      for (uint32_t bits = byteMb; bits; bits &= bits - 1, r++) {
        const uint32_t pos = 8 * (t + 256) + __ffs(bits) - 1;
        if (r >= M || pos >= L) { bad = true; break; }
        const uint32_t v = mant_value(mstream, Mex + r);
        if (v == 0) bad = true; else s_mask[pos] = (uint16_t)v;
      }
    }
    __syncthreads();
    // scatter the rare values; a position already holding a mantissa value is malformed
    if (listR) {
      if ((uint32_t)t < R) {
        const uint32_t pos = xaR + aR;
        const uint32_t v = load_u16(rstream + 2 * t);
        if (pos >= L || (v & kSignExp) == 0 || s_mask[pos] != 0) bad = true;
        else s_mask[pos] = (uint16_t)v;
      }
    } else {
      if (totaR + totbR != R) bad = true;
      uint32_t r = xaR;
      for (uint32_t bits = byteRa; bits; bits &= bits - 1, r++) {
        const uint32_t pos = 8 * t + __ffs(bits) - 1;
        if (r >= R || pos >= L) { bad = true; break; }
        const uint32_t v = load_u16(rstream + 2 * r);
        if ((v & kSignExp) == 0 || s_mask[pos] != 0) bad = true; else s_mask[pos] = (uint16_t)v;
      }
      r = xbR;
      for (uint32_t bits = byteRb; bits; bits &= bits - 1, r++) {
        const uint32_t pos = 8 * (t + 256) + __ffs(bits) - 1;
        if (r >= R || pos >= L) { bad = true; break; }
        const uint32_t v = load_u16(rstream + 2 * r);
        if ((v & kSignExp) == 0 || s_mask[pos] != 0) bad = true; else s_mask[pos] = (uint16_t)v;
      }
    }
    if (bad) s_bad = 1;
    __syncthreads();
    const bool chunk_bad = s_bad != 0;
    if (!chunk_bad) {
      const uint4 ma = s_mask4[t], mb = s_mask4[t + 256];
      const uint4 ra = make_uint4(oa.x ^ ma.x, oa.y ^ ma.y, oa.z ^ ma.z, oa.w ^ ma.w);
      const uint4 rb = make_uint4(ob.x ^ mb.x, ob.y ^ mb.y, ob.z ^ mb.z, ob.w ^ mb.w);
      const uint64_t words = (n + 3) >> 2;
      ck += group_hash(ra, ea >> 3, words) + group_hash(rb, eb >> 3, words);
      const bool inplace = J.out == J.old;
      const bool cha = (ma.x | ma.y | ma.z | ma.w) != 0, chb = (mb.x | mb.y | mb.z | mb.w) != 0;
      uint16_t* out = J.out;
      if (ea < n && (!inplace || cha)) {
        if (ea + 8 <= n) *reinterpret_cast<uint4*>(out + ea) = ra;
        else for (int i = 0; ea + i < n; i++) out[ea + i] = (uint16_t)elem_of(ra, i);
      }
      if (eb < n && (!inplace || chb)) {
        if (eb + 8 <= n) *reinterpret_cast<uint4*>(out + eb) = rb;
        else for (int i = 0; eb + i < n; i++) out[eb + i] = (uint16_t)elem_of(rb, i);
      }
    }
    __syncthreads();
    if (t == 0 && chunk_bad) {
      record_status(&info[j].chunk_err, BD_ERR_FORMAT);
      s_bad = 0;
    }
    __syncthreads();
  }
  if (cur_job != 0xFFFFFFFFu) {
    const uint64_t s = warp_sum64(ck);
    if (lane == 0) s_ck[w] = s;
    __syncthreads();
    if (t == 0) {
      uint64_t tot = 0;
      for (int q = 0; q < kWarps; q++) tot += s_ck[q];
      atomicAdd(reinterpret_cast<unsigned long long*>(ck_base + (uint64_t)cur_job * kCkBytes) +
                    (blockIdx.x & (kCkSlots - 1)) * kCkStride,
                (unsigned long long)tot);
    }
  }
}

// ------------------------------------------------------------------------ decode

struct DecodeSmem {
  uint16_t posM[256], valM[256], posR[256], valR[256];
};

// Number of values < x in the ascending array a[0..k).
__device__ __forceinline__ uint32_t lower_bound16(const uint16_t* a, uint32_t k, uint32_t x) {
  uint32_t lo = 0, hi = k;
  while (lo < hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Decodes the k ascending positions of one class (block at blk, chunk of length L whose
// bitmap has B bytes) into pos[0..k).  Returns true when the block is malformed.
__device__ __forceinline__ bool decode_positions(const uint8_t* __restrict__ blk, uint32_t k,
                                                 uint32_t L, uint32_t B, uint16_t* pos) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
  if (2 * k < B) {  // delta list: d_0 = p_0, d_i = p_i - p_{i-1} >= 1
    uint32_t carry = 0;
    for (uint32_t base = 0; base < k; base += 32) {
      const uint32_t i = base + lane;
      uint32_t d = 0;
      if (i < k) {
        d = load_u16(blk + 2 * i);
        if (i > 0 && d == 0) bad = true;
      }
      const uint32_t p = carry + warp_incl_scan(d);
      if (i < k) {
        if (p >= L) bad = true;
        pos[i] = (uint16_t)(p < L ? p : 0);
      }
      carry = __shfl_sync(0xFFFFFFFFu, p, 31);
    }
  } else {  // bitmap: lane handles bytes [16 lane, 16 lane + 16)
    uint32_t bytes[4] = {0, 0, 0, 0};
    uint32_t cnt = 0;
    for (int q = 0; q < 16; q++) {
      const uint32_t bi = 16 * lane + q;
      const uint32_t v = bi < B ? blk[bi] : 0u;
      bytes[q >> 2] |= v << (8 * (q & 3));
      cnt += __popc(v);
    }
    const uint32_t incl = warp_incl_scan(cnt);
    if (__shfl_sync(0xFFFFFFFFu, incl, 31) != k) bad = true;
    uint32_t r = incl - cnt;
    for (int q = 0; q < 4; q++) {
      for (uint32_t bits = bytes[q]; bits; bits &= bits - 1) {
        const uint32_t p = 16 * 8 * lane + 32 * q + __ffs(bits) - 1;
        if (p >= L || r >= k) { bad = true; break; }
        pos[r++] = (uint16_t)p;
      }
    }
  }
  return bad;
}

__global__ void __launch_bounds__(kThreads)
k_decode(const DJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
         const uint64_t* __restrict__ tile_start, uint32_t k, uint64_t total_chunks,
         const uint4* __restrict__ loc, const TileSum* __restrict__ tile_pre,
         JobInfo* __restrict__ info, uint8_t* __restrict__ slots,
         uint32_t* __restrict__ list_count, uint32_t* __restrict__ list) {
  __shared__ DecodeSmem s_dec[kWarps];
  const int lane = threadIdx.x & 31;
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  DecodeSmem* sm = &s_dec[threadIdx.x >> 5];
  uint32_t j = 0xFFFFFFFFu;
  for (uint64_t g = gwarp; g < total_chunks; g += nwarps) {
    j = advance_job(chunk_start, k, j, g);
    const uint4 lc = loc[g];
    if (info[j].status != BD_OK) continue;
    const DJob& J = jobs[j];
    const uint64_t c = g - chunk_start[j];
    const uint64_t e0 = c * kChunk;
    const uint32_t L = (J.n - e0) < kChunk ? (uint32_t)(J.n - e0) : kChunk;
    const uint32_t B = (L + 7) >> 3;
    const uint8_t* __restrict__ payload = J.payload;
    const uint32_t cnt = reinterpret_cast<const uint32_t*>(payload + kHeader)[c];
    const uint32_t M = cnt & 0xFFFFu, R = cnt >> 16;
    uint32_t* slot = reinterpret_cast<uint32_t*>(slots + g * kSlotBytes);
    if (M + R > kSlotEntries) {
      if (lane == 0) {
        slot[0] = kSlotOverflow;
        list[atomicAdd(list_count, 1u)] = (uint32_t)g;
      }
      continue;
    }
    const TileSum pre = tile_pre[tile_start[j] + c / kTileChunks];
    const uint64_t Pex = pre.p + lc.x, Mex = pre.m + lc.y, Rex = pre.r + lc.z;
    const JobInfo& I = info[j];
    const uint8_t* mblk = payload + I.p_start + Pex;
    const uint8_t* rblk = mblk + block_bytes(M, B);
    const uint8_t* mstream = payload + I.m_start;
    const uint8_t* rstream = payload + I.r_start + 2 * Rex;

    bool bad = decode_positions(mblk, M, L, B, sm->posM);
    bad |= decode_positions(rblk, R, L, B, sm->posR);
    for (uint32_t r = lane; r < M; r += 32) {
      const uint32_t v = mant_value(mstream, Mex + r);
      if (v == 0) bad = true;
      sm->valM[r] = (uint16_t)v;
    }
    for (uint32_t r = lane; r < R; r += 32) {
      const uint32_t v = load_u16(rstream + 2 * r);
      if ((v & kSignExp) == 0) bad = true;
      sm->valR[r] = (uint16_t)v;
    }
    __syncwarp();
    // merge the two ascending lists into position order; a shared position is malformed
    uint32_t* entries = slot + kSlotHeader / 4;
    for (uint32_t r = lane; r < M; r += 32) {
      const uint32_t p = sm->posM[r];
      const uint32_t less = lower_bound16(sm->posR, R, p);
      if (less < R && sm->posR[less] == p) bad = true;
      entries[r + less] = (p << 16) | sm->valM[r];
    }
    for (uint32_t r = lane; r < R; r += 32) {
      const uint32_t p = sm->posR[r];
      entries[r + lower_bound16(sm->posM, M, p)] = (p << 16) | sm->valR[r];
    }
    // step_end[s]: entries with position < 512 (s + 1)
    uint32_t se = 0;
    if (lane < 8) {
      const uint32_t bound = 512u * (lane + 1);
      se = lower_bound16(sm->posM, M, bound) + lower_bound16(sm->posR, R, bound);
    }
    uint32_t w0 = 0, w1 = 0;
#pragma unroll
    for (int q = 0; q < 4; q++) {
      w0 |= __shfl_sync(0xFFFFFFFFu, se, q) << (8 * q);
      w1 |= __shfl_sync(0xFFFFFFFFu, se, q + 4) << (8 * q);
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
      slot[0] = (M + R) | (bad ? kSlotBad : 0u);
      slot[2] = w0;
      slot[3] = w1;
      if (bad) record_status(&info[j].chunk_err, BD_ERR_FORMAT);
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------------ apply_stream

struct StreamSmem {
  uint32_t ent[kSlotEntries + 4];
  uint4 mask4[64];   // 512 u16: the XOR mask of one step
};

template <bool FULL>
__device__ __forceinline__ void stream_chunk(const uint16_t* __restrict__ old,
                                             uint16_t* __restrict__ out, bool inplace,
                                             uint64_t n, uint64_t e0, uint32_t w0, uint32_t w1,
                                             StreamSmem* sm, uint64_t& ck) {
  const int lane = threadIdx.x & 31;
  const uint64_t words = (n + 3) >> 2;
  uint16_t* mask = reinterpret_cast<uint16_t*>(sm->mask4);
  uint64_t e = e0 + lane * 16;
  uint4 o0, o1;
  if (FULL) {
    o0 = __ldg(reinterpret_cast<const uint4*>(old + e));
    o1 = __ldg(reinterpret_cast<const uint4*>(old + e + 8));
  } else {
    o0 = load8(old, e, n);
    o1 = load8(old, e + 8, n);
  }
  uint64_t key = ((e >> 2) + 1) * kGamma;
  uint32_t lo = 0;
#pragma unroll 1
  for (int s = 0; s < 8; s++) {
    const uint4 c0 = o0, c1 = o1;
    if (s < 7) {
      if (FULL) {
        o0 = __ldg(reinterpret_cast<const uint4*>(old + e + 512));
        o1 = __ldg(reinterpret_cast<const uint4*>(old + e + 520));
      } else {
        o0 = load8(old, e + 512, n);
        o1 = load8(old, e + 520, n);
      }
    }
    const uint32_t hi = ((s < 4 ? w0 : w1) >> (8 * (s & 3))) & 0xFFu;
    uint4 m0 = make_uint4(0, 0, 0, 0), m1 = m0;
    if (__any_sync(0xFFFFFFFFu, hi > lo)) {
      sm->mask4[2 * lane] = m0;
      sm->mask4[2 * lane + 1] = m1;
      __syncwarp();
      for (uint32_t i = lo + lane; i < hi; i += 32) {
        const uint32_t en = sm->ent[i];
        mask[(en >> 16) & 511] = (uint16_t)(en & 0xFFFFu);
      }
      __syncwarp();
      m0 = sm->mask4[2 * lane];
      m1 = sm->mask4[2 * lane + 1];
      __syncwarp();
    }
    lo = hi;
    const uint4 r0 = make_uint4(c0.x ^ m0.x, c0.y ^ m0.y, c0.z ^ m0.z, c0.w ^ m0.w);
    const uint4 r1 = make_uint4(c1.x ^ m1.x, c1.y ^ m1.y, c1.z ^ m1.z, c1.w ^ m1.w);
    const bool ch0 = (m0.x | m0.y | m0.z | m0.w) != 0, ch1 = (m1.x | m1.y | m1.z | m1.w) != 0;
    if (FULL) {
      const uint64_t a0 = (uint64_t)r0.x | ((uint64_t)r0.y << 32);
      const uint64_t a1 = (uint64_t)r0.z | ((uint64_t)r0.w << 32);
      const uint64_t a2 = (uint64_t)r1.x | ((uint64_t)r1.y << 32);
      const uint64_t a3 = (uint64_t)r1.z | ((uint64_t)r1.w << 32);
      ck += mix64(a0 ^ key) + mix64(a1 ^ (key + kGamma)) + mix64(a2 ^ (key + 2 * kGamma)) +
            mix64(a3 ^ (key + 3 * kGamma));
      if (!inplace || ch0) *reinterpret_cast<uint4*>(out + e) = r0;
      if (!inplace || ch1) *reinterpret_cast<uint4*>(out + e + 8) = r1;
    } else {
      ck += group_hash(r0, e >> 3, words) + group_hash(r1, (e >> 3) + 1, words);
      if (e < n && (!inplace || ch0)) {
        if (e + 8 <= n) *reinterpret_cast<uint4*>(out + e) = r0;
        else for (int i = 0; e + i < n; i++) out[e + i] = (uint16_t)elem_of(r0, i);
      }
      if (e + 8 < n && (!inplace || ch1)) {
        if (e + 16 <= n) *reinterpret_cast<uint4*>(out + e + 8) = r1;
        else for (int i = 0; e + 8 + i < n; i++) out[e + 8 + i] = (uint16_t)elem_of(r1, i);
      }
    }
    e += 512;
    key += 128 * kGamma;
  }
}

__global__ void __launch_bounds__(kThreads)
k_apply_stream(const DJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
               uint32_t k, uint64_t total_chunks, const JobInfo* __restrict__ info,
               const uint8_t* __restrict__ slots, uint8_t* __restrict__ ck_base) {
  __shared__ StreamSmem s_st[kWarps];
  const int lane = threadIdx.x & 31;
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  StreamSmem* sm = &s_st[threadIdx.x >> 5];
  uint32_t j = 0xFFFFFFFFu, cur = 0xFFFFFFFFu;
  uint64_t ck = 0;
  for (uint64_t g = gwarp; g < total_chunks; g += nwarps) {
    j = advance_job(chunk_start, k, j, g);
    const uint4 hdr = *reinterpret_cast<const uint4*>(slots + g * kSlotBytes);
    if (info[j].status != BD_OK || (hdr.x & (kSlotOverflow | kSlotBad))) continue;
    if (j != cur) {
      if (cur != 0xFFFFFFFFu) {
        const uint64_t s = warp_sum64(ck);
        if (lane == 0)
          atomicAdd(reinterpret_cast<unsigned long long*>(ck_base + (uint64_t)cur * kCkBytes) +
                        (gwarp & (kCkSlots - 1)) * kCkStride,
                    (unsigned long long)s);
      }
      cur = j;
      ck = 0;
    }
    const uint32_t kk = hdr.x & 0xFFFFu;
    const uint32_t* ent = reinterpret_cast<const uint32_t*>(slots + g * kSlotBytes + kSlotHeader);
    for (uint32_t i = lane; i < kk; i += 32) sm->ent[i] = ent[i];
    __syncwarp();
    const DJob& J = jobs[j];
    const uint64_t e0 = (g - chunk_start[j]) * kChunk;
    const bool inplace = J.out == J.old;
    if (e0 + kChunk <= J.n)
      stream_chunk<true>(J.old, J.out, inplace, J.n, e0, hdr.z, hdr.w, sm, ck);
    else
      stream_chunk<false>(J.old, J.out, inplace, J.n, e0, hdr.z, hdr.w, sm, ck);
    __syncwarp();
  }
  if (cur != 0xFFFFFFFFu) {
    const uint64_t s = warp_sum64(ck);
    if (lane == 0)
      atomicAdd(reinterpret_cast<unsigned long long*>(ck_base + (uint64_t)cur * kCkBytes) +
                    (gwarp & (kCkSlots - 1)) * kCkStride,
                (unsigned long long)s);
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
    const uint64_t* ck = reinterpret_cast<const uint64_t*>(ck_base + j * kCkBytes);
    uint64_t sum = 0;
    for (int s = 0; s < kCkSlots; s++) sum += ck[s * kCkStride];
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

cudaError_t launch_decode(const LaunchCtx& c) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm = blocks_per_sm(k_decode);
  const uint64_t grid = std::min<uint64_t>((c.chunks + kWarps - 1) / kWarps, (uint64_t)per_sm * c.sms);
  k_decode<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const DJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.tile_start), c.k, c.chunks,
      reinterpret_cast<const uint4*>(c.ws + c.lay.loc),
      reinterpret_cast<const TileSum*>(c.ws + c.lay.tile_pre),
      reinterpret_cast<JobInfo*>(c.ws + c.lay.info), c.ws + c.lay.slots,
      reinterpret_cast<uint32_t*>(c.ws + c.lay.overflow),
      reinterpret_cast<uint32_t*>(c.ws + c.lay.ovf_list));
  return cudaGetLastError();
}

cudaError_t launch_apply_stream(const LaunchCtx& c) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm = blocks_per_sm(k_apply_stream);
  const uint64_t grid = std::min<uint64_t>((c.chunks + kWarps - 1) / kWarps, (uint64_t)per_sm * c.sms);
  k_apply_stream<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const DJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start), c.k, c.chunks,
      reinterpret_cast<const JobInfo*>(c.ws + c.lay.info), c.ws + c.lay.slots, c.ws + c.lay.ck);
  return cudaGetLastError();
}

cudaError_t launch_apply(const LaunchCtx& c) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm = blocks_per_sm(k_apply_dense);
  const uint64_t grid = std::min<uint64_t>(c.chunks, (uint64_t)per_sm * c.sms);
  k_apply_dense<<<(unsigned)grid, kThreads, 0, c.stream>>>(
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

cudaError_t launch_apply_finish(const LaunchCtx& c, int32_t* d_status_all) {
  const unsigned threads = 128;
  const unsigned grid = (unsigned)((c.k + threads - 1) / threads);
  k_apply_finish<<<grid, threads, 0, c.stream>>>(
      reinterpret_cast<const DJob*>(c.ws + c.lay.jobs), c.k,
      reinterpret_cast<JobInfo*>(c.ws + c.lay.info), c.ws + c.lay.ck, d_status_all);
  return cudaGetLastError();
}

}  // namespace bd
