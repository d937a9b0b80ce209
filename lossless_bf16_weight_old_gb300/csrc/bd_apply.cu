// bd_apply.cu -- decompress (apply) kernels of libbf16delta.
//
// "GPU-accelerated Weight Teleportation", section "Delta update algebra": the rollout side
// XORs the mask into its old weights to obtain the new ones.  "Every byte counts: ARCv3 and
// the case for cross-region RL": both streams are applied to the previous checkpoint and the
// result is checksummed against the trainer's original.
//
// After the count scan (bd_scan.cu):
//   decode        one warp per chunk: requests the chunk's position blocks and values in one
//                 round, decodes the positions (delta list -> prefix sum, or bitmap ->
//                 popcount rank) and writes (position, XOR) entries into the chunk's workspace
//                 slot, mantissa-only from the front and rare from the back, checking the
//                 format rules.  Chunks with more changes than a slot holds are listed for
//                 apply_dense.
//   apply_stream  two warps per chunk, the streaming pass over old: the chunk's 8 KiB of old are
//                 copied into shared memory with cp.async while the previous chunk is processed
//                 (double buffer) and its slot is prefetched into registers; the entries are
//                 XORed into the staged data with shared-memory atomics (a position taken
//                 twice is malformed), then each warp checksums half of the result, two steps
//                 at a time, and writes back only the 16-byte groups that changed (in place)
//                 or every group (out of place).
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

// 16-byte asynchronous global -> shared copy; src_bytes < 16 zero-fills the rest.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, uint32_t src_bytes) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// 4-byte asynchronous global -> shared copy; src_bytes < 4 zero-fills the rest.
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem, uint32_t src_bytes) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(s), "l"(gmem),
               "r"(src_bytes)
               : "memory");
}


// Staging capacity per warp, in 32-bit words, of the three payload byte ranges of one chunk
// whose changes fit a slot (M + R <= kSlotEntries): position blocks (delta lists up to 504
// bytes, or bitmaps of a ragged last chunk up to 2 x 511 bytes), mantissa bytes (up to 221)
// and rare values (up to 504 bytes), each widened to whole aligned words.
constexpr int kStageP = 9, kStageM = 2, kStageR = 4;   // words per lane
struct DecodeSmem {
  uint32_t wp[32 * kStageP], wm[32 * kStageM], wr[32 * kStageR];
};

__device__ __forceinline__ uint32_t sbyte(const uint32_t* w, uint32_t i) {
  return (w[i >> 2] >> (8 * (i & 3))) & 0xFFu;
}
__device__ __forceinline__ uint32_t su16(const uint32_t* w, uint32_t i) {
  return sbyte(w, i) | (sbyte(w, i + 1) << 8);
}

// Decodes the k ascending positions of one class from the staged block (byte offset `boff`
// in the word buffer w; chunk of length L whose bitmap has B bytes) and hands each one to
// sink(rank, position).  Returns true when the block is malformed.
template <typename SINK>
__device__ __forceinline__ bool decode_positions(const uint32_t* w, uint32_t boff, uint32_t k,
                                                 uint32_t L, uint32_t B, SINK sink) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
  if (2 * k < B) {  // delta list: d_0 = p_0, d_i = p_i - p_{i-1} >= 1
    uint32_t carry = 0;
    for (uint32_t base = 0; base < k; base += 32) {
      const uint32_t i = base + lane;
      uint32_t d = 0;
      if (i < k) {
        d = su16(w, boff + 2 * i);
        if (i > 0 && d == 0) bad = true;
      }
      const uint32_t p = carry + warp_incl_scan(d);
      if (i < k) {
        if (p >= L) bad = true;
        else sink(i, p);
      }
      carry = __shfl_sync(0xFFFFFFFFu, p, 31);
    }
  } else {  // bitmap: lane handles bytes [16 lane, 16 lane + 16)
    uint32_t bytes[4] = {0, 0, 0, 0};
    uint32_t cnt = 0;
#pragma unroll
    for (int q = 0; q < 16; q++) {
      const uint32_t bi = 16 * lane + q;
      const uint32_t v = bi < B ? sbyte(w, boff + bi) : 0u;
      bytes[q >> 2] |= v << (8 * (q & 3));
      cnt += __popc(v);
    }
    const uint32_t incl = warp_incl_scan(cnt);
    if (__shfl_sync(0xFFFFFFFFu, incl, 31) != k) bad = true;
    uint32_t r = incl - cnt;
    for (int q = 0; q < 4; q++) {
      for (uint32_t bits = bytes[q]; bits; bits &= bits - 1) {
        const uint32_t p = 128 * lane + 32 * q + __ffs(bits) - 1;
        if (p >= L || r >= k) { bad = true; break; }
        sink(r++, p);
      }
    }
  }
  return bad;
}

// One chunk's payload pieces, as aligned word ranges.
struct WordRange {
  uint64_t first;   // byte offset (multiple of 4) of the first word
  uint32_t words;   // words to stage
  uint32_t skip;    // offset of the range's first byte inside the first word
};
__device__ __forceinline__ WordRange word_range(uint64_t a, uint64_t b) {
  WordRange r;
  r.first = a & ~3ull;
  r.skip = (uint32_t)(a - r.first);
  r.words = b > a ? (uint32_t)((((b + 3) & ~3ull) - r.first) >> 2) : 0u;
  return r;
}

// Starts the asynchronous copy of word w of range r (payload of `size` bytes) to dst.
__device__ __forceinline__ void stage_word(uint32_t* dst, const uint8_t* __restrict__ payload,
                                           const WordRange& r, uint32_t w, uint64_t size) {
  if (w >= r.words) return;
  const uint64_t off = r.first + 4ull * w;
  const uint32_t bytes = off + 4 <= size ? 4u : (off < size ? (uint32_t)(size - off) : 0u);
  cp_async4(dst, bytes ? payload + off : payload, bytes);
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
    // level 1: everything addressed by g and j alone
    const DJob& J = jobs[j];
    const JobInfo& I = info[j];
    const uint64_t c = g - chunk_start[j];
    const uint4 lc = loc[g];
    const TileSum pre = tile_pre[tile_start[j] + c / kTileChunks];
    const int32_t status = I.status;
    const uint8_t* __restrict__ payload = J.payload;
    if (status != BD_OK) continue;
    const uint32_t cnt = reinterpret_cast<const uint32_t*>(payload + kHeader)[c];
    const uint64_t n = J.n, size = J.size;
    const uint64_t e0 = c * kChunk;
    const uint32_t L = (n - e0) < kChunk ? (uint32_t)(n - e0) : kChunk;
    const uint32_t B = (L + 7) >> 3;
    const uint32_t M = cnt & 0xFFFFu, R = cnt >> 16;
    uint32_t* slot = reinterpret_cast<uint32_t*>(slots + g * kSlotBytes);
    if (M + R > kSlotEntries) {
      if (lane == 0) {
        slot[0] = kSlotOverflow;
        list[atomicAdd(list_count, 1u)] = (uint32_t)g;
      }
      continue;
    }
    const uint64_t Pex = pre.p + lc.x, Mex = pre.m + lc.y, Rex = pre.r + lc.z;
    const uint32_t blkM = block_bytes(M, B), blkR = block_bytes(R, B);
    // level 2: the chunk's three payload ranges, all words requested before any is used
    const uint64_t pa = I.p_start + Pex;
    const WordRange wp = word_range(pa, pa + blkM + blkR);
    const uint64_t ma = I.m_start + ((7 * Mex) >> 3);
    const WordRange wm = word_range(ma, I.m_start + ((7 * (Mex + M) + 7) >> 3));
    const uint64_t ra = I.r_start + 2 * Rex;
    const WordRange wr = word_range(ra, ra + 2 * R);
#pragma unroll
    for (int q = 0; q < kStageP; q++) stage_word(&sm->wp[lane + 32 * q], payload, wp, lane + 32 * q, size);
#pragma unroll
    for (int q = 0; q < kStageM; q++) stage_word(&sm->wm[lane + 32 * q], payload, wm, lane + 32 * q, size);
#pragma unroll
    for (int q = 0; q < kStageR; q++) stage_word(&sm->wr[lane + 32 * q], payload, wr, lane + 32 * q, size);
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();

    // entries: mantissa-only at [0, M), rare at [M, M+R) (collisions are checked when the
    // chunk is applied)
    uint32_t* entries = slot + kSlotHeader / 4;
    bool bad = false;
    const uint32_t mbit0 = 8 * wm.skip + (uint32_t)((7 * Mex) & 7);
    const uint32_t* wmv = sm->wm;
    bad |= decode_positions(sm->wp, wp.skip, M, L, B, [&](uint32_t r, uint32_t p) {
      const uint32_t bit = mbit0 + 7 * r;
      const uint32_t v = (su16(wmv, bit >> 3) >> (bit & 7)) & kMant;
      if (v == 0) bad = true;
      entries[r] = (p << 16) | v;
    });
    const uint32_t* wrv = sm->wr;
    const uint32_t rskip = wr.skip;
    bad |= decode_positions(sm->wp, wp.skip + blkM, R, L, B, [&](uint32_t r, uint32_t p) {
      const uint32_t v = su16(wrv, rskip + 2 * r);
      if ((v & kSignExp) == 0) bad = true;
      entries[M + r] = (p << 16) | v;
    });
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
      slot[0] = slot_info(M, R) | (bad ? kSlotBad : 0u);
      if (bad) record_status(&info[j].chunk_err, BD_ERR_FORMAT);
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------------ apply_stream

constexpr int kStreamThreads = 256;  // 4 pairs of warps, one chunk per pair
constexpr int kStreamPairs = kStreamThreads / 64;
struct PairSmem {
  uint4 buf[2][kChunk / 8];       // two 8 KiB chunk buffers (double-buffered old data)
  uint32_t touched[kChunk / 32];  // 512 B: positions written in the current chunk
  uint32_t flag;                  // a position was taken twice
  uint32_t pad[3];
};

// Barrier over the 64 threads of one warp pair (ids 1..4; 0 is __syncthreads).
__device__ __forceinline__ void pair_sync(int pair) {
  asm volatile("bar.sync %0, 64;\n" ::"r"(pair + 1) : "memory");
}

// Starts copying chunk [e0, e0 + 4096) of old into buf: pair thread pt copies groups
// 64 t + pt (group q = elements e0 + 8q .. +8), elements past n read as zero.
__device__ __forceinline__ void issue_chunk(uint4* buf, const uint16_t* __restrict__ old,
                                            uint64_t n, uint64_t e0, uint32_t pt) {
#pragma unroll
  for (int t = 0; t < 8; t++) {
    const uint32_t q = 64 * t + pt;
    const uint64_t e = e0 + 8 * q;
    const uint32_t bytes = e + 8 <= n ? 16u : (e < n ? (uint32_t)(2 * (n - e)) : 0u);
    cp_async16(&buf[q], bytes ? old + e : old, bytes);
  }
}

// XORs one entry into the staged chunk; returns true when its position was already taken.
__device__ __forceinline__ bool xor_entry(uint32_t* data32, uint32_t* touched, uint32_t e) {
  const uint32_t pos = (e >> 16) & (kChunk - 1);
  atomicXor(&data32[pos >> 1], (e & 0xFFFFu) << (16 * (pos & 1)));
  return (atomicOr(&touched[pos >> 5], 1u << (pos & 31)) >> (pos & 31)) & 1u;
}

// Checksums and writes back the two 16-byte groups of this lane in step s (elements
// e0 + 512 s + 16 lane ..); tmask = the 16 touched bits of those elements.
template <bool FULL>
__device__ __forceinline__ void put_groups(uint4 r0, uint4 r1, uint32_t tmask, uint64_t e,
                                           uint64_t key, uint64_t n, uint64_t words,
                                           uint16_t* __restrict__ out, bool inplace,
                                           uint64_t& ck) {
  if (FULL) {
    const uint64_t a0 = (uint64_t)r0.x | ((uint64_t)r0.y << 32);
    const uint64_t a1 = (uint64_t)r0.z | ((uint64_t)r0.w << 32);
    const uint64_t a2 = (uint64_t)r1.x | ((uint64_t)r1.y << 32);
    const uint64_t a3 = (uint64_t)r1.z | ((uint64_t)r1.w << 32);
    ck += mix64(a0 ^ key) + mix64(a1 ^ (key + kGamma)) + mix64(a2 ^ (key + 2 * kGamma)) +
          mix64(a3 ^ (key + 3 * kGamma));
    if (!inplace || (tmask & 0xFFu)) *reinterpret_cast<uint4*>(out + e) = r0;
    if (!inplace || (tmask >> 8)) *reinterpret_cast<uint4*>(out + e + 8) = r1;
  } else {
    ck += group_hash(r0, e >> 3, words) + group_hash(r1, (e >> 3) + 1, words);
    if (e < n && (!inplace || (tmask & 0xFFu))) {
      if (e + 8 <= n) *reinterpret_cast<uint4*>(out + e) = r0;
      else for (int i = 0; e + i < n; i++) out[e + i] = (uint16_t)elem_of(r0, i);
    }
    if (e + 8 < n && (!inplace || (tmask >> 8))) {
      if (e + 16 <= n) *reinterpret_cast<uint4*>(out + e + 8) = r1;
      else for (int i = 0; e + 8 + i < n; i++) out[e + 8 + i] = (uint16_t)elem_of(r1, i);
    }
  }
}

// Steps s0 and s0 + 1 of a staged chunk, interleaved (eight independent hash chains per lane).
template <bool FULL>
__device__ __forceinline__ void stream_two_steps(const uint4* buf, const uint32_t* touched,
                                                 int s0, uint64_t e0, uint64_t n,
                                                 uint16_t* __restrict__ out, bool inplace,
                                                 uint64_t& ck) {
  const int lane = threadIdx.x & 31;
  const uint64_t words = (n + 3) >> 2;
  const uint4 a0 = buf[64 * s0 + 2 * lane], a1 = buf[64 * s0 + 2 * lane + 1];
  const uint4 b0 = buf[64 * (s0 + 1) + 2 * lane], b1 = buf[64 * (s0 + 1) + 2 * lane + 1];
  const uint32_t ta = (touched[16 * s0 + (lane >> 1)] >> (16 * (lane & 1))) & 0xFFFFu;
  const uint32_t tb = (touched[16 * (s0 + 1) + (lane >> 1)] >> (16 * (lane & 1))) & 0xFFFFu;
  const uint64_t ea = e0 + 512 * s0 + 16 * lane, eb = ea + 512;
  const uint64_t ka = ((ea >> 2) + 1) * kGamma, kb = ka + 128 * kGamma;
  uint64_t c0 = 0, c1 = 0;
  put_groups<FULL>(a0, a1, ta, ea, ka, n, words, out, inplace, c0);
  put_groups<FULL>(b0, b1, tb, eb, kb, n, words, out, inplace, c1);
  ck += c0 + c1;
}

__global__ void __launch_bounds__(kStreamThreads)
k_apply_stream(const DJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
               uint32_t k, uint64_t total_chunks, JobInfo* __restrict__ info,
               const uint8_t* __restrict__ slots, uint8_t* __restrict__ ck_base) {
  extern __shared__ uint4 s_dyn[];
  const int lane = threadIdx.x & 31;
  const int pair = threadIdx.x >> 6, half = (threadIdx.x >> 5) & 1;
  const uint32_t pt = threadIdx.x & 63;
  const uint64_t gpair = (uint64_t)blockIdx.x * kStreamPairs + pair;
  const uint64_t npairs = (uint64_t)gridDim.x * kStreamPairs;
  const uint64_t gwarp = 2 * gpair + half;
  PairSmem* sm = reinterpret_cast<PairSmem*>(s_dyn) + pair;
  sm->touched[2 * pt] = 0;
  sm->touched[2 * pt + 1] = 0;
  if (pt == 0) sm->flag = 0;

  uint32_t j = 0xFFFFFFFFu, cur = 0xFFFFFFFFu;
  uint64_t ck = 0;
  int b = 0;
  // prologue: the first chunk's old data and slot (the pair's 64 threads hold its 64
  // 16-byte pieces: the header in piece 0, entries 4 p - 4 .. 4 p - 1 in piece p)
  uint4 pre = make_uint4(0, 0, 0, 0);
  uint32_t pre_hdr = 0;
  if (gpair < total_chunks) {
    const uint32_t j0 = find_job(chunk_start, k, gpair);
    issue_chunk(sm->buf[0], jobs[j0].old, jobs[j0].n, (gpair - chunk_start[j0]) * kChunk, pt);
    pre = reinterpret_cast<const uint4*>(slots + gpair * kSlotBytes)[pt];
    pre_hdr = *reinterpret_cast<const uint32_t*>(slots + gpair * kSlotBytes);
  }
  cp_async_commit();
  for (uint64_t g = gpair; g < total_chunks; g += npairs, b ^= 1) {
    j = advance_job(chunk_start, k, j, g);
    const uint4 cur_pre = pre;
    const uint32_t hdr = pre_hdr;
    // the next chunk's old data goes into the other buffer, its slot into registers
    const uint64_t gn = g + npairs;
    if (gn < total_chunks) {
      const uint32_t jn = advance_job(chunk_start, k, j, gn);
      issue_chunk(sm->buf[b ^ 1], jobs[jn].old, jobs[jn].n, (gn - chunk_start[jn]) * kChunk, pt);
      pre = reinterpret_cast<const uint4*>(slots + gn * kSlotBytes)[pt];
      pre_hdr = *reinterpret_cast<const uint32_t*>(slots + gn * kSlotBytes);
    }
    cp_async_commit();
    const DJob& J = jobs[j];
    const uint64_t n = J.n;
    const uint64_t e0 = (g - chunk_start[j]) * kChunk;
    // this chunk's copies (every group but the one just issued) must land before its buffer
    // is read, or reused two iterations later when the chunk is skipped
    cp_async_wait<1>();
    pair_sync(pair);
    if (info[j].status != BD_OK || (hdr & (kSlotOverflow | kSlotBad))) continue;
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
    const uint32_t kk = (hdr & 0xFFFu) + ((hdr >> 12) & 0xFFFu);  // M + R entries
    uint32_t* data32 = reinterpret_cast<uint32_t*>(sm->buf[b]);
    bool taken = false;
    if (pt > 0) {
      const uint32_t i0 = 4 * pt - 4;  // entries held in this thread's piece of the slot
      if (i0 + 0 < kk) taken |= xor_entry(data32, sm->touched, cur_pre.x);
      if (i0 + 1 < kk) taken |= xor_entry(data32, sm->touched, cur_pre.y);
      if (i0 + 2 < kk) taken |= xor_entry(data32, sm->touched, cur_pre.z);
      if (i0 + 3 < kk) taken |= xor_entry(data32, sm->touched, cur_pre.w);
    }
    if (taken) sm->flag = 1;
    pair_sync(pair);
    if (sm->flag == 0) {
      uint16_t* __restrict__ out = J.out;
      const bool inplace = out == J.old;
      if (e0 + kChunk <= n) {
        stream_two_steps<true>(sm->buf[b], sm->touched, 4 * half, e0, n, out, inplace, ck);
        stream_two_steps<true>(sm->buf[b], sm->touched, 4 * half + 2, e0, n, out, inplace, ck);
      } else {
        stream_two_steps<false>(sm->buf[b], sm->touched, 4 * half, e0, n, out, inplace, ck);
        stream_two_steps<false>(sm->buf[b], sm->touched, 4 * half + 2, e0, n, out, inplace, ck);
      }
    } else if (pt == 0) {
      record_status(&info[j].chunk_err, BD_ERR_FORMAT);
    }
    pair_sync(pair);
    sm->touched[2 * pt] = 0;
    sm->touched[2 * pt + 1] = 0;
    if (pt == 0) sm->flag = 0;
  }
  cp_async_wait<0>();
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
  constexpr size_t smem = kStreamPairs * sizeof(PairSmem);  // ~66 KiB
  static const int per_sm = [] {
    if (cudaFuncSetAttribute(k_apply_stream, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return 0;
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, k_apply_stream, kStreamThreads, smem) !=
            cudaSuccess || v < 1)
      v = 1;
    return v;
  }();
  if (per_sm == 0) return cudaErrorInvalidValue;
  const uint64_t grid = std::min<uint64_t>((c.chunks + kStreamPairs - 1) / kStreamPairs,
                                           (uint64_t)per_sm * c.sms);
  k_apply_stream<<<(unsigned)grid, kStreamThreads, smem, c.stream>>>(
      reinterpret_cast<const DJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start), c.k, c.chunks,
      reinterpret_cast<JobInfo*>(c.ws + c.lay.info), c.ws + c.lay.slots, c.ws + c.lay.ck);
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
