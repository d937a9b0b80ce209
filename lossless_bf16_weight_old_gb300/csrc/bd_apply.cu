// bd_apply.cu -- decompress (apply) kernels of libbf16delta.
//
// "GPU-accelerated Weight Teleportation", section "Delta update algebra": the rollout side
// XORs the mask into its old weights to obtain the new ones.  "Every byte counts: ARCv3 and
// the case for cross-region RL": both streams are applied to the previous checkpoint and the
// result is checksummed against the trainer's original.
//
//   apply         one CTA per 4096-element chunk (persistent loop): reads the old chunk,
//                 decodes the M and R position blocks (delta list -> prefix sum, or bitmap ->
//                 popcount rank), gathers the 7-bit and 16-bit XOR values, builds the chunk's
//                 XOR mask in shared memory, XORs it in, checksums the result and writes back
//                 only the 16-byte groups that changed (in place) or the whole chunk (out of
//                 place).  Malformed chunks are detected before any write and left unwritten.
//   apply_finish  one thread per tensor: checks the M-stream pad bits, compares the checksum
//                 with the expected value and publishes the status.
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
k_apply(const DJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
        const uint64_t* __restrict__ tile_start, uint32_t k, uint64_t total_chunks,
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

  for (uint64_t g = blockIdx.x; g < total_chunks; g += gridDim.x) {
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

}  // namespace

cudaError_t launch_apply(const LaunchCtx& c) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm = [] {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, k_apply, kThreads, 0) != cudaSuccess ||
        v < 1)
      v = 1;
    return v;
  }();
  const uint64_t grid = std::min<uint64_t>(c.chunks, (uint64_t)per_sm * c.sms);
  k_apply<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const DJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.tile_start), c.k, c.chunks,
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
