// bd_encode.cu -- compress kernels of libbf16delta.
//
// "Every byte counts: ARCv3 and the case for cross-region RL", figure "How ARCv3 encodes a
// block of weights": XOR each old/new pair, classify by the changed field, omit unchanged
// values, keep only the mantissa bits of mantissa-only changes and pack exponent/sign changes
// separately as one block; the API returns a checksum beside the payload.
//
// Three passes, none of which waits on another CTA:
//   encode_slots  reads old and new once (the only full-size read): per 4096-element chunk
//                 it counts the M and R classes, accumulates the checksum of new and stores
//                 the chunk's nonzero XORs (position, value) in a fixed 1 KiB slot of the
//                 workspace; a chunk with more changes than a slot holds is marked overflow.
//   (count scan in bd_scan.cu: per-chunk offsets of every section, header, size.)
//   emit          writes the count table, the R stream and the position blocks straight to
//                 their final payload offsets and stages the 7-bit M values as bytes;
//                 overflow chunks re-read old/new instead of the slot.
//   pack_mant     packs the staged M bytes into the 7-bit stream; each output byte is
//                 written by the chunk that holds the element its first bit belongs to.
#include "bd_internal.cuh"

namespace bd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint64_t* ck_slot(uint8_t* ck_base, uint32_t job, uint64_t salt) {
  return reinterpret_cast<uint64_t*>(ck_base + (uint64_t)job * kCkBytes) +
         (salt & (kCkSlots - 1)) * kCkStride;
}

// ------------------------------------------------------------------------ encode_slots
__global__ void __launch_bounds__(kThreads)
k_encode_slots(const CJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
               uint32_t k, uint64_t total_chunks, uint32_t* __restrict__ counts,
               uint8_t* __restrict__ slots, uint8_t* __restrict__ ck_base) {
  const int lane = threadIdx.x & 31;
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;

  uint32_t cur_job = 0xFFFFFFFFu;
  uint64_t ck = 0;
  for (uint64_t g = gwarp; g < total_chunks; g += nwarps) {
    const uint32_t j = find_job(chunk_start, k, g);
    if (j != cur_job) {
      if (cur_job != 0xFFFFFFFFu) {
        uint64_t s = warp_sum64(ck);
        if (lane == 0) atomicAdd(reinterpret_cast<unsigned long long*>(ck_slot(ck_base, cur_job, gwarp)),
                                 (unsigned long long)s);
      }
      cur_job = j;
      ck = 0;
    }
    const uint16_t* __restrict__ old = jobs[j].old;
    const uint16_t* __restrict__ neu = jobs[j].neu;
    const uint64_t n = jobs[j].n;
    const uint64_t c = g - chunk_start[j];
    const uint64_t e0 = c * kChunk;
    const uint64_t words = (n + 3) >> 2;
    uint32_t* __restrict__ slot = reinterpret_cast<uint32_t*>(slots + g * kSlotBytes);

    uint32_t running = 0, mcnt = 0, rcnt = 0;
    // two-stage register pipeline over the 8 steps of 512 elements
    uint64_t e = e0 + lane * 16;
    uint4 o0 = load8_stream(old, e, n), o1 = load8_stream(old, e + 8, n);
    uint4 n0 = load8_stream(neu, e, n), n1 = load8_stream(neu, e + 8, n);
#pragma unroll 1
    for (int s = 0; s < 8; s++) {
      uint4 po0 = o0, po1 = o1, pn0 = n0, pn1 = n1;
      if (s < 7) {
        const uint64_t en = e0 + (s + 1) * 512 + lane * 16;
        o0 = load8_stream(old, en, n); o1 = load8_stream(old, en + 8, n);
        n0 = load8_stream(neu, en, n); n1 = load8_stream(neu, en + 8, n);
      }
      const uint32_t eloc = s * 512 + lane * 16;
      const uint64_t q = (e0 + eloc) >> 3;
      ck += group_hash(pn0, q, words) + group_hash(pn1, q + 1, words);
      const uint4 x0 = make_uint4(po0.x ^ pn0.x, po0.y ^ pn0.y, po0.z ^ pn0.z, po0.w ^ pn0.w);
      const uint4 x1 = make_uint4(po1.x ^ pn1.x, po1.y ^ pn1.y, po1.z ^ pn1.z, po1.w ^ pn1.w);
      uint32_t m0, r0, m1, r1;
      classify8(x0, m0, r0);
      classify8(x1, m1, r1);
      const uint32_t mm = m0 | (m1 << 8), rm = r0 | (r1 << 8), nz = mm | rm;
      mcnt += __popc(mm);
      rcnt += __popc(rm);
      const uint32_t cnt = __popc(nz);
      const uint32_t incl = warp_incl_scan(cnt);
      const uint32_t tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
      uint32_t idx = running + incl - cnt;
      uint32_t bits = nz;
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        if (idx < kSlotEntries) {
          const uint32_t xv = elem_of(b < 8 ? x0 : x1, b & 7);
          slot[1 + idx] = ((eloc + b) << 16) | xv;
        }
        idx++;
      }
      running += tot;
    }
    mcnt = warp_incl_scan(mcnt);
    rcnt = warp_incl_scan(rcnt);
    if (lane == 31) {
      counts[g] = mcnt | (rcnt << 16);
      slot[0] = running > kSlotEntries ? (kSlotOverflow | kSlotEntries) : running;
    }
  }
  if (cur_job != 0xFFFFFFFFu) {
    uint64_t s = warp_sum64(ck);
    if (lane == 0) atomicAdd(reinterpret_cast<unsigned long long*>(ck_slot(ck_base, cur_job, gwarp)),
                             (unsigned long long)s);
  }
}

// ------------------------------------------------------------------------ emit

// Where one chunk's output goes.
struct EmitCtx {
  uint8_t* mblk;       // M position block
  uint8_t* rblk;       // R position block
  uint16_t* rstream;   // R stream at this chunk's first R element
  uint8_t* mbytes;     // staged M bytes at this chunk's first M element
  uint32_t* bm;        // shared bitmaps of this warp: [0..128) M, [128..256) R
  uint32_t M, R;       // the chunk's counts: no write goes past them
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
      if (cx.listM) {
        store_u16(cx.mblk + 2 * rm, (uint16_t)(pos - (uint32_t)prevM));
      } else {
        atomicOr(&cx.bm[pos >> 5], 1u << (pos & 31));
      }
      cx.mbytes[rm] = (uint8_t)(x & kMant);
      prevM = (int32_t)pos;
      rm++;
    } else {
      if (rr >= cx.R) continue;
      if (cx.listR) {
        store_u16(cx.rblk + 2 * rr, (uint16_t)(pos - (uint32_t)prevR));
      } else {
        atomicOr(&cx.bm[128 + (pos >> 5)], 1u << (pos & 31));
      }
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

__global__ void __launch_bounds__(kThreads)
k_emit(const CJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
       const uint64_t* __restrict__ tile_start, uint32_t k, uint64_t total_chunks,
       const uint32_t* __restrict__ counts, const uint8_t* __restrict__ slots,
       const uint4* __restrict__ loc, const TileSum* __restrict__ tile_pre,
       const JobInfo* __restrict__ info, uint8_t* __restrict__ mbytes) {
  __shared__ uint32_t s_bm[kWarps][256];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  uint32_t* bm = s_bm[wib];

  for (uint64_t g = gwarp; g < total_chunks; g += nwarps) {
    const uint32_t j = find_job(chunk_start, k, g);
    if (info[j].status != BD_OK) continue;
    const CJob& J = jobs[j];
    const uint64_t n = J.n;
    const uint64_t c = g - chunk_start[j];
    const uint64_t e0 = c * kChunk;
    const uint32_t L = (uint32_t)((n - e0) < kChunk ? (n - e0) : kChunk);
    const uint32_t B = (L + 7) >> 3;
    const uint32_t cnt = counts[g];
    const uint32_t M = cnt & 0xFFFFu, R = cnt >> 16;
    const TileSum pre = tile_pre[tile_start[j] + c / kTileChunks];
    const uint4 lc = loc[g];
    const uint64_t Pex = pre.p + lc.x, Mex = pre.m + lc.y, Rex = pre.r + lc.z;
    uint8_t* payload = J.payload;
    if (lane == 0) reinterpret_cast<uint32_t*>(payload + kHeader)[c] = cnt;

    EmitCtx cx;
    cx.listM = 2 * M < B;
    cx.listR = 2 * R < B;
    cx.mblk = payload + info[j].p_start + Pex;
    cx.rblk = cx.mblk + block_bytes(M, B);
    cx.rstream = reinterpret_cast<uint16_t*>(payload + info[j].r_start) + Rex;
    cx.mbytes = mbytes + J.m_base + Mex;
    cx.bm = bm;
    cx.M = M;
    cx.R = R;
    if (!cx.listM || !cx.listR) {
      for (int i = lane; i < 256; i += 32) bm[i] = 0;
      __syncwarp();
    }
    EmitState st{0, 0, 0, 0};

    const uint32_t* slot = reinterpret_cast<const uint32_t*>(slots + g * kSlotBytes);
    const uint32_t hdr = slot[0];
    if (!(hdr & kSlotOverflow)) {
      const uint32_t kk = hdr;
      for (uint32_t base = 0; base < kk; base += 32) {
        const uint32_t i = base + lane;
        uint32_t ent = 0, mm = 0, rmk = 0;
        if (i < kk) {
          ent = slot[1 + i];
          const uint32_t x = ent & 0xFFFFu;
          if (x & kSignExp) rmk = 1; else mm = 1;
        }
        emit_batch(ent >> 16, mm, rmk, [ent](int) { return ent & 0xFFFFu; }, st, cx);
      }
    } else {
      // Overflow: derive the chunk's changes again from old and new.
      const uint16_t* __restrict__ old = J.old;
      const uint16_t* __restrict__ neu = J.neu;
      for (int s = 0; s < 8; s++) {
        const uint32_t eloc = s * 512 + lane * 16;
        const uint64_t e = e0 + eloc;
        const uint4 o0 = load8(old, e, n), o1 = load8(old, e + 8, n);
        const uint4 n0 = load8(neu, e, n), n1 = load8(neu, e + 8, n);
        const uint4 x0 = make_uint4(o0.x ^ n0.x, o0.y ^ n0.y, o0.z ^ n0.z, o0.w ^ n0.w);
        const uint4 x1 = make_uint4(o1.x ^ n1.x, o1.y ^ n1.y, o1.z ^ n1.z, o1.w ^ n1.w);
        uint32_t m0, r0, m1, r1;
        classify8(x0, m0, r0);
        classify8(x1, m1, r1);
        emit_batch(eloc, m0 | (m1 << 8), r0 | (r1 << 8),
                   [x0, x1](int b) { return elem_of(b < 8 ? x0 : x1, b & 7); }, st, cx);
      }
    }
    if (!cx.listM || !cx.listR) {
      __syncwarp();
      if (!cx.listM) store_bitmap(cx.mblk, bm, B);
      if (!cx.listR) store_bitmap(cx.rblk, bm + 128, B);
      __syncwarp();
    }
  }
}

// ------------------------------------------------------------------------ pack_mant
__global__ void __launch_bounds__(kThreads)
k_pack_mant(const CJob* __restrict__ jobs, const uint64_t* __restrict__ chunk_start,
            const uint64_t* __restrict__ tile_start, uint32_t k, uint64_t total_chunks,
            const uint32_t* __restrict__ counts, const uint4* __restrict__ loc,
            const TileSum* __restrict__ tile_pre, const JobInfo* __restrict__ info,
            const uint8_t* __restrict__ mbytes) {
  const int lane = threadIdx.x & 31;
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  for (uint64_t g = gwarp; g < total_chunks; g += nwarps) {
    const uint32_t M = counts[g] & 0xFFFFu;
    if (M == 0) continue;
    const uint32_t j = find_job(chunk_start, k, g);
    if (info[j].status != BD_OK) continue;
    const uint64_t c = g - chunk_start[j];
    const TileSum pre = tile_pre[tile_start[j] + c / kTileChunks];
    const uint64_t Mex = pre.m + loc[g].y;
    const uint64_t sum_m = info[j].sum_m;
    const uint8_t* __restrict__ mb = mbytes + jobs[j].m_base;
    uint8_t* out = jobs[j].payload + info[j].m_start;
    // this chunk owns the bytes whose first bit lies in one of its elements
    const uint64_t b0 = (7 * Mex + 7) >> 3;
    const uint64_t b1 = (7 * (Mex + M) + 7) >> 3;
    for (uint64_t b = b0 + lane; b < b1; b += 32) {
      const uint64_t jj = (8 * b) / 7;
      const uint32_t s = (uint32_t)(8 * b - 7 * jj);
      const uint32_t v0 = mb[jj];
      const uint32_t v1 = (jj + 1 < sum_m) ? mb[jj + 1] : 0u;
      out[b] = (uint8_t)((v0 >> s) | (v1 << (7 - s)));
    }
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

cudaError_t launch_encode_slots(const LaunchCtx& c) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm = blocks_per_sm(k_encode_slots, kThreads);
  const uint64_t grid = cap_grid((uint64_t)per_sm * c.sms, kWarps, c.chunks);
  k_encode_slots<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const CJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start), c.k, c.chunks,
      reinterpret_cast<uint32_t*>(c.ws + c.lay.counts), c.ws + c.lay.slots, c.ws + c.lay.ck);
  return cudaGetLastError();
}

cudaError_t launch_emit(const LaunchCtx& c) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm = blocks_per_sm(k_emit, kThreads);
  const uint64_t grid = cap_grid((uint64_t)per_sm * c.sms, kWarps, c.chunks);
  k_emit<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const CJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.tile_start), c.k, c.chunks,
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.counts), c.ws + c.lay.slots,
      reinterpret_cast<const uint4*>(c.ws + c.lay.loc),
      reinterpret_cast<const TileSum*>(c.ws + c.lay.tile_pre),
      reinterpret_cast<const JobInfo*>(c.ws + c.lay.info), c.ws + c.lay.mbytes);
  return cudaGetLastError();
}

cudaError_t launch_pack_mant(const LaunchCtx& c) {
  if (c.chunks == 0) return cudaSuccess;
  static const int per_sm = blocks_per_sm(k_pack_mant, kThreads);
  const uint64_t grid = cap_grid((uint64_t)per_sm * c.sms, kWarps, c.chunks);
  k_pack_mant<<<(unsigned)grid, kThreads, 0, c.stream>>>(
      reinterpret_cast<const CJob*>(c.ws + c.lay.jobs),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.chunk_start),
      reinterpret_cast<const uint64_t*>(c.ws + c.lay.tile_start), c.k, c.chunks,
      reinterpret_cast<const uint32_t*>(c.ws + c.lay.counts),
      reinterpret_cast<const uint4*>(c.ws + c.lay.loc),
      reinterpret_cast<const TileSum*>(c.ws + c.lay.tile_pre),
      reinterpret_cast<const JobInfo*>(c.ws + c.lay.info), c.ws + c.lay.mbytes);
  return cudaGetLastError();
}

}  // namespace bd
