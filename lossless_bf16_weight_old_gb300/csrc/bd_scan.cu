// bd_scan.cu -- the count scan of libbf16delta, shared by compress and decompress.
//
// The payload sections are laid out chunk-major, so every chunk needs the exclusive prefix of
// four per-chunk quantities over the chunks before it in its tensor: position-section bytes
// P_c (two version-1 blocks, or a compact block of version 3 or 4), mantissa-only count M_c, rare
// count R_c and escaped gaps E_c (X-stream values of a compact block, else 0).
//   scan_tiles  one CTA per tile of 1024 chunks: per-chunk prefix inside the tile, tile total.
//               Compress decides here which chunks of a version-3 or -4 payload are compact.  For
//               decompress the counts come from the untrusted payload, so it also checks
//               that the count table lies inside the payload, that each entry is well formed
//               for the version and that M_c + R_c <= L_c.
//   scan_jobs   one warp per tensor: prefix of the tile totals, section offsets and the
//               payload size.  Compress writes the header, the size and the checksum of new;
//               decompress checks the header against the count table and the size given.
#include <algorithm>

#include "bd_internal.cuh"

namespace bd {
namespace {

constexpr int kThreads = 256;

struct JobView {
  uint64_t n, nchunks, chunk_base;
  const uint8_t* payload;
  uint64_t size;
};

template <bool DEC>
__device__ __forceinline__ JobView view(const void* jobs, uint32_t j) {
  JobView v;
  if (DEC) {
    const DJob& J = reinterpret_cast<const DJob*>(jobs)[j];
    v.n = J.n; v.nchunks = J.nchunks; v.chunk_base = J.chunk_base;
    v.payload = J.payload; v.size = J.size;
  } else {
    const CJob& J = reinterpret_cast<const CJob*>(jobs)[j];
    v.n = J.n; v.nchunks = J.nchunks; v.chunk_base = J.chunk_base;
    v.payload = nullptr; v.size = 0;
  }
  return v;
}

// Version of a payload as the scan reads it (0 when too short to hold one).
__device__ __forceinline__ uint32_t payload_version(const uint8_t* payload, uint64_t size) {
  return size >= 16 ? reinterpret_cast<const uint32_t*>(payload)[2] : 0;
}

template <bool DEC>
__global__ void __launch_bounds__(kThreads)
k_scan_tiles(const void* __restrict__ jobs, const uint64_t* __restrict__ tile_start, uint32_t k,
             uint64_t total_tiles, const uint32_t* __restrict__ counts_ws, uint4* __restrict__ loc,
             TileSum* __restrict__ tile_tot, JobInfo* __restrict__ info) {
  __shared__ uint32_t s_w[kThreads / 32][4];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  for (uint64_t u = blockIdx.x; u < total_tiles; u += gridDim.x) {
    const uint32_t j = find_job(tile_start, k, u);
    const JobView J = view<DEC>(jobs, j);
    const uint64_t c0 = (u - tile_start[j]) * kTileChunks;
    const uint64_t c1 = min(c0 + kTileChunks, J.nchunks);
    const uint32_t* cnt;
    uint32_t version;
    if (DEC) {
      // the header length follows the version (checked again with the whole header in
      // scan_jobs); the count table must lie inside the payload
      version = payload_version(J.payload, J.size);
      if (J.size < header_bytes(version) + 4 * J.nchunks) {
        if (t == 0) record_status(&info[j].status, BD_ERR_FORMAT);
        continue;
      }
      cnt = reinterpret_cast<const uint32_t*>(J.payload + header_bytes(version));
    } else {
      version = reinterpret_cast<const CJob*>(jobs)[j].version;
      cnt = counts_ws + J.chunk_base;
    }

    uint32_t vP[4], vM[4], vR[4], vE[4];
    uint32_t sP = 0, sM = 0, sR = 0, sE = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const uint64_t c = c0 + 4 * t + i;
      vP[i] = vM[i] = vR[i] = vE[i] = 0;
      if (c < c1) {
        const uint32_t v = cnt[c];
        const uint64_t L64 = J.n - c * kChunk;
        const uint32_t L = L64 < kChunk ? (uint32_t)L64 : kChunk;
        const uint32_t B = (L + 7) >> 3;
        ChunkCount cc{};
        if (DEC) {
          cc = parse_count(v, version);
          if (cc.bad || cc.M + cc.R > L) bad = true;
        } else {
          cc.M = wcount_m(v);
          cc.R = wcount_r(v);
          if (version == 4) {
            cc.M = v4count_m(v);
            cc.R = v4count_r(v);
            cc.compact = cc.rice = rice_compact(v, B);
            cc.nb = (v >> 21) & 0x3FFu;
          } else {
            cc.compact = version == 3 && choose_compact(cc.M, cc.R, wcount_e(v), B);
            cc.E = cc.compact ? wcount_e(v) : 0;
          }
        }
        vM[i] = cc.M;
        vR[i] = cc.R;
        vE[i] = cc.E;
        vP[i] = chunk_pos_bytes(cc, B);
      }
      sP += vP[i]; sM += vM[i]; sR += vR[i]; sE += vE[i];
    }
    // block-wide exclusive scan of (sP, sM, sR, sE) in thread order
    const uint32_t iP = warp_incl_scan(sP), iM = warp_incl_scan(sM), iR = warp_incl_scan(sR),
                   iE = warp_incl_scan(sE);
    if (lane == 31) { s_w[w][0] = iP; s_w[w][1] = iM; s_w[w][2] = iR; s_w[w][3] = iE; }
    __syncthreads();
    uint32_t bP = 0, bM = 0, bR = 0, bE = 0, tP = 0, tM = 0, tR = 0, tE = 0;
    for (int q = 0; q < kThreads / 32; q++) {
      if (q < w) { bP += s_w[q][0]; bM += s_w[q][1]; bR += s_w[q][2]; bE += s_w[q][3]; }
      tP += s_w[q][0]; tM += s_w[q][1]; tR += s_w[q][2]; tE += s_w[q][3];
    }
    uint32_t eP = bP + iP - sP, eM = bM + iM - sM, eR = bR + iR - sR, eE = bE + iE - sE;
#pragma unroll
    for (int i = 0; i < 4; i++) {
      const uint64_t c = c0 + 4 * t + i;
      if (c < c1) loc[J.chunk_base + c] = make_uint4(eP, eM, eR, eE);
      eP += vP[i]; eM += vM[i]; eR += vR[i]; eE += vE[i];
    }
    if (t == 0) tile_tot[u] = TileSum{tP, tM, tR, tE};
    if (bad) record_status(&info[j].status, BD_ERR_FORMAT);
    __syncthreads();
  }
}

__device__ __forceinline__ uint64_t warp_incl_scan64(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint64_t o = __shfl_up_sync(0xFFFFFFFFu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

template <bool DEC>
__global__ void __launch_bounds__(kThreads)
k_scan_jobs(const void* __restrict__ jobs, const uint64_t* __restrict__ tile_start, uint32_t k,
            const TileSum* __restrict__ tile_tot, TileSum* __restrict__ tile_pre,
            JobInfo* __restrict__ info, const uint8_t* __restrict__ ck_base,
            int32_t* __restrict__ status_all, uint32_t* __restrict__ v3_flag) {
  const int lane = threadIdx.x & 31;
  const uint64_t gwarp = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const uint64_t nwarps = ((uint64_t)gridDim.x * kThreads) >> 5;
  for (uint64_t jj = gwarp; jj < k; jj += nwarps) {
    const uint32_t j = (uint32_t)jj;
    const uint64_t tb = tile_start[j], U = tile_start[j + 1] - tb;
    uint64_t rP = 0, rM = 0, rR = 0, rE = 0;
    for (uint64_t b = 0; b < U; b += 32) {
      TileSum ts{0, 0, 0, 0};
      if (b + lane < U) ts = tile_tot[tb + b + lane];
      const uint64_t iP = warp_incl_scan64(ts.p), iM = warp_incl_scan64(ts.m),
                     iR = warp_incl_scan64(ts.r), iE = warp_incl_scan64(ts.e);
      if (b + lane < U) tile_pre[tb + b + lane] = TileSum{rP + iP - ts.p, rM + iM - ts.m,
                                                          rR + iR - ts.r, rE + iE - ts.e};
      rP += __shfl_sync(0xFFFFFFFFu, iP, 31);
      rM += __shfl_sync(0xFFFFFFFFu, iM, 31);
      rR += __shfl_sync(0xFFFFFFFFu, iR, 31);
      rE += __shfl_sync(0xFFFFFFFFu, iE, 31);
    }
    if (lane != 0) continue;

    JobInfo I{};
    I.sum_p = rP; I.sum_m = rM; I.sum_r = rR; I.sum_e = rE;
    I.chunk_err = 0;
    if (!DEC) {
      finish_compress_job(reinterpret_cast<const CJob*>(jobs)[j], j, I, ck_base, info,
                          status_all);
    } else {
      const DJob& J = reinterpret_cast<const DJob*>(jobs)[j];
      int32_t st = info[j].status;
      const uint32_t version = payload_version(J.payload, J.size);
      const uint64_t hdr = header_bytes(version);
      I.version = version;
      const uint64_t flags = version >= 2 && J.size >= kHeaderV2
                                 ? reinterpret_cast<const uint64_t*>(J.payload)[9] : 0;
      I.flags = (uint32_t)(flags & kFlagOverwrite);
      // the general apply build decodes compact blocks and applies overwrites
      if (version >= 3 || I.flags != 0) *v3_flag = 1u;
      if (I.flags != 0) v3_flag[kFlagOwWord - kFlagV3Word] = 1u;
      I.r_start = hdr + 4 * J.nchunks;
      I.x_start = I.r_start + 2 * rR;
      I.p_start = I.x_start + 2 * rE;
      I.m_start = I.p_start + rP;
      I.total = I.m_start + (7 * rM + 7) / 8;
      if (J.size < hdr) {
        st = BD_ERR_FORMAT;
      } else if (st == BD_OK) {
        const uint64_t* h = reinterpret_cast<const uint64_t*>(J.payload);
        const bool ok = h[0] == kMagic && version >= 1 && version <= 4 &&
                        h[1] == ((uint64_t)version | ((uint64_t)kChunk << 32)) &&
                        h[2] == J.n && h[3] == J.nchunks && h[4] == rM && h[5] == rR &&
                        h[6] == rP && h[7] == J.size && I.total == J.size &&
                        (version == 1 || (h[9] & ~(uint64_t)kFlagOverwrite) == 0);
        if (!ok) st = BD_ERR_FORMAT;
        // a payload bound to a base version is applied incrementally to that version only
        else if (version >= 2 && J.d_ck_old && h[8] != *J.d_ck_old) st = BD_ERR_BASE;
      }
      I.status = st;
      info[j] = I;
    }
  }
}

template <typename K>
int blocks_per_sm(K kernel) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return per_sm;
}

}  // namespace

cudaError_t launch_scan_tiles(const LaunchCtx& c, bool decompress) {
  if (c.tiles == 0) return cudaSuccess;
  const void* jobs = c.ws + c.lay.jobs;
  const uint64_t* ts = reinterpret_cast<const uint64_t*>(c.ws + c.lay.tile_start);
  const uint32_t* counts = decompress ? nullptr : reinterpret_cast<const uint32_t*>(c.ws + c.lay.counts);
  uint4* loc = reinterpret_cast<uint4*>(c.ws + c.lay.loc);
  TileSum* tt = reinterpret_cast<TileSum*>(c.ws + c.lay.tile_tot);
  JobInfo* info = reinterpret_cast<JobInfo*>(c.ws + c.lay.info);
  if (decompress) {
    static const int per_sm = blocks_per_sm(k_scan_tiles<true>);
    const uint64_t grid = std::min<uint64_t>(c.tiles, (uint64_t)per_sm * c.sms);
    k_scan_tiles<true><<<(unsigned)grid, kThreads, 0, c.stream>>>(jobs, ts, c.k, c.tiles, counts,
                                                                 loc, tt, info);
  } else {
    static const int per_sm = blocks_per_sm(k_scan_tiles<false>);
    const uint64_t grid = std::min<uint64_t>(c.tiles, (uint64_t)per_sm * c.sms);
    k_scan_tiles<false><<<(unsigned)grid, kThreads, 0, c.stream>>>(jobs, ts, c.k, c.tiles, counts,
                                                                  loc, tt, info);
  }
  return cudaGetLastError();
}

cudaError_t launch_scan_jobs(const LaunchCtx& c, bool decompress, int32_t* d_status_all) {
  const void* jobs = c.ws + c.lay.jobs;
  const uint64_t* ts = reinterpret_cast<const uint64_t*>(c.ws + c.lay.tile_start);
  const TileSum* tt = reinterpret_cast<const TileSum*>(c.ws + c.lay.tile_tot);
  TileSum* tp = reinterpret_cast<TileSum*>(c.ws + c.lay.tile_pre);
  JobInfo* info = reinterpret_cast<JobInfo*>(c.ws + c.lay.info);
  const uint64_t warps_per_block = kThreads / 32;
  const uint64_t grid = std::min<uint64_t>((c.k + warps_per_block - 1) / warps_per_block,
                                      (uint64_t)8 * c.sms);
  if (decompress)
    k_scan_jobs<true><<<(unsigned)grid, kThreads, 0, c.stream>>>(
        jobs, ts, c.k, tt, tp, info, c.ws + c.lay.ck, d_status_all,
        reinterpret_cast<uint32_t*>(c.ws + c.lay.overflow) + kFlagV3Word);
  else
    k_scan_jobs<false><<<(unsigned)grid, kThreads, 0, c.stream>>>(
        jobs, ts, c.k, tt, tp, info, c.ws + c.lay.ck, d_status_all, nullptr);
  return cudaGetLastError();
}

}  // namespace bd
