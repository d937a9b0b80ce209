// bd_noalloc.cu -- bd_decompress_noalloc: the apply path without a caller workspace.
//
// Some callers cannot allocate device memory: an inference engine whose allocator has
// already reserved nearly all of HBM for weights and KV cache, or any process where a
// cudaMalloc would fail, fragment the engine's pool or stall the device.  This entry point
// takes its scratch from one fixed array in the library's device memory instead of a
// workspace argument.  It runs the same scan kernels as bd_decompress and applies every
// chunk with the block-level decoder, which needs only a few bytes of scratch per chunk.
#include <algorithm>

#include "bd_internal.cuh"

namespace bd {
namespace {

// The scratch array.  In host code `g_scratch` names a host-side stand-in, not a device
// address: the device address is looked up with cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_scratch[BD_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  It is looked up on every call
// (a cheap host call) rather than cached, so that a device reset or a re-created primary
// context never leaves a stale address behind; the first lookup on a device also loads the
// library's module there.
int scratch_address(uint8_t** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
  if (e != cudaSuccess || p == nullptr) return BD_ERR_CUDA;
  *out = static_cast<uint8_t*>(p);
  return BD_OK;
}

inline uint64_t up256(uint64_t x) { return (x + 255) / 256 * 256; }

// Scratch layout for one tensor of at most BD_NOALLOC_MAX_ELEMS elements (no slots).
WsLayout noalloc_layout(uint64_t chunks, uint64_t tiles) {
  WsLayout L{};
  uint64_t off = 0;
  L.state = off;
  L.ck = off;
  off = up256(off + kCkBytes);
  L.info = off;
  off = up256(off + sizeof(JobInfo));
  L.overflow = off;
  off = up256(off + 16);
  L.state_bytes = off - L.state;
  L.jobs = off;
  off = up256(off + sizeof(DJob));
  L.chunk_start = off;
  off = up256(off + 2 * sizeof(uint64_t));
  L.tile_start = off;
  off = up256(off + 2 * sizeof(uint64_t));
  L.loc = off;
  off = up256(off + chunks * 16);
  L.tile_tot = off;
  off = up256(off + tiles * sizeof(TileSum));
  L.tile_pre = off;
  off = up256(off + tiles * sizeof(TileSum));
  L.ovf_list = off;
  off = up256(off + chunks * 4);
  L.slots = 0;
  L.counts = 0;
  L.total = off;
  return L;
}

constexpr uint64_t kMaxChunks = BD_NOALLOC_MAX_ELEMS / kChunk;
static_assert(kMaxChunks * (16 + 4) + 8 * 1024 + 2 * 64 * ((kMaxChunks + kTileChunks - 1) / kTileChunks) <=
                  BD_NOALLOC_SCRATCH_BYTES,
              "scratch array too small for BD_NOALLOC_MAX_ELEMS");

// Writes the one-tensor table into the scratch and lists every chunk for the block decoder.
__global__ void k_noalloc_setup(const DJob job, DJob* __restrict__ jobs,
                                uint64_t* __restrict__ chunk_start,
                                uint64_t* __restrict__ tile_start, uint32_t* __restrict__ count,
                                uint32_t* __restrict__ list, uint32_t chunks, uint32_t tiles) {
  const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t == 0) {
    jobs[0] = job;
    chunk_start[0] = 0;
    chunk_start[1] = chunks;
    tile_start[0] = 0;
    tile_start[1] = tiles;
    *count = chunks;
  }
  for (uint32_t i = t; i < chunks; i += gridDim.x * blockDim.x) list[i] = i;
}

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}
inline bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && x < y + nb && y < x + na;
}
int check(cudaError_t e) { return e == cudaSuccess ? BD_OK : BD_ERR_CUDA; }

}  // namespace
}  // namespace bd

using namespace bd;

extern "C" int bd_decompress_noalloc(const uint16_t* d_old, uint64_t n, const void* d_payload,
                                     uint64_t size, const uint64_t* d_expected, uint16_t* d_out,
                                     int32_t* d_status, void* stream) {
  if (n > BD_NOALLOC_MAX_ELEMS) return BD_ERR_INVALID_ARG;  // larger than the scratch covers
  if (!d_status || !aligned(d_status, 4) || !d_expected || !aligned(d_expected, 8))
    return BD_ERR_INVALID_ARG;
  if (n > 0 && (!d_old || !d_out || !aligned(d_old, 16) || !aligned(d_out, 16)))
    return BD_ERR_INVALID_ARG;
  if (d_out != d_old && overlaps(d_out, 2 * n, d_old, 2 * n)) return BD_ERR_INVALID_ARG;
  if (size > 0 && (!d_payload || !aligned(d_payload, 16))) return BD_ERR_INVALID_ARG;
  if (overlaps(d_out, 2 * n, d_payload, size)) return BD_ERR_INVALID_ARG;

  uint8_t* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != BD_OK) return rc;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return BD_ERR_CUDA;

  const uint64_t chunks = (n + kChunk - 1) / kChunk;
  const uint64_t tiles = (chunks + kTileChunks - 1) / kTileChunks;
  const WsLayout lay = noalloc_layout(chunks, tiles);
  if (lay.total > BD_NOALLOC_SCRATCH_BYTES) return BD_ERR_INVALID_ARG;

  DJob job{};
  job.old = d_old;
  job.out = d_out;
  job.payload = static_cast<const uint8_t*>(d_payload);
  job.n = n;
  job.size = size;
  job.d_expected = d_expected;
  job.d_status = nullptr;
  job.chunk_base = 0;
  job.nchunks = chunks;
  job.tile_base = 0;

  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchCtx c{s, sms, scratch, lay, 1u, chunks, tiles};
  // the scratch keeps the previous call's contents: clear the accumulators and the status
  if ((rc = check(cudaMemsetAsync(scratch + lay.state, 0, lay.state_bytes, s)))) return rc;
  if ((rc = check(cudaMemsetAsync(d_status, 0, sizeof(int32_t), s)))) return rc;
  const unsigned setup_grid = (unsigned)(chunks > 0 ? std::min<uint64_t>((chunks + 255) / 256, 1024) : 1);
  k_noalloc_setup<<<setup_grid, 256, 0, s>>>(
      job, reinterpret_cast<DJob*>(scratch + lay.jobs),
      reinterpret_cast<uint64_t*>(scratch + lay.chunk_start),
      reinterpret_cast<uint64_t*>(scratch + lay.tile_start),
      reinterpret_cast<uint32_t*>(scratch + lay.overflow),
      reinterpret_cast<uint32_t*>(scratch + lay.ovf_list), (uint32_t)chunks, (uint32_t)tiles);
  if ((rc = check(cudaGetLastError()))) return rc;
  if ((rc = check(launch_scan_tiles(c, true)))) return rc;
  if ((rc = check(launch_scan_jobs(c, true, nullptr)))) return rc;
  if (d_out != d_old && (rc = check(launch_copy_jobs(c)))) return rc;
  if ((rc = check(launch_apply(c)))) return rc;
  return check(launch_apply_finish(c, d_status));
}
