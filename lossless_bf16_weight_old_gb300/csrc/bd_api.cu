// bd_api.cu -- the C ABI of libbf16delta (include/bf16delta.h): argument checks, workspace
// layout, the per-call tensor table and the kernel sequence of each operation.
//
// Operations follow "Every byte counts: ARCv3 and the case for cross-region RL" (API listing:
// delta_compress(src, dst) -> (compressed_diff, checksum); delta_decompress(src,
// compressed_diff, checksum) -> restored) and "GPU-accelerated Weight Teleportation",
// section "Delta update algebra" (old XOR mask = new).
#include <algorithm>
#include <cstring>
#include <memory>
#include <vector>

#include "bd_internal.cuh"
#include "bf16delta_debug.h"

namespace bd {
namespace {

constexpr uint64_t kAlign = 256;
inline uint64_t up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

struct Sizes {
  uint64_t chunks = 0, tiles = 0, batches = 0;
  uint32_t bchunks = 1;
};

// Chunks per batch of the fused compress: as many as keep about four batches per resident warp
// (32 per SM), at most kMaxBatchChunks.  Fewer, larger batches cost less to hand out and to
// publish; small calls keep one warp per chunk.  The workspace size assumes the smallest.
uint32_t batch_chunks(uint64_t chunks, int sms) {
  const uint64_t per = chunks / ((uint64_t)(sms > 0 ? sms : 1) * 32 * 4);
  return (uint32_t)(per < 1 ? 1 : per > kMaxBatchChunks ? kMaxBatchChunks : per);
}

bool sizes_of(const uint64_t* ns, uint32_t k, Sizes& s, uint32_t bchunks = 1) {
  s = Sizes{};
  s.bchunks = bchunks;
  for (uint32_t i = 0; i < k; i++) {
    const uint64_t n = ns[i];
    if (n > BD_MAX_ELEMS) return false;
    const uint64_t C = (n + kChunk - 1) / kChunk;
    s.chunks += C;
    s.tiles += (C + kTileChunks - 1) / kTileChunks;
    s.batches += tensor_batches(C, bchunks);
  }
  return true;
}

WsLayout make_layout(uint32_t k, const Sizes& s, bool compress) {
  WsLayout L{};
  uint64_t off = 0;
  L.state = off;
  L.ck = off;
  off = up(off + (uint64_t)k * kCkBytes, kAlign);
  L.info = off;
  off = up(off + (uint64_t)k * sizeof(JobInfo), kAlign);
  L.overflow = off;  // count of chunks listed for the dense kernels (+ selection words)
  off = up(off + 16, kAlign);
  if (compress) {
    L.fused_ctl = off;
    off = up(off + ((uint64_t)kCtlTensors + 2 * (uint64_t)k) * 4, kAlign);
  }
  L.state_bytes = off - L.state;
  L.jobs = off;
  off = up(off + (uint64_t)k * 128, kAlign);
  L.chunk_start = off;
  off = up(off + ((uint64_t)k + 1) * 8, kAlign);
  L.tile_start = off;
  off = up(off + ((uint64_t)k + 1) * 8, kAlign);
  if (compress) {   // uploaded with the tensor table
    L.batch_start = off;
    off = up(off + ((uint64_t)k + 1) * 8, kAlign);
  }
  L.loc = off;
  off = up(off + s.chunks * 16, kAlign);
  L.tile_tot = off;
  off = up(off + s.tiles * sizeof(TileSum), kAlign);
  L.tile_pre = off;
  off = up(off + s.tiles * sizeof(TileSum), kAlign);
  L.ovf_list = off;  // chunks too dense for a slot / for the thread-level apply
  off = up(off + s.chunks * 4, kAlign);
  L.ovf_job = off;   // their tensors
  off = up(off + s.chunks * 4, kAlign);
  if (compress) {
    L.slots = off;
    off = up(off + s.chunks * kSlotBytes, kAlign);
    L.counts = off;
    off = up(off + s.chunks * 4, kAlign);
    L.batch_tot = off;
    off = up(off + s.batches * 16, kAlign);
    L.batch_pre = off;
    off = up(off + s.batches * sizeof(TileSum), kAlign);
  }
  L.total = off;
  return L;
}

// ---- host -> device upload of the tensor table through kernel parameters -----------------
// Kernel parameters are copied at launch, so the host table may be released as soon as the
// call returns and no pageable-memory copy (which may synchronise) is involved.
constexpr uint32_t kBlobWords = 30 * 1024 / 16;
struct Blob {
  uint32_t words;
  uint32_t pad[3];
  uint4 data[kBlobWords];
};

// One 16-byte word per thread, spread over several blocks: the words of the parameter blob
// differ from thread to thread and the constant cache serves one address at a time, so a
// single block looping over a 30 KiB blob took about 8 µs per launch.
__global__ void k_put(const __grid_constant__ Blob b, uint4* __restrict__ dst) {
  const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < b.words) dst[i] = b.data[i];
}

cudaError_t upload(const std::vector<uint8_t>& host, uint8_t* dst, cudaStream_t s) {
  static_assert(sizeof(Blob) <= 32000, "kernel parameter limit");
  const uint64_t words = host.size() / 16;
  std::unique_ptr<Blob> b(new Blob);
  for (uint64_t w0 = 0; w0 < words; w0 += kBlobWords) {
    const uint32_t cnt = (uint32_t)((words - w0) < kBlobWords ? (words - w0) : kBlobWords);
    b->words = cnt;
    std::memcpy(b->data, host.data() + w0 * 16, (size_t)cnt * 16);
    k_put<<<(cnt + 127) / 128, 128, 0, s>>>(*b, reinterpret_cast<uint4*>(dst) + w0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// [a, a+na) and [b, b+nb) intersect
inline bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

int check(cudaError_t e) { return e == cudaSuccess ? BD_OK : BD_ERR_CUDA; }

// -------------------------------------------------------------------------------- compress
// bases == nullptr: version 1; else version `format & 0xFF` (2, or 3 or 4 with compact
// position blocks), an overwrite payload when format has BD_FORMAT_OVERWRITE.  stall < k: the
// fused compress with tensor `stall` never published (bd_debug_compress_stall).
constexpr uint32_t kNoStall = 0xFFFFFFFFu;
int compress_impl(const bd_compress_item* items, const uint64_t* const* bases, uint32_t format,
                  uint32_t k, void* ws, uint64_t ws_bytes, int32_t* status_all, cudaStream_t s,
                  uint32_t stall = kNoStall) {
  if (k > 0 && items == nullptr) return BD_ERR_INVALID_ARG;
  const uint32_t vfmt = format & 0xFFu;
  const bool overwrite = bases && (format & BD_FORMAT_OVERWRITE) != 0;
  if (bases && (vfmt < 2 || vfmt > 4 || (format & ~(0xFFu | BD_FORMAT_OVERWRITE)) != 0))
    return BD_ERR_INVALID_ARG;
  const uint32_t version = bases ? vfmt : 1;
  if (bases)
    for (uint32_t i = 0; i < k; i++)
      if (!bases[i] || !aligned(bases[i], 8)) return BD_ERR_INVALID_ARG;
  std::vector<uint64_t> ns(k);
  for (uint32_t i = 0; i < k; i++) {
    const bd_compress_item& it = items[i];
    if (it.n > BD_MAX_ELEMS) return BD_ERR_INVALID_ARG;
    if (it.n > 0 && (!it.d_old || !it.d_new || !aligned(it.d_old, 16) || !aligned(it.d_new, 16)))
      return BD_ERR_INVALID_ARG;
    if (it.cap > 0 && (!it.d_payload || !aligned(it.d_payload, 16))) return BD_ERR_INVALID_ARG;
    if (!it.d_size || !it.d_checksum) return BD_ERR_INVALID_ARG;
    if (overlaps(it.d_payload, it.cap, it.d_old, 2 * it.n) ||
        overlaps(it.d_payload, it.cap, it.d_new, 2 * it.n))
      return BD_ERR_INVALID_ARG;
    ns[i] = it.n;
  }
  // (the layout for one-chunk batches, the most there can be, is the size the caller was told)
  Sizes sz;
  if (!sizes_of(ns.data(), k, sz)) return BD_ERR_INVALID_ARG;
  const WsLayout lay = make_layout(k, sz, true);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < lay.total) return BD_ERR_INVALID_ARG;
  for (uint32_t i = 0; i < k; i++)
    if (overlaps(items[i].d_payload, items[i].cap, ws, lay.total)) return BD_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms <= 0) return BD_ERR_CUDA;
  const uint32_t bchunks = batch_chunks(sz.chunks, sms);

  // tensor table
  std::vector<uint8_t> host(lay.loc - lay.jobs, 0);
  CJob* jobs = reinterpret_cast<CJob*>(host.data());
  uint64_t* cstart = reinterpret_cast<uint64_t*>(host.data() + (lay.chunk_start - lay.jobs));
  uint64_t* tstart = reinterpret_cast<uint64_t*>(host.data() + (lay.tile_start - lay.jobs));
  uint64_t* bstart = reinterpret_cast<uint64_t*>(host.data() + (lay.batch_start - lay.jobs));
  uint64_t cb = 0, tb = 0, bb = 0, most_batches = 0;
  for (uint32_t i = 0; i < k; i++) {
    const bd_compress_item& it = items[i];
    CJob& J = jobs[i];
    J.old = it.d_old;
    J.neu = it.d_new;
    J.payload = static_cast<uint8_t*>(it.d_payload);
    J.n = it.n;
    J.cap = it.cap;
    J.d_size = it.d_size;
    J.d_checksum = it.d_checksum;
    J.d_status = it.d_status;
    J.d_base = bases ? bases[i] : nullptr;
    J.version = version;
    J.flags = overwrite ? kFlagOverwrite : 0;
    J.nchunks = (it.n + kChunk - 1) / kChunk;
    J.chunk_base = cb;
    J.tile_base = tb;
    cstart[i] = cb;
    tstart[i] = tb;
    bstart[i] = bb;
    cb += J.nchunks;
    tb += (J.nchunks + kTileChunks - 1) / kTileChunks;
    bb += tensor_batches(J.nchunks, bchunks);
    most_batches = std::max(most_batches, tensor_batches(J.nchunks, bchunks));
  }
  cstart[k] = cb;
  tstart[k] = tb;
  bstart[k] = bb;
  if (stall != kNoStall && (stall >= k || bases || most_batches > kMaxFusedBatches))
    return BD_ERR_INVALID_ARG;   // (the hook needs a call that takes the fused compress)

  uint8_t* w = static_cast<uint8_t*>(ws);
  LaunchCtx c{s, sms, w, lay, k, sz.chunks, sz.tiles, bb, bchunks};
  int rc;
  if ((rc = check(cudaMemsetAsync(w + lay.state, 0, lay.state_bytes, s)))) return rc;
  if (status_all && (rc = check(cudaMemsetAsync(status_all, 0, sizeof(int32_t), s)))) return rc;
  if (k == 0) return BD_OK;
  if ((rc = check(upload(host, w + lay.jobs, s)))) return rc;
  // the kernel builds: version 4, version 3 (also every overwrite payload of version 2), or
  // the XOR payloads of versions 1 and 2
  const uint32_t fmt = version == 4 ? 4u : (version == 3 || overwrite) ? 3u : 0u;
  if (most_batches <= kMaxFusedBatches) {   // the fused compress, then the dense chunks
    // the hook: tensor `stall` starts with a chunk count that never reaches its chunks
    if (stall != kNoStall &&
        (rc = check(cudaMemsetAsync(w + lay.fused_ctl + 4 * (kCtlTensors + 2 * (uint64_t)stall),
                                    0x80, 4, s))))
      return rc;
    if ((rc = check(launch_compress_fused(c, fmt, overwrite, status_all)))) return rc;
    return check(launch_emit_dense(c, true));
  }
  if ((rc = check(launch_encode_slots(c, fmt, overwrite)))) return rc;
  if ((rc = check(launch_scan_tiles(c, false)))) return rc;
  if ((rc = check(launch_scan_jobs(c, false, status_all)))) return rc;
  if ((rc = check(launch_emit(c, fmt, overwrite)))) return rc;
  return check(launch_emit_dense(c));
}

// ------------------------------------------------------------------------------ decompress
// One tensor of a decompress call, from either public item type.
struct DecItem {
  const uint16_t* old;
  uint16_t* out;
  uint64_t n;
  const void* payload;
  uint64_t size;
  const uint64_t* expected;
  const uint64_t* ck_old;   // incremental verification only
  uint64_t* ck_out;         // incremental verification only (optional)
  int32_t* status;
};

int decompress_impl(const DecItem* items, uint32_t k, void* ws, uint64_t ws_bytes,
                    int32_t* status_all, cudaStream_t s, bool incremental,
                    bool clear_status = true) {
  if (k > 0 && items == nullptr) return BD_ERR_INVALID_ARG;
  if (!status_all || !aligned(status_all, 4)) return BD_ERR_INVALID_ARG;
  std::vector<uint64_t> ns(k);
  for (uint32_t i = 0; i < k; i++) {
    const DecItem& it = items[i];
    if (it.n > BD_MAX_ELEMS) return BD_ERR_INVALID_ARG;
    if (it.n > 0 && (!it.old || !it.out || !aligned(it.old, 16) || !aligned(it.out, 16)))
      return BD_ERR_INVALID_ARG;
    if (it.out != it.old && overlaps(it.out, 2 * it.n, it.old, 2 * it.n))
      return BD_ERR_INVALID_ARG;
    if (it.size > 0 && (!it.payload || !aligned(it.payload, 16))) return BD_ERR_INVALID_ARG;
    if (overlaps(it.out, 2 * it.n, it.payload, it.size)) return BD_ERR_INVALID_ARG;
    if (!it.expected || !aligned(it.expected, 8)) return BD_ERR_INVALID_ARG;
    if (incremental) {
      if (it.out != it.old || !it.ck_old || !aligned(it.ck_old, 8)) return BD_ERR_INVALID_ARG;
      if (it.ck_out && !aligned(it.ck_out, 8)) return BD_ERR_INVALID_ARG;
    }
    ns[i] = it.n;
  }
  Sizes sz;
  if (!sizes_of(ns.data(), k, sz)) return BD_ERR_INVALID_ARG;
  const WsLayout lay = make_layout(k, sz, false);
  if (!ws || !aligned(ws, kAlign) || ws_bytes < lay.total) return BD_ERR_INVALID_ARG;
  for (uint32_t i = 0; i < k; i++)
    if (overlaps(items[i].out, 2 * items[i].n, ws, lay.total)) return BD_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms <= 0) return BD_ERR_CUDA;

  std::vector<uint8_t> host(lay.loc - lay.jobs, 0);
  DJob* jobs = reinterpret_cast<DJob*>(host.data());
  uint64_t* cstart = reinterpret_cast<uint64_t*>(host.data() + (lay.chunk_start - lay.jobs));
  uint64_t* tstart = reinterpret_cast<uint64_t*>(host.data() + (lay.tile_start - lay.jobs));
  uint64_t cb = 0, tb = 0;
  bool any_out_of_place = false;
  for (uint32_t i = 0; i < k; i++) {
    const DecItem& it = items[i];
    if (it.out != it.old) any_out_of_place = true;
    DJob& J = jobs[i];
    J.old = it.old;
    J.out = it.out;
    J.payload = static_cast<const uint8_t*>(it.payload);
    J.n = it.n;
    J.size = it.size;
    J.d_expected = it.expected;
    J.d_status = it.status;
    J.d_ck_old = incremental ? it.ck_old : nullptr;
    J.d_ck_out = incremental ? it.ck_out : nullptr;
    J.nchunks = (it.n + kChunk - 1) / kChunk;
    J.chunk_base = cb;
    J.tile_base = tb;
    cstart[i] = cb;
    tstart[i] = tb;
    cb += J.nchunks;
    tb += (J.nchunks + kTileChunks - 1) / kTileChunks;
  }
  cstart[k] = cb;
  tstart[k] = tb;

  uint8_t* w = static_cast<uint8_t*>(ws);
  LaunchCtx c{s, sms, w, lay, k, sz.chunks, sz.tiles};
  int rc;
  if ((rc = check(cudaMemsetAsync(w + lay.state, 0, lay.state_bytes, s)))) return rc;
  if (clear_status && (rc = check(cudaMemsetAsync(status_all, 0, sizeof(int32_t), s)))) return rc;
  if (k == 0) return BD_OK;
  if ((rc = check(upload(host, w + lay.jobs, s)))) return rc;
  if ((rc = check(launch_scan_tiles(c, true)))) return rc;
  if ((rc = check(launch_scan_jobs(c, true, nullptr)))) return rc;
  if (any_out_of_place && (rc = check(launch_copy_jobs(c)))) return rc;
  if (incremental) {
    if ((rc = check(launch_apply_incremental(c)))) return rc;
  } else {
    if ((rc = check(launch_apply_chunks(c)))) return rc;
  }
  if ((rc = check(launch_apply_bitmap(c, incremental)))) return rc;
  return check(launch_apply_finish(c, status_all));
}

// Events of one streamed decompress, destroyed when the call returns (the runtime releases an
// event's resources once the work recorded on it has completed).
struct StreamEvents {
  cudaEvent_t e[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  ~StreamEvents() {
    for (cudaEvent_t& x : e)
      if (x) cudaEventDestroy(x);
  }
  cudaError_t create() {
    for (cudaEvent_t& x : e) {
      const cudaError_t r = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
      if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
  }
};

// bd_decompress_batch with the payloads in host memory, streamed through two device slots:
// the items are cut, in order, into groups whose payloads (each at a 256-byte boundary) fit
// one slot; group g's payloads are copied into slot g % 2 on the copy stream while the apply
// of group g - 1 runs on the compute stream, and group g's apply waits for its copies only.
// A slot is refilled (group g + 2) once the apply that read it is done.
int decompress_streamed_impl(const bd_decompress_item* items, uint32_t k, void* staging,
                             uint64_t slot_bytes, void* ws, uint64_t ws_bytes,
                             int32_t* status_all, cudaStream_t s, cudaStream_t cs) {
  if (k > 0 && !items) return BD_ERR_INVALID_ARG;
  if (!status_all || !aligned(status_all, 4)) return BD_ERR_INVALID_ARG;
  if (!cs || cs == s) return BD_ERR_INVALID_ARG;   // a stream of its own for the copies
  if (k > 0 && (!staging || !aligned(staging, kAlign) || slot_bytes == 0 ||
                slot_bytes % 256 != 0 || slot_bytes > (1ull << 40)))
    return BD_ERR_INVALID_ARG;
  // everything checked before anything is enqueued (the per-group calls then cannot refuse)
  std::vector<uint64_t> ns(k);
  std::vector<uint32_t> group_start;
  uint64_t used = 0;
  for (uint32_t i = 0; i < k; i++) {
    const bd_decompress_item& it = items[i];
    if (it.n > BD_MAX_ELEMS) return BD_ERR_INVALID_ARG;
    if (it.n > 0 && (!it.d_old || !it.d_out || !aligned(it.d_old, 16) || !aligned(it.d_out, 16)))
      return BD_ERR_INVALID_ARG;
    if (it.d_out != it.d_old && overlaps(it.d_out, 2 * it.n, it.d_old, 2 * it.n))
      return BD_ERR_INVALID_ARG;
    if (it.size > 0 && !it.d_payload) return BD_ERR_INVALID_ARG;
    if (!it.d_expected || !aligned(it.d_expected, 8)) return BD_ERR_INVALID_ARG;
    if (overlaps(it.d_out, 2 * it.n, staging, 2 * slot_bytes)) return BD_ERR_INVALID_ARG;
    const uint64_t need = up(it.size, 256);
    if (need > slot_bytes) return BD_ERR_INVALID_ARG;   // a payload larger than a slot
    if (i == 0 || used + need > slot_bytes) {
      group_start.push_back(i);
      used = 0;
    }
    used += need;
    ns[i] = it.n;
  }
  group_start.push_back(k);
  Sizes sz;
  if (!sizes_of(ns.data(), k, sz)) return BD_ERR_INVALID_ARG;
  const WsLayout lay = make_layout(k, sz, false);   // covers the layout of every group
  if (!ws || !aligned(ws, kAlign) || ws_bytes < lay.total) return BD_ERR_INVALID_ARG;
  if (k > 0 && overlaps(ws, lay.total, staging, 2 * slot_bytes)) return BD_ERR_INVALID_ARG;
  for (uint32_t i = 0; i < k; i++)
    if (overlaps(items[i].d_out, 2 * items[i].n, ws, lay.total)) return BD_ERR_INVALID_ARG;

  int rc;
  if ((rc = check(cudaMemsetAsync(status_all, 0, sizeof(int32_t), s)))) return rc;
  if (k == 0) return BD_OK;
  StreamEvents ev;   // 0, 1: slot copied; 2, 3: slot free; 4: the call's start
  if ((rc = check(ev.create()))) return rc;
  // the copies may not overwrite a slot that work enqueued before this call still reads
  if ((rc = check(cudaEventRecord(ev.e[4], s)))) return rc;
  if ((rc = check(cudaStreamWaitEvent(cs, ev.e[4], 0)))) return rc;
  uint8_t* const base = static_cast<uint8_t*>(staging);
  std::vector<DecItem> dec;
  for (size_t g = 0; g + 1 < group_start.size(); g++) {
    const uint32_t slot = (uint32_t)(g & 1), i0 = group_start[g], i1 = group_start[g + 1];
    uint8_t* const sb = base + slot * slot_bytes;
    if (g >= 2 && (rc = check(cudaStreamWaitEvent(cs, ev.e[2 + slot], 0)))) return rc;
    dec.clear();
    // one copy per run of payloads laid out in host memory as they go into the slot (each at
    // the slot offset's distance from the run's first): thousands of small tensors would
    // otherwise cost one host call each
    uint64_t off = 0, run_off = 0, run_len = 0;
    const uint8_t* run_src = nullptr;
    for (uint32_t i = i0; i < i1; i++) {
      const bd_decompress_item& x = items[i];
      const uint8_t* src = static_cast<const uint8_t*>(x.d_payload);
      if (x.size > 0) {
        if (run_src && src == run_src + (off - run_off)) {
          run_len = off - run_off + x.size;
        } else {
          if (run_src && (rc = check(cudaMemcpyAsync(sb + run_off, run_src, run_len,
                                                     cudaMemcpyHostToDevice, cs))))
            return rc;
          run_src = src;
          run_off = off;
          run_len = x.size;
        }
      }
      dec.push_back(DecItem{x.d_old, x.d_out, x.n, sb + off, x.size, x.d_expected, nullptr,
                            nullptr, x.d_status});
      off += up(x.size, 256);
    }
    if (run_src &&
        (rc = check(cudaMemcpyAsync(sb + run_off, run_src, run_len, cudaMemcpyHostToDevice, cs))))
      return rc;
    if ((rc = check(cudaEventRecord(ev.e[slot], cs)))) return rc;
    if ((rc = check(cudaStreamWaitEvent(s, ev.e[slot], 0)))) return rc;
    if ((rc = decompress_impl(dec.data(), i1 - i0, ws, ws_bytes, status_all, s, false, false)))
      return rc;
    if ((rc = check(cudaEventRecord(ev.e[2 + slot], s)))) return rc;
  }
  return BD_OK;
}

uint64_t le64(const uint8_t* p) {
  uint64_t v = 0;
  for (int i = 0; i < 8; i++) v |= (uint64_t)p[i] << (8 * i);
  return v;
}

}  // namespace
}  // namespace bd

using namespace bd;

extern "C" {

uint64_t bd_compress_bound(uint64_t n) {
  if (n > BD_MAX_ELEMS) return 0;
  const uint64_t C = (n + kChunk - 1) / kChunk;
  const uint64_t full = n / kChunk, tail = n % kChunk;
  const uint64_t bitmaps = full * kChunkBitmap + (tail + 7) / 8;
  // per chunk: 2 bytes per R element + 7/8 byte per M element <= 2 bytes per element, and
  // at most two bitmaps of position bytes; one byte of M-stream rounding
  return kHeaderV2 + 4 * C + 2 * n + 2 * bitmaps + 1;
}

uint64_t bd_compress_workspace_size(const uint64_t* h_n, uint32_t k) {
  if (k > 0 && !h_n) return 0;
  Sizes s;
  if (!sizes_of(h_n, k, s)) return 0;
  return make_layout(k, s, true).total;
}

uint64_t bd_decompress_workspace_size(const uint64_t* h_n, uint32_t k) {
  if (k > 0 && !h_n) return 0;
  Sizes s;
  if (!sizes_of(h_n, k, s)) return 0;
  return make_layout(k, s, false).total;
}

int bd_compress(const uint16_t* d_old, const uint16_t* d_new, uint64_t n, void* d_payload,
                uint64_t cap, void* d_ws, uint64_t ws_bytes, uint64_t* d_size,
                uint64_t* d_checksum, int32_t* d_status, void* stream) {
  bd_compress_item it{d_old, d_new, n, d_payload, cap, d_size, d_checksum, nullptr};
  return compress_impl(&it, nullptr, 1, 1, d_ws, ws_bytes, d_status,
                       static_cast<cudaStream_t>(stream));
}

int bd_compress_batch(const bd_compress_item* h_items, uint32_t k, void* d_ws,
                      uint64_t ws_bytes, int32_t* d_status, void* stream) {
  return compress_impl(h_items, nullptr, 1, k, d_ws, ws_bytes, d_status,
                       static_cast<cudaStream_t>(stream));
}

int bd_debug_compress_stall(const bd_compress_item* h_items, uint32_t k, uint32_t stall,
                            void* d_ws, uint64_t ws_bytes, int32_t* d_status, void* stream) {
  if (stall >= k) return BD_ERR_INVALID_ARG;
  return compress_impl(h_items, nullptr, 1, k, d_ws, ws_bytes, d_status,
                       static_cast<cudaStream_t>(stream), stall);
}

int bd_compress_versioned(const uint16_t* d_old, const uint16_t* d_new, uint64_t n,
                          void* d_payload, uint64_t cap, void* d_ws, uint64_t ws_bytes,
                          uint64_t* d_size, uint64_t* d_checksum,
                          const uint64_t* d_base_checksum, uint32_t format, int32_t* d_status,
                          void* stream) {
  bd_compress_item it{d_old, d_new, n, d_payload, cap, d_size, d_checksum, nullptr};
  const uint64_t* bases[1] = {d_base_checksum};
  return compress_impl(&it, bases, format, 1, d_ws, ws_bytes, d_status,
                       static_cast<cudaStream_t>(stream));
}

int bd_compress_versioned_batch(const bd_compress_item* h_items,
                                const uint64_t* const* h_base_checksums, uint32_t k,
                                uint32_t format, void* d_ws, uint64_t ws_bytes,
                                int32_t* d_status, void* stream) {
  if (k > 0 && !h_base_checksums) return BD_ERR_INVALID_ARG;
  return compress_impl(h_items, h_base_checksums, format, k, d_ws, ws_bytes, d_status,
                       static_cast<cudaStream_t>(stream));
}

int bd_decompress(const uint16_t* d_old, uint64_t n, const void* d_payload, uint64_t size,
                  const uint64_t* d_expected, uint16_t* d_out, void* d_ws, uint64_t ws_bytes,
                  int32_t* d_status, void* stream) {
  DecItem it{d_old, d_out, n, d_payload, size, d_expected, nullptr, nullptr, nullptr};
  return decompress_impl(&it, 1, d_ws, ws_bytes, d_status, static_cast<cudaStream_t>(stream),
                         false);
}

int bd_decompress_batch(const bd_decompress_item* h_items, uint32_t k, void* d_ws,
                        uint64_t ws_bytes, int32_t* d_status, void* stream) {
  if (k > 0 && !h_items) return BD_ERR_INVALID_ARG;
  std::vector<DecItem> it(k);
  for (uint32_t i = 0; i < k; i++) {
    const bd_decompress_item& x = h_items[i];
    it[i] = DecItem{x.d_old, x.d_out, x.n, x.d_payload, x.size, x.d_expected, nullptr, nullptr,
                    x.d_status};
  }
  return decompress_impl(it.data(), k, d_ws, ws_bytes, d_status,
                         static_cast<cudaStream_t>(stream), false);
}

int bd_decompress_batch_streamed(const bd_decompress_item* h_items, uint32_t k, void* d_staging,
                                 uint64_t slot_bytes, void* d_ws, uint64_t ws_bytes,
                                 int32_t* d_status, void* stream, void* copy_stream) {
  return decompress_streamed_impl(h_items, k, d_staging, slot_bytes, d_ws, ws_bytes, d_status,
                                  static_cast<cudaStream_t>(stream),
                                  static_cast<cudaStream_t>(copy_stream));
}

int bd_decompress_incremental(uint16_t* d_w, uint64_t n, const void* d_payload, uint64_t size,
                              const uint64_t* d_ck_old, const uint64_t* d_expected,
                              uint64_t* d_ck_out, void* d_ws, uint64_t ws_bytes,
                              int32_t* d_status, void* stream) {
  DecItem it{d_w, d_w, n, d_payload, size, d_expected, d_ck_old, d_ck_out, nullptr};
  return decompress_impl(&it, 1, d_ws, ws_bytes, d_status, static_cast<cudaStream_t>(stream),
                         true);
}

int bd_decompress_incremental_batch(const bd_incremental_item* h_items, uint32_t k, void* d_ws,
                                    uint64_t ws_bytes, int32_t* d_status, void* stream) {
  if (k > 0 && !h_items) return BD_ERR_INVALID_ARG;
  std::vector<DecItem> it(k);
  for (uint32_t i = 0; i < k; i++) {
    const bd_incremental_item& x = h_items[i];
    it[i] = DecItem{x.d_w, x.d_w, x.n, x.d_payload, x.size, x.d_expected, x.d_ck_old,
                    x.d_ck_out, x.d_status};
  }
  return decompress_impl(it.data(), k, d_ws, ws_bytes, d_status,
                         static_cast<cudaStream_t>(stream), true);
}

int bd_checksum(const uint16_t* d_w, uint64_t n, uint64_t* d_out, void* stream) {
  if (!d_out || !aligned(d_out, 8) || n > BD_MAX_ELEMS) return BD_ERR_INVALID_ARG;
  if (n > 0 && (!d_w || !aligned(d_w, 16))) return BD_ERR_INVALID_ARG;
  const int sms = sm_count();
  if (sms <= 0) return BD_ERR_CUDA;
  return check(launch_checksum(d_w, n, d_out, static_cast<cudaStream_t>(stream), sms));
}

int bd_payload_info(const void* h_header, uint64_t bytes, bd_payload_info_t* out) {
  if (!h_header || !out || bytes < kHeader) return BD_ERR_INVALID_ARG;
  const uint8_t* p = static_cast<const uint8_t*>(h_header);
  if (std::memcmp(p, "BF16DLT1", 8) != 0) return BD_ERR_FORMAT;
  bd_payload_info_t I;
  I.version = (uint32_t)(le64(p + 8) & 0xFFFFFFFFu);
  I.chunk_elems = (uint32_t)(le64(p + 8) >> 32);
  I.n = le64(p + 16);
  I.chunks = le64(p + 24);
  I.n_mant = le64(p + 32);
  I.n_rare = le64(p + 40);
  I.position_bytes = le64(p + 48);
  I.total_size = le64(p + 56);
  I.base_checksum = 0;
  I.n_escapes = 0;
  I.flags = 0;
  if (I.version < 1 || I.version > 4 || I.chunk_elems != kChunk || I.n > BD_MAX_ELEMS)
    return BD_ERR_FORMAT;
  const uint64_t hdr = I.version >= 2 ? kHeaderV2 : kHeader;
  if (I.version >= 2) {
    if (bytes < kHeaderV2) return BD_ERR_INVALID_ARG;
    I.base_checksum = le64(p + 64);
    I.flags = le64(p + 72);
    if ((I.flags & ~(uint64_t)kFlagOverwrite) != 0) return BD_ERR_FORMAT;
  }
  if (I.chunks != (I.n + kChunk - 1) / kChunk) return BD_ERR_FORMAT;
  if (I.n_mant > I.n || I.n_rare > I.n - I.n_mant) return BD_ERR_FORMAT;
  if (I.position_bytes > 2 * (uint64_t)kChunkBitmap * I.chunks) return BD_ERR_FORMAT;
  const uint64_t want = hdr + 4 * I.chunks + 2 * I.n_rare + I.position_bytes +
                        (7 * I.n_mant + 7) / 8;
  if (I.version == 3) {
    // the X stream's length is not in the header: whatever the other sections leave, in u16
    // values, at most kCompactMax per chunk
    if (I.total_size < want || (I.total_size - want) % 2 != 0 ||
        (I.total_size - want) / 2 > (uint64_t)kCompactMax * I.chunks)
      return BD_ERR_FORMAT;
    I.n_escapes = (I.total_size - want) / 2;
  } else if (want != I.total_size) {
    return BD_ERR_FORMAT;
  }
  *out = I;
  return BD_OK;
}

int bd_status_sync(const int32_t* d_status, void* stream) {
  if (!d_status) return BD_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return BD_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, d_status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return BD_ERR_CUDA;
  return v;
}

const char* bd_status_string(int code) {
  switch (code) {
    case BD_OK: return "ok";
    case BD_ERR_INVALID_ARG: return "invalid argument";
    case BD_ERR_CAPACITY: return "payload larger than the capacity given";
    case BD_ERR_FORMAT: return "malformed payload";
    case BD_ERR_CHECKSUM: return "checksum mismatch";
    case BD_ERR_CUDA: return "CUDA error";
    case BD_ERR_BASE: return "payload bound to another base version";
    default: return "unknown status";
  }
}

}  // extern "C"
