// bd_checksum.cu -- the standalone checksum of libbf16delta.
//
// "Every byte counts: ARCv3 and the case for cross-region RL": the rollout side checksums the
// reconstructed weights against the trainer's original.  The checksum is a wrapping sum of
// position-keyed SplitMix64 mixes of 64-bit words (definition in include/bf16delta.h), so
// every CTA can reduce its share independently and add it with one atomic.
#include "bd_internal.cuh"

namespace bd {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
k_checksum(const uint16_t* __restrict__ w, uint64_t n, unsigned long long* __restrict__ out) {
  __shared__ uint64_t s_part[kThreads / 32];
  const uint64_t groups = (n + 7) >> 3, words = (n + 3) >> 2;
  uint64_t acc = 0;
  const uint64_t stride = (uint64_t)gridDim.x * kThreads;
  uint64_t q = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
  // two groups in flight per thread
  for (; q + stride < groups; q += 2 * stride) {
    const uint4 a = load8_stream(w, 8 * q, n);
    const uint4 b = load8_stream(w, 8 * (q + stride), n);
    acc += group_hash(a, q, words) + group_hash(b, q + stride, words);
  }
  if (q < groups) acc += group_hash(load8_stream(w, 8 * q, n), q, words);
  acc = warp_sum64(acc);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t tot = 0;
    for (int i = 0; i < kThreads / 32; i++) tot += s_part[i];
    atomicAdd(out, (unsigned long long)tot);
  }
}

}  // namespace

cudaError_t launch_checksum(const uint16_t* w, uint64_t n, uint64_t* out, cudaStream_t s,
                            int sms) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(uint64_t), s);
  if (e != cudaSuccess || n == 0) return e;
  static const int per_sm = [] {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, k_checksum, kThreads, 0) !=
            cudaSuccess || v < 1)
      v = 1;
    return v;
  }();
  const uint64_t groups = (n + 7) >> 3;
  uint64_t grid = (uint64_t)per_sm * sms;
  const uint64_t need = (groups + kThreads - 1) / kThreads;
  if (need < grid) grid = need;
  k_checksum<<<(unsigned)grid, kThreads, 0, s>>>(w, n, reinterpret_cast<unsigned long long*>(out));
  return cudaGetLastError();
}

}  // namespace bd
