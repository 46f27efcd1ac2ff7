// probe.cu -- a streaming-read probe: how fast one kernel of the GEMM's shape
// (one CTA per SM, a ring of bulk copies into shared memory) can read a
// buffer from HBM when it does nothing else.  The benchmark reads as many
// bytes as the layer's GEMM launch streams and reports the GEMM's bandwidth
// against it, next to the copy-bandwidth peak.
#include <cstdint>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kProbeStage = 18432;  // bytes per copy: the narrow-tile GEMM's weight stage
constexpr int kProbeRing = 8;

// CTA c reads chunks c, c + gridDim.x, ... of kProbeStage bytes.  Warp 0's
// elected lane issues the copies, warp 1 waits for each and frees its slot.
__global__ void __launch_bounds__(64, 1) stream_probe_kernel(const uint8_t* __restrict__ src, long long nchunks,
                                                              int* __restrict__ status, unsigned* __restrict__ sink) {
  extern __shared__ __align__(1024) uint8_t ring[];
  __shared__ __align__(8) uint64_t bars[2 * kProbeRing];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto full = [&](int r) { return smem_u32(&bars[r]); };
  auto empty = [&](int r) { return smem_u32(&bars[kProbeRing + r]); };
  if (threadIdx.x == 0) {
    for (int r = 0; r < kProbeRing; ++r) {
      mbar_init(full(r), 1);
      mbar_init(empty(r), 1);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const long long mine = nchunks > blockIdx.x ? (nchunks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (warp == 0) {
    long long j = 0;
    for (; j < mine; ++j) {
      const int r = (int)(j % kProbeRing);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty(r), ((uint32_t)(j / kProbeRing) & 1u) ^ 1u, &abort_flag, status)))
        break;
      if (elect_one_sync()) {
        mbar_arrive_expect_tx(full(r), kProbeStage);
        bulk_copy_g2s(smem_u32(ring + (size_t)r * kProbeStage), src + (size_t)(blockIdx.x + j * gridDim.x) * kProbeStage,
                      kProbeStage, full(r));
      }
      __syncwarp();
    }
    for (long long q = (j > kProbeRing ? j - kProbeRing : 0); q < j; ++q)  // drain
      mbar_wait(full((int)(q % kProbeRing)), (uint32_t)(q / kProbeRing) & 1u, nullptr, status, kDrainTimeoutNs);
  } else {
    unsigned acc = 0;
    for (long long j = 0; j < mine; ++j) {
      const int r = (int)(j % kProbeRing);
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(full(r), (uint32_t)(j / kProbeRing) & 1u, &abort_flag, status))) break;
      acc += ring[(size_t)r * kProbeStage + lane];
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(r));
    }
    if (acc == 0xFFFFFFFFu) *sink = acc;  // keeps the reads
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_stream_probe(const void* src, size_t bytes, int* status, cudaStream_t s) {
  const long long nchunks = (long long)(bytes / kProbeStage);
  if (nchunks == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const int smem = kProbeRing * kProbeStage;
  err = cudaFuncSetAttribute(stream_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  // the sink word: the int after the status word (never written in practice)
  return launch_pdl(stream_probe_kernel, dim3(sms), dim3(64), (size_t)smem, s, static_cast<const uint8_t*>(src),
                    nchunks, status, reinterpret_cast<unsigned*>(status + 1));
}

}  // namespace moe
