// router.cu -- the gate logits of the MoE layer: logits = x * Wr^T (+ bias).
//
// The Atlas article (f.mffb.com.cn/a/497905.html), section "KV Cache量化、MTP推测
// 解码和调试工具链", traces the layer as gate input -> gate logits -> expert IDs.
// Top-k routing compares logits exactly, so the logits are computed in one
// fixed fp32 order that does not depend on the launch shape:
//  * the hidden dimension is cut into 8-element (16-byte) chunks; lane l of
//    the warp takes chunks l, l+32, l+64, ... and accumulates x*w over its
//    elements in ascending h with fmaf, starting from 0;
//  * the 32 lane sums are combined by an xor butterfly (strides 16, 8, 4, 2,
//    1: lane l adds lane l^stride, and fp32 addition is commutative, so every
//    lane ends with the same value);
//  * the bias, if any, is added last.
#include <cstdint>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kRouterWarps = 8;
constexpr int kRouterExpertsPerBlock = 64;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// grid (ceil(E / 64), T); warp w of block (bx, t) takes experts bx*64 + w, + 8, ...
__global__ void __launch_bounds__(kRouterWarps * 32) router_logits_kernel(const uint16_t* __restrict__ x,
                                                                           const uint16_t* __restrict__ wr,
                                                                           const float* __restrict__ bias, int H,
                                                                           int E, float* __restrict__ logits) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.y;
  pdl_wait();
  pdl_trigger();
  const int nch = H / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  for (int i = 0; i < kRouterExpertsPerBlock / kRouterWarps; ++i) {
    const int e = blockIdx.x * kRouterExpertsPerBlock + i * kRouterWarps + warp;
    if (e >= E) break;
    const uint4* wrow = reinterpret_cast<const uint4*>(wr + (size_t)e * H);
    float acc = 0.f;
    for (int ch = lane; ch < nch; ch += 32) {
      const uint4 xv = xr[ch], wv = wrow[ch];
      acc = fmaf(bf16_lo(xv.x), bf16_lo(wv.x), acc);
      acc = fmaf(bf16_hi(xv.x), bf16_hi(wv.x), acc);
      acc = fmaf(bf16_lo(xv.y), bf16_lo(wv.y), acc);
      acc = fmaf(bf16_hi(xv.y), bf16_hi(wv.y), acc);
      acc = fmaf(bf16_lo(xv.z), bf16_lo(wv.z), acc);
      acc = fmaf(bf16_hi(xv.z), bf16_hi(wv.z), acc);
      acc = fmaf(bf16_lo(xv.w), bf16_lo(wv.w), acc);
      acc = fmaf(bf16_hi(xv.w), bf16_hi(wv.w), acc);
    }
#pragma unroll
    for (int stride = 16; stride >= 1; stride >>= 1) acc = acc + __shfl_xor_sync(0xFFFFFFFFu, acc, stride);
    if (lane == 0) logits[(size_t)t * E + e] = bias != nullptr ? acc + bias[e] : acc;
  }
}

}  // namespace

cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* wr, const float* bias, int T, int H, int E,
                                 float* logits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((E + kRouterExpertsPerBlock - 1) / kRouterExpertsPerBlock, T);
  return launch_pdl(router_logits_kernel, grid, dim3(kRouterWarps * 32), 0, s, x, wr, bias, H, E, logits);
}

}  // namespace moe
