// gemm_simt.cu -- CUDA-core reference of the grouped W4A16 GEMMs over the
// packed weights (same dequantiser, fp32 FMA accumulation).  Used only to
// cross-check the tcgen05 kernels while they are brought up.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kSimtTok = 8;

// grid (MT, E), 128 threads: thread r owns packed tile row r.
template <int MODE>
__global__ void __launch_bounds__(128) simt_gemm_kernel(const uint16_t* __restrict__ act,
                                                        const uint8_t* __restrict__ packed,
                                                        const float* __restrict__ gscale,
                                                        const int32_t* __restrict__ offsets, void* __restrict__ out,
                                                        int N, int K, int out_ld) {
  const int mt = blockIdx.x, e = blockIdx.y, r = threadIdx.x, lane = r & 31, q = r >> 5;
  const int MT = N / kTileM, KB = K / kBlockK;
  const int off = offsets[e], cnt = offsets[e + 1] - off;
  const float gsc = gscale[e] * 128.0f;
  for (int tb = 0; tb < cnt; tb += kSimtTok) {
    float acc[kSimtTok];
#pragma unroll
    for (int i = 0; i < kSimtTok; ++i) acc[i] = 0.f;
    for (int kb = 0; kb < KB; ++kb) {
      const uint8_t* blk = packed + ((size_t)(e * MT + mt) * KB + kb) * kWBlockBytes;
      for (int half = 0; half < 2; ++half) {
        const uint4 cw = *reinterpret_cast<const uint4*>(blk + (half * 128 + r) * 16);
        const uint16_t sc = *reinterpret_cast<const uint16_t*>(blk + 4096 + r * 4 + half * 2);
        uint32_t s0, s1, v[16];
        e4m3x2_to_scaleprime(sc, s0, s1);
        dequant_word(cw.x, s0, v + 0);
        dequant_word(cw.y, s0, v + 4);
        dequant_word(cw.z, s1, v + 8);
        dequant_word(cw.w, s1, v + 12);
        const int k0 = kb * kBlockK + half * 32;
#pragma unroll
        for (int i = 0; i < kSimtTok; ++i) {
          if (tb + i >= cnt) break;
          const uint16_t* xr = act + (size_t)(off + tb + i) * K + k0;
          float a = acc[i];
          for (int j = 0; j < 16; ++j) {
            const uint32_t xx = *reinterpret_cast<const uint32_t*>(xr + 2 * j);
            a = fmaf(__uint_as_float(v[j] << 16), __uint_as_float(xx << 16), a);
            a = fmaf(__uint_as_float(v[j] & 0xFFFF0000u), __uint_as_float(xx & 0xFFFF0000u), a);
          }
          acc[i] = a;
        }
      }
    }
    if (MODE == 0) {
      const int f = mt * 64 + 16 * q + (lane & 15);
      uint16_t* h = reinterpret_cast<uint16_t*>(out);
#pragma unroll
      for (int i = 0; i < kSimtTok; ++i) {
        const float partner = __shfl_xor_sync(0xFFFFFFFFu, acc[i], 16);
        if (lane < 16 && tb + i < cnt) {
          const float g = acc[i] * gsc, u = partner * gsc;
          const float hv = g / (1.0f + __expf(-g)) * u;
          h[(size_t)(off + tb + i) * out_ld + f] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
        }
      }
    } else {
      float* y = reinterpret_cast<float*>(out);
      const int n = mt * kTileM + r;
#pragma unroll
      for (int i = 0; i < kSimtTok; ++i)
        if (tb + i < cnt) y[(size_t)(off + tb + i) * out_ld + n] = acc[i] * gsc;
    }
  }
}

cudaError_t launch_gemm_simt(int mode, const GemmArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  dim3 grid(a.N / kTileM, a.E);
  if (mode == 0)
    simt_gemm_kernel<0><<<grid, 128, 0, s>>>(a.act, a.packed, a.gscale, a.offsets, a.out, a.N, a.K, a.out_ld);
  else
    simt_gemm_kernel<1><<<grid, 128, 0, s>>>(a.act, a.packed, a.gscale, a.offsets, a.out, a.N, a.K, a.out_ld);
  return cudaGetLastError();
}

}  // namespace moe
