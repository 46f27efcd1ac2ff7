// gemm_common.cuh -- device pieces of the grouped W4A16 GEMM (gemm_w4a16.cu):
// the device-side tile list, the packed-block loader and the block
// dequantiser.
#pragma once
#include <cstdint>

#include "device_common.cuh"
#include "kernels.h"

namespace moe {

struct TileCoord {
  int e, mt, nt;
};

// Tile t of a projection with MT weight tiles per expert: expert e owns tiles
// tprefix[e] * MT .. tprefix[e+1] * MT - 1, where tprefix is the prefix sum of
// the experts' token-tile counts (experts without tokens own none); inside
// them the token tile varies fastest, so the token tiles of one weight tile
// are adjacent.
__device__ __forceinline__ TileCoord decode_tile(int t, const int32_t* tprefix, int E, int MT) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tprefix[mid] * MT <= t) lo = mid;
    else hi = mid;
  }
  const int nt_count = tprefix[lo + 1] - tprefix[lo];
  const int local = t - tprefix[lo] * MT;
  TileCoord c;
  c.e = lo;
  c.mt = local / nt_count;
  c.nt = local - c.mt * nt_count;
  return c;
}

// One 64-column block of row r: codes at blk + r*16 and blk + 2048 + r*16,
// the four block scales at blk + 4096 + r*4.
struct BlockCodes {
  uint4 c0, c1;
  uint32_t sc;
};

__device__ __forceinline__ BlockCodes load_block(const uint8_t* blk, int r) {
  BlockCodes b;
  b.c0 = *reinterpret_cast<const uint4*>(blk + r * 16);
  b.c1 = *reinterpret_cast<const uint4*>(blk + 2048 + r * 16);
  b.sc = *reinterpret_cast<const uint32_t*>(blk + 4096 + r * 4);
  return b;
}

// Dequantise a loaded block into 32 bf16x2 columns.
__device__ __forceinline__ void dequant_block(const BlockCodes& b, uint32_t (&v)[32]) {
  uint32_t s0, s1, s2, s3;
  e4m3x2_to_scaleprime((uint16_t)(b.sc & 0xFFFFu), s0, s1);
  e4m3x2_to_scaleprime((uint16_t)(b.sc >> 16), s2, s3);
  dequant_word(b.c0.x, s0, v + 0);
  dequant_word(b.c0.y, s0, v + 4);
  dequant_word(b.c0.z, s1, v + 8);
  dequant_word(b.c0.w, s1, v + 12);
  dequant_word(b.c1.x, s2, v + 16);
  dequant_word(b.c1.y, s2, v + 20);
  dequant_word(b.c1.z, s3, v + 24);
  dequant_word(b.c1.w, s3, v + 28);
}

// Token-tile table of a grouped GEMM, built in shared memory by the whole
// CTA: s_off[0..E] = the expert offsets, s_tprefix[e] = the token tiles
// (ceil(count / BN)) of experts before e, s_tprefix[E] = *ntok = all token
// tiles.  Every thread calls it; it ends with the table visible to all.
__device__ __forceinline__ void build_tile_table(const int32_t* offsets, int E, int BN, int32_t* s_off,
                                                 int32_t* s_tprefix, volatile uint32_t* ntok) {
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = offsets[i];
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int sum = 0;
    for (int e = e0; e < e0 + per && e < E; ++e) sum += (s_off[e + 1] - s_off[e] + BN - 1) / BN;
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += y;
    }
    int run = incl - sum;
    for (int e = e0; e < e0 + per && e < E; ++e) {
      s_tprefix[e] = run;
      run += (s_off[e + 1] - s_off[e] + BN - 1) / BN;
    }
    if (lane == 31) {
      s_tprefix[E] = incl;
      *ntok = (uint32_t)incl;
    }
  }
  __syncthreads();
}

}  // namespace moe
