// gemm_w4a4.cu -- the block-scaled FP4 variant of the layer (W4A4): NVFP4
// weights AND NVFP4 activations multiplied natively by tcgen05.mma
// kind::mxf4nvf4 (E2M1 x E2M1 with one E4M3 scale per 16 K elements on each
// side, fp32 accumulate), which GB300 has and GB10 lacks (the Atlas article,
// section "编译时内核选择和W4A16 Grouped GEMM", falls back to W4A16 on GB10 for
// that reason; the ATOM article, section "8.2 量化并非单一格式，而是一套执行契约",
// treats a 4-bit-activation format as an execution contract of its own).
//
// Activation quantizer (x before gate_up, h before down): per 16 consecutive
// elements s = RNE_e4m3(min(amax16 / 6, 448)) (amax16 / 6 in fp32) and the
// codes RNE_e2m1 of the exact quotient v / e4m3(s), ties to the even
// mantissa, saturating at +-6, all codes 0 when e4m3(s) is 0; no global
// scale.  h is quantized from its fp32 value.  Weights keep their NVFP4 format in the
// natural layout (codes [E][N][K/2], scales [E][N][K/16], global scale [E]),
// read by TMA straight from it; the fp32 global scale is applied in the
// epilogue.
//
// Scale factors in tensor memory (measured on this GPU with a probe that
// writes known words and selects one K block at a time): for one MMA of
// K = 64, row m of A reads lane m, column sfa + m / 32, byte kb (the scale of
// its K elements 16 kb .. 16 kb + 15); column n of B, for the rows of A in
// lane quadrant q, reads lane 32 q + n % 32, column sfb + n / 32, byte kb --
// B's scales are held once per lane quadrant.  Every scale address given to the MMA is kept
// on a 4-column (128-bit) boundary, as in the probe.
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace moe {

// ------------------------------------------------------------- quantizer
// One 16-element block of NVFP4 (no global scale): the E4M3 scale s =
// RNE_e4m3(min(amax / 6, 448)) and the E2M1 codes of v / e4m3(s), each the
// grid value nearest to the exact quotient, ties to the even mantissa,
// saturating at 6, all codes 0 when e4m3(s) is 0.

// RNE_e4m3(min(amax / 6, 448)).  The quotient is amax * RN(1/6) corrected by
// one FMA on the exact remainder, within half an ulp (plus 2^-24 ulp) of
// amax / 6.  An E4M3 rounding midpoint m has 5 significant bits, so 6 m is
// exact in fp32 and amax / 6 is either m itself (the corrected quotient is
// then m) or at least 2/3 ulp away from it: the E4M3 rounding of the
// corrected quotient is that of amax / 6, and of an IEEE division.
__device__ __forceinline__ uint32_t e4m3_scale_of_amax(float amax) {
  constexpr float kSixth = 0.16666667f;
  const float q0 = amax * kSixth;
  const float q = fmaf(fmaf(-6.0f, q0, amax), kSixth, q0);
  return (uint32_t)__nv_cvt_float_to_fp8(fminf(q, 448.0f), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Quotient v / d rounded to E2M1 by the hardware conversion.  d (an E4M3
// value) has at most 4 significant bits: with rc within an ulp of 1 / d, q0 =
// v rc is within a few ulps of v / d, so the remainder v - d q0 is exact and
// q = q0 + (v - d q0) rc lies within half an ulp (plus 2^-22 ulp) of v / d.
// Each E2M1 midpoint t has at most 3 significant bits, so t d is exact in
// fp32 and v / d is either t (q is then t) or more than 0.53 ulp from it:
// rounding q to E2M1 rounds v / d.
__device__ __forceinline__ float e2m1_quotient(float v, float d, float rc) {
  const float q0 = v * rc;
  return fmaf(fmaf(-d, q0, v), rc, q0);
}

// Eight quotients -> one word of E2M1 codes, element i in bits 4i..4i+3;
// codes of magnitude 0 carry no sign.
__device__ __forceinline__ uint32_t e2m1x8(const float (&q)[16], int o) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w)
      : "f"(q[o]), "f"(q[o + 1]), "f"(q[o + 2]), "f"(q[o + 3]), "f"(q[o + 4]), "f"(q[o + 5]), "f"(q[o + 6]),
        "f"(q[o + 7]));
  const uint32_t mag = w & 0x77777777u;
  const uint32_t nonzero = (mag + 0x77777777u) & 0x88888888u;  // bit 3 of a nibble: magnitude != 0
  return mag | (w & nonzero);
}

// One 16-element block: the E4M3 scale byte and 8 code bytes (element 2i in
// the low nibble).
struct Nvfp4Block {
  uint32_t scale;
  uint32_t codes[2];  // 8 bytes
};

__device__ __forceinline__ Nvfp4Block quant_block16(const float (&v)[16]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  Nvfp4Block b;
  b.scale = e4m3_scale_of_amax(amax);
  const float d = __half2float(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b.scale, __NV_E4M3));
  const float rc = rcp_approx(d);
  float q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) q[i] = e2m1_quotient(v[i], d, rc);
  b.codes[0] = b.scale != 0u ? e2m1x8(q, 0) : 0u;
  b.codes[1] = b.scale != 0u ? e2m1x8(q, 8) : 0u;
  return b;
}

// Quantize and gather: row p of the grouped view gets the NVFP4 form of
// x[src[p]] (or x[p] when src is null), x bf16 or fp32.  One thread per
// 16-element block; codes [n][K/2], scales [n][K/16].
__device__ __forceinline__ void load_block16(const uint16_t* xp, float (&v)[16]) {
  const uint4* p = reinterpret_cast<const uint4*>(xp);
  const uint4 w0 = p[0], w1 = p[1];
  const uint32_t wd[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(wd[i] << 16);
    v[2 * i + 1] = __uint_as_float(wd[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void load_block16(const float* xp, float (&v)[16]) {
  const float4* p = reinterpret_cast<const float4*>(xp);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = p[i];
    v[4 * i] = f.x;
    v[4 * i + 1] = f.y;
    v[4 * i + 2] = f.z;
    v[4 * i + 3] = f.w;
  }
}

template <typename T>
__global__ void __launch_bounds__(256) quant_gather_kernel(const T* __restrict__ x, const int32_t* __restrict__ src,
                                                            long long nblocks, int bpr, uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  for (long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x; g < nblocks;
       g += (long long)gridDim.x * blockDim.x) {
    const long long p = g / bpr;
    const int b = (int)(g - p * bpr);
    const long long row = src != nullptr ? (long long)src[p] : p;
    float v[16];
    load_block16(x + row * (long long)bpr * 16 + b * 16, v);
    const Nvfp4Block q = quant_block16(v);
    *reinterpret_cast<uint2*>(codes + p * (long long)bpr * 8 + b * 8) = make_uint2(q.codes[0], q.codes[1]);
    scales[p * (long long)bpr + b] = (uint8_t)q.scale;
  }
}

template <typename T>
cudaError_t launch_quant_gather(const T* x, const int32_t* src, int n, int K, uint8_t* codes, uint8_t* scales,
                                cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int bpr = K / 16;
  const long long nblocks = (long long)n * bpr;
  long long blocks = (nblocks + 255) / 256;
  if (blocks > 8192) blocks = 8192;
  return launch_pdl(quant_gather_kernel<T>, dim3((unsigned)blocks), dim3(256), 0, s, x, src, nblocks, bpr, codes,
                    scales);
}

// ------------------------------------------------------------- the GEMMs
// Persistent, one CTA per SM, static tile stride (u = blockIdx.x, +
// gridDim.x, ...) over the tile list of gemm_common.cuh.  A stage is K 256:
// 128 code bytes (128-byte swizzled) and 16 scale bytes per row of A and B,
// consumed by 4 block-scaled MMAs of K 64 (M 128, N = NB).  Warp roles:
//   0..3  epilogue (TMEM lane quadrant = warp);
//   4..7  scale factors: per stage, the E4M3 scales of A (rows 32q..32q+31)
//         and a copy of B's, read from the stage in shared memory and stored
//         into the warp's lane quadrant of a TMEM slot in the MMA's layout;
//   8     TMA producer;
//   9     TMEM owner and MMA issue.
// gate_up (MODE 0) puts the tokens in the accumulator's lanes: A = TT
// activation rows (the MMA still reads 128; rows TT.. of its result are not
// used), B = 64 gate rows then the 64 matching up rows of the expert, so one
// epilogue thread holds whole 16-feature blocks of h (gate columns 16 b..,
// up columns 64 + 16 b..) and quantizes them without exchanging data.  down
// (MODE 1) puts 128 weight rows (output features) in A and TT tokens in B.
constexpr int kW4Warps = 10;
constexpr int kW4Threads = kW4Warps * 32;
constexpr int kW4WarpSf0 = 4;
constexpr int kW4WarpTma = 8;
constexpr int kW4WarpMma = 9;
constexpr int kW4StageK = 256;
constexpr uint32_t kW4TmemCols = 512;
constexpr int kGuFeat = 64;  // h features of a gate_up tile (MMA N = 2 * 64)

template <int NB>
struct Cfg4 {
  // a stage: A codes (128 rows x 128 B, swizzled), B codes (NB rows x 128 B,
  // swizzled), A scales (128 rows x 16 B), B scales (NB rows x 16 B)
  static constexpr int kA = 128 * 128;
  static constexpr int kB = NB * 128;
  static constexpr int kOffAs = kA + kB;
  static constexpr int kOffBs = kOffAs + 128 * 16;
  static constexpr int kStage = ((kOffBs + NB * 16 + 1023) / 1024) * 1024;
  static constexpr int NS0 = (200 * 1024) / kStage;
  static constexpr int NS = NS0 > 8 ? 8 : NS0;
  static constexpr int ND = 2;
  static constexpr int kSfbPerMma = NB / 32 > 0 ? NB / 32 : 1;  // SFB columns an MMA reads
  // every MMA's scale vectors start on a 4-column (128-bit) boundary
  static constexpr int kSfbStride = ((kSfbPerMma + 3) / 4) * 4;
  static constexpr int kSfSlot = 16 + 4 * kSfbStride;  // SFA (4 MMAs x 4 columns) + SFB
  static_assert(kSfSlot % 4 == 0 && (ND * NB) % 4 == 0, "scale vectors on 4-column boundaries");
  static constexpr int NSF0 = (int)(512 - ND * NB) / kSfSlot;
  static constexpr int NSF = NSF0 > 6 ? 6 : NSF0;
  static_assert(NSF >= 2 && NS >= 2, "rings need two slots");
  static constexpr int kOffBar = NS * kStage;
  // full[NS], empty[NS], sffull[NSF], sfempty[NSF], dfull[ND], dempty[ND], drain
  static constexpr int kNumBars = 2 * NS + 2 * NSF + 2 * ND + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // [0] tmem base, [1] abort, [2] token tiles
  static constexpr int kOffTables = kOffMisc + 16;
  static_assert(kA % 1024 == 0 && kB % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static int bytes(int E) { return kOffTables + 2 * (E + 1) * 4 + 1024; }
};

__device__ __forceinline__ void tc_mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

// Instruction descriptor of kind::mxf4nvf4: A and B E2M1 (format 1 at bits
// 7-9 and 10-12), K-major, N >> 3 at bits 17-22, UE4M3 scales (bit 23 = 0),
// M >> 4 at bits 24-28, scale-factor ids 0.
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

struct W4a4Launch {
  const float* gscale;       // [E]
  const int32_t* offsets;
  void* out;                 // MODE 0: h codes [rows][I/2]; MODE 1: y f32 [rows][H]
  uint8_t* out_scales;       // MODE 0: h scales [rows][I/16]
  int* status;
  int E, N, K, rows, out_ld;  // out_ld: I (MODE 0) or H (MODE 1)
  int I;                      // the expert intermediate size (gate_up: N = 2I)
};

// MODE 0: gate_up + SwiGLU, h quantized to NVFP4; MODE 1: down, fp32 y.  TT
// is the token tile.
template <int MODE, int TT>
__global__ void __launch_bounds__(kW4Threads, 1)
    w4a4_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_as,
                     const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_bs,
                     const __grid_constant__ W4a4Launch L) {
  constexpr int NB = MODE == 0 ? 2 * kGuFeat : TT;  // MMA N
  constexpr int kRowsA = MODE == 0 ? TT : kTileM;   // rows of A a stage delivers
  using C = Cfg4<NB>;
  constexpr int NS = C::NS, NSF = C::NSF, ND = C::ND;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (NS + s); };
  auto sffull_bar = [&](int f) { return bar0 + 8u * (2 * NS + f); };
  auto sfempty_bar = [&](int f) { return bar0 + 8u * (2 * NS + NSF + f); };
  auto dfull_bar = [&](int d) { return bar0 + 8u * (2 * NS + 2 * NSF + d); };
  auto dempty_bar = [&](int d) { return bar0 + 8u * (2 * NS + 2 * NSF + ND + d); };
  const uint32_t drain_bar = bar0 + 8u * (2 * NS + 2 * NSF + 2 * ND);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const int E = L.E;
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + C::kOffTables);
  int32_t* s_tprefix = s_off + (E + 1);
  int* status = L.status;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full_bar(s), 1);   // the producer's expect_tx arrival (+ the copied bytes)
      mbar_init(empty_bar(s), 1);  // the MMA commit
    }
    for (int f = 0; f < NSF; ++f) {
      mbar_init(sffull_bar(f), 4);  // the four scale-factor warps
      mbar_init(sfempty_bar(f), 1); // the MMA commit
    }
    for (int d = 0; d < ND; ++d) {
      mbar_init(dfull_bar(d), 1);
      mbar_init(dempty_bar(d), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kW4WarpTma && lane == 0) {
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_as);
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_bs);
  }
  if (warp == kW4WarpMma) {
    tmem_alloc(sbase + C::kOffMisc, kW4TmemCols);
    tmem_relinquish();
  }
  // The expert offsets come from the routing kernel, which had completed
  // before the kernel this one depends on got past its own dependency wait
  // (every kernel of the layer waits on its predecessor before it lets its
  // dependents launch), so the tile table is built before this kernel's wait.
  build_tile_table(L.offsets, E, TT, s_off, s_tprefix, misc + 2);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const int ntok = (int)misc[2];
  const int MT = MODE == 0 ? L.I / kGuFeat : L.N / kTileM;  // weight tiles per expert
  const int total = ntok * MT;
  const int KS = L.K / kW4StageK;
  const uint32_t sf_col0 = (uint32_t)(ND * NB);  // scale-factor slots after the accumulators
  constexpr uint32_t kTx = (uint32_t)((kRowsA + NB) * (128 + 16));  // bytes a stage's copies deliver

  // the weight rows of stage ks of tile c (MODE 0: 64 gate rows 64 mt.. of
  // expert e, then the matching up rows, I further on; MODE 1: 128 rows), and
  // the tile's activation rows p0..
  auto load_weights = [&](uint32_t st, const TileCoord& c, int ks, uint32_t bar) {
    if (MODE == 0) {
      const int gate_row = c.e * L.N + c.mt * kGuFeat;
      const int up_row = gate_row + L.I;
      tma_load_2d(st + C::kA, &tm_b, ks * 128, gate_row, bar);
      tma_load_2d(st + C::kA + (uint32_t)(kGuFeat * 128), &tm_b, ks * 128, up_row, bar);
      tma_load_2d(st + C::kOffBs, &tm_bs, ks * 16, gate_row, bar);
      tma_load_2d(st + C::kOffBs + (uint32_t)(kGuFeat * 16), &tm_bs, ks * 16, up_row, bar);
    } else {
      const int row = c.e * L.N + c.mt * kTileM;
      tma_load_2d(st, &tm_a, ks * 128, row, bar);
      tma_load_2d(st + C::kOffAs, &tm_as, ks * 16, row, bar);
    }
  };
  auto load_activations = [&](uint32_t st, int p0, int ks, uint32_t bar) {
    if (MODE == 0) {
      tma_load_2d(st, &tm_a, ks * 128, p0, bar);
      tma_load_2d(st + C::kOffAs, &tm_as, ks * 16, p0, bar);
    } else {
      tma_load_2d(st + C::kA, &tm_b, ks * 128, p0, bar);
      tma_load_2d(st + C::kOffBs, &tm_bs, ks * 16, p0, bar);
    }
  };

  // Before the dependency wait the producer issues the weight half of the
  // first NS stages (the weights do not come from the kernels before; their
  // slots are free in a fresh ring), so the weight stream starts while the
  // kernel before is still finishing.  The activation half follows the wait.
  int npre = 0;
  if (warp == kW4WarpTma) {
    for (int u = blockIdx.x; u < total && npre < NS; u += gridDim.x) {
      const TileCoord c = decode_tile(u, s_tprefix, E, MT);
      for (int ks = 0; ks < KS && npre < NS; ++ks, ++npre) {
        if (elect_one_sync()) {
          mbar_arrive_expect_tx(full_bar(npre), kTx);
          load_weights(sbase + (uint32_t)(npre * C::kStage), c, ks, full_bar(npre));
        }
        __syncwarp();
      }
    }
  }
  pdl_wait();
  pdl_trigger();

  if (warp == kW4WarpTma) {
    // ------------------------------------------------------------ producer
    // (stages below npre have their weights in flight already; their empty
    // waits pass at once, the ring being fresh, so none of them is left
    // without its activation half)
    int i = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const TileCoord c = decode_tile(u, s_tprefix, E, MT);
      const int p0 = s_off[c.e] + c.nt * TT;
      for (int ks = 0; ks < KS; ++ks, ++i) {
        const int s = i % NS;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty_bar(s), ((uint32_t)(i / NS) & 1u) ^ 1u, abort_flag, status))) {
          ok = false;
          break;
        }
        if (elect_one_sync()) {
          const uint32_t st = sbase + (uint32_t)(s * C::kStage);
          if (i >= npre) {
            mbar_arrive_expect_tx(full_bar(s), kTx);
            load_weights(st, c, ks, full_bar(s));
          }
          load_activations(st, p0, ks, full_bar(s));
        }
        __syncwarp();
      }
    }
    for (int j = (i > NS ? i - NS : 0); j < i; ++j)
      mbar_wait(full_bar(j % NS), (uint32_t)(j / NS) & 1u, nullptr, status, kDrainTimeoutNs);
  } else if (warp >= kW4WarpSf0 && warp < kW4WarpSf0 + 4) {
    // ------------------------------------------------------- scale factors
    // Row m = 32 q + lane of A and column n = 32 cb + lane of B: the 4 scale
    // bytes of MMA j (K elements 64 j .. 64 j + 63 of the stage) form one
    // 32-bit word, stored at lane m, column slot + 4 j + q (A; zero for the
    // rows a stage does not deliver) and lane 32 q + n % 32, column slot + 16
    // + j * kSfbStride + n / 32 (B, one copy per lane quadrant).
    const int q = warp - kW4WarpSf0;
    const uint32_t t_lane = tmem_base + ((uint32_t)(32 * q) << 16);
    int i = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      for (int ks = 0; ks < KS; ++ks, ++i) {
        const int s = i % NS, f = i % NSF;
        const bool got = mbar_wait(full_bar(s), (uint32_t)(i / NS) & 1u, abort_flag, status) &&
                         mbar_wait(sfempty_bar(f), ((uint32_t)(i / NSF) & 1u) ^ 1u, abort_flag, status);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = smem + s * C::kStage;
        uint4 wa = make_uint4(0u, 0u, 0u, 0u);
        if (32 * q < kRowsA) wa = *reinterpret_cast<const uint4*>(st + C::kOffAs + (32 * q + lane) * 16);
        const uint32_t col = sf_col0 + (uint32_t)(f * C::kSfSlot);
        tmem_st1(t_lane + col + 0u + q, wa.x);
        tmem_st1(t_lane + col + 4u + q, wa.y);
        tmem_st1(t_lane + col + 8u + q, wa.z);
        tmem_st1(t_lane + col + 12u + q, wa.w);
#pragma unroll
        for (int cb = 0; cb < C::kSfbPerMma; ++cb) {
          const int n = 32 * cb + lane;
          uint4 wb = make_uint4(0u, 0u, 0u, 0u);
          if (n < NB) wb = *reinterpret_cast<const uint4*>(st + C::kOffBs + n * 16);
          const uint32_t cbase = col + 16u + (uint32_t)cb;
          tmem_st1(t_lane + cbase + 0u * C::kSfbStride, wb.x);
          tmem_st1(t_lane + cbase + 1u * C::kSfbStride, wb.y);
          tmem_st1(t_lane + cbase + 2u * C::kSfbStride, wb.z);
          tmem_st1(t_lane + cbase + 3u * C::kSfbStride, wb.w);
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sffull_bar(f));
      }
    }
  } else if (warp == kW4WarpMma) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t idesc = idesc_mxf4(kTileM, NB);
    int i = 0, it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++it) {
      const int d = it % ND;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(dempty_bar(d), ((uint32_t)(it / ND) & 1u) ^ 1u, abort_flag, status)))
        break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(d * NB);
      for (int ks = 0; ks < KS; ++ks, ++i) {
        const int s = i % NS, f = i % NSF;
        const bool got = mbar_wait(full_bar(s), (uint32_t)(i / NS) & 1u, abort_flag, status) &&
                         mbar_wait(sffull_bar(f), (uint32_t)(i / NSF) & 1u, abort_flag, status);
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t st = sbase + (uint32_t)(s * C::kStage);
        const uint64_t a_desc = smem_desc_sw128(st), b_desc = smem_desc_sw128(st + C::kA);
        const uint32_t sf = tmem_base + sf_col0 + (uint32_t)(f * C::kSfSlot);
        if (elect_one_sync()) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma_mxf4(d_tmem, a_desc + (uint64_t)(2 * j), b_desc + (uint64_t)(2 * j), idesc, sf + 4u * j,
                        sf + 16u + (uint32_t)(j * C::kSfbStride), (ks | j) != 0);
          tc_commit(empty_bar(s));
          tc_commit(sfempty_bar(f));
        }
        __syncwarp();
      }
      if (ok) {
        if (elect_one_sync()) tc_commit(dfull_bar(d));
        __syncwarp();
      }
    }
    if (elect_one_sync()) tc_commit(drain_bar);
    __syncwarp();
    mbar_wait(drain_bar, 0, nullptr, status, kDrainTimeoutNs);
  } else if (warp < 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp;
    int it = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++it) {
      const TileCoord c = decode_tile(u, s_tprefix, E, MT);
      const int d = it % ND;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(dfull_bar(d), (uint32_t)(it / ND) & 1u, abort_flag, status))) break;
      tc_fence_after();
      const int p0 = s_off[c.e] + c.nt * TT;
      const int nvalid = min(TT, s_off[c.e + 1] - p0);
      const float gsc = __ldg(L.gscale + c.e);
      const uint32_t t_acc = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(d * NB);
      if (MODE == 0) {
        // this thread's token: row r of the tile; h block b = SwiGLU of gate
        // columns 16 b.. and up columns 64 + 16 b.., then its NVFP4 form
        const int r = 32 * q + lane;
        uint32_t words[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        uint32_t sc = 0u;
        if (32 * q < TT && 32 * q < nvalid) {
#pragma unroll
          for (int b = 0; b < kGuFeat / 16; ++b) {
            uint32_t vg[16], vu[16];
            tmem_ld16(t_acc + (uint32_t)(16 * b), vg);
            tmem_ld16(t_acc + (uint32_t)(kGuFeat + 16 * b), vu);
            tc_wait_ld();
            float h[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float g = __uint_as_float(vg[j]) * gsc;
              const float up = __uint_as_float(vu[j]) * gsc;
              h[j] = __fdividef(g, 1.0f + __expf(-g)) * up;
            }
            const Nvfp4Block nb = quant_block16(h);
            words[2 * b] = nb.codes[0];
            words[2 * b + 1] = nb.codes[1];
            sc |= nb.scale << (8 * b);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dempty_bar(d));
        if (r < nvalid) {
          const size_t p = (size_t)(p0 + r);
          uint4* hc = reinterpret_cast<uint4*>(static_cast<uint8_t*>(L.out) + p * (size_t)(L.out_ld / 2) +
                                               (size_t)c.mt * (kGuFeat / 2));
          hc[0] = make_uint4(words[0], words[1], words[2], words[3]);
          hc[1] = make_uint4(words[4], words[5], words[6], words[7]);
          *reinterpret_cast<uint32_t*>(L.out_scales + p * (size_t)(L.out_ld / 16) + (size_t)c.mt * (kGuFeat / 16)) =
              sc;
        }
      } else {
        const int n = c.mt * kTileM + 32 * q + lane;
        float* y = reinterpret_cast<float*>(L.out);
#pragma unroll 1
        for (int cc = 0; cc < NB / 16; ++cc) {
          uint32_t v[16];
          tmem_ld16(t_acc + (uint32_t)(cc * 16), v);
          tc_wait_ld();
          if (cc * 16 >= nvalid) continue;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = cc * 16 + j;
            if (col < nvalid) y[(size_t)(p0 + col) * L.out_ld + n] = __uint_as_float(v[j]) * gsc;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dempty_bar(d));
      }
    }
  }
  // warps 4..7 (scale factors) and the producer are done; everyone meets here
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kW4WarpMma) tmem_dealloc(tmem_base, kW4TmemCols);
}

// ------------------------------------------------------------------ launch
using PFN_encodeTiled4 = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled4 encode_fn4() {
  static PFN_encodeTiled4 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled4>(p);
  }
  return fn;
}

// A 2-D byte matrix [rows][cols] with a (box_cols x box_rows) box.
static bool encode_u8(CUtensorMap* m, const void* base, long long cols, long long rows, int box_cols, int box_rows,
                      bool swizzle) {
  PFN_encodeTiled4 enc = encode_fn4();
  if (enc == nullptr) return false;
  memset(m, 0, sizeof(*m));
  const cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)cols};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct W4a4Args {
  const uint8_t* w_codes;  // [E][N][K/2]
  const uint8_t* w_scales; // [E][N][K/16]
  const float* gscale;     // [E]
  const uint8_t* a_codes;  // [rows][K/2]
  const uint8_t* a_scales; // [rows][K/16]
  const int32_t* offsets;
  void* out;
  uint8_t* out_scales;
  int* status;
  int rows, E, N, K, I, out_ld;
};

template <int MODE, int TT>
static cudaError_t launch_w4a4_cfg(const W4a4Args& a, cudaStream_t s) {
  constexpr int NB = MODE == 0 ? 2 * kGuFeat : TT;
  using C = Cfg4<NB>;
  CUtensorMap tm[4];
  const long long wrows = (long long)a.E * a.N;
  // MODE 0: A = activations (TT-row boxes), B = weights (64-row boxes);
  // MODE 1: A = weights (128-row boxes), B = activations (TT-row boxes)
  const bool ok = MODE == 0 ? encode_u8(&tm[0], a.a_codes, a.K / 2, a.rows, 128, TT, true) &&
                                  encode_u8(&tm[1], a.a_scales, a.K / 16, a.rows, 16, TT, false) &&
                                  encode_u8(&tm[2], a.w_codes, a.K / 2, wrows, 128, kGuFeat, true) &&
                                  encode_u8(&tm[3], a.w_scales, a.K / 16, wrows, 16, kGuFeat, false)
                            : encode_u8(&tm[0], a.w_codes, a.K / 2, wrows, 128, kTileM, true) &&
                                  encode_u8(&tm[1], a.w_scales, a.K / 16, wrows, 16, kTileM, false) &&
                                  encode_u8(&tm[2], a.a_codes, a.K / 2, a.rows, 128, TT, true) &&
                                  encode_u8(&tm[3], a.a_scales, a.K / 16, a.rows, 16, TT, false);
  if (!ok) return cudaErrorInvalidValue;
  W4a4Launch L;
  L.gscale = a.gscale;
  L.offsets = a.offsets;
  L.out = a.out;
  L.out_scales = a.out_scales;
  L.status = a.status;
  L.E = a.E;
  L.N = a.N;
  L.K = a.K;
  L.rows = a.rows;
  L.out_ld = a.out_ld;
  L.I = a.I;
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const long long n = a.rows;
  const long long mt = MODE == 0 ? a.I / kGuFeat : a.N / kTileM;
  const long long max_tiles = mt * (n / TT + (n < a.E ? n : a.E));
  const int grid = (int)(max_tiles < sms ? max_tiles : sms);
  if (grid <= 0) return cudaSuccess;
  const int smem = C::bytes(a.E);
  auto kern = w4a4_gemm_kernel<MODE, TT>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, dim3(grid), dim3(kW4Threads), smem, s, tm[0], tm[1], tm[2], tm[3], L);
}

// Token tile of the W4A4 GEMMs: 32, 64 or 128 rows, about twice the mean rows per expert.
int w4a4_token_tile(int rows, int E) {
  const long long mean2 = 2LL * rows / (E > 0 ? E : 1);
  return mean2 <= 32 ? 32 : mean2 <= 64 ? 64 : 128;
}

cudaError_t launch_w4a4(int mode, const W4a4Args& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  switch (w4a4_token_tile(a.rows, a.E) * 2 + mode) {
    case 64: return launch_w4a4_cfg<0, 32>(a, s);
    case 65: return launch_w4a4_cfg<1, 32>(a, s);
    case 128: return launch_w4a4_cfg<0, 64>(a, s);
    case 129: return launch_w4a4_cfg<1, 64>(a, s);
    case 256: return launch_w4a4_cfg<0, 128>(a, s);
    default: return launch_w4a4_cfg<1, 128>(a, s);
  }
}

}  // namespace moe

// ------------------------------------------------------------ entry points
#include "moe_w4a16.h"

namespace {

constexpr size_t kAlign4 = 256;
inline size_t up4(size_t v) { return (v + kAlign4 - 1) & ~(kAlign4 - 1); }
inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Layout4 {
  size_t status, perm, ids, w, counts, offsets, sorted, inv, xc, xs, hc, hs, y, total;
};

Layout4 layout4(const moe_dims& d) {
  Layout4 L{};
  const size_t n = (size_t)d.T * d.k;
  size_t o = 0;
  L.status = o;
  o = up4(o + sizeof(int));
  L.perm = o;
  o = up4(o + moe::perm_scratch_bytes(d.T, d.E, d.k));
  L.ids = o;
  o = up4(o + n * 4);
  L.w = o;
  o = up4(o + n * 4);
  L.counts = o;
  o = up4(o + (size_t)d.E * 4);
  L.offsets = o;
  o = up4(o + (size_t)(d.E + 1) * 4);
  L.sorted = o;
  o = up4(o + n * 4);
  L.inv = o;
  o = up4(o + n * 4);
  L.xc = o;
  o = up4(o + n * (size_t)d.H / 2);
  L.xs = o;
  o = up4(o + n * (size_t)d.H / 16);
  L.hc = o;
  o = up4(o + n * (size_t)d.I / 2);
  L.hs = o;
  o = up4(o + n * (size_t)d.I / 16);
  L.y = o;
  o = up4(o + n * (size_t)d.H * 4);
  L.total = o;
  return L;
}

int check4(const moe_dims& d) {
  if (d.T < 0 || d.H <= 0 || d.I <= 0 || d.E < 1 || d.k < 1 || d.k > d.E || d.k > 32 || d.E > 1024)
    return MOE_ERR_INVALID_ARG;
  if (d.H % 256 != 0 || d.I % 256 != 0 || d.H > 65536 || d.I > 65536 || (long long)d.T * d.k >= (1LL << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

int cuda_rc(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  (void)cudaGetLastError();
  return MOE_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t moe_w4a4_workspace_bytes(moe_dims d) {
  if (check4(d) != MOE_OK) return 0;
  return layout4(d).total;
}

int moe_w4a4_kernel_launches(moe_dims d) {
  const int rc = check4(d);
  if (rc != MOE_OK) return -rc;
  if (d.T == 0) return 0;
  // routing + grouping, quantize + gather of x, gate_up, down, combine
  return moe::route_group_launches(d.T, d.E, d.k, false) + 4;
}

int moe_layer_forward_w4a4_profiled(const uint16_t* x, const float* logits, moe_w4n w_gate_up, moe_w4n w_down,
                                    moe_dims d, uint16_t* out, int32_t* topk_ids, float* topk_w, void* ws,
                                    size_t ws_bytes, void* stream, void* const* ev);

int moe_layer_forward_w4a4(const uint16_t* x, const float* logits, moe_w4n w_gate_up, moe_w4n w_down, moe_dims d,
                           uint16_t* out, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, void* stream) {
  return moe_layer_forward_w4a4_profiled(x, logits, w_gate_up, w_down, d, out, topk_ids, topk_w, ws, ws_bytes, stream,
                                         nullptr);
}

int moe_layer_forward_w4a4_profiled(const uint16_t* x, const float* logits, moe_w4n w_gate_up, moe_w4n w_down,
                                    moe_dims d, uint16_t* out, int32_t* topk_ids, float* topk_w, void* ws,
                                    size_t ws_bytes, void* stream, void* const* ev) {
  const int rc = check4(d);
  if (rc != MOE_OK) return rc;
  if (d.T == 0) return MOE_OK;
  const void* need[] = {x, logits, w_gate_up.codes, w_gate_up.scales, w_gate_up.global_scale, w_down.codes,
                        w_down.scales, w_down.global_scale, out, ws};
  for (const void* p : need)
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
  for (const void* p : need)
    if (!al16(p)) return MOE_ERR_MISALIGNED;
  if ((topk_ids != nullptr && !al16(topk_ids)) || (topk_w != nullptr && !al16(topk_w))) return MOE_ERR_MISALIGNED;
  const Layout4 L = layout4(d);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t* ids = topk_ids ? topk_ids : reinterpret_cast<int32_t*>(w + L.ids);
  float* wts = topk_w ? topk_w : reinterpret_cast<float*>(w + L.w);
  int32_t* offs = reinterpret_cast<int32_t*>(w + L.offsets);
  int32_t* sorted = reinterpret_cast<int32_t*>(w + L.sorted);
  int32_t* inv = reinterpret_cast<int32_t*>(w + L.inv);
  const int rows = d.T * d.k;
  auto mark = [&](int i) -> int {
    if (ev == nullptr || ev[i] == nullptr) return MOE_OK;
    return cuda_rc(cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[i]), s));
  };
  int e = mark(0);
  if (e != MOE_OK) return e;
  e = cuda_rc(moe::launch_route_group(logits, d.T, d.E, d.k, false, ids, wts,
                                          reinterpret_cast<int32_t*>(w + L.counts), offs, sorted, inv,
                                          reinterpret_cast<int32_t*>(w + L.perm), nullptr, s));
  if (e != MOE_OK || (e = mark(1)) != MOE_OK) return e;
  e = cuda_rc(moe::launch_quant_gather(x, sorted, rows, d.H, w + L.xc, w + L.xs, s));
  if (e != MOE_OK || (e = mark(2)) != MOE_OK) return e;
  moe::W4a4Args a{};
  a.w_codes = static_cast<const uint8_t*>(w_gate_up.codes);
  a.w_scales = static_cast<const uint8_t*>(w_gate_up.scales);
  a.gscale = w_gate_up.global_scale;
  a.a_codes = w + L.xc;
  a.a_scales = w + L.xs;
  a.offsets = offs;
  a.out = w + L.hc;
  a.out_scales = w + L.hs;
  a.status = reinterpret_cast<int*>(w + L.status);
  a.rows = rows;
  a.E = d.E;
  a.N = 2 * d.I;
  a.K = d.H;
  a.I = d.I;
  a.out_ld = d.I;
  e = cuda_rc(moe::launch_w4a4(0, a, s));
  if (e != MOE_OK || (e = mark(3)) != MOE_OK) return e;
  moe::W4a4Args b = a;
  b.w_codes = static_cast<const uint8_t*>(w_down.codes);
  b.w_scales = static_cast<const uint8_t*>(w_down.scales);
  b.gscale = w_down.global_scale;
  b.a_codes = w + L.hc;
  b.a_scales = w + L.hs;
  b.out = w + L.y;
  b.out_scales = nullptr;
  b.N = d.H;
  b.K = d.I;
  b.out_ld = d.H;
  e = cuda_rc(moe::launch_w4a4(1, b, s));
  if (e != MOE_OK || (e = mark(4)) != MOE_OK) return e;
  e = cuda_rc(moe::launch_combine(reinterpret_cast<const float*>(w + L.y), inv, wts, d.T, d.H, d.k, false, out, s));
  if (e != MOE_OK) return e;
  return mark(5);
}

int moe_quantize_nvfp4(const uint16_t* x, const int32_t* rows_of, int32_t n, int32_t K, uint8_t* codes,
                       uint8_t* scales, void* stream) {
  if (n < 0 || K <= 0 || K % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (x == nullptr || codes == nullptr || scales == nullptr) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(codes) || !al16(scales)) return MOE_ERR_MISALIGNED;
  return cuda_rc(moe::launch_quant_gather(x, rows_of, n, K, codes, scales, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_quantize_nvfp4_f32(const float* x, const int32_t* rows_of, int32_t n, int32_t K, uint8_t* codes,
                           uint8_t* scales, void* stream) {
  if (n < 0 || K <= 0 || K % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  if (x == nullptr || codes == nullptr || scales == nullptr) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(codes) || !al16(scales)) return MOE_ERR_MISALIGNED;
  return cuda_rc(moe::launch_quant_gather(x, rows_of, n, K, codes, scales, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

extern "C" int moe_debug_w4a4_gemm(int32_t mode, const uint8_t* act_codes, const uint8_t* act_scales,
                                   const int32_t* offsets, moe_w4n w, moe_dims d, void* out, uint8_t* out_scales,
                                   void* ws, void* stream) {
  const int rc = check4(d);
  if (rc != MOE_OK) return rc;
  if (mode != 0 && mode != 1) return MOE_ERR_INVALID_ARG;
  if (act_codes == nullptr || act_scales == nullptr || offsets == nullptr || w.codes == nullptr ||
      w.scales == nullptr || w.global_scale == nullptr || out == nullptr || ws == nullptr ||
      (mode == 0 && out_scales == nullptr))
    return MOE_ERR_INVALID_ARG;
  if (!al16(act_codes) || !al16(act_scales) || !al16(w.codes) || !al16(w.scales) || !al16(out) ||
      (mode == 0 && !al16(out_scales)))
    return MOE_ERR_MISALIGNED;
  moe::W4a4Args a{};
  a.w_codes = w.codes;
  a.w_scales = w.scales;
  a.gscale = w.global_scale;
  a.a_codes = act_codes;
  a.a_scales = act_scales;
  a.offsets = offsets;
  a.out = out;
  a.out_scales = out_scales;
  a.status = static_cast<int*>(ws);
  a.rows = d.T * d.k;
  a.E = d.E;
  a.I = d.I;
  a.N = mode == 0 ? 2 * d.I : d.H;
  a.K = mode == 0 ? d.H : d.I;
  a.out_ld = mode == 0 ? d.I : d.H;
  return cuda_rc(moe::launch_w4a4(mode, a, reinterpret_cast<cudaStream_t>(stream)));
}
