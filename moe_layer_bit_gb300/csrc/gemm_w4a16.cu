// gemm_w4a16.cu -- the grouped W4A16 NVFP4 GEMMs (gate_up + SwiGLU, down) on
// tcgen05 tensor cores, the weight prepack and the dequantiser test kernel.
//
// What is computed: the Atlas article (f.mffb.com.cn/a/497905.html), section
// "编译时内核选择和W4A16 Grouped GEMM": both projections of every expert in one
// launch, packed FP4 weights dequantised to BF16 on chip and multiplied
// against BF16 activations by a BF16 MMA, dequant and GEMM fused (no BF16
// weight written back).  SwiGLU as in "Rust 实现深度学习推理引擎：从计算图到异构
// 硬件加速" (ybb.press/ai-applications/14151.html), section "三、计算图".
//
// How (sm_103a design; the article's GB10 kernel uses a 3D grid
// (ceil(N/64), max_m_tiles, num_experts) and dequantises into shared memory):
//  * swap-AB: the weight tile is the MMA's M=128 operand, the expert's tokens
//    are N (16..128), so a decode step with 2 tokens per expert still runs a
//    legal tcgen05 shape and every weight byte is read once per token tile;
//  * a persistent CTA per SM walks a device-side tile list built from the
//    expert offsets (no host sync, no empty CTAs);
//  * warp roles: one producer thread issues a 1-D bulk copy of the packed
//    weight block (codes + E4M3 scales, 4608 B) and a 2-D TMA copy of the
//    128-byte-swizzled activation tile per stage; eight dequant warps turn the
//    codes into exact bf16 (value * 2^-7) and store them straight into tensor
//    memory as the MMA's A operand (tcgen05.st), so no dequantised weight ever
//    touches shared memory; one thread issues tcgen05.mma (A from TMEM, B from
//    shared memory, fp32 accumulator in TMEM, double-buffered); four epilogue
//    warps read the accumulator (tcgen05.ld), apply global_scale * 2^7, and
//    write SwiGLU(bf16) or fp32 rows.
//  * every barrier wait is bounded (about 1 s); on expiry the CTA records a
//    timeout in the status word, drains its copies and MMAs and exits.
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kStages = 8;
constexpr int kWarpEpi0 = 0;       // warps 0..3: epilogue (TMEM lane quadrant = warp)
constexpr int kWarpDq0 = 4;        // warps 4..11: dequant (quadrant = warp % 4, K half = (warp-4)/4)
constexpr int kWarpProducer = 12;  // warp 12: copies
constexpr int kWarpMma = 13;       // warp 13: TMEM owner + MMA issue
constexpr int kThreads = 14 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemA0 = 256;  // A ring: columns [256, 256 + 32 * kStages)
constexpr int kMinSmem = 120 * 1024;  // keeps one CTA (one TMEM allocation) per SM

template <int BN>
struct Smem {
  static constexpr int kBTile = BN * 128;  // BN rows x 64 bf16, 128-byte swizzled
  static constexpr int kOffB = 0;
  static constexpr int kOffW = kStages * kBTile;
  static constexpr int kOffBar = kOffW + kStages * kWBlockBytes;
  // full[S], empty[S], afull[S], dfull[2], dempty[2], drain
  static constexpr int kNumBars = 3 * kStages + 5;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // [0] tmem base, [1] abort, [2] total tiles
  static constexpr int kOffTables = kOffMisc + 16;         // offsets[E+1], prefix[E+1]
  static int bytes(int E) {
    int b = kOffTables + 2 * (E + 1) * 4 + 1024;  // + alignment slack
    return b < kMinSmem ? kMinSmem : b;
  }
};

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }

struct TileCoord {
  int e, mt, nt;
};

// Largest e with prefix[e] <= t (experts with no tiles have prefix[e] == prefix[e+1]).
__device__ __forceinline__ TileCoord decode_tile(int t, const int32_t* prefix, const int32_t* offs, int E, int BN) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= t) lo = mid;
    else hi = mid;
  }
  const int cnt = offs[lo + 1] - offs[lo];
  const int nt_count = (cnt + BN - 1) / BN;
  const int local = t - prefix[lo];
  TileCoord c;
  c.e = lo;
  c.mt = local / nt_count;
  c.nt = local - c.mt * nt_count;
  return c;
}

template <int BN, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_gemm_kernel(const __grid_constant__ CUtensorMap tmap_act, const uint8_t* __restrict__ packed,
                      const float* __restrict__ gscale, const int32_t* __restrict__ offsets, void* __restrict__ out,
                      int* __restrict__ status, int E, int N, int K, int out_ld) {
  using L = Smem<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sB = sbase + L::kOffB;
  const uint32_t sW = sbase + L::kOffW;
  const uint32_t bar0 = sbase + L::kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto afull_bar = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
  auto dfull_bar = [&](int d) { return bar0 + 8u * (3 * kStages + d); };
  auto dempty_bar = [&](int d) { return bar0 + 8u * (3 * kStages + 2 + d); };
  const uint32_t drain_bar = bar0 + 8u * (3 * kStages + 4);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + L::kOffTables);
  int32_t* s_prefix = s_off + (E + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int MT = N / kTileM;
  const int KB = K / kBlockK;

  // ---- set-up: barriers, TMEM, tile table
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(afull_bar(s), 8);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(dfull_bar(d), 1);
      mbar_init(dempty_bar(d), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpProducer && lane == 0) prefetch_tmap(&tmap_act);
  if (warp == kWarpMma) {
    tmem_alloc(sbase + L::kOffMisc, kTmemCols);
    tmem_relinquish();
  }
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = __ldg(offsets + i);
  __syncthreads();
  if (warp == 0) {
    // prefix[e] = first tile of expert e; tiles of e = ceil(count/BN) * MT
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int sum = 0;
    for (int e = e0; e < e0 + per && e < E; ++e) sum += ((s_off[e + 1] - s_off[e] + BN - 1) / BN) * MT;
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += y;
    }
    int run = incl - sum;
    for (int e = e0; e < e0 + per && e < E; ++e) {
      s_prefix[e] = run;
      run += ((s_off[e + 1] - s_off[e] + BN - 1) / BN) * MT;
    }
    if (lane == 31) {
      s_prefix[E] = incl;
      misc[2] = (uint32_t)incl;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const int total = (int)misc[2];

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_par = 0;  // per-stage: issued at least once / parity of the last issue
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileCoord c = decode_tile(t, s_prefix, s_off, E, BN);
        const uint8_t* wsrc = packed + (size_t)(c.e * MT + c.mt) * KB * kWBlockBytes;
        const int row0 = s_off[c.e] + c.nt * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), (uint32_t)(kWBlockBytes + L::kBTile));
          bulk_copy_g2s(sW + stage * kWBlockBytes, wsrc + (size_t)kb * kWBlockBytes, kWBlockBytes, full_bar(stage));
          tma_load_2d(sB + stage * L::kBTile, &tmap_act, kb * kBlockK, row0, full_bar(stage));
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: every copy this thread issued has landed before the CTA exits
      for (int s = 0; s < kStages; ++s)
        if ((issued >> s) & 1u) mbar_wait(full_bar(s), (last_par >> s) & 1u, nullptr, status, kDrainTimeoutNs);
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTileM, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const int d = it & 1;
        const uint32_t dph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(dempty_bar(d), dph ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(d * BN);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(afull_bar(stage), phase, abort_flag, status) ||
              !mbar_wait(full_bar(stage), phase, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem_base + kTmemA0 + (uint32_t)stage * 32u;
          const uint32_t b_addr = sB + stage * L::kBTile;
#pragma unroll
          for (int kk = 0; kk < kBlockK / 16; ++kk)
            tc_mma_ts(d_tmem, a_tmem + kk * 8u, smem_desc_sw128(b_addr + kk * 32u), idesc, (kb | kk) != 0);
          tc_commit(empty_bar(stage));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit(dfull_bar(d));
      }
      // drain: all MMAs issued by this thread complete before TMEM is freed
      tc_commit(drain_bar);
      mbar_wait(drain_bar, 0, nullptr, status, kDrainTimeoutNs);
    }
  } else if (warp >= kWarpDq0) {
    // ------------------------------------------------------------- dequant
    const int q = warp & 3;
    const int half = (warp - kWarpDq0) >> 2;
    const int r = 32 * q + lane;
    const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + kTmemA0 + (uint32_t)(half * 16);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      for (int kb = 0; kb < KB; ++kb) {
        // every lane waits (each acquires the copied bytes); the warp acts as one
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(full_bar(stage), phase, abort_flag, status))) {
          ok = false;
          break;
        }
        const uint8_t* blk = smem + L::kOffW + stage * kWBlockBytes;
        const uint4 cw = *reinterpret_cast<const uint4*>(blk + (half * 128 + r) * 16);
        const uint16_t sc = *reinterpret_cast<const uint16_t*>(blk + 4096 + (half * 128 + r) * 2);
        uint32_t s0, s1;
        e4m3x2_to_scaleprime(sc, s0, s1);
        uint32_t v[16];
        dequant_word(cw.x, s0, v + 0);
        dequant_word(cw.y, s0, v + 4);
        dequant_word(cw.z, s1, v + 8);
        dequant_word(cw.w, s1, v + 12);
        tmem_st16(t_row + (uint32_t)stage * 32u, v);
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(afull_bar(stage));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp - kWarpEpi0;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const TileCoord c = decode_tile(t, s_prefix, s_off, E, BN);
      const int d = it & 1;
      const uint32_t dph = (uint32_t)(it >> 1) & 1u;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(dfull_bar(d), dph, abort_flag, status))) break;
      tc_fence_after();
      const int p0 = s_off[c.e] + c.nt * BN;
      const int nvalid = min(BN, s_off[c.e + 1] - p0);
      const float gsc = __ldg(gscale + c.e) * 128.0f;
      const uint32_t t_acc = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(d * BN);
#pragma unroll 1
      for (int cc = 0; cc < BN / 16; ++cc) {
        uint32_t v[16];
        tmem_ld16(t_acc + (uint32_t)(cc * 16), v);
        tc_wait_ld();
        if (MODE == 0) {
          // rows 32q..32q+15 hold gate features f, rows 32q+16.. the matching up rows
          const int f = c.mt * 64 + 16 * q + (lane & 15);
          const bool is_gate = lane < 16;
          uint16_t* h = reinterpret_cast<uint16_t*>(out);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float a = __uint_as_float(v[j]);
            const float b = __uint_as_float(v[j + 8]);
            const float send = is_gate ? b : a;
            const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, 16);
            const float own = is_gate ? a : b;
            const float g = (is_gate ? own : recv) * gsc;
            const float u = (is_gate ? recv : own) * gsc;
            const int col = cc * 16 + j + (is_gate ? 0 : 8);
            if (col < nvalid) {
              const float hv = g / (1.0f + __expf(-g)) * u;
              h[(size_t)(p0 + col) * out_ld + f] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
            }
          }
        } else {
          const int n = c.mt * kTileM + 32 * q + lane;
          float* y = reinterpret_cast<float*>(out);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = cc * 16 + j;
            if (col < nvalid) y[(size_t)(p0 + col) * out_ld + n] = __uint_as_float(v[j]) * gsc;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty_bar(d));
    }
  }

  // ---- teardown: everyone is here; the MMA thread drained its work
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem_base, kTmemCols);
}

// ------------------------------------------------------------------ launch
using PFN_encodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                     const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled get_encode_fn() {
  static PFN_encodeTiled fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  }
  return fn;
}

template <int BN, int MODE>
static cudaError_t launch_gemm_bn(const GemmArgs& a, cudaStream_t s) {
  PFN_encodeTiled enc = get_encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t gdim[2] = {(cuuint64_t)a.K, (cuuint64_t)a.rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)a.K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBlockK, (cuuint32_t)BN};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.act), gdim, gstride, box,
                   estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const int MT = a.N / kTileM;
  const long long n = a.rows;
  const long long max_tiles = (long long)MT * (n / BN + (n < a.E ? n : a.E));
  int grid = (int)(max_tiles < sms ? max_tiles : sms);
  if (grid <= 0) return cudaSuccess;
  const int smem = Smem<BN>::bytes(a.E);
  auto kern = w4a16_gemm_kernel<BN, MODE>;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  kern<<<grid, kThreads, smem, s>>>(tmap, a.packed, a.gscale, a.offsets, a.out, a.status, a.E, a.N, a.K, a.out_ld);
  return cudaGetLastError();
}

// Token tile width: the smallest of 16/32/64/128 that covers about twice the
// mean number of rows per expert (T*k/E), so a decode step is one tile per
// expert and prefill uses the widest tile.
static int pick_bn(int rows, int E) {
  const long long mean2 = 2LL * rows / (E > 0 ? E : 1);
  if (mean2 <= 16) return 16;
  if (mean2 <= 32) return 32;
  if (mean2 <= 64) return 64;
  return 128;
}

cudaError_t launch_gemm(int mode, const GemmArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  const int bn = pick_bn(a.rows, a.E);
  if (mode == 0) {
    switch (bn) {
      case 16: return launch_gemm_bn<16, 0>(a, s);
      case 32: return launch_gemm_bn<32, 0>(a, s);
      case 64: return launch_gemm_bn<64, 0>(a, s);
      default: return launch_gemm_bn<128, 0>(a, s);
    }
  }
  switch (bn) {
    case 16: return launch_gemm_bn<16, 1>(a, s);
    case 32: return launch_gemm_bn<32, 1>(a, s);
    case 64: return launch_gemm_bn<64, 1>(a, s);
    default: return launch_gemm_bn<128, 1>(a, s);
  }
}

// ------------------------------------------------------------------ prepack
// One thread per (expert, 128-row tile, 64-column block, K half, tile row):
// copies 16 code bytes (32 elements) into the packed word order and the two
// E4M3 scales of those 32 elements.  Packed word w of a K half holds elements
// 8w..8w+7: even elements in nibbles 0..3 of the low 16 bits, odd elements in
// nibbles 0..3 of the high 16 bits.
__global__ void prepack_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, int E, int N,
                               int K, int proj, uint8_t* __restrict__ packed) {
  const int MT = N / kTileM, KB = K / kBlockK;
  const long long total = (long long)E * MT * KB * 256;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= total) return;
  const int r = (int)(gid & 127);
  const int half = (int)((gid >> 7) & 1);
  long long blk = gid >> 8;  // (e * MT + mt) * KB + kb
  const int kb = (int)(blk % KB);
  const long long em = blk / KB;
  const int mt = (int)(em % MT);
  const int e = (int)(em / MT);
  int row;
  if (proj == 0) {
    const int I = N / 2, g = r >> 5, w = r & 31;
    row = (w < 16) ? (mt * 64 + 16 * g + w) : (I + mt * 64 + 16 * g + (w - 16));
  } else {
    row = mt * kTileM + r;
  }
  const size_t src_row = (size_t)e * N + row;
  const uint8_t* cs = codes + src_row * (K / 2) + kb * 32 + half * 16;
  uint32_t words[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t o = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t b = cs[4 * w + j];
      o |= (b & 0xFu) << (4 * j);
      o |= (b >> 4) << (16 + 4 * j);
    }
    words[w] = o;
  }
  uint8_t* dst = packed + blk * kWBlockBytes;
  *reinterpret_cast<uint4*>(dst + (half * 128 + r) * 16) = make_uint4(words[0], words[1], words[2], words[3]);
  const uint8_t* ss = scales + src_row * (K / 16) + kb * 4 + half * 2;
  dst[4096 + (half * 128 + r) * 2 + 0] = ss[0];
  dst[4096 + (half * 128 + r) * 2 + 1] = ss[1];
}

cudaError_t launch_prepack(const uint8_t* codes, const uint8_t* scales, int E, int N, int K, int proj,
                           uint8_t* packed, cudaStream_t s) {
  const long long total = (long long)E * (N / kTileM) * (K / kBlockK) * 256;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  prepack_kernel<<<(unsigned)blocks, threads, 0, s>>>(codes, scales, E, N, K, proj, packed);
  return cudaGetLastError();
}

// ------------------------------------------------------- dequantiser table
// Thread s builds packed words holding codes 0..15 and dequantises them with
// scale byte s in the low half of the scale pair and 255-s in the high half,
// exactly as the GEMM's dequant warps do; out[s*16 + c] takes the low-half
// result of scale s and out[4096 + (255-s)*16 + c] the high-half result.
// Both tables are scaled back by 2^7 (exact) to e2m1(c) * e4m3(scale).
__global__ void dequant_table_kernel(uint16_t* __restrict__ out) {
  const int s = threadIdx.x;
  const uint16_t pair = (uint16_t)(s | ((255 - s) << 8));
  uint32_t s_lo, s_hi;
  e4m3x2_to_scaleprime(pair, s_lo, s_hi);
  for (int w = 0; w < 2; ++w) {
    uint32_t q = 0;
    for (int j = 0; j < 4; ++j) {
      q |= (uint32_t)(8 * w + 2 * j) << (4 * j);
      q |= (uint32_t)(8 * w + 2 * j + 1) << (16 + 4 * j);
    }
    uint32_t lo[4], hi[4];
    dequant_word(q, s_lo, lo);
    dequant_word(q, s_hi, hi);
    const uint32_t two7 = 0x43004300u;  // bf16 128.0 in both halves
    for (int j = 0; j < 4; ++j) {
      const uint32_t a = bf16x2_mul(lo[j], two7), b = bf16x2_mul(hi[j], two7);
      const int c = 8 * w + 2 * j;
      out[s * 16 + c] = (uint16_t)(a & 0xFFFFu);
      out[s * 16 + c + 1] = (uint16_t)(a >> 16);
      out[4096 + (255 - s) * 16 + c] = (uint16_t)(b & 0xFFFFu);
      out[4096 + (255 - s) * 16 + c + 1] = (uint16_t)(b >> 16);
    }
  }
}

cudaError_t launch_dequant_table(uint16_t* out, cudaStream_t s) {
  dequant_table_kernel<<<1, 256, 0, s>>>(out);
  return cudaGetLastError();
}

// ------------------------------------------------------ bounded-wait probe
// Waits on an mbarrier that nothing ever arrives at; the bounded wait must
// give up and record a timeout.  Used by the failure-detection test.
__global__ void timeout_probe_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

cudaError_t launch_timeout_probe(int* status, unsigned long long limit_ns, cudaStream_t s) {
  timeout_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
