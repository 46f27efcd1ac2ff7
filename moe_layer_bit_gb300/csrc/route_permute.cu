// route_permute.cu -- top-k routing, the grouping permutation (histogram ->
// scan -> stable scatter + row gather) and the weighted combine.
//
// Routing and combine follow the ATOM article (itsolotime.com/archives/33112),
// section "8.1 MoE 路径：路由、专家并行与 MORI 通信" (routing, top-k selection,
// final combine) and the Atlas article (f.mffb.com.cn/a/497905.html), section
// "KV Cache量化、MTP推测解码和调试工具链" (gate logits -> expert IDs).  The
// permutation realises the per-expert row blocks that the Atlas article's
// grouped W4A16 GEMM (section "编译时内核选择和W4A16 Grouped GEMM") tiles over.
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "kernels.h"

namespace moe {

// Kernels here read what the kernel before them wrote, after pdl_wait(), so
// their loads use the coherent path (no ld.global.nc).

// --------------------------------------------------------------- routing
// Order-preserving map of a logit to an unsigned key: NaN ranks as -inf and
// -0 as +0 (they compare equal), every real logit maps above 0, and 0 marks
// an expert that is already chosen or does not exist.
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (isnan(v)) v = -INFINITY;
  if (v == 0.0f) v = 0.0f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One warp routes one token.  Lane l holds experts l, l+32, ..., NV per lane
// (NV * 32 >= E).  k rounds of a warp arg-max in (key desc, index asc) order:
// each lane's best (strict > over ascending experts keeps the lower index),
// then a warp max of the keys and a warp min of the indices holding it.  Gate
// weights: softmax over the k selected logits, fp32 with expf, summed in slot
// order.  Lane j < k returns slot j's expert and weight.
template <int NV>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k, int& out_id, float& out_w) {
  const int lane = threadIdx.x & 31;
  uint32_t key[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? logit_key(row[e]) : 0u;
  }
  uint32_t sel = 0;  // lane j keeps slot j's key and expert
  int sel_id = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t best = 0, bi = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      if (key[i] > best) {
        best = key[i];
        bi = (uint32_t)(lane + 32 * i);
      }
    }
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, best);  // > 0: k <= E real experts
    const uint32_t e_sel = __reduce_min_sync(0xFFFFFFFFu, best == m ? bi : 0xFFFFFFFFu);
    if ((int)(e_sel & 31u) == lane) {
#pragma unroll
      for (int i = 0; i < NV; ++i)
        if (i == (int)(e_sel >> 5)) key[i] = 0u;
    }
    if (lane == j) {
      sel = m;
      sel_id = (int)e_sel;
    }
  }
  const float sel_key = key_logit(sel);
  const float kmax = __shfl_sync(0xFFFFFFFFu, sel_key, 0);
  float z = 0.f;
  if (lane < k) z = (kmax == -INFINITY) ? 1.f : expf(sel_key - kmax);
  float sum = 0.f;  // ordered sum over slots 0..k-1 (same order on every lane)
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, z, j);
  out_id = sel_id;
  out_w = (kmax == -INFINITY) ? 1.f / (float)k : z / sum;
}

constexpr int kRouteWarps = 8;

template <int NV>
__global__ void __launch_bounds__(kRouteWarps * 32) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                                       int k, int32_t* __restrict__ ids,
                                                                       float* __restrict__ wts) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  pdl_wait();
  pdl_trigger();
  if (t >= T) return;
  int id;
  float w;
  route_token<NV>(logits + (size_t)t * E, E, k, id, w);
  if (lane < k) {
    ids[(size_t)t * k + lane] = id;
    wts[(size_t)t * k + lane] = w;
  }
}

// Values per lane: the smallest power of two >= ceil(E / 32).
static int route_nv(int E) {
  const int need = (E + 31) / 32;
  int nv = 1;
  while (nv < need) nv <<= 1;
  return nv;
}

#define MOE_DISPATCH_NV(nv, ...)                  \
  switch (nv) {                                   \
    case 1: { constexpr int NV = 1; __VA_ARGS__; } break;   \
    case 2: { constexpr int NV = 2; __VA_ARGS__; } break;   \
    case 4: { constexpr int NV = 4; __VA_ARGS__; } break;   \
    case 8: { constexpr int NV = 8; __VA_ARGS__; } break;   \
    case 16: { constexpr int NV = 16; __VA_ARGS__; } break; \
    default: { constexpr int NV = 32; __VA_ARGS__; } break; \
  }

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kRouteWarps - 1) / kRouteWarps;
  cudaError_t err;
  MOE_DISPATCH_NV(route_nv(E), err = launch_pdl(route_topk_kernel<NV>, dim3(blocks), dim3(kRouteWarps * 32), 0, s,
                                                logits, T, E, k, ids, w));
  return err;
}

// ------------------------------------------------------------ permutation
// Pairs i = t*k + j are cut into chunks of kPermChunk.  (a) per-chunk expert
// histograms; (b) per expert, an exclusive scan over chunks plus the expert
// offsets; (c) per chunk, a stable scatter.  Inside a block the stable rank of
// pair i among the block's pairs with the same expert and a lower index is
// (pairs of that expert in lower warps: a per-warp count table scanned over
// warps) + (lower lanes of the same warp: match_any + popc), so the result is
// independent of scheduling.
constexpr int kPermChunk = 1024;

// The grouped view of the (token, slot) pairs: ks slots per token, the first
// k routed (ids [T][k]) and, when ks == k + 1, a last slot for the shared
// expert, which takes index E_r (after the E_r routed experts).
__device__ __forceinline__ int pair_expert(const int32_t* ids, int g, int k, int ks, int E_r) {
  if (ks == k) return ids[g];
  const int t = g / ks, j = g - t * ks;
  return j < k ? ids[t * k + j] : E_r;
}

// The rank kernels run 32 warps (kPermChunk threads).  Rank table: uint16
// [E][32], expert-major, so a warp scans one expert's 32 per-warp counts with
// lane = warp index.
constexpr int kRankWarps = kPermChunk / 32;
static size_t rank_table_bytes(int E) { return (size_t)E * kRankWarps * sizeof(uint16_t); }

// Phase 1 of the stable rank (every thread of the block, pair e / valid):
// returns the pair's rank among the lower lanes of its warp with the same
// expert and records the warp's count of e in tab[e][warp].  `tab` is zero
// on entry; a __syncthreads must follow before block_rank_scan.
__device__ __forceinline__ int warp_rank_and_count(int e, bool valid, uint16_t* tab) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int key = valid ? e : -1 - lane;  // padding pairs: unique keys
  const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key);
  if (valid && lane == __ffs(peers) - 1) tab[e * kRankWarps + warp] = (uint16_t)__popc(peers);
  return __popc(peers & ((1u << lane) - 1u));
}

// Phase 2: per expert, the exclusive prefix over warps replaces tab[e][w];
// cnt[e] (if cnt != nullptr) receives the block's count of e.  Warp w scans
// experts w, w+32, ...  A __syncthreads must follow.
__device__ __forceinline__ void block_rank_scan(uint16_t* tab, int32_t* cnt, int E) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = warp; e < E; e += kRankWarps) {
    const uint32_t c = tab[e * kRankWarps + lane];
    uint32_t incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += y;
    }
    tab[e * kRankWarps + lane] = (uint16_t)(incl - c);
    if (cnt != nullptr && lane == 31) cnt[e] = (int32_t)incl;
  }
}

__global__ void __launch_bounds__(256) perm_hist_kernel(const int32_t* __restrict__ ids, int n, int E, int k, int ks,
                                                        int32_t* __restrict__ chunk_counts) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const int base = blockIdx.x * kPermChunk;
  for (int i = threadIdx.x; i < kPermChunk; i += blockDim.x) {
    const int g = base + i;
    if (g < n) atomicAdd(&hist[pair_expert(ids, g, k, ks, E - (ks - k))], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(size_t)blockIdx.x * E + e] = hist[e];
}

// Exclusive scan of E <= 1024 values held one per thread (blockDim 1024 or
// >= E); returns this thread's exclusive prefix and the total via *total.
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t x, int32_t* warp_tot, int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t incl = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += y;
    }
    warp_tot[lane] = w;  // inclusive
  }
  __syncthreads();
  *total = warp_tot[(blockDim.x >> 5) - 1];
  return incl - x + (warp > 0 ? warp_tot[warp - 1] : 0);
}

// One block of 1024 threads; thread e owns expert e.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ chunk_counts, int nchunks, int E,
                                                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                         int32_t* __restrict__ zero_e) {
  __shared__ int32_t warp_tot[32];
  const int e = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  int32_t run = 0;
  if (e < E) {
    for (int b = 0; b < nchunks; ++b) {
      const int32_t c = chunk_counts[(size_t)b * E + e];
      chunk_counts[(size_t)b * E + e] = run;
      run += c;
    }
    counts[e] = run;
    if (zero_e != nullptr) zero_e[e] = 0;
  }
  if (zero_e != nullptr && e < kSchedInts) zero_e[E + e] = 0;  // the schedule counters after them
  int32_t total;
  const int32_t excl = block_exclusive_scan(run, warp_tot, &total);
  if (e < E) {
    offsets[e] = excl;
    for (int b = 0; b < nchunks; ++b) chunk_counts[(size_t)b * E + e] += excl;
    if (e == E - 1) offsets[E] = excl + run;
  }
}

// Shared memory of the scatter kernel: base[E] int32, then the rank table.
static size_t scatter_smem_bytes(int E) { return (size_t)E * sizeof(int32_t) + rank_table_bytes(E); }

// One block of kPermChunk threads per chunk; thread i owns pair base + i.
__global__ void __launch_bounds__(kPermChunk) perm_scatter_kernel(const int32_t* __restrict__ ids, int n, int E, int k,
                                                                  int ks,
                                                                  const int32_t* __restrict__ chunk_base,
                                                                  int32_t* __restrict__ sorted_token,
                                                                  int32_t* __restrict__ inv_perm) {
  extern __shared__ int32_t smem_i[];
  int32_t* base = smem_i;
  uint16_t* tab = reinterpret_cast<uint16_t*>(smem_i + E);
  const int g = blockIdx.x * kPermChunk + threadIdx.x;
  const int warp = threadIdx.x >> 5;
  for (int x = threadIdx.x; x < E * kRankWarps; x += blockDim.x) tab[x] = 0;
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < E; e += blockDim.x) base[e] = chunk_base[(size_t)blockIdx.x * E + e];
  const bool valid = g < n;
  const int e = valid ? pair_expert(ids, g, k, ks, E - (ks - k)) : 0;
  __syncthreads();
  const int rank = warp_rank_and_count(e, valid, tab);
  __syncthreads();
  block_rank_scan(tab, nullptr, E);
  __syncthreads();
  if (valid) {
    const int pos = base[e] + tab[e * kRankWarps + warp] + rank;
    sorted_token[pos] = g / ks;
    inv_perm[g] = pos;
  }
}

// All pairs in one block (T*k <= kPermChunk), routing optionally included:
// with logits != nullptr the block first routes its T tokens (one warp per
// token, warps striding), writing ids / weights; then per-warp counts, the
// scans over warps and over experts, and the stable scatter, in one launch.
// 16-byte vectors each thread of a copy block moves (64 KiB per 1024-thread block)
constexpr int kCopyVecPerThread = 4;

template <int NV>
__global__ void __launch_bounds__(kPermChunk) route_permute_small_kernel(
    const float* __restrict__ logits, int T, int E, int k, int ks, int32_t* __restrict__ ids, float* __restrict__ wts,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_token,
    int32_t* __restrict__ inv_perm, int32_t* __restrict__ zero_e, const uint4* __restrict__ copy_src,
    uint4* __restrict__ copy_dst, long long copy_vec) {
  if (blockIdx.x > 0) {
    // a copy block: its share of the copy (kCopyVecPerThread 16-byte vectors
    // per thread, loads before stores), ordered after the kernels before
    pdl_wait();
    pdl_trigger();
    const long long v0 = (long long)(blockIdx.x - 1) * blockDim.x * kCopyVecPerThread + threadIdx.x;
    uint4 v[kCopyVecPerThread];
#pragma unroll
    for (int u = 0; u < kCopyVecPerThread; ++u) {
      const long long i = v0 + (long long)u * blockDim.x;
      if (i < copy_vec) v[u] = copy_src[i];
    }
#pragma unroll
    for (int u = 0; u < kCopyVecPerThread; ++u) {
      const long long i = v0 + (long long)u * blockDim.x;
      if (i < copy_vec) copy_dst[i] = v[u];
    }
    return;
  }
  // E routed experts; the grouping sees EG = E + (ks - k) (the shared expert last)
  const int EG = E + (ks - k);
  extern __shared__ int32_t smem_i[];
  int32_t* base = smem_i;                                  // [EG] counts, then offsets
  int32_t* s_ids = smem_i + EG;                            // [kPermChunk]
  uint16_t* tab = reinterpret_cast<uint16_t*>(smem_i + EG + kPermChunk);
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = T * ks;
  for (int x = tid; x < EG * kRankWarps; x += blockDim.x) tab[x] = 0;
  pdl_wait();
  pdl_trigger();
  if (logits != nullptr) {
    for (int t = warp; t < T; t += kRankWarps) {
      int id;
      float w;
      route_token<NV>(logits + (size_t)t * E, E, k, id, w);
      if (lane < k) {
        s_ids[t * ks + lane] = id;
        ids[(size_t)t * k + lane] = id;
        wts[(size_t)t * k + lane] = w;
      }
      if (ks > k && lane == k) s_ids[t * ks + k] = E;
    }
  } else {
    for (int i = tid; i < n; i += blockDim.x) s_ids[i] = pair_expert(ids, i, k, ks, E);
  }
  __syncthreads();
  const bool valid = tid < n;
  const int e = valid ? s_ids[tid] : 0;
  const int t = tid / ks;
  // When this block routed the tokens itself, a token meets an expert at most
  // once, so the pairs of expert e in pair order are its tokens in token
  // order.  Then, for T <= 256, the block keeps per expert a bitmap of its
  // tokens (W words, in the zeroed rank table): the count is its popcount and
  // a pair's rank the popcount of the lower bits.  Otherwise (ids given, or
  // larger T) it uses the per-warp count table.
  const int W = (T + 31) >> 5;
  const bool bitmap = logits != nullptr && W <= 8;
  uint32_t* bm = reinterpret_cast<uint32_t*>(tab);  // [EG][W]
  int rank = 0;
  if (bitmap) {
    if (valid) atomicOr(&bm[e * W + (t >> 5)], 1u << (t & 31));
    __syncthreads();
    for (int ex = tid; ex < EG; ex += blockDim.x) {
      int cnt = 0;
      for (int w = 0; w < W; ++w) cnt += __popc(bm[ex * W + w]);
      base[ex] = cnt;
    }
  } else {
    rank = warp_rank_and_count(e, valid, tab);
    __syncthreads();
    block_rank_scan(tab, base, EG);  // base[e] = count of e
  }
  __syncthreads();
  const int32_t c = tid < EG ? base[tid] : 0;
  int32_t total;
  const int32_t excl = block_exclusive_scan(c, warp_tot, &total);
  if (tid < EG) {
    counts[tid] = c;
    offsets[tid] = excl;
    base[tid] = excl;
    if (tid == EG - 1) offsets[EG] = excl + c;
    if (zero_e != nullptr) zero_e[tid] = 0;
  }
  if (zero_e != nullptr && tid < kSchedInts) zero_e[EG + tid] = 0;  // the schedule counters after them
  __syncthreads();
  if (valid) {
    int pos = base[e];
    if (bitmap) {
      for (int w = 0; w < (t >> 5); ++w) pos += __popc(bm[e * W + w]);
      pos += __popc(bm[e * W + (t >> 5)] & ((1u << (t & 31)) - 1u));
    } else {
      pos += tab[e * kRankWarps + warp] + rank;
    }
    sorted_token[pos] = t;
    inv_perm[tid] = pos;
  }
}

static size_t small_smem_bytes(int E) { return (size_t)(E + kPermChunk) * sizeof(int32_t) + rank_table_bytes(E); }

// x_perm[p] = x[sorted_token[p]] (H % 8 == 0): one warp copies a row at a
// time, its lanes taking the row's 16-byte vectors c = lane, lane + 32, ...,
// kGatherUnroll loads in flight per lane before their stores; warps stride
// over the rows (no per-vector index division).
constexpr int kGatherUnroll = 8;
__global__ void __launch_bounds__(256) perm_gather_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ sorted_token, int n,
                                                          int vec_per_row, uint16_t* __restrict__ x_perm) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int nwarps = (int)(gridDim.x * blockDim.x) >> 5;
  for (int p = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); p < n; p += nwarps) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)sorted_token[p] * vec_per_row * 8);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)p * vec_per_row * 8);
    for (int c0 = 0; c0 < vec_per_row; c0 += 32 * kGatherUnroll) {
      uint4 v[kGatherUnroll];
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) {
        const int c = c0 + 32 * u + lane;
        if (c < vec_per_row) v[u] = __ldg(src + c);
      }
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) {
        const int c = c0 + 32 * u + lane;
        if (c < vec_per_row) dst[c] = v[u];
      }
    }
  }
}

size_t perm_scratch_bytes(int T, int E, int k) {
  const size_t n = (size_t)T * k;
  const size_t nchunks = (n + kPermChunk - 1) / kPermChunk;
  return (nchunks > 0 ? nchunks : 1) * (size_t)E * sizeof(int32_t);
}

cudaError_t launch_gather(const uint16_t* x, const int32_t* sorted_token, int n, int H, uint16_t* x_perm,
                                 cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int vpr = H / 8;
  // one row per warp, at most 16 blocks of 8 warps per SM
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  long long blocks = ((long long)n + 7) / 8;
  if (blocks > 16LL * sms) blocks = 16LL * sms;
  return launch_pdl(perm_gather_kernel, dim3((unsigned)blocks), dim3(256), 0, s, x, sorted_token, n, vpr, x_perm);
}

// E routed experts, k routed slots, ks slots per token in the grouped view
// (k + 1 with the shared expert, which groups as expert E).
// Block 0 routes and groups; blocks 1.. (when copy_bytes > 0) copy.
template <int NV>
static cudaError_t launch_small(const float* logits, int T, int E, int k, int ks, int32_t* ids, float* w,
                                int32_t* counts, int32_t* offsets, int32_t* sorted_token, int32_t* inv_perm,
                                int32_t* zero_e, cudaStream_t s, const void* copy_src = nullptr,
                                void* copy_dst = nullptr, size_t copy_bytes = 0) {
  const size_t smem = small_smem_bytes(E + (ks - k));
  auto kern = route_permute_small_kernel<NV>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const long long nvec = (long long)(copy_bytes / 16);
  const long long per_block = (long long)kPermChunk * kCopyVecPerThread;
  const long long copy_blocks = (nvec + per_block - 1) / per_block;
  return launch_pdl(kern, dim3((unsigned)(1 + copy_blocks)), dim3(kPermChunk), smem, s, logits, T, E, k, ks, ids, w,
                    counts, offsets, sorted_token, inv_perm, zero_e, static_cast<const uint4*>(copy_src),
                    static_cast<uint4*>(copy_dst), nvec);
}

static cudaError_t launch_chunked(const int32_t* ids, int T, int E, int k, int ks, int32_t* counts, int32_t* offsets,
                                  int32_t* sorted_token, int32_t* inv_perm, int32_t* scratch, int32_t* zero_e,
                                  cudaStream_t s) {
  const int n = T * ks, EG = E + (ks - k);
  const int nchunks = (n + kPermChunk - 1) / kPermChunk;
  cudaError_t err =
      launch_pdl(perm_hist_kernel, dim3(nchunks), dim3(256), EG * sizeof(int32_t), s, ids, n, EG, k, ks, scratch);
  if (err != cudaSuccess) return err;
  err = launch_pdl(perm_scan_kernel, dim3(1), dim3(1024), 0, s, scratch, nchunks, EG, counts, offsets, zero_e);
  if (err != cudaSuccess) return err;
  const size_t smem = scatter_smem_bytes(EG);
  err = cudaFuncSetAttribute(perm_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(perm_scatter_kernel, dim3(nchunks), dim3(kPermChunk), smem, s, ids, n, EG, k, ks,
                    (const int32_t*)scratch, sorted_token, inv_perm);
}

cudaError_t launch_permute(const int32_t* ids, const uint16_t* x, int T, int H, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* sorted_token, int32_t* inv_perm, uint16_t* x_perm,
                           int32_t* scratch, cudaStream_t s) {
  const int n = T * k;
  cudaError_t err = (n <= kPermChunk)
                        ? launch_small<1>(nullptr, T, E, k, k, const_cast<int32_t*>(ids), nullptr, counts, offsets,
                                          sorted_token, inv_perm, nullptr, s)
                        : launch_chunked(ids, T, E, k, k, counts, offsets, sorted_token, inv_perm, scratch, nullptr, s);
  if (err != cudaSuccess) return err;
  return launch_gather(x, sorted_token, n, H, x_perm, s);
}

// Routing runs inside the single grouping block only while the logits are
// small enough for one SM to read quickly (T*E floats, 128 KiB).
constexpr long long kFusedRouteLogits = 32768;

int route_group_launches(int T, int E, int k, bool shared) {
  const int n = T * (k + (shared ? 1 : 0));
  if (n <= kPermChunk && (long long)T * E <= kFusedRouteLogits) return 1;
  return n <= kPermChunk ? 2 : 4;
}

bool route_group_copies(int T, int E, int k, bool shared) { return route_group_launches(T, E, k, shared) == 1; }

cudaError_t launch_route_group(const float* logits, int T, int E, int k, bool shared, int32_t* ids, float* w,
                               int32_t* counts, int32_t* offsets, int32_t* sorted_token, int32_t* inv_perm,
                               int32_t* scratch, int32_t* zero_e, cudaStream_t s, const void* copy_src,
                               void* copy_dst, size_t copy_bytes) {
  const int ks = k + (shared ? 1 : 0);
  const int n = T * ks;
  cudaError_t err;
  if (copy_bytes > 0 && (!route_group_copies(T, E, k, shared) || copy_bytes % 16 != 0 || copy_src == nullptr ||
                         copy_dst == nullptr || (reinterpret_cast<uintptr_t>(copy_src) & 15u) != 0 ||
                         (reinterpret_cast<uintptr_t>(copy_dst) & 15u) != 0))
    return cudaErrorInvalidValue;
  if (n <= kPermChunk && (long long)T * E <= kFusedRouteLogits) {
    MOE_DISPATCH_NV(route_nv(E), err = (launch_small<NV>(logits, T, E, k, ks, ids, w, counts, offsets, sorted_token,
                                                         inv_perm, zero_e, s, copy_src, copy_dst, copy_bytes)));
    return err;
  }
  err = launch_route_topk(logits, T, E, k, ids, w, s);
  if (err != cudaSuccess) return err;
  if (n <= kPermChunk)
    return launch_small<1>(nullptr, T, E, k, ks, ids, nullptr, counts, offsets, sorted_token, inv_perm, zero_e, s);
  return launch_chunked(ids, T, E, k, ks, counts, offsets, sorted_token, inv_perm, scratch, zero_e, s);
}

// ------------------------------------------------------------------ combine
// out[t, c] = bf16_rne(sum_j w[t,j] * y[inv[t*ks+j], c]) with the fp32 sum in
// ascending j over the k routed slots, then, with a shared expert (ks == k +
// 1), plus y[inv[t*ks+k], c] (weight 1).  A block of kCombineThreads takes
// 4 * kCombineThreads columns of one token; the token's rows and weights are
// staged in shared memory first so the row loads of a thread are independent.
constexpr int kCombineThreads = 128;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const float* __restrict__ y,
                                                                  const int32_t* __restrict__ inv,
                                                                  const float* __restrict__ w, int T, int H, int k,
                                                                  int ks, uint16_t* __restrict__ out) {
  __shared__ int32_t s_row[33];
  __shared__ float s_w[33];
  const int t = blockIdx.y;
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < ks) {
    s_row[threadIdx.x] = inv[(size_t)t * ks + threadIdx.x];
    s_w[threadIdx.x] = threadIdx.x < k ? w[(size_t)t * k + threadIdx.x] : 1.0f;
  }
  __syncthreads();
  if (c4 * 4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int j = 0; j < k; ++j) {
    const float wj = s_w[j];
    const float4 v = reinterpret_cast<const float4*>(y + (size_t)s_row[j] * H)[c4];
    acc.x = fmaf(wj, v.x, acc.x);
    acc.y = fmaf(wj, v.y, acc.y);
    acc.z = fmaf(wj, v.z, acc.z);
    acc.w = fmaf(wj, v.w, acc.w);
  }
  if (ks > k) {
    const float4 v = reinterpret_cast<const float4*>(y + (size_t)s_row[k] * H)[c4];
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(out + (size_t)t * H)[c4] = pk;
}

cudaError_t launch_combine(const float* y, const int32_t* inv, const float* w, int T, int H, int k, bool shared,
                           uint16_t* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  dim3 grid((H / 4 + kCombineThreads - 1) / kCombineThreads, T);
  return launch_pdl(combine_kernel, grid, dim3(kCombineThreads), 0, s, y, inv, w, T, H, k, k + (shared ? 1 : 0), out);
}

}  // namespace moe
