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

#include "kernels.h"

namespace moe {

// --------------------------------------------------------------- routing
// One warp per token.  Lane l holds experts l, l+32, ... (up to 32 each, E <=
// 1024).  k rounds of a warp arg-max with (key desc, index asc) order, where
// key = logit with NaN mapped to -inf.  Gate weights: softmax over the k
// selected keys, fp32, expf, summed in slot order.
constexpr int kRouteWarps = 8;

__global__ void __launch_bounds__(kRouteWarps * 32) route_topk_kernel(const float* __restrict__ logits, int T, int E,
                                                                       int k, int32_t* __restrict__ ids,
                                                                       float* __restrict__ wts) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* row = logits + (size_t)t * E;
  float key[32];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int e = lane + 32 * i;
    float v = -INFINITY;
    if (e < E) {
      v = __ldg(row + e);
      if (isnan(v)) v = -INFINITY;
    }
    key[i] = v;
    if (e >= E) taken |= (1u << i);  // not a real expert
  }
  float sel_key = -INFINITY;   // lane j keeps the key of slot j
  int sel_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const bool ok = !((taken >> i) & 1u);
      const int e = lane + 32 * i;
      if (ok && (bi == 0x7FFFFFFF || key[i] > bv)) {  // ascending e: strict > keeps the lower index
        bv = key[i];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
      if (oi != 0x7FFFFFFF && (bi == 0x7FFFFFFF || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      sel_key = bv;
      sel_id = bi;
    }
  }
  const float kmax = __shfl_sync(0xFFFFFFFFu, sel_key, 0);
  float z = 0.f;
  if (lane < k) z = (kmax == -INFINITY) ? 1.f : expf(sel_key - kmax);
  // ordered sum over slots 0..k-1 (same order on every lane)
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, z, j);
  if (lane < k) {
    ids[(size_t)t * k + lane] = sel_id;
    wts[(size_t)t * k + lane] = (kmax == -INFINITY) ? 1.f / (float)k : z / sum;
  }
}

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kRouteWarps - 1) / kRouteWarps;
  route_topk_kernel<<<blocks, kRouteWarps * 32, 0, s>>>(logits, T, E, k, ids, w);
  return cudaGetLastError();
}

// ------------------------------------------------------------ permutation
// Pairs i = t*k + j are cut into chunks of kPermChunk.  (a) per-chunk expert
// histograms; (b) per expert, an exclusive scan over chunks plus the expert
// offsets; (c) per chunk, a stable scatter: the rank of pair i among the
// chunk's pairs with the same expert and a lower index is found warp by warp
// (match_any + popc), so the result is independent of scheduling.
constexpr int kPermChunk = 1024;

__global__ void __launch_bounds__(256) perm_hist_kernel(const int32_t* __restrict__ ids, int n, int E,
                                                        int32_t* __restrict__ chunk_counts) {
  extern __shared__ int32_t hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * kPermChunk;
  for (int i = threadIdx.x; i < kPermChunk; i += blockDim.x) {
    const int g = base + i;
    if (g < n) atomicAdd(&hist[__ldg(ids + g)], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(size_t)blockIdx.x * E + e] = hist[e];
}

// One block of 1024 threads; thread e owns expert e.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int32_t* __restrict__ chunk_counts, int nchunks, int E,
                                                         int32_t* __restrict__ counts, int32_t* __restrict__ offsets) {
  __shared__ int32_t warp_tot[32];
  const int e = threadIdx.x;
  int32_t run = 0;
  if (e < E) {
    for (int b = 0; b < nchunks; ++b) {
      const int32_t c = chunk_counts[(size_t)b * E + e];
      chunk_counts[(size_t)b * E + e] = run;
      run += c;
    }
    counts[e] = run;
  }
  // block exclusive scan of run over e
  const int lane = e & 31, warp = e >> 5;
  int32_t x = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t w = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += y;
    }
    warp_tot[lane] = w;  // inclusive
  }
  __syncthreads();
  const int32_t excl = x - run + (warp > 0 ? warp_tot[warp - 1] : 0);
  if (e < E) {
    offsets[e] = excl;
    for (int b = 0; b < nchunks; ++b) chunk_counts[(size_t)b * E + e] += excl;
    if (e == E - 1) offsets[E] = excl + run;
  }
}

// Stable rank of each pair among the block's pairs routed to the same expert:
// warp w's pairs follow warps 0..w-1 (ascending pair index), and inside a warp
// match_any + popc orders equal experts by lane.  `run[e]` starts at the first
// sorted row of expert e available to this block and ends past its last.
__device__ __forceinline__ int block_stable_position(int e, bool valid, int32_t* run) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int key = valid ? e : -1 - lane;   // invalid pairs: unique keys
  const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  const int leader = __ffs(peers) - 1;
  int pos = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    if (warp == w && valid) {
      pos = run[e] + rank;
      __syncwarp(peers);
      if (lane == leader) run[e] += __popc(peers);
    }
    __syncthreads();
  }
  return pos;
}

// One block of kPermChunk threads per chunk; thread i owns pair base + i.
__global__ void __launch_bounds__(kPermChunk) perm_scatter_kernel(const int32_t* __restrict__ ids, int n, int E, int k,
                                                                  const int32_t* __restrict__ chunk_base,
                                                                  int32_t* __restrict__ sorted_token,
                                                                  int32_t* __restrict__ inv_perm) {
  extern __shared__ int32_t run[];            // [E] running position per expert
  const int g = blockIdx.x * kPermChunk + threadIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) run[e] = chunk_base[(size_t)blockIdx.x * E + e];
  const bool valid = g < n;
  const int e = valid ? __ldg(ids + g) : 0;
  __syncthreads();
  const int pos = block_stable_position(e, valid, run);
  if (valid) {
    sorted_token[pos] = g / k;
    inv_perm[g] = pos;
  }
}

// All pairs in one block (T*k <= kPermChunk): histogram, scan and stable
// scatter in a single launch.
__global__ void __launch_bounds__(kPermChunk) perm_single_kernel(const int32_t* __restrict__ ids, int n, int E, int k,
                                                                 int32_t* __restrict__ counts,
                                                                 int32_t* __restrict__ offsets,
                                                                 int32_t* __restrict__ sorted_token,
                                                                 int32_t* __restrict__ inv_perm) {
  extern __shared__ int32_t run[];            // [E]
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += blockDim.x) run[e] = 0;
  __syncthreads();
  const bool valid = tid < n;
  const int e = valid ? __ldg(ids + tid) : 0;
  if (valid) atomicAdd(&run[e], 1);
  __syncthreads();
  // exclusive scan of the counts (E <= 1024 = blockDim)
  const int32_t c = tid < E ? run[tid] : 0;
  int32_t x = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int32_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t w = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xFFFFFFFFu, w, off);
      if (lane >= off) w += y;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  const int32_t excl = x - c + (warp > 0 ? warp_tot[warp - 1] : 0);
  if (tid < E) {
    counts[tid] = c;
    offsets[tid] = excl;
    run[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + c;
  }
  __syncthreads();
  const int pos = block_stable_position(e, valid, run);
  if (valid) {
    sorted_token[pos] = tid / k;
    inv_perm[tid] = pos;
  }
}

// x_perm[p] = x[sorted_token[p]]: one thread per 16-byte vector (H % 8 == 0).
__global__ void __launch_bounds__(256) perm_gather_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ sorted_token, long long nvec,
                                                          int vec_per_row, uint16_t* __restrict__ x_perm) {
  for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += (long long)gridDim.x * blockDim.x) {
    const long long p = v / vec_per_row;
    const int c = (int)(v - p * vec_per_row);
    const int t = __ldg(sorted_token + p);
    reinterpret_cast<uint4*>(x_perm)[v] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * vec_per_row * 8) + c);
  }
}

size_t perm_scratch_bytes(int T, int E, int k) {
  const size_t n = (size_t)T * k;
  const size_t nchunks = (n + kPermChunk - 1) / kPermChunk;
  return (nchunks > 0 ? nchunks : 1) * (size_t)E * sizeof(int32_t);
}

cudaError_t launch_permute(const int32_t* ids, const uint16_t* x, int T, int H, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* sorted_token, int32_t* inv_perm, uint16_t* x_perm,
                           int32_t* scratch, cudaStream_t s) {
  const int n = T * k;
  const int nchunks = (n + kPermChunk - 1) / kPermChunk;
  cudaError_t err;
  if (nchunks <= 1) {
    perm_single_kernel<<<1, kPermChunk, E * sizeof(int32_t), s>>>(ids, n, E, k, counts, offsets, sorted_token,
                                                                   inv_perm);
    err = cudaGetLastError();
  } else {
    perm_hist_kernel<<<nchunks, 256, E * sizeof(int32_t), s>>>(ids, n, E, scratch);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    perm_scan_kernel<<<1, 1024, 0, s>>>(scratch, nchunks, E, counts, offsets);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    perm_scatter_kernel<<<nchunks, kPermChunk, E * sizeof(int32_t), s>>>(ids, n, E, k, scratch, sorted_token,
                                                                         inv_perm);
    err = cudaGetLastError();
  }
  if (err != cudaSuccess || n == 0) return err;
  const int vpr = H / 8;
  const long long nvec = (long long)n * vpr;
  long long blocks = (nvec + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  perm_gather_kernel<<<(unsigned)blocks, 256, 0, s>>>(x, sorted_token, nvec, vpr, x_perm);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ combine
// out[t, c] = bf16_rne(sum_j w[t,j] * y[inv[t*k+j], c]) with the fp32 sum in
// ascending j.  One thread per 4 consecutive columns.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y, const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w, int T, int H, int k,
                                                      uint16_t* __restrict__ out) {
  const int t = blockIdx.y;
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
  if (c4 * 4 >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int p = __ldg(inv + (size_t)t * k + j);
    const float wj = __ldg(w + (size_t)t * k + j);
    const float4 v = __ldg(reinterpret_cast<const float4*>(y + (size_t)p * H) + c4);
    acc.x = fmaf(wj, v.x, acc.x);
    acc.y = fmaf(wj, v.y, acc.y);
    acc.z = fmaf(wj, v.z, acc.z);
    acc.w = fmaf(wj, v.w, acc.w);
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(out + (size_t)t * H)[c4] = pk;
}

cudaError_t launch_combine(const float* y, const int32_t* inv, const float* w, int T, int H, int k, uint16_t* out,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  dim3 grid((H / 4 + 255) / 256, T);
  combine_kernel<<<grid, 256, 0, s>>>(y, inv, w, T, H, k, out);
  return cudaGetLastError();
}

}  // namespace moe
