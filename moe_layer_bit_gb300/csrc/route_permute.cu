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
// One warp routes one token.  Lane l holds experts l, l+32, ..., NV per lane
// (NV * 32 >= E).  k rounds of a warp arg-max with (key desc, index asc)
// order, key = logit with NaN mapped to -inf.  Gate weights: softmax over the
// k selected keys, fp32 with expf, summed in slot order.  Lane j < k returns
// slot j's expert and weight.
template <int NV>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k, int& out_id, float& out_w) {
  const int lane = threadIdx.x & 31;
  float key[NV];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    float v = -INFINITY;
    if (e < E) {
      v = __ldg(row + e);
      if (isnan(v)) v = -INFINITY;
    } else {
      taken |= 1u << i;  // not a real expert
    }
    key[i] = v;
  }
  float sel_key = -INFINITY;  // lane j keeps the key of slot j
  int sel_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const bool ok = !((taken >> i) & 1u);
      if (ok && (bi == 0x7FFFFFFF || key[i] > bv)) {  // ascending e: strict > keeps the lower index
        bv = key[i];
        bi = lane + 32 * i;
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
  MOE_DISPATCH_NV(route_nv(E), (route_topk_kernel<NV><<<blocks, kRouteWarps * 32, 0, s>>>(logits, T, E, k, ids, w)));
  return cudaGetLastError();
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

// Shared memory of the rank table: uint16 [warps][E].
static size_t rank_table_bytes(int warps, int E) { return (size_t)warps * E * sizeof(uint16_t); }

// Every thread of the block calls this with its pair (valid == false for
// padding).  `base[e]` is the first sorted row of expert e available to this
// block.  `tab` is zeroed by the caller (and a __syncthreads follows).
__device__ __forceinline__ int block_stable_position(int e, bool valid, const int32_t* base, uint16_t* tab, int E) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int key = valid ? e : -1 - lane;  // padding pairs: unique keys
  const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key);
  const int rank = __popc(peers & ((1u << lane) - 1u));
  if (valid && lane == __ffs(peers) - 1) tab[warp * E + e] = (uint16_t)__popc(peers);
  __syncthreads();
  for (int ex = threadIdx.x; ex < E; ex += blockDim.x) {  // exclusive prefix over warps, per expert
    uint16_t run = 0;
    for (int w = 0; w < nwarps; ++w) {
      const uint16_t c = tab[w * E + ex];
      tab[w * E + ex] = run;
      run = (uint16_t)(run + c);
    }
  }
  __syncthreads();
  return valid ? base[e] + tab[warp * E + e] + rank : 0;
}

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
  int32_t total;
  const int32_t excl = block_exclusive_scan(run, warp_tot, &total);
  if (e < E) {
    offsets[e] = excl;
    for (int b = 0; b < nchunks; ++b) chunk_counts[(size_t)b * E + e] += excl;
    if (e == E - 1) offsets[E] = excl + run;
  }
}

// Shared memory of the scatter kernels: base[E] int32, then the rank table.
static size_t scatter_smem_bytes(int warps, int E) { return (size_t)E * sizeof(int32_t) + rank_table_bytes(warps, E); }

// One block of kPermChunk threads per chunk; thread i owns pair base + i.
__global__ void __launch_bounds__(kPermChunk) perm_scatter_kernel(const int32_t* __restrict__ ids, int n, int E, int k,
                                                                  const int32_t* __restrict__ chunk_base,
                                                                  int32_t* __restrict__ sorted_token,
                                                                  int32_t* __restrict__ inv_perm) {
  extern __shared__ int32_t smem_i[];
  int32_t* base = smem_i;
  uint16_t* tab = reinterpret_cast<uint16_t*>(smem_i + E);
  const int g = blockIdx.x * kPermChunk + threadIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) base[e] = chunk_base[(size_t)blockIdx.x * E + e];
  for (int x = threadIdx.x; x < (int)(blockDim.x >> 5) * E; x += blockDim.x) tab[x] = 0;
  const bool valid = g < n;
  const int e = valid ? __ldg(ids + g) : 0;
  __syncthreads();
  const int pos = block_stable_position(e, valid, base, tab, E);
  if (valid) {
    sorted_token[pos] = g / k;
    inv_perm[g] = pos;
  }
}

// All pairs in one block (T*k <= kPermChunk), routing optionally included:
// with logits != nullptr the block first routes its T tokens (one warp per
// token, warps striding), writing ids / weights; then histogram, scan and
// stable scatter, all in one launch.
template <int NV>
__global__ void __launch_bounds__(kPermChunk) route_permute_small_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ ids, float* __restrict__ wts,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_token,
    int32_t* __restrict__ inv_perm) {
  extern __shared__ int32_t smem_i[];
  int32_t* base = smem_i;                                  // [E] counts, then offsets
  int32_t* s_ids = smem_i + E;                             // [kPermChunk]
  uint16_t* tab = reinterpret_cast<uint16_t*>(smem_i + E + kPermChunk);
  __shared__ int32_t warp_tot[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int n = T * k;
  for (int e = tid; e < E; e += blockDim.x) base[e] = 0;
  for (int x = tid; x < nwarps * E; x += blockDim.x) tab[x] = 0;
  if (logits != nullptr) {
    for (int t = warp; t < T; t += nwarps) {
      int id;
      float w;
      route_token<NV>(logits + (size_t)t * E, E, k, id, w);
      if (lane < k) {
        s_ids[t * k + lane] = id;
        ids[(size_t)t * k + lane] = id;
        wts[(size_t)t * k + lane] = w;
      }
    }
  } else {
    for (int i = tid; i < n; i += blockDim.x) s_ids[i] = __ldg(ids + i);
  }
  __syncthreads();
  const bool valid = tid < n;
  const int e = valid ? s_ids[tid] : 0;
  if (valid) atomicAdd(&base[e], 1);
  __syncthreads();
  const int32_t c = tid < E ? base[tid] : 0;
  int32_t total;
  const int32_t excl = block_exclusive_scan(c, warp_tot, &total);
  if (tid < E) {
    counts[tid] = c;
    offsets[tid] = excl;
    base[tid] = excl;
    if (tid == E - 1) offsets[E] = excl + c;
  }
  __syncthreads();
  const int pos = block_stable_position(e, valid, base, tab, E);
  if (valid) {
    sorted_token[pos] = tid / k;
    inv_perm[tid] = pos;
  }
}

static size_t small_smem_bytes(int E) {
  return (size_t)(E + kPermChunk) * sizeof(int32_t) + rank_table_bytes(kPermChunk / 32, E);
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

cudaError_t launch_gather(const uint16_t* x, const int32_t* sorted_token, int n, int H, uint16_t* x_perm,
                                 cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int vpr = H / 8;
  const long long nvec = (long long)n * vpr;
  long long blocks = (nvec + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  perm_gather_kernel<<<(unsigned)blocks, 256, 0, s>>>(x, sorted_token, nvec, vpr, x_perm);
  return cudaGetLastError();
}

template <int NV>
static cudaError_t launch_small(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* counts,
                                int32_t* offsets, int32_t* sorted_token, int32_t* inv_perm, cudaStream_t s) {
  const size_t smem = small_smem_bytes(E);
  auto kern = route_permute_small_kernel<NV>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  kern<<<1, kPermChunk, smem, s>>>(logits, T, E, k, ids, w, counts, offsets, sorted_token, inv_perm);
  return cudaGetLastError();
}

static cudaError_t launch_chunked(const int32_t* ids, int n, int E, int k, int32_t* counts, int32_t* offsets,
                                  int32_t* sorted_token, int32_t* inv_perm, int32_t* scratch, cudaStream_t s) {
  const int nchunks = (n + kPermChunk - 1) / kPermChunk;
  perm_hist_kernel<<<nchunks, 256, E * sizeof(int32_t), s>>>(ids, n, E, scratch);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  perm_scan_kernel<<<1, 1024, 0, s>>>(scratch, nchunks, E, counts, offsets);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t smem = scatter_smem_bytes(kPermChunk / 32, E);
  err = cudaFuncSetAttribute(perm_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  perm_scatter_kernel<<<nchunks, kPermChunk, smem, s>>>(ids, n, E, k, scratch, sorted_token, inv_perm);
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* ids, const uint16_t* x, int T, int H, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* sorted_token, int32_t* inv_perm, uint16_t* x_perm,
                           int32_t* scratch, cudaStream_t s) {
  const int n = T * k;
  cudaError_t err = (n <= kPermChunk)
                        ? launch_small<1>(nullptr, T, E, k, const_cast<int32_t*>(ids), nullptr, counts, offsets,
                                          sorted_token, inv_perm, s)
                        : launch_chunked(ids, n, E, k, counts, offsets, sorted_token, inv_perm, scratch, s);
  if (err != cudaSuccess) return err;
  return launch_gather(x, sorted_token, n, H, x_perm, s);
}

cudaError_t launch_route_group(const float* logits, int T, int E, int k, int32_t* ids, float* w, int32_t* counts,
                               int32_t* offsets, int32_t* sorted_token, int32_t* inv_perm, int32_t* scratch,
                               cudaStream_t s) {
  const int n = T * k;
  if (n <= kPermChunk) {
    cudaError_t err;
    MOE_DISPATCH_NV(route_nv(E), err = (launch_small<NV>(logits, T, E, k, ids, w, counts, offsets, sorted_token,
                                                         inv_perm, s)));
    return err;
  }
  const cudaError_t err = launch_route_topk(logits, T, E, k, ids, w, s);
  if (err != cudaSuccess) return err;
  return launch_chunked(ids, n, E, k, counts, offsets, sorted_token, inv_perm, scratch, s);
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
