// permute_noalloc.cu -- moe_permute for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc at all: code running inside a memory
// pool or arena that owns every device allocation, code that must not
// allocate after start-up (latency-critical serving loops, or a process
// whose allocator is frozen), and plug-ins whose host framework hands them only
// input and output buffers.  For them, moe_permute_noalloc keeps the one
// piece of scratch moe_permute needs (the per-chunk expert histograms) in a
// fixed-size array that is part of the loaded library image, so the caller
// passes inputs and outputs only.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "kernels.h"
#include "moe_w4a16.h"

namespace {

// Capacity of the built-in scratch, in int32 entries: the permutation needs
// ceil(T*k / 1024) * E of them (nothing at all when T*k <= 1024).  256 KiB of
// device memory, held by every GPU that loads the library until the process
// exits.
constexpr size_t kNoAllocScratchInts = 65536;
__device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

// Device address of g_permute_scratch, resolved once per device and
// context.  In host code the symbol itself is only a host-side stand-in,
// never a device address.  The address belongs to the module loaded into
// the context that was current when it was looked up: after cudaDeviceReset
// (or any other way the device's primary context is destroyed and created
// again) the module is loaded anew, possibly elsewhere, so each record also
// holds the context's process-unique ID and is looked up again when the
// current context's ID differs.
using PFN_ctxGetCurrent = CUresult (*)(CUcontext*);
using PFN_ctxGetId = CUresult (*)(CUcontext, unsigned long long*);

struct ScratchRecord {
  unsigned long long ctx_id;
  int32_t* addr;
};
constexpr int kMaxDevices = 64;
ScratchRecord g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// The current context's process-unique ID (CUDA driver cuCtxGetId), or 0 if it
// cannot be had.
unsigned long long current_context_id() {
  static PFN_ctxGetCurrent get_current = nullptr;
  static PFN_ctxGetId get_id = nullptr;
  static bool resolved = false;
  if (!resolved) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_ctxGetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_ctxGetId>(p);
    (void)cudaGetLastError();
    resolved = true;
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

int scratch_address(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchRecord& rec = g_scratch_addr[dev];
  // 0 while no context is current yet on this thread (nothing has touched
  // the device): then the lookup below creates the primary context
  const unsigned long long ctx = current_context_id();
  if (rec.addr == nullptr || ctx == 0 || rec.ctx_id != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    rec.addr = static_cast<int32_t*>(p);
    rec.ctx_id = current_context_id();
  }
  *out = rec.addr;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int moe_permute_noalloc(const int32_t* topk_ids, const uint16_t* x, moe_dims d, int32_t* counts,
                                   int32_t* offsets, int32_t* sorted_token, int32_t* inv_perm, uint16_t* x_perm,
                                   void* stream) {
  // the same argument rules as moe_permute
  if (d.T < 0 || d.H <= 0 || d.I <= 0 || d.E < 1 || d.k < 1 || d.k > d.E || d.k > 32 || d.E > 1024)
    return MOE_ERR_INVALID_ARG;
  if (d.H % 128 != 0 || d.I % 64 != 0 || d.H > 65536 || d.I > 65536 || (long long)d.T * d.k >= (1LL << 31))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  const void* need[] = {topk_ids, x, counts, offsets, sorted_token, inv_perm, x_perm};
  const int n_need = d.T == 0 ? 2 : 7;  // T == 0: only counts and offsets are written
  const void* const* ptrs = d.T == 0 ? need + 2 : need;
  for (int i = 0; i < n_need; ++i)
    if (ptrs[i] == nullptr) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n_need; ++i)
    if (!aligned16(ptrs[i])) return MOE_ERR_MISALIGNED;
  // sizes beyond the built-in scratch are refused before anything runs
  if (moe::perm_scratch_bytes(d.T, d.E, d.k) > sizeof(g_permute_scratch)) return MOE_ERR_UNSUPPORTED_SHAPE;
  int32_t* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != MOE_OK) return rc;
  // The histogram kernel writes every scratch entry it later reads, so the
  // previous call's contents need no clearing.
  const cudaError_t e = moe::launch_permute(topk_ids, x, d.T, d.H, d.E, d.k, counts, offsets, sorted_token, inv_perm,
                                            x_perm, scratch, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
