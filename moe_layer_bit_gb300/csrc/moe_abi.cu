// moe_abi.cu -- the extern "C" entry points of libmoe_w4a16.so (declared in
// include/moe_w4a16.h): argument validation, workspace carving and launches.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "moe_w4a16.h"
#include "kernels.h"

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Workspace layout: the status word always sits at offset 0.
struct Layout {
  size_t status, perm, ids, w, counts, offsets, ready, sorted_token, inv_perm, x_perm, h, y, hx, hlogits, hout,
      stage_total, total;
};

// A shared expert adds one slot per token and one expert group (needs E < 1024).
bool shared_possible(const moe_dims& d) { return d.E < 1024; }

Layout layout_of(const moe_dims& d, bool shared) {
  Layout L{};
  const int ks = d.k + (shared ? 1 : 0), EG = d.E + (shared ? 1 : 0);
  const size_t nr = (size_t)d.T * d.k;  // routed (token, slot) pairs
  const size_t n = (size_t)d.T * ks;    // grouped rows
  size_t o = 0;
  L.status = o;
  o = align_up(o + sizeof(int));
  L.perm = o;
  o = align_up(o + moe::perm_scratch_bytes(d.T, EG, ks));
  L.stage_total = o;
  L.ids = o;
  o = align_up(o + nr * sizeof(int32_t));
  L.w = o;
  o = align_up(o + nr * sizeof(float));
  L.counts = o;
  o = align_up(o + (size_t)EG * sizeof(int32_t));
  L.offsets = o;
  o = align_up(o + (size_t)(EG + 1) * sizeof(int32_t));
  L.ready = o;  // per-group readiness counters, then the schedule counters
  o = align_up(o + (size_t)(EG + moe::kSchedInts) * sizeof(int32_t));
  L.sorted_token = o;
  o = align_up(o + n * sizeof(int32_t));
  L.inv_perm = o;
  o = align_up(o + n * sizeof(int32_t));
  L.x_perm = o;
  o = align_up(o + n * (size_t)d.H * 2);
  L.h = o;
  o = align_up(o + n * (size_t)d.I * 2);
  L.y = o;
  o = align_up(o + n * (size_t)d.H * sizeof(float));
  L.hx = o;
  o = align_up(o + (size_t)d.T * d.H * 2);
  L.hlogits = o;
  o = align_up(o + (size_t)d.T * d.E * sizeof(float));
  L.hout = o;
  o = align_up(o + (size_t)d.T * d.H * 2);
  L.total = o;
  return L;
}

// The workspace the layer entry points ask for covers the shared-expert
// layout (a superset) whenever a shared expert is possible.
Layout layout_of(const moe_dims& d) { return layout_of(d, shared_possible(d)); }

int check_dims(const moe_dims& d) {
  if (d.T < 0 || d.H <= 0 || d.I <= 0 || d.E < 1 || d.k < 1) return MOE_ERR_INVALID_ARG;
  if (d.k > d.E || d.k > 32 || d.E > 1024) return MOE_ERR_INVALID_ARG;
  if (d.H % 128 != 0 || d.I % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (d.H > 65536 || d.I > 65536) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)d.T * d.k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
  for (const void* p : ps)
    if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  (void)cudaGetLastError();
  return MOE_ERR_CUDA;
}

cudaError_t run_gemm(int mode, const moe::GemmArgs& a, cudaStream_t s) { return moe::launch_gemm(mode, a, s); }

#define MOE_TRY(expr)            \
  do {                           \
    int _rc = (expr);            \
    if (_rc != MOE_OK) return _rc; \
  } while (0)

#define MOE_TRY_NEG(expr)           \
  do {                              \
    int _rc = (expr);               \
    if (_rc != MOE_OK) return -_rc; \
  } while (0)

}  // namespace

extern "C" {

size_t moe_packed_w4_bytes(int32_t E, int32_t N, int32_t K) {
  if (E <= 0 || N <= 0 || K <= 0) return 0;
  return (size_t)E * (size_t)N * (size_t)K * 9 / 16;
}

int moe_prepack_w4(const uint8_t* codes, const uint8_t* scales, int32_t E, int32_t N, int32_t K, int32_t proj,
                   void* packed, void* stream) {
  if (E < 1 || N <= 0 || K <= 0 || (proj != MOE_PROJ_GATE_UP && proj != MOE_PROJ_DOWN)) return MOE_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (codes == nullptr || scales == nullptr || packed == nullptr) return MOE_ERR_INVALID_ARG;
  if (!aligned16(packed)) return MOE_ERR_MISALIGNED;
  return cuda_status(moe::launch_prepack(codes, scales, E, N, K, proj, static_cast<uint8_t*>(packed),
                                         as_stream(stream)));
}

size_t moe_workspace_bytes(moe_dims d) {
  if (check_dims(d) != MOE_OK) return 0;
  return layout_of(d).total;
}

int moe_layer_kernel_launches(moe_dims d) {
  MOE_TRY_NEG(check_dims(d));
  if (d.T == 0) return 0;
  const moe::GemmPlan p = moe::plan_layer(d.T * d.k, d.E, d.H, d.I);
  return moe::route_group_launches(d.T, d.E, d.k, false) + (p.gathers ? 0 : 1) + (p.fused ? 1 : 2) + 1;
}

int moe_layer_projections_fused(moe_dims d) {
  MOE_TRY_NEG(check_dims(d));
  return d.T > 0 && moe::plan_layer(d.T * d.k, d.E, d.H, d.I).fused ? 1 : 0;
}

size_t moe_stage_workspace_bytes(moe_dims d) {
  if (check_dims(d) != MOE_OK) return 0;
  return layout_of(d).stage_total;
}

int moe_router_logits(const uint16_t* x, const uint16_t* router_weight, const float* router_bias, moe_dims d,
                      float* logits, void* stream) {
  MOE_TRY(check_dims(d));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({x, router_weight, logits}));
  if (router_bias != nullptr && (reinterpret_cast<uintptr_t>(router_bias) & 3u) != 0) return MOE_ERR_MISALIGNED;
  return cuda_status(
      moe::launch_router_logits(x, router_weight, router_bias, d.T, d.H, d.E, logits, as_stream(stream)));
}

int moe_route_topk(const float* logits, moe_dims d, int32_t* topk_ids, float* topk_w, void* stream) {
  MOE_TRY(check_dims(d));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({logits, topk_ids, topk_w}));
  return cuda_status(moe::launch_route_topk(logits, d.T, d.E, d.k, topk_ids, topk_w, as_stream(stream)));
}

int moe_permute(const int32_t* topk_ids, const uint16_t* x, moe_dims d, int32_t* counts, int32_t* offsets,
                int32_t* sorted_token, int32_t* inv_perm, uint16_t* x_perm, void* ws, size_t ws_bytes,
                void* stream) {
  MOE_TRY(check_dims(d));
  if (d.T == 0) MOE_TRY(check_ptrs({counts, offsets, ws}));
  else MOE_TRY(check_ptrs({topk_ids, x, counts, offsets, sorted_token, inv_perm, x_perm, ws}));
  const Layout L = layout_of(d);
  if (ws_bytes < L.stage_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  return cuda_status(moe::launch_permute(topk_ids, x, d.T, d.H, d.E, d.k, counts, offsets, sorted_token, inv_perm,
                                         x_perm, reinterpret_cast<int32_t*>(w + L.perm), as_stream(stream)));
}

int moe_w4a16_gate_up_swiglu(const uint16_t* x_perm, const int32_t* offsets, moe_w4 w_gate_up, moe_dims d,
                             uint16_t* h, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(d));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({x_perm, offsets, w_gate_up.packed, w_gate_up.global_scale, h, ws}));
  const Layout L = layout_of(d);
  if (ws_bytes < L.stage_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe::GemmArgs a{};
  a.act = x_perm;
  a.packed = static_cast<const uint8_t*>(w_gate_up.packed);
  a.gscale = w_gate_up.global_scale;
  a.offsets = offsets;
  a.out = h;
  a.status = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + L.status);
  a.rows = d.T * d.k;
  a.E = d.E;
  a.N = 2 * d.I;
  a.K = d.H;
  a.out_ld = d.I;
  a.T = d.T;
  a.k = d.k;
  return cuda_status(run_gemm(0, a, as_stream(stream)));
}

int moe_w4a16_down(const uint16_t* h, const int32_t* offsets, moe_w4 w_down, moe_dims d, float* y_perm, void* ws,
                   size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(d));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({h, offsets, w_down.packed, w_down.global_scale, y_perm, ws}));
  const Layout L = layout_of(d);
  if (ws_bytes < L.stage_total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe::GemmArgs a{};
  a.act = h;
  a.packed = static_cast<const uint8_t*>(w_down.packed);
  a.gscale = w_down.global_scale;
  a.offsets = offsets;
  a.out = y_perm;
  a.status = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + L.status);
  a.rows = d.T * d.k;
  a.E = d.E;
  a.N = d.H;
  a.K = d.I;
  a.out_ld = d.H;
  a.T = d.T;
  a.k = d.k;
  return cuda_status(run_gemm(1, a, as_stream(stream)));
}

int moe_unpermute_combine(const float* y_perm, const int32_t* inv_perm, const float* topk_w, moe_dims d,
                          uint16_t* out, void* stream) {
  MOE_TRY(check_dims(d));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({y_perm, inv_perm, topk_w, out}));
  return cuda_status(moe::launch_combine(y_perm, inv_perm, topk_w, d.T, d.H, d.k, false, out, as_stream(stream)));
}

}  // extern "C"

namespace {

// The layer, optionally recording ev[0..5] around the five stages
// (ev[i] before stage i, ev[5] after the last).  shared_gu / shared_dn: the
// shared expert's projections (both or neither), packed as one-expert
// matrices of the routed experts' shapes.
int layer_forward_impl(const uint16_t* x, const float* logits, moe_w4 w_gate_up, moe_w4 w_down,
                       const moe_w4* shared_gu, const moe_w4* shared_dn, moe_dims d, uint16_t* out,
                       int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, void* stream, void* const* ev,
                       int force_bn = -1, int force_sched = -1, const uint16_t* x_copy_src = nullptr) {
  MOE_TRY(check_dims(d));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({x, logits, w_gate_up.packed, w_gate_up.global_scale, w_down.packed, w_down.global_scale, out,
                      ws}));
  if ((topk_ids != nullptr && !aligned16(topk_ids)) || (topk_w != nullptr && !aligned16(topk_w)))
    return MOE_ERR_MISALIGNED;
  const bool shared = shared_gu != nullptr;
  if (shared) {
    if (shared_dn == nullptr) return MOE_ERR_INVALID_ARG;
    if (!shared_possible(d) || d.k >= 32) return MOE_ERR_UNSUPPORTED_SHAPE;  // E + 1 groups, k + 1 slots
    MOE_TRY(check_ptrs({shared_gu->packed, shared_gu->global_scale, shared_dn->packed, shared_dn->global_scale}));
  }
  const Layout L = layout_of(d);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  cudaStream_t s = as_stream(stream);
  // NVTX ranges name the launches of each stage for a profiler's timeline
  // (no-ops when no tool is attached); the guard closes an open range on
  // every return.
  static const char* const kStageNames[5] = {"moe:route_group", "moe:gather", "moe:gate_up", "moe:down",
                                             "moe:combine"};
  struct NvtxStage {
    bool open = false;
    void next(int i) {
      if (open) nvtxRangePop();
      open = i < 5;
      if (open) nvtxRangePushA(kStageNames[i]);
    }
    ~NvtxStage() {
      if (open) nvtxRangePop();
    }
  } nvtx_stage;
  auto mark = [&](int i) -> int {
    nvtx_stage.next(i);
    if (ev == nullptr || ev[i] == nullptr) return MOE_OK;
    return cuda_status(cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[i]), s));
  };
  int32_t* ids = topk_ids ? topk_ids : reinterpret_cast<int32_t*>(w + L.ids);
  float* wts = topk_w ? topk_w : reinterpret_cast<float*>(w + L.w);
  int32_t* counts = reinterpret_cast<int32_t*>(w + L.counts);
  int32_t* offs = reinterpret_cast<int32_t*>(w + L.offsets);
  int32_t* sorted = reinterpret_cast<int32_t*>(w + L.sorted_token);
  int32_t* inv = reinterpret_cast<int32_t*>(w + L.inv_perm);
  uint16_t* xp = reinterpret_cast<uint16_t*>(w + L.x_perm);
  uint16_t* h = reinterpret_cast<uint16_t*>(w + L.h);
  float* y = reinterpret_cast<float*>(w + L.y);
  // grouped view: with a shared expert every token has k + 1 rows and the
  // shared expert is group E
  const int rows = d.T * (d.k + (shared ? 1 : 0));
  const int EG = d.E + (shared ? 1 : 0);
  MOE_TRY(mark(0));
  // readiness counters [EG], then the schedule counters; the grouping kernel zeroes them
  int32_t* ready = reinterpret_cast<int32_t*>(w + L.ready);
  int32_t* claim = ready + EG;
  const moe::GemmPlan plan = moe::plan_layer(rows, EG, d.H, d.I, force_bn, force_sched);
  // x_copy_src (host-buffer calls): x's bytes, copied to x by extra blocks of
  // the routing launch, which the caller has checked can carry them
  MOE_TRY(cuda_status(moe::launch_route_group(logits, d.T, d.E, d.k, shared, ids, wts, counts, offs, sorted, inv,
                                              reinterpret_cast<int32_t*>(w + L.perm), ready, s, x_copy_src,
                                              const_cast<uint16_t*>(x), x_copy_src != nullptr ? (size_t)d.T * d.H * 2
                                                                                              : 0)));
  MOE_TRY(mark(1));
  // the narrow-tile GEMM gathers the rows of x itself; the wide one reads x_perm
  if (!plan.gathers) MOE_TRY(cuda_status(moe::launch_gather(x, sorted, rows, d.H, xp, s)));
  MOE_TRY(mark(2));
  moe::GemmArgs a{};
  a.offsets = offs;
  a.status = reinterpret_cast<int*>(w + L.status);
  a.claim = claim;
  a.rows = rows;
  a.E = EG;
  a.T = d.T;
  a.k = d.k;
  a.act = plan.gathers ? x : xp;
  a.gather_rows = plan.gathers ? sorted : nullptr;
  a.packed = static_cast<const uint8_t*>(w_gate_up.packed);
  a.gscale = w_gate_up.global_scale;
  a.shared_packed = shared ? static_cast<const uint8_t*>(shared_gu->packed) : nullptr;
  a.shared_gscale = shared ? shared_gu->global_scale : nullptr;
  a.out = h;
  a.N = 2 * d.I;
  a.K = d.H;
  a.out_ld = d.I;
  moe::GemmArgs b = a;
  b.act = h;
  b.gather_rows = nullptr;
  b.claim = claim + 1;
  b.packed = static_cast<const uint8_t*>(w_down.packed);
  b.gscale = w_down.global_scale;
  b.shared_packed = shared ? static_cast<const uint8_t*>(shared_dn->packed) : nullptr;
  b.shared_gscale = shared ? shared_dn->global_scale : nullptr;
  b.out = y;
  b.N = d.H;
  b.K = d.I;
  b.out_ld = d.H;
  if (plan.fused) {
    // one launch for both projections: stage 2 spans it, stage 3 is empty
    MOE_TRY(cuda_status(moe::launch_gemm_layer(a, b, ready, plan, s)));
    MOE_TRY(mark(3));
  } else {
    MOE_TRY(cuda_status(moe::launch_gemm_planned(0, a, plan, s)));
    MOE_TRY(mark(3));
    MOE_TRY(cuda_status(moe::launch_gemm_planned(1, b, plan, s)));
  }
  MOE_TRY(mark(4));
  MOE_TRY(cuda_status(moe::launch_combine(y, inv, wts, d.T, d.H, d.k, shared, out, s)));
  return mark(5);
}

}  // namespace

extern "C" {

int moe_layer_forward(const uint16_t* x, const float* logits, moe_w4 w_gate_up, moe_w4 w_down, moe_dims d,
                      uint16_t* out, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, void* stream) {
  return layer_forward_impl(x, logits, w_gate_up, w_down, nullptr, nullptr, d, out, topk_ids, topk_w, ws, ws_bytes,
                            stream, nullptr);
}

int moe_layer_forward_profiled(const uint16_t* x, const float* logits, moe_w4 w_gate_up, moe_w4 w_down, moe_dims d,
                               uint16_t* out, int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes,
                               void* stream, void* const* stage_events) {
  return layer_forward_impl(x, logits, w_gate_up, w_down, nullptr, nullptr, d, out, topk_ids, topk_w, ws, ws_bytes,
                            stream, stage_events);
}

int moe_debug_layer_forward_config(const uint16_t* x, const float* logits, moe_w4 w_gate_up, moe_w4 w_down,
                                   moe_dims d, uint16_t* out, int32_t* topk_ids, float* topk_w, void* ws,
                                   size_t ws_bytes, int32_t token_tile, int32_t schedule, void* stream,
                                   void* const* stage_events) {
  if (token_tile != -1 && token_tile != 16 && token_tile != 32 && token_tile != 64 && token_tile != 128)
    return MOE_ERR_INVALID_ARG;
  if (schedule < -1 || schedule > moe::kSchedGrid3D) return MOE_ERR_INVALID_ARG;
  return layer_forward_impl(x, logits, w_gate_up, w_down, nullptr, nullptr, d, out, topk_ids, topk_w, ws, ws_bytes,
                            stream, stage_events, token_tile, schedule);
}

int moe_layer_forward_router(const uint16_t* x, const uint16_t* router_weight, const float* router_bias,
                             moe_w4 w_gate_up, moe_w4 w_down, moe_dims d, uint16_t* out, float* logits_out,
                             int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(d));
  if (d.T == 0) return MOE_OK;
  MOE_TRY(check_ptrs({x, router_weight, ws}));
  if (router_bias != nullptr && (reinterpret_cast<uintptr_t>(router_bias) & 3u) != 0) return MOE_ERR_MISALIGNED;
  if (logits_out != nullptr && !aligned16(logits_out)) return MOE_ERR_MISALIGNED;
  const Layout L = layout_of(d);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  float* logits = logits_out != nullptr ? logits_out : reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + L.hlogits);
  MOE_TRY(cuda_status(
      moe::launch_router_logits(x, router_weight, router_bias, d.T, d.H, d.E, logits, as_stream(stream))));
  return layer_forward_impl(x, logits, w_gate_up, w_down, nullptr, nullptr, d, out, topk_ids, topk_w, ws, ws_bytes,
                            stream, nullptr);
}

int moe_layer_forward_shared(const uint16_t* x, const float* logits, const uint16_t* router_weight,
                             const float* router_bias, moe_w4 w_gate_up, moe_w4 w_down, moe_w4 shared_gate_up,
                             moe_w4 shared_down, moe_dims d, uint16_t* out, float* logits_out, int32_t* topk_ids,
                             float* topk_w, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(d));
  if (d.T == 0) return MOE_OK;
  if ((logits == nullptr) == (router_weight == nullptr)) return MOE_ERR_INVALID_ARG;  // exactly one source
  MOE_TRY(check_ptrs({x, ws}));
  const Layout L = layout_of(d);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (router_weight != nullptr) {
    if (!aligned16(router_weight)) return MOE_ERR_MISALIGNED;
    if (router_bias != nullptr && (reinterpret_cast<uintptr_t>(router_bias) & 3u) != 0) return MOE_ERR_MISALIGNED;
    if (logits_out != nullptr && !aligned16(logits_out)) return MOE_ERR_MISALIGNED;
    float* lg = logits_out != nullptr ? logits_out
                                      : reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + L.hlogits);
    MOE_TRY(cuda_status(
        moe::launch_router_logits(x, router_weight, router_bias, d.T, d.H, d.E, lg, as_stream(stream))));
    logits = lg;
  }
  return layer_forward_impl(x, logits, w_gate_up, w_down, &shared_gate_up, &shared_down, d, out, topk_ids, topk_w, ws,
                            ws_bytes, stream, nullptr);
}

}  // extern "C"

namespace {

// The device address of page-locked host memory that kernels can access
// directly (mapped), else nullptr.
void* mapped_device_ptr(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

bool page_locked(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

// The copies and kernels of one host-buffer call, enqueued on `s`.
// x is copied into the workspace (the GEMM reads its rows many times).  When
// the host logits and output are mapped page-locked memory, the routing
// kernel reads the logits and the combine writes the output through their
// device addresses, so those two transfers need no copy of their own;
// otherwise they are copied too.
int enqueue_host_call(const uint16_t* host_x, const float* host_logits, moe_w4 w_gate_up, moe_w4 w_down, moe_dims d,
                      uint16_t* host_out, void* ws, size_t ws_bytes, cudaStream_t s) {
  const Layout L = layout_of(d);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const size_t xb = (size_t)d.T * d.H * 2, lb = (size_t)d.T * d.E * sizeof(float);
  uint16_t* dx = reinterpret_cast<uint16_t*>(w + L.hx);
  const float* ml = static_cast<const float*>(mapped_device_ptr(host_logits));
  uint16_t* mo = static_cast<uint16_t*>(mapped_device_ptr(host_out));
  const uint16_t* mx = static_cast<const uint16_t*>(mapped_device_ptr(host_x));
  if (ml != nullptr && mo != nullptr && aligned16(ml) && aligned16(mo)) {
    // x mapped too, and routing in one launch: extra blocks of that launch
    // copy x, so the call needs no copy of its own (it would otherwise run
    // before the routing, on the copy engine)
    if (mx != nullptr && aligned16(mx) && moe::route_group_copies(d.T, d.E, d.k, false))
      return layer_forward_impl(dx, ml, w_gate_up, w_down, nullptr, nullptr, d, mo, nullptr, nullptr, ws, ws_bytes, s,
                                nullptr, -1, -1, mx);
    MOE_TRY(cuda_status(cudaMemcpyAsync(dx, host_x, xb, cudaMemcpyHostToDevice, s)));
    return moe_layer_forward(dx, ml, w_gate_up, w_down, d, mo, nullptr, nullptr, ws, ws_bytes, s);
  }
  MOE_TRY(cuda_status(cudaMemcpyAsync(dx, host_x, xb, cudaMemcpyHostToDevice, s)));
  float* dl = reinterpret_cast<float*>(w + L.hlogits);
  uint16_t* dout = reinterpret_cast<uint16_t*>(w + L.hout);
  MOE_TRY(cuda_status(cudaMemcpyAsync(dl, host_logits, lb, cudaMemcpyHostToDevice, s)));
  MOE_TRY(moe_layer_forward(dx, dl, w_gate_up, w_down, d, dout, nullptr, nullptr, ws, ws_bytes, s));
  return cuda_status(cudaMemcpyAsync(host_out, dout, xb, cudaMemcpyDeviceToHost, s));
}

}  // namespace

// A host plan: one host-buffer call recorded once as a CUDA graph (its
// copies and kernels, bound to the plan's host buffers, workspace and
// stream) and replayed by every run.  The caller owns it: the graph lives
// until moe_host_plan_destroy, and the library keeps no reference to it.
struct moe_host_plan {
  cudaGraphExec_t exec;
  cudaStream_t stream;
  int dev;
};

extern "C" {

int moe_layer_forward_host(const uint16_t* host_x, const float* host_logits, moe_w4 w_gate_up, moe_w4 w_down,
                           moe_dims d, uint16_t* host_out, void* ws, size_t ws_bytes, void* stream) {
  MOE_TRY(check_dims(d));
  if (d.T == 0) return MOE_OK;
  if (host_x == nullptr || host_logits == nullptr || host_out == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ptrs({w_gate_up.packed, w_gate_up.global_scale, w_down.packed, w_down.global_scale, ws}));
  const Layout L = layout_of(d);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = as_stream(stream);
  MOE_TRY(enqueue_host_call(host_x, host_logits, w_gate_up, w_down, d, host_out, ws, ws_bytes, s));
  return cuda_status(cudaStreamSynchronize(s));
}

int moe_host_plan_create(const uint16_t* host_x, const float* host_logits, moe_w4 w_gate_up, moe_w4 w_down,
                         moe_dims d, uint16_t* host_out, void* ws, size_t ws_bytes, void* stream,
                         moe_host_plan** plan) {
  if (plan == nullptr) return MOE_ERR_INVALID_ARG;
  *plan = nullptr;
  MOE_TRY(check_dims(d));
  if (host_x == nullptr || host_logits == nullptr || host_out == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ptrs({w_gate_up.packed, w_gate_up.global_scale, w_down.packed, w_down.global_scale, ws}));
  const Layout L = layout_of(d);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = as_stream(stream);
  if (s == nullptr) return MOE_ERR_INVALID_ARG;  // the legacy default stream cannot be captured
  if (!page_locked(host_x) || !page_locked(host_logits) || !page_locked(host_out)) return MOE_ERR_INVALID_ARG;
  int dev = 0;
  MOE_TRY(cuda_status(cudaGetDevice(&dev)));
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  MOE_TRY(cuda_status(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal)));
  const int rc = d.T == 0 ? MOE_OK
                          : enqueue_host_call(host_x, host_logits, w_gate_up, w_down, d, host_out, ws, ws_bytes, s);
  const cudaError_t ec = cudaStreamEndCapture(s, &graph);
  if (rc != MOE_OK || ec != cudaSuccess || graph == nullptr) {
    if (graph != nullptr) cudaGraphDestroy(graph);
    (void)cudaGetLastError();
    return rc != MOE_OK ? rc : MOE_ERR_CUDA;
  }
  const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess) return cuda_status(ei);
  moe_host_plan* p = static_cast<moe_host_plan*>(std::malloc(sizeof(moe_host_plan)));
  if (p == nullptr) {
    cudaGraphExecDestroy(exec);
    return MOE_ERR_CUDA;
  }
  p->exec = exec;
  p->stream = s;
  p->dev = dev;
  *plan = p;
  return MOE_OK;
}

int moe_host_plan_run(moe_host_plan* plan) {
  if (plan == nullptr) return MOE_ERR_INVALID_ARG;
  int dev = 0;
  MOE_TRY(cuda_status(cudaGetDevice(&dev)));
  if (dev != plan->dev) return MOE_ERR_INVALID_ARG;
  MOE_TRY(cuda_status(cudaGraphLaunch(plan->exec, plan->stream)));
  return cuda_status(cudaStreamSynchronize(plan->stream));
}

int moe_host_plan_destroy(moe_host_plan* plan) {
  if (plan == nullptr) return MOE_OK;
  const cudaError_t e = cudaGraphExecDestroy(plan->exec);
  std::free(plan);
  return cuda_status(e);
}

int moe_get_device_status(void* ws, void* stream) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return cuda_status(cudaErrorUnknown);
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return cuda_status(cudaErrorUnknown);
  if (v != 0) {
    if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return cuda_status(cudaErrorUnknown);
  }
  return v == 0 ? MOE_OK : (v == MOE_ERR_DEVICE_TIMEOUT ? MOE_ERR_DEVICE_TIMEOUT : MOE_ERR_CUDA);
}

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_debug_dequant_table(uint16_t* out, void* stream) {
  MOE_TRY(check_ptrs({out}));
  return cuda_status(moe::launch_dequant_table(out, as_stream(stream)));
}

int moe_debug_timeout_probe(void* ws, uint64_t limit_ns, void* stream) {
  MOE_TRY(check_ptrs({ws}));
  return cuda_status(moe::launch_timeout_probe(static_cast<int*>(ws), (unsigned long long)limit_ns,
                                               as_stream(stream)));
}

int moe_debug_stream_read(const void* src, size_t bytes, void* ws, void* stream) {
  MOE_TRY(check_ptrs({src, ws}));
  return cuda_status(moe::launch_stream_probe(src, bytes, static_cast<int*>(ws), as_stream(stream)));
}

int moe_debug_counter_timeout_probe(void* ws, uint64_t limit_ns, void* stream) {
  MOE_TRY(check_ptrs({ws}));
  int* base = static_cast<int*>(ws);
  cudaStream_t s = as_stream(stream);
  // the counter: the int at byte 128 of ws, zeroed here
  MOE_TRY(cuda_status(cudaMemsetAsync(base + 32, 0, sizeof(int), s)));
  return cuda_status(moe::launch_counter_timeout_probe(base, base + 32, (unsigned long long)limit_ns, s));
}

}  // extern "C"
