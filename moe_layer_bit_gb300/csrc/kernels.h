// kernels.h -- host-side launchers of the library's kernels (internal).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

namespace moe {

// Launches `kern` with programmatic stream serialization: it may start its
// on-chip set-up while the previous kernel in `s` finishes (the kernels call
// pdl_wait() before touching global memory, and pdl_trigger() once the next
// kernel may start its own set-up).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Packed NVFP4 layout: tiles of 128 weight rows x 64 K elements, 4608 bytes each.
constexpr int kTileM = 128;
constexpr int kBlockK = 64;
constexpr int kWBlockBytes = 4608;

// Gate logits [T][E] = x [T][H] * Wr^T (Wr bf16 [E][H]) (+ bias [E]) in the
// library's fixed fp32 order (router.cu).
cudaError_t launch_router_logits(const uint16_t* x, const uint16_t* wr, const float* bias, int T, int H, int E,
                                 float* logits, cudaStream_t s);

cudaError_t launch_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t s);

size_t perm_scratch_bytes(int T, int E, int k);
cudaError_t launch_permute(const int32_t* ids, const uint16_t* x, int T, int H, int E, int k, int32_t* counts,
                           int32_t* offsets, int32_t* sorted_token, int32_t* inv_perm, uint16_t* x_perm,
                           int32_t* scratch, cudaStream_t s);

// Routing and grouping of the layer: top-k routing (ids / w [T][k]), then
// counts, offsets, sorted_token and inv_perm of the grouped view: with
// `shared`, every token has a (k+1)-th slot for the shared expert, grouped as
// expert E (so E+1 groups, T*(k+1) rows).  zero_e (one int32 per group,
// then kSchedInts more; may be null) is zeroed.  T*(k+shared) <= 1024 with T*E <= 32768 runs as one
// single-block launch; otherwise routing, then one grouping block or
// histogram + scan + scatter.
// With copy_bytes > 0 (a multiple of 16, both pointers 16-byte aligned) the
// launch also copies copy_bytes from copy_src (e.g. mapped page-locked host
// memory) to copy_dst, in extra blocks of the single-block launch, so the copy
// overlaps the routing; only when route_group_copies() says that launch is
// taken (cudaErrorInvalidValue otherwise).
cudaError_t launch_route_group(const float* logits, int T, int E, int k, bool shared, int32_t* ids, float* w,
                               int32_t* counts, int32_t* offsets, int32_t* sorted_token, int32_t* inv_perm,
                               int32_t* scratch, int32_t* zero_e, cudaStream_t s, const void* copy_src = nullptr,
                               void* copy_dst = nullptr, size_t copy_bytes = 0);
// True when launch_route_group routes and groups in its single-block launch,
// which can carry a copy.
bool route_group_copies(int T, int E, int k, bool shared);
// x_perm[p] = x[sorted_token[p]] for p < n.
cudaError_t launch_gather(const uint16_t* x, const int32_t* sorted_token, int n, int H, uint16_t* x_perm,
                          cudaStream_t s);

// out = sum over the k routed slots of w * y (+ the shared expert's row).
cudaError_t launch_combine(const float* y, const int32_t* inv, const float* w, int T, int H, int k, bool shared,
                           uint16_t* out, cudaStream_t s);

cudaError_t launch_prepack(const uint8_t* codes, const uint8_t* scales, int E, int N, int K, int proj,
                           uint8_t* packed, cudaStream_t s);

cudaError_t launch_dequant_table(uint16_t* out, cudaStream_t s);

// Tile schedules of the grouped GEMM (how a CTA learns its tiles):
//  static: a persistent CTA per SM takes tiles blockIdx.x, + gridDim.x, ...
//  claim:  a persistent CTA per SM takes the next tile of a global counter
//          (list order: all gate_up tiles are handed out before any down tile,
//          so the one-launch layer never waits on a CTA that has not started);
//  grid3d: one CTA per (weight tile, token tile, expert), the token-tile
//          count bounded by ceil(rows per expert bound / BN) -- the article's
//          3-D grid; CTAs without a tile exit.  One projection per launch.
constexpr int kSchedStatic = 0;
constexpr int kSchedClaim = 1;
constexpr int kSchedGrid3D = 2;
// Schedule counters after the per-group readiness counters in the layer's
// workspace (zeroed by the grouping kernel): [0] the one-launch layer's or
// the gate_up launch's claim counter, [1] the down launch's.
constexpr int kSchedInts = 4;

// Grouped W4A16 GEMM.  mode 0: gate_up + SwiGLU -> bf16 h [rows][I];
// mode 1: down -> fp32 y [rows][H].  `act` is the bf16 activation matrix
// [rows = T*k][K]; N = rows of the weight per expert (2I or H).
struct GemmArgs {
  const uint16_t* act;
  // nullptr: activation row p is act row p (a permuted copy); otherwise it is
  // act row gather_rows[p] (narrow token tiles only, see GemmPlan::gathers)
  const int32_t* gather_rows;
  const uint8_t* packed;
  const float* gscale;
  // with a shared expert: its one-expert packed matrix and global scale; it is
  // the last of the E experts the offsets describe (E - 1 routed ones)
  const uint8_t* shared_packed;
  const float* shared_gscale;
  const int32_t* offsets;
  void* out;
  int* status;
  int32_t* claim;  // the claim schedule's counter (zero before the launch), else unused
  int rows;        // T*k (T*(k+1) with a shared expert)
  int E, N, K;
  int out_ld;      // I (mode 0) or H (mode 1)
  int T, k;
};

// How the layer's projections run for given sizes: the token-tile width, the
// tile schedule, whether the GEMM gathers activation rows itself (narrow
// tiles) and whether both projections run as one launch.
struct GemmPlan {
  int bn;
  int sched;
  bool gathers;
  bool fused;
};
// force_bn (16/32/64/128) and force_sched (kSched*) override the choice when
// >= 0 (a measurement hook); -1 keeps the library's choice.  fused needs
// narrow tiles and a persistent schedule.
GemmPlan plan_layer(int rows, int E, int H, int I, int force_bn = -1, int force_sched = -1);

// One projection with the library's choice of tile width and the static
// schedule (the stage entry points).
cudaError_t launch_gemm(int mode, const GemmArgs& a, cudaStream_t s);
// One projection with the given plan's tile width and schedule.
cudaError_t launch_gemm_planned(int mode, const GemmArgs& a, const GemmPlan& plan, cudaStream_t s);

// Both projections of the layer in one persistent launch (narrow token tiles
// only): gate_up + SwiGLU tiles first, then down tiles, whose activation
// loads wait per expert until that expert's h rows are written.  `ready`:
// E int32 zeroed before the launch (and the claim counter, plan.sched ==
// kSchedClaim, in gate_up.claim).
cudaError_t launch_gemm_layer(const GemmArgs& gate_up, const GemmArgs& down, int32_t* ready, const GemmPlan& plan,
                              cudaStream_t s);

// Kernel-side view of one projection (a phase) of a launch.
struct GemmPhase {
  const uint8_t* packed;
  const float* gscale;
  const uint8_t* shared_packed;
  const float* shared_gscale;
  int E_routed;  // experts >= E_routed take the shared weights
  void* out;
  const uint16_t* act;
  const int32_t* gather_rows;
  int N, K, out_ld, mode;
};
struct GemmLaunch {
  GemmPhase ph[2];
  int nph;
  const int32_t* offsets;
  int32_t* ready;  // per expert: epilogue warps done with phase-0 tiles (nph == 2)
  int32_t* claim;  // kSchedClaim: the global tile counter
  int* status;
  int E;
  int sched;
};

// Kernel launches made by launch_route_group for these sizes.
int route_group_launches(int T, int E, int k, bool shared);

// Streaming-read probe (probe.cu): reads floor(bytes / 18432) stages of 18432
// bytes from src with one CTA per SM and a ring of bulk copies, nothing else.
// status: the status word (the int after it is a sink that is never written).
cudaError_t launch_stream_probe(const void* src, size_t bytes, int* status, cudaStream_t s);

// Bounded-wait self test: a kernel waits on a barrier nobody arrives at and
// must give up after `limit_ns`, recording a timeout in `status`.
cudaError_t launch_timeout_probe(int* status, unsigned long long limit_ns, cudaStream_t s);
// The same for the cross-CTA counter wait: `ctr` is a zero int nothing increments.
cudaError_t launch_counter_timeout_probe(int* status, const int* ctr, unsigned long long limit_ns, cudaStream_t s);

}  // namespace moe
