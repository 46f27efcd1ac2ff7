/*
 * moe_w4a16.h -- C ABI of libmoe_w4a16.so: a W4A16 NVFP4 mixture-of-experts
 * FFN layer for NVIDIA GB300 (sm_103a).
 *
 * The layer (top-k routing -> permutation grouped by expert -> grouped
 * gate_up GEMM with SwiGLU -> grouped down GEMM -> weighted combine) is the
 * MoE layer described by:
 *   [Atlas]  "告别Python堆栈：Atlas用纯Rust重写LLM推理，在GB10上跑赢vLLM"
 *            (f.mffb.com.cn/a/497905.html), section "编译时内核选择和W4A16 Grouped
 *            GEMM": per-expert gate_up and down projections run by ONE grouped
 *            launch over all experts; packed FP4 weights are dequantised to
 *            BF16 on chip and fed to a BF16 MMA, with no BF16 weight written
 *            back to memory.  Section "KV Cache量化、MTP推测解码和调试工具链":
 *            gate logits -> expert IDs -> routed output.
 *   [ATOM]   "AMD ATOM推理引擎：如何用分页KV缓存和分段编译实现大模型推理性能翻倍"
 *            (itsolotime.com/archives/33112), section "8.1 MoE 路径": routing,
 *            top-k selection, expert compute, combine; section "8.2 量化并非单一
 *            格式，而是一套执行契约": a quantisation format fixes dtype, scale
 *            shape and whether weights are pre-shuffled for the kernel.
 *   [Rust DL] "Rust 实现深度学习推理引擎：从计算图到异构硬件加速"
 *            (ybb.press/ai-applications/14151.html), section "三、计算图":
 *            SiLU / SwiGLU activation.
 *
 * Conventions for every entry point
 *  - Shapes: T tokens, H hidden, I expert intermediate, E experts, k top-k.
 *    Row-major everywhere.  Supported: T >= 0, H % 128 == 0, I % 64 == 0,
 *    1 <= k <= min(E, 32), 1 <= E <= 1024, T*k < 2^31, H, I <= 65536.
 *  - bf16 arrays are passed as uint16_t bit patterns.
 *  - All pointers are DEVICE pointers unless the name says host_; the caller
 *    owns every buffer.  Device arrays must be 16-byte aligned.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and does not synchronise, except where stated.
 *  - Arguments are validated before anything is launched; on error nothing
 *    is launched and no output is touched.
 *  - Return value: a moe_status.  A launch failure returns MOE_ERR_CUDA and
 *    clears the CUDA error state (cudaGetLastError).
 *  - A kernel whose internal wait (a pipeline barrier) runs past about one
 *    second gives up, records MOE_ERR_DEVICE_TIMEOUT in the workspace's status
 *    word and returns; moe_get_device_status() reads it.
 *  - The library allocates no device memory: every intermediate lives in the
 *    caller's workspace `ws`.  The one allocation of any entry point is the
 *    caller-owned host plan (moe_host_plan_create / _destroy).  Global
 *    mutable state: the fixed scratch array of moe_permute_noalloc with its
 *    per-device address record, and the once-resolved address of the
 *    driver's tensor-map encoder; nothing else.
 */
#ifndef MOE_W4A16_H
#define MOE_W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,        /* null pointer, k > E, k > 32, E > 1024, negative size */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* H % 128, I % 64, or a size beyond the limits above */
    MOE_ERR_MISALIGNED = 3,         /* a device pointer not 16-byte aligned */
    MOE_ERR_WORKSPACE_TOO_SMALL = 4,
    MOE_ERR_CUDA = 5,               /* a CUDA runtime / driver call failed */
    MOE_ERR_DEVICE_TIMEOUT = 6      /* a kernel's bounded wait expired (reported by moe_get_device_status) */
} moe_status;

typedef struct {
    int32_t T, H, I, E, k;
} moe_dims;

/* Which projection a packed weight buffer holds. */
typedef enum {
    MOE_PROJ_GATE_UP = 0,  /* N = 2I rows (rows 0..I-1 gate, I..2I-1 up), K = H */
    MOE_PROJ_DOWN = 1      /* N = H rows, K = I */
} moe_projection;

/* ------------------------------------------------------------------------
 * NVFP4 weights.
 * Interchange ("natural") layout of one projection with N rows and K columns
 * per expert:
 *   codes   uint8 [E][N][K/2]  E2M1 codes, element 2i in the low nibble,
 *                              2i+1 in the high nibble;
 *   scales  uint8 [E][N][K/16] one E4M3 block scale per 16 consecutive K;
 *   global  float [E]          one fp32 global scale per expert matrix;
 *   weight[e][n][kk] = e2m1(code) * e4m3(scale) * global[e].
 * The GEMM entry points read the "packed" layout made once by
 * moe_prepack_w4 (the pre-shuffle of [ATOM] section 8.2): same bytes,
 * reordered into 128-row x 64-column tiles so that each pipeline stage is one
 * contiguous copy.  The packed buffer has exactly E*N*K*9/16 bytes.
 * ------------------------------------------------------------------------ */
typedef struct {
    const void *packed;          /* from moe_prepack_w4, device */
    const float *global_scale;   /* [E], device */
} moe_w4;

/* Bytes of a packed buffer for E experts of an N x K projection. */
size_t moe_packed_w4_bytes(int32_t E, int32_t N, int32_t K);

/* One-time re-layout of natural NVFP4 weights (device codes/scales) into the
 * packed layout (device `packed`, moe_packed_w4_bytes bytes, must not overlap
 * the inputs).  `proj` selects the row order: gate_up rows are interleaved
 * gate/up in groups of 16 so that one 128-row tile holds 64 gate rows and
 * the 64 matching up rows.  N, K as for `proj` (gate_up: N = 2I, K = H;
 * down: N = H, K = I); N % 128 == 0, K % 64 == 0.  Pure byte permutation. */
int moe_prepack_w4(const uint8_t *codes, const uint8_t *scales, int32_t E, int32_t N, int32_t K,
                   int32_t proj, void *packed, void *stream);

/* ------------------------------------------------------------------------
 * Workspace.  moe_workspace_bytes(d) is the size that moe_layer_forward and
 * moe_layer_forward_host need; the stage entry points need at least
 * moe_stage_workspace_bytes(d).  Device memory, 256-byte aligned, owned by
 * the caller.  The first 4 bytes are the device status word: zero-fill the
 * workspace (or at least those bytes) once before its first use; kernels only
 * ever write a timeout code there, and moe_get_device_status clears it after
 * reading.  Nothing else in the workspace needs initialisation.
 * T == 0 is valid everywhere: nothing is launched except that moe_permute
 * writes zero counts and offsets; token-sized arrays may then be NULL.
 * ------------------------------------------------------------------------ */
size_t moe_workspace_bytes(moe_dims d);

/* Number of kernels one moe_layer_forward call with these dims launches on
 * its stream (0 for T == 0); minus a moe_status code if d is invalid.  Host
 * only: touches no device. */
int moe_layer_kernel_launches(moe_dims d);

/* 1 if moe_layer_forward runs gate_up + SwiGLU and down as ONE kernel launch
 * for these dims (narrow token tiles: decode-sized batches), 0 if as two;
 * minus a moe_status code if d is invalid.  Host only. */
int moe_layer_projections_fused(moe_dims d);
size_t moe_stage_workspace_bytes(moe_dims d);

/* Gate logits of the layer (Atlas: gate input -> gate logits -> expert IDs,
 * section «KV Cache量化、MTP推测解码和调试工具链»):
 *   logits[t][e] = sum_h x[t][h] * router_weight[e][h]  (+ router_bias[e])
 * x bf16 [T][H], router_weight bf16 [E][H], router_bias f32 [E] or NULL,
 * logits f32 [T][E] out.  Computed in one fixed fp32 order, independent of
 * the launch shape, so routing on the result is reproducible bit for bit: the
 * hidden dimension is cut into 8-element chunks, part l (0..31) sums x*w over
 * chunks l, l+32, ... in ascending h with fused multiply-adds from 0, the 32
 * parts are combined pairwise (part l + part l^s for s = 16, 8, 4, 2, 1) and
 * the bias is added last.  x, router_weight, logits 16-byte aligned. */
int moe_router_logits(const uint16_t *x, const uint16_t *router_weight, const float *router_bias,
                      moe_dims d, float *logits, void *stream);

/* [Atlas] "KV Cache量化…" (gate logits -> expert IDs), [ATOM] 8.1 (top-k).
 * logits  float [T][E]   router logits (NaN is treated as -infinity)
 * topk_ids int32 [T][k]  out: selected experts, slot order = descending logit,
 *                        ties to the lower expert index
 * topk_w  float [T][k]   out: softmax over the k selected logits (equal to
 *                        softmax over E renormalised over the k); 1/k each if
 *                        the best logit is -infinity. */
int moe_route_topk(const float *logits, moe_dims d, int32_t *topk_ids, float *topk_w, void *stream);

/* Permutation grouped by expert ([Atlas] per-expert M tiles; [ATOM] 8.1).
 * topk_ids int32 [T][k]; x bf16 [T][H].
 * counts   int32 [E]    out: pairs (t, j) routed to each expert
 * offsets  int32 [E+1]  out: exclusive scan of counts, offsets[E] = T*k
 * sorted_token int32 [T*k] out: token of sorted row p; rows sorted by (expert, token)
 * inv_perm int32 [T*k]  out: sorted row of pair (t, j) at index t*k+j
 * x_perm   bf16 [T*k][H] out: x_perm[p] = x[sorted_token[p]]
 * Deterministic and bit-exact.  Needs moe_stage_workspace_bytes(d) of ws. */
int moe_permute(const int32_t *topk_ids, const uint16_t *x, moe_dims d, int32_t *counts,
                int32_t *offsets, int32_t *sorted_token, int32_t *inv_perm, uint16_t *x_perm,
                void *ws, size_t ws_bytes, void *stream);

/* moe_permute for callers that cannot allocate device memory: code whose
 * device memory all belongs to a pool or arena it may not grow, serving loops
 * that must not allocate after start-up, and plug-ins that are handed only
 * their input and output buffers.  The pages have no counterpart of this
 * entry point; it exists only for such callers.
 * Same arguments, results and rules as moe_permute, minus the workspace: the
 * per-chunk histogram scratch lives in a fixed array inside the library
 * (65536 int32 = 256 KiB of device memory, held by every GPU that loads the
 * library until the process exits).  The call allocates nothing.
 * Limit: ceil(T*k / 1024) * E <= 65536 (e.g. T*k <= 65536 with E <= 1024);
 * larger sizes return MOE_ERR_UNSUPPORTED_SHAPE before anything runs.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, and so does the first
 * call after the device's context was created anew (cudaDeviceReset); make
 * those calls before any stream capture.  Every call uses the same array, so calls whose
 * work overlaps on the GPU (other streams, other host threads) race; the
 * array needs no clearing between calls. */
int moe_permute_noalloc(const int32_t *topk_ids, const uint16_t *x, moe_dims d, int32_t *counts,
                        int32_t *offsets, int32_t *sorted_token, int32_t *inv_perm, uint16_t *x_perm,
                        void *stream);

/* Grouped gate_up GEMM + SwiGLU, one launch over all experts ([Atlas] W4A16
 * Grouped GEMM; [Rust DL] SwiGLU).  For expert e and rows p in
 * [offsets[e], offsets[e+1]):
 *   g = x_perm[p] . Wgate_e^T,  u = x_perm[p] . Wup_e^T  (fp32 accumulation of
 *   bf16 x bf16 products; weights dequantised exactly to bf16 on chip),
 *   h[p] = bf16_rne(silu(g) * u),  silu(z) = z / (1 + exp(-z)).
 * x_perm bf16 [T*k][H]; offsets int32 [E+1] (from moe_permute);
 * w_gate_up packed gate_up weights; h bf16 [T*k][I] out. */
int moe_w4a16_gate_up_swiglu(const uint16_t *x_perm, const int32_t *offsets, moe_w4 w_gate_up,
                             moe_dims d, uint16_t *h, void *ws, size_t ws_bytes, void *stream);

/* Grouped down GEMM ([Atlas]: the same grouped W4A16 launch for "down").
 *   y_perm[p] = h[p] . Wdown_e^T   (fp32 accumulation, fp32 result)
 * h bf16 [T*k][I]; y_perm float [T*k][H] out. */
int moe_w4a16_down(const uint16_t *h, const int32_t *offsets, moe_w4 w_down, moe_dims d,
                   float *y_perm, void *ws, size_t ws_bytes, void *stream);

/* Weighted combine back to token order ([ATOM] 8.1 "combine"):
 *   out[t] = bf16_rne( sum_{j=0..k-1} topk_w[t][j] * y_perm[inv_perm[t*k+j]] ),
 * fp32 sum in ascending j.  Every element of out is written. */
int moe_unpermute_combine(const float *y_perm, const int32_t *inv_perm, const float *topk_w,
                          moe_dims d, uint16_t *out, void *stream);

/* The whole layer: route -> permute -> gate_up+SwiGLU -> down -> combine,
 * stream-ordered, no host synchronisation.  topk_ids / topk_w may be NULL
 * (then they live in ws).  Needs moe_workspace_bytes(d) of ws.
 * When moe_layer_projections_fused(d), both projections run as one launch
 * of one CTA per SM whose CTAs wait on one another; it relies on all of them
 * becoming resident, which holds when nothing else keeps SMs busy for long.
 * Such launches of calls on several streams that start at the same moment
 * can split the SMs between them; their waits then give up after about a
 * second and report MOE_ERR_DEVICE_TIMEOUT (nothing hangs).  Issue
 * concurrent layer calls on one stream. */
int moe_layer_forward(const uint16_t *x, const float *logits, moe_w4 w_gate_up, moe_w4 w_down,
                      moe_dims d, uint16_t *out, int32_t *topk_ids, float *topk_w, void *ws,
                      size_t ws_bytes, void *stream);

/* moe_layer_forward with per-stage timing: stage_events points to 6
 * cudaEvent_t handles (created by the caller; any entry may be NULL).
 * stage_events[i] is recorded on `stream` just before stage i (0 routing and
 * grouping: top-k ids and weights, counts, offsets, sorted_token, inv_perm;
 * 1 the row gather into x_perm, empty when the GEMM gathers rows itself;
 * 2 gate_up+SwiGLU, 3 down, 4 combine; when moe_layer_projections_fused(d),
 * stage 2 spans the one launch of both projections and stage 3 is empty) and
 * stage_events[5] after
 * the last, so cudaEventElapsedTime(ev[2], ev[3]) is the gate_up launch.
 * Same results and launches as moe_layer_forward. */
int moe_layer_forward_profiled(const uint16_t *x, const float *logits, moe_w4 w_gate_up, moe_w4 w_down,
                               moe_dims d, uint16_t *out, int32_t *topk_ids, float *topk_w, void *ws,
                               size_t ws_bytes, void *stream, void *const *stage_events);

/* moe_layer_forward with the gate logits computed in the layer from the
 * router weights (moe_router_logits) instead of passed in.  logits_out:
 * f32 [T][E] that receives them, or NULL (then they live in ws).  Same
 * workspace as moe_layer_forward. */
int moe_layer_forward_router(const uint16_t *x, const uint16_t *router_weight, const float *router_bias,
                             moe_w4 w_gate_up, moe_w4 w_down, moe_dims d, uint16_t *out, float *logits_out,
                             int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes, void *stream);

/* The layer with a shared expert.  The Atlas article's MoE layer produces a
 * routed output and a shared-expert output (section «KV Cache量化、MTP推测解码
 * 和调试工具链», which dumps both per layer); here
 *   out[t] = bf16( sum_j topk_w[t][j] * y_{ids[t][j]}(x[t])  +  y_shared(x[t]) )
 * with the routed sum in ascending j (fp32), then the shared term added with
 * weight 1.  y_shared is a SwiGLU FFN like a routed expert's, with
 * shared_gate_up / shared_down: one-expert NVFP4 matrices (moe_prepack_w4
 * with E = 1) of the routed experts' H and I.  It runs in the same grouped
 * launches as the routed experts, as an extra expert that every token uses.
 * Gate logits: `logits` (f32 [T][E]), or, with logits == NULL,
 * computed from router_weight (bf16 [E][H]) and router_bias (f32 [E] or
 * NULL) as moe_router_logits does, into logits_out (f32 [T][E], or ws when
 * NULL).  Exactly one of logits / router_weight is non-NULL.  Needs E < 1024
 * and k < 32 (else MOE_ERR_UNSUPPORTED_SHAPE).  Same workspace as
 * moe_layer_forward. */
int moe_layer_forward_shared(const uint16_t *x, const float *logits, const uint16_t *router_weight,
                             const float *router_bias, moe_w4 w_gate_up, moe_w4 w_down, moe_w4 shared_gate_up,
                             moe_w4 shared_down, moe_dims d, uint16_t *out, float *logits_out, int32_t *topk_ids,
                             float *topk_w, void *ws, size_t ws_bytes, void *stream);

/* The whole layer from HOST buffers: copies host_x (bf16 [T][H]) into ws,
 * runs moe_layer_forward on it and host_logits (float [T][E]), puts the
 * result in host_out (bf16 [T][H]) and synchronises `stream` before returning.
 * When host_logits and host_out are page-locked memory the device can address
 * (mapped, 16-byte aligned), the routing kernel reads the logits and the
 * combine writes the output through their device addresses; otherwise they
 * are copied through ws as well.  If host_x is mapped page-locked memory too
 * (16-byte aligned) and the routing runs as one single-block launch
 * (T*k <= 1024 and T*E <= 32768), extra blocks of that launch copy host_x into
 * ws while it routes; otherwise host_x is copied before the routing.  Host
 * buffers should be page-locked for full
 * transfer speed.  Weights stay on the device.  Needs moe_workspace_bytes(d)
 * of ws.  Every call issues its copies and launches afresh and keeps nothing
 * after it returns. */
int moe_layer_forward_host(const uint16_t *host_x, const float *host_logits, moe_w4 w_gate_up,
                           moe_w4 w_down, moe_dims d, uint16_t *host_out, void *ws, size_t ws_bytes,
                           void *stream);

/* A host plan: moe_layer_forward_host with fixed arguments, recorded once as
 * a CUDA graph (its copies and kernels) and replayed by moe_host_plan_run, so
 * that a serving loop calling the layer on the same buffers pays one graph
 * launch per call instead of the individual copies and launches.
 *   moe_host_plan_create: same arguments as moe_layer_forward_host, plus the
 *     plan out-pointer.  host_x, host_logits and host_out must be page-locked
 *     (cudaHostAlloc / cudaHostRegister); `stream` must be a created stream
 *     (not NULL), current device = the device of ws.  Records nothing on the
 *     GPU: the stream is captured, not run.  The plan holds the graph's
 *     driver resources and a small host record -- the only memory any entry
 *     point of this library allocates -- until moe_host_plan_destroy.
 *   moe_host_plan_run: reads the host buffers' CURRENT contents, runs the
 *     layer and writes host_out; synchronises the plan's stream before
 *     returning.  Call it with the plan's device current.
 *   moe_host_plan_destroy: frees the plan (NULL is a no-op).
 * The plan keeps the raw addresses it was created with: destroy it before
 * freeing, unregistering or reusing any of its buffers, its workspace or its
 * weights, and before destroying its stream; then create a new one.  The
 * library keeps no reference to a plan, so plans of different threads or
 * streams are independent; runs of one plan must not overlap. */
typedef struct moe_host_plan moe_host_plan;
int moe_host_plan_create(const uint16_t *host_x, const float *host_logits, moe_w4 w_gate_up,
                         moe_w4 w_down, moe_dims d, uint16_t *host_out, void *ws, size_t ws_bytes,
                         void *stream, moe_host_plan **plan);
int moe_host_plan_run(moe_host_plan *plan);
int moe_host_plan_destroy(moe_host_plan *plan);

/* ------------------------------------------------------------------------
 * W4A4: the block-scaled FP4 variant of the layer.  GB300 multiplies NVFP4
 * by NVFP4 natively (tcgen05.mma kind::mxf4nvf4), which the Atlas article's
 * GB10 lacks (section «编译时内核选择和W4A16 Grouped GEMM»: it falls back to
 * W4A16 there); the ATOM article (section «8.2 量化并非单一格式，而是一套执行契约»)
 * treats a 4-bit-activation format as its own execution contract.  Here the
 * activations entering each projection (x before gate_up, h before down) are
 * quantized to NVFP4 -- per 16 consecutive elements an E4M3 scale
 * s = RNE_e4m3(min(amax16 / 6, 448)) (amax16 / 6 in fp32) and the E2M1
 * codes of the exact quotient v / e4m3(s) rounded to nearest, ties to the
 * even mantissa, saturating at +-6, no global scale; h is quantized from its
 * fp32 value -- and both projections run as E2M1 x E2M1 products with both
 * sides' block scales applied by the MMA, fp32 accumulation, the weights'
 * global scale in the epilogue.  Different numerics from the W4A16 layer
 * (the activations lose precision): results are checked against the W4A4
 * definition, not the W4A16 one.
 * Weights in the natural NVFP4 layout (no prepack): */
typedef struct {
    const uint8_t *codes;        /* [E][N][K/2], device, 16-byte aligned */
    const uint8_t *scales;       /* [E][N][K/16] E4M3, device, 16-byte aligned */
    const float *global_scale;   /* [E], device */
} moe_w4n;

/* Workspace of moe_layer_forward_w4a4 (0 if d is invalid).  Supported: the
 * W4A16 limits and additionally H % 256 == 0, I % 256 == 0. */
size_t moe_w4a4_workspace_bytes(moe_dims d);

/* Host-only: the number of kernels one moe_layer_forward_w4a4 call launches
 * (the routing + grouping launches, then quantize-and-gather, gate_up, down
 * and combine); 0 for T == 0, minus the moe_status for invalid dims. */
int moe_w4a4_kernel_launches(moe_dims d);

/* The W4A4 layer: route -> group -> quantize and gather x -> gate_up +
 * SwiGLU (h quantized in the epilogue) -> down -> combine, as
 * moe_layer_forward with the activation quantization above.  out bf16 [T][H];
 * topk_ids / topk_w as for moe_layer_forward (may be NULL).  Needs
 * moe_w4a4_workspace_bytes(d) of ws (its first 4 bytes the status word). */
int moe_layer_forward_w4a4(const uint16_t *x, const float *logits, moe_w4n w_gate_up, moe_w4n w_down,
                           moe_dims d, uint16_t *out, int32_t *topk_ids, float *topk_w, void *ws,
                           size_t ws_bytes, void *stream);

/* moe_layer_forward_w4a4 with per-stage timing: stage_events points to 6
 * cudaEvent_t handles (any may be NULL), recorded on `stream` before routing
 * + grouping (0), the quantize-and-gather of x (1), gate_up + SwiGLU (2),
 * down (3), the combine (4), and after it (5).  Same results and launches. */
int moe_layer_forward_w4a4_profiled(const uint16_t *x, const float *logits, moe_w4n w_gate_up, moe_w4n w_down,
                                    moe_dims d, uint16_t *out, int32_t *topk_ids, float *topk_w, void *ws,
                                    size_t ws_bytes, void *stream, void *const *stage_events);

/* The activation quantizer alone: row r of the output is the NVFP4 form of
 * row rows_of[r] of x (bf16 [*][K]; row r when rows_of is NULL), r < n:
 * codes uint8 [n][K/2] (element 2i in the low nibble), scales E4M3 [n][K/16].
 * K % 16 == 0; x, codes, scales 16-byte aligned. */
int moe_quantize_nvfp4(const uint16_t *x, const int32_t *rows_of, int32_t n, int32_t K, uint8_t *codes,
                       uint8_t *scales, void *stream);

/* moe_quantize_nvfp4 for fp32 rows x [*][K] (the precision h has when the
 * layer quantizes it): the same quantizer, arguments and errors. */
int moe_quantize_nvfp4_f32(const float *x, const int32_t *rows_of, int32_t n, int32_t K, uint8_t *codes,
                           uint8_t *scales, void *stream);

/* Test hook: one W4A4 projection over grouped, already quantized activation
 * rows.  mode 0: gate_up + SwiGLU, act [T*k][H/2] codes + [T*k][H/16] scales,
 * w the gate_up weights (N = 2I, K = H), out = h codes [T*k][I/2] and
 * out_scales = h scales [T*k][I/16]; mode 1: down, act = h's NVFP4 form, w
 * the down weights (N = H, K = I), out = y float [T*k][H].  offsets [E+1] as
 * from moe_permute; ws: a status word.  Same limits as moe_layer_forward_w4a4. */
int moe_debug_w4a4_gemm(int32_t mode, const uint8_t *act_codes, const uint8_t *act_scales,
                        const int32_t *offsets, moe_w4n w, moe_dims d, void *out, uint8_t *out_scales,
                        void *ws, void *stream);

/* Synchronises `stream`, then reads and clears the device status word in ws
 * (any workspace passed to the calls above).  Returns MOE_OK,
 * MOE_ERR_DEVICE_TIMEOUT, or MOE_ERR_CUDA. */
int moe_get_device_status(void *ws, void *stream);

/* Human-readable name of a moe_status. */
const char *moe_status_string(int status);

/* Test hook: runs the GEMM kernels' on-chip NVFP4 -> bf16 dequantisation on
 * every (E4M3 scale, E2M1 code) pair and writes out[s*16 + c] =
 * bf16(e2m1(c) * e4m3(s)) (exact: at most 6 significant bits).
 * out: device uint16 [256*16]. */
int moe_debug_dequant_table(uint16_t *out, void *stream);

/* Test hook for failure detection: launches a kernel whose pipeline wait can
 * never complete (an mbarrier nobody arrives at) with a wait limit of
 * `limit_ns` nanoseconds.  The wait gives up, records MOE_ERR_DEVICE_TIMEOUT in
 * the status word at the start of `ws` and the kernel returns; read it with
 * moe_get_device_status.  Nothing faults and the context stays usable. */
int moe_debug_timeout_probe(void *ws, uint64_t limit_ns, void *stream);

/* Test hook for failure detection of the cross-CTA wait: when
 * moe_layer_projections_fused(d), a down tile waits on a per-expert counter
 * that the gate_up tiles of other CTAs increment.  This launches a kernel
 * that waits, with limit `limit_ns`, on a counter nothing increments (the int
 * at byte 128 of `ws`, zeroed first; ws must hold >= 132 bytes).  The wait
 * gives up and records MOE_ERR_DEVICE_TIMEOUT in the status word; nothing
 * faults and the context stays usable. */
int moe_debug_counter_timeout_probe(void *ws, uint64_t limit_ns, void *stream);

/* Measurement hook for choosing the GEMM's tile schedule and token-tile
 * width by measurement: moe_layer_forward_profiled with those two choices
 * forced.  token_tile: 16, 32, 64 or 128 rows per token tile (-1: the
 * library's choice); schedule: 0 static (a persistent CTA per SM takes
 * tiles blockIdx.x, + gridDim.x, ...), 1 claim (a persistent CTA per SM
 * takes the next tile of a global counter), 2 grid3d (one CTA per (weight
 * tile, token tile, expert), the Atlas article's 3-D grid
 * (ceil(N/BN), max token tiles, experts); one launch per projection), -1:
 * the library's choice.  16- and 32-row tiles gather activation rows in the
 * GEMM and, unless grid3d, run both projections as one launch; 64- and
 * 128-row tiles read a permuted copy of x.  Same results as
 * moe_layer_forward within the layer tolerance (the fp32 sums are the same
 * for every choice: a token tile's MMA K order does not depend on them).
 * Same workspace. */
int moe_debug_layer_forward_config(const uint16_t *x, const float *logits, moe_w4 w_gate_up, moe_w4 w_down,
                                   moe_dims d, uint16_t *out, int32_t *topk_ids, float *topk_w, void *ws,
                                   size_t ws_bytes, int32_t token_tile, int32_t schedule, void *stream,
                                   void *const *stage_events);

/* Measurement hook: a streaming-read probe.  Reads floor(bytes / 18432) *
 * 18432 bytes of device memory at src (16-byte aligned) with one CTA per SM,
 * each issuing 18432-byte bulk copies into a ring of 8 shared-memory slots and
 * doing nothing else -- the weight stream of the narrow-tile GEMM without its
 * work -- so that a caller can time how fast one kernel of that shape reads
 * that many bytes.  ws: the status word (and the int after it) of a workspace;
 * a stalled copy records MOE_ERR_DEVICE_TIMEOUT there. */
int moe_debug_stream_read(const void *src, size_t bytes, void *ws, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_W4A16_H */
