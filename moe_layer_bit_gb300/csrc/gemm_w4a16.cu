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
//    expert offsets (no host sync, no empty CTAs): one producer warp decides
//    the CTA's tiles (a fixed stride, or the next value of a global counter)
//    and publishes each through a shared-memory ring that every other role
//    follows; the article's 3-D grid is kept as a measured alternative;
//  * a pipeline stage is SB consecutive 64-column K blocks (a "superstage"),
//    so the per-stage barrier round trips of the single MMA-issuing warp are
//    paid once per SB*4 MMAs;
//  * warp roles (24 warps):
//    - one producer warp decides and publishes the tiles and issues one 1-D
//      bulk copy of the SB packed weight blocks (codes + E4M3 scales,
//      SB * 4608 B) per stage into a weight ring that is freed as soon as the
//      codes are in registers;
//    - activation tiles, 128-byte swizzled, go into a second ring freed by
//      the MMA commit: for wide token tiles one warp issues SB 2-D TMA copies
//      of a permuted copy of the rows; for narrow ones (16 or 32 rows:
//      decode) one warp copies row sorted_token[p] of x itself with 16-byte
//      cp.async, so no permuted copy is written;
//    - 16 dequant warps in groups (stages round-robin over groups) turn the
//      codes into exact bf16 (value * 2^-7) and store them straight into
//      tensor memory as the MMA's A operand (tcgen05.st), so no dequantised
//      weight touches shared memory;
//    - one MMA warp (operands warp-uniform, one elected lane issuing) runs
//      tcgen05.mma with A from TMEM, B from shared memory and an fp32
//      accumulator in TMEM, a ring of 2 (wide tiles) or 4 (narrow) across
//      tiles;
//    - four epilogue warps read the accumulator (tcgen05.ld), apply
//      global_scale * 2^7 and write SwiGLU(bf16) or fp32 rows;
//    - in the one-launch layer, one readiness warp (below);
//  * one launch can run both projections of the layer (narrow token tiles):
//    the schedule is the gate_up tiles, then the down tiles, the weight
//    stream runs on without a break, and a down tile's activation loads wait
//    (per expert, on a GPU-scope counter the gate_up epilogues publish with
//    release semantics, watched by the readiness warp) until that expert's
//    h rows are written.  CTAs take tiles from a global counter in list
//    order, so every gate_up tile belongs to a running CTA before any down
//    tile is handed out, and the waits end whatever the SM residency (other
//    streams, other processes, a partitioned GPU);
//  * every barrier wait is bounded (about 1 s); on expiry the CTA records a
//    timeout in the status word, drains its copies and MMAs and exits.
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "gemm_common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kWarpEpi0 = 0;       // warps 0..3: epilogue (TMEM lane quadrant = warp)
constexpr int kWarpDq0 = 4;        // warps 4..19: dequant (groups of 4 * kSplit warps)
constexpr int kDqWarps = 16;
constexpr int kWarpProducer = 20;  // warp 20: weight copies
constexpr int kWarpMma = 21;       // warp 21: TMEM owner + MMA issue
constexpr int kWarpProducerB = 22; // warps 22 ..: activation rows (gathered; warp 22 alone for TMA tiles)
constexpr int kBProducers = 1;     // gathering warps
constexpr int kWarpReady = kWarpProducerB + kBProducers;  // readiness of down tiles (one-launch layer)
constexpr int kThreads = (kWarpReady + 1) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kMinSmem = 120 * 1024;  // keeps one CTA (one TMEM allocation) per SM
constexpr int kSmemBudget = 216 * 1024;  // rings; the tile table (<= 8 KiB) and alignment slack on top
constexpr int kBInFlight = 2;  // activation stages a gathering producer lane keeps in flight
// 64-row (TMA) token tiles with at most 32 valid rows load and multiply only
// their first 32 rows (a 32-row box, MMA N = 32).
template <int BN>
constexpr bool kHalfTiles = BN == 64;

// Token-tile width BN and SB K blocks per stage: shared-memory rings of NSW
// weight stages (SB packed blocks) and NSB activation stages (SB sub-tiles),
// and a TMEM ring of NA A-operand slots of 32*SB columns (128 rows x 64*SB
// bf16) placed after the ND accumulators of BN columns.
template <int BN, int SB>
struct Cfg {
  static constexpr int kBSub = BN * 128;  // BN rows x 64 bf16, 128-byte swizzled
  static constexpr int kBTile = SB * kBSub;
  static constexpr int kWBytes = SB * kWBlockBytes;
  // ND fp32 accumulators of BN columns (tiles round-robin), so the MMA warp
  // runs ND - 1 tiles ahead of the epilogue: 4 for narrow tiles, whose tiles
  // are short (a down tile of a decode step is 3 stages), where TMEM has room.
  static constexpr int ND = BN <= 32 ? 4 : 2;
  static constexpr int A0 = (ND * BN < 32) ? 32 : ND * BN;
  static constexpr int kSlotCols = 32 * SB;
  static constexpr int NA = (int)(kTmemCols - A0) / kSlotCols;
  // A stage's SB blocks are split over kSplit warps per TMEM lane quadrant,
  // so a dequant group has 4 * kSplit warps; groups take stages round-robin.
  // 16-row tiles (SB = 4): two groups of 8 warps, 2 blocks per warp.  With
  // fewer groups than TMEM slots, a group's next stage waits on the MMA of
  // the other group's stage, not on its own (measured faster on decode than
  // three groups of 4 warps on three slots).  32-row tiles (SB = 4) measured
  // the other way round: three groups of 4 warps beat two of 8 (grouped
  // layer 175 vs 163 us of GEMM).  64/128-row tiles (SB = 4, two TMEM slots
  // next to the two accumulators): two groups of 8 warps (prefill layer
  // 2,414 -> 2,102 us against SB = 2 with four groups of 4).
  static constexpr int kSplit = ((BN == 16 || BN >= 64) && SB == 4) ? 2 : 1;
  static constexpr int kGroupWarps = 4 * kSplit;
  static constexpr int kGroups0 = kDqWarps / kGroupWarps;
  static constexpr int G = kGroups0 < NA ? kGroups0 : NA;
  // Two shared-memory rings: NSB activation tiles (freed by the MMA commit)
  // and NSW weight blocks (freed as soon as the dequant warps hold the codes in
  // registers, so weight prefetch depth does not wait on the MMA).
  // Narrow token tiles (BN <= 32: decode-sized batches) gather their
  // activation rows with cp.async (row sorted_token[p] of x, or row p); an
  // activation stage is then released kBInFlight stages after it was issued,
  // so that ring is deeper: 6 stages of 8 KiB (16-row tiles) or 16 KiB
  // (32-row tiles), which leaves room for 8 weight stages (16-row tiles: a
  // 10-stage activation ring with 6 weight stages measured 1.1% slower on
  // decode).  Wider tiles read permuted rows with TMA: at SB = 4 (K 256 per
  // stage) 3 stages of 32 KiB for 64-row tiles, next to 6 weight stages (the
  // weight-streaming grouped shape: gate_up 97 -> 84 us against 2 activation
  // and 8 weight stages; 4 + 4 measured 86 us), and 2 of 64 KiB for 128-row
  // tiles; 4 at smaller SB.  An activation stage is refilled only after its
  // MMAs complete, so with 2 stages the refill had only the next stage's MMAs
  // to hide behind.  (Activation slots of one K block each, refilled block by
  // block, and MMAs trimmed to a partial tile's valid rows both measured
  // slower on every wide-tile workload.)
  static constexpr bool kGatherB = BN <= 32;
  static constexpr int NSB = kGatherB ? 4 + kBInFlight : (SB == 4 ? (BN == 64 ? 3 : 2) : 4);
  static_assert(!kGatherB || NSB > kBInFlight, "the gathering producer must not wait on a stage it has not released");
  static constexpr int NSW0 = (kSmemBudget - NSB * kBTile) / kWBytes;
  static constexpr int NSW1 = NSW0 > 12 ? 12 : NSW0;
  // Parity waits are exact only while the awaited barrier cannot be two
  // phases behind the waiter.  A dequant group waits for (a) TMEM slot i % NA
  // to be free (MMA of stage i - NA done) and (b) weight slot i % NSW to hold
  // stage i.
  // (a) Its own previous stage i - G waited for the MMA of stage i - G - NA,
  //     which covers stage i - 2 NA only when G <= NA.
  // (b) Stage i - NSW (the slot's previous phase) must have landed; copies do
  //     not complete in issue order, so G | NSW makes it the group's own,
  //     already waited on.
  // The activation ring is waited on in stage order: by the MMA warp, or for
  // gathered stages by the stage's dequant group, whose previous stage's wait
  // (with the producer's in-order releases and NSB >= G) covers stage
  // i - NSB, and whose own arrival the release of stage i + NSB waits behind.
  static constexpr int NSW = NSW1 < G ? G : (NSW1 / G) * G;
  // TMA stages with as many activation stages as TMEM A slots (64- and
  // 128-row tiles at SB = 4): stage i takes activation stage i % NSB and A
  // slot i % NA, both free once the stage's MMAs complete, so the A slot's
  // barrier frees both and the MMA warp commits once per stage (prefill
  // gate_up -1.5%, grouped -2%).
  static constexpr bool kOneFreeBar = !kGatherB && NSB == NA;
  static_assert(G <= NA && NSW % G == 0 && (!kGatherB || NSB >= G), "dequant groups must fit the rings");
  // The tile ring: the weight producer publishes each tile of the CTA's
  // schedule (phase, expert, weight tile, token tile) into entry j % kRing;
  // the MMA warp, the epilogue warps and the activation producers read it,
  // and in the one-launch layer the readiness warp too.
  static constexpr int kRing = 32;
  static constexpr int kRingReaders = 1 + 4 + (kGatherB ? kBProducers : 1);
  static constexpr int kOffB = 0;
  static constexpr int kOffW = NSB * kBTile;
  static constexpr int kOffBar = kOffW + NSW * kWBytes;
  // fullw[NSW], emptyw[NSW], fullb[NSB], emptyb[NSB], afull[NA], aempty[NA],
  // dfull[ND], dempty[ND], drain, tfull[kRing], tempty[kRing], rdy[kRing]
  static constexpr int kNumBars = 2 * NSW + 2 * NSB + 2 * NA + 2 * ND + 1 + 3 * kRing;
  static constexpr int kOffRing = ((kOffBar + kNumBars * 8 + 15) / 16) * 16;  // int4 [kRing]
  static constexpr int kOffWFlag = kOffRing + kRing * 16;           // int [NSW]: 1 = weight stage, 0 = end
  static constexpr int kOffMisc = kOffWFlag + ((NSW * 4 + 15) / 16) * 16;  // [0] tmem base, [1] abort, [2] tiles
  static constexpr int kOffTables = kOffMisc + 16;                  // offsets[E+1], prefix[E+1]
  static_assert(NA >= 1, "TMEM ring needs a slot");
  static_assert(kOffW % 1024 == 0, "swizzled tiles need 1024-byte alignment");
  static_assert(kOffRing % 16 == 0, "ring entries are 16-byte vectors");
  static int bytes(int E) {
    int b = kOffTables + 2 * (E + 1) * 4 + 1024;  // + alignment slack
    return b < kMinSmem ? kMinSmem : b;
  }
};

__device__ __forceinline__ int4 ld_shared_v4(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// MODE 0 / 1: one phase, gate_up + SwiGLU / down, fixed at compile time;
// MODE 2: the phases' own modes (the one-launch layer).
template <int BN, int SB, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_gemm_kernel(const __grid_constant__ CUtensorMap tmap_act, const __grid_constant__ CUtensorMap tmap_half,
                      const __grid_constant__ GemmLaunch L) {
  using C = Cfg<BN, SB>;
  constexpr int NSW = C::NSW, NSB = C::NSB, NA = C::NA, R = C::kRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sB = sbase + C::kOffB;
  const uint32_t sW = sbase + C::kOffW;
  const uint32_t bar0 = sbase + C::kOffBar;
  auto fullw_bar = [&](int s) { return bar0 + 8u * s; };
  auto emptyw_bar = [&](int s) { return bar0 + 8u * (NSW + s); };
  auto fullb_bar = [&](int s) { return bar0 + 8u * (2 * NSW + s); };
  auto emptyb_bar = [&](int s) { return bar0 + 8u * (2 * NSW + NSB + s); };
  auto afull_bar = [&](int a) { return bar0 + 8u * (2 * NSW + 2 * NSB + a); };
  auto aempty_bar = [&](int a) { return bar0 + 8u * (2 * NSW + 2 * NSB + NA + a); };
  constexpr int ND = C::ND;
  auto dfull_bar = [&](int d) { return bar0 + 8u * (2 * NSW + 2 * NSB + 2 * NA + d); };
  auto dempty_bar = [&](int d) { return bar0 + 8u * (2 * NSW + 2 * NSB + 2 * NA + ND + d); };
  const uint32_t drain_bar = bar0 + 8u * (2 * NSW + 2 * NSB + 2 * NA + 2 * ND);
  auto tfull_bar = [&](int t) { return drain_bar + 8u * (1 + t); };
  auto tempty_bar = [&](int t) { return drain_bar + 8u * (1 + R + t); };
  // tile j's rows of h are written (down tiles of the one-launch layer)
  auto rdy_bar = [&](int t) { return drain_bar + 8u * (1 + 2 * R + t); };
  const bool ready_warp = C::kGatherB && L.nph > 1;
  const uint32_t s_ring = sbase + C::kOffRing;
  volatile int* s_wflag = reinterpret_cast<volatile int*>(smem + C::kOffWFlag);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const int E = L.E;
  int32_t* s_off = reinterpret_cast<int32_t*>(smem + C::kOffTables);
  int32_t* s_tprefix = s_off + (E + 1);
  int* status = L.status;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- set-up: barriers and TMEM (on-chip only), then the tile table
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSW; ++s) {
      mbar_init(fullw_bar(s), 1);
      mbar_init(emptyw_bar(s), C::kGroupWarps);  // the stage's dequant warps
    }
    for (int s = 0; s < NSB; ++s) {
      mbar_init(fullb_bar(s), C::kGatherB ? kBProducers : 1);  // each gathering warp, or the TMA bytes
      mbar_init(emptyb_bar(s), 1);  // the MMA commit
    }
    for (int a = 0; a < NA; ++a) {
      mbar_init(afull_bar(a), C::kGroupWarps);
      mbar_init(aempty_bar(a), 1);
    }
    for (int d = 0; d < ND; ++d) {
      mbar_init(dfull_bar(d), 1);
      mbar_init(dempty_bar(d), 4);
    }
    mbar_init(drain_bar, 1);
    for (int t = 0; t < R; ++t) {
      mbar_init(tfull_bar(t), 1);                                          // the weight producer
      mbar_init(tempty_bar(t), C::kRingReaders + (ready_warp ? 1 : 0));  // every reader of the entry
      mbar_init(rdy_bar(t), 1);                                            // the readiness warp
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (!C::kGatherB && warp == kWarpProducerB && lane == 0) {
    prefetch_tmap(&tmap_act);
    if (kHalfTiles<BN>) prefetch_tmap(&tmap_half);
  }
  if (C::kGatherB && L.sched != kSchedGrid3D && warp == kWarpProducer && lane == 0) {
    // The packed weights do not come from the kernels before, so while they
    // run this CTA pulls into L2 the weights of one likely early tile: tile
    // blockIdx.x of the phase-0 list if every expert had one token tile.  Of
    // a decode step's first round of tiles most are these (whichever CTA
    // takes them); a wrong guess only costs bandwidth that is idle here.
    const GemmPhase& P0 = L.ph[0];
    const int MT0 = P0.N / kTileM;
    const int e = (int)blockIdx.x / MT0, mt = (int)blockIdx.x % MT0;
    if (e < P0.E_routed) {
      const uint32_t tile_bytes = (uint32_t)(P0.K / kBlockK) * kWBlockBytes;
      const uint8_t* src = P0.packed + (size_t)(e * MT0 + mt) * tile_bytes;
      for (uint32_t o = 0; o < tile_bytes; o += C::kWBytes)
        prefetch_l2_bulk(src + o, min((uint32_t)C::kWBytes, tile_bytes - o));
    }
  }
  if (warp == kWarpMma) {
    tmem_alloc(sbase + C::kOffMisc, kTmemCols);
    tmem_relinquish();
  }
  // everything above is on-chip; the offsets, the activations and the
  // schedule counters come from the kernels before
  pdl_wait();
  pdl_trigger();
  // the claim schedule's first tile: issued now, its latency hidden behind
  // the table build
  int first_claim = 0;
  if (L.sched == kSchedClaim && warp == kWarpProducer && lane == 0) first_claim = atomicAdd(L.claim, 1);
  build_tile_table(L.offsets, E, BN, s_off, s_tprefix, misc + 2);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];

  // Tiles of the launch: the phase-0 tile list, then the phase-1 list.
  const int ntok = (int)misc[2];
  const int MT0 = L.ph[0].N / kTileM;
  const int MT1 = L.nph > 1 ? L.ph[1].N / kTileM : 0;
  const int T0 = ntok * MT0;
  const int total = T0 + ntok * MT1;
  const int KS0 = L.ph[0].K / (kBlockK * SB);
  const int KS1 = L.nph > 1 ? L.ph[1].K / (kBlockK * SB) : 0;
  struct TileRef {
    int ph;  // phase; -1: the end of the CTA's schedule
    TileCoord c;
  };
  // Tile u of the launch, decoded by a whole warp: the expert is the last e
  // with tprefix[e] * MT <= t, found by ballots over 32 candidates at a time
  // (two rounds for up to 1024 experts, three for 1025), so the producer's
  // per-tile decode is a few dependent steps, not a serial binary search.
  auto tile_of = [&](int u) {
    TileRef r;
    r.ph = u < T0 ? 0 : 1;
    const int t = r.ph == 0 ? u : u - T0;
    const int MT = r.ph == 0 ? MT0 : MT1;
    int lo = 0, span = E;
    while (span > 1) {
      const int part = (span + 31) >> 5;
      const int b = lo + lane * part;
      const bool p = lane * part < span && s_tprefix[b] * MT <= t;
      const uint32_t m = __ballot_sync(0xFFFFFFFFu, p);
      const int last = 31 - __clz(m);  // lane 0 always holds: tprefix[lo] * MT <= t
      lo += last * part;
      span = min(part, span - last * part);
    }
    const int ntc = s_tprefix[lo + 1] - s_tprefix[lo];
    const int local = t - s_tprefix[lo] * MT;
    r.c.e = lo;
    r.c.mt = local / ntc;
    r.c.nt = local - r.c.mt * ntc;
    return r;
  };
  // A reader's wait for entry j of the tile ring; every lane reads it, then
  // one lane frees it (unless `release` is false: then the reader frees it
  // itself later).  False if the CTA aborted.
  auto ring_read = [&](int j, TileRef& tr, bool release = true) -> bool {
    const int slot = j % R;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(tfull_bar(slot), (uint32_t)(j / R) & 1u, abort_flag, status)))
      return false;
    const int4 v = ld_shared_v4(s_ring + 16u * slot);
    __syncwarp();
    if (release && lane == 0) mbar_arrive(tempty_bar(slot));
    tr.ph = v.x;
    tr.c.e = v.y;
    tr.c.mt = v.z;
    tr.c.nt = v.w;
    return true;
  };

  if (warp == kWarpProducer) {
    // --------------------------------------------------- schedule + weights
    // This warp decides the CTA's tiles -- u = blockIdx.x, + gridDim.x, ...
    // (static); u = the next value of a global counter (claim: tiles are
    // taken in list order, so every phase-0 tile belongs to a running CTA
    // before any phase-1 tile is handed out); or the one tile of a 3-D grid
    // CTA -- publishes each in the tile ring and streams its packed weight
    // blocks (phase after phase, with no break in between) into the weight
    // ring, one bulk copy per stage issued by one lane.  After the last
    // tile it publishes the end, then one empty weight stage per dequant
    // group flagged as the end of the stream.
    int u;
    if (L.sched == kSchedStatic) {
      u = (int)blockIdx.x;
    } else if (L.sched == kSchedClaim) {
      u = __shfl_sync(0xFFFFFFFFu, first_claim, 0);
    } else {
      // 3-D grid (weight tile, token tile, expert): one tile, if it exists
      const int e = (int)blockIdx.z, nt = (int)blockIdx.y, mt = (int)blockIdx.x;
      const int ntc = e < E ? s_tprefix[e + 1] - s_tprefix[e] : 0;
      u = (e < E && nt < ntc && mt < MT0) ? s_tprefix[e] * MT0 + mt * ntc + nt : total;
    }
    int i = 0;  // weight stages issued
    bool ok = true;
    // Publish tile j (the end when u >= total).  False if the CTA aborted.
    auto publish = [&](int j, int uj, TileRef& tr) -> bool {
      if (uj < total) {
        tr = tile_of(uj);
      } else {
        tr.ph = -1;
        tr.c.e = tr.c.mt = tr.c.nt = 0;
      }
      const int slot = j % R;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(tempty_bar(slot), ((uint32_t)(j / R) & 1u) ^ 1u, abort_flag, status)))
        return false;
      if (lane == 0) {
        asm volatile("st.shared.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(s_ring + 16u * slot), "r"(tr.ph), "r"(tr.c.e),
                     "r"(tr.c.mt), "r"(tr.c.nt)
                     : "memory");
        mbar_arrive(tfull_bar(slot));
      }
      __syncwarp();
      return true;
    };
    // Tile j + 1 is published right after tile j's first weight copy, so
    // that the readers (the gathering warp above all) never wait for it at a
    // tile boundary and the first copy is not held up.  The claim schedule
    // keeps one claim in flight ahead of that: the claim of tile j + 2 is
    // issued when tile j + 1 is published and read a tile later, so its
    // latency is not waited for.  A CTA's claims are increasing, so a claimed
    // but unpublished tile is never a phase-0 tile behind a phase-1 one.
    TileRef tr;
    ok = publish(0, u, tr);
    int pending = 0;  // lane 0: the claim in flight (the claim schedule)
    if (ok && L.sched == kSchedClaim && tr.ph >= 0 && lane == 0) pending = atomicAdd(L.claim, 1);
    for (int j = 0; ok && tr.ph >= 0; ++j) {
      const TileRef cur = tr;
      const GemmPhase& P = L.ph[cur.ph];
      const int MT = cur.ph == 0 ? MT0 : MT1, KS = cur.ph == 0 ? KS0 : KS1;
      // experts 0 .. E_routed-1 are the routed ones; the next (if any) is the
      // shared expert, whose weights are a separate one-expert matrix
      const uint8_t* wsrc = cur.c.e < P.E_routed
                                ? P.packed + (size_t)(cur.c.e * MT + cur.c.mt) * KS * SB * kWBlockBytes
                                : P.shared_packed + (size_t)cur.c.mt * KS * SB * kWBlockBytes;
      for (int ks = 0; ks < KS; ++ks, ++i) {
        const int s = i % NSW;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(emptyw_bar(s), ((uint32_t)(i / NSW) & 1u) ^ 1u, abort_flag, status))) {
          ok = false;
          break;
        }
        if (elect_one_sync()) {
          s_wflag[s] = 1;
          mbar_arrive_expect_tx(fullw_bar(s), (uint32_t)C::kWBytes);
          bulk_copy_g2s(sW + s * C::kWBytes, wsrc + (size_t)ks * C::kWBytes, C::kWBytes, fullw_bar(s));
        }
        __syncwarp();
        if (ks == 0) {
          int u_next;
          if (L.sched == kSchedStatic) u_next = u + (int)gridDim.x;
          else if (L.sched == kSchedClaim) u_next = __shfl_sync(0xFFFFFFFFu, pending, 0);
          else u_next = total;
          if (!publish(j + 1, u_next, tr)) {
            ok = false;
            break;
          }
          if (L.sched == kSchedClaim && tr.ph >= 0 && lane == 0) pending = atomicAdd(L.claim, 1);
          u = u_next;
        }
      }
    }
    // the end of the weight stream: one flagged stage per dequant group
    for (int g = 0; g < C::G && ok; ++g, ++i) {
      const int s = i % NSW;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(emptyw_bar(s), ((uint32_t)(i / NSW) & 1u) ^ 1u, abort_flag, status)))
        break;
      if (lane == 0) {
        s_wflag[s] = 0;
        mbar_arrive(fullw_bar(s));
      }
      __syncwarp();
    }
    // drain: every copy this warp issued has landed before the CTA exits
    for (int j = (i > NSW ? i - NSW : 0); j < i; ++j)
      mbar_wait(fullw_bar(j % NSW), (uint32_t)(j / NSW) & 1u, nullptr, status, kDrainTimeoutNs);
  } else if (!C::kGatherB && warp == kWarpProducerB) {
    // ------------------------------------------- activation tiles by TMA
    // (wide token tiles, one phase): SB 2-D boxes of the permuted rows per
    // stage, issued by one lane.
    int i = 0;
    bool ok = true;
    for (int j = 0; ok; ++j) {
      TileRef tr;
      if (!ring_read(j, tr) || tr.ph < 0) break;
      const int KS = tr.ph == 0 ? KS0 : KS1;
      const int row0 = s_off[tr.c.e] + tr.c.nt * BN;
      const bool half = kHalfTiles<BN> && 2 * (s_off[tr.c.e + 1] - row0) <= BN;
      const CUtensorMap* tm = half ? &tmap_half : &tmap_act;
      for (int ks = 0; ks < KS; ++ks, ++i) {
        const int s = i % NSB;
        const uint32_t freed = C::kOneFreeBar ? aempty_bar(s) : emptyb_bar(s);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(freed, ((uint32_t)(i / NSB) & 1u) ^ 1u, abort_flag, status))) {
          ok = false;
          break;
        }
        if (elect_one_sync()) {
          mbar_arrive_expect_tx(fullb_bar(s), (uint32_t)(half ? C::kBTile / 2 : C::kBTile));
#pragma unroll
          for (int b = 0; b < SB; ++b)
            tma_load_2d(sB + s * C::kBTile + b * C::kBSub, tm, (ks * SB + b) * kBlockK, row0, fullb_bar(s));
        }
        __syncwarp();
      }
    }
    for (int j = (i > NSB ? i - NSB : 0); j < i; ++j)
      mbar_wait(fullb_bar(j % NSB), (uint32_t)(j / NSB) & 1u, nullptr, status, kDrainTimeoutNs);
  } else if (C::kGatherB && warp >= kWarpProducerB && warp < kWarpProducerB + kBProducers) {
    // ------------------------------------- activation rows, gathered (BN <= 32)
    // The gathering warps split every row's 16-byte chunks (with one warp,
    // a 16-row tile takes two lanes per row).  Lane -> (row r, chunks
    // c0 .. c0 + kChunks - 1 of every 64-column block); chunk c of row r lands
    // at r * 128 + ((c ^ (r & 7)) * 16), the 128-byte swizzle the MMA's
    // shared-memory descriptor expects.  Rows past the expert's last token are
    // zero-filled, not read.  A phase-1 tile of expert e first waits until
    // every phase-0 tile of e has written its rows.
    constexpr int kChunks = (BN == 16 ? 4 : 8) / kBProducers;
    const int part = warp - kWarpProducerB;
    const int r = BN == 16 ? (lane & 15) : lane;
    const int c0 = (BN == 16 ? (lane >> 4) * 4 : 0) + part * kChunks;
    uint32_t dst_off[kChunks];
#pragma unroll
    for (int j = 0; j < kChunks; ++j) dst_off[j] = (uint32_t)(r * 128 + (((c0 + j) ^ (r & 7)) * 16));
    // Stages [released, issued) are copied or in flight but not yet handed to
    // the MMA warp; a stage is handed over once at most kBInFlight newer ones
    // are pending, or all at once before a wait on another CTA (so this CTA's
    // own phase-0 tiles never wait behind that wait).
    int issued = 0, released = 0;
    auto release_all = [&]() {
      cp_async_wait_group<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0)
        for (int j = released; j < issued; ++j) mbar_arrive(fullb_bar(j % NSB));
      released = issued;
    };
    // A phase-1 tile of expert e needs every phase-0 tile of e finished (4
    // epilogue warps each); the readiness warp waits for that and signals
    // the tile's rdy barrier, so this warp only waits on shared memory.  Its
    // ring entry is freed after that wait, which keeps the rdy barrier on
    // this tile's lap.
    bool ok = true;
    for (int j = 0; ok; ++j) {
      TileRef tr;
      const int slot = j % R;
      // about to wait for the next tile's entry: hand the pending stages over
      // first, so that the MMA never waits on them meanwhile
      if (!__all_sync(0xFFFFFFFFu, mbar_test_wait(tfull_bar(slot), (uint32_t)(j / R) & 1u))) release_all();
      if (!ring_read(j, tr, false)) break;
      if (tr.ph == 1) {
        const uint32_t par = (uint32_t)(j / R) & 1u;
        if (!__all_sync(0xFFFFFFFFu, mbar_test_wait(rdy_bar(slot), par))) {
          // hand every pending stage over before waiting on other CTAs
          release_all();
          ok = __all_sync(0xFFFFFFFFu, mbar_wait(rdy_bar(slot), par, abort_flag, status));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(slot));
      if (!ok || tr.ph < 0) break;
      const GemmPhase& P = L.ph[tr.ph];
      const int KS = tr.ph == 0 ? KS0 : KS1;
      const int p0 = s_off[tr.c.e] + tr.c.nt * BN;
      const bool valid = r < s_off[tr.c.e + 1] - p0;
      const size_t src_row = valid ? (size_t)(P.gather_rows != nullptr ? P.gather_rows[p0 + r] : p0 + r) : 0;
      const uint16_t* rowp = P.act + src_row * (size_t)P.K + c0 * 8;
      const uint32_t nbytes = valid ? 16u : 0u;
      for (int ks = 0; ks < KS; ++ks) {
        const int s = issued % NSB;
        if (!__all_sync(0xFFFFFFFFu,
                        mbar_wait(emptyb_bar(s), ((uint32_t)(issued / NSB) & 1u) ^ 1u, abort_flag, status))) {
          ok = false;
          break;
        }
        const uint32_t dst = sB + s * C::kBTile;
#pragma unroll
        for (int b = 0; b < SB; ++b) {
          const uint16_t* src = rowp + (ks * SB + b) * kBlockK;
#pragma unroll
          for (int c = 0; c < kChunks; ++c) cp_async16(dst + b * C::kBSub + dst_off[c], src + c * 8, nbytes);
        }
        cp_async_commit();
        ++issued;
        if (issued - released > kBInFlight) {
          // the oldest pending stage has landed for this lane; after the proxy
          // fence and the warp sync it is complete for the MMA to read
          cp_async_wait_group<kBInFlight>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(fullb_bar(released % NSB));
          ++released;
        }
      }
    }
    if (ok) {
      release_all();
    } else {
      cp_async_wait_group<0>();  // nothing may land after the CTA exits
    }
  } else if (warp == kWarpReady) {
    // ------------------------------------------- readiness (one-launch layer)
    // Follows the tile ring; for a phase-1 tile of expert e waits (bounded,
    // acquire loads) until every phase-0 tile of e has published its rows of
    // h (4 epilogue warps each), then arrives on the tile's rdy barrier, whose
    // release / acquire hands that ordering on to the gathering warps.  It
    // runs ahead of them, so their phase-1 tiles rarely wait.  Phase-0 tiles
    // are passed at once.  A CTA's phase-0 tiles all come before its phase-1
    // tiles, so this wait never holds back the CTA's own gate_up work.
    if (ready_warp) {
      for (int j = 0;; ++j) {
        const int slot = j % R;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(tfull_bar(slot), (uint32_t)(j / R) & 1u, abort_flag, status))) break;
        const int4 v = ld_shared_v4(s_ring + 16u * slot);
        bool ok = true;
        if (v.x == 1) {
          const int target = 4 * MT0 * (s_tprefix[v.y + 1] - s_tprefix[v.y]);
          ok = __all_sync(0xFFFFFFFFu, wait_counter(L.ready + v.y, target, abort_flag, status));
        }
        __syncwarp();
        if (lane == 0) {
          if (ok) mbar_arrive(rdy_bar(slot));
          mbar_arrive(tempty_bar(slot));
        }
        if (!ok || v.x < 0) break;
      }
    }
  } else if (warp >= kWarpProducerB) {
    // TMA tiles: warp 22 is the producer above; warp 23 has nothing to do
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issue
    // The whole warp waits and computes the (uniform) operands; one elected
    // lane issues the MMAs and commits.
    constexpr uint32_t idesc = idesc_bf16_f32(kTileM, BN);
    constexpr uint32_t idesc_half = idesc_bf16_f32(kTileM, BN >= 32 ? BN / 2 : 16);
    int i = 0;
    bool ok = true;
    // one entry of lookahead: tile it + 1 is usually published when tile it
    // starts, and reading it then keeps the ring read off the path between
    // the tiles' MMAs
    TileRef nxt;
    bool have_nxt = false;
    for (int it = 0; ok; ++it) {
      TileRef tr;
      if (have_nxt) {
        tr = nxt;
      } else if (!ring_read(it, tr)) {
        break;
      }
      have_nxt = false;
      if (tr.ph < 0) break;
      if (__all_sync(0xFFFFFFFFu, mbar_test_wait(tfull_bar((it + 1) % R), (uint32_t)((it + 1) / R) & 1u)))
        have_nxt = ring_read(it + 1, nxt);
      const int KS = tr.ph == 0 ? KS0 : KS1;
      const int d = it % ND;
      // a 64-row tile with at most 32 valid rows: the producer loaded only
      // those, and the MMAs multiply them alone (both shapes compile-time)
      const bool half = kHalfTiles<BN> && 2 * (s_off[tr.c.e + 1] - (s_off[tr.c.e] + tr.c.nt * BN)) <= BN;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(dempty_bar(d), ((uint32_t)(it / ND) & 1u) ^ 1u, abort_flag, status)))
        break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(d * BN);
      for (int ks = 0; ks < KS; ++ks, ++i) {
        const int s = i % NSB, a = i % NA;
        // gathered activation stages are waited on by the dequant group
        // (afull implies fullb); TMA stages here
        const bool got = mbar_wait(afull_bar(a), (uint32_t)(i / NA) & 1u, abort_flag, status) &&
                         (C::kGatherB || mbar_wait(fullb_bar(s), (uint32_t)(i / NSB) & 1u, abort_flag, status));
        if (!__all_sync(0xFFFFFFFFu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_tmem = tmem_base + (uint32_t)(C::A0 + C::kSlotCols * a);
        const uint64_t b_desc = smem_desc_sw128(sB + s * C::kBTile);
        if (elect_one_sync()) {
          if (half) {
#pragma unroll
            for (int b = 0; b < SB; ++b)
#pragma unroll
              for (int kk = 0; kk < kBlockK / 16; ++kk)
                tc_mma_ts(d_tmem, a_tmem + (uint32_t)(32 * b + 8 * kk),
                          b_desc + (uint64_t)((b * C::kBSub + kk * 32) >> 4), idesc_half, (ks | b | kk) != 0);
          } else {
#pragma unroll
            for (int b = 0; b < SB; ++b)
#pragma unroll
              for (int kk = 0; kk < kBlockK / 16; ++kk)
                tc_mma_ts(d_tmem, a_tmem + (uint32_t)(32 * b + 8 * kk),
                          b_desc + (uint64_t)((b * C::kBSub + kk * 32) >> 4), idesc, (ks | b | kk) != 0);
          }
          tc_commit(aempty_bar(a));
          if (!C::kOneFreeBar) tc_commit(emptyb_bar(s));
        }
        __syncwarp();
      }
      if (ok) {
        if (elect_one_sync()) tc_commit(dfull_bar(d));
        __syncwarp();
      }
    }
    // drain: all MMAs issued by this warp complete before TMEM is freed
    if (elect_one_sync()) tc_commit(drain_bar);
    __syncwarp();
    mbar_wait(drain_bar, 0, nullptr, status, kDrainTimeoutNs);
  } else if (warp >= kWarpDq0) {
    // ------------------------------------------------------------- dequant
    // Stages round-robin over the groups, in the weight ring's order, until a
    // stage flagged as the end of the stream.
    constexpr int G = C::G, kBlocksPerWarp = SB / C::kSplit;
    const int dw = warp - kWarpDq0;
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int group = dw / C::kGroupWarps;
    const int part = (dw % C::kGroupWarps) >> 2;
    const int r = 32 * q + lane;
    const uint32_t t_row = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)C::A0;
#pragma unroll 1
    for (int i = group; group < G; i += G) {
      const int s = i % NSW, a = i % NA;
      // every lane waits (each acquires the copied bytes); the warp acts as one
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(fullw_bar(s), (uint32_t)(i / NSW) & 1u, abort_flag, status))) break;
      // the stage's flag is loaded with its first block's codes (an end stage
      // holds no codes; what is loaded there is dropped)
      const uint8_t* stage_w = smem + C::kOffW + s * C::kWBytes + part * kBlocksPerWarp * kWBlockBytes;
      const int wflag = s_wflag[s];
      // software-pipelined: the next block's codes are loaded while this one is
      // converted, hiding the shared-memory latency
      BlockCodes cur = load_block(stage_w, r);
      if (wflag == 0) break;  // the end of the weight stream
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(aempty_bar(a), ((uint32_t)(i / NA) & 1u) ^ 1u, abort_flag, status)))
        break;
      tc_fence_after();
      // 16-row tiles unroll the loop, so the conversions of a warp's two
      // blocks interleave (measured: a steadier weight stream on decode);
      // wider tiles measured faster one block at a time
#pragma unroll(C::kSplit == 2 ? kBlocksPerWarp : 1)
      for (int bb = 0; bb < kBlocksPerWarp; ++bb) {
        BlockCodes nxt = cur;
        if (bb + 1 < kBlocksPerWarp) nxt = load_block(stage_w + (bb + 1) * kWBlockBytes, r);
        if (bb + 1 == kBlocksPerWarp) {
          __syncwarp();
          if (lane == 0) mbar_arrive(emptyw_bar(s));  // codes are in registers: the slot may be refilled
        }
        uint32_t v[32];
        dequant_block(cur, v);
        tmem_st32(t_row + (uint32_t)(C::kSlotCols * a + 32 * (part * kBlocksPerWarp + bb)), v);
        cur = nxt;
      }
      tc_wait_st();
      tc_fence_before();
      if (C::kGatherB && q == 0 && part == 0) {
        // The stage's activation rows too, so that the MMA warp waits on one
        // barrier per stage.  Gathered stages are released in order, so the
        // in-order fullb phases cannot alias across the groups that wait here.
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(fullb_bar(i % C::NSB), (uint32_t)(i / C::NSB) & 1u, abort_flag,
                                               status)))
          break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(afull_bar(a));
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp - kWarpEpi0;
    for (int it = 0;; ++it) {
      TileRef tr;
      if (!ring_read(it, tr) || tr.ph < 0) break;
      const GemmPhase& P = L.ph[tr.ph];
      const TileCoord c = tr.c;
      const int d = it % ND;
      const uint32_t dph = (uint32_t)(it / ND) & 1u;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(dfull_bar(d), dph, abort_flag, status))) break;
      tc_fence_after();
      const int p0 = s_off[c.e] + c.nt * BN;
      const int nvalid = min(BN, s_off[c.e + 1] - p0);
      const float gsc = __ldg(c.e < P.E_routed ? P.gscale + c.e : P.shared_gscale) * 128.0f;
      const uint32_t t_acc = tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(d * BN);
      // only the accumulator columns of valid rows are read (a partial tile
      // of a 128-row width loaded all 8 column chunks before: skewed gate_up
      // 366 -> 345 us)
#pragma unroll 1
      for (int cc = 0; cc * 16 < nvalid; ++cc) {
        uint32_t v[16];
        tmem_ld16(t_acc + (uint32_t)(cc * 16), v);
        tc_wait_ld();
        if ((MODE == 2 ? P.mode : MODE) == 0) {
          // rows 32q..32q+15 hold gate features f, rows 32q+16.. the matching up rows
          const int f = c.mt * 64 + 16 * q + (lane & 15);
          const bool is_gate = lane < 16;
          uint16_t* h = reinterpret_cast<uint16_t*>(P.out);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float a = __uint_as_float(v[j]);
            const float b = __uint_as_float(v[j + 8]);
            const float send = is_gate ? b : a;
            const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, 16);
            const float own = is_gate ? a : b;
            const float g = (is_gate ? own : recv) * gsc;
            const float up = (is_gate ? recv : own) * gsc;
            const int col = cc * 16 + j + (is_gate ? 0 : 8);
            if (col < nvalid) {
              // silu(g) * up with the fast exponential and the fast, branch-free
              // division: an IEEE division's slow-path branch kept the loop's
              // iterations from overlapping, and the epilogue then bounded
              // short tiles (skewed gate_up 438 -> 340 us)
              const float hv = __fdividef(g, 1.0f + __expf(-g)) * up;
              h[(size_t)(p0 + col) * P.out_ld + f] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
            }
          }
        } else {
          const int n = c.mt * kTileM + 32 * q + lane;
          float* y = reinterpret_cast<float*>(P.out);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = cc * 16 + j;
            if (col < nvalid) y[(size_t)(p0 + col) * P.out_ld + n] = __uint_as_float(v[j]) * gsc;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dempty_bar(d));
      if (tr.ph == 0 && L.nph > 1) {
        // this warp's rows of h are written: publish them to phase-1 tiles
        __threadfence();
        __syncwarp();
        if (lane == 0) counter_add_release(L.ready + c.e, 1);
      }
    }
  }

  // ---- teardown: everyone is here; the MMA warp drained its work
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

static GemmPhase phase_of(int mode, const GemmArgs& a) {
  GemmPhase p;
  p.packed = a.packed;
  p.gscale = a.gscale;
  p.shared_packed = a.shared_packed;
  p.shared_gscale = a.shared_gscale;
  p.E_routed = a.shared_packed != nullptr ? a.E - 1 : a.E;
  p.out = a.out;
  p.act = a.act;
  p.gather_rows = a.gather_rows;
  p.N = a.N;
  p.K = a.K;
  p.out_ld = a.out_ld;
  p.mode = mode;
  return p;
}

// `rows` activation rows (T*k); the phases of L share them and the offsets.
template <int BN, int SB, int MODE>
static cudaError_t launch_gemm_cfg(const GemmLaunch& L, int rows, int T, cudaStream_t s) {
  using C = Cfg<BN, SB>;
  // TMA tiles: boxes of 64 columns x BN rows (a token tile) and x BN/2 rows
  // (a tile with at most half its rows valid, kHalfTiles)
  CUtensorMap tmap, tmap_half;
  memset(&tmap, 0, sizeof(tmap));
  memset(&tmap_half, 0, sizeof(tmap_half));
  if (!C::kGatherB) {
    // TMA tiles read a permuted copy, one phase per launch
    if (L.nph != 1 || L.ph[0].gather_rows != nullptr) return cudaErrorInvalidValue;
    PFN_encodeTiled enc = get_encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    const cuuint64_t gdim[2] = {(cuuint64_t)L.ph[0].K, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)L.ph[0].K * 2};
    const cuuint32_t estride[2] = {1, 1};
    for (int m = 0; m < (kHalfTiles<BN> ? 2 : 1); ++m) {
      const cuuint32_t box[2] = {(cuuint32_t)kBlockK, (cuuint32_t)(m == 0 ? BN : BN / 2)};
      CUresult r = enc(m == 0 ? &tmap : &tmap_half, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                       const_cast<uint16_t*>(L.ph[0].act), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                       CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
  }
  const int smem = C::bytes(L.E);
  auto kern = w4a16_gemm_kernel<BN, SB, MODE>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  if (L.sched == kSchedGrid3D) {
    // (weight tiles, token tiles of the largest possible expert, experts): an
    // expert receives each token at most once, so it has at most T rows
    if (L.nph != 1 || T <= 0) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(L.ph[0].N / kTileM), (unsigned)((T + BN - 1) / BN), (unsigned)L.E);
    return launch_pdl(kern, grid, dim3(kThreads), smem, s, tmap, tmap_half, L);
  }
  if (L.sched == kSchedClaim && L.claim == nullptr) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const long long n = rows;
  long long max_tiles = 0;
  for (int p = 0; p < L.nph; ++p) max_tiles += (long long)(L.ph[p].N / kTileM) * (n / BN + (n < L.E ? n : L.E));
  const int grid = (int)(max_tiles < sms ? max_tiles : sms);
  if (grid <= 0) return cudaSuccess;
  // Persistent: at most one CTA per SM (a CTA takes a whole SM's shared
  // memory and TMEM).  The one-launch layer's down tiles wait on gate_up
  // tiles of other CTAs; with the claim schedule every gate_up tile is taken
  // by a running CTA before any down tile is handed out, so the waits end
  // whatever the residency.  The launch is programmatic, so its CTAs start
  // on the free SMs while the kernel before finishes (a cooperative launch
  // measured about 2.4 us more per decode step).
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, tmap, tmap_half, L);
}

// Token tile width: the smallest of 16/32/64/128 that covers about twice the
// mean number of rows per expert (T*k/E), so a decode step is one tile per
// expert, the grouped 800-token layer (25 rows per expert) takes 64-row tiles
// and prefill the widest.  Measured on all four workloads (every width x
// schedule): the choice is the fastest or within 1% of it.
static int pick_bn(int rows, int E) {
  const long long mean2 = 2LL * rows / (E > 0 ? E : 1);
  if (mean2 <= 16) return 16;
  if (mean2 <= 32) return 32;
  if (mean2 <= 64) return 64;
  return 128;
}

// K blocks per stage: 4 (K 256 per stage amortises the per-stage handoffs
// between the dequant groups and the MMA warp: measured faster for every
// token-tile width), or 2 or 1 when a phase's K/64 is not a multiple of 4.
static int pick_sb(const int* kb, int nph) {
  int sb = 4;
  for (;;) {
    bool ok = true;
    for (int p = 0; p < nph; ++p) ok = ok && kb[p] % sb == 0;
    if (ok || sb == 1) return sb;
    sb >>= 1;
  }
}

template <int BN, int MODE>
static cudaError_t launch_gemm_mode(const GemmLaunch& L, int rows, int T, cudaStream_t s) {
  int kb[2];
  for (int p = 0; p < L.nph; ++p) kb[p] = L.ph[p].K / kBlockK;
  switch (pick_sb(kb, L.nph)) {
    case 4: return launch_gemm_cfg<BN, 4, MODE>(L, rows, T, s);
    case 2: return launch_gemm_cfg<BN, 2, MODE>(L, rows, T, s);
    default: return launch_gemm_cfg<BN, 1, MODE>(L, rows, T, s);
  }
}

template <int BN>
static cudaError_t launch_gemm_bn(const GemmLaunch& L, int rows, int T, cudaStream_t s) {
  if (L.nph > 1) {
    if constexpr (BN <= 32) return launch_gemm_mode<BN, 2>(L, rows, T, s);
    return cudaErrorInvalidValue;  // one-launch layers use narrow token tiles only
  }
  return L.ph[0].mode == 0 ? launch_gemm_mode<BN, 0>(L, rows, T, s) : launch_gemm_mode<BN, 1>(L, rows, T, s);
}

static cudaError_t launch_gemm_any(const GemmLaunch& L, int rows, int T, int bn, cudaStream_t s) {
  switch (bn) {
    case 16: return launch_gemm_bn<16>(L, rows, T, s);
    case 32: return launch_gemm_bn<32>(L, rows, T, s);
    case 64: return launch_gemm_bn<64>(L, rows, T, s);
    case 128: return launch_gemm_bn<128>(L, rows, T, s);
    default: return cudaErrorInvalidValue;
  }
}

GemmPlan plan_layer(int rows, int E, int /*H*/, int /*I*/, int force_bn, int force_sched) {
  GemmPlan p;
  p.bn = force_bn > 0 ? force_bn : pick_bn(rows, E);
  p.gathers = p.bn <= 32;
  // narrow tiles: both projections in one launch with the claim schedule
  // (its down tiles wait on gate_up tiles of other CTAs; claim keeps that
  // independent of SM residency); wide tiles: one launch per projection with
  // the static stride.  Measured: the 3-D grid is 2-10x slower on every
  // workload; static and claim are within a few per cent of each other.
  p.sched = force_sched >= 0 ? force_sched : (p.gathers ? kSchedClaim : kSchedStatic);
  p.fused = rows > 0 && p.gathers && p.sched != kSchedGrid3D;
  return p;
}

cudaError_t launch_gemm_planned(int mode, const GemmArgs& a, const GemmPlan& plan, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  GemmLaunch L;
  memset(&L, 0, sizeof(L));
  L.ph[0] = phase_of(mode, a);
  L.nph = 1;
  L.offsets = a.offsets;
  L.status = a.status;
  L.claim = a.claim;
  L.E = a.E;
  L.sched = plan.sched;
  if (a.gather_rows != nullptr && !plan.gathers) return cudaErrorInvalidValue;
  return launch_gemm_any(L, a.rows, a.T, plan.bn, s);
}

cudaError_t launch_gemm(int mode, const GemmArgs& a, cudaStream_t s) {
  GemmPlan p = plan_layer(a.rows, a.E, 0, 0, -1, kSchedStatic);
  return launch_gemm_planned(mode, a, p, s);
}

cudaError_t launch_gemm_layer(const GemmArgs& gate_up, const GemmArgs& down, int32_t* ready, const GemmPlan& plan,
                              cudaStream_t s) {
  if (gate_up.rows == 0) return cudaSuccess;
  if (!plan.fused || ready == nullptr) return cudaErrorInvalidValue;
  GemmLaunch L;
  memset(&L, 0, sizeof(L));
  L.ph[0] = phase_of(0, gate_up);
  L.ph[1] = phase_of(1, down);
  L.nph = 2;
  L.offsets = gate_up.offsets;
  L.ready = ready;
  L.claim = gate_up.claim;
  L.status = gate_up.status;
  L.E = gate_up.E;
  L.sched = plan.sched;
  return launch_gemm_any(L, gate_up.rows, gate_up.T, plan.bn, s);
}

// ------------------------------------------------------------------ prepack
// Packed block of a 128-row x 64-column tile (4608 bytes):
//   codes  [half 0..1][row 0..127][16 B] at (half * 128 + row) * 16: K
//          elements 32*half .. 32*half+31 of the row as 4 words of 8;
//   scales [row][4] at 4096 + row * 4: the row's four E4M3 block scales.
// Packed word w holds elements 8w..8w+7 in the slot placement of
// nvfp4_pack_word (device_common.cuh).
// One thread per (expert, tile, K block, half, row) moves 16 code bytes and
// the two scales of those 32 elements.
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
    uint32_t c8[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t b = cs[4 * w + j];  // elements 8w+2j (low nibble) and 8w+2j+1 (high nibble)
      c8[2 * j] = b & 0xFu;
      c8[2 * j + 1] = b >> 4;
    }
    words[w] = nvfp4_pack_word(c8);
  }
  uint8_t* dst = packed + blk * kWBlockBytes;
  *reinterpret_cast<uint4*>(dst + (half * 128 + r) * 16) = make_uint4(words[0], words[1], words[2], words[3]);
  const uint8_t* ss = scales + src_row * (K / 16) + kb * 4 + half * 2;
  dst[4096 + r * 4 + half * 2 + 0] = ss[0];
  dst[4096 + r * 4 + half * 2 + 1] = ss[1];
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
    uint32_t c8[8];
    for (int j = 0; j < 8; ++j) c8[j] = (uint32_t)(8 * w + j);
    const uint32_t q = nvfp4_pack_word(c8);
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

// Waits, like a down tile of the one-launch projections, on a GPU-scope
// readiness counter that nothing increments (`ctr`, zero, target 1); the
// bounded wait must give up and record a timeout.
__global__ void counter_timeout_probe_kernel(int* status, const int* ctr, unsigned long long limit_ns) {
  wait_counter(ctr, 1, nullptr, status, limit_ns);
}

cudaError_t launch_counter_timeout_probe(int* status, const int* ctr, unsigned long long limit_ns, cudaStream_t s) {
  counter_timeout_probe_kernel<<<1, 32, 0, s>>>(status, ctr, limit_ns);
  return cudaGetLastError();
}

}  // namespace moe
