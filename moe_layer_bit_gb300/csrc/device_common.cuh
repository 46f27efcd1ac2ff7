// device_common.cuh -- device-side helpers shared by the library's kernels:
// status word, bounded waits, inline-PTX wrappers for mbarrier / bulk copy /
// TMA / tcgen05, and the on-chip NVFP4 -> bf16 dequantiser.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace moe {

// Status codes written to the device status word (same values as moe_status).
constexpr int kStatusOk = 0;
constexpr int kStatusDeviceTimeout = 6;

// A pipeline wait gives up after this long (globaltimer nanoseconds).
constexpr unsigned long long kWaitTimeoutNs = 1000ull * 1000ull * 1000ull;  // ~1 s
// Waits on the drain path at kernel exit (copies / MMAs still in flight).
constexpr unsigned long long kDrainTimeoutNs = 200ull * 1000ull * 1000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may begin while the
// kernel before it in the stream is still running.  pdl_wait() blocks until
// that predecessor grid has completed and its memory writes are visible (it
// returns at once when there is no programmatic predecessor); every kernel of
// the library calls it before its first global-memory access, so the overlap
// covers only launch and on-chip set-up.  pdl_trigger() lets the successor
// start launching once every CTA of this grid has called it or exited.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// try_wait with a suspend-time hint: a waiting thread sleeps in hardware until
// the phase completes or about `hint_ns` pass, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns = 1000000u) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Non-blocking test of a phase: returns at once.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// One lane of the (fully active) warp returns true.
__device__ __forceinline__ bool elect_one_sync() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .b32 r;\n\t.reg .pred p;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// if the CTA-wide abort flag is raised or the wait exceeds `limit_ns`; in the
// latter case it raises the abort flag and records a timeout in `status`.
// try_wait gives up after a short hardware-chosen time, so a long wait loops;
// a waiter off the critical path passes `sleep_ns` to yield its issue slots
// between polls, and the abort flag and clock are read every 16th poll only.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, unsigned long long limit_ns = kWaitTimeoutNs,
                                          uint32_t sleep_ns = 0) {
  if (mbar_test_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
#pragma unroll 1
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if (sleep_ns != 0) __nanosleep(sleep_ns);
    if ((n & 15u) != 0) continue;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      if (abort_flag != nullptr) *abort_flag = 1;
      if (status != nullptr) atomicExch(status, kStatusDeviceTimeout);
      return false;
    }
  }
}

// Acquire load of a GPU-scope counter.
__device__ __forceinline__ int counter_load_acquire(const int* ctr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
  return v;
}
// Bounded wait until the GPU-scope counter *ctr reaches `target`, polled with
// acquire loads (so this thread's later reads see what the writers published
// before their release increments) and a short sleep between polls.  Same
// abort / timeout behaviour as mbar_wait.
__device__ __forceinline__ bool wait_counter(const int* ctr, int target, volatile int* abort_flag, int* status,
                                             unsigned long long limit_ns = kWaitTimeoutNs) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
  if (v >= target) return true;
  const unsigned long long t0 = globaltimer_ns();
#pragma unroll 1
  for (uint32_t n = 1;; ++n) {
    __nanosleep(128);
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= target) return true;
    if ((n & 15u) != 0) continue;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      if (abort_flag != nullptr) *abort_flag = 1;
      if (status != nullptr) atomicExch(status, kStatusDeviceTimeout);
      return false;
    }
  }
}
// Adds v to a GPU-scope counter with release semantics.
__device__ __forceinline__ void counter_add_release(int* ctr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(ctr), "r"(v) : "memory");
}

// ----------------------------------------------------------- bulk / TMA copy
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t c0, int32_t c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(dst),
      "l"(tmap), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
// Hint: pull `bytes` (a multiple of 16, 16-byte aligned) of global memory
// into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// 16-byte cp.async into shared memory through L2 (no L1 allocation); the
// bytes past `src_bytes` (0 or 16) are zero-filled and not read.  Completion
// is tracked per thread with commit / wait groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's committed groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Makes this thread's completed generic-proxy shared-memory writes (plain
// stores, cp.async) visible to later async-proxy reads (tcgen05.mma operands).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]; kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 columns store (thread i -> lane base+i, registers -> columns).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzle: rows of 128 B, 8-row swizzle atoms 1024 B apart.
//   bits  0-13 start address >> 4, 16-29 leading byte offset >> 4 (unused for
//   swizzled K-major, set to 1), 32-45 stride byte offset >> 4 (1024 B),
//   46-47 descriptor version (1), 61-63 swizzle mode (2 = 128 B).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor for kind::f16: D fp32 (bits 4-5 = 1), A bf16 (bits 7-9
// = 1), B bf16 (bits 10-12 = 1), both K-major, N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------- NVFP4 dequantiser
// An E2M1 code s.e1.e0.m whose sign sits at bf16 bit 15 and whose e1.e0.m sit
// at bits 8..6 is the bf16 pattern of value * 2^-126 (e1.e0 = exponent field,
// m = top mantissa bit; exponent 0 is the bf16 subnormal m * 2^-127 =
// 0.5m * 2^-126).  Multiplying by S' = scale * 2^119 (exact in bf16: the E4M3
// scale has 4 significant bits and S' <= 1.75 * 2^127) gives
// value * scale * 2^-7, exact (<= 6 significant bits, >= 2^-17, normal).  The
// epilogue multiplies by global_scale * 2^7.
//
// Packed word of 8 consecutive K elements e0..e7: the low 16 bits hold the even
// elements, the high 16 bits the odd ones (element 2j+1 at the same bit
// positions + 16 as element 2j).  Per half, the four codes sit in slots
//   A (e0/e1): s 15, e1 8,  e0 7,  m 6    -> already in place
//   B (e2/e3): s 12, e1 5,  e0 4,  m 3    -> shift left 3
//   C (e4/e5): s 9,  e1 2,  e0 1,  m 0    -> shift left 6
//   D (e6/e7): s 11, e1 10, e0 14, m 13   -> from the isolated slot:
//              sign << 4, e1 >> 2, e0.m >> 7
// so every output column is one mask of a shifted word, and no shifted copy
// drops a foreign bit onto a kept position (bits 15, 8..6 of each half).
constexpr uint32_t kBf16PatternMask = 0x81C081C0u;

__device__ __host__ __forceinline__ uint32_t nvfp4_slot_bits(uint32_t code, int slot) {
  const uint32_t s = (code >> 3) & 1u, e1 = (code >> 2) & 1u, e0 = (code >> 1) & 1u, m = code & 1u;
  switch (slot) {
    case 0: return (s << 15) | (e1 << 8) | (e0 << 7) | (m << 6);
    case 1: return (s << 12) | (e1 << 5) | (e0 << 4) | (m << 3);
    case 2: return (s << 9) | (e1 << 2) | (e0 << 1) | m;
    default: return (s << 11) | (e1 << 10) | (e0 << 14) | (m << 13);
  }
}

// Packed word from the 8 codes of elements e0..e7.
__device__ __host__ __forceinline__ uint32_t nvfp4_pack_word(const uint32_t (&codes)[8]) {
  uint32_t w = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) w |= nvfp4_slot_bits(codes[2 * j], j) | (nvfp4_slot_bits(codes[2 * j + 1], j) << 16);
  return w;
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Two E4M3 scale bytes (lo, hi of a 16-bit value) -> S' = scale * 2^119 as bf16,
// duplicated into both halves of a 32-bit word, for each of the two scales.
__device__ __forceinline__ void e4m3x2_to_scaleprime(uint16_t two, uint32_t& s_lo, uint32_t& s_hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
  const float f_lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * 0x1p119f;
  const float f_hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * 0x1p119f;
  asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(s_lo) : "f"(f_lo));
  asm("cvt.rn.bf16x2.f32 %0, %1, %1;" : "=r"(s_hi) : "f"(f_hi));
}

// Dequantise one packed word (8 elements, one block scale S') into 4 bf16x2
// columns: column j = (e_{2j}, e_{2j+1}).
__device__ __forceinline__ void dequant_word(uint32_t q, uint32_t sprime, uint32_t* out4) {
  const uint32_t d = q & 0x6C006C00u;  // slot D, isolated
  out4[0] = bf16x2_mul(q & kBf16PatternMask, sprime);
  out4[1] = bf16x2_mul((q << 3) & kBf16PatternMask, sprime);
  out4[2] = bf16x2_mul((q << 6) & kBf16PatternMask, sprime);
  out4[3] = bf16x2_mul(((d << 4) | (d >> 2) | (d >> 7)) & kBf16PatternMask, sprime);
}

}  // namespace moe
