// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// (tiled tensor and 1-D bulk copies), and the tcgen05 tensor-core family
// (TMEM alloc/dealloc, MMA, commit, TMEM loads/stores, fences).
//
// Every wait in this library is bounded by a time limit (counted in SM clock
// cycles): a wait that runs out records FIA_ERR_TIMEOUT in the call's device
// status word and returns false so the caller can unwind instead of spinning
// forever.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace fia {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per wait
constexpr uint64_t kShortestWaitLimitNs = 100000;   // limits below this (tests only) skip the blocking first try

// Waits are timed with the SM's cycle counter (a register read; the global
// nanosecond timer is far slower to read and sat on every wait's path).  The
// limits are converted at kCyclesPerNs, above the 2.07 GHz maximum SM clock,
// so a limit never expires early.
constexpr uint64_t kCyclesPerNs = 3;
__device__ __forceinline__ uint64_t cycles() { return static_cast<uint64_t>(clock64()); }

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Rounds a dynamic shared-memory pointer up to a 1024-byte boundary (the
// 128-byte swizzle atom) with pointer arithmetic, so the compiler still knows
// the result is a shared-memory address and emits ld/st.shared.
__device__ __forceinline__ uint8_t* align_smem_1024(uint8_t* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  return p + ((1024u - (a & 1023u)) & 1023u);
}

__device__ __forceinline__ bool elect_lane0() { return (threadIdx.x & 31) == 0; }

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// One arrival per warp: the warp barrier orders every lane's earlier writes
// before lane 0's (releasing) arrive; a barrier counting warps instead of
// threads keeps the arrival traffic small.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Non-blocking check: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Device status word of one call: (epoch << 8) | code, where the epoch is a
// per-call number from the host.  The first CTA stamps (epoch << 8) when it
// starts; an error raises the word with atomicMax, so the newest call's worst
// code wins whatever order the writes land in, and no per-call reset is needed.
struct DevStatus {
  unsigned long long* word;
  unsigned long long epoch;
  // Limit of the waits that can give up (the ones that unwind a CTA); the
  // waits that let in-flight copies and products finish before a CTA exits
  // always use kWaitLimitNs.  (No default member initializer: the parameter
  // structs that hold a DevStatus stay trivial types.)
  unsigned long long limit_ns;
};

// Tag of a call in the high half of a per-unit completion counter.  The
// counters live in the caller's workspace, whose bytes may hold whatever an
// earlier call left there (plan entries, partial results): a bare epoch, a
// small integer, would match such leftovers.  The epoch is spread over 31
// bits (multiplicative hashing with the golden-ratio constant, Knuth) and the
// top bit set, so a stale word matches a given call with probability 2^-31.
__device__ __forceinline__ unsigned long long unit_tag(unsigned long long epoch) {
  const uint32_t x = (uint32_t(epoch) ^ uint32_t(epoch >> 32)) * 2654435761u;
  return (unsigned long long)(x | 0x80000000u) << 32;
}

// Increments a counter word (tag << 32) | count that belongs to the call
// with this tag (unit_tag of its epoch) and returns the new count.  A word
// left by an earlier call, or any other bytes, is claimed for this call by the
// first increment that sees it (the claim sets the count to 1); every other
// increment is one atomic add, so many CTAs bumping one word at once cost
// one round trip each, not a compare-and-swap retry each.
__device__ __forceinline__ unsigned tagged_increment(unsigned long long* ctr, unsigned long long tag) {
  unsigned long long old = atomicAdd(ctr, 1ull);
  while ((old & 0xffffffff00000000ull) != tag) {
    const unsigned long long prev = atomicCAS(ctr, old + 1ull, tag | 1ull);
    if (prev == old + 1ull) return 1u;
    if ((prev & 0xffffffff00000000ull) == tag) {
      old = atomicAdd(ctr, 1ull);
    } else {
      old = prev - 1ull;   // another stale increment came in between: claim from its value
    }
  }
  return unsigned(old & 0xffffffffull) + 1u;
}

// tagged_increment with acquire-release semantics at device scope: the
// increment publishes every write that happens before it (the partial
// results other warps of the CTA handed over through a CTA barrier), and the
// increment that sees the final count observes every earlier increment's
// writes.  Lighter than a sequentially consistent fence on each side.
__device__ __forceinline__ unsigned long long atom_add_acq_rel(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}
__device__ __forceinline__ unsigned long long atom_cas_acq_rel(unsigned long long* p, unsigned long long cmp,
                                                               unsigned long long val) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.cas.b64 %0, [%1], %2, %3;" : "=l"(old) : "l"(p), "l"(cmp), "l"(val) : "memory");
  return old;
}
__device__ __forceinline__ unsigned tagged_increment_acq_rel(unsigned long long* ctr, unsigned long long tag) {
  unsigned long long old = atom_add_acq_rel(ctr, 1ull);
  while ((old & 0xffffffff00000000ull) != tag) {
    const unsigned long long prev = atom_cas_acq_rel(ctr, old + 1ull, tag | 1ull);
    if (prev == old + 1ull) return 1u;
    if ((prev & 0xffffffff00000000ull) == tag) {
      old = atom_add_acq_rel(ctr, 1ull);
    } else {
      old = prev - 1ull;   // another stale increment came in between: claim from its value
    }
  }
  return unsigned(old & 0xffffffffull) + 1u;
}

// The stamp is a compare-and-swap loop keyed on the epoch: it replaces
// whatever an earlier call (or uninitialised memory) left, and never clears a
// code this call has already raised.
__device__ __forceinline__ void status_stamp(const DevStatus& st) {
  if (st.word == nullptr) return;
  unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(st.word);
  while ((cur >> 8) != st.epoch) {
    const unsigned long long prev = atomicCAS(st.word, cur, st.epoch << 8);
    if (prev == cur) break;
    cur = prev;
  }
}

// The stamp above has set the word to this call's epoch, so a raise is one
// atomic maximum (the newest epoch's worst code wins).
__device__ __forceinline__ void status_raise(const DevStatus& st, unsigned code) {
  if (st.word != nullptr) atomicMax(st.word, (st.epoch << 8) | code);
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// (after recording FIA_ERR_TIMEOUT) if the limit passes or another role of the
// CTA has already given up (*abort != 0).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          const DevStatus status) {
  // The status comes by value: the call site copies it out of the kernel
  // parameters into registers (constant-bank reads, hoisted out of loops).
  // A reference into the parameters would make the limit a generic memory
  // load on every wait.  The first probe does not block; then one try_wait
  // that may suspend the thread until the phase completes -- skipped under a
  // limit shorter than such a suspension (a test's), which is checked first.
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t limit_ns = abort != nullptr ? status.limit_ns : kWaitLimitNs;
  if (limit_ns >= kShortestWaitLimitNs && mbar_try_wait(bar, parity)) return true;
  const uint64_t limit = limit_ns * kCyclesPerNs;
  const uint64_t t0 = cycles();
  while (true) {
    if (cycles() - t0 > limit) {
      if (abort != nullptr) *abort = 1;
      status_raise(status, 10u /* FIA_ERR_TIMEOUT */);
      return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
  }
}

// ------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialisation may start while the
// kernel before it on the stream is still running: grid_dep_wait() blocks until
// that kernel has completed and its writes are visible, so every read of an
// input and every write of an output or of the workspace comes after it.
// grid_dep_launch() lets the next such kernel start launching (its CTAs still
// wait for this one to complete before touching memory).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The wait of the two-tile prefill, MLA decode and FP8 block-sparse kernels,
// whose issuing and softmax warps sit at the register limit with many inlined
// wait sites: the fast path is one suspending try_wait and nothing else; the
// limit (the status's, read through the reference) and the clock are touched
// only once that first try has come back empty.  Same-box A/B against
// mbar_wait: varlen TND prefill 0.384 -> 0.365 ms, MLA decode 0.245 -> 0.237
// ms (the single-tile block-sparse kernel measured 1% slower with it and keeps
// mbar_wait).  Under a test's short limit the wait gives up once the first
// suspension ends; the paged decode kernels, whose tests make every wait give
// up, keep mbar_wait (no blocking first try under such a limit).
__device__ __forceinline__ bool mbar_wait_lean(uint64_t* bar, uint32_t parity, volatile int* abort,
                                               const DevStatus& status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t limit_ns = abort != nullptr ? status.limit_ns : kWaitLimitNs;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer() - t0 > limit_ns) {
      if (abort != nullptr) *abort = 1;
      status_raise(status, 10u /* FIA_ERR_TIMEOUT */);
      return false;
    }
  }
}

// ----------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* desc) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(desc)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const void* desc, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// Warms L2 with a tile a later tma_load_2d of the same coordinates will read
// (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* desc, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(desc)),
               "r"(c0), "r"(c1)
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_4d(const void* desc, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(desc)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const void* desc, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const void* desc, uint64_t* bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}


__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Per-thread asynchronous copy of N (4, 8 or 16) bytes global -> shared.  Only
// src_bytes (<= N) are read; the rest of the destination is zero-filled.  Both
// addresses are N-byte aligned.  Completion: cp_async_commit + cp_async_wait_all
// by the issuing thread, which then sees the data.
template <int N>
__device__ __forceinline__ void cp_async_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  static_assert(N == 4 || N == 8 || N == 16, "cp.async size");
  if constexpr (N == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(dst), "l"(src), "n"(N), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Bit k (k = 0..3) set when byte k of w is nonzero: the high bit of
// ((b & 0x7f) + 0x7f) | b is set iff b != 0 (no carry leaves a byte), and the
// multiply gathers bits 7, 15, 23, 31 into bits 28..31 (the partial products
// land on distinct positions, so nothing carries into them).
__device__ __forceinline__ uint32_t nonzero_bytes4(uint32_t w) {
  const uint32_t hi = (((w & 0x7f7f7f7fu) + 0x7f7f7f7fu) | w) & 0x80808080u;
  return (hi * 0x00204081u) >> 28;
}

// ------------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
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

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on an mbarrier when all previously issued tcgen05 async ops of
// this thread have completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// tcgen05.ld fills its destination registers asynchronously: they hold the
// data only once tcgen05.wait::ld has returned.  The compiler does not know
// that, so the wait names the registers as read-write operands -- every use
// then depends on the wait and cannot be scheduled ahead of it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
        "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
        "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

// For further register sets loaded before the same wait: an empty statement
// that keeps their uses after it (volatile asm statements keep their order).
__device__ __forceinline__ void tmem_regs_after_wait(uint32_t (&r)[32]) {
  asm volatile(""
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
        "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
        "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}
// The same for smaller register sets (4, 8 or 16 columns).
template <int N>
__device__ __forceinline__ void tmem_regs_after_wait_n(uint32_t (&r)[N]) {
  static_assert(N == 4 || N == 8 || N == 16, "column count");
  if constexpr (N == 4) {
    asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]));
  } else if constexpr (N == 8) {
    asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]));
  } else {
    asm volatile(""
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
  }
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (taddr.lane + i), registers r[c] = column (taddr.col + c).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Narrower loads (4, 8 or 16 consecutive columns), each with its register-tied
// wait.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[4]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3])
      :
      : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
      :
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
      :
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// --------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;   // version
  d |= (uint64_t)2 << 61;   // SWIZZLE_128B
  return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation.
//   a_bf16/b_bf16: operand type (0 = f16, 1 = bf16); a_mn/b_mn: 1 = MN-major.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t M, uint32_t N, uint32_t is_bf16, uint32_t a_mn,
                                                 uint32_t b_mn) {
  return (1u << 4)                 // D = f32
         | (is_bf16 << 7)          // A type
         | (is_bf16 << 10)         // B type
         | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// ---------------------------------------------------------------- numerics
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum in one instruction (sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Pairs of fp32 in one 64-bit register, for the packed f32x2 arithmetic of
// sm_100 and later (one instruction does both lanes).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Maximum of x[0..N) with 8 independent accumulators (short dependency chains).
template <int N>
__device__ __forceinline__ float tree_max(const float* x) {
  static_assert(N % 8 == 0, "N must be a multiple of 8");
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = x[k];
#pragma unroll
  for (int c = 8; c < N; c += 8)
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = fmaxf(a[k], x[c + k]);
  return fmaxf(fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])), fmaxf(fmaxf(a[4], a[5]), fmaxf(a[6], a[7])));
}

// x[c] <- 2^(x[c] * sl2 - mo) in place; returns the sum (8 independent accumulators).
template <int N>
__device__ __forceinline__ float exp2_and_sum(float* x, float sl2, float mo) {
  static_assert(N % 8 == 0, "N must be a multiple of 8");
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = 0.f;
#pragma unroll
  for (int c = 0; c < N; c += 8)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float y = fast_exp2(fmaf(x[c + k], sl2, -mo));
      x[c + k] = y;
      a[k] += y;
    }
  return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace fia
