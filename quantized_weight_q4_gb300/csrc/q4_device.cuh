// Device-side helpers shared by the sm_103a kernels: inline PTX for mbarriers,
// TMA tensor copies, programmatic dependent launch, clusters and packed fp32x2
// arithmetic.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace q4 {

constexpr int kBlockBytes = 18;   // sizeof(block_q4_0)
constexpr int kBlockCols = 32;    // weights per block

// Device status bits (mirrors Q4_DEVERR_* of the public header).
constexpr unsigned kDevErrIndex = 0x1u;
constexpr unsigned kDevErrTimeout = 0x2u;

// Upper bound of any spin-wait, in nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- GPU-scope acquire / release between CTAs ----------------------------
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// ticket = *p; *p += 1, with release semantics for this thread's earlier
// writes and those ordered before them (cumulative), and acquire semantics
// for its later reads, at GPU scope: one round trip, no full fences.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}
// *p += 1 with release semantics at GPU scope; nothing is returned, so the
// thread does not wait for the round trip.
__device__ __forceinline__ void red_add_release_gpu(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---- mbarrier -------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

// Like mbar_try_wait, but the thread may be suspended for up to `hint_ns`
// nanoseconds waiting for the phase instead of returning at once: a waiting
// warp then issues no instructions.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` to complete, giving up after kWaitLimitNs.
// Returns false on timeout; the caller records the error and stops.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) return false;
  }
}

// The wait every kernel uses on its pipeline barriers: returns true once phase
// `parity` of `bar` completes.  Gives up (returns false) if the CTA already
// failed, or after `limit_ns`: then it marks the CTA failed (`*fail`) and
// records Q4_DEVERR_TIMEOUT in the device status word, so that no thread of
// the CTA waits again and the host learns of it.  Between tries the thread is
// suspended in the barrier (hint 2 us) rather than spinning.
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* fail,
                                             unsigned* err,
                                             unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*fail) return false;
  const unsigned long long t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i)
      if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
    if (*fail) return false;
    if (globaltimer() - t0 > limit_ns) {
      *fail = 1;
      atomicOr(err, kDevErrTimeout);
      return false;
    }
  }
}

// ---- TMA tensor copy: a 3-D box of a tensor map -> shared, completes on an mbarrier
// (coordinates in elements; the tensor map must live in param/const/global space)
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// ---- programmatic dependent launch ------------------------------------------
// pdl_wait: blocks until every grid this grid depends on has completed and its
// memory operations are visible (a no-op when launched without the attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// pdl_launch_dependents: lets the next kernel on the stream begin launching.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- thread-block clusters ----------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives, then waits: shared-memory
// writes before it are visible to cluster peers after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address, in the cluster's shared window, of `local` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}
// Stores to a peer's shared memory (made visible by the next cluster barrier).
__device__ __forceinline__ void st_peer(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// ---- packed fp32x2 arithmetic (sm_100+) -------------------------------------
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 dup2(float x) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---- Q4_0 blocks in shared memory -------------------------------------------
// Reads the 18-byte block at byte offset `off` of a 4-byte-aligned shared
// row: returns the fp16 scale bits and the four 32-bit words of qs.
__device__ __forceinline__ void load_block_smem(const uint8_t* row, uint32_t off, uint32_t& dbits,
                                                uint32_t (&qs)[4]) {
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(row + (off & ~3u));
  const uint32_t w0 = wp[0], w1 = wp[1], w2 = wp[2], w3 = wp[3], w4 = wp[4];
  const uint32_t odd = off & 2u;   // block starts at 2 mod 4
  dbits = odd ? (w0 >> 16) : (w0 & 0xFFFFu);
  const uint32_t sh = odd ? 32u : 16u;
  qs[0] = __funnelshift_rc(w0, w1, sh);
  qs[1] = __funnelshift_rc(w1, w2, sh);
  qs[2] = __funnelshift_rc(w2, w3, sh);
  qs[3] = __funnelshift_rc(w3, w4, sh);
}

__device__ __forceinline__ float fp16_bits_to_f32(uint32_t bits) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits) {
  return __uint_as_float(bits << 16);
}

}  // namespace q4
