// tcgen05 / TMA helpers and the exact bf16 dequant of Q4_0 blocks into
// swizzled tensor-core tiles, shared by the GEMM forms of q4_gemm_sm103.cu and
// the few-row GEMM of q4_gemm_skinny.cu (sm_103a).
#pragma once

#include <cstdint>

#include "q4_device.cuh"
#include "q4_kernels.h"

namespace q4 {
namespace gemm {

constexpr int BN = 256, BK = 64;
constexpr int kBBytes = BN * BK * 2;                            // 32768
constexpr int kRawRowBytes = (BN / kBlockCols) * kBlockBytes;   // 144
constexpr int kRawBytes = BK * kRawRowBytes;                    // 9216
// A rows are BK * 2 bytes: one swizzle span of that width (128 or 64 bytes)
constexpr int kARowBytes = BK * 2;
static_assert(kARowBytes == 128 || kARowBytes == 64, "A rows must fill one swizzle span");
constexpr int kMaxSplit = 16;   // non-portable thread-block cluster size limit

// ---- tcgen05 / TMA wrappers ------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// D[tmem] (+)= A[smem desc] . B[smem desc]
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// TMA tensor store of a 2-D box from shared memory (1024-byte aligned for a
// 128-byte swizzle) to global memory, in this thread's current bulk
// async-group.  The box may reach past the tensor's end (clipped there); its
// start must lie inside the tensor.
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}
// Closes this thread's current bulk async-group.
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's bulk async-groups still read their
// shared-memory sources (the sources may then be overwritten).
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until at most N of this thread's bulk async-groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// 32 lanes x 32 columns of 32-bit accumulators: thread i gets its lane's 32.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (16-byte units), descriptor version 1, swizzle mode in bits 61-63
// (2 = 128-byte swizzle, 4 = 64-byte swizzle).
constexpr uint64_t kSwizzle128 = 2, kSwizzle64 = 4;
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint64_t swizzle) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= swizzle << 61;
  return d;
}
// A (K-major): rows of kARowBytes, 8-row swizzle atoms kARowBytes * 8 apart.
constexpr uint64_t kASwizzle = (kARowBytes == 128) ? kSwizzle128 : kSwizzle64;
constexpr uint32_t kASbo = kARowBytes * 8;

// Instruction descriptor of kind::f16: fp32 D, bf16 A and B, A K-major,
// B MN-major, N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (1u << 16) |
                            (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);

// Bounded wait that leaves the failure visible to the whole CTA (bounded_wait).
__device__ __forceinline__ bool gwait(uint64_t* bar, uint32_t parity, volatile int* fail,
                                      unsigned* err) {
  return bounded_wait(bar, parity, fail, err);
}

// ---- dequant of one raw stage into an MN-major swizzled bf16 B tile --------
// B tile layout (K = BK rows, N = 256): 128-byte swizzle atoms of 8 K rows x
// 64 N; atom (na, ka) at (na * BK/8 + ka) * 1024 bytes; inside it K row kr is
// 128 bytes at kr * 128 with 16-byte chunk c stored at chunk c ^ kr.
// Descriptor: leading byte offset (between atoms along N) BK/8 * 1024, stride
// byte offset (between atoms along K) 1024.
constexpr uint32_t kBLbo = (BK / 8) * 1024;
__device__ __forceinline__ uint32_t b_offset(int k, int n) {
  const int ka = k >> 3, kr = k & 7, na = n >> 6, c = (n & 63) >> 3;
  return static_cast<uint32_t>((na * (BK / 8) + ka) * 1024 + kr * 128 + ((c ^ kr) << 4));
}

// bf16x2 arithmetic, round to nearest even.
__device__ __forceinline__ uint32_t bf2_add(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Column order inside each 8-column chunk of a B tile: the decode packs
// nibbles j and j + 4 of a 32-bit word into one bf16 pair, so slot s of a
// chunk holds column chunk_col(s) of it.  The epilogue applies the inverse.
__host__ __device__ constexpr int chunk_col(int s) { return (s >> 1) + 4 * (s & 1); }

// Scale of one block for the bf16 decode: d = dh + dl with dh the bf16
// truncation of d (toward zero) and dl the remaining (at most 3) low bits of
// the fp16 significand, carrying d's sign also when it is zero.  Non-finite d
// keeps dh = d (a canonical NaN for NaN) and dl = signed zero.
__device__ __forceinline__ void split_scale(uint32_t dbits16, uint32_t& dh2, uint32_t& dl2) {
  const float d = fp16_bits_to_f32(dbits16);
  const uint32_t db = __float_as_uint(d);
  const bool finite = (db & 0x7F800000u) != 0x7F800000u;
  const uint32_t hb = (d != d) ? 0x7FC00000u : (db & 0xFFFF0000u);
  const float dl = finite ? d - __uint_as_float(hb) : 0.0f;   // exact: at most 3 bits
  const uint32_t lb = __float_as_uint(dl) | (db & 0x80000000u);
  const uint32_t h16 = hb >> 16, l16 = lb >> 16;                // dl is exact in bf16
  dh2 = h16 | (h16 << 16);
  dl2 = l16 | (l16 << 16);
}

// bf16_rn((q - 8) * d) for nibbles j (low half) and j + 4 (high half) of w:
// x = bf16(128 + q) from the bits, q - 8 exactly by one add, (q - 8) * dl
// exactly (at most 7 significant bits), then (q - 8) * dh plus that, rounded
// once.
__device__ __forceinline__ uint32_t decode_pair(uint32_t w_shifted, uint32_t dh2, uint32_t dl2) {
  const uint32_t x = (w_shifted & 0x000F000Fu) | 0x43004300u;   // 128 + q, 128 + q'
  const uint32_t xq = bf2_add(x, 0xC308C308u);                    // - 136
  return bf2_fma(xq, dh2, bf2_mul(xq, dl2));
}

// A stage is BK/8 row groups x 2 parities of (8 rows x 4 blocks) units; warp
// wd decodes units wd * UPW + i, i < UPW.  In unit u (row group u/2,
// parity u%2), lane = 8*s + r takes row 8*(u/2) + r and block 2*s + u%2.
//  * 16-byte stores are served eight lanes at a time; those eight lanes hold
//    eight different rows of one block, i.e. eight different chunk positions
//    of the 128-byte swizzle: no bank conflict.
//  * 32-bit raw reads: the rows are 36 words apart (4 banks), and the even
//    (odd) blocks start at words 0, 9, 18, 27 (4, 13, 22, 31) of a row, one
//    per residue mod 4: the 32 lanes hit 32 different banks.
template <int UPW>
__device__ __forceinline__ void dequant_stage(const uint8_t* raw, uint8_t* btile, int wd,
                                              int lane) {
#pragma unroll
  for (int i = 0; i < UPW; ++i) {
    const int u = wd * UPW + i;
    const int k = (u >> 1) * 8 + (lane & 7);
    const int b = 2 * (lane >> 3) + (u & 1);
    uint32_t dbits, qs[4];
    load_block_smem(raw + k * kRawRowBytes, static_cast<uint32_t>(b * kBlockBytes), dbits, qs);
    uint32_t dh2, dl2;
    split_scale(dbits, dh2, dl2);
    // word t holds columns 8t .. 8t+7 of the block (nibble j = column 8t + j);
    // it becomes chunk t, slots in chunk_col order
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t w = qs[t];
      const uint4 o = make_uint4(decode_pair(w, dh2, dl2), decode_pair(w >> 4, dh2, dl2),
                                 decode_pair(w >> 8, dh2, dl2), decode_pair(w >> 12, dh2, dl2));
      *reinterpret_cast<uint4*>(btile + b_offset(k, b * 32 + t * 8)) = o;
    }
  }
}

__device__ __forceinline__ uint32_t bf16_bits(float v) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

}  // namespace gemm
}  // namespace q4
