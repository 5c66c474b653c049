// Prefill Q4_0 GEMM on the 5th-generation tensor cores (sm_103a).
//
// C[M, N] = A[M, K] . W[K, N] with bf16 A, the weights W in the block layout of
// the C++ DeepSeek engine page (§2.2-§2.3: K rows of ceil(N/32) 18-byte
// blocks, each spanning 32 output columns) and fp32 accumulation; the page
// batches the prompt's tokens into one big matmul (§5.2).  Each weight is
// dequantised once per CTA tile to bf16: bf16_rn((q - 8) * d), the exact
// product rounded once (bf16x2 arithmetic on a split of d, see split_scale).
//
// Structure (one CTA per SM, persistent over 256 x 256 output tiles):
//  * warp 0, producer: TMA loads of A (64 K x 256 rows, 128-byte swizzle,
//    K-major) and of the raw Q4 tile (64 rows x 8 blocks) into rings;
//  * warps 2..9, dequant + epilogue: decode each raw block (one K row, 32
//    consecutive N) into 64 contiguous bytes of an MN-major, 128-byte-swizzled
//    bf16 B tile; after a tile's last K step, read the accumulators out of
//    tensor memory and store C;
//  * warp 1, MMA: allocates 512 tensor-memory columns (two 128 x 256 fp32
//    accumulators), issues tcgen05.mma (M = 128, N = 256, K = 16; two per K16
//    step, one per half of the tile's rows, both reading the same B tile) and
//    signals stage and accumulator readiness with tcgen05.commit.
// Every wait on an mbarrier is bounded: on a timeout the CTA records an error
// in the device status word, stops issuing work, drains the tensor core and
// frees its tensor memory before returning.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "q4_device.cuh"
#include "q4_kernels.h"

namespace q4 {
namespace gemm {

constexpr int BM = 256, BN = 256, BK = 64;
// CTAs of a thread-block cluster take the same rows of A and adjacent column
// tiles: each loads 1/kCluster of the A tile and multicasts it to all.
constexpr int kCluster = 1;
constexpr int kASlice = BM / kCluster;                 // A rows loaded per CTA
constexpr uint16_t kClusterMask = (1u << kCluster) - 1;
constexpr int kStagesA = 3;     // A ring: 3 x 32 KB
constexpr int kStagesRaw = 3;   // raw Q4 ring: 3 x 9 KB
constexpr int kStagesB = 3;     // dequantised B ring: 3 x 32 KB
constexpr int kABytes = BM * BK * 2;                   // 32768
constexpr int kBBytes = BN * BK * 2;                   // 32768
// A rows are BK * 2 bytes: one swizzle span of that width (128 or 64 bytes)
constexpr int kARowBytes = BK * 2;
static_assert(kARowBytes == 128 || kARowBytes == 64, "A rows must fill one swizzle span");
constexpr int kBarBytes = 512;
constexpr int kRawRowBytes = (BN / kBlockCols) * kBlockBytes;   // 144
constexpr int kRawBytes = BK * kRawRowBytes;           // 9216
constexpr int kDequantWarps = 8;
constexpr int kThreads = (2 + kDequantWarps) * 32;     // 320
constexpr uint32_t kTmemCols = 512;

struct Smem {
  uint32_t a, b, raw, bars, total;
};
__host__ __device__ constexpr Smem plan() {
  // A and B stages need 1024-byte alignment (swizzle atoms)
  return Smem{0, kStagesA * kABytes, kStagesA * kABytes + kStagesB * kBBytes,
              kStagesA * kABytes + kStagesB * kBBytes + kStagesRaw * kRawBytes,
              kStagesA * kABytes + kStagesB * kBBytes + kStagesRaw * kRawBytes + kBarBytes + 1024};
}

static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0 && plan().raw % 1024 == 0 &&
                  kRawBytes % 128 == 0 && plan().bars % 8 == 0,
              "TMA destinations need alignment");
static_assert((2 * kStagesA + 2 * kStagesRaw + 2 * kStagesB + 3) * 8 + 8 <= kBarBytes,
              "barrier region overflows");
static_assert(plan().total <= 227 * 1024, "shared memory plan exceeds the per-CTA limit");

// ---- tcgen05 / TMA wrappers ------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// The same box into the same shared offset of every CTA in `mask`; each
// destination's mbarrier (same offset) receives the bytes it got.
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const void* tmap, int c0, int c1,
                                               uint64_t* bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "h"(mask)
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
// Arrives once on the mbarrier at this offset in every CTA of `mask` when the
// MMAs issued so far by this thread are complete.
__device__ __forceinline__ void tc_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)), "h"(mask)
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

// Bounded wait that leaves the failure visible to the whole CTA.
__device__ __forceinline__ bool gwait(uint64_t* bar, uint32_t parity, volatile int* fail,
                                      unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*fail) return false;
  const unsigned long long t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 8; ++i)
      if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
    if (*fail) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *fail = 1;
      atomicOr(err, kDevErrTimeout);
      return false;
    }
  }
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
// wd decodes units wd * BK/32 + i, i < BK/32.  In unit u (row group u/2,
// parity u%2), lane = 8*s + r takes row 8*(u/2) + r and block 2*s + u%2.
//  * 16-byte stores are served eight lanes at a time; those eight lanes hold
//    eight different rows of one block, i.e. eight different chunk positions
//    of the 128-byte swizzle: no bank conflict.
//  * 32-bit raw reads: the rows are 36 words apart (4 banks), and the even
//    (odd) blocks start at words 0, 9, 18, 27 (4, 13, 22, 31) of a row, one
//    per residue mod 4: the 32 lanes hit 32 different banks.
__device__ __forceinline__ void dequant_stage(const uint8_t* raw, uint8_t* btile, int wd,
                                              int lane) {
#pragma unroll
  for (int i = 0; i < BK / 32; ++i) {
    const int u = wd * (BK / 32) + i;
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

// 32 consecutive accumulators of one row of C, columns col0 .. col0+31 (< N).
__device__ __forceinline__ void store_row32(const GemmParams& p, int row, int col0,
                                            const uint32_t (&acc)[32]) {
  // tensor-memory column 8t + s holds output column 8t + chunk_col(s)
  uint32_t v[32];
#pragma unroll
  for (int t = 0; t < 4; ++t)
#pragma unroll
    for (int s = 0; s < 8; ++s) v[8 * t + chunk_col(s)] = acc[8 * t + s];
  const size_t base = static_cast<size_t>(row) * p.N + col0;
  const bool whole = col0 + 32 <= p.N && (p.N & 7) == 0;
  if (p.c_dtype == 0) {
    float* dst = reinterpret_cast<float*>(p.C) + base;
    if (whole) {
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<uint4*>(dst + j) = make_uint4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    } else {
      for (int j = 0; j < 32 && col0 + j < p.N; ++j) dst[j] = __uint_as_float(v[j]);
    }
  } else {
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.C) + base;
    if (whole) {
#pragma unroll
      for (int j = 0; j < 32; j += 8) {
        uint4 o;
        o.x = bf16_bits(__uint_as_float(v[j])) | (bf16_bits(__uint_as_float(v[j + 1])) << 16);
        o.y = bf16_bits(__uint_as_float(v[j + 2])) | (bf16_bits(__uint_as_float(v[j + 3])) << 16);
        o.z = bf16_bits(__uint_as_float(v[j + 4])) | (bf16_bits(__uint_as_float(v[j + 5])) << 16);
        o.w = bf16_bits(__uint_as_float(v[j + 6])) | (bf16_bits(__uint_as_float(v[j + 7])) << 16);
        *reinterpret_cast<uint4*>(dst + j) = o;
      }
    } else {
      for (int j = 0; j < 32 && col0 + j < p.N; ++j)
        dst[j] = static_cast<uint16_t>(bf16_bits(__uint_as_float(v[j])));
    }
  }
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
    q4_gemm_tc_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr Smem L = plan();
  // 128-byte swizzled stages need 1024-byte aligned shared addresses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  static_assert(BK == 32 || BK == 64, "the dequant mapping covers BK = 32 or 64");
  uint8_t* sA = smem + L.a;
  uint8_t* sB = smem + L.b;
  uint8_t* sRaw = smem + L.raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* full_a = bars;                          // [kStagesA]
  uint64_t* empty_a = full_a + kStagesA;            // [kStagesA]
  uint64_t* full_raw = empty_a + kStagesA;          // [kStagesRaw]
  uint64_t* empty_raw = full_raw + kStagesRaw;      // [kStagesRaw]
  uint64_t* full_b = empty_raw + kStagesRaw;        // [kStagesB]
  uint64_t* empty_b = full_b + kStagesB;            // [kStagesB]
  uint64_t* tmem_full = empty_b + kStagesB;         // [1]
  uint64_t* tmem_empty = tmem_full + 1;             // [1]
  uint64_t* drain = tmem_empty + 1;                 // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_fail = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // work unit: a group of kCluster adjacent column tiles of one row tile; the
  // CTAs of a cluster take the group's tiles by rank
  const int rank = static_cast<int>(cluster_ctarank());
  const int tiles_m = (p.M + BM - 1) / BM;
  const int groups_n = (p.N + BN * kCluster - 1) / (BN * kCluster);
  const int ngroups = tiles_m * groups_n;
  const int first = blockIdx.x / kCluster, stride = gridDim.x / kCluster;
  const int ksteps = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesA; ++i) {
      mbar_init(&full_a[i], 1);
      mbar_init(&empty_a[i], kCluster);   // one commit from every CTA's MMA thread
    }
    for (int i = 0; i < kStagesRaw; ++i) {
      mbar_init(&full_raw[i], 1);
      mbar_init(&empty_raw[i], kDequantWarps);
    }
    for (int i = 0; i < kStagesB; ++i) {
      mbar_init(&full_b[i], kDequantWarps);
      mbar_init(&empty_b[i], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, kDequantWarps);
    mbar_init(drain, 1);
    *s_fail = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  // every CTA's barriers are initialised before any peer multicasts into them
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ================= producer =================
    if (lane == 0) {
      int ga = 0, gr = 0;   // loads issued into the A and raw rings
      for (int g = first; g < ngroups && !*s_fail; g += stride) {
        const int m0 = (g % tiles_m) * BM, n0 = ((g / tiles_m) * kCluster + rank) * BN;
        for (int ks = 0; ks < ksteps; ++ks) {
          const int sa = ga % kStagesA, sr = gr % kStagesRaw;
          // the stage is free once the MMAs of every CTA in the cluster read it
          if (ga >= kStagesA && !gwait(&empty_a[sa], ((ga / kStagesA) - 1) & 1, s_fail, p.err))
            break;
          mbar_arrive_expect_tx(&full_a[sa], kABytes);
          tma_load_2d_mc(sA + sa * kABytes + rank * kASlice * (BK * 2), &p.tmap_a, ks * BK,
                         m0 + rank * kASlice, &full_a[sa], kClusterMask);
          ++ga;
          if (gr >= kStagesRaw &&
              !gwait(&empty_raw[sr], ((gr / kStagesRaw) - 1) & 1, s_fail, p.err))
            break;
          mbar_arrive_expect_tx(&full_raw[sr], kRawBytes);
          tma_load_2d(sRaw + sr * kRawBytes, &p.tmap_b, (n0 / kBlockCols) * (kBlockBytes / 2),
                      ks * BK, &full_raw[sr]);
          ++gr;
        }
      }
      // No copy may still be writing shared memory when the CTA exits: wait
      // (bounded) for the last load issued into every stage.  On the normal
      // path these phases completed long ago.
      for (int g = ga - 1; g >= 0 && g >= ga - kStagesA; --g)
        (void)mbar_wait(&full_a[g % kStagesA], (g / kStagesA) & 1);
      for (int g = gr - 1; g >= 0 && g >= gr - kStagesRaw; --g)
        (void)mbar_wait(&full_raw[g % kStagesRaw], (g / kStagesRaw) & 1);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      int ga = 0, gb = 0, tl = 0;
      for (int g = first; g < ngroups && !*s_fail; g += stride, ++tl) {
        // the epilogue of the previous tile must have drained the accumulators
        if (tl > 0 && !gwait(tmem_empty, (tl - 1) & 1, s_fail, p.err)) break;
        tc_fence_after();
        bool ok = true;
        for (int ks = 0; ks < ksteps; ++ks, ++ga, ++gb) {
          const int sa = ga % kStagesA, sb = gb % kStagesB;
          ok = gwait(&full_a[sa], (ga / kStagesA) & 1, s_fail, p.err) &&
               gwait(&full_b[sb], (gb / kStagesB) & 1, s_fail, p.err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + sa * kABytes);
          const uint32_t b_base = smem_u32(sB + sb * kBBytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // B: MN-major, one K16 step = two 8-row swizzle atoms = 2048 bytes
            const uint64_t bdesc = smem_desc(b_base + kk * 2048, kBLbo, 1024, kSwizzle128);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              // A: K-major, 32 bytes per K16 step, 128 rows per accumulator
              const uint64_t adesc =
                  smem_desc(a_base + mt * 128 * kARowBytes + kk * 32, 16, kASbo, kASwizzle);
              tc_mma(tmem + mt * BN, adesc, bdesc, kIdesc, (ks > 0 || kk > 0) ? 1u : 0u);
            }
          }
          // frees the A stage (in every CTA of the cluster) and the B stage
          // once these MMAs are done
          tc_commit_mc(&empty_a[sa], kClusterMask);
          tc_commit(&empty_b[sb]);
        }
        if (!ok) break;
        tc_commit(tmem_full);
      }
      // every MMA this thread issued must be complete before the tensor memory
      // is freed and the CTA exits (bounded wait, also after a failure)
      tc_commit(drain);
      (void)mbar_wait(drain, 0);
    }
  } else {
    // ================= dequant + epilogue =================
    const int wd = warp - 2;   // 0..7
    int gr = 0, gb = 0, tl = 0;
    bool ok = true;
    for (int g = first; g < ngroups && ok && !*s_fail; g += stride, ++tl) {
      const int m0 = (g % tiles_m) * BM, n0 = ((g / tiles_m) * kCluster + rank) * BN;
      for (int ks = 0; ks < ksteps; ++ks, ++gr, ++gb) {
        const int sr = gr % kStagesRaw, sb = gb % kStagesB;
        int w = 1;
        if (lane == 0) {
          w = gwait(&full_raw[sr], (gr / kStagesRaw) & 1, s_fail, p.err) ? 1 : 0;
          if (w && gb >= kStagesB)
            w = gwait(&empty_b[sb], ((gb / kStagesB) - 1) & 1, s_fail, p.err) ? 1 : 0;
        }
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        if (!ok) break;
        dequant_stage(sRaw + sr * kRawBytes, sB + sb * kBBytes, wd, lane);
        fence_async_smem();   // the tensor core reads B through the async proxy
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full_b[sb]);
          mbar_arrive(&empty_raw[sr]);
        }
      }
      if (!ok) break;
      // ---- epilogue: accumulators -> C ----
      int w = 1;
      if (lane == 0) w = gwait(tmem_full, tl & 1, s_fail, p.err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, w, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const int q = warp & 3;   // the tensor-memory lane quarter this warp may access
      {
        const int mt = wd >> 2;   // warps 2..5 drain the first accumulator, 6..9 the second
        const int row = m0 + mt * 128 + q * 32 + lane;
#pragma unroll 1
        for (int cc = 0; cc < BN / 32; ++cc) {
          uint32_t v[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + mt * BN + cc * 32, v);
          const int col0 = n0 + cc * 32;
          if (row < p.M && col0 < p.N) store_row32(p, row, col0, v);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty);
    }
  }
  // everyone (the MMA thread after its drain) meets here before the tensor
  // memory is released
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // no CTA leaves while a peer may still multicast into it or arrive on its
  // barriers (every wait above is bounded, so all CTAs get here)
  cluster_sync();
}

}  // namespace gemm

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}

bool gemm_supported(int64_t M, int64_t N, int64_t K) {
  const int64_t nb = (N + 31) / 32;
  return M >= 1 && nb % 8 == 0 && K % 8 == 0 && K >= 1 && M <= (1LL << 30) && N <= (1LL << 30);
}

uint32_t gemm_smem_bytes() { return gemm::plan().total; }

cudaError_t launch_gemm(void* C, int c_dtype, const void* A, const void* B, int64_t M, int64_t N,
                        int64_t K, unsigned* err, int sms, cudaStream_t st) {
  using namespace gemm;
  auto encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  GemmParams p;
  // A: bf16 [M][K], box BK x kASlice rows (one CTA's share), swizzled rows
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 2)};
    const cuuint32_t box[2] = {BK, kASlice};
    const CUtensorMapSwizzle swz =
        (kARowBytes == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const cuuint32_t es[2] = {1, 1};
    if (encode(&p.tmap_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(A), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // raw Q4: uint16 [K][nb*9], box 72 halfwords (8 blocks) x 64 rows, no swizzle
  {
    const int64_t nb = (N + 31) / 32;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nb * 9), static_cast<cuuint64_t>(K)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nb * kBlockBytes)};
    const cuuint32_t box[2] = {72, BK};   // 8 blocks x BK rows
    const cuuint32_t es[2] = {1, 1};
    if (encode(&p.tmap_b, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(B), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  p.C = C;
  p.c_dtype = c_dtype;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.err = err;
  const uint32_t smem = plan().total;
  cudaError_t e = cudaFuncSetAttribute(gemm::q4_gemm_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent grid: as many clusters as can be resident at once (one CTA per
  // SM), at most one per work group
  static int resident[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (resident[dev] == 0) {
    cfg.gridDim = dim3(static_cast<unsigned>((sms / kCluster) * kCluster));
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, gemm::q4_gemm_tc_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    resident[dev] = n;
  }
  const int64_t groups = ((M + BM - 1) / BM) * ((N + BN * kCluster - 1) / (BN * kCluster));
  const int64_t clusters = groups < resident[dev] ? groups : resident[dev];
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * kCluster));
  e = cudaLaunchKernelEx(&cfg, gemm::q4_gemm_tc_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace q4
