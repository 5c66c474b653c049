// Q4_0 GEMM on the 5th-generation tensor cores (sm_103a).
//
// C[M, N] = A[M, K] . W[K, N] with bf16 A, the weights W in the block layout of
// the C++ DeepSeek engine page (§2.2-§2.3: K rows of ceil(N/32) 18-byte
// blocks, each spanning 32 output columns) and fp32 accumulation; the page
// batches the prompt's tokens into one big matmul (§5.2).  Each weight is
// dequantised once per CTA tile to bf16: bf16_rn((q - 8) * d), the exact
// product rounded once (bf16x2 arithmetic on a split of d, see split_scale).
//
// One kernel template, two forms:
//  * prefill (MT = 2): one CTA per SM, persistent over 256 x 256 output tiles;
//  * small M (MT = 1, SPLIT): 128 x 256 output tiles, each split along K over
//    the S CTAs of a thread-block cluster; the partial sums meet in shared
//    memory over DSMEM and are added in rank order (deterministic).
// Roles inside a CTA:
//  * warp 0, producer: TMA loads of A (64 K x 128*MT rows, 128-byte swizzle,
//    K-major) and of the raw Q4 tile (64 rows x 8 blocks) into rings;
//  * warps 2 .. DW+1, dequant + epilogue: decode each raw block (one K row,
//    32 consecutive N) into 64 bytes of an MN-major, 128-byte-swizzled bf16 B
//    tile; after a tile's last K step, read the accumulators out of tensor
//    memory and store C (or push the partial sums to their owner);
//  * warp 1, MMA: allocates MT*256 tensor-memory columns (MT accumulators of
//    128 x 256 fp32), issues tcgen05.mma (M = 128, N = 256, K = 16; MT per
//    K16 step, all reading the same B tile) and signals stage and
//    accumulator readiness with tcgen05.commit.
// Every wait on an mbarrier is bounded: on a timeout the CTA records an error
// in the device status word, stops issuing work, drains the tensor core and
// its copies and frees its tensor memory before returning.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "q4_device.cuh"
#include "q4_kernels.h"
#include "q4_tc_core.cuh"

namespace q4 {
namespace gemm {


// Compile-time shape of one kernel form.
template <int MT, int DW, bool SPLIT>
struct Cfg {
  static constexpr int kBM = 128 * MT;                 // rows of A per tile
  static constexpr int kThreads = (2 + DW) * 32;
  // ring depths: the prefill form re-reads A from L2 for every column tile
  // and needs its A ring deep; the small-M form streams each weight once
  // from HBM and needs its raw ring deep
  static constexpr int kStagesA = (MT == 2) ? 3 : 4;   // 32 KB or 16 KB per stage
  static constexpr int kStagesB = 3;                   // 32 KB per stage
  static constexpr int kStagesRaw = (MT == 2) ? 3 : 6; // 9 KB per stage
  static constexpr int kABytes = kBM * BK * 2;
  static constexpr uint32_t kTmemCols = MT * BN;
  // with kGroups > 1 the dequant warps form groups that take alternate
  // stages; both forms measured faster with one group (every warp on every
  // stage).  Dequant units (8 rows x 4 blocks) per warp and stage follow.
  static constexpr int kGroups = 1;
  static constexpr int kGroupWarps = DW / kGroups;
  static constexpr int kUnitsPerWarp = (BK / 4) / kGroupWarps;
  // epilogue: the DW/4 warps of one tensor-memory lane quarter split the
  // MT * BN accumulator columns
  static constexpr int kEpiCols = MT * BN / (DW / 4);
  // shared memory plan; A and B stages need 1024-byte alignment
  static constexpr uint32_t kOffB = kStagesA * kABytes;
  static constexpr uint32_t kOffRaw = kOffB + kStagesB * kBBytes;
  static constexpr uint32_t kOffBars = kOffRaw + kStagesRaw * kRawBytes;
  static constexpr uint32_t kBarBytes = 256;
  static constexpr uint32_t kSmemBytes = kOffBars + kBarBytes + 1024;
  static_assert(MT == 1 || (MT == 2 && !SPLIT), "forms: prefill (MT 2) and split small M (MT 1)");
  static_assert(kUnitsPerWarp >= 1 && (BK / 4) % kGroupWarps == 0 && DW % 4 == 0 &&
                    DW % kGroups == 0,
                "dequant warps");
  static_assert(kEpiCols % 32 == 0 && BN % kEpiCols == 0, "epilogue column split");
  static_assert(kABytes % 1024 == 0 && kOffRaw % 1024 == 0 && kRawBytes % 128 == 0,
                "TMA destinations need alignment");
  static_assert((2 * kStagesA + 2 * kStagesRaw + 2 * kStagesB + 3) * 8 + 8 <= kBarBytes,
                "barrier region overflows");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory plan exceeds the per-CTA limit");
};

// Split form: the partial sums of a 128 x 256 tile travel as rows of 32
// columns, padded to 36 floats (16-byte aligned, conflict-free 16-byte
// stores of eight consecutive rows).  Owner of 32-column chunk c: rank c % S.
constexpr int kRedRowFloats = 36;
__host__ __device__ constexpr uint32_t red_bytes(int S, int rows) {
  return static_cast<uint32_t>(((BN / 32 + S - 1) / S) * S * rows * kRedRowFloats * 4);
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


// Four consecutive fp32 results of one row of C, columns col .. col+3.
__device__ __forceinline__ void store_group4(const GemmParams& p, int row, int col, float4 v) {
  if (row >= p.M || col >= p.N) return;
  const size_t base = static_cast<size_t>(row) * p.N + col;
  const bool whole = col + 4 <= p.N && (p.N & 3) == 0;
  if (p.c_dtype == 0) {
    float* dst = reinterpret_cast<float*>(p.C) + base;
    if (whole) {
      *reinterpret_cast<float4*>(dst) = v;
    } else {
      const float f[4] = {v.x, v.y, v.z, v.w};
      for (int j = 0; j < 4 && col + j < p.N; ++j) dst[j] = f[j];
    }
  } else {
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.C) + base;
    if (whole) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(bf16_bits(v.x) | (bf16_bits(v.y) << 16),
                                                  bf16_bits(v.z) | (bf16_bits(v.w) << 16));
    } else {
      const float f[4] = {v.x, v.y, v.z, v.w};
      for (int j = 0; j < 4 && col + j < p.N; ++j) dst[j] = static_cast<uint16_t>(bf16_bits(f[j]));
    }
  }
}

// A unit of work: one output tile (rows m0.., columns n0..) over K steps
// [kb, ke) of BK rows.  Prefill form: `role` 0 stores the tile; in the tail,
// 1 is the part holding the tile's last K step (it adds the earlier parts,
// those of CTAs [c1, c1 + nc), and stores), 2 an earlier part (it writes its
// partial tile for that one).
struct Work {
  int m0, n0, kb, ke;
  int role, c1, nc;
};

// Start of the tail's part c: the tail's K steps [0, T) cut into `parts`
// equal ranges.
__host__ __device__ __forceinline__ int64_t tail_start(int64_t T, int parts, int c) {
  return static_cast<int64_t>(c) * T / parts;
}

// Prefill form: the it-th unit of CTA c of a grid of G (false when there is
// none).  Tiles c, c + G, ... below full_tiles over all K, then the pieces
// of CTA c's range of the tail, one per tile it crosses (at most two: a
// range is never longer than a tile), the later tile's first.  So a CTA's
// earlier part (role 2, which never waits) comes before its last-step part
// (role 1), and a last-step part waits only for CTAs of lower index, which
// start no later than it does: no chain of waits, and no wait on a CTA that
// cannot start.  Host and device share this function (the host lists the
// units for tests).
template <int MT>
__host__ __device__ __forceinline__ bool prefill_unit(int M, int N, int K, int full_tiles,
                                                      int tail_ctas, int c, int G, int it,
                                                      Work& w) {
  constexpr int kBM = 128 * MT;
  const int tiles_m = (M + kBM - 1) / kBM;
  const int tiles_n = (N + BN - 1) / BN;
  const int ksteps = (K + BK - 1) / BK;
  int tile;
  w.role = 0;
  w.c1 = 0;
  w.nc = 0;
  const int mine = full_tiles > c ? (full_tiles - c + G - 1) / G : 0;
  if (it < mine) {
    tile = c + it * G;
    w.kb = 0;
    w.ke = ksteps;
  } else {
    if (c >= tail_ctas) return false;
    const int64_t T = static_cast<int64_t>(tiles_m * tiles_n - full_tiles) * ksteps;
    const int64_t lo = tail_start(T, tail_ctas, c), hi = tail_start(T, tail_ctas, c + 1);
    if (lo >= hi) return false;
    const int64_t t = (hi - 1) / ksteps - (it - mine);   // tile of the tail, later first
    const int64_t t0 = t * ksteps;
    if (t0 + ksteps <= lo) return false;
    w.kb = static_cast<int>((lo > t0 ? lo : t0) - t0);
    w.ke = static_cast<int>((hi < t0 + ksteps ? hi : t0 + ksteps) - t0);
    tile = full_tiles + static_cast<int>(t);
    if (w.kb > 0 && w.ke == ksteps) {
      // the parts of CTAs c1 .. c - 1 hold this tile's earlier K steps
      w.role = 1;
      int e = c - 1;
      while (e > 0 && tail_start(T, tail_ctas, e) > t0) --e;
      w.c1 = e;
      w.nc = c - e;
    } else if (w.ke < ksteps) {
      w.role = 2;
    }
  }
  if (tile >= tiles_m * tiles_n) return false;
  w.m0 = (tile % tiles_m) * kBM;
  w.n0 = (tile / tiles_m) * BN;
  return true;
}

// The it-th unit of this CTA (false when there is none): the prefill form's
// (above), or for the split form the one tile of the cluster, this CTA's
// share of K (cluster rank = blockIdx.x % S).
template <int MT, bool SPLIT>
__device__ __forceinline__ bool work_item(const GemmParams& p, int it, Work& w) {
  if (!SPLIT)
    return prefill_unit<MT>(p.M, p.N, p.K, p.full_tiles, p.tail_ctas, blockIdx.x, gridDim.x, it,
                            w);
  constexpr int kBM = 128 * MT;
  const int tiles_m = (p.M + kBM - 1) / kBM;
  const int tiles_n = (p.N + BN - 1) / BN;
  const int ksteps = (p.K + BK - 1) / BK;
  w.role = 0;
  w.c1 = 0;
  w.nc = 0;
  if (it > 0) return false;
  const int tile = blockIdx.x / p.nsplit;
  const int s = blockIdx.x % p.nsplit;
  w.kb = s * ksteps / p.nsplit;
  w.ke = (s + 1) * ksteps / p.nsplit;
  if (tile >= tiles_m * tiles_n) return false;
  w.m0 = (tile % tiles_m) * kBM;
  w.n0 = (tile / tiles_m) * BN;
  return true;
}

// Prefill tail: the partial tile of CTA c's part, the tensor-memory image of
// 128 lanes x cols fp32 stored as float4 [cols / 32][8][128]: element (lane
// r, column c + 4j + i) of 32-column chunk c at float4 (c / 32 * 8 + j) * 128
// + r, component i, so that a warp's 32 lanes (consecutive rows) move 512
// contiguous bytes per access.
__device__ __forceinline__ float4* tail_slot(const GemmParams& p, int c, int cols) {
  return reinterpret_cast<float4*>(p.part + static_cast<size_t>(c) * 128 * cols);
}

// Waits (bounded, one thread) until the parts of CTAs [c1, c1 + nc) have
// released their partial tiles.  On a timeout it marks the CTA failed and
// records Q4_DEVERR_TIMEOUT.
__device__ __forceinline__ bool wait_parts(const GemmParams& p, int c1, int nc,
                                           volatile int* fail) {
  const unsigned long long t0 = globaltimer();
  for (int i = 0; i < nc; ++i) {
    while (ld_acquire_gpu(&p.tickets[c1 + i]) == 0u) {
      if (*fail || globaltimer() - t0 > kWaitLimitNs) {
        if (!*fail) {
          *fail = 1;
          atomicOr(p.err, kDevErrTimeout);
        }
        return false;
      }
      __nanosleep(256);
    }
  }
  return true;
}

// acc (32 accumulators of lane `r`, tensor-memory columns c .. c+31, fp32
// bits) += the partials of CTAs c1, c1 + 1, ... in that order (K order).
template <int COLS>
__device__ __forceinline__ void add_parts(const GemmParams& p, int c1, int nc, int r, int c,
                                          uint32_t (&acc)[32]) {
  for (int i = 0; i < nc; ++i) {
    const float4* src = tail_slot(p, c1 + i, COLS) + (c / 32) * 8 * 128 + r;
    float4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __ldcg(src + j * 128);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      acc[4 * j] = __float_as_uint(__uint_as_float(acc[4 * j]) + v[j].x);
      acc[4 * j + 1] = __float_as_uint(__uint_as_float(acc[4 * j + 1]) + v[j].y);
      acc[4 * j + 2] = __float_as_uint(__uint_as_float(acc[4 * j + 2]) + v[j].z);
      acc[4 * j + 3] = __float_as_uint(__uint_as_float(acc[4 * j + 3]) + v[j].w);
    }
  }
}

// 16 bytes global -> shared, asynchronous, through L2 only (cp.async.cg).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The last-step part of a tail tile, TMA epilogue: one lane's rows of the
// earlier parts' partial tiles, staged in shared memory two (chunk, part) pairs ahead
// of their use, so that the L2 round trips overlap.  Pair k = chunk k / nc of
// the warp's columns, part k % nc, lands in slot k % 3 of the warp's 12 KB
// (float4 [3][8][32]); each lane copies and later reads only its own row, so
// no lane waits for another.  The buffer is the A ring, idle by then: a
// last-step part is always its CTA's last unit.
template <int COLS>
struct PartPrefetch {
  const GemmParams& p;
  float4* buf;
  int c1, nc, r, lane, chunk0, npairs;
  __device__ __forceinline__ void issue(int k) {
    if (k < npairs) {
      const int ch = k / nc, i = k - ch * nc;
      const float4* src = tail_slot(p, c1 + i, COLS) + (chunk0 + ch) * 8 * 128 + r;
      float4* dst = buf + (k % 3) * 256 + lane;
#pragma unroll
      for (int j = 0; j < 8; ++j) cp_async16(dst + j * 32, src + j * 128);
    }
    cp_async_commit();   // empty groups keep the count of groups uniform
  }
  // acc += the later parts' rows of chunk `ch`, in part (K) order
  __device__ __forceinline__ void add(int ch, uint32_t (&acc)[32]) {
    for (int i = 0; i < nc; ++i) {
      const int k = ch * nc + i;
      issue(k + 2);
      cp_async_wait<2>();   // pair k has landed
      const float4* src = buf + (k % 3) * 256 + lane;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 v = src[j * 32];
        acc[4 * j] = __float_as_uint(__uint_as_float(acc[4 * j]) + v.x);
        acc[4 * j + 1] = __float_as_uint(__uint_as_float(acc[4 * j + 1]) + v.y);
        acc[4 * j + 2] = __float_as_uint(__uint_as_float(acc[4 * j + 2]) + v.z);
        acc[4 * j + 3] = __float_as_uint(__uint_as_float(acc[4 * j + 3]) + v.w);
      }
    }
  }
};

// ---------------------------------------------------------------------------
template <int MT, int DW, bool SPLIT>
__global__ void __launch_bounds__(Cfg<MT, DW, SPLIT>::kThreads, 1)
    q4_gemm_tc_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<MT, DW, SPLIT>;
  constexpr int kStagesA = C::kStagesA, kStagesB = C::kStagesB, kStagesRaw = C::kStagesRaw;
  extern __shared__ uint8_t smem_raw[];
  // swizzled stages need 1024-byte aligned shared addresses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::kOffB;
  uint8_t* sRaw = smem + C::kOffRaw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
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

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesA; ++i) {
      mbar_init(&full_a[i], 1);
      mbar_init(&empty_a[i], 1);
    }
    for (int i = 0; i < kStagesRaw; ++i) {
      mbar_init(&full_raw[i], 1);
      mbar_init(&empty_raw[i], C::kGroupWarps);
    }
    for (int i = 0; i < kStagesB; ++i) {
      mbar_init(&full_b[i], C::kGroupWarps);
      mbar_init(&empty_b[i], 1);
    }
    mbar_init(tmem_full, 1);
    mbar_init(tmem_empty, DW);
    mbar_init(drain, 1);
    *s_fail = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ================= producer =================
    if (lane == 0) {
      int ga = 0, gr = 0;   // loads issued into the A and raw rings
      Work w;
      for (int it = 0; work_item<MT, SPLIT>(p, it, w) && !*s_fail; ++it) {
        for (int ks = w.kb; ks < w.ke; ++ks) {
          const int sa = ga % kStagesA, sr = gr % kStagesRaw;
          if (ga >= kStagesA && !gwait(&empty_a[sa], ((ga / kStagesA) - 1) & 1, s_fail, p.err))
            break;
          // the A box holds p.a_rows rows (the tile's rows, rounded up to 16);
          // the MMA also reads the stage's remaining rows, whose accumulator
          // rows are never stored
          mbar_arrive_expect_tx(&full_a[sa], static_cast<uint32_t>(p.a_rows * kARowBytes));
          tma_load_2d(sA + sa * C::kABytes, &p.tmap_a, ks * BK, w.m0, &full_a[sa]);
          ++ga;
          if (gr >= kStagesRaw &&
              !gwait(&empty_raw[sr], ((gr / kStagesRaw) - 1) & 1, s_fail, p.err))
            break;
          mbar_arrive_expect_tx(&full_raw[sr], kRawBytes);
          tma_load_2d(sRaw + sr * kRawBytes, &p.tmap_b, (w.n0 / kBlockCols) * (kBlockBytes / 2),
                      ks * BK, &full_raw[sr]);
          ++gr;
        }
      }
      // No copy may still be writing shared memory when the CTA exits or the
      // rings are reused: wait (bounded) for the last load issued into every
      // stage.  On the normal path these phases completed long ago.
      for (int g = ga - 1; g >= 0 && g >= ga - kStagesA; --g)
        (void)mbar_wait(&full_a[g % kStagesA], (g / kStagesA) & 1);
      for (int g = gr - 1; g >= 0 && g >= gr - kStagesRaw; --g)
        (void)mbar_wait(&full_raw[g % kStagesRaw], (g / kStagesRaw) & 1);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      int ga = 0, gb = 0;
      Work w;
      for (int it = 0; work_item<MT, SPLIT>(p, it, w) && !*s_fail; ++it) {
        // the epilogue of the previous tile must have drained the accumulators
        if (it > 0 && !gwait(tmem_empty, (it - 1) & 1, s_fail, p.err)) break;
        tc_fence_after();
        bool ok = true;
        for (int ks = w.kb; ks < w.ke; ++ks, ++ga, ++gb) {
          const int sa = ga % kStagesA, sb = gb % kStagesB;
          ok = gwait(&full_a[sa], (ga / kStagesA) & 1, s_fail, p.err) &&
               gwait(&full_b[sb], (gb / kStagesB) & 1, s_fail, p.err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + sa * C::kABytes);
          const uint32_t b_base = smem_u32(sB + sb * kBBytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // B: MN-major, one K16 step = two 8-row swizzle atoms = 2048 bytes
            const uint64_t bdesc = smem_desc(b_base + kk * 2048, kBLbo, 1024, kSwizzle128);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
              // A: K-major, 32 bytes per K16 step, 128 rows per accumulator
              const uint64_t adesc =
                  smem_desc(a_base + mt * 128 * kARowBytes + kk * 32, 16, kASbo, kASwizzle);
              tc_mma(tmem + mt * BN, adesc, bdesc, kIdesc, (ks > w.kb || kk > 0) ? 1u : 0u);
            }
          }
          // frees the A and B stages once these MMAs are done
          tc_commit(&empty_a[sa]);
          tc_commit(&empty_b[sb]);
        }
        if (!ok) break;
        tc_commit(tmem_full);
      }
      // every MMA this thread issued must be complete before the tensor memory
      // is freed, the rings are reused or the CTA exits (bounded wait, also
      // after a failure)
      tc_commit(drain);
      (void)mbar_wait(drain, 0);
    }
  } else {
    // ================= dequant + epilogue =================
    const int wd = warp - 2;   // 0 .. DW-1
    const int q = warp & 3;    // the tensor-memory lane quarter this warp may access
    const int grp = wd / C::kGroupWarps, wg = wd % C::kGroupWarps;
    int gr = 0, gb = 0;
    bool ok = true;
    Work w;
    for (int it = 0; ok && work_item<MT, SPLIT>(p, it, w) && !*s_fail; ++it) {
      for (int ks = w.kb; ks < w.ke; ++ks, ++gr, ++gb) {
        if (gb % C::kGroups != grp) continue;   // the other group's stage
        const int sr = gr % kStagesRaw, sb = gb % kStagesB;
        int v = 1;
        if (lane == 0) {
          v = gwait(&full_raw[sr], (gr / kStagesRaw) & 1, s_fail, p.err) ? 1 : 0;
          if (v && gb >= kStagesB)
            v = gwait(&empty_b[sb], ((gb / kStagesB) - 1) & 1, s_fail, p.err) ? 1 : 0;
        }
        ok = __shfl_sync(0xffffffffu, v, 0) != 0;
        if (!ok) break;
        dequant_stage<C::kUnitsPerWarp>(sRaw + sr * kRawBytes, sB + sb * kBBytes, wg, lane);
        fence_async_smem();   // the tensor core reads B through the async proxy
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full_b[sb]);
          mbar_arrive(&empty_raw[sr]);
        }
      }
      if (!ok) break;
      int v = 1;
      if (lane == 0) v = gwait(tmem_full, it & 1, s_fail, p.err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, v, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      if (SPLIT) break;   // the split form's epilogue follows below
      if (w.role == 2) {
        // ---- a later part of a tail tile: its partial tile, released once
        //      every warp's stores are done (after the meet below) ----
        float4* slot = tail_slot(p, blockIdx.x, C::kTmemCols);
        const int c0 = (wd >> 2) * C::kEpiCols;
        const int r = q * 32 + lane;
#pragma unroll 1
        for (int c = c0; c < c0 + C::kEpiCols; c += 32) {
          uint32_t acc[32];
          tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, acc);
          float4* dst = slot + (c / 32) * 8 * 128 + r;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            __stcg(dst + j * 128, make_float4(__uint_as_float(acc[4 * j]), __uint_as_float(acc[4 * j + 1]),
                                        __uint_as_float(acc[4 * j + 2]),
                                        __uint_as_float(acc[4 * j + 3])));
        }
      } else {
      // the last-step part of a tail tile adds the earlier parts' partial tiles
      bool add = false;
      if (w.role == 1) {
        int v = 1;
        if (lane == 0) v = wait_parts(p, w.c1, w.nc, s_fail) ? 1 : 0;
        add = __shfl_sync(0xffffffffu, v, 0) != 0;
      }
      // ---- epilogue: accumulators -> C ----
      {
        // column c of the MT x BN accumulator columns is column c % BN of
        // accumulator c / BN; the warps of one lane quarter split them
        const int c0 = (wd >> 2) * C::kEpiCols;
        const int mt = c0 / BN;
        const int row0 = w.m0 + mt * 128 + q * 32;   // the warp's 32 rows
        const int row = row0 + lane;
        if (p.use_tma_c) {
          // Through shared memory and TMA tensor stores: boxes of 32 rows x
          // 128 bytes (32 fp32 or 64 bf16 columns), 128-byte swizzled (each
          // lane writes its row's 16-byte chunks at chunk ^ (row % 8): no bank
          // conflicts), two in flight per warp.  The staging boxes sit in the
          // B ring, which no MMA reads and no dequant writes between tiles.
          uint8_t* stg = sB + wd * 8192;
          const int box_cols = p.c_dtype == 0 ? 32 : 64;
          static_assert(SPLIT || kStagesA * C::kABytes >= DW * 12288, "partial staging in the A ring");
          PartPrefetch<C::kTmemCols> pf{p, reinterpret_cast<float4*>(sA + wd * 12288), w.c1,
                                        w.nc, q * 32 + lane, lane, c0 / 32,
                                        add ? (C::kEpiCols / 32) * w.nc : 0};
          if (add) {
            pf.issue(0);
            pf.issue(1);
          }
          int nbox = 0;
#pragma unroll 1
          for (int c = c0; c < c0 + C::kEpiCols; c += box_cols, ++nbox) {
            uint8_t* box = stg + (nbox & 1) * 4096;
            if (nbox >= 2) {   // the store issued from this box two boxes ago has read it
              if (lane == 0) bulk_wait_read<1>();
              __syncwarp();
            }
#pragma unroll 1
            for (int h = 0; h < box_cols / 32; ++h) {
              uint32_t acc[32], v[32];
              tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c + 32 * h, acc);
              if (add) pf.add((c - c0) / 32 + h, acc);
              // tensor-memory column 8t + s holds output column 8t + chunk_col(s)
#pragma unroll
              for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int s8 = 0; s8 < 8; ++s8) v[8 * t + chunk_col(s8)] = acc[8 * t + s8];
              uint8_t* rowp = box + lane * 128;
              if (p.c_dtype == 0) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7)) << 4)) =
                      make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint4 o;
                  o.x = bf16_bits(__uint_as_float(v[8 * j])) |
                        (bf16_bits(__uint_as_float(v[8 * j + 1])) << 16);
                  o.y = bf16_bits(__uint_as_float(v[8 * j + 2])) |
                        (bf16_bits(__uint_as_float(v[8 * j + 3])) << 16);
                  o.z = bf16_bits(__uint_as_float(v[8 * j + 4])) |
                        (bf16_bits(__uint_as_float(v[8 * j + 5])) << 16);
                  o.w = bf16_bits(__uint_as_float(v[8 * j + 6])) |
                        (bf16_bits(__uint_as_float(v[8 * j + 7])) << 16);
                  *reinterpret_cast<uint4*>(rowp + (((4 * h + j) ^ (lane & 7)) << 4)) = o;
                }
              }
            }
            fence_async_smem();   // the TMA store reads the box through the async proxy
            __syncwarp();
            const int col = w.n0 + (c - mt * BN);
            if (lane == 0) {
              if (row0 < p.M && col < p.N) tma_store_2d(&p.tmap_c, box, col, row0);
              bulk_commit();
            }
          }
          // the boxes are read before the B ring takes the next tile's stages
          if (lane == 0) bulk_wait_read<0>();
          if (add) cp_async_wait<0>();   // no copy into the A ring outlives the unit
          __syncwarp();
        } else {
#pragma unroll 1
          for (int c = c0; c < c0 + C::kEpiCols; c += 32) {
            uint32_t acc[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, acc);
            if (add) add_parts<C::kTmemCols>(p, w.c1, w.nc, row - w.m0 - mt * 128, c, acc);
            const int col0 = w.n0 + (c - mt * BN);
            if (row < p.M && col0 < p.N) store_row32(p, row, col0, acc);
          }
        }
      }
      }   // role 0 or 1
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tmem_empty);
      if (p.use_tma_c || w.role != 0) {
        // all warps meet: every warp's staging boxes (in the B ring) have
        // been read before any warp writes the next tile's B stages over
        // them, and in the tail every warp's partial stores or partial reads
        // are done
        int v2 = 1;
        if (lane == 0) v2 = gwait(tmem_empty, it & 1, s_fail, p.err) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, v2, 0) != 0;
        if (ok && wd == 0 && lane == 0) {
          if (w.role == 2) {
            // the stores the meet ordered before this thread, then the ticket
            __threadfence();
            red_add_release_gpu(&p.tickets[blockIdx.x], 1u);
          } else if (w.role == 1) {
            for (int i = 0; i < w.nc; ++i) p.tickets[w.c1 + i] = 0u;   // zero for the next launch
          }
        }
      }
    }
  }

  if (SPLIT && p.gsplit) {
    // ---- split-K combine through global memory ----
    // (1) the accumulator is complete: the MMA thread waited for its MMAs
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int S = p.nsplit;
    const int tile = blockIdx.x / S, split = blockIdx.x % S;
    Work w;
    const bool have = work_item<MT, SPLIT>(p, 0, w);
    const int rows = min(p.M - w.m0, 128);   // valid rows of the tile
    const size_t tile_floats = static_cast<size_t>(rows) * BN;
    if (warp >= 2 && have && !*s_fail) {
      // (2) this split's partial tile, rows x 256 fp32, row-major: each lane
      //     writes its row's 32 columns of a chunk as eight 16-byte stores
      float* mine = p.part + (static_cast<size_t>(tile) * S + split) * tile_floats;
      const int wd = warp - 2, q = warp & 3;
      const int c0 = (wd >> 2) * C::kEpiCols;
      const int row = q * 32 + lane;
#pragma unroll 1
      for (int c = c0; c < c0 + C::kEpiCols; c += 32) {
        uint32_t acc[32], v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, acc);
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
          for (int s = 0; s < 8; ++s) v[8 * t + chunk_col(s)] = acc[8 * t + s];
        if (row < rows) {
          float4* dst = reinterpret_cast<float4*>(mine + static_cast<size_t>(row) * BN + c);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                 __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
        }
      }
    }
    // (3) every split takes one ticket after its partial is visible; the one
    //     that takes the last adds the S partials in split order and stores C
    __threadfence();
    __syncthreads();
    __shared__ int s_last;
    if (threadIdx.x == 0)
      s_last = (atomicAdd(&p.tickets[tile], 1u) == static_cast<unsigned>(S - 1)) ? 1 : 0;
    __syncthreads();
    if (s_last) {
      __threadfence();
      if (warp >= 2 && have && !*s_fail) {
        const float* base = p.part + static_cast<size_t>(tile) * S * tile_floats;
        const int items = rows * (BN / 4);
        for (int i = threadIdx.x - 64; i < items; i += DW * 32) {
          const int r = i / (BN / 4), c4 = (i % (BN / 4)) * 4;
          const float* src = base + static_cast<size_t>(r) * BN + c4;
          float4 acc = __ldcg(reinterpret_cast<const float4*>(src));
          for (int s = 1; s < S; ++s) {
            const float4 t = __ldcg(reinterpret_cast<const float4*>(src + s * tile_floats));
            acc.x += t.x;
            acc.y += t.y;
            acc.z += t.z;
            acc.w += t.w;
          }
          store_group4(p, w.m0 + r, w.n0 + c4, acc);
        }
      }
      if (threadIdx.x == 0) p.tickets[tile] = 0u;   // zero again for the next launch
    }
  } else if (SPLIT) {
    // ---- split-K combine over the cluster ----
    // (1) Every CTA of the cluster is past its main loop: its MMAs and copies
    //     are complete (the MMA thread and the producer waited for them), so
    //     its rings (A, B and raw) may take partial sums.
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const int S = p.nsplit;
    const int rank = static_cast<int>(cluster_ctarank());
    Work w;
    const bool have = work_item<MT, SPLIT>(p, 0, w);
    const int rows = min(p.M - w.m0, 128);   // valid rows of the tile
    float* red = reinterpret_cast<float*>(smem);
    if (warp >= 2 && have && !*s_fail) {
      // (2) push: each warp reads its lane quarter's columns of the
      //     accumulator and stores the 32-column chunks, in output column
      //     order, into the owning CTA's buffer [chunk/S][source rank][row]
      const int wd = warp - 2, q = warp & 3;
      const int c0 = (wd >> 2) * C::kEpiCols;
      const int row = q * 32 + lane;
#pragma unroll 1
      for (int c = c0; c < c0 + C::kEpiCols; c += 32) {
        uint32_t acc[32], v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, acc);
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
          for (int s = 0; s < 8; ++s) v[8 * t + chunk_col(s)] = acc[8 * t + s];
        const int chunk = c / 32, owner = chunk % S, jj = chunk / S;
        if (row < rows) {
          const uint32_t dst = peer_addr(
              red + ((static_cast<size_t>(jj) * S + rank) * rows + row) * kRedRowFloats, owner);
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + j * 4),
                         "r"(v[j]), "r"(v[j + 1]), "r"(v[j + 2]), "r"(v[j + 3])
                         : "memory");
        }
      }
    }
    // (3) all partial sums have arrived
    tc_fence_before();
    cluster_sync();
    if (warp >= 2 && have && !*s_fail) {
      // (4) the owner adds the S partial sums of its chunks in rank order and
      //     stores C: consecutive threads take consecutive 4-column groups
      const int mine = (BN / 32 - rank + S - 1) / S;   // chunks rank, rank + S, ...
      const int items = mine * rows * 8;
      for (int i = threadIdx.x - 64; i < items; i += DW * 32) {
        const int jj = i / (rows * 8), r = (i / 8) % rows, g4 = i % 8;
        const float* src = red + (static_cast<size_t>(jj) * S * rows + r) * kRedRowFloats + g4 * 4;
        float4 acc = *reinterpret_cast<const float4*>(src);
        for (int s = 1; s < S; ++s) {
          const float4 t =
              *reinterpret_cast<const float4*>(src + static_cast<size_t>(s) * rows * kRedRowFloats);
          acc.x += t.x;
          acc.y += t.y;
          acc.z += t.z;
          acc.w += t.w;
        }
        store_group4(p, w.m0 + r, w.n0 + (rank + jj * S) * 32 + g4 * 4, acc);
      }
    }
  }

  // the epilogue's TMA stores are complete before the CTA ends
  if (!SPLIT && warp >= 2 && lane == 0) bulk_wait<0>();
  // everyone (the MMA thread after its drain) meets here before the tensor
  // memory is released
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace gemm

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

// Dequant warps of the small-M form.
constexpr int kSmallDW = 8;
using PrefillCfg = gemm::Cfg<2, 8, false>;
using SmallCfg = gemm::Cfg<1, kSmallDW, true>;

template <int MT, int DW, bool SPLIT>
cudaLaunchConfig_t make_cfg(cudaLaunchAttribute* attr, int grid, int S, cudaStream_t st) {
  using C = gemm::Cfg<MT, DW, SPLIT>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int MT, int DW, bool SPLIT>
cudaError_t prepare() {
  using C = gemm::Cfg<MT, DW, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(gemm::q4_gemm_tc_kernel<MT, DW, SPLIT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::kSmemBytes));
  if (e != cudaSuccess) return e;
  if (SPLIT)
    e = cudaFuncSetAttribute(gemm::q4_gemm_tc_kernel<MT, DW, SPLIT>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

// Clusters of S CTAs of the small-M form that fit on the device at once
// (cached per device; 0 if that size cannot launch).
int small_resident(int S) {
  static int cache[64][gemm::kMaxSplit + 1] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev][S] == 0) {
    if (prepare<1, kSmallDW, true>() != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = make_cfg<1, kSmallDW, true>(attr, S, S, nullptr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm::q4_gemm_tc_kernel<1, kSmallDW, true>, &cfg) !=
        cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    cache[dev][S] = n > 0 ? n : -1;
  }
  return cache[dev][S] > 0 ? cache[dev][S] : 0;
}

bool encode_maps(GemmParams& p, const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                 int a_rows) {
  p.a_rows = a_rows;
  auto encode = get_encode();
  if (!encode) return false;
  // A: bf16 [M][K], boxes of BK x a_rows, rows swizzled in their 128 bytes
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 2)};
    const cuuint32_t box[2] = {gemm::BK, static_cast<cuuint32_t>(a_rows)};
    const cuuint32_t es[2] = {1, 1};
    const CUtensorMapSwizzle swz =
        (gemm::kARowBytes == 128) ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (encode(&p.tmap_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(A), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  // raw Q4: uint16 [K][nb*9], boxes of 72 halfwords (8 blocks) x BK rows
  {
    const int64_t nb = (N + 31) / 32;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nb * 9), static_cast<cuuint64_t>(K)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nb * kBlockBytes)};
    const cuuint32_t box[2] = {72, gemm::BK};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&p.tmap_b, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(B), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

// C for the prefill form's TMA stores: [M][N] fp32 or bf16, boxes of 128 bytes
// x 32 rows, 128-byte swizzle.  False (the epilogue then stores row by row)
// when the row pitch is not a multiple of 16 bytes.
bool encode_c_map(GemmParams& p, void* C, int c_dtype, int64_t M, int64_t N) {
  auto encode = get_encode();
  const int64_t es = c_dtype == 0 ? 4 : 2;
  if (!encode || (N * es) % 16 != 0) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N * es)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / es), 32};
  const cuuint32_t estr[2] = {1, 1};
  return encode(&p.tmap_c,
                c_dtype == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gemm_supported(int64_t M, int64_t N, int64_t K) {
  const int64_t nb = (N + 31) / 32;
  return M >= 1 && nb % 8 == 0 && K % 8 == 0 && K >= 1 && M <= (1LL << 30) && N <= (1LL << 30);
}

int gemm_small_split(int64_t M, int64_t N, int64_t K) {
  if (M > 128) return 0;
  const int64_t tiles = (N + gemm::BN - 1) / gemm::BN;
  const int64_t ksteps = (K + gemm::BK - 1) / gemm::BK;
  const int rows = static_cast<int>(M);
  int best = 0;
  int64_t best_cost = 0;
  for (int S = 1; S <= gemm::kMaxSplit && S <= ksteps; ++S) {
    // the partial sums take the A, B and raw rings (free after the main loop)
    if (gemm::red_bytes(S, rows) > SmallCfg::kOffBars) continue;
    const int active = small_resident(S);
    if (active <= 0) continue;
    const int64_t waves = (tiles + active - 1) / active;
    // a wave also pays its start (first loads) and the combine: about as
    // long as kWaveSteps K steps
    constexpr int64_t kWaveSteps = 10;
    const int64_t cost = waves * ((ksteps + S - 1) / S + kWaveSteps);
    if (best == 0 || cost < best_cost) {
      best = S;
      best_cost = cost;
    }
  }
  return best;
}

int gemm_global_split(int64_t M, int64_t N, int64_t K, int sms) {
  // the partial tiles grow with M: on K = 5120, N = 12288 (48 tiles) the
  // global form with 3 splits against the cluster form with 2 measured
  // +26% / +19% / +8% / +4% at M = 8 / 16 / 32 / 40, even at 48, -4% at 56
  // and -8% at 64 (GB300)
  if (M > 40 || sms <= 0) return 0;
  const int64_t tiles = (N + gemm::BN - 1) / gemm::BN;
  const int64_t ksteps = (K + gemm::BK - 1) / gemm::BK;
  if (tiles > kMaxGemmTickets) return 0;
  // one CTA per SM (the shared-memory plan allows no more): every split of
  // every tile in one wave
  int64_t S = sms / tiles;
  if (S > gemm::kMaxSplit) S = gemm::kMaxSplit;
  if (S > ksteps) S = ksteps;
  if (S < 2) return 0;
  // the cluster form combines on chip; the global form pays a write and a
  // read of the partial tiles, so it runs only where it has more splits
  const int sc = gemm_small_split(M, N, K);
  if (sc > 0 && S <= sc) return 0;
  return static_cast<int>(S);
}

PrefillPlan prefill_plan(int64_t M, int64_t N, int64_t K, int sms) {
  PrefillPlan pl;
  const int64_t tiles = ((M + PrefillCfg::kBM - 1) / PrefillCfg::kBM) * ((N + gemm::BN - 1) / gemm::BN);
  const int64_t ksteps = (K + gemm::BK - 1) / gemm::BK;
  pl.grid = static_cast<int>(tiles < sms ? tiles : sms);
  pl.full_tiles = static_cast<int>(tiles);
  pl.tail_ctas = 0;
  if (sms <= 0 || tiles <= 0) return pl;
  const int64_t rem = tiles % sms;
  if (rem == 0) return pl;
  // the last round's tiles: their K steps shared by up to kTailParts CTAs per
  // tile, each CTA's range no longer than a tile; worth it when a range plus
  // the partial tile's write and read (about kTailCostSteps K steps) is
  // shorter than a whole tile
  constexpr int64_t kTailParts = 4, kTailCostSteps = 6;
  const int64_t T = rem * ksteps;
  int64_t ctas = std::min<int64_t>(sms, rem * kTailParts);
  ctas = std::min<int64_t>(ctas, T);
  if ((T + ctas - 1) / ctas + kTailCostSteps > ksteps) return pl;
  // every CTA of the grid has work: whole tiles (then the grid fills the
  // SMs) or a part of the tail
  pl.grid = tiles >= sms ? sms : static_cast<int>(ctas);
  pl.full_tiles = static_cast<int>(tiles - rem);
  pl.tail_ctas = static_cast<int>(ctas);
  return pl;
}

int64_t prefill_units(int64_t M, int64_t N, int64_t K, int sms, int32_t* out, int64_t cap) {
  const PrefillPlan pl = prefill_plan(M, N, K, sms);
  const int64_t tiles =
      ((M + PrefillCfg::kBM - 1) / PrefillCfg::kBM) * ((N + gemm::BN - 1) / gemm::BN);
  const bool tail = pl.tail_ctas > 0;
  const int G = tail ? pl.grid : static_cast<int>(tiles < sms ? tiles : sms);
  const int full = tail ? pl.full_tiles : static_cast<int>(tiles);
  int64_t n = 0;
  for (int c = 0; c < G; ++c) {
    gemm::Work w;
    for (int it = 0; gemm::prefill_unit<2>(static_cast<int>(M), static_cast<int>(N),
                                            static_cast<int>(K), full, pl.tail_ctas, c, G, it, w);
         ++it, ++n) {
      if (n < cap) {
        int32_t* r = out + n * 9;
        r[0] = c;
        r[1] = it;
        r[2] = w.m0;
        r[3] = w.n0;
        r[4] = w.kb;
        r[5] = w.ke;
        r[6] = w.role;
        r[7] = w.c1;
        r[8] = w.nc;
      }
    }
  }
  return n;
}

size_t prefill_tail_ticket_bytes(const PrefillPlan& pl) {
  return (static_cast<size_t>(pl.tail_ctas) * sizeof(unsigned) + 255) / 256 * 256;
}

size_t prefill_tail_bytes(const PrefillPlan& pl) {
  if (pl.tail_ctas <= 0) return 0;
  return prefill_tail_ticket_bytes(pl) +
         static_cast<size_t>(pl.tail_ctas) * 128 * PrefillCfg::kTmemCols * sizeof(float);
}

size_t gemm_part_bytes(int64_t M, int64_t N, int S) {
  const int64_t tiles = (N + gemm::BN - 1) / gemm::BN;
  const int64_t rows = M < 128 ? M : 128;
  return static_cast<size_t>(tiles) * S * rows * gemm::BN * sizeof(float);
}

cudaError_t launch_gemm(void* C, int c_dtype, const void* A, const void* B, int64_t M, int64_t N,
                        int64_t K, unsigned* err, int sms, cudaStream_t st, float* part,
                        unsigned* tickets) {
  GemmParams p;
  p.use_tma_c = 0;
  p.gsplit = 0;
  p.part = nullptr;
  p.tickets = nullptr;
  p.full_tiles = 0;
  p.tail_ctas = 0;
  p.C = C;
  p.c_dtype = c_dtype;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.err = err;
  cudaLaunchAttribute attr[1];
  if (M > 128) {
    // prefill form: persistent, one CTA per SM at most
    if (!encode_maps(p, A, B, M, N, K, PrefillCfg::kBM)) return cudaErrorInvalidValue;
    p.use_tma_c = encode_c_map(p, C, c_dtype, M, N) ? 1 : 0;
    p.nsplit = 1;
    cudaError_t e = prepare<2, 8, false>();
    if (e != cudaSuccess) return e;
    // the last round's K steps shared over the grid when the caller gives
    // the tail's tickets and partial tiles (prefill_tail_bytes)
    const PrefillPlan pl = prefill_plan(M, N, K, sms);
    const bool tail = pl.tail_ctas > 0 && part && tickets;
    const int64_t tiles = ((M + PrefillCfg::kBM - 1) / PrefillCfg::kBM) * ((N + gemm::BN - 1) / gemm::BN);
    p.full_tiles = tail ? pl.full_tiles : static_cast<int>(tiles);
    p.tail_ctas = tail ? pl.tail_ctas : 0;
    p.part = tail ? part : nullptr;
    p.tickets = tail ? tickets : nullptr;
    const int grid = tail ? pl.grid : static_cast<int>(tiles < sms ? tiles : sms);
    cudaLaunchConfig_t cfg = make_cfg<2, 8, false>(attr, grid, 1, st);
    return cudaLaunchKernelEx(&cfg, gemm::q4_gemm_tc_kernel<2, 8, false>, p);
  }
  const int a_rows = static_cast<int>(((M + 15) / 16) * 16);   // M <= 128
  // small-M form through global memory: S independent CTAs per tile
  const int Sg = (part && tickets) ? gemm_global_split(M, N, K, sms) : 0;
  if (Sg > 0) {
    if (!encode_maps(p, A, B, M, N, K, a_rows)) return cudaErrorInvalidValue;
    p.nsplit = Sg;
    p.gsplit = 1;
    p.part = part;
    p.tickets = tickets;
    cudaError_t e = prepare<1, kSmallDW, true>();
    if (e != cudaSuccess) return e;
    const int64_t tiles = (N + gemm::BN - 1) / gemm::BN;
    cudaLaunchConfig_t cfg = make_cfg<1, kSmallDW, true>(attr, static_cast<int>(tiles * Sg), 1, st);
    return cudaLaunchKernelEx(&cfg, gemm::q4_gemm_tc_kernel<1, kSmallDW, true>, p);
  }
  // small-M form: one 128 x 256 tile per cluster of S CTAs splitting K
  const int S = gemm_small_split(M, N, K);
  if (S <= 0) return cudaErrorInvalidConfiguration;
  if (!encode_maps(p, A, B, M, N, K, a_rows)) return cudaErrorInvalidValue;
  p.nsplit = S;
  cudaError_t e = prepare<1, kSmallDW, true>();
  if (e != cudaSuccess) return e;
  const int64_t tiles = (N + gemm::BN - 1) / gemm::BN;
  cudaLaunchConfig_t cfg = make_cfg<1, kSmallDW, true>(attr, static_cast<int>(tiles * S), S, st);
  return cudaLaunchKernelEx(&cfg, gemm::q4_gemm_tc_kernel<1, kSmallDW, true>, p);
}

}  // namespace q4
