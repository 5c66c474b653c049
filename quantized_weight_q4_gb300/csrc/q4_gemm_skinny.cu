// Q4_0 GEMM for a few rows of A on the tensor cores (sm_103a), operands swapped.
//
// C[M, N] = A[M, K] . W[K, N] for 1 <= M <= 32 rows of bf16 A (a batch of
// decode tokens: the C++ DeepSeek engine page batches the tokens of a prompt
// into one matmul, §5.2), with each weight dequantised once to the bf16 tile
// element bf16_rn((q - 8) * d) and fp32 accumulation in tensor memory, as the
// prefill GEMM does.
//
// With so few rows the matmul is bound by streaming the weights from HBM; the
// tensor cores only take the products off the CUDA cores.  The weights are the
// MMA's A operand (M = 128 output columns per instruction, MN-major) and the
// activations its B operand (N = 16 or 32 token rows, K-major), so the
// tokens are not padded to a 128-row tile.  A CTA owns one column tile of 256
// columns (two MMA tiles) and one slice of K:
//  * warp 0 streams the raw weights in 18 KB TMA boxes (128 rows x 8 blocks)
//    and warp 10 the activations in boxes of 64 K x NT rows (128-byte
//    swizzle), each on its own ring, so that the weights run ahead of the
//    MMAs by the whole raw ring;
//  * warps 2..9 dequantise each 64-row half of a raw stage into an MN-major,
//    128-byte-swizzled bf16 tile (q4_tc_core.cuh), then, after the last
//    stage, read the accumulators out of tensor memory;
//  * warp 1 allocates tensor memory and issues tcgen05.mma (two per 16 rows
//    of K), freeing the tile and activation stages with tcgen05.commit.
// The K slices of a tile add their fp32 partial tiles through global memory:
// each CTA writes its partial, takes a ticket from the tile's counter, and the
// CTA with the last ticket adds the partials in slice order (deterministic),
// stores C and returns the counter to zero.  Every wait is bounded; on a
// timeout the CTA records Q4_DEVERR_TIMEOUT, stops issuing, waits (bounded)
// for its copies and MMAs and frees its tensor memory.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "q4_device.cuh"
#include "q4_kernels.h"
#include "q4_tc_core.cuh"

namespace q4 {
namespace skinny {

using namespace gemm;

constexpr int kTileCols = 256;                              // output columns per CTA
constexpr int kRawRows = 128;                               // K rows of one raw stage
constexpr int kRawStageBytes = kRawRows * kRawRowBytes;     // 18432
constexpr int kDW = 8;                                      // dequant warps
constexpr int kEW = 8;                                      // epilogue warps (the first kEW)
constexpr int kActWarp = 2 + kDW;                           // the activation loader
constexpr int kThreads = (3 + kDW) * 32;
constexpr int kUPW = (BK / 4) / kDW;                        // dequant units per warp
static_assert(kDW >= kEW && (BK / 4) % kDW == 0, "dequant and epilogue warps");

template <int NT>
struct Cfg {
  static constexpr int kActBytes = BK * NT * 2;             // one 64-K activation stage
  static constexpr int kStagesRaw = 6;
  static constexpr int kStagesBt = 3;                       // bf16 weight tiles of 32 KB
  static constexpr int kStagesAct = NT == 16 ? 8 : 4;          // 16 KB
  static constexpr uint32_t kTmemCols = 2 * NT < 32 ? 32 : 2 * NT;
  static constexpr uint32_t kOffBt = kStagesRaw * kRawStageBytes;
  static constexpr uint32_t kOffAct = kOffBt + kStagesBt * kBBytes;
  static constexpr uint32_t kOffBars = kOffAct + kStagesAct * kActBytes;
  static constexpr uint32_t kBarBytes = 512;
  static constexpr uint32_t kSmemBytes = kOffBars + kBarBytes + 1024;
  // instruction descriptor of kind::f16: fp32 D, bf16 A and B, A MN-major
  // (the dequantised weight tile), B K-major (the activations), N = NT,
  // M = 128
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) |
                                     (0u << 16) | (static_cast<uint32_t>(NT >> 3) << 17) |
                                     (static_cast<uint32_t>(128 >> 4) << 24);
  static_assert(NT == 16 || NT == 32, "token tile");
  static_assert(kOffBt % 1024 == 0 && kOffAct % 1024 == 0 && kActBytes % 1024 == 0,
                "swizzled stages need 1024-byte alignment");
  static_assert((2 * kStagesRaw + 2 * kStagesBt + 2 * kStagesAct + 1) * 8 + 16 <= kBarBytes,
                "barrier region overflows");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory plan exceeds the per-CTA limit");
};

// 32 lanes x 16 columns of 32-bit accumulators: thread i gets its lane's 16.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Output column (within the tile) of tile position p: the dequant packs
// nibbles j and j + 4 of a word into one bf16 pair, so within each chunk of 8
// positions slot s holds column chunk_col(s).
__device__ __forceinline__ int column_of(int p) { return (p & ~7) | chunk_col(p & 7); }

__device__ __forceinline__ void store_c(const SkinnyParams& p, int row, int col, float v) {
  const size_t i = static_cast<size_t>(row) * p.N + col;
  if (p.c_dtype == 0) reinterpret_cast<float*>(p.C)[i] = v;
  else reinterpret_cast<uint16_t*>(p.C)[i] = static_cast<uint16_t>(bf16_bits(v));
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) q4_skinny_kernel(const __grid_constant__ SkinnyParams p) {
  using C = Cfg<NT>;
  constexpr int SR = C::kStagesRaw, SB = C::kStagesBt, SA = C::kStagesAct;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sRaw = smem;
  uint8_t* sBt = smem + C::kOffBt;
  uint8_t* sAct = smem + C::kOffAct;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* full_raw = bars;                 // [SR] TMA bytes
  uint64_t* empty_raw = full_raw + SR;       // [SR] dequant warps
  uint64_t* full_bt = empty_raw + SR;        // [SB] dequant warps
  uint64_t* empty_bt = full_bt + SB;         // [SB] MMA commit
  uint64_t* full_act = empty_bt + SB;        // [SA] TMA bytes
  uint64_t* empty_act = full_act + SA;       // [SA] MMA commit
  uint64_t* drain = empty_act + SA;          // [1]  MMA commit after the last MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* s_fail = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* s_last = s_fail + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.nsplit;
  const int tile = blockIdx.x / S, split = blockIdx.x % S;
  const int ksteps = (p.K + kRawRows - 1) / kRawRows;          // raw stages of the whole K
  const int r0 = split * ksteps / S, r1 = (split + 1) * ksteps / S;
  const int nraw = r1 - r0;                                     // raw stages of this slice
  const int nsub = 2 * nraw;                                    // 64-row sub-stages

  if (threadIdx.x == 0) {
    for (int i = 0; i < SR; ++i) {
      mbar_init(&full_raw[i], 1);
      mbar_init(&empty_raw[i], kDW);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&full_bt[i], kDW);
      mbar_init(&empty_bt[i], 1);
    }
    for (int i = 0; i < SA; ++i) {
      mbar_init(&full_act[i], 1);
      mbar_init(&empty_act[i], 1);
    }
    mbar_init(drain, 1);
    *s_fail = 0;
    *s_last = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ================= producer: weights =================
    if (lane == 0) {
      int gr = 0;
      for (int r = 0; r < nraw && !*s_fail; ++r, ++gr) {
        const int sr = gr % SR;
        if (gr >= SR && !gwait(&empty_raw[sr], ((gr / SR) - 1) & 1, s_fail, p.err)) break;
        mbar_arrive_expect_tx(&full_raw[sr], kRawStageBytes);
        tma_load_2d(sRaw + sr * kRawStageBytes, &p.tmap_w, tile * (kTileCols / kBlockCols) * 9,
                    (r0 + r) * kRawRows, &full_raw[sr]);
      }
      // no copy may still be writing shared memory when the CTA exits: wait
      // (bounded) for the latest load of every slot
      for (int g = gr - 1; g >= 0 && g >= gr - SR; --g)
        (void)mbar_wait(&full_raw[g % SR], (g / SR) & 1);
    }
  } else if (warp == kActWarp) {
    // ================= producer: activations =================
    if (lane == 0) {
      pdl_wait();   // the activations may come from the kernel before
      int ga = 0;
      for (int g = 0; g < nsub && !*s_fail; ++g, ++ga) {
        const int sa = ga % SA;
        if (ga >= SA && !gwait(&empty_act[sa], ((ga / SA) - 1) & 1, s_fail, p.err)) break;
        mbar_arrive_expect_tx(&full_act[sa], C::kActBytes);
        tma_load_2d(sAct + sa * C::kActBytes, &p.tmap_a, r0 * kRawRows + g * BK, 0,
                    &full_act[sa]);
      }
      for (int g = ga - 1; g >= 0 && g >= ga - SA; --g)
        (void)mbar_wait(&full_act[g % SA], (g / SA) & 1);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      for (int g = 0; g < nsub; ++g) {
        const int sb = g % SB, sa = g % SA;
        if (!gwait(&full_bt[sb], (g / SB) & 1, s_fail, p.err) ||
            !gwait(&full_act[sa], (g / SA) & 1, s_fail, p.err))
          break;
        tc_fence_after();
        const uint32_t bt = smem_u32(sBt + sb * kBBytes);
        const uint32_t act = smem_u32(sAct + sa * C::kActBytes);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // activations: K-major, 32 bytes per 16 K, 8-row atoms 1024 bytes apart
          const uint64_t bdesc = smem_desc(act + kk * 32, 16, 1024, kSwizzle128);
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            // weights: MN-major; an MMA tile of 128 columns is two 64-column
            // swizzle atoms kBLbo apart; 16 rows of K are two 8-row atoms
            const uint64_t adesc =
                smem_desc(bt + mt * 2 * kBLbo + kk * 2048, kBLbo, 1024, kSwizzle128);
            tc_mma(tmem + mt * NT, adesc, bdesc, C::kIdesc, (g > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc_commit(&empty_bt[sb]);
        tc_commit(&empty_act[sa]);
      }
      // every MMA issued is complete before the accumulators are read, the
      // rings reused or the tensor memory freed (bounded, also after a failure)
      tc_commit(drain);
      (void)mbar_wait(drain, 0);
    }
  } else {
    // ================= dequant (warps 2 .. kDW+1) =================
    const int wd = warp - 2;
    int gb = 0;
    bool ok = true;
    for (int r = 0; r < nraw && ok; ++r) {
      const int sr = r % SR;
      int v = 1;
      if (lane == 0) v = gwait(&full_raw[sr], (r / SR) & 1, s_fail, p.err) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, v, 0) != 0;
      if (!ok) break;
      for (int h = 0; h < 2; ++h, ++gb) {
        const int sb = gb % SB;
        v = 1;
        if (lane == 0 && gb >= SB)
          v = gwait(&empty_bt[sb], ((gb / SB) - 1) & 1, s_fail, p.err) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, v, 0) != 0;
        if (!ok) break;
        dequant_stage<kUPW>(sRaw + sr * kRawStageBytes + h * BK * kRawRowBytes, sBt + sb * kBBytes,
                            wd, lane);
        fence_async_smem();   // the tensor core reads the tile through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_bt[sb]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_raw[sr]);
    }
  }

  // ---- epilogue: every thread reaches every barrier below on every path ----
  // (1) the accumulators are complete (the MMA thread waited for its MMAs)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool epi = warp >= 2 && warp < 2 + kEW && !*s_fail && nsub > 0;
  const int wd = warp - 2;
  const int q = warp & 3;                      // the tensor-memory lane quarter of this warp
  const int mt = (wd >> 2) & 1;                // its MMA tile
  const int pos = mt * 128 + q * 32 + lane;    // its tile position (one per thread)
  const int col = tile * kTileCols + column_of(pos);
  const int M = p.M;
  if (epi) {
    // (2) this slice's partial sums: thread = one column, NT token values
    uint32_t acc[NT];
#pragma unroll
    for (int c = 0; c < NT; c += 16) {
      uint32_t r[16];
      tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + mt * NT + c, r);
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[c + j] = r[j];
    }
    if (S == 1) {
      if (col < p.N)
#pragma unroll
        for (int t = 0; t < NT; ++t)
          if (t < M) store_c(p, t, col, __uint_as_float(acc[t]));
    } else {
      float* mine = p.part + (static_cast<size_t>(tile) * S + split) * M * kTileCols;
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (t < M) __stcg(mine + t * kTileCols + pos, __uint_as_float(acc[t]));
    }
  }
  if (S > 1) {
    // (3) every slice takes a ticket after its partial is visible; the one
    //     with the last ticket adds the S partials in slice order
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const unsigned t = atomicAdd(&p.tickets[tile], 1u);
      __threadfence();
      *s_last = (t == static_cast<unsigned>(S - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (*s_last) {
      if (epi && col < p.N) {
        const float* base = p.part + static_cast<size_t>(tile) * S * M * kTileCols + pos;
        const size_t stride = static_cast<size_t>(M) * kTileCols;
        for (int t = 0; t < M; ++t) {
          float s = 0.f;
          for (int s0 = 0; s0 < S; s0 += 8) {
            float v[8];
#pragma unroll
            for (int b = 0; b < 8; ++b)
              v[b] = (s0 + b < S) ? __ldcg(base + (s0 + b) * stride + t * kTileCols) : 0.f;
#pragma unroll
            for (int b = 0; b < 8; ++b)
              if (s0 + b < S) s = (s0 + b == 0) ? v[b] : s + v[b];
          }
          store_c(p, t, col, s);
        }
      }
      if (threadIdx.x == 0) p.tickets[tile] = 0u;   // zero again for the next launch
    }
  }
  // (4) everyone meets before the tensor memory is released
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace skinny

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 skinny_encoder() {
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

int token_tile(int64_t M) { return M <= 16 ? 16 : 32; }

template <int NT>
cudaError_t launch_nt(const SkinnyParams& p, int grid, cudaStream_t st) {
  using C = skinny::Cfg<NT>;
  cudaError_t e = cudaFuncSetAttribute(skinny::q4_skinny_kernel<NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::kSmemBytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(skinny::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, skinny::q4_skinny_kernel<NT>, p);
}

}  // namespace

bool skinny_supported(int64_t M, int64_t N, int64_t K) {
  const int64_t nb = (N + 31) / 32;
  return M >= 1 && M <= 32 && nb % 8 == 0 && K % 8 == 0 && K >= 1 && N <= (1LL << 30) &&
         K <= (1LL << 30);
}

int skinny_split(int64_t N, int64_t K, int sms) {
  const int64_t tiles = (N + skinny::kTileCols - 1) / skinny::kTileCols;
  const int64_t ksteps = (K + skinny::kRawRows - 1) / skinny::kRawRows;
  if (tiles > kMaxSkinnyTickets) return 1;
  // one CTA per SM: every slice of every tile in one wave
  int64_t S = sms / tiles;
  if (S > 64) S = 64;
  if (S > ksteps) S = ksteps;
  return static_cast<int>(S < 1 ? 1 : S);
}

size_t skinny_part_bytes(int64_t M, int64_t N, int S) {
  if (S <= 1) return 0;
  const int64_t tiles = (N + skinny::kTileCols - 1) / skinny::kTileCols;
  return static_cast<size_t>(tiles) * S * M * skinny::kTileCols * sizeof(float);
}

cudaError_t launch_skinny(void* C, int c_dtype, const void* A, const void* B, int64_t M, int64_t N,
                          int64_t K, unsigned* err, int S, float* part, unsigned* tickets,
                          cudaStream_t st) {
  if (!skinny_supported(M, N, K) || S < 1 || (S > 1 && (!part || !tickets)))
    return cudaErrorInvalidValue;
  auto encode = skinny_encoder();
  if (!encode) return cudaErrorInvalidValue;
  SkinnyParams p;
  p.C = C;
  p.c_dtype = c_dtype;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.nsplit = S;
  p.part = part;
  p.tickets = tickets;
  p.err = err;
  const int NT = token_tile(M);
  {
    // activations: bf16 [M][K], boxes of 64 K x NT rows (rows past M read as
    // zero), 128-byte swizzle
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 2)};
    const cuuint32_t box[2] = {gemm::BK, static_cast<cuuint32_t>(NT)};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&p.tmap_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(A), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // raw weights: uint16 [K][nb*9], boxes of 72 halfwords (8 blocks) x 128 rows
    const int64_t nb = (N + 31) / 32;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nb * 9), static_cast<cuuint64_t>(K)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nb * kBlockBytes)};
    const cuuint32_t box[2] = {72, static_cast<cuuint32_t>(skinny::kRawRows)};
    const cuuint32_t es[2] = {1, 1};
    if (encode(&p.tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(B), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int64_t tiles = (N + skinny::kTileCols - 1) / skinny::kTileCols;
  const int64_t grid = tiles * S;
  if (grid > (1LL << 31) - 1) return cudaErrorInvalidValue;
  return NT == 16 ? launch_nt<16>(p, static_cast<int>(grid), st)
                  : launch_nt<32>(p, static_cast<int>(grid), st);
}

}  // namespace q4
