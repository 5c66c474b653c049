// Split-K Q4_0 GEMV for small M and the grouped routed-expert GEMVs (sm_103a).
//
// What it computes: C[i, j] = sum_k A[i, k] * (q[k, j] - 8) * d[k, j/32], the
// fused dequant-matmul loop of the C++ DeepSeek engine page (§3.4), over the
// block layout of its §2.2-§2.3 (K rows of ceil(N/32) 18-byte blocks, each
// block spanning 32 output columns of one row).
//
// How (GB300-first, not the page's CPU loop):
//  * A CTA owns a column tile of up to 8 blocks (256 columns, 144 bytes of a
//    row) and a contiguous slice of rows (split-K).  One producer warp streams
//    the slice's row segments into a 4-stage shared-memory ring with TMA bulk
//    copies (cp.async.bulk, completion on mbarriers); eight consumer warps
//    decode the nibbles in registers and accumulate in fp32 with packed
//    fp32x2 FMAs.  Rows whose segments are not 16-byte aligned are staged by
//    the producer warp with plain loads instead.
//  * Partial sums over the split are combined in a fixed order (split 0, 1,
//    ...) by the last CTA of each tile to arrive (an atomic ticket), so the
//    result is deterministic and no CTA ever waits on another.
//  * Programmatic dependent launch: the producer starts streaming weights
//    before griddepcontrol.wait; A is read, and workspace written, only after.
//
// The routed-expert kernels (KTransformers DeepSeek-V2 page, «优化三»: 6 of
// 160 experts per token, run as batched GEMVs; «规则二»: gate -> top-k) reuse
// the same core: every CTA re-derives, from topk_idx, the sorted list of
// experts in use and the (token, slot) list of its expert, so no routing
// kernel and no host synchronisation is needed.
#include <cstdint>
#include <cuda_runtime.h>

#include "q4_device.cuh"
#include "q4_kernels.h"

namespace q4 {

constexpr int kTileBlocks = 8;                         // blocks per column tile
constexpr int kRowsPerStage = 64;
constexpr int kStages = 4;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;        // 256
constexpr int kThreads = kConsumers + 32;              // + producer warp
constexpr int kRowPhases = kConsumers / kTileBlocks;   // 32 rows in flight per CTA
constexpr int kRowBytes = kTileBlocks * kBlockBytes;   // 144
constexpr int kStageBytes = kRowsPerStage * kRowBytes + 16;   // + tail pad for 20-byte reads

// ---------------------------------------------------------------------------
// Shared-memory plan
// ---------------------------------------------------------------------------
struct SmemPlan {
  uint32_t ring, red, bars, a, list, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

template <int MR>
__host__ __device__ inline SmemPlan smem_plan(int rows_per_split, int list_cap) {
  SmemPlan p;
  p.ring = 0;
  p.red = align_up(kStages * kStageBytes, 16);
  p.bars = p.red + kConsumerWarps * MR * 256 * 4;
  p.a = p.bars + 2 * kStages * 8;
  p.list = align_up(p.a + MR * rows_per_split * 4, 16);
  p.total = align_up(p.list + list_cap * 4 + 64, 128);
  return p;
}

// ---------------------------------------------------------------------------
// Consumer arithmetic: one block of one row into the accumulators
// ---------------------------------------------------------------------------
// acc[m][4t + i] holds columns (8t + 2i, 8t + 2i + 1) of the block.
//
// Word t of qs holds columns 8t..8t+7 as nibbles 0..7 (bits 4n..4n+3).  Nibbles
// 0..4 are decoded in place (positions 0..4); nibbles 5..7 from w >> 12, where
// they sit at positions 2..4.  Pairs (0,1), (2,3), (4,5), (6,7) therefore use
// positions (0,1), (2,3), (4,2), (3,4).
struct PairConsts {
  f32x2 b01, b23, b42, b34;   // -(2^23 + 8*16^p) per half
};

__device__ __forceinline__ PairConsts pair_consts() {
  PairConsts c;
  c.b01 = pack2(neg_bias(0), neg_bias(1));
  c.b23 = pack2(neg_bias(2), neg_bias(3));
  c.b42 = pack2(neg_bias(4), neg_bias(2));
  c.b34 = pack2(neg_bias(3), neg_bias(4));
  return c;
}

// s01.. are (x * 16^-p) pairs for the positions above; x = a*d (M = 1) or d.
struct PairScales {
  f32x2 s01, s23, s42, s34;
};

__device__ __forceinline__ PairScales pair_scales(float x) {
  PairScales s;
  const f32x2 xx = pack2(x, x);
  s.s01 = mul2(xx, pack2(1.0f, 0.0625f));
  s.s23 = mul2(xx, pack2(0.00390625f, 0.000244140625f));
  s.s42 = mul2(xx, pack2(1.52587890625e-05f, 0.00390625f));
  s.s34 = mul2(xx, pack2(0.000244140625f, 1.52587890625e-05f));
  return s;
}

// The four signed, power-of-two-scaled codes of word w as pairs.
struct WordCodes {
  f32x2 c01, c23, c45, c67;
};

__device__ __forceinline__ WordCodes word_codes(uint32_t w, const PairConsts& k) {
  const uint32_t y = w >> 12;
  WordCodes c;
  c.c01 = add2(pack2(nib_f(w, 0x0000000Fu), nib_f(w, 0x000000F0u)), k.b01);
  c.c23 = add2(pack2(nib_f(w, 0x00000F00u), nib_f(w, 0x0000F000u)), k.b23);
  c.c45 = add2(pack2(nib_f(w, 0x000F0000u), nib_f(y, 0x00000F00u)), k.b42);
  c.c67 = add2(pack2(nib_f(y, 0x0000F000u), nib_f(y, 0x000F0000u)), k.b34);
  return c;
}

template <int MR>
__device__ __forceinline__ void accumulate_block(f32x2 (&acc)[MR][16], uint32_t dbits,
                                                 const uint32_t (&qs)[4], const float* a,
                                                 int a_ld, const PairConsts& k) {
  const float d = fp16_bits_to_f32(dbits);
  if constexpr (MR == 1) {
    // acc += (a*d * 16^-p) * (16^p (q - 8))
    const PairScales s = pair_scales(a[0] * d);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const WordCodes c = word_codes(qs[t], k);
      acc[0][4 * t + 0] = fma2(s.s01, c.c01, acc[0][4 * t + 0]);
      acc[0][4 * t + 1] = fma2(s.s23, c.c23, acc[0][4 * t + 1]);
      acc[0][4 * t + 2] = fma2(s.s42, c.c45, acc[0][4 * t + 2]);
      acc[0][4 * t + 3] = fma2(s.s34, c.c67, acc[0][4 * t + 3]);
    }
  } else {
    // w = (d * 16^-p) * (16^p (q - 8)) is the exact weight; acc[m] += a_m * w
    const PairScales s = pair_scales(d);
    f32x2 am[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) am[m] = pack2(a[m * a_ld], a[m * a_ld]);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const WordCodes c = word_codes(qs[t], k);
      const f32x2 w01 = mul2(s.s01, c.c01);
      const f32x2 w23 = mul2(s.s23, c.c23);
      const f32x2 w45 = mul2(s.s42, c.c45);
      const f32x2 w67 = mul2(s.s34, c.c67);
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        acc[m][4 * t + 0] = fma2(am[m], w01, acc[m][4 * t + 0]);
        acc[m][4 * t + 1] = fma2(am[m], w23, acc[m][4 * t + 1]);
        acc[m][4 * t + 2] = fma2(am[m], w45, acc[m][4 * t + 2]);
        acc[m][4 * t + 3] = fma2(am[m], w67, acc[m][4 * t + 3]);
      }
    }
  }
}

// Waits on `bar`, unless the CTA has already failed; on a timeout records the
// error and marks the CTA failed so that no thread waits again.  Threads never
// leave their loops early, so every named barrier is still reached.
__device__ __forceinline__ bool wait_or_fail(uint64_t* bar, uint32_t parity, volatile int* fail,
                                             unsigned* err) {
  if (*fail) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*fail) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *fail = 1;
      atomicOr(err, kDevErrTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// Producer: stage row segments [k0 + s*R, ...) of the tile into the ring
// ---------------------------------------------------------------------------
struct StreamDesc {
  const uint8_t* B;   // matrix base
  int nb;             // blocks per row
  int b0, tb;         // first block of the tile, blocks in the tile
  int k0, rows;       // row slice
  bool bulk;          // row segments are 16-byte aligned and 16-byte sized
};

__device__ __forceinline__ bool produce_stage(const StreamDesc& sd, int s, uint8_t* stage,
                                              uint64_t* full, int lane) {
  const int r0 = s * kRowsPerStage;
  const int nr = min(kRowsPerStage, sd.rows - r0);
  const uint32_t seg = static_cast<uint32_t>(sd.tb) * kBlockBytes;
  if (sd.bulk) {
    if (lane == 0) mbar_arrive_expect_tx(full, seg * static_cast<uint32_t>(nr));
    __syncwarp();
    for (int r = lane; r < nr; r += 32) {
      const uint8_t* src =
          sd.B + (static_cast<size_t>(sd.k0 + r0 + r) * sd.nb + sd.b0) * kBlockBytes;
      bulk_g2s(stage + r * kRowBytes, src, seg, full);
    }
  } else {
    // 2-byte aligned rows: copy with 16-bit loads (every block offset is even)
    const int halves = static_cast<int>(seg / 2);
    for (int r = 0; r < nr; ++r) {
      const uint16_t* src = reinterpret_cast<const uint16_t*>(
          sd.B + (static_cast<size_t>(sd.k0 + r0 + r) * sd.nb + sd.b0) * kBlockBytes);
      uint16_t* dst = reinterpret_cast<uint16_t*>(stage + r * kRowBytes);
      for (int h = lane; h < halves; h += 32) dst[h] = __ldg(src + h);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(full);
  }
  return true;
}

// ---------------------------------------------------------------------------
// The consumer-side reduction of one tile: warp shuffles, then across warps
// through shared memory.  Returns, in `out`, the value of column `tid` of the
// tile (tid in [0, 256)) for each of the MR rows.
// ---------------------------------------------------------------------------
template <int MR>
__device__ __forceinline__ void reduce_tile(f32x2 (&acc)[MR][16], float* red, int warp, int lane,
                                            int tid, float (&out)[MR]) {
  const bool hi16 = (lane & 16) != 0;
  const bool hi8 = (lane & 8) != 0;
  const int b = lane & 7;
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    f32x2 h[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const f32x2 send = hi16 ? acc[m][i] : acc[m][8 + i];
      const f32x2 keep = hi16 ? acc[m][8 + i] : acc[m][i];
      const f32x2 recv = __shfl_xor_sync(0xffffffffu, send, 16);
      h[i] = add2(keep, recv);
    }
    f32x2 q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const f32x2 send = hi8 ? h[i] : h[4 + i];
      const f32x2 keep = hi8 ? h[4 + i] : h[i];
      const f32x2 recv = __shfl_xor_sync(0xffffffffu, send, 8);
      q[i] = add2(keep, recv);
    }
    // lane now holds columns col0 .. col0+7 of block b
    const int col0 = (hi16 ? 16 : 0) + (hi8 ? 8 : 0);
    float* dst = red + (warp * MR + m) * 256 + b * 32 + col0;
    float v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) unpack2(q[i], v[2 * i], v[2 * i + 1]);
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) s += red[(w * MR + m) * 256 + tid];
    out[m] = s;
  }
}

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
}

// Called by all consumers after their partials are stored: returns true in
// the CTA that arrived last on `ticket` (expecting `arrivals` CTAs), which
// then owns the final combine.  The last CTA resets the ticket to zero.
__device__ __forceinline__ bool last_arrival(unsigned* ticket, unsigned arrivals, int tid,
                                             int* s_flag) {
  __threadfence();
  consumers_sync();
  if (tid == 0) {
    const unsigned old = atomicAdd(ticket, 1u);
    const int last = (old == arrivals - 1) ? 1 : 0;
    if (last) *ticket = 0u;
    *s_flag = last;
  }
  consumers_sync();
  const bool last = *s_flag != 0;
  if (last) __threadfence();
  return last;
}

// ---------------------------------------------------------------------------
// Routing helpers for the expert kernels
// ---------------------------------------------------------------------------
// j-th expert id (ascending) among those named by a valid topk_idx entry, or
// -1; computed by warp 0.  `present` is a scratch bitmap of ceil(E/32) words.
__device__ int jth_active_expert(const int32_t* idx, int nslots, int E, int j, unsigned* present,
                                 int lane) {
  const int words = (E + 31) / 32;
  for (int w = lane; w < words; w += 32) present[w] = 0u;
  __syncwarp();
  for (int s = lane; s < nslots; s += 32) {
    const int e = idx[s];
    if (e >= 0 && e < E) atomicOr(&present[e >> 5], 1u << (e & 31));
  }
  __syncwarp();
  int result = -1;
  int base = 0;
  for (int w0 = 0; w0 < words; w0 += 32) {
    const int w = w0 + lane;
    const unsigned bits = (w < words) ? present[w] : 0u;
    const int cnt = __popc(bits);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = base + incl - cnt;
    if (j >= excl && j < excl + cnt) {
      // the (j - excl)-th set bit of `bits`
      unsigned b = bits;
      for (int r = j - excl; r > 0; --r) b &= b - 1;
      result = w * 32 + (__ffs(b) - 1);
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) result = max(result, __shfl_xor_sync(0xffffffffu, result, o));
  return result;
}

// Slots s (ascending) with idx[s] == e, written to list; returns the count.
__device__ int slots_of_expert(const int32_t* idx, int nslots, int e, int* list, int lane) {
  int n = 0;
  for (int s0 = 0; s0 < nslots; s0 += 32) {
    const int s = s0 + lane;
    const bool hit = (s < nslots) && (idx[s] == e);
    const unsigned bal = __ballot_sync(0xffffffffu, hit);
    if (hit) list[n + __popc(bal & ((1u << lane) - 1u))] = s;
    n += __popc(bal);
  }
  return n;
}

__device__ __forceinline__ void store_out(const GemvParams& p, size_t i, float v) {
  if (p.c_dtype == 0)
    reinterpret_cast<float*>(p.C)[i] = v;
  else
    reinterpret_cast<__nv_bfloat16*>(p.C)[i] = __float2bfloat16_rn(v);
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int MR>
__global__ void __launch_bounds__(kThreads, 1) q4_gemv_kernel(GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemPlan plan = smem_plan<MR>(p.rows_per_split, p.list_cap);
  uint8_t* ring = smem + plan.ring;
  float* red = reinterpret_cast<float*>(smem + plan.red);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + plan.bars);
  uint64_t* empty = full + kStages;
  float* a_s = reinterpret_cast<float*>(smem + plan.a);
  int* list = reinterpret_cast<int*>(smem + plan.list);
  int* s_misc = list + p.list_cap;   // [0] ticket flag, [1] expert, [2] list length, [3] failed
  volatile int* s_fail = s_misc + 3;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int tile = blockIdx.x;
  const int split = blockIdx.y;
  const int z = blockIdx.z;

  // ---- resolve the problem of this CTA ----
  // mode GEMV: z = chunk of MR rows.  mode GATE_UP: z = 2*j + {0: gate, 1: up}
  // for the j-th active expert.  mode DOWN: z = j.
  int expert = 0;
  int nrows_total;   // rows of A for this problem (tokens / slots / M)
  const uint8_t* Bmat = p.B;
  if (p.mode == kModeGemv) {
    nrows_total = p.M;
  } else {
    // topk_idx may come from the kernel just before on the stream: the gate/up
    // kernel reads it only after that kernel has completed.  The down kernel
    // follows the gate/up kernel, whose CTAs all passed this wait before
    // letting it launch, so its early read is ordered too.
    if (p.mode == kModeGateUp) pdl_wait();
    if (warp == 0) {
      const int j = (p.mode == kModeGateUp) ? (z >> 1) : z;
      const int e =
          jth_active_expert(p.topk_idx, p.nslots, p.E, j, reinterpret_cast<unsigned*>(list), lane);
      __syncwarp();
      int n = 0;
      if (e >= 0) n = slots_of_expert(p.topk_idx, p.nslots, e, list, lane);
      if (lane == 0) {
        s_misc[1] = e;
        s_misc[2] = n;
      }
      // one CTA records routing indices outside [0, E)
      if (p.mode == kModeGateUp && blockIdx.x == 0 && blockIdx.y == 0 && z == 0) {
        bool bad = false;
        for (int s = lane; s < p.nslots; s += 32) {
          const int ee = p.topk_idx[s];
          bad |= (ee < 0 || ee >= p.E);
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.err, kDevErrIndex);
      }
    }
    __syncthreads();
    expert = s_misc[1];
    if (expert < 0) return;   // fewer distinct experts than grid slices
    nrows_total = s_misc[2];
    const int which = (p.mode == kModeGateUp) ? (z & 1) : 0;
    Bmat = (which ? p.B2 : p.B) + static_cast<size_t>(expert) * p.b_stride;
  }

  const int b0 = tile * kTileBlocks;
  const int tb = min(kTileBlocks, p.nb - b0);
  const int k0 = split * p.rows_per_split;
  const int rows = min(p.rows_per_split, p.K - k0);
  const int nstages = (rows + kRowsPerStage - 1) / kRowsPerStage;
  const int m_begin = (p.mode == kModeGemv) ? z * MR : 0;
  const int passes =
      (p.mode == kModeGemv) ? 1 : (nrows_total + MR - 1) / MR;   // expert tokens in chunks
  if (rows <= 0 || passes <= 0) return;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    *s_fail = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  StreamDesc sd;
  sd.B = Bmat;
  sd.nb = p.nb;
  sd.b0 = b0;
  sd.tb = tb;
  sd.k0 = k0;
  sd.rows = rows;
  sd.bulk = p.bulk != 0;

  if (warp == kConsumerWarps) {
    // ================= producer warp =================
    int gs = 0;
    for (int pass = 0; pass < passes; ++pass) {
      for (int s = 0; s < nstages; ++s, ++gs) {
        const int slot = gs % kStages;
        if (gs >= kStages) {
          bool ok = true;
          if (lane == 0) ok = wait_or_fail(&empty[slot], ((gs / kStages) - 1) & 1, s_fail, p.err);
          if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) return;   // failed: issue nothing more
        }
        produce_stage(sd, s, ring + slot * kStageBytes, &full[slot], lane);
      }
    }
    return;
  }

  // ================= consumer warps =================
  pdl_wait();   // A (and the workspace) may belong to the previous kernel
  const PairConsts kc = pair_consts();
  const int b = lane & 7;
  const int rp = warp * 4 + (lane >> 3);   // row phase 0..31
  const bool active_b = b < tb;
  const int ncols = p.N;
  int gs = 0;

  for (int pass = 0; pass < passes; ++pass) {
    // ---- rows of A for this pass, as fp32 in shared memory ----
    const int m0 = (p.mode == kModeGemv) ? m_begin : pass * MR;
    int mvalid = min(MR, nrows_total - m0);
    if (mvalid < 0) mvalid = 0;
    for (int i = tid; i < MR * rows; i += kConsumers) {
      const int m = i / rows;
      const int r = i - m * rows;
      float v = 0.f;
      if (m < mvalid) {
        size_t arow;
        if (p.mode == kModeGemv) arow = static_cast<size_t>(m0 + m);
        else if (p.mode == kModeGateUp) arow = static_cast<size_t>(list[m0 + m] / p.topk);
        else arow = static_cast<size_t>(list[m0 + m]);
        const size_t ai = arow * p.a_ld + k0 + r;
        v = (p.a_dtype == 0) ? reinterpret_cast<const float*>(p.A)[ai]
                             : bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.A)[ai]);
      }
      a_s[m * rows + r] = v;
    }
    consumers_sync();

    f32x2 acc[MR][16];
#pragma unroll
    for (int m = 0; m < MR; ++m)
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[m][i] = 0ull;

    for (int s = 0; s < nstages; ++s, ++gs) {
      const int slot = gs % kStages;
      const bool ready = wait_or_fail(&full[slot], (gs / kStages) & 1, s_fail, p.err);
      const uint8_t* stage = ring + slot * kStageBytes;
      const int r0 = s * kRowsPerStage;
      const int nr = min(kRowsPerStage, rows - r0);
#pragma unroll
      for (int i = 0; i < kRowsPerStage / kRowPhases; ++i) {
        const int r = rp + i * kRowPhases;
        if (ready && active_b && r < nr) {
          uint32_t dbits, qs[4];
          load_block_smem(stage + r * kRowBytes, b * kBlockBytes, dbits, qs);
          accumulate_block<MR>(acc, dbits, qs, a_s + r0 + r, rows, kc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ---- reduce the 32 row phases ----
    float colv[MR];
    reduce_tile<MR>(acc, red, warp, lane, tid, colv);
    const int col = b0 * kBlockCols + tid;   // tid = block * 32 + lane-in-block
    const bool col_ok = (tid < tb * kBlockCols) && (col < ncols);

    if (p.mode == kModeGemv) {
      if (p.nsplit == 1) {
        if (col_ok)
          for (int m = 0; m < mvalid; ++m) store_out(p, static_cast<size_t>(m0 + m) * ncols + col, colv[m]);
      } else {
        if (col_ok)
          for (int m = 0; m < mvalid; ++m)
            p.part[(static_cast<size_t>(split) * p.M + m0 + m) * ncols + col] = colv[m];
        unsigned* ticket = p.tickets + static_cast<size_t>(z) * gridDim.x + tile;
        if (last_arrival(ticket, p.nsplit, tid, s_misc)) {
          if (col_ok)
            for (int m = 0; m < mvalid; ++m) {
              float acc_s = 0.f;
              for (int sp = 0; sp < p.nsplit; ++sp)
                acc_s += __ldcg(p.part + (static_cast<size_t>(sp) * p.M + m0 + m) * ncols + col);
              store_out(p, static_cast<size_t>(m0 + m) * ncols + col, acc_s);
            }
        }
      }
    } else {
      // partial rows are indexed by slot; gate and up partials are separate planes
      const int which = (p.mode == kModeGateUp) ? (z & 1) : 0;
      float* part = p.part + static_cast<size_t>(which) * p.nsplit * p.nslots * ncols;
      if (col_ok)
        for (int m = 0; m < mvalid; ++m)
          part[(static_cast<size_t>(split) * p.nslots + list[m0 + m]) * ncols + col] = colv[m];
    }
    consumers_sync();   // red and a_s are reused by the next pass
  }

  if (p.mode != kModeGemv) {
    const int j = (p.mode == kModeGateUp) ? (z >> 1) : z;
    const unsigned arrivals = (p.mode == kModeGateUp) ? 2u * p.nsplit : p.nsplit;
    unsigned* ticket = p.tickets + static_cast<size_t>(j) * gridDim.x + tile;
    if (!last_arrival(ticket, arrivals, tid, s_misc)) return;
    const int col = b0 * kBlockCols + tid;
    if (!((tid < tb * kBlockCols) && (col < ncols))) return;
    const size_t plane = static_cast<size_t>(p.nsplit) * p.nslots * ncols;
    for (int m = 0; m < nrows_total; ++m) {
      const int slot = list[m];
      if (p.mode == kModeGateUp) {
        float g = 0.f, u = 0.f;
        for (int sp = 0; sp < p.nsplit; ++sp) {
          const size_t o = (static_cast<size_t>(sp) * p.nslots + slot) * ncols + col;
          g += __ldcg(p.part + o);
          u += __ldcg(p.part + plane + o);
        }
        // SiLU(g) * u, SiLU(g) = g * sigmoid(g)
        const float silu = g / (1.0f + __expf(-g));
        p.h[static_cast<size_t>(slot) * ncols + col] = silu * u;
      } else {
        float y = 0.f;
        for (int sp = 0; sp < p.nsplit; ++sp)
          y += __ldcg(p.part + (static_cast<size_t>(sp) * p.nslots + slot) * ncols + col);
        p.y[static_cast<size_t>(slot) * ncols + col] = y;
      }
    }
  }
}

// out[t, j] = sum_k w[t, k] * y[t*topk + k, j] in slot order; invalid slots skipped.
__global__ void __launch_bounds__(256) q4_moe_combine_kernel(float* out, const float* y,
                                                             const int32_t* idx, const float* w,
                                                             int T, int topk, int E, int H) {
  pdl_wait();
  pdl_launch_dependents();
  const size_t n = static_cast<size_t>(T) * H;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / H);
    const int j = static_cast<int>(i - static_cast<size_t>(t) * H);
    float acc = 0.f;
    for (int k = 0; k < topk; ++k) {
      const int s = t * topk + k;
      const int e = idx[s];
      if (e < 0 || e >= E) continue;
      acc = fmaf(w[s], y[static_cast<size_t>(s) * H + j], acc);
    }
    out[i] = acc;
  }
}

// ---------------------------------------------------------------------------
// Host-side launch helpers
// ---------------------------------------------------------------------------
template <int MR>
static cudaError_t launch_mr(const GemvParams& p, dim3 grid, cudaStream_t st, bool pdl) {
  const SmemPlan plan = smem_plan<MR>(p.rows_per_split, p.list_cap);
  cudaError_t e = cudaFuncSetAttribute(q4_gemv_kernel<MR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(plan.total));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = plan.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, q4_gemv_kernel<MR>, p);
}

cudaError_t launch_gemv(const GemvParams& p, int mr, dim3 grid, cudaStream_t st, bool pdl) {
  switch (mr) {
    case 1: return launch_mr<1>(p, grid, st, pdl);
    case 2: return launch_mr<2>(p, grid, st, pdl);
    case 4: return launch_mr<4>(p, grid, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

uint32_t gemv_smem_bytes(int mr, int rows_per_split, int list_cap) {
  switch (mr) {
    case 1: return smem_plan<1>(rows_per_split, list_cap).total;
    case 2: return smem_plan<2>(rows_per_split, list_cap).total;
    default: return smem_plan<4>(rows_per_split, list_cap).total;
  }
}

cudaError_t launch_moe_combine(float* out, const float* y, const int32_t* idx, const float* w,
                               int T, int topk, int E, int H, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  const size_t n = static_cast<size_t>(T) * H;
  size_t nblocks = (n + 255) / 256;
  if (nblocks > 1184) nblocks = 1184;
  cfg.gridDim = dim3(static_cast<unsigned>(nblocks));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, q4_moe_combine_kernel, out, y, idx, w, T, topk, E, H);
}

int gemv_tile_blocks() { return kTileBlocks; }

}  // namespace q4
