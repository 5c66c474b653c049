// Split-K Q4_0 GEMV for small M and the grouped routed-expert GEMVs (sm_103a).
//
// What it computes: C[i, j] = sum_k A[i, k] * (q[k, j] - 8) * d[k, j/32], the
// fused dequant-matmul loop of the C++ DeepSeek engine page (§3.4), over the
// block layout of its §2.2-§2.3 (K rows of ceil(N/32) 18-byte blocks, each
// block spanning 32 output columns of one row).
//
// How (GB300-first, not the page's CPU loop):
//  * A CTA owns a column tile of 8*BPT blocks (256*BPT columns) and a
//    contiguous slice of rows (split-K).  One producer warp streams the slice
//    into a shared-memory ring, one 18 KB box (64 or 128 rows) per TMA tensor copy
//    (cp.async.bulk.tensor, completion on mbarriers); eight consumer warps
//    decode nibbles in registers and accumulate in fp32 with packed fp32x2
//    arithmetic.  Eight consecutive lanes share a row, each owning BPT
//    consecutive blocks; a warp covers four rows, the CTA 32.  Weights whose
//    rows are not 16-byte aligned (ceil(N/32) not a multiple of 8) are staged
//    by the producer warp with plain loads instead.
//  * The splits of one column tile run as one thread-block cluster (at most
//    16 CTAs).  Each CTA leaves its partial sums in its own shared memory;
//    after a cluster barrier the cluster's rank-0 CTA adds them over DSMEM in
//    fixed split order (split 0, 1, ...) and writes the result, so the sum is
//    deterministic and needs no global scratch and no global round trip.
//  * Programmatic dependent launch: the producer streams weights before
//    griddepcontrol.wait; A is read, and workspace written, only after.
//
// Nibble decoding (exact, one AND per weight): a word masked down to its
// nibble q at bits 4p..4p+3 (p <= 3), read as an fp32 bit pattern, is the
// subnormal number q * 16^p * 2^-149, exactly.  Multiplying it by
// a' = (a * 2^64) * d in a fused multiply-add adds a*d*q*16^p*2^-85 with one
// rounding: subnormal operands are taken at full precision (no flush to zero)
// and, for |a*d| >= 2^-41, the product is a normal number.  The -8 of every
// code is not applied per weight: C = sum a*d*q - 8 * sum a*d, and each
// thread keeps sum a' for each of its blocks and subtracts 8 times it once,
// after its last stage, when it also removes the power-of-two factors.
// Preconditions: |a| and |a*d| below 2^64 (so that a' stays finite).  Word w
// (columns 8t..8t+7 as nibbles 0..7) is decoded as pairs (0,1) and (2,3) of w
// and of w >> 16, so only the positions p = 0..3 occur.
//
// The routed-expert kernels (KTransformers DeepSeek-V2 page, «优化三»: 6 of
// 160 experts per token, run as batched GEMVs; «规则二»: gate -> top-k) reuse
// the same core: every CTA re-derives, from topk_idx, the sorted list of
// experts in use and the (token, slot) list of its expert, so no routing
// kernel and no host synchronisation is needed.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "q4_device.cuh"
#include "q4_gemv_core.cuh"
#include "q4_kernels.h"

namespace q4 {

// ---------------------------------------------------------------------------
// Shared-memory plan
// ---------------------------------------------------------------------------
struct SmemPlan {
  uint32_t ring, red, cpart, bars, a, list, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// senders: the CTAs of a cluster (the split count; twice it for gate/up),
// whose partial sums of every column cluster rank 0 receives.
template <int MR, int BPT, bool BIG, int FMT>
__host__ __device__ inline SmemPlan smem_plan(int rows_per_split, int list_cap, int senders) {
  using T = TileCfg<BPT, BIG, FMT>;
  SmemPlan p;
  p.ring = 0;   // the dynamic shared-memory base is 128-byte aligned
  p.red = align_up(T::kStages * T::kStageBytes, 16);
  p.cpart = p.red + Crew<MR>::kWarps * MR * kRedStride<BPT> * 4;
  p.bars = p.cpart + MR * T::kCols * senders * 4;   // partials received from the cluster
  p.a = p.bars + 2 * T::kStages * 8;
  p.list = align_up(p.a + MR * align_up(rows_per_split, T::kRows) * 4, 16);
  p.total = align_up(p.list + list_cap * 4 + 64, 128);
  return p;
}


// Waits on `bar` (bounded_wait: gives up if the CTA failed or after the wait
// limit, recording the timeout).  Threads never leave their loops early, so
// every named barrier is still reached.
__device__ __forceinline__ bool wait_or_fail(uint64_t* bar, uint32_t parity, volatile int* fail,
                                             unsigned* err) {
  return bounded_wait(bar, parity, fail, err);
}

// ---------------------------------------------------------------------------
// Producer: stage rows [k0 + s*32, +32) of the tile into ring slot `stage`
// ---------------------------------------------------------------------------
struct StreamDesc {
  const uint8_t* B;   // matrix base
  const void* tmap;   // tensor map of the weight stack (TMA path) or null
  const void* tmap2;  // planar: tensor map of the scale plane
  long long qs_offset;   // planar: byte offset of the nibble plane from B
  int expert;         // expert index in the stack (0 for a single matrix)
  int nb;             // blocks per row
  int b0, tb;         // first block of the tile, blocks in the tile
  int k0, rows;       // row slice
};

template <int BPT, bool BIG, int FMT>
__device__ __forceinline__ void produce_stage(const StreamDesc& sd, int s, uint8_t* stage,
                                              uint64_t* full, int lane) {
  using T = TileCfg<BPT, BIG, FMT>;
  constexpr int kBB = Fmt<FMT>::kBytes;
  const int r0 = s * T::kRows;
  if constexpr (Fmt<FMT>::kPlanar) {
    if (sd.tmap) {
      // two boxes of kRows rows: the nibbles (uint32, 4 per block) and the
      // scales (uint16, 1 per block); rows past K read as zero
      if (lane == 0) {
        mbar_arrive_expect_tx(full, T::kStageBytes);
        tma_load_3d(stage, sd.tmap, sd.b0 * 4, sd.k0 + r0, 0, full);
        tma_load_3d(stage + T::kQsBytes, sd.tmap2, sd.b0, sd.k0 + r0, 0, full);
      }
    } else {
      // 16-byte nibble units and 2-byte scales; rows past the slice and
      // blocks past the row are written as zeros, as the tensor copies do
      const int nr = min(T::kRows, sd.rows - r0);
      const uint4* qsrc = reinterpret_cast<const uint4*>(sd.B + sd.qs_offset);
      const uint16_t* dsrc = reinterpret_cast<const uint16_t*>(sd.B);
      uint4* qdst = reinterpret_cast<uint4*>(stage);
      uint16_t* ddst = reinterpret_cast<uint16_t*>(stage + T::kQsBytes);
      for (int u = lane; u < T::kRows * T::kBlocks; u += 32) {
        const int r = u / T::kBlocks;
        const int b = u - r * T::kBlocks;
        const bool in = (r < nr && b < sd.tb);
        const size_t e = static_cast<size_t>(sd.k0 + r0 + r) * sd.nb + sd.b0 + b;
        qdst[u] = in ? __ldg(qsrc + e) : make_uint4(0u, 0u, 0u, 0u);
        ddst[u] = in ? __ldg(dsrc + e) : static_cast<uint16_t>(0);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(full);
    }
    return;
  }
  if (sd.tmap) {
    // one box of kRows rows x kRowBytes; rows past K and blocks past the row
    // read as zero (a slice is a whole number of boxes, except the last one,
    // which ends at K)
    if (lane == 0) {
      mbar_arrive_expect_tx(full, T::kStageBytes);
      tma_load_3d(stage, sd.tmap, sd.b0 * kBB / Fmt<FMT>::kTmaElem, sd.k0 + r0, sd.expert, full);
    }
  } else {
    // 2-byte aligned rows: copy with 16-bit loads (every block offset is even);
    // rows past the slice and blocks past the row are written as zeros, as
    // the tensor copy does, so that the consumers need no bounds checks
    const int nr = min(T::kRows, sd.rows - r0);
    const int halves = sd.tb * (kBB / 2);
    for (int r = 0; r < T::kRows; ++r) {
      const uint16_t* src = reinterpret_cast<const uint16_t*>(
          sd.B + (static_cast<size_t>(sd.k0 + r0 + r) * sd.nb + sd.b0) * kBB);
      uint16_t* dst = reinterpret_cast<uint16_t*>(stage + r * T::kRowBytes);
      for (int h = lane; h < T::kRowBytes / 2; h += 32)
        dst[h] = (r < nr && h < halves) ? __ldg(src + h) : static_cast<uint16_t>(0);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(full);
  }
}

template <int MR>
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(Crew<MR>::kConsumers) : "memory");
}

// ---------------------------------------------------------------------------
// Reduction of the row phases of a tile: warp shuffles (halving exchange
// over the four rows of a warp), then across warps through shared memory.
// out[m][i] = column tid + 256*i of the tile for row m.
// ---------------------------------------------------------------------------
template <int MR, int BPT, int FMT>
__device__ __forceinline__ void reduce_tile(f32x2 (&acc)[MR][16 * BPT], float* red, int warp,
                                            int lane, int tid, float (&out)[MR][BPT]) {
  constexpr int P = 16 * BPT;   // pairs per thread
  const bool hi16 = (lane & 16) != 0;
  const bool hi8 = (lane & 8) != 0;
  const int pi = lane & 7;
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    f32x2 h[P / 2];
#pragma unroll
    for (int i = 0; i < P / 2; ++i) {
      const f32x2 send = hi16 ? acc[m][i] : acc[m][P / 2 + i];
      const f32x2 keep = hi16 ? acc[m][P / 2 + i] : acc[m][i];
      h[i] = add2(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
    f32x2 q[P / 4];
#pragma unroll
    for (int i = 0; i < P / 4; ++i) {
      const f32x2 send = hi8 ? h[i] : h[P / 4 + i];
      const f32x2 keep = hi8 ? h[P / 4 + i] : h[i];
      q[i] = add2(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
    // the lane now holds pairs j0 + i, i < P/4, of its thread's accumulators
    const int j0 = (hi16 ? P / 2 : 0) + (hi8 ? P / 4 : 0);
    float* dst = red + (warp * MR + m) * kRedStride<BPT> + pi * BPT * 33;
#pragma unroll
    for (int i = 0; i < P / 4; ++i) {
      // pair j = j0 + i: block j >> 4, columns acc_col_pair(j & 15) and + kPairGap
      const int j = j0 + i;
      const int c = 33 * (j >> 4) + acc_col_pair<FMT>(j & 15);
      float v0, v1;
      unpack2(q[i], v0, v1);
      dst[c] = v0;
      dst[c + Fmt<FMT>::kPairGap] = v1;
    }
  }
  consumers_sync<MR>();
  // threads 0..255 finish columns tid + 256*i; column c = 32*(BPT*pi + blk) + cc
  const int t = tid & 255;
#pragma unroll
  for (int m = 0; m < MR; ++m)
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      const int c = t + 256 * i;
      const int off = (c >> 5) * 33 + (c & 31);
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < Crew<MR>::kWarps; ++w) s += red[(w * MR + m) * kRedStride<BPT> + off];
      out[m][i] = s;
    }
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
template <int MODE, int MR, int BPT, bool BIG, int FMT>
__global__ void __launch_bounds__(Crew<MR>::kThreads, 1)
    q4_gemv_kernel(const __grid_constant__ GemvParams p) {
  using T = TileCfg<BPT, BIG, FMT>;
  constexpr int kGroups = Crew<MR>::kWarps / T::kGroupWarps;
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemPlan plan = smem_plan<MR, BPT, BIG, FMT>(p.rows_per_split, p.list_cap,
                                                     MODE == kModeGateUp ? 2 * p.nsplit : p.nsplit);
  uint8_t* ring = smem + plan.ring;
  float* red = reinterpret_cast<float*>(smem + plan.red);
  float* cpart = reinterpret_cast<float*>(smem + plan.cpart);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + plan.bars);
  uint64_t* empty = full + T::kStages;
  float* a_s = reinterpret_cast<float*>(smem + plan.a);
  int* list = reinterpret_cast<int*>(smem + plan.list);
  int* s_misc = list + p.list_cap;   // [0] unused, [1] expert, [2] list length, [3] failed
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
  if constexpr (MODE == kModeGemv) {
    nrows_total = p.M;
  } else {
    // topk_idx may come from the kernel just before on the stream: the gate/up
    // kernel reads it only after that kernel has completed.  The down kernel
    // follows the gate/up kernel, whose CTAs all passed this wait before
    // letting it launch, so its early read is ordered too.
    if (MODE == kModeGateUp) pdl_wait();
    if (warp == 0) {
      const int j = (MODE == kModeGateUp) ? (z >> 1) : z;
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
      if (MODE == kModeGateUp && blockIdx.x == 0 && blockIdx.y == 0 && z == 0) {
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
  }
  const int which = (MODE == kModeGateUp) ? (z & 1) : 0;   // gate (0) or up (1)

  const int b0 = tile * T::kBlocks;
  const int tb = min(T::kBlocks, p.nb - b0);
  const int k0 = split * p.rows_per_split;
  const int rows = min(p.rows_per_split, p.K - k0);
  const int nstages = (rows + T::kRows - 1) / T::kRows;
  const int m_begin = (MODE == kModeGemv) ? z * MR : 0;
  const int passes = (MODE == kModeGemv) ? 1 : (nrows_total + MR - 1) / MR;
  if (rows <= 0 || passes <= 0) return;

  if (tid == 0) {
    for (int i = 0; i < T::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], T::kGroupWarps);
    }
    *s_fail = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == Crew<MR>::kWarps) {
    // ================= producer warp =================
    StreamDesc sd;
    sd.tmap = p.use_tma ? static_cast<const void*>(&p.tmap[which]) : nullptr;
    sd.tmap2 = (Fmt<FMT>::kPlanar && p.use_tma) ? static_cast<const void*>(&p.tmap[1]) : nullptr;
    sd.qs_offset = p.qs_offset;
    sd.expert = expert;
    sd.B = (which ? p.B2 : p.B) + static_cast<size_t>(expert) * p.b_stride;
    sd.nb = p.nb;
    sd.b0 = b0;
    sd.tb = tb;
    sd.k0 = k0;
    sd.rows = rows;
    int gs = 0;
    bool failed = false;
    for (int pass = 0; pass < passes; ++pass) {
      for (int s = 0; s < nstages && !failed; ++s, ++gs) {
        const int slot = gs % T::kStages;
        if (gs >= T::kStages) {
          bool ok = true;
          if (lane == 0)
            ok = wait_or_fail(&empty[slot], ((gs / T::kStages) - 1) & 1, s_fail, p.err);
          failed = !__shfl_sync(0xffffffffu, ok ? 1 : 0, 0);   // failed: issue nothing more
          if (failed) break;
        }
        produce_stage<BPT, BIG, FMT>(sd, s, ring + slot * T::kStageBytes, &full[slot], lane);
      }
      // the cluster barriers of this pass's combine (see the consumers)
      cluster_sync();
      if (pass + 1 < passes) cluster_sync();
    }
    return;
  }

  // ================= consumer warps =================
  pdl_wait();   // A (and the workspace) may belong to the previous kernel
  const DecodeConsts kc = load_consts(p);
  const int pi = lane & 7;                                 // lane within its row
  const int group = warp / T::kGroupWarps;                 // stages s = group mod kGroups
  // row phase: the thread decodes rows rp, rp + kGroupRows, ... of each stage
  const int rp = (warp % T::kGroupWarps) * 4 + (lane >> 3);
  const uint32_t boff = static_cast<uint32_t>(pi * BPT * Fmt<FMT>::kBytes);
  const bool odd = (boff & 2u) != 0;
  const int ncols = p.N;
  const int tile_cols = tb * kBlockCols;
  const int a_ld_s = nstages * T::kRows;   // rows of A in shared memory, stage-padded

  for (int pass = 0; pass < passes; ++pass) {
    // ---- rows of A for this pass, as fp32 in shared memory ----
    const int m0 = (MODE == kModeGemv) ? m_begin : pass * MR;
    int mvalid = min(MR, nrows_total - m0);
    if (mvalid < 0) mvalid = 0;
    for (int i = tid; i < MR * a_ld_s; i += Crew<MR>::kConsumers) {
      const int m = i / a_ld_s;
      const int r = i - m * a_ld_s;
      float v = 0.f;
      if (m < mvalid && r < rows) {
        size_t arow;
        if (MODE == kModeGemv) arow = static_cast<size_t>(m0 + m);
        else if (MODE == kModeGateUp) arow = static_cast<size_t>(list[m0 + m] / p.topk);
        else arow = static_cast<size_t>(list[m0 + m]);
        const size_t ai = arow * p.a_ld + k0 + r;
        v = (p.a_dtype == 0) ? reinterpret_cast<const float*>(p.A)[ai]
                             : bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.A)[ai]);
        v *= kAScale;
      }
      a_s[m * a_ld_s + r] = v;
    }
    consumers_sync<MR>();

    f32x2 acc[MR][16 * BPT];
    float sad[MR][BPT];
#pragma unroll
    for (int m = 0; m < MR; ++m) {
#pragma unroll
      for (int i = 0; i < 16 * BPT; ++i) acc[m][i] = 0ull;
#pragma unroll
      for (int bb = 0; bb < BPT; ++bb) sad[m][bb] = 0.f;
    }

    for (int s = group; s < nstages; s += kGroups) {
      const int gs = pass * nstages + s;   // the producer's stage counter
      const int slot = gs % T::kStages;
      // every lane waits on the stage itself (no divergence, no broadcast).
      // Rows past the slice need no check: they exist only past K, where the
      // stage holds zeros and the rows of A are zero too.
      const bool ready = wait_or_fail(&full[slot], (gs / T::kStages) & 1, s_fail, p.err);
      if (ready) {
        // two rows at a time: more would keep too many words live for MR > 1
#pragma unroll 2
        for (int rr = 0; rr < T::kRowsPerThread; ++rr) {
          const int rs = rp + rr * T::kGroupRows;   // row within the stage
          uint32_t dbits[BPT], qs[BPT][Fmt<FMT>::kWords];
          if constexpr (Fmt<FMT>::kPlanar) {
            const uint8_t* st = ring + slot * T::kStageBytes;
            load_planar<BPT>(st + (rs * T::kBlocks + pi * BPT) * 16,
                             st + T::kQsBytes + (rs * T::kBlocks + pi * BPT) * 2, dbits, qs);
          } else {
            const uint8_t* row = ring + slot * T::kStageBytes + rs * T::kRowBytes;
            load_blocks<BPT, FMT>(row, boff, odd, dbits, qs);
          }
          const float* a = a_s + s * T::kRows + rs;
#pragma unroll
          for (int bb = 0; bb < BPT; ++bb)
            accumulate_block<MR, BPT, FMT>(acc, sad, bb, dbits[bb], qs[bb], a, a_ld_s, kc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ---- reduce the row phases ----
    finish_acc<MR, BPT, FMT>(acc, sad);
    float colv[MR][BPT];
    reduce_tile<MR, BPT, FMT>(acc, red, warp, lane, tid, colv);

    // ---- combine the splits of the cluster in fixed order ----
    // Cluster rank 0 receives every sender's partial of every column, as
    // [m][sender][column], and finishes the tile alone, adding in fixed rank
    // order (gate/up: senders 0..ns-1 hold gate partials, ns..2ns-1 up
    // partials).  After the last pass the other CTAs exit right after the
    // barrier, so that their SMs can take the next kernel's clusters while
    // rank 0 adds and stores.
    {
      const int rank = static_cast<int>(cluster_ctarank());
      const int ns = p.nsplit;
      const int csize = (MODE == kModeGateUp) ? 2 * ns : ns;
      if (tid < 256) {
#pragma unroll
        for (int m = 0; m < MR; ++m)
#pragma unroll
          for (int i = 0; i < BPT; ++i) {
            float* dst = cpart + (m * csize + rank) * T::kCols + tid + 256 * i;
            st_peer(peer_addr(dst, 0), colv[m][i]);
          }
      }
      cluster_sync();   // every partial has reached rank 0
      if (rank == 0) {
        for (int c = tid; c < tile_cols; c += Crew<MR>::kConsumers) {
          const int col = b0 * kBlockCols + c;
          if (col >= ncols) break;
          for (int m = 0; m < mvalid; ++m) {
            const float* v = cpart + m * csize * T::kCols + c;
            if constexpr (MODE == kModeGateUp) {
              float g = 0.f, u = 0.f;
              for (int sp = 0; sp < ns; ++sp) {
                g += v[sp * T::kCols];
                u += v[(ns + sp) * T::kCols];
              }
              // SiLU(g) * u, SiLU(g) = g * sigmoid(g)
              const float silu = g / (1.0f + __expf(-g));
              const size_t o = static_cast<size_t>(list[m0 + m]) * ncols + col;
              p.h[o] = silu * u;
              if (p.g_trace) {
                p.g_trace[o] = g;
                p.u_trace[o] = u;
              }
            } else {
              float acc_s = 0.f;
              for (int sp = 0; sp < ns; ++sp) acc_s += v[sp * T::kCols];
              if constexpr (MODE == kModeGemv)
                store_out(p, static_cast<size_t>(m0 + m) * ncols + col, acc_s);
              else
                p.y[static_cast<size_t>(list[m0 + m]) * ncols + col] = acc_s;
            }
          }
        }
      }
      // another pass will push into rank 0's buffer again: wait until it has
      // read this pass's partials
      if (pass + 1 < passes) cluster_sync();
    }
  }
}

// out[t, j] = sum_k w[t, k] * y[t*topk + k, j] in slot order (invalid slots
// skipped), then + addend[t, j] when an addend is given.
__global__ void __launch_bounds__(256) q4_moe_combine_kernel(float* out, const float* y,
                                                             const int32_t* idx, const float* w,
                                                             const float* addend, int T, int topk,
                                                             int E, int H) {
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
    out[i] = addend ? acc + addend[i] : acc;
  }
}

// h[i] = SiLU(g[i]) * u[i] = g / (1 + exp(-g)) * u, in fp32 (the expert
// chain's middle step when gate and up run as separate matmuls).
__global__ void __launch_bounds__(256) q4_silu_mul_kernel(float* h, const float* g, const float* u,
                                                          size_t n) {
  pdl_wait();
  pdl_launch_dependents();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float gv = g[i];
    h[i] = gv / (1.0f + __expf(-gv)) * u[i];
  }
}

cudaError_t launch_silu_mul(float* h, const float* g, const float* u, size_t n, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  size_t nblocks = (n + 255) / 256;
  if (nblocks > 1184) nblocks = 1184;
  cfg.gridDim = dim3(static_cast<unsigned>(nblocks));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, q4_silu_mul_kernel, h, g, u, n);
}

// ---------------------------------------------------------------------------
// Host-side launch helpers
// ---------------------------------------------------------------------------
template <int MODE, int MR, int BPT, bool BIG, int FMT>
static cudaError_t launch_cfg(const GemvParams& p, dim3 grid, dim3 cluster, cudaStream_t st,
                              bool pdl) {
  const SmemPlan plan = smem_plan<MR, BPT, BIG, FMT>(p.rows_per_split, p.list_cap,
                                                     MODE == kModeGateUp ? 2 * p.nsplit : p.nsplit);
  auto fn = q4_gemv_kernel<MODE, MR, BPT, BIG, FMT>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(plan.total));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Crew<MR>::kThreads);
  cfg.dynamicSmemBytes = plan.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster.x;
  attr[0].val.clusterDim.y = cluster.y;
  attr[0].val.clusterDim.z = cluster.z;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

template <int MODE, bool BIG, int FMT>
static cudaError_t launch_mode(const GemvParams& p, int mr, int bpt, dim3 grid, dim3 cluster,
                               cudaStream_t st, bool pdl) {
  if (bpt == 2 && mr == 1) return launch_cfg<MODE, 1, 2, BIG, FMT>(p, grid, cluster, st, pdl);
  if (bpt == 1 && mr == 1) return launch_cfg<MODE, 1, 1, BIG, FMT>(p, grid, cluster, st, pdl);
  if (bpt == 1 && mr == 2) return launch_cfg<MODE, 2, 1, BIG, FMT>(p, grid, cluster, st, pdl);
  if (bpt == 1 && mr == 4) return launch_cfg<MODE, 4, 1, BIG, FMT>(p, grid, cluster, st, pdl);
  return cudaErrorInvalidValue;
}

template <bool BIG>
static cudaError_t launch_big(const GemvParams& p, int mr, int bpt, dim3 grid, dim3 cluster,
                              cudaStream_t st, bool pdl) {
  switch (p.mode) {
    case kModeGemv: return launch_mode<kModeGemv, BIG, kFmtQ4>(p, mr, bpt, grid, cluster, st, pdl);
    case kModeGateUp: return launch_mode<kModeGateUp, BIG, kFmtQ4>(p, mr, bpt, grid, cluster, st, pdl);
    case kModeDown: return launch_mode<kModeDown, BIG, kFmtQ4>(p, mr, bpt, grid, cluster, st, pdl);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemv(const GemvParams& p, int mr, int bpt, bool big, int fmt, dim3 grid,
                        dim3 cluster, cudaStream_t st, bool pdl) {
  if (fmt == kFmtQ8) {   // the plain GEMV, 32-row stages only
    if (p.mode != kModeGemv || big) return cudaErrorInvalidValue;
    return launch_mode<kModeGemv, false, kFmtQ8>(p, mr, bpt, grid, cluster, st, pdl);
  }
  if (fmt == kFmtQ4P) {   // the plain GEMV
    if (p.mode != kModeGemv) return cudaErrorInvalidValue;
    return big ? launch_mode<kModeGemv, true, kFmtQ4P>(p, mr, bpt, grid, cluster, st, pdl)
               : launch_mode<kModeGemv, false, kFmtQ4P>(p, mr, bpt, grid, cluster, st, pdl);
  }
  return big ? launch_big<true>(p, mr, bpt, grid, cluster, st, pdl)
             : launch_big<false>(p, mr, bpt, grid, cluster, st, pdl);
}

template <bool BIG, int FMT>
static void pick_instance(int mode, int mr, int bpt, int rows_per_split, int list_cap,
                          int senders, const void** fn, uint32_t* smem) {
#define Q4_PICK(MO)                                                                      \
  if (mode == MO) {                                                                      \
    if (bpt == 2 && mr == 1) *fn = (const void*)q4_gemv_kernel<MO, 1, 2, BIG, FMT>;      \
    else if (bpt == 1 && mr == 1) *fn = (const void*)q4_gemv_kernel<MO, 1, 1, BIG, FMT>; \
    else if (bpt == 1 && mr == 2) *fn = (const void*)q4_gemv_kernel<MO, 2, 1, BIG, FMT>; \
    else if (bpt == 1 && mr == 4) *fn = (const void*)q4_gemv_kernel<MO, 4, 1, BIG, FMT>; \
  }
  Q4_PICK(kModeGemv)
  if constexpr (FMT == kFmtQ4) {
    Q4_PICK(kModeGateUp)
    Q4_PICK(kModeDown)
  }
#undef Q4_PICK
  if (bpt == 2) *smem = smem_plan<1, 2, BIG, FMT>(rows_per_split, list_cap, senders).total;
  else if (mr == 1) *smem = smem_plan<1, 1, BIG, FMT>(rows_per_split, list_cap, senders).total;
  else if (mr == 2) *smem = smem_plan<2, 1, BIG, FMT>(rows_per_split, list_cap, senders).total;
  else *smem = smem_plan<4, 1, BIG, FMT>(rows_per_split, list_cap, senders).total;
}

int max_active_clusters(int mode, int mr, int bpt, bool big, int fmt, int rows_per_split,
                        int list_cap, dim3 cluster) {
  // occupancy query for the kernel instance that launch_gemv would pick
  const void* fn = nullptr;
  uint32_t smem = 0;
  const int senders = static_cast<int>(cluster.y * cluster.z);
  if (fmt == kFmtQ8) {
    if (big || mode != kModeGemv) return 0;
    pick_instance<false, kFmtQ8>(mode, mr, bpt, rows_per_split, list_cap, senders, &fn, &smem);
  } else if (fmt == kFmtQ4P) {
    if (mode != kModeGemv) return 0;
    if (big) pick_instance<true, kFmtQ4P>(mode, mr, bpt, rows_per_split, list_cap, senders, &fn, &smem);
    else pick_instance<false, kFmtQ4P>(mode, mr, bpt, rows_per_split, list_cap, senders, &fn, &smem);
  } else if (big) {
    pick_instance<true, kFmtQ4>(mode, mr, bpt, rows_per_split, list_cap, senders, &fn, &smem);
  } else {
    pick_instance<false, kFmtQ4>(mode, mr, bpt, rows_per_split, list_cap, senders, &fn, &smem);
  }
  if (!fn) return 0;
  // a failed query leaves no error pending for the caller's next launch
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess ||
      cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    cudaGetLastError();   // tolerated: the query below then counts what fits
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster.x, cluster.y, cluster.z);
  cfg.blockDim = dim3(mr == 1 ? Crew<1>::kThreads : mr == 2 ? Crew<2>::kThreads : Crew<4>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster.x;
  attr[0].val.clusterDim.y = cluster.y;
  attr[0].val.clusterDim.z = cluster.z;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_moe_combine(float* out, const float* y, const int32_t* idx, const float* w,
                               const float* addend, int T, int topk, int E, int H,
                               cudaStream_t st, bool pdl) {
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
  return cudaLaunchKernelEx(&cfg, q4_moe_combine_kernel, out, y, idx, w, addend, T, topk, E, H);
}

int gemv_tile_blocks(int bpt) { return kLanesPerRow * bpt; }

int gemv_stage_rows(int bpt, bool big) {
  if (big) return bpt == 2 ? TileCfg<2, true>::kRows : TileCfg<1, true>::kRows;
  return bpt == 2 ? TileCfg<2, false>::kRows : TileCfg<1, false>::kRows;
}

void fill_decode_consts(GemvParams& p, int fmt) {
  if (fmt == kFmtQ8) {
    for (int i = 0; i < 3; ++i) p.kmask[i] = 0xFFu << (8 * i);
    p.kmask[3] = 0x80808080u;   // sign flips: b = q + 128 in every byte
  } else {
    for (int i = 0; i < 4; ++i) p.kmask[i] = 0xFu << (4 * i);
  }
}

// cuTensorMapEncodeTiled from the driver (null if unavailable).
static PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return encode;
}

bool encode_weight_tmap(CUtensorMap* map, const void* base, int64_t K, int64_t nb,
                        int64_t experts, int64_t matrix_bytes, int bpt, bool big, int fmt) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode) return false;
  if (nb % kLanesPerRow != 0) return false;
  // Q4_0: uint16 elements, a row is nb*9 of them; Q8_0: uint32 elements, a
  // row is nb*34/4 (nb is a multiple of 8, so the tile starts, 8*bpt blocks
  // apart, are whole elements and 16-byte aligned).  A box is one tile row
  // segment (8*bpt blocks) by the stage's rows.
  const bool q8 = (fmt == kFmtQ8);
  const int64_t bb = q8 ? Fmt<kFmtQ8>::kBytes : Fmt<kFmtQ4>::kBytes;
  const int64_t es = q8 ? Fmt<kFmtQ8>::kTmaElem : Fmt<kFmtQ4>::kTmaElem;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(nb * bb / es), static_cast<cuuint64_t>(K),
                              static_cast<cuuint64_t>(experts)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(nb * bb),
                                 static_cast<cuuint64_t>(matrix_bytes)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kLanesPerRow * bpt * bb / es),
                             static_cast<cuuint32_t>(q8 ? 32 : gemv_stage_rows(bpt, big)), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = encode(map, q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16,
                            3, const_cast<void*>(base), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_planar_tmaps(CUtensorMap* maps, const void* base, int64_t K, int64_t nb,
                         int64_t qs_offset, int bpt, bool big) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tmap_encoder();
  if (!encode) return false;
  // nb % 8 == 0 makes the scale rows (nb * 2 bytes) 16-byte multiples and
  // every tile start (8*bpt blocks apart) a whole, 16-byte aligned element
  if (nb % kLanesPerRow != 0 || qs_offset % 16 != 0) return false;
  const cuuint32_t rows = static_cast<cuuint32_t>(gemv_stage_rows(bpt, big));
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  // the nibble plane: uint32 [1][K][nb*4], boxes of 8*bpt blocks (32*bpt words)
  const cuuint64_t qdims[3] = {static_cast<cuuint64_t>(nb * 4), static_cast<cuuint64_t>(K), 1u};
  const cuuint64_t qstrides[2] = {static_cast<cuuint64_t>(nb * 16),
                                  static_cast<cuuint64_t>(K * nb * 16)};
  const cuuint32_t qbox[3] = {static_cast<cuuint32_t>(kLanesPerRow * bpt * 4), rows, 1u};
  CUresult r = encode(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT32, 3,
                      const_cast<uint8_t*>(static_cast<const uint8_t*>(base) + qs_offset), qdims,
                      qstrides, qbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  // the scale plane: uint16 [1][K][nb], boxes of 8*bpt scales
  const cuuint64_t ddims[3] = {static_cast<cuuint64_t>(nb), static_cast<cuuint64_t>(K), 1u};
  const cuuint64_t dstrides[2] = {static_cast<cuuint64_t>(nb * 2),
                                  static_cast<cuuint64_t>(K * nb * 2)};
  const cuuint32_t dbox[3] = {static_cast<cuuint32_t>(kLanesPerRow * bpt), rows, 1u};
  r = encode(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), ddims,
             dstrides, dbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace q4
