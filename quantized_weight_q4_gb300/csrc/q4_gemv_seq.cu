// Persistent Q4_0 decode: a whole sequence of M = 1 GEMVs in one launch.
//
// What it computes: for every op i of the sequence, C_i[j] = sum_k A_i[k] *
// W_i[k, j] with W_i in the block layout of the C++ DeepSeek engine page
// (§2.2-§2.3, the fused loop of §3.4): the token-by-token decode of its §2.1
// streams every weight matrix of the model once per token, one GEMV each.
//
// How (GB300-first): instead of one launch per matrix, whose pipeline fill,
// reduction and drain leave the HBM idle for microseconds each time, one
// resident grid (two CTAs per SM) streams all of the sequence's weights.
//  * The work is cut into units of (op, column tile of 16 blocks = 512
//    columns, K slice of 64 to 4096 rows, chosen per op).  Units are numbered op by op, and within
//    an op tile by tile; a global counter hands them out in that order.
//  * In each CTA a producer warp issues one TMA tensor copy per 64-row stage
//    (18 KB) into a ring, and a second warp copies the stage's 64 entries of A
//    (cp.async.bulk) onto the same mbarrier once the op's dependencies have
//    completed, so that weights keep streaming while an op waits for its
//    input.  Eight consumer warps decode and accumulate with the same exact
//    arithmetic as the split-K GEMV (q4_gemv_core.cuh).
//  * At the end of a unit the consumers reduce their partial sums over the
//    CTA, write the unit's 512 partial sums to global scratch and take a
//    ticket of its column tile; the CTA that takes the tile's last ticket adds
//    the slices' partials in slice order (deterministic), stores C and counts
//    the tile as done for the op.  An op whose dependency list names earlier
//    ops reads its A only after all their tiles are done.
//  * Every wait is bounded; on a timeout the CTA records Q4_DEVERR_TIMEOUT and
//    its warps stop.  The consumers synchronise through an mbarrier with a
//    bounded wait rather than a named barrier, so that no thread can be left
//    waiting on one that has stopped.
#include <cstdint>
#include <cstring>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "q4_device.cuh"
#include "q4_gemv_core.cuh"
#include "q4_kernels.h"

namespace q4 {
namespace seq {

constexpr int kBPT = 2;                                  // blocks per consumer thread
constexpr int kTileBlocks = kLanesPerRow * kBPT;         // 16 blocks per column tile
constexpr int kTileCols = kTileBlocks * kBlockCols;      // 512 columns
constexpr int kRowBytes = kTileBlocks * kBlockBytes;     // 288 bytes of a tile row
constexpr int kStageRows = 64;
constexpr int kStageBytes = kStageRows * kRowBytes;      // 18432 bytes
constexpr int kDefaultSliceStages = 8;                   // stages of a unit by default
constexpr int kMaxSliceStages = 64;                      // stages of the longest unit
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 64;                // + producer warp + A warp
constexpr int kRowsPerPass = kConsumerWarps * 32 / kLanesPerRow;   // 32
constexpr int kRowsPerThread = kStageRows / kRowsPerPass;          // 2
constexpr int kARowBytes = 4;                            // A slots hold up to fp32
static_assert(kStageBytes % 128 == 0, "TMA destinations must be 128-byte aligned");
static_assert(kTileCols == 2 * kConsumers, "each consumer thread finishes two columns");

// What the producer tells the A warp and the consumers about a ring slot.
struct SlotMeta {
  int unit;    // global unit index, -1: end of the sequence
  int op;
  int tile;
  int flags;   // bit 0: the unit's last stage; bit 1: A is bf16; bit 2: end
  int k0;      // first row of the stage
  int rows;    // rows of the stage below K (1..64)
  int pad[2];
};

struct Smem {
  uint32_t ring, aring, red, meta, bars, misc, total;
};

template <int STAGES>
__host__ __device__ constexpr Smem smem_layout() {
  Smem s{};
  s.ring = 0;
  s.aring = STAGES * kStageBytes;
  s.red = s.aring + STAGES * kStageRows * kARowBytes;
  s.meta = s.red + kConsumerWarps * kRedStride<kBPT> * 4;
  s.bars = (s.meta + STAGES * static_cast<uint32_t>(sizeof(SlotMeta)) + 7) / 8 * 8;
  s.misc = s.bars + (3 * STAGES + 1) * 8;
  s.total = (s.misc + 64 + 127) / 128 * 128;
  return s;
}

// ---- memory-model helpers ---------------------------------------------------
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
// Orders this thread's earlier generic-proxy view of global memory before its
// later async-proxy (bulk copy) reads.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async;" ::: "memory");
}
// cp.async.bulk: `bytes` (a multiple of 16) from global `src` (16-byte aligned)
// to shared `dst`, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ uint32_t mbar_arrive_state(uint64_t* bar) {
  uint64_t st;
  asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];" : "=l"(st) : "r"(smem_u32(bar))
               : "memory");
  return static_cast<uint32_t>(st);
}

// The consumers' barrier: lane 0 of every consumer warp arrives on `bar`
// (count kConsumerWarps) after the warp's __syncwarp, and every thread waits,
// bounded, for the phase to complete.  `phase` is the
// thread's count of barriers passed.  False if the CTA failed or the wait ran
// out (then the thread stops using the barrier).
__device__ __forceinline__ bool consumers_meet(uint64_t* bar, uint32_t& phase, volatile int* fail,
                                               unsigned* err) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive_state(bar);
  const bool ok = bounded_wait(bar, phase & 1u, fail, err);
  ++phase;
  return ok;
}

// Waits for phase `parity` of `bar` for at most `limit_ns`, whatever the
// CTA's failure state (used to drain copies already issued).
constexpr unsigned long long kDrainNs = 100000000ull;
__device__ __forceinline__ bool wait_limit(uint64_t* bar, uint32_t parity,
                                           unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait_sleep(bar, parity, 1000u))
    if (globaltimer() - t0 > limit_ns) return false;
  return true;
}

// Bytes of A that the bulk copy moves for a stage of `rows` rows (the rest,
// fewer than 16 bytes, and the zeros past K are written by the A warp).
__device__ __forceinline__ uint32_t a_bulk_bytes(int rows, int a_dtype) {
  const uint32_t es = a_dtype == 0 ? 4u : 2u;
  return (static_cast<uint32_t>(rows) * es) & ~15u;
}

// Index of the op holding unit u: the last op whose unit_base <= u.
__device__ __forceinline__ int op_of_unit(const SeqOpDesc* ops, int nops, int u) {
  int lo = 0, hi = nops - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&ops[mid].unit_base) <= u) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <int STAGES>
__global__ void __launch_bounds__(kThreads, 2) q4_gemv_seq_kernel(const SeqParams p) {
  constexpr Smem L = smem_layout<STAGES>();
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem + L.ring;
  uint8_t* aring = smem + L.aring;
  float* red = reinterpret_cast<float*>(smem + L.red);
  SlotMeta* meta = reinterpret_cast<SlotMeta*>(smem + L.meta);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + STAGES;
  uint64_t* claimed = empty + STAGES;
  uint64_t* csync = claimed + STAGES;
  int* misc = reinterpret_cast<int*>(smem + L.misc);
  volatile int* s_fail = misc;
  volatile int* s_last = misc + 1;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 2);                  // producer (bytes) + A warp
      mbar_init(&empty[i], kConsumerWarps);
      mbar_init(&claimed[i], 1);
    }
    mbar_init(csync, kConsumerWarps);
    *s_fail = 0;
    *s_last = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // The counters this launch uses were cleared by the stream operation just
  // before it, and A may come from the kernel before: wait for both.
  pdl_wait();

  if (warp == kConsumerWarps) {
    // ===================== producer: weights =====================
    if (lane != 0) return;
    int gs = 0;
    int posted = 0;   // ring phases posted: stages, then the end marker
    bool failed = false;
    while (!failed) {
      // take a unit only once the ring has room for its first stage, so that
      // no CTA holds a unit that it cannot start loading while others idle
      if (gs >= STAGES &&
          !bounded_wait(&empty[gs % STAGES], ((gs / STAGES) - 1) & 1, s_fail, p.err)) {
        failed = true;
        break;
      }
      const int u = static_cast<int>(atomicAdd(p.queue, 1u));
      const bool end = (u >= p.total_units);
      int op = 0, tile = 0, slice = 0, nst = 1, K = 0, srows = 0;
      if (!end) {
        op = op_of_unit(p.ops, p.nops, u);
        const SeqOpDesc& d = p.ops[op];
        const int local = u - d.unit_base;
        tile = local / d.nslices;
        slice = local - tile * d.nslices;
        K = d.K;
        srows = d.slice_rows;
        const int rows = min(srows, K - slice * srows);
        nst = (rows + kStageRows - 1) / kStageRows;
      }
      for (int st = 0; st < nst; ++st, ++gs) {
        const int slot = gs % STAGES;
        if (st > 0 && gs >= STAGES &&
            !bounded_wait(&empty[slot], ((gs / STAGES) - 1) & 1, s_fail, p.err)) {
          failed = true;
          break;
        }
        SlotMeta& m = meta[slot];
        if (end) {
          m.unit = -1;
          m.flags = 4;
          mbar_arrive(&full[slot]);
          mbar_arrive(&claimed[slot]);
          posted = gs + 1;
          break;
        }
        const int k0 = slice * srows + st * kStageRows;
        const int rows = min(kStageRows, K - k0);
        const SeqOpDesc& d = p.ops[op];
        m.unit = u;
        m.op = op;
        m.tile = tile;
        m.flags = ((st == nst - 1) ? 1 : 0) | (d.a_dtype == 0 ? 0 : 2);
        m.k0 = k0;
        m.rows = rows;
        mbar_arrive_expect_tx(&full[slot], kStageBytes + a_bulk_bytes(rows, d.a_dtype));
        tma_load_3d(ring + slot * kStageBytes, &d.tmap, tile * kTileBlocks * 9, k0, 0,
                    &full[slot]);
        mbar_arrive(&claimed[slot]);
        posted = gs + 1;
      }
      if (end) break;
    }
    // every stage issued has landed before the CTA may exit: wait for the
    // latest phase posted on each slot (bounded: after a failure a stage whose
    // A copy was never issued cannot complete)
    for (int i = posted > STAGES ? posted - STAGES : 0; i < posted; ++i)
      wait_limit(&full[i % STAGES], (i / STAGES) & 1, kDrainNs);
    return;
  }

  if (warp == kConsumerWarps + 1) {
    // ===================== A warp: activations after dependencies =====================
    fence_proxy_async();
    int gs = 0;
    int verified = -1;   // ops up to this one have their dependencies done
    bool failed = false; // after a failure: serve the remaining slots unchecked
    while (true) {
      const int slot = gs % STAGES;
      bool got = failed ? wait_limit(&claimed[slot], (gs / STAGES) & 1, kDrainNs)
                        : bounded_wait(&claimed[slot], (gs / STAGES) & 1, s_fail, p.err);
      if (!got && !failed) {
        failed = true;
        got = wait_limit(&claimed[slot], (gs / STAGES) & 1, kDrainNs);
      }
      if (!got) break;
      const SlotMeta m = meta[slot];
      if (m.unit < 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[slot]);
        break;
      }
      const SeqOpDesc& d = p.ops[m.op];
      if (!failed && m.op > verified) {
        int ok = 1;
        if (lane == 0) {
          const unsigned long long t0 = globaltimer();
          for (int i = 0; i < d.ndeps && ok; ++i) {
            const int dep = d.deps[i];
            const unsigned need = static_cast<unsigned>(p.ops[dep].ntiles);
            while (ld_acquire_gpu(&p.done[dep]) < need) {
              if (*s_fail || globaltimer() - t0 > kWaitLimitNs) {
                if (!*s_fail) {
                  *s_fail = 1;
                  atomicOr(p.err, kDevErrTimeout);
                }
                ok = 0;
                break;
              }
              __nanosleep(200);
            }
          }
          fence_proxy_async();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        if (ok) verified = m.op;
        else failed = true;
      }
      const uint32_t es = d.a_dtype == 0 ? 4u : 2u;
      const uint32_t bulk = a_bulk_bytes(m.rows, d.a_dtype);
      uint8_t* dst = aring + slot * (kStageRows * kARowBytes);
      const uint8_t* src = static_cast<const uint8_t*>(d.A) + static_cast<size_t>(m.k0) * es;
      if (lane == 0 && bulk) bulk_load(dst, src, bulk, &full[slot]);
      // the last few entries below K, then zeros up to the stage's 64 rows
      for (uint32_t b = bulk + lane * es; b < kStageRows * es; b += 32 * es) {
        const uint32_t r = b / es;
        if (es == 4) {
          const float v =
              (static_cast<int>(r) < m.rows) ? __ldcg(reinterpret_cast<const float*>(src) + r) : 0.f;
          reinterpret_cast<float*>(dst)[r] = v;
        } else {
          const uint16_t v = (static_cast<int>(r) < m.rows)
                                 ? __ldcg(reinterpret_cast<const unsigned short*>(src) + r)
                                 : static_cast<uint16_t>(0);
          reinterpret_cast<uint16_t*>(dst)[r] = v;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&full[slot]);
      ++gs;
    }
    return;
  }

  // ===================== consumers =====================
  DecodeConsts kc;
#pragma unroll
  for (int i = 0; i < 4; ++i) kc.mask[i] = p.kmask[i];
  const int pi = lane & 7;
  const int rp = warp * 4 + (lane >> 3);              // row phase within a stage
  const uint32_t boff = static_cast<uint32_t>(pi * kBPT * kBlockBytes);
  uint32_t cphase = 0;

  f32x2 acc[1][16 * kBPT];
  float sad[1][kBPT];
#pragma unroll
  for (int i = 0; i < 16 * kBPT; ++i) acc[0][i] = 0ull;
#pragma unroll
  for (int bb = 0; bb < kBPT; ++bb) sad[0][bb] = 0.f;

  const volatile SlotMeta* vmeta = meta;
  for (int gs = 0;; ++gs) {
    const int slot = gs % STAGES;
    if (!bounded_wait(&full[slot], (gs / STAGES) & 1, s_fail, p.err)) break;
    const int flags = vmeta[slot].flags;
    if (flags & 4) break;
    const uint8_t* stage = ring + slot * kStageBytes;
    const uint8_t* as = aring + slot * (kStageRows * kARowBytes);
#pragma unroll
    for (int rr = 0; rr < kRowsPerThread; ++rr) {
      const int rs = rp + rr * kRowsPerPass;
      uint32_t dbits[kBPT], qs[kBPT][4];
      load_blocks<kBPT, kFmtQ4>(stage + rs * kRowBytes, boff, false, dbits, qs);
      float a = (flags & 2) ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(as)[rs])
                            : reinterpret_cast<const float*>(as)[rs];
      a *= kAScale;
#pragma unroll
      for (int bb = 0; bb < kBPT; ++bb)
        accumulate_block<1, kBPT, kFmtQ4>(acc, sad, bb, dbits[bb], qs[bb], &a, 0, kc);
    }
    __syncwarp();
    if (!(flags & 1)) {
      if (lane == 0) mbar_arrive(&empty[slot]);
      continue;
    }
    // the unit's last stage: its slot is released only once the unit's
    // identity has been read from it
    const int unit = vmeta[slot].unit;
    const int op = vmeta[slot].op;
    const int tile = vmeta[slot].tile;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    const SeqOpDesc& d = p.ops[op];

    // ---- the unit is complete: reduce over the CTA ----
    finish_acc<1, kBPT, kFmtQ4>(acc, sad);
    {
      constexpr int P = 16 * kBPT;
      const bool hi16 = (lane & 16) != 0;
      const bool hi8 = (lane & 8) != 0;
      f32x2 h[P / 2];
#pragma unroll
      for (int i = 0; i < P / 2; ++i) {
        const f32x2 send = hi16 ? acc[0][i] : acc[0][P / 2 + i];
        const f32x2 keep = hi16 ? acc[0][P / 2 + i] : acc[0][i];
        h[i] = add2(keep, __shfl_xor_sync(0xffffffffu, send, 16));
      }
      f32x2 q[P / 4];
#pragma unroll
      for (int i = 0; i < P / 4; ++i) {
        const f32x2 send = hi8 ? h[i] : h[P / 4 + i];
        const f32x2 keep = hi8 ? h[P / 4 + i] : h[i];
        q[i] = add2(keep, __shfl_xor_sync(0xffffffffu, send, 8));
      }
      const int j0 = (hi16 ? P / 2 : 0) + (hi8 ? P / 4 : 0);
      float* dst = red + warp * kRedStride<kBPT> + pi * kBPT * 33;
#pragma unroll
      for (int i = 0; i < P / 4; ++i) {
        const int j = j0 + i;
        const int c = 33 * (j >> 4) + acc_col_pair<kFmtQ4>(j & 15);
        float v0, v1;
        unpack2(q[i], v0, v1);
        dst[c] = v0;
        dst[c + Fmt<kFmtQ4>::kPairGap] = v1;
      }
    }
#pragma unroll
    for (int i = 0; i < 16 * kBPT; ++i) acc[0][i] = 0ull;
#pragma unroll
    for (int bb = 0; bb < kBPT; ++bb) sad[0][bb] = 0.f;
    if (!consumers_meet(csync, cphase, s_fail, p.err)) break;
    // thread t finishes columns t and t + 256 of the tile
    float colv[kBPT];
#pragma unroll
    for (int i = 0; i < kBPT; ++i) {
      const int c = tid + 256 * i;
      const int off = (c >> 5) * 33 + (c & 31);
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) s += red[w * kRedStride<kBPT> + off];
      colv[i] = s;
    }
    const int nslices = d.nslices;
    if (nslices == 1) {
      // the unit is the whole tile: store C directly
#pragma unroll
      for (int i = 0; i < kBPT; ++i) {
        const int col = tile * kTileCols + tid + 256 * i;
        if (col < d.N) {
          if (d.c_dtype == 0) reinterpret_cast<float*>(d.C)[col] = colv[i];
          else reinterpret_cast<__nv_bfloat16*>(d.C)[col] = __float2bfloat16_rn(colv[i]);
        }
      }
    } else {
      // ---- partial sums of the unit -> global scratch, then the tile's ticket ----
      float* part = p.part + static_cast<size_t>(unit) * kTileCols;
#pragma unroll
      for (int i = 0; i < kBPT; ++i) __stcg(part + tid + 256 * i, colv[i]);
      if (!consumers_meet(csync, cphase, s_fail, p.err)) break;
      if (tid == 0) {
        // every consumer's partial store is ordered before this by the meet
        const unsigned t = atom_add_acq_rel_gpu(&p.tickets[d.ticket_base + tile], 1u);
        *s_last = (t == static_cast<unsigned>(nslices - 1)) ? 1 : 0;
      }
      if (!consumers_meet(csync, cphase, s_fail, p.err)) break;
      if (!*s_last) continue;
      // every slice of the tile has written its partial: add them in slice order
      const float* base =
          p.part + static_cast<size_t>(d.unit_base + tile * nslices) * kTileCols;
      float sums[kBPT];
#pragma unroll
      for (int i = 0; i < kBPT; ++i) sums[i] = 0.f;
      // the loads of a batch are independent, so their L2 latencies overlap;
      // the additions keep slice order
      constexpr int kBatch = 8;
      for (int sl0 = 0; sl0 < nslices; sl0 += kBatch) {
        float v[kBPT][kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
#pragma unroll
          for (int i = 0; i < kBPT; ++i)
            v[i][b] = (sl0 + b < nslices)
                          ? __ldcg(base + static_cast<size_t>(sl0 + b) * kTileCols + tid + 256 * i)
                          : 0.f;
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
#pragma unroll
          for (int i = 0; i < kBPT; ++i)
            if (sl0 + b < nslices) sums[i] = (sl0 + b == 0) ? v[i][b] : sums[i] + v[i][b];
      }
#pragma unroll
      for (int i = 0; i < kBPT; ++i) {
        const int c = tid + 256 * i;
        const int col = tile * kTileCols + c;
        const float sum = sums[i];
        if (col < d.N) {
          if (d.c_dtype == 0) reinterpret_cast<float*>(d.C)[col] = sum;
          else reinterpret_cast<__nv_bfloat16*>(d.C)[col] = __float2bfloat16_rn(sum);
        }
      }
    }
    // the tile's C is stored: count it for the op (after every thread's stores)
    if (!consumers_meet(csync, cphase, s_fail, p.err)) break;
    if (tid == 0) red_add_release_gpu(&p.done[op], 1u);
  }
}

}  // namespace seq

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
int seq_ctas_per_sm(int stages) {
  const void* fn = stages == 4 ? (const void*)seq::q4_gemv_seq_kernel<4>
                               : (const void*)seq::q4_gemv_seq_kernel<5>;
  const uint32_t smem = stages == 4 ? seq::smem_layout<4>().total : seq::smem_layout<5>().total;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return 0;
  cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, seq::kThreads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int seq_tile_cols() { return seq::kTileCols; }
int seq_stage_rows() { return seq::kStageRows; }
int seq_max_slice_rows() { return seq::kMaxSliceStages * seq::kStageRows; }
int seq_default_slice_rows() { return seq::kDefaultSliceStages * seq::kStageRows; }

cudaError_t launch_gemv_seq(const SeqParams& p, int grid, int stages, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(seq::kThreads);
  cfg.stream = st;
  if (stages == 4) {
    cfg.dynamicSmemBytes = seq::smem_layout<4>().total;
    return cudaLaunchKernelEx(&cfg, seq::q4_gemv_seq_kernel<4>, p);
  }
  cfg.dynamicSmemBytes = seq::smem_layout<5>().total;
  return cudaLaunchKernelEx(&cfg, seq::q4_gemv_seq_kernel<5>, p);
}

}  // namespace q4
