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
//    columns, K slice of 64 to 4096 rows, chosen per op).  Units are
//    numbered op by op, and within an op tile by tile; a global counter hands
//    them out in that order.
//  * In each CTA a producer warp issues two TMA tensor copies (64-row boxes)
//    per 128-row stage (36 KB) into a three-stage ring, and a second warp
//    copies the stage's 128 entries of A (cp.async.bulk; zeros past the
//    unit's rows, so that a half stage adds nothing) onto the same mbarrier
//    once the op's dependencies have
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
constexpr int kStageRows = 128;                          // two 64-row TMA boxes
constexpr int kStageBytes = kStageRows * kRowBytes;      // 36864 bytes
constexpr int kDefaultSliceStages = 4;                   // stages of a unit by default
constexpr int kMaxSliceStages = 32;                      // stages of the longest unit
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
  int flags;   // bit 0: the unit's last stage; bit 1: A is bf16; bit 2: end;
               // bit 3: the unit's expert index is invalid
  int k0;      // first row of A of the stage
  int rows;    // rows of the stage inside the unit and below K (1..128)
  int slice;   // the unit's K slice
  int seg;     // the unit's segment (0 for unsegmented ops)
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

// ---- memory-model helpers (the GPU-scope ones are in q4_device.cuh) ---------
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

// Index of the op holding unit u: the last op whose unit_base <= u.  (With
// SEG the ops may sit in the kernel's parameters: generic loads.)
template <bool SEG>
__device__ __forceinline__ int op_of_unit(const SeqOpDesc* ops, int nops, int u) {
  int lo = 0, hi = nops - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((SEG ? ops[mid].unit_base : __ldg(&ops[mid].unit_base)) <= u) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Expert of segment `seg` of op d (0 without an index list; a pair op's
// segments 2s and 2s + 1 both belong to slot s), and whether it lies in
// [0, E).
template <bool SEG>
__device__ __forceinline__ int seg_expert(const SeqOpDesc& d, int seg, bool& valid) {
  if (!SEG || !d.eidx) {
    valid = true;
    return 0;
  }
  const int e = __ldcg(d.eidx + (d.pair ? (seg >> 1) : seg));
  valid = (e >= 0 && e < d.E);
  return e;
}

// Tile and K slice of unit `local` (0-based within op d): tile-major.
__device__ __forceinline__ void unit_coords(const SeqOpDesc& d, int local, int& tile, int& slice) {
  tile = local / d.nslices;
  slice = local - tile * d.nslices;
}

// Output columns of tile `tile` of op d: the segment it belongs to, its first
// column within the segment, the segment's width, and where the segment's
// row of C starts (a pair op's odd segments go to C2).
struct TileCols {
  int seg, c0, width;
  size_t row;   // element offset of the segment's row in `out`
  void* out;
};
template <bool SEG>
__device__ __forceinline__ TileCols tile_cols(const SeqOpDesc& d, int tile) {
  TileCols t;
  if (SEG && d.seg_mode == 1) {
    t.seg = tile / d.seg_tiles;
    t.c0 = (tile - t.seg * d.seg_tiles) * kTileCols;
    t.width = d.seg_len;
    const int row = d.pair ? (t.seg >> 1) : t.seg;
    t.row = static_cast<size_t>(row) * d.seg_len;
    t.out = (d.pair && (t.seg & 1)) ? d.C2 : d.C;
  } else {
    t.seg = 0;
    t.c0 = tile * kTileCols;
    t.width = d.N;
    t.row = 0;
    t.out = d.C;
  }
  return t;
}

// SEG: the ops may be segmented, paired or in the parameters, and the launch
// may reset its counters; without it, every op is a plain GEMV read from
// global memory and none of that code is compiled in.
template <int STAGES, bool SEG>
__global__ void __launch_bounds__(kThreads, 2) q4_gemv_seq_kernel(const __grid_constant__ SeqParams p) {
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
  // before it (or by the launch before, `reset`), and A and the expert
  // indices may come from the kernel before: wait for all of them.
  pdl_wait();
  pdl_launch_dependents();
  const SeqOpDesc* ops = (SEG && !p.ops) ? p.inl : p.ops;

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
      // the unit's weight rows [w0, w0 + urows) of matrix `expert`, columns
      // from cx (uint16 elements), and its first row of A
      int op = 0, tile = 0, nst = 1, urows = 0, w0 = 0, a0 = 0, cx = 0, expert = 0;
      int uslice = 0, useg = 0;
      bool valid = true, second = false;
      if (!end) {
        op = op_of_unit<SEG>(ops, p.nops, u);
        const SeqOpDesc& d = ops[op];
        int slice;
        unit_coords(d, u - d.unit_base, tile, slice);
        uslice = slice;
        int seg = 0;
        const int sl = slice, klen = d.K;
        const TileCols tc = tile_cols<SEG>(d, tile);
        if (SEG && d.seg_mode == 1) seg = tc.seg;
        useg = seg;
        second = SEG && d.pair && (seg & 1);
        cx = (tc.c0 / kTileCols) * kTileBlocks * 9;
        w0 = sl * d.slice_rows;
        urows = min(d.slice_rows, klen - w0);
        // the segment's row of A (routed tokens: one row per token)
        a0 = ((SEG && d.a_seg_div) ? (seg / d.a_seg_div) * d.a_seg_stride : 0) + w0;
        expert = seg_expert<SEG>(d, seg, valid);
        if (!valid) atomicOr(p.err, kDevErrIndex);
        nst = (urows + kStageRows - 1) / kStageRows;
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
        const int rows = min(kStageRows, urows - st * kStageRows);
        const SeqOpDesc& d = ops[op];
        m.unit = u;
        m.op = op;
        m.tile = tile;
        m.flags = ((st == nst - 1) ? 1 : 0) | (d.a_dtype != 0 ? 2 : 0) | (valid ? 0 : 8);
        m.k0 = a0 + st * kStageRows;
        m.rows = rows;
        m.slice = uslice;
        m.seg = useg;
        // a segment with an expert index outside [0, E) reads no weights: its
        // stages hold stale data and its outputs are not written
        const uint32_t tx = (valid ? kStageBytes : 0u) + a_bulk_bytes(rows, d.a_dtype);
        if (tx) mbar_arrive_expect_tx(&full[slot], tx);
        else mbar_arrive(&full[slot]);
        if (valid) {
          // two 64-row boxes (the weight maps' box); rows past the unit's
          // end meet zeros in A, and rows past K read as zeros
          const CUtensorMap* tm = second ? &d.tmap2 : &d.tmap;
          const int r0 = w0 + st * kStageRows;
          tma_load_3d(ring + slot * kStageBytes, tm, cx, r0, expert, &full[slot]);
          tma_load_3d(ring + slot * kStageBytes + kStageBytes / 2, tm, cx, r0 + kStageRows / 2,
                      expert, &full[slot]);
        }
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
    int vseg_op = -1, vseg = -1;   // segments up to vseg of op vseg_op have theirs
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
      const SeqOpDesc& d = ops[m.op];
      // a segment waits for its own slot's inputs
      if (SEG && !failed && d.seg_need > 0 && (m.op != vseg_op || m.seg > vseg)) {
        int ok = 1;
        if (lane == 0) {
          const unsigned long long t0 = globaltimer();
          const unsigned* c = p.seg_done + ops[d.seg_dep].seg_done_base + m.seg;
          while (ld_acquire_gpu(c) < static_cast<unsigned>(d.seg_need)) {
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
          fence_proxy_async();
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        __syncwarp();
        if (ok) {
          vseg_op = m.op;
          vseg = m.seg;
        } else {
          failed = true;
        }
      }
      if (!failed && m.op > verified) {
        int ok = 1;
        if (lane == 0) {
          const unsigned long long t0 = globaltimer();
          for (int i = 0; i < d.ndeps && ok; ++i) {
            const int dep = d.deps[i];
            const unsigned need = static_cast<unsigned>(ops[dep].ntiles);
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
      uint8_t* dst = aring + slot * (kStageRows * kARowBytes);
      const uint32_t es = d.a_dtype == 0 ? 4u : 2u;
      const uint32_t bulk = a_bulk_bytes(m.rows, d.a_dtype);
      const uint8_t* src = static_cast<const uint8_t*>(d.A) + static_cast<size_t>(m.k0) * es;
      if (lane == 0 && bulk) bulk_load(dst, src, bulk, &full[slot]);
      // the last few entries below K, then zeros up to the stage's rows
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
  kc.hi16 = (kc.mask[0] & 0x1u) << 16;   // 2^16 (mask[0] = 0xF)
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
    if (flags & 4) {
      // the end of the sequence for this CTA: with `reset`, the last CTA to
      // get here zeroes the counters for the next launch (every producer has
      // stopped taking units and every tile is complete by then)
      if (SEG && p.reset && consumers_meet(csync, cphase, s_fail, p.err) && tid == 0) {
        const unsigned n = atom_add_acq_rel_gpu(p.exits, 1u);
        if (n == gridDim.x - 1) {
          *p.queue = 0u;
          for (int i = 0; i < p.nops; ++i) p.done[i] = 0u;
          for (int i = 0; i < p.ntickets; ++i) p.tickets[i] = 0u;
          for (int i = 0; i < p.nseg_done; ++i) p.seg_done[i] = 0u;
          __threadfence();
          *p.exits = 0u;
        }
      }
      break;
    }
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
        accumulate_block<1, kBPT, kFmtQ4, true>(acc, sad, bb, dbits[bb], qs[bb], &a, 0, kc);
    }
    __syncwarp();
    if (!(flags & 1)) {
      if (lane == 0) mbar_arrive(&empty[slot]);
      continue;
    }
    // the unit's last stage: its slot is released only once the unit's
    // identity has been read from it
    const int op = vmeta[slot].op;
    const int tile = vmeta[slot].tile;
    const int uslice = vmeta[slot].slice;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    const SeqOpDesc& d = ops[op];

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
    const TileCols tc = tile_cols<SEG>(d, tile);
    const bool unit_valid = !SEG || !(flags & 8);
    const bool pair = SEG && d.pair;
    // a pair op's tile shares one ticket with its partner (the slot's other
    // product on the same columns): the last of their slices combines both
    const int pslot = tc.seg >> 1;
    const int ptile = pslot * d.seg_tiles + tc.c0 / kTileCols;
    if (nslices == 1 && !pair) {
      // the unit is the whole tile: store C directly
#pragma unroll
      for (int i = 0; i < kBPT; ++i) {
        const int c = tc.c0 + tid + 256 * i;
        if (unit_valid && c < tc.width) {
          const size_t col = tc.row + c;
          if (d.c_dtype == 0) reinterpret_cast<float*>(tc.out)[col] = colv[i];
          else reinterpret_cast<__nv_bfloat16*>(tc.out)[col] = __float2bfloat16_rn(colv[i]);
        }
      }
    } else {
      // ---- partial sums of the unit -> global scratch, then the tile's ticket ----
      // (partial rows are kept tile by tile, slice by slice, whatever the
      // order in which the units are handed out)
      const float* base =
          p.part + static_cast<size_t>(d.unit_base + tile * nslices) * kTileCols;
      float* part = const_cast<float*>(base) + static_cast<size_t>(uslice) * kTileCols;
#pragma unroll
      for (int i = 0; i < kBPT; ++i) __stcg(part + tid + 256 * i, colv[i]);
      if (!consumers_meet(csync, cphase, s_fail, p.err)) break;
      if (tid == 0) {
        // every consumer's partial store is ordered before this by the meet
        const int ti = pair ? ptile : tile;
        const unsigned need = static_cast<unsigned>(pair ? 2 * nslices : nslices);
        const unsigned t = atom_add_acq_rel_gpu(&p.tickets[d.ticket_base + ti], 1u);
        *s_last = (t == need - 1u) ? 1 : 0;
      }
      if (!consumers_meet(csync, cphase, s_fail, p.err)) break;
      if (!*s_last) continue;
      // every slice has written its partial: add them in slice order
      {
        // the tile's sum (a pair: both products' sums, then h = SiLU(g) * u)
        const int t0 = pair ? (2 * pslot) * d.seg_tiles + tc.c0 / kTileCols : tile;
        const float* b0 = p.part + static_cast<size_t>(d.unit_base + t0 * nslices) * kTileCols;
        const float* b1 = b0 + static_cast<size_t>(d.seg_tiles) * nslices * kTileCols;
        const int nsum = pair ? 2 : 1;
        float sums[2][kBPT];
#pragma unroll
        for (int i = 0; i < kBPT; ++i) sums[0][i] = sums[1][i] = 0.f;
        constexpr int kBatch = 8;
        for (int sl0 = 0; sl0 < nslices; sl0 += kBatch) {
          float v[2][kBPT][kBatch];
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int b = 0; b < kBatch; ++b)
#pragma unroll
              for (int i = 0; i < kBPT; ++i)
                v[q][i][b] = (q < nsum && sl0 + b < nslices)
                                 ? __ldcg((q ? b1 : b0) + static_cast<size_t>(sl0 + b) * kTileCols +
                                          tid + 256 * i)
                                 : 0.f;
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int b = 0; b < kBatch; ++b)
#pragma unroll
              for (int i = 0; i < kBPT; ++i)
                if (sl0 + b < nslices)
                  sums[q][i] = (sl0 + b == 0) ? v[q][i][b] : sums[q][i] + v[q][i][b];
        }
#pragma unroll
        for (int i = 0; i < kBPT; ++i) {
          const int c = tc.c0 + tid + 256 * i;
          if (unit_valid && c < tc.width) {
            const size_t col = tc.row + c;
            if (pair) {
              const float g = sums[0][i], u = sums[1][i];
              reinterpret_cast<float*>(d.C)[col] = g;
              reinterpret_cast<float*>(d.C2)[col] = u;
              d.h[col] = g / (1.0f + __expf(-g)) * u;
            } else if (d.c_dtype == 0) {
              reinterpret_cast<float*>(tc.out)[col] = sums[0][i];
            } else {
              reinterpret_cast<__nv_bfloat16*>(tc.out)[col] = __float2bfloat16_rn(sums[0][i]);
            }
          }
        }
      }
    }
    if (pair) {
      // the slot's h is stored on these columns: count them for the slot
      if (!consumers_meet(csync, cphase, s_fail, p.err)) break;
      if (tid == 0) {
        red_add_release_gpu(&p.seg_done[d.seg_done_base + pslot], 1u);
        red_add_release_gpu(&p.done[op], 2u);
      }
      continue;
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
int seq_ctas_per_sm(int stages, bool seg) {
  const void* fn = stages == 2 ? (seg ? (const void*)seq::q4_gemv_seq_kernel<2, true>
                                      : (const void*)seq::q4_gemv_seq_kernel<2, false>)
                               : (seg ? (const void*)seq::q4_gemv_seq_kernel<3, true>
                                      : (const void*)seq::q4_gemv_seq_kernel<3, false>);
  const uint32_t smem = stages == 2 ? seq::smem_layout<2>().total : seq::smem_layout<3>().total;
  // a failed call leaves no error pending for the caller's next launch
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    cudaGetLastError();   // tolerated: the occupancy query below counts what fits
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, seq::kThreads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

int seq_tile_cols() { return seq::kTileCols; }
int seq_stage_rows() { return seq::kStageRows; }
int seq_slice_rows_unit() { return seq::kStageRows / 2; }
int seq_max_slice_rows() { return seq::kMaxSliceStages * seq::kStageRows; }
int seq_default_slice_rows() { return seq::kDefaultSliceStages * seq::kStageRows; }

cudaError_t launch_gemv_seq(const SeqParams& p, int grid, int stages, cudaStream_t st,
                            bool pdl, bool seg) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(seq::kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (stages == 2) {
    cfg.dynamicSmemBytes = seq::smem_layout<2>().total;
    return seg ? cudaLaunchKernelEx(&cfg, seq::q4_gemv_seq_kernel<2, true>, p)
               : cudaLaunchKernelEx(&cfg, seq::q4_gemv_seq_kernel<2, false>, p);
  }
  cfg.dynamicSmemBytes = seq::smem_layout<3>().total;
  return seg ? cudaLaunchKernelEx(&cfg, seq::q4_gemv_seq_kernel<3, true>, p)
             : cudaLaunchKernelEx(&cfg, seq::q4_gemv_seq_kernel<3, false>, p);
}

}  // namespace q4
