// The decode and accumulation core of the Q4_0 GEMV kernels: weight
// formats, tile shapes, the exact nibble decode and the fp32x2 accumulation
// (one AND per weight, see q4_gemv.cu for the arithmetic), shared by the
// split-K GEMV (q4_gemv.cu) and the persistent decode sequence
// (q4_gemv_seq.cu).
#pragma once

#include <cstdint>

#include "q4_device.cuh"
#include "q4_kernels.h"

namespace q4 {

constexpr int kLanesPerRow = 8;     // consumer lanes sharing one row

// Consumer warps: one or two rows of A, 16 warps; four rows, 8 warps (their
// accumulators need the registers).  They work in groups that take the ring
// stages in turn (TileCfg).
template <int MR>
struct Crew {
  static constexpr int kWarps = (MR <= 2) ? 16 : 8;
  static constexpr int kConsumers = kWarps * 32;
  static constexpr int kThreads = kConsumers + 32;   // + producer warp
};

// Weight formats behind the same kernel (the block runs along the output
// columns of one row in both):
//   kFmtQ4: block_q4_0 {fp16 d; 16 bytes of nibbles}, w = (q - 8) * d;
//   kFmtQ8: Q8_0 {fp16 d; int8 q[32]}, w = q * d (decoded as b = q + 128,
//           so the offset removed per block is 128).
template <int FMT>
struct Fmt;
template <>
struct Fmt<kFmtQ4> {
  static constexpr int kBytes = 18;        // bytes per block
  static constexpr int kWords = 4;         // 32-bit words of codes per block
  static constexpr int kBias = 8;          // code offset removed after the loop
  static constexpr int kPairGap = 8;       // second column of an accumulator pair
  static constexpr int kTmaElem = 2;       // tensor-map element size (uint16)
  static constexpr bool kPlanar = false;
};
template <>
struct Fmt<kFmtQ8> {
  static constexpr int kBytes = 34;
  static constexpr int kWords = 8;
  static constexpr int kBias = 128;
  static constexpr int kPairGap = 4;
  static constexpr int kTmaElem = 4;       // uint32: a 2-block-per-thread row segment is 544 B
  static constexpr bool kPlanar = false;
};
// Planar Q4_0: the same blocks and arithmetic, stored as a plane of fp16
// scales d[K][nb] and a plane of nibbles qs[K][nb][16].  A stage holds its
// rows' nibbles [rows][tile blocks][16] followed by their scales
// [rows][tile blocks]: every block's codes are 16-byte aligned.
template <>
struct Fmt<kFmtQ4P> : Fmt<kFmtQ4> {
  static constexpr bool kPlanar = true;
};

// A stage is one TMA box.  Long slices use 18 KB boxes (BIG): bulk copies of
// that size keep HBM near its copy bandwidth from 128 SMs, where 9 KB boxes
// reach about two thirds of it (measured on GB300, data movement alone).
// Short slices use 32-row boxes: fewer rows per stage fill and drain the
// pipeline sooner.  Either way the ring holds ~147 KB.  (Q8_0 rows are
// already 272 or 544 bytes: it keeps 32-row boxes.)
template <int BPT, bool BIG, int FMT = kFmtQ4>
struct TileCfg {
  static constexpr int kBlocks = kLanesPerRow * BPT;                // blocks per column tile
  static constexpr int kCols = kBlocks * kBlockCols;                // 256 * BPT
  static constexpr int kRowBytes = kBlocks * Fmt<FMT>::kBytes;      // 144 or 272 per BPT
  static constexpr int kRows = (BIG && FMT != kFmtQ8) ? 128 / BPT : 32;   // rows of one stage
  static constexpr int kStageBytes = kRows * kRowBytes;
  static constexpr int kQsBytes = kRows * kBlocks * 16;             // planar: nibbles, then scales
  static constexpr int kStages = (147456 / kStageBytes);            // 8, 16 or 32
  static constexpr int kGroupWarps = BIG ? 8 : 4;                   // warps sharing a stage
  static constexpr int kGroupRows = kGroupWarps * 32 / kLanesPerRow;
  static constexpr int kRowsPerThread = kRows / kGroupRows;         // per consumer thread per stage
  static_assert(kRows % kGroupRows == 0, "a warp group covers a stage in whole passes");
  // TMA tensor copies need 128-byte-aligned shared destinations; a block's
  // word-aligned 20-byte read ends at most at the row's last byte, so rows
  // carry no padding.
  static_assert(kStageBytes % 128 == 0, "TMA destinations must be 128-byte aligned");
  static_assert(kQsBytes % 128 == 0, "the planar scale box must start 128-byte aligned");
};

// Reduction buffer of one (warp, row of A): 8 lanes-in-row x BPT blocks x 32
// columns, each block row padded to 33 floats so that the lanes' stores and
// the column-wise reads fall in distinct banks.
template <int BPT>
constexpr int kRedStride = kLanesPerRow * BPT * 33;

// ---------------------------------------------------------------------------
// Consumer arithmetic
// ---------------------------------------------------------------------------
// The code masks, held in registers across the main loop (loaded from the
// parameters so that the compiler does not re-create immediates): Q4_0, the
// nibble masks 0xF << 4p, p = 0..3; Q8_0, the byte masks 0xFF << 8p,
// p = 0..2, and the sign flips 0x80808080.
struct DecodeConsts {
  uint32_t mask[4];
  uint32_t hi16;   // 2^16, from a parameter (see accumulate_block's HI_MUL)
};

__device__ __forceinline__ DecodeConsts load_consts(const GemvParams& p) {
  DecodeConsts c;
#pragma unroll
  for (int i = 0; i < 4; ++i) c.mask[i] = p.kmask[i];
  c.hi16 = (c.mask[0] & 0x1u) << 16;
  return c;
}

// The subnormals (q0 * 16^p * 2^-149, q1 * 16^p * 2^-149) of nibble p of
// words w0 and w1: one AND per half, both written into one register pair.
__device__ __forceinline__ f32x2 code_pair(uint32_t w0, uint32_t w1, uint32_t mask) {
  f32x2 r;
  asm("{\n\t.reg .b32 lo, hi;\n\t"
      "and.b32 lo, %1, %3;\n\t"
      "and.b32 hi, %2, %3;\n\t"
      "mov.b64 %0, {lo, hi};\n\t}"
      : "=l"(r)
      : "r"(w0), "r"(w1), "r"(mask));
  return r;
}

// Q8_0: the subnormals ((byte p of w0 ^ 0x80) * 256^p * 2^-149, same for w1),
// p = 0..2: one three-input logic op per half, (w ^ flip) & mask.
__device__ __forceinline__ f32x2 byte_pair(uint32_t w0, uint32_t w1, uint32_t mask,
                                           uint32_t flip) {
  f32x2 r;
  asm("{\n\t.reg .b32 lo, hi;\n\t"
      "lop3.b32 lo, %1, %4, %3, 0x28;\n\t"   // (w0 ^ flip) & mask
      "lop3.b32 hi, %2, %4, %3, 0x28;\n\t"   // (w1 ^ flip) & mask
      "mov.b64 %0, {lo, hi};\n\t}"
      : "=l"(r)
      : "r"(w0), "r"(w1), "r"(mask), "r"(flip));
  return r;
}

// Q8_0 byte 3 of w0 and w1 as ((w >> 24) ^ 0x80) * 2^-149.
__device__ __forceinline__ f32x2 top_byte_pair(uint32_t w0, uint32_t w1) {
  return pack2(__uint_as_float((w0 >> 24) ^ 0x80u), __uint_as_float((w1 >> 24) ^ 0x80u));
}

// 2^64: the factor of the activations staged in shared memory.
constexpr float kAScale = 18446744073709551616.0f;

// Accumulator layout of one block (32 columns, 16 pairs).  Q4_0: words t = 2h
// and 2h + 1 are decoded together, nibble p of each forming a pair, so
//   acc[8h + p]     holds columns (16h + p,     16h + 8 + p)
//   acc[8h + 4 + p] holds columns (16h + 4 + p, 16h + 12 + p)
// each scaled by 16^p * 2^-85.  Q8_0: words 2h and 2h + 1, byte p of each:
//   acc[4h + p]     holds columns (8h + p, 8h + 4 + p), scaled by
// 256^p * 2^-85 for p < 3 and 2^-85 for p = 3.  acc_col_pair() maps a pair
// back to its first column (the second is kPairGap further) and finish_acc()
// removes the power-of-two factors (exact) and the code offset.
template <int FMT>
__device__ __forceinline__ int acc_col_pair(int j) {   // first column of pair j
  if constexpr (FMT == kFmtQ8) {
    return 8 * (j >> 2) + (j & 3);
  } else {
    const int h = j >> 3, p = j & 3, hi = (j >> 2) & 1;
    return 16 * h + 4 * hi + p;
  }
}

// Adds block bb of a staged row (scale bits dbits, codes qs) for MR rows of A
// (a[m * a_ld], already times 2^64): acc[m][16bb + j] += a'_m * codes of pair
// j, sad[m][bb] += a'_m.  HI_MUL: a word's upper half comes down as
// mul.hi(w, 2^16), which the FMA pipe executes, instead of a shift on the
// integer pipe (the same value); k.hi16 holds 2^16 read from a parameter, so
// that the compiler keeps the multiply.  The decode-sequence kernel, whose
// integer pipe is its busiest unit, takes it.
template <int MR, int BPT, int FMT, bool HI_MUL = false>
__device__ __forceinline__ void accumulate_block(f32x2 (&acc)[MR][16 * BPT],
                                                 float (&sad)[MR][BPT], int bb, uint32_t dbits,
                                                 const uint32_t (&qs)[Fmt<FMT>::kWords],
                                                 const float* a, int a_ld,
                                                 const DecodeConsts& k) {
  const float d = fp16_bits_to_f32(dbits);
  f32x2 ad[MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    const float x = a[m * a_ld] * d;
    sad[m][bb] += x;
    ad[m] = dup2(x);
  }
  if constexpr (FMT == kFmtQ8) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint32_t w0 = qs[2 * h], w1 = qs[2 * h + 1];
      f32x2 code[4];
#pragma unroll
      for (int p = 0; p < 3; ++p) code[p] = byte_pair(w0, w1, k.mask[p], k.mask[3]);
      code[3] = top_byte_pair(w0, w1);
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          f32x2* acc0 = &acc[m][16 * bb + 4 * h];
          acc0[p] = fma2(ad[m], code[p], acc0[p]);
        }
    }
    return;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t w0 = qs[2 * h], w1 = qs[2 * h + 1];
    const uint32_t y0 = HI_MUL ? __umulhi(w0, k.hi16) : w0 >> 16;
    const uint32_t y1 = HI_MUL ? __umulhi(w1, k.hi16) : w1 >> 16;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const f32x2 lo = code_pair(w0, w1, k.mask[p]);
      const f32x2 hi = code_pair(y0, y1, k.mask[p]);
#pragma unroll
      for (int m = 0; m < MR; ++m) {
        f32x2* acc0 = &acc[m][16 * bb + 8 * h];
        acc0[p] = fma2(ad[m], lo, acc0[p]);
        acc0[4 + p] = fma2(ad[m], hi, acc0[4 + p]);
      }
    }
  }
}

// Turns the accumulators into sums of a*w: pair j of block bb becomes
// acc * (power of two of its position) - bias * sad * 2^-64 (Q4_0: 2^(85-4p),
// p = j & 3, bias 8; Q8_0: 2^(85-8p) for p = j & 3 < 3, 2^85 for p = 3,
// bias 128; the scalings are exact).
template <int MR, int BPT, int FMT>
__device__ __forceinline__ void finish_acc(f32x2 (&acc)[MR][16 * BPT],
                                           const float (&sad)[MR][BPT]) {
  f32x2 sc[4];
  if constexpr (FMT == kFmtQ8) {
    sc[0] = dup2(0x1p85f); sc[1] = dup2(0x1p77f); sc[2] = dup2(0x1p69f); sc[3] = dup2(0x1p85f);
  } else {
    sc[0] = dup2(0x1p85f); sc[1] = dup2(0x1p81f); sc[2] = dup2(0x1p77f); sc[3] = dup2(0x1p73f);
  }
  constexpr float kCorr = -static_cast<float>(Fmt<FMT>::kBias) * 0x1p-64f;   // exact
#pragma unroll
  for (int m = 0; m < MR; ++m)
#pragma unroll
    for (int bb = 0; bb < BPT; ++bb) {
      const f32x2 corr = dup2(sad[m][bb] * kCorr);
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[m][16 * bb + j] = fma2(acc[m][16 * bb + j], sc[j & 3], corr);
    }
}

// The BPT consecutive blocks a thread owns in one staged row.  `off` is the
// byte offset of its first block; for BPT = 2 it is a multiple of 36 (Q4_0)
// or 68 (Q8_0), 4-byte aligned; for BPT = 1 a multiple of 18 or 34 whose
// parity (2 mod 4 or not) is fixed per thread.  Either format's block is a
// 2-byte scale followed by its code words, so a block that starts 4-byte
// aligned has its codes 2 bytes off the word grid.
template <int BPT, int FMT>
__device__ __forceinline__ void load_blocks(const uint8_t* row, uint32_t off, bool odd,
                                            uint32_t (&dbits)[BPT],
                                            uint32_t (&qs)[BPT][Fmt<FMT>::kWords]) {
  if constexpr (FMT == kFmtQ8) {
    constexpr int W = Fmt<FMT>::kWords;   // 8
    if constexpr (BPT == 2) {
      const uint32_t* wp = reinterpret_cast<const uint32_t*>(row + off);
      uint32_t w[2 * W + 1];
#pragma unroll
      for (int i = 0; i < 2 * W + 1; ++i) w[i] = wp[i];
      dbits[0] = w[0] & 0xFFFFu;
#pragma unroll
      for (int t = 0; t < W; ++t) qs[0][t] = __funnelshift_r(w[t], w[t + 1], 16);
      dbits[1] = w[W] >> 16;
#pragma unroll
      for (int t = 0; t < W; ++t) qs[1][t] = w[W + 1 + t];
    } else {
      const uint32_t* wp = reinterpret_cast<const uint32_t*>(row + (off & ~3u));
      uint32_t w[W + 1];
#pragma unroll
      for (int i = 0; i < W + 1; ++i) w[i] = wp[i];
      if (odd) {
        dbits[0] = w[0] >> 16;
#pragma unroll
        for (int t = 0; t < W; ++t) qs[0][t] = w[t + 1];
      } else {
        dbits[0] = w[0] & 0xFFFFu;
#pragma unroll
        for (int t = 0; t < W; ++t) qs[0][t] = __funnelshift_r(w[t], w[t + 1], 16);
      }
    }
  } else if constexpr (BPT == 2) {
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(row + off);
    uint32_t w[9];
#pragma unroll
    for (int i = 0; i < 9; ++i) w[i] = wp[i];
    dbits[0] = w[0] & 0xFFFFu;
#pragma unroll
    for (int t = 0; t < 4; ++t) qs[0][t] = __funnelshift_r(w[t], w[t + 1], 16);
    dbits[1] = w[4] >> 16;
#pragma unroll
    for (int t = 0; t < 4; ++t) qs[1][t] = w[5 + t];
  } else {
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(row + (off & ~3u));
    uint32_t w[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) w[i] = wp[i];
    if (odd) {   // block starts at 2 mod 4
      dbits[0] = w[0] >> 16;
#pragma unroll
      for (int t = 0; t < 4; ++t) qs[0][t] = w[t + 1];
    } else {
      dbits[0] = w[0] & 0xFFFFu;
#pragma unroll
      for (int t = 0; t < 4; ++t) qs[0][t] = __funnelshift_r(w[t], w[t + 1], 16);
    }
  }
}

// Planar Q4_0: the BPT consecutive blocks a thread owns in one staged row, the
// codes from the row's nibbles at `qs_row` (16-byte aligned, one 16-byte read
// per block), the scales from its scale row at `d_row` (2 * BPT bytes,
// aligned to their size).
template <int BPT>
__device__ __forceinline__ void load_planar(const uint8_t* qs_row, const uint8_t* d_row,
                                            uint32_t (&dbits)[BPT], uint32_t (&qs)[BPT][4]) {
#pragma unroll
  for (int bb = 0; bb < BPT; ++bb) {
    const uint4 v = reinterpret_cast<const uint4*>(qs_row)[bb];
    qs[bb][0] = v.x;
    qs[bb][1] = v.y;
    qs[bb][2] = v.z;
    qs[bb][3] = v.w;
  }
  if constexpr (BPT == 2) {
    const uint32_t both = *reinterpret_cast<const uint32_t*>(d_row);
    dbits[0] = both & 0xFFFFu;
    dbits[1] = both >> 16;
  } else {
    dbits[0] = *reinterpret_cast<const uint16_t*>(d_row);
  }
}

}  // namespace q4
