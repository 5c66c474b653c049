// Dequantisation and the lossless planar repack of Q4_0 weights (sm_103a).
//
// Dequant [C++ DeepSeek engine page §2.2]: W[k, 32b + l] = (q - 8) * d with q
// the low nibble of qs[l/2] for even l and the high nibble for odd l.  The fp32
// product of the small integer q - 8 and the fp16 scale d is exact, so every
// correct implementation agrees bit for bit; the bf16 form rounds that exact
// value to nearest-even, as the tensor-core operand tiles do.
//
// Planar layout: the scales of all blocks, row-major [K][nb] fp16, then (from a
// 16-byte aligned offset) the nibble bytes [K][nb][16].  Moving a block is a
// byte copy, so repack followed by unpack returns the input bit for bit.
#include <cstdint>
#include <cuda_runtime.h>

#include "q4_device.cuh"
#include "q4_kernels.h"

namespace q4 {

// One thread per block; 32 outputs per thread.
template <bool BF16>
__global__ void __launch_bounds__(256) q4_dequant_kernel(void* W, const uint8_t* B, int64_t K,
                                                         int64_t N, int64_t nb) {
  const int64_t nblk = K * nb;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nblk;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t k = i / nb;
    const int64_t b = i - k * nb;
    const uint16_t* blk = reinterpret_cast<const uint16_t*>(B + i * kBlockBytes);   // 2-aligned
    const float d = fp16_bits_to_f32(blk[0]);
    const int64_t j0 = b * kBlockCols;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const uint32_t two = blk[1 + h];   // bytes qs[2h] (low) and qs[2h+1] (high)
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int l = 4 * h + n;   // byte 2h holds l = 4h, 4h+1; byte 2h+1 holds 4h+2, 4h+3
        const int q = static_cast<int>((two >> (4 * n)) & 0xFu);
        const int64_t j = j0 + l;
        if (j < N) {
          const float w = static_cast<float>(q - 8) * d;
          if (BF16)
            reinterpret_cast<__nv_bfloat16*>(W)[k * N + j] = __float2bfloat16_rn(w);
          else
            reinterpret_cast<float*>(W)[k * N + j] = w;
        }
      }
    }
  }
}

// to_planar: blocks -> planar; else planar -> blocks.  One thread per block.
template <bool TO_PLANAR>
__global__ void __launch_bounds__(256) q4_repack_kernel(uint8_t* dst, const uint8_t* src,
                                                        int64_t nblk, int64_t qs_off) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nblk;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint16_t* s16;
    uint16_t* d16;
    if (TO_PLANAR) {
      s16 = reinterpret_cast<const uint16_t*>(src + i * kBlockBytes);
      reinterpret_cast<uint16_t*>(dst)[i] = s16[0];
      d16 = reinterpret_cast<uint16_t*>(dst + qs_off + i * 16);
#pragma unroll
      for (int h = 0; h < 8; ++h) d16[h] = s16[1 + h];
    } else {
      d16 = reinterpret_cast<uint16_t*>(dst + i * kBlockBytes);
      d16[0] = reinterpret_cast<const uint16_t*>(src)[i];
      s16 = reinterpret_cast<const uint16_t*>(src + qs_off + i * 16);
#pragma unroll
      for (int h = 0; h < 8; ++h) d16[1 + h] = s16[h];
    }
  }
}

static unsigned grid_for(int64_t n) {
  int64_t g = (n + 255) / 256;
  if (g > 152 * 16) g = 152 * 16;
  if (g < 1) g = 1;
  return static_cast<unsigned>(g);
}

cudaError_t launch_dequant(void* W, int w_dtype, const uint8_t* B, int64_t K, int64_t N,
                           cudaStream_t st) {
  const int64_t nb = (N + kBlockCols - 1) / kBlockCols;
  const unsigned g = grid_for(K * nb);
  (void)cudaGetLastError();   // report this launch's error, not an earlier one's
  if (w_dtype == 0)
    q4_dequant_kernel<false><<<g, 256, 0, st>>>(W, B, K, N, nb);
  else
    q4_dequant_kernel<true><<<g, 256, 0, st>>>(W, B, K, N, nb);
  return cudaGetLastError();
}

cudaError_t launch_repack(uint8_t* dst, const uint8_t* src, int64_t K, int64_t N, bool to_planar,
                          cudaStream_t st) {
  const int64_t nb = (N + kBlockCols - 1) / kBlockCols;
  const int64_t nblk = K * nb;
  const int64_t qs_off = (nblk * 2 + 15) / 16 * 16;
  const unsigned g = grid_for(nblk);
  (void)cudaGetLastError();   // report this launch's error, not an earlier one's
  if (to_planar)
    q4_repack_kernel<true><<<g, 256, 0, st>>>(dst, src, nblk, qs_off);
  else
    q4_repack_kernel<false><<<g, 256, 0, st>>>(dst, src, nblk, qs_off);
  return cudaGetLastError();
}

// Q4_0 encoder [C++ DeepSeek engine page §2.2-§2.3 block layout; the pages
// give no scale rule]: per block (row k, columns 32b .. 32b+31), m = the
// element of largest magnitude (first on ties), d = m / -8 stored as fp16
// (nearest even), code q = min(15, trunc(w * (1/d) + 8.5)) with each step
// one fp32 operation (explicitly rounded: no fused multiply-add), 1/d := 0
// when d = 0; padding columns (>= N) get code 8.  One thread per block.
template <bool BF16>
__global__ void __launch_bounds__(256) q4_quantize_kernel(uint8_t* B, const void* W, int64_t K,
                                                          int64_t N, int64_t nb) {
  const int64_t nblk = K * nb;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nblk;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t k = i / nb;
    const int64_t b = i - k * nb;
    const int64_t c0 = b * kBlockCols;
    const int n = static_cast<int>((N - c0) < kBlockCols ? (N - c0) : kBlockCols);
    float v[kBlockCols];
    const size_t base = static_cast<size_t>(k) * N + c0;
    if (BF16) {
      const uint16_t* w = static_cast<const uint16_t*>(W) + base;
#pragma unroll
      for (int l = 0; l < kBlockCols; ++l) v[l] = (l < n) ? bf16_bits_to_f32(w[l]) : 0.f;
    } else {
      const float* w = static_cast<const float*>(W) + base;
      if (n == kBlockCols && (N & 3) == 0) {
#pragma unroll
        for (int l = 0; l < kBlockCols; l += 4) {
          const float4 f = *reinterpret_cast<const float4*>(w + l);
          v[l] = f.x;
          v[l + 1] = f.y;
          v[l + 2] = f.z;
          v[l + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int l = 0; l < kBlockCols; ++l) v[l] = (l < n) ? w[l] : 0.f;
      }
    }
    float amax = 0.f, mx = 0.f;
#pragma unroll
    for (int l = 0; l < kBlockCols; ++l) {
      if (l < n && amax < fabsf(v[l])) {
        amax = fabsf(v[l]);
        mx = v[l];
      }
    }
    const float d = __fdiv_rn(mx, -8.0f);
    const float id = (d != 0.f) ? __fdiv_rn(1.0f, d) : 0.f;
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int l = 0; l < kBlockCols; ++l) {
      int q = 8;
      if (l < n) {
        const float t = __fadd_rn(__fmul_rn(v[l], id), 8.5f);
        q = __float2int_rz(t);
        q = q > 15 ? 15 : (q < 0 ? 0 : q);
      }
      packed[l >> 3] |= static_cast<uint32_t>(q) << (4 * (l & 7));
    }
    uint16_t* dst = reinterpret_cast<uint16_t*>(B + i * kBlockBytes);   // 2-byte aligned
    dst[0] = __half_as_ushort(__float2half_rn(d));
#pragma unroll
    for (int h = 0; h < 8; ++h)
      dst[1 + h] = static_cast<uint16_t>(packed[h >> 1] >> (16 * (h & 1)));
  }
}

cudaError_t launch_quantize(uint8_t* B, const void* W, int w_dtype, int64_t K, int64_t N,
                            cudaStream_t st) {
  const int64_t nb = (N + kBlockCols - 1) / kBlockCols;
  const int64_t nblk = K * nb;
  int64_t grid = (nblk + 255) / 256;
  if (grid > 65536) grid = 65536;
  (void)cudaGetLastError();   // report this launch's error, not an earlier one's
  if (w_dtype == 1)
    q4_quantize_kernel<true><<<static_cast<unsigned>(grid), 256, 0, st>>>(B, W, K, N, nb);
  else
    q4_quantize_kernel<false><<<static_cast<unsigned>(grid), 256, 0, st>>>(B, W, K, N, nb);
  return cudaGetLastError();
}

// One CTA waits, with bounded_wait and a limit of `limit_ns`, on an mbarrier
// that only `arrive` ever completes: the path every pipeline wait takes, run
// to its timeout on purpose (no fault, no hang: the wait gives up, records
// Q4_DEVERR_TIMEOUT in the status word and the kernel returns).
__global__ void __launch_bounds__(32) q4_wait_selftest_kernel(unsigned* err,
                                                              unsigned long long limit_ns,
                                                              int arrive) {
  __shared__ uint64_t bar;
  __shared__ int fail;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fail = 0;
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    if (arrive) mbar_arrive(&bar);
    (void)bounded_wait(&bar, 0, &fail, err, limit_ns);
  }
}

cudaError_t launch_wait_selftest(unsigned* err, unsigned long long limit_ns, bool arrive,
                                 cudaStream_t st) {
  (void)cudaGetLastError();   // report this launch's error, not an earlier one's
  q4_wait_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns, arrive ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace q4
