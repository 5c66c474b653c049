// Internal interface between the C-ABI layer and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace q4 {

enum : int { kModeGemv = 0, kModeGateUp = 1, kModeDown = 2 };

// Arguments of q4_gemv_kernel (one struct, passed by value).
struct GemvParams {
  int mode;
  // weights: one matrix (GEMV) or expert stacks (B = gate or down, B2 = up)
  const uint8_t* B;
  const uint8_t* B2;
  long long b_stride;   // bytes per expert matrix
  int K, N, nb;
  // split-K tiling (grid.x = column tiles of 8 blocks, grid.y = splits)
  int nsplit, rows_per_split;
  int bulk;             // row segments may use TMA bulk copies
  // activations
  const void* A;
  int a_dtype;          // 0 fp32, 1 bf16
  long long a_ld;       // elements per row of A
  int M;                // GEMV rows
  // outputs
  void* C;
  int c_dtype;
  float* part;          // split partials
  unsigned* tickets;    // one per (z-group, tile); zero between launches
  // routed experts
  const int32_t* topk_idx;
  int nslots, topk, E;
  int list_cap;         // shared-memory list entries (>= nslots, >= ceil(E/32))
  float* h;             // [nslots, I] SiLU(g) * u
  float* y;             // [nslots, H] down outputs
  unsigned* err;        // device status word
};

cudaError_t launch_gemv(const GemvParams& p, int mr, dim3 grid, cudaStream_t st, bool pdl);
uint32_t gemv_smem_bytes(int mr, int rows_per_split, int list_cap);
int gemv_tile_blocks();
cudaError_t launch_moe_combine(float* out, const float* y, const int32_t* idx, const float* w,
                               int T, int topk, int E, int H, cudaStream_t st, bool pdl);

// q4_misc.cu
cudaError_t launch_dequant(void* W, int w_dtype, const uint8_t* B, int64_t K, int64_t N,
                           cudaStream_t st);
cudaError_t launch_repack(uint8_t* dst, const uint8_t* src, int64_t K, int64_t N, bool to_planar,
                          cudaStream_t st);

}  // namespace q4
