// Host-streamed weights: a sequence of Q4_0 matmuls whose weights live in
// page-locked host memory (host-side scheduling only; the arithmetic is the
// GEMV/GEMM of q4_matmul_ex).
//
// The AirLLM deep-dive page (§1.2) keeps layers in host memory, pinned so
// that host-to-device copies take the DMA path, and has a worker bring the
// next layer while the GPU computes the current one; its §6 moves the packed
// quantised bytes and expands them on the GPU.  Here the packed Q4_0 blocks
// cross the host link (NVLink-C2C on GB300) on a copy stream, into a ring of
// device slots, and each matmul dequantises in its inner loop as usual:
//
//   copy stream:    H2D(B_0 -> s0)  H2D(B_1 -> s1)  H2D(B_2 -> s2)  [wait mm_0] H2D(B_3 -> s0) ...
//   compute stream:   [wait copy_0] mm_0  [wait copy_1] mm_1  ...
//
// Copy i reuses slot i % slots only after matmul i - slots has finished
// reading it; matmul i starts once copy i has landed.  The copy stream is
// forked from and joined back into the compute stream, so the whole sequence
// is ordered after earlier work on `stream`, everything later on `stream` is
// ordered after it, and the sequence can be captured into a CUDA graph.
#include <cstdint>
#include <cstring>
#include <vector>
#include <cuda_runtime.h>

#include "q4.h"

namespace {

constexpr size_t kSlotAlign = 256;

size_t weight_bytes(const q4_seq_op& op) {
  return static_cast<size_t>(op.K) * static_cast<size_t>((op.N + 31) / 32) * 18u;
}

size_t slot_pitch(const q4_seq_op* ops, int n) {
  size_t m = 0;
  for (int i = 0; i < n; ++i) {
    const size_t b = weight_bytes(ops[i]);
    if (b > m) m = b;
  }
  return (m + kSlotAlign - 1) / kSlotAlign * kSlotAlign;
}

bool pinned_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

// Events of one call, destroyed when it returns (destruction waits for no
// stream: a recorded event is released once its work completes).
struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  bool make(size_t n) {
    ev.reserve(n);
    for (size_t i = 0; i < n; ++i) {
      cudaEvent_t e;
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
      ev.push_back(e);
    }
    return true;
  }
};

}  // namespace

extern "C" {

size_t q4_host_stream_slot_bytes(const q4_seq_op* ops, int n) {
  if (!ops || n <= 0) return 0;
  for (int i = 0; i < n; ++i)
    if (ops[i].K <= 0 || ops[i].N <= 0) return 0;
  return slot_pitch(ops, n);
}

int q4_matmul_host_stream(const q4_seq_op* ops, int n, void* staging, size_t staging_bytes,
                          int slots, void* stream, void* copy_stream) {
  if (!ops || n <= 0 || !staging || slots <= 0 || stream == copy_stream) return Q4_ERR_ARG;
  // everything is checked before anything is enqueued, so that a rejected
  // call leaves no forked stream behind (which would break a graph capture)
  for (int i = 0; i < n; ++i) {
    const q4_seq_op& op = ops[i];
    if (!op.C || !op.A || !op.B || op.M <= 0 || op.N <= 0 || op.K <= 0) return Q4_ERR_ARG;
    if (op.M > (1LL << 30) || op.N > (1LL << 30) || op.K > (1LL << 30)) return Q4_ERR_SHAPE;
    if ((op.a_dtype != Q4_F32 && op.a_dtype != Q4_BF16) ||
        (op.c_dtype != Q4_F32 && op.c_dtype != Q4_BF16))
      return Q4_ERR_DTYPE;
    if (reinterpret_cast<uintptr_t>(op.C) % 16 || reinterpret_cast<uintptr_t>(op.A) % 16)
      return Q4_ERR_ALIGN;
  }
  if (reinterpret_cast<uintptr_t>(staging) % kSlotAlign != 0) return Q4_ERR_ALIGN;
  const size_t pitch = slot_pitch(ops, n);
  if (staging_bytes / pitch < static_cast<size_t>(slots)) return Q4_ERR_WORKSPACE;
  for (int i = 0; i < n; ++i)
    if (!pinned_host(ops[i].B)) return Q4_ERR_ARG;   // page-locked host memory only

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t cp = static_cast<cudaStream_t>(copy_stream);
  const int ns = slots < n ? slots : n;
  Events e;   // [0] fork, [1] join, then per slot: copy done, matmul done
  if (!e.make(2 + 2 * static_cast<size_t>(ns))) return Q4_ERR_CUDA;
  cudaEvent_t fork = e.ev[0], join = e.ev[1];
  auto copy_done = [&](int s) { return e.ev[2 + 2 * s]; };
  auto mm_done = [&](int s) { return e.ev[3 + 2 * s]; };

  if (cudaEventRecord(fork, st) != cudaSuccess || cudaStreamWaitEvent(cp, fork, 0) != cudaSuccess)
    return Q4_ERR_CUDA;
  uint8_t* base = static_cast<uint8_t*>(staging);
  for (int i = 0; i < n; ++i) {
    const q4_seq_op& op = ops[i];
    const int s = i % ns;
    uint8_t* slot = base + static_cast<size_t>(s) * pitch;
    if (i >= ns && cudaStreamWaitEvent(cp, mm_done(s), 0) != cudaSuccess) return Q4_ERR_CUDA;
    if (cudaMemcpyAsync(slot, op.B, weight_bytes(op), cudaMemcpyHostToDevice, cp) != cudaSuccess)
      return Q4_ERR_CUDA;
    if (cudaEventRecord(copy_done(s), cp) != cudaSuccess ||
        cudaStreamWaitEvent(st, copy_done(s), 0) != cudaSuccess)
      return Q4_ERR_CUDA;
    const int rc = q4_matmul_ex(op.C, op.c_dtype, op.A, op.a_dtype, slot, Q4_LAYOUT_BLOCKS, op.M,
                                op.N, op.K, nullptr, 0, stream);
    if (rc != Q4_OK) return rc;
    if (cudaEventRecord(mm_done(s), st) != cudaSuccess) return Q4_ERR_CUDA;
  }
  // join: later work on `stream` follows the last copy too
  if (cudaEventRecord(join, cp) != cudaSuccess || cudaStreamWaitEvent(st, join, 0) != cudaSuccess)
    return Q4_ERR_CUDA;
  return Q4_OK;
}

}  // extern "C"
