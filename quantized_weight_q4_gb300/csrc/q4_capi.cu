// C ABI of the Q4_0 dequant-matmul library: argument checks, launch shapes,
// workspace management and the device status word.  See include/q4.h.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "q4.h"
#include "q4_kernels.h"

namespace {

// Device status word (Q4_DEVERR_* bits), one per device that loads the library.
__device__ unsigned int g_q4_status = 0u;

constexpr int kMaxDevices = 64;
constexpr int kMaxRowsPerSplit = 2048;   // bounds the shared-memory copy of A

struct DeviceState {
  bool init = false;
  int sms = 0;
  unsigned* status = nullptr;   // device address of g_q4_status
  void* ws = nullptr;           // library-owned workspace
  size_t ws_bytes = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
unsigned g_last_flags = 0u;

int current_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return Q4_ERR_CUDA;
  DeviceState& s = g_dev[dev];
  if (!s.init) {
    if (cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return Q4_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_q4_status) != cudaSuccess) return Q4_ERR_CUDA;
    s.status = static_cast<unsigned*>(p);
    s.init = true;
  }
  *out = &s;
  return Q4_OK;
}

// Library-owned workspace of at least `bytes`, zero-filled when (re)allocated.
int owned_workspace(DeviceState* s, size_t bytes, void** ws) {
  if (bytes == 0) {
    *ws = s->ws;
    return Q4_OK;
  }
  if (s->ws_bytes < bytes) {
    if (s->ws) {
      if (cudaDeviceSynchronize() != cudaSuccess) return Q4_ERR_CUDA;
      cudaFree(s->ws);
      s->ws = nullptr;
      s->ws_bytes = 0;
    }
    size_t want = bytes + bytes / 4;
    if (cudaMalloc(&s->ws, want) != cudaSuccess) return Q4_ERR_CUDA;
    if (cudaMemset(s->ws, 0, want) != cudaSuccess) return Q4_ERR_CUDA;
    s->ws_bytes = want;
  }
  *ws = s->ws;
  return Q4_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// GEMV launch shape
// ---------------------------------------------------------------------------
struct GemvShape {
  int mr, nchunks, ntiles, nsplit, rows_per_split;
  size_t ticket_bytes, part_bytes;
};

GemvShape gemv_shape(int64_t M, int64_t N, int64_t K, int sms) {
  GemvShape g;
  const int64_t nb = ceil_div(N, 32);
  g.mr = (M == 1) ? 1 : (M == 2) ? 2 : 4;
  g.nchunks = static_cast<int>(ceil_div(M, g.mr));
  g.ntiles = static_cast<int>(ceil_div(nb, q4::gemv_tile_blocks()));
  const int64_t target = 2LL * sms;
  int64_t nsplit = target / (static_cast<int64_t>(g.ntiles) * g.nchunks);
  if (nsplit < 1) nsplit = 1;
  const int64_t max_split = ceil_div(K, 32);   // at least 32 rows per split
  if (nsplit > max_split) nsplit = max_split;
  const int64_t min_split = ceil_div(K, kMaxRowsPerSplit);
  if (nsplit < min_split) nsplit = min_split;
  int64_t rows = ceil_div(K, nsplit);
  rows = round_up(static_cast<size_t>(rows), 8);
  g.rows_per_split = static_cast<int>(rows);
  g.nsplit = static_cast<int>(ceil_div(K, rows));
  g.ticket_bytes = round_up(static_cast<size_t>(g.ntiles) * g.nchunks * 4, 256);
  g.part_bytes = (g.nsplit > 1) ? static_cast<size_t>(g.nsplit) * M * N * 4 : 0;
  return g;
}

// ---------------------------------------------------------------------------
// Expert launch shapes
// ---------------------------------------------------------------------------
struct MoeShape {
  int nslots, nexp, list_cap;
  int ntiles_gu, nsplit_gu, rows_gu;
  int ntiles_d, nsplit_d, rows_d;
  size_t off_tk_gu, off_tk_d, off_part_gu, off_h, off_part_d, off_y, total;
};

void split_for(int64_t K, int64_t ctas_per_split, int sms, int* nsplit, int* rows) {
  int64_t ns = (2LL * sms) / (ctas_per_split > 0 ? ctas_per_split : 1);
  if (ns < 1) ns = 1;
  if (ns > ceil_div(K, 32)) ns = ceil_div(K, 32);
  if (ns < ceil_div(K, kMaxRowsPerSplit)) ns = ceil_div(K, kMaxRowsPerSplit);
  int64_t r = round_up(static_cast<size_t>(ceil_div(K, ns)), 8);
  *rows = static_cast<int>(r);
  *nsplit = static_cast<int>(ceil_div(K, r));
}

MoeShape moe_shape(int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I, int sms) {
  MoeShape m;
  m.nslots = static_cast<int>(T * topk);
  m.nexp = static_cast<int>(E < m.nslots ? E : m.nslots);
  const int tbk = q4::gemv_tile_blocks();
  m.list_cap = static_cast<int>(m.nslots > ceil_div(E, 32) ? m.nslots : ceil_div(E, 32));
  m.ntiles_gu = static_cast<int>(ceil_div(ceil_div(I, 32), tbk));
  m.ntiles_d = static_cast<int>(ceil_div(ceil_div(H, 32), tbk));
  split_for(H, 2LL * m.ntiles_gu * m.nexp, sms, &m.nsplit_gu, &m.rows_gu);
  split_for(I, 1LL * m.ntiles_d * m.nexp, sms, &m.nsplit_d, &m.rows_d);
  size_t o = 0;
  m.off_tk_gu = o;
  o += round_up(static_cast<size_t>(m.nexp) * m.ntiles_gu * 4, 256);
  m.off_tk_d = o;
  o += round_up(static_cast<size_t>(m.nexp) * m.ntiles_d * 4, 256);
  m.off_part_gu = o;
  o += round_up(2ULL * m.nsplit_gu * m.nslots * I * 4, 256);
  m.off_h = o;
  o += round_up(static_cast<size_t>(m.nslots) * I * 4, 256);
  m.off_part_d = o;
  o += round_up(static_cast<size_t>(m.nsplit_d) * m.nslots * H * 4, 256);
  m.off_y = o;
  o += round_up(static_cast<size_t>(m.nslots) * H * 4, 256);
  m.total = o;
  return m;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? Q4_OK : Q4_ERR_CUDA; }

}  // namespace

extern "C" {

int q4_version(void) { return 100; }

const char* q4_status_str(int status) {
  switch (status) {
    case Q4_OK: return "ok";
    case Q4_ERR_ARG: return "invalid argument (null pointer, non-positive size or bad enum)";
    case Q4_ERR_DTYPE: return "unsupported dtype combination";
    case Q4_ERR_ALIGN: return "pointer not 16-byte aligned";
    case Q4_ERR_CUDA: return "CUDA runtime error";
    case Q4_ERR_WORKSPACE: return "workspace too small";
    case Q4_ERR_SHAPE: return "shape not supported by this entry point";
    case Q4_ERR_DEVICE: return "device-side error recorded (see q4_last_device_flags)";
    default: return "unknown status";
  }
}

size_t q4_matmul_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  DeviceState* s = nullptr;
  int sms = 152;
  if (current_state(&s) == Q4_OK) sms = s->sms;
  const GemvShape g = gemv_shape(M, N, K, sms);
  return g.ticket_bytes + g.part_bytes;
}

int q4_matmul_ex(void* C, int c_dtype, const void* A, int a_dtype, const void* B, int b_layout,
                 int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                 void* stream) {
  if (!C || !A || !B || M <= 0 || N <= 0 || K <= 0) return Q4_ERR_ARG;
  if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30)) return Q4_ERR_SHAPE;
  if ((c_dtype != Q4_F32 && c_dtype != Q4_BF16) || (a_dtype != Q4_F32 && a_dtype != Q4_BF16))
    return Q4_ERR_DTYPE;
  if (b_layout != Q4_LAYOUT_BLOCKS) return (b_layout == Q4_LAYOUT_PLANAR) ? Q4_ERR_SHAPE : Q4_ERR_ARG;
  if (!aligned16(C) || !aligned16(A) || !aligned16(B) || (workspace && !aligned16(workspace)))
    return Q4_ERR_ALIGN;

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int rc = current_state(&s);
  if (rc != Q4_OK) return rc;
  const GemvShape g = gemv_shape(M, N, K, s->sms);
  const size_t need = g.ticket_bytes + g.part_bytes;
  void* ws = workspace;
  if (ws) {
    if (workspace_bytes < need) return Q4_ERR_WORKSPACE;
  } else {
    rc = owned_workspace(s, need, &ws);
    if (rc != Q4_OK) return rc;
  }

  q4::GemvParams p;
  std::memset(&p, 0, sizeof(p));
  p.mode = q4::kModeGemv;
  p.B = static_cast<const uint8_t*>(B);
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.nb = static_cast<int>(ceil_div(N, 32));
  p.nsplit = g.nsplit;
  p.rows_per_split = g.rows_per_split;
  p.bulk = (p.nb % q4::gemv_tile_blocks() == 0) ? 1 : 0;
  p.A = A;
  p.a_dtype = a_dtype;
  p.a_ld = K;
  p.M = static_cast<int>(M);
  p.C = C;
  p.c_dtype = c_dtype;
  p.tickets = static_cast<unsigned*>(ws);
  p.part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + g.ticket_bytes);
  p.list_cap = 0;
  p.err = s->status;
  const dim3 grid(g.ntiles, g.nsplit, g.nchunks);
  return launch_status(q4::launch_gemv(p, g.mr, grid, static_cast<cudaStream_t>(stream), true));
}

int q4_matmul(float* C, const float* A, const void* B, int64_t M, int64_t N, int64_t K) {
  return q4_matmul_ex(C, Q4_F32, A, Q4_F32, B, Q4_LAYOUT_BLOCKS, M, N, K, nullptr, 0, nullptr);
}

size_t q4_moe_workspace_size(int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I) {
  if (T <= 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0) return 0;
  DeviceState* s = nullptr;
  int sms = 152;
  if (current_state(&s) == Q4_OK) sms = s->sms;
  return moe_shape(T, topk, E, H, I, sms).total;
}

int q4_moe_experts_ex(float* out, const void* x, int x_dtype, const void* W_gate, const void* W_up,
                      const void* W_down, const int32_t* topk_idx, const float* topk_w, int64_t T,
                      int64_t topk, int64_t E, int64_t H, int64_t I, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!out || !x || !W_gate || !W_up || !W_down || !topk_idx || !topk_w) return Q4_ERR_ARG;
  if (T <= 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0) return Q4_ERR_ARG;
  if (topk > 16 || T * topk > 8192 || E > (1 << 20) || H > (1 << 24) || I > (1 << 24))
    return Q4_ERR_SHAPE;
  if (x_dtype != Q4_F32 && x_dtype != Q4_BF16) return Q4_ERR_DTYPE;
  if (!aligned16(out) || !aligned16(x) || !aligned16(W_gate) || !aligned16(W_up) ||
      !aligned16(W_down) || !aligned16(topk_idx) || !aligned16(topk_w) ||
      (workspace && !aligned16(workspace)))
    return Q4_ERR_ALIGN;

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int rc = current_state(&s);
  if (rc != Q4_OK) return rc;
  const MoeShape m = moe_shape(T, topk, E, H, I, s->sms);
  void* ws = workspace;
  if (ws) {
    if (workspace_bytes < m.total) return Q4_ERR_WORKSPACE;
  } else {
    rc = owned_workspace(s, m.total, &ws);
    if (rc != Q4_OK) return rc;
  }
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t nbI = ceil_div(I, 32), nbH = ceil_div(H, 32);
  float* h = reinterpret_cast<float*>(w8 + m.off_h);
  float* y = reinterpret_cast<float*>(w8 + m.off_y);

  q4::GemvParams p;
  std::memset(&p, 0, sizeof(p));
  p.topk_idx = topk_idx;
  p.nslots = m.nslots;
  p.topk = static_cast<int>(topk);
  p.E = static_cast<int>(E);
  p.list_cap = m.list_cap;
  p.h = h;
  p.y = y;
  p.err = s->status;
  p.c_dtype = 0;

  // gate and up: K = H, N = I; A rows are tokens
  p.mode = q4::kModeGateUp;
  p.B = static_cast<const uint8_t*>(W_gate);
  p.B2 = static_cast<const uint8_t*>(W_up);
  p.b_stride = static_cast<long long>(H) * nbI * 18;
  p.K = static_cast<int>(H);
  p.N = static_cast<int>(I);
  p.nb = static_cast<int>(nbI);
  p.nsplit = m.nsplit_gu;
  p.rows_per_split = m.rows_gu;
  p.bulk = (p.nb % q4::gemv_tile_blocks() == 0 && p.b_stride % 16 == 0) ? 1 : 0;
  p.A = x;
  p.a_dtype = x_dtype;
  p.a_ld = H;
  p.part = reinterpret_cast<float*>(w8 + m.off_part_gu);
  p.tickets = reinterpret_cast<unsigned*>(w8 + m.off_tk_gu);
  cudaError_t e = q4::launch_gemv(p, 4, dim3(m.ntiles_gu, m.nsplit_gu, 2 * m.nexp), st, true);
  if (e != cudaSuccess) return Q4_ERR_CUDA;

  // down: K = I, N = H; A rows are slots of h
  p.mode = q4::kModeDown;
  p.B = static_cast<const uint8_t*>(W_down);
  p.B2 = nullptr;
  p.b_stride = static_cast<long long>(I) * nbH * 18;
  p.K = static_cast<int>(I);
  p.N = static_cast<int>(H);
  p.nb = static_cast<int>(nbH);
  p.nsplit = m.nsplit_d;
  p.rows_per_split = m.rows_d;
  p.bulk = (p.nb % q4::gemv_tile_blocks() == 0 && p.b_stride % 16 == 0) ? 1 : 0;
  p.A = h;
  p.a_dtype = 0;
  p.a_ld = I;
  p.part = reinterpret_cast<float*>(w8 + m.off_part_d);
  p.tickets = reinterpret_cast<unsigned*>(w8 + m.off_tk_d);
  e = q4::launch_gemv(p, 4, dim3(m.ntiles_d, m.nsplit_d, m.nexp), st, true);
  if (e != cudaSuccess) return Q4_ERR_CUDA;

  e = q4::launch_moe_combine(out, y, topk_idx, topk_w, static_cast<int>(T), static_cast<int>(topk),
                             static_cast<int>(E), static_cast<int>(H), st, true);
  return launch_status(e);
}

int q4_moe_experts(float* out, const void* x, const void* W_gate, const void* W_up,
                   const void* W_down, const int32_t* topk_idx, const float* topk_w, int64_t T,
                   int64_t E, int64_t H, int64_t I) {
  return q4_moe_experts_ex(out, x, Q4_BF16, W_gate, W_up, W_down, topk_idx, topk_w, T, 6, E, H, I,
                           nullptr, 0, nullptr);
}

size_t q4_planar_qs_offset(int64_t K, int64_t N) {
  if (K <= 0 || N <= 0) return 0;
  return round_up(static_cast<size_t>(K * ceil_div(N, 32)) * 2, 16);
}

size_t q4_planar_bytes(int64_t K, int64_t N) {
  if (K <= 0 || N <= 0) return 0;
  return q4_planar_qs_offset(K, N) + static_cast<size_t>(K * ceil_div(N, 32)) * 16;
}

int q4_repack(void* dst, const void* src, int64_t K, int64_t N, void* stream) {
  if (!dst || !src || K <= 0 || N <= 0) return Q4_ERR_ARG;
  if (!aligned16(dst) || !aligned16(src)) return Q4_ERR_ALIGN;
  return launch_status(q4::launch_repack(static_cast<uint8_t*>(dst),
                                         static_cast<const uint8_t*>(src), K, N, true,
                                         static_cast<cudaStream_t>(stream)));
}

int q4_unpack(void* dst, const void* src, int64_t K, int64_t N, void* stream) {
  if (!dst || !src || K <= 0 || N <= 0) return Q4_ERR_ARG;
  if (!aligned16(dst) || !aligned16(src)) return Q4_ERR_ALIGN;
  return launch_status(q4::launch_repack(static_cast<uint8_t*>(dst),
                                         static_cast<const uint8_t*>(src), K, N, false,
                                         static_cast<cudaStream_t>(stream)));
}

int q4_dequant(float* W, const void* B, int64_t K, int64_t N, void* stream) {
  if (!W || !B || K <= 0 || N <= 0) return Q4_ERR_ARG;
  if (!aligned16(W) || !aligned16(B)) return Q4_ERR_ALIGN;
  return launch_status(q4::launch_dequant(W, 0, static_cast<const uint8_t*>(B), K, N,
                                          static_cast<cudaStream_t>(stream)));
}

int q4_dequant_bf16(uint16_t* W, const void* B, int64_t K, int64_t N, void* stream) {
  if (!W || !B || K <= 0 || N <= 0) return Q4_ERR_ARG;
  if (!aligned16(W) || !aligned16(B)) return Q4_ERR_ALIGN;
  return launch_status(q4::launch_dequant(W, 1, static_cast<const uint8_t*>(B), K, N,
                                          static_cast<cudaStream_t>(stream)));
}

int q4_get_device_status(void* stream) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int rc = current_state(&s);
  if (rc != Q4_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return Q4_ERR_CUDA;
  unsigned flags = 0;
  if (cudaMemcpy(&flags, s->status, sizeof(flags), cudaMemcpyDeviceToHost) != cudaSuccess)
    return Q4_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpy(s->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return Q4_ERR_CUDA;
  if ((flags & Q4_DEVERR_TIMEOUT) && s->ws) {
    // a CTA that gave up may have left split-K tickets set
    if (cudaMemset(s->ws, 0, s->ws_bytes) != cudaSuccess) return Q4_ERR_CUDA;
  }
  g_last_flags = flags;
  return flags ? Q4_ERR_DEVICE : Q4_OK;
}

unsigned int q4_last_device_flags(void) { return g_last_flags; }

}  // extern "C"
