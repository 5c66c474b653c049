// C ABI of the Q4_0 dequant-matmul library: argument checks, launch shapes,
// workspace management and the device status word.  See include/q4.h.
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <map>
#include <new>
#include <mutex>
#include <tuple>
#include <vector>

#include <cuda_runtime.h>

#include "q4.h"
#include "q4_kernels.h"

namespace {

// Device status word (Q4_DEVERR_* bits), one per device that loads the library.
__device__ unsigned int g_q4_status = 0u;

constexpr int kMaxDevices = 64;
// The rows of A a CTA uses are copied to shared memory: MR * rows * 4 bytes.
constexpr int64_t kMaxASliceBytes = 64 * 1024;
// Every routed-expert workspace starts with this many bytes of counters for
// the persistent form (zero before the first call, left zero by every call
// whose waits do not time out); nothing else is stored there.
constexpr size_t kMoeHeaderBytes = 64 * 1024;
// From this many rows of bf16 A on, a matmul runs on the tensor cores (the
// split-K small-M form up to 128 rows, the persistent prefill form above);
// below it, and for fp32 A, as split-K GEMVs on the CUDA cores.
constexpr int64_t kMinTensorRows = 8;

struct GemvShape {
  int mr, bpt, nchunks, ntiles, nsplit, rows_per_split;
  bool big;
};

struct MoeShape {
  int mr;
  int nslots, nexp, list_cap;
  int bpt_gu, ntiles_gu, nsplit_gu, rows_gu;
  int bpt_d, ntiles_d, nsplit_d, rows_d;
  bool big_gu, big_d;
  size_t off_h, off_y, total;
};

struct DeviceState {
  bool init = false;
  int sms = 0;
  unsigned* status = nullptr;   // device address of g_q4_status
  void* ws = nullptr;           // library-owned workspace
  size_t ws_bytes = 0;
  // launch shapes already chosen for a problem size (the choice runs occupancy queries)
  std::map<std::tuple<int64_t, int64_t, int64_t, int>, GemvShape> gemv_shapes;
  std::map<std::tuple<int64_t, int64_t, int64_t, int64_t, int64_t>, MoeShape> moe_shapes;
  // per stream (keyed by its cudaStreamGetId, so that one handle naming a
  // different stream in each host thread, as cudaStreamPerThread does, gets
  // one entry per stream): the small-M GEMM's partial tiles and its zeroed
  // tile tickets.  Only eager calls use it; a stream being captured never
  // does, so no CUDA graph holds these pointers.
  struct GemmScratch {
    float* part = nullptr;
    size_t part_bytes = 0;
    unsigned* tickets = nullptr;
  };
  std::map<unsigned long long, GemmScratch> gemm_scratch;
  // library-owned workspaces replaced by larger ones: a CUDA graph captured
  // while one was current may still use it, so it is kept until
  // q4_release_scratch()
  std::vector<void*> retired;
  // the persistent sequence kernel's ring depth and resident CTAs per SM
  // (0 until first needed)
  int seq_stages = 0, seq_per_sm = 0;
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

// True if `st` is being captured into a CUDA graph (or its state cannot be read).
bool capturing(cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
    cudaGetLastError();
    return true;
  }
  return cs != cudaStreamCaptureStatusNone;
}

// The small-M GEMM's library scratch for stream `st`: partial tiles (at least
// `bytes`) and a zeroed ticket array.  Eager calls only: it returns false for
// a stream being captured (no graph may hold library scratch, whose buffers a
// later, larger call replaces) and when it cannot allocate; the caller then
// takes the cluster form.  A buffer outgrown by a later call is freed after
// the stream has drained, since only that stream's kernels use it.
bool gemm_scratch(DeviceState* s, cudaStream_t st, size_t bytes, float** part,
                  unsigned** tickets) {
  if (capturing(st)) return false;
  unsigned long long id = 0;
  if (cudaStreamGetId(st, &id) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  DeviceState::GemmScratch& g = s->gemm_scratch[id];
  if (!g.tickets) {
    unsigned* t = nullptr;
    const size_t tb = q4::kMaxGemmTickets * sizeof(unsigned);
    if (cudaMalloc(&t, tb) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (cudaMemsetAsync(t, 0, tb, st) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(t);
      return false;
    }
    g.tickets = t;
  }
  if (g.part_bytes < bytes) {
    if (g.part) {   // kernels on this stream may still read the old buffer
      if (cudaStreamSynchronize(st) != cudaSuccess) return false;
      cudaFree(g.part);
      g.part = nullptr;
      g.part_bytes = 0;
    }
    const size_t want = bytes + bytes / 4;
    if (cudaMalloc(&g.part, want) != cudaSuccess) {
      cudaGetLastError();
      g.part = nullptr;
      return false;
    }
    g.part_bytes = want;
  }
  *part = g.part;
  *tickets = g.tickets;
  return true;
}

// Library-owned workspace of at least `bytes`.  A larger one is allocated
// only outside stream capture (Q4_ERR_WORKSPACE while `st` is captured); the
// one it replaces is retired, not freed, because a graph captured earlier may
// still use it.
int owned_workspace(DeviceState* s, size_t bytes, cudaStream_t st, void** ws) {
  if (bytes == 0) {
    *ws = s->ws;
    return Q4_OK;
  }
  if (s->ws_bytes < bytes) {
    if (capturing(st)) return Q4_ERR_WORKSPACE;
    const size_t want = bytes + bytes / 4;
    void* p = nullptr;
    if (cudaMalloc(&p, want) != cudaSuccess) {
      cudaGetLastError();
      return Q4_ERR_CUDA;
    }
    // zero (the routed-expert counters in its header start at zero)
    if (cudaMemset(p, 0, want) != cudaSuccess) {
      cudaFree(p);
      return Q4_ERR_CUDA;
    }
    if (s->ws) s->retired.push_back(s->ws);
    s->ws = p;
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
// Rows per split for `nsplit` splits: a multiple of the TMA box height.
int64_t split_rows(int64_t K, int64_t nsplit, int bpt, bool big) {
  return static_cast<int64_t>(round_up(static_cast<size_t>(ceil_div(K, nsplit)),
                                       q4::gemv_stage_rows(bpt, big)));
}

constexpr double kCtaFixedBytes = 48.0 * 1024;
// Slices of at least this many 18 KB stages stream with them; shorter slices
// keep 32-row stages, which fill and drain the pipeline sooner.  With two or
// four rows of A the decode per stage is longer and the 18 KB stages pay off
// sooner (measured on GB300).
int64_t big_min_stages(int mr) { return mr == 1 ? 16 : 4; }

// Picks the blocks-per-thread and the split count (at most `max_split`; the
// splits of a column tile form one cluster of `pair * nsplit` CTAs) that
// minimise the bytes the busiest SM must stream: waves of resident clusters
// (from the occupancy query) times the CTAs per SM within a wave times the
// bytes per CTA plus its fixed cost.  Ties go to fewer CTAs.
void choose_split(int mode, int mr, int fmt, int list_cap, int64_t K, int64_t nb, int64_t z_groups,
                  int pair, int sms, int max_split, bool allow_bpt2, int* bpt_out,
                  int* nsplit_out, int* rows_out, int* ntiles_out, bool* big_out) {
  const double block_bytes = (fmt == q4::kFmtQ8) ? 34.0 : 18.0;
  double best = -1.0;
  int64_t best_ctas = 0;
  *bpt_out = 1;
  *nsplit_out = 1;
  *big_out = false;
  *rows_out = static_cast<int>(split_rows(K, 1, 1, false));
  *ntiles_out = static_cast<int>(ceil_div(nb, q4::gemv_tile_blocks(1)));
  for (int bpt = 2; bpt >= 1; --bpt) {
    if (bpt == 2 && !allow_bpt2) continue;
    const int64_t ntiles = ceil_div(nb, q4::gemv_tile_blocks(bpt));
    for (int64_t ns = 1; ns <= max_split; ++ns) {
      const int64_t rows = split_rows(K, ns, bpt, false);
      const int64_t nsplit = ceil_div(K, rows);
      if (nsplit != ns) continue;
      const int64_t csize = pair * nsplit;
      const int64_t clusters = ntiles * z_groups;
      const int64_t ctas = clusters * csize;
      const int active = q4::max_active_clusters(mode, mr, bpt, false, fmt, static_cast<int>(rows),
                                                 list_cap,
                                                 dim3(1, static_cast<unsigned>(nsplit),
                                                      static_cast<unsigned>(pair)));
      if (active <= 0) continue;
      const int64_t waves = ceil_div(clusters, active);
      const int64_t per_wave = (clusters < active ? clusters : active) * csize;
      // a CTA's fixed cost (first loads, reduction, cluster combine: ~2.5 us)
      // is worth about kCtaFixedBytes of streaming
      const double per_cta = static_cast<double>(rows) * q4::gemv_tile_blocks(bpt) * block_bytes +
                             kCtaFixedBytes;
      double cost = per_cta * static_cast<double>(waves * ceil_div(per_wave, sms));
      if (bpt == 1 && allow_bpt2) cost *= 1.03;   // more instructions per weight
      if (best < 0 || cost < best * 0.999 || (cost <= best * 1.001 && ctas < best_ctas)) {
        best = cost;
        best_ctas = ctas;
        *bpt_out = bpt;
        *nsplit_out = static_cast<int>(nsplit);
        *rows_out = static_cast<int>(rows);
        *ntiles_out = static_cast<int>(ntiles);
      }
    }
  }
  // long slices: the same split with 18 KB stages, if it keeps its split count
  // and its residency
  const int bpt = *bpt_out;
  const int64_t big_rows = q4::gemv_stage_rows(bpt, true);
  if (fmt != q4::kFmtQ8 && *rows_out >= big_min_stages(mr) * big_rows) {
    const int64_t rows = split_rows(K, *nsplit_out, bpt, true);
    const dim3 cl(1, static_cast<unsigned>(*nsplit_out), static_cast<unsigned>(pair));
    if (ceil_div(K, rows) == *nsplit_out &&
        q4::max_active_clusters(mode, mr, bpt, true, fmt, static_cast<int>(rows), list_cap, cl) >=
            q4::max_active_clusters(mode, mr, bpt, false, fmt, *rows_out, list_cap, cl)) {
      *big_out = true;
      *rows_out = static_cast<int>(rows);
    }
  }
}

GemvShape gemv_shape(int64_t M, int64_t N, int64_t K, int fmt, int sms) {
  GemvShape g;
  const int64_t nb = ceil_div(N, 32);
  // rows of A per pass: three rows run as three one-row chunks (1.76 TB/s on
  // 5120x12288, bf16 A) rather than one four-row chunk with a padded row
  // (1.43 TB/s); two and four rows keep one chunk (measured on GB300)
  g.mr = (M == 1 || M == 3) ? 1 : (M == 2) ? 2 : 4;
  g.nchunks = static_cast<int>(ceil_div(M, g.mr));
  choose_split(q4::kModeGemv, g.mr, fmt, 0, K, nb, g.nchunks, 1, sms, q4::kMaxCluster, g.mr == 1,
               &g.bpt, &g.nsplit, &g.rows_per_split, &g.ntiles, &g.big);
  return g;
}

// ---------------------------------------------------------------------------
// Expert launch shapes
// ---------------------------------------------------------------------------
MoeShape moe_shape(int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I, int sms) {
  MoeShape m;
  m.nslots = static_cast<int>(T * topk);
  m.nexp = static_cast<int>(E < m.nslots ? E : m.nslots);
  // one token per expert is the common case at T = 1; larger T gathers a few
  m.mr = (T == 1) ? 1 : 2;
  m.list_cap = static_cast<int>(m.nslots > ceil_div(E, 32) ? m.nslots : ceil_div(E, 32));
  // gate and up of one expert tile share a cluster: at most 8 splits each
  choose_split(q4::kModeGateUp, m.mr, q4::kFmtQ4, m.list_cap, H, ceil_div(I, 32), m.nexp, 2, sms,
               q4::kMaxCluster / 2, m.mr == 1, &m.bpt_gu, &m.nsplit_gu, &m.rows_gu, &m.ntiles_gu,
               &m.big_gu);
  choose_split(q4::kModeDown, m.mr, q4::kFmtQ4, m.list_cap, I, ceil_div(H, 32), m.nexp, 1, sms,
               q4::kMaxCluster, m.mr == 1, &m.bpt_d, &m.nsplit_d, &m.rows_d, &m.ntiles_d, &m.big_d);
  size_t o = 0;
  m.off_h = o;
  o += round_up(static_cast<size_t>(m.nslots) * I * 4, 256);
  m.off_y = o;
  o += round_up(static_cast<size_t>(m.nslots) * H * 4, 256);
  m.total = o;
  return m;
}

const GemvShape& cached_gemv_shape(DeviceState* s, int64_t M, int64_t N, int64_t K, int fmt) {
  const auto key = std::make_tuple(M, N, K, fmt);
  auto it = s->gemv_shapes.find(key);
  if (it == s->gemv_shapes.end())
    it = s->gemv_shapes.emplace(key, gemv_shape(M, N, K, fmt, s->sms)).first;
  return it->second;
}

const MoeShape& cached_moe_shape(DeviceState* s, int64_t T, int64_t topk, int64_t E, int64_t H,
                                 int64_t I) {
  const auto key = std::make_tuple(T, topk, E, H, I);
  auto it = s->moe_shapes.find(key);
  if (it == s->moe_shapes.end())
    it = s->moe_shapes.emplace(key, moe_shape(T, topk, E, H, I, s->sms)).first;
  return it->second;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? Q4_OK : Q4_ERR_CUDA; }

// The persistent sequence kernel's ring depth (3 stages of 36 KB where two
// CTAs fit on an SM, else 2) and resident CTAs per SM; Q4_ERR_CUDA if it
// cannot launch.
int seq_residency(DeviceState* s) {
  if (s->seq_per_sm == 0) {
    int stages = 3;
    int per_sm = q4::seq_ctas_per_sm(stages, true);
    if (per_sm < 2) {
      stages = 2;
      per_sm = q4::seq_ctas_per_sm(stages, true);
    }
    if (per_sm < 1) return Q4_ERR_CUDA;
    s->seq_stages = stages;
    s->seq_per_sm = per_sm;
  }
  return Q4_OK;
}

}  // namespace

namespace {

// The split-K GEMV of q4_matmul_ex for a validated problem (the caller holds
// g_mu): C [M, N] = A [M, K] . W, weights in format `fmt`.
int gemv_run(DeviceState* s, void* C, int c_dtype, const void* A, int a_dtype, const void* B,
             int fmt, int64_t M, int64_t N, int64_t K, cudaStream_t st) {
  const GemvShape& g = cached_gemv_shape(s, M, N, K, fmt);
  if (g.nchunks > 65535 || 4LL * g.mr * g.rows_per_split > kMaxASliceBytes) return Q4_ERR_SHAPE;

  q4::GemvParams p;
  std::memset(&p, 0, sizeof(p));
  p.mode = q4::kModeGemv;
  p.B = static_cast<const uint8_t*>(B);
  p.K = static_cast<int>(K);
  p.N = static_cast<int>(N);
  p.nb = static_cast<int>(ceil_div(N, 32));
  p.nsplit = g.nsplit;
  p.rows_per_split = g.rows_per_split;
  q4::fill_decode_consts(p, fmt);
  const int64_t block_bytes = (fmt == q4::kFmtQ8) ? 34 : 18;
  if (fmt == q4::kFmtQ4P) {
    p.qs_offset = static_cast<long long>(q4_planar_qs_offset(K, N));
    p.use_tma = (p.nb % 8 == 0 &&
                 q4::encode_planar_tmaps(p.tmap, B, K, p.nb, p.qs_offset, g.bpt, g.big))
                    ? 1 : 0;
  } else {
    p.use_tma = (p.nb % 8 == 0 &&
                 q4::encode_weight_tmap(&p.tmap[0], B, K, p.nb, 1, K * p.nb * block_bytes, g.bpt,
                                        g.big, fmt))
                    ? 1 : 0;
  }
  p.A = A;
  p.a_dtype = a_dtype;
  p.a_ld = K;
  p.M = static_cast<int>(M);
  p.C = C;
  p.c_dtype = c_dtype;
  p.list_cap = 0;
  p.err = s->status;
  const dim3 grid(g.ntiles, g.nsplit, g.nchunks);
  return launch_status(q4::launch_gemv(p, g.mr, g.bpt, g.big, fmt, grid, dim3(1, g.nsplit, 1),
                                       st, true));
}

// ---------------------------------------------------------------------------
// Routed experts of several tokens on the persistent sequence kernel: one
// launch for every slot's gate, up and down, then the slot combine.  Op 0
// pairs gate and up of each slot (s = t * topk + k, expert topk_idx[s], A =
// x[t]); the last K slice of a slot's column tile adds both products and
// forms h = SiLU(g) * u there, then counts the tile for the slot.  Op 1, down,
// is segmented over the slots along its output (y[s] = h[s] . W_down[e]);
// each slot's units wait only for that slot's h.  The launch takes its
// counters from the workspace header and leaves them zero.  Below
// kMoeSeqMinTokens tokens the three-launch form measured faster (DeepSeek-V2
// experts, GB/s of distinct expert weights: one token 1974 against 2796, two
// tokens 2464 against 2623; four tokens 3537 against 2641).
// ---------------------------------------------------------------------------
constexpr int64_t kMoeSeqMinTokens = 4;
constexpr int64_t kMoeSeqMaxSlots = 512;
// Most K rows per gate/up unit (DeepSeek-V2 experts, GB/s at 4 / 8 / 32
// tokens: slices of 2560 rows 3562 / 4163 / 3138; 2048 + 2048 + 1024 rows
// 3101 / 3930 / 3086; 1024 rows 3537 / 3850 / 2996).
constexpr int kMoeGuRows = 2560;

struct MoeSeqPlan {
  bool ok = false;
  int rows_gu = 0, rows_d = 0;        // K rows per unit of gate/up and of down
  int seg_tiles = 0, slices_gu = 0;   // gate/up: column tiles per slot, K slices
  int tiles_d = 0, slices_d = 0;      // down: column tiles per slot, K slices
  int units_gu = 0, units = 0, ntickets = 0;
  size_t off_g = 0, off_u = 0, off_h = 0, off_y = 0, off_part = 0, total = 0;   // data layout
};

MoeSeqPlan moe_seq_plan(int64_t T, int64_t topk, int64_t H, int64_t I, int x_dtype) {
  MoeSeqPlan q;
  const int64_t S = T * topk;
  const int64_t es = x_dtype == Q4_F32 ? 4 : 2;
  // whole 16-byte tensor-map rows; rows of x and of h start 16-byte aligned
  if (T < kMoeSeqMinTokens || S > kMoeSeqMaxSlots || ceil_div(I, 32) % 8 != 0 ||
      ceil_div(H, 32) % 8 != 0 || (H * es) % 16 != 0 || I % 4 != 0)
    return q;
  const int64_t tc = q4::seq_tile_cols(), stage = q4::seq_stage_rows();
  q.seg_tiles = static_cast<int>(ceil_div(I, tc));
  q.tiles_d = static_cast<int>(ceil_div(H, tc));
  // K slices of equal length (whole stages): an uneven last slice leaves its
  // units short of the others at the end of the sweep
  auto even_rows = [stage](int64_t K, int64_t most) {
    return static_cast<int>(round_up(ceil_div(K, ceil_div(K, most)), stage));
  };
  q.rows_gu = even_rows(H, kMoeGuRows);
  q.rows_d = even_rows(I, q4::seq_max_slice_rows());
  q.slices_gu = static_cast<int>(ceil_div(H, q.rows_gu));
  q.slices_d = static_cast<int>(ceil_div(I, q.rows_d));
  const int64_t units_gu = 2 * S * q.seg_tiles * q.slices_gu;
  const int64_t units = units_gu + S * q.tiles_d * q.slices_d;
  const int64_t tickets = S * q.seg_tiles + (q.slices_d > 1 ? S * q.tiles_d : 0);
  if (units > (1 << 24) || 4 * (2 + 2 + S + tickets) > static_cast<int64_t>(kMoeHeaderBytes))
    return q;
  q.units_gu = static_cast<int>(units_gu);
  q.units = static_cast<int>(units);
  q.ntickets = static_cast<int>(tickets);
  size_t o = 0;
  for (size_t* off : {&q.off_g, &q.off_u, &q.off_h}) {
    *off = o;
    o += round_up(static_cast<size_t>(S * I) * 4, 256);
  }
  q.off_y = o;
  o += round_up(static_cast<size_t>(S * H) * 4, 256);
  q.off_part = o;
  o += static_cast<size_t>(q.slices_d > 1 ? units : units_gu) * tc * 4;
  q.total = o;
  q.ok = true;
  return q;
}

// Bytes after the header of a routed-expert workspace for the three-launch
// form (the least any call needs), and for the form the call prefers.
size_t moe_old_data_bytes(int64_t T, int64_t topk, int64_t H, int64_t I) {
  const size_t nslots = static_cast<size_t>(T * topk);
  return round_up(nslots * I * 4, 256) + round_up(nslots * H * 4, 256);
}
size_t moe_data_bytes(int64_t T, int64_t topk, int64_t H, int64_t I) {
  const MoeSeqPlan q = moe_seq_plan(T, topk, H, I, Q4_BF16);
  const MoeSeqPlan q32 = moe_seq_plan(T, topk, H, I, Q4_F32);
  size_t b = moe_old_data_bytes(T, topk, H, I);
  if (q.ok) b = std::max(b, q.total);
  if (q32.ok) b = std::max(b, q32.total);
  return b;
}

}  // namespace

namespace q4 {
size_t moe_min_workspace_bytes(int64_t T, int64_t topk, int64_t H, int64_t I) {
  return kMoeHeaderBytes + moe_old_data_bytes(T, topk, H, I);
}
}  // namespace q4

namespace {

int moe_seq_run(DeviceState* s, const MoeSeqPlan& q, void* counters, void* data, float* out,
                const void* x, int x_dtype, const void* W_gate, const void* W_up,
                const void* W_down, const int32_t* topk_idx, const float* topk_w, int64_t T,
                int64_t topk, int64_t E, int64_t H, int64_t I, const float* addend,
                cudaStream_t st, float* g_trace, float* u_trace, float* h_trace,
                float* y_trace) {
  int rc = seq_residency(s);
  if (rc != Q4_OK) return rc;
  const int64_t S = T * topk;
  uint8_t* d8 = static_cast<uint8_t*>(data);
  float* g = g_trace ? g_trace : reinterpret_cast<float*>(d8 + q.off_g);
  float* u = u_trace ? u_trace : reinterpret_cast<float*>(d8 + q.off_u);
  float* h = h_trace ? h_trace : reinterpret_cast<float*>(d8 + q.off_h);
  float* y = y_trace ? y_trace : reinterpret_cast<float*>(d8 + q.off_y);
  const int64_t nbI = ceil_div(I, 32), nbH = ceil_div(H, 32);

  q4::SeqParams p;
  std::memset(&p, 0, sizeof(p));
  q4::SeqOpDesc& gu = p.inl[0];
  if (!q4::encode_weight_tmap(&gu.tmap, W_gate, H, nbI, E, H * nbI * 18, 2, true, q4::kFmtQ4) ||
      !q4::encode_weight_tmap(&gu.tmap2, W_up, H, nbI, E, H * nbI * 18, 2, true, q4::kFmtQ4))
    return Q4_ERR_CUDA;
  gu.A = x;
  gu.C = g;
  gu.C2 = u;
  gu.h = h;
  gu.eidx = topk_idx;
  gu.K = static_cast<int>(H);
  gu.N = static_cast<int>(2 * S * I);
  gu.nb = static_cast<int>(nbI);
  gu.ntiles = static_cast<int>(2 * S) * q.seg_tiles;
  gu.nslices = q.slices_gu;
  gu.slice_rows = q.rows_gu;
  gu.unit_base = 0;
  gu.ticket_base = 0;
  gu.a_dtype = x_dtype;
  gu.c_dtype = Q4_F32;
  gu.seg_mode = 1;
  gu.nseg = static_cast<int>(2 * S);
  gu.seg_len = static_cast<int>(I);
  gu.seg_tiles = q.seg_tiles;
  gu.a_seg_div = static_cast<int>(2 * topk);   // segments 2s, 2s + 1: token s / topk
  gu.a_seg_stride = static_cast<int>(H);
  gu.pair = 1;
  gu.seg_done_base = 0;
  gu.seg_need = 0;   // no per-slot dependency
  gu.E = static_cast<int>(E);

  q4::SeqOpDesc& d = p.inl[1];
  if (!q4::encode_weight_tmap(&d.tmap, W_down, I, nbH, E, I * nbH * 18, 2, true, q4::kFmtQ4))
    return Q4_ERR_CUDA;
  d.A = h;
  d.C = y;
  d.eidx = topk_idx;
  d.K = static_cast<int>(I);
  d.N = static_cast<int>(S * H);
  d.nb = static_cast<int>(nbH);
  d.ntiles = static_cast<int>(S) * q.tiles_d;
  d.nslices = q.slices_d;
  d.slice_rows = q.rows_d;
  d.unit_base = q.units_gu;
  d.ticket_base = static_cast<int>(S) * q.seg_tiles;
  d.a_dtype = Q4_F32;
  d.c_dtype = Q4_F32;
  d.seg_mode = 1;
  d.nseg = static_cast<int>(S);
  d.seg_len = static_cast<int>(H);
  d.seg_tiles = q.tiles_d;
  d.a_seg_div = 1;
  d.a_seg_stride = static_cast<int>(I);
  d.seg_dep = 0;
  d.seg_need = q.seg_tiles;
  d.E = static_cast<int>(E);

  unsigned* c = static_cast<unsigned*>(counters);
  p.ops = nullptr;
  p.nops = 2;
  p.total_units = q.units;
  p.queue = c;
  p.exits = c + 1;
  p.done = c + 2;
  p.seg_done = c + 4;
  p.nseg_done = static_cast<int>(S);
  p.tickets = c + 4 + S;
  p.ntickets = q.ntickets;
  p.reset = 1;
  p.part = reinterpret_cast<float*>(d8 + q.off_part);
  p.err = s->status;
  for (int i = 0; i < 4; ++i) p.kmask[i] = 0xFu << (4 * i);
  const int grid = std::min(s->seq_per_sm * s->sms, q.units);
  cudaError_t e = q4::launch_gemv_seq(p, grid, s->seq_stages, st, true, true);
  if (e != cudaSuccess) return Q4_ERR_CUDA;
  if (!out) return Q4_OK;
  return launch_status(q4::launch_moe_combine(out, y, topk_idx, topk_w, addend,
                                              static_cast<int>(T), static_cast<int>(topk),
                                              static_cast<int>(E), static_cast<int>(H), st, true));
}

// Where moe_run with `out` null leaves the per-slot down outputs y [T*topk,
// H] in the data part `ws`.
float* moe_y_rows(void* ws, const MoeShape& m, bool seq_form, int64_t T, int64_t topk, int64_t H,
                  int64_t I, int x_dtype) {
  const size_t off = seq_form ? moe_seq_plan(T, topk, H, I, x_dtype).off_y : m.off_y;
  return reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + off);
}

// Whether the call runs the persistent form: its shape and a data part of
// `data_bytes` (the rest of the workspace after the header) large enough.
bool moe_takes_seq(int64_t T, int64_t topk, int64_t H, int64_t I, int x_dtype, size_t data_bytes) {
  const MoeSeqPlan q = moe_seq_plan(T, topk, H, I, x_dtype);
  return q.ok && data_bytes >= q.total;
}

// The routed experts for a validated problem: the persistent form
// (moe_seq_run) where moe_takes_seq, else the gate/up, down and slot combine
// kernels.  `counters` is the workspace header (kMoeHeaderBytes, zero), `ws`
// the rest (`data_bytes` of it, at least moe_old_data_bytes).  The combine
// adds `addend` (fp32 [T, H], or null) after the weighted sum.  With `out`
// null the combine is left out and the per-slot down outputs stay in the
// workspace (moe_y_rows).  The trace pointers, when given, receive g, u, h
// and y.
int moe_run(DeviceState* s, const MoeShape& m, float* out, const void* x, int x_dtype,
            const void* W_gate, const void* W_up, const void* W_down, const int32_t* topk_idx,
            const float* topk_w, int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I,
            void* counters, void* ws, size_t data_bytes, const float* addend, cudaStream_t st,
            float* g_trace = nullptr, float* u_trace = nullptr, float* h_trace = nullptr,
            float* y_trace = nullptr) {
  if (moe_takes_seq(T, topk, H, I, x_dtype, data_bytes))
    return moe_seq_run(s, moe_seq_plan(T, topk, H, I, x_dtype), counters, ws, out, x, x_dtype,
                       W_gate, W_up, W_down, topk_idx, topk_w, T, topk, E, H, I, addend, st,
                       g_trace, u_trace, h_trace, y_trace);
  if (4LL * m.mr * m.rows_gu > kMaxASliceBytes || 4LL * m.mr * m.rows_d > kMaxASliceBytes)
    return Q4_ERR_SHAPE;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
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
  p.g_trace = g_trace;
  p.u_trace = u_trace;
  p.err = s->status;
  p.c_dtype = 0;
  q4::fill_decode_consts(p, q4::kFmtQ4);

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
  p.use_tma = (p.nb % 8 == 0 && p.b_stride % 16 == 0 &&
               q4::encode_weight_tmap(&p.tmap[0], W_gate, H, p.nb, E, p.b_stride, m.bpt_gu,
                                      m.big_gu, q4::kFmtQ4) &&
               q4::encode_weight_tmap(&p.tmap[1], W_up, H, p.nb, E, p.b_stride, m.bpt_gu,
                                      m.big_gu, q4::kFmtQ4))
                  ? 1 : 0;
  p.A = x;
  p.a_dtype = x_dtype;
  p.a_ld = H;
  cudaError_t e = q4::launch_gemv(p, m.mr, m.bpt_gu, m.big_gu, q4::kFmtQ4,
                                  dim3(m.ntiles_gu, m.nsplit_gu, 2 * m.nexp),
                                  dim3(1, m.nsplit_gu, 2), st, true);
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
  p.use_tma = (p.nb % 8 == 0 && p.b_stride % 16 == 0 &&
               q4::encode_weight_tmap(&p.tmap[0], W_down, I, p.nb, E, p.b_stride, m.bpt_d, m.big_d,
                                      q4::kFmtQ4))
                  ? 1 : 0;
  p.A = h;
  p.a_dtype = 0;
  p.a_ld = I;
  e = q4::launch_gemv(p, m.mr, m.bpt_d, m.big_d, q4::kFmtQ4, dim3(m.ntiles_d, m.nsplit_d, m.nexp),
                      dim3(1, m.nsplit_d, 1), st, true);
  if (e != cudaSuccess) return Q4_ERR_CUDA;

  if (h_trace && cudaMemcpyAsync(h_trace, h, static_cast<size_t>(m.nslots) * I * 4,
                                 cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return Q4_ERR_CUDA;
  if (y_trace && cudaMemcpyAsync(y_trace, y, static_cast<size_t>(m.nslots) * H * 4,
                                 cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return Q4_ERR_CUDA;
  if (!out) return Q4_OK;
  e = q4::launch_moe_combine(out, y, topk_idx, topk_w, addend, static_cast<int>(T),
                             static_cast<int>(topk), static_cast<int>(E), static_cast<int>(H), st,
                             true);
  return launch_status(e);
}


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

}  // extern "C"

namespace {
// Shapes the tensor-core GEMM takes at all (bf16 A).
bool gemm_shape_ok(int64_t M, int64_t N, int64_t K) {
  return M >= kMinTensorRows && q4::gemm_supported(M, N, K) &&
         (M > 128 || q4::gemm_small_split(M, N, K) > 0);
}

// Shapes whose q4_matmul_ex runs the tensor-core GEMM.  Below kMinTensorK the
// bf16 tile rounding (up to 2^-8 relative per weight) is not averaged out over
// enough products to keep |err| <= 1e-3 * sum|a*w| on random data, so short
// reductions take the exact-dequant GEMV.
constexpr int64_t kMinTensorK = 1024;
bool takes_gemm(int fmt, int a_dtype, int64_t M, int64_t N, int64_t K) {
  return fmt == q4::kFmtQ4 && a_dtype == Q4_BF16 && K >= kMinTensorK && gemm_shape_ok(M, N, K);
}

// Caller workspace of the tensor-core forms that add K slices through global
// memory: the tile tickets (zero before first use, left zero by every
// completed call), then the partial tiles.
size_t gemm_ticket_bytes(int64_t N) { return round_up(static_cast<size_t>(ceil_div(N, 256)) * 4, 256); }

// The few-row form (weights as the MMA's A operand) takes bf16 A with up to
// 32 rows.  Measured on 5120 x 12288 (GB/s of weights): 1425 / 1360 / 1253 /
// 1107 at M = 4 / 8 / 16 / 32 against 1396 (split-K GEMV) / 1085 / 1094 /
// 1152 (the GEMM's split forms); at M = 2 the GEMV (2110) and at M = 64 the
// cluster form (989 against 830) are faster.
constexpr int64_t kMaxSkinnyRows = 32;
constexpr int64_t kMinSkinnyRows = 4;
bool takes_skinny(int64_t M, int64_t N, int64_t K) {
  return M <= kMaxSkinnyRows && q4::skinny_supported(M, N, K);
}

// The few-row form for a validated problem (the caller holds g_mu).  Its K
// slices meet in the caller's workspace, else in the stream's library scratch
// (eager calls only); a call captured without a workspace returns
// Q4_ERR_SHAPE so that the caller takes another form.
int skinny_run(DeviceState* s, void* C, int c_dtype, const void* A, const void* B, int64_t M,
               int64_t N, int64_t K, void* workspace, size_t workspace_bytes, cudaStream_t st) {
  const int S = q4::skinny_split(N, K, s->sms);
  float* part = nullptr;
  unsigned* tickets = nullptr;
  if (S > 1) {
    const size_t tb = gemm_ticket_bytes(N);
    const size_t pb = q4::skinny_part_bytes(M, N, S);
    if (workspace && workspace_bytes >= tb + pb) {
      tickets = static_cast<unsigned*>(workspace);
      part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + tb);
    } else if (!gemm_scratch(s, st, pb, &part, &tickets)) {
      return Q4_ERR_SHAPE;
    }
  }
  return launch_status(
      q4::launch_skinny(C, c_dtype, A, B, M, N, K, s->status, S, part, tickets, st));
}

// The tensor-core GEMM for a validated problem (the caller holds g_mu).
int gemm_run(DeviceState* s, void* C, int c_dtype, const void* A, const void* B, int64_t M,
             int64_t N, int64_t K, void* workspace, size_t workspace_bytes, cudaStream_t st) {
  float* part = nullptr;
  unsigned* tickets = nullptr;
  if (M > 128) {
    // prefill form: the last round's tiles share K over the grid when the
    // tail's tickets and partial tiles are at hand (the caller's workspace,
    // else the stream's library scratch for an eager call)
    const q4::PrefillPlan pl = q4::prefill_plan(M, N, K, s->sms);
    const size_t need = q4::prefill_tail_bytes(pl);
    if (need > 0) {
      const size_t tb = q4::prefill_tail_ticket_bytes(pl);
      if (workspace && workspace_bytes >= need) {
        tickets = static_cast<unsigned*>(workspace);
        part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + tb);
      } else if (!gemm_scratch(s, st, need - tb, &part, &tickets)) {
        part = nullptr;
        tickets = nullptr;
      }
    }
    return launch_status(
        q4::launch_gemm(C, c_dtype, A, B, M, N, K, s->status, s->sms, st, part, tickets));
  }
  const int sg = q4::gemm_global_split(M, N, K, s->sms);
  if (sg > 0) {
    const size_t tb = gemm_ticket_bytes(N);
    const size_t need = tb + q4::gemm_part_bytes(M, N, sg);
    if (workspace && workspace_bytes >= need) {
      tickets = static_cast<unsigned*>(workspace);
      part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + tb);
    } else if (!gemm_scratch(s, st, q4::gemm_part_bytes(M, N, sg), &part, &tickets)) {
      part = nullptr;
      tickets = nullptr;
    }
  }
  return launch_status(
      q4::launch_gemm(C, c_dtype, A, B, M, N, K, s->status, s->sms, st, part, tickets));
}
}  // namespace

extern "C" {

size_t q4_matmul_workspace_size(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  if (current_state(&s) != Q4_OK) return 0;
  if (takes_skinny(M, N, K)) {
    const int S = q4::skinny_split(N, K, s->sms);
    return S > 1 ? gemm_ticket_bytes(N) + q4::skinny_part_bytes(M, N, S) : 0;
  }
  if (!gemm_shape_ok(M, N, K)) return 0;
  if (M > 128) return q4::prefill_tail_bytes(q4::prefill_plan(M, N, K, s->sms));
  const int sg = q4::gemm_global_split(M, N, K, s->sms);
  if (sg <= 0) return 0;
  return gemm_ticket_bytes(N) + q4::gemm_part_bytes(M, N, sg);
}

int q4_matmul_ex(void* C, int c_dtype, const void* A, int a_dtype, const void* B, int b_layout,
                 int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                 void* stream) {
  if (!C || !A || !B || M <= 0 || N <= 0 || K <= 0) return Q4_ERR_ARG;
  if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30)) return Q4_ERR_SHAPE;
  if ((c_dtype != Q4_F32 && c_dtype != Q4_BF16) || (a_dtype != Q4_F32 && a_dtype != Q4_BF16))
    return Q4_ERR_DTYPE;
  if (b_layout != Q4_LAYOUT_BLOCKS && b_layout != Q4_LAYOUT_Q8_0 && b_layout != Q4_LAYOUT_PLANAR)
    return Q4_ERR_ARG;
  const int fmt = (b_layout == Q4_LAYOUT_Q8_0)    ? q4::kFmtQ8
                  : (b_layout == Q4_LAYOUT_PLANAR) ? q4::kFmtQ4P
                                                   : q4::kFmtQ4;
  if (!aligned16(C) || !aligned16(A) || !aligned16(B) || (workspace && !aligned16(workspace)))
    return Q4_ERR_ALIGN;

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int rc = current_state(&s);
  if (rc != Q4_OK) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (fmt == q4::kFmtQ4 && a_dtype == Q4_BF16 && M >= kMinSkinnyRows && K >= kMinTensorK &&
      takes_skinny(M, N, K)) {
    rc = skinny_run(s, C, c_dtype, A, B, M, N, K, workspace, workspace_bytes, st);
    if (rc != Q4_ERR_SHAPE) return rc;   // else: captured without a workspace
  }
  if (takes_gemm(fmt, a_dtype, M, N, K))
    return gemm_run(s, C, c_dtype, A, B, M, N, K, workspace, workspace_bytes, st);
  return gemv_run(s, C, c_dtype, A, a_dtype, B, fmt, M, N, K, st);
}

int q4_matmul_bf16_tiles(void* C, int c_dtype, const void* A, const void* B, int64_t M, int64_t N,
                         int64_t K, void* workspace, size_t workspace_bytes, void* stream) {
  if (!C || !A || !B || M <= 0 || N <= 0 || K <= 0) return Q4_ERR_ARG;
  if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30)) return Q4_ERR_SHAPE;
  if (c_dtype != Q4_F32 && c_dtype != Q4_BF16) return Q4_ERR_DTYPE;
  if (!aligned16(C) || !aligned16(A) || !aligned16(B) || (workspace && !aligned16(workspace)))
    return Q4_ERR_ALIGN;
  if (!takes_skinny(M, N, K) && !gemm_shape_ok(M, N, K)) return Q4_ERR_SHAPE;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int rc = current_state(&s);
  if (rc != Q4_OK) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (takes_skinny(M, N, K)) {
    rc = skinny_run(s, C, c_dtype, A, B, M, N, K, workspace, workspace_bytes, st);
    if (rc != Q4_ERR_SHAPE || !gemm_shape_ok(M, N, K)) return rc;
  }
  return gemm_run(s, C, c_dtype, A, B, M, N, K, workspace, workspace_bytes, st);
}

int q4_matmul(float* C, const float* A, const void* B, int64_t M, int64_t N, int64_t K) {
  return q4_matmul_ex(C, Q4_F32, A, Q4_F32, B, Q4_LAYOUT_BLOCKS, M, N, K, nullptr, 0, nullptr);
}

size_t q4_moe_workspace_size(int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I) {
  if (T <= 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0) return 0;
  // the counter header, then the preferred form's rows and partial sums
  return kMoeHeaderBytes + moe_data_bytes(T, topk, H, I);
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
  const MoeShape& m = cached_moe_shape(s, T, topk, E, H, I);
  void* ws = workspace;
  size_t bytes = workspace_bytes;
  if (ws) {
    if (bytes < kMoeHeaderBytes + moe_old_data_bytes(T, topk, H, I)) return Q4_ERR_WORKSPACE;
  } else {
    bytes = kMoeHeaderBytes + moe_data_bytes(T, topk, H, I);
    rc = owned_workspace(s, bytes, static_cast<cudaStream_t>(stream), &ws);
    if (rc != Q4_OK) return rc;
  }
  return moe_run(s, m, out, x, x_dtype, W_gate, W_up, W_down, topk_idx, topk_w, T, topk, E, H, I,
                 ws, static_cast<uint8_t*>(ws) + kMoeHeaderBytes, bytes - kMoeHeaderBytes,
                 nullptr, static_cast<cudaStream_t>(stream));
}

int q4_moe_experts_trace(float* out, const void* x, int x_dtype, const void* W_gate,
                         const void* W_up, const void* W_down, const int32_t* topk_idx,
                         const float* topk_w, int64_t T, int64_t topk, int64_t E, int64_t H,
                         int64_t I, void* workspace, size_t workspace_bytes, float* g, float* u,
                         float* h, float* y, void* stream) {
  if (!out || !x || !W_gate || !W_up || !W_down || !topk_idx || !topk_w || !workspace || !g ||
      !u || !h || !y)
    return Q4_ERR_ARG;
  if (T <= 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0) return Q4_ERR_ARG;
  if (topk > 16 || T * topk > 8192 || E > (1 << 20) || H > (1 << 24) || I > (1 << 24))
    return Q4_ERR_SHAPE;
  if (x_dtype != Q4_F32 && x_dtype != Q4_BF16) return Q4_ERR_DTYPE;
  if (!aligned16(out) || !aligned16(x) || !aligned16(W_gate) || !aligned16(W_up) ||
      !aligned16(W_down) || !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(workspace) ||
      !aligned16(g) || !aligned16(u) || !aligned16(h) || !aligned16(y))
    return Q4_ERR_ALIGN;

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int rc = current_state(&s);
  if (rc != Q4_OK) return rc;
  const MoeShape& m = cached_moe_shape(s, T, topk, E, H, I);
  if (workspace_bytes < kMoeHeaderBytes + moe_old_data_bytes(T, topk, H, I))
    return Q4_ERR_WORKSPACE;
  return moe_run(s, m, out, x, x_dtype, W_gate, W_up, W_down, topk_idx, topk_w, T, topk, E, H, I,
                 workspace, static_cast<uint8_t*>(workspace) + kMoeHeaderBytes,
                 workspace_bytes - kMoeHeaderBytes, nullptr, static_cast<cudaStream_t>(stream), g,
                 u, h, y);
}

int q4_moe_experts(float* out, const void* x, const void* W_gate, const void* W_up,
                   const void* W_down, const int32_t* topk_idx, const float* topk_w, int64_t T,
                   int64_t E, int64_t H, int64_t I) {
  return q4_moe_experts_ex(out, x, Q4_BF16, W_gate, W_up, W_down, topk_idx, topk_w, T, 6, E, H, I,
                           nullptr, 0, nullptr);
}

int q4_moe_gate(int32_t* topk_idx, float* topk_w, const float* logits, int64_t T, int64_t E,
                int64_t topk, void* stream) {
  if (!topk_idx || !topk_w || !logits || T <= 0 || E <= 0 || topk <= 0) return Q4_ERR_ARG;
  if (E > q4::kGateMaxExperts || topk > q4::kGateMaxTopk || topk > E || T > (1 << 24))
    return Q4_ERR_SHAPE;
  if (!aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(logits)) return Q4_ERR_ALIGN;
  return launch_status(q4::launch_moe_gate(topk_idx, topk_w, logits, static_cast<int>(T),
                                           static_cast<int>(E), static_cast<int>(topk), nullptr,
                                           nullptr, static_cast<cudaStream_t>(stream)));
}

namespace {
// Workspace of q4_moe_block: routing, the shared expert's routing, its output
// (dense path) or its own expert workspace (one-expert path, whose per-slot
// down output is the addend of the routed combine), then the routed problem's
// expert workspace.
struct BlockLayout {
  size_t idx, w, sidx, sw, ys, sg, su, sh, moe_s, moe, total;
};

// The shared expert runs as one (E = 1) routed expert at T = 1, where gate and
// up share a kernel; with more tokens it is a dense FFN over all T rows: two
// GEMVs (gate, up) whose row chunks run side by side, SiLU(g)*u, and a GEMV
// for down -- rather than one expert kernel passing over its weights once per
// few tokens.
bool shared_dense(int64_t T) { return T > 1; }
BlockLayout block_layout(int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I, int64_t Is) {
  BlockLayout b;
  size_t o = kMoeHeaderBytes;   // the routed-expert counters (both expert calls)
  b.idx = o;
  o += round_up(static_cast<size_t>(T * topk) * 4, 256);
  b.w = o;
  o += round_up(static_cast<size_t>(T * topk) * 4, 256);
  b.sidx = o;
  o += round_up(static_cast<size_t>(T) * 4, 256);
  b.sw = o;
  o += round_up(static_cast<size_t>(T) * 4, 256);
  b.ys = o;
  o += (Is > 0 && shared_dense(T)) ? round_up(static_cast<size_t>(T * H) * 4, 256) : 0;
  const size_t tis = (Is > 0 && shared_dense(T)) ? round_up(static_cast<size_t>(T * Is) * 4, 256) : 0;
  b.sg = o;
  o += tis;
  b.su = o;
  o += tis;
  b.sh = o;
  o += tis;
  b.moe_s = o;
  o += (Is > 0 && !shared_dense(T)) ? round_up(moe_data_bytes(T, 1, H, Is), 256) : 0;
  b.moe = o;
  b.total = o + moe_data_bytes(T, topk, H, I);
  return b;
}
}  // namespace

size_t q4_moe_block_workspace_size(int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I,
                                   int64_t Is) {
  if (T <= 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0 || Is < 0) return 0;
  return block_layout(T, topk, E, H, I, Is).total;
}

int q4_moe_block(float* out, const void* x, int x_dtype, const float* logits, const void* W_gate,
                 const void* W_up, const void* W_down, int64_t T, int64_t topk, int64_t E,
                 int64_t H, int64_t I, const void* S_gate, const void* S_up, const void* S_down,
                 int64_t Is, void* workspace, size_t workspace_bytes, void* stream) {
  if (!out || !x || !logits || !W_gate || !W_up || !W_down) return Q4_ERR_ARG;
  if (T <= 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0 || Is < 0) return Q4_ERR_ARG;
  if (Is > 0 && (!S_gate || !S_up || !S_down)) return Q4_ERR_ARG;
  if (E > q4::kGateMaxExperts || topk > q4::kGateMaxTopk || topk > E || T * topk > 8192 ||
      H > (1 << 24) || I > (1 << 24) || Is > (1 << 24))
    return Q4_ERR_SHAPE;
  if (x_dtype != Q4_F32 && x_dtype != Q4_BF16) return Q4_ERR_DTYPE;
  if (!aligned16(out) || !aligned16(x) || !aligned16(logits) || !aligned16(W_gate) ||
      !aligned16(W_up) || !aligned16(W_down) || (workspace && !aligned16(workspace)) ||
      (Is > 0 && (!aligned16(S_gate) || !aligned16(S_up) || !aligned16(S_down))))
    return Q4_ERR_ALIGN;

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int rc = current_state(&s);
  if (rc != Q4_OK) return rc;
  const MoeShape& m = cached_moe_shape(s, T, topk, E, H, I);
  if (!moe_seq_plan(T, topk, H, I, x_dtype).ok &&
      (4LL * m.mr * m.rows_gu > kMaxASliceBytes || 4LL * m.mr * m.rows_d > kMaxASliceBytes))
    return Q4_ERR_SHAPE;
  const MoeShape* ms = nullptr;
  if (Is > 0 && !shared_dense(T)) {
    ms = &cached_moe_shape(s, T, 1, 1, H, Is);
    if (4LL * ms->mr * ms->rows_gu > kMaxASliceBytes || 4LL * ms->mr * ms->rows_d > kMaxASliceBytes)
      return Q4_ERR_SHAPE;
  }
  if (Is > 0 && shared_dense(T)) {
    for (const auto& kn : {std::make_pair(H, Is), std::make_pair(Is, H)}) {
      const GemvShape& g = cached_gemv_shape(s, T, kn.second, kn.first, q4::kFmtQ4);
      if (g.nchunks > 65535 || 4LL * g.mr * g.rows_per_split > kMaxASliceBytes) return Q4_ERR_SHAPE;
    }
  }
  const BlockLayout b = block_layout(T, topk, E, H, I, Is);
  void* ws = workspace;
  if (ws) {
    if (workspace_bytes < b.total) return Q4_ERR_WORKSPACE;
  } else {
    rc = owned_workspace(s, b.total, static_cast<cudaStream_t>(stream), &ws);
    if (rc != Q4_OK) return rc;
  }
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  int32_t* idx = reinterpret_cast<int32_t*>(w8 + b.idx);
  float* w = reinterpret_cast<float*>(w8 + b.w);
  int32_t* sidx = reinterpret_cast<int32_t*>(w8 + b.sidx);
  float* sw = reinterpret_cast<float*>(w8 + b.sw);
  float* ys = reinterpret_cast<float*>(w8 + b.ys);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);

  // router (and the shared expert's unit routing)
  cudaError_t e = q4::launch_moe_gate(idx, w, logits, static_cast<int>(T), static_cast<int>(E),
                                      static_cast<int>(topk), Is > 0 ? sidx : nullptr,
                                      Is > 0 ? sw : nullptr, st);
  if (e != cudaSuccess) return Q4_ERR_CUDA;
  // shared expert: every token, weight 1.  On the one-expert path its down
  // output, one slot per token, is already the shared expert's result
  // ([T, H]): no combine of its own, the routed combine adds it.
  if (Is > 0 && !shared_dense(T)) {
    const size_t sbytes = moe_data_bytes(T, 1, H, Is);
    rc = moe_run(s, *ms, nullptr, x, x_dtype, S_gate, S_up, S_down, sidx, sw, T, 1, 1, H, Is,
                 w8, w8 + b.moe_s, sbytes, nullptr, st);
    if (rc != Q4_OK) return rc;
    ys = moe_y_rows(w8 + b.moe_s, *ms, moe_takes_seq(T, 1, H, Is, x_dtype, sbytes), T, 1, H, Is,
                    x_dtype);
  } else if (Is > 0) {
    float* sg = reinterpret_cast<float*>(w8 + b.sg);
    float* su = reinterpret_cast<float*>(w8 + b.su);
    float* sh = reinterpret_cast<float*>(w8 + b.sh);
    rc = gemv_run(s, sg, Q4_F32, x, x_dtype, S_gate, q4::kFmtQ4, T, Is, H, st);
    if (rc == Q4_OK) rc = gemv_run(s, su, Q4_F32, x, x_dtype, S_up, q4::kFmtQ4, T, Is, H, st);
    if (rc != Q4_OK) return rc;
    if (q4::launch_silu_mul(sh, sg, su, static_cast<size_t>(T * Is), st) != cudaSuccess)
      return Q4_ERR_CUDA;
    rc = gemv_run(s, ys, Q4_F32, sh, Q4_F32, S_down, q4::kFmtQ4, T, H, Is, st);
    if (rc != Q4_OK) return rc;
  }
  // routed experts; the shared expert's rows are added after the weighted sum
  return moe_run(s, m, out, x, x_dtype, W_gate, W_up, W_down, idx, w, T, topk, E, H, I,
                 w8, w8 + b.moe, moe_data_bytes(T, topk, H, I), Is > 0 ? ys : nullptr, st);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode sequence: many M = 1 GEMVs in one persistent launch
// ---------------------------------------------------------------------------
struct q4_gemv_seq {
  int device;
  uint8_t* buf;
  int nops, total_units, grid, stages;
  size_t counters_off, counters_bytes, part_off;
  unsigned* status;
};

namespace {
struct SeqLayout {
  size_t descs, counters, counters_bytes, part, total;
  int units, tiles;
};

// Checks the ops and lays out the plan buffer: op descriptors, the counters
// cleared before every run (unit queue, done tiles per op, tile tickets),
// then one 512-float partial row per unit.
// Rows per unit of each op: the caller's choice; else 512 for an op that a
// later op waits for (it must finish soon after its last unit is handed out);
// else the longest of 4096, 2048, 1024 and 512 rows whose units, kSeqTailRounds
// per CTA of a full grid (kSeqNominalCtas), still fit in the weights from this
// op to the end of the sequence, so that units shorten as the sweep nears its
// end and the CTAs finish together.  Each unit ends in a reduction over its
// CTA and, with more than one slice per tile, a ticket of its tile, which its
// consumers wait for: long units spread that cost (independent sweep on
// GB300: 4421 GB/s at 512 rows, 5413 at 2048, 5552 at 4096, 5698 at 4096 with
// the last 192 MB in 512-row units), while ops that others wait for run best
// with short ones (layer-ordered sweep: 1745 GB/s at 512 rows, 817 at 2048).
constexpr double kSeqTailRounds = 0.5;
constexpr int64_t kSeqNominalCtas = 304;   // 152 SMs x 2 CTAs

int64_t op_weight_bytes(const q4_gemv_op& o) { return o.K * ceil_div(o.N, 32) * 18; }

// rows[i] = rows per unit of op i (ops already checked).
void seq_plan_rows(const q4_gemv_op* ops, int n, std::vector<int64_t>* rows) {
  rows->assign(static_cast<size_t>(n), 0);
  std::vector<char> waited(static_cast<size_t>(n), 0);
  for (int j = 0; j < n; ++j)
    for (int k = 0; k < ops[j].ndeps; ++k) waited[ops[j].deps[k]] = 1;
  int64_t remaining = 0;
  for (int i = n - 1; i >= 0; --i) {
    remaining += op_weight_bytes(ops[i]);
    int64_t r = ops[i].slice_rows;
    if (r == 0 && waited[i]) r = q4::seq_default_slice_rows();
    if (r == 0) {
      r = q4::seq_max_slice_rows();
      const int64_t unit_bytes_per_row = q4::seq_tile_cols() / 32 * 18;
      while (r > q4::seq_default_slice_rows() &&
             static_cast<double>(remaining) <
                 kSeqTailRounds * kSeqNominalCtas * unit_bytes_per_row * r)
        r /= 2;
    }
    (*rows)[i] = r;
  }
}

int seq_layout(const q4_gemv_op* ops, int n, SeqLayout* L) {
  if (!ops || n <= 0 || n > (1 << 20)) return Q4_ERR_ARG;
  const int64_t tc = q4::seq_tile_cols();
  int64_t units = 0, tiles = 0;
  for (int i = 0; i < n; ++i) {
    const q4_gemv_op& o = ops[i];
    if (!o.C || !o.A || !o.B || o.N <= 0 || o.K <= 0) return Q4_ERR_ARG;
    if (o.N > (1LL << 30) || o.K > (1LL << 30)) return Q4_ERR_SHAPE;
    if ((o.a_dtype != Q4_F32 && o.a_dtype != Q4_BF16) ||
        (o.c_dtype != Q4_F32 && o.c_dtype != Q4_BF16))
      return Q4_ERR_DTYPE;
    if (o.ndeps < 0 || o.ndeps > 4) return Q4_ERR_ARG;
    for (int j = 0; j < o.ndeps; ++j)
      if (o.deps[j] < 0 || o.deps[j] >= i) return Q4_ERR_ARG;
    if (!aligned16(o.C) || !aligned16(o.A) || !aligned16(o.B)) return Q4_ERR_ALIGN;
    if (ceil_div(o.N, 32) % 8 != 0) return Q4_ERR_SHAPE;   // 16-byte row pitch for TMA
    if (o.slice_rows < 0 || o.slice_rows > q4::seq_max_slice_rows() ||
        o.slice_rows % q4::seq_slice_rows_unit() != 0)
      return Q4_ERR_ARG;
  }
  std::vector<int64_t> rows;
  seq_plan_rows(ops, n, &rows);
  for (int i = 0; i < n; ++i) {
    const q4_gemv_op& o = ops[i];
    const int64_t nt = ceil_div(o.N, tc), ns = ceil_div(o.K, rows[i]);
    units += nt * ns;
    tiles += nt;
  }
  if (units > (1LL << 30)) return Q4_ERR_SHAPE;
  L->units = static_cast<int>(units);
  L->tiles = static_cast<int>(tiles);
  L->descs = 0;
  L->counters = round_up(sizeof(q4::SeqOpDesc) * n, 256);
  L->counters_bytes = round_up(static_cast<size_t>(1 + n + tiles) * 4, 256);
  L->part = L->counters + L->counters_bytes;
  L->total = L->part + static_cast<size_t>(units) * tc * 4;
  return Q4_OK;
}
}  // namespace

extern "C" {

size_t q4_gemv_seq_bytes(const q4_gemv_op* ops, int n) {
  SeqLayout L;
  return seq_layout(ops, n, &L) == Q4_OK ? L.total : 0;
}

int q4_gemv_seq_create(const q4_gemv_op* ops, int n, void* buf, size_t buf_bytes,
                       q4_gemv_seq** plan) {
  if (!plan) return Q4_ERR_ARG;
  *plan = nullptr;
  SeqLayout L;
  int rc = seq_layout(ops, n, &L);
  if (rc != Q4_OK) return rc;
  if (!buf) return Q4_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(buf) & 255u) != 0) return Q4_ERR_ALIGN;
  if (buf_bytes < L.total) return Q4_ERR_WORKSPACE;

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  rc = current_state(&s);
  if (rc != Q4_OK) return rc;
  int stages = 3;
  int per_sm = q4::seq_ctas_per_sm(stages, false);
  if (per_sm < 2) {
    stages = 2;
    per_sm = q4::seq_ctas_per_sm(stages, false);
  }
  if (per_sm < 1) return Q4_ERR_CUDA;

  std::vector<q4::SeqOpDesc> d(static_cast<size_t>(n));
  std::memset(d.data(), 0, sizeof(q4::SeqOpDesc) * n);
  const int64_t tc = q4::seq_tile_cols();
  std::vector<int64_t> rows;
  seq_plan_rows(ops, n, &rows);
  int unit_base = 0, ticket_base = 0;
  for (int i = 0; i < n; ++i) {
    const q4_gemv_op& o = ops[i];
    q4::SeqOpDesc& e = d[i];
    const int64_t nb = ceil_div(o.N, 32);
    if (!q4::encode_weight_tmap(&e.tmap, o.B, o.K, nb, 1, o.K * nb * 18, 2, true, q4::kFmtQ4))
      return Q4_ERR_CUDA;
    e.A = o.A;
    e.C = o.C;
    e.K = static_cast<int>(o.K);
    e.N = static_cast<int>(o.N);
    e.nb = static_cast<int>(nb);
    e.ntiles = static_cast<int>(ceil_div(o.N, tc));
    const int64_t sr = rows[i];
    e.slice_rows = static_cast<int>(sr);
    e.nslices = static_cast<int>(ceil_div(o.K, sr));
    e.unit_base = unit_base;
    e.ticket_base = ticket_base;
    e.a_dtype = o.a_dtype;
    e.c_dtype = o.c_dtype;
    e.ndeps = o.ndeps;
    for (int j = 0; j < o.ndeps; ++j) e.deps[j] = o.deps[j];
    unit_base += e.ntiles * e.nslices;
    ticket_base += e.ntiles;
  }
  uint8_t* b8 = static_cast<uint8_t*>(buf);
  if (cudaMemcpy(b8 + L.descs, d.data(), sizeof(q4::SeqOpDesc) * n, cudaMemcpyHostToDevice) !=
          cudaSuccess ||
      cudaMemset(b8 + L.counters, 0, L.counters_bytes) != cudaSuccess)
    return Q4_ERR_CUDA;
  q4_gemv_seq* h = new (std::nothrow) q4_gemv_seq;
  if (!h) return Q4_ERR_ARG;
  cudaGetDevice(&h->device);
  h->buf = b8;
  h->nops = n;
  h->total_units = L.units;
  h->stages = stages;
  h->grid = per_sm * s->sms;
  h->counters_off = L.counters;
  h->counters_bytes = L.counters_bytes;
  h->part_off = L.part;
  h->status = s->status;
  *plan = h;
  return Q4_OK;
}

int q4_gemv_seq_run(const q4_gemv_seq* plan, void* stream) {
  if (!plan) return Q4_ERR_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device) return Q4_ERR_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(plan->buf + plan->counters_off, 0, plan->counters_bytes, st) != cudaSuccess)
    return Q4_ERR_CUDA;
  q4::SeqParams p;
  std::memset(&p, 0, sizeof(p));
  p.ops = reinterpret_cast<const q4::SeqOpDesc*>(plan->buf);
  p.nops = plan->nops;
  p.total_units = plan->total_units;
  unsigned* c = reinterpret_cast<unsigned*>(plan->buf + plan->counters_off);
  p.queue = c;
  p.done = c + 1;
  p.tickets = c + 1 + plan->nops;
  p.part = reinterpret_cast<float*>(plan->buf + plan->part_off);
  p.err = plan->status;
  for (int i = 0; i < 4; ++i) p.kmask[i] = 0xFu << (4 * i);
  return launch_status(q4::launch_gemv_seq(p, plan->grid, plan->stages, st));
}

void q4_gemv_seq_destroy(q4_gemv_seq* plan) { delete plan; }

int q4_gemv_seq_grid(const q4_gemv_seq* plan) { return plan ? plan->grid : 0; }

int q4_quantize(void* B, const void* W, int w_dtype, int64_t K, int64_t N, void* stream) {
  if (!B || !W || K <= 0 || N <= 0) return Q4_ERR_ARG;
  if (K > (1LL << 30) || N > (1LL << 30)) return Q4_ERR_SHAPE;
  if (w_dtype != Q4_F32 && w_dtype != Q4_BF16) return Q4_ERR_DTYPE;
  if (!aligned16(B) || !aligned16(W)) return Q4_ERR_ALIGN;
  return launch_status(q4::launch_quantize(static_cast<uint8_t*>(B), W, w_dtype, K, N,
                                           static_cast<cudaStream_t>(stream)));
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

int64_t q4_prefill_units(int64_t M, int64_t N, int64_t K, int sms, int32_t* out, int64_t cap) {
  if (M <= 128 || N <= 0 || K <= 0 || sms <= 0 || cap < 0 || (cap > 0 && !out))
    return Q4_ERR_ARG;
  if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30)) return Q4_ERR_SHAPE;
  return q4::prefill_units(M, N, K, sms, out, cap);
}

int q4_selftest_wait(int64_t limit_ns, int arrive, void* stream) {
  if (limit_ns <= 0 || limit_ns > 1000000000LL || (arrive != 0 && arrive != 1)) return Q4_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int rc = current_state(&s);
  if (rc != Q4_OK) return rc;
  return launch_status(q4::launch_wait_selftest(s->status,
                                                static_cast<unsigned long long>(limit_ns),
                                                arrive != 0, static_cast<cudaStream_t>(stream)));
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
  g_last_flags = flags;
  return flags ? Q4_ERR_DEVICE : Q4_OK;
}

unsigned int q4_last_device_flags(void) { return g_last_flags; }

int q4_release_scratch(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int rc = current_state(&s);
  if (rc != Q4_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return Q4_ERR_CUDA;
  for (auto& kv : s->gemm_scratch) {
    cudaFree(kv.second.part);
    cudaFree(kv.second.tickets);
  }
  s->gemm_scratch.clear();
  for (void* p : s->retired) cudaFree(p);
  s->retired.clear();
  cudaFree(s->ws);
  s->ws = nullptr;
  s->ws_bytes = 0;
  return Q4_OK;
}

}  // extern "C"
