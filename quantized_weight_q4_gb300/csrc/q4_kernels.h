// Internal interface between the C-ABI layer and the kernel translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace q4 {

enum : int { kModeGemv = 0, kModeGateUp = 1, kModeDown = 2 };
// Weight formats of the GEMV kernel (values of the public Q4_LAYOUT_* codes
// are not used here: the host maps Q4_LAYOUT_BLOCKS -> kFmtQ4,
// Q4_LAYOUT_Q8_0 -> kFmtQ8 and Q4_LAYOUT_PLANAR -> kFmtQ4P, the Q4_0 blocks
// split into a scale plane and a nibble plane; plain GEMV mode only).
enum : int { kFmtQ4 = 0, kFmtQ8 = 1, kFmtQ4P = 2 };

// Arguments of q4_gemv_kernel (one struct, passed by value as a __grid_constant__
// parameter so that the tensor maps inside it are addressable by TMA).
struct GemvParams {
  // TMA tensor maps of the weights (B and B2) as 3-D uint16 tensors
  // [experts][K rows][nb*9 halfwords]; valid when use_tma != 0.  Planar
  // Q4_0 (kFmtQ4P): tmap[0] maps the nibble plane, tmap[1] the scale plane.
  // GEMV mode only.
  CUtensorMap tmap[2];
  int use_tma;
  int mode;
  // weights: one matrix (GEMV) or expert stacks (B = gate or down, B2 = up)
  const uint8_t* B;
  const uint8_t* B2;
  long long b_stride;   // bytes per expert matrix
  long long qs_offset;  // kFmtQ4P: byte offset of the nibble plane from B
  int K, N, nb;
  // split-K tiling (grid.x = column tiles of 8*BPT blocks, grid.y = splits;
  // the splits of a tile form one thread-block cluster)
  int nsplit, rows_per_split;
  uint32_t kmask[4];    // nibble masks (fill_decode_consts)
  // activations
  const void* A;
  int a_dtype;          // 0 fp32, 1 bf16
  long long a_ld;       // elements per row of A
  int M;                // GEMV rows
  // outputs
  void* C;
  int c_dtype;
  // routed experts
  const int32_t* topk_idx;
  int nslots, topk, E;
  int list_cap;         // shared-memory list entries (>= nslots, >= ceil(E/32))
  float* h;             // [nslots, I] SiLU(g) * u
  float* y;             // [nslots, H] down outputs
  float* g_trace;       // gate/up: if not null, g and u [nslots, I] are also
  float* u_trace;       //   written there (q4_moe_experts_trace)
  unsigned* err;        // device status word
};

// mr: rows of A per pass (1, 2 or 4); bpt: blocks per thread (1 or 2; 2 only with mr 1);
// big: 18 KB pipeline stages instead of 32-row ones (rows_per_split a multiple of
// gemv_stage_rows(bpt, big) either way).
// cluster: (1, nsplit, 1), or (1, nsplit, 2) for the gate/up kernel.
// fmt: kFmtQ4 (block_q4_0), kFmtQ8 (Q8_0: plain GEMV mode and big = false only)
// or kFmtQ4P (planar Q4_0: plain GEMV mode only).
cudaError_t launch_gemv(const GemvParams& p, int mr, int bpt, bool big, int fmt, dim3 grid,
                        dim3 cluster, cudaStream_t st, bool pdl);
constexpr int kMaxCluster = 16;   // non-portable thread-block cluster size limit
// Clusters of shape `cluster` that can be resident at once for that kernel
// configuration (0 if the configuration cannot launch).
int max_active_clusters(int mode, int mr, int bpt, bool big, int fmt, int rows_per_split,
                        int list_cap, dim3 cluster);
// Rows of one TMA box (one pipeline stage) of the GEMV kernel.
int gemv_stage_rows(int bpt, bool big);
// Blocks per column tile for `bpt` blocks per thread.
int gemv_tile_blocks(int bpt);
void fill_decode_consts(GemvParams& p, int fmt);
// Encodes the tensor map of `experts` stacked K x nb-block Q4_0 matrices,
// `matrix_bytes` apart, with boxes of one tile row segment (8*bpt blocks) by one
// stage of rows.  Needs nb % 8 == 0 and a 16-byte aligned base.
bool encode_weight_tmap(CUtensorMap* map, const void* base, int64_t K, int64_t nb,
                        int64_t experts, int64_t matrix_bytes, int bpt, bool big, int fmt);
// Planar Q4_0 (Q4_LAYOUT_PLANAR, one K x nb matrix at `base`): maps[0] = the
// nibble plane at base + qs_offset as uint32 [K][nb*4], maps[1] = the scale
// plane at base as uint16 [K][nb]; boxes of one tile row segment (8*bpt
// blocks) by one stage of rows.  Needs nb % 8 == 0, a 16-byte aligned base and
// qs_offset a multiple of 16.
bool encode_planar_tmaps(CUtensorMap* maps, const void* base, int64_t K, int64_t nb,
                         int64_t qs_offset, int bpt, bool big);
// h[i] = SiLU(g[i]) * u[i] for i < n, fp32 (programmatic dependent launch).
cudaError_t launch_silu_mul(float* h, const float* g, const float* u, size_t n, cudaStream_t st);
// out[t] = sum_k w[t,k] * y[t*topk+k] (slot order), plus addend[t] if given.
cudaError_t launch_moe_combine(float* out, const float* y, const int32_t* idx, const float* w,
                               const float* addend, int T, int topk, int E, int H,
                               cudaStream_t st, bool pdl);

// q4_gemv_seq.cu: a sequence of M = 1 GEMVs in one persistent launch.
// One op of the sequence, as the kernel reads it from global memory (a plan)
// or from its parameters (inline ops).
//
// An op may be segmented over the slots of routed tokens (segmented along
// its output columns): segment s holds the product A_s . W[eidx[s]] in
// C[s] (seg_len columns, seg_tiles column tiles), the expert eidx[s] picking
// the matrix of a tensor map over E experts, and A_s = A + (s / a_seg_div) *
// a_seg_stride.  With `pair`, segments 2s and 2s + 1 are slot s's products
// with the matrices of tmap (into C[s]) and tmap2 (into C2[s]); one ticket
// serves both tiles of a column, and the last of their K slices adds both
// products, stores them and h[s] = SiLU(C[s]) * C2[s] on those columns, and
// counts the column tile in seg_done[seg_done_base + s].  With seg_need > 0,
// segment s reads A only once op seg_dep's seg_done[.. + s] has reached
// seg_need (a zeroed descriptor has no such dependency).  Segments whose index lies outside [0, E) read no weights and
// write nothing.
struct SeqOpDesc {      // 64-byte aligned through its tensor maps
  CUtensorMap tmap;     // weights: uint16 [E][K][nb*9], boxes of 144 x 64
  CUtensorMap tmap2;    // pair: the second matrices
  const void* A;        // [K] (or per segment, see a_seg_div), fp32 (a_dtype 0) or bf16 (1)
  void* C;              // [N], fp32 (c_dtype 0) or bf16 (1)
  void* C2;             // pair: the second products, fp32 [nseg / 2][seg_len]
  float* h;             // pair: SiLU(C) * C2, fp32 [nseg / 2][seg_len]
  const int32_t* eidx;  // expert of each slot, or null (matrix 0)
  int K, N, nb;         // the op's K and N (segmented: N = nseg x seg_len)
  int ntiles, nslices;  // column tiles of 512 columns, K slices of slice_rows rows
  int slice_rows;       // a multiple of 64, at most 4096
  int unit_base;        // first unit of the op (units: tile-major, slice-minor)
  int ticket_base;      // first tile counter of the op
  int a_dtype, c_dtype;
  int seg_mode;         // 0: none; 1: segmented along N
  int nseg, seg_len;    // segments, and columns of each
  int seg_tiles;        // column tiles per segment
  int a_seg_div;        // segments per row of A (0: one A for all segments)
  int a_seg_stride;     // elements between rows of A
  int pair;             // segments form (tmap, tmap2) pairs of one slot
  int seg_done_base;    // pair: first per-slot counter in seg_done
  int seg_dep, seg_need;// per-segment dependency on op seg_dep (seg_need 0: none)
  int E;                // experts of the tensor maps (valid eidx values: [0, E))
  int ndeps;
  int deps[4];          // earlier ops whose outputs must be complete before A is read
};
constexpr int kSeqInlineOps = 2;
struct SeqParams {
  const SeqOpDesc* ops; // the ops in global memory, or null: the inline ops below
  int nops, total_units;
  unsigned* queue;      // unit counter (zero at launch)
  unsigned* done;       // [nops] completed tiles per op (zero at launch)
  unsigned* tickets;    // [ntickets] slices added per tile (pairs: per tile pair) (zero at launch)
  unsigned* seg_done;   // [nseg_done] completed column tiles per slot of pair ops (zero at launch)
  unsigned* exits;      // reset != 0: CTAs finished (zero at launch)
  int ntickets, nseg_done;
  int reset;            // nonzero: the last CTA to finish zeroes the counters
  float* part;          // [total_units][512] partial sums
  unsigned* err;        // device status word
  uint32_t kmask[4];    // nibble masks (fill as for the GEMV)
  SeqOpDesc inl[kSeqInlineOps];
};
// q4_capi.cu: the least workspace a routed-expert call of this shape takes
// (the counter header and the three-launch form's rows); calls with more may
// run the persistent form.
size_t moe_min_workspace_bytes(int64_t T, int64_t topk, int64_t H, int64_t I);
// CTAs per SM that the persistent kernel with `stages` ring slots (4 or 5)
// can keep resident (0 if it cannot launch).
int seq_ctas_per_sm(int stages, bool seg);   // seg: the segmented instance
int seq_tile_cols();       // columns of a unit (512)
int seq_stage_rows();      // rows of one pipeline stage (128: two 64-row TMA boxes)
int seq_slice_rows_unit(); // units are multiples of this many rows (64; a last stage may be half)
int seq_max_slice_rows();      // rows of the longest unit (4096)
int seq_default_slice_rows();  // rows of a unit by default (512)
// `pdl`: launched with programmatic stream serialization (the kernel waits
// for the previous grid before touching memory).
// seg: the instance for segmented or inline ops and counter resets; without
// it, the ops must be plain GEMVs in global memory and `reset` zero.
cudaError_t launch_gemv_seq(const SeqParams& p, int grid, int stages, cudaStream_t st,
                            bool pdl = false, bool seg = false);

// q4_gemm_sm103.cu: the prefill GEMM on the tensor cores.
struct GemmParams {
  CUtensorMap tmap_a;   // A: bf16 [M][K], boxes of 64 K x 256 rows, 128-byte swizzle
  CUtensorMap tmap_b;   // weights: uint16 [K][nb*9], boxes of 72 halfwords x 64 rows
  CUtensorMap tmap_c;   // prefill form, use_tma_c: C [M][N], boxes of 128 bytes x 32 rows,
                        // 128-byte swizzle (written with TMA stores)
  int use_tma_c;
  void* C;              // [M][N] fp32 (c_dtype 0) or bf16 (1)
  int c_dtype;
  int M, N, K;
  int nsplit;           // small-M form: K splits per tile (the cluster size)
  int a_rows;           // rows of one A box (tile rows, or M rounded up to 16)
  unsigned* err;        // device status word
  // small-M form through global memory (gsplit != 0): the K splits of a tile
  // are independent CTAs (no cluster); each writes its fp32 partial tile to
  // part [tile][split][rows][256] and takes a ticket from tickets[tile]; the
  // CTA with the last ticket adds the partials in split order, stores C and
  // returns the ticket to zero
  int gsplit;
  float* part;
  unsigned* tickets;
  // prefill form: tiles [0, full_tiles) run whole, round-robin over the grid;
  // with tail_ctas > 0 the K steps of the remaining tiles, taken in tile
  // order as one range, are cut into tail_ctas equal parts, CTA c taking
  // part c.  The part of a tile that holds its last K step adds the earlier
  // parts' fp32 partial tiles (part [tail_ctas][128][MT*256], each written
  // by the CTA whose part it is, ready once tickets[c] is nonzero) in K
  // order to its own sums and stores C; it returns those tickets to zero.
  int full_tiles, tail_ctas;
};
// Shapes the tensor-core GEMM accepts: nb = ceil(N/32) a multiple of 8 (whole
// 256-column tiles of blocks, 16-byte row pitch) and K a multiple of 8
// (16-byte row pitch of A).
bool gemm_supported(int64_t M, int64_t N, int64_t K);
// A: bf16, 16-byte aligned; B: blocks layout, 16-byte aligned.  M > 128 runs
// the persistent prefill form (`sms` bounds its grid; with `part` and
// `tickets` laid out as prefill_plan() asks, its last round shares K), M <=
// 128 the split-K small-M form.
// M <= 128 with `part` and `tickets` given and gemm_global_split() > 0 runs
// the small-M form through global memory (part: gemm_part_bytes() bytes;
// tickets: at least ceil(N/256) counters, zero, left zero by every launch;
// both owned by one stream at a time).
cudaError_t launch_gemm(void* C, int c_dtype, const void* A, const void* B, int64_t M, int64_t N,
                        int64_t K, unsigned* err, int sms, cudaStream_t st, float* part = nullptr,
                        unsigned* tickets = nullptr);
// K splits the small-M form uses for this shape (0: the form cannot take it).
int gemm_small_split(int64_t M, int64_t N, int64_t K);
// The prefill form (M > 128) on `sms` SMs: its grid, the tiles run whole and
// the CTAs sharing the K steps of the last round's tiles (0: no tail, every
// tile whole).  The tail needs prefill_tail_bytes() of caller memory: the
// tickets (prefill_tail_ticket_bytes(), zero, left zero by every launch) and
// then the partial tiles; launch_gemm takes them as `tickets` and `part`.
struct PrefillPlan {
  int grid, full_tiles, tail_ctas;
};
PrefillPlan prefill_plan(int64_t M, int64_t N, int64_t K, int sms);
size_t prefill_tail_ticket_bytes(const PrefillPlan& pl);
size_t prefill_tail_bytes(const PrefillPlan& pl);
// The units the prefill form's CTAs run for this shape on `sms` SMs, in
// each CTA's order: rows of 9 ints (CTA, unit, m0, n0, first and end K
// step, role, first helper CTA, helper count) into out[cap][9]; returns the
// number of units (host only, no CUDA call).
int64_t prefill_units(int64_t M, int64_t N, int64_t K, int sms, int32_t* out, int64_t cap);
// Tile counters a stream's ticket array holds (N up to 1,048,576 columns).
constexpr int kMaxGemmTickets = 4096;
// K splits of the global-memory small-M form (0: the cluster form is chosen:
// the global form runs for M <= 40, where it fits more CTAs in one wave).
int gemm_global_split(int64_t M, int64_t N, int64_t K, int sms);
// Bytes of partial tiles the global-memory form needs for that split.
size_t gemm_part_bytes(int64_t M, int64_t N, int S);

// q4_gemm_skinny.cu: the few-row GEMM (1 <= M <= 32, bf16 A) with the weights
// as the MMA's A operand and the tokens as its N.
struct SkinnyParams {
  CUtensorMap tmap_a;   // activations: bf16 [M][K], boxes of 64 K x NT rows, 128-byte swizzle
  CUtensorMap tmap_w;   // weights: uint16 [K][nb*9], boxes of 72 halfwords x 128 rows
  void* C;              // [M][N] fp32 (c_dtype 0) or bf16 (1)
  int c_dtype;
  int M, N, K;
  int nsplit;           // K slices per 256-column tile (CTAs per tile)
  float* part;          // nsplit > 1: [tiles][nsplit][M][256] partial sums
  unsigned* tickets;    // nsplit > 1: [tiles] counters, zero at launch, left zero
  unsigned* err;        // device status word
};
constexpr int kMaxSkinnyTickets = 4096;
bool skinny_supported(int64_t M, int64_t N, int64_t K);
// K slices per column tile: one CTA per SM over all tiles and slices.
int skinny_split(int64_t N, int64_t K, int sms);
size_t skinny_part_bytes(int64_t M, int64_t N, int S);
cudaError_t launch_skinny(void* C, int c_dtype, const void* A, const void* B, int64_t M, int64_t N,
                          int64_t K, unsigned* err, int S, float* part, unsigned* tickets,
                          cudaStream_t st);

// q4_misc.cu
cudaError_t launch_dequant(void* W, int w_dtype, const uint8_t* B, int64_t K, int64_t N,
                           cudaStream_t st);
cudaError_t launch_repack(uint8_t* dst, const uint8_t* src, int64_t K, int64_t N, bool to_planar,
                          cudaStream_t st);
// q4_misc.cu: the Q4_0 encoder (w_dtype 0 fp32, 1 bf16).
cudaError_t launch_quantize(uint8_t* B, const void* W, int w_dtype, int64_t K, int64_t N,
                            cudaStream_t st);

// q4_moe_gate.cu: the router (one warp per token).  Optionally also writes the
// shared expert's routing (index 0, weight 1) for every token.
constexpr int kGateMaxExperts = 1024;
constexpr int kGateMaxTopk = 16;
cudaError_t launch_moe_gate(int32_t* topk_idx, float* topk_w, const float* logits, int T, int E,
                            int topk, int32_t* shared_idx, float* shared_w, cudaStream_t st);

// One bounded pipeline wait run to its limit (arrive = false) or completed.
cudaError_t launch_wait_selftest(unsigned* err, unsigned long long limit_ns, bool arrive,
                                 cudaStream_t st);

}  // namespace q4
