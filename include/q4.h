/*
 * q4.h -- C ABI of the GB300 (sm_103a) Q4_0 weight-only dequant-matmul library.
 *
 * The operation (C++ DeepSeek engine page, "用两千行 C++ 重写一个 DeepSeek 推理引擎",
 * §2.2 block_q4_0 / dequantize, §2.3 layout and padding, §3.4 matmul_q4_0):
 *
 *   B holds a K x N weight matrix W as K rows of nb = ceil(N/32) blocks
 *   block_q4_0 { uint16 d (IEEE fp16, little-endian); uint8 qs[16]; }  (18 bytes).
 *   Block (k, b) sits at byte offset (k*nb + b)*18 and covers columns 32b..32b+31
 *   of row k.  Element l of a block is the low nibble of qs[l/2] for even l and
 *   the high nibble for odd l; its value is W[k, 32b + l] = (q - 8) * d.
 *   Columns >= N in the last block of a row are padding: they are never read
 *   into any output.
 *
 *   C[i, j] = sum_k A[i, k] * W[k, j]   (A: M x K row-major, C: M x N row-major)
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers (cudaMalloc / torch CUDA tensors)
 *     on the current CUDA device.  The caller owns every buffer; the library
 *     never frees caller memory.
 *   - Calls are asynchronous on the given stream (NULL = legacy default
 *     stream); none synchronises the host.  Outputs are overwritten.
 *   - B, A, C, x, out and workspace must be 16-byte aligned, else Q4_ERR_ALIGN.
 *   - Integer sizes must be > 0 (K, N, M, T, E, H, I), else Q4_ERR_ARG.
 *   - Return value: Q4_OK (0) or a negative Q4_ERR_* code; no call traps or
 *     aborts.  Errors found on the device (a routing index outside [0, E) or
 *     a wait that timed out) are recorded in a per-device status word that
 *     q4_get_device_status() reads.
 *   - There is no CPU fallback: every call runs on the GPU or returns an error.
 */
#ifndef Q4_GB300_H
#define Q4_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define Q4_API __attribute__((visibility("default")))
#else
#define Q4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define Q4_OK              0
#define Q4_ERR_ARG        (-1)   /* null pointer, size <= 0, bad enum value      */
#define Q4_ERR_DTYPE      (-2)   /* unsupported dtype combination                */
#define Q4_ERR_ALIGN      (-3)   /* a pointer is not 16-byte aligned             */
#define Q4_ERR_CUDA       (-4)   /* a CUDA runtime call or launch failed         */
#define Q4_ERR_WORKSPACE  (-5)   /* workspace smaller than the *_workspace_size  */
#define Q4_ERR_SHAPE      (-6)   /* shape outside what this entry point supports */
#define Q4_ERR_DEVICE     (-7)   /* q4_get_device_status: device-side error seen */

/* device status bits (q4_get_device_status() returns Q4_ERR_DEVICE and
 * q4_last_device_flags() the bits) */
#define Q4_DEVERR_INDEX    0x1u  /* a topk_idx entry outside [0, E) was skipped  */
#define Q4_DEVERR_TIMEOUT  0x2u  /* a bounded wait gave up; outputs are invalid  */

/* ---- element types ---- */
#define Q4_F32   0   /* IEEE fp32                        */
#define Q4_BF16  1   /* bfloat16, passed as raw uint16   */

/* ---- weight layouts ---- */
#define Q4_LAYOUT_BLOCKS 0   /* the 18-byte block_q4_0 array described above */
#define Q4_LAYOUT_PLANAR 1   /* q4_repack output: scales plane then nibble plane */
#define Q4_LAYOUT_Q8_0   2   /* Q8_0 blocks {fp16 d; int8 q[32]} (34 bytes), laid out
                                as the Q4_0 blocks above: w = q * d (see q4_matmul_ex) */

/*
 * q4_matmul -- C = A . W, fp32 A [M, K], fp32 C [M, N], B in Q4_LAYOUT_BLOCKS,
 * on the legacy default stream.
 * [engine page §3.4: matmul_q4_0(A, B, C, M, N, K), C overwritten as in §3.2]
 * Allocates nothing: fp32 activations take the split-K GEMV, whose partial
 * sums are combined on chip.
 */
Q4_API int q4_matmul(float *C, const float *A, const void *B, int64_t M, int64_t N, int64_t K);

/*
 * q4_matmul_ex -- C = A . W with explicit types, layout, workspace and stream.
 *   C          [M, N] row-major, c_dtype Q4_F32 or Q4_BF16 (bf16 = RN of fp32)
 *   A          [M, K] row-major, a_dtype Q4_F32 or Q4_BF16
 *   B          weights in b_layout: Q4_LAYOUT_BLOCKS; or Q4_LAYOUT_Q8_0, the
 *              second format (the engine page, §2.1-§2.2, names Q8_0 but
 *              prints no layout; reading: blocks {fp16 d; int8 q[32]} of 34
 *              bytes, 32 output columns of one row each, K rows of
 *              ceil(N/32) blocks, w = q * d); or Q4_LAYOUT_PLANAR
 *              (q4_repack's output for this K x N).  Both run the split-K
 *              GEMV below for every M (more than 4 rows in chunks of up to
 *              4, each chunk streaming the weights again); planar weights
 *              give C bit-identical to the Q4_LAYOUT_BLOCKS GEMV result for
 *              the same shape
 *   workspace  may be NULL.  Shapes whose tensor-core GEMM splits K over
 *              independent CTAs (bf16 A, 8 <= M <= 40; and M > 128 when the
 *              256 x 256 tiles leave a last round that does not fill the
 *              SMs: its tiles' K steps are then shared by up to four CTAs
 *              per tile) add the splits' partial tiles through scratch:
 *              q4_matmul_workspace_size(M, N, K) bytes of it (0 for every
 *              other shape; about 38 MB for M = 2048, K = 5120, N = 12288
 *              on 152 SMs).  A workspace of at
 *              least that size is used for it; its bytes must be zero before
 *              the first call that uses them and every completed call leaves
 *              them zero (zero it again after a Q4_ERR_DEVICE status).  With
 *              no such workspace an eager call uses scratch the library owns
 *              per stream (cudaMalloc'd by the first such call on the stream,
 *              replaced by a larger one when a later call needs more, after
 *              that stream has drained), and a call made while the stream is
 *              captured into a CUDA graph combines the splits on chip
 *              (M > 128: runs every tile over all of K) instead, so that no
 *              graph holds library-owned scratch.
 *              Calls that share one workspace must not overlap on the GPU;
 *              that includes replays of graphs captured with it.
 *   stream     cudaStream_t (NULL = legacy default stream)
 * Kernel choice:
 *   - fp32 A, M < 4, K < 1024, Q8_0 or planar weights, or a shape the GEMMs
 *     below do not take: the split-K GEMV on the CUDA cores, in chunks of
 *     up to 4 rows of A.  The splits of each column tile run as one
 *     thread-block cluster and are added on chip in fixed order.  Exact fp32
 *     dequantisation: |C - A.W| <= 1e-3 * sum|a*w| + 1e-6 for any input.
 *   - bf16 A with 4 <= M, K >= 1024, ceil(N/32) % 8 == 0 and K % 8 == 0:
 *     the tensor-core GEMM (prompt batching, engine page §5.2), as
 *     q4_matmul_bf16_tiles below: up to 32 rows the few-row form (the
 *     weights as the MMA's 128-row operand, the tokens as its N), which needs
 *     the workspace described above when captured into a graph (without one
 *     a captured call takes the split-K GEMV below 8 rows, the cluster form
 *     from 8), above 32 rows the split-K and persistent forms.
 *     Its result A . bf16_rn(W) deviates from A . W by at most 2^-8 *
 *     sum|a*w| plus the fp32 accumulation error; the rounding errors of the
 *     weights have random signs, and from K = 1024 on their sum stays within
 *     1e-3 * sum|a*w| + 1e-6 on random data.  An input built so that every
 *     weight's rounding has the sign of its activation can reach 2^-8 *
 *     sum|a*w|: callers that need the stated bound for any input pass fp32
 *     activations.
 *   Both are deterministic (no floating-point atomics, fixed orders).
 * Launches use programmatic dependent launch: a kernel may start streaming
 * its weights while the previous kernel on the stream finishes, and reads A
 * only after that kernel has completed.  Consequently B must not be written
 * by the kernel launched immediately before on the same stream (weights are
 * expected to be static; order such a write with an event or a
 * synchronisation).
 */
Q4_API int q4_matmul_ex(void *C, int c_dtype, const void *A, int a_dtype,
                 const void *B, int b_layout, int64_t M, int64_t N, int64_t K,
                 void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace q4_matmul_ex and q4_matmul_bf16_tiles use for this shape
 * (the partial tiles of the small-M tensor-core form and of the prefill
 * form's shared last round, bf16 A; 0 for shapes that need none).  0 also
 * when no CUDA device can be queried. */
Q4_API size_t q4_matmul_workspace_size(int64_t M, int64_t N, int64_t K);

/*
 * q4_matmul_bf16_tiles -- C = A . bf16_rn(W) on the tensor cores (tcgen05),
 * for any K [engine page §5.2: a prompt's tokens batched into one matmul].
 * Every weight is dequantised once to the bf16 tile element
 * bf16_rn((q - 8) * d) (q4_dequant_bf16 gives the same values) and the bf16 x
 * bf16 products are accumulated in fp32 in tensor memory.  A is bf16 [M, K];
 * C fp32 or bf16 (RN of the fp32 result) [M, N]; B in Q4_LAYOUT_BLOCKS.
 * Shapes: ceil(N/32) % 8 == 0, K % 8 == 0 (16-byte row pitches), else
 * Q4_ERR_SHAPE.  M <= 32 runs the few-row form: CTAs of 256 output columns
 * and a K slice, the dequantised weights as the MMA's A operand (M = 128)
 * and the tokens as N = 16, 32 or 64, the slices added through the
 * workspace described under q4_matmul_ex; a call captured without that
 * workspace returns Q4_ERR_SHAPE below 8 rows and takes the split form from
 * 8.  32 < M <= 128 splits K over 2..16 CTAs per 128 x 256 tile, combined in
 * fixed order over a cluster or, up to 40 rows, through the workspace;
 * M > 128 runs the persistent prefill form (256 x 256 output tiles, one
 * CTA per SM taking tiles round-robin; the tiles of an incomplete last round
 * share their K steps over the grid through the workspace, the part holding
 * a tile's last K step adding the earlier parts' partial tiles in K order to
 * its own sums).
 * Deterministic: the parts and their order depend only on the shape and the
 * SM count.
 */
Q4_API int q4_matmul_bf16_tiles(void *C, int c_dtype, const void *A, const void *B,
                                int64_t M, int64_t N, int64_t K, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * q4_release_scratch -- waits for the current device to finish all work,
 * then frees every buffer the library owns on it: the per-stream scratch of
 * the small-M GEMM and the library-owned workspace of the routed-expert calls
 * (with the ones larger calls replaced, kept until now because CUDA graphs
 * captured earlier may use them).  A graph captured with a NULL workspace
 * must not be replayed after this call.  Returns Q4_OK or Q4_ERR_CUDA.
 */
Q4_API int q4_release_scratch(void);

/*
 * q4_moe_experts -- DeepSeek-V2-style routed experts on the legacy default
 * stream with the library-owned workspace and top-k = 6
 * [KTransformers DeepSeek-V2 page, «优化三»: 160 experts, 6 active per token,
 *  run as batched GEMVs; «规则二»: gate -> top-k indices and weights].
 *   out       fp32 [T, H]
 *   x         bf16 [T, H] (raw uint16)
 *   W_gate    [E] experts x (H rows x ceil(I/32) blocks), Q4_LAYOUT_BLOCKS
 *   W_up      same shape as W_gate
 *   W_down    [E] experts x (I rows x ceil(H/32) blocks)
 *   topk_idx  int32 [T, 6]; entries outside [0, E) are skipped and flagged
 *   topk_w    fp32 [T, 6]
 * out[t] = sum_{k=0..5} topk_w[t,k] * ( SiLU(x_t.Wg[e]) * (x_t.Wu[e]) ) . Wd[e],
 * e = topk_idx[t,k], SiLU(g) = g * sigmoid(g), summed in slot order k.
 */
Q4_API int q4_moe_experts(float *out, const void *x, const void *W_gate, const void *W_up,
                   const void *W_down, const int32_t *topk_idx, const float *topk_w,
                   int64_t T, int64_t E, int64_t H, int64_t I);

/* q4_moe_experts with x_dtype (Q4_F32 / Q4_BF16), any topk in [1, 16],
 * an explicit workspace and a stream.
 * From 4 tokens up (and at most 512 slots T * topk, with ceil(I/32) and
 * ceil(H/32) multiples of 8, H * sizeof(x) and I * 4 multiples of 16 bytes)
 * the slots run in one launch of the persistent decode kernel: every slot's
 * gate and up (the last K slice of a column tile forms SiLU(g) * u there),
 * then every slot's down, each slot waiting only for its own SiLU(g) * u,
 * then the slot combine.  Fewer tokens, other shapes, or a workspace below
 * q4_moe_workspace_size run three launches (gate/up, down, slot combine).
 * The results satisfy the same bound either way.
 * The workspace (>= q4_moe_workspace_size bytes for the persistent form; the
 * three-launch form needs less) begins with 64 KB of counters that must be
 * zero before its first use (e.g. cudaMemset once); every call leaves them
 * zero unless one of its waits times out (Q4_DEVERR_TIMEOUT), after which
 * they must be cleared again.  The rest holds the intermediate rows and
 * partial sums and needs no initialisation.  NULL selects a library-owned
 * workspace (zeroed when allocated), allocated (cudaMalloc) by the first call
 * that needs more than it has.  No allocation happens while the stream is being captured: such a
 * call returns Q4_ERR_WORKSPACE, so make one call of the largest shape before
 * capturing a CUDA graph.  A workspace that a larger one replaces stays
 * allocated until q4_release_scratch(), since graphs may still use it.
 * Calls sharing a workspace must not overlap in time (the library-owned one
 * is shared by every stream of the device). */
Q4_API int q4_moe_experts_ex(float *out, const void *x, int x_dtype, const void *W_gate,
                      const void *W_up, const void *W_down, const int32_t *topk_idx,
                      const float *topk_w, int64_t T, int64_t topk, int64_t E,
                      int64_t H, int64_t I, void *workspace, size_t workspace_bytes,
                      void *stream);

Q4_API size_t q4_moe_workspace_size(int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I);

/*
 * q4_moe_experts_trace -- q4_moe_experts_ex (same kernels, same results) that
 * also returns the chain's intermediate values, so that each stage can be
 * checked on its own [KTransformers page, «优化三»: gate and up, SiLU(g) * u,
 * down, the weighted sum of the slots; C++ DeepSeek engine page §8.2:
 * checking a forward pass stage by stage on fixed inputs].
 * Row s = t * topk + k of each array belongs to slot k of token t:
 *   g, u  fp32 [T * topk, I]   the gate and up matmul outputs
 *   h     fp32 [T * topk, I]   SiLU(g) * u, the down projection's input
 *   y     fp32 [T * topk, H]   the down outputs, before the routing weights
 * Rows of slots whose index lies outside [0, E) are not written.  The
 * workspace is required (>= q4_moe_workspace_size bytes).  All pointers are
 * device pointers, 16-byte aligned.
 */
Q4_API int q4_moe_experts_trace(float *out, const void *x, int x_dtype, const void *W_gate,
                                const void *W_up, const void *W_down,
                                const int32_t *topk_idx, const float *topk_w, int64_t T,
                                int64_t topk, int64_t E, int64_t H, int64_t I,
                                void *workspace, size_t workspace_bytes, float *g, float *u,
                                float *h, float *y, void *stream);

/*
 * q4_moe_experts_noalloc -- q4_moe_experts_ex without a workspace argument,
 * for callers that cannot allocate device memory: code running while a CUDA
 * graph is captured in global mode, loops that must not allocate once
 * started, or hosts whose own allocator owns all device memory.  (This entry
 * point has no counterpart on the pages: it only changes where the scratch
 * lives.)
 *   The scratch is a fixed device array built into the library, of
 *   q4_moe_static_scratch_bytes() bytes (8 MiB) on every GPU that loads the
 *   library, held until the process exits.  Calls whose
 *   three-launch form's workspace (see q4_moe_experts_ex) exceeds it return
 *   Q4_ERR_WORKSPACE; a call runs the persistent form only when that form's
 *   workspace fits too.  No call allocates or frees device memory.
 *   The first call on a device looks up the array's device address; make it
 *   before capturing a stream into a CUDA graph.
 *   All calls on a device share the one array and leave their intermediate
 *   rows in it.  The array starts zeroed, so its counter header (see
 *   q4_moe_experts_ex) is zero before the first call; after a call whose
 *   wait timed out (Q4_DEVERR_TIMEOUT) it is not restored and later calls on
 *   the persistent form time out too.  Calls that overlap on the
 *   GPU (different streams without ordering) race on the array.
 */
Q4_API int q4_moe_experts_noalloc(float *out, const void *x, int x_dtype, const void *W_gate,
                                  const void *W_up, const void *W_down,
                                  const int32_t *topk_idx, const float *topk_w, int64_t T,
                                  int64_t topk, int64_t E, int64_t H, int64_t I, void *stream);
Q4_API size_t q4_moe_static_scratch_bytes(void);

/*
 * q4_repack / q4_unpack -- lossless change of layout, bit-exact both ways.
 * Q4_LAYOUT_PLANAR for K x N: the fp16 scales d[K][nb] (little-endian), then,
 * from byte offset q4_planar_qs_offset(K, N) (a multiple of 16), the nibble
 * bytes qs[K][nb][16]; q4_planar_bytes(K, N) bytes in all.
 * dst and src must not overlap.
 */
Q4_API int q4_repack(void *dst, const void *src, int64_t K, int64_t N, void *stream);
Q4_API int q4_unpack(void *dst, const void *src, int64_t K, int64_t N, void *stream);
Q4_API size_t q4_planar_qs_offset(int64_t K, int64_t N);
Q4_API size_t q4_planar_bytes(int64_t K, int64_t N);

/*
 * q4_dequant -- W [K, N] fp32 = (q - 8) * d, exact  [engine page §2.2].
 * q4_dequant_bf16 -- W [K, N] bf16 bits = bf16 round-to-nearest-even of the
 * same value: the 16-bit operand the tensor-core path multiplies.
 */
Q4_API int q4_dequant(float *W, const void *B, int64_t K, int64_t N, void *stream);
Q4_API int q4_dequant_bf16(uint16_t *W, const void *B, int64_t K, int64_t N, void *stream);

/*
 * Host-streamed weights [AirLLM deep-dive page, §1.2: layers kept in pinned
 * host memory and brought in by a worker while the GPU computes the previous
 * one; §6: the packed quantised bytes cross the link, expansion on the GPU].
 *
 * q4_seq_op -- one matmul C = A . W of a sequence; C and A are DEVICE
 * pointers as everywhere else, B is a PAGE-LOCKED HOST pointer
 * (cudaHostAlloc / cudaHostRegister, e.g. torch pin_memory) to Q4_0 blocks.
 */
typedef struct q4_seq_op {
  void *C;            /* device [M, N], c_dtype                 */
  const void *A;      /* device [M, K], a_dtype                 */
  const void *B;      /* pinned host, K x ceil(N/32) blocks      */
  int64_t M, N, K;
  int a_dtype, c_dtype;
} q4_seq_op;

/* Bytes of one staging slot for `ops`: the largest B, rounded up to 256.
 * 0 if ops is NULL, n <= 0 or a size is <= 0. */
Q4_API size_t q4_host_stream_slot_bytes(const q4_seq_op *ops, int n);

/*
 * q4_matmul_host_stream -- runs ops[0..n) in order on `stream`, each as
 * q4_matmul_ex would (same kernels, same results bit for bit), with its
 * weights copied from host memory into one of `slots` device slots of
 * `staging` on `copy_stream` while earlier matmuls run.  Copy i reuses slot
 * i % slots only after matmul i - slots has finished; matmul i waits for copy
 * i.  `copy_stream` is forked from and joined back into `stream`: the
 * sequence follows earlier work on `stream`, later work on `stream` follows
 * it, and it can be captured into a CUDA graph.
 *   staging      device buffer, 256-byte aligned, >= slots *
 *                q4_host_stream_slot_bytes(ops, n) bytes (else
 *                Q4_ERR_WORKSPACE); owned by the caller and in use until the
 *                sequence completes.
 *   slots        >= 1 (2 or more overlap copies with matmuls).
 *   copy_stream  a stream other than `stream` (else Q4_ERR_ARG).
 * Every op is checked before anything is enqueued: a B that is not
 * page-locked host memory, or a bad size, gives Q4_ERR_ARG; dtype and
 * alignment errors as in q4_matmul_ex.
 */
Q4_API int q4_matmul_host_stream(const q4_seq_op *ops, int n, void *staging, size_t staging_bytes,
                                 int slots, void *stream, void *copy_stream);

/*
 * Decode sequence -- a list of M = 1 GEMVs (C_i = A_i . W_i) run by ONE
 * persistent launch [engine page §2.1: decoding a token streams every weight
 * matrix of the model once, one matrix-vector product each; §3.4 the fused
 * Q4_0 loop].  One launch keeps the HBM busy across the matrices instead of
 * filling and draining a pipeline per matrix.
 *
 * q4_gemv_op -- one GEMV of the sequence:
 *   C       device [N], c_dtype Q4_F32 or Q4_BF16 (RN of the fp32 result)
 *   A       device [K], a_dtype Q4_F32 or Q4_BF16
 *   B       device, K rows of ceil(N/32) block_q4_0 (Q4_LAYOUT_BLOCKS);
 *           ceil(N/32) must be a multiple of 8 (else Q4_ERR_SHAPE)
 *   deps    indices of up to 4 EARLIER ops of the same sequence whose C must
 *           be complete before this op reads A (e.g. when A is, or is
 *           computed from, their output); ndeps = 0 for none.  Weights are
 *           streamed regardless; only the reads of A wait.
 *   slice_rows  rows of K per unit of work: 0 for the library's choice,
 *           else a multiple of 64 up to 4096 (else Q4_ERR_ARG).  Every unit
 *           ends in a reduction over its CTA and adds one partial row to its
 *           tile's combine, so shorter units cost more, while long units near
 *           the end of the sequence leave CTAs idle.  The library's choice:
 *           512 for an op that a later op depends on (so that it completes
 *           soon after its last unit starts); otherwise the longest of 4096,
 *           2048, 1024 and 512 rows such that the weights from this op to the
 *           end of the sequence hold at least half a unit for each of 304
 *           CTAs (152 SMs x 2), i.e. 4096 rows while 179.3 MB or more remain,
 *           2048 from 89.7 MB, 1024 from 44.8 MB, 512 below.
 * Every C is overwritten.  Results are deterministic (each output is summed
 * in a fixed order) and equal A . W within 1e-3 * sum|a*w| + 1e-6, like
 * q4_matmul_ex (the same exact dequantisation; other summation splits).
 */
typedef struct q4_gemv_op {
  void *C;
  const void *A;
  const void *B;
  int64_t N, K;
  int a_dtype, c_dtype;
  int ndeps;
  int deps[4];
  int slice_rows;
} q4_gemv_op;

/* Opaque plan of a decode sequence (host object). */
typedef struct q4_gemv_seq q4_gemv_seq;

/* Bytes of device buffer a plan for `ops` needs (0 if the ops are invalid):
 * the ops' descriptors, counters, and 2 KB of partial sums per unit of work
 * (a unit: 512 output columns x slice_rows rows of one op). */
Q4_API size_t q4_gemv_seq_bytes(const q4_gemv_op *ops, int n);

/*
 * q4_gemv_seq_create -- checks the ops and writes their descriptors into
 * `buf` (a device buffer of >= q4_gemv_seq_bytes bytes, 256-byte aligned,
 * owned by the caller, which must keep it, the weights and the A and C
 * buffers alive while the plan is used).  Synchronous; not for use while a
 * stream is being captured.  The pointers of every op are fixed in the plan:
 * new inputs are written into the same A buffers.  Errors: Q4_ERR_ARG (null
 * pointer, size <= 0, a dependency that is not an earlier op), Q4_ERR_DTYPE,
 * Q4_ERR_ALIGN (a pointer not 16-byte aligned, buf not 256-byte aligned),
 * Q4_ERR_SHAPE, Q4_ERR_WORKSPACE (buf too small), Q4_ERR_CUDA.
 */
Q4_API int q4_gemv_seq_create(const q4_gemv_op *ops, int n, void *buf, size_t buf_bytes,
                              q4_gemv_seq **plan);

/*
 * q4_gemv_seq_run -- runs the whole sequence on `stream`: one small clear of
 * the plan's counters, then one launch of a resident grid (two CTAs per SM)
 * that takes units of work in op order from a shared counter.  Asynchronous;
 * can be captured into a CUDA graph.  Runs of one plan must not overlap on the
 * GPU.  The current device must be the plan's.  A wait that runs out (1 s)
 * records Q4_DEVERR_TIMEOUT (q4_get_device_status).
 */
Q4_API int q4_gemv_seq_run(const q4_gemv_seq *plan, void *stream);

/* Frees the host object of a plan (the caller's device buffer is untouched). */
Q4_API void q4_gemv_seq_destroy(q4_gemv_seq *plan);

/* CTAs of the plan's launch (for measurement). */
Q4_API int q4_gemv_seq_grid(const q4_gemv_seq *plan);

/* Synchronises `stream`, then reads and clears the device status word of the
 * current device: Q4_OK, Q4_ERR_DEVICE (bits in q4_last_device_flags()) or
 * Q4_ERR_CUDA. */
Q4_API int q4_get_device_status(void *stream);
Q4_API unsigned int q4_last_device_flags(void);

/*
 * q4_quantize -- Q4_0 encoder: W [K, N] row-major (w_dtype Q4_F32 or Q4_BF16)
 * -> B [K, ceil(N/32) * 18 bytes] in Q4_LAYOUT_BLOCKS (engine page §2.2-§2.3).
 * The pages give no scale rule; this one, per block (row k, 32 consecutive
 * columns): m = the element of largest magnitude (the first on ties),
 * d = m / -8 (so that m maps to code 0 exactly), stored as fp16 rounded to
 * nearest even; code q = min(15, trunc(w * (1/d) + 8.5)), each step one
 * fp32 operation; 1/d is taken as 0 when d = 0; columns >= N get code 8.
 * Values must be finite.  Pointers 16-byte aligned; B is overwritten.
 */
Q4_API int q4_quantize(void *B, const void *W, int w_dtype, int64_t K, int64_t N, void *stream);

/*
 * q4_moe_gate -- the router in front of the routed experts
 * [KTransformers page, «规则二»: the gate gives the top-k indices and weights].
 *   topk_idx  int32 [T, topk] (out): for each token the topk largest of its
 *             E logits, in descending order; equal logits: lower index first
 *   topk_w    fp32 [T, topk] (out): softmax over the E logits with the maximum
 *             subtracted (engine page §5.1), restricted to the chosen experts
 *             and renormalised: w_i = exp(l_i - l_max) / sum_j exp(l_j - l_max)
 *   logits    fp32 [T, E], finite values
 * The choice compares the fp32 logits exactly.  E <= 1024, topk <= 16 and
 * topk <= E (else Q4_ERR_SHAPE); pointers 16-byte aligned.  The outputs are
 * the inputs q4_moe_experts_ex takes.
 */
Q4_API int q4_moe_gate(int32_t *topk_idx, float *topk_w, const float *logits,
                int64_t T, int64_t E, int64_t topk, void *stream);

/*
 * q4_moe_block -- one DeepSeek-V2-style MoE block on the GPU: router, shared
 * expert and routed experts, in one call that can be captured into a CUDA
 * graph [KTransformers page, «规则二» (gate, then the experts) and «优化三»
 * (the shared expert stays on the GPU with the rest of the block)].
 *   out[t] = sum_k topk_w[t,k] * expert_{topk_idx[t,k]}(x_t) + shared(x_t)
 * with (topk_idx, topk_w) = q4_moe_gate(logits), expert_e as in
 * q4_moe_experts_ex (W_gate, W_up, W_down: E experts, intermediate size I)
 * and shared(x) = (SiLU(x.S_gate) * (x.S_up)) . S_down with intermediate size
 * Is (S_gate, S_up: H rows x ceil(Is/32) blocks; S_down: Is rows x
 * ceil(H/32) blocks).  Is = 0 means no shared expert (S_* may be NULL).  The
 * routed sum is taken in slot order and the shared term added last.
 *   out  fp32 [T, H]; x  [T, H] fp32 or bf16 (x_dtype); logits fp32 [T, E]
 * Workspace: q4_moe_block_workspace_size bytes whose first 64 KB are zero
 * before its first use (as for q4_moe_experts_ex),
 * or NULL for the library-owned workspace shared with q4_moe_experts_ex.
 * Limits as for q4_moe_gate and q4_moe_experts_ex.
 */
Q4_API int q4_moe_block(float *out, const void *x, int x_dtype, const float *logits,
                 const void *W_gate, const void *W_up, const void *W_down,
                 int64_t T, int64_t topk, int64_t E, int64_t H, int64_t I,
                 const void *S_gate, const void *S_up, const void *S_down, int64_t Is,
                 void *workspace, size_t workspace_bytes, void *stream);

Q4_API size_t q4_moe_block_workspace_size(int64_t T, int64_t topk, int64_t E, int64_t H,
                                   int64_t I, int64_t Is);

/*
 * q4_selftest_wait -- failure-detection self-test; no counterpart on the
 * pages.  Launches one CTA that waits on a pipeline barrier with the same
 * bounded wait every kernel uses, but with a limit of `limit_ns`
 * (1 .. 1e9 ns; the kernels use 1 s).  With arrive = 0 nothing completes
 * the barrier: the wait runs out, records Q4_DEVERR_TIMEOUT in the device
 * status word and the kernel returns (no trap, no hang; the context stays
 * usable).  With arrive = 1 the CTA completes the barrier first and the wait
 * succeeds.  Read the outcome with q4_get_device_status(stream).
 * Returns Q4_OK, Q4_ERR_ARG (limit or arrive out of range) or Q4_ERR_CUDA.
 */
Q4_API int q4_selftest_wait(int64_t limit_ns, int arrive, void *stream);

/*
 * q4_prefill_units -- test hook; no counterpart on the pages.  Lists, on
 * the host (no CUDA call), the units of work the persistent prefill form
 * (q4_matmul_bf16_tiles with M > 128 and its tail workspace) gives each of
 * its CTAs for this shape on `sms` SMs, computed by the function the kernel
 * itself runs.  Row i of out[cap][9] (int32): CTA, unit index within the
 * CTA, first row m0, first column n0, first and end K step (of 64 rows),
 * role (0: a whole tile; 1: the part holding the tile's last K step, which
 * adds the earlier parts; 2: an earlier part, which writes its partial
 * tile), and for role 1 the first CTA and the number of CTAs whose parts it
 * adds.  Returns the number of units (rows beyond cap are counted, not
 * written), or Q4_ERR_ARG (M <= 128, non-positive sizes or sms, out NULL
 * with cap > 0) or Q4_ERR_SHAPE (a size above 2^30).
 */
Q4_API int64_t q4_prefill_units(int64_t M, int64_t N, int64_t K, int sms, int32_t *out,
                                int64_t cap);

/* Human-readable text of a status code (static storage). */
Q4_API const char *q4_status_str(int status);

/* Library ABI version (major*100 + minor). */
Q4_API int q4_version(void);

#ifdef __cplusplus
}
#endif
#endif /* Q4_GB300_H */
