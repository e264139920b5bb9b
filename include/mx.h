/*
 * mx.h - C ABI of libmx: low-batch MXFP8 block-scaled projections on GB300 (sm_103a).
 *
 * MXFP8 here means: E4M3 (fn) values with one UE8M0 power-of-two scale per 32
 * consecutive elements along K (sf_vec_size 32), as the vLLM page
 * "vllm.models.deepseek_v41.nvidia.specialized_decode.attention.mxfp8"
 * describes for fused_wqa_wkv, wq_b and wo_b (module docstring;
 * `compile_low_latency`: Float8E4M3FN operands, Float8E8M0FNU scales, bf16 out).
 *
 * Conventions shared by every entry point:
 *  - Every data pointer is a DEVICE pointer owned by the caller, except that the
 *    bf16 input x of mx_quantize_rows and the bf16 output out of mx_gemm may
 *    also be host memory the device addresses directly (pinned: cudaHostAlloc,
 *    cudaHostRegister): those kernels touch them with plain loads and stores,
 *    so a step can read its activations from and write its results to the host
 *    without copy-engine transfers. No call allocates or frees memory. mx_create allocates the handle's device memory
 *    once: a status word, the per-tile counters of the persistent chain kernel
 *    (64 KiB), the activation scratch of wo_a_grouped's two-launch form
 *    (8.25 MiB) and the block sums of squares of mx_gemm_chain_norm's
 *    three-launch form (64 KiB); mx_gemm_chain_noalloc also uses a fixed
 *    array inside the library.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream) and must be made with the handle's
 *    device current.
 *  - Arguments are validated before anything is launched: on any error the
 *    outputs are left untouched and nothing is enqueued (the page
 *    "vllm.models.deepseek_v41.nvidia.ops.cute_dsl", `_consumer`: a bad
 *    argument raises before the call's first launch).
 *  - MX_OK from a launching entry point means the work was enqueued. A bounded
 *    device-side wait that expires makes the kernel skip its remaining work
 *    instead of hanging, so the outputs of every call since the last check are
 *    defined only once mx_device_status reports MX_OK.
 *  - Activation scales and weight scales use the F8_128x4 swizzled layout:
 *    the [rows, K/32] scale matrix is padded to ceil128(rows) x ceil4(K/32)
 *    and cut into 128x4 tiles of 512 contiguous bytes (tiles row-major); inside
 *    a tile, (r, c) sits at byte 16*(r%32) + 4*(r/32) + c. Buffer size:
 *    mx_scale_bytes(rows, K).
 *  - Weights are [N, K] row-major E4M3 (K contiguous), i.e. the column-major
 *    [K, N] weight of `launch_low_latency`.
 */
#ifndef MX_H_
#define MX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
  MX_OK = 0,
  MX_ERR_INVALID_ARG = 1, /* null/misaligned pointer, size out of range        */
  MX_ERR_UNSUPPORTED = 2, /* shape outside what the kernels take: caller falls
                             back (the page's functions return None there)    */
  MX_ERR_DEVICE = 3,      /* not a compute-capability 10.3 device, or a call
                             made with another device current                 */
  MX_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed             */
  MX_ERR_TIMEOUT = 5      /* a bounded device-side wait expired (see
                             mx_device_status)                                 */
};

/* Flags for mx_gemm. */
#define MX_FLAG_PDL 1u /* launch with programmatic stream serialization: the
                          kernel streams its weights before waiting for the
                          previous kernel on the stream (`launch_low_latency`
                          / module docstring of the mxfp8 page)              */

typedef struct mx_handle mx_handle;

/* Weight operand of one projection: E4M3 [n, k] plus swizzled scales. */
typedef struct mx_weight {
  const void* w;        /* [n, k] E4M3, 16-byte aligned                      */
  const void* w_scales; /* mx_scale_bytes(n, k) bytes, 32-byte aligned       */
  int n;                /* output features, multiple of 128                  */
  int k;                /* input features, multiple of 128                   */
} mx_weight;

/* Create a handle for `device`. Checks compute capability 10.3 (the device
 * gate of `_cute_dsl_runner` / `_wide_supported` on the mxfp8 page), loads the
 * kernels and allocates the handle's device memory (the status word, the
 * persistent chain's counters, zeroed, and wo_a_grouped's scratch). The handle also caches
 * the tensor maps of the buffers it has seen (host memory only), so one handle
 * is used by one host thread at a time; give each thread its own handle.
 * Returns MX_ERR_DEVICE on another architecture, MX_ERR_CUDA if no device. */
int mx_create(mx_handle** h, int device);
int mx_destroy(mx_handle* h);

/* Bytes of a swizzled scale buffer for a [rows, k] MXFP8 operand:
 * ceil128(rows) * ceil4(k/32) (`mxfp8_scale_bytes` on the mxfp8 page, `_zeros`).
 * Returns 0 for rows < 0 or k not a multiple of 32. */
size_t mx_scale_bytes(int rows, int k);

/* Quantize bf16 rows to MXFP8 (the role of `mxfp8_e4m3_quantize(a,
 * is_sf_swizzled_layout=True)` in `wide_mm` / `pinned_mm` on the mxfp8 page).
 *   x      [M, K] bf16, row stride ldx elements (ldx >= K, ldx % 8 == 0),
 *          16-byte aligned.
 *   q      [M, K] E4M3 out, row stride K, 16-byte aligned.
 *   scales out: swizzled (mx_scale_bytes(M, K) bytes, padding written as 0)
 *          when swizzled != 0, else plain row-major [M, K/32].
 * Per 32-block: e = floor(log2 amax) - 8 clamped to [-127, 127] (e = -127
 * for a zero block), codes = E4M3 saturating round-to-nearest-even of
 * x * 2^-e, scale byte e + 127; a block holding NaN/Inf gets scale 0xFF and
 * NaN codes. Constraints: 1 <= M <= 65536, K % 32 == 0, K > 0. */
int mx_quantize_rows(mx_handle* h, int M, int K, const void* x, long ldx,
                     void* q, void* scales, int swizzled, void* stream);

/* RMS normalization then MX quantization of each row: y = bf16(x / sqrt(mean
 * over the row of x^2 + eps) * norm_weight), computed in float32, then y
 * quantized as mx_quantize_rows does. The squares are summed in a fixed order:
 * per 32-block the pairwise tree over its elements (element j with j ^ 16, then
 * j ^ 8, j ^ 4, j ^ 2, j ^ 1), then the block sums from the first block on;
 * the reciprocal RMS is 1 / sqrt(sum / K + eps) with correctly rounded division
 * and square root. This is the split between the first two
 * projections of a decode step (`qr, qr_scale, kv = attn._split_qkv_and_norm(
 * qr_kv)` in `AttentionStep.run`, step page; the pages show only the call: the
 * reading is an RMS norm of qr with a given weight and epsilon).
 *   x           [M, K] bf16, row stride ldx elements (ldx >= K, ldx % 8 == 0),
 *               16-byte aligned.
 *   norm_weight [K] bf16, 16-byte aligned; eps >= 0.
 *   y           optional [M, K] bf16 out (row stride K), or null.
 *   q, scales   as in mx_quantize_rows.
 * Constraints: 1 <= M <= 65536, K % 32 == 0. */
int mx_rmsnorm_quantize_rows(mx_handle* h, int M, int K, const void* x, long ldx,
                             const void* norm_weight, float eps, void* y, void* q,
                             void* scales, int swizzled, void* stream);

/* out = dequant(A) x dequant(W)^T (`launch_low_latency`: out = a times the
 * column-major [K, N] weight; bf16 out, float32 accumulation, no scale/bias).
 *   a        [M, K] E4M3, row stride K, 16-byte aligned.
 *   a_scales mx_scale_bytes(M, K) bytes, swizzled, 16-byte aligned.
 *   w        [N, K] E4M3, 16-byte aligned; w_scales swizzled, 32-byte aligned.
 *   out      [M, N] bf16 row-major, 16-byte aligned; rows >= M untouched.
 * Constraints: 1 <= M <= 256, N % 128 == 0, K % 128 == 0 (`mxfp8_eligible`:
 * weight K a multiple of 128), else MX_ERR_UNSUPPORTED / MX_ERR_INVALID_ARG.
 * flags: MX_FLAG_PDL. */
int mx_gemm(mx_handle* h, int M, int N, int K, const void* a, const void* a_scales,
            const void* w, const void* w_scales, void* out, unsigned flags,
            void* stream);

/* mx_gemm with bf16 activations quantized inside the GEMM: out equals, bit for
 * bit, mx_quantize_rows(x) (swizzled scales) followed by mx_gemm on the same
 * stream (the mxfp8 page's `wide_mm` / `pinned_mm` quantize the bf16 x and
 * then run the MXFP8 GEMM: two launches; here one). Each CTA quantizes the
 * K-range it contracts, in shared memory; the MXFP8 activation is not written.
 *   x        [M, K] bf16, row stride ldx elements (ldx >= K, ldx % 8 == 0),
 *            16-byte aligned.
 *   w, w_scales, out, flags: as in mx_gemm.
 * Constraints: as mx_gemm; MX_ERR_UNSUPPORTED also when the K-range's
 * quantized rows do not fit in one CTA's shared memory (large M with few
 * K-splits): the caller then uses mx_quantize_rows + mx_gemm.
 * Cost: every CTA quantizes the K-range it contracts (each 32-block split
 * over up to 8 threads when the rows are few), so the N/128 weight tiles
 * repeat that work; it saves a launch, and on GB300 at N = 2048, K = 5120 it
 * is faster than mx_quantize_rows + mx_gemm from one to four rows (4.44 /
 * 4.46 / 4.81 us at 1 / 2 / 4 rows against 1.17 us + 3.85 / 3.89 / 4.03 us),
 * slower at eight (5.57 against 1.17 + 4.01 us). */
int mx_gemm_bf16(mx_handle* h, int M, int N, int K, const void* x, long ldx,
                 const void* w, const void* w_scales, void* out, unsigned flags,
                 void* stream);

/* The three projections of a decode step's attention on one stream
 * (fused_wqa_wkv -> wq_b -> wo_b on the mxfp8 page and in `AttentionStep.run`
 * of the page "...specialized_decode.attention.step"), every kernel launched
 * with programmatic dependent launch so its weight read overlaps the previous
 * kernel (mxfp8 page, module docstring):
 *   out1 = G1(a1)                         [M, w[0].n]
 *   a2   = MXFP8(bf16(out1)[:, :g1_cols])  fused into G1's epilogue
 *   out2 = G2(a2)                         [M, w[1].n], w[1].k == g1_cols
 *   a3   = MXFP8(bf16(out2))              fused into G2's epilogue, w[2].k == w[1].n
 *   out  = G3(a3)                         [M, w[2].n] bf16
 * a2/a2_scales/a3/a3_scales are caller-owned intermediates ([M, K] E4M3 and
 * mx_scale_bytes(M, K) swizzled bytes each). debug_out1 / debug_out2
 * (nullable) receive the bf16 out1 / out2. Constraints as mx_gemm, plus
 * g1_cols % 128 == 0 and g1_cols <= w[0].n. */
int mx_gemm_chain(mx_handle* h, int M, const void* a1, const void* a1_scales,
                  const mx_weight w[3], int g1_cols, void* a2, void* a2_scales,
                  void* a3, void* a3_scales, void* out, void* debug_out1,
                  void* debug_out2, void* stream);

/* mx_gemm_chain with the split between G1 and G2 of `AttentionStep.run`:
 * G1 writes its whole bf16 output to out1 ([M, N1]: qr = columns [0, g1_cols),
 * kv = the rest, which the caller reads from out1), qr is RMS-normalized with
 * norm_weight / eps and MX-quantized into a2 / a2_scales (bit for bit what
 * mx_rmsnorm_quantize_rows writes), then G2 (+ requantization into a3) and G3
 * as in mx_gemm_chain. On one stream, with PDL. Up to 16 rows in three
 * launches: G1's epilogue also writes each 32-block's sum of squares of qr to
 * the handle's scratch, and G2 reads qr in bf16, adds those sums in block
 * order for each row's RMS and normalizes and quantizes the K-range it
 * contracts in its prologue (the CTAs of the first weight tile also store a2,
 * a2_scales and debug_y). Above 16 rows, where every CTA of G2 repeating the
 * quantization of its K-range costs more than a launch, the norm kernel runs
 * between G1 and G2 (four launches). Both forms give the same bits as
 * mx_rmsnorm_quantize_rows between mx_gemm calls. Calls on one handle whose
 * work overlaps on the GPU race on the scratch (as for wo_a_grouped).
 *   norm_weight [g1_cols] bf16, 16-byte aligned; eps >= 0.
 *   out1        [M, N1] bf16, required.
 *   debug_y     optional [M, g1_cols] bf16: the normalized qr before quantization.
 * Other arguments and constraints as in mx_gemm_chain. */
int mx_gemm_chain_norm(mx_handle* h, int M, const void* a1, const void* a1_scales,
                       const mx_weight w[3], int g1_cols, const void* norm_weight, float eps,
                       void* out1, void* a2, void* a2_scales, void* a3, void* a3_scales,
                       void* out, void* debug_y, void* debug_out2, void* stream);

/* mx_gemm_chain for callers that cannot allocate device memory. Some callers
 * have no way to provide the chain's two intermediate buffers: code that runs
 * while a stream is being captured into a CUDA graph (cudaMalloc is not a
 * stream operation and may synchronize the device), engines that hand a
 * kernel library only the input and output buffers because they budget every
 * byte of device memory themselves, and plugin hosts with no allocator exposed
 * to the plugin. This entry point takes only the inputs and the output:
 *   out = G3(MXFP8(G2(MXFP8(G1(a1)[:, :g1_cols])))), exactly as mx_gemm_chain
 * computes it with debug_out1 = debug_out2 = NULL.
 * The intermediates (a2 and a3 with their swizzled scales, each rounded up to
 * 256 bytes) live in one fixed 1 MiB device array inside the library, which
 * every GPU that loads the library holds until the process exits. The call
 * allocates nothing and calls no allocating routine.
 * Limit: round256(M*g1_cols) + round256(mx_scale_bytes(M, g1_cols)) +
 * round256(M*w[1].n) + round256(mx_scale_bytes(M, w[1].n)) <= 1 MiB (for
 * g1_cols = 1536 and w[1].n = 8192: M <= 99); larger problems return
 * MX_ERR_UNSUPPORTED before anything is launched - use mx_gemm_chain with
 * caller buffers then.
 * The first call on a device looks up the array's device address with that
 * device current (a one-time set-up per device); make that first call before
 * any stream capture. Every call shares the array, and it keeps the last call's
 * contents: each byte the kernels read is written earlier in the same call, so
 * nothing has to start at zero. Calls whose work overlaps on the GPU (two
 * streams, or a graph replay next to another call) race on the array: order
 * them on one stream. The paper has no counterpart: this is an addition for
 * callers without an allocator.
 * Other arguments, constraints and errors as in mx_gemm_chain. */
int mx_gemm_chain_noalloc(mx_handle* h, int M, const void* a1, const void* a1_scales,
                          const mx_weight w[3], int g1_cols, void* out, void* stream);

/* Grouped WO-A with RoPE, writing MXFP8 for wo_b (`dsv41_o_proj` and
 * `_can_fuse_wo_a` on the page "vllm.models.deepseek_v41.nvidia.ops.o_proj").
 *   x          [T, >= G*H heads, d_nope + d_rope] bf16; token stride ldx
 *              elements (ldx >= G*H*(d_nope+d_rope), ldx % 8 == 0), head
 *              stride d_nope + d_rope; heads gH..gH+H-1 form group g.
 *   positions  [T] int64 token positions, 0 <= pos < max_pos.
 *   cos_sin    [max_pos, d_rope] float32: row p = [cos(p f_i) | sin(p f_i)].
 *   w          [G*R, H*(d_nope+d_rope)] E4M3 (group g = rows gR..gR+R-1),
 *              w_scales swizzled over those [G*R, H*D/32] scales.
 *   q, q_scales  out: [T, G*R] E4M3 (row stride G*R) and mx_scale_bytes(T, G*R)
 *              swizzled bytes: the MXFP8 activation handed to wo_b.
 *   debug_z    nullable [T, G*R] bf16 z before requantization.
 *   debug_xq, debug_xs  nullable [T, G*H*D] E4M3 and plain [T, G*H*D/32] scale
 *              bytes of the RoPE'd, quantized activation the contraction reads.
 * The rope dims (the last d_rope of each head) are rotated on adjacent pairs
 * by -pos * f_i in float32 (a' = a c + b s, b' = b c - a s, no fused
 * multiply-add), quantized per 32 with the nope dims (never rounded to bf16),
 * contracted per group to R = o_lora_rank with float32 accumulation, rounded
 * to bf16 and quantized again.
 * Constraints: d_nope == 448, d_rope == 64, H <= 8, R % 128 == 0,
 * 1 <= T <= 128; else MX_ERR_UNSUPPORTED (the unfused path's domain).
 * early_trigger != 0: the dependent kernel (wo_b) may launch right after
 * this kernel has allocated its tensor memory (`dsv41_o_proj`).
 * Above 8 tokens, when debug_xq and debug_xs are null and the quantized
 * activation (T*G*H*D bytes plus its scales) fits the handle's 8.25 MiB
 * scratch, the call runs wo_a_grouped_unfused's two launches on that scratch
 * instead of the fused kernel (faster there on GB300: T = 32 takes 9.9 us
 * against 15.8 us); q, q_scales and debug_z mean the same, the dependent kernel
 * may launch once the second launch's GEMM releases it, and two such calls on
 * one handle whose work overlaps on the GPU race on the scratch: give each
 * stream its own handle. */
int wo_a_grouped(mx_handle* h, int T, const void* x, long ldx, const int64_t* positions,
                 const float* cos_sin, int max_pos, const void* w, const void* w_scales,
                 int G, int H, int d_nope, int d_rope, int R, void* q, void* q_scales,
                 void* debug_z, void* debug_xq, void* debug_xs, int early_trigger,
                 void* stream);

/* The same projection as wo_a_grouped in two launches, for token counts the
 * fused kernel does not take (the o_proj page's fallback: `grouped_forward`
 * when the tokens exceed the fused limit, z then fed to wo_b):
 *   1. inverse RoPE + per-32 MX quantization of every head -> xq, xq_scales;
 *   2. one grouped block-scaled GEMM: the R output rows of group g contract
 *      the group's K-slice of xq; z rounded to bf16 and requantized to q.
 *   xq         [T, G*H*D] E4M3 (caller-owned intermediate), 16-byte aligned.
 *   xq_scales  mx_scale_bytes(T, G*H*D) bytes, swizzled, 16-byte aligned.
 *   z          optional [T, G*R] bf16 (the pre-quantization output), or null.
 *   other arguments as in wo_a_grouped (H is not limited to 8 here).
 * q / q_scales equal mx_quantize_rows of bf16(z). On GB300 the fused kernel is
 * faster up to 8 tokens and this path from 10 on (T = 10: 7.85 vs 8.04 us;
 * T = 32: 9.9 vs 15.8 us; T = 128: 19.4 vs 74.7 us), so wo_a_grouped itself
 * takes this path above 8 tokens. Constraints: 1 <= T <= 256,
 * d_nope = 448, d_rope = 64, R % 128 == 0, else MX_ERR_UNSUPPORTED. A position
 * outside [0, max_pos) reads cache row 0 and is reported by mx_device_status,
 * as in wo_a_grouped. */
int wo_a_grouped_unfused(mx_handle* h, int T, const void* x, long ldx,
                         const int64_t* positions, const float* cos_sin, int max_pos,
                         const void* w, const void* w_scales, int G, int H, int d_nope,
                         int d_rope, int R, void* xq, void* xq_scales, void* z, void* q,
                         void* q_scales, void* stream);

/* Bytes of device scratch mx_warmup needs for these weights and row counts:
 * round256(the largest rows*k) for the zero activation's codes, then
 * round256(the largest mx_scale_bytes(rows, k)) for its scales, then one
 * round256(rows*n*2)-byte bf16 output per (shape, row count) run, in the order
 * of mx_warmup. 0 for invalid arguments (no weight or row count, rows < 1,
 * k not a multiple of 32). Host-only: touches no device. */
size_t mx_warmup_bytes(const mx_weight* w, int nw, const int* rows, int nrows);

/* Readies the kernels for the weight shapes a model will run, before its first
 * real call (the mxfp8 page's `compile_pinned`, `run_zeros` and `_zeros` over
 * `shape_representatives`): for each distinct (n, k) among w[0..nw), in
 * increasing (n, k) order, using the first weight of that shape, and for each
 * row count rows[0..nrows) in the given order, computes and keeps the handle's
 * GEMM plan, encodes the tensor maps and runs mx_gemm once on a zero MXFP8
 * activation (zero codes, zero scale bytes), with PDL, on stream.
 *   scratch  device buffer of at least mx_warmup_bytes(...) bytes, 256-byte
 *            aligned: the call zeroes the activation part and writes each
 *            run's [rows, n] bf16 output after it, in the layout
 *            mx_warmup_bytes describes. With finite weights every output is 0.
 * Every run is validated and prepared before the first launch: an invalid
 * weight or row count (as mx_gemm would reject it: rows > 256, n % 128 or
 * k % 128 != 0, a misaligned pointer) returns its error with nothing enqueued.
 * Call it after mx_create and before any stream capture. The paper's
 * counterpart compiles kernels; this library's kernels are loaded at mx_create,
 * so what it readies are the plans, the tensor maps and the first launch. */
int mx_warmup(mx_handle* h, const mx_weight* w, int nw, const int* rows, int nrows,
              void* scratch, size_t scratch_bytes, void* stream);

/* ------------------------------------------------------------ plan queries
 * Host-only (no device, no handle): the launch plans the entry points make,
 * the mxfp8 page's fixed tactic per (shape, row range) as this library picks
 * it, for inspection and tests. The tuning overrides of the environment
 * (MX_SPLITS, MX_STAGES, MX_PLAN_AT, MX_PUSH_ROWS) apply as at mx_create. */

/* How a plan sums the K-splits' fp32 partials (every form in rank order, so
 * all give the same bits): peer loads of 32-column items, of whole rows, or
 * the push exchange (each CTA stores the partials another rank owns into that
 * rank's shared memory) with a receive slot per rank or, compact, per peer. */
#define MX_REDUCE_ITEMS 0
#define MX_REDUCE_ROWS 1
#define MX_REDUCE_PUSH 2
#define MX_REDUCE_PUSH_COMPACT 3
/* The receive area a plan may take for the push exchange (mx_gemm: FULL). */
#define MX_PUSH_NONE 0
#define MX_PUSH_COMPACT 1
#define MX_PUSH_FULL 2

typedef struct mx_plan_info {
  int splits;     /* K-splits: the CTAs of one cluster */
  int stages;     /* weight ring depth */
  int mtile;      /* rows padded to a multiple of 16 (the MMA's N) */
  int tmem_cols;  /* tensor-memory columns per CTA */
  int reduction;  /* MX_REDUCE_* */
  size_t smem;    /* dynamic shared memory per CTA, bytes (above 232448: the
                     shape is unsupported and the entry point rejects it) */
} mx_plan_info;

/* The plan of a [M, K] x [N, K]^T launch on a device with sm_count SMs, as
 * mx_gemm (fused = 0) or mx_gemm_bf16 (fused = 1; norm = 1: the chain-norm's
 * G2 with the RMS norm in its prologue) makes it, allowing the push exchange
 * with receive area `push` (MX_PUSH_*). Returns MX_ERR_INVALID_ARG for
 * M outside 1..256, N or K not a multiple of 128, sm_count < 1 or a null out. */
int mx_plan_gemm(int M, int N, int K, int sm_count, int fused, int norm, int push,
                 mx_plan_info* out);

/* The push receive area (MX_PUSH_*) each of the three projections w[0..2] of
 * mx_gemm_chain (norm = 0) or mx_gemm_chain_norm (norm = 1) takes at M rows on
 * a device with sm_count SMs, smem_per_sm bytes of shared memory per SM and
 * smem_reserved bytes reserved per resident block. Under PDL the next grid's
 * CTAs start beside the previous grid's only where both fit an SM; for every
 * pair of neighbours (G3 of the previous step before G1) that fits without the
 * receive areas, the chosen forms fit too, the later projection stepping down
 * first (full, compact, none). Shapes as for mx_gemm_chain; MX_ERR_INVALID_ARG
 * otherwise. */
int mx_plan_chain_push(int M, const mx_weight w[3], int norm, int sm_count, size_t smem_per_sm,
                       size_t smem_reserved, int modes[3]);

/* Read and clear the device status word: MX_OK, or MX_ERR_TIMEOUT if a kernel
 * gave up on a bounded wait since the last call. Synchronizes the device. */
int mx_device_status(mx_handle* h, int* status);

/* Diagnostic of the failure path. Launches one thread that waits, through the
 * bounded mbarrier wait every kernel's pipeline uses, on a barrier that nothing
 * completes. After the wait's limit (one second of the GPU's global timer) the
 * thread records a timeout in the handle's status word and the kernel returns,
 * so the next mx_device_status reports MX_ERR_TIMEOUT and the context stays
 * usable: a wait that cannot complete ends as a status, not as a hung GPU.
 * Asynchronous on stream; returns MX_OK once launched, MX_ERR_INVALID_ARG for a
 * null handle, MX_ERR_DEVICE if another device is current. */
int mx_wait_selftest(mx_handle* h, void* stream);

/* Human-readable name of a status code. */
const char* mx_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* MX_H_ */
