/*
 * nvfp4moe.h -- C ABI of the NVFP4 Mixture-of-Experts expert forward for one
 * GB300 GPU (sm_103a).
 *
 * The operation is the one the "NVFP4 MegaMoE Kernel" README describes in
 * "MoE Runner" (six steps) with the fused L1 epilogue of "Fused SwiGLU - How
 * It Works": route tokens and permute them into per-expert groups, quantize
 * the BF16 activations to NVFP4, run the L1 grouped GEMM whose epilogue
 * computes silu(gate)*up and requantizes it to NVFP4, run the L2 grouped
 * GEMM, and add the expert outputs back per token, weighted by the routing
 * weights.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is a DEVICE pointer unless its comment says "host".
 *   The caller allocates and owns all memory, including the workspaces; the
 *   library never allocates or frees memory and never synchronises a stream
 *   (nvfp4moe_last_device_status is the one call that waits on its stream).
 * - Every launching call takes a cudaStream_t (passed as void*, NULL = the
 *   legacy default stream), enqueues its kernels on it and returns at once.
 * - Global scales are f32 values in device memory so that no call needs a
 *   host round trip.
 * - Return value: NVFP4MOE_OK, or a negative status (below). Arguments are
 *   checked on the host before anything is launched; a call that returns an
 *   error has launched nothing, except NVFP4MOE_ERR_LAUNCH, which reports the
 *   CUDA error of a launch.
 *
 * Data formats
 * ------------
 * - BF16 matrices: row-major, leading dimension in elements.
 * - NVFP4 matrix (rows x cols), cols a multiple of 16 (README "What We Have":
 *   per-16-element FP8 scales, FP32 global scale):
 *     codes: rows x cols/2 bytes, row-major; element c of a row is the E2M1
 *            code in the low nibble of byte c/2 when c is even, the high nibble
 *            when c is odd. E2M1 values {0,0.5,1,1.5,2,3,4,6}, bit 3 = sign.
 *     scales: one E4M3 byte per 16 consecutive elements of a row.
 *     value(r, c) = e2m1(code) * e4m3(scale) / gs.
 * - Scale layouts:
 *     NVFP4_SF_ROWMAJOR: rows x cols/16 bytes, row-major.
 *     NVFP4_SF_TILED:    the layout the tensor-core block-scaled MMA reads.
 *       Rows are padded to a multiple of 128 and scale columns to a multiple
 *       of 4; the scale of row r, 16-element block b lives at byte
 *         ((r / 128) * C4 + b / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + b % 4
 *       with C4 = ceil(cols / 64). Size: nvfp4_sf_bytes(rows, cols, TILED).
 *       The grouped GEMMs read their weight (B) scales in this layout.
 *     NVFP4_SF_TILED_ROWS: tiles of 128 rows x 16 scale columns (2048 bytes),
 *       row-major inside: the scale of row r, block b lives at byte
 *         ((r / 128) * S + b / 16) * 2048 + (r % 128) * 16 + b % 16
 *       with S = ceil(cols / 256); rows padded to 128, scale columns to 16.
 *       The grouped GEMMs read their activation (A) scales in this layout:
 *       one 256-element K stage of 128 rows is 2048 contiguous bytes, and a
 *       row's 16 consecutive blocks are 16 contiguous bytes, so a quantizer
 *       that scatters rows writes whole 16-byte pieces. Size:
 *       nvfp4_sf_bytes(rows, cols, TILED_ROWS).
 * - Quantization rule (README "Correctness Bugs Fixed", bugs 3 and 4): per
 *   block, p = amax * gs; a block with amax == 0 or p < 6 * 2^-9 gets scale
 *   byte 0 and all codes 0; otherwise sf = E4M3_rn_satfinite(p / 6) and
 *   code_i = E2M1_rn_satfinite((x_i * gs) / value(sf)), each step one f32
 *   operation; a negative element whose code magnitude rounds to 0 keeps the
 *   sign bit (code 0x8).
 * - Global scale: gs = 2688 / amax over the tensor (2688 = 6 * 448); 1 when
 *   the tensor is all zero.
 * - Grouped-padded rows: an activation operand grouped by expert, with counts
 *   n_e given by offsets (offsets[0] = 0, offsets[e+1] = offsets[e] + n_e,
 *   offsets[E] = M), stores group e at rows [P_e, P_e + n_e) where
 *     P_e = 128 * sum_{e' < e} ceil(n_e' / 128).
 *   Rows between groups are padding; their contents never reach a valid
 *   output. Capacity needed: nvfp4moe_padded_rows(M, E) rows. This is the
 *   README "Key Lessons" 4 layout: compact data scattered into a padded
 *   buffer, never a padded buffer quantized and sliced.
 * - Expert weights for the grouped GEMMs: B (E, N, K) NVFP4 with K contiguous
 *   (README "Bridge Layer": make_b_k_major), codes E x N x K/2 bytes, scales
 *   NVFP4_SF_TILED per expert with expert e at byte e * nvfp4_sf_bytes(N, K,
 *   NVFP4_SF_TILED), global scales gs_b[E] (README "What We Have": per-expert
 *   global scales).
 * - W1 of the fused L1 GEMM holds 2I rows whose gate and up rows are
 *   interleaved at granularity 8 (README "Fused SwiGLU - How It Works"):
 *   row 16*(i/8) + i%8 is gate row i, row 16*(i/8) + 8 + i%8 is up row i.
 *   nvfp4moe_interleave_row_map gives the source row of each interleaved row.
 */
#ifndef NVFP4MOE_H
#define NVFP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  NVFP4MOE_OK = 0,
  NVFP4MOE_ERR_INVALID = -1,        /* null/negative/misaligned argument      */
  NVFP4MOE_ERR_UNSUPPORTED = -2,    /* shape outside the supported range     */
  NVFP4MOE_ERR_WORKSPACE = -3,      /* workspace missing or too small         */
  NVFP4MOE_ERR_LAUNCH = -4,         /* a kernel launch failed (CUDA error)    */
  NVFP4MOE_ERR_DEVICE_TIMEOUT = -5  /* a kernel gave up a bounded wait        */
};

#define NVFP4_SF_ROWMAJOR 0
#define NVFP4_SF_TILED 1
#define NVFP4_SF_TILED_ROWS 2

/* Routed rows (T * k) up to which moe_dispatch and moe_dispatch_static do the
 * quantize + scatter inside their cooperative kernel; above, a second kernel
 * does it (measured faster there). */
#define NVFP4MOE_FRONT_FUSED_QUANTIZE_MAX_ROWS 32768

/* Short description of a status code (static string). */
const char* nvfp4moe_status_string(int status);

/* Bytes of the scale array of a (rows x cols) NVFP4 matrix in the given
 * layout; 0 for an invalid layout or negative sizes. Host only. */
size_t nvfp4_sf_bytes(int64_t rows, int64_t cols, int sf_layout);

/* Row capacity of a grouped-padded operand holding M rows in E groups:
 * 128 * ceil((M + min(E, M) * 127) / 128). Host only. */
int64_t nvfp4moe_padded_rows(int64_t M, int E);

/* Host: fills map_host[0 .. two_i) with the source row (in [gate | up] order)
 * of each interleaved W1 row (granularity 8). two_i must be a multiple of 16.
 * Returns NVFP4MOE_OK or NVFP4MOE_ERR_INVALID. */
int nvfp4moe_interleave_row_map(int64_t two_i, int32_t* map_host);

/*
 * Offline layout helpers (README "Bridge Layer": assemble_scales_2d_side /
 * assemble_scales_3d_side assemble scale factors into the layout the MMA
 * reads; interleave_l1_weights / deinterleave_l1_weights). Untimed weight
 * preparation; each launches one gather kernel on `stream` and allocates
 * nothing. Inputs and outputs must not overlap.
 *
 * nvfp4_sf_to_tiled -- `batch` scale matrices of (rows x cols) elements, each
 * rows x cols/16 row-major bytes (matrix m at byte m * rows * cols/16), into
 * the tiled layout sf_layout (NVFP4_SF_TILED or NVFP4_SF_TILED_ROWS), matrix m
 * at byte m * nvfp4_sf_bytes(rows, cols, sf_layout). Every byte of the tiled
 * output is written; padding rows and columns get 0. For the expert weights
 * of the grouped GEMMs: batch = E, (rows, cols) = (N, K), NVFP4_SF_TILED.
 * nvfp4_sf_from_tiled -- the inverse: the rows x cols/16 valid bytes of each
 * tiled matrix, row-major.
 * Errors: INVALID (cols % 16 != 0, negative sizes, null pointer, bad layout),
 * LAUNCH.
 */
int nvfp4_sf_to_tiled(const uint8_t* sf, int64_t batch, int64_t rows, int64_t cols, int sf_layout,
                      uint8_t* sf_tiled, void* stream);
int nvfp4_sf_from_tiled(const uint8_t* sf_tiled, int64_t batch, int64_t rows, int64_t cols, int sf_layout,
                        uint8_t* sf, void* stream);

/*
 * nvfp4_interleave_gate_up -- README "Fused SwiGLU - How It Works": W1's 2I
 * rows [gate 0..I-1 | up 0..I-1] reordered so that rows are interleaved at
 * granularity 8 ([g0-7, u0-7, g8-15, u8-15, ...]: row 16*(i/8) + i%8 is gate
 * row i and row 16*(i/8) + 8 + i%8 is up row i), or back (inverse = 1). Whole
 * NVFP4 rows move, since the 16-element blocks run along K.
 *   codes / codes_out  batch x two_i x K/2 bytes (NULL both to skip).
 *   sf / sf_out        batch scale matrices of (two_i, K) in sf_layout
 *                      (NVFP4_SF_ROWMAJOR, NVFP4_SF_TILED or
 *                      NVFP4_SF_TILED_ROWS), matrix m at byte
 *                      m * nvfp4_sf_bytes(two_i, K, sf_layout); the same
 *                      layout in and out, tiled padding written 0 (NULL both
 *                      to skip).
 * Requires two_i % 16 == 0, K % 16 == 0, batch <= 65535. Errors: INVALID,
 * UNSUPPORTED, LAUNCH.
 */
int nvfp4_interleave_gate_up(const uint8_t* codes, const uint8_t* sf, int64_t batch, int64_t two_i, int64_t K,
                             int sf_layout, int inverse, uint8_t* codes_out, uint8_t* sf_out, void* stream);

/* Workspace bytes nvfp4_quantize needs when it computes the global scale. */
size_t nvfp4_quantize_workspace_size(void);

/*
 * nvfp4_quantize -- BF16 -> NVFP4 block quantization (README "Bridge Layer":
 * quantize_to_nvfp4 / quantize_activation_nvfp4 / quantize_weight_to_nvfp4).
 *
 *   x        BF16 source, row-major, leading dimension ldx (elements); its base
 *            address and ldx*2 must be multiples of 16 bytes.
 *   rows     output rows (>= 0); cols: elements per row, a multiple of 16.
 *   gs_in    device f32 global scale to use (pre-computed), or NULL to compute
 *            gs = 2688 / amax over the source rows this call reads.
 *   gs_out   device f32 that receives the global scale used, or NULL. May
 *            alias gs_in.
 *   row_src  NULL (output row r reads x row r) or a device int32 array of
 *            `rows` entries: output row r reads x row row_src[r]; a negative
 *            entry makes output row r all-zero (codes 0, scales 0).
 *   codes    rows x cols/2 bytes (output, 8-byte aligned).
 *   sf       scales (output) in layout sf_layout (NVFP4_SF_ROWMAJOR,
 *            NVFP4_SF_TILED or NVFP4_SF_TILED_ROWS); in the tiled layouts
 *            the padding rows/columns are not written.
 *   ws       when gs_in == NULL: >= nvfp4_quantize_workspace_size() bytes,
 *            16-byte aligned; otherwise ignored (may be NULL).
 * Errors: INVALID (null pointer, cols % 16 != 0, misalignment, bad layout),
 * WORKSPACE, LAUNCH.
 */
int nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ldx,
                   const float* gs_in, float* gs_out, const int32_t* row_src,
                   uint8_t* codes, uint8_t* sf, int sf_layout,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * moe_route_topk -- router step (stage 1): for each of T tokens, the k
 * largest of its E logits (ties to the lower expert index), ordered by
 * descending logit, and softmax weights over those k logits (f32, expf).
 *   logits  (T, E) f32 row-major.  topk_ids (T, k) int32, topk_w (T, k) f32.
 * Supports 1 <= k <= 16, k <= E <= 1024. Logits may be -inf (never chosen
 * before a finite one); a NaN logit ranks below every other logit (as -inf).
 */
int moe_route_topk(const float* logits, int64_t T, int E, int k,
                   int32_t* topk_ids, float* topk_w, void* stream);

/* Workspace bytes moe_permute needs. */
size_t moe_permute_workspace_size(int64_t T, int k, int E);

/*
 * moe_permute -- group the T*k routed slots by expert (README "Correctness
 * Bugs Fixed" bug 5: counts per expert, then an exclusive prefix sum).
 *   topk_ids      (T, k) int32 in [0, E).
 *   offsets       (E + 1) int32: offsets[e] = number of slots routed to
 *                 experts < e; offsets[E] = T*k.
 *   perm_to_flat  (T*k) int32: row r of the grouped order holds flat slot
 *                 f = t*k + j; inside one expert, rows follow ascending f.
 *   flat_to_perm  (T*k) int32: the inverse permutation.
 * Out-of-range expert ids are not checked on the device.
 */
int moe_permute(const int32_t* topk_ids, int64_t T, int k, int E,
                int32_t* offsets, int32_t* perm_to_flat, int32_t* flat_to_perm,
                void* ws, size_t ws_bytes, void* stream);

/*
 * moe_permute_static_ws -- moe_permute without a workspace argument. The
 * pages have no counterpart: this entry point serves callers that cannot
 * allocate device memory where they call it (for example inside another
 * framework's execution callback that forbids allocation, or on a path that
 * must not risk the device synchronisation an allocation can bring) and have
 * no workspace to pass. Results are identical to moe_permute's.
 *   Scratch: a fixed 1 MiB device array inside the library, which every GPU
 *   that loads the library holds until the process exits. It must fit
 *   ceil(T*k / 1024) * E int32 entries (<= 262144); larger requests return
 *   NVFP4MOE_ERR_WORKSPACE before anything is launched.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   All calls share the one array: calls whose kernels may overlap on the GPU
 *   (several streams, several host threads) race on it. Nothing in it has to
 *   start at zero; each call overwrites what it reads.
 *   The call itself allocates nothing.
 */
int moe_permute_static_ws(const int32_t* topk_ids, int64_t T, int k, int E,
                          int32_t* offsets, int32_t* perm_to_flat, int32_t* flat_to_perm,
                          void* stream);

/* Workspace bytes moe_quantize_dispatch needs. */
size_t moe_quantize_dispatch_workspace_size(int E);

/*
 * moe_quantize_dispatch -- stage 2: quantize each token row of x (T, K) once
 * and write it to the grouped-padded row of every one of its k routed slots:
 * slot f = t*k + j of expert e = topk_ids[f] goes to padded row
 * P_e + (flat_to_perm[f] - offsets[e]).
 *   gs_in / gs_out as in nvfp4_quantize (gs_in == NULL: gs = 2688 / amax(x),
 *   recomputed every call, CURRENT_BUG.md "What Works").
 *   a_codes  a_rows x K/2 bytes, a_sf NVFP4_SF_TILED_ROWS for (a_rows, K);
 *   a_rows >= nvfp4moe_padded_rows(T*k, E). Padding rows are not written.
 * K must be a multiple of 64.
 */
int moe_quantize_dispatch(const void* x, int64_t T, int64_t K, int64_t ldx, int k, int E,
                          const int32_t* topk_ids, const int32_t* offsets,
                          const int32_t* flat_to_perm, const float* gs_in, float* gs_out,
                          uint8_t* a_codes, uint8_t* a_sf, int64_t a_rows,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * nvfp4_grouped_gemm -- README "ScaledGroupedGemmKernel": A(M, K) x B(E, K, N)
 * -> C(M, N), block-scaled on both operands, per-expert global scales.
 *   A        grouped-padded NVFP4 activation: a_codes a_rows x K/2, a_sf
 *            NVFP4_SF_TILED_ROWS for (a_rows, K), global scale *gs_a.
 *   B        expert weights (E, N, K) as described above, gs_b[E].
 *   offsets  (E + 1) int32 group boundaries (compact rows).
 *   C        BF16, COMPACT rows: C[offsets[e] + i, n] =
 *            sum_k A[P_e + i, k] * B[e, n, k] / (gs_a * gs_b[e]), f32
 *            accumulation rounded once to BF16; leading dimension ldc.
 * Requires K % 64 == 0, N % 128 == 0, 1 <= E <= 1024, a_rows >=
 * nvfp4moe_padded_rows(offsets[E], E); 16-byte aligned pointers, ldc % 8 == 0.
 * C is written in whole 32-byte sectors when C is 32-byte aligned and
 * ldc % 16 == 0 (faster), else in 16-byte pieces.
 */
int nvfp4_grouped_gemm(const uint8_t* a_codes, const uint8_t* a_sf, const float* gs_a,
                       int64_t a_rows, const uint8_t* b_codes, const uint8_t* b_sf,
                       const float* gs_b, const int32_t* offsets, int E, int64_t N, int64_t K,
                       void* c, int64_t ldc, void* stream);

/*
 * nvfp4_grouped_gemm_swiglu -- stages 3 and 4: the L1 grouped GEMM with W1
 * (E, 2I, K) (gate/up rows interleaved at granularity 8), whose epilogue
 * scales by 1 / (gs_a * gs_w1[e]), forms h_i = silu(gate_i) * up_i in f32
 * (silu(g) = g / (1 + exp(-g))) and requantizes h to NVFP4 with the
 * pre-computed global scale *gs_h (README "Bridge Layer":
 * quantize_activation_nvfp4 with pre-computed gs; "Fused SwiGLU - Remaining
 * Steps" 2-4: quantize in the epilogue and store FP4 + scales straight into
 * the padded L2 input).
 *   h_codes  a_rows x I/2 bytes (32-byte aligned), h_sf NVFP4_SF_TILED_ROWS
 *            for (a_rows, I), in the same grouped-padded rows as A (padding
 *            rows are not written): the A operand of the L2 GEMM.
 * Requires I % 64 == 0, K % 64 == 0, 1 <= E <= 1024.
 */
int nvfp4_grouped_gemm_swiglu(const uint8_t* a_codes, const uint8_t* a_sf, const float* gs_a,
                              int64_t a_rows, const uint8_t* w1_codes, const uint8_t* w1_sf,
                              const float* gs_w1, const int32_t* offsets, int E, int64_t I,
                              int64_t K, const float* gs_h, uint8_t* h_codes, uint8_t* h_sf,
                              void* stream);

/*
 * nvfp4_rmsnorm_rope_quantize -- fused front end for attention projections
 * (README "THE PLAN", item 3: "Q norm -> RoPE -> NVFP4 quant", all in one
 * pass): per row of D elements
 *   y = x / sqrt(mean(x^2) + eps) * gamma            (f32),
 *   the last rope_dims elements rotated in adjacent pairs (2j, 2j+1) by the
 *   angle whose cosine / sine are cos_tab / sin_tab[positions[row], j],
 *   then y quantized to NVFP4 with the pre-computed global scale *gs.
 *   x          (rows, D) BF16, leading dimension ldx (16-byte aligned rows).
 *   gamma      D f32 (device, 16-byte aligned).  eps >= 0.
 *   positions  rows int32 (device), each in [0, max_pos); a position outside
 *              it gives that row all-zero codes and scales and records
 *              NVFP4MOE_ERR_INVALID in the device status word.
 *   cos_tab, sin_tab  (max_pos, rope_dims / 2) f32, row-major (device,
 *              16-byte aligned).
 *              With rope_dims == 0 positions and tables are not read.
 *   codes      (rows, D/2) bytes; sf in NVFP4_SF_ROWMAJOR, NVFP4_SF_TILED or
 *              NVFP4_SF_TILED_ROWS.
 *   y_out      NULL, or (rows, D) f32 that receives y (16-byte aligned).
 * Requires D % 16 == 0, rope_dims % 16 == 0, rope_dims <= D.
 */
int nvfp4_rmsnorm_rope_quantize(const void* x, int64_t rows, int64_t D, int64_t ldx,
                                const float* gamma, float eps, int64_t rope_dims,
                                const int32_t* positions, const float* cos_tab,
                                const float* sin_tab, int64_t max_pos, const float* gs,
                                uint8_t* codes, uint8_t* sf, int sf_layout, float* y_out,
                                void* stream);

/* Workspace bytes nvfp4_linear needs (the row bounds of its single group). */
size_t nvfp4_linear_workspace_size(void);

/*
 * nvfp4_linear -- one NVFP4 x NVFP4 linear with BF16 output, for shared
 * experts and projections (README "NVFP4 Linear": CuTeDSLNvfp4Linear, a
 * single-expert NVFP4 GEMM): C[m, n] = sum_k A[m, k] * W[n, k] / (gs_a * gs_w)
 * for m < M, f32 accumulation rounded once to BF16. It is the grouped GEMM
 * with one group, so it can run on its own stream beside the routed experts.
 *   A   a_rows x K/2 codes, row-major (nvfp4_quantize output), with
 *       a_rows >= 128 * ceil(M / 128) allocated rows (rows >= M are read and
 *       their products discarded), scales NVFP4_SF_TILED_ROWS for (a_rows, K),
 *       global scale *gs_a (device).
 *   W   N x K/2 codes, scales NVFP4_SF_TILED for (N, K), *gs_w (device).
 *   C   M x N BF16, leading dimension ldc (alignment as nvfp4_grouped_gemm).
 *   ws  >= nvfp4_linear_workspace_size() bytes, 16-byte aligned, device; it
 *       holds the group bounds and must not be shared by calls in flight.
 * Requires K % 64 == 0, N % 128 == 0. Errors as nvfp4_grouped_gemm, plus
 * WORKSPACE.
 */
int nvfp4_linear(const uint8_t* a_codes, const uint8_t* a_sf, const float* gs_a, int64_t M,
                 int64_t a_rows, const uint8_t* w_codes, const uint8_t* w_sf, const float* gs_w,
                 int64_t N, int64_t K, void* c, int64_t ldc, void* ws, size_t ws_bytes,
                 void* stream);

/*
 * moe_combine -- stage 6 (README "MoE Runner" step 6, scatter with routing
 * weights): y[t, :] = sum_{j<k} topk_w[t, j] * out[flat_to_perm[t*k + j], :],
 * summed in f32 in j order and rounded once to BF16.
 *   out (T*k, K) BF16 compact rows, leading dimension ldo; y (T, K) BF16,
 *   leading dimension ldy. K % 8 == 0, ldo % 8 == 0, ldy % 8 == 0.
 */
int moe_combine(const void* out, int64_t ldo, const float* topk_w,
                const int32_t* flat_to_perm, int64_t T, int k, int64_t K,
                void* y, int64_t ldy, void* stream);

/* Workspace bytes moe_forward needs. */
size_t moe_forward_workspace_size(int64_t T, int64_t K, int64_t I, int E, int k);

/* Byte offsets inside the moe_forward workspace of its intermediates, written
 * to offs_host[0..11] in this order: topk_ids, topk_w, offsets, perm_to_flat,
 * flat_to_perm, gs_x, a_codes, a_sf, h_codes, h_sf, out, a_rows (the last one
 * is the row capacity, not an offset). Host only; for inspection and tests. */
int moe_forward_workspace_layout(int64_t T, int64_t K, int64_t I, int E, int k,
                                 int64_t* offs_host);

/*
 * moe_forward -- the whole expert forward (README "MoE Runner" steps 1-6 with
 * the fused L1 of "Fused SwiGLU"):
 *   x              (T, K) BF16, leading dimension K.
 *   router_logits  (T, E) f32.
 *   w1_*           (E, 2I, K) NVFP4, gate/up interleaved, tiled scales,
 *                  gs_w1[E].
 *   w2_*           (E, K, I) NVFP4 (reduction over I), tiled scales, gs_w2[E].
 *   gs_h           device f32, the pre-computed global scale of h.
 *   y              (T, K) BF16 output.
 *   ws             >= moe_forward_workspace_size(T, K, I, E, k) bytes,
 *                  256-byte aligned.
 * Requires K % 128 == 0, I % 64 == 0, 1 <= k <= 16, k <= E <= 1024, T >= 0.
 * Stages 1-2 run as moe_dispatch (the fused front) when
 * moe_forward_uses_fused_dispatch(T, E, k), else as moe_route_topk,
 * moe_permute and moe_quantize_dispatch; the intermediates are the same bit
 * for bit. Then the
 * L1+SwiGLU+requant, L2 and combine kernels. Everything is enqueued on
 * `stream` without any host synchronisation, so the call can be captured in
 * a CUDA graph.
 */
int moe_forward(const void* x, const float* router_logits, int64_t T, int64_t K, int64_t I,
                int E, int k, const uint8_t* w1_codes, const uint8_t* w1_sf,
                const float* gs_w1, const uint8_t* w2_codes, const uint8_t* w2_sf,
                const float* gs_w2, const float* gs_h, void* y, void* ws, size_t ws_bytes,
                void* stream);

/* Workspace bytes moe_dispatch_static and moe_dispatch need (T >= 1). */
size_t moe_dispatch_static_workspace_size(int64_t T, int E);

/*
 * moe_dispatch_static -- stages 1 and 2 fused, with a pre-computed activation
 * global scale *gs_x (README "Bridge Layer": quantize_activation_nvfp4 with
 * pre-computed gs; "MoE Runner" steps 1-2): moe_route_topk, moe_permute and
 * moe_quantize_dispatch (with gs_in = gs_x) in one cooperative kernel with
 * two grid-wide barriers, each bounded by the wait limit (a timeout sets the
 * device status; offsets and flat_to_perm are then all zero, so every slot's
 * codes land in padded row 0). Above NVFP4MOE_FRONT_FUSED_QUANTIZE_MAX_ROWS
 * routed rows the cooperative kernel stops after the permutation and a
 * second kernel does the quantize + scatter (the same bits).
 * Outputs as those three calls: topk_ids / topk_w (T, k); offsets (E + 1);
 * perm_to_flat / flat_to_perm (T*k); a_codes / a_sf in the grouped-padded
 * rows of (a_rows, K) with a_rows >= nvfp4moe_padded_rows(T*k, E).
 * ws >= moe_dispatch_static_workspace_size(T, E) bytes, 256-byte aligned.
 * Requires K % 64 == 0, 1 <= k <= 16, k <= E <= 1024, and T * k <= 4096 * G
 * (G = co-resident blocks of the kernel, at least one per SM).
 */
int moe_dispatch_static(const void* x, int64_t ldx, const float* router_logits, int64_t T,
                        int64_t K, int E, int k, const float* gs_x, int32_t* topk_ids,
                        float* topk_w, int32_t* offsets, int32_t* perm_to_flat,
                        int32_t* flat_to_perm, uint8_t* a_codes, uint8_t* a_sf, int64_t a_rows,
                        void* ws, size_t ws_bytes, void* stream);

/* 1 if T tokens at top-k over E experts fit the co-resident blocks of the
 * fused dispatch kernel (moe_dispatch, moe_dispatch_static), else 0. Host
 * only (queries the device's occupancy). */
int moe_dispatch_supported(int64_t T, int E, int k);

/* 1 if moe_forward runs stages 1-2 as moe_dispatch for this shape: whenever
 * moe_dispatch_supported, else 0 (the separate moe_route_topk, moe_permute
 * and moe_quantize_dispatch). Host only. */
int moe_forward_uses_fused_dispatch(int64_t T, int E, int k);

/*
 * moe_dispatch -- moe_dispatch_static with the activation global scale
 * computed in the same kernel (README "Bridge Layer": quantize_activation_nvfp4;
 * CURRENT_BUG "What Works": recomputed every call): max |x| over all T tokens
 * before the first grid barrier, gs = 2688 / max|x| (1 for an all-zero x)
 * after it, written to *gs_out (device f32). Outputs, workspace
 * (moe_dispatch_static_workspace_size) and requirements as
 * moe_dispatch_static; the same bits as moe_route_topk + moe_permute +
 * moe_quantize_dispatch with gs_in = NULL.
 */
int moe_dispatch(const void* x, int64_t ldx, const float* router_logits, int64_t T, int64_t K,
                 int E, int k, float* gs_out, int32_t* topk_ids, float* topk_w, int32_t* offsets,
                 int32_t* perm_to_flat, int32_t* flat_to_perm, uint8_t* a_codes, uint8_t* a_sf,
                 int64_t a_rows, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_forward_static -- moe_forward with a pre-computed activation global
 * scale (README "Bridge Layer": quantize_activation_nvfp4, the CUDA-graph-safe
 * quantizer with a pre-computed gs; "CUDAGraph-safe": workspace pre-allocated,
 * no runtime allocation): moe_dispatch_static (routing, permutation,
 * quantization and scatter as one kernel), then the L1, L2 and combine
 * kernels of moe_forward.
 *   gs_x  device f32: the global scale x is quantized with (codes and scales
 *         as nvfp4_quantize with gs_in = gs_x). Values of |x| * gs_x beyond
 *         the E4M3 x E2M1 range saturate.
 * Other arguments, workspace and layout as moe_forward; the intermediates sit
 * at the same workspace offsets (the gs_x slot is not written). Also needs
 * T * k <= 4096 * G, G the co-resident blocks of the front kernel (at least
 * one per SM: 77 824 tokens at k = 8 on 152 SMs); UNSUPPORTED beyond.
 */
int moe_forward_static(const void* x, const float* router_logits, int64_t T, int64_t K, int64_t I,
                       int E, int k, const float* gs_x, const uint8_t* w1_codes,
                       const uint8_t* w1_sf, const float* gs_w1, const uint8_t* w2_codes,
                       const uint8_t* w2_sf, const float* gs_w2, const float* gs_h, void* y,
                       void* ws, size_t ws_bytes, void* stream);

/* Waits for `stream`, then reads and clears the device status word that the
 * GEMM and fused-front kernels set when a bounded wait runs out (and
 * nvfp4_rmsnorm_rope_quantize sets on a position out of range) (README "Key Lessons" 5: no
 * silent failure). Returns NVFP4MOE_OK, NVFP4MOE_ERR_DEVICE_TIMEOUT or
 * NVFP4MOE_ERR_LAUNCH (a CUDA error on the stream). */
int nvfp4moe_last_device_status(void* stream);

/* Test hook: the wait limit of the GEMM kernels' bounded waits, in
 * nanoseconds (default 4e9). Host only; affects launches made afterwards. */
void nvfp4moe_set_wait_limit_ns(uint64_t ns);

/* Test hook for the failure path: while set (non-zero), the MMA-issuing
 * thread of every GEMM CTA that has work first waits on a barrier that
 * nothing arrives on, so that bounded wait runs out after the wait limit and
 * the kernel takes its abort path; and block 0 of the fused front
 * (moe_forward_static) leaves before its first grid barrier, so the other
 * blocks' bounded barrier waits run out. Host only; affects launches made
 * afterwards. */
void nvfp4moe_set_test_stall(int on);

/* Which grouped-GEMM kernel the GEMM entry points launch (host only; affects
 * launches made afterwards). 0 (default): one CTA per tile of 128 activation
 * rows x 256 weight rows. 1: a tile of 256 activation rows x 256 weight rows
 * on a pair of SMs (a thread-block cluster of two CTAs sharing one 2-SM
 * tcgen05 MMA, each CTA loading its 128 activation rows and half of the
 * weight tile) whenever N % 256 == 0, else one CTA per tile. Both give the
 * same results bit for bit; on this GB300 the pairs measured slower (their
 * cross-SM hand-offs lengthen the load round trip that bounds both kernels),
 * so they are not the default. Returns NVFP4MOE_OK or NVFP4MOE_ERR_INVALID. */
int nvfp4moe_set_gemm_mode(int mode);

/* Number of streaming multiprocessors of the current device (grid size of the
 * persistent GEMM kernels). Host only. */
int nvfp4moe_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4MOE_H */
