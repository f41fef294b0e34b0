/*
 * gq.h -- C ABI of the grouped FP8 quantizer and grouped expert GEMMs for
 * MoE training on GB300 (sm_103a).
 *
 * The hot path has two parts:
 *   1. gq_quantize: a bf16 token buffer partitioned by split_sizes is cast to
 *      FP8 e4m3 with per-block scales, rowwise and/or columnwise.  Recipes:
 *      MXFP8 1x32 with E8M0 scales in the swizzled
 *      [outer/128][inner/128][32][4][4] layout (TransformerEngine issue 3484,
 *      "Describe the bug"; TransformerEngine PR 3224, the group_quantize_mxfp8
 *      fix), a per-channel 128-row fp32-scale recipe (DeepGEMM issue 365,
 *      _per_channel_cast_to_fp8), and NVFP4 (E2M1 codes, 16-element E4M3
 *      scales and a per-group fp32 scale; see GQ_RECIPE_NVFP4_1X16).
 *   2. gq_gemm_fprop / gq_gemm_dgrad / gq_gemm_wgrad: grouped GEMMs that
 *      consume those operands; the wgrad contracts only over each group's
 *      live rows (TransformerEngine issue 3484, "Additional context: Scope").
 *      Fused variants: gq_gemm_fprop_bias, gq_quantize_dbias,
 *      gq_gemm_fprop_srelu_quant and gq_gemm_fprop_swiglu_quant.
 * gq_check_wait_limit is a diagnostic: it runs the kernels' bounded-wait
 * failure path (GQ_ERR_TIMEOUT) without a fault.
 *
 * Conventions shared by every call
 *  - Pointers named d_* and every buffer inside gq_quantized are DEVICE
 *    pointers; descriptor structs themselves live in HOST memory.  The caller
 *    owns all memory; the library allocates no device memory.
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream) and never synchronises with the host, so a sequence of calls
 *    can be captured in a CUDA graph once each (device, shape) pair has been
 *    called once outside capture.  That first call's set-up (kernel
 *    attributes) is cached per CUDA context: after cudaDeviceReset, or in
 *    another context, the next call redoes it, and it too must come before
 *    any capture.
 *  - Buffers are row-major.  A token buffer has rows_cap rows R; group g
 *    owns rows [o_g, o_g + m_g) with o_g = m_0 + ... + m_{g-1} and
 *    L = sum(m_g) <= R.  Rows >= L are padding: never read, never written,
 *    and their content (zeros, garbage, NaN) never affects any result.
 *  - split sizes: `d_split_sizes` is a device int32[num_groups]; NULL means
 *    the uniform split m_g = rows_cap / num_groups (rows_cap must divide;
 *    this is the single-grouped-weight case of TransformerEngine PR 3224).
 *    MX needs every m_g % 32 == 0, the per-channel recipe m_g % 128 == 0;
 *    all column counts must be multiples of 128.  1 <= num_groups <= 1024;
 *    0 <= rows_cap < 2^31 (a buffer may hold more than 2^31 elements).
 *  - Errors found on the host are returned synchronously and launch nothing.
 *    Errors found on the device (split sizes: negative, misaligned, or
 *    summing past rows_cap; a pipeline wait that timed out) are written to
 *    *d_status (first error wins) and the kernel leaves its outputs
 *    untouched.  Every kernel of every call first reads *d_status and does
 *    nothing when it is nonzero, so one bad split table turns the rest of a
 *    stream-ordered sequence into no-ops (the noop-flag semantics of
 *    TransformerEngine PR 3224's group_quantize).  The caller zeroes
 *    *d_status before a sequence and reads it afterwards.
 *  - L == 0 (every group empty) dereferences no data pointer (PR 3224's
 *    zero-row guard); the wgrad with accumulate == 0 still writes zeros.
 */
#ifndef GQ_H_
#define GQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t. */
typedef struct CUstream_st* gq_stream_t;

typedef enum gq_status {
    GQ_OK = 0,
    GQ_ERR_INVALID_ARG = -1,    /* null pointer, bad count, capacity too small */
    GQ_ERR_ALIGNMENT = -2,      /* cols % 128, rows_cap % num_groups, pointer alignment */
    GQ_ERR_SPLITS = -3,         /* (device) a split is negative, misaligned, or they overflow rows_cap */
    GQ_ERR_UNSUPPORTED = -4,    /* recipe / orientation / dtype combination not provided */
    GQ_ERR_CUDA = -5,           /* a CUDA runtime call or launch failed */
    GQ_ERR_TIMEOUT = -6,        /* (device) a pipeline wait gave up; outputs are undefined */
    GQ_ERR_SHAPE_MISMATCH = -7  /* descriptor disagrees with the call (groups, rows, cols, recipe) */
} gq_status;

typedef enum gq_recipe_kind {
    /* MXFP8 1x32: one E8M0 scale 2^e per 32 elements, e = floor(log2 amax) - 8
     * clamped to [-127, 127] (an all-zero block gets e = -127, byte 0);
     * codes = e4m3(x * 2^-e), nearest-even, saturating to +-448. */
    GQ_RECIPE_MXFP8_1X32 = 0,
    /* Per-channel 128-row fp32 scale (columnwise only), computed op by op in
     * fp32: sf = amax / 448; sf == 0 -> zero_scale; sf = max(sf, 1e-30);
     * codes = e4m3(x * (1 / sf)). */
    GQ_RECIPE_CHANNEL128_F32 = 1,
    /* NVFP4: FP4 E2M1 codes with one E4M3 scale per 16 elements along the
     * contraction axis and one fp32 second-level scale per group.
     * TransformerEngine PR 3224 names NVFP4 beside MXFP8 on the grouped paths
     * without defining it; this is the public NVFP4 format.  Per group
     * g: amax_g = max |x| over its live rows, S_g = 2688 / amax_g (1 when
     * amax_g == 0, clamped to FLT_MAX).  Per block, in fp32 op by op:
     * s = (amax_b / 6) * S_g, sf = e4m3(s) (nearest-even, saturating),
     * m = S_g / sf (0 when sf == 0, clamped to FLT_MAX), codes =
     * e2m1(x * m) (nearest-even, saturating to +-6).  A code stands for
     * e2m1 * sf / S_g. */
    GQ_RECIPE_NVFP4_1X16 = 2
} gq_recipe_kind;

typedef enum gq_dtype { GQ_DTYPE_F32 = 0, GQ_DTYPE_BF16 = 1 } gq_dtype;

typedef struct gq_recipe {
    int32_t kind;        /* gq_recipe_kind */
    int32_t rowwise;     /* 1: produce rowwise codes + scales (MX and NVFP4; the
                            per-channel recipe is columnwise only) */
    int32_t colwise;     /* 1: produce columnwise codes + scales */
    float zero_scale;    /* per-channel recipe: the scale of an all-zero block (the
                            page's sf_val); ignored by MX */
} gq_recipe;

/*
 * A grouped quantised tensor (the GroupedTensor of TransformerEngine PR
 * 3224), described by the caller and reusable across calls.
 *
 *  row_data / col_data : uint8 e4m3 codes, [rows_cap, cols] row-major.  Both
 *      orientations keep the buffer's orientation: columnwise codes of row r
 *      are stored in row r.  Only rows < L are written.
 *  row_scale (MX) : uint8 E8M0 bytes.  Group g's region starts at byte
 *      512 * (cols/128) * (T_0 + ... + T_{g-1}), T_h = ceil(m_h / 128), and
 *      holds T_g * (cols/128) atoms of 512 bytes ordered [row tile][col tile].
 *  col_scale (MX) : same region offsets; atoms ordered [col tile][row tile]:
 *      the row (m) tile is the inner stride and its extent is the group's own
 *      T_g, never the buffer's (TransformerEngine issue 3484).
 *      Inside an atom, the scale of (row r of a 128-row tile, scale column j
 *      of 4) -- for columnwise scales (channel r of a 128-channel tile,
 *      32-row block j of 4) -- is byte (r % 32) * 16 + (r / 32) * 4 + j.
 *      Entries of a group's last tile that cover no live row are 0.
 *  col_scale (per-channel) : fp32 [L/128][cols]: the scale of live rows
 *      [128 b, 128 b + 128) of channel c is element b * cols + c.
 *  NVFP4 : two E2M1 codes a byte, the element with the even index in the low
 *      nibble.  row_data is [rows_cap, cols/2]; col_data is stored
 *      TRANSPOSED, [cols, rows_cap/2] (row c holds column c's codes in blocks
 *      of 16 rows), so that every GEMM operand has its contraction axis
 *      contiguous (the tensor core takes packed 4-bit operands K-major only);
 *      columnwise quantisation needs rows_cap % 32 == 0.  Scale bytes (E4M3)
 *      use the same 512-byte atom with 16 elements a scale, so an atom
 *      covers 128 rows (channels) x 64 elements; group g's region starts at
 *      512 * (cols/64) * (T_0 + ... + T_{g-1}) in both orientations; rowwise
 *      atoms are ordered [128-row tile][64-column block], columnwise atoms
 *      [128-column tile][64-row block] (2 T_g inner).  Byte of (row r,
 *      16-column block j) -- columnwise (channel r, 16-row block j) -- inside
 *      an atom: (r % 32) * 16 + (r / 32) * 4 + j % 4.
 *  amax (NVFP4 only) : device fp32 [num_groups], the per-group amax the
 *      quantiser wrote (4-byte aligned); the GEMMs read it to undo S_g.
 *  *_scale_bytes : capacity in bytes of each scale buffer (checked).
 *
 * Device buffers must be 16-byte aligned.
 */
typedef struct gq_quantized {
    int32_t num_groups;
    int32_t reserved0;
    int64_t rows_cap;
    int64_t cols;
    gq_recipe recipe;
    void* row_data;
    void* row_scale;
    void* col_data;
    void* col_scale;
    uint64_t row_scale_bytes;
    uint64_t col_scale_bytes;
    float* amax;
} gq_quantized;

/* Human-readable name of a status code (static storage). */
const char* gq_status_string(int32_t status);

/* ABI version, (major << 16) | minor. */
int32_t gq_version(void);

/* Bytes a scale buffer needs for any split table of num_groups groups over
 * rows_cap rows: MX 512 * (cols/128) * (ceil(rows_cap/128) + num_groups);
 * NVFP4 512 * (cols/64) * (ceil(rows_cap/128) + num_groups); per-channel
 * 4 * cols * (rows_cap / 128).  0 on a bad argument. */
uint64_t gq_scale_bytes_bound(const gq_recipe* recipe, int32_t num_groups, int64_t rows_cap,
                              int64_t cols);

/*
 * gq_split_scan -- the partition of a token buffer by split sizes
 * (DeepGEMM issue 365, grouped_layout; TransformerEngine PR 3224, the m_splits
 * alignment contract).  Writes d_table (device int64[3 * (num_groups + 1)]):
 *   d_table[g]                     = o_g, the first row of group g (g = G: L)
 *   d_table[(G + 1) + g]           = T_0 + ... + T_{g-1}, T_h = ceil(m_h / 128)
 *   d_table[2 (G + 1) + g]         = byte offset of group g's scale region
 *                                    (MX: 512 (cols/128) sum T; NVFP4:
 *                                    512 (cols/64) sum T; per-channel:
 *                                    4 cols o_g / 128)
 * Split errors go to *d_status and leave d_table untouched.  Every other
 * call performs this scan inside its own kernels; this entry point exposes
 * it for callers that size or inspect buffers.
 */
gq_status gq_split_scan(const int32_t* d_split_sizes, int32_t num_groups, int64_t rows_cap,
                        int64_t cols, int32_t recipe_kind, int64_t* d_table, int32_t* d_status,
                        gq_stream_t stream);

/*
 * gq_quantize -- grouped quantisation of x_bf16 ([rows_cap, cols] bf16,
 * device) into the caller-described `out` (TransformerEngine PR 3224: output
 * reuse with num_tensors / logical-shape validation).
 *   out->num_groups, rows_cap, cols and recipe.kind must equal the call's
 *   (else GQ_ERR_SHAPE_MISMATCH); the orientations requested by `recipe`
 *   must have non-null buffers whose scale capacity is at least
 *   gq_scale_bytes_bound (else GQ_ERR_INVALID_ARG).  out->recipe is
 *   overwritten with *recipe.
 * Reads rows < L of x only; writes codes of rows < L and the grouped scale
 * regions (bytes past the last group's region are untouched).
 * NVFP4 runs three kernels: the split scan with amax[g] = 0, the per-group
 * amax over the live rows, then the codes and scales; out->amax must be set.
 */
gq_status gq_quantize(const void* x_bf16, int64_t rows_cap, int64_t cols,
                      const int32_t* d_split_sizes, int32_t num_groups, const gq_recipe* recipe,
                      gq_quantized* out, int32_t* d_status, gq_stream_t stream);

/*
 * gq_quantize_dbias -- gq_quantize (MX recipe) of an output gradient dY
 * fused with its bias gradient, the per-group dbiases that the grouped
 * linear's backward returns beside dinput and dweights (TransformerEngine
 * PR 3224, sequence diagram):
 *   d_dbias[g, c] = sum of dY[r, c] over the live rows r of group g
 * The quantiser sums each 128 x 128 tile's columns while it has them in
 * registers (one fp32 sum per column, in a fixed order) and writes them to
 * d_workspace; a second small kernel adds each group's tile sums in tile
 * order, so the result is the same on every call.
 *   d_dbias     : fp32 [num_groups, cols], 16-byte aligned; empty groups
 *                 (and L == 0) get 0.
 *   d_workspace : caller-owned device memory of at least
 *                 gq_dbias_workspace_bytes(num_groups, rows_cap, cols) bytes,
 *                 16-byte aligned; its content on entry does not matter.
 * Everything else as gq_quantize; GQ_ERR_UNSUPPORTED for the per-channel
 * recipe.
 */
uint64_t gq_dbias_workspace_bytes(int32_t num_groups, int64_t rows_cap, int64_t cols);
gq_status gq_quantize_dbias(const void* x_bf16, int64_t rows_cap, int64_t cols,
                            const int32_t* d_split_sizes, int32_t num_groups, const gq_recipe* recipe,
                            gq_quantized* out, float* d_dbias, void* d_workspace, uint64_t workspace_bytes,
                            int32_t* d_status, gq_stream_t stream);

/*
 * gq_gemm_fprop -- Y_g = X_g W_g^T for every group g (TransformerEngine PR
 * 3224, general_grouped_gemm_for_grouped_tensor in the forward sequence).
 *   x : MX rowwise, rows_cap R, cols k, split by d_split_sizes.
 *   w : MX rowwise, rows_cap num_groups * n, cols k, uniform split (W_g is
 *       rows [g n, g n + n)).
 *   y : [R, n] of out_dtype (GQ_DTYPE_F32 or GQ_DTYPE_BF16, nearest-even);
 *       rows < L written, rows >= L untouched.
 * n and k must be multiples of 128.
 * NVFP4 operands (x and w both NVFP4 rowwise): n and k must be multiples of
 * 256; the fp32 accumulator of the block-scaled MMAs is multiplied by
 * 1 / (S_x,g S_w,g) before the conversion.  Bias and the fused activation
 * take MX operands only.
 */
gq_status gq_gemm_fprop(const gq_quantized* x, const gq_quantized* w,
                        const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                        void* y, int32_t out_dtype, int32_t* d_status, gq_stream_t stream);

/*
 * gq_gemm_fprop_bias -- Y_g = X_g W_g^T + b_g: gq_gemm_fprop with the
 * grouped bias add that TransformerEngine PR 3224 runs after the grouped
 * GEMM (launch_grouped_bias_add in its forward sequence diagram), fused into
 * the GEMM's epilogue: the bias is added to the fp32 accumulator before the
 * conversion to out_dtype, so Y is written once.
 *   d_bias : [num_groups, n] device array of bias_dtype (GQ_DTYPE_F32 or
 *            GQ_DTYPE_BF16), 16-byte aligned; row g is added to every live
 *            row of group g.  Empty groups and L == 0 touch nothing (the
 *            page's zero-row guard).
 * Everything else as gq_gemm_fprop.
 */
gq_status gq_gemm_fprop_bias(const gq_quantized* x, const gq_quantized* w,
                             const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                             const void* d_bias, int32_t bias_dtype, void* y, int32_t out_dtype,
                             int32_t* d_status, gq_stream_t stream);

/*
 * gq_gemm_fprop_srelu_quant -- the fc1 forward with the activation and the
 * quantisation of fc2's input fused into the GEMM's epilogue: Y_g = X_g W_g^T
 * (+ b_g), and the MXFP8 rowwise and columnwise quantisation of
 *   A[r, c] = probs[r] * relu(Y[r, c])^2
 * computed from the fp32 accumulator (t = max(y, 0); t = t * t; a = t * p,
 * fp32 op by op), so A never exists in bf16 or in HBM.  This is the fc1 ->
 * ScaledSReLU -> fc2 sequence of TransformerEngine issue 3484's reproducer
 * (te.ops.ScaledSReLU fed with per-token probs); the pages name the
 * activation without printing it, and squared ReLU times the row's prob is
 * the plain reading.
 *   d_bias  : NULL, or as gq_gemm_fprop_bias (added before the activation).
 *   d_probs : fp32 [R] device array, 16-byte aligned (only rows < L read).
 *   y       : [R, n] of out_dtype, the pre-activation result (what the
 *             activation's backward needs), as gq_gemm_fprop.
 *   act_out : an MX descriptor with rowwise and colwise buffers, num_groups,
 *             rows_cap = x's rows_cap, cols = n; filled exactly as
 *             gq_quantize would fill it from A (same scale rule, codes,
 *             swizzled grouped atoms, zero entries past each group's end).
 * n must be a multiple of 256 (GQ_ERR_UNSUPPORTED otherwise).
 */
gq_status gq_gemm_fprop_srelu_quant(const gq_quantized* x, const gq_quantized* w,
                                    const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                                    const void* d_bias, int32_t bias_dtype, const float* d_probs, void* y,
                                    int32_t out_dtype, gq_quantized* act_out, int32_t* d_status,
                                    gq_stream_t stream);

/*
 * gq_gemm_fprop_swiglu_quant -- gq_gemm_fprop_srelu_quant with ScaledSwiGLU,
 * another activation TransformerEngine issue 3484 names without defining
 * (ScaledSwiGLU, beside ScaledClampedQGeGLU and ScaledSiTUGLU in its
 * 'Additional context').  Reading: the SwiGLU of "GLU Variants Improve
 * Transformer" scaled by the row's prob.  The fc1 output Y (width n) is split
 * into a gate half Y[:, 0:n/2] and a linear half Y[:, n/2:n] (W_g's rows in
 * the same order), and
 *   A[r, c] = (silu(Y[r, c]) * Y[r, n/2 + c]) * probs[r],
 *   silu(x) = x / (1 + exp(-x)),
 * fp32 op by op, with this library's own exp: argument clamped to [-87, 88],
 * Cody-Waite reduction by ln 2 (n = rint(x * log2(e)); r = x - n * ln2_hi -
 * n * ln2_lo, ln2_hi = 0x1.62e4p-1, ln2_lo = 0x1.7f7d1cp-20), the degree-7
 * Taylor polynomial of exp(r) in Horner form with fused multiply-adds, an
 * exact scaling by 2^n.  A is MX-quantised rowwise and columnwise into
 * act_out exactly as gq_quantize would quantise it.
 *   y       : [R, n] of out_dtype, the pre-activation result (both halves).
 *   act_out : MX rowwise + colwise, num_groups, rows_cap = x's rows_cap,
 *             cols = n / 2.
 * n must be a multiple of 256 (GQ_ERR_UNSUPPORTED otherwise); everything
 * else as gq_gemm_fprop_srelu_quant.
 */
gq_status gq_gemm_fprop_swiglu_quant(const gq_quantized* x, const gq_quantized* w,
                                     const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                                     const void* d_bias, int32_t bias_dtype, const float* d_probs, void* y,
                                     int32_t out_dtype, gq_quantized* act_out, int32_t* d_status,
                                     gq_stream_t stream);

/*
 * gq_gemm_dgrad -- dX_g = dY_g W_g (TransformerEngine issue 3484: M is a
 * free dimension of the dgrad).
 *   dy : MX rowwise, rows_cap R, cols n.
 *   w  : MX columnwise (32-row blocks along n, group-local layout), rows_cap
 *        num_groups * n, cols k.
 *   dx : [R, k] of out_dtype; rows < L written.
 * NVFP4: dy NVFP4 rowwise and w NVFP4 columnwise (stored [k, G n/2]); n and
 * k multiples of 256.
 */
gq_status gq_gemm_dgrad(const gq_quantized* dy, const gq_quantized* w,
                        const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                        void* dx, int32_t out_dtype, int32_t* d_status, gq_stream_t stream);

/*
 * gq_gemm_wgrad -- k-grouped weight gradient
 *   dW_g = (accumulate ? dW_g : 0) + dY_g^T X_g
 * contracting over group g's live rows only (TransformerEngine issue 3484;
 * DeepGEMM issue 365, k_grouped_fp8_gemm_nt_contiguous with recipe (1,1,128)).
 *   dy, x : both MX columnwise, both NVFP4 columnwise (k a multiple of 256;
 *           a group's last 64-row block may be half live: the scales of its
 *           dead 16-row blocks are 0), or both per-channel; rows_cap R; cols
 *           n and k.
 *   dw    : fp32 [num_groups, n, k].  accumulate = 1 adds into it (the
 *           accumulate_into_main_grad of TransformerEngine issue 3484); an
 *           empty group then leaves dW_g bit-unchanged, with accumulate = 0
 *           it writes +0.0.
 *   d_workspace : NULL, or caller-owned device memory of at least
 *           GQ_WGRAD_WORKSPACE_BYTES bytes, 16-byte aligned, that the call
 *           clears on `stream` before its kernel (cudaMemsetAsync) and uses
 *           as tile-claim counters.  With a workspace the MX wgrad hands out
 *           its output tiles at run time: 40% of the CTAs take tiles of the
 *           groups in decreasing order of m_g, the others in increasing
 *           order, until the two meet, so the long contractions of the
 *           largest groups overlap the main-grad traffic of the smallest
 *           (with skewed splits every CTA would otherwise work through the
 *           same group at the same time).  NULL keeps a static round-robin
 *           order.  Two calls that may run at the same time must not share a
 *           workspace.  The per-channel and NVFP4 recipes ignore it.
 *   workspace_bytes : size of d_workspace (ignored when it is NULL).
 * Deterministic: every output element is produced by one CTA in a fixed
 * order of additions, whichever CTA that is; repeated calls, with or without
 * a workspace, give bitwise identical results.
 */
#define GQ_WGRAD_WORKSPACE_BYTES 256
gq_status gq_gemm_wgrad(const gq_quantized* dy, const gq_quantized* x,
                        const int32_t* d_split_sizes, int32_t num_groups, int64_t n, int64_t k,
                        float* dw, int32_t accumulate, void* d_workspace, uint64_t workspace_bytes,
                        int32_t* d_status, gq_stream_t stream);

/*
 * gq_gemm_wgrad_noalloc -- gq_gemm_wgrad with the run-time tile order, for
 * callers that cannot supply a workspace.  The pages describe no such call:
 * it exists for hosts that have no device allocator of their own (a C or
 * Fortran program linking only this library) or that must not allocate on
 * this path (a cudaMalloc can wait for the whole device to go idle, and
 * memory pools owned by a framework may not be reachable from here).
 *
 * It allocates nothing.  The workspace is a GQ_WGRAD_WORKSPACE_BYTES-byte
 * array inside the library, one per device, held by every device that loads
 * the library until the process exits.  The first call in a CUDA context
 * looks up that array's device address there (cudaGetSymbolAddress, with the
 * context current; if no context is current yet, this makes the device's
 * primary context current, as any runtime call does) and keeps it, keyed by
 * the driver's context ID, which is never reused within a process.  So any
 * number of devices is served, and after cudaDeviceReset (a new context) the
 * next call looks the address up again.  Make the first call in each context
 * before any stream capture.  Each call clears the array's claim counter on
 * `stream` before its kernel.  All calls on a device share the one array, so
 * calls that may overlap on the GPU (on different streams without ordering
 * between them) race and must not be issued; serialise them, or use
 * gq_gemm_wgrad with one workspace per stream.
 *
 * Arguments, layouts, results and errors are those of gq_gemm_wgrad.  In
 * addition, a problem of 2^31 or more output tiles (num_groups * n/128 *
 * k/256, or k/128 when k % 256 != 0 -- the tiles the kernel itself runs)
 * exceeds the counter and returns GQ_ERR_INVALID_ARG before anything is
 * launched; GQ_ERR_CUDA when the set-up above fails.
 */
gq_status gq_gemm_wgrad_noalloc(const gq_quantized* dy, const gq_quantized* x,
                                const int32_t* d_split_sizes, int32_t num_groups, int64_t n,
                                int64_t k, float* dw, int32_t accumulate, int32_t* d_status,
                                gq_stream_t stream);

/*
 * gq_check_wait_limit -- a diagnostic of the library's failure path; the
 * pages describe no such call.  Every pipeline wait in the library's kernels
 * (an mbarrier phase: a TMA copy landing, a stage being freed, an
 * accumulator being handed over) gives up after 2 s of device time, records
 * GQ_ERR_TIMEOUT in *d_status (first error wins) and winds its CTA down:
 * the other roles see a shared abort flag, in-flight copies are waited for
 * (again bounded), tensor memory is freed, and the kernel returns.  This
 * call runs that path on purpose, without a fault: one CTA of two warps
 * waits on an mbarrier that nothing arrives on, until the limit passes.
 *
 *   d_status : device int32, 4-byte aligned, required.  Holds GQ_ERR_TIMEOUT
 *              afterwards when it held 0 before; when it was already nonzero
 *              the kernel does nothing (the noop flag).
 *   d_report : NULL, or device uint64[4], 8-byte aligned: for warp w = 0, 1,
 *              d_report[2w] = nanoseconds it waited (%globaltimer) and
 *              d_report[2w + 1] = 1 if the barrier's phase completed, else 0
 *              (it never completes).  Untouched by the noop path.
 * Asynchronous on `stream`; the kernel runs for about the wait limit (2 s)
 * and leaves the CUDA context usable.  Returns GQ_ERR_INVALID_ARG for a NULL
 * d_status, GQ_ERR_ALIGNMENT for a misaligned pointer, GQ_ERR_CUDA when the
 * launch fails.
 */
gq_status gq_check_wait_limit(int32_t* d_status, uint64_t* d_report, gq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GQ_H_ */
