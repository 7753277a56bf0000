/*
 * te_gb300.h -- C ABI of the fused normalization + feed-forward block for GB300 (sm_103a).
 *
 * The block is the one described by three TransformerEngine JAX pages:
 *   "Activation"       (activation(x, activation_type, quantizer, act_params)),
 *   "LayerNorm MLP"    (layernorm_mlp(x, gamma, beta, kernels, biases, norm_type, ...)),
 *   "LayerNorm Dense"  (layernorm_dense(x, kernel, gamma, beta, bias, norm_type, ...)).
 * Each entry point below names the page section that defines its operation.
 *
 * Conventions shared by every function:
 *   - Pointers are device pointers unless a comment says "host".  Every tensor is dense and
 *     row-major; leading batch/sequence dimensions are flattened into M rows (so the pages'
 *     transpose_batch_sequence flag has no counterpart).  Weights are stored [in, out], e.g.
 *     kernel1 is [H, F] (or [H, 2F] for a gated activation).
 *   - Device pointers must be 16-byte aligned.  Row lengths (H, N, F) must be multiples of 16
 *     elements for GEMM-carrying calls and multiples of 8 for the bandwidth-bound calls;
 *     otherwise the call returns TE_ERR_UNSUPPORTED and launches nothing.
 *   - The caller owns every buffer and the stream.  The library allocates no device memory;
 *     scratch space comes from the caller's `workspace` (size from te_workspace_size).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Every call
 *     is asynchronous on that stream and never synchronizes it.
 *   - Host-detectable errors are returned synchronously before any launch.  Device-side
 *     failures (a pipeline wait that timed out) are recorded in a device status word that
 *     te_get_device_status reads after the caller synchronizes.
 *   - FP8 is E4M3 (OCP "fn" variant), round to nearest even, saturating to +-448, with one fp32
 *     scale per tensor: q = E4M3(fp32(v * scale)), dequantized value = fp32(decode(q) * scale_inv).
 */
#ifndef TE_GB300_H
#define TE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TE_OK = 0,
  TE_ERR_INVALID_ARG = 1,  /* NULL required pointer, negative size, bad enum */
  TE_ERR_UNSUPPORTED = 2,  /* alignment or shape this build does not handle */
  TE_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
  TE_ERR_TIMEOUT = 4,      /* a device pipeline wait gave up (device status word only) */
  TE_ERR_WORKSPACE = 5,    /* workspace missing or smaller than te_workspace_size() */
  TE_ERR_TOO_LARGE = 6     /* problem exceeds the fixed scratch of te_dact_dbias_quantize_noalloc */
} te_status;

typedef enum { TE_F32 = 0, TE_BF16 = 1, TE_E4M3 = 2 } te_dtype;

/* norm_type: "layernorm" or "rmsnorm" (LayerNorm MLP page, I/O Contract). */
typedef enum { TE_LAYERNORM = 0, TE_RMSNORM = 1 } te_norm_type;

/* activation_type (Activation page, I/O Contract): ("relu",), ("gelu",) (tanh form),
 * ("silu",), and the gated pair ("silu", "linear") = SwiGLU.  TE_IDENTITY passes values
 * through (used for the plain bias-gradient reduction). */
/* Activations (Activation page: activation_type tuples).  TE_SWIGLU = ("silu", "linear"),
 * TE_GEGLU = ("gelu", "linear"), TE_REGLU = ("relu", "linear") are gated: their input has twice
 * the output's columns, [gate | linear], and the output is base(gate) * linear.  "gelu" is the
 * tanh form throughout. */
typedef enum {
  TE_IDENTITY = 0,
  TE_RELU = 1,
  TE_GELU = 2,
  TE_SILU = 3,
  TE_SWIGLU = 4,
  TE_GEGLU = 5,
  TE_REGLU = 6
} te_act_type;

/* How a quantizer obtains its scale.
 *   TE_SCALING_DELAYED: use *scale as given (e.g. from an earlier call's amax); one pass.
 *   TE_SCALING_CURRENT: compute this call's amax first, then scale = 448 / amax (1 if amax is
 *                       0 or not finite, FLT_MAX if the quotient overflows); two passes. */
typedef enum { TE_SCALING_DELAYED = 0, TE_SCALING_CURRENT = 1 } te_scaling;

/* One FP8 quantizer (the pages' Quantizer: the optional object that makes an output FP8).
 * All three pointers are device fp32 scalars.
 *   scale     DELAYED: read.  CURRENT: written (448 / amax).
 *   scale_inv written: 1 / scale, the factor that dequantizes this tensor.
 *   amax      written: max |v| over the fp32 values before the cast, for this call.
 * A quantizer whose `scale` is NULL is disabled (that tensor is not quantized). */
typedef struct {
  float* scale;
  float* scale_inv;
  float* amax;
  int32_t mode; /* te_scaling */
} te_quantizer;

/* The pages' QuantizerSet.  Passing NULL for a te_quantizer_set* is noop_quantizer_set. */
typedef struct {
  te_quantizer x;       /* normalized output (the first GEMM's A operand) */
  te_quantizer kernel1; /* kernel1, or the LayerNorm-Dense kernel */
  te_quantizer act;     /* activation output (the second GEMM's A operand) */
  te_quantizer kernel2; /* kernel2 */
  te_quantizer grad;    /* activation gradient dH in the backward pass */
} te_quantizer_set;

/* Operation ids for te_workspace_size. */
typedef enum {
  TE_OP_NORM_FWD = 0,
  TE_OP_ACT_LU = 1,
  TE_OP_DACT_DBIAS = 2,
  TE_OP_LAYERNORM_DENSE_FWD = 3,
  TE_OP_LAYERNORM_MLP_FWD = 4,
  TE_OP_NORM_BWD = 5,
  TE_OP_LAYERNORM_MLP_BWD = 6,
  TE_OP_LAYERNORM_DENSE_BWD = 7,
  TE_OP_LAYERNORM_MLP_FWD_HOST = 8,
  TE_OP_GEMM = 9 /* dims = {M, K, N}, dtype = the operands' dtype */
} te_op;

/* Human-readable name of a status code (static storage, never NULL). */
const char* te_status_string(te_status status);

/* ABI version of this library (major * 100 + minor). */
int te_version(void);

/* Reads and clears the device status word of the current device.  Synchronizes the device.
 * *device_status receives TE_OK, or the te_status a kernel recorded (e.g. TE_ERR_TIMEOUT). */
te_status te_get_device_status(int32_t* device_status);

/* Self-test of the failure reporting (no counterpart on the pages).  Launches on `stream` one
 * kernel whose single waiting thread waits `limit_us` microseconds (1 .. 1000000) on an
 * mbarrier that nothing completes -- the bounded wait every pipeline of this library uses --
 * so that the wait gives up and records TE_ERR_TIMEOUT in the device status word.  The kernel
 * then exits normally; nothing faults and the context stays usable.  Returns
 * TE_ERR_INVALID_ARG for a limit outside the range. */
te_status te_selftest_wait_timeout(int64_t limit_us, void* stream);

/* Bytes of workspace a call needs.  dims = {M, H, F or N}; `dtype` is the activation dtype,
 * `quantized` is nonzero when a quantizer set is passed, `kernel_dtype` the weights' storage
 * dtype.  Unused dims may be 0.  Returns 0 for operations that need none.
 * The size includes, at its end, scratch for splitting the GEMMs' last partial wave of tiles
 * along K; it depends on the current device's SM count (none without a device).  A workspace
 * that stops short of that scratch is accepted: the call then splits no tile. */
size_t te_workspace_size(te_op op, int64_t M, int64_t H, int64_t F_or_N, te_dtype dtype,
                         int quantized, te_dtype kernel_dtype, te_act_type act);

/* ---------------------------------------------------------------------------------------
 * te_norm_fwd -- LayerNorm or RMSNorm of each row (LayerNorm MLP page, Description, forward
 * step (1), the tex.normalization_fwd primitive; I/O Contract: norm_type, zero_centered_gamma,
 * epsilon).
 *   x      [M, H] in x_dtype (TE_F32 or TE_BF16); gamma, beta [H] in x_dtype.
 *   layernorm: y = (x - mean) / sqrt(var + epsilon) * g + beta, var the population variance;
 *              a NULL beta is taken as zero.
 *   rmsnorm:   y = x / sqrt(mean(x^2) + epsilon) * g; beta is ignored and may be NULL.
 *   g = gamma, or 1 + gamma when zero_centered_gamma != 0.  All arithmetic is fp32.
 *   out    [M, H] in out_dtype: TE_F32, TE_BF16, or TE_E4M3 (then q is required).
 *   q      NULL, or the quantizer of y: amax of the fp32 y is written to q->amax (also
 *          when out_dtype is not E4M3), and for E4M3 the codes use q's scale.
 *   mu, rsigma  [M] fp32, optional (NULL = not written): the row mean (0 for rmsnorm) and
 *          1 / sqrt(var + epsilon) (or 1 / sqrt(mean(x^2) + epsilon)).
 * H must be a multiple of 8 (16-byte rows) and at most 8192.
 */
te_status te_norm_fwd(const void* x, te_dtype x_dtype, int64_t M, int64_t H, const void* gamma,
                      const void* beta, te_norm_type norm_type, int zero_centered_gamma,
                      float epsilon, const te_quantizer* q, void* out, te_dtype out_dtype,
                      float* mu, float* rsigma, void* stream);

/* ---------------------------------------------------------------------------------------
 * te_act_lu -- activation with optional FP8 quantization (Activation page, Description: the
 * forward rule runs the tex.act_lu primitive, quantizing when asked, and returns the values
 * dequantized).
 *   x      [M, N_in] in x_dtype (TE_F32 / TE_BF16).  For a gated type, N_in = 2 * N_out and the
 *          columns are [gate | linear]: out = silu(x[:, :N_out]) * x[:, N_out:].
 *   out    [M, N_out] in out_dtype.
 *   q      NULL: out = act(x) rounded to out_dtype (TE_F32 / TE_BF16).
 *          non-NULL with out_dtype TE_E4M3: out holds the E4M3 codes.
 *          non-NULL with out_dtype TE_F32 / TE_BF16: out holds the dequantized values
 *          fp32(decode(q) * scale_inv), as the page's activation() returns them.
 * N_out must be a multiple of 8.
 */
te_status te_act_lu(const void* x, te_dtype x_dtype, int64_t M, int64_t N_in, te_act_type act,
                    const te_quantizer* q, void* out, te_dtype out_dtype, void* stream);

/* ---------------------------------------------------------------------------------------
 * te_dact_dbias_quantize -- the backward step that fuses the activation gradient, the bias
 * gradient reduction and the FP8 cast (LayerNorm MLP page, Description, backward pass:
 * tex.quantize_dact_dbias;
 * Activation page, Description: tex.dact_lu).
 *   dy        [M, N_out] in dtype: gradient w.r.t. the activation output.
 *   x_preact  [M, N_in] in dtype: the activation input saved by the forward (ignored for
 *             TE_IDENTITY, which makes dx = dy and dbias its column sums).
 *   dx        [M, N_in] in dx_dtype: dy * act'(x_preact) computed in fp32, then rounded
 *             (TE_F32 / TE_BF16) or quantized (TE_E4M3 with q).  Gated: [d_gate | d_linear].
 *   dbias     [N_in] fp32 or NULL: column sums of the fp32 dx before any rounding, reduced
 *             in a fixed order (deterministic).
 *   workspace te_workspace_size(TE_OP_DACT_DBIAS, M, 0, N_in, ...) bytes, needed when dbias
 *             is requested.
 */
te_status te_dact_dbias_quantize(const void* dy, const void* x_preact, te_dtype dtype, int64_t M,
                                 int64_t N_in, te_act_type act, const te_quantizer* q, void* dx,
                                 te_dtype dx_dtype, float* dbias, void* workspace,
                                 size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * te_quantize -- per-tensor E4M3 cast of a [M, N] tensor (LayerNorm Dense page, Description:
 * both the normalized output and the kernel are cast to FP8 before the GEMM).  x in x_dtype (TE_F32 / TE_BF16); out E4M3
 * codes [M, N]; q required (DELAYED uses *scale, CURRENT computes it).  N multiple of 8.
 */
te_status te_quantize(const void* x, te_dtype x_dtype, int64_t M, int64_t N,
                      const te_quantizer* q, void* out, void* stream);

/* ---------------------------------------------------------------------------------------
 * te_update_scales -- the delayed-scaling step between two calls: for each enabled quantizer
 * of qs[0 .. n-1] (a host array of n <= 16 structs; disabled ones, scale == NULL, are skipped),
 * *scale = 448 / *amax (1 if the amax is 0 or not finite, FLT_MAX if the quotient overflows)
 * and *scale_inv = 1 / *scale, on the device, in one launch on `stream`.  (The FP8 recipe the
 * pages leave open, read as per-tensor scaling from the amax; no page section defines this
 * step by name.)  Data-parallel callers reduce every rank's amax with MAX first, so that all
 * ranks derive the same scales.  An enabled quantizer needs an amax; NULL or misaligned
 * pointers and n outside 0 .. 16 give TE_ERR_INVALID_ARG.
 */
te_status te_update_scales(const te_quantizer* qs, int n, void* stream);

/* ---------------------------------------------------------------------------------------
 * te_gemm -- D = alpha * op(A) @ op(B) + bias on the tensor cores (LayerNorm MLP page,
 * Description, forward steps (2) and (4): the tex.gemm primitive with a bias).
 *   op(A) is [M, K]: A stored [M, K] (a_trans = 0) or [K, M] (a_trans = 1).
 *   op(B) is [K, N]: B stored [K, N] (b_trans = 0) or [N, K] (b_trans = 1).
 *   ab_dtype      TE_BF16, TE_E4M3 or TE_F32 (computed as TF32); A and B share it.
 *   a_scale_inv, b_scale_inv  device fp32 scalars or NULL (= 1); alpha is their product.
 *   bias          [N] in bias_dtype (TE_F32 / TE_BF16) or NULL.
 *   D             [M, N] in d_dtype (TE_F32 / TE_BF16).
 *   workspace     NULL, or te_workspace_size(TE_OP_GEMM, M, K, N, ab_dtype, ...) bytes,
 *                 16-byte aligned: with it, the tiles of the last partial wave are split along
 *                 K over the idle SM pairs (their fp32 partial sums added in a fixed order, so
 *                 repeated calls give identical results; the rounding differs from the unsplit
 *                 sum within fp32 accumulation error).
 * M >= 1; N and K multiples of 16.
 */
te_status te_gemm(const void* A, int a_trans, const void* B, int b_trans, te_dtype ab_dtype,
                  int64_t M, int64_t N, int64_t K, const float* a_scale_inv,
                  const float* b_scale_inv, const void* bias, te_dtype bias_dtype, void* D,
                  te_dtype d_dtype, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * te_layernorm_dense_fwd -- out = norm(x) @ kernel + bias (LayerNorm Dense page, Description
 * and Signature: layernorm_dense(x, kernel, gamma, beta, bias, norm_type, zero_centered_gamma,
 * epsilon, ..., quantizer_set)).
 *   dtype         activation dtype of x, gamma, beta, bias and out (TE_F32 or TE_BF16).
 *   x [M, H]; kernel [H, N] in kernel_dtype; bias [N] or NULL; out [M, N].
 *   qset NULL (no quantization): the normalized output is stored in dtype, kernel_dtype must
 *        equal dtype.  Non-NULL (FP8): qset->x and qset->kernel1 must be enabled; the
 *        normalized output is written once, as E4M3.  kernel_dtype TE_E4M3 means the kernel is
 *        already quantized and qset->kernel1.scale_inv holds its dequantization factor;
 *        kernel_dtype == dtype means it is quantized in this call with qset->kernel1.
 *   saved_ln_out  [M, H] (E4M3 with qset, else dtype) or NULL: keeps the GEMM operand.
 *   mu, rsigma    [M] fp32 or NULL.
 */
te_status te_layernorm_dense_fwd(const void* x, const void* kernel, te_dtype kernel_dtype,
                                 const void* gamma, const void* beta, const void* bias,
                                 te_norm_type norm_type, int zero_centered_gamma, float epsilon,
                                 const te_quantizer_set* qset, int64_t M, int64_t H, int64_t N,
                                 te_dtype dtype, void* out, void* saved_ln_out, float* mu,
                                 float* rsigma, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * te_layernorm_mlp_fwd -- norm -> GEMM1 + bias1 -> activation -> GEMM2 + bias2 (LayerNorm MLP
 * page, Description steps (1)-(4); Signature: layernorm_mlp(x, gamma, beta, kernels, biases,
 * norm_type, zero_centered_gamma, epsilon, ..., activation_type, quantizer_set)).
 *   dtype       activation dtype of x, gamma, beta, biases, out (TE_F32 or TE_BF16).
 *   x [M, H]; kernel1 [H, F'] with F' = 2F for a gated act (columns [gate | linear]) else F;
 *   kernel2 [F, H]; bias1 [F'] or NULL; bias2 [H] or NULL; out [M, H].
 *   GEMM1's output plus bias1 is rounded to dtype before the activation; the activation and
 *   the FP8 casts are fused into GEMM1's epilogue, bias2 into GEMM2's.
 *   qset  NULL, or FP8 mode: qset->x, kernel1, act, kernel2 enabled; kernel_dtype TE_E4M3
 *         means both kernels are pre-quantized (their scale_inv fields hold the factors),
 *         kernel_dtype == dtype means they are quantized in this call.
 *   saved_h      [M, F'] in dtype or NULL: GEMM1 output + bias1 (the activation input).
 *   saved_act    [M, F] (E4M3 codes with qset, else dtype) or NULL: the activation output as
 *                GEMM2 reads it.  When given, GEMM1's epilogue writes it there instead of into
 *                the workspace (the workspace size does not change).
 *   saved_ln_out [M, H] (E4M3 with qset, else dtype) or NULL.
 *   mu, rsigma   [M] fp32 or NULL.
 */
te_status te_layernorm_mlp_fwd(const void* x, const void* gamma, const void* beta,
                               const void* kernel1, const void* kernel2, te_dtype kernel_dtype,
                               const void* bias1, const void* bias2, te_norm_type norm_type,
                               int zero_centered_gamma, float epsilon, te_act_type act,
                               const te_quantizer_set* qset, int64_t M, int64_t H, int64_t F,
                               te_dtype dtype, void* out, void* saved_h, void* saved_act,
                               void* saved_ln_out, float* mu, float* rsigma, void* workspace,
                               size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * te_layernorm_mlp_fwd_host -- te_layernorm_mlp_fwd (LayerNorm MLP page, Description steps
 * (1)-(4)) with the activations in HOST memory: x_host [M, H] and out_host [M, H] are host
 * pointers (pinned -- cudaHostAlloc or cudaHostRegister -- for the copies to overlap); gamma,
 * beta, the kernels and the biases are device pointers as in te_layernorm_mlp_fwd.  No quantizer
 * set (a per-tensor FP8 scale needs every row before the cast) and no saved tensors.
 *   The rows are cut into at most `chunks` (1 .. 16) slices: the first and the last small (their
 *   copies are the ones no compute hides), the middle ones seven times larger, all but the last
 *   a multiple of 256 rows.  All host -> device copies are issued on a copy-in stream, each
 *   slice's forward runs on `stream` once
 *   its rows have landed, and its output returns on a copy-out stream as soon as it is
 *   computed; two such streams are created per device on first use and kept.  The copies start
 *   after the work already queued on `stream`, and `stream` waits for the last copy out before
 *   anything queued after the call, so the call is asynchronous and ordered like the others.
 *   Concurrent calls on one device from several host threads are not supported.
 *   workspace: te_workspace_size(TE_OP_LAYERNORM_MLP_FWD_HOST, M, H, F, dtype, 0, dtype, act)
 *   bytes, 256-byte aligned (device staging of x and out, and one forward's workspace).
 *   dtype TE_BF16 or TE_F32; the kernels in dtype.  Errors as for te_layernorm_mlp_fwd, plus
 *   TE_ERR_INVALID_ARG for `chunks` outside 1 .. 16.
 */
te_status te_layernorm_mlp_fwd_host(const void* x_host, const void* gamma, const void* beta,
                                    const void* kernel1, const void* kernel2, const void* bias1,
                                    const void* bias2, te_norm_type norm_type,
                                    int zero_centered_gamma, float epsilon, te_act_type act,
                                    int64_t M, int64_t H, int64_t F, te_dtype dtype,
                                    void* out_host, int chunks, void* workspace, size_t ws_bytes,
                                    void* stream);

/* ---------------------------------------------------------------------------------------
 * te_layernorm_mlp_bwd -- backward of te_layernorm_mlp_fwd (LayerNorm MLP page, Description:
 * the backward pass yields the gradient of every parameter and uses the fused activation
 * gradient + bias reduction + quantization step).
 * Sequence (all on `stream`): dbias2 = column sums of dy; a = act(saved_h) recomputed in dtype;
 * dkernel2 = a^T dy; da = dy kernel2^T; dH = da * act'(saved_h) with dbias1 = its fp32 column
 * sums, stored E4M3 (qset->grad) or in dtype; dln = dH kernel1^T; dkernel1 = ln^T dH; then the
 * norm backward gives dx, dgamma, dbeta.
 *   dy [M, H], x [M, H], gamma [H], kernel2 [F, H], saved_h [M, F'] in dtype (F' = 2F for
 *   a gated act); kernel1 [H, F'] in kernel_dtype; mu, rsigma [M] from the forward.
 *   saved_ln_out [M, H]: the forward's normalized output (E4M3 with qset, else dtype).
 *   qset NULL: every GEMM in dtype.  Non-NULL (FP8): qset->grad must be enabled and quantizes dH;
 *   qset->x.scale_inv dequantizes saved_ln_out; kernel1 is E4M3 (kernel_dtype TE_E4M3, factor in
 *   qset->kernel1.scale_inv) or is quantized here with qset->kernel1.  dln and dkernel1 then run
 *   as E4M3 x E4M3 GEMMs; dy, kernel2 and the recomputed activation stay in dtype.
 *   Outputs: dx [M, H] dtype; dgamma [H] fp32; dbeta [H] fp32 or NULL (rmsnorm: written
 *   with zeros, the gradient of the unused beta); dkernel1 [H, F'] and dkernel2 [F, H] in
 *   dtype; dbias1 [F'] and dbias2 [H] fp32 or NULL.
 *   saved_dh [M, F'] or NULL: when given, dH is written there (E4M3 codes with qset, else dtype)
 *   instead of into the workspace, as the dln and dkernel1 GEMMs read it.
 *   workspace: te_workspace_size(TE_OP_LAYERNORM_MLP_BWD, M, H, F, dtype, quantized,
 *   kernel_dtype, act) bytes.  H and F multiples of 16.
 */
te_status te_layernorm_mlp_bwd(const void* dy, const void* x, const void* gamma,
                               const void* kernel1, const void* kernel2, te_dtype kernel_dtype,
                               const void* saved_h, const void* saved_ln_out, const float* mu,
                               const float* rsigma, te_norm_type norm_type,
                               int zero_centered_gamma, te_act_type act,
                               const te_quantizer_set* qset, int64_t M, int64_t H, int64_t F,
                               te_dtype dtype, void* dx, float* dgamma, float* dbeta,
                               void* dkernel1, void* dkernel2, float* dbias1, float* dbias2,
                               void* saved_dh, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * te_layernorm_dense_bwd -- backward of te_layernorm_dense_fwd (LayerNorm Dense page,
 * Description: the gradients of x, the kernel, gamma, beta and the bias, with FP8 intermediate
 * gradients).
 * Sequence (all on `stream`): dbias = fp32 column sums of dy, taken over the unquantized dy in
 * the same pass that casts dy to E4M3 with qset->grad (FP8 mode); dln = dy kernel^T;
 * dkernel = ln^T dy; then the norm backward gives dx, dgamma, dbeta.
 *   dy [M, N], x [M, H], gamma [H] in dtype; kernel [H, N] in kernel_dtype; mu, rsigma [M]
 *   from the forward (mu unused for rmsnorm).
 *   saved_ln_out [M, H]: the forward's normalized output (E4M3 with qset, else dtype).
 *   qset NULL: both GEMMs in dtype (kernel_dtype must equal dtype).  Non-NULL (FP8): qset->grad
 *   must be enabled and quantizes dy; qset->x.scale_inv dequantizes saved_ln_out; the kernel is
 *   E4M3 (kernel_dtype TE_E4M3, factor in qset->kernel1.scale_inv) or is quantized here with
 *   qset->kernel1.  Both GEMMs then run as E4M3 x E4M3.
 *   Outputs (caller-owned): dx [M, H] dtype; dgamma [H] fp32; dbeta [H] fp32 or NULL
 *   (rmsnorm: written with zeros); dkernel [H, N] dtype; dbias [N] fp32 or NULL.
 *   workspace: te_workspace_size(TE_OP_LAYERNORM_DENSE_BWD, M, H, N, dtype, quantized,
 *   kernel_dtype, 0) bytes, 16-byte aligned.  dtype TE_BF16; H and N multiples of 16, H at most
 *   8192.  A NULL required pointer, a bad enum or a quantizer set without what FP8 mode needs
 *   gives TE_ERR_INVALID_ARG; sizes or alignment outside these limits TE_ERR_UNSUPPORTED; a
 *   missing or short workspace TE_ERR_WORKSPACE.  M = 0 zeroes every gradient.
 */
te_status te_layernorm_dense_bwd(const void* dy, const void* x, const void* gamma,
                                 const void* kernel, te_dtype kernel_dtype,
                                 const void* saved_ln_out, const float* mu, const float* rsigma,
                                 te_norm_type norm_type, int zero_centered_gamma,
                                 const te_quantizer_set* qset, int64_t M, int64_t H, int64_t N,
                                 te_dtype dtype, void* dx, float* dgamma, float* dbeta,
                                 void* dkernel, float* dbias, void* workspace, size_t ws_bytes,
                                 void* stream);

/* ---------------------------------------------------------------------------------------
 * te_norm_bwd -- gradients of te_norm_fwd (LayerNorm MLP page, Description: the backward pass
 * yields the gradient of every parameter; LayerNorm Dense page, Description: gradients of x,
 * gamma and beta).
 *   dz [M, H] upstream gradient and x [M, H] the forward input, both in dtype; mu, rsigma [M]
 *   from te_norm_fwd (mu unused for rmsnorm); gamma [H] in dtype.
 *   With xhat = (x - mu) * rsigma (layernorm) or x * rsigma (rmsnorm), g the applied gain and
 *   dxhat = dz * g:
 *     layernorm: dx = rsigma * (dxhat - mean(dxhat) - xhat * mean(dxhat * xhat))
 *     rmsnorm:   dx = rsigma * (dxhat - xhat * mean(dxhat * xhat))
 *   dx [M, H] in dtype; dgamma [H] fp32 = sum over rows of dz * xhat; dbeta [H] fp32 = sum over
 *   rows of dz (layernorm; may be NULL).  The column sums are reduced in a fixed order.
 *   workspace: te_workspace_size(TE_OP_NORM_BWD, M, H, ...) bytes.  H multiple of 8, at most
 *   8192 bf16 / 4096 fp32.
 */
te_status te_norm_bwd(const void* dz, const void* x, const float* mu, const float* rsigma,
                      const void* gamma, te_dtype dtype, int64_t M, int64_t H,
                      te_norm_type norm_type, int zero_centered_gamma, void* dx, float* dgamma,
                      float* dbeta, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * Instrumentation (no counterpart on the pages; used by benchmarks).
 * Between te_profile_begin and te_profile_end every kernel the library launches is bracketed
 * by CUDA events recorded on the launching stream.  te_profile_end synchronizes those events
 * and returns, per kernel kind, the summed device time (ms) and the number of launches.
 * Arrays have TE_KERNEL_KINDS entries (either may be NULL).  At most `max_records` launches
 * are timed (later ones are only counted).  Not thread-safe against concurrent calls.
 */
typedef enum {
  TE_KERNEL_NORM_FWD = 0,
  TE_KERNEL_QUANTIZE = 1,
  TE_KERNEL_ACT_LU = 2,
  TE_KERNEL_DACT_DBIAS = 3,
  TE_KERNEL_GEMM = 4,        /* GEMM + bias epilogue */
  TE_KERNEL_GEMM_ACT = 5,    /* GEMM + bias + activation (+ amax, E4M3) epilogue */
  TE_KERNEL_NORM_BWD = 6,
  TE_KERNEL_TRANSPOSE = 7,
  TE_KERNEL_KINDS = 8
} te_kernel_kind;

te_status te_profile_begin(int32_t max_records);
te_status te_profile_end(float* total_ms, int32_t* launches);

/* Streaming reference (no counterpart on the pages; used by benchmarks).  One launch of a plain
 * kernel that moves a bandwidth-bound kernel's traffic with no arithmetic: it reads
 * `ratio` x `write_bytes` bytes from `src` and writes `write_bytes` bytes to `dst`, each
 * 16-byte vector of dst from the next `ratio` vectors of src; write_bytes = 0 reads
 * `read_only_bytes` from src and writes nothing.  Its time is the floor a kernel with the same
 * traffic, size and access order can reach, below the bandwidth of a long copy for short
 * kernels.  src, dst 16-byte aligned, byte counts multiples of 16, ratio 1 .. 8; otherwise
 * TE_ERR_INVALID_ARG. */
te_status te_stream_probe(const void* src, void* dst, size_t write_bytes, int ratio,
                          size_t read_only_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * te_dact_dbias_quantize_noalloc -- te_dact_dbias_quantize for callers that cannot allocate
 * device memory at the call (no counterpart on the pages; an addition of this library).
 *
 * Who needs it: plugin hosts and runtimes that plan every device buffer ahead of time and give
 * an operator no allocator, and latency-critical code that cannot afford cudaMalloc's
 * device-wide synchronization.  Such callers cannot provide the workspace that
 * te_dact_dbias_quantize's bias reduction needs.
 *
 * Same arguments, results and rules as te_dact_dbias_quantize, without workspace/ws_bytes.  The
 * call allocates nothing: the bias reduction's partial sums live in one fixed device array of
 * te_dact_dbias_noalloc_capacity() floats (8 MiB) that every GPU loading the library holds
 * until the process exits.
 *   - A reduction needing more than the capacity (ceil(M / 128) * N_in floats, counted only when
 *     dbias is requested) returns TE_ERR_TOO_LARGE before launching.
 *   - The first call on a device looks up the array's device address once for that device;
 *     make that first call before any stream capture begins on the device.
 *   - All calls on a device share the array: calls that overlap on the GPU race on it (order
 *     them on one stream).  Nothing in it must start at zero; it keeps the last call's data.
 */
te_status te_dact_dbias_quantize_noalloc(const void* dy, const void* x_preact, te_dtype dtype,
                                         int64_t M, int64_t N_in, te_act_type act,
                                         const te_quantizer* q, void* dx, te_dtype dx_dtype,
                                         float* dbias, void* stream);

/* Floats of fixed scratch behind te_dact_dbias_quantize_noalloc. */
size_t te_dact_dbias_noalloc_capacity(void);

#ifdef __cplusplus
}
#endif

#endif /* TE_GB300_H */
