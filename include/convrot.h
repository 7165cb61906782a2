/*
 * convrot.h -- C ABI of libconvrot.so, the INT8 "convrot" linear layer on
 * NVIDIA GB300 (sm_103a).
 *
 * What the library computes (stable-diffusion.cpp documentation, page
 * "INT8 Convrot Safetensors"):
 *   - "How INT8 convrot works": R_G = H4^{(x)n}, the normalized Kronecker
 *     power of the regular Hadamard matrix H4 for a group size G = 4^n,
 *     applied to every contiguous group of G input features: X_rot = X R,
 *     W_rot = W R.
 *   - "Weight quantization": s_w[o] = max_i |W_rot[o,i]| / 127,
 *     Q_w[o,i] = clamp(round(W_rot[o,i] / s_w[o]), -127, 127).
 *   - "Runtime activation quantization": s_x[r] = max_i |X_rot[r,i]| / 127
 *     over the whole rotated row, Q_x by the same rule, the int32 product
 *     A[r,o] = sum_i Q_x[r,i] Q_w[o,i], and Y ~= A s_x[r] s_w[o] + b[o];
 *     linears sharing an input and a group size reuse one packed activation.
 *   - page "ggml operator extensions", section "sd.cpp integration": the
 *     output is float(A) * s_x * s_w + bias evaluated in that order, with the
 *     weight scale and the bias optional.
 *
 * Conventions for every entry point
 *   - Matrices are dense and row-major: X is [M,K] (K contiguous), W and the
 *     weight codes are [N,K], Y and A are [M,N].
 *   - Every array pointer is a DEVICE pointer on the current CUDA device,
 *     owned by the caller; the library keeps no pointer after a call returns
 *     and allocates no device memory. Arrays must start on a 16-byte boundary.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Work is enqueued asynchronously on it; the return value only
 *     reports argument checks and launch errors. Faults found later by a
 *     kernel (a bounded device-side wait that gave up) are reported by
 *     convrot_device_status().
 *   - Rounding: "round" is round-half-to-even; the two divisions of the
 *     quantizer are IEEE fp32 divisions; an all-zero row has scale 0 and
 *     codes 0.
 *   - The tensor cores of sm_103a have no 8-bit integer MMA, so the GEMM runs
 *     on the fp16 tensor-core path: int8 codes are exact in IEEE binary16, each
 *     K-chunk of at most 1024 products is summed exactly in fp32 (its partial
 *     sums stay below 2^24) and the chunk sums are added in int32. The int32
 *     result is therefore bit-exact. Weight codes are also kept as binary16
 *     ("Q_w16", written by convrot_prepare_weight) so the GEMM reads them
 *     directly.
 */
#ifndef CONVROT_H
#define CONVROT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. Every entry point returns one of these (as int). */
typedef enum convrot_status {
  CONVROT_OK = 0,
  CONVROT_ERR_ARG = 1,         /* NULL where an array is required, a size < 0,
                                  an unknown dtype, n_weights outside [1,8] */
  CONVROT_ERR_GROUP = 2,       /* G is not 4^n with 1 <= G <= 1024, or K % G != 0
                                  ("Checkpoint format": a power of four that
                                  divides the input feature dimension) */
  CONVROT_ERR_ALIGN = 3,       /* an array not 16-byte aligned, or K % 16 != 0 */
  CONVROT_ERR_OVERFLOW = 4,    /* K * 127^2 > INT32_MAX (K > 133144): the int32
                                  accumulation could overflow */
  CONVROT_ERR_ALIAS = 5,       /* an output array overlaps an input or another
                                  output */
  CONVROT_ERR_WORKSPACE = 6,   /* workspace NULL or smaller than the size query */
  CONVROT_ERR_UNSUPPORTED = 7, /* a shape beyond this build's limits (pack rows
                                  longer than CONVROT_PACK_MAX_K) */
  CONVROT_ERR_TIMEOUT = 8,     /* a kernel's bounded wait gave up (from
                                  convrot_device_status) */
  CONVROT_ERR_CUDA = 9,        /* a CUDA runtime call failed or a launch error;
                                  convrot_last_cuda_error() gives the code */
  CONVROT_ERR_DEVICE = 10,     /* the current device is not an sm_103 GPU */
  CONVROT_ERR_SCRATCH = 11     /* the packed activation does not fit in the
                                  library's fixed scratch array
                                  (convrot_linear_noalloc) */
} convrot_status;

/* Element type of the floating-point activation input X. */
typedef enum convrot_dtype {
  CONVROT_F32 = 0, /* IEEE binary32 */
  CONVROT_F16 = 1  /* IEEE binary16 (converted exactly to fp32 on load) */
} convrot_dtype;

/* Activation applied to a linear's output (convrot_mlp). */
typedef enum convrot_activation {
  CONVROT_ACT_NONE = 0,
  CONVROT_ACT_GELU = 1,  /* 0.5 y (1 + erf(y / sqrt 2)), fp32, erf by Abramowitz &
                            Stegun 7.1.28 (|error| <= 3e-7) */
  CONVROT_ACT_SWIGLU = 2 /* split SwiGLU: silu(gate) * up = (g / (1 + exp(-g))) * u
                            of two linears sharing the input (fp32, expf and an
                            IEEE division) */
} convrot_activation;

/* Longest activation row (K) the pack kernel holds on chip. */
#define CONVROT_PACK_MAX_K 32768
/* Largest K whose worst-case int32 accumulation fits: 133144 * 127^2 < 2^31. */
#define CONVROT_MAX_K 133144
/* Most linears one convrot_linear call may share a packed input across. */
#define CONVROT_MAX_LINEARS 8

/* Library version, major*10000 + minor*100 + patch. */
int convrot_version(void);

/* Static text for a convrot_status value. */
const char* convrot_strerror(int status);

/* The cudaError_t of the most recent CONVROT_ERR_CUDA on this host thread. */
int convrot_last_cuda_error(void);

/*
 * convrot_prepare_weight -- offline weight path ("Weight quantization").
 *   W      [N,K] fp32 weights (input).
 *   G      group size, 4^n in [1,1024], dividing K.
 *   Q_w    [N,K] int8 codes (output).
 *   s_w    [N] fp32 per-output-row scales (output).
 *   Q_w16  [N,K] the same codes as binary16 (output, may be NULL; required by
 *          convrot_linear and used by int8_linear when given).
 * Same rotation and quantizer as convrot_pack_activations, applied to W.
 * Errors: ERR_ARG, ERR_GROUP, ERR_ALIGN, ERR_ALIAS, ERR_UNSUPPORTED, ERR_CUDA.
 */
int convrot_prepare_weight(const float* W, int64_t N, int64_t K, int G,
                           int8_t* Q_w, float* s_w, uint16_t* Q_w16,
                           void* stream);

/*
 * convrot_pack_activations -- runtime activation quantization.
 *   X       [M,K] activations, fp32 or fp16 per x_dtype (input).
 *   Q_x     [M,K] int8 codes (output).
 *   s_x     [M] fp32 row scales (output).
 * One pass over X: group-wise rotation, row absmax over the whole rotated
 * row, quantization. M = 0 is a no-op. K <= CONVROT_PACK_MAX_K.
 * Errors: ERR_ARG, ERR_GROUP, ERR_ALIGN, ERR_ALIAS, ERR_UNSUPPORTED, ERR_CUDA.
 */
int convrot_pack_activations(const void* X, int x_dtype, int64_t M, int64_t K,
                             int G, int8_t* Q_x, float* s_x, void* stream);

/*
 * Bytes of the GEMM's hand-over words, part of every workspace below. When the
 * last wave of output tiles would leave CTA pairs idle, the GEMM splits the
 * remaining tiles by K over all pairs; a pair that ends inside a tile passes
 * its int32 partial sums (stored in that tile's output) to the pair that
 * finishes it, and these words say when they are ready (one 8-byte word per
 * CTA, up to 256 CTA pairs). Their content between calls needs no
 * initialization: a call writes a value unique to it and zeroes what it
 * consumed. A workspace must not be used by two calls that run at the same
 * time.
 */
#define CONVROT_GEMM_SYNC_BYTES 4096

/*
 * int8_linear_workspace_size -- device bytes int8_linear needs: room to widen
 * Q_x (and Q_w when Q_w16 is not given) to binary16 codes, and the GEMM's
 * hand-over words (CONVROT_GEMM_SYNC_BYTES).
 */
size_t int8_linear_workspace_size(int64_t M, int64_t N, int64_t K,
                                  int have_q_w16);

/*
 * int8_linear -- Y = float(Q_x Q_w^T) * s_x[r] * s_w[o] + bias[o].
 *   Q_x    [M,K] int8, s_x [M] fp32 (e.g. from convrot_pack_activations).
 *   Q_w    [N,K] int8 codes; may be NULL when Q_w16 is given.
 *   Q_w16  [N,K] binary16 codes, or NULL (then Q_w is widened in workspace).
 *   s_w    [N] fp32 or NULL (taken as 1).   bias [N] fp32 or NULL (none).
 *   Y      [M,N] fp32 (output).
 *   workspace / workspace_bytes: device scratch, at least
 *          int8_linear_workspace_size(M, N, K, Q_w16 != NULL) bytes.
 * Errors: ERR_ARG, ERR_ALIGN, ERR_OVERFLOW, ERR_ALIAS, ERR_WORKSPACE, ERR_CUDA.
 */
int int8_linear(const int8_t* Q_x, const float* s_x, int64_t M, int64_t K,
                const int8_t* Q_w, const uint16_t* Q_w16, const float* s_w,
                const float* bias, int64_t N, float* Y,
                void* workspace, size_t workspace_bytes, void* stream);

/* Longest K of a linear with packed 4-bit weights: 127 * 8 * 16384 < 2^24, so
 * the whole product stays exact in the tensor cores' fp32 accumulator. */
#define CONVROT_W4_MAX_K 16384

/*
 * One linear of a convrot_linear call. Its weight is either binary16 codes
 * (q16, from convrot_prepare_weight) or, for the packed INT4 convrot format
 * ("INT8 Convrot Safetensors", section "Packed INT4 convrot": convrot_w4a4,
 * signed 4-bit weights, low nibble first, with an F32 per-output weight
 * scale), the checkpoint's packed bytes (q4), which the S8 x S4 GEMM reads
 * as they are: no expanded copy is made. Exactly one of q16 and q4 is set.
 * A q4 linear needs K % 64 == 0 (ERR_ALIGN otherwise), K <= CONVROT_W4_MAX_K
 * (ERR_UNSUPPORTED) and N % 4 == 0 (ERR_ALIGN); linears of both kinds may
 * share one call (one GEMM launch per kind).
 */
typedef struct convrot_weight {
  const uint16_t* q16; /* [N,K] binary16 weight codes (convrot_prepare_weight), or NULL */
  const float* scale;  /* [N] s_w, or NULL (taken as 1) */
  const float* bias;   /* [N], or NULL (no bias) */
  int64_t N;           /* output features */
  float* Y;            /* [M,N] fp32 output */
  const int32_t* kchunk; /* [ceil(N/128)] exact-chunk plan from convrot_weight_chunks,
                            or NULL (chunks of 1024 products); unused for q4 */
  const uint8_t* q4;   /* [N,K/2] packed signed 4-bit weights (element 2j of a row
                          in the low nibble of byte j), or NULL */
} convrot_weight;

/*
 * convrot_w4_expand -- weights of the packed INT4 convrot format ("Packed
 * INT4 convrot", convrot_w4a4: signed 4-bit weights, low nibble first, with
 * an F32 per-output weight scale; activations use the INT8 convrot pack) into
 * the codes the GEMM reads. Element 2j of a row is the low nibble of byte j,
 * element 2j+1 the high nibble, each a two's-complement value in [-8, 7].
 * A W4A4 linear is then convrot_linear with these codes and the checkpoint's
 * weight scale.
 *   Q_w4   [N, K/2] packed bytes (input).
 *   Q_w    [N,K] int8 codes (output, may be NULL; feeds convrot_weight_chunks).
 *   Q_w16  [N,K] binary16 codes (output, may be NULL). Not both NULL.
 * Errors: ERR_ARG, ERR_ALIGN (K % 16, 16-byte arrays), ERR_ALIAS, ERR_CUDA.
 */
int convrot_w4_expand(const uint8_t* Q_w4, int64_t N, int64_t K, int8_t* Q_w,
                      uint16_t* Q_w16, void* stream);

/* Weight rows per entry of a chunk plan. */
#define CONVROT_CHUNK_ROWS 128

/*
 * convrot_weight_chunks -- offline exact-chunk plan of a weight for the GEMM.
 * The tensor-core GEMM accumulates runs of K-products in fp32 and adds the
 * runs in int32; a run is exact when every partial sum stays below 2^24.
 * Since every activation code has |q_x| <= 127, a run over the K range R is
 * exact for output row o whenever 127 * sum_{k in R} |Q_w[o,k]| < 2^24. For
 * every block of CONVROT_CHUNK_ROWS weight rows this writes the longest run
 * length L (in units of 64 K-elements; runs start at multiples of L) among
 * {16, 32, 64, ...} and "all of K" that satisfies that bound for every row of
 * the block and every run; L = 16 (1024 products) always does.
 *   Q_w     [N,K] int8 weight codes (convrot_prepare_weight).
 *   kchunk  [ceil(N/128)] int32 (output).
 * Errors: ERR_ARG, ERR_ALIGN, ERR_OVERFLOW, ERR_ALIAS, ERR_CUDA.
 */
int convrot_weight_chunks(const int8_t* Q_w, int64_t N, int64_t K, int32_t* kchunk,
                          void* stream);

/* Device bytes convrot_linear needs: the shared packed activation and the
 * GEMM's hand-over words (CONVROT_GEMM_SYNC_BYTES). */
size_t convrot_linear_workspace_size(int64_t M, int64_t K);

/*
 * convrot_linear -- n_weights linears sharing one input and group size:
 * X is packed once (rotation, row scales, codes) into the workspace, then one
 * grouped GEMM computes every Y_j = float(Q_x Q_wj^T) * s_x * s_wj + b_j.
 *   X         [M,K] fp32/fp16 activations.
 *   weights   host array of n_weights descriptors (1 <= n_weights <= 8); all
 *             Y_j must be distinct and must not overlap X or any weight.
 *   workspace at least convrot_linear_workspace_size(M, K) bytes.
 * Errors: ERR_ARG, ERR_GROUP, ERR_ALIGN, ERR_OVERFLOW, ERR_ALIAS,
 *         ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_CUDA.
 */
int convrot_linear(const void* X, int x_dtype, int64_t M, int64_t K, int G,
                   const convrot_weight* weights, int n_weights,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * convrot_linear_scaled -- convrot_linear for linears with an input scale
 * ("Runtime activation quantization": for input scales other than 1 the
 * activations are scaled before the convrot quantization and the output is
 * unscaled before the bias is added):
 *   X' = fp32(input_scale * X),  packed with G,
 *   Y_j = (((float(Q_x' Q_wj^T) * s_x') * s_wj) / input_scale) + b_j,
 * each operation one fp32 rounding. Linears sharing X, G and the input scale
 * share the packed activation. input_scale = 1 is exactly convrot_linear.
 *   input_scale  finite and > 0 (else ERR_ARG); other arguments as convrot_linear.
 * Errors: as convrot_linear.
 */
int convrot_linear_scaled(const void* X, int x_dtype, int64_t M, int64_t K, int G,
                          float input_scale, const convrot_weight* weights, int n_weights,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * int8_gemm_s32 -- the raw int32 product A = Q_x Q_w^T (no scales), through
 * the same tensor-core GEMM as int8_linear. For exactness checks.
 *   Arguments as int8_linear; kchunk: the weight's exact-chunk plan
 *   (convrot_weight_chunks) or NULL; A [M,N] int32 (output).
 * Errors: as int8_linear.
 */
int int8_gemm_s32(const int8_t* Q_x, int64_t M, int64_t K,
                  const int8_t* Q_w, const uint16_t* Q_w16, const int32_t* kchunk,
                  int64_t N, int32_t* A, void* workspace, size_t workspace_bytes,
                  void* stream);

/* Device bytes int8_gemm_s32_w4 needs: the widened Q_x and the GEMM's
 * hand-over words (CONVROT_GEMM_SYNC_BYTES). */
size_t int8_gemm_s32_w4_workspace_size(int64_t M, int64_t K);

/*
 * int8_gemm_s32_w4 -- the raw int32 product A = Q_x Q_w^T of int8 activation
 * codes and packed signed 4-bit weights ("Packed INT4 convrot", low nibble
 * first), through the S8 x S4 GEMM that the q4 linears of convrot_linear use.
 * For exactness checks.
 *   Q_x    [M,K] int8.   Q_w4 [N,K/2] packed bytes.   A [M,N] int32 (output).
 *   K % 64 == 0 and K <= CONVROT_W4_MAX_K.
 *   workspace  at least int8_gemm_s32_w4_workspace_size(M, K) bytes.
 * Errors: ERR_ARG, ERR_ALIGN, ERR_UNSUPPORTED, ERR_ALIAS, ERR_WORKSPACE, ERR_CUDA.
 */
int int8_gemm_s32_w4(const int8_t* Q_x, int64_t M, int64_t K, const uint8_t* Q_w4, int64_t N,
                     int32_t* A, void* workspace, size_t workspace_bytes, void* stream);

/*
 * convrot_pack_activations_f16 -- the pack of convrot_pack_activations, with
 * the codes written as binary16 integers: the packed activation in the form
 * the tensor-core GEMM reads. One packed activation can feed any number of
 * convrot_linear_packed calls ("Runtime activation quantization": linears
 * sharing an input and group size reuse the packed tensor).
 *   Q_x16  [M,K] binary16 codes (output).   s_x [M] fp32 (output).
 * Errors: as convrot_pack_activations.
 */
int convrot_pack_activations_f16(const void* X, int x_dtype, int64_t M, int64_t K,
                                 int G, uint16_t* Q_x16, float* s_x, void* stream);

/*
 * convrot_pack_gelu_f16 -- the MLP's repack: GELU (as CONVROT_ACT_GELU)
 * applied to every element of fp32 rows as they are loaded, then the convrot
 * pack with the codes written as binary16 (the tensor-core GEMM's operand).
 * GELU(X) itself is never stored.
 *   X [M,K] fp32, Q_x16 [M,K] binary16 codes (output), s_x [M] fp32 (output).
 * Errors: as convrot_pack_activations.
 */
int convrot_pack_gelu_f16(const float* X, int64_t M, int64_t K, int G, uint16_t* Q_x16, float* s_x,
                          void* stream);

/*
 * convrot_linear_packed -- the grouped GEMM of convrot_linear on an activation
 * packed by convrot_pack_activations_f16: every
 * Y_j = float(Q_x Q_wj^T) * s_x * s_wj + b_j.
 *   Q_x16 [M,K] binary16 codes, s_x [M] fp32; weights as convrot_linear.
 *   workspace  NULL, or CONVROT_GEMM_SYNC_BYTES bytes of device scratch
 *              (16-byte aligned) for the GEMM's hand-over words; without it
 *              the GEMM takes whole tiles only (same results, a less even
 *              last wave).
 * Errors: ERR_ARG, ERR_ALIGN, ERR_OVERFLOW, ERR_ALIAS, ERR_WORKSPACE (workspace
 *         given but smaller than CONVROT_GEMM_SYNC_BYTES), ERR_UNSUPPORTED, ERR_CUDA.
 */
int convrot_linear_packed(const uint16_t* Q_x16, const float* s_x, int64_t M, int64_t K,
                          const convrot_weight* weights, int n_weights,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * convrot_linear_packed_act -- convrot_linear_packed with an activation applied
 * in the GEMM's epilogue before the output is stored:
 *   CONVROT_ACT_NONE    exactly convrot_linear_packed;
 *   CONVROT_ACT_GELU    every Y_j = gelu(y_j) (as CONVROT_ACT_GELU);
 *   CONVROT_ACT_SWIGLU  weights = {gate, up} (n_weights == 2, the same N,
 *                       binary16 weights): weights[0].Y = silu(gate) * up
 *                       ("ggml operator extensions", sd.cpp integration:
 *                       split SwiGLU, the epilogue writes only the activated
 *                       output; weights[1].Y is unused).
 * The activation variants need N % 4 == 0. Other arguments as
 * convrot_linear_packed.
 * Errors: as convrot_linear_packed; ERR_UNSUPPORTED for split SwiGLU with
 *         packed 4-bit weights.
 */
int convrot_linear_packed_act(const uint16_t* Q_x16, const float* s_x, int64_t M, int64_t K,
                              const convrot_weight* weights, int n_weights, int activation,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * convrot_linear_host_workspace_size -- device bytes convrot_linear_host needs:
 * two sets of chunk buffers (input rows, binary16 codes, row scales and the
 * output rows of all linears, n_total = sum of their N) and the GEMM's
 * hand-over words (CONVROT_GEMM_SYNC_BYTES). chunk_rows = 0 picks
 * the library default (768 rows). Returns 0 for invalid arguments.
 */
size_t convrot_linear_host_workspace_size(int64_t M, int64_t K, int x_dtype,
                                          int64_t n_total, int64_t chunk_rows);

/*
 * convrot_linear_host -- convrot_linear with X and every Y_j in HOST memory
 * (the weights, scales and biases stay in device memory). The rows are
 * processed in chunks of chunk_rows: each chunk is copied in on
 * copy_in_stream, packed and multiplied on `stream`, and its output rows
 * copied out on copy_out_stream, so transfers overlap compute. Host arrays
 * should be pinned (page-locked) for the transfers to overlap.
 *   X_host     [M,K] fp32/fp16 host array.
 *   weights    as convrot_linear; every Y is a host array [M,N_j] fp32.
 *   chunk_rows rows per chunk (0 = the default: a first chunk of 256 rows, so
 *              that output copies start sooner, then chunks of 768; multiples
 *              of 256 suit the GEMM).
 *   workspace  device scratch, >= convrot_linear_host_workspace_size(...).
 *   stream, copy_in_stream, copy_out_stream: cudaStream_t (NULL copy streams
 *              mean `stream`: correct but without overlap). The call is
 *              ordered after earlier work on `stream`, and later work on
 *              `stream` runs after every output copy has completed.
 * Errors: ERR_ARG, ERR_GROUP, ERR_ALIGN, ERR_ALIAS, ERR_WORKSPACE,
 *         ERR_UNSUPPORTED, ERR_CUDA.
 */
int convrot_linear_host(const void* X_host, int x_dtype, int64_t M, int64_t K, int G,
                        const convrot_weight* weights, int n_weights, int64_t chunk_rows,
                        void* workspace, size_t workspace_bytes, void* stream,
                        void* copy_in_stream, void* copy_out_stream);

/*
 * An elementwise prologue applied to fp32 X before the convrot pack (the
 * normalization and modulation producers the pages fuse into ConvRot:
 * "RMSNorm -> Mul(weight) -> Modulate -> ConvRot", "Modulate -> ConvRot",
 * scale-only modulation). In this order, each step one fp32 rounding per
 * operation, absent parts skipped:
 *   x <- x * (1 / sqrt(mean_k(x^2) + eps))   if rmsnorm (mean over the row)
 *   x <- x * weight[k]                        if weight
 *   x <- x + x * scale[k]                     if scale
 *   x <- x + shift[k]                         if shift
 */
typedef struct convrot_prologue {
  int rmsnorm;          /* nonzero: normalize each row by its RMS first */
  float eps;            /* added to mean(x^2) before the square root */
  const float* weight;  /* [K] per-channel multiplier, or NULL */
  const float* scale;   /* [K] modulation scale, or NULL */
  const float* shift;   /* [K] modulation shift, or NULL */
} convrot_prologue;

/*
 * convrot_pack_prologue -- convrot_pack_activations of prologue(X) without
 * writing prologue(X): X fp32 [M,K] -> Q_x int8 [M,K], s_x [M].
 * Errors: as convrot_pack_activations; vectors must be 16-byte aligned.
 */
int convrot_pack_prologue(const float* X, int64_t M, int64_t K, int G,
                          const convrot_prologue* prologue, int8_t* Q_x, float* s_x,
                          void* stream);

/*
 * convrot_linear_prologue -- convrot_linear on prologue(X): one pack with the
 * prologue, one grouped GEMM. Arguments and workspace as convrot_linear.
 */
int convrot_linear_prologue(const float* X, int64_t M, int64_t K, int G,
                            const convrot_prologue* prologue, const convrot_weight* weights,
                            int n_weights, void* workspace, size_t workspace_bytes, void* stream);

/* Device bytes convrot_mlp needs: both packed activations, H and the GEMM's
 * hand-over words (CONVROT_GEMM_SYNC_BYTES). */
size_t convrot_mlp_workspace_size(int64_t M, int64_t K, int64_t N_up);

/*
 * convrot_mlp -- an up linear, an activation and a down linear on the device
 * (the transformer MLP built from two convrot linears):
 *   Y_up = float(Q_x Q_up^T) * s_x * s_up + b_up,
 *   H = act(Y_up), applied in the up GEMM's epilogue (fp32 [M, N_up]),
 *   Y = float(Q_h Q_down^T) * s_h * s_down + b_down  (H packed with G_down).
 *   X        [M,K] fp32/fp16 activations.
 *   up       the up linear's descriptor: q16 [N_up,K] (or packed 4-bit q4),
 *            scale, bias, kchunk as in convrot_linear; Y = NULL (H stays in
 *            the workspace) or an fp32 [M,N_up] device array that receives H.
 *            With CONVROT_ACT_SWIGLU, `up` points to TWO descriptors, the gate
 *            linear then the up linear (same N_up, binary16 weights; "ggml
 *            operator extensions", sd.cpp integration: split SwiGLU of two
 *            GEMMs sharing the quantized input), and H = silu(gate) * up;
 *            the first descriptor's Y receives H.
 *   activation  CONVROT_ACT_NONE, CONVROT_ACT_GELU or CONVROT_ACT_SWIGLU.
 *   down     weight of the down linear: q16 [N_down,N_up] (or q4), ...; Y [M,N_down].
 *   G_up / G_down  group sizes (4^n) dividing K / N_up.
 *   workspace  >= convrot_mlp_workspace_size(M, K, N_up) bytes.
 * Errors: ERR_ARG, ERR_GROUP, ERR_ALIGN, ERR_ALIAS, ERR_WORKSPACE,
 *         ERR_UNSUPPORTED (split SwiGLU with packed 4-bit weights), ERR_CUDA.
 */
int convrot_mlp(const void* X, int x_dtype, int64_t M, int64_t K, int G_up,
                const convrot_weight* up, int activation, int G_down,
                const convrot_weight* down, void* workspace, size_t workspace_bytes,
                void* stream);

/*
 * convrot_mlp_host_workspace_size -- device bytes convrot_mlp_host needs: two
 * sets of chunk buffers (input rows, output rows) and one convrot_mlp
 * workspace for a chunk. chunk_rows = 0 picks the default (1536 rows).
 * Returns 0 for invalid arguments.
 */
size_t convrot_mlp_host_workspace_size(int64_t M, int64_t K, int x_dtype, int64_t N_up,
                                       int64_t N_down, int64_t chunk_rows);

/*
 * convrot_mlp_host -- convrot_mlp with X and Y in HOST memory (weights,
 * scales and biases in device memory). The rows are independent, so they are
 * processed in chunks of chunk_rows: each chunk is copied in on
 * copy_in_stream, run through convrot_mlp on `stream`, and its rows of Y
 * copied out on copy_out_stream, so transfers overlap the other chunks'
 * compute. Results equal convrot_mlp's bit for bit. Host arrays should be
 * pinned for the transfers to overlap.
 *   X_host     [M,K] fp32/fp16 host array;  Y_host [M,N_down] fp32 host array.
 *   up, activation, down, G_up, G_down: as convrot_mlp; the descriptors' Y
 *              fields are ignored (H stays in the workspace, Y goes to Y_host).
 *   chunk_rows rows per chunk (0 = 1536; chunks much smaller than that leave
 *              the down GEMM's tiles on few SMs).
 *   workspace  device scratch, >= convrot_mlp_host_workspace_size(...).
 *   stream, copy_in_stream, copy_out_stream: as convrot_linear_host.
 * Errors: as convrot_mlp.
 */
int convrot_mlp_host(const void* X_host, int x_dtype, int64_t M, int64_t K, int G_up,
                     const convrot_weight* up, int activation, int G_down, const convrot_weight* down,
                     float* Y_host, int64_t chunk_rows, void* workspace, size_t workspace_bytes,
                     void* stream, void* copy_in_stream, void* copy_out_stream);

/*
 * convrot_linear_swiglu -- split SwiGLU of two linears that share an input
 * ("ggml operator extensions", sd.cpp integration: two INT8 GEMMs sharing a
 * quantized input fuse with split SwiGLU, a paired-column iterator reads the
 * separate gate and up weights, and the GEMM epilogue writes only the
 * activated output): X is packed once, and one GEMM computes
 *   g = float(Q_x Q_gate^T) * s_x * s_gate + b_gate,
 *   u = float(Q_x Q_up^T) * s_x * s_up + b_up,
 *   h = silu(g) * u = (g / (1 + exp(-g))) * u   (fp32: the hardware base-2
 *       exponential and a correctly rounded reciprocal, relative error of a
 *       few 1e-7),
 * writing h only.
 *   gate_up  host array of two descriptors: the gate linear, then the up
 *            linear; binary16 weights (q16), the same N (N % 4 == 0); h is
 *            written to gate_up[0].Y, [M,N] fp32 (gate_up[1].Y is unused).
 *   workspace  at least convrot_linear_workspace_size(M, K) bytes.
 * Errors: ERR_ARG, ERR_GROUP, ERR_ALIGN, ERR_ALIAS, ERR_WORKSPACE,
 *         ERR_UNSUPPORTED, ERR_CUDA.
 */
int convrot_linear_swiglu(const void* X, int x_dtype, int64_t M, int64_t K, int G,
                          const convrot_weight* gate_up, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Size of the fixed device array that convrot_linear_noalloc uses (32 MiB). */
#define CONVROT_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * convrot_linear_noalloc -- convrot_linear for callers that cannot allocate
 * device memory: a plugin that a host framework hands only its input and
 * output buffers, or a latency-bound loop where cudaMalloc (which can
 * synchronize the device) is not allowed. The pages have no counterpart; this
 * entry point is a property of this library, not of the method.
 *   Arguments and results as convrot_linear, without the workspace: the
 *   packed activation lives in one library-owned device array of
 *   CONVROT_NOALLOC_SCRATCH_BYTES bytes per GPU, held by every GPU that loads
 *   the library until the process exits. It must hold
 *   round256(M*K*2) + round256(M*4) bytes (round256 = round up to a multiple
 *   of 256), e.g. M = 4608, K = 3072 fits; larger calls return
 *   CONVROT_ERR_SCRATCH without launching anything.
 * The call allocates nothing. Its first call on a device looks up the array's
 * device address (cudaGetSymbolAddress) and remembers it with the identity of
 * the current CUDA context; a call in another context (e.g. after
 * cudaDeviceReset) looks it up again. Make the first call on a device, and
 * the first after a reset, before any stream capture. Every call on a device
 * shares the one array: calls that overlap on the GPU (different streams, or
 * host threads sharing a device) race and must be serialized by the caller.
 * Errors: ERR_ARG, ERR_GROUP, ERR_ALIGN, ERR_ALIAS, ERR_UNSUPPORTED,
 *         ERR_SCRATCH, ERR_CUDA.
 */
int convrot_linear_noalloc(const void* X, int x_dtype, int64_t M, int64_t K, int G,
                           const convrot_weight* weights, int n_weights,
                           void* stream);

/*
 * convrot_test_handover_timeout -- a test of the GEMM's timeout path, not part
 * of the method: convrot_linear_packed (binary16 weights, the hand-over words
 * in `workspace`) with every bounded device wait of the launch limited to
 * wait_ns nanoseconds, and the CTA pairs that finish split tiles waiting for a
 * hand-over value that no pair publishes. On a shape whose last wave is split
 * (e.g. M = 4608 with three 3072 x 3072 linears), those waits give up: the
 * kernel records CONVROT_ERR_TIMEOUT in the device's error word, skips its
 * remaining work, waits (bounded) for its copies in flight, releases its tensor
 * memory and exits; the outputs are incomplete. convrot_device_status then
 * returns CONVROT_ERR_TIMEOUT and clears the word; the device, the stream and
 * the workspace stay usable (the next launch publishes new hand-over values).
 * Nothing traps or hangs.
 * Errors: ERR_ARG (also wait_ns == 0 or packed 4-bit weights), ERR_ALIGN,
 *         ERR_WORKSPACE, ERR_OVERFLOW, ERR_ALIAS, ERR_UNSUPPORTED, ERR_CUDA.
 */
int convrot_test_handover_timeout(const uint16_t* Q_x16, const float* s_x, int64_t M, int64_t K,
                                  const convrot_weight* weights, int n_weights, void* workspace,
                                  size_t workspace_bytes, uint64_t wait_ns, void* stream);

/*
 * convrot_test_unscale_sweep -- a test of the GEMM epilogue's unscaling step,
 * not part of the method. The epilogue divides by a linear's input scale a
 * without a division per element (Markstein's correction step: r = RN(1/a),
 * q0 = RN(y r), RN(q0 + (y - q0 a) r) with the remainder exact in one FMA),
 * which equals the IEEE quotient while a, y and the quotient stay in the
 * normal range (a in [2^-20, 2^20], nonzero |y| in [2^-100, 2^100]; the
 * epilogue takes the IEEE division elsewhere). This call runs that step, on
 * the GPU, for each divisor divisors[i] (device, fp32, 16-byte aligned) and
 * every one of the 2^23 values y = 1.m * 2^y_exp, against the IEEE division.
 *   mismatches  device uint64, 8-byte aligned: the count of results that
 *               differ in any bit is added to it.
 *   first       device uint64: lowered (atomic min) to (i << 32 | bits of y)
 *               of the smallest differing pair; set it to ~0 beforehand.
 *   n_divisors  1 .. 65535;  y_exp  -98 .. 97.
 * Asynchronous on `stream`. Errors: ERR_ARG, ERR_ALIGN, ERR_CUDA.
 */
int convrot_test_unscale_sweep(const float* divisors, int n_divisors, int y_exp, uint64_t* mismatches,
                               uint64_t* first, void* stream);

/*
 * convrot_device_status -- synchronizes `stream`, then returns and clears the
 * device's sticky error word: CONVROT_OK, or CONVROT_ERR_TIMEOUT when a
 * kernel's bounded wait on a TMA or tensor-core completion barrier gave up
 * (the kernel then skipped its remaining work and released its resources).
 */
int convrot_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CONVROT_H */
