/*
 * vbq.h: C ABI of the VBQ mixed-bit decode library (sm_103a).
 *
 * VBQ (Variable Bit-width Quantization) stores a linear layer's weights packed.
 * Every run of 64 consecutive weights along the input dimension has its own
 * bit-width b_g from {1,2,4,8}. Source: "Variable Bit-width Quantization:
 * Learning Per-Group Precision for 'Bigger-but-Smaller' Language Models",
 * abstract: once learned, the per-group allocation is stored as packed low-bit
 * codes, and kernels that dequantize inside the multiply speed up token-by-token
 * decode, which memory bandwidth limits. The pages fix no code grid; this
 * library uses
 *
 *     w = s_g * (q - (2^b_g - 1) / 2),   s_g fp16,   q unsigned in [0, 2^b_g - 1],
 *
 * where group g of row r covers input columns [64g, 64g + 63].
 *
 * Conventions for every call:
 *  - "host" pointers are ordinary CPU memory, and "device" pointers are CUDA
 *    device memory of the current device (for example a torch tensor's
 *    data_ptr()). bf16 and fp16 values are passed as uint16_t bit patterns.
 *  - stream is a cudaStream_t cast to void*. NULL means the legacy default
 *    stream. Device work is enqueued on the stream asynchronously unless the
 *    call says otherwise. Output buffers are written when the stream reaches
 *    the work.
 *  - Arguments are validated on the host before any device work is enqueued.
 *    On a validation error nothing is enqueued and nothing is written.
 *  - A launch failure returns VBQ_ERR_CUDA, read with cudaGetLastError and
 *    without an implicit synchronization. vbq_last_error() gives the text.
 *  - Calls that share one vbq_matrix or vbq_model must not overlap on the GPU
 *    if the object holds per-call state (vbq_model does). Calls on different
 *    objects may run concurrently.
 */
#ifndef VBQ_H
#define VBQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define VBQ_API __attribute__((visibility("default")))
#else
#define VBQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct vbq_matrix vbq_matrix; /* packed matrix, owned by the library */
typedef struct vbq_model vbq_model;   /* decode-step stack, owned by the library */

typedef enum {
  VBQ_OK = 0,
  VBQ_ERR_INVALID_ARG = 1,  /* null pointer, bad count, mismatched objects */
  VBQ_ERR_SHAPE = 2,        /* K not a multiple of 64, sizes out of range */
  VBQ_ERR_CODE_RANGE = 3,   /* a code q >= 2^b of its group */
  VBQ_ERR_BITS = 4,         /* a bit-width outside {1,2,4,8} */
  VBQ_ERR_CUDA = 5,         /* a CUDA runtime call or a launch failed */
  VBQ_ERR_OOM = 6,          /* device or host allocation failed */
  VBQ_ERR_DEVICE_CHECK = 7, /* a kernel reported a failed internal check (bounded wait ran out) */
  VBQ_ERR_UNSUPPORTED = 8   /* valid request this build does not serve */
} vbq_status;

/* Sizes and storage accounting of a packed matrix. */
typedef struct {
  int64_t N, K;          /* rows (outputs) and columns (inputs) */
  int64_t code_bytes;    /* sum over groups of 64*b/8: the packed code bits */
  int64_t meta_bytes;    /* scales, row indices, step descriptors and offsets, tile table */
  int64_t total_bytes;   /* device bytes of the packed matrix */
  double mean_bits;      /* 8*code_bytes/(N*K): mean code bits per weight */
  int32_t n_tiles;       /* 256-row tiles of the layout */
  int32_t n_steps;       /* 32-entry steps of the layout (layout.h) */
  int64_t groups_by_bits[4]; /* groups at 1, 2, 4 and 8 bits */
} vbq_info;

/* Shapes of a decoder-only stack whose projections are VBQ matrices. */
typedef struct {
  int32_t n_layers;
  int32_t d;           /* model width */
  int32_t n_heads;     /* query heads */
  int32_t n_kv_heads;  /* key/value heads (n_heads % n_kv_heads == 0) */
  int32_t head_dim;
  int32_t d_ff;        /* SwiGLU hidden width */
  int32_t vocab;
  float rms_eps;       /* RMSNorm epsilon (unit gain) */
} vbq_model_desc;

/* Text for a status code. Static storage. */
VBQ_API const char* vbq_status_str(vbq_status s);

/* Detail of the last error raised on the calling host thread ("" if none). */
VBQ_API const char* vbq_last_error(void);

/*
 * vbq_quantize_rtn: dense weights onto the VBQ grid at a given bit map, by
 * absmax round-to-nearest per group (host; tooling for measuring how far a
 * quantized model's logits move from the dense ones, VBQ abstract's
 * distributional analysis). For each group: s = max|w| / c_b rounded to fp16
 * (nearest, ties to even), c_b = (2^b - 1)/2; q = the nearest integer (ties to
 * even) to w / s + c_b, clipped to [0, 2^b - 1]; q = 0 where s = 0. The pages
 * learn the allocation and the weights; this encoding is the plainest one for
 * a given allocation.
 *  W           host, float [N][K] row-major, finite
 *  bits        host, uint8 [N][K/64], each in {1,2,4,8}
 *  codes       host, uint8 [N][K] (out), ready for vbq_pack
 *  scales_f16  host, uint16 [N][K/64] (out), fp16 bit patterns
 * Errors: VBQ_ERR_SHAPE (K % 64), VBQ_ERR_BITS, VBQ_ERR_INVALID_ARG (NULL,
 * non-finite weight, a scale above fp16's range).
 */
VBQ_API vbq_status vbq_quantize_rtn(const float* W, int64_t N, int64_t K, const uint8_t* bits, uint8_t* codes,
                            uint16_t* scales_f16);

/*
 * Training-side fake quantization (VBQ abstract: precision learned by a
 * Gumbel-Softmax relaxation over precision logits, alternating with the
 * weights, gradients through the rounding by the straight-through estimator;
 * the formulas are this library's plainest reading). Per group g of 64
 * weights along K and bit-width b in {1,2,4,8} (index 0..3):
 *   Q_b(w) = s_b (q - c_b), c_b = (2^b - 1)/2, s_b = max|w_g| / c_b,
 *   q = rint(w r_b + c_b), r_b = c_b / max|w_g|, clipped to [0, 2^b - 1] (fp32, each operation
 *   rounded once; Q_b = 0 for an all-zero group),
 *   pi_b = softmax_b((alpha_gb - log(-log u_gb)) / tau),   W_mix = sum_b pi_b Q_b(W).
 * Backward for G = dL/dW_mix: dW = G (straight through, sum_b pi_b = 1), and
 * dalpha_b = (pi_b / tau) (D_b - sum_b' pi_b' D_b'), D_b = sum over the group of G Q_b(W).
 *  W, G, W_mix, dW  device, float [N][K] row-major, 16-byte aligned; K % 64 == 0
 *  alpha, u, dalpha device, float [N][K/64][4]; u in (0, 1), drawn by the caller
 *  tau              > 0
 * One launch each, eight lanes per group. Errors: VBQ_ERR_SHAPE, VBQ_ERR_INVALID_ARG, VBQ_ERR_CUDA.
 */
VBQ_API vbq_status vbq_fakequant_forward(const float* W, const float* alpha, const float* u, float tau, int64_t N,
                                 int64_t K, float* W_mix, void* stream);
VBQ_API vbq_status vbq_fakequant_backward(const float* W, const float* alpha, const float* u, float tau,
                                  const float* G, int64_t N, int64_t K, float* dW, float* dalpha, void* stream);

/*
 * vbq_pack: logical codes + per-group bit map + scales -> device layout.
 * Source: the VBQ abstract (a fixed per-group allocation is stored as packed
 * low-bit codes). The layout is this library's own design.
 *
 *  codes      host, uint8 [N][K] row-major; codes[r][k] < 2^bits[r][k/64]
 *  bits       host, uint8 [N][K/64]; each value in {1,2,4,8}
 *  scales_f16 host, uint16 [N][K/64]; the fp16 bit pattern of s_g
 *  N, K       N >= 0, K >= 0, K % 64 == 0, K/64 <= 65535, N < 2^31
 *  stream     the upload is enqueued on it. The call returns after the upload
 *             has finished, so the host arrays may be freed on return.
 *  out        receives the new handle. Release it with vbq_matrix_free.
 *
 * The host arrays stay owned by the caller. The handle owns its device memory,
 * allocated here with cudaMalloc on the current device.
 * Errors: VBQ_ERR_INVALID_ARG (null pointers), VBQ_ERR_SHAPE, VBQ_ERR_BITS,
 * VBQ_ERR_CODE_RANGE (nothing allocated), VBQ_ERR_OOM, VBQ_ERR_CUDA.
 */
VBQ_API vbq_status vbq_pack(const uint8_t* codes, const uint8_t* bits, const uint16_t* scales_f16,
                    int64_t N, int64_t K, void* stream, vbq_matrix** out);

/* Frees the handle and its device memory. It synchronizes the device first. NULL is a no-op. */
VBQ_API void vbq_matrix_free(vbq_matrix* m);

/* Fills *info from the handle. Host only, no device work. */
VBQ_API vbq_status vbq_matrix_info(const vbq_matrix* m, vbq_info* info);

/*
 * vbq_dequant: packed -> fp32 W (for checking). W[r][k] = s * (q - c_b),
 * computed exactly in fp32 (an fp16 scale has 11 significant bits and q - c_b
 * at most 9), so it equals the oracle bit for bit.
 * Source: the VBQ abstract (per-group bit-widths from {1,2,4,8}, stored as
 * packed low-bit codes); the grid w = s * (q - c_b) is this library's, as
 * stated at the top of this file.
 *  m      from vbq_pack, on the current device
 *  W_dev  device, float [N][K] row-major, caller-owned; every element is written.
 * One CTA per 1024-row super-tile; enqueued on stream.
 * Errors: VBQ_ERR_INVALID_ARG (NULL, misaligned or other-device arguments), VBQ_ERR_CUDA.
 */
VBQ_API vbq_status vbq_dequant(const vbq_matrix* m, float* W_dev, void* stream);

/*
 * vbq_gemv: y = W x for one bf16 activation vector.
 * Source: the VBQ abstract (dequantization fused with the multiply, for
 * batch-1 autoregressive decode).
 *  x_dev  device, bf16 [K] (uint16 bit patterns), 4-byte aligned
 *  y_dev  device, float [N], 4-byte aligned; every element is written (zeros when K == 0)
 * Arithmetic: each (row, group) contribution is rounded to an integer in units
 * of 2^-F, F = 30 - (e(L1) + e(max|x|)) (e(v): v < 2^e; L1 the largest row sum
 * of |w|), and summed in 32- then 64-bit integers: results do not depend on
 * timing, and the error per element is within the bound of the parity tests
 * (far below the normalized 2e-3 bar). One launch. K <= 16384 (larger K takes
 * the tensor-core path when the matrix is eligible, else VBQ_ERR_UNSUPPORTED).
 * Errors: VBQ_ERR_INVALID_ARG, VBQ_ERR_UNSUPPORTED, VBQ_ERR_CUDA.
 */
VBQ_API vbq_status vbq_gemv(const vbq_matrix* m, const uint16_t* x_dev, float* y_dev, void* stream);

/*
 * vbq_gemm_smallbatch: Y[j] = W X[j] for a batch of 1..64 bf16 vectors.
 * Source: the VBQ abstract (fused dequantize-and-multiply); with several
 * activation columns the product is a dense contraction, which this library
 * runs on the tensor cores.
 *  X_dev  device, bf16 [B][K] row-major, 4-byte aligned
 *  B      1 <= B <= 64 (else VBQ_ERR_INVALID_ARG, nothing written)
 *  Y_dev  device, float [B][N] row-major, 4-byte aligned; every element is written
 * B <= 3: one vbq_gemv launch per column. B >= 4: three launches (per-column
 * powers of two that keep x inside fp16's range, the fp16 activation tiles,
 * and one tcgen05 dequant-MMA launch for all columns), with weights rounded
 * once to fp16 and fp32 accumulation. Matrices whose scales exceed 512 (their
 * fp16 weights would overflow) take the per-column path at every B.
 * Errors: VBQ_ERR_INVALID_ARG, VBQ_ERR_OOM (first tensor-core call: its plan), VBQ_ERR_CUDA.
 */
VBQ_API vbq_status vbq_gemm_smallbatch(const vbq_matrix* m, const uint16_t* X_dev, int32_t B, float* Y_dev,
                               void* stream);

/*
 * vbq_gemm: Y[j] = W X[j] for any batch (prefill-sized included), in blocks of
 * 64 columns, each a vbq_gemm_smallbatch call on the same stream (so the
 * weights stream once per block of 64). Layouts and errors as
 * vbq_gemm_smallbatch; 1 <= B <= 2^24.
 */
VBQ_API vbq_status vbq_gemm(const vbq_matrix* m, const uint16_t* X_dev, int64_t B, float* Y_dev, void* stream);

/*
 * vbq_model_create: bind the packed projections of a decoder stack for vbq_decode_step.
 * Source: the VBQ abstract (token-by-token decode through VBQ projections);
 * the stack's shape and glue are this library's reading (see vbq_decode_step).
 *  desc  host; the shapes. Each matrix must match its projection's (N, K).
 *  mats  host array of n_layers*7 + 1 handles: per layer q, k, v, o, gate, up,
 *        down (in that order), then the LM head. The handles must stay alive
 *        while the model exists. The model does not own them.
 *  out   receives the model. It owns a device workspace (per projection group:
 *        64-bit sums, float outputs, arrival counters, flags) and the work
 *        plans of every GEMV of the step, built here once.
 * Limits: d and n_heads*head_dim at most 8192, d_ff at most 16384, all
 * multiples of 64 (VBQ_ERR_UNSUPPORTED / VBQ_ERR_SHAPE otherwise).
 * Errors: VBQ_ERR_INVALID_ARG, VBQ_ERR_SHAPE, VBQ_ERR_UNSUPPORTED, VBQ_ERR_OOM, VBQ_ERR_CUDA.
 */
VBQ_API vbq_status vbq_model_create(const vbq_model_desc* desc, const vbq_matrix* const* mats, vbq_model** out);

VBQ_API void vbq_model_free(vbq_model* model);

/*
 * vbq_decode_step: one batch-1 decode step (position 0) through the stack.
 * Source: the VBQ abstract (decode whose speed is set by memory bandwidth).
 * The glue between projections is this library's reading, since the pages
 * give no architecture:
 *   h = x;  per layer:  u = bf16(rmsnorm(h)); q,k,v = Wq u, Wk u, Wv u;
 *                       a = bf16(v of each head's kv group)   (softmax over one key = 1)
 *                       h += Wo a;  u = bf16(rmsnorm(h));
 *                       h += Wdown bf16(silu(Wgate u) * Wup u)
 *   logits = Whead bf16(rmsnorm(h))
 * The residual h is fp32; every projection sums in fixed point as vbq_gemv
 * does, so a step's logits do not depend on timing (two steps on the same
 * input agree bit for bit).
 * The step is one cooperative launch of a persistent kernel (one CTA per SM).
 * Dependent projections are linked by per-super-tile flags, not grid barriers:
 * the CTA that adds last into 1024 output rows converts them and sets their
 * flag; a CTA starts a projection once the rows it reads are flagged. Its
 * activations live in the model's workspace, so steps on the same model must
 * not overlap. Residual values must stay below 2^57 in magnitude (the RMSNorm
 * sums of squares are fp32).
 *  x_dev       device, bf16 [d], 4-byte aligned
 *  logits_dev  device, float [vocab], 4-byte aligned
 * Errors: VBQ_ERR_INVALID_ARG (NULL, misaligned, model on another device),
 * VBQ_ERR_CUDA; a bounded wait that ran out is reported by vbq_device_check (code 3).
 */
VBQ_API vbq_status vbq_decode_step(vbq_model* model, const uint16_t* x_dev, float* logits_dev, void* stream);

/*
 * Same step through host buffers: copies x_host (bf16 [d]) in, runs the step,
 * copies logits (float [vocab]) out and synchronizes the stream before
 * returning. Pinned host memory makes the copies asynchronous DMA.
 */
VBQ_API vbq_status vbq_decode_step_host(vbq_model* model, const uint16_t* x_host, float* logits_host, void* stream);

/*
 * The decode step at a position above 0 ("autoregressive decode", VBQ
 * abstract): the same projections and glue as vbq_decode_step, with each
 * layer's attention over a bf16 KV cache in place of the position-0 shortcut.
 * Per layer, q, k and v (the [q;k;v] projection's outputs, rounded to bf16)
 * are turned by the rotary embedding at pos (as vbq_rope_append: rotate-half
 * pairing, theta^(-2i/d), fp64 rounded to fp32 then bf16); k and v are written
 * to the layer's cache at pos; each query head attends over positions
 * 0 .. pos of its kv head (as vbq_attention_decode); and o reads the result,
 * rounded to bf16. At pos = 0 the logits equal vbq_decode_step's bit for bit.
 *
 * vbq_model_set_context: allocates the caches of every layer for max_context
 * positions (bf16 [n_kv_heads][max_context][head_dim] per layer for K and for
 * V, zeroed) and the programs of the segmented step; 0 frees them. theta is
 * the rotary base (10000 in the usual models). Needs head_dim 64 or 128 and at
 * most 8 query heads per kv head; max_context <= 65536. Synchronizes the
 * device.
 * vbq_model_kv_cache: the device addresses of layer's K and V caches (owned by
 * the model) and their position stride (max_context), for a caller that fills
 * or reads them.
 * vbq_decode_step_at: x_dev bf16 [d] and logits_dev float [vocab] as in
 * vbq_decode_step; 0 <= pos < max_context; positions below pos must already
 * hold the caller's keys and values. The step runs as n_layers + 1 launches of
 * the decode kernel (cut after each layer's [q;k;v]) with each layer's
 * attention between them; the trace, when enabled, covers it as it covers
 * vbq_decode_step. Errors as vbq_decode_step, and VBQ_ERR_INVALID_ARG without
 * a context.
 */
VBQ_API vbq_status vbq_model_set_context(vbq_model* model, int32_t max_context, double rope_theta);
VBQ_API vbq_status vbq_model_kv_cache(const vbq_model* model, int32_t layer, uint16_t** k_cache, uint16_t** v_cache,
                              int64_t* stride);
VBQ_API vbq_status vbq_decode_step_at(vbq_model* model, const uint16_t* x_dev, int32_t pos, float* logits_dev,
                              void* stream);

/*
 * Teacher-forcing trace. When enabled, each step also records, for every
 * projection p (layer-major, q..down per layer, then the head), the bf16
 * input it consumed and its fp32 output. vbq_model_trace_info gives the
 * offsets. The buffers live in the model, so nothing is recorded unless
 * enabled. Enabling re-uploads the step's item list (it synchronizes the device).
 */
VBQ_API vbq_status vbq_model_set_trace(vbq_model* model, int32_t enable);
/* in_off/out_off: host int64 [n_layers*7+1]; element offsets into the buffers below. */
VBQ_API vbq_status vbq_model_trace_info(const vbq_model* model, int64_t* in_off, int64_t* out_off,
                                int64_t* in_total, int64_t* out_total);
/* Copies the trace to host arrays (uint16 [in_total], float [out_total]). Synchronizes the device. */
VBQ_API vbq_status vbq_model_read_trace(const vbq_model* model, uint16_t* in_host, float* out_host);

/*
 * Dense bf16 GEMV baseline on the same shapes: y = W x, W bf16 [N][K]
 * row-major (device), x bf16 [K] (device), y float [N] (device). fp32
 * accumulation. K % 8 == 0.
 */
VBQ_API vbq_status vbq_dense_gemv_bf16(const uint16_t* W_dev, const uint16_t* x_dev, float* y_dev, int64_t N,
                               int64_t K, void* stream);

/*
 * Many dense bf16 GEMVs in one launch (the dense baseline of a whole decode
 * step, without a launch per matrix): for each job j, y_j = W_j x_j with the
 * layout and arithmetic of vbq_dense_gemv_bf16. Rows of all jobs are dealt to
 * the warps of one persistent grid in job order. jobs: host array of n_jobs
 * (at most VBQ_DENSE_MAX_JOBS) descriptors of device buffers, read before the
 * call returns. Every K % 8 == 0, 0 <= N, K < 2^31, W and x 16-byte aligned;
 * jobs with N == 0 are skipped, jobs with K == 0 get y = 0. An invalid job
 * fails the whole call before anything is launched. There is no counterpart
 * on the source pages: the pages compare against dense weights, and this is
 * the dense side of that comparison.
 */
#define VBQ_DENSE_MAX_JOBS 256
typedef struct {
  const uint16_t* W; /* bf16 [N][K], device */
  const uint16_t* x; /* bf16 [K], device */
  float* y;          /* float [N], device */
  int64_t N, K;
} vbq_dense_job;
VBQ_API vbq_status vbq_dense_gemv_bf16_many(const vbq_dense_job* jobs, int32_t n_jobs, void* stream);

/*
 * Decode attention for one new token over a bf16 KV cache (the other half of
 * a decode step beside the projections; the source pages name only
 * "autoregressive decode" in the VBQ abstract, so the operations below are the
 * standard definitions, read as stated).
 *
 * vbq_rope_append: rotary position embedding at position pos, rotate-half
 * pairing (for i < d/2 the pair (x_i, x_{i+d/2}) turns by the angle
 * pos * theta^(-2i/d)), computed in fp64, rounded to fp32 and then to bf16
 * (nearest even). q (bf16 [n_heads][head_dim], device) is turned in place;
 * k_new (bf16 [n_kv_heads][head_dim]) is turned into k_cache at position pos
 * and v_new copied into v_cache there. Caches: bf16
 * [n_kv_heads][kv_stride][head_dim], device. One launch.
 *
 * vbq_attention_decode: for each query head h (kv head g = h / (n_heads /
 * n_kv_heads)), out[h] = sum_j p_j v_g[j] with p = softmax_j(q_h . k_g[j] /
 * sqrt(head_dim)) over positions j < T. q bf16 [n_heads][head_dim], out float
 * [n_heads][head_dim], device. fp32 dot products and sums; each kv head's
 * positions are split into at most 64 spans (one CTA each, a running softmax
 * over sub-chunks of 64 positions) that the last CTA of the kv head merges in
 * span order, so results are deterministic. The library keeps a
 * per-device scratch for the merge (grown on demand; calls that overlap on
 * the GPU must not share a device).
 *
 * Both: head_dim 64 or 128, n_heads a multiple of n_kv_heads with at most 8
 * query heads per kv head; 1 <= T <= min(kv_stride, 65536); 0 <= pos <
 * kv_stride; theta > 1; q (for attention) and the caches 16-byte aligned.
 * A bad argument returns an
 * error with nothing launched. Device check code 5: a chunk copy never landed.
 */
VBQ_API vbq_status vbq_rope_append(uint16_t* q, const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_cache,
                           uint16_t* v_cache, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                           int64_t kv_stride, int32_t pos, double theta, void* stream);
VBQ_API vbq_status vbq_attention_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int64_t kv_stride,
                                int32_t T, float* out, void* stream);

/*
 * Reads and clears the device-side check word of the current device. Kernels
 * set it when a bounded wait runs out. Synchronizes the device. Returns
 * VBQ_OK, or VBQ_ERR_DEVICE_CHECK with *code set (code may be NULL).
 */
VBQ_API vbq_status vbq_device_check(int32_t* code);

/* Number of this library's kernel launches enqueued since the last reset (host counter). */
VBQ_API int64_t vbq_launch_count(int32_t reset);

/*
 * vbq_decode_step_noalloc: the step of vbq_decode_step for callers that may not
 * allocate device memory, or tie it to the model they step, at step time: for
 * example loops whose device memory is fixed before they start, or hosts that
 * hand out device memory only from their own pool. The pages have no
 * counterpart: this is an interface of this library.
 *
 * It launches the same kernel as vbq_decode_step with the step's scratch (per
 * projection group: 64-bit sums, float outputs, arrival counters, flags and
 * statistics) in one static device array instead of the model's workspace,
 * and gives the same logits bit for bit. The array has 4,194,304 8-byte words
 * (32 MiB) on every GPU that loads this library and lives until the process
 * exits. The call allocates nothing: no cudaMalloc, no cudaFree. It records no
 * trace, whether or not vbq_model_set_trace enabled one.
 *
 *  model       from vbq_model_create, on the current device
 *  x_dev       device, bf16 [d], 4-byte aligned
 *  logits_dev  device, float [vocab], 4-byte aligned
 *
 * Size limit: the model's scratch must fit the array (the 9B-shaped stack of
 * the tests needs about 2.2 million words). Larger models get VBQ_ERR_SHAPE,
 * the detail text gives the count, and nothing is enqueued.
 * Set-up: vbq_model_create looks up the array's device address with
 * cudaGetSymbolAddress on the model's device (once per device, with that
 * device current) and clears it, so the calls themselves do neither.
 * Sharing: every call on a device uses the same array. The sums and counters
 * must be zero when a step starts, and every step leaves them at zero; flags
 * hold a per-launch value, and every other value is written before it is read.
 * Calls that overlap on the GPU (two streams, or two host threads), with each
 * other or with vbq_decode_step on the same model, race and give undefined
 * results; serialize them.
 * Errors: VBQ_ERR_INVALID_ARG (NULL or misaligned pointers, model on another
 * device), VBQ_ERR_SHAPE (over the limit), VBQ_ERR_CUDA (the launch failed). A
 * bounded wait that runs out is recorded in the device check word; read it
 * with vbq_device_check.
 */
VBQ_API vbq_status vbq_decode_step_noalloc(vbq_model* model, const uint16_t* x_dev, float* logits_dev,
                                           void* stream);

/*
 * Test hooks; they change how later decode steps (vbq_decode_step and
 * vbq_decode_step_noalloc) behave in this process, and value 0 restores the
 * default.
 *  VBQ_DEBUG_WAIT_LIMIT     SM clock cycles a decode-step wait on another
 *                           CTA's flag may take before the kernel records
 *                           check code 3 and goes on (default 2e9, about a
 *                           second at 2 GHz).
 *  VBQ_DEBUG_NEVER_READY    nonzero: the waits look for a flag value that no
 *                           launch writes, so the first one runs out after
 *                           the limit and the rest give up at once. The step
 *                           completes with wrong logits and check code 3.
 *  VBQ_DEBUG_NOALLOC_WORDS  words of vbq_decode_step_noalloc's static array
 *                           that it may use (to test its size check).
 *  VBQ_DEBUG_ALLOC_CAP      bytes: a device allocation of this library above
 *                           the cap fails as if the device were out of memory
 *                           (VBQ_ERR_OOM), without reaching the driver.
 * Errors: VBQ_ERR_INVALID_ARG (unknown key, negative value).
 */
enum {
  VBQ_DEBUG_WAIT_LIMIT = 1,
  VBQ_DEBUG_NEVER_READY = 2,
  VBQ_DEBUG_NOALLOC_WORDS = 3,
  VBQ_DEBUG_ALLOC_CAP = 4
};
VBQ_API vbq_status vbq_debug_set(int32_t key, int64_t value);

#ifdef __cplusplus
}
#endif

#endif /* VBQ_H */
