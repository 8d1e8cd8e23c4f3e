/*
 * gpt2b300.h -- C ABI of a single-GPU GPT-2 training step for B300 (sm_103a).
 *
 * The step is the one the GPT-2 reproduction pages describe: forward and
 * backward of the pre-LN causal decoder (token + position embedding,
 * LayerNorm, QKV / projection / FC / FC-projection / LM-head matmuls, causal
 * multi-head attention, GELU, residuals), the softmax cross-entropy over the
 * padded vocabulary, global grad-norm clipping and AdamW on fp32 master
 * weights.  Sources (web pages, by title and section):
 *   [R]  "Let's reproduce GPT-2 (124M)" -- §Video özeti (mixed precision,
 *        flash attention, AdamW, warmup+cosine, gradient accumulation),
 *        §Bölümler 2 (GPT-2 nn.Module), §Bölümler 4 (cross-entropy loss and
 *        the overfit test).
 *   [L]  "llm.c kullanarak GPT-2 modelini düşük maliyetle yeniden uygulamak" --
 *        §Eğitimi çalıştırma (micro-batch -b, sequence length -t, total batch
 *        -d, recompute -r), §Eğitim süreci (clipping cures the early gradient
 *        explosion), §Kod yapısı (forward/backward of the Transformer).
 *   [G]  "Let's build GPT: from scratch" -- chapters 01:00:18 (position
 *        encoding), 01:02:00 / 01:16:56 (scaled self-attention, scale
 *        1/sqrt(head_size), errata: future tokens cannot communicate),
 *        01:21:59 (multi-head), 01:24:25 (feed-forward), 01:26:48 (residual),
 *        01:32:51 (LayerNorm).
 *
 * Conventions for every call
 *  - Return value: GPT2_OK (0) or a negative GPT2_ERR_* code; no C++ exception
 *    crosses this boundary.  gpt2_strerror() names a code.
 *  - Device pointers ("d_" prefix or documented as device) must point to memory
 *    of the current CUDA device; host pointers ("host_") to ordinary host memory.
 *  - All matrices are row-major.  Linear weights are [out_features, in_features].
 *  - bf16 buffers hold IEEE bfloat16 bit patterns (uint16 storage).
 *  - Work is enqueued on the CUDA stream given at build (model calls) or per call
 *    (op calls); calls return after enqueueing unless documented otherwise.
 */
#ifndef GPT2B300_H
#define GPT2B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define GPT2_OK                    0
#define GPT2_ERR_BAD_CONFIG       -1  /* config fields inconsistent or unsupported */
#define GPT2_ERR_BAD_SHAPE        -2  /* B > cfg.B, T > cfg.T, sizes <= 0 or misaligned */
#define GPT2_ERR_BAD_TOKEN        -3  /* a token or target outside [0, V) (seen on device) */
#define GPT2_ERR_ARENA_TOO_SMALL  -4  /* arena_bytes < gpt2_arena_bytes(cfg) */
#define GPT2_ERR_CUDA             -5  /* a CUDA runtime/driver call failed */
#define GPT2_ERR_NONFINITE        -6  /* loss or grad norm is NaN/Inf (update skipped) */
#define GPT2_ERR_TIMEOUT          -7  /* a bounded device wait gave up (no hang) */
#define GPT2_ERR_BAD_ARG          -8  /* NULL pointer, bad id, bad enum, short buffer */
#define GPT2_ERR_UNSUPPORTED      -9  /* device is not sm_103 / feature not built */
#define GPT2_ERR_STATE           -10  /* call order violated (backward without forward) */

/* ---- model configuration -------------------------------------------------- */
#define GPT2_DTYPE_FP32 0  /* all activations fp32, SIMT fp32 matmuls (no TF32) */
#define GPT2_DTYPE_BF16 1  /* bf16 activations, tcgen05 bf16 matmuls, fp32 master/grads/state */

typedef struct {
    int L;              /* layers */
    int C;              /* channels; head dim = C / H */
    int H;              /* heads */
    int V;              /* real vocabulary size: logits v >= V are masked out of the loss */
    int Vp;             /* padded vocabulary (rows of wte), Vp >= V */
    int T;              /* maximum sequence length (rows of wpe) */
    int B;              /* maximum micro-batch */
    int dtype;          /* GPT2_DTYPE_* */
    int recompute_gelu; /* 1: do not store GELU(h); recompute it in backward ([L] -r) */
    int fp8_forward;    /* 1 (bf16 only, C >= 128): the four per-block projections of the
                           forward (QKV, attention output, FC, FC output) multiply E4M3
                           codes -- activations scaled per row, weights per tensor -- and
                           the backward stays bf16 (straight-through); 0: bf16 throughout */
    int fused_lm_head;  /* 1 (bf16 only): the LM head and the cross-entropy without a [B*T, Vp]
                           logits buffer.  The forward's LM-head product keeps per-row
                           (max, sum exp) partials and the target logit in its epilogue; the
                           backward recomputes the logits in row chunks of up to 8,192
                           positions, turns them into dlogits in the epilogue and runs the
                           two LM-head gradient products per chunk.  A forward without
                           targets then serves at most that many positions (else
                           GPT2_ERR_UNSUPPORTED).  0: logits stored, classifier pass */
} gpt2_config;

typedef struct gpt2_model gpt2_model; /* opaque host handle */

/*
 * Device bytes a model of this config needs: fp32 params, grads, AdamW m and v,
 * bf16 weight copy (bf16 mode), activations for B*T tokens and scratch.
 * Returns 0 for an invalid config.
 */
size_t gpt2_arena_bytes(const gpt2_config *cfg);

/*
 * Build a model in a caller-owned device arena (>= gpt2_arena_bytes, 256-byte
 * aligned) and initialise it from `seed`: every 2-D weight N(0, 0.02^2), the
 * attention and FC output projections N(0, (0.02/sqrt(2L))^2), biases 0,
 * LayerNorm gains 1 ([R] §Bölümler 2); wte rows v >= V are 0.  The normal draws
 * are SplitMix64 counter draws + Box-Muller in double rounded once to fp32
 * (draw(seed, tensor_id, 2i) / (.., 2i+1)), computed on the host and copied
 * once.  Grads, m and v are zeroed; the AdamW step counter is 0.
 * `cuda_stream` (cudaStream_t, may be NULL for the legacy stream) is used by
 * every later model call.  The arena and stream stay owned by the caller and
 * must outlive the model; the handle owns only host memory.  Synchronises the
 * stream before returning.
 */
int gpt2_build(const gpt2_config *cfg, uint64_t seed, void *dev_arena, size_t arena_bytes,
               void *cuda_stream, gpt2_model **out);

/*
 * Forward pass over d_tokens [B, T] (device int32, B <= cfg.B, T <= cfg.T).
 * With d_targets (device int32 [B, T]) it also runs the fused classifier: the
 * loss is the mean over the B*T positions of logsumexp(z[0..V)) - z[target]
 * ([R] §Bölümler 4) and the logits buffer is overwritten in place by
 * dloss/dz (for a unit loss weight; backward applies grad_scale), with
 * dz[v >= V] = 0.  The scalar loss is copied to *loss_out (host), which
 * synchronises the stream.  With d_targets == NULL only the logits are
 * computed (no sync; loss_out untouched).  Out-of-range tokens give
 * GPT2_ERR_BAD_TOKEN (their rows are treated as token 0).
 */
int gpt2_forward(gpt2_model *m, const int32_t *d_tokens, const int32_t *d_targets, int B, int T,
                 float *loss_out);

/*
 * Backward of grad_scale * loss of the last forward with targets:
 * grads += d(grad_scale * loss)/d(params).  grad_scale = 1/accumulation_steps
 * gives the averaged gradient of [R] §Video özeti (gradient accumulation).
 * GPT2_ERR_STATE if no forward with targets preceded it.
 */
int gpt2_backward(gpt2_model *m, float grad_scale);

/* grads = 0 (enqueued). */
int gpt2_zero_grad(gpt2_model *m);

/*
 * CUDA-graph replay of the forward and backward launch sequences (on by
 * default).  The first gpt2_forward / gpt2_backward of a shape (B, T, with or
 * without targets; for the backward also grad_scale) launches its kernels
 * directly, the second captures them into a graph on a stream the library
 * creates and destroys, later calls replay that graph on the model's stream:
 * the same kernels with the same arguments, without the per-launch gaps.
 * Tokens and targets are copied into the model's own buffers before the
 * graph runs, so callers may pass different buffers on every call.  While
 * per-launch profiling is on (gpt2_profile) the kernels run directly.
 * enable = 0 drops the cached graphs and launches directly from then on.
 * GPT2_ERR_BAD_ARG for a NULL model or enable other than 0 or 1.
 */
int gpt2_set_graphs(gpt2_model *m, int enable);

/* Largest top_k of gpt2_generate and gpt2_op_sample. */
#define GPT2_MAX_TOP_K 128

/*
 * Autoregressive sampling with a key/value cache ("llm.c kullanarak GPT-2
 * modelini düşük maliyetle yeniden uygulamak", §Sampling and §SSS: sampling
 * works, conditionally or not; "Let's reproduce GPT-2 (124M)", §Bölümler 3).
 * d_seq: device int32 [B, T_total], row-major.  Columns [0, T0) hold the
 * prompt; columns [T0, T_total) receive the sampled tokens.
 * 1 <= T0 < T_total <= cfg.T, 1 <= B <= cfg.B.
 * d_uniforms: device float [T_total - T0, B] in [0, 1); the draw that picks
 * column t of row b is d_uniforms[(t - T0) * B + b] (the caller owns the
 * random numbers).
 * The rule for column t: z = the logits of position t - 1 over v < V (rounded
 * to bf16 in bf16 mode); candidates = the top_k largest, equal values lower
 * index first; w_i = exp((z_i - z_max) / temperature) (when z_max is not
 * finite, the limit of that rule: w_i = 1 where z_i == z_max, else 0); the
 * token is the first candidate, in that order, whose cumulative weight
 * exceeds u * sum(w).
 * top_k = 1 is greedy decoding.  1 <= top_k <= GPT2_MAX_TOP_K, temperature > 0.
 * The cache and the per-position work use the training step's activation
 * buffers: afterwards the first B rows of the logits buffer hold the logits
 * the last token was drawn from, and a backward needs a new forward with
 * targets (GPT2_ERR_STATE otherwise).  Out-of-range prompt tokens give
 * GPT2_ERR_BAD_TOKEN.  The position counter lives in device memory: the first
 * prompt position and the first drawing position run as plain launches, the
 * others replay a CUDA graph captured from them (on a stream the call creates
 * and destroys).  Synchronises the stream once, at the end.
 * Decoding always uses the bf16 weights, whatever fp8_forward is; with
 * fused_lm_head the B rows of logits fit in its one-chunk buffer.
 */
int gpt2_generate(gpt2_model *m, int32_t *d_seq, int B, int T_total, int T0, const float *d_uniforms,
                  float temperature, int top_k);

/*
 * One fused pass over all parameters ([L] §Eğitim süreci, [R] §Video özeti):
 *   n = sqrt(sum of all grads^2) (every tensor, fp32 data, fp64 reduction);
 *   c = min(1, clip / (n + 1e-6));  g = c * grad;
 *   t += 1;  m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   p = p (1 - lr wd [2-D weights only]) - lr (m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps);
 *   bf16 weight copy = RN(p).
 * The pre-clip norm is written to *grad_norm_out (host; synchronises).  If n is
 * not finite nothing is updated and GPT2_ERR_NONFINITE is returned.  Grads are
 * left unchanged (call gpt2_zero_grad before the next accumulation).
 */
int gpt2_clip_and_adamw(gpt2_model *m, float lr, float beta1, float beta2, float eps, float wd, float clip,
                        float *grad_norm_out);

/*
 * Test hook for the bounded device waits (not a step of the training path).
 * Sets, for this process, the time limit of the spin at the grid barrier of
 * gpt2_clip_and_adamw (wait_ns = 0 restores the default of 2 s).  With
 * never_arrive = 1 that barrier waits for one block more than its grid has,
 * so every block's wait runs out: gpt2_clip_and_adamw then returns
 * GPT2_ERR_TIMEOUT, updates nothing and leaves the step counter as it was,
 * and the model stays usable once the hook is reset (never_arrive = 0).
 * Returns GPT2_ERR_BAD_ARG for never_arrive other than 0 or 1.
 */
int gpt2_debug_set_barrier_wait(unsigned long long wait_ns, int never_arrive);

/* Number of parameter tensors: 2 + 12 L + 2. */
int gpt2_num_tensors(const gpt2_model *m);

/*
 * Name and shape of tensor `id` in the order wte, wpe, per layer
 * [ln1.g ln1.b qkv.w qkv.b proj.w proj.b ln2.g ln2.b fc.w fc.b fcproj.w fcproj.b], lnf.g, lnf.b.
 * *name points to static storage owned by the model.
 */
int gpt2_tensor_info(const gpt2_model *m, int id, const char **name, int *ndim, int64_t shape[2]);

/* Copy fp32 master params / grads / AdamW m / AdamW v of tensor `id` to host
 * (n = element count; synchronises). */
int gpt2_get_params(gpt2_model *m, int id, float *host_out, size_t n);
int gpt2_get_grads(gpt2_model *m, int id, float *host_out, size_t n);
int gpt2_get_adam_state(gpt2_model *m, int id, float *host_m, float *host_v, size_t n);

/* Overwrite fp32 master params of tensor `id` from host (and its bf16 copy). */
int gpt2_set_params(gpt2_model *m, int id, const float *host_in, size_t n);

/* Overwrite the fp32 gradient of tensor `id` from host (tests of the optimizer
 * on given gradients; synchronises). */
int gpt2_set_grads(gpt2_model *m, int id, const float *host_in, size_t n);

/*
 * Device pointer and byte size of an internal activation buffer, for tests:
 * "logits" ([B*T, Vp], dtype of the model; after a forward with targets it
 * holds dlogits), "loss_rows" (fp32 [B*T]), "lnf" (final LN output), "qkv.<l>",
 * "att.<l>", "lse.<l>", "resid.<l>" (input of layer l; resid.L is the final
 * residual stream), "ln1.<l>", "ln2.<l>", "resid_mid.<l>" (after attention),
 * "fch.<l>" (FC pre-activation [B*T, 4C]); with fp8_forward also "w8.<id>"
 * (E4M3 codes of tensor id, uint8 in its shape; filled for the four block
 * projection weights of every layer), "w8_inv" (fp32 [4L]: their
 * dequantisation factors, QKV / attention output / FC / FC output of layer 0,
 * then layer 1 ...), "a8" (uint8 [B*T, 4C]: the activation codes of the last
 * quantised product) and "a8_inv" (fp32 [B*T]).  GPT2_ERR_BAD_ARG for an
 * unknown name.
 */
int gpt2_debug_buffer(gpt2_model *m, const char *name, void **dev_ptr, size_t *bytes);

/* Step counter t of AdamW (number of clip_and_adamw calls that updated). */
int gpt2_adam_step(const gpt2_model *m, int *t_out);

void gpt2_free(gpt2_model *m);
const char *gpt2_strerror(int status);

/* Text of the last CUDA error seen by this thread (for diagnostics; "" if none). */
const char *gpt2_last_error_detail(void);

/* Number of kernels this library has launched in this process (all models and op calls). */
long long gpt2_launch_count(void);

/* ---- per-launch timing (measurement) ---------------------------------------
 * With profiling enabled, each kernel launch of the model calls is bracketed by
 * a pair of CUDA events on the model's stream and attributed to a category
 * together with its algorithmic work (FLOP for matmul and attention, bytes for
 * the memory-bound kernels).  gpt2_profile(m, 1) clears the totals and starts
 * recording, gpt2_profile(m, 0) stops; gpt2_profile_read synchronises the
 * stream and returns the totals of one category: event time, work, and the
 * number of kernels the recorded calls launched (an attention backward call
 * launches two or three).                                                   */
#define GPT2_PROF_MATMUL     0  /* tcgen05 / SIMT matmuls: work = 2 M N K FLOP */
#define GPT2_PROF_ATTENTION  1  /* causal attention: work = 4 hd T(T+1)/2 per head (fwd), 2x that (bwd) FLOP */
#define GPT2_PROF_CLASSIFIER 2  /* fused classifier: work = bytes read + written */
#define GPT2_PROF_ADAMW      3  /* clip + AdamW: bytes */
#define GPT2_PROF_LAYERNORM  4  /* LayerNorm forward/backward: bytes */
#define GPT2_PROF_OTHER      5  /* embedding, bias sums, GELU recompute, loss mean, E4M3 quantisers: bytes */
#define GPT2_PROF_MATMUL_E4M3 6 /* E4M3 matmuls of the fp8_forward mode: work = 2 M N K FLOP */
#define GPT2_PROF_NCAT       7
int gpt2_profile(gpt2_model *m, int enable);
int gpt2_profile_read(gpt2_model *m, int category, double *total_ms, double *total_work, long long *launches);

/* ---- op-level entry points (device pointers; enqueued on `stream`) ------- *
 * The model calls are built from these kernels; they are exposed for
 * per-kernel parity tests and for the isolated attention workload.          */

/*
 * Causal attention forward, flash style: the T x T score matrix is never
 * stored ([G] 01:02:00, 01:16:56; [R] §Video özeti, flash attention).
 * For each (b, h): O = softmax(Q K^T / sqrt(hd), j <= i) V and
 * lse[b,h,i] = logsumexp_j of the scaled scores.
 * q/k/v/o are bf16 with element (b, t, h, d) at ptr[(b*T + t)*row_stride + h*hd + d]
 * (row_stride in elements: 3C for a fused qkv buffer, H*hd for separate
 * tensors).  lse is fp32 [B, H, T].  hd must be 64; row strides multiples of 8;
 * all pointers 16-byte aligned; B*H <= 2^31-1 and T <= 4194240 (65535 blocks
 * of 64), else GPT2_ERR_BAD_SHAPE.
 */
int gpt2_op_attention_forward(const void *q, const void *k, const void *v, int64_t qkv_row_stride, void *o,
                              int64_t o_row_stride, float *lse, int B, int T, int H, int hd, void *stream);

/*
 * Causal attention backward from O, dO and lse of the forward:
 * D = rowsum(dO * O); P = exp(S - lse); dV = P^T dO; dP = dO V^T;
 * dS = P * (dP - D); dQ = dS K / sqrt(hd); dK = dS^T Q / sqrt(hd).
 * dq/dk/dv use qkv_row_stride (they may point into one fused dqkv buffer).
 * d_scratch: caller-owned fp32 workspace of B*H*T floats (holds D).
 * Shape, stride and alignment limits are those of gpt2_op_attention_forward.
 */
int gpt2_op_attention_backward(const void *q, const void *k, const void *v, int64_t qkv_row_stride,
                               const void *o, const void *dout, int64_t o_row_stride, const float *lse,
                               void *dq, void *dk, void *dv, float *d_scratch, int B, int T, int H, int hd,
                               void *stream);

/*
 * The same attention backward with the dS matrix kept: the kernel that forms
 * dK and dV also writes dS^T (bf16, in 64 x 64 blocks) of every causal block to
 * d_ds, and dQ =
 * dS K / sqrt(hd) is then one tensor-core product over those blocks, instead
 * of a second pass that recomputes S and dP for each block of queries.  Same
 * results up to rounding order (dS is rounded to bf16 once, as the dK product
 * uses it).
 * d_ds: caller-owned device workspace of at least
 * gpt2_attention_backward_ds_bytes(B, T, H) bytes, 16-byte aligned; its
 * contents need not be initialised and are overwritten.  The other arguments
 * are those of gpt2_op_attention_backward.  H*hd above 2048 returns
 * GPT2_ERR_UNSUPPORTED; a NULL or short d_ds returns GPT2_ERR_BAD_ARG.
 */
int gpt2_op_attention_backward_ds(const void *q, const void *k, const void *v, int64_t qkv_row_stride,
                                  const void *o, const void *dout, int64_t o_row_stride, const float *lse,
                                  void *dq, void *dk, void *dv, float *d_scratch, void *d_ds, size_t ds_bytes, int B,
                                  int T, int H, int hd, void *stream);

/* Bytes of the d_ds workspace: B*H*Tp*Tp*2 with Tp = T rounded up to a
 * multiple of 128 (0 for non-positive sizes). */
size_t gpt2_attention_backward_ds_bytes(int B, int T, int H);

/*
 * Attention backward that allocates nothing.  The source pages have no
 * counterpart to this entry point; it exists for callers of this library that
 * cannot allocate device memory when they call it (for example, when a
 * memory-pool owner has already reserved the device's memory, or when the
 * hosting runtime forbids allocation after start-up) and so cannot supply the
 * d_scratch workspace of gpt2_op_attention_backward.
 *
 * Same arguments and results as gpt2_op_attention_backward, without
 * d_scratch: the B*H*T-float workspace is a fixed array inside the library,
 * GPT2_NOALLOC_ATTN_MAX_ROWS floats (4 MiB) that every GPU loading the
 * library holds until the process exits.  B*H*T above that limit returns
 * GPT2_ERR_BAD_SHAPE.  The call makes no cudaMalloc / cudaFree and uses no
 * allocating library routine.  Each call looks up the array's device
 * address (cudaGetSymbolAddress) with the calling device current; the first
 * call on a device also loads the library there, so make that first call
 * before any stream capture.  All calls on a device
 * share the one array, which keeps the previous call's contents (the kernels
 * overwrite the part they read before reading it): calls that can overlap on
 * the GPU (different streams, or different host threads) race on it and must
 * be serialised by the caller.
 */
#define GPT2_NOALLOC_ATTN_MAX_ROWS (1 << 20)
int gpt2_op_attention_backward_noalloc(const void *q, const void *k, const void *v, int64_t qkv_row_stride,
                                       const void *o, const void *dout, int64_t o_row_stride, const float *lse,
                                       void *dq, void *dk, void *dv, int B, int T, int H, int hd, void *stream);

/*
 * LayerNorm over rows of C bf16 values ("Let's build GPT: from scratch",
 * 01:32:51): y = (x - mean) / sqrt(var + 1e-5) * g + b with biased variance;
 * mean and rstd (fp32 [N]) are written for the backward.  g, b fp32 [C];
 * C a multiple of 8 and at most 2048.
 */
int gpt2_op_layernorm_forward(const void *x, const float *g, const float *b, void *y, float *mean, float *rstd,
                              int N, int C, void *stream);

/*
 * LayerNorm backward: dres_out = dres_in + dx with
 * dx = rstd (dy*g - mean(dy*g) - xhat mean(dy*g*xhat)); dg += sum_rows dy*xhat,
 * db += sum_rows dy (fp32 [C], accumulated).  dres_in may be NULL (then dres_out
 * = dx) or equal dres_out (in place).  All bf16 [N, C] except the fp32 stats.
 */
int gpt2_op_layernorm_backward(const void *dy, const void *x, const float *mean, const float *rstd, const float *g,
                               const void *dres_in, void *dres_out, float *dg, float *db, int N, int C, void *stream);

/* Matmul epilogues of gpt2_op_matmul. */
#define GPT2_EPI_STORE        0  /* D = acc (+ bias)                      -> bf16 */
#define GPT2_EPI_RESIDUAL     1  /* D = acc + bias + R[m,n]              -> bf16 */
#define GPT2_EPI_GELU         2  /* D = acc + bias (h), D2 = gelu_tanh(h) -> bf16, bf16 */
#define GPT2_EPI_GELU_BWD     3  /* D = acc * gelu_tanh'(R[m,n])          -> bf16 */
#define GPT2_EPI_ACCUM_F32    4  /* D[m,n] += acc                         -> fp32 */

/*
 * bf16 matmul on the tcgen05 tensor cores, fp32 accumulation in TMEM:
 *   acc[m, n] = sum_k A(m, k) * B(n, k)
 * a_kmajor = 1: A(m,k) = A[m*lda + k]   (row-major [M, K])
 * a_kmajor = 0: A(m,k) = A[k*lda + m]   (row-major [K, M], i.e. A^T stored)
 * b_kmajor = 1: B(n,k) = B[n*ldb + k]   (row-major [N, K], a [out,in] weight)
 * b_kmajor = 0: B(n,k) = B[k*ldb + n]   (row-major [K, N])
 * D is row-major [M, N] with leading dimension ldd (R uses ldd too); bias is
 * fp32 [N] or NULL.  Requirements: lda, ldb, ldd multiples of 8, 16-byte
 * aligned pointers, K >= 1.  M, N, K need not be multiples of the tile.
 */
int gpt2_op_matmul(const void *A, int64_t lda, int a_kmajor, const void *B, int64_t ldb, int b_kmajor, void *D,
                   void *D2, const void *R, int64_t ldd, const float *bias, int M, int N, int K, int epilogue,
                   void *stream);

/*
 * Two weight-gradient products in one launch ("Let's reproduce GPT-2 (124M)",
 * §Video özeti: the backward pass of each linear layer):
 *   D0[m, n] += sum_k A0[k, m] B0[k, n]   (m < M0, n < N0)
 *   D1[m, n] += sum_k A1[k, m] B1[k, n]   (m < M1, n < N1)
 * A_i, B_i bf16 row-major [K, M_i] and [K, N_i] with leading dimensions lda_i,
 * ldb_i (the activation and the output gradient of a layer, as stored); D_i fp32
 * row-major [M_i, N_i] with leading dimension N_i.  Both products share K, run as
 * one persistent tcgen05 kernel whose work units are the tiles of both, and add
 * their fp32 results through TMA reduce-adds; results are those of two
 * gpt2_op_matmul calls with GPT2_EPI_ACCUM_F32 up to the order of fp32 additions.
 * Products with N_i < 256 run as two launches.  Requirements as for
 * gpt2_op_matmul (leading dimensions multiples of 8, 16-byte aligned pointers).
 */
int gpt2_op_matmul_accum2(const void *A0, int64_t lda0, const void *B0, int64_t ldb0, float *D0, int M0, int N0,
                          const void *A1, int64_t lda1, const void *B1, int64_t ldb1, float *D1, int M1, int N1, int K,
                          void *stream);

/* ---- E4M3 (FP8) matmul -------------------------------------------------------
 * The pages name FP8 as the next precision step of this training code ("llm.c
 * kullanarak GPT-2 modelini düşük maliyetle yeniden uygulamak", §SSS; the
 * "PyTorch Howsam" post on llm.c) and fix no format.  Format: E4M3 of the OCP
 * 8-bit floating point specification (largest finite 448), converted with
 * round to nearest even and saturation.  Codes are uint8 device arrays.
 *
 * gpt2_op_quantize_e4m3_rows: x bf16 [M, K] (row stride ldx) -> q [M, K]
 * (row stride ldq) and row_inv fp32 [M]: row m is multiplied by
 * s = 448 / amax_m (fp32) and rounded; it represents q * row_inv[m] with
 * row_inv[m] = amax_m / 448 (1 and codes 0 for a row of zeros).  K, ldx, ldq
 * multiples of 8; x and q 16-byte aligned.
 *
 * gpt2_op_quantize_e4m3_tensor: the same with one amax over x bf16 [n]
 * (n a multiple of 8): q [n], inv fp32 [1].  d_amax_work: one device uint of
 * caller-owned scratch (overwritten).
 *
 * gpt2_op_matmul_e4m3: D = a_row_inv[m] * b_inv[0] * sum_k A(m, k) B(n, k)
 * with the epilogues GPT2_EPI_STORE (+ bias), GPT2_EPI_RESIDUAL (+ bias + R)
 * or GPT2_EPI_GELU (D = h, D2 = gelu(h)), bf16 outputs; A [M, K] and B [N, K]
 * E4M3 codes K-major (lda, ldb in bytes, multiples of 16), fp32
 * accumulation in TMEM (tcgen05.mma kind::f8f6f4).  N >= 128 and a multiple
 * of 8; other requirements as gpt2_op_matmul.  GPT2_ERR_UNSUPPORTED or
 * GPT2_ERR_BAD_SHAPE otherwise.
 */
int gpt2_op_quantize_e4m3_rows(const void *x, int64_t ldx, int M, int K, uint8_t *q, int64_t ldq, float *row_inv,
                               void *stream);
int gpt2_op_quantize_e4m3_tensor(const void *x, int64_t n, uint8_t *q, float *inv, unsigned *d_amax_work,
                                 void *stream);
int gpt2_op_matmul_e4m3(const uint8_t *A, int64_t lda, const float *a_row_inv, const uint8_t *B, int64_t ldb,
                        const float *b_inv, void *D, void *D2, const void *R, int64_t ldd, const float *bias, int M,
                        int N, int K, int epilogue, void *stream);

/*
 * The sampling rule of gpt2_generate on bf16 logits rows [B, ldl] (columns
 * [0, V) are the candidates): out[b] = the token drawn with uniforms[b].
 * Device pointers; ldl >= V.
 */
int gpt2_op_sample(const void *logits, int64_t ldl, int B, int V, const float *uniforms, float temperature, int top_k,
                   int32_t *out, void *stream);

/*
 * Embedding backward ("Let's build GPT: from scratch", 01:00:18: token and
 * position embeddings are added, so each receives the residual gradient):
 *   dwte[tokens[b, t], :] += dx[b, t, :];   dwpe[t, :] += sum_b dx[b, t, :].
 * dx: device [B, T, C] of dtype GPT2_DTYPE_FP32 (float) or GPT2_DTYPE_BF16;
 * tokens: device int32 [B, T]; dwte: device fp32 [>= V, C]; dwpe: device fp32
 * [>= T, C]; both accumulated into (zero them for a plain result).  Tokens
 * outside [0, V) are added to row 0 (the forward reports them).
 * With d_workspace (device, 256-byte aligned, at least
 * gpt2_embedding_backward_workspace(B, T, C) bytes, owned by the caller) and
 * C a multiple of 8, V <= 65536: the positions are sorted by token (stable, in
 * chunks of 16384 positions) and every row of dwte is summed in one fixed
 * order, so the result is the same bits on every run.  With d_workspace NULL
 * the token rows are summed with fp32 atomics (order not fixed).  dwpe[t] is
 * always the batch rows added in order b = 0 .. B-1.  C a multiple of 4.
 */
size_t gpt2_embedding_backward_workspace(int B, int T, int C);
int gpt2_op_embedding_backward(const void *dx, int dtype, const int32_t *tokens, int B, int T, int C, int V,
                               float *dwte, float *dwpe, void *d_workspace, void *stream);

/*
 * Fused classifier over rows of bf16 logits [N, Vp] (in place):
 * loss_rows[i] = logsumexp(z[i, 0..V)) - z[i, target[i]];
 * z[i, v] <- (softmax(z[i, 0..V))[v] - [v == target[i]]) * dscale for v < V,
 * z[i, v] <- 0 for V <= v < Vp.  No probabilities are stored.
 */
int gpt2_op_classifier(void *logits, const int32_t *targets, float *loss_rows, int N, int V, int Vp, float dscale,
                       void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GPT2B300_H */
