// Launchers of the memory-bound kernels of the step and of the fp32-mode SIMT
// matmul / attention.  Template parameter T is the activation type: float
// (fp32 mode) or bf16.  Every launcher only enqueues work on `st`.
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace k {

// x[b,t,:] = wte[tok[b,t]] + wpe[t]   (fp32 master rows, one rounding to T)
template <typename T>
int embed_forward(const int *tok, const float *wte, const float *wpe, T *x, int B, int Tn, int C, int V, int *err,
                  cudaStream_t st);

// dwte[tok[b,t]] += dx[b,t];  dwpe[t] += sum_b dx[b,t].  With a workspace of
// embed_backward_workspace(B*T, C) bytes (and C % 8 == 0, V <= 65536) every row
// is summed in a fixed order (positions sorted by token); without one, with
// fp32 atomics.
template <typename T>
int embed_backward(const int *tok, const T *dx, float *dwte, float *dwpe, int B, int Tn, int C, int V,
                   cudaStream_t st, void *ws);
size_t embed_backward_workspace(int n, int C);

// y = (x - mean) * rstd * g + b per row of C; mean/rstd fp32 [N].  bf16 only:
// with q (uint8 [N, C]) and qinv (fp32 [N]) also the E4M3 copy of each stored
// row, scaled by 448 / amax of the row (qinv = amax / 448).
template <typename T>
int layernorm_forward(const T *x, const float *g, const float *b, T *y, float *mean, float *rstd, int N, int C,
                      cudaStream_t st, uint8_t *q = nullptr, float *qinv = nullptr);

// E4M3 with saturation, round to nearest even (CUDA's conversion)
__device__ __forceinline__ uint32_t e4m3_of(float x) {
    return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// E4M3 per-row copy of bf16 x [M, K] (rows scaled by 448 / amax; inv = amax / 448)
// Cross-entropy from the LM head's partials (the fused LM head): part[row * stride + j],
// j < nparts, holds (max, sum of exp(z - max)) over one half tile of the row's real
// logits (max -inf and sum 0 for none); zt[row] is the target's logit.  Writes
// lse[row] and loss_rows[row] = lse - zt; an invalid target raises the device
// error word (its row was computed as token 0).
int ce_combine(const float2 *part, int stride, int nparts, const float *zt, const int *targets, int N, int V,
               float *lse, float *loss_rows, int *err, cudaStream_t st);

int quantize_rows_e4m3(const bf16 *x, int64_t ldx, int M, int K, uint8_t *q, int64_t ldq, float *inv,
                       cudaStream_t st);
// E4M3 copies of several bf16 tensors of one flat array, one scale each:
// tensor t is w[off[t] .. off[t] + n[t]) -> q (same offsets), inv[t];
// amax_bits: [ntens] uint scratch (zeroed here).  off[t], n[t] multiples of 8.
int quantize_tensors_e4m3(const bf16 *w, const int64_t *d_off, const int64_t *d_n, int ntens, int64_t max_n,
                          uint8_t *q, float *inv, unsigned *amax_bits, cudaStream_t st);

// dres_out = dres_in (may be NULL) + LN'(dy); dg += sum dy*xhat; db += sum dy;
// dsum (may be NULL) += column sums of dres_out as stored, i.e. the bias
// gradient of a layer whose output gradient is dres_out (dres_in and dres_out
// may alias)
template <typename T>
int layernorm_backward(const T *dy, const T *x, const float *mean, const float *rstd, const float *g, const T *dres_in,
                       T *dres_out, float *dg, float *db, int N, int C, cudaStream_t st, float *dsum = nullptr);

// db[n] += sum_m dy[m, n]
template <typename T>
int column_sum(const T *dy, int M, int N, float *db, cudaStream_t st);

// fused softmax cross-entropy (in place), see gpt2_op_classifier
template <typename T>
int classifier(T *logits, const int *targets, float *loss_rows, int N, int V, int Vp, float dscale, int *err,
               cudaStream_t st);

// *out = mean(rows[0..N)) with a fixed-order fp64 reduction
int mean_rows(const float *rows, int N, float *out, cudaStream_t st);

// y = gelu_tanh(h) elementwise (GELU recompute)
template <typename T>
int gelu_forward(const T *h, T *y, int64_t n, cudaStream_t st);

int cast_f32_bf16(const float *x, bf16 *y, int64_t n, cudaStream_t st);

// SIMT matmul with the same epilogues as the tensor-core matmul:
//   acc[m,n] = sum_k A[m*sam + k*sak] * B[n*sbn + k*sbk]
template <typename T>
int matmul_simt(const T *A, int64_t sam, int64_t sak, const T *Bm, int64_t sbn, int64_t sbk, void *D, T *D2,
                const T *R, int64_t ldd, const float *bias, int M, int N, int K, int epi, float alpha,
                cudaStream_t st);

// SIMT causal attention (any head size <= 64), one thread per query / key row.
template <typename T>
int attention_forward_simt(const T *q, const T *kk, const T *v, int64_t rs, T *o, int64_t ors, float *lse, int B,
                           int Tn, int H, int hd, cudaStream_t st);
template <typename T>
int attention_backward_simt(const T *q, const T *kk, const T *v, int64_t rs, const T *o, const T *dout, int64_t ors,
                            const float *lse, T *dq, T *dk, T *dv, float *dscratch, int B, int Tn, int H, int hd,
                            cudaStream_t st);

// ---- forward-only decoding (generate.cu) ----------------------------------------
// The position pos is read from device memory (*d_pos) by the kernels.
// x[b, :] = wte[seq[b * ld + pos]] + wpe[pos]
template <typename T>
int embed_decode(const int *seq, int64_t ld, const int *d_pos, const float *wte, const float *wpe, T *x, int B, int C,
                 int V, int *err, cudaStream_t st);
// appends K, V of qkv_new [B, 3C] ([Q | K | V]) as cache row (b, pos), then
// out[b, h*hd:(h+1)*hd] = softmax_j<=pos(q . k_j / sqrt(hd)) v_j over the cache
// rows cache[(b * cache_T + j) * 3C]; pos <= max_pos < cache_T
template <typename T>
int attention_decode(T *cache, const T *qkv_new, int cache_T, const int *d_pos, int max_pos, int B, int H, int hd,
                     T *out, cudaStream_t st);
// the top-k sampled token of logits row b (see gpt2_generate) -> out[b * ld_out + col];
// col = col_out and u[b], or with d_pos col = *d_pos + 1 and u[(col - T0) * B + b]
template <typename T>
int sample_topk(const T *logits, int64_t ldl, int B, int V, const float *u, float temperature, int top_k, int *out,
                int64_t ld_out, int col_out, const int *d_pos, int T0, cudaStream_t st);
// *d_pos += 1
int advance_position(int *d_pos, cudaStream_t st);
// D[b, n] = epi(sum_k X[b, k] W[n, k] (+ bias[n])) for b < Bm <= SK_MAX_ROWS, W K-major [N, K]
// (ld K); epi: GPT2_EPI_STORE, GPT2_EPI_RESIDUAL (+ R[b, n]) or GPT2_EPI_GELU (D = h, D2 = gelu(h));
// R, D and D2 use the leading dimension ldd
constexpr int SK_MAX_ROWS = 16;
int skinny_gemm(const bf16 *X, int64_t ldx, const bf16 *W, int K, int N, int Bm, const float *bias, const bf16 *R,
                bf16 *D, bf16 *D2, int64_t ldd, int epi, int num_sms, cudaStream_t st);

struct AdamArgs {
    float lr, beta1, beta2, eps, wd, clip;
    float bc1, bc2;                // 1 - beta^t
    unsigned long long wait_ns;    // time limit of the grid barrier's spin
    unsigned extra_arrivals;       // blocks the barrier waits for beyond the grid (0; tests only)
};

// Fused global-norm + clip + AdamW over one flat parameter arena (see
// gpt2_clip_and_adamw).  Elements [0, n_decay) get weight decay.  `partials`
// holds >= max_blocks doubles and `counter` one zeroed uint (grid barrier).
int clip_adamw(float *p, const float *g, float *m, float *v, bf16 *shadow, int64_t n, int64_t n_decay,
               const AdamArgs &a, double *partials, unsigned *counter, int max_blocks, float *norm_out, int *err,
               int num_sms, cudaStream_t st);
int clip_adamw_max_blocks(int num_sms);

}  // namespace k
