// Flash-style causal attention for head dimension 64, bf16 in / out, fp32
// softmax statistics, on the tcgen05 tensor cores.  The T x T score matrix is
// never stored: scores live in TMEM one block at a time ("Let's reproduce GPT-2 (124M)",
// §Video özeti: flash attention; "Let's build GPT: from scratch", 01:02:00 and
// 01:16:56: causal self-attention scaled by 1/sqrt(head_size)).
#pragma once

#include "common.cuh"

namespace fa {

// O = softmax(Q K^T / sqrt(64), j <= i) V per (b, h); lse [B, H, T] fp32.
// Element (b, t, h, d) of q/k/v lives at ptr[(b*T + t)*rs + h*64 + d]; o uses ors.
int attention_forward(const bf16 *q, const bf16 *k, const bf16 *v, int64_t rs, bf16 *o, int64_t ors, float *lse,
                      int B, int T, int H, int hd, cudaStream_t st);

// tcgen05 implementation of attention_forward (attn_tc.cu).
int attention_forward_tc(const bf16 *q, const bf16 *k, const bf16 *v, int64_t rs, bf16 *o, int64_t ors, float *lse,
                         int B, int T, int H, cudaStream_t st);

// tcgen05 implementation of attention_backward (attn_tc.cu).
int attention_backward_tc(const bf16 *q, const bf16 *k, const bf16 *v, int64_t rs, const bf16 *o, const bf16 *dout,
                          int64_t ors, const float *lse, bf16 *dq, bf16 *dk, bf16 *dv, float *Dscr, int B, int T,
                          int H, cudaStream_t st, float *dbias = nullptr, bf16 *ds_ws = nullptr);

// Bytes of the dS workspace of attention_backward: B H Tp^2 bf16 with Tp = T
// rounded up to a multiple of 128.
size_t attention_backward_ds_bytes(int B, int T, int H);

// dq/dk/dv (row stride rs) from O, dO (row stride ors) and lse; Dscr holds
// D = rowsum(dO * O) as fp32 [B, H, T].  With dbias (fp32 [3 H 64], columns
// [q | k | v] as in the fused projection, H 64 <= 2048) the gradient of a bias
// added to q, k and v is added to it: the column sums of dq over all B*T rows
// for the query part; the column sums of dout for the value part (every row of
// P sums to one, so the rows of dv sum to the rows of dout); nothing for the
// key part, which is zero (a key bias moves all scores of a query by the same
// amount).
//
// ds_ws (optional, attention_backward_ds_bytes bytes, 16-byte aligned, contents
// need not be initialised): with it the dK/dV kernel also stores dS^T there and
// dQ = scale dS K is formed from it by one product over the causal blocks,
// instead of a second kernel that recomputes S and dP per query block.
int attention_backward(const bf16 *q, const bf16 *k, const bf16 *v, int64_t rs, const bf16 *o, const bf16 *dout,
                       int64_t ors, const float *lse, bf16 *dq, bf16 *dk, bf16 *dv, float *Dscr, int B, int T, int H,
                       int hd, cudaStream_t st, float *dbias = nullptr, bf16 *ds_ws = nullptr);

}  // namespace fa
