// Causal attention entry points (head dim 64): argument checks, then the
// tcgen05 kernels of attn_tc.cu.
#include "flash_attn.cuh"

namespace fa {

// The kernels launch a (B*H, T/64-or-coarser) grid: B*H must fit the x
// dimension and the block count the y dimension (at most 65535).
static bool grid_fits(int B, int T, int H) {
    return (int64_t)B * H <= 0x7fffffff && (T + 63) / 64 <= 65535;
}

int attention_forward(const bf16 *q, const bf16 *k, const bf16 *v, int64_t rs, bf16 *o, int64_t ors, float *lse,
                      int B, int T, int H, int hd, cudaStream_t st) {
    if (hd != 64 || rs % 8 || ors % 8 || B <= 0 || T <= 0 || H <= 0) return GPT2_ERR_BAD_SHAPE;
    if (!grid_fits(B, T, H)) return GPT2_ERR_BAD_SHAPE;
    return attention_forward_tc(q, k, v, rs, o, ors, lse, B, T, H, st);
}

int attention_backward(const bf16 *q, const bf16 *k, const bf16 *v, int64_t rs, const bf16 *o, const bf16 *dout,
                       int64_t ors, const float *lse, bf16 *dq, bf16 *dk, bf16 *dv, float *Dscr, int B, int T, int H,
                       int hd, cudaStream_t st, float *dbias, bf16 *ds_ws) {
    if (hd != 64 || rs % 8 || ors % 8 || B <= 0 || T <= 0 || H <= 0) return GPT2_ERR_BAD_SHAPE;
    if (!grid_fits(B, T, H)) return GPT2_ERR_BAD_SHAPE;
    return attention_backward_tc(q, k, v, rs, o, dout, ors, lse, dq, dk, dv, Dscr, B, T, H, st, dbias, ds_ws);
}

}  // namespace fa
