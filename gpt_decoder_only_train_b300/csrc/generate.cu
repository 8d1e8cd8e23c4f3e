// Forward-only decoding with a key/value cache and top-k sampling.
//
// "llm.c kullanarak GPT-2 modelini düşük maliyetle yeniden uygulamak"
// (§Sampling, §SSS) says a trained model can be sampled, conditionally or not,
// with small changes and no inference optimisation; "Let's reproduce GPT-2
// (124M)" (§Video özeti, §Bölümler 3) builds the forward pass and the sampling
// loop.  Neither page gives the sampling rule; the one implemented here (the
// reading the oracle follows too) is: the logits z[0..V) of the last position,
// candidates = the top_k largest (equal values: lower index first),
// w_i = exp((z_i - z_max) / temperature), and the token is the first candidate i
// in that order with w_0 + ... + w_i > u * sum(w) for a uniform u in [0, 1)
// supplied by the caller.  top_k = 1 is greedy decoding.
//
// Per generated position the model runs on B rows only: the new token's
// embedding, and per block LayerNorm, the QKV product (its K and V rows go
// straight into the cache), one query attending to the cached keys, and the
// rest of the block; the final LayerNorm, the LM head and the sampler run for
// the positions that produce a token.  The kernels read the position from
// device memory, so the host captures one position's launches as a CUDA graph
// and replays it (about 90 launches a position for the 124M model).
#include <algorithm>
#include <climits>

#include "kernels.cuh"

namespace k {

// The position being processed is read from device memory (*d_pos), so one
// captured CUDA graph of a position's launches serves every position.

// x[b, :] = wte[seq[b * ld + pos]] + wpe[pos]   (fp32 master rows, one rounding to T)
template <typename T>
__global__ void embed_decode_kernel(const int *__restrict__ seq, int64_t ld, const int *__restrict__ d_pos,
                                    const float *__restrict__ wte, const float *__restrict__ wpe, T *__restrict__ x,
                                    int B, int C, int V, int *err) {
    const int pos = *d_pos;
    const int c4 = C >> 2;
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= B * c4) return;
    const int b = idx / c4, c = (idx - b * c4) * 4;
    int tk = seq[(int64_t)b * ld + pos];
    if (tk < 0 || tk >= V) {
        raise_device_error(err, DEVERR_BAD_TOKEN);
        tk = 0;
    }
    const float4 a = *reinterpret_cast<const float4 *>(wte + (int64_t)tk * C + c);
    const float4 p = *reinterpret_cast<const float4 *>(wpe + (int64_t)pos * C + c);
    T *o = x + (int64_t)b * C + c;
    o[0] = from_f32<T>(a.x + p.x);
    o[1] = from_f32<T>(a.y + p.y);
    o[2] = from_f32<T>(a.z + p.z);
    o[3] = from_f32<T>(a.w + p.w);
}

template <typename T>
int embed_decode(const int *seq, int64_t ld, const int *d_pos, const float *wte, const float *wpe, T *x, int B, int C,
                 int V, int *err, cudaStream_t st) {
    if (C % 4) return GPT2_ERR_BAD_SHAPE;
    embed_decode_kernel<T><<<ceil_div((int64_t)B * (C / 4), 256), 256, 0, st>>>(seq, ld, d_pos, wte, wpe, x, B, C, V,
                                                                                 err);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// One query per (b, h) against the cached keys of positions 0..pos (causal:
// the position itself included), scale 1/sqrt(hd).  The new position's
// [Q | K | V] row (C columns each) is qkv_new[b * 3C]; the block first appends
// its head's K and V to the cache, whose row (b, j) is
// cache[(b * cache_T + j) * 3C] in the same column layout.
// One block per (b, h); scores in shared memory, fp32 softmax and sums.
constexpr int DEC_THREADS = 128;

template <typename T>
__global__ void __launch_bounds__(DEC_THREADS) attn_decode_kernel(T *__restrict__ cache, const T *__restrict__ qkv_new,
                                                                  int cache_T, const int *__restrict__ d_pos, int H,
                                                                  int hd, T *__restrict__ out, float scale) {
    extern __shared__ float dsm[];  // [pos + 1] scores, then [hd] query, then partial outputs
    const int b = blockIdx.x / H, h = blockIdx.x - (blockIdx.x / H) * H;
    const int C = H * hd, tid = threadIdx.x;
    const int pos = *d_pos;
    const int n = pos + 1;
    float *sc = dsm;
    float *qs = dsm + n;
    float *part = qs + hd;  // [DEC_THREADS / hd groups][hd]
    __shared__ float red[DEC_THREADS / 32];
    T *base = cache + (int64_t)b * cache_T * 3 * C;
    const T *nr = qkv_new + (int64_t)b * 3 * C;
    for (int d = tid; d < hd; d += DEC_THREADS) {
        qs[d] = to_f32(nr[h * hd + d]);
        base[(int64_t)pos * 3 * C + C + h * hd + d] = nr[C + h * hd + d];
        base[(int64_t)pos * 3 * C + 2 * C + h * hd + d] = nr[2 * C + h * hd + d];
    }
    __syncthreads();
    // scores
    float mx = -INFINITY;
    for (int j = tid; j < n; j += DEC_THREADS) {
        const T *kr = base + (int64_t)j * 3 * C + C + h * hd;
        float s = 0.f;
        for (int d = 0; d < hd; ++d) s = fmaf(qs[d], to_f32(kr[d]), s);
        s *= scale;
        sc[j] = s;
        mx = fmaxf(mx, s);
    }
    mx = warp_max(mx);
    if ((tid & 31) == 0) red[tid >> 5] = mx;
    __syncthreads();
    mx = red[0];
    for (int w = 1; w < DEC_THREADS / 32; ++w) mx = fmaxf(mx, red[w]);
    __syncthreads();
    float sum = 0.f;
    for (int j = tid; j < n; j += DEC_THREADS) {
        const float e = exp_t<T>(sc[j] - mx);
        sc[j] = e;
        sum += e;
    }
    sum = warp_sum(sum);
    if ((tid & 31) == 0) red[tid >> 5] = sum;
    __syncthreads();
    sum = 0.f;
    for (int w = 0; w < DEC_THREADS / 32; ++w) sum += red[w];
    // out[d] = sum_j p_j v_j[d]: thread (g, d) sums the positions j = g mod groups
    const int groups = DEC_THREADS / hd, g = tid / hd, d = tid - (tid / hd) * hd;
    if (g < groups) {
        float acc = 0.f;
        for (int j = g; j < n; j += groups) acc = fmaf(sc[j], to_f32(base[(int64_t)j * 3 * C + 2 * C + h * hd + d]), acc);
        part[g * hd + d] = acc;
    }
    __syncthreads();
    if (tid < hd) {
        float acc = 0.f;
        for (int gg = 0; gg < groups; ++gg) acc += part[gg * hd + tid];
        out[(int64_t)b * C + h * hd + tid] = from_f32<T>(acc / sum);
    }
}

template <typename T>
int attention_decode(T *cache, const T *qkv_new, int cache_T, const int *d_pos, int max_pos, int B, int H, int hd,
                     T *out, cudaStream_t st) {
    if (hd <= 0 || hd > 64 || DEC_THREADS % hd || max_pos >= cache_T) return GPT2_ERR_BAD_SHAPE;
    const size_t smem = (size_t)(max_pos + 1 + hd + DEC_THREADS) * sizeof(float);
    if (smem > 200 * 1024) return GPT2_ERR_BAD_SHAPE;
    if (smem > 48 * 1024)
        GPT2_CUDA_TRY(cudaFuncSetAttribute(attn_decode_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem));
    attn_decode_kernel<T><<<B * H, DEC_THREADS, smem, st>>>(cache, qkv_new, cache_T, d_pos, H, hd, out,
                                                            1.0f / sqrtf((float)hd));
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// ---- top-k sampling ------------------------------------------------------------------
// One block per row.  The candidates are found in rank order, one per round:
// round r takes the largest (value, lower index first) entry ranked below the
// one round r-1 took, so no element needs marking.  Thread 0 then forms the
// weights and walks the cumulative sum.
constexpr int SAMPLE_THREADS = 1024;

// (v, i) ranks before (w, j): larger value, or equal value and lower index
__device__ __forceinline__ bool ranks_before(float v, int i, float w, int j) { return v > w || (v == w && i < j); }

template <typename T>
__global__ void __launch_bounds__(SAMPLE_THREADS) sample_topk_kernel(const T *__restrict__ logits, int64_t ldl, int V,
                                                                     const float *__restrict__ u, float inv_temp,
                                                                     int top_k, int *__restrict__ out, int64_t ld_out,
                                                                     int col_out, const int *__restrict__ d_pos,
                                                                     int T0) {
    __shared__ float cv[GPT2_MAX_TOP_K];
    __shared__ int ci[GPT2_MAX_TOP_K];
    __shared__ float wv[SAMPLE_THREADS / 32];
    __shared__ int wi[SAMPLE_THREADS / 32];
    __shared__ int found;
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const T *z = logits + (int64_t)b * ldl;
    // with d_pos: the token of column *d_pos + 1, drawn with u[(column - T0) * B + b]
    const int col = d_pos ? *d_pos + 1 : col_out;
    const float ub = d_pos ? u[(int64_t)(col - T0) * gridDim.x + b] : u[b];
    float bv = INFINITY;
    int bi = -1;  // the entry taken last round (all later ones rank below it)
    int k = 0;
    for (; k < top_k; ++k) {
        float v = -INFINITY;
        int i = INT_MAX;
        for (int c = tid; c < V; c += SAMPLE_THREADS) {
            const float x = to_f32(z[c]);
            if (ranks_before(bv, bi, x, c) && ranks_before(x, c, v, i)) {
                v = x;
                i = c;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, v, o);
            const int oi = __shfl_xor_sync(0xffffffffu, i, o);
            if (ranks_before(ov, oi, v, i)) {
                v = ov;
                i = oi;
            }
        }
        if (lane == 0) {
            wv[wid] = v;
            wi[wid] = i;
        }
        __syncthreads();
        if (tid == 0) {
            float mv = wv[0];
            int mi = wi[0];
            for (int w = 1; w < SAMPLE_THREADS / 32; ++w)
                if (ranks_before(wv[w], wi[w], mv, mi)) {
                    mv = wv[w];
                    mi = wi[w];
                }
            found = mi != INT_MAX;
            cv[k] = mv;
            ci[k] = mi;
        }
        __syncthreads();
        if (!found) break;  // fewer than top_k ranked entries (NaN rows, V < top_k)
        bv = cv[k];
        bi = ci[k];
        __syncthreads();  // cv / ci of this round are read before thread 0 writes the next
    }
    if (tid == 0) {
        int pick = 0;
        if (k > 1) {
            // w_r = exp((z_r - z_max) / temperature); when z_max is not finite
            // (+inf, or every candidate -inf) the weights are the limit of that
            // rule: 1 for the candidates equal to z_max, 0 for the rest
            const float top = cv[0];
            const bool fin = isfinite(top);
            float s = 0.f;
            for (int r = 0; r < k; ++r) s += fin ? exp_t<T>((cv[r] - top) * inv_temp) : (cv[r] == top ? 1.f : 0.f);
            const float target = ub * s;
            float cum = 0.f;
            pick = k - 1;
            for (int r = 0; r < k; ++r) {
                cum += fin ? exp_t<T>((cv[r] - top) * inv_temp) : (cv[r] == top ? 1.f : 0.f);
                if (cum > target) {
                    pick = r;
                    break;
                }
            }
        }
        out[(int64_t)b * ld_out + col] = k > 0 ? ci[pick] : 0;
    }
}

template <typename T>
int sample_topk(const T *logits, int64_t ldl, int B, int V, const float *u, float temperature, int top_k, int *out,
                int64_t ld_out, int col_out, const int *d_pos, int T0, cudaStream_t st) {
    if (B <= 0 || V <= 0 || top_k < 1 || top_k > GPT2_MAX_TOP_K || !(temperature > 0.f)) return GPT2_ERR_BAD_ARG;
    // a finite scale: (z_i - z_max) * scale must stay 0 for ties with the maximum
    const float inv = 1.0f / temperature, inv_temp = isfinite(inv) ? inv : 3.0e38f;
    sample_topk_kernel<T><<<B, SAMPLE_THREADS, 0, st>>>(logits, ldl, V, u, inv_temp, top_k, out, ld_out, col_out,
                                                        d_pos, T0);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// ---- skinny matmul for the decode rows ------------------------------------------------------
// D[b, n] = epilogue(sum_k X[b, k] W[n, k]) for Bm <= SK_MAX_ROWS rows: the
// decode products are a few rows against a whole weight matrix, so the work
// is the weight stream.  Each warp takes one output column n at a time and
// reads W's row n (K-major, 16 bytes a lane) once for all rows; X sits in
// shared memory.  The sums are warp reductions; lane b finishes row b.
constexpr int SK_WARPS = 8;

template <int EPI>
__global__ void __launch_bounds__(SK_WARPS * 32)
    skinny_gemm_kernel(const bf16 *__restrict__ X, int64_t ldx, const bf16 *__restrict__ W, int K, int N, int Bm,
                       const float *__restrict__ bias, const bf16 *__restrict__ R, bf16 *__restrict__ D,
                       bf16 *__restrict__ D2, int64_t ldd) {
    extern __shared__ uint4 xs[];  // [Bm][K / 8] packets of X
    const int kp = K >> 3;
    for (int i = threadIdx.x; i < Bm * kp; i += blockDim.x) {
        const int b = i / kp, p = i - (i / kp) * kp;
        xs[i] = *reinterpret_cast<const uint4 *>(X + (int64_t)b * ldx + (int64_t)p * 8);
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int n = blockIdx.x * SK_WARPS + warp; n < N; n += gridDim.x * SK_WARPS) {
        float acc[SK_MAX_ROWS];
#pragma unroll
        for (int b = 0; b < SK_MAX_ROWS; ++b) acc[b] = 0.f;
        const uint4 *wr = reinterpret_cast<const uint4 *>(W + (int64_t)n * K);
        for (int p = lane; p < kp; p += 32) {
            const uint4 w = __ldg(wr + p);
            const float w0 = bf16_lo(w.x), w1 = bf16_hi(w.x), w2 = bf16_lo(w.y), w3 = bf16_hi(w.y);
            const float w4 = bf16_lo(w.z), w5 = bf16_hi(w.z), w6 = bf16_lo(w.w), w7 = bf16_hi(w.w);
#pragma unroll
            for (int b = 0; b < SK_MAX_ROWS; ++b) {
                if (b < Bm) {
                    const uint4 x = xs[b * kp + p];
                    float a = acc[b];
                    a = fmaf(w0, bf16_lo(x.x), a);
                    a = fmaf(w1, bf16_hi(x.x), a);
                    a = fmaf(w2, bf16_lo(x.y), a);
                    a = fmaf(w3, bf16_hi(x.y), a);
                    a = fmaf(w4, bf16_lo(x.z), a);
                    a = fmaf(w5, bf16_hi(x.z), a);
                    a = fmaf(w6, bf16_lo(x.w), a);
                    a = fmaf(w7, bf16_hi(x.w), a);
                    acc[b] = a;
                }
            }
        }
        float mine = 0.f;
#pragma unroll
        for (int b = 0; b < SK_MAX_ROWS; ++b) {
            if (b < Bm) {
                const float sum = warp_sum(acc[b]);
                if (lane == b) mine = sum;
            }
        }
        if (lane < Bm) {
            float v = mine + (bias ? bias[n] : 0.f);
            const int64_t o = (int64_t)lane * ldd + n;
            if (EPI == GPT2_EPI_RESIDUAL) v += __bfloat162float(R[o]);
            const bf16 h = __float2bfloat16_rn(v);
            D[o] = h;
            if (EPI == GPT2_EPI_GELU) D2[o] = __float2bfloat16_rn(gelu_tanh(__bfloat162float(h)));
        }
    }
}

// GPT2_ERR_UNSUPPORTED when X does not fit in shared memory (the caller then
// takes the general matmul).  The first call of each epilogue on a device sets
// the kernel's shared-memory limit there, so that call must not be inside a
// stream capture.
int skinny_gemm(const bf16 *X, int64_t ldx, const bf16 *W, int K, int N, int Bm, const float *bias, const bf16 *R,
                bf16 *D, bf16 *D2, int64_t ldd, int epi, int num_sms, cudaStream_t st) {
    if (Bm < 1 || Bm > SK_MAX_ROWS || K % 8 || ldx % 8 || N < 1) return GPT2_ERR_BAD_SHAPE;
    const size_t smem = (size_t)Bm * K * 2;
    const int grid = std::min(ceil_div(N, SK_WARPS), 4 * num_sms);
    auto go = [&](auto kern, PerDevice &lim_pd) -> int {
        int limit = 0;
        if (int rc = per_device(lim_pd, limit, [&](int &v) -> int {
                int dev = 0, optin = 0;
                GPT2_CUDA_TRY(cudaGetDevice(&dev));
                GPT2_CUDA_TRY(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
                GPT2_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin));
                v = optin;
                return GPT2_OK;
            }))
            return rc;
        if (smem > (size_t)limit) return GPT2_ERR_UNSUPPORTED;
        kern<<<grid, SK_WARPS * 32, smem, st>>>(X, ldx, W, K, N, Bm, bias, R, D, D2, ldd);
        GPT2_CUDA_TRY(cudaGetLastError());
        gpt2_note_launches(1);
        return GPT2_OK;
    };
    static PerDevice lim_store, lim_res, lim_gelu;
    switch (epi) {
        case GPT2_EPI_STORE: return go(skinny_gemm_kernel<GPT2_EPI_STORE>, lim_store);
        case GPT2_EPI_RESIDUAL: return R ? go(skinny_gemm_kernel<GPT2_EPI_RESIDUAL>, lim_res) : GPT2_ERR_BAD_ARG;
        case GPT2_EPI_GELU: return D2 ? go(skinny_gemm_kernel<GPT2_EPI_GELU>, lim_gelu) : GPT2_ERR_BAD_ARG;
        default: return GPT2_ERR_BAD_ARG;
    }
}

__global__ void advance_position_kernel(int *d_pos) { *d_pos += 1; }

int advance_position(int *d_pos, cudaStream_t st) {
    advance_position_kernel<<<1, 1, 0, st>>>(d_pos);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

#define INST_GEN(T)                                                                                              \
    template int embed_decode<T>(const int *, int64_t, const int *, const float *, const float *, T *, int, int,    \
                                 int, int *, cudaStream_t);                                                      \
    template int attention_decode<T>(T *, const T *, int, const int *, int, int, int, int, T *, cudaStream_t);     \
    template int sample_topk<T>(const T *, int64_t, int, int, const float *, float, int, int *, int64_t, int,      \
                                const int *, int, cudaStream_t);
INST_GEN(float)
INST_GEN(bf16)
#undef INST_GEN

}  // namespace k
