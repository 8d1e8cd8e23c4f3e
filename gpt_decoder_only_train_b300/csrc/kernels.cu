// Memory-bound kernels of the GPT-2 step (embedding, LayerNorm, classifier,
// bias gradients, fused clip + AdamW) and the fp32-mode SIMT matmul and
// attention.  Sources, by page title and section:
//   embedding / position encoding -- "Let's build GPT: from scratch", 01:00:18;
//   LayerNorm                     -- same page, 01:32:51;
//   cross-entropy                 -- "Let's reproduce GPT-2 (124M)", §Bölümler 4;
//   AdamW, clipping               -- same page §Video özeti; "llm.c kullanarak
//                                    GPT-2 ...", §Eğitim süreci.
#include <algorithm>
#include <math.h>

#include "kernels.cuh"

namespace k {

// ============================================================== embedding
template <typename T> __device__ __forceinline__ void store4(T *p, float a, float b, float c, float d);
template <> __device__ __forceinline__ void store4<float>(float *p, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}
template <> __device__ __forceinline__ void store4<bf16>(bf16 *p, float a, float b, float c, float d) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&lo);
    u.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = u;
}

template <typename T>
__global__ void embed_fwd_kernel(const int *__restrict__ tok, const float *__restrict__ wte,
                                 const float *__restrict__ wpe, T *__restrict__ x, int BT, int Tn, int C, int V,
                                 int *err) {
    const int c4 = C >> 2;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)BT * c4) return;
    const int row = (int)(idx / c4);
    const int c = (int)(idx - (int64_t)row * c4) * 4;
    const int t = row % Tn;
    int tk = tok[row];
    if (tk < 0 || tk >= V) {
        raise_device_error(err, DEVERR_BAD_TOKEN);
        tk = 0;
    }
    const float4 a = *reinterpret_cast<const float4 *>(wte + (int64_t)tk * C + c);
    const float4 p = *reinterpret_cast<const float4 *>(wpe + (int64_t)t * C + c);
    store4<T>(x + (int64_t)row * C + c, a.x + p.x, a.y + p.y, a.z + p.z, a.w + p.w);
}

template <typename T>
int embed_forward(const int *tok, const float *wte, const float *wpe, T *x, int B, int Tn, int C, int V, int *err,
                  cudaStream_t st) {
    if (C % 4) return GPT2_ERR_BAD_SHAPE;
    const int64_t n = (int64_t)B * Tn * (C / 4);
    embed_fwd_kernel<T><<<ceil_div(n, 256), 256, 0, st>>>(tok, wte, wpe, x, B * Tn, Tn, C, V, err);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

template <typename T>
__global__ void embed_bwd_wte_kernel(const int *__restrict__ tok, const T *__restrict__ dx, float *__restrict__ dwte,
                                     int BT, int C, int V) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)BT * C) return;
    const int row = (int)(idx / C), c = (int)(idx - (int64_t)row * C);
    int tk = tok[row];
    if (tk < 0 || tk >= V) tk = 0;
    atomicAdd(dwte + (int64_t)tk * C + c, to_f32(dx[idx]));
}

template <typename T>
__global__ void embed_bwd_wpe_kernel(const T *__restrict__ dx, float *__restrict__ dwpe, int B, int Tn, int C) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)Tn * C) return;
    float s = 0.f;
    for (int b = 0; b < B; ++b) s += to_f32(dx[(int64_t)b * Tn * C + idx]);
    dwpe[idx] += s;
}

// ---- token rows in a fixed order ----------------------------------------------
// The positions of a chunk (at most EMB_CHUNK of them) are sorted by token with
// a stable radix sort (so each token's positions stay in position order); the
// sorted list is cut into pieces of 32.  A warp sums the rows of each run of
// equal tokens in its piece in list order; a run that is a whole token
// segment is added to dwte[token] by that warp (its only writer), a run of a
// segment that crosses a piece boundary goes to a partial slot, and one block
// per crossing segment adds the slots in list order.  Every row of dwte is so
// summed in one fixed order: the result does not depend on scheduling.
constexpr int EMB_CHUNK = 16384;     // positions sorted by one CTA (keys in shared memory)
constexpr int EMB_SORT_THREADS = 1024;

// key = token << 16 | position in the chunk; stable LSD radix sort on the
// token's two bytes (shared-memory counts per warp and digit, digit-major
// exclusive scan, ranks within a warp from ballots of the digit bits).
// Lanes of the warp whose 8-bit digit equals this lane's, among the lanes with v set (one
// ballot per digit bit and one for v); 0 for a lane without v.
__device__ __forceinline__ uint32_t digit_peers(uint32_t d, bool v) {
    uint32_t peers = __ballot_sync(0xffffffffu, v);
#pragma unroll
    for (int bit = 0; bit < 8; ++bit) {
        const bool on = (d >> bit) & 1u;
        const uint32_t m = __ballot_sync(0xffffffffu, on);
        peers &= on ? m : ~m;
    }
    return v ? peers : 0u;
}

__global__ void __launch_bounds__(EMB_SORT_THREADS) embed_sort_kernel(const int *__restrict__ tok, int n, int V,
                                                                     uint32_t *__restrict__ keys_out) {
    extern __shared__ uint32_t esm[];
    uint32_t *buf0 = esm, *buf1 = esm + EMB_CHUNK;
    int *cnt = reinterpret_cast<int *>(esm + 2 * EMB_CHUNK);  // [32 warps][256 digits]
    __shared__ int wsum[32];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    for (int i = tid; i < n; i += EMB_SORT_THREADS) {
        int t = tok[i];
        if (t < 0 || t >= V) t = 0;  // the forward reported it; its row is treated as token 0
        buf0[i] = ((uint32_t)t << 16) | (uint32_t)i;
    }
    const int per_warp = (n + 31) / 32;  // each warp owns a contiguous range of the input order
    const int w0 = min(n, w * per_warp), w1 = min(n, w0 + per_warp);
    uint32_t *in = buf0, *out = buf1;
    for (int pass = 0; pass < 2; ++pass) {
        const int shift = 16 + 8 * pass;
        for (int i = tid; i < 32 * 256; i += EMB_SORT_THREADS) cnt[i] = 0;
        __syncthreads();
        for (int i = w0 + lane; i < w1; i += 32)  // counts need no order: shared atomics on the warp's row
            atomicAdd(&cnt[w * 256 + ((in[i] >> shift) & 255u)], 1);
        __syncthreads();
        // exclusive scan in digit-major order: entry (digit, warp) at index digit * 32 + warp
        int loc[8], run = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = tid * 8 + j, d = e >> 5, ww = e & 31;
            loc[j] = run;
            run += cnt[ww * 256 + d];
        }
        int x = run;  // inclusive scan of the per-thread totals
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[w] = x;
        __syncthreads();
        if (w == 0) {
            int z = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, z, o);
                if (lane >= o) z += y;
            }
            wsum[lane] = z - wsum[lane];  // exclusive
        }
        __syncthreads();
        const int base = wsum[w] + x - run;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = tid * 8 + j, d = e >> 5, ww = e & 31;
            cnt[ww * 256 + d] = base + loc[j];
        }
        __syncthreads();
        for (int b = w0; b < w1; b += 32) {
            const int i = b + lane;
            const bool v = i < w1;
            const uint32_t k = v ? in[i] : 0u;
            const uint32_t d = v ? (k >> shift) & 255u : 0u;
            const uint32_t peers = digit_peers(d, v);
            int dst = 0;
            if (v) dst = cnt[w * 256 + d] + __popc(peers & ((1u << lane) - 1u));
            __syncwarp();
            if (v) {
                out[dst] = k;
                if (lane == __ffs(peers) - 1) cnt[w * 256 + d] += __popc(peers);
            }
            __syncwarp();
        }
        __syncthreads();
        uint32_t *t = in;
        in = out;
        out = t;
    }
    for (int i = tid; i < n; i += EMB_SORT_THREADS) keys_out[i] = in[i];
}

// 8 consecutive elements of row `row` from column `col` as fp32
__device__ __forceinline__ void load8(const bf16 *p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[2 * k] = bf16_lo(w[k]);
        v[2 * k + 1] = bf16_hi(w[k]);
    }
}
__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}

// One warp per (piece of 32 sorted entries, slab of 256 columns; 8 per lane).
template <typename T>
__global__ void embed_runs_kernel(const uint32_t *__restrict__ keys, const T *__restrict__ dx, float *__restrict__ dwte,
                                  float *__restrict__ part, int n, int C) {
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int nslab = (C + 255) / 256, npieces = (n + 31) / 32;
    const int piece = gw / nslab, slab = gw - piece * nslab;
    if (piece >= npieces) return;
    const int i0 = piece * 32, cnt = min(32, n - i0);
    const uint32_t myk = lane < cnt ? keys[i0 + lane] : 0u;
    const int tok_before = i0 > 0 ? (int)(keys[i0 - 1] >> 16) : -1;
    const int tok_after = i0 + cnt < n ? (int)(keys[i0 + cnt] >> 16) : -1;
    const int col = slab * 256 + lane * 8;
    const bool active = col < C;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    int run_start = 0, cur = (int)(__shfl_sync(0xffffffffu, myk, 0) >> 16);
    auto flush = [&](int rs, int re) {
        const bool crosses = (rs == 0 && tok_before == cur) || (re == cnt && tok_after == cur);
        if (!active) return;
        if (crosses) {
            float4 *dst = reinterpret_cast<float4 *>(part + (int64_t)(rs == 0 ? piece : npieces + piece) * C + col);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        } else {
            // the segment's only addition into these elements: a reduction without a wait
            float *dst = dwte + (int64_t)cur * C + col;
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(acc[0]), "f"(acc[1]),
                         "f"(acc[2]), "f"(acc[3])
                         : "memory");
            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4), "f"(acc[4]), "f"(acc[5]),
                         "f"(acc[6]), "f"(acc[7])
                         : "memory");
        }
    };
    for (int j0 = 0; j0 < cnt; j0 += 8) {
        // the rows of up to 8 entries are requested together, then added in order
        float v[8][8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint32_t k = __shfl_sync(0xffffffffu, myk, (j0 + u) & 31);
            if (active && j0 + u < cnt) load8(dx + (int64_t)(k & 0xFFFFu) * C + col, v[u]);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int j = j0 + u;
            if (j >= cnt) break;
            const int tk = (int)(__shfl_sync(0xffffffffu, myk, j & 31) >> 16);
            if (tk != cur) {
                flush(run_start, j);
                run_start = j;
                cur = tk;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = 0.f;
            }
            if (active)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] += v[u][e];
        }
    }
    flush(run_start, cnt);
}

// One block per piece boundary b = 32 k: if a token segment crosses it and
// starts in piece k - 1, add its partial slots in list order to dwte[token].
__global__ void embed_cross_kernel(const uint32_t *__restrict__ keys, const float *__restrict__ part,
                                   float *__restrict__ dwte, int n, int C) {
    const int npieces = (n + 31) / 32, k = blockIdx.x + 1, b = 32 * k;
    if (b >= n) return;
    const uint32_t tk = keys[b] >> 16;
    if ((keys[b - 1] >> 16) != tk) return;                    // no segment crosses this boundary
    if (k >= 2 && (keys[32 * (k - 1) - 1] >> 16) == tk) return;  // it started before piece k - 1
    const bool starts_at_piece = (keys[32 * (k - 1)] >> 16) == tk;
    const int first = starts_at_piece ? k - 1 : npieces + k - 1;
    // pieces k .. last - 1 begin with this token: the first piece after k that begins with
    // another token, all boundaries tested at once (block-wide minimum)
    __shared__ int s_last;
    if (threadIdx.x == 0) s_last = npieces;
    __syncthreads();
    for (int q = k + 1 + threadIdx.x; q < npieces; q += blockDim.x)
        if ((keys[32 * q] >> 16) != tk) {
            atomicMin(&s_last, q);
            break;
        }
    __syncthreads();
    const int last = s_last;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        float s = part[(int64_t)first * C + c];
#pragma unroll 8
        for (int q = k; q < last; ++q) s += part[(int64_t)q * C + c];
        atomicAdd(dwte + (int64_t)tk * C + c, s);  // the segment's only addition into this element
    }
}

size_t embed_backward_workspace(int n, int C) {
    const int chunk = std::min(n, EMB_CHUNK), npieces = (chunk + 31) / 32;
    return (size_t)chunk * 4 + (size_t)2 * npieces * C * 4 + 256;
}

template <typename T>
int embed_backward(const int *tok, const T *dx, float *dwte, float *dwpe, int B, int Tn, int C, int V,
                   cudaStream_t st, void *ws) {
    const int n = B * Tn;
    if (!ws || C % 8 || V > 65536) {  // fp32 atomics: the order of additions into a shared row is not fixed
        const int64_t ne = (int64_t)n * C;
        embed_bwd_wte_kernel<T><<<ceil_div(ne, 256), 256, 0, st>>>(tok, dx, dwte, n, C, V);
        GPT2_CUDA_TRY(cudaGetLastError());
        gpt2_note_launches(1);
    } else {
        static PerDevice attr_pd;
        const int sort_smem = (2 * EMB_CHUNK + 32 * 256) * 4;
        int unused = 0;
        if (int rc = per_device(attr_pd, unused, [&](int &v) -> int {
                GPT2_CUDA_TRY(
                    cudaFuncSetAttribute(embed_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, sort_smem));
                v = 1;
                return GPT2_OK;
            }))
            return rc;
        uint32_t *keys = reinterpret_cast<uint32_t *>(ws);
        const int npieces_max = (std::min(n, EMB_CHUNK) + 31) / 32;
        float *part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ws) +
                                                (((size_t)std::min(n, EMB_CHUNK) * 4 + 255) & ~(size_t)255));
        (void)npieces_max;
        // chunks of positions in order; within a chunk, rows in sorted order
        for (int c0 = 0; c0 < n; c0 += EMB_CHUNK) {
            const int m = std::min(EMB_CHUNK, n - c0), npieces = (m + 31) / 32, nslab = (C + 255) / 256;
            embed_sort_kernel<<<1, EMB_SORT_THREADS, sort_smem, st>>>(tok + c0, m, V, keys);
            embed_runs_kernel<T><<<ceil_div(npieces * nslab, 8), 256, 0, st>>>(keys, dx + (int64_t)c0 * C, dwte, part,
                                                                                m, C);
            if (npieces > 1) embed_cross_kernel<<<npieces - 1, 256, 0, st>>>(keys, part, dwte, m, C);
            GPT2_CUDA_TRY(cudaGetLastError());
            gpt2_note_launches(npieces > 1 ? 3 : 2);
        }
    }
    embed_bwd_wpe_kernel<T><<<ceil_div((int64_t)Tn * C, 256), 256, 0, st>>>(dx, dwpe, B, Tn, C);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// ============================================================== LayerNorm
// One warp per row; the row stays in registers (VPL 16-byte packets per lane,
// packet p = lane + 32 i covers columns [p*E, p*E + E)).
template <int E> struct F4x {  // E fp32 values loaded as float4s
    float v[E];
    __device__ __forceinline__ void load(const float *p) {
#pragma unroll
        for (int i = 0; i < E; i += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(p + i);
            v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
        }
    }
};

template <typename T, int VPL>
__global__ void ln_fwd_kernel(const T *__restrict__ x, const float *__restrict__ g, const float *__restrict__ b,
                              T *__restrict__ y, float *__restrict__ mean, float *__restrict__ rstd, int N, int C) {
    constexpr int E = Pack16<T>::N;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= N) return;
    const int npk = C / E;
    const T *xr = x + (int64_t)row * C;
    Pack16<T> v[VPL];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int p = lane + 32 * i;
        if (p < npk) {
            v[i].load_stream(xr + p * E);
#pragma unroll
            for (int e = 0; e < E; ++e) s += v[i].get(e);
        }
    }
    const float mu = warp_sum(s) / C;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int p = lane + 32 * i;
        if (p < npk) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float d = v[i].get(e) - mu;
                q += d * d;
            }
        }
    }
    const float rs = rsqrt_t<T>(warp_sum(q) / C + 1e-5f);
    T *yr = y + (int64_t)row * C;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int p = lane + 32 * i;
        if (p < npk) {
            F4x<E> gg, bb;
            gg.load(g + p * E);
            bb.load(b + p * E);
            Pack16<T> o;
#pragma unroll
            for (int e = 0; e < E; ++e) o.set(e, (v[i].get(e) - mu) * rs * gg.v[e] + bb.v[e]);
            o.store(yr + p * E);
        }
    }
    if (lane == 0) {
        mean[row] = mu;
        rstd[row] = rs;
    }
}

// bf16 rows (forward and backward): the computation of the generic kernels with the packets handled as 32-bit words
// (a bf16 is the top half of an fp32, so unpacking is one shift or mask) and the
// output rounded two elements at a time.
__device__ __forceinline__ F2 bf16x2_f2(uint32_t w) { return f2(bf16_lo(w), bf16_hi(w)); }
__device__ __forceinline__ uint32_t f2_bf16x2(F2 v) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f2_lo(v), f2_hi(v));
    return *reinterpret_cast<uint32_t *>(&h);
}

// Rows of up to 1,024 bf16 (VPL <= 4 packets a lane): six blocks per SM (40 registers, no
// spills) instead of the five the unconstrained build allows; wider rows unconstrained.
template <int VPL>
__global__ void __launch_bounds__(256, (VPL <= 4 ? 6 : 1)) ln_fwd_bf16_kernel(const bf16 *__restrict__ x, const float *__restrict__ g,
                                   const float *__restrict__ b, bf16 *__restrict__ y, float *__restrict__ mean,
                                   float *__restrict__ rstd, int N, int C, uint8_t *__restrict__ q,
                                   float *__restrict__ qinv) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= N) return;
    const int npk = C / 8;
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + (int64_t)row * C);
    uint4 v[VPL];
    F2 s = f2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int p = lane + 32 * i;
        if (p < npk) {
            v[i] = __ldcs(xr + p);
            s = f2_add(s, f2_add(f2_add(bf16x2_f2(v[i].x), bf16x2_f2(v[i].y)),
                                 f2_add(bf16x2_f2(v[i].z), bf16x2_f2(v[i].w))));
        }
    }
    const float mu = warp_sum(f2_lo(s) + f2_hi(s)) / C;
    const F2 nmu = f2(-mu, -mu);
    F2 ss = f2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int p = lane + 32 * i;
        if (p < npk) {
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const F2 d = f2_add(bf16x2_f2(w[k]), nmu);
                ss = f2_fma(d, d, ss);
            }
        }
    }
    const float rs = rsqrtf(warp_sum(f2_lo(ss) + f2_hi(ss)) / C + 1e-5f);
    const F2 rs2 = f2(rs, rs);
    uint4 *yr = reinterpret_cast<uint4 *>(y + (int64_t)row * C);
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int p = lane + 32 * i;
        if (p < npk) {
            const float4 g0 = *reinterpret_cast<const float4 *>(g + p * 8);
            const float4 g1 = *reinterpret_cast<const float4 *>(g + p * 8 + 4);
            const float4 b0 = *reinterpret_cast<const float4 *>(b + p * 8);
            const float4 b1 = *reinterpret_cast<const float4 *>(b + p * 8 + 4);
            const F2 gk[4] = {f2(g0.x, g0.y), f2(g0.z, g0.w), f2(g1.x, g1.y), f2(g1.z, g1.w)};
            const F2 bk[4] = {f2(b0.x, b0.y), f2(b0.z, b0.w), f2(b1.x, b1.y), f2(b1.z, b1.w)};
            const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            uint32_t o[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) o[k] = f2_bf16x2(f2_fma(f2_mul(f2_add(bf16x2_f2(w[k]), nmu), rs2), gk[k], bk[k]));
            yr[p] = make_uint4(o[0], o[1], o[2], o[3]);
            v[i] = make_uint4(o[0], o[1], o[2], o[3]);  // the stored row, for the E4M3 copy
        }
    }
    if (lane == 0) {
        mean[row] = mu;
        rstd[row] = rs;
    }
    if (q) {
        // E4M3 copy of the stored (bf16) row: s = 448 / amax in fp32, one multiply, saturating
        // round to nearest even; qinv = amax / 448 (a row of zeros: codes 0, factor 1)
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int p = lane + 32 * i;
            if (p < npk) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
            }
        }
        amax = warp_max(amax);
        const float s = amax > 0.f ? 448.0f / amax : 1.0f;
        uint8_t *qr = q + (int64_t)row * C;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int p = lane + 32 * i;
            if (p < npk) {
                const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
                uint32_t lo = 0, hi = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t pair = e4m3_of(bf16_lo(w[k]) * s) | (e4m3_of(bf16_hi(w[k]) * s) << 8);
                    if (k < 2)
                        lo |= pair << (16 * k);
                    else
                        hi |= pair << (16 * (k - 2));
                }
                *reinterpret_cast<uint2 *>(qr + p * 8) = make_uint2(lo, hi);
            }
        }
        if (lane == 0) qinv[row] = amax > 0.f ? amax / 448.0f : 1.0f;
    }
}

template <typename T> static int ln_vpl(int C) {
    const int npk = C / Pack16<T>::N;
    const int per_lane = (npk + 31) / 32;
    return per_lane <= 8 ? per_lane : 0;
}

#define LN_VPL_SWITCH(VPLV, ...)                                         \
    switch (VPLV) {                                                      \
        case 1: { constexpr int V_ = 1; __VA_ARGS__; } break;            \
        case 2: { constexpr int V_ = 2; __VA_ARGS__; } break;            \
        case 3: { constexpr int V_ = 3; __VA_ARGS__; } break;            \
        case 4: { constexpr int V_ = 4; __VA_ARGS__; } break;            \
        case 5: { constexpr int V_ = 5; __VA_ARGS__; } break;            \
        case 6: { constexpr int V_ = 6; __VA_ARGS__; } break;            \
        case 7: { constexpr int V_ = 7; __VA_ARGS__; } break;            \
        case 8: { constexpr int V_ = 8; __VA_ARGS__; } break;            \
        default: return GPT2_ERR_BAD_SHAPE;                              \
    }

template <typename T>
int layernorm_forward(const T *x, const float *g, const float *b, T *y, float *mean, float *rstd, int N, int C,
                      cudaStream_t st, uint8_t *q, float *qinv) {
    if (C % Pack16<T>::N) return GPT2_ERR_BAD_SHAPE;
    const int warps = 8, grid = ceil_div(N, warps);
    if constexpr (sizeof(T) == 2) {
        LN_VPL_SWITCH(ln_vpl<T>(C),
                      ln_fwd_bf16_kernel<V_><<<grid, 32 * warps, 0, st>>>(x, g, b, y, mean, rstd, N, C, q, qinv))
    } else {
        if (q) return GPT2_ERR_UNSUPPORTED;  // the E4M3 copy is made from bf16 rows only
        LN_VPL_SWITCH(ln_vpl<T>(C), ln_fwd_kernel<T, V_><<<grid, 32 * warps, 0, st>>>(x, g, b, y, mean, rstd, N, C))
    }
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// dx = rstd (dy*g - mean(dy*g) - xhat mean(dy*g*xhat)).  One block of 16
// warps per SM; each warp takes one row at a time with its three input rows
// requested together.  Each lane keeps the dg / db / column-sum partials of
// its columns in registers over the rows its warp handles (VPL is the exact
// packet count per lane).  At the end every warp writes its partials to its
// own shared-memory row, the block sums the rows column by column (no shared
// atomics) and adds the result to the fp32 gradients with one atomic per
// column.
template <typename T, int VPL>
__global__ void __launch_bounds__(512, 1) ln_bwd_kernel(const T *__restrict__ dy, const T *__restrict__ x,
                                                        const float *__restrict__ mean,
                                                        const float *__restrict__ rstd, const float *__restrict__ g,
                                                        const T *dres_in, T *dres_out, float *__restrict__ dg,
                                                        float *__restrict__ db, float *__restrict__ dsum, int N,
                                                        int C) {
    constexpr int E = Pack16<T>::N, E2 = E / 2;  // elements per packet, element pairs per packet
    extern __shared__ float sh[];  // [warps][3C]: dg, db, column sums of dres_out
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, warps = blockDim.x >> 5;
    const int npk = C / E;
    // the arithmetic runs on element pairs (.f32x2)
    F2 adg[VPL][E2], adb[VPL][E2], ads[VPL][E2];
#pragma unroll
    for (int i = 0; i < VPL; ++i)
#pragma unroll
        for (int k = 0; k < E2; ++k) adg[i][k] = adb[i][k] = ads[i][k] = f2(0.f, 0.f);
    for (int row = blockIdx.x * warps + wid; row < N; row += gridDim.x * warps) {
        const int64_t off = (int64_t)row * C;
        // all three input rows are requested before any is used: one memory
        // round trip per row (dres_in may alias dres_out; rows are disjoint)
        Pack16<T> vdy[VPL], vx[VPL], vr[VPL];
        const float mu = mean[row], rs = rstd[row];
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int p = lane + 32 * i;
            if (p < npk) {
                vdy[i].load_stream(dy + off + p * E);
                vx[i].load_stream(x + off + p * E);
                if (dres_in) vr[i].load_stream(dres_in + off + p * E);
            }
        }
        const F2 rs2 = f2(rs, rs), nmr = f2(-mu * rs, -mu * rs);  // xhat = x rs - mu rs
        F2 s1 = f2(0.f, 0.f), s2 = f2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int p = lane + 32 * i;
            if (p < npk) {
                F4x<E> gg;
                gg.load(g + p * E);
#pragma unroll
                for (int k = 0; k < E2; ++k) {
                    const F2 d = f2(vdy[i].get(2 * k), vdy[i].get(2 * k + 1));
                    const F2 xh = f2_fma(f2(vx[i].get(2 * k), vx[i].get(2 * k + 1)), rs2, nmr);
                    const F2 dxh = f2_mul(d, f2(gg.v[2 * k], gg.v[2 * k + 1]));
                    s1 = f2_add(s1, dxh);
                    s2 = f2_fma(dxh, xh, s2);
                    adg[i][k] = f2_fma(d, xh, adg[i][k]);
                    adb[i][k] = f2_add(adb[i][k], d);
                }
            }
        }
        const float m1 = warp_sum(f2_lo(s1) + f2_hi(s1)) / C, m2 = warp_sum(f2_lo(s2) + f2_hi(s2)) / C;
        const F2 nm1 = f2(-m1, -m1), nm2 = f2(-m2, -m2);
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int p = lane + 32 * i;
            if (p < npk) {
                Pack16<T> o;
                F4x<E> gg;
                gg.load(g + p * E);
#pragma unroll
                for (int k = 0; k < E2; ++k) {
                    const F2 xh = f2_fma(f2(vx[i].get(2 * k), vx[i].get(2 * k + 1)), rs2, nmr);
                    // dx = rs (dy g - m1 - xhat m2)
                    const F2 t = f2_fma(xh, nm2, f2_fma(f2(vdy[i].get(2 * k), vdy[i].get(2 * k + 1)),
                                                         f2(gg.v[2 * k], gg.v[2 * k + 1]), nm1));
                    F2 ov = f2_mul(t, rs2);
                    if (dres_in) ov = f2_add(ov, f2(vr[i].get(2 * k), vr[i].get(2 * k + 1)));
                    o.set(2 * k, f2_lo(ov));
                    o.set(2 * k + 1, f2_hi(ov));
                    // column sums of the stored (rounded) output
                    ads[i][k] = f2_add(ads[i][k], f2(o.get(2 * k), o.get(2 * k + 1)));
                }
                o.store(dres_out + off + p * E);
            }
        }
    }
    float *my = sh + wid * 3 * C;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int p = lane + 32 * i;
        if (p < npk)
#pragma unroll
            for (int k = 0; k < E2; ++k) {
                my[p * E + 2 * k] = f2_lo(adg[i][k]);
                my[p * E + 2 * k + 1] = f2_hi(adg[i][k]);
                my[C + p * E + 2 * k] = f2_lo(adb[i][k]);
                my[C + p * E + 2 * k + 1] = f2_hi(adb[i][k]);
                my[2 * C + p * E + 2 * k] = f2_lo(ads[i][k]);
                my[2 * C + p * E + 2 * k + 1] = f2_hi(ads[i][k]);
            }
    }
    __syncthreads();
    const int ncol = dsum ? 3 * C : 2 * C;
    for (int c = threadIdx.x; c < ncol; c += blockDim.x) {
        float sum = 0.f;
        for (int w = 0; w < warps; ++w) sum += sh[w * 3 * C + c];
        atomicAdd(c < C ? dg + c : c < 2 * C ? db + (c - C) : dsum + (c - 2 * C), sum);
    }
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem_dst)),
                 "l"(gsrc)
                 : "memory");
}

template <int VPL>
__global__ void __launch_bounds__(512, 1) ln_bwd_bf16_kernel(const bf16 *__restrict__ dy, const bf16 *__restrict__ x,
                                                             const float *__restrict__ mean,
                                                             const float *__restrict__ rstd,
                                                             const float *__restrict__ g, const bf16 *dres_in,
                                                             bf16 *dres_out, float *__restrict__ dg,
                                                             float *__restrict__ db, float *__restrict__ dsum, int N,
                                                             int C) {
    // Per warp, 3C floats of shared memory (and C floats for the gain after all of them): while
    // rows are processed they hold
    // two row buffers (dy, x, dres_in: 3 x C bf16 each), the next row being
    // fetched (cp.async) while the current one is computed; at the end they hold
    // the warp's dg, db and column-sum partials.  A lane only ever touches its
    // own packets of a buffer, so no warp synchronisation is needed around them.
    extern __shared__ float sh[];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, warps = blockDim.x >> 5;
    const int npk = C / 8;
    uint8_t *wbuf = reinterpret_cast<uint8_t *>(sh + (size_t)wid * 3 * C);
    // the gain, staged once per block in shared memory after the warps' rows: both passes of
    // every row read it from there (global / L1 reads of it were measured 3% slower in the step)
    float *sg = sh + (size_t)warps * 3 * C;
    for (int c = threadIdx.x * 4; c < C; c += blockDim.x * 4)
        *reinterpret_cast<float4 *>(sg + c) = *reinterpret_cast<const float4 *>(g + c);
    __syncthreads();
    auto slot = [&](int b, int a) { return reinterpret_cast<uint4 *>(wbuf + (size_t)(b * 3 + a) * C * 2); };
    auto fetch = [&](int row, int b) {
        const int64_t off = (int64_t)row * C;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int p = lane + 32 * i;
            if (p < npk) {
                cp_async16(slot(b, 0) + p, reinterpret_cast<const uint4 *>(dy + off) + p);
                cp_async16(slot(b, 1) + p, reinterpret_cast<const uint4 *>(x + off) + p);
                if (dres_in) cp_async16(slot(b, 2) + p, reinterpret_cast<const uint4 *>(dres_in + off) + p);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    F2 adg[VPL][4], adb[VPL][4], ads[VPL][4];
#pragma unroll
    for (int i = 0; i < VPL; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) adg[i][k] = adb[i][k] = ads[i][k] = f2(0.f, 0.f);
    const int row0 = blockIdx.x * warps + wid, rstep = gridDim.x * warps;
    float nmu = 0.f, nrs = 0.f;
    if (row0 < N) {
        fetch(row0, 0);
        nmu = mean[row0];
        nrs = rstd[row0];
    }
    int b = 0;
    for (int row = row0; row < N; row += rstep, b ^= 1) {
        const int64_t off = (int64_t)row * C;
        const float mu = nmu, rs = nrs;
        if (row + rstep < N) {
            fetch(row + rstep, b ^ 1);
            nmu = mean[row + rstep];
            nrs = rstd[row + rstep];
        } else {
            asm volatile("cp.async.commit_group;" ::: "memory");  // keeps the group count uniform
        }
        asm volatile("cp.async.wait_group 1;" ::: "memory");  // this row's copies have landed
        // the row stays in shared memory: each pass reads the packets it needs
        const uint4 *vdy = slot(b, 0), *vx = slot(b, 1), *vr = slot(b, 2);
        const F2 rs2 = f2(rs, rs), nmr = f2(-mu * rs, -mu * rs);  // xhat = x rs - mu rs
        F2 s1 = f2(0.f, 0.f), s2 = f2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int p = lane + 32 * i;
            if (p < npk) {
                const float4 g0 = *reinterpret_cast<const float4 *>(sg + p * 8);
                const float4 g1 = *reinterpret_cast<const float4 *>(sg + p * 8 + 4);
                const F2 gk[4] = {f2(g0.x, g0.y), f2(g0.z, g0.w), f2(g1.x, g1.y), f2(g1.z, g1.w)};
                const uint4 pd = vdy[p], px = vx[p];
                const uint32_t wd[4] = {pd.x, pd.y, pd.z, pd.w};
                const uint32_t wx[4] = {px.x, px.y, px.z, px.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const F2 d = bf16x2_f2(wd[k]);
                    const F2 xh = f2_fma(bf16x2_f2(wx[k]), rs2, nmr);
                    const F2 dxh = f2_mul(d, gk[k]);
                    s1 = f2_add(s1, dxh);
                    s2 = f2_fma(dxh, xh, s2);
                    adg[i][k] = f2_fma(d, xh, adg[i][k]);
                    adb[i][k] = f2_add(adb[i][k], d);
                }
            }
        }
        const float m1 = warp_sum(f2_lo(s1) + f2_hi(s1)) / C, m2 = warp_sum(f2_lo(s2) + f2_hi(s2)) / C;
        const F2 nm1 = f2(-m1, -m1), nm2 = f2(-m2, -m2);
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int p = lane + 32 * i;
            if (p < npk) {
                const float4 g0 = *reinterpret_cast<const float4 *>(sg + p * 8);
                const float4 g1 = *reinterpret_cast<const float4 *>(sg + p * 8 + 4);
                const F2 gk[4] = {f2(g0.x, g0.y), f2(g0.z, g0.w), f2(g1.x, g1.y), f2(g1.z, g1.w)};
                const uint4 pd = vdy[p], px = vx[p], pr = dres_in ? vr[p] : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t wd[4] = {pd.x, pd.y, pd.z, pd.w};
                const uint32_t wx[4] = {px.x, px.y, px.z, px.w};
                const uint32_t wr[4] = {pr.x, pr.y, pr.z, pr.w};
                uint32_t wo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const F2 xh = f2_fma(bf16x2_f2(wx[k]), rs2, nmr);
                    // dx = rs (dy g - m1 - xhat m2)
                    const F2 t = f2_fma(xh, nm2, f2_fma(bf16x2_f2(wd[k]), gk[k], nm1));
                    F2 ov = f2_mul(t, rs2);
                    if (dres_in) ov = f2_add(ov, bf16x2_f2(wr[k]));
                    wo[k] = f2_bf16x2(ov);
                    // column sums of the stored (rounded) output
                    ads[i][k] = f2_add(ads[i][k], bf16x2_f2(wo[k]));
                }
                reinterpret_cast<uint4 *>(dres_out + off)[p] = make_uint4(wo[0], wo[1], wo[2], wo[3]);
            }
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncwarp();  // the row buffers become the partial rows
    float *my = sh + wid * 3 * C;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int p = lane + 32 * i;
        if (p < npk)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int c = p * 8 + 2 * k;
                *reinterpret_cast<float2 *>(my + c) = make_float2(f2_lo(adg[i][k]), f2_hi(adg[i][k]));
                *reinterpret_cast<float2 *>(my + C + c) = make_float2(f2_lo(adb[i][k]), f2_hi(adb[i][k]));
                *reinterpret_cast<float2 *>(my + 2 * C + c) = make_float2(f2_lo(ads[i][k]), f2_hi(ads[i][k]));
            }
    }
    __syncthreads();
    const int ncol = dsum ? 3 * C : 2 * C;
    for (int c = threadIdx.x; c < ncol; c += blockDim.x) {
        float sum = 0.f;
        for (int w = 0; w < warps; ++w) sum += sh[w * 3 * C + c];
        atomicAdd(c < C ? dg + c : c < 2 * C ? db + (c - C) : dsum + (c - 2 * C), sum);
    }
}

template <typename T>
int layernorm_backward(const T *dy, const T *x, const float *mean, const float *rstd, const float *g, const T *dres_in,
                       T *dres_out, float *dg, float *db, int N, int C, cudaStream_t st, float *dsum) {
    if (C % Pack16<T>::N) return GPT2_ERR_BAD_SHAPE;
    // 16 warps per block unless the per-warp partial rows (3C floats each) do not fit in shared memory
    const int warps = std::max(1, std::min(16, (int)((227 * 1024 - C * sizeof(float)) / (3 * C * sizeof(float)))));
    int dev = 0, sms = 0;
    GPT2_CUDA_TRY(cudaGetDevice(&dev));
    GPT2_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int grid = std::max(1, std::min(ceil_div(N, warps), sms));
    const size_t smem = (size_t)warps * 3 * C * sizeof(float) + (sizeof(T) == 2 ? C * sizeof(float) : 0);
    if constexpr (sizeof(T) == 2) {
        LN_VPL_SWITCH(ln_vpl<T>(C), {
            GPT2_CUDA_TRY(
                cudaFuncSetAttribute(ln_bwd_bf16_kernel<V_>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
            ln_bwd_bf16_kernel<V_><<<grid, 32 * warps, smem, st>>>(dy, x, mean, rstd, g, dres_in, dres_out, dg, db, dsum,
                                                                   N, C);
        })
    } else {
        LN_VPL_SWITCH(ln_vpl<T>(C), {
            GPT2_CUDA_TRY(
                cudaFuncSetAttribute(ln_bwd_kernel<T, V_>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
            ln_bwd_kernel<T, V_><<<grid, 32 * warps, smem, st>>>(dy, x, mean, rstd, g, dres_in, dres_out, dg, db, dsum, N,
                                                                 C);
        })
    }
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// ============================================================== bias gradient
// 256 threads: 8 column packets x 32 row lanes; partial sums reduced in shared
// memory, one atomic per column per block.
template <typename T>
__global__ void colsum_kernel(const T *__restrict__ dy, int M, int N, float *__restrict__ db, int rows_per_block) {
    constexpr int E = Pack16<T>::N;
    __shared__ float sh[32][8 * E + 1];
    const int cp = threadIdx.x & 7, rl = threadIdx.x >> 3;
    const int col = (blockIdx.x * 8 + cp) * E;
    const int r0 = blockIdx.y * rows_per_block, r1 = min(M, r0 + rows_per_block);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    if (col < N) {
        // four rows in flight per thread (the loads do not depend on each other)
        int r = r0 + rl;
        for (; r + 96 < r1; r += 128) {
            Pack16<T> v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u].load_stream(dy + (int64_t)(r + 32 * u) * N + col);
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] += v[u].get(e);
        }
        for (; r < r1; r += 32) {
            Pack16<T> v;
            v.load_stream(dy + (int64_t)r * N + col);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] += v.get(e);
        }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) sh[rl][cp * E + e] = acc[e];
    __syncthreads();
    if (threadIdx.x < 8 * E) {
        const int c = blockIdx.x * 8 * E + threadIdx.x;
        float s = 0.f;
        for (int r = 0; r < 32; ++r) s += sh[r][threadIdx.x];
        if (c < N) atomicAdd(db + c, s);
    }
}

template <typename T>
int column_sum(const T *dy, int M, int N, float *db, cudaStream_t st) {
    constexpr int E = Pack16<T>::N;
    if (N % E) return GPT2_ERR_BAD_SHAPE;
    const int gx = ceil_div(N, 8 * E);
    const int gy = std::max(1, std::min(ceil_div(M, 256), std::max(1, 592 / gx)));
    const int rpb = ceil_div(M, gy);
    colsum_kernel<T><<<dim3(gx, gy), 256, 0, st>>>(dy, M, N, db, rpb);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// ============================================================== classifier
template <typename T>
__device__ __forceinline__ void lse_merge(float &m, float &s, float om, float os) {
    if (om == -INFINITY) return;
    if (m == -INFINITY) {
        m = om;
        s = os;
        return;
    }
    const float mn = fmaxf(m, om);
    s = s * exp_t<T>(m - mn) + os * exp_t<T>(om - mn);
    m = mn;
}

// One block per row (grid-stride): pass 1 online max / sum-exp over v < V,
// pass 2 writes dz = (softmax - onehot) * dscale in place (0 for v >= V).
template <typename T>
__global__ void __launch_bounds__(1024) classifier_kernel(T *logits, const int *__restrict__ targets,
                                                          float *__restrict__ loss_rows, int N, int V, int Vp,
                                                          float dscale, int *err) {
    constexpr int E = Pack16<T>::N;
    __shared__ float sm_m[32], sm_s[32];
    __shared__ float sh_lse;
    __shared__ int sh_tg;
    const int npk = Vp / E;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int row = blockIdx.x; row < N; row += gridDim.x) {
        T *z = logits + (int64_t)row * Vp;
        float m = -INFINITY, s = 0.f;
        for (int p = threadIdx.x; p < npk; p += blockDim.x) {
            Pack16<T> v;
            v.load(z + p * E);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                if (p * E + e < V) {
                    const float x = v.get(e);
                    if (x > m) {
                        s = s * exp_t<T>(m - x) + 1.f;
                        m = x;
                    } else {
                        s += exp_t<T>(x - m);
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, s, o);
            lse_merge<T>(m, s, om, os);
        }
        if (lane == 0) {
            sm_m[wid] = m;
            sm_s[wid] = s;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            float M = sm_m[0], S = sm_s[0];
            for (int w = 1; w < nw; ++w) lse_merge<T>(M, S, sm_m[w], sm_s[w]);
            const float lse = M + logf(S);
            int tg = targets[row];
            if (tg < 0 || tg >= V) {
                raise_device_error(err, DEVERR_BAD_TOKEN);
                tg = 0;
            }
            loss_rows[row] = lse - to_f32(z[tg]);
            sh_lse = lse;
            sh_tg = tg;
        }
        __syncthreads();
        const float lse = sh_lse;
        const int tg = sh_tg;
        for (int p = threadIdx.x; p < npk; p += blockDim.x) {
            Pack16<T> v;
            v.load(z + p * E);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int c = p * E + e;
                float d = 0.f;
                if (c < V) {
                    d = exp_t<T>(v.get(e) - lse);
                    if (c == tg) d -= 1.f;
                    d *= dscale;
                }
                v.set(e, d);
            }
            v.store(z + p * E);
        }
        __syncthreads();
    }
}

// Register-resident variant: the row (NPK packets per thread) is read once,
// max and sum-exp are block reductions over registers, dz is written once.
template <typename T, int NPK>
__global__ void __launch_bounds__(1024) classifier_reg_kernel(T *logits, const int *__restrict__ targets,
                                                              float *__restrict__ loss_rows, int N, int V, int Vp,
                                                              float dscale, int *err) {
    constexpr int E = Pack16<T>::N;
    __shared__ float red_m[2][32], red_s[2][32];
    const int npk = Vp / E;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int par = 0;
    for (int row = blockIdx.x; row < N; row += gridDim.x, par ^= 1) {
        T *z = logits + (int64_t)row * Vp;
        int tg = targets[row];
        const bool bad = tg < 0 || tg >= V;
        if (bad) tg = 0;
        Pack16<T> v[NPK];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < NPK; ++i) {
            const int p = threadIdx.x + i * blockDim.x;
            if (p < npk) {
                v[i].load_stream(z + p * E);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    if (p * E + e < V) m = fmaxf(m, v[i].get(e));
            }
        }
        m = warp_max(m);
        if (lane == 0) red_m[par][wid] = m;
        __syncthreads();
        float M = red_m[par][0];
        for (int w = 1; w < nw; ++w) M = fmaxf(M, red_m[par][w]);
        float s = 0.f, zt = 0.f;
#pragma unroll
        for (int i = 0; i < NPK; ++i) {
            const int p = threadIdx.x + i * blockDim.x;
            if (p < npk) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int c = p * E + e;
                    if (c < V) s += exp_t<T>(v[i].get(e) - M);
                    if (c == tg) zt = v[i].get(e);
                }
            }
        }
        s = warp_sum(s);
        if (lane == 0) red_s[par][wid] = s;
        __syncthreads();
        float S = 0.f;
        for (int w = 0; w < nw; ++w) S += red_s[par][w];
        const float lse = M + logf(S);
        if (tg / E % blockDim.x == threadIdx.x) {  // the thread holding the target logit
            loss_rows[row] = lse - zt;
            if (bad) raise_device_error(err, DEVERR_BAD_TOKEN);
        }
#pragma unroll
        for (int i = 0; i < NPK; ++i) {
            const int p = threadIdx.x + i * blockDim.x;
            if (p < npk) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int c = p * E + e;
                    float d = 0.f;
                    if (c < V) {
                        d = exp_t<T>(v[i].get(e) - lse);
                        if (c == tg) d -= 1.f;
                        d *= dscale;
                    }
                    v[i].set(e, d);
                }
                v[i].store(z + p * E);
            }
        }
    }
}

// bf16 specialisation tuned for instruction count: bf16 pairs are unpacked
// with integer shifts, only the packet that straddles V takes per-element
// checks, and exp is evaluated once per logit: e = 2^(x log2e - M log2e) is
// summed in fp32 and kept as bf16 in the row registers, then
// dz = e * dscale / S.  The target logit's dz is recomputed in fp32 from the
// logit itself (p_t - 1 loses no precision when p_t is close to 1).
__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ uint32_t bf_pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <int NPK>
__global__ void __launch_bounds__(1024) classifier_bf16_kernel(bf16 *logits, const int *__restrict__ targets,
                                                               float *__restrict__ loss_rows, int N, int V, int Vp,
                                                               float dscale, int *err) {
    __shared__ float red_m[2][32], red_s[2][32];
    const int npk = Vp >> 3;
    const int full_pk = V >> 3;  // packets entirely below V
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const float L2E = 1.4426950408889634f;
    int par = 0;
    for (int row = blockIdx.x; row < N; row += gridDim.x, par ^= 1) {
        bf16 *z = logits + (int64_t)row * Vp;
        int tg = targets[row];
        const bool bad = tg < 0 || tg >= V;
        if (bad) tg = 0;
        uint4 v[NPK];
        float m = -INFINITY, zt = 0.f;
#pragma unroll
        for (int i = 0; i < NPK; ++i) {
            const int p = threadIdx.x + i * blockDim.x;
            if (p < npk) {
                v[i] = __ldcs(reinterpret_cast<const uint4 *>(z) + p);
                const uint32_t *u = &v[i].x;
                if (p == (tg >> 3)) {  // keep the target logit itself (fp32 of its bf16 value)
                    const int k = (tg & 7) >> 1;
                    const uint32_t w = k == 0 ? v[i].x : k == 1 ? v[i].y : k == 2 ? v[i].z : v[i].w;
                    zt = (tg & 1) ? bf_hi(w) : bf_lo(w);
                }
                if (p < full_pk) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) m = fmaxf(m, fmaxf(bf_lo(u[k]), bf_hi(u[k])));
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (p * 8 + 2 * k < V) m = fmaxf(m, bf_lo(u[k]));
                        if (p * 8 + 2 * k + 1 < V) m = fmaxf(m, bf_hi(u[k]));
                    }
                }
            }
        }
        m = warp_max(m);
        if (lane == 0) red_m[par][wid] = m;
        __syncthreads();
        float M = red_m[par][0];
        for (int w = 1; w < nw; ++w) M = fmaxf(M, red_m[par][w]);
        const float Mc = M * L2E;
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < NPK; ++i) {
            const int p = threadIdx.x + i * blockDim.x;
            if (p < npk) {
                uint32_t *u = &v[i].x;
                if (p < full_pk) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float a = exp2f(fmaf(bf_lo(u[k]), L2E, -Mc));
                        const float b = exp2f(fmaf(bf_hi(u[k]), L2E, -Mc));
                        s += a + b;
                        u[k] = bf_pack(a, b);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int c = p * 8 + 2 * k;
                        const float a = c < V ? exp2f(fmaf(bf_lo(u[k]), L2E, -Mc)) : 0.f;
                        const float b = c + 1 < V ? exp2f(fmaf(bf_hi(u[k]), L2E, -Mc)) : 0.f;
                        s += a + b;
                        u[k] = bf_pack(a, b);
                    }
                }
            }
        }
        s = warp_sum(s);
        if (lane == 0) red_s[par][wid] = s;
        __syncthreads();
        float S = 0.f;
        for (int w = 0; w < nw; ++w) S += red_s[par][w];
        const float lse = M + logf(S);
        const float scale = dscale / S;
#pragma unroll
        for (int i = 0; i < NPK; ++i) {
            const int p = threadIdx.x + i * blockDim.x;
            if (p < npk) {
                uint32_t *u = &v[i].x;
#pragma unroll
                for (int k = 0; k < 4; ++k) u[k] = bf_pack(bf_lo(u[k]) * scale, bf_hi(u[k]) * scale);
                reinterpret_cast<uint4 *>(z)[p] = v[i];
            }
        }
        if (threadIdx.x == (tg >> 3) % blockDim.x) {  // this thread loaded and stored the target's packet
            loss_rows[row] = lse - zt;
            z[tg] = __float2bfloat16_rn((__expf(zt - lse) - 1.0f) * dscale);
            if (bad) raise_device_error(err, DEVERR_BAD_TOKEN);
        }
    }
}

// Pipelined variant for large vocabularies: each row (Vp bf16) arrives by one
// bulk asynchronous copy into one of two shared-memory buffers; a row is moved
// to registers as soon as it has landed and its buffer is refilled, so three
// rows per SM are in flight (two copies and the one being computed).
// Per row: max (block reduction), e = 2^(x log2e - M log2e) rounded to bf16 and
// summed in fp32, then dz = e * dscale / S written with 16-byte stores; the
// target logit is read from the buffer and its dz recomputed in fp32.
constexpr int CLS_SMEM_THREADS = 1024;
constexpr int CLS_PPT = 7;  // 16-byte packets of a row per thread: Vp <= 7 * 1024 * 8

// 2^x with the hardware approximation (MUFU.EX2, flush-to-zero); the values
// are stored as bf16 and summed in fp32, far above its error.
__device__ __forceinline__ float ex2_hw(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t cls_su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__global__ void __launch_bounds__(CLS_SMEM_THREADS, 1)
    classifier_smem_kernel(bf16 *logits, const int *__restrict__ targets, float *__restrict__ loss_rows, int N, int V,
                           int Vp, int row_bytes_padded, float dscale, int *err) {
    extern __shared__ __align__(128) uint8_t cls_smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(cls_smem + 2 * row_bytes_padded);
    __shared__ float red_m[2][32], red_s[2][32];
    const int npk = Vp >> 3;
    const int full_pk = V >> 3;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const float L2E = 1.4426950408889634f;
    const uint32_t row_bytes = (uint32_t)Vp * 2;
    auto issue = [&](int row, int buf) {
        const uint32_t b = cls_su32(&bar[buf]);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(row_bytes) : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                cls_su32(cls_smem + buf * row_bytes_padded)),
            "l"(logits + (int64_t)row * Vp), "r"(row_bytes), "r"(b)
            : "memory");
    };
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(cls_su32(&bar[0])) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(cls_su32(&bar[1])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if ((int)blockIdx.x < N) issue(blockIdx.x, 0);
        if ((int)(blockIdx.x + gridDim.x) < N) issue(blockIdx.x + gridDim.x, 1);
    }
    __syncthreads();
    int i = 0;
    for (int row = blockIdx.x; row < N; row += gridDim.x, ++i) {
        const int buf = i & 1;
        uint4 *zs = reinterpret_cast<uint4 *>(cls_smem + buf * row_bytes_padded);
        // wait for this row's copy (bounded: a copy that never lands flags a timeout)
        {
            const uint32_t b = cls_su32(&bar[buf]), par = (i >> 1) & 1;
            uint32_t done = 0;
            const uint64_t t0 = global_timer_ns();
            while (true) {
                asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                             "selp.u32 %0, 1, 0, p;\n\t}\n"
                             : "=r"(done)
                             : "r"(b), "r"(par)
                             : "memory");
                if (done) break;
                if (global_timer_ns() - t0 > 2000000000ull) {
                    raise_device_error(err, DEVERR_TIMEOUT);
                    return;  // every thread of the block times out on the same copy
                }
            }
        }
        int tg = targets[row];
        const bool bad = tg < 0 || tg >= V;
        if (bad) tg = 0;
        // The row moves to registers (at most CLS_PPT packets per thread) and
        // its buffer is refilled with the row two ahead at once, so that copy
        // has the rest of this row and all of the next to land.
        uint4 ev[CLS_PPT];
#pragma unroll
        for (int j = 0; j < CLS_PPT; ++j) {
            const int p = threadIdx.x + j * CLS_SMEM_THREADS;
            if (p < npk) ev[j] = zs[p];
        }
        const float zt = __bfloat162float(reinterpret_cast<const bf16 *>(zs)[tg]);
        __syncthreads();  // every thread is done with this row's buffer
        if (threadIdx.x == 0 && row + 2 * (int)gridDim.x < N) issue(row + 2 * gridDim.x, buf);
        // Pass 1: row max.  Packets below full_pk hold only real columns; the
        // max of bf16 values is exact in bf16, two per instruction.
        uint32_t m2 = 0xff80ff80u;  // (-inf, -inf)
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < CLS_PPT; ++j) {
            const int p = threadIdx.x + j * CLS_SMEM_THREADS;
            if (p < full_pk) {
                asm("max.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(ev[j].x));
                asm("max.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(ev[j].y));
                asm("max.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(ev[j].z));
                asm("max.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(ev[j].w));
            } else if (p < npk) {  // the padded tail
                const uint32_t *u = &ev[j].x;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (p * 8 + 2 * k < V) m = fmaxf(m, bf_lo(u[k]));
                    if (p * 8 + 2 * k + 1 < V) m = fmaxf(m, bf_hi(u[k]));
                }
            }
        }
        m = fmaxf(m, fmaxf(bf_lo(m2), bf_hi(m2)));
        m = warp_max(m);
        if (lane == 0) red_m[buf][wid] = m;
        __syncthreads();
        float M = red_m[buf][0];
        for (int w = 1; w < nw; ++w) M = fmaxf(M, red_m[buf][w]);
        // Pass 2: e = 2^(x log2e - M log2e), rounded to bf16 in place, summed
        // in fp32; the arithmetic runs on column pairs (.f32x2).
        const F2 l2e2 = f2(L2E, L2E), nmc2 = f2(-M * L2E, -M * L2E);
        const float Mc = M * L2E;
        F2 sacc2 = f2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < CLS_PPT; ++j) {
            const int p = threadIdx.x + j * CLS_SMEM_THREADS;
            uint32_t *u = &ev[j].x;
            if (p < full_pk) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const F2 t = f2_fma(f2(bf_lo(u[k]), bf_hi(u[k])), l2e2, nmc2);
                    const float a = ex2_hw(f2_lo(t)), b2 = ex2_hw(f2_hi(t));
                    sacc2 = f2_add(sacc2, f2(a, b2));
                    u[k] = bf_pack(a, b2);
                }
            } else if (p < npk) {  // the padded tail: 0 past V
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int c = p * 8 + 2 * k;
                    const float a = c < V ? ex2_hw(fmaf(bf_lo(u[k]), L2E, -Mc)) : 0.f;
                    const float b2 = c + 1 < V ? ex2_hw(fmaf(bf_hi(u[k]), L2E, -Mc)) : 0.f;
                    sacc2 = f2_add(sacc2, f2(a, b2));
                    u[k] = bf_pack(a, b2);
                }
            }
        }
        const float sacc = warp_sum(f2_lo(sacc2) + f2_hi(sacc2));
        if (lane == 0) red_s[buf][wid] = sacc;
        __syncthreads();
        float S = 0.f;
        for (int w = 0; w < nw; ++w) S += red_s[buf][w];
        const float lse = M + logf(S);
        const float scale = dscale / S;
        const F2 scale2 = f2(scale, scale);
        // Pass 3: dz = e dscale / S from the registers, 16-byte stores
        uint4 *zg = reinterpret_cast<uint4 *>(logits + (int64_t)row * Vp);
#pragma unroll
        for (int j = 0; j < CLS_PPT; ++j) {
            const int p = threadIdx.x + j * CLS_SMEM_THREADS;
            if (p < npk) {
                uint4 v = ev[j];
                uint32_t *u = &v.x;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const F2 y = f2_mul(f2(bf_lo(u[k]), bf_hi(u[k])), scale2);
                    u[k] = bf_pack(f2_lo(y), f2_hi(y));
                }
                if (p == (tg >> 3)) {  // the target's dz from the logit itself, in fp32
                    bf16 *e8 = reinterpret_cast<bf16 *>(&v);
                    e8[tg & 7] = __float2bfloat16_rn((__expf(zt - lse) - 1.0f) * dscale);
                }
                zg[p] = v;
            }
        }
        if (threadIdx.x == 0) {
            loss_rows[row] = lse - zt;
            if (bad) raise_device_error(err, DEVERR_BAD_TOKEN);
        }
    }
}

template <typename T>
int classifier(T *logits, const int *targets, float *loss_rows, int N, int V, int Vp, float dscale, int *err,
               cudaStream_t st) {
    constexpr int E = Pack16<T>::N;
    if (Vp % E || V > Vp || V <= 0) return GPT2_ERR_BAD_SHAPE;
    const int npk = Vp / E;
    const int threads = std::min(1024, (npk + 31) / 32 * 32);
    const int npt = ceil_div(npk, threads);
    const int grid = std::min(N, 148 * 2);
    if constexpr (sizeof(T) == 2) {
        bf16 *lg = reinterpret_cast<bf16 *>(logits);
        // large rows: shared-memory pipeline (two rows of Vp bf16 in flight per SM)
        const int row_pad = (Vp * 2 + 127) / 128 * 128;
        const size_t cls_smem_bytes = 2 * (size_t)row_pad + 64;
        if (Vp >= 8192 && cls_smem_bytes <= 200 * 1024 && npk <= CLS_PPT * CLS_SMEM_THREADS) {
            static PerDevice attr_pd;
            int unused = 0;
            if (int rc = per_device(attr_pd, unused, [](int &v) -> int {
                    GPT2_CUDA_TRY(cudaFuncSetAttribute(classifier_smem_kernel,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024 + 64));
                    v = 1;
                    return GPT2_OK;
                }))
                return rc;
            int dev = 0, sms = 148;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            classifier_smem_kernel<<<std::min(N, sms), CLS_SMEM_THREADS, cls_smem_bytes, st>>>(
                lg, targets, loss_rows, N, V, Vp, row_pad, dscale, err);
            GPT2_CUDA_TRY(cudaGetLastError());
            gpt2_note_launches(1);
            return GPT2_OK;
        }
        switch (npt <= 1 ? 1 : npt <= 2 ? 2 : npt <= 4 ? 4 : npt <= 7 ? 7 : npt <= 8 ? 8 : 0) {
            case 1: classifier_bf16_kernel<1><<<grid, threads, 0, st>>>(lg, targets, loss_rows, N, V, Vp, dscale, err); break;
            case 2: classifier_bf16_kernel<2><<<grid, threads, 0, st>>>(lg, targets, loss_rows, N, V, Vp, dscale, err); break;
            case 4: classifier_bf16_kernel<4><<<grid, threads, 0, st>>>(lg, targets, loss_rows, N, V, Vp, dscale, err); break;
            case 7: classifier_bf16_kernel<7><<<grid, threads, 0, st>>>(lg, targets, loss_rows, N, V, Vp, dscale, err); break;
            case 8: classifier_bf16_kernel<8><<<grid, threads, 0, st>>>(lg, targets, loss_rows, N, V, Vp, dscale, err); break;
            default: classifier_kernel<T><<<std::min(N, 148 * 8), 512, 0, st>>>(logits, targets, loss_rows, N, V, Vp,
                                                                               dscale, err);
        }
        GPT2_CUDA_TRY(cudaGetLastError());
        gpt2_note_launches(1);
        return GPT2_OK;
    }
    switch (npt <= 1 ? 1 : npt <= 2 ? 2 : npt <= 4 ? 4 : npt <= 8 ? 8 : 0) {
        case 1: classifier_reg_kernel<T, 1><<<grid, threads, 0, st>>>(logits, targets, loss_rows, N, V, Vp, dscale, err); break;
        case 2: classifier_reg_kernel<T, 2><<<grid, threads, 0, st>>>(logits, targets, loss_rows, N, V, Vp, dscale, err); break;
        case 4: classifier_reg_kernel<T, 4><<<grid, threads, 0, st>>>(logits, targets, loss_rows, N, V, Vp, dscale, err); break;
        case 8: classifier_reg_kernel<T, 8><<<grid, threads, 0, st>>>(logits, targets, loss_rows, N, V, Vp, dscale, err); break;
        default: classifier_kernel<T><<<std::min(N, 148 * 8), 512, 0, st>>>(logits, targets, loss_rows, N, V, Vp,
                                                                            dscale, err);
    }
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

__global__ void mean_rows_kernel(const float *__restrict__ rows, int N, float *out) {
    __shared__ double sh[32];
    double s = 0.0;
    for (int i = threadIdx.x; i < N; i += blockDim.x) s += rows[i];
    s = warp_sum_d(s);
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += sh[w];
        out[0] = (float)(t / N);
    }
}

int mean_rows(const float *rows, int N, float *out, cudaStream_t st) {
    mean_rows_kernel<<<1, 1024, 0, st>>>(rows, N, out);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// One warp per row: the row's lse from its half-tile partials, combined in a fixed
// order (lane stride, then the warp tree), and its loss.
__global__ void ce_combine_kernel(const float2 *__restrict__ part, int stride, int nparts, const float *__restrict__ zt,
                                  const int *__restrict__ targets, int N, int V, float *__restrict__ lse,
                                  float *__restrict__ loss_rows, int *err) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= N) return;
    const float2 *p = part + (int64_t)row * stride;
    float m = -INFINITY;
    for (int j = lane; j < nparts; j += 32) m = fmaxf(m, p[j].x);
    m = warp_max(m);
    float s = 0.f;
    for (int j = lane; j < nparts; j += 32) {
        const float2 v = p[j];
        if (v.y > 0.f) s += v.y * expf(v.x - m);
    }
    s = warp_sum(s);
    if (lane == 0) {
        const float l = m + logf(s);
        lse[row] = l;
        loss_rows[row] = l - zt[row];
        const int t = targets[row];
        if (t < 0 || t >= V) raise_device_error(err, DEVERR_BAD_TOKEN);
    }
}

int ce_combine(const float2 *part, int stride, int nparts, const float *zt, const int *targets, int N, int V,
               float *lse, float *loss_rows, int *err, cudaStream_t st) {
    if (N <= 0 || nparts <= 0 || stride < nparts) return GPT2_ERR_BAD_SHAPE;
    ce_combine_kernel<<<ceil_div(N, 8), 256, 0, st>>>(part, stride, nparts, zt, targets, N, V, lse, loss_rows, err);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// ============================================================== GELU recompute, casts
template <typename T>
__global__ void gelu_fwd_kernel(const T *__restrict__ h, T *__restrict__ y, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    constexpr int E = Pack16<T>::N;
    if (i * E >= n) return;
    Pack16<T> v;
    v.load(h + i * E);
#pragma unroll
    for (int e = 0; e < E; ++e) v.set(e, gelu_tanh_t<T>(v.get(e)));
    v.store(y + i * E);
}

template <typename T>
int gelu_forward(const T *h, T *y, int64_t n, cudaStream_t st) {
    constexpr int E = Pack16<T>::N;
    if (n % E) return GPT2_ERR_BAD_SHAPE;
    gelu_fwd_kernel<T><<<ceil_div(n / E, 256), 256, 0, st>>>(h, y, n);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

__global__ void cast_kernel(const float *__restrict__ x, bf16 *__restrict__ y, int64_t n) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) y[i] = __float2bfloat16_rn(x[i]);
}

int cast_f32_bf16(const float *x, bf16 *y, int64_t n, cudaStream_t st) {
    cast_kernel<<<ceil_div(n, 256), 256, 0, st>>>(x, y, n);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// ============================================================== SIMT matmul
template <typename T>
__device__ __forceinline__ void simt_epilogue(int epi, float acc, int m, int n, void *D, T *D2, const T *R,
                                              int64_t ldd, const float *bias) {
    const int64_t o = (int64_t)m * ldd + n;
    const float bv = bias ? bias[n] : 0.f;
    switch (epi) {
        case GPT2_EPI_STORE: reinterpret_cast<T *>(D)[o] = from_f32<T>(acc + bv); break;
        case GPT2_EPI_RESIDUAL: reinterpret_cast<T *>(D)[o] = from_f32<T>(acc + bv + to_f32(R[o])); break;
        case GPT2_EPI_GELU: {
            const T h = from_f32<T>(acc + bv);
            reinterpret_cast<T *>(D)[o] = h;
            D2[o] = from_f32<T>(gelu_tanh_t<T>(to_f32(h)));
            break;
        }
        case GPT2_EPI_GELU_BWD: reinterpret_cast<T *>(D)[o] = from_f32<T>(acc * gelu_tanh_grad_t<T>(to_f32(R[o]))); break;
        case GPT2_EPI_ACCUM_F32: reinterpret_cast<float *>(D)[o] += acc; break;
    }
}

template <typename T>
__global__ void __launch_bounds__(256) matmul_simt_kernel(const T *__restrict__ A, int64_t sam, int64_t sak,
                                                          const T *__restrict__ Bm, int64_t sbn, int64_t sbk, void *D,
                                                          T *D2, const T *R, int64_t ldd, const float *bias, int M,
                                                          int N, int K, int epi, float alpha) {
    __shared__ float As[16][68], Bs[16][68];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int i = threadIdx.x; i < 16 * 64; i += 256) {
            const int kk = i & 15, r = i >> 4;
            const int gk = k0 + kk, gm = m0 + r, gn = n0 + r;
            As[kk][r] = (gm < M && gk < K) ? to_f32(A[(int64_t)gm * sam + (int64_t)gk * sak]) : 0.f;
            Bs[kk][r] = (gn < N && gk < K) ? to_f32(Bm[(int64_t)gn * sbn + (int64_t)gk * sbk]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
            if (m < M && n < N) simt_epilogue<T>(epi, acc[i][j] * alpha, m, n, D, D2, R, ldd, bias);
        }
}

template <typename T>
int matmul_simt(const T *A, int64_t sam, int64_t sak, const T *Bm, int64_t sbn, int64_t sbk, void *D, T *D2,
                const T *R, int64_t ldd, const float *bias, int M, int N, int K, int epi, float alpha,
                cudaStream_t st) {
    if (M <= 0 || N <= 0 || K <= 0) return GPT2_ERR_BAD_SHAPE;
    matmul_simt_kernel<T><<<dim3(ceil_div(N, 64), ceil_div(M, 64)), 256, 0, st>>>(A, sam, sak, Bm, sbn, sbk, D, D2, R,
                                                                                 ldd, bias, M, N, K, epi, alpha);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// ============================================================== SIMT attention
// Causal, scale 1/sqrt(hd) ("Let's build GPT: from scratch", 01:16:56 and the
// errata after 01:54:32).  One thread per query row (forward, dQ) or key row
// (dK, dV); K/V (or Q/dO) tiles staged in shared memory.
template <typename T, int HD>
__global__ void attn_fwd_simt_kernel(const T *__restrict__ q, const T *__restrict__ kk, const T *__restrict__ v,
                                     int64_t rs, T *__restrict__ o, int64_t ors, float *__restrict__ lse, int Tn,
                                     int H) {
    constexpr int BQ = 64, BKV = 32;
    __shared__ float Ks[BKV][HD], Vs[BKV][HD];
    const int bh = blockIdx.y, b = bh / H, h = bh % H;
    const int i = blockIdx.x * BQ + threadIdx.x;
    const bool valid = i < Tn;
    const float scale = 1.0f / sqrtf((float)HD);
    float qr[HD], acc[HD];
#pragma unroll
    for (int d = 0; d < HD; ++d) {
        qr[d] = valid ? to_f32(q[((int64_t)b * Tn + i) * rs + h * HD + d]) * scale : 0.f;
        acc[d] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const int kv_end = min(Tn, blockIdx.x * BQ + BQ);
    for (int j0 = 0; j0 < kv_end; j0 += BKV) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < BKV * HD; idx += BQ) {
            const int jj = idx / HD, d = idx % HD, j = j0 + jj;
            const int64_t off = ((int64_t)b * Tn + j) * rs + h * HD + d;
            Ks[jj][d] = j < Tn ? to_f32(kk[off]) : 0.f;
            Vs[jj][d] = j < Tn ? to_f32(v[off]) : 0.f;
        }
        __syncthreads();
        if (valid) {
            for (int jj = 0; jj < BKV; ++jj) {
                const int j = j0 + jj;
                if (j > i) break;
                float s = 0.f;
#pragma unroll
                for (int d = 0; d < HD; ++d) s = fmaf(qr[d], Ks[jj][d], s);
                const float mn = fmaxf(m, s);
                const float corr = expf(m - mn), p = expf(s - mn);
                l = l * corr + p;
#pragma unroll
                for (int d = 0; d < HD; ++d) acc[d] = acc[d] * corr + p * Vs[jj][d];
                m = mn;
            }
        }
    }
    if (valid) {
        const float inv = 1.0f / l;
#pragma unroll
        for (int d = 0; d < HD; ++d) o[((int64_t)b * Tn + i) * ors + h * HD + d] = from_f32<T>(acc[d] * inv);
        lse[(int64_t)bh * Tn + i] = m + logf(l);
    }
}

template <typename T, int HD>
__global__ void attn_bwd_dq_simt_kernel(const T *__restrict__ q, const T *__restrict__ kk, const T *__restrict__ v,
                                        int64_t rs, const T *__restrict__ o, const T *__restrict__ dout, int64_t ors,
                                        const float *__restrict__ lse, T *__restrict__ dq, float *__restrict__ Dsc,
                                        int Tn, int H) {
    constexpr int BQ = 64, BKV = 32;
    __shared__ float Ks[BKV][HD], Vs[BKV][HD];
    const int bh = blockIdx.y, b = bh / H, h = bh % H;
    const int i = blockIdx.x * BQ + threadIdx.x;
    const bool valid = i < Tn;
    const float scale = 1.0f / sqrtf((float)HD);
    float qr[HD], dor[HD], acc[HD];
    float Di = 0.f;
    const int64_t qoff = ((int64_t)b * Tn + i) * rs + h * HD, ooff = ((int64_t)b * Tn + i) * ors + h * HD;
#pragma unroll
    for (int d = 0; d < HD; ++d) {
        qr[d] = valid ? to_f32(q[qoff + d]) : 0.f;
        dor[d] = valid ? to_f32(dout[ooff + d]) : 0.f;
        Di += valid ? dor[d] * to_f32(o[ooff + d]) : 0.f;
        acc[d] = 0.f;
    }
    const float li = valid ? lse[(int64_t)bh * Tn + i] : 0.f;
    if (valid) Dsc[(int64_t)bh * Tn + i] = Di;
    const int kv_end = min(Tn, blockIdx.x * BQ + BQ);
    for (int j0 = 0; j0 < kv_end; j0 += BKV) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < BKV * HD; idx += BQ) {
            const int jj = idx / HD, d = idx % HD, j = j0 + jj;
            const int64_t off = ((int64_t)b * Tn + j) * rs + h * HD + d;
            Ks[jj][d] = j < Tn ? to_f32(kk[off]) : 0.f;
            Vs[jj][d] = j < Tn ? to_f32(v[off]) : 0.f;
        }
        __syncthreads();
        if (valid) {
            for (int jj = 0; jj < BKV; ++jj) {
                const int j = j0 + jj;
                if (j > i) break;
                float s = 0.f, dp = 0.f;
#pragma unroll
                for (int d = 0; d < HD; ++d) {
                    s = fmaf(qr[d], Ks[jj][d], s);
                    dp = fmaf(dor[d], Vs[jj][d], dp);
                }
                const float p = expf(s * scale - li);
                const float ds = p * (dp - Di);
#pragma unroll
                for (int d = 0; d < HD; ++d) acc[d] = fmaf(ds, Ks[jj][d], acc[d]);
            }
        }
    }
    if (valid) {
#pragma unroll
        for (int d = 0; d < HD; ++d) dq[qoff + d] = from_f32<T>(acc[d] * scale);
    }
}

template <typename T, int HD>
__global__ void attn_bwd_dkv_simt_kernel(const T *__restrict__ q, const T *__restrict__ kk, const T *__restrict__ v,
                                         int64_t rs, const T *__restrict__ dout, int64_t ors,
                                         const float *__restrict__ lse, const float *__restrict__ Dsc,
                                         T *__restrict__ dk, T *__restrict__ dv, int Tn, int H) {
    constexpr int BKV = 64, BQ = 32;
    __shared__ float Qs[BQ][HD], Ds[BQ][HD];
    __shared__ float Ls[BQ], Dd[BQ];
    const int bh = blockIdx.y, b = bh / H, h = bh % H;
    const int j = blockIdx.x * BKV + threadIdx.x;
    const bool valid = j < Tn;
    const float scale = 1.0f / sqrtf((float)HD);
    float kr[HD], vr[HD], adk[HD], adv[HD];
    const int64_t koff = ((int64_t)b * Tn + j) * rs + h * HD;
#pragma unroll
    for (int d = 0; d < HD; ++d) {
        kr[d] = valid ? to_f32(kk[koff + d]) : 0.f;
        vr[d] = valid ? to_f32(v[koff + d]) : 0.f;
        adk[d] = 0.f;
        adv[d] = 0.f;
    }
    const int q_start = blockIdx.x * BKV;
    for (int i0 = q_start; i0 < Tn; i0 += BQ) {
        __syncthreads();
        for (int idx = threadIdx.x; idx < BQ * HD; idx += BKV) {
            const int ii = idx / HD, d = idx % HD, i = i0 + ii;
            Qs[ii][d] = i < Tn ? to_f32(q[((int64_t)b * Tn + i) * rs + h * HD + d]) : 0.f;
            Ds[ii][d] = i < Tn ? to_f32(dout[((int64_t)b * Tn + i) * ors + h * HD + d]) : 0.f;
        }
        for (int ii = threadIdx.x; ii < BQ; ii += BKV) {
            const int i = i0 + ii;
            Ls[ii] = i < Tn ? lse[(int64_t)bh * Tn + i] : 0.f;
            Dd[ii] = i < Tn ? Dsc[(int64_t)bh * Tn + i] : 0.f;
        }
        __syncthreads();
        if (valid) {
            for (int ii = 0; ii < BQ; ++ii) {
                const int i = i0 + ii;
                if (i < j || i >= Tn) continue;
                float s = 0.f, dp = 0.f;
#pragma unroll
                for (int d = 0; d < HD; ++d) {
                    s = fmaf(Qs[ii][d], kr[d], s);
                    dp = fmaf(Ds[ii][d], vr[d], dp);
                }
                const float p = expf(s * scale - Ls[ii]);
                const float ds = p * (dp - Dd[ii]);
#pragma unroll
                for (int d = 0; d < HD; ++d) {
                    adv[d] = fmaf(p, Ds[ii][d], adv[d]);
                    adk[d] = fmaf(ds, Qs[ii][d], adk[d]);
                }
            }
        }
    }
    if (valid) {
#pragma unroll
        for (int d = 0; d < HD; ++d) {
            dk[koff + d] = from_f32<T>(adk[d] * scale);
            dv[koff + d] = from_f32<T>(adv[d]);
        }
    }
}

#define ATTN_HD_DISPATCH(HDV, ...)                  \
    switch (HDV) {                                  \
        case 8: { constexpr int HD = 8; __VA_ARGS__; } break;   \
        case 16: { constexpr int HD = 16; __VA_ARGS__; } break; \
        case 32: { constexpr int HD = 32; __VA_ARGS__; } break; \
        case 64: { constexpr int HD = 64; __VA_ARGS__; } break; \
        default: return GPT2_ERR_BAD_SHAPE;         \
    }

template <typename T>
int attention_forward_simt(const T *q, const T *kk, const T *v, int64_t rs, T *o, int64_t ors, float *lse, int B,
                           int Tn, int H, int hd, cudaStream_t st) {
    const dim3 grid(ceil_div(Tn, 64), B * H);
    ATTN_HD_DISPATCH(hd, (attn_fwd_simt_kernel<T, HD><<<grid, 64, 0, st>>>(q, kk, v, rs, o, ors, lse, Tn, H)));
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

template <typename T>
int attention_backward_simt(const T *q, const T *kk, const T *v, int64_t rs, const T *o, const T *dout, int64_t ors,
                            const float *lse, T *dq, T *dk, T *dv, float *dscratch, int B, int Tn, int H, int hd,
                            cudaStream_t st) {
    const dim3 grid(ceil_div(Tn, 64), B * H);
    ATTN_HD_DISPATCH(hd, (attn_bwd_dq_simt_kernel<T, HD><<<grid, 64, 0, st>>>(q, kk, v, rs, o, dout, ors, lse, dq,
                                                                                dscratch, Tn, H)));
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    ATTN_HD_DISPATCH(hd, (attn_bwd_dkv_simt_kernel<T, HD><<<grid, 64, 0, st>>>(q, kk, v, rs, dout, ors, lse, dscratch,
                                                                                 dk, dv, Tn, H)));
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

// ============================================================== clip + AdamW
constexpr int ADAM_THREADS = 256;
constexpr int ADAM_BLOCKS_PER_SM = 4;

__device__ __forceinline__ double block_sum_d(double v, double *sh) {
    v = warp_sum_d(v);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) sh[wid] = v;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0) {
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += sh[w];
        sh[0] = t;
    }
    __syncthreads();
    t = sh[0];
    __syncthreads();
    return t;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Phase 1: sum of squares of every gradient (fp32 per thread, fp64 per block);
// grid barrier (cooperative launch, spin bounded by a.wait_ns: a block whose
// wait runs out sets DEVERR_TIMEOUT and returns without updating); every block
// then reduces the block partials in the same fixed order, so all blocks see
// one norm.
// Phase 2: clip coefficient and the AdamW update, bf16 copy of the new weights.
__global__ void __launch_bounds__(ADAM_THREADS) clip_adamw_kernel(float *__restrict__ p, const float *__restrict__ g,
                                                                  float *__restrict__ m, float *__restrict__ v,
                                                                  bf16 *__restrict__ shadow, int64_t n,
                                                                  int64_t n_decay, AdamArgs a,
                                                                  double *__restrict__ partials, unsigned *counter,
                                                                  float *norm_out, int *err) {
    __shared__ double sh[32];
    __shared__ int ok;
    const int64_t n4 = n >> 2;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    float s = 0.f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 x = __ldcs(reinterpret_cast<const float4 *>(g) + i);
        s += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
    }
    const double bs = block_sum_d((double)s, sh);
    if (threadIdx.x == 0) {
        partials[blockIdx.x] = bs;
        __threadfence();
        atomicAdd(counter, 1u);
        ok = 1;
        const uint64_t t0 = global_timer_ns();
        const unsigned target = gridDim.x + a.extra_arrivals;
        while (ld_acquire(counter) < target) {
            if (global_timer_ns() - t0 > a.wait_ns) {
                ok = 0;
                raise_device_error(err, DEVERR_TIMEOUT);
                break;
            }
            __nanosleep(100);
        }
        __threadfence();
    }
    __syncthreads();
    if (!ok) return;
    double t = 0.0;
    for (int i = threadIdx.x; i < (int)gridDim.x; i += blockDim.x) t += __ldcg(partials + i);
    const double total = block_sum_d(t, sh);
    const double norm = sqrt(total);
    if (blockIdx.x == 0 && threadIdx.x == 0) *norm_out = (float)norm;
    if (!isfinite(norm)) return;
    const float coef = (float)fmin(1.0, (double)a.clip / (norm + 1e-6));
    const float decay_mul = 1.0f - a.lr * a.wd;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 gv = __ldcs(reinterpret_cast<const float4 *>(g) + i);
        float4 pv = reinterpret_cast<float4 *>(p)[i];
        float4 mv = reinterpret_cast<float4 *>(m)[i];
        float4 vv = reinterpret_cast<float4 *>(v)[i];
        const bool decay = i * 4 < n_decay;
        float *pp = &pv.x, *mp = &mv.x, *vp = &vv.x;
        const float *gp = &gv.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float gi = gp[e] * coef;
            mp[e] = a.beta1 * mp[e] + (1.0f - a.beta1) * gi;
            vp[e] = a.beta2 * vp[e] + (1.0f - a.beta2) * gi * gi;
            const float mhat = mp[e] / a.bc1, vhat = vp[e] / a.bc2;
            float pi = pp[e];
            if (decay) pi *= decay_mul;
            pp[e] = pi - a.lr * mhat / (sqrtf(vhat) + a.eps);
        }
        reinterpret_cast<float4 *>(p)[i] = pv;
        reinterpret_cast<float4 *>(m)[i] = mv;
        reinterpret_cast<float4 *>(v)[i] = vv;
        if (shadow) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(pv.x, pv.y), hi = __floats2bfloat162_rn(pv.z, pv.w);
            uint2 u;
            u.x = *reinterpret_cast<uint32_t *>(&lo);
            u.y = *reinterpret_cast<uint32_t *>(&hi);
            reinterpret_cast<uint2 *>(shadow)[i] = u;
        }
    }
}

int clip_adamw_max_blocks(int num_sms) { return num_sms * ADAM_BLOCKS_PER_SM; }

int clip_adamw(float *p, const float *g, float *m, float *v, bf16 *shadow, int64_t n, int64_t n_decay,
               const AdamArgs &a, double *partials, unsigned *counter, int max_blocks, float *norm_out, int *err,
               int num_sms, cudaStream_t st) {
    if (n % 4 || n_decay % 4) return GPT2_ERR_BAD_SHAPE;
    int occ = 0;
    GPT2_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, clip_adamw_kernel, ADAM_THREADS, 0));
    int grid = std::min(max_blocks, num_sms * std::min(occ, ADAM_BLOCKS_PER_SM));
    grid = std::max(1, std::min(grid, ceil_div(n / 4, ADAM_THREADS)));
    GPT2_CUDA_TRY(cudaMemsetAsync(counter, 0, sizeof(unsigned), st));
    void *args[] = {&p, &g, &m, &v, &shadow, &n, &n_decay, const_cast<AdamArgs *>(&a), &partials, &counter,
                    &norm_out, &err};
    GPT2_CUDA_TRY(cudaLaunchCooperativeKernel((void *)clip_adamw_kernel, dim3(grid), dim3(ADAM_THREADS), args, 0, st));
    gpt2_note_launches(1);
    return GPT2_OK;
}

// ============================================================== instantiations
#define INST(T)                                                                                                  \
    template int embed_forward<T>(const int *, const float *, const float *, T *, int, int, int, int, int *,       \
                                  cudaStream_t);                                                                 \
    template int embed_backward<T>(const int *, const T *, float *, float *, int, int, int, int, cudaStream_t,     \
                                   void *);                                                                      \
    template int layernorm_forward<T>(const T *, const float *, const float *, T *, float *, float *, int, int,    \
                                      cudaStream_t, uint8_t *, float *);                                         \
    template int layernorm_backward<T>(const T *, const T *, const float *, const float *, const float *,          \
                                       const T *, T *, float *, float *, int, int, cudaStream_t, float *);         \
    template int column_sum<T>(const T *, int, int, float *, cudaStream_t);                                        \
    template int classifier<T>(T *, const int *, float *, int, int, int, float, int *, cudaStream_t);              \
    template int gelu_forward<T>(const T *, T *, int64_t, cudaStream_t);                                           \
    template int matmul_simt<T>(const T *, int64_t, int64_t, const T *, int64_t, int64_t, void *, T *, const T *,  \
                                int64_t, const float *, int, int, int, int, float, cudaStream_t);                  \
    template int attention_forward_simt<T>(const T *, const T *, const T *, int64_t, T *, int64_t, float *, int,    \
                                           int, int, int, cudaStream_t);                                         \
    template int attention_backward_simt<T>(const T *, const T *, const T *, int64_t, const T *, const T *,        \
                                            int64_t, const float *, T *, T *, T *, float *, int, int, int, int,    \
                                            cudaStream_t);
INST(float)
INST(bf16)
#undef INST

}  // namespace k
