// Flash-style causal attention backward (head dim 64) on mma.sync bf16 tensor
// cores; the forward runs on tcgen05 (attn_tc.cu).
//
// K/V and Q/dO 64-row tiles stream through double-buffered cp.async rings
// (XOR-swizzled shared memory read by ldmatrix); scores and the softmax
// recompute stay in registers.  Two kernels without atomics --
//   dQ kernel   (per query block): D = rowsum(dO*O), then for each key block
//               S, P = exp(S - lse), dP = dO V^T, dS = P (dP - D), dQ += dS K;
//   dK/dV kernel (per key block): for each query block S^T, P^T, dP^T,
//               dV += P^T dO, dK += dS^T Q.
// Query blocks run heaviest-first to balance the causal triangle.
#include <algorithm>

#include "flash_attn.cuh"

namespace fa {

constexpr int HD = 64;
constexpr int NT = 128;  // 4 warps
constexpr int TILE = 64 * HD * 2;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// byte offset of 16-byte chunk c of row r in a swizzled 64 x 64 bf16 tile
__device__ __forceinline__ uint32_t toff(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(pred ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// rows [row0, row0 + 64) of one head's [T, 64] slice; rows >= T read as zero
__device__ __forceinline__ void load_tile(uint32_t tile, const bf16 *base, int64_t rs, int row0, int T) {
#pragma unroll
    for (int i = threadIdx.x; i < 64 * 8; i += NT) {
        const int r = i >> 3, c = i & 7, row = row0 + r;
        const bool ok = row < T;
        cp_async16(tile + toff(r, c), base + (int64_t)(ok ? row : row0) * rs + c * 8, ok);
    }
}

__device__ __forceinline__ void ldsm4(uint32_t a, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
__device__ __forceinline__ void ldsm4t(uint32_t a, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pk(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// A operand: 16 rows from rbase, k-step kk (columns 16kk..16kk+15)
__device__ __forceinline__ void ld_a(uint32_t tile, int rbase, int kk, uint32_t (&a)[4]) {
    const int l = threadIdx.x & 31;
    ldsm4(tile + toff(rbase + (l & 15), 2 * kk + (l >> 4)), a);
}
// B operand of two n-tiles whose n index is the tile row (rows nb..nb+15), k contiguous
__device__ __forceinline__ void ld_b_rows(uint32_t tile, int nb, int kk, uint32_t (&b)[4]) {
    const int l = threadIdx.x & 31;
    ldsm4(tile + toff(nb + (l & 7) + ((l >> 4) << 3), 2 * kk + ((l >> 3) & 1)), b);
}
// B operand whose k index is the tile row (rows 16kk..), n the column (n-tiles 2np, 2np+1)
__device__ __forceinline__ void ld_b_cols(uint32_t tile, int kk, int np, uint32_t (&b)[4]) {
    const int l = threadIdx.x & 31;
    ldsm4t(tile + toff(16 * kk + (l & 7) + (((l >> 3) & 1) << 3), 2 * np + (l >> 4)), b);
}

// acc[16 x 64] += A (4 k-steps, registers) * B where B's rows are n (row operand)
__device__ __forceinline__ void mm_rows(float (&acc)[8][4], const uint32_t (&a)[4][4], uint32_t tile) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t b[4];
            ld_b_rows(tile, 16 * np, kk, b);
            mma(acc[2 * np], a[kk], b[0], b[1]);
            mma(acc[2 * np + 1], a[kk], b[2], b[3]);
        }
}
// acc[16 x 64] += P (16 x 64 in accumulator layout, packed per k-step) * tile (rows are k)
__device__ __forceinline__ void mm_cols(float (&acc)[8][4], const float (&p)[8][4], uint32_t tile) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint32_t a[4] = {pk(p[2 * kk][0], p[2 * kk][1]), pk(p[2 * kk][2], p[2 * kk][3]),
                               pk(p[2 * kk + 1][0], p[2 * kk + 1][1]), pk(p[2 * kk + 1][2], p[2 * kk + 1][3])};
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t b[4];
            ld_b_cols(tile, kk, np, b);
            mma(acc[2 * np], a, b[0], b[1]);
            mma(acc[2 * np + 1], a, b[2], b[3]);
        }
    }
}

__device__ __forceinline__ void zero(float (&a)[8][4]) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) a[i][e] = 0.f;
}

// ----------------------------------------------------------------- backward: dQ (+ D)
__global__ void __launch_bounds__(NT) bwd_dq_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ k,
                                                    const bf16 *__restrict__ v, int64_t rs,
                                                    const bf16 *__restrict__ o, const bf16 *__restrict__ dout,
                                                    int64_t ors, const float *__restrict__ lse,
                                                    bf16 *__restrict__ dq, float *__restrict__ Dscr, int T, int H,
                                                    float sl2, float scale) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ float sD[64];
    const int nqb = (T + 63) / 64;
    const int qb = nqb - 1 - blockIdx.x;
    const int bh = blockIdx.y, b = bh / H, h = bh % H;
    const int64_t hoff = (int64_t)b * T * rs + h * HD, ooff = (int64_t)b * T * ors + h * HD;
    const bf16 *qg = q + hoff, *kg = k + hoff, *vg = v + hoff, *dog = dout + ooff, *og = o + ooff;
    const uint32_t sQ = su32(sm), sdO = sQ + TILE, sK = sQ + 2 * TILE, sV = sQ + 4 * TILE;
    load_tile(sQ, qg, rs, qb * 64, T);
    load_tile(sdO, dog, ors, qb * 64, T);
    load_tile(sK, kg, rs, 0, T);
    load_tile(sV, vg, rs, 0, T);
    cp_commit();
    {  // D = rowsum(dO * O): two threads per row, 32 columns each
        const int r = threadIdx.x >> 1, half = threadIdx.x & 1, row = qb * 64 + r;
        float d = 0.f;
        if (row < T) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int col = half * 32 + c * 8;
                Pack16<bf16> a, g;
                a.load(og + (int64_t)row * ors + col);
                g.load(dog + (int64_t)row * ors + col);
#pragma unroll
                for (int e = 0; e < 8; ++e) d += a.get(e) * g.get(e);
            }
        }
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        if (half == 0) {
            sD[r] = d;
            if (row < T) Dscr[(int64_t)bh * T + row] = d;
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
    const int row0 = qb * 64 + warp * 16 + gid;
    float lr[2], Dr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = row0 + 8 * r;
        lr[r] = row < T ? lse[(int64_t)bh * T + row] * LOG2E : 0.f;
    }
    float dqacc[8][4], s[8][4], dp[8][4];
    zero(dqacc);
    uint32_t qf[4][4], df[4][4];
    for (int j = 0; j <= qb; ++j) {
        const int buf = j & 1;
        if (j < qb) {
            load_tile(sK + (buf ^ 1) * TILE, kg, rs, (j + 1) * 64, T);
            load_tile(sV + (buf ^ 1) * TILE, vg, rs, (j + 1) * 64, T);
        }
        cp_commit();
        cp_wait1();
        __syncthreads();
        if (j == 0) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                ld_a(sQ, warp * 16, kk, qf[kk]);
                ld_a(sdO, warp * 16, kk, df[kk]);
            }
            Dr[0] = sD[warp * 16 + gid];
            Dr[1] = sD[warp * 16 + gid + 8];
        }
        zero(s);
        zero(dp);
        mm_rows(s, qf, sK + buf * TILE);
        mm_rows(dp, df, sV + buf * TILE);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = j * 64 + nt * 8 + 2 * t4 + (e & 1), row = row0 + (e >> 1) * 8;
                const float p = (key > row || key >= T) ? 0.f : exp2f(s[nt][e] * sl2 - lr[e >> 1]);
                s[nt][e] = p * (dp[nt][e] - Dr[e >> 1]);
            }
        mm_cols(dqacc, s, sK + buf * TILE);
        __syncthreads();
    }
    bf16 *dqg = dq + hoff;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = row0 + 8 * r;
        if (row < T)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
                *reinterpret_cast<uint32_t *>(dqg + (int64_t)row * rs + nt * 8 + 2 * t4) =
                    pk(dqacc[nt][2 * r] * scale, dqacc[nt][2 * r + 1] * scale);
    }
}

// ----------------------------------------------------------------- backward: dK, dV
__global__ void __launch_bounds__(NT) bwd_dkv_kernel(const bf16 *__restrict__ q, const bf16 *__restrict__ k,
                                                     const bf16 *__restrict__ v, int64_t rs,
                                                     const bf16 *__restrict__ dout, int64_t ors,
                                                     const float *__restrict__ lse, const float *__restrict__ Dscr,
                                                     bf16 *__restrict__ dk, bf16 *__restrict__ dv, int T, int H,
                                                     float sl2, float scale) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ float sL[2][64], sDd[2][64];
    const int nqb = (T + 63) / 64;
    const int kb = blockIdx.x;  // key block 0 has the most query blocks: launch it first
    const int bh = blockIdx.y, b = bh / H, h = bh % H;
    const int64_t hoff = (int64_t)b * T * rs + h * HD, ooff = (int64_t)b * T * ors + h * HD;
    const bf16 *qg = q + hoff, *kg = k + hoff, *vg = v + hoff, *dog = dout + ooff;
    const uint32_t sK = su32(sm), sV = sK + TILE, sQ = sK + 2 * TILE, sdO = sK + 4 * TILE;
    load_tile(sK, kg, rs, kb * 64, T);
    load_tile(sV, vg, rs, kb * 64, T);
    load_tile(sQ, qg, rs, kb * 64, T);
    load_tile(sdO, dog, ors, kb * 64, T);
    cp_commit();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
    const int key0 = kb * 64 + warp * 16 + gid;
    float dkacc[8][4], dvacc[8][4], st[8][4], dpt[8][4];
    zero(dkacc);
    zero(dvacc);
    uint32_t kf[4][4], vf[4][4];
    for (int i = kb; i < nqb; ++i) {
        const int buf = (i - kb) & 1;
        if (i + 1 < nqb) {
            load_tile(sQ + (buf ^ 1) * TILE, qg, rs, (i + 1) * 64, T);
            load_tile(sdO + (buf ^ 1) * TILE, dog, ors, (i + 1) * 64, T);
        }
        cp_commit();
        if (threadIdx.x < 64) {
            const int row = i * 64 + threadIdx.x;
            sL[buf][threadIdx.x] = row < T ? lse[(int64_t)bh * T + row] * LOG2E : 0.f;
            sDd[buf][threadIdx.x] = row < T ? Dscr[(int64_t)bh * T + row] : 0.f;
        }
        cp_wait1();
        __syncthreads();
        if (i == kb) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                ld_a(sK, warp * 16, kk, kf[kk]);
                ld_a(sV, warp * 16, kk, vf[kk]);
            }
        }
        zero(st);
        zero(dpt);
        mm_rows(st, kf, sQ + buf * TILE);
        mm_rows(dpt, vf, sdO + buf * TILE);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int qc = nt * 8 + 2 * t4 + (e & 1), qi = i * 64 + qc, key = key0 + (e >> 1) * 8;
                const float p = (qi < key || qi >= T) ? 0.f : exp2f(st[nt][e] * sl2 - sL[buf][qc]);
                st[nt][e] = p;
                dpt[nt][e] = p * (dpt[nt][e] - sDd[buf][qc]);
            }
        mm_cols(dvacc, st, sdO + buf * TILE);
        mm_cols(dkacc, dpt, sQ + buf * TILE);
        __syncthreads();
    }
    bf16 *dkg = dk + hoff, *dvg = dv + hoff;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int key = key0 + 8 * r;
        if (key < T)
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int64_t off = (int64_t)key * rs + nt * 8 + 2 * t4;
                *reinterpret_cast<uint32_t *>(dkg + off) = pk(dkacc[nt][2 * r] * scale, dkacc[nt][2 * r + 1] * scale);
                *reinterpret_cast<uint32_t *>(dvg + off) = pk(dvacc[nt][2 * r], dvacc[nt][2 * r + 1]);
            }
    }
}

// ----------------------------------------------------------------- launchers
static int smem_opt_in(const void *fn, int bytes) {
    GPT2_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
    return GPT2_OK;
}

int attention_forward(const bf16 *q, const bf16 *k, const bf16 *v, int64_t rs, bf16 *o, int64_t ors, float *lse,
                      int B, int T, int H, int hd, cudaStream_t st) {
    if (hd != HD || rs % 8 || ors % 8) return GPT2_ERR_BAD_SHAPE;
    return attention_forward_tc(q, k, v, rs, o, ors, lse, B, T, H, st);
}

int attention_backward(const bf16 *q, const bf16 *k, const bf16 *v, int64_t rs, const bf16 *o, const bf16 *dout,
                       int64_t ors, const float *lse, bf16 *dq, bf16 *dk, bf16 *dv, float *Dscr, int B, int T, int H,
                       int hd, cudaStream_t st) {
    if (hd != HD || rs % 8 || ors % 8) return GPT2_ERR_BAD_SHAPE;
    static bool init = false;
    const int smem = 6 * TILE;
    if (!init) {
        if (int rc = smem_opt_in((const void *)bwd_dq_kernel, smem)) return rc;
        if (int rc = smem_opt_in((const void *)bwd_dkv_kernel, smem)) return rc;
        init = true;
    }
    const float scale = 1.0f / sqrtf((float)HD), sl2 = LOG2E * scale;
    const dim3 grid((T + 63) / 64, B * H);
    bwd_dq_kernel<<<grid, NT, smem, st>>>(q, k, v, rs, o, dout, ors, lse, dq, Dscr, T, H, sl2, scale);
    GPT2_CUDA_TRY(cudaGetLastError());
    bwd_dkv_kernel<<<grid, NT, smem, st>>>(q, k, v, rs, dout, ors, lse, Dscr, dk, dv, T, H, sl2, scale);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(2);
    return GPT2_OK;
}

}  // namespace fa
