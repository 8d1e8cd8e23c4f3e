// Causal flash attention forward on the tcgen05 tensor cores (head dim 64).
//
// One CTA per (128-query block, b*h), heaviest blocks first; two CTAs per SM.
//   warp 0     TMA: Q once, then K_j / V_j of each 128-key block through a
//              3-slot shared-memory ring (128-byte swizzle);
//   warp 1     one thread issues tcgen05.mma: S = Q K_j^T into TMEM
//              (128 x 128 fp32), then O_j = P_j V_j into TMEM (128 x 64 fp32);
//   warps 2-9  softmax: two threads per query row (= TMEM lane), each owning
//              64 of the block's 128 keys and 32 of the 64 output columns.
//              They read S with tcgen05.ld, mask, exchange the row max through
//              shared memory, compute P in the log2 domain and write it as
//              bf16 into shared memory in the MMA's swizzled K-major layout,
//              then fold O_j into a register accumulator with the running
//              rescale.  O = acc / l and lse are written at the end.
// The T x T matrix is never stored ("Let's reproduce GPT-2 (124M)", §Video
// özeti: flash attention); the mask lets a query see itself and the past
// ("Let's build GPT: from scratch", 00:57:00 erratum; scale 1/sqrt(head_size),
// 01:20:05 erratum).  Every mbarrier wait is bounded (see tc_gemm.cuh).
#include "flash_attn.cuh"
#include "tc_gemm.cuh"

namespace fatc {

using namespace tcg;

constexpr int BQ = 128, BKV = 128, HD = 64;
constexpr int TILE = 128 * HD * 2;   // 16 KB: 128 rows of 128 B
constexpr int SLOTS = 3;             // K/V ring slots (K_j, V_j alternate)
constexpr int P_OFF = TILE * (1 + SLOTS);
constexpr int RED_OFF = P_OFF + 2 * TILE;          // exchange buffers [3][2 halves][128 rows] floats:
constexpr int BAR_OFF = RED_OFF + 3 * 2 * 128 * 4; // two alternate for the row max, the third for the row sum
constexpr int SMEM = 1024 + BAR_OFF + 256;
constexpr int SOFTMAX_WARPS = 8;                   // two per TMEM lane quadrant, one per half of the keys
constexpr int NT = 64 + 32 * SOFTMAX_WARPS;
constexpr uint32_t TMEM_COLS = 256;  // S: columns [0,128), O: [128,192)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// tcgen05.ld of 32 lanes x 32 fp32 columns into float registers
__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float (&f)[32]) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

struct Bars {
    uint64_t q_full, s_full, p_full, o_full, o_free, drain;
    uint64_t full[SLOTS], empty[SLOTS];
};

__global__ void __launch_bounds__(NT, 2)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, bf16 *__restrict__ o, int64_t ors, float *__restrict__ lse,
                  int T, int H, float sl2) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *bar = reinterpret_cast<Bars *>(sm + BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + BAR_OFF + sizeof(Bars));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    uint8_t *sQ = sm, *sP = sm + P_OFF;

    const int nqb = (T + BQ - 1) / BQ;
    const int qb = nqb - 1 - blockIdx.x;  // heaviest query blocks first
    const int bh = blockIdx.y, b = bh / H, h = bh % H;
    const int nkv = qb + 1;               // causal: key blocks 0..qb
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bar->q_full, 1);
        mbar_init(&bar->s_full, 1);
        mbar_init(&bar->p_full, SOFTMAX_WARPS);
        mbar_init(&bar->o_full, 1);
        mbar_init(&bar->o_free, SOFTMAX_WARPS);
        mbar_init(&bar->drain, 1);
        for (int s = 0; s < SLOTS; ++s) {
            mbar_init(&bar->full[s], 1);
            mbar_init(&bar->empty[s], 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tO = tmem + 128;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            mbar_expect_tx(&bar->q_full, TILE);
            tma_load_3d(sQ, &tq, &bar->q_full, h * HD, qb * BQ, b);
            uint32_t issued = 0, issued_phase = 0;
            bool ok = true;
            for (int i = 0; i < 2 * nkv && ok; ++i) {
                const int s = i % SLOTS;
                const uint32_t ph = (i / SLOTS) & 1;
                if (!mbar_wait(&bar->empty[s], ph ^ 1, abort_flag, nullptr)) {
                    ok = false;
                    break;
                }
                mbar_expect_tx(&bar->full[s], TILE);
                uint8_t *dst = sm + TILE * (1 + s);
                const int j = i >> 1;
                if ((i & 1) == 0)
                    tma_load_3d(dst, &tk, &bar->full[s], h * HD, j * BKV, b);
                else
                    tma_load_3d(dst, &tv, &bar->full[s], h * HD, j * BKV, b);
                issued |= 1u << s;
                issued_phase = (issued_phase & ~(1u << s)) | (ph << s);
            }
            if (!ok) {
                mbar_drain(&bar->q_full, 0);
                for (int s = 0; s < SLOTS; ++s)
                    if (issued & (1u << s)) mbar_drain(&bar->full[s], (issued_phase >> s) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t IDESC_S = instr_desc(BKV, false, false);  // 128 x 128, K-major x K-major
            constexpr uint32_t IDESC_O = instr_desc(HD, false, true);    // 128 x 64, P K-major, V MN-major
            const uint32_t aQ = smem_u32(sQ), aP = smem_u32(sP);
            bool ok = mbar_wait(&bar->q_full, 0, abort_flag, nullptr);
            auto issue_s = [&](int j) -> bool {
                const int s = (2 * j) % SLOTS;
                if (!mbar_wait(&bar->full[s], ((2 * j) / SLOTS) & 1, abort_flag, nullptr)) return false;
                tc_fence_after();
                const uint32_t aK = smem_u32(sm + TILE * (1 + s));
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    tc_mma(tS, smem_desc(aQ + kk * 32, 16, 1024), smem_desc(aK + kk * 32, 16, 1024), IDESC_S,
                           kk > 0 ? 1u : 0u);
                tc_commit(&bar->empty[s]);
                tc_commit(&bar->s_full);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; j < nkv && ok; ++j) {
                // softmax has turned S_j into P_j (and is done reading S)
                if (!(ok = mbar_wait(&bar->p_full, j & 1, abort_flag, nullptr))) break;
                if (j + 1 < nkv && !(ok = issue_s(j + 1))) break;
                if (j > 0 && !(ok = mbar_wait(&bar->o_free, (j - 1) & 1, abort_flag, nullptr))) break;
                const int s = (2 * j + 1) % SLOTS;
                if (!(ok = mbar_wait(&bar->full[s], ((2 * j + 1) / SLOTS) & 1, abort_flag, nullptr))) break;
                tc_fence_after();
                const uint32_t aV = smem_u32(sm + TILE * (1 + s));
#pragma unroll
                for (int kk = 0; kk < BKV / 16; ++kk)
                    tc_mma(tO, smem_desc(aP + (kk >> 2) * TILE + (kk & 3) * 32, 16, 1024),
                           smem_desc(aV + kk * 2048, 8192, 1024), IDESC_O, kk > 0 ? 1u : 0u);
                tc_commit(&bar->empty[s]);
                tc_commit(&bar->o_full);
            }
            tc_commit(&bar->drain);
            mbar_drain(&bar->drain, 0);
        }
    } else {
        // ---------------- softmax (warps 2..9): two threads per query row ----------------
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;    // keys [64 half, 64 half + 64), O columns [32 half, 32 half + 32)
        const int r = quad * 32 + lane;      // row within the block = TMEM lane
        const int q = qb * BQ + r;           // query index
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        float *red = reinterpret_cast<float *>(sm + RED_OFF);  // [3 buffers][2 halves][128 rows]
        auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory"); };
        float acc[32];
#pragma unroll
        for (int d = 0; d < 32; ++d) acc[d] = 0.f;
        float m = -INFINITY, l = 0.f, m_acc = -INFINITY, m_pend = -INFINITY;
        bool ok = true;
        auto fold_o = [&](int j) -> bool {   // acc = acc * 2^(m_acc - m_pend) + O_j (this thread's 32 columns)
            if (!mbar_wait(&bar->o_full, j & 1, abort_flag, nullptr)) return false;
            tc_fence_after();
            const float c = exp2f(m_acc - m_pend);
            float f[32];
            tmem_ld32f(tO + lane_off + half * 32, f);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = fmaf(acc[i], c, f[i]);
            m_acc = m_pend;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->o_free);
            return true;
        };
        for (int j = 0; j < nkv; ++j) {
            if (!(ok = mbar_wait(&bar->s_full, j & 1, abort_flag, nullptr))) break;
            tc_fence_after();
            const int kbase = j * BKV + half * 64;
            // keys of this thread's half that need a mask: causal diagonal block or past T
            const bool masked_block = (j == qb) || (kbase + 63 >= T);
            const int lim = min(T - 1 - kbase, (j == qb) ? r - half * 64 : 63);  // last visible column
            // pass 1: row max of the scaled, masked scores (two 32-column loads)
            float mx = -INFINITY;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                float f[32];
                tmem_ld32f(tS + lane_off + half * 64 + c0, f);
                if (!masked_block) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, f[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, c0 + i <= lim ? f[i] : -INFINITY);
                }
            }
            mx *= sl2;
            float *rb = red + (j & 1) * 256;
            rb[half * 128 + r] = mx;
            pair_sync();
            mx = fmaxf(rb[r], rb[128 + r]);
            const float m_new = fmaxf(m, mx);
            const float mu = (m_new == -INFINITY) ? 0.f : m_new;
            const float corr = exp2f(m - mu);
            // O_{j-1} is complete once PV_{j-1} has finished reading P: fold it
            // before P is overwritten.
            if (j > 0 && !(ok = fold_o(j - 1))) break;
            // pass 2: P = 2^(s*sl2 - m_new) as bf16 into this half's 64-key atom of the P tile
            float ls = 0.f;
            uint8_t *atom = sP + half * TILE + r * 128;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) {
                float f[32];
                tmem_ld32f(tS + lane_off + half * 64 + c0, f);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float p0 = exp2f(fmaf(f[i], sl2, -mu));
                    float p1 = exp2f(fmaf(f[i + 1], sl2, -mu));
                    if (masked_block) {
                        p0 = c0 + i <= lim ? p0 : 0.f;
                        p1 = c0 + i + 1 <= lim ? p1 : 0.f;
                    }
                    ls += p0 + p1;
                    __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);
                    pk[i >> 1] = *reinterpret_cast<uint32_t *>(&v2);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int cc = (c0 >> 3) + k;
                    *reinterpret_cast<uint4 *>(atom + ((cc ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
            }
            l = l * corr + ls;
            m = m_new;
            tc_fence_before();
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->p_full);
            m_pend = m_new;
        }
        if (ok) ok = fold_o(nkv - 1);
        // the row sum is split over the two halves
        float *rs2 = red + 2 * 256;
        rs2[half * 128 + r] = l;
        pair_sync();
        const float lt = rs2[r] + rs2[128 + r];
        if (ok && q < T) {
            const float inv = 1.0f / lt;
            bf16 *orow = o + ((int64_t)b * T + q) * ors + h * HD + half * 32;
#pragma unroll
            for (int d = 0; d < 32; d += 8) {
                uint4 w;
                w.x = pack_bf16x2(acc[d] * inv, acc[d + 1] * inv);
                w.y = pack_bf16x2(acc[d + 2] * inv, acc[d + 3] * inv);
                w.z = pack_bf16x2(acc[d + 4] * inv, acc[d + 5] * inv);
                w.w = pack_bf16x2(acc[d + 6] * inv, acc[d + 7] * inv);
                *reinterpret_cast<uint4 *>(orow + d) = w;
            }
            if (half == 0) lse[(int64_t)bh * T + q] = (m + log2f(lt)) * LN2;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// 3-D map over one operand: (column within H*64, row t, batch b), row stride rs
static int encode_qkv_map(CUtensorMap *tm, const bf16 *base, int64_t rs, int T, int B, int H) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) !=
                cudaSuccess ||
            qr != cudaDriverEntryPointSuccess)
            return GPT2_ERR_CUDA;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    cuuint64_t dims[3] = {(cuuint64_t)H * HD, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)rs * 2, (cuuint64_t)T * rs * 2};
    cuuint32_t box[3] = {HD, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<bf16 *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // namespace fatc

namespace fa {

int attention_forward_tc(const bf16 *q, const bf16 *k, const bf16 *v, int64_t rs, bf16 *o, int64_t ors, float *lse,
                         int B, int T, int H, cudaStream_t st) {
    using namespace fatc;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(o)) & 15)
        return GPT2_ERR_BAD_ARG;
    CUtensorMap mq, mk, mv;
    if (int rc = encode_qkv_map(&mq, q, rs, T, B, H)) return rc;
    if (int rc = encode_qkv_map(&mk, k, rs, T, B, H)) return rc;
    if (int rc = encode_qkv_map(&mv, v, rs, T, B, H)) return rc;
    static bool init = false;
    if (!init) {
        GPT2_CUDA_TRY(cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM));
        init = true;
    }
    const float sl2 = LOG2E / sqrtf((float)HD);
    fwd_tc_kernel<<<dim3((T + BQ - 1) / BQ, B * H), NT, SMEM, st>>>(mq, mk, mv, o, ors, lse, T, H, sl2);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

}  // namespace fa
