// Causal flash attention forward and backward on the tcgen05 tensor cores
// (head dim 64).
//
// Forward: one CTA per (128-query block, b*h), heaviest blocks first; two CTAs
// per SM.
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

// 2^x with the hardware approximation (MUFU.EX2, flush-to-zero): the results
// feed bf16 operands and fp32 sums whose error budget is far above its ~2 ulp.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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
            const float c = ex2(m_acc - m_pend);
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
        // A failed (timed-out) wait clears `ok`; the loop still runs to the end
        // so that every thread reaches every named barrier (bar.sync has no timeout).
        for (int j = 0; j < nkv; ++j) {
            if (ok) ok = mbar_wait(&bar->s_full, j & 1, abort_flag, nullptr);
            tc_fence_after();
            const int kbase = j * BKV + half * 64;
            // keys of this thread's half that need a mask: causal diagonal block or past T
            const bool masked_block = (j == qb) || (kbase + 63 >= T);
            const int lim = min(T - 1 - kbase, (j == qb) ? r - half * 64 : 63);  // last visible column
            // pass 1: row max of the scaled, masked scores (two 32-column loads)
            float mx = -INFINITY;
            if (ok) {
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
            }
            mx *= sl2;
            float *rb = red + (j & 1) * 256;
            rb[half * 128 + r] = mx;
            pair_sync();
            mx = fmaxf(rb[r], rb[128 + r]);
            if (!ok) continue;
            const float m_new = fmaxf(m, mx);
            const float mu = (m_new == -INFINITY) ? 0.f : m_new;
            const float corr = ex2(m - mu);
            // O_{j-1} is complete once PV_{j-1} has finished reading P: fold it
            // before P is overwritten.
            if (j > 0 && !(ok = fold_o(j - 1))) continue;
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
                    float p0 = ex2(fmaf(f[i], sl2, -mu));
                    float p1 = ex2(fmaf(f[i + 1], sl2, -mu));
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

// ===================================================================== backward
// Two kernels, no atomics.  D = rowsum(dO * O) is written by the dQ kernel and
// read by the dK/dV kernel, so the dQ kernel runs first.

__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float (&f)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(r[i]);
}

// 16 bf16 values (8 words) of row r into a swizzled 128-row x 128-byte atom at 16-byte chunks cc, cc+1
__device__ __forceinline__ void store_row_chunks(uint8_t *atom, int r, int cc, const uint32_t (&w)[8]) {
    uint8_t *row = atom + r * 128;
    *reinterpret_cast<uint4 *>(row + ((cc ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4 *>(row + (((cc + 1) ^ (r & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// ---------------------------------------------------------------- dQ kernel
// One CTA per (128-query block, b*h); key blocks of 64.  TMEM: S [0,64),
// dP [64,128), dQ [128,192).  Softmax threads: two per query row, 32 keys each.
namespace dq {
constexpr int BQ = 128, BK = 64, SLOTS = 4;
constexpr int TQ = BQ * HD * 2;      // 16 KB
constexpr int TK = BK * HD * 2;      // 8 KB
constexpr int OFF_DO = TQ, OFF_RING = 2 * TQ, OFF_DS = OFF_RING + SLOTS * TK, OFF_RED = OFF_DS + TQ;
constexpr int OFF_BAR = OFF_RED + 2 * 128 * 4;
constexpr int SMEM = 1024 + OFF_BAR + 256;
struct Bars {
    uint64_t qd_full, sp_full, ds_full, ds_free, dq_done, drain;
    uint64_t full[SLOTS], empty[SLOTS];
};
}  // namespace dq

__global__ void __launch_bounds__(NT, 2)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                     const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                     const bf16 *__restrict__ o, const bf16 *__restrict__ dout, int64_t ors,
                     const float *__restrict__ lse, bf16 *__restrict__ dqo, int64_t rs, float *__restrict__ Dscr,
                     int T, int H, float sl2, float scale) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    dq::Bars *bar = reinterpret_cast<dq::Bars *>(sm + dq::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + dq::OFF_BAR + sizeof(dq::Bars));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int nqb = (T + dq::BQ - 1) / dq::BQ;
    const int qb = nqb - 1 - blockIdx.x;
    const int bh = blockIdx.y, b = bh / H, h = bh % H;
    const int nkv = min((T + dq::BK - 1) / dq::BK, (qb + 1) * (dq::BQ / dq::BK));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bar->qd_full, 1);
        mbar_init(&bar->sp_full, 1);
        mbar_init(&bar->ds_full, SOFTMAX_WARPS);
        mbar_init(&bar->ds_free, 1);
        mbar_init(&bar->dq_done, 1);
        mbar_init(&bar->drain, 1);
        for (int i = 0; i < dq::SLOTS; ++i) {
            mbar_init(&bar->full[i], 1);
            mbar_init(&bar->empty[i], 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tdP = tmem + 64, tdQ = tmem + 128;

    if (warp == 0) {
        if (lane == 0) {
            mbar_expect_tx(&bar->qd_full, 2 * dq::TQ);
            tma_load_3d(sm, &tq, &bar->qd_full, h * HD, qb * dq::BQ, b);
            tma_load_3d(sm + dq::OFF_DO, &tdo, &bar->qd_full, h * HD, qb * dq::BQ, b);
            uint32_t issued = 0, iph = 0;
            bool ok = true;
            for (int i = 0; i < 2 * nkv && ok; ++i) {
                const int sl = i % dq::SLOTS;
                const uint32_t ph = (i / dq::SLOTS) & 1;
                if (!(ok = mbar_wait(&bar->empty[sl], ph ^ 1, abort_flag, nullptr))) break;
                mbar_expect_tx(&bar->full[sl], dq::TK);
                tma_load_3d(sm + dq::OFF_RING + sl * dq::TK, (i & 1) ? &tv : &tk, &bar->full[sl], h * HD, (i >> 1) * dq::BK, b);
                issued |= 1u << sl;
                iph = (iph & ~(1u << sl)) | (ph << sl);
            }
            if (!ok) {
                mbar_drain(&bar->qd_full, 0);
                for (int sl = 0; sl < dq::SLOTS; ++sl)
                    if (issued & (1u << sl)) mbar_drain(&bar->full[sl], (iph >> sl) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_S = instr_desc(dq::BK, false, false);   // 128 x 64, K-major x K-major
            constexpr uint32_t ID_DQ = instr_desc(HD, false, true);   // 128 x 64, dS K-major, K MN-major
            const uint32_t aQ = smem_u32(sm), aDO = smem_u32(sm + dq::OFF_DO), aDS = smem_u32(sm + dq::OFF_DS);
            bool ok = mbar_wait(&bar->qd_full, 0, abort_flag, nullptr);
            auto issue_sp = [&](int j) -> bool {
                const int sk = (2 * j) % dq::SLOTS, sv = (2 * j + 1) % dq::SLOTS;
                if (!mbar_wait(&bar->full[sk], ((2 * j) / dq::SLOTS) & 1, abort_flag, nullptr)) return false;
                if (!mbar_wait(&bar->full[sv], ((2 * j + 1) / dq::SLOTS) & 1, abort_flag, nullptr)) return false;
                tc_fence_after();
                const uint32_t aK = smem_u32(sm + dq::OFF_RING + sk * dq::TK), aV = smem_u32(sm + dq::OFF_RING + sv * dq::TK);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    tc_mma(tS, smem_desc(aQ + kk * 32, 16, 1024), smem_desc(aK + kk * 32, 16, 1024), ID_S,
                           kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    tc_mma(tdP, smem_desc(aDO + kk * 32, 16, 1024), smem_desc(aV + kk * 32, 16, 1024), ID_S,
                           kk > 0 ? 1u : 0u);
                tc_commit(&bar->sp_full);
                return true;
            };
            if (ok) ok = issue_sp(0);
            for (int j = 0; j < nkv && ok; ++j) {
                if (!(ok = mbar_wait(&bar->ds_full, j & 1, abort_flag, nullptr))) break;
                if (j + 1 < nkv && !(ok = issue_sp(j + 1))) break;
                const int sk = (2 * j) % dq::SLOTS, sv = (2 * j + 1) % dq::SLOTS;
                const uint32_t aK = smem_u32(sm + dq::OFF_RING + sk * dq::TK);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < dq::BK / 16; ++kk)
                    tc_mma(tdQ, smem_desc(aDS + kk * 32, 16, 1024), smem_desc(aK + kk * 2048, 8192, 1024), ID_DQ,
                           (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&bar->empty[sk]);
                tc_commit(&bar->empty[sv]);
                tc_commit(&bar->ds_free);
            }
            tc_commit(&bar->dq_done);
            tc_commit(&bar->drain);
            mbar_drain(&bar->drain, 0);
        }
    } else {
        const int quad = warp & 3, half = (warp - 2) >> 2;
        const int r = quad * 32 + lane, q = qb * dq::BQ + r;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        float *red = reinterpret_cast<float *>(sm + dq::OFF_RED);
        // D = rowsum(dO * O): each thread sums 32 of the 64 columns, partners exchange
        float part = 0.f;
        if (q < T) {
            const int64_t off = ((int64_t)b * T + q) * ors + h * HD + half * 32;
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
                Pack16<bf16> a, gd;
                a.load(o + off + c);
                gd.load(dout + off + c);
#pragma unroll
                for (int e = 0; e < 8; ++e) part = fmaf(a.get(e), gd.get(e), part);
            }
        }
        red[half * 128 + r] = part;
        asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
        const float Dq = red[r] + red[128 + r];
        if (half == 0 && q < T) Dscr[(int64_t)bh * T + q] = Dq;
        const float l2 = q < T ? lse[(int64_t)bh * T + q] * LOG2E : 0.f;
        uint8_t *sDS = sm + dq::OFF_DS;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            if (!(ok = mbar_wait(&bar->sp_full, j & 1, abort_flag, nullptr))) break;
            tc_fence_after();
            uint32_t w[2][8];
            // visible keys of this thread's 32: columns c <= lim (key <= q and key < T; none if q >= T)
            const int lim = q < T ? min(q, T - 1) - (j * dq::BK + half * 32) : -1;
            const bool full = lim >= 31;
#pragma unroll
            for (int c0 = 0; c0 < 32; c0 += 16) {
                float sv[16], dp[16];
                tmem_ld16f(tS + lane_off + half * 32 + c0, sv);
                tmem_ld16f(tdP + lane_off + half * 32 + c0, dp);
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    float p0 = ex2(fmaf(sv[i], sl2, -l2));
                    float p1 = ex2(fmaf(sv[i + 1], sl2, -l2));
                    if (!full) {
                        p0 = c0 + i <= lim ? p0 : 0.f;
                        p1 = c0 + i + 1 <= lim ? p1 : 0.f;
                    }
                    w[c0 >> 4][i >> 1] = pack_bf16x2(p0 * (dp[i] - Dq), p1 * (dp[i + 1] - Dq));
                }
            }
            tc_fence_before();
            if (j > 0 && !(ok = mbar_wait(&bar->ds_free, (j - 1) & 1, abort_flag, nullptr))) break;
            store_row_chunks(sDS, r, half * 4, w[0]);
            store_row_chunks(sDS, r, half * 4 + 2, w[1]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->ds_full);
        }
        if (ok && mbar_wait(&bar->dq_done, 0, abort_flag, nullptr)) {
            tc_fence_after();
            float f[32];
            tmem_ld32f(tdQ + lane_off + half * 32, f);
            if (q < T) {
                bf16 *row = dqo + ((int64_t)b * T + q) * rs + h * HD + half * 32;
#pragma unroll
                for (int d = 0; d < 32; d += 8) {
                    uint4 u;
                    u.x = pack_bf16x2(f[d] * scale, f[d + 1] * scale);
                    u.y = pack_bf16x2(f[d + 2] * scale, f[d + 3] * scale);
                    u.z = pack_bf16x2(f[d + 4] * scale, f[d + 5] * scale);
                    u.w = pack_bf16x2(f[d + 6] * scale, f[d + 7] * scale);
                    *reinterpret_cast<uint4 *>(row + d) = u;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- dK/dV kernel
// One CTA per (128-key block, b*h); query blocks of 64 from the key block on.
// TMEM: S^T [0,64), dP^T [64,128), dV [128,192), dK [192,256).  Softmax
// threads: two per key row, 32 queries each.
namespace dkv {
constexpr int BKY = 128, BQ = 64, SLOTS = 4;
constexpr int TKY = BKY * HD * 2;  // 16 KB
constexpr int TQ = BQ * HD * 2;    // 8 KB
constexpr int OFF_V = TKY, OFF_RING = 2 * TKY, OFF_P = OFF_RING + SLOTS * TQ, OFF_DS = OFF_P + TKY;
constexpr int OFF_LD = OFF_DS + TKY;  // [2 buffers][lse 64 | D 64] floats
constexpr int OFF_BAR = OFF_LD + 2 * 128 * 4;
constexpr int SMEM = 1024 + OFF_BAR + 256;
struct Bars {
    uint64_t kv_full, st_full, pds_full, pds_free, dkv_done, drain;
    uint64_t full[SLOTS], empty[SLOTS];
};
}  // namespace dkv

__global__ void __launch_bounds__(NT, 2)
    bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                      const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                      const float *__restrict__ lse, const float *__restrict__ Dscr, bf16 *__restrict__ dko,
                      bf16 *__restrict__ dvo, int64_t rs, int T, int H, float sl2, float scale) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    dkv::Bars *bar = reinterpret_cast<dkv::Bars *>(sm + dkv::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + dkv::OFF_BAR + sizeof(dkv::Bars));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int kb = blockIdx.x;  // key block 0 sees every query block: launch first
    const int bh = blockIdx.y, b = bh / H, h = bh % H;
    const int q0blk = kb * (dkv::BKY / dkv::BQ);
    const int nit = (T + dkv::BQ - 1) / dkv::BQ - q0blk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bar->kv_full, 1);
        mbar_init(&bar->st_full, 1);
        mbar_init(&bar->pds_full, SOFTMAX_WARPS);
        mbar_init(&bar->pds_free, 1);
        mbar_init(&bar->dkv_done, 1);
        mbar_init(&bar->drain, 1);
        for (int i = 0; i < dkv::SLOTS; ++i) {
            mbar_init(&bar->full[i], 1);
            mbar_init(&bar->empty[i], 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tSt = tmem, tdPt = tmem + 64, tdV = tmem + 128, tdK = tmem + 192;

    if (warp == 0) {
        if (lane == 0) {
            mbar_expect_tx(&bar->kv_full, 2 * dkv::TKY);
            tma_load_3d(sm, &tk, &bar->kv_full, h * HD, kb * dkv::BKY, b);
            tma_load_3d(sm + dkv::OFF_V, &tv, &bar->kv_full, h * HD, kb * dkv::BKY, b);
            uint32_t issued = 0, iph = 0;
            bool ok = true;
            for (int i = 0; i < 2 * nit && ok; ++i) {
                const int sl = i % dkv::SLOTS;
                const uint32_t ph = (i / dkv::SLOTS) & 1;
                if (!(ok = mbar_wait(&bar->empty[sl], ph ^ 1, abort_flag, nullptr))) break;
                mbar_expect_tx(&bar->full[sl], dkv::TQ);
                tma_load_3d(sm + dkv::OFF_RING + sl * dkv::TQ, (i & 1) ? &tdo : &tq, &bar->full[sl], h * HD,
                            (q0blk + (i >> 1)) * dkv::BQ, b);
                issued |= 1u << sl;
                iph = (iph & ~(1u << sl)) | (ph << sl);
            }
            if (!ok) {
                mbar_drain(&bar->kv_full, 0);
                for (int sl = 0; sl < dkv::SLOTS; ++sl)
                    if (issued & (1u << sl)) mbar_drain(&bar->full[sl], (iph >> sl) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_ST = instr_desc(dkv::BQ, false, false);  // 128 x 64: K/V K-major x Q/dO K-major
            constexpr uint32_t ID_G = instr_desc(HD, false, true);    // 128 x 64: P^T/dS^T K-major x dO/Q MN-major
            const uint32_t aK = smem_u32(sm), aV = smem_u32(sm + dkv::OFF_V);
            const uint32_t aP = smem_u32(sm + dkv::OFF_P), aDS = smem_u32(sm + dkv::OFF_DS);
            bool ok = mbar_wait(&bar->kv_full, 0, abort_flag, nullptr);
            auto issue_st = [&](int it) -> bool {
                const int sq = (2 * it) % dkv::SLOTS, sd = (2 * it + 1) % dkv::SLOTS;
                if (!mbar_wait(&bar->full[sq], ((2 * it) / dkv::SLOTS) & 1, abort_flag, nullptr)) return false;
                if (!mbar_wait(&bar->full[sd], ((2 * it + 1) / dkv::SLOTS) & 1, abort_flag, nullptr)) return false;
                tc_fence_after();
                const uint32_t aQ = smem_u32(sm + dkv::OFF_RING + sq * dkv::TQ), aDO = smem_u32(sm + dkv::OFF_RING + sd * dkv::TQ);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    tc_mma(tSt, smem_desc(aK + kk * 32, 16, 1024), smem_desc(aQ + kk * 32, 16, 1024), ID_ST,
                           kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    tc_mma(tdPt, smem_desc(aV + kk * 32, 16, 1024), smem_desc(aDO + kk * 32, 16, 1024), ID_ST,
                           kk > 0 ? 1u : 0u);
                tc_commit(&bar->st_full);
                return true;
            };
            if (ok) ok = issue_st(0);
            for (int it = 0; it < nit && ok; ++it) {
                if (!(ok = mbar_wait(&bar->pds_full, it & 1, abort_flag, nullptr))) break;
                if (it + 1 < nit && !(ok = issue_st(it + 1))) break;
                const int sq = (2 * it) % dkv::SLOTS, sd = (2 * it + 1) % dkv::SLOTS;
                const uint32_t aQ = smem_u32(sm + dkv::OFF_RING + sq * dkv::TQ), aDO = smem_u32(sm + dkv::OFF_RING + sd * dkv::TQ);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < dkv::BQ / 16; ++kk)
                    tc_mma(tdV, smem_desc(aP + kk * 32, 16, 1024), smem_desc(aDO + kk * 2048, 8192, 1024), ID_G,
                           (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < dkv::BQ / 16; ++kk)
                    tc_mma(tdK, smem_desc(aDS + kk * 32, 16, 1024), smem_desc(aQ + kk * 2048, 8192, 1024), ID_G,
                           (it > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&bar->empty[sq]);
                tc_commit(&bar->empty[sd]);
                tc_commit(&bar->pds_free);
            }
            tc_commit(&bar->dkv_done);
            tc_commit(&bar->drain);
            mbar_drain(&bar->drain, 0);
        }
    } else {
        const int quad = warp & 3, half = (warp - 2) >> 2;
        const int r = quad * 32 + lane, key = kb * dkv::BKY + r;
        const int sidx = threadIdx.x - 64;  // 0..255 over the softmax warps
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        float *ld = reinterpret_cast<float *>(sm + dkv::OFF_LD);  // [buf][0..63 lse*log2e | 64..127 D]
        auto load_ld = [&](int it, int buf) {
            if (sidx < 128 && it < nit) {
                const int q = (q0blk + it) * dkv::BQ + (sidx & 63);
                float v = 0.f;
                if (q < T) v = sidx < 64 ? lse[(int64_t)bh * T + q] * LOG2E : Dscr[(int64_t)bh * T + q];
                ld[buf * 128 + sidx] = v;
            }
        };
        auto group_sync = [&]() { asm volatile("bar.sync 5, 256;" ::: "memory"); };
        load_ld(0, 0);
        uint8_t *sP = sm + dkv::OFF_P, *sDS = sm + dkv::OFF_DS;
        bool ok = true;
        // A failed (timed-out) wait clears `ok`; the loop still runs to the end
        // so that every thread reaches every group barrier (bar.sync has no timeout).
        for (int it = 0; it < nit; ++it) {
            group_sync();               // buffer it&1 is filled; buffer (it+1)&1 is no longer read
            load_ld(it + 1, (it + 1) & 1);
            const float *L = ld + (it & 1) * 128, *Dv = L + 64;
            if (ok) ok = mbar_wait(&bar->st_full, it & 1, abort_flag, nullptr);
            if (!ok) continue;
            tc_fence_after();
            uint32_t wp[2][8], wd[2][8];
            const int qbase = (q0blk + it) * dkv::BQ + half * 32;
            // visible queries of this thread's 32: lo <= c <= hi (q >= key, q < T; none if key >= T)
            const int lo = key - qbase, hi = key < T ? T - 1 - qbase : -1;
            const bool full = lo <= 0 && hi >= 31;
#pragma unroll
            for (int c0 = 0; c0 < 32; c0 += 16) {
                float st[16], dpt[16], lv[16], dv[16];
                tmem_ld16f(tSt + lane_off + half * 32 + c0, st);
                tmem_ld16f(tdPt + lane_off + half * 32 + c0, dpt);
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 a = *reinterpret_cast<const float4 *>(L + half * 32 + c0 + i);
                    const float4 d4 = *reinterpret_cast<const float4 *>(Dv + half * 32 + c0 + i);
                    lv[i] = a.x; lv[i + 1] = a.y; lv[i + 2] = a.z; lv[i + 3] = a.w;
                    dv[i] = d4.x; dv[i + 1] = d4.y; dv[i + 2] = d4.z; dv[i + 3] = d4.w;
                }
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    float p0 = ex2(fmaf(st[i], sl2, -lv[i]));
                    float p1 = ex2(fmaf(st[i + 1], sl2, -lv[i + 1]));
                    if (!full) {
                        const int c = c0 + i;
                        p0 = (c >= lo && c <= hi) ? p0 : 0.f;
                        p1 = (c + 1 >= lo && c + 1 <= hi) ? p1 : 0.f;
                    }
                    wp[c0 >> 4][i >> 1] = pack_bf16x2(p0, p1);
                    wd[c0 >> 4][i >> 1] = pack_bf16x2(p0 * (dpt[i] - dv[i]), p1 * (dpt[i + 1] - dv[i + 1]));
                }
            }
            tc_fence_before();
            if (it > 0 && !(ok = mbar_wait(&bar->pds_free, (it - 1) & 1, abort_flag, nullptr))) continue;
            store_row_chunks(sP, r, half * 4, wp[0]);
            store_row_chunks(sP, r, half * 4 + 2, wp[1]);
            store_row_chunks(sDS, r, half * 4, wd[0]);
            store_row_chunks(sDS, r, half * 4 + 2, wd[1]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->pds_full);
        }
        if (ok && mbar_wait(&bar->dkv_done, 0, abort_flag, nullptr)) {
            tc_fence_after();
            float fv[32], fk[32];
            tmem_ld32f(tdV + lane_off + half * 32, fv);
            tmem_ld32f(tdK + lane_off + half * 32, fk);
            if (key < T) {
                const int64_t off = ((int64_t)b * T + key) * rs + h * HD + half * 32;
#pragma unroll
                for (int d = 0; d < 32; d += 8) {
                    uint4 u, w;
                    u.x = pack_bf16x2(fv[d], fv[d + 1]);
                    u.y = pack_bf16x2(fv[d + 2], fv[d + 3]);
                    u.z = pack_bf16x2(fv[d + 4], fv[d + 5]);
                    u.w = pack_bf16x2(fv[d + 6], fv[d + 7]);
                    w.x = pack_bf16x2(fk[d] * scale, fk[d + 1] * scale);
                    w.y = pack_bf16x2(fk[d + 2] * scale, fk[d + 3] * scale);
                    w.z = pack_bf16x2(fk[d + 4] * scale, fk[d + 5] * scale);
                    w.w = pack_bf16x2(fk[d + 6] * scale, fk[d + 7] * scale);
                    *reinterpret_cast<uint4 *>(dvo + off + d) = u;
                    *reinterpret_cast<uint4 *>(dko + off + d) = w;
                }
            }
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
static int encode_qkv_map(CUtensorMap *tm, const bf16 *base, int64_t rs, int T, int B, int H, int box_rows = 128) {
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
    cuuint32_t box[3] = {HD, (cuuint32_t)box_rows, 1};
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

int attention_backward_tc(const bf16 *q, const bf16 *k, const bf16 *v, int64_t rs, const bf16 *o, const bf16 *dout,
                          int64_t ors, const float *lse, bf16 *dq_out, bf16 *dk_out, bf16 *dv_out, float *Dscr, int B,
                          int T, int H, cudaStream_t st) {
    using namespace fatc;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq_out) |
         reinterpret_cast<uintptr_t>(dk_out) | reinterpret_cast<uintptr_t>(dv_out)) & 15)
        return GPT2_ERR_BAD_ARG;
    CUtensorMap q128, do128, k64, v64, k128, v128, q64, do64;
    if (int rc = encode_qkv_map(&q128, q, rs, T, B, H, 128)) return rc;
    if (int rc = encode_qkv_map(&do128, dout, ors, T, B, H, 128)) return rc;
    if (int rc = encode_qkv_map(&k64, k, rs, T, B, H, 64)) return rc;
    if (int rc = encode_qkv_map(&v64, v, rs, T, B, H, 64)) return rc;
    if (int rc = encode_qkv_map(&k128, k, rs, T, B, H, 128)) return rc;
    if (int rc = encode_qkv_map(&v128, v, rs, T, B, H, 128)) return rc;
    if (int rc = encode_qkv_map(&q64, q, rs, T, B, H, 64)) return rc;
    if (int rc = encode_qkv_map(&do64, dout, ors, T, B, H, 64)) return rc;
    static bool init = false;
    if (!init) {
        GPT2_CUDA_TRY(cudaFuncSetAttribute(bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dq::SMEM));
        GPT2_CUDA_TRY(cudaFuncSetAttribute(bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv::SMEM));
        init = true;
    }
    const float scale = 1.0f / sqrtf((float)HD), sl2 = LOG2E * scale;
    bwd_dq_tc_kernel<<<dim3((T + dq::BQ - 1) / dq::BQ, B * H), NT, dq::SMEM, st>>>(
        q128, do128, k64, v64, o, dout, ors, lse, dq_out, rs, Dscr, T, H, sl2, scale);
    GPT2_CUDA_TRY(cudaGetLastError());
    bwd_dkv_tc_kernel<<<dim3((T + dkv::BKY - 1) / dkv::BKY, B * H), NT, dkv::SMEM, st>>>(
        k128, v128, q64, do64, lse, Dscr, dk_out, dv_out, rs, T, H, sl2, scale);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(2);
    return GPT2_OK;
}

}  // namespace fa
