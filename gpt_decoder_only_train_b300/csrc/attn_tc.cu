// Causal flash attention forward and backward on the tcgen05 tensor cores
// (head dim 64).
//
// The forward, dQ and dK/dV kernels are persistent (one CTA per SM over a
// heaviest-first list of work items) and keep their fixed operand (Q, or K
// and V) in TMEM as the A operand of tcgen05.mma; each kernel's layout is
// described above it.
// The T x T matrix is never stored ("Let's reproduce GPT-2 (124M)", §Video
// özeti: flash attention); the mask lets a query see itself and the past
// ("Let's build GPT: from scratch", 00:57:00 erratum; scale 1/sqrt(head_size),
// 01:20:05 erratum).  Every mbarrier wait is bounded (see tc_gemm.cuh).
#include "flash_attn.cuh"
#include "tc_gemm.cuh"

namespace fatc {

using namespace tcg;

constexpr int HD = 64;  // head dimension
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

// Column sums over a warp's 32 rows (one row per lane, 16 values each) added to g[0, 16)
// (shared memory).
// A butterfly that keeps half of the columns at each step (16 shuffles in all) leaves
// lanes 2c and 2c + 1 with the sum of column c; the even lane adds it.
__device__ __forceinline__ void warp_colsum16_add(const float (&v)[16], float *g, int lane) {
    float a[8], b[4], c[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = (b4 ? v[8 + i] : v[i]) + __shfl_xor_sync(~0u, b4 ? v[i] : v[8 + i], 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = (b3 ? a[4 + i] : a[i]) + __shfl_xor_sync(~0u, b3 ? a[i] : a[4 + i], 8);
#pragma unroll
    for (int i = 0; i < 2; ++i) c[i] = (b2 ? b[2 + i] : b[i]) + __shfl_xor_sync(~0u, b2 ? b[i] : b[2 + i], 4);
    float d = (b1 ? c[1] : c[0]) + __shfl_xor_sync(~0u, b1 ? c[0] : c[1], 2);
    d += __shfl_xor_sync(~0u, d, 1);
    if (!(lane & 1)) atomicAdd(g + (lane >> 1), d);
}

// max of three fp32 values in one instruction (sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 2^x with the hardware approximation (MUFU.EX2, flush-to-zero): the results
// feed bf16 operands and fp32 sums whose error budget is far above its ~2 ulp.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// tcgen05.mma with the A operand in TMEM (kind::f16, fp32 accumulate)
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// 32 lanes x 8 columns of 32-bit words from registers into TMEM
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 4-byte asynchronous global -> shared copy; src_bytes 0 stores a zero
__device__ __forceinline__ void cp_async4(float *dst, const float *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 : "memory");
}
// the mbarrier counts one arrival when this thread's earlier cp.async copies have landed
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// 16 bf16 of row r, elements [16 sub, 16 sub + 16), from a 128-byte-swizzled tile (chunk c of
// row r at chunk c ^ (r & 7)) as 8 packed words
__device__ __forceinline__ void tile_row16(const uint8_t *tile, int r, int sub, uint32_t (&w)[8]) {
    const uint8_t *row = tile + r * 128;
    const uint4 a = *reinterpret_cast<const uint4 *>(row + (((2 * sub) ^ (r & 7)) << 4));
    const uint4 c = *reinterpret_cast<const uint4 *>(row + (((2 * sub + 1) ^ (r & 7)) << 4));
    w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w, w[4] = c.x, w[5] = c.y, w[6] = c.z, w[7] = c.w;
}
// L2 policy that evicts these lines first: for data written or read once (the stored dS)
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// Box of the blocked dS^T layout (see encode_ds_map) at query block qb, key block kb
// (blocks of 64), head bh; the two inner coordinates are always 0.
__device__ __forceinline__ void tma_load_ds_hint(void *dst, const CUtensorMap *tm, uint64_t *bar, int qb, int kb,
                                                 int bh, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(qb), "r"(kb), "r"(bh), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_store_ds_hint(const CUtensorMap *tm, const void *src, int qb, int kb, int bh,
                                                  uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %2, %3, %4, %5}], [%1], %6;" ::"l"(
            reinterpret_cast<uint64_t>(tm)),
        "r"(smem_u32(src)), "r"(0), "r"(qb), "r"(kb), "r"(bh), "l"(pol)
        : "memory");
}
// Item j of this CTA in a persistent grid: every gridDim.x-th entry of a
// heaviest-first list, in alternating direction, or -1 past the end.
__device__ __forceinline__ int item_of(int j, int nitems) {
    const int G = gridDim.x, c = blockIdx.x;
    const long long p = (long long)j * G + ((j & 1) ? G - 1 - c : c);
    return p < nitems ? (int)p : -1;
}

namespace fwd {
constexpr int BQ = 128, BKV = 128, SLOTS = 6, SWARPS = 8;
constexpr int NTH = 64 + 32 * SWARPS;
constexpr int TILE = 128 * HD * 2;         // 16 KB: a Q, K or V tile
constexpr int OFF_Q = SLOTS * TILE;        // [2 item slots] staged Q tiles
constexpr int OFF_RED = OFF_Q + 2 * TILE;  // [2 parities][2 halves][128 rows] row maxima, then [2][128] row sums
constexpr int OFF_BAR = OFF_RED + 3 * 2 * 128 * 4;
constexpr int SMEM = 1024 + OFF_BAR + 512;
constexpr uint32_t TCOLS = 512;
constexpr uint32_t C_S = 0, C_O = 256, C_Q = 384;  // S[b] [128b, +128), O[b] [256+64b, +64), Q[s] [384+32s, +32)
struct Bars {
    uint64_t drain;
    uint64_t q_sfull[2], q_sempty[2], q_tfull[2];
    uint64_t s_full[2], p_full[2], o_done[2], o_free[2];  // o_done: per block parity; o_free: per item parity
    uint64_t xmax[4][2], xsum[4];  // exchanges between the two softmax warps of a TMEM lane quadrant
    uint64_t full[SLOTS], empty[SLOTS];
};
}  // namespace fwd

// Forward.  Persistent: one CTA per SM walks the (128-query block, b*h)
// items, heaviest first; an item runs over the key blocks of 128 up to the
// diagonal.
//   warp 0     TMA: Q of the next item into a staging slot, K_j / V_j through
//              a ring of SLOTS shared-memory tiles (128-byte swizzle);
//   warp 1     one thread issues tcgen05.mma: S_j = Q K_j^T (A = Q in TMEM)
//              two key blocks ahead into a double-buffered S, and
//              O += P_j V_j (A = P_j in TMEM) into the item's O accumulator
//              (two, alternating by item);
//   warps 2-9  softmax: two threads per query row (= TMEM lane), each owning
//              64 of a block's 128 keys and 32 of the 64 output columns.  They
//              read S with tcgen05.ld, mask, exchange the row max, and write
//              P = 2^(s - m) as bf16 over the first 32 of their own 64 S
//              columns.  The reference max m of a row moves only when a block
//              exceeds it by more than 2^8; the O accumulated so far is then
//              rescaled in TMEM before P_j is released.  O / l and lse are
//              written per item.
// The T x T matrix is never stored ("Let's reproduce GPT-2 (124M)", §Video
// özeti: flash attention); the mask lets a query see itself and the past
// ("Let's build GPT: from scratch", 00:57:00 erratum; scale 1/sqrt(head_size),
// 01:20:05 erratum).  Every mbarrier wait is bounded (see tc_gemm.cuh).
__global__ void __launch_bounds__(fwd::NTH, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, bf16 *__restrict__ o, int64_t ors, float *__restrict__ lse,
                  int T, int H, int nitems, float sl2) {
    constexpr int BQ = fwd::BQ, BKV = fwd::BKV, SLOTS = fwd::SLOTS, SWARPS = fwd::SWARPS, TILE = fwd::TILE;
    constexpr int OFF_Q = fwd::OFF_Q, OFF_RED = fwd::OFF_RED, OFF_BAR = fwd::OFF_BAR;
    constexpr uint32_t TCOLS = fwd::TCOLS, C_S = fwd::C_S, C_O = fwd::C_O, C_Q = fwd::C_Q;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align_smem_1024(smem_raw);
    fwd::Bars *bar = reinterpret_cast<fwd::Bars *>(sm + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_BAR + sizeof(fwd::Bars));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int nqb = (T + BQ - 1) / BQ, BH = nitems / nqb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto item_qb = [&](int p) { return nqb - 1 - p / BH; };  // heaviest query blocks first
    if (threadIdx.x == 0) {
        mbar_init(&bar->drain, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar->q_sfull[i], 1);
            mbar_init(&bar->q_sempty[i], SWARPS);
            mbar_init(&bar->q_tfull[i], SWARPS);
            mbar_init(&bar->s_full[i], 1);
            mbar_init(&bar->p_full[i], SWARPS);
            mbar_init(&bar->o_done[i], 1);
            mbar_init(&bar->o_free[i], SWARPS);
        }
        for (int qd = 0; qd < 4; ++qd) {
            mbar_init(&bar->xmax[qd][0], 2);
            mbar_init(&bar->xmax[qd][1], 2);
            mbar_init(&bar->xsum[qd], 2);
        }
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
        tmem_alloc(tmem_slot, TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // Q of item j goes to staging slot j & 1 one item ahead; key block g
            // (counted over all items) puts K in ring tile 2g and V in 2g+1 (mod SLOTS).
            bool ok = true;
            int t = 0, nq = 0;
            auto stage_q = [&](int j) -> bool {
                const int p = item_of(j, nitems);
                if (p < 0) return true;
                const int s = j & 1, bh = p % BH;
                if (!mbar_wait(&bar->q_sempty[s], ((j >> 1) & 1) ^ 1, abort_flag, nullptr)) return false;
                mbar_expect_tx(&bar->q_sfull[s], TILE);
                tma_load_3d(sm + OFF_Q + s * TILE, &tq, &bar->q_sfull[s], (bh % H) * HD, item_qb(p) * BQ, bh / H);
                nq = j + 1;
                return true;
            };
            ok = stage_q(0);
            for (int j = 0; ok; ++j) {
                const int p = item_of(j, nitems);
                if (p < 0) break;
                if (!(ok = stage_q(j + 1))) break;
                const int bh = p % BH, b = bh / H, h = bh % H, nkv = item_qb(p) + 1;
                for (int i = 0; i < 2 * nkv && ok; ++i, ++t) {
                    const int s = t % SLOTS;
                    if (!(ok = mbar_wait(&bar->empty[s], ((t / SLOTS) & 1) ^ 1, abort_flag, nullptr))) break;
                    mbar_expect_tx(&bar->full[s], TILE);
                    tma_load_3d(sm + s * TILE, (i & 1) ? &tv : &tk, &bar->full[s], h * HD, (i >> 1) * BKV, b);
                }
            }
            if (!ok) {  // let the copies already issued land before the CTA exits
                for (int i = t > SLOTS ? t - SLOTS : 0; i < t; ++i) mbar_drain(&bar->full[i % SLOTS], (i / SLOTS) & 1);
                for (int j = nq > 2 ? nq - 2 : 0; j < nq; ++j) mbar_drain(&bar->q_sfull[j & 1], (j >> 1) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // S runs two key blocks ahead of O = P V: after PV_g the next score
            // block g+2 reuses S buffer g & 1 (the in-order pipe has read P_g).
            constexpr uint32_t ID_S = instr_desc(BKV, false, false);  // 128 x 128, B = K K-major
            constexpr uint32_t ID_O = instr_desc(HD, false, true);    // 128 x 64, B = V MN-major
            const uint64_t ring_k = smem_desc(smem_u32(sm), 16, 1024);     // K-major view of ring tile 0
            const uint64_t ring_mn = smem_desc(smem_u32(sm), 8192, 1024);  // MN-major view of ring tile 0
            auto item_len = [&](int j, int &n) -> bool {
                const int p = item_of(j, nitems);
                if (p < 0) return false;
                n = item_qb(p) + 1;
                return true;
            };
            int sj = 0, sit = 0, sn = 0, gs = 0, gj = 0, git = 0, gn = 0, go = 0;
            bool s_on = item_len(0, sn), o_on = s_on;
            gn = sn;
            auto issue_s = [&]() -> bool {  // S_gs = Q K^T into S[gs & 1]
                if (sit == 0 && !mbar_wait(&bar->q_tfull[sj & 1], (sj >> 1) & 1, abort_flag, nullptr)) return false;
                const int tk_ = 2 * gs, s = tk_ % SLOTS;
                if (!mbar_wait(&bar->full[s], (tk_ / SLOTS) & 1, abort_flag, nullptr)) return false;
                tc_fence_after();
                const uint32_t tQ = tmem + C_Q + 32 * (sj & 1), ts = tmem + C_S + 128 * (gs & 1);
                const uint64_t bk = ring_k + (uint64_t)(s * (TILE >> 4));
                tc_mma_ts(ts, tQ, bk, ID_S, 0u);
#pragma unroll
                for (int kk = 1; kk < HD / 16; ++kk) tc_mma_ts(ts, tQ + 8 * kk, bk + 2 * kk, ID_S, 1u);
                tc_commit(&bar->empty[s]);
                tc_commit(&bar->s_full[gs & 1]);
                ++gs;
                if (++sit == sn) sit = 0, s_on = item_len(++sj, sn);
                return true;
            };
            auto issue_o = [&]() -> bool {  // O[item] (+)= P_go V: the item's O accumulates in TMEM
                const int b2 = go & 1, tv_ = 2 * go + 1, s = tv_ % SLOTS, ob = gj & 1;
                if (!mbar_wait(&bar->p_full[b2], (go >> 1) & 1, abort_flag, nullptr)) return false;
                // the item two back used this O buffer: its read-out must be done
                if (git == 0 && gj >= 2 && !mbar_wait(&bar->o_free[ob], ((gj - 2) >> 1) & 1, abort_flag, nullptr))
                    return false;
                if (!mbar_wait(&bar->full[s], (tv_ / SLOTS) & 1, abort_flag, nullptr)) return false;
                tc_fence_after();
                const uint32_t pa = tmem + C_S + 128 * b2, to = tmem + C_O + 64 * ob;
                const uint64_t bv = ring_mn + (uint64_t)(s * (TILE >> 4));
                // K-step kk (keys 16kk..16kk+15): P columns 64 (kk / 4) + 8 (kk % 4)
                tc_mma_ts(to, pa, bv, ID_O, git > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 1; kk < BKV / 16; ++kk)
                    tc_mma_ts(to, pa + 64 * (kk >> 2) + 8 * (kk & 3), bv + 128 * kk, ID_O, 1u);
                tc_commit(&bar->empty[s]);
                tc_commit(&bar->o_done[b2]);
                ++go;
                if (++git == gn) git = 0, o_on = item_len(++gj, gn);
                return true;
            };
            bool ok = true;
            for (int i = 0; i < 2 && ok && s_on; ++i) ok = issue_s();
            while (ok && o_on) {
                if ((ok = issue_o()) && s_on) ok = issue_s();
            }
            tc_commit(&bar->drain);
            mbar_drain(&bar->drain, 0);
        }
    } else {
        const int quad = warp & 3, half = (warp - 2) >> 2;  // keys [64 half, +64), O columns [32 half, +32)
        const int r = quad * 32 + lane;                      // row within the block = TMEM lane
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        float *red = reinterpret_cast<float *>(sm + OFF_RED);
        // exchange a per-row value with the other warp of this quadrant (mbarrier, bounded)
        auto exchange = [&](float *buf, uint64_t *xb, uint32_t parity, float v, bool &ok) -> float {
            buf[half * 128 + r] = v;
            __syncwarp();
            if (lane == 0) mbar_arrive(xb);
            if (ok) ok = mbar_wait(xb, parity, abort_flag, nullptr);
            return buf[(half ^ 1) * 128 + r];
        };
        // Q rows of item j (this thread's 32 of the 64 head dims) into TMEM slot j & 1
        auto stage_in = [&](int j) -> bool {
            const int s = j & 1;
            if (!mbar_wait(&bar->q_sfull[s], (j >> 1) & 1, abort_flag, nullptr)) return false;
            const uint8_t *tile = sm + OFF_Q + s * TILE;
            uint32_t w0[8], w1[8];
            tile_row16(tile, r, 2 * half, w0);
            tile_row16(tile, r, 2 * half + 1, w1);
            tmem_st8(tmem + lane_off + C_Q + 32 * s + 16 * half, w0);
            tmem_st8(tmem + lane_off + C_Q + 32 * s + 16 * half + 8, w1);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar->q_tfull[s]);
                mbar_arrive(&bar->q_sempty[s]);
            }
            return true;
        };
        bool ok = stage_in(0);
        int g = 0;
        const F2 sl2x2 = f2(sl2, sl2);
        for (int j = 0; ok; ++j) {
            const int p = item_of(j, nitems);
            if (p < 0) break;
            const int qb = item_qb(p), bh = p % BH, b = bh / H, h = bh % H, nkv = qb + 1;
            const int q = qb * BQ + r;
            const int ob = j & 1;
            const uint32_t to = tmem + lane_off + C_O + 64 * ob + 32 * half;  // this thread's 32 O columns
            // m: the row's reference maximum (log2 units) of P and of the O accumulated so far.  It
            // moves only when a block's maximum exceeds it by more than RESCALE (always in the first
            // block): P then stays below 2^RESCALE and the accumulated O is rescaled once.
            constexpr float RESCALE = 8.0f;
            float m = -INFINITY, l = 0.f;
            // block gp's O product has completed (waits are taken in block order: at most one
            // completion of each barrier is pending, so its parity identifies it)
            auto o_done_wait = [&](int gp) -> bool {
                return mbar_wait(&bar->o_done[gp & 1], (gp >> 1) & 1, abort_flag, nullptr);
            };
            for (int jj = 0; jj < nkv; ++jj, ++g) {
                const int bb = g & 1;
                if (ok) ok = mbar_wait(&bar->s_full[bb], (g >> 1) & 1, abort_flag, nullptr);
                tc_fence_after();
                const uint32_t ts = tmem + lane_off + C_S + 128 * bb + 64 * half;
                const int kbase = jj * BKV + half * 64;
                // blocks below the diagonal and inside T need no mask (same for the whole CTA)
                const bool block_full = jj < qb && (jj + 1) * BKV <= T;
                const int lim = min(T - 1 - kbase, jj == qb ? r - half * 64 : 63);  // last visible column
                // the thread's 64 scores, read from TMEM once (both loads in flight, one wait)
                uint32_t sr[2][32];
                tmem_ld32(ts, sr[0]);
                tmem_ld32(ts + 32, sr[1]);
                tmem_ld_wait();
                // pass 1: row max of the masked scores (three-input max, four independent chains)
                float mx = -INFINITY;
                if (ok) {
                    float mc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        if (block_full) {
#pragma unroll
                            for (int i = 0; i < 32; i += 2)
                                mc[(i >> 1) & 3] = fmax3(mc[(i >> 1) & 3], __uint_as_float(sr[h2][i]),
                                                         __uint_as_float(sr[h2][i + 1]));
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                const int c = 32 * h2 + i;
                                mc[(i >> 1) & 3] = fmax3(mc[(i >> 1) & 3], c <= lim ? __uint_as_float(sr[h2][i]) : -INFINITY,
                                                         c + 1 <= lim ? __uint_as_float(sr[h2][i + 1]) : -INFINITY);
                            }
                        }
                    }
                    mx = fmax3(fmax3(mc[0], mc[1], mc[2]), mc[3], -INFINITY);
                }
                mx *= sl2;
                mx = fmaxf(mx, exchange(red + bb * 256, &bar->xmax[quad][bb], (g >> 1) & 1, mx, ok));
                if (!ok) break;
                const bool move = mx > m + RESCALE;
                const float m_new = move ? mx : m;
                if (jj > 0 && __any_sync(0xffffffffu, move)) {
                    // O holds blocks < jj: once the last of them has landed, scale this thread's columns
                    if (!(ok = o_done_wait(g - 1))) break;
                    tc_fence_after();
                    const float c = move ? ex2(m - m_new) : 1.0f;
                    const F2 c2 = f2(c, c);
                    uint32_t ov[32];
                    tmem_ld32(to, ov);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const F2 v = f2_mul(f2(__uint_as_float(ov[i]), __uint_as_float(ov[i + 1])), c2);
                        ov[i] = __float_as_uint(f2_lo(v));
                        ov[i + 1] = __float_as_uint(f2_hi(v));
                    }
#pragma unroll
                    for (int c8 = 0; c8 < 32; c8 += 8) {
                        uint32_t w8[8];
#pragma unroll
                        for (int k2 = 0; k2 < 8; ++k2) w8[k2] = ov[c8 + k2];
                        tmem_st8(to + c8, w8);
                    }
                    l *= c;
                }
                m = m_new;
                const float mu = (m == -INFINITY) ? 0.f : m;
                const F2 nmu = f2(-mu, -mu);
                // pass 2: P = 2^(s sl2 - m) as bf16 over the first 32 of this thread's 64 S columns
                F2 ls2 = f2(0.f, 0.f);
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    const uint32_t *f = sr[c0 >> 5];
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 32; i += 2) {
                        const F2 t = f2_fma(f2(__uint_as_float(f[i]), __uint_as_float(f[i + 1])), sl2x2, nmu);
                        float p0 = ex2(f2_lo(t)), p1 = ex2(f2_hi(t));
                        if (!block_full) {
                            p0 = c0 + i <= lim ? p0 : 0.f;
                            p1 = c0 + i + 1 <= lim ? p1 : 0.f;
                        }
                        ls2 = f2_add(ls2, f2(p0, p1));
                        pk[i >> 1] = pack_bf16x2(p0, p1);
                    }
                    uint32_t w0[8], w1[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) w0[k] = pk[k], w1[k] = pk[8 + k];
                    tmem_st8(ts + c0 / 2, w0);
                    tmem_st8(ts + c0 / 2 + 8, w1);
                }
                l += f2_lo(ls2) + f2_hi(ls2);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->p_full[bb]);
                if (jj > 0 && !(ok = o_done_wait(g - 1))) break;  // retire block g - 1 (normally long done)
                if (jj == 0 && item_of(j + 1, nitems) >= 0 && !(ok = stage_in(j + 1))) break;
            }
            if (!ok) break;
            // the item's O: once its last block has landed, read it and release the buffer
            if (!(ok = o_done_wait(g - 1))) break;
            tc_fence_after();
            float acc[32];
            tmem_ld32f(to, acc);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->o_free[ob]);
            // the row sum is split over the two halves
            const float lt = l + exchange(red + 2 * 256, &bar->xsum[quad], j & 1, l, ok);
            if (!ok) break;
            if (q < T) {
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
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TCOLS);
    }
}

// ===================================================================== backward
// Two kernels, no atomics.  D = rowsum(dO * O) is written by the dQ kernel and
// read by the dK/dV kernel, so the dQ kernel runs first.

// tcgen05.ld of 32 lanes x 16 columns without the wait (batch several loads,
// then one tmem_ld_wait)
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// ---------------------------------------------------------------- dQ kernel
// Persistent: one CTA per SM walks the (128-query block, b*h) items, heaviest
// first; an item iterates over the key blocks of 64 up to the diagonal.
//   S  = Q K^T      A = Q (TMEM)     B = K (K-major tile)
//   dP = dO V^T     A = dO (TMEM)    B = V (K-major tile)
//   dQ += dS K      A = dS (TMEM)    B = K (MN-major view)
// S / dP are double-buffered; the softmax warps write dS as bf16 over the
// first 8 of their 16 dP columns (K-step kk of the dQ product reads columns
// [16 kk, 16 kk + 8)).  Q, dO and O of the next item are staged by TMA while
// the current item runs; D = rowsum(dO * O) is computed from the staged tiles
// (every thread sums its own row in full) and written for the dK/dV kernel.
// TMEM columns: S[b] [64b, +64), dP[b] [128+64b, +64), dQ [256,320),
// Q[s] [320+64s, +32), dO[s] [352+64s, +32).
namespace dq {
constexpr int BQ = 128, BK = 64, NST = 6, SWARPS = 16;
constexpr int NTH = 64 + 32 * SWARPS;
constexpr int TQ = BQ * HD * 2;   // 16 KB: a Q, dO or O tile
constexpr int TK = BK * HD * 2;   // 8 KB: a K or V tile
constexpr int OFF_ITEM = NST * 2 * TK;      // [2 item slots][Q | dO | O]
constexpr int OFF_LSE = OFF_ITEM + 6 * TQ;  // [2][128] floats
constexpr int MAXC = 2048;                   // query- and value-bias partial sums of the CTA, [2][H * 64] floats
constexpr int OFF_BSUM = OFF_LSE + 2 * BQ * 4;
constexpr int OFF_BAR = OFF_BSUM + 2 * MAXC * 4;
constexpr int SMEM = 1024 + OFF_BAR + 512;
constexpr uint32_t TCOLS = 512;
constexpr uint32_t C_S = 0, C_DP = 128, C_DQ = 256, C_QD = 320;
struct Bars {
    uint64_t dq_done, dq_free, drain;
    uint64_t it_sfull[2], it_lfull[2], it_sempty[2], it_tfull[2];
    uint64_t sp_full[2], ds_full[2];
    uint64_t full[NST], empty[NST];  // per ring entry: K and V tiles of one key block
};
}  // namespace dq

__global__ void __launch_bounds__(dq::NTH, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                     const __grid_constant__ CUtensorMap to, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tv, const float *__restrict__ lse,
                     bf16 *__restrict__ dqo, int64_t rs, float *__restrict__ Dscr, int T, int H, int nitems,
                     float sl2, float scale, float *__restrict__ dbq, float *__restrict__ dbv) {
    constexpr int BQ = dq::BQ, BK = dq::BK, NST = dq::NST, SWARPS = dq::SWARPS;
    constexpr int TQ = dq::TQ, TK = dq::TK, OFF_ITEM = dq::OFF_ITEM, OFF_LSE = dq::OFF_LSE, OFF_BAR = dq::OFF_BAR;
    constexpr uint32_t TCOLS = dq::TCOLS, C_S = dq::C_S, C_DP = dq::C_DP, C_DQ = dq::C_DQ, C_QD = dq::C_QD;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align_smem_1024(smem_raw);
    dq::Bars *bar = reinterpret_cast<dq::Bars *>(sm + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_BAR + sizeof(dq::Bars));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *lsebuf = reinterpret_cast<float *>(sm + OFF_LSE);
    float *bsum = reinterpret_cast<float *>(sm + dq::OFF_BSUM), *bsum_v = bsum + dq::MAXC;
    if (dbq)
        for (int c = threadIdx.x; c < H * HD; c += blockDim.x) bsum[c] = bsum_v[c] = 0.f;
    const int nqb = (T + BQ - 1) / BQ, nkb = (T + BK - 1) / BK, BH = nitems / nqb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // item p: query block nqb - 1 - p / BH (heaviest first), b*h = p % BH
    auto item_qb = [&](int p) { return nqb - 1 - p / BH; };
    auto item_nkv = [&](int qb) { return min(nkb, (qb + 1) * (BQ / BK)); };
    if (threadIdx.x == 0) {
        mbar_init(&bar->dq_done, 1);
        mbar_init(&bar->dq_free, SWARPS);
        mbar_init(&bar->drain, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar->it_sfull[i], 1);
            mbar_init(&bar->it_lfull[i], 32);
            mbar_init(&bar->it_sempty[i], SWARPS);
            mbar_init(&bar->it_tfull[i], SWARPS);
            mbar_init(&bar->sp_full[i], 1);
            mbar_init(&bar->ds_full[i], SWARPS);
        }
        for (int i = 0; i < NST; ++i) {
            mbar_init(&bar->full[i], 1);
            mbar_init(&bar->empty[i], 1);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tdo);
        tma_prefetch_desc(&to);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // Q / dO / O / lse of item j go to staging slot j & 1 one item ahead; key
        // block g (counted over all items) uses ring entry g mod NST (K and V
        // tiles), refilled once the dQ product of the block that last used it
        // has completed.
        bool ok = true;
        int g = 0, nring = 0, nstage = 0;
        auto stage_item = [&](int j) -> bool {
            const int p = item_of(j, nitems);
            if (p < 0) return true;
            const int s = j & 1, qb = item_qb(p), bh = p % BH, b = bh / H, h = bh % H;
            if (!mbar_wait(&bar->it_sempty[s], ((j >> 1) & 1) ^ 1, abort_flag, nullptr)) return false;
            uint8_t *dst = sm + OFF_ITEM + s * 3 * TQ;
            if (lane == 0) {
                mbar_expect_tx(&bar->it_sfull[s], 3 * TQ);
                tma_load_3d(dst, &tq, &bar->it_sfull[s], h * HD, qb * BQ, b);
                tma_load_3d(dst + TQ, &tdo, &bar->it_sfull[s], h * HD, qb * BQ, b);
                tma_load_3d(dst + 2 * TQ, &to, &bar->it_sfull[s], h * HD, qb * BQ, b);
            }
            const float *src = lse + (int64_t)bh * T;
            float *ld = lsebuf + s * BQ + lane * 4;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int q = qb * BQ + lane * 4 + jj;
                cp_async4(ld + jj, src + (q < T ? q : 0), q < T ? 4u : 0u);
            }
            cp_async_arrive_noinc(&bar->it_lfull[s]);
            nstage = j + 1;
            return true;
        };
        ok = stage_item(0);
        for (int j = 0; ok; ++j) {
            const int p = item_of(j, nitems);
            if (p < 0) break;
            if (!(ok = stage_item(j + 1))) break;
            const int qb = item_qb(p), bh = p % BH, b = bh / H, h = bh % H, nkv = item_nkv(qb);
            for (int i = 0; i < nkv; ++i, ++g) {
                const int e = g % NST;
                if (!(ok = mbar_wait(&bar->empty[e], ((g / NST) & 1) ^ 1, abort_flag, nullptr))) break;
                if (lane == 0) {
                    mbar_expect_tx(&bar->full[e], 2 * TK);
                    tma_load_3d(sm + 2 * e * TK, &tk, &bar->full[e], h * HD, i * BK, b);
                    tma_load_3d(sm + (2 * e + 1) * TK, &tv, &bar->full[e], h * HD, i * BK, b);
                }
                nring = g + 1;
            }
        }
        if (!ok && lane == 0) {  // let the copies already issued land before the CTA exits
            for (int i = nring > NST ? nring - NST : 0; i < nring; ++i) mbar_drain(&bar->full[i % NST], (i / NST) & 1);
            for (int j = nstage > 2 ? nstage - 2 : 0; j < nstage; ++j) mbar_drain(&bar->it_sfull[j & 1], (j >> 1) & 1);
        }
        cp_async_wait_all();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_S = instr_desc(BK, false, false);  // 128 x 64, B = K / V K-major
            constexpr uint32_t ID_DQ = instr_desc(HD, false, true);  // 128 x 64, B = K MN-major
            const uint64_t ring_k = smem_desc(smem_u32(sm), 16, 1024);     // K-major view of ring slot 0
            const uint64_t ring_mn = smem_desc(smem_u32(sm), 8192, 1024);  // MN-major view of ring slot 0
            bool ok = true;
            // dQ product of key block gp, the it-th block of item j
            auto dq_mma = [&](int gp, int j, int it, bool last) -> bool {
                const int pb = gp & 1, pe = gp % NST;
                if (!mbar_wait(&bar->ds_full[pb], (gp >> 1) & 1, abort_flag, nullptr)) return false;
                if (it == 0 && j > 0 && !mbar_wait(&bar->dq_free, (j - 1) & 1, abort_flag, nullptr)) return false;
                tc_fence_after();
                const uint64_t bk = ring_mn + (uint64_t)(2 * pe * (TK >> 4));
                const uint32_t da = tmem + C_DP + pb * 64;
                tc_mma_ts(tmem + C_DQ, da, bk, ID_DQ, it > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 1; kk < BK / 16; ++kk) tc_mma_ts(tmem + C_DQ, da + 16 * kk, bk + 128 * kk, ID_DQ, 1u);
                tc_commit(&bar->empty[pe]);
                if (last) tc_commit(&bar->dq_done);
                return true;
            };
            int g = 0, pj = 0, pit = 0;
            bool plast = false;
            for (int j = 0; ok; ++j) {
                const int p = item_of(j, nitems);
                if (p < 0) break;
                const int nkv = item_nkv(item_qb(p));
                if (!(ok = mbar_wait(&bar->it_tfull[j & 1], (j >> 1) & 1, abort_flag, nullptr))) break;
                const uint32_t tQ = tmem + C_QD + 64 * (j & 1), tDO = tQ + 32;
                for (int it = 0; it < nkv; ++it, ++g) {
                    const int bb = g & 1, e = g % NST;
                    if (!(ok = mbar_wait(&bar->full[e], (g / NST) & 1, abort_flag, nullptr))) break;
                    tc_fence_after();
                    const uint64_t bk = ring_k + (uint64_t)(2 * e * (TK >> 4));
                    const uint64_t bv = ring_k + (uint64_t)((2 * e + 1) * (TK >> 4));
                    const uint32_t ts = tmem + C_S + bb * 64, tp = tmem + C_DP + bb * 64;
                    tc_mma_ts(ts, tQ, bk, ID_S, 0u);
#pragma unroll
                    for (int kk = 1; kk < HD / 16; ++kk) tc_mma_ts(ts, tQ + 8 * kk, bk + 2 * kk, ID_S, 1u);
                    tc_mma_ts(tp, tDO, bv, ID_S, 0u);
#pragma unroll
                    for (int kk = 1; kk < HD / 16; ++kk) tc_mma_ts(tp, tDO + 8 * kk, bv + 2 * kk, ID_S, 1u);
                    tc_commit(&bar->sp_full[bb]);
                    if (g > 0 && !(ok = dq_mma(g - 1, pj, pit, plast))) break;
                    pj = j, pit = it, plast = it == nkv - 1;
                }
            }
            if (ok && g > 0) dq_mma(g - 1, pj, pit, plast);
            tc_commit(&bar->drain);
            mbar_drain(&bar->drain, 0);
        }
    } else {
        const int quad = warp & 3, sub = (warp - 2) >> 2;  // sub: keys [16 sub, 16 sub + 16) of each block
        const int r = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        // Q / dO rows of item j (elements [16 sub, +16)) into TMEM slot j & 1,
        // plus lse * log2(e) and D = rowsum(dO * O) of row r
        auto stage_in = [&](int j, float &l2, float &Dr) -> bool {
            const int s = j & 1, p = item_of(j, nitems);
            if (!mbar_wait(&bar->it_sfull[s], (j >> 1) & 1, abort_flag, nullptr)) return false;
            if (!mbar_wait(&bar->it_lfull[s], (j >> 1) & 1, abort_flag, nullptr)) return false;
            const uint8_t *tile = sm + OFF_ITEM + s * 3 * TQ;
            uint32_t wq[8], wd[8];
            tile_row16(tile, r, sub, wq);
            tile_row16(tile + TQ, r, sub, wd);
            tmem_st8(tmem + lane_off + C_QD + 64 * s + sub * 8, wq);
            tmem_st8(tmem + lane_off + C_QD + 64 * s + 32 + sub * 8, wd);
            float acc = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {  // the whole row: 64 elements of dO and O
                uint32_t a[8], o8[8];
                tile_row16(tile + TQ, r, c, a);
                tile_row16(tile + 2 * TQ, r, c, o8);
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    acc = fmaf(bf16_lo(a[w]), bf16_lo(o8[w]), acc);
                    acc = fmaf(bf16_hi(a[w]), bf16_hi(o8[w]), acc);
                }
            }
            Dr = acc;
            l2 = lsebuf[s * BQ + r] * LOG2E;
            const int q = item_qb(p) * BQ + r;
            if (dbq) {  // value-bias gradient: column sums of dO (every row of P sums to one)
                float cv[16];
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    cv[2 * w] = q < T ? bf16_lo(wd[w]) : 0.f;
                    cv[2 * w + 1] = q < T ? bf16_hi(wd[w]) : 0.f;
                }
                warp_colsum16_add(cv, bsum_v + ((p % BH) % H) * HD + sub * 16, lane);
            }
            if (sub == 0 && q < T) Dscr[(int64_t)(p % BH) * T + q] = acc;
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar->it_tfull[s]);
                mbar_arrive(&bar->it_sempty[s]);
            }
            return true;
        };
        float l2 = 0.f, Dr = 0.f, l2n = 0.f, Drn = 0.f;
        bool ok = stage_in(0, l2, Dr);
        int g = 0;
        for (int j = 0; ok; ++j) {
            const int p = item_of(j, nitems);
            if (p < 0) break;
            const int qb = item_qb(p), bh = p % BH, b = bh / H, h = bh % H, nkv = item_nkv(qb);
            const int q = qb * BQ + r;
            const F2 sl2x2 = f2(sl2, sl2), nl2 = f2(-l2, -l2), dd = f2(Dr, Dr);
            for (int it = 0; it < nkv; ++it, ++g) {
                const int bb = g & 1;
                if (!(ok = mbar_wait(&bar->sp_full[bb], (g >> 1) & 1, abort_flag, nullptr))) break;
                tc_fence_after();
                const uint32_t cs = tmem + lane_off + C_S + bb * 64 + sub * 16;
                const uint32_t cp = tmem + lane_off + C_DP + bb * 64 + sub * 16;
                uint32_t ra[16], rb[16];
                tmem_ld16_nowait(cs, ra);
                tmem_ld16_nowait(cp, rb);
                tmem_ld_wait();
                const int k0 = it * BK, kbase = k0 + sub * 16;
                // Blocks wholly below the diagonal with every query below T need no
                // mask (same answer for the whole CTA); otherwise the visible keys of
                // this thread's 16 are columns c <= lim (key <= q, key < T; none if q >= T).
                const bool block_full = k0 + BK - 1 <= qb * BQ && qb * BQ + BQ <= T;
                const int lim = q < T ? min(q, T - 1) - kbase : -1;
                uint32_t wd[8];
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    const F2 t = f2_fma(f2(__uint_as_float(ra[c]), __uint_as_float(ra[c + 1])), sl2x2, nl2);
                    float p0 = ex2(f2_lo(t)), p1 = ex2(f2_hi(t));
                    if (!block_full) {
                        p0 = c <= lim ? p0 : 0.f;
                        p1 = c + 1 <= lim ? p1 : 0.f;
                    }
                    const F2 ds =
                        f2_mul(f2(p0, p1), f2_sub(f2(__uint_as_float(rb[c]), __uint_as_float(rb[c + 1])), dd));
                    wd[c >> 1] = pack_bf16x2(f2_lo(ds), f2_hi(ds));
                }
                tmem_st8(cp, wd);  // dS over the first 8 of this thread's dP columns
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->ds_full[bb]);
                if (it == 0 && item_of(j + 1, nitems) >= 0 && !(ok = stage_in(j + 1, l2n, Drn))) break;
            }
            if (!ok) break;
            l2 = l2n, Dr = Drn;
            // dQ of the item: read out of TMEM, release the accumulator, store
            if (!(ok = mbar_wait(&bar->dq_done, j & 1, abort_flag, nullptr))) break;
            tc_fence_after();
            uint32_t ra[16];
            tmem_ld16_nowait(tmem + lane_off + C_DQ + sub * 16, ra);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->dq_free);
            if (dbq) {  // query-bias gradient: column sums of dQ (one warp = 32 rows) into the CTA's partials
                float cv[16];
#pragma unroll
                for (int d = 0; d < 16; ++d) cv[d] = q < T ? __uint_as_float(ra[d]) * scale : 0.f;
                warp_colsum16_add(cv, bsum + h * HD + sub * 16, lane);
            }
            if (q < T) {
                bf16 *row = dqo + ((int64_t)b * T + q) * rs + h * HD + sub * 16;
#pragma unroll
                for (int d = 0; d < 16; d += 8) {
                    uint4 u;
                    u.x = pack_bf16x2(__uint_as_float(ra[d]) * scale, __uint_as_float(ra[d + 1]) * scale);
                    u.y = pack_bf16x2(__uint_as_float(ra[d + 2]) * scale, __uint_as_float(ra[d + 3]) * scale);
                    u.z = pack_bf16x2(__uint_as_float(ra[d + 4]) * scale, __uint_as_float(ra[d + 5]) * scale);
                    u.w = pack_bf16x2(__uint_as_float(ra[d + 6]) * scale, __uint_as_float(ra[d + 7]) * scale);
                    *reinterpret_cast<uint4 *>(row + d) = u;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TCOLS);
    }
    if (dbq)  // one atomic per head column and CTA
        for (int c = threadIdx.x; c < H * HD; c += blockDim.x) {
            if (bsum[c] != 0.f) atomicAdd(dbq + c, bsum[c]);
            if (bsum_v[c] != 0.f) atomicAdd(dbv + c, bsum_v[c]);
        }
}

// ---------------------------------------------------------------- dK/dV kernel
// Persistent: one CTA per SM walks a list of work items (128-key block, b*h),
// heaviest first, each CTA taking every gridDim.x-th item in alternating
// direction.  An item iterates over the query blocks of 64 from its key
// block on.  Every GEMM takes its A operand from TMEM, so shared memory only
// carries K / V (staging), the Q / dO tiles (B operands) and lse / D:
//   S^T  = K Q^T      A = K (TMEM)      B = Q  (K-major tile)
//   dP^T = V dO^T     A = V (TMEM)      B = dO (K-major tile)
//   dV  += P^T dO     A = P^T (TMEM)    B = dO (MN-major view)
//   dK  += dS^T Q     A = dS^T (TMEM)   B = Q  (MN-major view)
// S^T / dP^T are double-buffered.  The softmax warps read their 16 columns of
// S^T and dP^T and write P^T / dS^T as bf16 back over the first 8 of those
// columns, so that K-step kk of the dV / dK products reads columns
// [16 kk, 16 kk + 8) of the buffer.  tcgen05.mma operations issued by one
// thread execute in order, so S^T of block g+2 (issued after the dV / dK
// products of block g) never overwrites P^T / dS^T before they are read.
// K / V of the next item are staged (TMA) and copied into the second TMEM
// slot while the current item runs, and the dV / dK read-out of an item
// overlaps the first score products of the next one.
// TMEM columns: S^T[b] [64b, 64b+64), dP^T[b] [128+64b, ...), dV [256,320),
// dK [320,384), K[s] [384+64s, +32), V[s] [416+64s, +32) (bf16 pairs).
// Warps: 0 loads (TMA, cp.async), 1 issues the MMAs, 2-17 are the softmax
// warps: four per TMEM lane quadrant, each owning 16 of a block's 64 queries.
// With store_ds (the backward with the dS workspace), the softmax warps also
// write their dS^T values into the block's 128 x 64 staging tile (two tiles,
// by block parity) and fence them for the async proxy; once pds_full has
// completed, the MMA thread stores the tile with one TMA store (L2 evict-first)
// into the 64 x 64-blocked dS^T layout, and waits for the store of block g - 2
// to have read its tile before it lets block g's S^T be consumed.
namespace dkv {
constexpr int BKY = 128, BQ = 64, SLOTS = 12, SWARPS = 16, NLD = SLOTS / 2;
constexpr int NTH = 64 + 32 * SWARPS;
constexpr int TQ = BQ * HD * 2;    // 8 KB
constexpr int TKV = BKY * HD * 2;  // 16 KB: a K or V tile
constexpr int OFF_KV = SLOTS * TQ;  // [2 item slots][K | V]
constexpr int OFF_LD = OFF_KV + 4 * TKV;  // [NLD][lse 64 | D 64] floats
constexpr int TDS = BKY * BQ * 2;         // 16 KB: dS^T of one block, staged for its TMA store
constexpr int OFF_DS = OFF_LD + NLD * 2 * BQ * 4;  // [2 block parities]
constexpr int OFF_BAR = OFF_DS + 2 * TDS;
constexpr int SMEM = 1024 + OFF_BAR + 512;
constexpr uint32_t TCOLS = 512;
constexpr uint32_t C_ST = 0, C_DPT = 128, C_DV = 256, C_DK = 320, C_KV = 384;
static_assert(OFF_DS % 1024 == 0, "swizzled staging blocks start on 1024-byte boundaries");
struct Bars {
    uint64_t dkv_done, dkv_free, drain;
    uint64_t kv_sfull[2], kv_sempty[2], kv_tfull[2];
    uint64_t st_full[2], pds_full[2];
    uint64_t full[NLD], empty[NLD], ld_full[NLD];  // per ring entry: Q and dO slots + lse / D
};
}  // namespace dkv


__global__ void __launch_bounds__(dkv::NTH, 1)
    bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                      const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                      const __grid_constant__ CUtensorMap tds, const float *__restrict__ lse,
                      const float *__restrict__ Dscr, bf16 *__restrict__ dko, bf16 *__restrict__ dvo, int64_t rs,
                      int T, int H, int nitems, float sl2, float scale, int store_ds) {
    constexpr int BKY = dkv::BKY, BQ = dkv::BQ, SWARPS = dkv::SWARPS, NLD = dkv::NLD;
    constexpr int TQ = dkv::TQ, TKV = dkv::TKV, OFF_KV = dkv::OFF_KV, OFF_LD = dkv::OFF_LD, OFF_BAR = dkv::OFF_BAR;
    constexpr uint32_t TCOLS = dkv::TCOLS, C_ST = dkv::C_ST, C_DPT = dkv::C_DPT, C_DV = dkv::C_DV, C_DK = dkv::C_DK,
                       C_KV = dkv::C_KV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align_smem_1024(smem_raw);
    dkv::Bars *bar = reinterpret_cast<dkv::Bars *>(sm + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_BAR + sizeof(dkv::Bars));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *ldbuf = reinterpret_cast<float *>(sm + OFF_LD);
    const int nqb = (T + BQ - 1) / BQ, BH = nitems / ((T + BKY - 1) / BKY);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bar->dkv_done, 1);
        mbar_init(&bar->dkv_free, SWARPS);
        mbar_init(&bar->drain, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar->kv_sfull[i], 1);
            mbar_init(&bar->kv_sempty[i], SWARPS);
            mbar_init(&bar->kv_tfull[i], SWARPS);
            mbar_init(&bar->st_full[i], 1);
            mbar_init(&bar->pds_full[i], SWARPS);
        }
        for (int i = 0; i < NLD; ++i) {
            mbar_init(&bar->full[i], 1);
            mbar_init(&bar->empty[i], 1);
            mbar_init(&bar->ld_full[i], 32);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tdo);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // K / V of item j go to staging slot j & 1 one item ahead; query block g
        // (counted over all items) uses ring entry g mod NLD: shared-memory
        // slots 2e (Q) and 2e+1 (dO) and lse / D entry e, refilled once the
        // dV / dK products of the block that last used it have completed.
        bool ok = true;
        int g = 0, nring = 0, nkv = 0;
        auto load_kv = [&](int j) -> bool {
            const int p = item_of(j, nitems);
            if (p < 0) return true;
            const int s = j & 1, kb = p / BH, bh = p % BH;
            if (!mbar_wait(&bar->kv_sempty[s], ((j >> 1) & 1) ^ 1, abort_flag, nullptr)) return false;
            if (lane == 0) {
                mbar_expect_tx(&bar->kv_sfull[s], 2 * TKV);
                tma_load_3d(sm + OFF_KV + s * 2 * TKV, &tk, &bar->kv_sfull[s], (bh % H) * HD, kb * BKY, bh / H);
                tma_load_3d(sm + OFF_KV + s * 2 * TKV + TKV, &tv, &bar->kv_sfull[s], (bh % H) * HD, kb * BKY, bh / H);
            }
            nkv = j + 1;
            return true;
        };
        ok = load_kv(0);
        for (int j = 0; ok; ++j) {
            const int p = item_of(j, nitems);
            if (p < 0) break;
            if (!(ok = load_kv(j + 1))) break;
            const int kb = p / BH, bh = p % BH, b = bh / H, h = bh % H, nit = nqb - 2 * kb;
            for (int i = 0; i < nit; ++i, ++g) {
                const int e = g % NLD;
                const uint32_t ph = (g / NLD) & 1;
                if (!(ok = mbar_wait(&bar->empty[e], ph ^ 1, abort_flag, nullptr))) break;
                const int q0 = (2 * kb + i) * BQ;
                if (lane == 0) {
                    mbar_expect_tx(&bar->full[e], 2 * TQ);
                    tma_load_3d(sm + 2 * e * TQ, &tq, &bar->full[e], h * HD, q0, b);
                    tma_load_3d(sm + (2 * e + 1) * TQ, &tdo, &bar->full[e], h * HD, q0, b);
                }
                // lanes 0-15: lse of queries q0 + 4 lane + jj; lanes 16-31: D
                const float *src = (lane < 16 ? lse : Dscr) + (int64_t)bh * T;
                float *dst = ldbuf + e * 128 + lane * 4;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int q = q0 + (lane & 15) * 4 + jj;
                    cp_async4(dst + jj, src + (q < T ? q : 0), q < T ? 4u : 0u);
                }
                cp_async_arrive_noinc(&bar->ld_full[e]);
                nring = g + 1;
            }
        }
        if (!ok && lane == 0) {  // let the copies already issued land before the CTA exits
            for (int i = nring > NLD ? nring - NLD : 0; i < nring; ++i) mbar_drain(&bar->full[i % NLD], (i / NLD) & 1);
            for (int j = nkv > 2 ? nkv - 2 : 0; j < nkv; ++j) mbar_drain(&bar->kv_sfull[j & 1], (j >> 1) & 1);
        }
        cp_async_wait_all();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t ID_ST = instr_desc(BQ, false, false);  // 128 x 64, B = Q / dO K-major
            constexpr uint32_t ID_G = instr_desc(HD, false, true);    // 128 x 64, B = dO / Q MN-major
            const uint64_t ring_k = smem_desc(smem_u32(sm), 16, 1024);     // K-major view of slot 0
            const uint64_t ring_mn = smem_desc(smem_u32(sm), 8192, 1024);  // MN-major view of slot 0
            bool ok = true;
            // dV / dK products of query block gp, the it-th block of item j
            const uint64_t pol = l2_evict_first_policy();
            auto grads = [&](int gp, int j, int it, bool last) -> bool {
                const int pb = gp & 1, pe = gp % NLD;
                if (!mbar_wait(&bar->pds_full[pb], (gp >> 1) & 1, abort_flag, nullptr)) return false;
                if (store_ds) {  // dS^T of block gp, staged by the softmax warps: rows = its 128 keys
                    const int p = item_of(j, nitems), kb = p / BH, bh = p % BH;
                    tma_store_ds_hint(&tds, sm + dkv::OFF_DS + pb * dkv::TDS, 2 * kb + it, 2 * kb, bh, pol);
                    bulk_commit();
                }
                if (it == 0 && j > 0 && !mbar_wait(&bar->dkv_free, (j - 1) & 1, abort_flag, nullptr)) return false;
                tc_fence_after();
                const uint64_t bq = ring_mn + (uint64_t)(2 * pe * (TQ >> 4));
                const uint64_t bd = ring_mn + (uint64_t)((2 * pe + 1) * (TQ >> 4));
                const uint32_t pa = tmem + C_ST + pb * 64, da = tmem + C_DPT + pb * 64;
                const uint32_t acc0 = it > 0 ? 1u : 0u;
                tc_mma_ts(tmem + C_DV, pa, bd, ID_G, acc0);
#pragma unroll
                for (int kk = 1; kk < BQ / 16; ++kk) tc_mma_ts(tmem + C_DV, pa + 16 * kk, bd + 128 * kk, ID_G, 1u);
                tc_mma_ts(tmem + C_DK, da, bq, ID_G, acc0);
#pragma unroll
                for (int kk = 1; kk < BQ / 16; ++kk) tc_mma_ts(tmem + C_DK, da + 16 * kk, bq + 128 * kk, ID_G, 1u);
                tc_commit(&bar->empty[pe]);
                if (last) tc_commit(&bar->dkv_done);
                return true;
            };
            int g = 0, pj = 0, pit = 0;
            bool plast = false;
            for (int j = 0; ok; ++j) {
                const int p = item_of(j, nitems);
                if (p < 0) break;
                const int nit = nqb - 2 * (p / BH);
                if (!(ok = mbar_wait(&bar->kv_tfull[j & 1], (j >> 1) & 1, abort_flag, nullptr))) break;
                const uint32_t tK = tmem + C_KV + 64 * (j & 1), tV = tK + 32;
                for (int it = 0; it < nit; ++it, ++g) {
                    const int bb = g & 1, e = g % NLD;
                    if (!(ok = mbar_wait(&bar->full[e], (g / NLD) & 1, abort_flag, nullptr))) break;
                    tc_fence_after();
                    const uint64_t bq = ring_k + (uint64_t)(2 * e * (TQ >> 4));
                    const uint64_t bd = ring_k + (uint64_t)((2 * e + 1) * (TQ >> 4));
                    const uint32_t ts = tmem + C_ST + bb * 64, td = tmem + C_DPT + bb * 64;
                    tc_mma_ts(ts, tK, bq, ID_ST, 0u);
#pragma unroll
                    for (int kk = 1; kk < HD / 16; ++kk) tc_mma_ts(ts, tK + 8 * kk, bq + 2 * kk, ID_ST, 1u);
                    tc_mma_ts(td, tV, bd, ID_ST, 0u);
#pragma unroll
                    for (int kk = 1; kk < HD / 16; ++kk) tc_mma_ts(td, tV + 8 * kk, bd + 2 * kk, ID_ST, 1u);
                    // the staging block of this parity is rewritten once S^T of this block is ready:
                    // the store of block g - 2 must have read it by then
                    if (store_ds) bulk_wait_read<0>();
                    tc_commit(&bar->st_full[bb]);
                    if (g > 0 && !(ok = grads(g - 1, pj, pit, plast))) break;
                    pj = j, pit = it, plast = it == nit - 1;
                }
            }
            if (ok && g > 0) grads(g - 1, pj, pit, plast);
            if (store_ds) bulk_wait_all();
            tc_commit(&bar->drain);
            mbar_drain(&bar->drain, 0);
        }
    } else {
        const int quad = warp & 3, sub = (warp - 2) >> 2;  // sub: queries [16 sub, 16 sub + 16) of each block
        const int r = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        // Row r of the staged K and V tiles of item j, elements [16 sub, 16 sub + 16)
        // (128-byte swizzle: chunk c of row r sits at chunk c ^ (r & 7)), into TMEM slot j & 1.
        auto copy_kv = [&](int j) -> bool {
            const int s = j & 1;
            if (!mbar_wait(&bar->kv_sfull[s], (j >> 1) & 1, abort_flag, nullptr)) return false;
            const uint8_t *kt = sm + OFF_KV + s * 2 * TKV + r * 128, *vt = kt + TKV;
            const int c0 = ((2 * sub) ^ (r & 7)) << 4, c1 = ((2 * sub + 1) ^ (r & 7)) << 4;
            const uint4 k0 = *reinterpret_cast<const uint4 *>(kt + c0), k1 = *reinterpret_cast<const uint4 *>(kt + c1);
            const uint4 v0 = *reinterpret_cast<const uint4 *>(vt + c0), v1 = *reinterpret_cast<const uint4 *>(vt + c1);
            const uint32_t kr[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
            const uint32_t vr[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            tmem_st8(tmem + lane_off + C_KV + 64 * s + sub * 8, kr);
            tmem_st8(tmem + lane_off + C_KV + 64 * s + 32 + sub * 8, vr);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar->kv_tfull[s]);
                mbar_arrive(&bar->kv_sempty[s]);
            }
            return true;
        };
        bool ok = copy_kv(0);
        int g = 0;
        for (int j = 0; ok; ++j) {
            const int p = item_of(j, nitems);
            if (p < 0) break;
            const int kb = p / BH, bh = p % BH, b = bh / H, h = bh % H, nit = nqb - 2 * kb;
            const int key = kb * BKY + r;
            for (int it = 0; it < nit; ++it, ++g) {
                const int bb = g & 1, e = g % NLD;
                if (!(ok = mbar_wait(&bar->st_full[bb], (g >> 1) & 1, abort_flag, nullptr))) break;
                if (!(ok = mbar_wait(&bar->ld_full[e], (g / NLD) & 1, abort_flag, nullptr))) break;
                tc_fence_after();
                const uint32_t cs = tmem + lane_off + C_ST + bb * 64 + sub * 16;
                const uint32_t cd = tmem + lane_off + C_DPT + bb * 64 + sub * 16;
                uint32_t ra[16], rb[16];
                tmem_ld16_nowait(cs, ra);
                tmem_ld16_nowait(cd, rb);
                tmem_ld_wait();
                const float *L = ldbuf + e * 128 + sub * 16, *Dv = ldbuf + e * 128 + 64 + sub * 16;
                const int q0 = (2 * kb + it) * BQ, qbase = q0 + sub * 16;
                // Blocks past the diagonal with all keys and queries below T need no
                // mask (the same answer for the whole CTA).  Otherwise the visible
                // queries of this thread's 16 are lo <= c <= hi (q >= key, q < T;
                // none if key >= T).
                const bool block_full = q0 >= kb * BKY + BKY - 1 && q0 + BQ <= T && kb * BKY + BKY <= T;
                const int lo = key - qbase, hi = key < T ? T - 1 - qbase : -1;
                const F2 sl2x2 = f2(sl2, sl2), nlog2e = f2(-LOG2E, -LOG2E);
                uint32_t wp[8], wd[8];
#pragma unroll
                for (int i = 0; i < 16; i += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(L + i);
                    const float4 d4 = *reinterpret_cast<const float4 *>(Dv + i);
                    const F2 nl[2] = {f2_mul(f2(a4.x, a4.y), nlog2e), f2_mul(f2(a4.z, a4.w), nlog2e)};
                    const F2 dd[2] = {f2(d4.x, d4.y), f2(d4.z, d4.w)};
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int c = i + 2 * h2;
                        // s * scale * log2(e) - lse * log2(e), two columns per instruction
                        const F2 t = f2_fma(f2(__uint_as_float(ra[c]), __uint_as_float(ra[c + 1])), sl2x2, nl[h2]);
                        float p0 = ex2(f2_lo(t)), p1 = ex2(f2_hi(t));
                        if (!block_full) {
                            p0 = (c >= lo && c <= hi) ? p0 : 0.f;
                            p1 = (c + 1 >= lo && c + 1 <= hi) ? p1 : 0.f;
                        }
                        wp[c >> 1] = pack_bf16x2(p0, p1);
                        const F2 ds = f2_mul(f2(p0, p1),
                                             f2_sub(f2(__uint_as_float(rb[c]), __uint_as_float(rb[c + 1])), dd[h2]));
                        wd[c >> 1] = pack_bf16x2(f2_lo(ds), f2_hi(ds));
                    }
                }
                tmem_st8(cs, wp);  // P^T over the first 8 of this thread's S^T columns
                tmem_st8(cd, wd);  // dS^T over the first 8 of its dP^T columns
                if (store_ds) {  // the same 16 values of dS^T into the block's staging tile (row r, 128-byte swizzle)
                    uint8_t *row = sm + dkv::OFF_DS + bb * dkv::TDS + r * 128;
                    *reinterpret_cast<uint4 *>(row + (((2 * sub) ^ (r & 7)) << 4)) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                    *reinterpret_cast<uint4 *>(row + (((2 * sub + 1) ^ (r & 7)) << 4)) =
                        make_uint4(wd[4], wd[5], wd[6], wd[7]);
                    fence_async_smem();  // visible to the TMA store the MMA thread issues after pds_full
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar->pds_full[bb]);
                if (it == 0 && item_of(j + 1, nitems) >= 0 && !(ok = copy_kv(j + 1))) break;
            }
            if (!ok) break;
            // dV / dK of the item: read out of TMEM, release the accumulators, store
            if (!(ok = mbar_wait(&bar->dkv_done, j & 1, abort_flag, nullptr))) break;
            tc_fence_after();
            uint32_t ra[16], rb[16];
            tmem_ld16_nowait(tmem + lane_off + C_DV + sub * 16, ra);
            tmem_ld16_nowait(tmem + lane_off + C_DK + sub * 16, rb);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->dkv_free);
            if (key < T) {
                const int64_t off = ((int64_t)b * T + key) * rs + h * HD + sub * 16;
#pragma unroll
                for (int d = 0; d < 16; d += 8) {
                    uint4 u, w;
                    u.x = pack_bf16x2(__uint_as_float(ra[d]), __uint_as_float(ra[d + 1]));
                    u.y = pack_bf16x2(__uint_as_float(ra[d + 2]), __uint_as_float(ra[d + 3]));
                    u.z = pack_bf16x2(__uint_as_float(ra[d + 4]), __uint_as_float(ra[d + 5]));
                    u.w = pack_bf16x2(__uint_as_float(ra[d + 6]), __uint_as_float(ra[d + 7]));
                    w.x = pack_bf16x2(__uint_as_float(rb[d]) * scale, __uint_as_float(rb[d + 1]) * scale);
                    w.y = pack_bf16x2(__uint_as_float(rb[d + 2]) * scale, __uint_as_float(rb[d + 3]) * scale);
                    w.z = pack_bf16x2(__uint_as_float(rb[d + 4]) * scale, __uint_as_float(rb[d + 5]) * scale);
                    w.w = pack_bf16x2(__uint_as_float(rb[d + 6]) * scale, __uint_as_float(rb[d + 7]) * scale);
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
        tmem_dealloc(tmem, TCOLS);
    }
}

// ---------------------------------------------------------------- D and the value-bias sums
// D[b*H + h, t] = sum_d dO[b, t, h, d] O[b, t, h, d] (fp32) for the dK/dV
// kernel, and, with dbv, dbv[c] += the column sums of dO over all rows (the
// value-bias gradient: every row of P sums to one).  One warp per row at a time;
// in pass i lane l holds columns [8 (l + 32 i), +8), so the 8 lanes of a head
// finish its dot product with three shuffles.  NIT = ceil(C / 256) passes, C = 64 H <= 2048.
namespace rdot {
constexpr int WARPS = 16, MAXIT = 8;
}
template <int NIT>
__global__ void __launch_bounds__(32 * rdot::WARPS)
    bwd_rowdot_kernel(const bf16 *__restrict__ dout, const bf16 *__restrict__ o, int64_t ors,
                      float *__restrict__ Dscr, float *__restrict__ dbv, int BT, int T, int H) {
    __shared__ float cs[NIT * 256];
    const int C = H * HD, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (dbv)
        for (int c = threadIdx.x; c < NIT * 256; c += blockDim.x) cs[c] = 0.f;
    float acc[NIT][8];
#pragma unroll
    for (int i = 0; i < NIT; ++i)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[i][k] = 0.f;
    // RPI rows per pass: all of their loads are in flight before the first is used
    constexpr int RPI = NIT <= 4 ? 2 : 1;
    for (int row0 = (blockIdx.x * rdot::WARPS + warp) * RPI; row0 < BT; row0 += gridDim.x * rdot::WARPS * RPI) {
        uint4 a[RPI][NIT], v[RPI][NIT];
#pragma unroll
        for (int rr = 0; rr < RPI; ++rr)
#pragma unroll
            for (int i = 0; i < NIT; ++i) {
                const int row = row0 + rr, c = (lane + 32 * i) * 8;
                a[rr][i] = v[rr][i] = make_uint4(0u, 0u, 0u, 0u);
                if (row < BT && c < C) {
                    a[rr][i] = *reinterpret_cast<const uint4 *>(dout + (int64_t)row * ors + c);
                    v[rr][i] = *reinterpret_cast<const uint4 *>(o + (int64_t)row * ors + c);
                }
            }
#pragma unroll
        for (int rr = 0; rr < RPI; ++rr) {
            const int row = row0 + rr;
            if (row >= BT) break;  // the same for the whole warp
            const int b = row / T, t = row - b * T;
#pragma unroll
            for (int i = 0; i < NIT; ++i) {
                const int c = (lane + 32 * i) * 8;
                const uint32_t aw[4] = {a[rr][i].x, a[rr][i].y, a[rr][i].z, a[rr][i].w};
                const uint32_t vw[4] = {v[rr][i].x, v[rr][i].y, v[rr][i].z, v[rr][i].w};
                float s = 0.f;
#pragma unroll
                for (int w = 0; w < 4; ++w) {  // columns past C hold zeros
                    s = fmaf(bf16_lo(aw[w]), bf16_lo(vw[w]), s);
                    s = fmaf(bf16_hi(aw[w]), bf16_hi(vw[w]), s);
                    acc[i][2 * w] += bf16_lo(aw[w]);
                    acc[i][2 * w + 1] += bf16_hi(aw[w]);
                }
                s += __shfl_xor_sync(~0u, s, 1);
                s += __shfl_xor_sync(~0u, s, 2);
                s += __shfl_xor_sync(~0u, s, 4);
                if ((lane & 7) == 0 && c < C) Dscr[((int64_t)b * H + c / HD) * T + t] = s;
            }
        }
    }
    if (dbv) {
        __syncthreads();
#pragma unroll
        for (int i = 0; i < NIT; ++i) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int c = (lane + 32 * i) * 8 + k;
                if (c < C) atomicAdd(cs + c, acc[i][k]);
            }
        }
        __syncthreads();
        for (int c = threadIdx.x; c < C; c += blockDim.x)
            if (cs[c] != 0.f) atomicAdd(dbv + c, cs[c]);
    }
}

// ---------------------------------------------------------------- dQ from the stored dS
// dQ = scale dS K per (128-query block, b*h) item, over the key blocks of 64 up
// to the item's diagonal.  The dK/dV kernel stored dS^T as bf16 in 64 x 64 blocks
// (row = key, the queries contiguous; see encode_ds_map): the A operand (M =
// queries, K = keys) is MN-major; K is the MN-major B operand (N = the head's 64
// columns).  The
// accumulator (128 x 64 fp32) is double-buffered in TMEM, so the read-out of an
// item overlaps the products of the next.  With dbq, the column sums of dQ
// (query-bias gradient) are added to it.
// Warps: 0 loads (TMA), 1 issues the MMAs, 2-5 read out (one per TMEM lane quadrant).
namespace dqs {
constexpr int BQ = 128, BK = 64, NST = 8, EWARPS = 4;
constexpr int NTH = 64 + 32 * EWARPS;
constexpr int A_BYTES = BQ * BK * 2;  // 16 KB: two 64-query MN-major blocks
constexpr int B_BYTES = BK * HD * 2;  // 8 KB
constexpr int STAGE = A_BYTES + B_BYTES;
constexpr int MAXC = 2048;
constexpr int OFF_BSUM = NST * STAGE;
constexpr int OFF_BAR = OFF_BSUM + MAXC * 4;
constexpr int SMEM = 1024 + OFF_BAR + 256;
constexpr uint32_t TCOLS = 128;
}  // namespace dqs

__global__ void __launch_bounds__(dqs::NTH, 1)
    bwd_dq_from_ds_kernel(const __grid_constant__ CUtensorMap tds, const __grid_constant__ CUtensorMap tk,
                          bf16 *__restrict__ dqo, int64_t rs, int T, int H, int nitems, float scale,
                          float *__restrict__ dbq) {
    constexpr int BQ = dqs::BQ, BK = dqs::BK, NST = dqs::NST, EWARPS = dqs::EWARPS, A_BYTES = dqs::A_BYTES,
                  STAGE = dqs::STAGE;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align_smem_1024(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + dqs::OFF_BAR), *empty = full + NST, *tfull = empty + NST,
             *tempty = tfull + 2, *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *bsum = reinterpret_cast<float *>(sm + dqs::OFF_BSUM);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nqb = (T + BQ - 1) / BQ, nkb = (T + BK - 1) / BK, BH = nitems / nqb;
    // item p: query block nqb - 1 - p / BH (heaviest first), b*h = p % BH
    auto item_qb = [&](int p) { return nqb - 1 - p / BH; };
    auto item_nk = [&](int qb) { return min(nkb, 2 * (qb + 1)); };
    if (dbq)
        for (int c = threadIdx.x; c < H * HD; c += blockDim.x) bsum[c] = 0.f;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], EWARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tds);
        tma_prefetch_desc(&tk);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, dqs::TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued_mask = 0, issued_phase = 0;
            bool ok = true;
            const uint64_t pol = l2_evict_first_policy();  // dS is read once
            for (int j = 0; ok; ++j) {
                const int p = item_of(j, nitems);
                if (p < 0) break;
                const int qb = item_qb(p), bh = p % BH, b = bh / H, h = bh % H, nk = item_nk(qb);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!(ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, nullptr))) break;
                    uint8_t *a_dst = sm + stage * STAGE, *b_dst = a_dst + A_BYTES;
                    mbar_expect_tx(&full[stage], STAGE);
                    tma_load_ds_hint(a_dst, &tds, &full[stage], 2 * qb, kb, bh, pol);  // both 64-query halves
                    tma_load_3d(b_dst, &tk, &full[stage], h * HD, kb * BK, b);
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == NST) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok)  // let the copies already issued land before the CTA exits
                for (int s = 0; s < NST; ++s)
                    if (issued_mask & (1u << s)) mbar_drain(&full[s], (issued_phase >> s) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t IDESC = instr_desc(HD, true, true);  // 128 x 64, A and B MN-major
            int stage = 0, t = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int j = 0; ok; ++j, ++t) {
                const int p = item_of(j, nitems);
                if (p < 0) break;
                const int nk = item_nk(item_qb(p)), acc = t & 1;
                if (!(ok = mbar_wait(&tempty[acc], ((t >> 1) & 1) ^ 1, abort_flag, nullptr))) break;
                tc_fence_after();
                const uint32_t d = tmem + acc * HD;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!(ok = mbar_wait(&full[stage], phase, abort_flag, nullptr))) break;
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sm + stage * STAGE), b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma(d, smem_desc(a_addr + kk * 2048, A_BYTES / 2, 1024),
                               smem_desc(b_addr + kk * 2048, A_BYTES / 2, 1024), IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&empty[stage]);
                    if (++stage == NST) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(&tfull[acc]);
            }
            tc_commit(drain);  // all MMAs issued by this thread have completed once it flips
            mbar_drain(drain, 0);
        }
    } else {
        const int quad = warp & 3, r = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        int t = 0;
        for (int j = 0;; ++j, ++t) {
            const int p = item_of(j, nitems);
            if (p < 0) break;
            const int qb = item_qb(p), bh = p % BH, b = bh / H, h = bh % H, acc = t & 1;
            if (!mbar_wait(&tfull[acc], (t >> 1) & 1, abort_flag, nullptr)) break;
            tc_fence_after();
            uint32_t ra[32], rb[32];
            tmem_ld32(tmem + lane_off + acc * HD, ra);
            tmem_ld32(tmem + lane_off + acc * HD + 32, rb);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            const int q = qb * BQ + r;
            if (dbq) {  // query-bias gradient: column sums of dQ (one warp = 32 rows) into the CTA's partials
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    float cv[16];
#pragma unroll
                    for (int d = 0; d < 16; ++d)
                        cv[d] = q < T ? __uint_as_float(g < 2 ? ra[16 * g + d] : rb[16 * (g - 2) + d]) * scale : 0.f;
                    warp_colsum16_add(cv, bsum + h * HD + 16 * g, lane);
                }
            }
            if (q < T) {
                bf16 *row = dqo + ((int64_t)b * T + q) * rs + h * HD;
#pragma unroll
                for (int d = 0; d < 64; d += 8) {
                    const uint32_t *x = d < 32 ? ra + d : rb + (d - 32);
                    uint4 u;
                    u.x = pack_bf16x2(__uint_as_float(x[0]) * scale, __uint_as_float(x[1]) * scale);
                    u.y = pack_bf16x2(__uint_as_float(x[2]) * scale, __uint_as_float(x[3]) * scale);
                    u.z = pack_bf16x2(__uint_as_float(x[4]) * scale, __uint_as_float(x[5]) * scale);
                    u.w = pack_bf16x2(__uint_as_float(x[6]) * scale, __uint_as_float(x[7]) * scale);
                    *reinterpret_cast<uint4 *>(row + d) = u;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, dqs::TCOLS);
    }
    if (dbq)  // one atomic per head column and CTA
        for (int c = threadIdx.x; c < H * HD; c += blockDim.x)
            if (bsum[c] != 0.f) atomicAdd(dbq + c, bsum[c]);
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

// Map over the stored dS^T in blocks: for each b*h, key block kb and query block qb
// (blocks of 64), the 64 x 64 block [key][query] is contiguous (8 KB), blocks in
// (bh, kb, qb) order, so that a box of two query blocks (the dQ loads) is 16 KB of
// consecutive memory and one of two key blocks (the dK/dV stores) two runs of 8 KB.
// Dimensions, innermost first: query in block, key in block, qb, kb, bh; the box
// is 64 x 64 x box_qb x box_kb x 1, which lands in shared memory as box_qb * box_kb
// row-major 64 x 64 blocks (128-byte rows, 128-byte swizzle).
static int encode_ds_map(CUtensorMap *tm, const void *base, int BH, int Tp, int box_qb, int box_kb) {
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
    const cuuint64_t nb = (cuuint64_t)Tp / 64;
    cuuint64_t dims[5] = {64, 64, nb, nb, (cuuint64_t)BH};
    cuuint64_t strides[4] = {128, 8192, 8192 * nb, 8192 * nb * nb};
    cuuint32_t box[5] = {64, 64, (cuuint32_t)box_qb, (cuuint32_t)box_kb, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box, estr,
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
    static PerDevice init_pd;
    int unused = 0;
    if (int rc = per_device(init_pd, unused, [](int &v) -> int {
            GPT2_CUDA_TRY(cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::SMEM));
            v = 1;
            return GPT2_OK;
        }))
        return rc;
    const float sl2 = LOG2E / sqrtf((float)HD);
    int dev = 0, sms = 0;
    GPT2_CUDA_TRY(cudaGetDevice(&dev));
    GPT2_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    // persistent grid: one CTA per SM over (query block, b*h) items, heaviest first
    const int nitems = ((T + fwd::BQ - 1) / fwd::BQ) * B * H;
    fwd_tc_kernel<<<std::min(nitems, sms), fwd::NTH, fwd::SMEM, st>>>(mq, mk, mv, o, ors, lse, T, H, nitems, sl2);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

size_t attention_backward_ds_bytes(int B, int T, int H) {
    const int64_t Tp = ((int64_t)T + 127) / 128 * 128;
    return (size_t)B * H * Tp * Tp * 2;
}

int attention_backward_tc(const bf16 *q, const bf16 *k, const bf16 *v, int64_t rs, const bf16 *o, const bf16 *dout,
                          int64_t ors, const float *lse, bf16 *dq_out, bf16 *dk_out, bf16 *dv_out, float *Dscr, int B,
                          int T, int H, cudaStream_t st, float *dbias, bf16 *ds_ws) {
    using namespace fatc;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq_out) |
         reinterpret_cast<uintptr_t>(dk_out) | reinterpret_cast<uintptr_t>(dv_out)) & 15)
        return GPT2_ERR_BAD_ARG;
    CUtensorMap q128, do128, o128, k64, v64, q64, do64, k128, v128;
    if (dbias && H * HD > dq::MAXC) return GPT2_ERR_UNSUPPORTED;
    if (int rc = encode_qkv_map(&q128, q, rs, T, B, H, 128)) return rc;
    if (int rc = encode_qkv_map(&do128, dout, ors, T, B, H, 128)) return rc;
    if (int rc = encode_qkv_map(&o128, o, ors, T, B, H, 128)) return rc;
    if (int rc = encode_qkv_map(&k64, k, rs, T, B, H, 64)) return rc;
    if (int rc = encode_qkv_map(&v64, v, rs, T, B, H, 64)) return rc;
    if (int rc = encode_qkv_map(&q64, q, rs, T, B, H, 64)) return rc;
    if (int rc = encode_qkv_map(&k128, k, rs, T, B, H, 128)) return rc;
    if (int rc = encode_qkv_map(&v128, v, rs, T, B, H, 128)) return rc;
    if (int rc = encode_qkv_map(&do64, dout, ors, T, B, H, 64)) return rc;
    static PerDevice init_pd;
    int unused = 0;
    if (int rc = per_device(init_pd, unused, [](int &v) -> int {
            GPT2_CUDA_TRY(cudaFuncSetAttribute(bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dq::SMEM));
            GPT2_CUDA_TRY(
                cudaFuncSetAttribute(bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dkv::SMEM));
            GPT2_CUDA_TRY(
                cudaFuncSetAttribute(bwd_dq_from_ds_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dqs::SMEM));
            v = 1;
            return GPT2_OK;
        }))
        return rc;
    const float scale = 1.0f / sqrtf((float)HD), sl2 = LOG2E * scale;
    int dev = 0, sms = 0;
    GPT2_CUDA_TRY(cudaGetDevice(&dev));
    GPT2_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int nitems = ((T + dkv::BKY - 1) / dkv::BKY) * B * H;
    if (ds_ws && H * HD <= rdot::MAXIT * 256) {
        // D (and the value-bias sums) first; the dK/dV kernel stores dS^T, from which a
        // plain tcgen05 product forms dQ (and the query-bias sums)
        if (reinterpret_cast<uintptr_t>(ds_ws) & 15) return GPT2_ERR_BAD_ARG;
        const int Tp = (T + 127) / 128 * 128;
        CUtensorMap tds_ld, tds_st;  // boxes of 128 queries x 64 keys (dQ loads), 64 x 128 (dK/dV stores)
        if (int rc = encode_ds_map(&tds_ld, ds_ws, B * H, Tp, 2, 1)) return rc;
        if (int rc = encode_ds_map(&tds_st, ds_ws, B * H, Tp, 1, 2)) return rc;
        const int BT = B * T;
        const int rblocks = std::min((BT + 2 * rdot::WARPS - 1) / (2 * rdot::WARPS), sms);  // one per SM at most
        float *dbv = dbias ? dbias + 2 * H * HD : nullptr;
        switch ((H * HD + 255) / 256) {
#define ROWDOT_CASE(n)                                                                                      \
    case n:                                                                                                 \
        bwd_rowdot_kernel<n><<<rblocks, 32 * rdot::WARPS, 0, st>>>(dout, o, ors, Dscr, dbv, BT, T, H); \
        break;
            ROWDOT_CASE(1)
            ROWDOT_CASE(2)
            ROWDOT_CASE(3)
            ROWDOT_CASE(4)
            ROWDOT_CASE(5)
            ROWDOT_CASE(6)
            ROWDOT_CASE(7)
            ROWDOT_CASE(8)
#undef ROWDOT_CASE
        }
        GPT2_CUDA_TRY(cudaGetLastError());
        bwd_dkv_tc_kernel<<<std::min(nitems, sms), dkv::NTH, dkv::SMEM, st>>>(
            q64, do64, k128, v128, tds_st, lse, Dscr, dk_out, dv_out, rs, T, H, nitems, sl2, scale, 1);
        GPT2_CUDA_TRY(cudaGetLastError());
        const int nq_items = ((T + dqs::BQ - 1) / dqs::BQ) * B * H;
        bwd_dq_from_ds_kernel<<<std::min(nq_items, sms), dqs::NTH, dqs::SMEM, st>>>(tds_ld, k64, dq_out, rs, T, H,
                                                                                    nq_items, scale, dbias);
        GPT2_CUDA_TRY(cudaGetLastError());
        gpt2_note_launches(3);
        return GPT2_OK;
    }
    // persistent dQ grid: one CTA per SM over (query block, b*h) items, heaviest first
    const int nq_items = ((T + dq::BQ - 1) / dq::BQ) * B * H;
    bwd_dq_tc_kernel<<<std::min(nq_items, sms), dq::NTH, dq::SMEM, st>>>(q128, do128, o128, k64, v64, lse, dq_out, rs,
                                                                         Dscr, T, H, nq_items, sl2, scale, dbias,
                                                                         dbias ? dbias + 2 * H * HD : nullptr);
    GPT2_CUDA_TRY(cudaGetLastError());
    // persistent dK/dV grid: one CTA per SM over (key block, b*h) items, heaviest first
    bwd_dkv_tc_kernel<<<std::min(nitems, sms), dkv::NTH, dkv::SMEM, st>>>(
        q64, do64, k128, v128, q64 /* unused */, lse, Dscr, dk_out, dv_out, rs, T, H, nitems, sl2, scale, 0);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(2);
    return GPT2_OK;
}

}  // namespace fa
