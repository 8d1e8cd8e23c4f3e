// bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// Every dense contraction of the GPT-2 step (QKV, attention projection, FC,
// FC projection and the tied LM head, forward and both backward products) is
// one call of this kernel ("llm.c kullanarak GPT-2 modelini düşük maliyetle
// yeniden uygulamak", §Kod yapısı: the Transformer forward/backward is matmuls
// plus pointwise work; "Let's reproduce GPT-2 (124M)", §Bölümler 5: Tensor
// Cores).  acc[m, n] = sum_k A(m, k) B(n, k), fp32 accumulation in TMEM.
//
// Design (one CTA per SM, persistent over output tiles):
//   warp 0    one thread issues TMA loads of A/B k-blocks into a STAGES-deep
//             shared-memory ring (128-byte swizzle);
//   warp 1    allocates TMEM (2 accumulators x BN columns) and one thread
//             issues tcgen05.mma (M=128, N=BN, K=16) per 16-wide k slice,
//             committing each ring slot back to the producer and each finished
//             accumulator to the epilogue;
//   warps 2-9 epilogue: two warps per TMEM lane quadrant, each reading half of
//             the tile's columns with tcgen05.ld (32 lanes x 32 columns, two
//             loads in flight), fused bias / residual / GELU / GELU' / fp32
//             accumulate, 16-byte stores.
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
// Operands may be K-major (k contiguous) or MN-major (m or n contiguous), which
// covers Y = X W^T, dX = dY W and dW = dY^T X without transposes.
// Every mbarrier wait is bounded (globaltimer); on timeout the CTA records
// DEVERR_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and exits.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace tcg {

constexpr int BM = 128;            // rows of a tile = TMEM lanes
constexpr int BK = 64;             // 64 bf16 = one 128-byte swizzle row
constexpr int A_STAGE_BYTES = BM * BK * 2;
constexpr int MN_BLOCK_BYTES = 64 * BK * 2;  // one 64-wide MN-major TMA box (64 k rows x 128 B)
constexpr int EPI_WARPS = 8;  // two warps per TMEM lane quadrant, each owning half the tile's columns
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr uint64_t WAIT_LIMIT_NS = 4000000000ull;  // 4 s: far above any legitimate wait

// Epilogues of the LM head fused with the cross-entropy (not part of the C ABI's
// GPT2_EPI_* set).  Columns at or past `vocab` are padding and take no part.
//  EPI_LSE: no output; per row and per half tile (BN / 2 columns) the pair
//           (max, sum of exp(z - max)) goes to row_part[row * part_stride +
//           2 * n_tile + half], and z[row, tgt[row]] to row_zt[row].
//  EPI_DZ:  bf16 output dz = (exp(z - lse[row]) - [col == tgt[row]]) * dz_scale
//           for col < vocab, 0 past it.
constexpr int EPI_LSE = 100;
constexpr int EPI_DZ = 101;

struct Params {
    int M, N, K;
    int num_m_blocks, num_n_blocks, num_k_blocks;
    int splits, k_blocks_per_split;
    int n_fastest;  // tile raster: 1 = consecutive tiles share the A block (A is the large operand)
    int epi;
    float alpha;
    const float *bias;
    const bf16 *R;
    float *dbias;  // optional: += column sums of the stored bf16 output (bias gradient of the product)
    const float *a_scale;  // optional: per-row factor of acc (E4M3 operands: row dequantisation of A)
    const float *b_scale;  // optional: one factor of acc (E4M3 operands: dequantisation of B)
    // EPI_LSE / EPI_DZ (see above)
    int vocab, part_stride;
    const int *row_tgt;
    const float *row_lse;
    float2 *row_part;
    float *row_zt;
    float dz_scale;
    void *D;
    bf16 *D2;
    int64_t ldd;
    int *err;
    // Work units of the launch.  With ngroups = 2 a second product runs in the same
    // launch (fp32 accumulate, same K and splits): units at or past work1 are its
    // tiles, with the geometry below and the tensor maps of GroupMaps.
    int num_work, ngroups, work1;
    int g2_M, g2_N, g2_num_m_blocks, g2_num_n_blocks, g2_n_fastest;
};

// Tensor maps of the second product of a grouped launch (A, B, fp32 D); each
// CUtensorMap carries its own 128-byte alignment.
struct GroupMaps {
    CUtensorMap a, b, d;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 1024-byte aligned base inside the dynamic shared-memory array.  The offset is
// added to the array pointer itself (no round trip through an integer), so the
// compiler still knows the result points to shared memory and emits
// shared-memory loads and stores for it rather than generic ones.
__device__ __forceinline__ uint8_t *align_smem_1024(uint8_t *raw) {
    return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking test: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity; false on timeout or abort.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) {
            *abort_flag = 1;
            raise_device_error(err, DEVERR_TIMEOUT);
            return false;
        }
    }
}
// Bounded wait used only on the abort path (no abort check).
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_timer_ns() - t0 > 1000000000ull) return;
}

// ---- TMA --------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *tm, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *tm, uint64_t *bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}
// TMA store of a shared-memory box to global memory (bulk async-group of the issuing thread)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *tm, const void *src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
// TMA reduction of a shared-memory box into global memory: D[box] += smem, element
// type from the tensor map (fp32 here); same bulk async-group rules as the store.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *tm, const void *src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N of this thread's bulk groups still read shared memory
template <int N> __device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// wait until all of this thread's bulk groups have completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// make this thread's shared-memory writes visible to the async proxy (TMA, tensor cores)
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- tcgen05 ------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (>> 4), descriptor version 1 at bit 46, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor: fp32 accumulator (bit 4), A and B formats (bits 7-9,
// 10-12: 1 = bf16 for kind::f16, 0 = E4M3 for kind::f8f6f4), operand
// majorness, N >> 3 and M >> 4.
__host__ __device__ constexpr uint32_t instr_desc(int bn, bool a_mn, bool b_mn, bool f8 = false) {
    return (1u << 4) | ((f8 ? 0u : 1u) << 7) | ((f8 ? 0u : 1u) << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// Instruction descriptor for a CTA-pair MMA (cta_group::2): M = 256.
__host__ __device__ constexpr uint32_t instr_desc_pair(int bn, bool a_mn, bool b_mn, bool f8 = false) {
    return (1u << 4) | ((f8 ? 0u : 1u) << 7) | ((f8 ? 0u : 1u) << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
}

// E4M3 x E4M3 -> fp32 MMAs (kind::f8f6f4, K = 32 per instruction: the same
// 32 bytes of each operand row as a bf16 MMA with K = 16)
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ---- CTA pairs (cluster of two, cta_group::2) ------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// address of the same shared-memory object in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t smem_in_rank(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
// TMA load into this CTA's shared memory, completion counted on an mbarrier of either CTA of the pair
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *tm, uint32_t bar_cluster, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void tc_mma_pair_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive (when the MMAs issued so far complete) on the mbarrier at this offset in the CTAs of `mask`
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}
// Release of a TMEM accumulator to the even CTA of a pair.  The even CTA arrives
// on its own barrier; the odd CTA arrives remotely with relaxed semantics: its
// tcgen05.ld reads have completed (tcgen05.wait::ld) and are ordered before the
// arrive by tcgen05.fence::before_thread_sync, and there is no memory write
// that the MMA side has to observe, so a cluster-scope release is not needed.
__device__ __forceinline__ void release_accumulator(uint64_t *bar, uint32_t rank) {
    if (rank == 0)
        mbar_arrive(bar);
    else
        asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(smem_in_rank(bar, 0))
                     : "memory");
}

constexpr int EPI_STAGE_BYTES = 32 * 128;  // per epilogue warp: 32 rows x 64 bf16

// Epilogues with a second staging block per warp (3-deep ring single, 5-deep
// pair): operand-reading epilogues (residual, GELU input) fetch the next 32 x 64
// block of that operand (cp.async) into it while the current one is computed
// and stored; the GELU epilogue stores its two outputs from the two blocks.
// PAIR: a CTA pair shares one 256 x BN tile (cta_group::2), each CTA holding
// 128 rows of A and BN / 2 rows of B per stage; the R-reading variant of the
// pair kernel has 5 stages.
template <int BN, int STAGES, bool PAIR = false>
struct SmemLayout {
    static constexpr int B_STAGE_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    static constexpr int EPI_BUFS = (PAIR ? STAGES == 5 : STAGES == 3) ? 2 : 1;
    static constexpr int EPI_OFFSET = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFFSET = EPI_OFFSET + EPI_WARPS * EPI_BUFS * EPI_STAGE_BYTES;
    static constexpr int BAR_BYTES = (2 * STAGES + 5) * 8 + 16;
    static constexpr int TOTAL = 1024 /*alignment slack*/ + BAR_OFFSET + BAR_BYTES;
};

// Tile raster: m-fastest keeps one B block shared by the concurrently running
// tiles; n-fastest keeps one A block shared (used when A is the operand too
// large for L2 and N has few blocks, e.g. the LM-head backward over dlogits).
__device__ __forceinline__ int tile_m(const Params &P, int tile) {
    return P.n_fastest ? tile / P.num_n_blocks : tile % P.num_m_blocks;
}
__device__ __forceinline__ int tile_n(const Params &P, int tile) {
    return P.n_fastest ? tile % P.num_n_blocks : tile / P.num_m_blocks;
}

// Work unit w: its tile (m, n blocks), K-block range and product (0, or 1 for the
// second product of a grouped launch).
struct UnitView {
    int tm, tn, kb0, kb1, second;
};
__device__ __forceinline__ UnitView unit_view(const Params &P, int w) {
    UnitView u;
    u.second = P.ngroups > 1 && w >= P.work1;
    const int wl = u.second ? w - P.work1 : w;
    const int split = wl % P.splits, tile = wl / P.splits;
    if (u.second) {
        u.tm = P.g2_n_fastest ? tile / P.g2_num_n_blocks : tile % P.g2_num_m_blocks;
        u.tn = P.g2_n_fastest ? tile % P.g2_num_n_blocks : tile / P.g2_num_m_blocks;
    } else {
        u.tm = tile_m(P, tile);
        u.tn = tile_n(P, tile);
    }
    u.kb0 = split * P.k_blocks_per_split;
    u.kb1 = min(P.num_k_blocks, u.kb0 + P.k_blocks_per_split);
    return u;
}

// ---- epilogue -----------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// EPI_LSE: fold 64 columns of one row's logits (starting at col) into its
// running (max m, sum s of 2^((z - m) log2 e)); record z at the row's target.
__device__ __forceinline__ void lse_group(const Params &P, int row, int col, const uint32_t (&r0)[32],
                                          const uint32_t (&r1)[32], float &m, float &s);

// 2^x with the hardware approximation (MUFU.EX2, flush-to-zero): the
// cross-entropy's exponentials are summed in fp32 or stored as bf16, far above
// its error.
__device__ __forceinline__ float ex2_hw(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float LOG2E_F = 1.4426950408889634f;

__device__ __forceinline__ void lse_group(const Params &P, int row, int col, const uint32_t (&r0)[32],
                                          const uint32_t (&r1)[32], float &m, float &s) {
    const int nv = min(64, P.vocab - col);  // real columns of the group (may be <= 0)
    if (nv <= 0) return;
    float gm = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        gm = fmaxf(gm, i < nv ? __uint_as_float(r0[i]) : -INFINITY);
        gm = fmaxf(gm, 32 + i < nv ? __uint_as_float(r1[i]) : -INFINITY);
    }
    const float nm = fmaxf(m, gm), nb = -nm * LOG2E_F;
    float acc = s * ex2_hw((m - nm) * LOG2E_F);  // m = -inf: the factor is 0 (s is 0 too)
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        acc += i < nv ? ex2_hw(fmaf(__uint_as_float(r0[i]), LOG2E_F, nb)) : 0.f;
        acc += 32 + i < nv ? ex2_hw(fmaf(__uint_as_float(r1[i]), LOG2E_F, nb)) : 0.f;
    }
    m = nm;
    s = acc;
    if (row < P.M) {
        int tg = P.row_tgt[row];
        if (tg < 0 || tg >= P.vocab) tg = 0;  // an invalid target counts as token 0 (reported elsewhere)
        const int tc = tg - col;
        if (tc >= 0 && tc < 64) {
            float z = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                z = tc == i ? __uint_as_float(r0[i]) : z;
                z = tc == 32 + i ? __uint_as_float(r1[i]) : z;
            }
            P.row_zt[row] = z;
        }
    }
}

// 32 accumulator columns of one row -> global memory.
__device__ __forceinline__ void epilogue_chunk(const Params &P, int row, int col0, const uint32_t (&r)[32]) {
    if (row >= P.M) return;
    float fac = P.alpha;
    if (P.a_scale) fac *= P.a_scale[row];
    if (P.b_scale) fac *= *P.b_scale;
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(r[i]) * fac;
    if (P.epi == GPT2_EPI_ACCUM_F32) {
        float *D = reinterpret_cast<float *>(P.D) + (int64_t)row * P.ldd;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const int col = col0 + 4 * g;
            if (col >= P.N) break;
            float4 *p = reinterpret_cast<float4 *>(D + col);
            if (P.splits == 1) {
                float4 o = *p;
                o.x += acc[4 * g + 0];
                o.y += acc[4 * g + 1];
                o.z += acc[4 * g + 2];
                o.w += acc[4 * g + 3];
                *p = o;
            } else {  // split-K partial: one 16-byte vector reduction
                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(D + col), "f"(acc[4 * g + 0]),
                             "f"(acc[4 * g + 1]), "f"(acc[4 * g + 2]), "f"(acc[4 * g + 3])
                             : "memory");
            }
        }
        return;
    }
    bf16 *D = reinterpret_cast<bf16 *>(P.D) + (int64_t)row * P.ldd;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int col = col0 + 8 * g;
        if (col >= P.N) break;
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = acc[8 * g + i];
        if (P.bias && P.epi != GPT2_EPI_GELU_BWD) {
            const float4 b0 = *reinterpret_cast<const float4 *>(P.bias + col);
            const float4 b1 = *reinterpret_cast<const float4 *>(P.bias + col + 4);
            x[0] += b0.x; x[1] += b0.y; x[2] += b0.z; x[3] += b0.w;
            x[4] += b1.x; x[5] += b1.y; x[6] += b1.z; x[7] += b1.w;
        }
        if (P.epi == GPT2_EPI_RESIDUAL || P.epi == GPT2_EPI_GELU_BWD) {
            uint4 rv = *reinterpret_cast<const uint4 *>(P.R + (int64_t)row * P.ldd + col);
            const bf16 *rb = reinterpret_cast<const bf16 *>(&rv);
            if (P.epi == GPT2_EPI_RESIDUAL) {
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] += __bfloat162float(rb[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] *= gelu_tanh_grad(__bfloat162float(rb[i]));
            }
        }
        uint4 o;
        o.x = pack_bf16x2(x[0], x[1]);
        o.y = pack_bf16x2(x[2], x[3]);
        o.z = pack_bf16x2(x[4], x[5]);
        o.w = pack_bf16x2(x[6], x[7]);
        *reinterpret_cast<uint4 *>(D + col) = o;
        if (P.epi == GPT2_EPI_GELU) {
            // GELU of the bf16-rounded pre-activation, so a recompute from the
            // stored h reproduces the stored output bit for bit.
            const bf16 *hb = reinterpret_cast<const bf16 *>(&o);
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = gelu_tanh(__bfloat162float(hb[i]));
            uint4 og;
            og.x = pack_bf16x2(y[0], y[1]);
            og.y = pack_bf16x2(y[2], y[3]);
            og.z = pack_bf16x2(y[4], y[5]);
            og.w = pack_bf16x2(y[6], y[7]);
            *reinterpret_cast<uint4 *>(P.D2 + (int64_t)row * P.ldd + col) = og;
        }
    }
}

// ---- staged bf16 epilogue: 32 rows x 64 columns per warp ------------------------
// Each lane owns one row in TMEM order; the warp's tile passes through a
// swizzled shared-memory block so that global loads (residual / h) and stores
// are whole 128-byte row segments instead of 16 bytes from 32 different rows.
__device__ __forceinline__ uint4 *stage_at(uint8_t *stage, int row, int chunk) {
    return reinterpret_cast<uint4 *>(stage + row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void stage_load(uint8_t *stage, const bf16 *g, int64_t ld, int row0, int col0, int M, int N,
                                           int lane) {
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int rr = it * 4 + (lane >> 3), ch = lane & 7;
        const int row = row0 + rr, col = col0 + ch * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < M && col < N) v = *reinterpret_cast<const uint4 *>(g + (int64_t)row * ld + col);
        *stage_at(stage, rr, ch) = v;
    }
}

// Asynchronous version of stage_load (cp.async, 16 bytes per lane per step,
// zero fill outside [M, N)); complete it with cp_async_wait_all + __syncwarp.
__device__ __forceinline__ void stage_prefetch(uint8_t *stage, const bf16 *g, int64_t ld, int row0, int col0, int M,
                                               int N, int lane) {
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int rr = it * 4 + (lane >> 3), ch = lane & 7;
        const int row = row0 + rr, col = col0 + ch * 8;
        const bool ok = row < M && col < N;
        const bf16 *src = ok ? g + (int64_t)row * ld + col : g;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(stage_at(stage, rr, ch))),
                     "l"(src), "r"(ok ? 16 : 0)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// 32 accumulator columns of the warp's 32 rows added into the fp32 output: the
// scaled block passes through the warp's swizzled staging block (32 rows x 128
// bytes) and leaves as one TMA reduce-add, so the L2 receives whole 128-byte row
// segments instead of 16 bytes from each of 32 rows.  Rows at or past M and
// columns at or past N fall outside the tensor map and are not written.  The
// result is D + acc whether or not other work units add into the same block.
__device__ __forceinline__ void reduce_block32(const Params &P, const CUtensorMap *tmD, uint8_t *stage, int row0,
                                               int col, int lane, const uint32_t (&r)[32]) {
    float fac = P.alpha;
    if (P.a_scale) fac *= P.a_scale[min(row0 + lane, P.M - 1)];
    if (P.b_scale) fac *= *P.b_scale;
    if (lane == 0) bulk_wait_read<0>();  // the previous TMA store / reduce from this block has read it
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *stage_at(stage, lane, c) =
            make_uint4(__float_as_uint(__uint_as_float(r[4 * c]) * fac), __float_as_uint(__uint_as_float(r[4 * c + 1]) * fac),
                       __float_as_uint(__uint_as_float(r[4 * c + 2]) * fac),
                       __float_as_uint(__uint_as_float(r[4 * c + 3]) * fac));
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_reduce_add_2d(tmD, stage, col, row0);
        bulk_commit();
    }
}

// 64 accumulator columns (two 32-column TMEM loads) of the warp's 32 rows -> bf16
// outputs with the fused epilogue; row0 is the warp's first row, col0 the group's
// first column.
// rstage: if non-null, the block of R for this group is already being fetched
// there (stage_prefetch); otherwise R is loaded through `stage`.
// The bf16 outputs leave through TMA stores of the warp's staging block (the
// staging layout is the 128-byte swizzle of the store maps, box 64 x 32): lane 0
// issues them and, before a staging block is written again, waits until the
// store that last used it has read it.  `stage2` is a second staging block for
// the GELU output (or null: the first one is reused).
__device__ __forceinline__ void epilogue_group64(const Params &P, const CUtensorMap *tmD, const CUtensorMap *tmD2,
                                                 uint8_t *stage, uint8_t *stage2, uint8_t *rstage, int row0, int col0,
                                                 int lane, const uint32_t (&r0)[32], const uint32_t (&r1)[32]) {
    // x[i] holds columns 2i, 2i+1; the arithmetic runs on pairs (.f32x2)
    F2 x[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        x[i] = f2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
        x[16 + i] = f2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
    }
    if (P.alpha != 1.0f || P.a_scale || P.b_scale) {
        float fac = P.alpha;
        if (P.a_scale) fac *= P.a_scale[min(row0 + lane, P.M - 1)];
        if (P.b_scale) fac *= *P.b_scale;
        const F2 al = f2(fac, fac);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = f2_mul(x[i], al);
    }
    if (P.bias && P.epi != GPT2_EPI_GELU_BWD) {
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
            float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
            if (col0 + i < P.N) b = *reinterpret_cast<const float4 *>(P.bias + col0 + i);
            x[i / 2] = f2_add(x[i / 2], f2(b.x, b.y));
            x[i / 2 + 1] = f2_add(x[i / 2 + 1], f2(b.z, b.w));
        }
    }
    if (P.epi == EPI_DZ) {  // dz of the cross-entropy from the recomputed logits
        const int rr = min(row0 + lane, P.M - 1);
        const float nl = -P.row_lse[rr] * LOG2E_F;
        int tg = P.row_tgt[rr];
        if (tg < 0 || tg >= P.vocab) tg = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int c = col0 + 2 * i;
            float d0 = c < P.vocab ? ex2_hw(fmaf(f2_lo(x[i]), LOG2E_F, nl)) : 0.f;
            float d1 = c + 1 < P.vocab ? ex2_hw(fmaf(f2_hi(x[i]), LOG2E_F, nl)) : 0.f;
            if (c == tg) d0 -= 1.f;
            if (c + 1 == tg) d1 -= 1.f;
            x[i] = f2(d0 * P.dz_scale, d1 * P.dz_scale);
        }
    }
    // the output staging block is free once the TMA store that last used it has read it
    if (lane == 0) {
        if (stage2)
            bulk_wait_read<1>();  // the GELU output's store (other block) may still be reading
        else
            bulk_wait_read<0>();
    }
    __syncwarp();
    if (P.epi == GPT2_EPI_RESIDUAL || P.epi == GPT2_EPI_GELU_BWD) {
        uint8_t *rs = rstage;
        if (rs) {
            cp_async_wait_all();
        } else {
            rs = stage;
            stage_load(rs, P.R, P.ldd, row0, col0, P.M, P.N, lane);
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 v = *stage_at(rs, lane, c);
            const uint32_t rw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const F2 r = f2(bf16_lo(rw[k]), bf16_hi(rw[k]));
                x[4 * c + k] = P.epi == GPT2_EPI_RESIDUAL ? f2_add(x[4 * c + k], r) : f2_mul(x[4 * c + k], gelu_tanh_grad2(r));
            }
        }
        __syncwarp();
    }
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(f2_lo(x[i]), f2_hi(x[i]));
#pragma unroll
    for (int c = 0; c < 8; ++c) *stage_at(stage, lane, c) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tmD, stage, col0, row0);
        bulk_commit();
    }
    if (P.dbias) {
        // column sums of the stored (rounded) block: lane l reads columns 2l, 2l + 1 of each
        // of the warp's rows (rows at or past M excluded) and adds them to the bias gradient
        F2 cs = f2(0.f, 0.f);
        const int nrows = min(32, P.M - row0);
#pragma unroll 4
        for (int r = 0; r < nrows; ++r) {
            const uint32_t wv = *reinterpret_cast<const uint32_t *>(
                stage + r * 128 + ((((lane >> 2) ^ (r & 7)) << 4) | ((lane & 3) << 2)));
            cs = f2_add(cs, f2(bf16_lo(wv), bf16_hi(wv)));
        }
        const int c = col0 + 2 * lane;
        if (c < P.N)
            asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(P.dbias + c), "f"(f2_lo(cs)), "f"(f2_hi(cs))
                         : "memory");
    }
    if (P.epi == GPT2_EPI_GELU) {
        // GELU of the bf16-rounded pre-activation (a recompute from stored h matches bit for bit)
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const F2 y = gelu_tanh2(f2(bf16_lo(w[i]), bf16_hi(w[i])));
            w[i] = pack_bf16x2(f2_lo(y), f2_hi(y));
        }
        uint8_t *g2 = stage2 ? stage2 : stage;
        if (lane == 0) {
            if (stage2)
                bulk_wait_read<1>();  // the previous GELU store from stage2 has read it
            else
                bulk_wait_read<0>();  // the store just issued from `stage` has read it
        }
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *stage_at(g2, lane, c) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmD2, g2, col0, row0);
            bulk_commit();
        }
    }
}

// ---- the kernel -----------------------------------------------------------------
// PAIR: launched as clusters of two CTAs sharing 256 x BN tiles; the even CTA
// issues the cta_group::2 MMAs for both, each CTA loads its own 128 rows of A
// and BN / 2 rows of B (completions counted on the even CTA's barriers) and
// runs the epilogue of its own 128 rows.
// F8: E4M3 operands (K-major only); a k-block is then 128 elements (the same
// 128-byte rows), and the MMAs are kind::f8f6f4.
template <int BN, int STAGES, bool A_MN, bool B_MN, bool PAIR = false, bool F8 = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD2,
                   const __grid_constant__ GroupMaps gm, const Params P) {
    using Lay = SmemLayout<BN, STAGES, PAIR>;
    static_assert(!F8 || (!A_MN && !B_MN), "E4M3 operands are K-major");
    constexpr uint32_t IDESC = PAIR ? instr_desc_pair(BN, A_MN, B_MN, F8) : instr_desc(BN, A_MN, B_MN, F8);
    constexpr int BK_E = F8 ? 2 * BK : BK;  // elements of K per 128-byte k-block row
    constexpr uint32_t TMEM_COLS = 2 * BN;
    constexpr int TM = PAIR ? 2 * BM : BM;        // rows of a tile
    constexpr int BN_CTA = PAIR ? BN / 2 : BN;    // rows of B this CTA loads per stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_smem_1024(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::BAR_OFFSET);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = PAIR ? cluster_rank() : 0;               // CTA within the pair
    const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;  // first work unit
    const int ustep = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;    // units run concurrently
    const int row_off = PAIR ? (int)rank * BM : 0;                 // this CTA's rows within a tile
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], PAIR ? 2 * EPI_WARPS : EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if (P.epi != EPI_LSE) tma_prefetch_desc(&tmD);
        if (P.epi == GPT2_EPI_GELU) tma_prefetch_desc(&tmD2);
        if (P.ngroups > 1) {
            tma_prefetch_desc(&gm.a);
            tma_prefetch_desc(&gm.b);
            tma_prefetch_desc(&gm.d);
        }
    }
    if (warp == 1) {
        if constexpr (PAIR) {  // one warp of each CTA of the pair allocates collectively
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            tmem_alloc(tmem_slot, TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the even CTA's barriers exist before the odd CTA's copies signal them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_work = P.num_work;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;
            bool ok = true;
            for (int w = unit0; w < num_work && ok; w += ustep) {
                const UnitView u = unit_view(P, w);
                const int m0 = u.tm * TM + row_off, n0 = u.tn * BN + (PAIR ? (int)rank * BN_CTA : 0);
                const int kb0 = u.kb0, kb1 = u.kb1;
                const CUtensorMap *ta = u.second ? &gm.a : &tmA, *tb = u.second ? &gm.b : &tmB;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    uint8_t *a_dst = smem + stage * Lay::STAGE_BYTES;
                    uint8_t *b_dst = a_dst + A_STAGE_BYTES;
                    const int k0 = kb * BK_E;
                    if constexpr (PAIR) {
                        // both CTAs' bytes are counted on the even CTA's barrier, which it arms
                        if (rank == 0) mbar_expect_tx(&full[stage], 2 * Lay::STAGE_BYTES);
                        const uint32_t fb = smem_in_rank(&full[stage], 0);
                        if (!A_MN) {
                            tma_load_2d_pair(a_dst, ta, fb, k0, m0);
                        } else {
                            tma_load_2d_pair(a_dst, ta, fb, m0, k0);
                            tma_load_2d_pair(a_dst + MN_BLOCK_BYTES, ta, fb, m0 + 64, k0);
                        }
                        if (!B_MN) {
                            tma_load_2d_pair(b_dst, tb, fb, k0, n0);
                        } else {
#pragma unroll
                            for (int i = 0; i < BN_CTA / 64; ++i)
                                tma_load_2d_pair(b_dst + i * MN_BLOCK_BYTES, tb, fb, n0 + 64 * i, k0);
                        }
                    } else {
                        mbar_expect_tx(&full[stage], Lay::STAGE_BYTES);
                        if (!A_MN) {
                            tma_load_2d(a_dst, ta, &full[stage], k0, m0);
                        } else {
                            tma_load_2d(a_dst, ta, &full[stage], m0, k0);
                            tma_load_2d(a_dst + MN_BLOCK_BYTES, ta, &full[stage], m0 + 64, k0);
                        }
                        if (!B_MN) {
                            tma_load_2d(b_dst, tb, &full[stage], k0, n0);
                        } else {
#pragma unroll
                            for (int i = 0; i < BN / 64; ++i)
                                tma_load_2d(b_dst + i * MN_BLOCK_BYTES, tb, &full[stage], n0 + 64 * i, k0);
                        }
                    }
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok && rank == 0) {  // abort: let the copies already issued land before the CTA exits
                for (int s = 0; s < STAGES; ++s)
                    if (issued_mask & (1u << s)) mbar_drain(&full[s], (issued_phase >> s) & 1);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (the even CTA of a pair issues for both) ----------------
            int stage = 0;
            uint32_t phase = 0;
            int t = 0;
            bool ok = true;
            for (int w = unit0; w < num_work && ok; w += ustep, ++t) {
                const UnitView u = unit_view(P, w);
                const int kb0 = u.kb0, kb1 = u.kb1;
                const int acc = t & 1;
                const uint32_t aph = (t >> 1) & 1;
                if (!mbar_wait(&tempty[acc], aph ^ 1, abort_flag, P.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, P.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + stage * Lay::STAGE_BYTES);
                    const uint32_t b_addr = a_addr + A_STAGE_BYTES;
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j) {
                        const uint64_t ad = A_MN ? smem_desc(a_addr + j * 2048, MN_BLOCK_BYTES, 1024)
                                                 : smem_desc(a_addr + j * 32, 16, 1024);
                        const uint64_t bd = B_MN ? smem_desc(b_addr + j * 2048, MN_BLOCK_BYTES, 1024)
                                                 : smem_desc(b_addr + j * 32, 16, 1024);
                        const uint32_t accum = (kb > kb0 || j > 0) ? 1u : 0u;
                        if constexpr (PAIR && F8)
                            tc_mma_pair_f8(d_tmem, ad, bd, IDESC, accum);
                        else if constexpr (PAIR)
                            tc_mma_pair(d_tmem, ad, bd, IDESC, accum);
                        else if constexpr (F8)
                            tc_mma_f8(d_tmem, ad, bd, IDESC, accum);
                        else
                            tc_mma(d_tmem, ad, bd, IDESC, accum);
                    }
                    if constexpr (PAIR)
                        tc_commit_pair(&empty[stage], 3);
                    else
                        tc_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                if constexpr (PAIR)
                    tc_commit_pair(&tfull[acc], 3);
                else
                    tc_commit(&tfull[acc]);
            }
            // all MMAs issued by this thread have completed once `drain` flips
            if constexpr (PAIR)
                tc_commit_pair(drain, 1);
            else
                tc_commit(drain);
            mbar_drain(drain, 0);
        }
    } else {
        // ---------------- epilogue (warps 2..9) ----------------
        const int quad = warp & 3;                        // TMEM lanes this warp may access
        const int col_half = (warp - 2) >> 2;             // which half of the tile's columns
        uint8_t *stage = smem + Lay::EPI_OFFSET + (warp - 2) * Lay::EPI_BUFS * EPI_STAGE_BYTES;
        constexpr int HALF = BN / 2;
        if (Lay::EPI_BUFS > 1 && (P.epi == GPT2_EPI_RESIDUAL || P.epi == GPT2_EPI_GELU_BWD) &&
            unit0 < num_work) {
            const int t0 = unit0 / P.splits;
            const int ncol = tile_n(P, t0) * BN + col_half * HALF;
            if (ncol < P.N)
                stage_prefetch(stage + EPI_STAGE_BYTES, P.R, P.ldd, tile_m(P, t0) * TM + row_off + quad * 32, ncol, P.M, P.N,
                               lane);
        }
        int t = 0;
        for (int w = unit0; w < num_work; w += ustep, ++t) {
            const UnitView u = unit_view(P, w);
            const int m0 = u.tm * TM + row_off, n0 = u.tn * BN;
            const int Nu = u.second ? P.g2_N : P.N;  // the product's N (grouped launches: fp32 accumulate only)
            const int acc = t & 1;
            const uint32_t aph = (t >> 1) & 1;
            if (!mbar_wait(&tfull[acc], aph, abort_flag, P.err)) break;
            tc_fence_after();
            const int row = m0 + quad * 32 + lane;
            const int c_begin = col_half * HALF;
            const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * BN + c_begin);
            if constexpr (HALF >= 64) {
                if (P.epi == EPI_LSE) {  // cross-entropy partials of the row over this half tile; no output
                    float lm = -INFINITY, ls = 0.f;
#pragma unroll 1
                    for (int c0 = 0; c0 < HALF; c0 += 64) {
                        uint32_t r0[32], r1[32];
                        tmem_ld32(tbase + c0, r0);
                        tmem_ld32(tbase + c0 + 32, r1);
                        tmem_ld_wait();
                        if (c0 + 64 == HALF) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) {
                                if constexpr (PAIR)
                                    release_accumulator(&tempty[acc], rank);
                                else
                                    mbar_arrive(&tempty[acc]);
                            }
                        }
                        lse_group(P, row, n0 + c_begin + c0, r0, r1, lm, ls);
                    }
                    if (row < P.M) P.row_part[(int64_t)row * P.part_stride + 2 * (n0 / BN) + col_half] = make_float2(lm, ls);
                    continue;
                }
                const bool need_r = P.epi == GPT2_EPI_RESIDUAL || P.epi == GPT2_EPI_GELU_BWD;
                uint8_t *rstage = (Lay::EPI_BUFS > 1 && need_r) ? stage + EPI_STAGE_BYTES : nullptr;
                uint8_t *gstage = (Lay::EPI_BUFS > 1 && P.epi == GPT2_EPI_GELU) ? stage + EPI_STAGE_BYTES : nullptr;
                const int row0 = m0 + quad * 32;
#pragma unroll 1
                for (int c0 = 0; c0 < HALF; c0 += 64) {
                    const int col = n0 + c_begin + c0;
                    uint32_t r0[32], r1[32];
                    tmem_ld32(tbase + c0, r0);
                    tmem_ld32(tbase + c0 + 32, r1);
                    tmem_ld_wait();
                    if (c0 + 64 == HALF) {  // this warp's part of the accumulator is read: release it
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (PAIR)
                                release_accumulator(&tempty[acc], rank);
                            else
                                mbar_arrive(&tempty[acc]);
                        }
                    }
                    if (P.epi == GPT2_EPI_ACCUM_F32) {
                        const CUtensorMap *td = u.second ? &gm.d : &tmD;
                        if (col < Nu) reduce_block32(P, td, stage, row0, col, lane, r0);
                        if (col + 32 < Nu) reduce_block32(P, td, stage, row0, col + 32, lane, r1);
                    } else if (col < P.N) {
                        epilogue_group64(P, &tmD, &tmD2, stage, gstage, rstage, row0, col, lane, r0, r1);
                    }
                    // fetch the operand block of the next group (this tile or the next one)
                    if (rstage) {
                        __syncwarp();
                        int nrow0 = row0, ncol = col + 64;
                        if (c0 + 64 == HALF) {
                            const int wn = w + ustep;
                            if (wn < num_work) {
                                const int tn = wn / P.splits;
                                nrow0 = tile_m(P, tn) * TM + row_off + quad * 32;
                                ncol = tile_n(P, tn) * BN + c_begin;
                            } else {
                                ncol = P.N;  // nothing left: no fetch
                            }
                        }
                        if (ncol < P.N) stage_prefetch(rstage, P.R, P.ldd, nrow0, ncol, P.M, P.N, lane);
                    }
                }
            } else {
                uint32_t r0[32];
                tmem_ld32(tbase, r0);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        release_accumulator(&tempty[acc], rank);
                    else
                        mbar_arrive(&tempty[acc]);
                }
                const int col = n0 + c_begin;
                if (col < P.N) epilogue_chunk(P, row, col, r0);
            }
        }
    }
    if (warp >= 2 && lane == 0) bulk_wait_all();  // the epilogue's TMA stores have completed
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();  // the pair's MMAs and both epilogues are done with TMEM
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS)
                         : "memory");
        else
            tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---- host side ---------------------------------------------------------------------
int encode_tmap(CUtensorMap *tm, const void *ptr, uint64_t inner, uint64_t outer, uint64_t ld_elems, uint32_t box_inner,
                uint32_t box_outer);

struct GemmDesc {
    const bf16 *A = nullptr;
    int64_t lda = 0;
    bool a_kmajor = true;
    const bf16 *B = nullptr;
    int64_t ldb = 0;
    bool b_kmajor = true;
    void *D = nullptr;
    bf16 *D2 = nullptr;
    const bf16 *R = nullptr;
    int64_t ldd = 0;
    const float *bias = nullptr;
    int M = 0, N = 0, K = 0;
    int epi = GPT2_EPI_STORE;
    float alpha = 1.0f;  // acc is scaled by alpha before the epilogue
    int *err = nullptr;
    float *dbias = nullptr;  // bf16 epilogues: += column sums of the stored output (8-aligned fp32)
    // E4M3 operands (A and B K-major, bytes; lda / ldb multiples of 16): acc is
    // scaled by alpha * a_scale[row] (if given) * b_scale[0] (if given)
    bool fp8 = false;
    const float *a_scale = nullptr;
    const float *b_scale = nullptr;
    // EPI_LSE / EPI_DZ: vocabulary size, targets, per-row lse (EPI_DZ), partials and
    // target logits (EPI_LSE, part_stride >= 2 * ceil(N / 256) float2 per row), dz factor
    int vocab = 0, part_stride = 0;
    const int *row_tgt = nullptr;
    const float *row_lse = nullptr;
    float2 *row_part = nullptr;
    float *row_zt = nullptr;
    float dz_scale = 1.0f;
};

int launch_gemm_tc(const GemmDesc &g, int num_sms, cudaStream_t stream);

// Two fp32-accumulate products (both operands MN-major, the same K: the weight
// gradients of one block) in one persistent launch, their tiles sharing the
// waves and one prologue and drain; other pairs of products run as two launches.
int launch_gemm_tc_grouped(const GemmDesc &g0, const GemmDesc &g1, int num_sms, cudaStream_t stream);

}  // namespace tcg
