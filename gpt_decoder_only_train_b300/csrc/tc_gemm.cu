// Host side of the tcgen05 GEMM: tensor maps, tile/split choice, dispatch.
#include <algorithm>

#include "tc_gemm.cuh"

namespace tcg {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 2-D tensor map with 128-byte swizzle (bf16, or bytes for E4M3); OOB elements read as zero.
static int encode_tmap_t(CUtensorMap *tm, CUtensorMapDataType dt, uint32_t esize, const void *ptr, uint64_t inner,
                         uint64_t outer, uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return GPT2_ERR_CUDA;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld_elems * esize};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GPT2_OK : GPT2_ERR_CUDA;
}
int encode_tmap(CUtensorMap *tm, const void *ptr, uint64_t inner, uint64_t outer, uint64_t ld_elems, uint32_t box_inner,
                uint32_t box_outer) {
    return encode_tmap_t(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, inner, outer, ld_elems, box_inner, box_outer);
}

// Everything a launch passes to the kernel.  P.num_work work units (tiles x
// splits, of one or two products); the grid is one CTA per SM (or one pair of
// CTAs per two SMs) up to that count.
struct LaunchArgs {
    CUtensorMap ta, tb, td, td2;
    GroupMaps gm;
    Params P;
};

template <int BN, int STAGES, bool A_MN, bool B_MN, bool PAIR, bool F8 = false>
static int launch_one(const LaunchArgs &L, int num_sms, cudaStream_t st) {
    const int units = L.P.num_work;
    using Lay = SmemLayout<BN, STAGES, PAIR>;
    auto kern = gemm_tc_kernel<BN, STAGES, A_MN, B_MN, PAIR, F8>;
    static PerDevice attr_pd, pairs_pd;
    int unused = 0;
    if (int rc = per_device(attr_pd, unused, [&](int &v) -> int {
            GPT2_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::TOTAL));
            v = 1;
            return GPT2_OK;
        }))
        return rc;
    if constexpr (PAIR) {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = Lay::TOTAL;
        cfg.stream = st;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int max_pairs = 1;  // how many CTA pairs can be resident at once (about half the SMs)
        if (int rc = per_device(pairs_pd, max_pairs, [&](int &v) -> int {
                cfg.gridDim = dim3(2 * (num_sms / 2));
                int n = 0;
                GPT2_CUDA_TRY(cudaOccupancyMaxActiveClusters(&n, kern, &cfg));
                v = n > 0 ? n : 1;
                return GPT2_OK;
            }))
            return rc;
        cfg.gridDim = dim3(2 * std::min(units, max_pairs));
        GPT2_CUDA_TRY(cudaLaunchKernelEx(&cfg, kern, L.ta, L.tb, L.td, L.td2, L.gm, L.P));
    } else {
        kern<<<std::min(units, num_sms), NUM_THREADS, Lay::TOTAL, st>>>(L.ta, L.tb, L.td, L.td2, L.gm, L.P);
    }
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

template <int BN, int STAGES, bool PAIR>
static int dispatch_major(bool a_mn, bool b_mn, const LaunchArgs &L, int num_sms, cudaStream_t st) {
    if (!a_mn && !b_mn) return launch_one<BN, STAGES, false, false, PAIR>(L, num_sms, st);
    if (!a_mn && b_mn) return launch_one<BN, STAGES, false, true, PAIR>(L, num_sms, st);
    if (a_mn && b_mn) return launch_one<BN, STAGES, true, true, PAIR>(L, num_sms, st);
    return launch_one<BN, STAGES, true, false, PAIR>(L, num_sms, st);
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Argument checks of one product (no device or driver call).
static int check_desc(const GemmDesc &g) {
    if (g.M <= 0 || g.N <= 0 || g.K <= 0) return GPT2_ERR_BAD_SHAPE;
    const bool lse = g.epi == EPI_LSE, dz = g.epi == EPI_DZ;
    if (!g.A || !g.B || (!g.D && !lse)) return GPT2_ERR_BAD_ARG;
    if (lse || dz) {  // the cross-entropy epilogues: bf16 K-major operands, plain products
        if (g.fp8 || !g.a_kmajor || !g.b_kmajor || g.alpha != 1.0f || g.bias || g.dbias || g.N < 128 ||
            g.vocab <= 0 || g.vocab > g.N || !g.row_tgt)
            return GPT2_ERR_UNSUPPORTED;
        if (lse && (!g.row_part || !g.row_zt || g.part_stride < 2 * ceil_div(g.N, g.N >= 256 ? 256 : 128) ||
                    (reinterpret_cast<uintptr_t>(g.row_part) & 7)))
            return GPT2_ERR_BAD_ARG;
        if (dz && !g.row_lse) return GPT2_ERR_BAD_ARG;
    }
    if ((g.lda % 8) || (g.ldb % 8) || (g.ldd % 8) || (g.N % 8)) return GPT2_ERR_BAD_SHAPE;
    if (g.fp8 && (!g.a_kmajor || !g.b_kmajor || g.lda % 16 || g.ldb % 16 || g.N < 128 ||
                  g.epi == GPT2_EPI_ACCUM_F32 || g.epi == GPT2_EPI_GELU_BWD))
        return GPT2_ERR_UNSUPPORTED;  // E4M3: K-major operands, 16-byte rows, bf16 forward epilogues
    if ((g.a_scale && (reinterpret_cast<uintptr_t>(g.a_scale) & 3)) ||
        (g.b_scale && (reinterpret_cast<uintptr_t>(g.b_scale) & 3)))
        return GPT2_ERR_BAD_ARG;
    if (!aligned16(g.A) || !aligned16(g.B) || (!lse && !aligned16(g.D))) return GPT2_ERR_BAD_ARG;
    if ((g.epi < GPT2_EPI_STORE || g.epi > GPT2_EPI_ACCUM_F32) && !lse && !dz) return GPT2_ERR_BAD_ARG;
    if ((g.epi == GPT2_EPI_RESIDUAL || g.epi == GPT2_EPI_GELU_BWD) && (!g.R || !aligned16(g.R)))
        return GPT2_ERR_BAD_ARG;
    if (g.epi == GPT2_EPI_GELU && (!g.D2 || !aligned16(g.D2))) return GPT2_ERR_BAD_ARG;
    if (g.bias && (reinterpret_cast<uintptr_t>(g.bias) & 15)) return GPT2_ERR_BAD_ARG;
    if (g.dbias && (reinterpret_cast<uintptr_t>(g.dbias) & 7)) return GPT2_ERR_BAD_ARG;
    if (g.dbias && g.epi != GPT2_EPI_ACCUM_F32 && g.N <= 64) return GPT2_ERR_UNSUPPORTED;  // staged epilogue only
    return GPT2_OK;
}

// Checks one product and fills L (maps, tile and split choice).  other_tiles: the
// tiles of a second product launched with this one (the split-K choice then
// fills the waves of both together).
static int prepare(const GemmDesc &g, int num_sms, LaunchArgs &L, int &BN_out, bool &pair_out, int other_tiles) {
    if (int rc = check_desc(g)) return rc;
    const bool lse = g.epi == EPI_LSE;
    const int BN = g.N >= 256 ? 256 : (g.N > 64 ? 128 : 64);
    // CTA pairs on 256 x 256 tiles (cta_group::2): each SM reads half of the B
    // tile per stage, which keeps shared-memory traffic per MMA within what the
    // SM delivers, at the cost of pair synchronisation per tile.  Measured on
    // the model's shapes (one build, alternating), pairs pay off everywhere
    // except for short-K products that add a residual (16384 x 768 x 768: equal
    // times), which stay on single CTAs; the last to move were the plain and
    // the weight-gradient 768-wide products (-9% and -7%) and the GELU backward
    // (-3%).
    const bool pair = BN == 256 && (g.epi != GPT2_EPI_RESIDUAL || g.K >= 1024);
    const int conc = pair ? num_sms / 2 : num_sms;  // work units that run at once
    Params &P = L.P;
    P = Params{};
    P.M = g.M;
    P.N = g.N;
    P.K = g.K;
    P.num_m_blocks = ceil_div(g.M, pair ? 2 * BM : BM);
    P.num_n_blocks = ceil_div(g.N, BN);
    P.num_k_blocks = ceil_div(g.K, g.fp8 ? 2 * BK : BK);
    P.splits = 1;
    if (g.epi == GPT2_EPI_ACCUM_F32) {
        // Split K (partial products are added into D) so that the work units
        // fill whole waves of the persistent grid: the smallest split count
        // whose last wave is at least 95% busy, else the best one found.  Each
        // split keeps at least 4 K blocks.
        const int tiles = P.num_m_blocks * P.num_n_blocks + other_tiles;
        if (tiles < 2 * conc) {
            const int max_splits = std::max(1, P.num_k_blocks / 4);
            int best = 1;
            double best_eff = 0.0;
            for (int sp = 1; sp <= max_splits; ++sp) {
                const int kbps = ceil_div(P.num_k_blocks, sp), real = ceil_div(P.num_k_blocks, kbps);
                const long long units = (long long)tiles * real;
                const double eff = (double)units / ((double)ceil_div((int)units, conc) * conc);
                if (eff > best_eff + 1e-9) {
                    best_eff = eff;
                    best = real;
                }
                if (eff >= 0.95) break;
            }
            P.splits = best;
        }
    }
    P.k_blocks_per_split = ceil_div(P.num_k_blocks, P.splits);
    P.splits = ceil_div(P.num_k_blocks, P.k_blocks_per_split);
    // raster: share the A block across concurrent tiles when A is not small next
    // to L2 and B is (with m fastest, A would stream from HBM once per N block:
    // measured 2.3x the A bytes for 100 MB operands and N = 768)
    const double a_bytes = 2.0 * g.M * g.K, b_bytes = 2.0 * g.N * g.K;
    P.n_fastest = (P.num_n_blocks <= 8 && a_bytes > 32e6 && b_bytes < 96e6) ? 1 : 0;
    P.epi = g.epi;
    P.alpha = g.alpha;
    P.bias = g.bias;
    P.dbias = g.epi == GPT2_EPI_ACCUM_F32 ? nullptr : g.dbias;
    P.a_scale = g.a_scale;
    P.b_scale = g.b_scale;
    P.vocab = g.vocab;
    P.part_stride = g.part_stride;
    P.row_tgt = g.row_tgt;
    P.row_lse = g.row_lse;
    P.row_part = g.row_part;
    P.row_zt = g.row_zt;
    P.dz_scale = g.dz_scale;
    P.R = g.R;
    P.D = g.D;
    P.D2 = g.D2;
    P.ldd = g.ldd;
    P.err = g.err;

    CUtensorMap &ta = L.ta, &tb = L.tb;
    int rc;
    if (g.fp8) {  // bytes: 128 E4M3 values per 128-byte k-block row
        rc = encode_tmap_t(&ta, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.A, g.K, g.M, g.lda, 128, BM);
        if (rc) return rc;
        rc = encode_tmap_t(&tb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, g.B, g.K, g.N, g.ldb, 128, pair ? BN / 2 : BN);
        if (rc) return rc;
    } else {
        rc = g.a_kmajor ? encode_tmap(&ta, g.A, g.K, g.M, g.lda, 64, BM) : encode_tmap(&ta, g.A, g.M, g.K, g.lda, 64, 64);
        if (rc) return rc;
        rc = g.b_kmajor ? encode_tmap(&tb, g.B, g.K, g.N, g.ldb, 64, pair ? BN / 2 : BN)
                        : encode_tmap(&tb, g.B, g.N, g.K, g.ldb, 64, 64);
        if (rc) return rc;
    }

    // bf16 outputs leave through TMA stores from the epilogue's staging blocks (box 64 x 32)
    CUtensorMap &td = L.td, &td2 = L.td2;
    td = ta;  // unused copies when the output has no tensor map
    td2 = ta;
    if (g.epi != GPT2_EPI_ACCUM_F32 && !lse && (rc = encode_tmap(&td, g.D, g.N, g.M, g.ldd, 64, 32))) return rc;
    // fp32 outputs are added through TMA reduce-adds of 32 x 32 blocks (BN of 128 and up)
    if (g.epi == GPT2_EPI_ACCUM_F32 && BN >= 128 &&
        (rc = encode_tmap_t(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, g.D, g.N, g.M, g.ldd, 32, 32)))
        return rc;
    if (g.epi == GPT2_EPI_GELU && (rc = encode_tmap(&td2, g.D2, g.N, g.M, g.ldd, 64, 32))) return rc;

    P.num_work = P.num_m_blocks * P.num_n_blocks * P.splits;
    P.ngroups = 1;
    P.work1 = P.num_work;
    L.gm.a = ta;  // unused copies: no second product
    L.gm.b = tb;
    L.gm.d = td;
    BN_out = BN;
    pair_out = pair;
    return GPT2_OK;
}

static int dispatch(const GemmDesc &g, const LaunchArgs &L, int BN, bool pair, int num_sms, cudaStream_t stream) {
    const bool a_mn = !g.a_kmajor, b_mn = !g.b_kmajor;
    const bool reads_r = g.epi == GPT2_EPI_RESIDUAL || g.epi == GPT2_EPI_GELU_BWD;
    // epilogues with a second staging block per warp (the prefetched operand, or the GELU
    // output) trade a ring stage for it; the model uses them with K-major A only
    const bool two_bufs = (reads_r || g.epi == GPT2_EPI_GELU) && !a_mn;
    if (g.fp8) {  // E4M3 operands: K-major, BN 256 (pairs or single CTAs) or 128
        if (BN == 256 && pair)
            return two_bufs ? launch_one<256, 5, false, false, true, true>(L, num_sms, stream)
                            : launch_one<256, 6, false, false, true, true>(L, num_sms, stream);
        if (BN == 256)
            return two_bufs ? launch_one<256, 3, false, false, false, true>(L, num_sms, stream)
                            : launch_one<256, 4, false, false, false, true>(L, num_sms, stream);
        return launch_one<128, 6, false, false, false, true>(L, num_sms, stream);
    }
    if (BN == 256 && pair) {
        if (two_bufs)
            return b_mn ? launch_one<256, 5, false, true, true>(L, num_sms, stream)
                        : launch_one<256, 5, false, false, true>(L, num_sms, stream);
        return dispatch_major<256, 6, true>(a_mn, b_mn, L, num_sms, stream);
    }
    if (BN == 256) {
        if (two_bufs)
            return b_mn ? launch_one<256, 3, false, true, false>(L, num_sms, stream)
                        : launch_one<256, 3, false, false, false>(L, num_sms, stream);
        return dispatch_major<256, 4, false>(a_mn, b_mn, L, num_sms, stream);
    }
    if (BN == 128) return dispatch_major<128, 6, false>(a_mn, b_mn, L, num_sms, stream);
    return dispatch_major<64, 8, false>(a_mn, b_mn, L, num_sms, stream);
}

int launch_gemm_tc(const GemmDesc &g, int num_sms, cudaStream_t stream) {
    LaunchArgs L;
    int BN = 0;
    bool pair = false;
    if (int rc = prepare(g, num_sms, L, BN, pair, 0)) return rc;
    return dispatch(g, L, BN, pair, num_sms, stream);
}

int launch_gemm_tc_grouped(const GemmDesc &g0, const GemmDesc &g1, int num_sms, cudaStream_t stream) {
    // fp32-accumulate products on CTA pairs with both operands MN-major and the same K
    // (the weight gradients of one block); anything else runs as two launches.  Both
    // products are checked before either is launched.
    const auto groupable = [](const GemmDesc &g) {
        return g.epi == GPT2_EPI_ACCUM_F32 && !g.fp8 && !g.a_kmajor && !g.b_kmajor && !g.a_scale && !g.b_scale &&
               !g.bias && !g.dbias && g.N >= 256;
    };
    const bool grouped = groupable(g0) && groupable(g1) && g0.K == g1.K && g0.alpha == g1.alpha;
    const int tiles0 = grouped ? ceil_div(g0.M, 2 * BM) * ceil_div(g0.N, 256) : 0,
              tiles1 = grouped ? ceil_div(g1.M, 2 * BM) * ceil_div(g1.N, 256) : 0;
    if (int rc = check_desc(g0)) return rc;
    if (int rc = check_desc(g1)) return rc;
    LaunchArgs L, L1;
    int BN0 = 0, BN1 = 0;
    bool pair0 = false, pair1 = false;
    if (int rc = prepare(g0, num_sms, L, BN0, pair0, tiles1)) return rc;
    if (int rc = prepare(g1, num_sms, L1, BN1, pair1, tiles0)) return rc;
    if (!grouped) {
        if (int rc = dispatch(g0, L, BN0, pair0, num_sms, stream)) return rc;
        return dispatch(g1, L1, BN1, pair1, num_sms, stream);
    }
    Params &P = L.P;
    const Params &Q = L1.P;
    if (BN0 != 256 || BN1 != 256 || !pair0 || !pair1 || P.splits != Q.splits ||
        P.k_blocks_per_split != Q.k_blocks_per_split || P.num_m_blocks * P.num_n_blocks != tiles0 ||
        Q.num_m_blocks * Q.num_n_blocks != tiles1)
        return GPT2_ERR_UNSUPPORTED;  // the two choices agree by construction
    P.ngroups = 2;
    P.work1 = tiles0 * P.splits;
    P.num_work = (tiles0 + tiles1) * P.splits;
    P.g2_M = Q.M;
    P.g2_N = Q.N;
    P.g2_num_m_blocks = Q.num_m_blocks;
    P.g2_num_n_blocks = Q.num_n_blocks;
    P.g2_n_fastest = Q.n_fastest;
    L.gm.a = L1.ta;
    L.gm.b = L1.tb;
    L.gm.d = L1.td;
    return launch_one<256, 6, true, true, true>(L, num_sms, stream);
}

}  // namespace tcg
