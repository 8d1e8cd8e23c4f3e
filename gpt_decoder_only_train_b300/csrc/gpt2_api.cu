// C ABI of the GPT-2 training step: arena planning, host initialisation,
// and the launch sequence of forward, backward and the optimizer.
//
// The step follows "Let's reproduce GPT-2 (124M)" (§Bölümler 2: the GPT-2
// module; §Bölümler 4: cross-entropy; §Video özeti: AdamW, gradient
// accumulation, mixed precision) and "llm.c kullanarak GPT-2 modelini düşük
// maliyetle yeniden uygulamak" (§Eğitimi çalıştırma: -b/-t/-d/-r; §Eğitim
// süreci: gradient clipping).  Block order is pre-LN:
//   x1 = x + proj(attn(ln1(x)));  x' = x1 + fcproj(gelu(fc(ln2(x1))))
// with a final LayerNorm and an LM head tied to wte.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <string>
#include <thread>
#include <vector>

#include "flash_attn.cuh"
#include "kernels.cuh"
#include "tc_gemm.cuh"

// ------------------------------------------------------------------ errors
static thread_local char g_last_error[256] = "";

void gpt2_set_last_cuda_error(cudaError_t e, const char *what, int line) {
    snprintf(g_last_error, sizeof(g_last_error), "%s (%s) at gpt2_api line %d: %s", cudaGetErrorName(e),
             cudaGetErrorString(e), line, what);
}

extern "C" const char *gpt2_last_error_detail(void) { return g_last_error; }

static std::atomic<long long> g_launches{0};

// time limit of the clip + AdamW grid barrier, and the test hook that makes it unreachable
constexpr unsigned long long kDefaultBarrierWaitNs = 2000000000ull;
static std::atomic<unsigned long long> g_barrier_wait_ns{kDefaultBarrierWaitNs};
static std::atomic<unsigned> g_barrier_extra{0};
void gpt2_note_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
extern "C" long long gpt2_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" const char *gpt2_strerror(int s) {
    switch (s) {
        case GPT2_OK: return "ok";
        case GPT2_ERR_BAD_CONFIG: return "bad config";
        case GPT2_ERR_BAD_SHAPE: return "bad shape";
        case GPT2_ERR_BAD_TOKEN: return "token or target out of range";
        case GPT2_ERR_ARENA_TOO_SMALL: return "arena too small";
        case GPT2_ERR_CUDA: return "CUDA error";
        case GPT2_ERR_NONFINITE: return "non-finite loss or gradient norm";
        case GPT2_ERR_TIMEOUT: return "bounded device wait timed out";
        case GPT2_ERR_BAD_ARG: return "bad argument";
        case GPT2_ERR_UNSUPPORTED: return "unsupported device or feature";
        case GPT2_ERR_STATE: return "call order violated";
        default: return "unknown status";
    }
}

// ------------------------------------------------------------------ model
struct TensorInfo {
    std::string name;
    int ndim;
    int64_t shape[2];
    int64_t numel;
    int64_t offset;  // elements into the flat parameter arena
    bool decay;      // 2-D weight: receives weight decay
    int kind;        // 0 zeros, 1 ones, 2 normal (all rows), 3 normal (first V rows)
    double std;
};

struct LayerBuf {
    void *resid, *ln1, *qkv, *att, *resid_mid, *ln2, *fch, *fcg;
    float *ln1_mean, *ln1_rstd, *ln2_mean, *ln2_rstd, *lse;
};

struct LayerParams {
    int ln1g, ln1b, qkvw, qkvb, projw, projb, ln2g, ln2b, fcw, fcb, fcprojw, fcprojb;  // tensor ids
};

struct gpt2_model {
    gpt2_config cfg;
    cudaStream_t stream;
    uint8_t *arena;
    size_t arena_bytes;
    int num_sms;
    std::vector<TensorInfo> tensors;
    std::vector<LayerParams> lp;
    int64_t n_params, n_decay;
    float *params, *grads, *adam_m, *adam_v;
    bf16 *wbf;  // bf16 copy of the weights (bf16 mode)
    // E4M3 forward (fp8_forward): codes of the four projection weights of every
    // block (same offsets as the parameters), one dequantisation factor per
    // tensor, and one activation code buffer [B*T, 4C] with its row factors
    uint8_t *w8, *a8;
    float *w8_inv, *a8_inv;
    unsigned *w8_amax;
    int64_t *w8_off, *w8_n;  // device tables over the quantised tensors
    std::vector<int> w8_ids;  // tensor ids of the quantised tensors, in table order
    int64_t w8_maxn;
    // fused LM head (fused_lm_head): cross-entropy partials [B*T, ce_stride], target logits
    // and lse [B*T]; the logits buffer holds lm_rows rows (a chunk of the backward)
    float2 *ce_part;
    float *ce_zt, *ce_lse;
    int ce_stride, lm_rows;
    std::vector<LayerBuf> layers;
    void *resid_final, *lnf;
    float *lnf_mean, *lnf_rstd;
    void *logits;
    float *loss_rows, *loss_dev, *norm_dev;
    int *tokens, *targets;
    void *dres, *dbig, *dqkv, *datt, *dsmall, *gelu_buf;
    float *attn_D;
    void *attn_ds;  // attention backward: dS^T of the causal blocks (bf16 path, up to kMaxAttnDsBytes)
    void *emb_ws;  // embedding backward: sorted keys and partial sums
    double *norm_partials;
    unsigned *barrier;
    int *err_dev;
    int *gen_pos;  // device position counter of gpt2_generate
    int max_adam_blocks;
    int fwd_B, fwd_T;
    bool have_dlogits;
    int adam_t;
    // optional per-launch timing (gpt2_profile): event pairs recorded around launches
    struct Rec {
        cudaEvent_t a, b;
        int cat;
        double work;
        long long kernels;  // kernels the recorded call launched
    };
    std::vector<Rec> prof;
    size_t prof_used = 0;
    bool prof_on = false;
    // CUDA graphs of the forward and backward launch sequences, keyed by shape
    // (and, for the backward, the loss weight): replayed on the model's stream
    struct Graph {
        int kind, B, T;
        uint32_t key;
        cudaGraphExec_t exec;
        long long kernels;
        int uses;  // calls seen for this key; the first runs direct, the second captures
    };
    std::vector<Graph> graphs;
    bool graphs_on = true;
    double prof_ms[GPT2_PROF_NCAT] = {}, prof_work[GPT2_PROF_NCAT] = {};
    long long prof_n[GPT2_PROF_NCAT] = {};
};

// ------------------------------------------------------------------ layout
namespace {

struct Bump {
    uint8_t *base;
    size_t off = 0;
    template <typename P> P *take(size_t bytes) {
        off = (off + 255) & ~size_t(255);
        P *p = reinterpret_cast<P *>(base + off);
        off += bytes;
        return p;
    }
};

bool valid_config(const gpt2_config &c) {
    if (c.L <= 0 || c.C <= 0 || c.H <= 0 || c.V <= 0 || c.Vp < c.V || c.T <= 0 || c.B <= 0) return false;
    if (c.C % c.H) return false;
    if (c.dtype != GPT2_DTYPE_FP32 && c.dtype != GPT2_DTYPE_BF16) return false;
    if (c.fp8_forward != 0 && c.fp8_forward != 1) return false;
    if (c.fp8_forward && (c.dtype != GPT2_DTYPE_BF16 || c.C < 128)) return false;
    if (c.fused_lm_head != 0 && c.fused_lm_head != 1) return false;
    if (c.fused_lm_head && (c.dtype != GPT2_DTYPE_BF16 || c.Vp < 128)) return false;
    const int hd = c.C / c.H;
    if (c.dtype == GPT2_DTYPE_FP32) {
        if (c.C % 4 || c.Vp % 4 || (hd != 8 && hd != 16 && hd != 32 && hd != 64)) return false;
        if (c.C > 1024) return false;
    } else {
        if (hd != 64 || c.C % 64 || c.Vp % 64 || c.C > 2048) return false;
    }
    return true;
}

void make_tensors(const gpt2_config &c, std::vector<TensorInfo> &ts, std::vector<LayerParams> &lp, int64_t &n_params,
                  int64_t &n_decay) {
    ts.clear();
    lp.assign(c.L, LayerParams{});
    const double std = 0.02, rstd = 0.02 / sqrt(2.0 * c.L);
    auto add = [&](const std::string &name, int64_t r, int64_t cols, int kind, double s, bool decay) {
        TensorInfo t;
        t.name = name;
        t.ndim = cols ? 2 : 1;
        t.shape[0] = r;
        t.shape[1] = cols;
        t.numel = cols ? r * cols : r;
        t.decay = decay;
        t.kind = kind;
        t.std = s;
        t.offset = -1;
        ts.push_back(t);
        return (int)ts.size() - 1;
    };
    add("wte", c.Vp, c.C, 3, std, true);
    add("wpe", c.T, c.C, 2, std, true);
    for (int l = 0; l < c.L; ++l) {
        const std::string p = "h" + std::to_string(l) + ".";
        LayerParams &q = lp[l];
        q.ln1g = add(p + "ln1.g", c.C, 0, 1, 0, false);
        q.ln1b = add(p + "ln1.b", c.C, 0, 0, 0, false);
        q.qkvw = add(p + "qkv.w", 3 * c.C, c.C, 2, std, true);
        q.qkvb = add(p + "qkv.b", 3 * c.C, 0, 0, 0, false);
        q.projw = add(p + "proj.w", c.C, c.C, 2, rstd, true);
        q.projb = add(p + "proj.b", c.C, 0, 0, 0, false);
        q.ln2g = add(p + "ln2.g", c.C, 0, 1, 0, false);
        q.ln2b = add(p + "ln2.b", c.C, 0, 0, 0, false);
        q.fcw = add(p + "fc.w", 4 * c.C, c.C, 2, std, true);
        q.fcb = add(p + "fc.b", 4 * c.C, 0, 0, 0, false);
        q.fcprojw = add(p + "fcproj.w", c.C, 4 * c.C, 2, rstd, true);
        q.fcprojb = add(p + "fcproj.b", c.C, 0, 0, 0, false);
    }
    add("lnf.g", c.C, 0, 1, 0, false);
    add("lnf.b", c.C, 0, 0, 0, false);
    // physical order: all decayed (2-D) tensors first, each padded to 64 elements
    int64_t off = 0;
    for (int pass = 0; pass < 2; ++pass) {
        for (auto &t : ts) {
            if (t.decay != (pass == 0)) continue;
            t.offset = off;
            off += (t.numel + 63) / 64 * 64;
        }
        if (pass == 0) n_decay = off;
    }
    n_params = off;
}

template <typename P> P *take_opt(Bump &b, bool on, size_t bytes) { return on ? b.take<P>(bytes) : nullptr; }

constexpr int64_t kLmChunkRows = 8192;  // positions per chunk of the fused LM head's backward
// Largest stored-dS workspace of the attention backward the model keeps (B H T^2 bf16:
// 0.4 GB at B=16, T=1024, H=12; 6.4 GB at T=4096); past it the backward recomputes S
// and dP for dQ instead of growing the arena with T^2.
constexpr size_t kMaxAttnDsBytes = size_t(16) << 30;

void plan(gpt2_model &m, uint8_t *base) {
    const gpt2_config &c = m.cfg;
    const bool bf = c.dtype == GPT2_DTYPE_BF16;
    const size_t es = bf ? 2 : 4;
    const int64_t BT = (int64_t)c.B * c.T, C = c.C;
    Bump b{base};
    m.params = b.take<float>(m.n_params * 4);
    m.grads = b.take<float>(m.n_params * 4);
    m.adam_m = b.take<float>(m.n_params * 4);
    m.adam_v = b.take<float>(m.n_params * 4);
    m.wbf = take_opt<bf16>(b, bf, m.n_params * 2);
    const bool f8 = c.fp8_forward != 0;
    const size_t nq = f8 ? (size_t)4 * c.L : 0;
    m.w8 = take_opt<uint8_t>(b, f8, m.n_params);
    m.a8 = take_opt<uint8_t>(b, f8, BT * 4 * C);
    m.a8_inv = take_opt<float>(b, f8, BT * 4);
    m.w8_inv = take_opt<float>(b, f8, nq * 4);
    m.w8_amax = take_opt<unsigned>(b, f8, nq * 4);
    m.w8_off = take_opt<int64_t>(b, f8, nq * 8);
    m.w8_n = take_opt<int64_t>(b, f8, nq * 8);
    m.layers.assign(c.L, LayerBuf{});
    for (int l = 0; l < c.L; ++l) {
        LayerBuf &y = m.layers[l];
        y.resid = b.take<void>(BT * C * es);
        y.ln1 = b.take<void>(BT * C * es);
        y.qkv = b.take<void>(BT * 3 * C * es);
        y.att = b.take<void>(BT * C * es);
        y.resid_mid = b.take<void>(BT * C * es);
        y.ln2 = b.take<void>(BT * C * es);
        y.fch = b.take<void>(BT * 4 * C * es);
        y.fcg = take_opt<void>(b, !c.recompute_gelu, BT * 4 * C * es);
        y.ln1_mean = b.take<float>(BT * 4);
        y.ln1_rstd = b.take<float>(BT * 4);
        y.ln2_mean = b.take<float>(BT * 4);
        y.ln2_rstd = b.take<float>(BT * 4);
        y.lse = b.take<float>((int64_t)c.B * c.H * c.T * 4);
    }
    m.resid_final = b.take<void>(BT * C * es);
    m.lnf = b.take<void>(BT * C * es);
    m.lnf_mean = b.take<float>(BT * 4);
    m.lnf_rstd = b.take<float>(BT * 4);
    const bool fl = c.fused_lm_head != 0;
    m.lm_rows = (int)(fl ? std::min<int64_t>(BT, kLmChunkRows) : BT);
    m.logits = b.take<void>((int64_t)m.lm_rows * c.Vp * es);
    m.ce_stride = fl ? 2 * ceil_div(c.Vp, c.Vp >= 256 ? 256 : 128) : 0;
    m.ce_part = take_opt<float2>(b, fl, (size_t)BT * m.ce_stride * 8);
    m.ce_zt = take_opt<float>(b, fl, BT * 4);
    m.ce_lse = take_opt<float>(b, fl, BT * 4);
    m.loss_rows = b.take<float>(BT * 4);
    m.loss_dev = b.take<float>(64);
    m.norm_dev = b.take<float>(64);
    m.tokens = b.take<int>(BT * 4);
    m.targets = b.take<int>(BT * 4);
    m.dres = b.take<void>(BT * C * es);
    m.dbig = b.take<void>(BT * 4 * C * es);
    m.dqkv = b.take<void>(BT * 3 * C * es);
    m.datt = b.take<void>(BT * C * es);
    m.dsmall = b.take<void>(BT * C * es);
    m.gelu_buf = take_opt<void>(b, c.recompute_gelu != 0, BT * 4 * C * es);
    m.attn_D = b.take<float>((int64_t)c.B * c.H * c.T * 4);
    const size_t ds_bytes = fa::attention_backward_ds_bytes(c.B, c.T, c.H);
    m.attn_ds = take_opt<void>(b, c.dtype == GPT2_DTYPE_BF16 && ds_bytes <= kMaxAttnDsBytes, ds_bytes);
    m.emb_ws = b.take<void>(k::embed_backward_workspace((int)BT, c.C));
    m.norm_partials = b.take<double>((size_t)m.max_adam_blocks * 8);
    m.barrier = b.take<unsigned>(64);
    m.err_dev = b.take<int>(64);
    m.gen_pos = b.take<int>(64);
    m.arena_bytes = b.off + 256;
}

// SplitMix64 output for state x (Steele, Lea & Flood, OOPSLA 2014).
inline uint64_t sm64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Fill `n` fp32 values with N(0, std^2): counter draws (seed, id, 2i), (.., 2i+1),
// Box-Muller cosine branch in double, one rounding to fp32.
void fill_normal(uint64_t seed, uint64_t id, int64_t n, double sd, float *out) {
    const uint64_t key = sm64(sm64(seed) + id);
    const int nth = (int)std::max(1u, std::min(32u, std::thread::hardware_concurrency()));
    const int64_t chunk = (n + nth - 1) / nth;
    std::vector<std::thread> th;
    for (int t = 0; t < nth; ++t) {
        th.emplace_back([=]() {
            const int64_t a = t * chunk, e = std::min(n, a + chunk);
            for (int64_t i = a; i < e; ++i) {
                const uint64_t r1 = sm64(key + 2 * (uint64_t)i), r2 = sm64(key + 2 * (uint64_t)i + 1);
                const double u1 = ((double)(r1 >> 11) + 1.0) * (1.0 / 9007199254740992.0);
                const double u2 = (double)(r2 >> 11) * (1.0 / 9007199254740992.0);
                const double z = sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
                out[i] = (float)(sd * z);
            }
        });
    }
    for (auto &x : th) x.join();
}

int check_device(int &num_sms) {
    int dev = 0;
    GPT2_CUDA_TRY(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    GPT2_CUDA_TRY(cudaGetDeviceProperties(&prop, dev));
    num_sms = prop.multiProcessorCount;
    return (prop.major == 10 && prop.minor == 3) ? GPT2_OK : GPT2_ERR_UNSUPPORTED;
}

// ---- per-launch timing ---------------------------------------------------------
int prof_flush(gpt2_model *m) {
    if (!m->prof_used) return GPT2_OK;
    GPT2_CUDA_TRY(cudaStreamSynchronize(m->stream));
    for (size_t i = 0; i < m->prof_used; ++i) {
        float ms = 0.f;
        GPT2_CUDA_TRY(cudaEventElapsedTime(&ms, m->prof[i].a, m->prof[i].b));
        m->prof_ms[m->prof[i].cat] += ms;
        m->prof_work[m->prof[i].cat] += m->prof[i].work;
        m->prof_n[m->prof[i].cat] += m->prof[i].kernels;
    }
    m->prof_used = 0;
    return GPT2_OK;
}

// Record an event pair around `launch()` when profiling is on.
template <typename F> int timed(gpt2_model *m, int cat, double work, F &&launch) {
    if (!m->prof_on) return launch();
    if (m->prof_used == m->prof.size()) {
        if (m->prof.size() < 4096) {
            gpt2_model::Rec r{};
            GPT2_CUDA_TRY(cudaEventCreate(&r.a));
            GPT2_CUDA_TRY(cudaEventCreate(&r.b));
            m->prof.push_back(r);
        } else {
            if (int rc = prof_flush(m)) return rc;
        }
    }
    gpt2_model::Rec &r = m->prof[m->prof_used];
    r.cat = cat;
    r.work = work;
    GPT2_CUDA_TRY(cudaEventRecord(r.a, m->stream));
    const long long n0 = g_launches.load(std::memory_order_relaxed);
    const int rc = launch();
    r.kernels = g_launches.load(std::memory_order_relaxed) - n0;
    GPT2_CUDA_TRY(cudaEventRecord(r.b, m->stream));
    m->prof_used++;
    return rc;
}

// ---- typed helpers -------------------------------------------------------------
template <typename T> T *W(gpt2_model *m, int id);
template <> float *W<float>(gpt2_model *m, int id) { return m->params + m->tensors[id].offset; }
template <> bf16 *W<bf16>(gpt2_model *m, int id) { return m->wbf + m->tensors[id].offset; }
inline float *Pf(gpt2_model *m, int id) { return m->params + m->tensors[id].offset; }
inline float *Gf(gpt2_model *m, int id) { return m->grads + m->tensors[id].offset; }

#define TRY(x)                    \
    do {                          \
        int rc__ = (x);           \
        if (rc__) return rc__;    \
    } while (0)

// launch `expr` (an int-returning launcher call) under the per-launch timer
#define TIMED(cat, work, expr) TRY(timed(m, cat, (double)(work), [&]() -> int { return (expr); }))

// acc[m,n] = sum_k A(m,k) B(n,k) with the majorness conventions of gpt2_op_matmul.
template <typename T>
int mm(gpt2_model *m, const void *A, int64_t lda, bool a_km, const void *B, int64_t ldb, bool b_km, void *D, void *D2,
       const void *R, int64_t ldd, const float *bias, int M, int N, int K, int epi, float alpha = 1.0f,
       float *dbias = nullptr) {
    if constexpr (sizeof(T) == 2) {
        tcg::GemmDesc g;
        g.A = (const bf16 *)A;
        g.lda = lda;
        g.a_kmajor = a_km;
        g.B = (const bf16 *)B;
        g.ldb = ldb;
        g.b_kmajor = b_km;
        g.D = D;
        g.D2 = (bf16 *)D2;
        g.R = (const bf16 *)R;
        g.ldd = ldd;
        g.bias = bias;
        g.M = M;
        g.N = N;
        g.K = K;
        g.epi = epi;
        g.alpha = alpha;
        g.err = m->err_dev;
        g.dbias = dbias;
        return timed(m, GPT2_PROF_MATMUL, 2.0 * M * N * K, [&] { return tcg::launch_gemm_tc(g, m->num_sms, m->stream); });
    } else {
        return timed(m, GPT2_PROF_MATMUL, 2.0 * M * N * K, [&] {
            return k::matmul_simt<float>((const float *)A, a_km ? lda : 1, a_km ? 1 : lda, (const float *)B,
                                         b_km ? ldb : 1, b_km ? 1 : ldb, D, (float *)D2, (const float *)R, ldd, bias,
                                         M, N, K, epi, alpha, m->stream);
        });
    }
}

// Two weight-gradient products D_i += A_i^T B_i (A_i: [K, M_i], B_i: [K, N_i], both
// MN-major, K = B*T rows; D_i fp32 [M_i, N_i]) of one block: one grouped launch in
// bf16 mode, two products otherwise.
struct DwProduct {
    const void *A;
    int64_t lda;
    const void *B;
    int64_t ldb;
    float *D;
    int M, N;
};
template <typename T> int mm_dw2(gpt2_model *m, const DwProduct &x, const DwProduct &y, int K) {
    if constexpr (sizeof(T) == 2) {
        tcg::GemmDesc g[2];
        const DwProduct *d[2] = {&x, &y};
        for (int i = 0; i < 2; ++i) {
            g[i].A = (const bf16 *)d[i]->A;
            g[i].lda = d[i]->lda;
            g[i].a_kmajor = false;
            g[i].B = (const bf16 *)d[i]->B;
            g[i].ldb = d[i]->ldb;
            g[i].b_kmajor = false;
            g[i].D = d[i]->D;
            g[i].ldd = d[i]->N;
            g[i].M = d[i]->M;
            g[i].N = d[i]->N;
            g[i].K = K;
            g[i].epi = GPT2_EPI_ACCUM_F32;
            g[i].err = m->err_dev;
        }
        return timed(m, GPT2_PROF_MATMUL, 2.0 * K * ((double)x.M * x.N + (double)y.M * y.N),
                     [&] { return tcg::launch_gemm_tc_grouped(g[0], g[1], m->num_sms, m->stream); });
    } else {
        TRY(mm<T>(m, x.A, x.lda, false, x.B, x.ldb, false, x.D, nullptr, nullptr, x.N, nullptr, x.M, x.N, K,
                  GPT2_EPI_ACCUM_F32));
        return mm<T>(m, y.A, y.lda, false, y.B, y.ldb, false, y.D, nullptr, nullptr, y.N, nullptr, y.M, y.N, K,
                     GPT2_EPI_ACCUM_F32);
    }
}

// E4M3 product for the forward projections: D = a8_inv[m] w8_inv[slot] (A8 B8^T) + bias, with
// the bf16 epilogue `epi` (both operands K-major byte rows).
int mm8(gpt2_model *m, const uint8_t *A8, int64_t lda, const float *a_inv, int w_id, int slot, void *D, void *D2,
        const void *R, int64_t ldd, const float *bias, int M, int N, int K, int epi) {
    tcg::GemmDesc g;
    g.A = (const bf16 *)A8;
    g.lda = lda;
    g.a_kmajor = true;
    g.B = (const bf16 *)(m->w8 + m->tensors[w_id].offset);
    g.ldb = K;
    g.b_kmajor = true;
    g.D = D;
    g.D2 = (bf16 *)D2;
    g.R = (const bf16 *)R;
    g.ldd = ldd;
    g.bias = bias;
    g.M = M;
    g.N = N;
    g.K = K;
    g.epi = epi;
    g.alpha = 1.0f;
    g.err = m->err_dev;
    g.fp8 = true;
    g.a_scale = a_inv;
    g.b_scale = m->w8_inv + slot;
    return timed(m, GPT2_PROF_MATMUL_E4M3, 2.0 * M * N * K, [&] { return tcg::launch_gemm_tc(g, m->num_sms, m->stream); });
}

// The fused LM head's product z = y_f wte^T over rows [r0, r0 + rows) with a cross-entropy
// epilogue: EPI_LSE (forward: row partials and target logits) or EPI_DZ (backward:
// dlogits for a unit loss weight into the logits buffer).
int lm_head_ce(gpt2_model *m, int epi, int r0, int rows, int BT) {
    const gpt2_config &c = m->cfg;
    tcg::GemmDesc g;
    g.A = (const bf16 *)m->lnf + (int64_t)r0 * c.C;
    g.lda = c.C;
    g.B = W<bf16>(m, 0);
    g.ldb = c.C;
    g.D = epi == tcg::EPI_DZ ? m->logits : nullptr;
    g.ldd = c.Vp;
    g.M = rows;
    g.N = c.Vp;
    g.K = c.C;
    g.epi = epi;
    g.err = m->err_dev;
    g.vocab = c.V;
    g.row_tgt = m->targets + r0;
    g.row_lse = m->ce_lse + r0;
    g.row_part = m->ce_part + (int64_t)r0 * m->ce_stride;
    g.part_stride = m->ce_stride;
    g.row_zt = m->ce_zt + r0;
    g.dz_scale = 1.0f / BT;
    return timed(m, GPT2_PROF_MATMUL, 2.0 * rows * c.Vp * c.C,
                 [&] { return tcg::launch_gemm_tc(g, m->num_sms, m->stream); });
}

// Refresh the E4M3 weight codes from the bf16 weight copy (one amax per tensor).
int quantize_weights(gpt2_model *m) {
    if (!m->w8) return GPT2_OK;
    double n = 0;
    for (int id : m->w8_ids) n += (double)m->tensors[id].numel;
    return timed(m, GPT2_PROF_OTHER, 5.0 * n, [&] {  // bf16 read twice (amax, codes), one code byte written
        return k::quantize_tensors_e4m3(m->wbf, m->w8_off, m->w8_n, (int)m->w8_ids.size(), m->w8_maxn, m->w8,
                                        m->w8_inv, m->w8_amax, m->stream);
    });
}

// algorithmic FLOP of causal attention forward: 4 hd per causal (i, j) pair
inline double attn_flops(int B, int Tn, int H, int hd) { return 4.0 * hd * (0.5 * Tn * (Tn + 1.0)) * B * H; }

template <typename T>
int attn_fwd(gpt2_model *m, const T *qkv, T *o, float *lse, int B, int Tn) {
    const int C = m->cfg.C, H = m->cfg.H, hd = C / H;
    return timed(m, GPT2_PROF_ATTENTION, attn_flops(B, Tn, H, hd), [&] {
        if constexpr (sizeof(T) == 2)
            return fa::attention_forward(qkv, qkv + C, qkv + 2 * C, 3 * C, o, C, lse, B, Tn, H, hd, m->stream);
        else
            return k::attention_forward_simt<T>(qkv, qkv + C, qkv + 2 * C, 3 * C, o, C, lse, B, Tn, H, hd,
                                                m->stream);
    });
}

template <typename T>
int attn_bwd(gpt2_model *m, const T *qkv, const T *o, const T *dout, const float *lse, T *dqkv, int B, int Tn,
             float *dbias) {
    const int C = m->cfg.C, H = m->cfg.H, hd = C / H;
    return timed(m, GPT2_PROF_ATTENTION, 2.0 * attn_flops(B, Tn, H, hd), [&] {
        if constexpr (sizeof(T) == 2)
            return fa::attention_backward(qkv, qkv + C, qkv + 2 * C, 3 * C, o, dout, C, lse, dqkv, dqkv + C,
                                          dqkv + 2 * C, m->attn_D, B, Tn, H, hd, m->stream, dbias,
                                          (bf16 *)m->attn_ds);
        else
            return k::attention_backward_simt<T>(qkv, qkv + C, qkv + 2 * C, 3 * C, o, dout, C, lse, dqkv, dqkv + C,
                                                 dqkv + 2 * C, m->attn_D, B, Tn, H, hd, m->stream);
    });
}

// ---- forward ----------------------------------------------------------------------
// One transformer block with E4M3 projections.  The LayerNorms write the E4M3
// codes of their bf16 output rows next to it; the attention output and GELU
// output are quantised per row by a separate pass.  Every bf16 activation the
// backward reads is still stored.
int forward_block_e4m3(gpt2_model *m, int l, int BT, int B, int Tn, bf16 *next, bf16 *gbuf) {
    const gpt2_config &c = m->cfg;
    const int C = c.C;
    cudaStream_t st = m->stream;
    LayerBuf &y = m->layers[l];
    const LayerParams &p = m->lp[l];
    const double act = 2.0 * BT * C, stats = 8.0 * BT, codes = (double)BT * C + 4.0 * BT;
    TIMED(GPT2_PROF_LAYERNORM, 2 * act + stats + codes,
          k::layernorm_forward<bf16>((bf16 *)y.resid, Pf(m, p.ln1g), Pf(m, p.ln1b), (bf16 *)y.ln1, y.ln1_mean,
                                     y.ln1_rstd, BT, C, st, m->a8, m->a8_inv));
    TRY(mm8(m, m->a8, C, m->a8_inv, p.qkvw, 4 * l, y.qkv, nullptr, nullptr, 3 * C, Pf(m, p.qkvb), BT, 3 * C, C,
            GPT2_EPI_STORE));
    TRY(attn_fwd<bf16>(m, (bf16 *)y.qkv, (bf16 *)y.att, y.lse, B, Tn));
    TIMED(GPT2_PROF_OTHER, act + codes, k::quantize_rows_e4m3((bf16 *)y.att, C, BT, C, m->a8, C, m->a8_inv, st));
    TRY(mm8(m, m->a8, C, m->a8_inv, p.projw, 4 * l + 1, y.resid_mid, nullptr, y.resid, C, Pf(m, p.projb), BT, C, C,
            GPT2_EPI_RESIDUAL));
    TIMED(GPT2_PROF_LAYERNORM, 2 * act + stats + codes,
          k::layernorm_forward<bf16>((bf16 *)y.resid_mid, Pf(m, p.ln2g), Pf(m, p.ln2b), (bf16 *)y.ln2, y.ln2_mean,
                                     y.ln2_rstd, BT, C, st, m->a8, m->a8_inv));
    TRY(mm8(m, m->a8, C, m->a8_inv, p.fcw, 4 * l + 2, y.fch, gbuf, nullptr, 4 * C, Pf(m, p.fcb), BT, 4 * C, C,
            GPT2_EPI_GELU));
    TIMED(GPT2_PROF_OTHER, 4 * (act + codes),
          k::quantize_rows_e4m3(gbuf, 4 * C, BT, 4 * C, m->a8, 4 * C, m->a8_inv, st));
    TRY(mm8(m, m->a8, 4 * C, m->a8_inv, p.fcprojw, 4 * l + 3, next, nullptr, y.resid_mid, C, Pf(m, p.fcprojb), BT,
            C, 4 * C, GPT2_EPI_RESIDUAL));
    return GPT2_OK;
}

template <typename T>
int forward_impl(gpt2_model *m, bool with_targets, int B, int Tn) {
    const gpt2_config &c = m->cfg;
    const int BT = B * Tn, C = c.C;
    cudaStream_t st = m->stream;
    const double es = sizeof(T), act = (double)BT * C * es, stats = 8.0 * BT;
    TIMED(GPT2_PROF_OTHER, 4.0 * BT + (double)BT * C * 4 + (double)Tn * C * 4 + act,
          k::embed_forward<T>(m->tokens, Pf(m, 0), Pf(m, 1), (T *)m->layers[0].resid, B, Tn, C, c.V, m->err_dev, st));
    for (int l = 0; l < c.L; ++l) {
        LayerBuf &y = m->layers[l];
        const LayerParams &p = m->lp[l];
        T *next = (T *)(l + 1 < c.L ? m->layers[l + 1].resid : m->resid_final);
        T *gbuf = (T *)(c.recompute_gelu ? m->gelu_buf : y.fcg);
        if constexpr (sizeof(T) == 2) {
            if (c.fp8_forward) {
                TRY(forward_block_e4m3(m, l, BT, B, Tn, next, gbuf));
                continue;
            }
        }
        TIMED(GPT2_PROF_LAYERNORM, 2 * act + stats,
              k::layernorm_forward<T>((T *)y.resid, Pf(m, p.ln1g), Pf(m, p.ln1b), (T *)y.ln1, y.ln1_mean, y.ln1_rstd,
                                      BT, C, st));
        TRY(mm<T>(m, y.ln1, C, true, W<T>(m, p.qkvw), C, true, y.qkv, nullptr, nullptr, 3 * C, Pf(m, p.qkvb), BT,
                  3 * C, C, GPT2_EPI_STORE));
        TRY(attn_fwd<T>(m, (T *)y.qkv, (T *)y.att, y.lse, B, Tn));
        TRY(mm<T>(m, y.att, C, true, W<T>(m, p.projw), C, true, y.resid_mid, nullptr, y.resid, C, Pf(m, p.projb), BT,
                  C, C, GPT2_EPI_RESIDUAL));
        TIMED(GPT2_PROF_LAYERNORM, 2 * act + stats,
              k::layernorm_forward<T>((T *)y.resid_mid, Pf(m, p.ln2g), Pf(m, p.ln2b), (T *)y.ln2, y.ln2_mean,
                                      y.ln2_rstd, BT, C, st));
        TRY(mm<T>(m, y.ln2, C, true, W<T>(m, p.fcw), C, true, y.fch, gbuf, nullptr, 4 * C, Pf(m, p.fcb), BT, 4 * C, C,
                  GPT2_EPI_GELU));
        TRY(mm<T>(m, gbuf, 4 * C, true, W<T>(m, p.fcprojw), 4 * C, true, next, nullptr, y.resid_mid, C,
                  Pf(m, p.fcprojb), BT, C, 4 * C, GPT2_EPI_RESIDUAL));
    }
    const int nt = (int)m->tensors.size();
    TIMED(GPT2_PROF_LAYERNORM, 2 * act + stats,
          k::layernorm_forward<T>((T *)m->resid_final, Pf(m, nt - 2), Pf(m, nt - 1), (T *)m->lnf, m->lnf_mean,
                                  m->lnf_rstd, BT, C, st));
    if constexpr (sizeof(T) == 2) {
        if (c.fused_lm_head && with_targets) {  // no logits: row partials, then lse and the loss
            TRY(lm_head_ce(m, tcg::EPI_LSE, 0, BT, BT));
            TIMED(GPT2_PROF_CLASSIFIER, 8.0 * BT * m->ce_stride + 16.0 * BT,
                  k::ce_combine(m->ce_part, m->ce_stride, m->ce_stride, m->ce_zt, m->targets, BT, c.V, m->ce_lse,
                                m->loss_rows, m->err_dev, st));
            TIMED(GPT2_PROF_OTHER, 4.0 * BT, k::mean_rows(m->loss_rows, BT, m->loss_dev, st));
            return GPT2_OK;
        }
    }
    if (BT > m->lm_rows) return GPT2_ERR_UNSUPPORTED;  // fused LM head: logits of at most lm_rows positions
    TRY(mm<T>(m, m->lnf, C, true, W<T>(m, 0), C, true, m->logits, nullptr, nullptr, c.Vp, nullptr, BT, c.Vp, C,
              GPT2_EPI_STORE));
    if (with_targets) {
        TIMED(GPT2_PROF_CLASSIFIER, 2.0 * BT * c.Vp * es + 8.0 * BT,
              k::classifier<T>((T *)m->logits, m->targets, m->loss_rows, BT, c.V, c.Vp, 1.0f / BT, m->err_dev, st));
        TIMED(GPT2_PROF_OTHER, 4.0 * BT, k::mean_rows(m->loss_rows, BT, m->loss_dev, st));
    }
    return GPT2_OK;
}

// ---- backward ---------------------------------------------------------------------
template <typename T>
int backward_impl(gpt2_model *m, float grad_scale) {
    const gpt2_config &c = m->cfg;
    const int B = m->fwd_B, Tn = m->fwd_T, BT = B * Tn, C = c.C, Vp = c.Vp;
    cudaStream_t st = m->stream;
    const int nt = (int)m->tensors.size();
    const double es = sizeof(T), act = (double)BT * C * es, stats = 8.0 * BT;
    T *dres = (T *)m->dres, *dbig = (T *)m->dbig, *dqkv = (T *)m->dqkv, *datt = (T *)m->datt,
      *dsmall = (T *)m->dsmall;
    // LM head (tied): dy_f = alpha dz wte ; dwte += alpha dz^T y_f.  With the fused LM head dz
    // is recomputed chunk by chunk (logits, then dlogits in the product's epilogue).
    const int lm_rows = c.fused_lm_head ? m->lm_rows : BT;
    for (int r0 = 0; r0 < BT; r0 += lm_rows) {
        const int rows = std::min(lm_rows, BT - r0);
        if constexpr (sizeof(T) == 2) {
            if (c.fused_lm_head) TRY(lm_head_ce(m, tcg::EPI_DZ, r0, rows, BT));
        }
        TRY(mm<T>(m, m->logits, Vp, true, W<T>(m, 0), C, false, dsmall + (int64_t)r0 * C, nullptr, nullptr, C, nullptr,
                  rows, C, Vp, GPT2_EPI_STORE, grad_scale));
        TRY(mm<T>(m, m->logits, Vp, false, (T *)m->lnf + (int64_t)r0 * C, C, false, Gf(m, 0), nullptr, nullptr, C,
                  nullptr, Vp, C, rows, GPT2_EPI_ACCUM_F32, grad_scale));
    }
    // The LayerNorm backward kernels also add the column sums of the residual
    // gradient they produce into the bias gradient of the projection that
    // consumes it (the last block's MLP output projection here).
    TIMED(GPT2_PROF_LAYERNORM, 3 * act + stats,
          k::layernorm_backward<T>(dsmall, (T *)m->resid_final, m->lnf_mean, m->lnf_rstd, Pf(m, nt - 2), nullptr, dres,
                                   Gf(m, nt - 2), Gf(m, nt - 1), BT, C, st, Gf(m, m->lp[c.L - 1].fcprojb)));
    for (int l = c.L - 1; l >= 0; --l) {
        LayerBuf &y = m->layers[l];
        const LayerParams &p = m->lp[l];
        T *g_in = (T *)y.fcg;
        if (c.recompute_gelu) {
            g_in = (T *)m->gelu_buf;
            TIMED(GPT2_PROF_OTHER, 8 * act, k::gelu_forward<T>((T *)y.fch, g_in, (int64_t)BT * 4 * C, st));
        }
        // bf16: bias gradients from the kernels that read the gradients they sum: the GELU-backward
        // product sums its output's columns into the FC bias gradient; the attention backward adds
        // the QKV bias gradient (query part: column sums of dq; value part: column sums of dO, since
        // every row of P sums to one; key part: zero, a key bias moves all scores of a query alike)
        constexpr bool fold_bias = sizeof(T) == 2;
        // FC projection x' = x1 + g Wfcproj^T + b: dX (GELU backward) first, then both MLP weight
        // gradients (FC projection from dres and g, FC from dH and y2) as one launch
        TRY(mm<T>(m, dres, C, true, W<T>(m, p.fcprojw), 4 * C, false, dbig, nullptr, y.fch, 4 * C, nullptr, BT, 4 * C,
                  C, GPT2_EPI_GELU_BWD, 1.0f, fold_bias ? Gf(m, p.fcb) : nullptr));
        TRY(mm_dw2<T>(m, DwProduct{dres, C, g_in, 4 * C, Gf(m, p.fcprojw), C, 4 * C},
                      DwProduct{dbig, 4 * C, y.ln2, C, Gf(m, p.fcw), 4 * C, C}, BT));
        if (!fold_bias) TIMED(GPT2_PROF_OTHER, 4 * act, k::column_sum<T>(dbig, BT, 4 * C, Gf(m, p.fcb), st));
        TRY(mm<T>(m, dbig, 4 * C, true, W<T>(m, p.fcw), C, false, dsmall, nullptr, nullptr, C, nullptr, BT, C, 4 * C,
                  GPT2_EPI_STORE));
        TIMED(GPT2_PROF_LAYERNORM, 4 * act + stats,
              k::layernorm_backward<T>(dsmall, (T *)y.resid_mid, y.ln2_mean, y.ln2_rstd, Pf(m, p.ln2g), dres, dres,
                                       Gf(m, p.ln2g), Gf(m, p.ln2b), BT, C, st, Gf(m, p.projb)));
        // attention projection x1 = x + O Wproj^T + b: dO, the attention backward, then the
        // projection's and the QKV product's weight gradients (from dres and O, dqkv and y) as one
        // launch (dres keeps its value until the LN1 backward)
        TRY(mm<T>(m, dres, C, true, W<T>(m, p.projw), C, false, datt, nullptr, nullptr, C, nullptr, BT, C, C,
                  GPT2_EPI_STORE));
        TRY(attn_bwd<T>(m, (T *)y.qkv, (T *)y.att, datt, y.lse, dqkv, B, Tn, fold_bias ? Gf(m, p.qkvb) : nullptr));
        TRY(mm_dw2<T>(m, DwProduct{dres, C, y.att, C, Gf(m, p.projw), C, C},
                      DwProduct{dqkv, 3 * C, y.ln1, C, Gf(m, p.qkvw), 3 * C, C}, BT));
        if (!fold_bias) TIMED(GPT2_PROF_OTHER, 3 * act, k::column_sum<T>(dqkv, BT, 3 * C, Gf(m, p.qkvb), st));
        TRY(mm<T>(m, dqkv, 3 * C, true, W<T>(m, p.qkvw), C, false, dsmall, nullptr, nullptr, C, nullptr, BT, C, 3 * C,
                  GPT2_EPI_STORE));
        TIMED(GPT2_PROF_LAYERNORM, 4 * act + stats,
              k::layernorm_backward<T>(dsmall, (T *)y.resid, y.ln1_mean, y.ln1_rstd, Pf(m, p.ln1g), dres, dres,
                                       Gf(m, p.ln1g), Gf(m, p.ln1b), BT, C, st,
                                       l > 0 ? Gf(m, m->lp[l - 1].fcprojb) : nullptr));
    }
    TIMED(GPT2_PROF_OTHER, act + 8.0 * BT * C + 4.0 * BT,
          k::embed_backward<T>(m->tokens, dres, Gf(m, 0), Gf(m, 1), B, Tn, C, c.V, st, m->emb_ws));
    return GPT2_OK;
}

// ---- generation ----------------------------------------------------------------------
// Position t of all B rows at a time.  The key/value cache is the step's qkv
// buffer of each block with a row stride of cfg.T positions per sequence.
// Scratch for the B rows of one position: dres (residual stream), dqkv
// (mid-block residual), dsmall (LayerNorm outputs), datt (attention output),
// dqkv + B*C (the position's QKV row), dbig (MLP pre-activation and GELU
// output), layer 0's LayerNorm statistics.  The position lives in device
// memory (gen_pos), so the launches of one position do not depend on t: the
// first position of each kind (filling the cache from the prompt, or also
// drawing a token) runs directly, the rest replay a CUDA graph of it.
// the decode products: a few rows against a K-major weight; bf16 rows take the
// skinny weight-streaming kernel, the rest the general matmul
template <typename T>
int dmm(gpt2_model *m, const void *X, int ldx, const void *Wt, void *D, void *D2, const void *R, int64_t ldd,
        const float *bias, int Bm, int N, int K, int epi) {
    if constexpr (sizeof(T) == 2) {
        if (Bm <= k::SK_MAX_ROWS) {
            const int rc = k::skinny_gemm((const bf16 *)X, ldx, (const bf16 *)Wt, K, N, Bm, bias, (const bf16 *)R,
                                          (bf16 *)D, (bf16 *)D2, ldd, epi, m->num_sms, m->stream);
            if (rc != GPT2_ERR_UNSUPPORTED) return rc;
        }
    }
    return mm<T>(m, X, ldx, true, Wt, K, true, D, D2, R, ldd, bias, Bm, N, K, epi);
}

template <typename T>
int decode_position(gpt2_model *m, int *d_seq, int B, int T_total, int T0, const float *d_u, float temperature,
                    int top_k, bool draw) {
    const gpt2_config &c = m->cfg;
    const int C = c.C, hd = C / c.H, Tc = c.T;
    cudaStream_t st = m->stream;
    const int nt = (int)m->tensors.size();
    T *x = (T *)m->dres, *xm = (T *)m->dqkv, *qkv = xm + (size_t)B * C, *y = (T *)m->dsmall, *att = (T *)m->datt;
    T *hbuf = (T *)m->dbig, *gbuf = hbuf + (size_t)B * 4 * C;
    float *mean = m->layers[0].ln1_mean, *rstd = m->layers[0].ln1_rstd;
    TRY(k::embed_decode<T>(d_seq, T_total, m->gen_pos, Pf(m, 0), Pf(m, 1), x, B, C, c.V, m->err_dev, st));
    for (int l = 0; l < c.L; ++l) {
        const LayerParams &p = m->lp[l];
        TRY(k::layernorm_forward<T>(x, Pf(m, p.ln1g), Pf(m, p.ln1b), y, mean, rstd, B, C, st));
        TRY(dmm<T>(m, y, C, W<T>(m, p.qkvw), qkv, nullptr, nullptr, 3 * C, Pf(m, p.qkvb), B, 3 * C, C,
                   GPT2_EPI_STORE));
        TRY(k::attention_decode<T>((T *)m->layers[l].qkv, qkv, Tc, m->gen_pos, T_total - 2, B, c.H, hd, att, st));
        TRY(dmm<T>(m, att, C, W<T>(m, p.projw), xm, nullptr, x, C, Pf(m, p.projb), B, C, C, GPT2_EPI_RESIDUAL));
        TRY(k::layernorm_forward<T>(xm, Pf(m, p.ln2g), Pf(m, p.ln2b), y, mean, rstd, B, C, st));
        TRY(dmm<T>(m, y, C, W<T>(m, p.fcw), hbuf, gbuf, nullptr, 4 * C, Pf(m, p.fcb), B, 4 * C, C, GPT2_EPI_GELU));
        TRY(dmm<T>(m, gbuf, 4 * C, W<T>(m, p.fcprojw), x, nullptr, xm, C, Pf(m, p.fcprojb), B, C, 4 * C,
                   GPT2_EPI_RESIDUAL));
    }
    if (draw) {
        TRY(k::layernorm_forward<T>(x, Pf(m, nt - 2), Pf(m, nt - 1), y, mean, rstd, B, C, st));
        TRY(dmm<T>(m, y, C, W<T>(m, 0), m->logits, nullptr, nullptr, c.Vp, nullptr, B, c.Vp, C, GPT2_EPI_STORE));
        TRY(k::sample_topk<T>((const T *)m->logits, c.Vp, B, c.V, d_u, temperature, top_k, d_seq, T_total, 0,
                              m->gen_pos, T0, st));
    }
    return k::advance_position(m->gen_pos, st);
}

template <typename T>
int generate_impl(gpt2_model *m, int *d_seq, int B, int T_total, int T0, const float *d_u, float temperature,
                  int top_k) {
    GPT2_CUDA_TRY(cudaMemsetAsync(m->gen_pos, 0, sizeof(int), m->stream));
    const int n_pos = T_total - 1;  // positions 0 .. T_total - 2; position t draws column t + 1 when t + 1 >= T0
    int t = 0;
    while (t < n_pos) {
        const bool draw = t + 1 >= T0;
        const int run = draw ? n_pos - t : T0 - 1 - t;  // positions of this kind from t on
        TRY(decode_position<T>(m, d_seq, B, T_total, T0, d_u, temperature, top_k, draw));
        if (run > 1) {
            cudaStream_t cs;
            GPT2_CUDA_TRY(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
            cudaStream_t saved = m->stream;
            m->stream = cs;
            cudaGraph_t graph = nullptr;
            int rc = GPT2_OK;
            const long long counted0 = g_launches.load(std::memory_order_relaxed);
            if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
                rc = GPT2_ERR_CUDA;
            } else {
                rc = decode_position<T>(m, d_seq, B, T_total, T0, d_u, temperature, top_k, draw);
                if (cudaStreamEndCapture(cs, &graph) != cudaSuccess && !rc) rc = GPT2_ERR_CUDA;
            }
            m->stream = saved;
            // the launchers counted one position while capturing; each replay runs that many kernels
            const long long per_position = g_launches.load(std::memory_order_relaxed) - counted0;
            cudaGraphExec_t exec = nullptr;
            if (!rc && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) rc = GPT2_ERR_CUDA;
            for (int i = 1; !rc && i < run; ++i)
                if (cudaGraphLaunch(exec, m->stream) != cudaSuccess) rc = GPT2_ERR_CUDA;
            if (exec) cudaGraphExecDestroy(exec);
            if (graph) cudaGraphDestroy(graph);
            cudaStreamDestroy(cs);
            if (rc) return rc;
            gpt2_note_launches((int)((run - 2) * per_position));
        }
        t += run;
    }
    return GPT2_OK;
}

// Run `launch` (which enqueues work on m->stream) through a CUDA graph cached
// under (kind, B, T, key): the first call with a key launches directly (which
// also performs the per-device set-up of the kernels it uses), the second
// captures the launch sequence on a private stream and replays it, later
// calls replay.  The graph bakes in every kernel argument, so the key must
// cover what varies; buffers live in the arena at fixed addresses.  With
// profiling on, or if capturing fails, the launches run directly.
template <typename F> int run_graphed(gpt2_model *m, int kind, int B, int T, uint32_t key, F &&launch) {
    if (m->prof_on || !m->graphs_on) return launch();
    gpt2_model::Graph *gr = nullptr;
    for (auto &e : m->graphs)
        if (e.kind == kind && e.B == B && e.T == T && e.key == key) gr = &e;
    if (!gr) {
        m->graphs.push_back(gpt2_model::Graph{kind, B, T, key, nullptr, 0, 0});
        gr = &m->graphs.back();
    }
    if (gr->exec) {
        GPT2_CUDA_TRY(cudaGraphLaunch(gr->exec, m->stream));
        gpt2_note_launches((int)gr->kernels);
        return GPT2_OK;
    }
    if (gr->uses++ != 1) return launch();  // first call (or capture failed before): direct
    cudaStream_t cs;
    GPT2_CUDA_TRY(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
    cudaStream_t saved = m->stream;
    m->stream = cs;
    cudaGraph_t graph = nullptr;
    int rc = GPT2_OK;
    const long long n0 = g_launches.load(std::memory_order_relaxed);
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        rc = GPT2_ERR_CUDA;
    } else {
        rc = launch();
        if (cudaStreamEndCapture(cs, &graph) != cudaSuccess && !rc) rc = GPT2_ERR_CUDA;
    }
    m->stream = saved;
    const long long kernels = g_launches.load(std::memory_order_relaxed) - n0;
    g_launches.fetch_sub(kernels, std::memory_order_relaxed);  // captured, not launched
    cudaGraphExec_t exec = nullptr;
    if (!rc && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) rc = GPT2_ERR_CUDA;
    if (graph) cudaGraphDestroy(graph);
    cudaStreamDestroy(cs);
    cudaGetLastError();  // a failed capture leaves no sticky error
    if (rc) {  // run this call directly; later calls with this key stay direct
        if (exec) cudaGraphExecDestroy(exec);
        return launch();
    }
    gr->exec = exec;
    gr->kernels = kernels;
    GPT2_CUDA_TRY(cudaGraphLaunch(exec, m->stream));
    gpt2_note_launches((int)kernels);
    return GPT2_OK;
}

void drop_graphs(gpt2_model *m) {
    for (auto &e : m->graphs)
        if (e.exec) cudaGraphExecDestroy(e.exec);
    m->graphs.clear();
}

int read_error_word(gpt2_model *m, int &word) {
    GPT2_CUDA_TRY(cudaMemcpyAsync(&word, m->err_dev, sizeof(int), cudaMemcpyDeviceToHost, m->stream));
    GPT2_CUDA_TRY(cudaStreamSynchronize(m->stream));
    if (word) GPT2_CUDA_TRY(cudaMemsetAsync(m->err_dev, 0, sizeof(int), m->stream));
    return GPT2_OK;
}

int error_from_word(int word) {
    if (word & DEVERR_TIMEOUT) return GPT2_ERR_TIMEOUT;
    if (word & DEVERR_BAD_TOKEN) return GPT2_ERR_BAD_TOKEN;
    return GPT2_OK;
}

}  // namespace

// ================================================================== C ABI
extern "C" size_t gpt2_arena_bytes(const gpt2_config *cfg) {
    if (!cfg || !valid_config(*cfg)) return 0;
    gpt2_model m{};
    m.cfg = *cfg;
    make_tensors(m.cfg, m.tensors, m.lp, m.n_params, m.n_decay);
    m.max_adam_blocks = k::clip_adamw_max_blocks(160);
    plan(m, nullptr);
    return m.arena_bytes;
}

extern "C" int gpt2_build(const gpt2_config *cfg, uint64_t seed, void *dev_arena, size_t arena_bytes,
                          void *cuda_stream, gpt2_model **out) {
    if (!cfg || !out || !dev_arena) return GPT2_ERR_BAD_ARG;
    *out = nullptr;
    if (!valid_config(*cfg)) return GPT2_ERR_BAD_CONFIG;
    if (reinterpret_cast<uintptr_t>(dev_arena) & 255) return GPT2_ERR_BAD_ARG;
    int num_sms = 0;
    TRY(check_device(num_sms));
    if (arena_bytes < gpt2_arena_bytes(cfg)) return GPT2_ERR_ARENA_TOO_SMALL;
    gpt2_model *m = new gpt2_model{};
    m->cfg = *cfg;
    m->stream = (cudaStream_t)cuda_stream;
    m->arena = (uint8_t *)dev_arena;
    m->num_sms = num_sms;
    make_tensors(m->cfg, m->tensors, m->lp, m->n_params, m->n_decay);
    m->max_adam_blocks = k::clip_adamw_max_blocks(160);
    plan(*m, m->arena);
    // host init: one fp32 image of all parameters, copied once
    std::vector<float> host(m->n_params, 0.0f);
    for (size_t id = 0; id < m->tensors.size(); ++id) {
        const TensorInfo &t = m->tensors[id];
        float *dst = host.data() + t.offset;
        if (t.kind == 1) std::fill(dst, dst + t.numel, 1.0f);
        if (t.kind == 2) fill_normal(seed, id, t.numel, t.std, dst);
        if (t.kind == 3) fill_normal(seed, id, (int64_t)cfg->V * cfg->C, t.std, dst);
    }
    int rc = GPT2_OK;
    auto fail = [&](int r) {
        delete m;
        return r;
    };
    if (cudaMemcpyAsync(m->params, host.data(), m->n_params * 4, cudaMemcpyHostToDevice, m->stream) != cudaSuccess)
        return fail(GPT2_ERR_CUDA);
    if (cudaMemsetAsync(m->grads, 0, m->n_params * 4 * 3, m->stream) != cudaSuccess) return fail(GPT2_ERR_CUDA);
    if (m->wbf && (rc = k::cast_f32_bf16(m->params, m->wbf, m->n_params, m->stream))) return fail(rc);
    std::vector<int64_t> w8_tab;  // offsets then sizes of the E4M3 weight tensors (copied below)
    if (m->w8) {
        m->w8_maxn = 0;
        for (const LayerParams &p : m->lp)
            for (int id : {p.qkvw, p.projw, p.fcw, p.fcprojw}) {
                m->w8_ids.push_back(id);
                m->w8_maxn = std::max(m->w8_maxn, m->tensors[id].numel);
            }
        for (int id : m->w8_ids) w8_tab.push_back(m->tensors[id].offset);
        for (int id : m->w8_ids) w8_tab.push_back(m->tensors[id].numel);
        const size_t nb = m->w8_ids.size() * 8;
        if (cudaMemcpyAsync(m->w8_off, w8_tab.data(), nb, cudaMemcpyHostToDevice, m->stream) != cudaSuccess ||
            cudaMemcpyAsync(m->w8_n, w8_tab.data() + m->w8_ids.size(), nb, cudaMemcpyHostToDevice, m->stream) !=
                cudaSuccess)
            return fail(GPT2_ERR_CUDA);
        if ((rc = quantize_weights(m))) return fail(rc);
    }
    if (cudaMemsetAsync(m->err_dev, 0, 256, m->stream) != cudaSuccess) return fail(GPT2_ERR_CUDA);
    if (cudaStreamSynchronize(m->stream) != cudaSuccess) return fail(GPT2_ERR_CUDA);
    *out = m;
    return GPT2_OK;
}

extern "C" int gpt2_forward(gpt2_model *m, const int32_t *d_tokens, const int32_t *d_targets, int B, int T,
                            float *loss_out) {
    if (!m || !d_tokens) return GPT2_ERR_BAD_ARG;
    if (B <= 0 || T <= 0 || B > m->cfg.B || T > m->cfg.T) return GPT2_ERR_BAD_SHAPE;
    if (d_targets && !loss_out) return GPT2_ERR_BAD_ARG;
    m->have_dlogits = false;
    GPT2_CUDA_TRY(cudaMemcpyAsync(m->tokens, d_tokens, (size_t)B * T * 4, cudaMemcpyDeviceToDevice, m->stream));
    if (d_targets)
        GPT2_CUDA_TRY(
            cudaMemcpyAsync(m->targets, d_targets, (size_t)B * T * 4, cudaMemcpyDeviceToDevice, m->stream));
    const bool tg = d_targets != nullptr;
    const int rc = run_graphed(m, tg ? 1 : 0, B, T, 0u, [&]() -> int {
        return m->cfg.dtype == GPT2_DTYPE_BF16 ? forward_impl<bf16>(m, tg, B, T) : forward_impl<float>(m, tg, B, T);
    });
    if (rc) return rc;
    m->fwd_B = B;
    m->fwd_T = T;
    if (!d_targets) return GPT2_OK;
    GPT2_CUDA_TRY(cudaMemcpyAsync(loss_out, m->loss_dev, 4, cudaMemcpyDeviceToHost, m->stream));
    int word = 0;
    TRY(read_error_word(m, word));
    TRY(error_from_word(word));
    m->have_dlogits = true;
    return std::isfinite(*loss_out) ? GPT2_OK : GPT2_ERR_NONFINITE;
}

extern "C" int gpt2_backward(gpt2_model *m, float grad_scale) {
    if (!m) return GPT2_ERR_BAD_ARG;
    if (!m->have_dlogits) return GPT2_ERR_STATE;
    m->have_dlogits = false;  // dlogits are consumed
    uint32_t key;
    memcpy(&key, &grad_scale, 4);  // the loss weight is a kernel argument of the graph
    return run_graphed(m, 2, m->fwd_B, m->fwd_T, key, [&]() -> int {
        return m->cfg.dtype == GPT2_DTYPE_BF16 ? backward_impl<bf16>(m, grad_scale)
                                               : backward_impl<float>(m, grad_scale);
    });
}

extern "C" int gpt2_generate(gpt2_model *m, int32_t *d_seq, int B, int T_total, int T0, const float *d_uniforms,
                             float temperature, int top_k) {
    if (!m || !d_seq || !d_uniforms) return GPT2_ERR_BAD_ARG;
    if (B <= 0 || B > m->cfg.B || T0 < 1 || T_total <= T0 || T_total > m->cfg.T) return GPT2_ERR_BAD_SHAPE;
    if (top_k < 1 || top_k > GPT2_MAX_TOP_K || !(temperature > 0.f)) return GPT2_ERR_BAD_ARG;
    m->have_dlogits = false;  // the activation buffers are reused
    const bool prof = m->prof_on;  // no per-launch events inside captured graphs
    m->prof_on = false;
    const int rc = m->cfg.dtype == GPT2_DTYPE_BF16
                       ? generate_impl<bf16>(m, d_seq, B, T_total, T0, d_uniforms, temperature, top_k)
                       : generate_impl<float>(m, d_seq, B, T_total, T0, d_uniforms, temperature, top_k);
    m->prof_on = prof;
    if (rc) return rc;
    int word = 0;
    TRY(read_error_word(m, word));
    return error_from_word(word);
}

extern "C" int gpt2_zero_grad(gpt2_model *m) {
    if (!m) return GPT2_ERR_BAD_ARG;
    GPT2_CUDA_TRY(cudaMemsetAsync(m->grads, 0, m->n_params * 4, m->stream));
    return GPT2_OK;
}

extern "C" int gpt2_clip_and_adamw(gpt2_model *m, float lr, float beta1, float beta2, float eps, float wd, float clip,
                                   float *grad_norm_out) {
    if (!m || !grad_norm_out) return GPT2_ERR_BAD_ARG;
    const int t = m->adam_t + 1;
    k::AdamArgs a;
    a.lr = lr;
    a.beta1 = beta1;
    a.beta2 = beta2;
    a.eps = eps;
    a.wd = wd;
    a.clip = clip;
    a.bc1 = (float)(1.0 - pow((double)beta1, t));
    a.bc2 = (float)(1.0 - pow((double)beta2, t));
    a.wait_ns = g_barrier_wait_ns.load(std::memory_order_relaxed);
    a.extra_arrivals = g_barrier_extra.load(std::memory_order_relaxed);
    const double adam_bytes = (double)m->n_params * (m->wbf ? 34.0 : 32.0);
    TIMED(GPT2_PROF_ADAMW, adam_bytes,
          k::clip_adamw(m->params, m->grads, m->adam_m, m->adam_v, m->wbf, m->n_params, m->n_decay, a,
                        m->norm_partials, m->barrier, m->max_adam_blocks, m->norm_dev, m->err_dev, m->num_sms,
                        m->stream));
    TRY(quantize_weights(m));
    GPT2_CUDA_TRY(cudaMemcpyAsync(grad_norm_out, m->norm_dev, 4, cudaMemcpyDeviceToHost, m->stream));
    int word = 0;
    TRY(read_error_word(m, word));
    TRY(error_from_word(word));
    if (!std::isfinite(*grad_norm_out)) return GPT2_ERR_NONFINITE;
    m->adam_t = t;
    return GPT2_OK;
}

extern "C" int gpt2_debug_set_barrier_wait(unsigned long long wait_ns, int never_arrive) {
    if (never_arrive != 0 && never_arrive != 1) return GPT2_ERR_BAD_ARG;
    g_barrier_wait_ns.store(wait_ns ? wait_ns : kDefaultBarrierWaitNs, std::memory_order_relaxed);
    g_barrier_extra.store((unsigned)never_arrive, std::memory_order_relaxed);
    return GPT2_OK;
}

extern "C" int gpt2_set_graphs(gpt2_model *m, int enable) {
    if (!m || (enable != 0 && enable != 1)) return GPT2_ERR_BAD_ARG;
    m->graphs_on = enable != 0;
    if (!enable) drop_graphs(m);
    return GPT2_OK;
}

extern "C" int gpt2_num_tensors(const gpt2_model *m) { return m ? (int)m->tensors.size() : 0; }

extern "C" int gpt2_tensor_info(const gpt2_model *m, int id, const char **name, int *ndim, int64_t shape[2]) {
    if (!m || id < 0 || id >= (int)m->tensors.size()) return GPT2_ERR_BAD_ARG;
    const TensorInfo &t = m->tensors[id];
    if (name) *name = t.name.c_str();
    if (ndim) *ndim = t.ndim;
    if (shape) {
        shape[0] = t.shape[0];
        shape[1] = t.shape[1];
    }
    return GPT2_OK;
}

static int copy_out(gpt2_model *m, const float *base, int id, float *host, size_t n) {
    if (!m || !host || id < 0 || id >= (int)m->tensors.size()) return GPT2_ERR_BAD_ARG;
    const TensorInfo &t = m->tensors[id];
    if (n < (size_t)t.numel) return GPT2_ERR_BAD_ARG;
    GPT2_CUDA_TRY(cudaMemcpyAsync(host, base + t.offset, t.numel * 4, cudaMemcpyDeviceToHost, m->stream));
    GPT2_CUDA_TRY(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

extern "C" int gpt2_get_params(gpt2_model *m, int id, float *host_out, size_t n) {
    return copy_out(m, m ? m->params : nullptr, id, host_out, n);
}
extern "C" int gpt2_get_grads(gpt2_model *m, int id, float *host_out, size_t n) {
    return copy_out(m, m ? m->grads : nullptr, id, host_out, n);
}
extern "C" int gpt2_get_adam_state(gpt2_model *m, int id, float *host_m, float *host_v, size_t n) {
    TRY(copy_out(m, m ? m->adam_m : nullptr, id, host_m, n));
    return copy_out(m, m->adam_v, id, host_v, n);
}

extern "C" int gpt2_set_params(gpt2_model *m, int id, const float *host_in, size_t n) {
    if (!m || !host_in || id < 0 || id >= (int)m->tensors.size()) return GPT2_ERR_BAD_ARG;
    const TensorInfo &t = m->tensors[id];
    if (n < (size_t)t.numel) return GPT2_ERR_BAD_ARG;
    GPT2_CUDA_TRY(cudaMemcpyAsync(m->params + t.offset, host_in, t.numel * 4, cudaMemcpyHostToDevice, m->stream));
    if (m->wbf) TRY(k::cast_f32_bf16(m->params + t.offset, m->wbf + t.offset, t.numel, m->stream));
    TRY(quantize_weights(m));
    GPT2_CUDA_TRY(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

extern "C" int gpt2_set_grads(gpt2_model *m, int id, const float *host_in, size_t n) {
    if (!m || !host_in || id < 0 || id >= (int)m->tensors.size()) return GPT2_ERR_BAD_ARG;
    const TensorInfo &t = m->tensors[id];
    if (n < (size_t)t.numel) return GPT2_ERR_BAD_ARG;
    GPT2_CUDA_TRY(cudaMemcpyAsync(m->grads + t.offset, host_in, t.numel * 4, cudaMemcpyHostToDevice, m->stream));
    GPT2_CUDA_TRY(cudaStreamSynchronize(m->stream));
    return GPT2_OK;
}

extern "C" int gpt2_debug_buffer(gpt2_model *m, const char *name, void **dev_ptr, size_t *bytes) {
    if (!m || !name || !dev_ptr || !bytes) return GPT2_ERR_BAD_ARG;
    const gpt2_config &c = m->cfg;
    const size_t es = c.dtype == GPT2_DTYPE_BF16 ? 2 : 4;
    const size_t BT = (size_t)c.B * c.T;
    std::string s(name);
    auto layer_of = [&](const char *prefix, int lim) -> int {
        const size_t n = strlen(prefix);
        if (s.compare(0, n, prefix) != 0) return -1;
        const int l = atoi(s.c_str() + n);
        return (l >= 0 && l < lim) ? l : -1;
    };
    int l;
    if (s == "logits") { *dev_ptr = m->logits; *bytes = (size_t)m->lm_rows * c.Vp * es; }
    else if (s == "loss_rows") { *dev_ptr = m->loss_rows; *bytes = BT * 4; }
    else if (s == "lnf") { *dev_ptr = m->lnf; *bytes = BT * c.C * es; }
    else if ((l = layer_of("qkv.", c.L)) >= 0) { *dev_ptr = m->layers[l].qkv; *bytes = BT * 3 * c.C * es; }
    else if ((l = layer_of("att.", c.L)) >= 0) { *dev_ptr = m->layers[l].att; *bytes = BT * c.C * es; }
    else if ((l = layer_of("lse.", c.L)) >= 0) { *dev_ptr = m->layers[l].lse; *bytes = (size_t)c.B * c.H * c.T * 4; }
    else if ((l = layer_of("ln1.", c.L)) >= 0) { *dev_ptr = m->layers[l].ln1; *bytes = BT * c.C * es; }
    else if ((l = layer_of("ln2.", c.L)) >= 0) { *dev_ptr = m->layers[l].ln2; *bytes = BT * c.C * es; }
    else if ((l = layer_of("resid_mid.", c.L)) >= 0) { *dev_ptr = m->layers[l].resid_mid; *bytes = BT * c.C * es; }
    else if ((l = layer_of("fch.", c.L)) >= 0) { *dev_ptr = m->layers[l].fch; *bytes = BT * 4 * c.C * es; }
    else if ((l = layer_of("resid.", c.L + 1)) >= 0) {
        *dev_ptr = l < c.L ? m->layers[l].resid : m->resid_final;
        *bytes = BT * c.C * es;
    } else if (m->w8 && (l = layer_of("w8.", (int)m->tensors.size())) >= 0) {
        *dev_ptr = m->w8 + m->tensors[l].offset;
        *bytes = (size_t)m->tensors[l].numel;
    } else if (m->w8 && s == "w8_inv") { *dev_ptr = m->w8_inv; *bytes = m->w8_ids.size() * 4; }
    else if (m->w8 && s == "a8") { *dev_ptr = m->a8; *bytes = BT * 4 * c.C; }
    else if (m->w8 && s == "a8_inv") { *dev_ptr = m->a8_inv; *bytes = BT * 4; }
    else return GPT2_ERR_BAD_ARG;
    return GPT2_OK;
}

extern "C" int gpt2_adam_step(const gpt2_model *m, int *t_out) {
    if (!m || !t_out) return GPT2_ERR_BAD_ARG;
    *t_out = m->adam_t;
    return GPT2_OK;
}

extern "C" int gpt2_profile(gpt2_model *m, int enable) {
    if (!m) return GPT2_ERR_BAD_ARG;
    if (enable) {
        TRY(prof_flush(m));
        for (int c = 0; c < GPT2_PROF_NCAT; ++c) {
            m->prof_ms[c] = m->prof_work[c] = 0.0;
            m->prof_n[c] = 0;
        }
    }
    m->prof_on = enable != 0;
    return GPT2_OK;
}

extern "C" int gpt2_profile_read(gpt2_model *m, int category, double *total_ms, double *total_work,
                                 long long *launches) {
    if (!m || category < 0 || category >= GPT2_PROF_NCAT) return GPT2_ERR_BAD_ARG;
    TRY(prof_flush(m));
    if (total_ms) *total_ms = m->prof_ms[category];
    if (total_work) *total_work = m->prof_work[category];
    if (launches) *launches = m->prof_n[category];
    return GPT2_OK;
}

extern "C" void gpt2_free(gpt2_model *m) {
    if (!m) return;
    drop_graphs(m);
    for (auto &r : m->prof) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    delete m;
}

// ================================================================== op-level C ABI
static int op_sms() {
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 148;
    }
    return sms;
}

extern "C" int gpt2_op_attention_forward(const void *q, const void *kk, const void *v, int64_t qkv_row_stride,
                                         void *o, int64_t o_row_stride, float *lse, int B, int T, int H, int hd,
                                         void *stream) {
    if (!q || !kk || !v || !o || !lse) return GPT2_ERR_BAD_ARG;
    if (B <= 0 || T <= 0 || H <= 0 || hd != 64 || qkv_row_stride % 8 || o_row_stride % 8) return GPT2_ERR_BAD_SHAPE;
    return fa::attention_forward((const bf16 *)q, (const bf16 *)kk, (const bf16 *)v, qkv_row_stride, (bf16 *)o,
                                 o_row_stride, lse, B, T, H, hd, (cudaStream_t)stream);
}

extern "C" int gpt2_op_attention_backward(const void *q, const void *kk, const void *v, int64_t qkv_row_stride,
                                          const void *o, const void *dout, int64_t o_row_stride, const float *lse,
                                          void *dq, void *dk, void *dv, float *d_scratch, int B, int T, int H, int hd,
                                          void *stream) {
    if (!q || !kk || !v || !o || !dout || !lse || !dq || !dk || !dv || !d_scratch) return GPT2_ERR_BAD_ARG;
    if (B <= 0 || T <= 0 || H <= 0 || hd != 64 || qkv_row_stride % 8 || o_row_stride % 8) return GPT2_ERR_BAD_SHAPE;
    return fa::attention_backward((const bf16 *)q, (const bf16 *)kk, (const bf16 *)v, qkv_row_stride, (const bf16 *)o,
                                  (const bf16 *)dout, o_row_stride, lse, (bf16 *)dq, (bf16 *)dk, (bf16 *)dv, d_scratch,
                                  B, T, H, hd, (cudaStream_t)stream);
}

extern "C" size_t gpt2_attention_backward_ds_bytes(int B, int T, int H) {
    if (B <= 0 || T <= 0 || H <= 0) return 0;
    return fa::attention_backward_ds_bytes(B, T, H);
}

extern "C" int gpt2_op_attention_backward_ds(const void *q, const void *kk, const void *v, int64_t qkv_row_stride,
                                             const void *o, const void *dout, int64_t o_row_stride, const float *lse,
                                             void *dq, void *dk, void *dv, float *d_scratch, void *d_ds,
                                             size_t ds_bytes, int B, int T, int H, int hd, void *stream) {
    if (!q || !kk || !v || !o || !dout || !lse || !dq || !dk || !dv || !d_scratch) return GPT2_ERR_BAD_ARG;
    if (B <= 0 || T <= 0 || H <= 0 || hd != 64 || qkv_row_stride % 8 || o_row_stride % 8) return GPT2_ERR_BAD_SHAPE;
    if (H * hd > 2048) return GPT2_ERR_UNSUPPORTED;
    if (!d_ds || (reinterpret_cast<uintptr_t>(d_ds) & 15) || ds_bytes < fa::attention_backward_ds_bytes(B, T, H))
        return GPT2_ERR_BAD_ARG;
    return fa::attention_backward((const bf16 *)q, (const bf16 *)kk, (const bf16 *)v, qkv_row_stride, (const bf16 *)o,
                                  (const bf16 *)dout, o_row_stride, lse, (bf16 *)dq, (bf16 *)dk, (bf16 *)dv, d_scratch,
                                  B, T, H, hd, (cudaStream_t)stream, nullptr, (bf16 *)d_ds);
}

extern "C" int gpt2_op_matmul(const void *A, int64_t lda, int a_kmajor, const void *B, int64_t ldb, int b_kmajor,
                              void *D, void *D2, const void *R, int64_t ldd, const float *bias, int M, int N, int K,
                              int epilogue, void *stream) {
    tcg::GemmDesc g;
    g.A = (const bf16 *)A;
    g.lda = lda;
    g.a_kmajor = a_kmajor != 0;
    g.B = (const bf16 *)B;
    g.ldb = ldb;
    g.b_kmajor = b_kmajor != 0;
    g.D = D;
    g.D2 = (bf16 *)D2;
    g.R = (const bf16 *)R;
    g.ldd = ldd;
    g.bias = bias;
    g.M = M;
    g.N = N;
    g.K = K;
    g.epi = epilogue;
    g.alpha = 1.0f;
    g.err = nullptr;
    return tcg::launch_gemm_tc(g, op_sms(), (cudaStream_t)stream);
}

extern "C" int gpt2_op_matmul_accum2(const void *A0, int64_t lda0, const void *B0, int64_t ldb0, float *D0, int M0,
                                     int N0, const void *A1, int64_t lda1, const void *B1, int64_t ldb1, float *D1,
                                     int M1, int N1, int K, void *stream) {
    tcg::GemmDesc g[2];
    const void *A[2] = {A0, A1}, *Bp[2] = {B0, B1};
    const int64_t lda[2] = {lda0, lda1}, ldb[2] = {ldb0, ldb1};
    float *D[2] = {D0, D1};
    const int M[2] = {M0, M1}, N[2] = {N0, N1};
    for (int i = 0; i < 2; ++i) {
        g[i].A = (const bf16 *)A[i];
        g[i].lda = lda[i];
        g[i].a_kmajor = false;
        g[i].B = (const bf16 *)Bp[i];
        g[i].ldb = ldb[i];
        g[i].b_kmajor = false;
        g[i].D = D[i];
        g[i].ldd = N[i];
        g[i].M = M[i];
        g[i].N = N[i];
        g[i].K = K;
        g[i].epi = GPT2_EPI_ACCUM_F32;
        g[i].err = nullptr;
    }
    return tcg::launch_gemm_tc_grouped(g[0], g[1], op_sms(), (cudaStream_t)stream);
}

extern "C" int gpt2_op_layernorm_forward(const void *x, const float *g, const float *b, void *y, float *mean,
                                         float *rstd, int N, int C, void *stream) {
    if (!x || !g || !b || !y || !mean || !rstd) return GPT2_ERR_BAD_ARG;
    if (N <= 0 || C <= 0 || C % 8 || C > 2048) return GPT2_ERR_BAD_SHAPE;
    return k::layernorm_forward<bf16>((const bf16 *)x, g, b, (bf16 *)y, mean, rstd, N, C, (cudaStream_t)stream);
}

extern "C" int gpt2_op_layernorm_backward(const void *dy, const void *x, const float *mean, const float *rstd,
                                          const float *g, const void *dres_in, void *dres_out, float *dg, float *db,
                                          int N, int C, void *stream) {
    if (!dy || !x || !mean || !rstd || !g || !dres_out || !dg || !db) return GPT2_ERR_BAD_ARG;
    if (N <= 0 || C <= 0 || C % 8 || C > 2048) return GPT2_ERR_BAD_SHAPE;
    return k::layernorm_backward<bf16>((const bf16 *)dy, (const bf16 *)x, mean, rstd, g, (const bf16 *)dres_in,
                                       (bf16 *)dres_out, dg, db, N, C, (cudaStream_t)stream);
}

extern "C" int gpt2_op_sample(const void *logits, int64_t ldl, int B, int V, const float *uniforms, float temperature,
                              int top_k, int32_t *out, void *stream) {
    if (!logits || !uniforms || !out) return GPT2_ERR_BAD_ARG;
    if (B <= 0 || V <= 0 || ldl < V) return GPT2_ERR_BAD_SHAPE;
    return k::sample_topk<bf16>((const bf16 *)logits, ldl, B, V, uniforms, temperature, top_k, out, 1, 0, nullptr, 0,
                                (cudaStream_t)stream);
}

extern "C" size_t gpt2_embedding_backward_workspace(int B, int T, int C) {
    if (B <= 0 || T <= 0 || C <= 0) return 0;
    return k::embed_backward_workspace(B * T, C);
}

extern "C" int gpt2_op_embedding_backward(const void *dx, int dtype, const int32_t *tokens, int B, int T, int C,
                                          int V, float *dwte, float *dwpe, void *d_workspace, void *stream) {
    if (!dx || !tokens || !dwte || !dwpe) return GPT2_ERR_BAD_ARG;
    if (B <= 0 || T <= 0 || C <= 0 || V <= 0 || C % 4) return GPT2_ERR_BAD_SHAPE;
    if (reinterpret_cast<uintptr_t>(d_workspace) & 255) return GPT2_ERR_BAD_ARG;
    if (dtype == GPT2_DTYPE_FP32)
        return k::embed_backward<float>(tokens, (const float *)dx, dwte, dwpe, B, T, C, V, (cudaStream_t)stream,
                                        d_workspace);
    if (dtype == GPT2_DTYPE_BF16)
        return k::embed_backward<bf16>(tokens, (const bf16 *)dx, dwte, dwpe, B, T, C, V, (cudaStream_t)stream,
                                       d_workspace);
    return GPT2_ERR_BAD_ARG;
}

extern "C" int gpt2_op_classifier(void *logits, const int32_t *targets, float *loss_rows, int N, int V, int Vp,
                                  float dscale, void *stream) {
    if (!logits || !targets || !loss_rows) return GPT2_ERR_BAD_ARG;
    if (N <= 0) return GPT2_ERR_BAD_SHAPE;
    return k::classifier<bf16>((bf16 *)logits, targets, loss_rows, N, V, Vp, dscale, nullptr, (cudaStream_t)stream);
}
