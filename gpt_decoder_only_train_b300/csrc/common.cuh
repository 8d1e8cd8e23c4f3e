// Shared device helpers: bf16 <-> fp32, 16-byte vectors, warp reductions, and
// the error word that bounded device waits and index checks write into.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/gpt2b300.h"

typedef __nv_bfloat16 bf16;

#define GPT2_CUDA_TRY(expr)                                  \
    do {                                                     \
        cudaError_t e__ = (expr);                            \
        if (e__ != cudaSuccess) {                            \
            gpt2_set_last_cuda_error(e__, #expr, __LINE__);  \
            return GPT2_ERR_CUDA;                            \
        }                                                    \
    } while (0)

void gpt2_set_last_cuda_error(cudaError_t e, const char *what, int line);

// Process-wide count of kernel launches made by this library.
void gpt2_note_launches(int n);

// error-word bits written by kernels (the host reads the word after a step)
enum : int {
    DEVERR_BAD_TOKEN = 1,
    DEVERR_TIMEOUT = 2,
};

__device__ __forceinline__ void raise_device_error(int *err, int bit) {
    if (err) atomicOr(err, bit);
}

// ---- element conversions --------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float x) { return __float2bfloat16_rn(x); }

// A 16-byte packet of activations: 8 bf16 or 4 fp32.
template <typename T> struct Pack16 {
    static constexpr int N = 16 / sizeof(T);
    uint4 raw;
    __device__ __forceinline__ float get(int i) const {
        const T *p = reinterpret_cast<const T *>(&raw);
        return to_f32(p[i]);
    }
    __device__ __forceinline__ void set(int i, float v) {
        T *p = reinterpret_cast<T *>(&raw);
        p[i] = from_f32<T>(v);
    }
    __device__ __forceinline__ void load(const T *ptr) { raw = *reinterpret_cast<const uint4 *>(ptr); }
    __device__ __forceinline__ void load_stream(const T *ptr) {
        raw = __ldcs(reinterpret_cast<const uint4 *>(ptr));
    }
    __device__ __forceinline__ void store(T *ptr) const { *reinterpret_cast<uint4 *>(ptr) = raw; }
};

// The two bf16 halves of a packed word as fp32 (exact: a bf16 is the top half of an fp32)
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 values packed in one 64-bit register: the .f32x2 forms of
// fma / mul / add / sub (sm_100 and later) do the work of two scalar
// instructions with one issue slot.  Rounding is that of the scalar forms.
struct F2 {
    unsigned long long u;
};
__device__ __forceinline__ F2 f2(float lo, float hi) {
    F2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r.u) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float f2_lo(F2 v) { return __uint_as_float((uint32_t)v.u); }
__device__ __forceinline__ float f2_hi(F2 v) { return __uint_as_float((uint32_t)(v.u >> 32)); }
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
    F2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d.u) : "l"(a.u), "l"(b.u), "l"(c.u));
    return d;
}
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
    F2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d.u) : "l"(a.u), "l"(b.u));
    return d;
}
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) {
    F2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d.u) : "l"(a.u), "l"(b.u));
    return d;
}

__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
    F2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d.u) : "l"(a.u), "l"(b.u));
    return d;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Hardware tanh (MUFU.TANH, relative error ~2^-11): the GELU outputs and
// gradients are stored in bf16 (relative 2^-9), so the approximation is below
// the storage rounding.
__device__ __forceinline__ float tanh_hw(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// GELU, tanh form: gelu(h) = h/2 (1 + tanh(k (h + c h^3))), k = sqrt(2/pi),
// c = 0.044715, written as u = k + k c h^2, t = tanh(h u), gelu = h/2 + (h/2) t.
// Its derivative 1/2 (1 + t) + a (1 - t^2) with a = (k h / 2)(1 + 3 c h^2) is
// evaluated as 1/2 + t/2 - na + (na t) t with na = -a.  The scalar and paired
// versions run the same operations in the same order, so every kernel that
// uses them produces the same bits.
constexpr float GELU_K = 0.7978845608028654f, GELU_KC = 0.035677408136300125f;  // k, k c
constexpr float GELU_NA1 = -0.05351611220445019f, GELU_NA0 = -0.3989422804014327f;  // -3 k c / 2, -k / 2
__device__ __forceinline__ float gelu_tanh(float h) {
    const float h2 = h * h, u = fmaf(h2, GELU_KC, GELU_K), t = tanh_hw(h * u), hh = 0.5f * h;
    return fmaf(hh, t, hh);
}
__device__ __forceinline__ float gelu_tanh_grad(float h) {
    const float h2 = h * h, u = fmaf(h2, GELU_KC, GELU_K), t = tanh_hw(h * u);
    const float na = h * fmaf(h2, GELU_NA1, GELU_NA0);
    const float base = fmaf(t, 0.5f, 0.5f) - na;
    return fmaf(na * t, t, base);
}
__device__ __forceinline__ F2 gelu_tanh2(F2 h) {
    const F2 h2 = f2_mul(h, h), u = f2_fma(h2, f2(GELU_KC, GELU_KC), f2(GELU_K, GELU_K));
    const F2 a = f2_mul(h, u), t = f2(tanh_hw(f2_lo(a)), tanh_hw(f2_hi(a))), hh = f2_mul(h, f2(0.5f, 0.5f));
    return f2_fma(hh, t, hh);
}
__device__ __forceinline__ F2 gelu_tanh_grad2(F2 h) {
    const F2 h2 = f2_mul(h, h), u = f2_fma(h2, f2(GELU_KC, GELU_KC), f2(GELU_K, GELU_K));
    const F2 a = f2_mul(h, u), t = f2(tanh_hw(f2_lo(a)), tanh_hw(f2_hi(a)));
    const F2 na = f2_mul(h, f2_fma(h2, f2(GELU_NA1, GELU_NA1), f2(GELU_NA0, GELU_NA0)));
    const F2 base = f2_sub(f2_fma(t, f2(0.5f, 0.5f), f2(0.5f, 0.5f)), na);
    return f2_fma(f2_mul(na, t), t, base);
}

// Precision by element type.  bf16 data (relative rounding 2^-9) takes the
// hardware approximations above and __expf / rsqrtf; fp32 data takes CUDA's
// accurate tanhf / expf and a correctly rounded 1 / sqrt, so that the fp32
// mode computes in true fp32 throughout.
template <typename T> __device__ __forceinline__ float tanh_t(float x) { return tanh_hw(x); }
template <> __device__ __forceinline__ float tanh_t<float>(float x) { return tanhf(x); }
template <typename T> __device__ __forceinline__ float exp_t(float x) { return __expf(x); }
template <> __device__ __forceinline__ float exp_t<float>(float x) { return expf(x); }
template <typename T> __device__ __forceinline__ float rsqrt_t(float x) { return rsqrtf(x); }
template <> __device__ __forceinline__ float rsqrt_t<float>(float x) { return 1.0f / sqrtf(x); }

// GELU and its derivative at the precision of element type T: the same
// operations as gelu_tanh / gelu_tanh_grad, with tanh_t<T>.
template <typename T> __device__ __forceinline__ float gelu_tanh_t(float h) {
    const float h2 = h * h, u = fmaf(h2, GELU_KC, GELU_K), t = tanh_t<T>(h * u), hh = 0.5f * h;
    return fmaf(hh, t, hh);
}
template <typename T> __device__ __forceinline__ float gelu_tanh_grad_t(float h) {
    const float h2 = h * h, u = fmaf(h2, GELU_KC, GELU_K), t = tanh_t<T>(h * u);
    const float na = h * fmaf(h2, GELU_NA1, GELU_NA0);
    const float base = fmaf(t, 0.5f, 0.5f) - na;
    return fmaf(na * t, t, base);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

static inline int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

// Per-device one-time set-up.  A kernel's opt-in shared-memory limit and an
// occupancy result belong to one device, so they are set up and cached per
// device ordinal (up to 64), by `make(int &value)` on the first call made with
// that device current.  Thread-safe; `make` runs under the lock.
struct PerDevice {
    std::mutex mu;
    int val[64] = {};
    bool have[64] = {};
};
template <typename F> int per_device(PerDevice &pd, int &out, F &&make) {
    int dev = 0;
    GPT2_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return GPT2_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(pd.mu);
    if (!pd.have[dev]) {
        int v = 0;
        if (int rc = make(v)) return rc;
        pd.val[dev] = v;
        pd.have[dev] = true;
    }
    out = pd.val[dev];
    return GPT2_OK;
}
