// E4M3 quantisation and the E4M3 matmul entry points.
//
// The pages name FP8 as the next precision step of this training code
// ("llm.c kullanarak GPT-2 modelini düşük maliyetle yeniden uygulamak", §SSS;
// the "PyTorch Howsam" post on llm.c) without fixing a format or a scaling
// rule.  Format: E4M3 as the OCP 8-bit floating point specification defines
// it (largest finite 448), converted with round to nearest even and
// saturation.  Scaling: per row for activations and per tensor for weights,
// by s = 448 / amax computed in fp32, the element scaled by one fp32
// multiply; the dequantisation factor amax / 448 is kept beside the codes.
#include "kernels.cuh"
#include "tc_gemm.cuh"

namespace {

constexpr float E4M3_MAX = 448.0f;

__device__ __forceinline__ uint32_t to_e4m3(float x) { return k::e4m3_of(x); }

// One warp per row: amax of the row, then the codes of x * (448 / amax).
__global__ void quantize_rows_kernel(const bf16 *__restrict__ x, int64_t ldx, int M, int K, uint8_t *__restrict__ q,
                                     int64_t ldq, float *__restrict__ inv) {
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= M) return;
    const bf16 *xr = x + (int64_t)row * ldx;
    float amax = 0.f;
    for (int c = lane * 8; c < K; c += 256) {
        const uint4 u = *reinterpret_cast<const uint4 *>(xr + c);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
    }
    amax = warp_max(amax);
    const float s = amax > 0.f ? E4M3_MAX / amax : 1.0f;
    uint8_t *qr = q + (int64_t)row * ldq;
    for (int c = lane * 8; c < K; c += 256) {
        const uint4 u = *reinterpret_cast<const uint4 *>(xr + c);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t b0 = to_e4m3(bf16_lo(w[k]) * s), b1 = to_e4m3(bf16_hi(w[k]) * s);
            const uint32_t pair = b0 | (b1 << 8);
            if (k < 2)
                lo |= pair << (16 * k);
            else
                hi |= pair << (16 * (k - 2));
        }
        *reinterpret_cast<uint2 *>(qr + c) = make_uint2(lo, hi);
    }
    if (lane == 0) inv[row] = amax > 0.f ? amax / E4M3_MAX : 1.0f;
}

// amax of a tensor: block maxima combined with an integer atomic max on the
// bits of non-negative floats (ordered like the values).
__global__ void amax_kernel(const bf16 *__restrict__ x, int64_t n, unsigned *__restrict__ amax_bits) {
    float m = 0.f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n / 8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 u = reinterpret_cast<const uint4 *>(x)[i];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[k])), fabsf(bf16_hi(w[k]))));
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));
}

__global__ void quantize_tensor_kernel(const bf16 *__restrict__ x, int64_t n, const unsigned *__restrict__ amax_bits,
                                       uint8_t *__restrict__ q, float *__restrict__ inv) {
    const float amax = __uint_as_float(*amax_bits);
    const float s = amax > 0.f ? E4M3_MAX / amax : 1.0f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n / 8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 u = reinterpret_cast<const uint4 *>(x)[i];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t pair = to_e4m3(bf16_lo(w[k]) * s) | (to_e4m3(bf16_hi(w[k]) * s) << 8);
            if (k < 2)
                lo |= pair << (16 * k);
            else
                hi |= pair << (16 * (k - 2));
        }
        reinterpret_cast<uint2 *>(q)[i] = make_uint2(lo, hi);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *inv = amax > 0.f ? amax / E4M3_MAX : 1.0f;
}

// Several tensors of one flat bf16 array, one amax each: block (x, t) covers a
// chunk of tensor t.
__global__ void amax_multi_kernel(const bf16 *__restrict__ w, const int64_t *__restrict__ off,
                                  const int64_t *__restrict__ n, unsigned *__restrict__ amax_bits) {
    const int t = blockIdx.y;
    const int64_t n8 = n[t] / 8;
    const uint4 *src = reinterpret_cast<const uint4 *>(w + off[t]);
    float m = 0.f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 u = src[i];
        const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) m = fmaxf(m, fmaxf(fabsf(bf16_lo(ww[k])), fabsf(bf16_hi(ww[k]))));
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) atomicMax(amax_bits + t, __float_as_uint(m));
}

__global__ void quantize_multi_kernel(const bf16 *__restrict__ w, const int64_t *__restrict__ off,
                                      const int64_t *__restrict__ n, const unsigned *__restrict__ amax_bits,
                                      uint8_t *__restrict__ q, float *__restrict__ inv) {
    const int t = blockIdx.y;
    const int64_t n8 = n[t] / 8;
    const uint4 *src = reinterpret_cast<const uint4 *>(w + off[t]);
    uint2 *dst = reinterpret_cast<uint2 *>(q + off[t]);
    const float amax = __uint_as_float(amax_bits[t]);
    const float s = amax > 0.f ? E4M3_MAX / amax : 1.0f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 u = src[i];
        const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t pair = to_e4m3(bf16_lo(ww[k]) * s) | (to_e4m3(bf16_hi(ww[k]) * s) << 8);
            if (k < 2)
                lo |= pair << (16 * k);
            else
                hi |= pair << (16 * (k - 2));
        }
        dst[i] = make_uint2(lo, hi);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) inv[t] = amax > 0.f ? amax / E4M3_MAX : 1.0f;
}

int sms_of_current_device() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms > 0 ? sms : 148;
}

}  // namespace

extern "C" int gpt2_op_quantize_e4m3_rows(const void *x, int64_t ldx, int M, int K, uint8_t *q, int64_t ldq,
                                          float *row_inv, void *stream) {
    if (!x || !q || !row_inv) return GPT2_ERR_BAD_ARG;
    if (M <= 0 || K <= 0 || K % 8 || ldx % 8 || ldq % 8 || ldx < K || ldq < K) return GPT2_ERR_BAD_SHAPE;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(q)) & 15) return GPT2_ERR_BAD_ARG;
    quantize_rows_kernel<<<ceil_div(M, 8), 256, 0, (cudaStream_t)stream>>>((const bf16 *)x, ldx, M, K, q, ldq,
                                                                           row_inv);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

extern "C" int gpt2_op_quantize_e4m3_tensor(const void *x, int64_t n, uint8_t *q, float *inv, unsigned *d_amax_work,
                                            void *stream) {
    if (!x || !q || !inv || !d_amax_work) return GPT2_ERR_BAD_ARG;
    if (n <= 0 || n % 8) return GPT2_ERR_BAD_SHAPE;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(q)) & 15) return GPT2_ERR_BAD_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    GPT2_CUDA_TRY(cudaMemsetAsync(d_amax_work, 0, sizeof(unsigned), st));
    const int grid = (int)std::min<int64_t>(4 * sms_of_current_device(), std::max<int64_t>(1, (n / 8 + 255) / 256));
    amax_kernel<<<grid, 256, 0, st>>>((const bf16 *)x, n, d_amax_work);
    quantize_tensor_kernel<<<grid, 256, 0, st>>>((const bf16 *)x, n, d_amax_work, q, inv);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(2);
    return GPT2_OK;
}

extern "C" int gpt2_op_matmul_e4m3(const uint8_t *A, int64_t lda, const float *a_row_inv, const uint8_t *B, int64_t ldb,
                                   const float *b_inv, void *D, void *D2, const void *R, int64_t ldd,
                                   const float *bias, int M, int N, int K, int epilogue, void *stream) {
    if (!A || !B || !D || !a_row_inv || !b_inv) return GPT2_ERR_BAD_ARG;
    if (epilogue != GPT2_EPI_STORE && epilogue != GPT2_EPI_RESIDUAL && epilogue != GPT2_EPI_GELU)
        return GPT2_ERR_BAD_ARG;
    tcg::GemmDesc g;
    g.A = reinterpret_cast<const bf16 *>(A);  // bytes: the descriptor only carries the address
    g.lda = lda;
    g.a_kmajor = true;
    g.B = reinterpret_cast<const bf16 *>(B);
    g.ldb = ldb;
    g.b_kmajor = true;
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
    g.fp8 = true;
    g.a_scale = a_row_inv;
    g.b_scale = b_inv;
    return tcg::launch_gemm_tc(g, sms_of_current_device(), (cudaStream_t)stream);
}

namespace k {

int quantize_rows_e4m3(const bf16 *x, int64_t ldx, int M, int K, uint8_t *q, int64_t ldq, float *inv,
                       cudaStream_t st) {
    if (M <= 0 || K <= 0 || K % 8 || ldx % 8 || ldq % 8) return GPT2_ERR_BAD_SHAPE;
    quantize_rows_kernel<<<ceil_div(M, 8), 256, 0, st>>>(x, ldx, M, K, q, ldq, inv);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(1);
    return GPT2_OK;
}

int quantize_tensors_e4m3(const bf16 *w, const int64_t *d_off, const int64_t *d_n, int ntens, int64_t max_n,
                          uint8_t *q, float *inv, unsigned *amax_bits, cudaStream_t st) {
    if (ntens <= 0) return GPT2_OK;
    GPT2_CUDA_TRY(cudaMemsetAsync(amax_bits, 0, sizeof(unsigned) * ntens, st));
    const dim3 grid((unsigned)std::max<int64_t>(1, std::min<int64_t>(64, (max_n / 8 + 255) / 256)), (unsigned)ntens);
    amax_multi_kernel<<<grid, 256, 0, st>>>(w, d_off, d_n, amax_bits);
    quantize_multi_kernel<<<grid, 256, 0, st>>>(w, d_off, d_n, amax_bits, q, inv);
    GPT2_CUDA_TRY(cudaGetLastError());
    gpt2_note_launches(2);
    return GPT2_OK;
}

}  // namespace k
