// Attention backward for callers that cannot allocate device memory.
//
// The regular entry point, gpt2_op_attention_backward, asks the caller for a
// fp32 workspace of B*H*T floats (it holds D = rowsum(dO * O) between the
// dQ and dK/dV kernels).  Some callers cannot provide one: code that must not
// call cudaMalloc at this point (for example because a memory-pool owner has
// already claimed the device's memory, or because allocation is frozen after
// start-up in the hosting runtime), and callers that only hold the tensors
// they were handed.  This variant takes its workspace from a fixed array in
// the library instead, so it allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (4 MiB) until the process exits.  Host code cannot use the
// array's name as a device address, so every call looks the device address up
// with cudaGetSymbolAddress, with the calling device current.  Looking it up
// on each call (not once per device) keeps the address right after a device
// reset, which reloads the module at a new address.  The first call on a
// device loads the library's module there, so it must come before any stream
// capture.
#include "flash_attn.cuh"

namespace {

constexpr int64_t kMaxRows = GPT2_NOALLOC_ATTN_MAX_ROWS;  // B * H * T

static __device__ __align__(256) float g_attn_scratch[kMaxRows];

// Device address of g_attn_scratch on the current device.
int scratch_for_current_device(float **out) {
    void *p = nullptr;
    GPT2_CUDA_TRY(cudaGetSymbolAddress(&p, g_attn_scratch));
    *out = static_cast<float *>(p);
    return GPT2_OK;
}

}  // namespace

extern "C" int gpt2_op_attention_backward_noalloc(const void *q, const void *kk, const void *v,
                                                  int64_t qkv_row_stride, const void *o, const void *dout,
                                                  int64_t o_row_stride, const float *lse, void *dq, void *dk,
                                                  void *dv, int B, int T, int H, int hd, void *stream) {
    if (!q || !kk || !v || !o || !dout || !lse || !dq || !dk || !dv) return GPT2_ERR_BAD_ARG;
    if (B <= 0 || T <= 0 || H <= 0 || hd != 64 || qkv_row_stride % 8 || o_row_stride % 8) return GPT2_ERR_BAD_SHAPE;
    if ((int64_t)B * H * T > kMaxRows) return GPT2_ERR_BAD_SHAPE;  // workspace limit: B*H*T <= 2^20
    float *scratch = nullptr;
    if (int rc = scratch_for_current_device(&scratch)) return rc;
    // D is written in full by the dQ kernel before the dK/dV kernel reads it,
    // so the array needs no clearing between calls.
    return fa::attention_backward((const bf16 *)q, (const bf16 *)kk, (const bf16 *)v, qkv_row_stride,
                                  (const bf16 *)o, (const bf16 *)dout, o_row_stride, lse, (bf16 *)dq, (bf16 *)dk,
                                  (bf16 *)dv, scratch, B, T, H, hd, (cudaStream_t)stream);
}
