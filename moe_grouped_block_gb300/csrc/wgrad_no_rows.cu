// wgrad_no_rows.cu -- grouped wgrad when there are no rows at all.
//
// With M_cap = 0 every group of a wgrad (TransformerEngine gemm.py
// grouped_gemm, wgrad branch: dW[g] over the group's rows) is empty, so each
// dW_g is beta_g * dW_g, or 0 where there is no beta or beta_g is 0: what the
// GEMM epilogue writes for an empty group.  The GEMM kernels cannot run then,
// since the operands have no columns for tensor maps to describe.
#include <algorithm>

#include "mxg_device.cuh"

namespace mxg {

// dW is dense [G, N, K]; per_group = N * K is a multiple of 128 * 128, so
// the bf16 words (two elements each) never straddle two groups.
__global__ void __launch_bounds__(256) wgrad_no_rows_kernel(int64_t per_group, int64_t total,
                                                            const float* __restrict__ beta,
                                                            void* __restrict__ C, int out_bf16) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (out_bf16) {
    uint32_t* c = static_cast<uint32_t*>(C);  // two bf16 per word
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total / 2;
         i += stride) {
      const float b = beta ? beta[(2 * i) / per_group] : 0.0f;
      uint32_t w = 0;  // two bf16 zeros
      if (b != 0.0f) {
        const uint32_t old = c[i];
        w = cvt_bf16x2(0.0f + b * bf16lo(old), 0.0f + b * bf16hi(old));
      }
      c[i] = w;
    }
  } else {
    float* c = static_cast<float*>(C);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += stride) {
      const float b = beta ? beta[i / per_group] : 0.0f;
      c[i] = b != 0.0f ? 0.0f + b * c[i] : 0.0f;
    }
  }
}

cudaError_t launch_wgrad_no_rows(int G, int64_t N, int64_t K, const float* beta, void* C,
                                 int out_bf16, int num_sms, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(G) * N * K;
  const int64_t words = out_bf16 ? total / 2 : total;
  const int64_t blocks = std::min<int64_t>((words + 255) / 256, static_cast<int64_t>(num_sms) * 8);
  wgrad_no_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(N * K, total, beta, C,
                                                                          out_bf16);
  return cudaGetLastError();
}

}  // namespace mxg
