// dequantize.cu -- inverse swizzle + decode (TransformerEngine PR #2763's
// dequantizer unswizzles the pre-swizzled grouped scales before decoding).
// A test helper: one thread per scale block, not on the timed path.
#include "mxg_device.cuh"

namespace mxg {

namespace {

// E4M3 byte -> fp32 (exact; 0x7F / 0xFF -> NaN).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const float m = ue4m3_value(b & 0x7Fu);
  const bool nan = (b & 0x7Fu) == 0x7Fu;
  const float v = nan ? __uint_as_float(0x7FC00000u) : m;
  return (b & 0x80u) ? -v : v;
}

__device__ __forceinline__ float e2m1_value(uint32_t n) {
  const uint32_t e = (n >> 1) & 3u, m = n & 1u;
  const float mag = e == 0 ? 0.5f * m : __uint_as_float(((e + 126u) << 23) | (m << 22));
  return (n & 8u) ? -mag : mag;
}

__device__ __forceinline__ float e8m0_value(uint32_t b) {
  if (b == 0xFFu) return __uint_as_float(0x7FC00000u);
  if (b == 0) return __uint_as_float(0x00400000u);  // 2^-127 (subnormal)
  return __uint_as_float(b << 23);
}

__device__ __forceinline__ void store_out(void* out, int64_t idx, float v, int bf16) {
  if (bf16)
    static_cast<uint16_t*>(out)[idx] = static_cast<uint16_t>(f32_to_bf16_bits(v));
  else
    static_cast<float*>(out)[idx] = v;
}

}  // namespace

// MXFP8.  colwise = 0: q [rows, cols], sf swizzled [rows, cols/32].
//         colwise = 1: q [cols, rows] (transposed copy), sf [cols, rows/32];
//                      out is still [rows, cols].
__global__ void mxfp8_dequantize_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf,
                                        int64_t rows, int64_t cols, int colwise, void* out,
                                        int bf16) {
  const int64_t qrows = colwise ? cols : rows, qcols = colwise ? rows : cols;
  const int64_t nblk = qrows * (qcols >> 5);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nblk;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / (qcols >> 5), c = i % (qcols >> 5);
    const float s = e8m0_value(sf[swz_index(r, c, qcols >> 5)]);
    for (int j = 0; j < 32; ++j) {
      const float v = e4m3_value(q[r * qcols + c * 32 + j]) * s;
      const int64_t orow = colwise ? c * 32 + j : r, ocol = colwise ? r : c * 32 + j;
      store_out(out, orow * cols + ocol, v, bf16);
    }
  }
}

// Row-scaled NVFP4: q packed [rows, cols/2], sf swizzled [rows, cols/16],
// outer [rows] (NULL: 1).
__global__ void nvfp4_dequantize_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf,
                                        const float* __restrict__ outer, int64_t rows, int64_t cols,
                                        void* out, int bf16) {
  const int64_t nblk = rows * (cols >> 4);
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nblk;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / (cols >> 4), c = i % (cols >> 4);
    const float s = ue4m3_value(sf[swz_index(r, c, cols >> 4)] & 0x7Fu);
    const float o = outer ? outer[r] : 1.0f;
    for (int j = 0; j < 16; ++j) {
      const int64_t k = c * 16 + j;
      const uint32_t byte = q[r * (cols >> 1) + (k >> 1)];
      const uint32_t nib = (k & 1) ? (byte >> 4) : (byte & 15u);
      store_out(out, r * cols + k, e2m1_value(nib) * s * o, bf16);
    }
  }
}

cudaError_t launch_dequantize(int nvfp4, int colwise, const uint8_t* q, const uint8_t* sf,
                              const float* outer, int64_t rows, int64_t cols, void* out, int bf16,
                              int num_sms, cudaStream_t stream) {
  const int64_t nblk = nvfp4 ? rows * (cols >> 4) : rows * (cols >> 5);
  if (nblk == 0) return cudaSuccess;
  int64_t grid = (nblk + 255) / 256;
  if (grid > num_sms * 16) grid = num_sms * 16;
  if (nvfp4)
    nvfp4_dequantize_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(q, sf, outer, rows, cols, out,
                                                                      bf16);
  else
    mxfp8_dequantize_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(q, sf, rows, cols, colwise,
                                                                      out, bf16);
  return cudaGetLastError();
}

}  // namespace mxg
