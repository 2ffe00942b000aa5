// quantize_nvfp4.cu -- row-scaled NVFP4 grouped quantize with the per-row
// amax fused in and the swizzled E4M3 block scales written directly.
//
// TransformerEngine PR #3661: a single-launch row-scaled grouped NVFP4 cast
// with fused amax, baking the GEMM's swizzled scale layout into the cast;
// per-row FP32 outer scale amax / (6 * 448) (gemm.py
// _get_nvfp4_tensor_scale_inv), E2M1 data with E4M3 scales per 1x16 block.
// The per-block rule (every step an fp32 round-to-nearest operation):
//   S = 2688 / A_r;  sb = E4M3_RNE_satfinite((amax_b / 6) * S);
//   code = E2M1_RNE_satfinite(x * (S / sb)), signed zeros when sb or A_r = 0.
// Operations are explicit __fdiv_rn / __fmul_rn so the compiler cannot fuse
// or reassociate them.
//
// One warp per row: pass 1 reads the row (32 lanes x 16 bytes per step) for
// the row amax; pass 2 reads it again (from L1/L2) one 16-element block per
// lane, writes 8 packed bytes per lane (256 contiguous bytes per warp step)
// and gathers each run of 4 scale bytes -- which are contiguous in the
// swizzled layout -- into one 32-bit store.
#include "mxg_device.cuh"

namespace mxg {

namespace {

__device__ __forceinline__ int64_t live_rows_warp_nv(const int64_t* ws, int G, int64_t cap,
                                                     int32_t* status) {
  if (ws == nullptr) return cap;
  int64_t sum = 0;
  int32_t bits = 0;
  for (int g = static_cast<int>(lane_id()); g < G; g += 32) {
    int64_t s = ws[g];
    if (s < 0) {
      s = 0;
      bits |= MXG_DEV_NEG_SIZE;
    }
    if (s & 127) {
      s &= ~static_cast<int64_t>(127);
      bits |= MXG_DEV_MISALIGNED;
    }
    sum += s > cap ? cap : s;
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, d);
    bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, d);
  }
  if (sum > cap) {
    sum = cap;
    bits |= MXG_DEV_SUM_OVER_CAPACITY;
  }
  if (lane_id() == 0 && blockIdx.x == 0 && threadIdx.x == 0) status_set(status, bits);
  return sum;
}

__device__ __forceinline__ float amax8(const uint4 v) {
  float a = fmaxf(fabsf(bf16lo(v.x)), fabsf(bf16hi(v.x)));
  a = fmaxf(a, fmaxf(fabsf(bf16lo(v.y)), fabsf(bf16hi(v.y))));
  a = fmaxf(a, fmaxf(fabsf(bf16lo(v.z)), fabsf(bf16hi(v.z))));
  return fmaxf(a, fmaxf(fabsf(bf16lo(v.w)), fabsf(bf16hi(v.w))));
}

// Sign-only E2M1 nibbles of 8 bf16 values (for zero scales).
__device__ __forceinline__ uint32_t sign_nibbles8(const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o |= ((w[i] >> 15) & 1u) << (8 * i + 3);   // low element -> low nibble
    o |= ((w[i] >> 31) & 1u) << (8 * i + 7);   // high element -> high nibble
  }
  return o;
}

__device__ __forceinline__ uint32_t e2m1_8(const uint4 v, float ratio) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o |= cvt_e2m1x2(__fmul_rn(bf16lo(w[i]), ratio), __fmul_rn(bf16hi(w[i]), ratio)) << (8 * i);
  return o;
}

}  // namespace

__global__ void __launch_bounds__(256)
    nvfp4_quantize_kernel(const uint16_t* __restrict__ x, int64_t cap, int64_t cols,
                          const int64_t* __restrict__ group_ws, int G, uint8_t* __restrict__ q,
                          uint8_t* __restrict__ sf, float* __restrict__ outer, int32_t* status) {
  __shared__ int64_t live_s;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  if (warp == 0) {
    const int64_t l = live_rows_warp_nv(group_ws, G, cap, status);
    if (lane == 0) live_s = l;
  }
  __syncthreads();
  const int64_t live = live_s;
  const int64_t nb = cols >> 4;        // 16-element blocks per row
  const int64_t C4 = nb >> 2;          // swizzle tiles per 128-row band

  for (int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + warp; r < live;
       r += static_cast<int64_t>(gridDim.x) * 8) {
    const uint16_t* xr = x + r * cols;
    // pass 1: row amax
    float a = 0.f;
    for (int64_t c = 8 * lane; c < cols; c += 256)
      a = fmaxf(a, amax8(*reinterpret_cast<const uint4*>(xr + c)));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, d));
    const bool zero_row = !(a > 0.f);
    const float S = zero_row ? 0.f : __fdiv_rn(2688.0f, a);
    if (lane == 0) outer[r] = zero_row ? 0.f : __fdiv_rn(a, 2688.0f);

    // pass 2: blocks
    const int64_t rb = (r >> 7) * C4 * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4;
    for (int64_t b0 = 0; b0 < nb; b0 += 32) {
      const int64_t b = b0 + lane;
      const bool act = b < nb;  // nb % 4 == 0: groups of 4 lanes agree
      uint32_t sbyte = 0;
      if (act) {
        const uint4 v0 = *reinterpret_cast<const uint4*>(xr + 16 * b);
        const uint4 v1 = *reinterpret_cast<const uint4*>(xr + 16 * b + 8);
        uint2 o;
        if (!zero_row) {
          const float ab = fmaxf(amax8(v0), amax8(v1));
          const float t = __fmul_rn(__fdiv_rn(ab, 6.0f), S);
          sbyte = cvt_e4m3x2(t, 0.f) & 0x7Fu;
        }
        const float sbv = ue4m3_value(sbyte);
        if (sbv == 0.f) {
          o.x = sign_nibbles8(v0);
          o.y = sign_nibbles8(v1);
        } else {
          const float ratio = __fdiv_rn(S, sbv);
          o.x = e2m1_8(v0, ratio);
          o.y = e2m1_8(v1, ratio);
        }
        *reinterpret_cast<uint2*>(q + r * (cols >> 1) + 8 * b) = o;
      }
      // gather the 4 scale bytes of lanes 4i..4i+3 (consecutive c%4)
      const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 1);
      const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 2);
      const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 3);
      if (act && (lane & 3u) == 0) {
        const uint32_t word = sbyte | (b1 << 8) | (b2 << 16) | (b3 << 24);
        *reinterpret_cast<uint32_t*>(sf + rb + (b >> 2) * 512) = word;
      }
    }
  }
}

cudaError_t launch_nvfp4_quantize(const uint16_t* x, int64_t cap, int64_t cols,
                                  const int64_t* group_ws, int G, uint8_t* q, uint8_t* sf,
                                  float* outer, int32_t* status, int num_sms, cudaStream_t stream) {
  if (cap == 0) return cudaSuccess;
  const int64_t max_ctas = (cap + 7) / 8;
  const int grid = static_cast<int>(max_ctas < num_sms * 8 ? max_ctas : num_sms * 8);
  nvfp4_quantize_kernel<<<grid, 256, 0, stream>>>(x, cap, cols, group_ws, G, q, sf, outer, status);
  return cudaGetLastError();
}

}  // namespace mxg
