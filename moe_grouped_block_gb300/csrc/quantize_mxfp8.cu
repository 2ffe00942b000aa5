// quantize_mxfp8.cu -- grouped MXFP8 quantize, rowwise and/or colwise
// (transposed), writing the swizzled E8M0 scale layout directly.
//
// TransformerEngine PR #2763 moves the scale swizzle into the grouped
// quantize so the grouped GEMM consumes pre-swizzled scales; gemm.py
// swizzled_scale defines that layout (128x4 scale tiles of 512 bytes, the
// colwise scale matrix transposed first).  Because every group is a multiple
// of 128 rows, the per-group quantize and swizzle of rows [0, live) equal the
// dense ones, so the kernel only needs the live row count from the offsets
// workspace.
//
// Work unit: a 128-row x 128-column tile of bf16 (32 KB read).  Its rowwise
// scales are exactly one 512-byte swizzle tile of sf_row, and its colwise
// scales exactly one 512-byte tile of sf_col, so both are staged in shared
// memory and written as 16-byte stores.
//   phase 1: each half-warp reads one row segment (16 lanes x 16 bytes),
//            a 4-lane shuffle gives the 1x32 block amax, and the E4M3 bytes
//            go straight out (8 bytes per lane, 128 contiguous per row).
//            For the colwise copy the bf16 words are also kept in shared
//            memory (row-major; 16-byte stores are conflict-free per phase).
//   phase 2: thread (column pair, 32-row block) reads 32 words down the
//            tile (a warp reads 32 consecutive words per row: no bank
//            conflicts), forms the 32x1 block amax of both columns and
//            writes 32 contiguous bytes of each transposed row.
#include "mxg_device.cuh"

namespace mxg {

namespace {

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Live rows = sum of the group sizes in the offsets workspace, each taken
// as non-negative and 128-aligned, clamped to the capacity.  Called by warp
// 0; returns the value in every lane.
__device__ __forceinline__ int64_t live_rows_warp(const int64_t* ws, int G, int64_t cap,
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
  if (lane_id() == 0 && blockIdx.x == 0) status_set(status, bits);
  return sum;
}

// 8 bf16 scaled by 2^-e -> 8 E4M3 bytes.
__device__ __forceinline__ uint2 quant8(const uint4 v, float s) {
  uint2 o;
  o.x = cvt_e4m3x2(bf16lo(v.x) * s, bf16hi(v.x) * s) |
        (cvt_e4m3x2(bf16lo(v.y) * s, bf16hi(v.y) * s) << 16);
  o.y = cvt_e4m3x2(bf16lo(v.z) * s, bf16hi(v.z) * s) |
        (cvt_e4m3x2(bf16lo(v.w) * s, bf16hi(v.w) * s) << 16);
  return o;
}

__device__ __forceinline__ float amax8(const uint4 v) {
  float a = fmaxf(fabsf(bf16lo(v.x)), fabsf(bf16hi(v.x)));
  a = fmaxf(a, fmaxf(fabsf(bf16lo(v.y)), fabsf(bf16hi(v.y))));
  a = fmaxf(a, fmaxf(fabsf(bf16lo(v.z)), fabsf(bf16hi(v.z))));
  return fmaxf(a, fmaxf(fabsf(bf16lo(v.w)), fabsf(bf16hi(v.w))));
}

}  // namespace

template <bool ROW, bool COL>
__global__ void __launch_bounds__(256, 3)
    mxfp8_quantize_kernel(const uint16_t* __restrict__ x, int64_t cap, int64_t cols,
                          const int64_t* __restrict__ group_ws, int G, uint8_t* __restrict__ q_row,
                          uint8_t* __restrict__ sf_row, uint8_t* __restrict__ q_col,
                          uint8_t* __restrict__ sf_col, int32_t* status) {
  __shared__ __align__(16) uint32_t tile[COL ? 128 * 64 : 4];  // bf16 pairs, row-major
  __shared__ __align__(16) uint8_t sfr_s[512];
  __shared__ __align__(16) uint8_t sfc_s[512];
  __shared__ int64_t live_s;

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  if (warp == 0) {
    const int64_t l = live_rows_warp(group_ws, G, cap, status);
    if (lane == 0) live_s = l;
  }
  __syncthreads();
  const int64_t kt = cols >> 7;
  const int64_t tiles = (live_s >> 7) * kt;

  const uint32_t half = lane >> 4;  // which row of the pair
  const uint32_t cl = lane & 15u;   // 16-byte chunk: columns 8*cl .. 8*cl+7

  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t m0 = (t / kt) << 7, k0 = (t % kt) << 7;
    const uint16_t* xt = x + m0 * cols + k0 + 8 * cl;

    // ---- phase 1: rows
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t r = (h * 4 + i) * 16 + warp * 2 + half;
        v[i] = ld_stream16(xt + static_cast<int64_t>(r) * cols);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t r = (h * 4 + i) * 16 + warp * 2 + half;
        if (COL) reinterpret_cast<uint4*>(tile)[r * 16 + cl] = v[i];
        if (ROW) {
          float a = amax8(v[i]);
          a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
          a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
          const int e = mx_exponent(a);
          const uint2 o = quant8(v[i], pow2_neg(e));
          *reinterpret_cast<uint2*>(q_row + (m0 + r) * cols + k0 + 8 * cl) = o;
          if ((cl & 3u) == 0) sfr_s[(r & 31u) * 16 + (r >> 5) * 4 + (cl >> 2)] =
              static_cast<uint8_t>(e + 127);
        }
      }
    }
    __syncthreads();
    if (ROW && threadIdx.x < 32) {
      const int64_t atom = (m0 >> 7) * kt + (k0 >> 7);
      reinterpret_cast<uint4*>(sf_row + atom * 512)[threadIdx.x] =
          reinterpret_cast<const uint4*>(sfr_s)[threadIdx.x];
    }

    // ---- phase 2: columns (transposed output)
    if (COL) {
      const uint32_t cp = threadIdx.x & 63u;  // column pair 2cp, 2cp+1
      const uint32_t j = threadIdx.x >> 6;    // 32-row block
      uint32_t w[32];
      float alo = 0.f, ahi = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        w[i] = tile[(32 * j + i) * 64 + cp];
        alo = fmaxf(alo, fabsf(bf16lo(w[i])));
        ahi = fmaxf(ahi, fabsf(bf16hi(w[i])));
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int e = mx_exponent(c ? ahi : alo);
        const float s = pow2_neg(e);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float f0 = (c ? bf16hi(w[4 * i]) : bf16lo(w[4 * i])) * s;
          const float f1 = (c ? bf16hi(w[4 * i + 1]) : bf16lo(w[4 * i + 1])) * s;
          const float f2 = (c ? bf16hi(w[4 * i + 2]) : bf16lo(w[4 * i + 2])) * s;
          const float f3 = (c ? bf16hi(w[4 * i + 3]) : bf16lo(w[4 * i + 3])) * s;
          o[i] = cvt_e4m3x2(f0, f1) | (cvt_e4m3x2(f2, f3) << 16);
        }
        const uint32_t kk = 2 * cp + c;
        uint4* dst = reinterpret_cast<uint4*>(q_col + (k0 + kk) * cap + m0 + 32 * j);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        sfc_s[(kk & 31u) * 16 + (kk >> 5) * 4 + j] = static_cast<uint8_t>(e + 127);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        const int64_t atom = (k0 >> 7) * (cap >> 7) + (m0 >> 7);
        reinterpret_cast<uint4*>(sf_col + atom * 512)[threadIdx.x] =
            reinterpret_cast<const uint4*>(sfc_s)[threadIdx.x];
      }
    }
    __syncthreads();  // shared buffers are reused by the next tile
  }
}

cudaError_t launch_mxfp8_quantize(bool row, bool col, const uint16_t* x, int64_t cap, int64_t cols,
                                  const int64_t* group_ws, int G, uint8_t* q_row, uint8_t* sf_row,
                                  uint8_t* q_col, uint8_t* sf_col, int32_t* status, int num_sms,
                                  cudaStream_t stream) {
  const int64_t max_tiles = (cap >> 7) * (cols >> 7);
  if (max_tiles == 0) return cudaSuccess;
  const int64_t per_sm = col ? 3 : 6;
  const int grid = static_cast<int>(max_tiles < num_sms * per_sm ? max_tiles : num_sms * per_sm);
  if (row && col)
    mxfp8_quantize_kernel<true, true><<<grid, 256, 0, stream>>>(x, cap, cols, group_ws, G, q_row,
                                                                 sf_row, q_col, sf_col, status);
  else if (row)
    mxfp8_quantize_kernel<true, false><<<grid, 256, 0, stream>>>(x, cap, cols, group_ws, G, q_row,
                                                                  sf_row, q_col, sf_col, status);
  else
    mxfp8_quantize_kernel<false, true><<<grid, 256, 0, stream>>>(x, cap, cols, group_ws, G, q_row,
                                                                  sf_row, q_col, sf_col, status);
  return cudaGetLastError();
}

}  // namespace mxg
