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
// Rowwise: rows of up to 7168 columns go through shared memory -- one lane
// brings a whole row in with one bulk copy and a pair of warps works it (the
// row amax, then one 16-element block per lane: 8 packed bytes per lane and
// each run of 4 scale bytes, contiguous in the swizzled layout, as one 32-bit
// store); wider rows take one warp per row that reads the row twice from
// global memory.
// Colwise (the wgrad operands, per-(group, column) outer scale), one launch:
// a CTA owns one group's rows in a 64-column strip; an amax pass streams the
// strip's 256 x 64 TMA tiles and writes the strip's outer scales A / 2688, a
// quantize pass streams them again in reverse order (starting on the tiles
// still in L2) and writes the transposed codes and swizzled scales.
// Products are packed fp32x2 multiplies; four E2M1 conversions fill a word.
#include <algorithm>

#include "mxg_device.cuh"
#include "mxg_host.h"

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

// Two fp32 products with one packed multiply (each rounded to nearest even,
// as two separate multiplies would be).
__device__ __forceinline__ void fmul2_rn(float a0, float a1, float b, float& p0, float& p1) {
  uint64_t x, y, z;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(y) : "f"(b));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(z) : "l"(x), "l"(y));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(p0), "=f"(p1) : "l"(z));
}

// Eight fp32 values -> eight E2M1 codes (RN, satfinite) in one 32-bit word,
// value 2i in the low nibble of byte i: four conversions whose bytes go
// straight into the word (14 % fewer instructions in the colwise kernel
// than widening each byte and merging them).
__device__ __forceinline__ uint32_t e2m1x8_packed(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// E2M1 codes of 8 bf16 values (a row's consecutive elements) times ratio.
__device__ __forceinline__ uint32_t e2m1_8(const uint4 v, float ratio) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float p[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) fmul2_rn(bf16lo(w[i]), bf16hi(w[i]), ratio, p[2 * i], p[2 * i + 1]);
  return e2m1x8_packed(p);
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
    // pass 1: row amax, 8 independent 16-byte loads in flight per lane; the
    // remainder loop covers rows that are not a multiple of 2048 elements
    float a = 0.f;
    int64_t c = 8 * lane;
    for (; c + 7 * 256 < cols; c += 8 * 256) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = *reinterpret_cast<const uint4*>(xr + c + u * 256);
#pragma unroll
      for (int u = 0; u < 8; ++u) a = fmaxf(a, amax8(v[u]));
    }
    for (; c < cols; c += 256) a = fmaxf(a, amax8(*reinterpret_cast<const uint4*>(xr + c)));
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

// ------------------------------------------------------------------------
// Rows staged in shared memory.  A pair of warps owns one row buffer; one
// lane brings a whole row in with a single bulk copy (completing on the
// buffer's mbarrier), so HBM and L2 see every row once and both passes read
// shared memory.  Each warp of the pair reduces half of the row for the row
// amax (combined through shared memory at a pair barrier) and quantizes half
// of its blocks.  The block arithmetic is the one above, step for step; the
// row amax uses the packed bf16 maximum (exact).  The per-block chain (two
// IEEE divisions, then the conversions) is latency bound, so what counts is
// warps per SM: two warps per staged row give 32 warps on the 16 rows that
// fit (measured on the 16384 x 7168 activations: 0.085 ms with 8 warps of
// two buffers each, 0.068 ms with 16 warps of one).  Used for cols <= 7168,
// where two CTAs of 8 rows fit in an SM's shared memory.
// ------------------------------------------------------------------------
constexpr int kNvRowPairs = 8;  // rows in flight per CTA, two warps each
constexpr int64_t kNvRowMaxCols = 7168;

__device__ __forceinline__ float amax8_packed(const uint4 v) {
  const uint32_t m = bf16x2_max_abs(bf16x2_max_abs(v.x, v.y), bf16x2_max_abs(v.z, v.w));
  return fmaxf(__uint_as_float((m & 0x7FFFu) << 16), __uint_as_float(m & 0x7FFF0000u));
}

// Barrier over the 64 threads of warp pair `pair` (named barrier pair + 1).
__device__ __forceinline__ void pair_sync(uint32_t pair) {
  asm volatile("bar.sync %0, 64;" ::"r"(pair + 1) : "memory");
}

// Same, returning whether `ok` holds in every thread of the pair.
__device__ __forceinline__ bool pair_all(uint32_t pair, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %2, 0;\n\t"
      "bar.red.and.pred q, %1, 64, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pair + 1), "r"(ok ? 1u : 0u)
      : "memory");
  return r != 0;
}

__global__ void __launch_bounds__(64 * kNvRowPairs, 2)
    nvfp4_quantize_rows_smem_kernel(const uint16_t* __restrict__ x, int64_t cap, int64_t cols,
                                    const int64_t* __restrict__ group_ws, int G,
                                    uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                    float* __restrict__ outer, int32_t* status) {
  extern __shared__ __align__(128) uint8_t nsm[];
  __shared__ uint64_t bars[kNvRowPairs];
  __shared__ float part[kNvRowPairs][2];
  __shared__ int64_t live_s;
  __shared__ int abort_s;
  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const uint32_t pair = warp >> 1, half = warp & 1u;
  const bool leader = half == 0 && lane == 0;
  const uint32_t row_bytes = static_cast<uint32_t>(cols * 2);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNvRowPairs; ++i) mbar_init(smem_u32(&bars[i]), 1);
    abort_s = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    const int64_t l = live_rows_warp_nv(group_ws, G, cap, status);
    if (lane == 0) live_s = l;
  }
  __syncthreads();
  const int64_t live = live_s;
  const int64_t nb = cols >> 4;   // 16-element blocks per row (a multiple of 8)
  const int64_t C4 = nb >> 2;     // swizzle tiles per 128-row band
  const int64_t hb = nb >> 1;     // blocks per warp of the pair (a multiple of 4)
  const int64_t hc = cols >> 4;   // 16-byte chunks per warp of the pair (cols / 8 / 2)
  volatile int* abort_flag = &abort_s;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kNvRowPairs;
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kNvRowPairs + pair;
  uint8_t* buf = nsm + static_cast<size_t>(pair) * row_bytes;
  const uint32_t bar = smem_u32(&bars[pair]);
  auto issue = [&](int64_t r) {
    mbar_arrive_expect_tx(bar, row_bytes);
    bulk_load(smem_u32(buf), x + r * cols, row_bytes, bar);
  };
  if (leader && r0 < live) issue(r0);
  uint32_t parity = 0u;
  bool pending = r0 < live;
  for (int64_t r = r0; r < live; r += stride) {
    // both warps of the pair take the same decision, so neither is left at a
    // pair barrier the other never reaches
    if (!pair_all(pair, mbar_wait(bar, parity, abort_flag, status))) break;
    parity ^= 1u;
    pending = false;
    const uint4* row = reinterpret_cast<const uint4*>(buf);
    // pass 1: row amax (this warp's half of the chunks, then the pair's)
    float a = 0.f;
    for (int64_t c = half * hc + lane; c < (half + 1) * hc; c += 32) a = fmaxf(a, amax8_packed(row[c]));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, d));
    if (lane == 0) part[pair][half] = a;
    pair_sync(pair);
    a = fmaxf(part[pair][0], part[pair][1]);
    const bool zero_row = !(a > 0.f);
    const float S = zero_row ? 0.f : __fdiv_rn(2688.0f, a);
    if (leader) outer[r] = zero_row ? 0.f : __fdiv_rn(a, 2688.0f);
    // pass 2: this warp's half of the blocks (lane = block within a run of 32)
    const int64_t rb = (r >> 7) * C4 * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4;
    const int64_t bend = (half + 1) * hb;
    for (int64_t b0 = half * hb; b0 < bend; b0 += 32) {
      const int64_t blk = b0 + lane;
      const bool act = blk < bend;  // hb % 4 == 0: groups of 4 lanes agree
      uint32_t sbyte = 0;
      if (act) {
        const uint4 v0 = row[2 * blk], v1 = row[2 * blk + 1];
        uint2 o;
        if (!zero_row) {
          const float ab = fmaxf(amax8_packed(v0), amax8_packed(v1));
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
        *reinterpret_cast<uint2*>(q + r * (cols >> 1) + 8 * blk) = o;
      }
      const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 1);
      const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 2);
      const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 3);
      if (act && (lane & 3u) == 0)
        *reinterpret_cast<uint32_t*>(sf + rb + (blk >> 2) * 512) =
            sbyte | (s1 << 8) | (s2 << 16) | (s3 << 24);
    }
    // both warps are done with the buffer (and part[]) before it is refilled
    fence_proxy_async_shared();
    pair_sync(pair);
    if (leader && r + stride < live) {
      issue(r + stride);
      pending = true;
    }
  }
  // a copy still in flight (only after an abort) lands before the CTA exits
  if (leader && pending) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
      if (globaltimer() - t0 > kWaitTimeoutNs) break;
  }
}

// ------------------------------------------------------------------------
// Colwise (transposed) row-scaled NVFP4: the copy wgrad consumes (PR #3661
// sizes the columnwise amax per column and splits it per expert).  For group
// g and column k the outer scale is A[g,k] / 2688 with A the column amax over
// the group's rows; R2 then runs down the column in 16-row blocks.  Output
// qT[k, m/2] (rows m, m+1 in the low / high nibble), E4M3 scales swizzled
// over [cols, cap/16], outer [G, cols].
//
// One launch.  A work unit is one group's rows in a strip of 64 columns, and
// one CTA owns it whole: pass 1 streams the strip's 256-row tiles (32 KB; TMA,
// a ring of three buffers, two loads ahead) for the column amax and writes
// the outer scales; pass 2 streams the same tiles again, in reverse order,
// and quantizes, finding most of them still in L2.  So the input crosses
// HBM about once and a half instead of twice, and no atomics, no zeroing or
// finishing launch and no wait on another CTA are needed.  Units are dealt
// to the CTAs in rounds, forwards and backwards in turn, over the groups
// sorted by size (up to 64 groups; unsorted beyond), so that every CTA gets
// about the same number of rows.  (Measured against it and slower: 32- and
// size-dependent strip widths, deeper buffer rings with one CTA per SM, and
// three CTAs per SM with two buffers.)
// ------------------------------------------------------------------------

// Sanitised row offsets of the groups into shared memory (warp 0).
__device__ __forceinline__ void build_row_offsets(const int64_t* ws, int G, int64_t cap,
                                                  int64_t* row_off) {
  const uint32_t lane = lane_id();
  if (ws == nullptr) {
    if (lane == 0) {
      row_off[0] = 0;
      row_off[1] = cap;
    }
    return;
  }
  int64_t carry = 0;
  for (int base = 0; base < G; base += 32) {
    const int g = base + static_cast<int>(lane);
    int64_t s = 0;
    if (g < G) {
      s = ws[g];
      s = s < 0 ? 0 : (s & ~static_cast<int64_t>(127));
      s = s > cap ? cap : s;
    }
    int64_t incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= static_cast<uint32_t>(d)) incl += v;
    }
    if (g < G) row_off[g] = min(carry + incl - s, cap);
    carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  if (lane == 0) row_off[G] = min(carry, cap);
}

constexpr int kNvsCols = 64;                       // columns of a strip (128-byte rows)
constexpr int kNvsRows = 256;                      // rows of a tile (one TMA box)
constexpr int kNvsPairs = kNvsCols / 2;            // column pairs: the lanes of a warp
constexpr int kNvsTileBytes = kNvsRows * kNvsCols * 2;
constexpr int kNvsBufs = 3;                        // tile buffers: loads run 2 tiles ahead
constexpr int kNvsSortMax = 64;                    // groups sorted by size up to this many
// dynamic shared memory: the tile ring, alignment slack; then the row offsets
// (G + 1 int64) and the unit order (G int32)
constexpr int kNvsSmem = kNvsBufs * kNvsTileBytes + 1024;

// A unit of the colwise quantize: group g's rows [r0, r0 + rows) in the
// 64-column strip at k0, and its tiles.
struct StripUnit {
  int64_t r0, rows, k0;
  int g, nt;
};

// An unsigned E4M3 byte -> its value, exactly, by the hardware conversion to
// f16 (every E4M3 value is an f16 value): fewer instructions than decoding
// the bits.
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2;
  float v;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(byte & 0xFFu)));
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}"
      : "=f"(v)
      : "r"(h2));
  return v;
}

__global__ void __launch_bounds__(256)
    nvfp4_col_strip_kernel(const __grid_constant__ CUtensorMap tmap_x, int64_t cap, int64_t cols,
                           const int64_t* __restrict__ ws, int G, float* __restrict__ outer,
                           uint8_t* __restrict__ qT, uint8_t* __restrict__ sfT) {
  extern __shared__ uint8_t nsm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(nsm_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bars[kNvsBufs];
  __shared__ int abort_s;
  __shared__ uint32_t red[256];  // pass 1: per (slice, column pair), packed |x| max
  __shared__ float Ss[kNvsCols], As[kNvsCols];
  __shared__ float sixth[128];  // sixth[M - 128] = RN(M / 6) for the 8-bit significands M
  const int Gt = ws ? G : 1;
  int64_t* row_off = reinterpret_cast<int64_t*>(sm + kNvsBufs * kNvsTileBytes);
  int32_t* order = reinterpret_cast<int32_t*>(row_off + Gt + 1);
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
  if (tid == 0) {
    for (int i = 0; i < kNvsBufs; ++i) mbar_init(smem_u32(&bars[i]), 1);
    abort_s = 0;
    fence_barrier_init();
  }
  if (warp == 0) build_row_offsets(ws, G, cap, row_off);
  if (tid < 128) sixth[tid] = __fdiv_rn(static_cast<float>(128 + tid), 6.0f);
  __syncthreads();
  if (warp == 0) {  // units go largest group first (ties: group index)
    for (int g = static_cast<int>(lane); g < Gt; g += 32) {
      int rank = g;
      if (Gt <= kNvsSortMax) {
        const int64_t sg = row_off[g + 1] - row_off[g];
        rank = 0;
        for (int h = 0; h < Gt; ++h) {
          const int64_t sh = row_off[h + 1] - row_off[h];
          rank += (sh > sg || (sh == sg && h < g)) ? 1 : 0;
        }
      }
      order[rank] = g;
    }
  }
  __syncthreads();
  volatile int* abort_flag = &abort_s;
  const uint32_t S = static_cast<uint32_t>(cols / kNvsCols);
  const uint32_t units = static_cast<uint32_t>(Gt) * S;
  const uint32_t P = gridDim.x, c = blockIdx.x;
  // the CTA's n-th unit: rounds of P units dealt forwards in even rounds and
  // backwards in odd ones; false past the last
  auto unit_of = [&](uint32_t n, StripUnit& u) -> bool {
    const uint32_t i = n * P + ((n & 1u) ? P - 1 - c : c);
    if (i >= units) return false;
    u.g = order[i / S];
    u.k0 = static_cast<int64_t>(i % S) * kNvsCols;
    u.r0 = row_off[u.g];
    u.rows = row_off[u.g + 1] - u.r0;
    u.nt = static_cast<int>((u.rows + kNvsRows - 1) / kNvsRows);
    return true;
  };

  // Thread 0's load cursor runs kNvsBufs - 1 tiles ahead of the work: unit
  // an (decoded in au), tile ordinal aj within it (pass 1: tiles 0..nt-1,
  // then pass 2: tiles nt-1..0).
  uint32_t an = 0;
  int aj = 0;
  StripUnit au;
  bool ahead = false;
  auto ahead_first = [&]() {  // the first unit with rows at or after an
    for (;; ++an) {
      if (!unit_of(an, au)) return false;
      if (au.rows > 0) return true;
    }
  };
  auto issue = [&](int b) {
    const int64_t j = aj < au.nt ? aj : 2 * au.nt - 1 - aj;
    const uint32_t bar = smem_u32(&bars[b]);
    mbar_arrive_expect_tx(bar, kNvsTileBytes);
    tma_load_2d(smem_u32(sm + b * kNvsTileBytes), &tmap_x, bar, static_cast<int32_t>(au.k0),
                static_cast<int32_t>(au.r0 + j * kNvsRows));
    if (++aj == 2 * au.nt) {
      aj = 0;
      ++an;
      ahead = ahead_first();
    }
  };
  uint32_t parity = 0u, pending = 0u;
  if (tid == 0) {
    ahead = ahead_first();
    if (ahead) prefetch_tmap(&tmap_x);
    for (int i = 0; i < kNvsBufs - 1 && ahead; ++i) {
      issue(i);
      pending |= 1u << i;
    }
  }

  int b = 0;
  const int64_t C4 = cap >> 6;  // swizzle tiles per 128-column band along the rows
  // thread: column pair cp (columns 2 cp, 2 cp + 1 of the strip), rows
  // 32 slice .. 32 slice + 31 of every tile
  const uint32_t cp = tid % kNvsPairs, slice = tid / kNvsPairs;
  StripUnit u;
  for (uint32_t n = 0; unit_of(n, u); ++n) {
    if (u.rows == 0) {  // a group without rows: its outer scales are 0
      if (tid < kNvsCols) outer[static_cast<int64_t>(u.g) * cols + u.k0 + tid] = 0.0f;
      continue;
    }
    uint32_t colmax = 0;  // pass 1 running packed maximum
    for (int job = 0; job < 2 * u.nt; ++job) {
      if (!mbar_wait(smem_u32(&bars[b]), (parity >> b) & 1u, abort_flag, nullptr)) *abort_flag = 1;
      parity ^= 1u << b;
      pending &= ~(1u << b);
      __syncthreads();  // the previous job's buffer is free; Ss / As of this unit are set (pass 2)
      if (*abort_flag) break;
      if (tid == 0 && ahead) {
        const int bl = (b + kNvsBufs - 1) % kNvsBufs;  // the previous job's buffer
        issue(bl);
        pending |= 1u << bl;
      }
      const bool pass1 = job < u.nt;
      const int64_t j = pass1 ? job : 2 * u.nt - 1 - job;
      const int64_t valid = min(static_cast<int64_t>(kNvsRows), u.rows - j * kNvsRows);
      const uint32_t* tile = reinterpret_cast<const uint32_t*>(sm + b * kNvsTileBytes);
      if (pass1) {
        // column maximum of |x| over this thread's 32 rows, both columns of
        // the pair at once (packed bf16, exact)
        if (static_cast<int64_t>(32 * slice) < valid) {
#pragma unroll 8
          for (int i = 0; i < 32; ++i)
            colmax = bf16x2_max_abs(colmax, tile[(32 * slice + i) * kNvsPairs + cp]);
        }
        if (job + 1 == u.nt) {
          red[tid] = colmax & 0x7FFF7FFFu;  // = red[slice * kNvsPairs + cp]
          __syncthreads();
          if (tid < kNvsCols) {
            uint32_t m = 0;
#pragma unroll
            for (int q = 0; q < 256 / kNvsPairs; ++q) m = bf16x2_max_abs(m, red[q * kNvsPairs + (tid >> 1)]);
            const float A = (tid & 1) ? bf16hi(m & 0x7FFF7FFFu) : bf16lo(m & 0x7FFF7FFFu);
            As[tid] = A;
            Ss[tid] = A > 0.f ? __fdiv_rn(2688.0f, A) : 0.f;
            outer[static_cast<int64_t>(u.g) * cols + u.k0 + tid] =
                A > 0.f ? __fdiv_rn(A, 2688.0f) : 0.0f;
          }
          // Ss / As are read in pass 2, after the next job's barrier
        }
      } else if (static_cast<int64_t>(32 * slice) < valid) {
        // columns 2 cp, 2 cp + 1 (one 32-bit word), rows 32 slice .. 32 slice
        // + 31 of the tile: two 16-row blocks of each column
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = tile[(32 * slice + i) * kNvsPairs + cp];
        uint32_t bm[2];  // block maxima of |x|, both columns packed (exact)
#pragma unroll
        for (int bk = 0; bk < 2; ++bk) {
          uint32_t mm = 0;
#pragma unroll
          for (int i = 0; i < 16; ++i) mm = bf16x2_max_abs(mm, w[16 * bk + i]);
          bm[bk] = mm & 0x7FFF7FFFu;
        }
        const int64_t m = u.r0 + j * kNvsRows + 32 * slice;  // first row
        const int64_t cb = m >> 4;                     // first 16-row block (even)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const uint32_t kc = 2 * cp + cc;
          const float A = As[kc], Sv = Ss[kc];
          const bool zero = !(A > 0.f);
          uint32_t o[4];
          uint32_t sword = 0;
#pragma unroll
          for (int bk = 0; bk < 2; ++bk) {
            const float ab = cc ? bf16hi(bm[bk]) : bf16lo(bm[bk]);
            uint32_t sbyte = 0;
            if (!zero) {
              // RN(ab / 6): ab is a bf16 value, M * 2^E with an 8-bit significand
              // M; for ab >= 2^-123 the quotient is a normal fp32 and equals
              // RN(M / 6) * 2^E exactly (a power-of-two scaling commutes with
              // rounding), so the table entry is scaled instead of dividing
              const uint32_t ub = __float_as_uint(ab);
              const uint32_t ex = ub >> 23;  // biased exponent (ab >= 0)
              const float q6 = ex >= 4u ? __uint_as_float(__float_as_uint(sixth[(ub >> 16) & 127u]) +
                                                          ((ex - 134u) << 23))
                                        : __fdiv_rn(ab, 6.0f);
              sbyte = cvt_e4m3x2(__fmul_rn(q6, Sv), 0.f) & 0x7Fu;
            }
            const float sbv = e4m3_to_f32(sbyte);
#pragma unroll
            for (int h = 0; h < 2; ++h) o[2 * bk + h] = 0;
            if (sbv == 0.f) {  // codes are the signs of x
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const uint32_t w0 = w[16 * bk + 8 * h + 2 * i], w1 = w[16 * bk + 8 * h + 2 * i + 1];
                  const uint32_t s0 = cc ? (w0 >> 31) : ((w0 >> 15) & 1u);
                  const uint32_t s1 = cc ? (w1 >> 31) : ((w1 >> 15) & 1u);
                  o[2 * bk + h] |= ((s0 << 3) | (s1 << 7)) << (8 * i);
                }
            } else {
              const float ratio = __fdiv_rn(Sv, sbv);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                float pp[8];  // the products of rows 8h .. 8h + 7 of the block
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const uint32_t w0 = w[16 * bk + 8 * h + 2 * i], w1 = w[16 * bk + 8 * h + 2 * i + 1];
                  fmul2_rn(cc ? bf16hi(w0) : bf16lo(w0), cc ? bf16hi(w1) : bf16lo(w1), ratio,
                           pp[2 * i], pp[2 * i + 1]);
                }
                o[2 * bk + h] = e2m1x8_packed(pp);
              }
            }
            sword |= sbyte << (8 * bk);
          }
          const int64_t k = u.k0 + kc;
          *reinterpret_cast<uint4*>(qT + k * (cap >> 1) + (m >> 1)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint16_t*>(sfT + ((k >> 7) * C4 + (cb >> 2)) * 512 + (k & 31) * 16 +
                                       ((k & 127) >> 5) * 4 + (cb & 3)) = static_cast<uint16_t>(sword);
        }
      }
      b = (b + 1) % kNvsBufs;
    }
    if (*abort_flag) break;
  }
  // a load still in flight (only after an abort) lands before the CTA exits
  if (tid == 0)
    for (int bb = 0; bb < kNvsBufs; ++bb)
      if (pending & (1u << bb)) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&bars[bb]), (parity >> bb) & 1u))
          if (globaltimer() - t0 > kWaitTimeoutNs) break;
      }
}

cudaError_t launch_nvfp4_quantize_colwise(const uint16_t* x, int64_t cap, int64_t cols,
                                          const int64_t* group_ws, int G, uint8_t* qT,
                                          uint8_t* sfT, float* outer, int num_sms,
                                          cudaStream_t stream) {
  const int Gt = group_ws ? G : 1;
  CUtensorMap tm;
  if (!make_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, static_cast<uint64_t>(cols),
                    static_cast<uint64_t>(cap), static_cast<uint64_t>(cols) * 2, kNvsCols, kNvsRows,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  auto kern = nvfp4_col_strip_kernel;
  const int smem = kNvsSmem + 8 * (Gt + 1) + 4 * Gt;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // persistent grid: as many CTAs as are resident at once, at most one per unit
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t units = static_cast<int64_t>(Gt) * (cols / kNvsCols);
  const int grid = static_cast<int>(std::min<int64_t>(units, static_cast<int64_t>(num_sms) * per_sm));
  kern<<<grid, 256, smem, stream>>>(tm, cap, cols, group_ws, G, outer, qT, sfT);
  return cudaGetLastError();
}

cudaError_t launch_nvfp4_quantize(const uint16_t* x, int64_t cap, int64_t cols,
                                  const int64_t* group_ws, int G, uint8_t* q, uint8_t* sf,
                                  float* outer, int32_t* status, int num_sms, cudaStream_t stream) {
  if (cap == 0) return cudaSuccess;
  if (cols <= kNvRowMaxCols) {  // one row per warp pair in shared memory
    const size_t smem = static_cast<size_t>(kNvRowPairs) * static_cast<size_t>(cols) * 2;
    auto kern = nvfp4_quantize_rows_smem_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 64 * kNvRowPairs, smem) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    const int64_t max_ctas = (cap + kNvRowPairs - 1) / kNvRowPairs;
    const int64_t full = static_cast<int64_t>(num_sms) * per_sm;
    const int grid = static_cast<int>(max_ctas < full ? max_ctas : full);
    kern<<<grid, 64 * kNvRowPairs, smem, stream>>>(x, cap, cols, group_ws, G, q, sf, outer,
                                                   status);
    return cudaGetLastError();
  }
  const int64_t max_ctas = (cap + 7) / 8;
  const int grid = static_cast<int>(max_ctas < num_sms * 8 ? max_ctas : num_sms * 8);
  nvfp4_quantize_kernel<<<grid, 256, 0, stream>>>(x, cap, cols, group_ws, G, q, sf, outer, status);
  return cudaGetLastError();
}

}  // namespace mxg
