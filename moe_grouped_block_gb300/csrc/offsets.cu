// offsets.cu -- group sizes -> [G int64 sizes | G+1 int64 element offsets].
//
// TransformerEngine PR #2763 adds two small kernels for this (an int32 ->
// int64 widening with a multiplier and a single-thread exclusive prefix sum
// of size * last_dim); its review thread suggests a warp-shuffle scan for
// large G.  Here one warp does both in a single pass: each lane widens and
// sanitises one size per round of 32 groups, a shuffle scan forms the
// prefix, and a carry links the rounds.
//
// Sanitisation (this library's contract, recorded in the status word): a
// negative size counts as 0, a size that is not a multiple of 128 is rounded
// down (unless round128 is 0: the unaligned-group entry points keep every
// size), and rows past rows_capacity are dropped.  With P_g the running sum
// of the (non-negative, rounded) sizes, the kept prefix is min(P_g, cap), so
// the kept size of group g is min(P_{g+1}, cap) - min(P_g, cap).
#include "mxg_device.cuh"

namespace mxg {

__global__ void __launch_bounds__(32, 1)
    group_offsets_kernel(const void* __restrict__ sizes, int is_int64, int G, int64_t mult,
                         int64_t last_dim, int64_t cap, int64_t* __restrict__ ws, int32_t* status,
                         int round128) {
  const uint32_t lane = threadIdx.x;
  int64_t carry = 0;  // unclamped running sum before this round
  int32_t bits = 0;
  if (lane == 0) ws[G] = 0;
  for (int base = 0; base < G; base += 32) {
    const int g = base + static_cast<int>(lane);
    int64_t s = 0;
    if (g < G) {
      s = is_int64 ? static_cast<const int64_t*>(sizes)[g]
                   : static_cast<int64_t>(static_cast<const int32_t*>(sizes)[g]);
      if (s < 0) {  // rows = size * multiplier with multiplier >= 1: negative iff size is
        bits |= MXG_DEV_NEG_SIZE;
        s = 0;
      } else if (s > INT64_MAX / mult) {
        // size * multiplier does not fit in 64 bits.  The host bounds
        // multiplier <= 2^31 and cap <= 2^62, so the exact product is far
        // above cap + 127: its rounded value is clamped to cap.  Whether it
        // is a multiple of 128 follows from the factors modulo 128.
        if (round128 && (((s & 127) * (mult & 127)) & 127)) bits |= MXG_DEV_MISALIGNED;
        s = cap;
      } else {
        s *= mult;
        if (round128 && (s & 127)) {
          bits |= MXG_DEV_MISALIGNED;
          s &= ~static_cast<int64_t>(127);
        }
        if (s > cap) s = cap;  // keeps the running sum far from overflow
      }
    }
    // inclusive warp scan of s
    int64_t incl = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= static_cast<uint32_t>(d)) incl += v;
    }
    const int64_t p_before = carry + incl - s, p_after = carry + incl;
    const int64_t kb = p_before < cap ? p_before : cap;
    const int64_t ka = p_after < cap ? p_after : cap;
    if (g < G) {
      if (p_after > cap && s > 0) bits |= MXG_DEV_SUM_OVER_CAPACITY;
      ws[g] = ka - kb;
      ws[G + 1 + g] = ka * last_dim;
    }
    carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  // one atomic per warp
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, d);
  if (lane == 0) status_set(status, bits);
}

cudaError_t launch_group_offsets(const void* sizes, int is_int64, int G, int64_t mult,
                                 int64_t last_dim, int64_t cap, int64_t* ws, int32_t* status,
                                 cudaStream_t stream, int round128) {
  group_offsets_kernel<<<1, 32, 0, stream>>>(sizes, is_int64, G, mult, last_dim, cap, ws, status,
                                             round128);
  return cudaGetLastError();
}

}  // namespace mxg
