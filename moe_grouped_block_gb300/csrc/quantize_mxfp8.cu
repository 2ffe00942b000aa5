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
// scales exactly one 512-byte tile of sf_col; each thread writes its scale
// bytes straight to their swizzled places.
//   load:    one thread issues the TMA copies (two 64-column boxes with the
//            128-byte swizzle) of the CTA's next tile into the second of two
//            shared-memory buffers while all threads work on the current one,
//            so a tile's HBM latency overlaps the previous tile's arithmetic
//            and stores; one __syncthreads per tile.
//   phase 1: a lane owns one 1x32 block: four 16-byte loads (the 8 lanes of a
//            load phase read 8 rows of one block, 8 distinct swizzled chunk
//            positions: conflict-free), its amax and scale, one 32-byte store.
//   phase 2: thread (column pair, 32-row block) walks 32 words down the tile
//            twice through precomputed swizzled offsets (a warp reads 32
//            distinct chunk words per row: no bank conflicts) -- once for the
//            32x1 block amax of both columns, once to quantize -- and writes
//            32 contiguous bytes of each transposed row.
//   arithmetic: amax and the scaling by 2^-e run on packed bf16 pairs.  The
//            maximum of magnitudes is exact; so is the product by a power of
//            two whenever it is a normal bf16 (|x| 2^-e <= 448 bounds it
//            above), and a product below the normal range is under 2^-126,
//            which the E4M3 conversion takes to a signed zero in any case.
//            Only that final conversion goes through fp32.
#include "mxg_device.cuh"
#include "mxg_host.h"

namespace mxg {

namespace {

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

// Unaligned groups: one warp builds row_off (data rows: sizes taken as
// non-negative, the running sum capped at cap), prow_off (each kept size
// rounded up to 128: the padded row where the group's scales and colwise slab
// start) and tile_off (128-row tiles per group, prefix) in shared memory.
__device__ __forceinline__ void unaligned_tables_warp(const int64_t* ws, int G, int64_t cap,
                                                      int32_t* row_off, int32_t* prow_off,
                                                      int32_t* tile_off, int32_t* status) {
  const uint32_t lane = lane_id();
  auto scan = [&](int64_t v) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t u = __shfl_up_sync(0xFFFFFFFFu, v, d);
      if (lane >= static_cast<uint32_t>(d)) v += u;
    }
    return v;
  };
  int64_t carry = 0, carry_pad = 0;
  int32_t bits = 0;
  for (int base = 0; base < G; base += 32) {
    const int g = base + static_cast<int>(lane);
    int64_t s = 0;
    if (g < G) {
      s = ws[g];
      if (s < 0) {
        s = 0;
        bits |= MXG_DEV_NEG_SIZE;
      }
      if (s > cap) s = cap;
    }
    const int64_t incl = scan(s);
    const int64_t before = min(carry + incl - s, cap), after = min(carry + incl, cap);
    if (carry + incl > cap && s > 0) bits |= MXG_DEV_SUM_OVER_CAPACITY;
    const int64_t pad = ((after - before) + 127) & ~static_cast<int64_t>(127);
    const int64_t pincl = scan(pad);
    if (g < G) {
      row_off[g] = static_cast<int32_t>(before);
      prow_off[g] = static_cast<int32_t>(carry_pad + pincl - pad);
      tile_off[g] = static_cast<int32_t>((carry_pad + pincl - pad) >> 7);
    }
    carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    carry_pad += __shfl_sync(0xFFFFFFFFu, pincl, 31);
  }
  if (lane == 0) {
    row_off[G] = static_cast<int32_t>(min(carry, cap));
    prow_off[G] = static_cast<int32_t>(carry_pad);
    tile_off[G] = static_cast<int32_t>(carry_pad >> 7);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, d);
  if (lane == 0 && blockIdx.x == 0) status_set(status, bits);
}

// Largest g with tile_off[g] <= rt (binary search over G + 1 entries).
__device__ __forceinline__ int group_of_tile(const int32_t* tile_off, int G, int64_t rt) {
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tile_off[mid] <= rt)
      lo = mid;
    else
      hi = mid;
  }
  return lo;
}

// Scaled bf16 pair (already multiplied by 2^-e, exact) -> two E4M3 bytes.
__device__ __forceinline__ uint32_t e4m3_pair(uint32_t w) { return cvt_e4m3x2(bf16lo(w), bf16hi(w)); }

// 8 bf16 (one row chunk) scaled by the packed power of two s2 -> 8 E4M3 bytes.
__device__ __forceinline__ uint2 quant8(const uint4 v, uint32_t s2) {
  uint2 o;
  o.x = e4m3_pair(bf16x2_mul(v.x, s2)) | (e4m3_pair(bf16x2_mul(v.y, s2)) << 16);
  o.y = e4m3_pair(bf16x2_mul(v.z, s2)) | (e4m3_pair(bf16x2_mul(v.w, s2)) << 16);
  return o;
}

// |x| of the low / high bf16 of a packed value, as fp32 (exact).
__device__ __forceinline__ float abs_lo(uint32_t m) { return __uint_as_float((m & 0x7FFFu) << 16); }
__device__ __forceinline__ float abs_hi(uint32_t m) { return __uint_as_float(m & 0x7FFF0000u); }

}  // namespace

// Shared memory: two 32 KB bf16 tiles (TMA double buffer), two mbarriers, the
// live-row count and the abort flag; with unaligned groups, three int32
// tables of G + 1 entries after them.
constexpr int kQTileBytes = 128 * 128 * 2;
constexpr int kQSmemBytes = 2 * kQTileBytes + 2 * 8 + 16 + 1024;

// UNA: group sizes of any value.  Tiles are then 128-row tiles of each group
// (the last one may extend past the group: those rows are zeroed in shared
// memory after the load), written densely to q_row but at the group's padded
// row offset in sf_row, q_col and sf_col; cap_col is the row count of the
// colwise copy (cap, or cap + 128 G when padded).
template <bool ROW, bool COL, bool UNA>
__global__ void __launch_bounds__(256, 3)
    mxfp8_quantize_kernel(const __grid_constant__ CUtensorMap tmap_x, int64_t cap, int64_t cols,
                          const int64_t* __restrict__ group_ws, int G, uint8_t* __restrict__ q_row,
                          uint8_t* __restrict__ sf_row, uint8_t* __restrict__ q_col,
                          uint8_t* __restrict__ sf_col, int qcol_v8, int qrow_v8, int64_t cap_col,
                          int32_t* status) {
  extern __shared__ uint8_t qsmem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsmem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + 2 * kQTileBytes);
  int64_t* live_s = reinterpret_cast<int64_t*>(bars + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(live_s + 1);
  int32_t* row_off = reinterpret_cast<int32_t*>(live_s + 2);  // UNA only
  int32_t* prow_off = row_off + (G + 1);
  int32_t* tile_off = prow_off + (G + 1);

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    if (UNA) {
      unaligned_tables_warp(group_ws, G, cap, row_off, prow_off, tile_off, status);
      if (lane == 0) *live_s = 0;
    } else {
      const int64_t l = live_rows_warp(group_ws, G, cap, status);
      if (lane == 0) *live_s = l;
    }
  }
  __syncthreads();
  const int64_t kt = cols >> 7;
  const int64_t row_tiles = UNA ? static_cast<int64_t>(tile_off[G]) : (*live_s >> 7);
  const int64_t tiles = row_tiles * kt;
  // row tile rt -> first data row, first padded row, rows of the group in it
  struct RowTile {
    int64_t m0, mp;
    int valid;
  };
  auto row_tile = [&](int64_t rt) {
    RowTile r;
    if (UNA) {
      const int g = group_of_tile(tile_off, G, rt);
      const int64_t i = rt - tile_off[g];
      r.m0 = row_off[g] + 128 * i;
      r.mp = prow_off[g] + 128 * i;
      const int64_t left = row_off[g + 1] - r.m0;
      r.valid = static_cast<int>(left < 128 ? left : 128);
    } else {
      r.m0 = r.mp = rt << 7;
      r.valid = 128;
    }
    return r;
  };

  // thread 0 issues the TMA loads of tile t into buffer b: two 64-column
  // boxes (128 rows x 128 bytes each, 128-byte swizzle: 16-byte chunk c of row
  // r sits at chunk position c ^ (r & 7))
  auto issue = [&](int64_t t, int b) {
    const uint32_t bar = smem_u32(&bars[b]);
    const int32_t x0 = static_cast<int32_t>((t % kt) << 7);
    const int32_t y = static_cast<int32_t>(row_tile(t / kt).m0);
    mbar_arrive_expect_tx(bar, kQTileBytes);
    tma_load_2d(smem_u32(sm + b * kQTileBytes), &tmap_x, bar, x0, y);
    tma_load_2d(smem_u32(sm + b * kQTileBytes + kQTileBytes / 2), &tmap_x, bar, x0 + 64, y);
  };
  if (threadIdx.x == 0 && static_cast<int64_t>(blockIdx.x) < tiles) {
    prefetch_tmap(&tmap_x);
    issue(blockIdx.x, 0);
  }

  uint32_t parity = 0u;  // bit b: phase parity of buffer b
  uint32_t pending = static_cast<int64_t>(blockIdx.x) < tiles ? 1u : 0u;  // thread 0's loads
  int b = 0;
  // One __syncthreads per tile: once every thread has passed it, the previous
  // tile's buffer is no longer read, so thread 0 refills it with the tile
  // after this one; the scale bytes go straight to their swizzled positions in
  // global memory (no staging, no second barrier).
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x, b ^= 1) {
    if (!mbar_wait(smem_u32(&bars[b]), (parity >> b) & 1u, abort_flag, status)) *abort_flag = 1;
    parity ^= 1u << b;
    pending &= ~(1u << b);
    __syncthreads();
    if (*abort_flag) break;
    if (threadIdx.x == 0 && t + gridDim.x < tiles) {
      issue(t + gridDim.x, b ^ 1);
      pending |= 1u << (b ^ 1);
    }

    const RowTile rtl = row_tile(t / kt);
    const int64_t m0 = rtl.m0, mp = rtl.mp, k0 = (t % kt) << 7;
    const uint32_t* tile = reinterpret_cast<const uint32_t*>(sm + b * kQTileBytes);
    if (UNA && rtl.valid < 128) {
      // rows past the group: zeros (their scales come out 0, their colwise
      // bytes are the padding); ordered before the buffer's next TMA write
      uint32_t* wt = reinterpret_cast<uint32_t*>(sm + b * kQTileBytes);
      for (int w = static_cast<int>(threadIdx.x); w < 128 * 64; w += 256)
        if (((w & 4095) >> 5) >= rtl.valid) wt[w] = 0;  // word w: box w >> 12, row (w >> 5) & 127
      fence_proxy_async_shared();
      __syncthreads();
    }

    // ---- phase 1: rows.  A lane owns one 32-element block (row r, block blk):
    // four 16-byte loads, its own amax and scale, one 32-byte store.  The 8
    // lanes of each 8-lane phase read 8 rows of one block: 8 different chunk
    // positions under the swizzle, so the loads are conflict-free.
    if (ROW) {
      uint8_t* sfr = sf_row + ((mp >> 7) * kt + (k0 >> 7)) * 512;  // this tile's scale tile
      const uint32_t rl = lane & 7u, blk = lane >> 3;
      const uint4* box = reinterpret_cast<const uint4*>(tile + (blk >> 1) * 4096);
      const uint32_t c0 = (blk & 1u) * 4u;  // the block's first chunk in its 128-byte row
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint32_t r = static_cast<uint32_t>(i) * 64u + warp * 8u + rl;
        uint4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = box[r * 8 + ((c0 + q) ^ (r & 7u))];
        uint32_t m = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          m = bf16x2_max_abs(m, bf16x2_max_abs(bf16x2_max_abs(v[q].x, v[q].y),
                                               bf16x2_max_abs(v[q].z, v[q].w)));
        const int e = mx_exponent(fmaxf(abs_lo(m), abs_hi(m)));
        const uint32_t sb = bf16_pow2_neg_bits(e), s2 = sb | (sb << 16);
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint2 h = quant8(v[q], s2);
          o[2 * q] = h.x;
          o[2 * q + 1] = h.y;
        }
        if (!UNA || static_cast<int>(r) < rtl.valid) {
          uint8_t* dst = q_row + (m0 + r) * cols + k0 + 32 * blk;
          if (qrow_v8) {
            st_global_32B(dst, o);
          } else {
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
            reinterpret_cast<uint4*>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        sfr[(r & 31u) * 16 + (r >> 5) * 4 + blk] = static_cast<uint8_t>(e + 127);
      }
    }

    // ---- phase 2: columns (transposed output)
    if (COL) {
      const uint32_t cp = threadIdx.x & 63u;  // column pair 2cp, 2cp+1 (one 32-bit word)
      const uint32_t j = threadIdx.x >> 6;    // 32-row block
      // pass A: block amax of both columns at once (packed); pass B: re-read,
      // scale both halves by their own power of two and convert.  A warp reads
      // 32 consecutive words per row: no bank conflicts.
      // word (row 32j + i, pair cp) of the swizzled tile: box cp >> 5, chunk
      // ((cp & 31) >> 2) ^ (i & 7), word cp & 3 of the chunk (32 words a row)
      const uint32_t* col = tile + (cp >> 5) * 4096 + (32 * j) * 32;
      uint32_t off[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) off[k] = ((((cp & 31u) >> 2) ^ static_cast<uint32_t>(k)) << 2) | (cp & 3u);
      auto word = [&](int i) { return col[i * 32 + off[i & 7]]; };
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) m = bf16x2_max_abs(m, word(i));
      const int elo = mx_exponent(abs_lo(m)), ehi = mx_exponent(abs_hi(m));
      const uint32_t s2 = bf16_pow2_neg_bits(elo) | (bf16_pow2_neg_bits(ehi) << 16);
      uint32_t olo[8], ohi[8];  // 32 E4M3 bytes of column 2cp / 2cp+1
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t u0 = bf16x2_mul(word(4 * i), s2);
        const uint32_t u1 = bf16x2_mul(word(4 * i + 1), s2);
        const uint32_t u2 = bf16x2_mul(word(4 * i + 2), s2);
        const uint32_t u3 = bf16x2_mul(word(4 * i + 3), s2);
        olo[i] = cvt_e4m3x2(bf16lo(u0), bf16lo(u1)) | (cvt_e4m3x2(bf16lo(u2), bf16lo(u3)) << 16);
        ohi[i] = cvt_e4m3x2(bf16hi(u0), bf16hi(u1)) | (cvt_e4m3x2(bf16hi(u2), bf16hi(u3)) << 16);
      }
      uint8_t* dlo = q_col + (k0 + 2 * cp) * cap_col + mp + 32 * j;
      uint8_t* dhi = dlo + cap_col;
      if (qcol_v8) {
        st_global_32B(dlo, olo);
        st_global_32B(dhi, ohi);
      } else {
        reinterpret_cast<uint4*>(dlo)[0] = make_uint4(olo[0], olo[1], olo[2], olo[3]);
        reinterpret_cast<uint4*>(dlo)[1] = make_uint4(olo[4], olo[5], olo[6], olo[7]);
        reinterpret_cast<uint4*>(dhi)[0] = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
        reinterpret_cast<uint4*>(dhi)[1] = make_uint4(ohi[4], ohi[5], ohi[6], ohi[7]);
      }
      const uint32_t klo = 2 * cp, khi = klo + 1;
      uint8_t* sfc = sf_col + ((k0 >> 7) * (cap_col >> 7) + (mp >> 7)) * 512;
      sfc[(klo & 31u) * 16 + (klo >> 5) * 4 + j] = static_cast<uint8_t>(elo + 127);
      sfc[(khi & 31u) * 16 + (khi >> 5) * 4 + j] = static_cast<uint8_t>(ehi + 127);
    }
  }
  // a prefetch still in flight (only after an abort) lands before the CTA exits
  if (threadIdx.x == 0)
    for (int bb = 0; bb < 2; ++bb)
      if (pending & (1u << bb)) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&bars[bb]), (parity >> bb) & 1u))
          if (globaltimer() - t0 > kWaitTimeoutNs) break;
      }
}

// unaligned: group sizes of any value (group_ws required); the colwise copy
// and the scales are then padded per group (cap + 128 G rows).
cudaError_t launch_mxfp8_quantize(bool row, bool col, const uint16_t* x, int64_t cap, int64_t cols,
                                  const int64_t* group_ws, int G, uint8_t* q_row, uint8_t* sf_row,
                                  uint8_t* q_col, uint8_t* sf_col, int32_t* status, int num_sms,
                                  cudaStream_t stream, bool unaligned) {
  const int64_t cap_col = unaligned ? cap + 128 * static_cast<int64_t>(G) : cap;
  const int64_t max_tiles = (cap_col >> 7) * (cols >> 7);
  if (max_tiles == 0) return cudaSuccess;
  CUtensorMap tm;
  if (!make_tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, x, static_cast<uint64_t>(cols),
                    static_cast<uint64_t>(cap), static_cast<uint64_t>(cols) * 2, 64, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int smem = kQSmemBytes + (unaligned ? 12 * (G + 1) + 16 : 0);
  auto launch = [&](auto kern) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // persistent grid: as many CTAs as are resident at once
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    const int64_t full = static_cast<int64_t>(num_sms) * per_sm;
    const int grid = static_cast<int>(max_tiles < full ? max_tiles : full);
    const int qcol_v8 = (reinterpret_cast<uintptr_t>(q_col) & 31u) == 0 ? 1 : 0;
    const int qrow_v8 = (reinterpret_cast<uintptr_t>(q_row) & 31u) == 0 ? 1 : 0;
    kern<<<grid, 256, smem, stream>>>(tm, cap, cols, group_ws, G, q_row, sf_row, q_col, sf_col,
                                       qcol_v8, qrow_v8, cap_col, status);
    return cudaGetLastError();
  };
  if (unaligned) {
    if (row && col) return launch(mxfp8_quantize_kernel<true, true, true>);
    if (row) return launch(mxfp8_quantize_kernel<true, false, true>);
    return launch(mxfp8_quantize_kernel<false, true, true>);
  }
  if (row && col) return launch(mxfp8_quantize_kernel<true, true, false>);
  if (row) return launch(mxfp8_quantize_kernel<true, false, false>);
  return launch(mxfp8_quantize_kernel<false, true, false>);
}

}  // namespace mxg
