// gemm.cu -- persistent grouped block-scaled GEMM on tcgen05 (sm_103a).
//
// What it computes (TransformerEngine gemm.py grouped_gemm and PR #2763's V2
// grouped GEMM; PR #3661 for the row-scaled NVFP4 variant):
//   fprop TN (ragged rows):        C[off_g+i, n] = alpha_g * sum_k A[off_g+i, k] B[g*N+n, k]
//   wgrad NT (ragged contraction): dW[g, n, k]   = alpha_g * sum_{m in g} A[n, m] B[k, m]
//   dgrad NN (ragged rows):        dX[off_g+i, k] = alpha_g * sum_n A[off_g+i, n] B[k, g*N+n]
// (+ beta_g * previous C), with E4M3 x E8M0/1x32 (MXFP8) or E2M1 x
// E4M3/1x16 (NVFP4) operands whose scales arrive pre-swizzled from the
// grouped quantize, FP32 accumulation in tensor memory and an epilogue that
// applies alpha, beta and -- for NVFP4 -- the per-row / per-column FP32
// outer scales (PR #3661 runs the GEMM with neutral outer scales into an FP32
// scratch and scales afterwards; here the scratch is tensor memory and the
// scaling is fused into the read-out).
//
// Design (GB300-first, no library):
//   * one CTA per SM, persistent; work units are walked in a static
//     round-robin order derived on the device from the offsets workspace, so
//     there is no host sync and the launch is graph-safe (PR #2763's
//     motivation).
//   * default: grouped_gemm_pair_kernel, 2-CTA clusters computing 256 x 256
//     units with the cta_group::2 MMA (each CTA holds 128 rows of A and half
//     of B); warp 0 lane 0 TMA producer, warp 1 lane 0 MMA issuer (even CTA),
//     warps 2-9 epilogue (one TMEM lane quarter and 128 columns each), warps
//     10-11 scale copies (even CTA).  The producer publishes each unit's
//     shape (K blocks, MMAs of the last one, half width) to the MMA thread
//     and the copy warps, so that they decode nothing between units.  128
//     bytes of K per pipeline stage (4 MMAs of 32 bytes: 32 E4M3 or 64 E2M1
//     elements), 256 bytes for MXFP8 fprop when K % 256 == 0 and for MXFP8
//     wgrad (a group may end inside its last stage), 64 for NVFP4 fprop with
//     K % 256 != 0.  The epilogue warps copy their columns' operands (NVFP4
//     column outer scales, bias) into shared memory while they wait.
//   * grouped_gemm_kernel: single-CTA 128 x BN tiles (BN 256 or 128) for the
//     cases the pair does not cover (B with fewer than 256 rows); warps
//     0 / 1 / 2.. as above, scale copies inline on the MMA thread.
//   * scales: each 128x4 swizzled scale tile (512 bytes) is copied into 4
//     TMEM columns by tcgen05.cp 32x128b.warpx4 -- the swizzled layout is
//     exactly the one that copy and the block-scaled MMA consume.  Each
//     pipeline stage owns its own scale columns, so refilling a stage never
//     races an MMA that still reads the previous scales.
//   * fprop orders tiles group-major, then n, then m: the CTAs in flight
//     share one weight tile and the group's activations stay in L2.
//   * every mbarrier wait is bounded (mbar_wait); after a timeout the CTA
//     drains its in-flight copies and MMAs, frees TMEM and returns.
#include "mxg_device.cuh"
#include "mxg_host.h"

namespace mxg {

struct GemmParams {
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  const float* a_outer;
  const float* b_outer;
  const int64_t* group_ws;
  const float* alpha;
  const float* beta;
  const float* bias;  // [G, out_cols] or null
  void* C;
  int32_t* status;
  int64_t M_cap, N, K;
  int64_t a_atoms_row;  // 512-byte scale tiles per 128-row band of A
  int64_t b_atoms_row;  // ... of B
  int64_t kb_uniform;   // K blocks (128 bytes) of one fprop / dgrad tile
  int64_t out_cols;     // columns of C (N for fprop, K for dgrad and wgrad)
  uint64_t timeout_ns;  // bound on every pipeline wait
  int G;
  int mode;  // 0 fprop, 1 wgrad, 2 dgrad
  int out_bf16;
  int inject;  // test hook: bit 0 withholds the first accumulator-ready arrival of CTA 0
  int c_align32;  // C is 32-byte aligned (whole-sector epilogue stores)
  int vec_col;    // bias and the NVFP4 column outer scales are 16-byte aligned
  int unaligned;  // group sizes of any value (MXFP8, CTA-pair kernel only)
};

// BK: bytes of K per pipeline stage (128 with the 128-byte swizzle, or 64
// with the 64-byte swizzle for row-scaled NVFP4: half-size stages, twice as
// many of them).
template <int BN, int STAGES, int ACC, bool NVF4, int BK = 128>
struct GemmCfg {
  static_assert(BK == 128 || (BK == 64 && NVF4), "64-byte stages are for NVFP4");
  static constexpr int kEpiWarps = 4 * (BN / 128);
  static constexpr int kThreads = 32 * (2 + kEpiWarps);
  static constexpr int kATile = 128 * BK;
  static constexpr int kBTile = BN * BK;
  static constexpr int kMmas = BK / 32;          // MMAs (32 bytes of K each) per stage
  static constexpr int kSwizzle = BK == 128 ? 2 : 4;  // descriptor swizzle mode (128B / 64B)
  static constexpr int kSbo = 8 * BK;            // bytes between 8-row core-matrix groups
  // scale tiles along K per stage and band: NVFP4 one per MMA (64 elements);
  // MXFP8 one 128-element tile
  static constexpr int kAtomsK = NVF4 ? kMmas : 1;
  static constexpr int kSfaBytes = 512 * kAtomsK;
  static constexpr int kSfbBytes = 512 * kAtomsK * (BN / 128);
  static constexpr int kStageBytes =
      ((kATile + kBTile + kSfaBytes + kSfbBytes + 1023) / 1024) * 1024;
  static constexpr uint32_t kTxBytes = kATile + kBTile + kSfaBytes + kSfbBytes;
  static constexpr int kSfaCols = 4 * kAtomsK;
  static constexpr int kSfCols = kSfaCols * (1 + BN / 128);  // TMEM columns per stage
  static constexpr int kTmemCols = 512;
  static_assert(ACC * BN + STAGES * kSfCols <= kTmemCols, "tensor memory budget");
  // barriers: full[S], empty[S], tfull[ACC], tempty[ACC], drain; then the
  // TMEM base address and the abort flag
  static constexpr int kBarBytes = 8 * (2 * STAGES + 2 * ACC + 1) + 16;
  static size_t smem_bytes(int G) {
    return 1024 + static_cast<size_t>(STAGES) * kStageBytes + kBarBytes + 8 * (G + 1) + 16;
  }
  // Instruction descriptor: A/B formats at bits 7 / 10 (E4M3 = 0 for
  // mxf8f6f4, E2M1 = 1 for mxf4nvf4), N >> 3 at bit 17, scale format at bit
  // 23 (1 = UE8M0, 0 = UE4M3), M >> 4 at bit 24; K-major A and B; scale
  // data ids at bits 4 (B) and 29 (A) are added per MMA.
  static constexpr uint32_t kIdesc = (NVF4 ? ((1u << 7) | (1u << 10)) : 0u) |
                                     (static_cast<uint32_t>(BN >> 3) << 17) |
                                     (NVF4 ? 0u : (1u << 23)) | ((128u >> 4) << 24);
};

struct TileInfo {
  int g;
  int64_t a_row, b_row;      // first row of the A / B tile (TMA coordinate 1)
  int64_t a_sf_row;          // row of A's scales: the padded row when groups are unaligned
  int64_t kb_count;          // K blocks (BK bytes) of this tile
  int64_t a_kb0, b_kb0;      // single-CTA kernel: first K block of A and of B
  int64_t a_k0, b_k0;        // CTA-pair kernel: first contraction element of A and of B
  int last_mmas;             // CTA-pair kernel: MMAs of the last K block (a wgrad group
                             // may end inside it; the others run all of theirs)
  int64_t c_row, c_col;      // top-left output element
  int64_t row_end;           // rows of C at or beyond this are not written
  bool half_n;               // CTA-pair unit whose last 128 output columns are past the
                             // output width: its MMAs run with N = 128
};

// Work unit t of the single-CTA kernel -> one 128 x BN output tile.
// K blocks are BK bytes: BK elements of E4M3, 2*BK of packed E2M1 (EPB =
// elements per byte).
template <int BN, int BK, int EPB>
__device__ __forceinline__ TileInfo map_tile(int64_t t, const GemmParams& p, const int32_t* row_off,
                                             const int32_t* tile_off) {
  TileInfo ti;
  if (p.mode != 1) {  // fprop / dgrad: ragged output rows
    int lo = 0, hi = p.G;  // largest g with tile_off[g] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tile_off[mid] <= t)
        lo = mid;
      else
        hi = mid;
    }
    const int g = lo;
    const int64_t mt = (row_off[g + 1] - row_off[g]) >> 7;  // row tiles per column tile
    const int64_t local = t - tile_off[g];
    const int64_t n_tile = local / mt, m_tile = local % mt;
    ti.g = g;
    ti.a_row = row_off[g] + 128 * m_tile;
    // fprop: B rows are expert g's weight rows; dgrad: B is the transposed
    // weight copy [K, G*N] and expert g is its K-slab g*N .. g*N+N-1
    ti.b_row = p.mode == 0 ? static_cast<int64_t>(g) * p.N + BN * n_tile : BN * n_tile;
    ti.kb_count = p.kb_uniform;
    ti.a_kb0 = 0;
    ti.b_kb0 = p.mode == 0 ? 0 : (static_cast<int64_t>(g) * p.N) / (BK * EPB);
    ti.c_row = ti.a_row;
    ti.c_col = BN * n_tile;
    ti.row_end = row_off[g + 1];
  } else {
    const int64_t nt = p.N >> 7;
    const int64_t kt = p.K / BN, tpg = nt * kt;
    const int g = static_cast<int>(t / tpg);
    const int64_t local = t % tpg;
    const int64_t n_tile = local / kt, k_tile = local % kt;
    ti.g = g;
    ti.a_row = 128 * n_tile;
    ti.b_row = BN * k_tile;
    ti.kb_count = (row_off[g + 1] - row_off[g]) / (BK * EPB);
    ti.a_kb0 = ti.b_kb0 = row_off[g] / (BK * EPB);
    ti.c_row = static_cast<int64_t>(g) * p.N + ti.a_row;
    ti.c_col = ti.b_row;
    ti.row_end = static_cast<int64_t>(g + 1) * p.N;
  }
  ti.a_sf_row = ti.a_row;
  ti.half_n = false;
  return ti;
}

// Bounded wait used only while tearing down: ignores the abort flag.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity, int32_t* status,
                                                uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > timeout_ns) {
      status_set(status, MXG_DEV_TIMEOUT);
      return;
    }
  }
}

// Group tables in shared memory, built by one warp: sanitised row offsets
// (sizes clamped at 0, rounded down to 128 unless p.unaligned, the running
// sum capped at M_cap); padded row offsets (each kept size rounded up to
// 128: where a group's scales, and its slab of a colwise copy, start when
// groups are unaligned; equal to the row offsets otherwise), written when
// prow_off is not null; and, for fprop / dgrad, each group's first work unit
// -- a unit is one 128-row tile, or two (pair_units) -- times the column
// tiles of width bn.  CTA 0 records the sanitisation bits in the status word.
__device__ __forceinline__ void build_group_tables(const GemmParams& p, int32_t* row_off,
                                                   int32_t* prow_off, int32_t* tile_off,
                                                   uint32_t lane, bool pair_units, int bn) {
  int64_t carry_rows = 0, carry_pad = 0, carry_tiles = 0;
  int32_t bits = 0;
  const int64_t ntiles_n = (p.out_cols + bn - 1) / bn;  // a last unit may be half wide
  auto scan = [&](int64_t v) {  // inclusive warp scan
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t u = __shfl_up_sync(0xFFFFFFFFu, v, d);
      if (lane >= static_cast<uint32_t>(d)) v += u;
    }
    return v;
  };
  for (int base = 0; base < p.G; base += 32) {
    const int g = base + static_cast<int>(lane);
    int64_t s = 0;
    if (g < p.G) {
      s = p.group_ws[g];
      if (s < 0) {
        s = 0;
        bits |= MXG_DEV_NEG_SIZE;
      }
      if (!p.unaligned && (s & 127)) {
        s &= ~static_cast<int64_t>(127);
        bits |= MXG_DEV_MISALIGNED;
      }
      if (s > p.M_cap) s = p.M_cap;
    }
    const int64_t incl = scan(s);
    const int64_t before = min(carry_rows + incl - s, p.M_cap);
    const int64_t after = min(carry_rows + incl, p.M_cap);
    if (carry_rows + incl > p.M_cap && s > 0) bits |= MXG_DEV_SUM_OVER_CAPACITY;
    const int64_t pad = ((after - before) + 127) & ~static_cast<int64_t>(127);
    const int64_t pincl = scan(pad);
    const int64_t mt_g = pad >> 7;
    const int64_t tiles_g = p.mode != 1 ? (pair_units ? (mt_g + 1) >> 1 : mt_g) * ntiles_n : 0;
    const int64_t tincl = scan(tiles_g);
    if (g < p.G) {
      row_off[g] = static_cast<int32_t>(before);
      if (prow_off) prow_off[g] = static_cast<int32_t>(carry_pad + pincl - pad);
      tile_off[g] = static_cast<int32_t>(carry_tiles + tincl - tiles_g);
    }
    carry_rows += __shfl_sync(0xFFFFFFFFu, incl, 31);
    carry_pad += __shfl_sync(0xFFFFFFFFu, pincl, 31);
    carry_tiles += __shfl_sync(0xFFFFFFFFu, tincl, 31);
  }
  if (lane == 0) {
    row_off[p.G] = static_cast<int32_t>(min(carry_rows, p.M_cap));
    if (prow_off) prow_off[p.G] = static_cast<int32_t>(carry_pad);
    tile_off[p.G] = static_cast<int32_t>(carry_tiles);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, d);
  if (lane == 0 && blockIdx.x == 0) status_set(p.status, bits);
}

// Four consecutive fp32 values at p (16-byte aligned when vec, else any
// 4-byte alignment).
__device__ __forceinline__ float4 load4(const float* p, bool vec) {
  if (vec) return *reinterpret_cast<const float4*>(p);
  return make_float4(p[0], p[1], p[2], p[3]);
}

// A 16-byte shared-memory load the compiler keeps where it is written
// (neither hoisted nor merged with its neighbours).
__device__ __forceinline__ float4 lds_f4_volatile(uint32_t addr) {
  float4 v;
  asm volatile("ld.volatile.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// Column operands of an epilogue warp's 128 columns in the single-CTA
// kernel, read once per unit before the accumulator is (in flight while the
// warp waits for it): lane l holds columns 4l .. 4l+3 of the NVFP4 column
// outer scales (cs) and of the bias (bs); column j is lane j / 4's component
// j % 4, fetched with a shuffle.  (Loading them per 16-column chunk instead
// put a load latency in front of every chunk: the NVFP4 epilogue took twice
// as long.)  The CTA-pair kernel copies them to shared memory instead.
struct EpiCols {
  float4 cs, bs;
};

template <bool NVF4>
__device__ __forceinline__ EpiCols epi_cols(const GemmParams& p, const TileInfo& ti, uint32_t col0,
                                            uint32_t lane) {
  EpiCols e;
  e.cs = make_float4(1.0f, 1.0f, 1.0f, 1.0f);
  e.bs = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (ti.c_col + col0 >= p.out_cols) return e;  // upper half of a half-wide unit: not stored
  if (NVF4)  // fprop: per weight row; wgrad: per (group, column) of X
    e.cs = load4(p.b_outer + (p.mode == 1 ? static_cast<int64_t>(ti.g) * p.K : 0) + ti.b_row +
                     col0 + 4 * lane,
                 p.vec_col);
  if (p.bias)
    e.bs = load4(p.bias + static_cast<int64_t>(ti.g) * p.out_cols + ti.c_col + col0 + 4 * lane,
                 p.vec_col);
  return e;
}

// Component j % 4 of lane j / 4's value (j a compile-time constant after
// unrolling; every lane of the warp takes part).
__device__ __forceinline__ float col_value(const float4& v4, int j) {
  const int c = j & 3;
  const float x = c == 0 ? v4.x : (c == 1 ? v4.y : (c == 2 ? v4.z : v4.w));
  return __shfl_sync(0xFFFFFFFFu, x, j >> 2);
}

// One output row of the epilogue: 128 accumulator columns (v, four loads of
// 32) starting at column c_col + col0, turned into
//   alpha_g * acc [* outer_row * outer_col (NVFP4)] [+ bias] [+ beta_g * C]
// and stored as fp32 or bf16 (round to nearest even).  Rows at or beyond the
// tile's row_end, and the upper half of a half-wide last column unit, are
// skipped.  Each thread owns a row, so a store instruction touches 32 rows:
// with a 32-byte-aligned C every store fills whole 32-byte sectors (16 bf16
// or 8 fp32 per store), else 16-byte stores are used.  The column operands
// (NVFP4 column outer scales, bias) come from ec by shuffle, or with SMCOLS
// from the warp's shared-memory copy (scs: the 128 column outer scales, sbs:
// the 128 bias values), one broadcast 16-byte load per 4 columns; either way
// every lane of the warp runs the transform (rows past row_end only skip the
// loads and stores); beta and bias checks are made once per row, not per
// element.
template <bool NVF4, bool SMCOLS = false>
__device__ __forceinline__ void epilogue_row(const GemmParams& p, const TileInfo& ti, int64_t row,
                                             uint32_t col0, uint32_t (&v)[4][32], bool has_k,
                                             const EpiCols& ec, const float* scs = nullptr,
                                             const float* sbs = nullptr) {
  if (ti.c_col + col0 >= p.out_cols) return;  // warp-uniform
  const bool valid = row < ti.row_end;
  const int64_t cbase = row * p.out_cols + ti.c_col + col0;
  const float alpha = p.alpha ? p.alpha[ti.g] : 1.0f;
  const float beta = valid && p.beta ? p.beta[ti.g] : 0.0f;  // old C read for valid rows only
  const bool bs = p.bias != nullptr;
  const float rs = NVF4 ? (valid ? p.a_outer[row] : 0.0f) : 1.0f;
  const float rsa = rs * alpha;  // the row's factor (shared-memory column path)
  // 16 columns at a time (32 bytes of bf16 or 64 of fp32), transformed in
  // place in the accumulator registers
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint32_t* a = &v[k >> 1][16 * (k & 1)];
    const int j0 = 16 * k;  // first column of the 16
    if (SMCOLS) {
      // pairs of columns: (acc * (alpha * outer_row)) * outer_col [+ bias],
      // two lanes per packed instruction
#pragma unroll
      for (int e = 0; e < 16; e += 4) {
        float x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = has_k ? __uint_as_float(a[e + i]) : 0.0f;
        f32x2_mul(x[0], x[1], rsa, rsa);
        f32x2_mul(x[2], x[3], rsa, rsa);
        // NVFP4: volatile loads, kept next to their use, so the compiler does
        // not hoist all 128 columns' operands into registers beside the
        // accumulator (that kernel spilled 104 bytes without them); the MXFP8
        // kernel has the registers and schedules plain loads better
        if (NVF4) {
          const float4 c4 = lds_f4_volatile(smem_u32(scs + j0 + e));
          f32x2_mul(x[0], x[1], c4.x, c4.y);
          f32x2_mul(x[2], x[3], c4.z, c4.w);
        }
        if (bs) {
          const float4 b4 = NVF4 ? lds_f4_volatile(smem_u32(sbs + j0 + e))
                                 : *reinterpret_cast<const float4*>(sbs + j0 + e);
          f32x2_add(x[0], x[1], b4.x, b4.y);
          f32x2_add(x[2], x[3], b4.z, b4.w);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) a[e + i] = __float_as_uint(x[i]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float x = has_k ? __uint_as_float(a[e]) : 0.0f;
        if (NVF4) x = x * rs * col_value(ec.cs, j0 + e);
        x *= alpha;
        if (bs) x += col_value(ec.bs, j0 + e);
        a[e] = __float_as_uint(x);
      }
    }
    if (p.out_bf16) {
      uint16_t* dst = static_cast<uint16_t*>(p.C) + cbase + j0;
      uint32_t w[8];
      if (beta != 0.0f) {
        const uint4 q0 = reinterpret_cast<const uint4*>(dst)[0];
        const uint4 q1 = reinterpret_cast<const uint4*>(dst)[1];
        const uint32_t old[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int q = 0; q < 8; ++q)
          w[q] = cvt_bf16x2(__uint_as_float(a[2 * q]) + beta * bf16lo(old[q]),
                            __uint_as_float(a[2 * q + 1]) + beta * bf16hi(old[q]));
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          w[q] = cvt_bf16x2(__uint_as_float(a[2 * q]), __uint_as_float(a[2 * q + 1]));
      }
      if (!valid) {
      } else if (p.c_align32) {
        st_global_32B(dst, w);
      } else {
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    } else {
      float* out = static_cast<float*>(p.C) + cbase + j0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // 8 columns = 32 bytes
        float* dst = out + 8 * h;
        uint32_t w[8];
        if (beta != 0.0f) {
          const float4 q0 = reinterpret_cast<const float4*>(dst)[0];
          const float4 q1 = reinterpret_cast<const float4*>(dst)[1];
          const float old[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
          for (int q = 0; q < 8; ++q)
            w[q] = __float_as_uint(__uint_as_float(a[8 * h + q]) + beta * old[q]);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) w[q] = a[8 * h + q];
        }
        if (!valid) {
        } else if (p.c_align32) {
          st_global_32B(dst, w);
        } else {
          reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
          reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
  }
}

// Single-CTA kernel: one 128 x BN output tile per work unit, ACC
// accumulators in tensor memory (the MMA of the next tile starts while the
// epilogue drains the previous one when ACC = 2).
template <int BN, int STAGES, int ACC, bool NVF4, int BK>
__global__ void __launch_bounds__(GemmCfg<BN, STAGES, ACC, NVF4, BK>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
  using Cfg = GemmCfg<BN, STAGES, ACC, NVF4, BK>;
  constexpr int EPB = NVF4 ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* bar_area = smem + STAGES * Cfg::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(bar_area);
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(bar_area + 8 * (2 * STAGES + 2 * ACC + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_s + 1);
  int32_t* row_off = reinterpret_cast<int32_t*>(bar_area + Cfg::kBarBytes);
  int32_t* tile_off = row_off + (p.G + 1);

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const uint32_t smem_base = smem_u32(smem);
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[STAGES + s]); };
  auto tfull_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + a]); };
  auto tempty_bar = [&](int a) { return smem_u32(&bars[2 * STAGES + ACC + a]); };
  const uint32_t drain_bar = smem_u32(&bars[2 * STAGES + 2 * ACC]);

  // ------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < ACC; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), Cfg::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_base_s), Cfg::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 1) build_group_tables(p, row_off, nullptr, tile_off, lane, false, BN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_s;
  const int64_t unit0 = blockIdx.x;
  const int64_t ustride = gridDim.x;
  const int64_t total_tiles = p.mode != 1 ? static_cast<int64_t>(tile_off[p.G])
                                          : p.G * (p.N >> 7) * (p.K / BN);

  // ------------------------------------------------------------ producer
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmap_a);
      prefetch_tmap(&tmap_b);
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, last_parity = 0;  // per stage, for the final drain
      bool ok = true;
      for (int64_t t = unit0; ok && t < total_tiles; t += ustride) {
        const TileInfo ti = map_tile<BN, BK, EPB>(t, p, row_off, tile_off);
        for (int64_t kb = 0; kb < ti.kb_count; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_base + stage * Cfg::kStageBytes;
          const uint32_t sb = sa + Cfg::kATile;
          const uint32_t ssfa = sb + Cfg::kBTile;
          const uint32_t ssfb = ssfa + Cfg::kSfaBytes;
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, Cfg::kTxBytes);
          const int64_t ka = ti.a_kb0 + kb, kbb = ti.b_kb0 + kb;
          tma_load_2d(sa, &tmap_a, fb, static_cast<int32_t>(ka * BK), static_cast<int32_t>(ti.a_row));
          tma_load_2d(sb, &tmap_b, fb, static_cast<int32_t>(kbb * BK),
                      static_cast<int32_t>(ti.b_row));
          // first scale tile of this stage along K (MXFP8: tiles of 128 bytes of K)
          const int64_t a_atom = NVF4 ? ka * Cfg::kAtomsK : (ka * BK) >> 7;
          const int64_t b_atom = NVF4 ? kbb * Cfg::kAtomsK : (kbb * BK) >> 7;
          bulk_load(ssfa, p.a_sf + ((ti.a_row >> 7) * p.a_atoms_row + a_atom) * 512,
                    Cfg::kSfaBytes, fb);
#pragma unroll
          for (int i = 0; i < BN / 128; ++i)
            bulk_load(ssfb + i * 512 * Cfg::kAtomsK,
                      p.b_sf + (((ti.b_row >> 7) + i) * p.b_atoms_row + b_atom) * 512,
                      512 * Cfg::kAtomsK, fb);
          issued_mask |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every copy this thread issued has landed before the CTA may exit
      for (int s = 0; s < STAGES; ++s)
        if (issued_mask & (1u << s)) mbar_wait_drain(full_bar(s), (last_parity >> s) & 1u, p.status, p.timeout_ns);
    }
  }
  // ------------------------------------------------------------ MMA issuer
  else if (warp == 1) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int64_t t = unit0; ok && t < total_tiles; t += ustride) {
        const TileInfo ti = map_tile<BN, BK, EPB>(t, p, row_off, tile_off);
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.status, p.timeout_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int64_t kb = 0; kb < ti.kb_count; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_base + stage * Cfg::kStageBytes;
          const uint32_t sb = sa + Cfg::kATile;
          const uint32_t ssfa = sb + Cfg::kBTile;
          const uint32_t ssfb = ssfa + Cfg::kSfaBytes;
          const uint32_t sfa_t = tmem_base + ACC * BN + stage * Cfg::kSfCols;
          const uint32_t sfb_t = sfa_t + Cfg::kSfaCols;
          // scale tiles -> TMEM.  A: tile a at column 4a.  B: for K-step a,
          // band i at column a * 4 * (BN/128) + 4i (the bands of one MMA are
          // adjacent, 4 columns each).
#pragma unroll
          for (int a = 0; a < Cfg::kAtomsK; ++a)
            tc_cp_scales(sfa_t + 4 * a, smem_desc(ssfa + 512 * a, 0, 128, 0));
#pragma unroll
          for (int i = 0; i < BN / 128; ++i)
#pragma unroll
            for (int a = 0; a < Cfg::kAtomsK; ++a)
              tc_cp_scales(sfb_t + a * 4 * (BN / 128) + 4 * i,
                           smem_desc(ssfb + i * 512 * Cfg::kAtomsK + 512 * a, 0, 128, 0));
          // MXFP8: byte (K block within the 128-element scale tile) of each MMA
          const uint32_t sf_id0 = NVF4 ? 0u : static_cast<uint32_t>(((ti.a_kb0 + kb) * BK & 127) >> 5);
#pragma unroll
          for (int kk = 0; kk < Cfg::kMmas; ++kk) {
            const uint64_t adesc = smem_desc(sa + 32 * kk, 16, Cfg::kSbo, Cfg::kSwizzle);
            const uint64_t bdesc = smem_desc(sb + 32 * kk, 16, Cfg::kSbo, Cfg::kSwizzle);
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            if (NVF4) {
              tc_mma_nvf4(d_tmem, adesc, bdesc, Cfg::kIdesc, sfa_t + 4 * kk,
                          sfb_t + kk * 4 * (BN / 128), accum);
            } else {
              const uint32_t sid = sf_id0 + kk;
              const uint32_t idesc = Cfg::kIdesc | (sid << 4) | (sid << 29);
              tc_mma_mxf8(d_tmem, adesc, bdesc, idesc, sfa_t, sfb_t, accum);
            }
          }
          tc_commit(empty_bar(stage));  // frees the stage once these MMAs finish
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // accumulator ready (immediately if no K blocks); the test hook withholds
        // this arrival once so that the epilogue's bounded wait runs out
        if (!((p.inject & 1) && blockIdx.x == 0 && t == blockIdx.x)) tc_commit(tfull_bar(acc));
        if (++acc == ACC) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // all MMAs this thread issued have completed before TMEM is freed
      tc_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0, p.status, p.timeout_ns);
    }
  }
  // ------------------------------------------------------------ epilogue
  else {
    const uint32_t ew = warp - 2;
    const uint32_t quarter = warp & 3u;  // TMEM lanes 32*quarter .. +31
    const uint32_t col0 = 128u * (ew >> 2);
    uint32_t acc = 0, acc_phase = 0;
    for (int64_t t = unit0; t < total_tiles; t += ustride) {
      const TileInfo ti = map_tile<BN, BK, EPB>(t, p, row_off, tile_off);
      const EpiCols ec = epi_cols<NVF4>(p, ti, col0, lane);  // in flight during the wait
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.status, p.timeout_ns)) break;
      tc_fence_after();
      uint32_t v[4][32];
      const bool has_k = ti.kb_count > 0;
      if (has_k) {
        const uint32_t taddr = tmem_base + ((32u * quarter) << 16) + acc * BN + col0;
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(taddr + 32 * c, v[c]);
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(tempty_bar(acc));  // no memory published
      if (++acc == ACC) {
        acc = 0;
        acc_phase ^= 1u;
      }
      epilogue_row<NVF4>(p, ti, ti.c_row + 32 * quarter + lane, col0, v, has_k, ec);
    }
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ---------------------------------------------------------------- CTA-pair kernel
// A 2-CTA cluster computes one 256 x 256 output unit with the .cta_group::2
// MMA: the even CTA issues every MMA and scale copy, and each one runs on both
// SMs.  CTA rank r holds rows 128r..128r+127 of the unit's A tile and of its
// B tile (the B halves are exchanged by the tensor cores, not copied), the
// full 256-row B scale tile, and accumulates its 128 x 256 half of the unit
// in its own tensor memory.  Per SM and pipeline stage that is 32 KB of
// operands for a 128 x 256 x 128 MMA step, against 48 KB for the single-CTA
// 128 x 256 tile, and half the MMA instructions.
// BKB: bytes of K per stage.  256 for MXFP8 fprop with K % 256 == 0: 8 MMAs
// per stage halve the MMA thread's per-stage wait and commit (3 stages then
// fill shared memory instead of 6).  128 in
// general (128-byte swizzle); 64 (64-byte swizzle) for row-scaled NVFP4 where
// a 256-element K block does not fit: wgrad over 128-row groups (64 bytes of
// E2M1 along the contraction) and fprop with K % 256 != 0.
template <int STAGES, bool NVF4, int BKB = 128>
struct PairCfg {
  static constexpr int BN = 256, BK = BKB;
  static_assert(BK == 128 || (BK == 256 && !NVF4) || (BK == 64 && NVF4),
                "256-byte stages are for MXFP8, 64-byte stages for NVFP4");
  // a stage holds BK bytes of K as kSubTiles swizzled sub-tiles with rows of
  // kSubK bytes (a swizzled TMA box and a K-major MMA descriptor span at most
  // 128 bytes of a row)
  static constexpr int kSubK = BK > 128 ? 128 : BK;
  static constexpr int kSubTiles = BK / kSubK;
  static constexpr int kSwizzle = kSubK == 128 ? 2 : 4;  // descriptor swizzle mode
  static constexpr int kEpiWarps = 8;
  // scale-copy warps (even CTA): each tcgen05 instruction costs the issuing
  // thread about as long as a quarter of a stage's MMA work, so the scale
  // copies run on their own warps, beside the MMA thread
  static constexpr int kSfWarps = 2;
  static constexpr int kThreads = 32 * (2 + kEpiWarps + kSfWarps);
  static constexpr int kATile = 128 * BK;  // this CTA's rows of A
  static constexpr int kBTile = 128 * BK;  // this CTA's half of B
  static constexpr int kMmas = BK / 32;
  static constexpr int kMmasPerSub = kSubK / 32;
  // 512-byte scale tiles along K per stage and band: one per MMA with NVFP4
  // (4 scales of 16 elements per row), one per 128 elements with MXFP8
  static constexpr int kAtomsK = NVF4 ? kMmas : BK / 128;
  static constexpr int kSfaBytes = 512 * kAtomsK;
  static constexpr int kSfbBytes = 512 * kAtomsK * 2;
  static constexpr int kStageBytes =
      ((kATile + kBTile + kSfaBytes + kSfbBytes + 1023) / 1024) * 1024;
  // bytes landing per stage in BOTH CTAs, counted on the even CTA's barriers:
  // the operand tiles on full[s], the scale tiles on sffull[s]
  static constexpr uint32_t kTxBytes = 2u * (kATile + kBTile);
  static constexpr uint32_t kTxSfBytes = 2u * (kSfaBytes + kSfbBytes);
  static constexpr int kSfaCols = 4 * kAtomsK;
  static constexpr int kSfCols = kSfaCols * 3;
  static constexpr int kTmemCols = 512;
  static_assert(BN + STAGES * kSfCols <= kTmemCols, "tensor memory budget");
  static constexpr int kSfCopies = 3 * kAtomsK;  // scale tiles per stage (A, then B bands)
  // full[S], empty[S], sffull[S], tfull, tempty, drain, sfdrain,
  // info_full[2], info_empty[2], two unit words; TMEM base; abort flag
  static constexpr int kBarBytes = 8 * (3 * STAGES + 10) + 16;
  // column operands staged per epilogue warp (128 floats each): the NVFP4
  // column outer scales, the bias
  static size_t col_bytes(bool bias) {
    return static_cast<size_t>((NVF4 ? 1 : 0) + (bias ? 1 : 0)) * kEpiWarps * 128 * 4;
  }
  static size_t smem_bytes(int G, bool bias) {
    return 1024 + static_cast<size_t>(STAGES) * kStageBytes + kBarBytes + 12 * (G + 1) + 16 +
           col_bytes(bias);
  }
  // M = 256 (the pair), N = 256; other fields as in GemmCfg
  static constexpr uint32_t kIdesc = (NVF4 ? ((1u << 7) | (1u << 10)) : 0u) |
                                     (static_cast<uint32_t>(BN >> 3) << 17) |
                                     (NVF4 ? 0u : (1u << 23)) | ((256u >> 4) << 24);
  // the same with N = 128, for a half-wide last column unit: each CTA then
  // supplies 64 rows of B (the first 64 of its tile)
  static constexpr uint32_t kIdescN128 = (kIdesc & ~(0x3Fu << 17)) | ((128u >> 3) << 17);
};

// Work unit t -> this CTA's half.  fprop / dgrad: 256 rows of one group (the
// upper half may run past the group's end: it is computed but not stored)
// times 256 output columns, walked group-major.  wgrad: 256 rows of dW_g times 256 columns.
// When the output width is an odd multiple of 128 the last column unit is
// half wide (half_n): its MMAs run with N = 128, for which each CTA supplies
// 64 rows of B, so CTA r loads its B tile from b_row + 64 r (the tile's last
// 64 rows are loaded but not read).
// a_row is this CTA's first A row; b_row is the unit's first B row (this CTA
// loads b_row + 128 * rank, or b_row + 64 * rank when half wide).  Row units and the wgrad contraction are counted
// on the padded offsets, so unaligned groups (a last 128-row tile partly past
// the group) need nothing else: A's data rows start at the group's row
// offset, its scale rows (a_sf_row) and its colwise slabs at the padded one.
// a / b for a >= 0, b > 0: the 32-bit division when both fit (always, for
// the unit counts of any output that fits in memory), the 64-bit one
// otherwise.  A 64-bit division is a long dependent chain, and the unit
// decode runs on single threads between units.
__device__ __forceinline__ int64_t udiv(int64_t a, int64_t b) {
  if (((static_cast<uint64_t>(a) | static_cast<uint64_t>(b)) >> 32) == 0)
    return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
  return a / b;
}

template <int EPB, int BK>
__device__ __forceinline__ TileInfo map_unit_pair(int64_t t, const GemmParams& p,
                                                  const int32_t* row_off, const int32_t* prow_off,
                                                  const int32_t* tile_off, uint32_t rank) {
  TileInfo ti;
  if (p.mode != 1) {
    int lo = 0, hi = p.G;  // largest g with tile_off[g] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tile_off[mid] <= t)
        lo = mid;
      else
        hi = mid;
    }
    const int g = lo;
    const int64_t mu = (((prow_off[g + 1] - prow_off[g]) >> 7) + 1) >> 1;
    const int64_t local = t - tile_off[g];
    // fprop: column unit, then row unit: the clusters in flight share one
    // weight tile and the expert's activation rows stay in L2.  dgrad (whose
    // contraction runs over the FFN width, so that an expert's dY rows and
    // its transposed weight slab are tens of MB each): the same order while
    // the expert's dY rows fit in an L2 budget; else blocks of column units
    // whose weight tiles fit that budget, walked row unit by row unit, so
    // that the block's weight tiles stay in L2 and each dY row unit is read
    // once per block.
    int64_t n_tile = udiv(local, mu), mu_i = local - n_tile * mu;
    if (p.mode == 2) {
      constexpr int64_t kL2Budget = 32ll << 20;
      const int64_t ncu = (p.out_cols + 255) >> 8;
      if ((prow_off[g + 1] - prow_off[g]) * p.N > kL2Budget) {
        int64_t cb = 256 * p.N > kL2Budget ? 1 : udiv(kL2Budget, 256 * p.N);
        cb = cb > ncu ? ncu : cb;
        const int64_t blk = udiv(local, mu * cb);
        const int64_t width = (blk + 1) * cb <= ncu ? cb : ncu - blk * cb;
        const int64_t rem = local - blk * mu * cb;
        mu_i = udiv(rem, width);
        n_tile = blk * cb + (rem - mu_i * width);
      }
    }
    ti.g = g;
    ti.a_row = row_off[g] + 256 * mu_i + 128 * rank;
    ti.a_sf_row = prow_off[g] + 256 * mu_i + 128 * rank;
    ti.b_row = (p.mode == 0 ? static_cast<int64_t>(g) * p.N : 0) + 256 * n_tile;
    ti.kb_count = p.kb_uniform;
    ti.a_k0 = 0;
    ti.b_k0 = p.mode == 0 ? 0 : static_cast<int64_t>(g) * p.N;
    ti.last_mmas = BK / 32;
    ti.c_row = ti.a_row;
    ti.c_col = 256 * n_tile;
    ti.row_end = row_off[g + 1];
  } else {
    const int64_t nu = ((p.N >> 7) + 1) >> 1, kt = (p.K + 255) >> 8, tpg = nu * kt;
    const int64_t gq = udiv(t, tpg);
    const int g = static_cast<int>(gq);
    const int64_t local = t - gq * tpg;
    const int64_t nu_i = udiv(local, kt), k_tile = local - nu_i * kt;
    ti.g = g;
    ti.a_row = 256 * nu_i + 128 * rank;
    ti.a_sf_row = ti.a_row;
    ti.b_row = 256 * k_tile;
    // the group's padded rows (a multiple of 128) in K blocks of BK * EPB
    // elements; when they end inside the last block only its first MMAs
    // (32 bytes, i.e. 32 * EPB elements, each) belong to the group
    const int64_t rows = prow_off[g + 1] - prow_off[g], kel = BK * EPB;
    ti.kb_count = (rows + kel - 1) / kel;  // kel and 32 * EPB: powers of two
    ti.last_mmas = static_cast<int>((rows - (ti.kb_count - 1) * kel) / (32 * EPB));
    ti.a_k0 = ti.b_k0 = prow_off[g];
    ti.c_row = static_cast<int64_t>(g) * p.N + ti.a_row;
    ti.c_col = ti.b_row;
    ti.row_end = static_cast<int64_t>(g + 1) * p.N;
  }
  ti.half_n = ti.c_col + 256 > p.out_cols;
  return ti;
}

template <int STAGES, bool NVF4, int BKB>
__global__ void __launch_bounds__(PairCfg<STAGES, NVF4, BKB>::kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                             const __grid_constant__ CUtensorMap tmap_b,
                             const __grid_constant__ CUtensorMap tmap_sfa,
                             const __grid_constant__ CUtensorMap tmap_sfb, const GemmParams p) {
  using Cfg = PairCfg<STAGES, NVF4, BKB>;
  constexpr int BK = Cfg::BK, EPB = NVF4 ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* bar_area = smem + STAGES * Cfg::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(bar_area);
  // after the stage and accumulator barriers: info_full[2], info_empty[2],
  // the two published unit words, then the TMEM base and the abort flag
  uint64_t* info_word = bars + 3 * STAGES + 8;
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(bar_area + 8 * (3 * STAGES + 10));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_s + 1);
  int32_t* row_off = reinterpret_cast<int32_t*>(bar_area + Cfg::kBarBytes);
  int32_t* tile_off = row_off + (p.G + 1);
  int32_t* prow_off = tile_off + (p.G + 1);
  // after the tables: the epilogue warps' column operands (NVFP4 column
  // outer scales, then bias), 128 floats per warp each
  float* colsm = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(prow_off + (p.G + 1)) + 15) & ~static_cast<uintptr_t>(15));

  const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t rank = cluster_ctarank();
  auto full_bar = [&](int s) { return smem_u32(&bars[s]); };
  auto empty_bar = [&](int s) { return smem_u32(&bars[STAGES + s]); };
  auto sffull_bar = [&](int s) { return smem_u32(&bars[2 * STAGES + s]); };
  const uint32_t tfull_bar = smem_u32(&bars[3 * STAGES]);
  const uint32_t tempty_bar = smem_u32(&bars[3 * STAGES + 1]);
  const uint32_t drain_bar = smem_u32(&bars[3 * STAGES + 2]);
  const uint32_t sfdrain_bar = smem_u32(&bars[3 * STAGES + 3]);
  auto info_full_bar = [&](uint32_t i) { return smem_u32(&bars[3 * STAGES + 4 + i]); };
  auto info_empty_bar = [&](uint32_t i) { return smem_u32(&bars[3 * STAGES + 6 + i]); };
  constexpr uint64_t kInfoKbMask = (1ull << 48) - 1;
  constexpr uint32_t kFirstSfWarp = 2 + Cfg::kEpiWarps;

  // ------------------------------------------------------------ set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // even CTA: its producer's arrival + both CTAs' bytes + the scale-copy
      // warps' commits (scale tiles in tensor memory)
      mbar_init(full_bar(s), 1 + Cfg::kSfWarps);
      mbar_init(empty_bar(s), 1);  // the pair's MMA commit
      mbar_init(sffull_bar(s), 1);  // even CTA: its producer's arrival + both CTAs' scale bytes
    }
    mbar_init(tfull_bar, 1);
    mbar_init(tempty_bar, 2 * Cfg::kEpiWarps);  // even CTA: both CTAs' epilogue warps
    mbar_init(drain_bar, 1);
    mbar_init(sfdrain_bar, Cfg::kSfWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(info_full_bar(i), 1);                   // the producer
      mbar_init(info_empty_bar(i), 1 + Cfg::kSfWarps);  // the MMA thread, the scale-copy warps
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {  // collective over the pair: both CTAs get the same columns
    tmem_alloc_pair(smem_u32(tmem_base_s), Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  if (warp == 1) build_group_tables(p, row_off, prow_off, tile_off, lane, true, Cfg::BN);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the even CTA's barriers exist before the odd CTA's copies signal them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_base_s;
  const int64_t unit0 = blockIdx.x >> 1;
  const int64_t ustride = gridDim.x >> 1;
  const int64_t total_units =
      p.mode != 1 ? static_cast<int64_t>(tile_off[p.G])
                  : p.G * ((((p.N >> 7) + 1) >> 1) * ((p.K + 255) / 256));

  // ------------------------------------------------------------ producers (both CTAs)
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmap_a);
      prefetch_tmap(&tmap_b);
      prefetch_tmap(&tmap_sfa);
      prefetch_tmap(&tmap_sfb);
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, last_parity = 0;
      bool ok = true;
      for (int64_t t = unit0, u = 0; ok && t < total_units; t += ustride, ++u) {
        const TileInfo ti = map_unit_pair<EPB, BK>(t, p, row_off, prow_off, tile_off, rank);
        if (rank == 0) {
          // publish the unit's shape to the MMA thread and the scale-copy
          // warps (two slots: at most two units ahead of them)
          const uint32_t slot = static_cast<uint32_t>(u & 1), ipar = static_cast<uint32_t>((u >> 1) & 1);
          if (!mbar_wait(info_empty_bar(slot), ipar ^ 1u, abort_flag, p.status, p.timeout_ns)) break;
          info_word[slot] = (static_cast<uint64_t>(ti.kb_count) & kInfoKbMask) |
                            (static_cast<uint64_t>(ti.last_mmas & 0xFF) << 48) |
                            (static_cast<uint64_t>(ti.half_n ? 1 : 0) << 56);
          mbar_arrive(info_full_bar(slot));
        }
        // this CTA's half of B: rows 128r.. of the unit, or 64r.. when the
        // unit is half wide and its MMAs run with N = 128
        const int32_t b_half = static_cast<int32_t>(ti.b_row + (ti.half_n ? 64 : 128) * rank);
        const int32_t a_band = static_cast<int32_t>(ti.a_sf_row >> 7);
        const int32_t b_band = static_cast<int32_t>(ti.b_row >> 7);
        for (int64_t kb = 0; kb < ti.kb_count; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_base + stage * Cfg::kStageBytes;
          const uint32_t sb = sa + Cfg::kATile;
          const uint32_t ssfa = sb + Cfg::kBTile;
          const uint32_t ssfb = ssfa + Cfg::kSfaBytes;
          if (rank == 0) {
            mbar_arrive_expect_tx(sffull_bar(stage), Cfg::kTxSfBytes);
            mbar_arrive_expect_tx(full_bar(stage), Cfg::kTxBytes);
          }
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          const uint32_t sfb_bar = mapa_shared(sffull_bar(stage), 0);
          // first contraction element of this K block in A and in B (a
          // multiple of 128: a scale tile boundary)
          const int64_t ea = ti.a_k0 + kb * (BK * EPB), eb = ti.b_k0 + kb * (BK * EPB);
          // scale tiles first, on their own barrier: this CTA's A band, both B
          // bands of the unit.  They land well before the operand tiles, so
          // the copy warps move them into tensor memory meanwhile.  A scale
          // tile covers 128 (MXFP8) or 64 (NVFP4) elements of the contraction.
          const int64_t a_atom = ea / (NVF4 ? 64 : 128);
          const int64_t b_atom = eb / (NVF4 ? 64 : 128);
          tma_load_2d_pair(ssfa, &tmap_sfa, sfb_bar, 0,
                           static_cast<int32_t>(a_band * p.a_atoms_row + a_atom));
          tma_load_3d_pair(ssfb, &tmap_sfb, sfb_bar, 0, static_cast<int32_t>(b_atom), b_band);
#pragma unroll
          for (int sub = 0; sub < Cfg::kSubTiles; ++sub) {
            const uint32_t off = static_cast<uint32_t>(sub * 128 * Cfg::kSubK);
            tma_load_2d_pair(sa + off, &tmap_a, fb,
                             static_cast<int32_t>(ea / EPB + sub * Cfg::kSubK),
                             static_cast<int32_t>(ti.a_row));
            tma_load_2d_pair(sb + off, &tmap_b, fb,
                             static_cast<int32_t>(eb / EPB + sub * Cfg::kSubK), b_half);
          }
          issued_mask |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // the even CTA's full and scale barriers count both CTAs' bytes: once
      // they have completed, every copy of the pair has landed
      if (rank == 0)
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask & (1u << s)) {
            mbar_wait_drain(full_bar(s), (last_parity >> s) & 1u, p.status, p.timeout_ns);
            mbar_wait_drain(sffull_bar(s), (last_parity >> s) & 1u, p.status, p.timeout_ns);
          }
    }
  }
  // ------------------------------------------------------------ MMA issuer (even CTA)
  else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      uint32_t stage = 0, phase = 0, acc_phase = 0;
      bool ok = true;
      for (int64_t t = unit0, u = 0; ok && t < total_units; t += ustride, ++u) {
        // the unit's shape, as the producer published it
        const uint32_t slot = static_cast<uint32_t>(u & 1), ipar = static_cast<uint32_t>((u >> 1) & 1);
        if (!mbar_wait(info_full_bar(slot), ipar, abort_flag, p.status, p.timeout_ns)) break;
        const uint64_t info = info_word[slot];
        mbar_arrive(info_empty_bar(slot));
        const int64_t kb_count = static_cast<int64_t>(info & kInfoKbMask);
        const int last_mmas = static_cast<int>((info >> 48) & 0xFFu);
        const bool half_n = (info >> 56) & 1u;
        if (!mbar_wait(tempty_bar, acc_phase ^ 1u, abort_flag, p.status, p.timeout_ns)) break;
        tc_fence_after();
        for (int64_t kb = 0; kb < kb_count; ++kb) {
          // operands landed, and their scale tiles are in tensor memory
          if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_base + stage * Cfg::kStageBytes;
          const uint32_t sb = sa + Cfg::kATile;
          const uint32_t sfa_t = tmem_base + Cfg::BN + stage * Cfg::kSfCols;
          const uint32_t sfb_t = sfa_t + Cfg::kSfaCols;
          const uint32_t idesc = half_n ? Cfg::kIdescN128 : Cfg::kIdesc;
          const int nmma = kb + 1 == kb_count ? last_mmas : Cfg::kMmas;
#pragma unroll
          for (int kk = 0; kk < Cfg::kMmas; ++kk) {
            if (kk >= nmma) break;  // rows of the next group (wgrad): loaded, not used
            // K step kk: sub-tile kk / kMmasPerSub, 32 bytes further along the
            // row per step within it (16-byte units)
            const int sub = kk / Cfg::kMmasPerSub, ks = kk % Cfg::kMmasPerSub;
            const uint32_t off = static_cast<uint32_t>(sub * 128 * Cfg::kSubK);
            const uint64_t adesc = smem_desc(sa + off, 16, 8 * Cfg::kSubK, Cfg::kSwizzle) + 2 * ks;
            const uint64_t bdesc = smem_desc(sb + off, 16, 8 * Cfg::kSubK, Cfg::kSwizzle) + 2 * ks;
            const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
            if (NVF4) {
              tc_mma_nvf4_pair(tmem_base, adesc, bdesc, idesc, sfa_t + 4 * kk, sfb_t + 8 * kk,
                               accum);
            } else {
              // scale tile kk / 4 (A at 4 columns per tile, B's two bands at 8),
              // byte kk % 4 of its 32-bit columns
              const uint32_t sid = static_cast<uint32_t>(kk & 3), atom = static_cast<uint32_t>(kk >> 2);
              tc_mma_mxf8_pair(tmem_base, adesc, bdesc, idesc | (sid << 4) | (sid << 29),
                               sfa_t + 4 * atom, sfb_t + 8 * atom, accum);
            }
          }
          tc_commit_pair_mc(empty_bar(stage), 0x3);  // stage free in both CTAs
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // accumulator ready in both CTAs (the test hook withholds the first
        // arrival of cluster 0 so that the epilogues' bounded waits run out)
        if (!((p.inject & 1) && blockIdx.x == 0 && t == unit0)) tc_commit_pair_mc(tfull_bar, 0x3);
        acc_phase ^= 1u;
      }
      tc_commit_pair(drain_bar);
      mbar_wait_drain(drain_bar, 0, p.status, p.timeout_ns);
    }
  }
  // ------------------------------------------------------------ scale copies (even CTA)
  else if (warp >= kFirstSfWarp) {
    if (lane == 0 && rank == 0) {
      const int j = static_cast<int>(warp - kFirstSfWarp);
      uint32_t stage = 0, phase = 0;
      for (int64_t t = unit0, u = 0; t < total_units; t += ustride, ++u) {
        const uint32_t slot = static_cast<uint32_t>(u & 1), ipar = static_cast<uint32_t>((u >> 1) & 1);
        if (!mbar_wait(info_full_bar(slot), ipar, abort_flag, p.status, p.timeout_ns)) break;
        const int64_t kb_count = static_cast<int64_t>(info_word[slot] & kInfoKbMask);
        mbar_arrive(info_empty_bar(slot));
        bool ok = true;
        for (int64_t kb = 0; kb < kb_count; ++kb) {
          // the stage's previous MMAs finished before its producer refilled it
          // (empty barrier), so its scale columns are free once its scale
          // tiles have landed
          if (!mbar_wait(sffull_bar(stage), phase, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ssfa = smem_base + stage * Cfg::kStageBytes + Cfg::kATile + Cfg::kBTile;
          const uint32_t ssfb = ssfa + Cfg::kSfaBytes;
          const uint32_t sfa_t = tmem_base + Cfg::BN + stage * Cfg::kSfCols;
          const uint32_t sfb_t = sfa_t + Cfg::kSfaCols;
          // copy c: A tile a = c at column 4a; B (band i, K-step a) at 8a + 4i
#pragma unroll
          for (int c = 0; c < Cfg::kSfCopies; ++c) {
            if (c % Cfg::kSfWarps != j) continue;
            if (c < Cfg::kAtomsK) {
              tc_cp_scales_pair(sfa_t + 4 * c, smem_desc(ssfa + 512 * c, 0, 128, 0));
            } else {
              const int i = (c - Cfg::kAtomsK) / Cfg::kAtomsK, a = (c - Cfg::kAtomsK) % Cfg::kAtomsK;
              tc_cp_scales_pair(sfb_t + 8 * a + 4 * i,
                                smem_desc(ssfb + i * 512 * Cfg::kAtomsK + 512 * a, 0, 128, 0));
            }
          }
          // one of the full barrier's arrivals: the MMA thread waits there for
          // the operand bytes and these scale copies alike
          tc_commit_pair(full_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      // every copy this thread issued has completed before TMEM is freed
      tc_commit_pair(sfdrain_bar);
      mbar_wait_drain(sfdrain_bar, 0, p.status, p.timeout_ns);
    }
  }
  // ------------------------------------------------------------ epilogue (both CTAs)
  else {
    const uint32_t ew = warp - 2;
    const uint32_t quarter = warp & 3u;
    const uint32_t col0 = 128u * (ew >> 2);
    const uint32_t tempty_even = mapa_shared(tempty_bar, 0);
    uint32_t acc_phase = 0;
    for (int64_t t = unit0; t < total_units; t += ustride) {
      const TileInfo ti = map_unit_pair<EPB, BK>(t, p, row_off, prow_off, tile_off, rank);
      // this warp's 128 columns' operands (NVFP4 column outer scales, bias)
      // copied into its shared-memory slots while it waits (lane l: columns
      // 4l..4l+3), read back by every lane in the epilogue
      float* scs = colsm + ew * 128;
      float* sbs = colsm + ((NVF4 ? Cfg::kEpiWarps : 0) + ew) * 128;
      __syncwarp();  // the previous unit's reads of the slots are done
      if ((NVF4 || p.bias) && ti.c_col + col0 < p.out_cols) {
        const float* srcs[2] = {
            NVF4 ? p.b_outer + (p.mode == 1 ? static_cast<int64_t>(ti.g) * p.K : 0) + ti.b_row +
                       col0 + 4 * lane
                 : nullptr,
            p.bias ? p.bias + static_cast<int64_t>(ti.g) * p.out_cols + ti.c_col + col0 + 4 * lane
                   : nullptr};
        float* dsts[2] = {scs + 4 * lane, sbs + 4 * lane};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          if (!srcs[q]) continue;
          if (p.vec_col) {
            cp_async_16(smem_u32(dsts[q]), srcs[q]);
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) cp_async_4(smem_u32(dsts[q] + c), srcs[q] + c);
          }
        }
      }
      cp_async_commit();
      if (!mbar_wait(tfull_bar, acc_phase, abort_flag, p.status, p.timeout_ns)) {
        cp_async_wait_all();  // no copy into this CTA's shared memory outlives it
        break;
      }
      tc_fence_after();
      uint32_t v[4][32];
      const bool has_k = ti.kb_count > 0;
      if (has_k) {
        const uint32_t taddr = tmem_base + ((32u * quarter) << 16) + col0;
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(taddr + 32 * c, v[c]);
        tmem_ld_wait();
      }
      // the loads have completed (wait::ld): TMEM may be overwritten.  The
      // arrival is relaxed so that it does not wait for this warp's stores
      // of the previous unit to drain
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(tempty_even);
      acc_phase ^= 1u;
      cp_async_wait_all();
      __syncwarp();  // every lane's copies have landed
      epilogue_row<NVF4, true>(p, ti, ti.c_row + 32 * quarter + lane, col0, v, has_k, EpiCols{},
                               scs, sbs);
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no copy, commit or remote arrival still targets either CTA
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
namespace {

// 2-D byte tensor [rows, inner_bytes] with rows row_bytes apart, box
// [box_rows, bk bytes], with the swizzle of the same width (the layout the
// K-major MMA descriptors above describe).
bool make_tmap(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows,
               uint64_t row_bytes, uint32_t box_rows, int bk) {
  const int box = bk > 128 ? 128 : bk;  // a 256-byte stage is loaded as two boxes
  return make_tmap_2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, inner_bytes, rows, row_bytes,
                      static_cast<uint32_t>(box), box_rows,
                      box == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

// Launch as 2-CTA clusters: as many co-resident clusters as the device holds
// (one CTA per SM), at most max_units of them.
template <typename Kern, typename... Args>
cudaError_t launch_clusters(Kern kern, int threads, size_t smem, int64_t max_units, int num_sms,
                            cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1), 1, 1);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1)
    clusters = num_sms / 2;
  const int64_t n = max_units < clusters ? max_units : clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * n), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int BN, int STAGES, int ACC, bool NVF4, int BK>
cudaError_t launch_variant(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                           int64_t max_units, int num_sms, cudaStream_t stream) {
  using Cfg = GemmCfg<BN, STAGES, ACC, NVF4, BK>;
  auto kern = grouped_gemm_kernel<BN, STAGES, ACC, NVF4, BK>;
  const size_t smem = Cfg::smem_bytes(p.G);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (max_units <= 0) return cudaSuccess;
  const int grid = static_cast<int>(max_units < num_sms ? max_units : num_sms);
  kern<<<grid, Cfg::kThreads, smem, stream>>>(ta, tb, p);
  return cudaGetLastError();
}

template <int STAGES, bool NVF4, int BKB>
cudaError_t launch_pair_variant(const CUtensorMap& ta, const CUtensorMap& tb,
                                const CUtensorMap& tsa, const CUtensorMap& tsb,
                                const GemmParams& p, int64_t max_units, int num_sms,
                                cudaStream_t stream) {
  using Cfg = PairCfg<STAGES, NVF4, BKB>;
  auto kern = grouped_gemm_pair_kernel<STAGES, NVF4, BKB>;
  const size_t smem = Cfg::smem_bytes(p.G, p.bias != nullptr);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (max_units <= 0) return cudaSuccess;
  return launch_clusters(kern, Cfg::kThreads, smem, max_units, num_sms, stream, ta, tb, tsa, tsb,
                         p);
}

}  // namespace

// Kernel choice.  Default (tile_n = 0): the CTA-pair kernel, 256 x 256
// units, whenever B has at least 256 rows; otherwise the single-CTA kernel.
// tile_n = 256 or 128 forces the single-CTA kernel with that tile width (256
// needs an output width that allows it); stage_bytes = 128 forces 128-byte K
// stages where the default would take 256 (MXFP8 fprop with K % 256 == 0).
// Both overrides exist for the parity tests of every kernel variant.
cudaError_t launch_grouped_gemm(bool nvfp4, int mode, const void* a_data, const uint8_t* a_sf,
                                const float* a_outer, const void* b_data, const uint8_t* b_sf,
                                const float* b_outer, const int64_t* group_ws, int G, int64_t M_cap,
                                int64_t N, int64_t K, const float* alpha, const float* beta,
                                const float* bias, void* C, int out_bf16, int32_t* status,
                                int num_sms, int tile_n, int stage_bytes, int inject,
                                uint64_t timeout_ns, int unaligned, int64_t a_ld_bytes,
                                int64_t b_ld_bytes, cudaStream_t stream) {
  GemmParams p;
  p.unaligned = unaligned;
  p.inject = inject;
  p.timeout_ns = timeout_ns;
  p.a_sf = a_sf;
  p.b_sf = b_sf;
  p.a_outer = a_outer;
  p.b_outer = b_outer;
  p.group_ws = group_ws;
  p.alpha = alpha;
  p.beta = beta;
  p.bias = bias;
  p.C = C;
  p.c_align32 = (reinterpret_cast<uintptr_t>(C) & 31u) == 0 ? 1 : 0;
  p.vec_col = ((reinterpret_cast<uintptr_t>(b_outer) | reinterpret_cast<uintptr_t>(bias)) & 15u) == 0
                  ? 1 : 0;
  p.status = status;
  p.M_cap = M_cap;
  p.N = N;
  p.K = K;
  p.G = G;
  p.mode = mode;
  p.out_bf16 = out_bf16;
  // operand geometry: rows x contraction length (elements) of A and B
  //   fprop: A [M_cap, K], B [G*N, K];  wgrad: A [N, M_cap], B [K, M_cap];
  //   dgrad: A [M_cap, N], B [K, G*N]  (the transposed weight copy)
  // With unaligned groups the colwise copies and A's scales are padded per
  // group: M_pad = M_cap + 128 G rows replace M_cap there.
  const int64_t M_pad = unaligned ? M_cap + 128 * static_cast<int64_t>(G) : M_cap;
  const int64_t a_rows = mode == 0 ? M_cap : (mode == 1 ? N : M_cap);
  const int64_t b_rows = mode == 0 ? G * N : K;
  const int64_t a_kdim = mode == 0 ? K : (mode == 1 ? M_pad : N);
  const int64_t b_kdim = mode == 0 ? K : (mode == 1 ? M_pad : G * N);
  const int64_t a_sf_rows = mode == 1 ? a_rows : M_pad;  // rows of A's scale matrix
  const int64_t blk = nvfp4 ? 16 : 32;
  p.a_atoms_row = a_kdim / blk / 4;
  p.b_atoms_row = b_kdim / blk / 4;
  const bool pair_kernel = tile_n == 0 && b_rows >= 256;
  if (unaligned && !(pair_kernel && !nvfp4)) return cudaErrorInvalidValue;
  // bytes of K per pipeline stage.  An NVFP4 fprop whose K is not a multiple
  // of 256 elements needs 64, and so does NVFP4 wgrad on the single-CTA
  // kernel (a 128-row group is 64 bytes of E2M1 along the contraction).
  // 256-byte stages: MXFP8 fprop on the CTA-pair kernel with K % 256 == 0
  // (measured: fine-grained fprop 2.5 % faster, Mixtral fprop unchanged;
  // dgrad lost 2 % with 3 stages instead of 6 and keeps 128) and MXFP8 wgrad
  // on it.  The CTA-pair kernel lets a wgrad group end inside its last K
  // block (only that block's first MMAs run), so wgrad takes the wide stages
  // there: 8 MMAs per stage (MXFP8), 4 (NVFP4, 128 bytes), where 4 and 2
  // left the MMA thread's per-stage wait and commit on the critical path.
  const bool need64 = nvfp4 && ((mode == 1 && !pair_kernel) || (mode == 0 && (K % 256) != 0));
  const bool wide = !nvfp4 && stage_bytes == 0 && pair_kernel &&
                    ((mode == 0 && K % 256 == 0) || mode == 1);
  const int BKB = need64 ? 64 : (wide ? 256 : 128);
  p.kb_uniform = mode == 0 ? (nvfp4 ? K / 2 : K) / BKB : (mode == 2 ? N / BKB : 0);
  p.out_cols = mode == 0 ? N : K;

  if (pair_kernel) {
    CUtensorMap ta, tb, tsa, tsb;
    const int atoms = nvfp4 ? BKB / 32 : BKB / 128;  // scale tiles along K per stage and band
    const uint64_t b_bands = static_cast<uint64_t>(b_rows / 128);
    const uint64_t sfb_dims[3] = {128, static_cast<uint64_t>(p.b_atoms_row), b_bands};
    const uint64_t sfb_strides[2] = {512, static_cast<uint64_t>(512 * p.b_atoms_row)};
    const uint32_t sfb_box[3] = {128, static_cast<uint32_t>(atoms), 2};
    const int64_t ebn = nvfp4 ? 1 : 2;  // bytes per element x 2
    if (!make_tmap(&ta, a_data, static_cast<uint64_t>(a_kdim * ebn / 2), a_rows,
                   static_cast<uint64_t>(a_ld_bytes), 128, BKB) ||
        !make_tmap(&tb, b_data, static_cast<uint64_t>(b_kdim * ebn / 2), b_rows,
                   static_cast<uint64_t>(b_ld_bytes), 128, BKB) ||
        !make_tmap_2d(&tsa, CU_TENSOR_MAP_DATA_TYPE_UINT32, a_sf, 128,
                      static_cast<uint64_t>((a_sf_rows / 128) * p.a_atoms_row), 512, 128,
                      static_cast<uint32_t>(atoms), CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_tmap_3d(&tsb, CU_TENSOR_MAP_DATA_TYPE_UINT32, b_sf, sfb_dims, sfb_strides, sfb_box))
      return cudaErrorInvalidValue;
    const int64_t units = mode == 1 ? G * (((N / 128) + 1) / 2) * ((K + 255) / 256)
                                    : (((M_cap / 128) + G + 1) / 2) * ((p.out_cols + 255) / 256);
    if (nvfp4 && BKB == 64)
      return launch_pair_variant<10, true, 64>(ta, tb, tsa, tsb, p, units, num_sms, stream);
    if (nvfp4) return launch_pair_variant<5, true, 128>(ta, tb, tsa, tsb, p, units, num_sms, stream);
    if (BKB == 256)
      return launch_pair_variant<3, false, 256>(ta, tb, tsa, tsb, p, units, num_sms, stream);
    return launch_pair_variant<6, false, 128>(ta, tb, tsa, tsb, p, units, num_sms, stream);
  }

  // single-CTA kernel: tile width 256 where asked for (or by default) and the
  // output width allows it, else 128
  const int bn = (tile_n == 128 || p.out_cols % 256 != 0) ? 128 : 256;
  const int64_t ebytes_num = nvfp4 ? 1 : 2;  // bytes per element x 2
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, a_data, static_cast<uint64_t>(a_kdim * ebytes_num / 2), a_rows,
                 static_cast<uint64_t>(a_ld_bytes), 128, BKB) ||
      !make_tmap(&tb, b_data, static_cast<uint64_t>(b_kdim * ebytes_num / 2), b_rows,
                 static_cast<uint64_t>(b_ld_bytes), bn, BKB))
    return cudaErrorInvalidValue;
  // upper bound on the work units (device-side group sizes are unknown here)
  const int64_t max_units = mode == 1 ? G * (N / 128) * (K / bn)
                                      : (M_cap / 128) * (p.out_cols / bn);
  if (BKB == 64) {  // NVFP4 with half-size stages, twice as many
    if (bn == 256) return launch_variant<256, 7, 1, true, 64>(ta, tb, p, max_units, num_sms, stream);
    return launch_variant<128, 10, 2, true, 64>(ta, tb, p, max_units, num_sms, stream);
  }
  if (nvfp4) {
    if (bn == 256) return launch_variant<256, 4, 1, true, 128>(ta, tb, p, max_units, num_sms, stream);
    return launch_variant<128, 5, 2, true, 128>(ta, tb, p, max_units, num_sms, stream);
  }
  if (bn == 256) return launch_variant<256, 4, 1, false, 128>(ta, tb, p, max_units, num_sms, stream);
  return launch_variant<128, 6, 2, false, 128>(ta, tb, p, max_units, num_sms, stream);
}

}  // namespace mxg
