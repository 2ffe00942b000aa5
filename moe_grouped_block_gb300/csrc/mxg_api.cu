// mxg_api.cu -- the C ABI declared in include/mxg.h: argument validation,
// device checks and kernel dispatch.  Host code only; no allocation, no
// synchronisation.
#include <atomic>
#include <mutex>

#include "mxg_device.cuh"

namespace mxg {
cudaError_t launch_group_offsets(const void* sizes, int is_int64, int G, int64_t mult,
                                 int64_t last_dim, int64_t cap, int64_t* ws, int32_t* status,
                                 cudaStream_t stream, int round128);
cudaError_t launch_mxfp8_quantize(bool row, bool col, const uint16_t* x, int64_t cap, int64_t cols,
                                  const int64_t* group_ws, int G, uint8_t* q_row, uint8_t* sf_row,
                                  uint8_t* q_col, uint8_t* sf_col, int32_t* status, int num_sms,
                                  cudaStream_t stream, bool unaligned);
cudaError_t launch_nvfp4_quantize(const uint16_t* x, int64_t cap, int64_t cols,
                                  const int64_t* group_ws, int G, uint8_t* q, uint8_t* sf,
                                  float* outer, int32_t* status, int num_sms, cudaStream_t stream);
cudaError_t launch_nvfp4_quantize_colwise(const uint16_t* x, int64_t cap, int64_t cols,
                                          const int64_t* group_ws, int G, uint8_t* qT,
                                          uint8_t* sfT, float* outer, int num_sms,
                                          cudaStream_t stream);
cudaError_t launch_dequantize(int nvfp4, int colwise, const uint8_t* q, const uint8_t* sf,
                              const float* outer, int64_t rows, int64_t cols, void* out, int bf16,
                              int num_sms, cudaStream_t stream);
cudaError_t launch_grouped_gemm(bool nvfp4, int mode, const void* a_data, const uint8_t* a_sf,
                                const float* a_outer, const void* b_data, const uint8_t* b_sf,
                                const float* b_outer, const int64_t* group_ws, int G, int64_t M_cap,
                                int64_t N, int64_t K, const float* alpha, const float* beta,
                                const float* bias, void* C, int out_bf16, int32_t* status,
                                int num_sms, int tile_n, int stage_bytes, int inject,
                                uint64_t timeout_ns, int unaligned, int64_t a_ld_bytes,
                                int64_t b_ld_bytes, cudaStream_t stream);
cudaError_t launch_wgrad_no_rows(int G, int64_t N, int64_t K, const float* beta, void* C,
                                 int out_bf16, int num_sms, cudaStream_t stream);
constexpr uint64_t kDefaultWaitNs = 1000000000ull;
}  // namespace mxg

namespace {

std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
struct DevInfo {
  int checked = 0;  // 0 unknown, 1 sm_103, -1 other
  int num_sms = 0;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Confirms the current device is sm_103 (GB300) and returns its SM count.
mxg_status_t current_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return MXG_ERR_UNSUPPORTED_ARCH;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.checked == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MXG_ERR_UNSUPPORTED_ARCH;
    d.checked = (major == 10 && minor == 3) ? 1 : -1;
    d.num_sms = sms;
  }
  if (d.checked != 1) return MXG_ERR_UNSUPPORTED_ARCH;
  *num_sms = d.num_sms;
  return MXG_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool mult128(int64_t v) { return v >= 0 && (v & 127) == 0; }

mxg_status_t launched(cudaError_t e, uint64_t n) {
  if (e != cudaSuccess) return MXG_ERR_LAUNCH;
  g_launches.fetch_add(n, std::memory_order_relaxed);
  return MXG_OK;
}

// The kernels index rows (and the padded rows of groups of any size) with
// 32-bit integers in their group tables.
constexpr int64_t kMaxRows = 0x7FFFFF80LL;

// Arguments of the offsets entry points.  Bounds on the multiplier (2^31)
// and on the capacity (2^62, and capacity * last_dim within int64) keep every
// product the kernel forms -- sanitised rows times the multiplier, offsets
// times last_dim -- inside 64 bits.
bool offsets_args_ok(const void* sizes, const int64_t* ws, int G, int64_t multiplier,
                     int64_t last_dim, int64_t rows_capacity) {
  return sizes != nullptr && ws != nullptr && G >= 1 && G <= 65536 && multiplier >= 1 &&
         multiplier <= (1LL << 31) && last_dim >= 1 && rows_capacity >= 0 &&
         rows_capacity <= (1LL << 62) && rows_capacity <= INT64_MAX / last_dim;
}

// Checks an operand descriptor's rows / cols (0 = as the mode implies) and
// leading dimension (0 = dense) and returns the data's row stride in bytes.
mxg_status_t operand_shape(const mxg_operand_t* op, int64_t rows, int64_t cols, bool nvfp4,
                           int64_t* ld_bytes) {
  if ((op->rows != 0 && op->rows != rows) || (op->cols != 0 && op->cols != cols))
    return MXG_ERR_INVALID_ARG;
  const int64_t ld = op->ld == 0 ? cols : op->ld;
  if (ld < cols) return MXG_ERR_INVALID_ARG;
  if (nvfp4 && (ld & 1)) return MXG_ERR_ALIGNMENT;
  const int64_t bytes = nvfp4 ? ld / 2 : ld;
  if (bytes % 16 != 0) return MXG_ERR_ALIGNMENT;
  *ld_bytes = bytes;
  return MXG_OK;
}

}  // namespace

extern "C" {

size_t mxg_offsets_workspace_bytes(int G) {
  return G < 1 ? 0 : static_cast<size_t>(2 * G + 1) * sizeof(int64_t);
}

mxg_status_t mxg_group_offsets(const void* sizes, int sizes_is_int64, int G, int64_t multiplier,
                               int64_t last_dim, int64_t rows_capacity, int64_t* ws,
                               int32_t* dev_status, mxg_stream_t stream) {
  if (!offsets_args_ok(sizes, ws, G, multiplier, last_dim, rows_capacity))
    return MXG_ERR_INVALID_ARG;
  int sms = 0;
  const mxg_status_t st = current_device(&sms);
  if (st != MXG_OK) return st;
  return launched(mxg::launch_group_offsets(sizes, sizes_is_int64 ? 1 : 0, G, multiplier, last_dim,
                                            rows_capacity, ws, dev_status,
                                            reinterpret_cast<cudaStream_t>(stream), 1),
                  1);
}

mxg_status_t mxg_group_offsets_unaligned(const void* sizes, int sizes_is_int64, int G,
                                         int64_t multiplier, int64_t last_dim,
                                         int64_t rows_capacity, int64_t* ws, int32_t* dev_status,
                                         mxg_stream_t stream) {
  if (!offsets_args_ok(sizes, ws, G, multiplier, last_dim, rows_capacity))
    return MXG_ERR_INVALID_ARG;
  int sms = 0;
  const mxg_status_t st = current_device(&sms);
  if (st != MXG_OK) return st;
  return launched(mxg::launch_group_offsets(sizes, sizes_is_int64 ? 1 : 0, G, multiplier, last_dim,
                                            rows_capacity, ws, dev_status,
                                            reinterpret_cast<cudaStream_t>(stream), 0),
                  1);
}

int64_t mxg_unaligned_rows_capacity(int64_t rows_capacity, int G) {
  if (rows_capacity < 0 || G < 1) return 0;
  return rows_capacity + 128 * static_cast<int64_t>(G);
}

mxg_status_t mxg_group_quantize_unaligned(mxg_qlayout_t layout, const void* x,
                                          int64_t rows_capacity, int64_t cols,
                                          const int64_t* group_ws, int G, uint8_t* q_row,
                                          uint8_t* sf_row, uint8_t* q_col, uint8_t* sf_col,
                                          int32_t* dev_status, mxg_stream_t stream) {
  if (x == nullptr || group_ws == nullptr || G < 1 || G > 1024) return MXG_ERR_INVALID_ARG;
  if (layout != MXG_ROWWISE && layout != MXG_COLWISE && layout != MXG_BOTH)
    return MXG_ERR_INVALID_ARG;
  const bool row = (layout & MXG_ROWWISE) != 0, col = (layout & MXG_COLWISE) != 0;
  if ((row && (q_row == nullptr || sf_row == nullptr)) ||
      (col && (q_col == nullptr || sf_col == nullptr)))
    return MXG_ERR_INVALID_ARG;
  if (!mult128(rows_capacity) || !mult128(cols) || cols == 0) return MXG_ERR_ALIGNMENT;
  if (rows_capacity + 128 * static_cast<int64_t>(G) > kMaxRows) return MXG_ERR_INVALID_ARG;
  if (!aligned16(x) || (row && (!aligned16(q_row) || !aligned16(sf_row))) ||
      (col && (!aligned16(q_col) || !aligned16(sf_col))))
    return MXG_ERR_ALIGNMENT;
  int sms = 0;
  const mxg_status_t st = current_device(&sms);
  if (st != MXG_OK) return st;
  if (rows_capacity == 0) return MXG_OK;
  return launched(mxg::launch_mxfp8_quantize(row, col, static_cast<const uint16_t*>(x),
                                             rows_capacity, cols, group_ws, G, q_row, sf_row,
                                             q_col, sf_col, dev_status, sms,
                                             reinterpret_cast<cudaStream_t>(stream), true),
                  1);
}

mxg_status_t mxg_group_quantize(mxg_format_t fmt, mxg_qlayout_t layout, const void* x,
                                int64_t rows_capacity, int64_t cols, const int64_t* group_ws,
                                int G, void* q_row, uint8_t* sf_row, void* q_col, uint8_t* sf_col,
                                float* outer_row, float* outer_col, int32_t* dev_status,
                                mxg_stream_t stream) {
  if (x == nullptr || (group_ws != nullptr && (G < 1 || G > 65536))) return MXG_ERR_INVALID_ARG;
  if (layout != MXG_ROWWISE && layout != MXG_COLWISE && layout != MXG_BOTH)
    return MXG_ERR_INVALID_ARG;
  const bool row = (layout & MXG_ROWWISE) != 0, col = (layout & MXG_COLWISE) != 0;
  if (fmt == MXG_MXFP8_E4M3) {
    if ((row && (q_row == nullptr || sf_row == nullptr)) ||
        (col && (q_col == nullptr || sf_col == nullptr)))
      return MXG_ERR_INVALID_ARG;
  } else if (fmt == MXG_NVFP4_ROWSCALED) {
    if ((row && (q_row == nullptr || sf_row == nullptr || outer_row == nullptr)) ||
        (col && (q_col == nullptr || sf_col == nullptr || outer_col == nullptr)) ||
        (col && group_ws != nullptr && G > 1024))
      return MXG_ERR_INVALID_ARG;
  } else {
    return MXG_ERR_INVALID_ARG;
  }
  if (!mult128(rows_capacity) || !mult128(cols) || cols == 0) return MXG_ERR_ALIGNMENT;
  if (!aligned16(x) || (row && (!aligned16(q_row) || !aligned16(sf_row))) ||
      (col && (!aligned16(q_col) || !aligned16(sf_col))))
    return MXG_ERR_ALIGNMENT;
  int sms = 0;
  const mxg_status_t st = current_device(&sms);
  if (st != MXG_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (rows_capacity == 0) {
    // no rows: every group is empty, and the NVFP4 colwise outer scales of an
    // empty group are 0 (the colwise kernel needs rows for its tensor map)
    if (fmt == MXG_NVFP4_ROWSCALED && col &&
        cudaMemsetAsync(outer_col, 0,
                        static_cast<size_t>(group_ws ? G : 1) * static_cast<size_t>(cols) *
                            sizeof(float),
                        s) != cudaSuccess)
      return MXG_ERR_LAUNCH;
    return MXG_OK;
  }
  if (fmt == MXG_MXFP8_E4M3)
    return launched(mxg::launch_mxfp8_quantize(row, col, static_cast<const uint16_t*>(x),
                                               rows_capacity, cols, group_ws, G,
                                               static_cast<uint8_t*>(q_row), sf_row,
                                               static_cast<uint8_t*>(q_col), sf_col, dev_status,
                                               sms, s, false),
                    1);
  if (row) {
    const mxg_status_t r = launched(
        mxg::launch_nvfp4_quantize(static_cast<const uint16_t*>(x), rows_capacity, cols, group_ws,
                                   G, static_cast<uint8_t*>(q_row), sf_row, outer_row, dev_status,
                                   sms, s),
        1);
    if (r != MXG_OK || !col) return r;
  }
  return launched(mxg::launch_nvfp4_quantize_colwise(static_cast<const uint16_t*>(x), rows_capacity,
                                                     cols, group_ws, G,
                                                     static_cast<uint8_t*>(q_col), sf_col,
                                                     outer_col, sms, s),
                  1);
}

static mxg_status_t grouped_gemm_impl(mxg_format_t fmt, mxg_gemm_mode_t mode,
                                      const mxg_operand_t* A, const mxg_operand_t* B,
                                      const int64_t* group_ws, int G, int64_t M_cap, int64_t N,
                                      int64_t K, const float* alpha, const float* beta,
                                      const float* bias, void* C, mxg_out_t out_type,
                                      int32_t* dev_status, int tile_n, int stage_bytes,
                                      int inject, uint64_t timeout_ns, mxg_stream_t stream,
                                      int unaligned) {
  if (A == nullptr || B == nullptr || C == nullptr || group_ws == nullptr || G < 1 || G > 1024)
    return MXG_ERR_INVALID_ARG;
  if (fmt != MXG_MXFP8_E4M3 && fmt != MXG_NVFP4_ROWSCALED) return MXG_ERR_INVALID_ARG;
  if (mode != MXG_FPROP_TN && mode != MXG_WGRAD_NT && mode != MXG_DGRAD_NN)
    return MXG_ERR_INVALID_ARG;
  if (out_type != MXG_OUT_F32 && out_type != MXG_OUT_BF16) return MXG_ERR_INVALID_ARG;
  if (A->data == nullptr || A->scale == nullptr || B->data == nullptr || B->scale == nullptr)
    return MXG_ERR_INVALID_ARG;
  const bool nv = fmt == MXG_NVFP4_ROWSCALED;
  if (nv && (mode == MXG_DGRAD_NN || beta != nullptr || A->outer == nullptr || B->outer == nullptr))
    return MXG_ERR_INVALID_ARG;  // row-scaled NVFP4: fprop and wgrad, no beta
  if (bias != nullptr && mode == MXG_WGRAD_NT) return MXG_ERR_INVALID_ARG;
  // unaligned groups: MXFP8 on the CTA-pair kernel, whose B spans >= 256 rows
  if (unaligned && (nv || (mode == MXG_FPROP_TN ? N * static_cast<int64_t>(G) : K) < 256))
    return MXG_ERR_INVALID_ARG;
  if (!mult128(M_cap) || !mult128(N) || !mult128(K) || N == 0 || K == 0)
    return MXG_ERR_ALIGNMENT;

  if (M_cap + (unaligned ? 128 * static_cast<int64_t>(G) : 0) > kMaxRows ||
      N * static_cast<int64_t>(G) > kMaxRows)
    return MXG_ERR_INVALID_ARG;
  if (!aligned16(A->data) || !aligned16(A->scale) || !aligned16(B->data) || !aligned16(B->scale) ||
      !aligned16(C))
    return MXG_ERR_ALIGNMENT;
  // operand shapes the mode implies (rows x contraction elements) and the
  // leading dimensions of the data, in bytes
  const int64_t M_pad = M_cap + (unaligned ? 128 * static_cast<int64_t>(G) : 0);
  const int64_t a_rows = mode == MXG_WGRAD_NT ? N : M_cap;
  const int64_t a_cols = mode == MXG_FPROP_TN ? K : (mode == MXG_WGRAD_NT ? M_pad : N);
  const int64_t b_rows = mode == MXG_FPROP_TN ? N * static_cast<int64_t>(G) : K;
  const int64_t b_cols = mode == MXG_FPROP_TN ? K : (mode == MXG_WGRAD_NT ? M_pad : N * G);
  int64_t a_ld = 0, b_ld = 0;
  mxg_status_t sh = operand_shape(A, a_rows, a_cols, nv, &a_ld);
  if (sh != MXG_OK) return sh;
  if ((sh = operand_shape(B, b_rows, b_cols, nv, &b_ld)) != MXG_OK) return sh;
  int sms = 0;
  const mxg_status_t st = current_device(&sms);
  if (st != MXG_OK) return st;
  if (M_cap == 0) {
    // no rows: the fprop and dgrad outputs are empty; every wgrad group is
    // empty, and each dW_g is written as for an empty group
    if (mode != MXG_WGRAD_NT) return MXG_OK;
    return launched(mxg::launch_wgrad_no_rows(G, N, K, beta, C, out_type == MXG_OUT_BF16 ? 1 : 0,
                                              sms, reinterpret_cast<cudaStream_t>(stream)),
                    1);
  }
  return launched(mxg::launch_grouped_gemm(
                      nv, mode == MXG_WGRAD_NT ? 1 : (mode == MXG_DGRAD_NN ? 2 : 0), A->data, A->scale, A->outer, B->data,
                      B->scale, B->outer, group_ws, G, M_cap, N, K, alpha, beta, bias, C,
                      out_type == MXG_OUT_BF16 ? 1 : 0, dev_status, sms, tile_n, stage_bytes,
                      inject, timeout_ns, unaligned, a_ld, b_ld,
                      reinterpret_cast<cudaStream_t>(stream)),
                  1);
}

mxg_status_t mxg_grouped_gemm(mxg_format_t fmt, mxg_gemm_mode_t mode, const mxg_operand_t* A,
                              const mxg_operand_t* B, const int64_t* group_ws, int G,
                              int64_t M_cap, int64_t N, int64_t K, const float* alpha,
                              const float* beta, const float* bias, void* C, mxg_out_t out_type,
                              void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              mxg_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  return grouped_gemm_impl(fmt, mode, A, B, group_ws, G, M_cap, N, K, alpha, beta, bias, C,
                           out_type, dev_status, 0, 0, 0, mxg::kDefaultWaitNs, stream, 0);
}

mxg_status_t mxg_grouped_gemm_debug(mxg_format_t fmt, mxg_gemm_mode_t mode, const mxg_operand_t* A,
                                    const mxg_operand_t* B, const int64_t* group_ws, int G,
                                    int64_t M_cap, int64_t N, int64_t K, const float* alpha,
                                    const float* beta, const float* bias, void* C,
                                    mxg_out_t out_type, int32_t* dev_status, int tile_n,
                                    int stage_bytes, int inject_flags, int64_t wait_timeout_ns,
                                    mxg_stream_t stream) {
  if (wait_timeout_ns < 0 || (inject_flags & ~1)) return MXG_ERR_INVALID_ARG;
  if ((tile_n != 0 && tile_n != 128 && tile_n != 256) || (stage_bytes != 0 && stage_bytes != 128))
    return MXG_ERR_INVALID_ARG;
  const uint64_t t = wait_timeout_ns == 0 ? mxg::kDefaultWaitNs
                                          : static_cast<uint64_t>(wait_timeout_ns);
  return grouped_gemm_impl(fmt, mode, A, B, group_ws, G, M_cap, N, K, alpha, beta, bias, C,
                           out_type, dev_status, tile_n, stage_bytes, inject_flags, t, stream, 0);
}

mxg_status_t mxg_grouped_gemm_unaligned(mxg_gemm_mode_t mode, const mxg_operand_t* A,
                                        const mxg_operand_t* B, const int64_t* group_ws, int G,
                                        int64_t M_cap, int64_t N, int64_t K, const float* alpha,
                                        const float* beta, const float* bias, void* C,
                                        mxg_out_t out_type, int32_t* dev_status,
                                        mxg_stream_t stream) {
  return grouped_gemm_impl(MXG_MXFP8_E4M3, mode, A, B, group_ws, G, M_cap, N, K, alpha, beta, bias,
                           C, out_type, dev_status, 0, 0, 0, mxg::kDefaultWaitNs, stream, 1);
}

size_t mxg_grouped_gemm_workspace_bytes(mxg_format_t fmt, mxg_gemm_mode_t mode, int G,
                                        int64_t M_cap, int64_t N) {
  (void)fmt;
  (void)mode;
  (void)G;
  (void)M_cap;
  (void)N;
  return 0;
}

mxg_status_t mxg_dequantize(mxg_format_t fmt, mxg_qlayout_t layout, const void* q,
                            const uint8_t* sf, const float* outer, int64_t rows, int64_t cols,
                            void* out, mxg_out_t out_type, mxg_stream_t stream) {
  if (q == nullptr || sf == nullptr || out == nullptr) return MXG_ERR_INVALID_ARG;
  if (fmt != MXG_MXFP8_E4M3 && fmt != MXG_NVFP4_ROWSCALED) return MXG_ERR_INVALID_ARG;
  if (layout != MXG_ROWWISE && layout != MXG_COLWISE) return MXG_ERR_INVALID_ARG;
  if (out_type != MXG_OUT_F32 && out_type != MXG_OUT_BF16) return MXG_ERR_INVALID_ARG;
  if (fmt == MXG_NVFP4_ROWSCALED && layout == MXG_COLWISE) return MXG_ERR_UNSUPPORTED;
  if (!mult128(rows) || !mult128(cols)) return MXG_ERR_ALIGNMENT;
  int sms = 0;
  const mxg_status_t st = current_device(&sms);
  if (st != MXG_OK) return st;
  return launched(mxg::launch_dequantize(fmt == MXG_NVFP4_ROWSCALED ? 1 : 0,
                                         layout == MXG_COLWISE ? 1 : 0,
                                         static_cast<const uint8_t*>(q), sf, outer, rows, cols, out,
                                         out_type == MXG_OUT_BF16 ? 1 : 0, sms,
                                         reinterpret_cast<cudaStream_t>(stream)),
                  1);
}

const char* mxg_status_string(mxg_status_t status) {
  switch (status) {
    case MXG_OK: return "MXG_OK";
    case MXG_ERR_INVALID_ARG: return "MXG_ERR_INVALID_ARG";
    case MXG_ERR_ALIGNMENT: return "MXG_ERR_ALIGNMENT";
    case MXG_ERR_UNSUPPORTED_ARCH: return "MXG_ERR_UNSUPPORTED_ARCH";
    case MXG_ERR_LAUNCH: return "MXG_ERR_LAUNCH";
    case MXG_ERR_WORKSPACE_TOO_SMALL: return "MXG_ERR_WORKSPACE_TOO_SMALL";
    case MXG_ERR_UNSUPPORTED: return "MXG_ERR_UNSUPPORTED";
  }
  return "MXG_ERR_UNKNOWN";
}

int mxg_version(void) { return 100; }

uint64_t mxg_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
