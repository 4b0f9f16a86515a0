// mxq_api.cu -- the extern "C" entry points declared in include/mxq.h:
// argument validation, device checks, TMA descriptor encoding and dispatch
// to the kernels.  Host code only; it allocates nothing and never
// synchronises.

#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "mxq.h"
#include "mxq_internal.h"

namespace {

using mxq::DEFAULT_TIMEOUT_NS;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int checked = 0;     // 0 unknown, 1 sm_103, -1 other
  int num_sms = 0;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_device_mutex;

// Looks up (once per device) whether the current device is sm_103 and how
// many SMs it has.
mxq_status current_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXQ_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return MXQ_EARCH;
  std::lock_guard<std::mutex> lock(g_device_mutex);
  DeviceInfo& d = g_devices[dev];
  if (d.checked == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MXQ_ECUDA;
    d.checked = (major == 10 && minor == 3) ? 1 : -1;
    d.num_sms = sms;
  }
  if (d.checked < 0) return MXQ_EARCH;
  *num_sms = d.num_sms;
  return MXQ_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool load_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// Encodes a tensor map of `rank` dimensions (innermost first) with no
// swizzle; out-of-range loads read 0 and out-of-range stores are dropped.
mxq_status encode_map(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base,
                      const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                      const cuuint32_t* box,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  if (!load_encoder()) return MXQ_ECUDA;
  const cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  const CUresult r = g_encode(map, type, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
                              dims, strides_bytes, box, elem_strides,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MXQ_OK : MXQ_ECUDA;
}

// 2-D bf16 map over x[rows][cols] (row stride ldx elements).
mxq_status encode_bf16_map(CUtensorMap* map, const void* x, int64_t rows, int64_t cols,
                           int64_t ldx, int box_cols, int box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, dims, strides, box);
}

// Colwise-code map of an MXFP8 call quantizing an M x K matrix: [K][M]
// seen as [k % 8][k / 8][m], box 128 m x 16 x 8, 128-byte swizzle.
mxq_status encode_mx_qcol_map(CUtensorMap* map, int64_t M, int64_t K, uint8_t* q_col) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 8), 8};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(8 * M), static_cast<cuuint64_t>(M)};
  const cuuint32_t box[3] = {128, mxq::MX_TILE_K / 8, 8};
  return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, q_col, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
}

// Rowwise-code map: `width` columns of a [M][pitch] byte matrix starting at
// base, box 128 columns x `band` rows, 128-byte swizzle.
mxq_status encode_mx_qrow_map(CUtensorMap* map, uint8_t* base, int64_t M, int64_t width,
                              int64_t pitch, int band) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(mxq::MX_TILE_K), static_cast<cuuint32_t>(band)};
  return encode_map(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B);
}

// NVFP4 code maps: rowwise [M][K/2] seen as [m % 8][m / 8][k / 2] and
// transposed [K][M/2] seen as [k % 8][k / 8][m / 2]; boxes of one tile's
// codes (64 bytes x 16 x 8) with the 64-byte swizzle.
mxq_status encode_nv_code_maps(mxq::NvMaps* maps, uint32_t flags, int64_t M, int64_t K,
                               uint8_t* q_row, uint8_t* q_t) {
  if (flags & MXQ_ROWWISE) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(M / 8), 8};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(4 * K), static_cast<cuuint64_t>(K / 2)};
    const cuuint32_t box[3] = {mxq::NV_TILE_COLS / 2, mxq::NV_TILE_ROWS / 8, 8};
    mxq_status st = encode_map(&maps->q_row, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, q_row, dims,
                               strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
    if (st != MXQ_OK) return st;
  }
  if (flags & MXQ_COLWISE) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(M / 2), static_cast<cuuint64_t>(K / 8), 8};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(4 * M), static_cast<cuuint64_t>(M / 2)};
    const cuuint32_t box[3] = {mxq::NV_TILE_ROWS / 2, mxq::NV_TILE_COLS / 8, 8};
    mxq_status st = encode_map(&maps->q_t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, q_t, dims, strides,
                               box, CU_TENSOR_MAP_SWIZZLE_64B);
    if (st != MXQ_OK) return st;
  }
  return MXQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

mxq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MXQ_OK : MXQ_ECUDA; }

// Shared checks of the MXFP8 entry points; `width` is the quantized width.
mxq_status check_mx_outputs(uint32_t flags, int64_t width, const uint8_t* q_row,
                            const uint8_t* s_row, const uint8_t* q_col, const uint8_t* s_col) {
  (void)width;
  if ((flags & MXQ_ROWWISE) && (!q_row || !s_row)) return MXQ_EINVAL;
  if ((flags & MXQ_COLWISE) && (!q_col || !s_col)) return MXQ_EINVAL;
  if ((flags & MXQ_ROWWISE) && (!aligned(q_row, 16) || !aligned(s_row, 16))) return MXQ_EALIGN;
  if ((flags & MXQ_COLWISE) && (!aligned(q_col, 16) || !aligned(s_col, 16))) return MXQ_EALIGN;
  return MXQ_OK;
}

// The MXFP8 kernels built for the call's scale layout.
cudaError_t launch_mx_for(const mxq::MxMaps& maps, const mxq::MxArgs& a, int mode, bool dbias,
                          int act, int num_sms, cudaStream_t stream) {
  return a.scale_tiled ? mxq::launch_mx_tiled(maps, a, mode, dbias, act, num_sms, stream)
                       : mxq::launch_mx(maps, a, mode, dbias, act, num_sms, stream);
}

int direction_mode(uint32_t flags) {
  return ((flags & MXQ_ROWWISE) ? mxq::MX_ROW : 0) | ((flags & MXQ_COLWISE) ? mxq::MX_COL : 0);
}

}  // namespace

namespace mxq {

// mx_quantize_rowcol, with the colwise scale row pitch as a parameter.
mxq_status rowcol_panel(const void* x, int64_t M, int64_t K, int64_t ldx, uint32_t flags,
                        uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                        int64_t scol_ld, float* dbias, void* workspace, size_t workspace_bytes,
                        uint32_t* dev_err, cudaStream_t stream) {
  const uint32_t known = MXQ_ROWWISE | MXQ_COLWISE | MXQ_DBIAS | MXQ_ACT_GELU_TANH |
                         MXQ_SCALE_RCEIL | MXQ_SCALE_SWIZZLED;
  if (flags & ~known) return MXQ_EINVAL;
  if (!(flags & (MXQ_ROWWISE | MXQ_COLWISE))) return MXQ_EINVAL;
  if ((flags & MXQ_DBIAS) && (flags & MXQ_ACT_GELU_TANH)) return MXQ_EINVAL;
  if (M < 0 || K < 0 || ldx < K) return MXQ_ESHAPE;
  if ((M % 32) || (K % 32)) return MXQ_ESHAPE;
  if (M > (int64_t(1) << 30) || K > (int64_t(1) << 30) || M * K > (int64_t(1) << 40))
    return MXQ_ESHAPE;
  const bool want_dbias = (flags & MXQ_DBIAS) != 0;
  if (want_dbias && !dbias) return MXQ_EINVAL;
  if (want_dbias && !aligned(dbias, 16)) return MXQ_EALIGN;
  int sms = 0;
  mxq_status st = current_device(&sms);
  if (st != MXQ_OK) return st;
  if (M == 0 || K == 0) {
    if (want_dbias && K > 0)
      return from_cuda(cudaMemsetAsync(dbias, 0, static_cast<size_t>(K) * sizeof(float), stream));
    return MXQ_OK;
  }
  if (!x) return MXQ_EINVAL;
  if (!aligned(x, 16) || (ldx % 8)) return MXQ_EALIGN;
  st = check_mx_outputs(flags, K, q_row, s_row, q_col, s_col);
  if (st != MXQ_OK) return st;

  const int act = (flags & MXQ_ACT_GELU_TANH) ? mxq::ACT_GELU : mxq::ACT_NONE;
  const int band = mxq::mx_band_rows(act);
  mxq::MxArgs a{};
  a.scale_ceil = (flags & MXQ_SCALE_RCEIL) != 0;
  a.scale_tiled = (flags & MXQ_SCALE_SWIZZLED) != 0;
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.tiles_m = static_cast<int>((M + band - 1) / band);
  a.kin = static_cast<int>(K);
  a.tiles_k = static_cast<int>((K + mxq::MX_TILE_K - 1) / mxq::MX_TILE_K);
  a.q_row = q_row;
  a.s_row = s_row;
  a.q_col = q_col;
  a.s_col = s_col;
  a.scol_ld = scol_ld;
  a.dev_err = dev_err;
  a.timeout_ns = DEFAULT_TIMEOUT_NS;
  if (want_dbias) {
    const size_t need = static_cast<size_t>(a.tiles_m) * static_cast<size_t>(K) * sizeof(float);
    if (!workspace || workspace_bytes < need) return MXQ_EWORKSPACE;
    if (!aligned(workspace, 16)) return MXQ_EALIGN;
    a.dbias_ws = static_cast<float*>(workspace);
  }
  mxq::MxMaps maps{};
  st = encode_bf16_map(&maps.x, x, M, K, ldx, mxq::MX_TILE_K, mxq::mx_load_rows(act, want_dbias));
  if (st != MXQ_OK) return st;
  maps.x2 = maps.x;
  if (flags & MXQ_COLWISE) {
    st = encode_mx_qcol_map(&maps.q_col, M, K, q_col);
    if (st != MXQ_OK) return st;
  }
  maps.q_col2 = maps.q_col;
  if (flags & MXQ_ROWWISE) {
    st = encode_mx_qrow_map(&maps.q_row, q_row, M, K, K, band);
    if (st != MXQ_OK) return st;
  }
  maps.q_row2 = maps.q_row;
  st = from_cuda(launch_mx_for(maps, a, direction_mode(flags), want_dbias, act, sms, stream));
  if (st != MXQ_OK || !want_dbias) return st;
  return from_cuda(mxq::launch_dbias_finalize(a.dbias_ws, a.tiles_m, a.K, dbias, stream));
}
}  // namespace mxq

extern "C" {

const char* mxq_status_string(int status) {
  switch (status) {
    case MXQ_OK: return "MXQ_OK";
    case MXQ_EINVAL: return "MXQ_EINVAL: null pointer or bad flags";
    case MXQ_ESHAPE: return "MXQ_ESHAPE: bad matrix shape";
    case MXQ_EALIGN: return "MXQ_EALIGN: misaligned pointer or stride";
    case MXQ_EARCH: return "MXQ_EARCH: device is not sm_103";
    case MXQ_EWORKSPACE: return "MXQ_EWORKSPACE: workspace missing or too small";
    case MXQ_ECUDA: return "MXQ_ECUDA: CUDA error";
    default: return "unknown mxq status";
  }
}

size_t mxq_workspace_bytes(int op, int64_t M, int64_t K, uint32_t flags) {
  if (M <= 0 || K <= 0) return 0;
  if (op == MXQ_OP_NVFP4) return 16;   // one fp32 amax, padded
  if (op == MXQ_OP_ROWCOL_HOST) return mxq::host_workspace_bytes(M, K);
  if ((op != MXQ_OP_ROWCOL && op != MXQ_OP_DACT) || !(flags & MXQ_DBIAS)) return 0;
  const int64_t band = mxq::mx_band_rows(op == MXQ_OP_DACT ? mxq::ACT_DGELU : mxq::ACT_NONE);
  const int64_t bands = (M + band - 1) / band;
  return static_cast<size_t>(bands) * static_cast<size_t>(K) * sizeof(float);
}

mxq_status mx_quantize_rowcol(const void* x, int64_t M, int64_t K, int64_t ldx, uint32_t flags,
                              uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                              float* dbias, void* workspace, size_t workspace_bytes,
                              uint32_t* dev_err, mxq_stream_t stream) {
  return mxq::rowcol_panel(x, M, K, ldx, flags, q_row, s_row, q_col, s_col, M / 32, dbias,
                           workspace, workspace_bytes, dev_err, stream);
}


mxq_status mx_quantize_gated(const void* x, int64_t M, int64_t N, int64_t ldx, uint32_t flags,
                             uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                             uint32_t* dev_err, mxq_stream_t stream) {
  if (flags & ~static_cast<uint32_t>(MXQ_ROWWISE | MXQ_COLWISE | MXQ_ACT_GELU_TANH | MXQ_ACT_SILU |
                                     MXQ_SCALE_RCEIL | MXQ_SCALE_SWIZZLED))
    return MXQ_EINVAL;
  if (!(flags & (MXQ_ROWWISE | MXQ_COLWISE))) return MXQ_EINVAL;
  if ((flags & MXQ_ACT_GELU_TANH) && (flags & MXQ_ACT_SILU)) return MXQ_EINVAL;
  if (M < 0 || N < 0 || ldx < 2 * N) return MXQ_ESHAPE;
  if ((M % 32) || (N % 32)) return MXQ_ESHAPE;
  if (M > (int64_t(1) << 30) || N > (int64_t(1) << 29) || M * N > (int64_t(1) << 40))
    return MXQ_ESHAPE;
  int sms = 0;
  mxq_status st = current_device(&sms);
  if (st != MXQ_OK) return st;
  if (M == 0 || N == 0) return MXQ_OK;
  if (!x) return MXQ_EINVAL;
  if (!aligned(x, 16) || (ldx % 8)) return MXQ_EALIGN;
  st = check_mx_outputs(flags, N, q_row, s_row, q_col, s_col);
  if (st != MXQ_OK) return st;

  const int act = (flags & MXQ_ACT_GELU_TANH) ? mxq::ACT_GEGLU : mxq::ACT_SWIGLU;
  const int band = mxq::mx_band_rows(act);
  mxq::MxArgs a{};
  a.scale_ceil = (flags & MXQ_SCALE_RCEIL) != 0;
  a.scale_tiled = (flags & MXQ_SCALE_SWIZZLED) != 0;
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(N);
  a.kin = static_cast<int>(N);
  a.tiles_m = static_cast<int>((M + band - 1) / band);
  a.tiles_k = static_cast<int>((N + mxq::MX_TILE_K - 1) / mxq::MX_TILE_K);
  a.up_col = static_cast<int>(N);
  a.q_row = q_row;
  a.s_row = s_row;
  a.q_col = q_col;
  a.s_col = s_col;
  a.scol_ld = M / 32;
  a.dev_err = dev_err;
  a.timeout_ns = DEFAULT_TIMEOUT_NS;
  mxq::MxMaps maps{};
  // The input map spans [gate | up]; gate boxes start at column k, up boxes
  // at N + k.
  st = encode_bf16_map(&maps.x, x, M, 2 * N, ldx, mxq::MX_TILE_K, band);
  if (st != MXQ_OK) return st;
  maps.x2 = maps.x;
  if (flags & MXQ_COLWISE) {
    st = encode_mx_qcol_map(&maps.q_col, M, N, q_col);
    if (st != MXQ_OK) return st;
  }
  maps.q_col2 = maps.q_col;
  if (flags & MXQ_ROWWISE) {
    st = encode_mx_qrow_map(&maps.q_row, q_row, M, N, N, band);
    if (st != MXQ_OK) return st;
  }
  maps.q_row2 = maps.q_row;
  return from_cuda(launch_mx_for(maps, a, direction_mode(flags), false, act, sms, stream));
}

mxq_status mx_quantize_dact(const void* grad, const void* x, int64_t M, int64_t K, int64_t ldg,
                            int64_t ldx, uint32_t flags, uint8_t* q_row, uint8_t* s_row,
                            uint8_t* q_col, uint8_t* s_col, float* dbias, void* workspace,
                            size_t workspace_bytes, uint32_t* dev_err, mxq_stream_t stream) {
  const uint32_t known =
      MXQ_ROWWISE | MXQ_COLWISE | MXQ_DBIAS | MXQ_ACT_GELU_TANH | MXQ_ACT_SILU | MXQ_SCALE_RCEIL |
      MXQ_SCALE_SWIZZLED;
  if (flags & ~known) return MXQ_EINVAL;
  if (!(flags & (MXQ_ROWWISE | MXQ_COLWISE))) return MXQ_EINVAL;
  const bool gelu = (flags & MXQ_ACT_GELU_TANH) != 0, silu = (flags & MXQ_ACT_SILU) != 0;
  if (gelu == silu) return MXQ_EINVAL;   // exactly one activation
  if (M < 0 || K < 0 || ldg < K || ldx < K) return MXQ_ESHAPE;
  if ((M % 32) || (K % 32)) return MXQ_ESHAPE;
  if (M > (int64_t(1) << 30) || K > (int64_t(1) << 30) || M * K > (int64_t(1) << 40))
    return MXQ_ESHAPE;
  const bool want_dbias = (flags & MXQ_DBIAS) != 0;
  if (want_dbias && !dbias) return MXQ_EINVAL;
  if (want_dbias && !aligned(dbias, 16)) return MXQ_EALIGN;
  int sms = 0;
  mxq_status st = current_device(&sms);
  if (st != MXQ_OK) return st;
  if (M == 0 || K == 0) {
    if (want_dbias && K > 0)
      return from_cuda(cudaMemsetAsync(dbias, 0, static_cast<size_t>(K) * sizeof(float), stream));
    return MXQ_OK;
  }
  if (!grad || !x) return MXQ_EINVAL;
  if (!aligned(grad, 16) || !aligned(x, 16) || (ldg % 8) || (ldx % 8)) return MXQ_EALIGN;
  st = check_mx_outputs(flags, K, q_row, s_row, q_col, s_col);
  if (st != MXQ_OK) return st;

  const int act = gelu ? mxq::ACT_DGELU : mxq::ACT_DSILU;
  const int band = mxq::mx_band_rows(act);
  mxq::MxArgs a{};
  a.scale_ceil = (flags & MXQ_SCALE_RCEIL) != 0;
  a.scale_tiled = (flags & MXQ_SCALE_SWIZZLED) != 0;
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.kin = static_cast<int>(K);
  a.tiles_m = static_cast<int>((M + band - 1) / band);
  a.tiles_k = static_cast<int>((K + mxq::MX_TILE_K - 1) / mxq::MX_TILE_K);
  a.q_row = q_row;
  a.s_row = s_row;
  a.q_col = q_col;
  a.s_col = s_col;
  a.scol_ld = M / 32;
  a.dev_err = dev_err;
  a.timeout_ns = DEFAULT_TIMEOUT_NS;
  if (want_dbias) {
    const size_t need = static_cast<size_t>(a.tiles_m) * static_cast<size_t>(K) * sizeof(float);
    if (!workspace || workspace_bytes < need) return MXQ_EWORKSPACE;
    if (!aligned(workspace, 16)) return MXQ_EALIGN;
    a.dbias_ws = static_cast<float*>(workspace);
  }
  mxq::MxMaps maps{};
  st = encode_bf16_map(&maps.x, grad, M, K, ldg, mxq::MX_TILE_K, band);
  if (st != MXQ_OK) return st;
  st = encode_bf16_map(&maps.x2, x, M, K, ldx, mxq::MX_TILE_K, band);
  if (st != MXQ_OK) return st;
  if (flags & MXQ_COLWISE) {
    st = encode_mx_qcol_map(&maps.q_col, M, K, q_col);
    if (st != MXQ_OK) return st;
  }
  maps.q_col2 = maps.q_col;
  if (flags & MXQ_ROWWISE) {
    st = encode_mx_qrow_map(&maps.q_row, q_row, M, K, K, band);
    if (st != MXQ_OK) return st;
  }
  maps.q_row2 = maps.q_row;
  st = from_cuda(launch_mx_for(maps, a, direction_mode(flags), want_dbias, act, sms, stream));
  if (st != MXQ_OK || !want_dbias) return st;
  return from_cuda(mxq::launch_dbias_finalize(a.dbias_ws, a.tiles_m, a.K, dbias, stream));
}

mxq_status mx_quantize_dgated(const void* grad, const void* x, int64_t M, int64_t N, int64_t ldg,
                              int64_t ldx, uint32_t flags, uint8_t* q_row, uint8_t* s_row,
                              uint8_t* q_col, uint8_t* s_col, uint32_t* dev_err,
                              mxq_stream_t stream) {
  if (flags & ~static_cast<uint32_t>(MXQ_ROWWISE | MXQ_COLWISE | MXQ_ACT_GELU_TANH | MXQ_ACT_SILU |
                                     MXQ_SCALE_RCEIL | MXQ_SCALE_SWIZZLED))
    return MXQ_EINVAL;
  if (!(flags & (MXQ_ROWWISE | MXQ_COLWISE))) return MXQ_EINVAL;
  if ((flags & MXQ_ACT_GELU_TANH) && (flags & MXQ_ACT_SILU)) return MXQ_EINVAL;
  if (M < 0 || N < 0 || ldg < N || ldx < 2 * N) return MXQ_ESHAPE;
  if ((M % 32) || (N % 32)) return MXQ_ESHAPE;
  // Tiled scales: the d-up half must start on a 128-column tile boundary.
  if ((flags & MXQ_SCALE_SWIZZLED) && (N % 128)) return MXQ_ESHAPE;
  if (M > (int64_t(1) << 30) || N > (int64_t(1) << 29) || M * N > (int64_t(1) << 39))
    return MXQ_ESHAPE;
  int sms = 0;
  mxq_status st = current_device(&sms);
  if (st != MXQ_OK) return st;
  if (M == 0 || N == 0) return MXQ_OK;
  if (!grad || !x) return MXQ_EINVAL;
  if (!aligned(grad, 16) || !aligned(x, 16) || (ldg % 8) || (ldx % 8)) return MXQ_EALIGN;
  st = check_mx_outputs(flags, 2 * N, q_row, s_row, q_col, s_col);
  if (st != MXQ_OK) return st;

  const int act = (flags & MXQ_ACT_GELU_TANH) ? mxq::ACT_DGEGLU : mxq::ACT_DSWIGLU;
  const int band = mxq::mx_band_rows(act);
  mxq::MxArgs a{};
  a.scale_ceil = (flags & MXQ_SCALE_RCEIL) != 0;
  a.scale_tiled = (flags & MXQ_SCALE_SWIZZLED) != 0;
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(2 * N);       // output width
  a.kin = static_cast<int>(N);
  a.out_half = static_cast<int>(N);    // d up starts at output column N
  a.tiles_m = static_cast<int>((M + band - 1) / band);
  a.tiles_k = static_cast<int>((N + mxq::MX_TILE_K - 1) / mxq::MX_TILE_K);
  a.up_col = 0;                        // gate: columns 0.. of x
  a.up_col2 = static_cast<int>(N);     // up: columns N.. of x
  a.q_row = q_row;
  a.s_row = s_row;
  a.q_col = q_col;
  a.s_col = s_col;
  a.scol_ld = M / 32;
  a.dev_err = dev_err;
  a.timeout_ns = DEFAULT_TIMEOUT_NS;
  mxq::MxMaps maps{};
  st = encode_bf16_map(&maps.x, grad, M, N, ldg, mxq::MX_TILE_K, band);
  if (st != MXQ_OK) return st;
  st = encode_bf16_map(&maps.x2, x, M, 2 * N, ldx, mxq::MX_TILE_K, band);
  if (st != MXQ_OK) return st;
  if (flags & MXQ_COLWISE) {
    // One map per output tile, each clipped at its N code rows, so a ragged
    // last tile of d gate cannot spill into the rows of d up.
    st = encode_mx_qcol_map(&maps.q_col, M, N, q_col);
    if (st != MXQ_OK) return st;
    st = encode_mx_qcol_map(&maps.q_col2, M, N, q_col + static_cast<size_t>(N) * M);
    if (st != MXQ_OK) return st;
  }
  if (flags & MXQ_ROWWISE) {
    // Likewise for the rowwise codes: columns [0, N) and [N, 2N) of [M][2N].
    st = encode_mx_qrow_map(&maps.q_row, q_row, M, N, 2 * N, band);
    if (st != MXQ_OK) return st;
    st = encode_mx_qrow_map(&maps.q_row2, q_row + N, M, N, 2 * N, band);
    if (st != MXQ_OK) return st;
  }
  return from_cuda(launch_mx_for(maps, a, direction_mode(flags), false, act, sms, stream));
}

mxq_status bf16_amax(const void* x, int64_t M, int64_t K, int64_t ldx, float* amax_out,
                     mxq_stream_t stream) {
  if (!amax_out) return MXQ_EINVAL;
  if (M < 0 || K < 0 || ldx < K) return MXQ_ESHAPE;
  if (K % 8) return MXQ_ESHAPE;
  if (!aligned(amax_out, 4)) return MXQ_EALIGN;
  int sms = 0;
  mxq_status st = current_device(&sms);
  if (st != MXQ_OK) return st;
  if (M > 0 && K > 0) {
    if (!x) return MXQ_EINVAL;
    if (!aligned(x, 16) || (ldx % 8)) return MXQ_EALIGN;
  }
  return from_cuda(mxq::launch_bf16_amax(x, M, K, ldx, amax_out, sms, stream));
}

mxq_status nvfp4_quantize_transpose(const void* x, int64_t M, int64_t K, int64_t ldx,
                                    uint32_t flags, const float* amax_in, float* global_scale,
                                    uint8_t* q_row, uint8_t* s_row, uint8_t* q_t, uint8_t* s_t,
                                    void* workspace, size_t workspace_bytes, uint32_t* dev_err,
                                    mxq_stream_t stream) {
  if (flags & ~static_cast<uint32_t>(MXQ_ROWWISE | MXQ_COLWISE | MXQ_NVFP4_2D)) return MXQ_EINVAL;
  if (!(flags & (MXQ_ROWWISE | MXQ_COLWISE))) return MXQ_EINVAL;
  if (M < 0 || K < 0 || ldx < K) return MXQ_ESHAPE;
  if ((M % 32) || (K % 32)) return MXQ_ESHAPE;
  if (M > (int64_t(1) << 30) || K > (int64_t(1) << 30) || M * K > (int64_t(1) << 40))
    return MXQ_ESHAPE;
  if (!global_scale) return MXQ_EINVAL;
  if (!aligned(global_scale, 4)) return MXQ_EALIGN;
  int sms = 0;
  mxq_status st = current_device(&sms);
  if (st != MXQ_OK) return st;
  if (M == 0 || K == 0) {
    // Nothing to quantize; G = amax / 2688 from the caller's amax, else 0.
    if (!amax_in) return from_cuda(cudaMemsetAsync(global_scale, 0, sizeof(float), stream));
    return from_cuda(mxq::launch_nv_global_scale(amax_in, global_scale, stream));
  }
  const float* amax = amax_in;
  if (!amax) {
    if (!workspace || workspace_bytes < sizeof(float)) return MXQ_EWORKSPACE;
    if (!aligned(workspace, 16)) return MXQ_EALIGN;
  }
  if (!x) return MXQ_EINVAL;
  if (!aligned(x, 16) || (ldx % 8)) return MXQ_EALIGN;
  if ((flags & MXQ_ROWWISE) && (!q_row || !s_row)) return MXQ_EINVAL;
  if ((flags & MXQ_COLWISE) && (!q_t || !s_t)) return MXQ_EINVAL;
  if ((flags & MXQ_ROWWISE) && (!aligned(q_row, 16) || !aligned(s_row, 16))) return MXQ_EALIGN;
  if ((flags & MXQ_COLWISE) && (!aligned(q_t, 16) || !aligned(s_t, 16))) return MXQ_EALIGN;

  if (!amax) {
    float* ws_amax = static_cast<float*>(workspace);
    st = from_cuda(mxq::launch_bf16_amax(x, M, K, ldx, ws_amax, sms, stream));
    if (st != MXQ_OK) return st;
    amax = ws_amax;
  }
  const bool two_d = (flags & MXQ_NVFP4_2D) != 0;
  mxq::NvArgs a{};
  a.M = static_cast<int>(M);
  a.K = static_cast<int>(K);
  a.tiles_m = static_cast<int>((M + mxq::NV_TILE_ROWS - 1) / mxq::NV_TILE_ROWS);
  a.tiles_k = static_cast<int>((K + mxq::NV_TILE_COLS - 1) / mxq::NV_TILE_COLS);
  a.amax = amax;
  a.global_scale = global_scale;
  a.q_row = q_row;
  a.s_row = s_row;
  a.q_t = q_t;
  a.s_t = s_t;
  a.dev_err = dev_err;
  a.timeout_ns = DEFAULT_TIMEOUT_NS;
  mxq::NvMaps maps{};
  const int mode = direction_mode(flags);
  st = encode_bf16_map(&maps.x, x, M, K, ldx, mxq::nv_load_cols(), mxq::NV_TILE_ROWS);
  if (st != MXQ_OK) return st;
  st = encode_nv_code_maps(&maps, flags, M, K, q_row, q_t);
  if (st != MXQ_OK) return st;
  return from_cuda(mxq::launch_nvfp4(maps, a, mode, two_d, amax_in == nullptr, stream));
}

mxq_status mxq_selftest_bounded_wait(uint64_t timeout_ns, uint32_t* dev_err, mxq_stream_t stream) {
  if (!dev_err) return MXQ_EINVAL;
  if (timeout_ns < 1000ull || timeout_ns > 5000000000ull) return MXQ_EINVAL;
  int sms = 0;
  mxq_status st = current_device(&sms);
  if (st != MXQ_OK) return st;
  return from_cuda(mxq::launch_selftest_wait(timeout_ns, dev_err, stream));
}

}  // extern "C"
