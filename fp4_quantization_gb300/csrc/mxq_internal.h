// mxq_internal.h -- launch arguments and launchers shared between the kernel
// translation units and the C ABI layer (mxq_api.cu).  Not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "mxq.h"

namespace mxq {

// MXFP8: each warp quantizes 32 rows (one colwise block) x 128 columns
// (four rowwise blocks); a CTA takes a band of mx_band_rows() rows x 128
// columns per step.
constexpr int MX_TILE_M = 32;
constexpr int MX_TILE_K = 128;


constexpr uint64_t DEFAULT_TIMEOUT_NS = 1000000000ull;   // 1 s per wait

enum : int { MX_ROW = 1, MX_COL = 2 };
// Element functions of the MXFP8 kernel: the input itself, GELU, the gated
// SwiGLU / GeGLU, the backward dGELU / dSiLU (grad * act'(x)) and the gated
// backward (two outputs: d gate, d up).
enum : int {
  ACT_NONE = 0, ACT_GELU = 1, ACT_SWIGLU = 2, ACT_GEGLU = 3, ACT_DGELU = 4, ACT_DSILU = 5,
  ACT_DSWIGLU = 6, ACT_DGEGLU = 7
};

struct MxArgs {
  int M, K;                 // shape of y (the quantized matrix)
  int kin;                  // input columns per output tile (K, or N of a 2N-wide output)
  int out_half;             // output column of the second output tile (gated backward), else 0
  int tiles_m, tiles_k;     // bands of mx_band_rows() rows, 128-column steps over kin
  int up_col;               // column of the second operand in x2 (gated: N; else 0)
  int up_col2;              // column of the third operand in x2 (gated backward: N)
  int scale_ceil;           // 1: ceil-style E8M0 rule (MXQ_SCALE_RCEIL); 0: floor rule
  int scale_tiled;          // 1: scales in 128 x 4 tiles (MXQ_SCALE_SWIZZLED); 0: row-major
  uint8_t* q_row;
  uint8_t* s_row;
  uint8_t* q_col;
  uint8_t* s_col;
  int64_t scol_ld;          // bytes between rows of row-major colwise scales (M / 32, or
                            // the full matrix's when a row panel writes into it)
  float* dbias_ws;          // [tiles_m][K] column sums of each band
  uint32_t* dev_err;
  uint64_t timeout_ns;
};

// TMA descriptors of one MXFP8 call: the bf16 inputs (box 128 columns x one
// band; x2 is the second input tensor, or x again) and the colwise codes
// [K][M] viewed as the 3-D tensor [k % 8][k / 8][m] (box 128 x 16 x 8,
// 128-byte swizzle); q_col2 covers the second output tile's rows [N, 2N) of
// the gated backward (else q_col again).
struct MxMaps {
  CUtensorMap x;
  CUtensorMap x2;
  CUtensorMap q_col;
  CUtensorMap q_col2;
  // Rowwise codes [M][K] (box 128 columns x one band, 128-byte swizzle);
  // q_row2 covers the second output tile's columns [N, 2N) of the gated
  // backward, and q_row its first N columns (else q_row again).
  CUtensorMap q_row;
  CUtensorMap q_row2;
};

// NVFP4: one CTA per tile of NV_TILE_ROWS x NV_TILE_COLS.
constexpr int NV_TILE_ROWS = 128;
constexpr int NV_TILE_COLS = 128;
// Columns of one input copy of a tile (the input map's box).
int nv_load_cols();

// TMA descriptors of one NVFP4 call: the bf16 input (box nv_load_cols()
// columns x NV_TILE_ROWS rows), the
// rowwise codes [M][K/2] seen as [m % 8][m / 8][k / 2] and the transposed
// codes [K][M/2] seen as [k % 8][k / 8][m / 2] (boxes of 64 bytes x 16 x 8,
// 64-byte swizzle).
struct NvMaps {
  CUtensorMap x;
  CUtensorMap q_row;
  CUtensorMap q_t;
};

struct NvArgs {
  int M, K;
  int tiles_m, tiles_k;     // tile rows and columns of the grid
  const float* amax;        // device tensor amax
  float* global_scale;      // device, receives amax / 2688
  uint8_t* q_row;
  uint8_t* s_row;
  uint8_t* q_t;
  uint8_t* s_t;
  uint32_t* dev_err;
  uint64_t timeout_ns;
  int reverse;              // take the tiles last first
};

// Rows per band (per CTA step) of the MXFP8 kernel for activation `act`.
int mx_band_rows(int act);
// Rows of one input copy (the input map's box) of the kernel that runs
// element function `act` (with dbias or not): a band, or half a tile.
int mx_load_rows(int act, bool dbias);

cudaError_t launch_mx(const MxMaps& maps, const MxArgs& a, int mode, bool dbias, int act,
                      int num_sms, cudaStream_t stream);
// The same kernels built to write the scales in 128 x 4 tiles (a.scale_tiled).
cudaError_t launch_mx_tiled(const MxMaps& maps, const MxArgs& a, int mode, bool dbias, int act,
                            int num_sms, cudaStream_t stream);
cudaError_t launch_dbias_finalize(const float* ws, int bands, int K, float* dbias,
                                  cudaStream_t stream);
// after_amax: launched right after this call's own bf16_amax grid (as its
// programmatic dependent).
cudaError_t launch_nvfp4(const NvMaps& maps, const NvArgs& a, int mode, bool two_d,
                         bool after_amax, cudaStream_t stream);
cudaError_t launch_bf16_amax(const void* x, int64_t M, int64_t K, int64_t ldx, float* out,
                             int num_sms, cudaStream_t stream);
cudaError_t launch_nv_global_scale(const float* amax, float* global_scale, cudaStream_t stream);
// Device workspace of mx_quantize_rowcol_host (two sets of panel buffers and
// the colwise scales of the whole matrix).
size_t host_workspace_bytes(int64_t M, int64_t K);
// mx_quantize_rowcol with the row-major colwise scales written scol_ld bytes
// apart (a row panel of a wider matrix; scol_ld >= M / 32).
mxq_status rowcol_panel(const void* x, int64_t M, int64_t K, int64_t ldx, uint32_t flags,
                        uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                        int64_t scol_ld, float* dbias, void* workspace, size_t workspace_bytes,
                        uint32_t* dev_err, cudaStream_t stream);
cudaError_t launch_selftest_wait(uint64_t timeout_ns, uint32_t* dev_err, cudaStream_t stream);

}  // namespace mxq
