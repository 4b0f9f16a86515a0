// mx_kernels.cu -- MXFP8 quantization kernels for sm_103a.
//
// One kernel template covers the MXFP8 paths of TE PR #3291 "Fix pointer
// arithmatic to generate correct LDS/STS instructions" (results tables
// "MXFP8 generic quantize kernel": plain / dbias / gelu; "MXFP8 specialized
// cast-only kernel (bidimensional)": plain row / both; "MXFP8 gated (swiglu /
// geglu) kernel": swiglu) and the colwise "dim1" cast of torchao PR #12
// "Multiply with inverse scale in loop instead of dividing".
//
// Design (HBM-bound; no tensor-core work on this path):
//  * Every warp runs its own TMA pipeline: STAGES shared-memory slots, one
//    mbarrier each; lane 0 issues a 2-D TMA box of 32 rows x 128 columns
//    (8 KiB of bf16) per slot.  Warps never wait on each other.
//  * The grid is persistent (one CTA per SM); warp g takes tiles
//    g, g + W, g + 2W, ... (W = warps in the grid), or, with dbias, a fixed
//    column strip and every P-th row tile so its column sums stay in
//    registers.
//  * Lane (h, c) = (lane / 16, lane % 16) owns rows 16h..16h+15 and
//    columns 8c..8c+7 of the tile: 16 conflict-free 16-byte shared loads
//    (each quarter warp reads one contiguous 128-byte row segment).
//    Colwise 32x1 amax: in-thread over 16 rows + one xor-16 shuffle.
//    Rowwise 1x32 amax: in-thread over 8 columns + xor-1 / xor-2 shuffles,
//    two rows packed per 32-bit register.
//  * The shared scale is read off the exponent field of the amax and the
//    elements are multiplied by the exact power of two 2^-e (one multiply
//    per element, no division; torchao PR #12, rationale), then converted
//    two at a time by cvt.rn.satfinite.e4m3x2.f32.
//  * Stores: rowwise codes 8 bytes per lane per row (a half warp writes one
//    contiguous 128-byte row segment); colwise codes 16 bytes per lane per
//    column (lanes h = 0, 1 fill one 32-byte sector of the [K][M] output).

#include "mxq_internal.h"
#include "mxq_ptx.cuh"

namespace mxq {
namespace {

// ---------------------------------------------------------------------------
// Activations (fp32, no intermediate bf16 rounding)
// ---------------------------------------------------------------------------

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh-form GELU, 0.5 x (1 + tanh(u)) with u = sqrt(2/pi) (x + 0.044715 x^3),
// evaluated through the identity 0.5 (1 + tanh(u)) = 1 / (1 + e^(-2u)) and
// e^z = 2^(z log2 e).  A few fp32 ulps from the exact value.
__device__ __forceinline__ float gelu_tanh_f32(float x) {
  constexpr float kNeg2SqrtTwoOverPiLog2e = -2.0f * 0.7978845608028654f * 1.4426950408889634f;
  const float inner = x * fmaf(0.044715f, x * x, 1.0f);
  const float e = ex2_approx(kNeg2SqrtTwoOverPiLog2e * inner);
  return x * rcp_approx(1.0f + e);
}

// silu(g) * u with silu(g) = g / (1 + e^-g).
__device__ __forceinline__ float swiglu_f32(float g, float u) {
  constexpr float kNegLog2e = -1.4426950408889634f;
  const float e = ex2_approx(kNegLog2e * g);
  return g * rcp_approx(1.0f + e) * u;
}

// ---------------------------------------------------------------------------
// Tile schedule
// ---------------------------------------------------------------------------

struct Schedule {
  int count;      // tiles this warp processes
  int first;      // plain: first linear tile; dbias: first row tile
  int step;       // plain: warps in the grid; dbias: row groups
  int strip;      // dbias: fixed column tile; -1 for the plain schedule
  int tiles_k;

  __device__ void coords(int j, int& tm, int& tk) const {
    if (strip >= 0) {
      tm = first + j * step;
      tk = strip;
    } else {
      const int t = first + j * step;
      tm = t / tiles_k;
      tk = t - tm * tiles_k;
    }
  }
};

__device__ __forceinline__ Schedule make_schedule(const MxArgs& a, int gw, int warps_in_grid,
                                                  bool dbias) {
  Schedule s;
  s.tiles_k = a.tiles_k;
  if (dbias) {
    const int P = a.dbias_groups;
    const int p = gw / a.tiles_k;
    s.strip = gw - p * a.tiles_k;
    s.first = p;
    s.step = P;
    s.count = (p < P && p < a.tiles_m) ? (a.tiles_m - p + P - 1) / P : 0;
  } else {
    const int total = a.tiles_m * a.tiles_k;
    s.strip = -1;
    s.first = gw;
    s.step = warps_in_grid;
    s.count = gw < total ? (total - gw + warps_in_grid - 1) / warps_in_grid : 0;
  }
  return s;
}

// ---------------------------------------------------------------------------
// Shared per-tile arithmetic
// ---------------------------------------------------------------------------

// Packed exponents (two 16-bit lanes) -> two E8M0 codes (two 16-bit lanes).
__device__ __forceinline__ uint32_t e8m0_pair(uint32_t e2) {
  // max(E, 8) - 8 on both halves; no borrow crosses halves because each
  // half is >= 8 after the max.
  return vmax_u16x2(e2, 0x00080008u) - 0x00080008u;
}

template <int WARPS, int STAGES, int STAGE_BYTES>
struct MxSmemLayout {
  static constexpr int kStageBytes = STAGE_BYTES;
  static constexpr int kDynamicBytes = WARPS * STAGES * STAGE_BYTES + 128;  // + alignment pad
};

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

template <int MODE, bool DBIAS, int ACT, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32, 1)
mx_quantize_kernel(const __grid_constant__ CUtensorMap tmap, const MxArgs a) {
  constexpr bool ROW = (MODE & MX_ROW) != 0;
  constexpr bool COL = (MODE & MX_COL) != 0;
  constexpr int OPERANDS = (ACT == ACT_SWIGLU) ? 2 : 1;
  constexpr int TILE_BYTES = MX_TILE_M * MX_TILE_K * 2;
  constexpr int STAGE_BYTES = TILE_BYTES * OPERANDS;
  constexpr int ROW_PITCH = MX_TILE_K * 2;   // bytes per tile row in shared memory
  static_assert(!(DBIAS && ACT != ACT_NONE), "dbias is defined on the plain path only");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[WARPS][STAGES];
  __shared__ __align__(16) uint32_t row_scale_stage[WARPS][32];

  uint8_t* smem = align_up_shared<128>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = lane >> 4;     // which 16-row half of the tile
  const int c = lane & 15;     // which 8-column chunk
  const uint32_t stage0 = smem_addr(smem) + warp * STAGES * STAGE_BYTES;
  const uint32_t bar0 = smem_addr(&bars[warp][0]);
  const uint32_t rs_stage = smem_addr(&row_scale_stage[warp][0]);

  const Schedule sched = make_schedule(a, blockIdx.x * WARPS + warp, gridDim.x * WARPS, DBIAS);
  if (sched.count == 0) return;

  if (lane == 0) {
    prefetch_tensormap(&tmap);
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_barrier_init();
  }
  __syncwarp();

  auto issue = [&](int j) {   // lane 0 only
    int tm, tk;
    sched.coords(j, tm, tk);
    const int s = j % STAGES;
    const uint32_t bar = bar0 + 8 * s;
    const uint32_t dst = stage0 + s * STAGE_BYTES;
    mbar_arrive_expect_tx(bar, STAGE_BYTES);
    tma_load_2d(dst, &tmap, tk * MX_TILE_K, tm * MX_TILE_M, bar);
    if (OPERANDS == 2) tma_load_2d(dst + TILE_BYTES, &tmap, a.up_col + tk * MX_TILE_K, tm * MX_TILE_M, bar);
  };

  if (lane == 0) {
    const int pre = sched.count < STAGES ? sched.count : STAGES;
    for (int j = 0; j < pre; ++j) issue(j);
  }

  float dsum[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) dsum[j] = 0.0f;
  int last_tk = 0;

  for (int j = 0; j < sched.count; ++j) {
    const int s = j % STAGES;
    const uint32_t parity = (j / STAGES) & 1;
    const bool ok = mbar_wait_bounded(bar0 + 8 * s, parity, a.timeout_ns);
    if (__any_sync(0xFFFFFFFFu, !ok)) {
      // A copy never landed.  Record it, let this warp's other copies in
      // flight finish (bounded), and stop without touching more output.
      if (lane == 0 && a.dev_err) atomicOr(a.dev_err, 1u);
      const int last = (j + STAGES < sched.count) ? j + STAGES : sched.count;
      for (int jj = j + 1; jj < last; ++jj)
        mbar_wait_bounded(bar0 + 8 * (jj % STAGES), (jj / STAGES) & 1, a.timeout_ns);
      return;
    }

    int tm, tk;
    sched.coords(j, tm, tk);
    last_tk = tk;
    const uint32_t tile = stage0 + s * STAGE_BYTES;
    const uint32_t my_row0 = tile + (16 * h) * ROW_PITCH + c * 16;

    // ---- load this lane's 16 x 8 block; reduce to exponent maxima -------
    // ce[p]: packed exponent maxima of columns 2p (low half), 2p+1 (high).
    // re[q]: packed exponent maxima of rows 2q (low half), 2q+1 (high).
    uint32_t ce[4], re[8];
    uint32_t xr[16][4];
    float y[(ACT == ACT_NONE) ? 1 : 16][(ACT == ACT_NONE) ? 1 : 8];

    if constexpr (ACT == ACT_NONE) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint4 v = lds128(my_row0 + i * ROW_PITCH);
        xr[i][0] = v.x; xr[i][1] = v.y; xr[i][2] = v.z; xr[i][3] = v.w;
      }
      uint32_t cm[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        uint32_t t[2];
#pragma unroll
        for (int di = 0; di < 2; ++di) {
          const uint32_t a0 = xr[i + di][0] & 0x7FFF7FFFu;
          const uint32_t a1 = xr[i + di][1] & 0x7FFF7FFFu;
          const uint32_t a2 = xr[i + di][2] & 0x7FFF7FFFu;
          const uint32_t a3 = xr[i + di][3] & 0x7FFF7FFFu;
          cm[0] = vmax_u16x2(cm[0], a0);
          cm[1] = vmax_u16x2(cm[1], a1);
          cm[2] = vmax_u16x2(cm[2], a2);
          cm[3] = vmax_u16x2(cm[3], a3);
          t[di] = vmax_u16x2(vmax_u16x2(a0, a1), vmax_u16x2(a2, a3));
        }
        // low halves = even columns, high = odd; fold to one max per row.
        const uint32_t rm = vmax_u16x2(prmt(t[0], t[1], 0x5410), prmt(t[0], t[1], 0x7632));
        re[i / 2] = (rm >> 7) & 0x00FF00FFu;      // bf16 magnitude -> exponent field
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) ce[p] = (cm[p] >> 7) & 0x00FF00FFu;
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint4 v = lds128(my_row0 + i * ROW_PITCH);
        uint32_t u[4] = {0u, 0u, 0u, 0u};
        if constexpr (ACT == ACT_SWIGLU) {
          const uint4 w = lds128(my_row0 + TILE_BYTES + i * ROW_PITCH);
          u[0] = w.x; u[1] = w.y; u[2] = w.z; u[3] = w.w;
        }
        const uint32_t g[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          if constexpr (ACT == ACT_GELU) {
            y[i][2 * p] = gelu_tanh_f32(bf16_lo(g[p]));
            y[i][2 * p + 1] = gelu_tanh_f32(bf16_hi(g[p]));
          } else {
            y[i][2 * p] = swiglu_f32(bf16_lo(g[p]), bf16_lo(u[p]));
            y[i][2 * p + 1] = swiglu_f32(bf16_hi(g[p]), bf16_hi(u[p]));
          }
        }
      }
      uint32_t cmx[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      uint32_t rmx[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        rmx[i] = 0u;
#pragma unroll
        for (int jc = 0; jc < 8; ++jc) {
          const uint32_t b = __float_as_uint(y[i][jc]) & 0x7FFFFFFFu;
          cmx[jc] = max(cmx[jc], b);
          rmx[i] = max(rmx[i], b);
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) re[q] = (rmx[2 * q] >> 23) | ((rmx[2 * q + 1] >> 23) << 16);
#pragma unroll
      for (int p = 0; p < 4; ++p) ce[p] = (cmx[2 * p] >> 23) | ((cmx[2 * p + 1] >> 23) << 16);
    }

    // ---- every value of the slot is in registers: hand it back to TMA ----
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && j + STAGES < sched.count) issue(j + STAGES);

    // ---- complete the block maxima across lanes -------------------------
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      re[q] = vmax_u16x2(re[q], __shfl_xor_sync(0xFFFFFFFFu, re[q], 1));
      re[q] = vmax_u16x2(re[q], __shfl_xor_sync(0xFFFFFFFFu, re[q], 2));
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) ce[p] = vmax_u16x2(ce[p], __shfl_xor_sync(0xFFFFFFFFu, ce[p], 16));

    const int col0 = tk * MX_TILE_K + c * 8;      // first column of this lane
    const bool col_ok = col0 < a.K;
    const int row0 = tm * MX_TILE_M + 16 * h;     // first row of this lane

    auto val = [&](int i, int jc) -> float {
      if constexpr (ACT == ACT_NONE) {
        return (jc & 1) ? bf16_hi(xr[i][jc >> 1]) : bf16_lo(xr[i][jc >> 1]);
      } else {
        return y[i][jc];
      }
    };

    // ---- rowwise: scale codes, codes, stores ----------------------------
    if constexpr (ROW) {
      uint32_t rc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) rc[q] = e8m0_pair(re[q]);
      uint8_t* qrow = a.q_row + static_cast<size_t>(row0) * a.K + col0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t code = (rc[i >> 1] >> (16 * (i & 1))) & 0xFFu;
        const float inv = inv_scale_from_e8m0(code);
        const uint32_t w0 = cvt_e4m3x4(val(i, 0) * inv, val(i, 1) * inv, val(i, 2) * inv, val(i, 3) * inv);
        const uint32_t w1 = cvt_e4m3x4(val(i, 4) * inv, val(i, 5) * inv, val(i, 6) * inv, val(i, 7) * inv);
        if (col_ok) stg64(qrow + static_cast<size_t>(i) * a.K, w0, w1);
      }
      // Scale bytes: lane (h, c) holds the codes of block c/4 for its 16
      // rows; it stages rows 4t + (c & 3) into a [32 rows][4 blocks] byte
      // array, then lane L writes row L's 4 bytes.
      const int r = c & 3, b = c >> 2;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t pair = (r >> 1) ? rc[2 * t + 1] : rc[2 * t];
        sts8(rs_stage + (16 * h + 4 * t + r) * 4 + b, (pair >> (16 * (r & 1))) & 0xFFu);
      }
      __syncwarp();
      const uint32_t w = lds32(rs_stage + lane * 4);
      const int kb0 = tk * (MX_TILE_K / 32);
      const int nkb = a.K / 32;
      const int valid = min(4, nkb - kb0);
      uint8_t* srow = a.s_row + static_cast<size_t>(tm * MX_TILE_M + lane) * nkb + kb0;
      if (valid == 4 && (nkb & 3) == 0) {
        stg32(srow, w);
      } else {
        for (int bb = 0; bb < valid; ++bb) stg8(srow + bb, (w >> (8 * bb)) & 0xFFu);
      }
    }

    // ---- colwise: scale codes, codes, stores ----------------------------
    if constexpr (COL) {
      uint32_t cc[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) cc[p] = e8m0_pair(ce[p]);
      uint8_t* qcol = a.q_col + static_cast<size_t>(col0) * a.M + row0;
#pragma unroll
      for (int jc = 0; jc < 8; ++jc) {
        const uint32_t code = (cc[jc >> 1] >> (16 * (jc & 1))) & 0xFFu;
        const float inv = inv_scale_from_e8m0(code);
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          w[q] = cvt_e4m3x4(val(4 * q, jc) * inv, val(4 * q + 1, jc) * inv,
                            val(4 * q + 2, jc) * inv, val(4 * q + 3, jc) * inv);
        if (col_ok) stg128(qcol + static_cast<size_t>(jc) * a.M, w[0], w[1], w[2], w[3]);
      }
      // Lane h = 0 writes the scale bytes of columns 0-3, h = 1 of 4-7.
      const int nmb = a.M / 32;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const uint32_t pair = h ? cc[2 + (jj >> 1)] : cc[jj >> 1];
        const uint32_t code = (pair >> (16 * (jj & 1))) & 0xFFu;
        if (col_ok)
          stg8(a.s_col + static_cast<size_t>(col0 + 4 * h + jj) * nmb + tm, code);
      }
    }

    // ---- dbias: column sums of this tile, pairwise over rows -------------
    if constexpr (DBIAS) {
#pragma unroll
      for (int jc = 0; jc < 8; ++jc) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = val(i, jc);
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) v[i] = v[i] + v[i + w];
        const float tile_sum = v[0] + __shfl_xor_sync(0xFFFFFFFFu, v[0], 16);
        dsum[jc] += tile_sum;
      }
    }
    __syncwarp();   // row_scale_stage is rewritten by the next tile
  }

  if constexpr (DBIAS) {
    // This warp's column strip is fixed; write its partial sums once.
    const int col0 = last_tk * MX_TILE_K + c * 8;
    if (h == 0 && col0 < a.K) {
      const int p = sched.first;
      float* dst = a.dbias_ws + static_cast<size_t>(p) * a.K + col0;
      stg128(dst, __float_as_uint(dsum[0]), __float_as_uint(dsum[1]),
             __float_as_uint(dsum[2]), __float_as_uint(dsum[3]));
      stg128(dst + 4, __float_as_uint(dsum[4]), __float_as_uint(dsum[5]),
             __float_as_uint(dsum[6]), __float_as_uint(dsum[7]));
    }
  }
}

// dbias[k] = sum over row groups of the partial sums, in group order.
__global__ void dbias_finalize_kernel(const float* __restrict__ ws, int groups, int K,
                                      float* __restrict__ dbias) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= K) return;
  float s = 0.0f;
  for (int p = 0; p < groups; ++p) s += ws[static_cast<size_t>(p) * K + k];
  dbias[k] = s;
}

// ---------------------------------------------------------------------------
// Launch configuration per variant
// ---------------------------------------------------------------------------

template <int ACT>
struct MxConfig {
  // 8 warps x 3 slots x 8 KiB = 192 KiB of tiles per SM.
  static constexpr int WARPS = 8;
  static constexpr int STAGES = 3;
};
template <>
struct MxConfig<ACT_SWIGLU> {
  // gate + up per slot: 6 warps x 2 slots x 16 KiB = 192 KiB per SM.
  static constexpr int WARPS = 6;
  static constexpr int STAGES = 2;
};

template <int MODE, bool DBIAS, int ACT>
cudaError_t launch_variant(const CUtensorMap& map, const MxArgs& a, int num_sms,
                           cudaStream_t stream) {
  constexpr int WARPS = MxConfig<ACT>::WARPS;
  constexpr int STAGES = MxConfig<ACT>::STAGES;
  constexpr int STAGE_BYTES = MX_TILE_M * MX_TILE_K * 2 * (ACT == ACT_SWIGLU ? 2 : 1);
  constexpr int SMEM = WARPS * STAGES * STAGE_BYTES + 128;
  auto kernel = mx_quantize_kernel<MODE, DBIAS, ACT, WARPS, STAGES>;

  static int configured_device = -1;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (configured_device != dev) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (err != cudaSuccess) return err;
    configured_device = dev;
  }

  int grid;
  if (DBIAS) {
    const int warps_needed = a.dbias_groups * a.tiles_k;
    grid = (warps_needed + WARPS - 1) / WARPS;
  } else {
    const int64_t tiles = static_cast<int64_t>(a.tiles_m) * a.tiles_k;
    const int64_t ctas_for_tiles = (tiles + WARPS - 1) / WARPS;
    grid = static_cast<int>(ctas_for_tiles < num_sms ? ctas_for_tiles : num_sms);
  }
  if (grid < 1) grid = 1;
  kernel<<<grid, WARPS * 32, SMEM, stream>>>(map, a);
  return cudaGetLastError();
}

template <bool DBIAS, int ACT>
cudaError_t launch_mode(const CUtensorMap& map, const MxArgs& a, int mode, int num_sms,
                        cudaStream_t stream) {
  switch (mode) {
    case MX_ROW: return launch_variant<MX_ROW, DBIAS, ACT>(map, a, num_sms, stream);
    case MX_COL: return launch_variant<MX_COL, DBIAS, ACT>(map, a, num_sms, stream);
    default: return launch_variant<MX_ROW | MX_COL, DBIAS, ACT>(map, a, num_sms, stream);
  }
}

}  // namespace

int mx_dbias_groups(int tiles_m, int tiles_k, int num_sms) {
  const int warp_capacity = num_sms * MxConfig<ACT_NONE>::WARPS;
  int groups = warp_capacity / tiles_k;
  if (groups < 1) groups = 1;
  if (groups > tiles_m) groups = tiles_m;
  return groups;
}

cudaError_t launch_mx(const CUtensorMap& map, const MxArgs& a, int mode, bool dbias, int act,
                      int num_sms, cudaStream_t stream) {
  if (dbias) return launch_mode<true, ACT_NONE>(map, a, mode, num_sms, stream);
  switch (act) {
    case ACT_GELU: return launch_mode<false, ACT_GELU>(map, a, mode, num_sms, stream);
    case ACT_SWIGLU: return launch_mode<false, ACT_SWIGLU>(map, a, mode, num_sms, stream);
    default: return launch_mode<false, ACT_NONE>(map, a, mode, num_sms, stream);
  }
}

cudaError_t launch_dbias_finalize(const float* ws, int groups, int K, float* dbias,
                                  cudaStream_t stream) {
  const int threads = 256;
  const int blocks = (K + threads - 1) / threads;
  dbias_finalize_kernel<<<blocks, threads, 0, stream>>>(ws, groups, K, dbias);
  return cudaGetLastError();
}

}  // namespace mxq
