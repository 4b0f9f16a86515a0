// nvfp4_kernels.cu -- NVFP4 quantize-transpose, the tensor amax it needs,
// and the bounded-wait self test, for sm_103a.
//
// NVFP4 quantize-transpose is the "NVFP4 quantize-transpose" kernel family
// of TE PR #3291 "Fix pointer arithmatic to generate correct LDS/STS
// instructions" (results table "NVFP4 2D quantize-transpose kernel" and the
// 1D kernel named in its "Patched but not measurable" section); this file
// implements the 1D (1x16 block) variant.
//
// Same pipeline shape as the MXFP8 kernels: one TMA ring per warp, 64 x 64
// bf16 tiles (8 KiB).  Lane (h, c) = (lane / 8, lane % 8) owns rows
// 16h..16h+15 and columns 8c..8c+7, so each transposed 16x1 block lies
// entirely in one lane and each 1x16 row block in a lane pair.  Per block the
// scale arithmetic runs in IEEE fp32 with explicit rounding intrinsics in
// the fixed order (b / 6) / G -> E4M3 -> value * G -> 1 / d; each element
// then takes one multiply by that reciprocal (no per-element division, as
// in torchao PR #12 "Multiply with inverse scale in loop instead of
// dividing", rationale) and cvt.rn.satfinite.e2m1x2.f32.

#include <cfloat>

#include "mxq_internal.h"
#include "mxq_ptx.cuh"

namespace mxq {
namespace {

constexpr int NV_WARPS = 8;
constexpr int NV_STAGES = 3;

struct NvSchedule {
  int count, first, step, tiles_k;
  __device__ void coords(int j, int& tm, int& tk) const {
    const int t = first + j * step;
    tm = t / tiles_k;
    tk = t - tm * tiles_k;
  }
};

// Block scale of one NVFP4 block from its amax b (exact fp32).
__device__ __forceinline__ void nv_block_scale(float b, float G, uint32_t& code, float& inv) {
  code = 0u;
  inv = 0.0f;
  if (G == 0.0f) return;
  const float sf = __fdiv_rn(__fdiv_rn(b, 6.0f), G);
  code = cvt_e4m3x2(sf, 0.0f) & 0xFFu;
  const float d = __fmul_rn(e4m3_to_f32(code), G);
  if (code != 0u && d != 0.0f) {
    inv = __frcp_rn(d);
    if (isinf(inv)) inv = FLT_MAX;
  }
}

template <int MODE>
__global__ void __launch_bounds__(NV_WARPS * 32, 1)
nvfp4_quantize_kernel(const __grid_constant__ CUtensorMap tmap, const NvArgs a) {
  constexpr bool ROW = (MODE & MX_ROW) != 0;
  constexpr bool COL = (MODE & MX_COL) != 0;
  constexpr int STAGE_BYTES = NV_TILE_M * NV_TILE_K * 2;
  constexpr int ROW_PITCH = NV_TILE_K * 2;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[NV_WARPS][NV_STAGES];
  __shared__ __align__(16) uint32_t row_scale_stage[NV_WARPS][64];

  uint8_t* smem = align_up_shared<128>(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = lane >> 3;   // 16-row group 0..3
  const int c = lane & 7;    // 8-column chunk 0..7
  const uint32_t stage0 = smem_addr(smem) + warp * NV_STAGES * STAGE_BYTES;
  const uint32_t bar0 = smem_addr(&bars[warp][0]);
  const uint32_t rs_stage = smem_addr(&row_scale_stage[warp][0]);

  const float A = *a.amax;
  const float G = __fdiv_rn(A, 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) *a.global_scale = G;

  NvSchedule sched;
  const int gw = blockIdx.x * NV_WARPS + warp;
  const int W = gridDim.x * NV_WARPS;
  const int total = a.tiles_m * a.tiles_k;
  sched.first = gw;
  sched.step = W;
  sched.tiles_k = a.tiles_k;
  sched.count = gw < total ? (total - gw + W - 1) / W : 0;
  if (sched.count == 0) return;

  if (lane == 0) {
    prefetch_tensormap(&tmap);
#pragma unroll
    for (int s = 0; s < NV_STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
    fence_barrier_init();
  }
  __syncwarp();

  auto issue = [&](int j) {
    int tm, tk;
    sched.coords(j, tm, tk);
    const int s = j % NV_STAGES;
    mbar_arrive_expect_tx(bar0 + 8 * s, STAGE_BYTES);
    tma_load_2d(stage0 + s * STAGE_BYTES, &tmap, tk * NV_TILE_K, tm * NV_TILE_M, bar0 + 8 * s);
  };
  if (lane == 0) {
    const int pre = sched.count < NV_STAGES ? sched.count : NV_STAGES;
    for (int j = 0; j < pre; ++j) issue(j);
  }

  for (int j = 0; j < sched.count; ++j) {
    const int s = j % NV_STAGES;
    const bool ok = mbar_wait_bounded(bar0 + 8 * s, (j / NV_STAGES) & 1, a.timeout_ns);
    if (__any_sync(0xFFFFFFFFu, !ok)) {
      if (lane == 0 && a.dev_err) atomicOr(a.dev_err, 1u);
      const int last = (j + NV_STAGES < sched.count) ? j + NV_STAGES : sched.count;
      for (int jj = j + 1; jj < last; ++jj)
        mbar_wait_bounded(bar0 + 8 * (jj % NV_STAGES), (jj / NV_STAGES) & 1, a.timeout_ns);
      return;
    }
    int tm, tk;
    sched.coords(j, tm, tk);
    const uint32_t my_row0 = stage0 + s * STAGE_BYTES + (16 * h) * ROW_PITCH + c * 16;

    uint32_t xr[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint4 v = lds128(my_row0 + i * ROW_PITCH);
      xr[i][0] = v.x; xr[i][1] = v.y; xr[i][2] = v.z; xr[i][3] = v.w;
    }
    // cm[p]: magnitude maxima of columns 2p / 2p+1 over this lane's 16 rows
    // (complete transposed blocks).  rm[q]: rows 2q / 2q+1 over 8 columns.
    uint32_t cm[4] = {0u, 0u, 0u, 0u};
    uint32_t rm[8];
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
      rm[i / 2] = vmax_u16x2(prmt(t[0], t[1], 0x5410), prmt(t[0], t[1], 0x7632));
    }

    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && j + NV_STAGES < sched.count) issue(j + NV_STAGES);

    const int col0 = tk * NV_TILE_K + c * 8;
    const int row0 = tm * NV_TILE_M + 16 * h;
    const bool col_ok = col0 < a.K;
    const bool row_ok = row0 < a.M;

    if constexpr (ROW) {
      // 1x16 row blocks span lanes c = 2b, 2b+1.
#pragma unroll
      for (int q = 0; q < 8; ++q) rm[q] = vmax_u16x2(rm[q], __shfl_xor_sync(0xFFFFFFFFu, rm[q], 1));
      uint8_t* qrow = a.q_row + static_cast<size_t>(row0) * (a.K / 2) + col0 / 2;
      uint32_t codes[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float b = __uint_as_float(((rm[i >> 1] >> (16 * (i & 1))) & 0xFFFFu) << 16);
        float inv;
        nv_block_scale(b, G, codes[i], inv);
        const uint32_t w = cvt_e2m1x8(
            bf16_lo(xr[i][0]) * inv, bf16_hi(xr[i][0]) * inv, bf16_lo(xr[i][1]) * inv,
            bf16_hi(xr[i][1]) * inv, bf16_lo(xr[i][2]) * inv, bf16_hi(xr[i][2]) * inv,
            bf16_lo(xr[i][3]) * inv, bf16_hi(xr[i][3]) * inv);
        if (col_ok && row_ok) stg32(qrow + static_cast<size_t>(i) * (a.K / 2), w);
      }
      // Scale bytes: lanes c = 2b (rows i even) and 2b+1 (rows i odd) stage
      // block b of their rows into [64 rows][4 blocks]; lane L then writes
      // rows 2L and 2L+1.
      const int b = c >> 1, r = c & 1;
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const uint32_t code = r ? codes[i + 1] : codes[i];
        sts8(rs_stage + (16 * h + i + r) * 4 + b, code);
      }
      __syncwarp();
      const int nkb = a.K / 16;
      const int kb0 = tk * (NV_TILE_K / 16);
      const int valid = min(4, nkb - kb0);
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int tr = 2 * lane + rr;
        const int grow = tm * NV_TILE_M + tr;
        const uint32_t w = lds32(rs_stage + tr * 4);
        if (grow < a.M) {
          uint8_t* srow = a.s_row + static_cast<size_t>(grow) * nkb + kb0;
          if (valid == 4 && (nkb & 3) == 0) {
            stg32(srow, w);
          } else {
            for (int bb = 0; bb < valid; ++bb) stg8(srow + bb, (w >> (8 * bb)) & 0xFFu);
          }
        }
      }
    }

    if constexpr (COL) {
      uint8_t* qt = a.q_t + static_cast<size_t>(col0) * (a.M / 2) + row0 / 2;
      const int nmb = a.M / 16;
#pragma unroll
      for (int jc = 0; jc < 8; ++jc) {
        const uint32_t mag = (cm[jc >> 1] >> (16 * (jc & 1))) & 0xFFFFu;
        uint32_t code;
        float inv;
        nv_block_scale(__uint_as_float(mag << 16), G, code, inv);
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          v[i] = ((jc & 1) ? bf16_hi(xr[i][jc >> 1]) : bf16_lo(xr[i][jc >> 1])) * inv;
        const uint32_t w0 = cvt_e2m1x8(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
        const uint32_t w1 = cvt_e2m1x8(v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]);
        if (col_ok && row_ok) {
          stg64(qt + static_cast<size_t>(jc) * (a.M / 2), w0, w1);
          stg8(a.s_t + static_cast<size_t>(col0 + jc) * nmb + row0 / 16, code);
        }
      }
    }
    __syncwarp();   // row_scale_stage is rewritten by the next tile
  }
}

// Largest |x| of a bf16 matrix.  Each block takes whole rows; 16-byte loads;
// the bf16 magnitude bits are order-preserving, so the maximum is taken on
// integers and the fp32 bit pattern (bf16 << 16) is folded into *out with
// atomicMax, which gives the same result in any order.
__global__ void __launch_bounds__(256)
bf16_amax_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                 unsigned int* __restrict__ out) {
  const int64_t chunks = K / 8;
  uint32_t m = 0u;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const uint4* p = reinterpret_cast<const uint4*>(x + row * ldx);
    for (int64_t ch = threadIdx.x; ch < chunks; ch += blockDim.x) {
      const uint4 v = __ldcs(p + ch);
      m = vmax_u16x2(m, vmax_u16x2(vmax_u16x2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                   vmax_u16x2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu)));
    }
  }
  m = max(m & 0xFFFFu, m >> 16);
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t warp_max[8];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t v = threadIdx.x < (blockDim.x >> 5) ? warp_max[threadIdx.x] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (threadIdx.x == 0 && v != 0u) atomicMax(out, v << 16);
  }
}

// G = amax / 2688 alone, for an empty input with a caller-supplied amax.
__global__ void nv_global_scale_kernel(const float* amax, float* global_scale) {
  *global_scale = __fdiv_rn(*amax, 2688.0f);
}

// One warp waits on a barrier that nothing completes; the bounded wait
// gives up after timeout_ns and the kernel reports it in *dev_err.
__global__ void selftest_wait_kernel(uint64_t timeout_ns, uint32_t* dev_err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncwarp();
  const bool ok = mbar_wait_bounded(b, 0, timeout_ns);
  if (__any_sync(0xFFFFFFFFu, !ok) && threadIdx.x == 0) atomicOr(dev_err, 1u);
}

template <int MODE>
cudaError_t launch_nv_variant(const CUtensorMap& map, const NvArgs& a, int num_sms,
                              cudaStream_t stream) {
  constexpr int SMEM = NV_WARPS * NV_STAGES * NV_TILE_M * NV_TILE_K * 2 + 128;
  auto kernel = nvfp4_quantize_kernel<MODE>;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (configured_device != dev) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (err != cudaSuccess) return err;
    configured_device = dev;
  }
  const int64_t tiles = static_cast<int64_t>(a.tiles_m) * a.tiles_k;
  const int64_t ctas = (tiles + NV_WARPS - 1) / NV_WARPS;
  const int grid = static_cast<int>(ctas < num_sms ? ctas : num_sms);
  kernel<<<grid < 1 ? 1 : grid, NV_WARPS * 32, SMEM, stream>>>(map, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_nvfp4(const CUtensorMap& map, const NvArgs& a, int mode, int num_sms,
                         cudaStream_t stream) {
  switch (mode) {
    case MX_ROW: return launch_nv_variant<MX_ROW>(map, a, num_sms, stream);
    case MX_COL: return launch_nv_variant<MX_COL>(map, a, num_sms, stream);
    default: return launch_nv_variant<MX_ROW | MX_COL>(map, a, num_sms, stream);
  }
}

cudaError_t launch_bf16_amax(const void* x, int64_t M, int64_t K, int64_t ldx, float* out,
                             int num_sms, cudaStream_t stream) {
  cudaError_t err = cudaMemsetAsync(out, 0, sizeof(float), stream);
  if (err != cudaSuccess) return err;
  if (M == 0 || K == 0) return cudaSuccess;
  int64_t blocks = static_cast<int64_t>(num_sms) * 8;
  if (blocks > M) blocks = M;
  bf16_amax_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(x), M, K, ldx, reinterpret_cast<unsigned int*>(out));
  return cudaGetLastError();
}

cudaError_t launch_nv_global_scale(const float* amax, float* global_scale, cudaStream_t stream) {
  nv_global_scale_kernel<<<1, 1, 0, stream>>>(amax, global_scale);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(uint64_t timeout_ns, uint32_t* dev_err, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns, dev_err);
  return cudaGetLastError();
}

}  // namespace mxq
