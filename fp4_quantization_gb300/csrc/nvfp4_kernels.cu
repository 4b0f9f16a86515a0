// nvfp4_kernels.cu -- NVFP4 quantize-transpose, the tensor amax it needs,
// and the bounded-wait self test, for sm_103a.
//
// NVFP4 quantize-transpose is the "NVFP4 quantize-transpose" kernel family
// of TE PR #3291 "Fix pointer arithmatic to generate correct LDS/STS
// instructions" (results table "NVFP4 2D quantize-transpose kernel" and the
// 1D kernel named in its "Patched but not measurable" section); this file
// implements both: 1D (1x16 rowwise / 16x1 transposed blocks) and 2D (one
// scale per 16x16 block, used by both outputs).
//
// Layout of the work:
//  * One CTA (4 warps) per 128 x 128 tile of the input, the grid numbered
//    along K inside a 128-row band so the block scheduler hands tiles out in
//    address order; five CTAs share an SM.  Two TMA copies bring the tile
//    in, one per 64-column pass; the code staging reuses the first copy's
//    buffer once pass 0 has read it.
//  * The tile is taken in two 64-column passes.  Warp w owns rows
//    32w..32w+31; lane (h, c) = (lane / 8, lane % 8) owns rows 8h..8h+7 and
//    columns 8c..8c+7 of the pass (eight conflict-free 16-byte shared
//    loads).  A 1x16 row block spans lanes c = 2b, 2b+1 and a 16x1
//    transposed block spans lanes h = 2g, 2g+1: one xor shuffle each; a
//    16x16 block spans both pairs.
//  * Block scales follow the recipe's fixed fp32 order (b / 6) / G -> E4M3
//    -> value * G -> 1 / d: the code is decided from one multiply when that
//    is safe, else by the recipe's divisions (NvFastScale); 1/d comes from a
//    per-CTA table by code.  Each element then takes one multiply by 1/d
//    (two per mul.rn.f32x2; no per-element division, as in torchao PR #12
//    "Multiply with inverse scale in loop instead of dividing", rationale)
//    and cvt.rn.satfinite.e2m1x2.f32.
//  * Codes are staged per tile and leave through one 3-D TMA store per
//    direction, over [M][K/2] seen as [m % 8][m / 8][k / 2] and [K][M/2]
//    seen as [k % 8][k / 8][m / 2] (64-byte rows, 64-byte swizzle); scale
//    bytes as one 8-byte run per row and per column.

#include <cfloat>

#include "mxq_internal.h"
#include "mxq_ptx.cuh"

namespace mxq {
namespace {

// One bf16 magnitude of a packed pair of maxima, as its 15 magnitude bits
// (the sign bit left by max.xorsign.abs carries no meaning and is dropped).
__device__ __forceinline__ uint32_t mag16(uint32_t pair, int which) {
  return (pair >> (16 * which)) & 0x7FFFu;
}

// v[i] for a lane-dependent i without dynamic register indexing.
__device__ __forceinline__ uint32_t pick4(const uint32_t v[4], int i) {
  return (i & 2) ? ((i & 1) ? v[3] : v[2]) : ((i & 1) ? v[1] : v[0]);
}

// Shared memory of a CTA: the tile arrives as two 64-column copies (one per
// pass), and the code staging reuses the first copy's 16 KiB once pass 0
// has read it, so a CTA needs 35 KiB; with values widened to fp32 at each
// use (96 registers) five CTAs share an SM.  Measured on GB300 against one
// 32 KiB copy, separate staging and four CTAs per SM: 2D 16384 x 8192
// 65.2 -> 62.6 us, 2D 8192^2 37.0 -> 35.1 us, 1D 16384 x 8192 68.0 -> 68.2
// (six CTAs per SM spill: 1D 80.2 us).
constexpr int NT_CPS = 5;                                        // resident CTAs per SM
constexpr int NT_WARPS = 4;
constexpr int NT_ROWS = NV_TILE_ROWS;
constexpr int NT_COLS = NV_TILE_COLS;
constexpr int NT_TILE_BYTES = NT_ROWS * NT_COLS * 2;            // 32 KiB of bf16
constexpr int NT_LOADS = 2;                                      // input copies per tile
constexpr int NT_LOAD_BYTES = NT_TILE_BYTES / NT_LOADS;          // [128 rows][128 B] each
constexpr int NT_OFF_QR = 0;                                     // [m % 8][m / 8][64 B]
constexpr int NT_OFF_QT = NT_OFF_QR + NT_ROWS * NT_COLS / 2;     // [k % 8][k / 8][64 B]
constexpr int NT_OFF_RSC = NT_TILE_BYTES;                        // [128 rows][8 blocks]
constexpr int NT_OFF_TSC = NT_OFF_RSC + NT_ROWS * 8;             // [8 blocks][128 columns]
constexpr int NT_OFF_INV = NT_OFF_TSC + NT_COLS * 8;             // [128 codes] fp32 1/d
constexpr int NT_SMEM = NT_OFF_INV + 128 * 4 + 1024;             // + alignment pad
static_assert(NT_CPS * (NT_SMEM + 1024) <= 228 * 1024, "CTAs per SM");
static_assert(NT_OFF_QT + NT_COLS * NT_ROWS / 2 <= NT_LOAD_BYTES,
              "the staging fits in the first copy's buffer");

// Byte offset inside a [rows][64 B] staging block whose TMA map uses the
// 64-byte swizzle: the 16-byte chunk index is xor-ed with (row / 2) % 4.
__device__ __forceinline__ uint32_t swz64(int row, int byte) {
  return row * 64 + ((((byte >> 4) ^ ((row >> 1) & 3)) << 4) | (byte & 15));
}

// Scale codes without a per-amax table.  q = b * K with K = 1 / (6 G) is
// within a few units in the last place of the recipe's (b / 6) / G (two
// roundings each side); the codes of the fp32 values 16 units below and
// above q bound the recipe's code, so when they agree it is that code.  They
// disagree only within 16 units of an E4M3 rounding boundary -- in practice
// exact ties, e.g. G a power of two -- and those blocks, like every block
// when G is below 2^-100 (where b / 6 may round as a subnormal), take the
// recipe's division sequence.  1/d depends on the code alone: a 128-entry
// table built once per CTA with the recipe's operations.
struct NvFastScale {
  float K;            // 1 / (6 G), rounded twice
  float G;
  bool fast;          // 2^-100 <= G <= FLT_MAX
  uint32_t inv_tab;   // shared address of the [128] table of 1/d by code
};

__device__ __forceinline__ uint32_t nv_code_try(uint32_t mag, float K, uint32_t& miss) {
  const int q = __float_as_int(__fmul_rn(__uint_as_float(mag << 16), K));
  const uint32_t pair = cvt_e4m3x2(__int_as_float(max(q - 16, 0)),
                                   __int_as_float(min(q + 16, 0x7F7FFFFF)));
  miss |= pair ^ (pair >> 8);   // low byte nonzero: the two codes differ
  return pair & 0xFFu;
}

// The recipe's code for block amax bits `mag`: E4M3((b / 6) / G).
__device__ __forceinline__ uint32_t nv_code_exact(uint32_t mag, float G) {
  if (G == 0.0f) return 0u;
  return cvt_e4m3x2(__fdiv_rn(__fdiv_rn(__uint_as_float(mag << 16), 6.0f), G), 0.0f) & 0xFFu;
}

// A shared load the compiler may schedule freely: the table it reads is
// written before the CTA's first barrier and never again.
__device__ __forceinline__ float lds_table_f32(uint32_t addr) {
  float v;
  asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// Codes and reciprocals of N blocks whose amax bits are the bf16 halves of
// m[0..N/2) (block i: half i & 1 of m[i / 2]).
template <int N>
__device__ __forceinline__ void nv_scales(const uint32_t* m, const NvFastScale& fs,
                                          uint32_t* code, float* inv) {
  uint32_t miss = fs.fast ? 0u : 1u;
#pragma unroll
  for (int i = 0; i < N; ++i) code[i] = nv_code_try(mag16(m[i >> 1], i & 1), fs.K, miss);
  if (miss & 0xFFu) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      uint32_t one = fs.fast ? 0u : 1u;
      nv_code_try(mag16(m[i >> 1], i & 1), fs.K, one);
      if (one & 0xFFu) code[i] = nv_code_exact(mag16(m[i >> 1], i & 1), fs.G);
    }
  }
#pragma unroll
  for (int i = 0; i < N; ++i) inv[i] = lds_table_f32(fs.inv_tab + 4 * code[i]);
}

template <int MODE, bool TWO_D>
__global__ void __launch_bounds__(NT_WARPS * 32, NT_CPS)
nvfp4_tile_kernel(const __grid_constant__ CUtensorMap tmap_x,
                  const __grid_constant__ CUtensorMap tmap_qrow,
                  const __grid_constant__ CUtensorMap tmap_qt, const NvArgs a) {
  constexpr bool ROW = (MODE & MX_ROW) != 0;
  constexpr bool COL = (MODE & MX_COL) != 0;
  constexpr int ROW_PITCH = NT_LOAD_BYTES / NT_ROWS;   // bytes per row of one input copy

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[NT_LOADS];
  uint8_t* smem = align_up_shared<1024>(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h = lane >> 3;   // 8-row group 0..3 of the warp's 32 rows
  const int c = lane & 7;    // 8-column chunk 0..7 of the pass's 64 columns
  const uint32_t bar0 = smem_addr(&full_bar[0]);
  const unsigned t = a.reverse ? gridDim.x - 1u - blockIdx.x : blockIdx.x;
  const int band = static_cast<int>(t / static_cast<unsigned>(a.tiles_k));
  const int tk = static_cast<int>(t) - band * a.tiles_k;

  if (tid == 0) {
    if (ROW) prefetch_tensormap(&tmap_qrow);
    if (COL) prefetch_tensormap(&tmap_qt);
#pragma unroll
    for (int l = 0; l < NT_LOADS; ++l) mbar_init(bar0 + 8 * l, 1);
    fence_barrier_init();
#pragma unroll
    for (int l = 0; l < NT_LOADS; ++l) {
      mbar_arrive_expect_tx(bar0 + 8 * l, NT_LOAD_BYTES);
      tma_load_2d(sbase + l * NT_LOAD_BYTES, &tmap_x, tk * NT_COLS + l * (NT_COLS / NT_LOADS),
                  band * NT_ROWS, bar0 + 8 * l);
    }
  }
  // The tensor amax, read while the copy is in flight (after the amax grid
  // this one may depend on has completed), and the table of 1/d by code
  // (the recipe's d = value(s) * G, 1/d rounded to nearest).
  grid_dependency_wait();
  NvFastScale fs;
  {
    const float A = *a.amax;
    fs.G = __fdiv_rn(A, 2688.0f);
    fs.K = __frcp_rn(__fmul_rn(6.0f, fs.G));
    fs.fast = fs.G >= 0x1p-100f && fs.G <= FLT_MAX;
    fs.inv_tab = sbase + NT_OFF_INV;
    if (t == 0 && tid == 0) *a.global_scale = fs.G;
    float inv = 0.0f;
    if (tid != 0) {
      const float d = __fmul_rn(e4m3_to_f32(static_cast<uint32_t>(tid)), fs.G);
      if (d != 0.0f) {
        inv = __frcp_rn(d);
        if (isinf(inv)) inv = FLT_MAX;
      }
    }
    sts32(fs.inv_tab + 4 * tid, __float_as_uint(inv));
  }
  __syncthreads();

#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    {
      const bool ok = mbar_wait_bounded(bar0 + 8 * pass, 0, a.timeout_ns);
      if (__syncthreads_or(!ok)) {
        // A copy never landed: record it, let the copies finish (bounded)
        // and stop.
        if (tid == 0) {
          if (a.dev_err) atomicOr(a.dev_err, 1u);
          for (int l = pass; l < NT_LOADS; ++l) mbar_wait_bounded(bar0 + 8 * l, 0, a.timeout_ns);
        }
        return;
      }
    }
    // ---- this lane's 8 x 8 block; magnitude maxima ---------------------------
    const uint32_t my_row0 = sbase + pass * NT_LOAD_BYTES + (32 * warp + 8 * h) * ROW_PITCH + 16 * c;
    uint32_t xr[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 v = lds128(my_row0 + i * ROW_PITCH);
      xr[i][0] = v.x; xr[i][1] = v.y; xr[i][2] = v.z; xr[i][3] = v.w;
    }
    uint32_t cm[4] = {0u, 0u, 0u, 0u};   // columns 2p / 2p+1 over the lane's 8 rows
    uint32_t rm[4] = {0u, 0u, 0u, 0u};   // rows 2q / 2q+1 over the lane's 8 columns
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      uint32_t tt[2];
#pragma unroll
      for (int di = 0; di < 2; ++di) {
#pragma unroll
        for (int p = 0; p < 4; ++p) cm[p] = absmax_bf16x2(cm[p], xr[i + di][p]);
        tt[di] = absmax_bf16x2(absmax_bf16x2(xr[i + di][0], xr[i + di][1]),
                               absmax_bf16x2(xr[i + di][2], xr[i + di][3]));
      }
      rm[i / 2] = absmax_bf16x2(prmt(tt[0], tt[1], 0x5410), prmt(tt[0], tt[1], 0x7632));
    }

    // 2D: the 16x16 block's amax over the four lanes that hold it, and its
    // one scale.
    uint32_t code2d = 0u;
    float inv2d = 0.0f;
    if constexpr (TWO_D) {
      uint32_t m2 = absmax_bf16x2(absmax_bf16x2(rm[0], rm[1]), absmax_bf16x2(rm[2], rm[3]));
      m2 = absmax_bf16x2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 1));
      m2 = absmax_bf16x2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 8));
      const uint32_t mm = max(mag16(m2, 0), mag16(m2, 1));
      nv_scales<1>(&mm, fs, &code2d, &inv2d);
    }

    auto xv = [&](int i, int p) { return make_float2(bf16_lo(xr[i][p]), bf16_hi(xr[i][p])); };
    // Codes of the pass, stored to the staging below (pass 0 stores them only
    // after every warp has read the first copy, whose buffer they reuse).
    uint32_t qrw[8], qtw[8];

    // ---- rowwise: block scales (split over the c pair), codes, scale bytes --
    if constexpr (ROW) {
      const int mine = c & 1;               // this lane gathers the scale bytes of rows 4*mine..
      uint32_t rcode[4];
      float rinv[8];
      if constexpr (TWO_D) {
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) rcode[tq] = code2d;
#pragma unroll
        for (int i = 0; i < 8; ++i) rinv[i] = inv2d;
      } else {
        // This lane decides the blocks of its rows 4*mine..4*mine+3 (maxima
        // completed with the partner's half) and swaps 1/d with the partner
        // (both lanes deciding all eight: 71.6 instead of 68.2 us for
        // 16384 x 8192, measured on GB300).
        uint32_t mown[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t send = mine ? rm[q] : rm[2 + q];
          mown[q] = absmax_bf16x2(mine ? rm[2 + q] : rm[q],
                                  __shfl_xor_sync(0xFFFFFFFFu, send, 1));
        }
        float inv4[4];
        nv_scales<4>(mown, fs, rcode, inv4);
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) {
          const float other = __shfl_xor_sync(0xFFFFFFFFu, inv4[tq], 1);
          rinv[tq] = mine ? other : inv4[tq];
          rinv[4 + tq] = mine ? inv4[tq] : other;
        }
      }
      // Codes of row i: 8 values -> 4 bytes at byte 32 * pass + 4c of the
      // row's 64; staging row (m % 8) * 16 + m / 8.
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 iv = make_float2(rinv[i], rinv[i]);
        const float2 v0 = mul_f32x2(xv(i, 0), iv);
        const float2 v1 = mul_f32x2(xv(i, 1), iv);
        const float2 v2 = mul_f32x2(xv(i, 2), iv);
        const float2 v3 = mul_f32x2(xv(i, 3), iv);
        qrw[i] = cvt_e2m1x8(v0.x, v0.y, v1.x, v1.y, v2.x, v2.y, v3.x, v3.y);
      }
      // Scale bytes: the four lanes c = mine, mine + 2, mine + 4, mine + 6
      // hold blocks 0..3 of the pass for the same four rows; lane b = c / 2
      // gathers row 4 * mine + b (three shuffles) and stores one word.
      const int b = c >> 1;
      uint32_t word = pick4(rcode, b) << (8 * b);
#pragma unroll
      for (int k = 1; k < 4; ++k) {
        const int src_b = (b + k) & 3;
        const uint32_t got = __shfl_sync(0xFFFFFFFFu, pick4(rcode, (b - k) & 3),
                                         (lane & ~7) | (2 * src_b + mine));
        word |= got << (8 * src_b);
      }
      sts32(sbase + NT_OFF_RSC + (32 * warp + 8 * h + 4 * mine + b) * 8 + 4 * pass, word);
    }

    // ---- transposed: block scales (split over the h pair), codes, scales ----
    if constexpr (COL) {
      const int mine = h & 1;               // this lane stores the scale bytes of columns 4*mine..
      uint32_t tcode[4];
      float tinv[8];
      if constexpr (TWO_D) {
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) tcode[tq] = code2d;
#pragma unroll
        for (int j = 0; j < 8; ++j) tinv[j] = inv2d;
      } else {
        // This lane decides the blocks of its columns 4*mine..4*mine+3 and
        // swaps 1/d with the partner 8 rows away.
        uint32_t mown[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint32_t send = mine ? cm[q] : cm[2 + q];
          mown[q] = absmax_bf16x2(mine ? cm[2 + q] : cm[q],
                                  __shfl_xor_sync(0xFFFFFFFFu, send, 8));
        }
        float inv4[4];
        nv_scales<4>(mown, fs, tcode, inv4);
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) {
          const float other = __shfl_xor_sync(0xFFFFFFFFu, inv4[tq], 8);
          tinv[tq] = mine ? other : inv4[tq];
          tinv[4 + tq] = mine ? inv4[tq] : other;
        }
      }
      // Codes of column k = 64 * pass + 8c + j: 8 rows -> 4 bytes at byte
      // 16w + 4h of the column's 64; staging row (k % 8) * 16 + k / 8.
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float2 iv = make_float2(tinv[2 * p], tinv[2 * p + 1]);
        float2 r[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) r[i] = mul_f32x2(xv(i, p), iv);
        qtw[2 * p] = cvt_e2m1x8(r[0].x, r[1].x, r[2].x, r[3].x, r[4].x, r[5].x, r[6].x, r[7].x);
        qtw[2 * p + 1] = cvt_e2m1x8(r[0].y, r[1].y, r[2].y, r[3].y, r[4].y, r[5].y, r[6].y, r[7].y);
      }
      // Scale bytes [block][column]: the lane's four columns are adjacent.
      sts32(sbase + NT_OFF_TSC + (2 * warp + (h >> 1)) * NT_COLS + 64 * pass + 8 * c + 4 * mine,
            tcode[0] | (tcode[1] << 8) | (tcode[2] << 16) | (tcode[3] << 24));
    }

    // ---- the pass's codes to the staging ------------------------------------
    if (pass == 0) __syncthreads();   // the first copy is read: its buffer is free
    if constexpr (ROW) {
      // row i: 4 bytes at byte 32 * pass + 4c of the row's 64; staging row
      // (m % 8) * 16 + m / 8.
#pragma unroll
      for (int i = 0; i < 8; ++i)
        sts32(sbase + NT_OFF_QR + swz64(16 * i + 4 * warp + h, 32 * pass + 4 * c), qrw[i]);
    }
    if constexpr (COL) {
      // column k = 64 * pass + 8c + j: 4 bytes at byte 16w + 4h of the
      // column's 64; staging row (k % 8) * 16 + k / 8.
#pragma unroll
      for (int j = 0; j < 8; ++j)
        sts32(sbase + NT_OFF_QT + swz64(16 * j + 8 * pass + c, 16 * warp + 4 * h), qtw[j]);
    }
  }

  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0) {
    if (ROW) tma_store_3d(&tmap_qrow, sbase + NT_OFF_QR, tk * (NT_COLS / 2), band * (NT_ROWS / 8), 0);
    if (COL) tma_store_3d(&tmap_qt, sbase + NT_OFF_QT, band * (NT_ROWS / 2), tk * (NT_COLS / 8), 0);
    bulk_commit();
  }
  const uint64_t policy = l2_policy_evict_last();
  if (ROW) {
    // row tid: blocks 8 tk .. 8 tk + 7 of s_row [M][K / 16]
    const int nkb = a.K / 16;
    const int row = band * NT_ROWS + tid;
    const int nb = min(8, nkb - 8 * tk);
    if (row < a.M) {
      uint8_t* dst = a.s_row + static_cast<size_t>(row) * nkb + 8 * tk;
      const uint32_t src = sbase + NT_OFF_RSC + tid * 8;
      if (nb == 8 && (reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
        const uint2 w = lds64(src);
        stg64_hint(dst, w.x, w.y, policy);
      } else {
        for (int bb = 0; bb < nb; ++bb) stg8(dst + bb, ld_shared_u8(src + bb));
      }
    }
  }
  if (COL) {
    // column tid: blocks 8 band .. 8 band + 7 of s_t [K][M / 16]
    const int nmb = a.M / 16;
    const int k = tk * NT_COLS + tid;
    const int nb = min(8, nmb - 8 * band);
    if (k < a.K) {
      uint8_t* dst = a.s_t + static_cast<size_t>(k) * nmb + 8 * band;
      const uint32_t src = sbase + NT_OFF_TSC + tid;
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int bb = 0; bb < 8; ++bb) w[bb >> 2] |= ld_shared_u8(src + bb * NT_COLS) << (8 * (bb & 3));
      if (nb == 8 && (reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
        stg64_hint(dst, w[0], w[1], policy);
      } else {
        for (int bb = 0; bb < nb; ++bb) stg8(dst + bb, (w[bb >> 2] >> (8 * (bb & 3))) & 0xFFu);
      }
    }
  }
  // The staged codes must have left shared memory before the CTA exits.
  if (tid == 0) bulk_wait_read<0>();
}

// Largest |x| of a bf16 matrix.  Each block takes whole rows; 16-byte loads;
// the bf16 magnitude bits are order-preserving, so the maximum is taken on
// integers and the fp32 bit pattern (bf16 << 16) is folded into *out with
// atomicMax, which gives the same result in any order.
__global__ void __launch_bounds__(256)
bf16_amax_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                 unsigned int* __restrict__ out) {
  // A quantize grid launched as a programmatic dependent may be scheduled
  // now: it reads only the input until it has waited for this grid.
  grid_launch_dependents();
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

// One launch: one CTA per 128 x 128 tile, in address order.  Right after
// this call's own amax grid it is launched as that grid's programmatic
// dependent (the first copies and the set-up overlap the amax grid's tail;
// the kernel waits for it before reading the amax); never after a caller's
// kernel, which may still be writing the input.
template <int MODE, bool TWO_D>
cudaError_t launch_nv_tile_variant(const NvMaps& maps, const NvArgs& a, bool after_amax,
                                   cudaStream_t stream) {
  static int configured_device = -1;
  auto kernel = nvfp4_tile_kernel<MODE, TWO_D>;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (configured_device != dev) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, NT_SMEM);
    if (err != cudaSuccess) return err;
    configured_device = dev;
  }
  const int64_t tiles = static_cast<int64_t>(a.tiles_m) * a.tiles_k;
  if (tiles < 1 || tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles));
  cfg.blockDim = dim3(NT_WARPS * 32);
  cfg.dynamicSmemBytes = NT_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_amax ? 1 : 0;
  // After the call's own amax pass the tiles go last first: the first ones
  // find the input the amax pass read last still in L2.
  NvArgs args = a;
  args.reverse = after_amax ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, maps.x, maps.q_row, maps.q_t, args);
}

template <bool TWO_D>
cudaError_t launch_nv_mode(const NvMaps& maps, const NvArgs& a, int mode, bool after_amax,
                           cudaStream_t stream) {
  switch (mode) {
    case MX_ROW: return launch_nv_tile_variant<MX_ROW, TWO_D>(maps, a, after_amax, stream);
    case MX_COL: return launch_nv_tile_variant<MX_COL, TWO_D>(maps, a, after_amax, stream);
    default: return launch_nv_tile_variant<MX_ROW | MX_COL, TWO_D>(maps, a, after_amax, stream);
  }
}

}  // namespace

int nv_load_cols() { return NT_COLS / NT_LOADS; }

cudaError_t launch_nvfp4(const NvMaps& maps, const NvArgs& a, int mode, bool two_d,
                         bool after_amax, cudaStream_t stream) {
  return two_d ? launch_nv_mode<true>(maps, a, mode, after_amax, stream)
               : launch_nv_mode<false>(maps, a, mode, after_amax, stream);
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
