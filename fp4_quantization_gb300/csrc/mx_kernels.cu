// mx_kernels.cu -- MXFP8 quantization kernels for sm_103a.
//
// Two kernels cover the MXFP8 paths of TE PR #3291 "Fix pointer arithmatic
// to generate correct LDS/STS instructions" (results tables "MXFP8 generic
// quantize kernel": plain / dbias / gelu; "MXFP8 specialized cast-only
// kernel (bidimensional)": plain row / both; "MXFP8 gated (swiglu / geglu)
// kernel": swiglu) and the colwise "dim1" cast of torchao PR #12 "Multiply
// with inverse scale in loop instead of dividing":
//  * the plain cast, with or without dbias, runs mx_cast_tile_kernel, one
//    short CTA per 128 x 128 tile dispatched in address order (see its
//    comment: a persistent grid reads and writes HBM more slowly on GB300);
//  * the activation paths (GELU, SwiGLU / GeGLU, the backward fusions, with
//    their dbias) run the persistent mx_quantize_kernel described here,
//    whose TMA ring overlaps the next tile's copy with the arithmetic they
//    need.
// Both use the same lane layout and arithmetic.
//
// The path is bound by HBM traffic, and on GB300 the write side costs by
// the number of L2 write requests rather than by bytes: a 1-byte store costs
// as much as a 32-byte one.  The persistent kernel is laid out so every
// output leaves in whole sectors or lines:
//  * One CTA of WARPS warps per SM (persistent) walks a contiguous range of
//    "steps"; a step is a band of BAND = 16 * WARPS rows x 128 columns,
//    loaded by one TMA box into a ring of STAGES slots (one mbarrier per
//    slot).  Bands are taken GROUP at a time, and inside a group the steps
//    run column by column with the group's bands interleaved.
//  * Warp w owns rows 16w..16w+15 of the band; lane (h, c) = (lane / 16,
//    lane % 16) owns rows 8h..8h+7 and columns 8c..8c+7 of those: 8
//    conflict-free 16-byte shared loads (a quarter warp reads one contiguous
//    128-byte row segment).  Colwise 32x1 amax: in-thread over 8 rows, one
//    xor-16 shuffle, then the two warps of a 32-row block swap their halves
//    through shared memory at the step's first barrier; rowwise 1x32 amax:
//    in-thread over 8 columns + xor-1 / xor-2 shuffles, two rows per
//    register.
//  * The shared scale is read off the exponent field of the amax; elements
//    are multiplied by the exact power of two 2^-e (two per mul.rn.f32x2, no
//    division; torchao PR #12, rationale) and converted two at a time by
//    cvt.rn.satfinite.e4m3x2.f32.
//  * Rowwise codes go straight to global memory (a half warp writes one full
//    128-byte line per streaming-store instruction) or, for the variants
//    where that measured faster, are staged in shared memory (128-byte
//    swizzle) and leave by one 2-D bulk tensor store per step.
//  * Colwise codes of the band are staged in shared memory and leave through
//    3-D TMA stores over the [K][M] output viewed as [k % 8][k / 8][m] with
//    128-byte swizzle: every global segment is a full 128-byte line, and the
//    swizzle spreads one shared store instruction over all banks.  The
//    group's bands follow one another along m, so a CTA writes GROUP * 128
//    contiguous bytes of each colwise code row in consecutive steps.
//  * Rowwise scale bytes of 8 consecutive column steps (1024 columns) are
//    gathered in shared memory and written as one 32-byte sector per row;
//    colwise scale bytes of the group's bands (GROUP * BAND / 32 blocks)
//    leave as one run per column.
//  * dbias: per step, the band's column sums are combined across warps in
//    shared memory and written once per (band, column); a second small
//    kernel adds the bands.

#include "mxq_internal.h"
#include "mxq_ptx.cuh"

// This file is compiled twice: with MXQ_TILED_SCALES 0 (row-major scale
// output; exports launch_mx and the shared helpers) and 1 (scales in 128 x 4
// tiles; exports launch_mx_tiled), so neither variant carries the other's
// scale code.
#ifndef MXQ_TILED_SCALES
#define MXQ_TILED_SCALES 0
#endif
// The two builds' kernels carry different names, so that a profile tells
// them apart.
#if MXQ_TILED_SCALES
#define MX_KERNEL mx_quantize_tiled_kernel
#define MX_TILE_KERNEL mx_cast_tile_tiled_kernel
#else
#define MX_KERNEL mx_quantize_kernel
#define MX_TILE_KERNEL mx_cast_tile_kernel
#endif
// L2 policies (tuning builds): input copies 1 evict-first, 2 evict-last,
// 3 evict-normal; colwise code stores 0 none, 1 evict-first, 2 evict-last,
// 3 evict-normal; rowwise code stores streaming (.cs) or plain.  Copies two
// ring slots at a time when MXQ_LOAD_PAIR (even slot counts).
#ifndef MXQ_LOAD_POLICY
#define MXQ_LOAD_POLICY 3
#endif
#ifndef MXQ_QCOL_POLICY
#define MXQ_QCOL_POLICY 0
#endif
#ifndef MXQ_QROW_CS
#define MXQ_QROW_CS 1
#endif
#ifndef MXQ_LOAD_PAIR
#define MXQ_LOAD_PAIR 0
#endif
// L2 policy of the colwise scale runs (row-major scales): 2 evict-last,
// 3 evict-normal.
// Rowwise codes of the plain cast by bulk tensor store (tuning builds).
#ifndef MXQ_PLAIN_RTMA
#define MXQ_PLAIN_RTMA 0
#endif
#ifndef MXQ_CSC_POLICY
#define MXQ_CSC_POLICY 2
#endif

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

// Operand tiles per step and output tiles per step of each activation.
__host__ __device__ constexpr int act_operands(int act) {
  return act == ACT_NONE || act == ACT_GELU ? 1
         : (act == ACT_DSWIGLU || act == ACT_DGEGLU) ? 3 : 2;
}
__host__ __device__ constexpr int act_outputs(int act) {
  return (act == ACT_DSWIGLU || act == ACT_DGEGLU) ? 2 : 1;
}

// Element functions, evaluated on two elements at a time: the fp32
// arithmetic runs as packed f32x2 instructions (two lanes per instruction,
// measured 3-14% faster than scalar code on the fused paths), ex2 / rcp
// stay scalar.  The results are a few fp32 ulps from the exact values.
__device__ __forceinline__ float2 f2(float v) { return make_float2(v, v); }

__device__ __forceinline__ float2 ex2_pair(float2 v) {
  return make_float2(ex2_approx(v.x), ex2_approx(v.y));
}
__device__ __forceinline__ float2 rcp_pair(float2 v) {
  return make_float2(rcp_approx(v.x), rcp_approx(v.y));
}

// tanh-form GELU, 0.5 x (1 + tanh(u)) with u = sqrt(2/pi) (x + 0.044715 x^3),
// through the identity 0.5 (1 + tanh(u)) = 1 / (1 + e^(-2u)):
// gelu_tanh(x) = x / (1 + 2^(x (k + k a x^2))), k = -2 sqrt(2/pi) log2(e).
__device__ __forceinline__ float2 gelu_tanh_pair(float2 x) {
  constexpr float k = -2.0f * 0.7978845608028654f * 1.4426950408889634f;
  const float2 x2 = mul_f32x2(x, x);
  const float2 arg = mul_f32x2(x, fma_f32x2(x2, f2(k * 0.044715f), f2(k)));
  return mul_f32x2(x, rcp_pair(add_f32x2(ex2_pair(arg), f2(1.0f))));
}

// silu(g) = g / (1 + e^-g).
__device__ __forceinline__ float2 silu_pair(float2 g) {
  constexpr float kNegLog2e = -1.4426950408889634f;
  const float2 e = ex2_pair(mul_f32x2(g, f2(kNegLog2e)));
  return mul_f32x2(g, rcp_pair(add_f32x2(e, f2(1.0f))));
}

// gelu_tanh(x) and its derivative
//   0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) sqrt(2/pi) (1 + 3 * 0.044715 x^2),
// both from s = e^(-2|u|) in (0, 1]: 1 + tanh u is 2 / (1 + s) for u >= 0 and
// 2 s / (1 + s) below, 1 - tanh^2 u = 4 s / (1 + s)^2 (no cancellation, no
// overflow).
__device__ __forceinline__ void gelu_tanh_d_pair(float2 x, float2& value, float2& deriv) {
  constexpr float kC = 0.7978845608028654f;
  constexpr float kNeg2Log2e = -2.0f * 1.4426950408889634f;
  const float2 x2 = mul_f32x2(x, x);
  const float2 u = mul_f32x2(x, fma_f32x2(x2, f2(kC * 0.044715f), f2(kC)));
  const float2 sv = ex2_pair(mul_f32x2(make_float2(fabsf(u.x), fabsf(u.y)), f2(kNeg2Log2e)));
  const float2 r = rcp_pair(add_f32x2(sv, f2(1.0f)));
  const float2 num = make_float2(u.x >= 0.0f ? 2.0f : 2.0f * sv.x, u.y >= 0.0f ? 2.0f : 2.0f * sv.y);
  const float2 one_plus_tanh = mul_f32x2(num, r);
  const float2 sech2 = mul_f32x2(mul_f32x2(sv, f2(4.0f)), mul_f32x2(r, r));
  value = mul_f32x2(mul_f32x2(x, f2(0.5f)), one_plus_tanh);
  const float2 slope = mul_f32x2(mul_f32x2(x, sech2), f2(0.5f * kC));
  deriv = fma_f32x2(slope, fma_f32x2(x2, f2(3.0f * 0.044715f), f2(1.0f)),
                    mul_f32x2(one_plus_tanh, f2(0.5f)));
}

// silu(x) = x sigma(x) and its derivative sigma(x) (1 + x sigma(-x)), from
// t = e^(-|x|) in (0, 1] (sigma of the negative side is t / (1 + t)).
__device__ __forceinline__ void silu_d_pair(float2 x, float2& value, float2& deriv) {
  constexpr float kNegLog2e = -1.4426950408889634f;
  const float2 t = ex2_pair(mul_f32x2(make_float2(fabsf(x.x), fabsf(x.y)), f2(kNegLog2e)));
  const float2 r = rcp_pair(add_f32x2(t, f2(1.0f)));
  const float2 tr = mul_f32x2(t, r);
  const float2 sp = make_float2(x.x >= 0.0f ? r.x : tr.x, x.y >= 0.0f ? r.y : tr.y);
  const float2 sm = make_float2(x.x >= 0.0f ? tr.x : r.x, x.y >= 0.0f ? tr.y : r.y);
  value = mul_f32x2(x, sp);
  deriv = mul_f32x2(sp, fma_f32x2(x, sm, f2(1.0f)));
}

// y of output t from the operands of two elements: x (plain / GELU), gate
// and up (SwiGLU / GeGLU), grad and x (dGELU / dSiLU), grad, gate and up (the
// gated backward: t = 0 is d gate = grad * up * act'(gate), t = 1 is
// d up = grad * act(gate)).
template <int ACT>
__device__ __forceinline__ float2 act_pair(float2 o0, float2 o1, float2 o2, int t) {
  if constexpr (ACT == ACT_GELU) {
    return gelu_tanh_pair(o0);
  } else if constexpr (ACT == ACT_SWIGLU) {
    return mul_f32x2(silu_pair(o0), o1);
  } else if constexpr (ACT == ACT_GEGLU) {
    return mul_f32x2(gelu_tanh_pair(o0), o1);
  } else if constexpr (ACT == ACT_DGELU || ACT == ACT_DSILU) {
    float2 v, d;
    if constexpr (ACT == ACT_DGELU) gelu_tanh_d_pair(o1, v, d);
    else silu_d_pair(o1, v, d);
    return mul_f32x2(o0, d);
  } else {
    float2 v, d;
    if constexpr (ACT == ACT_DGEGLU) gelu_tanh_d_pair(o1, v, d);
    else silu_d_pair(o1, v, d);
    return t == 0 ? mul_f32x2(mul_f32x2(o0, o2), d) : mul_f32x2(o0, v);
  }
}

// Both outputs of the gated backward from one evaluation of act and act':
// d gate = grad * up * act'(gate), d up = grad * act(gate) (o0 grad, o1 gate,
// o2 up; the same fp32 operations as act_pair for t = 0 and t = 1).
template <int ACT>
__device__ __forceinline__ void dgated_pair(float2 o0, float2 o1, float2 o2, float2& dgate,
                                            float2& dup) {
  float2 v, d;
  if constexpr (ACT == ACT_DGEGLU) gelu_tanh_d_pair(o1, v, d);
  else silu_d_pair(o1, v, d);
  dgate = mul_f32x2(mul_f32x2(o0, o2), d);
  dup = mul_f32x2(o0, v);
}

// ---------------------------------------------------------------------------
// Small helpers
// ---------------------------------------------------------------------------

// Packed exponents (two 16-bit lanes) -> two E8M0 codes (two 16-bit lanes):
// max(E, 8) - 8 on both halves (no borrow crosses halves after the max).
__device__ __forceinline__ uint32_t e8m0_pair(uint32_t e2) {
  return vmax_u16x2(e2, 0x00080008u) - 0x00080008u;
}

__device__ __forceinline__ uint32_t half16(uint32_t pair, int which) {
  return (pair >> (16 * which)) & 0xFFFFu;
}

// Scale exponents of a packed pair of bf16 maxima (two 16-bit lanes; the
// sign bits carry no meaning) under the selected rule.  Floor rule
// (ceil_add = 0): the exponent field E.  Ceil rule (ceil_add = 0x001F001F):
// E + 1 where the significand is above 1.75, i.e. where the 7 stored
// mantissa bits exceed 0x60 -- adding 0x1F to them carries into the
// exponent field exactly then.  (2^(E-127) * m > 448 * 2^(E-135) exactly
// when m > 1.75, so E - 8 + [m > 1.75] is ceil(log2(amax / 448)) + 127.)
// For finite maxima the carry never leaves its lane.  The code is monotone
// in the amax, so block maxima may be combined on these values.
__device__ __forceinline__ uint32_t bf16_scale_exponents(uint32_t m, uint32_t ceil_add) {
  return ((m + ceil_add) >> 7) & 0x00FF00FFu;
}

// The same for one fp32 magnitude (bits without the sign); ceil_add is 0 or
// 0x1FFFFF (23 mantissa bits above 0x600000 carry into the exponent).
__device__ __forceinline__ uint32_t f32_scale_exponent(uint32_t b, uint32_t ceil_add) {
  return (b + ceil_add) >> 23;
}

// Largest of three floats (one three-input max instruction).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void bar_sync_cta(int threads) {
  asm volatile("bar.sync 1, %0;" :: "r"(threads) : "memory");
}

// ---------------------------------------------------------------------------
// Shared-memory layout of one CTA
// ---------------------------------------------------------------------------

template <int WARPS, int OPERANDS, int NSTAGES, int GROUP, int QBUF, int CPITCH, int NOUT,
          bool RTMA>
struct MxLayout {
  static constexpr int BAND = 16 * WARPS;
  static constexpr int BPB = BAND / 32;                              // colwise blocks per band
  static constexpr int TILE_BYTES = BAND * MX_TILE_K * 2;            // one bf16 operand
  static constexpr int STAGE_BYTES = TILE_BYTES * OPERANDS;
  static constexpr int STAGES = NSTAGES;
  static constexpr int QCOL_HALF = 128 * MX_TILE_K;                  // 128 m x 128 k codes
  static constexpr int QCOL_HALVES = BAND / 128;
  static constexpr int QCOL_BUF = QCOL_HALVES * QCOL_HALF;            // one step's codes
  static constexpr int OFF_QCOL = STAGES * STAGE_BYTES;              // 1024-aligned
  // [NOUT outputs][GROUP bands][BAND rows][8 steps][4 blocks]
  // Rowwise code staging when the rowwise codes leave by bulk store (not
  // for the three-operand steps: no room).
  static constexpr bool ROW_TMA = RTMA && OPERANDS < 3;
  static constexpr int QROW_BYTES = ROW_TMA ? BAND * MX_TILE_K : 0;
  static constexpr int OFF_QROW = OFF_QCOL + QBUF * QCOL_BUF;
  static constexpr int OFF_RSC = OFF_QROW + QROW_BYTES;
  // Colwise scale bytes, GROUP * BPB blocks of 128 columns: [128 columns]
  // [CPITCH bytes] when there are four blocks (one 4-byte word per column),
  // else [blocks][128 columns].
  static constexpr bool CSC_BY_COL = GROUP * BPB == 4;
  static_assert(CPITCH == 4 || CPITCH == 8, "column pitch of the scale staging");
  static constexpr int OFF_CSC = OFF_RSC + NOUT * GROUP * BAND * 32;
  static constexpr int CSC_BYTES = CSC_BY_COL ? MX_TILE_K * CPITCH : GROUP * BPB * MX_TILE_K;
  // Column sums of each warp's 16 rows, [WARPS][128] fp32, column 8c + j of
  // the step at position (j / 4) * 64 + 4c + j % 4 of the warp's row.
  static constexpr int OFF_DB = OFF_CSC + CSC_BYTES;
  static constexpr int OFF_XCH = OFF_DB + WARPS * MX_TILE_K * 4;     // [WARPS][16][4] u32
  static constexpr int BYTES = OFF_XCH + WARPS * 16 * 16;
  static constexpr int DYNAMIC = BYTES + 1024;                       // + alignment pad
  __device__ static constexpr int csc(int blk, int col) {
    return CSC_BY_COL ? col * CPITCH + blk : blk * MX_TILE_K + col;
  }
};

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

template <int MODE, bool DBIAS, int ACT, int WARPS, int STAGES, int GROUP, int QBUF,
          int CPITCH, int CPS, bool RTMA>
__global__ void __launch_bounds__(WARPS * 32, CPS)
MX_KERNEL(const __grid_constant__ CUtensorMap tmap_x,
                   const __grid_constant__ CUtensorMap tmap_x2,
                   const __grid_constant__ CUtensorMap tmap_qcol,
                   const __grid_constant__ CUtensorMap tmap_qcol2,
                   const __grid_constant__ CUtensorMap tmap_qrow,
                   const __grid_constant__ CUtensorMap tmap_qrow2, const MxArgs a) {
  constexpr bool ROW = (MODE & MX_ROW) != 0;
  constexpr bool COL = (MODE & MX_COL) != 0;
  constexpr int OPERANDS = act_operands(ACT);
  constexpr int NOUT = act_outputs(ACT);
  using L = MxLayout<WARPS, OPERANDS, STAGES, GROUP, QBUF, CPITCH, NOUT, RTMA>;
  constexpr int THREADS = WARPS * 32;
  constexpr int BAND = L::BAND;
  constexpr int ROW_PITCH = MX_TILE_K * 2;   // bf16 tile row, bytes
  static_assert(!DBIAS || ACT == ACT_NONE || ACT == ACT_DGELU || ACT == ACT_DSILU,
                "dbias is defined on the plain and single-input backward paths");
  static_assert(NOUT == 1 || GROUP == 1, "two-output steps keep one band per CTA");
  static_assert(BAND % 128 == 0 && BAND <= 256, "colwise codes leave in 128-row halves");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[L::STAGES];

  uint8_t* smem = align_up_shared<1024>(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h = lane >> 4;     // which 8-row half of the warp's 16 rows
  const int c = lane & 15;     // which 8-column chunk
  const uint32_t bar0 = smem_addr(&full_bar[0]);

  // This CTA's contiguous range of steps.  Bands are taken GROUP at a time;
  // inside a group the steps run column by column, the group's bands
  // interleaved, so the colwise output of GROUP consecutive bands (and their
  // colwise scale bytes) is written by one CTA in consecutive steps.
  // dbias: the finalize grid (launched as a programmatic dependent) may be
  // scheduled now; it waits for this grid's completion before reading.
  if constexpr (DBIAS) grid_launch_dependents();

  const int64_t total = static_cast<int64_t>(a.tiles_m) * a.tiles_k;
  const int t0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * total / gridDim.x);
  const int t1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * total / gridDim.x);
  const int count = t1 - t0;
  if (count <= 0) return;

  // Position of a step: group g (bands g * GROUP ..), its band count nb,
  // band index bi inside the group and column step tk.  Decoded once for
  // the range's first step, then advanced step by step.
  struct Pos {
    int g, nb, bi, tk;
    __device__ int band() const { return g * GROUP + bi; }
    __device__ void advance(int tiles_m, int tiles_k) {
      if (++bi < nb) return;
      bi = 0;
      if (++tk < tiles_k) return;
      tk = 0;
      ++g;
      nb = min(GROUP, tiles_m - g * GROUP);
    }
  };
  Pos p0;
  {
    const int gsteps = GROUP * a.tiles_k;
    p0.g = t0 / gsteps;
    const int local = t0 - p0.g * gsteps;
    p0.nb = min(GROUP, a.tiles_m - p0.g * GROUP);
    p0.tk = local / p0.nb;
    p0.bi = local - p0.tk * p0.nb;
  }
  Pos lpos = p0;   // next step to load (thread 0)
  // L2 policies.  Rowwise codes leave with the streaming (.cs) operator, so
  // L2 gives their lines up first and writes them back while the reads
  // stream in; the colwise scale runs (row-major scales: an eighth of a
  // sector each, completed by other CTAs later) are kept with evict-last
  // until their sectors are whole; the input tiles are loaded evict-normal,
  // below the scale runs.  Measured on GB300 against evict-last input tiles:
  // 16384^2 184.5 -> 180.4 us, 8192x28672 173.0 -> 159.7 us, 16384x28672
  // 363.4 -> 317.8 us (the wider the matrix, the more scale runs wait in L2).
  const uint64_t csc_policy = MXQ_CSC_POLICY == 3 ? l2_policy_evict_normal() : l2_policy_evict_last();
#if MXQ_LOAD_POLICY == 1
  const uint64_t load_policy = l2_policy_evict_first();
#elif MXQ_LOAD_POLICY == 3
  const uint64_t load_policy = l2_policy_evict_normal();
#else
  const uint64_t load_policy = l2_policy_evict_last();
#endif

  auto issue_load = [&](int j) {   // thread 0 only, for j = 0, 1, 2, ... in order
    const int s = j % STAGES;
    const uint32_t dst = sbase + s * L::STAGE_BYTES;
    mbar_arrive_expect_tx(bar0 + 8 * s, L::STAGE_BYTES);
    tma_load_2d_hint(dst, &tmap_x, lpos.tk * MX_TILE_K, lpos.band() * BAND, bar0 + 8 * s,
                     load_policy);
    if (OPERANDS >= 2)
      tma_load_2d_hint(dst + L::TILE_BYTES, &tmap_x2, a.up_col + lpos.tk * MX_TILE_K,
                       lpos.band() * BAND, bar0 + 8 * s, load_policy);
    if (OPERANDS >= 3)
      tma_load_2d_hint(dst + 2 * L::TILE_BYTES, &tmap_x2, a.up_col2 + lpos.tk * MX_TILE_K,
                       lpos.band() * BAND, bar0 + 8 * s, load_policy);
    lpos.advance(a.tiles_m, a.tiles_k);
  };

  if (tid == 0) {
    prefetch_tensormap(&tmap_x);
    if (OPERANDS >= 2) prefetch_tensormap(&tmap_x2);
    if (COL) prefetch_tensormap(&tmap_qcol);
    if (COL && NOUT == 2) prefetch_tensormap(&tmap_qcol2);
    if (ROW && L::ROW_TMA) prefetch_tensormap(&tmap_qrow);
    if (ROW && L::ROW_TMA && NOUT == 2) prefetch_tensormap(&tmap_qrow2);
#pragma unroll
    for (int st = 0; st < STAGES; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_barrier_init();
    for (int jj = 0; jj < STAGES && jj < count; ++jj) issue_load(jj);
  }
  __syncthreads();

  // Scale rule: the carry constants of bf16_scale_exponents / f32_scale_exponent.
  const uint32_t ceil_bf16 = a.scale_ceil ? 0x001F001Fu : 0u;
  const uint32_t ceil_f32 = a.scale_ceil ? 0x001FFFFFu : 0u;
  const int nmb = a.M / 32;    // colwise scale bytes per column
  const int nkb = a.K / 32;    // rowwise scale bytes per row

  Pos pos = p0;
  for (int j = 0; j < count; ++j, pos.advance(a.tiles_m, a.tiles_k)) {
    const int s = j % STAGES;
    const int band = pos.band();
    const int tk = pos.tk;
    const bool ok = mbar_wait_bounded(bar0 + 8 * s, (j / STAGES) & 1, a.timeout_ns);

    // One pass per output tile of the step (two for the gated backward,
    // which writes d gate and d up from the same loaded tiles).
    for (int t = 0; t < NOUT; ++t) {
      const uint32_t my_row0 =
          sbase + s * L::STAGE_BYTES + (16 * warp + 8 * h) * ROW_PITCH + c * 16;

      // ---- load this lane's 8 x 8 block and reduce it to magnitude maxima ---
      // The plain path keeps the packed bf16 pairs (xr) and widens them where
      // they are used; the activation paths hold y in fp32.  ce[p] / re[q]:
      // exponent fields of the largest magnitudes of columns 2p, 2p+1 / rows
      // 2q, 2q+1, packed as two 16-bit lanes.
      uint32_t xr[ACT == ACT_NONE ? 8 : 1][4];
      float y[ACT == ACT_NONE ? 1 : 8][8];
      uint32_t ce[4] = {0u, 0u, 0u, 0u};
      uint32_t re[4] = {0u, 0u, 0u, 0u};
      if (ok) {
        if constexpr (ACT == ACT_NONE) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v = lds128(my_row0 + i * ROW_PITCH);
            xr[i][0] = v.x; xr[i][1] = v.y; xr[i][2] = v.z; xr[i][3] = v.w;
          }
          uint32_t cm[4] = {0u, 0u, 0u, 0u};
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
            // low halves: even columns, high halves: odd columns; fold per row.
            re[i / 2] = bf16_scale_exponents(
                absmax_bf16x2(prmt(tt[0], tt[1], 0x5410), prmt(tt[0], tt[1], 0x7632)), ceil_bf16);
          }
#pragma unroll
          for (int p = 0; p < 4; ++p) ce[p] = bf16_scale_exponents(cm[p], ceil_bf16);
        } else {
          if (NOUT == 2 && t == 1) {
            // Gated backward, d up: grad * act(gate) was computed in the
            // d-gate pass and parked, as fp32, in this lane's own gate and up
            // bytes of the slot (row i: columns 0-3 in the gate tile, 4-7 in
            // the up tile).
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 lo = lds128(my_row0 + L::TILE_BYTES + i * ROW_PITCH);
              const uint4 hi = lds128(my_row0 + 2 * L::TILE_BYTES + i * ROW_PITCH);
              y[i][0] = __uint_as_float(lo.x); y[i][1] = __uint_as_float(lo.y);
              y[i][2] = __uint_as_float(lo.z); y[i][3] = __uint_as_float(lo.w);
              y[i][4] = __uint_as_float(hi.x); y[i][5] = __uint_as_float(hi.y);
              y[i][6] = __uint_as_float(hi.z); y[i][7] = __uint_as_float(hi.w);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 v = lds128(my_row0 + i * ROW_PITCH);
              uint32_t u[4] = {0u, 0u, 0u, 0u}, w2[4] = {0u, 0u, 0u, 0u};
              if constexpr (OPERANDS >= 2) {
                const uint4 w = lds128(my_row0 + L::TILE_BYTES + i * ROW_PITCH);
                u[0] = w.x; u[1] = w.y; u[2] = w.z; u[3] = w.w;
              }
              if constexpr (OPERANDS >= 3) {
                const uint4 w = lds128(my_row0 + 2 * L::TILE_BYTES + i * ROW_PITCH);
                w2[0] = w.x; w2[1] = w.y; w2[2] = w.z; w2[3] = w.w;
              }
              const uint32_t g[4] = {v.x, v.y, v.z, v.w};
              if constexpr (NOUT == 2) {
                // Both outputs from one evaluation of act and act': d gate kept
                // in y, d up parked in the lane's own gate / up bytes (which no
                // other lane reads) for the second pass.
                float yu[8];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                  float2 dg, du;
                  dgated_pair<ACT>(make_float2(bf16_lo(g[p]), bf16_hi(g[p])),
                                   make_float2(bf16_lo(u[p]), bf16_hi(u[p])),
                                   make_float2(bf16_lo(w2[p]), bf16_hi(w2[p])), dg, du);
                  y[i][2 * p] = dg.x;
                  y[i][2 * p + 1] = dg.y;
                  yu[2 * p] = du.x;
                  yu[2 * p + 1] = du.y;
                }
                sts128(my_row0 + L::TILE_BYTES + i * ROW_PITCH, __float_as_uint(yu[0]),
                       __float_as_uint(yu[1]), __float_as_uint(yu[2]), __float_as_uint(yu[3]));
                sts128(my_row0 + 2 * L::TILE_BYTES + i * ROW_PITCH, __float_as_uint(yu[4]),
                       __float_as_uint(yu[5]), __float_as_uint(yu[6]), __float_as_uint(yu[7]));
              } else {
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                  const float2 v = act_pair<ACT>(make_float2(bf16_lo(g[p]), bf16_hi(g[p])),
                                                 make_float2(bf16_lo(u[p]), bf16_hi(u[p])),
                                                 make_float2(bf16_lo(w2[p]), bf16_hi(w2[p])), t);
                  y[i][2 * p] = v.x;
                  y[i][2 * p + 1] = v.y;
                }
              }
            }
          }
          // Largest magnitudes of the lane's rows and columns: float max on
          // |y| (the absolute value is an operand modifier, no instruction of
          // its own), three-input max trees (four instructions per eight
          // values); non-negative floats order as their bits.
          auto max8 = [](float a0, float a1, float a2, float a3, float a4, float a5, float a6,
                         float a7) {
            return fmax3(fmax3(fabsf(a0), fabsf(a1), fabsf(a2)), fmax3(fabsf(a3), fabsf(a4), fabsf(a5)),
                         fmaxf(fabsf(a6), fabsf(a7)));
          };
          uint32_t cmx[8], rmx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            rmx[i] = __float_as_uint(max8(y[i][0], y[i][1], y[i][2], y[i][3], y[i][4], y[i][5],
                                          y[i][6], y[i][7]));
#pragma unroll
          for (int jc = 0; jc < 8; ++jc)
            cmx[jc] = __float_as_uint(max8(y[0][jc], y[1][jc], y[2][jc], y[3][jc], y[4][jc],
                                           y[5][jc], y[6][jc], y[7][jc]));
#pragma unroll
          for (int q = 0; q < 4; ++q)
            re[q] = f32_scale_exponent(rmx[2 * q], ceil_f32) |
                    (f32_scale_exponent(rmx[2 * q + 1], ceil_f32) << 16);
#pragma unroll
          for (int p = 0; p < 4; ++p)
            ce[p] = f32_scale_exponent(cmx[2 * p], ceil_f32) |
                    (f32_scale_exponent(cmx[2 * p + 1], ceil_f32) << 16);
        }
      }
      // Column maxima over the warp's 16 rows, published for the partner warp
      // that holds the other 16 rows of the same 32-row block.
#pragma unroll
      for (int p = 0; p < 4; ++p) ce[p] = vmax_u16x2(ce[p], __shfl_xor_sync(0xFFFFFFFFu, ce[p], 16));
      const uint32_t xch = sbase + L::OFF_XCH + (warp * 16 + c) * 16;
      if (COL && h == 0) sts128(xch, ce[0], ce[1], ce[2], ce[3]);

      // ---- barrier A: the slot has been read by every warp, the colwise
      // staging is free (thread 0 waited for the previous store), the column
      // maxima are published, and every thread knows whether the copy landed.
      fence_proxy_async_smem();
      if ((COL || (ROW && L::ROW_TMA)) && tid == 0) bulk_wait_read<QBUF - 1>();
      if (__syncthreads_or(!ok)) {
        // A copy never landed: record it, let the other copies in flight and
        // the pending stores finish (bounded), and stop without more output.
        if (tid == 0) {
          if (a.dev_err) atomicOr(a.dev_err, 1u);
          // Copies issued so far: steps below j + STAGES (paired issue: one
          // fewer before an odd step's pair).
          const int issued = j + STAGES - ((MXQ_LOAD_PAIR && STAGES % 2 == 0) ? (j & 1) : 0);
          for (int jj = j + 1; jj < issued && jj < count; ++jj)
            mbar_wait_bounded(bar0 + 8 * (jj % STAGES), (jj / STAGES) & 1, a.timeout_ns);
          bulk_wait_all();
        }
        return;
      }
      if (tid == 0 && t == NOUT - 1) {
        if constexpr (MXQ_LOAD_PAIR && STAGES % 2 == 0) {
          // Two slots at a time: the copies of consecutive steps leave together.
          if (j & 1) {
            if (j + STAGES - 1 < count) issue_load(j + STAGES - 1);
            if (j + STAGES < count) issue_load(j + STAGES);
          }
        } else if (j + STAGES < count) {
          issue_load(j + STAGES);
        }
      }

      // ---- complete the block maxima --------------------------------------
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        re[q] = vmax_u16x2(re[q], __shfl_xor_sync(0xFFFFFFFFu, re[q], 1));
        re[q] = vmax_u16x2(re[q], __shfl_xor_sync(0xFFFFFFFFu, re[q], 2));
      }
      if constexpr (COL) {
        const uint4 other = lds128(sbase + L::OFF_XCH + ((warp ^ 1) * 16 + c) * 16);
        ce[0] = vmax_u16x2(ce[0], other.x);
        ce[1] = vmax_u16x2(ce[1], other.y);
        ce[2] = vmax_u16x2(ce[2], other.z);
        ce[3] = vmax_u16x2(ce[3], other.w);
      }

      const int col0 = tk * MX_TILE_K + c * 8;            // first column of this lane
      const bool col_ok = col0 < a.kin;
      const int obase = t * a.out_half;                   // output column of input column 0
      const int row0 = band * BAND + 16 * warp + 8 * h;   // first row of this lane
      const bool row_ok = row0 < a.M;
      const int slot = tk & 7;                            // rowwise scale gathering slot

      // Values of row i, columns 2p and 2p+1 as an fp32 pair.
      auto pair_at = [&](int i, int p) -> float2 {
        if constexpr (ACT == ACT_NONE) {
          return make_float2(bf16_lo(xr[i][p]), bf16_hi(xr[i][p]));
        } else {
          return make_float2(y[i][2 * p], y[i][2 * p + 1]);
        }
      };

      // ---- rowwise: codes to global (or staging), scale bytes to staging ----
      if constexpr (ROW) {
        uint32_t rc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) rc[q] = e8m0_pair(re[q]);
        uint8_t* qrow = a.q_row + static_cast<size_t>(row0) * a.K + obase + col0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float inv = inv_scale_from_e8m0(half16(rc[i >> 1], i & 1));
          const float2 iv = make_float2(inv, inv);
          uint32_t w[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float2 v = mul_f32x2(pair_at(i, p), iv);
            w[p] = cvt_e4m3x2(v.x, v.y);
          }
          if constexpr (L::ROW_TMA) {
            // Staging [BAND rows][128 B], 16-byte chunk index xor-ed with the
            // row modulo 8 (the store map's 128-byte swizzle).
            const int rl = 16 * warp + 8 * h + i;
            sts64(sbase + L::OFF_QROW + rl * 128 + ((((c >> 1) ^ (rl & 7)) << 4) | (8 * (c & 1))),
                  w[0] | (w[1] << 16), w[2] | (w[3] << 16));
          } else if (col_ok && row_ok) {
#if MXQ_QROW_CS
            stg64_cs(qrow + static_cast<size_t>(i) * a.K, w[0] | (w[1] << 16), w[2] | (w[3] << 16));
#else
            stg64(qrow + static_cast<size_t>(i) * a.K, w[0] | (w[1] << 16), w[2] | (w[3] << 16));
#endif
          }
        }
        // Lane (h, c) holds block c/4's codes for its 8 rows; it stages rows
        // r and r + 4 (r = c & 3) into [BAND rows][8 slots][4 blocks].
        const int r = c & 3, b = c >> 2;
        const uint32_t rs =
            sbase + L::OFF_RSC + ((t * GROUP + pos.bi) * BAND + 16 * warp + 8 * h + r) * 32 +
            slot * 4 + b;
        const int sh = 16 * (r & 1);
        sts8(rs, ((r >> 1 ? rc[1] : rc[0]) >> sh) & 0xFFu);
        sts8(rs + 4 * 32, ((r >> 1 ? rc[3] : rc[2]) >> sh) & 0xFFu);
      }

      // ---- colwise: codes and scale bytes to staging -------------------------
      if constexpr (COL) {
        uint32_t cc[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) cc[p] = e8m0_pair(ce[p]);
        // Staging half (warp / 8) holds m = 128 * half + 0..127 as
        // [k % 8][k / 8][128 m], the 16-byte chunk index xor-ed with (k / 8) % 8
        // (the 128-byte swizzle of the store's tensor map).  The lane's 8 rows
        // are the h-th 8-byte half of chunk (warp % 8).
        const uint32_t qs = sbase + L::OFF_QCOL + (j % QBUF) * L::QCOL_BUF +
                            (warp >> 3) * L::QCOL_HALF + c * 128 +
                            (((warp & 7) ^ (c & 7)) << 4) + 8 * h;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float2 iv = make_float2(inv_scale_from_e8m0(half16(cc[p], 0)),
                                        inv_scale_from_e8m0(half16(cc[p], 1)));
          uint32_t we[4], wo[4];   // codes of columns 2p (even) and 2p+1 (odd), two rows each
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            const float2 r0 = mul_f32x2(pair_at(i, p), iv);
            const float2 r1 = mul_f32x2(pair_at(i + 1, p), iv);
            we[i / 2] = cvt_e4m3x2(r0.x, r1.x);
            wo[i / 2] = cvt_e4m3x2(r0.y, r1.y);
          }
          sts64(qs + (2 * p) * 2048, we[0] | (we[1] << 16), we[2] | (we[3] << 16));
          sts64(qs + (2 * p + 1) * 2048, wo[0] | (wo[1] << 16), wo[2] | (wo[3] << 16));
        }
        // Scale bytes of block (band bi, warp / 2); both warps of a block hold
        // the same codes, the even one writes them (h = 0: columns 0-3, h = 1:
        // columns 4-7 of the lane's chunk).
        if ((warp & 1) == 0) {
          const int blk = pos.bi * L::BPB + (warp >> 1);
          if constexpr (L::CSC_BY_COL) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const uint32_t pair = h ? cc[2 + (jj >> 1)] : cc[jj >> 1];
              sts8(sbase + L::OFF_CSC + L::csc(blk, c * 8 + 4 * h + jj),
                   (pair >> (16 * (jj & 1))) & 0xFFu);
            }
          } else {
            sts32(sbase + L::OFF_CSC + L::csc(blk, c * 8 + 4 * h),
                  h ? prmt(cc[2], cc[3], 0x6420) : prmt(cc[0], cc[1], 0x6420));
          }
        }
      }

      // ---- dbias: column sums of the warp's 16 rows, pairwise ----------------
      if constexpr (DBIAS) {
        // Columns 2p and 2p + 1 together (add.rn.f32x2: two independent fp32
        // sums, the same pairwise order per column).
        float s16[8];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          float2 v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = pair_at(i, p);
#pragma unroll
          for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) v[i] = add_f32x2(v[i], v[i + w]);
          const float2 o = make_float2(__shfl_xor_sync(0xFFFFFFFFu, v[0].x, 16),
                                       __shfl_xor_sync(0xFFFFFFFFu, v[0].y, 16));
          const float2 t = add_f32x2(v[0], o);
          s16[2 * p] = t.x;
          s16[2 * p + 1] = t.y;
        }
        // Two 16-byte stores per lane, 16 lanes side by side (no conflicts).
        if (h == 0) {
          const uint32_t db = sbase + L::OFF_DB + (warp * MX_TILE_K + 4 * c) * 4;
          sts128(db, __float_as_uint(s16[0]), __float_as_uint(s16[1]), __float_as_uint(s16[2]),
                 __float_as_uint(s16[3]));
          sts128(db + 64 * 4, __float_as_uint(s16[4]), __float_as_uint(s16[5]),
                 __float_as_uint(s16[6]), __float_as_uint(s16[7]));
        }
      }

      // ---- barrier B: the band's staging is complete -------------------------
      fence_proxy_async_smem();
      bar_sync_cta(THREADS);

      if (tid == 0 && (COL || (ROW && L::ROW_TMA))) {
        if constexpr (COL) {
#pragma unroll
          for (int half = 0; half < L::QCOL_HALVES; ++half)
#if MXQ_QCOL_POLICY
            tma_store_3d_hint(t == 0 ? &tmap_qcol : &tmap_qcol2,
                              sbase + L::OFF_QCOL + (j % QBUF) * L::QCOL_BUF + half * L::QCOL_HALF,
                              band * BAND + 128 * half, tk * (MX_TILE_K / 8), 0,
                              MXQ_QCOL_POLICY == 1 ? l2_policy_evict_first()
                              : MXQ_QCOL_POLICY == 2 ? l2_policy_evict_last()
                                                     : l2_policy_evict_normal());
#else
            tma_store_3d(t == 0 ? &tmap_qcol : &tmap_qcol2,
                         sbase + L::OFF_QCOL + (j % QBUF) * L::QCOL_BUF + half * L::QCOL_HALF,
                         band * BAND + 128 * half, tk * (MX_TILE_K / 8), 0);
#endif
        }
        if constexpr (ROW && L::ROW_TMA)
          tma_store_2d(t == 0 ? &tmap_qrow : &tmap_qrow2, sbase + L::OFF_QROW, tk * MX_TILE_K,
                       band * BAND);
        bulk_commit();
      }
      if constexpr (COL) {
        // Colwise scale bytes, once the group's last band (or this CTA's last
        // step) is staged: one run of up to GROUP * BAND / 32 blocks per column.
        if (pos.bi + 1 == pos.nb || j + 1 == count) {
          constexpr int NB = GROUP * L::BPB;
          constexpr int CH = NB < 16 ? NB : 16;               // bytes per store
          const int fb = (pos.g == p0.g && tk == p0.tk) ? p0.bi : 0;   // first band staged
          const int mb0 = (pos.g * GROUP + fb) * L::BPB;     // its first block along m
          const int nblk = min((pos.bi + 1 - fb) * L::BPB, nmb - mb0);
          if constexpr (MXQ_TILED_SCALES) {
            // Tiled layout: band bb's 4 blocks of the step's 128 columns are
            // the 128 x 4 tile (k / 128, band); lane L writes its 16 bytes,
            // columns L, L + 32, L + 64, L + 96 (4 blocks each).
            static_assert(L::BPB == 4, "one 128 x 4 tile per band and step");
            const int tiles_m = (nmb + 3) / 4;
            const int ktile = (obase >> 7) + tk;
            for (int it = tid; it < (pos.bi + 1 - fb) * 32; it += THREADS) {
              const int bb = fb + (it >> 5), ln = it & 31;
              uint32_t w[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int kc = ln + 32 * q;
                if constexpr (L::CSC_BY_COL) {
                  w[q] = lds32(sbase + L::OFF_CSC + L::csc(0, kc));
                } else {
                  w[q] = 0u;
#pragma unroll
                  for (int cb = 0; cb < 4; ++cb)
                    w[q] |= ld_shared_u8(sbase + L::OFF_CSC + L::csc(bb * 4 + cb, kc)) << (8 * cb);
                }
              }
              uint8_t* dst = a.s_col +
                             (static_cast<size_t>(ktile) * tiles_m + pos.g * GROUP + bb) * 512 + 16 * ln;
              stg128(dst, w[0], w[1], w[2], w[3]);
            }
          } else if (nblk == NB && (nmb % CH) == 0 && (a.scol_ld % CH) == 0) {
            // Item i = (chunk, column); warp w takes items w * IPW .. + IPW - 1.
            constexpr int ITEMS = MX_TILE_K * (NB / CH);
            constexpr int IPW = ITEMS / WARPS;
            static_assert(ITEMS % WARPS == 0 && IPW <= 32, "one item per lane");
            if (lane < IPW) {
              const int i = warp * IPW + lane;
              const int kc = i % MX_TILE_K, ch = i / MX_TILE_K;
              const int k = tk * MX_TILE_K + kc;
              uint32_t w[4] = {0u, 0u, 0u, 0u};
              if constexpr (L::CSC_BY_COL) {
                w[0] = lds32(sbase + L::OFF_CSC + L::csc(0, kc));
              } else {
#pragma unroll
                for (int bb = 0; bb < CH; ++bb)
                  w[bb >> 2] |= ld_shared_u8(sbase + L::OFF_CSC + L::csc(ch * CH + bb, kc))
                                << (8 * (bb & 3));
              }
              uint8_t* dst = a.s_col + static_cast<size_t>(obase + k) * a.scol_ld + mb0 + ch * CH;
              if (k < a.kin) {
                // Evict-last: a run is part of a 32-byte sector that other
                // CTAs complete later; kept in L2 until then, the sector is
                // written back whole (plain stores: 181.8 -> 176.9 us for
                // the 16384^2 rowwise + colwise cast, measured on GB300).
                if (CH == 16) stg128_hint(dst, w[0], w[1], w[2], w[3], csc_policy);
                else if (CH == 8) stg64_hint(dst, w[0], w[1], csc_policy);
                else stg32_hint(dst, w[0], csc_policy);
              }
            }
          } else {
            for (int kc = tid; kc < MX_TILE_K; kc += THREADS) {
              const int k = tk * MX_TILE_K + kc;
              if (k >= a.kin) continue;
              uint8_t* dst = a.s_col + static_cast<size_t>(obase + k) * a.scol_ld + mb0;
              for (int bb = 0; bb < nblk; ++bb)
                stg8(dst + bb, ld_shared_u8(sbase + L::OFF_CSC + L::csc(fb * L::BPB + bb, kc)));
            }
          }
        }
      }

      if constexpr (ROW) {
        // This band's next step in this CTA, if any, is j + nb.
        const bool flush = (slot == 7) || (tk + 1 == a.tiles_k) || (j + pos.nb >= count);
        if constexpr (MXQ_TILED_SCALES) {
          // Tiled layout: the step's 4 blocks of the band's 128 rows are the
          // 128 x 4 tile (band, column / 128), written every step by one warp:
          // lane L holds rows L, L + 32, L + 64, L + 96 (4 blocks each).
          if (warp == WARPS - 1) {
            const int tiles_k = (nkb + 3) / 4;
            const uint32_t src = sbase + L::OFF_RSC + ((t * GROUP + pos.bi) * BAND + lane) * 32 + slot * 4;
            uint8_t* dst = a.s_row +
                           (static_cast<size_t>(band) * tiles_k + (obase >> 7) + tk) * 512 + 16 * lane;
            stg128(dst, lds32(src), lds32(src + 32 * 32), lds32(src + 64 * 32), lds32(src + 96 * 32));
          }
        } else if (flush) {
          // Rowwise scale bytes of steps rsc_first..slot of this group of eight
          // (the CTA's first step for this band may fall inside the group):
          // one 32-byte sector per row when all eight steps are present,
          // written by two neighbouring threads in one instruction (16 bytes
          // each) so that the sector leaves as one request.
          const int first_tk = (pos.g == p0.g) ? p0.tk + (pos.bi < p0.bi ? 1 : 0) : 0;
          const int rsc_first = first_tk > (tk & ~7) ? (first_tk & 7) : 0;
          const int kb0 = (tk - slot) * 4;   // first k-block of the group
          // Two 16-byte halves: every row start must be 16-byte aligned.
          const bool full = rsc_first == 0 && slot == 7 && ((nkb | (obase >> 5)) & 15) == 0;
          if (full) {
            for (int it = tid; it < 2 * BAND; it += THREADS) {
              const int rr = it >> 1, half = it & 1;
              const int row = band * BAND + rr;
              if (row >= a.M) continue;
              uint8_t* dst = a.s_row + static_cast<size_t>(row) * nkb + (obase >> 5) + kb0;
              const uint32_t src = sbase + L::OFF_RSC + ((t * GROUP + pos.bi) * BAND + rr) * 32;
              const uint4 v = lds128(src + 16 * half);
              stg128(dst + 16 * half, v.x, v.y, v.z, v.w);
            }
          } else {
            // A partial group: eight neighbouring threads per row, thread w
            // writing the 4 bytes of step slot w when the group has them,
            // so that the row's run leaves as one request (a step past the
            // last valid column has fewer bytes).
            const int b_end = (a.kin >> 5) - kb0;   // valid scale bytes from kb0 on
            for (int it = tid; it < 8 * BAND; it += THREADS) {
              const int rr = it >> 3, w = it & 7;
              const int row = band * BAND + rr;
              if (row >= a.M || w < rsc_first || w > slot || 4 * w >= b_end) continue;
              uint8_t* dst = a.s_row + static_cast<size_t>(row) * nkb + (obase >> 5) + kb0 + 4 * w;
              const uint32_t src =
                  sbase + L::OFF_RSC + ((t * GROUP + pos.bi) * BAND + rr) * 32 + 4 * w;
              if (4 * w + 4 <= b_end && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
                stg32(dst, lds32(src));
              } else {
                for (int bb = 0; bb < 4 && 4 * w + bb < b_end; ++bb)
                  stg8(dst + bb, ld_shared_u8(src + bb));
              }
            }
          }
        }
      }

      if constexpr (DBIAS) {
        // The band's sum of each column: pairwise over the warps' 16-row sums;
        // warp w adds up 128 / WARPS columns.
        constexpr int COLS_PER_WARP = MX_TILE_K / WARPS;
        if (lane < COLS_PER_WARP) {
          const int kc = warp * COLS_PER_WARP + lane;
          const int k = tk * MX_TILE_K + kc;
          const float* db = reinterpret_cast<const float*>(smem + L::OFF_DB) +
                            ((kc & 7) >> 2) * 64 + 4 * (kc >> 3) + (kc & 3);
          float v[WARPS];
#pragma unroll
          for (int w = 0; w < WARPS; ++w) v[w] = db[w * MX_TILE_K];
#pragma unroll
          for (int w = WARPS / 2; w >= 1; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) v[i] = v[i] + v[i + w];
          if (k < a.kin) a.dbias_ws[static_cast<size_t>(band) * a.K + k] = v[0];
        }
      }
    }
  }
  // The staged codes must have left shared memory before the CTA exits.
  if (tid == 0) bulk_wait_all();
}

// ---------------------------------------------------------------------------
// The plain cast (with or without dbias) as one CTA per 128 x 128 tile
// ---------------------------------------------------------------------------
//
// A persistent grid walks 152 separate address ranges at once, and on GB300
// HBM that costs bandwidth: a copy kernel of the same bytes measured about
// 12% slower persistent (one CTA per SM, contiguous ranges) than as short
// CTAs that the block scheduler hands out in address order, which keeps all
// SMs inside one narrow window of memory.  The plain cast therefore runs as
// one CTA of 4 warps per 128-row x 128-column tile, tiles numbered along K
// inside a band: the tile arrives by two TMA copies of 64 rows, the 4 warps
// take its rows in two 64-row passes (the lane layout and the arithmetic of
// mx_quantize_kernel), and five CTAs share an SM (at most 96 registers a
// thread), so one CTA's copies overlap the others' work.  The colwise
// staging reuses the first copy's buffer (36 instead of 53 KiB a CTA;
// against one copy, separate staging and four CTAs per SM, measured on
// GB300: 16384^2 162.7 -> 161.7 us, colwise only 122.8 -> 119.4 us; dbias
// 8192^2 at five CTAs per SM instead of four 51.5 -> 50.2 us).
// Rowwise codes leave
// by streaming stores from registers, colwise codes by one bulk tensor store
// of the staged tile, scale bytes as one 4-byte run per row and column (or
// one 512-byte tile each in the tiled layout).  With dbias each lane adds
// its column values in row order as they are widened, and the tile's 128
// column sums (lane pair, then the four warps in a fixed order) go to the
// band's row of the workspace for the finalize kernel (8192^2 with dbias
// 53.0 -> 52.1 us against the persistent kernel, measured on GB300).
// L2 policies of the tile kernel's stores (overridable for tuning builds):
// colwise and rowwise scale runs 0 none / 1 evict-first / 2 evict-last;
// colwise code bulk stores 0 none / 1 evict-first / 2 evict-last / 3
// evict-normal.  A scale run is 4 bytes of a 32-byte sector that the
// neighbouring tiles complete; kept with evict-last, the sector is written
// back whole.  Measured on GB300 (16384^2, median of 100 calls, warm / with
// L2 flushed before each call): rowwise runs evict-last 168.1 / 170.6 ->
// 162.8 / 164.5 us; colwise runs without a policy 167.8 -> 173.0 us,
// evict-first 172.9 us; colwise codes evict-first 169.9 us, evict-last
// 166.8 us (within run-to-run noise of the default).
#ifndef MXQ_TILE_CSC_POLICY
#define MXQ_TILE_CSC_POLICY 2
#endif
#ifndef MXQ_TILE_RSC_POLICY
#define MXQ_TILE_RSC_POLICY 2
#endif
#ifndef MXQ_TILE_QCOL_POLICY
#define MXQ_TILE_QCOL_POLICY 0
#endif
__device__ __forceinline__ uint64_t tile_policy(int which) {
  return which == 1 ? l2_policy_evict_first()
         : which == 2 ? l2_policy_evict_last() : l2_policy_evict_normal();
}

// MXQ_TILE_HALVES 1: the tile arrives as two 64-row copies, one per pass,
// and the colwise staging reuses the first copy's 16 KiB (pass 0 writes it
// only after the CTA barrier that follows its loads), so a CTA needs 36 KiB
// and MXQ_TILE_CPS CTAs share an SM; 0: one 32 KiB copy and separate
// staging, four CTAs per SM (tuning comparisons).
#ifndef MXQ_TILE_HALVES
#define MXQ_TILE_HALVES 1
#endif
#ifndef MXQ_TILE_CPS
#define MXQ_TILE_CPS 5
#endif
struct MxTileLayout {
  static constexpr int WARPS = 4;
  static constexpr int ROWS = 128;                           // rows of a tile
  static constexpr int LOADS = MXQ_TILE_HALVES ? 2 : 1;      // input copies per tile
  static constexpr int LOAD_ROWS = ROWS / LOADS;
  static constexpr int OFF_TILE = 0;                         // [128 rows][256 B] bf16
  static constexpr int OFF_QCOL = MXQ_TILE_HALVES ? 0 : ROWS * MX_TILE_K * 2;   // [k % 8][k / 8][128 m]
  static constexpr int OFF_RSC = MXQ_TILE_HALVES ? ROWS * MX_TILE_K * 2
                                                 : OFF_QCOL + ROWS * MX_TILE_K;   // [128 rows][4 blocks]
  static constexpr int OFF_CSC = OFF_RSC + ROWS * 4;            // [128 columns][4 blocks]
  static constexpr int OFF_XCH = OFF_CSC + MX_TILE_K * 4;       // [2 passes][4 warps][16][16 B]
  static constexpr int BYTES = OFF_XCH + 2 * WARPS * 16 * 16;
  static constexpr int DYNAMIC = BYTES + 1024;               // + alignment pad
};

template <int MODE, bool DBIAS>
__global__ void __launch_bounds__(MxTileLayout::WARPS * 32, MXQ_TILE_HALVES ? MXQ_TILE_CPS : 4)
MX_TILE_KERNEL(const __grid_constant__ CUtensorMap tmap_x,
               const __grid_constant__ CUtensorMap tmap_qcol, const MxArgs a) {
  using L = MxTileLayout;
  constexpr bool ROW = (MODE & MX_ROW) != 0;
  constexpr bool COL = (MODE & MX_COL) != 0;
  constexpr int THREADS = L::WARPS * 32;
  constexpr int ROW_PITCH = MX_TILE_K * 2;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[L::LOADS];

  uint8_t* smem = align_up_shared<1024>(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h = lane >> 4;
  const int c = lane & 15;
  const uint32_t bar = smem_addr(&full_bar[0]);
  const int band = static_cast<int>(blockIdx.x) / a.tiles_k;
  const int tk = static_cast<int>(blockIdx.x) - band * a.tiles_k;
  // The dbias finalize grid, launched as this grid's programmatic
  // dependent, may be scheduled once every CTA has started; it waits for
  // this grid to finish before reading the column sums.
  if constexpr (DBIAS) grid_launch_dependents();

  if (tid == 0) {
#pragma unroll
    for (int l = 0; l < L::LOADS; ++l) mbar_init(bar + 8 * l, 1);
    fence_barrier_init();
#pragma unroll
    for (int l = 0; l < L::LOADS; ++l) {
      mbar_arrive_expect_tx(bar + 8 * l, L::LOAD_ROWS * ROW_PITCH);
      tma_load_2d(sbase + L::OFF_TILE + l * L::LOAD_ROWS * ROW_PITCH, &tmap_x, tk * MX_TILE_K,
                  band * L::ROWS + l * L::LOAD_ROWS, bar + 8 * l);
    }
  }
  __syncthreads();
  bool ok = mbar_wait_bounded(bar, 0, a.timeout_ns);

  const uint32_t ceil_bf16 = a.scale_ceil ? 0x001F001Fu : 0u;
  const int col0 = tk * MX_TILE_K + c * 8;      // first column of this lane
  const bool col_ok = col0 < a.kin;
  // dbias: this lane's column sums (columns 8c + 2p, 8c + 2p + 1) over its
  // rows of both passes, added in row order as the values are widened.
  float2 dsum[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                    make_float2(0.0f, 0.0f)};

#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    if (L::LOADS == 2 && pass == 1) ok = mbar_wait_bounded(bar + 8, 0, a.timeout_ns);
    const int vw = 4 * pass + warp;             // 16-row slice of the tile, 0..7
    const uint32_t my_row0 = sbase + L::OFF_TILE + (16 * vw + 8 * h) * ROW_PITCH + c * 16;
    uint32_t xr[8][4];
    uint32_t ce[4] = {0u, 0u, 0u, 0u};
    uint32_t re[4] = {0u, 0u, 0u, 0u};
    if (ok) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = lds128(my_row0 + i * ROW_PITCH);
        xr[i][0] = v.x; xr[i][1] = v.y; xr[i][2] = v.z; xr[i][3] = v.w;
      }
      uint32_t cm[4] = {0u, 0u, 0u, 0u};
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
        re[i / 2] = bf16_scale_exponents(
            absmax_bf16x2(prmt(tt[0], tt[1], 0x5410), prmt(tt[0], tt[1], 0x7632)), ceil_bf16);
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) ce[p] = bf16_scale_exponents(cm[p], ceil_bf16);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) xr[i][0] = xr[i][1] = xr[i][2] = xr[i][3] = 0u;
    }
    // Column maxima over the warp's 16 rows, published for the partner warp
    // (the other 16 rows of the same 32-row block); one exchange buffer per
    // pass, so pass 1 never overwrites what the partner still reads.
#pragma unroll
    for (int p = 0; p < 4; ++p) ce[p] = vmax_u16x2(ce[p], __shfl_xor_sync(0xFFFFFFFFu, ce[p], 16));
    const uint32_t xch = sbase + L::OFF_XCH + ((pass * L::WARPS + warp) * 16 + c) * 16;
    if (COL && h == 0) sts128(xch, ce[0], ce[1], ce[2], ce[3]);
    if (pass < L::LOADS) {
      // After this barrier every warp has read the pass's copy (with two
      // copies, pass 0's buffer becomes the colwise staging).
      if (__syncthreads_or(!ok)) {
        // A copy never landed: record it, let the copies finish (bounded)
        // and stop.
        if (tid == 0) {
          if (a.dev_err) atomicOr(a.dev_err, 1u);
          for (int l = pass; l < L::LOADS; ++l) mbar_wait_bounded(bar + 8 * l, 0, a.timeout_ns);
        }
        return;
      }
    } else {
      bar_sync_cta(THREADS);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      re[q] = vmax_u16x2(re[q], __shfl_xor_sync(0xFFFFFFFFu, re[q], 1));
      re[q] = vmax_u16x2(re[q], __shfl_xor_sync(0xFFFFFFFFu, re[q], 2));
    }
    if constexpr (COL) {
      const uint4 other =
          lds128(sbase + L::OFF_XCH + ((pass * L::WARPS + (warp ^ 1)) * 16 + c) * 16);
      ce[0] = vmax_u16x2(ce[0], other.x);
      ce[1] = vmax_u16x2(ce[1], other.y);
      ce[2] = vmax_u16x2(ce[2], other.z);
      ce[3] = vmax_u16x2(ce[3], other.w);
    }
    const int rl = 16 * vw + 8 * h;                 // first tile row of this lane
    const int row0 = band * L::ROWS + rl;
    const bool row_ok = row0 < a.M;

    if constexpr (ROW) {
      uint32_t rc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) rc[q] = e8m0_pair(re[q]);
      uint8_t* qrow = a.q_row + static_cast<size_t>(row0) * a.K + col0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float inv = inv_scale_from_e8m0(half16(rc[i >> 1], i & 1));
        const float2 iv = make_float2(inv, inv);
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float2 xv = make_float2(bf16_lo(xr[i][p]), bf16_hi(xr[i][p]));
          if constexpr (DBIAS && !COL) dsum[p] = add_f32x2(dsum[p], xv);
          const float2 v = mul_f32x2(xv, iv);
          w[p] = cvt_e4m3x2(v.x, v.y);
        }
        if (col_ok && row_ok)
          stg64_cs(qrow + static_cast<size_t>(i) * a.K, w[0] | (w[1] << 16), w[2] | (w[3] << 16));
      }
      // Lane (h, c) holds block c / 4 of its 8 rows; it stages rows r and
      // r + 4 (r = c & 3) into [128 rows][4 blocks].
      const int r = c & 3, b = c >> 2;
      const int sh = 16 * (r & 1);
      sts8(sbase + L::OFF_RSC + (rl + r) * 4 + b, ((r >> 1 ? rc[1] : rc[0]) >> sh) & 0xFFu);
      sts8(sbase + L::OFF_RSC + (rl + r + 4) * 4 + b, ((r >> 1 ? rc[3] : rc[2]) >> sh) & 0xFFu);
    }

    if constexpr (COL) {
      uint32_t cc[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) cc[p] = e8m0_pair(ce[p]);
      // Staging [k % 8][k / 8][128 m] with the 128-byte swizzle: the lane's
      // 8 rows are the h-th 8-byte half of chunk vw of each k row.
      const uint32_t qs = sbase + L::OFF_QCOL + c * 128 + ((vw ^ (c & 7)) << 4) + 8 * h;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float2 iv = make_float2(inv_scale_from_e8m0(half16(cc[p], 0)),
                                      inv_scale_from_e8m0(half16(cc[p], 1)));
        uint32_t we[4], wo[4];
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const float2 x0 = make_float2(bf16_lo(xr[i][p]), bf16_hi(xr[i][p]));
          const float2 x1 = make_float2(bf16_lo(xr[i + 1][p]), bf16_hi(xr[i + 1][p]));
          if constexpr (DBIAS) dsum[p] = add_f32x2(add_f32x2(dsum[p], x0), x1);
          const float2 r0 = mul_f32x2(x0, iv);
          const float2 r1 = mul_f32x2(x1, iv);
          we[i / 2] = cvt_e4m3x2(r0.x, r1.x);
          wo[i / 2] = cvt_e4m3x2(r0.y, r1.y);
        }
        sts64(qs + (2 * p) * 2048, we[0] | (we[1] << 16), we[2] | (we[3] << 16));
        sts64(qs + (2 * p + 1) * 2048, wo[0] | (wo[1] << 16), wo[2] | (wo[3] << 16));
      }
      // Scale bytes of block vw / 2 of the tile: the even warp of the pair
      // writes them, [128 columns][4 blocks].
      if ((vw & 1) == 0) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const uint32_t pair = h ? cc[2 + (jj >> 1)] : cc[jj >> 1];
          sts8(sbase + L::OFF_CSC + (c * 8 + 4 * h + jj) * 4 + (vw >> 1),
               (pair >> (16 * (jj & 1))) & 0xFFu);
        }
      }
    }
  }

  // ---- the tile's staging is complete: bulk store and scale runs --------
  fence_proxy_async_smem();
  bar_sync_cta(THREADS);
  if constexpr (DBIAS) {
    // Column sums of the tile: the lane pair 16 apart (the other 8 rows of
    // each pass), then the four warps through the exchange buffer, which no
    // warp reads any more ([4 warps][128 columns] fp32), added in a fixed
    // order; one value per column of the band to the workspace.
#pragma unroll
    for (int p = 0; p < 4; ++p)
      dsum[p] = add_f32x2(dsum[p], make_float2(__shfl_xor_sync(0xFFFFFFFFu, dsum[p].x, 16),
                                               __shfl_xor_sync(0xFFFFFFFFu, dsum[p].y, 16)));
    const uint32_t db = sbase + L::OFF_XCH;
    if (h == 0) {
      sts128(db + (warp * MX_TILE_K + 8 * c) * 4, __float_as_uint(dsum[0].x),
             __float_as_uint(dsum[0].y), __float_as_uint(dsum[1].x), __float_as_uint(dsum[1].y));
      sts128(db + (warp * MX_TILE_K + 8 * c + 4) * 4, __float_as_uint(dsum[2].x),
             __float_as_uint(dsum[2].y), __float_as_uint(dsum[3].x), __float_as_uint(dsum[3].y));
    }
    bar_sync_cta(THREADS);
    const float v = (__uint_as_float(lds32(db + tid * 4)) +
                     __uint_as_float(lds32(db + (MX_TILE_K + tid) * 4))) +
                    (__uint_as_float(lds32(db + (2 * MX_TILE_K + tid) * 4)) +
                     __uint_as_float(lds32(db + (3 * MX_TILE_K + tid) * 4)));
    const int k = tk * MX_TILE_K + tid;
    if (k < a.kin) a.dbias_ws[static_cast<size_t>(band) * a.K + k] = v;
  }
  if (COL && tid == 0) {
    if (MXQ_TILE_QCOL_POLICY)
      tma_store_3d_hint(&tmap_qcol, sbase + L::OFF_QCOL, band * L::ROWS, tk * (MX_TILE_K / 8), 0,
                        tile_policy(MXQ_TILE_QCOL_POLICY));
    else
      tma_store_3d(&tmap_qcol, sbase + L::OFF_QCOL, band * L::ROWS, tk * (MX_TILE_K / 8), 0);
    bulk_commit();
  }
  const int nmb = a.M / 32;    // colwise scale bytes per column
  const int nkb = a.K / 32;    // rowwise scale bytes per row
  if constexpr (MXQ_TILED_SCALES) {
    // One 512-byte tile each: entry (r, c) at (r % 32) * 16 + (r / 32) * 4 + c;
    // lane L writes rows (columns) L, L + 32, L + 64, L + 96.
    if (ROW && warp == 0) {
      const int tiles_kb = (nkb + 3) / 4;
      const uint32_t src = sbase + L::OFF_RSC + lane * 4;
      stg128(a.s_row + (static_cast<size_t>(band) * tiles_kb + tk) * 512 + 16 * lane, lds32(src),
             lds32(src + 32 * 4), lds32(src + 64 * 4), lds32(src + 96 * 4));
    }
    if (COL && warp == 1) {
      const int tiles_mb = (nmb + 3) / 4;
      const uint32_t src = sbase + L::OFF_CSC + lane * 4;
      stg128(a.s_col + (static_cast<size_t>(tk) * tiles_mb + band) * 512 + 16 * lane, lds32(src),
             lds32(src + 32 * 4), lds32(src + 64 * 4), lds32(src + 96 * 4));
    }
  } else {
    if (ROW) {
      // row tid: blocks 4 tk .. 4 tk + 3, one 4-byte run when aligned
      const int row = band * L::ROWS + tid;
      const int nb = min(4, (a.kin >> 5) - 4 * tk);
      if (row < a.M && nb > 0) {
        uint8_t* dst = a.s_row + static_cast<size_t>(row) * nkb + 4 * tk;
        const uint32_t src = sbase + L::OFF_RSC + tid * 4;
        if (nb == 4 && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
          if (MXQ_TILE_RSC_POLICY) stg32_hint(dst, lds32(src), tile_policy(MXQ_TILE_RSC_POLICY));
          else stg32(dst, lds32(src));
        } else {
          for (int bb = 0; bb < nb; ++bb) stg8(dst + bb, ld_shared_u8(src + bb));
        }
      }
    }
    if (COL) {
      // column tid: blocks 4 band .. 4 band + 3 (fewer in the last band).
      // Evict-last: a run is part of a 32-byte sector that neighbouring
      // tiles complete, kept in L2 until the sector is whole.
      const int k = tk * MX_TILE_K + tid;
      const int nb = min(4, nmb - 4 * band);
      if (k < a.kin) {
        uint8_t* dst = a.s_col + static_cast<size_t>(k) * a.scol_ld + 4 * band;
        const uint32_t src = sbase + L::OFF_CSC + tid * 4;
        if (nb == 4 && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
          if (MXQ_TILE_CSC_POLICY) stg32_hint(dst, lds32(src), tile_policy(MXQ_TILE_CSC_POLICY));
          else stg32(dst, lds32(src));
        } else {
          for (int bb = 0; bb < nb; ++bb) stg8(dst + bb, ld_shared_u8(src + bb));
        }
      }
    }
  }
  // The staged codes must have left shared memory before the CTA exits.
  if (COL && tid == 0) bulk_wait_read<0>();
}

// dbias[k] = sum over bands of the band sums.  A block takes 64 columns with
// 256 threads: thread (g, q) adds columns 4q .. 4q + 3 (one 16-byte load
// per band) over band group g (bands g * per .. g * per + per - 1, in band
// order), and the 16 group sums are then added pairwise in a fixed tree
// (g + 8, g + 4, g + 2, g + 1) -- a fixed order, so the result does not
// depend on scheduling; all of a thread's loads are independent, so the
// pass costs about one memory latency.
constexpr int kFinalizeCols = 64;
constexpr int kFinalizeGroups = 16;
__global__ void __launch_bounds__(kFinalizeGroups * kFinalizeCols / 4)
dbias_finalize_kernel(const float* __restrict__ ws, int bands, int K, float* __restrict__ dbias) {
  __shared__ float4 part[kFinalizeGroups][kFinalizeCols / 4];
  grid_dependency_wait();   // the band sums of the quantize grid before it
  const int q = threadIdx.x % (kFinalizeCols / 4), g = threadIdx.x / (kFinalizeCols / 4);
  const int k = blockIdx.x * kFinalizeCols + 4 * q;   // K is a multiple of 32
  const int per = (bands + kFinalizeGroups - 1) / kFinalizeGroups;
  const int b0 = g * per, b1 = min(bands, b0 + per);
  float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (k < K) {
#pragma unroll 4
    for (int b = b0; b < b1; ++b) {
      const float4 v = *reinterpret_cast<const float4*>(ws + static_cast<size_t>(b) * K + k);
      sum.x += v.x;
      sum.y += v.y;
      sum.z += v.z;
      sum.w += v.w;
    }
  }
  part[g][q] = sum;
  __syncthreads();
#pragma unroll
  for (int w = kFinalizeGroups / 2; w >= 1; w >>= 1) {
    if (g < w) {
      const float4 a = part[g][q], b = part[g + w][q];
      part[g][q] = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
    }
    __syncthreads();
  }
  if (g == 0 && k < K) *reinterpret_cast<float4*>(dbias + k) = part[0][q];
}

// ---------------------------------------------------------------------------
// Launch configuration per variant
// ---------------------------------------------------------------------------

// Warps per CTA (= 16-row slices of a band), ring slots and resident CTAs
// per SM, overridable at build time for tuning sweeps.  Measured on GB300:
// the plain cast runs best with one CTA per SM and three slots (two CTAs of
// two slots each: 214 vs 196 us); GELU with two CTAs per SM of two slots
// each (108 vs 112 us: one CTA's barriers no longer stall the whole SM).
#ifndef MXQ_PLAIN_WARPS
#define MXQ_PLAIN_WARPS 8
#endif
#ifndef MXQ_PLAIN_STAGES
#define MXQ_PLAIN_STAGES 3
#endif
#ifndef MXQ_GELU_WARPS
#define MXQ_GELU_WARPS 8
#endif
#ifndef MXQ_GELU_STAGES
#define MXQ_GELU_STAGES 2
#endif
#ifndef MXQ_SWIGLU_WARPS
#define MXQ_SWIGLU_WARPS 8
#endif
#ifndef MXQ_SWIGLU_STAGES
#define MXQ_SWIGLU_STAGES 2
#endif
#ifndef MXQ_PLAIN_GROUP
#define MXQ_PLAIN_GROUP 1
#endif
#ifndef MXQ_DBIAS_STAGES
#define MXQ_DBIAS_STAGES 4   // dbias 8192^2: 60.5 us (3 slots: 63 us; 2 CTAs/SM x 2: 64.6 us)
#endif
#ifndef MXQ_DBIAS_CPS
#define MXQ_DBIAS_CPS 1
#endif
#ifndef MXQ_PLAIN_GROUP_COL
#define MXQ_PLAIN_GROUP_COL 8
#endif
#ifndef MXQ_PLAIN_QBUF
#define MXQ_PLAIN_QBUF 1
#endif
#ifndef MXQ_PLAIN_CPS
#define MXQ_PLAIN_CPS 1
#endif
#ifndef MXQ_PLAIN_CPITCH
#define MXQ_PLAIN_CPITCH 8
#endif
#ifndef MXQ_GELU_GROUP
#define MXQ_GELU_GROUP 1
#endif
#ifndef MXQ_GELU_GROUP_COL
#define MXQ_GELU_GROUP_COL 8
#endif
#ifndef MXQ_GELU_QBUF
#define MXQ_GELU_QBUF 1
#endif
#ifndef MXQ_GELU_CPS
#define MXQ_GELU_CPS 2
#endif
#ifndef MXQ_SWIGLU_GROUP
#define MXQ_SWIGLU_GROUP 1
#endif
#ifndef MXQ_SWIGLU_GROUP_COL
#define MXQ_SWIGLU_GROUP_COL 8
#endif
#ifndef MXQ_SWIGLU_QBUF
#define MXQ_SWIGLU_QBUF 1
#endif
#ifndef MXQ_SWIGLU_CPS
#define MXQ_SWIGLU_CPS 1
#endif
template <int ACT>
struct MxConfig {   // plain / dbias: band of 16 * WARPS rows
  static constexpr int WARPS = MXQ_PLAIN_WARPS;
  static constexpr int STAGES = MXQ_PLAIN_STAGES;
  static constexpr int GROUP = MXQ_PLAIN_GROUP;          // with rowwise output
  static constexpr int GROUP_COL = MXQ_PLAIN_GROUP_COL;  // colwise only
  static constexpr int QBUF = MXQ_PLAIN_QBUF;            // colwise staging buffers
  static constexpr int CPS = MXQ_PLAIN_CPS;              // resident CTAs per SM
};
template <>
struct MxConfig<ACT_GELU> {
  static constexpr int WARPS = MXQ_GELU_WARPS;
  static constexpr int STAGES = MXQ_GELU_STAGES;
  static constexpr int GROUP = MXQ_GELU_GROUP;          // with rowwise output
  static constexpr int GROUP_COL = MXQ_GELU_GROUP_COL;  // colwise only
  static constexpr int QBUF = MXQ_GELU_QBUF;            // colwise staging buffers
  static constexpr int CPS = MXQ_GELU_CPS;              // resident CTAs per SM
};
template <>
struct MxConfig<ACT_SWIGLU> {   // gate + up per slot
  static constexpr int WARPS = MXQ_SWIGLU_WARPS;
  static constexpr int STAGES = MXQ_SWIGLU_STAGES;
  static constexpr int GROUP = MXQ_SWIGLU_GROUP;          // with rowwise output
  static constexpr int GROUP_COL = MXQ_SWIGLU_GROUP_COL;  // colwise only
  static constexpr int QBUF = MXQ_SWIGLU_QBUF;            // colwise staging buffers
  static constexpr int CPS = MXQ_SWIGLU_CPS;              // resident CTAs per SM
};
// The other two-operand paths (GeGLU; grad + x of the backward fusions)
// share the SwiGLU configuration.
template <>
struct MxConfig<ACT_GEGLU> : MxConfig<ACT_SWIGLU> {};
// The single-input backward fusions (grad + x per slot): two CTAs per SM of
// one slot each (128 registers), measured on GB300 against one CTA of two
// slots: dbias_dgelu 8192x14336 141.7 -> 137.9 us.
#ifndef MXQ_DACT_STAGES
#define MXQ_DACT_STAGES 1
#endif
#ifndef MXQ_DACT_CPS
#define MXQ_DACT_CPS 2
#endif
struct MxConfigDact : MxConfig<ACT_SWIGLU> {
  static constexpr int STAGES = MXQ_DACT_STAGES;
  static constexpr int CPS = MXQ_DACT_CPS;
};
template <>
struct MxConfig<ACT_DGELU> : MxConfigDact {};
template <>
struct MxConfig<ACT_DSILU> : MxConfigDact {};
// Gated backward: grad, gate and up per slot (96 KiB), two slots, one band
// per CTA (two outputs per step).
struct MxConfigDGated {
  static constexpr int WARPS = 8;
  static constexpr int STAGES = 2;
  static constexpr int GROUP = 1;
  static constexpr int GROUP_COL = 1;
  static constexpr int QBUF = 1;
  static constexpr int CPS = 1;
};
template <>
struct MxConfig<ACT_DSWIGLU> : MxConfigDGated {};
template <>
struct MxConfig<ACT_DGEGLU> : MxConfigDGated {};

// The plain cast (no activation) as one CTA per tile (see MX_TILE_KERNEL);
// MXQ_PLAIN_PERSISTENT=1 builds keep the persistent kernel for it instead
// (tuning comparisons).
#ifndef MXQ_PLAIN_PERSISTENT
#define MXQ_PLAIN_PERSISTENT 0
#endif
// The plain cast with dbias on the tile kernel (1) or the persistent one (0).
#ifndef MXQ_DBIAS_TILES
#define MXQ_DBIAS_TILES 1
#endif

template <int MODE, bool DBIAS>
cudaError_t launch_tile_variant(const MxMaps& maps, const MxArgs& a, cudaStream_t stream) {
  using L = MxTileLayout;
  static_assert((MXQ_TILE_HALVES ? MXQ_TILE_CPS : 4) * (L::DYNAMIC + 1024) <= 228 * 1024,
                "the CTAs per SM must fit");
  static_assert(L::WARPS * 32 == MX_TILE_K && 2 * L::WARPS * 16 * 16 >= 4 * L::WARPS * MX_TILE_K,
                "dbias: one thread per column; the exchange buffer holds the warps' sums");
  auto kernel = MX_TILE_KERNEL<MODE, DBIAS>;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (configured_device != dev) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::DYNAMIC);
    if (err != cudaSuccess) return err;
    configured_device = dev;
  }
  const int64_t tiles = static_cast<int64_t>(a.tiles_m) * a.tiles_k;
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  kernel<<<static_cast<unsigned>(tiles), L::WARPS * 32, L::DYNAMIC, stream>>>(maps.x, maps.q_col,
                                                                             a);
  return cudaGetLastError();
}

template <int MODE, bool DBIAS, int ACT>
cudaError_t launch_variant(const MxMaps& maps, const MxArgs& a, int num_sms,
                           cudaStream_t stream) {
  if constexpr (ACT == ACT_NONE && !MXQ_PLAIN_PERSISTENT && (!DBIAS || MXQ_DBIAS_TILES)) {
    static_assert(16 * MxConfig<ACT_NONE>::WARPS == MxTileLayout::ROWS,
                  "the tile kernel takes the plain cast's bands (and the dbias workspace's)");
    return launch_tile_variant<MODE, DBIAS>(maps, a, stream);
  }
  constexpr int WARPS = MxConfig<ACT>::WARPS;
  constexpr bool PLAIN_DBIAS = DBIAS && ACT == ACT_NONE;   // its own ring / residency
  constexpr int STAGES = PLAIN_DBIAS ? MXQ_DBIAS_STAGES : MxConfig<ACT>::STAGES;
  // Rowwise code lines want each CTA to stay on one band along K; the
  // colwise-only cast gains from interleaving bands (longer colwise runs).
  constexpr int GROUP = (MODE & MX_ROW) ? MxConfig<ACT>::GROUP : MxConfig<ACT>::GROUP_COL;
  constexpr int QBUF = MxConfig<ACT>::QBUF;
  // Band groups (colwise-only) need more staging than two CTAs can share.
  constexpr int CPS = GROUP != 1 ? 1 : PLAIN_DBIAS ? MXQ_DBIAS_CPS : MxConfig<ACT>::CPS;
  // Column pitch of the colwise scale staging (four blocks per column).  The
  // pitch changes how the warps' store phases line up; measured on GB300,
  // 8 bytes is faster for the plain cast and 4 bytes for the fused paths.
  constexpr int CPITCH = (ACT == ACT_NONE && !DBIAS) ? MXQ_PLAIN_CPITCH : 4;
  // Rowwise codes: staged and sent by one bulk store per step, or streaming
  // stores straight from registers.  Measured on GB300 (A/B): the bulk store
  // is faster for GELU (108 -> 94 us), dbias (64.6 -> 63 us) and the
  // single-input backward (dbias_dgelu 164 -> 157 us), slower for the plain
  // cast (196 -> 210 us) and the gated forward (121 -> 123 us).
  constexpr bool RTMA = ACT == ACT_GELU || DBIAS || ACT == ACT_DGELU || ACT == ACT_DSILU ||
                        (MXQ_PLAIN_RTMA && ACT == ACT_NONE);
  using L = MxLayout<WARPS, act_operands(ACT), STAGES, GROUP, QBUF, CPITCH, act_outputs(ACT),
                     RTMA>;
  static_assert(L::DYNAMIC <= 227 * 1024, "shared memory per CTA");
  static_assert(CPS == 1 || CPS * (L::DYNAMIC + 1024) <= 228 * 1024, "CTAs per SM must fit");
  auto kernel =
      MX_KERNEL<MODE, DBIAS, ACT, WARPS, STAGES, GROUP, QBUF, CPITCH, CPS, RTMA>;

  static int configured_device = -1;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (configured_device != dev) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::DYNAMIC);
    if (err != cudaSuccess) return err;
    configured_device = dev;
  }
  const int64_t steps = static_cast<int64_t>(a.tiles_m) * a.tiles_k;
  const int64_t slots = static_cast<int64_t>(CPS) * num_sms;   // persistent CTAs
  const int grid = static_cast<int>(steps < slots ? steps : slots);
  kernel<<<grid < 1 ? 1 : grid, WARPS * 32, L::DYNAMIC, stream>>>(
      maps.x, maps.x2, maps.q_col, maps.q_col2, maps.q_row, maps.q_row2, a);
  return cudaGetLastError();
}

template <bool DBIAS, int ACT>
cudaError_t launch_mode(const MxMaps& maps, const MxArgs& a, int mode, int num_sms,
                        cudaStream_t stream) {
  switch (mode) {
    case MX_ROW: return launch_variant<MX_ROW, DBIAS, ACT>(maps, a, num_sms, stream);
    case MX_COL: return launch_variant<MX_COL, DBIAS, ACT>(maps, a, num_sms, stream);
    default: return launch_variant<MX_ROW | MX_COL, DBIAS, ACT>(maps, a, num_sms, stream);
  }
}

}  // namespace

#if MXQ_TILED_SCALES
#define MXQ_LAUNCH_NAME launch_mx_tiled
#else
#define MXQ_LAUNCH_NAME launch_mx
int mx_load_rows(int act, bool dbias) {
  (void)dbias;
  return (act == ACT_NONE && !MXQ_PLAIN_PERSISTENT && (!dbias || MXQ_DBIAS_TILES))
             ? MxTileLayout::LOAD_ROWS
             : mx_band_rows(act);
}

int mx_band_rows(int act) {
  switch (act) {
    case ACT_GELU: return 16 * MxConfig<ACT_GELU>::WARPS;
    case ACT_SWIGLU: return 16 * MxConfig<ACT_SWIGLU>::WARPS;
    case ACT_GEGLU: return 16 * MxConfig<ACT_GEGLU>::WARPS;
    case ACT_DGELU: return 16 * MxConfig<ACT_DGELU>::WARPS;
    case ACT_DSILU: return 16 * MxConfig<ACT_DSILU>::WARPS;
    case ACT_DSWIGLU: return 16 * MxConfig<ACT_DSWIGLU>::WARPS;
    case ACT_DGEGLU: return 16 * MxConfig<ACT_DGEGLU>::WARPS;
    default: return 16 * MxConfig<ACT_NONE>::WARPS;
  }
}

cudaError_t launch_dbias_finalize(const float* ws, int bands, int K, float* dbias,
                                  cudaStream_t stream) {
  // Launched as a programmatic dependent of the quantize grid just before it
  // on the stream, so its launch overlaps that grid's last steps.
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((K + kFinalizeCols - 1) / kFinalizeCols);
  cfg.blockDim = dim3(kFinalizeGroups * kFinalizeCols / 4);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, dbias_finalize_kernel, ws, bands, K, dbias);
}

#endif

cudaError_t MXQ_LAUNCH_NAME(const MxMaps& maps, const MxArgs& a, int mode, bool dbias, int act,
                      int num_sms, cudaStream_t stream) {
  if (dbias) {
    switch (act) {
      case ACT_DGELU: return launch_mode<true, ACT_DGELU>(maps, a, mode, num_sms, stream);
      case ACT_DSILU: return launch_mode<true, ACT_DSILU>(maps, a, mode, num_sms, stream);
      default: return launch_mode<true, ACT_NONE>(maps, a, mode, num_sms, stream);
    }
  }
  switch (act) {
    case ACT_GELU: return launch_mode<false, ACT_GELU>(maps, a, mode, num_sms, stream);
    case ACT_SWIGLU: return launch_mode<false, ACT_SWIGLU>(maps, a, mode, num_sms, stream);
    case ACT_GEGLU: return launch_mode<false, ACT_GEGLU>(maps, a, mode, num_sms, stream);
    case ACT_DGELU: return launch_mode<false, ACT_DGELU>(maps, a, mode, num_sms, stream);
    case ACT_DSILU: return launch_mode<false, ACT_DSILU>(maps, a, mode, num_sms, stream);
    case ACT_DSWIGLU: return launch_mode<false, ACT_DSWIGLU>(maps, a, mode, num_sms, stream);
    case ACT_DGEGLU: return launch_mode<false, ACT_DGEGLU>(maps, a, mode, num_sms, stream);
    default: return launch_mode<false, ACT_NONE>(maps, a, mode, num_sms, stream);
  }
}

}  // namespace mxq
