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
// Layout of the work (same principles as the MXFP8 kernel: every output
// leaves in whole lines or sectors, because the write side costs by L2
// request, not by byte):
//  * One CTA (8 warps, one CTA per SM) walks a contiguous range of steps; a
//    step is a band of 256 rows x 64 columns (32 KiB of bf16) from a 3-slot
//    TMA ring.  Steps run along K inside a band.
//  * Warp w owns rows 32w..32w+31; lane (h, c) = (lane / 8, lane % 8) owns
//    rows 8h..8h+7 and columns 8c..8c+7 of those (eight conflict-free
//    16-byte shared loads).  A 1x16 row block spans lanes c = 2b, 2b+1 and a
//    16x1 transposed block spans lanes h = 2g, 2g+1: one xor shuffle each.
//  * Block scales come from a per-CTA table (NvScaleTables): both lanes of a
//    pair look up all eight blocks they multiply (a clamp and one shared
//    load each, cheaper than swapping reciprocals by shuffle), and each
//    stages the codes of its four.  A 16x16 block spans the four lanes (h
//    pair) x (c pair): its amax takes the xor-1 and xor-8 shuffles and every
//    lane looks its one scale up.  The table holds the scale arithmetic,
//    IEEE fp32 with explicit rounding intrinsics in the fixed order
//    (b / 6) / G -> E4M3 -> value * G -> 1 / d; each element then
//    takes one multiply by that reciprocal (two per mul.rn.f32x2; no
//    per-element division, as in torchao PR #12 "Multiply with inverse
//    scale in loop instead of dividing", rationale) and
//    cvt.rn.satfinite.e2m1x2.f32.
//  * Transposed codes of a step (64 k-rows x 128 bytes) leave through one
//    3-D TMA store over [K][M/2] seen as [k % 8][k / 8][m / 2] with 128-byte
//    swizzle; rowwise codes of four steps (256 rows x 128 bytes) leave
//    through one 3-D TMA store over [M][K/2] seen as [m % 8][m / 8][k / 2].
//    Both layouts keep the shared-memory stores free of bank conflicts.
//  * Rowwise scale bytes of eight steps are gathered into one 32-byte
//    sector per row; transposed scale bytes leave as 16 bytes per column
//    per step.  The partial groups at the ends of a CTA's range leave in
//    whole sectors too (codes: thread pairs, 16 bytes each, one instruction
//    per sector; scales: one request per row run).

#include <cfloat>

#include "mxq_internal.h"
#include "mxq_ptx.cuh"

namespace mxq {
namespace {

#ifndef MXQ_NV_STAGES
#define MXQ_NV_STAGES 3
#endif
// L2 policy of the input copies: 0 none, 1 evict-last, 2 evict-normal.
// Measured on GB300 (2D 8192^2 / 16384x8192): none 41.7 / 75.9 us,
// evict-last 43.1 / 76.4, evict-normal 43.0 / 76.3; ring slots 2 and 4 were
// slower than 3.
#ifndef MXQ_NV_LOAD_HINT
#define MXQ_NV_LOAD_HINT 0
#endif

// Tile order after this call's own amax pass (1: last tile first, so the
// first tiles find the input the amax pass read last still in L2) and the
// amax pass's loads (0: streaming, 1: L2 only).  Measured on GB300 for
// 16384 x 8192 with the amax pass: in order 110.8 us, last first 108.2,
// L2-only loads 118.6 (last first 112.6).
#ifndef MXQ_NV_REVERSE_AFTER_AMAX
#define MXQ_NV_REVERSE_AFTER_AMAX 1
#endif
#ifndef MXQ_AMAX_LOAD
#define MXQ_AMAX_LOAD 0
#endif

constexpr int NV_WARPS = 8;
constexpr int NV_STAGES = MXQ_NV_STAGES;
constexpr int NV_BAND = 32 * NV_WARPS;            // 256 rows per step
constexpr int NV_STEP_K = 64;                     // columns per step
constexpr int NV_STAGE_BYTES = NV_BAND * NV_STEP_K * 2;          // 32 KiB
constexpr int NV_OFF_QT = NV_STAGES * NV_STAGE_BYTES;            // [8][8][128 B]
constexpr int NV_OFF_QR = NV_OFF_QT + NV_STEP_K * NV_BAND / 2;   // [8][32][128 B]
// Rowwise scale bytes [256 rows][8 slots][4 blocks], rows 36 bytes apart so
// that consecutive rows fall in different banks.
constexpr int NV_RSC_PITCH = 36;
constexpr int NV_OFF_RSC = NV_OFF_QR + NV_BAND * 128;
// Transposed scale bytes [64 cols][16 blocks]; the four 4-byte words of
// column k are rotated by (k / 8) % 4 so that the lanes storing the columns
// 8 apart use different banks.
constexpr int NV_OFF_TSC = NV_OFF_RSC + NV_BAND * NV_RSC_PITCH;
constexpr int NV_TAB_BINADES = 21;                               // scale table: binades kept
// Scale table: [21 x 128 + 2] entries of {fp32 1/d, code} (see NvScaleTables).
constexpr int NV_OFF_TAB = NV_OFF_TSC + NV_STEP_K * 16;
constexpr int NV_TAB_ENTRIES = NV_TAB_BINADES * 128 + 2;
constexpr int NV_SMEM = NV_OFF_TAB + NV_TAB_ENTRIES * 8 + 1024;   // + alignment pad

__device__ __forceinline__ void bar_sync_nv() {
  asm volatile("bar.sync 1, %0;" :: "r"(NV_WARPS * 32) : "memory");
}

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

// One bf16 magnitude of a packed pair of maxima, as its 15 magnitude bits
// (the sign bit left by max.xorsign.abs carries no meaning and is dropped).
__device__ __forceinline__ uint32_t mag16(uint32_t pair, int which) {
  return (pair >> (16 * which)) & 0x7FFFu;
}

// Scale code of a block and the reciprocal its elements are multiplied by.
// With G fixed for the tensor, both depend only on the block amax b, so they
// come from one per-CTA table filled with the exact arithmetic of
// nv_block_scale, one 8-byte entry {1/d, code} per bf16 magnitude of the
// NV_TAB_BINADES binades at and below the tensor amax, plus one entry on
// each side:
//  * below: anything smaller gives b / (6 G) below 2^-10, i.e. code 0;
//  * above (a block amax beyond the tensor amax's binade, possible only when
//    the caller's amax is smaller than the data): b > A, so b / (6 G) rounds
//    to at least 448 and saturates to code 0x7E (0 when G is 0), the result
//    of nv_block_scale for the first magnitude above the table; the code is
//    monotone in b and 1/d depends only on the code.
// The lookup is a clamp and one 8-byte shared load, without a branch.
struct NvScaleTables {
  uint32_t tab;    // shared address of entry 0 (the "below" entry)
  int base;        // magnitude bits of entry 1, minus 1
  int top;         // index of the "above" entry

  __device__ __forceinline__ void lookup(uint32_t mag, uint32_t& code, float& inv) const {
    const int idx = min(max(static_cast<int>(mag) - base, 0), top);
    const uint2 e = lds64(tab + 8 * idx);
    inv = __uint_as_float(e.x);
    code = e.y;
  }
};

// Fills this CTA's scale table (see NvScaleTables) for tensor amax A and
// G = A / 2688; the caller synchronises the CTA before the first lookup.
__device__ __forceinline__ NvScaleTables nv_build_tables(uint32_t sbase, float A, float G, int tid) {
  NvScaleTables tabs;
  tabs.tab = sbase + NV_OFF_TAB;
  const int ea = static_cast<int>((__float_as_uint(A) >> 23) & 0xFFu);
  const int lo_e = ea > NV_TAB_BINADES - 1 ? ea - (NV_TAB_BINADES - 1) : 0;
  const int lo_bits = lo_e << 7;
  const int hi_bits = (ea << 7) | 0x7F;
  tabs.base = lo_bits - 1;
  tabs.top = hi_bits - lo_bits + 2;
  for (int e = tid; e <= tabs.top; e += NV_WARPS * 32) {
    uint32_t code = 0u;
    float inv = 0.0f;
    if (e > 0) nv_block_scale(__uint_as_float(static_cast<uint32_t>(tabs.base + e) << 16), G, code, inv);
    sts64(tabs.tab + 8 * e, __float_as_uint(inv), code);
  }
  return tabs;
}

// Swizzled byte offset inside a [rows][128 B] staging block whose TMA map
// uses the 128-byte swizzle: the 16-byte chunk index is xor-ed with the
// row index modulo 8.
__device__ __forceinline__ uint32_t swz128(int row, int byte) {
  return row * 128 + ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15));
}

// Byte offset of block `blk` of column `col` in the transposed scale staging.
__device__ __forceinline__ uint32_t tsc_offset(int col, int blk) {
  return col * 16 + ((((blk >> 2) + (col >> 3)) & 3) << 2) + (blk & 3);
}

__device__ __forceinline__ uint32_t pick4(const uint32_t v[4], int i) {
  return (i & 2) ? ((i & 1) ? v[3] : v[2]) : ((i & 1) ? v[1] : v[0]);
}

// Transposed scale bytes of one step (staged as [64 columns][16 blocks],
// word j of column k rotated to (j + k / 8) % 4): 16 bytes per column; warp w
// writes columns 8w .. 8w + 7.  A run is half of a 32-byte sector whose other
// half the CTA of the next band writes: evict-last keeps it in L2 until the
// sector is whole.
__device__ __forceinline__ void nv_flush_tscales(const NvArgs& a, uint32_t sbase, int band, int tk,
                                                 int warp, int lane, uint64_t tsc_policy) {
  const int nmb = a.M / 16;
  if (lane < NV_STEP_K / NV_WARPS) {
    const int kc = warp * (NV_STEP_K / NV_WARPS) + lane;
    const int k = tk * NV_STEP_K + kc;
    const int mb0 = band * (NV_BAND / 16);
    const int nvalid = min(NV_BAND / 16, nmb - mb0);
    if (k < a.K) {
      uint8_t* dst = a.s_t + static_cast<size_t>(k) * nmb + mb0;
      const uint4 v = lds128(sbase + NV_OFF_TSC + kc * 16);
      const uint32_t rot[4] = {v.x, v.y, v.z, v.w};
      const int r = (kc >> 3) & 3;   // word j of the column is stored at (j + r) % 4
      const uint32_t wv[4] = {pick4(rot, r), pick4(rot, (r + 1) & 3), pick4(rot, (r + 2) & 3),
                              pick4(rot, (r + 3) & 3)};
      if (nvalid == 16 && (nmb & 15) == 0) {
        stg128_hint(dst, wv[0], wv[1], wv[2], wv[3], tsc_policy);
      } else {
        for (int bb = 0; bb < nvalid; ++bb) stg8(dst + bb, (wv[bb >> 2] >> (8 * (bb & 3))) & 0xFFu);
      }
    }
  }
}

// Rowwise scale bytes of steps first..slot8 of a group of eight (staged as
// [256 rows][36-byte pitch], 4 bytes per step): eight steps are one 32-byte
// sector per row, written by two neighbouring threads in one instruction (16
// bytes each) so the sector leaves as one request.
__device__ __forceinline__ void nv_flush_rscales(const NvArgs& a, uint32_t sbase, int band, int tk,
                                                 int first, int slot8, int tid) {
  const int nkb = a.K / 16;
  const int kb0 = (tk - slot8) * (NV_STEP_K / 16);
  // Two 16-byte halves: every row start must be 16-byte aligned.
  const bool full = first == 0 && slot8 == 7 && (nkb & 15) == 0;
  if (full) {
    for (int it = tid; it < 2 * NV_BAND; it += NV_WARPS * 32) {
      const int rr = it >> 1, half = it & 1;
      const int row = band * NV_BAND + rr;
      if (row >= a.M) continue;
      const uint32_t s16 = sbase + NV_OFF_RSC + rr * NV_RSC_PITCH + 16 * half;
      stg128(a.s_row + static_cast<size_t>(row) * nkb + kb0 + 16 * half, lds32(s16),
             lds32(s16 + 4), lds32(s16 + 8), lds32(s16 + 12));
    }
    return;
  }
  // A partial group: eight neighbouring threads per row, thread w writing
  // the 4 bytes of slot w when the group has them, so the row's run leaves
  // as one request.  A slot past the last column (K % 64 == 32) has 2 bytes.
  const int b_end = nkb - kb0;   // scale bytes of this group inside the row
  for (int it = tid; it < 8 * NV_BAND; it += NV_WARPS * 32) {
    const int rr = it >> 3, w = it & 7;
    const int row = band * NV_BAND + rr;
    if (row >= a.M || w < first || w > slot8 || 4 * w >= b_end) continue;
    uint8_t* dst = a.s_row + static_cast<size_t>(row) * nkb + kb0 + 4 * w;
    const uint32_t src = sbase + NV_OFF_RSC + rr * NV_RSC_PITCH + 4 * w;
    if (4 * w + 4 <= b_end && (reinterpret_cast<uintptr_t>(dst) & 3u) == 0) {
      stg32(dst, lds32(src));
    } else {
      for (int bb = 0; bb < 4 && 4 * w + bb < b_end; ++bb) stg8(dst + bb, ld_shared_u8(src + bb));
    }
  }
}

template <int MODE, bool TWO_D>
__global__ void __launch_bounds__(NV_WARPS * 32, 1)
nvfp4_quantize_kernel(const __grid_constant__ CUtensorMap tmap_x,
                      const __grid_constant__ CUtensorMap tmap_qrow,
                      const __grid_constant__ CUtensorMap tmap_qt, const NvArgs a) {
  constexpr bool ROW = (MODE & MX_ROW) != 0;
  constexpr bool COL = (MODE & MX_COL) != 0;
  constexpr int ROW_PITCH = NV_STEP_K * 2;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[NV_STAGES];

  uint8_t* smem = align_up_shared<1024>(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h = lane >> 3;   // 8-row group 0..3 of the warp's 32 rows
  const int c = lane & 7;    // 8-column chunk 0..7
  const uint32_t bar0 = smem_addr(&full_bar[0]);

  const int64_t total = static_cast<int64_t>(a.tiles_m) * a.tiles_k;
  const int t0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * total / gridDim.x);
  const int t1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * total / gridDim.x);
  const int count = t1 - t0;

  auto issue_load = [&](int j) {   // thread 0 only
    const int t = t0 + j;
    const int band = t / a.tiles_k;
    const int tk = t - band * a.tiles_k;
    const int s = j % NV_STAGES;
    mbar_arrive_expect_tx(bar0 + 8 * s, NV_STAGE_BYTES);
#if MXQ_NV_LOAD_HINT
    tma_load_2d_hint(sbase + s * NV_STAGE_BYTES, &tmap_x, tk * NV_STEP_K, band * NV_BAND,
                     bar0 + 8 * s,
                     MXQ_NV_LOAD_HINT == 2 ? l2_policy_evict_normal() : l2_policy_evict_last());
#else
    tma_load_2d(sbase + s * NV_STAGE_BYTES, &tmap_x, tk * NV_STEP_K, band * NV_BAND, bar0 + 8 * s);
#endif
  };

  if (tid == 0) {
    prefetch_tensormap(&tmap_x);
    if (ROW) prefetch_tensormap(&tmap_qrow);
    if (COL) prefetch_tensormap(&tmap_qt);
#pragma unroll
    for (int st = 0; st < NV_STAGES; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_barrier_init();
    for (int jj = 0; jj < NV_STAGES && jj < count; ++jj) issue_load(jj);
  }

  // The tensor amax, read while the first copies are in flight (after the
  // amax grid this one may depend on has completed).
  grid_dependency_wait();
  const float A = *a.amax;
  const float G = __fdiv_rn(A, 2688.0f);
  if (blockIdx.x == 0 && tid == 0) *a.global_scale = G;
  if (count <= 0) return;

  // Scale tables (see NvScaleTables).
  const NvScaleTables tabs = nv_build_tables(sbase, A, G, tid);
  __syncthreads();

  const uint64_t tsc_policy = l2_policy_evict_last();
  int rq_first = -1;          // first slot of the rowwise code group gathered
  int rs_first = -1;          // first slot of the rowwise scale group gathered

  for (int j = 0; j < count; ++j) {
    const int s = j % NV_STAGES;
    const int t = t0 + j;
    const int band = t / a.tiles_k;
    const int tk = t - band * a.tiles_k;
    const bool ok = mbar_wait_bounded(bar0 + 8 * s, (j / NV_STAGES) & 1, a.timeout_ns);

    // ---- load this lane's 8 x 8 block; magnitude maxima ---------------------
    const uint32_t my_row0 = sbase + s * NV_STAGE_BYTES + (32 * warp + 8 * h) * ROW_PITCH + c * 16;
    uint32_t xr[8][4];
    uint32_t cm[4] = {0u, 0u, 0u, 0u};   // columns 2p / 2p+1 over the lane's 8 rows
    uint32_t rm[4] = {0u, 0u, 0u, 0u};   // rows 2q / 2q+1 over the lane's 8 columns
    if (ok) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = lds128(my_row0 + i * ROW_PITCH);
        xr[i][0] = v.x; xr[i][1] = v.y; xr[i][2] = v.z; xr[i][3] = v.w;
      }
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
    }

    // ---- barrier A: slot read by all warps, code staging free ---------------
    fence_proxy_async_smem();
    if (tid == 0) bulk_wait_read<0>();
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        if (a.dev_err) atomicOr(a.dev_err, 1u);
        for (int jj = j + 1; jj < j + NV_STAGES && jj < count; ++jj)
          mbar_wait_bounded(bar0 + 8 * (jj % NV_STAGES), (jj / NV_STAGES) & 1, a.timeout_ns);
        bulk_wait_all();
      }
      return;
    }
    if (tid == 0 && j + NV_STAGES < count) issue_load(j + NV_STAGES);

    // 2D: the 16x16 block's amax over the four lanes that hold it, and its
    // one scale.
    uint32_t code2d = 0u;
    float inv2d = 0.0f;
    if constexpr (TWO_D) {
      uint32_t m2 = absmax_bf16x2(absmax_bf16x2(rm[0], rm[1]), absmax_bf16x2(rm[2], rm[3]));
      m2 = absmax_bf16x2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 1));
      m2 = absmax_bf16x2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 8));
      tabs.lookup(max(mag16(m2, 0), mag16(m2, 1)), code2d, inv2d);
    }

    // The lane's values widened to fp32 once, for both directions.
    float2 xv[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int p = 0; p < 4; ++p) xv[i][p] = make_float2(bf16_lo(xr[i][p]), bf16_hi(xr[i][p]));
    auto pair_at = [&](int i, int p) -> float2 { return xv[i][p]; };

    // ---- rowwise: block scales (split over the c pair), codes, scale bytes --
    if constexpr (ROW) {
      const int mine = c & 1;               // this lane stages the codes of rows 4*mine .. 4*mine+3
      uint32_t rcode[4];
      float rinv[8];
      if constexpr (TWO_D) {
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) rcode[tq] = code2d;
#pragma unroll
        for (int i = 0; i < 8; ++i) rinv[i] = inv2d;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          rm[q] = absmax_bf16x2(rm[q], __shfl_xor_sync(0xFFFFFFFFu, rm[q], 1));
        // Both lanes of the pair look up all eight row blocks (a lookup is
        // one clamp and one shared load); each stages the codes of its four.
        uint32_t code8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) tabs.lookup(mag16(rm[i >> 1], i & 1), code8[i], rinv[i]);
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) rcode[tq] = mine ? code8[4 + tq] : code8[tq];
      }
      // Codes of row i: 8 values -> 4 bytes at k / 2 = 4c within this step.
      const int slot4 = tk & 3;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 iv = make_float2(rinv[i], rinv[i]);
        const float2 v0 = mul_f32x2(pair_at(i, 0), iv);
        const float2 v1 = mul_f32x2(pair_at(i, 1), iv);
        const float2 v2 = mul_f32x2(pair_at(i, 2), iv);
        const float2 v3 = mul_f32x2(pair_at(i, 3), iv);
        const uint32_t w = cvt_e2m1x8(v0.x, v0.y, v1.x, v1.y, v2.x, v2.y, v3.x, v3.y);
        // staging [m % 8][m / 8][128 B]: row index i * 32 + (4 * warp + h)
        const int srow = i * 32 + 4 * warp + h;
        sts32(sbase + NV_OFF_QR + swz128(srow, slot4 * 32 + 4 * c), w);
      }
      // Scale bytes: [256 rows][8 slots][4 blocks of 16 columns].  The four
      // lanes c = mine, mine + 2, mine + 4, mine + 6 hold blocks 0..3 of the
      // same four rows; lane b = c / 2 gathers row 4 * mine + b from the
      // other three (three shuffles) and stores one 4-byte word.
      const int slot8 = tk & 7;
      const int b = c >> 1;
      uint32_t word = pick4(rcode, b) << (8 * b);
#pragma unroll
      for (int k = 1; k < 4; ++k) {
        const int src_b = (b + k) & 3;   // the lane this one reads
        const uint32_t got = __shfl_sync(0xFFFFFFFFu, pick4(rcode, (b - k) & 3),
                                         (lane & ~7) | (2 * src_b + mine));
        word |= got << (8 * src_b);
      }
      sts32(sbase + NV_OFF_RSC + (32 * warp + 8 * h + 4 * mine + b) * NV_RSC_PITCH + slot8 * 4,
            word);
    }

    // ---- transposed: block scales (split over the h pair), codes, scales ----
    if constexpr (COL) {
      const int mine = h & 1;               // this lane stages the codes of columns 4*mine .. 4*mine+3
      uint32_t tcode[4];
      float tinv[8];
      if constexpr (TWO_D) {
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) tcode[tq] = code2d;
#pragma unroll
        for (int i = 0; i < 8; ++i) tinv[i] = inv2d;
      } else {
#pragma unroll
        for (int p = 0; p < 4; ++p)
          cm[p] = absmax_bf16x2(cm[p], __shfl_xor_sync(0xFFFFFFFFu, cm[p], 8));
        // Both lanes of the pair look up all eight column blocks; each
        // stages the codes of its four.
        uint32_t code8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) tabs.lookup(mag16(cm[j >> 1], j & 1), code8[j], tinv[j]);
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) tcode[tq] = mine ? code8[4 + tq] : code8[tq];
      }
      // Codes of column jc: 8 rows -> 4 bytes at m / 2 = 16 * warp + 4h.
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const float2 iv = make_float2(tinv[2 * p], tinv[2 * p + 1]);
        float2 r[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) r[i] = mul_f32x2(pair_at(i, p), iv);
        const uint32_t we = cvt_e2m1x8(r[0].x, r[1].x, r[2].x, r[3].x, r[4].x, r[5].x, r[6].x, r[7].x);
        const uint32_t wo = cvt_e2m1x8(r[0].y, r[1].y, r[2].y, r[3].y, r[4].y, r[5].y, r[6].y, r[7].y);
        // staging [k % 8][k / 8][128 B]: row index jc * 8 + c
        sts32(sbase + NV_OFF_QT + swz128((2 * p) * 8 + c, 16 * warp + 4 * h), we);
        sts32(sbase + NV_OFF_QT + swz128((2 * p + 1) * 8 + c, 16 * warp + 4 * h), wo);
      }
      // Scale bytes: [64 columns][16 blocks of 16 rows].
#pragma unroll
      for (int tq = 0; tq < 4; ++tq)
        sts8(sbase + NV_OFF_TSC + tsc_offset(8 * c + 4 * mine + tq, 2 * warp + (h >> 1)), tcode[tq]);
    }

    // ---- barrier B: staging complete --------------------------------------
    fence_proxy_async_smem();
    bar_sync_nv();

    if constexpr (COL) {
      if (tid == 0) {
        tma_store_3d(&tmap_qt, sbase + NV_OFF_QT, band * (NV_BAND / 2), tk * (NV_STEP_K / 8), 0);
        bulk_commit();
      }
      nv_flush_tscales(a, sbase, band, tk, warp, lane, tsc_policy);
    }

    if constexpr (ROW) {
      // Rowwise codes: a group of four steps is one 256 x 128-byte TMA store;
      // a partial group (range or band edge) is written by the threads.
      const int slot4 = tk & 3;
      if (rq_first < 0) rq_first = slot4;
      const bool end = (tk + 1 == a.tiles_k) || (j + 1 == count);
      if (slot4 == 3 || end) {
        const int kbyte0 = (tk - slot4) * (NV_STEP_K / 2);   // first code byte of the group
        if (rq_first == 0 && slot4 == 3) {
          if (tid == 0) {
            tma_store_3d(&tmap_qrow, sbase + NV_OFF_QR, kbyte0, band * (NV_BAND / 8), 0);
            bulk_commit();
          }
        } else {
          // A partial group (range or band edge): slots rq_first..slot4 of
          // every row, each slot's 32 bytes written by two neighbouring
          // threads in one instruction (16 bytes each), so that it leaves as
          // one whole sector.  K is a multiple of 32, so a 16-byte half
          // (32 columns) is either wholly inside the matrix or wholly out.
          // (One 4-byte store per thread and word instead: 90.4 -> 80.5 us
          // for the 16384 x 8192 cast, measured on GB300.)
          const int nsl = slot4 + 1 - rq_first;
          for (int it = tid; it < NV_BAND * nsl * 2; it += NV_WARPS * 32) {
            const int rr = it / (2 * nsl);
            const int rem = it - rr * 2 * nsl;
            const int sl = rq_first + (rem >> 1), half = rem & 1;
            const int row = band * NV_BAND + rr;
            if (row < a.M && (tk - slot4 + sl) * NV_STEP_K + 32 * half < a.K) {
              const int srow = (rr & 7) * 32 + (rr >> 3);
              const uint4 v = lds128(sbase + NV_OFF_QR + swz128(srow, sl * 32 + 16 * half));
              stg128(a.q_row + static_cast<size_t>(row) * (a.K / 2) + kbyte0 + sl * 32 + 16 * half,
                     v.x, v.y, v.z, v.w);
            }
          }
        }
        rq_first = -1;
      }
      // Rowwise scale bytes, once per group of eight steps.
      const int slot8 = tk & 7;
      if (rs_first < 0) rs_first = slot8;
      if (slot8 == 7 || end) {
        nv_flush_rscales(a, sbase, band, tk, rs_first, slot8, tid);
        rs_first = -1;
      }
    }
  }
  if (tid == 0) bulk_wait_all();
}

// ---------------------------------------------------------------------------
// One CTA per 128 x 128 tile
// ---------------------------------------------------------------------------
//
// Short CTAs handed out in address order read and write HBM faster on GB300
// than a persistent grid, but a short CTA cannot afford the persistent
// kernel's scale table (one entry per possible block amax).  This kernel
// keeps only a 128-entry table of 1/d by scale code and decides each code
// from one multiply (NvFastScale); the rare blocks the multiply cannot decide
// take the recipe's own division sequence.  One CTA of 4 warps takes a
// 128 x 128 tile (one TMA copy) in two 64-column passes with the persistent
// kernel's lane layout (lane (h, c) of warp w: rows 32w + 8h + 0..7,
// columns 8c..8c+7 of the pass); of the eight row (column) blocks a lane
// pair multiplies by, each lane decides four and the pair swaps 1/d by
// shuffle (71.6 -> 68.2 us for 16384 x 8192 against both lanes deciding all
// eight, measured on GB300).  Codes are staged per tile and leave by one
// 3-D bulk tensor store per direction (64-byte rows, 64-byte swizzle); scale
// bytes as one 8-byte run per row and per column, evict-last (a quarter of a
// 32-byte sector that the neighbouring tiles complete).  Four CTAs share an
// SM.
constexpr int NT_WARPS = 4;
constexpr int NT_ROWS = 128;
constexpr int NT_COLS = 128;
constexpr int NT_TILE_BYTES = NT_ROWS * NT_COLS * 2;            // 32 KiB of bf16
constexpr int NT_OFF_QR = NT_TILE_BYTES;                         // [m % 8][m / 8][64 B]
constexpr int NT_OFF_QT = NT_OFF_QR + NT_ROWS * NT_COLS / 2;     // [k % 8][k / 8][64 B]
constexpr int NT_OFF_RSC = NT_OFF_QT + NT_COLS * NT_ROWS / 2;    // [128 rows][8 blocks]
constexpr int NT_OFF_TSC = NT_OFF_RSC + NT_ROWS * 8;             // [8 blocks][128 columns]
constexpr int NT_OFF_INV = NT_OFF_TSC + NT_COLS * 8;             // [128 codes] fp32 1/d
constexpr int NT_SMEM = NT_OFF_INV + 128 * 4 + 1024;             // + alignment pad
static_assert(4 * (NT_SMEM + 1024) <= 228 * 1024, "four CTAs per SM");

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
__global__ void __launch_bounds__(NT_WARPS * 32, 4)
nvfp4_tile_kernel(const __grid_constant__ CUtensorMap tmap_x,
                  const __grid_constant__ CUtensorMap tmap_qrow,
                  const __grid_constant__ CUtensorMap tmap_qt, const NvArgs a) {
  constexpr bool ROW = (MODE & MX_ROW) != 0;
  constexpr bool COL = (MODE & MX_COL) != 0;
  constexpr int ROW_PITCH = NT_COLS * 2;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar;
  uint8_t* smem = align_up_shared<1024>(smem_raw);
  const uint32_t sbase = smem_addr(smem);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h = lane >> 3;   // 8-row group 0..3 of the warp's 32 rows
  const int c = lane & 7;    // 8-column chunk 0..7 of the pass's 64 columns
  const uint32_t bar = smem_addr(&full_bar);
  const unsigned t = a.reverse ? gridDim.x - 1u - blockIdx.x : blockIdx.x;
  const int band = static_cast<int>(t / static_cast<unsigned>(a.tiles_k));
  const int tk = static_cast<int>(t) - band * a.tiles_k;

  if (tid == 0) {
    if (ROW) prefetch_tensormap(&tmap_qrow);
    if (COL) prefetch_tensormap(&tmap_qt);
    mbar_init(bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar, NT_TILE_BYTES);
    tma_load_2d(sbase, &tmap_x, tk * NT_COLS, band * NT_ROWS, bar);
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
  const bool ok = mbar_wait_bounded(bar, 0, a.timeout_ns);
  if (__syncthreads_or(!ok)) {
    // The copy never landed: record it, let it finish (bounded) and stop.
    if (tid == 0) {
      if (a.dev_err) atomicOr(a.dev_err, 1u);
      mbar_wait_bounded(bar, 0, a.timeout_ns);
    }
    return;
  }

#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    // ---- this lane's 8 x 8 block; magnitude maxima ---------------------------
    const uint32_t my_row0 = sbase + (32 * warp + 8 * h) * ROW_PITCH + (64 * pass + 8 * c) * 2;
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

    float2 xv[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int p = 0; p < 4; ++p) xv[i][p] = make_float2(bf16_lo(xr[i][p]), bf16_hi(xr[i][p]));

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
        // completed with the partner's half) and swaps 1/d with the partner.
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
        const float2 v0 = mul_f32x2(xv[i][0], iv);
        const float2 v1 = mul_f32x2(xv[i][1], iv);
        const float2 v2 = mul_f32x2(xv[i][2], iv);
        const float2 v3 = mul_f32x2(xv[i][3], iv);
        sts32(sbase + NT_OFF_QR + swz64(16 * i + 4 * warp + h, 32 * pass + 4 * c),
              cvt_e2m1x8(v0.x, v0.y, v1.x, v1.y, v2.x, v2.y, v3.x, v3.y));
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
        for (int i = 0; i < 8; ++i) r[i] = mul_f32x2(xv[i][p], iv);
        const int srow = 16 * (2 * p) + 8 * pass + c;
        sts32(sbase + NT_OFF_QT + swz64(srow, 16 * warp + 4 * h),
              cvt_e2m1x8(r[0].x, r[1].x, r[2].x, r[3].x, r[4].x, r[5].x, r[6].x, r[7].x));
        sts32(sbase + NT_OFF_QT + swz64(srow + 16, 16 * warp + 4 * h),
              cvt_e2m1x8(r[0].y, r[1].y, r[2].y, r[3].y, r[4].y, r[5].y, r[6].y, r[7].y));
      }
      // Scale bytes [block][column]: the lane's four columns are adjacent.
      sts32(sbase + NT_OFF_TSC + (2 * warp + (h >> 1)) * NT_COLS + 64 * pass + 8 * c + 4 * mine,
            tcode[0] | (tcode[1] << 8) | (tcode[2] << 16) | (tcode[3] << 24));
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
#if MXQ_AMAX_LOAD == 1
      const uint4 v = __ldcg(p + ch);
#else
      const uint4 v = __ldcs(p + ch);
#endif
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

using NvKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, NvArgs);

// One launch of an NVFP4 kernel: one persistent CTA per SM (or per step).
// Right after this call's own amax grid it is launched as that grid's
// programmatic dependent: the first input copies and the set-up overlap the
// amax grid's tail (the kernel waits for it before reading the amax).  Never
// after a caller's kernel, which may still be writing the input.
cudaError_t launch_nv_kernel(NvKernel kernel, int& configured_device, const NvMaps& maps,
                             const NvArgs& a, int num_sms, bool after_amax, cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (configured_device != dev) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, NV_SMEM);
    if (err != cudaSuccess) return err;
    configured_device = dev;
  }
  const int64_t steps = static_cast<int64_t>(a.tiles_m) * a.tiles_k;
  const int grid = static_cast<int>(steps < num_sms ? steps : num_sms);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid < 1 ? 1 : grid);
  cfg.blockDim = dim3(NV_WARPS * 32);
  cfg.dynamicSmemBytes = NV_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_amax ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, maps.x, maps.q_row, maps.q_t, a);
}

template <int MODE, bool TWO_D>
cudaError_t launch_nv_variant(const NvMaps& maps, const NvArgs& a, int num_sms, bool after_amax,
                              cudaStream_t stream) {
  static int configured_device = -1;
  return launch_nv_kernel(nvfp4_quantize_kernel<MODE, TWO_D>, configured_device, maps, a, num_sms,
                          after_amax, stream);
}

// One launch of the tile kernel: one CTA per 128 x 128 tile, in address
// order (programmatic dependent of this call's own amax grid, as above).
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
  NvArgs args = a;
  args.reverse = after_amax && MXQ_NV_REVERSE_AFTER_AMAX;
  return cudaLaunchKernelEx(&cfg, kernel, maps.x, maps.q_row, maps.q_t, args);
}

// Which kernel takes 1D and 2D blocks: the tile kernel (1) or the
// persistent kernel (0).
#ifndef MXQ_NV1D_TILES
#define MXQ_NV1D_TILES 1
#endif
#ifndef MXQ_NV2D_TILES
#define MXQ_NV2D_TILES 1
#endif

template <bool TWO_D>
cudaError_t launch_nv_mode(const NvMaps& maps, const NvArgs& a, int mode, int num_sms,
                           bool after_amax, cudaStream_t stream) {
  constexpr bool TILES = TWO_D ? MXQ_NV2D_TILES != 0 : MXQ_NV1D_TILES != 0;
  if constexpr (TILES) {
    switch (mode) {
      case MX_ROW: return launch_nv_tile_variant<MX_ROW, TWO_D>(maps, a, after_amax, stream);
      case MX_COL: return launch_nv_tile_variant<MX_COL, TWO_D>(maps, a, after_amax, stream);
      default:
        return launch_nv_tile_variant<MX_ROW | MX_COL, TWO_D>(maps, a, after_amax, stream);
    }
  } else {
    switch (mode) {
      case MX_ROW: return launch_nv_variant<MX_ROW, TWO_D>(maps, a, num_sms, after_amax, stream);
      case MX_COL: return launch_nv_variant<MX_COL, TWO_D>(maps, a, num_sms, after_amax, stream);
      default:
        return launch_nv_variant<MX_ROW | MX_COL, TWO_D>(maps, a, num_sms, after_amax, stream);
    }
  }
}

}  // namespace

NvShape nv_shape(bool two_d) {
  const bool tiles = two_d ? MXQ_NV2D_TILES != 0 : MXQ_NV1D_TILES != 0;
  return tiles ? NvShape{true, NT_ROWS, NT_COLS} : NvShape{false, NV_BAND, NV_STEP_K};
}

cudaError_t launch_nvfp4(const NvMaps& maps, const NvArgs& a, int mode, bool two_d,
                         int num_sms, bool after_amax, cudaStream_t stream) {
  return two_d ? launch_nv_mode<true>(maps, a, mode, num_sms, after_amax, stream)
               : launch_nv_mode<false>(maps, a, mode, num_sms, after_amax, stream);
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
