// mxq_host.cu -- mx_quantize_rowcol_host: the MXFP8 rowwise/colwise cast of
// a matrix in host memory, pipelined through the device in row panels.
//
// Each panel of P rows (a multiple of the kernel's 128-row band) is copied
// to the device, quantized by the same kernels as mx_quantize_rowcol, and
// its outputs are copied back: rowwise codes and scales as contiguous
// blocks, colwise codes and scales (the panel's columns of the [K][M] and
// [K][M/32] outputs) as 2-D copies straight into the host layout.  Two sets
// of device buffers alternate, and the copies in and out run on two
// library-owned streams, so panel i+1's input copy overlaps panel i's cast
// and panel i-1's output copies.  Row-major colwise scales are the
// exception: a panel's part is only P / 32 bytes of each [M/32] row, and
// copies of rows that short run far below the copy engines' rate (64-byte
// rows: 16 GB/s against 190 GB/s for 2 KiB rows, measured on GB300), so the
// panels write them into one device copy of the whole [K][M/32] matrix,
// which leaves in one contiguous copy after the last panel.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "mxq.h"
#include "mxq_internal.h"

namespace {

#ifndef MXQ_HOST_PANEL_ROWS
#define MXQ_HOST_PANEL_ROWS 2048
#endif
constexpr int64_t kPanelRows = MXQ_HOST_PANEL_ROWS;
static_assert(kPanelRows % 128 == 0, "panels of whole 128-row bands");
#ifndef MXQ_HOST_BUFFERS
#define MXQ_HOST_BUFFERS 2
#endif
constexpr int kBuffers = MXQ_HOST_BUFFERS;
constexpr int kMaxDevices = 64;

struct HostPipe {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t loaded[kBuffers] = {};   // panel input on the device
  cudaEvent_t done[kBuffers] = {};     // panel quantized
  cudaEvent_t freed[kBuffers] = {};    // panel outputs copied out (buffer reusable)
  cudaEvent_t tail = nullptr;          // the whole-matrix colwise scales copied out
  bool ready = false;
};
HostPipe g_pipes[kMaxDevices];
std::mutex g_pipe_mutex;

mxq_status pipe_on_current_device(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXQ_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return MXQ_EARCH;
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  HostPipe& p = g_pipes[dev];
  if (!p.ready) {
    const unsigned ev = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, ev) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.tail, ev) != cudaSuccess)
      return MXQ_ECUDA;
    for (int b = 0; b < kBuffers; ++b)
      if (cudaEventCreateWithFlags(&p.loaded[b], ev) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.done[b], ev) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.freed[b], ev) != cudaSuccess)
        return MXQ_ECUDA;
    p.ready = true;
  }
  *out = &p;
  return MXQ_OK;
}

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Device bytes of one panel's buffers: input, codes and scales of both
// directions, and the workspace mx_quantize_rowcol needs (none without dbias).
struct PanelLayout {
  int64_t x, q_row, s_row, q_col, s_col, bytes;
  PanelLayout(int64_t P, int64_t K) {
    x = 0;
    q_row = x + round256(P * K * 2);
    s_row = q_row + round256(P * K);
    // Scale buffers sized for the tiled layout too (128 x 4 tiles, padded).
    q_col = s_row + round256(ceil_div(P, 128) * 128 * ceil_div(K / 32, 4) * 4);
    s_col = q_col + round256(K * P);
    bytes = s_col + round256(ceil_div(K, 128) * 128 * ceil_div(P / 32, 4) * 4);
  }
};

int64_t panel_rows(int64_t M) { return M < kPanelRows ? M : kPanelRows; }

}  // namespace

namespace mxq {
size_t host_workspace_bytes(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0) return 0;
  return static_cast<size_t>(kBuffers * PanelLayout(panel_rows(M), K).bytes +
                             round256(K * (M / 32)));
}
}  // namespace mxq

extern "C" mxq_status mx_quantize_rowcol_host(const void* x, int64_t M, int64_t K, int64_t ldx,
                                              uint32_t flags, uint8_t* q_row, uint8_t* s_row,
                                              uint8_t* q_col, uint8_t* s_col, void* workspace,
                                              size_t workspace_bytes, mxq_stream_t stream) {
  if (flags & ~static_cast<uint32_t>(MXQ_ROWWISE | MXQ_COLWISE | MXQ_SCALE_RCEIL | MXQ_SCALE_SWIZZLED))
    return MXQ_EINVAL;
  if (!(flags & (MXQ_ROWWISE | MXQ_COLWISE))) return MXQ_EINVAL;
  if (M < 0 || K < 0 || ldx < K) return MXQ_ESHAPE;
  if ((M % 32) || (K % 32)) return MXQ_ESHAPE;
  if (M == 0 || K == 0) return MXQ_OK;
  if (!x) return MXQ_EINVAL;
  if ((flags & MXQ_ROWWISE) && (!q_row || !s_row)) return MXQ_EINVAL;
  if ((flags & MXQ_COLWISE) && (!q_col || !s_col)) return MXQ_EINVAL;
  if (!workspace || workspace_bytes < mxq::host_workspace_bytes(M, K)) return MXQ_EWORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MXQ_EALIGN;
  HostPipe* p = nullptr;
  mxq_status st = pipe_on_current_device(&p);
  if (st != MXQ_OK) return st;
  // The streams and events are per device: calls from several host threads
  // enqueue one after another.
  std::lock_guard<std::mutex> lock(g_pipe_mutex);

  const int64_t P = panel_rows(M);
  const PanelLayout L(P, K);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const bool row = (flags & MXQ_ROWWISE) != 0, col = (flags & MXQ_COLWISE) != 0;
  const bool tiled = (flags & MXQ_SCALE_SWIZZLED) != 0;
  const int64_t tiles_k = ceil_div(K / 32, 4);   // tile columns of the rowwise scales
  const int64_t tiles_m = ceil_div(M, 128);      // tile columns of the colwise scales
  auto cu = [](cudaError_t e) { return e == cudaSuccess ? MXQ_OK : MXQ_ECUDA; };

  // Everything below runs after the work already queued on `stream`.
  if ((st = cu(cudaEventRecord(p->start, stream))) != MXQ_OK) return st;
  if ((st = cu(cudaStreamWaitEvent(p->h2d, p->start, 0))) != MXQ_OK) return st;
  if ((st = cu(cudaStreamWaitEvent(p->d2h, p->start, 0))) != MXQ_OK) return st;

  // Row-major colwise scales of the whole matrix, [K][M/32], after the panel buffers.
  const bool whole_scol = col && !tiled;
  uint8_t* scol_all = ws + kBuffers * L.bytes;

  const int64_t panels = (M + P - 1) / P;
  for (int64_t i = 0; i < panels; ++i) {
    const int b = static_cast<int>(i % kBuffers);
    uint8_t* buf = ws + b * L.bytes;
    const int64_t m0 = i * P;
    const int64_t rows = (M - m0) < P ? (M - m0) : P;
    // Input: wait until the buffer's previous panel has been copied out.
    if (i >= kBuffers && (st = cu(cudaStreamWaitEvent(p->h2d, p->freed[b], 0))) != MXQ_OK)
      return st;
    st = cu(cudaMemcpy2DAsync(buf + L.x, K * 2, static_cast<const uint8_t*>(x) + m0 * ldx * 2,
                              ldx * 2, K * 2, rows, cudaMemcpyHostToDevice, p->h2d));
    if (st != MXQ_OK) return st;
    if ((st = cu(cudaEventRecord(p->loaded[b], p->h2d))) != MXQ_OK) return st;
    // Cast on the caller's stream.
    if ((st = cu(cudaStreamWaitEvent(stream, p->loaded[b], 0))) != MXQ_OK) return st;
    uint8_t* scol_dev = whole_scol ? scol_all + m0 / 32 : (col ? buf + L.s_col : nullptr);
    st = mxq::rowcol_panel(buf + L.x, rows, K, K, flags, row ? buf + L.q_row : nullptr,
                           row ? buf + L.s_row : nullptr, col ? buf + L.q_col : nullptr, scol_dev,
                           whole_scol ? M / 32 : rows / 32, nullptr, nullptr, 0, nullptr, stream);
    if (st != MXQ_OK) return st;
    if ((st = cu(cudaEventRecord(p->done[b], stream))) != MXQ_OK) return st;
    // Outputs back: rows contiguous, columns as 2-D copies into [K][M].
    if ((st = cu(cudaStreamWaitEvent(p->d2h, p->done[b], 0))) != MXQ_OK) return st;
    if (row) {
      st = cu(cudaMemcpyAsync(q_row + m0 * K, buf + L.q_row, rows * K, cudaMemcpyDeviceToHost,
                              p->d2h));
      // Tiled rowwise scales: the panel's tile rows are contiguous in both.
      if (st == MXQ_OK)
        st = tiled ? cu(cudaMemcpyAsync(s_row + (m0 / 128) * tiles_k * 512, buf + L.s_row,
                                        ceil_div(rows, 128) * tiles_k * 512,
                                        cudaMemcpyDeviceToHost, p->d2h))
                   : cu(cudaMemcpyAsync(s_row + m0 * (K / 32), buf + L.s_row, rows * (K / 32),
                                        cudaMemcpyDeviceToHost, p->d2h));
      if (st != MXQ_OK) return st;
    }
    if (col) {
      st = cu(cudaMemcpy2DAsync(q_col + m0, M, buf + L.q_col, rows, rows, K,
                                cudaMemcpyDeviceToHost, p->d2h));
      // Tiled colwise scales: the panel's tiles of every tile row (row-major
      // ones leave with the whole matrix, below).
      if (st == MXQ_OK && tiled)
        st = cu(cudaMemcpy2DAsync(s_col + (m0 / 128) * 512, tiles_m * 512, buf + L.s_col,
                                  ceil_div(rows, 128) * 512, ceil_div(rows, 128) * 512,
                                  ceil_div(K, 128), cudaMemcpyDeviceToHost, p->d2h));
      if (st != MXQ_OK) return st;
    }
    if ((st = cu(cudaEventRecord(p->freed[b], p->d2h))) != MXQ_OK) return st;
  }
  // The whole-matrix colwise scales, once the last panel is cast (the d2h
  // stream waited for it above; every earlier cast precedes it on `stream`).
  if (whole_scol) {
    if ((st = cu(cudaMemcpyAsync(s_col, scol_all, K * (M / 32), cudaMemcpyDeviceToHost, p->d2h))) !=
        MXQ_OK)
      return st;
    if ((st = cu(cudaEventRecord(p->tail, p->d2h))) != MXQ_OK) return st;
    if ((st = cu(cudaStreamWaitEvent(stream, p->tail, 0))) != MXQ_OK) return st;
  }
  // The caller's stream continues once the last outputs are on the host.
  for (int b = 0; b < kBuffers && b < panels; ++b)
    if ((st = cu(cudaStreamWaitEvent(stream, p->freed[(panels - 1 - b) % kBuffers], 0))) != MXQ_OK)
      return st;
  return MXQ_OK;
}
