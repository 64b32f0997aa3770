// host_pipeline.cu -- the RMSNorm + AdaLN producer on host buffers: x read from
// and the codes and scales written to host memory, the copies inside the call.
//
// The rows are cut into chunks of chunk_rows (a multiple of 128).  Rows are
// independent and the scales of a 128-row tile are one contiguous byte range of
// the swizzled matrix, so each chunk is one producer launch on device staging
// buffers and two copies back.  Three staging slots rotate: while the caller's
// stream runs the producer on chunk i, an internal stream copies chunk i+1 in
// and another copies chunk i-1's codes and scales out (both directions of the
// host link busy at once).  Events order the three streams and guard the slots.
// The row -> frame array, when rows_per_frame is given, is written on the device
// into the workspace, so chunks need not line up with frames.
#include <mutex>

#include "../../include/h3q.h"
#include "h3q_internal.h"

namespace h3q {
namespace {

constexpr int kDepth = 3;  // staging slots: the layout of h3q_host_workspace_bytes
constexpr int kMaxContexts = 64;

// Internal streams and events of one CUDA context, created on its first host
// call and kept.  The mutex serialises the enqueueing of host calls in the
// context (they share the streams and events); the calls themselves stay
// asynchronous.  Keyed on the context's unique id, so a context the caller
// destroys and re-creates gets fresh streams and events instead of dead handles.
struct DevicePipe {
  std::mutex mu;
  unsigned long long context = 0;  // 0: slot unused (context ids start at 1)
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t loaded[kDepth] = {}, computed[kDepth] = {}, drained[kDepth] = {};
};
std::mutex g_pipes_mu;
DevicePipe g_pipes[kMaxContexts];

// The slot of the current context, claimed on its first call; nullptr once
// kMaxContexts contexts have claimed one.
DevicePipe* pipe_of(unsigned long long context) {
  std::lock_guard<std::mutex> lock(g_pipes_mu);
  for (DevicePipe& p : g_pipes)
    if (p.context == context) return &p;
  for (DevicePipe& p : g_pipes)
    if (p.context == 0) {
      p.context = context;
      return &p;
    }
  return nullptr;
}

cudaError_t init_pipe(DevicePipe& p) {
  cudaError_t err = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking);
  if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking);
  cudaEvent_t* all[2 + 3 * kDepth] = {&p.start, &p.done};
  for (int i = 0; i < kDepth; ++i) {
    all[2 + i] = &p.loaded[i];
    all[2 + kDepth + i] = &p.computed[i];
    all[2 + 2 * kDepth + i] = &p.drained[i];
  }
  for (cudaEvent_t* e : all)
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
  if (err == cudaSuccess) p.ready = true;
  return err;
}

__global__ void fill_frames_kernel(int32_t* __restrict__ frames, int64_t rows, int64_t rows_per_frame) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < rows;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    frames[i] = static_cast<int32_t>(i / rows_per_frame);
}

}  // namespace

cudaError_t launch_adaln_host(const uint16_t* x_host, int64_t rows, int64_t cols, const uint16_t* gamma,
                              const uint16_t* table, int64_t num_frames, const int32_t* row_frame,
                              int64_t rows_per_frame, float eps, const float* gsf, uint8_t* codes_host,
                              uint8_t* scales_host, uint8_t* workspace, int64_t chunk_rows,
                              cudaStream_t stream) {
  unsigned long long context = 0;
  cudaError_t err = current_context_id(&context);
  if (err != cudaSuccess) return err;
  DevicePipe* slot = pipe_of(context);
  if (slot == nullptr) return cudaErrorNotSupported;  // more contexts than slots
  DevicePipe& p = *slot;
  std::lock_guard<std::mutex> lock(p.mu);
  if (!p.ready && (err = init_pipe(p)) != cudaSuccess) return err;

  // workspace: kDepth slots of (x chunk, codes chunk, scales chunk), then frames
  uint16_t* xs[kDepth];
  uint8_t* cs[kDepth];
  uint8_t* ss[kDepth];
  uint8_t* w = workspace;
  for (int s = 0; s < kDepth; ++s) {
    xs[s] = reinterpret_cast<uint16_t*>(w);
    w += h3q_align256(chunk_rows * cols * 2);
    cs[s] = w;
    w += h3q_align256(chunk_rows * cols / 2);
    ss[s] = w;
    w += h3q_align256(chunk_rows * cols / 16);
  }
  const int32_t* frames = row_frame;

  // the call follows the work already queued on the caller's stream
  if ((err = cudaEventRecord(p.start, stream)) != cudaSuccess) return err;
  if ((err = cudaStreamWaitEvent(p.h2d, p.start, 0)) != cudaSuccess) return err;
  if (frames == nullptr) {
    int32_t* f = reinterpret_cast<int32_t*>(w);
    const int64_t blocks = (rows + 255) / 256 < 1024 ? (rows + 255) / 256 : 1024;
    fill_frames_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(f, rows, rows_per_frame);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    frames = f;
  }

  const int64_t quads = cols / 64;
  for (int64_t i = 0, r0 = 0; r0 < rows; ++i, r0 += chunk_rows) {
    const int s = static_cast<int>(i % kDepth);
    const int64_t n = rows - r0 < chunk_rows ? rows - r0 : chunk_rows;
    const int64_t pad_n = (n + 127) / 128 * 128;
    if (i >= kDepth && (err = cudaStreamWaitEvent(p.h2d, p.computed[s], 0)) != cudaSuccess) return err;
    if ((err = cudaMemcpyAsync(xs[s], x_host + r0 * cols, n * cols * 2, cudaMemcpyHostToDevice, p.h2d)) !=
        cudaSuccess)
      return err;
    if ((err = cudaEventRecord(p.loaded[s], p.h2d)) != cudaSuccess) return err;
    if ((err = cudaStreamWaitEvent(stream, p.loaded[s], 0)) != cudaSuccess) return err;
    if (i >= kDepth && (err = cudaStreamWaitEvent(stream, p.drained[s], 0)) != cudaSuccess) return err;
    if ((err = launch_adaln(xs[s], cols, gamma, table, num_frames, frames + r0, 0, eps, n, cols, gsf, cs[s],
                            ss[s], nullptr, stream)) != cudaSuccess)
      return err;
    if ((err = cudaEventRecord(p.computed[s], stream)) != cudaSuccess) return err;
    if ((err = cudaStreamWaitEvent(p.d2h, p.computed[s], 0)) != cudaSuccess) return err;
    if ((err = cudaMemcpyAsync(codes_host + r0 * cols / 2, cs[s], n * cols / 2, cudaMemcpyDeviceToHost,
                               p.d2h)) != cudaSuccess)
      return err;
    // the scales of rows r0.. (r0 a multiple of 128) start at (r0 / 128) atoms of quads words
    if ((err = cudaMemcpyAsync(scales_host + r0 / 128 * quads * 512, ss[s], pad_n * cols / 16,
                               cudaMemcpyDeviceToHost, p.d2h)) != cudaSuccess)
      return err;
    if ((err = cudaEventRecord(p.drained[s], p.d2h)) != cudaSuccess) return err;
  }
  // the caller's stream continues once every copy back has been issued before it
  if ((err = cudaEventRecord(p.done, p.d2h)) != cudaSuccess) return err;
  return cudaStreamWaitEvent(stream, p.done, 0);
}

}  // namespace h3q
