// dit_modulation_static: the per-step modulation without any caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// modulation: a plugin inside a host framework that owns every device buffer and hands
// the plugin only its input and output tensors, or a serving loop that forbids
// allocation after start-up (cudaMalloc can synchronise the device and can fail once
// memory is fragmented).  For them this entry point keeps its two small fp32 scratch
// vectors (the timestep-MLP hidden state and SiLU(e), each [batch, hidden]) in a
// file-scope __device__ array instead of the caller's workspace.  The array lives in
// every GPU that loads the library until the process exits, so its size is fixed and
// modest: batch <= 8 and hidden <= 4096, 256 KB in total.
//
// The array's host-side name is only a stand-in for the device symbol, so host code
// asks the runtime for its device address (cudaGetSymbolAddress) once per device, with
// that device current, on the first call made on it, and passes that address to the
// kernels.  Every call shares the one array: two calls that overlap on the GPU (on
// different streams) race on it.  Both scratch vectors are completely written before
// they are read, so nothing needs clearing between calls.
#include <mutex>

#include "../../include/dit.h"
#include "runtime.h"

namespace {
constexpr int kStaticMaxBatch = 8;
constexpr int kStaticMaxHidden = 4096;
constexpr int kMaxDevices = 64;
}  // namespace

// The scratch: [0, 8*4096) holds SiLU(t_in s), [8*4096, 2*8*4096) holds SiLU(e).
static __device__ __align__(256) float g_static_scratch[2 * kStaticMaxBatch * kStaticMaxHidden];

namespace dit {
namespace {

std::mutex g_static_mu;
float* g_static_addr[kMaxDevices] = {nullptr};

// Device address of g_static_scratch on the current device, looked up once per device.
cudaError_t static_scratch(float** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) {
      // Clear the runtime's last-error slot so that a later, unrelated call does not report
      // this failure as its own (a lookup refused during a stream capture, for example).
      (void)cudaGetLastError();
      return e;
    }
    g_static_addr[dev] = static_cast<float*>(p);
  }
  *out = g_static_addr[dev];
  return cudaSuccess;
}

inline bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dit

extern "C" dit_status dit_modulation_static(const dit_weights* w, const float* sigma_dev, int batch, void* mod_dev,
                                            dit_stream_t stream) {
  using namespace dit;
  if (!w) return DIT_ERR_INVALID_ARG;
  // The public size query validates the configuration without touching the device.
  const dit_shape one{1, 1, 1, 0};
  size_t unused = 0;
  const dit_status cs = dit_workspace_size(&w->cfg, &one, &unused);
  if (cs != DIT_OK) return cs;
  if (batch < 1) return DIT_ERR_INVALID_ARG;
  if (batch > kStaticMaxBatch || w->cfg.hidden > kStaticMaxHidden) return DIT_ERR_UNSUPPORTED;
  if (!aligned16(w->mod.t_in) || !aligned16(w->mod.t_out) || !aligned16(w->mod.mod) || !aligned16(sigma_dev) ||
      !aligned16(mod_dev))
    return DIT_ERR_INVALID_ARG;
  float* scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) return DIT_ERR_CUDA;
  float* h1 = scratch;
  float* h2 = scratch + kStaticMaxBatch * kStaticMaxHidden;
  const int H = w->cfg.hidden;
  const cudaStream_t st = (cudaStream_t)stream;
  if (launch_timestep_in((const bf16*)w->mod.t_in, H, 256, sigma_dev, batch, h1, st) != cudaSuccess)
    return DIT_ERR_CUDA;
  if (launch_gemv((const bf16*)w->mod.t_out, H, H, h1, batch, 1, h2, nullptr, st) != cudaSuccess)
    return DIT_ERR_CUDA;
  if (launch_gemv((const bf16*)w->mod.mod, 17 * H, H, h2, batch, 0, nullptr, (bf16*)mod_dev, st) != cudaSuccess)
    return DIT_ERR_CUDA;
  return DIT_OK;
}
