// noalloc.cu -- cbt_greedy_head_noalloc: the final RMSNorm + lm_head projection + greedy
// argmax for callers that cannot allocate device memory.  Its scratch is one fixed array in
// the library's own device memory instead of anything obtained from cudaMalloc.
#include <cuda_runtime.h>

#include <mutex>

#include "cbt.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchFloats = CBT_NOALLOC_SCRATCH_BYTES / sizeof(float);

// The scratch: normalised rows, then the split-K partial sums.  Host code must not pass
// this symbol to a kernel (in host code it is only a stand-in); it passes the device address
// that cudaGetSymbolAddress returns.
static __device__ __align__(256) float g_head_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
cbt_status scratch_on_current_device(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CBT_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_head_scratch) != cudaSuccess || !p) return CBT_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return CBT_OK;
}

int slice_of(int K) {
  for (int ks : {1024, 512, 256})
    if (K % ks == 0) return ks;
  return 0;
}

}  // namespace

extern "C" cbt_status cbt_greedy_head_noalloc(const cbt_model_config* cfg, const float* hidden,
                                              int32_t n, const void* final_norm,
                                              const cbt_linear* lm_head, float* logits,
                                              int32_t* next_tokens, void* stream) {
  if (!cfg || !lm_head) return CBT_ERR_NULL;
  if (n < 0 || cfg->d_model <= 0 || cfg->vocab <= 0) return CBT_ERR_INVALID;
  if (n == 0) return CBT_OK;
  if (!hidden || !final_norm || !logits || !lm_head->w) return CBT_ERR_NULL;
  if (cfg->weight_format != CBT_WEIGHTS_BF16 && cfg->weight_format != CBT_WEIGHTS_AFFINE4)
    return CBT_ERR_INVALID;
  if (cfg->weight_format == CBT_WEIGHTS_AFFINE4) {
    if (cfg->group_size != 64) return CBT_ERR_UNSUPPORTED;
    if (!lm_head->scales || !lm_head->biases) return CBT_ERR_NULL;
  }
  const int d = cfg->d_model, V = cfg->vocab;
  const int ks = slice_of(d);
  if (ks == 0) return CBT_ERR_UNSUPPORTED;
  if (n > CBT_NOALLOC_MAX_ROWS) return CBT_ERR_LIMIT;
  const size_t h_floats = ((size_t)n * d + 63) & ~size_t(63);  // 256-byte aligned split
  const size_t part_floats = (size_t)(d / ks) * n * V;
  if (h_floats + part_floats > kScratchFloats) return CBT_ERR_LIMIT;

  float* scratch = nullptr;
  cbt_status st = scratch_on_current_device(&scratch);
  if (st != CBT_OK) return st;
  float* h = scratch;
  float* part = scratch + h_floats;
  const size_t part_cap = kScratchFloats - h_floats;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LinearW W{lm_head->w, static_cast<const uint16_t*>(lm_head->scales),
            static_cast<const uint16_t*>(lm_head->biases), cfg->weight_format};
  // each launch's own status: an error left behind by unrelated earlier work is not this call's
  cudaError_t rc = launch_rmsnorm(hidden, static_cast<const uint16_t*>(final_norm), n, d,
                                  cfg->rms_eps, h, s);
  if (rc == cudaSuccess) rc = launch_linear(h, n, d, W, V, EPI_STORE, logits, part, part_cap, s);
  if (rc == cudaSuccess && next_tokens) rc = launch_argmax(logits, n, V, next_tokens, s);
  return rc == cudaSuccess ? CBT_OK : CBT_ERR_CUDA;
}
