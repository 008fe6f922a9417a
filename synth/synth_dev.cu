// synth_dev.cu -- device-side fills for the seeded synthetic inputs, giving the
// same bits as synth_host.c (integer generator, explicit round-to-nearest
// double multiply and add, so no fused multiply-add changes a value).
// Inputs only: no transformer arithmetic lives here.
#include <cuda_runtime.h>
#include "synth.h"

static __device__ __forceinline__ uint16_t affine_bf16_dev(double mean, double sigma, double z) {
  double p = __dmul_rn(sigma, z);
  double s = __dadd_rn(mean, p);
  return syn_bf16_from_double(s);
}

__global__ void syn_fill_normal_kernel(uint16_t* out, uint64_t n, uint64_t seed, uint64_t stream,
                                       uint64_t first, double mean, double sigma) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = affine_bf16_dev(mean, sigma, syn_normal(seed, stream, first + i));
}

__global__ void syn_fill_kv_kernel(uint16_t* out, int row, int kv, int Hkv, long long per,
                                   uint64_t seed, double sigma) {
  int blk = blockIdx.y;
  int l = blk / Hkv, h = blk % Hkv;
  uint64_t st = syn_stream_kv(row, l, kv, h);
  uint16_t* o = out + (long long)blk * per;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < per;
       i += (long long)gridDim.x * blockDim.x)
    o[i] = affine_bf16_dev(0.0, sigma, syn_normal(seed, st, (uint64_t)i));
}

__global__ void syn_fill_tokens_kernel(int32_t* out, uint64_t n, uint64_t seed, uint64_t stream,
                                       uint64_t first, uint32_t vocab) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
       i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = (int32_t)syn_uniform_int(syn_u64(seed, stream, first + i), vocab);
}

static int grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  if (g > 65535ull * 4) g = 65535ull * 4;
  if (g < 1) g = 1;
  return (int)g;
}

extern "C" {

int syn_dev_fill_normal_bf16(void* out, uint64_t n, uint64_t seed, uint64_t stream, uint64_t first,
                             double mean, double sigma, void* cuda_stream) {
  if (n == 0) return 0;
  syn_fill_normal_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(
      (uint16_t*)out, n, seed, stream, first, mean, sigma);
  return (int)cudaGetLastError();
}

int syn_dev_fill_kv(void* out, int row, int kv, int L, int Hkv, int n_tok, int hd, uint64_t seed,
                    double sigma, void* cuda_stream) {
  long long per = (long long)n_tok * hd;
  if (per == 0) return 0;
  dim3 grid((unsigned)((per + 255) / 256 > 1024 ? 1024 : (per + 255) / 256), (unsigned)(L * Hkv));
  syn_fill_kv_kernel<<<grid, 256, 0, (cudaStream_t)cuda_stream>>>((uint16_t*)out, row, kv, Hkv,
                                                                   per, seed, sigma);
  return (int)cudaGetLastError();
}

int syn_dev_fill_tokens(int32_t* out, uint64_t n, uint64_t seed, uint64_t stream, uint64_t first,
                        uint32_t vocab, void* cuda_stream) {
  if (n == 0) return 0;
  syn_fill_tokens_kernel<<<grid_for(n), 256, 0, (cudaStream_t)cuda_stream>>>(out, n, seed, stream,
                                                                           first, vocab);
  return (int)cudaGetLastError();
}

}  // extern "C"
