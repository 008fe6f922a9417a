// gemm_simt.cu -- CUDA-core projections y = x W^T (x fp32 [n][K], W bf16 or 4-bit affine).
//
//  * gemv_splitk: the skinny decode case (n <= 32).  A block owns 64 weight rows and one
//    K-slice; every weight element is loaded once (16-byte loads, or one 32-bit word of eight
//    4-bit codes) and used for all n rows, whose activations sit in shared memory.  Partial
//    sums go to a [slices][n][M] buffer; splitk_reduce adds the slices in order and applies
//    the epilogue, so results do not depend on scheduling.
//  * gemm_tiled: prefill (n > 32), 64x64 output tiles staged through shared memory.
#include "kernels.h"

namespace {

constexpr int GEMV_ROWS = 64;     // weight rows per block (8 warps x 8 rows)
constexpr int GEMV_THREADS = 256;

CBT_D float dot8_bf16(uint4 w, const float* x) {
  float a = x[0] * bf16_lo(w.x);
  a = fmaf(x[1], bf16_hi(w.x), a);
  a = fmaf(x[2], bf16_lo(w.y), a);
  a = fmaf(x[3], bf16_hi(w.y), a);
  a = fmaf(x[4], bf16_lo(w.z), a);
  a = fmaf(x[5], bf16_hi(w.z), a);
  a = fmaf(x[6], bf16_lo(w.w), a);
  a = fmaf(x[7], bf16_hi(w.w), a);
  return a;
}

// eight 4-bit codes of one word, dequantised as scale*q + bias
CBT_D void deq8(uint32_t word, float sc, float bi, float* w) {
#pragma unroll
  for (int k = 0; k < 8; ++k) w[k] = fmaf(sc, (float)((word >> (4 * k)) & 0xFu), bi);
}

template <int NB, bool Q4>
__global__ void __launch_bounds__(GEMV_THREADS) gemv_splitk(const float* __restrict__ x, int n,
                                                            int K, LinearW W, int M, int Ks,
                                                            float* __restrict__ part) {
  pdl_wait();
  pdl_launch();
  extern __shared__ float xs[];  // [NB][Ks]
  const int k0 = blockIdx.y * Ks;
  for (int i = threadIdx.x; i < n * Ks; i += blockDim.x) {
    int b = i / Ks, kk = i % Ks;
    xs[i] = x[(size_t)b * K + k0 + kk];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = 0; r < GEMV_ROWS / 8; ++r) {
    const int m = blockIdx.x * GEMV_ROWS + warp * (GEMV_ROWS / 8) + r;
    if (m >= M) break;
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
    for (int kk = lane * 8; kk < Ks; kk += 256) {
      float wf[8];
      if (!Q4) {
        uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(W.w) +
                                                       (size_t)m * K + k0 + kk));
        wf[0] = bf16_lo(w.x); wf[1] = bf16_hi(w.x); wf[2] = bf16_lo(w.y); wf[3] = bf16_hi(w.y);
        wf[4] = bf16_lo(w.z); wf[5] = bf16_hi(w.z); wf[6] = bf16_lo(w.w); wf[7] = bf16_hi(w.w);
      } else {
        int k = k0 + kk;
        uint32_t word = __ldg(static_cast<const uint32_t*>(W.w) + (size_t)m * (K / 8) + k / 8);
        size_t gi = (size_t)m * (K / 64) + k / 64;
        deq8(word, bf16_to_f32(W.scales[gi]), bf16_to_f32(W.biases[gi]), wf);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b < n) {
          const float* xb = xs + b * Ks + kk;
          float4 x0 = *reinterpret_cast<const float4*>(xb);
          float4 x1 = *reinterpret_cast<const float4*>(xb + 4);
          float a = acc[b];
          a = fmaf(wf[0], x0.x, a); a = fmaf(wf[1], x0.y, a);
          a = fmaf(wf[2], x0.z, a); a = fmaf(wf[3], x0.w, a);
          a = fmaf(wf[4], x1.x, a); a = fmaf(wf[5], x1.y, a);
          a = fmaf(wf[6], x1.z, a); a = fmaf(wf[7], x1.w, a);
          acc[b] = a;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b < n) {
        float v = warp_sum(acc[b]);
        if (lane == 0) part[((size_t)blockIdx.y * n + b) * M + m] = v;
      }
    }
  }
}

__global__ void splitk_reduce(const float* __restrict__ part, int S, int n, int M, int epi,
                              float* __restrict__ out) {
  pdl_wait();
  pdl_launch();
  const int Mo = epi == EPI_SWIGLU ? M / 2 : M;
  long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (idx >= (long long)n * Mo) return;
  int b = (int)(idx / Mo), m = (int)(idx % Mo);
  float v = 0.f;
  for (int s = 0; s < S; ++s) v += part[((size_t)s * n + b) * M + m];
  if (epi == EPI_STORE) {
    out[idx] = v;
  } else if (epi == EPI_ADD) {
    out[idx] += v;
  } else {
    float u = 0.f;
    for (int s = 0; s < S; ++s) u += part[((size_t)s * n + b) * M + m + Mo];
    out[idx] = v / (1.f + expf(-v)) * u;
  }
}

// ---- tiled GEMM for many tokens -----------------------------------------------------------
constexpr int TT = 64, TM = 64, TK = 16;

template <bool Q4, int EPI>
__global__ void __launch_bounds__(256) gemm_tiled(const float* __restrict__ x, int n, int K,
                                                  LinearW W, int M, float* __restrict__ out) {
  pdl_wait();
  pdl_launch();
  // SWIGLU: columns j of the tile are gate row j and up row j + M/2
  __shared__ float xs[TK][TT + 4];
  __shared__ float ws[TK][TM + 4];
  __shared__ float us[TK][TM + 4];
  const int Mo = EPI == EPI_SWIGLU ? M / 2 : M;
  const int t0 = blockIdx.y * TT, m0 = blockIdx.x * TM;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;  // 16 x 16 threads, 4 x 4 each
  float acc[4][4] = {}, accu[4][4] = {};
  for (int kb = 0; kb < K; kb += TK) {
    for (int i = threadIdx.x; i < TK * TT; i += 256) {
      int kk = i % TK, tt = i / TK;
      int t = t0 + tt;
      xs[kk][tt] = t < n ? x[(size_t)t * K + kb + kk] : 0.f;
    }
    for (int i = threadIdx.x; i < TK * TM; i += 256) {
      int kk = i % TK, mm = i / TK;
      int m = m0 + mm, k = kb + kk;
      float wv = 0.f, uv = 0.f;
      if (m < Mo) {
        for (int which = 0; which < (EPI == EPI_SWIGLU ? 2 : 1); ++which) {
          int row = m + which * Mo;
          float v;
          if (!Q4) {
            v = bf16_to_f32(static_cast<const uint16_t*>(W.w)[(size_t)row * K + k]);
          } else {
            uint32_t word = static_cast<const uint32_t*>(W.w)[(size_t)row * (K / 8) + k / 8];
            size_t gi = (size_t)row * (K / 64) + k / 64;
            v = fmaf(bf16_to_f32(W.scales[gi]), (float)((word >> (4 * (k % 8))) & 0xFu),
                     bf16_to_f32(W.biases[gi]));
          }
          if (which == 0) wv = v; else uv = v;
        }
      }
      ws[kk][mm] = wv;
      us[kk][mm] = uv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float xv[4], wv[4], uv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xv[i] = xs[kk][ty * 4 + i];
        wv[i] = ws[kk][tx * 4 + i];
        uv[i] = us[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
          if (EPI == EPI_SWIGLU) accu[i][j] = fmaf(xv[i], uv[j], accu[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int t = t0 + ty * 4 + i, m = m0 + tx * 4 + j;
      if (t < n && m < Mo) {
        float v = acc[i][j];
        float* o = out + (size_t)t * Mo + m;
        if (EPI == EPI_STORE) *o = v;
        else if (EPI == EPI_ADD) *o += v;
        else *o = v / (1.f + expf(-v)) * accu[i][j];
      }
    }
}

int pick_slice(int K) {
  for (int ks : {1024, 512, 256})
    if (K % ks == 0) return ks;
  return 0;
}

template <int NB>
cudaError_t run_gemv(const float* x, int n, int K, const LinearW& W, int M, int Ks, float* part,
                     cudaStream_t s) {
  dim3 grid((M + GEMV_ROWS - 1) / GEMV_ROWS, K / Ks);
  size_t smem = sizeof(float) * (size_t)NB * Ks;
  cudaError_t rc;
  if (W.fmt == CBT_WEIGHTS_BF16) {
    rc = cudaFuncSetAttribute(gemv_splitk<NB, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (rc != cudaSuccess) return rc;
    return launch_pdl((gemv_splitk<NB, false>), dim3(grid), dim3(GEMV_THREADS), smem, s, x, n, K, W, M, Ks, part);
  }
  rc = cudaFuncSetAttribute(gemv_splitk<NB, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (rc != cudaSuccess) return rc;
  return launch_pdl((gemv_splitk<NB, true>), dim3(grid), dim3(GEMV_THREADS), smem, s, x, n, K, W, M, Ks, part);
}

template <int EPI>
cudaError_t run_tiled(const float* x, int n, int K, const LinearW& W, int M, float* out, cudaStream_t s) {
  int Mo = EPI == EPI_SWIGLU ? M / 2 : M;
  dim3 grid((Mo + TM - 1) / TM, (n + TT - 1) / TT);
  if (W.fmt == CBT_WEIGHTS_BF16)
    return launch_pdl((gemm_tiled<false, EPI>), dim3(grid), dim3(256), 0, s, x, n, K, W, M, out);
  return launch_pdl((gemm_tiled<true, EPI>), dim3(grid), dim3(256), 0, s, x, n, K, W, M, out);
}

}  // namespace

cudaError_t launch_linear(const float* x, int n, int K, const LinearW& W, int M, Epilogue epi,
                          float* out, float* partials, size_t partial_floats, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  int Ks = pick_slice(K);
  if (n <= 32 && Ks > 0 && (size_t)(K / Ks) * n * M <= partial_floats) {
    cudaError_t rc;
    if (n <= 8) rc = run_gemv<8>(x, n, K, W, M, Ks, partials, s);
    else if (n <= 16) rc = run_gemv<16>(x, n, K, W, M, Ks, partials, s);
    else rc = run_gemv<32>(x, n, K, W, M, Ks, partials, s);
    if (rc != cudaSuccess) return rc;
    int Mo = epi == EPI_SWIGLU ? M / 2 : M;
    long long tot = (long long)n * Mo;
    return launch_pdl(splitk_reduce, dim3((unsigned)((tot + 255) / 256)), dim3(256), 0, s,
                      partials, K / Ks, n, M, epi, out);
  }
  if (epi == EPI_STORE) return run_tiled<EPI_STORE>(x, n, K, W, M, out, s);
  if (epi == EPI_ADD) return run_tiled<EPI_ADD>(x, n, K, W, M, out, s);
  return run_tiled<EPI_SWIGLU>(x, n, K, W, M, out, s);
}
