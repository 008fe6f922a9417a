// basic.cu -- the step's small kernels: embedding, RMSNorm, RoPE tables, RoPE + KV append,
// plain per-token attention, greedy argmax, row gather and the 4-bit quantiser.
#include <math.h>

#include <algorithm>

#include "kernels.h"

// ---- embedding: x[i] = E[token[i]] (fp32); out-of-range ids set the error word ------------
// With ss, also what the first RMSNorm needs when it is folded into the QKV projection: the
// row's sums of squares over each 128-element tile, ss[tile * ss_ld + i], and the operand
// x * gain as bf16 hi (row i of act) and lo (row lo_rows + i) parts.
// Embedding rows (one block of 256 threads per token) and, in the blocks after them, the RoPE
// cos/sin table of the call's positions (fp32 [n][head_dim / 2] each, angles in double): one
// launch for the step's two independent prologue kernels.  A token's row is read with 16-byte
// loads, eight columns a thread, all in flight together; the same values give the first
// RMSNorm's per-128-column sums of squares (16 threads per tile).
__global__ void k_embed_rope(const int32_t* tokens, int n, int d, int vocab,
                             const uint16_t* table, float* x, int* err, float* ss, int ss_ld,
                             const uint16_t* gain, uint16_t* act, int lo_rows,
                             const QueryRow* rows, int half, int head_dim, double theta,
                             float* cosv, float* sinv) {
  pdl_wait();
  pdl_launch();
  if ((int)blockIdx.x >= n) {  // RoPE table
    const int idx = (blockIdx.x - n) * blockDim.x + threadIdx.x;
    if (idx >= n * half) return;
    const int t = idx / half, i = idx % half;
    const double freq = pow(theta, -2.0 * (double)i / (double)head_dim);
    const double ang = (double)rows[t].pos * freq;
    double sv, cv;
    sincos(ang, &sv, &cv);
    cosv[idx] = (float)cv;
    sinv[idx] = (float)sv;
    return;
  }
  const int i = blockIdx.x;
  const int t = tokens[i];
  float* xr = x + (size_t)i * d;
  const bool bad = t < 0 || t >= vocab;
  if (bad && threadIdx.x == 0) set_device_error(err, CBT_DEV_TOKEN_RANGE, i);
  const uint16_t* er = table + (size_t)(bad ? 0 : t) * d;
  if ((d & 127) == 0 && (reinterpret_cast<uintptr_t>(table) & 15) == 0 &&
      (!act || (reinterpret_cast<uintptr_t>(gain) & 15) == 0)) {
    constexpr int kU = 4;  // 8-column chunks per thread in flight
    const int nch = d >> 3;
    for (int c0 = threadIdx.x; c0 < nch; c0 += blockDim.x * kU) {
      uint4 e[kU], g[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + u * (int)blockDim.x;
        e[u] = (c < nch && !bad) ? __ldg(reinterpret_cast<const uint4*>(er) + c) : make_uint4(0, 0, 0, 0);
        g[u] = (c < nch && act) ? __ldg(reinterpret_cast<const uint4*>(gain) + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int c = c0 + u * (int)blockDim.x;
        const uint32_t ew[4] = {e[u].x, e[u].y, e[u].z, e[u].w};
        const uint32_t gw[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
        float v[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[2 * k] = bf16_lo(ew[k]);
          v[2 * k + 1] = bf16_hi(ew[k]);
        }
        float sq = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) sq = fmaf(v[k], v[k], sq);
        if (c < nch) {
          *reinterpret_cast<float4*>(xr + 8 * c) = make_float4(v[0], v[1], v[2], v[3]);
          *reinterpret_cast<float4*>(xr + 8 * c + 4) = make_float4(v[4], v[5], v[6], v[7]);
          if (act) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float a0 = v[2 * k] * bf16_lo(gw[k]), a1 = v[2 * k + 1] * bf16_hi(gw[k]);
              const uint16_t h0 = f32_to_bf16(a0), h1 = f32_to_bf16(a1);
              hw[k] = (uint32_t)h0 | ((uint32_t)h1 << 16);
              lw[k] = (uint32_t)f32_to_bf16(a0 - bf16_to_f32(h0)) |
                      ((uint32_t)f32_to_bf16(a1 - bf16_to_f32(h1)) << 16);
            }
            *reinterpret_cast<uint4*>(act + (size_t)i * d + 8 * c) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            if (lo_rows > 0)
              *reinterpret_cast<uint4*>(act + (size_t)(lo_rows + i) * d + 8 * c) =
                  make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        if (ss) {  // the 16 chunks of a 128-column tile sit in 16 consecutive lanes
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
          if ((threadIdx.x & 15) == 0 && c < nch) ss[(size_t)(c >> 4) * ss_ld + i] = sq;
        }
      }
    }
    return;
  }
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    const float v = bad ? 0.f : bf16_to_f32(er[j]);
    xr[j] = v;
    if (act) {
      const float a = v * bf16_to_f32(gain[j]);
      const uint16_t hi = f32_to_bf16(a);
      act[(size_t)i * d + j] = hi;
      if (lo_rows > 0) act[(size_t)(lo_rows + i) * d + j] = f32_to_bf16(a - bf16_to_f32(hi));
    }
  }
  if (ss) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int tile = warp; tile * 128 < d; tile += nw) {
      float sum = 0.f;
      for (int j = tile * 128 + lane; j < d && j < tile * 128 + 128; j += 32) {
        const float v = bad ? 0.f : bf16_to_f32(er[j]);
        sum = fmaf(v, v, sum);
      }
      sum = warp_sum(sum);
      if (lane == 0) ss[(size_t)tile * ss_ld + i] = sum;
    }
  }
}

void launch_embed_rope(const int32_t* tokens, int n, const uint16_t* table, int d, int vocab,
                       float* x, int* err, float* ss, int ss_ld, const uint16_t* gain,
                       uint16_t* act, int lo_rows, const QueryRow* rows, int head_dim,
                       double theta, float* cosv, float* sinv, cudaStream_t s) {
  if (n <= 0) return;
  const int half = head_dim / 2;
  const int rope_blocks = (n * half + 255) / 256;
  launch_pdl(k_embed_rope, dim3(n + rope_blocks), dim3(256), 0, s, tokens, n, d, vocab, table, x,
             err, ss, ss_ld, gain, act, lo_rows, rows, half, head_dim, theta, cosv, sinv);
}

// ---- RMSNorm: h = x / sqrt(mean(x^2) + eps) * g -----------------------------------------
__global__ void k_rmsnorm(const float* x, const uint16_t* gain, int d, float eps, float* h) {
  pdl_wait();
  pdl_launch();
  __shared__ float red[32];
  const float* xr = x + (size_t)blockIdx.x * d;
  float ss = 0.f;
  for (int j = threadIdx.x; j < d; j += blockDim.x) ss = fmaf(xr[j], xr[j], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  float r = rsqrtf(red[0] / (float)d + eps);
  float* hr = h + (size_t)blockIdx.x * d;
  for (int j = threadIdx.x; j < d; j += blockDim.x) hr[j] = xr[j] * r * bf16_to_f32(gain[j]);
}

cudaError_t launch_rmsnorm(const float* x, const uint16_t* gain, int n, int d, float eps,
                           float* h, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(k_rmsnorm, dim3(n), dim3(256), 0, s, x, gain, d, eps, h);
}

// bf16 operand of a tensor-core projection: hi = bf16(v), and lo = bf16(v - hi) in rows
// shifted by lo_rows when lo_rows > 0 (hi + lo carries about 16 significant bits)
CBT_D void store_act(uint16_t* act, int row, int K, int k, int lo_rows, float v) {
  const uint16_t hi = f32_to_bf16(v);
  act[(size_t)row * K + k] = hi;
  if (lo_rows > 0) act[(size_t)(lo_rows + row) * K + k] = f32_to_bf16(v - bf16_to_f32(hi));
}

__global__ void k_rmsnorm_act(const float* x, const uint16_t* gain, int d, float eps,
                              uint16_t* act, int lo_rows) {
  pdl_wait();
  pdl_launch();
  __shared__ float red[32];
  const float* xr = x + (size_t)blockIdx.x * d;
  float ss = 0.f;
  for (int j = threadIdx.x; j < d; j += blockDim.x) ss = fmaf(xr[j], xr[j], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float r = rsqrtf(red[0] / (float)d + eps);
  for (int j = threadIdx.x; j < d; j += blockDim.x)
    store_act(act, blockIdx.x, d, j, lo_rows, xr[j] * r * bf16_to_f32(gain[j]));
}

void launch_rmsnorm_act(const float* x, const uint16_t* gain, int n, int d, float eps,
                        uint16_t* act, int lo_rows, cudaStream_t s) {
  if (n <= 0) return;
  launch_pdl(k_rmsnorm_act, dim3(n), dim3(256), 0, s, x, gain, d, eps, act, lo_rows);
}

__global__ void k_f32_to_act(const float* src, int K, uint16_t* act, int lo_rows) {
  pdl_wait();
  pdl_launch();
  const float* sr = src + (size_t)blockIdx.x * K;
  for (int k = threadIdx.x; k < K; k += blockDim.x) store_act(act, blockIdx.x, K, k, lo_rows, sr[k]);
}

void launch_f32_to_act(const float* src, int n, int K, uint16_t* act, int lo_rows, cudaStream_t s) {
  if (n <= 0) return;
  launch_pdl(k_f32_to_act, dim3(n), dim3(256), 0, s, src, K, act, lo_rows);
}

// ---- RoPE angles once per call: cos/sin of pos * theta^(-2i/hd), evaluated in double -------
// ---- RoPE q, k in place at the token's position; append k, v to its own slab at pos ------
__global__ void k_rope_append(float* qkv, const QueryRow* rows, int layer, int n_heads,
                              int n_kv_heads, int head_dim, const float* cosv, const float* sinv,
                              uint16_t* arena, uint8_t* qtile, uint16_t* qb, int q_lo_row) {
  pdl_wait();
  pdl_launch();
  int t = blockIdx.x;
  int half = head_dim / 2;
  int qd = n_heads * head_dim, kvd = n_kv_heads * head_dim;
  float* row = qkv + (size_t)t * (qd + 2 * kvd);
  const float* cr = cosv + (size_t)t * half;
  const float* sr = sinv + (size_t)t * half;
  QueryRow r = rows[t];
  int pairs = (n_heads + n_kv_heads) * half;
  for (int p = threadIdx.x; p < pairs; p += blockDim.x) {
    int h = p / half, i = p % half;
    float* v = row + (size_t)h * head_dim;  // q heads then k heads are contiguous
    float a = v[i], b = v[i + half], c = cr[i], s = sr[i];
    float ra = a * c - b * s;
    float rb = a * s + b * c;
    v[i] = ra;
    v[i + half] = rb;
    if (h >= n_heads) {
      uint16_t* kd = arena + k_index(r, layer, h - n_heads, r.pos, 0, n_kv_heads, head_dim);
      kd[i] = f32_to_bf16(ra);
      kd[i + half] = f32_to_bf16(rb);
    } else if (qb) {
      // the prefill attention's Q operand, scaled by 1/sqrt(head_dim): bf16 high parts at row
      // t, the bf16 rounding of the remainders at row q_lo_row + t
      const float qs = rsqrtf((float)head_dim);
      const float a = ra * qs, b = rb * qs;
      const uint16_t ah = f32_to_bf16(a), bh = f32_to_bf16(b);
      uint16_t* hi = qb + (size_t)t * qd + (size_t)h * head_dim;
      uint16_t* lo = hi + (size_t)q_lo_row * qd;
      hi[i] = ah;
      hi[i + half] = bh;
      lo[i] = f32_to_bf16(a - bf16_to_f32(ah));
      lo[i + half] = f32_to_bf16(b - bf16_to_f32(bh));
    } else if (qtile) {
      // the decode attention's Q operand of this row and kv head: [16 rows][head_dim] bf16 in
      // the MMA's swizzled layout; row j < G holds the hi part of q head g*G + j scaled by
      // 1/sqrt(head_dim), row 8 + j its lo part (rows beyond stay zero)
      const int G = n_heads / n_kv_heads, g = h / G, j = h % G;
      uint8_t* tile = qtile + ((size_t)t * n_kv_heads + g) * (16 * head_dim * 2);
      const float qs = rsqrtf((float)head_dim);
      const float vals[2] = {ra * qs, rb * qs};
      const int cols[2] = {i, i + half};
      for (int u = 0; u < 2; ++u) {
        const uint16_t hi = f32_to_bf16(vals[u]);
        const uint16_t lo = f32_to_bf16(vals[u] - bf16_to_f32(hi));
        *reinterpret_cast<uint16_t*>(tile + sw128_offset(j, cols[u], 2048)) = hi;
        *reinterpret_cast<uint16_t*>(tile + sw128_offset(8 + j, cols[u], 2048)) = lo;
      }
    }
  }
  const float* vv = row + qd + kvd;
  for (int e = threadIdx.x; e < kvd; e += blockDim.x) {
    int g = e / head_dim, j = e % head_dim;
    arena[v_index(r, layer, g, r.pos, j, n_kv_heads, head_dim)] = f32_to_bf16(vv[e]);
  }
}

void launch_rope_append(float* qkv, const QueryRow* rows, int n, int layer, int n_heads,
                        int n_kv_heads, int head_dim, const float* cosv, const float* sinv,
                        uint16_t* arena, uint8_t* qtile, uint16_t* qb, int q_lo_row,
                        cudaStream_t s) {
  if (n <= 0) return;
  launch_pdl(k_rope_append, dim3(n), dim3(256), 0, s, qkv, rows, layer, n_heads, n_kv_heads,
             head_dim, cosv, sinv, arena, qtile, qb, q_lo_row);
}

// ---- V of one layer between the plain [kv head][plain_n positions][head_dim] layout and a slab
// (or page) -- to_slab: plain -> slab, else slab -> plain; positions [t0, t0 + n)
__global__ void k_v_convert(uint16_t* plain, uint16_t* arena, QueryRow r, int layer,
                            int n_kv_heads, int t0, int n, int plain_n, int head_dim, int to_slab) {
  pdl_wait();
  pdl_launch();
  long long tot = (long long)n_kv_heads * n * head_dim;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < tot;
       i += (long long)gridDim.x * blockDim.x) {
    int d = (int)(i % head_dim);
    long long rest = i / head_dim;
    int t = t0 + (int)(rest % n), g = (int)(rest / n);
    long long at = v_index(r, layer, g, t, d, n_kv_heads, head_dim);
    long long pi = ((long long)g * plain_n + t) * head_dim + d;
    if (to_slab) arena[at] = plain[pi];
    else plain[pi] = arena[at];
  }
}

void launch_v_convert(uint16_t* plain, uint16_t* arena, const QueryRow& r, int layer,
                      int n_kv_heads, int t0, int n, int plain_n, int head_dim, bool to_slab,
                      cudaStream_t s) {
  long long tot = (long long)n_kv_heads * n * head_dim;
  if (tot <= 0) return;
  int grid = (int)std::min<long long>((tot + 255) / 256, 4096);
  launch_pdl(k_v_convert, dim3(grid), dim3(256), 0, s, plain, arena, r, layer, n_kv_heads, t0, n,
             plain_n, head_dim, to_slab ? 1 : 0);
}

// ---- plain attention: one block per (token, q head), keys [0, pos] of its own slab -------
__global__ void k_attention_naive(const float* qkv, const QueryRow* rows,
                                  const long long* pagetab, const int* tok_pages, int layer,
                                  int n_heads, int n_kv_heads, int head_dim,
                                  const uint16_t* arena, float* o) {
  pdl_wait();
  pdl_launch();
  extern __shared__ float sm[];
  __shared__ float red[32];
  int t = blockIdx.x, hq = blockIdx.y;
  int qd = n_heads * head_dim, kvd = n_kv_heads * head_dim;
  int g = hq / (n_heads / n_kv_heads);
  QueryRow r = rows[t];
  int nk = r.pos + 1;
  float* qs = sm;              // head_dim
  float* sc = sm + head_dim;   // nk scores
  const float* q = qkv + (size_t)t * (qd + 2 * kvd) + (size_t)hq * head_dim;
  for (int j = threadIdx.x; j < head_dim; j += blockDim.x) qs[j] = q[j];
  __syncthreads();
  // the slab (or, for a paged sequence, the page) holding key k, as a QueryRow
  const int tp = tok_pages ? tok_pages[t] : -1;
  auto holder = [&](int k) -> QueryRow {
    return tp < 0 ? r : QueryRow{pagetab[tp + k / r.cap], 0, r.cap};
  };
  float scale = rsqrtf((float)head_dim);
  float mx = -INFINITY;
  for (int k = threadIdx.x; k < nk; k += blockDim.x) {
    const uint4* kr = reinterpret_cast<const uint4*>(
        arena + k_index(holder(k), layer, g, k, 0, n_kv_heads, head_dim));
    float dot = 0.f;
    for (int c = 0; c < head_dim / 8; ++c) {
      uint4 w = kr[c];
      const float* qq = qs + c * 8;
      dot = fmaf(qq[0], bf16_lo(w.x), dot); dot = fmaf(qq[1], bf16_hi(w.x), dot);
      dot = fmaf(qq[2], bf16_lo(w.y), dot); dot = fmaf(qq[3], bf16_hi(w.y), dot);
      dot = fmaf(qq[4], bf16_lo(w.z), dot); dot = fmaf(qq[5], bf16_hi(w.z), dot);
      dot = fmaf(qq[6], bf16_lo(w.w), dot); dot = fmaf(qq[7], bf16_hi(w.w), dot);
    }
    float sv = dot * scale;
    sc[k] = sv;
    mx = fmaxf(mx, sv);
  }
  mx = warp_max(mx);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : -INFINITY;
    v = warp_max(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  mx = red[0];
  __syncthreads();
  float z = 0.f;
  for (int k = threadIdx.x; k < nk; k += blockDim.x) {
    float p = expf(sc[k] - mx);
    sc[k] = p;
    z += p;
  }
  z = warp_sum(z);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = z;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  float inv = 1.f / red[0];
  float* orow = o + (size_t)t * qd + (size_t)hq * head_dim;
  for (int j = threadIdx.x; j < head_dim; j += blockDim.x) {
    float acc = 0.f;
    for (int k0 = 0; k0 < nk; k0 += r.cap) {  // one slab, or page by page
      const QueryRow h = holder(k0);
      const int k1 = min(nk, k0 + r.cap);
      for (int k = k0; k < k1; ++k)
        acc = fmaf(sc[k], bf16_to_f32(arena[v_index(h, layer, g, k, j, n_kv_heads, head_dim)]), acc);
    }
    orow[j] = acc * inv;
  }
}

void launch_attention_naive(const float* qkv, const QueryRow* rows, const long long* pagetab,
                            const int* tok_pages, int n, int layer, int n_heads, int n_kv_heads,
                            int head_dim, int max_keys, const uint16_t* arena, float* o,
                            cudaStream_t s) {
  if (n <= 0) return;
  size_t smem = sizeof(float) * (size_t)(head_dim + max_keys);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(k_attention_naive, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_pdl(k_attention_naive, dim3(dim3(n, n_heads)), dim3(128), smem, s, qkv, rows, pagetab,
             tok_pages, layer, n_heads, n_kv_heads,
                                                         head_dim, arena, o);
}

// ---- greedy argmax, lowest index among equal maxima ----------------------------------------
__global__ void k_argmax(const float* logits, int vocab, int32_t* out) {
  pdl_wait();
  pdl_launch();
  __shared__ float bv[32];
  __shared__ int bi[32];
  const float* r = logits + (size_t)blockIdx.x * vocab;
  float best = -INFINITY;
  int idx = 0x7fffffff;
  if ((vocab & 3) == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0) {
    // 16-byte loads, kU of them in flight per thread (one load per iteration leaves the
    // scan a chain of memory latencies); each thread still visits its indices in increasing
    // order, so the earlier index is kept on ties
    constexpr int kU = 8;
    const float4* r4 = reinterpret_cast<const float4*>(r);
    const int n4 = vocab >> 2;
    for (int base = threadIdx.x; base < n4; base += blockDim.x * kU) {
      float4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * (int)blockDim.x;
        v[u] = i < n4 ? __ldcg(r4 + i) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = 4 * (base + u * (int)blockDim.x);
        if (v[u].x > best) { best = v[u].x; idx = i; }
        if (v[u].y > best) { best = v[u].y; idx = i + 1; }
        if (v[u].z > best) { best = v[u].z; idx = i + 2; }
        if (v[u].w > best) { best = v[u].w; idx = i + 3; }
      }
    }
  } else {
    for (int i = threadIdx.x; i < vocab; i += blockDim.x) {
      float v = r[i];
      if (v > best) { best = v; idx = i; }  // strided scan: earlier index kept on ties
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, best, off);
    int oi = __shfl_xor_sync(0xffffffffu, idx, off);
    if (ov > best || (ov == best && oi < idx)) { best = ov; idx = oi; }
  }
  if ((threadIdx.x & 31) == 0) { bv[threadIdx.x >> 5] = best; bi[threadIdx.x >> 5] = idx; }
  __syncthreads();
  if (threadIdx.x < 32) {
    int nw = blockDim.x >> 5;
    best = threadIdx.x < nw ? bv[threadIdx.x] : -INFINITY;
    idx = threadIdx.x < nw ? bi[threadIdx.x] : 0x7fffffff;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, best, off);
      int oi = __shfl_xor_sync(0xffffffffu, idx, off);
      if (ov > best || (ov == best && oi < idx)) { best = ov; idx = oi; }
    }
    if (threadIdx.x == 0) out[blockIdx.x] = idx == 0x7fffffff ? 0 : idx;
  }
}

cudaError_t launch_argmax(const float* logits, int n, int vocab, int32_t* out, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(k_argmax, dim3(n), dim3(512), 0, s, logits, vocab, out);
}

__global__ void k_gather_rows(const float* src, const int32_t* idx, int d, float* dst) {
  pdl_wait();
  pdl_launch();
  const float* sr = src + (size_t)idx[blockIdx.x] * d;
  float* dr = dst + (size_t)blockIdx.x * d;
  for (int j = threadIdx.x; j < d; j += blockDim.x) dr[j] = sr[j];
}

void launch_gather_rows(const float* src, const int32_t* idx, int n, int d, float* dst,
                        cudaStream_t s) {
  if (n <= 0) return;
  launch_pdl(k_gather_rows, dim3(n), dim3(256), 0, s, src, idx, d, dst);
}

// ---- MLX-style 4-bit affine quantisation, one thread per (row, group) ----------------------
__global__ void k_quantize_affine4(const uint16_t* w, int rows, int cols, int group,
                                   uint32_t* packed, uint16_t* scales, uint16_t* biases) {
  pdl_wait();
  pdl_launch();
  long long gid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  int ng = cols / group;
  if (gid >= (long long)rows * ng) return;
  int r = (int)(gid / ng), g = (int)(gid % ng);
  const uint16_t* src = w + (size_t)r * cols + (size_t)g * group;
  float mn = bf16_to_f32(src[0]), mx = mn;
  for (int i = 1; i < group; ++i) {
    float x = bf16_to_f32(src[i]);
    mn = fminf(mn, x);
    mx = fmaxf(mx, x);
  }
  // (mx - mn) is exact in double; divide, round to float, then to bf16
  uint16_t sb = f32_to_bf16((float)(((double)mx - (double)mn) / 15.0));
  uint16_t bb = f32_to_bf16(mn);
  double sc = bf16_to_f32(sb), bi = bf16_to_f32(bb);
  scales[gid] = sb;
  biases[gid] = bb;
  uint32_t* dst = packed + (size_t)r * (cols / 8) + (size_t)g * (group / 8);
  for (int j = 0; j < group / 8; ++j) {
    uint32_t word = 0;
    for (int k = 0; k < 8; ++k) {
      double x = bf16_to_f32(src[8 * j + k]);
      int q = 0;
      if (sc != 0.0) {
        double t = rint((x - bi) / sc);
        q = t < 0.0 ? 0 : (t > 15.0 ? 15 : (int)t);
      }
      word |= (uint32_t)q << (4 * k);
    }
    dst[j] = word;
  }
}

void launch_quantize_affine4(const uint16_t* w, int rows, int cols, int group, uint32_t* packed,
                             uint16_t* scales, uint16_t* biases, cudaStream_t s) {
  long long n = (long long)rows * (cols / group);
  if (n <= 0) return;
  launch_pdl(k_quantize_affine4, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, w, rows, cols, group, packed,
                                                                 scales, biases);
}
