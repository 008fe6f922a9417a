// kv8.cu -- 8-bit affine KV (the mlx-bun batching design's quantised KV cache: affine groups of
// 64 values along head_dim, a bf16 scale and bias per group, as its 4-bit weights).
//
// An 8-bit slab holds, per (layer, K|V, kv head) block of a slab of capacity cap:
//   codes  [cap][head_dim]          uint8
//   scales [cap][head_dim / 64]     bf16
//   biases [cap][head_dim / 64]     bf16
// (kv8_block_bytes).  A value reads back as scale * code + bias.  Keys and values are both
// stored position-major: the attention below reads them on CUDA cores, one key per thread for
// the scores and one dimension per thread for P.V.
//
// Kernels:
//   k_quantize_kv8   rows of bf16 into codes / scales / biases (the quantiser, one warp a group)
//   k_kv8_convert    positions of bf16 slabs (or one-page staging slabs) into 8-bit slabs
//   k_attn_decode_kv8  split flash decoding over 8-bit slabs: one 128-key item per iteration of a
//                    persistent grid, partial (max, sum, output) per item and q head
//   k_attn_merge_kv8 the splits of each (row, q head) combined in item order
#include "kernels.h"

namespace {

constexpr int kItemKeys = 128;  // keys per attention item (one 128-key sub-chunk)
constexpr int kAttnThreads = 128;

// One warp quantises one group of 64 values; lane j holds values 2j and 2j + 1.  scale =
// bf16((max - min) / 255), bias = bf16(min), code = clamp(rint((x - bias) / scale), 0, 255)
// (0 when scale is 0); the code is decided in double.  Writes the lane's two codes as one
// 16-bit store and, from lane 0, the scale and bias.
CBT_D void quantize_group(float x0, float x1, uint8_t* codes, uint16_t* scale, uint16_t* bias,
                          int lane) {
  float mn = fminf(x0, x1), mx = fmaxf(x0, x1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  // (mx - mn) is exact in double; divide, round to float, then to bf16
  const uint16_t sb = f32_to_bf16((float)(((double)mx - (double)mn) / 255.0));
  const uint16_t bb = f32_to_bf16(mn);
  const double sc = bf16_to_f32(sb), bi = bf16_to_f32(bb);
  uint32_t q[2] = {0u, 0u};
  const float xs[2] = {x0, x1};
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (sc != 0.0) {
      const double t = rint(((double)xs[k] - bi) / sc);
      q[k] = t < 0.0 ? 0u : (t > 255.0 ? 255u : (uint32_t)t);
    }
  }
  reinterpret_cast<uint16_t*>(codes)[lane] = (uint16_t)(q[0] | (q[1] << 8));
  if (lane == 0) {
    *scale = sb;
    *bias = bb;
  }
}

__global__ void k_quantize_kv8(const uint16_t* x, int rows, int cols, uint8_t* codes,
                               uint16_t* scales, uint16_t* biases) {
  pdl_wait();
  pdl_launch();
  const int ng = cols / 64, lane = threadIdx.x & 31;
  const long long grp = blockIdx.x * (long long)(blockDim.x / 32) + threadIdx.x / 32;
  if (grp >= (long long)rows * ng) return;
  const long long r = grp / ng, g = grp % ng;
  const uint16_t* src = x + r * cols + g * 64;
  const uint32_t w = reinterpret_cast<const uint32_t*>(src)[lane];
  quantize_group(bf16_lo(w), bf16_hi(w), codes + r * cols + g * 64, scales + grp, biases + grp,
                 lane);
}

// block (layer, kv, head) of an 8-bit slab at byte offset `off` with layout capacity `cap`
CBT_D long long kv8_block(long long off, int cap, int layer, int kv, int head, int n_kv_heads,
                          int head_dim) {
  return off + (((long long)layer * 2 + kv) * n_kv_heads + head) * kv8_block_bytes(cap, head_dim);
}

// One warp per (job, position, layer, K|V, kv head, group of 64 dims).  Job j converts positions
// [t0, t0 + n) of layers [l0, l0 + nl).
__global__ void k_kv8_convert(const Kv8Job* jobs, int l0, int nl, int n_kv_heads, int head_dim,
                              uint8_t* arena) {
  pdl_wait();
  pdl_launch();
  const Kv8Job jb = jobs[blockIdx.y];
  const int ng = head_dim / 64, lane = threadIdx.x & 31;
  long long u = blockIdx.x * (long long)(blockDim.x / 32) + threadIdx.x / 32;
  if (u >= (long long)jb.n * nl * 2 * n_kv_heads * ng) return;
  const int gr = (int)(u % ng);
  u /= ng;
  const int g = (int)(u % n_kv_heads);
  u /= n_kv_heads;
  const int kv = (int)(u % 2);
  u /= 2;
  const int layer = l0 + (int)(u % nl);
  const int pos = jb.t0 + (int)(u / nl);
  const uint16_t* a16 = reinterpret_cast<const uint16_t*>(arena);
  const QueryRow src{jb.src_base, pos, jb.src_cap};
  const int d = gr * 64 + 2 * lane;
  float x0, x1;
  if (kv == 0) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(
        a16 + k_index(src, layer, g, pos, d, n_kv_heads, head_dim));
    x0 = bf16_lo(w);
    x1 = bf16_hi(w);
  } else {
    x0 = bf16_to_f32(a16[v_index(src, layer, g, pos, d, n_kv_heads, head_dim)]);
    x1 = bf16_to_f32(a16[v_index(src, layer, g, pos, d + 1, n_kv_heads, head_dim)]);
  }
  const long long blk = kv8_block(jb.dst, jb.dst_cap, layer, kv, g, n_kv_heads, head_dim);
  uint16_t* sc = reinterpret_cast<uint16_t*>(arena + blk + (long long)jb.dst_cap * head_dim);
  uint16_t* bi = sc + (long long)jb.dst_cap * ng;
  quantize_group(x0, x1, arena + blk + (long long)pos * head_dim + gr * 64, sc + (long long)pos * ng + gr,
                 bi + (long long)pos * ng + gr, lane);
}

template <int G, int HD>
struct AttnSmem {
  static constexpr int kPitch = HD + 16;  // bytes per key row of K codes (16-byte loads
                                          // from consecutive rows land in distinct banks)
  float q[G][HD];                         // the group's q heads, scaled by 1/sqrt(head_dim)
  float qsum[G][HD / 64];                 // their sums over each group of 64 dims
  float s[G][kItemKeys];                  // scores, then softmax weights
  float ksc[kItemKeys][HD / 64], kbi[kItemKeys][HD / 64];
  float vsc[kItemKeys][HD / 64], vbi[kItemKeys][HD / 64];
  float2 ml[G];
  alignas(16) uint8_t kc[kItemKeys * kPitch];
  alignas(16) uint8_t vc[kItemKeys * HD];
};

// One item (row b, kv head g, 128-key sub-chunk s0) per iteration.  Scores: thread j takes key
// j, s = sum over groups of scale * (q . codes) + bias * sum(q); softmax over the item's keys
// per q head; P.V: thread t takes dimension t.  Partial outputs are relative to the item's own
// running max; k_attn_merge_kv8 combines them.
template <int G, int HD>
__global__ void __launch_bounds__(kAttnThreads) k_attn_decode_kv8(Kv8AttnArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  auto& S = *reinterpret_cast<AttnSmem<G, HD>*>(smem_raw);
  constexpr int NG = HD / 64;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int qd = a.n_heads * HD, nqkv = qd + 2 * a.n_kv_heads * HD;
  const float inv_sqrt = rsqrtf((float)HD);
  pdl_wait();
  pdl_launch();
  const int total = *a.n_items;
  for (int it = blockIdx.x; it < total; it += gridDim.x) {
    const AttnItem w = a.items[it];
    const Kv8Job jb = a.rows[w.b];
    const int k0 = w.s0 * kItemKeys;
    const int nk = min(kItemKeys, jb.t0 + 1 - k0);
    if (w.s1 != w.s0 + 1 || nk <= 0) {  // the work list is built one sub-chunk per item
      if (t == 0) set_device_error(a.err, CBT_DEV_WORK_ITEM, it);
      continue;
    }
    // q of the group's heads (rotated in place by the RoPE kernel), and its group sums
    for (int i = t; i < G * HD; i += kAttnThreads) {
      const int h = i / HD, dd = i % HD;
      S.q[h][dd] = a.qkv[(long long)w.b * nqkv + (w.g * G + h) * HD + dd] * inv_sqrt;
    }
    // codes of the item's keys (16-byte loads), and their scales and biases
    const long long kblk = kv8_block(jb.dst, jb.dst_cap, a.layer, 0, w.g, a.n_kv_heads, HD);
    const long long vblk = kv8_block(jb.dst, jb.dst_cap, a.layer, 1, w.g, a.n_kv_heads, HD);
    for (int i = t; i < nk * (HD / 16); i += kAttnThreads) {
      const int j = i / (HD / 16), c = i % (HD / 16);
      const long long at = (long long)(k0 + j) * HD + c * 16;
      *reinterpret_cast<uint4*>(S.kc + j * S.kPitch + c * 16) =
          *reinterpret_cast<const uint4*>(a.arena + kblk + at);
      *reinterpret_cast<uint4*>(S.vc + j * HD + c * 16) =
          *reinterpret_cast<const uint4*>(a.arena + vblk + at);
    }
    for (int i = t; i < nk * NG; i += kAttnThreads) {
      const int j = i / NG, gr = i % NG;
      const long long gi = (long long)(k0 + j) * NG + gr;
      const uint16_t* ks = reinterpret_cast<const uint16_t*>(a.arena + kblk + (long long)jb.dst_cap * HD);
      const uint16_t* vs = reinterpret_cast<const uint16_t*>(a.arena + vblk + (long long)jb.dst_cap * HD);
      S.ksc[j][gr] = bf16_to_f32(ks[gi]);
      S.kbi[j][gr] = bf16_to_f32(ks[(long long)jb.dst_cap * NG + gi]);
      S.vsc[j][gr] = bf16_to_f32(vs[gi]);
      S.vbi[j][gr] = bf16_to_f32(vs[(long long)jb.dst_cap * NG + gi]);
    }
    __syncthreads();
    if (t < G * NG) {
      const int h = t / NG, gr = t % NG;
      float sum = 0.f;
      for (int i = 0; i < 64; ++i) sum += S.q[h][gr * 64 + i];
      S.qsum[h][gr] = sum;
    }
    __syncthreads();
    // scores: thread t takes key t
    {
      float acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = 0.f;
      if (t < nk) {
        const uint8_t* row = S.kc + t * S.kPitch;
#pragma unroll
        for (int gr = 0; gr < NG; ++gr) {
          float part[G];
#pragma unroll
          for (int h = 0; h < G; ++h) part[h] = 0.f;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + gr * 64 + c * 16);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e4 = 0; e4 < 4; ++e4) {
#pragma unroll
              for (int by = 0; by < 4; ++by) {
                const float code = (float)((wv[e4] >> (8 * by)) & 0xFFu);
                const int dd = gr * 64 + c * 16 + e4 * 4 + by;
#pragma unroll
                for (int h = 0; h < G; ++h) part[h] = fmaf(S.q[h][dd], code, part[h]);
              }
            }
          }
#pragma unroll
          for (int h = 0; h < G; ++h)
            acc[h] += S.ksc[t][gr] * part[h] + S.kbi[t][gr] * S.qsum[h][gr];
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) S.s[h][t] = t < nk ? acc[h] : -INFINITY;
    }
    __syncthreads();
    // softmax per q head: warp w takes heads w, w + 4, ...
    for (int h = warp; h < G; h += kAttnThreads / 32) {
      float m = -INFINITY;
      for (int j = lane; j < kItemKeys; j += 32) m = fmaxf(m, S.s[h][j]);
      m = warp_max(m);
      float l = 0.f;
      for (int j = lane; j < kItemKeys; j += 32) {
        const float p = j < nk ? expf(S.s[h][j] - m) : 0.f;
        S.s[h][j] = p;
        l += p;
      }
      l = warp_sum(l);
      if (lane == 0) S.ml[h] = make_float2(m, l);
    }
    __syncthreads();
    // P.V: thread t takes dimension t
    if (t < HD) {
      float acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = 0.f;
      const int gr = t / 64;
      for (int j = 0; j < nk; ++j) {
        const float v = fmaf(S.vsc[j][gr], (float)S.vc[j * HD + t], S.vbi[j][gr]);
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = fmaf(S.s[h][j], v, acc[h]);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) a.part_o[((long long)it * G + h) * HD + t] = acc[h];
    }
    if (t < G) a.part_ml[(long long)it * G + t] = S.ml[t];
    __syncthreads();  // shared memory is refilled by the next item
  }
}

// One block per (q head, row): the row's items for that head's kv head, combined in order.
__global__ void k_attn_merge_kv8(Kv8AttnArgs a, int G, int head_dim) {
  pdl_wait();
  pdl_launch();
  const int hq = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int g = hq / G, h = hq % G;
  const int cnt = a.item_count[b], base = a.item_base[b] + g * cnt;
  float M = -INFINITY;
  for (int sp = 0; sp < cnt; ++sp) M = fmaxf(M, a.part_ml[(long long)(base + sp) * G + h].x);
  float L = 0.f, acc = 0.f;
  for (int sp = 0; sp < cnt; ++sp) {
    const float2 ml = a.part_ml[(long long)(base + sp) * G + h];
    const float f = expf(ml.x - M);
    L += f * ml.y;
    acc += f * a.part_o[((long long)(base + sp) * G + h) * head_dim + d];
  }
  if (d < head_dim) a.o[(long long)b * a.n_heads * head_dim + hq * head_dim + d] = acc / L;
}

template <int G, int HD>
bool launch_attn_kv8_t(const Kv8AttnArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = sizeof(AttnSmem<G, HD>);
  // set on every launch: the attribute belongs to the current device's copy of the kernel
  if (cudaFuncSetAttribute(k_attn_decode_kv8<G, HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return false;
  const int per_sm = std::max(1, std::min(4, (int)((200u << 10) / smem)));
  if (launch_pdl(k_attn_decode_kv8<G, HD>, dim3(num_sms * per_sm), dim3(kAttnThreads), smem, s, a) !=
      cudaSuccess)
    return false;
  return launch_pdl(k_attn_merge_kv8, dim3(a.n_heads, a.B), dim3(HD), 0, s, a, G, HD) == cudaSuccess;
}

template <int HD>
bool launch_attn_kv8_hd(const Kv8AttnArgs& a, int G, int num_sms, cudaStream_t s) {
  switch (G) {
    case 1: return launch_attn_kv8_t<1, HD>(a, num_sms, s);
    case 2: return launch_attn_kv8_t<2, HD>(a, num_sms, s);
    case 4: return launch_attn_kv8_t<4, HD>(a, num_sms, s);
    case 8: return launch_attn_kv8_t<8, HD>(a, num_sms, s);
    default: return false;
  }
}

}  // namespace

void launch_quantize_kv8(const uint16_t* x, int rows, int cols, uint8_t* codes, uint16_t* scales,
                         uint16_t* biases, cudaStream_t s) {
  const long long groups = (long long)rows * (cols / 64);
  if (groups <= 0) return;
  launch_pdl(k_quantize_kv8, dim3((unsigned)((groups + 7) / 8)), dim3(256), 0, s, x, rows, cols,
             codes, scales, biases);
}

void launch_kv8_convert(const Kv8Job* jobs, int n_jobs, int max_n, int l0, int nl, int n_kv_heads,
                        int head_dim, uint8_t* arena, cudaStream_t s) {
  const long long units = (long long)max_n * nl * 2 * n_kv_heads * (head_dim / 64);
  if (units <= 0 || n_jobs <= 0) return;
  launch_pdl(k_kv8_convert, dim3((unsigned)((units + 7) / 8), n_jobs), dim3(256), 0, s, jobs, l0,
             nl, n_kv_heads, head_dim, arena);
}

bool launch_attn_decode_kv8(const Kv8AttnArgs& a, int num_sms, cudaStream_t s) {
  const int G = a.n_heads / a.n_kv_heads;
  if (a.head_dim == 64) return launch_attn_kv8_hd<64>(a, G, num_sms, s);
  if (a.head_dim == 128) return launch_attn_kv8_hd<128>(a, G, num_sms, s);
  return false;
}
