// kvq.cu -- affine KV of 8 or 4 bits (the mlx-bun batching design's quantised KV cache,
// "--kv-quant 4|8": affine groups of 64 values along head_dim, a bf16 scale and bias per group,
// as its weights; "quantized KV multiplies the budget (~4x at 4-bit)").
//
// A quantised slab (or page) of capacity cap holds, per (layer, K|V, kv head) block:
//   codes  [cap][head_dim * bits / 8]   uint8 (4 bits: element 2i in the low nibble of byte i)
//   scales [cap][head_dim / 64]         bf16
//   biases [cap][head_dim / 64]         bf16
// (kvq_block_bytes).  A value reads back as scale * code + bias.
//
// Kernels:
//   k_quantize_kv      rows of bf16 into codes / scales / biases (the quantiser, a warp a group)
//   k_kvq_convert      positions of bf16 slabs (or staging pages) into quantised slabs or pages
//   k_attn_decode_q    split flash decoding over quantised slabs on the tensor cores (mma.sync):
//                      a persistent grid over the decode work list, one 128-key item at a time
//                      while the next item's codes stream into the other shared-memory stage
//   k_attn_prefill_q   a prefill token's attention over quantised positions (CUDA cores): the
//                      chunks of a prompt that continue a quantised slab
//   k_kvq_export       quantised positions back to plain bf16 rows
#include <cuda_fp16.h>

#include "kernels.h"

namespace {

constexpr int kItemKeys = 128;  // keys per attention item (one 128-key sub-chunk)
constexpr int kAttnWarps = 8;                        // each takes 16 keys of an item
constexpr int kAttnThreads = 32 * kAttnWarps;
constexpr int kKeysPerWarp = kItemKeys / kAttnWarps;
constexpr int kNt = kKeysPerWarp / 8;                // score tiles (n8) per warp
constexpr int kKs = kKeysPerWarp / 16;               // P.V k16 steps per warp

// One warp quantises one group of 64 values; lane j holds values 2j and 2j + 1.  With
// L = 2^BITS - 1: scale = bf16((max - min) / L), bias = bf16(min), code = clamp(rint((x - bias) /
// scale), 0, L) (0 when scale is 0), decided in double.  Writes the lane's two codes (one
// 16-bit store at 8 bits, one byte at 4 bits) and, from lane 0, the scale and bias.
template <int BITS>
CBT_D void quantize_group(float x0, float x1, uint8_t* codes, uint16_t* scale, uint16_t* bias,
                          int lane) {
  float mn = fminf(x0, x1), mx = fmaxf(x0, x1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  constexpr int kLevels = (1 << BITS) - 1;
  // (mx - mn) is exact in double; divide, round to float, then to bf16
  const uint16_t sb = f32_to_bf16((float)(((double)mx - (double)mn) / (double)kLevels));
  const uint16_t bb = f32_to_bf16(mn);
  const double sc = bf16_to_f32(sb), bi = bf16_to_f32(bb);
  uint32_t q[2] = {0u, 0u};
  const float xs[2] = {x0, x1};
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (sc != 0.0) {
      const double t = rint(((double)xs[k] - bi) / sc);
      q[k] = t < 0.0 ? 0u : (t > (double)kLevels ? (uint32_t)kLevels : (uint32_t)t);
    }
  }
  if (BITS == 8)
    reinterpret_cast<uint16_t*>(codes)[lane] = (uint16_t)(q[0] | (q[1] << 8));
  else
    codes[lane] = (uint8_t)(q[0] | (q[1] << 4));
  if (lane == 0) {
    *scale = sb;
    *bias = bb;
  }
}

template <int BITS>
__global__ void k_quantize_kv(const uint16_t* x, int rows, int cols, uint8_t* codes,
                              uint16_t* scales, uint16_t* biases) {
  pdl_wait();
  pdl_launch();
  const int ng = cols / 64, lane = threadIdx.x & 31;
  const long long grp = blockIdx.x * (long long)(blockDim.x / 32) + threadIdx.x / 32;
  if (grp >= (long long)rows * ng) return;
  const long long r = grp / ng, g = grp % ng;
  const uint16_t* src = x + r * cols + g * 64;
  const uint32_t w = reinterpret_cast<const uint32_t*>(src)[lane];
  quantize_group<BITS>(bf16_lo(w), bf16_hi(w), codes + r * (cols * BITS / 8) + g * (8 * BITS),
                       scales + grp, biases + grp, lane);
}

// One warp per (job, position, layer, K|V, kv head, group of 64 dims).  Job j converts positions
// [t0, t0 + n) of layers [l0, l0 + nl) from its bf16 source into its quantised destination,
// whose position p sits at local index p - dst_p0.
template <int BITS>
__global__ void k_kvq_convert(const Kv8Job* jobs, int l0, int nl, int n_kv_heads, int head_dim,
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
  const long long loc = pos - jb.dst_p0;
  const int row_bytes = head_dim * BITS / 8;
  const long long blk = kvq_block(jb.dst, jb.dst_cap, layer, kv, g, n_kv_heads, head_dim, BITS);
  uint16_t* sc = reinterpret_cast<uint16_t*>(arena + blk + (long long)jb.dst_cap * row_bytes);
  uint16_t* bi = sc + (long long)jb.dst_cap * ng;
  quantize_group<BITS>(x0, x1, arena + blk + loc * row_bytes + gr * (8 * BITS), sc + loc * ng + gr,
                       bi + loc * ng + gr, lane);
}

// ---- decode attention over quantised KV on the tensor cores --------------------------------
CBT_D void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}
CBT_D void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
CBT_D void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// D += A B, m16n8k16, fp16 operands, fp32 accumulators
CBT_D void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two codes (low 16 bits: c0 | c1 << 8) as an fp16 pair holding exactly (c0, c1): the bytes
// become the low mantissa bits of 1024 + c (exponent bits 0x64), and 1024 is subtracted exactly.
CBT_D uint32_t codes8_to_half2(uint32_t c01) {
  const uint32_t h = __byte_perm(c01, 0x6464u, 0x5140u);
  const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(
                                                                   __ushort_as_half(0x6400u),
                                                                   __ushort_as_half(0x6400u)));
  return *reinterpret_cast<const uint32_t*>(&v);
}
// two 4-bit codes (c0 in bits 0..3, c1 in bits 16..19) the same way
CBT_D uint32_t codes4_to_half2(uint32_t c01) {
  const uint32_t h = c01 | 0x64006400u;
  const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&h), __halves2half2(
                                                                   __ushort_as_half(0x6400u),
                                                                   __ushort_as_half(0x6400u)));
  return *reinterpret_cast<const uint32_t*>(&v);
}
CBT_D uint32_t pack_half2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Shared memory of the decode attention: two stages (one item each) and the reductions.
template <int G, int HD, int BITS>
struct QAttnSmem {
  static constexpr int kRow = HD * BITS / 8;  // code bytes of one key
  static constexpr int kPitch = kRow + 16;    // padded: the fragment loads of a warp hit
                                              // distinct banks
  static constexpr int NG = HD / 64;
  struct Stage {
    alignas(16) uint8_t kc[kItemKeys * kPitch];
    alignas(16) uint8_t vc[kItemKeys * kPitch];
    alignas(16) uint16_t ks[kItemKeys * NG], kb[kItemKeys * NG];
    alignas(16) uint16_t vs[kItemKeys * NG], vb[kItemKeys * NG];
    alignas(16) uint8_t q[16 * HD * 2];  // the Q operand image (bf16 hi rows 0..7, lo 8..15)
  };
  Stage st[2];
  alignas(16) uint32_t qfrag[(HD / 16) * 32 * 4];  // the item's Q fragments, [k-step][lane][4]
  float qks[HD / 16][8];                           // sum of q over each k-step's dims, per head
  float ored[kAttnWarps][G][HD];  // per warp: its keys' share of P.V
  float redm[kAttnWarps][8], redl[kAttnWarps][8];
  float redb[kAttnWarps][8][NG];
};

// One item (row b, kv head g, 128-key sub-chunk s0) per iteration; each of the 8 warps takes
// 16 of its keys (16 w .. 16 w + 15), so a short chain per warp and 16 warps per SM.  Scores S[h][key] = sum over 64-dim groups of
// scale * (q . codes) + bias * sum(q): an m16n8k16 MMA per 16 dims and 8 keys, the A rows being
// the group's q heads as fp16 high parts (rows 0..7) and remainders (rows 8..15), the codes
// converted exactly to fp16, one accumulator per group folded with its key's scale and bias.
// Softmax per head over the item's keys.  P.V: for each group, p' = p * scale of the key is the
// A operand (fp16 high part + remainder rows), V's codes the B operand, and sum(p * bias) is
// added per group.  Partial outputs are relative to the item's own max; k_attn_merge combines
// them in item order.
template <int G, int HD, int BITS>
__global__ void __launch_bounds__(kAttnThreads)
    k_attn_decode_q(KvqAttnArgs a) {
  using S = QAttnSmem<G, HD, BITS>;
  constexpr int kRow = S::kRow, kPitch = S::kPitch, NG = S::NG;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;  // fragment row group and thread in group
  const int total = *a.n_items;  // step inputs (the work list): readable before the wait

  // stage an item: codes of its keys (rows past the row's position zero-filled), their scales
  // and biases (whole 16-byte chunks up to the last valid key; the rest masked later) -- and
  // its Q image (prefetch_q)
  auto prefetch_codes = [&](const AttnItem& w, int si) {
    const int nk = min(kItemKeys, w.n - w.s0 * kItemKeys);
    const long long loc = (long long)w.s0 * kItemKeys - w.p0;
    typename S::Stage& st = sm.st[si];
    const uint8_t* kblk = a.arena + kvq_block(w.kbase, w.cap, a.layer, 0, w.g, a.n_kv_heads, HD, BITS);
    const uint8_t* vblk = a.arena + kvq_block(w.kbase, w.cap, a.layer, 1, w.g, a.n_kv_heads, HD, BITS);
    constexpr int kChunks = kRow / 16;
    for (int i = tid; i < kItemKeys * kChunks; i += kAttnThreads) {
      const int key = i / kChunks, c = i % kChunks;
      const bool ok = key < nk;
      const long long at = ok ? (loc + key) * kRow + c * 16 : 0;
      cp_async16(st.kc + key * kPitch + c * 16, kblk + at, ok ? 16u : 0u);
      cp_async16(st.vc + key * kPitch + c * 16, vblk + at, ok ? 16u : 0u);
    }
    // scales / biases: kItemKeys * NG bf16 = 16 * NG chunks each
    const long long sc_off = (long long)w.cap * kRow;
    const long long bi_off = sc_off + (long long)w.cap * NG * 2;
    constexpr int kKeysPerChunk = 8 / NG;
    for (int i = tid; i < 4 * 16 * NG; i += kAttnThreads) {
      const int which = i / (16 * NG), c = i % (16 * NG);
      const bool ok = c * kKeysPerChunk < nk;
      const uint8_t* blk = which < 2 ? kblk : vblk;
      const long long off = ((which & 1) ? bi_off : sc_off) + loc * NG * 2 + c * 16;
      uint16_t* dst = which == 0 ? st.ks : which == 1 ? st.kb : which == 2 ? st.vs : st.vb;
      cp_async16(reinterpret_cast<uint8_t*>(dst) + c * 16, blk + (ok ? off : 0), ok ? 16u : 0u);
    }
  };
  auto prefetch_q = [&](const AttnItem& w, int si) {
    const uint8_t* qsrc = a.qtile + ((size_t)w.b * a.n_kv_heads + w.g) * (16 * HD * 2);
    for (int i = tid; i < 16 * HD * 2 / 16; i += kAttnThreads)
      cp_async16(sm.st[si].q + i * 16, qsrc + i * 16, 16u);
  };

  // The first item's codes are requested before waiting for the previous kernel when they were
  // written by earlier steps (the item does not hold the row's new position); its Q image, and
  // the codes of an item that holds the new position, after it.
  int si = 0;
  AttnItem wc{};
  bool codes_early = false;
  if ((int)blockIdx.x < total) {
    wc = a.items[blockIdx.x];
    if ((wc.s0 + 1) * kItemKeys < wc.n) {
      prefetch_codes(wc, 0);
      codes_early = true;
    }
  }
  pdl_wait();
  pdl_launch();
  if (tid == 0) stamp_begin(a.stamp);
  if ((int)blockIdx.x < total) {
    if (!codes_early) prefetch_codes(wc, 0);
    prefetch_q(wc, 0);
  }
  cp_async_commit();
  for (int it = blockIdx.x; it < total; it += gridDim.x, si ^= 1) {
    cp_async_wait_all();
    __syncthreads();  // stage si holds item it; every warp is done with the previous item
    // the next item's descriptor, requested now and used once this item's scores are done
    // (its copies then go out without a load round trip on the path)
    const int itn = it + (int)gridDim.x;
    AttnItem wn{};
    if (itn < total) wn = a.items[itn];
    typename S::Stage& st = sm.st[si];
    const AttnItem w = wc;
    const int n = w.n;
    const int nk = min(kItemKeys, n - w.s0 * kItemKeys);
    if (w.s1 != w.s0 + 1 || nk <= 0) {  // the work list is built one sub-chunk per item
      if (tid == 0) set_device_error(a.err, CBT_DEV_WORK_ITEM, it);
      if (itn < total) {
        prefetch_codes(wn, si ^ 1);
        prefetch_q(wn, si ^ 1);
      }
      cp_async_commit();
      wc = wn;
      continue;
    }
    // ---- Q fragments (head gq: high parts in A rows gq, remainders in rows gq + 8), built once
    // per item by the whole CTA: thread (k, l) converts fragment k of lane l and the k-step's
    // sum of q for head l / 4; contraction slots 2 tq, 2 tq + 1 (half 0) and 2 tq + 8, 2 tq + 9
    // (half 1) of k-step k hold dims 16 k + 4 tq + 2 half + {0, 1}: a thread's four dims are
    // consecutive, so one load gives its key codes (the same order on the K side below)
    if (tid < (HD / 16) * 32) {
      const int k = tid >> 5, fgq = lane >> 2, ftq = lane & 3;
      uint32_t f[4];
      float fs = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int d = 16 * k + 4 * ftq + 2 * half;
        const uint32_t hi = *reinterpret_cast<const uint32_t*>(st.q + sw128_offset(fgq, d, 2048));
        const uint32_t lo = *reinterpret_cast<const uint32_t*>(st.q + sw128_offset(8 + fgq, d, 2048));
        const float q0 = bf16_lo(hi) + bf16_lo(lo), q1 = bf16_hi(hi) + bf16_hi(lo);
        const __half2 h = __floats2half2_rn(q0, q1);
        const float2 hf = __half22float2(h);
        f[2 * half] = *reinterpret_cast<const uint32_t*>(&h);
        f[2 * half + 1] = pack_half2(q0 - hf.x, q1 - hf.y);
        fs += q0 + q1;
      }
      reinterpret_cast<uint4*>(sm.qfrag)[tid] = make_uint4(f[0], f[1], f[2], f[3]);
      fs += __shfl_xor_sync(0xffffffffu, fs, 1);
      fs += __shfl_xor_sync(0xffffffffu, fs, 2);
      if (ftq == 0) sm.qks[k][fgq] = fs;  // sum over the k-step's 16 dims of head fgq
    }
    __syncthreads();
    uint32_t qa[HD / 16][4];
    float qsum[NG];
#pragma unroll
    for (int k = 0; k < HD / 16; ++k) {
      const uint4 f = reinterpret_cast<const uint4*>(sm.qfrag)[k * 32 + lane];
      qa[k][0] = f.x;
      qa[k][1] = f.y;
      qa[k][2] = f.z;
      qa[k][3] = f.w;
    }
#pragma unroll
    for (int gr = 0; gr < NG; ++gr)  // the group's four k-steps, in order
      qsum[gr] = ((sm.qks[4 * gr][gq] + sm.qks[4 * gr + 1][gq]) + sm.qks[4 * gr + 2][gq]) +
                 sm.qks[4 * gr + 3][gq];
    // ---- scores of this warp's 16 keys: s[nt][j] is key 16 w + 8 nt + 2 tq + j, head gq
    float s[kNt][2];
#pragma unroll
    for (int nt = 0; nt < kNt; ++nt) s[nt][0] = s[nt][1] = 0.f;
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) {
      float acc[kNt][4];
#pragma unroll
      for (int nt = 0; nt < kNt; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int k = 4 * gr + kk;
#pragma unroll
        for (int nt = 0; nt < kNt; ++nt) {
          const uint8_t* row = st.kc + (kKeysPerWarp * warp + 8 * nt + gq) * kPitch;
          uint32_t b0, b1;
          if (BITS == 8) {  // codes of dims 16 k + 4 tq .. + 3
            const uint32_t c = *reinterpret_cast<const uint32_t*>(row + 16 * k + 4 * tq);
            b0 = codes8_to_half2(c);
            b1 = codes8_to_half2(c >> 16);
          } else {
            const uint32_t c = *reinterpret_cast<const uint16_t*>(row + 8 * k + 2 * tq);
            b0 = codes4_to_half2((c & 0xFu) | ((c & 0xF0u) << 12));
            b1 = codes4_to_half2(((c >> 8) & 0xFu) | ((c & 0xF000u) << 4));
          }
          mma_f16(acc[nt], qa[k], b0, b1);
        }
      }
#pragma unroll
      for (int nt = 0; nt < kNt; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int key = kKeysPerWarp * warp + 8 * nt + 2 * tq + j;
          const float sc = bf16_to_f32(st.ks[key * NG + gr]), bi = bf16_to_f32(st.kb[key * NG + gr]);
          s[nt][j] += sc * (acc[nt][j] + acc[nt][j + 2]) + bi * qsum[gr];
        }
    }
    if (itn < total) {  // the next item into the other stage (every warp is past its data)
      prefetch_codes(wn, si ^ 1);
      prefetch_q(wn, si ^ 1);
    }
    cp_async_commit();
    wc = wn;
    // ---- softmax of head gq over the item's keys
    float mx = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < kNt; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int key = kKeysPerWarp * warp + 8 * nt + 2 * tq + j;
        if (key >= nk) s[nt][j] = -INFINITY;
        mx = fmaxf(mx, s[nt][j]);
      }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (tq == 0) sm.redm[warp][gq] = mx;
    __syncthreads();
    float m = sm.redm[0][gq];
#pragma unroll
    for (int w = 1; w < kAttnWarps; ++w) m = fmaxf(m, sm.redm[w][gq]);
    float l = 0.f;
    float p[kNt][2];
#pragma unroll
    for (int nt = 0; nt < kNt; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        p[nt][j] = s[nt][j] == -INFINITY ? 0.f : __expf(s[nt][j] - m);
        l += p[nt][j];
      }
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (tq == 0) sm.redl[warp][gq] = l;
    // ---- P.V over this warp's keys, group by group
#pragma unroll
    for (int gr = 0; gr < NG; ++gr) {
      uint32_t pa[kKs][4];
      float bsum = 0.f;
#pragma unroll
      for (int ks = 0; ks < kKs; ++ks)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int nt = 2 * ks + half;
          float pv[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int key = kKeysPerWarp * warp + 8 * nt + 2 * tq + j;
            const bool ok = key < nk;  // masked keys may hold stale scales and biases
            pv[j] = ok ? p[nt][j] * bf16_to_f32(st.vs[key * NG + gr]) : 0.f;
            bsum += ok ? p[nt][j] * bf16_to_f32(st.vb[key * NG + gr]) : 0.f;
          }
          const __half2 h = __floats2half2_rn(pv[0], pv[1]);
          const float2 hf = __half22float2(h);
          pa[ks][2 * half] = *reinterpret_cast<const uint32_t*>(&h);
          pa[ks][2 * half + 1] = pack_half2(pv[0] - hf.x, pv[1] - hf.y);
        }
      bsum += __shfl_xor_sync(0xffffffffu, bsum, 1);
      bsum += __shfl_xor_sync(0xffffffffu, bsum, 2);
      if (tq == 0) sm.redb[warp][gq][gr] = bsum;
      // V codes: output tile t's column n is dim 64 gr + 8 n + t, so this thread's B column
      // (n = gq) in tiles 0..7 is the 8 consecutive dims from 64 gr + 8 gq: one load per key
      // row gives all eight tiles' codes
      float o[8][4];
#pragma unroll
      for (int t = 0; t < 8; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[t][i] = 0.f;
#pragma unroll
      for (int ks = 0; ks < kKs; ++ks) {
        const int key0 = kKeysPerWarp * warp + 16 * ks + 2 * tq;
        const int rows[4] = {key0, key0 + 1, key0 + 8, key0 + 9};
        uint32_t w[4][2];  // per row: codes of the 8 dims (8 bits: two words; 4 bits: one)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (BITS == 8) {
            const uint2 v = *reinterpret_cast<const uint2*>(st.vc + rows[r] * kPitch + 64 * gr + 8 * gq);
            w[r][0] = v.x;
            w[r][1] = v.y;
          } else {
            w[r][0] = *reinterpret_cast<const uint32_t*>(st.vc + rows[r] * kPitch + 32 * gr + 4 * gq);
            w[r][1] = 0u;
          }
        }
#pragma unroll
        for (int t = 0; t < 8; t += 2) {
          // b0 of tile t: (key0, key0 + 1) codes of dim t; b1: (key0 + 8, key0 + 9)
          uint32_t b[2][2];  // [tile t, t + 1][b0, b1]
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const uint32_t x = w[2 * hb][0], y = w[2 * hb + 1][0];
            if (BITS == 8) {
              const uint32_t xs = t < 4 ? x : w[2 * hb][1], ys = t < 4 ? y : w[2 * hb + 1][1];
              const int by = t & 3;  // bytes by and by + 1 of the rows' word
              const uint32_t u = __byte_perm(xs, ys, (uint32_t)(by | ((4 + by) << 4) | ((by + 1) << 8) |
                                                                ((5 + by) << 12)));
              b[0][hb] = codes8_to_half2(u);        // (x_t, y_t)
              b[1][hb] = codes8_to_half2(u >> 16);  // (x_t+1, y_t+1)
            } else {
              const int by = t >> 1;  // byte by holds dims t (low nibble) and t + 1 (high)
              const uint32_t u = __byte_perm(x, y, (uint32_t)(by | ((4 + by) << 8)));  // x.by in 0, y.by in 2
              b[0][hb] = codes4_to_half2(u & 0x000F000Fu);
              b[1][hb] = codes4_to_half2((u >> 4) & 0x000F000Fu);
            }
          }
          mma_f16(o[t], pa[ks], b[0][0], b[0][1]);
          mma_f16(o[t + 1], pa[ks], b[1][0], b[1][1]);
        }
      }
      if (gq < G) {  // rows gq (high parts) + gq + 8 (remainders): head gq
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int d0 = 64 * gr + 16 * tq + t;  // columns 2 tq and 2 tq + 1 of tile t
          sm.ored[warp][gq][d0] = o[t][0] + o[t][2];
          sm.ored[warp][gq][d0 + 8] = o[t][1] + o[t][3];
        }
      }
    }
    __syncthreads();
    // ---- this item's partial output per q head: the warps' shares in warp order
    for (int i = tid; i < G * HD; i += kAttnThreads) {
      const int h = i / HD, d = i % HD, gr = d / 64;
      float o = 0.f, bsum = 0.f;
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {  // the warps' shares in warp order
        o += sm.ored[w][h][d];
        bsum += sm.redb[w][h][gr];
      }
      o += bsum;
      a.part_o[((long long)it * G + h) * HD + d] = o;
    }
    if (tid < G) {
      float mm = sm.redm[0][tid], ll = 0.f;
#pragma unroll
      for (int w = 1; w < kAttnWarps; ++w) mm = fmaxf(mm, sm.redm[w][tid]);
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) ll += sm.redl[w][tid];
      a.part_ml[(long long)it * G + tid] = make_float2(mm, ll);
    }
  }
  cp_async_wait_all();  // no copy in flight at exit
  if (tid == 0) stamp_end(a.stamp);
}

template <int G, int HD, int BITS>
bool launch_attn_q_t(const KvqAttnArgs& a, int num_sms, cudaStream_t s) {
  const size_t smem = sizeof(QAttnSmem<G, HD, BITS>);
  // set on every launch: the attribute belongs to the current device's copy of the kernel
  if (cudaFuncSetAttribute(k_attn_decode_q<G, HD, BITS>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return false;
  const int per_sm = std::max(1, std::min(4, (int)((224u << 10) / (smem + 1024))));
  return launch_pdl(k_attn_decode_q<G, HD, BITS>, dim3(num_sms * per_sm), dim3(kAttnThreads),
                    smem, s, a) == cudaSuccess;
}

template <int HD, int BITS>
bool launch_attn_q_hd(const KvqAttnArgs& a, int G, int num_sms, cudaStream_t s) {
  switch (G) {
    case 1: return launch_attn_q_t<1, HD, BITS>(a, num_sms, s);
    case 2: return launch_attn_q_t<2, HD, BITS>(a, num_sms, s);
    case 4: return launch_attn_q_t<4, HD, BITS>(a, num_sms, s);
    case 8: return launch_attn_q_t<8, HD, BITS>(a, num_sms, s);
    default: return false;
  }
}

// ---- prefill attention over quantised positions (CUDA cores) ----------------------------------
// One block per (token, q head): token t attends to positions [0, pos_t] of its sequence, whose
// quantised pages (or one slab) are at qpages[tok_first[t] + key / cap_t] (byte offsets).
template <int BITS>
__global__ void k_attn_prefill_q(const float* qkv, const QueryRow* rows, const long long* qpages,
                                 const int* tok_first, const int* tok_cap, int layer, int n_heads,
                                 int n_kv_heads, int head_dim, const uint8_t* arena, float* o) {
  pdl_wait();
  pdl_launch();
  extern __shared__ float sc[];  // [head_dim] q, then the scores
  float* q = sc;
  float* sco = sc + head_dim;
  __shared__ float red[32];
  const int t = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int G = n_heads / n_kv_heads, g = h / G;
  const int qd = n_heads * head_dim, nqkv = qd + 2 * n_kv_heads * head_dim;
  const int n = rows[t].pos + 1, cap = tok_cap[t], first = tok_first[t];
  const int ng = head_dim / 64, row_bytes = head_dim * BITS / 8;
  const float inv_sqrt = rsqrtf((float)head_dim);
  for (int d = tid; d < head_dim; d += blockDim.x) q[d] = qkv[(long long)t * nqkv + h * head_dim + d];
  __syncthreads();
  auto code_at = [&](const uint8_t* c, int d) -> int {
    if (BITS == 8) return c[d];
    return (c[d >> 1] >> (4 * (d & 1))) & 0xF;
  };
  float mx = -INFINITY;
  for (int key = tid; key < n; key += blockDim.x) {
    const long long blk = kvq_block(qpages[first + key / cap], cap, layer, 0, g, n_kv_heads,
                                    head_dim, BITS);
    const int loc = key % cap;
    const uint8_t* c = arena + blk + (long long)loc * row_bytes;
    const uint16_t* s16 = reinterpret_cast<const uint16_t*>(arena + blk + (long long)cap * row_bytes);
    const uint16_t* b16 = s16 + (long long)cap * ng;
    float acc = 0.f;
    for (int gr = 0; gr < ng; ++gr) {
      float qc = 0.f, qs = 0.f;
      for (int i = 0; i < 64; ++i) {
        qc = fmaf(q[gr * 64 + i], (float)code_at(c, gr * 64 + i), qc);
        qs += q[gr * 64 + i];
      }
      acc += bf16_to_f32(s16[loc * ng + gr]) * qc + bf16_to_f32(b16[loc * ng + gr]) * qs;
    }
    acc *= inv_sqrt;
    sco[key] = acc;
    mx = fmaxf(mx, acc);
  }
  mx = warp_max(mx);
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  if (tid < 32) {
    float v = tid < (int)(blockDim.x >> 5) ? red[tid] : -INFINITY;
    v = warp_max(v);
    if (tid == 0) red[0] = v;
  }
  __syncthreads();
  mx = red[0];
  __syncthreads();
  float l = 0.f;
  for (int key = tid; key < n; key += blockDim.x) {
    const float p = __expf(sco[key] - mx);
    sco[key] = p;
    l += p;
  }
  l = warp_sum(l);
  if ((tid & 31) == 0) red[tid >> 5] = l;
  __syncthreads();
  if (tid < 32) {
    float v = tid < (int)(blockDim.x >> 5) ? red[tid] : 0.f;
    v = warp_sum(v);
    if (tid == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = 1.f / red[0];
  for (int d = tid; d < head_dim; d += blockDim.x) {
    const int gr = d / 64;
    float acc = 0.f;
    for (int key = 0; key < n; ++key) {
      const long long blk = kvq_block(qpages[first + key / cap], cap, layer, 1, g, n_kv_heads,
                                      head_dim, BITS);
      const int loc = key % cap;
      const uint8_t* c = arena + blk + (long long)loc * row_bytes;
      const uint16_t* s16 = reinterpret_cast<const uint16_t*>(arena + blk + (long long)cap * row_bytes);
      const uint16_t* b16 = s16 + (long long)cap * ng;
      const float v = bf16_to_f32(s16[loc * ng + gr]) * (float)code_at(c, d) +
                      bf16_to_f32(b16[loc * ng + gr]);
      acc = fmaf(sco[key], v, acc);
    }
    o[(long long)t * qd + h * head_dim + d] = acc * inv;
  }
}

// ---- export: quantised positions [0, n) of one layer as plain bf16 [n_kv_heads][n][head_dim] --
// value = bf16(fp32(scale * code + bias)), the product and sum evaluated in double
template <int BITS>
__global__ void k_kvq_export(const uint8_t* arena, const long long* pages, int cap, int layer,
                             int n_kv_heads, int head_dim, int n, uint16_t* k, uint16_t* v) {
  pdl_wait();
  pdl_launch();
  const long long tot = (long long)n_kv_heads * n * head_dim;
  const int ng = head_dim / 64, row_bytes = head_dim * BITS / 8;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < tot;
       i += (long long)gridDim.x * blockDim.x) {
    const int d = (int)(i % head_dim);
    const int pos = (int)((i / head_dim) % n);
    const int g = (int)(i / ((long long)head_dim * n));
    const int loc = pos % cap;
    for (int kv = 0; kv < 2; ++kv) {
      const long long blk = kvq_block(pages[pos / cap], cap, layer, kv, g, n_kv_heads, head_dim, BITS);
      const uint8_t* c = arena + blk + (long long)loc * row_bytes;
      const uint16_t* s16 = reinterpret_cast<const uint16_t*>(arena + blk + (long long)cap * row_bytes);
      const uint16_t* b16 = s16 + (long long)cap * ng;
      const int code = BITS == 8 ? c[d] : (c[d >> 1] >> (4 * (d & 1))) & 0xF;
      const double val = (double)bf16_to_f32(s16[loc * ng + d / 64]) * code +
                         (double)bf16_to_f32(b16[loc * ng + d / 64]);
      (kv ? v : k)[i] = f32_to_bf16(__double2float_rn(val));
    }
  }
}

}  // namespace

bool launch_quantize_kv(const uint16_t* x, int rows, int cols, int bits, uint8_t* codes,
                        uint16_t* scales, uint16_t* biases, cudaStream_t s) {
  const long long groups = (long long)rows * (cols / 64);
  if (groups <= 0) return true;
  const dim3 grid((unsigned)((groups + 7) / 8));
  if (bits == 8)
    return launch_pdl(k_quantize_kv<8>, grid, dim3(256), 0, s, x, rows, cols, codes, scales,
                      biases) == cudaSuccess;
  if (bits == 4)
    return launch_pdl(k_quantize_kv<4>, grid, dim3(256), 0, s, x, rows, cols, codes, scales,
                      biases) == cudaSuccess;
  return false;
}

bool launch_kvq_convert(const Kv8Job* jobs, int n_jobs, int max_n, int l0, int nl, int n_kv_heads,
                        int head_dim, int bits, uint8_t* arena, cudaStream_t s) {
  const long long units = (long long)max_n * nl * 2 * n_kv_heads * (head_dim / 64);
  if (units <= 0 || n_jobs <= 0) return true;
  const dim3 grid((unsigned)((units + 7) / 8), n_jobs);
  if (bits == 8)
    return launch_pdl(k_kvq_convert<8>, grid, dim3(256), 0, s, jobs, l0, nl, n_kv_heads, head_dim,
                      arena) == cudaSuccess;
  if (bits == 4)
    return launch_pdl(k_kvq_convert<4>, grid, dim3(256), 0, s, jobs, l0, nl, n_kv_heads, head_dim,
                      arena) == cudaSuccess;
  return false;
}

bool launch_attn_decode_q(const KvqAttnArgs& a, int bits, int num_sms, cudaStream_t s) {
  if (a.n_heads % a.n_kv_heads) return false;
  const int G = a.n_heads / a.n_kv_heads;
  if (bits == 8) {
    if (a.head_dim == 64) return launch_attn_q_hd<64, 8>(a, G, num_sms, s);
    if (a.head_dim == 128) return launch_attn_q_hd<128, 8>(a, G, num_sms, s);
  } else if (bits == 4) {
    if (a.head_dim == 64) return launch_attn_q_hd<64, 4>(a, G, num_sms, s);
    if (a.head_dim == 128) return launch_attn_q_hd<128, 4>(a, G, num_sms, s);
  }
  return false;
}

bool launch_attn_prefill_q(const float* qkv, const QueryRow* rows, const long long* qpages,
                           const int* tok_first, const int* tok_cap, int n, int layer, int n_heads,
                           int n_kv_heads, int head_dim, int max_keys, int bits,
                           const uint8_t* arena, float* o, cudaStream_t s) {
  if (n <= 0) return true;
  const size_t smem = sizeof(float) * (size_t)(head_dim + max_keys);
  auto kern = bits == 8 ? k_attn_prefill_q<8> : k_attn_prefill_q<4>;
  if (bits != 8 && bits != 4) return false;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return false;
  return launch_pdl(kern, dim3(n, n_heads), dim3(128), smem, s, qkv, rows, qpages, tok_first,
                    tok_cap, layer, n_heads, n_kv_heads, head_dim, arena, o) == cudaSuccess;
}

bool launch_kvq_export(const uint8_t* arena, const long long* pages, int cap, int layer,
                       int n_kv_heads, int head_dim, int n, int bits, uint16_t* k, uint16_t* v,
                       cudaStream_t s) {
  const long long tot = (long long)n_kv_heads * n * head_dim;
  if (tot <= 0) return true;
  const dim3 grid((unsigned)std::min<long long>((tot + 255) / 256, 4096));
  if (bits == 8)
    return launch_pdl(k_kvq_export<8>, grid, dim3(256), 0, s, arena, pages, cap, layer,
                      n_kv_heads, head_dim, n, k, v) == cudaSuccess;
  if (bits == 4)
    return launch_pdl(k_kvq_export<4>, grid, dim3(256), 0, s, arena, pages, cap, layer,
                      n_kv_heads, head_dim, n, k, v) == cudaSuccess;
  return false;
}
