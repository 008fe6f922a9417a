// tc_epilogue.cuh -- epilogues of the tensor-core projections (decode and prefill), shared by
// the stream-K kernel (gemm_tc.cu) and the cluster split-K kernel (gemm_csk.cu): RMSNorm scale,
// residual add with the next RMSNorm's statistics and operand, SwiGLU, and for QKV the RoPE
// rotation, the K/V append and the decode attention's Q operand image.
#pragma once
#include "kernels.h"
#include "tc_common.cuh"

namespace tcepi {

// Residual values out[tok0 + j][m] of tile row r for an EPI_ADD epilogue, all loads issued
// before any is used (the epilogue's latency is a chain of global round trips otherwise)
template <int CNT>
__device__ __forceinline__ void load_residual(const TcParams& p, int rb, int r, int tok0,
                                              float* res) {
  const int m = rb * 128 + r;
#pragma unroll
  for (int j = 0; j < CNT; ++j) {
    const int t = tok0 + j;
    res[j] = (p.epi == EPI_ADD && m < p.M && t < p.n_act) ? __ldcg(p.out + (size_t)t * p.ldo + m)
                                                          : 0.f;
  }
}

// Where finish() reads the values it needs besides the accumulator: the row table and the RoPE
// cos/sin (global memory, or shared-memory copies), and optionally the next RMSNorm gain of
// this thread's output row, loaded earlier (each global load here is a round trip at the end
// of the projection, when latency is all that is left).
struct EpiSrc {
  const QueryRow* rows;  // [n_act]
  const float* cosv;     // [n_act][head_dim / 2]
  const float* sinv;
  float gn;              // next_gain[m] (valid when has_gn)
  bool has_gn;
};

__device__ __forceinline__ EpiSrc epi_src_global(const TcParams& p) {
  return EpiSrc{p.rows, p.cosv, p.sinv, 0.f, false};
}

// next_gain of tile row r of row block rb (EPI_ADD with a next operand), 0 otherwise
__device__ __forceinline__ float load_next_gain(const TcParams& p, int rb, int r) {
  const int m = rb * 128 + r;
  return (p.next_act && m < p.M) ? bf16_to_f32(p.next_gain[m]) : 0.f;
}

// Final epilogue of CNT (<= 32) columns (tokens tok0 .. tok0+CNT-1) of tile row r of row
// block rb.  All 128 epilogue threads call it together.  rinv (when p.ss_in) holds each
// column's RMSNorm factor; res the residual values from load_residual (EPI_ADD).
template <int CNT>
__device__ __forceinline__ void finish(const TcParams& p, int rb, int r, float* vals, int tok0,
                                       float* swx, const float* rinv, const float* res,
                                       const EpiSrc& src) {
  if (p.ss_in) {
#pragma unroll
    for (int j = 0; j < CNT; ++j) vals[j] *= rinv[j];
  }
  if (p.epi == EPI_QKV) {
    // Row r of the tile is dim i of head `head` of q|k|v (heads are head_dim-aligned in the
    // tile); its RoPE partner is dim i ^ half of the same head, held by tile row r ^ half.
    const int hd = p.head_dim, half = hd >> 1;
    const int row = rb * 128 + r, head = row / hd, i = row % hd;
    const bool rope = head < p.n_heads + p.n_kv_heads;
    float cs[CNT], sn[CNT];
#pragma unroll
    for (int j = 0; j < CNT; ++j) {
      const bool ok = rope && j < p.n_act;
      cs[j] = ok ? src.cosv[j * half + (i & (half - 1))] : 1.f;
      sn[j] = ok ? src.sinv[j * half + (i & (half - 1))] : 0.f;
    }
    tc::named_bar_sync(1, 128);
#pragma unroll
    for (int j = 0; j < CNT; ++j) swx[r * (CNT + 1) + j] = vals[j];
    tc::named_bar_sync(1, 128);
    const int pr = r ^ half;
    const int G = p.n_heads / p.n_kv_heads;
#pragma unroll
    for (int j = 0; j < CNT; ++j) {
      if (j >= p.n_act || row >= p.M) break;
      float v = vals[j];
      if (rope) {  // q and k turn by pos * theta^(-2(i%half)/hd)
        const float w = swx[pr * (CNT + 1) + j];
        v = i < half ? v * cs[j] - w * sn[j] : w * sn[j] + v * cs[j];
      }
      if (head < p.n_heads) {
        // Q operand image of row j, kv head head / G: hi part in tile row head % G, lo part
        // in row 8 + head % G, scaled by 1/sqrt(head_dim)
        uint8_t* tile = p.qtile + ((size_t)j * p.n_kv_heads + head / G) * (16 * hd * 2);
        const float qv = v * rsqrtf((float)hd);
        const uint16_t hi = f32_to_bf16(qv);
        *reinterpret_cast<uint16_t*>(tile + sw128_offset(head % G, i, 2048)) = hi;
        *reinterpret_cast<uint16_t*>(tile + sw128_offset(8 + head % G, i, 2048)) =
            f32_to_bf16(qv - bf16_to_f32(hi));
      } else {
        const QueryRow qr = src.rows[j];
        if (head < p.n_heads + p.n_kv_heads)
          p.arena[k_index(qr, p.layer, head - p.n_heads, qr.pos, i, p.n_kv_heads, hd)] =
              f32_to_bf16(v);
        else
          p.arena[v_index(qr, p.layer, head - p.n_heads - p.n_kv_heads, qr.pos, i, p.n_kv_heads,
                          hd)] = f32_to_bf16(v);
      }
    }
    return;
  }
  if (p.epi != EPI_SWIGLU) {
    const int m = rb * 128 + r;
    const float gn = src.has_gn ? src.gn : load_next_gain(p, rb, r);
    float sq[CNT];
#pragma unroll
    for (int j = 0; j < CNT; ++j) {
      const int t = tok0 + j;
      sq[j] = 0.f;
      if (m < p.M && t < p.n_act) {
        const float v = p.epi == EPI_ADD ? vals[j] + res[j] : vals[j];
        p.out[(size_t)t * p.ldo + m] = v;
        sq[j] = v * v;
        if (p.next_act) {  // the next projection's operand x * g, as hi/lo parts
          const float a = v * gn;
          const uint16_t hi = f32_to_bf16(a);
          p.next_act[(size_t)t * p.ldo + m] = hi;
          if (p.next_lo)
            p.next_act[(size_t)(p.next_lo + t) * p.ldo + m] = f32_to_bf16(a - bf16_to_f32(hi));
        }
      }
    }
    if (p.ss_out) {
      // sums of squares of the updated rows over this tile's 128 rows, for the next RMSNorm;
      // the CNT warp reductions interleaved level by level, so their shuffles overlap
      const int w = r >> 5, lane = r & 31;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float t[CNT];
#pragma unroll
        for (int j = 0; j < CNT; ++j) t[j] = __shfl_xor_sync(0xffffffffu, sq[j], o);
#pragma unroll
        for (int j = 0; j < CNT; ++j) sq[j] += t[j];
      }
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < CNT; ++j) swx[w * 32 + j] = sq[j];
      }
      tc::named_bar_sync(1, 128);
      if (r < CNT && tok0 + r < p.n_act)
        p.ss_out[(size_t)rb * p.ss_ld + tok0 + r] = swx[r] + swx[32 + r] + swx[64 + r] + swx[96 + r];
      tc::named_bar_sync(1, 128);
    }
    return;
  }
  // SwiGLU: tile rows 0..63 are gate rows, 64..127 the up rows of the same 64 features
  tc::named_bar_sync(1, 128);
  if (r >= 64) {
#pragma unroll
    for (int j = 0; j < CNT; ++j) swx[(r - 64) * (CNT + 1) + j] = vals[j];
  }
  tc::named_bar_sync(1, 128);
  if (r < 64) {
    const int f = rb * 64 + r;
    if (f < p.F) {
#pragma unroll
      for (int j = 0; j < CNT; ++j) {
        const int t = tok0 + j;
        if (t < p.n_act) {
          const float g = vals[j], u = swx[r * (CNT + 1) + j];
          const float a = g / (1.f + expf(-g)) * u;
          const uint16_t hi = f32_to_bf16(a);
          p.act[(size_t)t * p.act_ld + f] = hi;
          if (p.act_lo) p.act[(size_t)(p.act_lo + t) * p.act_ld + f] = f32_to_bf16(a - bf16_to_f32(hi));
        }
      }
    }
  }
}

}  // namespace tcepi
