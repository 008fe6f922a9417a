// tc_epilogue.cuh -- epilogues of the projections (decode and prefill), shared by the prefill
// GEMM (gemm_tc.cu), the cluster split-K decode kernel (gemm_csk.cu) and the 4-bit decode
// kernels (gemm_q4r.cu): RMSNorm scale, residual add with the next RMSNorm's statistics and
// operand, SwiGLU, and for QKV the RoPE rotation, the K/V append (or its quantisation) and the
// decode attention's Q operand image.
#pragma once
#include "kernels.h"
#include "tc_common.cuh"

namespace tcepi {

// Residual values out[tok0 + j][m] of tile row r for an EPI_ADD epilogue (columns jlo <= j <
// jhi), all loads issued before any is used (the epilogue's latency is a chain of global round
// trips otherwise).  EPI_T >= 0: the epilogue fixed at compile time (only its code is
// generated), else p.epi.
template <int CNT, int EPI_T = -1>
__device__ __forceinline__ void load_residual(const TcParams& p, int rb, int r, int tok0,
                                              float* res, int jlo = 0, int jhi = CNT) {
  const int epi = EPI_T >= 0 ? EPI_T : p.epi;
  const int m = rb * 128 + r;
#pragma unroll
  for (int j = 0; j < CNT; ++j) {
    const int t = tok0 + j;
    res[j] = (epi == EPI_ADD && m < p.M && t < p.n_act && j >= jlo && j < jhi)
                 ? __ldcg(p.out + (size_t)t * p.ldo + m)
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

// The new K/V of a quantised-KV engine, quantised where they are produced: tile row r holds dim
// i of a K or V head for the CNT decode rows (x[j], already rounded to bf16; rows jlo <= j <
// jhi are written).  Per row j and 64-dim group: L = 2^bits - 1, scale = bf16((max - min) / L),
// bias = bf16(min), code = clamp(rint((x - bias) / scale), 0, L) with the quotient the
// correctly rounded double one (q0 = d / s through the group's reciprocal, then one
// exact-residual correction: the reciprocal is computed once per (row, group) and the division
// of every element is three double operations instead of one).  The codes, scale and bias go
// to the row's quantised slab or page (kvq_jobs[j]); nothing is written in bf16.
template <int CNT>
__device__ __forceinline__ void kvq_append(const TcParams& p, int rb, int r, const float (&x)[CNT],
                                           float* swx, const EpiSrc& src, int jlo, int jhi) {
  const int hd = p.head_dim, bits = p.kvq_bits;
  const int row = rb * 128 + r, head = row / hd, i = row % hd;
  const bool isv = head >= p.n_heads + p.n_kv_heads;
  const int g = head - p.n_heads - (isv ? p.n_kv_heads : 0);
  const int lane = r & 31, wq = r >> 5, grp = r >> 6;  // 64-row groups of the tile
  const int L = (1 << bits) - 1;
  float mn[CNT], mx[CNT];
#pragma unroll
  for (int j = 0; j < CNT; ++j) mn[j] = mx[j] = x[j];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float a[CNT], b[CNT];
#pragma unroll
    for (int j = 0; j < CNT; ++j) {
      a[j] = __shfl_xor_sync(0xffffffffu, mn[j], o);
      b[j] = __shfl_xor_sync(0xffffffffu, mx[j], o);
    }
#pragma unroll
    for (int j = 0; j < CNT; ++j) {
      mn[j] = fminf(mn[j], a[j]);
      mx[j] = fmaxf(mx[j], b[j]);
    }
  }
  float* wmm = swx;                                   // [4 warps][CNT][min, max]
  float* gsb = swx + 8 * CNT;                         // [2 groups][CNT][scale, bias]
  double* ginv = reinterpret_cast<double*>(
      (reinterpret_cast<uintptr_t>(swx + 12 * CNT) + 7) & ~uintptr_t(7));  // [2 groups][CNT]
  tc::named_bar_sync(1, 128);  // the exchange buffer is free again
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < CNT; ++j) {
      wmm[(wq * CNT + j) * 2] = mn[j];
      wmm[(wq * CNT + j) * 2 + 1] = mx[j];
    }
  }
  tc::named_bar_sync(1, 128);
  const int jj = r & 63;  // thread jj of a group prepares row jj's scale, bias and reciprocal
  if (jj < CNT && jj >= jlo && jj < jhi) {
    const int w0 = 2 * grp, w1 = 2 * grp + 1;
    const float gmn = fminf(wmm[(w0 * CNT + jj) * 2], wmm[(w1 * CNT + jj) * 2]);
    const float gmx = fmaxf(wmm[(w0 * CNT + jj) * 2 + 1], wmm[(w1 * CNT + jj) * 2 + 1]);
    const uint16_t sb = f32_to_bf16((float)(((double)gmx - (double)gmn) / (double)L));
    const float sc = bf16_to_f32(sb);
    gsb[(grp * CNT + jj) * 2] = sc;
    gsb[(grp * CNT + jj) * 2 + 1] = bf16_to_f32(f32_to_bf16(gmn));
    ginv[grp * CNT + jj] = sc != 0.f ? 1.0 / (double)sc : 0.0;
  }
  tc::named_bar_sync(1, 128);
  uint8_t* arena8 = reinterpret_cast<uint8_t*>(p.arena);
  const int ng = hd / 64, gr = i / 64, row_bytes = hd * bits / 8;
#pragma unroll
  for (int j = 0; j < CNT; ++j) {
    if (j < jlo || j >= jhi) continue;
    const float sc = gsb[(grp * CNT + j) * 2], bi = gsb[(grp * CNT + j) * 2 + 1];
    uint32_t code = 0u;
    if (sc != 0.f) {
      const double s = sc, d = (double)x[j] - (double)bi, inv = ginv[grp * CNT + j];
      const double q0 = d * inv;
      const double q1 = fma(fma(-q0, s, d), inv, q0);  // the correctly rounded d / s
      const double t = rint(q1);
      code = t < 0.0 ? 0u : (t > (double)L ? (uint32_t)L : (uint32_t)t);
    }
    const Kv8Job jb = p.kvq_jobs[j];
    const long long loc = (long long)src.rows[j].pos - jb.dst_p0;
    const long long blk = kvq_block(jb.dst, jb.dst_cap, p.layer, isv ? 1 : 0, g, p.n_kv_heads, hd,
                                    bits);
    if (bits == 8) {
      arena8[blk + loc * row_bytes + i] = (uint8_t)code;
    } else {  // dims 2k (low nibble) and 2k + 1 are adjacent lanes
      const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
      if ((i & 1) == 0) arena8[blk + loc * row_bytes + (i >> 1)] = (uint8_t)(code | (hi << 4));
    }
    if ((i & 63) == 0) {
      uint16_t* sp = reinterpret_cast<uint16_t*>(arena8 + blk + (long long)jb.dst_cap * row_bytes);
      sp[loc * ng + gr] = f32_to_bf16(sc);
      sp[(long long)jb.dst_cap * ng + loc * ng + gr] = f32_to_bf16(bi);
    }
  }
}

// Final epilogue of CNT (<= 32) columns (tokens tok0 .. tok0+CNT-1) of tile row r of row
// block rb, of which columns jlo <= j < jhi are written.  All 128 epilogue threads call it
// together (it synchronises them on named barrier 1).  rinv (when p.ss_in) holds each column's RMSNorm factor; res the residual values from
// load_residual (EPI_ADD).  The tile's values are staged in swx ([row][CNT + 1]) and every
// per-column step below is a rolled loop over them: unrolled over 32 columns, the three store
// paths of a launch grow past the instruction cache and the epilogue waits on instruction
// fetches.
template <int CNT, int EPI_T = -1>
__device__ __forceinline__ void finish(const TcParams& p, int rb, int r, float* vals, int tok0,
                                       float* swx, const float* rinv, const float* res,
                                       const EpiSrc& src, int jlo = 0, int jhi = CNT) {
  const int epi = EPI_T >= 0 ? EPI_T : p.epi;
  constexpr int LD = CNT + 1;  // staged row pitch: a column's 32 rows sit in 32 banks
  if (p.ss_in) {
#pragma unroll
    for (int j = 0; j < CNT; ++j) vals[j] *= rinv[j];
  }
  const int n = min(jhi, p.n_act - tok0);  // columns [jlo, n) are tokens to write
  tc::named_bar_sync(1, 128);              // swx is free
  if (epi == EPI_QKV || epi == EPI_QKVQ) {
    // Row r of the tile is dim i of head `head` of q|k|v (heads are head_dim-aligned in the
    // tile); its RoPE partner is dim i ^ half of the same head, held by tile row r ^ half.
    const int hd = p.head_dim, half = hd >> 1;
    const int row = rb * 128 + r, head = row / hd, i = row % hd;
    const bool rope = head < p.n_heads + p.n_kv_heads;
#pragma unroll
    for (int j = 0; j < CNT; ++j) swx[r * LD + j] = vals[j];
    tc::named_bar_sync(1, 128);
    const int pr = r ^ half, ci = i & (half - 1);
    const int G = p.n_heads / p.n_kv_heads;
    // q and k turn by pos * theta^(-2(i%half)/hd)
    auto rotated = [&](int j) {
      float v = swx[r * LD + j];
      if (rope) {
        const float w = swx[pr * LD + j];
        const float c = src.cosv[j * half + ci], sn = src.sinv[j * half + ci];
        v = i < half ? v * c - w * sn : w * sn + v * c;
      }
      return v;
    };
    if (epi == EPI_QKVQ && rb * 128 >= p.n_heads * hd) {
      // a tile of K/V heads on a quantised-KV engine (uniform over the tile: the q rows end on
      // a 256-row boundary) quantises its rows once they are all rotated
      float xq[CNT];
#pragma unroll
      for (int j = 0; j < CNT; ++j)
        xq[j] = (j >= jlo && j < n && row < p.M) ? bf16_to_f32(f32_to_bf16(rotated(j))) : 0.f;
      kvq_append<CNT>(p, rb, r, xq, swx, src, jlo, n);
      return;
    }
    if (row >= p.M) return;
    if (head < p.n_heads) {
      // Q operand image of row j, kv head head / G: hi part in tile row head % G, lo part in
      // row 8 + head % G, scaled by 1/sqrt(head_dim)
      const size_t img = (size_t)16 * hd * 2;
      uint8_t* tile = p.qtile + (size_t)(head / G) * img;
      const uint32_t ohi = sw128_offset(head % G, i, 2048), olo = sw128_offset(8 + head % G, i, 2048);
      const float qs = rsqrtf((float)hd);
#pragma unroll 2
      for (int j = jlo; j < n; ++j) {
        const float qv = rotated(j) * qs;
        const uint16_t hi = f32_to_bf16(qv);
        uint8_t* t = tile + (size_t)j * p.n_kv_heads * img;
        *reinterpret_cast<uint16_t*>(t + ohi) = hi;
        *reinterpret_cast<uint16_t*>(t + olo) = f32_to_bf16(qv - bf16_to_f32(hi));
      }
    } else if (rope) {
#pragma unroll 2
      for (int j = jlo; j < n; ++j) {
        const QueryRow qr = src.rows[j];
        p.arena[k_index(qr, p.layer, head - p.n_heads, qr.pos, i, p.n_kv_heads, hd)] =
            f32_to_bf16(rotated(j));
      }
    } else {
#pragma unroll 2
      for (int j = jlo; j < n; ++j) {
        const QueryRow qr = src.rows[j];
        p.arena[v_index(qr, p.layer, head - p.n_heads - p.n_kv_heads, qr.pos, i, p.n_kv_heads,
                        hd)] = f32_to_bf16(swx[r * LD + j]);
      }
    }
    return;
  }
  if (epi != EPI_SWIGLU) {
    const int m = rb * 128 + r;
    const float gn = src.has_gn ? src.gn : load_next_gain(p, rb, r);
#pragma unroll
    for (int j = 0; j < CNT; ++j)
      swx[r * LD + j] = m < p.M ? (epi == EPI_ADD ? vals[j] + res[j] : vals[j]) : 0.f;
    if (m < p.M) {
#pragma unroll 2
      for (int j = jlo; j < n; ++j) {
        const size_t t = (size_t)(tok0 + j);
        const float v = swx[r * LD + j];
        p.out[t * p.ldo + m] = v;
        if (p.next_act) {  // the next projection's operand x * g, as hi/lo parts
          const float a = v * gn;
          const uint16_t hi = f32_to_bf16(a);
          p.next_act[t * p.ldo + m] = hi;
          if (p.next_lo) p.next_act[(p.next_lo + t) * p.ldo + m] = f32_to_bf16(a - bf16_to_f32(hi));
        }
      }
    }
    if (p.ss_out) {
      // sums of squares of the updated rows over this tile's 128 rows, for the next RMSNorm:
      // column j = r / 4; thread w = r % 4 adds rows 32 w .. 32 w + 31 (from row 32 w + w,
      // wrapping, so the four threads of a column read four banks), then (w0 + w1) + (w2 + w3)
      tc::named_bar_sync(1, 128);
      const int j = r >> 2, w = r & 3;
      float sq = 0.f;
      if (j >= jlo && j < n) {
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
          const float v = swx[(32 * w + ((k + w) & 31)) * LD + j];
          sq += v * v;
        }
      }
      sq += __shfl_xor_sync(0xffffffffu, sq, 1);
      sq += __shfl_xor_sync(0xffffffffu, sq, 2);
      if (w == 0 && j >= jlo && j < n) p.ss_out[(size_t)rb * p.ss_ld + tok0 + j] = sq;
    }
    return;
  }
  if (epi == EPI_SWIGLU) {
    // SwiGLU: tile rows 0..63 are gate rows, 64..127 the up rows of the same 64 features; two
    // threads per feature take alternate columns
#pragma unroll
    for (int j = 0; j < CNT; ++j) swx[r * LD + j] = vals[j];
    tc::named_bar_sync(1, 128);
    const int fr = r & 63, f = rb * 64 + fr;
    if (f < p.F) {
#pragma unroll 2
      for (int j = jlo + (r >> 6); j < n; j += 2) {
        const size_t t = (size_t)(tok0 + j);
        const float g = swx[fr * LD + j], u = swx[(64 + fr) * LD + j];
        const float a = g / (1.f + expf(-g)) * u;
        const uint16_t hi = f32_to_bf16(a);
        p.act[t * p.act_ld + f] = hi;
        if (p.act_lo) p.act[(p.act_lo + t) * p.act_ld + f] = f32_to_bf16(a - bf16_to_f32(hi));
      }
    }
  }
}

}  // namespace tcepi
