// gemm_q4r.cu -- decode projections y = x W^T over 4-bit affine weights (groups of 64 columns,
// w = s * q + b with q in 0..15 and bf16 s, b), dequantised in registers.
//
// A decode step has few rows (B <= 32), so the contraction is a weight stream: every weight is
// used by at most B operand rows.  Here the codes never leave the registers between the load and
// the multiply:
//   * each warp copies its 32 rows of a 128-row x 128-column weight block (2 KB of codes plus
//     the rows' scales and biases) into a private shared-memory ring with cp.async, three
//     blocks ahead, so no other warp ever waits for it;
//   * it turns each pair of codes into one bf16x2 register holding (128 + q, 128 + q') -- the
//     codes sit in the low mantissa bits of 128.0, so the values are exact -- and feeds them as
//     the A fragment of mma.sync m16n8k16 (A from registers is what keeps the dequantisation
//     in registers; tcgen05 takes A only from shared or tensor memory);
//   * the B fragment is the operand, 8 rows per n8 block (bf16 hi parts, then lo parts, so the
//     operand carries fp32-grade precision), staged once per CTA in shared memory for the
//     CTA's whole k-range together with each operand row's sum over every group of 64 columns;
//   * every group of 64 columns is its own accumulation, folded in with the row's scale and
//     bias in fp32:  y += s * sum_k (128 + q_k) x_k  +  (b - 128 s) * sum_k x_k.
// No dequantised weight is rounded; the result is that of the exact dequantised weights and
// the fp32 operand up to fp32 accumulation.
//
// Work split (the cluster split-K of the bf16 decode projections): tile t of 128 rows belongs
// to cluster t % NC; rank r of the cluster takes superblocks [r SB / C, (r + 1) SB / C) of its
// tiles; inside a CTA, warps 0-3 take the first half of those superblocks and warps 4-7 the
// second half, warp w holding tile rows 32 (w % 4) .. + 31 as two m16 row blocks that share
// the operand fragments.  The two halves meet in shared memory, the C ranks in the tile
// owner's shared memory (st.async, added in rank order), and the owner's warps 0-3 run the
// shared epilogue (RMSNorm scale, residual add and the next norm's statistics and operand,
// SwiGLU, RoPE + K/V append + the attention's Q operand).  C is chosen from the matrix shape
// and the number of clusters of C CTAs that fit on the GPU at once.
//
// Up to 8 batch rows (k_q4_rd): the operand slice of the CTA's whole k-range is staged in
// shared memory once, with its group sums.  9 to 32 rows (k_q4_rs): 16 rows (32 operand
// columns) per pass over the weights (gridDim.y passes); the slice no longer fits, so the
// operand streams superblock by superblock through a ring shared by the four warps of a set,
// whose 128 threads also add up that superblock's group sums (two barriers per superblock).
// A row's arithmetic -- the k split, the group order, the fold, the order in which its group
// sums are added -- depends on the matrix shape alone (MMA columns do not mix), so a row's
// result does not depend on how many rows share the step, nor on which kernel takes it.
//
// The weights are the native block layout of gemm_q4.cu: per (128-row tile, 128-column
// superblock) [4 chunks][128 rows][16 bytes] of codes (chunk c holds columns 32c .. 32c + 31 of
// a row as four words; word i's pair p: bits 4p..4p+3 column 8i + 2p, bits 16+4p..19+4p column
// 8i + 2p + 1), then [128 rows][s0, b0, s1, b1] bf16.
#include <algorithm>
#include <map>
#include <tuple>

#include "csk_common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_epilogue.cuh"

namespace {

constexpr int kWarps = 8;                // two sets of 4 warps, one per half of the k-range
constexpr int kThreads = 32 * kWarps;
constexpr int kRows = 32;                // tile rows per warp (two m16 row blocks)
constexpr int kDepth = 4;                // ring slots per warp (kDepth - 1 blocks in flight)
constexpr int kChunkPitch = 576;         // a ring chunk: 32 rows x 16 bytes, padded so the
                                         // fragment loads of one half-warp hit 32 distinct banks
constexpr int kScaleOff = 4 * kChunkPitch;
constexpr int kStage = kScaleOff + kRows * 8;  // codes of 32 rows, then their scales and biases
constexpr int kCodeBytes = 128 * 64;
constexpr int kMaxSlots = 4;
constexpr int kMaxSbPerRank = 24;        // bounds the operand slice kept in shared memory
constexpr int kSmemBudget = 227 * 1024;
constexpr int kMaxSsTiles = 64;          // RMSNorm statistics tiles (d_model <= 8192)

struct Q4rPlan {
  int C;       // CTAs per cluster (split of the k-range)
  int NC;      // clusters
  int slots;   // inbox slots: most tiles one CTA owns
  int sb_max;  // most superblocks of one rank
};

__host__ __device__ constexpr size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// Shared-memory carve-up for N operand columns (H = N / 2 batch rows)
struct Layout {
  size_t ring, xs, xsum, sacc, inbox, swx, rinv, cosv, sinv, rows, ssq, bars, flags, total;
  int pitch;  // bytes per operand row of xs
};

__host__ __device__ inline Layout layout(int N, const Q4rPlan& q) {
  const int H = N / 2;
  Layout L;
  L.pitch = q.sb_max * 256 + 16;  // == 16 (mod 128): conflict-free 16-byte fragment loads
  size_t o = 0;
  L.ring = o;
  o += (size_t)kWarps * kDepth * kStage;
  L.xs = o;
  o = align16(o + (size_t)N * L.pitch);
  L.xsum = o;
  o = align16(o + (size_t)2 * q.sb_max * N * 4);
  L.sacc = o;
  o = align16(o + (size_t)2 * 2 * 128 * H * 4);  // [tile parity][warp set][128 rows][H]
  L.inbox = o;
  o = align16(o + (size_t)q.slots * (q.C > 1 ? q.C - 1 : 0) * 128 * H * 4);
  L.swx = o;
  o = align16(o + (size_t)(128 * (H + 1) + 32) * 4);
  L.rinv = o;
  o = align16(o + 32 * 4);
  L.cosv = o;
  o = align16(o + (size_t)H * 64 * 4);
  L.sinv = o;
  o = align16(o + (size_t)H * 64 * 4);
  L.rows = o;
  o = align16(o + (size_t)8 * sizeof(QueryRow));
  L.ssq = o;
  o = align16(o + (size_t)kMaxSsTiles * 8 * 4);
  L.bars = o;
  o = align16(o + kMaxSlots * 8);
  L.flags = o;
  o += 16;
  L.total = o;
  return L;
}

// 16 bytes global -> shared (L2 only); src_bytes < 16: the rest of the 16 bytes are zero-filled
__device__ __forceinline__ void cp_async16_zfill_s(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
// 16 bytes global -> shared (L2 only), with an L2 eviction policy
__device__ __forceinline__ void cp_async16s(uint32_t dst, const void* src, uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "l"(pol)
               : "memory");
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// D += A B for one m16n8k16 tile: bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// the same with a zero accumulator in
__device__ __forceinline__ void mma16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                           uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// (a & m) | c in one logic op; m and c are held in registers (opaque_const), so each pair of
// codes costs one shift and this one instruction
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t m, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(m), "r"(c));
  return r;
}
// a constant the compiler keeps in a register instead of re-creating it at every use
__device__ __forceinline__ uint32_t opaque_const(uint32_t v) {
  uint32_t r;
  asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(v));
  return r;
}
// pair p of a native code word as a bf16x2 word (128 + q_even, 128 + q_odd): the codes sit in
// the low mantissa bits of 128.0 (m = 0x000F000F, c = 0x43004300)
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w, int p, uint32_t m, uint32_t c) {
  return and_or(w >> (4 * p), m, c);
}

// sum of 32 consecutive bf16 operand values (four 16-byte pieces) in index order; a group's
// sum over its 64 columns is (first 32) + (last 32) in both kernels
__device__ __forceinline__ float sum32(const uint4* v) {
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 u = v[c];
    s += bf16_lo(u.x);
    s += bf16_hi(u.x);
    s += bf16_lo(u.y);
    s += bf16_hi(u.y);
    s += bf16_lo(u.z);
    s += bf16_hi(u.z);
    s += bf16_lo(u.w);
    s += bf16_hi(u.w);
  }
  return s;
}

__device__ __forceinline__ void report_timeout(const TcParams& p, volatile int* abort, int role) {
  *abort = 1;
  if (atomicCAS(p.err, 0, CBT_DEV_TIMEOUT) == 0) p.err[1] = 500 + role;
}

// The projection's parameters for batch rows [R pass, R pass + R): every per-row pointer moves
// to the pass's first row; lo-part row offsets are absolute and stay.
__device__ __forceinline__ TcParams pass_params(const TcParams& p0, int pass, int R) {
  TcParams p = p0;
  const int r0 = R * pass;
  p.n_act = min(R, p0.n_act - r0);
  if (p.out) p.out += (size_t)r0 * p.ldo;
  if (p.next_act) p.next_act += (size_t)r0 * p.ldo;
  if (p.act) p.act += (size_t)r0 * p.act_ld;
  if (p.ss_in) p.ss_in += r0;
  if (p.ss_out) p.ss_out += r0;
  if (p.rows) p.rows += r0;
  if (p.cosv) p.cosv += (size_t)r0 * (p.head_dim / 2);
  if (p.sinv) p.sinv += (size_t)r0 * (p.head_dim / 2);
  if (p.qtile) p.qtile += (size_t)r0 * p.n_kv_heads * 16 * p.head_dim * 2;
  if (p.kvq_jobs) p.kvq_jobs += r0;
  return p;
}

// ---- k_q4_rd: up to 8 rows, the operand slice staged once ------------------------------------
// One CTA: k-range [sb0, sb1) of tiles cid, cid + NC, ... for batch rows [8 y, 8 y + 8).
// NB8 n8 blocks of operand columns: NB8 = 1 takes up to 4 rows (hi parts in columns 0-3, lo
// parts in 4-7), NB8 = 2 up to 8 rows (hi block, then lo block).
template <int NB8>
__global__ void __launch_bounds__(kThreads, 1)
    k_q4_rd(const __grid_constant__ TcParams p0, const uint16_t* __restrict__ x, int x_lo,
            const Q4rPlan q) {
  constexpr int N = 8 * NB8, H = N / 2;
  extern __shared__ __align__(16) uint8_t smem[];
  const Layout L = layout(N, q);
  uint8_t* ring = smem + L.ring;
  uint8_t* xs = smem + L.xs;
  float* xsum = reinterpret_cast<float*>(smem + L.xsum);
  float* sacc = reinterpret_cast<float*>(smem + L.sacc);
  float* inbox = reinterpret_cast<float*>(smem + L.inbox);
  float* swx = reinterpret_cast<float*>(smem + L.swx);
  float* rinv = reinterpret_cast<float*>(smem + L.rinv);
  float* scos = reinterpret_cast<float*>(smem + L.cosv);
  float* ssin = reinterpret_cast<float*>(smem + L.sinv);
  QueryRow* srows = reinterpret_cast<QueryRow*>(smem + L.rows);
  float* ssq = reinterpret_cast<float*>(smem + L.ssq);
  uint64_t* inbox_full = reinterpret_cast<uint64_t*>(smem + L.bars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.flags);

  const int pass = blockIdx.y;
  const TcParams p = pass_params(p0, pass, 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int C = q.C;
  const uint32_t rank = C > 1 ? csk::cluster_rank() : 0u;
  const int cid = blockIdx.x / C, NC = gridDim.x / C;
  const int Tc = cid < p.RB ? (p.RB - cid + NC - 1) / NC : 0;
  const int SB = p.K / 128;
  const int sb0 = (int)((long long)rank * SB / C);
  const int sb1 = (int)((long long)(rank + 1) * SB / C);
  const int nsb = sb1 - sb0;
  const int owned = Tc > (int)rank ? (Tc - (int)rank + C - 1) / C : 0;
  const int pitch = nsb * 256 + 16;
  // warp set h takes local superblocks [kbase, kbase + nh) of every tile; warp w of a set holds
  // tile rows 32 w .. 32 w + 31
  const int h = warp >> 2, rw = kRows * (warp & 3);
  const int n0 = (nsb + 1) >> 1;
  const int nh = h ? nsb - n0 : n0, kbase = h ? n0 : 0;
  const int nst = Tc * nh;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxSlots; ++s) tc::mbar_init(&inbox_full[s], 1);
    if (C > 1)
      for (int s = 0; s < owned; ++s)
        tc::mbar_expect_tx(&inbox_full[s], (uint32_t)((C - 1) * 128 * H * 4));
    abort_flag[0] = 0;
    tc::mbar_fence_init();
  }
  __syncthreads();
  if (C > 1) csk::cluster_sync();
  pdl_launch();

  // ---- weight blocks: this warp's 16 rows, kDepth - 1 blocks ahead (weights only: these may
  // be requested before the previous kernel has finished)
  const uint32_t wring = tc::smem_u32(ring) + (uint32_t)(warp * kDepth * kStage);
  // issue cursor: this lane's source addresses in the next block (code row rw + lane of each
  // chunk; lanes 0-15 also 16 bytes of the rows' scales and biases), and its ring slot
  const uint8_t* blk0 = p.wq + ((size_t)cid * SB + sb0 + kbase) * kQ4BlockBytes;
  const uint8_t* pcode = blk0 + (rw + lane) * 16;
  const uint8_t* pscale = blk0 + kCodeBytes + rw * 8 + (lane & 15) * 16;
  const size_t tile_skip = ((size_t)NC * SB - nh) * kQ4BlockBytes;  // last block -> next tile
  // the weights are read once per step: first out of L2
  const uint64_t pol_w = tc::policy_evict_first();
  int is_n = 0, is_k = 0;
  uint32_t is_dst = wring + lane * 16;
  const uint32_t ring_end = wring + kDepth * kStage;
  auto issue = [&]() {
    if (is_n < nst) {
      cp_async16s(is_dst, pcode, pol_w);
      cp_async16s(is_dst + kChunkPitch, pcode + 2048, pol_w);
      cp_async16s(is_dst + 2 * kChunkPitch, pcode + 2 * 2048, pol_w);
      cp_async16s(is_dst + 3 * kChunkPitch, pcode + 3 * 2048, pol_w);
      if (lane < 16) cp_async16s(is_dst + kScaleOff, pscale, pol_w);
      pcode += kQ4BlockBytes;
      pscale += kQ4BlockBytes;
      if (++is_k == nh) {
        is_k = 0;
        pcode += tile_skip;
        pscale += tile_skip;
      }
      ++is_n;
      is_dst += kStage;
      if (is_dst >= ring_end) is_dst -= kDepth * kStage;
    }
    cp_async_commit();
  };
  for (int s = 0; s < kDepth - 1; ++s) issue();

  pdl_wait();
  if (threadIdx.x == 0) stamp_begin(p.stamp);
  // ---- the operand slice of this k-range (zero columns past the pass's rows), all pieces in
  // flight at once; RMSNorm factors and the QKV epilogue's per-row inputs meanwhile
  {
    const int per_row = nsb * 16;  // 16-byte pieces; warp w copies operand rows w, w + 8, ...
    for (int n = warp; n < N; n += kWarps) {
      const int b = n % H;
      const bool valid = b < p.n_act;
      const size_t row = n >= H ? (size_t)(x_lo + 8 * pass + b) : (size_t)(8 * pass + b);
      const uint16_t* src = x + row * p.K + (size_t)sb0 * 128;
      const uint32_t dst = tc::smem_u32(xs + (size_t)n * pitch);
      for (int c = lane; c < per_row; c += 32)
        cp_async16_zfill_s(dst + c * 16, valid ? src + c * 8 : x, valid ? 16u : 0u);
    }
    cp_async_commit();
  }
  // the folded RMSNorm's per-tile sums of squares: every value requested at once (one per
  // thread), added up in tile order after the barrier
  if (p.ss_in)
    for (int i = threadIdx.x; i < p.ss_tiles * p.n_act; i += kThreads) {
      const int tt = i / p.n_act, b = i - tt * p.n_act;
      ssq[i] = __ldcg(p.ss_in + (size_t)tt * p.ss_ld + b);
    }
  tcepi::EpiSrc src = tcepi::epi_src_global(p);
  if (p.epi == EPI_QKV || p.epi == EPI_QKVQ) {
    const int half = p.head_dim >> 1;
    for (int i = threadIdx.x; i < p.n_act * half; i += kThreads) {
      scos[i] = p.cosv[i];
      ssin[i] = p.sinv[i];
    }
    if (threadIdx.x < p.n_act) srows[threadIdx.x] = p.rows[threadIdx.x];
    src.rows = srows;
    src.cosv = scos;
    src.sinv = ssin;
  }
  cp_async_wait<0>();  // the operand slice (and the weight blocks requested before it)
  __syncthreads();
  if (p.ss_in && threadIdx.x < p.n_act) {
    float s = 0.f;
    for (int tt = 0; tt < p.ss_tiles; ++tt) s += ssq[tt * p.n_act + threadIdx.x];
    rinv[threadIdx.x] = rsqrtf(s / (float)p.K + p.eps);
  }
  // each operand column's sum over every group of 64 columns, in a fixed order
  for (int idx = threadIdx.x; idx < 2 * nsb * N; idx += kThreads) {
    const int gl = idx / N, n = idx - gl * N;
    const uint4* v = reinterpret_cast<const uint4*>(xs + (size_t)n * pitch + gl * 128);
    xsum[gl * N + n] = sum32(v) + sum32(v + 4);
  }
  __syncthreads();

  float y[2][NB8][4];  // [row block u][n8 block][fragment]
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int nb = 0; nb < NB8; ++nb)
#pragma unroll
      for (int c = 0; c < 4; ++c) y[u][nb][c] = 0.f;
  // per-lane views: code words of rows 16u + g / 16u + g + 8 (chunk 2G + t/2, half t&1),
  // scales, operand
  const uint32_t lane_w = (t >> 1) * kChunkPitch + g * 16 + 8 * (t & 1);
  const uint32_t xlane = tc::smem_u32(xs) + (uint32_t)(g * pitch + 32 * t + kbase * 256);
  const uint32_t xsl = tc::smem_u32(xsum) + (uint32_t)((2 * kbase * N + 2 * t) * 4);
  const uint32_t pitch8 = 8u * (uint32_t)pitch;
  uint32_t st = wring;  // the ring slot consumed next
  const uint32_t km = opaque_const(0x000F000Fu), kc = opaque_const(0x43004300u);
  for (int j = 0; j < Tc; ++j) {
    float res[H];
    const uint32_t owner = (uint32_t)(j % C);
    if (warp < 4 && rank == owner) {  // epilogue inputs of this tile, requested early
      const int rb = cid + j * NC;
      tcepi::load_residual<H>(p, rb, threadIdx.x, 0, res);
      src.gn = tcepi::load_next_gain(p, rb, threadIdx.x);
      src.has_gn = true;
    }
    for (int k = 0; k < nh; ++k) {
      issue();
      cp_async_wait<kDepth - 1>();  // block of this stage has landed (this lane's copies) ...
      __syncwarp();                 // ... and every lane's
      uint2 sv[2][2];               // [u][row g, row g + 8]: (s0, b0), (s1, b1)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        sv[u][0] = lds64(st + kScaleOff + (16 * u + g) * 8);
        sv[u][1] = lds64(st + kScaleOff + (16 * u + g + 8) * 8);
      }
#pragma unroll
      for (int G = 0; G < 2; ++G) {
        // operand fragments of group G (both row blocks use them): column nb * 8 + g, the
        // sixteen columns 64 G + 16 t .. + 15 as bf16 pairs, 8 per MMA pair jp
        const uint32_t xg = xlane + k * 256 + G * 128;
        uint4 xv[2][NB8];
        float2 X[NB8];
#pragma unroll
        for (int nb = 0; nb < NB8; ++nb) {
          xv[0][nb] = lds128(xg + nb * pitch8);
          xv[1][nb] = lds128(xg + nb * pitch8 + 16);
          const uint2 Xw = lds64(xsl + ((2 * k + G) * N + nb * 8) * 4);
          X[nb] = make_float2(__uint_as_float(Xw.x), __uint_as_float(Xw.y));
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          // lane (g, t): columns 64 G + 16 t .. + 15 of rows 16u + g and 16u + g + 8
          const uint32_t wa = st + lane_w + G * 2 * kChunkPitch + u * 256;
          const uint2 wA = lds64(wa), wB = lds64(wa + 128);
          float acc[NB8][4];
#pragma unroll
          for (int jp = 0; jp < 2; ++jp) {
            // word jp holds columns 16 t + 8 jp .. + 7: MMA 2 jp takes its pairs 0 and 1,
            // MMA 2 jp + 1 its pairs 2 and 3 (k index 2t, 2t+1 -> first pair, 2t+8, 2t+9 ->
            // second)
            const uint32_t a = jp ? wA.y : wA.x, b = jp ? wB.y : wB.x;
            const uint32_t A0[4] = {unpack_pair(a, 0, km, kc), unpack_pair(b, 0, km, kc),
                                    unpack_pair(a, 1, km, kc), unpack_pair(b, 1, km, kc)};
            const uint32_t A1[4] = {unpack_pair(a, 2, km, kc), unpack_pair(b, 2, km, kc),
                                    unpack_pair(a, 3, km, kc), unpack_pair(b, 3, km, kc)};
#pragma unroll
            for (int nb = 0; nb < NB8; ++nb) {
              if (jp == 0) mma16816_z(acc[nb], A0, xv[0][nb].x, xv[0][nb].y);
              else mma16816(acc[nb], A0, xv[jp][nb].x, xv[jp][nb].y);
              mma16816(acc[nb], A1, xv[jp][nb].z, xv[jp][nb].w);
            }
          }
          const uint32_t swa = G ? sv[u][0].y : sv[u][0].x, swb = G ? sv[u][1].y : sv[u][1].x;
          const float s_a = bf16_lo(swa), s_b = bf16_lo(swb);
          const float c_a = fmaf(-128.f, s_a, bf16_hi(swa));
          const float c_b = fmaf(-128.f, s_b, bf16_hi(swb));
#pragma unroll
          for (int nb = 0; nb < NB8; ++nb) {
            y[u][nb][0] = fmaf(s_a, acc[nb][0], fmaf(c_a, X[nb].x, y[u][nb][0]));
            y[u][nb][1] = fmaf(s_a, acc[nb][1], fmaf(c_a, X[nb].y, y[u][nb][1]));
            y[u][nb][2] = fmaf(s_b, acc[nb][2], fmaf(c_b, X[nb].x, y[u][nb][2]));
            y[u][nb][3] = fmaf(s_b, acc[nb][3], fmaf(c_b, X[nb].y, y[u][nb][3]));
          }
        }
      }
      st += kStage;
      if (st >= ring_end) st = wring;
      __syncwarp();  // the slot is refilled by the next iteration's copies
    }

    // ---- end of tile j: hi + lo parts into the warp set's half of the hand-off buffer
    float* sa = sacc + (size_t)((j & 1) * 2 + h) * 128 * H;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r0 = rw + 16 * u + g;
      if constexpr (NB8 == 1) {
        float v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) v[c] = y[u][0][c] + __shfl_xor_sync(0xffffffffu, y[u][0][c], 2);
        if (t < 2) {
          *reinterpret_cast<float2*>(sa + r0 * H + 2 * t) = make_float2(v[0], v[1]);
          *reinterpret_cast<float2*>(sa + (r0 + 8) * H + 2 * t) = make_float2(v[2], v[3]);
        }
      } else {
#pragma unroll
        for (int nb = 0; nb < NB8 / 2; ++nb) {
          const float* lo = y[u][nb + NB8 / 2];
          *reinterpret_cast<float2*>(sa + r0 * H + nb * 8 + 2 * t) =
              make_float2(y[u][nb][0] + lo[0], y[u][nb][1] + lo[1]);
          *reinterpret_cast<float2*>(sa + (r0 + 8) * H + nb * 8 + 2 * t) =
              make_float2(y[u][nb][2] + lo[2], y[u][nb][3] + lo[3]);
        }
      }
#pragma unroll
      for (int nb = 0; nb < NB8; ++nb)
#pragma unroll
        for (int c = 0; c < 4; ++c) y[u][nb][c] = 0.f;
    }
    tc::named_bar_sync(2, kThreads);
    if (warp < 4) {
      // ---- tile row r: both halves, then the cluster's partials, then the epilogue
      const int r = threadIdx.x;
      const float* s0 = sacc + (size_t)((j & 1) * 2) * 128 * H + r * H;
      const float* s1 = s0 + 128 * H;
      float vals[H];
#pragma unroll
      for (int b = 0; b < H; ++b) vals[b] = s0[b] + s1[b];
      const int rb = cid + j * NC;
      float sum[H];
      const int got = csk::combine_partials<H>(vals, sum, inbox, inbox_full, j / C, rank, owner,
                                               C, r, abort_flag);
      if (got < 0) report_timeout(p, abort_flag, 1);
      tc::named_bar_sync(1, 128);  // the same decision in all 128 threads
      if (got > 0 && *abort_flag == 0) tcepi::finish<H>(p, rb, r, sum, 0, swx, rinv, res, src);
    }
  }
  cp_async_wait<0>();  // (only empty groups remain: every issued block was consumed)
  if (threadIdx.x == 0) stamp_end(p.stamp);
  if (C > 1 && threadIdx.x == 0)
    for (int s = 0; s < owned; ++s) tc::mbar_wait(&inbox_full[s], 0);
  if (C > 1) csk::cluster_sync();
}

// ---- k_q4_rs: 9 to 32 rows, 16 per pass, the operand streamed ------------------------------
constexpr int kRsN = 32;                 // operand columns of a pass: 16 rows, hi and lo parts
constexpr int kRsH = kRsN / 2;
constexpr int kRsDepth = 3;              // ring slots per warp (weights) and per set (operand)
constexpr int kXPitch = 272;             // bytes per operand row of a ring slot (128 bf16 + 16:
                                         // conflict-free 16-byte fragment loads)
constexpr int kXSlot = kRsN * kXPitch;   // one operand ring slot: 32 rows of one superblock

struct LayoutRs {
  size_t ring, xr, xsb, sacc, inbox, swx, rinv, cosv, sinv, rows, ssq, bars, flags, total;
};

__host__ __device__ inline LayoutRs layout_rs(const Q4rPlan& q) {
  constexpr int N = kRsN, H = kRsH;
  LayoutRs L;
  size_t o = 0;
  L.ring = o;
  o += (size_t)kWarps * kRsDepth * kStage;
  L.xr = o;  // [warp set][slot][N rows][kXPitch]
  o = align16(o + (size_t)2 * kRsDepth * kXSlot);
  L.xsb = o;  // [warp set][parity][group][N]: group sums of two consecutive superblocks
  o = align16(o + (size_t)2 * 2 * 2 * N * 4);
  L.sacc = o;
  o = align16(o + (size_t)2 * 2 * 128 * H * 4);  // [tile parity][warp set][128 rows][H]
  L.inbox = o;
  o = align16(o + (size_t)q.slots * (q.C > 1 ? q.C - 1 : 0) * 128 * H * 4);
  L.swx = o;
  o = align16(o + (size_t)(128 * (H + 1) + 32) * 4);
  L.rinv = o;
  o = align16(o + 32 * 4);
  L.cosv = o;
  o = align16(o + (size_t)H * 64 * 4);
  L.sinv = o;
  o = align16(o + (size_t)H * 64 * 4);
  L.rows = o;
  o = align16(o + (size_t)H * sizeof(QueryRow));
  L.ssq = o;
  o = align16(o + (size_t)kMaxSsTiles * H * 4);
  L.bars = o;
  o = align16(o + kMaxSlots * 8);
  L.flags = o;
  o += 16;
  L.total = o;
  return L;
}

// One CTA: k-range [sb0, sb1) of tiles cid, cid + NC, ... for batch rows [16 y, 16 y + 16).
// The work split, the weight ring, the MMAs and the fold are those of k_q4_rd at four n8
// blocks (hi parts of the 16 rows, then their lo parts); per superblock the set's threads wait
// for their copies of this superblock and the next, meet at the set's barrier (both have
// landed, the slots of the superblock before are free), issue the copies kRsDepth - 1
// superblocks ahead, add up the next superblock's 64 group sums (a pair of threads per sum;
// this superblock's were added in the previous iteration), then multiply.
__global__ void __launch_bounds__(kThreads, 1)
    k_q4_rs(const __grid_constant__ TcParams p0, const uint16_t* __restrict__ x, int x_lo,
            const Q4rPlan q) {
  constexpr int NB8 = 4, N = kRsN, H = kRsH;
  constexpr int kXPieces = N * 16 / 128;  // 16-byte operand pieces per thread of a set
  extern __shared__ __align__(16) uint8_t smem[];
  const LayoutRs L = layout_rs(q);
  uint8_t* ring = smem + L.ring;
  float* sacc = reinterpret_cast<float*>(smem + L.sacc);
  float* inbox = reinterpret_cast<float*>(smem + L.inbox);
  float* swx = reinterpret_cast<float*>(smem + L.swx);
  float* rinv = reinterpret_cast<float*>(smem + L.rinv);
  float* scos = reinterpret_cast<float*>(smem + L.cosv);
  float* ssin = reinterpret_cast<float*>(smem + L.sinv);
  QueryRow* srows = reinterpret_cast<QueryRow*>(smem + L.rows);
  float* ssq = reinterpret_cast<float*>(smem + L.ssq);
  uint64_t* inbox_full = reinterpret_cast<uint64_t*>(smem + L.bars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.flags);

  const int pass = blockIdx.y;
  const TcParams p = pass_params(p0, pass, H);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int C = q.C;
  const uint32_t rank = C > 1 ? csk::cluster_rank() : 0u;
  const int cid = blockIdx.x / C, NC = gridDim.x / C;
  const int Tc = cid < p.RB ? (p.RB - cid + NC - 1) / NC : 0;
  const int SB = p.K / 128;
  const int sb0 = (int)((long long)rank * SB / C);
  const int sb1 = (int)((long long)(rank + 1) * SB / C);
  const int nsb = sb1 - sb0;
  const int owned = Tc > (int)rank ? (Tc - (int)rank + C - 1) / C : 0;
  // warp set h takes local superblocks [kbase, kbase + nh) of every tile; warp w of a set holds
  // tile rows 32 w .. 32 w + 31
  const int h = warp >> 2, rw = kRows * (warp & 3);
  const int n0 = (nsb + 1) >> 1;
  const int nh = h ? nsb - n0 : n0, kbase = h ? n0 : 0;
  const int nst = Tc * nh;
  uint8_t* xr = smem + L.xr + (size_t)h * kRsDepth * kXSlot;  // this set's operand ring
  float* xsb = reinterpret_cast<float*>(smem + L.xsb) + h * 2 * 2 * N;
  const int bar = 3 + h;  // the set's named barrier

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxSlots; ++s) tc::mbar_init(&inbox_full[s], 1);
    if (C > 1)
      for (int s = 0; s < owned; ++s)
        tc::mbar_expect_tx(&inbox_full[s], (uint32_t)((C - 1) * 128 * H * 4));
    abort_flag[0] = 0;
    tc::mbar_fence_init();
  }
  // operand rows past the pass's rows are zero in every slot (no copy ever writes them)
  for (int i = threadIdx.x; i < 2 * kRsDepth * N * (kXPitch / 16); i += kThreads) {
    const int n = (i / (kXPitch / 16)) % N;
    if (n % H >= p.n_act)
      reinterpret_cast<uint4*>(smem + L.xr)[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  if (C > 1) csk::cluster_sync();
  pdl_launch();

  // ---- weight blocks: this warp's 32 rows, kRsDepth - 1 blocks ahead (weights only: these may
  // be requested before the previous kernel has finished)
  const uint32_t wring = tc::smem_u32(ring) + (uint32_t)(warp * kRsDepth * kStage);
  const uint8_t* blk0 = p.wq + ((size_t)cid * SB + sb0 + kbase) * kQ4BlockBytes;
  const uint8_t* pcode = blk0 + (rw + lane) * 16;
  const uint8_t* pscale = blk0 + kCodeBytes + rw * 8 + (lane & 15) * 16;
  const size_t tile_skip = ((size_t)NC * SB - nh) * kQ4BlockBytes;  // last block -> next tile
  const uint64_t pol_w = tc::policy_evict_first();
  int is_n = 0, is_k = 0;
  uint32_t is_dst = wring + lane * 16;
  const uint32_t ring_end = wring + kRsDepth * kStage;
  auto issue_w = [&]() {
    if (is_n < nst) {
      cp_async16s(is_dst, pcode, pol_w);
      cp_async16s(is_dst + kChunkPitch, pcode + 2048, pol_w);
      cp_async16s(is_dst + 2 * kChunkPitch, pcode + 2 * 2048, pol_w);
      cp_async16s(is_dst + 3 * kChunkPitch, pcode + 3 * 2048, pol_w);
      if (lane < 16) cp_async16s(is_dst + kScaleOff, pscale, pol_w);
      pcode += kQ4BlockBytes;
      pscale += kQ4BlockBytes;
      if (++is_k == nh) {
        is_k = 0;
        pcode += tile_skip;
        pscale += tile_skip;
      }
      ++is_n;
      is_dst += kStage;
      if (is_dst >= ring_end) is_dst -= kRsDepth * kStage;
    }
  };
  // operand pieces of this thread (the set's 128 threads copy a superblock's N rows x 256
  // bytes): piece m is row n = (sti + 128 m) / 16, 16-byte column c = (sti + 128 m) % 16
  const int sti = (warp & 3) * 32 + lane;
  const uint16_t* xsrc[kXPieces];
  uint32_t xdst[kXPieces];
  bool xval[kXPieces];
#pragma unroll
  for (int m = 0; m < kXPieces; ++m) {
    const int pi = sti + 128 * m, n = pi >> 4, c = pi & 15;
    const int b = n % H;
    xval[m] = b < p.n_act;
    const size_t row = n >= H ? (size_t)(x_lo + H * pass + b) : (size_t)(H * pass + b);
    xsrc[m] = x + row * p.K + (size_t)(sb0 + kbase) * 128 + c * 8;
    xdst[m] = (uint32_t)(n * kXPitch + c * 16);
  }
  const uint32_t xr_u32 = tc::smem_u32(xr);
  // the operand of iteration io (superblock kbase + io % nh of the k-range) into slot
  // io % kRsDepth
  auto issue_x = [&](int io) {
    if (io < nst) {
      const size_t col = (size_t)(io % nh) * 128;
      const uint32_t slot = xr_u32 + (uint32_t)((io % kRsDepth) * kXSlot);
#pragma unroll
      for (int m = 0; m < kXPieces; ++m)
        if (xval[m]) cp_async16_zfill_s(slot + xdst[m], xsrc[m] + col, 16u);
    }
  };
  for (int s = 0; s < kRsDepth - 1; ++s) {
    issue_w();
    cp_async_commit();
  }

  pdl_wait();
  if (threadIdx.x == 0) stamp_begin(p.stamp);
  for (int s = 0; s < kRsDepth - 1; ++s) issue_x(s);
  cp_async_commit();
  // the folded RMSNorm's per-tile sums of squares: every value requested at once (one per
  // thread), added up in tile order after the barrier
  if (p.ss_in)
    for (int i = threadIdx.x; i < p.ss_tiles * p.n_act; i += kThreads) {
      const int tt = i / p.n_act, b = i - tt * p.n_act;
      ssq[i] = __ldcg(p.ss_in + (size_t)tt * p.ss_ld + b);
    }
  tcepi::EpiSrc src = tcepi::epi_src_global(p);
  if (p.epi == EPI_QKV || p.epi == EPI_QKVQ) {
    const int half = p.head_dim >> 1;
    for (int i = threadIdx.x; i < p.n_act * half; i += kThreads) {
      scos[i] = p.cosv[i];
      ssin[i] = p.sinv[i];
    }
    if (threadIdx.x < p.n_act) srows[threadIdx.x] = p.rows[threadIdx.x];
    src.rows = srows;
    src.cosv = scos;
    src.sinv = ssin;
  }
  // group sums of iteration io (slot io % kRsDepth) into parity io & 1: this thread pair takes
  // group gs, column ns; half hs of the 64 values each, then (first 32) + (last 32)
  const int gs = (sti >> 1) / N, ns = (sti >> 1) % N, hs = sti & 1;
  auto group_sums = [&](int io) {
    const uint4* v = reinterpret_cast<const uint4*>(xr + (io % kRsDepth) * kXSlot + ns * kXPitch +
                                                    gs * 128 + hs * 64);
    const float sh = sum32(v);
    const float o = __shfl_xor_sync(0xffffffffu, sh, 1);
    if (hs == 0) xsb[(io & 1) * 2 * N + gs * N + ns] = sh + o;
  };
  cp_async_wait<0>();  // the first superblocks' operand (and the weight blocks before it)
  __syncthreads();
  if (p.ss_in && threadIdx.x < p.n_act) {
    float s = 0.f;
    for (int tt = 0; tt < p.ss_tiles; ++tt) s += ssq[tt * p.n_act + threadIdx.x];
    rinv[threadIdx.x] = rsqrtf(s / (float)p.K + p.eps);
  }
  if (nst > 0) group_sums(0);  // (read after the first iteration's barrier)

  float y[2][NB8][4];  // [row block u][n8 block][fragment]
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int nb = 0; nb < NB8; ++nb)
#pragma unroll
      for (int c = 0; c < 4; ++c) y[u][nb][c] = 0.f;
  // per-lane views: code words of rows 16u + g / 16u + g + 8 (chunk 2G + t/2, half t&1),
  // scales, operand column g of each n8 block
  const uint32_t lane_w = (t >> 1) * kChunkPitch + g * 16 + 8 * (t & 1);
  const uint32_t xlane = xr_u32 + (uint32_t)(g * kXPitch + 32 * t);
  const uint32_t xsl = tc::smem_u32(xsb) + (uint32_t)(2 * t * 4);
  uint32_t st = wring;  // the ring slot consumed next
  const uint32_t km = opaque_const(0x000F000Fu), kc = opaque_const(0x43004300u);
  int it = 0;  // iteration (tile, superblock) of this warp set
  for (int j = 0; j < Tc; ++j) {
    float res[H];
    const uint32_t owner = (uint32_t)(j % C);
    if (warp < 4 && rank == owner) {  // epilogue inputs of this tile, requested early
      const int rb = cid + j * NC;
      tcepi::load_residual<H>(p, rb, threadIdx.x, 0, res);
      src.gn = tcepi::load_next_gain(p, rb, threadIdx.x);
      src.has_gn = true;
    }
    for (int k = 0; k < nh; ++k, ++it) {
      cp_async_wait<0>();            // this thread's copies of iterations it, it + 1 ...
      tc::named_bar_sync(bar, 128);  // ... and the set's; the slots of it - 1 are free, the
                                     // sums of it are in
      issue_w();
      issue_x(it + kRsDepth - 1);
      cp_async_commit();
      if (it + 1 < nst) group_sums(it + 1);
      const uint32_t xo = (uint32_t)((it % kRsDepth) * kXSlot);
      const uint32_t xsp = xsl + (uint32_t)((it & 1) * 2 * N * 4);
      uint2 sv[2][2];                // [u][row g, row g + 8]: (s0, b0), (s1, b1)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        sv[u][0] = lds64(st + kScaleOff + (16 * u + g) * 8);
        sv[u][1] = lds64(st + kScaleOff + (16 * u + g + 8) * 8);
      }
#pragma unroll
      for (int G = 0; G < 2; ++G) {
        // operand fragments of group G (both row blocks use them): column nb * 8 + g, the
        // sixteen k 64 G + 16 t .. + 15 as bf16 pairs, 8 per MMA pair jp
        const uint32_t xg = xlane + xo + G * 128;
        uint4 xv[2][NB8];
        float2 X[NB8];
#pragma unroll
        for (int nb = 0; nb < NB8; ++nb) {
          xv[0][nb] = lds128(xg + nb * 8 * kXPitch);
          xv[1][nb] = lds128(xg + nb * 8 * kXPitch + 16);
          const uint2 Xw = lds64(xsp + (G * N + nb * 8) * 4);
          X[nb] = make_float2(__uint_as_float(Xw.x), __uint_as_float(Xw.y));
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          // lane (g, t): columns 64 G + 16 t .. + 15 of rows 16u + g and 16u + g + 8
          const uint32_t wa = st + lane_w + G * 2 * kChunkPitch + u * 256;
          const uint2 wA = lds64(wa), wB = lds64(wa + 128);
          float acc[NB8][4];
#pragma unroll
          for (int jp = 0; jp < 2; ++jp) {
            const uint32_t a = jp ? wA.y : wA.x, b = jp ? wB.y : wB.x;
            const uint32_t A0[4] = {unpack_pair(a, 0, km, kc), unpack_pair(b, 0, km, kc),
                                    unpack_pair(a, 1, km, kc), unpack_pair(b, 1, km, kc)};
            const uint32_t A1[4] = {unpack_pair(a, 2, km, kc), unpack_pair(b, 2, km, kc),
                                    unpack_pair(a, 3, km, kc), unpack_pair(b, 3, km, kc)};
#pragma unroll
            for (int nb = 0; nb < NB8; ++nb) {
              if (jp == 0) mma16816_z(acc[nb], A0, xv[0][nb].x, xv[0][nb].y);
              else mma16816(acc[nb], A0, xv[jp][nb].x, xv[jp][nb].y);
              mma16816(acc[nb], A1, xv[jp][nb].z, xv[jp][nb].w);
            }
          }
          const uint32_t swa = G ? sv[u][0].y : sv[u][0].x, swb = G ? sv[u][1].y : sv[u][1].x;
          const float s_a = bf16_lo(swa), s_b = bf16_lo(swb);
          const float c_a = fmaf(-128.f, s_a, bf16_hi(swa));
          const float c_b = fmaf(-128.f, s_b, bf16_hi(swb));
#pragma unroll
          for (int nb = 0; nb < NB8; ++nb) {
            y[u][nb][0] = fmaf(s_a, acc[nb][0], fmaf(c_a, X[nb].x, y[u][nb][0]));
            y[u][nb][1] = fmaf(s_a, acc[nb][1], fmaf(c_a, X[nb].y, y[u][nb][1]));
            y[u][nb][2] = fmaf(s_b, acc[nb][2], fmaf(c_b, X[nb].x, y[u][nb][2]));
            y[u][nb][3] = fmaf(s_b, acc[nb][3], fmaf(c_b, X[nb].y, y[u][nb][3]));
          }
        }
      }
      st += kStage;
      if (st >= ring_end) st = wring;
    }

    // ---- end of tile j: hi + lo parts into the warp set's half of the hand-off buffer
    float* sa = sacc + (size_t)((j & 1) * 2 + h) * 128 * H;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r0 = rw + 16 * u + g;
#pragma unroll
      for (int nb = 0; nb < NB8 / 2; ++nb) {
        const float* lo = y[u][nb + NB8 / 2];
        *reinterpret_cast<float2*>(sa + r0 * H + nb * 8 + 2 * t) =
            make_float2(y[u][nb][0] + lo[0], y[u][nb][1] + lo[1]);
        *reinterpret_cast<float2*>(sa + (r0 + 8) * H + nb * 8 + 2 * t) =
            make_float2(y[u][nb][2] + lo[2], y[u][nb][3] + lo[3]);
      }
#pragma unroll
      for (int nb = 0; nb < NB8; ++nb)
#pragma unroll
        for (int c = 0; c < 4; ++c) y[u][nb][c] = 0.f;
    }
    tc::named_bar_sync(2, kThreads);
    if (warp < 4) {
      // ---- tile row r: both halves, then the cluster's partials, then the epilogue
      const int r = threadIdx.x;
      const float* s0 = sacc + (size_t)((j & 1) * 2) * 128 * H + r * H;
      const float* s1 = s0 + 128 * H;
      float vals[H];
#pragma unroll
      for (int b = 0; b < H; ++b) vals[b] = s0[b] + s1[b];
      const int rb = cid + j * NC;
      float sum[H];
      const int got = csk::combine_partials<H>(vals, sum, inbox, inbox_full, j / C, rank, owner,
                                               C, r, abort_flag);
      if (got < 0) report_timeout(p, abort_flag, 1);
      tc::named_bar_sync(1, 128);  // the same decision in all 128 threads
      if (got > 0 && *abort_flag == 0) tcepi::finish<H>(p, rb, r, sum, 0, swx, rinv, res, src);
    }
  }
  cp_async_wait<0>();  // (only empty groups remain: every issued block was consumed)
  if (threadIdx.x == 0) stamp_end(p.stamp);
  if (C > 1 && threadIdx.x == 0)
    for (int s = 0; s < owned; ++s) tc::mbar_wait(&inbox_full[s], 0);
  if (C > 1) csk::cluster_sync();
}

template <int NB8>
size_t q4r_smem(const Q4rPlan& q) {
  return layout(8 * NB8, q).total;
}

size_t q4rs_smem(const Q4rPlan& q) { return layout_rs(q).total; }

using Q4Kernel = void (*)(TcParams, const uint16_t*, int, Q4rPlan);

// most clusters of C CTAs of kern (each with `smem` bytes) resident at once, cached
int q4_active_clusters(Q4Kernel kern, int C, size_t smem) {
  static std::map<std::tuple<const void*, int, size_t>, int> cache;
  const auto key = std::make_tuple(reinterpret_cast<const void*>(kern), C, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  return cache[key] = n;
}

// clusters of the plan's C that both kernels can keep resident (0: a kernel does not fit)
int q4_plan_fit(const Q4rPlan& q) {
  if (q.slots > kMaxSlots || q4r_smem<2>(q) > (size_t)kSmemBudget ||
      q4rs_smem(q) > (size_t)kSmemBudget)
    return 0;
  return std::min(q4_active_clusters(k_q4_rd<2>, q.C, q4r_smem<2>(q)),
                  q4_active_clusters(k_q4_rs, q.C, q4rs_smem(q)));
}

// The split of the k-range (C) follows from the matrix shape alone -- so a row's arithmetic
// does not depend on the number of rows -- by the cost of the busiest CTA: superblocks it
// streams, plus a little for each cluster hand-off.  How many clusters of C CTAs run at once is
// asked of the occupancy calculator (clusters are placed within GPCs, so fewer than
// num_sms / C may fit), for both kernels at their widest operand.
bool q4r_split(int RB, int SB, int num_sms, Q4rPlan* out) {
  static const int kSizes[] = {1, 2, 3, 4, 6, 8};
  double best = 1e30;
  Q4rPlan bp{};
  for (int C : kSizes) {
    if (C > SB || C > num_sms) continue;
    Q4rPlan q{};
    q.C = C;
    q.sb_max = (SB + C - 1) / C;
    if (q.sb_max > kMaxSbPerRank) continue;
    q.NC = std::min(RB, num_sms / C);
    q.slots = C > 1 ? ((RB + q.NC - 1) / q.NC + C - 1) / C : 0;
    const int fit = q4_plan_fit(q);
    if (fit <= 0) continue;
    if (fit < q.NC) {
      q.NC = fit;
      q.slots = C > 1 ? ((RB + q.NC - 1) / q.NC + C - 1) / C : 0;
      if (q4_plan_fit(q) < q.NC) continue;
    }
    const int tmax = (RB + q.NC - 1) / q.NC;
    const double cost = (double)tmax * q.sb_max + (C > 1 ? 1.0 : 0.0) + 0.01 * C;
    if (cost < best) {
      best = cost;
      bp = q;
    }
  }
  if (best >= 1e30) return false;
  *out = bp;
  return true;
}

bool q4_launch(Q4Kernel kern, size_t smem, const TcParams& p, const uint16_t* x, int x_lo,
               const Q4rPlan& q, int passes, cudaStream_t s) {
  // the plan's clusters fit at both kernels' widest operand, so at this one too
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(q.NC * q.C, passes);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = q.C;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kern, p, x, x_lo, q) == cudaSuccess;
}

}  // namespace

bool launch_q4_rd(TcParams p, const uint16_t* x, int x_lo, int num_sms, cudaStream_t s) {
  if (!p.wq || !x || p.K % 128 || p.K <= 0 || p.n_act <= 0 || p.n_act > 32) return false;
  if (p.epi == EPI_SWIGLU && (p.F % 64 || p.M != 2 * p.F)) return false;
  if ((p.epi == EPI_QKV || p.epi == EPI_QKVQ) && (p.head_dim > 128 || p.head_dim % 2)) return false;
  if (p.ss_in && p.ss_tiles > kMaxSsTiles) return false;
  p.RB = p.epi == EPI_SWIGLU ? p.F / 64 : (p.M + 127) / 128;
  p.KS = p.K / 64;
  p.NT = 1;
  static std::map<std::tuple<int, int, int>, Q4rPlan> plans;
  const auto key = std::make_tuple(p.RB, p.K / 128, num_sms);
  auto it = plans.find(key);
  Q4rPlan q;
  if (it != plans.end()) {
    q = it->second;
  } else {
    if (!q4r_split(p.RB, p.K / 128, num_sms, &q)) return false;
    plans[key] = q;
  }
  if (p.n_act <= 4) return q4_launch(k_q4_rd<1>, q4r_smem<1>(q), p, x, x_lo, q, 1, s);
  if (p.n_act <= 8) return q4_launch(k_q4_rd<2>, q4r_smem<2>(q), p, x, x_lo, q, 1, s);
  return q4_launch(k_q4_rs, q4rs_smem(q), p, x, x_lo, q, (p.n_act + kRsH - 1) / kRsH, s);
}
