// gemm_q4.cu -- decode projections y = x W^T over 4-bit affine weights (groups of 64 columns,
// w = s * q + b with q in 0..15 and bf16 s, b) on the 5th-generation tensor cores (sm_103a).
//
// The codes enter the MMA as exact integers, so no dequantised weight is ever rounded:
//   * a converter warp group unpacks each 128-row x 128-column block of codes from shared
//     memory into tensor memory as bf16 (128 + q), two per 32-bit column -- the layout in which
//     tcgen05.mma reads its A operand from TMEM;
//   * the same warps add up the operand's 64-column groups (sum_k x[k] of each operand row) on
//     the CUDA cores;
//   * each group of 64 columns is its own MMA chain (codes x operand) into a ring of TMEM
//     accumulators;
//   * the epilogue warps fold every group in with its scale and bias, in fp32:
//       y[m] += s[m,g] * sum_k (128 + q[m,k]) x[k]  +  (b[m,g] - 128 s[m,g]) * sum_k x[k].
// The operand is the bf16 hi/lo pair of the other decode projections, so the result is that of
// the fp32 operand and the exactly dequantised weights, up to fp32 accumulation.
// A 4-bit block carries four times the weights of a bf16 one per byte, so a stage needs four
// times the MMAs per byte streamed; one thread issues a tcgen05.mma only every ~60 ns, so two
// warps issue them (one per stage parity), and eight warps unpack.  An
// mbarrier wait tells phases apart only by parity, so a waiter that could run two phases ahead
// of a barrier would misread it: every barrier instance is used by its waiters in order (the
// issuers of one parity touch only the stages, A slots and accumulator slots of that parity,
// which needs an even pipeline depth).
//
// Everything else is the cluster split-K of gemm_csk.cu: tile t belongs to cluster t % NC, rank
// r of the cluster streams super-blocks [r SB / C, (r + 1) SB / C) of each of its tiles, the
// partial sums of a tile meet in its owner's shared memory (st.async) and are added in rank
// order, and the owner runs the shared epilogue (residual add, SwiGLU, RoPE + KV append, RMSNorm
// statistics).
//
// The weights live on the device in a layout of their own, written once by q4_repack from the
// interchange format (uint32 words of eight codes, element 8j + t in bits 4t..4t+3 of word j;
// bf16 scales and biases [rows][cols / 64]): per (128-row tile, 128-column super-block) one
// contiguous 9 KB block that a single bulk copy brings in,
//   [4 chunks][128 rows][16 bytes]  codes: chunk c of a row holds columns 32c .. 32c + 31 as
//                                   four words, word i's pair p = (bits 4p..4p+3: column 8i+2p,
//                                   bits 16+4p..19+4p: column 8i+2p+1), so one shift and one
//                                   logic op turn a pair into a bf16x2 word;
//   [128 rows][s0, b0, s1, b1]      bf16 scale and bias of the block's two groups.
// SwiGLU tiles hold 64 gate rows and then the same 64 features' up rows.
#include <algorithm>
#include <map>
#include <tuple>

#include "csk_common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_epilogue.cuh"

namespace {

using csk::cluster_rank;
using csk::cluster_sync;
using tcepi::finish;
// every wait of this kernel suspends instead of spinning: most warps wait most of the time
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return csk::wait_or_abort_sleep(bar, parity, abort);
}
using tcepi::load_residual;

constexpr int kMmaWarps = 2;   // MMA issuers: warp par takes the stages of parity par
constexpr int kConvWarps = 8;  // two per TMEM lane quarter, one 64-column group each
// 15 warps: at most four share an SM sub-partition's 16 K registers, so 128 per thread
constexpr int kConvWarp0 = 1 + kMmaWarps, kEpiWarp0 = kConvWarp0 + kConvWarps;
constexpr int kThreads = 32 * (kEpiWarp0 + 4);  // TMA, MMA issuers, converters, 4 epilogue
constexpr int kNK = 2;         // 64-column groups per stage
constexpr int kCodeBytes = 128 * 64;
constexpr int kWBytes = kQ4BlockBytes;  // codes + scales/biases of one stage
constexpr int kMaxStages = 8;
constexpr int kMaxSlots = 4;
constexpr int kSmemBudget = 227 * 1024;
// tensor memory: A ring [0, 256), accumulator slots (BN columns each) from column 256
constexpr int kRA = 4;
constexpr uint32_t kAccCol = 256, kTmemCols = 512;

template <int BN>
__host__ __device__ constexpr int acc_slots() {
  return BN == 64 ? 4 : 8;
}

__device__ __forceinline__ void report_timeout(const TcParams& p, volatile int* abort, int role) {
  *abort = 1;
  if (atomicCAS(p.err, 0, CBT_DEV_TIMEOUT) == 0) p.err[1] = 400 + role;
}

struct Smem {
  uint8_t *x, *w;
  float* xs;  // [stages][kNK][BN/2]: each operand row's sum (hi + lo) over each group
  float *inbox, *swx, *rinv;
  float *cosv, *sinv;
  QueryRow* rows;
  uint64_t *full, *empty, *afull, *aempty, *xsf, *accf, *acce, *done, *inbox_full;
  uint32_t* tmem_slot;
  volatile int* sflag;
};

template <int BN>
__host__ __device__ constexpr size_t inbox_floats(int C, int slots) {
  return (size_t)slots * (C - 1) * 128 * (BN / 2);
}
template <int BN>
__host__ __device__ constexpr size_t rope_floats() {
  return (size_t)(BN / 2) * 64 * 2;
}
template <int BN>
__host__ __device__ size_t q4_smem_bytes(const CskPlan& q, bool qkv) {
  return 1024 + (size_t)q.stages * (kNK * BN * 128 + kWBytes + kNK * (BN / 2) * 4) +
         inbox_floats<BN>(q.C, q.slots) * 4 + (128 * 33 + 32) * 4 +
         (qkv ? rope_floats<BN>() * 4 + 32 * sizeof(QueryRow) : 0) + 640;
}

template <int BN>
__device__ __forceinline__ Smem carve(uint8_t* smem, const CskPlan& q, bool qkv) {
  Smem s;
  s.x = smem;  // operand tiles first: each stage's tiles stay 1024-byte aligned (swizzle)
  s.w = s.x + q.stages * kNK * BN * 128;
  s.xs = reinterpret_cast<float*>(s.w + q.stages * kWBytes);
  s.inbox = s.xs + q.stages * kNK * (BN / 2);
  s.swx = s.inbox + inbox_floats<BN>(q.C, q.slots);
  s.rinv = s.swx + 128 * 33;
  s.cosv = s.rinv + 32;
  s.sinv = s.cosv + (qkv ? rope_floats<BN>() / 2 : 0);
  s.rows = reinterpret_cast<QueryRow*>(s.sinv + (qkv ? rope_floats<BN>() / 2 : 0));
  s.full = reinterpret_cast<uint64_t*>(s.rows + (qkv ? 32 : 0));
  s.empty = s.full + kMaxStages;
  s.afull = s.empty + kMaxStages;
  s.aempty = s.afull + kRA;
  s.xsf = s.aempty + kRA;
  s.accf = s.xsf + kMaxStages;
  s.acce = s.accf + 8;
  s.done = s.acce + 8;
  s.inbox_full = s.done + kMmaWarps;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.inbox_full + kMaxSlots);
  s.sflag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);
  return s;
}

// pair p of a native code word as a bf16x2 word (128 + q_even, 128 + q_odd): the codes sit in
// the low mantissa bits of 128.0
__device__ __forceinline__ uint32_t unpack_pair(uint32_t w, int p) {
  return ((w >> (4 * p)) & 0x000F000Fu) | 0x43004300u;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    k_q4_csk(const __grid_constant__ CUtensorMap tx, const TcParams p, const CskPlan q) {
  constexpr int H = BN / 2;  // operand rows: H hi parts, then H lo parts
  constexpr int RG = acc_slots<BN>();
  constexpr int kXBytes = BN * 128;
  constexpr uint32_t kIdesc = tc::idesc_bf16(128, BN);
  constexpr uint32_t kPartBytes = 128 * H * 4;
  constexpr int CH = H < 16 ? H : 16;  // accumulator columns read per TMEM load
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const Smem sm = carve<BN>(base, q, p.epi == EPI_QKV);
  const int S = q.stages, C = q.C;
  const int stage_x = kNK * kXBytes;
  volatile int* abort_flag = sm.sflag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = C > 1 ? cluster_rank() : 0u;
  const int cid = blockIdx.x / C, NC = gridDim.x / C;
  const int Tc = cid < p.RB ? (p.RB - cid + NC - 1) / NC : 0;
  const int SB = p.KS / kNK;
  const int sb0 = (int)((long long)rank * SB / C);
  const int sb1 = (int)((long long)(rank + 1) * SB / C);
  const int nsb = sb1 - sb0;
  const int nst = Tc * nsb;  // stages this CTA streams: (tile j, super-block sb0 + i % nsb)
  const int owned = Tc > (int)rank ? (Tc - (int)rank + C - 1) / C : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&sm.full[s], 1);
      tc::mbar_init(&sm.empty[s], 1 + 4);     // the stage's MMA commit, the epilogue warps
      tc::mbar_init(&sm.xsf[s], kConvWarps);  // each converter warp's rows of the group sums
    }
    for (int a = 0; a < kRA; ++a) {
      tc::mbar_init(&sm.afull[a], kConvWarps);
      tc::mbar_init(&sm.aempty[a], 1);
    }
    for (int a = 0; a < RG; ++a) {
      tc::mbar_init(&sm.accf[a], 1);
      tc::mbar_init(&sm.acce[a], 4);
    }
    for (int m = 0; m < kMmaWarps; ++m) tc::mbar_init(&sm.done[m], 1);
    for (int s = 0; s < kMaxSlots; ++s) tc::mbar_init(&sm.inbox_full[s], 1);
    if (C > 1)
      for (int s = 0; s < owned; ++s) tc::mbar_expect_tx(&sm.inbox_full[s], (C - 1) * kPartBytes);
    sm.sflag[0] = 0;
    sm.sflag[1] = 0;
    tc::mbar_fence_init();
    tc::tma_prefetch_desc(&tx);
  }
  if (warp == 1) tc::tmem_alloc(sm.tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (C > 1) cluster_sync();
  const uint32_t tmem = *sm.tmem_slot;
  pdl_launch();

  if (warp == 0) {
    if (lane == 0) {  // ---- producer: weight blocks (bulk copies) and operand tiles (TMA)
      const uint64_t pol_x = tc::policy_evict_last();
      int pend_k[kMaxStages], pend_st[kMaxStages];
      int npend = 0;
      bool dep_done = false;
      auto flush_pending = [&]() {
        pdl_wait();
        dep_done = true;
        for (int i = 0; i < npend; ++i)
          tc::tma_load_3d(sm.x + pend_st[i] * stage_x, &tx, &sm.full[pend_st[i]], 0, 0,
                          pend_k[i] * kNK, pol_x);
        npend = 0;
      };
      int issued = 0;
      for (int i = 0; i < nst; ++i) {
        const int rb = cid + (i / nsb) * NC, sb = sb0 + i % nsb;
        const int stage = i % S;
        if (!wait_or_abort(&sm.empty[stage], ((i / S) & 1) ^ 1, abort_flag)) {
          report_timeout(p, abort_flag, 1);
          break;
        }
        tc::mbar_expect_tx(&sm.full[stage], kWBytes + stage_x);
        tc::bulk_load(sm.w + stage * kWBytes, p.wq + ((size_t)rb * SB + sb) * kWBytes, kWBytes,
                      &sm.full[stage]);
        if (dep_done) {
          tc::tma_load_3d(sm.x + stage * stage_x, &tx, &sm.full[stage], 0, 0, sb * kNK, pol_x);
        } else {
          pend_k[npend] = sb;
          pend_st[npend] = stage;
          if (++npend == S) flush_pending();
        }
        ++issued;
      }
      if (!dep_done) flush_pending();
      // never leave with copies in flight: the last loads of each stage
      for (int i = issued - 1; i >= 0 && i >= issued - S; --i)
        tc::mbar_wait(&sm.full[i % S], (i / S) & 1);
    }
  } else if (warp <= kMmaWarps) {
    // ---- MMA warps: warp par issues the eight MMAs (two groups) of stages par, par + 2, ...
    // Once the stage's codes are in tensor memory (so its loads have landed), lane 0 waits for
    // the groups' accumulator slots and issues.
    const int par = warp - 1;
    if (lane == 0) {
      bool ok = true;
      for (int i = par; i < nst && ok; i += 2) {
        const int stage = i % S, as = i % kRA;
        // afull first: the converters saw the stage land, so the stage's own full phase is
        // the one complete now (waited too, for the operand tile's visibility to the MMA)
        if (!wait_or_abort(&sm.afull[as], (i / kRA) & 1, abort_flag) ||
            !wait_or_abort(&sm.full[stage], (i / S) & 1, abort_flag)) {
          report_timeout(p, abort_flag, 3);
          break;
        }
        for (int jj = 0; jj < kNK; ++jj) {
          const int g = i * kNK + jj, slot = g % RG;
          if (!wait_or_abort(&sm.acce[slot], ((g / RG) & 1) ^ 1, abort_flag)) {
            report_timeout(p, abort_flag, 3);
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t dq = tmem + kAccCol + (uint32_t)(slot * BN);
          const uint64_t xd =
              tc::sdesc_sw128(tc::smem_u32(sm.x + stage * stage_x + jj * kXBytes));
          const uint32_t acol = tmem + (uint32_t)(as * 64 + jj * 32);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16_ta(dq, acol + 8 * kk, xd + 2 * kk, kIdesc, kk > 0 ? 1u : 0u);
          tc::mma_commit(&sm.accf[slot]);
        }
        if (!ok) break;
        tc::mma_commit(&sm.aempty[as]);
        tc::mma_commit(&sm.empty[stage]);
      }
      // all MMAs of this thread complete before TMEM is released
      tc::mma_commit(&sm.done[par]);
      tc::mbar_wait(&sm.done[par], 0);
    }
  } else if (warp < kEpiWarp0) {
    // ---- converters: warp (quarter qd, group half) unpacks columns [64 half, 64 half + 64) of
    // tile rows 32 qd .. 32 qd + 31 into the A ring in TMEM, then adds up operand rows
    // [qd H/4, (qd + 1) H/4) of the group (hi and lo parts, 16-byte chunks, 8 lanes a row)
    const int qd = warp & 3, half = (warp - kConvWarp0) >> 2;
    const int r = qd * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
    for (int i = 0; i < nst; ++i) {
      const int stage = i % S, as = i % kRA;
      if (!wait_or_abort(&sm.full[stage], (i / S) & 1, abort_flag) ||
          !wait_or_abort(&sm.aempty[as], ((i / kRA) & 1) ^ 1, abort_flag)) {
        report_timeout(p, abort_flag, 4);
        break;
      }
      const uint8_t* codes = sm.w + stage * kWBytes + r * 16;
      uint32_t a[32];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const uint4 v = *reinterpret_cast<const uint4*>(codes + (2 * half + cc) * 2048);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int pp = 0; pp < 4; ++pp) a[cc * 16 + k * 4 + pp] = unpack_pair(wv[k], pp);
      }
      tc::tmem_st32(lane_base + (uint32_t)(as * 64 + half * 32), a);
      tc::tmem_st_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.afull[as]);
      float* xs = sm.xs + stage * kNK * H;
      const uint8_t* tile = sm.x + stage * stage_x + half * kXBytes;
#pragma unroll
      for (int e = 0; e < (2 * H + 31) / 32; ++e) {  // (row, chunk): H/4 x 8
        const int pidx = lane + 32 * e;
        const bool valid = pidx < 2 * H;
        const int row = qd * (H / 4) + (pidx >> 3), c = pidx & 7, lo = row + H;
        float sum = 0.f;
        if (valid) {
          const uint4 v = *reinterpret_cast<const uint4*>(tile + row * 128 + ((c ^ (row & 7)) << 4));
          const uint4 u = *reinterpret_cast<const uint4*>(tile + lo * 128 + ((c ^ (lo & 7)) << 4));
          sum = ((bf16_lo(v.x) + bf16_hi(v.x)) + (bf16_lo(v.y) + bf16_hi(v.y))) +
                ((bf16_lo(v.z) + bf16_hi(v.z)) + (bf16_lo(v.w) + bf16_hi(v.w)));
          sum += ((bf16_lo(u.x) + bf16_hi(u.x)) + (bf16_lo(u.y) + bf16_hi(u.y))) +
                 ((bf16_lo(u.z) + bf16_hi(u.z)) + (bf16_lo(u.w) + bf16_hi(u.w)));
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        if (valid && c == 0) xs[half * H + row] = sum;
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.xsf[stage]);
    }
  } else {  // ---- epilogue warps: TMEM lanes 32q .. 32q + 31 = tile rows
    pdl_wait();
    const int qd = warp & 3;
    const int r = qd * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
    if (p.ss_in) {
      if (r < p.n_act) {
        float s = 0.f;
        for (int t = 0; t < p.ss_tiles; ++t) s += p.ss_in[(size_t)t * p.ss_ld + r];
        sm.rinv[r] = rsqrtf(s / (float)p.K + p.eps);
      }
    }
    tcepi::EpiSrc src = tcepi::epi_src_global(p);
    if (p.epi == EPI_QKV) {
      const int half = p.head_dim >> 1;
      for (int i = r; i < p.n_act * half; i += 128) {
        sm.cosv[i] = p.cosv[i];
        sm.sinv[i] = p.sinv[i];
      }
      if (r < p.n_act) sm.rows[r] = p.rows[r];
      src.rows = sm.rows;
      src.cosv = sm.cosv;
      src.sinv = sm.sinv;
    }
    tc::named_bar_sync(1, 128);
    bool ok = true;
    int i = 0;  // stage counter
    for (int j = 0; j < Tc && ok; ++j) {
      const int rb = cid + j * NC;
      const uint32_t owner = (uint32_t)(j % C);
      const int tslot = j / C;
      float res[H];
      if (rank == owner) {
        load_residual<H>(p, rb, r, 0, res);
        src.gn = tcepi::load_next_gain(p, rb, r);
        src.has_gn = true;
      }
      float y[H];
#pragma unroll
      for (int n = 0; n < H; ++n) y[n] = 0.f;
      for (int k = 0; k < nsb; ++k, ++i) {
        const int stage = i % S;
        // the stage's scales and biases (landed with the stage) and operand group sums
        if (!wait_or_abort(&sm.full[stage], (i / S) & 1, abort_flag) ||
            !wait_or_abort(&sm.xsf[stage], (i / S) & 1, abort_flag)) {
          report_timeout(p, abort_flag, 5);
          ok = false;
          break;
        }
        const uint2 sbw =
            *reinterpret_cast<const uint2*>(sm.w + stage * kWBytes + kCodeBytes + r * 8);
        const uint32_t sbv[2] = {sbw.x, sbw.y};
        const float* xs = sm.xs + stage * kNK * H;
        if constexpr (H <= 16) {
          // both groups of the stage: wait for both accumulators, one round of TMEM loads
          uint32_t qh[kNK][H], ql[kNK][H];
#pragma unroll
          for (int jj = 0; jj < kNK; ++jj) {
            const int g = i * kNK + jj, slot = g % RG;
            if (!wait_or_abort(&sm.accf[slot], (g / RG) & 1, abort_flag)) {
              report_timeout(p, abort_flag, 6);
              ok = false;
              break;
            }
          }
          if (!ok) break;
          tc::tc_fence_after();
#pragma unroll
          for (int jj = 0; jj < kNK; ++jj) {
            const uint32_t ta = lane_base + kAccCol + (uint32_t)(((i * kNK + jj) % RG) * BN);
            if constexpr (H == 16) {
              tc::tmem_ld16(ta, qh[jj]);
              tc::tmem_ld16(ta + H, ql[jj]);
            } else {
              tc::tmem_ld8(ta, qh[jj]);
              tc::tmem_ld8(ta + H, ql[jj]);
            }
          }
          tc::tmem_ld_wait();
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0)
            for (int jj = 0; jj < kNK; ++jj) tc::mbar_arrive(&sm.acce[(i * kNK + jj) % RG]);
#pragma unroll
          for (int jj = 0; jj < kNK; ++jj) {
            const float s = bf16_to_f32((uint16_t)(sbv[jj] & 0xFFFFu));
            const float b1 = bf16_to_f32((uint16_t)(sbv[jj] >> 16)) - 128.f * s;
#pragma unroll
            for (int n = 0; n < H; n += 4) {
              const float4 f = *reinterpret_cast<const float4*>(xs + jj * H + n);
              const float xv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float vq = __uint_as_float(qh[jj][n + e]) + __uint_as_float(ql[jj][n + e]);
                y[n + e] = fmaf(s, vq, fmaf(b1, xv[e], y[n + e]));
              }
            }
          }
        } else {
#pragma unroll
          for (int jj = 0; jj < kNK; ++jj) {
            const int g = i * kNK + jj, slot = g % RG;
            const float s = bf16_to_f32((uint16_t)(sbv[jj] & 0xFFFFu));
            const float b1 = bf16_to_f32((uint16_t)(sbv[jj] >> 16)) - 128.f * s;
            if (!wait_or_abort(&sm.accf[slot], (g / RG) & 1, abort_flag)) {
              report_timeout(p, abort_flag, 6);
              ok = false;
              break;
            }
            tc::tc_fence_after();
            const uint32_t ta = lane_base + kAccCol + (uint32_t)(slot * BN);
#pragma unroll
            for (int c0 = 0; c0 < H; c0 += CH) {
              uint32_t qh[CH], ql[CH];
              if constexpr (CH == 16) {
                tc::tmem_ld16(ta + c0, qh);
                tc::tmem_ld16(ta + H + c0, ql);
              } else {
                tc::tmem_ld8(ta + c0, qh);
                tc::tmem_ld8(ta + H + c0, ql);
              }
              tc::tmem_ld_wait();
              float xv[CH];
#pragma unroll
              for (int n = 0; n < CH; n += 4) {
                const float4 f = *reinterpret_cast<const float4*>(xs + jj * H + c0 + n);
                xv[n] = f.x;
                xv[n + 1] = f.y;
                xv[n + 2] = f.z;
                xv[n + 3] = f.w;
              }
#pragma unroll
              for (int n = 0; n < CH; ++n) {
                const float vq = __uint_as_float(qh[n]) + __uint_as_float(ql[n]);
                y[c0 + n] = fmaf(s, vq, fmaf(b1, xv[n], y[c0 + n]));
              }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&sm.acce[slot]);
          }
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm.empty[stage]);  // the stage may be refilled
      }
      if (!ok) break;
      float sum[H];
      const int got = csk::combine_partials<H>(y, sum, sm.inbox, sm.inbox_full, tslot, rank,
                                               owner, C, r, abort_flag);
      if (got < 0) {
        report_timeout(p, abort_flag, 7);
        break;
      }
      if (got > 0) finish<H>(p, rb, r, sum, 0, sm.swx, sm.rinv, res, src);
    }
    if (C > 1 && threadIdx.x == 32 * kEpiWarp0)
      for (int s = 0; s < owned; ++s) tc::mbar_wait(&sm.inbox_full[s], 0);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  if (C > 1) cluster_sync();
}

template <int BN>
cudaError_t launch_q4(const CUtensorMap& tx, const TcParams& p, const CskPlan& q, cudaStream_t s) {
  const size_t smem = q4_smem_bytes<BN>(q, p.epi == EPI_QKV);
  auto kern = k_q4_csk<BN>;
  cudaError_t rc = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (rc != cudaSuccess) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(q.NC * q.C);
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
  return cudaLaunchKernelEx(&cfg, kern, tx, p, q);
}

template <int BN>
int active_clusters(int C, size_t smem) {
  static std::map<std::pair<int, size_t>, int> cache;
  auto key = std::make_pair(C, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  auto kern = k_q4_csk<BN>;
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

// The cluster shape depends on the matrix shape alone (as for the bf16 weights), so a row's
// result does not depend on how many rows share the step.
bool q4_plan(int RB, int KS, int BN, int num_sms, CskPlan* out) {
  if (RB <= 0 || KS <= 0 || num_sms <= 0 || KS % kNK) return false;
  static const int kSizes[] = {1, 2, 3, 4, 6, 8};
  double best = 1e30;
  CskPlan bp{};
  const int SB = KS / kNK;
  for (int C : kSizes) {
    if (C > SB || C > num_sms) continue;
    CskPlan q{};
    q.nk = kNK;
    q.C = C;
    q.NC = std::min(RB, num_sms / C);
    const int tmax = (RB + q.NC - 1) / q.NC;
    q.slots = C > 1 ? (tmax + C - 1) / C : 0;
    if (q.slots > kMaxSlots) continue;
    q.stages = 2;
    if (q4_smem_bytes<64>(q, true) > (size_t)kSmemBudget) continue;
    const int fit = active_clusters<64>(C, q4_smem_bytes<64>(q, true));
    if (fit <= 0) continue;
    if (fit < q.NC) q.NC = fit;
    const int tmax2 = (RB + q.NC - 1) / q.NC;
    q.slots = C > 1 ? (tmax2 + C - 1) / C : 0;
    if (q.slots > kMaxSlots) continue;
    const double cost = (double)tmax2 * ((SB + C - 1) / C) * kNK + (C > 1 ? 2.0 : 0.0) + 0.01 * C;
    if (cost < best) {
      best = cost;
      bp = q;
    }
  }
  if (best >= 1e30) return false;
  bp.stages = kMaxStages;
  auto smem = [&](const CskPlan& q) {
    return BN == 16 ? q4_smem_bytes<16>(q, true)
                    : BN == 32 ? q4_smem_bytes<32>(q, true) : q4_smem_bytes<64>(q, true);
  };
  while (bp.stages > 2 && smem(bp) > (size_t)kSmemBudget) --bp.stages;
  bp.stages &= ~1;  // even: the issuers of one stage parity own half of the stages
  if (bp.stages < 2 || smem(bp) > (size_t)kSmemBudget) return false;
  *out = bp;
  return true;
}

// ---- the native layout, from the interchange format -------------------------------------------
// One thread per tile row of one block; invalid rows (past the matrix) are zero codes with zero
// scale and bias, so they contribute nothing.
__global__ void k_q4_repack(const uint32_t* __restrict__ packed, const uint16_t* __restrict__ scales,
                            const uint16_t* __restrict__ biases, int M, int K, int F, int SB,
                            uint8_t* __restrict__ out) {
  const int blk = blockIdx.x, r = threadIdx.x;
  const int rb = blk / SB, sb = blk % SB;
  int src;
  bool valid;
  if (F > 0) {  // SwiGLU: gate rows, then the same features' up rows
    const int f = rb * 64 + (r & 63);
    valid = f < F;
    src = r < 64 ? f : F + f;
  } else {
    src = rb * 128 + r;
    valid = src < M;
  }
  uint8_t* dst = out + (size_t)blk * kQ4BlockBytes;
#pragma unroll 1
  for (int i = 0; i < 16; ++i) {  // word i: columns sb*128 + 8i .. + 7
    const uint32_t w = valid ? packed[(size_t)src * (K / 8) + sb * 16 + i] : 0u;
    uint32_t o = 0;
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      o |= ((w >> (8 * pp)) & 0xFu) << (4 * pp);
      o |= ((w >> (8 * pp + 4)) & 0xFu) << (16 + 4 * pp);
    }
    // chunk i / 4 of row r, word i % 4
    reinterpret_cast<uint32_t*>(dst + (i >> 2) * 2048 + r * 16)[i & 3] = o;
  }
  uint16_t* sbd = reinterpret_cast<uint16_t*>(dst + kCodeBytes + r * 8);
#pragma unroll
  for (int jj = 0; jj < kNK; ++jj) {
    const size_t gi = (size_t)src * (K / 64) + sb * kNK + jj;
    sbd[2 * jj] = valid ? scales[gi] : (uint16_t)0;
    sbd[2 * jj + 1] = valid ? biases[gi] : (uint16_t)0;
  }
}

}  // namespace

size_t q4_native_bytes(int M, int K, int F) {
  if (K % 128) return 0;
  const int RB = F > 0 ? (F + 63) / 64 : (M + 127) / 128;
  return (size_t)RB * (K / 128) * kQ4BlockBytes;
}

bool launch_q4_repack(const uint32_t* packed, const uint16_t* scales, const uint16_t* biases,
                      int M, int K, int F, uint8_t* out, cudaStream_t s) {
  if (K % 128 || M <= 0 || (F > 0 && M != 2 * F)) return false;
  const int RB = F > 0 ? (F + 63) / 64 : (M + 127) / 128;
  const int SB = K / 128;
  k_q4_repack<<<RB * SB, 128, 0, s>>>(packed, scales, biases, M, K, F, SB, out);
  count_launch();
  return cudaGetLastError() == cudaSuccess;
}

bool launch_q4_csk(const CUtensorMap& tx, TcParams p, int BN, int num_sms, cudaStream_t s) {
  if (!p.wq || p.K % 128 || p.K <= 0 || p.n_act <= 0 || 2 * p.n_act > BN) return false;
  if (p.epi == EPI_SWIGLU && (p.F % 64 || p.M != 2 * p.F)) return false;
  p.RB = p.epi == EPI_SWIGLU ? p.F / 64 : (p.M + 127) / 128;
  p.KS = p.K / 64;
  p.NT = 1;
  static std::map<std::tuple<int, int, int, int>, CskPlan> plans;
  const auto key = std::make_tuple(p.RB, p.KS, BN, num_sms);
  auto it = plans.find(key);
  CskPlan q;
  if (it != plans.end()) {
    q = it->second;
  } else {
    if (!q4_plan(p.RB, p.KS, BN, num_sms, &q)) return false;
    plans[key] = q;
  }
  if (q.stages % 2) return false;
  cudaError_t rc;
  if (BN == 16) rc = launch_q4<16>(tx, p, q, s);
  else if (BN == 32) rc = launch_q4<32>(tx, p, q, s);
  else if (BN == 64) rc = launch_q4<64>(tx, p, q, s);
  else return false;
  return rc == cudaSuccess;
}
