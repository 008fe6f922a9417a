// gemm_tc.cu -- projections y = x W^T on the 5th-generation tensor cores (sm_103a).
//
// Swap-AB: the weight rows are the MMA's M side (128 per tile), the activation rows its N
// side, so a decode step with B rows is one 128 x N x 64 MMA chain per weight tile and every
// weight byte crosses HBM once.  Per CTA: one TMA producer thread streams 128x64 bf16 weight
// tiles and Nx64 activation tiles into a ring of 128-byte-swizzled shared-memory stages;
// one thread issues tcgen05.mma into a double-buffered TMEM accumulator; four epilogue warps
// read the accumulator back (tcgen05.ld) and apply the epilogue (store, residual add, or
// SwiGLU into the next projection's bf16 operand).
//
// Decode (SPLIT): activations enter as bf16 hi/lo pairs (x = hi + lo), rows [0, BN/2) hi and
// [BN/2, BN) lo, summed in the epilogue -- fp32-grade operands at no cost, since the N side
// is padded anyway.  Work is split stream-K: the (row block, k-step) units are divided evenly
// over the grid, so every CTA streams the same number of weight bytes; a row block cut
// between CTAs is finished by whichever CTA completes it last, summing the partial sums in
// a fixed order, so results do not depend on timing.
//
// RMSNorm without a kernel of its own (decode): RMSNorm(x) W^T = rsqrt(mean(x^2) + eps) *
// ((x * g) W^T), so the residual-add epilogue that produces x also writes x * g (the next
// projection's operand, hi/lo) and x's sums of squares over its 128-row tile; the consuming
// projection scales each accumulated column by the row's rsqrt(mean(x^2) + eps).
// Prefill (!SPLIT): N tiles of up to 128 tokens, whole tiles per CTA.  The activations are
// bf16 hi/lo pairs here too (lo parts at row act_lo + t): each stage carries both operand
// tiles and the MMA chain runs over both.  The tensor core's fp32 accumulation rounds toward
// zero (measured: a relative bias of -4e-6 over K = 4096, -1.5e-5 over K = 14336), and over a
// deep prefill the bias reaches the logits through the bf16 rounding of every appended K/V;
// so every kDrainEvery k-blocks the MMAs start a fresh accumulator (kPrefillAcc of them in
// rotation, which fill the tensor memory) and the epilogue warps add the finished one into fp32
// sums with round to nearest while the next k-blocks run: only the MMAs of one group truncate.
// Measured on a 4 x 1024-token 7B prefill: groups of 1, 2, 4 and 16 k-blocks take 260, 247,
// 233 and 177 ms a call (the original 16-k-block interleave 142 ms); a 32-layer prefill then
// decode stays within 1.6-1.7e-2 of the double-precision oracle for groups of up to 4 and
// exceeds 2e-2 at 16.
// Prefill over 4-bit weights (WLO): the matrix arrives expanded into bf16 hi and lo parts, each
// stage carries both weight tiles, and the chain adds lo . x_hi to hi . x_hi + hi . x_lo (the
// lo . x_lo term is below 2^-16 of the product).
#include <cudaTypedefs.h>

#include <algorithm>

#include "kernels.h"
#include "tc_common.cuh"
#include "tc_epilogue.cuh"

namespace {

using tcepi::finish;
using tcepi::load_residual;

constexpr int kThreads = 192;       // warp 0 TMA, warp 1 MMA (+TMEM alloc), warps 2..5 epilogue
constexpr int kABytes = 128 * 128;  // 128 rows x 64 bf16
// Decode stages: 8 x (16 KB of weights + the operand tile) keeps 128 KB of weights in flight
// per SM (5 stages, which would let a second CTA share the SM, measured slower).
constexpr int kSplitStages = 8;
constexpr int kPrefillAcc = 4;   // prefill accumulators in rotation
constexpr int kDrainEvery = 4;   // k-blocks an accumulator takes before the epilogue adds it up

struct Sched {
  long long u, u1;
  int t;
  __device__ void init(const TcParams& p) {
    if (p.streamk) {
      u = (long long)blockIdx.x * p.U / gridDim.x;
      u1 = (long long)(blockIdx.x + 1) * p.U / gridDim.x;
    } else {
      t = blockIdx.x;
    }
  }
  __device__ bool next(const TcParams& p, int& tile, int& kb, int& ke) {
    if (p.streamk) {
      if (u >= u1) return false;
      tile = (int)(u / p.KS);
      kb = (int)(u % p.KS);
      long long rem = u1 - u;
      ke = (int)((long long)p.KS < kb + rem ? (long long)p.KS : kb + rem);
      u += ke - kb;
      return true;
    }
    if (t >= p.RB * p.NT) return false;
    tile = t;
    kb = 0;
    ke = p.KS;
    t += gridDim.x;
    return true;
  }
};

// CTA whose stream-K range holds unit u (ranges are [c*U/G, (c+1)*U/G))
__host__ __device__ inline int cta_of_unit(long long U, long long G, long long u) {
  long long c = u * G / U;
  while (c + 1 < G && (c + 1) * U / G <= u) ++c;
  while (c > 0 && c * U / G > u) --c;
  return (int)c;
}

__device__ __forceinline__ void report_timeout(const TcParams& p, volatile int* abort, int role) {
  *abort = 1;
  if (atomicCAS(p.err, 0, CBT_DEV_TIMEOUT) == 0) p.err[1] = role;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < tc::kSpinLimit; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 1023) == 1023 && *abort) return false;
    if (i > 256) __nanosleep(32);
  }
  return false;
}


template <int BN, int STAGES, bool SPLIT, bool WLO>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_linear(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx,
                const __grid_constant__ CUtensorMap twl, const TcParams p) {
  static_assert(!(WLO && SPLIT), "weight lo parts are a prefill form");
  constexpr int kXTile = BN * 128;                     // one [BN rows][64] operand tile
  constexpr int kXBytes = SPLIT ? kXTile : 2 * kXTile;  // prefill stages: hi and lo tiles
  constexpr int kAStage = WLO ? 2 * kABytes : kABytes;  // weight tile (+ its lo parts)
  constexpr uint32_t kTmemCols = SPLIT ? (2 * BN < 32 ? 32 : 2 * BN) : kPrefillAcc * BN;
  constexpr uint32_t kIdesc = tc::idesc_bf16(128, BN);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sX = smem + STAGES * kAStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(sX + STAGES * kXBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;  // per accumulator: MMAs done / drained by the epilogue
  uint64_t* acce = accf + kPrefillAcc;
  uint64_t* done = acce + kPrefillAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* sflag = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] last, [1] abort
  float* swx = reinterpret_cast<float*>(smem + STAGES * (kAStage + kXBytes) + 512);
  float* rinv = swx + 128 * 33;  // [32] RMSNorm factor of each decode column

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < kPrefillAcc; ++a) {
      tc::mbar_init(&accf[a], 1);
      tc::mbar_init(&acce[a], 4);
    }
    tc::mbar_init(done, 1);
    sflag[0] = 0;
    sflag[1] = 0;
    tc::mbar_fence_init();
    tc::tma_prefetch_desc(&tw);
    tc::tma_prefetch_desc(&tx);
    if (WLO) tc::tma_prefetch_desc(&twl);
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_launch();
  Sched sch;
  sch.init(p);
  int tile, kb, ke;
  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      const uint64_t pol_w = tc::policy_evict_first(), pol_x = tc::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      // The weights never depend on the previous kernel: the first STAGES weight tiles are
      // requested before waiting for it; their activation tiles follow once it has finished.
      int pend_k[STAGES], pend_nt[STAGES], pend_st[STAGES];
      int npend = 0;
      bool dep_done = false;
      auto flush_pending = [&]() {
        pdl_wait();
        dep_done = true;
        for (int i = 0; i < npend; ++i) {
          tc::tma_load_2d(sX + pend_st[i] * kXBytes, &tx, &full[pend_st[i]], pend_k[i] * 64,
                          pend_nt[i] * BN, pol_x);
          if (!SPLIT)
            tc::tma_load_2d(sX + pend_st[i] * kXBytes + kXTile, &tx, &full[pend_st[i]],
                            pend_k[i] * 64, p.act_lo + pend_nt[i] * BN, pol_x);
        }
        npend = 0;
      };
      while (ok && sch.next(p, tile, kb, ke)) {
        const int rb = tile / p.NT, nt = tile % p.NT;
        const int y0 = p.epi == EPI_SWIGLU ? rb * 64 : rb * 128;
        const int y1 = p.epi == EPI_SWIGLU ? p.F + rb * 64 : rb * 128 + 64;
        for (int k = kb; k < ke; ++k) {
          if (!wait_or_abort(&empty[stage], phase ^ 1, sflag + 1)) {
            report_timeout(p, sflag + 1, 1);
            ok = false;
            break;
          }
          tc::mbar_expect_tx(&full[stage], kAStage + kXBytes);
          tc::tma_load_2d(sA + stage * kAStage, &tw, &full[stage], k * 64, y0, pol_w);
          tc::tma_load_2d(sA + stage * kAStage + 8192, &tw, &full[stage], k * 64, y1, pol_w);
          if (WLO) {
            tc::tma_load_2d(sA + stage * kAStage + kABytes, &twl, &full[stage], k * 64, y0, pol_w);
            tc::tma_load_2d(sA + stage * kAStage + kABytes + 8192, &twl, &full[stage], k * 64, y1,
                            pol_w);
          }
          if (dep_done) {
            tc::tma_load_2d(sX + stage * kXBytes, &tx, &full[stage], k * 64, nt * BN, pol_x);
            if (!SPLIT)
              tc::tma_load_2d(sX + stage * kXBytes + kXTile, &tx, &full[stage], k * 64,
                              p.act_lo + nt * BN, pol_x);
          } else {
            pend_k[npend] = k;
            pend_nt[npend] = nt;
            pend_st[npend] = stage;
            if (++npend == STAGES) flush_pending();
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!dep_done) flush_pending();
      // never leave with copies in flight: wait for the last loads issued to each stage
      for (int i = 0; i < STAGES && i < issued; ++i) {
        if (--stage < 0) {
          stage = STAGES - 1;
          phase ^= 1;
        }
        tc::mbar_wait(&full[stage], phase);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && !SPLIT) {  // ---- MMA issuer, prefill: a fresh accumulator per k-block
      int stage = 0, a = 0;
      uint32_t phase = 0, aphase = 0;
      bool ok = true;
      while (ok && sch.next(p, tile, kb, ke)) {
        for (int k = kb; k < ke; ++k) {
          const bool first = (k - kb) % kDrainEvery == 0;
          const bool last = (k - kb) % kDrainEvery == kDrainEvery - 1 || k == ke - 1;
          if (first && !wait_or_abort(&acce[a], aphase ^ 1, sflag + 1)) {  // drained
            report_timeout(p, sflag + 1, 2);
            ok = false;
            break;
          }
          if (!wait_or_abort(&full[stage], phase, sflag + 1)) {
            report_timeout(p, sflag + 1, 3);
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t d = tmem + (uint32_t)(a * BN);
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sA + stage * kAStage));
          const uint64_t xd = tc::sdesc_sw128(tc::smem_u32(sX + stage * kXBytes));
          const uint64_t ld = tc::sdesc_sw128(tc::smem_u32(sX + stage * kXBytes + kXTile));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // hi parts (the group's first MMA overwrites)
            tc::mma_bf16(d, ad + 2 * kk, xd + 2 * kk, kIdesc, (kk > 0 || !first) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(d, ad + 2 * kk, ld + 2 * kk, kIdesc, 1u);
          if (WLO) {  // the weights' lo parts against the operand's hi parts
            const uint64_t al = tc::sdesc_sw128(tc::smem_u32(sA + stage * kAStage + kABytes));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(d, al + 2 * kk, xd + 2 * kk, kIdesc, 1u);
          }
          tc::mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (last) {
            tc::mma_commit(&accf[a]);
            if (++a == kPrefillAcc) {
              a = 0;
              aphase ^= 1;
            }
          }
        }
      }
      tc::mma_commit(done);
      tc::mbar_wait(done, 0);
    } else if (lane == 0) {  // ---- MMA issuer, decode: one accumulator per tile, two buffers
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      while (ok && sch.next(p, tile, kb, ke)) {
        if (!wait_or_abort(&acce[acc], acc_phase ^ 1, sflag + 1)) {
          report_timeout(p, sflag + 1, 2);
          break;
        }
        tc::tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        for (int k = kb; k < ke; ++k) {
          if (!wait_or_abort(&full[stage], phase, sflag + 1)) {
            report_timeout(p, sflag + 1, 3);
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sA + stage * kAStage));
          const uint64_t xd = tc::sdesc_sw128(tc::smem_u32(sX + stage * kXBytes));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16(d, ad + 2 * kk, xd + 2 * kk, kIdesc, (k > kb || kk > 0) ? 1u : 0u);
          tc::mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit(&accf[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // all MMAs of this thread complete before TMEM is released
      tc::mma_commit(done);
      tc::mbar_wait(done, 0);
    }
  } else {  // ---- epilogue warps 2..5
    pdl_wait();  // outputs and the stream-K scratch are shared with the previous kernel
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    if (SPLIT && p.ss_in) {  // RMSNorm factor of each decode row, from the per-tile sums
      if (r < p.n_act) {
        float s = 0.f;
        for (int t = 0; t < p.ss_tiles; ++t) s += p.ss_in[(size_t)t * p.ss_ld + r];
        rinv[r] = rsqrtf(s / (float)p.K + p.eps);
      }
      tc::named_bar_sync(1, 128);
    }
    if (!SPLIT) {
      // prefill: every k-block's accumulator is added into fp32 sums (round to nearest) as soon
      // as its MMAs are done, then handed back; the tile's epilogue runs on the sums
      int a = 0;
      uint32_t aphase = 0;
      bool ok = true;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
      while (ok && sch.next(p, tile, kb, ke)) {
        const int rb = tile / p.NT, nt = tile % p.NT;
        float sums[BN];
#pragma unroll
        for (int j = 0; j < BN; ++j) sums[j] = 0.f;
        for (int k = kb; k < ke; k += kDrainEvery) {
          if (!wait_or_abort(&accf[a], aphase, sflag + 1)) {
            report_timeout(p, sflag + 1, 4);
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < BN; c0 += 64) {
            uint32_t raw[64];
#pragma unroll
            for (int c = 0; c < 4; ++c) tc::tmem_ld16(tbase + (uint32_t)(a * BN + c0 + 16 * c), raw + 16 * c);
            tc::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 64; ++j) sums[c0 + j] += __uint_as_float(raw[j]);
          }
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&acce[a]);
          if (++a == kPrefillAcc) {
            a = 0;
            aphase ^= 1;
          }
        }
        if (!ok) break;
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float res[32];
          load_residual<32>(p, rb, r, nt * BN + c0, res);
          finish<32>(p, rb, r, sums + c0, nt * BN + c0, swx, rinv, res, tcepi::epi_src_global(p));
        }
      }
    } else {
    int acc = 0;
    uint32_t acc_phase = 0;
    while (sch.next(p, tile, kb, ke)) {
      if (!wait_or_abort(&accf[acc], acc_phase, sflag + 1)) {
        report_timeout(p, sflag + 1, 4);
        break;
      }
      tc::tc_fence_after();
      const int rb = tile / p.NT, nt = tile % p.NT;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (SPLIT) {
        constexpr int H = BN / 2;
        uint32_t raw[BN];
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) tc::tmem_ld16(taddr + 16 * c, raw + 16 * c);
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acce[acc]);
        float vals[H];
#pragma unroll
        for (int n = 0; n < H; ++n) vals[n] = __uint_as_float(raw[n]) + __uint_as_float(raw[n + H]);
        if (kb == 0 && ke == p.KS) {
          float res[H];
          load_residual<H>(p, rb, r, 0, res);
          finish<H>(p, rb, r, vals, 0, swx, rinv, res, tcepi::epi_src_global(p));
        } else {
          const int first = cta_of_unit(p.U, gridDim.x, (long long)tile * p.KS);
          const int slot = blockIdx.x - first;
          float* pp = p.part + ((size_t)tile * p.slots + slot) * H * 128;
#pragma unroll
          for (int n = 0; n < H; ++n)
            if (n < p.n_act) pp[n * 128 + r] = vals[n];
          __threadfence();
          tc::named_bar_sync(1, 128);
          if (threadIdx.x == 64) {
            const int old = atomicAdd(p.cnt + tile, ke - kb);
            sflag[0] = (old + (ke - kb) == p.KS) ? 1 : 0;
          }
          tc::named_bar_sync(1, 128);
          if (sflag[0]) {
            __threadfence();
            const int last = cta_of_unit(p.U, gridDim.x, (long long)tile * p.KS + p.KS - 1);
            float res[H], sum[H];
            load_residual<H>(p, rb, r, 0, res);
#pragma unroll
            for (int n = 0; n < H; ++n) sum[n] = 0.f;
            // partial slots in order (a fixed summation order keeps results reproducible),
            // the loads of kChunk slots in flight together
            constexpr int kChunk = H <= 16 ? 4 : 2;
            const int nslots = last - first + 1;
            for (int s0 = 0; s0 < nslots; s0 += kChunk) {
              float ld[kChunk][H];
#pragma unroll
              for (int i = 0; i < kChunk; ++i) {
                const float* ps = p.part + ((size_t)tile * p.slots + s0 + i) * H * 128;
#pragma unroll
                for (int n = 0; n < H; ++n)
                  ld[i][n] = (s0 + i < nslots && n < p.n_act) ? __ldcg(ps + n * 128 + r) : 0.f;
              }
#pragma unroll
              for (int i = 0; i < kChunk; ++i)
                if (s0 + i < nslots) {
#pragma unroll
                  for (int n = 0; n < H; ++n) sum[n] += ld[i][n];
                }
            }
            finish<H>(p, rb, r, sum, 0, swx, rinv, res, tcepi::epi_src_global(p));
            if (threadIdx.x == 64) p.cnt[tile] = 0;
          }
        }
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int BN, int STAGES, bool SPLIT, bool WLO = false>
cudaError_t launch_inst(const CUtensorMap& tw, const CUtensorMap& tx, const TcParams& p, int grid,
                        cudaStream_t s, const CUtensorMap* twl = nullptr) {
  constexpr size_t smem = 1024 + STAGES * (kABytes * (WLO ? 2 : 1) + BN * 128 * (SPLIT ? 1 : 2)) +
                          512 + 128 * 33 * 4 + 256;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  auto kern = k_tc_linear<BN, STAGES, SPLIT, WLO>;
  cudaError_t rc = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (rc != cudaSuccess) return rc;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, tw, tx, WLO ? *twl : tw, p);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

}  // namespace

bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15) || (inner * 2) % 16) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_kblocks(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows,
                       uint32_t nk, uint64_t pair_rows) {
  auto fn = encode_fn();
  if (!fn || !base || (reinterpret_cast<uintptr_t>(base) & 15) || K % 64 || nk < 1 || box_rows > 256)
    return false;
  const cuuint32_t es[4] = {1, 1, 1, 1};
  if (pair_rows == 0) {
    // [k-block][row][64 columns]: one box is nk consecutive 64-column blocks of box_rows rows
    cuuint64_t dims[3] = {64, rows, K / 64};
    cuuint64_t strides[2] = {K * 2, 128};
    cuuint32_t box[3] = {64, box_rows, nk};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  // rows [0, 2 pair_rows) as two halves (gate, up): [k-block][half][row][64 columns]
  if (rows != 2 * pair_rows) return false;
  cuuint64_t dims[4] = {64, pair_rows, 2, K / 64};
  cuuint64_t strides[3] = {K * 2, pair_rows * K * 2, 128};
  cuuint32_t box[4] = {64, box_rows, 2, nk};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_split_bn(int n) { return n <= 8 ? 16 : (n <= 16 ? 32 : 64); }
int tc_plain_bn(int n) { return n <= 64 ? 64 : 128; }

// Plan and launch one projection.  p carries shapes, epilogue and outputs; this fills the
// schedule.  Returns false if the shape is outside what the kernel supports.
bool launch_tc_linear(const CUtensorMap& tw, const CUtensorMap& tx, TcParams p, bool split, int BN,
                      int num_sms, size_t part_floats, cudaStream_t s, const CUtensorMap* twl) {
  if (twl && split) return false;
  if (p.K % 64 || p.K <= 0 || p.n_act <= 0) return false;
  if (p.epi == EPI_SWIGLU && (p.F % 64 || p.M != 2 * p.F)) return false;
  if (!split && p.ss_in) return false;  // the per-column RMSNorm factors exist for decode rows only
  if (!split && p.act_lo < p.n_act) return false;  // prefill operands carry their lo parts
  p.RB = p.epi == EPI_SWIGLU ? p.F / 64 : (p.M + 127) / 128;
  p.KS = p.K / 64;
  if (split) {
    if (2 * p.n_act > BN) return false;
    p.NT = 1;
    p.streamk = 1;
    p.U = (long long)p.RB * p.KS;
    int G = (int)std::min<long long>(num_sms, p.U);
    // partial slots per tile: most CTAs whose ranges meet one tile
    for (;;) {
      int slots = 1;
      for (int t = 0; t < p.RB; ++t) {
        int f = cta_of_unit(p.U, G, (long long)t * p.KS);
        int l = cta_of_unit(p.U, G, (long long)t * p.KS + p.KS - 1);
        slots = std::max(slots, l - f + 1);
      }
      if ((size_t)p.RB * slots * (BN / 2) * 128 <= part_floats || G == 1) {
        p.slots = slots;
        break;
      }
      G = std::max(1, G / 2);
    }
    if ((size_t)p.RB * p.slots * (BN / 2) * 128 > part_floats) return false;
    cudaError_t rc;
    if (BN == 16) rc = launch_inst<16, kSplitStages, true>(tw, tx, p, G, s);
    else if (BN == 32) rc = launch_inst<32, kSplitStages, true>(tw, tx, p, G, s);
    else if (BN == 64) rc = launch_inst<64, kSplitStages, true>(tw, tx, p, G, s);
    else return false;
    return rc == cudaSuccess;
  }
  p.NT = (p.n_act + BN - 1) / BN;
  p.streamk = 0;
  p.U = (long long)p.RB * p.NT * p.KS;
  p.slots = 0;
  const int tiles = p.RB * p.NT;
  const int G = std::min(tiles, num_sms);
  cudaError_t rc;
  if (twl) {  // weights as hi + lo parts: a third tile per stage
    if (BN == 64) rc = launch_inst<64, 4, false, true>(tw, tx, p, G, s, twl);
    else if (BN == 128) rc = launch_inst<128, 3, false, true>(tw, tx, p, G, s, twl);
    else return false;
  } else if (BN == 64) rc = launch_inst<64, 6, false>(tw, tx, p, G, s);
  else if (BN == 128) rc = launch_inst<128, 4, false>(tw, tx, p, G, s);
  else return false;
  return rc == cudaSuccess;
}
