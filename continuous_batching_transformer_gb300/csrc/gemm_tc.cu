// gemm_tc.cu -- prefill projections y = x W^T on the 5th-generation tensor cores (sm_103a).
//
// Swap-AB: the weight rows are the MMA's M side (128 per tile), N tiles of 64 or 128 tokens
// its N side, whole tiles per CTA over a persistent grid.  Per CTA: one TMA producer thread
// streams 128x64 bf16 weight tiles and the tokens' 64-column operand tiles into a ring of
// 128-byte-swizzled shared-memory stages; two threads issue tcgen05.mma into TMEM; four
// epilogue warps read the accumulators back (tcgen05.ld) and apply the epilogue (store,
// residual add, or SwiGLU into the next projection's bf16 operand).
//
// The activations are bf16 hi/lo pairs (x = hi + lo: lo parts at row act_lo + t), so the
// operand carries fp32-grade precision; a stage holds both operand tiles.  One thread issues a
// tcgen05.mma only about every 60 ns whatever its shape, so the products are split over two
// issuers, each into accumulators of its own: issuer 0 takes hi(W) . x_hi, issuer 1 takes
// hi(W) . x_lo (and, for 4-bit weights expanded into bf16 hi + lo parts (WLO), lo(W) . x_hi;
// the lo . lo term is below 2^-16 of the product).
//
// The tensor core's fp32 accumulation rounds toward zero (measured: a relative bias of -4e-6
// over K = 4096, -1.5e-5 over K = 14336), and over a deep prefill the bias reaches the logits
// through the bf16 rounding of every appended K/V.  So every kDrainEvery k-blocks the issuers
// start fresh accumulators (two groups in flight, each a pair of accumulators, which fills the
// tensor memory at N = 128) and the epilogue warps add the finished pair into fp32 sums with
// round to nearest while the next group runs: the large accumulator takes only the hi . hi
// MMAs of one group.  Measured on a 4 x 1024-token 7B prefill (bf16): groups of 4, 8 and 16
// k-blocks take 226, 217 and 203 ms a call, against 142 ms for accumulators that run the whole
// K range and are read once per tile; a 32-layer prefill then decode stays within 1.6-1.8e-2
// of the double-precision oracle up to 8 k-blocks a group and exceeds 2e-2 at 16 and beyond.
#include <cudaTypedefs.h>

#include <algorithm>

#include "kernels.h"
#include "tc_common.cuh"
#include "tc_epilogue.cuh"

namespace {

using tcepi::finish;
using tcepi::load_residual;

// warp 0 TMA, warps 1 and 6 MMA (warp 1 also allocates TMEM), warps 2..5 epilogue
constexpr int kThreads = 224;
constexpr int kABytes = 128 * 128;  // 128 rows x 64 bf16
constexpr int kDrainEvery = 8;      // k-blocks a group of accumulators takes

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

template <int BN, int STAGES, bool WLO>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_linear(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx,
                const __grid_constant__ CUtensorMap twl, const TcParams p) {
  constexpr int kXTile = BN * 128;                      // one [BN tokens][64] operand tile
  constexpr int kXBytes = 2 * kXTile;                   // its hi and lo tiles
  constexpr int kAStage = WLO ? 2 * kABytes : kABytes;  // weight tile (+ its lo parts)
  constexpr uint32_t kTmemCols = 4 * BN;                // 2 groups x (issuer 0, issuer 1)
  constexpr uint32_t kIdesc = tc::idesc_bf16(128, BN);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sX = smem + STAGES * kAStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(sX + STAGES * kXBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;  // per group buffer: both issuers' MMAs done
  uint64_t* acce = accf + 2;        // per group buffer: added up by the epilogue
  uint64_t* done = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* sflag = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [1] abort
  float* swx = reinterpret_cast<float*>(smem + STAGES * (kAStage + kXBytes) + 512);
  float* rinv = swx + 128 * 33;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 2);  // both issuers' MMAs have read the stage
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&accf[b], 2);
      tc::mbar_init(&acce[b], 4);
    }
    tc::mbar_init(done, 2);
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
  const int tiles = p.RB * p.NT;

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
      auto load_x = [&](int st, int k, int nt) {
        tc::tma_load_2d(sX + st * kXBytes, &tx, &full[st], k * 64, nt * BN, pol_x);
        tc::tma_load_2d(sX + st * kXBytes + kXTile, &tx, &full[st], k * 64, p.act_lo + nt * BN,
                        pol_x);
      };
      auto flush_pending = [&]() {
        pdl_wait();
        dep_done = true;
        for (int i = 0; i < npend; ++i) load_x(pend_st[i], pend_k[i], pend_nt[i]);
        npend = 0;
      };
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        const int rb = tile / p.NT, nt = tile % p.NT;
        const int y0 = p.epi == EPI_SWIGLU ? rb * 64 : rb * 128;
        const int y1 = p.epi == EPI_SWIGLU ? p.F + rb * 64 : rb * 128 + 64;
        for (int k = 0; k < p.KS; ++k) {
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
            load_x(stage, k, nt);
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
  } else if (warp == 1 || warp == 6) {
    if (lane == 0) {  // ---- MMA issuers
      const int iss = warp == 1 ? 0 : 1;
      int stage = 0, b = 0;
      uint32_t phase = 0, bphase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        for (int k = 0; k < p.KS; ++k) {
          const bool first = k % kDrainEvery == 0;
          const bool last = k % kDrainEvery == kDrainEvery - 1 || k == p.KS - 1;
          if (first && !wait_or_abort(&acce[b], bphase ^ 1, sflag + 1)) {  // added up
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
          const uint32_t d = tmem + (uint32_t)((2 * b + iss) * BN);
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sA + stage * kAStage));
          const uint64_t xd = tc::sdesc_sw128(tc::smem_u32(sX + stage * kXBytes + iss * kXTile));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // a group's first MMA overwrites the accumulator
            tc::mma_bf16(d, ad + 2 * kk, xd + 2 * kk, kIdesc, (kk > 0 || !first) ? 1u : 0u);
          if (WLO && iss == 1) {  // the weights' lo parts against the operand's hi parts
            const uint64_t al = tc::sdesc_sw128(tc::smem_u32(sA + stage * kAStage + kABytes));
            const uint64_t xh = tc::sdesc_sw128(tc::smem_u32(sX + stage * kXBytes));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) tc::mma_bf16(d, al + 2 * kk, xh + 2 * kk, kIdesc, 1u);
          }
          tc::mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
          if (last) {
            tc::mma_commit(&accf[b]);
            b ^= 1;
            if (b == 0) bphase ^= 1;
          }
        }
      }
      // all MMAs of both issuers complete before TMEM is released
      tc::mma_commit(done);
      tc::mbar_wait(done, 0);
    }
  } else {  // ---- epilogue warps 2..5
    pdl_wait();  // outputs are shared with the previous kernel
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16);
    int b = 0;
    uint32_t bphase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      const int rb = tile / p.NT, nt = tile % p.NT;
      float sums[BN];
#pragma unroll
      for (int j = 0; j < BN; ++j) sums[j] = 0.f;
      for (int k = 0; k < p.KS; k += kDrainEvery) {
        if (!wait_or_abort(&accf[b], bphase, sflag + 1)) {
          report_timeout(p, sflag + 1, 4);
          ok = false;
          break;
        }
        tc::tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t hi[32], lo[32];
          tc::tmem_ld16(tbase + (uint32_t)(2 * b * BN + c0), hi);
          tc::tmem_ld16(tbase + (uint32_t)(2 * b * BN + c0 + 16), hi + 16);
          tc::tmem_ld16(tbase + (uint32_t)((2 * b + 1) * BN + c0), lo);
          tc::tmem_ld16(tbase + (uint32_t)((2 * b + 1) * BN + c0 + 16), lo + 16);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) sums[c0 + j] += __uint_as_float(hi[j]) + __uint_as_float(lo[j]);
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&acce[b]);
        b ^= 1;
        if (b == 0) bphase ^= 1;
      }
      if (tc::named_bar_any(1, 128, !ok)) {  // one decision for the 128 threads
        ok = false;
        break;
      }
      // one copy of the (large) epilogue code: each 16-column chunk is moved out of the sums
      // by constant indices (so they stay in registers) and finished in a loop that is not
      // unrolled -- four inlined copies crowd the issuing warps out of the instruction cache
#pragma unroll 1
      for (int c = 0; c < BN / 16; ++c) {
        float v[16], res[16];
#pragma unroll
        for (int cc = 0; cc < BN / 16; ++cc)
          if (cc == c) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = sums[16 * cc + j];
          }
        load_residual<16>(p, rb, r, nt * BN + 16 * c, res);
        finish<16>(p, rb, r, v, nt * BN + 16 * c, swx, rinv, res, tcepi::epi_src_global(p));
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

template <int BN, int STAGES, bool WLO>
cudaError_t launch_inst(const CUtensorMap& tw, const CUtensorMap& tx, const TcParams& p, int grid,
                        cudaStream_t s, const CUtensorMap* twl) {
  constexpr size_t smem =
      1024 + STAGES * (kABytes * (WLO ? 2 : 1) + 2 * BN * 128) + 512 + 128 * 33 * 4 + 256;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  auto kern = k_tc_linear<BN, STAGES, WLO>;
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

// Plan and launch one prefill projection: N tiles of BN (64 or 128) tokens, whole tiles per CTA
// over min(tiles, SMs) CTAs.  p carries shapes, epilogue and outputs.  Returns false if the
// shape is outside what the kernel supports (decode rows go to launch_tc_csk / launch_q4_rd).
bool launch_tc_linear(const CUtensorMap& tw, const CUtensorMap& tx, TcParams p, bool split, int BN,
                      int num_sms, cudaStream_t s, const CUtensorMap* twl) {
  if (split) return false;
  if (p.K % 64 || p.K <= 0 || p.n_act <= 0) return false;
  if (p.epi == EPI_SWIGLU && (p.F % 64 || p.M != 2 * p.F)) return false;
  if (p.ss_in) return false;               // the folded RMSNorm is a decode form
  if (p.act_lo < p.n_act) return false;    // the operand carries its lo parts
  p.RB = p.epi == EPI_SWIGLU ? p.F / 64 : (p.M + 127) / 128;
  p.KS = p.K / 64;
  p.NT = (p.n_act + BN - 1) / BN;
  const int G = std::min(p.RB * p.NT, num_sms);
  cudaError_t rc;
  if (twl) {  // weights as hi + lo parts: a third tile per stage
    if (BN == 64) rc = launch_inst<64, 4, true>(tw, tx, p, G, s, twl);
    else if (BN == 128) rc = launch_inst<128, 3, true>(tw, tx, p, G, s, twl);
    else return false;
  } else if (BN == 64) {
    rc = launch_inst<64, 6, false>(tw, tx, p, G, s, nullptr);
  } else if (BN == 128) {
    rc = launch_inst<128, 4, false>(tw, tx, p, G, s, nullptr);
  } else {
    return false;
  }
  return rc == cudaSuccess;
}
