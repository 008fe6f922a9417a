// gemm_csk.cu -- decode projections y = x W^T with cluster split-K on the 5th-generation tensor
// cores (sm_103a).
//
// Decode streams every weight once per step, so a projection is an HBM-bound stream split over
// all SMs.  With a few 128-row weight tiles per matrix (32 for a 4096-row output) the K
// dimension has to be split too, and the partial sums of a tile meet somewhere.  Through global
// memory that hand-off is slow on a streaming SM: a store, or any release fence, waits behind
// the ~128 KB of weight tiles the SM keeps in flight (microseconds).  Here the CTAs that split a
// tile form a thread-block cluster and reduce-scatter their partial sums through distributed
// shared memory: the tile's N/2 output columns (tokens) are cut into one chunk per rank, each
// CTA writes every peer's columns of its 128-row partial sums into that peer's inbox with
// st.async (which signals the peer's mbarrier with the byte count), and each CTA adds the C
// partials of its own columns in rank order (a fixed order, so results do not depend on timing
// or on which CTA adds them) and runs the epilogue for those columns.  No partial sum touches
// global memory, no fence is executed, and the combine and epilogue are spread over the
// cluster instead of falling on one CTA per tile.
//
// Layout of the work: tile t of the matrix belongs to cluster t % NC (clusters take tiles
// cid, cid + NC, ...), rank r of the cluster streams k-blocks [r*KS/C, (r+1)*KS/C) of each of
// its cluster's tiles and finishes columns [r*chunk, (r+1)*chunk) of each.  Per CTA
// the pipeline: a TMA producer warp for the weights (which stream from the kernel's start, before
// the previous kernel finishes), a TMA producer warp for the operand tiles (after it), two MMA
// warps (swap-AB: 128 weight rows x N operand rows, bf16 hi/lo operand parts, fp32
// accumulators in TMEM), four epilogue warps.
#include <algorithm>
#include <map>
#include <tuple>

#include "kernels.h"
#include "csk_common.cuh"
#include "tc_common.cuh"
#include "tc_epilogue.cuh"

namespace {

using tcepi::finish;
using tcepi::load_residual;

// warp 0 TMA (weights), warp 7 TMA (operand), warps 1 and 6 MMA (warp 1 also allocates TMEM),
// warps 2..5 epilogue
constexpr int kThreads = 256;
constexpr int kABytes = 128 * 128;  // 128 rows x 64 bf16
constexpr int kMaxStages = 8;
constexpr int kMaxSlots = 16;       // tiles of one cluster in a launch (an inbox barrier each)
constexpr int kSmemBudget = 227 * 1024;
// One thread issues a tcgen05.mma about every 60 ns whatever its shape, so at N = 16..64 one
// issuer caps an SM near 65 GB/s of weights (8 MMAs a 32 KB stage); two issuers, each taking
// one of a stage's two 64-column blocks into accumulators of its own, lift that cap.
constexpr int kIssuers = 2;
constexpr int kAcc = 2;             // accumulators per issuer and tile (see k_tc_csk)

using csk::cluster_rank;
using csk::cluster_sync;
using csk::wait_or_abort;

__device__ __forceinline__ void report_timeout(const TcParams& p, volatile int* abort, int role) {
  *abort = 1;
  if (atomicCAS(p.err, 0, CBT_DEV_TIMEOUT) == 0) p.err[1] = 200 + role;
}

struct Smem {
  uint8_t *a, *x;
  float *inbox, *swx, *rinv;
  float *cosv, *sinv;  // shared copies of the RoPE tables [n_act][64] (QKV)
  QueryRow* rows;      // shared copy of the row table [32] (QKV)
  uint64_t *full, *empty, *accf, *acce, *done, *inbox_full;
  uint32_t* tmem_slot;
  volatile int* sflag;
};

// inbox of a CTA: per tile of its cluster, the C - 1 other ranks' partial sums of its columns
template <int BN>
__host__ __device__ inline size_t inbox_floats(int C, int slots) {
  return C > 1 ? (size_t)slots * (C - 1) * 128 * csk::rs_chunk(BN / 2, C) : 0;
}

// shared copies of the RoPE tables: BN/2 rows x up to 64 pairs, cos and sin
template <int BN>
__host__ __device__ constexpr size_t rope_floats() {
  return (size_t)(BN / 2) * 64 * 2;
}

// qkv: the launch keeps shared copies of the RoPE tables and the row table
template <int BN>
__host__ __device__ size_t csk_smem_bytes(const CskPlan& q, bool qkv) {
  return 1024 + (size_t)q.stages * q.nk * (kABytes + BN * 128) + inbox_floats<BN>(q.C, q.slots) * 4 +
         (128 * 33 + 32) * 4 + (qkv ? rope_floats<BN>() * 4 + 32 * sizeof(QueryRow) : 0) + 512;
}

template <int BN>
__device__ __forceinline__ Smem carve(uint8_t* smem, const CskPlan& q, bool qkv) {
  Smem s;
  s.a = smem;
  s.x = s.a + q.stages * q.nk * kABytes;
  s.inbox = reinterpret_cast<float*>(s.x + q.stages * q.nk * BN * 128);
  s.swx = s.inbox + inbox_floats<BN>(q.C, q.slots);
  s.rinv = s.swx + 128 * 33;
  s.cosv = s.rinv + 32;
  s.sinv = s.cosv + (qkv ? rope_floats<BN>() / 2 : 0);
  s.rows = reinterpret_cast<QueryRow*>(s.sinv + (qkv ? rope_floats<BN>() / 2 : 0));
  s.full = reinterpret_cast<uint64_t*>(s.rows + (qkv ? 32 : 0));
  s.empty = s.full + kMaxStages;
  s.accf = s.empty + kMaxStages;
  s.acce = s.accf + 2;
  s.done = s.acce + 2;
  s.inbox_full = s.done + 1;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.inbox_full + kMaxSlots);
  s.sflag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);  // [1] abort
  return s;
}

// EPI: the launch's epilogue (p.epi), a template parameter so that each launch carries only
// its own epilogue code (all four inlined together crowd the instruction cache)
template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_csk(const __grid_constant__ CUtensorMap tw, const __grid_constant__ CUtensorMap tx,
             const TcParams p, const CskPlan q) {
  constexpr int H = BN / 2;  // operand rows: H hi parts, then H lo parts
  constexpr int kXBytes = BN * 128;  // operand tile of one 64-column block
  // two buffers (tiles in flight) of kIssuers x kAcc accumulators: issuer i's block of
  // super-block sb accumulates into its accumulator (sb - sb0) % kAcc, and the epilogue adds
  // all of them in fp32 (round to nearest) -- the tensor core's own fp32 accumulation rounds
  // toward zero, and the split divides that bias by kIssuers x kAcc
  static_assert(kCskBlocks == kIssuers, "one 64-column block of a stage per issuer");
  constexpr uint32_t kTmemCols = 2 * kIssuers * kAcc * BN < 32 ? 32 : 2 * kIssuers * kAcc * BN;
  constexpr uint32_t kIdesc = tc::idesc_bf16(128, BN);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const Smem sm = carve<BN>(base, q, EPI == EPI_QKV || EPI == EPI_QKVQ);
  const int S = q.stages, C = q.C, NK = q.nk;
  const int stage_a = NK * kABytes, stage_x = NK * kXBytes;  // bytes per stage
  volatile int* abort_flag = sm.sflag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = C > 1 ? cluster_rank() : 0u;
  const uint32_t lim = p.spin_limit ? p.spin_limit : tc::kSpinLimit;  // every wait's bound
  const int cid = blockIdx.x / C, NC = gridDim.x / C;
  const int Tc = cid < p.RB ? (p.RB - cid + NC - 1) / NC : 0;  // tiles cid, cid + NC, ...
  // this rank's stages: super-blocks of NK 64-column blocks [sb0, sb1) of each tile
  const int SB = p.KS / NK;
  const int sb0 = (int)((long long)rank * SB / C);
  const int sb1 = (int)((long long)(rank + 1) * SB / C);
  // this rank's columns of every tile (reduce-scatter), none for the last ranks of a wide split
  const int t0 = min(H, (int)rank * csk::rs_chunk(H, C)), t1 = min(H, t0 + csk::rs_chunk(H, C));
  const int owned = t1 > t0 ? Tc : 0;  // tiles whose inbox this CTA waits for

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&sm.full[s], 1);
      tc::mbar_init(&sm.empty[s], kIssuers);  // every issuer's MMAs have read the stage
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&sm.accf[a], kIssuers);
      tc::mbar_init(&sm.acce[a], 4);
    }
    tc::mbar_init(sm.done, kIssuers);
    for (int s = 0; s < kMaxSlots; ++s) tc::mbar_init(&sm.inbox_full[s], 1);
    // each tile's inbox receives the C - 1 other ranks' partial sums of this CTA's columns
    if (C > 1)
      for (int s = 0; s < owned; ++s)
        tc::mbar_expect_tx(&sm.inbox_full[s], (uint32_t)((C - 1) * 128 * (t1 - t0) * 4));
    sm.sflag[0] = 0;
    sm.sflag[1] = 0;
    tc::mbar_fence_init();
    tc::tma_prefetch_desc(&tw);
    tc::tma_prefetch_desc(&tx);
  }
  if (warp == 1) tc::tmem_alloc(sm.tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (C > 1) cluster_sync();  // peers' barriers are initialised before any st.async reaches them
  const uint32_t tmem = *sm.tmem_slot;
  pdl_launch();

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer of the weight tiles
      // The weights never depend on the previous kernel: they stream from the start, while the
      // operand producer (warp 7) waits for it.  Each stage's barrier expects both halves.
      const uint64_t pol_w = tc::policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int j = 0; j < Tc && ok && !p.stall_loads; ++j) {
        const int rb = cid + j * NC;
        for (int sb = sb0; sb < sb1; ++sb) {
          if (!wait_or_abort(&sm.empty[stage], phase ^ 1, abort_flag, lim)) {
            report_timeout(p, abort_flag, 1);
            ok = false;
            break;
          }
          tc::mbar_expect_tx(&sm.full[stage], stage_a + stage_x);
          // NK blocks of the tile's 128 weight rows (SwiGLU: 64 gate rows, then the same 64
          // features' up rows) in one box, each block a swizzled [128][64] tile
          if (EPI == EPI_SWIGLU)
            tc::tma_load_4d(sm.a + stage * stage_a, &tw, &sm.full[stage], 0, rb * 64, 0, sb * NK, pol_w);
          else
            tc::tma_load_3d(sm.a + stage * stage_a, &tw, &sm.full[stage], 0, rb * 128, sb * NK, pol_w);
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // never leave with copies in flight: wait for the last loads issued to each stage (weights
      // and operands complete the same barrier)
      for (int i = 0; i < S && i < issued; ++i) {
        if (--stage < 0) {
          stage = S - 1;
          phase ^= 1;
        }
        tc::mbar_wait(&sm.full[stage], phase, lim);
      }
    }
  } else if (warp == 7) {
    if (lane == 0) {  // ---- TMA producer of the operand tiles, once the previous kernel is done
      // A stage's operand may land before the weight producer's expect-tx: the barrier's
      // transaction count goes below zero until then, and the phase cannot complete without
      // that arrival.  Waiting on the same empty phases keeps this thread within one ring pass.
      const uint64_t pol_x = tc::policy_evict_last();
      pdl_wait();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int j = 0; j < Tc && ok && !p.stall_loads; ++j) {
        for (int sb = sb0; sb < sb1; ++sb) {
          if (!wait_or_abort(&sm.empty[stage], phase ^ 1, abort_flag, lim)) {
            report_timeout(p, abort_flag, 6);
            ok = false;
            break;
          }
          tc::tma_load_3d(sm.x + stage * stage_x, &tx, &sm.full[stage], 0, 0, sb * NK, pol_x);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1 || warp == 6) {
    if (lane == 0) {  // ---- MMA issuers: issuer iss takes block iss of every stage
      const int iss = warp == 1 ? 0 : 1;
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int j = 0; j < Tc && ok; ++j) {
        if (!wait_or_abort(&sm.acce[acc], acc_phase ^ 1, abort_flag, lim)) {
          report_timeout(p, abort_flag, 2);
          break;
        }
        tc::tc_fence_after();
        const uint32_t d0 = tmem + (uint32_t)((acc * kIssuers + iss) * kAcc * BN);
        for (int sb = sb0; sb < sb1; ++sb) {
          const uint32_t d = d0 + (uint32_t)(((sb - sb0) % kAcc) * BN);
          if (!wait_or_abort(&sm.full[stage], phase, abort_flag, lim)) {
            report_timeout(p, abort_flag, 3);
            ok = false;
            break;
          }
          tc::tc_fence_after();
          for (int jj = iss; jj < NK; jj += kIssuers) {
            const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sm.a + stage * stage_a + jj * kABytes));
            const uint64_t xd = tc::sdesc_sw128(tc::smem_u32(sm.x + stage * stage_x + jj * kXBytes));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_bf16(d, ad + 2 * kk, xd + 2 * kk, kIdesc,
                           (sb - sb0 >= kAcc || jj > iss || kk > 0) ? 1u : 0u);
          }
          tc::mma_commit(&sm.empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc::mma_commit(&sm.accf[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // all MMAs of this thread complete before TMEM is released
      tc::mma_commit(sm.done);
      tc::mbar_wait(sm.done, 0, lim);
    }
  } else {  // ---- epilogue warps 2..5: TMEM lanes 32q .. 32q + 31 = tile rows
    pdl_wait();  // outputs and norm statistics are shared with the previous kernel
    if (threadIdx.x == 64) stamp_begin(p.stamp);
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    if (p.ss_in) {  // RMSNorm factor of each decode row, from the per-tile sums of squares
      if (r < p.n_act) {
        float s = 0.f;
        for (int t = 0; t < p.ss_tiles; ++t) s += p.ss_in[(size_t)t * p.ss_ld + r];
        sm.rinv[r] = rsqrtf(s / (float)p.K + p.eps);
      }
    }
    tcepi::EpiSrc src = tcepi::epi_src_global(p);
    if (EPI == EPI_QKV || EPI == EPI_QKVQ) {
      // the row table and the RoPE tables in shared memory, loaded while the weights stream
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
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int j = 0; j < Tc; ++j) {
      const int rb = cid + j * NC;
      // the global inputs of this CTA's columns of the tile, requested before its accumulator
      // is ready
      float res[H];
      if (owned) {
        load_residual<H, EPI>(p, rb, r, 0, res, t0, t1);
        src.gn = tcepi::load_next_gain(p, rb, r);
        src.has_gn = true;
      }
      if (!wait_or_abort(&sm.accf[acc], acc_phase, abort_flag, lim)) {
        report_timeout(p, abort_flag, 4);
        break;
      }
      tc::tc_fence_after();
      float vals[H];
#pragma unroll
      for (int n = 0; n < H; ++n) vals[n] = 0.f;
      const uint32_t taddr =
          tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(acc * kIssuers * kAcc * BN);
      const int nacc = sb1 - sb0 < kAcc ? sb1 - sb0 : kAcc;  // per issuer
      const int niss = NK < kIssuers ? NK : kIssuers;        // issuers that had a block
      for (int a = 0; a < niss * kAcc; ++a) {  // issuer-major, a fixed order; hi + lo per column
        if (a % kAcc >= nacc) continue;
        uint32_t raw[BN];
#pragma unroll
        for (int c = 0; c < BN / 16; ++c)
          tc::tmem_ld16(taddr + (uint32_t)(a * BN) + 16 * c, raw + 16 * c);
        tc::tmem_ld_wait();
#pragma unroll
        for (int n = 0; n < H; ++n) vals[n] += __uint_as_float(raw[n]) + __uint_as_float(raw[n + H]);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm.acce[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
      float sum[H];
      const int got = csk::reduce_scatter<H>(vals, sum, sm.inbox, sm.inbox_full, j, rank, C, r,
                                             abort_flag, lim);
      // one decision for the 128 threads (the epilogue synchronises them)
      if (tc::named_bar_any(1, 128, got < 0)) {
        if (got < 0) report_timeout(p, abort_flag, 5);
        break;
      }
      if (got > 0) finish<H, EPI>(p, rb, r, sum, 0, sm.swx, sm.rinv, res, src, t0, t1);
    }
    // a CTA leaves only after its inboxes have been filled (bounded: a peer that gave up sends
    // nothing), so no st.async can land in a CTA that has exited
    if (C > 1 && threadIdx.x == 64)
      for (int s = 0; s < owned; ++s) tc::mbar_wait(&sm.inbox_full[s], 0, lim);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) stamp_end(p.stamp);
  if (C > 1) cluster_sync();
}

// cluster dims and PDL on one launch
template <int BN, int EPI>
cudaError_t launch_csk(const CUtensorMap& tw, const CUtensorMap& tx, const TcParams& p,
                       const CskPlan& q, cudaStream_t s) {
  const size_t smem = csk_smem_bytes<BN>(q, EPI == EPI_QKV || EPI == EPI_QKVQ);
  auto kern = k_tc_csk<BN, EPI>;
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
  return cudaLaunchKernelEx(&cfg, kern, tw, tx, p, q);
}

template <int BN>
cudaError_t launch_csk_epi(const CUtensorMap& tw, const CUtensorMap& tx, const TcParams& p,
                           const CskPlan& q, cudaStream_t s) {
  switch (p.epi) {
    case EPI_STORE: return launch_csk<BN, EPI_STORE>(tw, tx, p, q, s);
    case EPI_ADD: return launch_csk<BN, EPI_ADD>(tw, tx, p, q, s);
    case EPI_SWIGLU: return launch_csk<BN, EPI_SWIGLU>(tw, tx, p, q, s);
    case EPI_QKV: return launch_csk<BN, EPI_QKV>(tw, tx, p, q, s);
    case EPI_QKVQ: return launch_csk<BN, EPI_QKVQ>(tw, tx, p, q, s);
  }
  return cudaErrorInvalidValue;
}

// most clusters of C CTAs (each with `smem` bytes) resident at once, cached per configuration
template <int BN>
int active_clusters(int C, size_t smem) {
  static std::map<std::pair<int, size_t>, int> cache;
  auto key = std::make_pair(C, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  auto kern = k_tc_csk<BN, EPI_ADD>;  // every epilogue's instance has the same shape
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

}  // namespace

// The cluster shape is chosen from the matrix shape alone (the same for every operand width),
// so a row's result does not depend on how many rows share the step: minimise the k-blocks
// the busiest CTA streams, ceil(RB / NC) * ceil(KS / C), over cluster sizes whose clusters can
// all be resident at once.
bool csk_plan(int RB, int KS, int BN, int num_sms, CskPlan* out) {
  if (RB <= 0 || KS <= 0 || num_sms <= 0) return false;
  static const int kSizes[] = {1, 2, 3, 4, 6, 8};
  double best = 1e30;
  CskPlan bp{};
  if (KS % kCskBlocks) return false;
  const int SB = KS / kCskBlocks;
  for (int C : kSizes) {
    if (C > SB || C > num_sms) continue;
    // shape part of the plan, sized for the widest operand (N = 64)
    CskPlan q{};
    q.nk = kCskBlocks;
    q.C = C;
    q.NC = std::min(RB, num_sms / C);
    const int tmax = (RB + q.NC - 1) / q.NC;
    q.slots = C > 1 ? tmax : 0;
    if (q.slots > kMaxSlots) continue;
    q.stages = 2;  // the shallowest pipeline a launch may get
    if (csk_smem_bytes<64>(q, true) > (size_t)kSmemBudget) continue;
    const int fit = active_clusters<64>(C, csk_smem_bytes<64>(q, true));
    if (fit <= 0) continue;
    if (fit < q.NC) q.NC = fit;
    const int tmax2 = (RB + q.NC - 1) / q.NC;
    q.slots = C > 1 ? tmax2 : 0;
    if (q.slots > kMaxSlots) continue;
    const double cost = (double)tmax2 * ((SB + C - 1) / C) * kCskBlocks + (C > 1 ? 2.0 : 0.0) + 0.01 * C;
    if (cost < best) {
      best = cost;
      bp = q;
    }
  }
  if (best >= 1e30) return false;
  // pipeline depth for this operand width (the deepest that fits any epilogue)
  bp.stages = kMaxStages;
  auto smem = [&](const CskPlan& q) {
    return BN == 16 ? csk_smem_bytes<16>(q, true)
                    : BN == 32 ? csk_smem_bytes<32>(q, true) : csk_smem_bytes<64>(q, true);
  };
  while (bp.stages > 2 && smem(bp) > (size_t)kSmemBudget) --bp.stages;
  if (smem(bp) > (size_t)kSmemBudget) return false;
  *out = bp;
  return true;
}

bool launch_tc_csk(const CUtensorMap& tw, const CUtensorMap& tx, TcParams p, int BN, int num_sms,
                   cudaStream_t s) {
  if (p.K % 64 || p.K <= 0 || p.n_act <= 0 || 2 * p.n_act > BN) return false;
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
    if (!csk_plan(p.RB, p.KS, BN, num_sms, &q)) return false;
    plans[key] = q;
  }
  cudaError_t rc;
  if (BN == 16) rc = launch_csk_epi<16>(tw, tx, p, q, s);
  else if (BN == 32) rc = launch_csk_epi<32>(tw, tx, p, q, s);
  else if (BN == 64) rc = launch_csk_epi<64>(tw, tx, p, q, s);
  else return false;
  return rc == cudaSuccess;
}
