// gemm_csk.cu -- decode projections y = x W^T with cluster split-K on the 5th-generation tensor
// cores (sm_103a), one projection per launch or a chain of them.
//
// Decode streams every weight once per step, so a projection is an HBM-bound stream split over
// all SMs.  With a few 128-row weight tiles per matrix (32 for a 4096-row output) the K
// dimension has to be split too, and the partial sums of a tile meet somewhere.  Through global
// memory that hand-off is slow on a streaming SM: a store, or any release fence, waits behind
// the ~128 KB of weight tiles the SM keeps in flight (microseconds).  Here the CTAs that split a
// tile form a thread-block cluster and hand their partial sums to the tile's owner through
// distributed shared memory: each sender writes its 128 rows x N/2 fp32 sums into the owner's
// inbox with st.async, which signals the owner's mbarrier with the byte count; the owner adds
// the partials in rank order (a fixed order, so results do not depend on timing) and runs the
// epilogue.  No partial sum touches global memory and no fence is executed.
//
// Layout of the work: tile t of the matrix belongs to cluster t % NC (clusters take tiles
// cid, cid + NC, ...), rank r of the cluster streams k-blocks [r*KS/C, (r+1)*KS/C) of each of
// its cluster's tiles, and tile j of a cluster (in that order) is owned by rank j % C.  Per CTA
// the pipeline is the one of gemm_tc.cu: a TMA producer warp (weights requested before the
// previous kernel finishes, operand tiles after), an MMA warp (swap-AB: 128 weight rows x N
// operand rows, bf16 hi/lo operand parts, fp32 accumulators in TMEM), four epilogue warps.
//
// A chain runs up to four projections of a decode step that follow each other with nothing in
// between -- O, gate/up, down and the next layer's QKV (or the lm_head) -- in one persistent
// launch.  Between two phases all CTAs meet at a grid barrier (a counter in global memory): a
// phase's operand and its epilogue's inputs are the previous phases' outputs.  The weights do
// not depend on anything, so the producer keeps streaming the next phase's weight tiles into
// the ring while the current phase's last MMAs, partial-sum hand-offs, epilogues and the
// barrier complete; only the (small) operand tiles wait for the barrier.  The kernel
// boundaries of those projections, and the pipeline fill each of them would start with, go.
#include <algorithm>
#include <map>
#include <tuple>
#include <vector>

#include "kernels.h"
#include "csk_common.cuh"
#include "tc_common.cuh"
#include "tc_epilogue.cuh"

namespace {

using tcepi::finish;
using tcepi::load_residual;

constexpr int kThreads = 192;       // warp 0 TMA, warp 1 MMA (+TMEM alloc), warps 2..5 epilogue
constexpr int kABytes = 128 * 128;  // 128 rows x 64 bf16
constexpr int kMaxStages = 8;
constexpr int kMaxSlots = 4;        // tiles one CTA owns in one phase
constexpr int kSmemBudget = 227 * 1024;
constexpr int kAcc = 4;             // accumulators per tile (see k_tc_csk)

using csk::cluster_rank;
using csk::cluster_sync;
using csk::wait_or_abort;

// one projection of a launch: its weights and operand as tensor maps, its epilogue parameters
struct CskPhase {
  CUtensorMap tw, tx;
  TcParams p;
};

struct CskChainArgs {
  CskPhase ph[kMaxCskPhases];
  int n;                    // phases
  unsigned long long* bar;  // [n - 1] grid barrier counters, zero at the launch's start
  unsigned long long* stamp;
};

__device__ __forceinline__ void report_timeout(const TcParams& p, volatile int* abort, int role) {
  *abort = 1;
  if (atomicCAS(p.err, 0, CBT_DEV_TIMEOUT) == 0) p.err[1] = 200 + role;
}

struct Smem {
  uint8_t *a, *x;
  float *inbox, *swx, *rinv;
  float *cosv, *sinv;  // shared copies of the RoPE tables [n_act][64] (QKV)
  QueryRow* rows;      // shared copy of the row table [32] (QKV)
  uint64_t *full, *empty, *accf, *acce, *done, *inbox_full;  // inbox_full: [phase][slot]
  uint64_t* bar_target;  // [phase]: the count barrier `phase` completes at (0: not yet known)
  uint32_t* tmem_slot;
  volatile int* sflag;
};

// inbox of a CTA: per owned tile, the partial sums of the C - 1 other ranks
template <int BN>
__host__ __device__ constexpr size_t inbox_floats(int C, int slots) {
  return (size_t)slots * (C - 1) * 128 * (BN / 2);
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
         (128 * 33 + 32) * 4 + (qkv ? rope_floats<BN>() * 4 + 32 * sizeof(QueryRow) : 0) + 768;
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
  s.bar_target = s.inbox_full + kMaxCskPhases * kMaxSlots;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.bar_target + kMaxCskPhases);
  s.sflag = reinterpret_cast<volatile int*>(s.tmem_slot + 1);  // [1] abort
  return s;
}

// where a CTA works in one phase: its tiles cid, cid + NC, ... and its k-range [sb0, sb1) of
// super-blocks of each
struct Geo {
  int Tc, sb0, sb1, owned;
};
__device__ __forceinline__ Geo geo_of(const TcParams& p, int cid, int NC, int C, uint32_t rank,
                                      int NK) {
  Geo g;
  g.Tc = cid < p.RB ? (p.RB - cid + NC - 1) / NC : 0;
  const int SB = p.KS / NK;
  g.sb0 = (int)((long long)rank * SB / C);
  g.sb1 = (int)((long long)(rank + 1) * SB / C);
  g.owned = g.Tc > (int)rank ? (g.Tc - (int)rank + C - 1) / C : 0;
  return g;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until grid barrier k has been passed by every CTA: first for this CTA's own
// arrival (which records the count the barrier completes at), then for the count.
__device__ __forceinline__ bool grid_wait(const CskChainArgs& ch, const Smem& sm, int k,
                                          volatile int* abort) {
  volatile uint64_t* tgt = sm.bar_target + k;
  uint32_t i = 0;
  for (; i < tc::kSpinLimit && *tgt == 0; ++i) {
    if ((i & 1023) == 1023 && *abort) return false;
    if (i > 64) __nanosleep(64);
  }
  if (*tgt == 0) return false;
  const unsigned long long target = *tgt;
  for (i = 0; i < tc::kSpinLimit; ++i) {
    if (ld_acquire_u64(ch.bar + k) >= target) return true;
    if ((i & 255) == 255 && *abort) return false;
    __nanosleep(64);
  }
  return false;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_csk(const __grid_constant__ CskChainArgs ch, const CskPlan q) {
  constexpr int H = BN / 2;  // operand rows: H hi parts, then H lo parts
  constexpr int kXBytes = BN * 128;  // operand tile of one 64-column block
  // two buffers (tiles in flight) of kAcc accumulators: super-block sb accumulates into
  // accumulator (sb - sb0) % kAcc, and the epilogue adds them in fp32 (round to nearest) --
  // the tensor core's own fp32 accumulation rounds toward zero, and the split divides that
  // bias by kAcc
  constexpr uint32_t kTmemCols = 2 * kAcc * BN < 32 ? 32 : 2 * kAcc * BN;
  constexpr uint32_t kIdesc = tc::idesc_bf16(128, BN);
  constexpr uint32_t kPartBytes = 128 * H * 4;  // one CTA's partial sums of one tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  bool any_qkv = false;
  for (int k = 0; k < ch.n; ++k) any_qkv |= ch.ph[k].p.epi == EPI_QKV;
  const Smem sm = carve<BN>(base, q, any_qkv);
  const int S = q.stages, C = q.C, NK = q.nk, NP = ch.n;
  const int stage_a = NK * kABytes, stage_x = NK * kXBytes;  // bytes per stage
  volatile int* abort_flag = sm.sflag + 1;
  const TcParams& p0 = ch.ph[0].p;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = C > 1 ? cluster_rank() : 0u;
  const int cid = blockIdx.x / C, NC = gridDim.x / C;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&sm.full[s], 1);
      tc::mbar_init(&sm.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&sm.accf[a], 1);
      tc::mbar_init(&sm.acce[a], 4);
    }
    tc::mbar_init(sm.done, 1);
    for (int s = 0; s < kMaxCskPhases * kMaxSlots; ++s) tc::mbar_init(&sm.inbox_full[s], 1);
    // each tile this CTA owns, in every phase, receives the partial sums of the C - 1 other
    // ranks; armed before any peer can send (the cluster barrier below)
    if (C > 1)
      for (int k = 0; k < NP; ++k) {
        const Geo g = geo_of(ch.ph[k].p, cid, NC, C, rank, NK);
        for (int s = 0; s < g.owned; ++s)
          tc::mbar_expect_tx(&sm.inbox_full[k * kMaxSlots + s], (C - 1) * kPartBytes);
      }
    for (int k = 0; k < kMaxCskPhases; ++k) sm.bar_target[k] = 0;
    sm.sflag[0] = 0;
    sm.sflag[1] = 0;
    tc::mbar_fence_init();
    for (int k = 0; k < NP; ++k) {
      tc::tma_prefetch_desc(&ch.ph[k].tw);
      tc::tma_prefetch_desc(&ch.ph[k].tx);
    }
  }
  if (warp == 1) tc::tmem_alloc(sm.tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (C > 1) cluster_sync();  // peers' barriers are initialised before any st.async reaches them
  const uint32_t tmem = *sm.tmem_slot;
  pdl_launch();

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      const uint64_t pol_w = tc::policy_evict_first(), pol_x = tc::policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      // The weights never depend on earlier work: each stage's weight tile is requested as soon
      // as the ring has room.  A phase's operand tiles wait for what produces them -- the
      // previous kernel (phase 0) or grid barrier k - 1 (phase k) -- so until then they are
      // kept pending (stage, super-block, phase) and requested in order once it has passed.
      int pend_sb[kMaxStages], pend_st[kMaxStages], pend_ph[kMaxStages];
      int npend = 0, dep = -1;  // operands of phases <= dep may be requested
      auto satisfy = [&](int k) -> bool {
        pdl_wait();
        if (k > 0 && !grid_wait(ch, sm, k - 1, abort_flag)) return false;
        // the operand was written by other CTAs' generic stores and is read through TMA
        asm volatile("fence.proxy.async.global;" ::: "memory");
        dep = k;
        return true;
      };
      auto flush_pending = [&]() -> bool {
        for (int i = 0; i < npend; ++i) {
          if (pend_ph[i] > dep && !satisfy(pend_ph[i])) return false;
          tc::tma_load_3d(sm.x + pend_st[i] * stage_x, &ch.ph[pend_ph[i]].tx, &sm.full[pend_st[i]],
                          0, 0, pend_sb[i] * NK, pol_x);
        }
        npend = 0;
        return true;
      };
      for (int k = 0; k < NP && ok; ++k) {
        const CskPhase& A = ch.ph[k];
        const Geo g = geo_of(A.p, cid, NC, C, rank, NK);
        for (int j = 0; j < g.Tc && ok; ++j) {
          const int rb = cid + j * NC;
          for (int sb = g.sb0; sb < g.sb1; ++sb) {
            if (!wait_or_abort(&sm.empty[stage], phase ^ 1, abort_flag)) {
              report_timeout(p0, abort_flag, 1);
              ok = false;
              break;
            }
            tc::mbar_expect_tx(&sm.full[stage], stage_a + stage_x);
            // NK blocks of the tile's 128 weight rows (SwiGLU: 64 gate rows, then the same 64
            // features' up rows) in one box, each block a swizzled [128][64] tile
            if (A.p.epi == EPI_SWIGLU)
              tc::tma_load_4d(sm.a + stage * stage_a, &A.tw, &sm.full[stage], 0, rb * 64, 0, sb * NK,
                              pol_w);
            else
              tc::tma_load_3d(sm.a + stage * stage_a, &A.tw, &sm.full[stage], 0, rb * 128, sb * NK,
                              pol_w);
            if (dep >= k) {
              tc::tma_load_3d(sm.x + stage * stage_x, &A.tx, &sm.full[stage], 0, 0, sb * NK, pol_x);
            } else {
              pend_sb[npend] = sb;
              pend_st[npend] = stage;
              pend_ph[npend] = k;
              // a ring of nothing but pending stages: the consumer can take none of them
              if (++npend == S && !flush_pending()) {
                report_timeout(p0, abort_flag, 6);
                ok = false;
              }
            }
            ++issued;
            if (++stage == S) {
              stage = 0;
              phase ^= 1;
            }
            if (!ok) break;
          }
        }
      }
      if (ok && npend > 0 && !flush_pending()) report_timeout(p0, abort_flag, 6);
      // never leave with copies in flight: wait for the last loads issued to each stage
      for (int i = 0; i < S && i < issued; ++i) {
        if (--stage < 0) {
          stage = S - 1;
          phase ^= 1;
        }
        tc::mbar_wait(&sm.full[stage], phase);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int k = 0; k < NP && ok; ++k) {
        const Geo g = geo_of(ch.ph[k].p, cid, NC, C, rank, NK);
        for (int j = 0; j < g.Tc && ok; ++j) {
          if (!wait_or_abort(&sm.acce[acc], acc_phase ^ 1, abort_flag)) {
            report_timeout(p0, abort_flag, 2);
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t d0 = tmem + (uint32_t)(acc * kAcc * BN);
          for (int sb = g.sb0; sb < g.sb1; ++sb) {
            const uint32_t d = d0 + (uint32_t)(((sb - g.sb0) % kAcc) * BN);
            if (!wait_or_abort(&sm.full[stage], phase, abort_flag)) {
              report_timeout(p0, abort_flag, 3);
              ok = false;
              break;
            }
            tc::tc_fence_after();
            for (int jj = 0; jj < NK; ++jj) {
              const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sm.a + stage * stage_a + jj * kABytes));
              const uint64_t xd = tc::sdesc_sw128(tc::smem_u32(sm.x + stage * stage_x + jj * kXBytes));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tc::mma_bf16(d, ad + 2 * kk, xd + 2 * kk, kIdesc,
                             (sb - g.sb0 >= kAcc || jj > 0 || kk > 0) ? 1u : 0u);
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
      }
      // all MMAs of this thread complete before TMEM is released
      tc::mma_commit(sm.done);
      tc::mbar_wait(sm.done, 0);
    }
  } else {  // ---- epilogue warps 2..5: TMEM lanes 32q .. 32q + 31 = tile rows
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int k = 0; k < NP; ++k) {
      const TcParams& p = ch.ph[k].p;
      const Geo g = geo_of(p, cid, NC, C, rank, NK);
      // this phase's inputs (operand statistics, residual, the row and RoPE tables) are the
      // previous kernel's (phase 0) or the earlier phases' outputs (grid barrier k - 1)
      if (k == 0) {
        pdl_wait();
        if (threadIdx.x == 64) stamp_begin(ch.stamp);
      } else {
        bool good = ok;
        if (threadIdx.x == 64 && ok && !grid_wait(ch, sm, k - 1, abort_flag)) {
          report_timeout(p, abort_flag, 7);
          good = false;
        }
        if (threadIdx.x == 64) sm.sflag[0] = good ? 0 : 1;
        tc::named_bar_sync(1, 128);
        ok = sm.sflag[0] == 0;
        tc::named_bar_sync(1, 128);  // everyone has read the flag before it is reused
      }
      if (!ok) break;
      if (p.ss_in) {  // RMSNorm factor of each decode row, from the per-tile sums of squares
        if (r < p.n_act) {
          float s = 0.f;
          for (int t = 0; t < p.ss_tiles; ++t) s += p.ss_in[(size_t)t * p.ss_ld + r];
          sm.rinv[r] = rsqrtf(s / (float)p.K + p.eps);
        }
      }
      tcepi::EpiSrc src = tcepi::epi_src_global(p);
      if (p.epi == EPI_QKV) {
        // the row table and the RoPE tables in shared memory
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
      for (int j = 0; j < g.Tc; ++j) {
        const int rb = cid + j * NC;
        const uint32_t owner = (uint32_t)(j % C);
        const int slot = j / C;
        // the owner's global inputs of this tile, requested before its accumulator is ready
        float res[H];
        if (rank == owner) {
          load_residual<H>(p, rb, r, 0, res);
          src.gn = tcepi::load_next_gain(p, rb, r);
          src.has_gn = true;
        }
        if (!wait_or_abort(&sm.accf[acc], acc_phase, abort_flag)) {
          report_timeout(p, abort_flag, 4);
          ok = false;
          break;
        }
        tc::tc_fence_after();
        float vals[H];
#pragma unroll
        for (int n = 0; n < H; ++n) vals[n] = 0.f;
        const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(acc * kAcc * BN);
        const int nacc = g.sb1 - g.sb0 < kAcc ? g.sb1 - g.sb0 : kAcc;
        for (int a = 0; a < nacc; ++a) {  // accumulators in a fixed order; hi + lo per column
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
        const int got = csk::combine_partials<H>(vals, sum, sm.inbox, sm.inbox_full + k * kMaxSlots,
                                                 slot, rank, owner, C, r, abort_flag);
        if (got < 0) {
          report_timeout(p, abort_flag, 5);
          ok = false;
          break;
        }
        if (got > 0) finish<H>(p, rb, r, sum, 0, sm.swx, sm.rinv, res, src);
      }
      if (!ok) break;
      if (k + 1 < NP) {
        // arrive at grid barrier k once every epilogue thread's phase-k writes are done; the
        // count the barrier completes at is the next multiple of the grid size
        tc::named_bar_sync(1, 128);
        if (threadIdx.x == 64) {
          __threadfence();
          const unsigned long long t = atomicAdd(ch.bar + k, 1ull);
          const unsigned long long G = gridDim.x;
          sm.bar_target[k] = (t / G + 1) * G;
        }
      }
    }
    // an owner leaves only after its inboxes have been filled (bounded: a peer that gave up
    // sends nothing), so no st.async can land in a CTA that has exited
    if (C > 1 && threadIdx.x == 64)
      for (int k = 0; k < NP; ++k) {
        const Geo g = geo_of(ch.ph[k].p, cid, NC, C, rank, NK);
        for (int s = 0; s < g.owned; ++s) tc::mbar_wait(&sm.inbox_full[k * kMaxSlots + s], 0);
      }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) stamp_end(ch.stamp);
  if (C > 1) cluster_sync();
}

// cluster dims and PDL on one launch
template <int BN>
cudaError_t launch_csk(const CskChainArgs& ch, const CskPlan& q, bool any_qkv, cudaStream_t s) {
  const size_t smem = csk_smem_bytes<BN>(q, any_qkv);
  auto kern = k_tc_csk<BN>;
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
  return cudaLaunchKernelEx(&cfg, kern, ch, q);
}

// most clusters of C CTAs (each with `smem` bytes) resident at once, cached per configuration
template <int BN>
int active_clusters(int C, size_t smem) {
  static std::map<std::pair<int, size_t>, int> cache;
  auto key = std::make_pair(C, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  auto kern = k_tc_csk<BN>;
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

// The cluster shape is chosen from the matrix shapes alone (the same for every operand width),
// so a row's result does not depend on how many rows share the step: minimise the k-blocks the
// busiest CTA streams over all phases, sum_k ceil(RB_k / NC) * ceil(KS_k / C), over cluster
// sizes whose clusters can all be resident at once (a chain's grid barriers need every CTA
// resident).
bool csk_plan(const int* RB, const int* KS, int n, int BN, int num_sms, CskPlan* out) {
  if (n <= 0 || n > kMaxCskPhases || num_sms <= 0) return false;
  int rb_max = 0;
  for (int k = 0; k < n; ++k) {
    if (RB[k] <= 0 || KS[k] <= 0 || KS[k] % kCskBlocks) return false;
    rb_max = std::max(rb_max, RB[k]);
  }
  static const int kSizes[] = {1, 2, 3, 4, 6, 8};
  double best = 1e30;
  CskPlan bp{};
  for (int C : kSizes) {
    bool fits = C <= num_sms;
    for (int k = 0; k < n; ++k) fits = fits && C <= KS[k] / kCskBlocks;
    if (!fits) continue;
    // shape part of the plan, sized for the widest operand (N = 64)
    CskPlan q{};
    q.nk = kCskBlocks;
    q.C = C;
    q.NC = std::min(rb_max, num_sms / C);
    auto slots_of = [&](const CskPlan& pl) {
      int sl = 0;
      for (int k = 0; k < n; ++k) {
        const int tmax = (RB[k] + pl.NC - 1) / pl.NC;
        sl = std::max(sl, C > 1 ? (tmax + C - 1) / C : 0);
      }
      return sl;
    };
    q.slots = slots_of(q);
    if (q.slots > kMaxSlots) continue;
    q.stages = 2;  // the shallowest pipeline a launch may get
    if (csk_smem_bytes<64>(q, true) > (size_t)kSmemBudget) continue;
    const int fit = active_clusters<64>(C, csk_smem_bytes<64>(q, true));
    if (fit <= 0) continue;
    if (fit < q.NC) q.NC = fit;
    q.slots = slots_of(q);
    if (q.slots > kMaxSlots) continue;
    double cost = 0.01 * C;
    for (int k = 0; k < n; ++k) {
      const int SB = KS[k] / kCskBlocks;
      const int tmax = (RB[k] + q.NC - 1) / q.NC;
      cost += (double)tmax * ((SB + C - 1) / C) * kCskBlocks + (C > 1 ? 2.0 : 0.0);
    }
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

bool launch_tc_csk_chain(const CskChainPhase* phs, int n, int BN, int num_sms,
                         unsigned long long* bar, unsigned long long* stamp, cudaStream_t s) {
  if (n <= 0 || n > kMaxCskPhases || (n > 1 && !bar)) return false;
  CskChainArgs ch{};
  ch.n = n;
  ch.bar = bar;
  ch.stamp = stamp;
  std::vector<int> key{BN, num_sms};
  int RB[kMaxCskPhases], KS[kMaxCskPhases];
  bool any_qkv = false;
  for (int k = 0; k < n; ++k) {
    TcParams p = phs[k].p;
    if (!phs[k].tw || !phs[k].tx) return false;
    if (p.K % 64 || p.K <= 0 || p.n_act <= 0 || 2 * p.n_act > BN) return false;
    if (p.epi == EPI_SWIGLU && (p.F % 64 || p.M != 2 * p.F)) return false;
    p.RB = p.epi == EPI_SWIGLU ? p.F / 64 : (p.M + 127) / 128;
    p.KS = p.K / 64;
    p.NT = 1;
    ch.ph[k].tw = *phs[k].tw;
    ch.ph[k].tx = *phs[k].tx;
    ch.ph[k].p = p;
    RB[k] = p.RB;
    KS[k] = p.KS;
    key.push_back(p.RB);
    key.push_back(p.KS);
    any_qkv |= p.epi == EPI_QKV;
  }
  static std::map<std::vector<int>, CskPlan> plans;
  auto it = plans.find(key);
  CskPlan q;
  if (it != plans.end()) {
    q = it->second;
  } else {
    if (!csk_plan(RB, KS, n, BN, num_sms, &q)) return false;
    plans[key] = q;
  }
  cudaError_t rc;
  if (BN == 16) rc = launch_csk<16>(ch, q, any_qkv, s);
  else if (BN == 32) rc = launch_csk<32>(ch, q, any_qkv, s);
  else if (BN == 64) rc = launch_csk<64>(ch, q, any_qkv, s);
  else return false;
  return rc == cudaSuccess;
}

bool launch_tc_csk(const CUtensorMap& tw, const CUtensorMap& tx, TcParams p, int BN, int num_sms,
                   cudaStream_t s) {
  const CskChainPhase ph{&tw, &tx, p};
  return launch_tc_csk_chain(&ph, 1, BN, num_sms, nullptr, p.stamp, s);
}
