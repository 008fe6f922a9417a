// attn_prefill.cu -- segmented prefill attention on the 5th-generation tensor cores (sm_103a).
//
// Flash attention over each segment's own slab, causal inside the segment (query at position
// p attends keys [0, p]).  A unit is one q head of a block of 128 consecutive queries of one
// segment; its kv head is q head / G (grouped-query attention).  Per key block of 128:
//   S = Q K^T      tcgen05.mma, M = 128 queries, N = 128 keys, K = head_dim   (TMEM, 128 cols)
//   online softmax: two threads per query row (TMEM lane = query), each reading the whole
//                   row of S for the running max and sum, writing P for half the keys
//   O_b = P V      tcgen05.mma, M = 128 queries, N = head_dim, K = 128 keys   (TMEM)
// and each thread accumulates half of its row's O in registers with the running-max rescale.
// Q comes from a copy the RoPE kernel writes, scaled by 1/sqrt(head_dim) and split into a bf16
// high part and the bf16 rounding of the remainder; S accumulates both products, so the
// scores carry the rounding of K alone (as the decode attention's do); P enters the second
// product the same way, as bf16 hi and lo tiles.  K and V^T tiles come straight from the slab
// through the arena-wide TMA maps the decode attention uses: two K blocks in flight, one V
// block (its load overlaps the next block's Q K^T and softmax).  Keys past the segment's end are masked in S and their V^T
// columns zeroed in shared memory (the slab holds no values there).  One CTA per SM walks a
// list of units ordered by decreasing work.
#include "kernels.h"
#include "tc_common.cuh"

namespace {

constexpr int kBlk = 128;       // queries per unit and keys per key block
constexpr int kBox = 16384;     // one [128 rows][64 bf16] swizzled tile
constexpr int kRing = 2;        // K blocks in flight
constexpr int kCompute = 256;   // warps 2..9: two per TMEM lane quarter (halves of head_dim)
constexpr int kThreads = 64 + kCompute;

__device__ __forceinline__ void st_bf16(uint8_t* base, uint32_t off, uint16_t v) {
  *reinterpret_cast<uint16_t*>(base + off) = v;
}

__device__ __forceinline__ void flag_timeout(int* err, volatile int* abort_flag, int where) {
  *abort_flag = 1;
  if (atomicCAS(err, 0, CBT_DEV_TIMEOUT) == 0) err[1] = 300 + where;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort) {
  for (uint32_t i = 0; i < tc::kSpinLimit; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 1023) == 1023 && *abort) return false;
    if (i > 256) __nanosleep(32);
  }
  return false;
}

// key blocks a unit visits: up to the one holding its last query
__device__ __forceinline__ int key_blocks(const PrefillUnit& u) {
  return (u.q0 + u.nq - 1) / kBlk + 1;
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_prefill(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const PrefillUnit* __restrict__ units,
                   const long long* __restrict__ pagetab, int n_units, int q_lo_row, int layer,
                   int n_heads, int n_kv_heads, float* __restrict__ o, int* err) {
  constexpr int nKh = HD / 64;               // 64-dim boxes of Q and K
  constexpr uint32_t kQBytes = 2 * nKh * kBox;  // Q tile [hi, lo][128 queries][HD]
  constexpr uint32_t kKBytes = nKh * kBox;   // K tile [128 keys][HD]
  constexpr uint32_t kVBytes = 2 * HD * 128; // V^T tile: two [HD dims][64 keys] boxes
  constexpr int kVBox = HD * 128;            // bytes of one V^T box
  constexpr int kHalf = HD / 2;              // O columns per compute thread
  constexpr uint32_t kIdescS = tc::idesc_bf16(128, 128);
  constexpr uint32_t kIdescO = tc::idesc_bf16(128, HD);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;                          // 2 x nKh boxes: hi, lo
  uint8_t* sK = sQ + kQBytes;                  // [kRing] x nKh boxes
  uint8_t* sV = sK + kRing * kKBytes;          // 2 V^T boxes
  uint8_t* sP = sV + kVBytes;                  // [hi, lo][128 queries][128 keys] bf16: 4 boxes
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 4 * kBox);
  uint64_t *qfull = bars, *qempty = bars + 1;
  uint64_t *kfull = bars + 2, *kempty = bars + 2 + kRing;
  uint64_t *vfull = bars + 2 + 2 * kRing, *vempty = vfull + 1;
  uint64_t *s_full = vfull + 2, *s_free = s_full + 1, *p_full = s_full + 2;
  uint64_t *o_full = s_full + 3, *o_free = s_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_free + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = n_heads / n_kv_heads;
  if (tid == 0) {
    tc::mbar_init(qfull, 1);
    tc::mbar_init(qempty, 1);
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(&kfull[i], 1);
      tc::mbar_init(&kempty[i], 1);
    }
    tc::mbar_init(vfull, 1);
    tc::mbar_init(vempty, 1);
    tc::mbar_init(s_full, 1);
    tc::mbar_init(s_free, kCompute / 32);
    tc::mbar_init(p_full, kCompute / 32);
    tc::mbar_init(o_full, 1);
    tc::mbar_init(o_free, kCompute / 32);
    *abort_flag = 0;
    tc::mbar_fence_init();
    tc::tma_prefetch_desc(&tq);
    tc::tma_prefetch_desc(&tk);
    tc::tma_prefetch_desc(&tv);
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, 256);  // S: columns 0..127, O: 128..128+HD
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // Q, K and V come from the previous kernels
  pdl_launch();

  if (warp == 0) {
    if (lane == 0) {  // ---- TMA producer
      const uint64_t pol = tc::policy_evict_first();
      uint32_t un = 0, kn = 0, vn = 0;  // Q tiles, K blocks and V blocks issued
      for (int ui = blockIdx.x; ui < n_units; ui += gridDim.x) {
        const PrefillUnit u = units[ui];
        const int g = u.head / G;
        const QueryRow r{u.base, 0, u.cap};
        long long krow = kv_block(r, layer, 0, g, n_kv_heads, HD) / HD;
        long long vrow = kv_block(r, layer, 1, g, n_kv_heads, HD) / 64;
        if (!wait_or_abort(qempty, (un & 1) ^ 1, abort_flag)) {
          flag_timeout(err, abort_flag, 1);
          break;
        }
        tc::mbar_expect_tx(qfull, kQBytes);
#pragma unroll
        for (int h = 0; h < nKh; ++h) {
          tc::tma_load_2d(sQ + h * kBox, &tq, qfull, u.head * HD + h * 64, u.tok0, pol);
          tc::tma_load_2d(sQ + (nKh + h) * kBox, &tq, qfull, u.head * HD + h * 64,
                          q_lo_row + u.tok0, pol);
        }
        ++un;
        const int nkb = key_blocks(u);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (u.pages >= 0) {  // paged: the key block's own page (blocks never straddle pages)
            const QueryRow rp{pagetab[u.pages + kb * kBlk / u.cap], 0, u.cap};
            krow = kv_block(rp, layer, 0, g, n_kv_heads, HD) / HD;
            vrow = kv_block(rp, layer, 1, g, n_kv_heads, HD) / 64;
          }
          const int st = (int)(kn % kRing);
          if (!wait_or_abort(&kempty[st], ((kn / kRing) & 1) ^ 1, abort_flag)) {
            flag_timeout(err, abort_flag, 2);
            ok = false;
            break;
          }
          tc::mbar_expect_tx(&kfull[st], kKBytes);
#pragma unroll
          for (int h = 0; h < nKh; ++h)
            tc::tma_load_2d(sK + st * kKBytes + h * kBox, &tk, &kfull[st], h * 64,
                            (int)(krow + kb * kBlk), pol);
          ++kn;
          if (!wait_or_abort(vempty, (vn & 1) ^ 1, abort_flag)) {
            flag_timeout(err, abort_flag, 9);
            ok = false;
            break;
          }
          tc::mbar_expect_tx(vfull, kVBytes);
#pragma unroll
          for (int j = 0; j < 2; ++j)
            tc::tma_load_2d(sV + j * kVBox, &tv, vfull, 0,
                            (int)(vrow + (long long)(2 * kb + j) * HD), pol);
          ++vn;
        }
        if (!ok) break;
      }
      // never leave with copies in flight
      if (un > 0) tc::mbar_wait(qfull, (un - 1) & 1);
      for (uint32_t i = 0; i < (uint32_t)kRing && i < kn; ++i)
        tc::mbar_wait(&kfull[(kn - 1 - i) % kRing], ((kn - 1 - i) / kRing) & 1);
      if (vn > 0) tc::mbar_wait(vfull, (vn - 1) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---- MMA issuer
      uint32_t un = 0, kn = 0;
      bool ok = true;
      for (int ui = blockIdx.x; ui < n_units && ok; ui += gridDim.x, ++un) {
        const PrefillUnit u = units[ui];
        const int nkb = key_blocks(u);
        if (!wait_or_abort(qfull, un & 1, abort_flag)) {
          flag_timeout(err, abort_flag, 3);
          break;
        }
        for (int kb = 0; kb < nkb; ++kb, ++kn) {
          const int st = (int)(kn % kRing);
          // S = Q K^T once K has landed and the compute warps are done with the last S
          if (!wait_or_abort(&kfull[st], (kn / kRing) & 1, abort_flag) ||
              !wait_or_abort(s_free, (kn & 1) ^ 1, abort_flag)) {
            flag_timeout(err, abort_flag, 4);
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 2 * HD / 16; ++kk) {  // Q_hi K^T, then Q_lo K^T
            const int kd = kk % (HD / 16);
            const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sQ + (kk >> 2) * kBox)) + 2 * (kk & 3);
            const uint64_t bd =
                tc::sdesc_sw128(tc::smem_u32(sK + st * kKBytes + (kd >> 2) * kBox)) + 2 * (kd & 3);
            tc::mma_bf16(tmem, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
          }
          tc::mma_commit(s_full);
          tc::mma_commit(&kempty[st]);                // K of this block is free
          if (kb == nkb - 1) tc::mma_commit(qempty);  // Q is not read again by this unit
          // O_b = P V once P is written, V has landed and the compute warps have taken the
          // last O_b
          if (!wait_or_abort(p_full, kn & 1, abort_flag) ||
              !wait_or_abort(o_free, (kn & 1) ^ 1, abort_flag) ||
              !wait_or_abort(vfull, kn & 1, abort_flag)) {
            flag_timeout(err, abort_flag, 5);
            ok = false;
            break;
          }
          tc::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 2 * kBlk / 16; ++kk) {  // P_hi V, then P_lo V
            const int kd = kk % (kBlk / 16);
            const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sP + (kk >> 2) * kBox)) + 2 * (kk & 3);
            const uint64_t bd =
                tc::sdesc_sw128(tc::smem_u32(sV + (kd >> 2) * kVBox)) + 2 * (kd & 3);
            tc::mma_bf16(tmem + 128, ad, bd, kIdescO, kk > 0 ? 1u : 0u);
          }
          tc::mma_commit(o_full);
          tc::mma_commit(vempty);  // V of this block is free
        }
      }
    }
  } else {
    // ---- compute warps: query row = TMEM lane (32 * (warp % 4) + lane); `half` picks the
    // head_dim half this thread accumulates and the 64 keys of each block it writes P for
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    uint32_t kn = 0;
    bool ok = true;
    for (int ui = blockIdx.x; ui < n_units && ok; ui += gridDim.x) {
      const PrefillUnit u = units[ui];
      const int nkb = key_blocks(u);
      const int qpos = u.q0 + row;  // this row's position in the segment
      const bool live_row = row < u.nq;
      float m = -INFINITY, l = 0.f;
      float oacc[kHalf];
#pragma unroll
      for (int c = 0; c < kHalf; ++c) oacc[c] = 0.f;
      for (int kb = 0; kb < nkb; ++kb, ++kn) {
        if (!wait_or_abort(s_full, kn & 1, abort_flag)) {
          flag_timeout(err, abort_flag, 6);
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const int k0 = kb * kBlk;
        // pass 1: the row's maximum over its visible keys
        float mloc = -INFINITY;
#pragma unroll 1
        for (int c0 = 0; c0 < kBlk; c0 += 16) {
          uint32_t raw[16];
          tc::tmem_ld16(lane_base + c0, raw);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (live_row && k0 + c0 + j <= qpos) mloc = fmaxf(mloc, __uint_as_float(raw[j]));
        }
        const float mn = fmaxf(m, mloc);
        const float scl = (m == -INFINITY) ? 0.f : __expf(m - mn);
        // pass 2: P = exp(S - max) for the row, as bf16 hi/lo parts into the P tiles (this
        // thread's 64 keys, 16-byte stores of 8 keys), the row sum over all 128
        float psum = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < kBlk; c0 += 16) {
          uint32_t raw[16];
          tc::tmem_ld16(lane_base + c0, raw);
          tc::tmem_ld_wait();
          uint32_t hp[8], lp[8];
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const int key = k0 + c0 + j;
            const bool v0 = live_row && key <= qpos, v1 = live_row && key + 1 <= qpos;
            const float p0 = v0 ? __expf(__uint_as_float(raw[j]) - mn) : 0.f;
            const float p1 = v1 ? __expf(__uint_as_float(raw[j + 1]) - mn) : 0.f;
            psum += p0 + p1;
            const uint16_t h0 = f32_to_bf16(p0), h1 = f32_to_bf16(p1);
            const uint16_t l0 = f32_to_bf16(p0 - bf16_to_f32(h0));
            const uint16_t l1 = f32_to_bf16(p1 - bf16_to_f32(h1));
            hp[j >> 1] = (uint32_t)h0 | ((uint32_t)h1 << 16);
            lp[j >> 1] = (uint32_t)l0 | ((uint32_t)l1 << 16);
          }
          if ((c0 >> 6) == half) {
            const int chunk = (c0 & 63) >> 3;
#pragma unroll
            for (int v = 0; v < 2; ++v) {
              const uint32_t off = (uint32_t)(row * 128 + (((chunk + v) ^ (row & 7)) << 4));
              *reinterpret_cast<uint4*>(sP + half * kBox + off) =
                  make_uint4(hp[4 * v], hp[4 * v + 1], hp[4 * v + 2], hp[4 * v + 3]);
              *reinterpret_cast<uint4*>(sP + (2 + half) * kBox + off) =
                  make_uint4(lp[4 * v], lp[4 * v + 1], lp[4 * v + 2], lp[4 * v + 3]);
            }
          }
        }
        // keys past the segment's end: their V^T columns hold no values; zero this thread's
        // share of them (P is zero there) once the tile has landed
        if (k0 + kBlk > u.len) {
          if (!wait_or_abort(vfull, kn & 1, abort_flag)) {
            flag_timeout(err, abort_flag, 7);
            ok = false;
          } else {
            const int t = (warp - 2) * 32 + lane;  // 0..255: key (t & 127), dims half (t >> 7)
            const int key = t & 127;
            if (k0 + key >= u.len) {
              uint8_t* vt = sV + (key >> 6) * kVBox;
              for (int d = (t >> 7) * kHalf; d < (t >> 7) * kHalf + kHalf; ++d)
                st_bf16(vt, sw128_offset(d, key & 63, 0), 0);
            }
          }
        }
        m = mn;
        l = l * scl + psum;
        tc::fence_proxy_async_smem();  // P and the zeroed V columns are read by the MMA
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(s_free);
          tc::mbar_arrive(p_full);
        }
        if (!ok) break;
        // this block's P V into the running output
        if (!wait_or_abort(o_full, kn & 1, abort_flag)) {
          flag_timeout(err, abort_flag, 8);
          ok = false;
          break;
        }
        tc::tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < kHalf; c0 += 16) {
          uint32_t raw[16];
          tc::tmem_ld16(lane_base + 128 + half * kHalf + c0, raw);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) oacc[c0 + j] = oacc[c0 + j] * scl + __uint_as_float(raw[j]);
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(o_free);
      }
      if (!ok) break;
      if (live_row) {
        const float inv = 1.f / l;
        float* dst = o + (size_t)(u.tok0 + row) * (n_heads * HD) + u.head * HD + half * kHalf;
#pragma unroll
        for (int c = 0; c < kHalf; c += 4)
          *reinterpret_cast<float4*>(dst + c) =
              make_float4(oacc[c] * inv, oacc[c + 1] * inv, oacc[c + 2] * inv, oacc[c + 3] * inv);
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 256);
  }
}

template <int HD>
cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillUnit* units, const long long* pagetab, int n_units,
                           int q_lo_row, int layer, int n_heads, int n_kv_heads, float* o,
                           int* err, int grid, cudaStream_t s) {
  constexpr int nKh = HD / 64;
  constexpr size_t smem =
      1024 + 2 * nKh * kBox + kRing * nKh * kBox + 2 * HD * 128 + 4 * kBox + 256;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  cudaError_t rc =
      cudaFuncSetAttribute(k_attn_prefill<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (rc != cudaSuccess) return rc;
  return launch_pdl(k_attn_prefill<HD>, dim3(grid), dim3(kThreads), smem, s, tq, tk, tv, units,
                    pagetab, n_units, q_lo_row, layer, n_heads, n_kv_heads, o, err);
}

}  // namespace

bool launch_attn_prefill_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const PrefillUnit* units, const long long* pagetab, int n_units,
                            int q_lo_row, int layer, int n_heads, int n_kv_heads, int head_dim,
                            float* o, int* err, int num_sms, cudaStream_t s) {
  if (n_units <= 0) return true;
  if (n_heads % n_kv_heads) return false;
  const int grid = n_units < num_sms ? n_units : num_sms;
  cudaError_t rc;
  if (head_dim == 128)
    rc = launch_prefill<128>(tq, tk, tv, units, pagetab, n_units, q_lo_row, layer, n_heads,
                             n_kv_heads, o, err, grid, s);
  else if (head_dim == 64)
    rc = launch_prefill<64>(tq, tk, tv, units, pagetab, n_units, q_lo_row, layer, n_heads,
                            n_kv_heads, o, err, grid, s);
  else
    return false;
  return rc == cudaSuccess;
}
