// csk_common.cuh -- pieces shared by the cluster split-K decode projections (bf16 weights in
// gemm_csk.cu, 4-bit affine weights in gemm_q4.cu): cluster rank and distributed-shared-memory
// addressing, the cluster barrier, st.async into a peer's inbox, bounded mbarrier waits, the
// hand-off of a tile's partial sums to its owner and their reduce-scatter over the cluster.
#pragma once
#include "tc_common.cuh"

namespace csk {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t peer_addr(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// 16 bytes into a peer's shared memory; completes `bytes` on the peer's mbarrier
__device__ __forceinline__ void st_async_f4(uint32_t raddr, float a, float b, float c, float d,
                                            uint32_t rbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          raddr),
      "f"(a), "f"(b), "f"(c), "f"(d), "r"(rbar)
      : "memory");
}

// the same, suspending between polls instead of spinning
__device__ __forceinline__ bool wait_or_abort_sleep(uint64_t* bar, uint32_t parity,
                                                    volatile int* abort) {
  for (uint32_t i = 0; i < (1u << 23); ++i) {
    if (tc::mbar_try_wait_sleep(bar, parity, 1000)) return true;
    if ((i & 63) == 63 && *abort) return false;
  }
  return false;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              uint32_t limit = tc::kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 1023) == 1023 && *abort) return false;
    if (i > 256) __nanosleep(32);
  }
  return false;
}

// The C CTAs of a cluster that split one 128-row tile meet here.  Each holds its partial sums
// `vals` (row r of the tile, H operand rows).  A sender writes them into the owner's inbox
// (slot `slot`, sender index skipping the owner) and returns 0.  The owner waits for the C - 1
// partials and adds all C in rank order -- a fixed summation order -- into `sum`, returning 1;
// -1 if the wait timed out.
template <int H>
__device__ __forceinline__ int combine_partials(const float (&vals)[H], float (&sum)[H],
                                                float* inbox, uint64_t* inbox_full, int slot,
                                                uint32_t rank, uint32_t owner, int C, int r,
                                                volatile int* abort_flag,
                                                uint32_t limit = tc::kSpinLimit) {
  if (rank == owner) {
    if (C == 1) {
#pragma unroll
      for (int n = 0; n < H; ++n) sum[n] = vals[n];
      return 1;
    }
    if (!wait_or_abort(&inbox_full[slot], 0, abort_flag, limit)) return -1;
#pragma unroll
    for (int n = 0; n < H; ++n) sum[n] = 0.f;
    for (int src = 0; src < C; ++src) {
      if (src == (int)rank) {
#pragma unroll
        for (int n = 0; n < H; ++n) sum[n] += vals[n];
      } else {
        const int from = src - (src > (int)rank);  // sender slots skip the owner
        const float4* in = reinterpret_cast<const float4*>(
            inbox + ((size_t)(slot * (C - 1) + from) * 128 + r) * H);
#pragma unroll
        for (int c = 0; c < H / 4; ++c) {
          const float4 v = in[c];
          sum[4 * c] += v.x;
          sum[4 * c + 1] += v.y;
          sum[4 * c + 2] += v.z;
          sum[4 * c + 3] += v.w;
        }
      }
    }
    return 1;
  }
  const int from = (int)rank - ((int)rank > (int)owner);
  const uint32_t dst =
      peer_addr(tc::smem_u32(inbox + ((size_t)(slot * (C - 1) + from) * 128 + r) * H), owner);
  const uint32_t bar = peer_addr(tc::smem_u32(&inbox_full[slot]), owner);
#pragma unroll
  for (int c = 0; c < H / 4; ++c)
    st_async_f4(dst + 16 * c, vals[4 * c], vals[4 * c + 1], vals[4 * c + 2], vals[4 * c + 3], bar);
  return 0;
}

// Tokens [t0, t1) of a tile's H columns that rank `rank` of a C-CTA cluster finishes when the
// tile's partial sums are reduce-scattered over the cluster: chunks of a multiple of 4 columns
// (one st.async of 16 bytes each), possibly none for the last ranks.
__host__ __device__ __forceinline__ int rs_chunk(int H, int C) { return 4 * ((H + 4 * C - 1) / (4 * C)); }

// Reduce-scatter of one tile's partial sums over the C CTAs of a cluster: each CTA sends every
// peer that peer's columns of its `vals` (row r of the tile) into the peer's inbox for tile
// `tile` (sender index skipping the receiver), then waits for the C - 1 partials of its own
// columns [t0, t1) and adds all C in rank order -- the fixed order of a single owner -- into
// sum[t0 .. t1).  Returns 1 when it holds columns to finish, 0 when it has none, -1 if the wait
// timed out.  The inbox holds 128 x chunk floats per (tile, sender).
template <int H>
__device__ __forceinline__ int reduce_scatter(const float (&vals)[H], float (&sum)[H],
                                              float* inbox, uint64_t* inbox_full, int tile,
                                              uint32_t rank, int C, int r,
                                              volatile int* abort_flag,
                                              uint32_t limit = tc::kSpinLimit) {
  const int chunk = rs_chunk(H, C);
  for (int k = 0; k < C; ++k) {
    if (k == (int)rank) continue;
    const int k0 = min(H, k * chunk), k1 = min(H, k0 + chunk);
    if (k1 <= k0) continue;
    const int from = (int)rank - ((int)rank > k);
    const uint32_t dst = peer_addr(
        tc::smem_u32(inbox + ((size_t)(tile * (C - 1) + from) * 128 + r) * chunk), (uint32_t)k);
    const uint32_t bar = peer_addr(tc::smem_u32(&inbox_full[tile]), (uint32_t)k);
#pragma unroll
    for (int c = 0; c < H / 4; ++c)
      if (4 * c >= k0 && 4 * c < k1)
        st_async_f4(dst + 4 * (4 * c - k0), vals[4 * c], vals[4 * c + 1], vals[4 * c + 2],
                    vals[4 * c + 3], bar);
  }
  const int t0 = min(H, (int)rank * chunk), t1 = min(H, t0 + chunk);
  if (t1 <= t0) return 0;
  if (C == 1) {
#pragma unroll
    for (int n = 0; n < H; ++n) sum[n] = vals[n];
    return 1;
  }
#pragma unroll
  for (int n = 0; n < H; ++n) sum[n] = 0.f;
  if (!wait_or_abort(&inbox_full[tile], 0, abort_flag, limit)) return -1;
  for (int src = 0; src < C; ++src) {
    if (src == (int)rank) {
#pragma unroll
      for (int n = 0; n < H; ++n)
        if (n >= t0 && n < t1) sum[n] += vals[n];
    } else {
      const int from = src - (src > (int)rank);
      const float4* in = reinterpret_cast<const float4*>(
          inbox + ((size_t)(tile * (C - 1) + from) * 128 + r) * chunk);
#pragma unroll
      for (int c = 0; c < H / 4; ++c)
        if (4 * c >= t0 && 4 * c < t1) {
          const float4 v = in[(4 * c - t0) / 4];
          sum[4 * c] += v.x;
          sum[4 * c + 1] += v.y;
          sum[4 * c + 2] += v.z;
          sum[4 * c + 3] += v.w;
        }
    }
  }
  return 1;
}

}  // namespace csk
