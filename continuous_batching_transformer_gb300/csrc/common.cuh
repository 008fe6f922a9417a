// common.cuh -- small device helpers shared by the engine's kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "cbt.h"

#define CBT_HD __host__ __device__ __forceinline__
#define CBT_D __device__ __forceinline__

// bf16 bits <-> fp32.  Widening is exact; narrowing rounds to nearest even.
CBT_D float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
CBT_D float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
CBT_D float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }
CBT_D uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0x7FFFFFu) ? 0x40u : 0u));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// Where a decode row or a prefill token reads and writes its KV: the slab's element offset
// in the arena, the token's position and the slab's capacity (a multiple of 64).  A paged
// sequence keeps its positions in pages of `cap` positions (a multiple of 128), the page
// holding positions [s, s + cap) at element offset o; its rows carry base = o - s * head_dim,
// so the index helpers below take global positions unchanged (a page starts on a multiple of
// 64, so its V groups line up too).
// Slab layout (bf16): [layer][K|V][kv head] blocks of cap * head_dim elements; inside a K
// block key t, dim d sits at t*head_dim + d (one row per key); inside a V block the keys are
// grouped by 64 and transposed: key t, dim d sits at ((t/64)*head_dim + d)*64 + t%64, so a
// 64-key group is a [head_dim][64] tile.  Both attention contractions then read K-major
// tiles: Q.K^T with the keys' dims contiguous, P.V with the 64 keys of a dim contiguous.
struct QueryRow {
  long long base;  // element offset of the slab in the arena
  int pos;         // position of this token in its slab
  int cap;         // slab capacity (positions), a multiple of 64
};

CBT_HD long long kv_block(const QueryRow& r, int layer, int kv, int head, int n_kv_heads,
                          int head_dim) {
  return r.base + (((long long)layer * 2 + kv) * n_kv_heads + head) * (long long)r.cap * head_dim;
}
CBT_HD long long k_index(const QueryRow& r, int layer, int head, int key, int d, int n_kv_heads,
                         int head_dim) {
  return kv_block(r, layer, 0, head, n_kv_heads, head_dim) + (long long)key * head_dim + d;
}
CBT_HD long long v_index(const QueryRow& r, int layer, int head, int key, int d, int n_kv_heads,
                         int head_dim) {
  return kv_block(r, layer, 1, head, n_kv_heads, head_dim) +
         ((long long)(key >> 6) * head_dim + d) * 64 + (key & 63);
}

// Byte offset of bf16 element (row, col) in a K-major operand tile of 128-byte rows stored in
// the 128-byte swizzle (16-byte chunk index XOR row % 8), the layout TMA writes and tcgen05
// descriptors read; 64-column groups of the tile are `group_stride` bytes apart.
CBT_HD uint32_t sw128_offset(int row, int col, int group_stride) {
  const int g = col >> 6, c = col & 63;
  return (uint32_t)(g * group_stride + row * 128 + (((c >> 3) ^ (row & 7)) << 4) + (c & 7) * 2);
}

// One unit of decode attention: kv head g of row b over 128-key sub-chunks [s0, s1), whose
// keys sit in the slab (or page) at kbase (a QueryRow base: see above)
struct AttnItem {
  int b, g, s0, s1;
  long long kbase;
  int cap, p0;  // quantised KV: kbase is the byte offset of the slab or page, cap its layout
                // capacity, p0 its first position
  int n;        // the row's keys (its position + 1), so an item needs no second load
};

// Device error word: the first error wins (code, info).
CBT_D void set_device_error(int* err, int code, int info) {
  if (atomicCAS(err, 0, code) == 0) err[1] = info;
}

CBT_D float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

CBT_D float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Programmatic dependent launch: every kernel of a step is launched so that it may start
// while its predecessor drains; it must call pdl_wait() before touching memory the
// predecessor writes (or reads: buffers are reused), and calls pdl_launch() to let its own
// successor start early.  Without the launch attribute both are no-ops.
CBT_D void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
CBT_D void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Measurement stamps: a launch given a stamp slot s (2 words) records the earliest time one of
// its CTAs could start dependent work (min into s[0]) and the latest time one of its CTAs ended
// (max into s[1]), in globaltimer nanoseconds.  NULL: no stamps.
CBT_D unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
CBT_D void stamp_begin(unsigned long long* s) {
  if (s) atomicMin(s, globaltimer_ns());
}
CBT_D void stamp_end(unsigned long long* s) {
  if (s) atomicMax(s + 1, globaltimer_ns());
}

// Epilogues of a projection y = x W^T.
enum Epilogue : int {
  EPI_STORE = 0,   // out[n][m] = y
  EPI_ADD = 1,     // out[n][m] += y (residual)
  EPI_SWIGLU = 2,  // W = [gate; up] (2F rows): out[n][j] = silu(y_gate[j]) * y_up[j], j < F
  EPI_QKV = 3,     // W = [Wq; Wk; Wv]: RoPE, KV append and the attention's Q operand (decode)
  EPI_QKVQ = 4,    // EPI_QKV on a quantised-KV engine: the new K/V quantised into the slabs
};
