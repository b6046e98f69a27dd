// prefill_common.cuh -- device helpers of the head-pair prefill (prefill_pair.cu): work-item
// decoding, visible-key ranges, bias-box geometry, packed two-lane fp32 arithmetic and the
// bounded waits.
//
// What the kernels compute ("Support Inkling-NVFP4 model", TensorRT-LLM PR #17062, sections
// "Architecture" and "Implementation"): s_k = sm_scale <q, K[k]> + rel[t, h, min(p - k, E - 1)]
// over the visible keys, out = softmax(s) V; new tokens are the last n_b positions of the
// history, K/V rows come through the positional block table ("Inkling attn backend cleanup fake
// registry", TensorRT-LLM PR #17860).
#pragma once

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace ink {
namespace pf {
namespace {   // each kernel's translation unit has its own copy (internal linkage)

constexpr int PP_ROWS = PREFILL_ROWS;          // new tokens per item
constexpr int BR = PAIR_BIAS_ROWS;             // tokens per bias box
constexpr int NGR = PP_ROWS / BR;              // bias boxes per tile and head
constexpr float RESCALE_NAT = 5.545177444479562f;   // rescale O when a max grows by > 2^8


// Bias slot of one head and one tile: NGR boxes of BR rows; box gr holds buckets
// [x_gr, x_gr + COLS) of its rows, row i at +COLS i, x_gr = ALIGN floor((dmin0 + BR gr) / ALIGN)
// where dmin0 = pos0 - (k0 + 63) is row 0's smallest distance in the tile (x_gr is 16-byte
// aligned, as TMA wants).  Row r = BR gr + i finds the bucket of key k0 + c at
// offset (dmin_r - x_gr) + 63 - c, dmin_r - x_gr in [i, i + ALIGN - 1].  The row pitch plus the
// one-bucket skew between rows is odd (fp32: 101 words), so the 32 rows of a warp read 32
// different banks (bf16: at most two rows per bank).
template <bool BF16, int NSLOTS>
struct PBias {
  using T = typename std::conditional<BF16, __nv_bfloat16, float>::type;
  static constexpr int COLS = BF16 ? PAIR_BIAS_COLS_BF16 : PAIR_BIAS_COLS_F32;
  static constexpr int ALIGN = 16 / (int)sizeof(T);
  static constexpr int GROUP = BR * COLS;                       // elements per box
  static constexpr int SLOT_BYTES = NGR * GROUP * (int)sizeof(T);
  static constexpr int NB = NSLOTS;                             // ring slots per head
  static_assert(COLS >= TILE_KEYS + BR - 1 + ALIGN - 1, "bias box too narrow");
  static_assert((COLS * (int)sizeof(T)) % 16 == 0 && SLOT_BYTES % 1024 == 0, "TMA alignment");
};


struct PPItem {
  int b, kvh, h0, nh, t0, rows, n, L, pos0, lo_min, k_hi, kt0, ntile;
  bool bad_len;
};

// Item i: q-tile level (longest first), then sequence, KV head and head pair.
__device__ __forceinline__ bool pp_item(const PrefillArgs& a, int i, PPItem& it) {
  const int npair = (a.G + 1) >> 1;
  const int per_qt = a.B * a.Hkv * npair;
  const int qrev = i / per_qt;
  int r = i - qrev * per_qt;
  it.b = r / (a.Hkv * npair);
  r -= it.b * (a.Hkv * npair);
  it.kvh = r / npair;
  const int pair = r - it.kvh * npair;
  it.h0 = it.kvh * a.G + 2 * pair;
  it.nh = min(2, a.G - 2 * pair);
  const int qt = a.num_q_tiles - 1 - qrev;
  const int cu0 = __ldg(a.cu_q + it.b);
  it.n = __ldg(a.cu_q + it.b + 1) - cu0;
  if (qt * PP_ROWS >= it.n) return false;
  it.L = __ldg(a.seq_lens + it.b);
  it.t0 = cu0 + qt * PP_ROWS;
  it.rows = min(PP_ROWS, it.n - qt * PP_ROWS);
  it.bad_len = it.n > it.L;
  if (it.bad_len) {
    it.ntile = 0;
    return true;
  }
  it.pos0 = it.L - it.n + qt * PP_ROWS;
  const int p_max = it.pos0 + it.rows - 1;
  it.lo_min = a.W > 0 ? max(0, it.pos0 - a.W + 1) : 0;
  const long long cap = (long long)a.max_pages << a.log2_page;
  const int k_reach = (int)min((long long)it.L, cap) - 1;
  it.k_hi = min(p_max, k_reach);
  it.kt0 = it.lo_min / TILE_KEYS;
  it.ntile = it.k_hi >= it.lo_min ? it.k_hi / TILE_KEYS - it.kt0 + 1 : 0;
  return true;
}

// Visible keys of row position pr within tile k0 (kmin > kmax: none).
__device__ __forceinline__ void pp_row_keys(const PrefillArgs& a, const PPItem& it, int pr, int k0, int& kmin,
                                            int& kmax) {
  const int lor = a.W > 0 ? max(0, pr - a.W + 1) : 0;
  kmin = max(k0, lor);
  kmax = min(min(k0 + TILE_KEYS - 1, pr), it.k_hi);
}

// Every visible (row, key) pair of tile k0 is at distance >= E - 1: the tile reads bucket E - 1 only.
__device__ __forceinline__ bool pp_tile_needs_bias(int pos0, int k0, int E) {
  return pos0 - (k0 + TILE_KEYS - 1) < E - 1;
}

// Does bias box gr (rows BR gr .. BR gr + BR - 1) read any bucket below E - 1 in tile k0?
__device__ __forceinline__ bool pp_group_needed(const PrefillArgs& a, const PPItem& it, int k0, int gr) {
  const int r0 = BR * gr;
  if (r0 >= it.rows) return false;
  const int p_lo = it.pos0 + r0, p_hi = it.pos0 + min(r0 + BR - 1, it.rows - 1);
  const int lo_lo = a.W > 0 ? max(0, p_lo - a.W + 1) : 0;
  const bool any_key = p_hi >= k0 && lo_lo <= min(k0 + TILE_KEYS - 1, it.k_hi);
  const bool all_clamped = p_lo - (k0 + TILE_KEYS - 1) >= a.E - 1;
  return any_key && !all_clamped;
}

template <int ALIGN>
__device__ __forceinline__ int pp_group_x(int dmin0, int gr) {
  return (dmin0 + BR * gr) & ~(ALIGN - 1);
}

// Two fp32 lanes in one 64-bit register: packed FMA and add (sm_100-family), three-input max.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// The slow part of a bounded wait, out of line (one copy of the loop for every call site keeps
// the kernels' code small enough for the instruction caches).
__device__ __noinline__ bool pp_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* err, unsigned long long wait_ns) {
  if (*abort_flag) return false;
  if (mbar_wait_limit(bar, parity, wait_ns)) return true;
  record_error(err, INK_DEVERR_WAIT_TIMEOUT);
  *abort_flag = 1;
  return false;
}

// Bounded wait with the call's limit; gives up at once when another warp has timed out.
__device__ __forceinline__ bool pp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                       const PrefillArgs& a) {
  if (mbar_probe(bar, parity, a.wait_ns)) return true;
  return pp_wait_slow(bar, parity, abort_flag, a.err, a.wait_ns);
}

// The same, with every lane of the warp waiting and one answer for the whole warp.
__device__ __forceinline__ bool pp_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                            const PrefillArgs& a) {
  return __all_sync(0xffffffffu, pp_wait(bar, parity, abort_flag, a));
}

// After an abort: wait (with the full limit) until fill n of a ring slot has landed, for
// the last min(depth, issued) fills of the ring, so no copy is in flight at exit.
__device__ __forceinline__ void pp_drain_ring(uint64_t* full, int depth, int issued, uint32_t* err) {
#pragma unroll 1
  for (int n = max(0, issued - depth); n < issued; ++n)
    if (!mbar_wait_bounded(&full[n % depth], (uint32_t)(n / depth) & 1u)) record_error(err, INK_DEVERR_WAIT_TIMEOUT);
}

}  // namespace
}  // namespace pf
}  // namespace ink
