// prefill_pair.cu -- paged prefill on the 5th-generation tensor cores (tcgen05 + TMEM) with
// two query heads of one KV head per work item, so that every K and V tile staged in shared
// memory feeds two score products and two P V products.
//
// What it computes ("Support Inkling-NVFP4 model", TensorRT-LLM PR #17062, sections
// "Architecture" and "Implementation"): for each new token and query head,
//   s_k = sm_scale * <q, K[k]> + rel[t, h, min(p - k, E - 1)]   (bias added before the softmax)
// over the visible keys (sliding window of W keys on local layers, full causal on global
// ones), then out = softmax(s) V.  New tokens are the last n_b positions of the history; K/V
// rows are read through the positional block table, page = k >> log2(P), and only keys below
// seq_len are read ("Inkling attn backend cleanup fake registry", TensorRT-LLM PR #17860).
//
// Work item: 128 consecutive new tokens of one sequence, one KV head and two of its query
// heads (one head when the group has an odd head left over).  One CTA per SM walks the items
// in order of decreasing causal length (static round-robin); the two heads of an item share
// their tokens, hence their visible keys, masks and K/V tiles.
//
// Tensor memory (512 columns for D = 128), bf16 bias: Q of head 0 (the A operand of
// S_0 = Q_0 K^T, D/2 columns), S of head 0 and 1 (64 fp32 columns each), P of head 0 and 1
// (softmax numerators, 32 columns of bf16 pairs each: the A operand of O += P V), O of head 0
// and 1 (D fp32 columns each).  Q of head 1 does not fit and sits in shared memory
// (S_1 = Q_1 K^T reads both operands from there).  With P apart from S, the next S of a head
// is computed as soon as the softmax has read the current one, so the softmax never waits
// for its own P V product.  fp32 bias (whose bias ring leaves no room for Q of head 1): Q of
// both heads in TMEM, P over the first columns of S, and the next S of a head after its P V
// product; Q tiles come into TMEM through one shared-memory staging tile loaded by TMA.
//
// Warp roles (384 threads):
//   warp 0   K and V producer: one TMA box per 64-key tile (or one per page segment when
//            pages are shorter than a tile), block-table entries held 32 at a time in lanes.
//   warps 1, 3  MMA issuers of head 0 and head 1, per tile: S_h(j+1) = Q_h K(j+1)^T (M 128,
//            N 64) as soon as the softmax has read S_h(j), then O_h += P_h(j) V(j) (M 128, N D,
//            A = P from TMEM) once P_h(j) is written.  Before its P V product each zeroes the V
//            rows of keys that no row of the item may see (window edges, sequence end,
//            unreadable pages).
//   warp 2   bias producer: per tile that reads any bucket below E - 1 and per head, up to four
//            3-D TMA boxes (32 tokens x COLS buckets) into the head's ring.
//   warps 4-7, 8-11  softmax of head 0 and head 1: thread r owns row r (TMEM lane r).  Per
//            item it loads its Q row (bf16 bias, head 0: into TMEM; head 1: into shared
//            memory, in the 128-byte-swizzled layout of an MMA operand; fp32 bias: from the
//            staging tile into TMEM), the next item's as soon as the current item's last P is
//            written, so that the next S overlaps the last P V product and the epilogue; per
//            tile it reads its 64 scores, adds the bias,
//            masks, keeps the running max and sum (O rescaled in TMEM only when the max grows
//            by more than 2^8), writes P into TMEM; at the end it normalises O and stores bf16.  Pairs of
//            scores go through packed two-lane fp32 FMA and add (the same rounding as scalar
//            FMA and add), maxima through three-input max.
// Every wait is bounded; after a timeout the CTA records INK_DEVERR_WAIT_TIMEOUT, stops
// issuing copies and MMAs, waits for the copies and MMAs already issued, and exits.
#include <type_traits>

#include "prefill_common.cuh"

namespace ink {

namespace {

constexpr int PP_THREADS = 384;
using namespace pf;

// Bias ring slots per head: two for the bf16 bias, one for fp32 (shared-memory budget).
template <bool BF16>
using PairBias = PBias<BF16, BF16 ? 2 : 1>;

constexpr int PP_Q1_SUB = PP_ROWS * 128;   // Q_1 in shared memory: blocks of 128 rows x 64 bf16

// ES (early S, the bf16-bias kernel): Q_0 in TMEM, Q_1 in shared memory, P_h apart from S_h,
// so that S_h(j+1) follows as soon as the softmax has read S_h(j).  Otherwise (the fp32-bias
// kernel, whose bias ring takes the shared memory Q_1 would need): Q_h in TMEM and P_h over
// the first 32 columns of S_h, so that S_h(j+1) follows once O_h += P_h(j) V(j) is done.
template <int D, bool ES>
struct PPShape {
  static constexpr int CB = D / 64;
  static constexpr int KV_SUB = TILE_KEYS * 128;
  static constexpr int KV_TILE = CB * KV_SUB;
  static constexpr int NK = D == 128 ? (ES ? 3 : 2) : 4;   // K ring (freed when both S products are done)
  static constexpr int NV = D == 128 ? 2 : 4;   // V ring (freed when both P V products are done)
  static constexpr uint32_t QC = D / 2;          // TMEM columns of one Q tile (bf16 pairs)
  static constexpr uint32_t TQ = 0;              // Q_h at TQ + h QC (ES: Q_0 only)
  static constexpr uint32_t TS = ES ? QC : 2 * QC;            // S_h at TS + 64 h
  static constexpr uint32_t TP = ES ? QC + 128 : 2 * QC;      // P_h at TP + PSTRIDE h
  static constexpr uint32_t PSTRIDE = ES ? 32 : 64;
  static constexpr uint32_t TO = ES ? QC + 192 : 2 * QC + 128;   // O_h at TO + D h
  static_assert(TO + 2 * D <= 512, "tensor memory budget");
  // ES: Q_1, an MMA operand.  Otherwise the staging tile through which TMA brings each Q_h
  // tile on its way into TMEM.
  static constexpr int Q1_BYTES = CB * PP_Q1_SUB;
};

template <int D, bool BF16>
struct PPSmem {
  using S = PPShape<D, BF16>;
  using B = PairBias<BF16>;
  static constexpr size_t kst = 0;
  static constexpr size_t vst = kst + (size_t)S::NK * S::KV_TILE;
  static constexpr size_t q1 = vst + (size_t)S::NV * S::KV_TILE;
  static constexpr size_t bias = q1 + (size_t)S::Q1_BYTES;
  static constexpr size_t bars = bias + (size_t)2 * B::NB * B::SLOT_BYTES;
  // k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], q_ready[2], s_full[2], s_empty[2],
  // p_full[2], pv_done[2], b_full[2 NB], b_empty[2 NB], drain[2], qs_full[2], qs_empty[2]
  static constexpr int NBAR = 2 * S::NK + 2 * S::NV + 10 + 4 * B::NB + 6;
  static constexpr size_t vbad = bars + NBAR * 8;
  static constexpr size_t misc = vbad + S::NV * 8;
  static constexpr size_t total = misc + 32;
  static constexpr size_t alloc = total + 1024;
};

// S_h = Q_h K^T of one 64-key tile, D / 16 K-steps (B = the K tile, K-major with the 128-byte
// swizzle; descriptors of later K-steps add the byte offset / 16 to the start-address field).
// A = Q_0 from TMEM (QS false, a0 its column) or Q_1 from shared memory (QS true, a0 the
// address of its first block).  Executed by a converged warp; one elected lane issues.
template <int D, bool QS>
__device__ __forceinline__ void pair_issue_s(uint32_t d, uint32_t a0, uint64_t b0, uint64_t* done) {
  constexpr uint32_t IDESC_S = umma_idesc_bf16(PP_ROWS, TILE_KEYS, false, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t bk = b0 + (uint64_t)((((kk >> 2) * TILE_KEYS * 128) + (kk & 3) * 32) >> 4);
    if constexpr (QS)
      umma_ss_warp(d, umma_desc_sw128(a0 + (uint32_t)((kk >> 2) * PP_Q1_SUB + (kk & 3) * 32), 16, 1024), bk,
                   IDESC_S, kk > 0 ? 1u : 0u);
    else
      umma_ts_warp(d, a0 + kk * 8, bk, IDESC_S, kk > 0 ? 1u : 0u);
  }
  umma_commit_warp(done);
}

// O_h += P_h V of one 64-key tile (A = P from TMEM, 8 columns of bf16 pairs per 16 keys; B = the
// V tile, MN-major), four K-steps of 16 keys; the first product of an item overwrites O_h.
template <int D>
__device__ __forceinline__ void pair_issue_pv(uint32_t d, uint32_t a0, uint64_t b0, uint32_t acc0, uint64_t* done) {
  constexpr uint32_t IDESC_PV = umma_idesc_bf16(PP_ROWS, D, false, true);
#pragma unroll
  for (int ks = 0; ks < TILE_KEYS / 16; ++ks)
    umma_ts_warp(d, a0 + ks * 8, b0 + (uint64_t)((ks * 16 * 128) >> 4), IDESC_PV, (acc0 || ks > 0) ? 1u : 0u);
  umma_commit_warp(done);
}

// 32 bytes of a row (p 32-byte aligned when IO32, else 16): one 256-bit load, or two 128-bit
// ones.  A thread owns a whole row, so each load of a warp touches 32 rows; the wider load
// halves the L1 requests of a row.
template <bool IO32>
__device__ __forceinline__ void ldg_row32(const uint4* p, uint32_t (&r)[8]) {
  if constexpr (IO32) {
    asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "l"(p));
  } else {
    const uint4 x = __ldg(p), y = __ldg(p + 1);
    r[0] = x.x; r[1] = x.y; r[2] = x.z; r[3] = x.w;
    r[4] = y.x; r[5] = y.y; r[6] = y.z; r[7] = y.w;
  }
}
template <bool IO32>
__device__ __forceinline__ void stg_row32(uint4* p, const uint32_t (&r)[8]) {
  if constexpr (IO32) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]),
                 "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
  } else {
    p[0] = make_uint4(r[0], r[1], r[2], r[3]);
    p[1] = make_uint4(r[4], r[5], r[6], r[7]);
  }
}

// Load this thread's Q row (rows past the item's last are zero) into TMEM (D / 2 columns).
// Every load of the row is issued before the first store.
template <int D, bool IO32>
__device__ __forceinline__ void pair_load_q(const uint4* qsrc, bool rv, uint32_t tm_q) {
  uint32_t qv[D / 64][32];
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    uint32_t (&w)[8] = *reinterpret_cast<uint32_t(*)[8]>(&qv[c >> 2][8 * (c & 3)]);
    if (rv) {
      ldg_row32<IO32>(qsrc + 2 * c, w);
    } else {
#pragma unroll
      for (int x = 0; x < 8; ++x) w[x] = 0u;
    }
  }
#pragma unroll
  for (int half = 0; half < D / 64; ++half) tmem_st32(tm_q + 32 * half, qv[half]);
  tmem_wait_st();
}

// Store this thread's Q row (rows past the item's last are zero) into shared memory as row r of
// an MMA operand tile: CB blocks of 128 rows x 128 bytes, 16-byte chunk c of a row at chunk
// position c ^ (r & 7) (the 128-byte swizzle).
template <int D, bool IO32>
__device__ __forceinline__ void pair_store_q_smem(const uint4* qsrc, bool rv, uint8_t* qtile, int r) {
  uint32_t x[D / 16][8];
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    if (rv) {
      ldg_row32<IO32>(qsrc + 2 * c, x[c]);
    } else {
#pragma unroll
      for (int y = 0; y < 8; ++y) x[c][y] = 0u;
    }
  }
#pragma unroll
  for (int c = 0; c < D / 8; ++c)
    *reinterpret_cast<uint4*>(qtile + (c >> 3) * PP_Q1_SUB + r * 128 + (((c & 7) ^ (r & 7)) << 4)) =
        make_uint4(x[c >> 1][4 * (c & 1)], x[c >> 1][4 * (c & 1) + 1], x[c >> 1][4 * (c & 1) + 2],
                   x[c >> 1][4 * (c & 1) + 3]);
}

// Multiply this thread's row of O (D fp32 TMEM columns) by f.
template <int D>
__device__ __forceinline__ void pair_rescale_o(uint32_t tm_o, float f) {
#pragma unroll 1
  for (int c2 = 0; c2 < D / 32; ++c2) {
    uint32_t ov[32];
    tmem_ld32(tm_o + c2 * 32, ov);
    tmem_wait_ld();
#pragma unroll
    for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * f);
    tmem_st32(tm_o + c2 * 32, ov);
  }
  tmem_wait_st();
}

// out row = O / l in bf16 (written only when `store`), 32 columns per TMEM load.
template <int D, bool IO32>
__device__ __forceinline__ void pair_store_o(uint32_t tm_o, float inv, uint4* orow, bool store) {
#pragma unroll 1
  for (int c2 = 0; c2 < D / 32; ++c2) {
    uint32_t ov[32];
    tmem_ld32(tm_o + c2 * 32, ov);
    tmem_wait_ld();
    if (store) {
#pragma unroll
      for (int q8 = 0; q8 < 2; ++q8) {
        uint32_t w[8];
#pragma unroll
        for (int x = 0; x < 8; ++x)
          w[x] = pack_bf16(__uint_as_float(ov[16 * q8 + 2 * x]) * inv, __uint_as_float(ov[16 * q8 + 2 * x + 1]) * inv);
        stg_row32<IO32>(orow + c2 * 4 + 2 * q8, w);
      }
    }
  }
}

// 32-bit shared-memory load, kept after the barrier wait that precedes it.
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// One row's bias in a ring slot.  Key c's bucket is element 63 - c counted from the element of
// key 63 (`at`).  load(hh) brings keys 32 hh .. 32 hh + 31 into registers (bf16: every key at
// once), each load of a batch issued together; pair(c) hands out (b[c], b[c + 1]) for even c.
template <bool BF16>
struct BiasRow {   // fp32: one 32-bit load per key (the 32 rows of a warp hit 32 banks)
  uint32_t k63;    // shared address of key 63's element
  float fv[32];    // keys 32 hh + i at fv[31 - i]
  __device__ __forceinline__ void at(const float* p) { k63 = smem_u32(p); }
  __device__ __forceinline__ void load(int hh) {
#pragma unroll
    for (int u = 0; u < 32; ++u) fv[u] = __uint_as_float(lds32(k63 + 4u * (uint32_t)(32 - 32 * hh + u)));
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int u = 0; u < 32; ++u) fv[u] = 0.f;
  }
  __device__ __forceinline__ uint64_t pair(int c) const {
    const int i = c & 31;
    return f2_pack(fv[31 - i], fv[30 - i]);
  }
};
template <>
struct BiasRow<true> {   // bf16: 33 aligned 32-bit loads per row, pairs funnel-shifted into place
  uint32_t w0;           // shared address of the word holding key 63's element
  uint32_t sh;           // 16 when that element is the high half of its word
  uint32_t wv[33];
  __device__ __forceinline__ void at(const __nv_bfloat16* p) {
    const uint32_t a = smem_u32(p);
    w0 = a & ~3u;
    sh = (a & 2u) << 3;
  }
  __device__ __forceinline__ void load(int) {
#pragma unroll
    for (int u = 0; u < 33; ++u) wv[u] = lds32(w0 + 4u * (uint32_t)u);
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int u = 0; u < 33; ++u) wv[u] = 0u;
  }
  __device__ __forceinline__ uint64_t pair(int c) const {
    const int q = 31 - (c >> 1);   // elements 2q, 2q + 1 from key 63's: keys c + 1, c
    const uint32_t v = __funnelshift_r(wv[q], wv[q + 1], sh);
    return f2_pack(__uint_as_float(v & 0xffff0000u), __uint_as_float(v << 16));
  }
};

template <int D, bool BF16, bool IO32, bool AHEAD2>
__global__ void __launch_bounds__(PP_THREADS, 1)
prefill_pair_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmK3, const __grid_constant__ CUtensorMap tmV3,
                    const __grid_constant__ CUtensorMap tmQ3, const __grid_constant__ CUtensorMap tmB,
                    const PrefillArgs a) {
  constexpr bool ES = BF16;
  // fp32 bias: the next item's facts (its bucket E - 1, its page check) are read at the end
  // of the current item along with its Q row.  (With the bf16 bias the kernel measured
  // slower that way, and reads them at the item's start.)
  constexpr bool CARRY = !BF16;
  using S = PPShape<D, ES>;
  using L_ = PPSmem<D, BF16>;
  using BS = PairBias<BF16>;
  using BT = typename BS::T;
  constexpr int NK = S::NK, NV = S::NV, NB = BS::NB;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L_::bars);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* q_ready = v_empty + NV;   // [2] Q_h of the item in place
  uint64_t* s_full = q_ready + 2;     // [2] S_h in TMEM (and every earlier product of the MMA warp done)
  uint64_t* s_empty = s_full + 2;     // [2] S_h read by the softmax
  uint64_t* p_full = s_empty + 2;     // [2] P_h in TMEM
  uint64_t* pv_done = p_full + 2;     // [2] O_h += P_h V done (P_h may be rewritten; O_h stable)
  uint64_t* b_full = pv_done + 2;     // [2 NB] head h's slot s at h NB + s
  uint64_t* b_empty = b_full + 2 * NB;
  uint64_t* drain = b_empty + 2 * NB;   // [2] one per MMA-issuing warp
  uint64_t* qs_full = drain + 2;        // [2] (fp32 bias) Q_h tile staged in shared memory
  uint64_t* qs_empty = qs_full + 2;     // [2] (fp32 bias) head h's warps have read it
  uint64_t* vbad = reinterpret_cast<uint64_t*>(smem + L_::vbad);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L_::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L_::misc + 4);
  int* qs_issued = reinterpret_cast<int*>(smem + L_::misc + 8);   // [2] staged tiles issued per head

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = 1 << a.log2_page;
  const int total_items = a.num_q_tiles * a.B * a.Hkv * ((a.G + 1) >> 1);

  if (tid == 0) {
    for (int x = 0; x < NK; ++x) {
      mbar_init(&k_full[x], 1);
      mbar_init(&k_empty[x], 2);   // one tcgen05.commit from each MMA warp
    }
    for (int x = 0; x < NV; ++x) {
      mbar_init(&v_full[x], 1);
      mbar_init(&v_empty[x], 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_ready[x], 4);
      mbar_init(&s_full[x], 1);
      mbar_init(&s_empty[x], 4);
      mbar_init(&p_full[x], 4);
      mbar_init(&pv_done[x], 1);
    }
    for (int x = 0; x < 2 * NB; ++x) {
      mbar_init(&b_full[x], 1);
      mbar_init(&b_empty[x], 4);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(&qs_full[x], 1);
      mbar_init(&qs_empty[x], 4);
      qs_issued[x] = 0;
    }
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "n"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // -------------------------------------------------------------- K and V producer
    if (lane == 0) {
      prefetch_tensormap(&tmK);
      prefetch_tensormap(&tmV);
      if (P >= TILE_KEYS) {
        prefetch_tensormap(&tmK3);
        prefetch_tensormap(&tmV3);
      }
    }
    // Two cursors walk the same sequence of tiles, K one tile ahead of V: the S product of a
    // tile is issued about a tile before its P V product, and a V slot that is still busy must
    // not hold back the next K.
    const int seg = P < TILE_KEYS ? P : TILE_KEYS;
    const int nseg = TILE_KEYS / seg;
    struct Cursor {
      int i, j;                           // item index, tile within it
      PPItem it;
      int chunk_b, chunk_base, chunk_val; // block-table entries chunk_base + lane
      int n;                              // fills issued
    };
    // the next tile of the walk (false when none is left)
    auto advance = [&](Cursor& c) -> bool {
      if (++c.j < c.it.ntile) return true;
      for (c.i += gridDim.x; c.i < total_items; c.i += gridDim.x)
        if (pp_item(a, c.i, c.it) && c.it.ntile > 0) {
          c.j = 0;
          return true;
        }
      return false;
    };
    // one K or V fill of the cursor's tile into the next ring slot (false after an abort)
    auto issue = [&](Cursor& c, bool is_k) -> bool {
      const PPItem& it = c.it;
      const int32_t* bt = a.block_table + (size_t)it.b * a.max_pages;
      const int last_idx = it.k_hi >> a.log2_page;   // never read the table past here
      const int k0 = (it.kt0 + c.j) * TILE_KEYS;
      // lane sg < nseg takes segment sg of the tile: seg keys on one page
      const int pfirst = k0 >> a.log2_page, plast = (k0 + TILE_KEYS - 1) >> a.log2_page;
      if (c.chunk_b != it.b || pfirst < c.chunk_base || plast >= c.chunk_base + 32) {
        c.chunk_b = it.b;
        c.chunk_base = pfirst;
        const int idx = c.chunk_base + lane;
        const int v = __ldg(bt + min(idx, last_idx));   // in bounds even past the last entry
        c.chunk_val = idx <= last_idx ? v : -1;
      }
      const int ks = k0 + lane * seg;
      const bool want = lane < nseg && ks <= it.k_hi && ks + seg - 1 >= it.lo_min;
      const int page = __shfl_sync(0xffffffffu, c.chunk_val, min(max((ks >> a.log2_page) - c.chunk_base, 0), 31));
      const bool bad_seg = want && (page < 0 || page >= a.num_pages);
      const bool load = want && !bad_seg;
      const uint32_t lmask = __ballot_sync(0xffffffffu, load);
      const uint32_t bmask = __ballot_sync(0xffffffffu, bad_seg);
      const int my_row = ((page * a.Hkv + it.kvh) << a.log2_page) + (ks & (P - 1));
      const uint32_t bytes = (uint32_t)__popc(lmask) * (uint32_t)(seg * D * 2);
      const int NR = is_k ? NK : NV;
      const int st = c.n % NR;
      uint64_t* full = is_k ? k_full : v_full;
      if (c.n >= NR && !pp_wait_warp(is_k ? &k_empty[st] : &v_empty[st], (uint32_t)((c.n / NR) - 1) & 1u, abort_flag, a))
        return false;
      if (!is_k && lane == 0) {   // keys whose page is outside the pool: the MMA warps zero their V rows
        uint64_t bad = 0;
#pragma unroll 1
        for (uint32_t mm = bmask; mm; mm &= mm - 1)
          bad |= seg == 64 ? ~0ull : (((1ull << seg) - 1) << ((__ffs(mm) - 1) * seg));
        vbad[st] = bad;
      }
      if (is_k && bmask && lane == 0) record_error(a.err, INK_DEVERR_PAGE_OUT_OF_RANGE);
      __syncwarp();
      mbar_arrive_expect_tx_warp(&full[st], bytes);
      uint8_t* ring = smem + (is_k ? L_::kst : L_::vst) + (size_t)st * S::KV_TILE;
#pragma unroll 1
      for (uint32_t mm = lmask; mm; mm &= mm - 1) {
        const int sg = __ffs(mm) - 1;
        const int row = __shfl_sync(0xffffffffu, my_row, sg);
        uint8_t* dst = ring + sg * seg * 128;
        if (seg == TILE_KEYS) {
          tma_load_3d_warp(dst, is_k ? &tmK3 : &tmV3, 0, row, 0, &full[st]);   // whole tile: one box
        } else {
#pragma unroll
          for (int cb = 0; cb < S::CB; ++cb)
            tma_load_2d_warp(dst + cb * S::KV_SUB, is_k ? &tmK : &tmV, cb * 64, row, &full[st]);
        }
      }
      ++c.n;
      return true;
    };
    Cursor ck, cv;
    ck.i = blockIdx.x - (int)gridDim.x;
    ck.j = 0;
    ck.it.ntile = 0;
    ck.chunk_b = -1;
    ck.chunk_base = 0;
    ck.chunk_val = -1;
    ck.n = 0;
    cv = ck;
    bool hk = advance(ck), hv = advance(cv);
    bool go = true;
    if (hk) {
      go = issue(ck, true);
      hk = advance(ck);
    }
    while (go && hv) {
      if (hk) {
        go = issue(ck, true);
        if (!go) break;
        hk = advance(ck);
      }
      go = issue(cv, false);
      if (!go) break;
      hv = advance(cv);
    }
    if (lane == 0) {
      pp_drain_ring(k_full, NK, ck.n, a.err);
      pp_drain_ring(v_full, NV, cv.n, a.err);
    }
  } else if (warp == 1 || warp == 3) {
    // -------------------------------------------------------------- MMA issuers
    // Warp 1 issues head 0's products, warp 3 head 1's, so that neither head waits behind the
    // other's barriers.  Per tile j: S_h(j+1) once the softmax has read S_h(j) (s_empty) and
    // K(j+1) has landed, then O_h += P_h(j) V(j) once P_h(j) is written (p_full).  K and V
    // slots are released by one commit from each warp (a warp whose head is absent from an
    // item commits without products).  Every phase of the barriers a warp waits on is waited
    // for in order.
    const int h = warp == 1 ? 0 : 1;
    int g = 0;                     // tiles walked
    int qc = 0;                    // items of head h
    int sn = 0;                    // S products issued for head h
    int pc = 0;                    // P V products issued for head h
    bool go = true;
    const uint32_t q1addr = smem_u32(smem + L_::q1);
    // S_h of K slot kslot, once S_h is free: read by the softmax (ES), or, with P_h over S_h,
    // read by the last P V product
    auto issue_s = [&](int kslot) -> bool {
      if (ES) {
        if (sn > 0 && !pp_wait_warp(&s_empty[h], (uint32_t)(sn - 1) & 1u, abort_flag, a)) return false;
      } else {
        if (pc > 0 && !pp_wait_warp(&pv_done[h], (uint32_t)(pc - 1) & 1u, abort_flag, a)) return false;
      }
      tc_fence_after();
      const uint64_t kd = umma_desc_sw128(smem_u32(smem + L_::kst + (size_t)kslot * S::KV_TILE), 16, 1024);
      if (ES && h == 1)
        pair_issue_s<D, true>(tmem + S::TS + 64u, q1addr, kd, &s_full[1]);
      else
        pair_issue_s<D, false>(tmem + S::TS + 64u * h, tmem + S::TQ + S::QC * h, kd, &s_full[h]);
      __syncwarp();
      ++sn;
      return true;
    };
    for (int i = blockIdx.x; i < total_items && go; i += gridDim.x) {
      PPItem it;
      if (!pp_item(a, i, it) || it.ntile == 0) continue;
      const bool mine = h < it.nh;
      // S of tile 0 once Q_h is in place
      go = pp_wait_warp(&k_full[g % NK], (uint32_t)(g / NK) & 1u, abort_flag, a);
      if (go && mine) {
        go = pp_wait_warp(&q_ready[h], (uint32_t)qc & 1u, abort_flag, a);
        ++qc;
        if (go) go = issue_s(g % NK);
      }
      if (!go) break;
      umma_commit_warp(&k_empty[g % NK]);
      __syncwarp();
      for (int j = 0; j < it.ntile && go; ++j) {
        const int gj = g + j;
        const int k0 = (it.kt0 + j) * TILE_KEYS;
        const int vs = gj % NV;
        // S of the next tile (ES: before this tile's P V product; otherwise after it)
        auto next_s = [&]() -> bool {
          if (j + 1 >= it.ntile) return true;
          if (!pp_wait_warp(&k_full[(gj + 1) % NK], (uint32_t)((gj + 1) / NK) & 1u, abort_flag, a)) return false;
          if (mine && !issue_s((gj + 1) % NK)) return false;
          umma_commit_warp(&k_empty[(gj + 1) % NK]);
          __syncwarp();
          return true;
        };
        if (ES) {
          go = next_s();
          if (!go) break;
        }
        go = pp_wait_warp(&v_full[vs], (uint32_t)(gj / NV) & 1u, abort_flag, a);
        if (!go) break;
        if (mine) {
          // zero the V rows of keys that no row of the item may read (both warps write the same
          // zeros to the same rows, each before its own product)
          const uint64_t vb = vbad[vs];
          if (k0 < it.lo_min || k0 + TILE_KEYS - 1 > it.k_hi || vb) {
            uint8_t* vt = smem + L_::vst + (size_t)vs * S::KV_TILE;
#pragma unroll 1
            for (int rr = lane; rr < TILE_KEYS; rr += 32) {
              const int k = k0 + rr;
              if (k < it.lo_min || k > it.k_hi || ((vb >> rr) & 1ull)) {
#pragma unroll 1
                for (int cb = 0; cb < S::CB; ++cb) {
                  uint4* row = reinterpret_cast<uint4*>(vt + cb * S::KV_SUB + rr * 128);
#pragma unroll
                  for (int c = 0; c < 8; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
                }
              }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
          }
          go = pp_wait_warp(&p_full[h], (uint32_t)pc & 1u, abort_flag, a);
          if (!go) break;
          tc_fence_after();
          pair_issue_pv<D>(tmem + S::TO + (uint32_t)(D * h), tmem + S::TP + S::PSTRIDE * h,
                           umma_desc_sw128(smem_u32(smem + L_::vst + (size_t)vs * S::KV_TILE), S::KV_SUB, 1024),
                           j > 0 ? 1u : 0u, &pv_done[h]);
          ++pc;
        }
        umma_commit_warp(&v_empty[vs]);
        __syncwarp();
        if (!ES) go = next_s();
      }
      g += it.ntile;
    }
    // every MMA this warp issued is complete before tensor memory is released
    umma_commit_warp(&drain[h]);
    __syncwarp();
    if (!mbar_wait_bounded(&drain[h], 0)) record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
  } else if (warp == 2) {
    // -------------------------------------------------------------- bias producer
    // For each tile that reads any bucket below E - 1, and each head of the item, the boxes of
    // the 32-row groups that do, into that head's next ring slot.  Out-of-range buckets and
    // tokens arrive as zeros and are never used.
    if (lane == 0) prefetch_tensormap(&tmB);
    int cnt[2] = {0, 0};
    bool go = true;
    for (int i = blockIdx.x; i < total_items && go; i += gridDim.x) {
      PPItem it;
      if (!pp_item(a, i, it) || it.ntile == 0) continue;
      for (int j = 0; j < it.ntile && go; ++j) {
        const int k0 = (it.kt0 + j) * TILE_KEYS;
        if (!pp_tile_needs_bias(it.pos0, k0, a.E)) continue;
        const int dmin0 = it.pos0 - (k0 + TILE_KEYS - 1);
        const uint32_t nm = __ballot_sync(0xffffffffu, lane < NGR && pp_group_needed(a, it, k0, lane));
        if constexpr (!BF16 && !AHEAD2) {
          // fp32: one ring slot per head, so the slot frees late; start the boxes towards L2 now
#pragma unroll 1
          for (int hs = 0; hs < it.nh; ++hs)
#pragma unroll 1
            for (uint32_t mm = nm; mm; mm &= mm - 1) {
              const int gr = __ffs(mm) - 1;
              tma_prefetch_l2_3d_warp(&tmB, pp_group_x<BS::ALIGN>(dmin0, gr), it.h0 + hs, it.t0 + BR * gr);
            }
        }
        if constexpr (!BF16 && AHEAD2) {
          // the same a tile earlier (window layers, whose short items leave the first tiles
          // of each item little time): the next tile's boxes at every tile, and this tile's
          // when no earlier tile sent them
          const bool sent = j > 0 && pp_tile_needs_bias(it.pos0, k0 - TILE_KEYS, a.E);
#pragma unroll 1
          for (int jj = sent ? 1 : 0; jj <= 1; ++jj) {
            const int kp = k0 + jj * TILE_KEYS;
            if (j + jj >= it.ntile || !pp_tile_needs_bias(it.pos0, kp, a.E)) continue;
            const int dp = it.pos0 - (kp + TILE_KEYS - 1);
            const uint32_t np = jj == 0 ? nm : __ballot_sync(0xffffffffu, lane < NGR && pp_group_needed(a, it, kp, lane));
#pragma unroll 1
            for (int hs = 0; hs < it.nh; ++hs)
#pragma unroll 1
              for (uint32_t mm = np; mm; mm &= mm - 1) {
                const int gr = __ffs(mm) - 1;
                tma_prefetch_l2_3d_warp(&tmB, pp_group_x<BS::ALIGN>(dp, gr), it.h0 + hs, it.t0 + BR * gr);
              }
          }
        }
        for (int hs = 0; hs < it.nh; ++hs) {
          const int slot = hs * NB + cnt[hs] % NB;
          if (cnt[hs] >= NB && !pp_wait_warp(&b_empty[slot], (uint32_t)((cnt[hs] / NB) - 1) & 1u, abort_flag, a)) {
            go = false;
            break;
          }
          BT* sb = reinterpret_cast<BT*>(smem + L_::bias + (size_t)slot * BS::SLOT_BYTES);
          mbar_arrive_expect_tx_warp(&b_full[slot], (uint32_t)__popc(nm) * (uint32_t)(BS::GROUP * sizeof(BT)));
#pragma unroll 1
          for (uint32_t mm = nm; mm; mm &= mm - 1) {
            const int gr = __ffs(mm) - 1;
            tma_load_3d_warp(sb + gr * BS::GROUP, &tmB, pp_group_x<BS::ALIGN>(dmin0, gr), it.h0 + hs, it.t0 + BR * gr,
                             &b_full[slot]);
          }
          ++cnt[hs];
        }
      }
    }
    if (lane == 0) {
      pp_drain_ring(b_full, NB, cnt[0], a.err);
      pp_drain_ring(b_full + NB, NB, cnt[1], a.err);
    }
  } else {
    // -------------------------------------------------------------- softmax warpgroups
    const int hs = (warp - 4) >> 2;   // head slot
    const int sw = (warp - 4) & 3;    // TMEM lane quarter
    const int r = sw * 32 + lane;
    const uint32_t tlane = tmem + ((uint32_t)(sw * 32) << 16);
    const uint32_t tm_q = tlane + S::TQ + S::QC * hs;
    const uint32_t tm_s = tlane + S::TS + 64u * hs;
    const uint32_t tm_p = tlane + S::TP + S::PSTRIDE * hs;
    const uint32_t tm_o = tlane + S::TO + (uint32_t)(D * hs);
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    int th = 0, bcnt = 0, pvw = 0;   // tiles, bias tiles and pv_done phases seen, of this head slot
    int q_in = -1;                   // item whose Q row went in at the end of the previous one
    PPItem nx;                       // item q_in, with its row's bucket E - 1 and page check
    float nx_clamp = 0.f;
    bool nx_bad = false;
    // fp32 bias: Q tiles reach TMEM through one shared-memory staging tile, by TMA (128
    // rows, all column blocks, the 128-byte swizzle), in the order (item, head 0), (item,
    // head 1), (next item, head 0), ...  The warps of the head that has read a tile issue the
    // next one, so one tile is in flight at a time: head 0's tile of the next item arrives
    // while the current item is still running.  Rows past an item's last are other tokens'
    // queries (or zeros past the tensor): their scores are masked and never stored.
    constexpr bool QSTAGE = !ES;
    int qsn = 0;   // staged tiles this head slot has taken
    auto stage_q = [&](const PPItem& qi, int hq) {   // one thread
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&qs_full[hq], (uint32_t)S::Q1_BYTES);
      tma_load_3d(smem + L_::q1, &tmQ3, 0, qi.t0, (qi.h0 + hq) * S::CB, &qs_full[hq]);
      atomicAdd(&qs_issued[hq], 1);
    };
    // This thread's Q row of item qi (index qidx) into TMEM (fp32 bias: from the staging tile;
    // bf16 bias: head 0 from global memory, rows past the item's last zero; head 1 into shared
    // memory), then q_ready.  False after an abort.
    auto load_q = [&](const PPItem& qi, int qidx) -> bool {
      if constexpr (QSTAGE) {
        if (hs == 0 && qsn == 0 && sw == 0 && lane == 0) stage_q(qi, 0);   // the first tile
        if (!pp_wait_warp(&qs_full[hs], (uint32_t)qsn & 1u, abort_flag, a)) return false;
        ++qsn;
        {
          const uint8_t* st = smem + L_::q1;
          uint32_t qv[D / 64][32];
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {
            const uint4 x = *reinterpret_cast<const uint4*>(st + (c >> 3) * PP_Q1_SUB + r * 128 + (((c & 7) ^ (r & 7)) << 4));
            qv[c >> 3][4 * (c & 7)] = x.x;
            qv[c >> 3][4 * (c & 7) + 1] = x.y;
            qv[c >> 3][4 * (c & 7) + 2] = x.z;
            qv[c >> 3][4 * (c & 7) + 3] = x.w;
          }
#pragma unroll
          for (int half = 0; half < D / 64; ++half) tmem_st32(tm_q + 32 * half, qv[half]);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&q_ready[hs]);
          mbar_arrive(&qs_empty[hs]);
        }
        if (sw == 0) {   // the next tile, once this head's four warps have read this one
          if (!pp_wait_warp(&qs_empty[hs], (uint32_t)(qsn - 1) & 1u, abort_flag, a)) return false;
          if (hs == 0 && qi.nh == 2) {
            if (lane == 0) stage_q(qi, 1);
          } else {
            PPItem nq;
            for (int ni = qidx + (int)gridDim.x; ni < total_items; ni += gridDim.x)
              if (pp_item(a, ni, nq) && nq.ntile > 0) {
                if (lane == 0) stage_q(nq, 0);
                break;
              }
          }
        }
        return true;
      }
      const bool qv = r < qi.rows;
      const uint4* qsrc = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q) +
                                                         ((size_t)(qi.t0 + (qv ? r : 0)) * a.Hq + qi.h0 + hs) * D);
      if (!ES || hs == 0) {
        pair_load_q<D, IO32>(qsrc, qv, tm_q);
        tc_fence_before();
      } else {
        pair_store_q_smem<D, IO32>(qsrc, qv, smem + L_::q1, r);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_ready[hs]);
      return true;
    };
    // Bucket E - 1 of this thread's row of item qi (rows past the item's last read its last
    // row: in bounds), and whether some page holding a key of the item lies outside the pool
    // (then per-tile masks of unreadable keys are built); the table entries are read four
    // per lane at a time.
    auto item_clamp = [&](const PPItem& qi) -> float {
      const bool qv = r < qi.rows;
      const BT* relrow =
          static_cast<const BT*>(a.rel) + ((size_t)(qi.t0 + (qv ? r : qi.rows - 1)) * a.Hq + qi.h0 + hs) * a.E;
      return qv ? to_float_b(__ldg(relrow + a.E - 1)) : 0.f;
    };
    auto item_pages_bad = [&](const PPItem& qi) -> bool {
      const int32_t* bq = a.block_table + (size_t)qi.b * a.max_pages;
      const int p0 = qi.lo_min >> a.log2_page, p1 = qi.k_hi >> a.log2_page;
      bool bad = false;
#pragma unroll 1
      for (int pi = p0 + lane; pi <= p1; pi += 128) {
        int pg[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) pg[u] = __ldg(bq + min(pi + 32 * u, p1));
#pragma unroll
        for (int u = 0; u < 4; ++u) bad |= pg[u] < 0 || pg[u] >= a.num_pages;
      }
      return __any_sync(0xffffffffu, bad);
    };
    bool go = true;
    for (int i = blockIdx.x; i < total_items && go; i += gridDim.x) {
      PPItem it;
      if (CARRY && q_in == i)
        it = nx;
      else if (!pp_item(a, i, it))
        continue;
      if (hs == 0 && sw == 0 && lane == 0 && it.t0 == __ldg(a.cu_q + it.b) && it.h0 == 0) {
        if (it.n > a.max_q_len) record_error(a.err, INK_DEVERR_QLEN_EXCEEDS_MAX);
        if (it.bad_len) record_error(a.err, INK_DEVERR_QLEN_EXCEEDS_KV);
        else if ((long long)it.L > ((long long)a.max_pages << a.log2_page))
          record_error(a.err, INK_DEVERR_PAGE_OUT_OF_RANGE);
      }
      if (hs >= it.nh) continue;
      const int h = it.h0 + hs;
      const bool rv = r < it.rows;
      if (it.ntile == 0) {  // nothing visible (inconsistent lengths or no readable key): zeros
        if (rv) {
          uint4* o = reinterpret_cast<uint4*>(out + ((size_t)(it.t0 + r) * a.Hq + h) * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      // ---- Q row and the item's facts, unless they came in at the end of the previous item
      // (the previous item's S products that read Q_h are complete: their s_full was seen)
      float clampv;
      bool item_bad = false;
      if constexpr (CARRY) {
        if (q_in == i) {
          clampv = nx_clamp;
          item_bad = nx_bad;
        } else {
          clampv = item_clamp(it);
          if (!load_q(it, i)) {
            go = false;
            break;
          }
          item_bad = item_pages_bad(it);
        }
      } else {
        if (q_in != i) load_q(it, i);
        clampv = item_clamp(it);
        const int p0 = it.lo_min >> a.log2_page, p1 = it.k_hi >> a.log2_page;
        const int32_t* bq = a.block_table + (size_t)it.b * a.max_pages;
#pragma unroll 1
        for (int pi = p0 + lane; pi <= p1; pi += 32) {
          const int page = __ldg(bq + pi);
          item_bad |= page < 0 || page >= a.num_pages;
        }
        item_bad = __any_sync(0xffffffffu, item_bad);
      }
      const int pr = it.pos0 + r;
      const int32_t* bt = a.block_table + (size_t)it.b * a.max_pages;
      const int seg = P < TILE_KEYS ? P : TILE_KEYS;
      auto tile_bad = [&](int k0) {
        uint64_t bad = 0;
#pragma unroll 1
        for (int sg = 0; sg < TILE_KEYS / seg; ++sg) {
          const int ks = k0 + sg * seg;
          if (ks > it.k_hi || ks + seg - 1 < it.lo_min) continue;
          const int page = __ldg(bt + min(ks >> a.log2_page, it.k_hi >> a.log2_page));
          if (page < 0 || page >= a.num_pages) bad |= (seg == 64 ? ~0ull : (((1ull << seg) - 1) << (sg * seg)));
        }
        return bad;
      };
      float m = -INFINITY, l = 0.f;
      const uint64_t scale2 = f2_pack(a.sm_scale, a.sm_scale);
      const uint64_t log2e2 = f2_pack(LOG2E, LOG2E);
      const uint64_t scalelog2e2 = f2_pack(a.sm_scale * LOG2E, a.sm_scale * LOG2E);
      for (int j = 0; j < it.ntile; ++j, ++th) {
        const int k0 = (it.kt0 + j) * TILE_KEYS;
        const bool needs = pp_tile_needs_bias(it.pos0, k0, a.E);
        const uint64_t bad = item_bad ? tile_bad(k0) : 0ull;
        // visible columns of this row: [kmin - k0, kmax - k0] less unreadable keys
        int kmin, kmax;
        pp_row_keys(a, it, pr, k0, kmin, kmax);
        uint64_t vis = 0;
        if (rv && kmax >= kmin) vis = (~0ull >> (TILE_KEYS - 1 - (kmax - k0))) & (~0ull << (kmin - k0));
        vis &= ~bad;
        // key c sits at distance dmin + 63 - c; columns c <= cc read bucket E - 1
        const int dmin = pr - (k0 + TILE_KEYS - 1);
        const int cc = dmin + TILE_KEYS - a.E;
        const int bslot_i = hs * NB + bcnt % NB;
        const BT* bslot = reinterpret_cast<const BT*>(smem + L_::bias + (size_t)bslot_i * BS::SLOT_BYTES);
        // The tile's bias comes into registers while its scores are still being computed
        BiasRow<BF16> brow;
        if (needs) {
          go = pp_wait_warp(&b_full[bslot_i], (uint32_t)(bcnt / NB) & 1u, abort_flag, a);
          if (!go) break;
          const int gr = r / BR;
          brow.at(bslot + gr * BS::GROUP + (r % BR) * BS::COLS + (dmin - pp_group_x<BS::ALIGN>(dmin - r, gr)));
          brow.load(0);
        } else {
          brow.at(bslot);
          brow.zero();
        }
        go = pp_wait_warp(&s_full[hs], (uint32_t)th & 1u, abort_flag, a);
        if (!go) break;
        tc_fence_after();
        uint32_t sr[64];
        {
          uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
          uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
          tmem_ld32(tm_s, lo);
          tmem_ld32(tm_s + 32, hi);
          tmem_wait_ld();
        }
        if (ES) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[hs]);   // the MMA warp may compute the next S here
        }
        // ES: O_h and P_h are free once the previous tile's P V product is done (waited once per
        // tile).  Otherwise S_h(j) was issued after that product completed, and s_full covers it.
        auto wait_pv = [&]() -> bool {
          if (!ES || pvw >= th) return true;
          if (!pp_wait_warp(&pv_done[hs], (uint32_t)pvw & 1u, abort_flag, a)) return false;
          ++pvw;
          tc_fence_after();
          return true;
        };
        float mxv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        const bool all_vis = vis == ~0ull;
        bool raw_clamp = false;   // sr holds the raw scores, every key reading bucket E - 1
        if (__all_sync(0xffffffffu, all_vis && cc < 0)) {
          // every key visible, every bucket from the tile's bias rows
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            if (!BF16 && c == 32) brow.load(1);
            float x, y;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), scale2, brow.pair(c)), x, y);
            sr[c] = __float_as_uint(x);
            sr[c + 1] = __float_as_uint(y);
            mxv[(c >> 1) & 3] = fmax3(mxv[(c >> 1) & 3], x, y);
          }
        } else if (__all_sync(0xffffffffu, all_vis && cc >= TILE_KEYS - 1)) {
          // every key visible at distance >= E - 1: s sm_scale + clampv for every key, so the max
          // is taken over the raw scores and the row's constant goes into the exponent's FMA
#pragma unroll
          for (int c = 0; c < 64; c += 2)
            mxv[(c >> 1) & 3] = fmax3(mxv[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
          raw_clamp = true;
        } else {
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            if (!BF16 && c == 32) {
              if (needs) brow.load(1);
            }
            float b0, b1;
            f2_unpack(brow.pair(c), b0, b1);
            b0 = c <= cc ? clampv : b0;
            b1 = c + 1 <= cc ? clampv : b1;
            float x, y;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), scale2, f2_pack(b0, b1)), x, y);
            x = ((vis >> c) & 1ull) ? x : -INFINITY;
            y = ((vis >> (c + 1)) & 1ull) ? y : -INFINITY;
            sr[c] = __float_as_uint(x);
            sr[c + 1] = __float_as_uint(y);
            mxv[(c >> 1) & 3] = fmax3(mxv[(c >> 1) & 3], x, y);
          }
        }
        float mx = fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3]));
        if (raw_clamp) mx = fmaf(mx, a.sm_scale, clampv);
        if (needs) {
          // every bias value this thread read is consumed (mx depends on all of them)
          asm volatile("" ::"f"(mx) : "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(&b_empty[bslot_i]);
          ++bcnt;
        }
        const float m_new = fmaxf(m, mx);
        if (j == 0) {
          m = m_new;
        } else {
          const bool mine = m_new > m + RESCALE_NAT;
          if (__any_sync(0xffffffffu, mine)) {
            // O_h must hold every earlier tile's P V product before it is rescaled
            go = wait_pv();
            if (!go) break;
            const float f = mine ? fast_exp2((m - m_new) * LOG2E) : 1.f;
            pair_rescale_o<D>(tm_o, f);
            l *= f;
            if (mine) m = m_new;
          }
        }
        // p = 2^(s log2(e) - m log2(e)); masked keys (s = -inf) give exactly 0.  With raw
        // scores: 2^(raw sm_scale log2(e) + clampv log2(e) - m log2(e)).
        const float mb = m == -INFINITY ? 0.f : m * LOG2E;
        const float addv = (raw_clamp ? clampv * LOG2E : 0.f) - mb;
        const uint64_t nmb2 = f2_pack(addv, addv);
        const uint64_t mul2 = raw_clamp ? scalelog2e2 : log2e2;
        uint32_t pk[32];
        uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};   // four packed partial sums (+0.0f pairs)
        auto exp_pairs = [&](int c0) {
#pragma unroll
          for (int c = c0; c < c0 + 16; ++c) {
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), mul2, nmb2), t0, t1);
            const float p0 = fast_exp2(t0);
            const float p1 = fast_exp2(t1);
            ls2[c & 3] = f2_add(ls2[c & 3], f2_pack(p0, p1));
            pk[c] = pack_bf16(p0, p1);
          }
        };
        // P row r in two halves, the first stored while the second is computed (P_h is free
        // once the previous tile's product has read it)
        exp_pairs(0);
        go = wait_pv();
        if (!go) break;
        tmem_st16(tm_p, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
        exp_pairs(16);
        tmem_st16(tm_p + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
        {
          float a0, a1, b0, b1, c0, c1, d0, d1;
          f2_unpack(ls2[0], a0, a1);
          f2_unpack(ls2[1], b0, b1);
          f2_unpack(ls2[2], c0, c1);
          f2_unpack(ls2[3], d0, d1);
          l += ((a0 + b0) + (c0 + d0)) + ((a1 + b1) + (c1 + d1));
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[hs]);
      }
      if (!go) break;
      // ---- epilogue: O_h / l -> bf16 -> out, once the item's last P V product is done
      auto epilogue = [&]() -> bool {
        if (!ES || pvw < th) {
          if (!pp_wait_warp(&pv_done[hs], (uint32_t)(th - 1) & 1u, abort_flag, a)) return false;
          pvw = th;
        }
        tc_fence_after();
        pair_store_o<D, IO32>(tm_o, l > 0.f ? 1.f / l : 0.f,
                              reinterpret_cast<uint4*>(out + ((size_t)(it.t0 + r) * a.Hq + h) * D), rv);
        tc_fence_before();
        return true;
      };
      // Head 1's staged tile is issued once head 0 has read its own: head 1 writes its output
      // first, while that tile is on its way.
      const bool epilogue_first = QSTAGE && hs == 1;
      if (epilogue_first && !epilogue()) {
        go = false;
        break;
      }
      // ---- the next item's Q row goes in now, so that its first S product overlaps this
      // item's last P V product and epilogue (S_h(last), the last reader of Q_h, is complete;
      // the next item's first P V product, which overwrites O_h, follows this epilogue)
      {
        int ni = i + (int)gridDim.x;
        if constexpr (CARRY) {
          nx = PPItem{};   // (written on every path: nothing of it lives through the tile loop)
          nx_clamp = 0.f;
          nx_bad = false;
          for (; ni < total_items; ni += gridDim.x)
            if (pp_item(a, ni, nx) && hs < nx.nh && nx.ntile > 0) break;
          if (ni < total_items) {
            nx_clamp = item_clamp(nx);
            go = load_q(nx, ni);
            nx_bad = item_pages_bad(nx);
            q_in = ni;
          }
        } else {
          PPItem nq;
          for (; ni < total_items; ni += gridDim.x)
            if (pp_item(a, ni, nq) && hs < nq.nh && nq.ntile > 0) break;
          if (ni < total_items) {
            go = load_q(nq, ni);
            q_in = ni;
          }
        }
      }
      if (!go) break;
      if (!epilogue_first && !epilogue()) {
        go = false;
        break;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // a staged Q tile still in flight (after an abort) lands before the CTA exits
  if (!ES && tid == 0) {
    for (int x = 0; x < 2; ++x) {
      const int n = qs_issued[x];
      if (n > 0 && !mbar_wait_bounded(&qs_full[x], (uint32_t)(n - 1) & 1u)) record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(512));
  }
}

int num_sms_pp() {
  int dev = 0;
  const int n = current_device_sms(&dev);
  return n > 0 ? n : 148;
}

template <int D, bool BF16, bool IO32, bool AHEAD2>
cudaError_t launch_pair_t(const PrefillMaps& m, const PrefillArgs& a, cudaStream_t stream) {
  constexpr size_t smem = PPSmem<D, BF16>::alloc;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  static std::atomic<unsigned long long> opted{0};
  cudaError_t e = smem_opt_in_once(prefill_pair_kernel<D, BF16, IO32, AHEAD2>, (int)smem, opted);
  if (e != cudaSuccess) return e;
  const long long items = (long long)a.num_q_tiles * a.B * a.Hkv * ((a.G + 1) / 2);
  const int grid = (int)std::min<long long>(items, num_sms_pp());
  prefill_pair_kernel<D, BF16, IO32, AHEAD2><<<grid, PP_THREADS, smem, stream>>>(m.k, m.v, m.k3, m.v3, m.q3,
                                                                                 m.bias, a);
  return cudaGetLastError();
}

// The fp32-bias kernel of window layers sends its bias boxes towards L2 a tile earlier (a
// kernel of its own, so that the global layers' code stays as it is).
template <int D, bool BF16>
cudaError_t launch_pair_io(const PrefillMaps& m, const PrefillArgs& a, cudaStream_t stream) {
  if constexpr (!BF16) {
    if (a.W > 0)
      return a.io32 ? launch_pair_t<D, false, true, true>(m, a, stream) : launch_pair_t<D, false, false, true>(m, a, stream);
  }
  return a.io32 ? launch_pair_t<D, BF16, true, false>(m, a, stream) : launch_pair_t<D, BF16, false, false>(m, a, stream);
}

}  // namespace

cudaError_t launch_prefill_pair(const PrefillMaps& m, const PrefillArgs& a, int head_dim, cudaStream_t stream) {
  if (a.bias_bf16)
    return head_dim == 128 ? launch_pair_io<128, true>(m, a, stream) : launch_pair_io<64, true>(m, a, stream);
  return head_dim == 128 ? launch_pair_io<128, false>(m, a, stream) : launch_pair_io<64, false>(m, a, stream);
}

}  // namespace ink
