// prefill_tc.cu -- paged prefill on the 5th-generation tensor cores (tcgen05 + TMEM),
// with the relative-position bias and the window / causal mask fused into the score
// tile ("Support Inkling-NVFP4 model", TensorRT-LLM PR #17062, sections "Architecture"
// and "Implementation": the bias rel[t, h, distance] is added before the softmax; local
// layers see a 512-key window, global layers are full causal).  New tokens are the last
// n_b positions of the history and K/V are read through the positional block table
// ("Inkling attn backend cleanup fake registry", TensorRT-LLM PR #17860).
//
// Work item: 128 consecutive new tokens of one sequence and one query head.  One CTA
// per SM walks items in order of decreasing causal length (static round-robin, every other
// round reversed: sched_item).
// Warp roles (384 threads):
//   warps 0, 3  producers: TMA of the item's 128 query rows (q viewed as [tokens, Hq*D])
//           and of 64-key K tiles (warp 0) and V tiles (warp 3) into separate rings (K is
//           freed when S = Q K^T is done, V when O += P V is done; 128-byte swizzle);
//           block-table entries are held 32 at a time in lanes and looked up by shuffle.
//   warp 1  S issuer: S = Q K^T (M 128, N 64, fp32 in TMEM, double-buffered), issued by
//           one elected lane of the converged warp.
//   warp 2  bias: one 3-D TMA box (84 buckets x 16 tokens) per group of 16 rows that
//           reads any bucket below E - 1, into the slot of the softmax warpgroup that
//           owns the tile (4-byte cp.async when rows of rel are not 16-byte aligned);
//           keys at distance >= E - 1 use the row's bucket E - 1 instead.
//   warps 4-11  softmax, two warpgroups taking alternate key tiles: thread r of a
//           warpgroup owns row r (TMEM lane r): reads its 64 scores, adds bias, masks,
//           keeps the running max/sum and writes P (bf16) back to TMEM; then the
//           warpgroup's first warp issues O[wg] += P V (P from TMEM, V from shared
//           memory, fp32 O in TMEM), after zeroing the V rows of keys no row of the item
//           may see (edges of the window, the sequence end, unreadable pages), so any bit
//           pattern there is harmless.  O is rescaled in TMEM only when a row's max grows
//           by more than 2^8.  Epilogue: the two partial results are merged,
//           O / l -> bf16 -> out.
// Bias modes: fp32 or bf16 rel_logits (the slot loaded by TMA, as above), or the bias in
// low-rank form (BM_LOWRANK, 512 threads): there warp 2 issues tcgen05 MMAs of the item's r
// rows and projection rows into free TMEM columns, and warps 12-15 read the products out
// into fp16 slots; the softmax warpgroups are the same in every mode.
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace ink {

namespace {

constexpr int PT_ROWS = PREFILL_ROWS;
constexpr int PT_THREADS = 384;
// The low-rank mode adds a fourth warpgroup (warps 12-15, one per TMEM lane quarter) that
// reads the bias products out of TMEM, so it runs with 512 threads and rebalances registers
// with setmaxnreg: warps 0-3 and 12-15 give theirs to the softmax warpgroups.
constexpr int PT_THREADS_LR = 512;
constexpr int LR_REGS_PRODUCERS = 72, LR_REGS_SOFTMAX = 168, LR_REGS_BIAS = 104;
static_assert(LR_REGS_PRODUCERS + 2 * LR_REGS_SOFTMAX + LR_REGS_BIAS <= 4 * (65536 / PT_THREADS_LR),
              "the four warpgroups' registers must fit the 512-thread launch budget");
// Bias slot: 8 groups of 16 rows (tokens); group g holds buckets [x_g, x_g + COLS) of its
// rows, row i of it at +COLS i, x_g = ALIGN*floor((dmin0 + 16g)/ALIGN), where
// dmin0 = pos0 - (k0 + 63) is row 0's smallest distance in the tile (x_g is 16-byte
// aligned, as TMA wants).  Row r = 16g + i then finds the bucket of key k0 + c at offset
// boff + 63 - c with boff = (dmin0 mod ALIGN) + i, so 64 + 15 + ALIGN - 1 columns suffice.
// fp32: COLS 84 (the row pitch 85 is odd mod 32, so a row-per-thread read of one c hits
// each bank at most twice); bf16: COLS 88 (also at most two rows per bank word).
// Each softmax warpgroup owns PER_WG slots that it fills in turn; every slot then has one
// consumer taking its fills in order, so a parity wait never matches a phase two behind.
// Bias modes: BM_F32 and BM_BF16 load the slot from rel_logits by TMA; BM_LOWRANK builds an
// fp16 slot from tcgen05 products of r and the projection, one group at x_g = dmin0 + 16 g
// exactly (no TMA alignment to keep), so 64 + 15 = 79 buckets a row: 80 columns.  It keeps
// four slots, one per bias tile mod 4 (a tile's buckets are written as the products of
// three consecutive tiles arrive).
constexpr int BM_F32 = 0, BM_BF16 = 1, BM_LOWRANK = 2;

template <int BM>
struct BiasShape {
  using T = typename std::conditional<BM == BM_BF16, __nv_bfloat16,
                                      typename std::conditional<BM == BM_LOWRANK, __half, float>::type>::type;
  static constexpr int COLS = BM == BM_BF16 ? BIAS_BOX_COLS_BF16 : (BM == BM_LOWRANK ? 80 : BIAS_BOX_COLS);
  static constexpr int ALIGN = BM == BM_LOWRANK ? 1 : 16 / (int)sizeof(T);   // x_g is a multiple of ALIGN
  static constexpr int GROUP = BIAS_BOX_ROWS * COLS;          // elements per group
  static constexpr int NGROUP = PT_ROWS / BIAS_BOX_ROWS;      // groups per tile
  static constexpr int SLOT_BYTES = NGROUP * GROUP * (int)sizeof(T);
  static constexpr int PER_WG = 1;                            // slots per softmax warpgroup
  static constexpr int SLOTS = BM == BM_LOWRANK ? 4 : 2 * PER_WG;
  static_assert(COLS >= TILE_KEYS + BIAS_BOX_ROWS - 1 + ALIGN - 1, "bias box too narrow");
  static_assert((COLS * (int)sizeof(T)) % 16 == 0 && (GROUP * (int)sizeof(T)) % 128 == 0, "TMA alignment");
};

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

constexpr uint32_t TM_S = 0;     // S[2]: 64 fp32 columns each
constexpr uint32_t TM_P = 128;   // P[2]: 32 columns (64 bf16) each
constexpr uint32_t TM_BC = 192;  // low-rank mode: a bias chunk, 64 fp32 columns (128 rows x 64 buckets)
constexpr uint32_t TM_O = 256;   // O[2]: D fp32 columns each (one per softmax warpgroup)
constexpr uint32_t TM_COLS = 512;
constexpr float RESCALE_NAT = 5.545177444479562f;   // rescale O when a max grows by > 2^8

// Ring depths (D = 128): V gets two slots per softmax warpgroup (a V tile waits for the P V
// product two tiles back, so one slot each left the P V issue waiting for V); K gets three
// stages when the smaller bf16 bias slots leave room, two with the fp32 bias.
template <int D, int BM>
struct PtShape {
  static constexpr int CB = D / 64;
  static constexpr int Q_SUB = PT_ROWS * 128;
  static constexpr int Q_BYTES = CB * Q_SUB;
  static constexpr int KV_SUB = TILE_KEYS * 128;
  static constexpr int KV_TILE = CB * KV_SUB;   // one K or one V tile
  static constexpr int NK = D == 128 ? (BM == BM_BF16 ? 3 : 2) : 4;   // K ring: freed once S = Q K^T is done
  // V ring (even: slot g % NV serves warpgroup g % 2); the low-rank mode gives up two V
  // slots for its r tile and projection window
  static constexpr int NV = BM == BM_LOWRANK ? 2 : 4;
};

template <int D, int BM>
struct PtSmem {
  using S = PtShape<D, BM>;
  using BS = BiasShape<BM>;
  static constexpr size_t q = 0;
  static constexpr size_t kst = q + S::Q_BYTES;
  static constexpr size_t vst = kst + (size_t)S::NK * S::KV_TILE;
  static constexpr size_t bias = vst + (size_t)S::NV * S::KV_TILE;
  // low-rank mode: the item's r rows [128][64] and three chunks of projection rows
  // [64 buckets][64] (bf16, 128-byte swizzle as TMA lands them; MMA operands A and B)
  static constexpr size_t lr_r = bias + (size_t)BS::SLOTS * BS::SLOT_BYTES;
  static constexpr size_t lr_p = lr_r + (BM == BM_LOWRANK ? (size_t)PT_ROWS * LOWRANK_MAX_D * 2 : 0);
  static constexpr size_t bars = lr_p + (BM == BM_LOWRANK ? (size_t)3 * LOWRANK_CHUNK * LOWRANK_MAX_D * 2 : 0);
  // q_full, q_empty, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], s_full[2],
  // s_empty[2], o_done[2], o_free, b_full[NB], b_empty[NB], ml_full, ml_free,
  // pt_full[3], r_full, bc_full, bc_empty, drain[4] (one per MMA-issuing warp)
  static constexpr int NBAR = 2 + 2 * S::NK + 2 * S::NV + 2 + 2 + 2 + 1 + 2 * BS::SLOTS + 2 + 6 + 4;
  static constexpr size_t vbad = bars + NBAR * 8;
  static constexpr size_t ml1 = vbad + S::NV * 8;          // float2 [128]
  static constexpr size_t misc = ml1 + PT_ROWS * 8;
  static constexpr size_t total = misc + 32;
  static constexpr size_t alloc = total + 1024;
};

struct PItem {
  int b, h, kvh, t0, rows, n, L, pos0, lo_min, k_hi, kt0, ntile;
  bool bad_len;
};

__device__ __forceinline__ bool get_item(const PrefillArgs& a, int i_walk, PItem& it) {
  const int per_qt = a.B * a.Hq;
  const int i = sched_item(i_walk, a.num_q_tiles * per_qt);
  const int qrev = i / per_qt;
  const int r = i - qrev * per_qt;
  it.b = r / a.Hq;
  it.h = r - it.b * a.Hq;
  it.kvh = it.h / a.G;
  const int qt = a.num_q_tiles - 1 - qrev;
  const int cu0 = __ldg(a.cu_q + it.b);
  it.n = __ldg(a.cu_q + it.b + 1) - cu0;
  if (qt * PT_ROWS >= it.n) return false;
  it.L = __ldg(a.seq_lens + it.b);
  it.t0 = cu0 + qt * PT_ROWS;
  it.rows = min(PT_ROWS, it.n - qt * PT_ROWS);
  it.bad_len = it.n > it.L;
  if (it.bad_len) {
    it.ntile = 0;
    return true;
  }
  it.pos0 = it.L - it.n + qt * PT_ROWS;
  const int p_max = it.pos0 + it.rows - 1;
  it.lo_min = a.W > 0 ? max(0, it.pos0 - a.W + 1) : 0;
  const long long cap = (long long)a.max_pages << a.log2_page;
  const int k_reach = (int)min((long long)it.L, cap) - 1;
  it.k_hi = min(p_max, k_reach);
  it.kt0 = it.lo_min / TILE_KEYS;
  it.ntile = it.k_hi >= it.lo_min ? it.k_hi / TILE_KEYS - it.kt0 + 1 : 0;
  return true;
}

template <int ALIGN>
__device__ __forceinline__ int bias_group_x(int dmin0, int g) {
  return (dmin0 + BIAS_BOX_ROWS * g) & ~(ALIGN - 1);
}

// Visible keys of row position pr within tile k0 (kmin > kmax: none).
__device__ __forceinline__ void row_tile_keys(const PrefillArgs& a, const PItem& it, int pr, int k0, int& kmin,
                                              int& kmax) {
  const int lor = a.W > 0 ? max(0, pr - a.W + 1) : 0;
  kmin = max(k0, lor);
  kmax = min(min(k0 + TILE_KEYS - 1, pr), it.k_hi);
}

// Does bias group gr (rows 16 gr .. 16 gr + 15 of the item) read any bucket below E - 1 in
// tile k0?  The union of the group's visible ranges is [window start of its first row,
// its last row].
__device__ __forceinline__ bool bias_group_needed(const PrefillArgs& a, const PItem& it, int k0, int gr) {
  const int r0 = BIAS_BOX_ROWS * gr;
  if (r0 >= it.rows) return false;
  const int p_lo = it.pos0 + r0, p_hi = it.pos0 + min(r0 + BIAS_BOX_ROWS - 1, it.rows - 1);
  const int lo_lo = a.W > 0 ? max(0, p_lo - a.W + 1) : 0;
  const bool any_key = p_hi >= k0 && lo_lo <= min(k0 + TILE_KEYS - 1, it.k_hi);
  const bool all_clamped = p_lo - (k0 + TILE_KEYS - 1) >= a.E - 1;
  return any_key && !all_clamped;
}

// Every visible (row, key) pair of tile k0 lies at distance >= E - 1 (row 0 has the
// smallest position, key k0 + 63 the largest index): the whole tile reads bucket E - 1.
__device__ __forceinline__ bool tile_needs_bias(int pos0, int k0, int E) {
  return pos0 - (k0 + TILE_KEYS - 1) < E - 1;
}

// ---- low-rank bias: the chunk sequence of a CTA.  An item's tiles that need bias are its
// last ones (distances only shrink as k0 grows).  Tile t's bias window is the 192 buckets
// [x_0, x_0 + 192), x_0 = pos0 - (k0 + 63); the next tile's window starts 64 lower.  So the
// item's first bias tile needs three 64-bucket chunks [x_0 + 64 m, +64), m = 0..2, and every
// further tile one new chunk [x_0, x_0 + 64).
__device__ __forceinline__ int lr_first_bias_tile(const PrefillArgs& a, const PItem& it) {
  int j = 0;
  while (j < it.ntile && !tile_needs_bias(it.pos0, (it.kt0 + j) * TILE_KEYS, a.E)) ++j;
  return j;
}

struct LrCursor {
  PItem it;
  int i, j, m, jb;  // item, tile, chunk of the first bias tile (0..2), first bias tile
  int s;            // first bucket of the chunk
  bool first;       // first chunk of its item (the item's r rows are needed)
  bool valid;
};

__device__ __forceinline__ void lr_set(LrCursor& c) {
  const int x0 = c.it.pos0 - ((c.it.kt0 + c.j) * TILE_KEYS + TILE_KEYS - 1);
  c.s = c.j == c.jb ? x0 + LOWRANK_CHUNK * c.m : x0;
  c.first = c.j == c.jb && c.m == 0;
}

__device__ __forceinline__ void lr_seek(const PrefillArgs& a, int total_items, int i, LrCursor& c) {
  for (; i < total_items; i += gridDim.x) {
    if (!get_item(a, i, c.it) || c.it.ntile == 0) continue;
    const int jb = lr_first_bias_tile(a, c.it);
    if (jb >= c.it.ntile) continue;
    c.i = i;
    c.jb = jb;
    c.j = jb;
    c.m = 0;
    c.valid = true;
    lr_set(c);
    return;
  }
  c.valid = false;
}

__device__ __forceinline__ void lr_advance(const PrefillArgs& a, int total_items, LrCursor& c) {
  if (c.j == c.jb && c.m < 2) {
    ++c.m;
  } else if (c.j + 1 < c.it.ntile) {
    ++c.j;
    c.m = 0;
  } else {
    lr_seek(a, total_items, c.i + gridDim.x, c);
    return;
  }
  lr_set(c);
}

// A completed phase returns at once; otherwise give up at once if another warp of the
// CTA has timed out, else wait (bounded) and on a timeout record it and tell the others.
__device__ __forceinline__ bool wait_flag(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t* err,
                                          unsigned long long limit_ns) {
  if (mbar_probe(bar, parity, limit_ns)) return true;
  if (*abort_flag) return false;
  if (mbar_wait_limit(bar, parity, limit_ns)) return true;
  record_error(err, INK_DEVERR_WAIT_TIMEOUT);
  *abort_flag = 1;
  return false;
}

template <int D, int BM>
__global__ void __launch_bounds__(BM == BM_LOWRANK ? PT_THREADS_LR : PT_THREADS, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmK3, const __grid_constant__ CUtensorMap tmV3,
                  const __grid_constant__ CUtensorMap tmQ3, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmR, const __grid_constant__ CUtensorMap tmP,
                  const PrefillArgs a) {
  using S = PtShape<D, BM>;
  using L_ = PtSmem<D, BM>;
  using BS = BiasShape<BM>;
  using BT = typename BS::T;
  constexpr int NK = S::NK, NV = S::NV;
  constexpr uint32_t IDESC_S = umma_idesc_bf16(PT_ROWS, TILE_KEYS, false, false);
  constexpr uint32_t IDESC_PV = umma_idesc_bf16(PT_ROWS, D, false, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L_::bars);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;
  uint64_t* s_empty = s_full + 2;
  uint64_t* o_done = s_empty + 2;
  uint64_t* o_free = o_done + 2;
  uint64_t* b_full = o_free + 1;
  uint64_t* b_empty = b_full + BS::SLOTS;
  uint64_t* ml_full = b_empty + BS::SLOTS;
  uint64_t* ml_free = ml_full + 1;
  // low-rank mode: projection chunk n is in slot n % 3 (pt_full[3]); the item's r rows are in
  // (r_full); the bias product of chunk n is in TMEM (bc_full) / has been read out (bc_empty)
  uint64_t* pt_full = ml_free + 1;
  uint64_t* r_full = pt_full + 3;
  uint64_t* bc_full = r_full + 1;
  uint64_t* bc_empty = bc_full + 1;
  // every MMA a warp issued is complete before tensor memory is released: [0] the S issuer,
  // [1] the low-rank bias product issuer, [2 + wg] the P V issuer of softmax warpgroup wg
  uint64_t* drains = bc_empty + 1;
  float2* ml1 = reinterpret_cast<float2*>(smem + L_::ml1);
  uint64_t* vbad = reinterpret_cast<uint64_t*>(smem + L_::vbad);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L_::misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L_::misc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = 1 << a.log2_page;
  const int total_items = a.num_q_tiles * a.B * a.Hq;

  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int x = 0; x < NK; ++x) {
      mbar_init(&k_full[x], 1);
      mbar_init(&k_empty[x], 1);
    }
    for (int x = 0; x < NV; ++x) {
      mbar_init(&v_full[x], 1);
      mbar_init(&v_empty[x], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&s_empty[x], 4);
      mbar_init(&o_done[x], 1);
    }
    mbar_init(o_free, 4);
    mbar_init(ml_full, 4);
    mbar_init(ml_free, 4);
    for (int x = 0; x < 3; ++x) mbar_init(&pt_full[x], 1);
    mbar_init(r_full, 1);
    mbar_init(bc_full, 1);
    mbar_init(bc_empty, 4);
    for (int x = 0; x < 4; ++x) mbar_init(&drains[x], 1);
    for (int x = 0; x < BS::SLOTS; ++x) {
      mbar_init(&b_full[x], BM == BM_LOWRANK ? 128 : (a.bias_bulk ? 1 : 32));
      mbar_init(&b_empty[x], 4);
    }
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "n"(TM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 || warp == 3) {
    if constexpr (BM == BM_LOWRANK) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(LR_REGS_PRODUCERS));
    // -------------------------------------------------------------- producers (TMA)
    // warp 0 loads the query tile of each item and the K tiles, warp 3 the V tiles;
    // each walks the block table on its own (entries held 32 at a time in lanes).
    const bool is_k = warp == 0;
    const int NR = is_k ? NK : NV;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    const CUtensorMap* tm = is_k ? &tmK : &tmV;
    const CUtensorMap* tm3 = is_k ? &tmK3 : &tmV3;   // whole tiles, P >= 64
    uint8_t* ring = smem + (is_k ? L_::kst : L_::vst);
    if (lane == 0) {
      prefetch_tensormap(tm);
      if (P >= TILE_KEYS) prefetch_tensormap(tm3);
      if (is_k) prefetch_tensormap(&tmQ3);
    }
    int icount = 0, g = 0, q_issued = 0;   // items, ring fills issued (g), Q tiles issued
    int chunk_b = -1, chunk_base = 0, chunk_val = -1;
    const int seg = P < TILE_KEYS ? P : TILE_KEYS;
    const int nseg = TILE_KEYS / seg;
    bool go = true;
    for (int i = blockIdx.x; i < total_items && go; i += gridDim.x) {
      PItem it;
      if (!get_item(a, i, it) || it.ntile == 0) continue;
      if (is_k) {
        bool ok = true;
        if (lane == 0) {
          ok = icount == 0 || wait_flag(q_empty, (uint32_t)(icount - 1) & 1u, abort_flag, a.err, a.wait_ns);
          if (ok) {
            mbar_arrive_expect_tx(q_full, (uint32_t)S::Q_BYTES);
            tma_load_3d(smem + L_::q, &tmQ3, 0, it.t0, it.h * S::CB, q_full);   // 128 rows x all column blocks
          }
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
        ++q_issued;
      }
      const int32_t* bt = a.block_table + (size_t)it.b * a.max_pages;
      const int last_idx = it.k_hi >> a.log2_page;  // never read the table past here
      for (int j = 0; j < it.ntile; ++j, ++g) {
        const int st = g % NR;
        bool ok = true;
        if (lane == 0 && g >= NR) ok = wait_flag(&empty[st], (uint32_t)((g / NR) - 1) & 1u, abort_flag, a.err, a.wait_ns);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) {
          go = false;
          break;
        }
        const int k0 = (it.kt0 + j) * TILE_KEYS;
        // lane sg < nseg takes segment sg of the tile: seg keys on one page
        const int pfirst = k0 >> a.log2_page, plast = (k0 + TILE_KEYS - 1) >> a.log2_page;
        if (chunk_b != it.b || pfirst < chunk_base || plast >= chunk_base + 32) {
          chunk_b = it.b;
          chunk_base = pfirst;
          const int idx = chunk_base + lane;
          const int v = __ldg(bt + min(idx, last_idx));   // in bounds even past the last entry
          chunk_val = idx <= last_idx ? v : -1;
        }
        const int ks = k0 + lane * seg;
        const bool want = lane < nseg && ks <= it.k_hi && ks + seg - 1 >= it.lo_min;
        const int page = __shfl_sync(0xffffffffu, chunk_val, min(max((ks >> a.log2_page) - chunk_base, 0), 31));
        const bool bad_seg = want && (page < 0 || page >= a.num_pages);
        const bool load = want && !bad_seg;
        const uint32_t lmask = __ballot_sync(0xffffffffu, load);
        const uint32_t bmask = __ballot_sync(0xffffffffu, bad_seg);
        if (bmask) {  // error path: record it, and tell the MMA warp which V rows to zero
          if (lane == 0) {
            if (is_k) record_error(a.err, INK_DEVERR_PAGE_OUT_OF_RANGE);
            uint64_t bad = 0;
#pragma unroll 1
            for (uint32_t mm = bmask; mm; mm &= mm - 1)
              bad |= seg == 64 ? ~0ull : (((1ull << seg) - 1) << ((__ffs(mm) - 1) * seg));
            if (!is_k) vbad[st] = bad;
          }
        } else if (!is_k && lane == 0) {
          vbad[st] = 0;
        }
        __syncwarp();
        mbar_arrive_expect_tx_warp(&full[st], (uint32_t)__popc(lmask) * (uint32_t)(seg * D * 2));
        const int my_row = ((page * a.Hkv + it.kvh) << a.log2_page) + (ks & (P - 1));
#pragma unroll 1
        for (uint32_t mm = lmask; mm; mm &= mm - 1) {
          const int sg = __ffs(mm) - 1;
          const int row = __shfl_sync(0xffffffffu, my_row, sg);
          uint8_t* dst = ring + (size_t)st * S::KV_TILE + sg * seg * 128;
          if (seg == TILE_KEYS) {
            tma_load_3d_warp(dst, tm3, 0, row, 0, &full[st]);   // whole tile: one box
          } else {
#pragma unroll
            for (int cb = 0; cb < S::CB; ++cb) tma_load_2d_warp(dst + cb * S::KV_SUB, tm, cb * 64, row, &full[st]);
          }
        }
      }
      ++icount;
    }
    // the copies issued last into each ring slot (and the last Q tile) may still be landing
    // after an abort: wait for them (2 s each) so none is in flight when the CTA exits
    if (lane == 0) {
#pragma unroll 1
      for (int n = max(0, g - NR); n < g; ++n)
        if (!mbar_wait_bounded(&full[n % NR], (uint32_t)(n / NR) & 1u)) record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
      if (q_issued > 0 && !mbar_wait_bounded(q_full, (uint32_t)(q_issued - 1) & 1u))
        record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
    }
  } else if (warp == 1) {
    if constexpr (BM == BM_LOWRANK) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(LR_REGS_PRODUCERS));
    // -------------------------------------------------------------- S issuer
    // S(g) = Q K(g)^T into S buffer g % 2 as soon as K(g) is in and the warpgroup that
    // owns tile g - 2 has read S(g - 2) out of TMEM, which it does first thing, so each
    // warpgroup finds its next S computed when it finishes a P.  Q is freed after the
    // item's last S.
    int icount = 0, g = 0;
    bool go = true;
    for (int i = blockIdx.x; i < total_items && go; i += gridDim.x) {
      PItem it;
      if (!get_item(a, i, it) || it.ntile == 0) continue;
      go = __all_sync(0xffffffffu, wait_flag(q_full, (uint32_t)icount & 1u, abort_flag, a.err, a.wait_ns));
#pragma unroll 1
      for (int j = 0; j < it.ntile && go; ++j, ++g) {
        const int ks_ = g % NK;
        go = __all_sync(0xffffffffu, wait_flag(&k_full[ks_], (uint32_t)(g / NK) & 1u, abort_flag, a.err, a.wait_ns));
        if (go && g >= 2)
          go = __all_sync(0xffffffffu,
                          wait_flag(&s_empty[g & 1], (uint32_t)((g >> 1) - 1) & 1u, abort_flag, a.err, a.wait_ns));
        if (!go) break;   // after an abort no MMA is issued
        tc_fence_after();
        const uint32_t qbase = smem_u32(smem + L_::q);
        const uint32_t kbase = smem_u32(smem + L_::kst + (size_t)ks_ * S::KV_TILE);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = umma_desc_sw128(qbase + (kk >> 2) * S::Q_SUB + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = umma_desc_sw128(kbase + (kk >> 2) * S::KV_SUB + (kk & 3) * 32, 16, 1024);
          umma_ss_warp(tmem + TM_S + (g & 1) * 64, ad, bd, IDESC_S, kk > 0 ? 1u : 0u);
        }
        umma_commit_warp(&s_full[g & 1]);
        umma_commit_warp(&k_empty[ks_]);
        if (j == it.ntile - 1) umma_commit_warp(q_empty);   // the item's last S: Q may be replaced
        __syncwarp();
      }
      ++icount;
    }
    umma_commit_warp(&drains[0]);
    __syncwarp();
    if (!mbar_wait_bounded(&drains[0], 0)) record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
  } else if (warp == 2) {
    if constexpr (BM == BM_LOWRANK) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(LR_REGS_PRODUCERS));
    // -------------------------------------------------------------- bias loader
    // Fast path (rows of rel 16-byte aligned): one 3-D TMA box per group of 16 tokens
    // (84 buckets x 16 rows, laid out so the softmax reads see at most 2-way bank
    // conflicts); out-of-range buckets arrive as zeros and are never used.  Otherwise the
    // warp copies the visible buckets with 4-byte cp.async into the same layout.
    // Buckets at distance >= E - 1 are never read: the softmax uses the row's bucket
    // E - 1 for those keys.
    // Warpgroup w's tiles (g % 2 == w) fill its PER_WG slots in turn: each slot has one
    // consumer that takes its fills in order, so a parity wait never sees a phase two
    // behind.  (V slots follow the same rule: NV is even.)
    if (lane == 0 && a.bias_bulk) prefetch_tensormap(&tmB);
    if constexpr (BM == BM_LOWRANK) {
      // ------------------------------------------------------------ low-rank bias products
      // For each chunk n of the CTA's chunk sequence: bias[row, bucket] for the item's 128
      // rows and the chunk's 64 buckets, one tcgen05 MMA (M 128, N 64, K 64: four K-steps)
      // into TMEM columns TM_BC, A = the item's r rows, B = the chunk's projection rows
      // (both K-major, 128-byte swizzle).  Projection chunks are loaded two ahead into three
      // slots; the single TMEM chunk is reused once the bias warps have read it out.
      if (lane == 0) {
        prefetch_tensormap(&tmR);
        prefetch_tensormap(&tmP);
      }
      constexpr uint32_t PT_BYTES = LOWRANK_CHUNK * LOWRANK_MAX_D * 2;
      LrCursor cur, pf;
      lr_seek(a, total_items, blockIdx.x, cur);
      pf = cur;
      int issued = 0;
#pragma unroll 1
      for (int q = 0; q < 2 && pf.valid; ++q, ++issued) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&pt_full[q], PT_BYTES);
          tma_load_2d(smem + L_::lr_p + (size_t)q * PT_BYTES, &tmP, 0, pf.s, &pt_full[q]);
        }
        lr_advance(a, total_items, pf);
      }
      int n = 0, ritems = 0;
      bool r_pending = false;
      while (cur.valid) {
        bool ok = true;
        // the product of chunk n - 1 has been read out of TMEM: its MMA is complete, so
        // TMEM, the r rows and chunk slot (n - 1) % 3 are free
        if (n >= 1) ok = wait_flag(bc_empty, (uint32_t)(n - 1) & 1u, abort_flag, a.err, a.wait_ns);
        if (ok && cur.first) {
          if (lane == 0) {
            mbar_arrive_expect_tx(r_full, (uint32_t)(PT_ROWS * LOWRANK_MAX_D * 2));
            tma_load_3d(smem + L_::lr_r, &tmR, 0, cur.it.h, cur.it.t0, r_full);
          }
          r_pending = true;
          ok = wait_flag(r_full, (uint32_t)ritems & 1u, abort_flag, a.err, a.wait_ns);
          ++ritems;
          r_pending = !ok;
        }
        if (ok) ok = wait_flag(&pt_full[n % 3], (uint32_t)(n / 3) & 1u, abort_flag, a.err, a.wait_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t rb = smem_u32(smem + L_::lr_r);
        const uint32_t pb = smem_u32(smem + L_::lr_p + (size_t)(n % 3) * PT_BYTES);
#pragma unroll
        for (int kk = 0; kk < LOWRANK_MAX_D / 16; ++kk) {
          const uint64_t ad = umma_desc_sw128(rb + kk * 32, 16, 1024);
          const uint64_t bd = umma_desc_sw128(pb + kk * 32, 16, 1024);
          umma_ss_warp(tmem + TM_BC, ad, bd, IDESC_S, kk > 0 ? 1u : 0u);
        }
        umma_commit_warp(bc_full);
        __syncwarp();
        // chunk n + 2 into slot (n + 2) % 3, last read by MMA n - 1 (complete, see above)
        if (pf.valid) {
          if (lane == 0) {
            mbar_arrive_expect_tx(&pt_full[(n + 2) % 3], PT_BYTES);
            tma_load_2d(smem + L_::lr_p + (size_t)((n + 2) % 3) * PT_BYTES, &tmP, 0, pf.s, &pt_full[(n + 2) % 3]);
          }
          ++issued;
          lr_advance(a, total_items, pf);
        }
        lr_advance(a, total_items, cur);
        ++n;
      }
      if (lane == 0) {
        // after an abort, loads may still be landing: wait (bounded) for every load not yet
        // waited for, so none is in flight when the CTA exits
#pragma unroll 1
        for (int e = n; e < issued; ++e)
          if (!mbar_wait_bounded(&pt_full[e % 3], (uint32_t)(e / 3) & 1u)) record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
        if (r_pending && !mbar_wait_bounded(r_full, (uint32_t)(ritems - 1) & 1u)) record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
      }
      umma_commit_warp(&drains[1]);
      __syncwarp();
      if (!mbar_wait_bounded(&drains[1], 0)) record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
    } else {
    int bcnt[2] = {0, 0};   // bias tiles loaded per warpgroup
    int g = 0;
    bool go = true;
    for (int i = blockIdx.x; i < total_items && go; i += gridDim.x) {
      PItem it;
      if (!get_item(a, i, it) || it.ntile == 0) continue;
      for (int j = 0; j < it.ntile; ++j, ++g) {
        const int k0 = (it.kt0 + j) * TILE_KEYS;
        if (!tile_needs_bias(it.pos0, k0, a.E)) continue;
        const int u = bcnt[g & 1];
        const int slot = (g & 1) * BS::PER_WG + u % BS::PER_WG, use = u / BS::PER_WG;
        BT* sb = reinterpret_cast<BT*>(smem + L_::bias + (size_t)slot * BS::SLOT_BYTES);
        const int dmin0 = it.pos0 - (k0 + TILE_KEYS - 1);
        if (use >= 1 &&
            !__all_sync(0xffffffffu, wait_flag(&b_empty[slot], (uint32_t)(use - 1) & 1u, abort_flag, a.err, a.wait_ns))) {
          go = false;
          break;
        }
        ++bcnt[g & 1];
        if (a.bias_bulk) {
          // lane gr < NGROUP decides whether group gr of this tile is read; the warp loads those
          const uint32_t nm =
              __ballot_sync(0xffffffffu, lane < BS::NGROUP && bias_group_needed(a, it, k0, lane));
          mbar_arrive_expect_tx_warp(&b_full[slot], (uint32_t)__popc(nm) * (uint32_t)(BS::GROUP * sizeof(BT)));
#pragma unroll 1
          for (uint32_t mm = nm; mm; mm &= mm - 1) {
            const int gr = __ffs(mm) - 1;
            tma_load_3d_warp(sb + gr * BS::GROUP, &tmB, bias_group_x<BS::ALIGN>(dmin0, gr), it.h,
                             it.t0 + BIAS_BOX_ROWS * gr, &b_full[slot]);
          }
        } else if constexpr (BM == BM_F32) {   // fp32 rows that are not 16-byte aligned (never bf16)
#pragma unroll 1
          for (int r = 0; r < it.rows; ++r) {
            const int pr = it.pos0 + r;
            int kmin, kmax;
            row_tile_keys(a, it, pr, k0, kmin, kmax);
            const float* srcr = static_cast<const float*>(a.rel) + ((size_t)(it.t0 + r) * a.Hq + it.h) * a.E;
            const int gr = r / BIAS_BOX_ROWS, ii = r % BIAS_BOX_ROWS;
            const int xg = bias_group_x<BS::ALIGN>(dmin0, gr);
            // bucket d sits at group_base + ii*COLS + (d - x_g); visible keys give d >= x_g
            const uint32_t rb = smem_u32(sb + gr * BS::GROUP + ii * BS::COLS);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int c = lane + 32 * half;
              const int k = k0 + c;
              const int d = pr - k;
              if (k >= kmin && k <= kmax && d < a.E - 1) cp_async_4(rb + (uint32_t)((d - xg) * 4), srcr + d);
            }
          }
          cp_async_mbar_arrive_noinc(&b_full[slot]);
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // TMA path: the last fill of each slot may still be landing after an abort
    if (a.bias_bulk && lane == 0) {
#pragma unroll 1
      for (int w = 0; w < 2; ++w)
#pragma unroll 1
        for (int u = max(0, bcnt[w] - BS::PER_WG); u < bcnt[w]; ++u)
          if (!mbar_wait_bounded(&b_full[w * BS::PER_WG + u % BS::PER_WG], (uint32_t)(u / BS::PER_WG) & 1u))
            record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
    }
    }
  } else if (warp >= 12) {
    if constexpr (BM == BM_LOWRANK) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(LR_REGS_BIAS));
    // -------------------------------------------------------------- bias warps (low-rank)
    // Warp 12 + q reads TMEM lanes 32 q .. 32 q + 31 (rows of the item) of every bias chunk
    // and writes each row's 64 values, as fp16, into the slots of the (up to three) tiles
    // whose windows hold the chunk: tile t + k sees chunk [s, s + 64) at window offset
    // (s - x_0(t)) + 64 k.  Slot t % 4 row r (group g = r / 16) holds the 80 buckets
    // x_0 + 16 g + [0, 80).  Before the first write into a slot for tile t', the tile that
    // used it before (t' - 4) must have been consumed by its softmax warpgroup.
    if constexpr (BM == BM_LOWRANK) {
      const int q = warp - 12;
      const int row = 32 * q + lane, grp = row >> 4, irow = row & 15;
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + TM_BC;
      int t = 0, n = 0, waited = -1;
      for (int i = blockIdx.x; i < total_items; i += gridDim.x) {
        PItem it;
        if (!get_item(a, i, it) || it.ntile == 0) continue;
        const int jb = lr_first_bias_tile(a, it);
        for (int j = jb; j < it.ntile; ++j, ++t) {
          const int nch = j == jb ? 3 : 1;
#pragma unroll 1
          for (int m = 0; m < nch; ++m) {
            const bool ok = wait_flag(bc_full, (uint32_t)n & 1u, abort_flag, a.err, a.wait_ns);
            ++n;
            tc_fence_after();
            uint32_t h[32];   // this row's 64 buckets of the chunk, fp16 pairs
            {
              uint32_t v[32];
              tmem_ld32(taddr, v);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) h[e] = pack_half2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
              tmem_ld32(taddr + 32, v);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e)
                h[16 + e] = pack_half2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bc_empty);   // TMEM may take the next product
            if (!ok) continue;
            const int off0 = j == jb ? LOWRANK_CHUNK * m : 0;   // the chunk's offset in tile t's window
#pragma unroll 1
            for (int k = 0; k < 3; ++k) {
              const int off = off0 + LOWRANK_CHUNK * k;
              if (off >= 3 * LOWRANK_CHUNK || j + k >= it.ntile) break;
              const int tt = t + k, sl = tt & 3;
              if (tt > waited) {
                if (tt >= 4) (void)wait_flag(&b_empty[sl], (uint32_t)((tt >> 2) - 1) & 1u, abort_flag, a.err, a.wait_ns);
                waited = tt;
              }
              __half* dst = reinterpret_cast<__half*>(smem + L_::bias + (size_t)sl * BS::SLOT_BYTES) +
                            grp * BS::GROUP + irow * BS::COLS;
#pragma unroll
              for (int qv = 0; qv < 8; ++qv) {
                const int col = off + 8 * qv - BIAS_BOX_ROWS * grp;   // slot column of bucket s + 8 qv
                if (col >= 0 && col < BS::COLS)
                  *reinterpret_cast<uint4*>(dst + col) = make_uint4(h[4 * qv], h[4 * qv + 1], h[4 * qv + 2], h[4 * qv + 3]);
              }
              if (k == 0 && m == nch - 1) mbar_arrive(&b_full[sl]);   // all 32 lanes: tile t is complete
            }
          }
        }
      }
    }
  } else {
    if constexpr (BM == BM_LOWRANK) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(LR_REGS_SOFTMAX));
    // -------------------------------------------------------------- softmax warpgroups
    // Warpgroup wg (warps 4-7: wg 0, warps 8-11: wg 1) owns the tiles g with g % 2 == wg
    // and its own O accumulator in TMEM; thread r of a warpgroup owns row r.  At the end
    // of an item wg 1 hands (max, sum) of its rows to wg 0 through shared memory and wg 0
    // merges both partial results and writes the output.
    const int wg = (warp - 4) >> 2;
    const int sw = (warp - 4) & 3;
    const int r = sw * 32 + lane;
    const uint32_t tlane = tmem + ((uint32_t)(sw * 32) << 16);
    const uint32_t tm_o = tlane + TM_O + (uint32_t)(wg * D);
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
    int icount = 0, g = 0, buse = 0;  // buse: bias tiles this warpgroup has consumed
    int btile = 0;                     // low-rank mode: bias tiles of the CTA so far (both warpgroups)
    for (int i = blockIdx.x; i < total_items; i += gridDim.x) {
      PItem it;
      if (!get_item(a, i, it)) continue;
      const bool rv = r < it.rows;
      if (wg == 0 && sw == 0 && lane == 0 && it.t0 == __ldg(a.cu_q + it.b) && it.h == 0) {
        if (it.n > a.max_q_len) record_error(a.err, INK_DEVERR_QLEN_EXCEEDS_MAX);
        if (it.bad_len) record_error(a.err, INK_DEVERR_QLEN_EXCEEDS_KV);
        else if ((long long)it.L > ((long long)a.max_pages << a.log2_page))
          record_error(a.err, INK_DEVERR_PAGE_OUT_OF_RANGE);
      }
      if (it.ntile == 0) {  // nothing visible (inconsistent lengths or no readable key): zeros
        if (wg == 0 && rv) {
          uint4* o = reinterpret_cast<uint4*>(out + ((size_t)(it.t0 + r) * a.Hq + it.h) * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      const int pr = it.pos0 + r;
      float clamp_ld;
      if constexpr (BM == BM_LOWRANK) {
        // bucket E - 1 of this row: r[t, h, :] . proj_t[E - 1, :], in fp32
        const uint4* rr = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.lr_r) +
                                                         ((size_t)(it.t0 + (rv ? r : it.rows - 1)) * a.Hq + it.h) * a.d_rel);
        const uint4* pe = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.lr_proj_t) +
                                                         (size_t)(a.E - 1) * a.d_rel);
        float acc = 0.f;
#pragma unroll 1
        for (int w8 = 0; w8 < a.d_rel / 8; ++w8) {
          const uint4 x = __ldg(rr + w8), y = __ldg(pe + w8);
          const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), acc);
            acc = fmaf(__uint_as_float(xs[e] & 0xFFFF0000u), __uint_as_float(ys[e] & 0xFFFF0000u), acc);
          }
        }
        clamp_ld = acc;
      } else {
        // (rows past the item's last use its last row's address: never outside rel)
        const BT* relrow = static_cast<const BT*>(a.rel) + ((size_t)(it.t0 + (rv ? r : it.rows - 1)) * a.Hq + it.h) * a.E;
        clamp_ld = to_float(__ldg(relrow + a.E - 1));
      }
      const float clampv = rv ? clamp_ld : 0.f;   // bucket of distances >= E - 1
      const int32_t* bt = a.block_table + (size_t)it.b * a.max_pages;
      const int seg = P < TILE_KEYS ? P : TILE_KEYS;
      // Does some page holding a key of the item lie outside the pool?  (Checked once per
      // item; only then are per-tile masks of unreadable keys built.)
      bool item_bad = false;
      {
        const int p0 = it.lo_min >> a.log2_page, p1 = it.k_hi >> a.log2_page;
#pragma unroll 1
        for (int pi = p0 + lane; pi <= p1; pi += 32) {
          const int page = __ldg(bt + pi);
          item_bad |= page < 0 || page >= a.num_pages;
        }
        item_bad = __any_sync(0xffffffffu, item_bad);
      }
      // unreadable keys of a tile (same rule as the producers: segments holding a key some
      // row of the item may see, with a page id outside the pool)
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
      const int g0 = g;
      // running max (natural units) and sum of this warpgroup's tiles
      float m = -INFINITY, l = 0.f;
      bool fresh = true;  // no tile of this item seen yet by this warpgroup
      for (int j = 0; j < it.ntile; ++j, ++g) {
        const int k0 = (it.kt0 + j) * TILE_KEYS;
        const bool needs = tile_needs_bias(it.pos0, k0, a.E);
        const int my_bt = btile;
        if (BM == BM_LOWRANK && needs) ++btile;
        if ((g & 1) != wg) continue;  // the other warpgroup's tile
        // this tile's bias slot: the warpgroup's next fill, or (low-rank) bias tile my_bt % 4
        const int bslot_i = BM == BM_LOWRANK ? (my_bt & 3) : wg * BS::PER_WG + buse % BS::PER_WG;
        const uint32_t bpar = BM == BM_LOWRANK ? (uint32_t)(my_bt >> 2) & 1u : (uint32_t)(buse / BS::PER_WG) & 1u;
        const BT* bslot = reinterpret_cast<const BT*>(smem + L_::bias + (size_t)bslot_i * BS::SLOT_BYTES);
        uint64_t bad = item_bad ? tile_bad(k0) : 0ull;
        bool ok = wait_flag(&s_full[g & 1], (uint32_t)(g >> 1) & 1u, abort_flag, a.err, a.wait_ns);
        tc_fence_after();
        uint32_t sr[64];
        {
          uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
          uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
          tmem_ld32(tlane + TM_S + (g & 1) * 64, lo);
          tmem_ld32(tlane + TM_S + (g & 1) * 64 + 32, hi);
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[g & 1]);
        if (!ok) bad = ~0ull;
        // visible columns of this row: [kmin - k0, kmax - k0] less unreadable keys
        int kmin, kmax;
        row_tile_keys(a, it, pr, k0, kmin, kmax);
        uint64_t vis = 0;
        if (rv && kmax >= kmin) vis = (~0ull >> (TILE_KEYS - 1 - (kmax - k0))) & (~0ull << (kmin - k0));
        vis &= ~bad;
        // key c sits at distance dmin + 63 - c; columns c <= cc read bucket E - 1
        const int dmin = pr - (k0 + TILE_KEYS - 1);
        const int cc = dmin + TILE_KEYS - a.E;
        // bucket of key c at brow[-c] (group_base + i*COLS + (d - x_g)); any address in the
        // slot when the tile reads no bucket from it
        const BT* brow = bslot + (TILE_KEYS - 1);
        if (needs) {
          (void)wait_flag(&b_full[bslot_i], bpar, abort_flag, a.err, a.wait_ns);
          const int gr = r / BIAS_BOX_ROWS;
          brow = bslot + gr * BS::GROUP + (r % BIAS_BOX_ROWS) * BS::COLS + (dmin - bias_group_x<BS::ALIGN>(dmin - r, gr)) +
                 (TILE_KEYS - 1);
        }
        float mxv[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        const bool all_vis = vis == ~0ull;
        if (__all_sync(0xffffffffu, all_vis && cc < 0)) {
          // every key visible, every bucket from the tile's bias rows
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float sv = fmaf(__uint_as_float(sr[c]), a.sm_scale, to_float(brow[-c]));
            sr[c] = __float_as_uint(sv);
            mxv[c & 3] = fmaxf(mxv[c & 3], sv);
          }
        } else if (__all_sync(0xffffffffu, all_vis && cc >= TILE_KEYS - 1)) {
          // every key visible at distance >= E - 1
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float sv = fmaf(__uint_as_float(sr[c]), a.sm_scale, clampv);
            sr[c] = __float_as_uint(sv);
            mxv[c & 3] = fmaxf(mxv[c & 3], sv);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float bsv = c <= cc ? clampv : to_float(brow[-c]);
            const float sv = ((vis >> c) & 1ull) ? fmaf(__uint_as_float(sr[c]), a.sm_scale, bsv) : -INFINITY;
            sr[c] = __float_as_uint(sv);
            mxv[c & 3] = fmaxf(mxv[c & 3], sv);
          }
        }
        const float mx = fmaxf(fmaxf(mxv[0], mxv[1]), fmaxf(mxv[2], mxv[3]));
        if (needs) {
          // every bias value this thread read is consumed (mx depends on all of them)
          asm volatile("" ::"f"(mx) : "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(&b_empty[bslot_i]);
          ++buse;
        }
        const float m_new = fmaxf(m, mx);
        if (fresh) {
          m = m_new;
        } else {
          const bool mine = m_new > m + RESCALE_NAT;
          if (__any_sync(0xffffffffu, mine)) {
            // this warpgroup's O must be stable: its previous P V product (tile g - 2) is done
            (void)wait_flag(&o_done[g & 1], (uint32_t)((g - 2) >> 1) & 1u, abort_flag, a.err, a.wait_ns);
            tc_fence_after();
            const float f = mine ? fast_exp2((m - m_new) * LOG2E) : 1.f;
#pragma unroll 1
            for (int cc2 = 0; cc2 < D / 32; ++cc2) {
              uint32_t ov[32];
              tmem_ld32(tm_o + cc2 * 32, ov);
              tmem_wait_ld();
#pragma unroll
              for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * f);
              tmem_st32(tm_o + cc2 * 32, ov);
            }
            tmem_wait_st();
            l *= f;
            if (mine) m = m_new;
          }
        }
        // p = 2^(s log2(e) - m log2(e)); masked keys (s = -inf) give exactly 0
        const float mb = m == -INFINITY ? 0.f : m * LOG2E;
        uint32_t pk[32];
        float lsv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(sr[2 * c]), LOG2E, -mb));
          const float p1 = fast_exp2(fmaf(__uint_as_float(sr[2 * c + 1]), LOG2E, -mb));
          lsv[c & 3] += p0 + p1;
          pk[c] = pack_bf16(p0, p1);
        }
        l += (lsv[0] + lsv[1]) + (lsv[2] + lsv[3]);
        // P buffer g & 1 was last read by the P V product of tile g - 2
        if (g >= 2) (void)wait_flag(&o_done[g & 1], (uint32_t)((g - 2) >> 1) & 1u, abort_flag, a.err, a.wait_ns);
        tmem_st32(tlane + TM_P + (g & 1) * 32, pk);
        tmem_wait_st();
        tc_fence_before();
        named_barrier_sync(1 + wg, 128);   // all 128 rows of P(g) are in TMEM
        if (sw == 0) {
          // O[wg] += P(g) V(g), issued by this warpgroup's first warp
          const int vs = g % NV;   // NV is even: this warpgroup's own V slots
          bool pv_ok = wait_flag(&v_full[vs], (uint32_t)(g / NV) & 1u, abort_flag, a.err, a.wait_ns);
          // warpgroup 1's first product of an item overwrites O[1], which the previous
          // item's epilogue (warpgroup 0) reads: wait until it has
          if (fresh && wg == 1 && icount > 0) pv_ok = wait_flag(o_free, (uint32_t)(icount - 1) & 1u, abort_flag, a.err, a.wait_ns) && pv_ok;
          // zero the V rows of keys that no row of this item may read
          const uint64_t vb = pv_ok ? vbad[vs] : ~0ull;
          uint8_t* vt = smem + L_::vst + (size_t)vs * S::KV_TILE;
          if (k0 < it.lo_min || k0 + TILE_KEYS - 1 > it.k_hi || vb) {
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
          pv_ok = __all_sync(0xffffffffu, pv_ok);
          tc_fence_after();
          if (pv_ok) {
            const uint32_t vbase = smem_u32(vt);
#pragma unroll
            for (int ks = 0; ks < TILE_KEYS / 16; ++ks) {
              const uint64_t bdesc = umma_desc_sw128(vbase + ks * 16 * 128, S::KV_SUB, 1024);
              umma_ts_warp(tmem + TM_O + (uint32_t)(wg * D), tmem + TM_P + (g & 1) * 32 + ks * 8, bdesc, IDESC_PV,
                           (fresh && ks == 0) ? 0u : 1u);
            }
          }
          umma_commit_warp(&v_empty[vs]);
          umma_commit_warp(&o_done[g & 1]);
          __syncwarp();
        }
        fresh = false;
      }
      // ---- item epilogue
      const int g_last = g - 1;
      if (wg == 1) {
        if (icount > 0) (void)wait_flag(ml_free, (uint32_t)(icount - 1) & 1u, abort_flag, a.err, a.wait_ns);
        ml1[r] = make_float2(m, l);
        __syncwarp();
        if (lane == 0) mbar_arrive(ml_full);
      } else {
        // Warpgroup 1 first: once it has stored its last P it has waited for its P V
        // product two tiles back, so o_done[1] is at most one phase short of the count
        // awaited below.  Waiting on o_done[1] earlier could see a phase two behind,
        // whose parity matches, and read O_1 before its last product lands.
        (void)wait_flag(ml_full, (uint32_t)icount & 1u, abort_flag, a.err, a.wait_ns);
        // both warpgroups' last P V products of the item are done
        (void)wait_flag(&o_done[g_last & 1], (uint32_t)(g_last >> 1) & 1u, abort_flag, a.err, a.wait_ns);
        if (g_last > g0)
          (void)wait_flag(&o_done[(g_last - 1) & 1], (uint32_t)((g_last - 1) >> 1) & 1u, abort_flag, a.err, a.wait_ns);
        tc_fence_after();
        const float2 o1 = ml1[r];
        __syncwarp();
        if (lane == 0) mbar_arrive(ml_free);
        const float M = fmaxf(m, o1.x);
        const float Mu = M == -INFINITY ? 0.f : M;
        const bool has0 = l > 0.f, has1 = o1.y > 0.f;   // a warpgroup without tiles holds stale O
        const float f0 = has0 ? fast_exp2((m - Mu) * LOG2E) : 0.f;
        const float f1 = has1 ? fast_exp2((o1.x - Mu) * LOG2E) : 0.f;
        const float Lt = l * f0 + o1.y * f1;
        const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
        const float c0 = f0 * inv, c1 = f1 * inv;
        uint4* orow = reinterpret_cast<uint4*>(out + ((size_t)(it.t0 + r) * a.Hq + it.h) * D);
        const uint32_t t_o0 = tlane + TM_O, t_o1 = tlane + TM_O + D;
        const bool store = rv && !*abort_flag;   // after an abort the rows are left untouched
#pragma unroll 1
        for (int cc = 0; cc < D / 16; ++cc) {
          uint32_t ov[16], ow[16];
          tmem_ld16(t_o0 + cc * 16, ov);
          tmem_ld16(t_o1 + cc * 16, ow);
          tmem_wait_ld();
          if (store) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float a0 = has0 ? __uint_as_float(ov[2 * e]) * c0 : 0.f;
              const float a1 = has1 ? __uint_as_float(ow[2 * e]) * c1 : 0.f;
              const float b0 = has0 ? __uint_as_float(ov[2 * e + 1]) * c0 : 0.f;
              const float b1 = has1 ? __uint_as_float(ow[2 * e + 1]) * c1 : 0.f;
              w[e] = pack_bf16(a0 + a1, b0 + b1);
            }
            if (a.io32) {
              asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(orow + cc * 2), "r"(w[0]),
                           "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                           : "memory");
            } else {
              orow[cc * 2] = make_uint4(w[0], w[1], w[2], w[3]);
              orow[cc * 2 + 1] = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free);
      }
      ++icount;
    }
    if (sw == 0) {   // this warpgroup's P V products are complete before tensor memory is released
      umma_commit_warp(&drains[2 + wg]);
      __syncwarp();
      if (!mbar_wait_bounded(&drains[2 + wg], 0)) record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(TM_COLS));
  }
}

int num_sms_pf() {
  int dev = 0;
  const int n = current_device_sms(&dev);
  return n > 0 ? n : 148;
}

template <int D, int BM>
cudaError_t launch_prefill_tc_t(const PrefillMaps& m, const PrefillArgs& a, cudaStream_t stream) {
  constexpr size_t smem = PtSmem<D, BM>::alloc;
  static_assert(smem <= 227 * 1024, "shared memory budget");
  static_assert(PtShape<D, BM>::NV % 2 == 0, "each V slot must serve one softmax warpgroup");
  static std::atomic<unsigned long long> opted{0};
  cudaError_t e = smem_opt_in_once(prefill_tc_kernel<D, BM>, (int)smem, opted);
  if (e != cudaSuccess) return e;
  const long long items = (long long)a.num_q_tiles * a.B * a.Hq;
  const int grid = (int)std::min<long long>(items, num_sms_pf());
  prefill_tc_kernel<D, BM><<<grid, BM == BM_LOWRANK ? PT_THREADS_LR : PT_THREADS, smem, stream>>>(
      m.k, m.v, m.k3, m.v3, m.q3, m.bias, m.lr_r, m.lr_p, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillMaps& m, const PrefillArgs& a, int head_dim, cudaStream_t stream) {
  if (a.bias_lowrank)
    return head_dim == 128 ? launch_prefill_tc_t<128, BM_LOWRANK>(m, a, stream)
                           : launch_prefill_tc_t<64, BM_LOWRANK>(m, a, stream);
  if (a.bias_bf16)
    return head_dim == 128 ? launch_prefill_tc_t<128, BM_BF16>(m, a, stream) : launch_prefill_tc_t<64, BM_BF16>(m, a, stream);
  return head_dim == 128 ? launch_prefill_tc_t<128, BM_F32>(m, a, stream) : launch_prefill_tc_t<64, BM_F32>(m, a, stream);
}

}  // namespace ink
