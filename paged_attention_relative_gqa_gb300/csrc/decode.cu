// decode.cu -- persistent split-K flash-decode over a paged K/V cache with a per-token
// relative-position bias ("Support Inkling-NVFP4 model", TensorRT-LLM PR #17062,
// sections "Architecture" and "Implementation": one new token per request attends to
// its paged history, the bias rel[b, h, distance] added before the softmax; 512-key
// windows on local layers, full causal on global layers).
//
// Work unit: (split s, sequence b, KV head, chunk of <= 16 query heads sharing that KV
// head).  A split is a run of `tiles_per_split` 64-key tiles of the sequence's visible
// range [lo, p], p = L - 1.  One CTA per SM walks units blockIdx.x, +gridDim.x, ...;
// units whose split lies past the sequence's visible range are skipped by every warp
// alike, so the producer and consumers need no unit hand-off.
//
// Two CTAs per SM.  Warp roles:
//   warp 4 (producer, one lane): block-table walk (page of key k is
//     block_table[b][k / P]; entries past the sequence's own pages are never read),
//     then 2-D TMA loads of K and V rows into a ring of NSTAGE shared-memory stages
//     (128-byte swizzle, full/empty mbarriers).  Whole 64-key tiles use 64-row boxes;
//     tiles cut by the window start or the sequence end load only the 16-row segments
//     that hold visible keys.  The first tile of a unit also carries the unit's query
//     rows (TMA over q viewed as [B*Hq, D]).  The producer runs ahead across units.
//   warps 0-3 (consumers): each takes 16 keys of every tile: S = Q K^T (mma.sync,
//     query heads are the 16 MMA rows), s2 = S * sm_scale * log2(e) + bias * log2(e),
//     keys outside [lo, p] or in unreadable pages -> -inf, online softmax in base 2 (the
//     running max moves only when a score passes it by more than 8, so most tiles skip
//     the cross-lane max and the rescale of O),
//     O += P V with V rows of masked keys zeroed in registers.  The bias values of the
//     next tile are prefetched into registers while the current one is computed.
// Unit epilogue: the 4 warps' (max, sum, O) are merged through shared memory; a
// sequence with one split writes bf16 output, otherwise fp32 partials go to the
// workspace and the last CTA to finish that sequence (atomic ticket, no spinning)
// merges all partials in split order -- the result does not depend on arrival order --
// and resets the ticket.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace ink {

namespace {

constexpr int DEC_CONSUMERS = 4;
// With at most 8 query heads per unit two CTAs share an SM: 8 consumer warps per SM hide
// each other's latencies, which matters more than a deeper ring (registers are capped
// at 65536 / (2 * 160) = 204).  16-head units need the room of a whole SM.
template <int HB>
constexpr int dec_ctas_per_sm() { return HB == 8 ? 2 : 1; }
constexpr int DEC_THREADS = (DEC_CONSUMERS + 1) * 32;
constexpr int QROWS = 16;       // query-head rows per unit (MMA M)
constexpr int SEG_ROWS = 16;    // fine TMA box rows for partial tiles
constexpr int PTAB = 576;       // staged block-table entries per unit (>= 64 tiles x 64/8 + 2)
constexpr int L2_AHEAD = 1;     // whole tiles prefetched into L2 ahead of their loads

template <int D>
struct DecShape {
  static constexpr int COL_BLOCKS = D / 64;             // 128-byte column blocks
  // K and V tiles are staged group-major: [16-key group][column block][16 rows x 128 B],
  // 2 KB blocks with the 128-byte swizzle; consumer warp w reads group w.
  static constexpr int BLOCK_BYTES = 16 * 128;
  static constexpr int GROUP_BYTES = COL_BLOCKS * BLOCK_BYTES;
  static constexpr int TILE_BYTES = (TILE_KEYS / 16) * GROUP_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;    // K tile + V tile
  static constexpr int QSUB_BYTES = QROWS * 128;        // one column block of the query rows
  static constexpr int QSLOT_BYTES = COL_BLOCKS * QSUB_BYTES;
  static constexpr int OPITCH = D + 4;                  // fp32 merge buffer row pitch
};

constexpr int BIAS_DIST = 3;               // tiles a consumer warp stages its bias ahead of use
constexpr int BIAS_SLOTS = BIAS_DIST + 1;
constexpr int BIAS_PITCH = 20;             // floats per staged (head) row of a warp's 16 keys

template <int D, int NSTAGE, int HB>
struct DecSmem {
  using S = DecShape<D>;
  static constexpr size_t stages = 0;
  static constexpr size_t q = stages + (size_t)NSTAGE * S::STAGE_BYTES;
  static constexpr size_t bias = q + 2 * S::QSLOT_BYTES;
  static constexpr size_t obuf = bias + (size_t)DEC_CONSUMERS * BIAS_SLOTS * HB * BIAS_PITCH * 4;
  static constexpr size_t red = obuf + (size_t)DEC_CONSUMERS * HB * S::OPITCH * 4;
  static_assert((size_t)DEC_CONSUMERS * HB * S::OPITCH * 4 >= 16 * MAX_DECODE_SPLITS * 8, "merge scratch in obuf");
  static constexpr size_t wts = red + (2 * DEC_CONSUMERS * 16 + 2 * 16) * 4;
  static constexpr size_t bars = wts + 16 * MAX_DECODE_SPLITS * 4;  // 8-byte aligned
  static constexpr size_t badmask = bars + (2 * NSTAGE + 4 + DEC_CONSUMERS * BIAS_SLOTS) * 8;
  static constexpr size_t flags = badmask + NSTAGE * 8;
  static constexpr size_t ptab = flags + 16;
  static constexpr size_t total = ptab + 3 * PTAB * 4;
  static constexpr size_t alloc = total + 1024;  // base alignment slack
};

struct Unit {
  int b, kvh, hc, s, h0, nh, L, p, lo, tb, n_my, nact;
};

// Decode potential unit u.  Returns false when the unit has nothing to do.  A sequence
// with L <= 0 yields one unit (split 0) with n_my = 0: its output rows are zeroed.
__device__ __forceinline__ bool get_unit(const DecodeArgs& a, int u, Unit& w) {
  const int per_s = a.B * a.Hkv * a.head_chunks;
  w.s = u / per_s;
  int r = u - w.s * per_s;
  const int per_b = a.Hkv * a.head_chunks;
  w.b = r / per_b;
  r -= w.b * per_b;
  w.kvh = r / a.head_chunks;
  w.hc = r - w.kvh * a.head_chunks;
  w.h0 = w.kvh * a.G + w.hc * QROWS;
  w.nh = min(QROWS, a.G - w.hc * QROWS);
  int L = __ldg(a.seq_lens + w.b);
  if (L <= 0) {
    w.L = 0;
    w.n_my = 0;
    w.nact = 1;
    return w.s == 0;
  }
  const long long cap = (long long)a.max_pages << a.log2_page;
  if (L > cap) L = (int)cap;  // keys past the table's reach are not readable (error recorded)
  w.L = L;
  w.p = L - 1;
  w.lo = a.W > 0 ? max(0, w.p - a.W + 1) : 0;
  const int t_first = w.lo / TILE_KEYS, t_last = w.p / TILE_KEYS;
  const int ntiles = t_last - t_first + 1;
  w.nact = min((ntiles + a.tiles_per_split - 1) / a.tiles_per_split, a.num_splits);
  if (w.s >= w.nact) return false;
  w.tb = t_first + w.s * a.tiles_per_split;
  w.n_my = (w.s == w.nact - 1) ? (t_last + 1 - w.tb) : a.tiles_per_split;
  return true;
}

// First and last block-table index a unit reads (pages holding its visible keys).
__device__ __forceinline__ void unit_page_span(const DecodeArgs& a, const Unit& w, int& first, int& count) {
  const int kf = max(w.tb * TILE_KEYS, w.lo);
  const int kl = min((w.tb + w.n_my) * TILE_KEYS - 1, w.p);
  first = kf >> a.log2_page;
  count = (kl >> a.log2_page) - first + 1;
}

// Segments of tile i of unit w to fetch: `whole` (one 64-row box) when every key of the
// tile is visible and the page holds the whole tile, else 16-row (or P-row) segments
// that hold at least one visible key.  rows[sg] is the pool row of segment sg, or -1
// (nothing to fetch), or -2 (unreadable page: its keys are masked).  Page ids come from
// the unit's slice of the block table, staged in shared memory (ptab[j] = entry first+j).
// Does tile k0 of unit w need its own bias values?  Not when every visible key of the
// tile is at distance >= E - 1: those all read the clamped bucket E - 1.
__device__ __forceinline__ bool tile_needs_bias(const Unit& w, int k0, int E) {
  return max(w.p - (k0 + TILE_KEYS - 1), 0) < E - 1;
}

__device__ __forceinline__ void named_barrier_consumers() {
  asm volatile("bar.sync 1, %0;" ::"n"(DEC_CONSUMERS * 32) : "memory");
}

// Wait on an mbarrier phase unless the CTA has aborted; on timeout, record the error
// and abort the CTA (every later wait returns at once).
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              uint32_t* err, unsigned long long limit_ns) {
  if (*abort_flag) return false;
  if (mbar_wait_limit(bar, parity, limit_ns)) return true;
  record_error(err, INK_DEVERR_WAIT_TIMEOUT);
  *abort_flag = 1;
  return false;
}

// One split of a unit has its partials in the workspace: take the unit's ticket, and the
// last of its splits to arrive merges all of them in split order and resets the ticket.
// Run by the 128 consumer threads alike.  Out of line: it is off the tile loop's path.
// Ordering: every thread's partial stores come before the CTA barrier, thread 0's ticket
// add releases them at GPU scope and acquires the other splits' (the pattern of a
// grid-wide semaphore), and the barrier after it hands that on to the threads that read.
// The (max, sum) pairs of all splits are read at once into `scratch` (shared memory of at
// least 16 x MAX_DECODE_SPLITS float2, free at this point), so the merge costs two round
// trips to L2 rather than one per split.
template <int D>
__device__ __noinline__ void finish_split_unit(const float* part_o, const float* part_ml, int32_t* tickets,
                                               __nv_bfloat16* out, int Hq, int Hkv, int head_chunks, int num_splits,
                                               int b, int kvh, int hc, int h0, int nh, int nact, int tid,
                                               int* flags, float* wts, float2* scratch) {
  const size_t rowbase = (size_t)b * Hq + h0;
  named_barrier_consumers();
  const size_t ticket = ((size_t)b * Hkv + kvh) * head_chunks + hc;
  if (tid == 0) {
    int prev;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(tickets + ticket) : "memory");
    flags[0] = prev == nact - 1;
  }
  named_barrier_consumers();
  if (!flags[0]) return;
  // scratch[r * MAX_DECODE_SPLITS + sp] <- (max, sum) of split sp of row r
  for (int i = tid; i < nh * nact; i += DEC_CONSUMERS * 32) {
    const int r = i / nact, sp = i - r * nact;
    scratch[r * MAX_DECODE_SPLITS + sp] = __ldcg(reinterpret_cast<const float2*>(part_ml) + (rowbase + r) * num_splits + sp);
  }
  named_barrier_consumers();
  if (tid < nh) {
    const float2* row = scratch + tid * MAX_DECODE_SPLITS;
    float M = -INFINITY;
    for (int sp = 0; sp < nact; ++sp) M = fmaxf(M, row[sp].x);
    const float Mu = M == -INFINITY ? 0.f : M;
    float Lt = 0.f;
    for (int sp = 0; sp < nact; ++sp) Lt += row[sp].y * fast_exp2(row[sp].x - Mu);
    const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
    for (int sp = 0; sp < nact; ++sp) wts[tid * MAX_DECODE_SPLITS + sp] = fast_exp2(row[sp].x - Mu) * inv;
  }
  named_barrier_consumers();
  for (int idx = tid; idx < nh * (D / 4); idx += DEC_CONSUMERS * 32) {
    const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
    const size_t pi0 = (rowbase + r) * num_splits;
    const float* w = wts + r * MAX_DECODE_SPLITS;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int sp = 0; sp < nact; ++sp) {
      const float wt = w[sp];
      const float4 v = __ldcg(reinterpret_cast<const float4*>(part_o + (pi0 + sp) * D + d));
      acc.x += wt * v.x;
      acc.y += wt * v.y;
      acc.z += wt * v.z;
      acc.w += wt * v.w;
    }
    *reinterpret_cast<uint2*>(out + (rowbase + r) * D + d) = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
  }
  if (tid == 0) tickets[ticket] = 0;  // ready for the next call
}

template <int D, int NSTAGE, int HB>
__global__ void __launch_bounds__(DEC_THREADS, dec_ctas_per_sm<HB>())
decode_persistent_kernel(const __grid_constant__ CUtensorMap tmKs, const __grid_constant__ CUtensorMap tmVs,
                         const __grid_constant__ CUtensorMap tmKt, const __grid_constant__ CUtensorMap tmVt,
                         const __grid_constant__ CUtensorMap tmKg, const __grid_constant__ CUtensorMap tmVg,
                         const __grid_constant__ CUtensorMap tmQ3, const DecodeArgs a) {
  using S = DecShape<D>;
  using L_ = DecSmem<D, NSTAGE, HB>;
  constexpr int KSTEPS = D / 16;
  static_assert(HB == 8 || HB == 16, "heads per unit");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L_::bars);
  uint64_t* empty = full + NSTAGE;
  uint64_t* qempty = empty + NSTAGE;  // [2]
  uint64_t* badmask = reinterpret_cast<uint64_t*>(smem + L_::badmask);
  int* flags = reinterpret_cast<int*>(smem + L_::flags);  // [0] ticket winner, [1] abort
  float* red_m = reinterpret_cast<float*>(smem + L_::red);
  float* red_l = red_m + DEC_CONSUMERS * 16;
  float* head_ml = red_l + DEC_CONSUMERS * 16;  // [16][2]: a unit's (max, sum) per head
  float* obuf = reinterpret_cast<float*>(smem + L_::obuf);
  float* wts = reinterpret_cast<float*>(smem + L_::wts);
  volatile int* abort_flag = flags + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = 1 << a.log2_page;
  const int total_units = a.num_splits * a.B * a.Hkv * a.head_chunks;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], DEC_CONSUMERS);
    }
    mbar_init(&qempty[0], DEC_CONSUMERS);
    mbar_init(&qempty[1], DEC_CONSUMERS);
    for (int x = 0; x < DEC_CONSUMERS * BIAS_SLOTS; ++x) mbar_init(&qempty[2 + x], 32);
    fence_mbar_init();
    flags[0] = 0;
    flags[1] = 0;
  }
  __syncthreads();

  if (warp == DEC_CONSUMERS) {
    // ------------------------------------------------------------------ producer
    // The warp stages each unit's slice of the block table into shared memory with
    // cp.async two units ahead (3-slot ring), so no tile waits on a table read; lane 0
    // alone then issues the unit's tiles into the shared-memory ring.  Whole tiles take
    // a short path (one page lookup, four TMA copies for D = 128).
    int* ptab = reinterpret_cast<int*>(smem + L_::ptab);
    if (lane == 0) {
      prefetch_tensormap(&tmQ3);
      if (P >= TILE_KEYS) {
        prefetch_tensormap(&tmKt);
        prefetch_tensormap(&tmVt);
      }
      if (P >= 16) {
        prefetch_tensormap(&tmKg);
        prefetch_tensormap(&tmVg);
      } else {
        prefetch_tensormap(&tmKs);
        prefetch_tensormap(&tmVs);
      }
    }
    const int per_b = a.Hkv * a.head_chunks, per_s = a.B * per_b;
    auto next_active = [&](int u, Unit& w) -> int {
      for (; u < total_units; u += gridDim.x) {
        // warm L1 with the length of the unit four strides on (read by every warp later)
        const int uf = u + 4 * (int)gridDim.x;
        if (uf < total_units) prefetch_l1(a.seq_lens + (uf % per_s) / per_b);
        if (get_unit(a, u, w) && w.n_my > 0) return u;
      }
      return total_units;
    };
    auto stage_ptab = [&](const Unit* w, int slot) {  // w == nullptr: empty group
      if (w) {
        int first, count;
        unit_page_span(a, *w, first, count);
        const int32_t* src = a.block_table + (size_t)w->b * a.max_pages + first;
        const uint32_t dst = smem_u32(ptab + slot * PTAB);
        for (int j = lane; j < count; j += 32) cp_async_4(dst + 4 * j, src + j);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    Unit cur, nxt, nxt2;
    int ucur = next_active(blockIdx.x, cur);
    int unxt = ucur < total_units ? next_active(ucur + gridDim.x, nxt) : total_units;
    stage_ptab(ucur < total_units ? &cur : nullptr, 0);
    stage_ptab(unxt < total_units ? &nxt : nullptr, 1);
    int n = 0, uc = 0;
    bool go = true;
    while (ucur < total_units && go) {
      const int unxt2 = unxt < total_units ? next_active(unxt + gridDim.x, nxt2) : total_units;
      stage_ptab(unxt2 < total_units ? &nxt2 : nullptr, (uc + 2) % 3);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
      __syncwarp();
      const int slot = uc & 1;  // Q slot
      const int* tab = ptab + (uc % 3) * PTAB;
      int pfirst, pcount;
      unit_page_span(a, cur, pfirst, pcount);
      const int row_kv = cur.kvh << a.log2_page;       // + page * Hkv * P
      const int hkvp = a.Hkv << a.log2_page;
      constexpr uint32_t WHOLE_BYTES = 2u * TILE_KEYS * D * 2u;
      // The ring holds NSTAGE tiles; each load issue also starts the K and V boxes of the
      // whole tile L2_AHEAD tiles on (in this unit or the next, whose table slice is staged)
      // towards L2, so that the loads into the ring find them there.
      int nfirst = 0, ncount = 0;
      if (unxt < total_units) unit_page_span(a, nxt, nfirst, ncount);
      const int* ntab = ptab + ((uc + 1) % 3) * PTAB;
      auto prefetch_whole = [&](const Unit& w, const int* wtab, int wfirst, int i) {
        const int k0 = (w.tb + i) * TILE_KEYS;
        if (P < TILE_KEYS || k0 < w.lo || k0 + TILE_KEYS - 1 > w.p) return;
        const int page = wtab[(k0 >> a.log2_page) - wfirst];
        if (page < 0 || page >= a.num_pages) return;
        const int row = page * hkvp + (w.kvh << a.log2_page) + (k0 & (P - 1));
        tma_prefetch_l2_4d(&tmKt, 0, 0, 0, row >> 4);
        tma_prefetch_l2_4d(&tmVt, 0, 0, 0, row >> 4);
      };
      if (uc >= 2) {
        if (lane == 0) go = wait_or_abort(&qempty[slot], (uint32_t)((uc >> 1) - 1) & 1u, abort_flag, a.err, a.wait_ns);
        go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
      }
      for (int i = 0; i < cur.n_my && go; ++i, ++n) {
        const int st = n % NSTAGE;
        if (n >= NSTAGE) {
          if (lane == 0) go = wait_or_abort(&empty[st], (uint32_t)((n / NSTAGE) - 1) & 1u, abort_flag, a.err, a.wait_ns);
          go = __shfl_sync(0xffffffffu, go ? 1 : 0, 0) != 0;
          if (!go) break;
        }
        const int k0 = (cur.tb + i) * TILE_KEYS;
        if (lane == 0) {
          if (i + L2_AHEAD < cur.n_my)
            prefetch_whole(cur, tab, pfirst, i + L2_AHEAD);
          else if (unxt < total_units && i + L2_AHEAD - cur.n_my < nxt.n_my)
            prefetch_whole(nxt, ntab, nfirst, i + L2_AHEAD - cur.n_my);
          uint8_t* kdst = smem + L_::stages + (size_t)st * S::STAGE_BYTES;
          uint8_t* vdst = kdst + S::TILE_BYTES;
          const uint32_t qbytes = i == 0 ? (uint32_t)(S::COL_BLOCKS * QROWS * 128) : 0u;
          if (P >= TILE_KEYS && k0 >= cur.lo && k0 + TILE_KEYS - 1 <= cur.p) {
            const int page = tab[(k0 >> a.log2_page) - pfirst];
            const bool okp = page >= 0 && page < a.num_pages;
            badmask[st] = okp ? 0ull : ~0ull;
            if (!okp) record_error(a.err, INK_DEVERR_PAGE_OUT_OF_RANGE);
            mbar_arrive_expect_tx(&full[st], (okp ? WHOLE_BYTES : 0u) + qbytes);
            if (okp) {
              // one box per tensor: the tile's 4 groups x every column block
              const int row = page * hkvp + row_kv + (k0 & (P - 1));
              tma_load_4d(kdst, &tmKt, 0, 0, 0, row >> 4, &full[st]);
              tma_load_4d(vdst, &tmVt, 0, 0, 0, row >> 4, &full[st]);
            }
          } else {
            // the tile's copies of seg keys (one 16-key group, or an 8-key page) that hold
            // a visible key; pages outside the pool are skipped and their keys masked
            const int seg = P < 16 ? P : 16;
            const int kfirst = max(k0, cur.lo), klast = min(k0 + TILE_KEYS - 1, cur.p);
            uint64_t bad = 0;
            uint32_t bytes = qbytes;
            for (int ks = k0; ks < k0 + TILE_KEYS; ks += seg) {
              if (ks > klast || ks + seg - 1 < kfirst) continue;
              const int page = tab[(ks >> a.log2_page) - pfirst];
              if (page < 0 || page >= a.num_pages) {
                bad |= ((1ull << seg) - 1) << (ks - k0);
                record_error(a.err, INK_DEVERR_PAGE_OUT_OF_RANGE);
              } else {
                bytes += 2u * seg * D * 2u;
              }
            }
            badmask[st] = bad;
            mbar_arrive_expect_tx(&full[st], bytes);
            for (int ks = k0; ks < k0 + TILE_KEYS; ks += seg) {
              if (ks > klast || ks + seg - 1 < kfirst) continue;
              const int page = tab[(ks >> a.log2_page) - pfirst];
              if (page < 0 || page >= a.num_pages) continue;
              const int row = page * hkvp + row_kv + (ks & (P - 1));
              const int off = ((ks - k0) >> 4) * S::GROUP_BYTES;
              if (seg == 16) {
                tma_load_4d(kdst + off, &tmKg, 0, 0, 0, row >> 4, &full[st]);
                tma_load_4d(vdst + off, &tmVg, 0, 0, 0, row >> 4, &full[st]);
              } else {
                const int r16 = ((ks - k0) & 15) * 128;
#pragma unroll
                for (int cb = 0; cb < S::COL_BLOCKS; ++cb) {
                  tma_load_2d(kdst + off + cb * S::BLOCK_BYTES + r16, &tmKs, cb * 64, row, &full[st]);
                  tma_load_2d(vdst + off + cb * S::BLOCK_BYTES + r16, &tmVs, cb * 64, row, &full[st]);
                }
              }
            }
          }
          if (i == 0) {
            uint8_t* qdst = smem + L_::q + slot * S::QSLOT_BYTES;
            tma_load_3d(qdst, &tmQ3, 0, cur.b * a.Hq + cur.h0, 0, &full[st]);
          }
        }
      }
      ++uc;
      cur = nxt;
      ucur = unxt;
      nxt = nxt2;
      unxt = unxt2;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // drain: the last load issued into each stage must land before the CTA exits
    if (lane == 0)
      for (int k = max(0, n - NSTAGE); k < n; ++k)
        (void)mbar_wait_bounded(&full[k % NSTAGE], (uint32_t)(k / NSTAGE) & 1u);
    return;
  }

  // -------------------------------------------------------------------- consumers
  // Transposed products, so no MMA row is padding: S^T = K Q^T has the warp's 16 keys as
  // MMA rows and the unit's query heads as MMA columns (NB blocks of 8), and
  // O^T = V^T P^T.  A thread owns keys (gq, gq + 8) and heads (8j + 2cq, 8j + 2cq + 1):
  // the same two heads in its S^T and O^T fragments, so each thread keeps the running
  // max / sum of exactly the heads whose O^T columns it rescales.
  constexpr int NB = HB / 8;
  const int gq = lane >> 2, cq = lane & 3, mi = lane >> 3;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
  int n = 0, uc = 0;

  // find the first unit with tiles (or a zero-length unit) starting at u
  auto next_unit = [&](int u, Unit& w) -> int {
    for (; u < total_units; u += gridDim.x)
      if (get_unit(a, u, w)) return u;
    return total_units;
  };

  Unit cur, nxt;
  int ucur = next_unit(blockIdx.x, cur);

  // Bias ring of this warp: for stream position t (the t-th tile this CTA consumes) the
  // lanes copy rel[b, h0 + r, min(p - k, E - 1)] for the warp's 16 keys k and the unit's
  // heads r into slot t % BIAS_SLOTS with 4-byte cp.async, BIAS_DIST tiles ahead of use;
  // completion is counted on the slot's mbarrier (32 arrivals, one per lane).
  float* bring = reinterpret_cast<float*>(smem + L_::bias) + warp * BIAS_SLOTS * HB * BIAS_PITCH;
  uint64_t* bfull = qempty + 2 + warp * BIAS_SLOTS;
  Unit bu = cur;          // unit of the next position to stage
  int bu_idx = ucur, bi = 0, bpos = 0;
  auto stage_bias = [&]() {
    // skip zero-length units: they have no tiles in the stream
    while (bu_idx < total_units && bi >= bu.n_my) {
      bu_idx = next_unit(bu_idx + gridDim.x, bu);
      bi = 0;
    }
    const int slot = bpos % BIAS_SLOTS;
    if (bu_idx < total_units) {
      const int k0 = (bu.tb + bi) * TILE_KEYS;
      if (tile_needs_bias(bu, k0, a.E)) {
        const uint32_t dst = smem_u32(bring + slot * HB * BIAS_PITCH);
        const int kw = k0 + 16 * warp;
        const float* relu = a.rel + ((size_t)bu.b * a.Hq + bu.h0) * a.E;
        for (int idx = lane; idx < bu.nh * 16; idx += 32) {
          const int r = idx >> 4, kk = idx & 15, k = kw + kk;
          if (k >= bu.lo && k <= bu.p)
            cp_async_4(dst + (uint32_t)((r * BIAS_PITCH + kk) * 4), relu + (size_t)r * a.E + min(bu.p - k, a.E - 1));
        }
      }
      ++bi;
    }
    cp_async_mbar_arrive_noinc(&bfull[slot]);
    ++bpos;
  };
  for (int x = 0; x < BIAS_DIST; ++x) stage_bias();

  while (ucur < total_units) {
    const int unxt = next_unit(ucur + gridDim.x, nxt);
    if (cur.n_my == 0) {  // zero-length sequence: zeros, nothing read
      for (int i = tid; i < cur.nh * D; i += DEC_CONSUMERS * 32)
        out[((size_t)cur.b * a.Hq + cur.h0 + i / D) * D + i % D] = __float2bfloat16(0.f);
      cur = nxt;
      ucur = unxt;
      continue;
    }
    // bucket E - 1 of this thread's heads: the bias of every key at distance >= E - 1
    float clampv[NB][2];
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 8 * j + 2 * cq + e;
        // heads past the unit's last read head h0's bucket instead: never outside rel
        const float ld = __ldg(a.rel + ((size_t)cur.b * a.Hq + cur.h0 + (h < cur.nh ? h : 0)) * a.E + a.E - 1);
        clampv[j][e] = h < cur.nh ? ld : 0.f;
      }
    const int qslot = uc & 1;
    uint32_t qb[NB][KSTEPS][2];  // B fragments of Q^T
    float m_r[NB][2], l_r[NB][2];
    float o[D / 16][NB][4];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      m_r[j][0] = m_r[j][1] = -INFINITY;
      l_r[j][0] = l_r[j][1] = 0.f;
    }
#pragma unroll
    for (int dn = 0; dn < D / 16; ++dn)
#pragma unroll
      for (int j = 0; j < NB; ++j) o[dn][j][0] = o[dn][j][1] = o[dn][j][2] = o[dn][j][3] = 0.f;

    for (int i = 0; i < cur.n_my; ++i, ++n) {
      const int st = n % NSTAGE;
      const bool ok = wait_or_abort(&full[st], (uint32_t)(n / NSTAGE) & 1u, abort_flag, a.err, a.wait_ns) &&
                      wait_or_abort(&bfull[n % BIAS_SLOTS], (uint32_t)(n / BIAS_SLOTS) & 1u, abort_flag, a.err, a.wait_ns);
      if (i == 0) {
        const uint32_t qbase = smem_u32(smem + L_::q + qslot * S::QSLOT_BYTES);
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          const bool hv = ok && 8 * j + gq < cur.nh;
#pragma unroll
          for (int kk = 0; kk < KSTEPS; kk += 2) {
            const int row = 8 * j + (lane & 7);
            const int chunk = 2 * kk + mi;
            uint32_t r0, r1, r2, r3;
            ldmatrix_x4(qbase + (chunk >> 3) * S::QSUB_BYTES + swz128(row, chunk & 7), r0, r1, r2, r3);
            qb[j][kk][0] = hv ? r0 : 0u;
            qb[j][kk][1] = hv ? r1 : 0u;
            qb[j][kk + 1][0] = hv ? r2 : 0u;
            qb[j][kk + 1][1] = hv ? r3 : 0u;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&qempty[qslot]);
      }
      const int kw = (cur.tb + i) * TILE_KEYS + 16 * warp;
      const uint64_t bad = ok ? badmask[st] : ~0ull;
      // keys kw + j (j < 16) with lo <= key <= p, minus keys of unreadable pages
      const int jlo = max(cur.lo - kw, 0), jhi = min(cur.p - kw, 15);
      uint32_t valid16 = jhi >= jlo ? ((0xFFFFu >> (15 - jhi)) & (0xFFFFu << jlo)) : 0u;
      valid16 &= ~(uint32_t)(bad >> (16 * warp)) & 0xFFFFu;
      if (valid16 != 0) {
        const uint32_t kbase = smem_u32(smem + L_::stages + (size_t)st * S::STAGE_BYTES);
        const uint32_t vbase = kbase + S::TILE_BYTES;
        float acc[NB][4];
#pragma unroll
        for (int j = 0; j < NB; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
          const int krow = 16 * warp + (mi & 1) * 8 + (lane & 7);
          const int chunk = 2 * kk + (mi >> 1);
          uint32_t ka[4];
          ldmatrix_x4(kbase + warp * S::GROUP_BYTES + (chunk >> 3) * S::BLOCK_BYTES + swz128(krow & 15, chunk & 7),
                      ka[0], ka[1], ka[2], ka[3]);
#pragma unroll
          for (int j = 0; j < NB; ++j) mma_bf16_16816(acc[j], ka, qb[j][kk][0], qb[j][kk][1]);
        }
        // V fragments (A operand of O^T = V^T P^T) into registers, masked keys zeroed;
        // then the stage goes back to the producer before the softmax and PV run
        const bool all_valid = valid16 == 0xFFFFu;
        const uint32_t mlo = pair_mask((valid16 >> (2 * cq)) & 1u, (valid16 >> (2 * cq + 1)) & 1u);
        const uint32_t mhi = pair_mask((valid16 >> (8 + 2 * cq)) & 1u, (valid16 >> (9 + 2 * cq)) & 1u);
        uint32_t va[D / 16][4];
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          const int vrow = 16 * warp + (mi >> 1) * 8 + (lane & 7);
          const int chunk = 2 * dn + (mi & 1);
          ldmatrix_x4_trans(vbase + warp * S::GROUP_BYTES + (chunk >> 3) * S::BLOCK_BYTES + swz128(vrow & 15, chunk & 7),
                            va[dn][0], va[dn][1],
                            va[dn][2], va[dn][3]);
          if (!all_valid) { va[dn][0] &= mlo; va[dn][1] &= mlo; va[dn][2] &= mhi; va[dn][3] &= mhi; }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        const bool v0 = (valid16 >> gq) & 1u, v1 = (valid16 >> (gq + 8)) & 1u;
        // bias: this warp's staged rows [head][key], or the clamped bucket
        float bias[NB][4];
        if (tile_needs_bias(cur, (cur.tb + i) * TILE_KEYS, a.E)) {
          const float* bsm = bring + (n % BIAS_SLOTS) * HB * BIAS_PITCH + gq;
#pragma unroll
          for (int j = 0; j < NB; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const bool hv = 8 * j + 2 * cq + e < cur.nh;  // rows past nh are never staged
              const float* br = bsm + (8 * j + 2 * cq + e) * BIAS_PITCH;
              bias[j][e] = hv ? br[0] : 0.f;
              bias[j][2 + e] = hv ? br[8] : 0.f;
            }
        } else {
#pragma unroll
          for (int j = 0; j < NB; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) bias[j][e] = bias[j][2 + e] = clampv[j][e];
        }
        uint32_t pb0[NB], pb1[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          // Scores in base 2.  The running max m_r moves only when a score passes it by more than
          // 8 (so p = 2^(s - m_r) < 256): most tiles skip the cross-lane max and the rescale of O.
          float sv[2][2];
          bool up = false;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            sv[e][0] = v0 ? fmaf(acc[j][e], a.scale_log2, bias[j][e] * LOG2E) : -INFINITY;
            sv[e][1] = v1 ? fmaf(acc[j][2 + e], a.scale_log2, bias[j][2 + e] * LOG2E) : -INFINITY;
            up |= fmaxf(sv[e][0], sv[e][1]) > m_r[j][e] + 8.f;
          }
          if (__any_sync(0xffffffffu, up)) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float mx = fmaxf(sv[e][0], sv[e][1]);
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
              const float mn = fmaxf(m_r[j][e], mx);   // the same in the 8 lanes of this head
              if (mn > m_r[j][e]) {
                const float al = fast_exp2(m_r[j][e] - mn);
                m_r[j][e] = mn;
                l_r[j][e] *= al;
#pragma unroll
                for (int dn = 0; dn < D / 16; ++dn) {
                  o[dn][j][e] *= al;
                  o[dn][j][2 + e] *= al;
                }
              }
            }
          }
          float pr[4];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float mu = m_r[j][e] == -INFINITY ? 0.f : m_r[j][e];
            pr[e] = fast_exp2(sv[e][0] - mu);
            pr[2 + e] = fast_exp2(sv[e][1] - mu);
            l_r[j][e] += pr[e] + pr[2 + e];
          }
          // P^T into the B-fragment layout: thread (g, c) needs keys 2c, 2c+1 (and +8) of head g
          const uint32_t X = pack_bf16(pr[0], pr[1]);  // key gq,   heads 2cq, 2cq+1
          const uint32_t Y = pack_bf16(pr[2], pr[3]);  // key gq+8, heads 2cq, 2cq+1
          const int src0 = 8 * cq + (gq >> 1), src1 = src0 + 4;
          const uint32_t x0 = __shfl_sync(0xffffffffu, X, src0), x1 = __shfl_sync(0xffffffffu, X, src1);
          const uint32_t y0 = __shfl_sync(0xffffffffu, Y, src0), y1 = __shfl_sync(0xffffffffu, Y, src1);
          const uint32_t sel = (gq & 1) ? 0x7632u : 0x5410u;
          pb0[j] = __byte_perm(x0, x1, sel);
          pb1[j] = __byte_perm(y0, y1, sel);
        }
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn)
#pragma unroll
          for (int j = 0; j < NB; ++j) mma_bf16_16816(o[dn][j], va[dn], pb0[j], pb1[j]);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      stage_bias();  // position n + BIAS_DIST reuses the slot just read
    }
    ++uc;

    // ---- unit epilogue: merge the 4 warps' partial softmax states
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float l = l_r[j][e];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        l_r[j][e] = l;
        if (gq == 0) {
          red_m[warp * 16 + 8 * j + 2 * cq + e] = m_r[j][e];
          red_l[warp * 16 + 8 * j + 2 * cq + e] = l;
        }
      }
    named_barrier_consumers();
    // Each thread weighs its own heads' O rows: 2^(m_w - M) over the unit's sum (the sum
    // alone when the unit is one split of several); then the 4 warps' rows are added,
    // 4 channels per thread.
    const bool single = cur.nact == 1;
#pragma unroll
    for (int j = 0; j < NB; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 8 * j + 2 * cq + e;
        if (h >= cur.nh) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < DEC_CONSUMERS; ++w) M = fmaxf(M, red_m[w * 16 + h]);
        const float Mu = M == -INFINITY ? 0.f : M;
        float Lt = 0.f;
#pragma unroll
        for (int w = 0; w < DEC_CONSUMERS; ++w) Lt += red_l[w * 16 + h] * fast_exp2(red_m[w * 16 + h] - Mu);
        float f = fast_exp2(m_r[j][e] - Mu);
        if (single) f *= Lt > 0.f ? 1.f / Lt : 0.f;
        if (warp == 0 && gq == 0) {
          head_ml[2 * h] = M;
          head_ml[2 * h + 1] = Lt;
        }
        float* row = obuf + (warp * HB + h) * S::OPITCH;
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          row[16 * dn + gq] = o[dn][j][e] * f;
          row[16 * dn + gq + 8] = o[dn][j][2 + e] * f;
        }
      }
    named_barrier_consumers();
    const size_t rowbase = (size_t)cur.b * a.Hq + cur.h0;
    for (int idx = tid; idx < cur.nh * (D / 4); idx += DEC_CONSUMERS * 32) {
      const int r = idx / (D / 4), d = (idx % (D / 4)) * 4;
      float4 acc = *reinterpret_cast<const float4*>(obuf + r * S::OPITCH + d);
#pragma unroll
      for (int w = 1; w < DEC_CONSUMERS; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(obuf + (w * HB + r) * S::OPITCH + d);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      if (single) {
        *reinterpret_cast<uint2*>(out + (rowbase + r) * D + d) = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
      } else {
        const size_t pi = (rowbase + r) * a.num_splits + cur.s;
        *reinterpret_cast<float4*>(a.part_o + pi * D + d) = acc;
        if (d == 0) {
          a.part_ml[pi * 2 + 0] = head_ml[2 * r];
          a.part_ml[pi * 2 + 1] = head_ml[2 * r + 1];
        }
      }
    }
    if (!single)
      finish_split_unit<D>(a.part_o, a.part_ml, a.tickets, out, a.Hq, a.Hkv, a.head_chunks, a.num_splits, cur.b,
                           cur.kvh, cur.hc, cur.h0, cur.nh, cur.nact, tid, flags, wts, reinterpret_cast<float2*>(obuf));
    named_barrier_consumers();  // red/obuf/wts/flags are reused by the next unit
    cur = nxt;
    ucur = unxt;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

}  // namespace

int current_device_sms(int* dev_out) {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  *dev_out = dev;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

namespace {

int num_sms() {
  int dev = 0;
  const int n = current_device_sms(&dev);
  return n > 0 ? n : 148;
}

template <int D, int NSTAGE, int HB>
cudaError_t launch_decode_t(const DecodeMaps& m, const DecodeArgs& a, cudaStream_t stream) {
  constexpr size_t smem = DecSmem<D, NSTAGE, HB>::alloc;
  constexpr int ctas = dec_ctas_per_sm<HB>();
  static_assert(smem * ctas <= 228 * 1024 - ctas * 1024, "shared memory budget");
  static std::atomic<unsigned long long> opted{0};
  cudaError_t e = smem_opt_in_once(decode_persistent_kernel<D, NSTAGE, HB>, (int)smem, opted);
  if (e != cudaSuccess) return e;
  const long long units = (long long)a.num_splits * a.B * a.Hkv * a.head_chunks;
  const int grid = (int)std::min<long long>(units, (long long)dec_ctas_per_sm<HB>() * num_sms());
  decode_persistent_kernel<D, NSTAGE, HB><<<grid, DEC_THREADS, smem, stream>>>(
      m.k_seg, m.v_seg, m.k_tile, m.v_tile, m.k_grp, m.v_grp, m.q3, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeMaps& m, const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  const bool narrow = a.G <= 8;  // one 8-wide column block of query heads per unit
  if (head_dim == 128)
    return narrow ? launch_decode_t<128, 2, 8>(m, a, stream) : launch_decode_t<128, 4, 16>(m, a, stream);
  return narrow ? launch_decode_t<64, 4, 8>(m, a, stream) : launch_decode_t<64, 8, 16>(m, a, stream);
}

}  // namespace ink
