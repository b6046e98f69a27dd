// decode.cu -- split-K flash-decode over a paged K/V cache with a per-token
// relative-position bias ("Support Inkling-NVFP4 model", TensorRT-LLM PR #17062,
// sections "Architecture" and "Implementation": one new token per request attends to
// its paged history, bias added before the softmax).
//
// Grid: (split, KV head x head-chunk, sequence).  One CTA owns up to 16 query heads
// that share one KV head (GQA, query head h reads KV head h / G) and a contiguous run
// of 64-key tiles of one sequence.  Per tile:
//   * thread 0 reads the block-table entries (positional: page of key k is
//     block_table[b][k / P]) and issues 2-D TMA loads of the K and V rows into a ring
//     of NSTAGE shared-memory stages (128-byte swizzle, completion on an mbarrier);
//   * each of the 4 warps takes 16 keys: S = Q K^T with mma.sync (query heads are the
//     16 MMA rows), scale, add the gathered bias rel[b, h, min(p - k, E - 1)], mask
//     keys outside [lo, p] (window) or in unreadable pages, online softmax in base 2;
//     O += P V with mma.sync, V rows of masked keys zeroed in registers.
// The 4 warps' (max, sum, O) are merged in shared memory.  A sequence that needs more
// than one split writes fp32 partials to the workspace; the last CTA of that sequence
// to finish (atomic ticket, no spinning) merges the partials in split order, so the
// result does not depend on which CTA finishes last, and resets the ticket to 0.
#include "common.cuh"
#include "kernels.h"

namespace ink {

namespace {

constexpr int DEC_WARPS = 4;
constexpr int DEC_THREADS = DEC_WARPS * 32;

template <int D>
struct DecodeShape {
  static constexpr int COL_BLOCKS = D / 64;               // 128-byte column blocks
  static constexpr int SUB_BYTES = TILE_KEYS * 128;       // one column block of a tile
  static constexpr int TILE_BYTES = COL_BLOCKS * SUB_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;      // K tile + V tile
  static constexpr int OPITCH = D + 4;                    // fp32 merge buffer row pitch
};

template <int D, int NSTAGE>
constexpr size_t decode_smem_bytes() {
  using S = DecodeShape<D>;
  return 1024 /* alignment slack */ + (size_t)NSTAGE * S::STAGE_BYTES +
         NSTAGE * 16 /* barriers + masks */ + 2 * DEC_WARPS * 16 * 4 +
         16 * MAX_DECODE_SPLITS * 4 + 16;
}

template <int D, int NSTAGE>
__global__ void __launch_bounds__(DEC_THREADS, 2)
decode_splitk_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const DecodeArgs a) {
  using S = DecodeShape<D>;
  static_assert(NSTAGE >= 2, "merge buffer reuses two stages");
  static_assert(DEC_WARPS * 16 * S::OPITCH * 4 <= NSTAGE * S::STAGE_BYTES, "merge buffer");
  constexpr int KSTEPS = D / 16;
  constexpr int DBLK = D / 8;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSTAGE * S::STAGE_BYTES);
  uint64_t* badmask = full + NSTAGE;
  float* red_m = reinterpret_cast<float*>(badmask + NSTAGE);
  float* red_l = red_m + DEC_WARPS * 16;
  float* wts = red_l + DEC_WARPS * 16;
  int* flags = reinterpret_cast<int*>(wts + 16 * MAX_DECODE_SPLITS);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3;  // mma fragment row / column-pair
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / a.head_chunks, hc = blockIdx.y % a.head_chunks;
  const int b = blockIdx.z;
  const int h0 = kvh * a.G + hc * 16;
  const int nh = min(16, a.G - hc * 16);
  const int P = 1 << a.log2_page;

  int L = a.seq_lens[b];
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
  if (L <= 0) {  // padding row: zeros, nothing read
    if (split == 0)
      for (int i = tid; i < nh * D; i += DEC_THREADS)
        out[((size_t)b * a.Hq + h0 + i / D) * D + i % D] = __float2bfloat16(0.f);
    return;
  }
  const long long cap = (long long)a.max_pages * P;
  if (L > cap) {  // history longer than the table row: use what the table covers
    if (split == 0 && blockIdx.y == 0 && tid == 0) record_error(a.err, INK_DEVERR_PAGE_OUT_OF_RANGE);
    L = (int)cap;
  }
  const int p = L - 1;
  const int lo = a.W > 0 ? max(0, p - a.W + 1) : 0;
  const int t_first = lo / TILE_KEYS, t_last = p / TILE_KEYS;
  const int ntiles = t_last - t_first + 1;
  const int nact = min((ntiles + a.tiles_per_split - 1) / a.tiles_per_split, a.num_splits);
  if (split >= nact) return;
  const int tb = t_first + split * a.tiles_per_split;
  const int n_my = (split == nact - 1) ? (t_last + 1 - tb) : a.tiles_per_split;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    flags[0] = 0;
    flags[1] = 0;
  }
  __syncthreads();

  // Producer: block-table walk + TMA for tile index i (relative to tb) into stage s.
  auto issue = [&](int i, int s) {
    const int k0 = (tb + i) * TILE_KEYS;
    uint8_t* kdst = smem + s * S::STAGE_BYTES;
    uint8_t* vdst = kdst + S::TILE_BYTES;
    const int32_t* bt = a.block_table + (size_t)b * a.max_pages;
    uint64_t bad = 0;
    uint32_t bytes = 0;
    const int seg_keys = P < TILE_KEYS ? P : TILE_KEYS;
    const int nseg = TILE_KEYS / seg_keys;
    int rows[TILE_KEYS / 8];
    for (int sg = 0; sg < nseg; ++sg) {
      const int ks = k0 + sg * seg_keys;
      rows[sg] = -1;
      if (ks > p || ks + seg_keys - 1 < lo) continue;  // no visible key in this segment
      const int pidx = ks >> a.log2_page;
      const int page = bt[pidx];
      if (page < 0 || page >= a.num_pages) {
        bad |= (seg_keys == 64 ? ~0ull : (((1ull << seg_keys) - 1) << (sg * seg_keys)));
        record_error(a.err, INK_DEVERR_PAGE_OUT_OF_RANGE);
        continue;
      }
      rows[sg] = ((page * a.Hkv + kvh) << a.log2_page) + (ks & (P - 1));
      bytes += 2u * seg_keys * D * 2u;
    }
    badmask[s] = bad;
    mbar_arrive_expect_tx(&full[s], bytes);
    for (int sg = 0; sg < nseg; ++sg) {
      if (rows[sg] < 0) continue;
#pragma unroll
      for (int cb = 0; cb < S::COL_BLOCKS; ++cb) {
        tma_load_2d(kdst + cb * S::SUB_BYTES + sg * seg_keys * 128, &tmK, cb * 64, rows[sg], &full[s]);
        tma_load_2d(vdst + cb * S::SUB_BYTES + sg * seg_keys * 128, &tmV, cb * 64, rows[sg], &full[s]);
      }
    }
  };

  if (tid == 0)
    for (int i = 0; i < min(NSTAGE, n_my); ++i) issue(i, i);

  // Q fragments (A operand, 16 heads x D), loaded once.
  const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(a.q) + ((size_t)b * a.Hq + h0) * D;
  uint32_t qa[KSTEPS][4];
#pragma unroll
  for (int kk = 0; kk < KSTEPS; ++kk) {
    const int c0 = kk * 16 + 2 * cq;
    qa[kk][0] = gq < nh ? *reinterpret_cast<const uint32_t*>(qb + gq * D + c0) : 0u;
    qa[kk][1] = gq + 8 < nh ? *reinterpret_cast<const uint32_t*>(qb + (gq + 8) * D + c0) : 0u;
    qa[kk][2] = gq < nh ? *reinterpret_cast<const uint32_t*>(qb + gq * D + c0 + 8) : 0u;
    qa[kk][3] = gq + 8 < nh ? *reinterpret_cast<const uint32_t*>(qb + (gq + 8) * D + c0 + 8) : 0u;
  }
  const float* rel0 = a.rel + ((size_t)b * a.Hq + h0 + gq) * a.E;
  const float* rel1 = rel0 + (size_t)8 * a.E;
  const bool row0 = gq < nh, row1 = gq + 8 < nh;

  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  float o[DBLK][4];
#pragma unroll
  for (int n = 0; n < DBLK; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

  bool timed_out = false;
  for (int i = 0; i < n_my; ++i) {
    const int s = i % NSTAGE;
    const uint32_t par = (uint32_t)(i / NSTAGE) & 1u;
    const int kw = (tb + i) * TILE_KEYS + 16 * warp;  // this warp's first key

    // bias gather for this warp's 4 keys per thread, issued before the wait
    float bias[2][2][2];
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int k = kw + 8 * nb + 2 * cq + e;
        const bool vis = k >= lo && k <= p;
        const int d = min(p - k, a.E - 1);
        bias[nb][e][0] = (vis && row0) ? __ldg(rel0 + d) : 0.f;
        bias[nb][e][1] = (vis && row1) ? __ldg(rel1 + d) : 0.f;
      }

    if (!mbar_wait_bounded(&full[s], par)) {
      timed_out = true;
      record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
      flags[1] = 1;
    }
    const uint64_t bad = badmask[s];
    uint32_t valid16 = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int k = kw + j;
      const bool ok = k >= lo && k <= p && !((bad >> (16 * warp + j)) & 1ull);
      valid16 |= (ok ? 1u : 0u) << j;
    }
    if (!timed_out && valid16 != 0) {
      const uint32_t kbase = smem_u32(smem + s * S::STAGE_BYTES);
      const uint32_t vbase = kbase + S::TILE_BYTES;
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const int mi = lane >> 3;
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        const int krow = 16 * warp + (mi >> 1) * 8 + (lane & 7);
        const int chunk = 2 * kk + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(kbase + (chunk >> 3) * S::SUB_BYTES + swz128(krow, chunk & 7), b0, b1, b2, b3);
        mma_bf16_16816(sacc[0], qa[kk], b0, b1);
        mma_bf16_16816(sacc[1], qa[kk], b2, b3);
      }
      // scores in log2 units, masked keys -> -inf
      float sc[2][4];
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool ok = (valid16 >> (8 * nb + 2 * cq + e)) & 1u;
          sc[nb][e] = ok ? fmaf(sacc[nb][e], a.scale_log2, bias[nb][e][0] * LOG2E) : -INFINITY;
          sc[nb][2 + e] = ok ? fmaf(sacc[nb][2 + e], a.scale_log2, bias[nb][e][1] * LOG2E) : -INFINITY;
        }
      float mx0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      float mx1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m_r[0], mx0), mn1 = fmaxf(m_r[1], mx1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = fast_exp2(m_r[0] - mu0), al1 = fast_exp2(m_r[1] - mu1);
      m_r[0] = mn0;
      m_r[1] = mn1;
      float pr[2][4];
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int nb = 0; nb < 2; ++nb) {
        pr[nb][0] = fast_exp2(sc[nb][0] - mu0);
        pr[nb][1] = fast_exp2(sc[nb][1] - mu0);
        pr[nb][2] = fast_exp2(sc[nb][2] - mu1);
        pr[nb][3] = fast_exp2(sc[nb][3] - mu1);
        rs0 += pr[nb][0] + pr[nb][1];
        rs1 += pr[nb][2] + pr[nb][3];
      }
      l_r[0] = l_r[0] * al0 + rs0;
      l_r[1] = l_r[1] * al1 + rs1;
#pragma unroll
      for (int n = 0; n < DBLK; ++n) {
        o[n][0] *= al0; o[n][1] *= al0;
        o[n][2] *= al1; o[n][3] *= al1;
      }
      uint32_t pa[4];
      pa[0] = pack_bf16(pr[0][0], pr[0][1]);
      pa[1] = pack_bf16(pr[0][2], pr[0][3]);
      pa[2] = pack_bf16(pr[1][0], pr[1][1]);
      pa[3] = pack_bf16(pr[1][2], pr[1][3]);
      const bool all_valid = valid16 == 0xFFFFu;
      const uint32_t mlo = pair_mask((valid16 >> (2 * cq)) & 1u, (valid16 >> (2 * cq + 1)) & 1u);
      const uint32_t mhi = pair_mask((valid16 >> (8 + 2 * cq)) & 1u, (valid16 >> (9 + 2 * cq)) & 1u);
#pragma unroll
      for (int dn = 0; dn < D / 16; ++dn) {
        const int vrow = 16 * warp + (mi & 1) * 8 + (lane & 7);
        const int chunk = 2 * dn + (mi >> 1);
        uint32_t v0, v1, v2, v3;
        ldmatrix_x4_trans(vbase + (chunk >> 3) * S::SUB_BYTES + swz128(vrow, chunk & 7), v0, v1, v2, v3);
        if (!all_valid) { v0 &= mlo; v1 &= mhi; v2 &= mlo; v3 &= mhi; }
        mma_bf16_16816(o[2 * dn], pa, v0, v1);
        mma_bf16_16816(o[2 * dn + 1], pa, v2, v3);
      }
    }
    __syncthreads();  // every warp is done with stage s
    if (tid == 0 && !flags[1] && i + NSTAGE < n_my) issue(i + NSTAGE, s);
  }
  if (flags[1] && tid == 0) {
    // a copy never completed: give the outstanding ones one more bounded wait
    for (int i = max(0, n_my - NSTAGE); i < n_my; ++i)
      (void)mbar_wait_bounded(&full[i % NSTAGE], (uint32_t)(i / NSTAGE) & 1u);
  }

  // ---- merge the 4 warps' partial softmax states
  l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], 1);
  l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], 2);
  l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], 1);
  l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], 2);
  if (cq == 0) {
    red_m[warp * 16 + gq] = m_r[0];
    red_m[warp * 16 + gq + 8] = m_r[1];
    red_l[warp * 16 + gq] = l_r[0];
    red_l[warp * 16 + gq + 8] = l_r[1];
  }
  __syncthreads();
  float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
  for (int w = 0; w < DEC_WARPS; ++w) {
    M0 = fmaxf(M0, red_m[w * 16 + gq]);
    M1 = fmaxf(M1, red_m[w * 16 + gq + 8]);
  }
  const float f0 = fast_exp2(m_r[0] - (M0 == -INFINITY ? 0.f : M0));
  const float f1 = fast_exp2(m_r[1] - (M1 == -INFINITY ? 0.f : M1));
  float* obuf = reinterpret_cast<float*>(smem);
#pragma unroll
  for (int n = 0; n < DBLK; ++n) {
    const int col = 8 * n + 2 * cq;
    float* r0p = obuf + (warp * 16 + gq) * S::OPITCH + col;
    float* r1p = obuf + (warp * 16 + gq + 8) * S::OPITCH + col;
    r0p[0] = o[n][0] * f0; r0p[1] = o[n][1] * f0;
    r1p[0] = o[n][2] * f1; r1p[1] = o[n][3] * f1;
  }
  __syncthreads();

  const bool single = nact == 1;
  const size_t rowbase = (size_t)b * a.Hq + h0;
  for (int idx = tid; idx < nh * D; idx += DEC_THREADS) {
    const int r = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) M = fmaxf(M, red_m[w * 16 + r]);
    const float Mu = M == -INFINITY ? 0.f : M;
    float acc = 0.f, Lt = 0.f;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) {
      acc += obuf[(w * 16 + r) * S::OPITCH + d];
      Lt += red_l[w * 16 + r] * fast_exp2(red_m[w * 16 + r] - Mu);
    }
    if (single) {
      out[(rowbase + r) * D + d] = __float2bfloat16(Lt > 0.f ? acc / Lt : 0.f);
    } else {
      const size_t pi = (rowbase + r) * a.num_splits + split;
      a.part_o[pi * D + d] = acc;
      if (d == 0) {
        a.part_ml[pi * 2 + 0] = M;
        a.part_ml[pi * 2 + 1] = Lt;
      }
    }
  }
  if (single) return;

  // ---- split-K ticket: the last CTA of this (sequence, head chunk) merges
  __threadfence();
  __syncthreads();
  const size_t ticket = (size_t)b * gridDim.y + blockIdx.y;
  if (tid == 0) flags[0] = (atomicAdd(&a.tickets[ticket], 1) == nact - 1);
  __syncthreads();
  if (!flags[0]) return;
  __threadfence();
  if (tid < nh) {
    const size_t pi0 = (rowbase + tid) * a.num_splits;
    float M = -INFINITY;
    for (int sp = 0; sp < nact; ++sp) M = fmaxf(M, __ldcg(a.part_ml + (pi0 + sp) * 2));
    const float Mu = M == -INFINITY ? 0.f : M;
    float Lt = 0.f;
    for (int sp = 0; sp < nact; ++sp)
      Lt += __ldcg(a.part_ml + (pi0 + sp) * 2 + 1) * fast_exp2(__ldcg(a.part_ml + (pi0 + sp) * 2) - Mu);
    const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
    for (int sp = 0; sp < nact; ++sp)
      wts[tid * MAX_DECODE_SPLITS + sp] = fast_exp2(__ldcg(a.part_ml + (pi0 + sp) * 2) - Mu) * inv;
  }
  __syncthreads();
  for (int idx = tid; idx < nh * D; idx += DEC_THREADS) {
    const int r = idx / D, d = idx % D;
    const size_t pi0 = (rowbase + r) * a.num_splits;
    float acc = 0.f;
    for (int sp = 0; sp < nact; ++sp)
      acc += wts[r * MAX_DECODE_SPLITS + sp] * __ldcg(a.part_o + (pi0 + sp) * D + d);
    out[(rowbase + r) * D + d] = __float2bfloat16(acc);
  }
  if (tid == 0) a.tickets[ticket] = 0;  // ready for the next call
}

template <int D, int NSTAGE>
cudaError_t launch_decode_t(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeArgs& a,
                            cudaStream_t stream) {
  constexpr size_t smem = decode_smem_bytes<D, NSTAGE>();
  cudaError_t e = cudaFuncSetAttribute(decode_splitk_kernel<D, NSTAGE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_splits, a.Hkv * a.head_chunks, a.B);
  decode_splitk_kernel<D, NSTAGE><<<grid, DEC_THREADS, smem, stream>>>(tmK, tmV, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const CUtensorMap& tmK, const CUtensorMap& tmV, const DecodeArgs& a,
                          int head_dim, cudaStream_t stream) {
  if (head_dim == 128) return launch_decode_t<128, 3>(tmK, tmV, a, stream);
  return launch_decode_t<64, 4>(tmK, tmV, a, stream);
}

}  // namespace ink
