// prefill_mma.cu -- paged prefill with the relative bias fused into the score tile,
// warp-level tensor cores (mma.sync bf16).  Used for head_dim 64 and as the baseline
// the tcgen05 prefill kernel is measured against.
//
// "Support Inkling-NVFP4 model" (TensorRT-LLM PR #17062), "Architecture": the bias
// rel[t, h, distance] is added before the softmax; local layers see a 512-key window,
// global layers are full causal.  New tokens are the last n_b positions of the
// sequence's history, read through the positional block table
// ("Inkling attn backend cleanup fake registry", TensorRT-LLM PR #17860).
//
// Grid: (query head, sequence, query tile) with the query-tile index reversed so the
// longest causal rows start first.  A CTA owns 64 query rows of one head (4 warps x
// 16 rows) and walks the 64-key tiles that intersect their visible band.  Per tile:
// thread 0 issues the K/V TMA loads; all threads stage the tile's bias values into
// shared memory with 4-byte cp.async (a skewed gather: row r needs
// rel[t_r, h, p_r - k0 - 63 .. p_r - k0], clamped at E - 1), completion counted on the
// same mbarrier.  Each warp computes S = Q K^T (16 x 64), adds bias, masks, runs the
// online softmax in base 2, and accumulates O += P V.
#include "common.cuh"
#include "kernels.h"

namespace ink {

namespace {

constexpr int PF_WARPS = 4;
constexpr int PF_THREADS = PF_WARPS * 32;
constexpr int PF_ROWS = 64;
constexpr int BIAS_PITCH = 72;  // floats per staged bias row

template <int D>
struct PrefillShape {
  static constexpr int COL_BLOCKS = D / 64;
  static constexpr int SUB_BYTES = TILE_KEYS * 128;
  static constexpr int TILE_BYTES = COL_BLOCKS * SUB_BYTES;
  static constexpr int BIAS_BYTES = PF_ROWS * BIAS_PITCH * 4;  // 18 KB, 1024-multiple
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES + BIAS_BYTES;
};

template <int D, int NSTAGE>
constexpr size_t prefill_smem_bytes() {
  return 1024 + (size_t)NSTAGE * PrefillShape<D>::STAGE_BYTES + NSTAGE * 16 + 16;
}

template <int D, int NSTAGE>
__global__ void __launch_bounds__(PF_THREADS, 2)
prefill_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillArgs a) {
  using S = PrefillShape<D>;
  constexpr int KSTEPS = D / 16;
  constexpr int DBLK = D / 8;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NSTAGE * S::STAGE_BYTES);
  uint64_t* badmask = full + NSTAGE;
  int* flags = reinterpret_cast<int*>(badmask + NSTAGE);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3;
  const int h = blockIdx.x, b = blockIdx.y;
  const int qt = gridDim.z - 1 - blockIdx.z;
  const int kvh = h / a.G;
  const int P = 1 << a.log2_page;

  const int cu0 = a.cu_q[b];
  const int n = a.cu_q[b + 1] - cu0;
  int L = a.seq_lens[b];
  if (qt == 0 && h == 0 && tid == 0 && n > a.max_q_len) record_error(a.err, INK_DEVERR_QLEN_EXCEEDS_MAX);
  const int r_begin = qt * PF_ROWS;
  if (r_begin >= n) return;
  const int r_end = min(n, r_begin + PF_ROWS);
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out);
  if (n > L || L <= 0) {  // inconsistent lengths (or padding): zeros
    if (n > L && h == 0 && tid == 0) record_error(a.err, INK_DEVERR_QLEN_EXCEEDS_KV);
    for (int i = tid; i < (r_end - r_begin) * D; i += PF_THREADS)
      out[((size_t)(cu0 + r_begin + i / D) * a.Hq + h) * D + i % D] = __float2bfloat16(0.f);
    return;
  }
  const long long cap = (long long)a.max_pages * P;
  const int pos0 = L - n;  // absolute position of new token 0
  const int p_first = pos0 + r_begin, p_last = pos0 + r_end - 1;
  // keys at or past the table's reach are unreadable: they are masked (error recorded)
  const int k_reach = (int)min((long long)L, cap) - 1;
  if (k_reach < L - 1 && tid == 0 && qt == 0) record_error(a.err, INK_DEVERR_PAGE_OUT_OF_RANGE);
  const int lo_first = a.W > 0 ? max(0, p_first - a.W + 1) : 0;
  const int k_hi = min(p_last, k_reach);
  const int tb = lo_first / TILE_KEYS;
  const int n_my = k_hi >= lo_first ? k_hi / TILE_KEYS - tb + 1 : 0;

  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(&full[s], 1 + PF_THREADS);
    fence_mbar_init();
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    flags[0] = 0;
  }
  __syncthreads();

  // Per-thread row bookkeeping for the bias staging: warp w stages rows 16w..16w+15.
  const float* relh = a.rel + (size_t)h * a.E;
  const size_t rel_row_stride = (size_t)a.Hq * a.E;

  auto issue_kv = [&](int i, int s) {
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
      if (ks > k_hi || ks + seg_keys - 1 < lo_first) continue;
      const int page = bt[ks >> a.log2_page];
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

  // All threads: stage bias[r][kl] = rel[t_r, h, min(p_r - k, E-1)] for visible (r, k).
  auto issue_bias = [&](int i, int s) {
    const int k0 = (tb + i) * TILE_KEYS;
    const uint32_t bdst = smem_u32(smem + s * S::STAGE_BYTES + 2 * S::TILE_BYTES);
#pragma unroll 4
    for (int rr = 0; rr < 16; ++rr) {
      const int r = warp * 16 + rr;
      const int ri = r_begin + r;
      if (ri >= r_end) break;
      const int pr = pos0 + ri;
      const int lor = a.W > 0 ? max(0, pr - a.W + 1) : 0;
      const float* src = relh + (size_t)(cu0 + ri) * rel_row_stride;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int kl = lane + 32 * half;
        const int k = k0 + kl;
        if (k >= lor && k <= pr && k <= k_reach)
          cp_async_4(bdst + (r * BIAS_PITCH + kl) * 4, src + min(pr - k, a.E - 1));
      }
    }
    cp_async_mbar_arrive_noinc(&full[s]);
  };

  for (int i = 0; i < min(NSTAGE, n_my); ++i) {
    if (tid == 0) issue_kv(i, i);
    issue_bias(i, i);
  }

  // Q fragments for this warp's 16 rows
  const int ra = r_begin + warp * 16 + gq, rb = ra + 8;
  const bool va = ra < r_end, vb = rb < r_end;
  const __nv_bfloat16* q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* qra = q + ((size_t)(cu0 + ra) * a.Hq + h) * D;
  const __nv_bfloat16* qrb = q + ((size_t)(cu0 + rb) * a.Hq + h) * D;
  uint32_t qa[KSTEPS][4];
#pragma unroll
  for (int kk = 0; kk < KSTEPS; ++kk) {
    const int c0 = kk * 16 + 2 * cq;
    qa[kk][0] = va ? *reinterpret_cast<const uint32_t*>(qra + c0) : 0u;
    qa[kk][1] = vb ? *reinterpret_cast<const uint32_t*>(qrb + c0) : 0u;
    qa[kk][2] = va ? *reinterpret_cast<const uint32_t*>(qra + c0 + 8) : 0u;
    qa[kk][3] = vb ? *reinterpret_cast<const uint32_t*>(qrb + c0 + 8) : 0u;
  }
  const int pa_ = pos0 + ra, pb_ = pos0 + rb;
  const int loa = a.W > 0 ? max(0, pa_ - a.W + 1) : 0;
  const int lob = a.W > 0 ? max(0, pb_ - a.W + 1) : 0;
  // this warp's visible band: union over its valid rows
  const int wr0 = r_begin + warp * 16;
  const int wr1 = min(r_end, wr0 + 16) - 1;
  const bool warp_live = wr0 < r_end;
  const int wp0 = pos0 + wr0, wp1 = pos0 + wr1;
  const int wlo0 = a.W > 0 ? max(0, wp0 - a.W + 1) : 0;   // smallest lo of the warp
  const int wlo1 = a.W > 0 ? max(0, wp1 - a.W + 1) : 0;   // largest lo of the warp
  const int whi = min(wp1, k_reach);

  float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
  float o[DBLK][4];
#pragma unroll
  for (int nn = 0; nn < DBLK; ++nn) o[nn][0] = o[nn][1] = o[nn][2] = o[nn][3] = 0.f;
  const int mi = lane >> 3;

  for (int i = 0; i < n_my; ++i) {
    const int s = i % NSTAGE;
    const uint32_t par = (uint32_t)(i / NSTAGE) & 1u;
    const int k0 = (tb + i) * TILE_KEYS;
    bool ok_wait = mbar_wait_bounded(&full[s], par);
    if (!ok_wait) {
      record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
      flags[0] = 1;
    }
    const uint64_t bad = badmask[s];
    const bool touches = warp_live && k0 <= whi && k0 + TILE_KEYS - 1 >= wlo0;
    if (ok_wait && touches) {
      const uint32_t kbase = smem_u32(smem + s * S::STAGE_BYTES);
      const uint32_t vbase = kbase + S::TILE_BYTES;
      const float* bsm = reinterpret_cast<const float*>(smem + s * S::STAGE_BYTES + 2 * S::TILE_BYTES);
      float sacc[8][4];
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) sacc[nb][0] = sacc[nb][1] = sacc[nb][2] = sacc[nb][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int krow = np * 16 + (mi >> 1) * 8 + (lane & 7);
          const int chunk = 2 * kk + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kbase + (chunk >> 3) * S::SUB_BYTES + swz128(krow, chunk & 7), b0, b1, b2, b3);
          mma_bf16_16816(sacc[2 * np], qa[kk], b0, b1);
          mma_bf16_16816(sacc[2 * np + 1], qa[kk], b2, b3);
        }
      }
      // a tile is "interior" for this warp when every row sees every key of it
      const bool interior = bad == 0 && k0 >= wlo1 && k0 + TILE_KEYS - 1 <= wp0 &&
                            k0 + TILE_KEYS - 1 <= k_reach && wr1 - wr0 == 15;
      const float* ba = bsm + (warp * 16 + gq) * BIAS_PITCH;
      const float* bb = ba + 8 * BIAS_PITCH;
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nb = 0; nb < 8; ++nb)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kl = 8 * nb + 2 * cq + e;
          const int k = k0 + kl;
          bool oka = true, okb = true;
          if (!interior) {
            const bool kb = !((bad >> kl) & 1ull) && k <= k_reach;
            oka = va && kb && k >= loa && k <= pa_;
            okb = vb && kb && k >= lob && k <= pb_;
          }
          sacc[nb][e] = oka ? fmaf(sacc[nb][e], a.scale_log2, ba[kl] * LOG2E) : -INFINITY;
          sacc[nb][2 + e] = okb ? fmaf(sacc[nb][2 + e], a.scale_log2, bb[kl] * LOG2E) : -INFINITY;
          mx0 = fmaxf(mx0, sacc[nb][e]);
          mx1 = fmaxf(mx1, sacc[nb][2 + e]);
        }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m_r[0], mx0), mn1 = fmaxf(m_r[1], mx1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = fast_exp2(m_r[0] - mu0), al1 = fast_exp2(m_r[1] - mu1);
      m_r[0] = mn0;
      m_r[1] = mn1;
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int nb = 0; nb < 8; ++nb) {
        sacc[nb][0] = fast_exp2(sacc[nb][0] - mu0);
        sacc[nb][1] = fast_exp2(sacc[nb][1] - mu0);
        sacc[nb][2] = fast_exp2(sacc[nb][2] - mu1);
        sacc[nb][3] = fast_exp2(sacc[nb][3] - mu1);
        rs0 += sacc[nb][0] + sacc[nb][1];
        rs1 += sacc[nb][2] + sacc[nb][3];
      }
      l_r[0] = l_r[0] * al0 + rs0;
      l_r[1] = l_r[1] * al1 + rs1;
#pragma unroll
      for (int nn = 0; nn < DBLK; ++nn) {
        o[nn][0] *= al0; o[nn][1] *= al0;
        o[nn][2] *= al1; o[nn][3] *= al1;
      }
      // keys no row of this warp may read get their V rows zeroed (NaN-safe)
      const bool v_clean = bad == 0 && k0 >= wlo0 && k0 + TILE_KEYS - 1 <= whi;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t pa[4];
        pa[0] = pack_bf16(sacc[2 * ks][0], sacc[2 * ks][1]);
        pa[1] = pack_bf16(sacc[2 * ks][2], sacc[2 * ks][3]);
        pa[2] = pack_bf16(sacc[2 * ks + 1][0], sacc[2 * ks + 1][1]);
        pa[3] = pack_bf16(sacc[2 * ks + 1][2], sacc[2 * ks + 1][3]);
        uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
        if (!v_clean) {
          auto kv_ok = [&](int kl) {
            const int k = k0 + kl;
            return !((bad >> kl) & 1ull) && k >= wlo0 && k <= whi;
          };
          const int kb = 16 * ks + 2 * cq;
          mlo = pair_mask(kv_ok(kb), kv_ok(kb + 1));
          mhi = pair_mask(kv_ok(kb + 8), kv_ok(kb + 9));
        }
#pragma unroll
        for (int dn = 0; dn < D / 16; ++dn) {
          const int vrow = 16 * ks + (mi & 1) * 8 + (lane & 7);
          const int chunk = 2 * dn + (mi >> 1);
          uint32_t v0, v1, v2, v3;
          ldmatrix_x4_trans(vbase + (chunk >> 3) * S::SUB_BYTES + swz128(vrow, chunk & 7), v0, v1, v2, v3);
          v0 &= mlo; v1 &= mhi; v2 &= mlo; v3 &= mhi;
          mma_bf16_16816(o[2 * dn], pa, v0, v1);
          mma_bf16_16816(o[2 * dn + 1], pa, v2, v3);
        }
      }
    }
    __syncthreads();
    if (!flags[0] && i + NSTAGE < n_my) {
      if (tid == 0) issue_kv(i + NSTAGE, s);
      issue_bias(i + NSTAGE, s);
    }
  }
  if (flags[0] && tid == 0)
    for (int i = max(0, n_my - NSTAGE); i < n_my; ++i)
      (void)mbar_wait_bounded(&full[i % NSTAGE], (uint32_t)(i / NSTAGE) & 1u);
  asm volatile("cp.async.wait_all;" ::: "memory");

  l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], 1);
  l_r[0] += __shfl_xor_sync(0xffffffffu, l_r[0], 2);
  l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], 1);
  l_r[1] += __shfl_xor_sync(0xffffffffu, l_r[1], 2);
  const float inv0 = l_r[0] > 0.f ? 1.f / l_r[0] : 0.f;
  const float inv1 = l_r[1] > 0.f ? 1.f / l_r[1] : 0.f;
  __nv_bfloat16* oa = out + ((size_t)(cu0 + ra) * a.Hq + h) * D;
  __nv_bfloat16* ob = out + ((size_t)(cu0 + rb) * a.Hq + h) * D;
#pragma unroll
  for (int nn = 0; nn < DBLK; ++nn) {
    const int col = 8 * nn + 2 * cq;
    if (va) *reinterpret_cast<uint32_t*>(oa + col) = pack_bf16(o[nn][0] * inv0, o[nn][1] * inv0);
    if (vb) *reinterpret_cast<uint32_t*>(ob + col) = pack_bf16(o[nn][2] * inv1, o[nn][3] * inv1);
  }
}

template <int D, int NSTAGE>
cudaError_t launch_prefill_t(const CUtensorMap& tmK, const CUtensorMap& tmV, const PrefillArgs& a,
                             cudaStream_t stream) {
  constexpr size_t smem = prefill_smem_bytes<D, NSTAGE>();
  cudaError_t e = cudaFuncSetAttribute(prefill_mma_kernel<D, NSTAGE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.Hq, a.B, a.num_q_tiles);
  prefill_mma_kernel<D, NSTAGE><<<grid, PF_THREADS, smem, stream>>>(tmK, tmV, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& tmK, const CUtensorMap& tmV, const PrefillArgs& a,
                           int head_dim, cudaStream_t stream) {
  if (head_dim == 128) return launch_prefill_t<128, 2>(tmK, tmV, a, stream);
  return launch_prefill_t<64, 3>(tmK, tmV, a, stream);
}

}  // namespace ink
