// kv_conv.cu -- the step before attention: the causal short convolution of the step's K
// and V rows, written into the paged K/V cache, and the convolution state carried to the
// next step.
//
// Operation ("Support Inkling-NVFP4 model", TensorRT-LLM PR #17062, section
// "Architecture"; the state and the in-backend KV write from the commits of "Inkling attn
// backend cleanup fake registry", TensorRT-LLM PR #17860): per channel (g, d) of each of K
// and V, with x the raw projection rows of a request in position order,
//     y[p] = sum_{j < ks} w[g, d, j] * x[p - (ks - 1) + j]
// where the ks - 1 rows before the step's first new token come from the carried state.
// y goes to cache[block_table[b][p / P], g, p % P, :] rounded to bf16; the new state is
// the last ks - 1 raw rows of (state, new rows).
//
// The work is pure streaming: every input row is read once from HBM and every output row
// written once, so it is HBM-bound.  Two kernels do it:
//  - kv_conv_staged_kernel, for steps with at least one tile of K and one of V per SM
//    (prefill): persistent, token tiles bulk-copied into a shared-memory ring (see the
//    comment above it);
//  - kv_conv_write_kernel, for smaller steps (decode): one thread owns one 16-byte vector
//    (8 channels) of either K or V over a run of TOK consecutive tokens (1 or 8).  It loads
//    its TOK rows up front (TOK independent 16-byte loads in flight), keeps the last
//    ks - 1 rows in registers as a sliding window, and reloads the window only where a run
//    starts or crosses into the next request.  Consecutive threads take consecutive vectors
//    of a row, so every load and store of a warp is 512 contiguous bytes of one row (or 256
//    bytes per KV head in the cache).
// In both, extra threads of the same launch copy the carried state: one thread per 16-byte
// vector of a request's state, all KS - 1 rows (loads issued together).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace ink {
namespace {

constexpr int KV_CONV_THREADS = 256;

__device__ __forceinline__ uint4 ld_row16(const uint16_t* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void unpack8(const uint4 r, float (&f)[8]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Index b of the request that owns packed token t: the last b with cu_q[b] <= t.
// Returns -1 when t lies before cu_q[0] or at/after cu_q[B].
__device__ __forceinline__ int find_seq(const int32_t* cu_q, int B, int t) {
  if (B <= 0 || t < __ldg(cu_q) || t >= __ldg(cu_q + B)) return -1;
  int lo = 0, hi = B;   // cu_q[lo] <= t < cu_q[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(cu_q + mid) <= t) lo = mid; else hi = mid;
  }
  return lo;
}

// find_seq over a copy of cu_q in shared memory.
__device__ __forceinline__ int find_seq_shared(const int* cu_q, int B, int t) {
  if (B <= 0 || t < cu_q[0] || t >= cu_q[B]) return -1;
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu_q[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

// Carried state of item sid = (tensor z, request b, vector v): the KS - 1 rows after the step,
// the last KS - 1 rows of [state before; the request's new rows].  All loads are issued
// before the stores.  cu holds cu_q (in shared memory when `cached`, else global).
template <int KS>
__device__ __forceinline__ void copy_state_item(const KvConvArgs& a, long long sid, const int* cu_s, bool cached,
                                                int row_elems) {
  const int v = (int)(sid % a.nvec);
  const long long rest = sid / a.nvec;
  const int b = (int)(rest % a.B);
  const int z = (int)(rest / a.B);
  const int col = v * 8;
  const int seq_start = cached ? cu_s[b] : __ldg(a.cu_q + b);
  const int n = max((cached ? cu_s[b + 1] : __ldg(a.cu_q + b + 1)) - seq_start, 0);
  uint4 rows[KS - 1];
#pragma unroll
  for (int r = 0; r < KS - 1; ++r) {
    rows[r] = make_uint4(0, 0, 0, 0);
    if (r + n < KS - 1) {
      rows[r] = ld_row16(a.st_in[z] + ((size_t)b * (KS - 1) + (r + n)) * row_elems + col);
    } else {
      const int t = seq_start + r + n - (KS - 1);
      if (t >= 0 && t < a.T) rows[r] = ld_row16(a.x[z] + (size_t)t * row_elems + col);
      else record_error(a.err, INK_DEVERR_BAD_ROWS);
    }
  }
#pragma unroll
  for (int r = 0; r < KS - 1; ++r)
    *reinterpret_cast<uint4*>(a.st_out[z] + ((size_t)b * (KS - 1) + r) * row_elems + col) = rows[r];
}

// Requests whose offsets and lengths the per-thread kernel stages in shared memory (one
// parallel load per block instead of a chain of dependent loads per thread).
constexpr int KV_SMALL_CACHED_SEQS = 1023;

template <int KS, int TOK>
__global__ void __launch_bounds__(KV_CONV_THREADS, 2) kv_conv_write_kernel(const KvConvArgs a) {
  const long long gid = (long long)blockIdx.x * KV_CONV_THREADS + threadIdx.x;
  const int row_elems = a.nvec * 8;
  __shared__ int cu_s[KV_SMALL_CACHED_SEQS + 1];
  __shared__ int len_s[KV_SMALL_CACHED_SEQS];
  const bool cached = a.B <= KV_SMALL_CACHED_SEQS;
  const bool conv = gid < a.conv_items;
  // A convolution thread's rows and taps depend on nothing else: their loads go out before
  // the block stages the request offsets, so the two round trips overlap.
  int v = 0, chunk = 0, z = 0;
  if (conv) {
    v = (int)(gid % a.nvec);
    const long long rest = gid / a.nvec;
    chunk = (int)(rest % a.nchunks);
    z = (int)(rest / a.nchunks);                     // 0: K, 1: V
  }
  const uint16_t* __restrict__ x = a.x[z];
  const int col = v * 8;                             // element offset inside a row
  const int g = col / a.D, d = col % a.D;
  const int t0 = chunk * TOK;
  // this run's raw rows, loaded first so that TOK loads are in flight together, and the
  // taps of these 8 channels: w[g, d + e, j] at ((g*D + d + e) * KS + j).  Threads past the
  // convolution items issue no load (T may be 0, and x then points at nothing).
  uint4 raw[TOK];
  float flat[8 * KS];
#pragma unroll
  for (int k = 0; k < TOK; ++k) raw[k] = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int q = 0; q < 8 * KS; ++q) flat[q] = 0.f;
  if (conv) {
#pragma unroll
    for (int k = 0; k < TOK; ++k)
      if (t0 + k < a.T) raw[k] = ld_row16(x + (size_t)(t0 + k) * row_elems + col);
    const float4* wp = reinterpret_cast<const float4*>(a.w[z] + (size_t)(g * a.D + d) * KS);
#pragma unroll
    for (int q = 0; q < 2 * KS; ++q) {
      const float4 f = __ldg(wp + q);
      flat[4 * q] = f.x; flat[4 * q + 1] = f.y; flat[4 * q + 2] = f.z; flat[4 * q + 3] = f.w;
    }
  }
  float w[KS][8];
#pragma unroll
  for (int e = 0; e < 8; ++e)
#pragma unroll
    for (int j = 0; j < KS; ++j) w[j][e] = flat[e * KS + j];
  if (cached) {
    for (int j = threadIdx.x; j <= a.B; j += KV_CONV_THREADS) {
      cu_s[j] = __ldg(a.cu_q + j);
      if (j < a.B) len_s[j] = __ldg(a.seq_lens + j);
    }
  }
  __syncthreads();
  if (conv) {
    // ---------------------------------------------------------------- convolution
    uint16_t* __restrict__ cache = a.cache[z];

    float win[KS > 1 ? KS - 1 : 1][8];   // rows at positions p - (KS-1) .. p - 1
    // The run is cut at request boundaries into segments [k, k_end); each segment loads
    // its request's scalars and window once, then convolves its tokens.
    int k = 0;
    while (k < TOK && t0 + k < a.T) {
      const int t = t0 + k;
      const int b = cached ? find_seq_shared(cu_s, a.B, t) : find_seq(a.cu_q, a.B, t);
      if (b < 0) {                                    // token outside every request
        record_error(a.err, INK_DEVERR_BAD_ROWS);
        ++k;
        continue;
      }
      const int seq_start = cached ? cu_s[b] : __ldg(a.cu_q + b);
      const int seq_end = cached ? cu_s[b + 1] : __ldg(a.cu_q + b + 1);
      const int k_end = min(TOK, seq_end - t0);
      if (seq_start < 0) {                            // request rows named before row 0
        record_error(a.err, INK_DEVERR_BAD_ROWS);
        k = k_end;
        continue;
      }
      const int n = seq_end - seq_start;
      const int L = cached ? len_s[b] : __ldg(a.seq_lens + b);
      const bool seq_ok = n <= L;
      if (!seq_ok) record_error(a.err, INK_DEVERR_QLEN_EXCEEDS_KV);
      const int i0 = t - seq_start;                   // index of token t among the request's new rows
      const int pos_t0 = L - n - seq_start + t0;      // position of run token 0 if it were in b
      const int* bt_row = a.block_table + (size_t)b * a.max_pages;
      // the page of the segment's first token, loaded beside the window rows
      const int pidx0 = (pos_t0 + k) >> a.log2_page;
      const int page0 = seq_ok && pidx0 >= 0 && pidx0 < a.max_pages ? __ldg(bt_row + pidx0) : -1;
#pragma unroll
      for (int m = 0; m < KS - 1; ++m) {
        const int r = i0 - (KS - 1) + m;              // row of the new rows, or of the state if < 0
        const uint16_t* src = r >= 0 ? x + (size_t)(seq_start + r) * row_elems + col
                                     : a.st_in[z] + ((size_t)b * (KS - 1) + (KS - 1 + r)) * row_elems + col;
        unpack8(ld_row16(src), win[m]);
      }
#pragma unroll
      for (int kk = 0; kk < TOK; ++kk) {
        if (kk < k || kk >= k_end) continue;
        float cur[8];
        unpack8(raw[kk], cur);
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float s = 0.f;
#pragma unroll
          for (int j = 0; j < KS - 1; ++j) s = fmaf(w[j][e], win[j][e], s);
          y[e] = fmaf(w[KS - 1][e], cur[e], s);
        }
#pragma unroll
        for (int m = 0; m + 1 < KS - 1; ++m)
#pragma unroll
          for (int e = 0; e < 8; ++e) win[m][e] = win[m + 1][e];
        if constexpr (KS > 1) {
#pragma unroll
          for (int e = 0; e < 8; ++e) win[KS - 2][e] = cur[e];
        }
        if (!seq_ok) continue;
        const int p = pos_t0 + kk;
        const int pidx = p >> a.log2_page;
        const int page = pidx == pidx0 ? page0 : (pidx < a.max_pages ? __ldg(bt_row + pidx) : -1);
        if (page < 0 || page >= a.num_pages) {
          record_error(a.err, INK_DEVERR_PAGE_OUT_OF_RANGE);
          continue;
        }
        const size_t slot = (((size_t)page * a.Hkv + g) << a.log2_page) + (p & ((1 << a.log2_page) - 1));
        *reinterpret_cast<uint4*>(cache + slot * a.D + d) = pack8(y);
      }
      k = k_end;
    }
    return;
  }
  if constexpr (KS > 1) {
    // ---------------------------------------------------------------- carried state
    if (gid < a.conv_items + a.state_items) copy_state_item<KS>(a, gid - a.conv_items, cu_s, cached, row_elems);
  }
}

// One output row of 8 channels: y = sum_j w[j] * (window rows, then the current row), in
// fp32 with one fma per tap; then the current row enters the window.
template <int KS>
__device__ __forceinline__ void conv_step(const float (&w)[KS][8], float (&win)[KS > 1 ? KS - 1 : 1][8],
                                          const uint4 raw, float (&y)[8]) {
  float cur[8];
  unpack8(raw, cur);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < KS - 1; ++j) acc = fmaf(w[j][e], win[j][e], acc);
    y[e] = fmaf(w[KS - 1][e], cur[e], acc);
  }
#pragma unroll
  for (int mm = 0; mm + 1 < KS - 1; ++mm)
#pragma unroll
    for (int e = 0; e < 8; ++e) win[mm][e] = win[mm + 1][e];
  if constexpr (KS > 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) win[KS - 2][e] = cur[e];
  }
}

// ---------------------------------------------------------------------------------------
// Staged kernel for steps with many new rows (prefill).  The step's rows of K (or V) are
// one contiguous array in token order, so a tile of TT consecutive tokens plus the ks - 1
// rows before it is one contiguous run of bytes: a single 1-D bulk async copy brings it
// into shared memory.  One CTA per SM walks the tiles (K and V tiles interleaved) through
// a ring of NS stages.  Each stage has its own producer warp, which issues the copy of a
// tile and then computes the tile's per-token metadata (request, index inside the request,
// destination slot) while the copy is in flight; the request offsets and lengths are held
// in shared memory, so that chain is one block-table load.  Eight consumer warps convolve
// from shared memory and store each 16-byte result straight to its cache slot.

constexpr int KVS_CONSUMER_WARPS = 8;
constexpr int KVS_CONSUMERS = KVS_CONSUMER_WARPS * 32;
constexpr int KVS_MAX_TT = 32;
constexpr int KVS_MAX_STAGES = 4;
constexpr int KVS_THREADS = KVS_CONSUMERS + 32 * KVS_MAX_STAGES;   // one producer warp per stage
constexpr int KVS_MAX_CACHED_SEQS = 2047;   // cu_q / seq_lens held in shared memory up to this B

struct KvsMeta {
  long long slot[KVS_MAX_TT];   // element offset of the token's cache row for head 0, or -1
  int b[KVS_MAX_TT];            // request of the token (-1: none)
  int i[KVS_MAX_TT];            // index of the token among its request's new rows
  uint32_t starts;              // bit r: token r has no earlier row of its request here (i == 0)
  uint32_t pad[31];
};

// Shared memory: barriers and flag (128 B), per-stage metadata, cached cu_q and seq_lens,
// then the stages (128-byte aligned).
constexpr size_t KVS_STAGE_OFFSET =
    (128 + KVS_MAX_STAGES * sizeof(KvsMeta) + (2 * KVS_MAX_CACHED_SEQS + 1) * sizeof(int) + 127) / 128 * 128;

template <int KS>
__global__ void __launch_bounds__(KVS_THREADS, 1) kv_conv_staged_kernel(const KvConvArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);               // [NS]
  uint64_t* empty = full + KVS_MAX_STAGES;                          // [NS]
  int* abort_flag = reinterpret_cast<int*>(empty + KVS_MAX_STAGES);
  KvsMeta* meta = reinterpret_cast<KvsMeta*>(smem + 128);           // [NS]
  int* cu_s = reinterpret_cast<int*>(smem + 128 + KVS_MAX_STAGES * sizeof(KvsMeta));   // [B + 1]
  int* len_s = cu_s + (KVS_MAX_CACHED_SEQS + 1);                                          // [B]
  unsigned char* stage_base = smem + KVS_STAGE_OFFSET;
  const bool cached = a.B <= KVS_MAX_CACHED_SEQS;
  const int NS = a.stages, TT = a.tile_tokens;
  const int row_elems = a.nvec * 8;
  const size_t row_bytes = (size_t)row_elems * 2;
  const size_t stage_bytes = (size_t)(TT + KS - 1) * row_bytes;
  const int ntiles = (a.T + TT - 1) / TT;
  const int units = 2 * ntiles;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 33);
      mbar_init(&empty[s], KVS_CONSUMER_WARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (cached) {
    for (int j = threadIdx.x; j <= a.B; j += KVS_THREADS) {
      cu_s[j] = __ldg(a.cu_q + j);
      if (j < a.B) len_s[j] = __ldg(a.seq_lens + j);
    }
  }
  __syncthreads();

  if (warp >= KVS_CONSUMER_WARPS) {
    // ------------------------------------------------------------ producer warps
    // Producer warp s fills stage s: local units k = s, s + NS, ...  Their metadata
    // chains (request lookup, block-table load) thus run NS at a time.
    const int ps = warp - KVS_CONSUMER_WARPS;
    if (ps >= NS) return;
    int k = ps;
    int issued = 0;
    for (int u = blockIdx.x + ps * gridDim.x; u < units; u += NS * gridDim.x, k += NS) {
      const int s = ps;
      if (k >= NS && !mbar_wait_limit(&empty[s], ((k / NS) - 1) & 1, a.wait_ns)) {
        if (lane == 0) record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
        *reinterpret_cast<volatile int*>(abort_flag) = 1;
        break;
      }
      const int z = u & 1, tile = u >> 1;
      const int t0 = tile * TT;
      const int t_end = min(a.T, t0 + TT);
      const int row0 = max(0, t0 - (KS - 1));
      if (lane == 0) {
        const uint32_t bytes = (uint32_t)((size_t)(t_end - row0) * row_bytes);
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_copy_g2s(smem_u32(stage_base + (size_t)s * stage_bytes), a.x[z] + (size_t)row0 * row_elems, bytes,
                      &full[s]);
      }
      // metadata of token t0 + lane while the copy is in flight
      if (lane < TT) {
        const int t = t0 + lane;
        long long slot = -1;
        int b = -1, i = 0;
        if (t < a.T) {
          b = cached ? find_seq_shared(cu_s, a.B, t) : find_seq(a.cu_q, a.B, t);
          if (b < 0) {
            if (z == 0) record_error(a.err, INK_DEVERR_BAD_ROWS);
          } else {
            const int seq_start = cached ? cu_s[b] : __ldg(a.cu_q + b);
            const int n = (cached ? cu_s[b + 1] : __ldg(a.cu_q + b + 1)) - seq_start;
            const int L = cached ? len_s[b] : __ldg(a.seq_lens + b);
            i = t - seq_start;
            if (seq_start < 0) {
              if (z == 0) record_error(a.err, INK_DEVERR_BAD_ROWS);
              b = -1;
              i = 0;                      // no window rows from the stage for a bad request
            } else if (n > L) {
              if (z == 0) record_error(a.err, INK_DEVERR_QLEN_EXCEEDS_KV);
            } else {
              const int p = L - n + i;
              const int pidx = p >> a.log2_page;
              const int page = pidx < a.max_pages ? __ldg(a.block_table + (size_t)b * a.max_pages + pidx) : -1;
              if (page < 0 || page >= a.num_pages) {
                if (z == 0) record_error(a.err, INK_DEVERR_PAGE_OUT_OF_RANGE);
              } else {
                slot = ((((long long)page * a.Hkv) << a.log2_page) + (p & ((1 << a.log2_page) - 1))) * a.D;
              }
            }
          }
        }
        meta[s].slot[lane] = slot;
        meta[s].b[lane] = b;
        meta[s].i[lane] = i;
      }
      const uint32_t starts = __ballot_sync(0xffffffffu, lane < TT && meta[s].i[lane] == 0);
      if (lane == 0) meta[s].starts = starts;
      mbar_arrive(&full[s]);
      ++issued;
    }
    // drain: wait (bounded) until the last copy into this stage has landed, so none is in
    // flight into shared memory when the CTA exits
    if (lane == 0 && issued > 0) {
      const int last = ps + (issued - 1) * NS;   // local index of this stage's last unit
      if (!mbar_wait_bounded(&full[ps], (last / NS) & 1)) record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
    }
    return;
  }

  // -------------------------------------------------------------- consumer warps
  // carried-state rows first (plain copies, a few per thread)
  if constexpr (KS > 1) {
    for (long long sid = (long long)blockIdx.x * KVS_CONSUMERS + threadIdx.x; sid < a.state_items;
         sid += (long long)gridDim.x * KVS_CONSUMERS)
      copy_state_item<KS>(a, sid, cu_s, cached, row_elems);
  }

  const int nseg = max(1, KVS_CONSUMERS / a.nvec);
  const int seg_len = (TT + nseg - 1) / nseg;
  const int items = a.nvec * nseg;
  // A thread's filter taps stay in registers while its (tensor, vector) pair repeats: with
  // an even grid every tile of a CTA is of the same tensor, and with at most one item per
  // thread every tile gives the thread the same vector.
  float w[KS][8];
  int w_key = -1;
  int k = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x, ++k) {
    const int s = k % NS;
    const bool ok = mbar_wait_limit(&full[s], (k / NS) & 1, a.wait_ns);
    if (!ok || *reinterpret_cast<volatile int*>(abort_flag)) {
      if (!ok) record_error(a.err, INK_DEVERR_WAIT_TIMEOUT);
      break;
    }
    const int z = u & 1, tile = u >> 1;
    const int t0 = tile * TT;
    const int n_tile = min(a.T, t0 + TT) - t0;
    const int row0 = max(0, t0 - (KS - 1));
    const unsigned char* stage = stage_base + (size_t)s * stage_bytes;
    const KvsMeta& m = meta[s];
    uint16_t* __restrict__ cache = a.cache[z];
    const uint64_t starts = m.starts;
    for (int it = threadIdx.x; it < items; it += KVS_CONSUMERS) {
      const int v = it % a.nvec, seg = it / a.nvec;
      const int r0 = seg * seg_len, r1 = min(n_tile, r0 + seg_len);
      if (r0 >= r1) continue;
      const int col = v * 8;
      const int g = col / a.D, d = col % a.D;
      if (w_key != z * a.nvec + v) {
        w_key = z * a.nvec + v;
        const float4* wp = reinterpret_cast<const float4*>(a.w[z] + (size_t)(g * a.D + d) * KS);
        float flat[8 * KS];
#pragma unroll
        for (int q = 0; q < 2 * KS; ++q) {
          const float4 f = __ldg(wp + q);
          flat[4 * q] = f.x; flat[4 * q + 1] = f.y; flat[4 * q + 2] = f.z; flat[4 * q + 3] = f.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e)
#pragma unroll
          for (int jj = 0; jj < KS; ++jj) w[jj][e] = flat[e * KS + jj];
      }
      // stage row of tile token r: col_base + (t0 + r - row0) * row_bytes
      const unsigned char* col_base = stage + (size_t)col * 2 + (size_t)(t0 - row0) * row_bytes;
      uint16_t* cache_col = cache + ((size_t)g << a.log2_page) * a.D + d;
      const uint16_t* st_col = a.st_in[z] + col;
      float win[KS > 1 ? KS - 1 : 1][8];
      {
        // window of token r0: earlier rows of its request from the stage, else state rows
        const int b0 = m.b[r0], i0 = m.i[r0];
#pragma unroll
        for (int mm = 0; mm < KS - 1; ++mm) {
          const int rr = i0 - (KS - 1) + mm;
          uint4 row = make_uint4(0, 0, 0, 0);
          if (rr >= 0)
            row = *reinterpret_cast<const uint4*>(col_base + (ptrdiff_t)(r0 - (KS - 1) + mm) * (ptrdiff_t)row_bytes);
          else if (b0 >= 0)
            row = ld_row16(st_col + ((size_t)b0 * (KS - 1) + (KS - 1 + rr)) * row_elems);
          unpack8(row, win[mm]);
        }
      }
      int r = r0;
      while (r < r1) {
        if (r != r0 && ((starts >> r) & 1)) {
          // first new row of the next request: its window is that request's state
          const int b = m.b[r];
#pragma unroll
          for (int mm = 0; mm < KS - 1; ++mm) {
            uint4 row = make_uint4(0, 0, 0, 0);
            if (b >= 0) row = ld_row16(st_col + ((size_t)b * (KS - 1) + mm) * row_elems);
            unpack8(row, win[mm]);
          }
        }
        if (r + 8 <= r1 && ((starts >> (r + 1)) & 0x7Full) == 0) {
          // eight tokens of one request: unrolled, the window shift is register renaming
          uint4 raw[8];
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            raw[kk] = *reinterpret_cast<const uint4*>(col_base + (size_t)(r + kk) * row_bytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            float y[8];
            conv_step<KS>(w, win, raw[kk], y);
            const long long slot = m.slot[r + kk];
            if (slot >= 0) *reinterpret_cast<uint4*>(cache_col + slot) = pack8(y);
          }
          r += 8;
        } else {
          float y[8];
          conv_step<KS>(w, win, *reinterpret_cast<const uint4*>(col_base + (size_t)r * row_bytes), y);
          const long long slot = m.slot[r];
          if (slot >= 0) *reinterpret_cast<uint4*>(cache_col + slot) = pack8(y);
          ++r;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
}

template <int KS>
cudaError_t launch_ks(const KvConvArgs& a, int tok, cudaStream_t stream) {
  if (a.stages >= 2) {
    static std::atomic<unsigned long long> opted{0};
    const cudaError_t e = smem_opt_in_once(kv_conv_staged_kernel<KS>, KV_STAGED_SMEM_MAX, opted);
    if (e != cudaSuccess) return e;
    const int units = 2 * ((a.T + a.tile_tokens - 1) / a.tile_tokens);
    int dev = 0;
    const int sms = current_device_sms(&dev);
    const int grid = units < sms ? units : sms;
    const size_t smem = kv_staged_smem_bytes(a.tile_tokens, KS, a.nvec, a.stages);
    kv_conv_staged_kernel<KS><<<grid, KVS_THREADS, smem, stream>>>(a);
    return cudaGetLastError();
  }
  const long long items = a.conv_items + a.state_items;
  const unsigned blocks = (unsigned)((items + KV_CONV_THREADS - 1) / KV_CONV_THREADS);
  if (tok == 8) kv_conv_write_kernel<KS, 8><<<blocks, KV_CONV_THREADS, 0, stream>>>(a);
  else kv_conv_write_kernel<KS, 1><<<blocks, KV_CONV_THREADS, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t kv_staged_smem_bytes(int tile_tokens, int kernel_size, int nvec, int stages) {
  return KVS_STAGE_OFFSET + (size_t)stages * (tile_tokens + kernel_size - 1) * (size_t)nvec * 16;
}

void kv_conv_plan(KvConvArgs& a, int kernel_size, int num_sms) {
  // Staged path: tiles of about 32 KB of new rows, up to four stages in KV_STAGED_SMEM_MAX
  // bytes, and enough tiles for every SM; otherwise (few rows, or rows too long for two
  // stages) the one-thread-per-vector kernel.
  const size_t row_bytes = (size_t)a.nvec * 16;
  int tt = (int)(32768 / row_bytes);
  tt = tt < 1 ? 1 : (tt > KVS_MAX_TT ? KVS_MAX_TT : tt);
  int stages = 0;
  while (true) {
    const size_t fixed = kv_staged_smem_bytes(tt, kernel_size, a.nvec, 0);
    const size_t per = kv_staged_smem_bytes(tt, kernel_size, a.nvec, 1) - fixed;
    stages = (int)((KV_STAGED_SMEM_MAX - fixed) / per);
    if (stages >= 2 || tt == 1) break;
    --tt;
  }
  if (stages > KVS_MAX_STAGES) stages = KVS_MAX_STAGES;
  const long long units = 2ll * ((a.T + tt - 1) / tt);
  a.tile_tokens = tt;
  a.stages = (stages >= 2 && units >= num_sms) ? stages : 0;
  a.tok = kv_conv_tokens_per_thread(a.T, a.nvec, num_sms);
  a.nchunks = (a.T + a.tok - 1) / a.tok;
  a.conv_items = 2ll * a.nchunks * a.nvec;
}

int kv_conv_tokens_per_thread(long long total_q, int nvec, int num_sms) {
  // Runs of 8 tokens amortise the window reload and keep 8 loads in flight per thread,
  // but leave few threads when the step has few tokens (decode: one token per request,
  // where every token also starts a new request); there one token per thread keeps the
  // GPU's threads busy instead (at least 1024 threads per SM at 8).
  const long long threads_at_8 = 2ll * nvec * ((total_q + 7) / 8);
  return threads_at_8 >= (long long)num_sms * 1024 ? 8 : 1;
}

cudaError_t launch_kv_conv(const KvConvArgs& a, int kernel_size, cudaStream_t stream) {
  const int tok = a.tok;
  if (tok != 1 && tok != 8) return cudaErrorInvalidValue;
  if (a.conv_items + a.state_items <= 0) return cudaSuccess;
  switch (kernel_size) {
    case 1: return launch_ks<1>(a, tok, stream);
    case 2: return launch_ks<2>(a, tok, stream);
    case 3: return launch_ks<3>(a, tok, stream);
    case 4: return launch_ks<4>(a, tok, stream);
    case 5: return launch_ks<5>(a, tok, stream);
    case 6: return launch_ks<6>(a, tok, stream);
    case 7: return launch_ks<7>(a, tok, stream);
    case 8: return launch_ks<8>(a, tok, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ink
