// kernels.h -- argument blocks and launchers shared between the host API (api.cu)
// and the kernel translation units.
#pragma once

#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ink {

// Keys per K/V tile: one TMA box is 64 rows of 128 bytes (64 bf16 of head_dim).
constexpr int TILE_KEYS = 64;

// Largest number of key splits a decode launch may use (bounds the merge scratch).
constexpr int MAX_DECODE_SPLITS = 64;

struct DecodeArgs {
  const void* q;              // bf16 [B, Hq, D]
  const int32_t* block_table; // [B, max_pages]
  const int32_t* seq_lens;    // [B]
  const float* rel;           // fp32 [B, Hq, E]
  void* out;                  // bf16 [B, Hq, D]
  float* part_o;              // fp32 [B, Hq, num_splits, D]
  float* part_ml;             // fp32 [B, Hq, num_splits, 2] (running max in log2 units, sum)
  int32_t* tickets;           // [B, Hkv * head_chunks]
  uint32_t* err;              // sticky error word
  int B, Hq, Hkv, G, head_chunks;
  int log2_page, max_pages, num_pages, E, W;
  float scale_log2;           // sm_scale * log2(e)
  int tiles_per_split, num_splits;
  unsigned long long wait_ns; // limit of one pipeline wait (the drain waits keep 2 s)
};

struct PrefillArgs {
  const void* q;              // bf16 [total_q, Hq, D]
  const int32_t* cu_q;        // [B+1]
  const int32_t* block_table; // [B, max_pages]
  const int32_t* seq_lens;    // [B]
  const void* rel;            // [total_q, Hq, E], fp32, or bf16 when bias_bf16
  void* out;                  // bf16 [total_q, Hq, D]
  uint32_t* err;
  int B, Hq, Hkv, G;
  int log2_page, max_pages, num_pages, E, W;
  float scale_log2;
  float sm_scale;             // multiplies q.k (the bias is added unscaled)
  int max_q_len, num_q_tiles;
  int bias_bulk;              // rows of rel are 16-byte aligned (E a multiple of 16 bytes, aligned base)
  int bias_bf16;              // rel holds bf16 values (always with bias_bulk)
  int bias_lowrank;           // bias from r and proj_t (rel unused)
  const void* lr_r;           // bf16 [total_q, Hq, d_rel]
  const void* lr_proj_t;      // bf16 [E, d_rel]
  int d_rel;                  // a multiple of 8 in [8, 64]
  unsigned long long wait_ns; // limit of one pipeline wait (the drain waits keep 2 s)
  int io32;                   // q and out 32-byte aligned: rows move in 256-bit loads and stores
};

// TMA descriptors of one decode call: K/V pools viewed as [num_pages*Hkv*P rows, D]
// with 64-row boxes (whole tiles) and 16-row boxes (tiles cut by the window start or
// the sequence end), and q viewed as [B*Hq rows, D] with 16-row boxes.
struct DecodeMaps {
  CUtensorMap k_seg, v_seg;   // 2-D, boxes of min(P, 16) rows x 64 columns (pages of 8 keys)
  CUtensorMap k_tile, v_tile; // 4-D group view, one box = 4 groups (a whole 64-key tile; P >= 64)
  CUtensorMap k_grp, v_grp;   // 4-D group view, one box = 1 group of 16 keys (P >= 16)
  CUtensorMap q3;             // 16 query rows, all column blocks in one box
};

// The current device's id and SM count, looked up once per device (host-only afterwards,
// so launches stay legal inside CUDA-graph stream capture).
int current_device_sms(int* dev_out);

// Opt a kernel into `bytes` of dynamic shared memory on the current device, once per
// device and kernel (the setting persists; repeating it inside stream capture is avoided).
template <typename Kernel>
inline cudaError_t smem_opt_in_once(Kernel kernel, int bytes, std::atomic<unsigned long long>& done) {
  int dev = 0;
  if (current_device_sms(&dev) <= 0 || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const unsigned long long bit = 1ull << dev;
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

cudaError_t launch_decode(const DecodeMaps& maps, const DecodeArgs& a, int head_dim,
                          cudaStream_t stream);
// TMA descriptors of one prefill call: K/V pools as for decode (min(P, 64)-row boxes) and
// q viewed as [total_q rows, Hq*D] with 128-row boxes (rows past total_q read as zero).
// bias: rel_logits viewed as [E, Hq, total_q] fp32 (innermost first) with boxes of
// 84 buckets x 1 head x 16 tokens (only built when rows of rel are 16-byte aligned).
struct PrefillMaps {
  CUtensorMap k, v, bias;
  CUtensorMap lr_r;     // low-rank bias: r viewed as {64, Hq, total_q}, box {64, 1, 128} (MMA operand A)
  CUtensorMap lr_p;     // low-rank bias: proj_t viewed as {64, E}, box {64, LOWRANK_CHUNK} (MMA operand B)
  CUtensorMap k3, v3;   // whole 64-key tiles, all column blocks in one box (P >= 64 only)
  CUtensorMap q3;       // 128 query rows of one head, all column blocks in one box
};

constexpr int BIAS_BOX_COLS = 84;   // buckets per bias box row
constexpr int BIAS_BOX_ROWS = 16;   // tokens per bias box
constexpr int BIAS_BOX_COLS_BF16 = 88;   // buckets per bias box row, bf16 bias
constexpr int PREFILL_ROWS = 128;        // new tokens per prefill work item
constexpr int LOWRANK_CHUNK = 64;        // projection rows per TMA box (one key tile's new buckets)
constexpr int LOWRANK_MAX_D = 64;        // largest d_rel of the low-rank bias (the MMA's K: four K-steps of 16)

cudaError_t launch_prefill_tc(const PrefillMaps& maps, const PrefillArgs& a, int head_dim,
                              cudaStream_t stream);

// The head-pair prefill (prefill_pair.cu): bias given as rel_logits with 16-byte rows, read by
// 3-D TMA boxes of PAIR_BIAS_ROWS tokens x PAIR_BIAS_COLS_* buckets of one head.
constexpr int PAIR_BIAS_ROWS = 32;
constexpr int PAIR_BIAS_COLS_F32 = 100;
constexpr int PAIR_BIAS_COLS_BF16 = 104;
cudaError_t launch_prefill_pair(const PrefillMaps& maps, const PrefillArgs& a, int head_dim,
                                cudaStream_t stream);

// One call of the K/V short convolution and paged write (kv_conv.cu).  Rows of the
// step's K/V and of the carried state are Hkv*D bf16 (nvec 16-byte vectors).
struct KvConvArgs {
  const uint16_t* x[2];        // k_new, v_new: bf16 [T, Hkv, D]
  const float* w[2];           // taps: fp32 [Hkv, D, ks]
  const uint16_t* st_in[2];    // bf16 [B, ks-1, Hkv, D], oldest row first
  uint16_t* st_out[2];         // same layout, never overlapping st_in
  uint16_t* cache[2];          // bf16 [num_pages, Hkv, P, D]
  const int32_t* cu_q;         // [B+1]
  const int32_t* seq_lens;     // [B]
  const int32_t* block_table;  // [B, max_pages]
  uint32_t* err;
  int B, T, Hkv, D, log2_page, max_pages, num_pages;
  int nvec;                    // Hkv * D / 8
  int tok;                     // tokens per thread (1 or 8)
  int nchunks;                 // ceil(T / tok)
  long long conv_items;        // 2 * nchunks * nvec threads of convolution
  long long state_items;       // 2 * B * nvec threads of state copy (each all ks-1 rows)
  int tile_tokens;             // staged kernel: new rows per tile (<= 32)
  int stages;                  // staged kernel: ring depth (0: use the per-thread kernel)
  unsigned long long wait_ns;  // limit of one pipeline wait (the drain waits keep 2 s)
};

// Largest dynamic shared memory of the staged K/V kernel.
constexpr size_t KV_STAGED_SMEM_MAX = 216 * 1024;

int kv_conv_tokens_per_thread(long long total_q, int nvec, int num_sms);
size_t kv_staged_smem_bytes(int tile_tokens, int kernel_size, int nvec, int stages);
// Fill tile_tokens, stages, tok, nchunks and conv_items of `a` (T, nvec, B set).
void kv_conv_plan(KvConvArgs& a, int kernel_size, int num_sms);
cudaError_t launch_kv_conv(const KvConvArgs& a, int kernel_size, cudaStream_t stream);

}  // namespace ink
