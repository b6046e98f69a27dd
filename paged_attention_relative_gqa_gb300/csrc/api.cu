// api.cu -- the C ABI of libinkling_attn.so (declared in include/inkling_attn.h):
// argument validation, workspace layout, TMA tensor-map encoding and kernel launch.
// Host code here touches only scalars and pointer values; it never synchronises,
// allocates or copies (except inkling_attn_read_device_error, which is documented to).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <cstring>

#include "../../include/inkling_attn.h"
#include "kernels.h"

namespace {

using ink::DecodeArgs;
using ink::PrefillArgs;

constexpr size_t kHeaderBytes = 256;  // error word lives at offset 0

// Limit of one pipeline wait inside the kernels launched from now on (default 2 s).
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

ink_status_t validate(const ink_attn_params_t* p) {
  if (!p) return INK_ERR_NULL_PTR;
  if (p->num_seqs < 0 || p->num_q_heads < 1 || p->num_kv_heads < 1 || p->rel_extent < 1 ||
      p->max_pages_per_seq < 1 || p->num_pages < 1)
    return INK_ERR_BAD_SHAPE;
  if (p->num_q_heads % p->num_kv_heads != 0) return INK_ERR_BAD_SHAPE;
  if (p->head_dim != 64 && p->head_dim != 128) return INK_ERR_BAD_SHAPE;
  if (!is_pow2(p->page_size) || p->page_size < 8 || p->page_size > (1 << 20))
    return INK_ERR_BAD_PAGE_SIZE;
  // TMA row coordinates and in-kernel row arithmetic are 32-bit
  const long long rows = (long long)p->num_pages * p->num_kv_heads * p->page_size;
  if (rows >= (1ll << 31)) return INK_ERR_TOO_LARGE;
  if ((long long)p->max_pages_per_seq * p->page_size >= (1ll << 31)) return INK_ERR_TOO_LARGE;
  if (!(p->sm_scale == p->sm_scale)) return INK_ERR_BAD_SHAPE;  // NaN scale
  return INK_OK;
}

struct DecodePlan {
  int head_chunks, tiles_per_split, num_splits;
};

// Split-K plan for decode.  Visible keys of one sequence span at most `max_tiles`
// 64-key tiles (window-limited on sliding-window layers).  The persistent decode kernel
// runs one CTA per SM over work units (split, sequence, KV head, head chunk); the tiles
// of a sequence are cut into splits so that there are about kTargetUnits units in the
// worst case, enough for an even spread over the SMs, while each split keeps at least
// two tiles.
constexpr long long kTargetUnits = 608;  // 4 units per SM on a 152-SM GB300

DecodePlan plan_decode(const ink_attn_params_t* p) {
  DecodePlan d;
  const int G = p->num_q_heads / p->num_kv_heads;
  d.head_chunks = (G + 15) / 16;
  const long long max_keys = (long long)p->max_pages_per_seq * p->page_size;
  long long max_tiles = (max_keys + ink::TILE_KEYS - 1) / ink::TILE_KEYS;
  if (p->window > 0) {
    const long long wt = (p->window + ink::TILE_KEYS - 1) / ink::TILE_KEYS + 1;
    if (wt < max_tiles) max_tiles = wt;
  }
  if (max_tiles < 1) max_tiles = 1;
  const long long units = (long long)(p->num_seqs > 0 ? p->num_seqs : 1) * p->num_kv_heads * d.head_chunks;
  long long tps = (units * max_tiles + kTargetUnits - 1) / kTargetUnits;
  if (tps < 2) tps = 2;
  if (tps > 64) tps = 64;
  long long splits = (max_tiles + tps - 1) / tps;
  if (splits > ink::MAX_DECODE_SPLITS) splits = ink::MAX_DECODE_SPLITS;
  tps = (max_tiles + splits - 1) / splits;  // rebalance
  splits = (max_tiles + tps - 1) / tps;
  d.tiles_per_split = (int)tps;
  d.num_splits = (int)splits;
  return d;
}

struct DecodeLayout {
  size_t tickets_off, part_o_off, part_ml_off, total;
};

DecodeLayout decode_layout(const ink_attn_params_t* p, const DecodePlan& d) {
  DecodeLayout l;
  const size_t B = (size_t)(p->num_seqs > 0 ? p->num_seqs : 1);
  const size_t nt = B * p->num_kv_heads * d.head_chunks;
  l.tickets_off = kHeaderBytes;
  l.part_o_off = align_up(l.tickets_off + nt * sizeof(int32_t), 256);
  const size_t rows = B * p->num_q_heads * (size_t)d.num_splits;
  l.part_ml_off = align_up(l.part_o_off + rows * p->head_dim * sizeof(float), 256);
  l.total = align_up(l.part_ml_off + rows * 2 * sizeof(float), 256);
  return l;
}

// ---- TMA tensor maps over a K or V pool viewed as [num_pages*Hkv*P rows, D] bf16

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// A bf16 matrix [rows, cols] (row pitch cols*2 bytes) with boxes of 64 columns x box_rows
// rows, 128-byte swizzle.
bool make_rows_map(CUtensorMap* map, const void* base, uint64_t rows, int cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same bf16 rows as a 3-D tensor {64 columns, rows, column blocks} (row pitch
// `pitch` elements, blocks 128 bytes apart): one box of box_rows rows x `blocks` column
// blocks lands in shared memory as the 128-byte-swizzled sub-tiles [block][row][64] that
// separate 2-D boxes would give, block stride box_rows * 128 bytes.
bool make_rows_map3(CUtensorMap* map, const void* base, uint64_t rows, uint64_t pitch, int blocks, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(pitch / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)pitch * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)blocks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A K or V pool of `rows` rows (a multiple of 16) as a 4-D tensor {64 columns, 16 rows,
// column blocks, 16-row groups}: one box of `groups` groups lands in shared memory as
// [group][block][16 rows][64], 2 KB blocks with the 128-byte swizzle.
bool make_group_map(CUtensorMap* map, const void* base, uint64_t rows, int D, int groups) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {64, 16, (cuuint64_t)(D / 64), (cuuint64_t)(rows / 16)};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, 128, (cuuint64_t)D * 2 * 16};
  cuuint32_t box[4] = {64, 16, (cuuint32_t)(D / 64), (cuuint32_t)groups};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

uint64_t pool_rows(const ink_attn_params_t* p) {
  return (uint64_t)p->num_pages * p->num_kv_heads * p->page_size;
}

// K or V pool as [num_pages*Hkv*P rows, D], boxes of min(P, box_cap) rows.
bool make_pool_map(CUtensorMap* map, const void* base, const ink_attn_params_t* p, int box_cap) {
  const int box_rows = p->page_size < box_cap ? p->page_size : box_cap;
  return make_rows_map(map, base, pool_rows(p), p->head_dim, box_rows);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// rel_logits [total_q, Hq, E] (fp32 or bf16) as a 3-D tensor {E, Hq, total_q}; boxes of
// box_cols buckets x 1 head x box_rows tokens, out-of-range elements read as 0.
bool make_bias_map(CUtensorMap* map, const void* rel, bool bf16, const ink_attn_params_t* p, int total_q,
                   int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t es = bf16 ? 2 : 4;
  cuuint64_t dims[3] = {(cuuint64_t)p->rel_extent, (cuuint64_t)p->num_q_heads, (cuuint64_t)total_q};
  cuuint64_t strides[2] = {(cuuint64_t)p->rel_extent * es, (cuuint64_t)p->rel_extent * es * p->num_q_heads};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                  const_cast<void*>(rel), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Low-rank bias operands: r [total_q, Hq, d_rel] as {d_rel, Hq, total_q} with boxes of 64
// columns x 128 tokens of one head, and proj_t [E, d_rel] as {d_rel, E} with boxes of 64
// columns x LOWRANK_CHUNK buckets; 128-byte rows with the 128-byte swizzle, as the bias MMA's
// K-major operands (K = 64) want them.  Columns past d_rel, tokens past total_q and buckets
// outside [0, E) read as zeros, so a smaller d_rel adds zero products.
bool make_lowrank_maps(ink::PrefillMaps* m, const void* r, const void* proj_t, const ink_attn_params_t* p,
                       int total_q, int d_rel) {
  auto fn = encode_fn();
  if (!fn) return false;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B;
  cuuint64_t dims_r[3] = {(cuuint64_t)d_rel, (cuuint64_t)p->num_q_heads, (cuuint64_t)total_q};
  cuuint64_t str_r[2] = {(cuuint64_t)d_rel * 2, (cuuint64_t)d_rel * 2 * p->num_q_heads};
  cuuint32_t box_r[3] = {(cuuint32_t)ink::LOWRANK_MAX_D, 1, (cuuint32_t)ink::PREFILL_ROWS};
  cuuint32_t e3[3] = {1, 1, 1};
  CUresult e = fn(&m->lr_r, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(r), dims_r, str_r, box_r, e3,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (e != CUDA_SUCCESS) return false;
  cuuint64_t dims_p[2] = {(cuuint64_t)d_rel, (cuuint64_t)p->rel_extent};
  cuuint64_t str_p[1] = {(cuuint64_t)d_rel * 2};
  cuuint32_t box_p[2] = {(cuuint32_t)ink::LOWRANK_MAX_D, (cuuint32_t)ink::LOWRANK_CHUNK};
  cuuint32_t e2[2] = {1, 1};
  e = fn(&m->lr_p, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(proj_t), dims_p, str_p, box_p, e2,
         CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return e == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

int32_t inkling_attn_version(void) { return 100; }

void inkling_attn_set_wait_limit_ns(uint64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns > 2000000000ull ? 2000000000ull : limit_ns, std::memory_order_relaxed);
}

const char* inkling_attn_status_string(ink_status_t s) {
  switch (s) {
    case INK_OK: return "ok";
    case INK_ERR_NULL_PTR: return "null pointer argument";
    case INK_ERR_BAD_SHAPE: return "bad shape (heads not divisible, head_dim not 64/128, or non-positive size)";
    case INK_ERR_BAD_PAGE_SIZE: return "page_size must be a power of two >= 8";
    case INK_ERR_WORKSPACE: return "workspace too small";
    case INK_ERR_ALIGNMENT: return "misaligned pointer (16 bytes for q/k/v/out, 4 for index and bias arrays)";
    case INK_ERR_CUDA: return "CUDA runtime error";
    case INK_ERR_TOO_LARGE: return "sizes overflow 32-bit coordinates";
  }
  return "unknown status";
}

size_t inkling_attn_workspace_bytes(const ink_attn_params_t* params, int is_decode) {
  if (validate(params) != INK_OK) return 0;
  if (!is_decode) return kHeaderBytes;
  return decode_layout(params, plan_decode(params)).total;
}

ink_status_t inkling_attn_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace) return INK_ERR_NULL_PTR;
  if (workspace_bytes < kHeaderBytes) return INK_ERR_WORKSPACE;
  if (cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream) != cudaSuccess)
    return INK_ERR_CUDA;
  return INK_OK;
}

ink_status_t inkling_attn_read_device_error(void* workspace, size_t workspace_bytes, void* stream,
                                            uint32_t* err_out, int clear) {
  if (!workspace || !err_out) return INK_ERR_NULL_PTR;
  if (workspace_bytes < kHeaderBytes) return INK_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return INK_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return INK_ERR_CUDA;
  *err_out = v;
  if (clear) {
    if (cudaMemsetAsync(workspace, 0, sizeof v, st) != cudaSuccess) return INK_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return INK_ERR_CUDA;
  }
  return INK_OK;
}

ink_status_t inkling_attn_decode(const ink_attn_params_t* params, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_table,
                                 const int32_t* seq_lens, const float* rel_logits, void* out,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  ink_status_t st = validate(params);
  if (st != INK_OK) return st;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !rel_logits || !out || !workspace)
    return INK_ERR_NULL_PTR;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(rel_logits, 4) ||
      !aligned(workspace, 256))
    return INK_ERR_ALIGNMENT;
  const DecodePlan plan = plan_decode(params);
  const DecodeLayout lay = decode_layout(params, plan);
  if (workspace_bytes < lay.total) return INK_ERR_WORKSPACE;
  if (params->num_seqs == 0) return INK_OK;
  ink::DecodeMaps maps;
  const int cblocks = params->head_dim / 64;
  if (!make_pool_map(&maps.k_seg, k_cache, params, 16) ||
      !make_pool_map(&maps.v_seg, v_cache, params, 16) ||
      !make_rows_map3(&maps.q3, q, (uint64_t)params->num_seqs * params->num_q_heads, params->head_dim, cblocks, 16))
    return INK_ERR_CUDA;
  std::memset(&maps.k_tile, 0, sizeof maps.k_tile);
  std::memset(&maps.v_tile, 0, sizeof maps.v_tile);
  std::memset(&maps.k_grp, 0, sizeof maps.k_grp);
  std::memset(&maps.v_grp, 0, sizeof maps.v_grp);
  if (params->page_size >= 16 &&
      (!make_group_map(&maps.k_grp, k_cache, pool_rows(params), params->head_dim, 1) ||
       !make_group_map(&maps.v_grp, v_cache, pool_rows(params), params->head_dim, 1)))
    return INK_ERR_CUDA;
  if (params->page_size >= ink::TILE_KEYS &&
      (!make_group_map(&maps.k_tile, k_cache, pool_rows(params), params->head_dim, ink::TILE_KEYS / 16) ||
       !make_group_map(&maps.v_tile, v_cache, pool_rows(params), params->head_dim, ink::TILE_KEYS / 16)))
    return INK_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeArgs a;
  a.q = q;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.rel = rel_logits;
  a.out = out;
  a.part_o = reinterpret_cast<float*>(ws + lay.part_o_off);
  a.part_ml = reinterpret_cast<float*>(ws + lay.part_ml_off);
  a.tickets = reinterpret_cast<int32_t*>(ws + lay.tickets_off);
  a.err = reinterpret_cast<uint32_t*>(ws);
  a.B = params->num_seqs;
  a.Hq = params->num_q_heads;
  a.Hkv = params->num_kv_heads;
  a.G = params->num_q_heads / params->num_kv_heads;
  a.head_chunks = plan.head_chunks;
  a.log2_page = ilog2(params->page_size);
  a.max_pages = params->max_pages_per_seq;
  a.num_pages = params->num_pages;
  a.E = params->rel_extent;
  a.W = params->window;
  a.scale_log2 = params->sm_scale * 1.4426950408889634f;
  a.tiles_per_split = plan.tiles_per_split;
  a.num_splits = plan.num_splits;
  a.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  if (ink::launch_decode(maps, a, params->head_dim, (cudaStream_t)stream) != cudaSuccess)
    return INK_ERR_CUDA;
  return INK_OK;
}

}  // extern "C"

namespace {

// The bias of a prefill call: rel_logits in fp32 or bf16, or its low-rank factors.
enum class BiasIn { F32, BF16, LOWRANK };

// Shared by the fp32-bias, bf16-bias and low-rank-bias prefill entry points.
ink_status_t prefill_impl(const ink_attn_params_t* params, const void* q, const int32_t* cu_q_lens,
                          int32_t max_q_len, int32_t total_q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, const int32_t* seq_lens, const void* rel_logits,
                          BiasIn bias_in, const void* lr_r, const void* lr_proj_t, int32_t d_rel, void* out,
                          void* workspace, size_t workspace_bytes, void* stream) {
  ink_status_t st = validate(params);
  if (st != INK_OK) return st;
  const bool bias_bf16 = bias_in == BiasIn::BF16, lowrank = bias_in == BiasIn::LOWRANK;
  if (!q || !cu_q_lens || !k_cache || !v_cache || !block_table || !seq_lens || !out || !workspace)
    return INK_ERR_NULL_PTR;
  if (lowrank ? (!lr_r || !lr_proj_t) : !rel_logits) return INK_ERR_NULL_PTR;
  if (max_q_len < 0 || total_q < 0) return INK_ERR_BAD_SHAPE;
  if (lowrank && (d_rel < 8 || d_rel > ink::LOWRANK_MAX_D || d_rel % 8 != 0)) return INK_ERR_BAD_SHAPE;
  if ((long long)total_q * params->num_q_heads >= (1ll << 31)) return INK_ERR_TOO_LARGE;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(cu_q_lens, 4) || !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(workspace, 256))
    return INK_ERR_ALIGNMENT;
  if (lowrank ? (!aligned(lr_r, 16) || !aligned(lr_proj_t, 16)) : !aligned(rel_logits, bias_bf16 ? 16 : 4))
    return INK_ERR_ALIGNMENT;
  if (bias_bf16 && params->rel_extent % 8 != 0) return INK_ERR_BAD_SHAPE;   // 16-byte bias rows
  if (workspace_bytes < kHeaderBytes) return INK_ERR_WORKSPACE;
  if (params->num_seqs == 0 || max_q_len == 0 || total_q == 0) return INK_OK;
  const int num_q_tiles = (max_q_len + ink::PREFILL_ROWS - 1) / ink::PREFILL_ROWS;
  if (num_q_tiles > 65535 || params->num_seqs > 65535) return INK_ERR_TOO_LARGE;
  ink::PrefillMaps maps;
  const int cblocks = params->head_dim / 64;
  std::memset(&maps.k3, 0, sizeof maps.k3);
  std::memset(&maps.v3, 0, sizeof maps.v3);
  if (params->page_size >= ink::TILE_KEYS &&
      (!make_rows_map3(&maps.k3, k_cache, pool_rows(params), params->head_dim, cblocks, ink::TILE_KEYS) ||
       !make_rows_map3(&maps.v3, v_cache, pool_rows(params), params->head_dim, cblocks, ink::TILE_KEYS)))
    return INK_ERR_CUDA;
  if (!make_pool_map(&maps.k, k_cache, params, ink::TILE_KEYS) ||
      !make_pool_map(&maps.v, v_cache, params, ink::TILE_KEYS) ||
      !make_rows_map3(&maps.q3, q, (uint64_t)total_q, (uint64_t)params->num_q_heads * params->head_dim, cblocks, 128))
    return INK_ERR_CUDA;
  PrefillArgs a;
  a.q = q;
  a.cu_q = cu_q_lens;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.rel = rel_logits;
  a.out = out;
  a.err = reinterpret_cast<uint32_t*>(workspace);
  a.B = params->num_seqs;
  a.Hq = params->num_q_heads;
  a.Hkv = params->num_kv_heads;
  a.G = params->num_q_heads / params->num_kv_heads;
  a.log2_page = ilog2(params->page_size);
  a.max_pages = params->max_pages_per_seq;
  a.num_pages = params->num_pages;
  a.E = params->rel_extent;
  a.W = params->window;
  a.scale_log2 = params->sm_scale * 1.4426950408889634f;
  a.sm_scale = params->sm_scale;
  a.max_q_len = max_q_len;
  a.num_q_tiles = num_q_tiles;
  a.bias_bf16 = bias_bf16 ? 1 : 0;
  a.bias_lowrank = lowrank ? 1 : 0;
  a.lr_r = lr_r;
  a.lr_proj_t = lr_proj_t;
  a.d_rel = d_rel;
  a.bias_bulk = !lowrank && (bias_bf16 || ((params->rel_extent % 4 == 0) && aligned(rel_logits, 16)));
  a.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  a.io32 = aligned(q, 32) && aligned(out, 32) ? 1 : 0;
  std::memset(&maps.bias, 0, sizeof maps.bias);
  std::memset(&maps.lr_r, 0, sizeof maps.lr_r);
  std::memset(&maps.lr_p, 0, sizeof maps.lr_p);
  if (lowrank && !make_lowrank_maps(&maps, lr_r, lr_proj_t, params, total_q, d_rel)) return INK_ERR_CUDA;
  if (a.bias_bulk) {
    // the head-pair kernel: 32-token bias boxes
    if (!make_bias_map(&maps.bias, rel_logits, bias_bf16, params, total_q,
                       bias_bf16 ? ink::PAIR_BIAS_COLS_BF16 : ink::PAIR_BIAS_COLS_F32, ink::PAIR_BIAS_ROWS))
      return INK_ERR_CUDA;
    if (ink::launch_prefill_pair(maps, a, params->head_dim, (cudaStream_t)stream) != cudaSuccess)
      return INK_ERR_CUDA;
    return INK_OK;
  }
  if (ink::launch_prefill_tc(maps, a, params->head_dim, (cudaStream_t)stream) != cudaSuccess)
    return INK_ERR_CUDA;
  return INK_OK;
}

}  // namespace

extern "C" {

ink_status_t inkling_attn_prefill(const ink_attn_params_t* params, const void* q,
                                  const int32_t* cu_q_lens, int32_t max_q_len, int32_t total_q,
                                  const void* k_cache,
                                  const void* v_cache, const int32_t* block_table,
                                  const int32_t* seq_lens, const float* rel_logits, void* out,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  return prefill_impl(params, q, cu_q_lens, max_q_len, total_q, k_cache, v_cache, block_table, seq_lens,
                      rel_logits, BiasIn::F32, nullptr, nullptr, 0, out, workspace, workspace_bytes, stream);
}

ink_status_t inkling_attn_prefill_bf16bias(const ink_attn_params_t* params, const void* q,
                                           const int32_t* cu_q_lens, int32_t max_q_len, int32_t total_q,
                                           const void* k_cache, const void* v_cache,
                                           const int32_t* block_table, const int32_t* seq_lens,
                                           const void* rel_logits_bf16, void* out, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  return prefill_impl(params, q, cu_q_lens, max_q_len, total_q, k_cache, v_cache, block_table, seq_lens,
                      rel_logits_bf16, BiasIn::BF16, nullptr, nullptr, 0, out, workspace, workspace_bytes, stream);
}

ink_status_t inkling_attn_prefill_lowrank_bias(const ink_attn_params_t* params, const void* q,
                                               const int32_t* cu_q_lens, int32_t max_q_len, int32_t total_q,
                                               const void* k_cache, const void* v_cache,
                                               const int32_t* block_table, const int32_t* seq_lens,
                                               const void* r, const void* rel_proj_t, int32_t d_rel, void* out,
                                               void* workspace, size_t workspace_bytes, void* stream) {
  return prefill_impl(params, q, cu_q_lens, max_q_len, total_q, k_cache, v_cache, block_table, seq_lens,
                      nullptr, BiasIn::LOWRANK, r, rel_proj_t, d_rel, out, workspace, workspace_bytes, stream);
}

ink_status_t inkling_attn_kv_conv_write(const ink_attn_params_t* params, const void* k_new,
                                        const void* v_new, const int32_t* cu_q_lens, int32_t total_q,
                                        const int32_t* seq_lens, const int32_t* block_table,
                                        const float* w_k, const float* w_v, int32_t kernel_size,
                                        const void* state_k_in, const void* state_v_in,
                                        void* state_k_out, void* state_v_out, void* k_cache,
                                        void* v_cache, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  ink_status_t st = validate(params);
  if (st != INK_OK) return st;
  if (kernel_size < 1 || kernel_size > 8 || total_q < 0) return INK_ERR_BAD_SHAPE;
  const bool has_state = kernel_size > 1;
  if (!k_new || !v_new || !cu_q_lens || !seq_lens || !block_table || !w_k || !w_v || !k_cache ||
      !v_cache || !workspace)
    return INK_ERR_NULL_PTR;
  if (has_state && (!state_k_in || !state_v_in || !state_k_out || !state_v_out)) return INK_ERR_NULL_PTR;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(w_k, 16) || !aligned(w_v, 16) || !aligned(cu_q_lens, 4) || !aligned(seq_lens, 4) ||
      !aligned(block_table, 4) || !aligned(workspace, 256))
    return INK_ERR_ALIGNMENT;
  if (has_state && (!aligned(state_k_in, 16) || !aligned(state_v_in, 16) || !aligned(state_k_out, 16) ||
                    !aligned(state_v_out, 16)))
    return INK_ERR_ALIGNMENT;
  if (workspace_bytes < kHeaderBytes) return INK_ERR_WORKSPACE;
  const int nvec = params->num_kv_heads * params->head_dim / 8;
  if ((long long)total_q * nvec * 8 >= (1ll << 40)) return INK_ERR_TOO_LARGE;
  ink::KvConvArgs a;
  a.x[0] = static_cast<const uint16_t*>(k_new);
  a.x[1] = static_cast<const uint16_t*>(v_new);
  a.w[0] = w_k;
  a.w[1] = w_v;
  a.st_in[0] = static_cast<const uint16_t*>(state_k_in);
  a.st_in[1] = static_cast<const uint16_t*>(state_v_in);
  a.st_out[0] = static_cast<uint16_t*>(state_k_out);
  a.st_out[1] = static_cast<uint16_t*>(state_v_out);
  a.cache[0] = static_cast<uint16_t*>(k_cache);
  a.cache[1] = static_cast<uint16_t*>(v_cache);
  a.cu_q = cu_q_lens;
  a.seq_lens = seq_lens;
  a.block_table = block_table;
  a.err = reinterpret_cast<uint32_t*>(workspace);
  a.B = params->num_seqs;
  a.T = total_q;
  a.Hkv = params->num_kv_heads;
  a.D = params->head_dim;
  a.log2_page = ilog2(params->page_size);
  a.max_pages = params->max_pages_per_seq;
  a.num_pages = params->num_pages;
  a.nvec = nvec;
  a.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  if (total_q == 0 && (params->num_seqs == 0 || !has_state)) return INK_OK;   // nothing to write
  int dev = 0;
  const int sms = ink::current_device_sms(&dev);
  if (sms <= 0) return INK_ERR_CUDA;
  ink::kv_conv_plan(a, kernel_size, sms);
  a.state_items = has_state ? 2ll * a.B * nvec : 0;   // each copies all ks - 1 rows of a vector
  if ((a.conv_items + a.state_items + 255) / 256 >= (1ll << 31)) return INK_ERR_TOO_LARGE;
  if (ink::launch_kv_conv(a, kernel_size, (cudaStream_t)stream) != cudaSuccess) return INK_ERR_CUDA;
  return INK_OK;
}

}  // extern "C"
