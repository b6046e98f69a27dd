// decode_noalloc.cu -- inkling_attn_decode_noalloc: paged decode for callers that can
// not allocate device memory, so cannot provide the workspace that
// inkling_attn_decode needs.  The split-K workspace (error word, tickets, partial
// softmax states) lives instead in one file-scope device array of fixed size that every
// GPU loading this library holds until the process exits.
//
// The call runs exactly the kernel and host path of inkling_attn_decode, handing it the
// address of that array as the workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/inkling_attn.h"

namespace {

// Largest workspace the allocation-free entry point can use (64 MiB per device).
constexpr size_t kStaticScratchBytes = size_t(64) << 20;

// The workspace every inkling_attn_decode_noalloc call on a device shares.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device.  In host code the array's
// name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, once per device, with that device current.
ink_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return INK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return INK_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return INK_OK;
}

}  // namespace

extern "C" ink_status_t inkling_attn_decode_noalloc(const ink_attn_params_t* params, const void* q,
                                                    const void* k_cache, const void* v_cache,
                                                    const int32_t* block_table,
                                                    const int32_t* seq_lens,
                                                    const float* rel_logits, void* out,
                                                    void* stream) {
  if (!params) return INK_ERR_NULL_PTR;
  const size_t need = inkling_attn_workspace_bytes(params, 1);
  if (need == 0) {
    // invalid parameters: let the regular entry point report which check failed
    // (it validates the scalars before it looks at any pointer)
    return inkling_attn_decode(params, q, k_cache, v_cache, block_table, seq_lens, rel_logits,
                               out, nullptr, 0, stream);
  }
  if (need > kStaticScratchBytes) return INK_ERR_WORKSPACE;
  void* scratch = nullptr;
  ink_status_t st = scratch_for_current_device(&scratch);
  if (st != INK_OK) return st;
  // The workspace starts with a 256-byte header (the device error word) followed by the
  // split-K tickets, one int32 per (sequence, KV head, 16-head chunk).  Both must be
  // zero when a call starts; earlier calls may have left anything there.
  const int G = params->num_q_heads / params->num_kv_heads;
  const size_t tickets = (size_t)params->num_seqs * params->num_kv_heads * ((G + 15) / 16);
  const size_t clear_bytes = 256 + ((tickets * sizeof(int32_t) + 255) / 256) * 256;
  if (cudaMemsetAsync(scratch, 0, clear_bytes, (cudaStream_t)stream) != cudaSuccess)
    return INK_ERR_CUDA;
  return inkling_attn_decode(params, q, k_cache, v_cache, block_table, seq_lens, rel_logits, out,
                             scratch, kStaticScratchBytes, stream);
}
