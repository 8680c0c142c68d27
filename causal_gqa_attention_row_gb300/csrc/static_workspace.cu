// static_workspace.cu -- attn_decode_paged_static_workspace: the paged decode
// for callers that cannot allocate device memory themselves.
//
// Who needs it: code that has no device allocator to call -- a host program
// whose GPU memory is entirely handed out up front by another component (for
// example a serving engine that reserves all free HBM for its KV pool), a plugin
// inside a framework that does not expose its allocator, or a loop that must
// not risk the implicit device synchronisation cudaMalloc/cudaFree can cause.
// Such a caller can pass the inputs and outputs it already owns, but not the
// split-K scratch that attn_decode_paged takes as `workspace`.
//
// Here that scratch is a fixed array in the library's own device data. The CUDA
// runtime places it on a device when it loads this file's module there: with
// lazy module loading (CUDA's default) that happens at the first call on the
// device, which looks up the array's address; with eager loading, when the
// context is created. From then on the device holds it until the process exits,
// and no call here allocates anything.
#include <atomic>
#include <climits>

#include "gqa_attn.h"
#include "internal.h"

namespace {

// Largest split-K scratch the static entry point offers.
constexpr size_t kStaticWorkspaceBytes = GQA_STATIC_WORKSPACE_BYTES;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

// Host-side device address of g_static_workspace, per device. In host code the
// name g_static_workspace is only a host-side stand-in, never a device address,
// so the address is fetched with that device current and cached. The cache is
// atomic: host threads making their first calls at the same time may each look
// the address up, and they store the same value.
void* static_workspace_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  static std::atomic<void*> cache[64];
  void* ptr = cache[dev].load(std::memory_order_acquire);
  if (!ptr) {
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || ptr == nullptr) return nullptr;
    cache[dev].store(ptr, std::memory_order_release);
  }
  return ptr;
}

}  // namespace

extern "C" gqa_status attn_decode_paged_static_workspace(const void* q, const void* k_pool, const void* v_pool,
                                                         const int32_t* block_tables, const int32_t* seq_lens,
                                                         void* out, int B, int max_blocks_per_seq, int num_blocks,
                                                         int block_size, int H, int Hkv, int d_k, int d_v,
                                                         float attention_scale, gqa_dtype dt, void* stream) {
  if (max_blocks_per_seq <= 0 || block_size <= 0 || (long long)max_blocks_per_seq * block_size > INT_MAX / 2)
    return GQA_ERR_INVALID_ARG;
  // Every call, B = 0 included, makes sure the array is on the current device
  // first, so that a call with B = 0 is a complete set-up call.
  void* ws = static_workspace_ptr();
  if (!ws) return GQA_ERR_CUDA;
  const size_t need = attn_decode_workspace_bytes(B, H, d_v, max_blocks_per_seq * block_size);
  if (need > kStaticWorkspaceBytes) return GQA_ERR_WORKSPACE;  // beyond the fixed maximum
  // Nothing in the scratch needs clearing: the plan's ticket counter is reset by
  // the call's own planning kernel, and every partial a call reads was written
  // earlier in the same call.
  return attn_decode_paged(q, k_pool, v_pool, block_tables, seq_lens, out, B, max_blocks_per_seq, num_blocks,
                           block_size, H, Hkv, d_k, d_v, attention_scale, dt, ws, kStaticWorkspaceBytes, stream);
}
