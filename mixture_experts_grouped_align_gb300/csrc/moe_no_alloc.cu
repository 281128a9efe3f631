// moe_forward_no_alloc: moe_forward with its scratch in a fixed device array of this
// library instead of a caller-provided workspace.
//
// Some callers cannot call cudaMalloc: code embedded in a host application that owns
// all device memory through its own pool and hands plug-ins only input and output
// buffers, or latency-critical threads that must not enter the CUDA allocator (it can
// synchronise the device and can fail under memory pressure at an arbitrary point).
// For them the layer's scratch (h, o and the f16 copy of x) lives in a file-scope
// device array of kNoAllocScratchBytes.  Every GPU that loads this library holds that
// array until the process exits.
#include "moe_common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = MOE_NO_ALLOC_SCRATCH_BYTES;

// The scratch.  Host code must not pass this symbol to a kernel: on the host it names a
// host-side stand-in, not device memory.  Its device address comes from
// cudaGetSymbolAddress on the current device.
static __device__ __align__(256) uint8_t g_no_alloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch on the current device.  Looked up on every call (the
// lookup allocates nothing and is cheap once the library's module is loaded on the
// device), so a context torn down and created again never leaves a stale address.
moe_status scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
  if (err != cudaSuccess || !p) {
    moe_host::set_error("moe_forward_no_alloc: cudaGetSymbolAddress: %s", cudaGetErrorString(err));
    return MOE_ERR_CUDA;
  }
  *out = p;
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_forward_no_alloc(
    const moe_weights* W, const void* x, const uint8_t* x_scale, int64_t T_rows, int64_t T_real,
    int32_t k, const float* topk_w, const int32_t* sorted_token_ids, const int32_t* expert_ids,
    const int32_t* num_tokens_post_padded, const int32_t* expert_offsets, int32_t block_m,
    int64_t cap_tokens, void* y, const moe_ctx* ctx) {
  if (!W) {
    moe_host::set_error("moe_forward_no_alloc: null weights");
    return MOE_ERR_INVALID_ARG;
  }
  // Only the size is checked here; moe_forward validates every argument itself (invalid
  // sizes give a workspace size of 0, which always fits, and are then rejected there).
  const size_t need = moe_forward_workspace_size(T_rows, k, W->K, W->I, cap_tokens);
  if (need > kNoAllocScratchBytes) {
    moe_host::set_error(
        "moe_forward_no_alloc: the call needs %zu bytes of scratch; the fixed array holds %zu "
        "(use moe_forward with a workspace for larger calls)",
        need, kNoAllocScratchBytes);
    return MOE_ERR_CAPACITY;
  }
  void* scratch = nullptr;
  moe_status st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  moe_ctx c{};
  if (ctx) c = *ctx;
  c.workspace = scratch;
  c.workspace_bytes = kNoAllocScratchBytes;
  return moe_forward(W, x, x_scale, T_rows, T_real, k, topk_w, sorted_token_ids, expert_ids,
                     num_tokens_post_padded, expert_offsets, block_m, cap_tokens, y, &c);
}
