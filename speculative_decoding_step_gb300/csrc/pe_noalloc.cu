// pe_draft_forward_noalloc: the drafter pass with its scratch in a fixed array
// that this library owns, for callers that cannot allocate device memory
// (a plugin whose host framework owns every device allocation, or a serving
// loop that must never call cudaMalloc).  See include/pe.h for the contract.
#include <mutex>

#include "pe_internal.h"

namespace {

// The scratch array.  In host code its name is only a host-side stand-in; the
// kernels receive the device address that cudaGetSymbolAddress returns.
static __device__ __align__(256) uint8_t g_noalloc_scratch[PE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {nullptr};
CUcontext g_ctx[kMaxDevices] = {nullptr};  // the context each cached address belongs to

// The calling thread's current context (the driver call found through the runtime, so the
// library links against the runtime alone); nullptr when none is current.
CUcontext current_context() {
  using Fn = CUresult (*)(CUcontext*);
  static Fn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (Fn) nullptr;
    return reinterpret_cast<Fn>(p);
  }();
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of the array on the current device.  Looked up once per device, and again
// when the device's context is no longer the one the address was taken in (after
// cudaDeviceReset the array lives at a new address in a new context).
pe_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  const CUcontext ctx = current_context();
  if (g_addr[dev] == nullptr || ctx == nullptr || ctx != g_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return PE_ERR_CUDA;
    g_addr[dev] = p;
    g_ctx[dev] = current_context();  // the lookup made the device's context current if none was
  }
  *out = g_addr[dev];
  return PE_OK;
}

}  // namespace

extern "C" pe_status pe_draft_forward_noalloc(const pe_config* cfg, const pe_weights* w, const pe_kv* kv,
                                              const int32_t* block_table, const void* x0, const int32_t* positions,
                                              const int64_t* slot_mapping, const int32_t* row_list,
                                              const int32_t* n_valid, const int32_t* draft_rows,
                                              int32_t* draft_tokens, float* logits_dbg, int32_t* err_word,
                                              pe_stream_t stream) {
  const pe_status st = pe_check_config(cfg);
  if (st != PE_OK) return st;
  const size_t need = pe_workspace_bytes(cfg);
  if (need == 0 || need > (size_t)PE_NOALLOC_SCRATCH_BYTES) return PE_ERR_SHAPE;
  void* scratch = nullptr;
  const pe_status sa = scratch_address(&scratch);
  if (sa != PE_OK) return sa;
  return pe_draft_forward(cfg, w, kv, block_table, x0, positions, slot_mapping, row_list, n_valid, draft_rows,
                          scratch, (size_t)PE_NOALLOC_SCRATCH_BYTES, draft_tokens, logits_dbg, err_word, stream);
}
