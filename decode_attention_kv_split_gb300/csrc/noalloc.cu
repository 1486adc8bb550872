// decode_attn_noalloc: decode attention for callers that cannot allocate
// device memory.
//
// The split path needs scratch for its per-split partial outputs.
// decode_attn_ex takes it from the caller and decode_attn allocates it with
// cudaMalloc.  Some callers can do neither: code that must not call
// cudaMalloc because it would synchronise the device in the middle of a
// latency-critical serving loop, code whose device memory is all owned and
// accounted by another allocator, or host runtimes that simply have no
// device allocator to call.  This entry point serves them from one buffer
// of fixed size that lives in the library itself.
//
// The buffer is a file-scope __device__ array, so every GPU that loads this
// library holds it (kNoAllocScratchBytes) until the process exits.  In host
// code the array's name is only a host-side stand-in for the symbol, never a
// usable device address: the address is looked up with cudaGetSymbolAddress,
// with the device current, on the first call made on that device, and cached
// together with the id of the context it belongs to; a call from a newer
// context of the device (after cudaDeviceReset) looks it up again.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(DA_NOALLOC_SCRATCH_BYTES);

// Partial outputs and log-sum-exps of the split kernel.  Nothing in it has to
// start at zero: every call overwrites what it later reads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxNoAllocDevices = 64;
struct ScratchEntry {
  unsigned long long ctx_id;  // the context the address belongs to (0: none yet)
  void* addr;
};
ScratchEntry g_scratch[kMaxNoAllocDevices] = {};
std::mutex g_scratch_mu;

// Driver entry points (no libcuda link): the current context and its
// process-unique id, so that an address looked up in a context that has since
// been destroyed (cudaDeviceReset) is never reused.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
std::once_flag g_ctx_fns_once;

int current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_fns_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!g_ctx_get_current || !g_ctx_get_id) return DA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return DA_ERR_CUDA;
  if (g_ctx_get_id(ctx, id) != CUDA_SUCCESS) return DA_ERR_CUDA;
  return DA_OK;
}

// Device address of g_noalloc_scratch in the current device's context.
int scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return DA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxNoAllocDevices) return DA_ERR_DEVICE;
  unsigned long long ctx_id = 0;
  int st = current_context_id(&ctx_id);
  void* fresh = nullptr;
  if (st != DA_OK) {
    // No context bound to this thread yet: the symbol lookup binds the
    // device's primary context (the one the launch will use); read its id then.
    e = cudaGetSymbolAddress(&fresh, g_noalloc_scratch);
    if (e != cudaSuccess || fresh == nullptr) return DA_ERR_CUDA;
    if ((st = current_context_id(&ctx_id)) != DA_OK) return st;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchEntry& ent = g_scratch[dev];
  if (ent.ctx_id != ctx_id || !ent.addr) {
    void* p = fresh;
    if (!p) {
      e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess || p == nullptr) return DA_ERR_CUDA;
    }
    ent.addr = p;
    ent.ctx_id = ctx_id;
  }
  *addr = ent.addr;
  return DA_OK;
}

}  // namespace

extern "C" int decode_attn_noalloc(const void* q, const void* K, const void* V,
                                   const int32_t* seq_lens, void* out, int B, int h_q, int h_kv,
                                   int d_k, int d_v, int n_max, float scale, int dtype,
                                   int num_splits, int32_t* dev_error, cudaStream_t stream) {
  if (!q || !K || !V || !seq_lens || !out) return DA_ERR_NULL;
  int st = DA_OK;
  size_t need = decode_attn_workspace_bytes(B, h_q, h_kv, d_k, d_v, n_max, dtype, num_splits,
                                            &st);
  if (st != DA_OK) return st;
  if (need > kNoAllocScratchBytes && num_splits == 0 &&
      da::library_takes_balanced(B, h_q, h_kv, d_k, d_v, n_max, dtype)) {
    // the library's balanced pieces do not fit: one split per sequence instead
    num_splits = 1;
    need = decode_attn_workspace_bytes(B, h_q, h_kv, d_k, d_v, n_max, dtype, num_splits, &st);
    if (st != DA_OK) return st;
  }
  if (need > kNoAllocScratchBytes) return DA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    st = scratch_address(&scratch);
    if (st != DA_OK) return st;
  }
  return decode_attn_ex(q, K, V, seq_lens, out, B, h_q, h_kv, d_k, d_v, n_max, scale, dtype,
                        num_splits, scratch, need > 0 ? kNoAllocScratchBytes : 0, dev_error, stream);
}
