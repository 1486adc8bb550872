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
// usable device address: the address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device, and cached.
#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(DA_NOALLOC_SCRATCH_BYTES);

// Partial outputs and log-sum-exps of the split kernel.  Nothing in it has to
// start at zero: every call overwrites what it later reads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxNoAllocDevices = 64;
void* g_scratch_addr[kMaxNoAllocDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on the current device.
int scratch_address(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return DA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxNoAllocDevices) return DA_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return DA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return DA_OK;
}

}  // namespace

extern "C" int decode_attn_noalloc(const void* q, const void* K, const void* V,
                                   const int32_t* seq_lens, void* out, int B, int h_q, int h_kv,
                                   int d_k, int d_v, int n_max, float scale, int dtype,
                                   int num_splits, int32_t* dev_error, cudaStream_t stream) {
  if (!q || !K || !V || !seq_lens || !out) return DA_ERR_NULL;
  int st = DA_OK;
  const size_t need = decode_attn_workspace_bytes(B, h_q, h_kv, d_k, d_v, n_max, dtype,
                                                  num_splits, &st);
  if (st != DA_OK) return st;
  if (need > kNoAllocScratchBytes) return DA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    st = scratch_address(&scratch);
    if (st != DA_OK) return st;
  }
  return decode_attn_ex(q, K, V, seq_lens, out, B, h_q, h_kv, d_k, d_v, n_max, scale, dtype,
                        num_splits, scratch, need > 0 ? kNoAllocScratchBytes : 0, dev_error, stream);
}
