// KV-cache append (sm_103a).
#include <math.h>

#include "common.cuh"

namespace da {

// ---------------------------------------------------------------------------
// KV append ("MoA-Structured Decode Attention", introduction item 3):
// row pos[b] of every (b, kv head) of K and V receives the new key / value
// row.  One thread moves 16 bytes; consecutive threads move consecutive
// 16-byte pieces of a row, so both the reads and the writes are coalesced.
// For an 8-bit cache the rows are codes, and the row scales (ks, vs: one
// float per cached row) receive the new rows' scales as well.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     uint4* __restrict__ K, uint4* __restrict__ V, const int32_t* __restrict__ pos,
                     int B, int h_kv, int kvec, int vvec, int n_max,
                     const float* __restrict__ ks_new, const float* __restrict__ vs_new,
                     float* __restrict__ ks, float* __restrict__ vs, int32_t* dev_error) {
  const int per_row = kvec + vvec;
  const long long total = (long long)B * h_kv * per_row;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int row = int(i / per_row);  // b * h_kv + h
  const int e = int(i % per_row);
  const int b = row / h_kv;
  const int p = __ldg(pos + b);
  if (p < 0 || p >= n_max) {
    if (e == 0 && row % h_kv == 0) flag_error(dev_error, DA_DEVERR_POS);
    return;
  }
  const size_t dst_row = size_t(row) * size_t(n_max) + size_t(p);
  if (e == 0 && ks) {
    ks[dst_row] = __ldg(ks_new + row);
    vs[dst_row] = __ldg(vs_new + row);
  }
  if (e < kvec)
    K[dst_row * kvec + e] = __ldg(k_new + size_t(row) * kvec + e);
  else
    V[dst_row * vvec + (e - kvec)] = __ldg(v_new + size_t(row) * vvec + (e - kvec));
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* K, void* V,
                             const int32_t* pos, int B, int h_kv, int row_bytes_k, int row_bytes_v,
                             int n_max, const float* ks_new, const float* vs_new, float* ks,
                             float* vs, int32_t* dev_error, cudaStream_t stream) {
  const int kvec = row_bytes_k / 16, vvec = row_bytes_v / 16;
  const long long total = (long long)B * h_kv * (kvec + vvec);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  kv_append_kernel<<<unsigned(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), static_cast<uint4*>(K),
      static_cast<uint4*>(V), pos, B, h_kv, kvec, vvec, n_max, ks_new, vs_new, ks, vs, dev_error);
  return cudaGetLastError();
}

}  // namespace da
