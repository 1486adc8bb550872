// Log-sum-exp combine across splits, and the KV-cache append (sm_103a).
#include <math.h>

#include "common.cuh"

namespace da {

// ---------------------------------------------------------------------------
// Combine.  One CTA of 4 warps per (b, query head).  Split s of sequence b
// holds the normalised partial output o_s of its rows and lse_s, the log2 of
// its softmax denominator taken on log2-domain scores.  With L = max_s lse_s,
// the whole-sequence result is
//     out = sum_s 2^(lse_s - L) o_s / sum_s 2^(lse_s - L),
// the same softmax over the union of the rows (the partial denominators add
// up to the full one).  Only the splits that hold rows are read: split s
// holds rows [s*chunk, min((s+1)*chunk, n_b)), so ceil(n_b / chunk) of them.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128)
    lse_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                       const int32_t* __restrict__ seq_lens, float* __restrict__ out, int h_q,
                       int num_splits, int chunk, int n_max) {
  constexpr int EPL = D / 32;
  __shared__ float red_m[4];
  __shared__ float red_w[4];
  __shared__ float red_acc[4][D];

  const int bh = blockIdx.x;
  const int b = bh / h_q;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int n = __ldg(seq_lens + b);
  n = n < 0 ? 0 : (n > n_max ? n_max : n);
  const int nv = (n + chunk - 1) / chunk;
  const float* lse = lse_part + size_t(bh) * num_splits;
  const float* op = o_part + size_t(bh) * num_splits * D;

  float mx = -INFINITY;
  for (int s = threadIdx.x; s < nv; s += blockDim.x) mx = fmaxf(mx, lse[s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red_m[warp] = mx;
  __syncthreads();
  const float L = fmaxf(fmaxf(red_m[0], red_m[1]), fmaxf(red_m[2], red_m[3]));

  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (L != -INFINITY) {
    for (int s = warp; s < nv; s += 4) {
      const float w = ex2(lse[s] - L);
      wsum += w;
      const float* row = op + size_t(s) * D + lane * EPL;
      if constexpr (EPL == 4) {
        const float4 x = *reinterpret_cast<const float4*>(row);
        acc[0] = fmaf(w, x.x, acc[0]);
        acc[1] = fmaf(w, x.y, acc[1]);
        acc[2] = fmaf(w, x.z, acc[2]);
        acc[3] = fmaf(w, x.w, acc[3]);
      } else {
        const float2 x = *reinterpret_cast<const float2*>(row);
        acc[0] = fmaf(w, x.x, acc[0]);
        acc[1] = fmaf(w, x.y, acc[1]);
      }
    }
  }
  if (lane == 0) red_w[warp] = wsum;
#pragma unroll
  for (int e = 0; e < EPL; ++e) red_acc[warp][lane * EPL + e] = acc[e];
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    const float W = red_w[0] + red_w[1] + red_w[2] + red_w[3];
    const float a = red_acc[0][d] + red_acc[1][d] + red_acc[2][d] + red_acc[3][d];
    out[size_t(bh) * D + d] = W > 0.f ? a / W : 0.f;
  }
}

cudaError_t launch_combine(const SplitParams& p, int d, cudaStream_t stream) {
  const int blocks = p.B * p.h_q;
  if (d == 128)
    lse_combine_kernel<128><<<blocks, 128, 0, stream>>>(p.o_part, p.lse_part, p.seq_lens, p.out,
                                                        p.h_q, p.num_splits, p.chunk, p.n_max);
  else
    lse_combine_kernel<64><<<blocks, 128, 0, stream>>>(p.o_part, p.lse_part, p.seq_lens, p.out,
                                                       p.h_q, p.num_splits, p.chunk, p.n_max);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// KV append ("MoA-Structured Decode Attention", introduction item 3):
// row pos[b] of every (b, kv head) of K and V receives the new key / value
// row.  One thread moves 16 bytes; consecutive threads move consecutive
// 16-byte pieces of a row, so both the reads and the writes are coalesced.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                     uint4* __restrict__ K, uint4* __restrict__ V, const int32_t* __restrict__ pos,
                     int B, int h_kv, int kvec, int vvec, int n_max, int32_t* dev_error) {
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
  if (e < kvec)
    K[dst_row * kvec + e] = __ldg(k_new + size_t(row) * kvec + e);
  else
    V[dst_row * vvec + (e - kvec)] = __ldg(v_new + size_t(row) * vvec + (e - kvec));
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* K, void* V,
                             const int32_t* pos, int B, int h_kv, int row_bytes_k, int row_bytes_v,
                             int n_max, int32_t* dev_error, cudaStream_t stream) {
  const int kvec = row_bytes_k / 16, vvec = row_bytes_v / 16;
  const long long total = (long long)B * h_kv * (kvec + vvec);
  const int threads = 256;
  const long long blocks = (total + threads - 1) / threads;
  kv_append_kernel<<<unsigned(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), static_cast<uint4*>(K),
      static_cast<uint4*>(V), pos, B, h_kv, kvec, vvec, n_max, dev_error);
  return cudaGetLastError();
}

}  // namespace da
