// Log-sum-exp combine of the split partials (sm_103a).
//
// Split s of sequence b holds the normalised output o_s of its rows and
// lse_s, the log2 of its softmax denominator on log2-domain scores.  With
// L = max_s lse_s the whole-sequence result is
//     out = sum_s 2^(lse_s - L) o_s / sum_s 2^(lse_s - L),
// the softmax of "MoA-Structured Decode Attention" (section 2, eq. 2 and 3)
// over the union of the rows: the partial denominators add up to the full
// one.  Sequences with a single split were written by the split kernel and
// are skipped here.
//
// The kernel is launched with programmatic stream serialisation: its CTAs
// may start while the split kernel runs and wait (griddepcontrol.wait) for
// that grid's completion before reading anything it wrote.
#include <math.h>

#include "common.cuh"

namespace da {

// One CTA of 8 warps per (b, query head).  Warp w takes splits w, w+8, ...;
// each lane holds D/32 consecutive columns.  The 8 partial sums meet in
// shared memory.
template <int D>
__global__ void __launch_bounds__(256)
    lse_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                       const int* __restrict__ chunk_in, const int32_t* __restrict__ seq_lens,
                       int append, float* __restrict__ out, int h_q, int max_splits, int n_max) {
  constexpr int EPL = D / 32;
  constexpr int kWarps = 8;
  __shared__ float red_m[kWarps];
  __shared__ float red_w[kWarps];
  __shared__ float red_acc[kWarps][D];

  wait_for_prerequisite_grid();

  const int bh = blockIdx.x;
  const int b = bh / h_q;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int n = __ldg(seq_lens + b);
  const bool appended = append && n >= 0 && n < n_max;  // same rule as the split kernel
  n = n < 0 ? 0 : (n > n_max ? n_max : n);
  if (appended) ++n;
  const int chunk = *reinterpret_cast<const volatile int*>(chunk_in);
  const int nv = n <= 0 ? 1 : (n + chunk - 1) / chunk;
  if (nv <= 1 || chunk <= 0) return;  // written by the split kernel
  const float* lse = lse_part + size_t(bh) * max_splits;
  const float* op = o_part + size_t(bh) * max_splits * D;

  float mx = -INFINITY;
  for (int s = threadIdx.x; s < nv; s += blockDim.x) mx = fmaxf(mx, __ldcg(lse + s));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red_m[warp] = mx;
  __syncthreads();
  float L = red_m[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) L = fmaxf(L, red_m[w]);

  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  int s = warp;
  for (; s + 3 * kWarps < nv; s += 4 * kWarps) {  // four splits in flight per warp
    float w[4], v[4][EPL];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      w[u] = __ldcg(lse + s + u * kWarps);
      const float* row = op + size_t(s + u * kWarps) * D + lane * EPL;
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[u][e] = __ldcg(row + e);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float e2 = ex2(w[u] - L);
      wsum += e2;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(e2, v[u][e], acc[e]);
    }
  }
  for (; s < nv; s += kWarps) {
    const float e2 = ex2(__ldcg(lse + s) - L);
    wsum += e2;
    const float* row = op + size_t(s) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = fmaf(e2, __ldcg(row + e), acc[e]);
  }
  if (lane == 0) red_w[warp] = wsum;
#pragma unroll
  for (int e = 0; e < EPL; ++e) red_acc[warp][lane * EPL + e] = acc[e];
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float W = 0.f, a = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      W += red_w[w];
      a += red_acc[w][d];
    }
    out[size_t(bh) * D + d] = W > 0.f ? a / W : 0.f;
  }
}

cudaError_t launch_combine(const float* o_part, const float* lse_part, const int* chunk_in,
                           const int32_t* seq_lens, int append, float* out, int B, int h_q, int d,
                           int max_splits, int n_max, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(B) * unsigned(h_q));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (d == 128)
    return cudaLaunchKernelEx(&cfg, lse_combine_kernel<128>, o_part, lse_part, chunk_in, seq_lens,
                              append, out, h_q, max_splits, n_max);
  return cudaLaunchKernelEx(&cfg, lse_combine_kernel<64>, o_part, lse_part, chunk_in, seq_lens,
                            append, out, h_q, max_splits, n_max);
}

}  // namespace da
