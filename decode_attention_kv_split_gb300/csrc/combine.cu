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

// One CTA of 16 warps per (b, query head).  Warp w merges splits w, w+16,
// ... in one pass, four in flight, keeping a running maximum of the lse
// values it has seen (the online form of the combine; every weight is taken
// against the same maximum that scales the warp's sum).  Each lane holds D/32
// consecutive columns.  The 16 warp results meet in shared memory and are
// merged the same way.
constexpr int kCombineWarps = 16;
// Dynamic shared memory of one combine CTA.  Only the first
// kCombineWarps * (D + 2) floats are used; the request is sized so that at
// most two CTAs share an SM.  The grid may launch while the split kernel
// drains, and without the cap its CTAs pile up on the first SMs to free up.
constexpr int kCombineSmemBytes = 96 * 1024;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
    lse_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                       const int* __restrict__ chunk_in, const int32_t* __restrict__ seq_lens,
                       int append, void* __restrict__ out, int out_bf16, int h_q, int max_splits,
                       int n_max, const int* __restrict__ unit_nv, int h_kv, int head_chunks,
                       int heads_per_cta) {
  constexpr int EPL = D / 32;
  constexpr int kWarps = kCombineWarps;
  extern __shared__ float csm[];
  float* red_acc = csm;                 // [kWarps][D]
  float* red_m = csm + kWarps * D;      // [kWarps]
  float* red_w = red_m + kWarps;        // [kWarps]

  // No early launch_dependents here: a next kernel whose CTAs sat resident
  // beside these ones, waiting for this grid, slowed the merge.  It launches
  // as these CTAs exit and waits for the grid to complete.
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
  int nv;
  if (chunk > 0) {  // chunked list: ceil(n / chunk) splits
    nv = n <= 0 ? 1 : (n + chunk - 1) / chunk;
  } else {          // balanced list: the unit's count, written by its first CTA
    const int group = h_q / h_kv, h = bh - b * h_q;
    const int kvh = h / group, hc = (h - kvh * group) / heads_per_cta;
    nv = __ldcg(unit_nv + (b * h_kv + kvh) * head_chunks + hc);
  }
  if (nv <= 1) return;  // written by the split kernel
  const float* lse = lse_part + size_t(bh) * max_splits;
  const float* op = o_part + size_t(bh) * max_splits * D + lane * EPL;

  float m = -INFINITY, wsum = 0.f, acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  for (int s = warp; s < nv; s += 4 * kWarps) {
    float l[4], v[4][EPL];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int su = s + u * kWarps;
      const bool ok = su < nv;
      l[u] = ok ? __ldcg(lse + su) : -INFINITY;
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[u][e] = ok ? __ldcg(op + size_t(su) * D + e) : 0.f;
    }
    const float mx = fmaxf(fmaxf(m, fmaxf(l[0], l[1])), fmaxf(l[2], l[3]));
    const float m_use = mx == -INFINITY ? 0.f : mx;  // only empty splits so far
    const float scale = ex2(m - m_use);              // 0 while m is -inf
    wsum *= scale;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] *= scale;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float f = ex2(l[u] - m_use);
      wsum += f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(f, v[u][e], acc[e]);
    }
    m = mx;
  }
  if (lane == 0) {
    red_m[warp] = m;
    red_w[warp] = wsum;
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) red_acc[warp * D + lane * EPL + e] = acc[e];
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w]);
    const float M_use = M == -INFINITY ? 0.f : M;
    float W = 0.f, a = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = ex2(red_m[w] - M_use);
      W += f * red_w[w];
      a += f * red_acc[w * D + d];
    }
    const float v = W > 0.f ? a / W : 0.f;
    if (out_bf16) static_cast<__nv_bfloat16*>(out)[size_t(bh) * D + d] = __float2bfloat16_rn(v);
    else static_cast<float*>(out)[size_t(bh) * D + d] = v;
  }
}

template <int D>
static cudaError_t launch_combine_d(const float* o_part, const float* lse_part,
                                    const int* chunk_in, const int32_t* seq_lens, int append,
                                    void* out, int out_bf16, int B, int h_q, int max_splits, int n_max,
                                    const int* unit_nv, int h_kv, int head_chunks,
                                    int heads_per_cta, cudaStream_t stream) {
  static_assert(kCombineWarps * (D + 2) * 4 <= kCombineSmemBytes, "combine scratch");
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(lse_combine_kernel<D>, kCombineSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  return launch_dependent(lse_combine_kernel<D>, B * h_q, kCombineWarps * 32,
                          size_t(kCombineSmemBytes), stream, o_part, lse_part, chunk_in, seq_lens,
                          append, out, out_bf16, h_q, max_splits, n_max, unit_nv, h_kv,
                          head_chunks, heads_per_cta);
}

cudaError_t launch_combine(const float* o_part, const float* lse_part, const int* chunk_in,
                           const int32_t* seq_lens, int append, void* out, int out_bf16, int B,
                           int h_q, int d, int max_splits, int n_max, const int* unit_nv, int h_kv,
                           int head_chunks, int heads_per_cta, cudaStream_t stream) {
  if (d == 256)
    return launch_combine_d<256>(o_part, lse_part, chunk_in, seq_lens, append, out, out_bf16, B,
                                 h_q, max_splits, n_max, unit_nv, h_kv, head_chunks,
                                 heads_per_cta, stream);
  if (d == 128)
    return launch_combine_d<128>(o_part, lse_part, chunk_in, seq_lens, append, out, out_bf16, B,
                                 h_q, max_splits, n_max, unit_nv, h_kv, head_chunks,
                                 heads_per_cta, stream);
  return launch_combine_d<64>(o_part, lse_part, chunk_in, seq_lens, append, out, out_bf16, B, h_q,
                              max_splits, n_max, unit_nv, h_kv, head_chunks, heads_per_cta,
                              stream);
}

}  // namespace da
