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

// One CTA of W warps per (b, query head).  Warp w merges splits w, w+W, ...
// in one pass, NB in flight, keeping a running maximum of the lse values it
// has seen (the online form of the combine; every weight is taken against the
// same maximum that scales the warp's sum).  Each lane holds D/32 consecutive
// columns.  The W warp results meet in shared memory and are merged the same
// way.  W = 16 when a head may have more than 8 * 17 splits (long contexts
// with hundreds of splits), else W = 8 (and always for balanced pieces), so
// that four CTAs fit on an SM and a batch of many heads merges in one wave.
// Dynamic shared memory of one combine CTA: only W * (D + 2) floats are used;
// the request caps the CTAs per SM (two of 16 warps, four of 8).  The grid
// may launch while the split kernel drains, and without the cap its CTAs pile
// up on the first SMs to free up.
template <int W>
constexpr int combine_smem_bytes() { return W == 16 ? 96 * 1024 : 48 * 1024; }

// EPL consecutive floats (EPL * 4-byte aligned) through L2, as vector loads.
template <int EPL>
__device__ __forceinline__ void ldcg_vec(float (&v)[EPL], const float* src) {
  if constexpr (EPL == 2) {
    const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
    v[0] = x.x, v[1] = x.y;
  } else {
#pragma unroll
    for (int i = 0; i < EPL; i += 4) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(src + i));
      v[i] = x.x, v[i + 1] = x.y, v[i + 2] = x.z, v[i + 3] = x.w;
    }
  }
}

// Splits the split kernel wrote for query head bh = b * h_q + h, given the
// sequence's seq_lens value: the same rules as its work list (the rows
// decoded for sequence b, then the chunked list's ceil(n / chunk) or, for
// balanced pieces, the count the unit's first CTA recorded).  Returns 1 when
// the split kernel wrote the output itself and 0 when a checked build finds
// the partial rows or the output row outside their buffers.
template <int D>
__device__ __forceinline__ int splits_of_head(const SplitParams& p, int bh, int seq_len,
                                              int heads_per_cta) {
  const int h_q = p.h_q;
  const int b = bh / h_q;
  int n = seq_len;
  const bool appended = p.append && n >= 0 && n < p.n_max;
  n = n < 0 ? 0 : (n > p.n_max ? p.n_max : n);
  if (appended) ++n;
  else n = max(0, min(n, p.row_lim) - p.row_off);
  const int chunk = *reinterpret_cast<const volatile int*>(p.chunk_out);
  int nv;
  if (chunk > 0) {  // chunked list: ceil(n / chunk) splits
    nv = n <= 0 ? 1 : (n + chunk - 1) / chunk;
  } else {          // balanced list: the unit's count, written by its first CTA
    const int group = h_q / p.h_kv, h = bh - b * h_q;
    const int kvh = h / group, hc = (h - kvh * group) / heads_per_cta;
    nv = __ldcg(p.unit_nv + (b * p.h_kv + kvh) * p.head_chunks + hc);
  }
  if (nv <= 1) return 1;
  // (checked builds: the partial rows and the output row stay inside their buffers)
  if (!DA_IN(p, size_t(bh) * p.max_splits + nv - 1, p.part_rows) ||
      !DA_IN(p, size_t(bh) * D + D - 1, p.out_elems))
    return 0;
  return nv;
}


// Merge of one query head's nv > 1 partials by the whole CTA.  Warp w takes
// splits w, w + kWarps, ... in passes of NB splits in flight (vector loads
// from L2), keeping a running maximum of the lse values it has seen (the
// online form of the combine: every weight is taken against the same maximum
// that scales the warp's sum).  Each lane holds D/32 consecutive columns.  The
// warp results meet in shared memory and are merged the same way; the output
// row and the head's natural-log lse are written.
template <int D, int kWarps, int NB>
__device__ __forceinline__ void merge_head(const SplitParams& p, int bh, int nv, float* red_acc,
                                           float* red_m, float* red_w) {
  constexpr int EPL = D / 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const float* lse = p.lse_part + size_t(bh) * p.max_splits;
  const float* op = p.o_part + size_t(bh) * p.max_splits * D + lane * EPL;

  float m = -INFINITY, wsum = 0.f, acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  for (int s = warp; s < nv; s += NB * kWarps) {
    float l[NB], v[NB][EPL];
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int su = s + u * kWarps;
      const bool ok = su < nv;
      l[u] = ok ? __ldcg(lse + su) : -INFINITY;
      if (ok) ldcg_vec<EPL>(v[u], op + size_t(su) * D);
      else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[u][e] = 0.f;
      }
    }
    float mx = m;
#pragma unroll
    for (int u = 0; u < NB; ++u) mx = fmaxf(mx, l[u]);
    const float m_use = mx == -INFINITY ? 0.f : mx;  // only empty splits so far
    const float scale = ex2(m - m_use);              // 0 while m is -inf
    wsum *= scale;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] *= scale;
#pragma unroll
    for (int u = 0; u < NB; ++u) {
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
    if (p.out_bf16) static_cast<__nv_bfloat16*>(p.out)[size_t(bh) * D + d] = __float2bfloat16_rn(v);
    else static_cast<float*>(p.out)[size_t(bh) * D + d] = v;
    if (d == 0 && p.lse_out) p.lse_out[bh] = W > 0.f ? (M_use + log2f(W)) * kLn2 : -INFINITY;
  }
}

template <int D, int W>
__global__ void __launch_bounds__(W * 32, 32 / W)
    lse_combine_kernel(const SplitParams p, int heads_per_cta) {
  constexpr int EPL = D / 32;
  constexpr int kWarps = W;
  extern __shared__ float csm[];
  float* red_acc = csm;                 // [kWarps][D]
  float* red_m = csm + kWarps * D;      // [kWarps]
  float* red_w = red_m + kWarps;        // [kWarps]

  // The next kernel on the stream may launch now: a split kernel's CTAs
  // cannot share an SM with a combine CTA (registers), so they take the SMs
  // this grid leaves free and wait there (griddepcontrol.wait) until it has
  // completed, with their set-up done and no launch latency left.  The
  // sequence's length is read before the wait: the split grid read the same
  // final value before it let this grid launch.
  const int bh = blockIdx.x;
  const int seq_len = __ldg(p.seq_lens + bh / p.h_q);
  allow_dependent_launch();
  wait_for_prerequisite_grid();

  const int nv = splits_of_head<D>(p, bh, seq_len, heads_per_cta);
  if (nv <= 1) return;  // written by the split kernel, or out of range (CTA-uniform)
  // NB splits per warp in flight at once: one pass covers NB * kWarps
  // splits, 272 for d <= 128 (256 splits and the one that rows appended past
  // n_max open).
  constexpr int NB = EPL == 4 ? 17 : (EPL == 2 ? 16 : 8);
  merge_head<D, kWarps, NB>(p, bh, nv, red_acc, red_m, red_w);
}

// Warp-per-head combine, for heads with few splits.  Eight warps per CTA, one
// query head each, at most 64 registers a thread and no shared memory, so
// that four CTAs share an SM: launched early, the grid waits on the first SMs
// the split grid frees and holds as few of them as it can from the next
// call's split CTAs.  The
// sequence's length is read before the wait (the split grid read the same
// final value before it let this grid launch); after the wait the split count
// and the first NB splits' partials are loaded together (slots past the count
// are allocated workspace, masked out once the count is known), so a head
// with at most NB splits is merged after one round trip.  Same online merge as
// merge_head, within one warp.
constexpr int kWarpCombineWarps = 8;

template <int D, int NB>
__global__ void __launch_bounds__(kWarpCombineWarps * 32, 4)
    lse_combine_warp_kernel(const SplitParams p, int heads_per_cta) {
  constexpr int EPL = D / 32;
  const int lane = threadIdx.x & 31;
  const long long head = (long long)blockIdx.x * kWarpCombineWarps + (threadIdx.x >> 5);
  const bool live = head < (long long)p.B * p.h_q;
  const int bh = live ? int(head) : 0;
  const int seq_len = __ldg(p.seq_lens + bh / p.h_q);
  allow_dependent_launch();
  wait_for_prerequisite_grid();
  if (!live) return;  // whole warps: nothing below synchronises the CTA
  const float* lse = p.lse_part + size_t(bh) * p.max_splits;
  const float* op = p.o_part + size_t(bh) * p.max_splits * D + lane * EPL;
  const int first = NB < p.max_splits ? NB : p.max_splits;
  float l[NB], v[NB][EPL];
#pragma unroll
  for (int u = 0; u < NB; ++u) {
    if (u < first) {
      l[u] = __ldcg(lse + u);
      ldcg_vec<EPL>(v[u], op + size_t(u) * D);
    }
  }
  const int nv = splits_of_head<D>(p, bh, seq_len, heads_per_cta);
  if (nv <= 1) return;  // written by the split kernel, or out of range
  float m = -INFINITY, wsum = 0.f, acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  for (int s = 0; s < nv; s += NB) {
    if (s > 0) {
#pragma unroll
      for (int u = 0; u < NB; ++u)
        if (s + u < nv) {
          l[u] = __ldcg(lse + s + u);
          ldcg_vec<EPL>(v[u], op + size_t(s + u) * D);
        }
    }
    // slots past the count hold anything: select them out, never multiply
#pragma unroll
    for (int u = 0; u < NB; ++u)
      if (s + u >= nv) {
        l[u] = -INFINITY;
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[u][e] = 0.f;
      }
    float mx = m;
#pragma unroll
    for (int u = 0; u < NB; ++u) mx = fmaxf(mx, l[u]);
    const float m_use = mx == -INFINITY ? 0.f : mx;  // only empty splits so far
    const float scale = ex2(m - m_use);              // 0 while m is -inf
    wsum *= scale;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] *= scale;
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const float f = ex2(l[u] - m_use);
      wsum += f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(f, v[u][e], acc[e]);
    }
    m = mx;
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) store_out(p, size_t(bh) * D + lane * EPL + e, acc[e] * inv);
  if (lane == 0 && p.lse_out) p.lse_out[bh] = wsum > 0.f ? (m + log2f(wsum)) * kLn2 : -INFINITY;
}

template <int D, int W>
static cudaError_t launch_combine_dw(const SplitParams& p, int heads_per_cta,
                                     cudaStream_t stream) {
  constexpr int kSmem = combine_smem_bytes<W>();
  static_assert(W * (D + 2) * 4 <= kSmem, "combine scratch");
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(lse_combine_kernel<D, W>, kSmem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_dependent(lse_combine_kernel<D, W>, p.B * p.h_q, W * 32, size_t(kSmem), stream,
                          p, heads_per_cta);
}

template <int D>
static cudaError_t launch_combine_d(const SplitParams& p, int heads_per_cta, int split_grid,
                                    cudaStream_t stream) {
  // One warp per head when a head's splits are expected to fit one pass of
  // NB: balanced pieces spread over about split_grid / units CTAs per unit,
  // chunked lists at most max_splits.  (Heads with more splits merge faster
  // across the warps of a CTA: measured 19 splits per head 4 % slower and 38
  // splits 2 % slower in one warp.)
  constexpr int NB = D == 256 ? 4 : (D == 128 ? 8 : 12);
  const long long units = (long long)p.B * p.h_kv * p.head_chunks;
  const long long expected = p.balanced ? (split_grid + units - 1) / units + 1 : p.max_splits;
  if (expected <= NB) {
    const long long heads = (long long)p.B * p.h_q;
    const int grid = int((heads + kWarpCombineWarps - 1) / kWarpCombineWarps);
    return launch_dependent(lse_combine_warp_kernel<D, NB>, grid, kWarpCombineWarps * 32, 0,
                            stream, p, heads_per_cta);
  }
  constexpr int NB8 = D == 128 ? 17 : (D == 64 ? 16 : 8);  // splits in flight per warp
  // balanced pieces: max_splits is one slot per CTA, but a unit rarely spans
  // more than a few pieces (8 warps take any count, in more than one pass)
  if (p.max_splits > 8 * NB8 && !p.balanced)
    return launch_combine_dw<D, 16>(p, heads_per_cta, stream);
  return launch_combine_dw<D, 8>(p, heads_per_cta, stream);
}

cudaError_t launch_combine(const SplitParams& p, int d, int heads_per_cta, int split_grid,
                           cudaStream_t stream) {
  if (d == 256) return launch_combine_d<256>(p, heads_per_cta, split_grid, stream);
  if (d == 128) return launch_combine_d<128>(p, heads_per_cta, split_grid, stream);
  return launch_combine_d<64>(p, heads_per_cta, split_grid, stream);
}

// ---------------------------------------------------------------------------
// Merge of S caller-gathered partials (the exchange step of a sequence-sharded
// decode).  Part s of head i holds the normalised output o_s of its rows and
// lse_s, the natural log of its softmax denominator; with L = max_s lse_s,
//     out = sum_s e^(lse_s - L) o_s / sum_s e^(lse_s - L),
//     lse = L + log(sum_s e^(lse_s - L)),
// the same identity as above in the natural-log domain.  One warp per head;
// each lane holds D/32 consecutive columns and walks the parts in order, with
// a running maximum (an online merge, four parts in flight).
// ---------------------------------------------------------------------------
constexpr int kMergeWarps = 8;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
    lse_merge_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts, int S,
                     void* __restrict__ out, int out_bf16, float* __restrict__ lse_out,
                     long long heads) {
  constexpr int EPL = D / 32;
  constexpr float kLog2e = 1.44269504088896341f;
  wait_for_prerequisite_grid();
  const long long i = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (i >= heads) return;
  const int lane = threadIdx.x & 31;
  const float* op = o_parts + i * D + lane * EPL;
  float m = -INFINITY, wsum = 0.f, acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  for (int s = 0; s < S; s += 4) {
    float l[4], v[4][EPL];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool ok = s + u < S;
      l[u] = ok ? __ldcg(lse_parts + (long long)(s + u) * heads + i) * kLog2e : -INFINITY;
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        v[u][e] = ok ? __ldcg(op + (long long)(s + u) * heads * D + e) : 0.f;
    }
    const float mx = fmaxf(fmaxf(m, fmaxf(l[0], l[1])), fmaxf(l[2], l[3]));
    const float m_use = mx == -INFINITY ? 0.f : mx;
    const float scale = ex2(m - m_use);
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
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const long long idx = i * D + lane * EPL + e;
    const float val = acc[e] * inv;
    if (out_bf16) static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(val);
    else static_cast<float*>(out)[idx] = val;
  }
  if (lane == 0 && lse_out)
    lse_out[i] = wsum > 0.f ? (m + log2f(wsum)) * kLn2 : -INFINITY;
}

cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int S, void* out,
                             int out_bf16, float* lse_out, long long heads, int d,
                             cudaStream_t stream) {
  const long long grid = (heads + kMergeWarps - 1) / kMergeWarps;
  if (d == 256)
    return launch_dependent(lse_merge_kernel<256>, int(grid), kMergeWarps * 32, 0, stream, o_parts,
                            lse_parts, S, out, out_bf16, lse_out, heads);
  if (d == 128)
    return launch_dependent(lse_merge_kernel<128>, int(grid), kMergeWarps * 32, 0, stream, o_parts,
                            lse_parts, S, out, out_bf16, lse_out, heads);
  return launch_dependent(lse_merge_kernel<64>, int(grid), kMergeWarps * 32, 0, stream, o_parts,
                          lse_parts, S, out, out_bf16, lse_out, heads);
}

}  // namespace da
