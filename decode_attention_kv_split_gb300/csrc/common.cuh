// Shared device helpers for the decode-attention kernels (sm_103a).
//
// Inline PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor), ldmatrix,
// movmatrix, the bf16 tensor-core MMA, ex2 and the global timer, plus the
// split geometry that the host launcher and every kernel must agree on.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/decode_attn.h"

namespace da {

// ---------------------------------------------------------------------------
// Launch parameters shared by the split kernels and the combine kernel.
// ---------------------------------------------------------------------------
struct SplitParams {
  const void* q;            // [B, h_q, d]
  const int32_t* seq_lens;  // [B]
  float* out;               // [B, h_q, d] (written when num_splits == 1)
  float* o_part;            // [B, h_q, num_splits, d]   (num_splits > 1)
  float* lse_part;          // [B, h_q, num_splits]      log2-domain lse
  int32_t* dev_error;       // nullable
  int B, h_q, h_kv, group;  // group = h_q / h_kv
  int n_max;
  int num_splits;           // S: splits per (b, kv head)
  int chunk;                // C: rows per split (multiple of the tile height)
  int head_chunks;          // query-head chunks per kv head
  int items;                // B * h_kv * head_chunks * num_splits
  float scale_log2;         // scale * log2(e)
};

// Wall-clock limit for any wait inside a kernel.  A pipeline wait that has
// not completed after this long means a copy never landed; the kernel then
// records DA_DEVERR_TIMEOUT and finishes without waiting further.
constexpr unsigned long long kWaitTimeoutNs = 1000ull * 1000ull * 1000ull;

// ---------------------------------------------------------------------------
// Small PTX wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed, for at most
// kWaitTimeoutNs.  Returns false on timeout.  `abort_flag` (shared memory)
// short-cuts the wait once any warp of the CTA has timed out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitTimeoutNs) return false;
    }
  }
  return false;
}

// 3-D tiled TMA load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policy for data that is read exactly once (the K/V stream).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Named barrier over a subset of warps (id 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 2^x on the special-function unit.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack two floats into bf16x2 (round to nearest even); `lo` lands in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo_to_f32(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t x) {
  return __uint_as_float(x & 0xffff0000u);
}

__device__ __forceinline__ void flag_error(int32_t* dev_error, int bit) {
  if (dev_error) atomicOr(dev_error, bit);
}

// What a split-kernel variant needs from the host: its stage height (split
// lengths are multiples of it), how many query heads one work item covers,
// and the TMA box it expects.
struct KernelShape {
  int tile_rows;
  int heads_per_cta;
  int box_cols;    // inner box width in elements
  int swizzle128;  // 1: 128-byte swizzle, 0: none
};

KernelShape bf16_shape(int d, int group);
KernelShape f32_shape(int d, int group);
cudaError_t launch_split_bf16(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int d, int grid, cudaStream_t stream);
cudaError_t launch_split_f32(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             int d, int grid, cudaStream_t stream);
cudaError_t launch_combine(const SplitParams& p, int d, cudaStream_t stream);
cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* K, void* V,
                             const int32_t* pos, int B, int h_kv, int row_bytes_k,
                             int row_bytes_v, int n_max, int32_t* dev_error, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Work items: (b, kv head, head chunk, split), split fastest.
// ---------------------------------------------------------------------------
struct Item {
  int b, kvh, hc, split;
  int row_begin, row_end;  // rows [row_begin, row_end) of this (b, kvh); empty if equal
  int tiles;
};

template <int TILE>
__device__ __forceinline__ Item decode_item(const SplitParams& p, int i, int32_t* err_sink,
                                            bool report) {
  Item it;
  it.split = i % p.num_splits;
  int rest = i / p.num_splits;
  it.hc = rest % p.head_chunks;
  rest /= p.head_chunks;
  it.kvh = rest % p.h_kv;
  it.b = rest / p.h_kv;
  int n = __ldg(p.seq_lens + it.b);
  if (n < 0 || n > p.n_max) {
    if (report) flag_error(err_sink, DA_DEVERR_SEQ_LEN);
    n = n < 0 ? 0 : p.n_max;
  }
  it.row_begin = it.split * p.chunk;
  int end = it.row_begin + p.chunk;
  it.row_end = end < n ? end : n;
  if (it.row_end < it.row_begin) it.row_end = it.row_begin;
  it.tiles = (it.row_end - it.row_begin + TILE - 1) / TILE;
  return it;
}

}  // namespace da
