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
// Launch parameters shared by the split kernels.
// ---------------------------------------------------------------------------
// Sequences per launch: the work list is built in shared memory from this many
// lengths; the host cuts larger batches into several launches.
constexpr int kMaxBatchPerLaunch = 512;

struct SplitParams {
  const void* q;                 // [B, h_q, d]  (this launch's slice of the batch)
  const int32_t* seq_lens;       // [B]
  float* out;                    // [B, h_q, d]
  float* o_part;                 // [B, h_q, max_splits, d]  normalised partial outputs
  float* lse_part;               // [B, h_q, max_splits]     log2-domain log-sum-exp
  int* chunk_out;                // workspace word receiving the split length used (nullable)
  int32_t* dev_error;            // nullable
  // Fused append (append != 0): before decoding, row seq_lens[b] of every kv
  // head of K/V receives k_new[b, h] / v_new[b, h] and takes part in the decode.
  const void* k_new;             // [B, h_kv, d]
  const void* v_new;             // [B, h_kv, d]
  void* k_cache;                 // K base (all sequences; b_offset applies)
  void* v_cache;                 // V base
  int32_t* seq_lens_out;         // nullable: receives the lengths after the append
  int append;
  int B, h_q, h_kv, group;       // group = h_q / h_kv
  int b_offset;                  // first sequence of this launch inside the tensor maps
  int n_max;
  int head_chunks;               // query-head chunks per kv head
  int chunk_fixed;               // > 0: rows per split chosen by the caller
  int chunk_min;                 // else: smallest rows per split the device may choose
  int max_splits;                // partial slots per query head (ceil(n_max / chunk))
  float cta_speed;               // one CTA's streaming rate / its even share (split-length model)
  float scale_log2;              // scale * log2(e)
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

// Contiguous bulk copy global -> shared (size a multiple of 16 bytes, both
// addresses 16-byte aligned), completing on an mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
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

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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

__device__ __forceinline__ bool lane_is_zero(int tid) { return (tid & 31) == 0; }

__device__ __forceinline__ void flag_error(int32_t* dev_error, int bit) {
  if (dev_error) atomicOr(dev_error, bit);
}

// What a split-kernel variant needs from the host: its stage height (split
// lengths are multiples of it), how many query heads one work item covers,
// and the TMA box it expects.
struct KernelShape {
  int tile_rows;
  int heads_per_cta;
  int box_cols;     // inner box width in elements
  int swizzle128;   // 1: 128-byte swizzle, 0: none
  float cta_speed;  // how fast one CTA streams relative to an even share of HBM (measured)
};

KernelShape bf16_shape(int d, int group);
KernelShape f32_shape(int d, int group);
KernelShape tc5_shape(int group);
cudaError_t launch_split_tc5(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             int grid, cudaStream_t stream);
cudaError_t launch_split_bf16(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int d, int grid, cudaStream_t stream);
cudaError_t launch_split_f32(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             int d, int grid, cudaStream_t stream);
cudaError_t launch_combine(const float* o_part, const float* lse_part, const int* chunk_in,
                           const int32_t* seq_lens, int append, float* out, int B, int h_q, int d,
                           int max_splits, int n_max, cudaStream_t stream);
cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* K, void* V,
                             const int32_t* pos, int B, int h_kv, int row_bytes_k,
                             int row_bytes_v, int n_max, int32_t* dev_error, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Work list.
//
// Sequence b is cut into nv_b = max(1, ceil(n_b / chunk)) splits of `chunk`
// rows.  Each (kv head, head chunk) of b is a unit; each (unit, split) is a
// work item.  Items are numbered sequence by sequence, unit by unit, split by
// split, so the splits of one unit are consecutive and units complete one
// after another.  Persistent CTAs take items i = blockIdx.x + k * gridDim.x.
// Every CTA builds the same list in shared memory from seq_lens.
// ---------------------------------------------------------------------------
struct Schedule {
  int* first;       // [B + 1] first item of sequence b (shared memory)
  int* lens;        // [B] rows to decode; bit 31 set when row (len - 1) is appended now
  int chunk;
  int total;
};

constexpr int kAppendFlag = int(0x80000000u);
__device__ __forceinline__ int len_of(int v) { return v & 0x7fffffff; }

struct Item {
  int b, kvh, hc, split, nv;
  int row_begin, row_end;  // rows [row_begin, row_end) of head (b, kvh)
  int tiles;
  int new_row;             // row appended by this call (-1: none); the unit's last row
};

template <int TILE>
__device__ __forceinline__ Item schedule_item(const SplitParams& p, const Schedule& s, int i) {
  // last b with first[b] <= i
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.first[mid] <= i) lo = mid; else hi = mid - 1;
  }
  Item it;
  it.b = lo;
  const int per_seq = p.h_kv * p.head_chunks;
  it.nv = (s.first[lo + 1] - s.first[lo]) / per_seq;
  const int r = i - s.first[lo];
  const int unit = r / it.nv;
  it.split = r - unit * it.nv;
  it.kvh = unit / p.head_chunks;
  it.hc = unit - it.kvh * p.head_chunks;
  const int n = len_of(s.lens[lo]);
  it.new_row = (s.lens[lo] & kAppendFlag) ? n - 1 : -1;
  it.row_begin = it.split * s.chunk;
  const int end = it.row_begin + s.chunk;
  it.row_end = end < n ? end : n;
  if (it.row_end < it.row_begin) it.row_end = it.row_begin;
  it.tiles = (it.row_end - it.row_begin + TILE - 1) / TILE;
  return it;
}

// Choose the split length when the caller left it to the library.  Lanes
// 0-15 of warp 0 score chunk_min * 2^k; lanes 16-31 score "balanced" lengths
// that cut the longest sequence into R * grid / units pieces (R = 1..16), so
// that the items fill whole rounds of the grid.  The estimated time in rows
// streamed by one CTA is the larger of the even share of all rows and the
// busiest CTA's rows divided by how fast one CTA can stream relative to its
// even share (p.cta_speed: above 1 when a lone CTA can pull more than its
// share of HBM bandwidth, below 1 when a CTA is compute-bound), plus one tile
// of epilogue per item and two tiles when partials must be merged.  Ties go
// to more, shorter items.  All threads call this.
__device__ __forceinline__ int choose_chunk(const SplitParams& p, const int* lens, int tile,
                                            int grid, int* red /* shared, >= 1 int */) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    const int k = tid;
    long long rows = 0;
    int nmax = 0;
    for (int b = 0; b < p.B; ++b) {
      const int n = len_of(lens[b]);
      rows += n;
      nmax = n > nmax ? n : nmax;
    }
    const long long longest = nmax > 0 ? nmax : 1;
    const int per_seq = p.h_kv * p.head_chunks;
    const long long units = (long long)p.B * per_seq;
    long long c;
    if (k < 16) {
      c = (long long)p.chunk_min << k;
    } else {
      long long pieces = (long long)(k - 15) * grid / units;
      if (pieces < 1) pieces = 1;
      c = (longest + pieces - 1) / pieces;
    }
    c = (c + tile - 1) / tile * tile;
    if (c < p.chunk_min) c = p.chunk_min;
    if (c > (1LL << 30)) c = 1LL << 30;
    // power-of-two candidates stop after the first one covering everything
    const bool candidate = k >= 16 || k == 0 || ((long long)p.chunk_min << (k - 1)) < longest;
    float t = 3.0e38f;
    if (candidate) {
      long long items = 0;
      const int ci = int(c);
      for (int b = 0; b < p.B; ++b) {
        const int n = len_of(lens[b]);
        items += n <= 0 ? 1 : (n + ci - 1) / ci;
      }
      const float fitems = float(items) * float(per_seq);
      const float rounds = ceilf(fitems / float(grid));
      const float share = float(rows) * float(per_seq) / float(grid);
      const float ceff = float(c < longest ? c : longest);
      t = fmaxf(share, rounds * ceff / p.cta_speed) + rounds * float(tile);
      if (c < longest) t += 2.f * float(tile);
    }
    // argmin over lanes; within 0.1% prefer the shorter chunk (more items)
    float best_t = t;
    long long best_c = c;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ot = __shfl_xor_sync(0xffffffffu, best_t, o);
      const long long oc = __shfl_xor_sync(0xffffffffu, best_c, o);
      const bool take = oc < best_c ? ot <= best_t * 1.001f
                                    : (oc == best_c ? false : ot * 1.001f < best_t);
      if (take) {
        best_t = ot;
        best_c = oc;
      }
    }
    if (k == 0) red[0] = int(best_c);
  }
  __syncthreads();
  const int chunk = red[0];
  __syncthreads();
  return chunk;
}

// Builds the work list in shared memory; every thread of the CTA must call it.
// `first` has room for kMaxBatchPerLaunch + 1 ints, `lens` for kMaxBatchPerLaunch,
// `red` for 48 ints.
template <int TILE>
__device__ __forceinline__ Schedule build_schedule(const SplitParams& p, int* first, int* lens,
                                                   int* red) {
  const int tid = threadIdx.x;
  bool bad = false;
  bool bad_pos = false;
  for (int b = tid; b < p.B; b += blockDim.x) {
    int n = __ldg(p.seq_lens + b);
    bool app = false;
    if (p.append) {
      app = n >= 0 && n < p.n_max;  // room for the new row
      bad_pos |= !app;
    }
    if (n < 0 || n > p.n_max) {
      bad = true;
      n = n < 0 ? 0 : p.n_max;
    }
    if (app) ++n;
    lens[b] = app ? (n | kAppendFlag) : n;
    if (blockIdx.x == 0 && p.seq_lens_out) p.seq_lens_out[b] = n;
  }
  if (bad && blockIdx.x == 0) flag_error(p.dev_error, DA_DEVERR_SEQ_LEN);
  if (bad_pos && blockIdx.x == 0) flag_error(p.dev_error, DA_DEVERR_POS);
  __syncthreads();
  Schedule s;
  s.first = first;
  s.lens = lens;
  s.chunk = p.chunk_fixed > 0 ? p.chunk_fixed : choose_chunk(p, lens, TILE, gridDim.x, red);
  // exclusive scan of items per sequence by warp 0
  const int per_seq = p.h_kv * p.head_chunks;
  if (tid < 32) {
    int carry = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + tid;
      int c = 0;
      if (b < p.B) {
        const int n = len_of(lens[b]);
        c = per_seq * (n <= 0 ? 1 : (n + s.chunk - 1) / s.chunk);
      }
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (tid >= o) x += y;
      }
      if (b < p.B) first[b] = carry + x - c;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (tid == 0) first[p.B] = carry;
  }
  __syncthreads();
  s.total = first[p.B];
  if (blockIdx.x == 0 && tid == 0 && p.chunk_out) *p.chunk_out = s.chunk;
  return s;
}

// ---------------------------------------------------------------------------
// End of a work item, shared by every split kernel.
//
// The consumer warps have written, per (key warp, head), their running max m
// (log2 domain), running sum l and unnormalised accumulator into shared
// slots.  This merges the KW key warps of each head group by log-sum-exp and
// writes the item's normalised output: straight to `out` when the sequence
// has a single split, else to its partial slot with its log-sum-exp for the
// combine kernel.  All consumer threads call it together.
// ---------------------------------------------------------------------------
template <int D, int HG, int KW, int HPW, int SLOT_STRIDE>
__device__ __forceinline__ void finish_item(const SplitParams& p, const Item& it,
                                            const float* epi_acc, const float* epi_m,
                                            const float* epi_l, int ctid, int nthreads,
                                            volatile int* abort_flag) {
  constexpr int GC = HG * HPW;  // query heads of this item
  if (*abort_flag) return;
  const int head0 = it.hc * GC;  // group-local index of the item's first head
  const size_t bh0 = (size_t(it.b) * p.h_q + size_t(it.kvh) * p.group);
  for (int idx = ctid; idx < GC * D; idx += nthreads) {
    const int h = idx / D;  // head inside the item
    const int d = idx - h * D;
    if (head0 + h >= p.group) continue;
    const int hg = h / HPW, hw = h - hg * HPW;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < KW; ++k) M = fmaxf(M, epi_m[(hg * KW + k) * HPW + hw]);
    float L = 0.f, sum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int k = 0; k < KW; ++k) {
        const int sid = hg * KW + k;
        const float f = ex2(epi_m[sid * HPW + hw] - M);
        L += f * epi_l[sid * HPW + hw];
        sum += f * epi_acc[(sid * HPW + hw) * SLOT_STRIDE + d];
      }
    }
    const float o = L > 0.f ? sum / L : 0.f;
    const size_t bh = bh0 + head0 + h;
    if (it.nv == 1) {
      p.out[bh * D + d] = o;
    } else {
      p.o_part[(bh * p.max_splits + it.split) * D + d] = o;
      if (d == 0) p.lse_part[bh * p.max_splits + it.split] = L > 0.f ? M + log2f(L) : -INFINITY;
    }
  }
}

// Fused append: copy the new K and V rows (shared-memory slot, K row then V
// row, ROW_BYTES each) into row `row` of kv head (b_offset + b, kvh) of the
// caches.  One warp; an exact copy of the bits.
template <int ROW_BYTES>
__device__ __forceinline__ void store_new_row(const SplitParams& p, const Item& it,
                                              const uint8_t* slot, int lane) {
  const size_t head = size_t(p.b_offset + it.b) * p.h_kv + it.kvh;
  const size_t off = (head * size_t(p.n_max) + size_t(it.new_row)) * ROW_BYTES;
  const uint4* ks = reinterpret_cast<const uint4*>(slot);
  const uint4* vs = reinterpret_cast<const uint4*>(slot + ROW_BYTES);
  uint4* kd = reinterpret_cast<uint4*>(static_cast<char*>(p.k_cache) + off);
  uint4* vd = reinterpret_cast<uint4*>(static_cast<char*>(p.v_cache) + off);
  for (int i = lane; i < ROW_BYTES / 16; i += 32) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

// Let a combine kernel launched with programmatic stream serialisation start
// its launch while this grid is still running (it waits for our completion).
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// In a dependent grid: wait until the preceding grid has completed and its
// memory operations are visible.
__device__ __forceinline__ void wait_for_prerequisite_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Producer: one thread streams every tile of the CTA's items into the ring.
// NBOX boxes of BOX_COLS columns per tensor per stage, each BOX_BYTES long.
// ---------------------------------------------------------------------------
// The query rows of an item (its head chunk of one kv group, contiguous in
// q) ride with the item's first stage into that stage's q slot.
// With a fused append, the new K and V rows of the unit ride with the stage
// that holds the unit's last row, into that stage's new-row slot
// (2 * ROW_BYTES: the K row, then the V row).
template <int TILE, int STAGES, int STAGE_BYTES, int NBOX, int BOX_COLS, int BOX_BYTES,
          int HEADS, int ROW_BYTES>
__device__ __forceinline__ void produce(const CUtensorMap* tmK, const CUtensorMap* tmV,
                                        const SplitParams& p, const Schedule& s, uint32_t ring,
                                        uint32_t qslots, uint32_t newslots, uint32_t full0,
                                        uint32_t empty0, volatile int* abort_flag) {
  prefetch_tmap(tmK);
  prefetch_tmap(tmV);
  const uint64_t policy = l2_policy_evict_first();
  constexpr int kTileBytes = STAGE_BYTES / 2;
  int stage = 0;
  uint32_t phase = 0, issued = 0, issued_parity = 0;
  bool aborted = false;
  for (int i = blockIdx.x; i < s.total && !aborted; i += gridDim.x) {
    const Item it = schedule_item<TILE>(p, s, i);
    const int z = (p.b_offset + it.b) * p.h_kv + it.kvh;
    for (int t = 0; t < it.tiles; ++t) {
      if (!mbar_wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag)) {
        *abort_flag = 1;
        flag_error(p.dev_error, DA_DEVERR_TIMEOUT);
        aborted = true;
        break;
      }
      const uint32_t bar = full0 + 8 * stage;
      const int y0 = it.row_begin + t * TILE;
      const bool with_new = it.new_row >= y0 && it.new_row < y0 + TILE;
      uint32_t extra = 0;
      if (HEADS > 0 && t == 0) {
        const int h0 = it.hc * HEADS;
        const int nh = min(HEADS, p.group - h0);
        extra += uint32_t(nh) * ROW_BYTES;
      }
      if (with_new) extra += 2 * ROW_BYTES;
      mbar_arrive_expect_tx(bar, STAGE_BYTES + extra);
      if (HEADS > 0 && t == 0) {
        const int h0 = it.hc * HEADS;
        const int nh = min(HEADS, p.group - h0);
        const char* qsrc = static_cast<const char*>(p.q) +
                           (size_t(it.b) * p.h_q + size_t(it.kvh) * p.group + h0) * ROW_BYTES;
        bulk_load(qslots + stage * (HEADS * ROW_BYTES), qsrc, uint32_t(nh) * ROW_BYTES, bar);
      }
      if (with_new) {
        const size_t src = (size_t(it.b) * p.h_kv + it.kvh) * ROW_BYTES;
        bulk_load(newslots + stage * (2 * ROW_BYTES), static_cast<const char*>(p.k_new) + src,
                  ROW_BYTES, bar);
        bulk_load(newslots + stage * (2 * ROW_BYTES) + ROW_BYTES,
                  static_cast<const char*>(p.v_new) + src, ROW_BYTES, bar);
      }
      const uint32_t kdst = ring + stage * STAGE_BYTES;
      const int y = it.row_begin + t * TILE;
#pragma unroll
      for (int h = 0; h < NBOX; ++h) {
        tma_load_3d(kdst + h * BOX_BYTES, tmK, h * BOX_COLS, y, z, bar, policy);
        tma_load_3d(kdst + kTileBytes + h * BOX_BYTES, tmV, h * BOX_COLS, y, z, bar, policy);
      }
      issued |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (aborted) {
    // Let every copy this thread started land before the CTA can exit.
    volatile int never = 0;
    for (int st = 0; st < STAGES; ++st)
      if (issued & (1u << st)) mbar_wait_bounded(full0 + 8 * st, (issued_parity >> st) & 1u, &never);
  }
}

}  // namespace da
