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

#include <atomic>

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
  void* out;                     // [B, h_q, d] float32, or bf16 when out_bf16
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
  // 8-bit caches only: one float32 scale per cached row, [B, h_kv, n_max]
  // (read through tensor maps; the appended row's scale is written here),
  // and the scales of the appended rows, [B, h_kv].
  float* k_scale;
  float* v_scale;
  const float* k_new_scale;
  const float* v_new_scale;
  int append;
  int out_bf16;                  // out holds bf16 (rounded once from the fp32 result)
  // Rows decoded per sequence: [row_off, min(row_lim, seq_lens[b])) (row_off = 0
  // and row_lim >= n_max decode every cached row).  Never combined with append.
  int row_off, row_lim;
  float* lse_out;                // nullable: [B, h_q] natural-log log-sum-exp of the decoded rows
  int B, h_q, h_kv, group;       // group = h_q / h_kv
  int b_offset;                  // first sequence of this launch inside the tensor maps
  int n_max;
  int head_chunks;               // query-head chunks per kv head
  int chunk_fixed;               // > 0: rows per split chosen by the caller
  int balanced;                  // 1: cut all units' rows into one equal piece per CTA
  int* unit_nv;                  // balanced: [units] partial count of each unit (workspace)
  int4* hints;                   // nullable: [gridDim.x] first tiles of each CTA (workspace)
  // Extents for the checked build (set on every launch): elements of `out`
  // in this slice, partial slots (B * h_q * max_splits), rows of K (and V) in
  // the whole cache.
  long long out_elems, part_rows, cache_rows;
  int chunk_min;                 // else: smallest rows per split the device may choose
  int max_splits;                // partial slots per query head (ceil(n_max / chunk))
  float cta_speed;               // one CTA's streaming rate / its even share (split-length model)
  float scale_log2;              // scale * log2(e)
#ifdef DA_TEST_HOOKS
  int withhold_cta;              // test builds: this CTA's producer never fills the last stage
                                 // of its first item (-1: none), so a wait must run out
#endif
};

// Wall-clock limit for any wait inside a kernel.  A pipeline wait that has
// not completed after this long means a copy never landed; the kernel then
// records DA_DEVERR_TIMEOUT and finishes without waiting further.  Test
// builds (DA_TEST_HOOKS) give up after 2 ms so that a test can make a wait
// run out quickly.
#ifdef DA_TEST_HOOKS
constexpr unsigned long long kWaitTimeoutNs = 2ull * 1000ull * 1000ull;
#else
constexpr unsigned long long kWaitTimeoutNs = 1000ull * 1000ull * 1000ull;
#endif

// Test builds only: whether this CTA's producer withholds stage t of its k-th
// item (the last stage of its first item of the CTA the test names).
__device__ __forceinline__ bool test_withhold(const SplitParams& p, int k, int t, int tiles) {
#ifdef DA_TEST_HOOKS
  return int(blockIdx.x) == p.withhold_cta && k == 0 && t == tiles - 1;
#else
  (void)p, (void)k, (void)t, (void)tiles;
  return false;
#endif
}

// ln 2: converts a log2-domain log-sum-exp to the natural log.
constexpr float kLn2 = 0.693147180559945309f;

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

// L2 policy for data a later kernel reads back soon (the split partials,
// which the combine merges after the K/V stream has passed through L2).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// A float store that asks L2 to keep the line (policy from l2_policy_evict_last).
__device__ __forceinline__ void st_keep(float* addr, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(addr), "f"(v), "l"(policy)
               : "memory");
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

// Checked builds (DA_BOUNDS_CHECK; the test build defines it): every index the
// kernels compute from the caller's data for a global or shared-memory access
// is checked against the extent of its buffer first; an index out of range
// sets DA_DEVERR_BOUNDS and the access is skipped (never a trap).  Product
// builds compile the checks away.
#ifdef DA_BOUNDS_CHECK
__device__ __forceinline__ bool in_range(int32_t* dev_error, long long i, long long n) {
  if (i >= 0 && i < n) return true;
  flag_error(dev_error, DA_DEVERR_BOUNDS);
  return false;
}
#else
__device__ __forceinline__ bool in_range(int32_t*, long long, long long) { return true; }
#endif
#define DA_IN(p, i, n) da::in_range((p).dev_error, (long long)(i), (long long)(n))

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

KernelShape bf16_shape(int d_k, int d_v, int group);
KernelShape f32_shape(int d, int group);
KernelShape tc5_shape(int group);
KernelShape q8_shape(int d);
cudaError_t launch_split_q8(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tks, const CUtensorMap& tvs, int d, int kind,
                            int grid, cudaStream_t stream);
cudaError_t launch_kv_quantize(const void* x, int x_bf16, void* codes, float* scales,
                               long long rows, int d, int kind, cudaStream_t stream);
cudaError_t launch_split_tc5(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             int grid, cudaStream_t stream);
cudaError_t launch_split_bf16(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int d_k, int d_v, int grid, cudaStream_t stream);
cudaError_t launch_split_f32(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             int d, int grid, cudaStream_t stream);
// split_grid: the CTAs of the split launch before it (the expected pieces per
// unit of a balanced list).
// Host: whether num_splits = 0 resolves to balanced pieces for this request
// (the allocation-free entry point takes one split instead when those pieces'
// partials do not fit its buffer).
bool library_takes_balanced(int B, int h_q, int h_kv, int d_k, int d_v, int n_max, int dtype);

cudaError_t launch_combine(const SplitParams& p, int d, int heads_per_cta, int split_grid,
                           cudaStream_t stream);
cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int S, void* out,
                             int out_bf16, float* lse_out, long long heads, int d,
                             cudaStream_t stream);
cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* K, void* V,
                             const int32_t* pos, int B, int h_kv, int row_bytes_k,
                             int row_bytes_v, int n_max, const float* ks_new, const float* vs_new,
                             float* ks, float* vs, int32_t* dev_error, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Work list.
//
// Sequence b is cut into nv_b = max(1, ceil(n_b / chunk)) splits of `chunk`
// rows.  Each (kv head, head chunk) of b is a unit; each (unit, split) is a
// work item.  Items are numbered in two runs: first every split but the last
// of every unit (sequence by sequence, unit by unit, split by split), then
// the last split of every unit, which is usually shorter than `chunk`.
// Persistent CTAs take items i = blockIdx.x + k * gridDim.x, so the full
// splits are dealt evenly and the short ones fill the last round.  Every CTA
// builds the same list in shared memory from seq_lens.
// ---------------------------------------------------------------------------
// Shared-memory words of the work list: first[] and lens[] of up to
// kMaxBatchPerLaunch sequences, reduction scratch for up to 16 warps, and the
// decoded items 0 .. kItemCache-1 of the CTA (later items are decoded on the
// fly).  Kernels reserve kSchedWords ints.
constexpr int kItemCache = 64;
constexpr int kItemWords = 8;
constexpr int kSchedRedWords = 16 * 32 + 64;
constexpr int kSchedLens = kMaxBatchPerLaunch + 1;          // offset of lens[]
constexpr int kSchedRed = kSchedLens + kMaxBatchPerLaunch;  // offset of the scratch
constexpr int kSchedItems = (kSchedRed + kSchedRedWords + 3) & ~3;
constexpr int kSchedWords = kSchedItems + kItemCache * kItemWords;

struct Schedule {
  int* w;           // kSchedWords ints of shared memory:
                    //   [0, B]      chunked: first item of sequence b's run of full
                    //               splits (first[B] = F, the items of that run);
                    //               balanced: stream offset of sequence b's rows per
                    //               unit, sum of max(n, 1) over earlier sequences
                    //   kSchedLens  rows to decode per sequence; bit 31 set when
                    //               row (len - 1) is appended now
                    //   kSchedItems this CTA's first items, decoded
  int chunk;        // chunked: rows per split
  int total;        // chunked: items in the list
  int mine;         // items of this CTA
  int balanced;     // 1: items are the units one equal piece of the row stream touches
  int u0;           // balanced: the first unit of this CTA's piece
  int piece;        // balanced: rows per piece before tile alignment
  const int* cuts;  // balanced: the gridDim.x + 1 boundaries, in shared memory
  __device__ __forceinline__ int first(int b) const { return w[b]; }
  __device__ __forceinline__ int lens(int b) const { return w[kSchedLens + b]; }
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
  const int per_seq = p.h_kv * p.head_chunks;
  const int F = s.first(p.B);
  Item it;
  int unit;
  if (i < F) {  // a full split: last b with first[b] <= i (then first[b + 1] > i)
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s.first(mid) <= i) lo = mid; else hi = mid - 1;
    }
    it.b = lo;
    const int full = (s.first(lo + 1) - s.first(lo)) / per_seq;  // nv - 1
    it.nv = full + 1;
    const int r = i - s.first(lo);
    unit = r / full;
    it.split = r - unit * full;
  } else {      // the last split of unit (i - F) % per_seq of sequence (i - F) / per_seq
    const int j = i - F;
    it.b = j / per_seq;
    unit = j - it.b * per_seq;
    const int n = len_of(s.lens(it.b));
    it.nv = n <= 0 ? 1 : (n - 1) / s.chunk + 1;
    it.split = it.nv - 1;
  }
  it.kvh = unit / p.head_chunks;
  it.hc = unit - it.kvh * p.head_chunks;
  const int lv = s.lens(it.b);
  const int n = len_of(lv);
  it.new_row = (lv & kAppendFlag) ? n - 1 : -1;
  it.row_begin = it.split * s.chunk;
  const int end = it.row_begin + s.chunk;
  it.row_end = end < n ? end : n;
  if (it.row_end < it.row_begin) it.row_end = it.row_begin;
  it.tiles = (it.row_end - it.row_begin + TILE - 1) / TILE;
  it.row_begin += p.row_off;  // rows counted from the start of the decoded range
  it.row_end += p.row_off;
  return it;
}

// ---------------------------------------------------------------------------
// Balanced work list.  The rows of every unit, unit after unit (units ordered
// as in the chunked list; an empty sequence counts one row so that its zero
// output is still written), form one stream of R rows.  Boundary c of the
// grid's pieces lies at c * piece, rounded down to a whole tile inside the
// unit it falls in; CTA c takes the rows between boundaries c and c + 1, an
// item for every unit they touch.  Every CTA computes the same boundaries.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int bal_len(const Schedule& s, int b) {
  const int n = len_of(s.lens(b));
  return n > 0 ? n : 1;
}

// Stream positions fit in 32 bits: the host only takes this list when the
// rows of a launch slice number fewer than 2^31, and a boundary c * piece is
// below R + piece < 2^32.

// The unit holding stream position x (0 <= x < R) and the position where it starts.
__device__ __forceinline__ int bal_unit(const SplitParams& p, const Schedule& s, uint32_t x,
                                        uint32_t& start) {
  const uint32_t per_seq = uint32_t(p.h_kv * p.head_chunks);
  int lo = 0, hi = p.B - 1;  // last b with per_seq * first[b] <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (per_seq * uint32_t(s.first(mid)) <= x) lo = mid; else hi = mid - 1;
  }
  const uint32_t len = uint32_t(bal_len(s, lo));
  const uint32_t base = per_seq * uint32_t(s.first(lo));
  const uint32_t j = (x - base) / len;
  start = base + j * len;
  return int(uint32_t(lo) * per_seq + j);
}

// Stream position of boundary c (0 .. gridDim.x), and in `tag` the unit that
// holds the rows from it on, times 2, plus 1 when the boundary is that unit's
// first row (for the last boundary: the unit count, times 2, plus 1).
template <int TILE>
__device__ __forceinline__ uint32_t bal_cut(const SplitParams& p, const Schedule& s, int c,
                                            int& tag) {
  const uint32_t per_seq = uint32_t(p.h_kv * p.head_chunks);
  const uint32_t R = per_seq * uint32_t(s.first(p.B));
  const uint32_t x = uint32_t(c) * uint32_t(s.piece);
  if (c <= 0) {
    tag = 1;  // unit 0, at its first row
    return 0;
  }
  if (x >= R) {
    tag = int(per_seq * uint32_t(p.B)) * 2 + 1;  // past the last unit
    return R;
  }
  uint32_t start;
  const int u = bal_unit(p, s, x, start);
  const uint32_t cut = start + (x - start) / TILE * TILE;
  tag = u * 2 + (cut == start ? 1 : 0);
  return cut;
}

// The item of CTA c on unit u (inlined into the work-list build, where it is
// on every CTA's start-up path; bal_item_far below is the out-of-line copy for
// items decoded on the fly past the item cache).
template <int TILE>
__device__ __forceinline__ Item bal_item(const SplitParams& p, const Schedule& s, int c, int u) {
  const int per_seq = p.h_kv * p.head_chunks;
  const int b = u / per_seq, j = u - (u / per_seq) * per_seq;
  const uint32_t len = uint32_t(bal_len(s, b));
  const uint32_t piece = uint32_t(s.piece);
  const uint32_t U = uint32_t(per_seq) * uint32_t(s.first(b)) + uint32_t(j) * len;
  const uint32_t lo = uint32_t(s.cuts[c]), hi = uint32_t(s.cuts[c + 1]);
  // first CTA whose piece reaches past U; last CTA whose piece starts before U + len
  int c0 = int(U / piece);
  while (c0 + 1 < int(gridDim.x) && uint32_t(s.cuts[c0 + 1]) <= U) ++c0;
  int c1 = int((U + len - 1) / piece);
  if (c1 > int(gridDim.x) - 1) c1 = int(gridDim.x) - 1;
  Item it;
  it.b = b;
  it.kvh = j / p.head_chunks;
  it.hc = j - it.kvh * p.head_chunks;
  it.split = c - c0;
  it.nv = c1 - c0 + 1;
  const int n = len_of(s.lens(b));
  const int beg = int((lo > U ? lo : U) - U);
  int end = int((hi < U + len ? hi : U + len) - U);
  if (end > n) end = n;  // an empty sequence's one stream row holds no data
  it.row_begin = beg < end ? beg : end;
  it.row_end = end;
  const int last = (s.lens(b) & kAppendFlag) ? n - 1 : -1;
  it.new_row = (last >= it.row_begin && last < it.row_end) ? last : -1;
  it.tiles = (it.row_end - it.row_begin + TILE - 1) / TILE;
  it.row_begin += p.row_off;  // rows counted from the start of the decoded range
  it.row_end += p.row_off;
  return it;
}

template <int TILE>
__device__ __noinline__ Item bal_item_far(const SplitParams& p, const Schedule& s, int c, int u) {
  return bal_item<TILE>(p, s, c, u);
}

// The k-th item of this CTA (k < s.mine), read back from shared memory when
// build_schedule decoded it.
template <int TILE>
__device__ __forceinline__ Item cta_item(const SplitParams& p, const Schedule& s, int k) {
  if (k >= kItemCache)
    return s.balanced ? bal_item_far<TILE>(p, s, int(blockIdx.x), s.u0 + k)
                      : schedule_item<TILE>(p, s, int(blockIdx.x) + k * int(gridDim.x));
  const int* w = s.w + kSchedItems + k * kItemWords;
  Item it;
  it.b = w[0];
  it.kvh = w[1];
  it.hc = w[2];
  it.split = w[3];
  it.nv = w[4];
  it.row_begin = w[5];
  it.row_end = w[6];
  it.new_row = w[7];
  it.tiles = (it.row_end - it.row_begin + TILE - 1) / TILE;
  return it;
}

// Choose the split length when the caller left it to the library.  Lane k of
// every warp stands for one candidate length: chunk_min * 2^k for k < 16, and
// for k >= 16 the "balanced" length that cuts the longest sequence into
// (k - 15) * grid / units pieces, so that the items fill whole rounds of the
// grid.  The estimated time in rows streamed by one CTA is the larger of the
// even share of all rows and the busiest CTA's rows divided by how fast one
// CTA can stream relative to its even share (p.cta_speed: above 1 when a lone
// CTA can pull more than its share of HBM bandwidth, below 1 when a CTA is
// compute-bound), plus one tile of epilogue per item and two tiles when
// partials must be merged.  Ties go to more, shorter items.  The item counts
// are summed over the sequences by all warps of the CTA; every reduction runs
// in a fixed order, so every CTA picks the same length.  All threads call this
// with the CTA-wide row total and longest length.
template <int TILE>
__device__ __forceinline__ int choose_chunk(const SplitParams& p, const int* lens, int grid,
                                            float rows, int nmax,
                                            int* red /* shared, kSchedRedWords */) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int longest = nmax > 0 ? nmax : 1;
  const int per_seq = p.h_kv * p.head_chunks;
  const int units = p.B * per_seq;
  const int k = lane;
  uint32_t c;  // candidate length, at most 2^30 (32-bit arithmetic throughout)
  if (k < 16) {
    const unsigned long long c64 = (unsigned long long)p.chunk_min << k;
    c = c64 > (1ull << 30) ? (1u << 30) : uint32_t(c64);
  } else {
    int pieces = (k - 15) * grid / units;
    if (pieces < 1) pieces = 1;
    c = uint32_t(longest / pieces + (longest % pieces != 0));
  }
  c = (c + TILE - 1) / TILE * TILE;
  if (c < uint32_t(p.chunk_min)) c = uint32_t(p.chunk_min);
  if (c > (1u << 30)) c = 1u << 30;
  const int ci = int(c);
  const int tile = TILE;
  // power-of-two candidates stop after the first one covering everything
  const bool candidate = k >= 16 || k == 0 || ((long long)p.chunk_min << (k - 1)) < longest;
  int items = 0;
  if (candidate) {
    int b = warp;
#pragma unroll 4
    for (; b < p.B; b += nwarps) {
      const int n = len_of(lens[b]);
      items += n <= 0 ? 1 : (n - 1) / ci + 1;
    }
  }
  red[warp * 32 + lane] = items;
  __syncthreads();
  if (warp == 0) {
    long long all = 0;
    for (int w = 0; w < nwarps; ++w) all += red[w * 32 + lane];
    float t = 3.0e38f;
    if (candidate) {
      const float fitems = float(all) * float(per_seq);
      const float rounds = ceilf(fitems / float(grid));
      const float share = rows * float(per_seq) / float(grid);
      const float ceff = float(ci < longest ? ci : longest);
      t = fmaxf(share, rounds * ceff / p.cta_speed) + rounds * float(tile);
      if (ci < longest) t += 2.f * float(tile);
    }
    // argmin over lanes; within 0.1% prefer the shorter chunk (more items)
    float best_t = t;
    int best_c = ci;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ot = __shfl_xor_sync(0xffffffffu, best_t, o);
      const int oc = __shfl_xor_sync(0xffffffffu, best_c, o);
      const bool take = oc < best_c ? ot <= best_t * 1.001f
                                    : (oc == best_c ? false : ot * 1.001f < best_t);
      if (take) {
        best_t = ot;
        best_c = oc;
      }
    }
    __syncwarp();
    if (lane == 0) red[kSchedRedWords - 1] = best_c;
  }
  __syncthreads();
  return red[kSchedRedWords - 1];
}

// The same choice made by one warp for a launch slice of at most 32
// sequences: lane b holds n_b (0 for lanes past the batch), and lane k
// evaluates candidate k over every sequence by shuffles, so the choice needs
// no barrier.  `rows` and `nmax` are the slice's row total and longest length,
// the same on every lane.  Every lane returns the chosen length.
template <int TILE>
__device__ __forceinline__ int choose_chunk_warp(const SplitParams& p, int n_lane, int grid,
                                                 float rows, int nmax) {
  const int k = threadIdx.x & 31;
  const int longest = nmax > 0 ? nmax : 1;
  const int per_seq = p.h_kv * p.head_chunks;
  const int units = p.B * per_seq;
  uint32_t c;  // candidate length, as in choose_chunk
  if (k < 16) {
    const unsigned long long c64 = (unsigned long long)p.chunk_min << k;
    c = c64 > (1ull << 30) ? (1u << 30) : uint32_t(c64);
  } else {
    int pieces = (k - 15) * grid / units;
    if (pieces < 1) pieces = 1;
    c = uint32_t(longest / pieces + (longest % pieces != 0));
  }
  c = (c + TILE - 1) / TILE * TILE;
  if (c < uint32_t(p.chunk_min)) c = uint32_t(p.chunk_min);
  if (c > (1u << 30)) c = 1u << 30;
  const int ci = int(c);
  const bool candidate = k >= 16 || k == 0 || ((long long)p.chunk_min << (k - 1)) < longest;
  long long all = 0;
  for (int b = 0; b < p.B; ++b) {  // warp-uniform bound
    const int n = __shfl_sync(0xffffffffu, n_lane, b);
    all += n <= 0 ? 1 : (n - 1) / ci + 1;
  }
  float t = 3.0e38f;
  if (candidate) {
    const float fitems = float(all) * float(per_seq);
    const float rounds = ceilf(fitems / float(grid));
    const float share = rows * float(per_seq) / float(grid);
    const float ceff = float(ci < longest ? ci : longest);
    t = fmaxf(share, rounds * ceff / p.cta_speed) + rounds * float(TILE);
    if (ci < longest) t += 2.f * float(TILE);
  }
  float best_t = t;
  int best_c = ci;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {  // argmin; within 0.1% the shorter length
    const float ot = __shfl_xor_sync(0xffffffffu, best_t, o);
    const int oc = __shfl_xor_sync(0xffffffffu, best_c, o);
    const bool take = oc < best_c ? ot <= best_t * 1.001f
                                  : (oc == best_c ? false : ot * 1.001f < best_t);
    if (take) {
      best_t = ot;
      best_c = oc;
    }
  }
  return best_c;
}

// The rows a sequence contributes to the work list, from its seq_lens value:
// clamped into [0, n_max], plus the appended row when there is room for it
// (kAppendFlag set), else cut to the decoded row range.  `n_out` receives the
// length after the append (the seq_lens_out value).
__device__ __forceinline__ int list_len(const SplitParams& p, int n, bool& bad, bool& bad_pos,
                                        int& n_out) {
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
  n_out = n;
  if (!app) {  // rows of the decoded range (all of them unless a range was asked for)
    n = min(n, p.row_lim) - p.row_off;
    n = n < 0 ? 0 : n;
  }
  return app ? (n | kAppendFlag) : n;
}

// Builds the work list in shared memory; every thread of the CTA must call it.
// `sched` points at kSchedWords ints (16-byte aligned).  It writes nothing
// but shared memory, so it may run before the wait for the previous grid,
// on lengths that grid may still be writing: commit_schedule checks them
// afterwards and builds again if any changed.
template <int TILE>
__device__ __forceinline__ Schedule build_schedule_core(const SplitParams& p, int* sched) {
  int* first = sched;
  int* lens = sched + kSchedLens;
  int* red = sched + kSchedRed;
  int* items = sched + kSchedItems;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  bool bad = false;
  bool bad_pos = false;
  float rows = 0.f;  // only feeds the split-length model; summed in a fixed order
  int nmax = 0;
  int my_n = 0;      // n of sequence tid (the one-warp path: B <= 32)
  for (int b = tid; b < p.B; b += blockDim.x) {
    int n_out;
    const int lv = list_len(p, __ldcg(p.seq_lens + b), bad, bad_pos, n_out);  // through L2
    const int n = len_of(lv);
    lens[b] = lv;
    rows += float(n);
    nmax = n > nmax ? n : nmax;
    my_n = n;
  }
  (void)bad, (void)bad_pos;
  Schedule s;
  s.w = sched;
  s.balanced = 0;
  s.u0 = 0;
  s.piece = 0;
  s.cuts = nullptr;
  s.chunk = 0;
  s.total = 0;
  s.mine = 0;
  const int per_seq = p.h_kv * p.head_chunks;
  if (p.balanced) {
    __syncthreads();  // lens[] complete
    if (tid < 32) {   // stream offsets: exclusive scan of max(n, 1) by warp 0
      int carry = 0;
      for (int base = 0; base < p.B; base += 32) {
        const int b = base + tid;
        const int c = b < p.B ? bal_len(s, b) : 0;
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
    s.balanced = 1;
    const uint32_t R = uint32_t(per_seq) * uint32_t(first[p.B]);
    uint32_t piece = (R + gridDim.x - 1) / gridDim.x;
    if (piece < TILE) piece = TILE;  // so that no two boundaries round to the same row
    s.piece = int(piece);
    // every boundary once, a thread each, into the reduction scratch: the
    // positions in its first half, the tags in its second (gridDim.x + 1 <=
    // kSchedRedWords / 2 words each; the host launches at most that many CTAs)
    int* tags = red + kSchedRedWords / 2;
    for (int c = tid; c <= int(gridDim.x); c += blockDim.x)
      if (DA_IN(p, c, kSchedRedWords / 2)) red[c] = int(bal_cut<TILE>(p, s, c, tags[c]));
    __syncthreads();
    s.cuts = red;
    const uint32_t lo = uint32_t(s.cuts[blockIdx.x]);
    const uint32_t hi = uint32_t(s.cuts[blockIdx.x + 1]);
    if (lo < hi) {
      s.u0 = tags[blockIdx.x] >> 1;  // the unit of row lo
      // the unit of row hi - 1: the one before hi's when hi is a unit's first row
      const int th = tags[blockIdx.x + 1];
      s.mine = (th >> 1) - (th & 1) - s.u0 + 1;
    }
    for (int t = tid; t < s.mine && t < kItemCache; t += blockDim.x) {
      const Item it = bal_item<TILE>(p, s, int(blockIdx.x), s.u0 + t);
      {
        int* w = items + t * kItemWords;
        w[0] = it.b;
        w[1] = it.kvh;
        w[2] = it.hc;
        w[3] = it.split;
        w[4] = it.nv;
        w[5] = it.row_begin;
        w[6] = it.row_end;
        w[7] = it.new_row;
      }
    }
    __syncthreads();
    return s;
  }
  if (p.B <= 32) {
    // One warp: the split length, then the scan of the full splits per
    // sequence, with shuffles only; the other warps wait at one barrier.
    if (warp == 0) {
      float wrows = rows;
      int wmax = nmax;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        wrows += __shfl_xor_sync(0xffffffffu, wrows, o);
        wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
      }
      const int chunk = p.chunk_fixed > 0
                            ? p.chunk_fixed
                            : choose_chunk_warp<TILE>(p, my_n, gridDim.x, wrows, wmax);
      const int c = lane < p.B ? per_seq * (my_n <= 0 ? 0 : (my_n - 1) / chunk) : 0;
      int x = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane < p.B) first[lane] = x - c;
      if (lane == 31) {
        first[p.B] = x;
        red[kSchedRedWords - 1] = chunk;
      }
    }
    __syncthreads();
    s.chunk = red[kSchedRedWords - 1];
  } else if (p.chunk_fixed > 0) {
    __syncthreads();
    s.chunk = p.chunk_fixed;
  } else {
    // CTA-wide row total and longest length, summed in a fixed order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      rows += __shfl_xor_sync(0xffffffffu, rows, o);
      nmax = max(nmax, __shfl_xor_sync(0xffffffffu, nmax, o));
    }
    if (lane == 0) {
      red[16 * 32 + warp] = __float_as_int(rows);
      red[16 * 32 + 32 + warp] = nmax;
    }
    __syncthreads();
    float all_rows = 0.f;
    int all_max = 0;
    for (int w = 0; w < nwarps; ++w) {
      all_rows += __int_as_float(red[16 * 32 + w]);
      all_max = max(all_max, red[16 * 32 + 32 + w]);
    }
    s.chunk = choose_chunk<TILE>(p, lens, gridDim.x, all_rows, all_max, red);
  }
  // exclusive scan of the full-split items per sequence by warp 0
  if (p.B > 32 && tid < 32) {
    int carry = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + tid;
      int c = 0;
      if (b < p.B) {
        const int n = len_of(lens[b]);
        c = per_seq * (n <= 0 ? 0 : (n - 1) / s.chunk);
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
  if (p.B > 32) __syncthreads();
  s.total = first[p.B] + per_seq * p.B;  // and one last split per unit
  // decode this CTA's first items, one per thread
  const int mine = s.total > int(blockIdx.x) ? (s.total - 1 - int(blockIdx.x)) / int(gridDim.x) + 1 : 0;
  s.mine = mine;
  if (tid < mine && tid < kItemCache) {
    const Item it = schedule_item<TILE>(p, s, int(blockIdx.x) + tid * int(gridDim.x));
    int* w = items + tid * kItemWords;
    w[0] = it.b;
    w[1] = it.kvh;
    w[2] = it.hc;
    w[3] = it.split;
    w[4] = it.nv;
    w[5] = it.row_begin;
    w[6] = it.row_end;
    w[7] = it.new_row;
  }
  __syncthreads();
  return s;
}

// After the wait for the previous grid: read seq_lens again (now final), build
// the list again if any length differs from the one it was built on, then
// make the list's global writes: seq_lens_out and the error bits (CTA 0), the
// split length or balanced marker for the combine (CTA 0) and, in balanced
// mode, each unit's partial count (its first CTA).  Every thread must call it.
template <int TILE>
__device__ __forceinline__ Schedule commit_schedule(const SplitParams& p, int* sched,
                                                    Schedule s) {
  const int* lens = sched + kSchedLens;
  const int tid = threadIdx.x;
  bool bad = false, bad_pos = false;
  int changed = 0;
  for (int b = tid; b < p.B; b += blockDim.x) {
    int n_out;
    const int lv = list_len(p, __ldcg(p.seq_lens + b), bad, bad_pos, n_out);
    changed |= lv != lens[b];
    if (blockIdx.x == 0 && p.seq_lens_out && DA_IN(p, b, p.B)) p.seq_lens_out[b] = n_out;
  }
  if (bad && blockIdx.x == 0) flag_error(p.dev_error, DA_DEVERR_SEQ_LEN);
  if (bad_pos && blockIdx.x == 0) flag_error(p.dev_error, DA_DEVERR_POS);
  if (__syncthreads_or(changed)) s = build_schedule_core<TILE>(p, sched);
  if (blockIdx.x == 0 && tid == 0 && p.chunk_out) *p.chunk_out = s.balanced ? -1 : s.chunk;
  if (s.balanced && p.unit_nv)
    for (int t = tid; t < s.mine; t += blockDim.x) {
      const Item it = bal_item<TILE>(p, s, int(blockIdx.x), s.u0 + t);
      if (it.split == 0 && DA_IN(p, s.u0 + t, p.B * p.h_kv * p.head_chunks))
        p.unit_nv[s.u0 + t] = it.nv;  // the unit's first CTA
    }
  return s;
}

// The whole work list when nothing can change under it (a single call).
template <int TILE>
__device__ __forceinline__ Schedule build_schedule(const SplitParams& p, int* sched) {
  return commit_schedule<TILE>(p, sched, build_schedule_core<TILE>(p, sched));
}

// One element of the final output, rounded to bf16 when the caller asked for it.
__device__ __forceinline__ void store_out(const SplitParams& p, size_t idx, float v) {
  if (!DA_IN(p, idx, p.out_elems)) return;
  if (p.out_bf16) static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
  else static_cast<float*>(p.out)[idx] = v;
}

// ---------------------------------------------------------------------------
// End of a work item, shared by the split kernels with consumer warps.
//
// The consumer warps have written, per (key warp, head), their running max m
// (log2 domain), running sum l and unnormalised accumulator into shared
// slots.  This merges the KW key warps of each head group by log-sum-exp and
// writes the item's normalised output: straight to `out` when the sequence
// has a single split, else to its partial slot with its log-sum-exp for the
// combine kernel.  All `nthreads` consumer threads call it together (it
// synchronises them on named barrier 1).
//   Phase A: one thread per head takes the maximum over the KW warps, the
//            weight f_k = 2^(m_k - M) of each warp and the denominator
//            L = sum_k f_k l_k, and leaves f_k in place of m_k and 1 / L in
//            place of the head's first l (no other thread reads them).
//   Phase B: all threads, one output element (head, column) at a time:
//            out = (sum_k f_k acc_k) / L, consecutive threads on consecutive
//            columns.
// ---------------------------------------------------------------------------
template <int D, int HG, int KW, int HPW, int SLOT_STRIDE>
__device__ __forceinline__ void finish_item(const SplitParams& p, const Item& it,
                                            const float* epi_acc, float* epi_m, float* epi_l,
                                            int ctid, int nthreads, volatile int* abort_flag) {
  constexpr int GC = HG * HPW;  // query heads of this item
  static_assert(KW >= 2, "phase A keeps 1 / L in the second l slot");
  const int head0 = it.hc * GC;  // group-local index of the item's first head
  const int nh = min(GC, p.group - head0);
  const size_t bh0 = size_t(it.b) * p.h_q + size_t(it.kvh) * p.group + head0;
  const bool single = it.nv == 1;
  if (ctid < GC) {
    const int h = ctid, hg = h / HPW, hw = h - hg * HPW;
    float m[KW], M = -INFINITY;
#pragma unroll
    for (int k = 0; k < KW; ++k) {
      m[k] = epi_m[(hg * KW + k) * HPW + hw];
      M = fmaxf(M, m[k]);
    }
    const float M_use = M == -INFINITY ? 0.f : M;  // an empty item: every l is 0
    float L = 0.f;
#pragma unroll
    for (int k = 0; k < KW; ++k) {
      const float f = ex2(m[k] - M_use);
      L += f * epi_l[(hg * KW + k) * HPW + hw];
      epi_m[(hg * KW + k) * HPW + hw] = f;
    }
    epi_l[(hg * KW + 1) * HPW + hw] = L > 0.f ? __fdividef(1.f, L) : 0.f;
    if (h < nh && !*abort_flag) {
      const float lse2 = L > 0.f ? M + log2f(L) : -INFINITY;
      if (!single) {
        if (DA_IN(p, (bh0 + h) * p.max_splits + it.split, p.part_rows))
          st_keep(p.lse_part + (bh0 + h) * p.max_splits + it.split, lse2, l2_policy_evict_last());
      } else if (p.lse_out && DA_IN(p, bh0 + h, p.out_elems / D)) {
        p.lse_out[bh0 + h] = lse2 * kLn2;
      }
    }
  }
  named_bar_sync(1, nthreads);
  const size_t stride = single ? size_t(D) : size_t(p.max_splits) * D;
  const size_t base = single ? bh0 * D : (bh0 * p.max_splits + it.split) * D;
  const uint64_t keep = l2_policy_evict_last();  // partials: read back by the combine
  for (int idx = ctid; idx < nh * D; idx += nthreads) {
    const int h = idx / D, d = idx - h * D;
    const int hg = h / HPW, hw = h - hg * HPW;
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < KW; ++k) {
      const int sid = hg * KW + k;
      sum += epi_m[sid * HPW + hw] * epi_acc[(sid * HPW + hw) * SLOT_STRIDE + d];
    }
    const float val = sum * epi_l[(hg * KW + 1) * HPW + hw];
    if (!*abort_flag) {
      if (single) store_out(p, base + h * stride + d, val);
      else if (DA_IN(p, base + h * stride + d, p.part_rows * D))
        st_keep(p.o_part + base + h * stride + d, val, keep);
    }
  }
}

// ---------------------------------------------------------------------------
// First-tile hints.  A decode call usually follows one of the same shape on
// the same workspace (the previous decode step), and a CTA's first tiles are
// then the same rows as last time.  Each CTA leaves the coordinates of its
// first tiles in the workspace; at the next launch its producer reads them
// and asks for those tiles to be brought into L2 before it waits for the
// previous grid and builds its work list (~1.5-4 us in which HBM would
// otherwise idle).  An L2 prefetch is only a hint: L2 stays coherent with
// any later write, so a stale or wrong guess costs bandwidth, never a result.
// Hint words: {z, y0, tiles, check} with check = z ^ y0 ^ tiles ^ kHintSeal.
// ---------------------------------------------------------------------------
constexpr int kHintSeal = 0x5a17c0de;
constexpr int kMaxHintCtas = 1024;

// L2 prefetch of one box of a 3-D tiled tensor map.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// L2 prefetch of one box of a 2-D tiled tensor map.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// This CTA's hint from the previous launch, if it is well formed and inside
// this launch's tensors: rows [y0, y0 + tiles * TILE) of kv head z.  Called
// before griddepcontrol.wait: the words may be stale, never unsafe to use.
// The hint word of this CTA, loaded through L2 without waiting for it: the
// caller issues the load at kernel entry and decodes the value once the work
// list is built, so the load's round trip overlaps the build.
__device__ __forceinline__ int4 load_hint(const SplitParams& p) {
  int4 h = make_int4(0, 0, 0, 0);
  if (p.hints && blockIdx.x < unsigned(kMaxHintCtas))
    asm volatile("ld.global.cg.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(h.x), "=r"(h.y), "=r"(h.z), "=r"(h.w)
                 : "l"(p.hints + blockIdx.x));
  return h;
}

// A hint word written by write_hint for this launch's shapes: its first tiles.
template <int TILE>
__device__ __forceinline__ bool read_hint(const SplitParams& p, int4 h, int max_tiles, int& z,
                                          int& y0, int& tiles) {
  if (!p.hints || blockIdx.x >= unsigned(kMaxHintCtas)) return false;
  z = h.x, y0 = h.y, tiles = h.z;
  if ((h.x ^ h.y ^ h.z ^ kHintSeal) != h.w) return false;
  const int z0 = p.b_offset * p.h_kv, z1 = (p.b_offset + p.B) * p.h_kv;
  if (z < z0 || z >= z1 || y0 < 0 || y0 >= p.n_max || tiles < 1) return false;
  if (tiles > max_tiles) tiles = max_tiles;
  return true;
}

// After the work list is built: record this CTA's first tiles for the next launch.
template <int TILE>
__device__ __forceinline__ void write_hint(const SplitParams& p, const Item& it, int max_tiles) {
  if (!p.hints || blockIdx.x >= unsigned(kMaxHintCtas)) return;
  const int z = (p.b_offset + it.b) * p.h_kv + it.kvh;
  const int y0 = it.row_begin;
  const int tiles = it.tiles < max_tiles ? it.tiles : max_tiles;
  p.hints[blockIdx.x] = make_int4(z, y0, tiles, z ^ y0 ^ tiles ^ kHintSeal);
}

// Producer lane, before waiting for the previous grid: L2 prefetch of the
// hinted tiles of K (NBOX_K boxes of BOX_COLS columns per tile) and V.
template <int TILE, int NBOX_K, int NBOX_V, int BOX_COLS>
__device__ __forceinline__ void prefetch_hinted(const SplitParams& p, int4 hint,
                                                const CUtensorMap* tmK, const CUtensorMap* tmV,
                                                int max_tiles) {
  int z, y0, tiles;
  if (!read_hint<TILE>(p, hint, max_tiles, z, y0, tiles)) return;
  for (int t = 0; t < tiles && y0 + t * TILE < p.n_max; ++t) {
#pragma unroll
    for (int h = 0; h < NBOX_K; ++h) tma_prefetch_3d(tmK, h * BOX_COLS, y0 + t * TILE, z);
#pragma unroll
    for (int h = 0; h < NBOX_V; ++h) tma_prefetch_3d(tmV, h * BOX_COLS, y0 + t * TILE, z);
  }
}

// Fused append: copy the new K and V rows (shared-memory slot, the K row of
// KROW bytes then the V row of VROW bytes) into row `it.new_row` of kv head
// (b_offset + b, kvh) of the caches.  One warp; an exact copy of the bits.
template <int KROW, int VROW>
__device__ __forceinline__ void store_new_row(const SplitParams& p, const Item& it,
                                              const uint8_t* slot, int lane) {
  const size_t head = size_t(p.b_offset + it.b) * p.h_kv + it.kvh;
  const size_t row = head * size_t(p.n_max) + size_t(it.new_row);
  if (!DA_IN(p, row, p.cache_rows) || !DA_IN(p, it.new_row, p.n_max)) return;
  const uint4* ks = reinterpret_cast<const uint4*>(slot);
  const uint4* vs = reinterpret_cast<const uint4*>(slot + KROW);
  uint4* kd = reinterpret_cast<uint4*>(static_cast<char*>(p.k_cache) + row * KROW);
  uint4* vd = reinterpret_cast<uint4*>(static_cast<char*>(p.v_cache) + row * VROW);
  for (int i = lane; i < KROW / 16; i += 32) kd[i] = ks[i];
  for (int i = lane; i < VROW / 16; i += 32) vd[i] = vs[i];
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

// Host: raise a kernel's dynamic shared-memory limit to `smem` on the current
// device, once per device.  `done` holds one bit per device ordinal (< 64);
// each kernel instantiation owns its own word.  Setting it twice is harmless.
template <class... Params>
cudaError_t set_smem_limit_once(void (*kernel)(Params...), size_t smem,
                                std::atomic<unsigned long long>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_relaxed);
  return e;
}

// Host: launch a kernel as a programmatic dependent of the work before it on
// the stream.  It may start while that grid drains (once every CTA of it has
// run griddepcontrol.launch_dependents, or exited) and must execute
// griddepcontrol.wait before it reads anything that grid wrote or writes
// anything it reads.
template <class... Params, class... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), int grid, int threads, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---------------------------------------------------------------------------
// Producer: one thread streams every tile of the CTA's items into the ring.
// A stage holds the K tile (NBOX_K boxes of BOX_COLS columns, BOX_BYTES each)
// and, V_OFFSET bytes in, the V tile (NBOX_V such boxes).  The item's q rows
// (QROW bytes each) ride with its first stage, an appended K row (KROW bytes)
// and V row (VROW bytes) with the stage that holds their position.
// ---------------------------------------------------------------------------
// The query rows of an item (its head chunk of one kv group, contiguous in
// q) ride with the item's first stage into that stage's q slot.
// With a fused append, the new K and V rows of the unit ride with the stage
// that holds the unit's last row, into that stage's new-row slot
// (2 * ROW_BYTES: the K row, then the V row).
template <int TILE, int STAGES, int STAGE_BYTES, int NBOX_K, int NBOX_V, int BOX_COLS,
          int BOX_BYTES, int V_OFFSET, int HEADS, int QROW, int KROW, int VROW>
__device__ __forceinline__ void produce(const CUtensorMap* tmK, const CUtensorMap* tmV,
                                        const SplitParams& p, const Schedule& s, uint32_t ring,
                                        uint32_t qslots, uint32_t newslots, uint32_t full0,
                                        uint32_t empty0, volatile int* abort_flag) {
  prefetch_tmap(tmK);
  prefetch_tmap(tmV);
  const uint64_t policy = l2_policy_evict_first();
  constexpr int kNewSlot = KROW + VROW;
  int stage = 0;
  uint32_t phase = 0, issued = 0, issued_parity = 0;
  bool aborted = false;
  for (int k = 0; k < s.mine && !aborted; ++k) {
    const Item it = cta_item<TILE>(p, s, k);
    const int z = (p.b_offset + it.b) * p.h_kv + it.kvh;
    for (int t = 0; t < it.tiles; ++t) {
      if (!mbar_wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag)) {
        *abort_flag = 1;
        flag_error(p.dev_error, DA_DEVERR_TIMEOUT);
        aborted = true;
        break;
      }
      if (test_withhold(p, k, t, it.tiles)) {  // never filled: its consumers' wait runs out
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        continue;
      }
      const uint32_t bar = full0 + 8 * stage;
      const int y0 = it.row_begin + t * TILE;
      const bool with_new = it.new_row >= y0 && it.new_row < y0 + TILE;
      // the item's q rows and the unit's new rows (checked builds: only from
      // inside their arrays, and only those bytes are expected)
      const int h0 = it.hc * (HEADS > 0 ? HEADS : 1);
      const int nh = HEADS > 0 ? min(HEADS, p.group - h0) : 0;
      const size_t bhq = size_t(it.b) * p.h_q + size_t(it.kvh) * p.group + h0;
      const bool load_q = HEADS > 0 && t == 0 && DA_IN(p, bhq + nh - 1, size_t(p.B) * p.h_q);
      const size_t src = size_t(it.b) * p.h_kv + it.kvh;
      const bool load_new = with_new && DA_IN(p, src, size_t(p.B) * p.h_kv);
      uint32_t extra = 0;
      if (load_q) extra += uint32_t(nh) * QROW;
      if (load_new) extra += KROW + VROW;
      mbar_arrive_expect_tx(bar, STAGE_BYTES + extra);
      if (load_q)
        bulk_load(qslots + stage * (HEADS * QROW), static_cast<const char*>(p.q) + bhq * QROW,
                  uint32_t(nh) * QROW, bar);
      if (load_new) {
        bulk_load(newslots + stage * kNewSlot, static_cast<const char*>(p.k_new) + src * KROW,
                  KROW, bar);
        bulk_load(newslots + stage * kNewSlot + KROW,
                  static_cast<const char*>(p.v_new) + src * VROW, VROW, bar);
      }
      const uint32_t kdst = ring + stage * STAGE_BYTES;
      const int y = it.row_begin + t * TILE;
#pragma unroll
      for (int h = 0; h < NBOX_K; ++h)
        tma_load_3d(kdst + h * BOX_BYTES, tmK, h * BOX_COLS, y, z, bar, policy);
#pragma unroll
      for (int h = 0; h < NBOX_V; ++h)
        tma_load_3d(kdst + V_OFFSET + h * BOX_BYTES, tmV, h * BOX_COLS, y, z, bar, policy);
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
