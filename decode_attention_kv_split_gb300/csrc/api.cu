// Host side of the C ABI declared in include/decode_attn.h: argument checks,
// split planning, TMA descriptor encoding, workspace handling and launches.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"

namespace {

using da::KernelShape;
using da::SplitParams;

std::atomic<uint64_t> g_launches{0};
#ifdef DA_TEST_HOOKS
std::atomic<int> g_test_withhold_cta{-1};  // test builds: see decode_attn_test_withhold
#endif
thread_local char g_last_cuda_error[256] = "";

int fail_cuda(cudaError_t e, const char* what) {
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%d)", what,
           cudaGetErrorString(e), int(e));
  return DA_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Device properties, cached per device ordinal.
// ---------------------------------------------------------------------------
struct DeviceInfo {
  int checked = 0;
  int ok = 0;
  int sms = 0;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int current_device(int* dev, int* sms) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return DA_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& di = g_dev[*dev];
  if (!di.checked) {
    int major = 0, minor = 0, count = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, *dev)) != cudaSuccess)
      return fail_cuda(e, "cudaDeviceGetAttribute");
    di.ok = (major == 10 && minor == 3);
    di.sms = count;
    di.checked = 1;
  }
  *sms = di.sms;
  return di.ok ? DA_OK : DA_ERR_DEVICE;
}

// ---------------------------------------------------------------------------
// Tensor-map encoding through the driver entry point (no libcuda link).
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

int get_encoder(EncodeTiledFn* fn) {
  std::call_once(g_encode_once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                    cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!g_encode) return fail_cuda(g_encode_err == cudaSuccess ? cudaErrorNotSupported : g_encode_err,
                                  "cuTensorMapEncodeTiled entry point");
  *fn = g_encode;
  return DA_OK;
}

// Recently encoded descriptors: decode steps reuse the same caches, and an
// encode costs more host time than the rest of a call.
struct MapCacheEntry {
  const void* base;
  int dtype, d, n_max, heads, rows, cols, swz;
  CUtensorMap map;
};
constexpr int kMapCacheSize = 32;
MapCacheEntry g_map_cache[kMapCacheSize];
int g_map_cache_next = 0;
std::mutex g_map_mu;

int encode_cache_map_uncached(CUtensorMap* map, const void* base, int dtype, int d, int n_max,
                              int heads, const KernelShape& ks);

// Bytes per cached element of a cache type; kScaleMap marks the tensor map
// of an 8-bit cache's row scales.
constexpr int kScaleMap = 100;
int elem_size(int dtype) { return dtype == DA_FP32 ? 4 : dtype == DA_BF16 ? 2 : 1; }
bool is_q8(int dtype) { return dtype == DA_INT8 || dtype == DA_FP8_E4M3; }

// A [rows_total = B*h_kv heads][n_max][d] cache viewed as a 3-D tensor
// (innermost first): x = column, y = row inside a head, z = b*h_kv + head.
int encode_cache_map(CUtensorMap* map, const void* base, int dtype, int d, int n_max, int heads,
                     const KernelShape& ks) {
  std::lock_guard<std::mutex> lk(g_map_mu);
  for (int i = 0; i < kMapCacheSize; ++i) {
    const MapCacheEntry& e = g_map_cache[i];
    if (e.base == base && e.dtype == dtype && e.d == d && e.n_max == n_max && e.heads == heads &&
        e.rows == ks.tile_rows && e.cols == ks.box_cols && e.swz == ks.swizzle128) {
      *map = e.map;
      return DA_OK;
    }
  }
  const int st = encode_cache_map_uncached(map, base, dtype, d, n_max, heads, ks);
  if (st == DA_OK) {
    MapCacheEntry& e = g_map_cache[g_map_cache_next];
    g_map_cache_next = (g_map_cache_next + 1) % kMapCacheSize;
    e = MapCacheEntry{base, dtype, d, n_max, heads, ks.tile_rows, ks.box_cols, ks.swizzle128, *map};
  }
  return st;
}

int encode_cache_map_uncached(CUtensorMap* map, const void* base, int dtype, int d, int n_max,
                              int heads, const KernelShape& ks) {
  EncodeTiledFn fn;
  int st = get_encoder(&fn);
  if (st != DA_OK) return st;
  CUresult r;
  const cuuint32_t estr[3] = {1, 1, 1};
  if (dtype == kScaleMap) {
    // row scales [heads][n_max] float32, one row of the tile per element
    const cuuint64_t dims[2] = {cuuint64_t(n_max), cuuint64_t(heads)};
    const cuuint64_t strides[1] = {cuuint64_t(n_max) * 4};
    const cuuint32_t box[2] = {cuuint32_t(ks.tile_rows), 1};
    r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const int es = elem_size(dtype);
    const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(n_max), cuuint64_t(heads)};
    const cuuint64_t strides[2] = {cuuint64_t(d) * es, cuuint64_t(n_max) * d * es};
    const cuuint32_t box[3] = {cuuint32_t(ks.box_cols), cuuint32_t(ks.tile_rows), 1};
    const CUtensorMapDataType ty = dtype == DA_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : dtype == DA_FP32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                      : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    r = fn(map, ty, 3, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE,
           ks.swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "cuTensorMapEncodeTiled failed (%d)",
             int(r));
    return DA_ERR_CUDA;
  }
  return DA_OK;
}

// ---------------------------------------------------------------------------
// Argument checks and split planning.
// ---------------------------------------------------------------------------
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The element type of q, K, V and whether `out` is bf16, from a dtype argument.
struct DtypeArg {
  int kv;        // DA_FP32 or DA_BF16
  bool out_bf16;
};
bool parse_dtype(int dtype, DtypeArg* a) {
  a->kv = dtype & 0xff;
  a->out_bf16 = (dtype & DA_OUT_BF16) != 0;
  return (dtype & ~(0xff | DA_OUT_BF16)) == 0 &&
         (a->kv == DA_FP32 || a->kv == DA_BF16 || a->kv == DA_INT8 || a->kv == DA_FP8_E4M3);
}

int check_sizes(int B, int h_q, int h_kv, int d_k, int d_v, int n_max, int dtype) {
  DtypeArg dt;
  if (!parse_dtype(dtype, &dt)) return DA_ERR_DTYPE;
  if (B <= 0 || h_q <= 0 || h_kv <= 0 || n_max <= 0) return DA_ERR_SHAPE;
  if (h_q % h_kv != 0) return DA_ERR_SHAPE;
  if (n_max > (1 << 30)) return DA_ERR_SHAPE;
  if ((long long)B * h_kv * (long long)n_max > 0x7fffffffLL) return DA_ERR_SHAPE;
  if ((long long)B * h_q > 0x7fffffffLL) return DA_ERR_SHAPE;
  // (d_k, d_v) pairs with kernels: 64/64 and 128/128 for every cache type;
  // 256/256 and 192/128 for bf16 caches
  const bool common = (d_k == 64 || d_k == 128) && d_v == d_k;
  const bool wide = dt.kv == DA_BF16 && ((d_k == 256 && d_v == 256) || (d_k == 192 && d_v == 128));
  if (!common && !wide) return DA_ERR_UNSUPPORTED;
  if (is_q8(dt.kv) && n_max % 4 != 0) return DA_ERR_SHAPE;  // row-scale tensor map stride
  return DA_OK;
}

struct Plan {
  KernelShape ks;
  bool tc5;            // bf16, d = 128, group > 8: the tcgen05 kernel
  int head_chunks;
  int chunk_fixed;     // > 0: rows per split fixed by the caller's num_splits
  int chunk_min;       // else: the device picks chunk_min * 2^k
  int max_splits;      // partial slots per query head
  int batch_per_launch;
  bool balanced;       // num_splits = -1: one equal piece of all rows per CTA
  int units;           // (sequence, kv head, head chunk) units of one launch slice
};

// The device-side cost model (choose_chunk) evaluated with every sequence at
// n_max: if even full-length sequences are best served by one split, shorter
// ones are too, and the launch needs neither partials nor a combine.
bool single_split_suffices(long long units, int n_max, int chunk_min, int tile, int sms,
                           float cta_speed) {
  const long long grid = sms;  // the device model uses the whole persistent grid
  const double share = double(n_max) * double(units) / double(grid);
  double best_t = 1e300;
  long long best_c = chunk_min;
  for (int k = 0; k < 32; ++k) {
    long long c;
    if (k < 16) {
      c = (long long)chunk_min << k;
      if (k > 0 && ((long long)chunk_min << (k - 1)) >= n_max) continue;
    } else {
      long long pieces = (long long)(k - 15) * grid / units;
      if (pieces < 1) pieces = 1;
      c = (n_max + pieces - 1) / pieces;
    }
    c = (c + tile - 1) / tile * tile;
    if (c < chunk_min) c = chunk_min;
    const long long per_seq_items = (n_max + c - 1) / c;
    const double items = double(per_seq_items) * double(units);
    const double rounds = ceil(items / double(grid));
    const double ceff = double(c < n_max ? c : n_max);
    double t = fmax(share, rounds * ceff / cta_speed) + rounds * tile;
    if (c < n_max) t += 2.0 * tile;
    if (t < best_t * 0.999 || (t <= best_t * 1.001 && c < best_c)) {
      best_t = t;
      best_c = c;
    }
  }
  return best_c >= n_max;
}

// Splits per sequence requested by the caller -> a split length that is a
// whole number of pipeline stages, as close as possible to n_max / S.  When
// the library chooses, the device picks the length from the actual sequence
// lengths; the host only bounds it from below so that the partial outputs of
// at most about 4 x SMs work items per launch need workspace.
int make_plan(int B, int h_q, int h_kv, int d, int d_v, int n_max, int dtype_arg, int requested,
              int sms, Plan* pl, bool balance_rule = true) {
  const int dtype = dtype_arg & 0xff;
  const int group = h_q / h_kv;
  pl->tc5 = dtype == DA_BF16 && d == 128 && d_v == 128 && group > 8;
  pl->ks = pl->tc5 ? da::tc5_shape(group)
           : is_q8(dtype) ? da::q8_shape(d)
                          : (dtype == DA_BF16 ? da::bf16_shape(d, d_v, group)
                                              : da::f32_shape(d, group));
  pl->head_chunks = (group + pl->ks.heads_per_cta - 1) / pl->ks.heads_per_cta;
  pl->batch_per_launch = B < da::kMaxBatchPerLaunch ? B : da::kMaxBatchPerLaunch;
  const long long tile = pl->ks.tile_rows;
  const long long max_tiles = (n_max + tile - 1) / tile;
  pl->balanced = false;
  pl->units = int((long long)pl->batch_per_launch * h_kv * pl->head_chunks);
  if (requested < -1) return DA_ERR_SHAPE;
  // Balanced pieces when the row stream fits an int and the partials of up
  // to one per SM per query head stay within 256 MiB.
  auto take_balanced = [&]() {
    const long long stream_rows = (long long)pl->units * n_max;
    const long long part_bytes = (long long)pl->batch_per_launch * h_q * sms * (d_v + 1) * 4;
    if (stream_rows >= (1LL << 31) || part_bytes > (256LL << 20)) return false;
    pl->balanced = true;
    pl->chunk_fixed = 0;
    pl->chunk_min = int(tile);
    pl->max_splits = sms;  // a unit has at most one piece per CTA
    return true;
  };
  if (requested == -1) {
    if (take_balanced()) return DA_OK;
    requested = 0;  // otherwise the library's usual choice
  }
  if (requested > 0) {
    long long tiles = (n_max + (long long)requested * tile / 2) / ((long long)requested * tile);
    if (tiles < 1) tiles = 1;
    pl->chunk_fixed = int(tiles * tile);
    pl->chunk_min = pl->chunk_fixed;
  } else {
    const long long units = (long long)pl->batch_per_launch * h_kv * pl->head_chunks;
    long long cap = (4LL * sms + units - 1) / units;
    if (cap > max_tiles) cap = max_tiles;
    if (cap < 1) cap = 1;
    const long long per = (n_max + cap - 1) / cap;
    pl->chunk_fixed = 0;
    pl->chunk_min = int((per + tile - 1) / tile * tile);
    if (single_split_suffices(units, n_max, pl->chunk_min, int(tile), sms, pl->ks.cta_speed)) {
      // One split per unit needs no partials and no combine, but when the
      // units fill the grid's rounds unevenly (fewer units than CTAs, or a
      // ragged last round) the CTAs without a unit idle while the longest
      // sequences stream.  Then balanced pieces, if each CTA's share is at
      // least 8 tiles (below that the merge costs more than the idle SMs).
      const long long rounds = (units + sms - 1) / sms;
      const bool uneven = double(units) < 0.9 * double(rounds * sms);
      const bool sizeable = units * (long long)n_max >= 8LL * tile * sms;
      if (balance_rule && uneven && sizeable && take_balanced()) return DA_OK;
      pl->chunk_fixed = int(max_tiles * tile);  // one split: no partials, no combine
      pl->chunk_min = pl->chunk_fixed;
    }
  }
  const long long splits = (n_max + pl->chunk_min - 1) / pl->chunk_min;
  if (splits >= (1 << 20)) return DA_ERR_SHAPE;
  pl->max_splits = int(splits);
  if ((long long)pl->batch_per_launch * h_q * pl->max_splits * (d_v + 1) > (1LL << 40))
    return DA_ERR_SHAPE;
  return DA_OK;
}

// Workspace of one launch: a header word (the split length the kernels
// used), partial outputs, partial log-sum-exps.
struct WorkspaceLayout {
  size_t header, o_part, lse_part, hints, total;
};

WorkspaceLayout workspace_layout(const Plan& pl, int h_q, int d) {
  WorkspaceLayout w{0, 0, 0, 0, 0};
  if (pl.max_splits <= 1) return w;
  const size_t heads = size_t(pl.batch_per_launch) * h_q;
  w.header = 0;
  // header word; in balanced mode the per-unit partial counts follow it
  w.o_part = pl.balanced ? 256 + (size_t(pl.units) * 4 + 255) / 256 * 256 : 256;
  w.lse_part = w.o_part + heads * pl.max_splits * d * sizeof(float);
  // then each CTA's first-tile hint for the next call (16 bytes per CTA)
  w.hints = (w.lse_part + heads * pl.max_splits * sizeof(float) + 255) / 256 * 256;
  w.total = w.hints + size_t(da::kMaxHintCtas) * 16;
  return w;
}

// Library-owned workspace for decode_attn(), one per device.
struct OwnedWorkspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};
OwnedWorkspace g_ws[kMaxDevices];
std::mutex g_ws_mu;

// Row scales of an 8-bit cache (and of the appended rows, for a fused append).
struct QuantArgs {
  float* k_scale;
  float* v_scale;
  const float* k_new_scale;
  const float* v_new_scale;
};

int run_decode(const void* q, const void* K, const void* V, const int32_t* seq_lens,
                      void* out, int B, int h_q, int h_kv, int d_k, int d_v, int n_max,
                      float scale, int dtype_arg, int num_splits, void* workspace,
                      size_t workspace_bytes, int32_t* dev_error, cudaStream_t stream,
                      const void* k_new, const void* v_new, int32_t* seq_lens_out,
                      const QuantArgs* qa, int row_off = 0, int row_lim = 0x7fffffff,
                      float* lse_out = nullptr) {
  if (!q || !K || !V || !seq_lens || !out) return DA_ERR_NULL;
  int st = check_sizes(B, h_q, h_kv, d_k, d_v, n_max, dtype_arg);
  if (st != DA_OK) return st;
  DtypeArg dta;
  parse_dtype(dtype_arg, &dta);
  const int dtype = dta.kv;
  // 8-bit caches go through the entry points that carry their row scales
  if (is_q8(dtype) != (qa != nullptr)) return DA_ERR_DTYPE;
  if (qa && (!qa->k_scale || !qa->v_scale || (k_new && (!qa->k_new_scale || !qa->v_new_scale))))
    return DA_ERR_NULL;
  if (qa && (!aligned16(qa->k_scale) || !aligned16(qa->v_scale))) return DA_ERR_ALIGN;
  // a row range starts the 8-bit row-scale tiles off their 16-byte grid
  if (qa && row_off != 0) return DA_ERR_UNSUPPORTED;
  if (k_new && (row_off != 0 || row_lim < n_max)) return DA_ERR_SHAPE;
  if (!isfinite(scale)) return DA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out) ||
      (workspace && !aligned16(workspace)))
    return DA_ERR_ALIGN;
  int dev, sms;
  if ((st = current_device(&dev, &sms)) != DA_OK) return st;
  Plan pl;
  if ((st = make_plan(B, h_q, h_kv, d_k, d_v, n_max, dtype, num_splits, sms, &pl)) != DA_OK)
    return st;
  const size_t out_es = dta.out_bf16 ? 2 : 4;
  const WorkspaceLayout wl = workspace_layout(pl, h_q, d_v);
  if (wl.total > 0 && (!workspace || workspace_bytes < wl.total)) return DA_ERR_WORKSPACE;

  CUtensorMap tk, tv, tks, tvs;
  if ((st = encode_cache_map(&tk, K, dtype, d_k, n_max, B * h_kv, pl.ks)) != DA_OK) return st;
  if ((st = encode_cache_map(&tv, V, dtype, d_v, n_max, B * h_kv, pl.ks)) != DA_OK) return st;
  if (qa) {
    if ((st = encode_cache_map(&tks, qa->k_scale, kScaleMap, 1, n_max, B * h_kv, pl.ks)) != DA_OK)
      return st;
    if ((st = encode_cache_map(&tvs, qa->v_scale, kScaleMap, 1, n_max, B * h_kv, pl.ks)) != DA_OK)
      return st;
  }

  const int es = elem_size(dtype);          // cached (and appended) elements
  const int q_es = qa ? 2 : es;             // q is bf16 with an 8-bit cache
  char* ws = static_cast<char*>(workspace);
  for (int b0 = 0; b0 < B; b0 += pl.batch_per_launch) {
    const int bn = (B - b0) < pl.batch_per_launch ? (B - b0) : pl.batch_per_launch;
    SplitParams p;
    p.q = static_cast<const char*>(q) + size_t(b0) * h_q * d_k * q_es;
    p.seq_lens = seq_lens + b0;
    p.out = static_cast<char*>(out) + size_t(b0) * h_q * d_v * out_es;
    p.out_bf16 = dta.out_bf16 ? 1 : 0;
    p.row_off = row_off;
    p.row_lim = row_lim;
    p.lse_out = lse_out ? lse_out + size_t(b0) * h_q : nullptr;
    p.o_part = wl.total ? reinterpret_cast<float*>(ws + wl.o_part) : nullptr;
    p.lse_part = wl.total ? reinterpret_cast<float*>(ws + wl.lse_part) : nullptr;
    p.chunk_out = wl.total ? reinterpret_cast<int*>(ws + wl.header) : nullptr;
    p.balanced = pl.balanced ? 1 : 0;
    p.unit_nv = pl.balanced ? reinterpret_cast<int*>(ws + 256) : nullptr;
    p.hints = wl.total ? reinterpret_cast<int4*>(ws + wl.hints) : nullptr;
    p.out_elems = (long long)bn * h_q * d_v;
    p.part_rows = wl.total ? (long long)bn * h_q * pl.max_splits : 0;
    p.cache_rows = (long long)B * h_kv * n_max;
    p.dev_error = dev_error;
    p.append = k_new != nullptr;
    p.k_new = k_new ? static_cast<const char*>(k_new) + size_t(b0) * h_kv * d_k * es : nullptr;
    p.v_new = v_new ? static_cast<const char*>(v_new) + size_t(b0) * h_kv * d_v * es : nullptr;
    p.k_cache = const_cast<void*>(K);
    p.v_cache = const_cast<void*>(V);
    p.seq_lens_out = seq_lens_out ? seq_lens_out + b0 : nullptr;
    p.k_scale = qa ? qa->k_scale : nullptr;
    p.v_scale = qa ? qa->v_scale : nullptr;
    p.k_new_scale = qa && qa->k_new_scale ? qa->k_new_scale + size_t(b0) * h_kv : nullptr;
    p.v_new_scale = qa && qa->v_new_scale ? qa->v_new_scale + size_t(b0) * h_kv : nullptr;
    p.B = bn;
    p.h_q = h_q;
    p.h_kv = h_kv;
    p.group = h_q / h_kv;
    p.b_offset = b0;
    p.n_max = n_max;
    p.head_chunks = pl.head_chunks;
    p.chunk_fixed = pl.chunk_fixed;
    p.chunk_min = pl.chunk_min;
    p.max_splits = pl.max_splits;
    p.cta_speed = pl.ks.cta_speed;
    p.scale_log2 = float(double(scale) * 1.4426950408889634);  // log2(e) = 1 / ln 2
#ifdef DA_TEST_HOOKS
    p.withhold_cta = b0 == 0 ? g_test_withhold_cta.load() : -1;
#endif
    const long long items = (long long)bn * h_kv * pl.head_chunks * pl.max_splits;
    // one persistent CTA per SM (the balanced list keeps a boundary and a unit
    // tag per CTA in the two halves of the work list's reduction scratch)
    const long long max_grid = da::kSchedRedWords / 2 - 1;
    const long long grid_cap = sms < max_grid ? sms : max_grid;
    const int grid = int(items < grid_cap ? items : grid_cap);
    cudaError_t err =
        pl.tc5 ? da::launch_split_tc5(p, tk, tv, grid, stream)
        : qa   ? da::launch_split_q8(p, tk, tv, tks, tvs, d_k, dtype == DA_INT8 ? 1 : 2, grid, stream)
        : dtype == DA_BF16 ? da::launch_split_bf16(p, tk, tv, d_k, d_v, grid, stream)
                           : da::launch_split_f32(p, tk, tv, d_k, grid, stream);
    if (err != cudaSuccess) return fail_cuda(err, "split kernel launch");
    g_launches.fetch_add(1);
    if (wl.total) {
      err = da::launch_combine(p, d_v, pl.ks.heads_per_cta, grid, stream);
      if (err != cudaSuccess) return fail_cuda(err, "combine kernel launch");
      g_launches.fetch_add(1);
    }
  }
  return DA_OK;
}


}  // namespace

namespace da {
// Whether the library's own split choice (num_splits = 0) takes balanced
// pieces by the uneven-grid rule of make_plan for this request.
bool library_takes_balanced(int B, int h_q, int h_kv, int d_k, int d_v, int n_max, int dtype) {
  if (check_sizes(B, h_q, h_kv, d_k, d_v, n_max, dtype) != DA_OK) return false;
  int dev = 0, sms = 0;
  if (current_device(&dev, &sms) != DA_OK) return false;
  Plan pl;
  if (make_plan(B, h_q, h_kv, d_k, d_v, n_max, dtype, 0, sms, &pl) != DA_OK) return false;
  return pl.balanced;
}
}  // namespace da

extern "C" {

const char* decode_attn_status_string(int status) {
  switch (status) {
    case DA_OK: return "ok";
    case DA_ERR_NULL: return "null pointer argument";
    case DA_ERR_SHAPE: return "size out of range or inconsistent";
    case DA_ERR_DTYPE: return "unknown dtype";
    case DA_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case DA_ERR_WORKSPACE: return "workspace missing or too small";
    case DA_ERR_CUDA: return "CUDA call failed";
    case DA_ERR_DEVICE: return "current device is not sm_103 (GB300)";
    case DA_ERR_UNSUPPORTED: return "unsupported head dimension combination";
    default: return "unknown status";
  }
}

const char* decode_attn_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t decode_attn_launch_count(void) { return g_launches.load(); }

#ifdef DA_TEST_HOOKS
// Test builds only (not part of the product library or its header): from the
// next decode call on, the producer of split-kernel CTA `cta` never fills the
// last pipeline stage of its first work item, so that a consumer's bounded
// wait runs out (2 ms in test builds) and the kernel takes its timeout path.
// -1 turns it off.
__attribute__((visibility("default"))) void decode_attn_test_withhold(int cta) {
  g_test_withhold_cta.store(cta);
}
#endif

int decode_attn_resolve_splits(int B, int h_q, int h_kv, int d_k, int d_v, int n_max, int dtype,
                               int num_splits) {
  int st = check_sizes(B, h_q, h_kv, d_k, d_v, n_max, dtype);
  if (st != DA_OK) return st;
  int dev, sms;
  if ((st = current_device(&dev, &sms)) != DA_OK) return st;
  Plan pl;
  if ((st = make_plan(B, h_q, h_kv, d_k, d_v, n_max, dtype, num_splits, sms, &pl)) != DA_OK)
    return st;
  return pl.max_splits;
}

size_t decode_attn_workspace_bytes(int B, int h_q, int h_kv, int d_k, int d_v, int n_max, int dtype,
                                   int num_splits, int* status) {
  int st = check_sizes(B, h_q, h_kv, d_k, d_v, n_max, dtype);
  int dev = 0, sms = 0;
  Plan pl;
  if (st == DA_OK) st = current_device(&dev, &sms);
  if (st == DA_OK) st = make_plan(B, h_q, h_kv, d_k, d_v, n_max, dtype, num_splits, sms, &pl);
  if (status) *status = st;
  return st == DA_OK ? workspace_layout(pl, h_q, d_v).total : 0;
}

int decode_attn_ex(const void* q, const void* K, const void* V, const int32_t* seq_lens, void* out,
                   int B, int h_q, int h_kv, int d_k, int d_v, int n_max, float scale, int dtype,
                   int num_splits, void* workspace, size_t workspace_bytes, int32_t* dev_error,
                   cudaStream_t stream) {
  return run_decode(q, K, V, seq_lens, out, B, h_q, h_kv, d_k, d_v, n_max, scale, dtype,
                    num_splits, workspace, workspace_bytes, dev_error, stream, nullptr, nullptr,
                    nullptr, nullptr);
}

int decode_attn_append(const void* q, const void* k_new, const void* v_new, void* K, void* V,
                       const int32_t* seq_lens, int32_t* seq_lens_out, void* out, int B, int h_q,
                       int h_kv, int d_k, int d_v, int n_max, float scale, int dtype,
                       int num_splits, void* workspace, size_t workspace_bytes,
                       int32_t* dev_error, cudaStream_t stream) {
  if (!k_new || !v_new) return DA_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new)) return DA_ERR_ALIGN;
  if (seq_lens_out && seq_lens_out == seq_lens) return DA_ERR_SHAPE;
  return run_decode(q, K, V, seq_lens, out, B, h_q, h_kv, d_k, d_v, n_max, scale, dtype,
                    num_splits, workspace, workspace_bytes, dev_error, stream, k_new, v_new,
                    seq_lens_out, nullptr);
}

int decode_attn_partial(const void* q, const void* K, const void* V, const int32_t* seq_lens,
                        int row_begin, int row_end, float* o, float* lse, int B, int h_q,
                        int h_kv, int d_k, int d_v, int n_max, float scale, int dtype,
                        int num_splits, void* workspace, size_t workspace_bytes,
                        int32_t* dev_error, cudaStream_t stream) {
  if (!lse) return DA_ERR_NULL;
  if ((dtype & DA_OUT_BF16) != 0) return DA_ERR_DTYPE;  // partials are float32
  if (row_begin < 0 || row_end < row_begin) return DA_ERR_SHAPE;
  return run_decode(q, K, V, seq_lens, o, B, h_q, h_kv, d_k, d_v, n_max, scale, dtype,
                    num_splits, workspace, workspace_bytes, dev_error, stream, nullptr, nullptr,
                    nullptr, nullptr, row_begin, row_end, lse);
}

int decode_attn_combine(const float* o_parts, const float* lse_parts, int S, void* out,
                        float* lse_out, int B, int h_q, int d_v, int out_dtype,
                        cudaStream_t stream) {
  if (S < 0 || B <= 0 || h_q <= 0) return DA_ERR_SHAPE;
  if (!out || (S > 0 && (!o_parts || !lse_parts))) return DA_ERR_NULL;  // S = 0 reads neither
  if (d_v != 64 && d_v != 128 && d_v != 256) return DA_ERR_UNSUPPORTED;
  if (out_dtype != DA_FP32 && out_dtype != (DA_FP32 | DA_OUT_BF16)) return DA_ERR_DTYPE;
  const long long heads = (long long)B * h_q;
  if (heads > (1LL << 36) || (long long)S * heads * d_v > (1LL << 46)) return DA_ERR_SHAPE;
  if (!aligned16(o_parts) || !aligned16(out)) return DA_ERR_ALIGN;
  int dev, sms;
  int st = current_device(&dev, &sms);
  if (st != DA_OK) return st;
  cudaError_t e = da::launch_lse_merge(o_parts, lse_parts, S, out, (out_dtype & DA_OUT_BF16) ? 1 : 0,
                                       lse_out, heads, d_v, stream);
  if (e != cudaSuccess) return fail_cuda(e, "lse merge launch");
  g_launches.fetch_add(1);
  return DA_OK;
}

int decode_attn(const void* q, const void* K, const void* V, const int32_t* seq_lens, void* out,
                int B, int h_q, int h_kv, int d_k, int d_v, int n_max, float scale, int dtype,
                cudaStream_t stream) {
  if (!q || !K || !V || !seq_lens || !out) return DA_ERR_NULL;
  int st = DA_OK;
  const size_t need =
      decode_attn_workspace_bytes(B, h_q, h_kv, d_k, d_v, n_max, dtype, 0, &st);
  if (st != DA_OK) return st;
  void* ws = nullptr;
  // Held through the launch so that a concurrent growth cannot free the
  // buffer between taking its address and enqueueing the kernels.
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (need > 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return DA_ERR_DEVICE;
    OwnedWorkspace& w = g_ws[dev];
    if (w.bytes < need) {
      if (w.ptr) {
        e = cudaFree(w.ptr);  // waits for work still using the old buffer
        w.ptr = nullptr;
        w.bytes = 0;
        if (e != cudaSuccess) return fail_cuda(e, "cudaFree(workspace)");
      }
      e = cudaMalloc(&w.ptr, need);
      if (e != cudaSuccess) {
        w.ptr = nullptr;
        return fail_cuda(e, "cudaMalloc(workspace)");
      }
      w.bytes = need;
    }
    ws = w.ptr;
  }
  return decode_attn_ex(q, K, V, seq_lens, out, B, h_q, h_kv, d_k, d_v, n_max, scale, dtype, 0, ws,
                        need, nullptr, stream);
}

namespace {
int append_rows(const void* k_new, const void* v_new, void* K, void* V, const int32_t* pos, int B,
                int h_kv, int d_k, int d_v, int n_max, int dtype, const float* ks_new,
                const float* vs_new, float* ks, float* vs, int32_t* dev_error,
                cudaStream_t stream) {
  if (!k_new || !v_new || !K || !V || !pos) return DA_ERR_NULL;
  if (B <= 0 || h_kv <= 0 || d_k <= 0 || d_v <= 0 || n_max <= 0) return DA_ERR_SHAPE;
  const int es = elem_size(dtype);
  if ((d_k * es) % 16 != 0 || (d_v * es) % 16 != 0) return DA_ERR_SHAPE;
  if ((long long)B * h_kv * (long long)n_max > 0x7fffffffLL) return DA_ERR_SHAPE;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(K) || !aligned16(V)) return DA_ERR_ALIGN;
  int dev, sms;
  int st = current_device(&dev, &sms);
  if (st != DA_OK) return st;
  cudaError_t e = da::launch_kv_append(k_new, v_new, K, V, pos, B, h_kv, d_k * es, d_v * es, n_max,
                                       ks_new, vs_new, ks, vs, dev_error, stream);
  if (e != cudaSuccess) return fail_cuda(e, "kv_append launch");
  g_launches.fetch_add(1);
  return DA_OK;
}
}  // namespace

int kv_append(const void* k_new, const void* v_new, void* K, void* V, const int32_t* pos, int B,
              int h_kv, int d_k, int d_v, int n_max, int dtype, int32_t* dev_error,
              cudaStream_t stream) {
  if (dtype != DA_FP32 && dtype != DA_BF16) return DA_ERR_DTYPE;
  return append_rows(k_new, v_new, K, V, pos, B, h_kv, d_k, d_v, n_max, dtype, nullptr, nullptr,
                     nullptr, nullptr, dev_error, stream);
}

int kv_append_q8(const void* k_new, const void* v_new, const float* k_new_scale,
                 const float* v_new_scale, void* K, void* V, float* k_scale, float* v_scale,
                 const int32_t* pos, int B, int h_kv, int d_k, int d_v, int n_max, int dtype,
                 int32_t* dev_error, cudaStream_t stream) {
  if (!is_q8(dtype)) return DA_ERR_DTYPE;
  if (!k_new_scale || !v_new_scale || !k_scale || !v_scale) return DA_ERR_NULL;
  return append_rows(k_new, v_new, K, V, pos, B, h_kv, d_k, d_v, n_max, dtype, k_new_scale,
                     v_new_scale, k_scale, v_scale, dev_error, stream);
}

int decode_attn_q8_ex(const void* q, const void* K, const void* V, const float* k_scale,
                      const float* v_scale, const int32_t* seq_lens, void* out, int B, int h_q,
                      int h_kv, int d_k, int d_v, int n_max, float scale, int dtype,
                      int num_splits, void* workspace, size_t workspace_bytes,
                      int32_t* dev_error, cudaStream_t stream) {
  if (!is_q8(dtype & 0xff)) return DA_ERR_DTYPE;
  const QuantArgs qa{const_cast<float*>(k_scale), const_cast<float*>(v_scale), nullptr, nullptr};
  return run_decode(q, K, V, seq_lens, out, B, h_q, h_kv, d_k, d_v, n_max, scale, dtype,
                    num_splits, workspace, workspace_bytes, dev_error, stream, nullptr, nullptr,
                    nullptr, &qa);
}

int decode_attn_q8_append(const void* q, const void* k_new, const void* v_new,
                          const float* k_new_scale, const float* v_new_scale, void* K, void* V,
                          float* k_scale, float* v_scale, const int32_t* seq_lens,
                          int32_t* seq_lens_out, void* out, int B, int h_q, int h_kv, int d_k,
                          int d_v, int n_max, float scale, int dtype, int num_splits,
                          void* workspace, size_t workspace_bytes, int32_t* dev_error,
                          cudaStream_t stream) {
  if (!is_q8(dtype & 0xff)) return DA_ERR_DTYPE;
  if (!k_new || !v_new || !k_new_scale || !v_new_scale) return DA_ERR_NULL;
  if (seq_lens_out && seq_lens_out == seq_lens) return DA_ERR_SHAPE;
  if (!aligned16(k_new) || !aligned16(v_new)) return DA_ERR_ALIGN;
  const QuantArgs qa{k_scale, v_scale, k_new_scale, v_new_scale};
  return run_decode(q, K, V, seq_lens, out, B, h_q, h_kv, d_k, d_v, n_max, scale, dtype,
                    num_splits, workspace, workspace_bytes, dev_error, stream, k_new, v_new,
                    seq_lens_out, &qa);
}

int kv_quantize(const void* x, int x_dtype, void* codes, float* scales, long long rows, int d,
                int code_dtype, cudaStream_t stream) {
  if (!x || !codes || !scales) return DA_ERR_NULL;
  if ((x_dtype != DA_FP32 && x_dtype != DA_BF16) || !is_q8(code_dtype)) return DA_ERR_DTYPE;
  if (rows < 0 || d <= 0 || d % 32 != 0 || d > 256 || rows > (1LL << 33)) return DA_ERR_SHAPE;
  if (rows == 0) return DA_OK;
  int dev, sms;
  int st = current_device(&dev, &sms);
  if (st != DA_OK) return st;
  cudaError_t e = da::launch_kv_quantize(x, x_dtype == DA_BF16, codes, scales, rows, d,
                                         code_dtype == DA_INT8 ? 1 : 2, stream);
  if (e != cudaSuccess) return fail_cuda(e, "kv_quantize launch");
  g_launches.fetch_add(1);
  return DA_OK;
}

}  // extern "C"
