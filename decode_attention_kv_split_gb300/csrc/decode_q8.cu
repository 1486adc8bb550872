// Split-KV decode attention over 8-bit KV caches (sm_103a).
//
// A cached row of K (and of V) is d one-byte codes plus one float32 scale;
// it stands for scale * value(code), value() being the int8 integer or the
// fp8 e4m3 number.  The page "Attention over the KV cache in the decode step"
// notes that such a cache halves the bytes streamed per row; the row format
// is this library's.  Steps I-III of "MoA-Structured Decode Attention"
// (section 2, eq. 1-3) factor over the row scales:
//   s[l]      = scale * ks[l] * sum_j q[j] * value(Kc[l][j])
//   out[h, d] = sum_l a[l] * vs[l] * value(Vc[l][d])
// so the tensor cores only ever see the codes' values, which fp16 holds
// exactly (int8: |x| <= 128; e4m3: 3 mantissa bits, exponents 2^-9 .. 2^8),
// and the scales are applied in fp32 to the scores and to the softmax weights.
//
// Structure (as the bf16 kernel): one persistent CTA per SM, a producer warp
// streaming each item's code tiles and scale tiles with TMA through a ring of
// stages, consumer warps that each own KBW blocks of 16 rows of a stage.  A
// consumer warp first converts its own rows' codes into an fp16 tile in
// shared memory (rows past the end become zeros, an appended row is taken
// from its slot), reads its rows' scales and releases the stage, then runs
// the fragment code of the bf16 kernel on fp16 MMAs:
//   S^T = K_rows . Q^T (mma.m16n8k16, rows of K as M, 8 query heads as N),
//   online softmax in the log2 domain, P scaled by the V row scales,
//   O^T += V_rows^T . P^T with P as an fp16 head plus an fp16 remainder.
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"

namespace da {

namespace q8 {

// D = A * B + D, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats -> f16x2 (round to nearest even); `lo` lands in bits 0..15.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float f16_lo(uint32_t x) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(x & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t x) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(x >> 16)));
}

// Four codes (code i in bits 8i..8i+7) -> their exact values as two f16x2
// words: lo = codes 0, 1; hi = codes 2, 3.
template <int KIND>
__device__ __forceinline__ void codes_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi);

// int8: the byte x ^ 0x80 = x + 128 placed under the fp16 exponent of 1024
// gives 1024 + x + 128 exactly; subtracting 1152 leaves x.
template <>
__device__ __forceinline__ void codes_to_f16<1>(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x7170);  // bytes u0, 0x64, u1, 0x64
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x7372);  // bytes u2, 0x64, u3, 0x64
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  const __half2 x = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  const __half2 y = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&x);
  hi = *reinterpret_cast<const uint32_t*>(&y);
}

// fp8 e4m3: the hardware conversion to f16x2 is exact.
template <>
__device__ __forceinline__ void codes_to_f16<2>(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// 2-D tiled TMA load into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

}  // namespace q8

// Producer lane, before waiting for the previous grid: L2 prefetch of the
// hinted tiles of the codes (one box per tile) and of their row scales.
template <int TILE>
__device__ __forceinline__ void prefetch_hinted_q8(const SplitParams& p, int4 hint,
                                                   const CUtensorMap* tmK, const CUtensorMap* tmV,
                                                   const CUtensorMap* tmKs, const CUtensorMap* tmVs,
                                                   int max_tiles) {
  int z, y0, tiles;
  if (!read_hint<TILE>(p, hint, max_tiles, z, y0, tiles)) return;
  if ((y0 & 3) != 0) return;  // the row-scale maps take x = row: 16-byte aligned starts only
  for (int t = 0; t < tiles && y0 + t * TILE < p.n_max; ++t) {
    tma_prefetch_3d(tmK, 0, y0 + t * TILE, z);
    tma_prefetch_3d(tmV, 0, y0 + t * TILE, z);
    tma_prefetch_2d(tmKs, y0 + t * TILE, z);
    tma_prefetch_2d(tmVs, y0 + t * TILE, z);
  }
}

template <int D_, int KW_, int KBW_, int STAGES_, int KIND_>
struct Q8Cfg {
  static constexpr int D = D_;            // head dim (d_k == d_v)
  static constexpr int KW = KW_;          // key warps
  static constexpr int KBW = KBW_;        // 16-row blocks per key warp per stage
  static constexpr int STAGES = STAGES_;
  static constexpr int KIND = KIND_;      // 1: int8 codes, 2: fp8 e4m3 codes
  static constexpr int HG = 1;            // one head group of 8 query heads
  static constexpr int kHPW = 8;          // heads per warp (one MMA N block)
  static constexpr int kHeadsPerCta = 8;
  static constexpr int kTile = 16 * KW * KBW;
  static constexpr int kConsumerWarps = KW;
  static constexpr int kConsumerThreads = 32 * KW;
  static constexpr int kThreads = kConsumerThreads + 32;
  static constexpr int kCodeBytes = kTile * D;            // one tensor's codes per stage
  static constexpr int kScaleBytes = kTile * 4;           // one tensor's row scales per stage
  static constexpr int kStageBytes = 2 * kCodeBytes + 2 * kScaleBytes;
  static constexpr int kHalfBytes = kTile * 128;          // a 64-column half of an fp16 tile
  static constexpr int kF16TileBytes = kTile * D * 2;     // one tensor, fp16
  static constexpr int kQBytes = kHeadsPerCta * D * 2;    // bf16 q rows of one item, per stage
  static constexpr int kNewBytes = 2 * D;                 // appended K and V code rows, per stage
  static constexpr int kSlotStride = D + 4;
  static constexpr int kEpiAccFloats = KW * kHPW * kSlotStride;
  static constexpr int kEpiMLFloats = 2 * KW * kHPW;
  static constexpr int kSchedWords = da::kSchedWords;
  static constexpr size_t kSmemBytes =
      1024 + size_t(STAGES) * (kStageBytes + kQBytes + kNewBytes) + 2 * size_t(kF16TileBytes) +
      size_t(kEpiAccFloats + kEpiMLFloats + kSchedWords) * 4 + 2 * STAGES * 8 + 16;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(KIND == 1 || KIND == 2, "code type");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kStageBytes % 1024 == 0, "stage alignment");
  static_assert((kEpiAccFloats + kEpiMLFloats) % 2 == 0, "mbarrier alignment");
};

// Byte offset of column `col` (a multiple of 8) of row `row` of an fp16
// tile: 64-column halves of 128-byte rows, 128-byte swizzle.
template <class Cfg>
__device__ __forceinline__ uint32_t swz_f16(int row, int col) {
  const int half = col >> 6;
  const int chunk = (col & 63) >> 3;
  return uint32_t(half * Cfg::kHalfBytes + row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Producer: one thread streams every stage of the CTA's items: the K and V
// code tiles and row scales, the item's bf16 q rows on its first stage, and
// the appended code rows on the stage that holds them.
template <class Cfg>
__device__ __forceinline__ void produce_q8(const CUtensorMap* tmK, const CUtensorMap* tmV,
                                           const CUtensorMap* tmKs, const CUtensorMap* tmVs,
                                           const SplitParams& p, const Schedule& s, uint32_t ring,
                                           uint32_t qslots, uint32_t newslots, uint32_t full0,
                                           uint32_t empty0, volatile int* abort_flag) {
  constexpr int T = Cfg::kTile, STAGES = Cfg::STAGES, D = Cfg::D;
  const uint64_t policy = l2_policy_evict_first();
  int stage = 0;
  uint32_t phase = 0, issued = 0, issued_parity = 0;
  bool aborted = false;
  for (int k = 0; k < s.mine && !aborted; ++k) {
    const Item it = cta_item<T>(p, s, k);
    const int z = (p.b_offset + it.b) * p.h_kv + it.kvh;
    for (int t = 0; t < it.tiles; ++t) {
      if (!mbar_wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag)) {
        *abort_flag = 1;
        flag_error(p.dev_error, DA_DEVERR_TIMEOUT);
        aborted = true;
        break;
      }
      if (test_withhold(p, k, t, it.tiles)) {  // test builds only: never filled
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        continue;
      }
      const uint32_t bar = full0 + 8 * stage;
      const int y0 = it.row_begin + t * T;
      const bool with_new = it.new_row >= y0 && it.new_row < y0 + T;
      uint32_t extra = 0;
      const int h0 = it.hc * Cfg::kHeadsPerCta;
      const int nh = min(Cfg::kHeadsPerCta, p.group - h0);
      // (checked builds: q and new rows only from inside their arrays)
      const size_t bhq = size_t(it.b) * p.h_q + size_t(it.kvh) * p.group + h0;
      const bool load_q = t == 0 && DA_IN(p, bhq + nh - 1, size_t(p.B) * p.h_q);
      const bool load_new = with_new && DA_IN(p, size_t(it.b) * p.h_kv + it.kvh, size_t(p.B) * p.h_kv);
      if (load_q) extra += uint32_t(nh) * (D * 2);
      if (load_new) extra += 2 * D;
      mbar_arrive_expect_tx(bar, Cfg::kStageBytes + extra);
      if (load_q) {
        const char* qsrc = static_cast<const char*>(p.q) + bhq * (D * 2);
        bulk_load(qslots + stage * Cfg::kQBytes, qsrc, uint32_t(nh) * (D * 2), bar);
      }
      if (load_new) {
        const size_t src = (size_t(it.b) * p.h_kv + it.kvh) * D;
        bulk_load(newslots + stage * Cfg::kNewBytes, static_cast<const char*>(p.k_new) + src, D,
                  bar);
        bulk_load(newslots + stage * Cfg::kNewBytes + D, static_cast<const char*>(p.v_new) + src,
                  D, bar);
      }
      const uint32_t dst = ring + stage * Cfg::kStageBytes;
      tma_load_3d(dst, tmK, 0, y0, z, bar, policy);
      tma_load_3d(dst + Cfg::kCodeBytes, tmV, 0, y0, z, bar, policy);
      q8::tma_load_2d(dst + 2 * Cfg::kCodeBytes, tmKs, y0, z, bar, policy);
      q8::tma_load_2d(dst + 2 * Cfg::kCodeBytes + Cfg::kScaleBytes, tmVs, y0, z, bar, policy);
      issued |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }
  }
  if (aborted) {
    volatile int never = 0;
    for (int st = 0; st < STAGES; ++st)
      if (issued & (1u << st)) mbar_wait_bounded(full0 + 8 * st, (issued_parity >> st) & 1u, &never);
  }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    split_decode_q8_kernel(const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmKs,
                           const __grid_constant__ CUtensorMap tmVs, const SplitParams p) {
  constexpr int D = Cfg::D, KW = Cfg::KW, KBW = Cfg::KBW, STAGES = Cfg::STAGES, T = Cfg::kTile;
  constexpr int kHPW = Cfg::kHPW;
  constexpr int MB = D / 16;       // 16-wide blocks of d
  constexpr int RW = KBW * 16;     // rows owned by one consumer warp
  constexpr int CPR = D / 16;      // 16-code chunks per row

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* kf16 = smem + size_t(STAGES) * Cfg::kStageBytes;  // fp16 K tile (1024-aligned)
  uint8_t* vf16 = kf16 + Cfg::kF16TileBytes;                 // fp16 V tile
  uint8_t* qslots = vf16 + Cfg::kF16TileBytes;
  uint8_t* newslots = qslots + size_t(STAGES) * Cfg::kQBytes;
  float* epi_acc = reinterpret_cast<float*>(newslots + size_t(STAGES) * Cfg::kNewBytes);
  float* epi_m = epi_acc + Cfg::kEpiAccFloats;
  float* epi_l = epi_m + KW * kHPW;
  int* sched_words = reinterpret_cast<int*>(epi_l + KW * kHPW);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sched_words + Cfg::kSchedWords);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * STAGES);
  const uint32_t ring = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, Cfg::kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {  // the tensor maps do not depend on the preceding grid
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmKs);
    prefetch_tmap(&tmVs);
  }
  if (threadIdx.x == Cfg::kConsumerThreads)  // producer lane: L2 prefetch of the hinted tiles
    prefetch_hinted_q8<T>(p, load_hint(p), &tmK, &tmV, &tmKs, &tmVs, STAGES);
  // Launched as a programmatic dependent: the set-up here overlaps the tail
  // of the previous grid on the stream, which may have produced seq_lens, q,
  // the caches or the new rows.  Before the wait below, only the hinted L2
  // prefetch and the work list touch them: the prefetch is a hint, and the
  // list is built on the lengths as they read now (shared memory only), then
  // checked and built again if they changed once the wait is over.  Here the
  // prefetch goes out before the build, for the most lead time (measured
  // faster for these kernels than issuing it after the build).
  Schedule sched = build_schedule_core<T>(p, sched_words);
  wait_for_prerequisite_grid();
  sched = commit_schedule<T>(p, sched_words, sched);
  allow_dependent_launch();
  if (threadIdx.x == 0 && sched.mine > 0) write_hint<T>(p, cta_item<T>(p, sched, 0), STAGES);

  // ------------------------------------------------------------------ producer
  if (warp == KW) {
    if (lane == 0)
      produce_q8<Cfg>(&tmK, &tmV, &tmKs, &tmVs, p, sched, ring, smem_u32(qslots),
                      smem_u32(newslots), full0, empty0, abort_flag);
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int kw = warp;
  const int r = lane >> 2;  // MMA fragment row group
  const int c = lane & 3;   // MMA fragment column pair
  const int key0 = kw * RW;  // first row of this warp inside a stage
  int stage = 0;
  uint32_t phase = 0;

  // Which 16-code chunks of its rows a lane converts: chunk u of lane L is
  // number L + 32 u of the warp's 2 * RW * CPR chunks (K rows, then V rows).
  // For d = 128 a quarter-warp covers two rows in opposite 64-column halves,
  // so neither the 16-byte code reads nor the swizzled fp16 writes share a
  // bank; for d = 64 (64-byte rows) it covers two whole rows.  Everything but
  // the stage base is fixed per lane.
  constexpr int kChunks = 2 * RW * CPR / 32;
  static_assert((RW * CPR) % 32 == 0, "chunks split evenly between K and V");
  int lane_row, chunk_col;
  if (D == 128) {
    const int qa = (lane >> 3) & 1, sub = lane & 7, r2 = sub >> 2;
    lane_row = 2 * (lane >> 4) + r2;   // rows step by 4 per 32 chunks
    chunk_col = (r2 ^ qa) * 64 + (sub & 3) * 16;
  } else {
    lane_row = lane >> 2;              // rows step by 8 per 32 chunks
    chunk_col = (lane & 3) * 16;
  }
  constexpr int kRowStep = 32 / CPR;   // rows advanced by 32 chunks
  auto chunk_tensor = [&](int u) { return u / (kChunks / 2); };
  auto chunk_row = [&](int u) { return key0 + lane_row + (u % (kChunks / 2)) * kRowStep; };
  const int src_off0 = (key0 + lane_row) * D + chunk_col;
  auto chunk_src = [&](int u) {
    return chunk_tensor(u) * Cfg::kCodeBytes + (u % (kChunks / 2)) * kRowStep * D;
  };
  auto chunk_dst = [&](int u, int c8) {
    return chunk_tensor(u) * Cfg::kF16TileBytes + int(swz_f16<Cfg>(chunk_row(u), chunk_col + c8));
  };

  for (int k = 0; k < sched.mine; ++k) {
    const Item it = cta_item<T>(p, sched, k);
    const int head_base = it.hc * Cfg::kHeadsPerCta;
    const size_t kvhead = size_t(p.b_offset + it.b) * p.h_kv + it.kvh;
    uint32_t qf[MB][2];

    float m_run[2], l_run[2];
    float acc[MB][4];
    m_run[0] = m_run[1] = -INFINITY;
    l_run[0] = l_run[1] = 0.f;
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mb][e] = 0.f;

    for (int t = 0; t < it.tiles; ++t) {
      if (!mbar_wait_bounded(full0 + 8 * stage, phase, abort_flag)) {
        if (!*abort_flag) {
          *abort_flag = 1;
          flag_error(p.dev_error, DA_DEVERR_TIMEOUT);
        }
      }
      const uint8_t* st = smem + size_t(stage) * Cfg::kStageBytes;
      const float* ks_t = reinterpret_cast<const float*>(st + 2 * Cfg::kCodeBytes);
      const float* vs_t = ks_t + T;
      const uint8_t* nslot = newslots + size_t(stage) * Cfg::kNewBytes;
      const int tile_row0 = it.row_begin + t * T;
      const int valid = min(T, it.row_end - tile_row0);
      const int new_local = (it.new_row >= tile_row0 && it.new_row < tile_row0 + T)
                                ? it.new_row - tile_row0
                                : -1;
      const bool mine_new = new_local >= key0 && new_local < key0 + RW;

      // ---- this warp's rows: codes -> fp16 tiles (zeros past the end)
      if (valid == T && new_local < 0) {  // a full tile with no appended row (warp-uniform)
#pragma unroll
        for (int u = 0; u < kChunks; ++u) {
          const uint4 w = *reinterpret_cast<const uint4*>(st + src_off0 + chunk_src(u));
          uint4 a, b;
          q8::codes_to_f16<Cfg::KIND>(w.x, a.x, a.y);
          q8::codes_to_f16<Cfg::KIND>(w.y, a.z, a.w);
          q8::codes_to_f16<Cfg::KIND>(w.z, b.x, b.y);
          q8::codes_to_f16<Cfg::KIND>(w.w, b.z, b.w);
          *reinterpret_cast<uint4*>(kf16 + chunk_dst(u, 0)) = a;
          *reinterpret_cast<uint4*>(kf16 + chunk_dst(u, 8)) = b;
        }
      } else {
#pragma unroll 2
        for (int u = 0; u < kChunks; ++u) {
          const int tensor = chunk_tensor(u), row = chunk_row(u), col = chunk_col;
          uint4 w = make_uint4(0, 0, 0, 0);
          if (row < valid) {
            const uint8_t* src = row == new_local ? nslot + tensor * D + col
                                                  : st + src_off0 + chunk_src(u);
            w = *reinterpret_cast<const uint4*>(src);
          }
          uint4 a, b;
          q8::codes_to_f16<Cfg::KIND>(w.x, a.x, a.y);
          q8::codes_to_f16<Cfg::KIND>(w.y, a.z, a.w);
          q8::codes_to_f16<Cfg::KIND>(w.z, b.x, b.y);
          q8::codes_to_f16<Cfg::KIND>(w.w, b.z, b.w);
          if (row >= valid) a = b = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(kf16 + chunk_dst(u, 0)) = a;
          *reinterpret_cast<uint4*>(kf16 + chunk_dst(u, 8)) = b;
        }
      }
      // ---- this lane's row scales (0 past the end; the appended row's own)
      float fk[KBW][2], fv[KBW][2];
#pragma unroll
      for (int kb = 0; kb < KBW; ++kb)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int row = key0 + kb * 16 + r + 8 * hh;
          float sk = ks_t[row], sv = vs_t[row];
          if (row == new_local) {
            sk = __ldg(p.k_new_scale + size_t(it.b) * p.h_kv + it.kvh);
            sv = __ldg(p.v_new_scale + size_t(it.b) * p.h_kv + it.kvh);
          }
          fk[kb][hh] = row < valid ? sk * p.scale_log2 : 0.f;
          fv[kb][hh] = row < valid ? sv : 0.f;
        }
      if (t == 0) {  // q rows of the item's heads, bf16 -> fp16 fragments
        const uint32_t* qs =
            reinterpret_cast<const uint32_t*>(qslots + size_t(stage) * Cfg::kQBytes);
        const bool ok = head_base + r < p.group;
#pragma unroll
        for (int ks = 0; ks < MB; ++ks) {
          const uint32_t a0 = ok ? qs[r * (D / 2) + ks * 8 + c] : 0u;
          const uint32_t a1 = ok ? qs[r * (D / 2) + ks * 8 + 4 + c] : 0u;
          qf[ks][0] = q8::pack_f16x2(bf16_lo_to_f32(a0), bf16_hi_to_f32(a0));
          qf[ks][1] = q8::pack_f16x2(bf16_lo_to_f32(a1), bf16_hi_to_f32(a1));
        }
      }
      // the appended row goes into the caches once per kv head, by the warp that owns it
      if (mine_new && it.hc == 0 && !*abort_flag &&
          DA_IN(p, kvhead * size_t(p.n_max) + size_t(it.new_row), p.cache_rows)) {
        const size_t row_off = kvhead * size_t(p.n_max) + size_t(it.new_row);
        if (lane < D / 16) {
          reinterpret_cast<uint4*>(static_cast<char*>(p.k_cache) + row_off * D)[lane] =
              reinterpret_cast<const uint4*>(nslot)[lane];
          reinterpret_cast<uint4*>(static_cast<char*>(p.v_cache) + row_off * D)[lane] =
              reinterpret_cast<const uint4*>(nslot + D)[lane];
        }
        if (lane == 0) {
          p.k_scale[row_off] = __ldg(p.k_new_scale + size_t(it.b) * p.h_kv + it.kvh);
          p.v_scale[row_off] = __ldg(p.v_new_scale + size_t(it.b) * p.h_kv + it.kvh);
        }
      }
      __syncwarp();
      // the stage's codes, scales and q are all in registers or the fp16 tiles now
      if (lane == 0) mbar_arrive(empty0 + 8 * stage);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }

      // warp-uniform (the MMAs and shuffles below need the whole warp)
      const bool live = __all_sync(0xffffffffu, !*abort_flag);
      if (live && key0 < valid) {
        const uint32_t kbase = smem_u32(kf16);
        const uint32_t vbase = smem_u32(vf16);
        // ---- Step I: scores for KBW blocks of 16 rows
        float s[KBW][4];
#pragma unroll
        for (int kb = 0; kb < KBW; ++kb)
#pragma unroll
          for (int e = 0; e < 4; ++e) s[kb][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < MB; ++ks) {
#pragma unroll
          for (int kb = 0; kb < KBW; ++kb) {
            const int row = key0 + kb * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int col = ks * 16 + (lane >> 4) * 8;
            uint32_t a[4];
            ldmatrix_x4(a, kbase + swz_f16<Cfg>(row, col));
            q8::mma_f16_16816(s[kb], a, qf[ks][0], qf[ks][1]);
          }
        }
        // ---- Step II: scale by the K row scales, mask, running max and sum
        float alpha[2];
        bool changed = false;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float mx = -INFINITY;
#pragma unroll
          for (int kb = 0; kb < KBW; ++kb) {
            const int row_lo = key0 + kb * 16 + r;
            s[kb][j] = row_lo < valid ? s[kb][j] * fk[kb][0] : -INFINITY;
            s[kb][j + 2] = row_lo + 8 < valid ? s[kb][j + 2] * fk[kb][1] : -INFINITY;
            mx = fmaxf(mx, fmaxf(s[kb][j], s[kb][j + 2]));
          }
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_run[j], mx);
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          alpha[j] = ex2(m_run[j] - m_use);
          changed |= (m_new != m_run[j]);
          m_run[j] = m_new;
          float sum = 0.f;
#pragma unroll
          for (int kb = 0; kb < KBW; ++kb) {
            s[kb][j] = ex2(s[kb][j] - m_use);
            s[kb][j + 2] = ex2(s[kb][j + 2] - m_use);
            sum += s[kb][j] + s[kb][j + 2];
          }
          l_run[j] = l_run[j] * alpha[j] + sum;
        }
        if (__any_sync(0xffffffffu, changed)) {
#pragma unroll
          for (int mb = 0; mb < MB; ++mb) {
            acc[mb][0] *= alpha[0];
            acc[mb][1] *= alpha[1];
            acc[mb][2] *= alpha[0];
            acc[mb][3] *= alpha[1];
          }
        }
        // ---- Step III: O^T += V^T . (P * vs)^T, P as fp16 head + fp16 remainder
#pragma unroll
        for (int kb = 0; kb < KBW; ++kb) {
          const float p0 = s[kb][0] * fv[kb][0], p1 = s[kb][1] * fv[kb][0];
          const float p2 = s[kb][2] * fv[kb][1], p3 = s[kb][3] * fv[kb][1];
          const uint32_t h0 = q8::pack_f16x2(p0, p1);  // row r
          const uint32_t h1 = q8::pack_f16x2(p2, p3);  // row r + 8
          const uint32_t l0 = q8::pack_f16x2(p0 - q8::f16_lo(h0), p1 - q8::f16_hi(h0));
          const uint32_t l1 = q8::pack_f16x2(p2 - q8::f16_lo(h1), p3 - q8::f16_hi(h1));
          const uint32_t ph0 = movmatrix_trans(h0), ph1 = movmatrix_trans(h1);
          const uint32_t pl0 = movmatrix_trans(l0), pl1 = movmatrix_trans(l1);
          const int blk0 = key0 + kb * 16;
#pragma unroll
          for (int mb = 0; mb < MB; ++mb) {
            const int row = blk0 + (lane & 7) + ((lane >> 4) & 1) * 8;
            const int col = mb * 16 + ((lane >> 3) & 1) * 8;
            uint32_t a[4];
            ldmatrix_x4_trans(a, vbase + swz_f16<Cfg>(row, col));
            q8::mma_f16_16816(acc[mb], a, ph0, ph1);
            q8::mma_f16_16816(acc[mb], a, pl0, pl1);
          }
        }
      }
      __syncwarp();  // the fp16 tiles are rewritten for the next stage
    }

    // ---- Epilogue: per-warp state to shared slots, then the shared finish.
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float v = l_run[j];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l_run[j] = v;
    }
    named_bar_sync(1, Cfg::kConsumerThreads);  // earlier readers of the slots are done
    float* slot = epi_acc + kw * kHPW * Cfg::kSlotStride;
    if (lane < 4) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        epi_m[kw * kHPW + 2 * lane + j] = m_run[j];
        epi_l[kw * kHPW + 2 * lane + j] = l_run[j];
      }
    }
#pragma unroll
    for (int mb = 0; mb < MB; ++mb) {
      const int d0 = mb * 16 + r;
      const int h0 = 2 * c;
      slot[h0 * Cfg::kSlotStride + d0] = acc[mb][0];
      slot[(h0 + 1) * Cfg::kSlotStride + d0] = acc[mb][1];
      slot[h0 * Cfg::kSlotStride + d0 + 8] = acc[mb][2];
      slot[(h0 + 1) * Cfg::kSlotStride + d0 + 8] = acc[mb][3];
    }
    named_bar_sync(1, Cfg::kConsumerThreads);
    finish_item<D, 1, KW, kHPW, Cfg::kSlotStride>(p, it, epi_acc, epi_m, epi_l, threadIdx.x,
                                                  Cfg::kConsumerThreads, abort_flag);
  }
}

// ---------------------------------------------------------------------------
// d = 128: MMA fragments built straight from the code tiles, in registers.
//
// The code tiles arrive with the 128-byte swizzle (16-byte chunk c of row r
// at chunk c ^ (r & 7)), so the reads below are bank-conflict free, and no
// fp16 copy of a stage is ever written to shared memory.  With lane = 4 g + t:
//   Step I  (S^T = K . Q^T, rows of K as M): lane (g, t) reads bytes
//           [32 t, 32 t + 32) of rows g and g + 8 of its 16-row block and
//           uses the 4 codes at 32 t + 4 kb as the A elements of k-block kb
//           at logical columns 2t, 2t+1, 2t+8, 2t+9.  This relabels the 128
//           columns of d one to one, and the B fragments (q) are taken in the
//           same order, so every score is the same sum of the same products.
//   Step III (O^T += V^T . P^T, d as M): lane (g, t) reads bytes
//           [16 g, 16 g + 16) of rows 2t, 2t+1, 2t+8, 2t+9; a byte permute
//           pairs each column of rows 2t and 2t+1 (the two k elements of an A
//           register), and m-block mb takes columns 16 g + 2 mb (as row g of
//           the block) and 16 g + 2 mb + 1 (as row g + 8).  The outputs of
//           lane (g, t) are then columns [16 g, 16 g + 16) of heads 2t, 2t+1.
// ---------------------------------------------------------------------------
template <int STAGES_, int KIND_>
struct Q8RCfg {
  static constexpr int D = 128;
  static constexpr int KW = 8;             // consumer warps, one 16-row block each
  static constexpr int STAGES = STAGES_;
  static constexpr int KIND = KIND_;
  static constexpr int HG = 1;
  static constexpr int kHPW = 8;
  static constexpr int kHeadsPerCta = 8;
  static constexpr int kTile = 16 * KW;
  static constexpr int kConsumerWarps = KW;
  static constexpr int kConsumerThreads = 32 * KW;
  static constexpr int kThreads = kConsumerThreads + 32;
  static constexpr int kCodeBytes = kTile * D;
  static constexpr int kScaleBytes = kTile * 4;
  static constexpr int kStageBytes = 2 * kCodeBytes + 2 * kScaleBytes;
  static constexpr int kQBytes = kHeadsPerCta * D * 2;
  static constexpr int kNewBytes = 2 * D;
  static constexpr int kSlotStride = D + 4;
  static constexpr int kEpiAccFloats = KW * kHPW * kSlotStride;
  static constexpr int kEpiMLFloats = 2 * KW * kHPW;
  static constexpr int kSchedWords = da::kSchedWords;
  static constexpr size_t kSmemBytes =
      1024 + size_t(STAGES) * (kStageBytes + kQBytes + kNewBytes) +
      size_t(kEpiAccFloats + kEpiMLFloats + kSchedWords) * 4 + 2 * STAGES * 8 + 16;
  static_assert(KIND == 1 || KIND == 2, "code type");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kStageBytes % 1024 == 0, "stage alignment (128-byte swizzle)");
  static_assert((kEpiAccFloats + kEpiMLFloats) % 2 == 0, "mbarrier alignment");
};

// 16 bytes of row `row` of a 128-byte-swizzled code tile, logical chunk `chunk`.
__device__ __forceinline__ uint4 ld_code_chunk(const uint8_t* tile, int row, int chunk) {
  return *reinterpret_cast<const uint4*>(tile + row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    split_decode_q8r_kernel(const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ CUtensorMap tmKs,
                            const __grid_constant__ CUtensorMap tmVs, const SplitParams p) {
  constexpr int D = Cfg::D, KW = Cfg::KW, STAGES = Cfg::STAGES, T = Cfg::kTile;
  constexpr int kHPW = Cfg::kHPW;
  constexpr int MB = D / 16;   // 16-wide blocks of d (Step III m-blocks; Step I k-blocks)
  constexpr int KIND = Cfg::KIND;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* qslots = smem + size_t(STAGES) * Cfg::kStageBytes;
  uint8_t* newslots = qslots + size_t(STAGES) * Cfg::kQBytes;
  float* epi_acc = reinterpret_cast<float*>(newslots + size_t(STAGES) * Cfg::kNewBytes);
  float* epi_m = epi_acc + Cfg::kEpiAccFloats;
  float* epi_l = epi_m + KW * kHPW;
  int* sched_words = reinterpret_cast<int*>(epi_l + KW * kHPW);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sched_words + Cfg::kSchedWords);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * STAGES);
  const uint32_t ring = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, Cfg::kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {  // the tensor maps do not depend on the preceding grid
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmKs);
    prefetch_tmap(&tmVs);
  }
  if (threadIdx.x == Cfg::kConsumerThreads)  // producer lane: L2 prefetch of the hinted tiles
    prefetch_hinted_q8<T>(p, load_hint(p), &tmK, &tmV, &tmKs, &tmVs, STAGES);
  // Launched as a programmatic dependent: the set-up here overlaps the tail
  // of the previous grid on the stream, which may have produced seq_lens, q,
  // the caches or the new rows.  Before the wait below, only the hinted L2
  // prefetch and the work list touch them: the prefetch is a hint, and the
  // list is built on the lengths as they read now (shared memory only), then
  // checked and built again if they changed once the wait is over.  Here the
  // prefetch goes out before the build, for the most lead time (measured
  // faster for these kernels than issuing it after the build).
  Schedule sched = build_schedule_core<T>(p, sched_words);
  wait_for_prerequisite_grid();
  sched = commit_schedule<T>(p, sched_words, sched);
  allow_dependent_launch();
  if (threadIdx.x == 0 && sched.mine > 0) write_hint<T>(p, cta_item<T>(p, sched, 0), STAGES);

  // ------------------------------------------------------------------ producer
  if (warp == KW) {
    if (lane == 0)
      produce_q8<Cfg>(&tmK, &tmV, &tmKs, &tmVs, p, sched, ring, smem_u32(qslots),
                      smem_u32(newslots), full0, empty0, abort_flag);
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int g = lane >> 2;   // MMA fragment row group
  const int t = lane & 3;    // MMA fragment column pair
  const int key0 = warp * 16;  // first row of this warp's block inside a stage
  const int rA = key0 + g, rB = rA + 8;             // Step I rows (and P rows)
  const int r0 = key0 + 2 * t, r1 = r0 + 1, r2 = r0 + 8, r3 = r0 + 9;  // Step III rows
  int stage = 0;
  uint32_t phase = 0;

  for (int k = 0; k < sched.mine; ++k) {
    const Item it = cta_item<T>(p, sched, k);
    const int head_base = it.hc * Cfg::kHeadsPerCta;
    const size_t kvhead = size_t(p.b_offset + it.b) * p.h_kv + it.kvh;
    uint32_t qf[MB][2];  // B fragments of q (head g), in the permuted column order

    float m_run[2], l_run[2];
    float acc[MB][4];
    m_run[0] = m_run[1] = -INFINITY;
    l_run[0] = l_run[1] = 0.f;
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[mb][e] = 0.f;

    for (int tt = 0; tt < it.tiles; ++tt) {
      if (!mbar_wait_bounded(full0 + 8 * stage, phase, abort_flag)) {
        if (!*abort_flag) {
          *abort_flag = 1;
          flag_error(p.dev_error, DA_DEVERR_TIMEOUT);
        }
      }
      const uint8_t* st = smem + size_t(stage) * Cfg::kStageBytes;
      const uint8_t* ktile = st;
      const uint8_t* vtile = st + Cfg::kCodeBytes;
      const float* ks_t = reinterpret_cast<const float*>(st + 2 * Cfg::kCodeBytes);
      const float* vs_t = ks_t + T;
      const uint8_t* nslot = newslots + size_t(stage) * Cfg::kNewBytes;
      const int tile_row0 = it.row_begin + tt * T;
      const int valid = min(T, it.row_end - tile_row0);
      const int new_local = (it.new_row >= tile_row0 && it.new_row < tile_row0 + T)
                                ? it.new_row - tile_row0
                                : -1;

      // ---- this lane's codes and row scales, into registers
      uint4 kA0 = ld_code_chunk(ktile, rA, 2 * t), kA1 = ld_code_chunk(ktile, rA, 2 * t + 1);
      uint4 kB0 = ld_code_chunk(ktile, rB, 2 * t), kB1 = ld_code_chunk(ktile, rB, 2 * t + 1);
      uint4 v0 = ld_code_chunk(vtile, r0, g), v1 = ld_code_chunk(vtile, r1, g);
      uint4 v2 = ld_code_chunk(vtile, r2, g), v3 = ld_code_chunk(vtile, r3, g);
      float skA = ks_t[rA], skB = ks_t[rB], svA = vs_t[rA], svB = vs_t[rB];
      if (new_local >= key0 && new_local < key0 + 16) {  // warp-uniform: the appended row
        const uint4* nk = reinterpret_cast<const uint4*>(nslot);
        const uint4* nv = reinterpret_cast<const uint4*>(nslot + D);
        const float nks = __ldg(p.k_new_scale + size_t(it.b) * p.h_kv + it.kvh);
        const float nvs = __ldg(p.v_new_scale + size_t(it.b) * p.h_kv + it.kvh);
        if (rA == new_local) kA0 = nk[2 * t], kA1 = nk[2 * t + 1], skA = nks, svA = nvs;
        if (rB == new_local) kB0 = nk[2 * t], kB1 = nk[2 * t + 1], skB = nks, svB = nvs;
        if (r0 == new_local) v0 = nv[g];
        if (r1 == new_local) v1 = nv[g];
        if (r2 == new_local) v2 = nv[g];
        if (r3 == new_local) v3 = nv[g];
      }
      // rows past the end may hold anything: their values must not reach O
      const uint4 zero = make_uint4(0, 0, 0, 0);
      if (r0 >= valid) v0 = zero;
      if (r1 >= valid) v1 = zero;
      if (r2 >= valid) v2 = zero;
      if (r3 >= valid) v3 = zero;
      const float fkA = rA < valid ? skA * p.scale_log2 : 0.f;
      const float fkB = rB < valid ? skB * p.scale_log2 : 0.f;
      const float fvA = rA < valid ? svA : 0.f;
      const float fvB = rB < valid ? svB : 0.f;
      if (tt == 0) {  // q of head g (rows past the group are zero), bf16 -> fp16 B fragments
        const bool ok = head_base + g < p.group;
        const uint4* qs = reinterpret_cast<const uint4*>(qslots + size_t(stage) * Cfg::kQBytes +
                                                         g * (D * 2) + t * 64);
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // 8 bf16 values = columns 32t + 8c .. + 7
          const uint4 w = ok ? qs[c] : zero;
          qf[2 * c][0] = q8::pack_f16x2(bf16_lo_to_f32(w.x), bf16_hi_to_f32(w.x));
          qf[2 * c][1] = q8::pack_f16x2(bf16_lo_to_f32(w.y), bf16_hi_to_f32(w.y));
          qf[2 * c + 1][0] = q8::pack_f16x2(bf16_lo_to_f32(w.z), bf16_hi_to_f32(w.z));
          qf[2 * c + 1][1] = q8::pack_f16x2(bf16_lo_to_f32(w.w), bf16_hi_to_f32(w.w));
        }
      }
      // the appended row goes into the caches once per kv head, by the warp that owns it
      if (new_local >= key0 && new_local < key0 + 16 && it.hc == 0 && !*abort_flag &&
          DA_IN(p, kvhead * size_t(p.n_max) + size_t(it.new_row), p.cache_rows)) {
        const size_t row_off = kvhead * size_t(p.n_max) + size_t(it.new_row);
        if (lane < D / 16) {
          reinterpret_cast<uint4*>(static_cast<char*>(p.k_cache) + row_off * D)[lane] =
              reinterpret_cast<const uint4*>(nslot)[lane];
          reinterpret_cast<uint4*>(static_cast<char*>(p.v_cache) + row_off * D)[lane] =
              reinterpret_cast<const uint4*>(nslot + D)[lane];
        }
        if (lane == 0) {
          p.k_scale[row_off] = __ldg(p.k_new_scale + size_t(it.b) * p.h_kv + it.kvh);
          p.v_scale[row_off] = __ldg(p.v_new_scale + size_t(it.b) * p.h_kv + it.kvh);
        }
      }
      __syncwarp();
      // every byte this warp needs from the stage is in registers now
      if (lane == 0) mbar_arrive(empty0 + 8 * stage);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }

      // warp-uniform (the MMAs and shuffles below need the whole warp)
      const bool live = __all_sync(0xffffffffu, !*abort_flag);
      if (live && key0 < valid) {
        // ---- Step I: two independent accumulation chains over the 8 k-blocks
        float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kb = 0; kb < MB; ++kb) {
          uint32_t a[4];
          q8::codes_to_f16<KIND>(word_of(kb < 4 ? kA0 : kA1, kb & 3), a[0], a[2]);
          q8::codes_to_f16<KIND>(word_of(kb < 4 ? kB0 : kB1, kb & 3), a[1], a[3]);
          if (kb & 1) q8::mma_f16_16816(s2, a, qf[kb][0], qf[kb][1]);
          else q8::mma_f16_16816(s, a, qf[kb][0], qf[kb][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) s[e] += s2[e];
        // ---- Step II: scale by the K row scales, mask, running max and sum
        float alpha[2];
        bool changed = false;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          s[j] = rA < valid ? s[j] * fkA : -INFINITY;
          s[j + 2] = rB < valid ? s[j + 2] * fkB : -INFINITY;
          float mx = fmaxf(s[j], s[j + 2]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_run[j], mx);
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          alpha[j] = ex2(m_run[j] - m_use);
          changed |= (m_new != m_run[j]);
          m_run[j] = m_new;
          s[j] = ex2(s[j] - m_use);
          s[j + 2] = ex2(s[j + 2] - m_use);
          l_run[j] = l_run[j] * alpha[j] + (s[j] + s[j + 2]);
        }
        if (__any_sync(0xffffffffu, changed)) {
#pragma unroll
          for (int mb = 0; mb < MB; ++mb) {
            acc[mb][0] *= alpha[0];
            acc[mb][1] *= alpha[1];
            acc[mb][2] *= alpha[0];
            acc[mb][3] *= alpha[1];
          }
        }
        // ---- Step III: O^T += V^T . (P * vs)^T, P as fp16 head + fp16 remainder
        const float p0 = s[0] * fvA, p1 = s[1] * fvA, p2 = s[2] * fvB, p3 = s[3] * fvB;
        const uint32_t h0 = q8::pack_f16x2(p0, p1);  // row g
        const uint32_t h1 = q8::pack_f16x2(p2, p3);  // row g + 8
        const uint32_t l0 = q8::pack_f16x2(p0 - q8::f16_lo(h0), p1 - q8::f16_hi(h0));
        const uint32_t l1 = q8::pack_f16x2(p2 - q8::f16_lo(h1), p3 - q8::f16_hi(h1));
        const uint32_t ph0 = movmatrix_trans(h0), ph1 = movmatrix_trans(h1);
        const uint32_t pl0 = movmatrix_trans(l0), pl1 = movmatrix_trans(l1);
#pragma unroll
        for (int mb = 0; mb < MB; ++mb) {
          const int w = mb >> 1;
          const uint32_t sel = (mb & 1) ? 0x7362u : 0x5140u;  // columns 2mb, 2mb+1 of the lane's 16
          const uint32_t x01 = __byte_perm(word_of(v0, w), word_of(v1, w), sel);
          const uint32_t x23 = __byte_perm(word_of(v2, w), word_of(v3, w), sel);
          uint32_t a[4];
          q8::codes_to_f16<KIND>(x01, a[0], a[1]);  // rows 2t, 2t+1 at columns 2mb (a0), 2mb+1 (a1)
          q8::codes_to_f16<KIND>(x23, a[2], a[3]);  // rows 2t+8, 2t+9
          q8::mma_f16_16816(acc[mb], a, ph0, ph1);
          q8::mma_f16_16816(acc[mb], a, pl0, pl1);
        }
      }
    }

    // ---- Epilogue: per-warp state to shared slots, then the shared finish.
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float v = l_run[j];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l_run[j] = v;
    }
    named_bar_sync(1, Cfg::kConsumerThreads);  // earlier readers of the slots are done
    float* slot = epi_acc + warp * kHPW * Cfg::kSlotStride;
    if (lane < 4) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        epi_m[warp * kHPW + 2 * lane + j] = m_run[j];
        epi_l[warp * kHPW + 2 * lane + j] = l_run[j];
      }
    }
#pragma unroll
    for (int mb = 0; mb < MB; ++mb) {
      const int d0 = 16 * g + 2 * mb;  // acc[mb][0..1]: column d0; acc[mb][2..3]: d0 + 1
      slot[(2 * t) * Cfg::kSlotStride + d0] = acc[mb][0];
      slot[(2 * t + 1) * Cfg::kSlotStride + d0] = acc[mb][1];
      slot[(2 * t) * Cfg::kSlotStride + d0 + 1] = acc[mb][2];
      slot[(2 * t + 1) * Cfg::kSlotStride + d0 + 1] = acc[mb][3];
    }
    named_bar_sync(1, Cfg::kConsumerThreads);
    finish_item<D, 1, KW, kHPW, Cfg::kSlotStride>(p, it, epi_acc, epi_m, epi_l, threadIdx.x,
                                                  Cfg::kConsumerThreads, abort_flag);
  }
}

// ---------------------------------------------------------------------------
// Variants and launcher.
// ---------------------------------------------------------------------------
template <int KIND>
using Q8D128 = Q8RCfg<5, KIND>;   // register-fragment kernel, 128-byte-swizzled code tiles
template <int KIND>
using Q8D64 = Q8Cfg<64, 8, 1, 6, KIND>;

KernelShape q8_shape(int d) {
  if (d == 128) return KernelShape{Q8D128<1>::kTile, 8, 128, 1, 1.0f};
  return KernelShape{Q8D64<1>::kTile, 8, 64, 0, 1.0f};
}

template <class Cfg>
static cudaError_t launch_q8_cfg(const SplitParams& p, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tks,
                                 const CUtensorMap& tvs, int grid, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(split_decode_q8_kernel<Cfg>, Cfg::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  return launch_dependent(split_decode_q8_kernel<Cfg>, grid, Cfg::kThreads, Cfg::kSmemBytes,
                          stream, tk, tv, tks, tvs, p);
}

template <class Cfg>
static cudaError_t launch_q8r_cfg(const SplitParams& p, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const CUtensorMap& tks,
                                  const CUtensorMap& tvs, int grid, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e =
      set_smem_limit_once(split_decode_q8r_kernel<Cfg>, Cfg::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  return launch_dependent(split_decode_q8r_kernel<Cfg>, grid, Cfg::kThreads, Cfg::kSmemBytes,
                          stream, tk, tv, tks, tvs, p);
}

cudaError_t launch_split_q8(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tks, const CUtensorMap& tvs, int d, int kind,
                            int grid, cudaStream_t stream) {
  if (d == 128)
    return kind == 1 ? launch_q8r_cfg<Q8D128<1>>(p, tk, tv, tks, tvs, grid, stream)
                     : launch_q8r_cfg<Q8D128<2>>(p, tk, tv, tks, tvs, grid, stream);
  return kind == 1 ? launch_q8_cfg<Q8D64<1>>(p, tk, tv, tks, tvs, grid, stream)
                   : launch_q8_cfg<Q8D64<2>>(p, tk, tv, tks, tvs, grid, stream);
}

}  // namespace da
