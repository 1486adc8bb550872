// Split-KV decode attention for bf16 caches on tensor cores (sm_103a).
//
// One persistent CTA per SM walks a static list of work items
// (b, kv head, query-head chunk, split).  A producer warp streams the K and
// V rows of each item through a ring of shared-memory stages with 3-D TMA
// loads (128-byte swizzle, evict-first L2 policy); consumer warps compute on
// each stage and hand it back through an mbarrier.  Every K/V byte is read
// from HBM once per CTA that needs it, and all query heads of a kv head live
// in the same CTA, so GQA/MQA groups are never broadcast in memory
// ("MoA-Structured Decode Attention", introduction item 4).
//
// Per 16 cached rows a consumer warp computes, for its 8*NB query heads:
//   Step I  (section 2, eq. 1): S^T = K_rows . Q^T with mma.m16n8k16, the
//           rows of K as the M operand (16 rows) and the query heads as N
//           (8 per block), so a group of 8 heads fills the MMA exactly;
//   Step II (section 2, eq. 2): a running max / running sum (online softmax)
//           in the log2 domain, exp(x) = 2^(x * log2 e) on the SFU;
//   Step III(section 2, eq. 3): O^T += V_rows^T . P^T with mma.m16n8k16, the
//           weights P split into a bf16 head plus a bf16 remainder so they
//           carry ~16 significant bits into the fp32 accumulators.
// Rows are read in their natural row-major layout: the K^T of the textbook
// formula is never formed (section 2, Step I), and lanes run along the
// contiguous d axis of each row (coalescing criterion of section 4).
#include <math.h>

#include "common.cuh"

namespace da {

template <int DK_, int DV_, int NB_, int HG_, int KW_, int KBW_, int STAGES_>
struct Bf16Cfg {
  static constexpr int DK = DK_;          // key / query head dim
  static constexpr int DV = DV_;          // value / output head dim
  static constexpr int NB = NB_;          // 8-head MMA blocks per warp
  static constexpr int HG = HG_;          // head groups (warps sharing rows, different heads)
  static constexpr int KW = KW_;          // key warps per head group
  static constexpr int KBW = KBW_;        // 16-row blocks per key warp per stage
  static constexpr int STAGES = STAGES_;
  static constexpr int kHalvesK = DK / 64;  // 64-column (128-byte) TMA boxes per K row
  static constexpr int kHalvesV = DV / 64;
  static constexpr int kTile = 16 * KW * KBW;
  static constexpr int kConsumerWarps = HG * KW;
  static constexpr int kConsumerThreads = 32 * kConsumerWarps;
  static constexpr int kThreads = kConsumerThreads + 32;
  static constexpr int kHPW = 8 * NB;            // heads per warp
  static constexpr int kHeadsPerCta = kHPW * HG;
  static constexpr int kHalfBytes = kTile * 128;
  static constexpr int kTileBytesK = kTile * DK * 2;  // the K tile; the V tile follows it
  static constexpr int kStageBytes = kTileBytesK + kTile * DV * 2;
  static constexpr int kSlotStride = DV + 4;     // padded row of the epilogue slots
  static constexpr int kEpiAccFloats = HG * KW * kHPW * kSlotStride;
  static constexpr int kEpiMLFloats = 2 * HG * KW * kHPW;
  // schedule: first[kMaxBatchPerLaunch + 1], lens[kMaxBatchPerLaunch], red[48]
  // (rounded up to an even count of 4-byte words)
  static constexpr int kSchedWords = da::kSchedWords;  // work list (common.cuh)
  static constexpr int kQBytes = kHeadsPerCta * DK * 2;   // q rows of one item, per stage
  static constexpr int kNewBytes = (DK + DV) * 2;          // appended K and V rows, per stage
  static constexpr size_t kSmemBytes = 1024 + size_t(STAGES) * (kStageBytes + kQBytes + kNewBytes) +
                                       size_t(kEpiAccFloats + kEpiMLFloats + kSchedWords) * 4 +
                                       2 * STAGES * 8 + 16;
  static_assert(DK % 64 == 0 && DV % 64 == 0 && DK <= 256 && DV <= 256, "head dims");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert((kEpiAccFloats + kEpiMLFloats) % 2 == 0, "mbarrier alignment");
};

// Byte offset of element column `col` (a multiple of 8) of tile row `row`
// inside one tensor's tile: 64-column halves, 128-byte rows, 128-byte swizzle.
template <class Cfg>
__device__ __forceinline__ uint32_t swz(int row, int col) {
  const int half = col >> 6;
  const int chunk = (col & 63) >> 3;
  return uint32_t(half * Cfg::kHalfBytes + row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    split_decode_bf16_kernel(const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
  constexpr int DK = Cfg::DK, DV = Cfg::DV, NB = Cfg::NB, KW = Cfg::KW, KBW = Cfg::KBW,
                STAGES = Cfg::STAGES;
  constexpr int kHPW = Cfg::kHPW;
  constexpr int MBK = DK / 16;  // 16-wide blocks of d_k (Step I)
  constexpr int MB = DV / 16;   // 16-wide blocks of d_v (Step III)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* qslots = smem + size_t(STAGES) * Cfg::kStageBytes;
  uint8_t* newslots = qslots + size_t(STAGES) * Cfg::kQBytes;
  float* epi_acc = reinterpret_cast<float*>(newslots + size_t(STAGES) * Cfg::kNewBytes);
  float* epi_m = epi_acc + Cfg::kEpiAccFloats;
  float* epi_l = epi_m + Cfg::HG * KW * kHPW;
  int* sched_words = reinterpret_cast<int*>(epi_l + Cfg::HG * KW * kHPW);
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
  }
  int4 hint = make_int4(0, 0, 0, 0);
  if (threadIdx.x == Cfg::kConsumerThreads) hint = load_hint(p);  // producer lane
  // Launched as a programmatic dependent: the set-up here overlaps the tail
  // of the previous grid on the stream, which may have produced seq_lens, q,
  // the caches or the new rows.  Before the wait below, only the hinted L2
  // prefetch and the work list touch them: the prefetch is a hint, and the
  // list is built on the lengths as they read now (shared memory only), then
  // checked and built again if they changed once the wait is over.  The hint
  // is loaded first and used after the build, so that its round trip does
  // not hold the build's first barrier.
  Schedule sched = build_schedule_core<Cfg::kTile>(p, sched_words);
  if (threadIdx.x == Cfg::kConsumerThreads)
    prefetch_hinted<Cfg::kTile, Cfg::kHalvesK, Cfg::kHalvesV, 64>(p, hint, &tmK, &tmV, STAGES);
  wait_for_prerequisite_grid();
  sched = commit_schedule<Cfg::kTile>(p, sched_words, sched);
  allow_dependent_launch();
  if (threadIdx.x == 0 && sched.mine > 0) write_hint<Cfg::kTile>(p, cta_item<Cfg::kTile>(p, sched, 0), STAGES);

  // ------------------------------------------------------------------ producer
  if (warp == Cfg::kConsumerWarps) {
    if (lane == 0)
      produce<Cfg::kTile, STAGES, Cfg::kStageBytes, Cfg::kHalvesK, Cfg::kHalvesV, 64,
              Cfg::kHalfBytes, Cfg::kTileBytesK, Cfg::kHeadsPerCta, DK * 2, DK * 2, DV * 2>(&tmK, &tmV, p, sched, ring, smem_u32(qslots),
                                        smem_u32(newslots), full0, empty0, abort_flag);
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int hg = warp / KW;
  const int kw = warp % KW;
  const int r = lane >> 2;  // MMA fragment row group
  const int c = lane & 3;   // MMA fragment column pair
  int stage = 0;
  uint32_t phase = 0;

  for (int k = 0; k < sched.mine; ++k) {
    const Item it = cta_item<Cfg::kTile>(p, sched, k);

    // Query heads of this warp: group-local index hl = hc*HeadsPerCta + hg*kHPW + nb*8 + n.
    // Their bf16 rows arrive with the item's first stage (rows past the group are zero).
    const int head_base = it.hc * Cfg::kHeadsPerCta + hg * kHPW;
    uint32_t qf[NB][MBK][2];

    float m_run[NB][2], l_run[NB][2];
    float acc[MB][NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      m_run[nb][0] = m_run[nb][1] = -INFINITY;
      l_run[nb][0] = l_run[nb][1] = 0.f;
    }
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mb][nb][e] = 0.f;

    for (int t = 0; t < it.tiles; ++t) {
      if (!mbar_wait_bounded(full0 + 8 * stage, phase, abort_flag)) {
        if (!*abort_flag) {
          *abort_flag = 1;
          flag_error(p.dev_error, DA_DEVERR_TIMEOUT);
        }
      }
      const uint32_t kbase = ring + stage * Cfg::kStageBytes;
      const uint32_t vbase = kbase + Cfg::kTileBytesK;
      const int tile_row0 = it.row_begin + t * Cfg::kTile;
      const int valid = min(Cfg::kTile, it.row_end - tile_row0);
      const int key0 = kw * KBW * 16;  // first row of this warp inside the stage
      // A row appended by this call replaces the stale cache row the tile load
      // brought in.
      const int new_local = (it.new_row >= tile_row0 && it.new_row < tile_row0 + Cfg::kTile)
                                ? it.new_row - tile_row0
                                : -1;
      if (new_local >= 0) {  // the same for every consumer warp
        if (warp == 0 && !*abort_flag) {
          // Put the appended rows into the stage, in the tile's swizzled layout,
          // and (once per kv head) into the caches.
          const uint8_t* slot = newslots + size_t(stage) * Cfg::kNewBytes;
          uint8_t* ktile = smem + size_t(stage) * Cfg::kStageBytes;
          uint8_t* vtile = ktile + Cfg::kTileBytesK;
          for (int ch = lane; ch < DK / 8; ch += 32) {
            const int col = ch * 8;
            *reinterpret_cast<uint4*>(ktile + swz<Cfg>(new_local, col)) =
                *reinterpret_cast<const uint4*>(slot + col * 2);
          }
          for (int ch = lane; ch < DV / 8; ch += 32) {
            const int col = ch * 8;
            *reinterpret_cast<uint4*>(vtile + swz<Cfg>(new_local, col)) =
                *reinterpret_cast<const uint4*>(slot + DK * 2 + col * 2);
          }
          if (it.hc == 0) store_new_row<DK * 2, DV * 2>(p, it, slot, lane);
          fence_proxy_async_smem();
        }
        named_bar_sync(2, Cfg::kConsumerThreads);
      }
      if (t == 0) {
        const uint32_t* qs =
            reinterpret_cast<const uint32_t*>(qslots + size_t(stage) * Cfg::kQBytes);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const int hloc = hg * kHPW + nb * 8 + r;  // head inside the item
          const bool ok = head_base + nb * 8 + r < p.group;
#pragma unroll
          for (int ks = 0; ks < MBK; ++ks) {
            qf[nb][ks][0] = ok ? qs[hloc * (DK / 2) + ks * 8 + c] : 0u;
            qf[nb][ks][1] = ok ? qs[hloc * (DK / 2) + ks * 8 + 4 + c] : 0u;
          }
        }
      }

      // warp-uniform (the MMAs and shuffles below need the whole warp)
      const bool live = __all_sync(0xffffffffu, !*abort_flag);
      if (live && key0 < valid) {
        // ---- Step I: scores for KBW blocks of 16 rows.
        float s[KBW][NB][4];
#pragma unroll
        for (int kb = 0; kb < KBW; ++kb)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[kb][nb][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < MBK; ++ks) {
#pragma unroll
          for (int kb = 0; kb < KBW; ++kb) {
            const int row = key0 + kb * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
            const int col = ks * 16 + (lane >> 4) * 8;
            uint32_t a[4];
            ldmatrix_x4(a, kbase + swz<Cfg>(row, col));
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(s[kb][nb], a, qf[nb][ks][0], qf[nb][ks][1]);
          }
        }

        // ---- Step II: mask rows past the end, scale, running max and sum.
        float alpha[NB][2];
        bool changed = false;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float mx = -INFINITY;
#pragma unroll
            for (int kb = 0; kb < KBW; ++kb) {
              const int row_lo = key0 + kb * 16 + r;
              s[kb][nb][j] = row_lo < valid ? s[kb][nb][j] * p.scale_log2 : -INFINITY;
              s[kb][nb][j + 2] = row_lo + 8 < valid ? s[kb][nb][j + 2] * p.scale_log2 : -INFINITY;
              mx = fmaxf(mx, fmaxf(s[kb][nb][j], s[kb][nb][j + 2]));
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float m_new = fmaxf(m_run[nb][j], mx);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            alpha[nb][j] = ex2(m_run[nb][j] - m_use);
            changed |= (m_new != m_run[nb][j]);
            m_run[nb][j] = m_new;
            float sum = 0.f;
#pragma unroll
            for (int kb = 0; kb < KBW; ++kb) {
              s[kb][nb][j] = ex2(s[kb][nb][j] - m_use);
              s[kb][nb][j + 2] = ex2(s[kb][nb][j + 2] - m_use);
              sum += s[kb][nb][j] + s[kb][nb][j + 2];
            }
            l_run[nb][j] = l_run[nb][j] * alpha[nb][j] + sum;
          }
        }
        if (__any_sync(0xffffffffu, changed)) {
#pragma unroll
          for (int mb = 0; mb < MB; ++mb)
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              acc[mb][nb][0] *= alpha[nb][0];
              acc[mb][nb][1] *= alpha[nb][1];
              acc[mb][nb][2] *= alpha[nb][0];
              acc[mb][nb][3] *= alpha[nb][1];
            }
        }

        // ---- Step III: O^T += V^T . P^T, P as bf16 head + bf16 remainder.
#pragma unroll
        for (int kb = 0; kb < KBW; ++kb) {
          uint32_t ph[NB][2], pl[NB][2];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const uint32_t h0 = pack_bf16x2(s[kb][nb][0], s[kb][nb][1]);  // row r
            const uint32_t h1 = pack_bf16x2(s[kb][nb][2], s[kb][nb][3]);  // row r + 8
            const uint32_t l0 = pack_bf16x2(s[kb][nb][0] - bf16_lo_to_f32(h0),
                                            s[kb][nb][1] - bf16_hi_to_f32(h0));
            const uint32_t l1 = pack_bf16x2(s[kb][nb][2] - bf16_lo_to_f32(h1),
                                            s[kb][nb][3] - bf16_hi_to_f32(h1));
            ph[nb][0] = movmatrix_trans(h0);
            ph[nb][1] = movmatrix_trans(h1);
            pl[nb][0] = movmatrix_trans(l0);
            pl[nb][1] = movmatrix_trans(l1);
          }
          const int blk0 = key0 + kb * 16;
          const bool partial = blk0 + 16 > valid;
          // rows held by this lane's A registers: {2c, 2c+1} and {8+2c, 9+2c}
          const uint32_t mlo = (blk0 + 2 * c < valid ? 0x0000ffffu : 0u) |
                               (blk0 + 2 * c + 1 < valid ? 0xffff0000u : 0u);
          const uint32_t mhi = (blk0 + 8 + 2 * c < valid ? 0x0000ffffu : 0u) |
                               (blk0 + 9 + 2 * c < valid ? 0xffff0000u : 0u);
#pragma unroll
          for (int mb = 0; mb < MB; ++mb) {
            const int row = blk0 + (lane & 7) + ((lane >> 4) & 1) * 8;
            const int col = mb * 16 + ((lane >> 3) & 1) * 8;
            uint32_t a[4];
            ldmatrix_x4_trans(a, vbase + swz<Cfg>(row, col));
            if (partial) {  // rows past the end may hold anything, even NaN
              a[0] &= mlo;
              a[1] &= mlo;
              a[2] &= mhi;
              a[3] &= mhi;
            }
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              mma_bf16_16816(acc[mb][nb], a, ph[nb][0], ph[nb][1]);
              mma_bf16_16816(acc[mb][nb], a, pl[nb][0], pl[nb][1]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * stage);
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    }

    // ---- Epilogue: per-warp state to shared slots, then the shared finish.
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float v = l_run[nb][j];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        l_run[nb][j] = v;
      }
    named_bar_sync(1, Cfg::kConsumerThreads);  // earlier readers of the slots are done
    const int slot_id = hg * KW + kw;
    float* slot = epi_acc + slot_id * kHPW * Cfg::kSlotStride;
    if (lane < 4) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          epi_m[slot_id * kHPW + nb * 8 + 2 * lane + j] = m_run[nb][j];
          epi_l[slot_id * kHPW + nb * 8 + 2 * lane + j] = l_run[nb][j];
        }
    }
#pragma unroll
    for (int mb = 0; mb < MB; ++mb)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int d0 = mb * 16 + r;
        const int h0 = nb * 8 + 2 * c;
        slot[h0 * Cfg::kSlotStride + d0] = acc[mb][nb][0];
        slot[(h0 + 1) * Cfg::kSlotStride + d0] = acc[mb][nb][1];
        slot[h0 * Cfg::kSlotStride + d0 + 8] = acc[mb][nb][2];
        slot[(h0 + 1) * Cfg::kSlotStride + d0 + 8] = acc[mb][nb][3];
      }
    named_bar_sync(1, Cfg::kConsumerThreads);
    finish_item<DV, Cfg::HG, KW, kHPW, Cfg::kSlotStride>(p, it, epi_acc, epi_m, epi_l, threadIdx.x,
                                                        Cfg::kConsumerThreads, abort_flag);
  }
}

// ---------------------------------------------------------------------------
// Variant table and launcher.
// ---------------------------------------------------------------------------
using Bf16G8D128 = Bf16Cfg<128, 128, 1, 1, 4, 2, 3>;
using Bf16G8D64 = Bf16Cfg<64, 64, 1, 1, 4, 2, 6>;
using Bf16G16D64 = Bf16Cfg<64, 64, 2, 1, 4, 1, 8>;
using Bf16G32D64 = Bf16Cfg<64, 64, 2, 2, 4, 1, 8>;
using Bf16G8D256 = Bf16Cfg<256, 256, 1, 1, 4, 1, 2>;   // 64-row stages of 64 KB
using Bf16G8D192V128 = Bf16Cfg<192, 128, 1, 1, 4, 1, 3>;

template <class Cfg>
static KernelShape shape_of() {
  return KernelShape{Cfg::kTile, Cfg::kHeadsPerCta, 64, 1, 1.5f};
}

// (d_k, d_v) pairs with a variant; groups above a variant's heads per work
// item are covered by several head chunks.
KernelShape bf16_shape(int d_k, int d_v, int group) {
  if (d_k == 256) return shape_of<Bf16G8D256>();
  if (d_k == 192) return shape_of<Bf16G8D192V128>();
  if (d_k == 128) return shape_of<Bf16G8D128>();  // larger groups use the tcgen05 kernel
  if (group <= 8) return shape_of<Bf16G8D64>();
  if (group <= 16) return shape_of<Bf16G16D64>();
  return shape_of<Bf16G32D64>();
}

template <class Cfg>
static cudaError_t launch_cfg(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int grid, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(split_decode_bf16_kernel<Cfg>, Cfg::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  return launch_dependent(split_decode_bf16_kernel<Cfg>, grid, Cfg::kThreads, Cfg::kSmemBytes, stream, tk, tv,
                          p);
}

cudaError_t launch_split_bf16(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                              int d_k, int d_v, int grid, cudaStream_t stream) {
  if (d_k == 256) return launch_cfg<Bf16G8D256>(p, tk, tv, grid, stream);
  if (d_k == 192) return launch_cfg<Bf16G8D192V128>(p, tk, tv, grid, stream);
  if (d_k == 128) return launch_cfg<Bf16G8D128>(p, tk, tv, grid, stream);
  if (p.group <= 8) return launch_cfg<Bf16G8D64>(p, tk, tv, grid, stream);
  if (p.group <= 16) return launch_cfg<Bf16G16D64>(p, tk, tv, grid, stream);
  return launch_cfg<Bf16G32D64>(p, tk, tv, grid, stream);
}

}  // namespace da
