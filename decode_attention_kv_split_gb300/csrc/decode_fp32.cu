// Split-KV decode attention for fp32 caches on CUDA cores (sm_103a).
//
// Same pipeline as the bf16 kernel (persistent CTAs, a producer warp feeding
// a ring of shared-memory stages with 3-D TMA loads, consumer warps, mbarrier
// hand-off), but the arithmetic stays in fp32 FMAs: with one query head per
// kv head the work is about half a flop per byte ("Attention over the KV
// cache in the decode step": arithmetic intensity = h_q/h_kv flop per bf16
// byte), far below what the CUDA cores deliver.
//
// Lanes run along the contiguous d axis of each cached row, so a warp reads
// one whole row per instruction (coalescing criterion of "MoA-Structured
// Decode Attention", section 4).  Each consumer warp owns a contiguous block
// of rows in every stage and keeps its own running max and running sum
// (section 2, Steps I-III evaluated as an online softmax); the warps are
// merged by log-sum-exp at the end of each work item.
#include <math.h>

#include "common.cuh"

namespace da {

template <int D_, int G_, int W_, int TILE_, int STAGES_>
struct F32Cfg {
  static constexpr int D = D_;        // head dim (d_k == d_v)
  static constexpr int G = G_;        // query heads per work item
  static constexpr int W = W_;        // consumer warps
  static constexpr int kTile = TILE_; // rows per stage
  static constexpr int STAGES = STAGES_;
  static constexpr int kEPL = D / 32; // elements per lane
  static constexpr int kRowsPerWarp = kTile / W;
  static constexpr int kConsumerThreads = 32 * W;
  static constexpr int kThreads = kConsumerThreads + 32;
  static constexpr int kTileBytes = kTile * D * 4;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kEpiAccFloats = W * G * D;
  static constexpr int kEpiMLFloats = 2 * W * G;
  static constexpr int kSchedWords = da::kSchedWords;  // work list (common.cuh)
  static constexpr int kQBytes = G * D * 4;  // q rows of one item, per stage
  static constexpr int kNewBytes = 2 * D * 4;  // appended K and V rows, per stage
  static constexpr size_t kSmemBytes = 1024 + size_t(STAGES) * (kStageBytes + kQBytes + kNewBytes) +
                                       size_t(kEpiAccFloats + kEpiMLFloats + kSchedWords) * 4 +
                                       2 * STAGES * 8 + 16;
  static_assert((kEpiAccFloats + kEpiMLFloats) % 2 == 0, "mbarrier alignment");
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(kTile % W == 0, "rows per warp");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

template <int N>
__device__ __forceinline__ void load_lane(float (&v)[N], const float* p) {
  if constexpr (N == 4) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
  } else {
    const float2 x = *reinterpret_cast<const float2*>(p);
    v[0] = x.x, v[1] = x.y;
  }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    split_decode_f32_kernel(const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
  constexpr int D = Cfg::D, G = Cfg::G, W = Cfg::W, STAGES = Cfg::STAGES, EPL = Cfg::kEPL;
  constexpr int RPW = Cfg::kRowsPerWarp;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* qslots = smem + size_t(STAGES) * Cfg::kStageBytes;
  uint8_t* newslots = qslots + size_t(STAGES) * Cfg::kQBytes;
  float* epi_acc = reinterpret_cast<float*>(newslots + size_t(STAGES) * Cfg::kNewBytes);
  float* epi_m = epi_acc + Cfg::kEpiAccFloats;
  float* epi_l = epi_m + W * G;
  int* sched_words = reinterpret_cast<int*>(epi_l + W * G);
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
      mbar_init(empty0 + 8 * s, W);
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
    prefetch_hinted<Cfg::kTile, 1, 1, 0>(p, hint, &tmK, &tmV, STAGES);
  wait_for_prerequisite_grid();
  sched = commit_schedule<Cfg::kTile>(p, sched_words, sched);
  allow_dependent_launch();
  if (threadIdx.x == 0 && sched.mine > 0) write_hint<Cfg::kTile>(p, cta_item<Cfg::kTile>(p, sched, 0), STAGES);

  // ------------------------------------------------------------------ producer
  if (warp == W) {
    if (lane == 0)
      produce<Cfg::kTile, STAGES, Cfg::kStageBytes, 1, 1, 0, 0, Cfg::kTileBytes, G, D * 4, D * 4,
              D * 4>(
          &tmK, &tmV, p, sched, ring, smem_u32(qslots), smem_u32(newslots), full0, empty0,
          abort_flag);
    return;
  }

  // ------------------------------------------------------------------ consumers
  int stage = 0;
  uint32_t phase = 0;

  for (int k = 0; k < sched.mine; ++k) {
    const Item it = cta_item<Cfg::kTile>(p, sched, k);

    const int head_base = it.hc * G;  // group-local index of this item's first head
    // q (pre-multiplied by scale * log2(e) once loaded, so scores come out in
    // the log2 domain) arrives with the item's first stage.
    float qv[G][EPL];

    float m_run[G], l_run[G], acc[G][EPL];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -INFINITY;
      l_run[g] = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[g][e] = 0.f;
    }

    for (int t = 0; t < it.tiles; ++t) {
      if (!mbar_wait_bounded(full0 + 8 * stage, phase, abort_flag)) {
        if (!*abort_flag) {
          *abort_flag = 1;
          flag_error(p.dev_error, DA_DEVERR_TIMEOUT);
        }
      }
      const float* ks = reinterpret_cast<const float*>(smem + size_t(stage) * Cfg::kStageBytes);
      const float* vs = ks + Cfg::kTile * D;
      if (t == 0) {
        const float* qs = reinterpret_cast<const float*>(qslots + size_t(stage) * Cfg::kQBytes);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float tmp[EPL];
          load_lane<EPL>(tmp, qs + g * D + lane * EPL);
          const bool ok = head_base + g < p.group;
#pragma unroll
          for (int e = 0; e < EPL; ++e) qv[g][e] = ok ? tmp[e] * p.scale_log2 : 0.f;
        }
      }
      const int tile_row0 = it.row_begin + t * Cfg::kTile;
      const int valid = min(Cfg::kTile, it.row_end - tile_row0);
      const int row0 = warp * RPW;
      const int nrows = min(RPW, valid - row0);  // may be <= 0
      // A row appended by this call replaces the stale cache row the tile load
      // brought in.
      const int new_local = (it.new_row >= tile_row0 && it.new_row < tile_row0 + Cfg::kTile)
                                ? it.new_row - tile_row0
                                : -1;
      if (new_local >= 0) {  // the same for every consumer warp
        if (warp == 0 && !*abort_flag) {
          // Put the appended rows into the stage and (once per kv head) into the caches.
          const uint8_t* slot = newslots + size_t(stage) * Cfg::kNewBytes;
          uint8_t* ktile = smem + size_t(stage) * Cfg::kStageBytes;
          uint8_t* vtile = ktile + Cfg::kTileBytes;
          for (int ch = lane; ch < D / 4; ch += 32) {
            reinterpret_cast<uint4*>(ktile + size_t(new_local) * D * 4)[ch] =
                reinterpret_cast<const uint4*>(slot)[ch];
            reinterpret_cast<uint4*>(vtile + size_t(new_local) * D * 4)[ch] =
                reinterpret_cast<const uint4*>(slot + D * 4)[ch];
          }
          if (it.hc == 0) store_new_row<D * 4, D * 4>(p, it, slot, lane);
          fence_proxy_async_smem();
        }
        named_bar_sync(2, Cfg::kConsumerThreads);
      }

      // warp-uniform (the shuffles below need the whole warp)
      const bool live = __all_sync(0xffffffffu, !*abort_flag);
      if (live && nrows > 0) {
        // Step I: s[g][r] = (scale*log2e*q_g) . K_row, reduced across the warp.
        float s[G][RPW];
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
          float kv[EPL];
          load_lane<EPL>(kv, ks + (row0 + rr) * D + lane * EPL);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float x = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) x = fmaf(qv[g][e], kv[e], x);
            s[g][rr] = x;
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int rr = 0; rr < RPW; ++rr) {
            float x = s[g][rr];
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            x += __shfl_xor_sync(0xffffffffu, x, 2);
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            s[g][rr] = rr < nrows ? x : -INFINITY;
          }
        // Step II: running max and sum (warp-uniform values).
        float alpha[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float mx = -INFINITY;
#pragma unroll
          for (int rr = 0; rr < RPW; ++rr) mx = fmaxf(mx, s[g][rr]);
          const float m_new = fmaxf(m_run[g], mx);
          const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
          alpha[g] = ex2(m_run[g] - m_use);
          m_run[g] = m_new;
          float sum = 0.f;
#pragma unroll
          for (int rr = 0; rr < RPW; ++rr) {
            s[g][rr] = ex2(s[g][rr] - m_use);
            sum += s[g][rr];
          }
          l_run[g] = l_run[g] * alpha[g] + sum;
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[g][e] *= alpha[g];
        }
        // Step III: acc += p * V_row over the valid rows of this warp.
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
          if (rr < nrows) {
            float vv[EPL];
            load_lane<EPL>(vv, vs + (row0 + rr) * D + lane * EPL);
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
              for (int e = 0; e < EPL; ++e) acc[g][e] = fmaf(s[g][rr], vv[e], acc[g][e]);
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

    // Epilogue: merge the W warps, normalise, store.
    named_bar_sync(1, Cfg::kConsumerThreads);
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        epi_m[warp * G + g] = m_run[g];
        epi_l[warp * G + g] = l_run[g];
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < EPL; ++e) epi_acc[(warp * G + g) * D + lane * EPL + e] = acc[g][e];
    named_bar_sync(1, Cfg::kConsumerThreads);
    finish_item<D, 1, W, G, D>(p, it, epi_acc, epi_m, epi_l, threadIdx.x,
                               Cfg::kConsumerThreads, abort_flag);
  }
}

// ---------------------------------------------------------------------------
// Variant table and launcher.
// ---------------------------------------------------------------------------
template <int D>
using F32G1 = F32Cfg<D, 1, 8, (D == 128 ? 32 : 64), 5>;
template <int D>
using F32G2 = F32Cfg<D, 2, 8, (D == 128 ? 32 : 64), 5>;
template <int D>
using F32G4 = F32Cfg<D, 4, 8, (D == 128 ? 32 : 64), 5>;
template <int D>
using F32G8 = F32Cfg<D, 8, 8, (D == 128 ? 32 : 64), 5>;

template <class Cfg>
static KernelShape f32_shape_of() {
  return KernelShape{Cfg::kTile, Cfg::G, Cfg::D, 0, 1.5f};
}

template <int D>
static KernelShape f32_shape_d(int group) {
  if (group <= 1) return f32_shape_of<F32G1<D>>();
  if (group <= 2) return f32_shape_of<F32G2<D>>();
  if (group <= 4) return f32_shape_of<F32G4<D>>();
  return f32_shape_of<F32G8<D>>();
}

KernelShape f32_shape(int d, int group) {
  return d == 128 ? f32_shape_d<128>(group) : f32_shape_d<64>(group);
}

template <class Cfg>
static cudaError_t launch_f32_cfg(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                  int grid, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(split_decode_f32_kernel<Cfg>, Cfg::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  return launch_dependent(split_decode_f32_kernel<Cfg>, grid, Cfg::kThreads, Cfg::kSmemBytes, stream, tk, tv,
                          p);
}

template <int D>
static cudaError_t launch_f32_d(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                                int grid, cudaStream_t stream) {
  if (p.group <= 1) return launch_f32_cfg<F32G1<D>>(p, tk, tv, grid, stream);
  if (p.group <= 2) return launch_f32_cfg<F32G2<D>>(p, tk, tv, grid, stream);
  if (p.group <= 4) return launch_f32_cfg<F32G4<D>>(p, tk, tv, grid, stream);
  return launch_f32_cfg<F32G8<D>>(p, tk, tv, grid, stream);
}

cudaError_t launch_split_f32(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             int d, int grid, cudaStream_t stream) {
  return d == 128 ? launch_f32_d<128>(p, tk, tv, grid, stream)
                  : launch_f32_d<64>(p, tk, tv, grid, stream);
}

}  // namespace da
