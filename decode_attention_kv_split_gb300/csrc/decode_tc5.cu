// Split-KV decode attention for bf16 caches and large query groups on the
// fifth-generation tensor cores (tcgen05, TMEM accumulators), sm_103a.
//
// For a group of NH query heads sharing one kv head (MQA-like), the score
// block of a 128-row stage is a real GEMM: S^T[128 rows x NH heads] =
// K_stage[128 x d] . Q^T[d x NH] ("MoA-Structured Decode Attention",
// section 2, Step I, lifted to NH query rows by the Omega rank argument),
// and the weighted sum is O^T[d x NH] += V_stage^T[d x 128] . P^T[128 x NH]
// (Step III).  Keeping the cached rows as the MMA's M dimension (128) means
// no MMA work is padding whatever NH is (16 or 32).
//
// Roles (352 threads):
//   warps 0-7  softmax: warp w owns stage rows 32*(w%4)..+31 of S^T (its TMEM
//              lane quarter; for the output, columns d of O^T) and half of the
//              heads.  Per stage: load the scores, mask rows past the end,
//              exponentiate against a lazily updated running max (a vote finds
//              scores more than 2^8 above it; only then is the exact per-head
//              maximum over the 128 rows taken and the accumulator rescaled),
//              and write P^T as a bf16 head plus a bf16 remainder into
//              swizzled shared memory.
//   warp 8     producer: TMA loads of the K and V stages (as the other kernels).
//   warp 9     score-MMA issuer: builds the swizzled Q of each item, patches an
//              appended K row into its stage, issues S^T = K . Q^T.
//   warp 10    P.V-MMA issuer: clears V rows past the end, patches an appended
//              V row, issues O^T += V^T . P^T.  The MMA commits release the
//              K and V slots and signal the softmax warps.
// Step II's online softmax is exact up to rounding: every exponent is taken
// against the same running max that scales the accumulator.
#include <math.h>

#include "common.cuh"

namespace da {
namespace tc5 {

__device__ __forceinline__ void alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D (TMEM) = A (smem) . B (smem)^T [+ D], bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once every MMA this thread issued so far has completed.
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void st8(uint32_t taddr, const float* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}
// n (8 or 16) consecutive columns.
__device__ __forceinline__ void ld16x(uint32_t taddr, float* v, int n) {
  if (n == 16) ld16(taddr, v); else ld8(taddr, v);
}
__device__ __forceinline__ void st16x(uint32_t taddr, const float* v, int n) {
  if (n == 16) st16(taddr, v); else st8(taddr, v);
}

// Shared-memory matrix descriptor, 128-byte swizzle.  K-major operands: rows
// of 128 bytes (64 bf16), SBO = 1024 between groups of 8 rows.  MN-major:
// LBO = byte distance between 64-element blocks along M/N, SBO = 1024
// between groups of 8 rows along K.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= uint64_t((saddr >> 4) & 0x3FFF);
  d |= uint64_t((lbo >> 4) & 0x3FFF) << 16;
  d |= uint64_t((sbo >> 4) & 0x3FFF) << 32;
  d |= uint64_t(1) << 46;  // descriptor version
  d |= uint64_t(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn_major) << 15) |
         (uint32_t(b_mn_major) << 16) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Byte offset of element (r, c) of a [rows][128] bf16 matrix stored as two
// [rows][64] halves with the 128-byte swizzle (the layout of the TMA stages).
__device__ __forceinline__ uint32_t sw128(int r, int c, int rows) {
  return uint32_t((c >> 6) * rows * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2);
}

}  // namespace tc5

template <int NH_, int KST_, int VST_>
struct Tc5Cfg {
  static constexpr int NH = NH_;    // query heads per item (MMA N)
  static constexpr int KST = KST_;  // K slots: freed when the score MMA completes
  static constexpr int VST = VST_;  // V slots: freed when the P.V MMA completes
  static constexpr int D = 128;
  static constexpr int kTile = 128;                    // rows per stage (MMA M)
  static constexpr int kHalfBytes = kTile * 128;       // one 64-column half of a tile
  static constexpr int kTileBytes = kTile * D * 2;     // one K or V tile
  static constexpr int kQBytes = NH * D * 2;           // swizzled Q of the current item
  // P^T of one stage as a [2 * NH rows][128 rows of the stage] K-major operand:
  // rows 0..NH-1 hold the bf16 head of P, rows NH..2NH-1 the bf16 remainder,
  // so one N = 2 * NH MMA accumulates both into O^T columns [0, NH) and [NH, 2NH).
  static constexpr int kPBytes = 2 * NH * kTile * 2;   // one buffer
  static constexpr int kRowBytes = D * 2;              // an appended row
  static constexpr int kSoftmaxWarps = 8;
  static constexpr int kThreads = 32 * (kSoftmaxWarps + 3);  // + producer + 2 MMA issuers
  static constexpr int kSchedWords = da::kSchedWords;  // work list (common.cuh)
  static constexpr int kRedGroup = 4 * (NH / 2) + 4;   // [4 quarters][NH/2] partials + 4 flags
  static constexpr int kRedFloats = 2 * 2 * kRedGroup; // two groups, double-buffered
  // kfull, kempty, vfull, vempty, s_full[2], p_full[2], pv_done[2], fin
  static constexpr int kBars = 2 * KST + 2 * VST + 2 + 2 + 2 + 1;
  static constexpr size_t kSmemBytes = 1024 + size_t(KST + VST) * (kTileBytes + kRowBytes) +
                                       kQBytes + 2 * kPBytes +
                                       size_t(kSchedWords + kRedFloats) * 4 + kBars * 8 + 32;
  static_assert(NH == 16 || NH == 32, "heads per item");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(kRedFloats % 2 == 0, "alignment");
};

// One ring of tile slots fed by one producer lane: every stage of the CTA's
// items, in order, into slot (stage % NSLOT).  Each load completes on the
// slot's full barrier; the slot is refilled after its empty barrier (an MMA
// commit).  The appended row of a unit rides with the tile that holds it.
template <int T, int NSLOT, int TILE_BYTES, int HALF_BYTES, int ROW_BYTES>
__device__ __forceinline__ void produce_ring(const CUtensorMap* map, const void* new_rows,
                                             const SplitParams& p, const Schedule& s,
                                             uint32_t slots, uint32_t newslots, uint32_t full0,
                                             uint32_t empty0, volatile int* abort_flag,
                                             bool may_withhold) {
  prefetch_tmap(map);
  const uint64_t policy = l2_policy_evict_first();
  int slot = 0;
  uint32_t phase = 0, issued = 0, issued_parity = 0;
  bool aborted = false;
  for (int k = 0; k < s.mine && !aborted; ++k) {
    const Item it = cta_item<T>(p, s, k);
    const int z = (p.b_offset + it.b) * p.h_kv + it.kvh;
    for (int t = 0; t < it.tiles; ++t) {
      if (!mbar_wait_bounded(empty0 + 8 * slot, phase ^ 1u, abort_flag)) {
        *abort_flag = 1;
        flag_error(p.dev_error, DA_DEVERR_TIMEOUT);
        aborted = true;
        break;
      }
      if (may_withhold && test_withhold(p, k, t, it.tiles)) {  // test builds only
        if (++slot == NSLOT) {
          slot = 0;
          phase ^= 1u;
        }
        continue;
      }
      const uint32_t bar = full0 + 8 * slot;
      const int y0 = it.row_begin + t * T;
      const bool with_new = it.new_row >= y0 && it.new_row < y0 + T;
      mbar_arrive_expect_tx(bar, TILE_BYTES + (with_new ? ROW_BYTES : 0));
      const uint32_t dst = slots + slot * TILE_BYTES;
      tma_load_3d(dst, map, 0, y0, z, bar, policy);
      tma_load_3d(dst + HALF_BYTES, map, 64, y0, z, bar, policy);
      if (with_new)  // (a checked build flags a row outside k_new / v_new and leaves the stage short)
        if (DA_IN(p, size_t(it.b) * p.h_kv + it.kvh, size_t(p.B) * p.h_kv))
          bulk_load(newslots + slot * ROW_BYTES,
                    static_cast<const char*>(new_rows) + (size_t(it.b) * p.h_kv + it.kvh) * ROW_BYTES,
                    ROW_BYTES, bar);
      issued |= 1u << slot;
      issued_parity = (issued_parity & ~(1u << slot)) | (phase << slot);
      if (++slot == NSLOT) {
        slot = 0;
        phase ^= 1u;
      }
    }
  }
  if (aborted) {
    volatile int never = 0;
    for (int st = 0; st < NSLOT; ++st)
      if (issued & (1u << st)) mbar_wait_bounded(full0 + 8 * st, (issued_parity >> st) & 1u, &never);
  }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, 1)
    split_decode_tc5_kernel(const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const SplitParams p) {
  constexpr int NH = Cfg::NH, KST = Cfg::KST, VST = Cfg::VST, D = Cfg::D, T = Cfg::kTile;
  // TMEM: S[2] (NH columns each), then O^T as two accumulation chains (even
  // and odd 16-row blocks of a stage), each 2 NH columns (head | remainder).
  constexpr uint32_t kTmemCols = 256;
  constexpr float kLazy = 8.f;         // rescale only when a max grows by > 2^8

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* kslots = smem;                                        // [KST] K tiles
  uint8_t* vslots = kslots + size_t(KST) * Cfg::kTileBytes;      // [VST] V tiles
  uint8_t* qsw = vslots + size_t(VST) * Cfg::kTileBytes;         // 1024-aligned
  uint8_t* p_buf = qsw + Cfg::kQBytes;  // [2 buffers][kPBytes], 1024-aligned
  uint8_t* knew = p_buf + 2 * Cfg::kPBytes;                      // [KST] appended K rows
  uint8_t* vnew = knew + size_t(KST) * Cfg::kRowBytes;           // [VST] appended V rows
  int* sched_words = reinterpret_cast<int*>(vnew + size_t(VST) * Cfg::kRowBytes);
  float* red = reinterpret_cast<float*>(sched_words + Cfg::kSchedWords);
  uint64_t* bars = reinterpret_cast<uint64_t*>(red + Cfg::kRedFloats);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::kBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t kfull0 = smem_u32(bars);
  const uint32_t kempty0 = kfull0 + 8 * KST;
  const uint32_t vfull0 = kempty0 + 8 * KST;
  const uint32_t vempty0 = vfull0 + 8 * VST;
  const uint32_t s_full0 = vempty0 + 8 * VST;  // per S buffer
  const uint32_t p_full0 = s_full0 + 16;       // per P buffer
  const uint32_t pv_done0 = p_full0 + 16;      // per P buffer
  const uint32_t fin = pv_done0 + 16;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < KST; ++s) {
      mbar_init(kfull0 + 8 * s, 1);
      mbar_init(kempty0 + 8 * s, 1);  // released by one tcgen05.commit
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(vfull0 + 8 * s, 1);
      mbar_init(vempty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full0 + 8 * b, 1);
      mbar_init(p_full0 + 8 * b, Cfg::kSoftmaxWarps);  // one arrival per softmax warp
      mbar_init(pv_done0 + 8 * b, 1);
    }
    mbar_init(fin, 2);  // one commit from each MMA issuer
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tc5::alloc(smem_u32(tmem_slot), kTmemCols);
    tc5::relinquish();
  }
  if (threadIdx.x == 32) {  // the tensor maps do not depend on the preceding grid
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  int4 hint = make_int4(0, 0, 0, 0);
  if (threadIdx.x == 8 * 32) hint = load_hint(p);  // producer warp
  // Launched as a programmatic dependent: the set-up here overlaps the tail
  // of the previous grid on the stream, which may have produced seq_lens, q,
  // the caches or the new rows.  Before the wait below, only the hinted L2
  // prefetch and the work list touch them: the prefetch is a hint, and the
  // list is built on the lengths as they read now (shared memory only), then
  // checked and built again if they changed once the wait is over.  The hint
  // is loaded first and used after the build, so that its round trip does
  // not hold the build's first barrier.
  tc5::fence_before();
  Schedule sched = build_schedule_core<T>(p, sched_words);
  if (threadIdx.x == 8 * 32) prefetch_hinted<T, 2, 2, 64>(p, hint, &tmK, &tmV, KST);
  wait_for_prerequisite_grid();
  sched = commit_schedule<T>(p, sched_words, sched);
  tc5::fence_after();
  allow_dependent_launch();
  if (threadIdx.x == 0 && sched.mine > 0) write_hint<T>(p, cta_item<T>(p, sched, 0), KST);
  const uint32_t tmem = *tmem_slot;
  const uint32_t s_col0 = tmem, o_col = tmem + 2 * NH;  // chain c at o_col + c * 2 NH

  // ------------------------------------------------------------------ producers
  if (warp == 8) {
    if (lane == 0)
      produce_ring<T, KST, Cfg::kTileBytes, Cfg::kHalfBytes, Cfg::kRowBytes>(
          &tmK, p.k_new, p, sched, smem_u32(kslots), smem_u32(knew), kfull0, kempty0, abort_flag,
          true);
    else if (lane == 1)
      produce_ring<T, VST, Cfg::kTileBytes, Cfg::kHalfBytes, Cfg::kRowBytes>(
          &tmV, p.v_new, p, sched, smem_u32(vslots), smem_u32(vnew), vfull0, vempty0, abort_flag,
          false);
    return;
  }

  // ------------------------------------------------------------------ MMA issuers
  // Warp 9 issues the score MMAs, warp 10 the P.V MMAs: two independent
  // accumulation chains that the tensor core overlaps.
  if (warp == 9 || warp == 10) {
    uint32_t j = 0;  // stages processed by this CTA (all items)
    bool aborted = false;
    // Whole warp: wait (lane 0) on a barrier; false on timeout.
    auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
      bool ok = true;
      if (lane == 0) ok = mbar_wait_bounded(bar, parity, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok && !aborted) {
        aborted = true;
        if (lane == 0) {
          *abort_flag = 1;
          flag_error(p.dev_error, DA_DEVERR_TIMEOUT);
        }
      }
      return ok;
    };
    if (warp == 9) {
      // ---- scores: S^T[j % 2] = K_j . Q^T
      const uint32_t idesc_s = tc5::idesc_bf16(128, NH, 0, 0);
      int kslot = 0;
      uint32_t kphase = 0;
      for (int k = 0; k < sched.mine && !aborted; ++k) {
        const Item it = cta_item<T>(p, sched, k);
        if (it.tiles == 0) continue;
        // Q of the item's NH heads, swizzled K-major (rows past the group are
        // zero).  The score MMAs of the previous stage are complete once the
        // softmax warps have read their result.
        if (j >= 1 && !warp_wait(p_full0 + 8 * ((j - 1) & 1), ((j - 1) >> 1) & 1)) break;
        {
          constexpr int kPerLane = NH * (D / 8) / 32;  // 16-byte pieces per lane
          const int h0 = it.hc * NH;
          const char* qbase = static_cast<const char*>(p.q) +
                              (size_t(it.b) * p.h_q + size_t(it.kvh) * p.group + h0) * (D * 2);
          uint4 v[kPerLane];
#pragma unroll
          for (int u = 0; u < kPerLane; ++u) {  // all loads in flight at once
            const int ch = lane + 32 * u;
            const int h = ch / (D / 8), c = (ch % (D / 8)) * 8;
            const size_t bhq = size_t(it.b) * p.h_q + size_t(it.kvh) * p.group + h0 + h;
            v[u] = h0 + h < p.group && DA_IN(p, bhq, size_t(p.B) * p.h_q)
                       ? __ldg(reinterpret_cast<const uint4*>(qbase + h * (D * 2) + c * 2))
                       : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int u = 0; u < kPerLane; ++u) {
            const int ch = lane + 32 * u;
            const int h = ch / (D / 8), c = (ch % (D / 8)) * 8;
            *reinterpret_cast<uint4*>(qsw + tc5::sw128(h, c, NH)) = v[u];
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        for (int t = 0; t < it.tiles; ++t, ++j) {
          // S buffer j % 2 is free once the softmax warps have read stage j - 2
          if (j >= 2 && !warp_wait(p_full0 + 8 * (j & 1), ((j - 2) >> 1) & 1)) break;
          if (!warp_wait(kfull0 + 8 * kslot, kphase)) break;
          const int row0 = it.row_begin + t * T;
          const int new_local =
              (it.new_row >= row0 && it.new_row < row0 + T) ? it.new_row - row0 : -1;
          uint8_t* kt = kslots + size_t(kslot) * Cfg::kTileBytes;
          if (new_local >= 0) {
            const uint8_t* slot = knew + size_t(kslot) * Cfg::kRowBytes;
            for (int ch = lane; ch < D / 8; ch += 32)
              *reinterpret_cast<uint4*>(kt + tc5::sw128(new_local, ch * 8, T)) =
                  reinterpret_cast<const uint4*>(slot)[ch];
            if (it.hc == 0 &&  // and into the K cache
                DA_IN(p, (size_t(p.b_offset + it.b) * p.h_kv + it.kvh) * size_t(p.n_max) + it.new_row,
                      p.cache_rows)) {
              const size_t head = size_t(p.b_offset + it.b) * p.h_kv + it.kvh;
              uint4* dst = reinterpret_cast<uint4*>(
                  static_cast<char*>(p.k_cache) + (head * size_t(p.n_max) + size_t(it.new_row)) * (D * 2));
              for (int ch = lane; ch < D / 8; ch += 32) dst[ch] = reinterpret_cast<const uint4*>(slot)[ch];
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          if (lane == 0) {
            tc5::fence_after();
            const uint32_t ka = smem_u32(kt);
            const uint32_t sd = s_col0 + (j & 1) * NH;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint64_t a = tc5::sdesc(ka + (ks >> 2) * Cfg::kHalfBytes + (ks & 3) * 32, 16, 1024);
              const uint64_t bq =
                  tc5::sdesc(smem_u32(qsw) + (ks >> 2) * (NH * 128) + (ks & 3) * 32, 16, 1024);
              tc5::mma(sd, a, bq, idesc_s, ks > 0);
            }
            tc5::commit(s_full0 + 8 * (j & 1));
            tc5::commit(kempty0 + 8 * kslot);
          }
          __syncwarp();
          if (++kslot == KST) {
            kslot = 0;
            kphase ^= 1u;
          }
        }
      }
    } else {
      // ---- weighted sums: O^T += V_j^T . P_j^T (head | remainder)
      const uint32_t idesc_o = tc5::idesc_bf16(128, 2 * NH, 1, 0);
      int vslot = 0;
      uint32_t vphase = 0;
      for (int k = 0; k < sched.mine && !aborted; ++k) {
        const Item it = cta_item<T>(p, sched, k);
        for (int t = 0; t < it.tiles; ++t, ++j) {
          const uint32_t b = j & 1;
          if (!warp_wait(p_full0 + 8 * b, (j >> 1) & 1)) break;
          if (!warp_wait(vfull0 + 8 * vslot, vphase)) break;
          uint8_t* vt = vslots + size_t(vslot) * Cfg::kTileBytes;
          const int row0 = it.row_begin + t * T;
          const int valid = min(T, it.row_end - row0);
          if (valid < T) {  // rows past the end may hold anything, even NaN
            for (int ch = lane; ch < (T - valid) * (D / 8); ch += 32) {
              const int r = valid + ch / (D / 8), col = (ch % (D / 8)) * 8;
              *reinterpret_cast<uint4*>(vt + tc5::sw128(r, col, T)) = make_uint4(0, 0, 0, 0);
            }
          }
          const int new_local =
              (it.new_row >= row0 && it.new_row < row0 + T) ? it.new_row - row0 : -1;
          if (new_local >= 0) {
            const uint8_t* slot = vnew + size_t(vslot) * Cfg::kRowBytes;
            for (int ch = lane; ch < D / 8; ch += 32)
              *reinterpret_cast<uint4*>(vt + tc5::sw128(new_local, ch * 8, T)) =
                  reinterpret_cast<const uint4*>(slot)[ch];
            if (it.hc == 0 &&  // and into the V cache
                DA_IN(p, (size_t(p.b_offset + it.b) * p.h_kv + it.kvh) * size_t(p.n_max) + it.new_row,
                      p.cache_rows)) {
              const size_t head = size_t(p.b_offset + it.b) * p.h_kv + it.kvh;
              uint4* dst = reinterpret_cast<uint4*>(
                  static_cast<char*>(p.v_cache) + (head * size_t(p.n_max) + size_t(it.new_row)) * (D * 2));
              for (int ch = lane; ch < D / 8; ch += 32) dst[ch] = reinterpret_cast<const uint4*>(slot)[ch];
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tc5::fence_after();
            const uint32_t va = smem_u32(vt);
            const uint32_t pb = smem_u32(p_buf) + b * Cfg::kPBytes;
#pragma unroll
            for (int ks = 0; ks < T / 16; ++ks) {  // even / odd blocks: two independent chains
              const uint64_t a = tc5::sdesc(va + ks * 16 * 128, Cfg::kHalfBytes, 1024);
              const uint32_t off = (ks >> 2) * (2 * NH * 128) + (ks & 3) * 32;
              tc5::mma(o_col + (ks & 1) * (2 * NH), a, tc5::sdesc(pb + off, 16, 1024), idesc_o,
                       t > 0 || ks > 1);
            }
            tc5::commit(vempty0 + 8 * vslot);
            tc5::commit(pv_done0 + 8 * b);
          }
          __syncwarp();
          if (++vslot == VST) {
            vslot = 0;
            vphase ^= 1u;
          }
        }
      }
    }
    // every MMA either issuer started has completed before TMEM is freed
    if (lane == 0) {
      if (j > 0) tc5::commit(fin);
      else mbar_arrive(fin);
      volatile int never = 0;
      mbar_wait_bounded(fin, 0, &never);
    }
    __syncwarp();
    // and everyone else is done with TMEM
    named_bar_sync(2, 320);
    if (warp == 9) {
      tc5::fence_after();
      tc5::dealloc(tmem, kTmemCols);
    }
    return;
  }

  // ------------------------------------------------------------------ softmax warps
  // Warp w (0..7) owns stage rows 32*(w%4) .. +31 (its TMEM lane quarter) and
  // heads HT*(w/4) .. +HT-1 of the item; the two halves of the heads are two
  // groups of 128 threads with their own named barrier.
  constexpr int HT = NH / 2;
  const int grp = warp >> 2;
  const int quarter = warp & 3;
  const int hb = grp * HT;                       // first head of this thread
  const int t_row = quarter * 32 + lane;         // stage row for S, column d for O
  const uint32_t lane_base = uint32_t(quarter * 32) << 16;
  const int bar_id = 3 + grp;
  // [2 groups][2 buffers][4 quarters][HT] partials + 4 flags
  auto gred_of = [&](uint32_t parity) { return red + (grp * 2 + parity) * Cfg::kRedGroup; };
  // byte offsets of this thread's P^T elements: row r, column t_row (swizzled)
  const uint32_t p_off0 = uint32_t((t_row >> 6) * (2 * NH) * 128 + (t_row & 7) * 2);
  const int chunk = (t_row & 63) >> 3;
  uint32_t j = 0;  // stages processed (same count as the MMA warp)
  // Wait for the P.V of stage number jj (buffer jj % 2, its (jj / 2)-th use).
  auto wait_pv = [&](uint32_t jj) {
    if (!mbar_wait_bounded(pv_done0 + 8 * (jj & 1), (jj >> 1) & 1, abort_flag)) {
      if (!*abort_flag) {
        *abort_flag = 1;
        flag_error(p.dev_error, DA_DEVERR_TIMEOUT);
      }
    }
    tc5::fence_after();
  };
  for (int k = 0; k < sched.mine; ++k) {
    const Item it = cta_item<T>(p, sched, k);
    const int head0 = it.hc * NH;
    const size_t bh0 = size_t(it.b) * p.h_q + size_t(it.kvh) * p.group + head0;
    const int nheads = min(NH, p.group - head0);
    float m_run[HT], l_part[HT];
#pragma unroll
    for (int h = 0; h < HT; ++h) {
      m_run[h] = -INFINITY;
      l_part[h] = 0.f;
    }
    for (int t = 0; t < it.tiles; ++t, ++j) {
      if (!mbar_wait_bounded(s_full0 + 8 * (j & 1), (j >> 1) & 1, abort_flag)) {
        if (!*abort_flag) {
          *abort_flag = 1;
          flag_error(p.dev_error, DA_DEVERR_TIMEOUT);
        }
      }
      tc5::fence_after();
      // warp-uniform: the TMEM loads below are .sync.aligned
      const bool live = __all_sync(0xffffffffu, !*abort_flag);
      const int valid = min(T, it.row_end - (it.row_begin + t * T));
      const bool row_ok = t_row < valid;
      float s[HT];
      if (live) {
        tc5::ld16x(s_col0 + (j & 1) * NH + hb + lane_base, s, HT);
        tc5::wait_ld();
      }
#pragma unroll
      for (int h = 0; h < HT; ++h) s[h] = (live && row_ok) ? s[h] * p.scale_log2 : -INFINITY;

      // Running max: exact on an item's first stage, else only when some score
      // exceeds it by more than 2^8 (a vote; the exponentials stay <= 2^8).
      // Scratch buffer j % 2: a warp rewrites it two stages later, after the
      // barrier of the stage in between, when every reader is done with it.
      float* gred = gred_of(j & 1);
      bool exact = (t == 0);
      if (!exact) {
        bool over = false;
#pragma unroll
        for (int h = 0; h < HT; ++h) over |= s[h] > m_run[h] + kLazy;
        over = __any_sync(0xffffffffu, over);
        if (lane == 0) reinterpret_cast<int*>(gred + 4 * HT)[quarter] = over;
        named_bar_sync(bar_id, 128);
        const int* flags = reinterpret_cast<const int*>(gred + 4 * HT);
        exact = (flags[0] | flags[1] | flags[2] | flags[3]) != 0;
      }
      float alpha[HT];
#pragma unroll
      for (int h = 0; h < HT; ++h) alpha[h] = 1.f;
      if (exact) {  // uniform across the group
#pragma unroll
        for (int h = 0; h < HT; ++h) {
          float v = s[h];
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
          v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
          if (lane == 0) gred[quarter * HT + h] = v;
        }
        named_bar_sync(bar_id, 128);
#pragma unroll
        for (int h = 0; h < HT; ++h) {
          const float tm = fmaxf(fmaxf(gred[h], gred[HT + h]), fmaxf(gred[2 * HT + h], gred[3 * HT + h]));
          const float m_new = fmaxf(m_run[h], tm);
          alpha[h] = (m_run[h] == -INFINITY) ? 0.f : ex2(m_run[h] - m_new);
          m_run[h] = m_new;
        }
      }
#pragma unroll
      for (int h = 0; h < HT; ++h) {
        const float m_use = m_run[h] == -INFINITY ? 0.f : m_run[h];
        s[h] = ex2(s[h] - m_use);  // 0 for masked rows
        l_part[h] = l_part[h] * alpha[h] + s[h];
      }
      // P buffer j % 2 is free once the P.V of stage j - 2 has completed; O may
      // be rescaled once the P.V of stage j - 1 has.  (Each pv_done barrier
      // completes once per use of its buffer, so neither wait can be lapped.)
      if (j >= 2) wait_pv(j - 2);
      if (exact && t > 0) {
        wait_pv(j - 1);
        if (live) {  // rescale this thread's row of O^T (column d = t_row): 2 chains x 2 halves
#pragma unroll
          for (int part = 0; part < 4; ++part) {
            float o[HT];
            tc5::ld16x(o_col + part * NH + hb + lane_base, o, HT);
            tc5::wait_ld();
#pragma unroll
            for (int u = 0; u < HT; ++u) o[u] *= alpha[u];
            tc5::st16x(o_col + part * NH + hb + lane_base, o, HT);
          }
          tc5::wait_st();
        }
      }
      // P^T (heads x stage rows), K-major over the rows: bf16 head + remainder
      uint8_t* pb = p_buf + (j & 1) * Cfg::kPBytes;
#pragma unroll
      for (int h = 0; h < HT; ++h) {
        const int hh = hb + h;   // head row; its remainder row is NH + hh (same swizzle phase)
        const uint32_t off = p_off0 + uint32_t(hh * 128) + uint32_t((chunk ^ (hh & 7)) << 4);
        const __nv_bfloat16 hi = __float2bfloat16_rn(s[h]);
        const __nv_bfloat16 lo = __float2bfloat16_rn(s[h] - __bfloat162float(hi));
        *reinterpret_cast<__nv_bfloat16*>(pb + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(pb + off + NH * 128) = lo;
      }
      fence_proxy_async_smem();
      tc5::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full0 + 8 * (j & 1));
    }
    // ---- item epilogue
    // The softmax sums are final: reduce them while the last P.V completes.
    float* gred = gred_of(j & 1);
    // per-head sums over the 128 rows
#pragma unroll
    for (int h = 0; h < HT; ++h) {
      float v = l_part[h];
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      if (lane == 0) gred[quarter * HT + h] = v;
    }
    named_bar_sync(bar_id, 128);
    float L[HT], inv_l[HT];
#pragma unroll
    for (int h = 0; h < HT; ++h) {
      L[h] = gred[h] + gred[HT + h] + gred[2 * HT + h] + gred[3 * HT + h];
      inv_l[h] = L[h] > 0.f ? __fdividef(1.f, L[h]) : 0.f;
    }
    if (it.tiles > 0) wait_pv(j - 1);  // O is complete in TMEM
    float o[HT];
    const bool epi_live = __all_sync(0xffffffffu, !*abort_flag);  // warp-uniform, as above
    if (it.tiles > 0 && epi_live) {
      // O^T = (even chain head + remainder) + (odd chain head + remainder)
      float r1[HT];
      tc5::ld16x(o_col + hb + lane_base, o, HT);
      tc5::ld16x(o_col + NH + hb + lane_base, r1, HT);
      tc5::wait_ld();
#pragma unroll
      for (int h = 0; h < HT; ++h) o[h] += r1[h];
      float r2[HT];
      tc5::ld16x(o_col + 2 * NH + hb + lane_base, r1, HT);
      tc5::ld16x(o_col + 3 * NH + hb + lane_base, r2, HT);
      tc5::wait_ld();
#pragma unroll
      for (int h = 0; h < HT; ++h) o[h] += r1[h] + r2[h];
    } else {
#pragma unroll
      for (int h = 0; h < HT; ++h) o[h] = 0.f;
    }
    if (!*abort_flag) {
      // column d = t_row of every head of this thread's half: one 128-byte
      // row segment per warp and head
      const bool single = it.nv == 1;
      const size_t stride = single ? size_t(D) : size_t(p.max_splits) * D;
      const size_t base = single ? (bh0 + hb) * D + t_row
                                 : ((bh0 + hb) * p.max_splits + it.split) * D + t_row;
      const uint64_t keep = l2_policy_evict_last();  // partials: read back by the combine
#pragma unroll
      for (int h = 0; h < HT; ++h)
        if (hb + h < nheads) {
          if (single) store_out(p, base + h * stride, o[h] * inv_l[h]);
          else if (DA_IN(p, base + h * stride, p.part_rows * D))
            st_keep(p.o_part + base + h * stride, o[h] * inv_l[h], keep);
        }
      if ((!single || p.lse_out) && quarter == 0 && lane < HT && hb + lane < nheads) {
        float m_h = m_run[0], l_h = L[0];
#pragma unroll
        for (int h = 1; h < HT; ++h)
          if (lane == h) {
            m_h = m_run[h];
            l_h = L[h];
          }
        const float lse2 = l_h > 0.f ? m_h + log2f(l_h) : -INFINITY;
        if (!single) {
          if (DA_IN(p, (bh0 + hb + lane) * p.max_splits + it.split, p.part_rows))
            st_keep(p.lse_part + (bh0 + hb + lane) * p.max_splits + it.split, lse2,
                    l2_policy_evict_last());
        } else if (DA_IN(p, bh0 + hb + lane, size_t(p.B) * p.h_q)) {
          p.lse_out[bh0 + hb + lane] = lse2 * kLn2;
        }
      }
    }
    // the next item's first P.V overwrites O: our TMEM reads are complete
    tc5::fence_before();
    named_bar_sync(bar_id, 128);
  }
  named_bar_sync(2, 320);
}

// ---------------------------------------------------------------------------
// Variants and launcher.
// ---------------------------------------------------------------------------
using Tc5G16 = Tc5Cfg<16, 3, 3>;
using Tc5G32 = Tc5Cfg<32, 3, 2>;

KernelShape tc5_shape(int group) {
  if (group <= 16) return KernelShape{Tc5G16::kTile, 16, 64, 1, 0.7f};
  return KernelShape{Tc5G32::kTile, 32, 64, 1, 0.7f};
}

template <class Cfg>
static cudaError_t launch_tc5_cfg(const SplitParams& p, const CUtensorMap& tk,
                                  const CUtensorMap& tv, int grid, cudaStream_t stream) {
  static std::atomic<unsigned long long> smem_set{0};
  const cudaError_t e = set_smem_limit_once(split_decode_tc5_kernel<Cfg>, Cfg::kSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  return launch_dependent(split_decode_tc5_kernel<Cfg>, grid, Cfg::kThreads, Cfg::kSmemBytes, stream, tk, tv,
                          p);
}

cudaError_t launch_split_tc5(const SplitParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             int grid, cudaStream_t stream) {
  if (p.group <= 16) return launch_tc5_cfg<Tc5G16>(p, tk, tv, grid, stream);
  return launch_tc5_cfg<Tc5G32>(p, tk, tv, grid, stream);
}

}  // namespace da
