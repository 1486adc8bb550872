// Row quantization into an 8-bit KV cache (sm_103a).
//
// The row format of the 8-bit caches (one float32 scale per cached row; the
// page "Attention over the KV cache in the decode step" names int8/fp8 caches
// but no format) with absmax scaling:
//   a = max_j |x[j]|,  s = a / Q  (float32 division; Q = 127 int8, 448 e4m3),
//   code[j] = round-to-nearest-even(x[j] / s) clamped to [-Q, Q]; all zero
//   when s = 0.
// One warp per row; lane i takes elements i, i + 32, ... so loads and stores
// are coalesced.  The divisions are the correctly rounded float32 ones.
#include "common.cuh"

namespace da {

template <int KIND, int X_BF16>
__global__ void __launch_bounds__(256)
    kv_quantize_kernel(const void* __restrict__ x, uint8_t* __restrict__ codes,
                       float* __restrict__ scales, long long rows, int d) {
  const long long row = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  constexpr float Q = KIND == 1 ? 127.f : 448.f;
  const int per = d / 32;  // d is a multiple of 32, at most 256
  float v[8];
  float a = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    v[u] = 0.f;
    if (u < per) {
      const long long idx = row * d + lane + 32 * u;
      v[u] = X_BF16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(x)[idx])
                    : static_cast<const float*>(x)[idx];
      a = fmaxf(a, fabsf(v[u]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const float s = __fdiv_rn(a, Q);
  if (lane == 0) scales[row] = s;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    if (u >= per) break;
    uint8_t c = 0;
    if (s != 0.f) {
      const float q = fminf(fmaxf(__fdiv_rn(v[u], s), -Q), Q);
      if (KIND == 1) {
        c = static_cast<uint8_t>(static_cast<int8_t>(__float2int_rn(q)));
      } else {
        uint16_t two;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(two) : "f"(0.f), "f"(q));
        c = static_cast<uint8_t>(two & 0xffu);
      }
    }
    codes[row * d + lane + 32 * u] = c;
  }
}

cudaError_t launch_kv_quantize(const void* x, int x_bf16, void* codes, float* scales,
                               long long rows, int d, int kind, cudaStream_t stream) {
  const int threads = 256;  // 8 rows per block
  const long long blocks = (rows + 7) / 8;
  uint8_t* c = static_cast<uint8_t*>(codes);
  if (kind == 1) {
    if (x_bf16) kv_quantize_kernel<1, 1><<<unsigned(blocks), threads, 0, stream>>>(x, c, scales, rows, d);
    else kv_quantize_kernel<1, 0><<<unsigned(blocks), threads, 0, stream>>>(x, c, scales, rows, d);
  } else {
    if (x_bf16) kv_quantize_kernel<2, 1><<<unsigned(blocks), threads, 0, stream>>>(x, c, scales, rows, d);
    else kv_quantize_kernel<2, 0><<<unsigned(blocks), threads, 0, stream>>>(x, c, scales, rows, d);
  }
  return cudaGetLastError();
}

}  // namespace da
