// Round-to-nearest 4-bit quantiser: fp32 weights -> the user layout that
// spear_linear_create takes (packed codes, bf16 scales, integer zeros).
//
// RTN is the quantisation backend of the per-channel results in "SPEAR: A
// System for Post-Quantization Error-Adaptive Recovery", section 3.1; the
// paper does not spell it out, so this is the usual asymmetric min/max form.
// Per group of G input channels of one output row:
//   lo = min(0, min w), hi = max(0, max w), range = max(hi - lo, 1e-8)
//   s  = bf16_RNE(range / 15),  z = clamp(rint(-lo / s), 0, 15),
//   q  = clamp(rint(w / s) + z, 0, 15),
// every step in fp32 with IEEE division and round half to even, so the codes
// are defined bit for bit. One warp per (row, group), 16-byte loads.
#include "internal.h"

namespace spear {
namespace {

constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads) rtn_kernel(const float* __restrict__ w, int N, int K, int G,
                                                            uint8_t* __restrict__ q, uint16_t* __restrict__ s,
                                                            uint8_t* __restrict__ zp) {
  const int n_groups = K / G;
  const long gw = (long)blockIdx.x * (kQuantThreads / 32) + threadIdx.x / 32;
  if (gw >= (long)N * n_groups) return;
  const int lane = threadIdx.x & 31;
  const int row = (int)(gw / n_groups), g = (int)(gw % n_groups);
  const float* src = w + (size_t)row * K + (size_t)g * G;
  float lo = 0.f, hi = 0.f;
  for (int k = 4 * lane; k < G; k += 128) {
    const float4 v = *reinterpret_cast<const float4*>(src + k);
    lo = fminf(lo, fminf(fminf(v.x, v.y), fminf(v.z, v.w)));
    hi = fmaxf(hi, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  const float range = fmaxf(hi - lo, 1e-8f);
  const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(range, 15.0f));
  const float sf = __bfloat162float(sb);
  const float zf = fminf(fmaxf(rintf(__fdiv_rn(-lo, sf)), 0.f), 15.f);
  if (lane == 0) {
    s[(size_t)row * n_groups + g] = __bfloat16_as_ushort(sb);
    zp[(size_t)row * n_groups + g] = (uint8_t)zf;
  }
  uint8_t* dst = q + (size_t)row * (K / 2) + (size_t)g * (G / 2);
  for (int k = 4 * lane; k < G; k += 128) {
    const float4 v = *reinterpret_cast<const float4*>(src + k);
    const float vv[4] = {v.x, v.y, v.z, v.w};
    unsigned c[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) c[e] = (unsigned)fminf(fmaxf(rintf(__fdiv_rn(vv[e], sf)) + zf, 0.f), 15.f);
    // byte j holds channel 2j in its low nibble and 2j + 1 in its high nibble
    *reinterpret_cast<uint16_t*>(dst + k / 2) = (uint16_t)(c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12));
  }
}

}  // namespace
}  // namespace spear

using namespace spear;

extern "C" spear_status_t spear_quantize_rtn(const float* w, int32_t N, int32_t K, int32_t group_size,
                                             uint8_t* qweight, void* scales, uint8_t* zeros, cudaStream_t stream) {
  if (!w || !qweight || !scales || !zeros) return SPEAR_ERR_INVALID_ARG;
  if (N <= 0 || K <= 0 || K % 128 != 0 || (group_size != 0 && group_size != 128)) return SPEAR_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w) & 15u) || (reinterpret_cast<uintptr_t>(qweight) & 1u) ||
      (reinterpret_cast<uintptr_t>(scales) & 1u))
    return SPEAR_ERR_INVALID_ARG;
  const int G = group_size == 0 ? K : group_size;
  const long warps = (long)N * (K / G);
  const long blocks = (warps + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
  if (blocks > 0x7FFFFFFFL) return SPEAR_ERR_UNSUPPORTED;
  rtn_kernel<<<(unsigned)blocks, kQuantThreads, 0, stream>>>(w, N, K, G, qweight, static_cast<uint16_t*>(scales),
                                                             zeros);
  return cudaGetLastError() == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}
