// Allocation-free decode entry point.
//
// Some callers cannot call cudaMalloc at all: a process whose device memory
// is entirely reserved up front by another allocator (every further
// cudaMalloc fails), or a latency-critical serving loop in which a device
// allocation, which may synchronise the device, is not allowed. Such callers
// cannot create a spear_linear_t (create allocates the kernel-side weight
// layouts and a workspace). spear_linear_forward_decode_noalloc serves them:
// it reads the weights straight from the caller's buffers in the documented
// user layout, and the only scratch it needs (the compensator's projection
// z = A x) lives in the file-scope array below, which every GPU that loads
// this library holds until the process exits.
//
// Two plain CUDA-core kernels on the caller's stream, ordered by the stream
// alone (no counter, no wait across blocks, nothing to clear between calls):
//  1. projection: one warp per row j of A writes z[j][0..M) (the whole dot
//     product over K, so every entry is written, never accumulated);
//  2. output: every CTA applies the gate u = alpha * gamma(z) * z into shared
//     memory, then one warp per output row n computes W x + B u with fp32
//     accumulation and one bf16 rounding. A lane reads 16 bytes of codes
//     (32 channels of one group) per step, the group's scale and zero once.
#include <mutex>

#include "internal.h"

namespace spear {
namespace {

constexpr int kNoallocMaxRank = 256;
constexpr int kNoallocMaxTokens = 32;
constexpr int kNoallocThreads = 256;
// z [rank][32] fp32
constexpr size_t kNoallocScratchBytes = (size_t)kNoallocMaxRank * kNoallocMaxTokens * 4;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct NoallocParams {
  const uint8_t* q;
  const uint16_t* s;
  const uint8_t* zp;
  const uint16_t* A;
  const uint16_t* B;
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  float* z;  // [rank][32]
  int K, N, G, n_groups, rank, M, gate;
  float alpha;
};

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Sum of 8 products of a bf16 octet (16 bytes) with another.
__device__ __forceinline__ float dot8(const uint4& a, const uint4& b) {
  float s = bf_lo(a.x) * bf_lo(b.x);
  s = fmaf(bf_hi(a.x), bf_hi(b.x), s);
  s = fmaf(bf_lo(a.y), bf_lo(b.y), s);
  s = fmaf(bf_hi(a.y), bf_hi(b.y), s);
  s = fmaf(bf_lo(a.z), bf_lo(b.z), s);
  s = fmaf(bf_hi(a.z), bf_hi(b.z), s);
  s = fmaf(bf_lo(a.w), bf_lo(b.w), s);
  return fmaf(bf_hi(a.w), bf_hi(b.w), s);
}

__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// z[j][m] = sum_k A[j][k] x[m][k]: warp w of CTA b takes row j = 8 b + w; lane
// l reads channels 8 l .. 8 l + 7 of every 256-channel step (16-byte loads).
__global__ void __launch_bounds__(kNoallocThreads) noalloc_project_kernel(const NoallocParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = blockIdx.x * (kNoallocThreads / 32) + warp;
  if (j >= p.rank) return;
  float acc[kNoallocMaxTokens];
#pragma unroll
  for (int m = 0; m < kNoallocMaxTokens; ++m) acc[m] = 0.f;
  const uint4* arow = reinterpret_cast<const uint4*>(p.A + (size_t)j * p.K);
  for (int k8 = lane; k8 < p.K / 8; k8 += 32) {
    const uint4 a = __ldg(arow + k8);
#pragma unroll
    for (int m = 0; m < kNoallocMaxTokens; ++m)
      if (m < p.M) acc[m] += dot8(a, __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)m * p.K) + k8));
  }
#pragma unroll
  for (int m = 0; m < kNoallocMaxTokens; ++m) {
    if (m >= p.M) break;
    const float v = warp_sum(acc[m]);
    if (lane == 0) p.z[j * kNoallocMaxTokens + m] = v;
  }
}

// y = W x + B u for one warp per output row n.
__global__ void __launch_bounds__(kNoallocThreads) noalloc_output_kernel(const NoallocParams p) {
  __shared__ float u[kNoallocMaxTokens * kNoallocMaxRank];  // u[m * rank + j]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < p.M * p.rank; i += kNoallocThreads) {
    const int m = i / p.rank, j = i % p.rank;
    const float zz = p.z[j * kNoallocMaxTokens + m];
    u[i] = p.alpha * (p.gate == SPEAR_GATE_ONE ? zz : zz * (1.0f / (1.0f + expf(-zz))));
  }
  __syncthreads();

  const int nwarps = kNoallocThreads / 32;
  for (int n = blockIdx.x * nwarps + warp; n < p.N; n += gridDim.x * nwarps) {
    float acc[kNoallocMaxTokens];
#pragma unroll
    for (int m = 0; m < kNoallocMaxTokens; ++m) acc[m] = 0.f;
    const uint4* qrow = reinterpret_cast<const uint4*>(p.q + (size_t)n * (p.K / 2));
    // lane l takes the 32 channels k0 = 32 (l + 32 i) .. k0 + 31, one group
    for (int c = lane; c < p.K / 32; c += 32) {
      const int k0 = 32 * c, g = k0 / p.G;
      const uint4 qv = __ldg(qrow + c);
      const float zero = p.zp ? (float)p.zp[(size_t)n * p.n_groups + g] : 8.f;
      const float sc = bf(p.s[(size_t)n * p.n_groups + g]);
      // (q - z) for the 32 channels, exact in fp32
      float w[32];
      const uint32_t words[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
      for (int b = 0; b < 4; ++b)
#pragma unroll
        for (int i = 0; i < 8; ++i) w[8 * b + i] = (float)((words[b] >> (4 * i)) & 0xFu) - zero;
#pragma unroll
      for (int m = 0; m < kNoallocMaxTokens; ++m) {
        if (m >= p.M) break;
        const uint4* xr = reinterpret_cast<const uint4*>(p.x + (size_t)m * p.K + k0);
        float part = 0.f;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint4 xv = __ldg(xr + b);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            part = fmaf(w[8 * b + 2 * i], bf_lo(xw[i]), part);
            part = fmaf(w[8 * b + 2 * i + 1], bf_hi(xw[i]), part);
          }
        }
        acc[m] = fmaf(sc, part, acc[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < kNoallocMaxTokens; ++m) {
      if (m >= p.M) break;
      const float v = warp_sum(acc[m]);
      float ec = 0.f;
      for (int j = lane; j < p.rank; j += 32) ec += bf(p.B[(size_t)n * p.rank + j]) * u[m * p.rank + j];
      ec = warp_sum(ec);
      if (lane == 0) p.y[(size_t)m * p.N + n] = __float2bfloat16_rn(v + ec);
    }
  }
}

// Device address of the scratch array, looked up once per device (with that
// device current) and cached.
void* scratch_address(spear_status_t* st) {
  static std::mutex mu;
  static void* addr[128] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    *st = SPEAR_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      *st = SPEAR_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = ptr;
  }
  *st = SPEAR_OK;
  return addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace spear

using namespace spear;

extern "C" spear_status_t spear_linear_forward_decode_noalloc(const spear_linear_desc_t* d, const void* x, void* y,
                                                              int32_t M, cudaStream_t stream) {
  if (!d || M < 0) return SPEAR_ERR_INVALID_ARG;
  if (M == 0) return SPEAR_OK;
  if (!x || !y || !d->qweight || !d->scales) return SPEAR_ERR_INVALID_ARG;
  if (d->K <= 0 || d->N <= 0 || d->K % 128 != 0 || d->N % 8 != 0) return SPEAR_ERR_INVALID_ARG;
  if (d->group_size != 0 && d->group_size != 128) return SPEAR_ERR_INVALID_ARG;
  if (d->rank < 0 || d->rank % 16 != 0 || (d->rank > 0 && (!d->A || !d->B))) return SPEAR_ERR_INVALID_ARG;
  if (d->gate == SPEAR_GATE_MLP) return SPEAR_ERR_UNSUPPORTED;
  if (d->gate != SPEAR_GATE_SIGMOID && d->gate != SPEAR_GATE_ONE) return SPEAR_ERR_INVALID_ARG;
  // 16-byte loads of codes, x and A
  if (!aligned16(x) || !aligned16(d->qweight) || (d->rank > 0 && !aligned16(d->A))) return SPEAR_ERR_INVALID_ARG;
  // beyond the scratch array's capacity
  if (M > kNoallocMaxTokens || d->rank > kNoallocMaxRank) return SPEAR_ERR_INVALID_ARG;

  spear_status_t st;
  unsigned char* scratch = static_cast<unsigned char*>(scratch_address(&st));
  if (st != SPEAR_OK) return st;

  NoallocParams p{};
  p.q = d->qweight;
  p.s = static_cast<const uint16_t*>(d->scales);
  p.zp = d->zeros;
  p.A = static_cast<const uint16_t*>(d->A);
  p.B = static_cast<const uint16_t*>(d->B);
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.z = reinterpret_cast<float*>(scratch);
  p.K = d->K;
  p.N = d->N;
  p.G = d->group_size == 0 ? d->K : d->group_size;
  p.n_groups = d->K / p.G;
  p.rank = d->rank;
  p.M = M;
  p.gate = d->gate;
  p.alpha = d->alpha;
  const int rows_per_cta = kNoallocThreads / 32;
  if (p.rank > 0) {
    noalloc_project_kernel<<<(p.rank + rows_per_cta - 1) / rows_per_cta, kNoallocThreads, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return SPEAR_ERR_CUDA;
  }
  noalloc_output_kernel<<<(d->N + rows_per_cta - 1) / rows_per_cta, kNoallocThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}
