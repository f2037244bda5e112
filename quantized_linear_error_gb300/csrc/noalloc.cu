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
// z = A x and a CTA arrival counter) lives in the file-scope array below,
// which every GPU that loads this library holds until the process exits.
//
// The kernel is a plain CUDA-core variant of the fused decode kernel: each
// CTA first computes whole rows of z (so no atomics are needed) and bumps an
// arrival counter, waits (bounded by %globaltimer) until every CTA has
// arrived, applies the gate u = alpha * gamma(z) * z in shared memory, then
// computes its output rows y = W x + B u with fp32 accumulation and one bf16
// rounding. It trades speed for having no set-up at all.
#include <mutex>

#include "internal.h"

namespace spear {
namespace {

constexpr int kNoallocMaxRank = 256;
constexpr int kNoallocMaxTokens = 32;
constexpr int kNoallocThreads = 256;
// Layout: [0, 256) counters (arrive, status); [256, 256 + 256 * 32 * 4) z [rank][32] fp32.
constexpr size_t kNoallocCounterBytes = 256;
constexpr size_t kNoallocScratchBytes = kNoallocCounterBytes + (size_t)kNoallocMaxRank * kNoallocMaxTokens * 4;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct NoallocParams {
  const uint8_t* q;
  const uint16_t* s;
  const uint8_t* zp;
  const uint16_t* A;
  const uint16_t* B;
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  unsigned* counters;  // [0] arrivals, [1] status
  float* z;            // [rank][32]
  int K, N, G, n_groups, rank, M, gate;
  float alpha;
  uint64_t wait_ns;
};

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x < kNoallocThreads / 32) t = red[threadIdx.x];
  if (warp == 0)
    for (int o = 4; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;  // valid in thread 0
}

__global__ void __launch_bounds__(kNoallocThreads) noalloc_decode_kernel(const NoallocParams p) {
  __shared__ float u[kNoallocMaxTokens * kNoallocMaxRank];  // u[m * rank + j]
  __shared__ float red[kNoallocThreads / 32];
  __shared__ int ok_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- compensator projection: CTA b owns rows j = b, b + grid, ... of z
  for (int j = blockIdx.x; j < p.rank; j += gridDim.x) {
    for (int m = 0; m < p.M; ++m) {
      float acc = 0.f;
      for (int k = threadIdx.x; k < p.K; k += kNoallocThreads)
        acc += bf(p.A[(size_t)j * p.K + k]) * __bfloat162float(p.x[(size_t)m * p.K + k]);
      acc = block_sum(acc, red);
      if (threadIdx.x == 0) p.z[j * 32 + m] = acc;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&p.counters[0], 1u);
  }

  // ---- wait for every CTA's rows of z, then gate
  if (threadIdx.x == 0) {
    int ok = 1;
    if (p.rank > 0) {
      const uint64_t t0 = globaltimer();
      while (ld_acquire_gpu(&p.counters[0]) < gridDim.x) {
        if (globaltimer() - t0 > p.wait_ns) {
          ok = 0;
          atomicOr(&p.counters[1], kStatusTimeoutZ);
          break;
        }
      }
    }
    ok_s = ok;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < p.M * p.rank; i += kNoallocThreads) {
    const int m = i / p.rank, j = i % p.rank;
    float v = 0.f;
    if (ok_s) {
      const float zz = __ldcg(p.z + j * 32 + m);
      v = p.alpha * (p.gate == SPEAR_GATE_ONE ? zz : zz * (1.0f / (1.0f + expf(-zz))));
    }
    u[i] = v;
  }
  __syncthreads();

  // ---- output rows: one warp per row, lanes stride over K
  const int nwarps = kNoallocThreads / 32;
  for (int n = blockIdx.x * nwarps + warp; n < p.N; n += gridDim.x * nwarps) {
    float acc[kNoallocMaxTokens];
#pragma unroll
    for (int m = 0; m < kNoallocMaxTokens; ++m) acc[m] = 0.f;
    for (int k = lane; k < p.K; k += 32) {
      const uint8_t byte = p.q[(size_t)n * (p.K / 2) + (k >> 1)];
      const int code = (k & 1) ? (byte >> 4) : (byte & 0xF);
      const int g = k / p.G;
      const int zero = p.zp ? p.zp[(size_t)n * p.n_groups + g] : 8;
      const float w = (float)(code - zero) * bf(p.s[(size_t)n * p.n_groups + g]);
#pragma unroll
      for (int m = 0; m < kNoallocMaxTokens; ++m)
        if (m < p.M) acc[m] += w * __bfloat162float(p.x[(size_t)m * p.K + k]);
    }
#pragma unroll
    for (int m = 0; m < kNoallocMaxTokens; ++m) {
      if (m >= p.M) break;
      float v = acc[m];
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      float ec = 0.f;
      for (int j = lane; j < p.rank; j += 32) ec += bf(p.B[(size_t)n * p.rank + j]) * u[m * p.rank + j];
      for (int o = 16; o > 0; o >>= 1) ec += __shfl_xor_sync(0xffffffffu, ec, o);
      if (lane == 0) p.y[(size_t)m * p.N + n] = __float2bfloat16_rn(v + ec);
    }
  }
}

// Device address of the scratch array, looked up once per device.
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
  // beyond the scratch array's capacity
  if (M > kNoallocMaxTokens || d->rank > kNoallocMaxRank) return SPEAR_ERR_INVALID_ARG;

  spear_status_t st;
  unsigned char* scratch = static_cast<unsigned char*>(scratch_address(&st));
  if (st != SPEAR_OK) return st;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SPEAR_ERR_CUDA;

  NoallocParams p{};
  p.q = d->qweight;
  p.s = static_cast<const uint16_t*>(d->scales);
  p.zp = d->zeros;
  p.A = static_cast<const uint16_t*>(d->A);
  p.B = static_cast<const uint16_t*>(d->B);
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.counters = reinterpret_cast<unsigned*>(scratch);
  p.z = reinterpret_cast<float*>(scratch + kNoallocCounterBytes);
  p.K = d->K;
  p.N = d->N;
  p.G = d->group_size == 0 ? d->K : d->group_size;
  p.n_groups = d->K / p.G;
  p.rank = d->rank;
  p.M = M;
  p.gate = d->gate;
  p.alpha = d->alpha;
  p.wait_ns = 100000000ull;
  // The array keeps the previous call's contents: start from zero counters.
  if (cudaMemsetAsync(scratch, 0, kNoallocCounterBytes, stream) != cudaSuccess) return SPEAR_ERR_CUDA;
  // One CTA per SM at most, so that all CTAs are resident for the z wait.
  const int rows_per_cta = kNoallocThreads / 32;
  int grid = (d->N + rows_per_cta - 1) / rows_per_cta;
  if (grid > sms) grid = sms;
  if (grid < 1) grid = 1;
  noalloc_decode_kernel<<<grid, kNoallocThreads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}
