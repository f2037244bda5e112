// Decode-phase kernel: the whole W4 + error-compensator linear for M <= 32
// tokens in one launch ("SPEAR: A System for Post-Quantization Error-Adaptive
// Recovery", section 2.2A: in the memory-bound decode phase the compensator is
// fused into the low-bit GEMM so the correction path is a single kernel).
//
// Design (one CTA per SM, persistent; 8 consumer warps + 1 producer warp):
//  * The CTA owns P consecutive 16-row tiles of W. A producer warp streams,
//    stage by stage along K, the tiles' packed codes, their scale/zero words
//    and the matching slice of x into shared memory with bulk async copies
//    (cp.async.bulk + mbarrier transaction counts).
//  * Consumer warps turn each 32-bit word into four bf16 A-fragment registers
//    with one LOP3 per pair (codes land in the mantissa of 128 + code) and one
//    bf16x2 subtraction of 128 + zero, which leaves the exact integer q - z.
//    Warp MMA (m16n8k16, fp32 accumulate) takes x as the 8-wide N operand
//    (tokens), and the group scale is applied once per group to the fp32
//    partial sum.
//  * The compensator's down-projection z = A x is split over all CTAs before
//    they start on W; partial sums are added into a workspace with vector
//    atomics and each CTA then bumps an arrival counter. After its W tiles a
//    CTA waits (bounded by %globaltimer) for all arrivals, applies the gate
//    u = alpha * gamma(z) * z, splits u into bf16 hi + lo and adds B u to its
//    fp32 accumulators with two more MMAs per step, then rounds y to bf16
//    once. The last CTA to read z clears it for the next call. HBM traffic is
//    W, scales/zeros, A and B once each.
#include "internal.h"

namespace spear {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;
constexpr int kBarrierBytes = 1024;

struct DecodeParams {
  const uint4* wq;
  const uint32_t* sz;
  const uint4* a_frag;
  const uint4* b_frag;
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  float* z;
  SyncWords* sync;
  int K, N, M, n_groups, rank, gate;
  float alpha;
  int nt16, P, KW, KC, NS, n_stages;
  uint32_t bytes_x, bytes_w, bytes_sz, stage_bytes;
  int xs_stride;  // bf16 elements per token row of a staged x slice
  uint64_t wait_ns;
  int skip_arrive;
};

SPEAR_DEVINL void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); }

// B fragments (k16 x n8, col) for MT token tiles from a token-major smem
// buffer: base[token * stride + k].
template <int MT>
SPEAR_DEVINL void load_token_frags(const __nv_bfloat16* base, int stride, int koff, int lane,
                                   uint32_t (&b)[MT][2]) {
  const int mat = lane >> 3, r = lane & 7;
  if constexpr (MT == 1) {
    ldmatrix_x2(b[0][0], b[0][1], base + r * stride + koff + 8 * (mat & 1));
  } else {
#pragma unroll
    for (int p = 0; p < MT / 2; ++p) {
      const int token = 8 * (2 * p + (mat >> 1)) + r;
      ldmatrix_x4(b[2 * p][0], b[2 * p][1], b[2 * p + 1][0], b[2 * p + 1][1],
                  base + token * stride + koff + 8 * (mat & 1));
    }
  }
}

SPEAR_DEVINL uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

SPEAR_DEVINL float gate_apply(float z, int gate) {
  return gate == SPEAR_GATE_ONE ? z : z * (1.0f / (1.0f + expf(-z)));
}

// z += A[:, this CTA's share] x, via warp MMA with A rows as the M side.
template <int MT>
SPEAR_DEVINL void ec_project(const DecodeParams& p, int warp, int lane) {
  const int kb128 = p.K / 128;
  const int units = (p.rank / 16) * kb128;
  const int u0 = (int)((long)blockIdx.x * units / gridDim.x);
  const int u1 = (int)((long)(blockIdx.x + 1) * units / gridDim.x);
  const int g = lane >> 2, tq = lane & 3;
  for (int ua = u0 + warp; ua < u1; ua += kConsumerWarps) {
    const int at = ua / kb128, kb = ua % kb128;
    float c[MT][4] = {};
#pragma unroll 2
    for (int kk = 0; kk < 8; ++kk) {
      const int k16 = kb * 8 + kk;
      const uint4 af = __ldg(p.a_frag + ((size_t)at * (p.K / 16) + k16) * 32 + lane);
      const uint32_t a[4] = {af.x, af.y, af.z, af.w};
#pragma unroll
      for (int n = 0; n < MT; ++n) {
        const int tok = 8 * n + g;
        uint32_t b0 = 0, b1 = 0;
        if (tok < p.M) {
          const uint32_t* xr = reinterpret_cast<const uint32_t*>(p.x + (size_t)tok * p.K + k16 * 16 + 2 * tq);
          b0 = __ldg(xr);
          b1 = __ldg(xr + 4);
        }
        mma_bf16_16816(c[n], a, b0, b1);
      }
    }
#pragma unroll
    for (int n = 0; n < MT; ++n) {
      red_add_v2(p.z + (16 * at + g) * 32 + 8 * n + 2 * tq, c[n][0], c[n][1]);
      red_add_v2(p.z + (16 * at + g + 8) * 32 + 8 * n + 2 * tq, c[n][2], c[n][3]);
    }
  }
}

template <int MT, int T, bool PC, bool EC>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + 16;
  uint64_t* szbar = full + 32;
  volatile int* flag = reinterpret_cast<volatile int*>(smem + 512);
  uint8_t* stages = smem + kBarrierBytes;
  uint32_t* szpc = reinterpret_cast<uint32_t*>(stages + (size_t)p.NS * p.stage_bytes);

  constexpr int Mp = 8 * MT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile0 = blockIdx.x * p.P;
  const int Pc = min(p.P, p.nt16 - tile0);
  const int K = p.K, KC = p.KC;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(szbar, 1);
    fence_mbar_init();
  }
  // Token rows M..Mp-1 of every staged x slice stay zero (never copied).
  for (int s = 0; s < p.NS; ++s) {
    __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(stages + (size_t)s * p.stage_bytes);
    for (int i = threadIdx.x; i < (Mp - p.M) * p.xs_stride; i += blockDim.x)
      xs[p.M * p.xs_stride + i] = __float2bfloat16_rn(0.f);
  }
  __syncthreads();

  // ------------------------------------------------------------ producer warp
  if (warp == kConsumerWarps) {
    const uint64_t pol = policy_evict_first();
    if (PC) {
      if (lane == 0) mbar_arrive_expect_tx(szbar, Pc * 64);
      __syncwarp();
      if (lane < Pc) bulk_g2s(szpc + lane * 16, p.sz + (size_t)(tile0 + lane) * 16, 64, szbar);
    }
    for (int i = 0; i < p.n_stages; ++i) {
      const int slot = i % p.NS;
      if (i >= p.NS && !mbar_wait_bounded(&empty[slot], ((i / p.NS) - 1) & 1, p.wait_ns)) {
        if (lane == 0) atomicOr(&p.sync->status, kStatusTimeoutPipe);
        return;
      }
      const int kc = i * KC;
      const int kcw = min(KC, K - kc);
      const int units = kcw / 128;
      const uint32_t bytes = (uint32_t)(p.M * kcw * 2 + Pc * (kcw / 64) * 512 + (PC ? 0 : Pc * units * 64));
      uint8_t* st = stages + (size_t)slot * p.stage_bytes;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], bytes);
      __syncwarp();
      const int ncopies = p.M + Pc * (PC ? 1 : 2);
      for (int c = lane; c < ncopies; c += 32) {
        if (c < p.M) {
          bulk_g2s(st + (size_t)c * p.xs_stride * 2, p.x + (size_t)c * K + kc, kcw * 2, &full[slot]);
        } else if (c < p.M + Pc) {
          const int t = c - p.M;
          bulk_g2s_stream(st + p.bytes_x + (size_t)t * (KC / 64) * 512,
                          p.wq + ((size_t)(tile0 + t) * (K / 64) + kc / 64) * 32, (kcw / 64) * 512, &full[slot],
                          pol);
        } else {
          const int t = c - p.M - Pc;
          bulk_g2s(st + p.bytes_x + p.bytes_w + (size_t)t * (KC / 128) * 64,
                   p.sz + ((size_t)(tile0 + t) * p.n_groups + kc / 128) * 16, units * 64, &full[slot]);
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumer warps
  const int pw_i = warp / p.KW, kw_i = warp % p.KW;
  const int g = lane >> 2, tq = lane & 3;

  if constexpr (EC) {
    ec_project<MT>(p, warp, lane);
    consumer_bar();
    if (threadIdx.x == 0 && !p.skip_arrive) {
      __threadfence();
      atomicAdd(&p.sync->arrive, 1u);
    }
  }

  float acc[T][MT][4];
  float accg[T][MT][4];
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int n = 0; n < MT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][n][e] = accg[t][n][e] = 0.f;

  uint32_t zzpc[T][2];
  float spc[T][2];
  bool ok = true;
  if constexpr (PC) {
    ok = mbar_wait_bounded(szbar, 0, p.wait_ns);
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const int tl = pw_i * T + t;
      const uint32_t w0 = tl < Pc ? szpc[tl * 16 + g] : 0u, w1 = tl < Pc ? szpc[tl * 16 + g + 8] : 0u;
      zzpc[t][0] = biased_zero_x2(w0 >> 16);
      zzpc[t][1] = biased_zero_x2(w1 >> 16);
      spc[t][0] = bf16_bits_to_float(w0 & 0xFFFF);
      spc[t][1] = bf16_bits_to_float(w1 & 0xFFFF);
    }
  }

  for (int i = 0; i < p.n_stages && ok; ++i) {
    const int slot = i % p.NS;
    if (!mbar_wait_bounded(&full[slot], (i / p.NS) & 1, p.wait_ns)) {
      ok = false;
      break;
    }
    const uint8_t* st = stages + (size_t)slot * p.stage_bytes;
    const __nv_bfloat16* xs = reinterpret_cast<const __nv_bfloat16*>(st);
    const uint4* wsm = reinterpret_cast<const uint4*>(st + p.bytes_x);
    const uint32_t* szs = reinterpret_cast<const uint32_t*>(st + p.bytes_x + p.bytes_w);
    const int units = min(KC, K - i * KC) / 128;
    for (int u = kw_i; u < units; u += p.KW) {
      uint4 wv[T][2];
      uint32_t zz[T][2];
      float sc[T][2];
#pragma unroll
      for (int t = 0; t < T; ++t) {
        const int tl = pw_i * T + t;
        if (tl < Pc) {
          wv[t][0] = wsm[(tl * (KC / 64) + 2 * u) * 32 + lane];
          wv[t][1] = wsm[(tl * (KC / 64) + 2 * u + 1) * 32 + lane];
          if constexpr (!PC) {
            const uint32_t w0 = szs[(tl * (KC / 128) + u) * 16 + g];
            const uint32_t w1 = szs[(tl * (KC / 128) + u) * 16 + g + 8];
            zz[t][0] = biased_zero_x2(w0 >> 16);
            zz[t][1] = biased_zero_x2(w1 >> 16);
            sc[t][0] = bf16_bits_to_float(w0 & 0xFFFF);
            sc[t][1] = bf16_bits_to_float(w1 & 0xFFFF);
          } else {
            zz[t][0] = zzpc[t][0];
            zz[t][1] = zzpc[t][1];
          }
        }
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b[MT][2];
        load_token_frags<MT>(xs, p.xs_stride, u * 128 + kk * 16, lane, b);
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const int tl = pw_i * T + t;
          if (tl < Pc) {
            const uint32_t w = word_of(wv[t][kk >> 2], kk & 3);
            const uint32_t a[4] = {bf16x2_sub(int4_pair_to_bf16x2_biased(w), zz[t][0]),
                                   bf16x2_sub(int4_pair_to_bf16x2_biased(w >> 4), zz[t][1]),
                                   bf16x2_sub(int4_pair_to_bf16x2_biased(w >> 8), zz[t][0]),
                                   bf16x2_sub(int4_pair_to_bf16x2_biased(w >> 12), zz[t][1])};
#pragma unroll
            for (int n = 0; n < MT; ++n) mma_bf16_16816(PC ? acc[t][n] : accg[t][n], a, b[n][0], b[n][1]);
          }
        }
      }
      if constexpr (!PC) {
#pragma unroll
        for (int t = 0; t < T; ++t)
#pragma unroll
          for (int n = 0; n < MT; ++n) {
            acc[t][n][0] = fmaf(sc[t][0], accg[t][n][0], acc[t][n][0]);
            acc[t][n][1] = fmaf(sc[t][0], accg[t][n][1], acc[t][n][1]);
            acc[t][n][2] = fmaf(sc[t][1], accg[t][n][2], acc[t][n][2]);
            acc[t][n][3] = fmaf(sc[t][1], accg[t][n][3], acc[t][n][3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) accg[t][n][e] = 0.f;
          }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  if (!ok && lane == 0) atomicOr(&p.sync->status, kStatusTimeoutPipe);

  if constexpr (PC) {
#pragma unroll
    for (int t = 0; t < T; ++t)
#pragma unroll
      for (int n = 0; n < MT; ++n) {
        acc[t][n][0] *= spc[t][0];
        acc[t][n][1] *= spc[t][0];
        acc[t][n][2] *= spc[t][1];
        acc[t][n][3] *= spc[t][1];
      }
  }

  // ------------------------------------------------------------ reduction over K warps
  consumer_bar();  // every warp is done with the stages: reuse them
  float* red = reinterpret_cast<float*>(stages);
  const size_t red_floats = (size_t)p.P * p.KW * 32 * 4 * MT;
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const int tl = pw_i * T + t;
    if (tl < Pc) {
      float* dst = red + ((size_t)(tl * p.KW + kw_i) * 32 + lane) * 4 * MT;
#pragma unroll
      for (int n = 0; n < MT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[n * 4 + e] = acc[t][n][e];
    }
  }

  // ------------------------------------------------------------ compensator gate
  const int us = p.rank + 8;  // bf16 elements per token row of u
  __nv_bfloat16* uh = reinterpret_cast<__nv_bfloat16*>(red + red_floats);
  __nv_bfloat16* ul = uh + Mp * us;
  bool ec_ok = false;
  if constexpr (EC) {
    if (threadIdx.x == 0) {
      bool arrived = ld_acquire_gpu(&p.sync->arrive) >= gridDim.x;
      if (!arrived) {
        const uint64_t t0 = globaltimer();
        while (!(arrived = ld_acquire_gpu(&p.sync->arrive) >= gridDim.x))
          if (globaltimer() - t0 > p.wait_ns) break;
      }
      if (!arrived) atomicOr(&p.sync->status, kStatusTimeoutZ);
      flag[0] = arrived ? 1 : 0;
    }
    consumer_bar();
    ec_ok = flag[0] != 0;
    for (int idx = threadIdx.x; idx < Mp * p.rank; idx += kConsumerWarps * 32) {
      const int m = idx / p.rank, j = idx % p.rank;
      float v = 0.f;
      if (ec_ok && m < p.M) v = p.alpha * gate_apply(__ldcg(p.z + j * 32 + m), p.gate);
      __nv_bfloat16 hi, lo;
      split_bf16(v, hi, lo);
      uh[m * us + j] = hi;
      ul[m * us + j] = lo;
    }
    consumer_bar();
    if (threadIdx.x == 0) {
      int last = 0;
      if (ec_ok) {
        __threadfence();
        last = atomicAdd(&p.sync->depart, 1u) == gridDim.x - 1;
        __threadfence();
      }
      flag[1] = last;
    }
    consumer_bar();
    if (flag[1]) {  // last reader: clear z and the counters for the next call
      for (int idx = threadIdx.x; idx < p.rank * 32; idx += kConsumerWarps * 32) p.z[idx] = 0.f;
      consumer_bar();
      if (threadIdx.x == 0) {
        p.sync->arrive = 0;
        p.sync->depart = 0;
        __threadfence();
      }
    }
  } else {
    consumer_bar();
  }

  // ------------------------------------------------------------ finalize tiles
  for (int tl = warp; tl < Pc; tl += kConsumerWarps) {
    float c[MT][4];
#pragma unroll
    for (int n = 0; n < MT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) c[n][e] = 0.f;
    for (int kw = 0; kw < p.KW; ++kw) {
      const float* src = red + ((size_t)(tl * p.KW + kw) * 32 + lane) * 4 * MT;
#pragma unroll
      for (int n = 0; n < MT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[n][e] += src[n * 4 + e];
    }
    const int tile = tile0 + tl;
    if constexpr (EC) {
      if (ec_ok) {
        for (int j16 = 0; j16 < p.rank / 16; ++j16) {
          const uint4 bf = __ldg(p.b_frag + ((size_t)tile * (p.rank / 16) + j16) * 32 + lane);
          const uint32_t a[4] = {bf.x, bf.y, bf.z, bf.w};
          uint32_t bh[MT][2], bl[MT][2];
          load_token_frags<MT>(uh, us, j16 * 16, lane, bh);
          load_token_frags<MT>(ul, us, j16 * 16, lane, bl);
#pragma unroll
          for (int n = 0; n < MT; ++n) {
            mma_bf16_16816(c[n], a, bh[n][0], bh[n][1]);
            mma_bf16_16816(c[n], a, bl[n][0], bl[n][1]);
          }
        }
      }
    }
    const int row0 = tile * 16 + g, row1 = row0 + 8;
#pragma unroll
    for (int n = 0; n < MT; ++n) {
      const int m0 = 8 * n + 2 * tq, m1 = m0 + 1;
      if (row0 < p.N) {
        if (m0 < p.M) p.y[(size_t)m0 * p.N + row0] = __float2bfloat16_rn(c[n][0]);
        if (m1 < p.M) p.y[(size_t)m1 * p.N + row0] = __float2bfloat16_rn(c[n][1]);
      }
      if (row1 < p.N) {
        if (m0 < p.M) p.y[(size_t)m0 * p.N + row1] = __float2bfloat16_rn(c[n][2]);
        if (m1 < p.M) p.y[(size_t)m1 * p.N + row1] = __float2bfloat16_rn(c[n][3]);
      }
    }
  }
}

template <int MT, int T, bool PC, bool EC>
cudaError_t launch_one(const DecodeParams& p, int grid, size_t smem, cudaStream_t st) {
  static bool configured = false;
  auto k = decode_kernel<MT, T, PC, EC>;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  k<<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

template <int MT, int T>
cudaError_t launch_mt_t(const DecodeParams& p, bool pc, bool ec, int grid, size_t smem, cudaStream_t st) {
  if (pc) return ec ? launch_one<MT, T, true, true>(p, grid, smem, st) : launch_one<MT, T, true, false>(p, grid, smem, st);
  return ec ? launch_one<MT, T, false, true>(p, grid, smem, st) : launch_one<MT, T, false, false>(p, grid, smem, st);
}

}  // namespace
}  // namespace spear

using namespace spear;

spear_status_t spear_launch_decode(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                   cudaStream_t stream) {
  DecodeParams p{};
  const int MT = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
  const int Mp = 8 * MT;
  const bool ec = h->rank > 0;
  const int P = (h->nt16 + h->sm_count - 1) / h->sm_count;
  const int grid = (h->nt16 + P - 1) / P;
  const int T = P > 4 ? 2 : 1;
  int pw = 1;
  while (pw < (P + T - 1) / T) pw *= 2;
  const int KW = kConsumerWarps / pw;
  int KC = 128 * KW < 256 ? 256 : 128 * KW;
  if (KC > h->K) KC = h->K;

  p.wq = h->wq_dec;
  p.sz = h->sz_dec;
  p.a_frag = h->a_dec;
  p.b_frag = h->b_dec;
  p.x = x;
  p.y = y;
  p.z = h->z_dec;
  p.sync = h->sync;
  p.K = h->K;
  p.N = h->N;
  p.M = M;
  p.n_groups = h->n_groups;
  p.rank = h->rank;
  p.gate = h->gate;
  p.alpha = h->alpha;
  p.nt16 = h->nt16;
  p.P = P;
  p.KW = KW;
  p.KC = KC;
  p.xs_stride = KC + 8;
  p.bytes_x = (uint32_t)(((size_t)Mp * p.xs_stride * 2 + 127) / 128 * 128);
  p.bytes_w = (uint32_t)((size_t)P * (KC / 64) * 512);
  p.bytes_sz = h->per_channel ? 0u : (uint32_t)((size_t)P * (KC / 128) * 64);
  p.stage_bytes = (p.bytes_x + p.bytes_w + p.bytes_sz + 127) / 128 * 128;
  p.n_stages = (h->K + KC - 1) / KC;
  p.wait_ns = h->wait_ns;
  p.skip_arrive = h->skip_arrive;

  const size_t red_bytes = (size_t)P * KW * 32 * 4 * MT * 4;
  const size_t u_bytes = ec ? (size_t)2 * Mp * (h->rank + 8) * 2 : 0;
  const size_t pc_bytes = h->per_channel ? (size_t)P * 64 : 0;
  const size_t budget = 227 * 1024 - kBarrierBytes - pc_bytes;
  int NS = (int)(budget / p.stage_bytes);
  if (NS > kMaxStages) NS = kMaxStages;
  if (NS > p.n_stages) NS = p.n_stages > 1 ? p.n_stages : 1;
  while ((size_t)NS * p.stage_bytes < red_bytes + u_bytes && (size_t)(NS + 1) * p.stage_bytes <= budget) ++NS;
  if (NS < 1 || (size_t)NS * p.stage_bytes < red_bytes + u_bytes) return SPEAR_ERR_UNSUPPORTED;
  p.NS = NS;
  const size_t smem = kBarrierBytes + (size_t)NS * p.stage_bytes + pc_bytes;

  cudaError_t e;
  if (MT == 1)
    e = T == 1 ? launch_mt_t<1, 1>(p, h->per_channel, ec, grid, smem, stream)
               : launch_mt_t<1, 2>(p, h->per_channel, ec, grid, smem, stream);
  else if (MT == 2)
    e = T == 1 ? launch_mt_t<2, 1>(p, h->per_channel, ec, grid, smem, stream)
               : launch_mt_t<2, 2>(p, h->per_channel, ec, grid, smem, stream);
  else
    e = T == 1 ? launch_mt_t<4, 1>(p, h->per_channel, ec, grid, smem, stream)
               : launch_mt_t<4, 2>(p, h->per_channel, ec, grid, smem, stream);
  return e == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}
