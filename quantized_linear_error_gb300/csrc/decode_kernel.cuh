// The fused decode kernel template (see decode.cu for the design), shared by
// the translation units that instantiate it for one token-tile count each
// (decode_mt1.cu, decode_mt2.cu, decode_mt4.cu), so that they compile in
// parallel.
#pragma once
#include <atomic>

#include "internal.h"

namespace spear {
namespace dec {


constexpr int kMaxStages = 8;
constexpr int kEcWarps = 4;  // compensator warps per CTA
constexpr int kBarrierBytes = 1024;
constexpr size_t kSmemCap = 200 * 1024;

struct DecodeParams {
  const uint8_t* wq;     // decode layout runs
  const uint32_t* sz;    // per-channel scale/zero words [nt16][16]
  const uint4* a_frag;
  const uint4* b_frag;
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  float* z;
  SyncWords* sync;
  int K, N, M, n_groups, rank, gate;
  float alpha;
  int nt16, P, KW, KC, NS, n_stages;
  uint32_t bytes_x, stage_bytes;  // x box bytes (KC * Mp * 2), bytes per stage buffer
  uint32_t b_late_off;            // nonzero: B fragments copied to the stage area at this offset after the W loop
  uint64_t wait_ns;
  int skip_arrive;
  const __nv_bfloat16* gw1;  // SPEAR_GATE_MLP: W1 [gh][rank]
  const __nv_bfloat16* gw2;  // SPEAR_GATE_MLP: W2 [rank][gh]
  int gh;
  // grouped handle: member i owns 16-row tiles [tile_start[i], tile_start[i + 1]),
  // its up-projection reads u columns [i rank_b, (i + 1) rank_b), scaled by alphas[i]
  int n_members, rank_b;
  int tile_start[kMaxGroup + 1];
  float alphas[kMaxGroup];
};

// Member of a grouped handle that owns 16-row tile `tile`.
SPEAR_DEVINL int member_of_tile(const DecodeParams& p, int tile) {
  int m = 0;
  while (m + 1 < p.n_members && tile >= p.tile_start[m + 1]) ++m;
  return m;
}

// Named barrier of the consumer warps. bar.sync counts whole warps, so each
// warp reconverges first (lane-0 branches precede both uses).
template <int NW>
SPEAR_DEVINL void consumer_bar() {
  __syncwarp();
  asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

// ldmatrix.x4 on a shared-space address.
SPEAR_DEVINL void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A B (no accumulator input: the first k16 step of a chain).
SPEAR_DEVINL void mma_bf16_16816_zero(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// Named barrier of the compensator warps (reconverged first: bar.sync counts warps).
SPEAR_DEVINL void ec_bar() {
  __syncwarp();
  asm volatile("bar.sync 2, %0;" ::"n"(kEcWarps * 32) : "memory");
}

// The x fragments of k16 step kk of a unit only (MT >= 2: fewer live registers).
template <int MT>
SPEAR_DEVINL void load_kk_x_frags(const uint32_t (&lane_base)[8], int kk, uint32_t (&b)[MT][2]) {
  constexpr int Mp = 8 * MT;
  const int c = (2 * kk) & 7;
  const uint32_t blk = (kk >> 2) * Mp * 128;
#pragma unroll
  for (int pr = 0; pr < MT / 2; ++pr)
    ldsm_x4(b[2 * pr][0], b[2 * pr][1], b[2 * pr + 1][0], b[2 * pr + 1][1], lane_base[c] + blk + pr * 16 * 128);
}

SPEAR_DEVINL uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// This CTA's share [u0, u1) of the projection units (one unit: 16 A rows x 128
// channels, 4 KB contiguous in fragment order).
SPEAR_DEVINL void ec_share(const DecodeParams& p, int& u0, int& u1) {
  // units <= 16 * (K / 128) and grid <= SM count keep the products in 32 bits
  const unsigned units = (unsigned)((p.rank / 16) * (p.K / 128));
  u0 = (int)(blockIdx.x * units / gridDim.x);
  u1 = (int)((blockIdx.x + 1) * units / gridDim.x);
}

SPEAR_DEVINL const uint4* ec_unit_ptr(const DecodeParams& p, int ua) {
  const int kb128 = p.K / 128;
  return p.a_frag + ((size_t)(ua / kb128) * (p.K / 16) + (ua % kb128) * 8) * 32;
}

// A does not depend on the previous kernel: pull this warp's units of it into
// L2 before waiting for x, one 128-byte line per lane and unit through the
// load path (a bulk prefetch would queue behind the weight copies of the
// copy engine and hold this warp back from its dependency wait).
SPEAR_DEVINL void ec_prefetch(const DecodeParams& p, int ew, int lane) {
  int u0, u1;
  ec_share(p, u0, u1);
  for (int ua = u0 + ew; ua < u1; ua += kEcWarps)
    prefetch_l2_line(reinterpret_cast<const uint8_t*>(ec_unit_ptr(p, ua)) + lane * 128);
}

// Bottleneck-MLP gate ("SPEAR", section 2.1A: gamma is a bottleneck MLP):
// u = alpha * sigmoid(W2 relu(W1 z)) (.) z per token, by the four compensator
// warps: z is staged transposed in shared memory (zs [M16][rank + 8], token
// rows M .. M16 - 1 zero, M16 = Mp rounded up to 16) next to W1 and W2
// (copied there, rows padded by 8, by three of the warps while the fourth
// waits for the grid), the two products run on warp MMAs (mlp_gate_logits),
// each of the four warps taking one 16-token block and a quarter (M16 = 16)
// or half (M16 = 32) of the rank columns (the hidden layer is computed by
// each); u is written split into bf16 hi + lo like the elementwise gates
// (zero for tokens M .. Mp - 1, and everywhere if z never arrived).
// One (16-token block, part of the rank columns) item of the MLP gate. Not
// inlined: its fragments would otherwise raise the register allocation of the
// whole kernel, consumer loop included.
template <int Mp>
__device__ __noinline__ void ec_u_mlp_item(const float* zs, int zst, int tb, int part, int parts, int r, int gh, int M,
                                           float alpha, bool arrived, const __nv_bfloat16* w1s,
                                           const __nv_bfloat16* w2s, int lane, __nv_bfloat16* uh,
                                           __nv_bfloat16* ul, int us) {
  const int nj8 = r / 8;
  mlp_gate_logits(zs, zst, 16 * tb, r, gh, w1s, r + 8, w2s, gh + 8, lane, part * nj8 / parts, (part + 1) * nj8 / parts,
                  [&](int m, int j, float g0, float g1) {
                    if (m >= Mp) return;
                    const bool live = arrived && m < M;
                    const float u0 = live ? alpha * zs[m * zst + j] * __fdividef(1.0f, 1.0f + __expf(-g0)) : 0.f;
                    const float u1 = live ? alpha * zs[m * zst + j + 1] * __fdividef(1.0f, 1.0f + __expf(-g1)) : 0.f;
                    __nv_bfloat16 h0, l0, h1, l1;
                    split_bf16(u0, h0, l0);
                    split_bf16(u1, h1, l1);
                    uh[m * us + j] = h0;
                    uh[m * us + j + 1] = h1;
                    ul[m * us + j] = l0;
                    ul[m * us + j + 1] = l1;
                  });
}

template <int Mp>
SPEAR_DEVINL void ec_u_mlp(const DecodeParams& p, const float* z, bool arrived, int ew, int lane, float* zs,
                           __nv_bfloat16* uh, __nv_bfloat16* ul, int us) {
  constexpr int M16 = Mp < 16 ? 16 : Mp;
  const int r = p.rank, M = p.M, zst = r + 8;
  // z [rank][32] -> zs [token][rank]: four tokens per float4, eight loads of a
  // thread in flight before any store (one L2 round trip for M16 <= 32, r <= 256)
  const int nv = r * (M16 / 4);
  for (int base = ew * 32 + lane; base < nv; base += 8 * kEcWarps * 32) {
    float4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int idx = base + k * kEcWarps * 32;
      const int j = idx / (M16 / 4), m0 = (idx % (M16 / 4)) * 4;
      v[k] = (arrived && idx < nv && m0 < M) ? __ldcg(reinterpret_cast<const float4*>(z + j * 32 + m0))
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int idx = base + k * kEcWarps * 32;
      if (idx < nv) {
        const int j = idx / (M16 / 4), m0 = (idx % (M16 / 4)) * 4;
        const float e[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) zs[(m0 + q) * zst + j] = m0 + q < M ? e[q] : 0.f;
      }
    }
  }
  ec_bar();
  constexpr int kParts = kEcWarps / (M16 / 16);  // one item per compensator warp
  for (int item = ew; item < (M16 / 16) * kParts; item += kEcWarps)
    ec_u_mlp_item<Mp>(zs, zst, item / kParts, item % kParts, kParts, r, p.gh, M, p.alpha, arrived,
                      reinterpret_cast<const __nv_bfloat16*>(zs + M16 * zst),
                      reinterpret_cast<const __nv_bfloat16*>(zs + M16 * zst) + p.gh * zst, lane, uh, ul, us);
}

// z += A[:, this CTA's share] x, via warp MMA with A rows as the M side.
template <int MT>
SPEAR_DEVINL void ec_project(const DecodeParams& p, float* z, int ew, int lane) {
  const int kb128 = p.K / 128;
  int u0, u1;
  ec_share(p, u0, u1);
  const int g = lane >> 2, tq = lane & 3;
  for (int ua = u0 + ew; ua < u1; ua += kEcWarps) {
    const int at = ua / kb128, kb = ua % kb128;
    const uint4* ag = ec_unit_ptr(p, ua) + lane;
    float c[2][MT][4] = {};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int k16 = kb * 8 + kk;
      const uint4 af = __ldg(ag + kk * 32);
      const uint32_t a[4] = {af.x, af.y, af.z, af.w};
#pragma unroll
      for (int n = 0; n < MT; ++n) {
        const int tok = 8 * n + g;
        // A's columns are in the quad order of the layout: lane tq takes
        // channels 4 tq .. 4 tq + 3 of the step, one 8-byte load
        uint2 bx = make_uint2(0u, 0u);
        if (tok < p.M) bx = __ldg(reinterpret_cast<const uint2*>(p.x + (size_t)tok * p.K + k16 * 16 + 4 * tq));
        const uint32_t b0 = bx.x, b1 = bx.y;
        mma_bf16_16816(c[kk & 1][n], a, b0, b1);
      }
    }
#pragma unroll
    for (int n = 0; n < MT; ++n) {
      red_add_v2(z + (16 * at + g) * 32 + 8 * n + 2 * tq, c[0][n][0] + c[1][n][0], c[0][n][1] + c[1][n][1]);
      red_add_v2(z + (16 * at + g + 8) * 32 + 8 * n + 2 * tq, c[0][n][2] + c[1][n][2], c[0][n][3] + c[1][n][3]);
    }
  }
}

template <int NW, int MT, int T, bool PC, bool EC>
__global__ void __launch_bounds__((NW + 1 + kEcWarps) * 32, 1)
    decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap xmap) {
  // Independent accumulator chains per tile (k16 step kk goes to chain
  // kk % NC). Grouped scales fold the chains into acc once per 128-channel
  // group; per-channel scales never fold until the end (there, 2 chains and
  // 1 at four token tiles measured 3-4% faster on the 70B MLP shapes than
  // 4 and 2).
  constexpr int NC = PC ? (MT == 4 ? 1 : 2) : (T == 1 && MT < 4 ? 2 : 1);
  constexpr int Mp = 8 * MT;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + 16;
  uint64_t* szbar = full + 32;
  uint64_t* ubar = full + 33;  // compensator warp -> consumers: u is in shared memory
  uint64_t* bbar = full + 34;  // B fragments of this CTA's tiles are in shared memory
  // stage buffers start on a 1024-byte boundary (the swizzle pattern of the x
  // box is defined on absolute shared-memory address bits)
  const uint32_t s0 = smem_u32(smem + kBarrierBytes);
  uint8_t* stages = smem + kBarrierBytes + (((s0 + 1023u) & ~1023u) - s0);
  uint32_t* szpc = reinterpret_cast<uint32_t*>(stages + (size_t)p.NS * p.stage_bytes);
  const int us = p.rank + 8;  // bf16 elements per token row of u
  __nv_bfloat16* uh = reinterpret_cast<__nv_bfloat16*>(szpc + (PC ? p.P * 16 : 0));
  __nv_bfloat16* ul = uh + Mp * us;
  float* zs_mlp = reinterpret_cast<float*>(ul + Mp * us);  // MLP gate: z^T [M16][rank + 8]
  constexpr int M16 = Mp < 16 ? 16 : Mp;
  // B fragments of this CTA's tiles [Pc][rank / 16][32] uint4 (16-byte aligned)
  // (or, with b_late_off, in the stage area behind the partial sums)
  const uint32_t bbuf_s =
      p.b_late_off ? smem_u32(stages) + p.b_late_off
                   : (smem_u32(zs_mlp + (p.gh > 0 ? M16 * (p.rank + 8) : 0)) +
                      (p.gh > 0 ? (uint32_t)(p.gh * (p.rank + 8) + p.rank * (p.gh + 8)) * 2u : 0u) + 15u) &
                         ~15u;

  const uint32_t stages_s = smem_u32(stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile0 = blockIdx.x * p.P;
  const int Pc = min(p.P, p.nt16 - tile0);
  const int K = p.K, KC = p.KC;
  const DecodeLayout L{K, p.nt16, p.P, PC};
  const size_t run_full = (size_t)Pc * L.stage_tile_bytes(kDecodeRun);

  // consumer warps with at least one tile: KW warps per row group of T tiles
  const int busy_warps = p.KW * ((Pc + T - 1) / T);
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], busy_warps);
    }
    mbar_init(szbar, 1);
    mbar_init(ubar, kEcWarps);
    mbar_init(bbar, 1);
    fence_mbar_init();
  }
  // Token rows M..Mp-1 of the staged x boxes are zero-filled by the copy
  // engine; in any case they only feed MMA output columns M..Mp-1, which are
  // never stored.
  __syncwarp();
  __syncthreads();
  // Let the next kernel in the stream launch now; it only touches its own
  // weights until its griddepcontrol.wait, which waits for this grid.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ------------------------------------------------------------ producer warp
  if (warp == NW) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      if (PC) {
        mbar_arrive_expect_tx(szbar, Pc * 64);
        bulk_g2s(szpc, p.sz + (size_t)tile0 * 16, Pc * 64, szbar);
      }
      // Weights and compensator factors are constant since create, x may be
      // produced by the previous kernel. The CTA that lands on the SM freed
      // last by the previous grid reaches the wait only after the issues made
      // before it, so before it go only the first stage's weights; right
      // after it, the first stage's x, then the other stages and the B
      // fragments. (Staging A here as well was measured to delay the wait.)
      const int prefetch = min(p.NS, p.n_stages);
      auto issue_weights = [&](int i) {
        const int slot = i % p.NS;
        const uint32_t run = (uint32_t)(Pc * L.stage_tile_bytes(min(KC, K - i * KC)));
        mbar_arrive_expect_tx(&full[slot], run + p.bytes_x);
        bulk_g2s_stream(stages + (size_t)slot * p.stage_bytes + p.bytes_x,
                        p.wq + L.run_offset(blockIdx.x, i * (KC / kDecodeRun)), run, &full[slot], pol);
      };
      auto issue_x = [&](int i) {
        const int slot = i % p.NS;
        tma_load_3d(stages + (size_t)slot * p.stage_bytes, &xmap, 0, 0, i * (KC / 64), &full[slot]);
      };
      prefetch_tensormap(&xmap);
      issue_weights(0);
      // CTAs start in block order as SMs free up, so high-numbered ones tend
      // to start last, when the previous grid ends; warm L2 with the first two
      // stages of the CTA half a grid away, whose own loads would otherwise
      // start only then. Measured worth it only with more than two stages:
      // on shorter calls the extra L2 traffic delays the compensator's
      // round trips more than it saves.
      if (p.n_stages > 2) {
        const int pb = (int)((blockIdx.x + gridDim.x / 2) % gridDim.x);
        for (int i = 0; i < 2; ++i)
          prefetch_l2(p.wq + L.run_offset(pb, i * (KC / kDecodeRun)),
                      (unsigned)(L.pc(pb) * L.stage_tile_bytes(min(KC, K - i * KC))));
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");
      issue_x(0);
      for (int i = 1; i < prefetch; ++i) {
        issue_weights(i);
        issue_x(i);
      }
      const unsigned bbytes = EC ? (unsigned)(Pc * (p.rank_b / 16) * 512) : 0u;
      const uint4* bsrc = p.b_frag + (size_t)tile0 * (p.rank_b / 16) * 32;
      if (EC) {
        // B fragments of this CTA's tiles (contiguous, constant since create)
        // into shared memory for the final up-projection (late: into L2 now)
        if (p.b_late_off) {
          prefetch_l2(bsrc, bbytes);
        } else {
          mbar_arrive_expect_tx(bbar, bbytes);
          bulk_g2s_shared_u32(bbuf_s, bsrc, bbytes, bbar);
        }
      }
      for (int i = prefetch; i < p.n_stages; ++i) {
        const int slot = i % p.NS;
        if (!mbar_wait_bounded(&empty[slot], ((i / p.NS) - 1) & 1, p.wait_ns)) {
          atomicOr(&p.sync->status, kStatusTimeoutPipe);
          break;
        }
        issue_weights(i);
        issue_x(i);
      }
      if (EC && p.b_late_off) {
        // the stage area is free once the last NS stages are released
        bool free = true;
        for (int i = max(0, p.n_stages - p.NS); free && i < p.n_stages; ++i)
          free = mbar_wait_bounded(&empty[i % p.NS], (i / p.NS) & 1, p.wait_ns);
        if (free) {
          mbar_arrive_expect_tx(bbar, bbytes);
          bulk_g2s_shared_u32(bbuf_s, bsrc, bbytes, bbar);
        } else {
          atomicOr(&p.sync->status, kStatusTimeoutPipe);
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------ compensator warps
  if (warp > NW) {
    if constexpr (EC) {
      const int ew = warp - NW - 1;
      volatile int* ec_flag = reinterpret_cast<volatile int*>(smem + 512);
      ec_prefetch(p, ew, lane);
      asm volatile("griddepcontrol.wait;" ::: "memory");
      // Calls alternate between two z buffers. `epoch` (calls completed so
      // far) is read by every CTA before its arrival and advanced by the last
      // CTA to arrive, after which no CTA of this call reads it; this call adds
      // into z[epoch % 2] and clears z[(epoch + 1) % 2] for the next call (the
      // previous call, which used that buffer, has completed). The arrival
      // counter is never reset: a call is complete at (epoch + 1) * grid.
      // (The epoch load is in flight during the projection's loads; only
      // the additions into z wait for it.)
      const unsigned ep = __ldcg(&p.sync->epoch);
      float* zc = p.z + (ep & 1u) * kZDecFloats;
      ec_project<MT>(p, zc, ew, lane);
      // Every lane's additions into z are visible device-wide before the
      // CTA's single arrival (release) on the grid-wide counter.
      __threadfence();
      ec_bar();
      if (ew == 0 && lane == 0) {
        const unsigned target = (ep + 1u) * gridDim.x;
        if (!p.skip_arrive) {
          const unsigned old = atomicAdd(&p.sync->arrive_acc, 1u);
          if (old == target - 1u) p.sync->epoch = ep + 1u;  // last to arrive: every CTA has read epoch
        }
        auto reached = [&]() { return (int)(ld_acquire_gpu(&p.sync->arrive_acc) - target) >= 0; };
        bool arrived = reached();
        if (!arrived) {
          const uint64_t t0 = globaltimer();
          while (!(arrived = reached())) {
            if (globaltimer() - t0 > p.wait_ns) break;
            __nanosleep(64);  // one poller per CTA, spaced out on the counter's L2 line
          }
        }
        if (!arrived) atomicOr(&p.sync->status, kStatusTimeoutZ);
        *ec_flag = arrived ? 1 : 0;
        __threadfence_block();
      } else if (ew > 0) {
        // While warp 0 waits for the grid, clear this CTA's slice of the
        // other buffer (after the arrival fence, which need not wait for
        // these stores; the next call reads it only after this grid ends).
        float4* zn = reinterpret_cast<float4*>(p.z + ((ep + 1u) & 1u) * kZDecFloats);
        const int n4 = p.rank * 8;  // float4 of [rank][32]
        const int c0 = (int)((long)blockIdx.x * n4 / gridDim.x), c1 = (int)((long)(blockIdx.x + 1) * n4 / gridDim.x);
        for (int i = c0 + (ew - 1) * 32 + lane; i < c1; i += (kEcWarps - 1) * 32) zn[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.gate == SPEAR_GATE_MLP) {
          // and the MLP gate's weights (constant since create) into shared
          // memory after z^T: W1 [gh][rank + 8], then W2 [rank][gh + 8].
          // (Copied before the grid-dependency wait, they delayed the
          // projection by ~1 us.)
          constexpr int M16 = Mp < 16 ? 16 : Mp;
          __nv_bfloat16* w1s = reinterpret_cast<__nv_bfloat16*>(zs_mlp + M16 * (p.rank + 8));
          const int tid = (ew - 1) * 32 + lane, nt = (kEcWarps - 1) * 32;
          stage_rows_padded(w1s, p.gw1, p.gh, p.rank, tid, nt);
          stage_rows_padded(w1s + p.gh * (p.rank + 8), p.gw2, p.rank, p.gh, tid, nt);
        }
      }
      ec_bar();
      const bool arrived = *ec_flag != 0;
      if (p.gate == SPEAR_GATE_MLP) {
        ec_u_mlp<Mp>(p, zc, arrived, ew, lane, zs_mlp, uh, ul, us);
      } else {
        // u = alpha * gamma(z) * z for 4 tokens per float4 of z ([rank][32] fp32).
        // Kept compact (fast exp and division for the sigmoid, ~1e-6
        // relative): this code runs once per launch, and a large unrolled
        // body here costs the consumer warps instruction fetch.
        // All loads of a round of four float4 per thread are issued before
        // any use, so that a round costs one L2 round trip.
        const int nv = p.rank * (Mp / 4);
        constexpr int kR = 4;
        for (int base = ew * 32 + lane; base < nv; base += kR * kEcWarps * 32) {
          float4 v[kR];
#pragma unroll
          for (int r = 0; r < kR; ++r) {
            const int idx = base + r * kEcWarps * 32;
            const int j = idx / (Mp / 4), m0 = (idx % (Mp / 4)) * 4;
            v[r] = (arrived && idx < nv) ? __ldcg(reinterpret_cast<const float4*>(zc + j * 32 + m0))
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int r = 0; r < kR; ++r) {
            const int idx = base + r * kEcWarps * 32;
            if (idx >= nv) break;
            const int j = idx / (Mp / 4), m0 = (idx % (Mp / 4)) * 4;
            const float zz[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float g = p.gate == SPEAR_GATE_ONE ? 1.0f : __fdividef(1.0f, 1.0f + __expf(-zz[e]));
              const float uval = (m0 + e < p.M) ? p.alphas[j / p.rank_b] * zz[e] * g : 0.f;
              __nv_bfloat16 hi, lo;
              split_bf16(uval, hi, lo);
              uh[(m0 + e) * us + j] = hi;
              ul[(m0 + e) * us + j] = lo;
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(ubar);  // release: this warp's share of u is visible to the consumers
    }
    return;
  }

  // ------------------------------------------------------------ consumer warps
  const int pw_i = warp / p.KW, kw_i = warp % p.KW;
  const int g = lane >> 2, tq = lane & 3;
  // The staged x box is laid out [k64 block][token][64] with the 128-byte
  // swizzle (16-byte chunk c of token row r sits at chunk c ^ (r & 7)).
  // x box addressing for ldmatrix: this lane supplies row (lane % 8) of matrix
  // lane / 8, i.e. token 8 * (lane / 16) + lane % 8 and k half (lane / 8) % 2
  const int mrow = lane & 7, mkh = (lane >> 3) & 1, mtok = 8 * (lane >> 4) + mrow;
  const uint32_t lane_off = mtok * 128;
  uint32_t swz[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) swz[c] = (uint32_t)((((c + mkh) & 7) ^ mrow) << 4);
  // M <= 8: one ldmatrix.x4 brings two k16 steps; lane l addresses token l % 8,
  // chunk c0 + l / 8 of the k64 block (c0 = 0 for steps 0-1, 4 for steps 2-3)
  const uint32_t lane_off1 = mrow * 128;
  const uint32_t swz1[2] = {(uint32_t)((((lane >> 3) & 7) ^ mrow) << 4),
                            (uint32_t)((((4 + (lane >> 3)) & 7) ^ mrow) << 4)};
  asm volatile("griddepcontrol.wait;" ::: "memory");

  float acc[T][MT][4];
  float accg[T][NC][MT][4];
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int n = 0; n < MT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[t][n][e] = 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) accg[t][c][n][e] = 0.f;
      }

  uint32_t zzpc[T][2];
  float spc[T][2];
  bool ok = true;
  if constexpr (PC) {
    ok = mbar_wait_bounded(szbar, 0, p.wait_ns);
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const int tl = pw_i * T + t;
      const uint32_t w0 = tl < Pc ? szpc[tl * 16 + g] : 0u, w1 = tl < Pc ? szpc[tl * 16 + g + 8] : 0u;
      zzpc[t][0] = frag_zero_lo(biased_zero_x2(w0 >> 16));
      zzpc[t][1] = frag_zero_hi(biased_zero_x2(w1 >> 16));
      spc[t][0] = bf16_bits_to_float(w0 & 0xFFFF);
      spc[t][1] = bf16_bits_to_float(w1 & 0xFFFF);
    }
  }

  // One 128-channel unit of this warp's tiles: wa[t] is this lane's first 16
  // bytes of tile t's codes (the unit's second k64 block is 512 bytes on), sa[t]
  // the scale/zero word of row g (row g + 8 is 32 bytes on), xa the lane's
  // ldmatrix row address of the unit's first k64 block of x, unswizzled.
  auto unit = [&](const uint32_t (&wa)[T], const uint32_t (&sa)[T], uint32_t xa) {
    uint4 wv[T][2];
    uint32_t zz[T][2];
    float sc[T][2];
#pragma unroll
    for (int t = 0; t < T; ++t) {
      {  // every CTA owns all P tiles (the layout is padded to whole CTAs)
        wv[t][0] = lds128(wa[t]);
        wv[t][1] = lds128(wa[t] + 512);
        if constexpr (!PC) {
          const uint32_t w0 = lds32(sa[t]);
          const uint32_t w1 = lds32(sa[t] + 32);
          zz[t][0] = frag_zero_lo(biased_zero_x2_of_word(w0));
          zz[t][1] = frag_zero_hi(biased_zero_x2_of_word(w1));
          sc[t][0] = bf16_bits_to_float(w0 & 0xFFFF);
          sc[t][1] = bf16_bits_to_float(w1 & 0xFFFF);
        } else {
          zz[t][0] = zzpc[t][0];
          zz[t][1] = zzpc[t][1];
        }
      }
    }
    uint32_t lane_base[8];
    // M <= 8: all eight k16 steps' x fragments at once (16 registers, four
    // ldmatrix.x4); wider M: per k16 step
    uint32_t bb[MT == 1 ? 8 : 1][MT][2];
    if constexpr (MT == 1) {
      const uint32_t a0 = xa + swz1[0], a1 = xa + swz1[1];
      ldsm_x4(bb[0][0][0], bb[0][0][1], bb[1][0][0], bb[1][0][1], a0);
      ldsm_x4(bb[2][0][0], bb[2][0][1], bb[3][0][0], bb[3][0][1], a1);
      ldsm_x4(bb[4][0][0], bb[4][0][1], bb[5][0][0], bb[5][0][1], a0 + Mp * 128);
      ldsm_x4(bb[6][0][0], bb[6][0][1], bb[7][0][0], bb[7][0][1], a1 + Mp * 128);
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) lane_base[c] = xa + swz[c];
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t bk[MT][2];
      if constexpr (MT > 1) load_kk_x_frags<MT>(lane_base, kk, bk);
      const uint32_t(&b)[MT][2] = MT == 1 ? bb[MT == 1 ? kk : 0] : bk;
#pragma unroll
      for (int t = 0; t < T; ++t) {
        {
          const uint32_t w = word_of(wv[t][kk >> 2], kk & 3);
          uint32_t a[4];
          decode_frag_unpack(w, zz[t][0], zz[t][1], a);
#pragma unroll
          for (int n = 0; n < MT; ++n) {
            // grouped scales restart the chains every group (folded below)
            if (!PC && kk < NC)
              mma_bf16_16816_zero(accg[t][kk % NC][n], a, b[n][0], b[n][1]);
            else
              mma_bf16_16816(accg[t][kk % NC][n], a, b[n][0], b[n][1]);
          }
        }
      }
    }
    if constexpr (!PC) {
      // grouped scales: fold the chains into acc once per group
#pragma unroll
      for (int t = 0; t < T; ++t)
#pragma unroll
        for (int n = 0; n < MT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v = accg[t][0][n][e];
#pragma unroll
            for (int c = 1; c < NC; ++c) v += accg[t][c][n][e];
            acc[t][n][e] = fmaf(sc[t][e >> 1], v * ((e >> 1) ? kFragScaleHi : kFragScaleLo), acc[t][n][e]);
          }
    }
  };

  // warps without a tile skip the stages (they are not counted on `empty`)
  const bool busy = pw_i * T < Pc;
  const uint32_t x_lane = MT == 1 ? lane_off1 : lane_off;
  // Full stages (KC channels) whose KC / 128 units split evenly over the K
  // warps: each warp takes the same NU <= 2 units of every stage (units
  // kw_i + j KW, j < NU), at offsets from the stage base fixed here.
  const int units_full = KC / 128;
  const int NU = units_full % p.KW == 0 && units_full / p.KW <= 2 ? units_full / p.KW : 0;
  const int n_fast = NU > 0 ? K / KC : 0;  // stages taken by the fixed-offset path
  uint32_t wo[2][T], so[2][T], xo[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int u = kw_i + j * p.KW;
    const int sr = u >> 1, uin = u & 1;
    const uint32_t run = p.bytes_x + (uint32_t)sr * (uint32_t)run_full;
#pragma unroll
    for (int t = 0; t < T; ++t) {
      const int tl = pw_i * T + t;
      wo[j][t] = run + (uint32_t)((tl * (kDecodeRun / 64) + 2 * uin) * 32 + lane) * 16;
      so[j][t] = run + (uint32_t)(Pc * (kDecodeRun / 64) * 512) +
                 (uint32_t)((tl * (kDecodeRun / 128) + uin) * 16 + g) * 4;
    }
    xo[j] = (uint32_t)(2 * u) * (Mp * 128) + x_lane;
  }
  for (int i = 0; i < p.n_stages && ok && busy; ++i) {
    const int slot = i % p.NS;
    if (!mbar_wait_bounded(&full[slot], (i / p.NS) & 1, p.wait_ns)) {
      ok = false;
      break;
    }
    const uint32_t st = stages_s + (uint32_t)slot * p.stage_bytes;
    if (i < n_fast) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (j < NU) {
          uint32_t wa[T], sa[T];
#pragma unroll
          for (int t = 0; t < T; ++t) {
            wa[t] = st + wo[j][t];
            sa[t] = st + so[j][t];
          }
          unit(wa, sa, st + xo[j]);
        }
      }
    } else {
      const int kcw = min(KC, K - i * KC);
      const int units = kcw / 128;
      // unit u of stage i is unit i * (KC / 128) + u of the whole K range; the
      // KW warps of a row group take those round-robin
      int u0 = kw_i - (i * units_full) % p.KW;
      if (u0 < 0) u0 += p.KW;
      for (int u = u0; u < units; u += p.KW) {
        // unit u is half uin of layout run sr inside this stage
        const int sr = u >> 1, uin = u & 1;
        const int kcw_r = min(kDecodeRun, kcw - sr * kDecodeRun);
        const uint32_t wsm = st + p.bytes_x + sr * (uint32_t)run_full;
        const uint32_t szs = wsm + (uint32_t)(Pc * (kcw_r / 64) * 512);
        uint32_t wa[T], sa[T];
#pragma unroll
        for (int t = 0; t < T; ++t) {
          const int tl = pw_i * T + t;
          wa[t] = wsm + ((tl * (kcw_r / 64) + 2 * uin) * 32 + lane) * 16;
          sa[t] = szs + ((tl * (kcw_r / 128) + uin) * 16 + g) * 4;
        }
        unit(wa, sa, st + (uint32_t)(2 * u) * (Mp * 128) + x_lane);
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
      for (int n = 0; n < MT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = accg[t][0][n][e];
#pragma unroll
          for (int c = 1; c < NC; ++c) v += accg[t][c][n][e];
          acc[t][n][e] = (v * ((e >> 1) ? kFragScaleHi : kFragScaleLo)) * spc[t][e >> 1];
        }
  }

  // ------------------------------------------------------------ reduction over K warps
  consumer_bar<NW>();  // every warp is done with the stages: reuse them
  float* red = reinterpret_cast<float*>(stages);
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

  // ------------------------------------------------------------ compensator term
  bool ec_ok = false;
  if constexpr (EC) ec_ok = mbar_wait_bounded(ubar, 0, 2 * p.wait_ns) && mbar_wait_bounded(bbar, 0, p.wait_ns);
  consumer_bar<NW>();  // partial sums of all K warps are in shared memory

  // ------------------------------------------------------------ finalize tiles
  // One (tile, 8-token column block) per warp and step, so that with several
  // token blocks (M > 8) all consumer warps share the reduction over the K
  // warps, the up-projection and the stores.
  const int mat = lane >> 3, mr = lane & 7;
  for (int it = warp; it < Pc * MT; it += NW) {
    const int tl = it / MT, n = it % MT;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kw = 0; kw < p.KW; ++kw) {
      const float* src = red + ((size_t)(tl * p.KW + kw) * 32 + lane) * 4 * MT + n * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) c[e] += src[e];
    }
    const int tile = tile0 + tl;
    if constexpr (EC) {
      if (ec_ok) {
        const int nj = p.rank_b / 16;
        const uint32_t bt = bbuf_s + (uint32_t)(((tl * nj) * 32 + lane) * 16);
        // this lane's ldmatrix row of u: token 8 n + lane % 8, k half lane / 8 % 2,
        // in the tile's member's columns of u
        const int uoff = (8 * n + mr) * us + 8 * (mat & 1) + member_of_tile(p, tile) * p.rank_b;
#pragma unroll 2
        for (int j = 0; j < nj; ++j) {
          const uint4 bf = lds128(bt + (uint32_t)j * 512);
          const uint32_t a[4] = {bf.x, bf.y, bf.z, bf.w};
          uint32_t h0, h1, l0, l1;  // u = hi + lo
          ldmatrix_x2(h0, h1, uh + uoff + j * 16);
          ldmatrix_x2(l0, l1, ul + uoff + j * 16);
          mma_bf16_16816(c, a, h0, h1);
          mma_bf16_16816(c, a, l0, l1);
        }
      }
    }
    const int row0 = tile * 16 + g, row1 = row0 + 8;
    const int m0 = 8 * n + 2 * tq, m1 = m0 + 1;
    if (row0 < p.N) {
      if (m0 < p.M) p.y[(size_t)m0 * p.N + row0] = __float2bfloat16_rn(c[0]);
      if (m1 < p.M) p.y[(size_t)m1 * p.N + row0] = __float2bfloat16_rn(c[1]);
    }
    if (row1 < p.N) {
      if (m0 < p.M) p.y[(size_t)m0 * p.N + row1] = __float2bfloat16_rn(c[2]);
      if (m1 < p.M) p.y[(size_t)m1 * p.N + row1] = __float2bfloat16_rn(c[3]);
    }
  }
}


// The kernel instantiation for (NW, MT, T, PC, EC) and the set-up it needs on a
// device (its shared-memory limit raised, once per device).
using DecodeKernelFn = void (*)(const DecodeParams, const CUtensorMap);
struct DecodeKernelRef {
  DecodeKernelFn fn = nullptr;
  cudaError_t (*configure)() = nullptr;
};

template <int NW, int MT, int T, bool PC, bool EC>
cudaError_t configure_t() {
  static std::atomic<uint64_t> configured{0};  // devices whose limit is raised
  return smem_limit_once(reinterpret_cast<const void*>(decode_kernel<NW, MT, T, PC, EC>), configured);
}

template <int NW, int MT, int T>
DecodeKernelRef kernel_t(bool pc, bool ec) {
  if (pc) return ec ? DecodeKernelRef{decode_kernel<NW, MT, T, true, true>, configure_t<NW, MT, T, true, true>}
                    : DecodeKernelRef{decode_kernel<NW, MT, T, true, false>, configure_t<NW, MT, T, true, false>};
  return ec ? DecodeKernelRef{decode_kernel<NW, MT, T, false, true>, configure_t<NW, MT, T, false, true>}
            : DecodeKernelRef{decode_kernel<NW, MT, T, false, false>, configure_t<NW, MT, T, false, false>};
}

// Instantiations per token-tile count MT (one translation unit each); an
// empty reference for a (NW, T) pair that is not instantiated.
DecodeKernelRef kernel_ref_mt1(int NW, int T, bool pc, bool ec);
DecodeKernelRef kernel_ref_mt2(int NW, int T, bool pc, bool ec);
DecodeKernelRef kernel_ref_mt4(int NW, int T, bool pc, bool ec);

}  // namespace dec
}  // namespace spear
