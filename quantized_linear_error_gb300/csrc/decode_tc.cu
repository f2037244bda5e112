// Decode-phase kernel on the tcgen05 tensor cores: the whole W4 + error-
// compensator linear for M <= 32 tokens in one launch ("SPEAR: A System for
// Post-Quantization Error-Adaptive Recovery", section 2.2A: in the
// memory-bound decode phase the compensator is fused into the low-bit GEMM,
// so the correction path is a single kernel).
//
// Design (persistent, one CTA per SM, 26 warps):
//  * Work: the weight matrix in 128-row tiles, K in units of 256 channels;
//    the (tile, unit) pairs are split into equal contiguous ranges, one per
//    CTA ("stream-K"), so every shape balances over the SMs. The
//    compensator's up-projection is one more unit per tile (its "tail":
//    A = the tile's rows of B, the MMA's N side = u = alpha gamma(z) z in
//    bf16, since W x + B u = [W | B] [x ; u]); tile t's tail runs on CTA
//    t mod grid after that CTA's weight units, so no CTA stalls on the
//    grid-wide z dependency in the middle of its stream.
//  * A producer warp streams each weight unit (16 KB of packed codes and its
//    scale/zero words, bulk copies; the first ones before the dependency on
//    the previous kernel) and the matching x box (3-D tensor map, 128-byte
//    swizzle, tokens past M zero-filled) into a ring of shared-memory slots.
//  * 16 dequantising warps (4 per tensor-memory lane quarter, each 64 channels
//    of a unit) turn one row's codes into bf16 (q - z) * s (the exported
//    dequantised value: one LOP3 per pair, a bf16x2 subtraction and product)
//    and store them into a 3-deep ring of A operands in tensor memory
//    (tcgen05.st; the store of one unit overlaps the conversion of the next).
//  * One thread issues tcgen05.mma (M = 128 weight rows, N = 16 or 32 tokens,
//    K = 16, A from tensor memory, B from shared memory) into a double-buffered
//    fp32 accumulator in tensor memory.
//  * 4 epilogue warps read each finished segment (lane = weight row); a tile
//    done by one segment (no compensator) is stored at once, otherwise every
//    segment stores its fp32 partial in its own slot and the last contributor
//    sums the slots in a fixed order (the result does not depend on which
//    CTA finishes first), rounds to bf16 once and stores y.
//  * 4 compensator warps compute the CTA's share of z = A x (warp MMA), add it
//    with vector atomics, make the CTA's single arrival on a grid-wide counter,
//    wait for every CTA (bounded by %globaltimer), and build u in the
//    swizzled K-major layout the tail units' MMAs read.
// HBM traffic: W, scales/zeros, A and B once each, x and y.
#include "internal.h"
#include "tcgen05.cuh"

namespace spear {
namespace {

constexpr int kDq = 16;                     // dequantising warps
constexpr int kEp = 4;                      // epilogue warps
constexpr int kWProd = kDq + kEp;           // 20: TMA producer, owns the TMEM allocation
constexpr int kWMma = kWProd + 1;           // 21: MMA issuer
constexpr int kWEc0 = kWMma + 1;            // 22..25: compensator
constexpr int kEc = 4;
constexpr int kThr = (kWEc0 + kEc) * 32;    // 832
constexpr int kStageK = 256;                // channels per unit
constexpr int kNA = 3;                      // A operands in tensor memory (128 columns each)
constexpr uint32_t kTmemD = kNA * 128;      // two accumulators of 32 columns after the A ring
constexpr int kMaxSlots = 8;
constexpr uint32_t kWBytes = 128 * kStageK / 2;  // packed codes of one unit
constexpr uint32_t kSzBytes = 1024;              // scale/zero words of one unit (<= 2 groups x 128 rows)

struct TcParams {
  const uint32_t* wq;            // [nt][K/64][128][8] packed codes
  const uint32_t* sz;            // [nt][n_groups][128] scale/zero words
  const uint4* a_frag;           // A in warp-MMA fragment order (projection)
  const __nv_bfloat16* b_rows;   // B, [nt * 128][rank] (zero rows past N)
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  float* y32;                    // [grid + 2 nt][128][32] fp32 partials
  unsigned* tile_cnt;            // [nt] contributors done, zero between calls
  float* z;                      // [256][32] fp32, zero between calls
  SyncWords* sync;
  const __nv_bfloat16* gw1;      // MLP gate W1 [gh][rank]
  const __nv_bfloat16* gw2;      // MLP gate W2 [rank][gh]
  int K, N, M, n_groups, G, rank, gate, gh;
  float alpha;
  int nt, spt, units;            // tiles, units per tile, weight units = nt * spt
  int NS;
  uint32_t slot_bytes, x_bytes, u_off, mlp_off;
  uint64_t wait_ns;
  int skip_arrive;
};

// CTA c's weight units [begin(c), begin(c + 1)) and the CTA that owns unit u.
struct Split {
  int units, grid;
  __device__ int begin(int c) const { return (int)((long)c * units / grid); }
  __device__ int owner(int u) const {
    int c = (int)(((long)u * grid) / units);
    while (c > 0 && begin(c) > u) --c;
    while (c + 1 < grid && begin(c + 1) <= u) ++c;
    return c;
  }
};

// The MMAs of one unit, fully unrolled: descriptors advance by compile-time
// offsets (start address >> 4 in the low bits; no carry: shared addresses are
// below 256 KB), so each MMA costs about one add next to the instruction
// itself. The issuing thread shares its scheduler with busy dequantising
// warps, so every instruction it saves shortens the unit.
template <int NT, int NK>
SPEAR_DEVINL void mma_unit(uint32_t d, uint32_t a0, uint64_t b0, uint32_t idesc, bool first) {
#pragma unroll
  for (int k = 0; k < NK; ++k)
    umma_ts_bf16(d, a0 + 8 * k, b0 + (uint64_t)(((k >> 2) * NT * 128 + 32 * (k & 3)) >> 4), idesc,
                 (first && k == 0) ? 0u : 1u);
}

SPEAR_DEVINL void epi_bar() {
  __syncwarp();
  asm volatile("bar.sync 1, 128;" ::: "memory");
}
SPEAR_DEVINL void ec_bar() {
  __syncwarp();
  asm volatile("bar.sync 2, %0;" ::"n"(kEc * 32) : "memory");
}

SPEAR_DEVINL uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

SPEAR_DEVINL float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
SPEAR_DEVINL float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// sum_k w[k] v[k] over 8 * n8 bf16 weights (16-byte rows) and fp32 values.
SPEAR_DEVINL float dot_bf16_f32(const uint4* w, const float4* v, int n8) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 4
  for (int k = 0; k < n8; ++k) {
    const uint4 wv = __ldg(w + k);
    const float4 v0 = v[2 * k], v1 = v[2 * k + 1];
    a0 = fmaf(bf_lo(wv.x), v0.x, a0);
    a1 = fmaf(bf_hi(wv.x), v0.y, a1);
    a2 = fmaf(bf_lo(wv.y), v0.z, a2);
    a3 = fmaf(bf_hi(wv.y), v0.w, a3);
    a0 = fmaf(bf_lo(wv.z), v1.x, a0);
    a1 = fmaf(bf_hi(wv.z), v1.y, a1);
    a2 = fmaf(bf_lo(wv.w), v1.z, a2);
    a3 = fmaf(bf_hi(wv.w), v1.w, a3);
  }
  return (a0 + a1) + (a2 + a3);
}

// u[m][j] as bf16 in the 128-byte-swizzled K-major layout of the tail MMAs'
// B operand: blocks of 64 channels, NT rows (tokens) of 128 bytes each.
template <int NT>
SPEAR_DEVINL void store_u(uint8_t* u_area, int m, int j, float v) {
  const int blk = j >> 6, c = j & 63;
  const uint32_t off = blk * NT * 128 + m * 128 + ((((c >> 3) ^ (m & 7)) & 7) << 4) + (c & 7) * 2;
  *reinterpret_cast<__nv_bfloat16*>(u_area + off) = __float2bfloat16_rn(v);
}

// The A down-projection's share of this CTA: pull it into L2 before the
// dependency on the previous kernel (A does not depend on it).
SPEAR_DEVINL void ec_prefetch(const TcParams& p, int ew, int lane) {
  const int kb128 = p.K / 128;
  const int units = (p.rank / 16) * kb128;
  const int u0 = (int)((long)blockIdx.x * units / gridDim.x);
  const int u1 = (int)((long)(blockIdx.x + 1) * units / gridDim.x);
  if (lane == 0)
    for (int ua = u0 + ew; ua < u1; ua += kEc) {
      const int at = ua / kb128, kb = ua % kb128;
      prefetch_l2(p.a_frag + ((size_t)at * (p.K / 16) + kb * 8) * 32, 8 * 32 * 16);
    }
}

// z += A[:, this CTA's share] x (warp MMA, A rows as the M side, MT token tiles of 8).
template <int MT>
SPEAR_DEVINL void ec_project(const TcParams& p, int ew, int lane) {
  const int kb128 = p.K / 128;
  const int units = (p.rank / 16) * kb128;
  const int u0 = (int)((long)blockIdx.x * units / gridDim.x);
  const int u1 = (int)((long)(blockIdx.x + 1) * units / gridDim.x);
  const int g = lane >> 2, tq = lane & 3;
  for (int ua = u0 + ew; ua < u1; ua += kEc) {
    const int at = ua / kb128, kb = ua % kb128;
    float c[2][MT][4] = {};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int k16 = kb * 8 + kk;
      const uint4 af = __ldg(p.a_frag + ((size_t)at * (p.K / 16) + k16) * 32 + lane);
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
      red_add_v2(p.z + (16 * at + g) * 32 + 8 * n + 2 * tq, c[0][n][0] + c[1][n][0], c[0][n][1] + c[1][n][1]);
      red_add_v2(p.z + (16 * at + g + 8) * 32 + 8 * n + 2 * tq, c[0][n][2] + c[1][n][2], c[0][n][3] + c[1][n][3]);
    }
  }
}

// u = alpha gamma(z) (.) z for tokens < M into the tail operand (zero for the
// other NT rows, and everywhere if z never arrived).
template <int NT>
SPEAR_DEVINL void ec_build_u(const TcParams& p, bool arrived, int tid, uint8_t* u_area, float* zs, float* ts) {
  constexpr int kT = kEc * 32;
  const int r = p.rank, M = p.M;
  if (p.gate == SPEAR_GATE_MLP) {
    // bottleneck MLP ("SPEAR", section 2.1A): gamma(z) = sigmoid(W2 relu(W1 z)), per token
    const int hh = p.gh;
    for (int i = tid; i < M * r; i += kT) {
      const int m = i / r, j = i - m * r;
      zs[i] = arrived ? __ldcg(p.z + j * 32 + m) : 0.f;
    }
    ec_bar();
    for (int i = tid; i < M * hh; i += kT) {
      const int m = i / hh, c = i - m * hh;
      ts[i] = fmaxf(dot_bf16_f32(reinterpret_cast<const uint4*>(p.gw1 + (size_t)c * r),
                                 reinterpret_cast<const float4*>(zs + m * r), r / 8), 0.f);
    }
    ec_bar();
    for (int i = tid; i < NT * r; i += kT) {
      const int m = i / r, j = i - m * r;
      float uv = 0.f;
      if (arrived && m < M) {
        const float g = dot_bf16_f32(reinterpret_cast<const uint4*>(p.gw2 + (size_t)j * hh),
                                     reinterpret_cast<const float4*>(ts + m * hh), hh / 8);
        uv = p.alpha * zs[m * r + j] * __fdividef(1.0f, 1.0f + __expf(-g));
      }
      store_u<NT>(u_area, m, j, uv);
    }
  } else {
    for (int i = tid; i < NT * r; i += kT) {
      const int j = i / NT, m = i - j * NT;
      float uv = 0.f;
      if (arrived && m < M) {
        const float zz = __ldcg(p.z + j * 32 + m);
        uv = p.alpha * zz * (p.gate == SPEAR_GATE_ONE ? 1.0f : __fdividef(1.0f, 1.0f + __expf(-zz)));
      }
      store_u<NT>(u_area, m, j, uv);
    }
  }
}

template <int NT, bool EC>
__global__ void __launch_bounds__(kThr, 1) decode_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap xmap) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxSlots;
  uint64_t* a_full = empty + kMaxSlots;
  uint64_t* a_empty = a_full + kNA;
  uint64_t* d_full = a_empty + kNA;
  uint64_t* d_empty = d_full + 2;
  uint64_t* u_ready = d_empty + 2;
  uint64_t* mma_done = u_ready + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 512);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + 576);
  volatile int* ec_flag = reinterpret_cast<volatile int*>(smem + 640);
  uint8_t* slots = smem + 1024;
  const uint32_t slots_s = smem_u32(slots);
  uint8_t* u_area = smem + p.u_off;
  float* mlp = reinterpret_cast<float*>(smem + p.mlp_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Split sp{p.units, (int)gridDim.x};
  const int ub = sp.begin(blockIdx.x), ue = sp.begin(blockIdx.x + 1);
  const int nW = ue - ub;
  const int nT = (EC && (int)blockIdx.x < p.nt) ? (p.nt - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int spt = p.spt, kb_tile = p.K / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDq + 1);  // 16 dequant warps read W, the MMA reads x
    }
    for (int s = 0; s < kNA; ++s) {
      mbar_init(&a_full[s], kDq);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&d_full[s], 1);
      mbar_init(&d_empty[s], kEp);
    }
    mbar_init(u_ready, kEc);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == kWProd) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp < kDq) {
    // ------------------------------------------------------------ dequantisers
    const int q = warp & 3, j = warp >> 2;
    const int r = 32 * q + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    int ga = 0, pending = -1;
    bool ok = true;
    for (int i = 0; i < nW + nT && ok; ++i, ++ga) {
      uint32_t v[32];
      bool live;
      if (i < nW) {
        const int u = ub + i, s = i % p.NS;
        if (!mbar_wait_bounded(&full[s], (i / p.NS) & 1, p.wait_ns)) {
          ok = false;
          break;
        }
        const int st = u % spt;
        live = st * 4 + j < kb_tile;
        if (live) {
          const uint32_t sl = slots_s + (uint32_t)s * p.slot_bytes;
          const uint4 w0 = lds128(sl + (uint32_t)((j * 128 + r) * 32));
          const uint4 w1 = lds128(sl + (uint32_t)((j * 128 + r) * 32 + 16));
          const uint32_t szw = lds32(sl + kWBytes + (uint32_t)(((p.G == 128 ? (j >> 1) : 0) * 128 + r) * 4));
          const uint32_t zz = biased_zero_x2_of_word(szw);
          const uint32_t sc = (szw & 0xFFFFu) | (szw << 16);
          const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int c = 0; c < 8; ++c)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              v[4 * c + jj] = bf16x2_mul(bf16x2_sub(int4_pair_to_bf16x2_biased(words[c] >> (4 * jj)), zz), sc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // this warp's reads of the slot are done
      } else {
        // compensator tail of tile t: row t * 128 + r of B, channels 64 j .. + 63
        const int t = (int)blockIdx.x + (i - nW) * (int)gridDim.x;
        live = 64 * j < p.rank;
        if (live) {
          const uint4* src = reinterpret_cast<const uint4*>(p.b_rows + (size_t)(t * 128 + r) * p.rank + 64 * j);
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const uint4 w = 64 * j + 8 * c8 < p.rank ? __ldg(src + c8) : make_uint4(0u, 0u, 0u, 0u);
            v[4 * c8] = w.x;
            v[4 * c8 + 1] = w.y;
            v[4 * c8 + 2] = w.z;
            v[4 * c8 + 3] = w.w;
          }
        }
      }
      if (pending >= 0) {
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[pending % kNA]);
        pending = -1;
      }
      const int ab = ga % kNA;
      if (ga >= kNA && !mbar_wait_bounded(&a_empty[ab], ((ga / kNA) - 1) & 1, p.wait_ns)) {
        ok = false;
        break;
      }
      if (live) tmem_st_x32(lane_base + ab * 128 + 32 * j, v);
      pending = ga;
    }
    if (pending >= 0) {
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[pending % kNA]);
    }
    if (!ok && lane == 0) atomicOr(&p.sync->status, kStatusTimeoutPipe);
  } else if (warp == kWProd) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      auto issue_w = [&](int i) {
        const int u = ub + i, s = i % p.NS;
        const int tile = u / spt, st = u % spt;
        const int kb0 = st * 4, nkb = min(4, kb_tile - kb0);
        const int g0 = p.G == 128 ? kb0 / 2 : 0, ng = p.G == 128 ? (nkb + 1) / 2 : 1;
        uint8_t* sl = slots + (size_t)s * p.slot_bytes;
        mbar_arrive_expect_tx(&full[s], (uint32_t)nkb * 4096u + (uint32_t)ng * 512u + p.x_bytes);
        bulk_g2s_stream(sl, p.wq + ((size_t)tile * kb_tile + kb0) * 1024, (uint32_t)nkb * 4096u, &full[s], pol);
        bulk_g2s(sl + kWBytes, p.sz + ((size_t)tile * p.n_groups + g0) * 128, (uint32_t)ng * 512u, &full[s]);
      };
      auto issue_x = [&](int i) {
        const int u = ub + i, s = i % p.NS;
        tma_load_3d(slots + (size_t)s * p.slot_bytes + kWBytes + kSzBytes, &xmap, 0, 0, (u % spt) * 4, &full[s]);
      };
      const int pre = min(p.NS, nW);
      for (int i = 0; i < pre; ++i) issue_w(i);  // weights do not depend on the previous kernel
      asm volatile("griddepcontrol.wait;" ::: "memory");
      for (int i = 0; i < pre; ++i) issue_x(i);
      int issued = pre;
      for (int i = pre; i < nW; ++i) {
        const int s = i % p.NS;
        if (!mbar_wait_bounded(&empty[s], ((i / p.NS) - 1) & 1, p.wait_ns)) {
          atomicOr(&p.sync->status, kStatusTimeoutPipe);
          break;
        }
        issue_w(i);
        issue_x(i);
        issued = i + 1;
      }
      // no copy into this CTA's shared memory may still be in flight at exit
      for (int i = issued > p.NS ? issued - p.NS : 0; i < issued; ++i)
        mbar_wait_bounded(&full[i % p.NS], (i / p.NS) & 1, p.wait_ns);
    }
  } else if (warp == kWMma) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, NT);
      int seg = 0, ga = 0;
      bool ok = true;
      for (int i = 0; i < nW && ok; ++seg) {
        const int tile = (ub + i) / spt;
        const int seg_end = min(nW, (tile + 1) * spt - ub);
        const int db = seg & 1;
        if (seg >= 2 && !(ok = mbar_wait_bounded(&d_empty[db], ((seg / 2) - 1) & 1, p.wait_ns))) break;
        for (bool first = true; i < seg_end; ++i, ++ga, first = false) {
          const int ab = ga % kNA, s = i % p.NS;
          if (!(ok = mbar_wait_bounded(&a_full[ab], (ga / kNA) & 1, p.wait_ns))) break;
          if (!(ok = mbar_wait_bounded(&full[s], (i / p.NS) & 1, p.wait_ns))) break;
          tc_fence_after_sync();
          const bool full_unit = p.K - ((ub + i) % spt) * kStageK >= kStageK;  // else 128 channels
          const uint64_t bd = sw128_kmajor_desc(slots_s + (uint32_t)s * p.slot_bytes + kWBytes + kSzBytes);
          if (full_unit)
            mma_unit<NT, 16>(tmem + kTmemD + 32 * db, tmem + ab * 128, bd, idesc, first);
          else
            mma_unit<NT, 8>(tmem + kTmemD + 32 * db, tmem + ab * 128, bd, idesc, first);
          umma_commit(&a_empty[ab]);
          umma_commit(&empty[s]);
        }
        umma_commit(&d_full[db]);
      }
      if constexpr (EC) {
        bool u_ok = false;
        const uint32_t us = smem_u32(u_area);
        for (int t = 0; t < nT && ok; ++t, ++seg, ++ga) {
          const int db = seg & 1, ab = ga % kNA;
          if (seg >= 2 && !(ok = mbar_wait_bounded(&d_empty[db], ((seg / 2) - 1) & 1, p.wait_ns))) break;
          if (!(ok = mbar_wait_bounded(&a_full[ab], (ga / kNA) & 1, p.wait_ns))) break;
          if (!u_ok && !(ok = u_ok = mbar_wait_bounded(u_ready, 0, 4 * p.wait_ns))) break;
          tc_fence_after_sync();
          // (a loop here: the unrolled, guarded form of mma_unit produced wrong
          // results for rank >= 32 in testing)
          for (int k = 0; k < p.rank / 16; ++k)
            umma_ts_bf16(tmem + kTmemD + 32 * db, tmem + ab * 128 + 8 * k,
                         sw128_kmajor_desc(us + (k >> 2) * NT * 128 + 32 * (k & 3)), idesc, k != 0);
          umma_commit(&a_empty[ab]);
          umma_commit(&d_full[db]);
        }
      }
      if (!ok) atomicOr(&p.sync->status, kStatusTimeoutPipe);
      umma_commit(mma_done);  // every MMA above has finished before tensor memory is freed
      mbar_wait_bounded(mma_done, 0, p.wait_ns);
    }
  } else if (warp >= kWEc0) {
    // ------------------------------------------------------------ compensator
    if constexpr (EC) {
      const int ew = warp - kWEc0;
      ec_prefetch(p, ew, lane);
      asm volatile("griddepcontrol.wait;" ::: "memory");
      ec_project<NT / 8>(p, ew, lane);
      __threadfence();
      ec_bar();
      if (ew == 0 && lane == 0) {
        if (!p.skip_arrive) atomicAdd(&p.sync->arrive, 1u);
        const unsigned target = gridDim.x;
        bool arrived = ld_acquire_gpu(&p.sync->arrive) >= target;
        if (!arrived) {
          const uint64_t t0 = globaltimer();
          while (!(arrived = ld_acquire_gpu(&p.sync->arrive) >= target)) {
            if (globaltimer() - t0 > p.wait_ns) break;
            __nanosleep(64);
          }
        }
        if (!arrived) atomicOr(&p.sync->status, kStatusTimeoutZ);
        *ec_flag = arrived ? 1 : 0;
        __threadfence_block();
      }
      ec_bar();
      const bool arrived = *ec_flag != 0;
      ec_build_u<NT>(p, arrived, ew * 32 + lane, u_area, mlp, mlp + p.M * p.rank);
      fence_proxy_async_smem();  // generic-proxy writes of u, read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(u_ready);
      // the last CTA (over the grid) to have read z clears it and the counters
      ec_bar();
      if (ew == 0) {
        int last = 0;
        if (lane == 0 && arrived) {
          __threadfence();
          last = atomicAdd(&p.sync->depart, 1u) == gridDim.x - 1;
          __threadfence();
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          for (int idx = lane; idx < p.rank * 8; idx += 32)
            reinterpret_cast<float4*>(p.z)[idx] = make_float4(0.f, 0.f, 0.f, 0.f);
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            p.sync->arrive = 0;
            p.sync->depart = 0;
            __threadfence();
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row = 32 * q + lane;
    bool alive = true;  // after a timeout the warp still takes part in every epi_bar, with zeros
    int seg = 0;
    auto segment = [&](int tile, int slot, bool whole, int c_first, int c_last) {
      const int db = seg & 1;
      if (alive && !mbar_wait_bounded(&d_full[db], (seg / 2) & 1, 4 * p.wait_ns)) {
        if (lane == 0) atomicOr(&p.sync->status, kStatusTimeoutPipe);
        alive = false;
      }
      float v[NT];
      if (alive) {
        tc_fence_after_sync();
#pragma unroll
        for (int c0 = 0; c0 < NT; c0 += 16) {
          uint32_t tv[16];
          tmem_ld_x16(tmem + ((uint32_t)(32 * q) << 16) + kTmemD + 32 * db + c0, tv);
          tmem_ld_wait();
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) v[c0 + jj] = __uint_as_float(tv[jj]);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&d_empty[db]);
      } else {
#pragma unroll
        for (int m = 0; m < NT; ++m) v[m] = 0.f;
      }
      ++seg;
      const int n = tile * 128 + row;
      bool fin = whole;
      if (!whole) {
        const unsigned contributors = (unsigned)(c_last - c_first + 1) + (EC ? 1u : 0u);
        float* mine = p.y32 + ((size_t)slot * 128 + row) * 32;
#pragma unroll
        for (int m = 0; m < NT; m += 4)
          if (m < p.M) __stcg(reinterpret_cast<float4*>(mine + m), make_float4(v[m], v[m + 1], v[m + 2], v[m + 3]));
        __threadfence();
        epi_bar();
        if (threadIdx.x == kDq * 32) {
          flags[0] = atomicAdd(&p.tile_cnt[tile], 1u) == contributors - 1;
          __threadfence();
        }
        epi_bar();
        fin = flags[0] != 0;
        if (fin) {
          // fixed order: the weight segments' slots by CTA, then the tail's slot
          const int n_sl = c_last - c_first + 1 + (EC ? 1 : 0);
          for (int k = 0; k < n_sl; ++k) {
            const int sl = k <= c_last - c_first ? c_first + k + tile : (int)gridDim.x + p.nt + tile;
            const float* part = p.y32 + ((size_t)sl * 128 + row) * 32;
#pragma unroll
            for (int m = 0; m < NT; m += 4)
              if (m < p.M) {
                const float4 t4 = __ldcg(reinterpret_cast<const float4*>(part + m));
                v[m] = k == 0 ? t4.x : v[m] + t4.x;
                v[m + 1] = k == 0 ? t4.y : v[m + 1] + t4.y;
                v[m + 2] = k == 0 ? t4.z : v[m + 2] + t4.z;
                v[m + 3] = k == 0 ? t4.w : v[m + 3] + t4.w;
              }
          }
          if (threadIdx.x == kDq * 32) p.tile_cnt[tile] = 0;
        }
        epi_bar();  // flags[0] is reused by the next segment
      }
      if (fin && n < p.N) {
#pragma unroll
        for (int m = 0; m < NT; ++m)
          if (m < p.M) p.y[(size_t)m * p.N + n] = __float2bfloat16_rn(v[m]);
      }
    };
    for (int i = 0; i < nW;) {
      const int tile = (ub + i) / spt;
      const int seg_end = min(nW, (tile + 1) * spt - ub);
      const int c_first = sp.owner(tile * spt), c_last = sp.owner((tile + 1) * spt - 1);
      const bool whole = !EC && (ub + i == tile * spt) && (ub + seg_end == (tile + 1) * spt);
      segment(tile, (int)blockIdx.x + tile, whole, c_first, c_last);
      i = seg_end;
    }
    if constexpr (EC) {
      for (int t = 0; t < nT; ++t) {
        const int tile = (int)blockIdx.x + t * (int)gridDim.x;
        const int c_first = sp.owner(tile * spt), c_last = sp.owner((tile + 1) * spt - 1);
        segment(tile, (int)gridDim.x + p.nt + tile, false, c_first, c_last);
      }
    }
  }

  // single-lane roles leave warps split: reconverge before the CTA barrier
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWProd) tmem_dealloc(tmem, 512);
}

template <int NT, bool EC>
cudaError_t launch_tc(const TcParams& p, const CUtensorMap& xmap, int grid, size_t smem, cudaStream_t st) {
  static bool configured = false;
  auto k = decode_tc_kernel<NT, EC>;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThr);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p, xmap);
}

}  // namespace
}  // namespace spear

using namespace spear;

spear_status_t spear_launch_decode_tc(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                      cudaStream_t stream) {
  const int NT = M <= 16 ? 16 : 32;
  const bool ec = h->rank > 0;
  TcParams p{};
  p.wq = h->wq_pre;
  p.sz = h->sz_pre;
  p.a_frag = h->a_dec;
  p.b_rows = h->b_pre;
  p.x = x;
  p.y = y;
  p.y32 = h->y32_tc;
  p.tile_cnt = h->tile_cnt_tc;
  p.z = h->z_dec;
  p.sync = h->sync;
  p.gw1 = h->gate_w1;
  p.gw2 = h->gate_w2;
  p.K = h->K;
  p.N = h->N;
  p.M = M;
  p.n_groups = h->n_groups;
  p.G = h->G;
  p.rank = h->rank;
  p.gate = h->gate;
  p.gh = h->gate_hidden;
  p.alpha = h->alpha;
  p.nt = h->nt128;
  p.spt = (h->K + kStageK - 1) / kStageK;
  p.units = p.nt * p.spt;
  p.wait_ns = h->wait_ns;
  p.skip_arrive = h->skip_arrive;
  const int grid = p.units < h->sm_count ? p.units : h->sm_count;

  p.x_bytes = (uint32_t)kStageK * NT * 2;
  p.slot_bytes = kWBytes + kSzBytes + p.x_bytes;
  const size_t u_bytes = ec ? (size_t)((h->rank + 63) / 64) * NT * 128 : 0;
  const size_t mlp_bytes = h->gate_hidden > 0 ? (size_t)M * (h->rank + h->gate_hidden) * 4 : 0;
  const size_t cap = 227 * 1024 - 1024 - 1024;  // alignment slack, barriers
  int NS = (int)((cap - u_bytes - mlp_bytes) / p.slot_bytes);
  if (NS > kMaxSlots) NS = kMaxSlots;
  if (NS < 2) return SPEAR_ERR_UNSUPPORTED;
  p.NS = NS;
  p.u_off = (uint32_t)(1024 + (size_t)NS * p.slot_bytes);
  p.mlp_off = (uint32_t)(p.u_off + u_bytes);
  const size_t smem = 1024 + (size_t)p.mlp_off + mlp_bytes;

  CUtensorMap xmap;
  if (!encode_x_map(&xmap, x, M, h->K, NT, kStageK)) return SPEAR_ERR_CUDA;
  cudaError_t e;
  if (NT == 16)
    e = ec ? launch_tc<16, true>(p, xmap, grid, smem, stream) : launch_tc<16, false>(p, xmap, grid, smem, stream);
  else
    e = ec ? launch_tc<32, true>(p, xmap, grid, smem, stream) : launch_tc<32, false>(p, xmap, grid, smem, stream);
  return e == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}
