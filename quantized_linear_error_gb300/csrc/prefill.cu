// Prefill-phase path ("SPEAR: A System for Post-Quantization Error-Adaptive
// Recovery", section 2.2A: for M > 1 the layer is compute-bound, and the
// compensator runs as a separate small kernel next to the low-bit GEMM).
//
// Two launches of one warp-specialised tcgen05 GEMM kernel, D = A B^T with
// bf16 operands in 128-byte-swizzled shared memory and an fp32 accumulator
// in tensor memory (128 rows x TN columns, one tile per CTA):
//
//  1. Compensator pre-kernel (rank > 0): A = x (128 tokens per tile), B = the
//     compensator's A matrix (rank rows), both by TMA; the epilogue applies
//     the gate and writes u' = bf16(alpha * gamma(z) * z), z = A x, [M][rank].
//  2. Main kernel: A = W rows, dequantised in the CTA: the TMA warp brings
//     the packed INT4 tile and its scale/zero words, four warps turn them into
//     bf16 (q - z) * s (one rounding, the exported dequantised value), one
//     row per thread, and write them straight into the stage's A slot in
//     tensor memory (tcgen05.st; one slot per pipeline stage), so the
//     dequantised tile never passes through shared memory; B = x tokens by
//     TMA. After the K blocks of W
//     come ceil(rank / 64) more K blocks with A = rows of the compensator's B
//     matrix (read by the same four warps into the same slots) and B = u' by
//     TMA: since W x + B u' = [W | B] [x ; u'],
//     the same accumulator absorbs the compensator term. The epilogue reads
//     TMEM (lane = output row n, column = token) and stores y in bf16.
//
// Warp roles: warp 0 issues TMA (one thread) and owns the TMEM allocation,
// warp 1 issues tcgen05.mma (one thread), warps 2-5 dequantise and then run
// the epilogue (warp w reads TMEM lanes 32 (w % 4) .. + 31). Every mbarrier
// wait is bounded; a timeout latches the handle's status word. The MMA
// thread's loop is on the critical path (a few hundred cycles of its own
// latency per K block would idle the tensor core), so it waits on one barrier
// per stage (TMA bytes and the dequantisers' arrivals together) and commits
// once, and all roles step the stage index by counting.
#include <algorithm>
#include <cstring>

#include "internal.h"
#include "tcgen05.cuh"

namespace spear {
namespace {

constexpr int kThreads = 192;
constexpr int kATileBytes = 128 * 128;         // 128 rows x 64 bf16
constexpr int kRawWBytes = 128 * 8 * 4;        // 128 rows x 64 codes, packed
constexpr int kRawBytes = kRawWBytes + 128 * 4;  // plus one scale/zero word per row
constexpr int kBarrierBytes = 1024;
constexpr int kMaxStages = 6;
constexpr uint32_t kHintNs = 100;  // suspend-time hint of the pipeline waits
constexpr uint32_t kTmemA = 256;       // main kernel: A operand of stage s at column 256 + 32 s (after the accumulator)
static_assert(kTmemA + 32 * kMaxStages <= 512, "the A slots of every stage fit in tensor memory");

struct GemmParams {
  int kblocks;      // K blocks of 64 from the main operands (per split for the pre-kernel)
  int kb_total;     // all K blocks (the last split may be shorter)
  int tail_blocks;  // compensator K blocks (main kernel: A rows of B through tensor memory, B = u' from mapBt)
  int TN;           // B rows per tile = MMA N (multiple of 16, <= 256)
  int a_rows;       // rows of the A operand (W rows, or tokens for the pre-kernel)
  int b_rows;       // rows of the B operand (tokens, or rank for the pre-kernel)
  int K;
  const uint32_t* wq;  // prefill-layout packed W
  const uint32_t* sz;  // prefill-layout scale/zero words
  int n_groups, G;
  __nv_bfloat16* out;
  int ld_out;
  float alpha;
  int gate;
  int rank_b;                // pre-kernel: column c of u' belongs to member c / rank_b (grouped handle)
  float alphas[kMaxGroup];   // pre-kernel: each member's alpha
  unsigned* status;
  uint64_t wait_ns;
  int skip_arrive;  // test surface: splits other than the leader skip their arrival on part_cnt
  int NS;
  uint32_t a_bytes, b_bytes, raw_bytes, stage_bytes;
  uint32_t tmem_cols;
  const __nv_bfloat16* bt;  // main kernel: compensator B rows [nt128 * 128][rank] (the K-tail's A operand)
  const __nv_bfloat16* gw1;  // pre-kernel, SPEAR_GATE_MLP: W1 [gh][rank]
  const __nv_bfloat16* gw2;  // pre-kernel, SPEAR_GATE_MLP: W2 [rank][gh]
  int gh;
  int mlp_stage_w;  // pre-kernel, SPEAR_GATE_MLP: W1 and W2 staged in shared memory (they fit)
  int rank;
  float* zacc;          // pre-kernel: fp32 [M][rank] partial sums of z (zero between calls)
  unsigned* tile_done;  // pre-kernel: per 128-token tile, splits finished
  int splits;
  // main kernel split over K (gridDim.z splits of kps K blocks; the last one
  // also runs the compensator K-tail): fp32 partial tiles
  // part [split][tile][128][TN] and per-tile counters of finished splits
  int kps;
  float* part;
  unsigned* part_cnt;
  // main kernel, compensator on a concurrent stream: the main contraction
  // writes its fp32 result to y32_out [M][N] instead of y; the K-tail launch
  // (no W blocks) adds y32_in [M][N] to its accumulator before the rounding
  float* y32_out;
  const float* y32_in;
};

SPEAR_DEVINL void fail(const GemmParams& p) { atomicOr(p.status, kStatusTimeoutPipe); }


SPEAR_DEVINL uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

SPEAR_DEVINL float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
SPEAR_DEVINL float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// sum_k w[k] v[k] over n = 8 * n8 bf16 weights (16-byte rows) and fp32 values.
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

SPEAR_DEVINL float gate_apply(float z, int gate) {
  return gate == SPEAR_GATE_ONE ? z : z * (1.0f / (1.0f + expf(-z)));
}

SPEAR_DEVINL void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

// Named barrier of the 4 epilogue warps; bar.sync counts whole warps, so a
// warp split by a single-thread branch reconverges first.
SPEAR_DEVINL void epilogue_bar() {
  __syncwarp();
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

template <bool DEQ, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const GemmParams p, const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                const __grid_constant__ CUtensorMap mapAt, const __grid_constant__ CUtensorMap mapBt) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  // Per stage s: full[s] = the stage's operands are ready for the MMA (B, and
  // A, in shared memory by TMA; main kernel: B by TMA plus the A operand in
  // tensor memory from the four dequantising warps), raw_full[s] = main
  // kernel: the packed W tile and its scale/zero words have landed (the
  // dequantisers' input), empty[s] = the MMAs of the stage have completed, so
  // its shared memory and its A slot in tensor memory may be refilled.
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* raw_full = full + 8;
  uint64_t* empty = full + 16;
  uint64_t* acc_full = full + 24;
  uint64_t* part_bar = full + 32;  // main kernel split over K: the other splits' partials are in smem
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 384);
  uint8_t* stages = smem + kBarrierBytes;
  const uint32_t stages_s = smem_u32(stages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a0 = blockIdx.x * 128;
  // main kernel: blockIdx.y is the token tile, blockIdx.z the K split;
  // pre-kernel: blockIdx.y is the K split
  const int b0 = EPI == 2 ? 0 : blockIdx.y * p.TN;
  const int kb0 = EPI == 2 ? blockIdx.y * p.kblocks : (DEQ ? blockIdx.z * p.kps : 0);
  const int kmain = EPI == 2 ? min(p.kblocks, p.kb_total - kb0) : (DEQ ? min(p.kps, p.kb_total - kb0) : p.kblocks);
  const int tail = (DEQ && blockIdx.z + 1 != gridDim.z) ? 0 : p.tail_blocks;
  const int total = kmain + tail;
  volatile int& last_split = *reinterpret_cast<volatile int*>(smem + 512);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(&full[s], DEQ ? 5 : 1);
      mbar_init(&raw_full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(part_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_d = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // Grid dependencies. The pre-kernel reads x, written by the previous kernel:
  // it waits for that grid, then lets the main kernel launch. The main kernel
  // can then read x at once (x's producer has completed) and waits for the
  // pre-kernel only before it loads u' for its compensator K-tail; without a
  // compensator it waits for its predecessor here. Either kernel lets the
  // next one launch early; the next one waits for it before reading anything
  // it writes.
  const bool late_wait = DEQ && tail > 0;
  if (!late_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      if (DEQ && tail > 0) prefetch_l2(p.bt + (size_t)a0 * p.rank, 128u * p.rank * 2u);
      // stage s and the parity of its current fill, advanced by counting (the
      // loops of the three roles are short enough that a division by the
      // runtime stage count would show in the time per K block)
      int s = 0;
      unsigned ph = 0;
      for (int it = 0; it < total; ++it) {
        if (it >= p.NS && !mbar_wait_bounded_hint(&empty[s], ph ^ 1u, p.wait_ns, kHintNs)) {
          fail(p);
          break;
        }
        uint8_t* st = stages + (size_t)s * p.stage_bytes;
        uint8_t* A = st;
        uint8_t* B = st + p.a_bytes;
        uint8_t* raw = B + p.b_bytes;
        if (it < kmain) {
          if constexpr (DEQ) {
            mbar_arrive_expect_tx(&raw_full[s], kRawBytes);
            bulk_g2s(raw, p.wq + ((size_t)blockIdx.x * p.kb_total + kb0 + it) * 1024, kRawWBytes, &raw_full[s]);
            bulk_g2s(raw + kRawWBytes, p.sz + ((size_t)blockIdx.x * p.n_groups + ((kb0 + it) * 64) / p.G) * 128,
                     512, &raw_full[s]);
            mbar_arrive_expect_tx(&full[s], p.b_bytes);
          } else {
            mbar_arrive_expect_tx(&full[s], kATileBytes + p.b_bytes);
            tma_load_2d(A, &mapA, (kb0 + it) * 64, a0, &full[s]);
          }
          tma_load_2d(B, &mapB, (kb0 + it) * 64, b0, &full[s]);
        } else {
          // compensator K-tail: A rows (read from global memory by the
          // dequantisers, who may fill the stage's A slot from now on) through
          // tensor memory, B = u' from the pre-kernel
          const int t = it - kmain;
          if (DEQ) mbar_arrive(&raw_full[s]);
          if (t == 0 && late_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
          mbar_arrive_expect_tx(&full[s], p.b_bytes);
          tma_load_2d(B, &mapBt, t * 64, b0, &full[s]);
        }
        if (++s == p.NS) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, p.TN);
      int s = 0;
      unsigned ph = 0;
      uint32_t a_s = stages_s;
      for (int it = 0; it < total; ++it) {
        if (!mbar_wait_bounded_hint(&full[s], ph, p.wait_ns, kHintNs)) {
          fail(p);
          break;
        }
        tc_fence_after_sync();
        const uint32_t b_s = a_s + p.a_bytes;
        if (DEQ) {
          // A from tensor memory: 8 columns (16 channels) per k16 step
#pragma unroll
          for (int k16 = 0; k16 < 4; ++k16)
            umma_ts_bf16(tmem_d, tmem_d + kTmemA + 32 * s + 8 * k16, sw128_kmajor_desc(b_s + 32 * k16), idesc,
                         (it | k16) != 0);
        } else {
#pragma unroll
          for (int k16 = 0; k16 < 4; ++k16)
            umma_bf16(tmem_d, sw128_kmajor_desc(a_s + 32 * k16), sw128_kmajor_desc(b_s + 32 * k16), idesc,
                      (it | k16) != 0);
        }
        umma_commit(&empty[s]);
        a_s += p.stage_bytes;
        if (++s == p.NS) {
          s = 0;
          ph ^= 1u;
          a_s = stages_s;
        }
      }
      umma_commit(acc_full);  // the accumulator is complete once every MMA above has finished
    }
  } else {
    // ---------------------------------------------------------- dequantisers
    // One thread per row: warp w owns tensor-memory lanes 32 (w % 4) .. + 31,
    // i.e. rows r = 32 (w % 4) + lane of the tile. Per K block a thread reads
    // its row's 8 packed words and scale/zero word, makes 32 bf16 pairs (pair
    // c = channels 2c, 2c + 1) and stores them as the 32 columns of the
    // stage's A slot. raw_full[s] also says that the slot is free: the
    // producer refills a stage only after the MMAs that read it completed.
    // The store of block it is still in flight while block it + 1 is
    // converted; block it counts towards full[s] once its store has completed.
    if constexpr (DEQ) {
      const int q = warp & 3;
      const int r = 32 * q + lane;
      const uint32_t lane_base = tmem_d + ((uint32_t)(32 * q) << 16) + kTmemA;
      int s = 0;
      unsigned ph = 0;
      uint32_t raw_sa = stages_s + p.a_bytes + p.b_bytes;
      int pending = -1;  // stage whose A store is in flight
      for (int it = 0; it < total; ++it) {
        uint32_t v[32];
        if (it < kmain) {
          if (!mbar_wait_bounded_hint(&raw_full[s], ph, p.wait_ns, kHintNs)) {
            fail(p);
            break;
          }
          const uint4 w0 = lds128(raw_sa + (uint32_t)(r * 32));
          const uint4 w1 = lds128(raw_sa + (uint32_t)(r * 32 + 16));
          const uint32_t szw = lds32(raw_sa + kRawWBytes + r * 4);
          const uint32_t zz = biased_zero_x2(szw >> 16);
          const uint32_t sc = (szw & 0xFFFFu) | (szw << 16);
          const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int c = 0; c < 8; ++c)
#pragma unroll
            for (int j = 0; j < 4; ++j)
              v[4 * c + j] = bf16x2_mul(bf16x2_sub(int4_pair_to_bf16x2_biased(words[c] >> (4 * j)), zz), sc);
        } else {
          // row a0 + r of the compensator's B, columns 64 t .. + 63 (zero past rank)
          const int t = it - kmain;
          const uint4* src = reinterpret_cast<const uint4*>(p.bt + (size_t)(a0 + r) * p.rank + t * 64);
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const uint4 w = t * 64 + c8 * 8 < p.rank ? __ldg(src + c8) : make_uint4(0u, 0u, 0u, 0u);
            v[4 * c8] = w.x;
            v[4 * c8 + 1] = w.y;
            v[4 * c8 + 2] = w.z;
            v[4 * c8 + 3] = w.w;
          }
          if (!mbar_wait_bounded_hint(&raw_full[s], ph, p.wait_ns, kHintNs)) {
            fail(p);
            break;
          }
        }
        if (pending >= 0) {
          tmem_st_wait();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[pending]);
        }
        tc_fence_after_sync();
        tmem_st_x32(lane_base + 32 * s, v);
        pending = s;
        raw_sa += p.stage_bytes;
        if (++s == p.NS) {
          s = 0;
          ph ^= 1u;
          raw_sa = stages_s + p.a_bytes + p.b_bytes;
        }
      }
      if (pending >= 0) {
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[pending]);
      }
    }

    // ---------------------------------------------------------- epilogue
    bool ok = mbar_wait_bounded(acc_full, 0, 4 * p.wait_ns);
    if (!ok && lane == 0) fail(p);
    tc_fence_after_sync();
    const int q = warp & 3;
    const int row = a0 + 32 * q + lane;
    // Split over K (main kernel): splits 0 .. S-2 store their fp32 partial
    // tile ([column][row]) and count themselves done; split S-1, which also
    // ran the compensator K-tail, waits for that count, pulls the S-1
    // partials into its now idle stage memory with one bulk copy each, and
    // adds them in split order to its own accumulator before the single
    // rounding to bf16. (A last-arriver pass that re-read every partial
    // through the load path was latency-bound.)
    const bool split = EPI == 0 && gridDim.z > 1;
    const bool leader = split && blockIdx.z + 1 == gridDim.z;
    const unsigned tile_id = blockIdx.y * gridDim.x + blockIdx.x;
    const size_t part_tile = (size_t)p.TN * 128;  // floats of one partial tile
    if (leader) {
      if (threadIdx.x == 64) {
        bool got = false;
        if (ok) {
          const unsigned want = gridDim.z - 1;
          const uint64_t t0 = globaltimer();
          while (!(got = ld_acquire_gpu(&p.part_cnt[tile_id]) >= want)) {
            if (globaltimer() - t0 > 4 * p.wait_ns) break;
            __nanosleep(64);
          }
          if (!got) fail(p);
        }
        last_split = got ? 1 : 0;
        if (got) {
          p.part_cnt[tile_id] = 0;  // every other split has counted itself: reset for the next call
          mbar_arrive_expect_tx(part_bar, (unsigned)(part_tile * 4 * (gridDim.z - 1)));
          for (unsigned z = 0; z + 1 < gridDim.z; ++z)
            bulk_g2s(stages + z * part_tile * 4, p.part + ((size_t)z * gridDim.x * gridDim.y + tile_id) * part_tile,
                     (unsigned)(part_tile * 4), part_bar);
        }
      }
      epilogue_bar();
      ok = last_split != 0 && mbar_wait_bounded(part_bar, 0, 4 * p.wait_ns);
      if (last_split != 0 && !ok && lane == 0) fail(p);
    }
    // main kernel: the bf16 y tile, after the leader's partials in the idle stage memory
    const uint32_t ytile_s = stages_s + (leader ? (uint32_t)((gridDim.z - 1) * part_tile * 4) : 0u);
    if (ok) {
      for (int c0 = 0; c0 < p.TN; c0 += 16) {
        uint32_t v[16];
        tmem_ld_x16(tmem_d + ((uint32_t)(32 * q) << 16) + c0, v);
        tmem_ld_wait();
        if constexpr (EPI == 0) {
          if (split && !leader) {
            // this split's fp32 partial tile, [column][row], so that a warp's
            // 32 rows of one column are 128 contiguous bytes
            float* dst = p.part + ((size_t)blockIdx.z * gridDim.x * gridDim.y + tile_id) * part_tile +
                         (size_t)c0 * 128 + 32 * q + lane;
#pragma unroll
            for (int j = 0; j < 16; ++j) __stcg(dst + j * 128, __uint_as_float(v[j]));
          } else if (p.y32_out != nullptr) {
            // fp32 result for the separate compensator K-tail: lane = row n
            // (consecutive lanes, consecutive addresses), columns = tokens
            if (row < p.a_rows)
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (b0 + c0 + j < p.b_rows)
                  __stcg(p.y32_out + (size_t)(b0 + c0 + j) * p.ld_out + row, __uint_as_float(v[j]));
          } else if (row < p.a_rows) {
            if (p.y32_in != nullptr) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (b0 + c0 + j < p.b_rows)
                  v[j] = __float_as_uint(__uint_as_float(v[j]) +
                                         __ldcg(p.y32_in + (size_t)(b0 + c0 + j) * p.ld_out + row));
            }
            if (leader) {
              // add the other splits' partials, in split order, from shared
              // memory (shared-space loads, all 16 of a split in flight at once)
              const uint32_t ps = stages_s + (uint32_t)((c0 * 128 + 32 * q + lane) * 4);
              float acc16[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) acc16[j] = 0.f;
              for (unsigned z = 0; z + 1 < gridDim.z; ++z) {
                uint32_t w16[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) w16[j] = lds32(ps + (uint32_t)((z * part_tile + j * 128) * 4));
#pragma unroll
                for (int j = 0; j < 16; ++j) acc16[j] = z == 0 ? __uint_as_float(w16[j]) : acc16[j] + __uint_as_float(w16[j]);
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(acc16[j] + __uint_as_float(v[j]));
            }
            // y tile staged in shared memory as bf16 [token][128 rows], stored below
            // with 16-byte vectors along n (lane = n here, columns = tokens)
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(v[j]));
              asm volatile("st.shared.b16 [%0], %1;" ::"r"(ytile_s + (uint32_t)(((c0 + j) * 128 + 32 * q + lane) * 2)),
                           "h"(*reinterpret_cast<const unsigned short*>(&h)));
            }
          }
        } else if constexpr (EPI == 1) {
          // u'[m][j] = bf16(alpha * gamma(z) * z): lane = token m, columns = rank index
          if (row < p.a_rows) {
            uint32_t pk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float al = p.alphas[(c0 + 2 * j) / p.rank_b];  // c0 + 2j and + 1: same member
              pk[j] = pack_bf16x2(al * gate_apply(__uint_as_float(v[2 * j]), p.gate),
                                  al * gate_apply(__uint_as_float(v[2 * j + 1]), p.gate));
            }
            uint4* dst = reinterpret_cast<uint4*>(p.out + (size_t)row * p.ld_out + c0);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        } else {
          // split-K partial of z: add into the fp32 accumulator
          if (row < p.a_rows) {
            float* dst = p.zacc + (size_t)row * p.ld_out + c0;
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              red_add_v4(dst + j, __uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                         __uint_as_float(v[j + 3]));
          }
        }
      }
    }
    if (EPI == 0 && !(split && !leader) && p.y32_out == nullptr) {
      // 16-byte stores of the staged tile: token m, rows a0 + 8 c8 .. + 7
      // (the barrier is unconditional: every epilogue warp reaches it)
      epilogue_bar();
      const int t = threadIdx.x - 64;  // the four epilogue warps
      for (int i = t; ok && i < p.TN * 16; i += 128) {
        const int mm = i >> 4, c8 = i & 15;
        const int m = b0 + mm, n0 = a0 + 8 * c8;
        if (m < p.b_rows && n0 < p.a_rows) {
          uint4 w;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                       : "r"(ytile_s + (uint32_t)((mm * 128 + 8 * c8) * 2)));
          *reinterpret_cast<uint4*>(p.out + (size_t)m * p.ld_out + n0) = w;
        }
      }
    }
    if (split && !leader) {
      // publish this split's partial tile to the leader
      __threadfence();
      epilogue_bar();
      if (threadIdx.x == 64 && ok && !p.skip_arrive) atomicAdd(&p.part_cnt[tile_id], 1u);
    }
    if constexpr (EPI == 2) {
      // The last split of this 128-token tile applies the gate to the complete z,
      // writes u' and clears z and the counter for the next call.
      __threadfence();
      epilogue_bar();
      if (threadIdx.x == 64) {
        last_split = ok && atomicAdd(&p.tile_done[blockIdx.x], 1u) == (unsigned)(p.splits - 1);
        __threadfence();
      }
      epilogue_bar();
      if (last_split && p.gate == SPEAR_GATE_MLP) {
        // Bottleneck-MLP gate: warp q stages z rows a0 + 32 q .. + 31 in the
        // (now idle) stage memory (rows padded by 8 floats: conflict-free
        // fragment reads), then evaluates the gate for its two 16-token blocks
        // on warp MMAs (mlp_gate_logits): u' = bf16(alpha sigmoid(W2 relu(W1 z)) (.) z).
        const int zst = p.TN + 8;
        float* zt = reinterpret_cast<float*>(stages);
        for (int rr = 0; rr < 32; ++rr) {
          const int m = a0 + 32 * q + rr;
          for (int c = lane; c < p.TN; c += 32)
            zt[(32 * q + rr) * zst + c] = m < p.a_rows ? __ldcg(p.zacc + (size_t)m * p.ld_out + c) : 0.f;
        }
        // W1 [gh][rank + 8] and W2 [rank][gh + 8] after the 128 z rows when
        // they fit the stage area, else read from global memory
        const __nv_bfloat16* w1 = p.gw1;
        const __nv_bfloat16* w2 = p.gw2;
        int w1s = p.TN, w2s = p.gh;
        if (p.mlp_stage_w) {
          __nv_bfloat16* s1 = reinterpret_cast<__nv_bfloat16*>(zt + 128 * zst);
          __nv_bfloat16* s2 = s1 + p.gh * (p.TN + 8);
          stage_rows_padded(s1, p.gw1, p.gh, p.TN, threadIdx.x - 64, 128);
          stage_rows_padded(s2, p.gw2, p.TN, p.gh, threadIdx.x - 64, 128);
          w1 = s1;
          w2 = s2;
          w1s = p.TN + 8;
          w2s = p.gh + 8;
        }
        epilogue_bar();
        for (int tb = 0; tb < 2; ++tb)
          mlp_gate_logits(zt, zst, 32 * q + 16 * tb, p.TN, p.gh, w1, w1s, w2, w2s, lane, 0, p.TN / 8,
                          [&](int lr, int j, float g0, float g1) {
                            const int m = a0 + lr;
                            if (m >= p.a_rows) return;
                            const float* zr = zt + lr * zst;
                            *reinterpret_cast<uint32_t*>(p.out + (size_t)m * p.ld_out + j) =
                                pack_bf16x2(p.alpha * zr[j] * (1.0f / (1.0f + expf(-g0))),
                                            p.alpha * zr[j + 1] * (1.0f / (1.0f + expf(-g1))));
                          });
        __syncwarp();
        for (int rr = 0; rr < 32; ++rr) {
          const int mm = a0 + 32 * q + rr;
          if (mm < p.a_rows)
            for (int c = lane * 4; c < p.TN; c += 128)
              *reinterpret_cast<float4*>(p.zacc + (size_t)mm * p.ld_out + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      } else if (last_split) {
        // Warp q finishes rows a0 + 32 q .. + 31, eight rows per round with all
        // loads in flight; lanes run along the row (coalesced), 4 columns each.
        for (int r0 = 0; r0 < 32; r0 += 8) {
          for (int c = lane * 4; c < p.TN; c += 128) {
            float4 zv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int m = a0 + 32 * q + r0 + j;
              zv[j] = m < p.a_rows ? __ldcg(reinterpret_cast<const float4*>(p.zacc + (size_t)m * p.ld_out + c))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int m = a0 + 32 * q + r0 + j;
              if (m < p.a_rows) {
                const float al = p.alphas[c / p.rank_b];  // columns c .. c + 3: one member
                const uint2 pk = make_uint2(pack_bf16x2(al * gate_apply(zv[j].x, p.gate),
                                                        al * gate_apply(zv[j].y, p.gate)),
                                            pack_bf16x2(al * gate_apply(zv[j].z, p.gate),
                                                        al * gate_apply(zv[j].w, p.gate)));
                *reinterpret_cast<uint2*>(p.out + (size_t)m * p.ld_out + c) = pk;
                *reinterpret_cast<float4*>(p.zacc + (size_t)m * p.ld_out + c) = make_float4(0.f, 0.f, 0.f, 0.f);
              }
            }
          }
        }
      }
      if (last_split && threadIdx.x == 64) p.tile_done[blockIdx.x] = 0;
    }
  }

  // single-thread roles leave warps split: reconverge before the CTA barrier
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_d, p.tmem_cols);
}

uint32_t tmem_cols_for(int n) {
  uint32_t c = 32;
  while (c < (uint32_t)n) c <<= 1;
  return c;
}

template <bool DEQ, int EPI>
cudaError_t launch(const GemmParams& p, dim3 grid, size_t smem, cudaStream_t st, const CUtensorMap& mA,
                   const CUtensorMap& mB, const CUtensorMap& mAt, const CUtensorMap& mBt) {
  static std::atomic<uint64_t> configured{0};  // devices whose limit is raised
  auto k = gemm_kernel<DEQ, EPI>;
  {
    cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(k), configured);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p, mA, mB, mAt, mBt);
}

// Stages that fit next to the barriers (one A tile, one B tile, raw W).
int stages_for(uint32_t stage_bytes) {
  const size_t budget = 227 * 1024 - kBarrierBytes - 1024;
  int ns = (int)(budget / stage_bytes);
  return ns > kMaxStages ? kMaxStages : ns;
}

}  // namespace
}  // namespace spear

using namespace spear;

// Tokens per tile: the fewest tiles of at most 256 tokens, split evenly and
// rounded up to the MMA's multiple of 16.
static int prefill_tn(int M) {
  const int tiles = (M + 255) / 256;
  int tn = (M + tiles - 1) / tiles;
  tn = (tn + 15) / 16 * 16;
  return tn < 16 ? 16 : tn;
}

// Compensator pre-kernel: u' [M][rank] = bf16(alpha gamma(A x) (.) A x).
// Sets *pre_ctas to the CTAs it runs on.
static spear_status_t launch_pre(spear_linear_s* h, const __nv_bfloat16* x, int M, cudaStream_t stream,
                                 int* pre_ctas) {
  const int K = h->K, r = h->rank;
  CUtensorMap none;
  memset(&none, 0, sizeof none);
  cudaError_t e;
  *pre_ctas = 0;
  {
    // ---- compensator projection and gate: u' [M][r]
    CUtensorMap mx, ma;
    if (!encode_2d_bf16(&mx, x, K, M, (uint64_t)K * 2, 64, 128) ||
        !encode_2d_bf16(&ma, h->a_pre, K, r, (uint64_t)K * 2, 64, r))
      return SPEAR_ERR_CUDA;
    GemmParams p{};
    const int kbt = K / 64, mt = (M + 127) / 128;
    // About 32 CTAs (at least 8 K blocks each): the pre-kernel runs on a few
    // SMs next to the main kernel, which needs u' only for its last K blocks.
    int splits = (32 + mt - 1) / mt;
    if (splits > kbt / 8) splits = kbt / 8;
    if (splits < 1) splits = 1;
    p.kblocks = (kbt + splits - 1) / splits;
    splits = (kbt + p.kblocks - 1) / p.kblocks;
    p.kb_total = kbt;
    p.splits = splits;
    p.zacc = h->z_pre;
    p.tile_done = h->pre_done;
    p.tail_blocks = 0;
    p.TN = r;
    p.a_rows = M;
    p.b_rows = r;
    p.K = K;
    p.out = h->u_pre;
    p.ld_out = r;
    p.alpha = h->alpha;
    p.gate = h->gate;
    p.rank_b = h->rank_b;
    for (int i = 0; i < h->n_members; ++i) p.alphas[i] = h->alphas[i];
    p.status = &h->sync->status;
    p.wait_ns = h->wait_ns;
    p.a_bytes = kATileBytes;
    p.b_bytes = (uint32_t)(r * 128 + 1023) / 1024 * 1024;
    p.raw_bytes = 0;
    p.stage_bytes = p.a_bytes + p.b_bytes;
    p.NS = stages_for(p.stage_bytes);
    p.gw1 = h->gate_w1;
    p.gw2 = h->gate_w2;
    p.gh = h->gate_hidden;
    if (h->gate_hidden > 0) {
      // the MLP gate stages 128 z rows in the stage area, and W1 and W2 after
      // them if that still fits
      const size_t need_z = (size_t)128 * (r + 8) * 4;
      const size_t need_w = need_z + ((size_t)h->gate_hidden * (r + 8) + (size_t)r * (h->gate_hidden + 8)) * 2;
      const size_t cap = 227 * 1024 - kBarrierBytes - 1024;
      const int ns_w = (int)((need_w + p.stage_bytes - 1) / p.stage_bytes);
      p.mlp_stage_w = ns_w <= 8 && (size_t)ns_w * p.stage_bytes <= cap;
      const size_t need = p.mlp_stage_w ? need_w : need_z;
      while ((size_t)p.NS * p.stage_bytes < need) ++p.NS;
      if (p.NS > 8 || kBarrierBytes + 1024 + (size_t)p.NS * p.stage_bytes > 227 * 1024) return SPEAR_ERR_UNSUPPORTED;
    }
    p.tmem_cols = tmem_cols_for(r);
    const size_t smem = kBarrierBytes + 1024 + (size_t)p.NS * p.stage_bytes;
    *pre_ctas = mt * splits;
    e = launch<false, 2>(p, dim3(mt, splits), smem, stream, mx, ma, none, none);
    if (e != cudaSuccess) return SPEAR_ERR_CUDA;
  }
  return SPEAR_OK;
}

// Main kernel. mode 0: W x plus the compensator K-tail, bf16 y; mode 1: W x
// only, fp32 result into h->y32; mode 2: the K-tail only, added to h->y32,
// bf16 y.
static spear_status_t launch_main(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                  cudaStream_t stream, int pre_ctas, int mode) {
  const int K = h->K, N = h->N;
  const int r = mode == 1 ? 0 : h->rank;
  CUtensorMap none;
  memset(&none, 0, sizeof none);
  cudaError_t e;
  // ---- main contraction with the compensator K-tail
  const int TN = prefill_tn(M);
  CUtensorMap mx, mut;
  if (!encode_2d_bf16(&mx, x, K, M, (uint64_t)K * 2, 64, TN)) return SPEAR_ERR_CUDA;
  if (r > 0) {
    if (!encode_2d_bf16(&mut, h->u_pre, r, M, (uint64_t)r * 2, 64, TN)) return SPEAR_ERR_CUDA;
  } else {
    mut = none;
  }
  GemmParams p{};
  const int kbt = K / 64, ntt = (M + TN - 1) / TN, tiles = h->nt128 * ntt;
  // Split K when the tiles fill less than one wave of CTAs (one per SM): up to
  // four splits of at least eight K blocks, (split, tile) pairs within the
  // SMs. Not with a compensator: its pre-kernel's CTAs run alongside, and the
  // split that runs the K-tail waits for them (measured slower than no split).
  int ks = 1;
  const int avail = h->sm_count - pre_ctas;
  if (h->part && r == 0 && mode == 0 && tiles < avail) {
    ks = std::min(std::min(4, avail / tiles), kbt / 8);
    if (ks < 1) ks = 1;
  }
  p.kps = (kbt + ks - 1) / ks;
  ks = (kbt + p.kps - 1) / p.kps;
  p.part = h->part;
  p.part_cnt = h->part_cnt;
  p.skip_arrive = h->skip_arrive;
  p.kblocks = mode == 2 ? 0 : kbt;
  p.kb_total = mode == 2 ? 0 : kbt;
  if (mode == 2) p.kps = 0;
  p.y32_out = mode == 1 ? h->y32 : nullptr;
  p.y32_in = mode == 2 ? h->y32 : nullptr;
  p.splits = 1;
  p.tail_blocks = (r + 63) / 64;
  p.TN = TN;
  p.a_rows = N;
  p.b_rows = M;
  p.K = K;
  p.wq = h->wq_pre;
  p.sz = h->sz_pre;
  p.n_groups = h->n_groups;
  p.G = h->G;
  p.out = y;
  p.ld_out = N;
  p.alpha = h->alpha;
  p.gate = h->gate;
  p.status = &h->sync->status;
  p.wait_ns = h->wait_ns;
  p.a_bytes = 0;  // every A operand of the main kernel lives in tensor memory
  p.bt = h->b_pre;
  p.rank = r;
  p.b_bytes = (uint32_t)(TN * 128 + 1023) / 1024 * 1024;
  p.raw_bytes = kRawBytes;
  p.stage_bytes = (p.a_bytes + p.b_bytes + kRawBytes + 1023) / 1024 * 1024;
  p.NS = stages_for(p.stage_bytes);
  // the split leader pulls the other splits' partial tiles into the stage area,
  // followed there by the bf16 y tile of the epilogue
  if ((size_t)TN * 256 > (size_t)p.NS * p.stage_bytes) return SPEAR_ERR_UNSUPPORTED;
  while (ks > 1 && (size_t)(ks - 1) * TN * 512 + (size_t)TN * 256 > (size_t)p.NS * p.stage_bytes) {
    --ks;
    p.kps = (kbt + ks - 1) / ks;
    ks = (kbt + p.kps - 1) / p.kps;
  }
  p.tmem_cols = 512;  // accumulator (TN <= 256 columns) + one A slot per stage from column 256
  const size_t smem = kBarrierBytes + 1024 + (size_t)p.NS * p.stage_bytes;
  e = launch<true, 0>(p, dim3(h->nt128, ntt, ks), smem, stream, none, mx, none, mut);
  return e == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}

spear_status_t spear_launch_prefill(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                    cudaStream_t stream) {
  int pre_ctas = 0;
  if (h->rank > 0) {
    spear_status_t st = launch_pre(h, x, M, stream, &pre_ctas);
    if (st != SPEAR_OK) return st;
  }
  return launch_main(h, x, y, M, stream, pre_ctas, 0);
}

// The compensator on a concurrent stream (the pages' semi-fused prefill): the
// pre-kernel runs on ec_stream next to the main contraction on `stream`, which
// writes fp32; after the join, the K-tail launch adds alpha B u' and rounds.
spear_status_t spear_launch_prefill_concurrent(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                               cudaStream_t stream, cudaStream_t ec_stream) {
  if (h->rank == 0) return spear_launch_prefill(h, x, y, M, stream);
  if (cudaEventRecord(h->ev_fork, stream) != cudaSuccess || cudaStreamWaitEvent(ec_stream, h->ev_fork, 0) != cudaSuccess)
    return SPEAR_ERR_CUDA;
  int pre_ctas = 0;
  spear_status_t st = launch_pre(h, x, M, ec_stream, &pre_ctas);
  if (st != SPEAR_OK) return st;
  st = launch_main(h, x, y, M, stream, 0, 1);
  if (st != SPEAR_OK) return st;
  if (cudaEventRecord(h->ev_join, ec_stream) != cudaSuccess || cudaStreamWaitEvent(stream, h->ev_join, 0) != cudaSuccess)
    return SPEAR_ERR_CUDA;
  return launch_main(h, x, y, M, stream, 0, 2);
}
