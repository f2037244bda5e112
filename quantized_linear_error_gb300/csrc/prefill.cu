// Prefill-phase path ("SPEAR: A System for Post-Quantization Error-Adaptive
// Recovery", section 2.2A: for M > 1 the layer is compute-bound; the
// compensator's skinny products run beside the low-bit GEMM).
//
// One persistent, warp-specialised tcgen05 GEMM kernel (main_kernel) with
// bf16 operands in 128-byte-swizzled shared memory and fp32 accumulators in
// tensor memory computes y = W x + B u', u' = bf16(alpha * gamma(z) * z),
// z = A x:
//
//  - Prologue (rank > 0): the compensator projection, one item per 128-token
//    tile, item i on CTA i (and i + G, ...): z = x A^T over all of K with
//    both operands by TMA, so z is complete in tensor memory; the epilogue
//    gates it there, builds the tile's u' rows in shared memory, writes
//    them with one bulk copy and raises the tile's "u' ready" flag. (Splits
//    over K with a cross-CTA reduction of z were slower: with every SM
//    streaming the main contraction, a round trip to L2 takes microseconds,
//    and fp32 atomics from every split queued up in L2 for longer still.)
//  - Main contraction: A = W rows, dequantised in the CTA: the TMA thread
//    brings the packed INT4 block and its scale/zero words, four warps turn
//    them into bf16 (q - z) * s (one rounding, the exported dequantised
//    value), one row per thread, and write them straight into the stage's A
//    slot in tensor memory (tcgen05.st), so the dequantised tile never passes
//    through shared memory; B = x tokens by TMA. A tile's compensator K-tail
//    (ceil(rank / 64) more K blocks, A = rows of the compensator's B matrix,
//    B = u') lands in the same accumulator, since W x + B u' = [W | B] [x ; u'].
//
// The main contraction follows a "stream-K" schedule: a tile (128 output rows
// x TN tokens) is kpt = tail + kbt work units, its K-tail blocks first and
// then its W blocks, and the G CTAs (at most one per SM) take contiguous
// ranges of all tiles' units, equal but for the CTAs that run prologue items
// (pro_d units each), so that every SM has the same work
// whatever the number of tiles. Range starts are moved back to the start of
// a tile when they would fall inside its K-tail, so a tile's K-tail belongs
// to the CTA that holds the tile's first unit (its owner). A range is a
// sequence of segments, one per tile it touches, each run as its W blocks and
// then (the owner's) K-tail blocks, so that u' is needed only late. Only a
// range's first segment can start after its tile's first unit: that CTA
// stores its fp32 partial tile in its own workspace slot and raises its flag.
// Only a range's last segment can be an owner's that stops before its tile's
// end: the owner waits for the flags of the CTAs that follow it (whose first
// segments are the rest of its tile), adds their partials in CTA order from
// shared memory and rounds once. Prologue items and contributors' first
// segments wait for no other CTA, so every wait on another CTA ends.
//
// pre_kernel is the projection on its own (split over K), for the form
// that runs it on a concurrent stream: there the main kernel writes its fp32
// sum, and a K-tail-only launch of it adds alpha B u' after the join.
//
// Warp roles: warp 0 owns the TMEM allocation and issues copies (one thread:
// in the main kernel the packed W; there warp 6 issues the x copies), warp 1
// issues tcgen05.mma (one thread), warps 2-5 dequantise and run the
// epilogues (warp w reads TMEM lanes 32 (w % 4) .. + 31); in the main kernel
// warps 7-10 dequantise the other half of each block's channels. Every mbarrier and
// flag wait is bounded; a timeout latches the handle's status word and the
// CTA runs through its remaining barriers without touching data. The MMA
// thread's loop is on the critical path, so it waits on one barrier per
// stage (TMA bytes and the dequantisers' arrivals together) and commits once,
// and all roles step the stage index by counting.
#include <algorithm>
#include <cstring>

#include "internal.h"
#include "tcgen05.cuh"

namespace spear {
namespace {

constexpr int kThreads = 192;      // pre-kernel: TMA, MMA, four epilogue warps
constexpr int kMainThreads = 352;  // main kernel: W producer, MMA, 4 dequantising + epilogue warps, x producer, 4 dequantising warps
constexpr int kATileBytes = 128 * 128;           // 128 rows x 64 bf16
constexpr int kRawWBytes = 128 * 8 * 4;          // 128 rows x 64 codes, packed
constexpr int kRawBytes = kRawWBytes + 128 * 4;  // plus one scale/zero word per row (one prefill-layout block)
static_assert(kRawBytes == kPrefillBlockWords * 4, "a stage's raw input is one prefill-layout block");
constexpr int kBarrierBytes = 1024;
constexpr int kMaxStages = 6;       // pre-kernel
constexpr int kMaxMainStages = 16;  // main kernel (barrier arrays of 16)
constexpr uint32_t kHintNs = 100;  // suspend-time hint of the pipeline waits
// Main kernel: the accumulator takes columns 0 .. TN - 1 of the 512 TMEM
// columns and stage s's A operand columns tmem_a + 32 s (tmem_a = TN rounded
// up to 32), so small token tiles leave room for more stages.
constexpr int kSlotFloats = 256 * 128;  // one partial tile: [256 columns][128 rows] fp32
// Dynamic shared memory of at least this much keeps a second CTA of either
// kernel off the SM (each allocates tensor memory for the whole launch).
constexpr size_t kOneCtaPerSmBytes = 116 * 1024;

// ------------------------------------------------------------------ params
// The compensator's gate: z [tiles * 128][rank] fp32 -> u' [M][rank] bf16.
struct GateArgs {
  float* zacc;  // fp32 sums of z (rows past M stay zero; cleared after use)
  __nv_bfloat16* u;
  int M, rank;
  int gate;
  float alpha;
  int rank_b;               // column c of u' belongs to member c / rank_b (grouped handle)
  float alphas[kMaxGroup];  // each member's alpha
  const __nv_bfloat16* gw1;  // SPEAR_GATE_MLP: W1 [gh][rank]
  const __nv_bfloat16* gw2;  // SPEAR_GATE_MLP: W2 [rank][gh]
  int gh;
};

struct PreParams {
  int kblocks;   // K blocks of 64 per split
  int kb_total;  // all K blocks (the last split may be shorter)
  int splits;
  unsigned* tile_done;  // per 128-token tile, splits finished
  unsigned* status;
  uint64_t wait_ns;
  int NS;
  uint32_t a_bytes, b_bytes, stage_bytes;
  uint32_t tmem_cols;
  GateArgs ga;
};

struct MainParams {
  int kbt;         // W blocks of 64 channels per tile (0: the K-tail-only launch)
  int tail;        // compensator K-tail blocks per tile
  int kpt;         // work units per tile, tail + kbt
  int nt128;       // tiles of 128 output rows (tile t: row tile t % nt128, token tile t / nt128)
  uint32_t units;  // all tiles' units
  int TN;          // tokens per tile = MMA N (multiple of 16, <= 256)
  int N, M;
  const uint32_t* wq;  // prefill-layout blocks: packed W, then the block's scale/zero words
  __nv_bfloat16* out;  // y [M][N]
  unsigned* status;
  uint64_t wait_ns;
  int skip_arrive;  // test surface: contributors skip raising their flag
  int late_wait;    // u' comes from the pre-kernel launched just before: only the K-tail loads wait for it
  int NS;
  uint32_t tmem_a;  // first TMEM column of the stages' A slots (after the accumulator)
  uint32_t b_bytes, stage_bytes;
  const __nv_bfloat16* bt;  // compensator B rows [nt128 * 128][rank] (the K-tail's A operand)
  int rank;
  float* part;          // [G][kSlotFloats]: each CTA's fp32 partial tile, [column][row]
  unsigned* part_flag;  // [G]: 1 = that CTA's partial tile is stored (reset by its owner)
  // compensator projection as a prologue (0 items: u' is already complete)
  int pro_items;        // items: one per 128-token tile, item i on CTA i mod G
  int pro_d;            // main-contraction units one item stands for in the schedule
  unsigned* u_ready;    // per token tile: 1 = its u' is written
  unsigned* cta_done;   // CTAs finished; the last one clears u_ready
  GateArgs ga;
  // compensator on a concurrent stream: the main contraction writes its fp32
  // result to y32_out [M][N] instead of y; the K-tail launch (no W blocks)
  // adds y32_in [M][N] to its accumulator before the rounding
  float* y32_out;
  const float* y32_in;
};

SPEAR_DEVINL void fail(unsigned* status) { atomicOr(status, kStatusTimeoutPipe); }

SPEAR_DEVINL uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

SPEAR_DEVINL float gate_apply(float z, int gate) {
  return gate == SPEAR_GATE_ONE ? z : z * (1.0f / (1.0f + expf(-z)));
}

SPEAR_DEVINL void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}

SPEAR_DEVINL void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's generic-proxy accesses of global memory with its
// bulk copies (async proxy) on either side of it.
SPEAR_DEVINL void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Bulk copy shared -> global (both 16-byte aligned, bytes a multiple of 16)
// in this thread's bulk group; bulk_commit_wait_all waits until the group's
// writes are complete.
SPEAR_DEVINL void bulk_s2g(void* dst, const void* src, unsigned bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}
SPEAR_DEVINL void bulk_commit_wait_all() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// 32 lanes x 32-bit, 16 consecutive columns per thread, registers -> TMEM.
SPEAR_DEVINL void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// One half of a K block's A operand for row r: channels 32 h .. 32 h + 31
// of the block as 16 bf16 pairs (TMEM columns 16 h .. 16 h + 15 of the
// stage's A slot), from the stage's raw input (words 4 h .. 4 h + 3 of the
// row, then the row's scale/zero word).
SPEAR_DEVINL void dequant_half(uint32_t raw_sa, int r, int h, uint32_t (&v)[16]) {
  const uint4 w = lds128(raw_sa + (uint32_t)(r * 32 + 16 * h));
  const uint32_t szw = lds32(raw_sa + kRawWBytes + r * 4);
  const uint32_t zz = biased_zero_x2(szw >> 16);
  const uint32_t sc = (szw & 0xFFFFu) | (szw << 16);
  const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int j = 0; j < 4; ++j)
      v[4 * c + j] = bf16x2_mul(bf16x2_sub(int4_pair_to_bf16x2_biased(words[c] >> (4 * j)), zz), sc);
}

// The same half of a K-tail block: row a0 + r of the compensator's B,
// columns 64 t + 32 h .. + 31 (zero past rank).
SPEAR_DEVINL void tail_half(const __nv_bfloat16* bt, int rank, int row, int t, int h, uint32_t (&v)[16]) {
  const uint4* src = reinterpret_cast<const uint4*>(bt + (size_t)row * rank + t * 64 + 32 * h);
#pragma unroll
  for (int c8 = 0; c8 < 4; ++c8) {
    const uint4 w = t * 64 + 32 * h + c8 * 8 < rank ? __ldg(src + c8) : make_uint4(0u, 0u, 0u, 0u);
    v[4 * c8] = w.x;
    v[4 * c8 + 1] = w.y;
    v[4 * c8 + 2] = w.z;
    v[4 * c8 + 3] = w.w;
  }
}

// 32 lanes x 32-bit, 32 consecutive columns per thread.
SPEAR_DEVINL void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Named barrier of the 4 epilogue warps; bar.sync counts whole warps, so a
// warp split by a single-thread branch reconverges first.
SPEAR_DEVINL void epilogue_bar() {
  __syncwarp();
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// A bounded wait whose outcome is the same for the whole warp (the tensor
// memory loads and stores that follow are warp-collective).
SPEAR_DEVINL bool warp_wait(uint64_t* bar, unsigned parity, uint64_t limit_ns, uint32_t hint_ns) {
  const bool ok =
      hint_ns ? mbar_wait_bounded_hint(bar, parity, limit_ns, hint_ns) : mbar_wait_bounded(bar, parity, limit_ns);
  return __all_sync(0xffffffffu, ok);
}

// Non-blocking test of an mbarrier phase (the producer's stage is usually
// free long before it is reused: a blocking try_wait cost it ~200 cycles per
// block even then).
SPEAR_DEVINL bool mbar_test_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Spin (bounded) until *flag is nonzero; acquire.
SPEAR_DEVINL bool wait_flag(const unsigned* flag, uint64_t limit_ns) {
  if (ld_acquire_gpu(flag) != 0u) return true;
  const uint64_t t0 = globaltimer();
  while (ld_acquire_gpu(flag) == 0u) {
    if (globaltimer() - t0 > limit_ns) return false;
    __nanosleep(64);
  }
  return true;
}

// z of this 128-token tile (tokens a0 + 32 q + lane: TMEM lane = token,
// column = rank index) added into the fp32 sum.
SPEAR_DEVINL void add_z_partial(const GateArgs& g, uint32_t lane_base, int token) {
  for (int c0 = 0; c0 < g.rank; c0 += 32) {
    uint32_t v[32];
    tmem_ld_x32(lane_base + c0, v);
    tmem_ld_wait();
    if (token < g.M) {
      float* dst = g.zacc + (size_t)token * g.rank + c0;
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        if (c0 + j < g.rank)
          red_add_v4(dst + j, __uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                     __uint_as_float(v[j + 3]));
    }
  }
}

// u' = bf16(alpha gamma(z) (.) z) for the 128-token tile starting at token
// a0, from its z rows in global memory (row stride zst floats, read through
// L2; rows past M are zero). Run by the four epilogue warps, warp q on tokens
// a0 + 32 q .. + 31. The MLP gate reads W1 [gh][rank + 8] and W2
// [rank][gh + 8] from shared memory (stage_mlp_weights).
SPEAR_DEVINL void gate_rows(const GateArgs& g, const float* z, int zst, int a0, int q, int lane,
                            const __nv_bfloat16* w1, const __nv_bfloat16* w2) {
  const int r = g.rank;
  auto ld4 = [&](const float* ptr) { return __ldcg(reinterpret_cast<const float4*>(ptr)); };
  if (g.gate == SPEAR_GATE_MLP) {
    // Bottleneck-MLP gate on warp MMAs (mlp_gate_logits) for the warp's two
    // 16-token blocks: u' = bf16(alpha sigmoid(W2 relu(W1 z)) (.) z).
    for (int tb = 0; tb < 2; ++tb)
      mlp_gate_logits(z, zst, 32 * q + 16 * tb, r, g.gh, w1, r + 8, w2, g.gh + 8, lane, 0, r / 8,
                      [&](int lr, int j, float g0, float g1) {
                        const int m = a0 + lr;
                        if (m >= g.M) return;
                        const float* zr = z + (size_t)lr * zst;
                        const float z0 = __ldcg(zr + j), z1 = __ldcg(zr + j + 1);
                        *reinterpret_cast<uint32_t*>(g.u + (size_t)m * r + j) =
                            pack_bf16x2(g.alpha * z0 * (1.0f / (1.0f + expf(-g0))),
                                        g.alpha * z1 * (1.0f / (1.0f + expf(-g1))));
                      });
    return;
  }
  // Elementwise gate: eight rows per round with all loads in flight; lanes
  // run along the row, 4 columns each.
  for (int r0 = 0; r0 < 32; r0 += 8) {
    for (int c = lane * 4; c < r; c += 128) {
      float4 zv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int lr = 32 * q + r0 + j;
        zv[j] = a0 + lr < g.M ? ld4(z + (size_t)lr * zst + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int m = a0 + 32 * q + r0 + j;
        if (m < g.M) {
          const float al = g.alphas[c / g.rank_b];  // columns c .. c + 3: one member
          const uint2 pk = make_uint2(pack_bf16x2(al * gate_apply(zv[j].x, g.gate), al * gate_apply(zv[j].y, g.gate)),
                                      pack_bf16x2(al * gate_apply(zv[j].z, g.gate), al * gate_apply(zv[j].w, g.gate)));
          *reinterpret_cast<uint2*>(g.u + (size_t)m * r + c) = pk;
        }
      }
    }
  }
}

// The MLP gate's W1 [gh][rank] and W2 [rank][gh] (constant since create) into
// shared memory at dst, rows padded by 8 elements: W1 then W2. By the four
// epilogue warps, which then synchronise. Read from global memory inside the
// gate's MMA loops, each k16 step waited for its own L2 round trip.
SPEAR_DEVINL void stage_mlp_weights(const GateArgs& g, __nv_bfloat16* dst) {
  stage_rows_padded(dst, g.gw1, g.gh, g.rank, threadIdx.x - 64, 128);
  stage_rows_padded(dst + (size_t)g.gh * (g.rank + 8), g.gw2, g.rank, g.gh, threadIdx.x - 64, 128);
  epilogue_bar();
}

// Shared-memory bytes of stage_mlp_weights.
__host__ __device__ inline size_t mlp_weight_bytes(int rank, int gh) {
  return ((size_t)gh * (rank + 8) + (size_t)rank * (gh + 8)) * 2;
}

// The last K split of the 128-token tile starting at token a0 (pre_kernel):
// u' from the fp32 sums of z in global memory, then z cleared for the next
// call. wbuf: free shared memory for the MLP gate's weights.
SPEAR_DEVINL void gate_tile(const GateArgs& g, int a0, int q, int lane, __nv_bfloat16* wbuf) {
  const int r = g.rank;
  if (g.gate == SPEAR_GATE_MLP) stage_mlp_weights(g, wbuf);
  gate_rows(g, g.zacc + (size_t)a0 * r, r, a0, q, lane, wbuf, wbuf + (size_t)g.gh * (r + 8));
  __syncwarp();
  for (int rr = 0; rr < 32; ++rr) {
    const int m = a0 + 32 * q + rr;
    if (m < g.M)
      for (int c = lane * 4; c < r; c += 128)
        *reinterpret_cast<float4*>(g.zacc + (size_t)m * r + c) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ------------------------------------------------------------------ compensator projection on its own
// z [M][rank] (+)= x A^T over this CTA's K split (tokens of tile blockIdx.x,
// K blocks of split blockIdx.y); the last split of the token tile gates z
// into u' and clears z and its counter for the next call.
__global__ void __launch_bounds__(kThreads, 1)
    pre_kernel(const PreParams p, const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapA) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  // full[s] = the stage's x and A tiles have landed; empty[s] = its MMAs completed
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + 16;
  uint64_t* acc_full = full + 24;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 384);
  volatile int& last_split = *reinterpret_cast<volatile int*>(smem + 512);
  uint8_t* stages = smem + kBarrierBytes;
  const uint32_t stages_s = smem_u32(stages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int a0 = blockIdx.x * 128;
  const int kb0 = blockIdx.y * p.kblocks;
  const int total = min(p.kblocks, p.kb_total - kb0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
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
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    if (lane == 0) {
      int s = 0;
      unsigned ph = 0;
      for (int it = 0; it < total; ++it) {
        if (it >= p.NS && !mbar_wait_bounded_hint(&empty[s], ph ^ 1u, p.wait_ns, kHintNs)) {
          fail(p.status);
          break;
        }
        uint8_t* A = stages + (size_t)s * p.stage_bytes;
        mbar_arrive_expect_tx(&full[s], p.a_bytes + p.b_bytes);
        tma_load_2d(A, &mapX, (kb0 + it) * 64, a0, &full[s]);
        tma_load_2d(A + p.a_bytes, &mapA, (kb0 + it) * 64, 0, &full[s]);
        if (++s == p.NS) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, p.ga.rank);
      int s = 0;
      unsigned ph = 0;
      uint32_t a_s = stages_s;
      bool bad = false;
      for (int it = 0; it < total; ++it) {
        if (!mbar_wait_bounded_hint(&full[s], ph, p.wait_ns, kHintNs)) {
          fail(p.status);
          bad = true;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int k16 = 0; k16 < 4; ++k16)
          umma_bf16(tmem_d, sw128_kmajor_desc(a_s + 32 * k16), sw128_kmajor_desc(a_s + p.a_bytes + 32 * k16), idesc,
                    (it | k16) != 0);
        umma_commit(&empty[s]);
        a_s += p.stage_bytes;
        if (++s == p.NS) {
          s = 0;
          ph ^= 1u;
          a_s = stages_s;
        }
      }
      if (!bad) umma_commit(acc_full);  // the accumulator is complete once every MMA above has finished
    }
  } else {
    const int q = warp & 3;
    bool ok = warp_wait(acc_full, 0, 4 * p.wait_ns, 0);
    if (!ok && lane == 0) fail(p.status);
    tc_fence_after_sync();
    if (ok) add_z_partial(p.ga, tmem_d + ((uint32_t)(32 * q) << 16), a0 + 32 * q + lane);
    __threadfence();
    epilogue_bar();
    if (threadIdx.x == 64) {
      last_split = ok && atomicAdd(&p.tile_done[blockIdx.x], 1u) == (unsigned)(p.splits - 1);
      __threadfence();
    }
    epilogue_bar();
    if (last_split) {
      gate_tile(p.ga, a0, q, lane, reinterpret_cast<__nv_bfloat16*>(stages));
      if (threadIdx.x == 64) p.tile_done[blockIdx.x] = 0;
    }
  }

  // single-thread roles leave warps split: reconverge before the CTA barrier
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_d, p.tmem_cols);
}

// ------------------------------------------------------------------ main kernel: schedule
// Prologue items on CTAs 0 .. c - 1 (item i runs on CTA i mod G).
__host__ __device__ inline uint64_t items_before(uint32_t c, uint32_t items, uint32_t G) {
  uint64_t n = 0;
  for (uint64_t k0 = 0; k0 < items; k0 += G) n += min((uint64_t)c, (uint64_t)items - k0);
  return n;
}

// First unit of CTA c's range among G CTAs (c = G: all units). The units
// plus pro_d per prologue item are shared equally, and a CTA's items take
// their part of its share; the start is then moved back to the tile's first
// unit when it would fall inside the tile's K-tail.
__host__ __device__ inline uint32_t range_start_of(const MainParams& p, uint32_t c, uint32_t G) {
  const uint64_t all = (uint64_t)p.units + (uint64_t)p.pro_items * p.pro_d;
  uint32_t b = (uint32_t)(((uint64_t)c * all) / G - items_before(c, (uint32_t)p.pro_items, G) * p.pro_d);
  const uint32_t j = b % (uint32_t)p.kpt;
  if (j != 0 && j < (uint32_t)p.tail) b -= j;
  return b;
}
SPEAR_DEVINL uint32_t range_start(const MainParams& p, uint32_t c) { return range_start_of(p, c, gridDim.x); }

// The part of one tile inside [u, end).
struct Segment {
  int tile;
  int wb0, nw;  // W blocks wb0 .. wb0 + nw - 1
  int ntail;    // K-tail blocks (the owner's: all of them)
  int len;      // units
  bool owner;   // holds the tile's first unit
  bool whole;   // holds all of the tile
};

SPEAR_DEVINL Segment segment_at(const MainParams& p, uint32_t u, uint32_t end) {
  Segment s;
  s.tile = (int)(u / (uint32_t)p.kpt);
  const int j0 = (int)(u - (uint32_t)s.tile * (uint32_t)p.kpt);
  const int j1 = (int)min((uint32_t)p.kpt, (uint32_t)j0 + (end - u));
  s.len = j1 - j0;
  s.owner = j0 == 0;
  s.whole = s.owner && j1 == p.kpt;
  s.wb0 = max(j0, p.tail) - p.tail;
  s.nw = max(j1 - p.tail, s.wb0) - s.wb0;
  s.ntail = s.owner ? p.tail : 0;
  return s;
}

// Columns c0 .. c0 + 31 of output row `row` = a0 + 32 q + lane (x: fp32,
// token b0 + c0 + j) to y (bf16) or to the fp32 result of the
// concurrent-stream form. For y, lanes 2i and 2i + 1 trade half of their
// values so that each stores a 32-bit word of two rows of one token (the
// even lane tokens c0 + 2k, the odd lane tokens c0 + 2k + 1): 16-bit stores
// from every lane ran several times slower. N is a multiple of 8, so a pair
// of rows is either inside y or past its end. All 32 lanes take part.
SPEAR_DEVINL void store_out(const MainParams& p, int row, int b0, int c0, float (&x)[32], int lane) {
  if (p.y32_out != nullptr) {
    if (row < p.N)
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int m = b0 + c0 + j;
        if (c0 + j < p.TN && m < p.M) __stcg(p.y32_out + (size_t)m * p.N + row, x[j]);
      }
    return;
  }
  if (p.y32_in != nullptr && row < p.N)
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int m = b0 + c0 + j;
      if (c0 + j < p.TN && m < p.M) x[j] += __ldcg(p.y32_in + (size_t)m * p.N + row);
    }
  const bool odd = (lane & 1) != 0;
  const int row0 = row & ~1;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float recv = __shfl_xor_sync(0xffffffffu, odd ? x[2 * k] : x[2 * k + 1], 1);
    const float lo = odd ? recv : x[2 * k];      // row0, token c0 + j
    const float hi = odd ? x[2 * k + 1] : recv;  // row0 + 1
    const int j = 2 * k + (odd ? 1 : 0);
    const int m = b0 + c0 + j;
    if (c0 + j < p.TN && m < p.M && row0 < p.N)
      *reinterpret_cast<uint32_t*>(p.out + (size_t)m * p.N + row0) = pack_bf16x2(lo, hi);
  }
}

// ------------------------------------------------------------------ main kernel: producers
// The stages are filled by two threads in different warps, stepping the same
// sequence of K blocks: the W producer (X = false) brings each block's packed
// W and scale/zero words (raw_full[s]; a plain arrival for prologue and
// K-tail blocks), the x producer (X = true) the B operand (full[s]: x, u' or,
// in the prologue, x and the compensator's A). One thread issuing both was
// the pace-setter of the whole kernel (~700 cycles per block against 512 of
// MMA at 256 tokens). Both wait for a stage's MMAs (empty[s]) before
// refilling it, and for each prologue item's epilogue (pro_done), which uses
// the stage memory, before the next item or the main contraction.
template <bool X>
SPEAR_DEVINL void produce(const MainParams& p, const CUtensorMap* mapX, const CUtensorMap* mapU,
                          const CUtensorMap* mapXp, const CUtensorMap* mapA, uint8_t* stages, uint64_t* full,
                          uint64_t* raw_full, uint64_t* empty, uint64_t* pro_done, uint32_t ub, uint32_t ue) {
  const uint32_t pro_a_bytes = kATileBytes;  // prologue stage: x tile, then the A tile
  int s = 0;
  unsigned ph = 0;
  bool waited = !X;
  if (X && !p.late_wait) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    waited = true;
  }
  int it = 0;
  bool bad = false;
  int k = 0;
  for (int item = blockIdx.x; item < p.pro_items && !bad; item += gridDim.x, ++k) {
    if (k > 0 && !mbar_wait_bounded(pro_done, (unsigned)((k - 1) & 1), 8 * p.wait_ns)) {
      fail(p.status);
      bad = true;
      break;
    }
    for (int i = 0; i < p.kbt; ++i, ++it) {
      if (it >= p.NS && !mbar_test_wait(&empty[s], ph ^ 1u) &&
          !mbar_wait_bounded_hint(&empty[s], ph ^ 1u, p.wait_ns, kHintNs)) {
        fail(p.status);
        bad = true;
        break;
      }
      if (X) {
        uint8_t* st = stages + (size_t)s * p.stage_bytes;
        mbar_arrive_expect_tx(&full[s], pro_a_bytes + (uint32_t)p.rank * 128u);
        tma_load_2d(st, mapXp, i * 64, item * 128, &full[s]);
        tma_load_2d(st + pro_a_bytes, mapA, i * 64, 0, &full[s]);
      } else {
        mbar_arrive(&raw_full[s]);
      }
      if (++s == p.NS) {
        s = 0;
        ph ^= 1u;
      }
    }
  }
  if (!bad && k > 0 && !mbar_wait_bounded(pro_done, (unsigned)((k - 1) & 1), 8 * p.wait_ns)) {
    fail(p.status);
    bad = true;
  }
  for (uint32_t u = ub; u < ue && !bad;) {
    const Segment g = segment_at(p, u, ue);
    u += g.len;
    const int rt = g.tile % p.nt128, b0 = (g.tile / p.nt128) * p.TN;
    if (!X && g.ntail > 0) prefetch_l2(p.bt + (size_t)rt * 128 * p.rank, 128u * p.rank * 2u);
    const uint32_t* wsrc = p.wq + ((size_t)rt * p.kbt + g.wb0) * kPrefillBlockWords;
    for (int i = 0; i < g.nw + g.ntail; ++i, ++it) {
      if (it >= p.NS && !mbar_test_wait(&empty[s], ph ^ 1u) &&
          !mbar_wait_bounded_hint(&empty[s], ph ^ 1u, p.wait_ns, kHintNs)) {
        fail(p.status);
        bad = true;
        break;
      }
      uint8_t* B = stages + (size_t)s * p.stage_bytes;
      if (i < g.nw) {
        if (X) {
          mbar_arrive_expect_tx(&full[s], p.b_bytes);
          tma_load_2d(B, mapX, (g.wb0 + i) * 64, b0, &full[s]);
        } else {
          mbar_arrive_expect_tx(&raw_full[s], kRawBytes);
          bulk_g2s(B + p.b_bytes, wsrc, kRawBytes, &raw_full[s]);
          wsrc += kPrefillBlockWords;
        }
      } else if (X) {
        // K-tail block: B = u' of this tile's tokens, once the prologue has
        // written it (or the pre-kernel's grid has completed)
        if (i == g.nw && p.pro_items > 0) {
          const int t_end = min(b0 + p.TN, p.M);
          for (int ti = b0 / 128; ti * 128 < t_end && !bad; ++ti)
            if (!wait_flag(&p.u_ready[ti], 4 * p.wait_ns)) bad = true;
          if (bad) {
            fail(p.status);
            break;
          }
          fence_proxy_async_global();
        }
        if (!waited) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          waited = true;
        }
        mbar_arrive_expect_tx(&full[s], p.b_bytes);
        tma_load_2d(B, mapU, (i - g.nw) * 64, b0, &full[s]);
      } else {
        // K-tail block: the dequantisers read A rows (the compensator's B)
        // from global memory and may fill the stage's A slot from now on
        mbar_arrive(&raw_full[s]);
      }
      if (++s == p.NS) {
        s = 0;
        ph ^= 1u;
      }
    }
  }
}

// ------------------------------------------------------------------ main kernel
// mapX: x tokens (box 64 x TN); mapU: u' (box 64 x TN); mapXp: x tokens for
// the prologue (box 64 x 128); mapA: the compensator's A (box 64 x rank).
__global__ void __launch_bounds__(kMainThreads, 1)
    main_kernel(const MainParams p, const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapU,
                const __grid_constant__ CUtensorMap mapXp, const __grid_constant__ CUtensorMap mapA) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
  // Per stage s: full[s] = the stage's operands are ready for the MMA (B by
  // TMA plus the A operand in tensor memory from the four dequantising
  // warps; prologue: both operands by TMA, the four warps only count in),
  // raw_full[s] = the stage's dequantiser input has landed (packed W block
  // and scale/zero words; for K-tail and prologue blocks a plain arrival),
  // which also says that the stage's A slot is free, since the producer
  // refills a stage only after its MMAs completed, and empty[s] = the MMAs of
  // the stage have completed. acc_full completes one phase per prologue item
  // and per segment; part_bar one per pass over the owner's partials.
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* raw_full = full + kMaxMainStages;
  uint64_t* empty = full + 2 * kMaxMainStages;
  uint64_t* acc_full = full + 3 * kMaxMainStages;
  uint64_t* part_bar = acc_full + 1;
  uint64_t* pro_done = acc_full + 2;  // a prologue item's epilogue is done: the stage memory is free
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 448);
  volatile int& epi_bad = *reinterpret_cast<volatile int*>(smem + 512);  // an epilogue warp gave up
  uint8_t* stages = smem + kBarrierBytes;
  const uint32_t stages_s = smem_u32(stages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ub = range_start(p, blockIdx.x), ue = range_start(p, blockIdx.x + 1);
  const uint32_t pro_a_bytes = kATileBytes;  // prologue stage: x tile, then the A tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.NS; ++s) {
      mbar_init(&full[s], 9);  // the x producer's expect_tx and the eight dequantising warps
      mbar_init(&raw_full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(part_bar, 1);
    mbar_init(pro_done, 1);
    epi_bad = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_d = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // Grid dependencies: only the x producer reads what preceding grids write
  // (x, u', and for the K-tail-only launch y32, which the epilogue reads
  // after MMAs that waited for the x producer's copies); every write of this
  // grid follows such an MMA too. So only the x producer waits for the
  // preceding grid, at its start, and the W producer and the dequantisers
  // fill the first stages' A operands meanwhile. After a separate
  // pre-kernel, which waited for x's producer before it let this grid
  // launch, x can be read at once and the x producer waits only before its
  // first u' load.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    // ---------------------------------------------------------- W producer
    if (lane == 0)
      produce<false>(p, &mapX, &mapU, &mapXp, &mapA, stages, full, raw_full, empty, pro_done, ub, ue);
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, p.TN);
      const uint32_t idesc_pro = idesc_bf16_f32(128, p.rank);
      int s = 0;
      unsigned ph = 0;
      uint32_t b_s = stages_s;
      bool bad = false;
      for (int item = blockIdx.x; item < p.pro_items && !bad; item += gridDim.x) {
        for (int i = 0; i < p.kbt; ++i) {
          if (!mbar_wait_bounded_hint(&full[s], ph, p.wait_ns, kHintNs)) {
            fail(p.status);
            bad = true;
            break;
          }
          tc_fence_after_sync();
          // D [128 tokens][rank] (+)= x A^T, both operands in shared memory
#pragma unroll
          for (int k16 = 0; k16 < 4; ++k16)
            umma_bf16(tmem_d, sw128_kmajor_desc(b_s + 32 * k16), sw128_kmajor_desc(b_s + pro_a_bytes + 32 * k16),
                      idesc_pro, (i | k16) != 0);
          umma_commit(&empty[s]);
          b_s += p.stage_bytes;
          if (++s == p.NS) {
            s = 0;
            ph ^= 1u;
            b_s = stages_s;
          }
        }
        if (!bad) umma_commit(acc_full);
      }
      for (uint32_t u = ub; u < ue && !bad;) {
        const Segment g = segment_at(p, u, ue);
        u += g.len;
        for (int i = 0; i < g.nw + g.ntail; ++i) {
          if (!mbar_wait_bounded_hint(&full[s], ph, p.wait_ns, kHintNs)) {
            fail(p.status);
            bad = true;
            break;
          }
          tc_fence_after_sync();
          // A from tensor memory: 8 columns (16 channels) per k16 step; B's
          // descriptor built once per stage, the k16 step added to its
          // address field (a 32-byte step is 2 in units of 16 bytes; the
          // field holds every shared-memory address, so nothing carries)
          const uint64_t bdesc = sw128_kmajor_desc(b_s);
          const uint32_t a_t = tmem_d + p.tmem_a + 32 * s;
          umma_ts_bf16(tmem_d, a_t, bdesc, idesc, i != 0);
          umma_ts_bf16(tmem_d, a_t + 8, bdesc + 2, idesc, 1u);
          umma_ts_bf16(tmem_d, a_t + 16, bdesc + 4, idesc, 1u);
          umma_ts_bf16(tmem_d, a_t + 24, bdesc + 6, idesc, 1u);
          umma_commit(&empty[s]);
          b_s += p.stage_bytes;
          if (++s == p.NS) {
            s = 0;
            ph ^= 1u;
            b_s = stages_s;
          }
        }
        if (!bad) umma_commit(acc_full);  // this segment's sum is complete once its MMAs have finished
      }
    }
  } else if (warp == 6) {
    // ---------------------------------------------------------- x producer
    if (lane == 0)
      produce<true>(p, &mapX, &mapU, &mapXp, &mapA, stages, full, raw_full, empty, pro_done, ub, ue);
  } else if (warp >= 7) {
    // ---------------------------------------------------------- second-half dequantisers
    // Warps 7-10 convert channels 32 .. 63 of every K block (TMEM columns
    // 16 .. 31 of the stage's A slot) while warps 2-5 convert 0 .. 31: one
    // warp per lane quarter took ~370 cycles a block. They run no epilogue:
    // the MMA thread needs every dequantiser's arrival for a stage, and warps
    // 2-5 arrive for a segment's first block only after its epilogue.
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_base = tmem_d + ((uint32_t)(32 * q) << 16);
    int s = 0;
    unsigned ph = 0;
    uint32_t raw_sa = stages_s + p.b_bytes;
    bool ok = true;
    for (int item = blockIdx.x; item < p.pro_items; item += gridDim.x) {
      for (int i = 0; ok && i < p.kbt; ++i) {
        ok = warp_wait(&raw_full[s], ph, p.wait_ns, kHintNs);
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
        raw_sa += p.stage_bytes;
        if (++s == p.NS) {
          s = 0;
          ph ^= 1u;
          raw_sa = stages_s + p.b_bytes;
        }
      }
    }
    for (uint32_t u = ub; ok && u < ue;) {
      const Segment g = segment_at(p, u, ue);
      u += g.len;
      const int a0 = (g.tile % p.nt128) * 128;
      for (int i = 0; ok && i < g.nw + g.ntail; ++i) {
        uint32_t v[16];
        if (i < g.nw) {
          ok = warp_wait(&raw_full[s], ph, p.wait_ns, kHintNs);
          if (!ok) break;
          dequant_half(raw_sa, r, 1, v);
        } else {
          tail_half(p.bt, p.rank, a0 + r, i - g.nw, 1, v);
          ok = warp_wait(&raw_full[s], ph, p.wait_ns, kHintNs);
          if (!ok) break;
        }
        tc_fence_after_sync();
        tmem_st_x16(lane_base + p.tmem_a + 32 * s + 16, v);
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
        raw_sa += p.stage_bytes;
        if (++s == p.NS) {
          s = 0;
          ph ^= 1u;
          raw_sa = stages_s + p.b_bytes;
        }
      }
    }
    if (!ok && lane == 0) fail(p.status);
  } else {
    // ---------------------------------------------------------- dequantisers + epilogues
    // One thread per row: warp w owns tensor-memory lanes 32 (w % 4) .. + 31,
    // i.e. rows r = 32 (w % 4) + lane of the tile. Per K block a thread reads
    // the first 4 of its row's 8 packed words and its scale/zero word, makes
    // 16 bf16 pairs (pair c = channels 2c, 2c + 1) and stores them as
    // columns 0 .. 15 of the stage's A slot (warps 7-10 do channels 32 .. 63). An epilogue reads the accumulator before these warps
    // arrive for the next segment's first block, so the MMA thread cannot
    // overwrite it early. Every warp runs every item and segment and every epilogue
    // barrier; after a failed wait it only skips the data.
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t lane_base = tmem_d + ((uint32_t)(32 * q) << 16);
    int s = 0;
    unsigned ph = 0;
    uint32_t raw_sa = stages_s + p.b_bytes;
    bool ok = true;
    int si = 0;  // acc_full phases consumed
    // Prologue items: token tile ti's z = x A^T over all of K is in tensor
    // memory (lane = token, column = rank index). Gate it there and build
    // the u' rows of the tile in shared memory (the MLP gate first stages z
    // rows [128][rank + 8] there), then write them with one bulk copy and
    // raise the tile's flag. The producer loads the next item, or starts the
    // main contraction, only after this epilogue's pro_done arrival, so the
    // stage memory is free here once the item's MMAs have completed.
    const int zst = p.rank + 8;
    float* zrows = reinterpret_cast<float*>(stages);
    __nv_bfloat16* utile = reinterpret_cast<__nv_bfloat16*>(
        stages + (p.ga.gate == SPEAR_GATE_MLP ? (size_t)128 * zst * 4 : (size_t)0));
    for (int item = blockIdx.x; item < p.pro_items; item += gridDim.x, ++si) {
      const int ti = item;
      const int a0t = ti * 128;
      for (int i = 0; ok && i < p.kbt; ++i) {
        ok = warp_wait(&raw_full[s], ph, p.wait_ns, kHintNs);
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
        raw_sa += p.stage_bytes;
        if (++s == p.NS) {
          s = 0;
          ph ^= 1u;
          raw_sa = stages_s + p.b_bytes;
        }
      }
      if (ok) ok = warp_wait(acc_full, (unsigned)(si & 1), 4 * p.wait_ns, 0);
      if (!ok && lane == 0) fail(p.status);
      tc_fence_after_sync();
      if (ok) {
        const GateArgs& g = p.ga;
        for (int c0 = 0; c0 < p.rank; c0 += 32) {
          uint32_t v[32];
          tmem_ld_x32(lane_base + c0, v);
          tmem_ld_wait();
          if (g.gate == SPEAR_GATE_MLP) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c0 + j < p.rank) zrows[r * zst + c0 + j] = __uint_as_float(v[j]);
          } else {
            // u'[token r][c0 .. c0 + 31] = bf16(alpha gamma(z) z), 16 bytes at a time
#pragma unroll
            for (int j8 = 0; j8 < 4; ++j8) {
              const int c = c0 + 8 * j8;
              if (c < p.rank) {
                const float al = g.alphas[c / g.rank_b];  // columns c .. c + 7: one member
                uint32_t pk[4];
#pragma unroll
                for (int h = 0; h < 4; ++h)
                  pk[h] = pack_bf16x2(al * gate_apply(__uint_as_float(v[8 * j8 + 2 * h]), g.gate),
                                      al * gate_apply(__uint_as_float(v[8 * j8 + 2 * h + 1]), g.gate));
                *reinterpret_cast<uint4*>(utile + (size_t)r * p.rank + c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              }
            }
          }
        }
        if (g.gate == SPEAR_GATE_MLP) {
          // warp q's z rows are its own: gate its two 16-token blocks on warp
          // MMAs, W1 and W2 staged after the u' rows
          __nv_bfloat16* w1 = utile + (size_t)128 * p.rank;
          stage_mlp_weights(g, w1);
          const __nv_bfloat16* w2 = w1 + (size_t)g.gh * (p.rank + 8);
          for (int tb = 0; tb < 2; ++tb)
            mlp_gate_logits(zrows, zst, 32 * q + 16 * tb, p.rank, g.gh, w1, p.rank + 8, w2, g.gh + 8, lane, 0,
                            p.rank / 8, [&](int lr, int j, float g0, float g1) {
                              const float* zr = zrows + lr * zst;
                              *reinterpret_cast<uint32_t*>(utile + (size_t)lr * p.rank + j) =
                                  pack_bf16x2(g.alpha * zr[j] * (1.0f / (1.0f + expf(-g0))),
                                              g.alpha * zr[j + 1] * (1.0f / (1.0f + expf(-g1))));
                            });
        }
      }
      if (!ok) epi_bad = 1;
      epilogue_bar();
      if (threadIdx.x == 64 && epi_bad == 0) {
        // the tile's u' rows (those below M) in one bulk copy, then the flag
        const int rows = min(128, p.M - a0t);
        fence_proxy_async_smem();
        bulk_s2g(p.ga.u + (size_t)a0t * p.rank, utile, (unsigned)(rows * p.rank * 2));
        bulk_commit_wait_all();
        fence_proxy_async_global();
        st_release_gpu(&p.u_ready[ti], 1u);
      }
      epilogue_bar();  // the bulk copy has read the tile: the stage memory is free again
      if (threadIdx.x == 64) {
        fence_proxy_async_smem();  // the stage memory's generic use above ends before the producer's copies
        mbar_arrive(pro_done);
      }
    }
    ok = ok && epi_bad == 0;
    for (uint32_t u = ub; u < ue; ++si) {
      const Segment g = segment_at(p, u, ue);
      u += g.len;
      const int rt = g.tile % p.nt128, a0 = rt * 128, b0 = (g.tile / p.nt128) * p.TN;
      for (int i = 0; ok && i < g.nw + g.ntail; ++i) {
        uint32_t v[16];
        if (i < g.nw) {
          ok = warp_wait(&raw_full[s], ph, p.wait_ns, kHintNs);
          if (!ok) break;
          dequant_half(raw_sa, r, 0, v);
        } else {
          tail_half(p.bt, p.rank, a0 + r, i - g.nw, 0, v);
          ok = warp_wait(&raw_full[s], ph, p.wait_ns, kHintNs);
          if (!ok) break;
        }
        // the block counts towards full[s] once its store has completed
        // (deferring that until the next block was converted, to overlap the
        // store, made the MMA wait for the next block's input)
        tc_fence_after_sync();
        tmem_st_x16(lane_base + p.tmem_a + 32 * s, v);
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
        raw_sa += p.stage_bytes;
        if (++s == p.NS) {
          s = 0;
          ph ^= 1u;
          raw_sa = stages_s + p.b_bytes;
        }
      }
      if (!ok && lane == 0) fail(p.status);

      // ------------------------------------------------------ epilogue of the segment
      if (ok) {
        ok = warp_wait(acc_full, (unsigned)(si & 1), 4 * p.wait_ns, 0);
        if (!ok && lane == 0) fail(p.status);
      }
      tc_fence_after_sync();
      const int row = a0 + r;
      if (!g.owner) {
        // A tile's later units: store the fp32 partial ([column][row]: a
        // warp's 32 rows of one column are 128 contiguous bytes), then raise
        // this CTA's flag for the owner.
        float* dst = p.part + (size_t)blockIdx.x * kSlotFloats + r;
        for (int c0 = 0; ok && c0 < p.TN; c0 += 32) {
          uint32_t v[32];
          tmem_ld_x32(lane_base + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c0 + j < p.TN) __stcg(dst + (size_t)(c0 + j) * 128, __uint_as_float(v[j]));
        }
        if (!ok) epi_bad = 1;
        __threadfence();
        epilogue_bar();
        if (threadIdx.x == 64 && epi_bad == 0 && !p.skip_arrive) st_release_gpu(&p.part_flag[blockIdx.x], 1u);
      } else if (g.whole) {
        for (int c0 = 0; ok && c0 < p.TN; c0 += 32) {
          uint32_t v[32];
          tmem_ld_x32(lane_base + c0, v);
          tmem_ld_wait();
          float x[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
          store_out(p, row, b0, c0, x, lane);
        }
      } else {
        // Owner of a tile whose later units other CTAs ran (this is the last
        // segment of the range, so the stage memory is idle): wait for their
        // flags, bring their partials into the stage memory with bulk copies,
        // in passes of `w` columns when they do not fit at once, and add them
        // in CTA order to this CTA's sum before the single rounding.
        const uint32_t tile_end = (uint32_t)(g.tile + 1) * (uint32_t)p.kpt;
        int n = 0;
        while (blockIdx.x + 1 + n < gridDim.x && range_start(p, blockIdx.x + 1 + n) < tile_end) ++n;
        if (!ok) epi_bad = 1;
        epilogue_bar();
        if (threadIdx.x == 64) {
          bool got = epi_bad == 0;
          for (int z = 1; got && z <= n; ++z) got = wait_flag(&p.part_flag[blockIdx.x + z], 4 * p.wait_ns);
          if (got) {
            for (int z = 1; z <= n; ++z) p.part_flag[blockIdx.x + z] = 0u;  // for the next call
            fence_proxy_async_global();
            fence_proxy_async_smem();
          } else if (epi_bad == 0) {
            fail(p.status);
          }
          if (!got) epi_bad = 1;
        }
        epilogue_bar();
        ok = epi_bad == 0;
        const int tnr = (p.TN + 31) / 32 * 32;
        int w = n > 0 ? min(tnr, (int)(((uint32_t)p.NS * p.stage_bytes) / ((uint32_t)n * 512u)) / 32 * 32) : tnr;
        if (w < 32) {  // the launch keeps 32 columns of every owner's partials within the stage memory
          if (threadIdx.x == 64) fail(p.status);
          ok = false;
          w = tnr;
        }
        int pass = 0;
        for (int cp = 0; cp < tnr; cp += w, ++pass) {
          const int wc = min(w, tnr - cp);
          if (threadIdx.x == 64 && ok) {
            mbar_arrive_expect_tx(part_bar, (unsigned)(n * wc * 512));
            for (int z = 0; z < n; ++z)
              bulk_g2s(stages + (size_t)z * wc * 512,
                       p.part + (size_t)(blockIdx.x + 1 + z) * kSlotFloats + (size_t)cp * 128, (unsigned)(wc * 512),
                       part_bar);
          }
          if (ok) {
            ok = warp_wait(part_bar, (unsigned)(pass & 1), 4 * p.wait_ns, 0);
            if (!ok && lane == 0) fail(p.status);
          }
          for (int c0 = cp; ok && c0 < cp + wc; c0 += 32) {
            uint32_t v[32];
            tmem_ld_x32(lane_base + c0, v);
            tmem_ld_wait();
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
            for (int z = 0; z < n; ++z) {
              const uint32_t ps = stages_s + (uint32_t)(((z * wc + (c0 - cp)) * 128 + r) * 4);
#pragma unroll
              for (int j = 0; j < 32; ++j) x[j] += __uint_as_float(lds32(ps + (uint32_t)(j * 512)));
            }
            store_out(p, row, b0, c0, x, lane);
          }
          epilogue_bar();  // every warp is done with this pass's partials
        }
      }
    }
  }

  // single-thread roles leave warps split: reconverge before the CTA barrier
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_d, 512);
  // The last CTA to finish clears the "u' ready" flags for the next call
  // (every reader has finished; the next launch waits for this grid).
  if (p.pro_items > 0 && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.cta_done, 1u) == gridDim.x - 1) {
      for (int i = 0; i < p.pro_items; ++i) p.u_ready[i] = 0u;
      *p.cta_done = 0u;
      __threadfence();
    }
  }
}

uint32_t tmem_cols_for(int n) {
  uint32_t c = 32;
  while (c < (uint32_t)n) c <<= 1;
  return c;
}

template <typename Kernel, typename Params, typename... Maps>
cudaError_t launch(Kernel k, int threads, std::atomic<uint64_t>& configured, const Params& p, dim3 grid, size_t smem,
                   cudaStream_t st, const Maps&... maps) {
  cudaError_t e = smem_limit_once(reinterpret_cast<const void*>(k), configured);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p, maps...);
}

// Stages that fit next to the barriers.
int stages_for(uint32_t stage_bytes, int max_stages = kMaxStages) {
  const size_t budget = 227 * 1024 - kBarrierBytes - 1024;
  int ns = (int)(budget / stage_bytes);
  return ns > max_stages ? max_stages : ns;
}

uint32_t host_range_start(const MainParams& p, uint32_t c, uint32_t G) { return range_start_of(p, c, G); }

// Every range of a grid of G CTAs is non-empty.
bool ranges_nonempty(const MainParams& p, uint32_t G) {
  for (uint32_t c = 0; c < G; ++c)
    if (host_range_start(p, c + 1, G) <= host_range_start(p, c, G)) return false;
  return true;
}

// Most partial tiles one owner adds under a grid of G CTAs.
int max_contributors(const MainParams& p, uint32_t G) {
  int worst = 0;
  for (uint32_t c = 0; c < G; ++c) {
    const uint32_t b = host_range_start(p, c, G), e = host_range_start(p, c + 1, G);
    if (e % (uint32_t)p.kpt == 0) continue;                     // the range ends at a tile boundary
    const uint32_t ts = e / (uint32_t)p.kpt * (uint32_t)p.kpt;  // start of the tile it ends in
    if (ts < b) continue;                                       // it holds no tile start there
    int n = 0;
    while (c + 1 + n < G && host_range_start(p, c + 1 + n, G) < ts + (uint32_t)p.kpt) ++n;
    worst = std::max(worst, n);
  }
  return worst;
}

GateArgs gate_args(const spear_linear_s* h, int M) {
  GateArgs g{};
  g.zacc = h->z_pre;
  g.u = h->u_pre;
  g.M = M;
  g.rank = h->rank;
  g.gate = h->gate;
  g.alpha = h->alpha;
  g.rank_b = h->rank_b;
  for (int i = 0; i < h->n_members; ++i) g.alphas[i] = h->alphas[i];
  g.gw1 = h->gate_w1;
  g.gw2 = h->gate_w2;
  g.gh = h->gate_hidden;
  return g;
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

// K splits of the pre-kernel: about 32 CTAs of at least 8 K blocks each.
static int pre_splits(int K, int M) {
  const int kbt = K / 64, mt = (M + 127) / 128;
  int splits = (32 + mt - 1) / mt;
  if (splits > kbt / 8) splits = kbt / 8;
  if (splits < 1) splits = 1;
  const int kblocks = (kbt + splits - 1) / splits;
  return (kbt + kblocks - 1) / kblocks;
}

// The compensator projection on its own: u' [M][rank] = bf16(alpha gamma(A x) (.) A x).
static spear_status_t launch_pre(spear_linear_s* h, const __nv_bfloat16* x, int M, cudaStream_t stream,
                                 int* pre_ctas) {
  static std::atomic<uint64_t> configured{0};  // devices whose shared-memory limit is raised
  const int K = h->K, r = h->rank;
  CUtensorMap mx, ma;
  if (!encode_2d_bf16(&mx, x, K, M, (uint64_t)K * 2, 64, 128) ||
      !encode_2d_bf16(&ma, h->a_pre, K, r, (uint64_t)K * 2, 64, r))
    return SPEAR_ERR_CUDA;
  PreParams p{};
  const int kbt = K / 64, mt = (M + 127) / 128;
  int splits = pre_splits(K, M);
  p.kblocks = (kbt + splits - 1) / splits;
  splits = (kbt + p.kblocks - 1) / p.kblocks;
  p.kb_total = kbt;
  p.splits = splits;
  p.tile_done = h->pre_done;
  p.status = &h->sync->status;
  p.wait_ns = h->wait_ns;
  p.a_bytes = kATileBytes;
  p.b_bytes = (uint32_t)(r * 128 + 1023) / 1024 * 1024;
  p.stage_bytes = p.a_bytes + p.b_bytes;
  p.NS = stages_for(p.stage_bytes);
  p.tmem_cols = tmem_cols_for(r);
  p.ga = gate_args(h, M);
  const size_t smem = std::max(kBarrierBytes + 1024 + (size_t)p.NS * p.stage_bytes, kOneCtaPerSmBytes);
  *pre_ctas = mt * splits;
  const cudaError_t e = launch(pre_kernel, kThreads, configured, p, dim3(mt, splits), smem, stream, mx, ma);
  return e == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}

// The main kernel's launch plan (host only): the schedule fields of p, the
// grid G and the dynamic shared memory. mode as for launch_main; r the rank
// the launch uses (0 for mode 1); gh the MLP gate's hidden width (0 for the
// elementwise gates); pre_ctas the SMs a preceding pre-kernel holds;
// has_part whether the handle has the stream-K partial workspace.
static spear_status_t plan_main(MainParams& p, int& G, size_t& smem, int K, int N, int nt128, int r, int gh,
                                int M, int mode, int sm_count, int pre_ctas, bool has_part) {
  const int TN = prefill_tn(M);
  const bool prologue = mode == 0 && r > 0;
  p.kbt = mode == 2 ? 0 : K / 64;
  p.tail = (r + 63) / 64;
  p.kpt = p.kbt + p.tail;
  p.nt128 = nt128;
  const int tiles = nt128 * ((M + TN - 1) / TN);
  const uint64_t units = (uint64_t)tiles * p.kpt;
  if (units >= (1ull << 31)) return SPEAR_ERR_UNSUPPORTED;
  p.units = (uint32_t)units;
  p.TN = TN;
  p.N = N;
  p.M = M;
  p.late_wait = mode == 3 && r > 0;
  p.rank = r;
  p.b_bytes = (uint32_t)(TN * 128 + 1023) / 1024 * 1024;
  uint32_t stage = (p.b_bytes + kRawBytes + 1023) / 1024 * 1024;
  if (prologue) stage = std::max<uint32_t>(stage, kATileBytes + (uint32_t)(r * 128 + 1023) / 1024 * 1024);
  p.stage_bytes = stage;
  p.tmem_a = (uint32_t)(TN + 31) / 32 * 32;
  p.NS = stages_for(p.stage_bytes, std::min<int>(kMaxMainStages, (int)(512 - p.tmem_a) / 32));
  // CTAs: one per tile for the K-tail-only launch and for handles without a
  // partial workspace (sized for decode token counts). Otherwise every SM,
  // with at least max(8, tail + 2, kpt / 3) units each (so that every range
  // is non-empty and an owner adds few partials), and fewer where an owner's
  // partials would not fit its stage memory 32 columns at a time.
  const bool stream_k = has_part && p.kbt > 0;
  const uint64_t area = (uint64_t)p.NS * p.stage_bytes;
  G = tiles;
  if (stream_k) {
    const uint64_t lmin = std::max<uint64_t>({8, (uint64_t)p.tail + 2, (uint64_t)(p.kpt + 2) / 3});
    G = (int)std::min<uint64_t>((uint64_t)std::max(1, sm_count - pre_ctas), units / lmin);
    if (G < 1) G = 1;
  }
  for (;;) {
    if (prologue) {
      // One item per 128-token tile. Its weight in main-contraction units:
      // its loads against a unit's (measured: CTAs with an item then finish
      // with the others; half of that left them 7 us late).
      p.pro_items = (M + 127) / 128;
      const uint32_t pro_bytes = kATileBytes + (uint32_t)r * 128u, unit_bytes = p.b_bytes + kRawBytes;
      p.pro_d = stream_k ? (int)((uint64_t)p.kbt * pro_bytes / unit_bytes) + 2 : 0;
      if (stream_k && !ranges_nonempty(p, (uint32_t)G)) p.pro_d = 0;
    }
    if (!stream_k || G == 1 ||
        (ranges_nonempty(p, (uint32_t)G) && (uint64_t)max_contributors(p, (uint32_t)G) * 32 * 512 <= area))
      break;
    --G;
  }
  smem = std::max(kBarrierBytes + 1024 + (size_t)p.NS * p.stage_bytes, kOneCtaPerSmBytes);
  if (prologue) {
    // an item's u' rows [128][rank] bf16 (the MLP gate: after z rows [128][rank + 8]
    // fp32, and followed by the gate's weights)
    const size_t need = (size_t)128 * r * 2 + (gh > 0 ? (size_t)128 * (r + 8) * 4 + mlp_weight_bytes(r, gh) : 0);
    smem = std::max(smem, kBarrierBytes + 1024 + need);
  }
  return SPEAR_OK;
}

// Main kernel. mode 0: compensator prologue, W x and the K-tail, bf16 y;
// mode 1: W x only, fp32 result into h->y32, next to the pre-kernel on
// another stream (pre_ctas SMs); mode 2: the K-tail only (u' complete), added
// to h->y32, bf16 y; mode 3: W x and the K-tail with u' from the pre-kernel
// launched just before on the same stream, which runs on pre_ctas SMs.
static spear_status_t launch_main(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                  cudaStream_t stream, int mode, int pre_ctas) {
  static std::atomic<uint64_t> configured{0};
  const int K = h->K, N = h->N;
  const int r = mode == 1 ? 0 : h->rank;
  const int TN = prefill_tn(M);
  CUtensorMap mx, mu, mxp, ma;
  memset(&mu, 0, sizeof mu);
  memset(&mxp, 0, sizeof mxp);
  memset(&ma, 0, sizeof ma);
  if (!encode_2d_bf16(&mx, x, K, M, (uint64_t)K * 2, 64, TN)) return SPEAR_ERR_CUDA;
  if (r > 0 && !encode_2d_bf16(&mu, h->u_pre, r, M, (uint64_t)r * 2, 64, TN)) return SPEAR_ERR_CUDA;
  const bool prologue = mode == 0 && r > 0;
  if (prologue && (!encode_2d_bf16(&mxp, x, K, M, (uint64_t)K * 2, 64, 128) ||
                   !encode_2d_bf16(&ma, h->a_pre, K, r, (uint64_t)K * 2, 64, r)))
    return SPEAR_ERR_CUDA;
  MainParams p{};
  int G = 0;
  size_t smem = 0;
  const spear_status_t ps = plan_main(p, G, smem, K, N, h->nt128, r, h->gate == SPEAR_GATE_MLP ? h->gate_hidden : 0, M, mode, h->sm_count,
                                      pre_ctas, h->part != nullptr);
  if (ps != SPEAR_OK) return ps;
  p.wq = h->wq_pre;
  p.out = y;
  p.status = &h->sync->status;
  p.wait_ns = h->wait_ns;
  p.skip_arrive = h->skip_arrive;
  p.bt = h->b_pre;
  p.part = h->part;
  p.part_flag = h->part_cnt;
  p.u_ready = h->u_ready;
  p.cta_done = h->pf_done;
  p.ga = gate_args(h, M);
  p.y32_out = mode == 1 ? h->y32 : nullptr;
  p.y32_in = mode == 2 ? h->y32 : nullptr;
  const cudaError_t e = launch(main_kernel, kMainThreads, configured, p, dim3(G), smem, stream, mx, mu, mxp, ma);
  return e == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}

// The projection goes into the main kernel's prologue when an item (one
// 128-token tile over all of K) weighs at most 3/4 of a CTA's share of the
// main contraction; otherwise the item would be the critical path of a short
// contraction, and a separate split-K pre-kernel runs first. (Measured on
// the mixed step's shapes: at 576 tokens the 4096 x 4096 and 11008 -> 4096
// projections ran 30% faster with the pre-kernel, 4096 -> 11008 20% slower.)
static bool prologue_pays(int K, int nt128, int rank, int gh, int M, int sm_count, bool has_part) {
  if (!has_part) return false;
  // an item's epilogue buffers (u' rows; the MLP gate's z rows and weights) fit
  const size_t need = (size_t)128 * rank * 2 + (gh > 0 ? (size_t)128 * (rank + 8) * 4 + mlp_weight_bytes(rank, gh) : 0);
  if (kBarrierBytes + 1024 + need > (size_t)227 * 1024) return false;
  const int TN = prefill_tn(M), kbt = K / 64;
  const uint64_t tiles = (uint64_t)nt128 * ((M + TN - 1) / TN);
  const uint64_t share = tiles * (kbt + (rank + 63) / 64) / (uint64_t)sm_count;
  const uint64_t unit_bytes = (uint64_t)(TN * 128 + 1023) / 1024 * 1024 + kRawBytes;
  const uint64_t pro_d = (uint64_t)kbt * (kATileBytes + (uint64_t)rank * 128) / unit_bytes + 2;
  return 4 * pro_d <= 3 * share;
}

spear_status_t spear_launch_prefill(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                    cudaStream_t stream) {
  if (h->rank > 0 && !prologue_pays(h->K, h->nt128, h->rank, h->gate == SPEAR_GATE_MLP ? h->gate_hidden : 0, M,
                                    h->sm_count, h->part != nullptr)) {
    int pre_ctas = 0;
    const spear_status_t st = launch_pre(h, x, M, stream, &pre_ctas);
    if (st != SPEAR_OK) return st;
    return launch_main(h, x, y, M, stream, 3, pre_ctas);
  }
  return launch_main(h, x, y, M, stream, 0, 0);
}

// The compensator on a concurrent stream (the pages' semi-fused prefill): the
// projection runs on ec_stream next to the main contraction on `stream`,
// which writes fp32; after the join, the K-tail launch adds alpha B u' and
// rounds.
spear_status_t spear_launch_prefill_concurrent(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                               cudaStream_t stream, cudaStream_t ec_stream) {
  if (h->rank == 0) return spear_launch_prefill(h, x, y, M, stream);
  if (cudaEventRecord(h->ev_fork, stream) != cudaSuccess || cudaStreamWaitEvent(ec_stream, h->ev_fork, 0) != cudaSuccess)
    return SPEAR_ERR_CUDA;
  int pre_ctas = 0;
  spear_status_t st = launch_pre(h, x, M, ec_stream, &pre_ctas);
  if (st != SPEAR_OK) return st;
  // the main contraction leaves the pre-kernel's SMs free: its stream-K
  // owners wait for later CTAs, which must all be resident
  st = launch_main(h, x, y, M, stream, 1, pre_ctas);
  if (st != SPEAR_OK) return st;
  if (cudaEventRecord(h->ev_join, ec_stream) != cudaSuccess || cudaStreamWaitEvent(stream, h->ev_join, 0) != cudaSuccess)
    return SPEAR_ERR_CUDA;
  return launch_main(h, x, y, M, stream, 2, 0);
}

// Test surface: the prefill launch plan of a handle of this shape, computed
// by the same host code as the launch (no device work).
spear_status_t spear_prefill_schedule(int32_t N, int32_t K, int32_t rank, int32_t gate_hidden, int32_t M,
                                      int32_t sm_count, int32_t with_workspace, int32_t* info, uint32_t* starts,
                                      int32_t starts_cap) {
  if (N <= 0 || K <= 0 || K % 64 != 0 || rank < 0 || rank > 256 || M < 1 || sm_count < 1 || !info || gate_hidden < 0 ||
      gate_hidden > kMaxGateHidden || gate_hidden % 16 != 0)
    return SPEAR_ERR_INVALID_ARG;
  const int nt128 = (N + 127) / 128;
  const bool has_part = with_workspace != 0;
  int mode = 0, pre_ctas = 0;
  if (rank > 0 && !prologue_pays(K, nt128, rank, gate_hidden, M, sm_count, has_part)) {
    mode = 3;
    pre_ctas = ((M + 127) / 128) * pre_splits(K, M);
  }
  MainParams p{};
  int G = 0;
  size_t smem = 0;
  const spear_status_t st = plan_main(p, G, smem, K, N, nt128, rank, gate_hidden, M, mode, sm_count, pre_ctas, has_part);
  if (st != SPEAR_OK) return st;
  const int32_t v[14] = {mode, G, p.TN, p.kpt, p.tail, (int32_t)p.units, p.pro_items, p.pro_d, p.NS,
                         (int32_t)p.stage_bytes, (int32_t)smem, pre_ctas, (int32_t)p.tmem_a,
                         max_contributors(p, (uint32_t)G)};
  for (int i = 0; i < 14; ++i) info[i] = v[i];
  if (starts) {
    if (starts_cap < G + 1) return SPEAR_ERR_INVALID_ARG;
    for (int c = 0; c <= G; ++c) starts[c] = host_range_start(p, (uint32_t)c, (uint32_t)G);
  }
  return SPEAR_OK;
}
