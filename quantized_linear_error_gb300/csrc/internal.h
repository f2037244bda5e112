// Handle layout and internal launch interfaces shared by the .cu files of the
// library (not part of the public ABI).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/spear.h"
#include "common.cuh"

// Kernel-side weight layouts (built once by spear_linear_create):
//
// Decode layout (warp MMA m16n8k16 fragments). Rows are grouped in tiles of
// 16. For a tile and a block of 64 input channels, lane l = 4g + t holds one
// uint4 (a 512-byte "k64 block" per tile); word s (k16 step s of the block)
// packs the eight codes that lane feeds to the MMA A fragment, nibble i at
// bits 4i..4i+3:
//   i: 0 (g, 2t)  1 (g+8, 2t)  2 (g, 2t+8)  3 (g+8, 2t+8)
//      4 (g, 2t+1) 5 (g+8, 2t+1) 6 (g, 2t+9) 7 (g+8, 2t+9)
// (row within the tile, k within the 16-step), so (w >> 4j) & 0x000F000F
// yields A-fragment register j as a bf16 pair. Scale/zero words are u32:
// bits 0..15 bf16 scale, 16..31 bf16(128 + zero), one 64-byte block of 16 rows
// per (tile, group).
//
// The blocks are ordered for the decode kernel's schedule, fixed at create:
// CTA c owns tiles [c*P, c*P + P) (nt16 is padded to a whole number of
// CTAs with zero tiles: rows past N, scale 0) and reads K in runs of 256 channels;
// everything one CTA needs for one run is contiguous,
//   [W: Pc tiles x kcw/64 k64 blocks][S: Pc tiles x kcw/128 group blocks]
// (kcw = channels in the run, 256 except maybe the last; S absent for
// per-channel scales), and a CTA's runs follow each other in K order, so a
// pipeline stage of any whole number of runs is a single bulk copy.
//   wq_dec  bytes, nt16 * dec_tile_bytes
//   sz_dec  u32 [nt16][16] (per-channel only)
//   a_dec   uint4 [rank/16][K/16][32]    A in A-fragment order (bf16 pairs), the 16 columns
//                                         of a k16 step in quad order (lane t: 4t .. 4t + 3)
//   b_dec   uint4 [nt16][rank/16][32]    B in A-fragment order (bf16 pairs)
//
// Prefill layout (row-major 16-byte chunks for the tensor-core tile loader).
// Rows are grouped in tiles of 128; for a tile and a block of 64 channels the
// 4 KB block holds, per row, eight u32 words; word c packs channels
// 8c .. 8c+7 with nibble order (0, 2, 4, 6, 1, 3, 5, 7) so that
// (w >> 4j) & 0x000F000F yields channels (2j, 2j+1) as a bf16 pair. The
// block's 128 scale/zero words (same encoding as sz_dec, of the group that
// holds the block) follow it, so one bulk copy brings a block's input.
//   wq_pre  u32   [nt128][K/64][1024 + 128]
//   a_pre   bf16  [rank][K]               copy of A
//   b_pre   bf16  [nt128*128][rank]       copy of B, zero rows past N

constexpr int kMaxGroup = 8;  // linears fused into one grouped handle, at most

struct spear_linear_s {
  int device = 0, sm_count = 0;
  int K = 0, N = 0, G = 0, n_groups = 0, rank = 0, max_tokens = 0;
  float alpha = 1.f;
  // Grouped handle (spear_linear_create_grouped): n_members linears sharing x,
  // rows [row_start[i], row_start[i + 1]) of y belong to member i. `rank` is
  // the stacked rank of all members' A (the projection and gate run over all
  // of it); member i's up-projection uses u columns [i rank_b, (i + 1) rank_b)
  // and its own alpha. An ordinary handle is a group of one.
  int n_members = 1, rank_b = 0;
  int row_start[kMaxGroup + 1] = {};
  float alphas[kMaxGroup] = {};
  int gate = 0;
  bool per_channel = false;

  int nt16 = 0, nt128 = 0;  // decode tiles of 16 rows (padded to whole CTAs), prefill tiles of 128
  // decode schedule (see the layout comment)
  int dec_P = 0;
  size_t dec_tile_bytes = 0;  // one tile over all of K: W blocks plus (grouped) scale blocks
  uint8_t* wq_dec = nullptr;
  uint32_t* sz_dec = nullptr;
  uint4* a_dec = nullptr;
  uint4* b_dec = nullptr;
  uint32_t* wq_pre = nullptr;
  __nv_bfloat16* a_pre = nullptr;
  __nv_bfloat16* b_pre = nullptr;

  // Workspace: SyncWords followed by z [256][32] fp32 (decode), then the
  // prefill buffers.
  void* ws = nullptr;
  spear::SyncWords* sync = nullptr;
  float* z_dec = nullptr;
  float* z_mma = nullptr;            // warp-MMA decode: z [2][256][32] fp32, alternating by call
  float* part = nullptr;             // prefill stream-K schedule: one fp32 partial tile per CTA, [sm_count][256][128]
  unsigned* part_cnt = nullptr;      // prefill stream-K schedule: [sm_count] flags, 1 = that CTA's partial is stored
  float* z_pre = nullptr;            // [ceil(max_tokens / 128) * 128][rank] fp32 (prefill projection; rows past M zero)
  __nv_bfloat16* u_pre = nullptr;    // [max_tokens][rank] bf16 (prefill gated, alpha-scaled)
  unsigned* pre_done = nullptr;      // [ceil(max_tokens / 128)] K splits of the projection finished per token tile
  unsigned* u_ready = nullptr;       // [ceil(max_tokens / 128)] 1 = that token tile's u' is written (prefill)
  unsigned* pf_done = nullptr;       // prefill main kernel: CTAs finished (the last clears u_ready)
  int gate_hidden = 0;               // SPEAR_GATE_MLP: hidden width h8 = h rounded up to 8
  __nv_bfloat16* gate_w1 = nullptr;  // SPEAR_GATE_MLP: W1 [h8][rank], rows h.. zero
  __nv_bfloat16* gate_w2 = nullptr;  // SPEAR_GATE_MLP: W2 [rank][h8], columns h.. zero
  size_t ws_bytes = 0;               // workspace size (zeroed at create and by a TIMEOUT check)
  // compensator on a concurrent stream (spear_linear_enable_concurrent_ec):
  // fp32 main result [max_tokens][N] and the fork / join events
  float* y32 = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // host-buffer batches: copy streams (inputs up, results down) and the
  // per-handle events that order them with the forwards
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_x_ready = nullptr, ev_done = nullptr, ev_y_taken = nullptr;
  __nv_bfloat16* x_stage = nullptr;  // host-path staging [max_tokens][K]
  __nv_bfloat16* y_stage = nullptr;  // host-path staging [max_tokens][N]

  uint64_t wait_ns = 100000000ull;   // bounded-wait limit (100 ms)
  int skip_arrive = 0;
};

constexpr int kDecodeMaxTokens = 32;
constexpr int kPrefillBlockWords = 1024 + 128;  // prefill layout: a block's code words, then its scale/zero words
constexpr int kMaxGateHidden = 64;  // widest hidden layer of the MLP gate

constexpr int kDecodeRun = 256;  // channels per layout run

// Byte offset, inside wq_dec, of tile `tile`'s k64 block `kb` (lane data
// follows at 16 bytes per lane) and of its scale block for group `grp`.
struct DecodeLayout {
  int K, nt16, P;
  bool per_channel;
  static constexpr int KC = kDecodeRun;
  __host__ __device__ size_t stage_tile_bytes(int kcw) const {
    return (size_t)(kcw / 64) * 512 + (per_channel ? 0 : (size_t)(kcw / 128) * 64);
  }
  __host__ __device__ size_t tile_bytes() const { return stage_tile_bytes(K); }
  __host__ __device__ int pc(int cta) const { return min(P, nt16 - cta * P); }
  // start of (cta, stage) run
  __host__ __device__ size_t run_offset(int cta, int stage) const {
    return (size_t)cta * P * tile_bytes() + (size_t)pc(cta) * stage * stage_tile_bytes(KC);
  }
  __host__ __device__ int kcw(int stage) const { return min(KC, K - stage * KC); }
  __host__ __device__ size_t w_offset(int tile, int kb) const {
    const int cta = tile / P, tl = tile % P, stage = (kb * 64) / KC, kin = kb - stage * (KC / 64);
    return run_offset(cta, stage) + ((size_t)tl * (kcw(stage) / 64) + kin) * 512;
  }
  __host__ __device__ size_t sz_offset(int tile, int grp) const {
    const int cta = tile / P, tl = tile % P, stage = (grp * 128) / KC, gin = grp - stage * (KC / 128);
    const int w = kcw(stage);
    return run_offset(cta, stage) + (size_t)pc(cta) * (w / 64) * 512 + ((size_t)tl * (w / 128) + gin) * 64;
  }
};

// Tiles of 16 rows per CTA (grid <= SM count); fixed at create.
inline int decode_tiles_per_cta(int nt16, int sm_count) { return (nt16 + sm_count - 1) / sm_count; }

// Per-call decode schedule: NW consumer warps, T tiles per warp, KW warps
// splitting K, KC channels per pipeline stage (a whole number of layout runs).
// The consumer warps of a CTA form ceil(P / T) row groups of KW warps each;
// only instantiated (NW, T) pairs may be chosen (decode_mt*.cu). Register
// budget: the CTA's NW + 5 warps share four 16K-register files, so 21-23 warps
// get 80 registers per thread, 20 warps 96 and 15 warps 128.
inline void decode_plan(int P, int K, int M, int* NW, int* T, int* KW, int* KC) {
  if (M > 16) {
    // four token tiles: one or two tiles take 8 warps (K split four ways,
    // measured faster than 16); five, six or ten tiles take two, two or one
    // K warps per tile at up to 128 registers (the 16-warp variant spills);
    // other tile counts keep 16 warps busy
    *NW = P <= 2 ? 8 : P == 5 ? 10 : P == 6 ? 12 : P == 10 ? 10 : 16;
    *T = 1;
  } else {
    // 16 consumer warps (16 / P along K), except ten tiles at M <= 8: five
    // tile pairs (T = 2) with three K warps each, so that 15 warps work
    // instead of 10 (fused gate/up: 15.6 -> 13.2 us). 15 or 18 warps for
    // three, five, six or nine tiles measured no faster than 16 with one or
    // two idle; two tiles per warp at M <= 16 spills registers.
    if (P == 10 && M <= 8) {
      *NW = 15;
      *T = 2;
    } else {
      *NW = 16;
      *T = 1;
    }
  }
  const int pw = (P + *T - 1) / *T;  // warps along rows
  *KW = *NW / pw;                    // warps along K; 128-channel units go round-robin
  // Two units per K warp per stage: measured faster than smaller stages,
  // whose fixed per-stage costs (two copies, barrier round trips) dominate.
  int kc = kDecodeRun * *KW;
  const int kr = (K + kDecodeRun - 1) / kDecodeRun * kDecodeRun;
  if (kc > kr) kc = kr;
  // x box of a stage (KC channels x Mp tokens, bf16) at most 64 KB
  const int mp = M <= 8 ? 8 : (M <= 16 ? 16 : 32);
  const int kx = 32768 / mp / kDecodeRun * kDecodeRun;
  if (kc > kx) kc = kx;
  *KC = kc;
}
constexpr int kDecodeMaxTilesPerCta = 16;  // 16 consumer warps x one tile each
constexpr size_t kZDecFloats = 256 * 32;

// Tensor map over x [M][K] bf16 viewed as {64, M, K/64} (strides K*2 and 128
// bytes) with box {64, Mp, KC/64} and the 128-byte swizzle. Returns false if
// the driver entry point is unavailable or rejects the map.
bool encode_x_map(CUtensorMap* map, const void* x, int M, int K, int Mp, int KC);

// 2-D tensor map over a row-major bf16 matrix (`inner` elements per row,
// `rows` rows, `row_bytes` apart) with a {box_inner, box_rows} box and the
// 128-byte swizzle; out-of-range elements read as zero.
bool encode_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                    uint32_t box_inner, uint32_t box_rows);

spear_status_t spear_launch_decode(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                   cudaStream_t stream);
spear_status_t spear_decode_check_residency(spear_linear_s* h);
spear_status_t spear_launch_prefill(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                    cudaStream_t stream);
spear_status_t spear_launch_prefill_concurrent(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                               cudaStream_t stream, cudaStream_t ec_stream);
// Builds every kernel layout from user-layout weights: q, scales, zeros and A
// from `d` (A with h->rank rows), B from `B_rows` ([N][h->rank_b], the members'
// B matrices one after the other).
spear_status_t spear_build_layouts(spear_linear_s* h, const spear_linear_desc_t* d, const void* B_rows,
                                   cudaStream_t stream);
spear_status_t spear_launch_dequant(spear_linear_s* h, int path, __nv_bfloat16* out, cudaStream_t stream);

// Raise `kernel`'s dynamic shared-memory limit to 227 KB on the current device,
// once per (kernel, device): `done` is the caller's per-kernel set of devices
// already configured (bit d for device ordinal d < 64; larger ordinals are
// configured on every call). Setting the attribute is idempotent, so threads
// racing on the first launch on a device do no harm.
inline cudaError_t smem_limit_once(const void* kernel, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}
