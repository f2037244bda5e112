// Handle layout and internal launch interfaces shared by the .cu files of the
// library (not part of the public ABI).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spear.h"
#include "common.cuh"

// Kernel-side weight layouts (built once by spear_linear_create):
//
// Decode layout (warp MMA m16n8k16 fragments). Rows are grouped in tiles of
// 16. For a tile and a block of 64 input channels, lane l = 4g + t holds one
// uint4; word s (k16 step s of the block) packs the eight codes that lane
// feeds to the MMA A fragment, nibble i at bits 4i..4i+3:
//   i: 0 (g, 2t)  1 (g+8, 2t)  2 (g, 2t+8)  3 (g+8, 2t+8)
//      4 (g, 2t+1) 5 (g+8, 2t+1) 6 (g, 2t+9) 7 (g+8, 2t+9)
// (row within the tile, k within the 16-step), so (w >> 4j) & 0x000F000F
// yields A-fragment register j as a bf16 pair.
//   wq_dec  uint4 [nt16][K/64][32]
//   sz_dec  u32   [nt16][n_groups][16]   bits 0..15 bf16 scale, 16..31 bf16(128 + zero)
//   a_dec   uint4 [rank/16][K/16][32]    A in A-fragment order (bf16 pairs)
//   b_dec   uint4 [nt16][rank/16][32]    B in A-fragment order (bf16 pairs)
//
// Prefill layout (row-major 16-byte chunks for the tensor-core tile loader).
// Rows are grouped in tiles of 128; for a tile and a block of 64 channels the
// 4 KB block holds, per row, eight u32 words; word c packs channels
// 8c .. 8c+7 with nibble order (0, 2, 4, 6, 1, 3, 5, 7) so that
// (w >> 4j) & 0x000F000F yields channels (2j, 2j+1) as a bf16 pair.
//   wq_pre  u32   [nt128][K/64][128][8]
//   sz_pre  u32   [nt128][n_groups][128] same encoding as sz_dec
//   a_pre   bf16  [rank][K]               copy of A
//   b_pre   bf16  [nt128*128][rank]       copy of B, zero rows past N

struct spear_linear_s {
  int device = 0, sm_count = 0;
  int K = 0, N = 0, G = 0, n_groups = 0, rank = 0, max_tokens = 0;
  float alpha = 1.f;
  int gate = 0;
  bool per_channel = false;

  int nt16 = 0, nt128 = 0;
  uint4* wq_dec = nullptr;
  uint32_t* sz_dec = nullptr;
  uint4* a_dec = nullptr;
  uint4* b_dec = nullptr;
  uint32_t* wq_pre = nullptr;
  uint32_t* sz_pre = nullptr;
  __nv_bfloat16* a_pre = nullptr;
  __nv_bfloat16* b_pre = nullptr;

  // Workspace: SyncWords followed by z [256][32] fp32 (decode), then the
  // prefill buffers.
  void* ws = nullptr;
  spear::SyncWords* sync = nullptr;
  float* z_dec = nullptr;
  float* z_pre = nullptr;            // [max_tokens][rank] fp32 (prefill projection)
  __nv_bfloat16* u_pre = nullptr;    // [max_tokens][rank] bf16 (prefill gated, alpha-scaled)
  __nv_bfloat16* x_stage = nullptr;  // host-path staging [max_tokens][K]
  __nv_bfloat16* y_stage = nullptr;  // host-path staging [max_tokens][N]

  uint64_t wait_ns = 100000000ull;   // bounded-wait limit (100 ms)
  int skip_arrive = 0;
};

constexpr int kDecodeMaxTokens = 32;
constexpr int kDecodeMaxTilesPerCta = 16;
constexpr size_t kZDecFloats = 256 * 32;

spear_status_t spear_launch_decode(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                   cudaStream_t stream);
spear_status_t spear_launch_prefill(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                    cudaStream_t stream);
spear_status_t spear_build_layouts(spear_linear_s* h, const spear_linear_desc_t* d, cudaStream_t stream);
spear_status_t spear_launch_dequant(spear_linear_s* h, int path, __nv_bfloat16* out, cudaStream_t stream);
