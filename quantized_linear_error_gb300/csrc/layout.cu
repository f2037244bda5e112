// One-time re-layout of user weights into the kernel layouts (run by
// spear_linear_create), and the dequantisation export used to test the unpack
// code of both layouts bit for bit.
#include "internal.h"

namespace spear {
namespace {

// Code of (row, k) from the user layout: byte k/2 of the row, even k low nibble.
__device__ __forceinline__ uint32_t user_code(const uint8_t* q, int K, int N, int row, int k) {
  if (row >= N) return 0u;
  const uint8_t b = q[(size_t)row * (K / 2) + (k >> 1)];
  return (k & 1) ? (b >> 4) : (b & 0xF);
}

__device__ __forceinline__ uint32_t user_sz(const uint16_t* s, const uint8_t* z, int n_groups, int N, int row,
                                            int g) {
  if (row >= N) return 0x4300u << 16;  // scale 0, zero 0: a padded row dequantises to 0
  const uint32_t sb = s[(size_t)row * n_groups + g];
  const uint32_t zp = z ? z[(size_t)row * n_groups + g] : 8u;
  return sb | ((0x4300u | zp) << 16);
}

__global__ void repack_w_decode(const uint8_t* __restrict__ q, int K, int N, DecodeLayout L, uint8_t* __restrict__ out) {
  const int kb64 = K / 64;
  const long total = (long)L.nt16 * kb64 * 32;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int lane = i % 32;
    const int kb = (i / 32) % kb64;
    const int tile = i / (32L * kb64);
    const int g = lane >> 2, t = lane & 3;
    const int r0 = tile * 16 + g, r1 = r0 + 8;
    uint32_t w[4];
    for (int s = 0; s < 4; ++s) {
      const int k = kb * 64 + s * 16 + 2 * t;
      w[s] = user_code(q, K, N, r0, k) | user_code(q, K, N, r1, k) << 4 | user_code(q, K, N, r0, k + 8) << 8 |
             user_code(q, K, N, r1, k + 8) << 12 | user_code(q, K, N, r0, k + 1) << 16 |
             user_code(q, K, N, r1, k + 1) << 20 | user_code(q, K, N, r0, k + 9) << 24 |
             user_code(q, K, N, r1, k + 9) << 28;
    }
    *reinterpret_cast<uint4*>(out + L.w_offset(tile, kb) + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__global__ void repack_sz_decode(const uint16_t* __restrict__ s, const uint8_t* __restrict__ z, int n_groups, int N,
                                 DecodeLayout L, uint8_t* __restrict__ out) {
  const long total = (long)L.nt16 * n_groups * 16;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int rl = i % 16;
    const int g = (i / 16) % n_groups;
    const int tile = i / (16L * n_groups);
    *reinterpret_cast<uint32_t*>(out + L.sz_offset(tile, g) + rl * 4) = user_sz(s, z, n_groups, N, tile * 16 + rl, g);
  }
}

// Prefill layout: per (row tile, 64-channel block) 1024 code words, then the
// block's 128 scale/zero words (kPrefillBlockWords in all).
__global__ void repack_w_prefill(const uint8_t* __restrict__ q, int K, int N, int nt128, uint32_t* __restrict__ out) {
  const int kb64 = K / 64;
  const long total = (long)nt128 * kb64 * 128 * 8;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int c = i % 8;
    const int rl = (i / 8) % 128;
    const int kb = (i / 1024) % kb64;
    const int tile = i / (1024L * kb64);
    const int row = tile * 128 + rl;
    const int k = kb * 64 + c * 8;
    uint32_t w = 0;
    // nibble slot j*4 holds channel 2j, slot 16 + j*4 holds channel 2j+1
    for (int j = 0; j < 4; ++j) {
      w |= user_code(q, K, N, row, k + 2 * j) << (4 * j);
      w |= user_code(q, K, N, row, k + 2 * j + 1) << (16 + 4 * j);
    }
    out[((long)tile * kb64 + kb) * kPrefillBlockWords + (i % 1024)] = w;
  }
}

// The scale/zero words of the prefill blocks: block (tile, kb), row rl holds
// the word of the group of channels kb * 64 (the same word in both blocks of
// a 128-channel group, and in every block of a per-channel row).
__global__ void repack_sz_prefill(const uint16_t* __restrict__ s, const uint8_t* __restrict__ z, int K, int G,
                                  int n_groups, int N, int nt128, uint32_t* __restrict__ out) {
  const int kb64 = K / 64;
  const long total = (long)nt128 * kb64 * 128;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int rl = i % 128;
    const int kb = (i / 128) % kb64;
    const int tile = i / (128L * kb64);
    out[((long)tile * kb64 + kb) * kPrefillBlockWords + 1024 + rl] =
        user_sz(s, z, n_groups, N, tile * 128 + rl, (kb * 64) / G);
  }
}

__global__ void repack_sz(const uint16_t* __restrict__ s, const uint8_t* __restrict__ z, int n_groups, int N,
                          int ntiles, int tile_rows, uint32_t* __restrict__ out) {
  const long total = (long)ntiles * n_groups * tile_rows;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int rl = i % tile_rows;
    const int g = (i / tile_rows) % n_groups;
    const int tile = i / ((long)tile_rows * n_groups);
    out[i] = user_sz(s, z, n_groups, N, tile * tile_rows + rl, g);
  }
}

// bf16 matrix [rows][cols] into m16n8k16 A-fragment order [rows/16][cols/16][32] uint4.
// With `quad`, the 16 columns of a k16 step are taken in the order that gives
// lane t the four consecutive columns 4t .. 4t + 3 (fragment columns 2t, 2t + 1,
// 2t + 8, 2t + 9), so that the matching B fragment of a row-major activation is
// one 8-byte load (the compensator's down-projection A).
__global__ void repack_frag(const uint16_t* __restrict__ m, int rows, int cols, int row_tiles, bool quad,
                            uint4* __restrict__ out) {
  const int ks = cols / 16;
  const long total = (long)row_tiles * ks * 32;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int lane = i % 32;
    const int kk = (i / 32) % ks;
    const int tile = i / (32L * ks);
    const int g = lane >> 2, t = lane & 3;
    const int r0 = tile * 16 + g, r1 = r0 + 8;
    const int k = kk * 16 + (quad ? 4 * t : 2 * t);
    const int k2 = quad ? k + 2 : k + 8;  // columns of registers 2 and 3
    auto at = [&](int r, int c) -> uint32_t { return r < rows ? (uint32_t)m[(size_t)r * cols + c] : 0u; };
    out[i] = make_uint4(at(r0, k) | at(r0, k + 1) << 16, at(r1, k) | at(r1, k + 1) << 16,
                        at(r0, k2) | at(r0, k2 + 1) << 16, at(r1, k2) | at(r1, k2 + 1) << 16);
  }
}

// Copy a bf16 [rows][cols] matrix into [rows_pad][cols], zero rows past `rows`.
__global__ void copy_pad_rows(const uint16_t* __restrict__ m, int rows, int rows_pad, int cols,
                              uint16_t* __restrict__ out) {
  const long total = (long)rows_pad * cols;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x)
    out[i] = (i / cols) < rows ? m[i] : (uint16_t)0;
}

// Block-diagonal prefill B of a grouped handle: out [rows_pad][n * rb], row r
// of member i (rows [start[i], start[i + 1])) holds that member's B row in
// columns [i rb, (i + 1) rb) and zeros elsewhere; rows past N are zero.
struct RowStarts {
  int n;
  int start[kMaxGroup + 1];
};
__global__ void expand_block_diag(const uint16_t* __restrict__ b, int N, int rb, RowStarts rs, int rows_pad,
                                  uint16_t* __restrict__ out) {
  const int cols = rs.n * rb;
  const long total = (long)rows_pad * cols;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int row = (int)(i / cols), c = (int)(i % cols);
    uint16_t v = 0;
    if (row < N) {
      int m = 0;
      while (m + 1 < rs.n && row >= rs.start[m + 1]) ++m;
      if (c / rb == m) v = b[(size_t)row * rb + (c - m * rb)];
    }
    out[i] = v;
  }
}

// (q - z) * s with one rounding: the exact difference d = (q - z) * 2^-e comes
// from the kernels' own unpack (e = 0 for the prefill layout; e = 7 or 3 for
// the decode layout), d * 2^e is exact, its product with s is exact in fp32
// (at most 4 + 8 significant bits) unless it overflows, and the conversion to
// bf16 rounds once to nearest even.
__device__ __forceinline__ __nv_bfloat16 scaled(uint32_t diff_bits16, float s, float pow2 = 1.f) {
  return __float2bfloat16_rn((bf16_bits_to_float(diff_bits16) * pow2) * s);
}

__global__ void dequant_from_decode(const uint8_t* __restrict__ wq, const uint32_t* __restrict__ sz_pc, int K, int N,
                                    DecodeLayout L, __nv_bfloat16* __restrict__ out) {
  const int kb64 = K / 64;
  const long total = (long)L.nt16 * kb64 * 32;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int lane = i % 32;
    const int kb = (i / 32) % kb64;
    const int tile = i / (32L * kb64);
    const int g = lane >> 2, t = lane & 3;
    const uint32_t* szb = L.per_channel ? sz_pc + (size_t)tile * 16
                                        : reinterpret_cast<const uint32_t*>(wq + L.sz_offset(tile, (kb * 64) / 128));
    const uint32_t sz0 = szb[g], sz1 = szb[g + 8];
    const uint32_t c0 = frag_zero_lo(biased_zero_x2(sz0 >> 16)), c1 = frag_zero_hi(biased_zero_x2(sz1 >> 16));
    const float s0 = bf16_bits_to_float(sz0 & 0xFFFF), s1 = bf16_bits_to_float(sz1 & 0xFFFF);
    const uint4 v = *reinterpret_cast<const uint4*>(wq + L.w_offset(tile, kb) + lane * 16);
    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
    const int r0 = tile * 16 + g, r1 = r0 + 8;
    for (int s = 0; s < 4; ++s) {
      // the decode kernel's own unpack: (q - z) * 2^-7 for rows r0, (q - z) * 2^-3
      // for rows r1, taken back by an exact power-of-two product before the scale
      uint32_t d[4];
      decode_frag_unpack(words[s], c0, c1, d);
      const uint32_t d0 = d[0], d1 = d[1], d2 = d[2], d3 = d[3];  // (r0, k..k+1) (r1, k..) (r0, k+8..) (r1, k+8..)
      const int k = kb * 64 + s * 16 + 2 * t;
      if (r0 < N) {
        out[(size_t)r0 * K + k] = scaled(d0 & 0xFFFF, s0, kFragScaleLo);
        out[(size_t)r0 * K + k + 1] = scaled(d0 >> 16, s0, kFragScaleLo);
        out[(size_t)r0 * K + k + 8] = scaled(d2 & 0xFFFF, s0, kFragScaleLo);
        out[(size_t)r0 * K + k + 9] = scaled(d2 >> 16, s0, kFragScaleLo);
      }
      if (r1 < N) {
        out[(size_t)r1 * K + k] = scaled(d1 & 0xFFFF, s1, kFragScaleHi);
        out[(size_t)r1 * K + k + 1] = scaled(d1 >> 16, s1, kFragScaleHi);
        out[(size_t)r1 * K + k + 8] = scaled(d3 & 0xFFFF, s1, kFragScaleHi);
        out[(size_t)r1 * K + k + 9] = scaled(d3 >> 16, s1, kFragScaleHi);
      }
    }
  }
}

__global__ void dequant_from_prefill(const uint32_t* __restrict__ wq, int K, int N, int nt128,
                                     __nv_bfloat16* __restrict__ out) {
  const int kb64 = K / 64;
  const long total = (long)nt128 * kb64 * 1024;
  for (long i = blockIdx.x * (long)blockDim.x + threadIdx.x; i < total; i += (long)gridDim.x * blockDim.x) {
    const int c = i % 8;
    const int rl = (i / 8) % 128;
    const int kb = (i / 1024) % kb64;
    const int tile = i / (1024L * kb64);
    const int row = tile * 128 + rl;
    if (row >= N) continue;
    const int k = kb * 64 + c * 8;
    const uint32_t* blk = wq + ((size_t)tile * kb64 + kb) * kPrefillBlockWords;
    const uint32_t szw = blk[1024 + rl];
    const uint32_t zz = biased_zero_x2(szw >> 16);
    const float s = bf16_bits_to_float(szw & 0xFFFF);
    const uint32_t w = blk[i % 1024];
    __align__(16) __nv_bfloat16 v[8];
    for (int j = 0; j < 4; ++j) {
      const uint32_t d = bf16x2_sub(int4_pair_to_bf16x2_biased(w >> (4 * j)), zz);
      v[2 * j] = scaled(d & 0xFFFF, s);
      v[2 * j + 1] = scaled(d >> 16, s);
    }
    *reinterpret_cast<uint4*>(out + (size_t)row * K + k) = *reinterpret_cast<uint4*>(v);
  }
}

inline int grid_for(long total, int threads) {
  long b = (total + threads - 1) / threads;
  return (int)(b < 1 ? 1 : (b > 65535L * 8 ? 65535L * 8 : b));
}

}  // namespace
}  // namespace spear

using namespace spear;

spear_status_t spear_build_layouts(spear_linear_s* h, const spear_linear_desc_t* d, const void* B_rows,
                                   cudaStream_t st) {
  const int K = h->K, N = h->N, r = h->rank, rb = h->rank_b;
  const uint16_t* s = static_cast<const uint16_t*>(d->scales);
  const int T = 256;
  long n;
  const DecodeLayout L{K, h->nt16, h->dec_P, h->per_channel};
  n = (long)h->nt16 * (K / 64) * 32;
  repack_w_decode<<<grid_for(n, T), T, 0, st>>>(d->qweight, K, N, L, h->wq_dec);
  if (h->per_channel) {
    n = (long)h->nt16 * 16;
    repack_sz<<<grid_for(n, T), T, 0, st>>>(s, d->zeros, 1, N, h->nt16, 16, h->sz_dec);
  } else {
    n = (long)h->nt16 * h->n_groups * 16;
    repack_sz_decode<<<grid_for(n, T), T, 0, st>>>(s, d->zeros, h->n_groups, N, L, h->wq_dec);
  }
  n = (long)h->nt128 * (K / 64) * 1024;
  repack_w_prefill<<<grid_for(n, T), T, 0, st>>>(d->qweight, K, N, h->nt128, h->wq_pre);
  n = (long)h->nt128 * (K / 64) * 128;
  repack_sz_prefill<<<grid_for(n, T), T, 0, st>>>(s, d->zeros, K, h->G, h->n_groups, N, h->nt128, h->wq_pre);
  if (r > 0) {
    const uint16_t* A = static_cast<const uint16_t*>(d->A);
    const uint16_t* B = static_cast<const uint16_t*>(B_rows);
    n = (long)(r / 16) * (K / 16) * 32;
    repack_frag<<<grid_for(n, T), T, 0, st>>>(A, r, K, r / 16, true, h->a_dec);
    n = (long)h->nt16 * (rb / 16) * 32;
    repack_frag<<<grid_for(n, T), T, 0, st>>>(B, N, rb, h->nt16, false, h->b_dec);
    n = (long)r * K;
    copy_pad_rows<<<grid_for(n, T), T, 0, st>>>(A, r, r, K, reinterpret_cast<uint16_t*>(h->a_pre));
    n = (long)h->nt128 * 128 * r;
    if (h->n_members == 1) {
      copy_pad_rows<<<grid_for(n, T), T, 0, st>>>(B, N, h->nt128 * 128, r, reinterpret_cast<uint16_t*>(h->b_pre));
    } else {
      RowStarts rs{};
      rs.n = h->n_members;
      for (int i = 0; i <= h->n_members; ++i) rs.start[i] = h->row_start[i];
      expand_block_diag<<<grid_for(n, T), T, 0, st>>>(B, N, rb, rs, h->nt128 * 128,
                                                      reinterpret_cast<uint16_t*>(h->b_pre));
    }
  }
  return cudaGetLastError() == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}

spear_status_t spear_launch_dequant(spear_linear_s* h, int path, __nv_bfloat16* out, cudaStream_t st) {
  const int T = 256;
  if (path == 0) {
    const DecodeLayout L{h->K, h->nt16, h->dec_P, h->per_channel};
    long n = (long)h->nt16 * (h->K / 64) * 32;
    dequant_from_decode<<<grid_for(n, T), T, 0, st>>>(h->wq_dec, h->sz_dec, h->K, h->N, L, out);
  } else {
    long n = (long)h->nt128 * (h->K / 64) * 1024;
    dequant_from_prefill<<<grid_for(n, T), T, 0, st>>>(h->wq_pre, h->K, h->N, h->nt128, out);
  }
  return cudaGetLastError() == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}
