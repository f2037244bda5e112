// Shared device helpers for the sm_103a kernels: inline PTX for mbarriers,
// bulk async copies, warp-level MMA, INT4 unpacking and bounded waits.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define SPEAR_DEVINL __device__ __forceinline__

namespace spear {

// Device status word bits (latched until spear_linear_check clears them).
enum : unsigned {
  kStatusTimeoutZ = 1u,      // grid-wide "compensator projection done" wait gave up
  kStatusTimeoutPipe = 2u,   // an mbarrier wait in a pipeline gave up
};

// Workspace of one handle (device memory, zero-initialised at create).
struct SyncWords {
  unsigned status;     // kStatus* bits
  unsigned epoch;      // decode: calls completed (selects the z buffer)
  unsigned arrive_acc; // decode: CTA arrivals summed over all calls (epoch * grid at a call's start)
  unsigned pad[29];    // keep the z buffer 128-byte aligned
};
static_assert(sizeof(SyncWords) == 128, "the decode z buffer follows at a 128-byte boundary");

SPEAR_DEVINL uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SPEAR_DEVINL uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
SPEAR_DEVINL void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

SPEAR_DEVINL void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

SPEAR_DEVINL void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

SPEAR_DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

SPEAR_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

SPEAR_DEVINL bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; gives up after `limit_ns`
// (returns false) so that a broken pipeline can never hang the GPU.
SPEAR_DEVINL bool mbar_wait_bounded(uint64_t* bar, unsigned parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// Same, but each try suspends the thread for at most `hint_ns` (the pipeline
// roles of the prefill kernel: a short suspension re-checks the phase sooner
// than the default time limit; measured ~5% per K block in a replica of the
// pipeline).
SPEAR_DEVINL bool mbar_try_wait_hint(uint64_t* bar, unsigned parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
SPEAR_DEVINL bool mbar_wait_bounded_hint(uint64_t* bar, unsigned parity, uint64_t limit_ns, uint32_t hint_ns) {
  if (mbar_try_wait_hint(bar, parity, hint_ns)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait_hint(bar, parity, hint_ns)) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------- bulk copies
// 1-D bulk copy global -> shared of the executing CTA, completion counted in
// bytes on `bar`. dst, src 16-byte aligned, bytes a multiple of 16.
SPEAR_DEVINL void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, destination given as a shared-space address.
SPEAR_DEVINL void bulk_g2s_shared_u32(uint32_t dst, const void* src, unsigned bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 evict-first hint for data read exactly once (weights).
SPEAR_DEVINL void bulk_g2s_stream(void* dst, const void* src, unsigned bytes, uint64_t* bar,
                                  uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 3-D tiled tensor copy global -> shared (box shape fixed by the map), counted
// on `bar`. c0 is the innermost coordinate; c0 * element size must be a
// multiple of 16 bytes.
SPEAR_DEVINL void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Fetch a tensor map (a kernel parameter) into the copy engine's descriptor
// cache ahead of its first use.
SPEAR_DEVINL void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Warm L2 with the 128-byte line holding p (an ordinary load-path prefetch).
SPEAR_DEVINL void prefetch_l2_line(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

// Warm L2 with [src, src + bytes) (16-byte aligned, multiple of 16 bytes).
SPEAR_DEVINL void prefetch_l2(const void* src, unsigned bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

SPEAR_DEVINL uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- shared loads
// Explicit shared-space loads on 32-bit shared addresses (generic loads of
// shared memory take the slower L1TEX path). Volatile so that they stay
// between the mbarrier wait and arrival that bracket their data.
SPEAR_DEVINL uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

SPEAR_DEVINL uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// ---------------------------------------------------------------- warp MMA
// D = A(16x16, row) * B(16x8, col) + C, bf16 inputs, fp32 accumulate.
// Not volatile: a pure register operation the compiler may schedule freely.
SPEAR_DEVINL void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

SPEAR_DEVINL void ldmatrix_x2(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r0), "=r"(r1)
               : "r"(smem_u32(p)));
}

// ---------------------------------------------------------------- INT4 unpack
// (w & 0x000F000F) | 0x43004300: the nibbles at bits 0..3 and 16..19 become the
// low mantissa bits of two bf16 values 128 + code (exact: bf16 has 8
// significant bits and 128..143 are integers in its [128, 256) binade).
SPEAR_DEVINL uint32_t int4_pair_to_bf16x2_biased(uint32_t w) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(0x000F000Fu), "r"(0x43004300u));
  return r;
}

// a - b on bf16x2; exact here because both operands are integers in [128, 143].
SPEAR_DEVINL uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// bf16 bits of (128 + z) in both halves.
SPEAR_DEVINL uint32_t biased_zero_x2(uint32_t zbits16) { return zbits16 | (zbits16 << 16); }

// The same pair from a scale/zero word (bits 16..31 = bf16(128 + z)): one byte permute.
SPEAR_DEVINL uint32_t biased_zero_x2_of_word(uint32_t w) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %1, 0x3232;" : "=r"(r) : "r"(w));
  return r;
}

SPEAR_DEVINL float bf16_bits_to_float(uint32_t b16) { return __uint_as_float(b16 << 16); }

// ---------------------------------------------------------------- decode-layout A fragments
// One code word w of the decode layout holds nibble j and j + 4 of A-fragment
// register j (j = 0..3; registers 0 and 2 are row g, 1 and 3 row g + 8).
// Masked without a shift, a nibble pair reads as a bf16 pair of tiny values:
// (w & 0x000F000F) puts code q in the mantissa with a zero exponent field, i.e.
// q * 2^-133; (w & 0x00F000F0) puts 16 q in bits 0..7, whose top bit is the
// exponent field's lowest bit, and since the subnormal binade and the first
// normal one share the spacing 2^-133 it reads as 16 q * 2^-133 for every q.
// One fma.rn.bf16x2 by 2^126 plus c, with c = -z * 2^-7 for the low nibbles
// and -z * 2^-3 for the high ones, then yields (q - z) * 2^-7 and
// (q - z) * 2^-3, both exact (bf16 arithmetic keeps subnormal inputs), so
// rows g carry the factor 2^-7 and rows g + 8 the factor 2^-3, which an exact
// fp32 multiplication by kFragScaleLo / kFragScaleHi takes back before the
// scale is applied (scaling s instead could overflow). One shift, four masks and
// four fmas per word, against three shifts, four masks and four subtractions
// for the biased form (bias 128 in the exponent, minus 128 + z).
constexpr float kFragScaleLo = 128.f;  // rows g: fragment values are (q - z) * 2^-7
constexpr float kFragScaleHi = 8.f;    // rows g + 8: fragment values are (q - z) * 2^-3

SPEAR_DEVINL uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// The additive terms from the pair bf16(128 + z) in both halves (exact).
SPEAR_DEVINL uint32_t frag_zero_lo(uint32_t biased_zz) {  // -z * 2^-7 = 1 - (128 + z) * 2^-7
  return bf16x2_fma(biased_zz, 0xBC00BC00u /* -2^-7 */, 0x3F803F80u /* 1 */);
}
SPEAR_DEVINL uint32_t frag_zero_hi(uint32_t biased_zz) {  // -z * 2^-3 = 16 - (128 + z) * 2^-3
  return bf16x2_fma(biased_zz, 0xBE00BE00u /* -2^-3 */, 0x41804180u /* 16 */);
}

SPEAR_DEVINL void decode_frag_unpack(uint32_t w, uint32_t c_lo, uint32_t c_hi, uint32_t (&a)[4]) {
  constexpr uint32_t k2p126 = 0x7E807E80u;  // 2^126 in both halves
  const uint32_t w8 = w >> 8;
  a[0] = bf16x2_fma(w & 0x000F000Fu, k2p126, c_lo);
  a[1] = bf16x2_fma(w & 0x00F000F0u, k2p126, c_hi);
  a[2] = bf16x2_fma(w8 & 0x000F000Fu, k2p126, c_lo);
  a[3] = bf16x2_fma(w8 & 0x00F000F0u, k2p126, c_hi);
}

SPEAR_DEVINL uint32_t pack_bf16x2(float lo, float hi);

// Copy a bf16 [rows][cols] matrix (cols a multiple of 8, 16-byte aligned rows)
// into shared memory with row stride cols + 8 (16-byte chunks, all loads of a
// thread's share in flight before any store): the MLP gate's weights.
SPEAR_DEVINL void stage_rows_padded(__nv_bfloat16* dst, const __nv_bfloat16* src, int rows, int cols, int tid,
                                    int nthreads) {
  const int c8 = cols / 8, n = rows * c8;
  for (int i0 = 0; i0 < n; i0 += 4 * nthreads) {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = i0 + k * nthreads + tid;
      v[k] = i < n ? __ldg(reinterpret_cast<const uint4*>(src) + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = i0 + k * nthreads + tid;
      if (i < n) *reinterpret_cast<uint4*>(dst + (i / c8) * (cols + 8) + (i % c8) * 8) = v[k];
    }
  }
}

// Bottleneck-MLP gate logits of one block of 16 tokens by warp MMA (bf16
// operands, fp32 accumulation), for the gate gamma(z) = sigmoid(W2 relu(W1 z)):
//   t = relu(z W1^T) (16 x gh),   g = t W2^T (16 x r),
// rows t0 .. t0 + 15 of z (fp32, shared memory, row stride zst floats; rows
// past the valid tokens must hold zeros). z enters the first product as bf16
// hi + lo (two MMAs per step), t the second as bf16. W1 is [gh][r] (row stride
// w1s elements), W2 [r][gh] (row stride w2s), bf16, in shared or global
// memory, with gh a multiple of 16 and r of 16 (gh <= 64). The C fragment of a
// 16 x 8 tile of t is the A fragment of the second product, so t never leaves
// registers. For each 8-column tile j8 of g in [j8_0, j8_1), out(row, col,
// g[row][col], g[row][col + 1]) is called for this lane's two pairs: rows
// t0 + lane / 4 and + 8, columns 8 j8 + 2 (lane % 4) and + 1.
template <class Out>
SPEAR_DEVINL void mlp_gate_logits(const float* z, int zst, int t0, int r, int gh, const __nv_bfloat16* W1, int w1s,
                                  const __nv_bfloat16* W2, int w2s, int lane, int j8_0, int j8_1, Out out) {
  const int g = lane >> 2, tq = lane & 3;
  const int nh8 = gh / 8;  // 8-unit tiles of the hidden layer, even
  float acc1[8][4];
#pragma unroll
  for (int c = 0; c < 8; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc1[c][e] = 0.f;
  for (int k16 = 0; k16 < r / 16; ++k16) {
    const float* z0 = z + (t0 + g) * zst + k16 * 16 + 2 * tq;
    const float* z1 = z0 + 8 * zst;
    const float2 v[4] = {*reinterpret_cast<const float2*>(z0), *reinterpret_cast<const float2*>(z1),
                         *reinterpret_cast<const float2*>(z0 + 8), *reinterpret_cast<const float2*>(z1 + 8)};
    uint32_t ah[4], al[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ah[i] = pack_bf16x2(v[i].x, v[i].y);
      al[i] = pack_bf16x2(v[i].x - __uint_as_float(ah[i] << 16), v[i].y - __uint_as_float(ah[i] & 0xFFFF0000u));
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      if (c < nh8) {
        const __nv_bfloat16* w = W1 + (size_t)(c * 8 + g) * w1s + k16 * 16 + 2 * tq;
        const uint32_t b0 = *reinterpret_cast<const unsigned int*>(w);
        const uint32_t b1 = *reinterpret_cast<const unsigned int*>(w + 8);
        mma_bf16_16816(acc1[c], ah, b0, b1);
        mma_bf16_16816(acc1[c], al, b0, b1);
      }
    }
  }
  uint32_t ta[4][4];  // relu(t) as A fragments, one per 16 hidden units
#pragma unroll
  for (int kh = 0; kh < 4; ++kh) {
    if (2 * kh < nh8) {
      ta[kh][0] = pack_bf16x2(fmaxf(acc1[2 * kh][0], 0.f), fmaxf(acc1[2 * kh][1], 0.f));
      ta[kh][1] = pack_bf16x2(fmaxf(acc1[2 * kh][2], 0.f), fmaxf(acc1[2 * kh][3], 0.f));
      ta[kh][2] = pack_bf16x2(fmaxf(acc1[2 * kh + 1][0], 0.f), fmaxf(acc1[2 * kh + 1][1], 0.f));
      ta[kh][3] = pack_bf16x2(fmaxf(acc1[2 * kh + 1][2], 0.f), fmaxf(acc1[2 * kh + 1][3], 0.f));
    }
  }
  for (int j8 = j8_0; j8 < j8_1; ++j8) {
    float c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kh = 0; kh < 4; ++kh) {
      if (2 * kh < nh8) {
        const __nv_bfloat16* w = W2 + (size_t)(j8 * 8 + g) * w2s + kh * 16 + 2 * tq;
        mma_bf16_16816(c2, ta[kh], *reinterpret_cast<const unsigned int*>(w),
                       *reinterpret_cast<const unsigned int*>(w + 8));
      }
    }
    out(t0 + g, j8 * 8 + 2 * tq, c2[0], c2[1]);
    out(t0 + g + 8, j8 * 8 + 2 * tq, c2[2], c2[3]);
  }
}

SPEAR_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Split v into bf16 hi + bf16 lo with hi + lo == v to ~2^-17 relative.
SPEAR_DEVINL void split_bf16(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

SPEAR_DEVINL void red_add_v2(float* addr, float a, float b) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(addr), "f"(a), "f"(b) : "memory");
}

SPEAR_DEVINL unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

}  // namespace spear
