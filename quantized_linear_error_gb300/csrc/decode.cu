// Decode-phase kernel: the whole W4 + error-compensator linear for M <= 32
// tokens in one launch ("SPEAR: A System for Post-Quantization Error-Adaptive
// Recovery", section 2.2A: in the memory-bound decode phase the compensator is
// fused into the low-bit GEMM so the correction path is a single kernel).
//
// Design (one CTA per SM; 16 consumer warps, or 8 / 10 for M > 16 with 2 / 5
// tiles per CTA, + 1 producer warp + 4 compensator warps):
//  * The CTA owns P consecutive 16-row tiles of W. A producer warp streams K
//    in stages: per stage one bulk copy brings the tiles' packed codes and
//    scale/zero words (laid out at create as one contiguous run per CTA and
//    stage, since every bulk copy has a fixed issue cost) and one 3-D tensor
//    copy brings x[0:Mp, k-slice] with a 128-byte swizzle (tokens past M are
//    zero-filled by the copy engine), both counted on one mbarrier.
//  * Consumer warps turn each 32-bit word into four bf16 A-fragment registers
//    with one shift, one mask per pair (the codes land in the mantissa of a
//    bf16 pair with an exponent field of 0 or 1) and one bf16x2 fma by 2^126
//    with -z * 2^-7 or -z * 2^-3, which leaves the exact (q - z) * 2^-7 or
//    (q - z) * 2^-3; the power of two is taken back in fp32.
//    Warp MMA (m16n8k16, fp32 accumulate) takes x as the 8-wide N operand
//    (tokens), and the group scale is applied once per group to the fp32
//    partial sum.
//  * A separate compensator warp per CTA runs concurrently with the W stream:
//    it computes the CTA's share of the down-projection z = A x (split over
//    all CTAs), adds it into a workspace with vector atomics, bumps an arrival
//    counter, waits (bounded by %globaltimer) for every CTA's arrival, applies
//    the gate u = alpha * gamma(z) * z, splits u into bf16 hi + lo in shared
//    memory and signals the consumers through an mbarrier. The last CTA to
//    read z clears it for the next call. After their W tiles the consumer
//    warps add B u to the fp32 accumulators with two more MMAs per step and
//    round y to bf16 once. HBM traffic is W, scales/zeros, A and B once each.
#include "decode_kernel.cuh"

namespace spear {
namespace dec {
namespace {

DecodeKernelRef kernel_for(int NW, int MT, int T, bool pc, bool ec) {
  if (MT == 1) return kernel_ref_mt1(NW, T, pc, ec);
  if (MT == 2) return kernel_ref_mt2(NW, T, pc, ec);
  return kernel_ref_mt4(NW, T, pc, ec);
}

// Everything a decode launch needs except the x tensor map.
struct DecodeLaunch {
  DecodeParams p;
  int grid = 0, NW = 0, MT = 0, T = 0;
  size_t smem = 0;
  DecodeKernelRef kernel;
};

spear_status_t decode_config(const spear_linear_s* h, int M, DecodeLaunch* out) {
  DecodeParams& p = out->p;
  p = DecodeParams{};
  const int MT = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
  const int Mp = 8 * MT;
  const bool ec = h->rank > 0;
  const int P = h->dec_P;
  int NW, T, KW, KC;
  decode_plan(P, h->K, M, &NW, &T, &KW, &KC);
  if (P > T * NW) return SPEAR_ERR_UNSUPPORTED;
  const DecodeLayout L{h->K, h->nt16, P, h->per_channel};

  p.wq = h->wq_dec;
  p.sz = h->sz_dec;
  p.a_frag = h->a_dec;
  p.b_frag = h->b_dec;
  p.z = h->z_mma;
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
  p.wait_ns = h->wait_ns;
  p.skip_arrive = h->skip_arrive;
  p.gw1 = h->gate_w1;
  p.gw2 = h->gate_w2;
  p.gh = h->gate_hidden;
  p.n_members = h->n_members;
  p.rank_b = h->rank_b;
  for (int i = 0; i <= h->n_members; ++i) p.tile_start[i] = h->row_start[i] / 16;
  for (int i = 0; i < h->n_members; ++i) p.alphas[i] = h->alphas[i];

  const size_t red_bytes = (size_t)P * KW * 32 * 4 * MT * 4;
  const size_t u_bytes = ec ? (size_t)2 * Mp * (h->rank + 8) * 2 : 0;
  // MLP gate: z^T [M16][rank + 8] fp32, W1 [gh][rank + 8] and W2 [rank][gh + 8] bf16
  const size_t mlp_bytes =
      h->gate_hidden > 0 ? (size_t)(Mp < 16 ? 16 : Mp) * (h->rank + 8) * 4 +
                               ((size_t)h->gate_hidden * (h->rank + 8) + (size_t)h->rank * (h->gate_hidden + 8)) * 2
                         : 0;
  const size_t pc_bytes = h->per_channel ? (size_t)P * 64 : 0;
  const size_t b_bytes = ec ? (size_t)P * (h->rank_b / 16) * 512 + 16 : 0;
  // barriers, alignment slack, per-channel words, u (hi and lo)
  const size_t base = kBarrierBytes + 1024 + pc_bytes + u_bytes + mlp_bytes;

  // The pipeline for kc channels per stage: stage size, stages next to the
  // fixed buffers. The B fragments of the CTA's tiles live next to the stages
  // for the whole call, unless that costs stages (rank 256: 8 KB per tile);
  // then they are copied into the stage area once the W loop has released it,
  // behind the partial sums (the reduction reuses the stage area too).
  struct StagePlan {
    int KC, n_stages, NS;
    uint32_t stage_bytes, b_late_off;
    size_t fixed;
  };
  auto stage_plan = [&](int kc) {
    StagePlan sp;
    sp.KC = kc;
    sp.stage_bytes = (uint32_t)(((size_t)kc * Mp * 2 + P * L.stage_tile_bytes(kc) + 1023) / 1024 * 1024);
    sp.n_stages = (h->K + kc - 1) / kc;
    auto stages_next_to = [&](size_t fixed, size_t area) {
      const size_t budget = kSmemCap > fixed ? kSmemCap - fixed : 0;
      int ns = (int)(budget / sp.stage_bytes);
      if (ns > kMaxStages) ns = kMaxStages;
      if (ns > sp.n_stages) ns = sp.n_stages;
      while ((size_t)ns * sp.stage_bytes < area) ++ns;
      return ns;
    };
    sp.fixed = base + b_bytes;
    sp.NS = stages_next_to(sp.fixed, red_bytes);
    sp.b_late_off = 0;
    if (ec) {
      const size_t red_al = (red_bytes + 127) / 128 * 128;
      const int ns_late = stages_next_to(base, red_al + b_bytes);
      if (ns_late > sp.NS && base + (size_t)ns_late * sp.stage_bytes <= 227 * 1024) {
        sp.fixed = base;
        sp.NS = ns_late;
        sp.b_late_off = (uint32_t)red_al;
      }
    }
    return sp;
  };
  StagePlan sp = stage_plan(KC);
  // One unit per K warp and stage where two would leave a single stage (x
  // boxes of 16 or 32 tokens at two tiles per CTA): double buffering pays
  // there, while elsewhere the two-unit stages measured faster.
  if (sp.NS < 2 && sp.n_stages > 1 && (KC / 2) % kDecodeRun == 0) {
    const StagePlan half = stage_plan(KC / 2);
    if (half.NS >= 2) sp = half;
  }
  KC = sp.KC;
  p.KC = KC;
  p.bytes_x = (uint32_t)(KC * Mp * 2);
  p.stage_bytes = sp.stage_bytes;
  p.n_stages = sp.n_stages;
  p.b_late_off = sp.b_late_off;
  const size_t fixed = sp.fixed;
  const int NS = sp.NS;
  if (NS < 1 || fixed + (size_t)NS * p.stage_bytes > 227 * 1024) return SPEAR_ERR_UNSUPPORTED;
  p.NS = NS;
  out->smem = fixed + (size_t)NS * p.stage_bytes;
  out->grid = (h->nt16 + P - 1) / P;
  out->NW = NW;
  out->MT = MT;
  out->T = T;
  out->kernel = kernel_for(NW, MT, T, h->per_channel, ec);
  if (!out->kernel.fn) return SPEAR_ERR_UNSUPPORTED;
  return SPEAR_OK;
}

}  // namespace
}  // namespace dec
}  // namespace spear

using namespace spear;
using namespace spear::dec;

spear_status_t spear_launch_decode(spear_linear_s* h, const __nv_bfloat16* x, __nv_bfloat16* y, int M,
                                   cudaStream_t stream) {
  DecodeLaunch d;
  spear_status_t st = decode_config(h, M, &d);
  if (st != SPEAR_OK) return st;
  d.p.x = x;
  d.p.y = y;
  CUtensorMap xmap;
  if (!encode_x_map(&xmap, x, M, h->K, 8 * d.MT, d.p.KC)) return SPEAR_ERR_CUDA;
  if (d.kernel.configure() != cudaSuccess) return SPEAR_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(d.grid);
  cfg.blockDim = dim3((d.NW + 1 + kEcWarps) * 32);
  cfg.dynamicSmemBytes = d.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, d.kernel.fn, d.p, xmap) == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}

// The decode kernel's CTAs wait for each other (the compensator's grid-wide
// z dependency), so a grid must fit on the device at once: one CTA per SM at
// most, with each plan's shared memory. Checked at create for every token
// count the handle accepts.
spear_status_t spear_decode_check_residency(spear_linear_s* h) {
  const int mmax = h->max_tokens < kDecodeMaxTokens ? h->max_tokens : kDecodeMaxTokens;
  for (int M : {1, 9, 17}) {
    if (M > mmax) break;
    DecodeLaunch d;
    spear_status_t st = decode_config(h, M, &d);
    if (st != SPEAR_OK) return st;
    if (d.kernel.configure() != cudaSuccess) return SPEAR_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, d.kernel.fn, (d.NW + 1 + kEcWarps) * 32, d.smem) !=
        cudaSuccess)
      return SPEAR_ERR_CUDA;
    if ((long)per_sm * h->sm_count < d.grid) return SPEAR_ERR_UNSUPPORTED;
  }
  return SPEAR_OK;
}

// Test surface: the decode launch plan of a handle of this shape, computed by
// the same host code as the launch (decode_config), with no device work.
spear_status_t spear_decode_schedule(int32_t N, int32_t K, int32_t rank_b, int32_t n_members, int32_t group_size,
                                     int32_t gate_hidden, int32_t M, int32_t sm_count, int32_t* info) {
  if (N <= 0 || K <= 0 || K % 128 != 0 || N % 8 != 0 || (group_size != 0 && group_size != 128) || rank_b < 0 ||
      rank_b % 16 != 0 || n_members < 1 || n_members > kMaxGroup || n_members * rank_b > 256 || gate_hidden < 0 ||
      gate_hidden > kMaxGateHidden || gate_hidden % 16 != 0 || (gate_hidden > 0 && rank_b == 0) || M < 1 ||
      M > kDecodeMaxTokens || sm_count < 1 || !info)
    return SPEAR_ERR_INVALID_ARG;
  spear_linear_s h;
  h.sm_count = sm_count;
  h.K = K;
  h.N = N;
  h.per_channel = group_size == 0;
  h.G = h.per_channel ? K : group_size;
  h.n_groups = K / h.G;
  h.n_members = n_members;
  h.rank_b = rank_b;
  h.rank = n_members * rank_b;
  for (int i = 0; i <= n_members; ++i) h.row_start[i] = (int)((int64_t)N * i / n_members);
  h.gate = gate_hidden > 0 ? SPEAR_GATE_MLP : SPEAR_GATE_SIGMOID;
  h.gate_hidden = gate_hidden;
  h.max_tokens = kDecodeMaxTokens;
  const int nt16_rows = (N + 15) / 16;
  if ((nt16_rows + sm_count - 1) / sm_count > kDecodeMaxTilesPerCta) return SPEAR_ERR_UNSUPPORTED;
  h.dec_P = decode_tiles_per_cta(nt16_rows, sm_count);
  h.nt16 = (nt16_rows + h.dec_P - 1) / h.dec_P * h.dec_P;
  DecodeLaunch d;
  const spear_status_t st = decode_config(&h, M, &d);
  if (st != SPEAR_OK) return st;
  const int32_t v[13] = {d.grid,
                         d.p.P,
                         d.NW,
                         d.T,
                         d.MT,
                         d.p.KW,
                         d.p.KC,
                         d.p.NS,
                         (int32_t)d.p.stage_bytes,
                         (int32_t)d.smem,
                         d.p.n_stages,
                         (d.NW + 1 + kEcWarps) * 32,
                         (int32_t)d.p.bytes_x};
  for (int i = 0; i < 13; ++i) info[i] = v[i];
  return SPEAR_OK;
}
