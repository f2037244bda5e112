// C ABI of the library: argument checking, handle lifetime, phase dispatch.
// All arithmetic of the layer runs in the kernels of decode.cu, prefill.cu and
// layout.cu; this file only validates, allocates at create and launches.
#include <cudaTypedefs.h>

#include <mutex>
#include <new>

#include "internal.h"

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return encode;
}

bool encode_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                    uint32_t box_inner, uint32_t box_rows) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_x_map(CUtensorMap* map, const void* x, int M, int K, int Mp, int KC) {
  auto encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[3] = {64, (cuuint64_t)M, (cuuint64_t)(K / 64)};
  const cuuint64_t strides[2] = {(cuuint64_t)K * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)Mp, (cuuint32_t)(KC / 64)};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <typename T>
cudaError_t alloc(T** p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) return cudaSuccess;
  return cudaMalloc(reinterpret_cast<void**>(p), bytes);
}

void free_all(spear_linear_s* h) {
  void* ptrs[] = {h->wq_dec, h->sz_dec,  h->a_dec,   h->b_dec,   h->wq_pre,  h->a_pre,
                  h->b_pre,  h->ws,      h->x_stage, h->y_stage, h->gate_w1, h->gate_w2, h->y32};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  for (cudaEvent_t ev : {h->ev_fork, h->ev_join, h->ev_start, h->ev_x_ready, h->ev_done, h->ev_y_taken})
    if (ev) cudaEventDestroy(ev);
  for (cudaStream_t st : {h->copy_in, h->copy_out})
    if (st) cudaStreamDestroy(st);
}

spear_status_t validate(const spear_linear_desc_t* d) {
  if (!d) return SPEAR_ERR_INVALID_ARG;
  if (d->K <= 0 || d->N <= 0 || d->K % 128 != 0 || d->N % 8 != 0) return SPEAR_ERR_INVALID_ARG;
  if (d->group_size != 0 && d->group_size != 128) return SPEAR_ERR_INVALID_ARG;
  if (!d->qweight || !d->scales) return SPEAR_ERR_INVALID_ARG;
  if (d->rank < 0 || d->rank > 256 || d->rank % 16 != 0) return SPEAR_ERR_INVALID_ARG;
  if (d->rank > 0 && (!d->A || !d->B)) return SPEAR_ERR_INVALID_ARG;
  if (d->gate != SPEAR_GATE_SIGMOID && d->gate != SPEAR_GATE_ONE && d->gate != SPEAR_GATE_MLP)
    return SPEAR_ERR_INVALID_ARG;
  if (d->gate == SPEAR_GATE_MLP) {
    if (d->rank == 0 || d->gate_hidden < 1 || d->gate_hidden > kMaxGateHidden || !d->gate_w1 || !d->gate_w2 ||
        !aligned16(d->gate_w1) || !aligned16(d->gate_w2))
      return SPEAR_ERR_INVALID_ARG;
  }
  if (d->max_tokens < 1) return SPEAR_ERR_INVALID_ARG;
  return SPEAR_OK;
}

spear_status_t check_io(spear_linear_t h, const void* x, void* y, int32_t M) {
  if (!h || M < 0) return SPEAR_ERR_INVALID_ARG;
  if (M == 0) return SPEAR_OK;
  if (!x || !y || M > h->max_tokens) return SPEAR_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y)) return SPEAR_ERR_INVALID_ARG;
  const char* xb = static_cast<const char*>(x);
  const char* yb = static_cast<const char*>(y);
  const size_t xs = (size_t)M * h->K * 2, ys = (size_t)M * h->N * 2;
  if (xb < yb + ys && yb < xb + xs) return SPEAR_ERR_INVALID_ARG;  // y overlaps x
  return SPEAR_OK;
}

// Members of a grouped handle (a group of one for spear_linear_create).
struct GroupInfo {
  int n = 1;
  int rank_b = 0;                      // each member's compensator rank
  int row_start[kMaxGroup + 1] = {};   // first output row of each member, then N
  float alphas[kMaxGroup] = {};
  const void* B_rows = nullptr;        // [N][rank_b]: the members' B, one after the other
};

spear_status_t create_impl(const spear_linear_desc_t* d, const GroupInfo& g, cudaStream_t stream, spear_linear_t* out) {
  *out = nullptr;

  spear_linear_s* h = new (std::nothrow) spear_linear_s();
  if (!h) return SPEAR_ERR_OOM;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    delete h;
    return SPEAR_ERR_CUDA;
  }
  h->K = d->K;
  h->N = d->N;
  h->per_channel = d->group_size == 0;
  h->G = h->per_channel ? d->K : d->group_size;
  h->n_groups = h->K / h->G;
  h->rank = d->rank;
  h->alpha = d->alpha;
  h->n_members = g.n;
  h->rank_b = g.rank_b;
  for (int i = 0; i <= g.n; ++i) h->row_start[i] = g.row_start[i];
  for (int i = 0; i < g.n; ++i) h->alphas[i] = g.alphas[i];
  h->gate = d->gate;
  // zero-padded to a multiple of 16 hidden units (one MMA k step): the extra
  // units are relu(0) = 0 and meet zero columns of W2
  h->gate_hidden = d->gate == SPEAR_GATE_MLP ? (d->gate_hidden + 15) / 16 * 16 : 0;
  h->max_tokens = d->max_tokens;
  const int nt16_rows = (h->N + 15) / 16;  // 16-row tiles holding output rows
  h->nt128 = (h->N + 127) / 128;
  if ((nt16_rows + h->sm_count - 1) / h->sm_count > kDecodeMaxTilesPerCta) {
    delete h;
    return SPEAR_ERR_UNSUPPORTED;
  }
  h->dec_P = decode_tiles_per_cta(nt16_rows, h->sm_count);
  // every decode CTA owns exactly dec_P tiles: the layout is padded with
  // zero tiles (rows past N, scale 0) up to whole CTAs
  h->nt16 = (nt16_rows + h->dec_P - 1) / h->dec_P * h->dec_P;
  h->dec_tile_bytes = DecodeLayout{h->K, h->nt16, h->dec_P, h->per_channel}.tile_bytes();

  const size_t K = h->K, r = h->rank, mt = h->max_tokens;
  const size_t pre_tiles = (mt + 127) / 128;
  // prefill compensator: z [pre_tiles * 128][rank] fp32 (rows past the tokens
  // stay zero), u' [max_tokens][rank] bf16, per 128-token tile a split
  // counter and a "u' ready" flag, and the count of finished CTAs
  const size_t ws_base =
      sizeof(spear::SyncWords) + kZDecFloats * 4 + pre_tiles * 128 * r * 4 + mt * r * 2 + pre_tiles * 8 + 4;
  const size_t z_mma_off = (ws_base + 127) / 128 * 128;
  // Prefill's stream-K schedule: one fp32 partial tile of 128 rows x 256
  // tokens and one flag per CTA (at most sm_count), for handles sized for
  // more than decode token counts.
  const bool want_part = mt > (size_t)kDecodeMaxTokens;
  const size_t part_off = z_mma_off + 2 * kZDecFloats * 4;
  const size_t part_floats = want_part ? (size_t)h->sm_count * 128 * 256 : 0;
  const size_t cnt_off = part_off + part_floats * 4;
  const size_t ws_bytes = cnt_off + (size_t)h->sm_count * 4;
  h->ws_bytes = ws_bytes;
  cudaError_t e = cudaSuccess;
  auto A = [&](cudaError_t x) {
    if (e == cudaSuccess) e = x;
  };
  A(alloc(&h->wq_dec, (size_t)h->nt16 * h->dec_tile_bytes));
  if (h->per_channel) A(alloc(&h->sz_dec, (size_t)h->nt16 * 16 * 4));
  A(alloc(&h->wq_pre, (size_t)h->nt128 * (K / 64) * kPrefillBlockWords * 4));
  if (r > 0) {
    A(alloc(&h->a_dec, (r / 16) * (K / 16) * 32 * 16));
    A(alloc(&h->b_dec, (size_t)h->nt16 * (h->rank_b / 16) * 32 * 16));
    A(alloc(&h->a_pre, r * K * 2));
    A(alloc(&h->b_pre, (size_t)h->nt128 * 128 * r * 2));
  }
  if (h->gate_hidden > 0) {
    A(alloc(&h->gate_w1, (size_t)h->gate_hidden * r * 2));
    A(alloc(&h->gate_w2, (size_t)h->gate_hidden * r * 2));
  }
  A(alloc(&h->ws, ws_bytes));
  A(alloc(&h->x_stage, mt * K * 2));
  A(alloc(&h->y_stage, mt * (size_t)h->N * 2));
  if (e != cudaSuccess) {
    cudaGetLastError();
    free_all(h);
    delete h;
    return e == cudaErrorMemoryAllocation ? SPEAR_ERR_OOM : SPEAR_ERR_CUDA;
  }
  char* w = static_cast<char*>(h->ws);
  h->sync = reinterpret_cast<spear::SyncWords*>(w);
  h->z_dec = reinterpret_cast<float*>(w + sizeof(spear::SyncWords));
  h->z_mma = reinterpret_cast<float*>(w + z_mma_off);
  h->part = want_part ? reinterpret_cast<float*>(w + part_off) : nullptr;
  h->part_cnt = reinterpret_cast<unsigned*>(w + cnt_off);
  h->z_pre = h->z_dec + kZDecFloats;
  h->u_pre = reinterpret_cast<__nv_bfloat16*>(h->z_pre + pre_tiles * 128 * r);
  h->pre_done = reinterpret_cast<unsigned*>(h->u_pre + mt * r);
  h->u_ready = h->pre_done + pre_tiles;
  h->pf_done = h->u_ready + pre_tiles;

  spear_status_t st = SPEAR_OK;
  if (cudaMemsetAsync(h->ws, 0, ws_bytes, stream) != cudaSuccess) st = SPEAR_ERR_CUDA;
  if (st == SPEAR_OK) st = spear_build_layouts(h, d, g.B_rows, stream);
  if (st == SPEAR_OK && h->gate_hidden > 0) {
    const size_t h8 = h->gate_hidden, hu = d->gate_hidden;
    if (cudaMemsetAsync(h->gate_w1, 0, h8 * r * 2, stream) != cudaSuccess ||
        cudaMemsetAsync(h->gate_w2, 0, h8 * r * 2, stream) != cudaSuccess ||
        cudaMemcpyAsync(h->gate_w1, d->gate_w1, hu * r * 2, cudaMemcpyDeviceToDevice, stream) != cudaSuccess ||
        cudaMemcpy2DAsync(h->gate_w2, h8 * 2, d->gate_w2, hu * 2, hu * 2, r, cudaMemcpyDeviceToDevice, stream) !=
            cudaSuccess)
      st = SPEAR_ERR_CUDA;
  }
  if (st == SPEAR_OK && cudaStreamSynchronize(stream) != cudaSuccess) st = SPEAR_ERR_CUDA;
  if (st == SPEAR_OK) st = spear_decode_check_residency(h);
  if (st != SPEAR_OK) {
    cudaGetLastError();
    free_all(h);
    delete h;
    return st;
  }
  *out = h;
  return SPEAR_OK;
}

}  // namespace

extern "C" {

spear_status_t spear_linear_create(const spear_linear_desc_t* d, cudaStream_t stream, spear_linear_t* out) {
  if (!out) return SPEAR_ERR_INVALID_ARG;
  *out = nullptr;
  spear_status_t v = validate(d);
  if (v != SPEAR_OK) return v;
  GroupInfo g;
  g.rank_b = d->rank;
  g.row_start[1] = d->N;
  g.alphas[0] = d->alpha;
  g.B_rows = d->B;
  return create_impl(d, g, stream, out);
}

spear_status_t spear_linear_create_grouped(const spear_linear_desc_t* descs, int32_t n, cudaStream_t stream,
                                           spear_linear_t* out) {
  if (!out) return SPEAR_ERR_INVALID_ARG;
  *out = nullptr;
  if (!descs || n < 1 || n > kMaxGroup) return SPEAR_ERR_INVALID_ARG;
  if (n == 1) return spear_linear_create(descs, stream, out);
  const spear_linear_desc_t& d0 = descs[0];
  int n_tot = 0, max_tokens = 0;
  bool any_zeros = false;
  for (int32_t i = 0; i < n; ++i) {
    const spear_linear_desc_t& d = descs[i];
    spear_status_t v = validate(&d);
    if (v != SPEAR_OK) return v;
    if (d.K != d0.K || d.group_size != d0.group_size || d.rank != d0.rank || d.gate != d0.gate || d.N % 16 != 0)
      return SPEAR_ERR_INVALID_ARG;
    if (d.gate == SPEAR_GATE_MLP) return SPEAR_ERR_UNSUPPORTED;
    n_tot += d.N;
    max_tokens = d.max_tokens > max_tokens ? d.max_tokens : max_tokens;
    any_zeros = any_zeros || d.zeros != nullptr;
  }
  const int r = d0.rank, K = d0.K, ng = d0.group_size == 0 ? 1 : K / d0.group_size;
  if (n * r > 256) return SPEAR_ERR_INVALID_ARG;
  // The members' weights side by side in temporary buffers (freed once the
  // layouts are built; create_impl synchronises the stream before returning).
  uint8_t *q = nullptr, *z = nullptr;
  void *s = nullptr, *A = nullptr, *B = nullptr;
  cudaError_t e = cudaSuccess;
  auto chk = [&](cudaError_t x) {
    if (e == cudaSuccess) e = x;
  };
  chk(alloc(&q, (size_t)n_tot * K / 2));
  chk(alloc(reinterpret_cast<uint8_t**>(&s), (size_t)n_tot * ng * 2));
  if (any_zeros) chk(alloc(&z, (size_t)n_tot * ng));
  if (r > 0) {
    chk(alloc(reinterpret_cast<uint8_t**>(&A), (size_t)n * r * K * 2));
    chk(alloc(reinterpret_cast<uint8_t**>(&B), (size_t)n_tot * r * 2));
  }
  GroupInfo g;
  g.n = n;
  g.rank_b = r;
  g.B_rows = B;
  size_t row = 0;
  for (int32_t i = 0; i < n && e == cudaSuccess; ++i) {
    const spear_linear_desc_t& d = descs[i];
    g.row_start[i] = (int)row;
    g.alphas[i] = d.alpha;
    chk(cudaMemcpyAsync(q + row * K / 2, d.qweight, (size_t)d.N * K / 2, cudaMemcpyDeviceToDevice, stream));
    chk(cudaMemcpyAsync(static_cast<uint8_t*>(s) + row * ng * 2, d.scales, (size_t)d.N * ng * 2,
                        cudaMemcpyDeviceToDevice, stream));
    if (any_zeros)
      chk(d.zeros ? cudaMemcpyAsync(z + row * ng, d.zeros, (size_t)d.N * ng, cudaMemcpyDeviceToDevice, stream)
                  : cudaMemsetAsync(z + row * ng, 8, (size_t)d.N * ng, stream));  // no zeros: z = 8
    if (r > 0) {
      chk(cudaMemcpyAsync(static_cast<uint8_t*>(A) + (size_t)i * r * K * 2, d.A, (size_t)r * K * 2,
                          cudaMemcpyDeviceToDevice, stream));
      chk(cudaMemcpyAsync(static_cast<uint8_t*>(B) + row * r * 2, d.B, (size_t)d.N * r * 2,
                          cudaMemcpyDeviceToDevice, stream));
    }
    row += d.N;
  }
  g.row_start[n] = n_tot;
  spear_status_t st = SPEAR_ERR_CUDA;
  if (e == cudaSuccess) {
    spear_linear_desc_t d = d0;
    d.N = n_tot;
    d.qweight = q;
    d.scales = s;
    d.zeros = z;
    d.rank = n * r;
    d.A = A;
    d.B = B;  // validated as present; the layouts take B from g.B_rows
    d.max_tokens = max_tokens;
    st = validate(&d);
    if (st == SPEAR_OK) st = create_impl(&d, g, stream, out);
  } else {
    st = e == cudaErrorMemoryAllocation ? SPEAR_ERR_OOM : SPEAR_ERR_CUDA;
    cudaGetLastError();
    cudaStreamSynchronize(stream);
  }
  for (void* p : {static_cast<void*>(q), s, static_cast<void*>(z), A, B})
    if (p) cudaFree(p);
  return st;
}

spear_status_t spear_linear_forward_decode(spear_linear_t h, const void* x, void* y, int32_t M,
                                           cudaStream_t stream) {
  spear_status_t v = check_io(h, x, y, M);
  if (v != SPEAR_OK || M == 0) return v;
  if (M > kDecodeMaxTokens) return SPEAR_ERR_INVALID_ARG;
  const auto* xb = static_cast<const __nv_bfloat16*>(x);
  auto* yb = static_cast<__nv_bfloat16*>(y);
  return spear_launch_decode(h, xb, yb, M, stream);
}

spear_status_t spear_linear_forward_prefill(spear_linear_t h, const void* x, void* y, int32_t M,
                                            cudaStream_t stream) {
  spear_status_t v = check_io(h, x, y, M);
  if (v != SPEAR_OK || M == 0) return v;
  return spear_launch_prefill(h, static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), M,
                              stream);
}

spear_status_t spear_linear_enable_concurrent_ec(spear_linear_t h) {
  if (!h) return SPEAR_ERR_INVALID_ARG;
  if (h->y32) return SPEAR_OK;
  if (h->rank == 0) return SPEAR_OK;  // nothing runs beside the main contraction
  float* y32 = nullptr;
  cudaEvent_t a = nullptr, b = nullptr;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&y32), (size_t)h->max_tokens * h->N * 4);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&a, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    cudaGetLastError();
    if (y32) cudaFree(y32);
    if (a) cudaEventDestroy(a);
    if (b) cudaEventDestroy(b);
    return e == cudaErrorMemoryAllocation ? SPEAR_ERR_OOM : SPEAR_ERR_CUDA;
  }
  h->y32 = y32;
  h->ev_fork = a;
  h->ev_join = b;
  return SPEAR_OK;
}

spear_status_t spear_linear_forward_prefill_concurrent(spear_linear_t h, const void* x, void* y, int32_t M,
                                                       cudaStream_t stream, cudaStream_t ec_stream) {
  spear_status_t v = check_io(h, x, y, M);
  if (v != SPEAR_OK || M == 0) return v;
  if (h->rank > 0 && (!h->y32 || ec_stream == stream)) return SPEAR_ERR_INVALID_ARG;
  return spear_launch_prefill_concurrent(h, static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y),
                                         M, stream, ec_stream);
}

spear_status_t spear_linear_forward(spear_linear_t h, const void* x, void* y, int32_t M, cudaStream_t stream) {
  if (M <= kDecodeMaxTokens) return spear_linear_forward_decode(h, x, y, M, stream);
  return spear_linear_forward_prefill(h, x, y, M, stream);
}

spear_status_t spear_linear_forward_host(spear_linear_t h, const void* x_host, void* y_host, int32_t M,
                                         cudaStream_t stream) {
  if (!h || M < 0) return SPEAR_ERR_INVALID_ARG;
  if (M == 0) return SPEAR_OK;
  if (!x_host || !y_host || M > h->max_tokens) return SPEAR_ERR_INVALID_ARG;
  const size_t xb = (size_t)M * h->K * 2, yb = (size_t)M * h->N * 2;
  if (cudaMemcpyAsync(h->x_stage, x_host, xb, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return SPEAR_ERR_CUDA;
  spear_status_t s = spear_linear_forward(h, h->x_stage, h->y_stage, M, stream);
  if (s != SPEAR_OK) return s;
  if (cudaMemcpyAsync(y_host, h->y_stage, yb, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return SPEAR_ERR_CUDA;
  return cudaStreamSynchronize(stream) == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}

// The copy streams and events of the host-buffer batch path, made on a
// handle's first batch (most handles never use that path).
static cudaError_t host_batch_sync_objects(spear_linear_s* h, bool streams) {
  cudaError_t e = cudaSuccess;
  for (cudaEvent_t* ev : {&h->ev_start, &h->ev_x_ready, &h->ev_done, &h->ev_y_taken})
    if (e == cudaSuccess && !*ev) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (streams)
    for (cudaStream_t* st : {&h->copy_in, &h->copy_out})
      if (e == cudaSuccess && !*st) e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking);
  return e;
}

spear_status_t spear_linear_forward_host_batch(const spear_linear_t* hs, const void* const* x_host,
                                               void* const* y_host, const int32_t* Ms, int32_t n,
                                               cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!hs || !x_host || !y_host || !Ms))) return SPEAR_ERR_INVALID_ARG;
  if (n == 0) return SPEAR_OK;
  // every argument is checked before anything is enqueued
  for (int32_t i = 0; i < n; ++i) {
    const spear_linear_t h = hs[i];
    if (!h || Ms[i] < 0 || Ms[i] > h->max_tokens) return SPEAR_ERR_INVALID_ARG;
    if (Ms[i] > 0 && (!x_host[i] || !y_host[i])) return SPEAR_ERR_INVALID_ARG;
  }
  // Inputs go up on one copy stream and results down on another (those of
  // hs[0]), so that copies overlap the forwards on `stream`. Per handle,
  // events order each call's steps: its input copy after the previous
  // forward on the handle has read the staging buffer (ev_done), its forward
  // after that copy (ev_x_ready) and after the previous result left the
  // staging buffer (ev_y_taken), its result copy after the forward. Every
  // wait is on an earlier call, so nothing waits in a cycle; the copy streams
  // start after the work already on `stream`.
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  for (int32_t k = 0; k < n; ++k)
    if (!ok(host_batch_sync_objects(hs[k], k == 0))) return SPEAR_ERR_CUDA;
  cudaStream_t cin = hs[0]->copy_in, cout = hs[0]->copy_out;
  if (!ok(cudaEventRecord(hs[0]->ev_start, stream)) || !ok(cudaStreamWaitEvent(cin, hs[0]->ev_start, 0)) ||
      !ok(cudaStreamWaitEvent(cout, hs[0]->ev_start, 0)))
    return SPEAR_ERR_CUDA;
  for (int32_t k = 0; k < n; ++k) {
    const spear_linear_t h = hs[k];
    if (Ms[k] == 0) continue;
    bool again = false;  // an earlier call of this batch used the handle
    for (int32_t j = 0; j < k && !again; ++j) again = hs[j] == h && Ms[j] > 0;
    if ((again && !ok(cudaStreamWaitEvent(cin, h->ev_done, 0))) ||
        !ok(cudaMemcpyAsync(h->x_stage, x_host[k], (size_t)Ms[k] * h->K * 2, cudaMemcpyHostToDevice, cin)) ||
        !ok(cudaEventRecord(h->ev_x_ready, cin)) || !ok(cudaStreamWaitEvent(stream, h->ev_x_ready, 0)) ||
        (again && !ok(cudaStreamWaitEvent(stream, h->ev_y_taken, 0))))
      return SPEAR_ERR_CUDA;
    const spear_status_t s = spear_linear_forward(h, h->x_stage, h->y_stage, Ms[k], stream);
    if (s != SPEAR_OK) return s;
    if (!ok(cudaEventRecord(h->ev_done, stream)) || !ok(cudaStreamWaitEvent(cout, h->ev_done, 0)) ||
        !ok(cudaMemcpyAsync(y_host[k], h->y_stage, (size_t)Ms[k] * h->N * 2, cudaMemcpyDeviceToHost, cout)) ||
        !ok(cudaEventRecord(h->ev_y_taken, cout)))
      return SPEAR_ERR_CUDA;
  }
  if (!ok(cudaStreamSynchronize(cin)) || !ok(cudaStreamSynchronize(cout))) return SPEAR_ERR_CUDA;
  return cudaStreamSynchronize(stream) == cudaSuccess ? SPEAR_OK : SPEAR_ERR_CUDA;
}

spear_status_t spear_linear_destroy(spear_linear_t h) {
  if (!h) return SPEAR_OK;
  // cudaFree itself waits for the work already queued on the device, so a
  // forward still in flight never sees its buffers freed under it.
  free_all(h);
  delete h;
  return SPEAR_OK;
}

spear_status_t spear_linear_dequantize(spear_linear_t h, int32_t path, void* w_out, cudaStream_t stream) {
  if (!h || !w_out || (path != 0 && path != 1) || !aligned16(w_out)) return SPEAR_ERR_INVALID_ARG;
  return spear_launch_dequant(h, path, static_cast<__nv_bfloat16*>(w_out), stream);
}

spear_status_t spear_linear_check(spear_linear_t h, cudaStream_t stream) {
  if (!h) return SPEAR_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SPEAR_ERR_CUDA;
  unsigned status = 0;
  if (cudaMemcpy(&status, &h->sync->status, sizeof status, cudaMemcpyDeviceToHost) != cudaSuccess)
    return SPEAR_ERR_CUDA;
  if (status == 0) return SPEAR_OK;
  // Reset the workspace (counters, status, accumulators) so the handle is usable again.
  if (cudaMemset(h->ws, 0, h->ws_bytes) != cudaSuccess) return SPEAR_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return SPEAR_ERR_CUDA;
  return SPEAR_ERR_TIMEOUT;
}

spear_status_t spear_linear_debug_set(spear_linear_t h, int64_t wait_ns, int32_t skip_arrive) {
  if (!h || wait_ns < 0) return SPEAR_ERR_INVALID_ARG;
  h->wait_ns = wait_ns == 0 ? 100000000ull : (uint64_t)wait_ns;
  h->skip_arrive = skip_arrive != 0;
  return SPEAR_OK;
}

const char* spear_status_string(spear_status_t s) {
  switch (s) {
    case SPEAR_OK: return "SPEAR_OK";
    case SPEAR_ERR_INVALID_ARG: return "SPEAR_ERR_INVALID_ARG";
    case SPEAR_ERR_UNSUPPORTED: return "SPEAR_ERR_UNSUPPORTED";
    case SPEAR_ERR_OOM: return "SPEAR_ERR_OOM";
    case SPEAR_ERR_CUDA: return "SPEAR_ERR_CUDA";
    case SPEAR_ERR_TIMEOUT: return "SPEAR_ERR_TIMEOUT";
  }
  return "SPEAR_ERR_UNKNOWN";
}

}  // extern "C"
