// moe_api.cu -- the C ABI declared in include/moe.h: host-side validation, the layout of
// the caller-owned workspace and forward context, and the order in which the layer's
// kernels are enqueued.  Nothing here allocates device memory or waits for the device
// (except moe_status).
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "internal.h"

using namespace moe;

namespace {

constexpr size_t ALIGN = 256;

size_t align_up(size_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }

moe_status_t validate(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T <= 0 || c->E <= 0 || c->k <= 0 || c->k > c->E || c->d <= 0 || c->ffn <= 0 ||
      c->ffn_shared < 0 || c->capacity < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->gate != MOE_GATE_SOFTMAX_TOPK && c->gate != MOE_GATE_SIGMOID_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->route_scale)) return MOE_ERR_INVALID_ARG;
  if ((c->drop_negative != 0 && c->drop_negative != 1) ||
      (c->recompute != 0 && c->recompute != 1) ||
      (c->drop_by_score != 0 && c->drop_by_score != 1) || (c->mxfp8 < 0 || c->mxfp8 > 2))
    return MOE_ERR_INVALID_ARG;
  if (c->select_bias && (reinterpret_cast<uintptr_t>(c->select_bias) & 3u))
    return MOE_ERR_INVALID_ARG;
  if (c->E > 256 || c->k > 8) return MOE_ERR_UNSUPPORTED;
  if (c->d % 64 || c->ffn % 64 || c->ffn_shared % 64) return MOE_ERR_UNSUPPORTED;
  // MXFP8: K blocks of 128 elements; the backward's FC1 rerun would be bf16, not MXFP8
  if (c->mxfp8 && (c->d % 128 || c->ffn % 128 || c->recompute)) return MOE_ERR_UNSUPPORTED;
  if (c->T * static_cast<int64_t>(c->k) >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  // 2f rows x d of one expert must be addressable with int32 tile coordinates
  if (static_cast<int64_t>(c->E) * 2 * c->ffn >= (int64_t(1) << 31) ||
      static_cast<int64_t>(c->E) * c->d >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// every pointer must be non-null and 16-byte aligned
template <typename... P>
bool ptrs_ok(P... ps) {
  const void* arr[] = {static_cast<const void*>(ps)...};
  for (const void* p : arr)
    if (!p || !aligned16(p)) return false;
  return true;
}

struct CtxLayout {
  size_t off[MOE_CTX_NFIELDS];
  size_t total;
};

CtxLayout ctx_layout(const moe_config_t* c) {
  const size_t T = static_cast<size_t>(c->T), k = c->k, E = c->E, d = c->d, f = c->ffn,
               fs = c->ffn_shared;
  const size_t R = T * k;
  size_t sz[MOE_CTX_NFIELDS];
  sz[MOE_CTX_TOPK_IDX] = R * 4;
  sz[MOE_CTX_TOPK_W] = R * 4;
  sz[MOE_CTX_COUNTS] = E * 4;
  sz[MOE_CTX_KEPT] = E * 4;
  sz[MOE_CTX_OFFSETS] = (E + 1) * 4;
  sz[MOE_CTX_DEST_ROW] = R * 4;
  sz[MOE_CTX_SRC_TOK] = R * 4;
  sz[MOE_CTX_SRC_SLOT] = R * 4;
  sz[MOE_CTX_DROP_MASK] = R;
  sz[MOE_CTX_XP] = R * d * 2;
  const bool keep_act = !c->recompute;   // with recompute, FC1's outputs live in ws
  sz[MOE_CTX_AB] = keep_act ? R * 2 * f * 2 : 0;
  sz[MOE_CTX_H] = keep_act ? R * f * 2 : 0;
  sz[MOE_CTX_YP] = R * d * 2;
  sz[MOE_CTX_AB_S] = keep_act ? T * 2 * fs * 2 : 0;
  sz[MOE_CTX_H_S] = keep_act ? T * fs * 2 : 0;
  sz[MOE_CTX_YS] = fs ? T * d * 2 : 0;
  CtxLayout L;
  size_t o = 0;
  for (int i = 0; i < MOE_CTX_NFIELDS; ++i) {
    L.off[i] = o;
    o += align_up(sz[i]);
  }
  L.total = o;
  return L;
}

struct WsLayout {
  size_t route, maps, dyp, dab, dxp, dab_s, dx_s, ab, h, ab_s, h_s, xq, x_sf, hq, h_sf, dyq,
      dy_sf, dabq, dab_sf, dyT, dyT_sf, hT, hT_sf, dabT, dabT_sf, xpT, xpT_sf, total;
};

WsLayout ws_layout(const moe_config_t* c) {
  const size_t T = static_cast<size_t>(c->T), k = c->k, d = c->d, f = c->ffn,
               fs = c->ffn_shared;
  const size_t R = T * k;
  WsLayout L;
  size_t o = WS_HEADER_BYTES;
  L.route = o; o += align_up(route_scratch_bytes(c));
  L.maps = o;  o += align_up(2 * static_cast<size_t>(c->E) * SEG_MAP_BYTES);
  L.dyp = o;   o += align_up(R * d * 2);
  L.dab = o;   o += align_up(R * 2 * f * 2);
  L.dxp = o;   o += align_up(R * d * 2);
  L.dab_s = o; o += align_up(T * 2 * fs * 2);
  L.dx_s = o;  o += align_up(fs ? T * d * 2 : 0);
  // selective rematerialisation: FC1's outputs are scratch, recomputed by the backward
  const bool rc = c->recompute != 0;
  L.ab = o;    o += align_up(rc ? R * 2 * f * 2 : 0);
  L.h = o;     o += align_up(rc ? R * f * 2 : 0);
  L.ab_s = o;  o += align_up(rc ? T * 2 * fs * 2 : 0);
  L.h_s = o;   o += align_up(rc ? T * fs * 2 : 0);
  // MXFP8 forward: the quantised activations and their scales
  const bool mx = c->mxfp8 != 0;
  L.xq = o;    o += align_up(mx ? R * d : 0);
  L.x_sf = o;  o += align_up(mx ? mx_act_scale_bytes(c->T * c->k, c->E, c->d) : 0);
  L.hq = o;    o += align_up(mx ? R * f : 0);
  L.h_sf = o;  o += align_up(mx ? mx_act_scale_bytes(c->T * c->k, c->E, c->ffn) : 0);
  // ... and the backward's: dyp and dab in MXFP8
  L.dyq = o;   o += align_up(mx ? R * d : 0);
  L.dy_sf = o; o += align_up(mx ? mx_act_scale_bytes(c->T * c->k, c->E, c->d) : 0);
  L.dabq = o;  o += align_up(mx ? R * 2 * f : 0);
  L.dab_sf = o; o += align_up(mx ? mx_act_scale_bytes(c->T * c->k, c->E, 2 * c->ffn) : 0);
  // ... and with mxfp8 = 2 the weight gradients' operands, quantised along the tokens:
  // dW2 = dyp^T h (dyp the M operand, h the N operand), dW1 = dab^T xp
  const bool mw = c->mxfp8 == 2;
  const int64_t Rc = c->T * c->k;
  const int E = c->E, D = c->d, F = c->ffn;
  L.dyT = o;     o += align_up(mw ? mx_tok_codes_bytes(Rc, E, D) : 0);
  L.dyT_sf = o;  o += align_up(mw ? mx_tok_scale_bytes(Rc, E, D, false) : 0);
  L.hT = o;      o += align_up(mw ? mx_tok_codes_bytes(Rc, E, F) : 0);
  L.hT_sf = o;   o += align_up(mw ? mx_tok_scale_bytes(Rc, E, F, true) : 0);
  L.dabT = o;    o += align_up(mw ? mx_tok_codes_bytes(Rc, E, 2 * F) : 0);
  L.dabT_sf = o; o += align_up(mw ? mx_tok_scale_bytes(Rc, E, 2 * F, false) : 0);
  L.xpT = o;     o += align_up(mw ? mx_tok_codes_bytes(Rc, E, D) : 0);
  L.xpT_sf = o;  o += align_up(mw ? mx_tok_scale_bytes(Rc, E, D, true) : 0);
  L.total = o;
  return L;
}

template <typename T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}
template <typename T>
const T* at(const void* base, size_t off) {
  return reinterpret_cast<const T*>(static_cast<const uint8_t*>(base) + off);
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                                        \
  do {                                                       \
    cudaError_t e_ = (expr);                                 \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA;              \
  } while (0)

GroupedGemmArgs gemm_args(int mode, const moe_config_t* c, const int32_t* offsets,
                          int64_t uniform_rows, int d, int f, const void* A, const void* B,
                          void* out0, void* out1, const void* aux, int* err) {
  GroupedGemmArgs a{};
  a.mode = mode;
  a.offsets = offsets;
  a.G = uniform_rows > 0 ? 1 : c->E;
  a.uniform_rows = uniform_rows;
  a.rows_cap = uniform_rows > 0 ? uniform_rows : c->T * c->k;
  a.d = d;
  a.f = f;
  a.A = A;
  a.B = B;
  a.out0 = out0;
  a.out1 = out1;
  a.aux = aux;
  a.err = err;
  return a;
}

// Rows of the FC1 input taken from x through src_tok (the fused permute), or none.
struct Gather {
  const int32_t* idx = nullptr;
  const void* src = nullptr;
  int64_t rows = 0;
};

void set_gather(GroupedGemmArgs& a, const Gather& gx) {
  a.gather_idx = gx.idx;
  a.gather_src = gx.src;
  a.gather_rows = gx.rows;
}

moe_status_t ffn_fwd(const moe_config_t* c, const void* xp, const int32_t* offsets,
                     int64_t uniform_rows, int f, const void* W1, const void* W2, void* ab,
                     void* h, void* yp, int* err, cudaStream_t st, Gather gx = {}) {
  GroupedGemmArgs a1 = gemm_args(GEMM_FC1_SWIGLU, c, offsets, uniform_rows, c->d, f, xp, W1, ab,
                                 h, nullptr, err);
  set_gather(a1, gx);
  MOE_TRY(launch_grouped_gemm(a1, st));
  GroupedGemmArgs a2 =
      gemm_args(GEMM_FC2, c, offsets, uniform_rows, c->d, f, h, W2, yp, nullptr, nullptr, err);
  MOE_TRY(launch_grouped_gemm(a2, st));
  return MOE_OK;
}

// The FC2 data-gradient's rows taken from dy through src_tok, each scaled by its slot's
// gate weight in the epilogue (the dispatch of dy fused into that GEMM), or none.
struct DyDispatch {
  Gather rows;
  const float* topk_w = nullptr;
  const int32_t* src_slot = nullptr;
  int64_t n_slots = 0;
};

moe_status_t ffn_bwd(const moe_config_t* c, const void* dyp, const void* xp,
                     const int32_t* offsets, int64_t uniform_rows, int f, const void* W1,
                     const void* W2, const void* ab, const void* h, void* dab, void* dxp,
                     void* dW1, void* dW2, void* seg_maps, int* err, cudaStream_t st,
                     Gather gx = {}, DyDispatch gd = {}) {
  GroupedGemmArgs g2 = gemm_args(GEMM_DGRAD2_SWIGLU, c, offsets, uniform_rows, c->d, f, dyp, W2,
                                 dab, nullptr, ab, err);
  if (gd.rows.idx) {
    set_gather(g2, gd.rows);
    g2.gate_w = gd.topk_w;
    g2.gate_slot = gd.src_slot;
    g2.n_slots = gd.n_slots;
  }
  MOE_TRY(launch_grouped_gemm(g2, st));
  GroupedGemmArgs w2 = gemm_args(GEMM_WGRAD, c, offsets, uniform_rows, c->d, f, dyp, h, dW2,
                                 nullptr, nullptr, err);
  w2.wg_M = c->d;
  w2.wg_N = f;
  w2.seg_maps = seg_maps;
  MOE_TRY(launch_grouped_gemm(w2, st));
  GroupedGemmArgs g1 = gemm_args(GEMM_DGRAD1, c, offsets, uniform_rows, c->d, f, dab, W1, dxp,
                                 nullptr, nullptr, err);
  MOE_TRY(launch_grouped_gemm(g1, st));
  GroupedGemmArgs w1 = gemm_args(GEMM_WGRAD, c, offsets, uniform_rows, c->d, f, dab, xp, dW1,
                                 nullptr, nullptr, err);
  w1.wg_M = 2 * f;
  w1.wg_N = c->d;
  w1.seg_maps = seg_maps;
  set_gather(w1, gx);
  MOE_TRY(launch_grouped_gemm(w1, st));
  return MOE_OK;
}

// A wait that nothing will complete: the bounded wait gives up, flags the timeout and the
// kernel returns (the path every pipeline wait of the grouped GEMM takes on a stall).
__global__ void selftest_wait_kernel(int* err, long long budget) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, err, budget);
}

}  // namespace

extern "C" {

int32_t moe_capacity_from_factor(int64_t T, int32_t k, int32_t E, double c) {
  if (T <= 0 || k <= 0 || E <= 0) return -1;
  if (!(c > 0.0)) return 0;
  const long double v = static_cast<long double>(c) * static_cast<long double>(T) *
                        static_cast<long double>(k) / static_cast<long double>(E);
  // absorb binary representation error of c (e.g. 1.25 is exact, 0.1 is not)
  const long double fl = std::floor(v + 1e-9L);
  if (fl > 2147483647.0L) return 2147483647;
  return static_cast<int32_t>(fl);
}

moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* ws_bytes, size_t* ctx_bytes) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (ws_bytes) *ws_bytes = ws_layout(cfg).total;
  if (ctx_bytes) *ctx_bytes = ctx_layout(cfg).total;
  return MOE_OK;
}

moe_status_t moe_ctx_offsets(const moe_config_t* cfg, size_t* offsets) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!offsets) return MOE_ERR_INVALID_ARG;
  CtxLayout L = ctx_layout(cfg);
  for (int i = 0; i < MOE_CTX_NFIELDS; ++i) offsets[i] = L.off[i];
  return MOE_OK;
}

moe_status_t moe_ws_init(void* ws, void* stream) {
  if (!ptrs_ok(ws)) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, WS_HEADER_BYTES, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_route(const moe_config_t* cfg, const float* logits, int32_t* topk_idx,
                       float* topk_w, int32_t* counts, int32_t* kept, int32_t* offsets,
                       int32_t* dest_row, int32_t* src_tok, int32_t* src_slot,
                       uint8_t* drop_mask, void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(logits, topk_idx, topk_w, counts, kept, offsets, dest_row, src_tok, src_slot,
               drop_mask, ws))
    return MOE_ERR_INVALID_ARG;
  WsLayout W = ws_layout(cfg);
  return cuda_status(launch_route(cfg, logits, topk_idx, topk_w, counts, kept, offsets,
                                  dest_row, src_tok, src_slot, drop_mask, at<uint8_t>(ws, W.route),
                                  static_cast<int*>(ws), static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_permute(const moe_config_t* cfg, const void* x, const int32_t* src_tok,
                         const int32_t* offsets, void* xp, void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(x, src_tok, offsets, xp, ws)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_permute(x, src_tok, offsets, cfg->E, cfg->T, cfg->T * cfg->k, cfg->d,
                                    xp, static_cast<int*>(ws),
                                    static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_grouped_ffn(const moe_config_t* cfg, const void* xp, const int32_t* offsets,
                             const void* W1, const void* W2, void* ab, void* h, void* yp,
                             void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(xp, offsets, W1, W2, ab, h, yp, ws)) return MOE_ERR_INVALID_ARG;
  return ffn_fwd(cfg, xp, offsets, 0, cfg->ffn, W1, W2, ab, h, yp, static_cast<int*>(ws),
                 static_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_ffn_gather(const moe_config_t* cfg, const void* x,
                                    const int32_t* src_tok, const int32_t* offsets,
                                    const void* W1, const void* W2, void* ab, void* h, void* yp,
                                    void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(x, src_tok, offsets, W1, W2, ab, h, yp, ws)) return MOE_ERR_INVALID_ARG;
  Gather gx;
  gx.idx = src_tok;
  gx.src = x;
  gx.rows = cfg->T;
  return ffn_fwd(cfg, nullptr, offsets, 0, cfg->ffn, W1, W2, ab, h, yp, static_cast<int*>(ws),
                 static_cast<cudaStream_t>(stream), gx);
}

moe_status_t moe_combine(const moe_config_t* cfg, const void* yp, const int32_t* dest_row,
                         const float* topk_w, const void* ys_or_null, void* y, void* ws,
                         void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(yp, dest_row, topk_w, y, ws)) return MOE_ERR_INVALID_ARG;
  if (ys_or_null && !aligned16(ys_or_null)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(yp, dest_row, topk_w, ys_or_null, cfg->T, cfg->k, cfg->d,
                                    cfg->T * cfg->k, y, static_cast<int*>(ws),
                                    static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_combine_bwd(const moe_config_t* cfg, const void* dy, const void* yp,
                             const float* logits, const int32_t* topk_idx, const float* topk_w,
                             const int32_t* dest_row, void* dyp, float* dlogits, void* ws,
                             void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(dy, yp, logits, topk_idx, topk_w, dest_row, dyp, dlogits, ws))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine_bwd(dy, yp, logits, topk_idx, topk_w, dest_row, cfg->T,
                                        cfg->E, cfg->k, cfg->d, cfg->gate, cfg->route_scale,
                                        cfg->T * cfg->k, dyp, dlogits, static_cast<int*>(ws),
                                        static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_grouped_ffn_bwd(const moe_config_t* cfg, const void* dyp, const void* xp,
                                 const int32_t* offsets, const void* W1, const void* W2,
                                 const void* ab, const void* h, void* dab, void* dxp, void* dW1,
                                 void* dW2, void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(dyp, xp, offsets, W1, W2, ab, h, dab, dxp, dW1, dW2, ws))
    return MOE_ERR_INVALID_ARG;
  return ffn_bwd(cfg, dyp, xp, offsets, 0, cfg->ffn, W1, W2, ab, h, dab, dxp, dW1, dW2,
                 at<uint8_t>(ws, ws_layout(cfg).maps), static_cast<int*>(ws),
                 static_cast<cudaStream_t>(stream));
}

moe_status_t moe_grouped_ffn_bwd_gather(const moe_config_t* cfg, const void* dyp, const void* x,
                                        const int32_t* src_tok, const int32_t* offsets,
                                        const void* W1, const void* W2, const void* ab,
                                        const void* h, void* dab, void* dxp, void* dW1,
                                        void* dW2, void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(dyp, x, src_tok, offsets, W1, W2, ab, h, dab, dxp, dW1, dW2, ws))
    return MOE_ERR_INVALID_ARG;
  Gather gx;
  gx.idx = src_tok;
  gx.src = x;
  gx.rows = cfg->T;
  return ffn_bwd(cfg, dyp, nullptr, offsets, 0, cfg->ffn, W1, W2, ab, h, dab, dxp, dW1, dW2,
                 at<uint8_t>(ws, ws_layout(cfg).maps), static_cast<int*>(ws),
                 static_cast<cudaStream_t>(stream), gx);
}

moe_status_t moe_grouped_ffn_bwd_dispatch(const moe_config_t* cfg, const void* dy,
                                          const float* topk_w, const int32_t* src_tok,
                                          const int32_t* src_slot, const void* dyp,
                                          const void* xp, const int32_t* offsets,
                                          const void* W1, const void* W2, const void* ab,
                                          const void* h, void* dab, void* dxp, void* dW1,
                                          void* dW2, void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(dy, topk_w, src_tok, src_slot, dyp, xp, offsets, W1, W2, ab, h, dab, dxp, dW1,
               dW2, ws))
    return MOE_ERR_INVALID_ARG;
  DyDispatch gd;
  gd.rows.idx = src_tok;
  gd.rows.src = dy;
  gd.rows.rows = cfg->T;
  gd.topk_w = topk_w;
  gd.src_slot = src_slot;
  gd.n_slots = cfg->T * cfg->k;
  return ffn_bwd(cfg, dyp, xp, offsets, 0, cfg->ffn, W1, W2, ab, h, dab, dxp, dW1, dW2,
                 at<uint8_t>(ws, ws_layout(cfg).maps), static_cast<int*>(ws),
                 static_cast<cudaStream_t>(stream), Gather{}, gd);
}

moe_status_t moe_unpermute_reduce(const moe_config_t* cfg, const void* dxp,
                                  const int32_t* dest_row, const void* dxs_or_null, void* dx,
                                  void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(dxp, dest_row, dx, ws)) return MOE_ERR_INVALID_ARG;
  if (dxs_or_null && !aligned16(dxs_or_null)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(dxp, dest_row, nullptr, dxs_or_null, cfg->T, cfg->k, cfg->d,
                                    cfg->T * cfg->k, dx, static_cast<int*>(ws),
                                    static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_fwd(const moe_config_t* cfg, const float* logits, const void* x,
                           const void* W1, const void* W2, const void* W1s, const void* W2s,
                           void* y, void* ctx, void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(logits, x, W1, W2, y, ctx, ws)) return MOE_ERR_INVALID_ARG;
  if (cfg->ffn_shared && !ptrs_ok(W1s, W2s)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(ws);
  CtxLayout C = ctx_layout(cfg);
  WsLayout W = ws_layout(cfg);
  int32_t* offsets = at<int32_t>(ctx, C.off[MOE_CTX_OFFSETS]);
  MOE_TRY(launch_route(cfg, logits, at<int32_t>(ctx, C.off[MOE_CTX_TOPK_IDX]),
                       at<float>(ctx, C.off[MOE_CTX_TOPK_W]),
                       at<int32_t>(ctx, C.off[MOE_CTX_COUNTS]),
                       at<int32_t>(ctx, C.off[MOE_CTX_KEPT]), offsets,
                       at<int32_t>(ctx, C.off[MOE_CTX_DEST_ROW]),
                       at<int32_t>(ctx, C.off[MOE_CTX_SRC_TOK]),
                       at<int32_t>(ctx, C.off[MOE_CTX_SRC_SLOT]),
                       at<uint8_t>(ctx, C.off[MOE_CTX_DROP_MASK]), at<uint8_t>(ws, W.route), err,
                       st));
  void* xp = at<uint8_t>(ctx, C.off[MOE_CTX_XP]);
  MOE_TRY(launch_permute(x, at<int32_t>(ctx, C.off[MOE_CTX_SRC_TOK]), offsets, cfg->E, cfg->T,
                         cfg->T * cfg->k, cfg->d, xp, err, st));
  void* yp = at<uint8_t>(ctx, C.off[MOE_CTX_YP]);
  const bool rc = cfg->recompute != 0;
  void* ab = rc ? at<uint8_t>(ws, W.ab) : at<uint8_t>(ctx, C.off[MOE_CTX_AB]);
  void* h = rc ? at<uint8_t>(ws, W.h) : at<uint8_t>(ctx, C.off[MOE_CTX_H]);
  s = ffn_fwd(cfg, xp, offsets, 0, cfg->ffn, W1, W2, ab, h, yp, err, st);
  if (s != MOE_OK) return s;
  const void* ys = nullptr;
  if (cfg->ffn_shared) {
    void* ysw = at<uint8_t>(ctx, C.off[MOE_CTX_YS]);
    void* ab_s = rc ? at<uint8_t>(ws, W.ab_s) : at<uint8_t>(ctx, C.off[MOE_CTX_AB_S]);
    void* h_s = rc ? at<uint8_t>(ws, W.h_s) : at<uint8_t>(ctx, C.off[MOE_CTX_H_S]);
    s = ffn_fwd(cfg, x, nullptr, cfg->T, cfg->ffn_shared, W1s, W2s, ab_s, h_s, ysw, err, st);
    if (s != MOE_OK) return s;
    ys = ysw;
  }
  MOE_TRY(launch_combine(yp, at<int32_t>(ctx, C.off[MOE_CTX_DEST_ROW]),
                         at<float>(ctx, C.off[MOE_CTX_TOPK_W]), ys, cfg->T, cfg->k, cfg->d,
                         cfg->T * cfg->k, y, err, st));
  return MOE_OK;
}

moe_status_t moe_mx_weights_size(const moe_config_t* cfg, size_t* bytes, size_t* offsets) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (cfg->d % 128 || cfg->ffn % 128) return MOE_ERR_UNSUPPORTED;
  const MxWeightLayout L = mx_weight_layout(cfg->E, cfg->d, cfg->ffn);
  if (bytes) *bytes = L.total;
  if (offsets) {
    offsets[0] = L.w1q;
    offsets[1] = L.w1sf;
    offsets[2] = L.w2q;
    offsets[3] = L.w2sf;
    offsets[4] = L.w2tq;
    offsets[5] = L.w2tsf;
    offsets[6] = L.w1tq;
    offsets[7] = L.w1tsf;
  }
  return MOE_OK;
}

moe_status_t moe_mx_act_scales_size(const moe_config_t* cfg, int32_t K, size_t* bytes) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (K <= 0 || K % 128 || !bytes) return MOE_ERR_INVALID_ARG;
  *bytes = mx_act_scale_bytes(cfg->T * cfg->k, cfg->E, K);
  return MOE_OK;
}

moe_status_t moe_mx_quantize_weights(const moe_config_t* cfg, const void* W1, const void* W2,
                                     void* wq, void* stream) {
  size_t bytes = 0;
  moe_status_t s = moe_mx_weights_size(cfg, &bytes, nullptr);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(W1, W2, wq) || (reinterpret_cast<uintptr_t>(wq) & 255u)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_mx_quant_weights(W1, W2, cfg->E, cfg->d, cfg->ffn, wq,
                                             static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_mx_permute_quant(const moe_config_t* cfg, const void* x, const int32_t* src_tok,
                                  const int32_t* offsets, void* xp_or_null, void* xq,
                                  uint8_t* x_sf, void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (cfg->d % 128) return MOE_ERR_UNSUPPORTED;
  if (!ptrs_ok(x, src_tok, offsets, xq, x_sf, ws)) return MOE_ERR_INVALID_ARG;
  if (xp_or_null && !aligned16(xp_or_null)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_mx_permute_quant(x, src_tok, offsets, cfg->E, cfg->T,
                                             cfg->T * cfg->k, cfg->d, xp_or_null, xq, x_sf,
                                             static_cast<int*>(ws),
                                             static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_grouped_ffn_mx(const moe_config_t* cfg, const void* xq, const uint8_t* x_sf,
                                const int32_t* offsets, const void* wq, void* ab, void* h,
                                uint8_t* hq, uint8_t* h_sf, void* yp, void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (cfg->d % 128 || cfg->ffn % 128) return MOE_ERR_UNSUPPORTED;
  if (!ptrs_ok(xq, x_sf, offsets, wq, ab, h, hq, h_sf, yp, ws)) return MOE_ERR_INVALID_ARG;
  MxFfnArgs a{};
  a.E = cfg->E;
  a.d = cfg->d;
  a.f = cfg->ffn;
  a.rows_cap = cfg->T * cfg->k;
  a.offsets = offsets;
  a.xq = xq;
  a.x_sf = x_sf;
  a.wq = wq;
  a.ab = ab;
  a.h = h;
  a.hq = hq;
  a.h_sf = h_sf;
  a.yp = yp;
  a.err = static_cast<int*>(ws);
  return cuda_status(launch_mx_ffn(a, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_fwd_mx(const moe_config_t* cfg, const float* logits, const void* x,
                              const void* wq, const void* W1s, const void* W2s, void* y,
                              void* ctx, void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!cfg->mxfp8) return MOE_ERR_INVALID_ARG;
  if (!ptrs_ok(logits, x, wq, y, ctx, ws)) return MOE_ERR_INVALID_ARG;
  if (cfg->ffn_shared && !ptrs_ok(W1s, W2s)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(ws);
  CtxLayout C = ctx_layout(cfg);
  WsLayout W = ws_layout(cfg);
  int32_t* offsets = at<int32_t>(ctx, C.off[MOE_CTX_OFFSETS]);
  const int32_t* src_tok = at<int32_t>(ctx, C.off[MOE_CTX_SRC_TOK]);
  MOE_TRY(launch_route(cfg, logits, at<int32_t>(ctx, C.off[MOE_CTX_TOPK_IDX]),
                       at<float>(ctx, C.off[MOE_CTX_TOPK_W]),
                       at<int32_t>(ctx, C.off[MOE_CTX_COUNTS]),
                       at<int32_t>(ctx, C.off[MOE_CTX_KEPT]), offsets,
                       at<int32_t>(ctx, C.off[MOE_CTX_DEST_ROW]),
                       at<int32_t>(ctx, C.off[MOE_CTX_SRC_TOK]),
                       at<int32_t>(ctx, C.off[MOE_CTX_SRC_SLOT]),
                       at<uint8_t>(ctx, C.off[MOE_CTX_DROP_MASK]), at<uint8_t>(ws, W.route), err,
                       st));
  void* xp = at<uint8_t>(ctx, C.off[MOE_CTX_XP]);
  MOE_TRY(launch_mx_permute_quant(x, src_tok, offsets, cfg->E, cfg->T, cfg->T * cfg->k, cfg->d,
                                  xp, at<uint8_t>(ws, W.xq), at<uint8_t>(ws, W.x_sf), err, st));
  MxFfnArgs a{};
  a.E = cfg->E;
  a.d = cfg->d;
  a.f = cfg->ffn;
  a.rows_cap = cfg->T * cfg->k;
  a.offsets = offsets;
  a.xq = at<uint8_t>(ws, W.xq);
  a.x_sf = at<uint8_t>(ws, W.x_sf);
  a.wq = wq;
  a.ab = at<uint8_t>(ctx, C.off[MOE_CTX_AB]);
  a.h = at<uint8_t>(ctx, C.off[MOE_CTX_H]);
  a.hq = at<uint8_t>(ws, W.hq);
  a.h_sf = at<uint8_t>(ws, W.h_sf);
  void* yp = at<uint8_t>(ctx, C.off[MOE_CTX_YP]);
  a.yp = yp;
  a.err = err;
  MOE_TRY(launch_mx_ffn(a, st));
  const void* ys = nullptr;
  if (cfg->ffn_shared) {   // the shared expert stays bf16
    void* ysw = at<uint8_t>(ctx, C.off[MOE_CTX_YS]);
    s = ffn_fwd(cfg, x, nullptr, cfg->T, cfg->ffn_shared, W1s, W2s,
                at<uint8_t>(ctx, C.off[MOE_CTX_AB_S]), at<uint8_t>(ctx, C.off[MOE_CTX_H_S]), ysw,
                err, st);
    if (s != MOE_OK) return s;
    ys = ysw;
  }
  MOE_TRY(launch_combine(yp, at<int32_t>(ctx, C.off[MOE_CTX_DEST_ROW]),
                         at<float>(ctx, C.off[MOE_CTX_TOPK_W]), ys, cfg->T, cfg->k, cfg->d,
                         cfg->T * cfg->k, y, err, st));
  return MOE_OK;
}

namespace {
// The MXFP8 backward of the routed experts' FFN: quantise dyp, DGRAD2 and DGRAD1 on MXFP8
// operands, then the two weight gradients: bf16 (mxfp8 = 1), or (mxfp8 = 2) on operands
// quantised along each segment's tokens.
moe_status_t ffn_bwd_mx(const moe_config_t* c, const void* dyp, const void* xp,
                        const int32_t* offsets, const void* wq, const void* ab, const void* h,
                        void* dab, void* dxp, void* dW1, void* dW2, void* ws, cudaStream_t st) {
  const WsLayout W = ws_layout(c);
  int* err = static_cast<int*>(ws);
  const int64_t R = c->T * c->k;
  MOE_TRY(launch_mx_permute_quant(dyp, nullptr, offsets, c->E, R, R, c->d, nullptr,
                                  at<uint8_t>(ws, W.dyq), at<uint8_t>(ws, W.dy_sf), err, st));
  MxDgradArgs a{};
  a.E = c->E;
  a.d = c->d;
  a.f = c->ffn;
  a.rows_cap = R;
  a.offsets = offsets;
  a.dyq = at<uint8_t>(ws, W.dyq);
  a.dy_sf = at<uint8_t>(ws, W.dy_sf);
  a.wq = wq;
  a.ab = ab;
  a.dab = dab;
  a.dabq = at<uint8_t>(ws, W.dabq);
  a.dab_sf = at<uint8_t>(ws, W.dab_sf);
  a.dxp = dxp;
  a.err = err;
  MOE_TRY(launch_mx_ffn_dgrad(a, st));
  if (c->mxfp8 == 2) {
    auto quant = [&](const void* X, int C, bool role_n, size_t q, size_t sf) {
      return launch_mx_quant_tok(X, offsets, c->E, R, C, role_n, at<uint8_t>(ws, q),
                                 at<uint8_t>(ws, sf), err, st);
    };
    MxWgradArgs g{};
    g.E = c->E;
    g.rows_cap = R;
    g.offsets = offsets;
    g.err = err;
    // dW2 [E][d][f] = dyp^T h
    MOE_TRY(quant(dyp, c->d, false, W.dyT, W.dyT_sf));
    MOE_TRY(quant(h, c->ffn, true, W.hT, W.hT_sf));
    g.M = c->d;
    g.N = c->ffn;
    g.aq = at<uint8_t>(ws, W.dyT);
    g.a_sf = at<uint8_t>(ws, W.dyT_sf);
    g.bq = at<uint8_t>(ws, W.hT);
    g.b_sf = at<uint8_t>(ws, W.hT_sf);
    g.dW = dW2;
    MOE_TRY(launch_mx_wgrad(g, st));
    // dW1 [E][2f][d] = dab^T xp
    MOE_TRY(quant(dab, 2 * c->ffn, false, W.dabT, W.dabT_sf));
    MOE_TRY(quant(xp, c->d, true, W.xpT, W.xpT_sf));
    g.M = 2 * c->ffn;
    g.N = c->d;
    g.aq = at<uint8_t>(ws, W.dabT);
    g.a_sf = at<uint8_t>(ws, W.dabT_sf);
    g.bq = at<uint8_t>(ws, W.xpT);
    g.b_sf = at<uint8_t>(ws, W.xpT_sf);
    g.dW = dW1;
    MOE_TRY(launch_mx_wgrad(g, st));
    return MOE_OK;
  }
  void* maps = at<uint8_t>(ws, W.maps);
  GroupedGemmArgs w2 = gemm_args(GEMM_WGRAD, c, offsets, 0, c->d, c->ffn, dyp, h, dW2, nullptr,
                                 nullptr, err);
  w2.wg_M = c->d;
  w2.wg_N = c->ffn;
  w2.seg_maps = maps;
  MOE_TRY(launch_grouped_gemm(w2, st));
  GroupedGemmArgs w1 = gemm_args(GEMM_WGRAD, c, offsets, 0, c->d, c->ffn, dab, xp, dW1, nullptr,
                                 nullptr, err);
  w1.wg_M = 2 * c->ffn;
  w1.wg_N = c->d;
  w1.seg_maps = maps;
  MOE_TRY(launch_grouped_gemm(w1, st));
  return MOE_OK;
}
}  // namespace

moe_status_t moe_grouped_ffn_bwd_mx(const moe_config_t* cfg, const void* dyp, const void* xp,
                                    const int32_t* offsets, const void* wq, const void* ab,
                                    const void* h, void* dab, void* dxp, void* dW1, void* dW2,
                                    void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!cfg->mxfp8) return MOE_ERR_INVALID_ARG;
  if (!ptrs_ok(dyp, xp, offsets, wq, ab, h, dab, dxp, dW1, dW2, ws)) return MOE_ERR_INVALID_ARG;
  return ffn_bwd_mx(cfg, dyp, xp, offsets, wq, ab, h, dab, dxp, dW1, dW2, ws,
                    static_cast<cudaStream_t>(stream));
}

namespace {
// The whole backward; wq != null runs the routed experts' data gradients on MXFP8 operands.
moe_status_t layer_bwd(const moe_config_t* cfg, const void* ctx, const float* logits,
                       const void* x, const void* dy, const void* W1, const void* W2,
                       const void* wq, const void* W1s, const void* W2s, void* dx, void* dW1,
                       void* dW2, void* dW1s, void* dW2s, float* dlogits, void* ws,
                       void* stream) {
  moe_status_t s = MOE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(ws);
  CtxLayout C = ctx_layout(cfg);
  WsLayout W = ws_layout(cfg);
  const int32_t* offsets = at<int32_t>(ctx, C.off[MOE_CTX_OFFSETS]);
  const int32_t* dest_row = at<int32_t>(ctx, C.off[MOE_CTX_DEST_ROW]);
  void* dyp = at<uint8_t>(ws, W.dyp);
  void* dab = at<uint8_t>(ws, W.dab);
  void* dxp = at<uint8_t>(ws, W.dxp);
  const bool rc = cfg->recompute != 0;
  const void* xp_saved = at<uint8_t>(ctx, C.off[MOE_CTX_XP]);
  const void* ab = at<uint8_t>(ctx, C.off[MOE_CTX_AB]);
  const void* h = at<uint8_t>(ctx, C.off[MOE_CTX_H]);
  const void* ab_s = at<uint8_t>(ctx, C.off[MOE_CTX_AB_S]);
  const void* h_s = at<uint8_t>(ctx, C.off[MOE_CTX_H_S]);
  if (rc) {
    // selective rematerialisation: rerun FC1 (+ SwiGLU) from the saved permuted tokens;
    // the grouped GEMM is deterministic, so ab and h equal the forward's bit for bit
    GroupedGemmArgs a1 = gemm_args(GEMM_FC1_SWIGLU, cfg, offsets, 0, cfg->d, cfg->ffn, xp_saved,
                                   W1, at<uint8_t>(ws, W.ab), at<uint8_t>(ws, W.h), nullptr, err);
    MOE_TRY(launch_grouped_gemm(a1, st));
    ab = at<uint8_t>(ws, W.ab);
    h = at<uint8_t>(ws, W.h);
    if (cfg->ffn_shared) {
      GroupedGemmArgs a2 = gemm_args(GEMM_FC1_SWIGLU, cfg, nullptr, cfg->T, cfg->d,
                                     cfg->ffn_shared, x, W1s, at<uint8_t>(ws, W.ab_s),
                                     at<uint8_t>(ws, W.h_s), nullptr, err);
      MOE_TRY(launch_grouped_gemm(a2, st));
      ab_s = at<uint8_t>(ws, W.ab_s);
      h_s = at<uint8_t>(ws, W.h_s);
    }
  }
  MOE_TRY(launch_combine_bwd(dy, at<uint8_t>(ctx, C.off[MOE_CTX_YP]), logits,
                             at<int32_t>(ctx, C.off[MOE_CTX_TOPK_IDX]),
                             at<float>(ctx, C.off[MOE_CTX_TOPK_W]), dest_row, cfg->T, cfg->E,
                             cfg->k, cfg->d, cfg->gate, cfg->route_scale, cfg->T * cfg->k, dyp,
                             dlogits, err, st));
  if (wq)
    s = ffn_bwd_mx(cfg, dyp, xp_saved, offsets, wq, ab, h, dab, dxp, dW1, dW2, ws, st);
  else
    s = ffn_bwd(cfg, dyp, xp_saved, offsets, 0, cfg->ffn, W1, W2, ab, h, dab, dxp, dW1, dW2,
                at<uint8_t>(ws, W.maps), err, st);
  if (s != MOE_OK) return s;
  const void* dxs = nullptr;
  if (cfg->ffn_shared) {
    void* dxsw = at<uint8_t>(ws, W.dx_s);
    s = ffn_bwd(cfg, dy, x, nullptr, cfg->T, cfg->ffn_shared, W1s, W2s, ab_s, h_s,
                at<uint8_t>(ws, W.dab_s), dxsw, dW1s, dW2s, nullptr, err, st);
    if (s != MOE_OK) return s;
    dxs = dxsw;
  }
  MOE_TRY(launch_combine(dxp, dest_row, nullptr, dxs, cfg->T, cfg->k, cfg->d, cfg->T * cfg->k,
                         dx, err, st));
  return MOE_OK;
}
}  // namespace

moe_status_t moe_layer_bwd(const moe_config_t* cfg, const void* ctx, const float* logits,
                           const void* x, const void* dy, const void* W1, const void* W2,
                           const void* W1s, const void* W2s, void* dx, void* dW1, void* dW2,
                           void* dW1s, void* dW2s, float* dlogits, void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!ptrs_ok(ctx, logits, x, dy, W1, W2, dx, dW1, dW2, dlogits, ws)) return MOE_ERR_INVALID_ARG;
  if (cfg->ffn_shared && !ptrs_ok(W1s, W2s, dW1s, dW2s)) return MOE_ERR_INVALID_ARG;
  return layer_bwd(cfg, ctx, logits, x, dy, W1, W2, nullptr, W1s, W2s, dx, dW1, dW2, dW1s, dW2s,
                   dlogits, ws, stream);
}

moe_status_t moe_layer_bwd_mx(const moe_config_t* cfg, const void* ctx, const float* logits,
                              const void* x, const void* dy, const void* wq, const void* W1s,
                              const void* W2s, void* dx, void* dW1, void* dW2, void* dW1s,
                              void* dW2s, float* dlogits, void* ws, void* stream) {
  moe_status_t s = validate(cfg);
  if (s != MOE_OK) return s;
  if (!cfg->mxfp8) return MOE_ERR_INVALID_ARG;
  if (!ptrs_ok(ctx, logits, x, dy, wq, dx, dW1, dW2, dlogits, ws)) return MOE_ERR_INVALID_ARG;
  if (cfg->ffn_shared && !ptrs_ok(W1s, W2s, dW1s, dW2s)) return MOE_ERR_INVALID_ARG;
  return layer_bwd(cfg, ctx, logits, x, dy, nullptr, nullptr, wq, W1s, W2s, dx, dW1, dW2, dW1s,
                   dW2s, dlogits, ws, stream);
}

moe_status_t moe_selftest_wait_timeout(void* ws, int64_t budget_cycles, void* stream) {
  if (!ptrs_ok(ws) || budget_cycles <= 0) return MOE_ERR_INVALID_ARG;
  const long long budget = budget_cycles > 2000000000LL ? 2000000000LL : budget_cycles;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<int*>(ws),
                                                                        budget);
  return cuda_status(cudaGetLastError());
}

moe_status_t moe_gemm_clock_trace(int enable) {
  if (moe::gemm_clock_trace_set(enable != 0) != cudaSuccess ||
      moe::mx_clock_trace_set(enable != 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_gemm_clock_read(uint64_t* cycles, uint64_t* ns, uint64_t* loops) {
  if (!cycles || !ns || !loops) return MOE_ERR_INVALID_ARG;
  unsigned long long sum[3] = {0, 0, 0};
  if (moe::gemm_clock_trace_add(sum) != cudaSuccess ||
      moe::mx_clock_trace_add(sum) != cudaSuccess)
    return MOE_ERR_CUDA;
  *cycles = sum[0];
  *ns = sum[1];
  *loops = sum[2];
  return MOE_OK;
}

moe_status_t moe_status(void* ws, void* stream, int32_t* flags) {
  if (!ptrs_ok(ws)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  if (h) {
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (flags) *flags = h;
  if (h & MOE_DEVERR_TIMEOUT) return MOE_ERR_TIMEOUT;
  return h ? MOE_ERR_DEVICE_FLAG : MOE_OK;
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_FLAG: return "MOE_ERR_DEVICE_FLAG";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
  }
  return "MOE_ERR_UNKNOWN";
}

}  // extern "C"
