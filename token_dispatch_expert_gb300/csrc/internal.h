// internal.h -- launchers shared between the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Number of 32-token chunks the routing histogram is built from.
inline int64_t route_chunks(int64_t T) { return (T + 31) / 32; }

// Scratch the routing step needs inside ws (after the 256-byte header): the per-chunk,
// per-expert counts; with drop-by-score also each expert's base among all eligible
// assignments (E+1 ints) and one 32-bit word per assignment (score key, then final rank).
struct RouteScratch {
  size_t chunk, cnt_base, list, total;
};
inline RouteScratch route_scratch_layout(int64_t T, int E, int k, bool by_score) {
  auto up = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
  RouteScratch r;
  r.chunk = 0;
  size_t o = up(static_cast<size_t>(route_chunks(T)) * static_cast<size_t>(E) * 4);
  r.cnt_base = o;
  if (by_score) o += up(static_cast<size_t>(E + 1) * 4);
  r.list = o;
  if (by_score) o += up(static_cast<size_t>(T) * static_cast<size_t>(k) * 4);
  r.total = o;
  return r;
}
inline bool route_by_score(const moe_config_t* c) {
  return c->drop_by_score != 0 && c->capacity > 0;
}
inline size_t route_scratch_bytes(const moe_config_t* c) {
  return route_scratch_layout(c->T, c->E, c->k, route_by_score(c)).total;
}

constexpr size_t WS_HEADER_BYTES = 256;

// F1 + F2 for config `c` (its routing variants included); scratch: route_scratch_bytes(c)
// bytes, 256-byte aligned.
cudaError_t launch_route(const moe_config_t* c, const float* logits, int32_t* topk_idx,
                         float* topk_w, int32_t* counts, int32_t* kept, int32_t* offsets,
                         int32_t* dest_row, int32_t* src_tok, int32_t* src_slot,
                         uint8_t* drop_mask, void* scratch, int* err, cudaStream_t st);

cudaError_t launch_permute(const void* x, const int32_t* src_tok, const int32_t* offsets,
                           int E, int64_t T, int64_t rows_cap, int d, void* xp, int* err,
                           cudaStream_t st);

// y[t] = sum_j w[t,j] * rows[dest_row[t,j]] (+ add[t]); w == nullptr means weight 1.
cudaError_t launch_combine(const void* rows, const int32_t* dest_row, const float* w,
                           const void* add, int64_t T, int k, int d, int64_t rows_cap, void* y,
                           int* err, cudaStream_t st);

cudaError_t launch_combine_bwd(const void* dy, const void* yp, const float* logits,
                               const int32_t* topk_idx, const float* topk_w,
                               const int32_t* dest_row, int64_t T, int E, int k, int d,
                               int gate, float scale, int64_t rows_cap, void* dyp,
                               float* dlogits, int* err, cudaStream_t st);

// ----------------------------------------------------------------- grouped GEMM
enum GemmMode : int {
  GEMM_FC1_SWIGLU = 0,  // [a|b] = A W1^T, h = silu(a) b          A K-major, B K-major
  GEMM_FC2 = 1,         // out = A W2^T                           A K-major, B K-major
  GEMM_DGRAD2_SWIGLU = 2,  // dh = A W2; da, db from ab           A K-major, B MN-major
  GEMM_DGRAD1 = 3,      // out = A W1                             A K-major, B MN-major
  GEMM_WGRAD = 4,       // dW[g] = A_g^T B_g (K = rows of g)      A MN-major, B MN-major
};

struct GroupedGemmArgs {
  int mode;
  // groups: offsets[G+1] on the device, or a single group of `uniform_rows` rows
  const int32_t* offsets;
  int G;
  int64_t uniform_rows;  // > 0: one group of this many rows, offsets ignored
  int64_t rows_cap;      // capacity (rows) of the row-indexed buffers
  int d;                 // model width of this expert set
  int f;                 // SwiGLU width of this expert set
  // operands (bf16)
  const void* A;   // FC1: xp [rows,d]  FC2: h [rows,f]  DGRAD2: dyp [rows,d]
                   // DGRAD1: dab [rows,2f]   WGRAD: [rows, M]
  const void* B;   // FC1: W1 [G,2f,d]  FC2: W2 [G,d,f]  DGRAD2: W2  DGRAD1: W1
                   // WGRAD: [rows, N]
  int wg_M;        // WGRAD: M (= d for dW2, 2f for dW1)
  int wg_N;        // WGRAD: N (= f for dW2, d for dW1)
  // outputs
  void* out0;      // FC1: ab  FC2: yp  DGRAD2: dab  DGRAD1: dxp  WGRAD: dW [G, M, N]
  void* out1;      // FC1: h
  const void* aux; // DGRAD2: ab (saved FC1 output)
  int* err;
  // WGRAD over segments: device scratch for 2 * G tensor maps (128-byte aligned) whose row
  // extent ends at each segment's end, so rows past it load as zeros
  void* seg_maps;
  // Gathered operand (FC1's A, DGRAD2's A, or the WGRAD's B): when gather_idx is set, row p
  // of that operand is row gather_idx[p] of gather_src [gather_rows, cols] instead of row p
  // of the row buffer -- a dispatch fused into the GEMM's loads (TMA gather4).
  const int32_t* gather_idx;
  const void* gather_src;
  int64_t gather_rows;
  // DGRAD2 with gathered rows (the rows of dy): dh of row p is scaled by
  // gate_w[gate_slot[p]], gate_slot entries in [0, n_slots)
  const float* gate_w;
  const int32_t* gate_slot;
  int64_t n_slots;
};

constexpr size_t SEG_MAP_BYTES = 128;   // one CUtensorMap

cudaError_t launch_grouped_gemm(const GroupedGemmArgs& a, cudaStream_t st);

// ----------------------------------------------------------------- MXFP8 forward
// Byte offsets inside the quantised-weight blob: E4M3 codes of W1 [E][2f][d] and W2
// [E][d][f], and their E8M0 scales in 512-byte atoms ([E][f/128][d/128][2][512] and
// [E][ceil(d/256)][f/128][2][512]); every part 256-byte aligned.
// The backward's parts: W2^T [E][f][d] quantised along d with atoms
// [E][ceil(f/256)][d/128][2][512], and W1^T [E][d][2f] quantised along 2f with atoms
// [E][ceil(d/256)][2f/128][2][512].
struct MxWeightLayout {
  size_t w1q, w1sf, w2q, w2sf, w2tq, w2tsf, w1tq, w1tsf, total;
};
MxWeightLayout mx_weight_layout(int E, int d, int f);

// Bytes of an activation scale array (atoms tiled by 128 rows inside each expert
// segment: block (offsets[e] >> 7) + e + l/128 for local row l, K/128 atoms per block).
inline size_t mx_act_scale_bytes(int64_t rows_cap, int E, int K) {
  return static_cast<size_t>((rows_cap >> 7) + E + 1) * static_cast<size_t>(K / 128) * 512;
}

cudaError_t launch_mx_quant_weights(const void* W1, const void* W2, int E, int d, int f,
                                    void* blob, cudaStream_t st);

cudaError_t launch_mx_permute_quant(const void* x, const int32_t* src_tok,
                                    const int32_t* offsets, int E, int64_t T, int64_t rows_cap,
                                    int d, void* xp_or_null, void* xq, uint8_t* x_sf, int* err,
                                    cudaStream_t st);

struct MxFfnArgs {
  int E, d, f;
  int64_t rows_cap;
  const int32_t* offsets;
  const void* xq;        // [rows_cap][d] E4M3
  const uint8_t* x_sf;   // activation scale atoms (mx_act_scale_bytes(rows_cap, E, d))
  const void* wq;        // quantised-weight blob
  void* ab;              // [rows_cap][2f] bf16
  void* h;               // [rows_cap][f] bf16
  uint8_t* hq;           // [rows_cap][f] E4M3
  uint8_t* h_sf;         // activation scale atoms (mx_act_scale_bytes(rows_cap, E, f))
  void* yp;              // [rows_cap][d] bf16
  int* err;
};
cudaError_t launch_mx_ffn(const MxFfnArgs& a, cudaStream_t st);

// The backward's data gradients on MXFP8 operands: DGRAD2 (dh from dyq and the W2^T codes,
// the SwiGLU backward from ab -> dab bf16 and its MXFP8 form), then DGRAD1 (dxp from the
// dab codes and the W1^T codes).
struct MxDgradArgs {
  int E, d, f;
  int64_t rows_cap;
  const int32_t* offsets;
  const void* dyq;       // [rows_cap][d] E4M3
  const uint8_t* dy_sf;  // activation scale atoms (K = d)
  const void* wq;        // quantised-weight blob
  const void* ab;        // [rows_cap][2f] bf16 (saved)
  void* dab;             // [rows_cap][2f] bf16 out
  uint8_t* dabq;         // [rows_cap][2f] E4M3 out
  uint8_t* dab_sf;       // activation scale atoms (K = 2f) out
  void* dxp;             // [rows_cap][d] bf16 out
  int* err;
};
cudaError_t launch_mx_ffn_dgrad(const MxDgradArgs& a, cudaStream_t st);

// MXFP8 weight gradients.  Their contraction runs over an expert segment's rows, so each
// operand is quantised along the rows: the segment is cut into K blocks of 128 rows (the
// last zero-padded) and expert e's blocks follow e-1's (block kb0_e + i, kb0_e the sum of
// ceil(n_e' / 128) over e' < e).  Codes go transposed, [C][128 * kb_cap] (K-major along
// the rows); scales as atoms for the GEMM role: the M operand [C/128][kb_cap][512], the N
// operand [ceil(C/256)][kb_cap][2][512].  kb_cap = ceil(rows_cap / 128) + E.
inline int64_t mx_tok_kb_cap(int64_t rows_cap, int E) { return (rows_cap + 127) / 128 + E; }
inline size_t mx_tok_codes_bytes(int64_t rows_cap, int E, int C) {
  return static_cast<size_t>(C) * 128 * static_cast<size_t>(mx_tok_kb_cap(rows_cap, E));
}
inline size_t mx_tok_scale_bytes(int64_t rows_cap, int E, int C, bool role_n) {
  const size_t kb = static_cast<size_t>(mx_tok_kb_cap(rows_cap, E));
  return role_n ? static_cast<size_t>((C + 255) / 256) * kb * 1024
                : static_cast<size_t>(C / 128) * kb * 512;
}
cudaError_t launch_mx_quant_tok(const void* X, const int32_t* offsets, int E, int64_t rows_cap,
                                int C, bool role_n, uint8_t* codes, uint8_t* scales, int* err,
                                cudaStream_t st);
struct MxWgradArgs {
  int E;
  int64_t rows_cap;
  const int32_t* offsets;
  int M, N;              // dW [E][M][N] = A^T B over each segment's rows
  const uint8_t* aq;     // [M][128 kb_cap] codes, role M
  const uint8_t* a_sf;
  const uint8_t* bq;     // [N][128 kb_cap] codes, role N
  const uint8_t* b_sf;
  void* dW;              // [E][M][N] bf16 out
  int* err;
};
cudaError_t launch_mx_wgrad(const MxWgradArgs& a, cudaStream_t st);

// Clock tracing of the tensor-core mainloops (moe_gemm_clock_trace): the bf16 grouped GEMMs
// and the MXFP8 GEMMs each keep their own device-side sums.  *_set(true) zeroes the sums
// and turns tracing on, *_set(false) turns it off and keeps them; *_add adds the sums to
// out[0..2] (SM cycles, nanoseconds, loops).  Synchronous; call with the device idle.
cudaError_t gemm_clock_trace_set(bool on);
cudaError_t gemm_clock_trace_add(unsigned long long out[3]);
cudaError_t mx_clock_trace_set(bool on);
cudaError_t mx_clock_trace_add(unsigned long long out[3]);

}  // namespace moe
