// dispatch.cu -- the HBM-bound row movers of the layer: permute (F3), combine (F7),
// combine backward + gate backward (B1) and the un-permute reduce (B6).
//
// "MoE Training Optimization with Primus", Figure 7 dataflow: the permutation into
// expert order before FC1, and the last step that un-permutes the expert outputs, scales
// them by the gate weights and sums them per token; MegaMoE section: the backward mirrors them by
// dispatch/combine duality.  X-MoE verdict page, key machinery: the padding-free token
// buffer these kernels fill and drain.
//
// Permute runs one warp per destination row, combine, its backward and the reduce one
// warp per token; each walks its rows in batches of 16-byte vectors (8 bf16) whose loads
// are all issued before any is used, so each lane keeps 12-18 independent loads in
// flight whatever k is; the backward's dot products are warp reductions.  Combine accumulates in fp32 in slot order j = 0..k-1.  Every output
// element is written by exactly one thread: results are deterministic.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int THREADS = 256;

int sm_count() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

// persistent grid of warps (8 CTAs of 8 warps per SM at most)
int grid_warps(int64_t warps) {
  const int64_t need = (warps + THREADS / 32 - 1) / (THREADS / 32);
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  return static_cast<int>(need < 1 ? 1 : (need < cap ? need : cap));
}

// xp[p] = x[src_tok[p]] for p < offsets[E].  One warp per destination row; the row is
// copied in batches of 16 vectors per lane whose loads are all issued first.
__global__ void __launch_bounds__(THREADS)
permute_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ src_tok,
               const int32_t* __restrict__ offsets, int E, int64_t T, int64_t rows_cap, int nvec,
               uint4* __restrict__ xp, int* err) {
  griddep_wait();   // see common.cuh: dependent launches
  constexpr int B = 16;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * THREADS) >> 5;
  int64_t n_rows = offsets[E];
  if (n_rows < 0 || n_rows > rows_cap) {
    if (gw == 0 && lane == 0) flag_error(err, MOE_DEVERR_BAD_OFFSETS);
    n_rows = n_rows < 0 ? 0 : rows_cap;
  }
  // the next row's source index is loaded while the current row is copied, so a warp
  // with several rows does not wait for an index load before each row's copies
  int t_next = gw < n_rows ? __ldg(src_tok + gw) : 0;
  for (int64_t p = gw; p < n_rows; p += nw) {
    const int t = t_next;
    if (p + nw < n_rows) t_next = __ldg(src_tok + p + nw);
    if (t < 0 || t >= T) {
      if (lane == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
      continue;
    }
    const uint4* src = x + static_cast<int64_t>(t) * nvec;
    uint4* dst = xp + p * nvec;
    for (int c0 = lane; c0 < nvec; c0 += 32 * B) {
      uint4 v[B];
#pragma unroll
      for (int b = 0; b < B; ++b)
        if (c0 + 32 * b < nvec) v[b] = __ldg(src + c0 + 32 * b);
#pragma unroll
      for (int b = 0; b < B; ++b)
        if (c0 + 32 * b < nvec) dst[c0 + 32 * b] = v[b];
    }
  }
  griddep_launch();
}

// Slot indices and weights of token t, one lane per slot, broadcast to the warp.
template <int KMAX>
__device__ __forceinline__ void load_slots(const int32_t* __restrict__ dest_row,
                                           const float* __restrict__ w, int64_t t, int k,
                                           int64_t rows_cap, int* err, int64_t* p, float* wt) {
  const int lane = threadIdx.x & 31;
  int my_p = -1;
  float my_w = 1.0f;
  if (lane < k) {
    my_p = __ldg(dest_row + t * k + lane);
    if (w) my_w = __ldg(w + t * k + lane);
    if (my_p >= rows_cap || my_p < -1) {
      flag_error(err, MOE_DEVERR_BAD_INDEX);
      my_p = -1;
    }
  }
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    p[j] = __shfl_sync(FULL_MASK, my_p, j);
    wt[j] = __shfl_sync(FULL_MASK, my_w, j);
    if (j >= k) p[j] = -1;
  }
}

// y[t] = sum_j w[t,j] rows[dest_row[t,j]] (+ add[t]); w == nullptr -> weight 1.
// One warp per token; the row is walked in batches of B vectors per lane whose KMAX * B
// loads are all issued before any is used (about 16 independent 16-byte loads in flight
// per lane, whatever k is).
template <int KMAX>
__global__ void __launch_bounds__(THREADS)
combine_kernel(const uint4* __restrict__ rows, const int32_t* __restrict__ dest_row,
               const float* __restrict__ w, const uint4* __restrict__ add, int64_t T, int k,
               int nvec, int64_t rows_cap, uint4* __restrict__ y, int* err) {
  griddep_wait();   // see common.cuh: dependent launches
  constexpr int B = KMAX == 6 ? 3 : 16 / KMAX;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * THREADS) >> 5;
  for (int64_t t = gw; t < T; t += nw) {
    int64_t p[KMAX];
    float wt[KMAX];
    load_slots<KMAX>(dest_row, w, t, k, rows_cap, err, p, wt);
    for (int c0 = lane; c0 < nvec; c0 += 32 * B) {
      uint4 v[B][KMAX];
      uint4 a[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int c = c0 + 32 * b;
        if (c < nvec) {
#pragma unroll
          for (int j = 0; j < KMAX; ++j)
            if (p[j] >= 0) v[b][j] = __ldg(rows + p[j] * nvec + c);
          if (add) a[b] = __ldg(add + t * nvec + c);
        }
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int c = c0 + 32 * b;
        if (c >= nvec) continue;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (p[j] >= 0) {
            float f[8];
            unpack8(v[b][j], f);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = fmaf(wt[j], f[q], acc[q]);
          }
        if (add) {
          float f[8];
          unpack8(a[b], f);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] += f[q];
        }
        y[t * nvec + c] = pack8(acc);
      }
    }
  }
  griddep_launch();
}

// One warp per token: dyp[p_j] = w_j dy[t]; dw_j = <dy[t], yp[p_j]> (warp reduction);
// dlogits from dw for the softmax or the sigmoid gate.  Batches of B vectors per lane with
// all (1 + KMAX) * B loads issued first.
template <int KMAX>
__global__ void __launch_bounds__(THREADS)
combine_bwd_kernel(const uint4* __restrict__ dy, const uint4* __restrict__ yp,
                   const float* __restrict__ logits, const int32_t* __restrict__ topk_idx,
                   const float* __restrict__ topk_w, const int32_t* __restrict__ dest_row,
                   int64_t T, int E, int k, int nvec, int gate, float scale, int64_t rows_cap,
                   uint4* __restrict__ dyp, float* __restrict__ dlogits, int* err) {
  griddep_wait();   // see common.cuh: dependent launches
  constexpr int B = KMAX >= 6 ? 2 : 16 / (KMAX + 2);
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * THREADS) >> 5;
  for (int64_t t = gw; t < T; t += nw) {
    int64_t p[KMAX];
    float wt[KMAX];
    load_slots<KMAX>(dest_row, topk_w, t, k, rows_cap, err, p, wt);
    int my_e = -1;
    if (lane < k) {
      my_e = __ldg(topk_idx + t * k + lane);
      if (my_e < 0 || my_e >= E) {
        flag_error(err, MOE_DEVERR_BAD_INDEX);
        my_e = -1;
      }
    }
    int se[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) se[j] = __shfl_sync(FULL_MASK, my_e, j);
    float dot[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) dot[j] = 0.0f;
    for (int c0 = lane; c0 < nvec; c0 += 32 * B) {
      uint4 g[B];
      uint4 v[B][KMAX];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int c = c0 + 32 * b;
        if (c < nvec) {
          g[b] = __ldg(dy + t * nvec + c);
#pragma unroll
          for (int j = 0; j < KMAX; ++j)
            if (p[j] >= 0) v[b][j] = __ldg(yp + p[j] * nvec + c);
        }
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int c = c0 + 32 * b;
        if (c >= nvec) continue;
        float gf[8];
        unpack8(g[b], gf);
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (p[j] >= 0) {
            float f[8], o[8];
            unpack8(v[b][j], f);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              dot[j] = fmaf(gf[q], f[q], dot[j]);
              o[q] = wt[j] * gf[q];
            }
            dyp[p[j] * nvec + c] = pack8(o);
          }
      }
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) dot[j] = warp_sum(dot[j]);
    // Both gates normalise over the k selected experts, so the gradient of slot j is
    // proportional to dot_j - sum_i u_i dot_i with sum_i u_i = 1 (u: the normalised
    // scores).  It is summed pairwise, sum_i u_i (dot_j - dot_i): when one score carries
    // almost all the weight the direct form subtracts two nearly equal fp32 numbers and
    // keeps only a few bits of a tiny result, the pairwise form keeps them all.
    float dl[KMAX];
    if (gate == MOE_GATE_SOFTMAX_TOPK) {
      // dl_j = w_j (dot_j - sum_i w_i dot_i)
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        float acc = 0.0f;
#pragma unroll
        for (int i = 0; i < KMAX; ++i)
          if (i < k && i != j) acc = fmaf(wt[i], dot[j] - dot[i], acc);
        dl[j] = wt[j] * acc;
      }
    } else {
      // w_j = scale s_j / S with s = sigma(logit), S = sum_i s_i:
      // dl_j = scale / S^2 (sum_i s_i (dot_j - dot_i)) s_j (1 - s_j), with 1 - s_j taken
      // as sigma(-logit) so that it does not round to 0 for large logits
      float sg[KMAX], sm[KMAX], S = 0.0f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        sg[j] = 0.0f;
        sm[j] = 0.0f;
        if (j < k && se[j] >= 0) {
          const float l = __ldg(logits + t * E + se[j]);
          sg[j] = 1.0f / (1.0f + expf(-l));
          sm[j] = 1.0f / (1.0f + expf(l));
          S += sg[j];
        }
      }
      const float c = scale / (S * S);
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        float acc = 0.0f;
#pragma unroll
        for (int i = 0; i < KMAX; ++i)
          if (i < k && i != j) acc = fmaf(sg[i], dot[j] - dot[i], acc);
        dl[j] = c * acc * sg[j] * sm[j];
      }
    }
    for (int e = lane; e < E; e += 32) {
      float val = 0.0f;
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (j < k && se[j] == e) val = dl[j];
      dlogits[t * E + e] = val;
    }
  }
  griddep_launch();
}

}  // namespace

cudaError_t launch_permute(const void* x, const int32_t* src_tok, const int32_t* offsets, int E,
                           int64_t T, int64_t rows_cap, int d, void* xp, int* err,
                           cudaStream_t st) {
  return launch_pdl(permute_kernel, dim3(grid_warps(rows_cap)), dim3(THREADS), 0, st, 1,
                    static_cast<const uint4*>(x), src_tok, offsets, E, T, rows_cap, d / 8,
                    static_cast<uint4*>(xp), err);
}

cudaError_t launch_combine(const void* rows, const int32_t* dest_row, const float* w,
                           const void* add, int64_t T, int k, int d, int64_t rows_cap, void* y,
                           int* err, cudaStream_t st) {
  const int grid = grid_warps(T);
#define MOE_COMBINE(KM)                                                                       \
  launch_pdl(combine_kernel<KM>, dim3(grid), dim3(THREADS), 0, st, 1,                         \
             static_cast<const uint4*>(rows), dest_row, w, static_cast<const uint4*>(add), T,  \
             k, d / 8, rows_cap, static_cast<uint4*>(y), err)
  if (k <= 2) return MOE_COMBINE(2);
  if (k <= 4) return MOE_COMBINE(4);
  if (k <= 6) return MOE_COMBINE(6);
  return MOE_COMBINE(8);
#undef MOE_COMBINE
}

cudaError_t launch_combine_bwd(const void* dy, const void* yp, const float* logits,
                               const int32_t* topk_idx, const float* topk_w,
                               const int32_t* dest_row, int64_t T, int E, int k, int d,
                               int gate, float scale, int64_t rows_cap, void* dyp,
                               float* dlogits, int* err, cudaStream_t st) {
  const int grid = grid_warps(T);
#define MOE_COMBINE_BWD(KM)                                                                   \
  launch_pdl(combine_bwd_kernel<KM>, dim3(grid), dim3(THREADS), 0, st, 1,                     \
             static_cast<const uint4*>(dy), static_cast<const uint4*>(yp), logits, topk_idx,   \
             topk_w, dest_row, T, E, k, d / 8, gate, scale, rows_cap,                          \
             static_cast<uint4*>(dyp), dlogits, err)
  if (k <= 2) return MOE_COMBINE_BWD(2);
  if (k <= 4) return MOE_COMBINE_BWD(4);
  if (k <= 6) return MOE_COMBINE_BWD(6);
  return MOE_COMBINE_BWD(8);
#undef MOE_COMBINE_BWD
}

}  // namespace moe
