// route.cu -- F1/F2: top-k gating, per-expert histogram, capacity, exclusive scan and the
// padding-free buffer's side arrays.
//
// "MoE Training Optimization with Primus", Figure 7 dataflow: the router scores each
// token and picks its top-k experts.  X-MoE verdict page (arXiv 2508.13337), key
// machinery: the padding-free token buffer with token ids, expert ids, per-expert
// token counts and combine weights; referee minor comment on section 4.1.1 Listing 1
// (max_token_count from the capacity factor) and major comment on section 5.6 (drop
// only on capacity overflow).
//
// Three kernels, all deterministic:
//   1. route_topk_chunk: one CTA per 32-token chunk.  Each warp selects the top-k of 4
//      tokens with k rounds of a warp argmax over packed 64-bit keys
//      (order-preserving fp32 bits << 32 | (0xFFFF - expert)), so the larger logit and
//      then the lower id wins and NaN (key 0) ranks below -inf.  The chunk then ORs one
//      bit per token into a per-expert 32-bit mask in shared memory; popc of the mask
//      gives the chunk's count of each expert and popc of the bits below a token its
//      rank inside the chunk -- an order fixed by token index, not by atomics.
//   2. route_scan: one CTA.  Per expert, an exclusive scan of the chunk counts (in
//      place) gives each chunk's base rank; kept = min(count, cap) and an exclusive
//      scan of kept gives the segment offsets.
//   3. route_assign: one thread per (t, j): rank = chunk base + rank in chunk; kept
//      slots get dest_row = offsets[e] + rank and fill the inverse maps.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int CHUNK = 32;
constexpr int ROUTE_THREADS = 256;   // 8 warps x 4 tokens = one 32-token chunk

__device__ __forceinline__ uint32_t order_key(float x, bool& is_nan) {
  uint32_t u = __float_as_uint(x);
  if (x != x) {
    is_nan = true;
    return 0u;   // below every real key (-inf maps to 0x007FFFFF)
  }
  if (x == 0.0f) u = 0u;   // +0 and -0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int VPL>
__global__ void __launch_bounds__(ROUTE_THREADS)
route_topk_chunk_kernel(const float* __restrict__ logits, int64_t T, int E, int k, int gate,
                        float scale, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                        int32_t* __restrict__ rank_out, int32_t* __restrict__ chunk_cnt,
                        int64_t nch, int* err) {
  __shared__ int s_idx[CHUNK][8];
  __shared__ uint32_t s_bits[256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t chunk = blockIdx.x;
  const int64_t t0 = chunk * CHUNK;
  for (int e = threadIdx.x; e < E; e += ROUTE_THREADS) s_bits[e] = 0u;

#pragma unroll 1
  for (int i = 0; i < CHUNK / 8; ++i) {
    const int tl = warp * (CHUNK / 8) + i;
    const int64_t t = t0 + tl;
    if (t >= T) {
      if (lane < 8) s_idx[tl][lane] = -1;
      continue;
    }
    const float* row = logits + t * E;
    float v[VPL];
    unsigned long long key[VPL];
    bool nan_here = false;
#pragma unroll
    for (int s = 0; s < VPL; ++s) {
      const int e = lane + 32 * s;
      if (e < E) {
        v[s] = row[e];
        const uint32_t kf = order_key(v[s], nan_here);
        key[s] = (static_cast<unsigned long long>(kf) << 32) | (0xFFFFu - static_cast<uint32_t>(e));
      } else {
        v[s] = 0.0f;
        key[s] = 0ull;   // padding never wins: k <= E real keys are all > 0
      }
    }
    if (__any_sync(FULL_MASK, nan_here) && lane == 0) flag_error(err, MOE_DEVERR_NAN_LOGIT);

    int sel_e[8];
    float sel_l[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      sel_e[j] = 0;
      sel_l[j] = 0.0f;
      if (j < k) {
        unsigned long long best = key[0];
#pragma unroll
        for (int s = 1; s < VPL; ++s) best = key[s] > best ? key[s] : best;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long other = __shfl_xor_sync(FULL_MASK, best, o);
          best = other > best ? other : best;
        }
        const int e = 0xFFFF - static_cast<int>(best & 0xFFFFull);
        const int owner = e & 31, slot = e >> 5;
        float mine = 0.0f;
#pragma unroll
        for (int s = 0; s < VPL; ++s)
          if (s == slot) {
            mine = v[s];
            if (lane == owner) key[s] = 0ull;   // remove the winner
          }
        sel_e[j] = e;
        sel_l[j] = __shfl_sync(FULL_MASK, mine, owner);
      }
    }

    // gate weights over the k selected (sel_l[0] is the largest selected logit)
    float w[8];
    float z = 0.0f;
    if (gate == MOE_GATE_SOFTMAX_TOPK) {
      const float m = sel_l[0];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < k) {
          w[j] = expf(sel_l[j] - m);
          z += w[j];
        }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < k) w[j] = w[j] / z;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < k) {
          w[j] = 1.0f / (1.0f + expf(-sel_l[j]));
          z += w[j];
        }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < k) w[j] = scale * w[j] / z;
    }
    int my_e = 0;
    float my_w = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j == lane) {
        my_e = sel_e[j];
        my_w = w[j];
      }
    if (lane < k) {
      topk_idx[t * k + lane] = my_e;
      topk_w[t * k + lane] = my_w;
      s_idx[tl][lane] = my_e;
    }
  }
  __syncthreads();

  // chunk histogram as per-expert token bitmasks (OR is order-free: deterministic)
  const int tok = threadIdx.x >> 3, j = threadIdx.x & 7;
  int e = -1;
  if (j < k) e = s_idx[tok][j];
  if (e >= 0) atomicOr(&s_bits[e], 1u << tok);
  __syncthreads();
  if (e >= 0) rank_out[(t0 + tok) * k + j] = __popc(s_bits[e] & ((1u << tok) - 1u));
  for (int x = threadIdx.x; x < E; x += ROUTE_THREADS)
    chunk_cnt[static_cast<int64_t>(x) * nch + chunk] = __popc(s_bits[x]);
}

__global__ void __launch_bounds__(1024)
route_scan_kernel(int32_t* __restrict__ chunk_cnt, int64_t nch, int E, int cap,
                  int32_t* __restrict__ counts, int32_t* __restrict__ kept,
                  int32_t* __restrict__ offsets) {
  __shared__ int s_kept[256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = warp; e < E; e += 32) {
    int32_t* col = chunk_cnt + static_cast<int64_t>(e) * nch;
    int running = 0;
    for (int64_t base = 0; base < nch; base += 32) {
      const int64_t c = base + lane;
      const int v = c < nch ? col[c] : 0;
      const int incl = warp_incl_scan(v);
      if (c < nch) col[c] = running + incl - v;   // chunk's base rank for expert e
      running += __shfl_sync(FULL_MASK, incl, 31);
    }
    if (lane == 0) {
      const int kp = (cap > 0 && running > cap) ? cap : running;
      counts[e] = running;
      kept[e] = kp;
      s_kept[e] = kp;
    }
  }
  __syncthreads();
  if (warp == 0) {
    int vals[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      vals[i] = e < E ? s_kept[e] : 0;
      sum += vals[i];
    }
    const int incl = warp_incl_scan(sum);
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < E) offsets[e] = run;
      run += vals[i];
    }
    if (lane == 31) offsets[E] = incl;
  }
}

__global__ void __launch_bounds__(256)
route_assign_kernel(const int32_t* __restrict__ topk_idx, int64_t T, int k, int E, int cap,
                    const int32_t* __restrict__ chunk_base, int64_t nch,
                    const int32_t* __restrict__ offsets, int32_t* __restrict__ dest_row,
                    int32_t* __restrict__ src_tok, int32_t* __restrict__ src_slot,
                    uint8_t* __restrict__ drop_mask) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t R = T * k;
  if (i >= R) return;
  const int total = offsets[E];
  if (i >= total) {
    src_tok[i] = -1;
    src_slot[i] = -1;
  }
  const int64_t t = i / k;
  const int e = topk_idx[i];
  const int r = chunk_base[static_cast<int64_t>(e) * nch + t / CHUNK] + dest_row[i];
  if (cap > 0 && r >= cap) {
    dest_row[i] = -1;
    drop_mask[i] = 1;
  } else {
    const int p = offsets[e] + r;
    dest_row[i] = p;
    drop_mask[i] = 0;
    src_tok[p] = static_cast<int32_t>(t);
    src_slot[p] = static_cast<int32_t>(i);
  }
}

}  // namespace

cudaError_t launch_route(const float* logits, int64_t T, int E, int k, int gate, float scale,
                         int capacity, int32_t* topk_idx, float* topk_w, int32_t* counts,
                         int32_t* kept, int32_t* offsets, int32_t* dest_row, int32_t* src_tok,
                         int32_t* src_slot, uint8_t* drop_mask, int32_t* chunk_scratch,
                         int* err, cudaStream_t st) {
  const int64_t nch = route_chunks(T);
  const dim3 g1(static_cast<unsigned>(nch));
#define MOE_ROUTE_LAUNCH(V)                                                                  \
  route_topk_chunk_kernel<V><<<g1, ROUTE_THREADS, 0, st>>>(logits, T, E, k, gate, scale,    \
                                                            topk_idx, topk_w, dest_row,      \
                                                            chunk_scratch, nch, err)
  if (E <= 32) MOE_ROUTE_LAUNCH(1);
  else if (E <= 64) MOE_ROUTE_LAUNCH(2);
  else if (E <= 128) MOE_ROUTE_LAUNCH(4);
  else MOE_ROUTE_LAUNCH(8);
#undef MOE_ROUTE_LAUNCH
  route_scan_kernel<<<1, 1024, 0, st>>>(chunk_scratch, nch, E, capacity, counts, kept, offsets);
  const int64_t R = T * k;
  route_assign_kernel<<<static_cast<unsigned>((R + 255) / 256), 256, 0, st>>>(
      topk_idx, T, k, E, capacity, chunk_scratch, nch, offsets, dest_row, src_tok, src_slot,
      drop_mask);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------------------
// moe_route_noalloc: the routing step for callers that cannot allocate device memory.
//
// Some callers cannot hand us a workspace: a plugin living inside a host framework that
// owns every byte of device memory through its own pool (and forbids cudaMalloc from
// anyone else), or a latency-critical caller that cannot risk the implicit device-wide
// synchronisation a cudaMalloc/cudaFree may bring.  For them this entry point keeps the
// routing histogram's scratch in a fixed array compiled into the library instead of in
// the caller's `ws`.  The caller still passes every input and output.
//
// The array below is MOE_NOALLOC_ROUTE_SCRATCH_BYTES (1 MiB) per GPU; every GPU that loads
// the library holds it until the process exits.  All calls share it and it keeps the last
// call's contents (the kernels overwrite every entry they read, so nothing needs
// clearing); calls whose execution overlaps on the GPU therefore race on it.
namespace {

__device__ __align__(256) int32_t g_noalloc_route_scratch[MOE_NOALLOC_ROUTE_SCRATCH_BYTES /
                                                          sizeof(int32_t)];

constexpr int kMaxDevices = 64;
std::once_flag g_noalloc_once[kMaxDevices];
int32_t* g_noalloc_ptr[kMaxDevices];
cudaError_t g_noalloc_err[kMaxDevices];

// The host-side name of a __device__ array is only a stand-in, not a device address:
// look the real address up once per device, with that device current.
cudaError_t noalloc_scratch(int dev, int32_t** out) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_noalloc_once[dev], [dev] {
    void* p = nullptr;
    g_noalloc_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_route_scratch);
    g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
  });
  *out = g_noalloc_ptr[dev];
  return g_noalloc_err[dev];
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route_noalloc(const moe_config_t* cfg, const float* logits,
                                          int32_t* topk_idx, float* topk_w, int32_t* counts,
                                          int32_t* kept, int32_t* offsets, int32_t* dest_row,
                                          int32_t* src_tok, int32_t* src_slot,
                                          uint8_t* drop_mask, int32_t* dev_flags_or_null,
                                          void* stream) {
  size_t ws_bytes = 0;
  const moe_status_t s = moe_workspace_size(cfg, &ws_bytes, nullptr);   // validates cfg
  if (s != MOE_OK) return s;
  const void* ptrs[] = {logits, topk_idx, topk_w, counts, kept, offsets, dest_row, src_tok,
                        src_slot, drop_mask};
  for (const void* p : ptrs)
    if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) return MOE_ERR_INVALID_ARG;
  if (dev_flags_or_null && (reinterpret_cast<uintptr_t>(dev_flags_or_null) & 3u))
    return MOE_ERR_INVALID_ARG;
  if (moe::route_scratch_bytes(cfg->T, cfg->E) > MOE_NOALLOC_ROUTE_SCRATCH_BYTES)
    return MOE_ERR_UNSUPPORTED;   // the fixed scratch is too small for this T x E
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t* scratch = nullptr;
  if (moe::noalloc_scratch(dev, &scratch) != cudaSuccess || !scratch) return MOE_ERR_CUDA;
  const cudaError_t e = moe::launch_route(
      logits, cfg->T, cfg->E, cfg->k, cfg->gate, cfg->route_scale, cfg->capacity, topk_idx,
      topk_w, counts, kept, offsets, dest_row, src_tok, src_slot, drop_mask, scratch,
      dev_flags_or_null, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
