// mx.cu -- the MXFP8 path of the routed experts: quantisation kernels and the block-scaled
// grouped GEMMs (FC1 + SwiGLU + quantisation of h, FC2; the FC2 data-gradient with the
// SwiGLU backward quantising dab, the FC1 data-gradient; and, at mxfp8 = 2, the weight
// gradients on operands quantised along each expert segment's tokens).
//
// "MoE Training Optimization with Primus", FP8 section: the MXFP8 recipe (OCP E4M3
// elements with per-block power-of-two scales) for the routed-expert grouped GEMMs, and
// weight-quantisation caching; MegaMoE section: the SwiGLU step quantises its own output,
// so the cast is never a separate pass.  Block rule (OCP Microscaling formats v1.0): a
// block is 32 consecutive elements along the contraction axis; its scale is the E8M0
// power of two 2^X with X = floor(log2(max |v|)) - 8 (8 = the exponent of E4M3's largest
// value, 448), clamped to [-127, 127], -127 for an all-zero block; elements are v / 2^X
// rounded to E4M3 (nearest, ties to even, saturating at 448).
//
// Tensor-core path: tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale, M 128 x N 256 x
// K 32 per instruction, E4M3 operands in 128-byte-swizzled shared memory (one K block =
// 128 elements = one 128-byte row), fp32 accumulation in TMEM.  The scales live in TMEM:
// the MMA reads row m's scale of A from lane m, column base + m/32, byte = the sub-block
// (0..3) named in the instruction descriptor, and column n's scale of B from lane n%32 of
// every lane quarter, column base + n/32.  tcgen05.cp.32x128b.warpx4 produces exactly that
// from a 512-byte "atom" in shared memory: byte 16*(m%32) + 4*(m/32) + k holds the scale of
// row m, sub-block k (the layout was measured with an in-bounds probe on GB300).
//
// Every scale is stored in atom order, so a stage's scales arrive by TMA like its
// operands: the weights' when they are quantised (cached by the caller), the activations'
// by the kernels that produce them -- tiled by 128 rows inside each expert segment (atom
// block (offsets[e] >> 7) + e + l/128 for local row l), so a tile's rows always fill whole
// atoms whatever the segment's start.
//
// Long segments run on CTA pairs (cta_group::2, M 256 x N 256): each CTA holds 128 rows of
// A and 128 rows of B; the MMA reads each CTA's A scales from that CTA's TMEM and, for its
// 128 output rows, the B scales of all 256 columns from the same CTA's TMEM, so both CTAs
// load the whole B scale pair; tcgen05.cp.cta_group::2 issued by the leader copies each
// CTA's own shared-memory atoms into its own TMEM (measured with a second probe).
//
// TMEM holds one 256-column accumulator and up to 6 stages x 12 scale columns.  There is
// no room for a second accumulator, so eight epilogue warps (two per lane quarter, each
// taking half the columns) copy the accumulator into registers and release it at once;
// the next tile's MMAs then overlap the epilogue's arithmetic and stores.
//
// Weight gradients (GEMM_WGRAD): dW[e] = A_e^T B_e with the contraction over the expert's
// rows.  mx_quant_tok_kernel writes each operand transposed ([C][128 kb_cap] codes, K-major
// along the rows) with each expert's rows as whole 128-row K blocks (the last one
// zero-padded), 32-row MX blocks starting at the segment's first row, and the scales in
// the atom layout of the operand's GEMM role; the GEMM walks every expert's fixed
// weight-shaped tile grid over its K blocks and writes dW through TMA stores.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp8.h>

#include <cstddef>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__device__ ClockTrace g_clock_trace;   // see ClockTrace (common.cuh)

constexpr int MX_BK = 128;                 // E4M3 elements (bytes) per K block
constexpr int MX_SFA_BYTES = 512;          // one scale atom
constexpr int MX_SFB_BYTES = 1024;         // a pair of atoms: 256 B rows
constexpr int MX_THREADS = 320;            // producer, MMA, 8 epilogue warps
constexpr int MX_EPI_WARPS = 8;
constexpr uint32_t MX_TMEM_COLS = 512;
constexpr uint32_t MX_SF_COL0 = 256;       // scale slots: 12 columns per stage (up to 6)
constexpr int MX_MAX_G = 256;
constexpr long long MX_WAIT_BUDGET = 4000000000LL;

// ------------------------------------------------------------------ quantisation helpers
// X = floor(log2(amax)) - 8, clamped to [-127, 127]; -127 when amax is 0 (or subnormal,
// whose floor(log2) lies below -127 anyway).
__device__ __forceinline__ int mx_exponent(float amax) {
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);
  if (e == 0) return -127;
  const int X = e - 127 - 8;
  return X < -127 ? -127 : X;   // at most 254 - 135 = 119: never above 127
}

// 2^n for n in [-126, 127] (normal fp32)
__device__ __forceinline__ float exp2_int(int n) {
  return __uint_as_float(static_cast<uint32_t>(n + 127) << 23);
}

// two values -> two E4M3 codes (round to nearest even, saturate to +-448); a in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE,
                                                        __NV_E4M3));
}

// Quantise one block of 32 values: 32 codes into c[8] (4 per word, element 0 lowest),
// returns the E8M0 scale code.
__device__ __forceinline__ uint32_t mx_block(const float* v, uint32_t* c) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int X = mx_exponent(amax);
  const float inv = exp2_int(-X);   // -X in [-119, 127]: exact scaling
#pragma unroll
  for (int w = 0; w < 8; ++w)
    c[w] = e4m3x2(v[4 * w] * inv, v[4 * w + 1] * inv) |
           (e4m3x2(v[4 * w + 2] * inv, v[4 * w + 3] * inv) << 16);
  return static_cast<uint32_t>(X + 127);
}

// mx_block on 32 bf16 values packed in 4 uint4 (element 0 in the low half of v[0].x).
__device__ __forceinline__ uint32_t mx_block_bf16(const uint4* v, uint32_t* c) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(v);
  auto lo = [](uint32_t x) { return __uint_as_float(x << 16); };
  auto hi = [](uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); };
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fmaxf(fabsf(lo(w[i])), fabsf(hi(w[i]))));
  const int X = mx_exponent(amax);
  const float inv = exp2_int(-X);
#pragma unroll
  for (int q = 0; q < 8; ++q)
    c[q] = e4m3x2(lo(w[2 * q]) * inv, hi(w[2 * q]) * inv) |
           (e4m3x2(lo(w[2 * q + 1]) * inv, hi(w[2 * q + 1]) * inv) << 16);
  return static_cast<uint32_t>(X + 127);
}

// Byte offset of (row m of a 128-row block, sub-block k) inside a scale atom.
__host__ __device__ __forceinline__ int atom_byte(int m, int k) {
  return 16 * (m & 31) + 4 * (m >> 5) + k;
}

// Byte of the scale of sub-block j (32 elements) of K block kb, for local row l of
// expert e (segment start seg0), in an activation atom array with KB K blocks per row.
__host__ __device__ __forceinline__ long long act_atom_byte(int seg0, int e, int l, int KB,
                                                            int kb, int j) {
  const long long blk = (seg0 >> 7) + e + (l >> 7);
  return (blk * KB + kb) * 512 + atom_byte(l & 127, j);
}

// Expert of row p: the e with offsets[e] <= p < offsets[e+1] (binary search; empty
// segments are skipped because their start equals the next one's).
__device__ __forceinline__ int expert_of_row(const int32_t* __restrict__ offsets, int E, int64_t p) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(offsets + mid) <= p) lo = mid;
    else hi = mid;
  }
  return lo;
}

// ------------------------------------------------------------------ F3 + quantisation
// Warp per destination row p < offsets[E]: x[src_tok[p]] (bf16, d elements) is quantised
// into xq[p] (E4M3) and its scales (E8M0 per 32 elements, into the activation atoms); with
// xp != null the bf16 row is also copied (the backward's saved input).  Lane l takes
// blocks l, l+32, ...
constexpr int QTHREADS = 256;

__global__ void __launch_bounds__(QTHREADS)
mx_permute_quant_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ src_tok,
                        const int32_t* __restrict__ offsets, int E, int64_t T, int64_t rows_cap,
                        int d, uint4* __restrict__ xp, uint4* __restrict__ xq,
                        uint8_t* __restrict__ x_sf, int* err) {
  griddep_wait();   // see common.cuh: dependent launches
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * QTHREADS + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * QTHREADS) >> 5;
  int64_t n_rows = offsets[E];
  if (n_rows < 0 || n_rows > rows_cap) {
    if (gw == 0 && lane == 0) flag_error(err, MOE_DEVERR_BAD_OFFSETS);
    n_rows = n_rows < 0 ? 0 : rows_cap;
  }
  const int nb = d / 32;
  for (int64_t p = gw; p < n_rows; p += nw) {
    // src_tok == null: the rows are quantised in place (x has rows_cap rows, t = p)
    const int t = src_tok ? __ldg(src_tok + p) : static_cast<int>(p);
    if (t < 0 || t >= T) {
      if (lane == 0) flag_error(err, MOE_DEVERR_BAD_INDEX);
      continue;
    }
    const uint4* src = x + static_cast<int64_t>(t) * (d / 8);
    const int e = expert_of_row(offsets, E, p);
    const int seg0 = __ldg(offsets + e);
    const int l = static_cast<int>(p - seg0);
    for (int b = lane; b < nb; b += 32) {
      uint4 raw[4];
      float v[32];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        raw[i] = __ldg(src + 4 * b + i);
        unpack8(raw[i], v + 8 * i);
      }
      if (xp) {
#pragma unroll
        for (int i = 0; i < 4; ++i) xp[p * (d / 8) + 4 * b + i] = raw[i];
      }
      uint32_t c[8];
      const uint32_t s = mx_block(v, c);
      uint4* dq = xq + p * (d / 16) + 2 * b;
      dq[0] = make_uint4(c[0], c[1], c[2], c[3]);
      dq[1] = make_uint4(c[4], c[5], c[6], c[7]);
      x_sf[act_atom_byte(seg0, e, l, d / 128, b >> 2, b & 3)] = static_cast<uint8_t>(s);
    }
  }
  griddep_launch();
}

// Weight quantisation, warp per weight row.  W1 [E][2f][d]: codes row-major into w1q,
// scales into atoms [E][f/128][d/128][2 halves][512 B] (half 0: gate rows, 1: up rows).
// W2 [E][d][f]: codes into w2q, scales into atoms [E][ceil(d/256)][f/128][2][512 B].
__global__ void __launch_bounds__(QTHREADS)
mx_weight_quant_kernel(const uint4* __restrict__ W, int64_t n_rows, int rows_per_expert,
                       int K, int which, int f, int n_blocks_mn, uint4* __restrict__ wq,
                       uint8_t* __restrict__ atoms) {
  griddep_wait();   // see common.cuh: dependent launches
  const int lane = threadIdx.x & 31;
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * QTHREADS + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * QTHREADS) >> 5;
  const int nb = K / 32, KB = K / 128;
  for (int64_t r = gw; r < n_rows; r += nw) {
    const int64_t e = r / rows_per_expert;
    const int re = static_cast<int>(r - e * rows_per_expert);
    int half, blk, m;
    if (which == 0) {   // W1: gate rows [0, f), up rows [f, 2f); 128-row blocks per half
      half = re >= f ? 1 : 0;
      const int rr = re - half * f;
      blk = rr >> 7;
      m = rr & 127;
    } else {            // W2: 256-row N tiles, two 128-row halves each
      blk = re >> 8;
      half = (re >> 7) & 1;
      m = re & 127;
    }
    const uint4* src = W + r * (K / 8);
    for (int b = lane; b < nb; b += 32) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 4; ++i) unpack8(__ldg(src + 4 * b + i), v + 8 * i);
      uint32_t c[8];
      const uint32_t s = mx_block(v, c);
      uint4* dq = wq + r * (K / 16) + 2 * b;
      dq[0] = make_uint4(c[0], c[1], c[2], c[3]);
      dq[1] = make_uint4(c[4], c[5], c[6], c[7]);
      const int kb = b >> 2, k1 = b & 3;
      const int64_t atom = ((e * n_blocks_mn + blk) * KB + kb) * 2 + half;
      atoms[atom * 512 + atom_byte(m, k1)] = static_cast<uint8_t>(s);
    }
  }
  griddep_launch();
}

// Transposed weight quantisation for the data-gradient GEMMs: for each expert, Wt = W^T
// ([C][Rk] from W [Rk][C]) quantised along Rk (the contraction axis of the backward GEMM),
// codes row-major into wtq and scales into atoms [E][ceil(C/256)][Rk/128][2][512] (the
// weight-atom layout of a B operand with N = C).  One CTA takes a 128 (Rk) x 64 (C) tile
// through shared memory: coalesced row reads, then one thread per (column, 32-row block).
constexpr int TQ_ROWS = 128, TQ_COLS = 64;

__global__ void __launch_bounds__(256)
mx_weight_quant_t_kernel(const __nv_bfloat16* __restrict__ W, int Rk, int C,
                         uint8_t* __restrict__ wtq, uint8_t* __restrict__ atoms) {
  griddep_wait();   // see common.cuh: dependent launches
  __shared__ __nv_bfloat16 tile[TQ_ROWS][TQ_COLS + 2];   // +2: stagger the banks
  const int e = blockIdx.z;
  const int r0 = blockIdx.y * TQ_ROWS, c0 = blockIdx.x * TQ_COLS;
  const __nv_bfloat16* src = W + static_cast<long long>(e) * Rk * C;
  for (int i = threadIdx.x; i < TQ_ROWS * TQ_COLS / 2; i += blockDim.x) {
    const int r = i / (TQ_COLS / 2), c2 = (i % (TQ_COLS / 2)) * 2;
    const __nv_bfloat162 v =
        *reinterpret_cast<const __nv_bfloat162*>(src + static_cast<long long>(r0 + r) * C + c0 + c2);
    tile[r][c2] = v.x;
    tile[r][c2 + 1] = v.y;
  }
  __syncthreads();
  const int c = threadIdx.x % TQ_COLS, blk = threadIdx.x / TQ_COLS;   // 4 blocks of 32 rows
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __bfloat162float(tile[32 * blk + i][c]);
  uint32_t code[8];
  const uint32_t sc = mx_block(v, code);
  const int col = c0 + c;                                   // the output row (N index)
  uint4* dq = reinterpret_cast<uint4*>(wtq + (static_cast<long long>(e) * C + col) * Rk + r0 +
                                       32 * blk);
  dq[0] = make_uint4(code[0], code[1], code[2], code[3]);
  dq[1] = make_uint4(code[4], code[5], code[6], code[7]);
  const int KB = Rk / 128, NT = (C + 255) / 256;
  const int kb = r0 / 128, j = blk;                          // r0 is a multiple of 128
  const long long atom = ((static_cast<long long>(e) * NT + col / 256) * KB + kb) * 2 + ((col >> 7) & 1);
  atoms[atom * 512 + atom_byte(col & 127, j)] = static_cast<uint8_t>(sc);
  griddep_launch();
}

// Along-token quantisation for the weight gradients: X [rows_cap][C] bf16 holds the expert
// segments; expert e's rows form K blocks kb0_e .. kb0_e + ceil(n_e / 128) - 1 of 128 rows
// (the last zero-padded).  For each column and each 32-row block: E4M3 codes into
// xtq[c][128 kb + 32 j ..] and the E8M0 scale into the atom of the column's GEMM role (M
// operand: atom (c / 128) kb_cap + kb; N operand: ((c / 256) kb_cap + kb) 2 + (c / 128) % 2).
// One CTA per (64 columns, K block): the 128 x 64 tile goes through shared memory.
constexpr int KQ_COLS = 64;

__global__ void __launch_bounds__(256)
mx_quant_tok_kernel(const __nv_bfloat16* __restrict__ X, const int32_t* __restrict__ offsets,
                    int E, long long rows_cap, int C, int kb_cap, int role_n,
                    uint8_t* __restrict__ xtq, uint8_t* __restrict__ atoms, int* err) {
  griddep_wait();   // see common.cuh: dependent launches
  __shared__ __nv_bfloat16 tile[128][KQ_COLS + 2];   // +2: stagger the banks
  __shared__ int s_kb0[MX_MAX_G + 1];
  __shared__ int s_wsum[8];
  __shared__ int s_bad;
  const int c0 = blockIdx.x * KQ_COLS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  // K blocks per expert and their exclusive prefix (E <= 256: one expert per thread)
  int nkb = 0;
  if (tid < E) {
    const int a = offsets[tid], b = offsets[tid + 1];
    if (a < 0 || b < a || b > rows_cap) s_bad = 1;
    nkb = b > a ? (b - a + 127) / 128 : 0;
  }
  const int incl = warp_incl_scan(nkb);
  if (lane == 31) s_wsum[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += s_wsum[w];
  if (tid < E) s_kb0[tid] = before + incl - nkb;
  if (tid == E - 1) s_kb0[E] = before + incl;
  __syncthreads();
  if (s_bad) {
    if (blockIdx.y == 0 && blockIdx.x == 0 && tid == 0) flag_error(err, MOE_DEVERR_BAD_OFFSETS);
    return;
  }
  // this CTA's K blocks: kb, kb + gridDim.y, ... below the experts' total.  The next
  // block's rows are loaded into registers while the current one is quantised.
  const int total = s_kb0[E];
  auto block_rows = [&](int kb, long long& r0, long long& r_end) {
    int lo = 0, hi = E;                            // s_kb0[lo] <= kb < s_kb0[lo + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_kb0[mid] <= kb) lo = mid;
      else hi = mid;
    }
    r0 = static_cast<long long>(offsets[lo]) + 128LL * (kb - s_kb0[lo]);
    r_end = offsets[lo + 1];
  };
  constexpr int PER = 128 * (KQ_COLS / 8) / 256;   // 16-byte pieces per thread (4)
  auto load_block = [&](int kb, uint4* reg) {
    long long r0, r_end;
    block_rows(kb, r0, r_end);
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = tid + 256 * u;
      const int r = i / (KQ_COLS / 8), c8 = (i % (KQ_COLS / 8)) * 8;
      reg[u] = r0 + r < r_end
                   ? __ldg(reinterpret_cast<const uint4*>(X + (r0 + r) * C + c0 + c8))
                   : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  uint4 cur[PER];
  if (static_cast<int>(blockIdx.y) < total) load_block(blockIdx.y, cur);
  for (int kb = blockIdx.y; kb < total; kb += gridDim.y) {
    __syncthreads();                               // the previous block's tile is consumed
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int i = tid + 256 * u;
      const int r = i / (KQ_COLS / 8), c8 = (i % (KQ_COLS / 8)) * 8;
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&cur[u]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        tile[r][c8 + 2 * q] = h2[q].x;
        tile[r][c8 + 2 * q + 1] = h2[q].y;
      }
    }
    __syncthreads();
    if (kb + static_cast<int>(gridDim.y) < total) load_block(kb + gridDim.y, cur);
    const int c = tid % KQ_COLS, j = tid / KQ_COLS;   // 4 blocks of 32 rows
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __bfloat162float(tile[32 * j + i][c]);
    uint32_t code[8];
    const uint32_t sc = mx_block(v, code);
    const int col = c0 + c;
    const long long kcap = 128LL * kb_cap;
    uint4* dq = reinterpret_cast<uint4*>(xtq + static_cast<long long>(col) * kcap + 128LL * kb +
                                         32 * j);
    dq[0] = make_uint4(code[0], code[1], code[2], code[3]);
    dq[1] = make_uint4(code[4], code[5], code[6], code[7]);
    const long long atom =
        role_n ? ((static_cast<long long>(col / 256) * kb_cap + kb) * 2 + ((col >> 7) & 1))
               : (static_cast<long long>(col / 128) * kb_cap + kb);
    atoms[atom * 512 + atom_byte(col & 127, j)] = static_cast<uint8_t>(sc);
  }
  griddep_launch();
}

// ------------------------------------------------------------------ block-scaled GEMM
// Per CTA and stage: A 128 rows x 128 B, B 128 rows (pair: this CTA's half of N) or 256
// rows (one CTA) x 128 B, the A scale atom (512 B) and the B scale pair (1 KB).  WG (the
// weight-gradient mode): 4 stages (its K is one expert's rows, a few K blocks) and a
// TMA-store staging area, two 32 x 64 bf16 boxes (4 KB each) per epilogue warp.
template <int PAIR, int MODE>
struct MxGeo {
  static constexpr bool WG = MODE == GEMM_WGRAD;
  // the CTA-pair FC2 data-gradient transposes fp32 dh through 4 KB per warp
  static constexpr bool XD2 = MODE == GEMM_DGRAD2_SWIGLU && PAIR == 2;
  static constexpr int B_ROWS = 256 / PAIR;
  static constexpr int A_BYTES = 128 * MX_BK;
  static constexpr int B_BYTES = B_ROWS * MX_BK;
  static constexpr int SFA_OFF = A_BYTES + B_BYTES;
  static constexpr int SFB_OFF = SFA_OFF + MX_SFA_BYTES;
  static constexpr int LOAD_BYTES = A_BYTES + B_BYTES + MX_SFA_BYTES + MX_SFB_BYTES;
  static constexpr int STAGE_BYTES = (LOAD_BYTES + 1023) / 1024 * 1024;
  static constexpr int STAGES = (WG || PAIR == 1) ? 4 : (XD2 ? 5 : 6);
  // WG: TMA-store staging; otherwise each epilogue warp's transpose block through which
  // its rows leave as 16-byte pieces: 2 KB (32 rows of 64 bytes), 4 KB for XD2
  static constexpr int STAGING_BYTES =
      WG ? MX_EPI_WARPS * 2 * 4096 : MX_EPI_WARPS * (XD2 ? 4096 : 2048);
  static constexpr int TILE_M = 128 * PAIR;
};
static_assert(MX_SF_COL0 + 12 * 6 <= MX_TMEM_COLS, "scale slots");

struct MxCtl {
  uint64_t full[6];
  uint64_t empty[6];
  uint64_t tfull;
  uint64_t tempty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int bad;
  int pad;
  int gstart[MX_MAX_G + 2];
  int tprefix[MX_MAX_G + 2];
  int kbpre[MX_MAX_G + 2];    // WGRAD: each expert's first K block (exclusive prefix)
};

template <int PAIR, int MODE>
constexpr size_t mx_smem_bytes() {
  using GE = MxGeo<PAIR, MODE>;
  return 1024 + GE::STAGES * GE::STAGE_BYTES + GE::STAGING_BYTES + sizeof(MxCtl);
}

struct MxParams {
  int G;
  long long rows_cap;
  int d, f;
  int num_n_tiles;
  int num_kb;
  int n_out;
  int n_blocks_mn;            // B atom blocks per expert (W1: f/128, W2: ceil(d/256))
  int b_rows;                 // B rows per expert for the 256-row N tiles (FC2 d, DGRAD2 f,
                              // DGRAD1 d)
  const int32_t* offsets;
  const __nv_bfloat16* aux;   // DGRAD2: the saved pre-activations ab [rows][2f]
  __nv_bfloat16* out0;        // FC1: ab  FC2: yp  DGRAD2: dab  DGRAD1: dxp
  __nv_bfloat16* out1;        // FC1: h
  uint8_t* out_q;             // FC1: hq [rows_cap][f]   DGRAD2: dab codes [rows_cap][2f]
  uint8_t* out_sf;            // FC1: h's scales (K blocks f/128)  DGRAD2: dab's (2f/128)
  int* err;
  // WGRAD: dW [G][wg_M][wg_N]; both operands along-token quantised (kb_cap K blocks)
  int wg_M, wg_N, wg_m_tiles, kb_cap;
};

__device__ __forceinline__ int mx_ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return make_smem_desc(saddr, 16, 1024);
}
// no-swizzle descriptor of a 32-row x 16-byte scale atom (8-row core matrices 128 B apart)
__device__ __forceinline__ uint64_t sdesc_atom(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>(128 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}
// kind::mxf8f6f4 instruction descriptor: E4M3 x E4M3, K-major A and B, UE8M0 scales;
// [4,6) B scale sub-block, [7,10) A type, [10,13) B type, [17,23) N>>3, [23] scale type
// UE8M0, [24,29) M>>4, [29,31) A scale sub-block.
__device__ __forceinline__ uint32_t idesc_mx(int M, int N, int sf_id) {
  return (static_cast<uint32_t>(sf_id) << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
         (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) |
         (static_cast<uint32_t>(sf_id) << 29);
}
template <int PAIR>
__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                          uint32_t accumulate) {
  if (PAIR == 2)
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
        "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
        "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}
template <int PAIR>
__device__ __forceinline__ void tc_cp_atom(uint32_t taddr, uint64_t sdesc) {
  if (PAIR == 2)
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
  else
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

__device__ __forceinline__ bool mx_warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                             int* err, long long budget) {
  return __all_sync(FULL_MASK, mbar_wait_bounded(bar, parity, abort, err, budget));
}

__device__ __forceinline__ float silu_mx(float a) { return a * sigmoid_fast(a); }
__device__ __forceinline__ void mx_st_shared_v4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 mx_ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float bf16r(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// tmA: the activation codes [rows, K] (box 128 x 128); tmB: the weight codes (box 128 x
// 128); tmSA: the activation scale atoms viewed as [*, 256] bytes (box 256 x 2 = one atom);
// tmSB: the weight scale atoms viewed as [*, 256] bytes (box 256 x 4 = one atom pair).
// WGRAD: A and B are along-token codes and atoms; tmC the gradient [E][M][N] bf16 (box
// 64 x 32 x 1), written with TMA stores (the other modes take a placeholder).
template <int MODE, int PAIR>
__global__ void __launch_bounds__(MX_THREADS, 1)
mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
               const __grid_constant__ CUtensorMap tmC, const MxParams p) {
  griddep_wait();   // see common.cuh: dependent launches
  using GE = MxGeo<PAIR, MODE>;
  constexpr int STAGES = GE::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  MxCtl* ctl =
      reinterpret_cast<MxCtl*>(smem + STAGES * GE::STAGE_BYTES + GE::STAGING_BYTES);
  const uint32_t staging_base = smem_u32(smem + STAGES * GE::STAGE_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  volatile int* abort_flag = &ctl->abort;
  const int rank = PAIR == 2 ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = rank == 0;
  const int unit = blockIdx.x / PAIR;
  const int num_units = gridDim.x / PAIR;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    mbar_init(smem_u32(&ctl->tfull), 1);
    mbar_init(smem_u32(&ctl->tempty), MX_EPI_WARPS * PAIR);
    mbar_init(smem_u32(&ctl->drain), 1);
    fence_mbar_init();
    ctl->abort = 0;
    ctl->bad = 0;
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmSA);
    tma_prefetch_desc(&tmSB);
    if (MODE == GEMM_WGRAD) tma_prefetch_desc(&tmC);
  }
  for (int g = threadIdx.x; g <= p.G; g += MX_THREADS) ctl->gstart[g] = p.offsets[g];
  __syncthreads();
  if (warp == 0) {
    // tiles per group: the segment's M tiles x the N tiles; WGRAD: the fixed weight-shaped
    // grid of every expert (an empty one still writes its zero gradient), and its K blocks
    auto tiles_of = [&](int a, int b) {
      if (MODE == GEMM_WGRAD) return p.wg_m_tiles * p.num_n_tiles;
      return b < a ? 0 : mx_ceil_div(b - a, GE::TILE_M) * p.num_n_tiles;
    };
    auto kblocks_of = [&](int a, int b) { return b > a ? mx_ceil_div(b - a, 128) : 0; };
    const int per = mx_ceil_div(p.G, 32);
    int local = 0, local_kb = 0, bad = 0;
    for (int i = 0; i < per; ++i) {
      const int g = lane * per + i;
      if (g < p.G) {
        const int a = ctl->gstart[g], b = ctl->gstart[g + 1];
        if (b < a || a < 0 || b > p.rows_cap) bad = 1;
        local += tiles_of(a, b);
        local_kb += kblocks_of(a, b);
      }
    }
    const int incl = warp_incl_scan(local);
    const int incl_kb = warp_incl_scan(local_kb);
    int run = incl - local, run_kb = incl_kb - local_kb;
    for (int i = 0; i < per; ++i) {
      const int g = lane * per + i;
      if (g < p.G) {
        ctl->tprefix[g] = run;
        ctl->kbpre[g] = run_kb;
        const int a = ctl->gstart[g], b = ctl->gstart[g + 1];
        run += tiles_of(a, b);
        run_kb += kblocks_of(a, b);
      }
    }
    if (lane == 31) {
      ctl->tprefix[p.G] = incl;
      ctl->kbpre[p.G] = incl_kb;
    }
    if (MODE == GEMM_WGRAD && incl_kb > p.kb_cap) bad = 1;
    if (ctl->gstart[0] != 0) bad = 1;
    bad = __any_sync(FULL_MASK, bad);
    if (lane == 0 && bad) {
      ctl->bad = 1;
      if (blockIdx.x == 0) flag_error(p.err, MOE_DEVERR_BAD_OFFSETS);
    }
  }
  if (warp == 1) {
    if (PAIR == 2) {
      tmem_alloc_pair(smem_u32(&ctl->tmem_base), MX_TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&ctl->tmem_base), MX_TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (PAIR == 2) cluster_sync_all();
  else __syncthreads();
  tc_fence_after();
  const int total = ctl->bad ? 0 : ctl->tprefix[p.G];
  const uint32_t tmem_base = ctl->tmem_base;

  auto map_tile = [&](int tile, int& g, int& mt, int& nt) {
    int lo = 0, hi = p.G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ctl->tprefix[mid] <= tile) lo = mid;
      else hi = mid;
    }
    g = lo;
    const int local = tile - ctl->tprefix[g];
    if (MODE == GEMM_WGRAD && p.wg_m_tiles > p.num_n_tiles) {
      // consecutive tiles share the M operand's (larger) tile and walk the N tiles, so the
      // larger operand streams through once and the smaller one is re-read from L2
      mt = local / p.num_n_tiles;
      nt = local - mt * p.num_n_tiles;
      return;
    }
    const int mtg = MODE == GEMM_WGRAD
                        ? p.wg_m_tiles
                        : mx_ceil_div(ctl->gstart[g + 1] - ctl->gstart[g], GE::TILE_M);
    nt = local / mtg;
    mt = local - nt * mtg;
  };

  if (warp == 0) {
    // -------------------------------------------------------------- producer (lane 0)
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tile = unit; tile < total && ok; tile += num_units) {
      int g, mt, nt;
      map_tile(tile, g, mt, nt);
      const int nkb = MODE == GEMM_WGRAD ? ctl->kbpre[g + 1] - ctl->kbpre[g] : p.num_kb;
      const int seg0 = ctl->gstart[g];
      const int lrow = mt * GE::TILE_M + 128 * rank;            // this CTA's first local row
      const int row0 = seg0 + lrow;
      const int a_atom_blk = (seg0 >> 7) + g + (lrow >> 7);     // its activation atom block
      const int b_atom = (g * p.n_blocks_mn + nt) * nkb;        // weight atom pair index
      for (int kb = 0; kb < nkb; ++kb) {
        if (!mx_warp_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, p.err, MX_WAIT_BUDGET)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t sa = smem_base + s * GE::STAGE_BYTES;
          const uint32_t sb = sa + GE::A_BYTES;
          const uint32_t full_local = smem_u32(&ctl->full[s]);
          const uint32_t full = PAIR == 2 ? mapa_shared(full_local, 0) : full_local;
          // the leader's single arrive announces both CTAs' bytes
          if (leader) mbar_arrive_expect_tx(full_local, PAIR * GE::LOAD_BYTES);
          auto load = [&](uint32_t dst, const CUtensorMap* m, int x, int y) {
            if (PAIR == 2) tma_load_2d_pair(dst, m, full, x, y);
            else tma_load_2d(dst, m, full, x, y);
          };
          const int k0 = kb * MX_BK;
          if (MODE == GEMM_WGRAD) {
            // K runs along the expert's rows: its K blocks sit at kbpre[g] .. in both
            // operands' along-token codes and scale atoms
            const int kbg = ctl->kbpre[g] + kb;
            const int arow = mt * GE::TILE_M + 128 * rank;
            load(sa, &tmA, kbg * MX_BK, arow);
            if (PAIR == 2) {
              load(sb, &tmB, kbg * MX_BK, nt * 256 + rank * 128);
            } else {
              load(sb, &tmB, kbg * MX_BK, nt * 256);
              load(sb + 128 * MX_BK, &tmB, kbg * MX_BK, nt * 256 + 128);
            }
            load(sa + GE::SFA_OFF, &tmSA, 0, ((arow >> 7) * p.kb_cap + kbg) * 2);
            load(sa + GE::SFB_OFF, &tmSB, 0, (nt * p.kb_cap + kbg) * 4);
          } else {
          load(sa, &tmA, k0, row0);
          if (MODE == GEMM_FC1_SWIGLU) {
            const int wrow = g * 2 * p.f + nt * 128;
            if (PAIR == 2) {
              load(sb, &tmB, k0, wrow + rank * p.f);                // CTA 0 gate, CTA 1 up
            } else {
              load(sb, &tmB, k0, wrow);
              load(sb + 128 * MX_BK, &tmB, k0, wrow + p.f);
            }
          } else {   // FC2 (W2), DGRAD2 (W2^T), DGRAD1 (W1^T): 256-row N tiles
            const int wrow = g * p.b_rows + nt * 256;
            if (PAIR == 2) {
              load(sb, &tmB, k0, wrow + rank * 128);
            } else {
              load(sb, &tmB, k0, wrow);
              load(sb + 128 * MX_BK, &tmB, k0, wrow + 128);
            }
          }
          load(sa + GE::SFA_OFF, &tmSA, 0, (a_atom_blk * nkb + kb) * 2);
          load(sa + GE::SFB_OFF, &tmSB, 0, (b_atom + kb) * 4);
          }
        }
        __syncwarp();
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    // every copy of this CTA is issued: the next kernel may be scheduled (it waits for
    // this one to complete before it touches memory)
    griddep_launch();
    for (int i = 0; i < STAGES && ok; ++i) {
      if (!mx_warp_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, p.err, MX_WAIT_BUDGET / 4))
        break;
      if (++s == STAGES) {
        s = 0;
        ph ^= 1u;
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer (leader)
    if (leader) {
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true, issued_any = false;
      const bool trace = g_clock_trace.on != 0;
      const long long trace_c0 = clock64();
      const unsigned long long trace_n0 = globaltimer_ns();
      for (int tile = unit; tile < total && ok; tile += num_units, ++it) {
        int nkb = p.num_kb;
        if (MODE == GEMM_WGRAD) {
          int g, mt, nt;
          map_tile(tile, g, mt, nt);
          nkb = ctl->kbpre[g + 1] - ctl->kbpre[g];
        }
        if (!mx_warp_wait(smem_u32(&ctl->tempty), (it & 1) ^ 1u, abort_flag, p.err,
                          MX_WAIT_BUDGET)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mx_warp_wait(smem_u32(&ctl->full[s]), ph, abort_flag, p.err, MX_WAIT_BUDGET)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_base + s * GE::STAGE_BYTES;
          const uint32_t sb = sa + GE::A_BYTES;
          // one scale slot per stage: a slot is rewritten only after the MMAs that read it
          // have completed (the producer refilled that stage after their commit)
          const uint32_t sf_col = tmem_base + MX_SF_COL0 + 12u * static_cast<uint32_t>(s);
          if (lane == 0) {
            // each CTA's own atoms into its own TMEM: A scales (its 128 rows) and the B
            // scales of all 256 columns
            tc_cp_atom<PAIR>(sf_col, sdesc_atom(sa + GE::SFA_OFF));
            tc_cp_atom<PAIR>(sf_col + 4, sdesc_atom(sa + GE::SFB_OFF));
            tc_cp_atom<PAIR>(sf_col + 8, sdesc_atom(sa + GE::SFB_OFF + 512));
#pragma unroll
            for (int kk = 0; kk < MX_BK / 32; ++kk)
              tc_mma_mx<PAIR>(tmem_base, sdesc_sw128(sa + kk * 32), sdesc_sw128(sb + kk * 32),
                              idesc_mx(GE::TILE_M, 256, kk), sf_col, sf_col + 4,
                              (kb | kk) != 0 ? 1u : 0u);
            if (PAIR == 2) tc_commit_pair_mc(smem_u32(&ctl->empty[s]), 0x3);
            else tc_commit(smem_u32(&ctl->empty[s]));
          }
          issued_any = true;
          __syncwarp();
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (lane == 0) {
          const uint32_t tf = smem_u32(&ctl->tfull);
          if (nkb > 0) {
            if (PAIR == 2) tc_commit_pair_mc(tf, 0x3);
            else tc_commit(tf);
          } else {   // an expert without rows (WGRAD): nothing to wait for
            mbar_arrive(tf);
            if (PAIR == 2) mbar_arrive_remote(mapa_shared(tf, 1));
          }
        }
        __syncwarp();
      }
      if (trace && ok && issued_any && lane == 0)
        clock_trace_add(&g_clock_trace, clock64() - trace_c0, globaltimer_ns() - trace_n0);
      if (!ok && issued_any && lane == 0) {
        if (PAIR == 2) tc_commit_pair(smem_u32(&ctl->drain));
        else tc_commit(smem_u32(&ctl->drain));
        long long t0 = clock64();
        while (!mbar_try_wait(smem_u32(&ctl->drain), 0) && clock64() - t0 < MX_WAIT_BUDGET / 4) {
        }
      }
      __syncwarp();
    }
  } else {
    // -------------------------------------------------------------- epilogue (8 warps)
    const int q = warp & 3;                  // the lane quarter this warp may access
    const int hh = (warp - 2) >> 2;          // which half of the columns
    const int r_in_tile = rank * 128 + q * 32 + lane;
    const uint32_t tempty_leader =
        PAIR == 2 ? mapa_shared(smem_u32(&ctl->tempty), 0) : smem_u32(&ctl->tempty);
    int store_buf = 0;                       // WGRAD: this warp's staging buffer in turn
    int it = 0;
    for (int tile = unit; tile < total; tile += num_units, ++it) {
      int g, mt, nt;
      map_tile(tile, g, mt, nt);
      const int seg0 = ctl->gstart[g];
      const int lrow = mt * GE::TILE_M + r_in_tile;
      // the output row: the segment's row, or WGRAD's row lrow of expert g's dW
      const long long prow = MODE == GEMM_WGRAD
                                 ? static_cast<long long>(g) * p.wg_M + lrow
                                 : static_cast<long long>(seg0) + lrow;
      const bool valid =
          MODE == GEMM_WGRAD ? lrow < p.wg_M : prow < ctl->gstart[g + 1];
      // WGRAD: an expert without rows has no accumulator to read, its gradient is zero
      const bool acc_zero = MODE == GEMM_WGRAD && ctl->kbpre[g + 1] == ctl->kbpre[g];
      // DGRAD2: the saved a, b of this row do not depend on the MMAs, so the first 32
      // columns are loaded before the accumulator is ready and each later chunk one chunk
      // ahead of its use (the epilogue was bound by these loads' latency)
      const int dg_n0 = nt * 256 + 128 * hh;
      const bool dg_ok = MODE == GEMM_DGRAD2_SWIGLU && !GE::XD2 && valid && dg_n0 < p.f;
      const uint4* dg_a = reinterpret_cast<const uint4*>(p.aux + prow * 2 * p.f + dg_n0);
      const uint4* dg_b = dg_a + p.f / 8;
      uint4 na[4], nb[4];
      if (dg_ok) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          na[v] = __ldg(dg_a + v);
          nb[v] = __ldg(dg_b + v);
        }
      }
      if (!mx_warp_wait(smem_u32(&ctl->tfull), it & 1, abort_flag, p.err, MX_WAIT_BUDGET)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      uint32_t acc[128];
      if (MODE == GEMM_FC1_SWIGLU) {
        // gate columns [64 hh, 64 hh + 64) and the matching up columns 128 + ...
        tmem_ld32(taddr + 64 * hh, acc);
        tmem_ld32(taddr + 64 * hh + 32, acc + 32);
        tmem_ld32(taddr + 128 + 64 * hh, acc + 64);
        tmem_ld32(taddr + 128 + 64 * hh + 32, acc + 96);
      } else if (!acc_zero) {
        tmem_ld32(taddr + 128 * hh, acc);
        tmem_ld32(taddr + 128 * hh + 32, acc + 32);
        tmem_ld32(taddr + 128 * hh + 64, acc + 64);
        tmem_ld32(taddr + 128 * hh + 96, acc + 96);
      } else {
#pragma unroll
        for (int i = 0; i < 128; ++i) acc[i] = 0u;
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {   // the accumulator is free (the leader counts both CTAs' warps)
        if (PAIR == 2) mbar_arrive_remote(tempty_leader);
        else mbar_arrive(tempty_leader);
      }
      if (MODE == GEMM_WGRAD) {
        // this warp's 32 rows of dW[g] and its 128 columns, as two 32 x 64 boxes written
        // through 128-byte-swizzled shared memory with TMA stores (rows past M and columns
        // past N: M and N are multiples of 128, so a box is wholly in or out)
        const int m_base = mt * GE::TILE_M + rank * 128 + q * 32;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int n0 = nt * 256 + 128 * hh + 64 * b;
          if (m_base >= p.wg_M || n0 >= p.wg_N) continue;
          const uint32_t buf_addr = staging_base +
                                    static_cast<uint32_t>(((warp - 2) * 2 + store_buf) * 4096);
          if (lane == 0) bulk_wait_group_read<1>();   // the store two boxes ago has read it
          __syncwarp();
          const uint32_t row_addr = buf_addr + lane * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(acc[64 * b + 8 * c + e]);
            const uint4 v = pack8(x);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                             row_addr + ((c ^ (lane & 7)) << 4)),
                         "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmC, buf_addr, n0, m_base, g);
            bulk_commit_group();
          }
          store_buf ^= 1;
        }
        continue;
      }
      if (MODE == GEMM_FC1_SWIGLU) {
        // gate columns [n0, n0 + 64) of f and their up columns; per 32-column block the
        // SwiGLU and the quantisation of h run on this lane's row, then a, b and h leave
        // through the warp's 2 KB block (64-byte rows, 16-byte pieces XOR-swizzled by row
        // pair: conflict-free both ways) as 16-byte row pieces of rows lane / 4 + 8 i,
        // four lanes per 64-byte row segment
        const int f = p.f;
        const int n0 = nt * 128 + 64 * hh;     // f is a multiple of 128: always in range
        const long long wrow0 = prow - lane;   // this warp's first row
        const uint32_t xb = staging_base + static_cast<uint32_t>((warp - 2) * 2048);
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          float h[32];
          uint4 pa[4], pb[4], phv[4];
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float a[8], b[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              a[e] = bf16r(__uint_as_float(acc[32 * blk + 8 * v + e]));
              b[e] = bf16r(__uint_as_float(acc[64 + 32 * blk + 8 * v + e]));
              h[8 * v + e] = bf16r(silu_mx(a[e]) * b[e]);
            }
            pa[v] = pack8(a);
            pb[v] = pack8(b);
            phv[v] = pack8(h + 8 * v);
          }
          if (valid) {
            // the SwiGLU step quantises its own (bf16) output for FC2
            uint32_t c[8];
            const uint32_t sc = mx_block(h, c);
            uint4* dq = reinterpret_cast<uint4*>(p.out_q + prow * f + n0 + 32 * blk);
            dq[0] = make_uint4(c[0], c[1], c[2], c[3]);
            dq[1] = make_uint4(c[4], c[5], c[6], c[7]);
            const int sub = n0 / 32 + blk;      // 32-element block of h's row
            p.out_sf[act_atom_byte(seg0, g, lrow, f / 128, sub >> 2, sub & 3)] =
                static_cast<uint8_t>(sc);
          }
#pragma unroll
          for (int o = 0; o < 3; ++o) {
            const uint4* src = o == 0 ? pa : (o == 1 ? pb : phv);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mx_st_shared_v4(xb + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4), src[k]);
            __syncwarp();
            // the four pieces are read out first, then stored
            uint4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = (lane >> 2) + 8 * i, k = lane & 3;
              v[i] = mx_ld_shared_v4(xb + r * 64 + ((k ^ ((r >> 1) & 3)) << 4));
            }
            __syncwarp();                       // the block is read before it is refilled
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const long long row = wrow0 + (lane >> 2) + 8 * i;
              if (row < ctl->gstart[g + 1]) {
                const int col = n0 + 32 * blk + 8 * (lane & 3);
                __nv_bfloat16* dst = o == 2 ? p.out1 + row * f + col
                                            : p.out0 + row * 2 * f + (o == 1 ? f : 0) + col;
                *reinterpret_cast<uint4*>(dst) = v[i];
              }
            }
          }
        }
        continue;
      }
      if (MODE == GEMM_FC2 || MODE == GEMM_DGRAD1) {
        // bf16 rows through the warp's 2 KB block as in FC1: 32 columns at a time, out as
        // 16-byte row pieces of rows lane / 4 + 8 i
        const int n0 = nt * 256 + 128 * hh;
        if (n0 < p.n_out) {                    // n_out is a multiple of 128: warp-uniform
          const long long wrow0 = prow - lane;
          const uint32_t xb = staging_base + static_cast<uint32_t>((warp - 2) * 2048);
#pragma unroll
          for (int blk = 0; blk < 4; ++blk) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              float x[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(acc[32 * blk + 8 * k + e]);
              mx_st_shared_v4(xb + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4), pack8(x));
            }
            __syncwarp();
            uint4 v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = (lane >> 2) + 8 * i, k = lane & 3;
              v[i] = mx_ld_shared_v4(xb + r * 64 + ((k ^ ((r >> 1) & 3)) << 4));
            }
            __syncwarp();                       // the block is read before it is refilled
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const long long row = wrow0 + (lane >> 2) + 8 * i;
              if (row < ctl->gstart[g + 1])
                *reinterpret_cast<uint4*>(p.out0 + row * p.n_out + n0 + 32 * blk +
                                          8 * (lane & 3)) = v[i];
            }
          }
        }
        continue;
      }
      if (GE::XD2) {
        // CTA pairs: dh goes through the warp's 4 KB block (128-byte fp32 rows, 16-byte
        // pieces XOR-swizzled by row) 32 columns at a time; each lane then takes the
        // 8-column piece lane % 4 of rows lane / 4 + 8 i, reads a, b and writes da, db as
        // 16-byte pieces, and the four lanes of a row share the 32-column MX block of dab:
        // its maximum by two shuffles, then 8 codes (8 bytes) per lane
        const int f = p.f;
        const int n0 = nt * 256 + 128 * hh;
        if (n0 < f) {                          // f is a multiple of 128: warp-uniform
          const long long wrow0 = prow - lane;
          const long long seg_end = ctl->gstart[g + 1];
          const uint32_t xb = staging_base + static_cast<uint32_t>((warp - 2) * 4096);
          const int kq = lane & 3;
          // the saved a, b of the lane's piece of row (blk, i), loaded one row ahead of
          // their use so that each load's latency overlaps the previous row's work (zero
          // past the segment's end)
          auto load_ab = [&](int blk, int i, uint4& xa, uint4& xv) {
            const long long row = wrow0 + (lane >> 2) + 8 * i;
            const long long base = row * 2 * f + n0 + 32 * blk + 8 * kq;
            xa = xv = make_uint4(0u, 0u, 0u, 0u);
            if (row < seg_end) {
              xa = __ldg(reinterpret_cast<const uint4*>(p.aux + base));
              xv = __ldg(reinterpret_cast<const uint4*>(p.aux + base + f));
            }
          };
#pragma unroll
          for (int blk = 0; blk < 4; ++blk) {
            uint4 na, nb;
            load_ab(blk, 0, na, nb);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mx_st_shared_v4(xb + lane * 128 + ((k ^ (lane & 7)) << 4),
                              make_uint4(acc[32 * blk + 4 * k], acc[32 * blk + 4 * k + 1],
                                         acc[32 * blk + 4 * k + 2], acc[32 * blk + 4 * k + 3]));
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 ca = na, cb = nb;
              if (i < 3) load_ab(blk, i + 1, na, nb);
              const int r = (lane >> 2) + 8 * i;
              const uint4 d0 = mx_ld_shared_v4(xb + r * 128 + (((2 * kq) ^ (r & 7)) << 4));
              const uint4 d1 = mx_ld_shared_v4(xb + r * 128 + (((2 * kq + 1) ^ (r & 7)) << 4));
              const float dh[8] = {__uint_as_float(d0.x), __uint_as_float(d0.y),
                                   __uint_as_float(d0.z), __uint_as_float(d0.w),
                                   __uint_as_float(d1.x), __uint_as_float(d1.y),
                                   __uint_as_float(d1.z), __uint_as_float(d1.w)};
              const long long row = wrow0 + r;
              const bool ok = row < seg_end;
              const int col = n0 + 32 * blk + 8 * kq;
              const long long base = row * 2 * f + col;
              float a[8], b[8], da[8], db[8];
              unpack8(ca, a);                   // bf16 zero bits: 0.0f past the end
              unpack8(cb, b);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float sg = sigmoid_fast(a[e]);
                const float silu = a[e] * sg;
                const float dsilu = sg * (1.0f + a[e] * (1.0f - sg));
                da[e] = dh[e] * b[e] * dsilu;
                db[e] = dh[e] * silu;
              }
              const uint4 pda = pack8(da), pdb = pack8(db);
              if (ok) {
                *reinterpret_cast<uint4*>(p.out0 + base) = pda;
                *reinterpret_cast<uint4*>(p.out0 + base + f) = pdb;
              }
              // dab quantised along 2f from its bf16 value, one 32-column block per four
              // lanes (a block never straddles the da | db boundary)
#pragma unroll
              for (int half = 0; half < 2; ++half) {
                const uint4 pv = half == 0 ? pda : pdb;
                const uint32_t w[4] = {pv.x, pv.y, pv.z, pv.w};
                float x[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  x[2 * e] = __uint_as_float(w[e] << 16);
                  x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
                }
                float amax = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
                amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, 2));
                const int X = mx_exponent(amax);
                const float inv = exp2_int(-X);
                const uint32_t c0 = e4m3x2(x[0] * inv, x[1] * inv) |
                                    (e4m3x2(x[2] * inv, x[3] * inv) << 16);
                const uint32_t c1 = e4m3x2(x[4] * inv, x[5] * inv) |
                                    (e4m3x2(x[6] * inv, x[7] * inv) << 16);
                if (ok) {
                  const long long qo = base + half * f;
                  *reinterpret_cast<uint2*>(p.out_q + qo) = make_uint2(c0, c1);
                  if (kq == 0) {
                    const int sub = (half * f + n0 + 32 * blk) / 32;
                    p.out_sf[act_atom_byte(seg0, g, static_cast<int>(row - seg0), 2 * f / 128,
                                           sub >> 2, sub & 3)] = static_cast<uint8_t>(X + 127);
                  }
                }
              }
            }
            __syncwarp();                       // the block is read before it is refilled
          }
        }
        continue;
      }
      if (!valid) continue;
      if (MODE == GEMM_DGRAD2_SWIGLU) {
        // dh of columns [n0, n0 + 128) of f; the SwiGLU backward from the saved a, b gives
        // da, db (bf16, for the bf16 weight gradient) and their MXFP8 form (for DGRAD1)
        const int f = p.f;
        const int n0 = dg_n0;
        if (dg_ok) {                           // f is a multiple of 128: all or nothing
          uint4* da_ = reinterpret_cast<uint4*>(p.out0 + prow * 2 * f + n0);
          uint4* db_ = reinterpret_cast<uint4*>(p.out0 + prow * 2 * f + f + n0);
#pragma unroll
          for (int c = 0; c < 4; ++c) {        // 32 columns = one MX block per chunk
            uint4 ca[4], cb[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              ca[v] = na[v];
              cb[v] = nb[v];
            }
            if (c + 1 < 4) {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                na[v] = __ldg(dg_a + 4 * (c + 1) + v);
                nb[v] = __ldg(dg_b + 4 * (c + 1) + v);
              }
            }
            uint4 pda[4], pdb[4];              // da, db as bf16 (what is stored)
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float a[8], b[8], da[8], db[8];
              unpack8(ca[v], a);
              unpack8(cb[v], b);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float dh = __uint_as_float(acc[32 * c + 8 * v + e]);
                const float sg = sigmoid_fast(a[e]);
                const float silu = a[e] * sg;
                const float dsilu = sg * (1.0f + a[e] * (1.0f - sg));
                da[e] = dh * b[e] * dsilu;
                db[e] = dh * silu;
              }
              pda[v] = pack8(da);
              pdb[v] = pack8(db);
              da_[4 * c + v] = pda[v];
              db_[4 * c + v] = pdb[v];
            }
            // dab quantised along 2f from its bf16 value (a block never straddles the
            // da | db boundary)
            uint32_t code[8];
            uint32_t sc = mx_block_bf16(pda, code);
            uint4* qa = reinterpret_cast<uint4*>(p.out_q + prow * 2 * f + n0 + 32 * c);
            qa[0] = make_uint4(code[0], code[1], code[2], code[3]);
            qa[1] = make_uint4(code[4], code[5], code[6], code[7]);
            int sub = (n0 + 32 * c) / 32;
            p.out_sf[act_atom_byte(seg0, g, lrow, 2 * f / 128, sub >> 2, sub & 3)] =
                static_cast<uint8_t>(sc);
            sc = mx_block_bf16(pdb, code);
            uint4* qb = reinterpret_cast<uint4*>(p.out_q + prow * 2 * f + f + n0 + 32 * c);
            qb[0] = make_uint4(code[0], code[1], code[2], code[3]);
            qb[1] = make_uint4(code[4], code[5], code[6], code[7]);
            sub = (f + n0 + 32 * c) / 32;
            p.out_sf[act_atom_byte(seg0, g, lrow, 2 * f / 128, sub >> 2, sub & 3)] =
                static_cast<uint8_t>(sc);
          }
        }
      }
    }
    if (MODE == GEMM_WGRAD && lane == 0) bulk_wait_group_all();   // stores done before exit
  }
  tc_fence_before();
  if (PAIR == 2) cluster_sync_all();
  else __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if (PAIR == 2) tmem_dealloc_pair(tmem_base, MX_TMEM_COLS);
    else tmem_dealloc(tmem_base, MX_TMEM_COLS);
  }
  griddep_launch();
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 mx_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D byte tensor map over a row-major [rows, cols] matrix: swizzled E4M3 tiles (box 128 x
// 128, 128-byte swizzle) or plain scale atoms (box 256 x box_rows, no swizzle).
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                 uint32_t box_cols, uint32_t box_rows, bool swizzle) {
  auto enc = mx_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 3-D bf16 tensor map over a weight gradient viewed as [groups][rows][cols], 128-byte
// swizzle, box 64 columns x 32 rows x 1 group (a store never crosses into the next
// group's rows)
bool make_map_dw(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                 uint64_t groups) {
  auto enc = mx_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, rows, groups};
  cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  cuuint32_t box[3] = {64, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

int grid_rows(int64_t rows) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (rows + (QTHREADS / 32) - 1) / (QTHREADS / 32);
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

template <int MODE, int PAIR>
cudaError_t launch_mx_mode(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa,
                           const CUtensorMap& tsb, const CUtensorMap& tc, const MxParams& kp,
                           cudaStream_t st) {
  auto kern = mx_gemm_kernel<MODE, PAIR>;
  constexpr size_t SMEM = mx_smem_bytes<PAIR, MODE>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  unsigned grid = static_cast<unsigned>(sms);
  if (PAIR == 2) {
    // persistent: as many CTA pairs as can be resident at once
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(MX_THREADS);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1));
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1)
      clusters = sms / 2;
    grid = static_cast<unsigned>(2 * clusters);
  }
  return launch_pdl(kern, dim3(grid), dim3(MX_THREADS), SMEM, st, PAIR, ta, tb, tsa, tsb, tc,
                    kp);
}

}  // namespace

MxWeightLayout mx_weight_layout(int E, int d, int f) {
  auto up = [](size_t b) { return (b + 255) & ~static_cast<size_t>(255); };
  MxWeightLayout L;
  const size_t Es = static_cast<size_t>(E), ds = static_cast<size_t>(d),
               fs = static_cast<size_t>(f);
  size_t o = 0;
  L.w1q = o;  o += up(Es * 2 * fs * ds);
  L.w1sf = o; o += up(Es * (fs / 128) * (ds / 128) * 1024);
  L.w2q = o;  o += up(Es * ds * fs);
  L.w2sf = o; o += up(Es * ((ds + 255) / 256) * (fs / 128) * 1024);
  // the backward's data-gradient operands: W2^T [E][f][d] along d, W1^T [E][d][2f] along 2f
  L.w2tq = o;  o += up(Es * fs * ds);
  L.w2tsf = o; o += up(Es * ((fs + 255) / 256) * (ds / 128) * 1024);
  L.w1tq = o;  o += up(Es * ds * 2 * fs);
  L.w1tsf = o; o += up(Es * ((ds + 255) / 256) * (2 * fs / 128) * 1024);
  L.total = o;
  return L;
}

cudaError_t launch_mx_quant_weights(const void* W1, const void* W2, int E, int d, int f,
                                    void* blob, cudaStream_t st) {
  const MxWeightLayout L = mx_weight_layout(E, d, f);
  uint8_t* b = static_cast<uint8_t*>(blob);
  // atom bytes of rows past an expert's last row are never written: give them scale 1
  cudaError_t e = cudaMemsetAsync(b + L.w1sf, 127, L.w2q - L.w1sf, st);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(b + L.w2sf, 127, L.w2tq - L.w2sf, st);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(b + L.w2tsf, 127, L.w1tq - L.w2tsf, st);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(b + L.w1tsf, 127, L.total - L.w1tsf, st);
  if (e != cudaSuccess) return e;
  const int64_t r1 = static_cast<int64_t>(E) * 2 * f, r2 = static_cast<int64_t>(E) * d;
  e = launch_pdl(mx_weight_quant_kernel, dim3(grid_rows(r1)), dim3(QTHREADS), 0, st, 1,
                 static_cast<const uint4*>(W1), r1, 2 * f, d, 0, f, f / 128,
                 reinterpret_cast<uint4*>(b + L.w1q), b + L.w1sf);
  if (e != cudaSuccess) return e;
  e = launch_pdl(mx_weight_quant_kernel, dim3(grid_rows(r2)), dim3(QTHREADS), 0, st, 1,
                 static_cast<const uint4*>(W2), r2, d, f, 1, f, (d + 255) / 256,
                 reinterpret_cast<uint4*>(b + L.w2q), b + L.w2sf);
  if (e != cudaSuccess) return e;
  // W2 [E][d][f] -> W2^T along d;  W1 [E][2f][d] -> W1^T along 2f
  e = launch_pdl(mx_weight_quant_t_kernel, dim3(f / TQ_COLS, d / TQ_ROWS, E), dim3(256), 0, st,
                 1, static_cast<const __nv_bfloat16*>(W2), d, f, b + L.w2tq, b + L.w2tsf);
  if (e != cudaSuccess) return e;
  return launch_pdl(mx_weight_quant_t_kernel, dim3(d / TQ_COLS, 2 * f / TQ_ROWS, E), dim3(256),
                    0, st, 1, static_cast<const __nv_bfloat16*>(W1), 2 * f, d, b + L.w1tq,
                    b + L.w1tsf);
}

cudaError_t launch_mx_permute_quant(const void* x, const int32_t* src_tok,
                                    const int32_t* offsets, int E, int64_t T, int64_t rows_cap,
                                    int d, void* xp_or_null, void* xq, uint8_t* x_sf, int* err,
                                    cudaStream_t st) {
  return launch_pdl(mx_permute_quant_kernel, dim3(grid_rows(rows_cap)), dim3(QTHREADS), 0, st, 1,
                    static_cast<const uint4*>(x), src_tok, offsets, E, T, rows_cap, d,
                    static_cast<uint4*>(xp_or_null), static_cast<uint4*>(xq), x_sf, err);
}

namespace {
// tc: WGRAD's output map; the other modes pass ta in its place (never used)
cudaError_t launch_mx_any(int mode, bool pair, const CUtensorMap& ta, const CUtensorMap& tb,
                          const CUtensorMap& tsa, const CUtensorMap& tsb, const MxParams& kp,
                          cudaStream_t st, const CUtensorMap* tc = nullptr) {
#define MOE_MX_CASE(M)                                                   \
  case M:                                                                \
    return pair ? launch_mx_mode<M, 2>(ta, tb, tsa, tsb, ta, kp, st)     \
                : launch_mx_mode<M, 1>(ta, tb, tsa, tsb, ta, kp, st);
  switch (mode) {
    MOE_MX_CASE(GEMM_FC1_SWIGLU)
    MOE_MX_CASE(GEMM_FC2)
    MOE_MX_CASE(GEMM_DGRAD2_SWIGLU)
    MOE_MX_CASE(GEMM_DGRAD1)
    case GEMM_WGRAD:
      if (!tc) return cudaErrorInvalidValue;
      return launch_mx_mode<GEMM_WGRAD, 2>(ta, tb, tsa, tsb, *tc, kp, st);
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_MX_CASE
}
}  // namespace

cudaError_t launch_mx_ffn(const MxFfnArgs& a, cudaStream_t st) {
  if (a.E < 1 || a.E > MX_MAX_G || a.d % 128 || a.f % 128) return cudaErrorInvalidValue;
  const MxWeightLayout L = mx_weight_layout(a.E, a.d, a.f);
  const uint8_t* wb = static_cast<const uint8_t*>(a.wq);
  const uint64_t rows = static_cast<uint64_t>(a.rows_cap);
  const uint64_t E = static_cast<uint64_t>(a.E), d = static_cast<uint64_t>(a.d),
                 f = static_cast<uint64_t>(a.f);
  // long segments on CTA pairs, as in the bf16 GEMMs
  const bool pair = static_cast<double>(a.rows_cap) / a.E >= 192.0;
  MxParams kp{};
  kp.G = a.E;
  kp.rows_cap = a.rows_cap;
  kp.d = a.d;
  kp.f = a.f;
  kp.offsets = a.offsets;
  kp.err = a.err;
  CUtensorMap ta, tb, tsa, tsb;
  auto launch = [&](int mode) {
    return launch_mx_any(mode, pair, ta, tb, tsa, tsb, kp, st);
  };
  // FC1: [a|b] = xq W1q^T (K = d), SwiGLU, h quantised
  const uint64_t KB1 = d / 128, NB1 = f / 128;
  kp.num_n_tiles = a.f / 128;
  kp.num_kb = a.d / MX_BK;
  kp.n_out = a.f;
  kp.n_blocks_mn = a.f / 128;
  kp.out0 = static_cast<__nv_bfloat16*>(a.ab);
  kp.out1 = static_cast<__nv_bfloat16*>(a.h);
  kp.out_q = a.hq;
  kp.out_sf = a.h_sf;
  if (!make_map_u8(&ta, a.xq, d, rows, 128, 128, true) ||
      !make_map_u8(&tb, wb + L.w1q, d, E * 2 * f, 128, 128, true) ||
      !make_map_u8(&tsa, a.x_sf, 256, mx_act_scale_bytes(a.rows_cap, a.E, a.d) / 256, 256, 2,
                   false) ||
      !make_map_u8(&tsb, wb + L.w1sf, 256, E * NB1 * KB1 * 4, 256, 4, false))
    return cudaErrorInvalidValue;
  cudaError_t e = launch(GEMM_FC1_SWIGLU);
  if (e != cudaSuccess) return e;
  // FC2: yp = hq W2q^T (K = f)
  const uint64_t KB2 = f / 128, NT2 = (d + 255) / 256;
  kp.num_n_tiles = static_cast<int>(NT2);
  kp.num_kb = a.f / MX_BK;
  kp.n_out = a.d;
  kp.n_blocks_mn = static_cast<int>(NT2);
  kp.b_rows = a.d;
  kp.out0 = static_cast<__nv_bfloat16*>(a.yp);
  kp.out1 = nullptr;
  kp.out_q = nullptr;
  kp.out_sf = nullptr;
  if (!make_map_u8(&ta, a.hq, f, rows, 128, 128, true) ||
      !make_map_u8(&tb, wb + L.w2q, f, E * d, 128, 128, true) ||
      !make_map_u8(&tsa, a.h_sf, 256, mx_act_scale_bytes(a.rows_cap, a.E, a.f) / 256, 256, 2,
                   false) ||
      !make_map_u8(&tsb, wb + L.w2sf, 256, E * NT2 * KB2 * 4, 256, 4, false))
    return cudaErrorInvalidValue;
  return launch(GEMM_FC2);
}

cudaError_t launch_mx_ffn_dgrad(const MxDgradArgs& a, cudaStream_t st) {
  if (a.E < 1 || a.E > MX_MAX_G || a.d % 128 || a.f % 128) return cudaErrorInvalidValue;
  const MxWeightLayout L = mx_weight_layout(a.E, a.d, a.f);
  const uint8_t* wb = static_cast<const uint8_t*>(a.wq);
  const uint64_t rows = static_cast<uint64_t>(a.rows_cap);
  const uint64_t E = static_cast<uint64_t>(a.E), d = static_cast<uint64_t>(a.d),
                 f = static_cast<uint64_t>(a.f);
  const bool pair = static_cast<double>(a.rows_cap) / a.E >= 192.0;
  MxParams kp{};
  kp.G = a.E;
  kp.rows_cap = a.rows_cap;
  kp.d = a.d;
  kp.f = a.f;
  kp.offsets = a.offsets;
  kp.err = a.err;
  CUtensorMap ta, tb, tsa, tsb;
  // DGRAD2: dh = dyq W2^T-quantised (K = d, N = f), SwiGLU backward, dab quantised
  const uint64_t NT_f = (f + 255) / 256, KB_d = d / 128;
  kp.num_n_tiles = static_cast<int>(NT_f);
  kp.num_kb = a.d / MX_BK;
  kp.n_out = a.f;
  kp.n_blocks_mn = static_cast<int>(NT_f);
  kp.b_rows = a.f;
  kp.aux = static_cast<const __nv_bfloat16*>(a.ab);
  kp.out0 = static_cast<__nv_bfloat16*>(a.dab);
  kp.out_q = a.dabq;
  kp.out_sf = a.dab_sf;
  if (!make_map_u8(&ta, a.dyq, d, rows, 128, 128, true) ||
      !make_map_u8(&tb, wb + L.w2tq, d, E * f, 128, 128, true) ||
      !make_map_u8(&tsa, a.dy_sf, 256, mx_act_scale_bytes(a.rows_cap, a.E, a.d) / 256, 256, 2,
                   false) ||
      !make_map_u8(&tsb, wb + L.w2tsf, 256, E * NT_f * KB_d * 4, 256, 4, false))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_mx_any(GEMM_DGRAD2_SWIGLU, pair, ta, tb, tsa, tsb, kp, st);
  if (e != cudaSuccess) return e;
  // DGRAD1: dxp = dabq W1^T-quantised (K = 2f, N = d)
  const uint64_t NT_d = (d + 255) / 256, KB_2f = 2 * f / 128;
  kp.num_n_tiles = static_cast<int>(NT_d);
  kp.num_kb = 2 * a.f / MX_BK;
  kp.n_out = a.d;
  kp.n_blocks_mn = static_cast<int>(NT_d);
  kp.b_rows = a.d;
  kp.aux = nullptr;
  kp.out0 = static_cast<__nv_bfloat16*>(a.dxp);
  kp.out_q = nullptr;
  kp.out_sf = nullptr;
  if (!make_map_u8(&ta, a.dabq, 2 * f, rows, 128, 128, true) ||
      !make_map_u8(&tb, wb + L.w1tq, 2 * f, E * d, 128, 128, true) ||
      !make_map_u8(&tsa, a.dab_sf, 256, mx_act_scale_bytes(a.rows_cap, a.E, 2 * a.f) / 256, 256,
                   2, false) ||
      !make_map_u8(&tsb, wb + L.w1tsf, 256, E * NT_d * KB_2f * 4, 256, 4, false))
    return cudaErrorInvalidValue;
  return launch_mx_any(GEMM_DGRAD1, pair, ta, tb, tsa, tsb, kp, st);
}

cudaError_t launch_mx_quant_tok(const void* X, const int32_t* offsets, int E, int64_t rows_cap,
                                int C, bool role_n, uint8_t* codes, uint8_t* scales, int* err,
                                cudaStream_t st) {
  if (E < 1 || E > MX_MAX_G || C % 128) return cudaErrorInvalidValue;
  const int64_t kb_cap = mx_tok_kb_cap(rows_cap, E);
  // each CTA walks up to 8 K blocks of its 64 columns (its expert prefix is built once)
  const unsigned gy = static_cast<unsigned>((kb_cap + 7) / 8);
  return launch_pdl(mx_quant_tok_kernel, dim3(C / KQ_COLS, gy), dim3(256), 0, st, 1,
                    static_cast<const __nv_bfloat16*>(X), offsets, E, rows_cap, C,
                    static_cast<int>(kb_cap), role_n ? 1 : 0, codes, scales, err);
}

// dW [E][M][N]: CTA pairs over 256 x 256 tiles of every expert's gradient, K = its rows
cudaError_t launch_mx_wgrad(const MxWgradArgs& a, cudaStream_t st) {
  if (a.E < 1 || a.E > MX_MAX_G || a.M % 128 || a.N % 128) return cudaErrorInvalidValue;
  const int64_t kb_cap = mx_tok_kb_cap(a.rows_cap, a.E);
  const uint64_t kcap = 128 * static_cast<uint64_t>(kb_cap);
  const uint64_t M = static_cast<uint64_t>(a.M), N = static_cast<uint64_t>(a.N);
  MxParams kp{};
  kp.G = a.E;
  kp.rows_cap = a.rows_cap;
  kp.offsets = a.offsets;
  kp.err = a.err;
  kp.wg_M = a.M;
  kp.wg_N = a.N;
  kp.wg_m_tiles = (a.M + 255) / 256;
  kp.kb_cap = static_cast<int>(kb_cap);
  kp.num_n_tiles = (a.N + 255) / 256;
  kp.n_out = a.N;
  kp.out0 = static_cast<__nv_bfloat16*>(a.dW);
  CUtensorMap ta, tb, tsa, tsb, tc;
  if (!make_map_u8(&ta, a.aq, kcap, M, 128, 128, true) ||
      !make_map_u8(&tb, a.bq, kcap, N, 128, 128, true) ||
      !make_map_u8(&tsa, a.a_sf, 256, (M / 128) * kb_cap * 2, 256, 2, false) ||
      !make_map_u8(&tsb, a.b_sf, 256, ((N + 255) / 256) * kb_cap * 4, 256, 4, false) ||
      !make_map_dw(&tc, a.dW, N, M, static_cast<uint64_t>(a.E)))
    return cudaErrorInvalidValue;
  return launch_mx_any(GEMM_WGRAD, true, ta, tb, tsa, tsb, kp, st, &tc);
}

cudaError_t mx_clock_trace_set(bool on) {
  if (on) {
    const ClockTrace t{1, 0, 0, 0};
    return cudaMemcpyToSymbol(g_clock_trace, &t, sizeof(t));
  }
  const int off = 0;
  return cudaMemcpyToSymbol(g_clock_trace, &off, sizeof(off), offsetof(ClockTrace, on));
}

cudaError_t mx_clock_trace_add(unsigned long long out[3]) {
  ClockTrace t;
  const cudaError_t e = cudaMemcpyFromSymbol(&t, g_clock_trace, sizeof(t));
  if (e != cudaSuccess) return e;
  out[0] += t.cycles;
  out[1] += t.ns;
  out[2] += t.loops;
  return cudaSuccess;
}

}  // namespace moe
