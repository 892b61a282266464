// grouped_gemm.cu -- the expert FFN's grouped GEMMs on the 5th-generation tensor cores.
//
// "MoE Training Optimization with Primus": Figure 7 (the grouped gate/up projection FC1,
// SwiGLU, the grouped down projection FC2), the MegaMoE section (the backward's FC2 and
// FC1 data-gradient GEMMs and the two weight-gradient GEMMs whose K is each expert's row
// count) and the JAX section
// (a single launch covers every expert's group of rows, each of its own length, in a
// layout sorted by expert).  X-MoE verdict page, key machinery: the groups are the padding-free
// buffer's expert segments -- no segment is padded; a tile that crosses a segment's
// end masks its stores, and in the weight-gradient GEMMs (K = the segment's rows) each
// segment gets its own copy of the operand maps whose row extent ends at the segment's
// end, so the rows of a K block past it load as zeros.
//
// One persistent kernel per mode, 192 threads per CTA, one CTA per SM:
//   warp 0      TMA producer: 128B-swizzled tiles of A and B into a shared-memory ring
//   warp 1      MMA issuer: one thread issues tcgen05.mma (bf16 in, fp32 accumulate in
//               TMEM); tcgen05.commit frees a stage / hands an accumulator to the epilogue
//   warps 2..5  epilogue: tcgen05.ld the accumulator (each warp its 32-lane quarter),
//               fused SwiGLU / SwiGLU-backward, bf16 rounding; each 32 x 32 block goes
//               through the warp's shared-memory block so that rows leave as 16-byte
//               pieces, four lanes per 64-byte row segment, not one row per lane
// Long segments run on CTA pairs (a cluster of 2 SMs): a 256 x 256 output tile, each CTA
// holding 128 rows of A and 128 rows of B in a 6-stage ring, the leader issuing
// M256 x N256 x K16 pair MMAs -- half the shared-memory traffic per SM of a one-CTA
// 128 x 256 tile.  Short segments (fine-grained experts) use one CTA with M128 x N256
// MMAs and a 4-stage ring.  Two 256-column fp32 accumulators in TMEM (512 columns) let
// the epilogue of one tile overlap the mainloop of the next.  The tile list is built on
// the device from the segment offsets (no host synchronisation): tiles are ordered
// expert-major, then N-tile, then M-tile, so CTAs running at the same time share one
// weight tile (read from HBM once, the rest from L2).  On CTA pairs a segment's last,
// partly filled M tile of at most TAIL_ROWS_MAX rows runs swapped (the weight rows as the
// MMA's M, the segment's rows as its N; see tail_tokens()), so its tensor time follows the
// rows present.  Every wait on an mbarrier is bounded; a wait that gives up sets
// MOE_DEVERR_TIMEOUT in the error word and the CTA drains and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstddef>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__device__ ClockTrace g_clock_trace;   // see ClockTrace (common.cuh)

// One tile is TILE_M x 256 of the output.  PAIR = 1: one CTA, M128 x N256 MMAs, A 128 rows
// and B 256 rows per CTA.  PAIR = 2: a CTA pair (cluster of 2) shares a 256 x 256 tile:
// each CTA holds 128 rows of A and 128 rows (N) of B, the leader issues M256 x N256 x K16
// pair MMAs that read both CTAs' shared memory, and each CTA's TMEM receives its own 128
// output rows.  The pair halves the shared-memory bytes each SM writes and reads per MMA.
template <int MODE, int PAIR>
struct Geo {
  static constexpr int BK = 64;
  static constexpr int TILE_M = 128 * PAIR;
  static constexpr int BN = 256;
  static constexpr int BN_CTA = BN / PAIR;
  static constexpr int A_BYTES = 128 * BK * 2;
  static constexpr int B_BYTES = BN_CTA * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // the weight-gradient epilogue stores through shared memory with TMA: each epilogue
  // warp double-buffers a 32-row x 64-column bf16 box (4 KB)
  static constexpr bool TMA_STORE = MODE == GEMM_WGRAD;
  // swap-AB tail tiles (CTA pairs, fixed-K modes): see tail_tokens()
  static constexpr bool TAIL = PAIR == 2 && MODE != GEMM_WGRAD;
  // the fixed-K epilogues transpose through shared memory: one block per epilogue warp
  // (a tail tile's 32 x 32 fp32 with rows padded to 144 bytes; an ordinary tile's 32
  // rows of 128 bytes, 16-byte pieces XOR-swizzled by row)
  static constexpr int XCH_BYTES = MODE != GEMM_WGRAD ? 4 * 32 * 144 : 0;
  static constexpr int STAGING_BYTES = (TMA_STORE ? 4 * 2 * 4096 : 0) + XCH_BYTES;
  static constexpr int STAGES = PAIR == 2 ? (TMA_STORE ? 5 : 6) : 4;
  // The fixed-K modes look each CTA's tiles up once, at the start, into a table in shared
  // memory (TileEnt); tiles past its end are looked up when they come.  The lookup (a
  // search over the groups' tile prefix, a division, a few loads) costs the issuing warps
  // 0.5-1.6k cycles per tile, and the tensor pipe, which runs barely ahead of the MMA warp,
  // waits for every cycle the MMA warp spends between two MMAs.
  static constexpr int TILE_TABLE = MODE == GEMM_WGRAD ? 0 : 1024;
};

struct TileEnt {
  uint16_t g, mt, nt, ntok;
};

constexpr int BK = 64;
constexpr int BN = 256;
constexpr int CHUNK_BYTES = 64 * BK * 2;     // one 64-element x 64-row MN-major box: 8 KB
constexpr int NUM_THREADS = 192;   // producer, MMA, 4 epilogue warps
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_G = 256;
constexpr int MAX_STAGES = 6;
constexpr long long WAIT_BUDGET = 4000000000LL;   // clock cycles (about 2 s)
// a segment's last M tile with at most this many rows runs as a swap-AB tail tile
constexpr int TAIL_ROWS_MAX = 160;

struct Ctl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t xfull[2][2];    // FC1 tail tiles: [warp pair][0] (one block per warp)
  uint64_t xempty[2][2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int bad;
  int pad;
  int gstart[MAX_G + 2];
  int tprefix[MAX_G + 2];
};

template <int MODE, int PAIR>
constexpr size_t smem_bytes() {
  using GE = Geo<MODE, PAIR>;
  return 1024 + GE::STAGES * GE::STAGE_BYTES + GE::STAGING_BYTES + sizeof(Ctl) +
         GE::TILE_TABLE * sizeof(TileEnt);
}

struct KParams {
  int G;
  long long uniform_rows;
  long long rows_cap;
  int d, f;
  int wg_M, wg_N;
  int num_n_tiles;
  int wg_m_tiles;
  int num_kb;          // K blocks of the fixed-K modes
  int n_out;           // valid output columns of the accumulator's N axis
  int wg_n_fast;       // WGRAD: walk N tiles fastest (when there are fewer N than M tiles)
  const int32_t* offsets;
  __nv_bfloat16* out0;
  __nv_bfloat16* out1;
  const __nv_bfloat16* aux;
  int* err;
  // WGRAD: per-segment copies of the two operand maps (row extent = segment end), or null
  const CUtensorMap* gmaps;
  // gathered operand rows (FC1's A, the FC2 data-gradient's A, WGRAD's B): source row of
  // each row-buffer row
  const int32_t* gidx;
  int gather_rows;
  // the FC2 data-gradient on gathered dy rows: dh of row p is scaled by gw[gslot[p]] (the
  // gate weight of the row's slot) in the epilogue; null otherwise
  const float* gw;
  const int32_t* gslot;
  long long n_slots;
  // a segment's last M tile with at most this many rows runs swapped (0: never)
  int tail_rows_max;
};

template <int MODE>
struct ModeTraits {
  static constexpr bool A_MN = (MODE == GEMM_WGRAD);
  static constexpr bool B_MN = (MODE == GEMM_DGRAD2_SWIGLU || MODE == GEMM_DGRAD1 ||
                                MODE == GEMM_WGRAD);
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Tile -> (group, m-tile, n-tile).
template <int MODE, int PAIR>
__device__ __forceinline__ void map_tile(const Ctl* ctl, const KParams& p, int tile, int& g,
                                         int& mt, int& nt) {
  if (MODE == GEMM_WGRAD) {
    // consecutive tiles share the operand chunk of the dimension with more tiles, so that
    // operand streams through once while the smaller one is re-read from L2
    const int per = p.wg_m_tiles * p.num_n_tiles;
    g = tile / per;
    const int r = tile - g * per;
    if (p.wg_n_fast) {
      mt = r / p.num_n_tiles;
      nt = r - mt * p.num_n_tiles;
    } else {
      nt = r / p.wg_m_tiles;
      mt = r - nt * p.wg_m_tiles;
    }
  } else {
    int lo = 0, hi = p.G;   // tprefix[0] = 0 <= tile < tprefix[G]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ctl->tprefix[mid] <= tile) lo = mid;
      else hi = mid;
    }
    g = lo;
    const int local = tile - ctl->tprefix[g];
    const int mtg = ceil_div(ctl->gstart[g + 1] - ctl->gstart[g], Geo<MODE, PAIR>::TILE_M);
    nt = local / mtg;
    mt = local - nt * mtg;
  }
}

__device__ __forceinline__ float silu_f(float a) { return a * sigmoid_fast(a); }

// Every lane of the warp waits; the result is made warp-uniform so that a timeout seen by
// one lane sends the whole warp down the same path (later warp-collective ops stay legal).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int* err, long long budget) {
  return __all_sync(FULL_MASK, mbar_wait_bounded(bar, parity, abort, err, budget));
}

// Source row of row-buffer row r for a gathered operand; an out-of-range entry is flagged
// and replaced by row 0, so no copy ever leaves the source matrix.
__device__ __forceinline__ int gather_row(const KParams& p, int r) {
  int v = __ldg(p.gidx + r);
  if (static_cast<unsigned>(v) >= static_cast<unsigned>(p.gather_rows)) {
    flag_error(p.err, MOE_DEVERR_BAD_INDEX);
    v = 0;
  }
  return v;
}

// Gate weight of row-buffer row r for the FC2 data-gradient on gathered dy rows (1 when
// the rows are the already-scaled dyp); an out-of-range slot is flagged and weighs 0.
__device__ __forceinline__ float row_gate_weight(const KParams& p, long long r) {
  if (!p.gw) return 1.0f;
  const int s = __ldg(p.gslot + r);
  if (s < 0 || s >= p.n_slots) {
    flag_error(p.err, MOE_DEVERR_BAD_INDEX);
    return 0.0f;
  }
  return __ldg(p.gw + s);
}

// Issue this CTA's share of the copies of one K block into stage (sa, sb).  With GATHER,
// the gathered operand (FC1's A, WGRAD's B) is left to the caller's gather4 copies.
template <int MODE, int PAIR, bool GATHER>
__device__ __forceinline__ void issue_loads(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                            const KParams& p, uint32_t sa, uint32_t sb,
                                            uint32_t bar, bool pair_form, int rank, int g,
                                            int mt, int nt, int seg0, int kb) {
  using GE = Geo<MODE, PAIR>;
  auto load = [&](uint32_t dst, const CUtensorMap* m, int x, int y) {
    if (pair_form) tma_load_2d_pair(dst, m, bar, x, y);
    else tma_load_2d(dst, m, bar, x, y);
  };
  const int k0 = kb * BK;
  const int arow = seg0 + mt * GE::TILE_M + 128 * rank;
  if (MODE == GEMM_FC1_SWIGLU) {
    if (!GATHER) load(sa, tmA, k0, arow);
    const int wrow = g * 2 * p.f + nt * (BN / 2);
    if (PAIR == 1) {
      load(sb, tmB, k0, wrow);                        // gate rows -> accumulator cols 0..127
      load(sb + GE::B_BYTES / 2, tmB, k0, wrow + p.f);  // up rows -> cols 128..255
    } else {
      load(sb, tmB, k0, wrow + rank * p.f);           // CTA 0: gate half, CTA 1: up half
    }
  } else if (MODE == GEMM_FC2) {
    load(sa, tmA, k0, arow);
    load(sb, tmB, k0, g * p.d + nt * BN + rank * GE::BN_CTA);
  } else if (MODE == GEMM_DGRAD2_SWIGLU || MODE == GEMM_DGRAD1) {
    if (!GATHER) load(sa, tmA, k0, arow);
    const int krow = (MODE == GEMM_DGRAD2_SWIGLU ? g * p.d : g * 2 * p.f) + k0;
#pragma unroll
    for (int j = 0; j < GE::BN_CTA / 64; ++j)
      load(sb + j * CHUNK_BYTES, tmB, nt * BN + rank * GE::BN_CTA + 64 * j, krow);
  } else {   // WGRAD: K rows run along the expert's segment
#pragma unroll
    for (int j = 0; j < 2; ++j)
      load(sa + j * CHUNK_BYTES, tmA, mt * GE::TILE_M + rank * 128 + 64 * j, seg0 + k0);
    if (!GATHER) {
#pragma unroll
      for (int j = 0; j < GE::BN_CTA / 64; ++j)
        load(sb + j * CHUNK_BYTES, tmB, nt * BN + rank * GE::BN_CTA + 64 * j, seg0 + k0);
    }
  }
}

// The tail tiles' segment-row maps: entry i has a box of 16 (i + 1) rows, the rows one
// CTA of a pair holds for N = 32 (i + 1), so each K block takes a single copy.
struct TailMaps {
  CUtensorMap m[8];
};

// Swap-AB tail tiles.  A segment's rows fill its M tiles of 256 except the last, which
// holds rem = rows - 256 (mtg - 1) rows.  When rem <= tail_rows_max that tile computes the
// transposed product, D^T = W_tile . X^T: the tile's 256 weight rows (output columns) are
// the MMA's M (128 per CTA) and its rows the MMA's N, rounded up to a multiple of 32, so
// the tensor-core time follows the rows present instead of a full 256.  Returns that N, or
// 0 for an ordinary tile.
template <int MODE, int PAIR>
__device__ __forceinline__ int tail_tokens(const Ctl* ctl, const KParams& p, int g, int mt) {
  if (!Geo<MODE, PAIR>::TAIL) return 0;
  const int rows = ctl->gstart[g + 1] - ctl->gstart[g];
  const int rem = rows - mt * 256;
  if (rem > 256 || rem <= 0 || rem > p.tail_rows_max) return 0;   // not the last tile
  return (rem + 31) & ~31;
}

// The copies of one K block of a tail tile: the weight rows into sb (as an ordinary tile's
// B operand, except FC1: 64 gate rows then the matching 64 up rows per CTA, through tmW)
// and this CTA's ntok / 2 rows of the segment into sa in one copy (tmT->m[ntok / 32 - 1]).
// With GATHER the segment rows are left to the caller's gather4 copies.
template <int MODE, bool GATHER>
__device__ __forceinline__ void issue_loads_tail(const CUtensorMap* tmB, const TailMaps* tmT,
                                                 const CUtensorMap* tmW, const KParams& p,
                                                 uint32_t sa, uint32_t sb, uint32_t bar,
                                                 int rank, int g, int mt, int nt, int seg0,
                                                 int kb, int ntok) {
  const int k0 = kb * BK;
  if (MODE == GEMM_FC1_SWIGLU) {
    const int wrow = g * 2 * p.f + nt * (BN / 2) + 64 * rank;
    tma_load_2d_pair(sb, tmW, bar, k0, wrow);                 // gate -> TMEM lanes 0..63
    tma_load_2d_pair(sb + 64 * BK * 2, tmW, bar, k0, wrow + p.f);   // up -> lanes 64..127
  } else if (MODE == GEMM_FC2) {
    tma_load_2d_pair(sb, tmB, bar, k0, g * p.d + nt * BN + rank * (BN / 2));
  } else {   // DGRAD2, DGRAD1: the weight operand is MN-major
    const int krow = (MODE == GEMM_DGRAD2_SWIGLU ? g * p.d : g * 2 * p.f) + k0;
#pragma unroll
    for (int j = 0; j < 2; ++j)
      tma_load_2d_pair(sb + j * CHUNK_BYTES, tmB, bar, nt * BN + rank * (BN / 2) + 64 * j, krow);
  }
  if (GATHER) return;
  const int trow = seg0 + mt * 256 + rank * (ntok / 2);
  tma_load_2d_pair(sa, &tmT->m[ntok / 32 - 1], bar, k0, trow);
}

__device__ __forceinline__ float bf16_round(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// Epilogue of a tail tile.  TMEM lane l of this CTA holds the tile's weight row (output
// column) rank * 128 + l, and TMEM column j the tile's row row0 + j, for j < ntok.  Each
// warp takes its 32 lanes x 32 rows per step, transposes them through its own block of
// shared memory (fp32, rows padded to 144 bytes so both the column writes and the 32-byte
// row reads are free of bank conflicts) and stores 16-byte pieces of 8 columns of a row.
// FC1: lanes 0..63 hold gate columns, 64..127 the matching up columns; the up warp
// (quarter 2 + i) only fills its block, and the gate warp (quarter i) reads both blocks and
// stores a, b and h.  Returns false if a wait gave up.
constexpr int XPOSE_PITCH = 144;                 // bytes per row of a transpose block
constexpr int XPOSE_BYTES = 32 * XPOSE_PITCH;    // one warp's block

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void ld_shared_f32x4(uint32_t addr, float* v) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ld_shared_f32x8(uint32_t addr, float* v) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(addr) : "memory");
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7]) : "r"(addr + 16) : "memory");
}

template <int MODE>
__device__ __forceinline__ bool tail_epilogue(const KParams& p, Ctl* ctl, uint32_t taddr,
                                              uint32_t xch_base, int q, int lane, int rank,
                                              int nt, long long row0, int nrows, int ntok,
                                              int& xc, volatile int* abort_flag) {
  const uint32_t blk = xch_base + static_cast<uint32_t>(q * XPOSE_BYTES);
  const int pi = q & 1;                      // FC1: warp pair (gate quarter pi, up pi + 2)
  const bool up = MODE == GEMM_FC1_SWIGLU && q >= 2;
  // the warp's first output column
  const int n0 = MODE == GEMM_FC1_SWIGLU ? nt * (BN / 2) + rank * 64 + pi * 32
                                         : nt * BN + rank * 128 + q * 32;
  const int n_lim = (MODE == GEMM_FC2 || MODE == GEMM_DGRAD1) ? p.n_out : p.f;
  const bool cols_ok = n0 < n_lim;           // d, f are multiples of 64: all 32 or none
#pragma unroll 1
  for (int c = 0; c < ntok / 32; ++c, ++xc) {
    // piece i of this lane: row j = lane / 4 + 8 i, columns n0 + 8 (lane % 4) + 0..7
    const int cc = 8 * (lane & 3);
    uint4 xa[4], xb[4];                      // FC2 data-gradient: the saved a, b
    if (MODE == GEMM_DGRAD2_SWIGLU) {
      // issued first, so that the four rows' loads are in flight together
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = lane / 4 + 8 * i;
        const long long base = (row0 + c * 32 + j) * 2 * p.f + n0 + cc;
        xa[i] = xb[i] = make_uint4(0u, 0u, 0u, 0u);
        if (cols_ok && c * 32 + j < nrows) {
          xa[i] = __ldg(reinterpret_cast<const uint4*>(p.aux + base));
          xb[i] = __ldg(reinterpret_cast<const uint4*>(p.aux + base + p.f));
        }
      }
    }
    uint32_t ra[32];
    tmem_ld32(taddr + c * 32, ra);
    tmem_ld_wait();
    const uint32_t xph = static_cast<uint32_t>(xc) & 1u;
    if (up && !warp_wait(smem_u32(&ctl->xempty[pi][0]), xph ^ 1u, abort_flag, p.err,
                         WAIT_BUDGET))
      return false;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(blk + j * XPOSE_PITCH + lane * 4),
                   "f"(__uint_as_float(ra[j]))
                   : "memory");
    __syncwarp();
    if (up) {
      mbar_arrive(smem_u32(&ctl->xfull[pi][0]));
      continue;
    }
    if (MODE == GEMM_FC1_SWIGLU &&
        !warp_wait(smem_u32(&ctl->xfull[pi][0]), xph, abort_flag, p.err, WAIT_BUDGET))
      return false;
    // the four pieces (and FC1's up pieces) are read out first and the blocks released,
    // then the four rows are computed and stored together
    float vs[4][8], us[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = lane / 4 + 8 * i;
      ld_shared_f32x8(blk + j * XPOSE_PITCH + cc * 4, vs[i]);
      if (MODE == GEMM_FC1_SWIGLU)   // the matching up values sit in the up warp's block
        ld_shared_f32x8(blk + 2 * XPOSE_BYTES + j * XPOSE_PITCH + cc * 4, us[i]);
    }
    __syncwarp();                            // the blocks are read before the next step
    if (MODE == GEMM_FC1_SWIGLU) mbar_arrive(smem_u32(&ctl->xempty[pi][0]));
    // the four rows are computed without branches (rows past the tile's end on zeros or
    // unused accumulator columns, not stored), then stored
    uint4 o0[4], o1[4], o2[4];
    if (MODE == GEMM_FC2 || MODE == GEMM_DGRAD1) {
#pragma unroll
      for (int i = 0; i < 4; ++i) o0[i] = pack8(vs[i]);
    } else if (MODE == GEMM_DGRAD2_SWIGLU) {
      float wr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = lane / 4 + 8 * i;
        wr[i] = cols_ok && c * 32 + j < nrows ? row_gate_weight(p, row0 + c * 32 + j) : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a[8], b[8], da[8], db[8];
        unpack8(xa[i], a);
        unpack8(xb[i], b);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float dh = vs[i][e] * wr[i];
          const float sg = sigmoid_fast(a[e]);
          const float silu = a[e] * sg;
          const float dsilu = sg * (1.0f + a[e] * (1.0f - sg));
          da[e] = dh * b[e] * dsilu;
          db[e] = dh * silu;
        }
        o0[i] = pack8(da);
        o1[i] = pack8(db);
      }
    } else {   // FC1, gate warp
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float a[8], b[8], h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          // round a, b to bf16 first: h is computed from the stored values
          a[e] = bf16_round(vs[i][e]);
          b[e] = bf16_round(us[i][e]);
          h[e] = silu_f(a[e]) * b[e];
        }
        o0[i] = pack8(a);
        o1[i] = pack8(b);
        o2[i] = pack8(h);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int j = lane / 4 + 8 * i;
      if (!(cols_ok && c * 32 + j < nrows)) continue;
      const long long row = row0 + c * 32 + j;
      if (MODE == GEMM_FC2 || MODE == GEMM_DGRAD1) {
        *reinterpret_cast<uint4*>(p.out0 + row * p.n_out + n0 + cc) = o0[i];
      } else {
        const long long base = row * 2 * p.f + n0 + cc;
        *reinterpret_cast<uint4*>(p.out0 + base) = o0[i];
        *reinterpret_cast<uint4*>(p.out0 + base + p.f) = o1[i];
        if (MODE == GEMM_FC1_SWIGLU)
          *reinterpret_cast<uint4*>(p.out1 + row * p.f + n0 + cc) = o2[i];
      }
    }
  }
  // FC1: the up warp's block is also its staging block for ordinary tiles, so it leaves
  // only once the gate warp has read the last step out of it
  if (up && ntok > 0 &&
      !warp_wait(smem_u32(&ctl->xempty[pi][0]), (static_cast<uint32_t>(xc) & 1u) ^ 1u,
                 abort_flag, p.err, WAIT_BUDGET))
    return false;
  return true;
}

template <int MODE, int PAIR, bool GATHER>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ TailMaps tmT,
                    const __grid_constant__ CUtensorMap tmW, const KParams p) {
  griddep_wait();   // see common.cuh: dependent launches
  using GE = Geo<MODE, PAIR>;
  constexpr int STAGES = GE::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + STAGES * GE::STAGE_BYTES + GE::STAGING_BYTES);
  TileEnt* table = reinterpret_cast<TileEnt*>(reinterpret_cast<uint8_t*>(ctl) + sizeof(Ctl));
  const uint32_t staging_base = smem_u32(smem + STAGES * GE::STAGE_BYTES);
  // the epilogue warps' transpose blocks (one per warp, used by every fixed-K tile) sit
  // after the TMA-store staging, which only the weight-gradient mode uses
  const uint32_t xch_base = staging_base + (GE::STAGING_BYTES - GE::XCH_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  volatile int* abort_flag = &ctl->abort;
  const int rank = PAIR == 2 ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = rank == 0;
  const int unit = blockIdx.x / PAIR;
  const int num_units = gridDim.x / PAIR;

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);   // the leader's arrive (+ both CTAs' bytes)
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl->tfull[b]), 1);
      mbar_init(smem_u32(&ctl->tempty[b]), 4 * PAIR);
      for (int w = 0; w < 2; ++w) {
        mbar_init(smem_u32(&ctl->xfull[w][b]), 32);   // every lane of the writing warp
        mbar_init(smem_u32(&ctl->xempty[w][b]), 32);  // every lane of the reading warp
      }
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    fence_mbar_init();
    ctl->abort = 0;
    ctl->bad = 0;
  }
  if (threadIdx.x == 32) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (GE::TMA_STORE) tma_prefetch_desc(&tmC);
    if (GE::TAIL && p.tail_rows_max > 0) {
      if (!GATHER)
        for (int i = 0; i < 8; ++i) tma_prefetch_desc(&tmT.m[i]);
      if (MODE == GEMM_FC1_SWIGLU) tma_prefetch_desc(&tmW);
    }
  }
  if (p.uniform_rows > 0) {
    if (threadIdx.x == 0) {
      ctl->gstart[0] = 0;
      ctl->gstart[1] = static_cast<int>(p.uniform_rows);
    }
  } else {
    for (int g = threadIdx.x; g <= p.G; g += NUM_THREADS) ctl->gstart[g] = p.offsets[g];
  }
  __syncthreads();
  if (warp == 0) {
    // validate the offsets and build the tile prefix (warp scan over the groups)
    const int per = ceil_div(p.G, 32);
    int local = 0, bad = 0;
    for (int i = 0; i < per; ++i) {
      const int g = lane * per + i;
      if (g < p.G) {
        const int a = ctl->gstart[g], b = ctl->gstart[g + 1];
        if (b < a || a < 0 || b > p.rows_cap) bad = 1;
        int tiles = (MODE == GEMM_WGRAD) ? p.wg_m_tiles * p.num_n_tiles
                                         : ceil_div(b - a, GE::TILE_M) * p.num_n_tiles;
        if (b < a) tiles = 0;
        local += tiles;
      }
    }
    const int incl = warp_incl_scan(local);
    int run = incl - local;
    for (int i = 0; i < per; ++i) {
      const int g = lane * per + i;
      if (g < p.G) {
        ctl->tprefix[g] = run;
        const int a = ctl->gstart[g], b = ctl->gstart[g + 1];
        int tiles = (MODE == GEMM_WGRAD) ? p.wg_m_tiles * p.num_n_tiles
                                         : ceil_div(b - a, GE::TILE_M) * p.num_n_tiles;
        if (b < a) tiles = 0;
        run += tiles;
      }
    }
    if (lane == 31) ctl->tprefix[p.G] = incl;
    if (ctl->gstart[0] != 0) bad = 1;
    bad = __any_sync(FULL_MASK, bad);
    if (lane == 0 && bad) {
      ctl->bad = 1;
      if (blockIdx.x == 0) flag_error(p.err, MOE_DEVERR_BAD_OFFSETS);
    }
  }
  if (warp == 1) {
    if (PAIR == 2) {
      tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (PAIR == 2) cluster_sync_all();   // barriers of both CTAs initialised before any remote use
  else __syncthreads();
  tc_fence_after();

  const int total = ctl->bad ? 0 : ctl->tprefix[p.G];
  const uint32_t tmem_base = ctl->tmem_base;
  // this CTA's tiles are unit, unit + num_units, ...: their lookups, shared by all roles
  // (entries hold 16-bit tile coordinates: segments of up to 2^24 rows, 2^16 N tiles)
  const bool fits16 = p.rows_cap <= 65535LL * GE::TILE_M && p.num_n_tiles <= 65535;
  const int n_mine = total > unit ? ceil_div(total - unit, num_units) : 0;
  const int n_table = !fits16 ? 0 : (n_mine < GE::TILE_TABLE ? n_mine : GE::TILE_TABLE);
  for (int i = threadIdx.x; i < n_table; i += NUM_THREADS) {
    int g, mt, nt;
    map_tile<MODE, PAIR>(ctl, p, unit + i * num_units, g, mt, nt);
    table[i] = TileEnt{static_cast<uint16_t>(g), static_cast<uint16_t>(mt),
                       static_cast<uint16_t>(nt),
                       static_cast<uint16_t>(tail_tokens<MODE, PAIR>(ctl, p, g, mt))};
  }
  __syncthreads();
  // the i-th tile of this CTA: from the table, or looked up now past its end
  auto tile_of = [&](int i, int tile, int& g, int& mt, int& nt, int& ntok) {
    if (i < n_table) {
      const TileEnt e = table[i];
      g = e.g;
      mt = e.mt;
      nt = e.nt;
      ntok = e.ntok;
    } else {
      map_tile<MODE, PAIR>(ctl, p, tile, g, mt, nt);
      ntok = tail_tokens<MODE, PAIR>(ctl, p, g, mt);
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (whole warp)
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    const CUtensorMap* mA = &tmA;
    const CUtensorMap* mB = &tmB;
    int map_g = -1;
    int pit = 0;
    for (int tile = unit; tile < total && ok; tile += num_units, ++pit) {
      int g, mt, nt, ntok;
      tile_of(pit, tile, g, mt, nt, ntok);
      const int seg0 = ctl->gstart[g];
      const int seg_rows = ctl->gstart[g + 1] - seg0;
      const int nkb = (MODE == GEMM_WGRAD) ? ceil_div(seg_rows, BK) : p.num_kb;
      // a tail tile copies the weight rows and ntok / 2 segment rows per CTA
      const uint32_t stage_tx =
          ntok > 0 ? static_cast<uint32_t>(PAIR * (GE::B_BYTES + ntok * BK))
                   : static_cast<uint32_t>(PAIR * GE::STAGE_BYTES);
      if (MODE == GEMM_WGRAD && p.gmaps != nullptr && g != map_g && nkb > 0) {
        // this segment's maps end at its last row: a K block that crosses the end loads
        // the rows past it as zeros (they belong to the next expert, or are unwritten).
        // A gathered B keeps the source map: its rows past the end repeat the segment's
        // last row and meet A's zero rows.
        mA = p.gmaps + 2 * g;
        mB = GATHER ? &tmB : mA + 1;
        map_g = g;
        if (lane == 0) {
          asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(mA)
                       : "memory");
          if (!GATHER)
            asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(mB)
                         : "memory");
        }
        __syncwarp();
      }
      // gathered rows.  FC1: this CTA's 128 A rows of the tile, 4 per lane, fixed for the
      // tile.  WGRAD: the 64 K rows of a K block, 4 per lane of lanes 0..15, fetched one K
      // block ahead.  Rows past the segment's end take its last row.
      const int seg_last = seg0 + seg_rows - 1;
      int gi[4] = {0, 0, 0, 0};
      if (GATHER && nkb > 0) {
        if (MODE == GEMM_FC1_SWIGLU || MODE == GEMM_DGRAD2_SWIGLU) {
          // a tail tile's CTA takes ntok / 2 rows: lanes below ntok / 8 copy them
          const int r0 = seg0 + mt * GE::TILE_M + (ntok > 0 ? ntok / 2 : 128) * rank + 4 * lane;
#pragma unroll
          for (int q = 0; q < 4; ++q) gi[q] = gather_row(p, min(r0 + q, seg_last));
        } else if (MODE == GEMM_WGRAD && lane < 16) {
#pragma unroll
          for (int q = 0; q < 4; ++q) gi[q] = gather_row(p, min(seg0 + 4 * lane + q, seg_last));
        }
      }
      for (int kb = 0; kb < nkb; ++kb) {
        int gc[4] = {gi[0], gi[1], gi[2], gi[3]};
        if (GATHER && MODE == GEMM_WGRAD && lane < 16 && kb + 1 < nkb) {
          const int r0 = seg0 + (kb + 1) * BK + 4 * lane;
#pragma unroll
          for (int q = 0; q < 4; ++q) gi[q] = gather_row(p, min(r0 + q, seg_last));
        }
        if (!warp_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, p.err, WAIT_BUDGET)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_base + s * GE::STAGE_BYTES;
        const uint32_t sb = sa + GE::A_BYTES;
        const uint32_t full_local = smem_u32(&ctl->full[s]);
        const uint32_t full_leader = PAIR == 2 ? mapa_shared(full_local, 0) : full_local;
        // the leader's single arrive announces both CTAs' bytes; the peer's copies count
        // down the leader's barrier directly (its stage is free, so the leader's barrier
        // for this stage has already completed its previous phase)
        if (lane == 0) {
          if (leader) mbar_arrive_expect_tx(full_local, stage_tx);
          if (GE::TAIL && ntok > 0)
            issue_loads_tail<MODE, GATHER>(mB, &tmT, &tmW, p, sa, sb, full_leader, rank, g, mt,
                                           nt, seg0, kb, ntok);
          else
            issue_loads<MODE, PAIR, GATHER>(mA, mB, p, sa, sb, full_leader, PAIR == 2, rank, g,
                                            mt, nt, seg0, kb);
        }
        if (GATHER) {
          __syncwarp();
          const int k0 = kb * BK;
          auto g4 = [&](uint32_t dst, const CUtensorMap* m, int x) {
            if (PAIR == 2) tma_gather4_pair(dst, m, full_leader, x, gc[0], gc[1], gc[2], gc[3]);
            else tma_gather4(dst, m, full_leader, x, gc[0], gc[1], gc[2], gc[3]);
          };
          if (MODE == GEMM_FC1_SWIGLU || MODE == GEMM_DGRAD2_SWIGLU) {
            if (ntok == 0 || lane < ntok / 8)
              g4(sa + lane * 512, mA, k0);            // rows 4*lane .. 4*lane+3 of the tile
          } else if (MODE == GEMM_WGRAD && lane < 16) {
            // K rows 4*lane.. of each 64-column chunk; a chunk past the last column (an N
            // tail) re-reads the last chunk instead: its output columns are never stored
#pragma unroll
            for (int j = 0; j < GE::BN_CTA / 64; ++j)
              g4(sb + j * CHUNK_BYTES + lane * 512, mB,
                 min(nt * BN + rank * GE::BN_CTA + 64 * j, p.wg_N - 64));
          }
        }
        if (++s == STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    // every copy of this CTA is issued: the next kernel may be scheduled (it waits for
    // this one to complete before it touches memory)
    griddep_launch();
    // wait until every stage is free again: all commits aimed at this CTA have landed
    for (int i = 0; i < STAGES && ok; ++i) {
      if (!warp_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort_flag, p.err, WAIT_BUDGET / 4))
        break;
      if (++s == STAGES) {
        s = 0;
        ph ^= 1u;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA)
    if (leader) {
      constexpr uint32_t IDESC = make_idesc_bf16(GE::TILE_M, BN, ModeTraits<MODE>::A_MN ? 1 : 0,
                                                 ModeTraits<MODE>::B_MN ? 1 : 0);
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true, issued_any = false;
      const bool trace = g_clock_trace.on != 0;
      const long long trace_c0 = clock64();
      const unsigned long long trace_n0 = globaltimer_ns();
      for (int tile = unit; tile < total && ok; tile += num_units, ++it) {
        int g, mt, nt, ntok;
        tile_of(it, tile, g, mt, nt, ntok);
        const int nkb = (MODE == GEMM_WGRAD)
                            ? ceil_div(ctl->gstart[g + 1] - ctl->gstart[g], BK) : p.num_kb;
        const int buf = it & 1;
        const uint32_t tph = (it >> 1) & 1;
        if (!warp_wait(smem_u32(&ctl->tempty[buf]), tph ^ 1u, abort_flag, p.err, WAIT_BUDGET)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * BN);
        // Operand descriptors for the whole tile, so the K loop below is the same
        // instruction stream for both tile forms.  An ordinary tile reads A (the segment's
        // rows) at sa and B (weights) at sb; a tail tile reads the weights at sb as its A
        // and the segment's rows at sa as its B, with N = ntok.  K-major operands step
        // 32 bytes per K16, MN-major ones one 64 x 16 core block (2 KB); descriptor start
        // addresses count 16-byte units, so stage and K offsets add to the low field.
        const bool tail = GE::TAIL && ntok > 0;
        const bool a_mn = tail ? ModeTraits<MODE>::B_MN : ModeTraits<MODE>::A_MN;
        const bool b_mn = tail ? false : ModeTraits<MODE>::B_MN;
        const uint32_t idesc =
            tail ? make_idesc_bf16(256, ntok, ModeTraits<MODE>::B_MN ? 1 : 0, 0) : IDESC;
        const uint64_t adesc0 = make_smem_desc(smem_base + (tail ? GE::A_BYTES : 0u),
                                               a_mn ? CHUNK_BYTES : 16u, 1024);
        const uint64_t bdesc0 = make_smem_desc(smem_base + (tail ? 0u : GE::A_BYTES),
                                               b_mn ? CHUNK_BYTES : 16u, 1024);
        const uint32_t astep = a_mn ? 2048 >> 4 : 32 >> 4;
        const uint32_t bstep = b_mn ? 2048 >> 4 : 32 >> 4;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!warp_wait(smem_u32(&ctl->full[s]), ph, abort_flag, p.err, WAIT_BUDGET)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint64_t so = static_cast<uint64_t>((s * GE::STAGE_BYTES) >> 4);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t adesc = adesc0 + so + kk * astep;
              const uint64_t bdesc = bdesc0 + so + kk * bstep;
              if (PAIR == 2) tc_mma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0);
              else tc_mma_bf16(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            // the stage is free (in both CTAs) once these MMAs have read it
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
          const uint32_t tf = smem_u32(&ctl->tfull[buf]);
          if (nkb > 0) {
            if (PAIR == 2) tc_commit_pair_mc(tf, 0x3);
            else tc_commit(tf);
          } else {   // an empty segment: nothing to accumulate, hand the buffer over
            mbar_arrive(tf);
            if (PAIR == 2) mbar_arrive_remote(mapa_shared(tf, 1));
          }
        }
        __syncwarp();
      }
      if (trace && ok && issued_any && lane == 0)
        clock_trace_add(&g_clock_trace, clock64() - trace_c0, globaltimer_ns() - trace_n0);
      if (!ok && issued_any && lane == 0) {
        // drain the MMAs in flight before TMEM is released
        if (PAIR == 2) tc_commit_pair(smem_u32(&ctl->drain));
        else tc_commit(smem_u32(&ctl->drain));
        long long t0 = clock64();
        while (!mbar_try_wait(smem_u32(&ctl->drain), 0) && clock64() - t0 < WAIT_BUDGET / 4) {
        }
      }
      __syncwarp();
    }
  } else if (warp <= 5) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    int store_buf = 0;                      // staging buffer of the TMA-store epilogue
    int it = 0;
    int xc = 0;                             // FC1 tail tiles: exchange blocks used so far
    for (int tile = unit; tile < total; tile += num_units, ++it) {
      int g, mt, nt, ntok;
      tile_of(it, tile, g, mt, nt, ntok);
      const int seg0 = ctl->gstart[g];
      const int seg_end = ctl->gstart[g + 1];
      const int buf = it & 1;
      const uint32_t tph = (it >> 1) & 1;
      if (!warp_wait(smem_u32(&ctl->tfull[buf]), tph, abort_flag, p.err, WAIT_BUDGET)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(buf * BN);
      if (GE::TAIL && ntok > 0) {
        const long long row0 = static_cast<long long>(seg0) + mt * GE::TILE_M;
        if (!tail_epilogue<MODE>(p, ctl, taddr, xch_base, q, lane, rank, nt, row0,
                                 static_cast<int>(seg_end - row0), ntok, xc, abort_flag))
          break;
      } else if (MODE == GEMM_FC1_SWIGLU) {
        // Transposed through the warp's block like the FC2 data-gradient below: per
        // 32-column chunk each lane writes bf16(a) and bf16(b) of its row (a's 16-byte
        // pieces at 2k, b's at 2k + 1, XOR-swizzled by row), then each lane takes four
        // 8-column pieces of rows lane / 4 + 8 i and stores a, b and h = silu(a) b.
        const int f = p.f;
        const long long wrow0 = static_cast<long long>(seg0) + mt * GE::TILE_M + rank * 128 +
                                q * 32;
        const uint32_t blk = xch_base + static_cast<uint32_t>(q * XPOSE_BYTES);
        const int cc = 8 * (lane & 3);
#pragma unroll 1
        for (int c = 0; c < (BN / 2) / 32; ++c) {
          const int n0 = nt * (BN / 2) + c * 32;
          if (n0 >= f) break;                   // f is a multiple of 64: warp-uniform
          uint32_t ra[32], rb[32];
          tmem_ld32(taddr + c * 32, ra);
          tmem_ld32(taddr + BN / 2 + c * 32, rb);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float x[8], y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              x[e] = __uint_as_float(ra[8 * k + e]);
              y[e] = __uint_as_float(rb[8 * k + e]);
            }
            const uint4 va = pack8(x), vb = pack8(y);
            st_shared_v4(blk + lane * 128 + (((2 * k) ^ (lane & 7)) << 4), va);
            st_shared_v4(blk + lane * 128 + (((2 * k + 1) ^ (lane & 7)) << 4), vb);
          }
          __syncwarp();
          // all four pieces are read out first and the block released, so that the
          // arithmetic and stores of the four rows interleave
          uint4 va[4], vb[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = (lane >> 2) + 8 * i;
            const int k = lane & 3;
            va[i] = ld_shared_v4(blk + r * 128 + (((2 * k) ^ (r & 7)) << 4));
            vb[i] = ld_shared_v4(blk + r * 128 + (((2 * k + 1) ^ (r & 7)) << 4));
          }
          __syncwarp();                         // the block is read before the next chunk
          uint4 vh[4];                          // h of the four rows, without branches
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a[8], b[8], h[8];
            unpack8(va[i], a);                  // a, b as stored: h comes from them
            unpack8(vb[i], b);
#pragma unroll
            for (int e = 0; e < 8; ++e) h[e] = silu_f(a[e]) * b[e];
            vh[i] = pack8(h);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const long long prow = wrow0 + (lane >> 2) + 8 * i;
            if (prow < seg_end) {
              *reinterpret_cast<uint4*>(p.out0 + prow * 2 * f + n0 + cc) = va[i];
              *reinterpret_cast<uint4*>(p.out0 + prow * 2 * f + f + n0 + cc) = vb[i];
              *reinterpret_cast<uint4*>(p.out1 + prow * f + n0 + cc) = vh[i];
            }
          }
        }
      } else if (MODE == GEMM_FC2 || MODE == GEMM_DGRAD1) {
        // Transposed through the warp's block: bf16 rows of 64 bytes (piece k at 2k,
        // XOR-swizzled by row), stored as 16-byte row pieces, four lanes per row segment.
        const int n_out = p.n_out;
        const long long wrow0 = static_cast<long long>(seg0) + mt * GE::TILE_M + rank * 128 +
                                q * 32;
        const uint32_t blk = xch_base + static_cast<uint32_t>(q * XPOSE_BYTES);
        const int cc = 8 * (lane & 3);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int n0 = nt * BN + c * 32;
          if (n0 >= n_out) break;               // n_out is a multiple of 64: warp-uniform
          uint32_t ra[32];
          tmem_ld32(taddr + c * 32, ra);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(ra[8 * k + e]);
            st_shared_v4(blk + lane * 128 + (((2 * k) ^ (lane & 7)) << 4), pack8(x));
          }
          __syncwarp();
          uint4 v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = (lane >> 2) + 8 * i;
            v[i] = ld_shared_v4(blk + r * 128 + (((2 * (lane & 3)) ^ (r & 7)) << 4));
          }
          __syncwarp();                         // the block is read before the next chunk
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const long long prow = wrow0 + (lane >> 2) + 8 * i;
            if (prow < seg_end)
              *reinterpret_cast<uint4*>(p.out0 + prow * n_out + n0 + cc) = v[i];
          }
        }
      } else if (MODE == GEMM_DGRAD2_SWIGLU) {
        // The warp's 32 rows (TMEM lanes) x 32 columns of each chunk go through its 4 KB
        // block of shared memory (128-byte rows, 16-byte pieces XOR-swizzled by row, free of
        // bank conflicts both ways); each lane then takes four 8-column pieces, of rows
        // lane / 4 + 8 i, so the saved a, b are read and da, db written as 16-byte pieces,
        // four lanes per 64-byte row segment, instead of one row per lane.  The next chunk's
        // a, b are loaded while the current one is computed.
        const int f = p.f;
        const long long wrow0 = static_cast<long long>(seg0) + mt * GE::TILE_M + rank * 128 +
                                q * 32;
        // (the same region of the staging area as this warp's tail-tile block: the warps
        // are not in step, so each keeps to its own)
        const uint32_t blk = xch_base + static_cast<uint32_t>(q * XPOSE_BYTES);
        const int cc = 8 * (lane & 3);
        auto load_ab = [&](int c, uint4* xa, uint4* xb) {
          const int n0 = nt * BN + c * 32;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const long long prow = wrow0 + (lane >> 2) + 8 * i;
            xa[i] = xb[i] = make_uint4(0u, 0u, 0u, 0u);
            if (prow < seg_end && n0 < f) {
              const long long base = prow * 2 * f + n0 + cc;
              xa[i] = __ldg(reinterpret_cast<const uint4*>(p.aux + base));
              xb[i] = __ldg(reinterpret_cast<const uint4*>(p.aux + base + f));
            }
          }
        };
        uint4 na[4], nb[4];
        load_ab(0, na, nb);
        // the gate weight of each of the lane's four rows, looked up once per tile (0 past
        // the segment's end)
        float wr[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const long long prow = wrow0 + (lane >> 2) + 8 * i;
          wr[i] = prow < seg_end ? row_gate_weight(p, prow) : 0.0f;
        }
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int n0 = nt * BN + c * 32;
          if (n0 >= f) break;                   // f is a multiple of 64: warp-uniform
          uint4 ca[4], cb[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            ca[i] = na[i];
            cb[i] = nb[i];
          }
          if (c + 1 < BN / 32) load_ab(c + 1, na, nb);
          uint32_t ra[32];
          tmem_ld32(taddr + c * 32, ra);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                             blk + lane * 128 + ((k ^ (lane & 7)) << 4)),
                         "r"(ra[4 * k]), "r"(ra[4 * k + 1]), "r"(ra[4 * k + 2]),
                         "r"(ra[4 * k + 3])
                         : "memory");
          __syncwarp();
          // all four pieces are read out first and the block released, so that the
          // arithmetic and stores of the four rows interleave
          float dhs[4][8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = (lane >> 2) + 8 * i;
            const int k0 = 2 * (lane & 3);
            ld_shared_f32x4(blk + r * 128 + ((k0 ^ (r & 7)) << 4), dhs[i]);
            ld_shared_f32x4(blk + r * 128 + (((k0 + 1) ^ (r & 7)) << 4), dhs[i] + 4);
          }
          __syncwarp();                         // the block is read before the next chunk
          // the SwiGLU backward of the four rows without branches (rows past the segment's
          // end compute on zeros and are not stored), so that their arithmetic interleaves
          uint4 oda[4], odb[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float a[8], b[8], da[8], db[8];
            unpack8(ca[i], a);
            unpack8(cb[i], b);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float dh = dhs[i][e] * wr[i];
              const float sg = sigmoid_fast(a[e]);
              const float silu = a[e] * sg;
              const float dsilu = sg * (1.0f + a[e] * (1.0f - sg));
              da[e] = dh * b[e] * dsilu;
              db[e] = dh * silu;
            }
            oda[i] = pack8(da);
            odb[i] = pack8(db);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const long long prow = wrow0 + (lane >> 2) + 8 * i;
            if (prow < seg_end) {
              const long long base = prow * 2 * f + n0 + cc;
              *reinterpret_cast<uint4*>(p.out0 + base) = oda[i];
              *reinterpret_cast<uint4*>(p.out0 + base + f) = odb[i];
            }
          }
        }
      } else {   // WGRAD: dW[g][m][n], written as 32 x 64 boxes through shared memory
        const int m_base = mt * GE::TILE_M + rank * 128 + q * 32;   // this warp's 32 rows
        const bool rows_ok = m_base < p.wg_M;
        const bool empty_seg = (seg_end - seg0) <= 0;
        const uint32_t stage0 = staging_base + static_cast<uint32_t>((warp - 2) * 8192);
#pragma unroll 1
        for (int box = 0; box < BN / 64; ++box) {
          uint32_t ra[32], rb[32];
          if (!empty_seg) {
            tmem_ld32(taddr + box * 64, ra);
            tmem_ld32(taddr + box * 64 + 32, rb);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) ra[e] = rb[e] = 0u;
          }
          const int n0 = nt * BN + box * 64;
          if (rows_ok && n0 < p.wg_N) {
            const uint32_t buf_addr = stage0 + static_cast<uint32_t>(store_buf * 4096);
            // the box written two stores ago must have been read out of this buffer
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            // row `lane` of the box: 128 bytes = 8 chunks of 16 bytes, 128B-swizzled
            const uint32_t row_addr = buf_addr + lane * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t* src = c < 4 ? &ra[c * 8] : &rb[(c - 4) * 8];
              float x[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(src[e]);
              const uint4 v = pack8(x);
              const uint32_t dst = row_addr + ((c ^ (lane & 7)) << 4);
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x),
                           "r"(v.y), "r"(v.z), "r"(v.w)
                           : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d_hint(&tmC, buf_addr, n0, m_base, g, l2_policy_evict_first());
              bulk_commit_group();
            }
            store_buf ^= 1;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t te = smem_u32(&ctl->tempty[buf]);
        if (PAIR == 2) mbar_arrive_remote(mapa_shared(te, 0));   // the leader's barrier
        else mbar_arrive(te);
      }
    }
    if (GE::TMA_STORE && lane == 0) bulk_wait_group_all();   // stores done before exit
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  if (PAIR == 2) cluster_sync_all();   // no CTA leaves while its peer may still signal it
  else __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    if (PAIR == 2) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
  griddep_launch();
}

// One thread per segment: copy the two operand maps of the weight-gradient GEMM into
// device memory and set their row extent to the segment's end (offsets[g+1]).
__global__ void prep_segment_maps(const __grid_constant__ CUtensorMap tmA,
                                  const __grid_constant__ CUtensorMap tmB,
                                  const int32_t* __restrict__ offsets, int G, long long rows_cap,
                                  CUtensorMap* out) {
  griddep_wait();   // see common.cuh: dependent launches
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= G) return;
  long long end = offsets[g + 1];
  end = end < 1 ? 1 : (end > rows_cap ? rows_cap : end);
  const uint4* sa = reinterpret_cast<const uint4*>(&tmA);
  const uint4* sb = reinterpret_cast<const uint4*>(&tmB);
  uint4* da = reinterpret_cast<uint4*>(out + 2 * g);
  uint4* db = reinterpret_cast<uint4*>(out + 2 * g + 1);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    da[i] = sa[i];
    db[i] = sb[i];
  }
  const uint32_t e32 = static_cast<uint32_t>(end);
  asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(da),
               "r"(e32)
               : "memory");
  asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(db),
               "r"(e32)
               : "memory");
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  griddep_launch();
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// 2-D bf16 tensor map over a row-major [rows, cols] matrix, 128-byte swizzle,
// box = 64 columns (128 bytes) x box_rows rows, zero fill out of bounds.
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 tensor map over dW viewed as [groups][rows][cols], 128-byte swizzle, box =
// 64 columns x 32 rows x 1 group: a store never crosses into the next group's rows.
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t groups) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {cols, rows, groups};
  cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  cuuint32_t box[3] = {64, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int MODE, int PAIR, bool GATHER = false>
cudaError_t launch_mode(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                        const TailMaps& tt, const CUtensorMap& tw, const KParams& kp,
                        cudaStream_t st) {
  auto kern = grouped_gemm_kernel<MODE, PAIR, GATHER>;
  constexpr size_t SMEM = smem_bytes<MODE, PAIR>();
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
    cfg.blockDim = dim3(NUM_THREADS);
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
  return launch_pdl(kern, dim3(grid), dim3(NUM_THREADS), SMEM, st, PAIR, ta, tb, tc, tt, tw, kp);
}

// tt, tw: the tail tiles' segment-row maps and, for FC1, weight map (64-row boxes); unused
// (tt zeroed, tw = tb) when the tail tiles are off
template <int MODE, bool GATHER = false>
cudaError_t launch_pick(bool pair, const CUtensorMap& ta, const CUtensorMap& tb,
                        const TailMaps& tt, const CUtensorMap& tw, const KParams& kp,
                        cudaStream_t st) {
  // the output map is used by the weight-gradient mode only; the others pass tb through
  return pair ? launch_mode<MODE, 2, GATHER>(ta, tb, tb, tt, tw, kp, st)
              : launch_mode<MODE, 1, GATHER>(ta, tb, tb, tt, tw, kp, st);
}

}  // namespace

cudaError_t launch_grouped_gemm(const GroupedGemmArgs& a, cudaStream_t st) {
  if (a.G < 1 || a.G > MAX_G) return cudaErrorInvalidValue;
  KParams kp{};
  kp.G = a.uniform_rows > 0 ? 1 : a.G;
  kp.uniform_rows = a.uniform_rows;
  kp.rows_cap = a.rows_cap;
  kp.d = a.d;
  kp.f = a.f;
  kp.wg_M = a.wg_M;
  kp.wg_N = a.wg_N;
  kp.offsets = a.offsets;
  kp.out0 = static_cast<__nv_bfloat16*>(a.out0);
  kp.out1 = static_cast<__nv_bfloat16*>(a.out1);
  kp.aux = static_cast<const __nv_bfloat16*>(a.aux);
  kp.err = a.err;
  kp.gmaps = nullptr;
  const bool gather = a.gather_idx != nullptr;
  if (gather && (!a.gather_src || a.gather_rows < 1 || a.gather_rows > INT32_MAX ||
                 (a.mode != GEMM_FC1_SWIGLU && a.mode != GEMM_DGRAD2_SWIGLU &&
                  a.mode != GEMM_WGRAD)))
    return cudaErrorInvalidValue;
  kp.gidx = a.gather_idx;
  kp.gather_rows = static_cast<int>(a.gather_rows);
  kp.gw = nullptr;
  kp.gslot = nullptr;
  kp.n_slots = 0;
  if (gather && a.mode == GEMM_DGRAD2_SWIGLU) {
    // the rows are dy's tokens: each needs the gate weight of its slot
    if (!a.gate_w || !a.gate_slot || a.n_slots < 1) return cudaErrorInvalidValue;
    kp.gw = a.gate_w;
    kp.gslot = a.gate_slot;
    kp.n_slots = a.n_slots;
  }
  const uint64_t G = static_cast<uint64_t>(kp.G);
  const uint64_t rows = static_cast<uint64_t>(a.rows_cap);
  const uint64_t d = static_cast<uint64_t>(a.d), f = static_cast<uint64_t>(a.f);
  // The CTA pair's 256-row tile pays off when the segments are long; with short segments
  // (e.g. many fine-grained experts) half of a 256-row tile would be masked, so the
  // single-CTA 128-row tile is used.  The weight-gradient modes tile the fixed weight
  // shape and always use the pair.
  const double rows_per_group = static_cast<double>(a.rows_cap) / static_cast<double>(kp.G);
  const bool pair_rows = rows_per_group >= 192.0;
  const bool pair = a.mode == GEMM_WGRAD ? true : pair_rows;
  const uint32_t b_rows = pair ? BN / 2 : BN;   // B rows (N) held by one CTA
  // swap-AB tail tiles: CTA pairs, fixed-K modes
  const bool tail = pair && a.mode != GEMM_WGRAD;
  kp.tail_rows_max = tail ? TAIL_ROWS_MAX : 0;
  CUtensorMap ta, tb, tw;
  TailMaps tt;
  memset(&tt, 0, sizeof(tt));
  // the segment rows of a tail tile, one map per N = 32 (i + 1): boxes of 16 (i + 1) rows
  auto tail_maps = [&](const void* base, uint64_t cols) {
    for (int i = 0; i < 8; ++i)
      if (!make_map(&tt.m[i], base, cols, rows, static_cast<uint32_t>(16 * (i + 1)))) return false;
    return true;
  };
  bool ok = true;
  switch (a.mode) {
    case GEMM_FC1_SWIGLU:
      kp.num_n_tiles = (a.f + BN / 2 - 1) / (BN / 2);
      kp.num_kb = a.d / BK;
      kp.n_out = a.f;
      ok = (gather ? make_map(&ta, a.gather_src, d, static_cast<uint64_t>(a.gather_rows), 1)
                   : make_map(&ta, a.A, d, rows, 128)) &&
           make_map(&tb, a.B, d, G * 2 * f, BN / 2);
      // the tail tiles' segment rows come through the gather copies when gathering
      tw = tb;
      if (ok && tail)
        ok = (gather || tail_maps(a.A, d)) && make_map(&tw, a.B, d, G * 2 * f, 64);
      if (!ok) return cudaErrorInvalidValue;
      return gather ? launch_pick<GEMM_FC1_SWIGLU, true>(pair, ta, tb, tt, tw, kp, st)
                    : launch_pick<GEMM_FC1_SWIGLU>(pair, ta, tb, tt, tw, kp, st);
    case GEMM_FC2:
      kp.num_n_tiles = (a.d + BN - 1) / BN;
      kp.num_kb = a.f / BK;
      kp.n_out = a.d;
      ok = make_map(&ta, a.A, f, rows, 128) && make_map(&tb, a.B, f, G * d, b_rows) &&
           (!tail || tail_maps(a.A, f));
      if (!ok) return cudaErrorInvalidValue;
      return launch_pick<GEMM_FC2>(pair, ta, tb, tt, tb, kp, st);
    case GEMM_DGRAD2_SWIGLU:
      kp.num_n_tiles = (a.f + BN - 1) / BN;
      kp.num_kb = a.d / BK;
      kp.n_out = a.f;
      // gathered: the rows of dy [gather_rows, d] (one-row boxes for the gather4 copies,
      // which also bring a tail tile's rows)
      ok = (gather ? make_map(&ta, a.gather_src, d, static_cast<uint64_t>(a.gather_rows), 1)
                   : make_map(&ta, a.A, d, rows, 128)) &&
           make_map(&tb, a.B, f, G * d, 64) && (!tail || gather || tail_maps(a.A, d));
      if (!ok) return cudaErrorInvalidValue;
      return gather ? launch_pick<GEMM_DGRAD2_SWIGLU, true>(pair, ta, tb, tt, tb, kp, st)
                    : launch_pick<GEMM_DGRAD2_SWIGLU>(pair, ta, tb, tt, tb, kp, st);
    case GEMM_DGRAD1:
      kp.num_n_tiles = (a.d + BN - 1) / BN;
      kp.num_kb = 2 * a.f / BK;
      kp.n_out = a.d;
      ok = make_map(&ta, a.A, 2 * f, rows, 128) && make_map(&tb, a.B, d, G * 2 * f, 64) &&
           (!tail || tail_maps(a.A, 2 * f));
      if (!ok) return cudaErrorInvalidValue;
      return launch_pick<GEMM_DGRAD1>(pair, ta, tb, tt, tb, kp, st);
    case GEMM_WGRAD:
      kp.num_n_tiles = (a.wg_N + BN - 1) / BN;
      kp.wg_m_tiles = (a.wg_M + 256 - 1) / 256;
      kp.wg_n_fast = kp.wg_m_tiles > kp.num_n_tiles ? 1 : 0;
      kp.n_out = a.wg_N;
      {
        CUtensorMap tc;
        ok = make_map(&ta, a.A, static_cast<uint64_t>(a.wg_M), rows, 64) &&
             (gather ? make_map(&tb, a.gather_src, static_cast<uint64_t>(a.wg_N),
                                static_cast<uint64_t>(a.gather_rows), 1)
                     : make_map(&tb, a.B, static_cast<uint64_t>(a.wg_N), rows, 64)) &&
             make_map_3d(&tc, a.out0, static_cast<uint64_t>(a.wg_N),
                         static_cast<uint64_t>(a.wg_M), G);
        if (!ok) return cudaErrorInvalidValue;
        if (a.uniform_rows <= 0) {
          // segments end inside the buffers: per-segment maps, prepared on the device
          if (!a.seg_maps || (reinterpret_cast<uintptr_t>(a.seg_maps) & 127u))
            return cudaErrorInvalidValue;
          CUtensorMap* maps = static_cast<CUtensorMap*>(a.seg_maps);
          const cudaError_t e =
              launch_pdl(prep_segment_maps, dim3((kp.G + 63) / 64), dim3(64), 0, st, 1, ta, tb,
                         a.offsets, kp.G, a.rows_cap, maps);
          if (e != cudaSuccess) return e;
          kp.gmaps = maps;
        }
        return gather ? launch_mode<GEMM_WGRAD, 2, true>(ta, tb, tc, tt, tb, kp, st)
                      : launch_mode<GEMM_WGRAD, 2>(ta, tb, tc, tt, tb, kp, st);
      }
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t gemm_clock_trace_set(bool on) {
  if (on) {
    const ClockTrace t{1, 0, 0, 0};
    return cudaMemcpyToSymbol(g_clock_trace, &t, sizeof(t));
  }
  const int off = 0;
  return cudaMemcpyToSymbol(g_clock_trace, &off, sizeof(off), offsetof(ClockTrace, on));
}

cudaError_t gemm_clock_trace_add(unsigned long long out[3]) {
  ClockTrace t;
  const cudaError_t e = cudaMemcpyFromSymbol(&t, g_clock_trace, sizeof(t));
  if (e != cudaSuccess) return e;
  out[0] += t.cycles;
  out[1] += t.ns;
  out[2] += t.loops;
  return cudaSuccess;
}

}  // namespace moe
