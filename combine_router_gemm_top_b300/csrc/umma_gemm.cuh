// Persistent, warp-specialised tcgen05 GEMM for sm_103a:
//   C[128 x BN tile] = A[rows, K] . B[cols, K]^T,  bf16 in, fp32 in TMEM.
//
// One CTA per SM, 10 warps:
//   warp 0      TMA producer (one elected lane): A and B tiles into a ring of
//               shared-memory stages (128-byte swizzle), completion counted
//               on per-stage "full" mbarriers.
//   warp 1      MMA issuer (one lane) and TMEM owner: 4 x tcgen05.mma
//               (128 x BN x 16) per 64-wide K block; tcgen05.commit frees the
//               stage ("empty" barrier) and, after the last K block,
//               publishes the accumulator ("tfull").  Two accumulators
//               alternate so the epilogue of tile i overlaps the MMAs of
//               tile i+1.
//   warps 2-9   epilogue: tcgen05.ld of their 32 TMEM lanes (one tile row
//               per thread), the mode's math, 16-byte stores, then "tempty".
//               Two warps share each lane quarter and take alternate column
//               chunks, so stores issue from 8 warps.
//
// Three modes share the pipeline and differ in tile scheduling, the B
// operand rows and the epilogue:
//   kRoute  router logits, split-K: tile = (m block, K split); writes fp32
//           partial logits [split][T][E], or with one split and a softmax
//           top-1/top-2 of at most 64 experts selects in the epilogue.
//   kUp     grouped SwiGLU up-projection: tile = (expert, n block, m block)
//           over ragged expert segments; B = 128 gate rows of W1 stacked on
//           the matching 128 up rows of W3 (BN = 256), epilogue
//           H = SiLU(gate) * up rounded to bf16.
//   kDown   grouped down-projection: B = 256 rows of W2, epilogue rounds to
//           bf16.
// Backward modes (training path; expert segments start on 64-row
// boundaries and padding rows are zero):
//   kDH     dH = dYp . W2_e: A = dYp rows (K = D, K-major), B = W2 [D, F]
//           read MN-major (F contiguous); bf16 out [rows, F].
//   kUpBwd  recomputes gate and up as kUp does; the epilogue reads dH and
//           writes dG = dH * up * SiLU'(gate) and dU = dH * SiLU(gate) into
//           dGU [rows, 2F] (W13's row order) and H = SiLU(gate) * up.
//   kDX     dXp = dGU . W13_e: A = dGU rows (K = 2F), B = W13 [2F, D] read
//           MN-major; bf16 out [rows, D].
//   kWG2    dW2_e = dYp_e^T . H_e and
//   kWG13   dW13_e = dGU_e^T . Xp_e: both operands MN-major over the
//           expert's token rows (the contraction), tile = (expert, 128
//           output rows, 256 output columns), fp32 out.  An expert with no
//           rows gets zeros.
// Router backward modes.  The fp32 logit gradient enters as two bf16 terms
// dl = hi + lo (hi = bf16(dl), lo = bf16(dl - hi)), stored side by side as
// dL2 [T, 2E]; each product with a bf16 operand is exact in the fp32
// accumulator, so the split carries dl to about 2^-17 relative.
//   kRDX    dx[t, :] += dL2[t, :] . [W_r; W_r]: A = dL2 rows (K = 2E,
//           K-major), B = W_r [E, D] read MN-major (K row = k mod E);
//           the epilogue adds into the bf16 dx in place.
//   kRDW    dW_r = [hi; lo]^T . [x; x]: A = dL2 read MN-major (expert
//           columns), B = x read MN-major, K = 2T with the hi and lo halves
//           of each 64-token block adjacent; split-K tiles write fp32
//           partials [split][E][D].
// Ragged tails (grouped modes): the last row block of an expert with at most
// 112 rows runs with the operands swapped.  The same shared-memory tiles
// feed two MMAs of shape 128 x n x 16, n = the tail rounded up to 16: the
// weight halves of the B tile are the 128-row A operands and the token
// tile is the n-row B operand.  TMEM then holds [feature, token] and the
// epilogue writes transposed.  This cuts the MMA work spent on padding rows
// from up to 127 rows per expert to at most 15.
// Every wait is time-bounded (see mbar_wait); on expiry the CTA stops
// issuing, drains its own copies and MMAs, frees TMEM, and reports
// MOE_ERR_TIMEOUT.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {

enum GemmMode {
  kRoute = 0, kUp = 1, kDown = 2,
  kDH = 3, kUpBwd = 4, kDX = 5, kWG2 = 6, kWG13 = 7,
  kRDX = 8, kRDW = 9
};

// Static properties of a mode.
template <int MODE>
struct ModeInfo {
  // token rows on M, ragged per expert (tiles from the expert offsets)
  static constexpr bool grouped_m = MODE == kUp || MODE == kDown ||
                                    MODE == kDH || MODE == kUpBwd ||
                                    MODE == kDX;
  // per-expert weight gradient: M x N output, K = the expert's token rows
  static constexpr bool wgrad = MODE == kWG2 || MODE == kWG13;
  static constexpr bool a_mn = wgrad || MODE == kRDW;
  static constexpr bool b_mn = MODE == kDH || MODE == kDX || wgrad ||
                               MODE == kRDX || MODE == kRDW;
  // fp32 output through the per-warp staging tiles
  static constexpr bool staged = wgrad || MODE == kRDW;
  static constexpr bool swap_tails = MODE == kUp || MODE == kDown;
  // B tile is gate rows stacked on up rows
  static constexpr bool gate_up = MODE == kUp || MODE == kUpBwd;
};

constexpr int kBM = 128;          // tile rows (TMEM lanes)
constexpr int kBK = 64;           // K elements per stage (one 128-byte row)
constexpr int kUmmaK = 16;        // K per tcgen05.mma for 16-bit inputs
constexpr int kMaxStages = 8;
constexpr int kEpiWarps = 8;      // two per TMEM lane quarter
constexpr int kGemmThreads = 64 + kEpiWarps * 32;
constexpr int kMaxGroups = 1024;  // experts the grouped scheduler handles
constexpr uint32_t kATileBytes = kBM * kBK * 2;
// Weight-gradient epilogue: a 32 x 32 fp32 staging tile per epilogue warp,
// rows padded to 36 floats (16-byte aligned, conflict-free float4 access).
constexpr int kStageLd = 36;
constexpr size_t kStageBytes = static_cast<size_t>(kEpiWarps) * 32 * kStageLd * 4;

// experts the router GEMM's epilogue selection holds in registers
constexpr int kRouteSelMaxE = 64;

struct GemmArgs {
  int32_t M;                // route: T ; grouped: rows allocated (max_rows)
  int32_t k_blocks;         // K / 64 (rounded up)
  int32_t BN;               // N tile (route: E rounded up to 16; else 256)
  int32_t stages;           // shared-memory ring depth
  int32_t tmem_cols;        // power of two >= 2 * BN
  // route
  int32_t splits, kb_per_split, E;
  // grouped
  int32_t groups;           // experts
  int32_t n_tiles;          // N blocks per expert
  int32_t F;                // up: gate/up row split inside W13
  int32_t b_rows_per_group; // up: 2F ; down: D
  const int32_t* offsets;   // [groups + 1] expert row offsets
  // output
  void* out;
  int32_t out_ld;           // elements per output row
  int32_t out_cols;         // valid output columns
  int32_t* status;
  uint64_t wait_limit_ns;
  // backward modes
  const void* aux_in;       // kUpBwd: dH [rows, F]
  void* out2;               // kUpBwd: H [rows, F]
  int32_t m_total;          // wgrad: output rows per expert (D or 2F)
  int32_t m_tiles;          // wgrad: m_total / 128
  int32_t n_fast;           // wgrad: column blocks vary fastest (keeps the
                            // smaller B operand resident in L2)
  // router backward
  int32_t row_limit;        // kRDW: output rows (E); 0 = no row mask
  int64_t split_stride;     // kRDW: elements between split partials
  // kRoute with one K split, softmax scores, no groups, k <= 2: the epilogue
  // selects (sel_idx != nullptr) instead of writing partial logits
  int32_t* sel_idx;         // [T, k] out
  float* sel_gate;          // [T, k] out
  float* sel_logits;        // [T, E] out or nullptr
  const float* sel_offset;  // [E] or nullptr, added to the logits
  int32_t sel_k;            // 1 or 2
  int32_t sel_full;         // 1: softmax over all E (else over the k)
};

struct TileInfo {
  int32_t a_row;      // first A row (TMA coordinate)
  int32_t rows;       // valid rows in the tile (1..128)
  int32_t b_row;      // first B row
  int32_t b_row2;     // second B half (up mode)
  int32_t out_col;    // first output column
  int32_t kb_begin, kb_end;
  int32_t split;      // route
  int32_t swap_n;     // grouped tail: MMA N of the swapped form, 0 = normal
};

struct GemmShared {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t xfull[2][4];   // route selection: half 1 -> half 0, per quarter
  uint32_t tmem_base;
  int32_t abort;
  int32_t total_tiles;
  int32_t prefix[kMaxGroups + 1];   // grouped: first tile of each expert
};

template <int MODE>
__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a,
                                                const GemmShared& sh, int t) {
  TileInfo ti;
  if (MODE == kRoute) {
    const int m_tiles = (a.M + kBM - 1) / kBM;
    const int m = t % m_tiles;
    ti.split = t / m_tiles;
    ti.a_row = m * kBM;
    ti.rows = min(kBM, a.M - ti.a_row);
    ti.b_row = 0;
    ti.b_row2 = 0;
    ti.out_col = 0;
    ti.kb_begin = ti.split * a.kb_per_split;
    ti.kb_end = min(a.k_blocks, ti.kb_begin + a.kb_per_split);
    ti.swap_n = 0;
    return ti;
  }
  if (MODE == kRDX || MODE == kRDW) {
    // kRDX: m = token block, K = the 2E columns of dL2.
    // kRDW: m = expert block, then column block, then K split.
    const int m_tiles = (a.M + kBM - 1) / kBM;
    const int m = t % m_tiles;
    const int rest = t / m_tiles;
    const int n = rest % a.n_tiles;
    ti.split = MODE == kRDW ? rest / a.n_tiles : 0;
    ti.swap_n = 0;
    ti.a_row = m * kBM;
    ti.rows = min(kBM, a.M - ti.a_row);
    ti.b_row = m * kBM;
    ti.b_row2 = 0;
    ti.out_col = n * 256;
    ti.kb_begin = ti.split * a.kb_per_split;
    ti.kb_end = min(a.k_blocks, ti.kb_begin + a.kb_per_split);
    return ti;
  }
  if (ModeInfo<MODE>::wgrad) {
    const int per_e = a.m_tiles * a.n_tiles;
    const int e = t / per_e;
    const int local = t - e * per_e;
    // tiles running at the same time share the operand that varies
    // slowest; the other one should be the one that fits L2
    const int n = a.n_fast ? local % a.n_tiles : local / a.m_tiles;
    const int m = a.n_fast ? local / a.n_tiles : local - n * a.m_tiles;
    ti.split = 0;
    ti.swap_n = 0;
    ti.a_row = e * a.m_total + m * kBM;   // output row of the tile
    ti.rows = kBM;
    ti.b_row = m * kBM;                    // A's MN coordinate
    ti.b_row2 = 0;
    ti.out_col = n * 256;                  // B's MN coordinate
    ti.kb_begin = __ldg(a.offsets + e) >> 6;
    ti.kb_end = __ldg(a.offsets + e + 1) >> 6;
    return ti;
  }
  // binary search: the expert whose tile range holds t
  int lo = 0, hi = a.groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sh.prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int row0 = __ldg(a.offsets + e);
  const int cnt = __ldg(a.offsets + e + 1) - row0;
  const int m_tiles = (cnt + kBM - 1) / kBM;
  const int local = t - sh.prefix[e];
  const int n = local / m_tiles;
  const int m = local - n * m_tiles;
  ti.split = 0;
  ti.a_row = row0 + m * kBM;
  ti.rows = min(kBM, cnt - m * kBM);
  ti.swap_n = ModeInfo<MODE>::swap_tails && ti.rows <= kBM - 16
                  ? (ti.rows + 15) & ~15
                  : 0;
  ti.kb_begin = 0;
  ti.kb_end = a.k_blocks;
  if (ModeInfo<MODE>::gate_up) {
    ti.b_row = e * a.b_rows_per_group + n * 128;
    ti.b_row2 = e * a.b_rows_per_group + a.F + n * 128;
    ti.out_col = n * 128;
  } else if (ModeInfo<MODE>::b_mn) {
    // MN-major B: b_row is the expert's first K row in B's row space
    ti.b_row = e * a.b_rows_per_group;
    ti.b_row2 = 0;
    ti.out_col = n * 256;
  } else {
    ti.b_row = e * a.b_rows_per_group + n * 256;
    ti.b_row2 = 0;
    ti.out_col = n * 256;
  }
  return ti;
}

__device__ __forceinline__ float silu_f32(float g) {
  return g / (1.0f + __expf(-g));
}

// Epilogue of one tile for the thread owning tile row `r` (TMEM lane r);
// `half` selects the alternate column chunks this warp handles.
template <int MODE>
__device__ __forceinline__ void epilogue_row(
    const GemmArgs& a, const TileInfo& ti, uint32_t tmem_row, int r, int half,
    float* stage, int parity = 0, uint64_t* xbar = nullptr,
    uint32_t xphase = 0, volatile int* abort_flag = nullptr) {
  if (MODE != kRoute && ti.swap_n != 0) {
    // swapped tail: TMEM lane r is output feature out_col + r (and, for the
    // down projection, out_col + 128 + r); column j is token row a_row + j
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) +
                         static_cast<int64_t>(ti.a_row) * a.out_ld +
                         ti.out_col + r;
    const int rows = min(ti.rows, a.M - ti.a_row);
    const bool lo_ok = ti.out_col + r < a.out_cols;
    const bool hi_ok = ti.out_col + 128 + r < a.out_cols;
#pragma unroll 1
    for (int c = 16 * half; c < ti.swap_n; c += 32) {
      float v0[16], v1[16];
      tmem_ld16(tmem_row + c, v0);
      tmem_ld16(tmem_row + 128 + c, v1);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int j = c + i;
        if (j < rows) {
          __nv_bfloat16* o = out + static_cast<int64_t>(j) * a.out_ld;
          if (MODE == kUp) {
            if (lo_ok) o[0] = __float2bfloat16_rn(silu_f32(v0[i]) * v1[i]);
          } else {
            if (lo_ok) o[0] = __float2bfloat16_rn(v0[i]);
            if (hi_ok) o[128] = __float2bfloat16_rn(v1[i]);
          }
        }
      }
    }
    return;
  }
  if (ModeInfo<MODE>::staged) {
    // fp32 weight-gradient rows; an expert with no token rows gets zeros.
    // Each 32 x 32 chunk goes through this warp's staging tile so that a
    // store instruction writes four whole 128-byte row segments instead of
    // one 16-byte piece of 32 different rows.
    const int lane = r & 31;
    const int row0 = ti.a_row + (r & ~31);       // the warp's first row
    const bool empty = ti.kb_end <= ti.kb_begin;
    float* obase = reinterpret_cast<float*>(a.out) + ti.split * a.split_stride;
#pragma unroll 1
    for (int c = 32 * half; c < 256; c += 64) {
      float v[32];
      if (empty) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
      } else {
        tmem_ld32(tmem_row + c, v);
      }
      if (ti.out_col + c < a.out_cols) {
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(stage + lane * kStageLd + i) =
              make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        __syncwarp();
        const int sub = lane >> 3;                // row within a group of 4
        const int col = (lane & 7) * 4;
#pragma unroll
        for (int rr = 0; rr < 32; rr += 4) {
          const int row = row0 + rr + sub;
          const float4 q =
              *reinterpret_cast<const float4*>(stage + (rr + sub) * kStageLd + col);
          if (a.row_limit == 0 || row < a.row_limit)
            *reinterpret_cast<float4*>(obase +
                                       static_cast<int64_t>(row) * a.out_ld +
                                       ti.out_col + c + col) = q;
        }
        __syncwarp();
      }
    }
    return;
  }
  const int64_t grow = static_cast<int64_t>(ti.a_row) + r;
  const bool valid = r < ti.rows && grow >= 0 && grow < a.M;
  if (MODE == kRoute && a.sel_idx != nullptr) {
    // The two epilogue warps on a token row's TMEM lanes share its E (<= 64)
    // logits: half 0 the first ceil(n/2) 16-column chunks, half 1 the rest,
    // each in registers.  Each keeps its top two in expert order (a
    // strictly larger key replaces, so ties keep the lower index) and, for
    // the full softmax, its maximum and the sum of its terms, independent of
    // each other once that maximum is known.  Half 1 hands its part to half
    // 0 through shared memory and an mbarrier per quarter (bounded wait),
    // and half 0 merges, half 1's experts losing ties.  Slots alternate with
    // the accumulator: half 1 rewrites one only for the tile after next,
    // whose accumulator half 0 must first have released.
    __shared__ float xk[2][4][32][4];
    __shared__ int xi[2][4][32][2];
    constexpr int kHalfE = kRouteSelMaxE / 2;
    const int E = a.E;
    const int quarter = r >> 5;
    const int lane = r & 31;
    const int nch = a.BN / 16;
    const int c_lo = half == 0 ? 0 : 16 * ((nch + 1) / 2);
    const int c_hi = half == 0 ? 16 * ((nch + 1) / 2) : a.BN;
    float v[kHalfE];
#pragma unroll
    for (int c = 0; c < kHalfE; c += 16) {
      if (c_lo + c < c_hi) {
        float t[16];
        tmem_ld16(tmem_row + c_lo + c, t);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[c + i] = t[i];
      }
    }
    float b0 = -INFINITY, b1 = -INFINITY, z = 0.0f;
    int i0 = -1, i1 = -1;
    if (valid) {
#pragma unroll
      for (int c = 0; c < kHalfE; ++c) {
        const int e = c_lo + c;
        if (e < c_hi && e < E) {
          float l = v[c];
          if (a.sel_offset != nullptr) l = __fadd_rn(l, __ldg(a.sel_offset + e));
          v[c] = l;
          if (l > b0) {
            b1 = b0;
            i1 = i0;
            b0 = l;
            i0 = e;
          } else if (l > b1) {
            b1 = l;
            i1 = e;
          }
        }
      }
      if (a.sel_logits != nullptr) {
        float* lout = a.sel_logits + grow * E;
#pragma unroll
        for (int c = 0; c < kHalfE; ++c)
          if (c_lo + c < c_hi && c_lo + c < E) lout[c_lo + c] = v[c];
      }
      if (a.sel_full && i0 >= 0) {
        float zs[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int c = 0; c < kHalfE; ++c)
          if (c_lo + c < c_hi && c_lo + c < E) zs[c & 3] += expf(v[c] - b0);
        z = (zs[0] + zs[1]) + (zs[2] + zs[3]);
      }
    }
    const int slot = parity & 1;
    uint64_t* bar = xbar + 4 * slot + quarter;
    if (half == 1) {
      xk[slot][quarter][lane][0] = b0;
      xk[slot][quarter][lane][1] = b1;
      xk[slot][quarter][lane][2] = z;
      xi[slot][quarter][lane][0] = i0;
      xi[slot][quarter][lane][1] = i1;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
      return;
    }
    bool ok = true;
    if (lane == 0) ok = mbar_wait(bar, xphase, abort_flag, a.wait_limit_ns);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    __syncwarp();
    if (!ok || !valid) return;
    const float c0 = xk[slot][quarter][lane][0];
    const float c1 = xk[slot][quarter][lane][1];
    const float zc = xk[slot][quarter][lane][2];
    const int j0 = xi[slot][quarter][lane][0];
    const int j1 = xi[slot][quarter][lane][1];
    float m0, m1;
    int k0, k1;
    if (c0 > b0) {
      m0 = c0;
      k0 = j0;
      if (c1 > b0) {
        m1 = c1;
        k1 = j1;
      } else {
        m1 = b0;
        k1 = i0;
      }
    } else {
      m0 = b0;
      k0 = i0;
      if (c0 > b1) {
        m1 = c0;
        k1 = j0;
      } else {
        m1 = b1;
        k1 = i1;
      }
    }
    float g0, g1 = 0.0f;
    if (a.sel_full) {
      // each half's sum is over its own maximum; m0 is the overall one
      float zt = 0.0f;
      if (i0 >= 0) zt += z * expf(b0 - m0);
      if (j0 >= 0) zt += zc * expf(c0 - m0);
      g0 = 1.0f / zt;
      if (a.sel_k > 1) g1 = expf(m1 - m0) / zt;
    } else if (a.sel_k > 1) {
      const float e1 = expf(m1 - m0);
      const float zz = 1.0f + e1;
      g0 = 1.0f / zz;
      g1 = e1 / zz;
    } else {
      g0 = 1.0f;
    }
    a.sel_idx[grow * a.sel_k] = k0;
    a.sel_gate[grow * a.sel_k] = g0;
    if (a.sel_k > 1) {
      a.sel_idx[grow * a.sel_k + 1] = k1;
      a.sel_gate[grow * a.sel_k + 1] = g1;
    }
    return;
  }
  if (MODE == kRoute) {
    // partial logits [split][T][E] fp32
    float* out = reinterpret_cast<float*>(a.out) +
                 (static_cast<int64_t>(ti.split) * a.M + grow) * a.E;
    for (int c = 16 * half; c < a.BN; c += 32) {
      float v[16];
      tmem_ld16(tmem_row + c, v);
      if (valid) {
        if ((a.E & 3) == 0 && c + 16 <= a.E) {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(out + c + i) =
                make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c + i < a.E) out[c + i] = v[i];
        }
      }
    }
  } else if (MODE == kUp) {
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) +
                         grow * a.out_ld + ti.out_col;
#pragma unroll 1
    for (int c = 32 * half; c < 128; c += 64) {
      float g[32], u[32];
      tmem_ld32(tmem_row + c, g);
      tmem_ld32(tmem_row + 128 + c, u);
      if (valid) {
        float h[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) h[i] = silu_f32(g[i]) * u[i];
#pragma unroll
        for (int i = 0; i < 32; i += 8)
          st_v4(out + c + i, Vec16<__nv_bfloat16>::from_f32(h + i));
      }
    }
  } else if (MODE == kUpBwd) {
    // recomputed gate g and up u; with dH: dU = dH * SiLU(g),
    // dG = dH * u * SiLU'(g), SiLU'(g) = s (1 + g (1 - s)), s = sigmoid(g);
    // H = SiLU(g) * u for the W2 gradient
    const int64_t F = a.F;
    const __nv_bfloat16* dh = reinterpret_cast<const __nv_bfloat16*>(
                                  a.aux_in) + grow * F + ti.out_col;
    __nv_bfloat16* dgu = reinterpret_cast<__nv_bfloat16*>(a.out) +
                         grow * 2 * F + ti.out_col;
    __nv_bfloat16* hout = reinterpret_cast<__nv_bfloat16*>(a.out2) +
                          grow * F + ti.out_col;
#pragma unroll 1
    for (int c = 32 * half; c < 128; c += 64) {
      float g[32], u[32];
      tmem_ld32(tmem_row + c, g);
      tmem_ld32(tmem_row + 128 + c, u);
      if (valid) {
        float d[32], dg[32], du[32], h[32];
#pragma unroll
        for (int i = 0; i < 32; i += 8)
          Vec16<__nv_bfloat16>::to_f32(ld_nc_v4(dh + c + i), d + i);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float sg = 1.0f / (1.0f + __expf(-g[i]));
          const float sl = g[i] * sg;
          du[i] = d[i] * sl;
          dg[i] = d[i] * u[i] * sg * (1.0f + g[i] * (1.0f - sg));
          h[i] = sl * u[i];
        }
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          st_v4(dgu + c + i, Vec16<__nv_bfloat16>::from_f32(dg + i));
          st_v4(dgu + F + c + i, Vec16<__nv_bfloat16>::from_f32(du + i));
          st_v4(hout + c + i, Vec16<__nv_bfloat16>::from_f32(h + i));
        }
      }
    }
  } else if (MODE == kRDX) {
    // dx += acc in place (bf16): each element is read and written by this
    // thread only
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) +
                         grow * a.out_ld + ti.out_col;
#pragma unroll 1
    for (int c = 32 * half; c < 256; c += 64) {
      float v[32];
      tmem_ld32(tmem_row + c, v);
      if (valid && ti.out_col + c < a.out_cols) {
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          float o[8];
          Vec16<__nv_bfloat16>::to_f32(
              *reinterpret_cast<const uint4*>(out + c + i), o);
#pragma unroll
          for (int q = 0; q < 8; ++q) o[q] += v[i + q];
          st_v4(out + c + i, Vec16<__nv_bfloat16>::from_f32(o));
        }
      }
    }
  } else {
    // kDown, kDH, kDX: 256 bf16 columns
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) +
                         grow * a.out_ld + ti.out_col;
#pragma unroll 1
    for (int c = 32 * half; c < 256; c += 64) {
      float v[32];
      tmem_ld32(tmem_row + c, v);
      if (valid && ti.out_col + c < a.out_cols) {
#pragma unroll
        for (int i = 0; i < 32; i += 8)
          st_v4(out + c + i, Vec16<__nv_bfloat16>::from_f32(v + i));
      }
    }
  }
}

__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity,
                                                uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    umma_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte-swizzled tiles
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* tiles = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  const uint32_t b_tile_bytes = static_cast<uint32_t>(a.BN) * kBK * 2;
  uint8_t* a_tiles = tiles;
  uint8_t* b_tiles = tiles + a.stages * kATileBytes;
  GemmShared& sh = *reinterpret_cast<GemmShared*>(
      b_tiles + static_cast<size_t>(a.stages) * b_tile_bytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sh.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.tfull[i], 1);
      mbar_init(&sh.tempty[i], kEpiWarps);
      for (int q = 0; q < 4; ++q) mbar_init(&sh.xfull[i][q], 1);
    }
    mbar_init(&sh.drain, 1);
    sh.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  // tile prefix over experts (grouped modes)
  if (ModeInfo<MODE>::wgrad) {
    if (warp == 2) {
      // every expert segment must start on a 64-row boundary (the K blocks
      // of one expert never reach into the next)
      bool aligned = true;
      for (int e = lane; e <= a.groups; e += 32)
        aligned = aligned && (__ldg(a.offsets + e) & 63) == 0;
      aligned = __all_sync(0xffffffffu, aligned);
      if (lane == 0) {
        sh.total_tiles = aligned ? a.groups * a.m_tiles * a.n_tiles : 0;
        if (!aligned) set_status(a.status, MOE_ERR_INVALID);
      }
    }
  } else if (ModeInfo<MODE>::grouped_m) {
    if (warp == 2) {
      int run = 0;
      for (int base = 0; base < a.groups; base += 32) {
        const int e = base + lane;
        int tiles_e = 0;
        if (e < a.groups) {
          const int cnt = __ldg(a.offsets + e + 1) - __ldg(a.offsets + e);
          tiles_e = (max(cnt, 0) + kBM - 1) / kBM * a.n_tiles;
        }
        int incl = tiles_e;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += v;
        }
        if (e < a.groups) sh.prefix[e] = run + incl - tiles_e;
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        sh.prefix[a.groups] = run;
        sh.total_tiles = run;
      }
    }
  } else if (threadIdx.x == 64) {
    const int m_tiles = (a.M + kBM - 1) / kBM;
    sh.total_tiles = MODE == kRDX   ? m_tiles * a.n_tiles
                     : MODE == kRDW ? m_tiles * a.n_tiles * a.splits
                                    : m_tiles * a.splits;
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int total = sh.total_tiles;
  const uint32_t tmem_base = sh.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      const uint32_t tx = kATileBytes + b_tile_bytes;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileInfo ti = decode_tile<MODE>(a, sh, t);
        for (int kb = ti.kb_begin; kb < ti.kb_end; ++kb) {
          if (!mbar_wait(&sh.empty[stage], phase ^ 1, abort_flag,
                         a.wait_limit_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sh.full[stage], tx);
          uint8_t* sa = a_tiles + stage * kATileBytes;
          uint8_t* sb = b_tiles + static_cast<size_t>(stage) * b_tile_bytes;
          if (ModeInfo<MODE>::a_mn) {
            // two 64-wide MN boxes of 64 K (token) rows; kRDW takes the hi
            // or lo half of dL2 for even or odd K blocks
            const int acol = MODE == kRDW ? ti.b_row + (kb & 1) * a.E : ti.b_row;
            const int arow = MODE == kRDW ? (kb >> 1) * kBK : kb * kBK;
            tma_load_2d(sa, &tmA, &sh.full[stage], acol, arow);
            tma_load_2d(sa + 8192, &tmA, &sh.full[stage], acol + 64, arow);
          } else {
            tma_load_2d(sa, &tmA, &sh.full[stage], kb * kBK, ti.a_row);
          }
          if (ModeInfo<MODE>::gate_up) {
            tma_load_2d(sb, &tmB, &sh.full[stage], kb * kBK, ti.b_row);
            tma_load_2d(sb + 128 * 128, &tmB, &sh.full[stage], kb * kBK,
                        ti.b_row2);
          } else if (ModeInfo<MODE>::b_mn) {
            // four 64-wide MN boxes; K rows start at the expert's first K
            // row in B (dgrad) or at the token row itself (wgrad)
            const int krow =
                MODE == kRDX   ? (kb * kBK) % a.E
                : MODE == kRDW ? (kb >> 1) * kBK
                               : (ModeInfo<MODE>::wgrad ? 0 : ti.b_row) + kb * kBK;
#pragma unroll
            for (int i = 0; i < 4; ++i)
              tma_load_2d(sb + i * 8192, &tmB, &sh.full[stage],
                          ti.out_col + 64 * i, krow);
          } else {
            tma_load_2d(sb, &tmB, &sh.full[stage], kb * kBK, ti.b_row);
          }
          ++issued;
          if (++stage == a.stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // drain the copies still in flight before the CTA may exit
        const int n = min(issued, a.stages);
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < n; ++i) {
          if (s == 0) {
            s = a.stages - 1;
            ph ^= 1;
          } else {
            --s;
          }
          mbar_wait_drain(&sh.full[s], ph, 50000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      const uint32_t idesc = umma_idesc_bf16_major(
          kBM, a.BN, ModeInfo<MODE>::a_mn, ModeInfo<MODE>::b_mn);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const TileInfo ti = decode_tile<MODE>(a, sh, t);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait(&sh.tempty[acc], acc_phase ^ 1, abort_flag,
                       a.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * a.BN;
        for (int kb = ti.kb_begin; kb < ti.kb_end; ++kb) {
          if (!mbar_wait(&sh.full[stage], phase, abort_flag,
                         a.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(a_tiles + stage * kATileBytes);
          const uint32_t sb =
              smem_u32(b_tiles + static_cast<size_t>(stage) * b_tile_bytes);
          // one K step of 16: +32 bytes along a K-major row (+2 in the
          // >>4 address field), or +16 rows of 128 bytes MN-major (+128)
          constexpr uint32_t a_step = ModeInfo<MODE>::a_mn ? 128u : 2u;
          constexpr uint32_t b_step = ModeInfo<MODE>::b_mn ? 128u : 2u;
          const uint64_t adesc = ModeInfo<MODE>::a_mn ? umma_desc_mn_sw128(sa)
                                                      : umma_desc_sw128(sa);
          const uint64_t bdesc = ModeInfo<MODE>::b_mn ? umma_desc_mn_sw128(sb)
                                                      : umma_desc_sw128(sb);
          if (MODE == kRoute || ti.swap_n == 0) {
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k) {
              umma_bf16(d_tmem, adesc + a_step * k, bdesc + b_step * k, idesc,
                        (kb > ti.kb_begin || k > 0) ? 1u : 0u);
            }
          } else {
            // swapped tail: each 128-row half of the weight tile is an A
            // operand, the first swap_n token rows are the B operand
            const uint32_t idesc_s = umma_idesc_bf16(kBM, ti.swap_n);
            const uint64_t bdesc_hi = umma_desc_sw128(sb + 128 * 128);
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k) {
              const uint32_t acc_in = (kb > ti.kb_begin || k > 0) ? 1u : 0u;
              umma_bf16(d_tmem, bdesc + 2 * k, adesc + 2 * k, idesc_s, acc_in);
              umma_bf16(d_tmem + 128, bdesc_hi + 2 * k, adesc + 2 * k, idesc_s,
                        acc_in);
            }
          }
          umma_commit(&sh.empty[stage]);
          if (++stage == a.stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&sh.tfull[acc]);
      }
      if (!ok) {
        umma_commit(&sh.drain);
        mbar_wait_drain(&sh.drain, 0, 50000000ull);
      }
    }
  } else {
    // ---------------- epilogue warps 2..9
    const int quarter = warp & 3;          // TMEM lanes 32*quarter ..
    const int half = (warp - 2) >> 2;      // alternate column chunks
    const int r = quarter * 32 + lane;     // tile row of this thread
    float* stage = reinterpret_cast<float*>(
                       reinterpret_cast<uint8_t*>(&sh) +
                       ((sizeof(GemmShared) + 15) & ~size_t(15))) +
                   (warp - 2) * 32 * kStageLd;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const TileInfo ti = decode_tile<MODE>(a, sh, t);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      bool ok = true;
      if (lane == 0)
        ok = mbar_wait(&sh.tfull[acc], acc_phase, abort_flag, a.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const uint32_t tmem_row =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
          acc * a.BN;
      epilogue_row<MODE>(a, ti, tmem_row, r, half, stage, acc,
                         &sh.xfull[0][0], acc_phase, abort_flag);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.tempty[acc]);
    }
  }

  __syncwarp();   // reconverge the single-lane producer / MMA roles
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, a.tmem_cols);
  }
  if (threadIdx.x == 0 && sh.abort) set_status(a.status, MOE_ERR_TIMEOUT);
}

// Shared-memory bytes of one launch (tiles + control block + alignment slack
// + the weight-gradient staging tiles when `staging`).
inline size_t umma_gemm_smem_bytes(int BN, int stages, bool staging = false) {
  return 1024 + static_cast<size_t>(stages) * (kATileBytes + BN * kBK * 2) +
         ((sizeof(GemmShared) + 15) & ~size_t(15)) +
         (staging ? kStageBytes : 0);
}

// One persistent launch (one CTA per SM) of a grouped or backward mode.
template <int MODE>
inline moe_status launch_umma(const CUtensorMap& tmA, const CUtensorMap& tmB,
                              const GemmArgs& g, cudaStream_t stream,
                              int num_sms) {
  static std::atomic<uint64_t> attr_done{0};
  if (!set_smem_limit_once(reinterpret_cast<const void*>(umma_gemm_kernel<MODE>),
                           227 * 1024, &attr_done))
    return MOE_ERR_CUDA;
  const size_t smem =
      umma_gemm_smem_bytes(g.BN, g.stages, ModeInfo<MODE>::staged);
  umma_gemm_kernel<MODE><<<num_sms, kGemmThreads, smem, stream>>>(tmA, tmB, g);
  return launch_status();
}

}  // namespace moe
