// Grouped SwiGLU FFN on pairs of SMs: the up and the down projection in one
// persistent launch of 2-CTA clusters, every MMA a 256-row tcgen05 MMA that
// the pair shares (cta_group::2) ("Expert Parallelism in LLMs", The
// Execution Pipeline, step 4: Expert_e(h) = W2_e (SiLU(W1_e h) * W3_e h)
// over each expert's rows).
//
// Why pairs: on one SM a 128 x 256 tile takes 48 KB of operands per 64-deep
// K block.  In a pair each SM holds its 128 token rows of A and its half of
// B (128 weight rows): 32 KB per K block for the same MMA work per SM, so
// the same shared memory holds 6 stages instead of 4 and the ring covers
// half as much again of the weight stream's latency.
//
// Row blocks are 256 token rows of one expert.  An expert with c rows has
// q = floor(c / 256) full blocks and r = c mod 256 rows left:
//   r > kPairSwapMax       one more block of 256 rows, the rows past c
//                          computed and not stored;
//   0 < r <= kPairSwapMax  a "swapped" tail block: the weights are the
//                          256-row operand (128 features per SM) and the r
//                          token rows the N side (r rounded up to 16, N/2
//                          rows per SM), so a few rows do not cost a whole
//                          256-row MMA; TMEM then holds [feature, token] and
//                          the epilogue writes transposed.
// Tiles:
//   up, normal     256 rows x (128 gate + 128 up features): SM 0 loads the
//                  gate rows, SM 1 the up rows, so each SM's TMEM row holds
//                  gate and up side by side and the epilogue writes
//                  H = SiLU(gate) * up for its 128 rows;
//   up, swapped    256 features x N tokens, gate and up in two MMAs that
//                  share the token tile;
//   down, normal   256 rows x 256 output features (A = H, B = W2);
//   down, swapped  256 output features x N tokens.
// Within an expert the tiles of one weight tile are adjacent: per 256
// gate/up features the normal blocks' two 128-feature tiles (blocks
// fastest), then the tail's tile; per 256 output features the normal
// blocks, then the tail.
//
// Scheduling: the pairs are persistent and claim tiles in list order from
// one global ticket, so the tiles in flight are always a contiguous window
// of the list and the pairs that share a weight tile read it from L2 at
// about the same time, whatever the tiles' lengths.  The leader SM's
// producer claims the next tile one tile ahead and publishes each claimed
// tile id through a small queue in both SMs' shared memory; the peer's
// producer, the MMA issuer and the epilogue warps of both SMs read it there
// and release the slot on the leader's "qempty" barrier.
//
// Cross-tile dependency: a down tile reads H of its row block, written by
// every up tile of that block.  Each up tile's 16 epilogue warps (8 per SM)
// add 1 to the block's counter with release semantics after their H stores;
// both producers of a down tile wait (bounded) for 16 x (up tiles per
// block), then issue the proxy fence and the TMA loads of H.  All up tiles
// precede all down tiles in the list, tiles are claimed in list order and
// up tiles wait for nothing, so every claimed down tile depends only on up
// tiles already claimed by running pairs (a pair claims one tile ahead, and
// a tile after a down tile is a down tile): no wait can be part of a cycle,
// and the launch needs no co-residency guarantee.
//
// Per SM: warp 0 is the TMA producer (both SMs load their own halves; the
// leader's "full" barrier counts the bytes of both), warp 1 of the leader
// issues the MMAs and commits to the "empty" and "tfull" barriers of both
// SMs at once, warps 2-9 of both SMs run the epilogue and report to the
// leader's "tempty" barrier.  Every wait is bounded; on expiry the SM stops
// issuing, drains its copies and MMAs and reports MOE_ERR_TIMEOUT.
#pragma once

#include "umma_ffn.cuh"

namespace moe {

constexpr int kPairRows = 256;                 // M of a pair MMA
constexpr int kPairStages = 6;
constexpr uint32_t kPairHalfBytes = 128 * kBK * 2;       // 16 KB: 128 rows
constexpr uint32_t kPairStageBytes = 2 * kPairHalfBytes;
constexpr int kPairSwapMax = 64;               // tails up to here run swapped
// a swapped tail's token half per stage, in a ring of its own after the A/B
// ring
constexpr uint32_t kPairTokBytes = (kPairSwapMax / 2) * kBK * 2;
constexpr int kPairMaxGroups = 256;            // experts the pair path takes
constexpr int kTileQ = 4;                       // tile-id queue slots
// readers of a queue slot: the peer's producer, the MMA issuer and the
// epilogue warps of both SMs
constexpr int kTileQReaders = 2 + 2 * kEpiWarps;

struct PairFfnArgs {
  int32_t E, D, F;
  int32_t kb_up;          // D / 64
  int32_t kb_dn;          // F / 64
  int32_t n_up;           // normal up tiles per row block: F / 128
  int32_t S;              // swapped up tiles per tail block: F / 256
  int32_t n_dn;           // down tiles per row block: ceil(D / 256)
  const int32_t* offsets; // [E + 1] expert row offsets
  int32_t max_rows;       // rows of Xp, H and Yp
  __nv_bfloat16* h;       // [max_rows, F]
  __nv_bfloat16* yp;      // [max_rows, D]
  uint32_t* ready;        // per row block, zeroed before the launch
  uint32_t* ticket;       // next tile to claim, zeroed before the launch
  int32_t ready_cap;
  int32_t* status;
  uint64_t wait_limit_ns;
};

struct PairShared {
  uint64_t full[kPairStages];
  uint64_t empty[kPairStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t qfull[kTileQ];              // tile id written into the slot
  uint64_t qempty[kTileQ];             // leader: every reader took it
  uint64_t drain;
  int32_t qtile[kTileQ];
  uint32_t tmem_base;
  int32_t abort;
  int32_t up_total;
  int32_t total;
  int32_t up_prefix[kPairMaxGroups + 1];   // first up tile of each expert
  int32_t dn_prefix[kPairMaxGroups + 1];   // first down tile of each expert
  int32_t blk_prefix[kPairMaxGroups + 1];  // first row block of each expert
};

struct PairTile {
  int32_t down;      // 0: up tile, 1: down tile
  int32_t swapped;   // tail block of <= kPairSwapMax rows, operands swapped
  int32_t e;
  int32_t row0;      // first token row of the block
  int32_t rows;      // valid token rows of the block (1..256)
  int32_t n_mma;     // MMA N: 256, or the swapped tail rounded up to 16
  int32_t col0;      // up: first H feature; down: first output feature
  int32_t blk;       // row block (ready counter)
};

// Normal blocks q and swapped tail (0 or 1) of an expert with c rows.
__device__ __forceinline__ void pair_blocks(int c, int& q, int& tail) {
  const int r = c & (kPairRows - 1);
  tail = (r > 0 && r <= kPairSwapMax) ? 1 : 0;
  q = c <= 0 ? 0 : (tail ? c / kPairRows : (c + kPairRows - 1) / kPairRows);
}

__device__ __forceinline__ int pair_find(const int32_t* prefix, int groups,
                                         int t) {
  int lo = 0, hi = groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Tile t: every up tile (expert-major; per 256 gate/up features the normal
// blocks' two 128-feature tiles, blocks fastest, then the tail's tile), then
// every down tile (expert-major; per 256 output features the normal blocks,
// then the tail).
__device__ __forceinline__ PairTile pair_decode(const PairFfnArgs& a,
                                                const PairShared& sh, int t) {
  PairTile p;
  p.down = t >= sh.up_total ? 1 : 0;
  const int local_all = p.down ? t - sh.up_total : t;
  const int32_t* prefix = p.down ? sh.dn_prefix : sh.up_prefix;
  const int e = pair_find(prefix, a.E, local_all);
  p.e = e;
  const int base = __ldg(a.offsets + e);
  const int c = __ldg(a.offsets + e + 1) - base;
  int q, tail;
  pair_blocks(c, q, tail);
  const int local = local_all - prefix[e];
  int m;
  if (!p.down) {
    const int per_s = 2 * q + tail;
    const int s = local / per_s;
    const int w = local - s * per_s;
    p.swapped = w >= 2 * q ? 1 : 0;
    if (p.swapped) {
      m = q;
      p.col0 = s * 256;
    } else {
      const int half = w >= q ? 1 : 0;
      m = w - half * q;
      p.col0 = s * 256 + half * 128;
    }
  } else {
    const int per_n = q + tail;
    const int n = local / per_n;
    m = local - n * per_n;
    p.swapped = m >= q ? 1 : 0;
    p.col0 = n * 256;
  }
  p.row0 = base + m * kPairRows;
  p.rows = min(kPairRows, c - m * kPairRows);
  p.n_mma = p.swapped ? (p.rows + 15) & ~15 : kPairRows;
  p.blk = sh.blk_prefix[e] + m;
  return p;
}

// Epilogue warps (of both SMs) that report each up tile, times the up tiles
// of the block: 2 per 256 features for a normal block, 1 for a swapped tail.
__device__ __forceinline__ uint32_t pair_ready_target(const PairFfnArgs& a,
                                                      const PairTile& p) {
  return static_cast<uint32_t>(2 * kEpiWarps * (p.swapped ? a.S : a.n_up));
}

// Bytes one SM loads per K block of a tile.
__device__ __forceinline__ uint32_t pair_stage_tx(const PairTile& p) {
  if (!p.swapped) return 2 * kPairHalfBytes;
  return (p.down ? 1u : 2u) * kPairHalfBytes + kPairTokBytes;
}

// Epilogue of one pair tile on this SM (`cta` 0 or 1) for the thread owning
// TMEM lane `r` of the accumulator at `tmem_row`; `half` picks alternate
// column chunks.  TMEM lane r is token row row0 + 128 cta + r.
__device__ __forceinline__ void pair_epilogue(const PairFfnArgs& a,
                                              const PairTile& p, int cta,
                                              uint32_t tmem_row, int r,
                                              int half) {
  const int row = 128 * cta + r;
  const int64_t grow = static_cast<int64_t>(p.row0) + row;
  const bool valid = row < p.rows && grow < a.max_rows;
  if (!p.down) {
    __nv_bfloat16* out = a.h + grow * a.F + p.col0;
#pragma unroll 1
    for (int c = 32 * half; c < 128; c += 64) {
      float g[32], u[32];
      tmem_ld32(tmem_row + c, g);
      tmem_ld32(tmem_row + 128 + c, u);
      if (valid) {
        float hv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) hv[i] = silu_f32(g[i]) * u[i];
#pragma unroll
        for (int i = 0; i < 32; i += 8)
          st_v4(out + c + i, Vec16<__nv_bfloat16>::from_f32(hv + i));
      }
    }
  } else {
    const int col0 = p.col0;
    __nv_bfloat16* out = a.yp + grow * a.D + col0;
#pragma unroll 1
    for (int c = 32 * half; c < 256; c += 64) {
      float v[32];
      tmem_ld32(tmem_row + c, v);
      if (valid && col0 + c < a.D) {
#pragma unroll
        for (int i = 0; i < 32; i += 8)
          st_v4(out + c + i, Vec16<__nv_bfloat16>::from_f32(v + i));
      }
    }
  }
}

// Reader side of the tile queue: the id in slot i % kTileQ once the leader
// has written it (the i-th tile this pair runs), the slot then released on
// the leader's barrier; -1 when the wait expired.
__device__ __forceinline__ int pair_queue_take(PairShared& sh, int i,
                                               uint32_t leader_qempty0,
                                               volatile int* abort_flag,
                                               uint64_t limit_ns) {
  const int slot = i % kTileQ;
  const uint32_t use = static_cast<uint32_t>(i / kTileQ);
  if (!mbar_wait_cluster(&sh.qfull[slot], use & 1, abort_flag, limit_ns))
    return -1;
  const int t = *reinterpret_cast<volatile int32_t*>(&sh.qtile[slot]);
  mbar_arrive_cluster(leader_qempty0 + 8u * slot);
  return t;
}

// Epilogue of a swapped tail tile on this SM: TMEM lane r is feature
// col0 + 128 cta + r, column j token row row0 + j.  Kept out of line so that
// the normal tiles' epilogue code stays as it is.
__device__ __noinline__ void pair_epilogue_swapped(const PairFfnArgs& a,
                                                   const PairTile& p, int cta,
                                                   uint32_t tmem_row, int r,
                                                   int half) {
  const int f = p.col0 + 128 * cta + r;
  const int rows = min(p.rows, a.max_rows - p.row0);
  if (!p.down) {
    const bool ok = f < a.F;
    __nv_bfloat16* out = a.h + static_cast<int64_t>(p.row0) * a.F + f;
#pragma unroll 1
    for (int c = 16 * half; c < p.n_mma; c += 32) {
      float g[16], u[16];
      tmem_ld16(tmem_row + c, g);
      tmem_ld16(tmem_row + 128 + c, u);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int j = c + i;
        if (ok && j < rows)
          out[static_cast<int64_t>(j) * a.F] =
              __float2bfloat16_rn(silu_f32(g[i]) * u[i]);
      }
    }
  } else {
    const bool ok = f < a.D;
    __nv_bfloat16* out = a.yp + static_cast<int64_t>(p.row0) * a.D + f;
#pragma unroll 1
    for (int c = 16 * half; c < p.n_mma; c += 32) {
      float v[16];
      tmem_ld16(tmem_row + c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int j = c + i;
        if (ok && j < rows)
          out[static_cast<int64_t>(j) * a.D] = __float2bfloat16_rn(v[i]);
      }
    }
  }
}

inline size_t umma_ffn_pair_smem_bytes() {
  return 1024 + static_cast<size_t>(kPairStages) * (kPairStageBytes + kPairTokBytes) +
         ((sizeof(PairShared) + 15) & ~size_t(15));
}

// tm_xp / tm_h: 128-row boxes over the token rows (normal tiles);
// tm_xp_t / tm_h_t: kPairSwapMax / 2-row boxes (a swapped tail's token
// half); tm_w13 / tm_w2: 128-row boxes over [E * 2F] and [E * D] rows.
__global__ void __launch_bounds__(kGemmThreads, 1)
    umma_ffn_pair_kernel(const __grid_constant__ CUtensorMap tm_xp,
                         const __grid_constant__ CUtensorMap tm_w13,
                         const __grid_constant__ CUtensorMap tm_h,
                         const __grid_constant__ CUtensorMap tm_w2,
                         const __grid_constant__ CUtensorMap tm_xp_t,
                         const __grid_constant__ CUtensorMap tm_h_t,
                         const PairFfnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* stages = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* tok = stages + static_cast<size_t>(kPairStages) * kPairStageBytes;
  PairShared& sh = *reinterpret_cast<PairShared*>(
      tok + static_cast<size_t>(kPairStages) * kPairTokBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = static_cast<int>(cluster_ctarank());
  const int pair = blockIdx.x >> 1;
  volatile int* abort_flag = &sh.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.tfull[i], 1);
      mbar_init(&sh.tempty[i], 2 * kEpiWarps);
    }
    for (int i = 0; i < kTileQ; ++i) {
      mbar_init(&sh.qfull[i], 1);
      mbar_init(&sh.qempty[i], kTileQReaders);
    }
    mbar_init(&sh.drain, 1);
    sh.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_xp);
    tma_prefetch_desc(&tm_w13);
    tma_prefetch_desc(&tm_h);
    tma_prefetch_desc(&tm_w2);
    tma_prefetch_desc(&tm_xp_t);
    tma_prefetch_desc(&tm_h_t);
  }
  if (warp == 2) {
    // per-expert tile and row-block prefixes (both SMs compute the same)
    int run_up = 0, run_dn = 0, run_blk = 0;
    for (int base = 0; base < a.E; base += 32) {
      const int e = base + lane;
      int up_e = 0, dn_e = 0, blk_e = 0;
      if (e < a.E) {
        const int c = max(__ldg(a.offsets + e + 1) - __ldg(a.offsets + e), 0);
        int q, tail;
        pair_blocks(c, q, tail);
        up_e = a.S * (2 * q + tail);
        dn_e = a.n_dn * (q + tail);
        blk_e = q + tail;
      }
      int iu = up_e, id = dn_e, ib = blk_e;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int vu = __shfl_up_sync(0xffffffffu, iu, d);
        const int vd = __shfl_up_sync(0xffffffffu, id, d);
        const int vb = __shfl_up_sync(0xffffffffu, ib, d);
        if (lane >= d) {
          iu += vu;
          id += vd;
          ib += vb;
        }
      }
      if (e < a.E) {
        sh.up_prefix[e] = run_up + iu - up_e;
        sh.dn_prefix[e] = run_dn + id - dn_e;
        sh.blk_prefix[e] = run_blk + ib - blk_e;
      }
      run_up += __shfl_sync(0xffffffffu, iu, 31);
      run_dn += __shfl_sync(0xffffffffu, id, 31);
      run_blk += __shfl_sync(0xffffffffu, ib, 31);
    }
    if (lane == 0) {
      sh.up_prefix[a.E] = run_up;
      sh.dn_prefix[a.E] = run_dn;
      sh.blk_prefix[a.E] = run_blk;
      // more row blocks than counters means the offsets overrun the rows
      // the buffers were sized for: run nothing
      const bool fits = run_blk <= a.ready_cap;
      sh.up_total = fits ? run_up : 0;
      sh.total = fits ? run_up + run_dn : 0;
      if (!fits && cta == 0 && pair == 0) set_status(a.status, MOE_ERR_INVALID);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(&sh.tmem_base, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // no TMA or commit from the peer may reach this SM's barriers before they
  // are initialised
  cluster_sync_all();
  tc_fence_after();

  const int total = sh.total;
  const uint32_t tmem_base = sh.tmem_base;
  const uint32_t leader_qempty0 = cluster_addr(&sh.qempty[0], 0);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both SMs)
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      // the leader claims tiles one ahead and publishes each to the queue;
      // the peer takes them from it
      uint32_t next = cta == 0 ? atomicAdd(a.ticket, 1u) : 0u;
      for (int qi = 0; ok; ++qi) {
        int t;
        if (cta == 0) {
          t = static_cast<int>(next);
          const int slot = qi % kTileQ;
          const uint32_t use = static_cast<uint32_t>(qi / kTileQ);
          if (!mbar_wait_cluster(&sh.qempty[slot], (use & 1) ^ 1, abort_flag,
                                 a.wait_limit_ns)) {
            ok = false;
            break;
          }
          sh.qtile[slot] = t;
          st_cluster_u32(cluster_addr(&sh.qtile[slot], 1),
                         static_cast<uint32_t>(t));
          mbar_arrive(&sh.qfull[slot]);
          mbar_arrive_cluster(cluster_addr(&sh.qfull[slot], 1));
          if (t < total) next = atomicAdd(a.ticket, 1u);
        } else {
          t = pair_queue_take(sh, qi, leader_qempty0, abort_flag,
                              a.wait_limit_ns);
          if (t < 0) {
            ok = false;
            break;
          }
        }
        if (t >= total) break;
        const PairTile p = pair_decode(a, sh, t);
        if (p.down) {
          // H of this row block must be complete before TMA reads it
          if (!ffn_wait_ready(a.ready + p.blk, pair_ready_target(a, p),
                              abort_flag, a.wait_limit_ns)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        const int kb_end = p.down ? a.kb_dn : a.kb_up;
        if (p.swapped) {
          // this SM's 128 weight rows (gate and up rows for the up
          // projection) and its N/2 token rows
          const int w_row = p.down ? p.e * a.D + p.col0 + 128 * cta
                                   : p.e * 2 * a.F + p.col0 + 128 * cta;
          const int t_row = p.row0 + (p.n_mma >> 1) * cta;
          const CUtensorMap* mw = p.down ? &tm_w2 : &tm_w13;
          const CUtensorMap* mt = p.down ? &tm_h_t : &tm_xp_t;
          const uint32_t tx = pair_stage_tx(p);
          for (int kb = 0; kb < kb_end; ++kb) {
            if (!mbar_wait(&sh.empty[stage], phase ^ 1, abort_flag,
                           a.wait_limit_ns)) {
              ok = false;
              break;
            }
            if (cta == 0) mbar_arrive_expect_tx(&sh.full[stage], 2 * tx);
            const uint32_t bar = cluster_addr(&sh.full[stage], 0);
            uint8_t* sx = stages + static_cast<size_t>(stage) * kPairStageBytes;
            tma_load_2d_pair(sx, mw, bar, kb * kBK, w_row);
            if (!p.down)
              tma_load_2d_pair(sx + kPairHalfBytes, mw, bar, kb * kBK,
                               w_row + a.F);
            tma_load_2d_pair(tok + static_cast<size_t>(stage) * kPairTokBytes,
                             mt, bar, kb * kBK, t_row);
            ++issued;
            if (++stage == kPairStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          continue;
        }
        const int a_row = p.row0 + 128 * cta;
        const int b_row = p.down ? p.e * a.D + p.col0 + 128 * cta
                                 : p.e * 2 * a.F + cta * a.F + p.col0;
        const CUtensorMap* ma = p.down ? &tm_h : &tm_xp;
        const CUtensorMap* mb = p.down ? &tm_w2 : &tm_w13;
        for (int kb = 0; kb < kb_end; ++kb) {
          if (!mbar_wait(&sh.empty[stage], phase ^ 1, abort_flag,
                         a.wait_limit_ns)) {
            ok = false;
            break;
          }
          if (cta == 0)
            mbar_arrive_expect_tx(&sh.full[stage], 2 * kPairStageBytes);
          const uint32_t bar = cluster_addr(&sh.full[stage], 0);
          uint8_t* sx = stages + static_cast<size_t>(stage) * kPairStageBytes;
          tma_load_2d_pair(sx, ma, bar, kb * kBK, a_row);
          tma_load_2d_pair(sx + kPairHalfBytes, mb, bar, kb * kBK, b_row);
          ++issued;
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok && cta == 0) {
        // drain the copies still in flight before the CTA may exit
        const int n = min(issued, kPairStages);
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < n; ++i) {
          if (s == 0) {
            s = kPairStages - 1;
            ph ^= 1;
          } else {
            --s;
          }
          mbar_wait_drain(&sh.full[s], ph, 50000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && cta == 0) {
      // ---------------- MMA issuer (the leader SM, for both)
      const uint32_t idesc = umma_idesc_bf16(kPairRows, 256);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int qi = 0; ok; ++qi, ++it) {
        const int t = pair_queue_take(sh, qi, leader_qempty0, abort_flag,
                                      a.wait_limit_ns);
        if (t < 0) {
          ok = false;
          break;
        }
        if (t >= total) break;
        const PairTile p = pair_decode(a, sh, t);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!mbar_wait_cluster(&sh.tempty[acc], acc_phase ^ 1, abort_flag,
                               a.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * 256;
        const int kb_end = p.down ? a.kb_dn : a.kb_up;
        if (p.swapped) {
          // [features x tokens]: the gate (or W2) rows, and for the up
          // projection the up rows into columns 128.., against the tokens
          const uint32_t idesc_s = umma_idesc_bf16(kPairRows, p.n_mma);
          for (int kb = 0; kb < kb_end; ++kb) {
            if (!mbar_wait_cluster(&sh.full[stage], phase, abort_flag,
                                   a.wait_limit_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sx =
                smem_u32(stages + static_cast<size_t>(stage) * kPairStageBytes);
            const uint64_t d0 = umma_desc_sw128(sx);
            const uint64_t d1 = umma_desc_sw128(sx + kPairHalfBytes);
            const uint64_t dt = umma_desc_sw128(
                smem_u32(tok + static_cast<size_t>(stage) * kPairTokBytes));
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k) {
              const uint32_t acc_in = (kb > 0 || k > 0) ? 1u : 0u;
              umma_bf16_pair(d_tmem, d0 + 2 * k, dt + 2 * k, idesc_s, acc_in);
              if (!p.down)
                umma_bf16_pair(d_tmem + 128, d1 + 2 * k, dt + 2 * k, idesc_s,
                               acc_in);
            }
            umma_commit_pair(&sh.empty[stage]);
            if (++stage == kPairStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          umma_commit_pair(&sh.tfull[acc]);
          continue;
        }
        for (int kb = 0; kb < kb_end; ++kb) {
          if (!mbar_wait_cluster(&sh.full[stage], phase, abort_flag,
                                 a.wait_limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sx =
              smem_u32(stages + static_cast<size_t>(stage) * kPairStageBytes);
          const uint64_t da = umma_desc_sw128(sx);
          const uint64_t db = umma_desc_sw128(sx + kPairHalfBytes);
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k)
            umma_bf16_pair(d_tmem, da + 2 * k, db + 2 * k, idesc,
                           (kb > 0 || k > 0) ? 1u : 0u);
          umma_commit_pair(&sh.empty[stage]);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit_pair(&sh.tfull[acc]);
      }
      if (!ok) {
        umma_commit_pair(&sh.drain);
        mbar_wait_drain(&sh.drain, 0, 50000000ull);
      }
    }
  } else {
    // ---------------- epilogue warps 2..9 (both SMs)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t leader_tempty0 = cluster_addr(&sh.tempty[0], 0);
    const uint32_t leader_tempty1 = cluster_addr(&sh.tempty[1], 0);
    int it = 0;
    for (int qi = 0;; ++qi, ++it) {
      int t = 0;
      if (lane == 0)
        t = pair_queue_take(sh, qi, leader_qempty0, abort_flag,
                            a.wait_limit_ns);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t < 0 || t >= total) break;
      const PairTile p = pair_decode(a, sh, t);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      bool ok = true;
      if (lane == 0)
        ok = mbar_wait_cluster(&sh.tfull[acc], acc_phase, abort_flag,
                               a.wait_limit_ns);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const uint32_t tmem_row =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * 256;
      if (p.swapped)
        pair_epilogue_swapped(a, p, cta, tmem_row, r, half);
      else
        pair_epilogue(a, p, cta, tmem_row, r, half);
      if (!p.down) {
        // this warp's part of the row block's H is written: count it
        __threadfence();
        __syncwarp();
        if (lane == 0) red_release_add_gpu(a.ready + p.blk, 1u);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0)
        mbar_arrive_cluster(acc ? leader_tempty1 : leader_tempty0);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // neither SM may leave while the other can still reach its shared memory
  // or TMEM
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
  if (threadIdx.x == 0 && sh.abort) set_status(a.status, MOE_ERR_TIMEOUT);
}

}  // namespace moe
