// Grouped SwiGLU FFN with the up and the down projection in one persistent
// launch ("Expert Parallelism in LLMs", The Execution Pipeline, step 4:
// Expert_e(h) = W2_e (SiLU(W1_e h) * W3_e h) over each expert's rows).
//
// The tile list is every up tile (kUp: H = SiLU(gate) * up for a 128-row
// block and 128 gate + 128 up columns) followed by every down tile (kDown:
// Yp for a 128-row block and 256 output columns), both over the same
// per-expert row blocks.  The CTAs walk it round-robin, as the two-launch
// path does, so an SM that runs out of up tiles starts down tiles while
// other SMs finish the up projection.
//
// A down tile reads the H rows of its row block, which all n_up up tiles
// of that block write.  Each of those tiles' 8 epilogue warps adds 1 to the
// block's counter with release semantics once its H stores are issued; the
// producer of a down tile waits (bounded) until the counter reaches
// 8 * n_up, then issues the proxy fence and the TMA loads of H.  Every up
// tile precedes every down tile in each CTA's order and up tiles wait for
// nothing, so the waits cannot form a cycle while all CTAs are resident
// (one per SM, grid = SM count).  A wait that expires stops the CTA like
// any other expired wait (MOE_ERR_TIMEOUT).
//
// Everything else -- the shared-memory ring, the MMAs, the swapped tail
// tiles, the epilogues -- is the grouped GEMM's (umma_gemm.cuh).
#pragma once

#include "umma_gemm.cuh"

namespace moe {

struct FfnArgs {
  GemmArgs up;          // kUp: A = Xp, B = W13, out = H
  GemmArgs dn;          // kDown: A = H, B = W2, out = Yp
  uint32_t* ready;      // per row block: up-tile epilogue warps done (zeroed)
  int32_t ready_cap;    // counters available
};

struct FfnTile {
  TileInfo ti;
  int down;             // 0: up tile, 1: down tile
  int rb;               // row block (for the ready counter)
};

// Tile t of the fused list.  sh.prefix[e] holds the row blocks of the
// experts before e; an expert's tiles run m-fastest within each phase.
__device__ __forceinline__ FfnTile ffn_decode(const FfnArgs& f,
                                              const GemmShared& sh, int t,
                                              int up_total) {
  FfnTile ft;
  ft.down = t >= up_total ? 1 : 0;
  const GemmArgs& a = ft.down ? f.dn : f.up;
  const int local_all = ft.down ? t - up_total : t;
  const int n_tiles = a.n_tiles;
  int lo = 0, hi = a.groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sh.prefix[mid] * n_tiles <= local_all) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int row0 = __ldg(a.offsets + e);
  const int cnt = __ldg(a.offsets + e + 1) - row0;
  const int m_tiles = (cnt + kBM - 1) / kBM;
  const int local = local_all - sh.prefix[e] * n_tiles;
  const int n = local / m_tiles;
  const int m = local - n * m_tiles;
  ft.rb = sh.prefix[e] + m;
  TileInfo& ti = ft.ti;
  ti.split = 0;
  ti.a_row = row0 + m * kBM;
  ti.rows = min(kBM, cnt - m * kBM);
  ti.swap_n = ti.rows <= kBM - 16 ? (ti.rows + 15) & ~15 : 0;
  ti.kb_begin = 0;
  ti.kb_end = a.k_blocks;
  if (!ft.down) {
    ti.b_row = e * a.b_rows_per_group + n * 128;
    ti.b_row2 = e * a.b_rows_per_group + a.F + n * 128;
    ti.out_col = n * 128;
  } else {
    ti.b_row = e * a.b_rows_per_group + n * 256;
    ti.b_row2 = 0;
    ti.out_col = n * 256;
  }
  return ft;
}

// Bounded wait of the producer for a row block's H: false when it expired
// (the abort flag is then set) or another thread aborted.
__device__ __forceinline__ bool ffn_wait_ready(const uint32_t* ready,
                                               uint32_t target,
                                               volatile int* abort_flag,
                                               uint64_t limit_ns) {
  if (ld_acquire_gpu(ready) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_gpu(ready) < target) {
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    umma_ffn_kernel(const __grid_constant__ CUtensorMap tm_xp,
                    const __grid_constant__ CUtensorMap tm_w13,
                    const __grid_constant__ CUtensorMap tm_h,
                    const __grid_constant__ CUtensorMap tm_w2,
                    const FfnArgs f) {
  extern __shared__ uint8_t smem_raw[];
  const GemmArgs& a = f.up;      // ring, TMEM and limits are the same
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
  }
  // row-block prefix over experts; the phase tile counts follow from it
  if (warp == 2) {
    int run = 0;
    for (int base = 0; base < a.groups; base += 32) {
      const int e = base + lane;
      int rb_e = 0;
      if (e < a.groups) {
        const int cnt = __ldg(a.offsets + e + 1) - __ldg(a.offsets + e);
        rb_e = (max(cnt, 0) + kBM - 1) / kBM;
      }
      int incl = rb_e;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      if (e < a.groups) sh.prefix[e] = run + incl - rb_e;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      sh.prefix[a.groups] = run;
      // row blocks; more than the counters cover means the offsets overrun
      // the rows the buffers were sized for: run nothing
      sh.total_tiles = run <= f.ready_cap ? run : 0;
      if (run > f.ready_cap) set_status(a.status, MOE_ERR_INVALID);
    }
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int row_blocks = sh.total_tiles;
  const int up_total = row_blocks * f.up.n_tiles;
  const int total = up_total + row_blocks * f.dn.n_tiles;
  const uint32_t tmem_base = sh.tmem_base;
  const uint32_t ready_target = static_cast<uint32_t>(kEpiWarps * f.up.n_tiles);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      const uint32_t tx = kATileBytes + b_tile_bytes;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const FfnTile ft = ffn_decode(f, sh, t, up_total);
        const TileInfo& ti = ft.ti;
        if (ft.down) {
          // H of this row block must be complete before TMA reads it
          if (!ffn_wait_ready(f.ready + ft.rb, ready_target, abort_flag,
                              a.wait_limit_ns)) {
            ok = false;
            break;
          }
          fence_proxy_async_global();
        }
        for (int kb = ti.kb_begin; kb < ti.kb_end; ++kb) {
          if (!mbar_wait(&sh.empty[stage], phase ^ 1, abort_flag,
                         a.wait_limit_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sh.full[stage], tx);
          uint8_t* sa = a_tiles + stage * kATileBytes;
          uint8_t* sb = b_tiles + static_cast<size_t>(stage) * b_tile_bytes;
          if (!ft.down) {
            tma_load_2d(sa, &tm_xp, &sh.full[stage], kb * kBK, ti.a_row);
            tma_load_2d(sb, &tm_w13, &sh.full[stage], kb * kBK, ti.b_row);
            tma_load_2d(sb + 128 * 128, &tm_w13, &sh.full[stage], kb * kBK,
                        ti.b_row2);
          } else {
            tma_load_2d(sa, &tm_h, &sh.full[stage], kb * kBK, ti.a_row);
            tma_load_2d(sb, &tm_w2, &sh.full[stage], kb * kBK, ti.b_row);
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
      // ---------------- MMA issuer (both phases: 128 x 256 tiles, K-major)
      const uint32_t idesc = umma_idesc_bf16_major(kBM, a.BN, false, false);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const TileInfo ti = ffn_decode(f, sh, t, up_total).ti;
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
          const uint64_t adesc = umma_desc_sw128(sa);
          const uint64_t bdesc = umma_desc_sw128(sb);
          if (ti.swap_n == 0) {
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k)
              umma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc,
                        (kb > ti.kb_begin || k > 0) ? 1u : 0u);
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
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const FfnTile ft = ffn_decode(f, sh, t, up_total);
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
      if (!ft.down) {
        epilogue_row<kUp>(f.up, ft.ti, tmem_row, r, half, nullptr);
        // this warp's part of the row block's H is written: count it
        __threadfence();
        __syncwarp();
        if (lane == 0) red_release_add_gpu(f.ready + ft.rb, 1u);
      } else {
        epilogue_row<kDown>(f.dn, ft.ti, tmem_row, r, half, nullptr);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.tempty[acc]);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, a.tmem_cols);
  }
  if (threadIdx.x == 0 && sh.abort) set_status(a.status, MOE_ERR_TIMEOUT);
}

}  // namespace moe
