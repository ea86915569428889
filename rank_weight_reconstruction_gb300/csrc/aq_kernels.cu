// aq_kernels.cu -- sm_103a kernels of the theta-bundle reconstruction linear
//   y = s . (W0 x) + U (V^T x)         ("How attnquant works", "The reconstruction identity")
//   W_eff = diag(s) W0 + U V^T         ("Execution paths", "Precompute-outside")
//
// aq_gemm_kernel         prefill (M > 32): tcgen05 GEMM over the K = in loop with a TMA-fed
//                        shared-memory ring, 128 tokens per tile as accumulator lanes and
//                        output rows as N, two accumulator buffers so a tile's epilogue
//                        overlaps the next tile's MMAs; the epilogue (eight warps, two per
//                        TMEM lane quadrant) scales the W0 x sum by s in TMEM, the rank-r
//                        up-projection is then added as extra K blocks
//                        into the same accumulator, and y is rounded once. t = x V runs as
//                        the first tiles of the same launch (or, for very large M, as a
//                        launch of its own). A CTA pair runs 2-SM MMAs (cta_group::2):
//                        each CTA of the pair loads its own half of the W0 / U rows with
//                        plain TMA loads (no multicast) and the even CTA's MMA reads both.
// aq_transpose_kernel    V [in, r] -> V^T [r, in] so the prefill t GEMM is K-major.
// aq_precompute_kernel   U V^T on tcgen05 (K = r), W0 tiles TMA-loaded and fused in the
//                        epilogue, W_eff written back with TMA stores; or, never forming
//                        the bf16 weight, the per-CTA max|W_eff| (amax pass) or W_eff
//                        quantized to NVFP4 in the epilogue ("Internals and extension",
//                        "Nvfp4Spec": E2M1 pairs per byte, an E4M3 scale per 16 values
//                        along K, one fp32 global scale).
#include <cuda.h>
#include <cuda_runtime.h>

#include "aq_internal.h"
#include "aq_ptx.cuh"

namespace aq {

__device__ int32_t g_device_status;  // AQ_OK or AQ_ERR_TIMEOUT, one word per device

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// Wait without honouring the abort flag (used to drain in-flight asynchronous work after
// an abort); bounded by its own limit.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

constexpr uint64_t kDrainNs = 20ull * 1000 * 1000;  // 20 ms per drained barrier

// Every lane waits; the outcome is made warp-uniform so that warp-collective tcgen05
// instructions after it are always executed by the whole warp or by none of it.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const AbortCtl& ctl) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl)) != 0;
}

// v[j] *= sc[j] for 16 columns: the scales as four 16-byte shared loads (sc 16-byte
// aligned), two columns per multiply instruction, each product rounded as a plain multiply
__device__ __forceinline__ void scale16(float (&v)[16], const float* sc) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 s4 = reinterpret_cast<const float4*>(sc)[q];
    fmul2_rn(v[4 * q], v[4 * q + 1], v[4 * q], v[4 * q + 1], s4.x, s4.y);
    fmul2_rn(v[4 * q + 2], v[4 * q + 3], v[4 * q + 2], v[4 * q + 3], s4.z, s4.w);
  }
}

// ------------------------------------------------------------------------------------
// GEMM with fused reconstruction epilogue
// ------------------------------------------------------------------------------------
struct TileCoord {
  int seg;
  int row0;
  int tok0;
};

// Work unit -> tile of this CTA: a unit is one row tile and `cluster` adjacent token tiles,
// one per CTA of the cluster (rank crank). Consecutive units (which run at the same time) share
// the operand that is re-read: token units fastest keep the token tiles in L2 while each row
// tile streams once; row tiles fastest (tok_major) keep the rows in L2 while each token tile
// streams once.
__device__ __forceinline__ TileCoord tile_coord(const GemmParams& p, int unit, int crank) {
  int si = 0;
#pragma unroll
  for (int j = 1; j < kMaxGemmSeg; ++j)
    if (j < p.nseg && unit >= p.seg[j].tile_begin) si = j;
  const int local = unit - p.seg[si].tile_begin;
  TileCoord c;
  c.seg = si;
  const int nrt = p.seg[si].n_row_tiles;
  const int tu = p.tok_major ? local / nrt : local % p.n_tok_units;
  const int rt = p.tok_major ? local - tu * nrt : local / p.n_tok_units;
  c.tok0 = (tu * p.cluster + crank) * p.tok_tile;
  c.row0 = rt * p.row_tile;
  return c;
}

// Two accumulator buffers of n_mma TMEM columns each, so a tile's epilogue overlaps the next
// tile's MMAs. The rank-r term needs no buffer of its own: once the W0 K loop of tile i is
// done, the epilogue scales the accumulator by s in place, and the MMA warp adds U t into it
// while the first head_kb k blocks of tile i+1 have covered the scale pass. Work items
// therefore reach the pipeline in the order
//   main(0), head(1), low(0), tail(1), head(2), low(1), tail(2), ..., low(last)
// (head + tail = main), which the producer and the MMA warp both walk with the same loop. The
// final pass of tile i then overlaps tail(i+1), so tile i+2, which reuses tile i's buffer,
// rarely waits for it.
//
// t = x V can run in the same launch: its segments come first in the unit order, so every
// cluster finishes its t tiles before any tile of its own that needs t. A t tile writes its
// rows of t (bf16, workspace) and bumps the flag of its token tile; the producer waits for
// the flag of a tile's token tile (bounded) before it loads t for the rank-r blocks. The
// last CTA to finish zeroes the flags again.
//
// With cluster = 2 the two CTAs of a cluster are one CTA pair of 2-SM MMAs (cta_group::2):
// each holds the 128-token tile of its own (A) and half of the row operand's N rows (B) per
// stage, and the even CTA issues M = 256 MMAs that read both CTAs' shared memory and write
// each CTA's TMEM. Per MMA a CTA's shared memory then moves 8 KB of operands instead of 12,
// and a stage takes 32 KB instead of 48. Both CTAs' TMA loads count on the even CTA's `full`
// barrier; its MMA commits arrive on both CTAs' `empty`, `acc_full` and `acc_done`; both
// CTAs' epilogue warps arrive on its `acc_scaled` and `acc_empty`.
// kPair: the CTA-pair (cluster = 2) variant; a function may not mix cta_group::1 and ::2.
//
// kSwap: the roles of the two operands are exchanged (the mid-M bucket, a few dozen to a few
// hundred tokens). The accumulator lanes are then 128 rows of the row operand (W0, V^T or U)
// and its N columns are the tokens (tok_tile = N <= 256): D[row, token]. One W0 tile feeds an
// MMA with all of a call's tokens, so W0 is streamed once even when the tokens are far fewer
// than 128, where the token-lane layout would pad most of every MMA. The epilogue owns one
// output row per thread: s is a per-thread scalar, and y is written down a column (32
// consecutive rows per warp-wide store). Not combined with CTA pairs.
template <bool kPair, bool kSwap>
__global__ void __launch_bounds__(kGemmThreads, 1) aq_gemm_kernel(const __grid_constant__ GemmParams p) {
  static_assert(!(kPair && kSwap), "the swapped-operand GEMM runs without CTA pairs");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint64_t* acc_full = empty + kMaxStages;   // [2] W0 loop of a tile done (MMA commit)
  uint64_t* acc_scaled = acc_full + 2;       // [2] accumulator scaled by s (one arrival per epilogue warp)
  uint64_t* acc_done = acc_scaled + 2;       // [2] rank-r blocks added (MMA commit)
  uint64_t* acc_empty = acc_done + 2;        // [2] accumulator drained (one arrival per epilogue warp)
  uint64_t* epi_bar = acc_empty + 2;         // epilogue warps' own barrier (every epilogue thread)
  uint64_t* mma_done = epi_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* last_cta = abort_flag + 1;
  float* sbuf = reinterpret_cast<float*>(smem + kHeaderBytes);   // s of the current tile, fp32
  uint8_t* ring = smem + kHeaderBytes + kGemmSBufBytes;
  uint8_t* ystage = ring + static_cast<size_t>(p.stages) * p.stage_bytes;   // output staging

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const AbortCtl ctl{abort_flag, p.status, p.timeout_ns};
  constexpr int cl = kPair ? 2 : 1;   // == p.cluster
  const int crank = kPair ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = crank == 0;   // issues the MMAs (the only CTA when unpaired)

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_scaled[b], kGemmEpiWarps * cl);   // one arrival per epilogue warp of each CTA
      mbar_init(&acc_done[b], 1);
      mbar_init(&acc_empty[b], kGemmEpiWarps * cl);
    }
    mbar_init(epi_bar, kGemmEpiWarps * 32);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_x);
    for (int j = 0; j < p.nseg; ++j) {
      tma_prefetch_desc(&p.seg[j].tm_w);
      if (p.seg[j].r > 0) {
        tma_prefetch_desc(&p.seg[j].tm_u);
        tma_prefetch_desc(&p.seg[j].tm_t);
      }
    }
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(tmem_slot, p.tmem_cols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, p.tmem_cols);
      tmem_relinquish();
    }
  }
  // The next kernel in the stream may now be scheduled and start its own weight
  // prefetch; it touches activations only after this grid has completed.
  pdl_launch_dependents();
  tc_fence_before();
  __syncthreads();
  // the peer's barriers are initialised before either CTA signals the other's
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int nkb_main = ceil_div_i(p.K, kBK);
  // bytes of one stage over the whole pair: each CTA's token tile and its share of the rows
  const uint32_t tx_bytes = static_cast<uint32_t>(cl) * static_cast<uint32_t>(p.row_tile / cl + p.tok_tile) * 128u;
  const int cid = static_cast<int>(blockIdx.x) / cl;
  const int ncl = static_cast<int>(gridDim.x) / cl;
  const int n_it = cid < p.total_tiles ? (p.total_tiles - 1 - cid) / ncl + 1 : 0;
  auto tile_of = [&](int it) { return cid + it * ncl; };
  // Work item it of this CTA: a unit's tile and one slice of its K (split K), or all of K.
  // Zero-initialised parameters mean no split.
  const int ksplit = p.ksplit > 1 ? p.ksplit : 1;
  const int kb_per = p.ksplit > 1 ? p.kb_per : nkb_main;
  struct Item {
    TileCoord tc;
    int ks, kb_lo, nkb;
  };
  auto item_of = [&](int it) {
    const int w = tile_of(it);
    Item m;
    m.ks = w % ksplit;
    m.tc = tile_coord(p, w / ksplit, crank);
    m.kb_lo = m.ks * kb_per;
    m.nkb = min(kb_per, nkb_main - m.kb_lo);
    return m;
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // the operand that later waves of tiles read again stays in L2 (evict-last); the other is
      // shared by the tiles running at the same time, so it keeps the normal policy (an
      // evict-first stream was measured to re-read it from DRAM)
      const uint64_t pol_tok = p.tok_major ? policy_evict_normal() : policy_evict_last();
      const uint64_t pol_row = p.tok_major ? policy_evict_last() : policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0, fill_par = 0;
      bool ok = true;
      // one box into this CTA's stage, counted on the even CTA's `full` barrier
      auto load = [&](uint8_t* dst, const CUtensorMap* m, int c0, int c1, uint64_t* bar, uint64_t pol) {
        if constexpr (kPair) {
          tma_load_2d_pair(dst, m, c0, c1, cluster_map(bar, 0), pol);
        } else {
          tma_load_2d(dst, m, c0, c1, bar, pol);
        }
      };
      // B: the whole N rows, or this CTA's half of them (rows n_mma / 2 apart)
      auto load_rows = [&](uint8_t* st, const CUtensorMap* m, int kb, int row0, int n_mma, uint64_t* bar) {
        load(st + kStageA, m, kb * kBK, row0 + crank * (n_mma / cl), bar, pol_row);
      };
      // one k block of work item (tile, low) into the next stage
      auto push = [&](const TileCoord& tc, const GemmSeg& sg, bool low, int kb) -> bool {
        if (!mbar_wait(&empty[stage], phase ^ 1, ctl)) return false;
        uint8_t* st = ring + static_cast<size_t>(stage) * p.stage_bytes;
        if (leader) mbar_arrive_expect_tx(&full[stage], tx_bytes);
        if constexpr (kSwap) {
          // A = 128 rows (W0, or U), B = the tokens (x, or t for the rank-r blocks)
          load(st, low ? &sg.tm_u : &sg.tm_w, kb * kBK, tc.row0, &full[stage], pol_row);
          load(st + kStageA, low ? &sg.tm_t : &p.tm_x, kb * kBK, tc.tok0, &full[stage], pol_tok);
        } else {
          // A = tokens (x, or t for the rank-r blocks), B = rows (W0, or U)
          load(st, low ? &sg.tm_t : &p.tm_x, kb * kBK, tc.tok0, &full[stage], pol_tok);
          load_rows(st, low ? &sg.tm_u : &sg.tm_w, kb, tc.row0, sg.n_mma, &full[stage]);
        }
        filled |= 1u << stage;
        fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1;
        }
        return true;
      };
      // the row operand of the first tile may be loaded before the previous grid completes
      // only when it is a weight (V^T of a t tile is written by the previous kernel)
      const bool pre_w = p.prefetch_w && n_it > 0 && !p.seg[item_of(0).tc.seg].t_seg;
      if (!pre_w) pdl_wait_prior_grid();
      for (int it = 0; ok && it <= n_it; ++it) {
        const Item cur = it < n_it ? item_of(it) : Item{};
        const int h = it == 0 ? cur.nkb : min(p.head_kb, cur.nkb);   // head k blocks of item it
        if (it < n_it) {
          const TileCoord tc = cur.tc;
          const GemmSeg& sg = p.seg[tc.seg];
          int kb = 0;
          if (it == 0 && pre_w) {
            // Weight tiles of the first stages go out before waiting on the previous grid.
            const int pre = cur.nkb < p.stages ? cur.nkb : p.stages;
            for (; kb < pre; ++kb) {
              uint8_t* st = ring + static_cast<size_t>(kb) * p.stage_bytes;
              if (leader) mbar_arrive_expect_tx(&full[kb], tx_bytes);
              if constexpr (kSwap) {
                load(st, &sg.tm_w, (cur.kb_lo + kb) * kBK, tc.row0, &full[kb], pol_row);
              } else {
                load_rows(st, &sg.tm_w, cur.kb_lo + kb, tc.row0, sg.n_mma, &full[kb]);
              }
              filled |= 1u << kb;
            }
            pdl_wait_prior_grid();
            for (int j = 0; j < pre; ++j) {
              uint8_t* st = ring + static_cast<size_t>(j) * p.stage_bytes;
              load(kSwap ? st + kStageA : st, &p.tm_x, (cur.kb_lo + j) * kBK, tc.tok0, &full[j], pol_tok);
            }
            stage = pre;
            if (stage == p.stages) {
              stage = 0;
              phase ^= 1;
            }
          }
          for (; ok && kb < h; ++kb) ok = push(tc, sg, false, cur.kb_lo + kb);
        }
        if (ok && it >= 1) {
          const TileCoord tc = item_of(it - 1).tc;
          const GemmSeg& sg = p.seg[tc.seg];
          const int nkb_low = sg.r > 0 ? ceil_div_i(sg.r, kBK) : 0;
          if (nkb_low > 0 && p.t_flags) {
            // t of this token tile is written by t tiles of this launch
            const int32_t* flag = p.t_flags + 1 + tc.tok0 / p.tok_tile;
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_gpu(flag) < p.t_need) {
              if (*reinterpret_cast<volatile int*>(abort_flag) || global_timer_ns() - t0 > p.timeout_ns) {
                *reinterpret_cast<volatile int*>(abort_flag) = 1;
                atomicExch(p.status, kStatusTimeout);
                ok = false;
                break;
              }
              __nanosleep(64);
            }
            fence_proxy_async_global();   // the TMA reads of t follow the acquire
          }
          for (int kb = 0; ok && kb < nkb_low; ++kb) ok = push(tc, sg, true, kb);
        }
        if (ok && it >= 1 && it < n_it) {
          const GemmSeg& sg = p.seg[cur.tc.seg];
          for (int kb = h; ok && kb < cur.nkb; ++kb) ok = push(cur.tc, sg, false, cur.kb_lo + kb);
        }
      }
      if (!ok && leader) {
        // Let every copy already issued land before the CTA can exit (a pair's copies all
        // count on the even CTA's barriers; both CTAs stay until the final cluster barrier).
        for (int s = 0; s < p.stages; ++s)
          if (filled & (1u << s)) mbar_wait_drain(&full[s], (fill_par >> s) & 1u, kDrainNs);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (the even CTA of a pair) ----------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = leader;
    // arrival on `bar` in this CTA and, for a pair, in the peer, once the MMAs so far finish
    auto commit_all = [&](uint64_t* bar) {
      if constexpr (kPair) {
        tc_commit_pair_multicast(bar, 0x3);
      } else {
        tc_commit(bar);
      }
    };
    const int mma_m = kMmaM * cl;
    // k blocks [kb0, kb1) of one work item into accumulator buffer b; `acc` = 1 adds to what
    // is there; rem_last: valid K of the last block when it is partial (rank-r blocks)
    auto run = [&](int kb0, int kb1, int rem_last, uint32_t b, uint32_t acc, uint32_t idesc) -> bool {
      const uint32_t d = tmem_base + b * static_cast<uint32_t>(p.n_mma);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!warp_wait(&full[stage], phase, ctl)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a_addr = smem_u32(ring + static_cast<size_t>(stage) * p.stage_bytes);
          const uint32_t b_addr = a_addr + kStageA;
          const int nk = (kb == kb1 - 1 && rem_last > 0) ? ceil_div_i(rem_last, kUmmaK) : kBK / kUmmaK;
          for (int j = 0; j < nk; ++j) {
            const uint32_t en = (acc || kb > 0 || j > 0) ? 1u : 0u;
            if constexpr (kPair) {
              tc_mma_bf16_pair(d, smem_desc_k128(a_addr + 32u * j), smem_desc_k128(b_addr + 32u * j), idesc, en);
            } else {
              tc_mma_bf16(d, smem_desc_k128(a_addr + 32u * j), smem_desc_k128(b_addr + 32u * j), idesc, en);
            }
          }
          commit_all(&empty[stage]);
        }
        __syncwarp();
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1;
        }
      }
      return true;
    };
    // Start the bounded waits only once the previous grid is done, so that a long
    // predecessor cannot be mistaken for a stalled pipeline.
    pdl_wait_prior_grid();
    // acc_scaled / acc_done are used only by tiles with a rank-r part: their phases advance
    // per use (bit b for buffer b), not per tile
    uint32_t lr_phase = 0;
    for (int it = 0; ok && it <= n_it; ++it) {   // (the odd CTA of a pair issues nothing)
      const Item cur = it < n_it ? item_of(it) : Item{};
      const int h = it == 0 ? cur.nkb : min(p.head_kb, cur.nkb);
      if (it < n_it) {
        const uint32_t b = it & 1;
        if (!warp_wait(&acc_empty[b], ((it >> 1) & 1) ^ 1, ctl)) break;
        tc_fence_after();
        ok = run(0, h, 0, b, 0u, idesc_bf16_f32(mma_m, p.seg[cur.tc.seg].n_mma));
      }
      if (ok && it >= 1) {
        const TileCoord tc = item_of(it - 1).tc;
        const GemmSeg& sg = p.seg[tc.seg];
        if (sg.r > 0) {
          const uint32_t b = (it - 1) & 1;
          if (!warp_wait(&acc_scaled[b], (lr_phase >> b) & 1u, ctl)) break;
          lr_phase ^= 1u << b;
          tc_fence_after();
          ok = run(0, ceil_div_i(sg.r, kBK), sg.r % kBK, b, 1u, idesc_bf16_f32(mma_m, sg.n_mma));
          if (ok && lane == 0) commit_all(&acc_done[b]);
          __syncwarp();
        }
      }
      if (ok && it < n_it) {
        const uint32_t b = it & 1;
        ok = run(h, cur.nkb, 0, b, 1u, idesc_bf16_f32(mma_m, p.seg[cur.tc.seg].n_mma));
        if (ok && lane == 0) commit_all(&acc_full[b]);
        __syncwarp();
      }
    }
    if (leader && lane == 0) {
      if constexpr (kPair) {
        tc_commit_pair(mma_done);
      } else {
        tc_commit(mma_done);
      }
      mbar_wait_drain(mma_done, 0, kDrainNs);
    }
    __syncwarp();
  } else {
    // ------- epilogue: warps 2.., two per TMEM lane quadrant, each one half of the columns -------
    const int q = warp & 3;
    const int et = q * 32 + lane;                 // 0..127: TMEM lane = token of the tile
    const int ect = threadIdx.x - 64;             // epilogue thread, 0..32 * kGemmEpiWarps - 1
    const int hw = (warp - 2) >> 2;               // column half of this warp
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    // this warp's accumulator columns of an n-column tile (n a multiple of 16): [c_lo, c_hi)
    auto col_lo = [&](int n) { return hw ? (((n >> 4) + 1) >> 1) << 4 : 0; };
    auto col_hi = [&](int n) { return hw ? n : (((n >> 4) + 1) >> 1) << 4; };
    // one arrival per warp on the MMA-issuing CTA's barrier
    auto mbar_arrive_lead = [&](uint64_t* bar) {
      if constexpr (kPair) {
        mbar_arrive_cluster(cluster_map(bar, 0));
      } else {
        mbar_arrive(bar);
      }
    };
    uint32_t ephase = 0;
    auto epi_sync = [&]() {
      mbar_arrive(epi_bar);
      const bool r = mbar_wait(epi_bar, ephase, ctl);
      ephase ^= 1u;
      return r;
    };
    pdl_wait_prior_grid();
    uint32_t lr_phase = 0;   // phases of acc_done[b] (bit b), advanced per rank-r use
    for (int it = 0; it < n_it; ++it) {
      const Item itm = item_of(it);
      const TileCoord tc = itm.tc;
      const GemmSeg& sg = p.seg[tc.seg];
      const bool has_lr = sg.r > 0;
      const uint32_t b = it & 1;
      const uint32_t par = (it >> 1) & 1;
      const uint32_t acc = t_lane + b * static_cast<uint32_t>(p.n_mma);
      if constexpr (kSwap) {
        // ---- lane = output row, columns = tokens ----
        const int row = tc.row0 + et;
        const bool row_ok = et < p.row_tile && row < sg.rows;
        // this row's scale, requested before the wait so that it lands while the MMAs run
        const float sc = (row_ok && sg.s) ? bf16_to_f32(sg.s[row]) : 1.0f;
        if (!warp_wait(&acc_full[b], par, ctl)) break;
        tc_fence_after();
        if (has_lr) {
          // scale the W0 x accumulator by s in place; the MMA warp then adds U t
          for (int c = col_lo(sg.n_mma); c < col_hi(sg.n_mma); c += 16) {
            float v[16];
            tmem_ld_16(acc + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] *= sc;
            tmem_st_16(acc + c, v);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_lead(&acc_scaled[b]);
          if (!warp_wait(&acc_done[b], (lr_phase >> b) & 1u, ctl)) break;
          lr_phase ^= 1u << b;
          tc_fence_after();
        }
        if (sg.part) {
          // split K: this slice's raw fp32 sums [slice][token][row], 32 consecutive rows per
          // warp-wide store
          float* pcol = sg.part + static_cast<int64_t>(itm.ks) * p.M * sg.ld_part + (row_ok ? row : 0);
          for (int c = col_lo(sg.n_mma); c < col_hi(sg.n_mma); c += 16) {
            float v[16];
            tmem_ld_16(acc + c, v);
            tmem_ld_wait();
            if (!row_ok) continue;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int tok = tc.tok0 + c + j;
              if (tok < p.M &&
                  dbg_in_bounds(static_cast<int64_t>(itm.ks) * p.M * sg.ld_part + static_cast<int64_t>(tok) * sg.ld_part + row,
                                static_cast<int64_t>(p.ksplit) * p.M * sg.ld_part, p.status))
                pcol[static_cast<int64_t>(tok) * sg.ld_part] = v[j];
            }
          }
        } else {
          uint16_t* ycol = sg.y + (row_ok ? row : 0);
          for (int c = col_lo(sg.n_mma); c < col_hi(sg.n_mma); c += 16) {
            float v[16];
            tmem_ld_16(acc + c, v);
            tmem_ld_wait();
            if (!row_ok) continue;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int tok = tc.tok0 + c + j;
              if (tok < p.M && dbg_in_bounds(static_cast<int64_t>(tok) * sg.ldy + row, dbg_extent(p.M, sg.ldy, sg.rows), p.status))
                ycol[static_cast<int64_t>(tok) * sg.ldy] = f32_to_bf16_rn(has_lr ? v[j] : v[j] * sc);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_lead(&acc_empty[b]);
        if (sg.t_seg && !sg.part) {
          // publish this token tile's t: every thread's stores, then one release
          __threadfence();
          fence_proxy_async_global();
          if (!epi_sync()) break;
          if (ect == 0) red_release_gpu_add(p.t_flags + 1 + tc.tok0 / p.tok_tile, 1);
        }
        continue;
      }
      // s of this tile's rows into shared memory (fp32, zero past the tile) while the
      // tensor core works on it
      if (!epi_sync()) break;   // every epilogue warp is done with the previous tile's s
      for (int c = ect; c < p.n_mma; c += kGemmEpiWarps * 32) {
        const int o = tc.row0 + c;
        sbuf[c] = (c < p.row_tile && o < sg.rows) ? (sg.s ? bf16_to_f32(sg.s[o]) : 1.0f) : 0.0f;
      }
      if (!epi_sync()) break;
      if (!warp_wait(&acc_full[b], par, ctl)) break;
      tc_fence_after();
      if (has_lr) {
        // scale the W0 x accumulator by s in place; the MMA warp then adds U t
        for (int c = col_lo(sg.n_mma); c < col_hi(sg.n_mma); c += 16) {
          float v[16];
          tmem_ld_16(acc + c, v);
          tmem_ld_wait();
          scale16(v, sbuf + c);
          tmem_st_16(acc + c, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_lead(&acc_scaled[b]);
        if (!warp_wait(&acc_done[b], (lr_phase >> b) & 1u, ctl)) break;
        lr_phase ^= 1u << b;
        tc_fence_after();
      }
      if (sg.tma_y) {
        // 64-column chunks (the two warps of a lane quadrant alternate) through this warp's
        // staging buffer (row = token, 128-byte swizzle), each written out by one bulk tensor
        // store; the tensor map clips rows past M and columns past the family's rows. A chunk
        // is converted into registers before the wait for the previous store's read.
        uint8_t* buf = ystage + static_cast<size_t>(warp - 2) * kYStageBytes;
        uint8_t* row = buf + lane * 128;
        int nst = 0;
        for (int c0 = 64 * hw; c0 < sg.n_mma; c0 += 128, ++nst) {
          uint32_t pk[32];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int c = c0 + q4 * 16;
            float v[16];
            tmem_ld_16(acc + c, v);
            tmem_ld_wait();
            if (!has_lr) scale16(v, sbuf + c);
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[8 * q4 + e] = pack_bf16x2_cvt(v[2 * e], v[2 * e + 1]);
          }
          if (nst > 0 && lane == 0) tma_store_wait_read_all();   // the previous chunk's store read the buffer
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 8; ++h)
            *reinterpret_cast<uint4*>(row + ((h ^ (lane & 7)) << 4)) =
                make_uint4(pk[4 * h], pk[4 * h + 1], pk[4 * h + 2], pk[4 * h + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&sg.tm_y, buf, tc.row0 + c0, tc.tok0 + q * 32);
            tma_store_commit();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_lead(&acc_empty[b]);
        if (lane == 0) tma_store_wait_read_all();   // the staging is free for the next tile
        __syncwarp();
        continue;
      }
      const int tok = tc.tok0 + et;
      const bool tok_ok = tok < p.M;
      if (sg.part) {
        // split K: this slice's raw fp32 sums (no scale, no rank-r part), summed in order
        // and finished by the finalize kernel; ld_part and the columns are multiples of 4
        float* prow = sg.part + (static_cast<int64_t>(itm.ks) * p.M + (tok_ok ? tok : 0)) * sg.ld_part;
        for (int c = col_lo(sg.n_mma); c < col_hi(sg.n_mma); c += 16) {
          float v[16];
          tmem_ld_16(acc + c, v);
          tmem_ld_wait();
          const int o0 = tc.row0 + c;
          if (!tok_ok || c >= p.row_tile || o0 >= sg.rows) continue;
          if (!dbg_in_bounds((static_cast<int64_t>(itm.ks) * p.M + tok) * sg.ld_part + min(o0 + 15, sg.rows - 1),
                             static_cast<int64_t>(p.ksplit) * p.M * sg.ld_part, p.status))
            continue;
          if ((c + 16 <= p.row_tile) && (o0 + 16 <= sg.rows)) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<float4*>(prow + o0 + 4 * q4) =
                  make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (c + j < p.row_tile && o0 + j < sg.rows) prow[o0 + j] = v[j];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_lead(&acc_empty[b]);
        continue;
      }
      uint16_t* yrow = sg.y + static_cast<int64_t>(tok) * sg.ldy;
      for (int c = col_lo(sg.n_mma); c < col_hi(sg.n_mma); c += 16) {
        float v[16];
        tmem_ld_16(acc + c, v);
        tmem_ld_wait();
        const int o0 = tc.row0 + c;
        if (!tok_ok || c >= p.row_tile || o0 >= sg.rows) continue;
        if (!dbg_in_bounds(static_cast<int64_t>(tok) * sg.ldy + min(o0 + 15, sg.rows - 1), dbg_extent(p.M, sg.ldy, sg.rows),
                           p.status))
          continue;
        if (!has_lr) scale16(v, sbuf + c);
        if ((c + 16 <= p.row_tile) && (o0 + 16 <= sg.rows)) {
          uint4 w0, w1;
          w0.x = pack_bf16x2_cvt(v[0], v[1]);
          w0.y = pack_bf16x2_cvt(v[2], v[3]);
          w0.z = pack_bf16x2_cvt(v[4], v[5]);
          w0.w = pack_bf16x2_cvt(v[6], v[7]);
          w1.x = pack_bf16x2_cvt(v[8], v[9]);
          w1.y = pack_bf16x2_cvt(v[10], v[11]);
          w1.z = pack_bf16x2_cvt(v[12], v[13]);
          w1.w = pack_bf16x2_cvt(v[14], v[15]);
          *reinterpret_cast<uint4*>(yrow + o0) = w0;
          *reinterpret_cast<uint4*>(yrow + o0 + 8) = w1;
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c + j < p.row_tile && o0 + j < sg.rows) yrow[o0 + j] = f32_to_bf16_rn(v[j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_lead(&acc_empty[b]);
      if (sg.t_seg) {
        // publish this token tile's t: every thread's stores, then one release
        __threadfence();
        fence_proxy_async_global();
        if (!epi_sync()) break;
        if (ect == 0) red_release_gpu_add(p.t_flags + 1 + tc.tok0 / p.tok_tile, 1);
      }
    }
    if (lane == 0) tma_store_wait_all();   // this warp's bulk stores of y are complete
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // a pair: both CTAs are done with the accumulators and with each other's barriers
  if constexpr (kPair) cluster_sync_all();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_dealloc_pair(tmem_base, p.tmem_cols);
    } else {
      tmem_dealloc(tmem_base, p.tmem_cols);
    }
  }
  if (p.t_flags) {
    // every CTA is past its last flag wait once all have counted themselves here: the last
    // one returns the flags to zero for the next call
    if (threadIdx.x == 0) {
      __threadfence();
      *last_cta = atomicAdd(p.t_flags, 1) == static_cast<int>(gridDim.x) - 1 ? 1 : 0;
    }
    __syncthreads();
    if (*last_cta) {
      for (int i = threadIdx.x; i < p.n_flags; i += blockDim.x) p.t_flags[1 + i] = 0;
      __syncthreads();
      if (threadIdx.x == 0) {
        p.t_flags[0] = 0;
        __threadfence();
      }
    }
  }
  if constexpr (kPair) cluster_sync_all();
}
// ------------------------------------------------------------------------------------
// Split-K finalize: y[m, o] = RN(s[o] * sum_k z_k[m, o] + sum_j U[o, j] * t[m, j]) with
// t[m, j] = sum_k t_k[m, j], every sum over the slices in slice order (deterministic).
// One thread per output (kFinRows consecutive rows of one token per block: the partial sums
// and y are read and written in 128-byte lines), the U row in registers, t of the block's
// token summed once into shared memory. The work per output is ksplit loads and r FMAs, so
// the kernel is a few round trips deep; enough threads keep those round trips overlapped.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kFinRows) aq_finalize_kernel(const __grid_constant__ FinalizeParams p) {
  __shared__ float ts[kFinMaxR];
  int si = 0;
#pragma unroll
  for (int j = 1; j < kMaxSeg; ++j)
    if (j < p.nseg && static_cast<int>(blockIdx.x) >= p.seg[j].block_begin) si = j;
  const FinalizeSeg& sg = p.seg[si];
  const int o = (static_cast<int>(blockIdx.x) - sg.block_begin) * kFinRows + static_cast<int>(threadIdx.x);
  const int m = static_cast<int>(blockIdx.y);
  const bool live = o < sg.rows;
  // weights before the dependency wait: this row's U and s
  float u[kSplitMaxRank];
#pragma unroll
  for (int j = 0; j < kSplitMaxRank; ++j) u[j] = 0.0f;
  if (live && sg.r > 0) {
    const uint16_t* urow = sg.U + static_cast<int64_t>(o) * sg.ldu;
#pragma unroll
    for (int j = 0; j < kSplitMaxRank; ++j)
      if (j < sg.r) u[j] = bf16_to_f32(urow[j]);
  }
  const float sc = (live && sg.s) ? bf16_to_f32(sg.s[o]) : 1.0f;
  pdl_wait_prior_grid();   // the partial sums are the previous grid's output
  if (static_cast<int>(threadIdx.x) < sg.r) {
    float v = 0.0f;
    for (int ks = 0; ks < p.ksplit; ++ks)
      v += sg.pt[ks * p.pt_slice + static_cast<int64_t>(m) * p.ld_pt + threadIdx.x];
    ts[threadIdx.x] = v;
  }
  float z = 0.0f;
  if (live) {
    const float* pz = sg.pz + static_cast<int64_t>(m) * p.ld_pz + o;
#pragma unroll 4
    for (int ks = 0; ks < p.ksplit; ++ks) z += pz[ks * p.pz_slice];
  }
  __syncthreads();
  pdl_launch_dependents();
  if (!live) return;
  float lr = 0.0f;
#pragma unroll
  for (int j = 0; j < kSplitMaxRank; ++j)
    if (j < sg.r) lr = fmaf(u[j], ts[j], lr);
  sg.y[static_cast<int64_t>(m) * sg.ldy + o] = f32_to_bf16_rn(fmaf(sc, z, lr));
}

// ------------------------------------------------------------------------------------
// V [in, r] -> V^T [r, in]
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) aq_transpose_kernel(const __grid_constant__ TransposeParams p) {
  __shared__ uint16_t tile[32][34];
  const TransposeSeg& sg = p.seg[blockIdx.z];
  const int i0 = blockIdx.x * 32;
  const int k0 = blockIdx.y * 32;
  pdl_launch_dependents();
  if (k0 >= sg.r) return;
  const int tx = threadIdx.x & 31;
  const int ty = threadIdx.x >> 5;
  // V is a weight: read it while the previous kernel finishes; the workspace it is written
  // to may still be in use until then
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int i = i0 + ty + 8 * j;
    const int k = k0 + tx;
    tile[ty + 8 * j][tx] = (i < p.K && k < sg.r) ? sg.V[static_cast<int64_t>(i) * sg.ldv + k] : 0;
  }
  __syncthreads();
  pdl_wait_prior_grid();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int k = k0 + ty + 8 * j;
    const int i = i0 + tx;
    if (k < sg.r && i < p.K) sg.Vt[static_cast<int64_t>(k) * sg.ldvt + i] = tile[tx][ty + 8 * j];
  }
}

// ------------------------------------------------------------------------------------
// W_eff = s * W0 + U V^T
// ------------------------------------------------------------------------------------
constexpr int kPreMaxCBufs = 8;   // W0 / W_eff tile buffers per CTA (p.cbufs of them used)
constexpr int kPreAcc = 2;     // TMEM accumulators
constexpr int kPreRedOffset = 768;   // header bytes holding the epilogue warps' maxima

// FP8 E4M3 byte of a non-negative fp32: nearest, ties to even, clamped to 448.
__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float a) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(a));
  return r & 0xFFu;
}

// Value of a finite non-negative E4M3 byte: exponent bias 7, 3 mantissa bits, subnormal
// step 2^-9 (exact in fp32).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u;
  const uint32_t m = b & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0x1p-9f;
}

// Eight fp32 values to E2M1 codes (nearest, ties to even, clamped to +-6, sign kept), the
// first value in the lowest nibble.
__device__ __forceinline__ uint32_t f32x8_to_e2m1(const float* q) {
  uint32_t r;
  asm("{\n"
      " .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n"
      "}"
      : "=r"(r)
      : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
  return r;
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// One block of 16 values: returns its E4M3 scale byte, codes in two words. a = max|v|,
// scale = E4M3(a * (1 / (6 g))), d = scale * g, code = E2M1(v * (1 / d)); each step one fp32
// operation rounded to nearest even (1 / (6 g) formed once per CTA; 1 / d per scale byte
// precomputed in inv_tbl, 0 where d is 0); d = 0 stores +0 codes.
__device__ __forceinline__ uint32_t nvfp4_block(const float* v, float inv6g, const float* inv_tbl, uint2* codes) {
  // max|v| as a tree of three-input maxima (max is exact in any order)
  float m[6];
#pragma unroll
  for (int j = 0; j < 5; ++j) m[j] = fmax3(fabsf(v[3 * j]), fabsf(v[3 * j + 1]), fabsf(v[3 * j + 2]));
  m[5] = fabsf(v[15]);
  const float a = fmaxf(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]));
  const uint32_t sf = f32_to_e4m3_satfinite(__fmul_rn(a, inv6g));
  const float inv = inv_tbl[sf];
  if (!(inv > 0.0f)) {
    *codes = make_uint2(0u, 0u);
    return sf;
  }
  float q[16];
#pragma unroll
  for (int j = 0; j < 16; j += 2) fmul2_rn(q[j], q[j + 1], v[j], v[j + 1], inv, inv);
  *codes = make_uint2(f32x8_to_e2m1(q), f32x8_to_e2m1(q + 8));
  return sf;
}

// Max over the 512 epilogue threads of the precompute kernel (named barrier 1); every
// epilogue thread gets the result.
__device__ __forceinline__ float epilogue_max(float m, float* red, int warp, int lane) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp - 2] = m;
  named_bar_sync(1, kPreThreads - 64);
  float r = 0.0f;
#pragma unroll
  for (int w = 0; w < (kPreThreads - 64) / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}

// This CTA's tiles: blockIdx.x, then every gridDim.x-th (so that the CTAs together sweep
// the weight front to back), walked last to first when reversed; (row band, column tile)
// stepped without divisions.
struct TileWalk {
  int count;     // tiles of this CTA
  int row, col;  // the current tile
  int n_col, drow, dcol;
  bool rev;
  __device__ __forceinline__ TileWalk(int total, int n_col_, bool rev_) : n_col(n_col_), rev(rev_) {
    const int g = static_cast<int>(gridDim.x);
    const int b = static_cast<int>(blockIdx.x);
    count = b < total ? (total - 1 - b) / g + 1 : 0;
    const int t = rev ? total - 1 - b : b;
    row = t / n_col;
    col = t - row * n_col;
    drow = g / n_col;
    dcol = g - drow * n_col;
  }
  __device__ __forceinline__ void next() {
    if (rev) {
      col -= dcol;
      row -= drow;
      if (col < 0) {
        col += n_col;
        --row;
      }
    } else {
      col += dcol;
      row += drow;
      if (col >= n_col) {
        col -= n_col;
        ++row;
      }
    }
  }
};

template <int kOut>
__global__ void __launch_bounds__(kPreThreads, 1)
    aq_precompute_kernel(const __grid_constant__ PrecomputeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint64_t* c_full = empty + kMaxStages;
  uint64_t* c_empty = c_full + kPreMaxCBufs;
  uint64_t* acc_full = c_empty + kPreMaxCBufs;
  uint64_t* acc_empty = acc_full + kPreAcc;
  uint64_t* epi_done = acc_empty + kPreAcc;
  uint64_t* mma_done = epi_done + kPreMaxCBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const uint32_t cbuf_bytes = static_cast<uint32_t>(p.bn) * 256u;  // bn/64 boxes of 128 x 128 B
  const int nkb = p.r > 0 ? ceil_div_i(p.r, kBK) : 0;
  uint8_t* cbuf = smem + kHeaderBytes;
  uint8_t* ring = cbuf + p.cbufs * cbuf_bytes;                              // U / V chunks
  // kPreNvfp4: 1/d for each of the 128 scale bytes
  float* inv_tbl = reinterpret_cast<float*>(ring + static_cast<size_t>(p.stages) * p.stage_bytes);
  float* red = reinterpret_cast<float*>(smem + kPreRedOffset);
  // tile order: last to first when the amax pass just walked them first to last
  const bool rev = kOut == kPreNvfp4 && p.reverse != 0;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const AbortCtl ctl{abort_flag, p.status, p.timeout_ns};
  const bool has_mma = p.r > 0;
  const int nbox = p.bn / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < p.cbufs; ++b) {
      mbar_init(&c_full[b], 1);
      // bf16: the leader frees a buffer after its store; otherwise every epilogue thread
      // frees it once it has read its row segment
      mbar_init(&c_empty[b], kOut == kPreBf16 ? 1 : kPreThreads - 64);
      mbar_init(&epi_done[b], kPreThreads - 64);
    }
    for (int b = 0; b < kPreAcc; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kPreThreads - 64);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_w0);
    if (kOut == kPreBf16) tma_prefetch_desc(&p.tm_we);
    if (has_mma) {
      tma_prefetch_desc(&p.tm_u);
      tma_prefetch_desc(&p.tm_v);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  // No early trigger of dependents here: the next call may read W_eff as its W0, and the
  // linear kernels fetch W0 before their dependency wait. Without the trigger the next
  // kernel starts only after every CTA has exited, its bulk stores complete.
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // Two independent producers: lane 0 streams W0 tiles as far ahead as the tile buffers
    // allow, lane 1 feeds the U / V chunks of the MMA. One thread doing both would tie the
    // W0 prefetch depth to the MMA's progress through the short U / V ring.
    if (lane == 0) {
      // the amax pass leaves W0 in L2 for the quantizing pass that follows it
      const uint64_t pol_stream = kOut == kPreAmax ? policy_evict_normal() : policy_evict_first();
      uint32_t cfilled = 0, cfill_par = 0;
      bool ok = true;
      pdl_wait_prior_grid();
      TileWalk tr(p.total_tiles, p.n_col_tiles, rev);
      TileWalk pf = tr;   // pf_ahead tiles ahead: prefetched into L2 beyond the tile buffers
      for (int a = 0; a < p.pf_ahead; ++a) pf.next();
      for (int it = 0; ok && it < tr.count; ++it, tr.next()) {
        const int o0 = tr.row * kMmaM;
        const int i0 = tr.col * p.bn;
        const int cb = it % p.cbufs;
        const uint32_t cph = static_cast<uint32_t>(it / p.cbufs) & 1u;
        if (!mbar_wait(&c_empty[cb], cph ^ 1u, ctl)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&c_full[cb], cbuf_bytes);
        for (int j = 0; j < nbox; ++j)
          tma_load_2d(cbuf + cb * cbuf_bytes + j * kStageA, &p.tm_w0, i0 + 64 * j, o0, &c_full[cb],
                      pol_stream);
        if (p.pf_ahead > 0 && it + p.pf_ahead < tr.count) {
          for (int j = 0; j < nbox; ++j) tma_prefetch_l2_2d(&p.tm_w0, pf.col * p.bn + 64 * j, pf.row * kMmaM);
          pf.next();
        }
        cfilled |= 1u << cb;
        cfill_par = (cfill_par & ~(1u << cb)) | (cph << cb);
      }
      if (!ok) {
        for (int b = 0; b < p.cbufs; ++b)
          if (cfilled & (1u << b)) mbar_wait_drain(&c_full[b], (cfill_par >> b) & 1u, kDrainNs);
      }
    } else if (lane == 1 && has_mma) {
      const uint64_t pol_keep = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t filled = 0, fill_par = 0;
      bool ok = true;
      TileWalk tr(p.total_tiles, p.n_col_tiles, rev);
      for (int it = 0; ok && it < tr.count; ++it, tr.next()) {
        const int o0 = tr.row * kMmaM;
        const int i0 = tr.col * p.bn;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, ctl)) {
            ok = false;
            break;
          }
          uint8_t* st = ring + static_cast<size_t>(stage) * p.stage_bytes;
          mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(kMmaM + p.bn) * 128u);
          tma_load_2d(st, &p.tm_u, kb * kBK, o0, &full[stage], pol_keep);
          tma_load_2d(st + kStageA, &p.tm_v, kb * kBK, i0, &full[stage], pol_keep);
          filled |= 1u << stage;
          fill_par = (fill_par & ~(1u << stage)) | (phase << stage);
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        for (int s2 = 0; s2 < p.stages; ++s2)
          if (filled & (1u << s2)) mbar_wait_drain(&full[s2], (fill_par >> s2) & 1u, kDrainNs);
      }
    }
  } else if (warp == 1) {
    if (has_mma) {
      const uint32_t idesc = idesc_bf16_f32(kMmaM, p.bn);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const int count = TileWalk(p.total_tiles, p.n_col_tiles, rev).count;
      for (int it = 0; ok && it < count; ++it) {
        const int ab = it & 1;
        const uint32_t aph = static_cast<uint32_t>(it >> 1) & 1u;
        if (!warp_wait(&acc_empty[ab], aph ^ 1u, ctl)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(ab * p.bn);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!warp_wait(&full[stage], phase, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a_addr = smem_u32(ring + static_cast<size_t>(stage) * p.stage_bytes);
            const uint32_t b_addr = a_addr + kStageA;
            const int rem = p.r - kb * kBK;
            const int nk = rem >= kBK ? kBK / kUmmaK : ceil_div_i(rem, kUmmaK);
            for (int j = 0; j < nk; ++j)
              tc_mma_bf16(d, smem_desc_k128(a_addr + 32u * j), smem_desc_k128(b_addr + 32u * j), idesc,
                          (kb > 0 || j > 0) ? 1u : 0u);
            tc_commit(&empty[stage]);
          }
          __syncwarp();
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok && lane == 0) tc_commit(&acc_full[ab]);
        __syncwarp();
      }
      if (lane == 0) {
        tc_commit(mma_done);
        mbar_wait_drain(mma_done, 0, kDrainNs);
      }
      __syncwarp();
    }
  } else {
    const int q = warp & 3;
    const int lrow = q * 32 + lane;  // row of the tile (TMEM lane) this thread owns
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const bool leader = (warp == 2 && lane == 0);
    const int et = threadIdx.x - 64;   // epilogue thread index, 0..511
    // four warps per TMEM lane quadrant, each 32 of the tile's 128 columns (bn = 128)
    const int c = ((warp - 2) >> 2) * 32;
    float amax = 0.0f;   // kPreAmax: this thread's max|W_eff|
    float inv6g = 0.0f;
    if (kOut == kPreNvfp4) {
      // the global scale: given, or amax / (6 * 448) from the amax pass's partial maxima
      pdl_wait_prior_grid();
      float g;
      if (p.scale_given) {
        g = *p.gscale;
      } else {
        float m = 0.0f;
        for (int i = et; i < p.n_partials; i += kPreThreads - 64) m = fmaxf(m, p.partials[i]);
        g = __fdiv_rn(epilogue_max(m, red, warp, lane), 2688.0f);
        if (blockIdx.x == 0 && et == 0) *p.gscale = g;
      }
      const float six_g = __fmul_rn(6.0f, g);
      inv6g = six_g > 0.0f ? __frcp_rn(six_g) : 0.0f;
      // 1/d for each scale byte a block can take: d = value(scale) * g, each one rounding
      if (et < 128) {
        const float dd = __fmul_rn(e4m3_value(static_cast<uint32_t>(et)), g);
        inv_tbl[et] = dd > 0.0f ? __frcp_rn(dd) : 0.0f;
      }
      named_bar_sync(1, kPreThreads - 64);
    }
    TileWalk tr(p.total_tiles, p.n_col_tiles, rev);
    int cb = 0, ab = 0;
    uint32_t cph = 0, aph = 0;
    // s of the row this thread owns, loaded one tile ahead (the load's latency is hidden
    // behind a tile)
    uint16_t s_next = (tr.row * kMmaM + lrow < p.out) ? p.s[tr.row * kMmaM + lrow] : uint16_t(0);
    for (int it = 0; it < tr.count; ++it) {
      const int o0 = tr.row * kMmaM;
      const int i0 = tr.col * p.bn;
      const float sc = bf16_to_f32(s_next);
      if (!warp_wait(&c_full[cb], cph, ctl)) break;
      const int o = o0 + lrow;
      uint8_t* ctile = cbuf + cb * cbuf_bytes;
      // W0 row segment: box (c / 64), four 16-byte chunks at swizzled positions.
      uint8_t* rowp = ctile + (c / 64) * kStageA + lrow * 128;
      const int ch0 = (c % 64) / 8;
      uint4 w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) w[h] = *reinterpret_cast<const uint4*>(rowp + (((ch0 + h) ^ (lrow & 7)) << 4));
      // amax / NVFP4 only read the tile: its buffer is free again once every thread has it
      // (the proxy fence orders these reads before the next TMA write into the buffer)
      if (kOut != kPreBf16) {
        fence_proxy_async_smem();
        mbar_arrive(&c_empty[cb]);
      }
      float d[32];
      if (has_mma) {
        if (!warp_wait(&acc_full[ab], aph, ctl)) break;
        tc_fence_after();
        float d0[16], d1[16];
        tmem_ld_16(t_lane + static_cast<uint32_t>(ab * p.bn + c), d0);
        tmem_ld_16(t_lane + static_cast<uint32_t>(ab * p.bn + c + 16), d1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          d[j] = d0[j];
          d[16 + j] = d1[j];
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) d[j] = 0.0f;
      }
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint32_t ww[4] = {w[h].x, w[h].y, w[h].z, w[h].w};
        uint32_t res[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // s * W0 + (U V^T), one rounding each; the quantising epilogues take two columns per
          // instruction (measured: the bf16 store path is 1.5 % slower that way)
          float lo, hi;
          if (kOut == kPreBf16) {
            lo = fmaf(sc, __uint_as_float(ww[e] << 16), d[h * 8 + 2 * e]);
            hi = fmaf(sc, __uint_as_float(ww[e] & 0xFFFF0000u), d[h * 8 + 2 * e + 1]);
          } else {
            ffma2_rn(lo, hi, sc, sc, __uint_as_float(ww[e] << 16), __uint_as_float(ww[e] & 0xFFFF0000u),
                     d[h * 8 + 2 * e], d[h * 8 + 2 * e + 1]);
          }
          if (kOut == kPreBf16) {
            res[e] = pack_bf16x2(lo, hi);
          } else {
            d[h * 8 + 2 * e] = lo;
            d[h * 8 + 2 * e + 1] = hi;
          }
        }
        if (kOut == kPreBf16)
          *reinterpret_cast<uint4*>(rowp + (((ch0 + h) ^ (lrow & 7)) << 4)) = make_uint4(res[0], res[1], res[2], res[3]);
      }
      if (has_mma) {
        tc_fence_before();
        mbar_arrive(&acc_empty[ab]);
      }
      if (kOut == kPreAmax) {
#pragma unroll
        for (int j = 0; j < 30; j += 6)
          amax = fmax3(amax, fmax3(fabsf(d[j]), fabsf(d[j + 1]), fabsf(d[j + 2])),
                       fmax3(fabsf(d[j + 3]), fabsf(d[j + 4]), fabsf(d[j + 5])));
        amax = fmax3(amax, fabsf(d[30]), fabsf(d[31]));
      } else if (kOut == kPreNvfp4) {
        uint2 codes[2];
        const uint32_t sf0 = nvfp4_block(d, inv6g, inv_tbl, &codes[0]);
        const uint32_t sf1 = nvfp4_block(d + 16, inv6g, inv_tbl, &codes[1]);
        const int col = i0 + c;   // first W_eff column of the two blocks (a multiple of 32)
        // codes straight from registers: a warp writes 16 bytes of each of 32 rows, the other
        // warps of the quadrant the rest of those rows' 64 bytes (measured faster than staging
        // the tile for full-row stores behind a per-tile barrier)
        if (o < p.out && col < p.in &&
            dbg_in_bounds(static_cast<int64_t>(o) * p.ldq + min(col + 31, p.in - 1) / 2, dbg_extent(p.out, p.ldq, p.in / 2),
                          p.status)) {
          uint8_t* dst = p.q + static_cast<int64_t>(o) * p.ldq + col / 2;
          if (col + 16 < p.in && p.q16) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(codes[0].x, codes[0].y, codes[1].x, codes[1].y);
          } else {
            *reinterpret_cast<uint2*>(dst) = codes[0];
            if (col + 16 < p.in) *reinterpret_cast<uint2*>(dst + 8) = codes[1];
          }
        }
        if (p.sf_layout == 0) {
          if (o < p.out) {
#pragma unroll
            for (int b = 0; b < 2; ++b)
              if (col + 16 * b < p.in &&
                  dbg_in_bounds(static_cast<int64_t>(o) * p.sf_cols + col / 16 + b, static_cast<int64_t>(p.out) * p.sf_cols,
                                p.status))
                p.sf[static_cast<int64_t>(o) * p.sf_cols + col / 16 + b] = static_cast<uint8_t>(b ? sf1 : sf0);
          }
        } else {
          // 128x4 tiles of 512 bytes, K tiles fastest; row r, column k of a tile at
          // 16 (r mod 32) + 4 (r div 32) + k. Rows past out and columns past in/16 up to the
          // padded shape hold the zero scales of their zero weights.
          const int kb0 = col / 16;
          const int64_t sf_tiles = static_cast<int64_t>(p.n_row_tiles) * p.sf_ktiles;
          if ((kb0 >> 2) < p.sf_ktiles &&
              dbg_in_bounds((static_cast<int64_t>(tr.row) * p.sf_ktiles + (kb0 >> 2)) * 512 + (lrow & 31) * 16 +
                                (lrow >> 5) * 4 + (kb0 & 3) + 1,
                            sf_tiles * 512, p.status))
            *reinterpret_cast<uint16_t*>(p.sf + (static_cast<int64_t>(tr.row) * p.sf_ktiles + (kb0 >> 2)) * 512 +
                                         (lrow & 31) * 16 + (lrow >> 5) * 4 + (kb0 & 3)) =
                static_cast<uint16_t>(sf0 | (sf1 << 8));
        }
      } else {
        // All epilogue threads publish their rows; the leader waits (bounded) for all of
        // them, then one TMA store per 64-column box writes the tile out.
        fence_proxy_async_smem();
        mbar_arrive(&epi_done[cb]);
        if (leader) {
          if (!mbar_wait(&epi_done[cb], cph, ctl)) break;
          for (int j = 0; j < nbox; ++j) tma_store_2d(&p.tm_we, ctile + j * kStageA, i0 + 64 * j, o0);
          tma_store_commit();
          // one store group may still be reading its buffer: release the previous tile's
          if (it > 0) {
            tma_store_wait_read_but_one();
            mbar_arrive(&c_empty[cb == 0 ? p.cbufs - 1 : cb - 1]);
          }
        }
      }
      // next tile of this CTA and its buffers
      tr.next();
      if (it + 1 < tr.count) s_next = (tr.row * kMmaM + lrow < p.out) ? p.s[tr.row * kMmaM + lrow] : uint16_t(0);
      if (++cb == p.cbufs) {
        cb = 0;
        cph ^= 1u;
      }
      ab ^= 1;
      if (ab == 0) aph ^= 1u;
    }
    if (kOut == kPreBf16 && leader) tma_store_wait_all();
    if (kOut == kPreAmax) {
      const float m = epilogue_max(amax, red, warp, lane);
      if (warp == 2 && lane == 0) p.partials[blockIdx.x] = m;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

// ------------------------------------------------------------------------------------
// Bounded-wait self test: one block waits on a barrier nobody arrives on.
// ------------------------------------------------------------------------------------
__global__ void aq_selftest_wait_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const AbortCtl ctl{&abort_flag, status, timeout_ns};
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, ctl);
  __syncthreads();
}

// Checked-build self test: two indices outside their extents, checked but never accessed.
__global__ void aq_selftest_bounds_kernel(int32_t* status) {
  (void)dbg_in_bounds(-1, 8, status);
  (void)dbg_in_bounds(8, 8, status);
}

// ------------------------------------------------------------------------------------
// host-side launch helpers
// ------------------------------------------------------------------------------------
static cudaError_t launch_ex(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             bool pdl, void** args, dim3 cluster = dim3(1, 1, 1)) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster.x * cluster.y * cluster.z > 1) {
    attrs[n].id = cudaLaunchAttributeClusterDimension;
    attrs[n].val.clusterDim.x = cluster.x;
    attrs[n].val.clusterDim.y = cluster.y;
    attrs[n].val.clusterDim.z = cluster.z;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_gemm(const GemmParams& p, int grid, size_t smem, cudaStream_t st, bool pdl) {
  void* args[] = {const_cast<GemmParams*>(&p)};
  if (p.cluster > 1)
    return launch_ex(reinterpret_cast<const void*>(&aq_gemm_kernel<true, false>), dim3(grid), dim3(kGemmThreads), smem,
                     st, pdl, args, dim3(2, 1, 1));
  if (p.swap)
    return launch_ex(reinterpret_cast<const void*>(&aq_gemm_kernel<false, true>), dim3(grid), dim3(kGemmThreads), smem,
                     st, pdl, args);
  return launch_ex(reinterpret_cast<const void*>(&aq_gemm_kernel<false, false>), dim3(grid), dim3(kGemmThreads), smem,
                   st, pdl, args);
}

cudaError_t gemm_max_clusters(size_t smem, int cluster, int* n) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = cluster;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(n, reinterpret_cast<const void*>(&aq_gemm_kernel<true, false>), &cfg);
}

cudaError_t launch_finalize(const FinalizeParams& p, int blocks, cudaStream_t st, bool pdl) {
  void* args[] = {const_cast<FinalizeParams*>(&p)};
  const dim3 grid(blocks, p.M);
  return launch_ex(reinterpret_cast<const void*>(&aq_finalize_kernel), grid, dim3(kFinRows), 0, st, pdl, args);
}

cudaError_t launch_transpose(const TransposeParams& p, int max_r, cudaStream_t st, bool pdl) {
  void* args[] = {const_cast<TransposeParams*>(&p)};
  dim3 grid((p.K + 31) / 32, (max_r + 31) / 32, p.nseg);
  return launch_ex(reinterpret_cast<const void*>(&aq_transpose_kernel), grid, dim3(256), 0, st, pdl,
                   args);
}

cudaError_t launch_precompute(const PrecomputeParams& p, int grid, size_t smem, cudaStream_t st,
                              bool pdl, int out_kind) {
  void* args[] = {const_cast<PrecomputeParams*>(&p)};
  const void* fn = out_kind == kPreAmax    ? reinterpret_cast<const void*>(&aq_precompute_kernel<kPreAmax>)
                   : out_kind == kPreNvfp4 ? reinterpret_cast<const void*>(&aq_precompute_kernel<kPreNvfp4>)
                                           : reinterpret_cast<const void*>(&aq_precompute_kernel<kPreBf16>);
  return launch_ex(fn, dim3(grid), dim3(kPreThreads), smem, st, pdl, args);
}

cudaError_t launch_bounds_selftest(int32_t* status, cudaStream_t st) {
  void* args[] = {&status};
  return launch_ex(reinterpret_cast<const void*>(&aq_selftest_bounds_kernel), dim3(1), dim3(1), 0, st, false, args);
}

cudaError_t launch_bounded_wait_selftest(int32_t* status, uint64_t timeout_ns, cudaStream_t st) {
  void* args[] = {&status, &timeout_ns};
  return launch_ex(reinterpret_cast<const void*>(&aq_selftest_wait_kernel), dim3(1), dim3(32), 0, st,
                   false, args);
}

cudaError_t configure_kernels(int device, size_t max_smem) {
  (void)device;
  cudaError_t e;
  const int s = static_cast<int>(max_smem);
  if ((e = cudaFuncSetAttribute(aq_gemm_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, s))) return e;
  if ((e = cudaFuncSetAttribute(aq_gemm_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, s))) return e;
  if ((e = cudaFuncSetAttribute(aq_gemm_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, s))) return e;
  if ((e = configure_decode(max_smem))) return e;
  if ((e = configure_decode2(max_smem))) return e;
  if ((e = cudaFuncSetAttribute(aq_precompute_kernel<kPreBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, s)))
    return e;
  if ((e = cudaFuncSetAttribute(aq_precompute_kernel<kPreAmax>, cudaFuncAttributeMaxDynamicSharedMemorySize, s)))
    return e;
  if ((e = cudaFuncSetAttribute(aq_precompute_kernel<kPreNvfp4>, cudaFuncAttributeMaxDynamicSharedMemorySize, s)))
    return e;
  return cudaSuccess;
}

int32_t* device_status_ptr(int device, cudaError_t* err) {
  (void)device;
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_device_status);
  return static_cast<int32_t*>(p);
}

}  // namespace aq
