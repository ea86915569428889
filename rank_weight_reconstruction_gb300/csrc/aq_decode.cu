// aq_decode.cu -- the decode kernel (M <= 32 tokens) of the reconstruction linear
//   y = s . (W0 x) + U (V^T x)            ("How attnquant works", "The reconstruction identity")
//
// At decode the work is an HBM stream of W0 with a tiny contraction per element, so the
// design is about keeping every SM's memory pipe full and the critical path short:
//   * every W0-streaming CTA owns a balanced, contiguous range of output rows of one
//     family over the whole K, so no partial sum of y ever leaves the CTA;
//   * warp 0 feeds a TMA ring (W0 boxes of the CTA's rows x 64, x boxes tok_tile x 64,
//     128-byte swizzle); warps 1..8 split the rows into 16-row slabs and, when there are
//     fewer than 8 slabs, split K between the warps of a slab; they run the M <= 32
//     contraction with mma.sync (m16n8k16, bf16 in, fp32 accumulate) from ldmatrix
//     fragments and add the warps' partial sums in shared memory in a fixed order.
//     A tcgen05.mma with M = 128, K = 16 costs about 148 cycles at any N on this part, so
//     one issuing thread moving a 128 x 16 W0 slice per instruction cannot keep up with
//     HBM, while eight warps of mma.sync use a small fraction of their rate here;
//   * a few extra CTAs compute t = V^T x, each over a slice of `in`, add their partial
//     sums in shared memory and then once per element into an fp32 accumulator in the
//     workspace's sync region; the streaming CTAs wait for them only in their epilogue,
//     y = RN_bf16(s * z + U t); the last CTA to finish clears the sync region.
#include <cuda.h>
#include <cuda_runtime.h>

#include "aq_internal.h"
#include "aq_ptx.cuh"

namespace aq {
namespace {

__device__ __forceinline__ uint8_t* align_1k(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Transposed load of two 8x8 b16 tiles (rows given by lanes 0..15): the B fragment of
// m16n8k16 from a [k][n] row-major tile.
__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Every lane waits; the outcome is made warp-uniform because ldmatrix and mma.sync that
// follow are warp-collective.
__device__ __forceinline__ bool warp_wait_all(uint64_t* bar, uint32_t parity, const AbortCtl& ctl) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, ctl)) != 0;
}

// Barrier of the 256 consumer threads on an mbarrier, so that a wait that never ends is
// bounded like every other wait in the kernel.
__device__ __forceinline__ bool cons_sync(uint64_t* bar, uint32_t& phase, const AbortCtl& ctl) {
  mbar_arrive(bar);
  const bool ok = mbar_wait(bar, phase, ctl);
  phase ^= 1u;
  return ok;
}

__device__ __forceinline__ int seg_of_cta(const DecodeParams& p, int g) {
  int si = 0;
#pragma unroll
  for (int j = 1; j < kMaxSeg; ++j)
    if (j < p.nseg && g >= p.seg[j].cta_begin) si = j;
  return si;
}

}  // namespace

// Shared-memory address of 16-byte chunk `c` of k block `b`, row `r` of a stage's W0 (or
// per-stage x) region, for the two box layouts (3-D: rows (r, b) interleaved; 2-D: one
// box per k block), both with the 128-byte swizzle.
__device__ __forceinline__ uint32_t stage_addr(uint32_t base, int w3d, int kbox, uint32_t box_bytes, int r, int b,
                                               int c) {
  if (w3d) {
    const int srow = r * kbox + b;
    return base + srow * 128 + ((c ^ (srow & 7)) << 4);
  }
  return base + b * box_bytes + r * 128 + ((c ^ (r & 7)) << 4);
}

// header: full[kMaxStages], empty[kMaxStages], cbar, vbar, tbar, two ints, then the s buffers
static_assert((2 * kMaxStages + 3) * 8 + 8 <= kSBufOffset, "s buffers overlap the barriers");
static_assert(kSBufOffset + 2 * kSBufBytes <= kHeaderBytes, "s buffers exceed the header");
static_assert(((kMmaM + 14) / 8) * 16 <= kSBufBytes, "s buffer too small for a 128-row chunk");

template <int NT>
__global__ void __launch_bounds__(kDecThreads, 2) aq_decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1k(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint64_t* cbar = empty + kMaxStages;
  uint64_t* vbar = cbar + 1;
  uint64_t* tbar = vbar + 1;   // t of this CTA's family is in shared memory (from the t CTAs)
  int* abort_flag = reinterpret_cast<int*>(tbar + 1);
  int* bcast = abort_flag + 1;
  uint8_t* epi = smem + kHeaderBytes;
  uint8_t* xres = epi + p.epi_bytes;
  uint8_t* vres = xres + p.xres_bytes;
  uint8_t* ures = vres + p.vres_bytes;
  uint8_t* ring = ures + p.ures_bytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grid = gridDim.x;
  const int cta = blockIdx.x;
  const bool t_cta = cta < p.t_ctas;
  const AbortCtl ctl{abort_flag, p.status, p.timeout_ns};
  constexpr int kTok = NT * 8;          // tokens per CTA tile: 8, 16 or 32
  constexpr int kMT = (NT + 1) / 2;      // 16-row tiles of tokens (local t, where tokens are rows)

  // this CTA's family and rows (streaming CTAs only)
  const int g = cta - p.t_ctas;
  const int si = t_cta ? 0 : seg_of_cta(p, g);
  const DecodeSeg& sg = p.seg[si];
  const int l = g - sg.cta_begin;
  const int R = sg.chunk_rows;
  const int nstage = (p.nkb + p.kbox - 1) / p.kbox;
  // Every streaming CTA reads the same x blocks; starting each CTA at a different k stage
  // spreads those reads over the L2 slices instead of all SMs hitting one block at once.
  const int rot = t_cta ? 0 : (g * 7) % nstage;
  const uint32_t xbox_bytes = static_cast<uint32_t>(p.tok_tile) * 128u;
  const bool local_t = !t_cta && p.t_local && sg.r > 0;
  // t from the t CTAs: small tiles are fetched early by lanes 1-31 of warp 0, large ones
  // (where 31 lanes would need many round trips) by all consumers in the first epilogue
  const bool early_t = !t_cta && sg.r > 0 && p.t_ctas > 0 && kTok * sg.r16 <= kEarlyTMax;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecConsumers / 32);
    }
    mbar_init(cbar, kDecConsumers);
    mbar_init(vbar, 1);
    mbar_init(tbar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    if (t_cta) {
      tma_prefetch_desc(&p.tm_xt);
      for (int j = 0; j < p.nseg; ++j)
        if (p.seg[j].r > 0) tma_prefetch_desc(&p.seg[j].tm_v);
    } else {
      tma_prefetch_desc(&sg.tm_w);
      if (!p.x_res) tma_prefetch_desc(&p.tm_x);
      if (local_t) tma_prefetch_desc(&sg.tm_v);
    }
  }
  // Release of the next kernel in the stream (griddepcontrol.launch_dependents; the first
  // thread of a CTA that issues it releases the whole CTA). Its CTAs then start their own
  // weight prefetch, which competes with this call's activation reads. Where those reads are
  // few and the rest of the call runs from shared memory (x resident, t computed locally),
  // the next call's weights are better on their way early: release now. Where x rides with
  // every W0 stage, or t comes from the t CTAs' reads of x, release only once this CTA's
  // activations have arrived (late_release).
  if (!p.late_release) pdl_launch_dependents();
  __syncthreads();

  if (warp == 0) {
    // ---------------- TMA producer (streaming CTAs) ----------------
    if (!t_cta && lane == 0) {
      int total = 0;
      for (int ch = 0; ch < sg.chunks; ++ch)
        if ((l * sg.chunks + ch) * R < sg.rows) total += nstage;
      const int pre = total < p.stages ? total : p.stages;
      uint32_t filled = 0, fill_par = 0;
      auto issue = [&](int q, int slot, bool weights, bool acts) {
        const int ch = q / nstage;
        const int st = (q - ch * nstage + rot) % nstage;
        const int row0 = (l * sg.chunks + ch) * R;
        const int kb0 = st * p.kbox;
        const int nb = min(p.kbox, p.nkb - kb0);
        uint8_t* base = ring + static_cast<size_t>(slot) * p.stage_bytes;
        uint8_t* xbase = base + p.wregion;
        if (weights) {
          // a 3-D box always covers kbox blocks (those past K read as zeros and still count)
          const uint32_t nbox = p.w3d ? static_cast<uint32_t>(p.kbox) : static_cast<uint32_t>(nb);
          const uint32_t xb = p.x_res ? 0u : static_cast<uint32_t>(p.M) * 128u;
          mbar_arrive_expect_tx(&full[slot], nbox * (static_cast<uint32_t>(R) * 128u + xb));
          if (p.w3d) {
            tma_load_3d(base, &sg.tm_w, 0, kb0, row0, &full[slot]);
          } else {
            for (int b = 0; b < nb; ++b)
              tma_load_2d_plain(base + b * p.wbox_bytes, &sg.tm_w, (kb0 + b) * kBK, row0, &full[slot]);
          }
        }
        if (acts && !p.x_res) {
          if (p.w3d) {
            tma_load_3d(xbase, &p.tm_x, 0, kb0, 0, &full[slot]);
          } else {
            for (int b = 0; b < nb; ++b)
              tma_load_2d_plain(xbase + b * xbox_bytes, &p.tm_x, (kb0 + b) * kBK, 0, &full[slot]);
          }
        }
      };
      // W0 of the first stages, and V when this CTA computes t itself, go out before
      // waiting on the previous grid.
      for (int q = 0; q < pre; ++q) {
        issue(q, q, true, false);
        filled |= 1u << q;
      }
      if (p.l2_prefetch) {
        // the rest of this CTA's W0 share streams into L2 now, while the previous call
        // finishes; after the dependency wait its stages then load from L2
        for (int q = pre; q < total; ++q) {
          const int ch = q / nstage;
          const int st = (q - ch * nstage + rot) % nstage;
          const int row0 = (l * sg.chunks + ch) * R;
          const int kb0 = st * p.kbox;
          if (p.w3d) {
            tma_prefetch_l2_3d(&sg.tm_w, 0, kb0, row0);
          } else {
            const int nb = min(p.kbox, p.nkb - kb0);
            for (int b = 0; b < nb; ++b) tma_prefetch_l2_2d(&sg.tm_w, (kb0 + b) * kBK, row0);
          }
        }
      }
      if (local_t) {
        const int nvb = (p.K + p.vbox - 1) / p.vbox;
        const uint32_t vb = static_cast<uint32_t>(p.vbox) * sg.r8 * 2u;
        mbar_arrive_expect_tx(vbar, nvb * vb);
        for (int b = 0; b < nvb; ++b) tma_load_2d_plain(vres + b * vb, &sg.tm_v, 0, b * p.vbox, vbar);
      }
      // x row g of the first M streaming CTAs into L2 while the previous kernel finishes,
      // so the reads of x after the dependency wait hit L2 (rows are 16-byte aligned and
      // K * 2 bytes long, a multiple of 16)
      if (g < p.M) prefetch_l2_bulk(p.x + static_cast<int64_t>(g) * p.ldx, static_cast<uint32_t>(p.K) * 2u);
      pdl_wait_prior_grid();
      for (int q = 0; q < pre; ++q) issue(q, q, false, true);
      int slot = pre == p.stages ? 0 : pre;
      uint32_t phase = pre == p.stages ? 1u : 0u;
      bool ok = true;
      for (int q = pre; q < total; ++q) {
        if (!mbar_wait(&empty[slot], phase ^ 1u, ctl)) {
          ok = false;
          break;
        }
        issue(q, slot, true, true);
        filled |= 1u << slot;
        fill_par = (fill_par & ~(1u << slot)) | (phase << slot);
        if (++slot == p.stages) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        for (int s = 0; s < p.stages; ++s)
          if (filled & (1u << s)) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&full[s], (fill_par >> s) & 1u))
              if (global_timer_ns() - t0 > 20000000ull) break;
          }
      }
      if (local_t) {  // no copy may still be landing when the CTA exits
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(vbar, 0u))
          if (global_timer_ns() - t0 > 20000000ull) break;
      }
    }
    if (!t_cta && lane > 0 && p.t_ctas > 0 && (early_t || sg.r == 0)) {
      // ---- t from the t CTAs, fetched by lanes 1-31 of this warp while lane 0 feeds the
      // ring and the consumers stream W0: wait for all t CTAs to publish, write t_hi / t_lo
      // for the epilogue, then count this CTA as done with the accumulator (t CTA 0 clears
      // it once every streaming CTA has) ----
      constexpr uint32_t kLanes = 0xFFFFFFFEu;
      pdl_wait_prior_grid();
      if (early_t) {
        bool got = true;
        if (lane == 1) {
          const uint64_t t0 = global_timer_ns();
          while (ld_acquire_gpu(&p.counters[0]) < p.t_ctas) {
            if (*reinterpret_cast<volatile int*>(abort_flag) || global_timer_ns() - t0 > p.timeout_ns) {
              *reinterpret_cast<volatile int*>(abort_flag) = 1;
              atomicExch(p.status, kStatusTimeout);
              got = false;
              break;
            }
            __nanosleep(64);
          }
        }
        got = __shfl_sync(kLanes, got ? 1 : 0, 1) != 0;
        if (got) {
          const int rs16 = sg.r16 + 8;
          uint16_t* tbh = reinterpret_cast<uint16_t*>(reinterpret_cast<float*>(epi) + p.ts_off);
          uint16_t* tbl = tbh + kTok * rs16;
          const int nt_el = kTok * sg.r16;
          for (int base = lane - 1; base < nt_el; base += 4 * 31) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {   // four loads in flight per lane
              const int idx = base + u * 31;
              const int m = idx / sg.r16, k = idx - m * sg.r16;
              v[u] = (idx < nt_el && m < p.M && k < sg.r) ? __ldcg(&p.t_acc[m * p.r_total + sg.t_col + k]) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int idx = base + u * 31;
              if (idx < nt_el) {
                const int m = idx / sg.r16, k = idx - m * sg.r16;
                const uint16_t h = f32_to_bf16_rn(v[u]);
                tbh[m * rs16 + k] = h;
                tbl[m * rs16 + k] = f32_to_bf16_rn(v[u] - bf16_to_f32(h));
              }
            }
          }
        }
        __syncwarp(kLanes);
      }
      if (lane == 1) {
        red_release_gpu_add(&p.counters[1], 1);
        if (early_t) mbar_arrive(tbar);   // also when the wait gave up: the epilogue sees the abort
      }
    }
  } else {
    const int cw = warp - 1;              // consumer warp 0..7
    const int ct = threadIdx.x - 32;      // 0..255
    const int gq = lane >> 2, qq = lane & 3;
    uint32_t cph = 0;
    bool ok = true;

    if (t_cta) {
      // ---- t = V^T x over this CTA's slice of `in`: every box of V and x is requested
      // at once (one round trip), V before the dependency wait ----
      // slices are whole 16-row k steps of the mma (and so start 16-byte aligned, as a TMA
      // box's innermost coordinate must)
      const int ks = ((p.K + p.t_ctas - 1) / p.t_ctas + 15) & ~15;
      const int i0 = cta * ks;
      const int i1 = min(p.K, i0 + ks);
      const int n = max(0, i1 - i0);
      const int nvb = (ks + p.vbox - 1) / p.vbox;
      const int trows = nvb * p.vbox;                                // staged rows of `in`
      const int ntot = p.M * p.r_total;
      const int tacc_bytes = (ntot * 4 + 1023) & ~1023;
      uint8_t* stage_area = epi + tacc_bytes;                        // per family [trows][r8]
      const uint16_t* xsb =                                          // per box [M][vbox]
          reinterpret_cast<const uint16_t*>(stage_area + static_cast<size_t>(trows) * p.r8_total * 2);
      // TMA writes shared memory at 128-byte aligned addresses: x boxes are spaced so
      const int xbs = ((p.vbox * p.M * 2 + 127) & ~127) / 2;        // elements per x box
      if (ct == 0 && n > 0) {
        mbar_arrive_expect_tx(&full[0], static_cast<uint32_t>(trows) * (p.r8_total + p.M) * 2u);  // box bytes
        int col = 0;
        for (int j = 0; j < p.nseg; ++j) {
          if (p.seg[j].r > 0)
            for (int b = 0; b < nvb; ++b)
              tma_load_2d_plain(stage_area + (static_cast<size_t>(trows) * col + b * p.vbox * p.seg[j].r8) * 2,
                                &p.seg[j].tm_v, 0, i0 + b * p.vbox, &full[0]);
          col += p.seg[j].r8;
        }
        pdl_wait_prior_grid();
        for (int b = 0; b < nvb; ++b)
          tma_load_2d_plain(const_cast<uint16_t*>(xsb) + b * xbs, &p.tm_xt, i0 + b * p.vbox, 0, &full[0]);
      }
      pdl_wait_prior_grid();
      if (n > 0) ok = mbar_wait(&full[0], 0u, ctl);
      if (p.late_release) pdl_launch_dependents();
      // t on the tensor cores: work items are (family, 8-column n tile, 16-token tile); when
      // there are fewer than 8 items, several warps split an item's k steps (ksplit) and
      // their fragments are summed in a fixed order. A: x [tokens][k] per box; B: the V
      // slice [k][r8] of a family (ldmatrix.trans). The slice length is a multiple of 16, so
      // every k step is whole; rows past K read as zero.
      const int kmt = (p.M + 15) / 16;
      int items = 0;
      for (int j = 0; j < p.nseg; ++j) items += (p.seg[j].r8 / 8) * kmt;
      const int ksplit = items >= 8 ? 1 : 8 / items;
      const int nsteps = (n + 15) / 16;
      const uint32_t vbase0 = smem_u32(stage_area);
      const uint32_t xbase0 = smem_u32(xsb);
      float* part = reinterpret_cast<float*>(stage_area);   // [items * ksplit][32 lanes][4], after the loop
      float fr[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      int my_item = -1;
      // item -> family, its column block in the staged V, n tile, token tile
      auto locate = [&](int item, int& j, int& vcol, int& nt, int& mt) {
        j = 0;
        vcol = 0;
        int rest = item;
        while (j < p.nseg - 1 && rest >= (p.seg[j].r8 / 8) * kmt) {
          rest -= (p.seg[j].r8 / 8) * kmt;
          vcol += p.seg[j].r8;
          ++j;
        }
        nt = rest / kmt;
        mt = rest - nt * kmt;
      };
      const int npairs = items * ksplit;
      for (int pr = cw; ok && pr < npairs; pr += 8) {
        const int item = pr / ksplit, kpart = pr - item * ksplit;
        int j, vcol, nt, mt;
        locate(item, j, vcol, nt, mt);
        const int r8 = p.seg[j].r8;
        const uint32_t vbase = vbase0 + static_cast<uint32_t>(trows) * vcol * 2;
        const int m = min(mt * 16 + (lane & 15), p.M - 1);   // rows past M repeat M-1; dropped
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int st = kpart; st < nsteps; st += ksplit) {
          const int k0 = st * 16;
          const int b = k0 / p.vbox, kk = k0 - b * p.vbox;
          uint32_t a0, a1, a2, a3, b0, b1;
          ldsm_x4(xbase0 + (b * xbs + m * p.vbox + kk + (lane >> 4) * 8) * 2, a0, a1, a2, a3);
          ldsm_x2_trans(vbase + ((k0 + (lane & 15)) * r8 + nt * 8) * 2, b0, b1);
          mma_16816(acc, a0, a1, a2, a3, b0, b1);
        }
        if (ksplit == 1) {
          // the only warp on this item: straight to the global accumulator
          const int gq = lane >> 2, qq = lane & 3;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int mm = mt * 16 + gq + 8 * (e >> 1), kc = nt * 8 + 2 * qq + (e & 1);
            if (mm < p.M && kc < p.seg[j].r) atomicAdd(&p.t_acc[mm * p.r_total + p.seg[j].t_col + kc], acc[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) fr[e] = acc[e];
          my_item = pr;
        }
      }
      if (ksplit > 1) {
        // partial fragments over the (no longer read) staging, then a fixed-order sum
        if (ok) ok = cons_sync(cbar, cph, ctl);
        if (ok && my_item >= 0) {
#pragma unroll
          for (int e = 0; e < 4; ++e) part[(my_item * 32 + lane) * 4 + e] = fr[e];
        }
        if (ok) ok = cons_sync(cbar, cph, ctl);
        if (ok && cw < items) {
          const int item = cw;
          int j, vcol, nt, mt;
          locate(item, j, vcol, nt, mt);
          const int gq = lane >> 2, qq = lane & 3;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v = 0.0f;
            for (int kp = 0; kp < ksplit; ++kp) v += part[((item * ksplit + kp) * 32 + lane) * 4 + e];
            const int mm = mt * 16 + gq + 8 * (e >> 1), kc = nt * 8 + 2 * qq + (e & 1);
            if (mm < p.M && kc < p.seg[j].r) atomicAdd(&p.t_acc[mm * p.r_total + p.seg[j].t_col + kc], v);
          }
        }
      }
      if (ok) {
        __threadfence();
        ok = cons_sync(cbar, cph, ctl);
        if (ok && ct == 0) atomicAdd(&p.counters[0], 1);
      }
      if (ok && cta == 0) {
        // Every streaming CTA counts itself once it has read t: then the accumulator and
        // both counters go back to zero for the next call (the sync region's invariant).
        if (ct == 0) {
          bool all = true;
          const uint64_t t0 = global_timer_ns();
          while (ld_acquire_gpu(&p.counters[1]) < grid - p.t_ctas) {
            if (*reinterpret_cast<volatile int*>(abort_flag) || global_timer_ns() - t0 > p.timeout_ns) {
              *reinterpret_cast<volatile int*>(abort_flag) = 1;
              atomicExch(p.status, kStatusTimeout);
              all = false;
              break;
            }
            __nanosleep(128);
          }
          *bcast = all ? 1 : 0;
        }
        ok = cons_sync(cbar, cph, ctl);
        if (ok && *bcast) {
          for (int idx = ct; idx < p.M * p.r_total; idx += kDecConsumers) p.t_acc[idx] = 0.0f;
          ok = cons_sync(cbar, cph, ctl);
          if (ok && ct == 0) {
            p.counters[0] = 0;
            p.counters[1] = 0;
            __threadfence();
          }
        }
      }
    } else {
      // s and the U rows of a chunk go to shared memory with cp.async when the chunk
      // starts (the first chunk's before the dependency wait: both are weights), so the
      // epilogue reads nothing from global memory. A load issued there would wait behind
      // this SM's whole queue of W0 traffic.
      auto sbuf = [&](int ch) { return reinterpret_cast<uint16_t*>(smem + kSBufOffset + (ch & 1) * kSBufBytes); };
      auto stage_ch = [&](int ch) {
        const int row0 = (l * sg.chunks + ch) * R;
        // s[row0 - (row0 & 7) ...] in 16-byte pieces, zero past the last row
        const int sb = row0 & ~7;
        const int spieces = (row0 + R - sb + 7) / 8;
        for (int idx = ct; idx < spieces; idx += kDecConsumers) {
          const int e0 = sb + idx * 8;
          cp_async_16_zfill(smem_u32(sbuf(ch)) + idx * 16, sg.s + e0, max(0, min(16, (sg.rows - e0) * 2)));
        }
        if (sg.r > 0) {   // U rows [R][r16], zero past r
          const uint32_t ub = smem_u32(ures) + (ch & 1) * p.ubuf_bytes;
          const int pieces = sg.r16 / 8;
          const int rs16 = sg.r16 + 8;   // row stride: 16 bytes of padding keep ldmatrix conflict-free
          for (int idx = ct; idx < R * pieces; idx += kDecConsumers) {
            const int rr = idx / pieces, c = idx - rr * pieces;
            const int o = row0 + rr;
            if (o < sg.rows)
              cp_async_16_zfill(ub + (rr * rs16 + c * 8) * 2, sg.U + static_cast<int64_t>(o) * sg.ldu + c * 8,
                                max(0, min(16, (sg.r - c * 8) * 2)));
          }
        }
        cp_async_commit();
      };
      stage_ch(0);
      pdl_wait_prior_grid();
      // ---- x resident in shared memory (dense rows, zero beyond K) ----
      if (p.x_res) {
        uint16_t* xs = reinterpret_cast<uint16_t*>(xres);
        const int kp = p.nkb * kBK;
        if ((p.K & 7) == 0) {
          const int per_row = kp / 8;
          const int tot = p.M * per_row;
          for (int base = ct; base < tot; base += 8 * kDecConsumers) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int idx = base + u * kDecConsumers;
              const int m = idx / per_row, c8 = idx - m * per_row;
              v[u] = (idx < tot && c8 * 8 < p.K)
                         ? __ldg(reinterpret_cast<const uint4*>(p.x + static_cast<int64_t>(m) * p.ldx) + c8)
                         : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int idx = base + u * kDecConsumers;
              if (idx < tot) {
                const int m = idx / per_row, c8 = idx - m * per_row;
                *reinterpret_cast<uint4*>(xs + m * p.xs_ld + c8 * 8) = v[u];
              }
            }
          }
        } else {
          for (int idx = ct; idx < p.M * kp; idx += kDecConsumers) {
            const int m = idx / kp, k = idx - m * kp;
            xs[m * p.xs_ld + k] = k < p.K ? p.x[static_cast<int64_t>(m) * p.ldx + k] : 0;
          }
        }
        ok = cons_sync(cbar, cph, ctl);
        if (p.late_release) pdl_launch_dependents();
      }
      float* red = reinterpret_cast<float*>(epi);          // [nslab * kg][16][kTok]
      // t of this CTA's family as a bf16 pair, t = t_hi + t_lo to about 16 significant
      // bits, each [kTok][r16] and zero past M and r: the B operand of U t in the epilogue
      // (rows padded by 16 bytes, like the staged U rows, so ldmatrix is conflict-free)
      const int rs16 = sg.r16 + 8;
      uint16_t* tbh = reinterpret_cast<uint16_t*>(red + p.ts_off);
      uint16_t* tbl = tbh + kTok * rs16;
      auto put_t = [&](int m, int k, float v) {
        const uint16_t h = f32_to_bf16_rn(v);
        tbh[m * rs16 + k] = h;
        tbl[m * rs16 + k] = f32_to_bf16_rn(v - bf16_to_f32(h));
      };
      const uint32_t xres_base = smem_u32(xres);
      // ---- t = V^T x of this CTA's family, from V staged before the dependency wait:
      // warps split `in` in 16-wide steps, mma.sync per step, fixed-order sum over warps ----
      if (ok && local_t) {
        ok = warp_wait_all(vbar, 0u, ctl);
        if (ok) {
          float* part = red;                                   // [8][kMT * 16][r8]
          const int r8 = sg.r8;
          const int ntn = r8 / 8;
          const uint32_t vbase = smem_u32(vres);
          float ta[kMT][kDecLocalMaxR8 / 8][4];
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
            for (int nt = 0; nt < kDecLocalMaxR8 / 8; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) ta[mt][nt][e] = 0.0f;
          const int nks = (p.K + 15) / 16;
          for (int kk = cw; kk < nks; kk += 8) {
            const int k0 = kk * 16;
            uint32_t bf[kDecLocalMaxR8 / 8][2];
#pragma unroll
            for (int nt = 0; nt < kDecLocalMaxR8 / 8; ++nt)
              if (nt < ntn) ldsm_x2_trans(vbase + ((k0 + (lane & 15)) * r8 + nt * 8) * 2, bf[nt][0], bf[nt][1]);
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt) {
              if (mt * 16 < p.M) {
                const int m = min(mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, p.M - 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(xres_base + (m * p.xs_ld + k0 + (lane >> 4) * 8) * 2, a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < kDecLocalMaxR8 / 8; ++nt)
                  if (nt < ntn) mma_16816(ta[mt][nt], a0, a1, a2, a3, bf[nt][0], bf[nt][1]);
              }
            }
          }
#pragma unroll
          for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
            for (int nt = 0; nt < kDecLocalMaxR8 / 8; ++nt)
              if (nt < ntn)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int m = mt * 16 + gq + 8 * h, c = nt * 8 + 2 * qq;
                  part[(cw * kMT * 16 + m) * r8 + c] = ta[mt][nt][2 * h];
                  part[(cw * kMT * 16 + m) * r8 + c + 1] = ta[mt][nt][2 * h + 1];
                }
          ok = cons_sync(cbar, cph, ctl);
          if (ok) {
            for (int idx = ct; idx < kTok * sg.r16; idx += kDecConsumers) {
              const int m = idx / sg.r16, k = idx - m * sg.r16;
              float v = 0.0f;
              if (m < p.M && k < sg.r)
                for (int w = 0; w < 8; ++w) v += part[(w * kMT * 16 + m) * r8 + k];
              put_t(m, k, v);
            }
          }
        }
      }
      // ---- stream this CTA's rows of W0 ----
      const int nslab = (R + 15) / 16;
      const int kg = 8 / nslab;                 // warps sharing one slab (split over K)
      const bool active = cw < nslab * kg;
      const int slab = cw / kg, kgi = cw - slab * kg;
      // B from resident x: this lane's token row in each n tile (rows past M repeat row
      // M-1, so every read stays inside x; those output columns are dropped) and k pair
      uint32_t xl[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) xl[nt] = xres_base + (min(8 * nt + gq, p.M - 1) * p.xs_ld + 2 * qq) * 2;

      int slot = 0;
      uint32_t phase = 0;
      for (int ch = 0; ok && ch < sg.chunks; ++ch) {
        const int row0 = (l * sg.chunks + ch) * R;
        if (row0 >= sg.rows) break;
        if (ch > 0) stage_ch(ch);
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
        // this lane's A row (rows past the chunk read row R-1 again; their sums are dropped,
        // so a stage holds exactly the chunk's rows)
        const int arow = min(16 * slab + (lane & 7) + ((lane >> 3) & 1) * 8, R - 1);
        const int ahi = lane >> 4;                                  // 8-wide half of a 16-wide step
        const int arowk = arow * p.kbox;
        const uint32_t arow_off = (arow << 7) + ((ahi ^ (arow & 7)) << 4);
        for (int sq = 0; sq < nstage; ++sq) {
          if (!warp_wait_all(&full[slot], phase, ctl)) {
            ok = false;
            break;
          }
          if (p.late_release && !p.x_res && ch == 0 && sq == 0) pdl_launch_dependents();
          const int st = (sq + rot) % nstage;
          const int nb = min(p.kbox, p.nkb - st * p.kbox);
          if (active) {
            const uint32_t wbase = smem_u32(ring + static_cast<size_t>(slot) * p.stage_bytes);
            const uint32_t xbase = wbase + p.wregion;
            const int kb_base = st * p.kbox;
            // The kg warps of a slab take whole 64-wide k blocks in turn by their index
            // in K (so the split stays balanced across stages), all four 16-wide steps of
            // each. Per block the swizzled row address is computed once; the steps differ
            // only in bits 5-6 of it.
            for (int b = (kgi - kb_base % kg + kg) % kg; b < nb; b += kg) {
              uint32_t rowaddr;
              if (p.w3d) {
                const int srow = arowk + b;
                rowaddr = wbase + (srow << 7) + ((ahi ^ (srow & 7)) << 4);
              } else {
                rowaddr = wbase + b * p.wbox_bytes + arow_off;
              }
              if (p.x_res) {
                const uint32_t xk = static_cast<uint32_t>(kb_base + b) << 7;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint32_t a0, a1, a2, a3;
                  ldsm_x4(rowaddr ^ (j << 5), a0, a1, a2, a3);
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt) {
                    uint32_t b0, b1;
                    const uint32_t ad = xl[nt] + xk + j * 32;
                    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b0) : "r"(ad));
                    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(b1) : "r"(ad + 16));
                    mma_16816(acc[nt], a0, a1, a2, a3, b0, b1);
                  }
                }
              } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  uint32_t a0, a1, a2, a3;
                  ldsm_x4(rowaddr ^ (j << 5), a0, a1, a2, a3);
                  if constexpr (NT == 1) {
                    uint32_t b0, b1;
                    ldsm_x2(stage_addr(xbase, p.w3d, p.kbox, xbox_bytes, lane & 7, b, 2 * j + ((lane >> 3) & 1)), b0,
                            b1);
                    mma_16816(acc[0], a0, a1, a2, a3, b0, b1);
                  } else {
#pragma unroll
                    for (int np = 0; np < NT / 2; ++np) {
                      const int brow = 16 * np + (lane & 7) + (lane >> 4) * 8;
                      uint32_t b0, b1, b2, b3;
                      ldsm_x4(stage_addr(xbase, p.w3d, p.kbox, xbox_bytes, brow, b, 2 * j + ((lane >> 3) & 1)), b0,
                              b1, b2, b3);
                      mma_16816(acc[2 * np], a0, a1, a2, a3, b0, b1);
                      mma_16816(acc[2 * np + 1], a0, a1, a2, a3, b2, b3);
                    }
                  }
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
          if (++slot == p.stages) {
            slot = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // ---- epilogue of this chunk: the lead warp of each slab (kgi == 0) adds its
        // partners' partial sums, runs U t on the tensor cores from the staged U rows and
        // t_hi / t_lo, and writes y = RN(s z + U t) straight from the mma fragments ----
        if (!(ok = cons_sync(cbar, cph, ctl))) break;   // red free
        if (active && kgi > 0) {
          float* my = red + (slab * kg + kgi) * 16 * kTok;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int rr = gq + 8 * h, tok = 8 * nt + 2 * qq;
              my[rr * kTok + tok] = acc[nt][2 * h];
              my[rr * kTok + tok + 1] = acc[nt][2 * h + 1];
            }
        }
        if (early_t && ch == 0) {   // t (from warp 0) stays for later chunks
          if (!(ok = warp_wait_all(tbar, 0u, ctl))) break;
          if (*reinterpret_cast<volatile int*>(abort_flag)) {
            ok = false;
            break;
          }
        } else if (sg.r > 0 && !p.t_local && ch == 0) {   // t stays in shared memory for later chunks
          if (ct == 0) {
            bool ready = true;
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire_gpu(&p.counters[0]) < p.t_ctas) {
              __nanosleep(128);   // many CTAs poll one word: keep the line free for the arrivals
              if (*reinterpret_cast<volatile int*>(abort_flag) || global_timer_ns() - t0 > p.timeout_ns) {
                *reinterpret_cast<volatile int*>(abort_flag) = 1;
                atomicExch(p.status, kStatusTimeout);
                ready = false;
                break;
              }
            }
            *bcast = ready ? 1 : 0;
          }
          if (!(ok = cons_sync(cbar, cph, ctl)) || !*bcast) {
            ok = false;
            break;
          }
          const int nt_el = kTok * sg.r16;
          for (int base = ct; base < nt_el; base += 8 * kDecConsumers) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {   // eight loads in flight per thread
              const int idx = base + u * kDecConsumers;
              const int m = idx / sg.r16, k = idx - m * sg.r16;
              v[u] = (idx < nt_el && m < p.M && k < sg.r) ? __ldcg(&p.t_acc[m * p.r_total + sg.t_col + k]) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int idx = base + u * kDecConsumers;
              const int m = idx / sg.r16, k = idx - m * sg.r16;
              if (idx < nt_el) put_t(m, k, v[u]);
            }
          }
          // all consumers have read t: count this CTA as done with the accumulator
          if (!(ok = cons_sync(cbar, cph, ctl))) break;
          if (ct == 0) red_release_gpu_add(&p.counters[1], 1);
        }
        cp_async_wait_all();
        if (!(ok = cons_sync(cbar, cph, ctl))) break;
        if (active && kgi == 0) {
          for (int k2 = 1; k2 < kg; ++k2) {
            const float* pr = red + (slab * kg + k2) * 16 * kTok;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int rr = gq + 8 * h, tok = 8 * nt + 2 * qq;
                acc[nt][2 * h] += pr[rr * kTok + tok];
                acc[nt][2 * h + 1] += pr[rr * kTok + tok + 1];
              }
          }
          float lw[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) lw[nt][e] = 0.0f;
          if (sg.r > 0) {
            const uint32_t ub = smem_u32(ures) + (ch & 1) * p.ubuf_bytes;
            const uint32_t th_base = smem_u32(tbh), tl_base = smem_u32(tbl);
            const int arow = min(16 * slab + (lane & 7) + ((lane >> 3) & 1) * 8, R - 1);
            for (int k0 = 0; k0 < sg.r16; k0 += 16) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4(ub + (arow * rs16 + k0 + (lane >> 4) * 8) * 2, a0, a1, a2, a3);
              if constexpr (NT == 1) {
                const uint32_t boff = ((lane & 7) * rs16 + k0 + ((lane >> 3) & 1) * 8) * 2;
                uint32_t b0, b1;
                ldsm_x2(th_base + boff, b0, b1);
                mma_16816(lw[0], a0, a1, a2, a3, b0, b1);
                ldsm_x2(tl_base + boff, b0, b1);
                mma_16816(lw[0], a0, a1, a2, a3, b0, b1);
              }
#pragma unroll
              for (int np = 0; np < NT / 2; ++np) {
                const int brow = 16 * np + (lane & 7) + (lane >> 4) * 8;
                const uint32_t boff = (brow * rs16 + k0 + ((lane >> 3) & 1) * 8) * 2;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(th_base + boff, b0, b1, b2, b3);
                mma_16816(lw[2 * np], a0, a1, a2, a3, b0, b1);
                mma_16816(lw[2 * np + 1], a0, a1, a2, a3, b2, b3);
                ldsm_x4(tl_base + boff, b0, b1, b2, b3);
                mma_16816(lw[2 * np], a0, a1, a2, a3, b0, b1);
                mma_16816(lw[2 * np + 1], a0, a1, a2, a3, b2, b3);
              }
            }
          }
          const uint16_t* sv = sbuf(ch);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int row = 16 * slab + gq + 8 * h;
            const int o = row0 + row;
            if (row < R && o < sg.rows) {
              const float sc = bf16_to_f32(sv[o - (row0 & ~7)]);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                  const int m = 8 * nt + 2 * qq + e;
                  const int64_t yi = static_cast<int64_t>(m) * sg.ldy + o;
                  if (m < p.M && dbg_in_bounds(yi, dbg_extent(p.M, sg.ldy, sg.rows), p.status))
                    sg.y[yi] = f32_to_bf16_rn(fmaf(sc, acc[nt][2 * h + e], lw[nt][2 * h + e]));
                }
            }
          }
        }
      }
    }

    if (!t_cta) cp_async_wait_all();   // no copy may still be landing when the CTA exits
  }
  __syncthreads();
}

cudaError_t launch_decode(const DecodeParams& p, int grid, size_t smem, cudaStream_t st, bool pdl) {
  void* args[] = {const_cast<DecodeParams*>(&p)};
  const void* fn = p.tok_tile > 16  ? reinterpret_cast<const void*>(&aq_decode_kernel<4>)
                   : p.tok_tile > 8 ? reinterpret_cast<const void*>(&aq_decode_kernel<2>)
                                    : reinterpret_cast<const void*>(&aq_decode_kernel<1>);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t configure_decode(size_t max_smem) {
  cudaError_t e;
  const int s = static_cast<int>(max_smem);
  if ((e = cudaFuncSetAttribute(aq_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, s))) return e;
  if ((e = cudaFuncSetAttribute(aq_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, s))) return e;
  return cudaFuncSetAttribute(aq_decode_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, s);
}

}  // namespace aq
