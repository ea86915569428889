// aq_decode2.cu -- the cluster decode kernel (M <= 16 tokens) of the reconstruction linear
//   y = s . (W0 x) + U (V^T x)            ("How attnquant works", "The reconstruction identity")
//
// A decode call moves a few MB of weights for a few tokens, so what bounds it is the chain
// of steps after the kernel's dependency wait, and whether the next call can already stream
// its weights while this one finishes. This kernel is built for both:
//   * A cluster of C CTAs owns a range of output rows of one family; CTA q of the cluster
//     covers K slice q of it. Each CTA therefore stages only its slice of V and of x, which
//     keeps every CTA within half of an SM's shared memory: the next call's CTAs fit beside
//     this call's and fill their W0 ring (issued before their dependency wait) while this
//     call computes.
//   * t = V^T x is not a phase of its own. It is formed inside the W0 loop: for every 16-wide
//     k step that a warp owns, the V slice (already in shared memory) supplies the A
//     fragments of V^T through ldmatrix.trans, and the x fragments the W0 product loads anyway
//     are the B operand. The t product is a second, independent mma chain of the same loop.
//   * After the loop every CTA holds partial sums over its K slice of W0 x (its rows) and of
//     t. They are added across the cluster through distributed shared memory, by stores only:
//     each CTA sums its own partials (k-block groups, warps) and pushes, with 16-byte stores
//     into the peers' shared memory, the W0 x sums of the rows peer q finishes (1/C of the
//     cluster's rows) to q and its t to every peer (its own share by plain shared stores; the
//     first push waits on a cluster barrier that every thread arrives on when it starts, so
//     no peer is written before it runs). The remote pushes are asynchronous stores that count
//     their bytes on the receiver's barrier, so a CTA starts its final phase as soon as its
//     own inputs have landed; a second cluster barrier phase, arrived on after the pushes and
//     waited on at exit, keeps every CTA alive while a peer may still push into it. Every CTA
//     adds the C partials it received, in rank order. y = RN_bf16(s * z + U t) is formed in
//     fp32 (U t on the FP32 pipes: r products per output) and rounded once.
// Warp 0 feeds the TMA ring (one lane); warps 1..8 run mma.sync m16n8k16 (bf16 in, fp32
// accumulate). Every wait on an mbarrier is bounded; a CTA whose wait expires records
// AQ_ERR_TIMEOUT, skips the remaining work and still takes part in every barrier, so the
// cluster never waits on a CTA that left.
#include <cuda.h>
#include <cuda_runtime.h>

#include "aq_internal.h"
#include "aq_ptx.cuh"

namespace aq {
namespace {

__device__ __forceinline__ uint8_t* align_1k2(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// shared::cluster address of the same offset in CTA `rank` of the cluster, from a shared::cta
// address.
__device__ __forceinline__ uint32_t mapa_u32(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

// The activations of the fused MLP, in fp32 with CUDA's tanhf / expf: the tanh approximation of
// GELU, v/2 (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))), and SiLU, v / (1 + e^-v).
__device__ __forceinline__ float gated_act(float v, int act) {
  if (act == kActSilu) return v / (1.0f + expf(-v));
  return 0.5f * v * (1.0f + tanhf(0.7978845608028654f * (v + 0.044715f * v * v * v)));
}

// Barrier of the 256 mma warps (named barrier 1). Every consumer thread reaches each call site
// on every path, a failed wait included, so it always completes.
__device__ __forceinline__ void cons_bar() { named_bar_sync(1, kDecConsumers); }

// 128-byte swizzled address of 16-byte chunk c of (row, k block b) in a 3-D box {64, kbox, rows}
// that starts on a 1 KB boundary: line row * kbox + b.
__device__ __forceinline__ uint32_t sw_addr(uint32_t base, int kbox, int row, int b, int c) {
  const int line = row * kbox + b;
  return base + line * 128 + ((c ^ (line & 7)) << 4);
}

// Asynchronous 16-byte store into a peer's shared memory that completes `16 bytes` of the
// transaction count of the peer's mbarrier (both shared::cluster addresses of that CTA).
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, float a, float b, float c, float d,
                                            uint32_t cluster_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   cluster_addr),
               "f"(a), "f"(b), "f"(c), "f"(d), "r"(cluster_bar)
               : "memory");
}

// Bounded wait on a phase that remote CTAs complete (acquire at cluster scope).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, const AbortCtl& ctl) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 31u) == 31u) {
      if (*reinterpret_cast<volatile int*>(ctl.abort_flag)) return false;
      if (global_timer_ns() - t0 > ctl.timeout_ns) {
        *reinterpret_cast<volatile int*>(ctl.abort_flag) = 1;
        atomicExch(ctl.status, kStatusTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void cluster_arrive_relaxed_end() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

// The cluster's start barrier in two halves: every thread arrives (relaxed) when it starts and
// waits before its first access to a peer's shared memory, by then long complete.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

}  // namespace

// kStaged: x and V ride in every stage behind its W0 box (Dec2Params::staged), a separate
// instantiation so that the resident layout keeps its own code
template <int NT, bool kStaged>
__global__ void __launch_bounds__(kDecThreads, 2) aq_decode2_kernel(const __grid_constant__ Dec2Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1k2(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint64_t* xbar = empty + kMaxStages;
  uint64_t* vbar = xbar + 1;
  uint64_t* rbar = vbar + 1;   // the peers' pushes into this CTA (transaction bytes)
  int* abort_flag = reinterpret_cast<int*>(rbar + 1);
  uint8_t* xs = smem + kHeaderBytes;                 // x slice: 3-D box {64, xkb, M}, swizzled
  uint8_t* xs2 = xs + p.x_bytes;                     // gated input: the second slice, same layout
  uint8_t* vs = xs2 + p.x2_bytes;                    // V slice: [kslice][vrow] bf16
  uint8_t* us = vs + p.v_bytes;                      // U rows this CTA finishes: [rf][r16] bf16
  uint8_t* ss = us + p.u_bytes;                      // s of those rows, bf16
  float* tf = reinterpret_cast<float*>(ss + p.s_bytes);  // t over the whole K: [r16][M] fp32
  // what the peers push: per sender rank, W0 x of the rows this CTA finishes [C][M][rf4], then
  // t [C][r16][M]; never aliased, so a peer may push while this CTA is still in its loop
  float* zrx = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(tf) + p.tf_bytes);
  uint8_t* ring = reinterpret_cast<uint8_t*>(zrx) + p.rx_bytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const AbortCtl ctl{abort_flag, p.status, p.timeout_ns};
  const int C = p.C;
  const int rank = static_cast<int>(cluster_ctarank());
  const int cid = static_cast<int>(blockIdx.x) / C;
  int si = 0;
#pragma unroll
  for (int j = 1; j < kMaxSeg; ++j)
    if (j < p.nseg && cid >= p.seg[j].cl_begin) si = j;
  const Dec2Seg& sg = p.seg[si];
  const int Rc = sg.rc;                                   // rows of this cluster (tile of the ring)
  const int row0 = (cid - sg.cl_begin) * Rc;              // first row of the cluster in the family
  const int rows_here = max(0, min(Rc, sg.rows - row0));
  const int kb_lo = rank * p.kb_per;                      // first k block of this CTA's slice
  const int kb_n = max(0, min(p.kb_per, p.nkb - kb_lo));  // k blocks of the slice
  const int nstage = (kb_n + p.kbox - 1) / p.kbox;
  const int r16 = sg.r16;
  const int M = p.M;
  // rows this CTA finishes
  const int rf = (Rc + C - 1) / C;
  const int rf4 = (rf + 3) & ~3;   // rows per token in the receive area: 16-byte pushes
  const int f0 = rank * rf;
  const int f_n = max(0, min(rf, rows_here - f0));

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kDecConsumers / 32);
    }
    mbar_init(xbar, 1);
    mbar_init(vbar, 1);
    mbar_init(rbar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    // every peer pushes the W0 x sums of this CTA's rows and its t here: (C - 1) (zn + tn) floats
    mbar_arrive_expect_tx(rbar, static_cast<uint32_t>(C - 1) * static_cast<uint32_t>((rf4 + r16) * M) * 4u);
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&sg.tm_w);
    tma_prefetch_desc(&p.tm_x);
    if (p.act >= 0) tma_prefetch_desc(&p.tm_x2);
    if (sg.r > 0) tma_prefetch_desc(&sg.tm_v);
  }
  // The next call may start now: its CTAs fit beside this one and stream their weights.
  pdl_launch_dependents();
  __syncthreads();
  cluster_arrive_relaxed();

  bool ok = true;
  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && rows_here > 0 && kb_n > 0) {
      const uint32_t wbytes = static_cast<uint32_t>(p.kbox) * static_cast<uint32_t>(Rc) * 128u;
      // staged: the stage's x box and V rows count on the same barrier (x after the wait)
      const uint32_t xsb = kStaged ? static_cast<uint32_t>(p.kbox) * static_cast<uint32_t>(M) * 128u : 0u;
      const uint32_t vkb = static_cast<uint32_t>(64 * p.vrow * 2);   // V bytes of one k block
      const uint32_t vsb = (kStaged && sg.r > 0) ? static_cast<uint32_t>(p.kbox) * vkb : 0u;
      auto issue = [&](int q, int slot, bool with_x) {
        uint8_t* st = ring + static_cast<size_t>(slot) * p.stage_bytes;
        mbar_arrive_expect_tx(&full[slot], wbytes + xsb + vsb);
        tma_load_3d(st, &sg.tm_w, 0, kb_lo + q * p.kbox, row0, &full[slot]);
        if (vsb)
          for (int b = 0; b < p.kbox; ++b)
            tma_load_2d_plain(st + p.sv_off + b * vkb, &sg.tm_v, 0, (kb_lo + q * p.kbox + b) * 64, &full[slot]);
        if (xsb && with_x) tma_load_3d(st + p.sx_off, &p.tm_x, 0, kb_lo + q * p.kbox, 0, &full[slot]);
      };
      const int pre = nstage < p.stages ? nstage : p.stages;
      uint32_t filled = 0, fill_par = 0;
      // weights first: W0 stages and this CTA's V slice, before the dependency wait
      for (int q = 0; q < pre; ++q) {
        issue(q, q, false);
        filled |= 1u << q;
      }
      if (sg.r > 0 && !kStaged) {
        const uint32_t vb = static_cast<uint32_t>(p.vbox) * static_cast<uint32_t>(p.vrow) * 2u;
        const int nvb = (kb_n * 64 + p.vbox - 1) / p.vbox;
        mbar_arrive_expect_tx(vbar, static_cast<uint32_t>(nvb) * vb);
        for (int b = 0; b < nvb; ++b)
          tma_load_2d_plain(vs + static_cast<size_t>(b) * vb, &sg.tm_v, 0, kb_lo * 64 + b * p.vbox, vbar);
      }
      // The stages that do not fit the ring go to L2 now, while the previous call finishes: after
      // the dependency wait they refill the ring from L2 instead of HBM, so a ring of half an
      // SM keeps the stream going.
      for (int q = pre; q < nstage; ++q) tma_prefetch_l2_3d(&sg.tm_w, 0, kb_lo + q * p.kbox, row0);
      // x rows of this slice into L2 (a hint; L2 keeps them coherent with the previous kernel)
      for (int m = 0; m < M; ++m) {
        const int kk = kb_lo * 64;
        const int len = min(kb_n * 64, p.K - kk);
        if (len > 0) prefetch_l2_bulk(p.x + static_cast<int64_t>(m) * p.ldx + kk, static_cast<uint32_t>(len) * 2u);
        if (len > 0 && p.act >= 0)
          prefetch_l2_bulk(p.x2 + static_cast<int64_t>(m) * p.ldx + kk, static_cast<uint32_t>(len) * 2u);
      }
      pdl_wait_prior_grid();
      if (kStaged) {
        // x of the stages already issued, onto their barriers
        for (int q = 0; q < pre; ++q)
          tma_load_3d(ring + static_cast<size_t>(q) * p.stage_bytes + p.sx_off, &p.tm_x, 0, kb_lo + q * p.kbox, 0,
                      &full[q]);
      } else {
        mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(p.xkb) * static_cast<uint32_t>(M) * 128u * (p.act >= 0 ? 2u : 1u));
        tma_load_3d(xs, &p.tm_x, 0, kb_lo, 0, xbar);
        if (p.act >= 0) tma_load_3d(xs2, &p.tm_x2, 0, kb_lo, 0, xbar);
      }
      int slot = pre == p.stages ? 0 : pre;
      uint32_t phase = pre == p.stages ? 1u : 0u;
      for (int q = pre; q < nstage; ++q) {
        if (!mbar_wait(&empty[slot], phase ^ 1u, ctl)) {
          ok = false;
          break;
        }
        issue(q, slot, true);
        filled |= 1u << slot;
        fill_par = (fill_par & ~(1u << slot)) | (phase << slot);
        if (++slot == p.stages) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        // no copy may still be landing when the CTA leaves
        for (int s = 0; s < p.stages; ++s)
          if (filled & (1u << s)) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&full[s], (fill_par >> s) & 1u))
              if (global_timer_ns() - t0 > 20000000ull) break;
          }
      }
      // the resident x and V copies land before the CTA can exit, whatever happened
      if (!kStaged) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(xbar, 0u))
          if (global_timer_ns() - t0 > 20000000ull) break;
        if (sg.r > 0)
          while (!mbar_try_wait(vbar, 0u))
            if (global_timer_ns() - t0 > 40000000ull) break;
      }
    }
    __syncwarp();
    cluster_wait();
  } else {
    // ---------------- mma warps ----------------
    const int cw = warp - 1;                 // 0..7
    const int ct = threadIdx.x - 32;         // 0..255
    const int gq = lane >> 2, qq = lane & 3;
    // U rows and s of the rows this CTA finishes (weights: before the dependency wait)
    if (f_n > 0) {
      const int pieces = r16 / 8;
      for (int idx = ct; idx < f_n * pieces; idx += kDecConsumers) {
        const int rr = idx / pieces, c = idx - rr * pieces;
        const int o = row0 + f0 + rr;
        cp_async_16_zfill(smem_u32(us) + (rr * r16 + c * 8) * 2, sg.U + static_cast<int64_t>(o) * sg.ldu + c * 8,
                          max(0, min(16, (sg.r - c * 8) * 2)));
      }
      const int sb = (row0 + f0) & ~7;   // s from an 8-aligned row, zero past the family
      const int spieces = (row0 + f0 + f_n - sb + 7) / 8;
      for (int idx = ct; idx < spieces; idx += kDecConsumers) {
        const int e0 = sb + idx * 8;
        cp_async_16_zfill(smem_u32(ss) + idx * 16, sg.s + e0, max(0, min(16, (sg.rows - e0) * 2)));
      }
    }
    cp_async_commit();
    // No dependency wait of their own: everything the mma warps read after this point came
    // through the producer's copies issued after its wait, and a CTA stores y only after its
    // W0 loop, which cannot end before x (copied after that wait) has landed.

    const int nslab = (Rc + 15) / 16;
    const int kg = nslab >= 8 ? 1 : 8 / nslab;          // warps sharing one slab (split over k blocks)
    const bool active = rows_here > 0 && cw < (nslab >= 8 ? 8 : nslab * kg);
    const int slab = nslab >= 8 ? cw : cw / kg;         // first slab of this warp
    const int kgi = nslab >= 8 ? 0 : cw - slab * kg;
    const int nmy = nslab >= 8 ? (nslab > 8 + cw ? 2 : 1) : 1;   // slabs of this warp: slab, slab + 8
    const int mtn = r16 / 16;                           // 16-row tiles of V^T (1 or 2)
    float acc[2][NT][4];
    float tacc[2][NT][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[a][nt][e] = tacc[a][nt][e] = 0.0f;

    if (rows_here > 0 && kb_n > 0 && !kStaged) {
      ok = __all_sync(0xffffffffu, mbar_wait(xbar, 0u, ctl)) != 0;
      if (ok && sg.r > 0) ok = __all_sync(0xffffffffu, mbar_wait(vbar, 0u, ctl)) != 0;
    }
    if (p.act >= 0) {
      // gated input: x = act(gate output) * up output, formed once in place over the whole
      // slice (both boxes share one layout; the zeros past K give act(0) * 0 = 0)
      if (ok && rows_here > 0 && kb_n > 0) {
        const int n8 = static_cast<int>(static_cast<uint32_t>(p.xkb) * static_cast<uint32_t>(M) * 128u / 16u);
        for (int e = ct; e < n8; e += kDecConsumers) {
          uint4* gp = reinterpret_cast<uint4*>(xs) + e;
          const uint4 gv = *gp, uv = reinterpret_cast<const uint4*>(xs2)[e];
          const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
          uint32_t hw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float g0 = __uint_as_float(gw[q] << 16), g1 = __uint_as_float(gw[q] & 0xFFFF0000u);
            const float u0 = __uint_as_float(uw[q] << 16), u1 = __uint_as_float(uw[q] & 0xFFFF0000u);
            hw[q] = pack_bf16x2(gated_act(g0, p.act) * u0, gated_act(g1, p.act) * u1);
          }
          *gp = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        }
      }
      cons_bar();
    }
    const uint32_t xbase = smem_u32(xs);
    const uint32_t vbase = smem_u32(vs);
    // this lane's A rows in each of its slabs (rows past the cluster's rows read the last one;
    // their sums are dropped)
    int arow[2];
#pragma unroll
    for (int a = 0; a < 2; ++a) arow[a] = min(16 * (slab + 8 * a) + (lane & 7) + ((lane >> 3) & 1) * 8, Rc - 1);
    const int ahi = lane >> 4;
    int slot = 0;
    uint32_t phase = 0;
    for (int sq = 0; ok && sq < nstage && rows_here > 0; ++sq) {
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&full[slot], phase, ctl)) != 0)) break;
      const int kb0 = sq * p.kbox;                     // first k block of the stage, within the slice
      const int nb = min(p.kbox, kb_n - kb0);
      const uint32_t wbase = smem_u32(ring + static_cast<size_t>(slot) * p.stage_bytes);
      // x and V of this stage: in the stage (staged) or in the resident slices
      const uint32_t sxbase = kStaged ? wbase + p.sx_off : xbase;
      const int sxkb = kStaged ? p.kbox : p.xkb;
      const uint32_t svbase = kStaged ? wbase + p.sv_off : vbase;
      const int sk0 = kStaged ? kb0 : 0;              // first k block held at svbase / sxbase
      if (active) {
        for (int b = (nslab >= 8) ? 0 : (kgi - kb0 % kg + kg) % kg; b < nb; b += (nslab >= 8 ? 1 : kg)) {
          const int bx = kb0 + b;                      // k block within the slice
          // t for this block: the slab-0 warps when the slabs are split over k blocks, else
          // warp (block mod 8)
          const bool t_own = sg.r > 0 && (nslab >= 8 ? ((kb_lo + bx) & 7) == cw : slab == 0);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // B: x^T fragments of this 16-wide step (token rows past M repeat the last token)
            uint32_t bfr[NT][2];
            if constexpr (NT == 1) {
              ldsm2(sw_addr(sxbase, sxkb, min(lane & 7, M - 1), bx - sk0, 2 * j + ((lane >> 3) & 1)), bfr[0][0],
                    bfr[0][1]);
            } else {
              uint32_t b0, b1, b2, b3;
              ldsm4(sw_addr(sxbase, sxkb, min((lane & 7) + (lane >> 4) * 8, M - 1), bx - sk0, 2 * j + ((lane >> 3) & 1)),
                    b0, b1, b2, b3);
              bfr[0][0] = b0;
              bfr[0][1] = b1;
              bfr[1][0] = b2;
              bfr[1][1] = b3;
            }
#pragma unroll
            for (int a = 0; a < 2; ++a) {
              if (a < nmy) {
                uint32_t a0, a1, a2, a3;
                ldsm4(sw_addr(wbase, p.kbox, arow[a], b, 2 * j + ahi), a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma16816(acc[a][nt], a0, a1, a2, a3, bfr[nt][0], bfr[nt][1]);
              }
            }
            if (t_own) {
              // A: V^T [16 ranks x 16 k] from the V slice [k][vrow] (ldmatrix.trans)
              const int kl = (bx - sk0) * 64 + 16 * j + (lane & 7) + ((lane >> 4) & 1) * 8;
#pragma unroll
              for (int mt = 0; mt < 2; ++mt) {
                if (mt < mtn) {
                  uint32_t a0, a1, a2, a3;
                  ldsm4_trans(svbase + (kl * p.vrow + 16 * mt + ((lane >> 3) & 1) * 8) * 2, a0, a1, a2, a3);
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt) mma16816(tacc[mt][nt], a0, a1, a2, a3, bfr[nt][0], bfr[nt][1]);
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
    cp_async_wait_all();
    cluster_wait();   // every CTA of the cluster has started: its shared memory may be written
    // ---- partial sums into this CTA's ring (no stage is in use any more) ----
    cons_bar();
    float* zex = reinterpret_cast<float*>(ring);               // [kg][M][Rc]: rows fastest
    float* tex = zex + static_cast<size_t>(kg) * Rc * M;       // [8][r16][M]
    if (active) {
#pragma unroll
      for (int a = 0; a < 2; ++a)
        if (a < nmy)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int row = 16 * (slab + 8 * a) + gq + 8 * h, tok = 8 * nt + 2 * qq + e;
                if (row < Rc && tok < M) zex[(static_cast<size_t>(kgi) * M + tok) * Rc + row] = acc[a][nt][2 * h + e];
              }
    }
    if (sg.r > 0) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
        if (mt < mtn)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int jr = 16 * mt + gq + 8 * h, tok = 8 * nt + 2 * qq + e;
                if (tok < M) tex[(static_cast<size_t>(cw) * r16 + jr) * M + tok] = tacc[mt][nt][2 * h + e];
              }
    }
    cons_bar();
    // push: the rows peer q finishes go to its receive area at this CTA's rank, and t to every
    // peer (this CTA included); each pushed value is this CTA's sum over its k-block groups (W0 x)
    // or its eight warps (t), in a fixed order. Stores only, no remote read.
    {
      // receive areas: z [C][M][rf4] (rows fastest), then t [C][r16][M]; 16-byte pushes
      const int zn = rf4 * M, tn = r16 * M;
      const size_t grp = static_cast<size_t>(Rc) * M;
      const uint32_t zr_me = smem_u32(zrx) + static_cast<uint32_t>(rank * zn) * 4u;
      const uint32_t tr_me = smem_u32(zrx) + static_cast<uint32_t>(C * zn + rank * tn) * 4u;
      const int zq = zn / 4;
      for (int idx = ct; idx < C * zq; idx += kDecConsumers) {
        const int q = idx / zq, e = (idx - q * zq) * 4;   // e = tok * rf4 + rr, rr a multiple of 4
        const int tok = e / rf4, rr = e - tok * rf4;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = q * rf + rr + i;
          v[i] = 0.0f;
          if (rr + i < rf && row < rows_here)
            for (int k = 0; k < kg; ++k) v[i] += zex[k * grp + tok * Rc + row];
        }
        if (q == rank)   // this CTA's own rows: a plain shared store
          *reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(zrx) + static_cast<size_t>(rank * zn + e) * 4u) =
              make_float4(v[0], v[1], v[2], v[3]);
        else
          st_async_v4(mapa_u32(zr_me + static_cast<uint32_t>(e) * 4u, static_cast<uint32_t>(q)), v[0], v[1], v[2], v[3],
                      mapa_u32(smem_u32(rbar), static_cast<uint32_t>(q)));
      }
      // t: this CTA's sum over its eight warps, formed once and pushed to every peer
      for (int e = 4 * ct; e < tn; e += 4 * kDecConsumers) {
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int w = 0; w < 8; ++w)
#pragma unroll
          for (int i = 0; i < 4; ++i) v[i] += tex[static_cast<size_t>(w) * tn + e + i];
        *reinterpret_cast<float4*>(reinterpret_cast<uint8_t*>(zrx) + static_cast<size_t>(C * zn + rank * tn + e) * 4u) =
            make_float4(v[0], v[1], v[2], v[3]);
        for (int q = 0; q < C; ++q)
          if (q != rank)
            st_async_v4(mapa_u32(tr_me + static_cast<uint32_t>(e) * 4u, static_cast<uint32_t>(q)), v[0], v[1], v[2], v[3],
                        mapa_u32(smem_u32(rbar), static_cast<uint32_t>(q)));
      }
    }
  }

  // The second cluster barrier phase: arrived once this thread's pushes are issued (the
  // producer warp: once its copies are done), waited on at the very end, so no CTA leaves
  // while a peer may still push into it.
  cluster_arrive_relaxed_end();
  if (warp > 0) {
    const int ct = threadIdx.x - 32;
    // the own pushes (plain stores) of every mma warp, then the peers' (their bytes on rbar)
    cons_bar();
    ok = __all_sync(0xffffffffu, mbar_wait_cluster(rbar, 0u, ctl)) != 0 && ok;
    ok = ok && !*reinterpret_cast<volatile int*>(abort_flag);
    const int zn = rf4 * M, tn = r16 * M;
    const float* zr = zrx;
    const float* tr = zrx + static_cast<size_t>(C) * zn;
    // t = sum over the cluster's slices, in rank order
    for (int idx = ct; idx < tn; idx += kDecConsumers) {
      float v = 0.0f;
      for (int q = 0; q < C; ++q) v += tr[q * tn + idx];
      tf[idx] = v;
    }
    cons_bar();
    // y for the rows this CTA finishes: z summed over the slices (rank order), U t in fp32, one
    // rounding
    if (ok && f_n > 0) {
      const uint16_t* urow_base = reinterpret_cast<const uint16_t*>(us);
      const uint16_t* sv = reinterpret_cast<const uint16_t*>(ss);
      const int soff = (row0 + f0) & 7;
      for (int idx = ct; idx < f_n * M; idx += kDecConsumers) {
        const int tok = idx / f_n, rr = idx - tok * f_n;   // rows fastest: coalesced stores of y
        float z = 0.0f;
        for (int q = 0; q < C; ++q) z += zr[q * zn + tok * rf4 + rr];
        // U row in 16-byte pieces (the row stride r16 * 2 is a multiple of 32 bytes)
        float lr = 0.0f;
        const uint4* ur = reinterpret_cast<const uint4*>(urow_base + rr * r16);
        for (int j8 = 0; j8 < r16 / 8; ++j8) {
          const uint4 w = ur[j8];
          const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = j8 * 8 + 2 * e;
            lr = fmaf(__uint_as_float(ww[e] << 16), tf[j * M + tok], lr);
            lr = fmaf(__uint_as_float(ww[e] & 0xFFFF0000u), tf[(j + 1) * M + tok], lr);
          }
        }
        const float sc = bf16_to_f32(sv[soff + rr]);
        const int64_t yi = static_cast<int64_t>(tok) * sg.ldy + row0 + f0 + rr;
        if (dbg_in_bounds(yi, dbg_extent(M, sg.ldy, sg.rows), p.status) && dbg_in_bounds(row0 + f0 + rr, sg.rows, p.status))
          sg.y[yi] = f32_to_bf16_rn(fmaf(sc, z, lr));
      }
    }
  }
  cluster_wait();
}

// h = RN_bf16(act(g) * u), in place of g: one thread per 8 elements (16-byte rows pieces).
__global__ void __launch_bounds__(256) aq_gated_act_kernel(uint16_t* g, const uint16_t* u, int64_t ld, int64_t M, int n,
                                                           int act) {
  const int per = (n + 7) / 8;
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  pdl_wait_prior_grid();   // g and u are the previous grid's outputs
  if (e >= M * per) return;
  const int64_t m = e / per;
  const int c = static_cast<int>(e - m * per) * 8;
  uint16_t* gr = g + m * ld + c;
  const uint16_t* ur = u + m * ld + c;
  for (int j = 0; j < 8 && c + j < n; ++j)
    gr[j] = f32_to_bf16_rn(gated_act(bf16_to_f32(gr[j]), act) * bf16_to_f32(ur[j]));
}

cudaError_t launch_gated_act(uint16_t* g, const uint16_t* u, int64_t ld, int64_t M, int32_t n, int32_t act,
                             cudaStream_t st, bool pdl) {
  const int64_t threads = M * ((n + 7) / 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((threads + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, aq_gated_act_kernel, g, u, ld, M, static_cast<int>(n), static_cast<int>(act));
}

cudaError_t launch_decode2(const Dec2Params& p, int grid, size_t smem, cudaStream_t st, bool pdl) {
  void* args[] = {const_cast<Dec2Params*>(&p)};
  const void* fn = p.staged ? (p.M > 8 ? reinterpret_cast<const void*>(&aq_decode2_kernel<2, true>)
                                       : reinterpret_cast<const void*>(&aq_decode2_kernel<1, true>))
                            : (p.M > 8 ? reinterpret_cast<const void*>(&aq_decode2_kernel<2, false>)
                                       : reinterpret_cast<const void*>(&aq_decode2_kernel<1, false>));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attrs[2];
  int n = 0;
  attrs[n].id = cudaLaunchAttributeClusterDimension;
  attrs[n].val.clusterDim.x = static_cast<unsigned>(p.C);
  attrs[n].val.clusterDim.y = 1;
  attrs[n].val.clusterDim.z = 1;
  ++n;
  if (pdl) {
    attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = n;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t configure_decode2(size_t max_smem) {
  cudaError_t e;
  const int s = static_cast<int>(max_smem);
  if ((e = cudaFuncSetAttribute(aq_decode2_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, s))) return e;
  if ((e = cudaFuncSetAttribute(aq_decode2_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, s))) return e;
  if ((e = cudaFuncSetAttribute(aq_decode2_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, s))) return e;
  return cudaFuncSetAttribute(aq_decode2_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, s);
}

}  // namespace aq
