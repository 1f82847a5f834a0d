// k_moe_down_persist.cuh -- down_combine's GEMV (vllm.models.flint.ops.
// moe_gemv, down_combine: y_j = bf16(fp32(act[pair] . W2[e] row h) *
// alpha2[e]), y_shared = bf16(fp32(sact[t] . Wsd row h) * gssd)) on a
// persistent grid, with the slab kernel's arithmetic (k_gemv_slab.cuh).
//
// The slab kernel's grouped form gives each CTA one work item: a chunk of up
// to 8 pairs routed to one expert (or a chunk of the shared expert's tokens)
// and a group of T row tiles of H.  Launched as one grid of items, the CTAs
// of the last round start late and finish late: at 8 tokens of the
// E = 128, top-8 block the SMs' CTA slots are ~74 % busy over the call.
// Here a grid of (CTAs per SM) x SMs CTAs takes the same items from a
// counter instead (item = column x groups + group): each CTA starts with item
// blockIdx.x and then claims the next free item, so every slot stays busy
// until the items run out, and the producer warp resolves and streams the
// next item's weights while the consumers finish the current one.
//
//   producer warp: resolves an item (inactive ones -- duplicate chunk
//     columns -- are skipped), writes its description into a ring of
//     kPersistDesc entries (one more than the deepest weight ring, so an
//     entry in use is never overwritten), and streams its T x stages weight
//     stages through the ring.  The counter is claimed only after the wait
//     for the previous grid: a following down_combine on the same workspace
//     may start early under PDL, and its CTAs must not see this call's
//     counter (the counter is tagged with the call's epoch, so the workspace
//     needs no initialisation).  When the items run out it completes the
//     next stage's full barrier with no copy and an empty description.
//   consumer warps: at an item's first stage they load the item's activation
//     rows into the slab (every 256-K stage's exponent range in the same
//     pass, then the stages that allow it to f16 with a power-of-two shift),
//     stream its stages and after each row tile write their rows of y.
//
// A CTA whose wait ran out tags every row tile's counter with this call's
// epoch; the combine kernel then leaves the whole output unwritten.
#pragma once

#include "k_gemv_slab.cuh"

namespace fp4 {

constexpr int kPersistDesc = kMaxStages + 1;

template <int kR>
__global__ void __launch_bounds__(kSlabThreads, kSlabMinBlocks) moe_down_persist_kernel(const __grid_constant__ GemvParams p) {
  using C = SlabCfg<kR>;
  constexpr int kChains = C::kChains;
  using Work = CtaWorkN<kSlabNT>;
  constexpr int kND = kPersistDesc;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t slab = (smem_u32(smem_raw) + 1023u) & ~1023u;  // activations of the current item
  const uint32_t ring = slab + p.x_off;                          // weight stages
  __shared__ __align__(8) uint64_t bar_full[kMaxStages];
  __shared__ __align__(8) uint64_t bar_empty[kMaxStages];
  __shared__ volatile int s_abort;
  __shared__ Work s_desc[kND];  // items in flight, producer -> consumers
  __shared__ int s_t0[kND];     // first row tile of the item
  __shared__ int s_ntl[kND];    // row tiles of the item (0: no more items)
  __shared__ int s_emax[kSlabMaxStages];
  __shared__ int s_emin[kSlabMaxStages];

  const int tid = threadIdx.x;
  const int warp = tid / 32;
  const int lane = tid % 32;
  const int cw = p.cw;  // consumer warps; warp cw is the producer
  const int ncons = cw * 32;
  const int nstages = p.nstages;
  const int trows = 16 * kR * cw;  // 128
  const int tiles_h = (p.n_out + 127) / 128;
  const int groups = p.routed_tiles;  // tile groups of up to T tiles
  const int cn = p.chunk > 0 && p.chunk < kSlabNT ? p.chunk : kSlabNT;
  const int ncols = p.P + (p.M + cn - 1) / cn;
  const int total = ncols * groups;
  const uint64_t pol_w = policy_evict_first();

  if (warp == cw && lane == 0) {
    prefetch_tensormap(&p.tm_w);
    prefetch_tensormap(&p.tm_w2);
    s_abort = 0;
    for (int i = 0; i < nstages; ++i) {
      mbar_init(smem_u32(&bar_full[i]), 1);
      mbar_init(smem_u32(&bar_empty[i]), cw);
    }
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0) pdl_launch_dependents();

  auto group_tiles = [&](int grp, int& t0, int& ntl) {
    t0 = grp * tiles_h / groups;
    ntl = (grp + 1) * tiles_h / groups - t0;
  };

  if (warp == cw) {
    // ------------------------------------------------------------------ producer
    // Next item: the counter holds [epoch:32 | next item:32].  One atomic
    // add per claim; a value with another epoch (an earlier call, or
    // never-initialised scratch) means this call's counter has not been
    // started yet: the CTA that swaps in [epoch | grid size + 1] takes item
    // gridDim.x, the others retry the swap on the value they saw until it
    // succeeds or the counter carries this epoch, then add again.
    auto claim = [&]() -> int {
      int it = 0;
      if (lane == 0) {
        constexpr unsigned long long kHi = 0xFFFFFFFF00000000ull;
        unsigned long long* ctr = p.counters + tiles_h;
        const unsigned long long tag = static_cast<unsigned long long>(p.epoch) << 32;
        unsigned long long old = atomicAdd(ctr, 1ull);
        while ((old & kHi) != tag) {
          const unsigned long long seen = atomicCAS(ctr, old + 1, tag | (gridDim.x + 1ull));
          if (seen == old + 1) {
            old = tag | gridDim.x;
          } else if ((seen & kHi) == tag) {
            old = atomicAdd(ctr, 1ull);
          } else {
            old = seen - 1;  // (the next swap expects `seen`)
          }
        }
        it = static_cast<int>(old & 0xFFFFFFFFull);
      }
      return __shfl_sync(0xFFFFFFFFu, it, 0);
    };
    int item = blockIdx.x, seq = 0, s = 0, issued = 0;
    bool waited = false;
    for (;;) {
      const int d = seq % kND;
      int t0 = 0, ntl = 0;
      while (item < total && !s_abort) {
        resolve_work_at<kMoeDown, kSlabNT, Work>(p, s_desc[d], 0, lane, item % groups, item / groups);
        if (s_desc[d].active) {
          group_tiles(item % groups, t0, ntl);
          break;
        }
        if (!waited) {
          pdl_wait();
          waited = true;
        }
        item = claim();
      }
      if (s_abort) break;
      const bool done = item >= total;
      if (lane == 0) {
        s_t0[d] = t0;
        s_ntl[d] = done ? 0 : ntl;
      }
      __syncwarp();
      const int nst_tile = done ? 1 : (s_desc[d].k_end + 255) / 256;
      const int nst_item = done ? 1 : ntl * nst_tile;  // (the end: one stage slot, no copy)
      bool ok = true;
      for (int i = 0; i < nst_item; ++i, ++s) {
        const int slot = s % nstages;
        if (s >= nstages)
          ok = __all_sync(0xFFFFFFFFu, !s_abort && mbar_wait_sleepy(smem_u32(&bar_empty[slot]),
                                                                    ((s / nstages) & 1) ^ 1, p.err, 64));
        if (!ok) break;
        if (lane == 0 && s != p.skip_stage) {  // (test hook: the skipped stage is never issued)
          const uint32_t fb = smem_u32(&bar_full[slot]);
          if (done) {
            mbar_arrive(fb);
          } else {
            const Work& w = s_desc[d];
            const int t = t0 + i / nst_tile, ks = i % nst_tile;
            const uint32_t st = ring + slot * p.stage_bytes;
            const int k0 = ks * 256;
            const int nchunks = min(256, w.k_end - k0) / kSubK;
            const CUtensorMap* tmw = w.shared ? &p.tm_w2 : &p.tm_w;
            const uint8_t* sfb = w.shared ? p.sf2 : p.sf + static_cast<size_t>(w.expert) * p.sf_expert_bytes;
            const int wrow = (w.shared ? 0 : w.expert * p.rows_per_expert) + t * 128;
            mbar_arrive_expect_tx(fb, static_cast<uint32_t>(trows * 128 + nchunks * 512));
            tma_load_2d(ring + slot * p.stage_bytes, tmw, k0 / 2, wrow, fb, pol_w);
            const size_t chunk = static_cast<size_t>(t) * (w.kbp / 4) + k0 / 64;
            bulk_load(st + trows * 128, sfb + chunk * 512, nchunks * 512, fb, pol_w);
          }
        }
        issued = s + 1;
      }
      if (!ok) {
        s_abort = 1;
        break;
      }
      if (done) break;
      ++seq;
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      item = claim();
    }
    // After an abort, let every copy still in flight land before the CTA
    // (and its shared memory) goes away: the latest fill of each slot.
    if (s_abort && lane == 0)
      for (int s2 = max(0, issued - nstages); s2 < issued; ++s2)
        if (s2 != p.skip_stage) (void)mbar_wait(smem_u32(&bar_full[s2 % nstages]), (s2 / nstages) & 1, p.err);
  } else {
    // ------------------------------------------------------------------ consumers
    // Every consumer warp walks every stage of every item: a warp whose wait
    // ran out sets s_abort and goes on without waiting or computing, so all
    // of them meet at the next item's barrier, which ORs the abort and lets
    // them leave together (the named barriers are not bounded waits).
    pdl_wait();  // the activations (gate_up's outputs) and the y scratch
    const int g = lane / 4, c = lane % 4;
    const int sg = (g % 2) * 4 + g / 2;  // sigma(g)
    const uint32_t key = static_cast<uint32_t>(sg);
    // shared-memory offsets of this thread's rows and of their scale bytes:
    // the same for every row tile (one 128-row scale group per tile)
    uint32_t w_off[kR][2], sf_off[kR][2];
#pragma unroll
    for (int b = 0; b < kR; ++b) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = (warp * kR + b) * 16 + sg + 8 * hr;
        w_off[b][hr] = (row / 8) * 1024 + (row % 8) * 128;
        sf_off[b][hr] = trows * 128 + (row % 32) * 16 + ((row % 128) / 32) * 4;
      }
    }
    float acc[kChains][kR][4];
    float accb[kR][4];
#pragma unroll
    for (int b = 0; b < kR; ++b) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        accb[b][e] = 0.0f;
#pragma unroll
        for (int q = 0; q < kChains; ++q) acc[q][b][e] = 0.0f;
      }
    }
    const float post = static_cast<float>(1 << kShift);
    int s = 0;
    for (int seq = 0;; ++seq) {
      const int d = seq % kND;
      // the item's first stage: its full barrier publishes the item
      bool ok = __all_sync(0xFFFFFFFFu, !s_abort && mbar_wait(smem_u32(&bar_full[s % nstages]), (s / nstages) & 1, p.err));
      if (!ok) s_abort = 1;
      if (bar_red_or<1>(ncons, s_abort != 0)) break;
      const int ntl = s_ntl[d];
      if (ntl == 0) break;  // no more items (the same for every consumer warp)
      const Work& w = s_desc[d];
      const int M = w.ntok;
      // (read before the item's last stage is released: the producer may
      // then reuse the item's description)
      int orow[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) orow[e] = 2 * c + e < M ? w.orow[2 * c + e] : 0;
      const int klen = w.k_end;
      const int nst_tile = (klen + 255) / 256;
      const int nchk = klen / 8;
      const int nslot = nst_tile * 32;
      const uint32_t slab_stage = static_cast<uint32_t>(M) * 512u;
      const uint16_t* xb = w.shared ? p.x2 : p.x;
      // the item's activation slab: bf16 chunks in with each stage's exponent
      // range (warp-reduced; a warp's 32 chunks share a row and a stage), then
      // the stages whose range allows it to x 2^s in f16
      for (int i = tid; i < nst_tile; i += ncons) {
        s_emax[i] = 0;
        s_emin[i] = 255;
      }
      cons_sync(ncons);
      constexpr int kFillBatch = 4;
      for (int q0 = tid; q0 < M * nslot; q0 += kFillBatch * ncons) {
        uint4 v[kFillBatch];
#pragma unroll
        for (int i = 0; i < kFillBatch; ++i) {
          const int q = q0 + i * ncons;
          const int n = q / nslot, kq = q % nslot;
          v[i] = make_uint4(0u, 0u, 0u, 0u);
          if (q < M * nslot && kq < nchk) v[i] = __ldg(reinterpret_cast<const uint4*>(xb + w.xoff[n] + 8 * kq));
        }
#pragma unroll
        for (int i = 0; i < kFillBatch; ++i) {
          const int q = q0 + i * ncons;
          if (q >= M * nslot) break;
          const int n = q / nslot, kq = q % nslot;
          const int st = kq / 32, u = (kq % 32) / 8, ch = kq % 8;
          sts128(slab + st * slab_stage + (u * M + n) * 128 + ((ch ^ (n & 7)) * 16), v[i]);
          int emx, emn;
          bf16x8_exp_range(v[i], emx, emn);
          emx = __reduce_max_sync(0xFFFFFFFFu, emx);
          emn = __reduce_min_sync(0xFFFFFFFFu, emn);
          if (lane == 0) {
            atomicMax(&s_emax[st], emx);
            atomicMin(&s_emin[st], emn);
          }
        }
      }
      cons_sync(ncons);
      for (int q = tid; q < M * nchk; q += ncons) {
        const int n = q / nchk, kq = q % nchk;
        const int st = kq / 32, u = (kq % 32) / 8, ch = kq % 8;
        const int sh = f16_shift(s_emax[st], s_emin[st]);
        if (sh < 0) continue;
        const uint32_t a = slab + st * slab_stage + (u * M + n) * 128 + ((ch ^ (n & 7)) * 16);
        sts128(a, bf16x8_to_f16x8_scaled(lds128(a), __int_as_float((127 + sh) << 23)));
      }
      cons_sync(ncons);
      const float sc = w.shared ? __ldg(p.gs) : __ldg(p.alpha + w.expert);
      uint16_t* dst = w.shared ? p.out2 : p.out;
      const int64_t ld = w.shared ? p.ldo2 : p.ldo;
      const int t0 = s_t0[d];
      for (int tt = 0; tt < ntl; ++tt) {
        for (int ks = 0; ks < nst_tile; ++ks, ++s) {
          const int slot = s % nstages;
          if (tt > 0 || ks > 0) {
            ok = __all_sync(0xFFFFFFFFu, !s_abort && mbar_wait(smem_u32(&bar_full[slot]), (s / nstages) & 1, p.err));
            if (!ok) s_abort = 1;
          }
          if (s_abort) continue;  // (the slot is not released: its copy may still land)
          const uint32_t st = ring + slot * p.stage_bytes;
          const uint32_t xs = slab + ks * slab_stage;
          const int kvalid = min(256, klen - ks * 256);
          const int sh = f16_shift(s_emax[ks], s_emin[ks]);
          if (sh >= 0) {
            const uint32_t sdown = f16x2_pow2_neg(sh);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              if (128 * h < kvalid) {
                if (128 * (h + 1) <= kvalid)
                  slab_half_f16<kR, kChains, true>(acc, st, xs, h, true, M, w_off, sf_off, key, g, c, sdown);
                else
                  slab_half_f16<kR, kChains, true>(acc, st, xs, h, 32 * (4 * h + c) < kvalid, M, w_off, sf_off, key, g,
                                                   c, sdown);
              }
            }
          } else {
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
              if (128 * h < kvalid)
                slab_half_bf16<kR>(accb, st, xs, h, 32 * (4 * h + c) < kvalid, M, w_off, sf_off, key, g, c);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bar_empty[slot]));
        }
        // the tile's y rows: y_j = bf16(acc * alpha2[e]) or y_shared =
        // bf16(acc * gssd); the accumulators restart
        const int h0 = (t0 + tt) * 128;
#pragma unroll
        for (int b = 0; b < kR; ++b) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int h = h0 + (warp * kR + b) * 16 + sg + 8 * hr;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float a = accb[b][2 * hr + e] * post;
              accb[b][2 * hr + e] = 0.0f;
#pragma unroll
              for (int q = 0; q < kChains; ++q) {
                a += acc[q][b][2 * hr + e];
                acc[q][b][2 * hr + e] = 0.0f;
              }
              const int n = 2 * c + e;
              if (!s_abort && n < M && h < p.n_out)
                dst[static_cast<int64_t>(orow[e]) * ld + h] = f32_to_bf16_rn(a * sc);
            }
          }
        }
      }
    }
  }
  __syncthreads();
  // a CTA that gave up tags every row tile: the combine leaves the output unwritten
  if (tid == 0 && s_abort)
    for (int t = 0; t < tiles_h; ++t) p.counters[t] = abort_tag(p.epoch);
}

}  // namespace fp4
