// tc_correction.cu -- second half of the tensor-core SLiM backward: the
// reverse state of the later segments.
//
// "Sub-Linear Memory: How to Make Performers SLiM", section 3.3, eq. (20)-(21).
// The backward kernel runs every segment from a reverse state of zero at its
// end, so dK and dV of segment s still lack the terms of G_end(s), the sum of
// the later segments' G totals (a reverse scan).  Both terms are linear in G:
//   dphi_k' = V G_V^T + 1 G_S^T,     u = phi_k * dphi_k'
//   dV     += phi_k G_V
//   dK     += u W^T - k rowsum(u)    (FAVOR+; elu+1: dK += dphi_k' * min(phi_k, 1))
// per 128-feature block h of G_end.  Tiles of segments 0 .. P-2 are
// independent here, so they are dealt out as flat (head, tile) units to one
// CTA per SM.
//
// Roles (16 warps): warp 0 streams K and V (and the bf16 image of G_end when
// the unit's segment changes) into shared memory and adds each unit's staged
// increments to dK and dV with TMA reduce-adds before it reuses the slots;
// warps 1, 2 and 3 issue the MMAs (F = K W and D = V G_V^T in 64-feature jobs
// through two TMEM buffers each; dV' and dK' per 128-feature block); warps
// 4-11 turn each job into phi_k and u (two threads per row, 32 columns each);
// warps 12-15 finish the unit: dK = dK' - k rowsum(u), both increments to
// bf16 in the unit's own K and V slots.  (Reading the backward's rows, adding
// and writing them back from the tail warps instead measured slower.)  Every
// hand-off is an mbarrier with a bounded wait.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace slim {
namespace tcc {

using namespace slim::tc;

constexpr int kTile = 128;
constexpr int D = 64;
constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;
constexpr int kSlots = 4;  // K, V of two units in flight (K in even slots, V in odd)
constexpr uint32_t kTileBytes = kTile * D * 2;

struct Params {
  int L, P, tps, BH;
  int H, wstride;  // heads; bf16 elements between per-head W^T images (0: one shared W)
  long long per_head;  // units per head: tiles of segments 0 .. P-2, or of every
                       // segment when a reverse state arrives from later rows
  __nv_bfloat16 *dk, *dv;
  const __nv_bfloat16 *wimg;  // W^T image [M][64] (FAVOR+)
  const unsigned char *grec;  // per (head, segment): G_end image [M][64] bf16, then G_S fp32 [M]
  int *status;
};

enum {
  B_FULL = 0,       // [4] TMA -> consumers
  B_EMPTY = 4,      // [4] MMAs done with the slot
  B_FFULL = 8,      // [2] feature job in TMEM buffer b
  B_FEMPTY = 10,    // [2] ... read out (8 warps)
  B_DFULL = 12,     // [2] V G_V^T job in TMEM buffer b
  B_DEMPTY = 14,    // [2] ... read out (8 warps)
  // phi_k and u are double-buffered, so each buffer has its own "stored"
  // barrier: the phi_k warps may run two blocks ahead of the dV', dK'
  // issuer (it can stall on B_OUTEMPTY), and one barrier for both buffers
  // would then be two phases ahead of the issuer's wait, whose parity test
  // cannot tell phase c from c + 2
  B_PHK = 16,       // [2] phi_k block stored in buffer b (8 warps)
  B_U = 18,         // [2] u block packed in TMEM buffer b (8 warps)
  B_PHFREE = 20,    // [2] dV' MMAs done with phi_k buffer b
  B_UFREE = 22,     // [2] dK' MMAs done with u buffer b
  B_OUTFULL = 24,   // dV', dK' complete
  B_OUTEMPTY = 25,  // dV', dK' read out (4 warps)
  B_GFULL = 26,     // G_end image landed
  B_GEMPTY = 27,    // G_end image no longer read (2 MMA commits + 8 warps)
  B_WFULL = 28,     // W image landed
  B_EPI = 29,       // [2] row sums of u written (8 warps), by unit parity
  B_STG = 31,       // [2] a unit's dK, dV increments staged in its slots (4 + 8 warps)
  B_DONE = 33,      // [3] MMA drain of each issuing thread
  B_COUNT = 36
};

template <int M>
struct Layout {
  uint32_t w, slots, g, gs, phk, usum, bars, total;
  __host__ __device__ Layout() {
    uint32_t o = 0;
    w = o; o += M * 128u;
    slots = o; o += kSlots * kTileBytes;
    g = o; o += M * 128u;   // G_end[:, 0:64] as bf16 [M][64], swizzled
    gs = o; o += M * 4u;    // G_end[:, 64] fp32 (directly after g: one bulk copy)
    o = (o + 1023u) & ~1023u;
    phk = o; o += 2 * kTile * 128 * 2;  // two phi_k blocks, used in turn
    usum = o; o += 2 * 2 * kTile * 4;  // [unit parity][part][row]
    bars = o; o += 8 * B_COUNT + 16;
    total = o;
  }
};

// TMEM columns: F jobs 2 x 64 | D jobs 2 x 64 | dV' 64 | dK' 64 | u, two
// 128-feature blocks of bf16 pairs (the A operand of dK' = u W^T) 2 x 64
constexpr uint32_t kF = 0, kDc = 128, kDV = 256, kDK = 320, kU = 384;

template <bool FAVOR, int M>
__global__ void __launch_bounds__(kThreads, 1)
    tc_corr_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV, Params p) {
  constexpr int nb = (M + 127) / 128, FB = M < 128 ? M : 128;
  constexpr int JT = M / 64;  // 64-feature jobs per unit (F and D alike)
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Layout<M> lay;
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + B_COUNT);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar + B_COUNT) + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // this CTA's units [u0, u1): unit u = (head, tile) over the first P-1
  // segments (every segment, the last one possibly short, when a reverse
  // state arrives from later rows)
  // with one W per head the grid is [CTAs per head][head]: a CTA's units stay
  // in head blockIdx.y, whose W it loads once
  const long long units = p.per_head * (gridDim.y > 1 ? 1 : p.BH);
  const long long u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
  const int nun = (int)(u1 - u0);
  // debug builds: a unit range outside the heads records SLIM_ERR_BOUNDS and the CTA does nothing
  if (!SLIM_DCHECK(p.status, nun >= 1 && (long long)blockIdx.y + (u1 - 1) / p.per_head < p.BH)) return;
  // every role walks the same units with counters (no divisions per unit):
  // head bh, tile t, segment seg and position pos of the tile in it; the
  // segment's G_end changes when pos wraps
  struct Cursor {
    int bh, t, seg, pos;
  };
  const int per_head = (int)p.per_head;
  Cursor first;
  const long long h0 = u0 / p.per_head;  // heads before this CTA's first unit (0 on a per-head grid)
  first.bh = (int)blockIdx.y + (int)h0;
  first.t = (int)(u0 - h0 * p.per_head);
  first.seg = first.t / p.tps;
  first.pos = first.t - first.seg * p.tps;
  auto advance = [&](Cursor &c) {
    ++c.t;
    if (++c.pos == p.tps) {
      c.pos = 0;
      ++c.seg;
    }
    if (c.t == per_head) {
      c.t = 0;
      c.seg = 0;
      c.pos = 0;
      ++c.bh;
    }
  };
  auto new_key = [&](int i, const Cursor &c) { return i == 0 || c.pos == 0; };
  auto last_of_key = [&](int i, const Cursor &c) {
    return i == nun - 1 || c.pos == p.tps - 1 || c.t == per_head - 1;
  };
  const uint32_t grec_bytes = (uint32_t)M * 132u;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar + B_FULL + s, 1);
      mbar_init(bar + B_EMPTY + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar + B_FFULL + b, 1);
      mbar_init(bar + B_FEMPTY + b, 8);
      mbar_init(bar + B_DFULL + b, 1);
      mbar_init(bar + B_DEMPTY + b, 8);
      mbar_init(bar + B_EPI + b, 8);
      mbar_init(bar + B_STG + b, 12);
      mbar_init(bar + B_PHFREE + b, 1);
      mbar_init(bar + B_UFREE + b, 1);
      mbar_init(bar + B_PHK + b, 8);
      mbar_init(bar + B_U + b, 8);
    }
    mbar_init(bar + B_OUTFULL, 1);
    mbar_init(bar + B_OUTEMPTY, 4);
    mbar_init(bar + B_GFULL, 1);
    mbar_init(bar + B_GEMPTY, 10);
    mbar_init(bar + B_WFULL, 1);
    for (int k = 0; k < 3; ++k) mbar_init(bar + B_DONE + k, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    if (FAVOR) {
      mbar_arrive_expect_tx(bar + B_WFULL, (uint32_t)M * 128u);
      bulk_load(smem + lay.w, p.wimg + (size_t)(blockIdx.y % p.H) * p.wstride, (uint32_t)M * 128u, bar + B_WFULL);
    }
  }
  if (warp == 0) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t s_w = sbase + lay.w, s_g = sbase + lay.g, s_phk = sbase + lay.phk;
  auto slot_addr = [&](int n) { return sbase + lay.slots + (uint32_t)(n % kSlots) * kTileBytes; };
  auto slot_par = [&](int n) { return (uint32_t)((n / kSlots) & 1); };
  bool ok = true;
  auto wait = [&](int b, uint32_t par) {
    if (ok) ok = mbar_wait(bar + b, par, p.status, abort_flag);
    return ok;
  };
  auto arrive = [&](int b) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar + b);
  };
  const int q4 = warp & 3, row = 32 * q4 + lane;
  const uint32_t lane_base = 32u * q4;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int n = 0, keys = 0;
      auto load = [&](const CUtensorMap *m, int t, int bh) {
        const int s = n % kSlots, u = n / kSlots;
        if (u > 0 && !wait(B_EMPTY + s, (u - 1) & 1)) return false;
        mbar_arrive_expect_tx(bar + B_FULL + s, kTileBytes);
        tma_load_3d(smem + lay.slots + s * kTileBytes, m, bar + B_FULL + s, 0, t * kTile, bh);
        ++n;
        return true;
      };
      // unit j's staged increments -> dK, dV; returns once its slots are read
      auto flush = [&](int j, const Cursor &c) {
        if (!wait(B_STG + (j & 1), (j >> 1) & 1)) return false;
        tma_reduce_add_3d(&tmDV, slot_addr(2 * j + 1), 0, c.t * kTile, c.bh);
        tma_reduce_add_3d(&tmDK, slot_addr(2 * j), 0, c.t * kTile, c.bh);
        tma_store_commit();
        tma_store_wait_read();
        return true;
      };
      Cursor cur = first, prev1 = first, prev2 = first;  // units i, i-1, i-2
      for (int i = 0; i < nun && ok; ++i) {
        if (i >= 2 && !flush(i - 2, prev2)) break;  // unit i takes unit i-2's slots
        if (!load(&tmK, cur.t, cur.bh) || !load(&tmV, cur.t, cur.bh)) break;
        if (new_key(i, cur)) {
          // the previous G_end is no longer read once its last unit is done
          if (keys > 0 && !wait(B_GEMPTY, (keys - 1) & 1)) break;
          mbar_arrive_expect_tx(bar + B_GFULL, grec_bytes);
          bulk_load(smem + lay.g, p.grec + (size_t)(cur.bh * p.P + cur.seg) * grec_bytes, grec_bytes, bar + B_GFULL);
          ++keys;
        }
        prev2 = prev1;
        prev1 = cur;
        advance(cur);
      }
      // the last two units (prev2 = unit nun-2, prev1 = unit nun-1)
      if (ok && nun >= 2) flush(nun - 2, prev2);
      if (ok && nun >= 1) flush(nun - 1, prev1);
      tma_store_wait_all();
      for (int m = max(0, n - kSlots); m < n; ++m) mbar_drain(bar + B_FULL + m % kSlots, slot_par(m));
      if (keys > 0) mbar_drain(bar + B_GFULL, (keys - 1) & 1);
      if (FAVOR) mbar_drain(bar + B_WFULL, 0);
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- MMA issuers
    if (lane == 0 && (FAVOR || warp != 1)) {
      const uint32_t id64 = make_idesc(128, 64, false, false);
      const uint32_t id_o = make_idesc(128, D, false, true);
      auto ks = [](int s, uint32_t rows) { return (uint64_t)((s >> 2) * rows * 8u + (s & 3) * 2u); };
      if (warp == 1) {
        // F = K W: job j = features [64 (j % JT), +64) of unit j / JT into buffer j & 1
        wait(B_WFULL, 0);
        const uint64_t d_w0 = desc_kmajor(s_w, M, 0, 0);
        for (int j = 0; j < nun * JT && ok; ++j) {
          const int i = j / JT, jj = j - i * JT, nK = 2 * i;
          if (j >= 2 && !wait(B_FEMPTY + (j & 1), ((j >> 1) - 1) & 1)) break;
          if (jj == 0 && !wait(B_FULL + nK % kSlots, slot_par(nK))) break;
          tc_fence_after();
          const uint64_t dx = desc_kmajor(slot_addr(nK), kTile, 0, 0), dw = d_w0 + (uint64_t)(jj * 512);
#pragma unroll
          for (int s = 0; s < D / 16; ++s)
            mma_bf16(tbase + kF + 64 * (j & 1), dx + ks(s, kTile), dw + ks(s, M), id64, s > 0);
          mma_commit(bar + B_FFULL + (j & 1));
          if (jj == JT - 1) mma_commit(bar + B_EMPTY + nK % kSlots);
        }
      } else if (warp == 2) {
        // D = V G_V^T, the same jobs
        int keys = 0;
        Cursor cur = first;
        for (int i = 0; i < nun && ok; ++i, advance(cur)) {
          const int nK = 2 * i, nV = 2 * i + 1;
          if (new_key(i, cur) && !wait(B_GFULL, keys++ & 1)) break;
          if (!wait(B_FULL + nV % kSlots, slot_par(nV))) break;
          const uint64_t dv = desc_kmajor(slot_addr(nV), kTile, 0, 0);
          for (int jj = 0; jj < JT && ok; ++jj) {
            const int j = i * JT + jj;
            if (j >= 2 && !wait(B_DEMPTY + (j & 1), ((j >> 1) - 1) & 1)) break;
            tc_fence_after();
            const uint64_t dg = desc_kmajor(s_g, M, 64 * jj, 0);
#pragma unroll
            for (int s = 0; s < D / 16; ++s)
              mma_bf16(tbase + kDc + 64 * (j & 1), dv + ks(s, kTile), dg + ks(s, M), id64, s > 0);
            mma_commit(bar + B_DFULL + (j & 1));
          }
          if (!ok) break;
          mma_commit(bar + B_EMPTY + nV % kSlots);
          if (!FAVOR) mma_commit(bar + B_EMPTY + nK % kSlots);  // K is read by the epilogue alone
          if (last_of_key(i, cur)) mma_commit(bar + B_GEMPTY);
        }
      } else {
        // dV' = phi_k G_V and dK' = u W^T, per 128-feature block
        if (FAVOR) wait(B_WFULL, 0);
        int keys = 0;
        Cursor cur = first;
        for (int i = 0; i < nun && ok; ++i, advance(cur)) {
          if (new_key(i, cur) && !wait(B_GFULL, keys++ & 1)) break;
          for (int h = 0; h < nb && ok; ++h) {
            const uint32_t c = (uint32_t)(i * nb + h), b = c & 1;
            if (!wait(B_PHK + b, (c >> 1) & 1)) break;
            if (h == 0 && i > 0 && !wait(B_OUTEMPTY, (i - 1) & 1)) break;
            tc_fence_after();
            const uint32_t s_ph = s_phk + b * kTile * 256;
#pragma unroll
            for (int s = 0; s < FB / 16; ++s)
              mma_bf16(tbase + kDV, desc_kmajor(s_ph, kTile, 0, s), desc_mnmajor(s_g, M, 0, 8 * h + s), id_o,
                       (h > 0 || s > 0) ? 1u : 0u);
            mma_commit(bar + B_PHFREE + b);
            if (FAVOR) {
              if (!wait(B_U + b, (c >> 1) & 1)) break;
              tc_fence_after();
#pragma unroll
              for (int s = 0; s < FB / 16; ++s)
                mma_bf16_ta(tbase + kDK, tbase + kU + 64 * b + 8 * s, desc_mnmajor(s_w, M, 0, 8 * h + s), id_o,
                            (h > 0 || s > 0) ? 1u : 0u);
              mma_commit(bar + B_UFREE + b);
            }
          }
          if (!ok) break;
          mma_commit(bar + B_OUTFULL);
          if (last_of_key(i, cur)) mma_commit(bar + B_GEMPTY);
        }
      }
      mma_commit(bar + B_DONE + (warp - 1));
      mbar_drain(bar + B_DONE + (warp - 1), 0);
    }
  } else if (warp < 12) {
    // ---------------------------------------------------------------- phi_k, u
    const int part = (warp - 4) >> 2;  // columns [32 part, +32) of every 64-feature job
    const float *gs = reinterpret_cast<const float *>(smem + lay.gs);
    float *usum = reinterpret_cast<float *>(smem + lay.usum);
    int keys = 0;
    Cursor cur = first;
    for (int i = 0; i < nun && ok; ++i, advance(cur)) {
      const int nK = 2 * i;
      const uint32_t s_k = slot_addr(nK);
      const bool dead = row >= min(kTile, p.L - cur.t * kTile);
      if (new_key(i, cur) && !wait(B_GFULL, keys++ & 1)) break;
      if (!wait(B_FULL + nK % kSlots, slot_par(nK))) break;
      // padding rows: F = 0 (zero-filled tile) and 2^-inf = 0, no select
      const float ck = FAVOR ? (dead ? -INFINITY : favor_row_const(tile_row_sqnorm(s_k, row, D), M)) : 0.f;
      float uk = 0.f;
      for (int h = 0; h < nb && ok; ++h) {
        const uint32_t c = (uint32_t)(i * nb + h), b = c & 1;
        const uint32_t s_ph = s_phk + b * kTile * 256;
        for (int half = 0; half < FB / 64 && ok; ++half) {
          const int j = (i * nb + h) * (FB / 64) + half;  // the job (F and D alike)
          const int col = 64 * half + 32 * part;          // column within the block
          float v[32];
          if (FAVOR) {
            if (!wait(B_FFULL + (j & 1), (j >> 1) & 1)) break;
            tc_fence_after();
            tmem_ld32(tmem_addr(tbase, lane_base, kF + 64 * (j & 1) + 32 * part), v);
            tc_fence_before();
            arrive(B_FEMPTY + (j & 1));
#pragma unroll
            for (int x = 0; x < 32; x += 2) favor_feature2(v[x], v[x + 1], ck);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              ld_bf16x8(s_k + sw128_offset(row, col + 8 * q, kTile), v + 8 * q);
#pragma unroll
              for (int x = 0; x < 8; ++x) v[8 * q + x] = dead ? 0.f : elu1_feature(v[8 * q + x]);
            }
          }
          // phi_k as the MMAs see it (bf16), and u from the same values
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            pk[x] = pack_bf16(v[2 * x], v[2 * x + 1]);
            v[2 * x] = __uint_as_float(pk[x] << 16);
            v[2 * x + 1] = __uint_as_float(pk[x] & 0xFFFF0000u);
          }
          // the buffer's last block has been read by its dV' MMAs
          if (half == 0 && c >= 2 && !wait(B_PHFREE + b, ((c >> 1) - 1) & 1)) break;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_shared_v4(s_ph + sw128_offset(row, col + 8 * q, kTile), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                         pk[4 * q + 3]);
          // u = phi_k * (V G_V^T + G_S)   (elu+1: dphi_k' * min(phi_k, 1))
          float dd[32];
          if (!wait(B_DFULL + (j & 1), (j >> 1) & 1)) break;
          tc_fence_after();
          tmem_ld32(tmem_addr(tbase, lane_base, kDc + 64 * (j & 1) + 32 * part), dd);
          tc_fence_before();
          arrive(B_DEMPTY + (j & 1));
          const float *g = gs + 128 * h + col;
          if (FAVOR) {
            // feature pairs in packed fp32x2 arithmetic
            const float2 *g2 = reinterpret_cast<const float2 *>(g);
#pragma unroll
            for (int x = 0; x < 32; x += 2) {
              const float2 u2 = __fmul2_rn(make_float2(v[x], v[x + 1]), __fadd2_rn(make_float2(dd[x], dd[x + 1]), g2[x >> 1]));
              dd[x] = u2.x;
              dd[x + 1] = u2.y;
              uk += u2.x;
              uk += u2.y;
            }
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) {
              const float dk = dd[x] + g[x];
              dd[x] = dk * fminf(v[x], 1.f);
              uk += dd[x];
            }
          }
          if (FAVOR) {
            // u as bf16 pairs into TMEM: feature f of the block -> column f / 2
            if (half == 0 && c >= 2 && !wait(B_UFREE + b, ((c >> 1) - 1) & 1)) break;
            float pu[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) pu[x] = __uint_as_float(pack_bf16(dd[2 * x], dd[2 * x + 1]));
            tmem_st16(tmem_addr(tbase, lane_base, kU + 64 * b + col / 2), pu);
          } else {
            // elu+1 (M = d): u is dK's increment (feature m = column m); it
            // takes the place of this thread's K values in the K slot
#pragma unroll
            for (int q = 0; q < 4; ++q) st_bf16x8(s_k + sw128_offset(row, 128 * h + col + 8 * q, kTile), dd + 8 * q);
          }
        }
        if (!ok) break;
        fence_async_smem();
        arrive(B_PHK + b);
        if (FAVOR) {
          tmem_st_wait();
          tc_fence_before();
          arrive(B_U + b);
        }
      }
      if (!ok) break;
      usum[((i & 1) * 2 + part) * kTile + row] = uk;
      arrive(B_EPI + (i & 1));
      if (last_of_key(i, cur)) arrive(B_GEMPTY);  // G_S read for the last time
      fence_async_smem();
      arrive(B_STG + (i & 1));
    }
    // a wait that gave up between a block's two halves leaves u's store of
    // the first half unwaited: TMEM is freed after this
    if (FAVOR) tmem_st_wait();
  } else {
    // ---------------------------------------------------------------- dK, dV increments
    const float *usum = reinterpret_cast<const float *>(smem + lay.usum);
    for (int i = 0; i < nun && ok; ++i) {
      const int nK = 2 * i, nV = 2 * i + 1;
      const uint32_t s_k = slot_addr(nK), s_v = slot_addr(nV);
      if (!wait(B_OUTFULL, i & 1)) break;
      tc_fence_after();
      {
        // dV' -> bf16 over V (the D MMAs are done with it)
        float dv[64];
        tmem_ld32x2(tmem_addr(tbase, lane_base, kDV), tmem_addr(tbase, lane_base, kDV + 32), dv, dv + 32);
#pragma unroll
        for (int q = 0; q < 8; ++q) st_bf16x8(s_v + sw128_offset(row, 8 * q, kTile), dv + 8 * q);
      }
      if (FAVOR) {
        // dK' - k rowsum(u) -> bf16 over K (whose values are read first)
        float dk[64];
        tmem_ld32x2(tmem_addr(tbase, lane_base, kDK), tmem_addr(tbase, lane_base, kDK + 32), dk, dk + 32);
        tc_fence_before();
        arrive(B_OUTEMPTY);
        if (!wait(B_EPI + (i & 1), (i >> 1) & 1)) break;
        const float sk = usum[((i & 1) * 2) * kTile + row] + usum[((i & 1) * 2 + 1) * kTile + row];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float xk[8];
          ld_bf16x8(s_k + sw128_offset(row, 8 * q, kTile), xk);
#pragma unroll
          for (int x = 0; x < 8; x += 2) {
            const float2 r = __ffma2_rn(make_float2(-xk[x], -xk[x + 1]), make_float2(sk, sk),
                                        make_float2(dk[8 * q + x], dk[8 * q + x + 1]));
            dk[8 * q + x] = r.x;
            dk[8 * q + x + 1] = r.y;
          }
          st_bf16x8(s_k + sw128_offset(row, 8 * q, kTile), dk + 8 * q);
        }
      } else {
        tc_fence_before();
        arrive(B_OUTEMPTY);
      }
      fence_async_smem();
      arrive(B_STG + (i & 1));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

// G_end(s) of every record s < nrec from the segments' G totals (gstates,
// features-major [BH][P][M][D + 1]) by a running sum from the last segment
// down: G_end(s) = g_last + sum over s' > s of total(s'), where g_last
// (features-major [BH][M][D + 1]) is the reverse state arriving from later
// rows, or zero.  nrec = P - 1, or P with g_last (then it is the last
// segment's G_end).  A record, per (head, segment): bf16 [M][64] swizzled
// image of columns 0..63, then fp32 column 64.  One thread per (head,
// feature, group of 8 columns); group 7 also carries column 64.  With keep
// the running sums also go back over totals 1 .. P - 1 (the carried-state
// gradient reads G_end(0) there).
__global__ void scan_prep_g_kernel(float *__restrict__ gstates, const float *__restrict__ g_last,
                                   unsigned char *__restrict__ grec, int M, int P, int nrec, int BH, int keep) {
  const int DP = D + 1;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)BH * M * 8) return;
  const int c = (int)(i & 7);
  const long long fm = i >> 3;
  const int bh = (int)(fm / M), f = (int)(fm - (long long)bh * M);
  const int n = c == 7 ? 9 : 8;
  const size_t per = (size_t)M * DP, base = (size_t)f * DP + 8 * c;
  float acc[9];
#pragma unroll
  for (int j = 0; j < 9; ++j) acc[j] = (j < n && g_last) ? g_last[(size_t)bh * per + base + j] : 0.f;
  for (int s = nrec - 1; s >= 0; --s) {
    if (s + 1 < P) {
      float *src = gstates + ((size_t)bh * P + s + 1) * per + base;
#pragma unroll
      for (int j = 0; j < 9; ++j)
        if (j < n) {
          acc[j] += src[j];
          if (keep) src[j] = acc[j];
        }
    }
    unsigned char *rec = grec + ((size_t)bh * P + s) * (size_t)M * 132u;
    *reinterpret_cast<uint4 *>(rec + sw128_offset(f, 8 * c, M)) =
        make_uint4(pack_bf16(acc[0], acc[1]), pack_bf16(acc[2], acc[3]), pack_bf16(acc[4], acc[5]),
                   pack_bf16(acc[6], acc[7]));
    if (c == 7) reinterpret_cast<float *>(rec + (size_t)M * 128u)[f] = acc[8];
  }
}

// ---------------------------------------------------------------------------
// dW's share of the later segments' reverse state (FAVOR+, learnable W).
// For a row k of segment s, with G = G_end(s):
//   dphi_k' = V G_V^T + G_S,  u' = phi_k * dphi_k',  dW += k^T u'
// (the same u' whose u' W^T the correction kernel adds to dK).  One CTA per
// (segment < P - 1, or every segment when a reverse state arrives from later
// rows; head) walks the segment's tiles in order, 512 threads,
// four per row (TMEM lane quadrant w % 4, a quarter of the features each):
//   F = K W -> TMEM; phi_k -> shared tile; D = V G_V^T -> the same TMEM
//   columns; u' = phi_k * (D + G_S) over phi_k in place; dW^T += u'^T K on
//   the tensor cores (features on the lanes, accumulated over the segment)
// K and V are double-buffered: tile t + 1 loads while tile t computes.  The
// segment's dW^T is added to its partial [M][D] at the end.
struct DwParams {
  int L, P, tps, nt, BH, M;
  int H, wstride;  // heads; bf16 elements between per-head W^T images (0: one shared W)
  const __nv_bfloat16 *wimg;  // W^T image [M][64]
  const unsigned char *grec;  // per (head, segment): G_end image [M][64] bf16, then G_S fp32 [M]
  float *dwpart;              // fp32 [BH][P][M][D]: dW^T partials
  int *status;
};

template <int M>
struct DwLayout {
  static constexpr uint32_t kPhCols = M < 128 ? 128 : M;
  uint32_t w, g, gs, kv, ph, nrm, bars, total;
  __host__ __device__ DwLayout() {
    uint32_t o = 0;
    w = o; o += M * 128u;
    g = o; o += M * 128u;
    gs = o; o += M * 4u;  // directly after g: one bulk copy of the record
    o = (o + 1023u) & ~1023u;
    kv = o; o += 2 * 2 * kTileBytes;      // [buffer][K, V]
    ph = o; o += kTile * kPhCols * 2u;    // phi_k, then u', [row][feature] swizzled
    nrm = o; o += 4 * kTile * 4u;         // [part][row] partial |k|^2
    bars = o; o += 64;
    total = o;
  }
};

template <int M>
__global__ void __launch_bounds__(kThreads, 1)
    tc_dw_corr_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, DwParams p) {
  constexpr int nb = (M + 127) / 128;       // 128-feature blocks (dW MMAs)
  constexpr int QF = M / 4;                 // features per thread
  constexpr uint32_t kFD = 0, kW = M;       // TMEM: F, then D | dW^T, nb x 64 columns
  constexpr uint32_t kCols = M == 256 ? 512u : (M == 128 ? 256u : 128u);
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const DwLayout<M> lay;
  const uint32_t sb = smem_u32(smem);
  uint64_t *ld_bar = reinterpret_cast<uint64_t *>(smem + lay.bars);  // [2]
  uint64_t *setup_bar = ld_bar + 2;
  uint64_t *mma_bar = ld_bar + 3;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(ld_bar + 4);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(ld_bar + 5);
  uint64_t *drain_bar = ld_bar + 6;  // used once, after a timed-out wait
  float *nrm = reinterpret_cast<float *>(smem + lay.nrm);
  const float *gs = reinterpret_cast<const float *>(smem + lay.gs);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, part = warp >> 2, row = 32 * q4 + lane;
  const int seg = blockIdx.x, bh = blockIdx.y;
  // debug builds: a segment outside the plan records SLIM_ERR_BOUNDS and the CTA does nothing
  if (!SLIM_DCHECK(p.status, seg < p.P && bh < p.BH && seg * p.tps < p.nt)) return;
  const int t0 = seg * p.tps, t1 = min(t0 + p.tps, p.nt);
  const uint32_t s_w = sb + lay.w, s_g = sb + lay.g, s_ph = sb + lay.ph;

  if (tid == 0) {
    mbar_init(ld_bar, 1);
    mbar_init(ld_bar + 1, 1);
    mbar_init(setup_bar, 1);
    mbar_init(mma_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    mbar_arrive_expect_tx(setup_bar, (uint32_t)M * 256u + (uint32_t)M * 4u);
    bulk_load(smem + lay.w, p.wimg + (size_t)(bh % p.H) * p.wstride, (uint32_t)M * 128u, setup_bar);
    bulk_load(smem + lay.g, p.grec + ((size_t)bh * p.P + seg) * (size_t)M * 132u, (uint32_t)M * 132u, setup_bar);
    if (t0 < t1) {
      mbar_arrive_expect_tx(ld_bar, 2 * kTileBytes);
      tma_load_3d(smem + lay.kv, &tmK, ld_bar, 0, t0 * kTile, bh);
      tma_load_3d(smem + lay.kv + kTileBytes, &tmV, ld_bar, 0, t0 * kTile, bh);
    }
  }
  if (warp == 0) tmem_alloc(tslot, kCols);
  if (M < 128) {  // features beyond M stay zero: the dW MMA reads 128
    for (int idx = tid; idx < kTile * 128; idx += kThreads) {
      const int r = idx >> 7, x = idx & 127;
      if (x >= M) *reinterpret_cast<__nv_bfloat16 *>(smem + lay.ph + sw128_offset(r, x, kTile)) = __float2bfloat16_rn(0.f);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tslot;
  // false once a wait of this thread has given up (or seen another give
  // up): thread 0 then issues nothing more.  A wait that returns true saw
  // its phase complete, so while thread 0's waits succeed the barriers it
  // arms are in step, whatever another thread's wait did.
  bool go = true;
  go &= mbar_wait(setup_bar, 0, p.status, abort_flag);

  uint32_t mphase = 0;
  auto wait_mma = [&]() {
    __syncwarp();
    go &= mbar_wait(mma_bar, mphase, p.status, abort_flag);
    mphase ^= 1;
    tc_fence_after();
  };
  auto cta_sync = [&]() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  const uint32_t id_f = make_idesc(128, M, false, false);
  const uint32_t id_w = make_idesc(128, 64, true, true);

  for (int i = 0; t0 + i < t1; ++i) {
    const int t = t0 + i, b = i & 1;
    const uint32_t s_k = sb + lay.kv + (uint32_t)b * 2u * kTileBytes, s_v = s_k + kTileBytes;
    const bool live = row < min(kTile, p.L - t * kTile);
    go &= mbar_wait(ld_bar + b, (uint32_t)(i >> 1) & 1u, p.status, abort_flag);
    // F = K W
    if (tid == 0 && go) {
      for (int s = 0; s < D / 16; ++s)
        mma_bf16(tb + kFD, desc_kmajor(s_k, kTile, 0, s), desc_kmajor(s_w, M, 0, s), id_f, s > 0);
      mma_commit(mma_bar);
    }
    nrm[part * kTile + row] = tile_row_sqnorm_part(s_k, row, 16 * part, 16);
    __syncthreads();
    const float ck = live ? favor_row_const((nrm[row] + nrm[kTile + row]) + (nrm[2 * kTile + row] + nrm[3 * kTile + row]), M)
                          : -INFINITY;
    wait_mma();
    // every MMA of the previous tile is complete (in order, one commit):
    // its K, V buffer takes tile t + 1
    if (tid == 0 && go && t + 1 < t1) {
      uint64_t *nb_bar = ld_bar + (b ^ 1);
      const uint32_t nk = sb + lay.kv + (uint32_t)(b ^ 1) * 2u * kTileBytes;
      mbar_arrive_expect_tx(nb_bar, 2 * kTileBytes);
      tma_load_3d(smem + (nk - sb), &tmK, nb_bar, 0, (t + 1) * kTile, bh);
      tma_load_3d(smem + (nk - sb) + kTileBytes, &tmV, nb_bar, 0, (t + 1) * kTile, bh);
    }
    // phi_k (padding rows: F = 0 and 2^-inf = 0)
#pragma unroll
    for (int c = 0; c < QF; c += 16) {
      float v[16];
      tmem_ld16(tmem_addr(tb, 32 * q4, kFD + QF * part + c), v);
#pragma unroll
      for (int x = 0; x < 16; x += 2) favor_feature2(v[x], v[x + 1], ck);
      st_bf16x8(s_ph + sw128_offset(row, QF * part + c, kTile), v);
      st_bf16x8(s_ph + sw128_offset(row, QF * part + c + 8, kTile), v + 8);
    }
    cta_sync();  // F is read out: D may overwrite it
    // D = V G_V^T
    if (tid == 0 && go) {
      for (int s = 0; s < D / 16; ++s)
        mma_bf16(tb + kFD, desc_kmajor(s_v, kTile, 0, s), desc_kmajor(s_g, M, 0, s), id_f, s > 0);
      mma_commit(mma_bar);
    }
    wait_mma();
    // u' = phi_k * (D + G_S), over phi_k
#pragma unroll
    for (int c = 0; c < QF; c += 16) {
      const int f0 = QF * part + c;
      float dv[16], ph[16], g[16];
      tmem_ld16(tmem_addr(tb, 32 * q4, kFD + f0), dv);
      ld_bf16x8(s_ph + sw128_offset(row, f0, kTile), ph);
      ld_bf16x8(s_ph + sw128_offset(row, f0 + 8, kTile), ph + 8);
#pragma unroll
      for (int x = 0; x < 16; x += 4) *reinterpret_cast<float4 *>(g + x) = *reinterpret_cast<const float4 *>(gs + f0 + x);
#pragma unroll
      for (int x = 0; x < 16; ++x) ph[x] *= dv[x] + g[x];
      st_bf16x8(s_ph + sw128_offset(row, f0, kTile), ph);
      st_bf16x8(s_ph + sw128_offset(row, f0 + 8, kTile), ph + 8);
    }
    fence_async_smem();
    cta_sync();
    // dW^T += u'^T K, per 128-feature block; no commit of its own: the next
    // tile's F commit covers it (MMAs complete in order), the last one is
    // committed after the loop
    if (tid == 0 && go) {
      for (int h = 0; h < nb; ++h)
        for (int s = 0; s < kTile / 16; ++s)
          mma_bf16(tb + kW + 64 * h, desc_mnmajor(s_ph, kTile, 128 * h, s), desc_mnmajor(s_k, kTile, 0, s), id_w,
                   i > 0 || s > 0);
    }
  }
  if (t0 < t1) {
    if (tid == 0) mma_commit(mma_bar);
    wait_mma();
    if (!*abort_flag) {
      float *base = p.dwpart + ((size_t)bh * p.P + seg) * (size_t)M * D;
#pragma unroll
      for (int h = 0; h < nb; ++h) {
        float v[16];
        tmem_ld16(tmem_addr(tb, 32 * q4, kW + 64 * h + 16 * part), v);
        const int f = 128 * h + row;
        if (f < M) {
#pragma unroll
          for (int x = 0; x < 16; x += 4)
            red_add_v4(base + (size_t)f * D + 16 * part + x, v[x], v[x + 1], v[x + 2], v[x + 3]);
        }
      }
    }
  }
  if (tid == 0 && *abort_flag) {
    // a wait gave up (nothing was issued after it): this CTA's MMAs and the
    // loads armed before that land before TMEM is freed and the CTA leaves
    // (an armed phase completes when its bytes land; one with nothing armed
    // gives up after 20 ms)
    mma_commit(drain_bar);
    mbar_drain(drain_bar, 0);
    uint64_t *const armed[3] = {ld_bar, ld_bar + 1, setup_bar};
    for (int i = 0; i < 3; ++i)
      for (uint32_t par = 0; par < 2; ++par) mbar_drain(armed[i], par, 20000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, kCols);
}

template <int M>
cudaError_t launch_dw(const Plan &pl, const Args &a, const CUtensorMap &mk, const CUtensorMap &mv, int nrec,
                      cudaStream_t st) {
  DwParams p{};
  p.L = pl.L; p.P = pl.P; p.tps = pl.cps; p.nt = pl.tc_tiles; p.BH = pl.BH; p.M = M;
  p.H = pl.H; p.wstride = pl.wh > 1 ? M * 64 : 0;
  p.wimg = reinterpret_cast<const __nv_bfloat16 *>(a.ws + pl.wimg_off);
  p.grec = reinterpret_cast<const unsigned char *>(a.ws + pl.gimg_off);
  p.dwpart = a.ws + pl.dwpart_off;
  p.status = a.status;
  const DwLayout<M> lay;
  const int smem = (int)lay.total + 1024;
  auto kern = tc_dw_corr_kernel<M>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(nrec, pl.BH), kThreads, smem, st>>>(mk, mv, p);
  return cudaGetLastError();
}

template <bool FAVOR, int M>
cudaError_t launch(const Plan &pl, const Args &a, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mdk,
                   const CUtensorMap &mdv, bool all_segments, cudaStream_t st) {
  Params p{};
  p.L = pl.L; p.P = pl.P; p.tps = pl.cps; p.BH = pl.BH;
  p.H = pl.H; p.wstride = pl.wh > 1 ? M * 64 : 0;
  p.per_head = all_segments ? (long long)pl.tc_tiles : (long long)(pl.P - 1) * pl.cps;
  p.dk = static_cast<__nv_bfloat16 *>(a.dk);
  p.dv = static_cast<__nv_bfloat16 *>(a.dv);
  p.wimg = reinterpret_cast<const __nv_bfloat16 *>(a.ws + pl.wimg_off);
  p.grec = reinterpret_cast<const unsigned char *>(a.ws + pl.gimg_off);
  p.status = a.status;
  const Layout<M> lay;
  const int smem = (int)lay.total + 1024;
  auto kern = tc_corr_kernel<FAVOR, M>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (p.wstride == 0) {
    const long long units = p.per_head * pl.BH;
    const int grid = (int)std::min<long long>(sms, units);
    kern<<<grid, kThreads, smem, st>>>(mk, mv, mdk, mdv, p);
  } else {
    // one W per head: each CTA stays in one head (every CTA gets >= 1 unit)
    const long long per_head_ctas = std::max<long long>(1, std::min<long long>(p.per_head, sms / std::max(pl.BH, 1)));
    kern<<<dim3((unsigned)per_head_ctas, pl.BH), kThreads, smem, st>>>(mk, mv, mdk, mdv, p);
  }
  return cudaGetLastError();
}

}  // namespace tcc

cudaError_t tc_correction(const Plan &pl, const Args &a, const float *g_last, cudaStream_t st) {
  const int nrec = g_last ? pl.P : pl.P - 1;
  if (nrec < 1) return cudaSuccess;
  CUtensorMap mk, mv, mdk, mdv;
  if (!make_map_bf16_3d(&mk, a.k, pl.BH, pl.L, tcc::D, tcc::kTile) ||
      !make_map_bf16_3d(&mv, a.v, pl.BH, pl.L, tcc::D, tcc::kTile) ||
      !make_map_bf16_3d(&mdk, a.dk, pl.BH, pl.L, tcc::D, tcc::kTile) ||
      !make_map_bf16_3d(&mdv, a.dv, pl.BH, pl.L, tcc::D, tcc::kTile))
    return cudaErrorInvalidValue;
  {
    ProfScope ps("prep_g", st);
    const long long threads = (long long)pl.BH * pl.M * 8;
    const int keep = a.g_out != nullptr && pl.P > 1;
    tcc::scan_prep_g_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
        a.ws + pl.gstates_off, g_last, reinterpret_cast<unsigned char *>(a.ws + pl.gimg_off), pl.M, pl.P, nrec,
        pl.BH, keep);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  ProfScope ps("tc_backward_fix", st);
  const bool all = g_last != nullptr;
  if (!pl.favor)
    return pl.M == 64 ? tcc::launch<false, 64>(pl, a, mk, mv, mdk, mdv, all, st) : cudaErrorInvalidValue;
  if (pl.M == 64) return tcc::launch<true, 64>(pl, a, mk, mv, mdk, mdv, all, st);
  if (pl.M == 128) return tcc::launch<true, 128>(pl, a, mk, mv, mdk, mdv, all, st);
  if (pl.M == 256) return tcc::launch<true, 256>(pl, a, mk, mv, mdk, mdv, all, st);
  return cudaErrorInvalidValue;
}

cudaError_t tc_dw_correction(const Plan &pl, const Args &a, const float *g_last, cudaStream_t st) {
  const int nrec = g_last ? pl.P : pl.P - 1;
  if (nrec < 1 || !pl.favor || !a.dw) return cudaSuccess;
  CUtensorMap mk, mv;
  if (!make_map_bf16_3d(&mk, a.k, pl.BH, pl.L, tcc::D, tcc::kTile) ||
      !make_map_bf16_3d(&mv, a.v, pl.BH, pl.L, tcc::D, tcc::kTile))
    return cudaErrorInvalidValue;
  ProfScope ps("tc_dw_fix", st);
  if (pl.M == 64) return tcc::launch_dw<64>(pl, a, mk, mv, nrec, st);
  if (pl.M == 128) return tcc::launch_dw<128>(pl, a, mk, mv, nrec, st);
  if (pl.M == 256) return tcc::launch_dw<256>(pl, a, mk, mv, nrec, st);
  return cudaErrorInvalidValue;
}

}  // namespace slim
