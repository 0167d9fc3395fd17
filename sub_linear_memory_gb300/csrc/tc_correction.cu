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
// Warp roles, as in the forward: warp 0 streams K and V (and the bf16 image
// of G_end when the unit's segment changes) into shared memory, warp 1 issues
// the MMAs, warps 2-9 run the epilogues, two threads per row.  The epilogue
// stages each unit's bf16 increments of dK and dV in that unit's K and V
// slots, and warp 0 adds them to dK and dV with TMA reduce-add copies before
// it reuses the slots, so no global read sits in the epilogue.  Every
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
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kSlots = 4;  // K, V of two units in flight
constexpr uint32_t kTileBytes = kTile * D * 2;

struct Params {
  int L, P, tps, BH;
  long long per_head;  // units per head: tiles of segments 0 .. P-2
  __nv_bfloat16 *dk, *dv;
  const __nv_bfloat16 *wimg;  // W^T image [M][64] (FAVOR+)
  const unsigned char *grec;  // per (head, segment): G_end image [M][64] bf16, then G_S fp32 [M]
  int *status;
};

enum {
  B_FULL = 0,       // [4] TMA -> consumers
  B_EMPTY = 4,      // [4] MMAs done with the slot
  B_FFULL = 8,      // [2] F ready
  B_FEMPTY = 10,    // [2] F read out
  B_DFULL = 12,     // V G_V^T ready
  B_DEMPTY = 13,    // V G_V^T read out
  B_PHK = 14,       // phi_k block stored
  B_PHFREE = 15,    // dV' MMA done with the phi_k block
  B_U = 16,         // u block stored
  B_UFREE = 17,     // dK' MMA done with the u block
  B_OUTFULL = 18,   // dV', dK' complete
  B_OUTEMPTY = 19,  // dV', dK' read out
  B_GFULL = 20,     // G_end image landed
  B_GEMPTY = 21,    // G_end image no longer read (1 MMA commit + 8 epilogue warps)
  B_WFULL = 22,     // W image landed
  B_EPI = 23,       // epilogue warps' row-sum halves written
  B_DONE = 24,
  B_STG = 25,       // [2] a unit's dK, dV increments staged in its slots (by unit parity)
  B_COUNT = 27
};

template <int M>
struct Layout {
  static constexpr bool kFavor = true;
  uint32_t w, slots, g, gs, phk, ub, usum, bars, total;
  __host__ __device__ Layout() {
    uint32_t o = 0;
    w = o; o += M * 128u;
    slots = o; o += kSlots * kTileBytes;
    g = o; o += M * 128u;   // G_end[:, 0:64] as bf16 [M][64], swizzled
    gs = o; o += M * 4u;    // G_end[:, 64] fp32 (directly after g: one bulk copy)
    o = (o + 1023u) & ~1023u;
    phk = o; o += kTile * 128 * 2;
    ub = o; o += kTile * 128 * 2;
    usum = o; o += 2 * 2 * kTile * 4;  // [unit parity][half][row]
    bars = o; o += 8 * B_COUNT + 16;
    total = o;
  }
};

// TMEM columns
constexpr uint32_t kF0 = 0, kF1 = 128, kDc = 256, kDV = 384, kDK = 448;

template <bool FAVOR, int M>
__global__ void __launch_bounds__(kThreads, 1)
    tc_corr_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV, Params p) {
  constexpr int nb = (M + 127) / 128, FB = M < 128 ? M : 128, FC = FB / 2;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Layout<M> lay;
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + B_COUNT);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar + B_COUNT) + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // this CTA's units [u0, u1): unit u = (head, tile) over the first P-1 segments
  const long long units = p.per_head * p.BH;
  const long long u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
  const int nun = (int)(u1 - u0);
  // every role walks the same units with counters (no divisions per unit):
  // head bh, tile t, segment seg and position pos of the tile in it; the
  // segment's G_end changes when pos wraps
  struct Cursor {
    int bh, t, seg, pos;
  };
  const int per_head = (int)p.per_head;  // a multiple of tps
  Cursor first;
  first.bh = (int)(u0 / p.per_head);
  first.t = (int)(u0 - (long long)first.bh * p.per_head);
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
      ++c.bh;
    }
  };
  auto new_key = [&](int i, const Cursor &c) { return i == 0 || c.pos == 0; };
  auto last_of_key = [&](int i, const Cursor &c) { return i == nun - 1 || c.pos == p.tps - 1; };
  const uint32_t grec_bytes = (uint32_t)M * 132u;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar + B_FULL + s, 1);
      mbar_init(bar + B_EMPTY + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar + B_FFULL + b, 1);
      mbar_init(bar + B_FEMPTY + b, kEpiWarps);
    }
    mbar_init(bar + B_DFULL, 1);
    mbar_init(bar + B_DEMPTY, kEpiWarps);
    mbar_init(bar + B_PHK, kEpiWarps);
    mbar_init(bar + B_PHFREE, 1);
    mbar_init(bar + B_U, kEpiWarps);
    mbar_init(bar + B_UFREE, 1);
    mbar_init(bar + B_OUTFULL, 1);
    mbar_init(bar + B_OUTEMPTY, kEpiWarps);
    mbar_init(bar + B_GFULL, 1);
    mbar_init(bar + B_GEMPTY, 1 + kEpiWarps);
    mbar_init(bar + B_WFULL, 1);
    mbar_init(bar + B_EPI, kEpiWarps);
    mbar_init(bar + B_DONE, 1);
    mbar_init(bar + B_STG, kEpiWarps);
    mbar_init(bar + B_STG + 1, kEpiWarps);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    if (FAVOR) {
      mbar_arrive_expect_tx(bar + B_WFULL, (uint32_t)M * 128u);
      bulk_load(smem + lay.w, p.wimg, (uint32_t)M * 128u, bar + B_WFULL);
    }
  }
  if (warp == 0) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t s_w = sbase + lay.w, s_g = sbase + lay.g, s_phk = sbase + lay.phk, s_ub = sbase + lay.ub;
  auto slot_addr = [&](int n) { return sbase + lay.slots + (uint32_t)(n % kSlots) * kTileBytes; };
  auto slot_par = [&](int n) { return (uint32_t)((n / kSlots) & 1); };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int n = 0, keys = 0;
      bool ok = true;
      auto load = [&](const CUtensorMap *m, int t, int bh) {
        const int s = n % kSlots, u = n / kSlots;
        if (u > 0 && !mbar_wait(bar + B_EMPTY + s, (u - 1) & 1, p.status, abort_flag)) return false;
        mbar_arrive_expect_tx(bar + B_FULL + s, kTileBytes);
        tma_load_3d(smem + lay.slots + s * kTileBytes, m, bar + B_FULL + s, 0, t * kTile, bh);
        ++n;
        return true;
      };
      // unit j's staged increments -> dK, dV; returns once its slots are read
      auto flush = [&](int j, const Cursor &c) {
        if (!mbar_wait(bar + B_STG + (j & 1), (j >> 1) & 1, p.status, abort_flag)) return false;
        tma_reduce_add_3d(&tmDV, slot_addr(2 * j + 1), 0, c.t * kTile, c.bh);
        tma_reduce_add_3d(&tmDK, slot_addr(2 * j), 0, c.t * kTile, c.bh);
        tma_store_commit();
        tma_store_wait_read();
        return true;
      };
      Cursor cur = first, prev1 = first, prev2 = first;  // units i, i-1, i-2
      for (int i = 0; i < nun && ok; ++i) {
        if (i >= 2 && !flush(i - 2, prev2)) break;  // unit i takes unit i-2's slots
        // K and V first: the MMA warp issues this unit's F early, before it
        // releases the previous G_end
        ok = load(&tmK, cur.t, cur.bh) && load(&tmV, cur.t, cur.bh);
        if (ok && new_key(i, cur)) {
          // the previous G_end is no longer read once its last unit is done
          if (keys > 0 && !mbar_wait(bar + B_GEMPTY, (keys - 1) & 1, p.status, abort_flag)) break;
          mbar_arrive_expect_tx(bar + B_GFULL, grec_bytes);
          bulk_load(smem + lay.g, p.grec + (size_t)(cur.bh * p.P + cur.seg) * grec_bytes, grec_bytes, bar + B_GFULL);
          ++keys;
        }
        prev2 = prev1;
        prev1 = cur;
        advance(cur);
      }
      // the last two units (prev2 = unit nun-2, prev1 = unit nun-1)
      if (ok && nun >= 2) ok = flush(nun - 2, prev2);
      if (ok && nun >= 1) ok = flush(nun - 1, prev1);
      tma_store_wait_all();
      for (int m = max(0, n - kSlots); m < n; ++m) mbar_drain(bar + B_FULL + m % kSlots, slot_par(m));
      if (keys > 0) mbar_drain(bar + B_GFULL, (keys - 1) & 1);
      if (FAVOR) mbar_drain(bar + B_WFULL, 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      auto wait = [&](int b, uint32_t par) {
        if (ok) ok = mbar_wait(bar + b, par, p.status, abort_flag);
        return ok;
      };
      const uint32_t id_f = make_idesc(128, FB, false, false);
      const uint32_t id_o = make_idesc(128, D, false, true);
      if (FAVOR) wait(B_WFULL, 0);
      int fj = 0, dj = 0, keys = 0;
      // F = K W_h of unit j: issued one unit ahead, while unit j-1's later
      // MMAs run, so the epilogue finds it ready when it starts unit j
      auto f_job = [&](int j, int h) {
        const int nK = 2 * j;
        if (h == 0 && !wait(B_FULL + nK % kSlots, slot_par(nK))) return;
        const int b = fj & 1, use = fj >> 1;
        if (use > 0 && !wait(B_FEMPTY + b, (use - 1) & 1)) return;
        tc_fence_after();
        for (int s = 0; s < D / 16; ++s)
          mma_bf16(tbase + (b ? kF1 : kF0), desc_kmajor(slot_addr(nK), kTile, 0, s), desc_kmajor(s_w, M, 128 * h, s),
                   id_f, s > 0);
        mma_commit(bar + B_FFULL + b);
        ++fj;
      };
      if (FAVOR && nun > 0)
        for (int h = 0; h < nb && ok; ++h) f_job(0, h);
      Cursor cur = first;
      for (int i = 0; i < nun && ok; ++i, advance(cur)) {
        const int nK = 2 * i, nV = 2 * i + 1;
        const uint32_t s_v = slot_addr(nV);
        if (new_key(i, cur)) {
          if (!wait(B_GFULL, keys & 1)) break;
          ++keys;
        }
        if (!wait(B_FULL + nK % kSlots, slot_par(nK))) break;
        if (!wait(B_FULL + nV % kSlots, slot_par(nV))) break;
        tc_fence_after();
        for (int h = 0; h < nb && ok; ++h) {
          // V G_V,h^T
          if (dj > 0 && !wait(B_DEMPTY, (dj - 1) & 1)) break;
          tc_fence_after();
          for (int s = 0; s < D / 16; ++s)
            mma_bf16(tbase + kDc, desc_kmajor(s_v, kTile, 0, s), desc_kmajor(s_g, M, 128 * h, s), id_f, s > 0);
          mma_commit(bar + B_DFULL);
          ++dj;
        }
        if (!ok) break;
        mma_commit(bar + B_EMPTY + nK % kSlots);  // K's last reader (F of this unit) was issued earlier
        mma_commit(bar + B_EMPTY + nV % kSlots);
        for (int h = 0; h < nb && ok; ++h) {
          const uint32_t c = (uint32_t)(i * nb + h);
          if (!wait(B_PHK, c & 1)) break;
          if (h == 0 && i > 0 && !wait(B_OUTEMPTY, (i - 1) & 1)) break;
          tc_fence_after();
          // dV' += phi_k,h G_V,h
          for (int s = 0; s < FB / 16; ++s)
            mma_bf16(tbase + kDV, desc_kmajor(s_phk, kTile, 0, s), desc_mnmajor(s_g, M, 0, 8 * h + s), id_o,
                     (h > 0 || s > 0) ? 1u : 0u);
          mma_commit(bar + B_PHFREE);
          // this block's F buffer has been read: the next unit's F_h may go in
          if (FAVOR && i + 1 < nun) f_job(i + 1, h);
          if (FAVOR) {
            if (!wait(B_U, c & 1)) break;
            tc_fence_after();
            // dK' += u_h W_h^T
            for (int s = 0; s < FB / 16; ++s)
              mma_bf16(tbase + kDK, desc_kmajor(s_ub, kTile, 0, s), desc_mnmajor(s_w, M, 0, 8 * h + s), id_o,
                       (h > 0 || s > 0) ? 1u : 0u);
            mma_commit(bar + B_UFREE);
          }
        }
        if (!ok) break;
        mma_commit(bar + B_OUTFULL);
        if (last_of_key(i, cur)) mma_commit(bar + B_GEMPTY);
      }
      mma_commit(bar + B_DONE);
      mbar_drain(bar + B_DONE, 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q4 = warp & 3, half = (warp - 2) >> 2, row = 32 * q4 + lane;
    const uint32_t lane_base = 32u * q4;
    bool ok = true;
    auto wait = [&](int b, uint32_t par) {
      if (ok) ok = mbar_wait(bar + b, par, p.status, abort_flag);
      return ok;
    };
    auto arrive = [&](int b) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar + b);
    };
    const float *gs = reinterpret_cast<const float *>(smem + lay.gs);
    float *usum = reinterpret_cast<float *>(smem + lay.usum);
    int fj = 0, dj = 0, keys = 0;
    Cursor cur = first;
    for (int i = 0; i < nun && ok; ++i, advance(cur)) {
      const int t = cur.t;
      const int nK = 2 * i, nV = 2 * i + 1;
      const uint32_t s_k = slot_addr(nK);
      const int valid = min(kTile, p.L - t * kTile);
      const bool dead = row >= valid;
      if (new_key(i, cur)) {
        if (!wait(B_GFULL, keys & 1)) break;
        ++keys;
      }
      if (!wait(B_FULL + nK % kSlots, slot_par(nK))) break;
      const float ck = FAVOR ? favor_row_const(tile_row_sqnorm(s_k, row, D), M) : 0.f;
      float uk = 0.f;
      for (int h = 0; h < nb && ok; ++h) {
        const uint32_t c = (uint32_t)(i * nb + h);
        const int f0 = 128 * h + FC * half;  // first feature of this thread
        float v[64];
        if (FAVOR) {
          const int b = fj & 1, use = fj >> 1;
          if (!wait(B_FFULL + b, use & 1)) break;
          tc_fence_after();
          const uint32_t a = tmem_addr(tbase, lane_base, (b ? kF1 : kF0) + FC * half);
          if (FC == 64)
            tmem_ld32x2(a, a + 32, v, v + 32);
          else
            tmem_ld32(a, v);
          tc_fence_before();
          arrive(B_FEMPTY + b);
          ++fj;
#pragma unroll
          for (int x = 0; x < 64; ++x)
            if (x < FC) v[x] = dead ? 0.f : favor_feature(v[x], ck);
        } else {
#pragma unroll
          for (int j = 0; j < FC / 8; ++j) {
            ld_bf16x8(s_k + sw128_offset(row, FC * half + 8 * j, kTile), v + 8 * j);
#pragma unroll
            for (int x = 0; x < 8; ++x) v[8 * j + x] = dead ? 0.f : elu1_feature(v[8 * j + x]);
          }
        }
        // phi_k block -> smem for dV' (after the previous block's dV' read it)
        if (c > 0 && !wait(B_PHFREE, (c - 1) & 1)) break;
#pragma unroll
        for (int j = 0; j < FC / 8; ++j) st_bf16x8(s_phk + sw128_offset(row, FC * half + 8 * j, kTile), v + 8 * j);
        fence_async_smem();
        arrive(B_PHK);
        // u = phi_k * (V G_V^T + G_S) with phi_k as stored (bf16)
        if (!wait(B_DFULL, dj & 1)) break;
        tc_fence_after();
        float d[64];
        {
          const uint32_t a = tmem_addr(tbase, lane_base, kDc + FC * half);
          if (FC == 64)
            tmem_ld32x2(a, a + 32, d, d + 32);
          else
            tmem_ld32(a, d);
        }
        tc_fence_before();
        arrive(B_DEMPTY);
        ++dj;
#pragma unroll
        for (int j = 0; j < FC / 8; ++j) {
          float fk[8];
          ld_bf16x8(s_phk + sw128_offset(row, FC * half + 8 * j, kTile), fk);
#pragma unroll
          for (int x = 0; x < 8; ++x) {
            const float dk = d[8 * j + x] + gs[f0 + 8 * j + x];
            d[8 * j + x] = FAVOR ? fk[x] * dk : dk * fminf(fk[x], 1.f);
            uk += d[8 * j + x];
          }
        }
        if (FAVOR) {
          if (c > 0 && !wait(B_UFREE, (c - 1) & 1)) break;
#pragma unroll
          for (int j = 0; j < FC / 8; ++j) st_bf16x8(s_ub + sw128_offset(row, FC * half + 8 * j, kTile), d + 8 * j);
          fence_async_smem();
          arrive(B_U);
        } else {
          // elu+1 (M = d): u is dK's increment (feature m = column m); it takes
          // the place of this thread's K values in the K slot
#pragma unroll
          for (int j = 0; j < FC / 8; ++j) st_bf16x8(s_k + sw128_offset(row, f0 + 8 * j, kTile), d + 8 * j);
        }
      }
      if (!ok) break;
      if (FAVOR) usum[((i & 1) * 2 + half) * kTile + row] = uk;
      arrive(B_EPI);
      if (last_of_key(i, cur)) arrive(B_GEMPTY);  // G_S read for the last time
      // dV += dV', dK += dK' - k rowsum(u)
      if (!wait(B_OUTFULL, i & 1)) break;
      tc_fence_after();
      float dv[32], dkk[32];
      tmem_ld32x2(tmem_addr(tbase, lane_base, kDV + 32 * half), tmem_addr(tbase, lane_base, kDK + 32 * half), dv,
                  dkk);
      tc_fence_before();
      arrive(B_OUTEMPTY);
      if (!wait(B_EPI, i & 1)) break;
      // increments -> bf16 in this unit's slots (dV over V; dK over K, whose
      // values this thread reads first); rows past L are clipped by the TMA
      const uint32_t s_v = slot_addr(nV);
#pragma unroll
      for (int j = 0; j < 4; ++j) st_bf16x8(s_v + sw128_offset(row, 32 * half + 8 * j, kTile), dv + 8 * j);
      if (FAVOR) {
        const float sk = usum[((i & 1) * 2) * kTile + row] + usum[((i & 1) * 2 + 1) * kTile + row];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float xk[8];
          ld_bf16x8(s_k + sw128_offset(row, 32 * half + 8 * j, kTile), xk);
#pragma unroll
          for (int x = 0; x < 8; ++x) dkk[8 * j + x] = fmaf(-xk[x], sk, dkk[8 * j + x]);
          st_bf16x8(s_k + sw128_offset(row, 32 * half + 8 * j, kTile), dkk + 8 * j);
        }
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

// G_end(s) = gstates[s + 1] (after the reverse scan) -> per (head, segment)
// record: bf16 [M][64] swizzled image of columns 0..63, then fp32 column 64.
__global__ void prep_g_kernel(const float *__restrict__ gstates, unsigned char *__restrict__ grec, int M, int P,
                              int BH) {
  const int DP = D + 1;
  const long long n = (long long)BH * (P - 1) * M * DP;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int e = (int)(idx % DP);
    const long long r = idx / DP;
    const int f = (int)(r % M);
    const long long hs = r / M;  // bh * (P - 1) + s
    const int s = (int)(hs % (P - 1));
    const int bh = (int)(hs / (P - 1));
    const float g = gstates[(((size_t)bh * P + s + 1) * M + f) * DP + e];
    unsigned char *rec = grec + ((size_t)bh * P + s) * (size_t)M * 132u;
    if (e < D)
      *reinterpret_cast<__nv_bfloat16 *>(rec + sw128_offset(f, e, M)) = __float2bfloat16_rn(g);
    else
      reinterpret_cast<float *>(rec + (size_t)M * 128u)[f] = g;
  }
}

template <bool FAVOR, int M>
cudaError_t launch(const Plan &pl, const Args &a, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mdk,
                   const CUtensorMap &mdv, cudaStream_t st) {
  Params p{};
  p.L = pl.L; p.P = pl.P; p.tps = pl.cps; p.BH = pl.BH;
  p.per_head = (long long)(pl.P - 1) * pl.cps;
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
  const long long units = p.per_head * pl.BH;
  const int grid = (int)std::min<long long>(sms, units);
  kern<<<grid, kThreads, smem, st>>>(mk, mv, mdk, mdv, p);
  return cudaGetLastError();
}

}  // namespace tcc

cudaError_t tc_correction(const Plan &pl, const Args &a, cudaStream_t st) {
  if (pl.P < 2) return cudaSuccess;
  CUtensorMap mk, mv, mdk, mdv;
  if (!make_map_bf16_3d(&mk, a.k, pl.BH, pl.L, tcc::D, tcc::kTile) ||
      !make_map_bf16_3d(&mv, a.v, pl.BH, pl.L, tcc::D, tcc::kTile) ||
      !make_map_bf16_3d(&mdk, a.dk, pl.BH, pl.L, tcc::D, tcc::kTile) ||
      !make_map_bf16_3d(&mdv, a.dv, pl.BH, pl.L, tcc::D, tcc::kTile))
    return cudaErrorInvalidValue;
  {
    ProfScope ps("prep_g", st);
    const long long n = (long long)pl.BH * (pl.P - 1) * pl.M * (tcc::D + 1);
    const int blocks = (int)std::min<long long>((n + 255) / 256, 4096);
    tcc::prep_g_kernel<<<blocks, 256, 0, st>>>(a.ws + pl.gstates_off,
                                               reinterpret_cast<unsigned char *>(a.ws + pl.gimg_off), pl.M, pl.P,
                                               pl.BH);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  ProfScope ps("tc_backward_fix", st);
  if (!pl.favor) return pl.M == 64 ? tcc::launch<false, 64>(pl, a, mk, mv, mdk, mdv, st) : cudaErrorInvalidValue;
  if (pl.M == 64) return tcc::launch<true, 64>(pl, a, mk, mv, mdk, mdv, st);
  if (pl.M == 128) return tcc::launch<true, 128>(pl, a, mk, mv, mdk, mdv, st);
  if (pl.M == 256) return tcc::launch<true, 256>(pl, a, mk, mv, mdk, mdv, st);
  return cudaErrorInvalidValue;
}

}  // namespace slim
