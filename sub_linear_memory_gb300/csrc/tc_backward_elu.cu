// tc_backward_elu.cu -- tensor-core (tcgen05 + TMA) SLiM backward for the
// elementwise map g(x) = elu(x) + 1 at d = M = 128, bf16 I/O.
//
// "Sub-Linear Memory: How to Make Performers SLiM", section 3.3.  The same
// per-tile recurrence as the d = 64 backward (tc_backward.cu), walked in
// reverse over a segment of 128-row tiles:
//   R -= phi_k^T V,  S -= phi_k^T 1            eq. (19)
//   A = tril(phi_q phi_k^T),  num = A V + phi_q R^T,  den = rowsum(A) + phi_q . S
//   dN = dY / den,  dD = -(dY . num) / den^2
//   dA = tril(dN V^T + dD 1^T)
//   dV = A^T dN + phi_k G^T
//   dphi_q = dA phi_k + dN R^T + dD S^T,   dphi_k = dA^T phi_q + V G^T + G_S
//   G += phi_q^T dN,  G_S += phi_q^T dD        eq. (20)
//   dQ = dphi_q * min(phi_q, 1), dK likewise  (g'(x) = min(g(x), 1))
// At d = 128 the states R and G are 128 x 128, too many TMEM columns for one
// CTA next to the two 128-column transients, so a segment runs on a cluster
// of two CTAs that split the value columns: CTA c owns columns
// [64c, 64c + 64) of R, G, V, num and dV, as double-float R (hi, lo) and
// fp32 G in TMEM (features on the lanes).  Every row-wise quantity is
// formed in full on both CTAs (phi, A, den, dN, dA): only dY . num, a sum
// over value columns, is swapped (one float per row, distributed shared
// memory).  dV is complete per CTA; dphi_q and dphi_k are sums over value
// columns, so each CTA adds its share (CTA 0 also the terms that need no
// value column) into the zeroed dQ, dK with TMA reduce-adds.  S and G_S
// (features only) are kept on the CUDA cores in shared memory, S as a
// double-float pair.  The later segments' G reaches dK and dV through the
// correction kernel below (elu_corr_kernel).
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace slim {
namespace tce {

using namespace slim::tc;

constexpr int kThreads = 512;
constexpr int kParts = 4;  // threads per row (TMEM lane): warps w, w + 4, w + 8, w + 12
constexpr int kTile = 128;
constexpr int D = 128;     // value columns (= features)
constexpr int DH = 64;     // value columns per CTA
constexpr uint32_t kTileBytes = kTile * D * 2;  // a 128 x 128 bf16 tile
constexpr uint32_t kHalfBytes = kTile * 64 * 2;  // one 64-column block of it

struct Params {
  int L, nt, P, tps, BH;
  __nv_bfloat16 *dv;
  const float *states;     // fp32 [BH][P][D][D + 1]: inclusive segment-end R' (high parts), features major
  const float *states_lo;  // low parts
  float *gstates;          // fp32 [BH][P][D][D + 1]: segment totals of G (out)
  int *status;
};

struct Layout {
  uint32_t q, k, v, dy, at, rb, gv, s_hi, s_lo, gs, dd, asum, dot, rx, bars, total;
  __host__ __device__ Layout() {
    uint32_t o = 0;
    q = o; o += kTileBytes;   // Q, then phi_q in place, then the dQ share
    k = o; o += kTileBytes;   // K, then phi_k in place, then the dK share
    v = o; o += kTileBytes;
    dy = o; o += kTileBytes;  // dY, then dN in place
    at = o; o += kTileBytes;  // masked A, then masked dA
    rb = o; o += kHalfBytes;  // bf16 copy of this CTA's R columns, [feature][column]
    gv = o; o += kHalfBytes;  // bf16 copy of this CTA's G columns
    s_hi = o; o += D * 4;     // S as a double-float pair
    s_lo = o; o += D * 4;
    gs = o; o += D * 4;       // G_S (CTA 0)
    dd = o; o += kTile * 4;   // dD per row
    asum = o; o += kParts * kTile * 4;  // [part][row] den partials; column sums of phi
    dot = o; o += kParts * kTile * 4;   // [part][row] dY . num partials; column sums of dD phi_q
    rx = o; o += kTile * 4;   // the peer's dY . num partial per row
    bars = o; o += 128;
    total = o;
  }
};

// TMEM: R (hi, lo) and G, 64 columns each, then two 128-column transients
constexpr uint32_t kRhi = 0, kRlo = 64, kG = 128, kT = 256, kX = 384;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    elu_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDY,
                   const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK, Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Layout lay;
  const uint32_t sb = smem_u32(smem);
  uint64_t *in_bar = reinterpret_cast<uint64_t *>(smem + lay.bars);  // Q, K
  uint64_t *in2_bar = in_bar + 1;                                     // V, dY
  uint64_t *mma_bar = in_bar + 2;
  uint64_t *mmb_bar = in_bar + 3;  // a group whose epilogue overlaps the group after it
  uint64_t *x1_full = in_bar + 4;  // the peer's dY . num partials landed
  uint64_t *x1_free = in_bar + 5;  // the peer may send them
  uint32_t *tslot = reinterpret_cast<uint32_t *>(in_bar + 6);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(in_bar + 7);
  // used once, after a timed-out wait: completes when every MMA issued so far has
  uint64_t *drain_bar = in_bar + 8;
  float *s_hi = reinterpret_cast<float *>(smem + lay.s_hi);
  float *s_lo = reinterpret_cast<float *>(smem + lay.s_lo);
  float *gs = reinterpret_cast<float *>(smem + lay.gs);
  float *dd = reinterpret_cast<float *>(smem + lay.dd);
  float *asum = reinterpret_cast<float *>(smem + lay.asum);
  float *dot = reinterpret_cast<float *>(smem + lay.dot);
  float *rx = reinterpret_cast<float *>(smem + lay.rx);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, part = warp >> 2, row = 32 * q4 + lane;
  const int rank = (int)cluster_rank(), peer = 1 - rank;
  const int cv = DH * rank;  // this CTA's first value column
  const int seg = blockIdx.x >> 1, bh = blockIdx.y;
  const int t0 = seg * p.tps, t1 = min(t0 + p.tps, p.nt);
  const uint32_t s_q = sb + lay.q, s_k = sb + lay.k, s_v = sb + lay.v, s_dy = sb + lay.dy;
  const uint32_t s_at = sb + lay.at, s_rb = sb + lay.rb, s_gv = sb + lay.gv;

  if (tid == 0) {
    mbar_init(in_bar, 1);
    mbar_init(in2_bar, 1);
    mbar_init(mma_bar, 1);
    mbar_init(mmb_bar, 1);
    mbar_init(x1_full, 1);
    mbar_init(x1_free, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDY);
  }
  if (warp == 0) tmem_alloc(tslot, 512);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer is running before any remote store
  tc_fence_after();
  const uint32_t tb = *tslot;
  // false once a wait of this thread has given up (or seen another give
  // up): thread 0 then issues nothing more.  A wait that returns true saw
  // its phase complete, so while thread 0's waits succeed the barriers it
  // arms are in step, whatever another thread's wait did.
  bool go = true;

  auto load_qk = [&](int t) {
    mbar_arrive_expect_tx(in_bar, 2 * kTileBytes);
    for (int c = 0; c < D; c += 64) {
      tma_load_3d(smem + lay.q + c * kTile * 2, &tmQ, in_bar, c, t * kTile, bh);
      tma_load_3d(smem + lay.k + c * kTile * 2, &tmK, in_bar, c, t * kTile, bh);
    }
  };
  auto load_v = [&](int t) {  // V and dY share in2_bar; dY is issued later
    mbar_arrive_expect_tx(in2_bar, 2 * kTileBytes);
    for (int c = 0; c < D; c += 64) tma_load_3d(smem + lay.v + c * kTile * 2, &tmV, in2_bar, c, t * kTile, bh);
  };
  auto load_dy = [&](int t) {
    for (int c = 0; c < D; c += 64) tma_load_3d(smem + lay.dy + c * kTile * 2, &tmDY, in2_bar, c, t * kTile, bh);
  };
  if (tid == 0 && t0 < t1) {
    load_qk(t1 - 1);
    load_v(t1 - 1);
    load_dy(t1 - 1);
  }

  // R <- this CTA's columns of the inclusive state at the segment end (hi, lo),
  // G <- 0; S (hi, lo) and G_S in shared memory
  {
    const size_t base = ((size_t)bh * p.P + seg) * (size_t)D * (D + 1);
    const float *sh = p.states + base + (size_t)row * (D + 1) + cv + 16 * part;
    const float *sl = p.states_lo + base + (size_t)row * (D + 1) + cv + 16 * part;
    float h[16], l[16], z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      h[i] = sh[i];
      l[i] = sl[i];
      z[i] = 0.f;
    }
    tmem_st16(tmem_addr(tb, 32 * q4, kRhi + 16 * part), h);
    tmem_st16(tmem_addr(tb, 32 * q4, kRlo + 16 * part), l);
    tmem_st16(tmem_addr(tb, 32 * q4, kG + 16 * part), z);
    if (tid < D) {
      s_hi[tid] = p.states[base + (size_t)tid * (D + 1) + D];
      s_lo[tid] = p.states_lo[base + (size_t)tid * (D + 1) + D];
      gs[tid] = 0.f;
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  uint32_t in_phase = 0, in2_phase = 0, mma_phase = 0, mmb_phase = 0, x_phase = 0;
  const uint32_t peer_x1_full = map_peer(smem_u32(x1_full), peer);
  const uint32_t peer_x1_free = map_peer(smem_u32(x1_free), peer);
  auto wait_mma = [&]() {
    __syncwarp();
    go &= mbar_wait(mma_bar, mma_phase, p.status, abort_flag);
    mma_phase ^= 1;
    tc_fence_after();
  };
  auto wait_mmb = [&]() {
    __syncwarp();
    go &= mbar_wait(mmb_bar, mmb_phase, p.status, abort_flag);
    mmb_phase ^= 1;
    tc_fence_after();
  };
  auto cta_sync = [&]() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  // thread 0 issues every MMA, copy and barrier arm; once a wait of this CTA
  // has given up it issues nothing more, so the drain after the loop covers
  // everything in flight
  auto issue0 = [&]() { return tid == 0 && go; };

  for (int t = t1 - 1; t >= t0; --t) {
    const int valid = min(kTile, p.L - t * kTile);
    const bool live = row < valid;
    go &= mbar_wait(in_bar, in_phase, p.status, abort_flag);
    in_phase ^= 1;
    if (issue0()) {
      mbar_arrive_expect_tx(x1_full, kTile * 4);
      if (t > t0) {
        tma_prefetch_3d(&tmQ, 0, (t - 1) * kTile, bh);
        tma_prefetch_3d(&tmQ, 64, (t - 1) * kTile, bh);
        tma_prefetch_3d(&tmK, 0, (t - 1) * kTile, bh);
        tma_prefetch_3d(&tmK, 64, (t - 1) * kTile, bh);
      }
    }

    // (b) phi = elu + 1 in place over Q and K (this thread: 32 columns of its
    // row); padding rows past L get phi = 0
    for (int side = 0; side < 2; ++side) {
      const uint32_t s_x = side ? s_k : s_q;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float v[8];
        const uint32_t a = s_x + sw128_offset(row, 32 * part + 8 * j, kTile);
        ld_bf16x8(a, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = live ? elu1_feature(v[i]) : 0.f;
        st_bf16x8(a, v);
      }
    }
    fence_async_smem();
    cta_sync();
    // my receive slot is free (read in the last tile's (f)): the peer may send
    if (tid == 32 && go) mbar_arrive_remote(peer_x1_free);

    // (c) A = phi_q phi_k^T -> X (its own commit), and eq. (19): this CTA's
    // increment phi_k^T V[:, own] -> T
    if (issue0()) {
      const uint32_t id = make_idesc(128, 128, false, false);
      for (int s = 0; s < kTile / 16; ++s)
        mma_bf16(tb + kX, desc_kmajor(s_q, kTile, 0, s), desc_kmajor(s_k, kTile, 0, s), id, s > 0);
      mma_commit(mmb_bar);
    }
    go &= mbar_wait(in2_bar, in2_phase, p.status, abort_flag);  // V (and dY, read in (f))
    in2_phase ^= 1;
    if (issue0()) {
      const uint32_t id = make_idesc(128, DH, true, true);
      for (int s = 0; s < kTile / 16; ++s)
        mma_bf16(tb + kT, desc_mnmajor(s_k, kTile, 0, s), desc_mnmajor(s_v, kTile, cv, s), id, s > 0);
      mma_commit(mma_bar);
    }
    // column sums of phi_k over this thread's quarter of the rows (S update)
    {
      const int f = tid & (D - 1), g = tid >> 7;
      float cs = 0.f;
      const unsigned char *kb = smem + lay.k;
#pragma unroll 8
      for (int j = 32 * g; j < 32 * g + 32; ++j)
        cs += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(kb + sw128_offset(j, f, kTile)));
      dot[g * kTile + f] = cs;
    }
    wait_mmb();
    // tril(A) (diagonal kept) -> bf16 tile, and this part's row sum of it
    {
      float v[32];
      tmem_ld32(tmem_addr(tb, 32 * q4, kX + 32 * part), v);
      // r4[i & 3] sums as two packed pairs: (0, 1), (2, 3)
      float2 r4[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        if (32 * part + i > row) v[i] = 0.f;
        if (32 * part + i + 1 > row) v[i + 1] = 0.f;
        r4[(i >> 1) & 1] = __fadd2_rn(r4[(i >> 1) & 1], make_float2(v[i], v[i + 1]));
      }
      asum[part * kTile + row] = (r4[0].x + r4[0].y) + (r4[1].x + r4[1].y);
#pragma unroll
      for (int j = 0; j < 4; ++j) st_bf16x8(s_at + sw128_offset(row, 32 * part + 8 * j, kTile), v + 8 * j);
    }
    wait_mma();
    // eq. (19) on the double-float master; the bf16 copy of R's own columns
    // ([feature][column]) for the MMAs
    {
      const int c = 16 * part;
      float x[16], h[16], l[16];
      tmem_ld16x3(tmem_addr(tb, 32 * q4, kT + c), tmem_addr(tb, 32 * q4, kRhi + c),
                  tmem_addr(tb, 32 * q4, kRlo + c), x, h, l);
#pragma unroll
      for (int i = 0; i < 16; ++i) df_add(h[i], l[i], -x[i]);
      tmem_st16(tmem_addr(tb, 32 * q4, kRhi + c), h);
      tmem_st16(tmem_addr(tb, 32 * q4, kRlo + c), l);
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = h[i] + l[i];
#pragma unroll
      for (int i = 0; i < 16; i += 8) st_bf16x8(s_rb + sw128_offset(row, c + i, D), x + i);
    }
    // no MMA reads the masters and only this thread rereads its columns (the
    // next tile): their stores are waited for after dN, off these barriers
    cta_sync();  // the column sums are in
    if (tid < D) {
      const float cs = (dot[tid] + dot[kTile + tid]) + (dot[2 * kTile + tid] + dot[3 * kTile + tid]);
      float h = s_hi[tid], l = s_lo[tid];
      df_add(h, l, -cs);
      s_hi[tid] = h;
      s_lo[tid] = l;
    }
    fence_async_smem();
    cta_sync();

    // (f) num = A V[:, own] + phi_q R[own]^T -> T; den = rowsum(tril A) +
    // phi_q . S on the CUDA cores while the MMAs run, and the bf16 copy of G
    if (issue0()) {
      const uint32_t id = make_idesc(128, DH, false, true);
      for (int s = 0; s < kTile / 16; ++s)
        mma_bf16(tb + kT, desc_kmajor(s_at, kTile, 0, s), desc_mnmajor(s_v, kTile, cv, s), id, s > 0);
      for (int s = 0; s < D / 16; ++s)
        mma_bf16(tb + kT, desc_kmajor(s_q, kTile, 0, s), desc_mnmajor(s_rb, D, 0, s), id, 1);
      mma_commit(mma_bar);
    }
    {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float fq[8];
        const int f0 = 32 * part + 8 * j;
        ld_bf16x8(s_q + sw128_offset(row, f0, kTile), fq);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i & 3] = fmaf(fq[i], s_hi[f0 + i] + s_lo[f0 + i], acc[i & 3]);
      }
      asum[part * kTile + row] += (acc[0] + acc[1]) + (acc[2] + acc[3]);
      float g[16];
      tmem_ld16(tmem_addr(tb, 32 * q4, kG + 16 * part), g);
#pragma unroll
      for (int i = 0; i < 16; i += 8) st_bf16x8(s_gv + sw128_offset(row, 16 * part + i, D), g + i);
    }
    wait_mma();
    {
      // dY . num over this CTA's columns; the peer sends its share (one float per row)
      float v[16], g[16];
      tmem_ld16(tmem_addr(tb, 32 * q4, kT + 16 * part), v);
#pragma unroll
      for (int j = 0; j < 2; ++j) ld_bf16x8(s_dy + sw128_offset(row, cv + 16 * part + 8 * j, kTile), g + 8 * j);
      float2 dyy2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < 16; i += 2) dyy2 = __ffma2_rn(make_float2(g[i], g[i + 1]), make_float2(v[i], v[i + 1]), dyy2);
      dot[part * kTile + row] = dyy2.x + dyy2.y;
    }
    __syncthreads();
    {
      float dsum = (dot[row] + dot[kTile + row]) + (dot[2 * kTile + row] + dot[3 * kTile + row]);
      const float den = (asum[row] + asum[kTile + row]) + (asum[2 * kTile + row] + asum[3 * kTile + row]);
      if (part == 0 && go) {
        go &= mbar_wait(x1_free, x_phase, p.status, abort_flag);
        st_async_f32(map_peer(sb + lay.rx + row * 4, peer), dsum, peer_x1_full);
      }
      go &= mbar_wait(x1_full, x_phase, p.status, abort_flag);
      // CTA 0 adds (own + peer), CTA 1 (peer + own): the same sum, a + b == b + a
      dsum = rank == 0 ? dsum + rx[row] : rx[row] + dsum;
      const float inv = live ? 1.0f / den : 0.f;
      // dN = dY / den over all 128 columns, in place
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float g[8];
        const uint32_t a = s_dy + sw128_offset(row, 32 * part + 8 * j, kTile);
        ld_bf16x8(a, g);
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const float2 gi = __fmul2_rn(make_float2(g[i], g[i + 1]), make_float2(inv, inv));
          g[i] = gi.x;
          g[i + 1] = gi.y;
        }
        st_bf16x8(a, g);
      }
      if (part == 0) dd[row] = live ? -(dsum * inv) * inv : 0.f;
    }
    tmem_st_wait();  // eq. (19)'s master stores, before the next tile rereads them
    fence_async_smem();
    cta_sync();

    // (g) dV[:, own] = A^T dN[:, own] + phi_k G[own]^T -> X; raw dA = dN V^T -> T
    if (issue0()) {
      const uint32_t id_v1 = make_idesc(128, DH, true, true);
      const uint32_t id_v2 = make_idesc(128, DH, false, true);
      for (int s = 0; s < kTile / 16; ++s)
        mma_bf16(tb + kX, desc_mnmajor(s_at, kTile, 0, s), desc_mnmajor(s_dy, kTile, cv, s), id_v1, s > 0);
      for (int s = 0; s < D / 16; ++s)
        mma_bf16(tb + kX, desc_kmajor(s_k, kTile, 0, s), desc_mnmajor(s_gv, D, 0, s), id_v2, 1);
      const uint32_t id_a = make_idesc(128, 128, false, false);
      for (int s = 0; s < D / 16; ++s)
        mma_bf16(tb + kT, desc_kmajor(s_dy, kTile, 0, s), desc_kmajor(s_v, kTile, 0, s), id_a, s > 0);
      mma_commit(mma_bar);
    }
    wait_mma();
    {
      const float dval = dd[row];
      float a[32];
      tmem_ld32(tmem_addr(tb, 32 * q4, kT + 32 * part), a);
#pragma unroll
      for (int i = 0; i < 32; ++i) a[i] = (32 * part + i > row) ? 0.f : a[i] + dval;
#pragma unroll
      for (int j = 0; j < 4; ++j) st_bf16x8(s_at + sw128_offset(row, 32 * part + 8 * j, kTile), a + 8 * j);
      float v[16];
      tmem_ld16(tmem_addr(tb, 32 * q4, kX + 16 * part), v);
      if (live) {
        uint4 *dst = reinterpret_cast<uint4 *>(p.dv + ((size_t)bh * p.L + (size_t)t * kTile + row) * D + cv + 16 * part);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          dst[j] = make_uint4(pack_bf16(v[8 * j], v[8 * j + 1]), pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                              pack_bf16(v[8 * j + 4], v[8 * j + 5]), pack_bf16(v[8 * j + 6], v[8 * j + 7]));
      }
    }
    fence_async_smem();
    cta_sync();

    // (h) this CTA's shares of dphi_q -> T and dphi_k -> X (one commit):
    //   CTA 0: dA phi_k + dN[:, 0:64] R[0:64]^T,  dA^T phi_q + V[:, 0:64] G[0:64]^T
    //   CTA 1:            dN[:, 64:] R[64:]^T,                V[:, 64:] G[64:]^T
    // then G[own] += phi_q^T dN[:, own] (its own commit, under the epilogue)
    if (issue0()) {
      if (rank == 0) {
        const uint32_t id1 = make_idesc(128, 128, false, true);
        for (int s = 0; s < kTile / 16; ++s)
          mma_bf16(tb + kT, desc_kmajor(s_at, kTile, 0, s), desc_mnmajor(s_k, kTile, 0, s), id1, s > 0);
      }
      const uint32_t id2 = make_idesc(128, 128, false, false);
      for (int s = 0; s < DH / 16; ++s)
        mma_bf16(tb + kT, desc_kmajor(s_dy, kTile, 0, (uint32_t)(cv / 16 + s)), desc_kmajor(s_rb, D, 0, s), id2,
                 rank == 0 || s > 0);
      if (rank == 0) {
        const uint32_t id3 = make_idesc(128, 128, true, true);
        for (int s = 0; s < kTile / 16; ++s)
          mma_bf16(tb + kX, desc_mnmajor(s_at, kTile, 0, s), desc_mnmajor(s_q, kTile, 0, s), id3, s > 0);
      }
      for (int s = 0; s < DH / 16; ++s)
        mma_bf16(tb + kX, desc_kmajor(s_v, kTile, 0, (uint32_t)(cv / 16 + s)), desc_kmajor(s_gv, D, 0, s), id2,
                 rank == 0 || s > 0);
      mma_commit(mmb_bar);
      const uint32_t id_g = make_idesc(128, DH, true, true);
      for (int s = 0; s < kTile / 16; ++s)
        mma_bf16(tb + kG, desc_mnmajor(s_q, kTile, 0, s), desc_mnmajor(s_dy, kTile, cv, s), id_g, 1);
      mma_commit(mma_bar);
    }
    // G_S's increment, sum over rows of dD phi_q (CTA 0; column sums over a
    // quarter of the rows each, added once the epilogue has used G_S)
    if (rank == 0) {
      const int f = tid & (D - 1), g = tid >> 7;
      float cs = 0.f;
      const unsigned char *qb = smem + lay.q;
#pragma unroll 8
      for (int j = 32 * g; j < 32 * g + 32; ++j)
        cs = fmaf(dd[j], __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(qb + sw128_offset(j, f, kTile))), cs);
      dot[g * kTile + f] = cs;
    }
    wait_mmb();
    if (issue0() && t > t0) load_v(t - 1);  // V is read by no later MMA of this tile
    // (i) dQ, dK shares = dphi * g'(x), g' = min(phi, 1); CTA 0 adds the dD S^T
    // and G_S terms.  dK goes over phi_k now, dQ over phi_q once the G
    // update has read phi_q
    uint32_t qpk[16];
    {
      const float dval = dd[row];
      float a[32], b[32];
      tmem_ld32x2(tmem_addr(tb, 32 * q4, kT + 32 * part), tmem_addr(tb, 32 * q4, kX + 32 * part), a, b);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int f0 = 32 * part + 8 * j;
        float fq[8], fk[8];
        ld_bf16x8(s_q + sw128_offset(row, f0, kTile), fq);
        ld_bf16x8(s_k + sw128_offset(row, f0, kTile), fk);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float dq = a[8 * j + i], dk = b[8 * j + i];
          if (rank == 0) {
            dq = fmaf(dval, s_hi[f0 + i] + s_lo[f0 + i], dq);
            dk += gs[f0 + i];
          }
          a[8 * j + i] = dq * fminf(fq[i], 1.f);
          b[8 * j + i] = dk * fminf(fk[i], 1.f);
        }
        st_bf16x8(s_k + sw128_offset(row, f0, kTile), b + 8 * j);
#pragma unroll
        for (int x = 0; x < 4; ++x) qpk[4 * j + x] = pack_bf16(a[8 * j + 2 * x], a[8 * j + 2 * x + 1]);
      }
    }
    cta_sync();  // every thread has read phi_q, phi_k and G_S
    wait_mma();  // the G update has read phi_q and dN
    if (issue0() && t > t0) load_dy(t - 1);
    if (rank == 0 && tid < D)
      gs[tid] += (dot[tid] + dot[kTile + tid]) + (dot[2 * kTile + tid] + dot[3 * kTile + tid]);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      st_shared_v4(s_q + sw128_offset(row, 32 * part + 8 * j, kTile), qpk[4 * j], qpk[4 * j + 1], qpk[4 * j + 2],
                   qpk[4 * j + 3]);
    fence_async_smem();
    cta_sync();
    if (issue0()) {
      for (int c = 0; c < D; c += 64) {
        tma_reduce_add_3d(&tmDQ, s_q + c * kTile * 2, c, t * kTile, bh);
        tma_reduce_add_3d(&tmDK, s_k + c * kTile * 2, c, t * kTile, bh);
      }
      tma_store_commit();
      if (t > t0) {
        // Q and K take the next tile once the reduce-adds have read them
        tma_store_wait_read();
        load_qk(t - 1);
      }
    }
    x_phase ^= 1;
  }

  if (tid == 0) tma_store_wait_all();
  if (tid == 0 && *abort_flag) {
    // a wait gave up: this CTA's MMAs and the loads armed before that land
    // before TMEM is freed and the CTA leaves (an armed phase completes when
    // its bytes land; one with nothing armed gives up after 20 ms)
    mma_commit(drain_bar);
    mbar_drain(drain_bar, 0);
    uint64_t *const armed[2] = {in_bar, in2_bar};
    for (int i = 0; i < 2; ++i)
      for (uint32_t par = 0; par < 2; ++par) mbar_drain(armed[i], par, 20000000ull);
  }
  // segment total of G (this CTA's columns; CTA 0 also G_S) -> gstates
  {
    const size_t base = ((size_t)bh * p.P + seg) * (size_t)D * (D + 1);
    float g[16];
    tmem_ld16(tmem_addr(tb, 32 * q4, kG + 16 * part), g);
    float *dst = p.gstates + base + (size_t)row * (D + 1) + cv + 16 * part;
#pragma unroll
    for (int i = 0; i < 16; ++i) dst[i] = g[i];
    if (rank == 0 && tid < D) p.gstates[base + (size_t)tid * (D + 1) + D] = gs[tid];
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote store may target an exited CTA
  if (warp == 0) tmem_dealloc(tb, 512);
}

// ---------------------------------------------------------------------------
// The later segments' reverse state (eq. (20)-(21)): the backward kernel runs
// every segment from G = 0 at its end, so dK and dV of segment s < P - 1 miss
// the terms of G_end(s) (the reverse scan of the later segments' totals).
// Both are linear in G; per row j of segment s:
//   dK_j += (V_j G^T + G_S) * min(phi_k,j, 1),   dV_j += phi_k,j G
// One CTA per (segment, head) walks the segment's tiles: phi_k in place over
// K, then D = V G^T and dV' = phi_k G on the tensor cores (G_end as a bf16
// [feature][column] image); the increments, in bf16 over the tile's own K
// and V slots, go into dK, dV by TMA reduce-add.  K and V are
// double-buffered.

struct CorrParams {
  int L, P, tps, nt, BH;
  const unsigned char *grec;  // per (head, segment): G_end image [128][128] bf16, then G_S fp32 [128]
  int *status;
};

constexpr uint32_t kRecBytes = kTileBytes + D * 4;

// G_end(s) = the scanned G total at index s + 1 -> image + G_S record of (bh, s)
__global__ void prep_g128_kernel(const float *__restrict__ gstates, unsigned char *__restrict__ grec, int P, int BH) {
  // x: the (feature, column) pairs of one record; y: its (head, segment)
  const int DP = D + 1;
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= D * DP) return;
  const int f = r / DP, e = r - f * DP;
  for (int hs = blockIdx.y; hs < BH * (P - 1); hs += gridDim.y) {
    const int bh = hs / (P - 1), s = hs - bh * (P - 1);
    const float g = gstates[((size_t)bh * P + s + 1) * (size_t)D * DP + r];
    unsigned char *rec = grec + ((size_t)bh * P + s) * (size_t)kRecBytes;
    if (e < D)
      *reinterpret_cast<__nv_bfloat16 *>(rec + sw128_offset(f, e, D)) = __float2bfloat16_rn(g);
    else
      reinterpret_cast<float *>(rec + kTileBytes)[f] = g;
  }
}

struct CorrLayout {
  uint32_t g, gs, kv, bars, total;
  __host__ __device__ CorrLayout() {
    uint32_t o = 0;
    g = o; o += kTileBytes;
    gs = o; o += D * 4;  // directly after g: one bulk copy of the record
    o = (o + 1023u) & ~1023u;
    kv = o; o += 2 * 2 * kTileBytes;  // [buffer][K, V]
    bars = o; o += 64;
    total = o;
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    elu_corr_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV, CorrParams p) {
  constexpr uint32_t kD = 0, kV = 128;  // TMEM: V G^T | phi_k G
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const CorrLayout lay;
  const uint32_t sb = smem_u32(smem);
  uint64_t *ld_bar = reinterpret_cast<uint64_t *>(smem + lay.bars);  // [2]
  uint64_t *setup_bar = ld_bar + 2;
  uint64_t *mma_bar = ld_bar + 3;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(ld_bar + 4);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(ld_bar + 5);
  uint64_t *drain_bar = ld_bar + 6;  // used once, after a timed-out wait
  const float *gs = reinterpret_cast<const float *>(smem + lay.gs);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, part = warp >> 2, row = 32 * q4 + lane;
  const int seg = blockIdx.x, bh = blockIdx.y;
  const int t0 = seg * p.tps, t1 = min(t0 + p.tps, p.nt);
  const uint32_t s_g = sb + lay.g;

  auto load = [&](int t, int b) {
    uint64_t *bar = ld_bar + b;
    unsigned char *kb = smem + lay.kv + (uint32_t)b * 2u * kTileBytes;
    mbar_arrive_expect_tx(bar, 2 * kTileBytes);
    for (int c = 0; c < D; c += 64) {
      tma_load_3d(kb + c * kTile * 2, &tmK, bar, c, t * kTile, bh);
      tma_load_3d(kb + kTileBytes + c * kTile * 2, &tmV, bar, c, t * kTile, bh);
    }
  };
  if (tid == 0) {
    mbar_init(ld_bar, 1);
    mbar_init(ld_bar + 1, 1);
    mbar_init(setup_bar, 1);
    mbar_init(mma_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    mbar_arrive_expect_tx(setup_bar, kRecBytes);
    bulk_load(smem + lay.g, p.grec + ((size_t)bh * p.P + seg) * (size_t)kRecBytes, kRecBytes, setup_bar);
    if (t0 < t1) load(t0, 0);
  }
  if (warp == 0) tmem_alloc(tslot, 256);
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
  const uint32_t id_d = make_idesc(128, 128, false, false);
  const uint32_t id_v = make_idesc(128, 128, false, true);
  for (int i = 0; t0 + i < t1; ++i) {
    const int t = t0 + i, b = i & 1;
    const uint32_t s_k = sb + lay.kv + (uint32_t)b * 2u * kTileBytes, s_v = s_k + kTileBytes;
    const bool live = row < min(kTile, p.L - t * kTile);
    go &= mbar_wait(ld_bar + b, (uint32_t)(i >> 1) & 1u, p.status, abort_flag);
    // phi_k in place over K (padding rows: 0)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float v[8];
      const uint32_t a = s_k + sw128_offset(row, 32 * part + 8 * j, kTile);
      ld_bf16x8(a, v);
#pragma unroll
      for (int x = 0; x < 8; ++x) v[x] = live ? elu1_feature(v[x]) : 0.f;
      st_bf16x8(a, v);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && go) {
      for (int s = 0; s < D / 16; ++s)
        mma_bf16(tb + kD, desc_kmajor(s_v, kTile, 0, s), desc_kmajor(s_g, D, 0, s), id_d, s > 0);
      for (int s = 0; s < D / 16; ++s)
        mma_bf16(tb + kV, desc_kmajor(s_k, kTile, 0, s), desc_mnmajor(s_g, D, 0, s), id_v, s > 0);
      mma_commit(mma_bar);
    }
    __syncwarp();
    go &= mbar_wait(mma_bar, mphase, p.status, abort_flag);
    mphase ^= 1;
    tc_fence_after();
    // every MMA up to this tile's is complete, and the last tile's reduce-adds
    // have read their sources: the other buffer takes tile t + 1
    if (tid == 0 && go && t + 1 < t1) {
      if (i > 0) tma_store_wait_read();
      load(t + 1, b ^ 1);
    }
    {
      float dk[32], dv[32];
      tmem_ld32x2(tmem_addr(tb, 32 * q4, kD + 32 * part), tmem_addr(tb, 32 * q4, kV + 32 * part), dk, dv);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int f0 = 32 * part + 8 * j;
        const uint32_t ak = s_k + sw128_offset(row, f0, kTile);
        float ph[8];
        ld_bf16x8(ak, ph);
#pragma unroll
        for (int x = 0; x < 8; ++x) dk[8 * j + x] = (dk[8 * j + x] + gs[f0 + x]) * fminf(ph[x], 1.f);
        // increments in place of this thread's own phi_k and V elements
        st_bf16x8(ak, dk + 8 * j);
        st_bf16x8(s_v + sw128_offset(row, f0, kTile), dv + 8 * j);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();  // TMEM and the increments are complete before the next tile's MMAs
    tc_fence_after();
    if (tid == 0 && go) {
      for (int c = 0; c < D; c += 64) {
        tma_reduce_add_3d(&tmDK, s_k + c * kTile * 2, c, t * kTile, bh);
        tma_reduce_add_3d(&tmDV, s_v + c * kTile * 2, c, t * kTile, bh);
      }
      tma_store_commit();
    }
  }
  if (tid == 0) tma_store_wait_all();
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
  __syncthreads();
  if (warp == 0) tmem_dealloc(tb, 256);
}

}  // namespace tce

bool tc_backward_elu128_supported(int d, int M, int chunk, bool favor) {
  (void)chunk;  // 128-row tiles for every slice size
  return !favor && d == tce::D && M == tce::D;
}

cudaError_t tc_backward_elu128(const Plan &pl, const Args &a, cudaStream_t st) {
  using namespace tce;
  CUtensorMap mq, mk, mv, mdy, mdq, mdk, mdv;
  if (!make_map_bf16_3d(&mq, a.q, pl.BH, pl.L, D, kTile) || !make_map_bf16_3d(&mk, a.k, pl.BH, pl.L, D, kTile) ||
      !make_map_bf16_3d(&mv, a.v, pl.BH, pl.L, D, kTile) || !make_map_bf16_3d(&mdy, a.dy, pl.BH, pl.L, D, kTile) ||
      !make_map_bf16_3d(&mdq, a.dq, pl.BH, pl.L, D, kTile) || !make_map_bf16_3d(&mdk, a.dk, pl.BH, pl.L, D, kTile) ||
      !make_map_bf16_3d(&mdv, a.dv, pl.BH, pl.L, D, kTile))
    return cudaErrorInvalidValue;
  // each CTA of a pair adds its share of dQ and dK: the state pass zeroes
  // them tile by tile while it runs
  cudaError_t e = tc_segment_states(pl, a, pl.P, 1 | 2, nullptr, st);
  if (e != cudaSuccess) return e;
  {
    Params p{};
    p.L = pl.L; p.nt = pl.tc_tiles; p.P = pl.P; p.tps = pl.cps; p.BH = pl.BH;
    p.dv = static_cast<__nv_bfloat16 *>(a.dv);
    p.states = a.ws + pl.states_off;
    p.states_lo = a.ws + pl.states_lo_off;
    p.gstates = a.ws + pl.gstates_off;
    p.status = a.status;
    const Layout lay;
    const int smem = (int)lay.total + 1024;
    e = cudaFuncSetAttribute(elu_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    ProfScope ps("tc_backward", st);
    elu_bwd_kernel<<<dim3(2 * pl.P, pl.BH), kThreads, smem, st>>>(mq, mk, mv, mdy, mdq, mdk, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (pl.P < 2) return cudaSuccess;
  {
    ProfScope ps("scan_states", st);
    // G_end(s) = sum over s' > s: reverse inclusive scan over segments 1..P-1
    e = scan_states_f32_rev(pl, a.ws + pl.gstates_off + (size_t)D * (D + 1), pl.P - 1, nullptr, st);
    if (e != cudaSuccess) return e;
  }
  {
    ProfScope ps("prep_g", st);
    const dim3 grid((D * (D + 1) + 255) / 256, (unsigned)std::min(pl.BH * (pl.P - 1), 65535));
    prep_g128_kernel<<<grid, 256, 0, st>>>(a.ws + pl.gstates_off, reinterpret_cast<unsigned char *>(a.ws + pl.gimg_off),
                                             pl.P, pl.BH);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  CorrParams cp{};
  cp.L = pl.L; cp.P = pl.P; cp.tps = pl.cps; cp.nt = pl.tc_tiles; cp.BH = pl.BH;
  cp.grec = reinterpret_cast<const unsigned char *>(a.ws + pl.gimg_off);
  cp.status = a.status;
  const CorrLayout lay;
  const int smem = (int)lay.total + 1024;
  e = cudaFuncSetAttribute(elu_corr_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  ProfScope ps("tc_backward_fix", st);
  elu_corr_kernel<<<dim3(pl.P - 1, pl.BH), kThreads, smem, st>>>(mk, mv, mdk, mdv, cp);
  return cudaGetLastError();
}

}  // namespace slim
