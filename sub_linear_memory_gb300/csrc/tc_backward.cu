// tc_backward.cu -- tensor-core (tcgen05 + TMA) SLiM backward for bf16 I/O.
//
// "Sub-Linear Memory: How to Make Performers SLiM", section 3.3.  One CTA
// walks one segment of 128-row tiles in reverse.  Per tile, with R' the
// stacked state [R ; S^T] and G the reverse state [G_V ; G_S] (rows d and
// d+1), both kept as fp32 masters in TMEM with features on the lanes:
//   R' -= phi_k^T [V, 1]                      eq. (19): state before the tile
//   A   = tril(phi_q phi_k^T),  num = A V + phi_q R^T,
//   den = rowsum(A) + phi_q . S,  Y = num / den
//   dN  = dY / den,  dD = -(dY . Y) / den     (dN' = [dN ; dD])
//   dA  = tril(dN V^T + dD 1^T)              (as diag(1/den) (dY V^T) + dD 1^T:
//                                             the MMA needs dY only, not dN)
//   dV  = A^T dN + phi_k G_V^T
//   dphi_q = dA phi_k + dN R^T + dD S^T
//   dphi_k = dA^T phi_q + V G_V^T + 1 G_S^T
//   G  += phi_q^T [dN, dD]                    eq. (20)
//   FAVOR+: u = phi * dphi, dX = u W^T - X rowsum(u);  elu+1: dX = dphi * min(phi, 1)
// G starts at zero at the end of each segment, so dK and dV here miss the
// later segments' G; the correction kernel adds G_end(s) (the reverse scan of
// the segments' G totals) afterwards: both terms are linear in G.
//
// With 256 features a segment runs on a two-CTA cluster, each CTA owning 128
// features.  dN' needs two row sums over all features, den and dY . num
// (dY . Y = dY . num / den), so the CTAs swap their partials of those two
// (distributed shared memory, two floats per row).  dV, dQ and dK are sums over
// features too, but nothing downstream needs them inside the kernel: each
// CTA rounds its partial to bf16 and adds it into the (zeroed) outputs with
// a TMA reduce-add.  The order of the two adds is not fixed, so those
// outputs may differ from run to run in the last bf16 bit.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace slim {
namespace tcb {

using namespace slim::tc;

constexpr int kThreads = 512;
constexpr int kParts = 4;  // threads per row (TMEM lane): warps w, w + 4, w + 8, w + 12
constexpr int kTile = 128;
constexpr int D = 64;
static_assert(16 * kParts == D, "the R update gives each part 16 value columns");

struct Params {
  int L, M, nt, P, tps, favor, BH;
  int H, wstride;  // heads; bf16 elements between per-head W^T images (0: one shared W)
  __nv_bfloat16 *dq, *dk, *dv;
  const float *w;
  const __nv_bfloat16 *wimg;  // W^T as the bf16 [M][64] swizzled shared-memory image
  const float *states;     // fp32 [BH][P][M][D + 1]: inclusive segment-end R', high parts
  const float *states_lo;  // low parts
  float *gstates;          // fp32 [BH][P][M][D + 1]: segment totals of G (out) / G_end (in)
  float *dwpart;           // learnable W: fp32 [BH][P][M][D] dW^T partial of each segment (added to)
  int *status;
};

struct Layout {
  uint32_t w, q, k, v, dy, phq, phk, at, gv, rb, ones, ddb;
  uint32_t asum, s_f, gs_f, dd, usq, usk, dot, rx, bars, total;
  __host__ __device__ explicit Layout(int MC) {
    uint32_t o = 0;
    const uint32_t tile = kTile * D * 2;
    w = o; o += (uint32_t)MC * 128u;
    q = o; o += tile;
    k = o; o += tile;
    v = o; o += tile;
    dy = o; o += tile;  // dY, then dN (in place)
    phq = o; o += kTile * 256;
    phk = o; o += kTile * 256;
    at = o; o += kTile * 256;  // masked A, then masked dA
    gv = o; o += tile;  // the bf16 copy of G_V; with a CTA pair, then the dQ partial
    rb = o; o += (uint32_t)MC * 128u;
    ones = o; o += 4096;
    ddb = o; o += 4096;
    asum = o; o += kParts * kTile * 4;  // [part][row]: row sums of tril(A), then den partials
    s_f = o; o += 128 * 4;
    gs_f = o; o += 128 * 4;
    dd = o; o += kTile * 4;
    usq = o; o += kParts * kTile * 4;  // [part][row] partial row sums of u_q
    usk = o; o += kParts * kTile * 4;
    // dY . Y partials: dead before u's row sums are written
    dot = usq;
    // cluster exchange, the peer's row partials of den and dY . num
    // ([2][128]): the peer writes them only after this CTA is past its
    // features (the last use of usk before (f)), and they are read before
    // u's row sums are written
    rx = usk;
    bars = o; o += 128;
    total = o;
  }
};

// TMEM columns: R' as a double-float (hi, lo) pair, G, two transients
constexpr uint32_t kRhi = 0, kRlo = 80, kG = 160, kT = 240, kX = 368;

__device__ __forceinline__ void st_bf16_scalar(unsigned char *smem, uint32_t off, float v) {
  *reinterpret_cast<__nv_bfloat16 *>(smem + off) = __float2bfloat16_rn(v);
}

// Copy columns [0, 64) of a TMEM state (features on lanes) into a bf16
// [MC][64] tile and column 64 into an fp32 vector.  Threads: feature
// f = 32 * (warp % 4) + lane, columns [16 part, +16); part 3 also column 64.
__device__ __forceinline__ void state_to_smem(uint32_t tbase, uint32_t col, int q4, int part, int f, int MC,
                                              uint32_t s_tile, float *vec) {
  float v[16];
  tmem_ld16(tmem_addr(tbase, 32 * q4, col + 16 * part), v);
  if (f < MC) {
#pragma unroll
    for (int j = 0; j < 2; ++j) st_bf16x8(s_tile + sw128_offset(f, 16 * part + 8 * j, MC), v + 8 * j);
  }
  if (part == kParts - 1) {
    const float s0 = tmem_ld1(tmem_addr(tbase, 32 * q4, col + 64));
    if (f < MC) vec[f] = s0;
  }
}

// CS = 1: one CTA per segment holds all M <= 128 features.
// CS = 2: a cluster of two CTAs per segment; CTA c owns features
// [128c, 128c + 128) with their R' and G, computes every per-feature term
// locally, and the two swap through distributed shared memory the row sums
// den and dY . num, so both form the same dN' for all 128 rows.  dV, dQ and
// dK partials go to global memory by TMA reduce-add.
// DW (learnable W, FAVOR+): each tile also forms dW^T = u_q^T Q + u_k^T K for
// this CTA's features on the tensor cores (u in the phi tiles, the result in
// the TMEM columns u leaves free) and adds it to the segment's dW partial.
template <bool FAVOR, int CS, int MC, bool DW>
__global__ void __launch_bounds__(kThreads, 1)
    tc_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDY,
                  const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
                  const __grid_constant__ CUtensorMap tmDV, Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // MC: features per CTA (<= 128)
  constexpr int QF = MC / kParts;  // feature columns per thread
  constexpr int QD = D / kParts;   // value columns per thread
  // 128 features per CTA: the two sides' features, dphi and dQ, dK MMAs
  // complete on barriers of their own, so one side's CUDA-core work runs
  // under the other side's MMAs; with 64 the MMAs and exponentials are short
  // and the extra hand-offs cost more than they hide (one commit for both)
  constexpr bool kSplit = MC == 128;
  const Layout lay(MC);
  const uint32_t sb = smem_u32(smem);
  uint64_t *in_bar = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint64_t *mma_bar = in_bar + 1;
  uint64_t *rl_bar = in_bar + 2;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(in_bar + 3);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(in_bar + 4);
  uint64_t *setup_bar = in_bar + 5;
  // cluster exchange of the den and dY . num partials: data received
  // (st.async bytes) and receive slots released by the peer (remote arrive),
  // one phase per tile
  uint64_t *x1_full = in_bar + 6, *x1_free = in_bar + 8;
  // inputs: Q, K on in_bar (needed first, by the features); V, dY on in2_bar
  // (needed from the state increment on), so a tile starts before they land
  uint64_t *in2_bar = in_bar + 10;
  // a second MMA-completion barrier, for a group whose epilogue overlaps the
  // group issued after it
  uint64_t *mmb_bar = in_bar + 11;
  // used once, after a timed-out wait: completes when every MMA issued so far has
  uint64_t *drain_bar = in_bar + 12;
  // dphi_q complete (dphi_k's completion is on mmb_bar); the dK MMAs complete
  uint64_t *mmc_bar = in_bar + 13, *mmd_bar = in_bar + 14;
  float *rx = reinterpret_cast<float *>(smem + lay.rx);
  float *s_f = reinterpret_cast<float *>(smem + lay.s_f);
  float *gs_f = reinterpret_cast<float *>(smem + lay.gs_f);
  float *dd = reinterpret_cast<float *>(smem + lay.dd);
  float *usq = reinterpret_cast<float *>(smem + lay.usq);
  float *usk = reinterpret_cast<float *>(smem + lay.usk);
  float *dot = reinterpret_cast<float *>(smem + lay.dot);
  float *asum = reinterpret_cast<float *>(smem + lay.asum);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, part = warp >> 2, row = 32 * q4 + lane;
  const int rank = CS == 2 ? (int)cluster_rank() : 0, peer = 1 - rank;
  const int seg = blockIdx.x / CS, bh = blockIdx.y;
  // debug builds: a segment outside the plan records SLIM_ERR_BOUNDS and the CTA does nothing
  if (!SLIM_DCHECK(p.status, seg < p.P && bh < p.BH && seg * p.tps < p.nt)) return;
  const int M = p.M, DP = D + 1;
  const int fbase = rank * MC;  // first feature of this CTA
  const int t0 = seg * p.tps, t1 = min(t0 + p.tps, p.nt);

  // this CTA's rows of the W^T image (its features are contiguous rows of
  // it, with the same swizzle phase) and its features' segment-end state
  // (high and low parts, staged in the phi / A tiles) by bulk copy
  const uint32_t st_bytes = (uint32_t)(MC * DP * 4);
  const uint32_t lo_stage = lay.phq + ((st_bytes + 1023u) & ~1023u);
  if (tid == 0) {
    mbar_init(in_bar, 1);
    mbar_init(in2_bar, 1);
    mbar_init(mmb_bar, 1);
    mbar_init(mma_bar, 1);
    mbar_init(rl_bar, 1);
    mbar_init(setup_bar, 1);
    mbar_init(x1_full, 1);
    mbar_init(x1_free, 1);
    mbar_init(drain_bar, 1);
    mbar_init(mmc_bar, 1);
    mbar_init(mmd_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    const size_t soff = ((size_t)bh * p.P + seg) * (size_t)M * DP + (size_t)fbase * DP;
    mbar_arrive_expect_tx(setup_bar, (FAVOR ? (uint32_t)MC * 128u : 0u) + 2 * st_bytes);
    if (FAVOR)
      bulk_load(smem + lay.w,
                reinterpret_cast<const unsigned char *>(p.wimg + (size_t)(bh % p.H) * p.wstride) + (size_t)fbase * 128,
                MC * 128u,
                setup_bar);
    bulk_load(smem + lay.phq, p.states + soff, st_bytes, setup_bar);
    bulk_load(smem + lo_stage, p.states_lo + soff, st_bytes, setup_bar);
  }
  if (warp == 0) tmem_alloc(tslot, 512);

  for (int idx = tid; idx < kTile * 16; idx += kThreads) {
    const int r = idx >> 4, x = idx & 15;
    st_bf16_scalar(smem, lay.ones + n16_offset(r, x), x == 0 ? 1.f : 0.f);
    st_bf16_scalar(smem, lay.ddb + n16_offset(r, x), 0.f);
  }
  tc_fence_before();
  __syncthreads();
  if (CS == 2) cluster_sync();  // the peer is running before any remote store
  tc_fence_after();
  const uint32_t tb = *tslot;
  // false once a wait of this thread has given up (or seen another give
  // up): thread 0 then issues nothing more.  A wait that returns true saw
  // its phase complete, so while thread 0's waits succeed the barriers it
  // arms are in step, whatever another thread's wait did.
  bool go = true;

  // R' <- inclusive state at the segment end (hi, lo); G <- 0
  {
    go &= mbar_wait(setup_bar, 0, p.status, abort_flag);
    const float *sh = reinterpret_cast<const float *>(smem + lay.phq);
    const float *sl = reinterpret_cast<const float *>(smem + lo_stage);
    const int f = row;
    for (int c = 16 * part; c < 80; c += 16 * kParts) {
      float h[16], l[16], z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int e = c + i;
        const bool in = f < MC && e <= D;
        h[i] = in ? sh[f * DP + e] : 0.f;
        l[i] = in ? sl[f * DP + e] : 0.f;
        z[i] = 0.f;
      }
      tmem_st16(tmem_addr(tb, 32 * q4, kRhi + c), h);
      tmem_st16(tmem_addr(tb, 32 * q4, kRlo + c), l);
      tmem_st16(tmem_addr(tb, 32 * q4, kG + c), z);
    }
    tmem_st_wait();
  }
  __syncthreads();  // the staging area is read before the zero padding goes in
  if (MC < 128) {  // features beyond MC stay zero in phi_q / phi_k
    for (int idx = tid; idx < kTile * 128; idx += kThreads) {
      const int r = idx >> 7, x = idx & 127;
      if (x >= MC) {
        st_bf16_scalar(smem, lay.phq + sw128_offset(r, x, kTile), 0.f);
        st_bf16_scalar(smem, lay.phk + sw128_offset(r, x, kTile), 0.f);
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t s_w = sb + lay.w, s_q = sb + lay.q, s_k = sb + lay.k, s_v = sb + lay.v;
  const uint32_t s_dy = sb + lay.dy, s_phq = sb + lay.phq, s_phk = sb + lay.phk;
  const uint32_t s_at = sb + lay.at, s_gv = sb + lay.gv, s_rb = sb + lay.rb;
  const uint32_t s_ones = sb + lay.ones, s_ddb = sb + lay.ddb;
  const uint32_t tile_bytes = kTile * D * 2;
  uint32_t in_phase = 0, in2_phase = 0, mma_phase = 0, mmb_phase = 0, mmc_phase = 0, mmd_phase = 0, rl_phase = 0,
           x_phase = 0;
  // the exchange: two fp32 row sums for each of the 128 rows
  constexpr uint32_t kX1Bytes = 2 * kTile * 4;
  const uint32_t peer_x1_full = CS == 2 ? map_peer(smem_u32(x1_full), peer) : 0u;
  const uint32_t peer_x1_free = CS == 2 ? map_peer(smem_u32(x1_free), peer) : 0u;

  auto issue_in = [&](int t) {
    mbar_arrive_expect_tx(in_bar, 2 * tile_bytes);
    tma_load_3d(smem + lay.q, &tmQ, in_bar, 0, t * kTile, bh);
    tma_load_3d(smem + lay.k, &tmK, in_bar, 0, t * kTile, bh);
    mbar_arrive_expect_tx(in2_bar, 2 * tile_bytes);
    tma_load_3d(smem + lay.v, &tmV, in2_bar, 0, t * kTile, bh);
    tma_load_3d(smem + lay.dy, &tmDY, in2_bar, 0, t * kTile, bh);
  };
  auto mma_done = [&]() {
    mma_commit(mma_bar);
  };
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
  auto wait_mmc = [&]() {
    __syncwarp();
    go &= mbar_wait(mmc_bar, mmc_phase, p.status, abort_flag);
    mmc_phase ^= 1;
    tc_fence_after();
  };
  auto wait_mmd = [&]() {
    __syncwarp();
    go &= mbar_wait(mmd_bar, mmd_phase, p.status, abort_flag);
    mmd_phase ^= 1;
    tc_fence_after();
  };
  auto cta_sync = [&]() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };
  // thread 0 issues every MMA, copy and barrier arm; once a wait of this CTA
  // has given up it issues nothing more (the other waits return at once),
  // so the drain after the loop covers everything in flight
  auto issue0 = [&]() { return tid == 0 && go; };

  if (tid == 0 && t0 < t1) issue_in(t1 - 1);

  for (int t = t1 - 1; t >= t0; --t) {
    const int valid = min(kTile, p.L - t * kTile);
    const bool live = row < valid;
    go &= mbar_wait(in_bar, in_phase, p.status, abort_flag);
    in_phase ^= 1;
    if (CS == 2 && issue0()) mbar_arrive_expect_tx(x1_full, kX1Bytes);
    if (issue0() && t > t0) {
      // the next tile's inputs head for L2 now; its TMA loads issue at the
      // end of this tile, when their buffers are free again
      tma_prefetch_3d(&tmQ, 0, (t - 1) * kTile, bh);
      tma_prefetch_3d(&tmK, 0, (t - 1) * kTile, bh);
      tma_prefetch_3d(&tmV, 0, (t - 1) * kTile, bh);
      tma_prefetch_3d(&tmDY, 0, (t - 1) * kTile, bh);
    }

    if constexpr (kSplit) {
      // (b) features: F_k -> T (its own commit), F_q -> X.  phi_k first, so
      // the state-increment MMA runs while phi_q is formed
      float ck = 0.f, cq = 0.f;
      if (FAVOR) {
        if (issue0()) {
          const uint32_t id = make_idesc(128, MC, false, false);
          for (int s = 0; s < D / 16; ++s)
            mma_bf16(tb + kT, desc_kmajor(s_k, kTile, 0, s), desc_kmajor(s_w, MC, 0, s), id, s > 0);
          mma_commit(mmb_bar);
          for (int s = 0; s < D / 16; ++s)
            mma_bf16(tb + kX, desc_kmajor(s_q, kTile, 0, s), desc_kmajor(s_w, MC, 0, s), id, s > 0);
          mma_done();
        }
        // |k|^2, |q|^2 of the row while the MMAs run, each part summing a
        // quarter of the columns (the u row-sum arrays are idle until (i))
        usq[part * kTile + row] = tile_row_sqnorm_part(s_k, row, QD * part, QD);
        usk[part * kTile + row] = tile_row_sqnorm_part(s_q, row, QD * part, QD);
        __syncthreads();
        const float nk = (usq[row] + usq[kTile + row]) + (usq[2 * kTile + row] + usq[3 * kTile + row]);
        const float nq = (usk[row] + usk[kTile + row]) + (usk[2 * kTile + row] + usk[3 * kTile + row]);
        ck = live ? favor_row_const(nk, M) : -INFINITY;
        cq = live ? favor_row_const(nq, M) : -INFINITY;
      }
      // one side's features: FAVOR+ from the TMEM pre-activations (padding
      // rows: F = 0 from the zero-filled tile and 2^-inf = 0), elu+1 from the
      // input tile
      auto features = [&](uint32_t col, float c, uint32_t s_x, uint32_t s_out) {
        const int c0 = QF * part;
        if (FAVOR) {
          float f[QF];
          if constexpr (QF == 32) {
            tmem_ld32(tmem_addr(tb, 32 * q4, col + c0), f);
          } else {
            tmem_ld16(tmem_addr(tb, 32 * q4, col + c0), f);
          }
#pragma unroll
          for (int i = 0; i < QF; i += 2) favor_feature2(f[i], f[i + 1], c);
#pragma unroll
          for (int j = 0; j < QF / 8; ++j) st_bf16x8(s_out + sw128_offset(row, c0 + 8 * j, kTile), f + 8 * j);
        } else {
          for (int cc = c0; cc < c0 + QF; cc += 8) {
            float v[8];
            ld_bf16x8(s_x + sw128_offset(row, cc, kTile), v);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = live ? elu1_feature(v[i]) : 0.f;
            st_bf16x8(s_out + sw128_offset(row, cc, kTile), v);
          }
        }
      };
      if (FAVOR) wait_mmb();
      features(kT, ck, s_k, s_phk);
      fence_async_smem();
      cta_sync();

      // (c) eq. (19): R' -= phi_k^T [V, 1], removing exactly the increment the
      // segment pre-pass added for this tile (increment -> T, its own commit),
      // while phi_q is formed
      go &= mbar_wait(in2_bar, in2_phase, p.status, abort_flag);  // V (and dY, read in (f))
      in2_phase ^= 1;
      if (issue0()) {
        // last tile's dQ, dK partials (staged in the G_V-copy and R-copy tiles) have
        // been read by their reduce-adds before this phase's epilogue reuses them
        if (CS == 2) tma_store_wait_read();
        issue_state_delta(tb + kT, s_phk, s_v, s_ones, D);
        mma_commit(mmb_bar);
      }
      if (FAVOR) wait_mma();
      features(kX, cq, s_q, s_phq);
      fence_async_smem();
      cta_sync();
      // my receive slots (in usk) are idle until (i): the peer may send its
      // row partials there (signalled off the MMA-issuing thread: the
      // cluster-scope release waits for this thread's earlier stores)
      if (CS == 2 && tid == 32 && go) mbar_arrive_remote(peer_x1_free);

      // A = phi_q phi_k^T -> X (its own commit: eq. (19) below runs under it)
      if (issue0()) {
        const uint32_t id = make_idesc(128, 128, false, false);
        for (int s = 0; s < MC / 16; ++s)
          mma_bf16(tb + kX, desc_kmajor(s_phq, kTile, 0, s), desc_kmajor(s_phk, kTile, 0, s), id, s > 0);
        mma_done();
      }
      wait_mmb();
      // eq. (19) on the double-float master, and from the updated values the
      // bf16 copy of R for the MMAs and fp32 S for the epilogues (R: 16
      // columns per part; S, column D, on part 3)
      {
        const int c = 16 * part;
        float x[16], h[16], l[16];
        tmem_ld16x3(tmem_addr(tb, 32 * q4, kT + c), tmem_addr(tb, 32 * q4, kRhi + c),
                    tmem_addr(tb, 32 * q4, kRlo + c), x, h, l);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          float2 h2 = make_float2(h[i], h[i + 1]), l2 = make_float2(l[i], l[i + 1]);
          df_sub2(h2, l2, make_float2(x[i], x[i + 1]));
          h[i] = h2.x;
          h[i + 1] = h2.y;
          l[i] = l2.x;
          l[i + 1] = l2.y;
        }
        tmem_st16(tmem_addr(tb, 32 * q4, kRhi + c), h);
        tmem_st16(tmem_addr(tb, 32 * q4, kRlo + c), l);
        if (row < MC) {
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = h[i] + l[i];
#pragma unroll
          for (int i = 0; i < 16; i += 8) st_bf16x8(s_rb + sw128_offset(row, c + i, MC), x + i);
        }
        if (part == kParts - 1) {
          float xs, hs, ls;
          tmem_ld1x3(tmem_addr(tb, 32 * q4, kT + D), tmem_addr(tb, 32 * q4, kRhi + D),
                     tmem_addr(tb, 32 * q4, kRlo + D), xs, hs, ls);
          df_add(hs, ls, -xs);
          tmem_st1(tmem_addr(tb, 32 * q4, kRhi + D), hs);
          tmem_st1(tmem_addr(tb, 32 * q4, kRlo + D), ls);
          if (row < MC) s_f[row] = hs + ls;
        }
      }
      wait_mma();
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
      // no MMA reads the masters and only this thread rereads its columns (the
      // next tile), so their stores are waited for later, off this barrier
      fence_async_smem();
      cta_sync();
    } else {
      // (b) features of both sides: F_k -> T, F_q -> X, one commit
      if (FAVOR) {
        if (issue0()) {
          const uint32_t id = make_idesc(128, MC, false, false);
          for (int s = 0; s < D / 16; ++s)
            mma_bf16(tb + kT, desc_kmajor(s_k, kTile, 0, s), desc_kmajor(s_w, MC, 0, s), id, s > 0);
          for (int s = 0; s < D / 16; ++s)
            mma_bf16(tb + kX, desc_kmajor(s_q, kTile, 0, s), desc_kmajor(s_w, MC, 0, s), id, s > 0);
          mma_done();
        }
        // |k|^2, |q|^2 of the row while the MMAs run, each part summing a
        // quarter of the columns (the u row-sum arrays are idle until (i))
        usq[part * kTile + row] = tile_row_sqnorm_part(s_k, row, QD * part, QD);
        usk[part * kTile + row] = tile_row_sqnorm_part(s_q, row, QD * part, QD);
        __syncthreads();
        const float nk = (usq[row] + usq[kTile + row]) + (usq[2 * kTile + row] + usq[3 * kTile + row]);
        const float nq = (usk[row] + usk[kTile + row]) + (usk[2 * kTile + row] + usk[3 * kTile + row]);
        const float ck = live ? favor_row_const(nk, M) : -INFINITY;
        const float cq = live ? favor_row_const(nq, M) : -INFINITY;
        wait_mma();
        {
          // both sides' F with one wait, so the two loads' latencies overlap
          const int c0 = QF * part;
          float fk[QF], fq[QF];
          if constexpr (QF == 32) {
            tmem_ld32x2(tmem_addr(tb, 32 * q4, kT + c0), tmem_addr(tb, 32 * q4, kX + c0), fk, fq);
          } else {
            tmem_ld16x2(tmem_addr(tb, 32 * q4, kT + c0), tmem_addr(tb, 32 * q4, kX + c0), fk, fq);
          }
          // padding rows: F = 0 (zero-filled tile) and 2^-inf = 0
#pragma unroll
          for (int i = 0; i < QF; i += 2) {
            favor_feature2(fk[i], fk[i + 1], ck);
            favor_feature2(fq[i], fq[i + 1], cq);
          }
#pragma unroll
          for (int j = 0; j < QF / 8; ++j) {
            st_bf16x8(s_phk + sw128_offset(row, c0 + 8 * j, kTile), fk + 8 * j);
            st_bf16x8(s_phq + sw128_offset(row, c0 + 8 * j, kTile), fq + 8 * j);
          }
        }
      } else {
        for (int side = 0; side < 2; ++side) {
          const uint32_t s_x = side ? s_q : s_k, s_out = side ? s_phq : s_phk;
          for (int c0 = QF * part; c0 < QF * (part + 1); c0 += 8) {
            float v[8];
            ld_bf16x8(s_x + sw128_offset(row, c0, kTile), v);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = live ? elu1_feature(v[i]) : 0.f;
            st_bf16x8(s_out + sw128_offset(row, c0, kTile), v);
          }
        }
      }
      fence_async_smem();
      cta_sync();
      // my receive slots (in usk) are idle until (i): the peer may send its
      // row partials there (signalled off the MMA-issuing thread: the
      // cluster-scope release waits for this thread's earlier stores)
      if (CS == 2 && tid == 32 && go) mbar_arrive_remote(peer_x1_free);

      // (c) A = phi_q phi_k^T -> X (its own commit: the mask below overlaps
      // the next group), and eq. (19): R' -= phi_k^T [V, 1], removing exactly
      // the increment the segment pre-pass added for this tile (increment -> T)
      if (issue0()) {
        // last tile's dQ, dK partials (staged in the G_V-copy and R-copy tiles) have
        // been read by their reduce-adds before this phase's epilogue reuses them
        if (CS == 2) tma_store_wait_read();
        const uint32_t id = make_idesc(128, 128, false, false);
        for (int s = 0; s < MC / 16; ++s)
          mma_bf16(tb + kX, desc_kmajor(s_phq, kTile, 0, s), desc_kmajor(s_phk, kTile, 0, s), id, s > 0);
        mma_commit(mmb_bar);
      }
      go &= mbar_wait(in2_bar, in2_phase, p.status, abort_flag);  // V (and dY, read in (f))
      in2_phase ^= 1;
      if (issue0()) {
        issue_state_delta(tb + kT, s_phk, s_v, s_ones, D);
        mma_done();
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
      // eq. (19) on the double-float master, and from the updated values the
      // bf16 copy of R for the MMAs and fp32 S for the epilogues (R: 16
      // columns per part; S, column D, on part 3)
      {
        const int c = 16 * part;
        float x[16], h[16], l[16];
        tmem_ld16x3(tmem_addr(tb, 32 * q4, kT + c), tmem_addr(tb, 32 * q4, kRhi + c),
                    tmem_addr(tb, 32 * q4, kRlo + c), x, h, l);
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          float2 h2 = make_float2(h[i], h[i + 1]), l2 = make_float2(l[i], l[i + 1]);
          df_sub2(h2, l2, make_float2(x[i], x[i + 1]));
          h[i] = h2.x;
          h[i + 1] = h2.y;
          l[i] = l2.x;
          l[i + 1] = l2.y;
        }
        tmem_st16(tmem_addr(tb, 32 * q4, kRhi + c), h);
        tmem_st16(tmem_addr(tb, 32 * q4, kRlo + c), l);
        if (row < MC) {
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = h[i] + l[i];
#pragma unroll
          for (int i = 0; i < 16; i += 8) st_bf16x8(s_rb + sw128_offset(row, c + i, MC), x + i);
        }
        if (part == kParts - 1) {
          float xs, hs, ls;
          tmem_ld1x3(tmem_addr(tb, 32 * q4, kT + D), tmem_addr(tb, 32 * q4, kRhi + D),
                     tmem_addr(tb, 32 * q4, kRlo + D), xs, hs, ls);
          df_add(hs, ls, -xs);
          tmem_st1(tmem_addr(tb, 32 * q4, kRhi + D), hs);
          tmem_st1(tmem_addr(tb, 32 * q4, kRlo + D), ls);
          if (row < MC) s_f[row] = hs + ls;
        }
      }
      // no MMA reads the masters and only this thread rereads its columns (the
      // next tile), so their stores are waited for later, off this barrier
      fence_async_smem();
      cta_sync();
    }

    // (f) num = A V + phi_q R^T -> T; Y, dN, dD.  den = rowsum(tril A) +
    // phi_q . S comes from the CUDA cores while the MMAs run
    if (issue0()) {
      const uint32_t id = make_idesc(128, D, false, true);
      for (int s = 0; s < kTile / 16; ++s)
        mma_bf16(tb + kT, desc_kmajor(s_at, kTile, 0, s), desc_mnmajor(s_v, kTile, 0, s), id, s > 0);
      for (int s = 0; s < MC / 16; ++s)
        mma_bf16(tb + kT, desc_kmajor(s_phq, kTile, 0, s), desc_mnmajor(s_rb, MC, 0, s), id, 1);
      mma_done();
      // dY V^T -> X (A is dead there since its mask, its loads complete
      // before the barrier above): dA before its row scaling by 1 / den,
      // which (g) applies, so dA needs no MMA after dN
      const uint32_t id_a = make_idesc(128, 128, false, false);
      for (int s = 0; s < D / 16; ++s)
        mma_bf16(tb + kX, desc_kmajor(s_dy, kTile, 0, s), desc_kmajor(s_v, kTile, 0, s), id_a, s > 0);
      mma_commit(mmb_bar);
    }
    {
      // this thread's features of phi_q . S (S after eq. (19), fp32), added
      // to its part of rowsum(tril A) in its own slot
      const int c0 = QF * part;
      // acc[i & 3] sums as two packed pairs: (0, 1), (2, 3)
      float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int j = 0; j < QF / 8; ++j) {
        float fq[8], sv[8];
        ld_bf16x8(s_phq + sw128_offset(row, c0 + 8 * j, kTile), fq);
        *reinterpret_cast<float4 *>(sv) = *reinterpret_cast<const float4 *>(s_f + c0 + 8 * j);
        *reinterpret_cast<float4 *>(sv + 4) = *reinterpret_cast<const float4 *>(s_f + c0 + 8 * j + 4);
#pragma unroll
        for (int i = 0; i < 8; i += 2)
          acc[(i >> 1) & 1] = __ffma2_rn(make_float2(fq[i], fq[i + 1]), make_float2(sv[i], sv[i + 1]), acc[(i >> 1) & 1]);
      }
      asum[part * kTile + row] += (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
    }
    // also while the MMAs run: the bf16 copy of G_V (G as the last tile
    // left it) into its tile, whose last reader (the previous dQ reduce-add
    // with a CTA pair) was waited for in (c); G_S as fp32
    state_to_smem(tb, kG, q4, part, row, MC, s_gv, gs_f);
    wait_mma();
    float inv;  // 1 / den of this thread's row (0 on padding rows)
    {
      // dN = dY / den and dD = -(dY . Y) / den with Y = num / den: only the
      // row sums den and dY . num are needed, both linear in the features,
      // so with a CTA pair each CTA forms its partials and the two swap two
      // floats per row
      float v[QD], g[QD];
      tmem_ld16(tmem_addr(tb, 32 * q4, kT + QD * part), v);
#pragma unroll
      for (int j = 0; j < QD / 8; ++j) ld_bf16x8(s_dy + sw128_offset(row, QD * part + 8 * j, kTile), g + 8 * j);
      float2 dyy2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < QD; i += 2) dyy2 = __ffma2_rn(make_float2(g[i], g[i + 1]), make_float2(v[i], v[i + 1]), dyy2);
      dot[part * kTile + row] = dyy2.x + dyy2.y;
      __syncthreads();
      float dsum = (dot[row] + dot[kTile + row]) + (dot[2 * kTile + row] + dot[3 * kTile + row]);
      float den = (asum[row] + asum[kTile + row]) + (asum[2 * kTile + row] + asum[3 * kTile + row]);
      if (CS == 2) {
        // the peer's receive slots (in its u row-sum array) are free once it
        // is past its features
        if (part == 0 && go) {
          go &= mbar_wait(x1_free, x_phase, p.status, abort_flag);
          st_async_f32(map_peer(sb + lay.rx + row * 4, peer), den, peer_x1_full);
          st_async_f32(map_peer(sb + lay.rx + (kTile + row) * 4, peer), dsum, peer_x1_full);
        }
        go &= mbar_wait(x1_full, x_phase, p.status, abort_flag);
        // a + b == b + a: both CTAs hold the same totals
        den += rx[row];
        dsum += rx[kTile + row];
      }
      inv = live ? 1.0f / den : 0.f;
#pragma unroll
      for (int i = 0; i < QD; i += 2) {
        const float2 gi = __fmul2_rn(make_float2(g[i], g[i + 1]), make_float2(inv, inv));
        g[i] = gi.x;
        g[i + 1] = gi.y;
      }
      wait_mmb();  // dY V^T has read dY
#pragma unroll
      for (int j = 0; j < QD / 8; ++j) st_bf16x8(s_dy + sw128_offset(row, QD * part + 8 * j, kTile), g + 8 * j);
      if (part == 0) {
        const float dval = live ? -(dsum * inv) * inv : 0.f;
        dd[row] = dval;
        st_bf16_scalar(smem, lay.ddb + n16_offset(row, 0), dval);
      }
    }
    tmem_st_wait();  // eq. (19)'s master stores, before the next tile rereads them
    fence_async_smem();
    cta_sync();

    // (g) dV = A^T dN + phi_k G_V^T -> T (num has been read there); while
    // its MMAs run, dA = tril(dN V^T + dD 1^T) = tril(diag(1/den) dY V^T +
    // dD 1^T) from the product in X, stored once the MMAs have read the
    // masked A out of its tile
    if (issue0()) {
      const uint32_t id_v1 = make_idesc(128, D, true, true);
      const uint32_t id_v2 = make_idesc(128, D, false, true);
      for (int s = 0; s < kTile / 16; ++s)
        mma_bf16(tb + kT, desc_mnmajor(s_at, kTile, 0, s), desc_mnmajor(s_dy, kTile, 0, s), id_v1, s > 0);
      for (int s = 0; s < MC / 16; ++s)
        mma_bf16(tb + kT, desc_kmajor(s_phk, kTile, 0, s), desc_mnmajor(s_gv, MC, 0, s), id_v2, 1);
      mma_done();
    }
    {
      const float dval = dd[row];
      uint32_t pa[16];
      {
        float a[32];
        tmem_ld32(tmem_addr(tb, 32 * q4, kX + 32 * part), a);
        const float2 inv2 = make_float2(inv, inv), dv2 = make_float2(dval, dval);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 ai = __ffma2_rn(inv2, make_float2(a[i], a[i + 1]), dv2);
          pa[i >> 1] = pack_bf16((32 * part + i > row) ? 0.f : ai.x, (32 * part + i + 1 > row) ? 0.f : ai.y);
        }
      }
      wait_mma();
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st_shared_v4(s_at + sw128_offset(row, 32 * part + 8 * j, kTile), pa[4 * j], pa[4 * j + 1], pa[4 * j + 2],
                     pa[4 * j + 3]);
      float v[QD];
      tmem_ld16(tmem_addr(tb, 32 * q4, kT + QD * part), v);
      if (CS == 2) {
        // this CTA's dV partial -> bf16 in the idle Q tile, for a reduce-add
#pragma unroll
        for (int j = 0; j < QD / 8; ++j) st_bf16x8(s_q + sw128_offset(row, QD * part + 8 * j, kTile), v + 8 * j);
      } else if (live) {
        uint4 *dst = reinterpret_cast<uint4 *>(p.dv + ((size_t)bh * p.L + (size_t)t * kTile + row) * D + QD * part);
#pragma unroll
        for (int j = 0; j < QD / 8; ++j)
          dst[j] = make_uint4(pack_bf16(v[8 * j], v[8 * j + 1]), pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                              pack_bf16(v[8 * j + 4], v[8 * j + 5]), pack_bf16(v[8 * j + 6], v[8 * j + 7]));
      }
    }
    fence_async_smem();
    cta_sync();
    if (CS == 2 && issue0()) {
      tma_reduce_add_3d(&tmDV, s_q, 0, t * kTile, bh);
      tma_store_commit();
    }

    // (h) dphi_k -> X (kSplit: its own commit, u_k starts on it while
    // dphi_q's MMAs run), dphi_q -> T, then the G update (its own commit:
    // it runs under u, which leaves phi_q, dN and dD, the update's operands,
    // in place)
    if (issue0()) {
      const uint32_t id_q2 = make_idesc(128, MC, false, false);
      const uint32_t id_k1 = make_idesc(128, MC, true, true);
      for (int s = 0; s < kTile / 16; ++s)
        mma_bf16(tb + kX, desc_mnmajor(s_at, kTile, 0, s), desc_mnmajor(s_phq, kTile, 0, s), id_k1, s > 0);
      for (int s = 0; s < D / 16; ++s)
        mma_bf16(tb + kX, desc_kmajor(s_v, kTile, 0, s), desc_kmajor(s_gv, MC, 0, s), id_q2, 1);
      if (kSplit) mma_commit(mmb_bar);
      const uint32_t id_q1 = make_idesc(128, MC, false, true);
      for (int s = 0; s < kTile / 16; ++s)
        mma_bf16(tb + kT, desc_kmajor(s_at, kTile, 0, s), desc_mnmajor(s_phk, kTile, 0, s), id_q1, s > 0);
      for (int s = 0; s < D / 16; ++s)
        mma_bf16(tb + kT, desc_kmajor(s_dy, kTile, 0, s), desc_kmajor(s_rb, MC, 0, s), id_q2, 1);
      mma_commit(kSplit ? mmc_bar : mmb_bar);
      const uint32_t id_g = make_idesc(128, D, true, true);
      const uint32_t id_g1 = make_idesc(128, 16, true, true);
      for (int s = 0; s < kTile / 16; ++s) {
        mma_bf16(tb + kG, desc_mnmajor(s_phq, kTile, 0, s), desc_mnmajor(s_dy, kTile, 0, s), id_g, 1);
        mma_bf16(tb + kG + D, desc_mnmajor(s_phq, kTile, 0, s), desc_n16(s_ddb, s), id_g1, 1);
      }
      mma_done();
      if (CS == 2 && t > t0) {
        // the K tile is idle since the features: the next tile's K streams
        // in while this one finishes (Q follows once the reduce-add has read
        // the dV partial out of the Q tile)
        mbar_arrive_expect_tx(in_bar, 2 * tile_bytes);
        tma_load_3d(smem + lay.k, &tmK, in_bar, 0, (t - 1) * kTile, bh);
      }
    }
    wait_mmb();
    // the next tile's inputs stream in as their tiles fall idle: V from
    // here, dY once the G update has read dN; Q and K at (h) with a CTA
    // pair, at the end of the tile alone
    if (issue0() && t > t0) {
      if (CS == 2) {
        tma_store_wait_read();
        tma_load_3d(smem + lay.q, &tmQ, in_bar, 0, (t - 1) * kTile, bh);
      }
      mbar_arrive_expect_tx(in2_bar, 2 * tile_bytes);
      tma_load_3d(smem + lay.v, &tmV, in2_bar, 0, (t - 1) * kTile, bh);
    }

    // (i) u = phi * dphi and its row sums, one side at a time: u_k (with
    // kSplit while dphi_q's MMAs run), then u_q.  FAVOR+: u as bf16 pairs
    // into TMEM over dphi (the A operand of (j)), with kSplit the dK MMAs
    // issued between the two sides; elu+1 writes dQ, dK here.  With DW, u_k also goes over phi_k
    // once dphi_q has read it, and u_q over phi_q once the G update has
    // read phi_q.  The dphi terms that are not MMAs are added here:
    // dphi_q += dD S, dphi_k += G_S (coef * vec, coef = dD or 1).
    auto u_side = [&](uint32_t col, uint32_t s_phi, const float *vec, float coef, float *usum,
                      uint32_t (&pairs)[QF / 2], __nv_bfloat16 *gout) {
      const int c0 = QF * part;
      float a[QF];
      if constexpr (QF == 32) {
        tmem_ld32(tmem_addr(tb, 32 * q4, col + c0), a);
      } else {
        tmem_ld16(tmem_addr(tb, 32 * q4, col + c0), a);
      }
      const float2 cf = make_float2(coef, coef);
      float2 ua = make_float2(0.f, 0.f), ub = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < QF / 8; ++j) {
        float fv[8], sv[8];
        ld_bf16x8(s_phi + sw128_offset(row, c0 + 8 * j, kTile), fv);
        // these 8 features' S or G_S (the same for every row): 128-bit loads
        *reinterpret_cast<float4 *>(sv) = *reinterpret_cast<const float4 *>(vec + c0 + 8 * j);
        *reinterpret_cast<float4 *>(sv + 4) = *reinterpret_cast<const float4 *>(vec + c0 + 8 * j + 4);
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          const float2 dphi = __ffma2_rn(cf, make_float2(sv[i], sv[i + 1]), make_float2(a[8 * j + i], a[8 * j + i + 1]));
          const float2 g = FAVOR ? make_float2(fv[i], fv[i + 1])
                                 : make_float2(fminf(fv[i], 1.f), fminf(fv[i + 1], 1.f));
          const float2 u = __fmul2_rn(g, dphi);
          a[8 * j + i] = u.x;
          a[8 * j + i + 1] = u.y;
          if (i & 2) {
            ub = __fadd2_rn(ub, u);
          } else {
            ua = __fadd2_rn(ua, u);
          }
        }
      }
      usum[part * kTile + row] = (ua.x + ua.y) + (ub.x + ub.y);
      if (FAVOR) {
        // feature m of u -> column m / 2 (low half of the pair first); the
        // four parts of a row share its TMEM lane, so every part's dphi
        // loads complete before any part stores
        float pk[QF / 2];
#pragma unroll
        for (int x = 0; x < QF / 2; ++x) pk[x] = __uint_as_float(pack_bf16(a[2 * x], a[2 * x + 1]));
        named_barrier_sync(1 + q4, kParts * 32);
        if constexpr (QF == 32) {
          tmem_st16(tmem_addr(tb, 32 * q4, col + c0 / 2), pk);
        } else {
          tmem_st8(tmem_addr(tb, 32 * q4, col + c0 / 2), pk);
        }
        if (DW) {
#pragma unroll
          for (int x = 0; x < QF / 2; ++x) pairs[x] = __float_as_uint(pk[x]);
        }
      } else if (live) {
        uint4 *g = reinterpret_cast<uint4 *>(gout + ((size_t)bh * p.L + (size_t)t * kTile + row) * D + c0);
#pragma unroll
        for (int j = 0; j < QF / 8; ++j)
          g[j] = make_uint4(pack_bf16(a[8 * j], a[8 * j + 1]), pack_bf16(a[8 * j + 2], a[8 * j + 3]),
                            pack_bf16(a[8 * j + 4], a[8 * j + 5]), pack_bf16(a[8 * j + 6], a[8 * j + 7]));
      }
    };
    uint32_t uq_pairs[QF / 2], uk_pairs[QF / 2];
    u_side(kX, s_phk, gs_f, 1.f, usk, uk_pairs, p.dk);
    if (FAVOR && kSplit) {
      // dK = u_k W^T (-> X + 64) under u_q
      tmem_st_wait();
      cta_sync();
      if (issue0()) {
        const uint32_t id = make_idesc(128, D, false, true);
        for (int s = 0; s < MC / 16; ++s)
          mma_bf16_ta(tb + kX + 64, tb + kX + 8 * s, desc_mnmajor(s_w, MC, 0, s), id, s > 0);
        mma_commit(mmd_bar);
      }
    }
    if (kSplit) wait_mmc();
    if (CS == 2) {
      // the dA tile is idle from here: Q and K come back into it for the
      // dQ, dK epilogue (the Q tile holds the dV partial, K the next K)
      if (issue0()) {
        mbar_arrive_expect_tx(rl_bar, 2 * tile_bytes);
        tma_load_3d(smem + lay.at, &tmQ, rl_bar, 0, t * kTile, bh);
        tma_load_3d(smem + lay.at + tile_bytes, &tmK, rl_bar, 0, t * kTile, bh);
      }
    }
    if (DW) {
      // phi_k has been read by dphi_q: u_k over it, for the dW MMAs
      const int c0 = QF * part;
#pragma unroll
      for (int j = 0; j < QF / 8; ++j)
        st_shared_v4(s_phk + sw128_offset(row, c0 + 8 * j, kTile), uk_pairs[4 * j], uk_pairs[4 * j + 1],
                     uk_pairs[4 * j + 2], uk_pairs[4 * j + 3]);
    }
    u_side(kT, s_phq, s_f, dd[row], usq, uq_pairs, p.dq);
    if (FAVOR) tmem_st_wait();
    // every thread is past the G update's phase before thread 0 can commit
    // the next group on the same barrier
    wait_mma();  // the G update: dN's tile takes the next dY
    cta_sync();
    if (issue0() && t > t0) tma_load_3d(smem + lay.dy, &tmDY, in2_bar, 0, (t - 1) * kTile, bh);
    if (DW) {
      // phi_q has been read by the G update: u_q over it, for the dW MMAs
      const int c0 = QF * part;
#pragma unroll
      for (int j = 0; j < QF / 8; ++j)
        st_shared_v4(s_phq + sw128_offset(row, c0 + 8 * j, kTile), uq_pairs[4 * j], uq_pairs[4 * j + 1],
                     uq_pairs[4 * j + 2], uq_pairs[4 * j + 3]);
      fence_async_smem();
      cta_sync();
    }

    if (FAVOR) {
      // (j) dQ = u_q W^T - q rowsum(u_q) -> T + 64, dK likewise -> X + 64
      // (its MMAs issued under u_q)
      if (issue0()) {
        const uint32_t id = make_idesc(128, D, false, true);
        for (int s = 0; s < MC / 16; ++s) {
          mma_bf16_ta(tb + kT + 64, tb + kT + 8 * s, desc_mnmajor(s_w, MC, 0, s), id, s > 0);
          if (!kSplit) mma_bf16_ta(tb + kX + 64, tb + kX + 8 * s, desc_mnmajor(s_w, MC, 0, s), id, s > 0);
        }
        mma_done();  // with kSplit, the dK MMAs issued under u_q too
      }
      uint32_t s_xq = s_q, s_xk = s_k;
      if (CS == 2) {
        s_xq = sb + lay.at;
        s_xk = sb + lay.at + tile_bytes;
      }
      auto issue_dw = [&]() {
        // dW^T = u_q^T Q + u_k^T K (features on the lanes) -> T: the dQ, dK
        // MMAs have read u's TMEM pairs there
        const uint32_t id_w = make_idesc(128, D, true, true);
        for (int s = 0; s < kTile / 16; ++s)
          mma_bf16(tb + kT, desc_mnmajor(s_phq, kTile, 0, s), desc_mnmajor(s_xq, kTile, 0, s), id_w, s > 0);
        for (int s = 0; s < kTile / 16; ++s)
          mma_bf16(tb + kT, desc_mnmajor(s_phk, kTile, 0, s), desc_mnmajor(s_xk, kTile, 0, s), id_w, 1);
        mma_commit(mmb_bar);
      };
      auto wait_rl = [&]() {
        if (CS == 2) {
          go &= mbar_wait(rl_bar, rl_phase, p.status, abort_flag);
          rl_phase ^= 1;
        }
      };
      // dQ = u_q W^T - q rowsum(u_q), dK likewise (this CTA's features)
      float oq[QD], ok[QD];
      if constexpr (kSplit) {
        // dK first: its MMAs ran under u_q (their own commit), so its
        // epilogue runs while the dQ MMAs do
        wait_mmd();
        {
          const float sk = (usk[row] + usk[kTile + row]) + (usk[2 * kTile + row] + usk[3 * kTile + row]);
          float b[QD];
          tmem_ld16(tmem_addr(tb, 32 * q4, kX + 64 + QD * part), b);
          wait_rl();
#pragma unroll
          for (int j = 0; j < QD / 8; ++j) {
            float xk[8];
            ld_bf16x8(s_xk + sw128_offset(row, QD * part + 8 * j, kTile), xk);
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
              const float2 k2 = __ffma2_rn(make_float2(-xk[i], -xk[i + 1]), make_float2(sk, sk),
                                           make_float2(b[8 * j + i], b[8 * j + i + 1]));
              ok[8 * j + i] = k2.x;
              ok[8 * j + i + 1] = k2.y;
            }
          }
        }
        wait_mma();
        if (DW && issue0()) issue_dw();
        const float sq = (usq[row] + usq[kTile + row]) + (usq[2 * kTile + row] + usq[3 * kTile + row]);
        float a[QD];
        tmem_ld16(tmem_addr(tb, 32 * q4, kT + 64 + QD * part), a);
#pragma unroll
        for (int j = 0; j < QD / 8; ++j) {
          float xq[8];
          ld_bf16x8(s_xq + sw128_offset(row, QD * part + 8 * j, kTile), xq);
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            const float2 q2 = __ffma2_rn(make_float2(-xq[i], -xq[i + 1]), make_float2(sq, sq),
                                         make_float2(a[8 * j + i], a[8 * j + i + 1]));
            oq[8 * j + i] = q2.x;
            oq[8 * j + i + 1] = q2.y;
          }
        }
      } else {
        wait_mma();
        const float sq = (usq[row] + usq[kTile + row]) + (usq[2 * kTile + row] + usq[3 * kTile + row]);
        const float sk = (usk[row] + usk[kTile + row]) + (usk[2 * kTile + row] + usk[3 * kTile + row]);
        float a[QD], b[QD];
        tmem_ld16x2(tmem_addr(tb, 32 * q4, kT + 64 + QD * part), tmem_addr(tb, 32 * q4, kX + 64 + QD * part), a, b);
        wait_rl();
        if (DW && issue0()) issue_dw();
#pragma unroll
        for (int j = 0; j < QD / 8; ++j) {
          float xq[8], xk[8];
          ld_bf16x8(s_xq + sw128_offset(row, QD * part + 8 * j, kTile), xq);
          ld_bf16x8(s_xk + sw128_offset(row, QD * part + 8 * j, kTile), xk);
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            const float2 q2 = __ffma2_rn(make_float2(-xq[i], -xq[i + 1]), make_float2(sq, sq),
                                         make_float2(a[8 * j + i], a[8 * j + i + 1]));
            const float2 k2 = __ffma2_rn(make_float2(-xk[i], -xk[i + 1]), make_float2(sk, sk),
                                         make_float2(b[8 * j + i], b[8 * j + i + 1]));
            oq[8 * j + i] = q2.x;
            oq[8 * j + i + 1] = q2.y;
            ok[8 * j + i] = k2.x;
            ok[8 * j + i + 1] = k2.y;
          }
        }
      }
      if (CS == 2) {
        // partials -> bf16 in the idle G_V-copy and R-copy tiles for reduce-adds
#pragma unroll
        for (int j = 0; j < QD / 8; ++j) {
          st_bf16x8(s_gv + sw128_offset(row, QD * part + 8 * j, kTile), oq + 8 * j);
          st_bf16x8(s_rb + sw128_offset(row, QD * part + 8 * j, kTile), ok + 8 * j);
        }
        fence_async_smem();
        cta_sync();
        if (issue0()) {
          tma_reduce_add_3d(&tmDQ, s_gv, 0, t * kTile, bh);
          tma_reduce_add_3d(&tmDK, s_rb, 0, t * kTile, bh);
          tma_store_commit();
        }
      } else if (live) {
        uint4 *gq = reinterpret_cast<uint4 *>(p.dq + ((size_t)bh * p.L + (size_t)t * kTile + row) * D + QD * part);
        uint4 *gk = reinterpret_cast<uint4 *>(p.dk + ((size_t)bh * p.L + (size_t)t * kTile + row) * D + QD * part);
#pragma unroll
        for (int j = 0; j < QD / 8; ++j) {
          gq[j] = make_uint4(pack_bf16(oq[8 * j], oq[8 * j + 1]), pack_bf16(oq[8 * j + 2], oq[8 * j + 3]),
                             pack_bf16(oq[8 * j + 4], oq[8 * j + 5]), pack_bf16(oq[8 * j + 6], oq[8 * j + 7]));
          gk[j] = make_uint4(pack_bf16(ok[8 * j], ok[8 * j + 1]), pack_bf16(ok[8 * j + 2], ok[8 * j + 3]),
                             pack_bf16(ok[8 * j + 4], ok[8 * j + 5]), pack_bf16(ok[8 * j + 6], ok[8 * j + 7]));
        }
      }
      if (DW) {
        // this tile's dW^T rows (features fbase + row, 16 value columns per
        // part) added to the segment's partial dW^T [M][D] without waiting
        wait_mmb();
        float wv[16];
        tmem_ld16(tmem_addr(tb, 32 * q4, kT + 16 * part), wv);
        if (row < MC) {
          float *dst = p.dwpart + (((size_t)bh * p.P + seg) * M + fbase + row) * D + 16 * part;
#pragma unroll
          for (int i = 0; i < 16; i += 4) red_add_v4(dst + i, wv[i], wv[i + 1], wv[i + 2], wv[i + 3]);
        }
      }
      // this tile's TMEM loads complete before the next tile's MMAs: with a
      // CTA pair (and no dW) the staging barrier above has ordered them
      if (CS == 1 || DW) cta_sync();
    }
    x_phase ^= 1;
    if (CS == 1 && issue0() && t > t0) {
      mbar_arrive_expect_tx(in_bar, 2 * tile_bytes);
      tma_load_3d(smem + lay.q, &tmQ, in_bar, 0, (t - 1) * kTile, bh);
      tma_load_3d(smem + lay.k, &tmK, in_bar, 0, (t - 1) * kTile, bh);
    }
  }

  if (CS == 2 && tid == 0) tma_store_wait_all();  // the last tile's reduce-adds
  if (tid == 0 && *abort_flag) {
    // a wait gave up: this CTA's MMAs and the loads armed before that land
    // before TMEM is freed and the CTA leaves.  An input barrier whose phase
    // is armed completes it when its bytes land (one of the two parities
    // passes at once); one with nothing armed gives up after 20 ms.
    mma_commit(drain_bar);
    mbar_drain(drain_bar, 0);
    uint64_t *const armed[4] = {in_bar, in2_bar, rl_bar, setup_bar};
    for (int i = 0; i < 4; ++i)
      for (uint32_t par = 0; par < 2; ++par) mbar_drain(armed[i], par, 20000000ull);
  }
  // segment total of G -> gstates, staged in the idle phi / A tiles for one
  // coalesced bulk store of this CTA's rows
  {
    float *stage = reinterpret_cast<float *>(smem + lay.phq);
    const int f = row;
    for (int c = 16 * part; c < 80; c += 16 * kParts) {
      float v[16];
      tmem_ld16(tmem_addr(tb, 32 * q4, kG + c), v);
      if (f < MC) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c + i <= D) stage[f * DP + c + i] = v[i];
      }
    }
  }
  fence_async_smem();
  cta_sync();
  if (tid == 0) {
    bulk_store(p.gstates + ((size_t)bh * p.P + seg) * (size_t)M * DP + (size_t)fbase * DP, sb + lay.phq,
               (uint32_t)(MC * DP * 4));
    tma_store_commit();
    tma_store_wait_read();
  }
  if (CS == 2) cluster_sync();  // no remote store may target an exited CTA
  if (warp == 0) tmem_dealloc(tb, 512);
}

// dQ, dK, dV = 0 before the CTA pairs add their partials (16-byte stores,
// a grid of whole waves over the SMs)
__global__ void zero3_kernel(uint4 *__restrict__ a, uint4 *__restrict__ b, uint4 *__restrict__ c, size_t n16) {
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x) {
    a[i] = z;
    b[i] = z;
    c[i] = z;
  }
}

cudaError_t zero_outputs(const Plan &pl, const Args &a, cudaStream_t st) {
  const size_t n16 = (size_t)pl.BH * pl.L * D * sizeof(__nv_bfloat16) / 16;  // d = 64: 8 per row
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int blocks = (int)std::max<size_t>(1, std::min<size_t>((n16 + 255) / 256, (size_t)sms * 8));
  ProfScope ps("zero_grads", st);
  zero3_kernel<<<blocks, 256, 0, st>>>(static_cast<uint4 *>(a.dq), static_cast<uint4 *>(a.dk),
                                       static_cast<uint4 *>(a.dv), n16);
  return cudaGetLastError();
}

template <bool FAVOR, int CS, int MC>
cudaError_t backward_family(const Plan &pl, const Args &a, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mdy;
  if (!make_map_bf16_3d(&mq, a.q, pl.BH, pl.L, D, kTile) || !make_map_bf16_3d(&mk, a.k, pl.BH, pl.L, D, kTile) ||
      !make_map_bf16_3d(&mv, a.v, pl.BH, pl.L, D, kTile) || !make_map_bf16_3d(&mdy, a.dy, pl.BH, pl.L, D, kTile))
    return cudaErrorInvalidValue;
  CUtensorMap mdq, mdk, mdv;
  if (CS == 2 && (!make_map_bf16_3d(&mdq, a.dq, pl.BH, pl.L, D, kTile) ||
                  !make_map_bf16_3d(&mdk, a.dk, pl.BH, pl.L, D, kTile) ||
                  !make_map_bf16_3d(&mdv, a.dv, pl.BH, pl.L, D, kTile)))
    return cudaErrorInvalidValue;
  if (CS == 1) mdq = mdk = mdv = mq;  // unused
  const bool want_dw = FAVOR && a.dw != nullptr;
  float *dwpart = a.ws + pl.dwpart_off;
  if (want_dw) {
    cudaError_t e = cudaMemsetAsync(dwpart, 0, sizeof(float) * (size_t)pl.BH * pl.P * D * pl.M, st);
    if (e != cudaSuccess) return e;
  }
  // carried states -> features-major: R'_0 of earlier rows (the scan starts
  // from it) and the reverse state G arriving from later rows
  float *init = nullptr, *g_last = nullptr;
  if (a.state_in) {
    init = a.ws + pl.carry_off;
    cudaError_t e = emajor_to_fm(pl, a.state_in, init, st);
    if (e != cudaSuccess) return e;
  }
  if (a.g_in) {
    g_last = a.ws + pl.carry_off + (size_t)pl.BH * pl.M * (D + 1);
    cudaError_t e = emajor_to_fm(pl, a.g_in, g_last, st);
    if (e != cudaSuccess) return e;
  }
  // R' totals of every segment, scanned; with two CTAs per segment the
  // outputs start at zero for the per-CTA reduce-adds.  With the end states
  // the forward left (same segments, same exact scan; its W image sits at
  // the same workspace offset, made from the same W) only the zeroed
  // outputs remain to be made.
  cudaError_t e = cudaSuccess;
  if (a.reuse_states) {
    if (CS == 2) e = zero_outputs(pl, a, st);
  } else {
    e = tc_segment_states(pl, a, pl.P, CS == 2 ? 7 : 0, init, st);
  }
  if (e != cudaSuccess) return e;
  Params p{};
  p.L = pl.L; p.M = pl.M; p.nt = pl.tc_tiles; p.P = pl.P; p.tps = pl.cps; p.favor = FAVOR;
  p.BH = pl.BH;
  p.H = pl.H; p.wstride = pl.wh > 1 ? pl.M * 64 : 0;
  p.dq = static_cast<__nv_bfloat16 *>(a.dq);
  p.dk = static_cast<__nv_bfloat16 *>(a.dk);
  p.dv = static_cast<__nv_bfloat16 *>(a.dv);
  p.w = a.w;
  p.wimg = reinterpret_cast<const __nv_bfloat16 *>(a.ws + pl.wimg_off);
  p.states = a.ws + pl.states_off;
  p.states_lo = a.ws + pl.states_lo_off;
  p.gstates = a.ws + pl.gstates_off;
  p.dwpart = dwpart;
  p.status = a.status;
  {
    const Layout lay(pl.M / CS);
    const int smem = (int)lay.total + 1024;
    auto kern = want_dw ? tc_bwd_kernel<FAVOR, CS, MC, FAVOR> : tc_bwd_kernel<FAVOR, CS, MC, false>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (CS > 1) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
      (void)e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.P * CS, pl.BH);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ProfScope ps("tc_backward", st);
    e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mdy, mdq, mdk, mdv, p);
    if (e != cudaSuccess) return e;
  }
  if (pl.P > 1 || g_last) {
    // G_end(s) = G arriving from later rows + sum over s' > s of the
    // segments' totals, formed by the correction's set-up kernel
    e = tc_correction(pl, a, g_last, st);
    if (e != cudaSuccess) return e;
    // dW's share of the later segments' reverse state
    if (want_dw) e = tc_dw_correction(pl, a, g_last, st);
    if (e != cudaSuccess) return e;
  }
  if (want_dw) e = reduce_dw_t(pl, dwpart, a.dw, st);
  if (e != cudaSuccess) return e;
  // gradient w.r.t. the carried incoming state: the reverse state before the
  // first row, segment 0's own total plus G_end(0)
  if (a.g_out) {
    if (pl.P > 1)
      e = fm_to_emajor(pl, a.ws + pl.gstates_off, pl.P, 0, a.ws + pl.gstates_off, pl.P, 1, a.g_out, st);
    else
      e = fm_to_emajor(pl, a.ws + pl.gstates_off, pl.P, 0, g_last, 1, 0, a.g_out, st);
  }
  return e;
}

}  // namespace tcb

bool tc_backward_supported(int d, int M, int chunk, bool favor) {
  if (tc_backward_elu128_supported(d, M, chunk, favor)) return true;
  if (d != 64) return false;  // 128-row tiles for every slice size
  return favor ? (M == 64 || M == 128 || M == 256) : M == 64;
}

cudaError_t tc_backward(const Plan &p, const Args &a, cudaStream_t st) {
  if (tc_backward_elu128_supported(p.d, p.M, p.C, p.favor != 0)) return tc_backward_elu128(p, a, st);
  if (p.d != 64) return cudaErrorInvalidValue;
  if (!p.favor) return p.M == 64 ? tcb::backward_family<false, 1, 64>(p, a, st) : cudaErrorInvalidValue;
  if (p.M == 256) return tcb::backward_family<true, 2, 128>(p, a, st);
  if (p.M == 128) return tcb::backward_family<true, 1, 128>(p, a, st);
  if (p.M == 64) return tcb::backward_family<true, 1, 64>(p, a, st);
  return cudaErrorInvalidValue;
}

}  // namespace slim
