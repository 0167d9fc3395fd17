// tc_forward.cu -- tensor-core (tcgen05 + TMA) forward for bf16 I/O.
//
// "Sub-Linear Memory: How to Make Performers SLiM", sections 2.1 and 3.2.
// One CTA owns one segment of consecutive 128-row tiles of one (b, h)
// problem and carries the stacked prefix-sum state R' = [R ; S^T] across
// tiles (the slice recurrence of eq. (16)-(18)).  Per tile (rows l of the
// tile, feature block h of at most 128 features):
//   F      = X W_h                     (MMA; X = Q or K, K-major operands)
//   phi    = exp(F - |x|^2/2)/sqrt(M)  (epilogue: TMEM -> bf16 swizzled smem)
//   A     += phi_q,h phi_k,h^T         (MMA, fp32 in TMEM)
//   num'  += phi_q,h [R_h, S_h]^T      (MMA; bf16 copies of R and of S as
//                                       a high and a low part in smem)
//   R'_h  += phi_k,h^T [V, 1]          (MMA; fp32 master state in TMEM)
// then A is masked to its lower triangle (diagonal kept) and rounded to bf16,
//   num'  += tril(A) [V, 1]
// and Y = num / den with den = num'[d] + num'[d + 1].  A tile of 128 rows
// holds two 64-row slices or half a 256-row slice; the paper's slice
// recurrence is exact for any slice size (section 3.4), so the tiling only
// changes rounding.
//
// MODE_STATE runs only the K side and writes the segment's total R' (the
// rows eq. (3) adds) for the segment scan.  With `exact` set (the backward's
// pre-pass) each tile's increment is formed by an MMA that restarts at zero
// and is added to a double-float (hi, lo) total, so the backward can later
// remove exactly the same values; otherwise (the forward's pre-pass, which
// never removes anything) the MMA accumulates in place.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace slim {
namespace tcf {

using namespace slim::tc;

constexpr int kThreads = 256;
constexpr int kTile = 128;

enum { MODE_STATE = 0, MODE_FWD = 1 };

struct Params {
  int L, M, nt, P, tps, favor, exact;
  __nv_bfloat16 *y;
  const float *w;
  float *states;     // fp32 [BH][P][M][D + 1]: high parts of the segment states
  float *states_lo;  // same layout: low parts
  int *status;
};

template <int D>
struct Layout {
  // shared memory (bytes from a 1024-aligned base)
  uint32_t w, q, k, v, phk, phq, rb, ones, sb, bars, total;
  // TMEM columns
  uint32_t t_f, t_f2, t_a, t_num, t_r;
  // TMEM columns of the state pre-pass: increment, (hi, lo) totals
  uint32_t s_delta, s_hi, s_lo;
  __host__ __device__ Layout(int M, bool favor) {
    const uint32_t tile = kTile * D * 2;  // one [128][D] bf16 tile
    uint32_t o = 0;
    w = o; o += favor ? (uint32_t)M * 128u : 0u;  // W^T as [M][64] bf16 (D == 64)
    q = o; o += tile;
    k = o; o += tile;
    v = o; o += tile;
    phk = o; o += kTile * 128 * 2;
    phq = o; o += kTile * 128 * 2;  // also the masked A tile
    rb = o; o += (uint32_t)M * D * 2;
    ones = o; o += 4096;            // [128][16] no-swizzle: column 0 = 1
    sb = o; o += (uint32_t)M * 32u; // [M][16] no-swizzle: columns 0, 1 = S high, S low
    bars = o; o += 64;
    total = o;
    const int nh = (M + 127) / 128;
    t_f = 0;
    t_a = nh > 1 ? 128u : 0u;
    t_num = nh > 1 ? 256u : 128u;
    t_r = t_num + D + 16;
    t_f2 = nh > 1 ? t_f : t_r + (uint32_t)(D + 16);  // a second feature buffer when it fits
    s_delta = 0;
    s_hi = (D + 16 > 128) ? (uint32_t)(D + 16) : 128u;
    s_lo = s_hi + nh * (D + 16);
  }
};

template <int D, bool FAVOR, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    tc_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Layout<D> lay(p.M, FAVOR);
  const uint32_t sbase = smem_u32(smem);
  uint64_t *qk_bar = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint64_t *v_bar = qk_bar + 1;
  uint64_t *mma_bar = qk_bar + 2;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(qk_bar + 3);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(qk_bar + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q4 = warp & 3, ch = warp >> 2, row = 32 * q4 + lane;
  const int seg = blockIdx.x, bh = blockIdx.y;
  const int M = p.M, nh = (M + 127) / 128, DP = D + 1;
  const int t0 = seg * p.tps, t1 = min(t0 + p.tps, p.nt);
  const bool exact = MODE == MODE_STATE && p.exact;
  // two feature buffers let the Q- and K-side feature MMAs run back to back
  const bool dual_f = FAVOR && MODE == MODE_FWD && nh == 1;

  if (tid == 0) {
    mbar_init(qk_bar, 1);
    mbar_init(v_bar, 1);
    mbar_init(mma_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    if (MODE == MODE_FWD) prefetch_tmap(&tmQ);
  }
  if (warp == 0) tmem_alloc(tslot, 512);

  // constant operands: W^T (bf16, K-major rows = features), the ones block,
  // zero padding of phi_k beyond M (the state MMA always reads 128 features)
  if (FAVOR) {
    for (int idx = tid; idx < M * D; idx += kThreads) {
      const int i = idx / M, m = idx - i * M;
      *reinterpret_cast<__nv_bfloat16 *>(smem + lay.w + sw128_offset(m, i, M)) =
          __float2bfloat16_rn(p.w[idx]);
    }
  }
  for (int idx = tid; idx < kTile * 16; idx += kThreads) {
    const int r = idx >> 4, x = idx & 15;
    *reinterpret_cast<__nv_bfloat16 *>(smem + lay.ones + n16_offset(r, x)) = __float2bfloat16_rn(x == 0 ? 1.f : 0.f);
  }
  if (MODE == MODE_FWD) {
    for (int idx = tid; idx < M * 16; idx += kThreads)
      *reinterpret_cast<__nv_bfloat16 *>(smem + lay.sb + n16_offset(idx >> 4, idx & 15)) = __float2bfloat16_rn(0.f);
  }
  if (M < 128) {
    for (int idx = tid; idx < kTile * 128; idx += kThreads) {
      const int r = idx >> 7, x = idx & 127;
      if (x >= M) *reinterpret_cast<__nv_bfloat16 *>(smem + lay.phk + sw128_offset(r, x, kTile)) =
          __float2bfloat16_rn(0.f);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  // S of feature f as the bf16 pair (high, low) in columns 0, 1 of the S block
  auto put_s = [&](int f, float sv) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(sv);
    *reinterpret_cast<__nv_bfloat16 *>(smem + lay.sb + n16_offset(f, 0)) = hi;
    *reinterpret_cast<__nv_bfloat16 *>(smem + lay.sb + n16_offset(f, 1)) =
        __float2bfloat16_rn(sv - __bfloat162float(hi));
  };

  // incoming state of the segment -> TMEM master, bf16 copies of R and S
  // (the pre-pass instead starts its totals at zero)
  const int ncols = D + 16, csplit = ((ncols / 16 + 1) / 2) * 16;
  if (MODE == MODE_STATE) {
    for (int b = 0; b < nh; ++b) {
      float z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0.f;
      for (int c = ch ? csplit : 0; c < (ch ? ncols : csplit); c += 16) {
        if (exact) {
          tmem_st16(tmem_addr(tbase, 32 * q4, lay.s_hi + b * ncols + c), z);
          tmem_st16(tmem_addr(tbase, 32 * q4, lay.s_lo + b * ncols + c), z);
        } else {
          tmem_st16(tmem_addr(tbase, 32 * q4, lay.t_r + b * ncols + c), z);
        }
      }
    }
    tmem_st_wait();
  } else {
    const size_t off = ((size_t)bh * p.P + seg - 1) * (size_t)M * DP;
    const float *st = seg > 0 ? p.states + off : nullptr;
    const float *st_lo = seg > 0 ? p.states_lo + off : nullptr;
    for (int b = 0; b < nh; ++b) {
      // warps 4b..4b+3 own block b when nh == 2; all warps split columns when nh == 1
      if (nh == 2 && ch != b) continue;
      const int f = 128 * b + row;
      const int c_lo = (nh == 2) ? 0 : (ch == 0 ? 0 : (ncols / 32) * 16);
      const int c_hi = (nh == 2) ? ncols : (ch == 0 ? (ncols / 32) * 16 : ncols);
      for (int c = c_lo; c < c_hi; c += 16) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = c + i;
          v[i] = (st && f < M && e <= D) ? st[(size_t)f * DP + e] + st_lo[(size_t)f * DP + e] : 0.f;
        }
        tmem_st16(tmem_addr(tbase, 32 * q4, lay.t_r + b * ncols + c), v);
        if (f < M) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int e = c + i;
            if (e < D)
              *reinterpret_cast<__nv_bfloat16 *>(smem + lay.rb + sw128_offset(f, e, M)) = __float2bfloat16_rn(v[i]);
            else if (e == D)
              put_s(f, v[i]);
          }
        }
      }
    }
    tmem_st_wait();
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tile_bytes = kTile * D * 2;
  uint32_t qk_phase = 0, v_phase = 0, mma_phase = 0;
  auto issue_qk = [&](int t) {
    const uint32_t bytes = (MODE == MODE_FWD ? 2u : 1u) * tile_bytes;
    mbar_arrive_expect_tx(qk_bar, bytes);
    for (int c = 0; c < D; c += 64) {
      tma_load_3d(smem + lay.k + c * kTile * 2, &tmK, qk_bar, c, t * kTile, bh);
      if (MODE == MODE_FWD) tma_load_3d(smem + lay.q + c * kTile * 2, &tmQ, qk_bar, c, t * kTile, bh);
    }
  };
  auto issue_v = [&](int t) {
    mbar_arrive_expect_tx(v_bar, tile_bytes);
    for (int c = 0; c < D; c += 64) tma_load_3d(smem + lay.v + c * kTile * 2, &tmV, v_bar, c, t * kTile, bh);
  };
  auto mma_sync_all = [&]() {
    __syncwarp();
    mbar_wait(mma_bar, mma_phase, p.status, abort_flag);
    mma_phase ^= 1;
    tc_fence_after();
  };
  auto cta_sync = [&]() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };

  if (tid == 0 && t0 < t1) {
    issue_qk(t0);
    issue_v(t0);
  }

  const uint32_t s_q = sbase + lay.q, s_k = sbase + lay.k, s_v = sbase + lay.v;
  const uint32_t s_phk = sbase + lay.phk, s_phq = sbase + lay.phq, s_rb = sbase + lay.rb;
  const uint32_t s_ones = sbase + lay.ones, s_w = sbase + lay.w, s_sb = sbase + lay.sb;

  // feature MMA: F = X W_h^T for feature block h (nu features)
  auto issue_features = [&](uint32_t s_x, uint32_t t_out, int h, int nu) {
    const uint32_t idesc = make_idesc(128, nu, false, false);
    for (int s = 0; s < D / 16; ++s)
      mma_bf16(tbase + t_out, desc_kmajor(s_x, kTile, 0, s), desc_kmajor(s_w, M, 128 * h, s), idesc, s > 0);
  };
  // phi = exp2(F log2 e + c) from TMEM into the swizzled bf16 tile
  auto favor_epilogue = [&](uint32_t t_in, uint32_t s_out, int cols, float c_row, bool zero_row) {
    if (cols == 64) {
      float v[64];
      tmem_ld32x2(tmem_addr(tbase, 32 * q4, t_in + 64 * ch), tmem_addr(tbase, 32 * q4, t_in + 64 * ch + 32), v,
                  v + 32);
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] = zero_row ? 0.f : favor_feature(v[i], c_row);
#pragma unroll
      for (int j = 0; j < 8; ++j) st_bf16x8(s_out + sw128_offset(row, 64 * ch + 8 * j, kTile), v + 8 * j);
      return;
    }
    for (int c0 = ch * cols; c0 < (ch + 1) * cols; c0 += 32) {
      float v[32];
      tmem_ld32(tmem_addr(tbase, 32 * q4, t_in + c0), v);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = favor_feature(v[i], c_row);
      if (zero_row) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) st_bf16x8(s_out + sw128_offset(row, c0 + 8 * j, kTile), v + 8 * j);
    }
  };
  auto elu_epilogue = [&](uint32_t s_x, uint32_t s_out, int cols, bool zero_row) {
    for (int c0 = ch * cols; c0 < (ch + 1) * cols; c0 += 8) {
      float v[8];
      ld_bf16x8(s_x + sw128_offset(row, c0, kTile), v);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = zero_row ? 0.f : elu1_feature(v[i]);
      st_bf16x8(s_out + sw128_offset(row, c0, kTile), v);
    }
  };

  for (int t = t0; t < t1; ++t) {
    const int valid = min(kTile, p.L - t * kTile);
    const bool dead = row >= valid;  // padding rows past L: features forced to zero
    mbar_wait(qk_bar, qk_phase, p.status, abort_flag);
    qk_phase ^= 1;
    float ck = 0.f, cq = 0.f;  // per-row exp2 offsets
    if (FAVOR) {
      ck = favor_row_const(tile_row_sqnorm(s_k, row, D), M);
      if (MODE == MODE_FWD) cq = favor_row_const(tile_row_sqnorm(s_q, row, D), M);
    }
    if (FAVOR && tid == 0) {
      issue_features(s_k, lay.t_f, 0, min(128, M));
      if (dual_f) issue_features(s_q, lay.t_f2, 0, M);
      mma_commit(mma_bar);
    }
    for (int h = 0; h < nh; ++h) {
      const int nu = min(128, M - 128 * h);  // features in this block
      const int cols = nu / 2;               // per thread (two threads per row)
      // K side (its feature MMA was issued already)
      if (FAVOR) {
        mma_sync_all();
        favor_epilogue(lay.t_f, s_phk, cols, ck, dead);
        if (dual_f) favor_epilogue(lay.t_f2, s_phq, cols, cq, dead);
      } else {
        elu_epilogue(s_k, s_phk, cols, dead);
        if (MODE == MODE_FWD) elu_epilogue(s_q, s_phq, cols, dead);
      }
      fence_async_smem();
      cta_sync();
      if (MODE == MODE_FWD && FAVOR && !dual_f) {
        if (tid == 0) {
          issue_features(s_q, lay.t_f, h, nu);
          mma_commit(mma_bar);
        }
        mma_sync_all();
        favor_epilogue(lay.t_f, s_phq, cols, cq, dead);
        fence_async_smem();
        cta_sync();
      }
      // next tile's Q/K can stream in once the last feature block is formed
      if (h == nh - 1 && tid == 0 && t + 1 < t1) issue_qk(t + 1);
      if (tid == 0) {
        if (MODE == MODE_FWD) {
          const uint32_t id_a = make_idesc(128, 128, false, false);
          const uint32_t id_n = make_idesc(128, D, false, true);
          const uint32_t id_s = make_idesc(128, 16, false, true);
          for (int s = 0; s < nu / 16; ++s)
            mma_bf16(tbase + lay.t_a, desc_kmajor(s_phq, kTile, 0, s), desc_kmajor(s_phk, kTile, 0, s), id_a,
                     (h > 0 || s > 0));
          for (int s = 0; s < nu / 16; ++s) {
            mma_bf16(tbase + lay.t_num, desc_kmajor(s_phq, kTile, 0, s), desc_mnmajor(s_rb, M, 0, 8 * h + s), id_n,
                     (h > 0 || s > 0));
            mma_bf16(tbase + lay.t_num + D, desc_kmajor(s_phq, kTile, 0, s), desc_n16(s_sb, 8 * h + s), id_s,
                     (h > 0 || s > 0));
          }
        }
        if (h == 0) {
          mbar_wait(v_bar, v_phase, p.status, abort_flag);
          v_phase ^= 1;
        }
        if (exact) {
          issue_state_delta(tbase + lay.s_delta, s_phk, s_v, s_ones, D);
        } else {
          // the running state only moves forward here: accumulate in place
          const uint32_t id_r = make_idesc(128, D, true, true);
          const uint32_t id_r1 = make_idesc(128, 16, true, true);
          const uint32_t t_r = tbase + lay.t_r + h * ncols;
          for (int s = 0; s < kTile / 16; ++s) {
            mma_bf16(t_r, desc_mnmajor(s_phk, kTile, 0, s), desc_mnmajor(s_v, kTile, 0, s), id_r, 1);
            mma_bf16(t_r + D, desc_mnmajor(s_phk, kTile, 0, s), desc_n16(s_ones, s), id_r1, 1);
          }
        }
        // the next feature block's K side shares this commit (F is free)
        if (FAVOR && h + 1 < nh && !exact) issue_features(s_k, lay.t_f, h + 1, min(128, M - 128 * (h + 1)));
        mma_commit(mma_bar);
      }
      if (exact) {
        mma_sync_all();
        // (hi, lo) total of block h += this tile's increment
        df_update_tmem(tbase, 32 * q4, lay.s_delta, lay.s_hi + h * ncols, lay.s_lo + h * ncols,
                       ch ? csplit : 0, ch ? ncols : csplit, 1.f);
        cta_sync();
        if (FAVOR && h + 1 < nh && tid == 0) {
          issue_features(s_k, lay.t_f, h + 1, min(128, M - 128 * (h + 1)));
          mma_commit(mma_bar);
        }
      } else if (h + 1 == nh || !FAVOR) {
        mma_sync_all();
      }
    }
    if (MODE == MODE_FWD) {
      // masked A (diagonal kept) -> bf16 into the phi_q buffer
      {
        float v[64];
        tmem_ld32x2(tmem_addr(tbase, 32 * q4, lay.t_a + 64 * ch), tmem_addr(tbase, 32 * q4, lay.t_a + 64 * ch + 32),
                    v, v + 32);
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (64 * ch + i > row) v[i] = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) st_bf16x8(s_phq + sw128_offset(row, 64 * ch + 8 * j, kTile), v + 8 * j);
      }
      fence_async_smem();
      cta_sync();
      if (tid == 0) {
        const uint32_t id_n = make_idesc(128, D, false, true);
        const uint32_t id_n1 = make_idesc(128, 16, false, true);
        for (int s = 0; s < kTile / 16; ++s) {
          mma_bf16(tbase + lay.t_num, desc_kmajor(s_phq, kTile, 0, s), desc_mnmajor(s_v, kTile, 0, s), id_n, 1);
          mma_bf16(tbase + lay.t_num + D, desc_kmajor(s_phq, kTile, 0, s), desc_n16(s_ones, s), id_n1, 1);
        }
        mma_commit(mma_bar);
      }
      mma_sync_all();
      if (tid == 0 && t + 1 < t1) issue_v(t + 1);
      // Y = num / den
      {
        float dv[16];
        tmem_ld16(tmem_addr(tbase, 32 * q4, lay.t_num + D), dv);
        const float inv = 1.0f / (dv[0] + dv[1]);
        __nv_bfloat16 *yrow = p.y + ((size_t)bh * p.L + (size_t)t * kTile + row) * D;
        for (int c0 = ch * (D / 2); c0 < (ch + 1) * (D / 2); c0 += 32) {
          float v[32];
          tmem_ld32(tmem_addr(tbase, 32 * q4, lay.t_num + c0), v);
          if (!dead) {
            uint4 *dst = reinterpret_cast<uint4 *>(yrow + c0);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(pack_bf16(v[8 * j] * inv, v[8 * j + 1] * inv),
                                  pack_bf16(v[8 * j + 2] * inv, v[8 * j + 3] * inv),
                                  pack_bf16(v[8 * j + 4] * inv, v[8 * j + 5] * inv),
                                  pack_bf16(v[8 * j + 6] * inv, v[8 * j + 7] * inv));
          }
        }
      }
      // refresh the bf16 copies of R' and S for the next tile
      for (int b = 0; b < nh; ++b) {
        if (nh == 2 && ch != b) continue;
        const int f = 128 * b + row;
        if (f >= M) continue;
        const int c_lo = (nh == 2) ? 0 : (ch == 0 ? 0 : (ncols / 32) * 16);
        const int c_hi = (nh == 2) ? ncols : (ch == 0 ? (ncols / 32) * 16 : ncols);
        for (int c = c_lo; c < c_hi; c += 16) {
          float v[16];
          tmem_ld16(tmem_addr(tbase, 32 * q4, lay.t_r + b * ncols + c), v);
#pragma unroll
          for (int i = 0; i < 16; i += 8) {
            if (c + i + 8 <= D) st_bf16x8(s_rb + sw128_offset(f, c + i, M), v + i);
          }
          if (c <= D && D < c + 16) put_s(f, v[D - c]);
        }
      }
      fence_async_smem();
      cta_sync();
    } else {
      if (tid == 0 && t + 1 < t1) issue_v(t + 1);
    }
  }

  if (MODE == MODE_STATE) {
    // segment total of R' -> fp32 [M][D + 1], high and low parts
    const size_t off = ((size_t)bh * p.P + seg) * (size_t)M * DP;
    for (int b = 0; b < nh; ++b) {
      const int f = 128 * b + row;
      for (int c = ch ? csplit : 0; c < (ch ? ncols : csplit); c += 16) {
        float h[16], l[16];
        if (exact) {
          tmem_ld16(tmem_addr(tbase, 32 * q4, lay.s_hi + b * ncols + c), h);
          tmem_ld16(tmem_addr(tbase, 32 * q4, lay.s_lo + b * ncols + c), l);
        } else {
          tmem_ld16(tmem_addr(tbase, 32 * q4, lay.t_r + b * ncols + c), h);
#pragma unroll
          for (int i = 0; i < 16; ++i) l[i] = 0.f;
        }
        if (f < M) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c + i <= D) {
              p.states[off + (size_t)f * DP + c + i] = h[i];
              p.states_lo[off + (size_t)f * DP + c + i] = l[i];
            }
        }
      }
    }
  }
  cta_sync();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

template <int D, bool FAVOR, int MODE>
cudaError_t launch(const Plan &pl, const Args &a, const CUtensorMap &mq, const CUtensorMap &mk,
                   const CUtensorMap &mv, int nseg, bool exact, cudaStream_t st) {
  Params p{};
  p.L = pl.L; p.M = pl.M; p.nt = pl.tc_tiles; p.P = pl.P; p.tps = pl.cps; p.favor = FAVOR;
  p.exact = exact ? 1 : 0;
  p.y = static_cast<__nv_bfloat16 *>(a.y);
  p.w = a.w;
  p.states = a.ws + pl.states_off;
  p.states_lo = a.ws + pl.states_lo_off;
  p.status = a.status;
  const Layout<D> lay(pl.M, FAVOR);
  const int smem = (int)lay.total + 1024;
  auto kern = tc_fwd_kernel<D, FAVOR, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(nseg, pl.BH), kThreads, smem, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

// Totals of R' over the first nseg segments, then their inclusive scan:
// states[s] = R' at the end of segment s.
template <int D, bool FAVOR>
cudaError_t segment_states(const Plan &pl, const Args &a, const CUtensorMap &mq,
                           const CUtensorMap &mk, const CUtensorMap &mv, int nseg, bool exact,
                           cudaStream_t st) {
  cudaError_t e;
  {
    ProfScope ps("tc_segment_state", st);
    e = launch<D, FAVOR, MODE_STATE>(pl, a, mq, mk, mv, nseg, exact, st);
    if (e != cudaSuccess) return e;
  }
  if (nseg > 1) {
    ProfScope ps("scan_states", st);
    e = scan_states_df(pl, a.ws + pl.states_off, a.ws + pl.states_lo_off, nseg, st);
  }
  return e;
}

template <int D, bool FAVOR>
cudaError_t forward_family(const Plan &pl, const Args &a, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_map_bf16_3d(&mq, a.q, pl.BH, pl.L, D, kTile) || !make_map_bf16_3d(&mk, a.k, pl.BH, pl.L, D, kTile) ||
      !make_map_bf16_3d(&mv, a.v, pl.BH, pl.L, D, kTile))
    return cudaErrorInvalidValue;
  cudaError_t e;
  if (pl.P > 1) {
    e = segment_states<D, FAVOR>(pl, a, mq, mk, mv, pl.P - 1, false, st);
    if (e != cudaSuccess) return e;
  }
  ProfScope ps("tc_forward", st);
  return launch<D, FAVOR, MODE_FWD>(pl, a, mq, mk, mv, pl.P, false, st);
}

}  // namespace tcf

size_t tc_smem_bytes(int d, int M, bool favor) {
  if (d == 64) return tcf::Layout<64>(M, favor).total + 1024;
  return tcf::Layout<128>(M, favor).total + 1024;
}

bool tc_forward_supported(int d, int M, int chunk, bool favor) {
  if (chunk < 64) return false;
  if (d == 64) return favor ? (M == 64 || M == 128 || M == 256) : M == 64;
  if (d == 128) return !favor && M == 128;
  return false;
}

cudaError_t tc_segment_states(const Plan &p, const Args &a, int nseg, cudaStream_t st) {
  CUtensorMap mk, mv;
  const int d = p.d;
  if (!make_map_bf16_3d(&mk, a.k, p.BH, p.L, d, tcf::kTile) || !make_map_bf16_3d(&mv, a.v, p.BH, p.L, d, tcf::kTile))
    return cudaErrorInvalidValue;
  if (d == 64 && p.favor) return tcf::segment_states<64, true>(p, a, mk, mk, mv, nseg, true, st);
  if (d == 64) return tcf::segment_states<64, false>(p, a, mk, mk, mv, nseg, true, st);
  if (d == 128 && !p.favor) return tcf::segment_states<128, false>(p, a, mk, mk, mv, nseg, true, st);
  return cudaErrorInvalidValue;
}

cudaError_t tc_forward(const Plan &p, const Args &a, cudaStream_t st) {
  if (p.d == 64 && p.favor) return tcf::forward_family<64, true>(p, a, st);
  if (p.d == 64) return tcf::forward_family<64, false>(p, a, st);
  if (p.d == 128 && !p.favor) return tcf::forward_family<128, false>(p, a, st);
  return cudaErrorInvalidValue;
}

}  // namespace slim
