// tc_forward.cu -- tensor-core (tcgen05 + TMA) forward for bf16 I/O.
//
// "Sub-Linear Memory: How to Make Performers SLiM", sections 2.1 and 3.2.
// One CTA owns one segment of consecutive 128-row tiles of one (b, h)
// problem and carries the stacked prefix-sum state R' = [R ; S^T] across
// tiles (the slice recurrence of eq. (16)-(18)).  Per tile, for each block h
// of at most 128 features:
//   F      = X W_h                     (MMA; X = K, then Q)
//   phi    = exp(F - |x|^2/2)/sqrt(M)  (epilogue: TMEM -> bf16 swizzled smem)
//   R'_h  += phi_k,h^T [V, 1]          (MMA; fp32 master state in TMEM)
//   A     += phi_q,h phi_k,h^T         (MMA)
//   num   += phi_q,h R_h^T             (MMA; bf16 copy of R(t-1) in smem)
//   den   += phi_q,h . S_h             (epilogue, fp32 S(t-1))
// then A is masked to its lower triangle (diagonal kept) and rounded to bf16,
//   [num, rowsum(A)] += tril(A) [V, 1]
// and Y = num / (den + rowsum(A)).  With d = 64 the ones column rides along
// V as a second 64-column operand block (one N = 80 MMA): every tcgen05.mma
// holds the tensor pipe for at least ~50 cycles, so N = 16 side MMAs for the
// normaliser would cost as much as the products themselves.  A tile of 128 rows
// holds two 64-row slices or half a 256-row slice; the paper's slice
// recurrence is exact for any slice size (section 3.4), so the tiling only
// changes rounding.
//
// The kernel is warp-specialised so that the tensor pipe, the exponentials
// and the loads overlap across tiles:
//   warp 0      TMA producer: K, Q, V tiles into a ring of shared slots;
//   warp 1      MMA issuer (one thread);
//   warps 2-9   epilogue: two threads per row, each half of the columns.
// Features and scores go through two TMEM buffers used in turn, so the next
// feature MMA runs while the epilogue turns the previous one into phi.  Every
// hand-off is an mbarrier; every wait is bounded.
//
// MODE_STATE runs only the K side and writes the segment's total R' (the
// rows eq. (3) adds) for the segment scan.  Each tile's increment is an MMA
// that restarts at zero, and the epilogue adds it into an fp32 master in
// TMEM, as a double-float (low part in shared memory) for the normaliser
// column S.  The backward recovers the first tiles' small states by
// subtracting increments from this total, so rounding in the total shows
// up there: accumulating in place on the tensor pipe cost dQ of the first
// tiles of a long segment a factor of two hundred, and plain fp32 still a
// factor of 2.6 through S, whose positive terms make its rounding errors
// add up; the signed R columns' errors do not.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tma_host.h"

namespace slim {
namespace tcf {

using namespace slim::tc;

constexpr int kTile = 128;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);

enum { MODE_STATE = 0, MODE_FWD = 1 };

struct Params {
  int L, M, nt, P, tps;
  int zero_grads;  // state pass of a two-CTA backward: zero dQ, dK, dV tile by tile
  __nv_bfloat16 *y;
  const __nv_bfloat16 *wimg;  // W^T shared-memory image (FAVOR+)
  float *states;     // fp32 [BH][P][M][D + 1]: high parts of the segment states
  float *states_lo;  // same layout: low parts
  int *status;
};

template <int D, bool FAVOR, int MODE>
struct Cfg {
  static constexpr int kSlots = D == 128 ? 3 : 4;         // ring of [128][D] bf16 tiles
  static constexpr int kLoads = MODE == MODE_FWD ? 3 : 2;  // per tile: K, (Q), V
  static constexpr int kNbuf = FAVOR && MODE == MODE_FWD ? 2 : 1;  // TMEM buffers for F and A
  static constexpr int kGroup = 1;                         // state pass: tiles per partial
  static constexpr uint32_t kTileBytes = kTile * D * 2;
  static constexpr int kCols = D + 16;                     // TMEM columns of num' or one R' block
};

// mbarrier indices
enum {
  B_FULL = 0,       // [slots] TMA -> consumers
  B_EMPTY = 4,      // [slots] consumers -> TMA (1 MMA arrival + 8 epilogue warps)
  B_FFULL = 8,      // [2] F or A ready in TMEM buffer
  B_FEMPTY = 10,    // [2] TMEM buffer read out by the epilogue
  B_PHK = 12,       // phi_k block stored
  B_PHQ = 13,       // phi_q block stored
  B_PHFREE = 14,    // MMAs reading the previous feature block done
  B_AFULL = 15,     // A and the tile's state update complete (state pass: group partial ready)
  B_ATFULL = 16,    // masked A stored
  B_NUMFULL = 17,   // num' complete
  B_NUMEMPTY = 18,  // num' read out
  B_RBFULL = 19,    // R(t) read out of TMEM, bf16 copies refreshed (state pass: partial free)
  B_DONE = 20,      // MMA drain
  B_SETUP = 21,     // set-up copies (W image, incoming state)
  B_EPI = 22,       // epilogue warps' S and den partials written
  B_COUNT = 23
};

template <int D, bool FAVOR, int MODE>
struct Layout {
  using C = Cfg<D, FAVOR, MODE>;
  // shared memory (bytes from a 1024-aligned base)
  uint32_t w, slots, phk, phq, rb, ones, ss, zero, lo, denp, bars, total;
  // TMEM columns
  uint32_t t_buf0, t_buf1, t_num, t_r, t_m;
  __host__ __device__ explicit Layout(int M) {
    uint32_t o = 0;
    w = o; o += FAVOR ? (uint32_t)M * 128u : 0u;  // W^T as [M][64] bf16 (D == 64)
    slots = o; o += C::kSlots * C::kTileBytes;
    phk = o; o += kTile * 128 * 2;                 // one feature block of phi_k
    phq = o; o += MODE == MODE_FWD ? kTile * 128 * 2 : 0u;  // phi_q block, then masked A
    rb = o; o += MODE == MODE_FWD ? (uint32_t)M * D * 2 : 0u;
    // column 0 = 1: a [128][64] 128-B-swizzled block placed after every V
    // slot (d = 64), else a [128][16] no-swizzle operand
    ones = o; o += D == 64 ? 16384u : 4096u;
    ss = o; o += MODE == MODE_FWD ? (uint32_t)M * 4u : 0u;        // fp32 S(t-1)
    // a zero tile (state pass of the two-CTA backward, d = 64 only)
    zero = o; o += (MODE == MODE_STATE && D == 64) ? C::kTileBytes : 0u;
    lo = o; o += MODE == MODE_STATE ? (uint32_t)M * (D + 1) * 4u : 0u;  // low parts [M][D + 1] (state pass)
    denp = o; o += MODE == MODE_FWD ? 2u * 2u * kTile * 4u : 0u;  // [tile parity][half][row]
    bars = o; o += 8 * B_COUNT + 16;
    total = o;
    t_buf0 = 0;
    t_buf1 = C::kNbuf > 1 ? 128u : 0u;
    const uint32_t used = (FAVOR || MODE == MODE_FWD) ? 128u * C::kNbuf : 0u;
    t_num = used;
    t_r = MODE == MODE_FWD ? t_num + C::kCols : used;  // R' (state pass: group partial)
    t_m = t_r + (M > 128 ? 2u : 1u) * C::kCols;        // state pass: fp32 master total
  }
};

template <int D, bool FAVOR, int MODE, int M>
__global__ void __launch_bounds__(kThreads, 1)
    tc_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDQ,
                  const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV, Params p) {
  using C = Cfg<D, FAVOR, MODE>;
  constexpr int NC = C::kCols;
  constexpr int nb = (M + 127) / 128, FB = M < 128 ? M : 128, DP = D + 1;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Layout<D, FAVOR, MODE> lay(M);
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + B_COUNT);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar + B_COUNT) + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x, bh = blockIdx.y;
  const int t0 = seg * p.tps, t1 = min(t0 + p.tps, p.nt), ntl = max(t1 - t0, 0);

  if (tid == 0) {
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar + B_FULL + s, 1);
      mbar_init(bar + B_EMPTY + s, 1 + kEpiWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar + B_FFULL + b, 1);
      mbar_init(bar + B_FEMPTY + b, kEpiWarps);
    }
    mbar_init(bar + B_PHK, kEpiWarps);
    mbar_init(bar + B_PHQ, kEpiWarps);
    mbar_init(bar + B_PHFREE, 1);
    mbar_init(bar + B_AFULL, 1);
    mbar_init(bar + B_ATFULL, kEpiWarps);
    mbar_init(bar + B_NUMFULL, 1);
    mbar_init(bar + B_NUMEMPTY, kEpiWarps);
    mbar_init(bar + B_RBFULL, kEpiWarps);
    mbar_init(bar + B_DONE, 1);
    mbar_init(bar + B_SETUP, 1);
    mbar_init(bar + B_EPI, kEpiWarps);
    *abort_flag = 0;
    fence_barrier_init();
    // W^T image and the incoming state (high parts: the forward's master is
    // fp32, below which the low parts do not register) by bulk copy
    const uint32_t wbytes = FAVOR ? (uint32_t)M * 128u : 0u;
    const uint32_t sbytes = (MODE == MODE_FWD && seg > 0) ? (uint32_t)(M * DP * 4) : 0u;
    if (wbytes + sbytes > 0) {
      mbar_arrive_expect_tx(bar + B_SETUP, wbytes + sbytes);
      if (wbytes) bulk_load(smem + lay.w, p.wimg, wbytes, bar + B_SETUP);
      if (sbytes)
        bulk_load(smem + lay.slots, p.states + ((size_t)bh * p.P + seg - 1) * (size_t)M * DP, sbytes, bar + B_SETUP);
    }
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    if (MODE == MODE_FWD) prefetch_tmap(&tmQ);
  }
  if (warp == 0) tmem_alloc(tslot, 512);

  // constant operands: the ones block, zero padding of phi_k beyond M (the
  // state MMA always reads 128 features)
  if (MODE == MODE_STATE) {
    if (D == 64)
      for (int idx = tid; idx < (int)(C::kTileBytes / 16); idx += kThreads)
        reinterpret_cast<uint4 *>(smem + lay.zero)[idx] = make_uint4(0u, 0u, 0u, 0u);
    for (int idx = tid; idx < M * (D + 1); idx += kThreads) reinterpret_cast<float *>(smem + lay.lo)[idx] = 0.f;
  }
  for (int idx = tid; idx < kTile * (D == 64 ? 64 : 16); idx += kThreads) {
    const int r = D == 64 ? idx >> 6 : idx >> 4, x = D == 64 ? idx & 63 : idx & 15;
    *reinterpret_cast<__nv_bfloat16 *>(smem + lay.ones + (D == 64 ? sw128_offset(r, x, kTile) : n16_offset(r, x))) =
        __float2bfloat16_rn(x == 0 ? 1.f : 0.f);
  }
  if (M < 128) {
    for (int idx = tid; idx < kTile * 128; idx += kThreads) {
      const int r = idx >> 7, x = idx & 127;
      if (x >= M)
        *reinterpret_cast<__nv_bfloat16 *>(smem + lay.phk + sw128_offset(r, x, kTile)) = __float2bfloat16_rn(0.f);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  // incoming state of the segment -> TMEM master (and, in the forward, its
  // bf16 copies); the state pass starts its master at zero.  The fp32
  // [M][D + 1] state arrived in the (still unused) load slots.
  {
    const bool in = MODE == MODE_FWD && seg > 0;
    if ((FAVOR || in) && !mbar_wait(bar + B_SETUP, 0, p.status, abort_flag)) {
      // nothing usable arrived: the tiles below are skipped by the abort flag
    }
    const float *stage = reinterpret_cast<const float *>(smem + lay.slots);  // [M][D + 1] fp32
    const int q4 = warp & 3, half = (warp - 2) >> 2, row = 32 * q4 + lane;
    const uint32_t t_dst = MODE == MODE_FWD ? lay.t_r : lay.t_m;
    constexpr int csplit = ((NC / 16 + 1) / 2) * 16;
    for (int b = 0; b < nb; ++b) {
      if (warp >= 2) {
        const int c_lo = nb == 2 ? 0 : (half ? csplit : 0);
        const int c_hi = nb == 2 ? (b == half ? NC : 0) : (half ? NC : csplit);
        const int f = 128 * b + row;
        for (int c = c_lo; c < c_hi; c += 16) {
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = (in && f < M && c + i <= D) ? stage[f * DP + c + i] : 0.f;
          tmem_st16(tmem_addr(tbase, 32u * q4, t_dst + b * NC + c), v);
          if (MODE == MODE_FWD && f < M) {
#pragma unroll
            for (int i = 0; i < 16; i += 8)
              if (c + i + 8 <= D) st_bf16x8(sbase + lay.rb + sw128_offset(f, c + i, M), v + i);
            if (c <= D && D < c + 16) reinterpret_cast<float *>(smem + lay.ss)[f] = v[D - c];
          }
        }
        tmem_st_wait();
      }
    }
    // num' columns d .. d+15 start at zero (only the ones product adds there)
    if (MODE == MODE_FWD && warp >= 2 && half == 0) {
      float z[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] = 0.f;
      tmem_st16(tmem_addr(tbase, 32u * q4, lay.t_num + D), z);
      tmem_st_wait();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  const uint32_t s_w = sbase + lay.w, s_phk = sbase + lay.phk, s_phq = sbase + lay.phq;
  const uint32_t s_rb = sbase + lay.rb, s_ones = sbase + lay.ones;
  auto t_buf = [&](int b) { return b ? lay.t_buf1 : lay.t_buf0; };
  auto slot_addr = [&](int n) { return sbase + lay.slots + (uint32_t)(n % C::kSlots) * C::kTileBytes; };
  auto slot_par = [&](int n) { return (uint32_t)((n / C::kSlots) & 1); };
  // the TMEM buffer of job j (features, then the tile's A, in issue order)
  // and the index of that use of the buffer
  auto job_buf = [&](int j) { return C::kNbuf > 1 ? (j & 1) : 0; };
  auto job_use = [&](int j) { return C::kNbuf > 1 ? (j >> 1) : j; };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int n = 0;
      bool ok = true;
      auto load = [&](const CUtensorMap *m, int t) {
        const int s = n % C::kSlots, u = n / C::kSlots;
        if (u > 0 && !mbar_wait(bar + B_EMPTY + s, (u - 1) & 1, p.status, abort_flag)) return false;
        mbar_arrive_expect_tx(bar + B_FULL + s, C::kTileBytes);
        for (int c = 0; c < D; c += 64)
          tma_load_3d(smem + lay.slots + s * C::kTileBytes + c * kTile * 2, m, bar + B_FULL + s, c, t * kTile, bh);
        ++n;
        return true;
      };
      for (int t = t0; t < t1 && ok; ++t) {
        ok = load(&tmK, t);
        if (ok && MODE == MODE_FWD) ok = load(&tmQ, t);
        if (ok) ok = load(&tmV, t);
        if (MODE == MODE_STATE && D == 64 && p.zero_grads) {
          // the two-CTA backward adds its per-CTA partials of dQ, dK, dV
          for (int c = 0; c < D; c += 64) {
            tma_store_3d(&tmDQ, smem + lay.zero + c * kTile * 2, c, t * kTile, bh);
            tma_store_3d(&tmDK, smem + lay.zero + c * kTile * 2, c, t * kTile, bh);
            tma_store_3d(&tmDV, smem + lay.zero + c * kTile * 2, c, t * kTile, bh);
          }
          tma_store_commit();
        }
      }
      if (MODE == MODE_STATE && D == 64 && p.zero_grads) tma_store_wait_all();
      // copies still in flight land before the CTA can leave
      for (int m = max(0, n - C::kSlots); m < n; ++m) mbar_drain(bar + B_FULL + m % C::kSlots, slot_par(m));
      if (FAVOR || (MODE == MODE_FWD && seg > 0)) mbar_drain(bar + B_SETUP, 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = true;
      auto wait = [&](int b, uint32_t par) {
        if (ok) ok = mbar_wait(bar + b, par, p.status, abort_flag);
        return ok;
      };
      constexpr uint32_t NV = D == 64 ? D + 16 : D;  // [V, 1] in one MMA when d = 64
      const uint32_t id_a = make_idesc(128, 128, false, false);
      const uint32_t id_n = make_idesc(128, D, false, true);
      const uint32_t id_nv = make_idesc(128, NV, false, true);
      const uint32_t id_s = make_idesc(128, 16, false, true);
      const uint32_t id_r = make_idesc(128, NV, true, true);
      const uint32_t id_r1 = make_idesc(128, 16, true, true);
      // [V, 1] as an MN-major operand: V's slot, then the ones block LBO bytes on
      auto desc_v1 = [&](uint32_t s_v, int s) {
        return make_desc(s_v, s_ones - s_v, 1024u, kSwizzle128) + (uint64_t)(s * 128u);
      };
      int job = 0, n = 0;
      // feature MMA into the next TMEM buffer: F = X W_h^T
      auto f_job = [&](uint32_t s_x, int h) {
        const int b = job_buf(job), u = job_use(job);
        if (u > 0 && !wait(B_FEMPTY + b, (u - 1) & 1)) return;
        tc_fence_after();
        const uint32_t idesc = make_idesc(128, min(128, M - 128 * h), false, false);
        for (int s = 0; s < D / 16; ++s)
          mma_bf16(tbase + t_buf(b), desc_kmajor(s_x, kTile, 0, s), desc_kmajor(s_w, M, 128 * h, s), idesc, s > 0);
        mma_commit(bar + B_FFULL + b);
        ++job;
      };
      // the epilogue's initial state (or zero totals) is in TMEM
      wait(B_RBFULL, 0);
      for (int i = 0; i < ntl && ok; ++i) {
        const int nK = n, nQ = n + 1, nV = n + C::kLoads - 1;
        n += C::kLoads;
        const uint32_t s_k = slot_addr(nK), s_q = slot_addr(nQ), s_v = slot_addr(nV);
        if (FAVOR) {
          if (!wait(B_FULL + nK % C::kSlots, slot_par(nK))) break;
          if (MODE == MODE_FWD && !wait(B_FULL + nQ % C::kSlots, slot_par(nQ))) break;
          tc_fence_after();
          for (int h = 0; h < nb && ok; ++h) {
            f_job(s_k, h);
            if (MODE == MODE_FWD) f_job(s_q, h);
          }
          if (!ok) break;
          mma_commit(bar + B_EMPTY + nK % C::kSlots);
          if (MODE == MODE_FWD) mma_commit(bar + B_EMPTY + nQ % C::kSlots);
        } else {
          // elu+1 features are formed from K and Q by the epilogue alone
          mbar_arrive(bar + B_EMPTY + nK % C::kSlots);
          if (MODE == MODE_FWD) mbar_arrive(bar + B_EMPTY + nQ % C::kSlots);
        }
        const int ja = job;  // the tile's A job
        const int gi = i % C::kGroup;  // state pass: position in the group
        for (int h = 0; h < nb && ok; ++h) {
          const uint32_t c = (uint32_t)(i * nb + h);
          if (!wait(B_PHK, c & 1)) break;
          if (h == 0) {
            if (!wait(B_FULL + nV % C::kSlots, slot_par(nV))) break;
            if (MODE == MODE_FWD && !wait(B_RBFULL, i & 1)) break;
            // the group partial restarts at zero once the epilogue has added it
            if (MODE == MODE_STATE && gi == 0 && i > 0 && !wait(B_RBFULL, (i / C::kGroup) & 1)) break;
          }
          tc_fence_after();
          // R'_h += phi_k,h^T [V, 1] (in place; the state pass restarts each group)
          const uint32_t t_r = tbase + lay.t_r + h * NC;
          for (int s = 0; s < kTile / 16; ++s) {
            const uint32_t acc = (MODE == MODE_FWD || gi > 0 || s > 0) ? 1u : 0u;
            if (D == 64) {
              mma_bf16(t_r, desc_mnmajor(s_phk, kTile, 0, s), desc_v1(s_v, s), id_r, acc);
            } else {
              mma_bf16(t_r, desc_mnmajor(s_phk, kTile, 0, s), desc_mnmajor(s_v, kTile, 0, s), id_r, acc);
              mma_bf16(t_r + D, desc_mnmajor(s_phk, kTile, 0, s), desc_n16(s_ones, s), id_r1, acc);
            }
          }
          if (MODE == MODE_FWD) {
            if (!wait(B_PHQ, c & 1)) break;
            if (h == 0) {
              const int u = job_use(ja);
              if (u > 0 && !wait(B_FEMPTY + job_buf(ja), (u - 1) & 1)) break;
              if (i > 0 && !wait(B_NUMEMPTY, (i - 1) & 1)) break;
            }
            tc_fence_after();
            const uint32_t t_a = tbase + t_buf(job_buf(ja));
            const int nu = min(128, M - 128 * h);
            for (int s = 0; s < nu / 16; ++s) {
              const uint32_t acc = (h > 0 || s > 0) ? 1u : 0u;
              const uint64_t aq = desc_kmajor(s_phq, kTile, 0, s);
              mma_bf16(t_a, aq, desc_kmajor(s_phk, kTile, 0, s), id_a, acc);
              mma_bf16(tbase + lay.t_num, aq, desc_mnmajor(s_rb, M, 0, 8 * h + s), id_n, acc);
            }
          }
          mma_commit(bar + B_PHFREE);
        }
        if (!ok) break;
        if (MODE == MODE_FWD) {
          // A fills its buffer like an F job: one phase of that buffer's barrier
          mma_commit(bar + B_FFULL + job_buf(ja));
          ++job;
          mma_commit(bar + B_AFULL);
          if (!wait(B_ATFULL, i & 1)) break;
          tc_fence_after();
          // num' += tril(A) [V, 1]
          for (int s = 0; s < kTile / 16; ++s) {
            const uint64_t aa = desc_kmajor(s_phq, kTile, 0, s);
            if (D == 64) {
              mma_bf16(tbase + lay.t_num, aa, desc_v1(s_v, s), id_nv, 1);
            } else {
              mma_bf16(tbase + lay.t_num, aa, desc_mnmajor(s_v, kTile, 0, s), id_n, 1);
              mma_bf16(tbase + lay.t_num + D, aa, desc_n16(s_ones, s), id_s, 1);
            }
          }
          mma_commit(bar + B_NUMFULL);
        }
        if (MODE == MODE_STATE && (gi == C::kGroup - 1 || i == ntl - 1)) mma_commit(bar + B_AFULL);
        mma_commit(bar + B_EMPTY + nV % C::kSlots);
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
    float *ss = reinterpret_cast<float *>(smem + lay.ss);
    float *denp = reinterpret_cast<float *>(smem + lay.denp);
    // columns [c_lo, c_hi) of R' block b handled by this thread: with two
    // blocks each half of the warps owns one, with one they split its columns
    const int csplit = ((NC / 16 + 1) / 2) * 16;
    auto r_cols = [&](int b, int &c_lo, int &c_hi) {
      if (nb == 2) {
        c_lo = 0;
        c_hi = b == half ? NC : 0;
      } else {
        c_lo = half ? csplit : 0;
        c_hi = half ? NC : csplit;
      }
    };
    auto put_rb = [&](int f, int c, const float *v) {
      if (f >= M) return;
#pragma unroll
      for (int i = 0; i < 16; i += 8)
        if (c + i + 8 <= D) st_bf16x8(s_rb + sw128_offset(f, c + i, M), v + i);
      if (c <= D && D < c + 16) ss[f] = v[D - c];
    };

    // the incoming state was placed in TMEM during set-up
    arrive(B_RBFULL);

    constexpr int FC = FAVOR ? 64 : D / 2;  // register columns of one phi half-row
    const int fcols = FAVOR ? FB / 2 : D / 2;
    auto store_phi = [&](uint32_t s_out, const float *v) {
#pragma unroll
      for (int j = 0; j < FC / 8; ++j)
        if (8 * j < fcols) st_bf16x8(s_out + sw128_offset(row, fcols * half + 8 * j, kTile), v + 8 * j);
    };
    int job = 0, n = 0;
    // the next F job from TMEM into registers; frees its buffer
    auto load_f = [&](float *v) {
      const int b = job_buf(job), u = job_use(job);
      if (!wait(B_FFULL + b, u & 1)) return;
      tc_fence_after();
      const uint32_t a = tmem_addr(tbase, lane_base, t_buf(b) + fcols * half);
      if (fcols == 64)
        tmem_ld32x2(a, a + 32, v, v + 32);
      else
        tmem_ld32(a, v);
      tc_fence_before();
      arrive(B_FEMPTY + b);
      ++job;
    };
    // phi of one half-row: FAVOR+ from the F job, elu+1 from the X tile
    auto make_phi = [&](uint32_t s_x, float c_row, bool dead, float *v) {
      if (FAVOR) {
        load_f(v);
#pragma unroll
        for (int x = 0; x < FC; ++x)
          if (x < fcols) v[x] = dead ? 0.f : favor_feature(v[x], c_row);
      } else {
#pragma unroll
        for (int j = 0; j < FC / 8; ++j) {
          ld_bf16x8(s_x + sw128_offset(row, FC * half + 8 * j, kTile), v + 8 * j);
#pragma unroll
          for (int x = 0; x < 8; ++x) v[8 * j + x] = dead ? 0.f : elu1_feature(v[8 * j + x]);
        }
      }
    };

    for (int i = 0; i < ntl && ok; ++i) {
      const int t = t0 + i;
      const int valid = min(kTile, p.L - t * kTile);
      const bool dead = row >= valid;  // padding rows past L: features forced to zero
      const int nK = n, nQ = n + 1, nV = n + C::kLoads - 1;
      n += C::kLoads;
      const uint32_t s_k = slot_addr(nK), s_q = slot_addr(nQ);
      if (!wait(B_FULL + nK % C::kSlots, slot_par(nK))) break;
      if (MODE == MODE_FWD && !wait(B_FULL + nQ % C::kSlots, slot_par(nQ))) break;
      float ck = 0.f, cq = 0.f;  // per-row exp2 offsets
      if (FAVOR) {
        ck = favor_row_const(tile_row_sqnorm(s_k, row, D), M);
        if (MODE == MODE_FWD) cq = favor_row_const(tile_row_sqnorm(s_q, row, D), M);
        arrive(B_EMPTY + nK % C::kSlots);
        if (MODE == MODE_FWD) arrive(B_EMPTY + nQ % C::kSlots);
      }
      float dpart = 0.f;  // phi_q . S(t-1) over this thread's features
      for (int h = 0; h < nb && ok; ++h) {
        const uint32_t c = (uint32_t)(i * nb + h);
        float v[FC];
        make_phi(s_k, ck, dead, v);
        if (c > 0 && !wait(B_PHFREE, (c - 1) & 1)) break;
        if (!ok) break;
        store_phi(s_phk, v);
        fence_async_smem();
        arrive(B_PHK);
        if (MODE == MODE_FWD) {
          make_phi(s_q, cq, dead, v);
          if (!ok) break;
#pragma unroll
          for (int x = 0; x < FC; ++x)
            if (x < fcols) dpart = fmaf(v[x], ss[128 * h + fcols * half + x], dpart);
          store_phi(s_phq, v);
          fence_async_smem();
          arrive(B_PHQ);
        }
      }
      if (!ok) break;
      if (MODE == MODE_FWD) denp[((i & 1) * 2 + half) * kTile + row] = dpart;
      if (!FAVOR) {
        arrive(B_EMPTY + nK % C::kSlots);
        if (MODE == MODE_FWD) arrive(B_EMPTY + nQ % C::kSlots);
      }
      if (MODE == MODE_STATE) {
        arrive(B_EMPTY + nV % C::kSlots);
        if (i % C::kGroup == C::kGroup - 1 || i == ntl - 1) {
          // master += this tile's increment (fp32; double-float for S)
          if (!wait(B_AFULL, (i / C::kGroup) & 1)) break;
          tc_fence_after();
          float *lo = reinterpret_cast<float *>(smem + lay.lo);
          for (int b = 0; b < nb; ++b) {
            int c_lo, c_hi;
            r_cols(b, c_lo, c_hi);
            const int f = 128 * b + row;
            for (int c = c_lo; c < c_hi; c += 16) {
              float x[16], m[16];
              tmem_ld16(tmem_addr(tbase, lane_base, lay.t_r + b * NC + c), x);
              tmem_ld16(tmem_addr(tbase, lane_base, lay.t_m + b * NC + c), m);
              const bool has_s = c <= D && D < c + 16;
              const float ms = has_s ? m[D - c] : 0.f, xs = has_s ? x[D - c] : 0.f;
#pragma unroll
              for (int e = 0; e < 16; ++e) m[e] += x[e];
              if (has_s && f < M) {
                float h = ms, l = lo[f * (D + 1) + D];
                df_add(h, l, xs);
                lo[f * (D + 1) + D] = l;
                m[D - c] = h;
              }
              tmem_st16(tmem_addr(tbase, lane_base, lay.t_m + b * NC + c), m);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          arrive(B_RBFULL);
        }
        continue;
      }
      // masked A (diagonal kept) -> bf16 into the phi_q buffer
      {
        if (!wait(B_AFULL, i & 1)) break;
        tc_fence_after();
        const int b = job_buf(job);
        float v[64];
        const uint32_t a = tmem_addr(tbase, lane_base, t_buf(b) + 64 * half);
        tmem_ld32x2(a, a + 32, v, v + 32);
        tc_fence_before();
        arrive(B_FEMPTY + b);
        ++job;
#pragma unroll
        for (int x = 0; x < 64; ++x)
          if (64 * half + x > row) v[x] = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) st_bf16x8(s_phq + sw128_offset(row, 64 * half + 8 * j, kTile), v + 8 * j);
        if (half == 0) {
          // num' columns d .. d+15 restart at zero: both halves read them
          // last tile, before either could get here
          float z[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) z[x] = 0.f;
          tmem_st16(tmem_addr(tbase, lane_base, lay.t_num + D), z);
          tmem_st_wait();
          tc_fence_before();
        }
        fence_async_smem();
        arrive(B_ATFULL);
      }
      // bf16 copies of R(t) for the next tile
      for (int b = 0; b < nb; ++b) {
        int c_lo, c_hi;
        r_cols(b, c_lo, c_hi);
        const int f = 128 * b + row;
        for (int c = c_lo; c < c_hi; c += 16) {
          float v[16];
          tmem_ld16(tmem_addr(tbase, lane_base, lay.t_r + b * NC + c), v);
          put_rb(f, c, v);
        }
      }
      fence_async_smem();
      tc_fence_before();
      arrive(B_RBFULL);
      arrive(B_EPI);  // this warp's S(t) and den partials are in shared memory
      // Y = num / den
      {
        if (!wait(B_NUMFULL, i & 1)) break;
        tc_fence_after();
        constexpr int YC = D / 2;  // value columns per thread
        float dv[16], v[YC];
        tmem_ld16(tmem_addr(tbase, lane_base, lay.t_num + D), dv);
        const uint32_t a = tmem_addr(tbase, lane_base, lay.t_num + YC * half);
        if constexpr (YC == 64)
          tmem_ld32x2(a, a + 32, v, v + 32);
        else
          tmem_ld32(a, v);
        tc_fence_before();
        arrive(B_NUMEMPTY);
        if (!wait(B_EPI, i & 1)) break;
        if (!dead) {
          const float inv =
              1.0f / (dv[0] + denp[((i & 1) * 2) * kTile + row] + denp[((i & 1) * 2 + 1) * kTile + row]);
          uint4 *dst = reinterpret_cast<uint4 *>(p.y + ((size_t)bh * p.L + (size_t)t * kTile + row) * D + YC * half);
#pragma unroll
          for (int j = 0; j < YC / 8; ++j)
            dst[j] = make_uint4(pack_bf16(v[8 * j] * inv, v[8 * j + 1] * inv),
                                pack_bf16(v[8 * j + 2] * inv, v[8 * j + 3] * inv),
                                pack_bf16(v[8 * j + 4] * inv, v[8 * j + 5] * inv),
                                pack_bf16(v[8 * j + 6] * inv, v[8 * j + 7] * inv));
        }
        arrive(B_EMPTY + nV % C::kSlots);
      }
    }

    if (MODE == MODE_STATE && ok) {
      // segment total of R' -> fp32 [M][D + 1] staged in the idle load slots
      // (and phi_k tile) for one coalesced bulk store after the final barrier
      float *stage = reinterpret_cast<float *>(smem + lay.slots);
      for (int b = 0; b < nb; ++b) {
        int c_lo, c_hi;
        r_cols(b, c_lo, c_hi);
        const int f = 128 * b + row;
        for (int c = c_lo; c < c_hi; c += 16) {
          float v[16];
          tmem_ld16(tmem_addr(tbase, lane_base, lay.t_m + b * NC + c), v);
          if (f < M) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              if (c + i <= D) stage[f * DP + c + i] = v[i];
          }
        }
      }
      fence_async_smem();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (MODE == MODE_STATE && tid == 0 && !*abort_flag) {
    const size_t off = ((size_t)bh * p.P + seg) * (size_t)M * DP;
    bulk_store(p.states + off, sbase + lay.slots, (uint32_t)(M * DP * 4));
    bulk_store(p.states_lo + off, sbase + lay.lo, (uint32_t)(M * DP * 4));
    tma_store_commit();
    tma_store_wait_read();
  }
  if (warp == 0) tmem_dealloc(tbase, 512);
}

template <int D, bool FAVOR, int MODE, int M>
cudaError_t launch_m(const Plan &pl, const Args &a, const CUtensorMap &mq, const CUtensorMap &mk,
                     const CUtensorMap &mv, const CUtensorMap *mz, int nseg, cudaStream_t st) {
  Params p{};
  p.L = pl.L; p.M = pl.M; p.nt = pl.tc_tiles; p.P = pl.P; p.tps = pl.cps;
  p.zero_grads = mz != nullptr;
  p.y = static_cast<__nv_bfloat16 *>(a.y);
  p.wimg = reinterpret_cast<const __nv_bfloat16 *>(a.ws + pl.wimg_off);
  p.states = a.ws + pl.states_off;
  p.states_lo = a.ws + pl.states_lo_off;
  p.status = a.status;
  const Layout<D, FAVOR, MODE> lay(M);
  const int smem = (int)lay.total + 1024;
  auto kern = tc_fwd_kernel<D, FAVOR, MODE, M>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(nseg, pl.BH), kThreads, smem, st>>>(mq, mk, mv, mz ? mz[0] : mk, mz ? mz[1] : mk, mz ? mz[2] : mk, p);
  return cudaGetLastError();
}

// M is a compile-time constant of the kernel: FAVOR+ with 64, 128 or 256
// features, elu+1 with M = d.
template <int D, bool FAVOR, int MODE>
cudaError_t launch(const Plan &pl, const Args &a, const CUtensorMap &mq, const CUtensorMap &mk,
                   const CUtensorMap &mv, const CUtensorMap *mz, int nseg, cudaStream_t st) {
  if constexpr (!FAVOR) {
    return pl.M == D ? launch_m<D, FAVOR, MODE, D>(pl, a, mq, mk, mv, mz, nseg, st) : cudaErrorInvalidValue;
  } else {
    if (pl.M == 64) return launch_m<D, FAVOR, MODE, 64>(pl, a, mq, mk, mv, mz, nseg, st);
    if (pl.M == 128) return launch_m<D, FAVOR, MODE, 128>(pl, a, mq, mk, mv, mz, nseg, st);
    if (pl.M == 256) return launch_m<D, FAVOR, MODE, 256>(pl, a, mq, mk, mv, mz, nseg, st);
    return cudaErrorInvalidValue;
  }
}

// W (fp32 [64][M]) -> the bf16 [M][64] swizzled image of W^T that the
// kernels copy into shared memory as the K-major B operand of F = X W.
__global__ void prep_w_kernel(const float *__restrict__ w, __nv_bfloat16 *__restrict__ img, int M) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= M * 64) return;
  const int i = idx / M, m = idx - i * M;
  img[sw128_offset(m, i, M) / 2] = __float2bfloat16_rn(w[idx]);
}

cudaError_t prep_w(const Plan &pl, const Args &a, cudaStream_t st) {
  if (!pl.favor) return cudaSuccess;
  ProfScope ps("prep_w", st);
  const int n = pl.M * 64;
  prep_w_kernel<<<(n + 255) / 256, 256, 0, st>>>(a.w, reinterpret_cast<__nv_bfloat16 *>(a.ws + pl.wimg_off), pl.M);
  return cudaGetLastError();
}

// Totals of R' over the first nseg segments, then their inclusive scan:
// states[s] = R' at the end of segment s.
template <int D, bool FAVOR>
cudaError_t segment_states(const Plan &pl, const Args &a, const CUtensorMap &mq,
                           const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap *mz, int nseg,
                           cudaStream_t st) {
  cudaError_t e;
  {
    ProfScope ps("tc_segment_state", st);
    e = launch<D, FAVOR, MODE_STATE>(pl, a, mq, mk, mv, mz, nseg, st);
    if (e != cudaSuccess) return e;
  }
  if (nseg > 1) {
    ProfScope ps("scan_states", st);
    e = scan_states_df(pl, a.ws + pl.states_off, a.ws + pl.states_lo_off, nseg, 1, st);
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
    e = segment_states<D, FAVOR>(pl, a, mq, mk, mv, nullptr, pl.P - 1, st);
    if (e != cudaSuccess) return e;
  }
  ProfScope ps("tc_forward", st);
  return launch<D, FAVOR, MODE_FWD>(pl, a, mq, mk, mv, nullptr, pl.P, st);
}

}  // namespace tcf

size_t tc_smem_bytes(int d, int M, bool favor) {
  if (d == 64 && favor) return tcf::Layout<64, true, tcf::MODE_FWD>(M).total + 1024;
  if (d == 64) return tcf::Layout<64, false, tcf::MODE_FWD>(M).total + 1024;
  return tcf::Layout<128, false, tcf::MODE_FWD>(M).total + 1024;
}

bool tc_forward_supported(int d, int M, int chunk, bool favor) {
  if (chunk < 64) return false;
  if (d == 64) return favor ? (M == 64 || M == 128 || M == 256) : M == 64;
  if (d == 128) return !favor && M == 128;
  return false;
}

cudaError_t tc_segment_states(const Plan &p, const Args &a, int nseg, bool zero_grads, cudaStream_t st) {
  CUtensorMap mk, mv, mz[3];
  const int d = p.d;
  cudaError_t e = tcf::prep_w(p, a, st);
  if (e != cudaSuccess) return e;
  if (!make_map_bf16_3d(&mk, a.k, p.BH, p.L, d, tcf::kTile) || !make_map_bf16_3d(&mv, a.v, p.BH, p.L, d, tcf::kTile))
    return cudaErrorInvalidValue;
  if (zero_grads &&
      (!make_map_bf16_3d(&mz[0], a.dq, p.BH, p.L, d, tcf::kTile) ||
       !make_map_bf16_3d(&mz[1], a.dk, p.BH, p.L, d, tcf::kTile) ||
       !make_map_bf16_3d(&mz[2], a.dv, p.BH, p.L, d, tcf::kTile)))
    return cudaErrorInvalidValue;
  const CUtensorMap *z = zero_grads ? mz : nullptr;
  if (d == 64 && p.favor) return tcf::segment_states<64, true>(p, a, mk, mk, mv, z, nseg, st);
  if (d == 64) return tcf::segment_states<64, false>(p, a, mk, mk, mv, z, nseg, st);
  if (d == 128 && !p.favor) return tcf::segment_states<128, false>(p, a, mk, mk, mv, z, nseg, st);
  return cudaErrorInvalidValue;
}

cudaError_t tc_forward(const Plan &p, const Args &a, cudaStream_t st) {
  cudaError_t e = tcf::prep_w(p, a, st);
  if (e != cudaSuccess) return e;
  if (p.d == 64 && p.favor) return tcf::forward_family<64, true>(p, a, st);
  if (p.d == 64) return tcf::forward_family<64, false>(p, a, st);
  if (p.d == 128 && !p.favor) return tcf::forward_family<128, false>(p, a, st);
  return cudaErrorInvalidValue;
}

}  // namespace slim
