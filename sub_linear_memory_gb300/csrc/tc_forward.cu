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
//   warps 2-9   epilogue: kParts = 2 threads per row, each half of the
//               columns (16 warps spill at M = 256 under the 96-register cap
//               of 576 threads and measured slower).
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
constexpr int kParts = kEpiWarps / 4;  // epilogue threads per row
constexpr int kThreads = 32 * (2 + kEpiWarps);

// n consecutive fp32 TMEM columns of this thread's lane (n = 16, 32 or 64)
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t a, float *v) {
  if constexpr (N == 16) {
    tmem_ld16(a, v);
  } else if constexpr (N == 32) {
    tmem_ld32(a, v);
  } else {
    static_assert(N == 64, "16, 32 or 64 columns");
    tmem_ld32x2(a, a + 32, v, v + 32);
  }
}

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
    denp = o; o += MODE == MODE_FWD ? 2u * kParts * kTile * 4u : 0u;  // [tile parity][part][row]
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
    const int q4 = warp & 3, part = (warp - 2) >> 2, row = 32 * q4 + lane;
    const uint32_t t_dst = MODE == MODE_FWD ? lay.t_r : lay.t_m;
    if (warp >= 2) {
      // 16-column chunks of the nb state blocks, dealt out over the parts
      constexpr int NCH = NC / 16;
      for (int k = part; k < nb * NCH; k += kParts) {
        const int b = k / NCH, c = (k - b * NCH) * 16, f = 128 * b + row;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = (in && f < M && c + i <= D) ? stage[f * DP + c + i] : 0.f;
        tmem_st16(tmem_addr(tbase, 32u * q4, t_dst + b * NC + c), v);
        if (MODE == MODE_FWD && f < M) {
#pragma unroll
          for (int i = 0; i < 16; i += 8)
            if (c + i + 8 <= D) st_bf16x8(sbase + lay.rb + sw128_offset(f, c + i, M), v + i);
          if (c == D) reinterpret_cast<float *>(smem + lay.ss)[f] = v[0];  // S opens chunk c = d
        }
      }
      tmem_st_wait();
    }
    // num' columns d .. d+15 start at zero (only the ones product adds there)
    if (MODE == MODE_FWD && warp >= 2 && part == 0) {
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
      // R'_h += phi_k,h^T [V, 1]; the forward accumulates in place, the state
      // pass restarts each tile's increment at zero
      auto issue_r = [&](int h, uint32_t s_v, bool fresh) {
        const uint32_t t_r = tbase + lay.t_r + h * NC;
        for (int s = 0; s < kTile / 16; ++s) {
          const uint32_t acc = (fresh && s == 0) ? 0u : 1u;
          if (D == 64) {
            mma_bf16(t_r, desc_mnmajor(s_phk, kTile, 0, s), desc_v1(s_v, s), id_r, acc);
          } else {
            mma_bf16(t_r, desc_mnmajor(s_phk, kTile, 0, s), desc_mnmajor(s_v, kTile, 0, s), id_r, acc);
            mma_bf16(t_r + D, desc_mnmajor(s_phk, kTile, 0, s), desc_n16(s_ones, s), id_r1, acc);
          }
        }
      };
      // feature MMA F = X W_h^T into TMEM buffer b; `uses` counts the jobs
      // issued on each buffer, whose previous job must have been read out
      int uses0 = 0, uses1 = 0;
      auto f_job = [&](uint32_t s_x, int h, int b) {
        int &u = b ? uses1 : uses0;
        if (u > 0 && !wait(B_FEMPTY + b, (u - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t idesc = make_idesc(128, min(128, M - 128 * h), false, false);
        for (int s = 0; s < D / 16; ++s)
          mma_bf16(tbase + t_buf(b), desc_kmajor(s_x, kTile, 0, s), desc_kmajor(s_w, M, 128 * h, s), idesc, s > 0);
        mma_commit(bar + B_FFULL + b);
        ++u;
        return true;
      };
      // the epilogue's initial state (or zero totals) is in TMEM
      wait(B_RBFULL, 0);
      if constexpr (MODE == MODE_FWD) {
        // Buffer plan (FAVOR+): buffer 0 carries phi_k,0(t), phi_k,1(t),
        // phi_q,1(t), phi_k,0(t+1), ...; buffer 1 carries phi_q,0(t) and then
        // the tile's A, which therefore never waits for a feature job.  The
        // epilogue finishes tile t-1 (mask, R copy, Y) between phi_k,0(t) and
        // phi_q,0(t), so the issue order below follows that.
        static_assert(nb <= 2, "at most 256 features");
        constexpr int bA = C::kNbuf > 1 ? 1 : 0;  // A's TMEM buffer
        auto slot_wait = [&](int n) { return wait(B_FULL + n % C::kSlots, slot_par(n)); };
        auto empty = [&](int n) { mma_commit(bar + B_EMPTY + n % C::kSlots); };
        // num' += tril(A) [V, 1] for the tile whose masked A is in phi_q's buffer
        auto issue_av = [&](uint32_t s_v) {
          for (int s = 0; s < kTile / 16; ++s) {
            const uint64_t aa = desc_kmajor(s_phq, kTile, 0, s);
            if (D == 64) {
              mma_bf16(tbase + lay.t_num, aa, desc_v1(s_v, s), id_nv, 1);
            } else {
              mma_bf16(tbase + lay.t_num, aa, desc_mnmajor(s_v, kTile, 0, s), id_n, 1);
              mma_bf16(tbase + lay.t_num + D, aa, desc_n16(s_ones, s), id_s, 1);
            }
          }
        };
        // A += phi_q,h phi_k,h^T and num += phi_q,h R_h^T
        auto issue_anum = [&](int h) {
          const uint32_t t_a = tbase + t_buf(bA);
          const int nu = min(128, M - 128 * h);
          for (int s = 0; s < nu / 16; ++s) {
            const uint32_t acc = (h > 0 || s > 0) ? 1u : 0u;
            const uint64_t aq = desc_kmajor(s_phq, kTile, 0, s);
            mma_bf16(t_a, aq, desc_kmajor(s_phk, kTile, 0, s), id_a, acc);
            mma_bf16(tbase + lay.t_num, aq, desc_mnmajor(s_rb, M, 0, 8 * h + s), id_n, acc);
          }
        };
        if (FAVOR && ntl > 0 && slot_wait(0) && slot_wait(1)) {
          f_job(slot_addr(0), 0, 0);
          if (nb == 1) empty(0);
          f_job(slot_addr(1), 0, 1);
          if (nb == 1) empty(1);
        }
        for (int i = 0; i < ntl && ok; ++i) {
          const int nK = 3 * i, nQ = nK + 1, nV = nK + 2;
          const uint32_t s_k = slot_addr(nK), s_q = slot_addr(nQ), s_v = slot_addr(nV);
          const uint32_t c = (uint32_t)(i * nb);
          if (FAVOR && nb > 1) {
            if (!f_job(s_k, 1, 0)) break;  // phi_k,1(t)
            empty(nK);
          }
          if (!FAVOR) {
            // elu+1 features are formed from K and Q by the epilogue alone
            mbar_arrive(bar + B_EMPTY + nK % C::kSlots);
            mbar_arrive(bar + B_EMPTY + nQ % C::kSlots);
          }
          if (i > 0) {
            // phi_q,0(t) once the mask of tile t-1 has read A out of buffer 1
            if (FAVOR) {
              if (!slot_wait(nQ) || !f_job(s_q, 0, 1)) break;
              if (nb == 1) empty(nQ);
            }
            // num'(t-1) += tril(A(t-1)) [V(t-1), 1]
            if (!wait(B_ATFULL, (i - 1) & 1)) break;
            tc_fence_after();
            issue_av(slot_addr(nV - 3));
            mma_commit(bar + B_NUMFULL);
            empty(nV - 3);
          }
          // block 0: R'_0 += ..., once R(t-1) has been copied out of TMEM
          if (!wait(B_PHK, c & 1) || !slot_wait(nV) || !wait(B_RBFULL, i & 1)) break;
          tc_fence_after();
          issue_r(0, s_v, false);
          if (FAVOR && nb == 1 && i + 1 < ntl) {
            // phi_k,0(t+1) ahead of A: buffer 0 is free once phi_k,0(t) is read
            if (!slot_wait(nK + 3) || !f_job(slot_addr(nK + 3), 0, 0)) break;
            empty(nK + 3);
          }
          if (!wait(B_PHQ, c & 1) || (i > 0 && !wait(B_NUMEMPTY, (i - 1) & 1))) break;
          {
            int &u = bA ? uses1 : uses0;
            if (u > 0 && !wait(B_FEMPTY + bA, (u - 1) & 1)) break;
          }
          tc_fence_after();
          issue_anum(0);
          mma_commit(bar + B_PHFREE);
          for (int h = 1; h < nb && ok; ++h) {
            if (!f_job(s_q, h, 0)) break;  // phi_q,1(t)
            empty(nQ);
            if (!wait(B_PHK, (c + h) & 1)) break;
            tc_fence_after();
            issue_r(h, s_v, false);
            if (i + 1 < ntl) {
              // phi_k,0(t+1) ahead of the last A block
              if (!slot_wait(nK + 3) || !f_job(slot_addr(nK + 3), 0, 0)) break;
            }
            if (!wait(B_PHQ, (c + h) & 1)) break;
            tc_fence_after();
            issue_anum(h);
            mma_commit(bar + B_PHFREE);
          }
          if (!ok) break;
          // A(t) complete: one phase of its buffer, like a feature job
          mma_commit(bar + B_FFULL + bA);
          ++(bA ? uses1 : uses0);
        }
        if (ok && ntl > 0 && wait(B_ATFULL, (ntl - 1) & 1)) {
          tc_fence_after();
          issue_av(slot_addr(3 * (ntl - 1) + 2));
          mma_commit(bar + B_NUMFULL);
          empty(3 * (ntl - 1) + 2);
        }
      } else {
        int n = 0;
        for (int i = 0; i < ntl && ok; ++i) {
          const int nK = n, nV = n + 1;
          n += C::kLoads;
          const uint32_t s_k = slot_addr(nK), s_v = slot_addr(nV);
          if (FAVOR) {
            if (!wait(B_FULL + nK % C::kSlots, slot_par(nK))) break;
            tc_fence_after();
            for (int h = 0; h < nb && ok; ++h) f_job(s_k, h, 0);
            if (!ok) break;
            mma_commit(bar + B_EMPTY + nK % C::kSlots);
          } else {
            mbar_arrive(bar + B_EMPTY + nK % C::kSlots);
          }
          for (int h = 0; h < nb && ok; ++h) {
            const uint32_t c = (uint32_t)(i * nb + h);
            if (!wait(B_PHK, c & 1)) break;
            if (h == 0) {
              if (!wait(B_FULL + nV % C::kSlots, slot_par(nV))) break;
              // the tile's increment restarts at zero once the epilogue has added the last
              if (i > 0 && !wait(B_RBFULL, i & 1)) break;
            }
            tc_fence_after();
            issue_r(h, s_v, true);
            mma_commit(bar + B_PHFREE);
          }
          if (!ok) break;
          mma_commit(bar + B_AFULL);
          mma_commit(bar + B_EMPTY + nV % C::kSlots);
        }
      }
      mma_commit(bar + B_DONE);
      mbar_drain(bar + B_DONE, 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q4 = warp & 3, part = (warp - 2) >> 2, row = 32 * q4 + lane;
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
    // R' state chunks (16 columns of one block) handled by this thread:
    // chunk k = part, part + kParts, ... of the nb * NC / 16
    constexpr int NCH = NC / 16;
    auto put_rb = [&](int f, int c, const float *v) {
      if (f >= M) return;
#pragma unroll
      for (int i = 0; i < 16; i += 8)
        if (c + i + 8 <= D) st_bf16x8(s_rb + sw128_offset(f, c + i, M), v + i);
      if (c == D) ss[f] = v[0];
    };

    // the incoming state was placed in TMEM during set-up
    arrive(B_RBFULL);

    constexpr int FC = (FAVOR ? FB : D) / kParts;  // phi columns of this thread
    auto store_phi = [&](uint32_t s_out, const float *v) {
#pragma unroll
      for (int j = 0; j < FC / 8; ++j) st_bf16x8(s_out + sw128_offset(row, FC * part + 8 * j, kTile), v + 8 * j);
    };
    // per-buffer counts of the TMEM jobs read out so far
    int got0 = 0, got1 = 0;
    // the next job of TMEM buffer b (FC columns of this thread) into registers; frees the buffer
    auto load_f = [&](int b, float *v) {
      int &u = b ? got1 : got0;
      if (!wait(B_FFULL + b, u & 1)) return;
      tc_fence_after();
      tmem_ldn<FC>(tmem_addr(tbase, lane_base, t_buf(b) + FC * part), v);
      tc_fence_before();
      arrive(B_FEMPTY + b);
      ++u;
    };
    // phi of this thread's columns: FAVOR+ from the F job in buffer b, elu+1 from the X tile
    auto make_phi = [&](int b, uint32_t s_x, float c_row, bool dead, float *v) {
      if (FAVOR) {
        load_f(b, v);
#pragma unroll
        for (int x = 0; x < FC; ++x) v[x] = dead ? 0.f : favor_feature(v[x], c_row);
      } else {
#pragma unroll
        for (int j = 0; j < FC / 8; ++j) {
          ld_bf16x8(s_x + sw128_offset(row, FC * part + 8 * j, kTile), v + 8 * j);
#pragma unroll
          for (int x = 0; x < 8; ++x) v[8 * j + x] = dead ? 0.f : elu1_feature(v[8 * j + x]);
        }
      }
    };

    if constexpr (MODE == MODE_FWD) {
      constexpr int bA = C::kNbuf > 1 ? 1 : 0;  // A's TMEM buffer (see the MMA issuer)
      // Finish tile j: masked A to bf16 (A's operand buffer), the bf16 copy of
      // R(j) for the next tile's num MMAs, then Y(j) = num / den.  Runs after
      // phi_k,0 of tile j + 1, once the MMAs that read tile j's last feature
      // block (hence A(j) and R(j)) are done.
      auto finish = [&](int j, bool refresh) {
        // masked A (diagonal kept) -> bf16 into the phi_q buffer
        {
          int &u = bA ? got1 : got0;
          if (!wait(B_FFULL + bA, u & 1)) return false;
          tc_fence_after();
          constexpr int AC = kTile / kParts;  // A columns of this thread, 32 at a time
#pragma unroll 1
          for (int c0 = AC * part; c0 < AC * (part + 1); c0 += 32) {
            float v[32];
            tmem_ld32(tmem_addr(tbase, lane_base, t_buf(bA) + c0), v);
#pragma unroll
            for (int x = 0; x < 32; ++x)
              if (c0 + x > row) v[x] = 0.f;
#pragma unroll
            for (int k = 0; k < 4; ++k) st_bf16x8(s_phq + sw128_offset(row, c0 + 8 * k, kTile), v + 8 * k);
          }
          tc_fence_before();
          arrive(B_FEMPTY + bA);
          ++u;
          if (part == 0) {
            // num' columns d .. d+15 restart at zero; every part read them for
            // Y(j-1) before the num MMAs of tile j, hence before this point
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
        // bf16 copies of R(j) and fp32 S(j) for tile j + 1
        if (refresh) {
          for (int k = part; k < nb * NCH; k += kParts) {
            const int b = k / NCH, c = (k - b * NCH) * 16;
            float v[16];
            tmem_ld16(tmem_addr(tbase, lane_base, lay.t_r + b * NC + c), v);
            put_rb(128 * b + row, c, v);
          }
          fence_async_smem();
          tc_fence_before();
          arrive(B_RBFULL);
        }
        arrive(B_EPI);  // this warp's S(j) and den partials of tile j are in shared memory
        // Y = num / den
        if (!wait(B_NUMFULL, j & 1)) return false;
        tc_fence_after();
        constexpr int YC = D / kParts;  // value columns per thread
        float v[YC];
        const float rowsum_a = tmem_ld1(tmem_addr(tbase, lane_base, lay.t_num + D));
        tmem_ldn<YC>(tmem_addr(tbase, lane_base, lay.t_num + YC * part), v);
        tc_fence_before();
        arrive(B_NUMEMPTY);
        if (!wait(B_EPI, j & 1)) return false;
        const int tj = t0 + j;
        if (row < min(kTile, p.L - tj * kTile)) {
          float den = rowsum_a;
#pragma unroll
          for (int q = 0; q < kParts; ++q) den += denp[((j & 1) * kParts + q) * kTile + row];
          const float inv = 1.0f / den;
          uint4 *dst = reinterpret_cast<uint4 *>(p.y + ((size_t)bh * p.L + (size_t)tj * kTile + row) * D + YC * part);
#pragma unroll
          for (int k = 0; k < YC / 8; ++k)
            dst[k] = make_uint4(pack_bf16(v[8 * k] * inv, v[8 * k + 1] * inv),
                                pack_bf16(v[8 * k + 2] * inv, v[8 * k + 3] * inv),
                                pack_bf16(v[8 * k + 4] * inv, v[8 * k + 5] * inv),
                                pack_bf16(v[8 * k + 6] * inv, v[8 * k + 7] * inv));
        }
        arrive(B_EMPTY + (3 * j + 2) % C::kSlots);  // V(j)
        return true;
      };

      for (int i = 0; i < ntl && ok; ++i) {
        const int t = t0 + i;
        const bool dead = row >= min(kTile, p.L - t * kTile);  // padding rows past L: features forced to zero
        const int nK = 3 * i, nQ = nK + 1;
        const uint32_t s_k = slot_addr(nK), s_q = slot_addr(nQ);
        if (!wait(B_FULL + nK % C::kSlots, slot_par(nK))) break;
        if (!wait(B_FULL + nQ % C::kSlots, slot_par(nQ))) break;
        float ck = 0.f, cq = 0.f;  // per-row exp2 offsets
        if (FAVOR) {
          ck = favor_row_const(tile_row_sqnorm(s_k, row, D), M);
          cq = favor_row_const(tile_row_sqnorm(s_q, row, D), M);
          arrive(B_EMPTY + nK % C::kSlots);
          arrive(B_EMPTY + nQ % C::kSlots);
        }
        float dpart[4] = {0.f, 0.f, 0.f, 0.f};  // phi_q . S(t-1) over this thread's features
#pragma unroll 1
        for (int h = 0; h < nb && ok; ++h) {
          const uint32_t c = (uint32_t)(i * nb + h);
          float v[FC];
          make_phi(0, s_k, ck, dead, v);
          if (c > 0 && !wait(B_PHFREE, (c - 1) & 1)) break;
          store_phi(s_phk, v);
          fence_async_smem();
          arrive(B_PHK);
          if (!FAVOR && h == nb - 1) arrive(B_EMPTY + nK % C::kSlots);
          if (h == 0 && i > 0 && !finish(i - 1, true)) break;
          make_phi(h == 0 ? (FAVOR ? 1 : 0) : 0, s_q, cq, dead, v);
          if (!ok) break;
#pragma unroll
          for (int x = 0; x < FC; ++x) dpart[x & 3] = fmaf(v[x], ss[128 * h + FC * part + x], dpart[x & 3]);
          store_phi(s_phq, v);
          fence_async_smem();
          arrive(B_PHQ);
          if (!FAVOR && h == nb - 1) arrive(B_EMPTY + nQ % C::kSlots);
        }
        if (!ok) break;
        denp[((i & 1) * kParts + part) * kTile + row] = (dpart[0] + dpart[1]) + (dpart[2] + dpart[3]);
      }
      if (ok && ntl > 0 && wait(B_PHFREE, (uint32_t)(ntl * nb - 1) & 1)) finish(ntl - 1, false);
    } else {
      int n = 0;
      for (int i = 0; i < ntl && ok; ++i) {
        const int t = t0 + i;
        const bool dead = row >= min(kTile, p.L - t * kTile);
        const int nK = n, nV = n + 1;
        n += C::kLoads;
        const uint32_t s_k = slot_addr(nK);
        if (!wait(B_FULL + nK % C::kSlots, slot_par(nK))) break;
        float ck = 0.f;
        if (FAVOR) {
          ck = favor_row_const(tile_row_sqnorm(s_k, row, D), M);
          arrive(B_EMPTY + nK % C::kSlots);
        }
        for (int h = 0; h < nb && ok; ++h) {
          const uint32_t c = (uint32_t)(i * nb + h);
          float v[FC];
          make_phi(0, s_k, ck, dead, v);
          if (c > 0 && !wait(B_PHFREE, (c - 1) & 1)) break;
          if (!ok) break;
          store_phi(s_phk, v);
          fence_async_smem();
          arrive(B_PHK);
        }
        if (!ok) break;
        if (!FAVOR) arrive(B_EMPTY + nK % C::kSlots);
        arrive(B_EMPTY + nV % C::kSlots);
        // master += this tile's increment (fp32; double-float for S)
        if (!wait(B_AFULL, i & 1)) break;
        tc_fence_after();
        float *lo = reinterpret_cast<float *>(smem + lay.lo);
        for (int k = part; k < nb * NCH; k += kParts) {
          const int b = k / NCH, c = (k - b * NCH) * 16, f = 128 * b + row;
          float x[16], m[16];
          tmem_ld16(tmem_addr(tbase, lane_base, lay.t_r + b * NC + c), x);
          tmem_ld16(tmem_addr(tbase, lane_base, lay.t_m + b * NC + c), m);
          const bool has_s = c == D;  // S is column 0 of chunk c = d
          const float ms = m[0], xs = x[0];
#pragma unroll
          for (int e = 0; e < 16; ++e) m[e] += x[e];
          if (has_s && f < M) {
            float hs = ms, l = lo[f * (D + 1) + D];
            df_add(hs, l, xs);
            lo[f * (D + 1) + D] = l;
            m[0] = hs;
          }
          tmem_st16(tmem_addr(tbase, lane_base, lay.t_m + b * NC + c), m);
        }
        tmem_st_wait();
        tc_fence_before();
        arrive(B_RBFULL);
      }
    }

    if (MODE == MODE_STATE && ok) {
      // segment total of R' -> fp32 [M][D + 1] staged in the idle load slots
      // (and phi_k tile) for one coalesced bulk store after the final barrier
      float *stage = reinterpret_cast<float *>(smem + lay.slots);
      for (int k = part; k < nb * NCH; k += kParts) {
        const int b = k / NCH, c = (k - b * NCH) * 16, f = 128 * b + row;
        float v[16];
        tmem_ld16(tmem_addr(tbase, lane_base, lay.t_m + b * NC + c), v);
        if (f < M) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c + i <= D) stage[f * DP + c + i] = v[i];
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

// ============================================================================
// Forward with role-specialised epilogue warpgroups.
//
// The serial epilogue above (one warp set walking phi_k, phi_q, the mask, the
// R copy and Y in turn) ran at about a third of the issue rate: each step
// waited on the one before it.  Here every step has warps of its own and the
// three epilogue warpgroups run concurrently, one thread per row (TMEM lane),
// walking columns in 32- or 64-wide chunks so that 128 registers suffice:
//   warp 0       TMA producer (K, Q, V ring);
//   warps 1, 2   K-side and Q-side feature MMAs F = X W (one thread each);
//   warp 3       the other MMAs, whichever is ready first: R'_h += phi_k,h^T
//                [V, 1], the A/num blocks, tril(A) [V, 1];
//   warps 4-7    phi_k blocks;
//   warps 8-11   phi_q blocks and den partials phi_q . S(t-1);
//   warps 12-15  the tile's tail: bf16 copy of R(t), masked A, Y = num/den.
// tcgen05.mma issue blocks for about the MMA's duration and each issuing
// warp shares its scheduler with three epilogue warps, so three issuing
// threads on three schedulers, each with few barriers to watch, keep the
// tensor pipe fed where one thread polling every barrier did not.
// Feature jobs are 64 features wide, one TMEM buffer per side, so A keeps a
// buffer of its own (TMEM at M = 256: F_k 64 | F_q 64 | A 128 | num' 80 |
// R' 2 x 80 of 512 columns).
namespace fw {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;

enum {
  F_FULL = 0,      // [4] slot loaded
  F_EMPTY = 4,     // [4] slot free: MMA commit + 4 consumer warps
  F_KJFULL = 12,   // K-side feature job in TMEM
  F_KJEMPTY = 13,  // ... read out (4 warps)
  F_QJFULL = 14,
  F_QJEMPTY = 15,
  F_PHK = 16,      // phi_k block stored (4 warps)
  F_PHQ = 17,      // phi_q block stored (4 warps)
  F_KFREE = 18,    // MMAs reading the phi_k buffer done
  F_QFREE = 19,    // MMAs reading the phi_q buffer done
  F_AFULL = 20,    // A and R' of the tile complete
  F_RBFULL = 21,   // R(t) and S(t) copied to shared memory (phase 0: incoming state)
  F_ATFULL = 23,   // masked A packed in TMEM (4 warps)
  F_NUMFULL = 24,  // num' complete
  F_NUMEMPTY = 25, // num' read out (4 warps)
  F_DEN = 26,      // [2] den partials of tile parity 0 / 1 (4 warps)
  F_SETUP = 28,
  F_DONE = 29,     // [3] MMA drain of each issuing thread
  F_COUNT = 32
};

template <int D, bool FAVOR, int M>
struct FwdLayout {
  static constexpr int kSlots = D == 128 ? 3 : 4;
  static constexpr uint32_t kTileBytes = kTile * D * 2;
  static constexpr int NC = D + 16;  // TMEM columns of num' and of one R' block
  static constexpr int nb = (M + 127) / 128;
  uint32_t w, slots, phk, phq, rb, ones, ss, den, bars, total;
  uint32_t t_fk, t_fq, t_a, t_num, t_r;
  __host__ __device__ FwdLayout() {
    uint32_t o = 0;
    w = o; o += FAVOR ? (uint32_t)M * 128u : 0u;      // W^T as [M][64] bf16
    slots = o; o += kSlots * kTileBytes;
    phk = o; o += kTile * 128 * 2;                     // one 128-feature block
    phq = o; o += kTile * 128 * 2;                     // one phi_q block
    rb = o; o += (uint32_t)M * D * 2;                  // bf16 R(t-1)
    ones = o; o += D == 64 ? 16384u : 4096u;
    ss = o; o += (uint32_t)M * 4u;                     // fp32 S(t-1)
    den = o; o += 2u * kTile * 4u;
    bars = o; o += 8 * F_COUNT + 16;
    total = o;
    t_fk = 0;
    t_fq = FAVOR ? 64u : 0u;
    t_a = FAVOR ? 128u : 0u;
    t_num = t_a + 128u;
    t_r = t_num + NC;
  }
};

template <int D, bool FAVOR, int M>
__global__ void __launch_bounds__(kThreads, 1)
    tc_fwd_ws_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, Params p) {
  using LY = FwdLayout<D, FAVOR, M>;
  constexpr int NC = LY::NC, nb = LY::nb, kS = LY::kSlots, DP = D + 1;
  constexpr int FB = M < 128 ? M : 128;  // features of one block
  constexpr int JT = FAVOR ? M / 64 : 0;  // feature jobs per side and tile
  constexpr int JTd = JT > 0 ? JT : 1;
  constexpr int NCH = NC / 16;
  static_assert(nb <= 2, "at most 256 features");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const LY lay;
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + F_COUNT);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar + F_COUNT) + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x, bh = blockIdx.y;
  const int t0 = seg * p.tps, t1 = min(t0 + p.tps, p.nt), ntl = max(t1 - t0, 0);

  if (tid == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(bar + F_FULL + s, 1);
      mbar_init(bar + F_EMPTY + s, 5);
    }
    mbar_init(bar + F_KJFULL, 1);
    mbar_init(bar + F_KJEMPTY, 4);
    mbar_init(bar + F_QJFULL, 1);
    mbar_init(bar + F_QJEMPTY, 4);
    mbar_init(bar + F_PHK, 4);
    mbar_init(bar + F_PHQ, 4);
    mbar_init(bar + F_KFREE, 1);
    mbar_init(bar + F_QFREE, 1);
    mbar_init(bar + F_AFULL, 1);
    mbar_init(bar + F_RBFULL, 4);
    mbar_init(bar + F_ATFULL, 4);
    mbar_init(bar + F_NUMFULL, 1);
    mbar_init(bar + F_NUMEMPTY, 4);
    mbar_init(bar + F_DEN, 4);
    mbar_init(bar + F_DEN + 1, 4);
    mbar_init(bar + F_SETUP, 1);
    for (int k = 0; k < 3; ++k) mbar_init(bar + F_DONE + k, 1);
    *abort_flag = 0;
    fence_barrier_init();
    // W^T image and the incoming state (fp32 [M][D + 1], staged in the load
    // slots and the phi_k buffer behind them) by bulk copy
    const uint32_t wbytes = FAVOR ? (uint32_t)M * 128u : 0u;
    const uint32_t sbytes = seg > 0 ? (uint32_t)(M * DP * 4) : 0u;
    if (wbytes + sbytes > 0) {
      mbar_arrive_expect_tx(bar + F_SETUP, wbytes + sbytes);
      if (wbytes) bulk_load(smem + lay.w, p.wimg, wbytes, bar + F_SETUP);
      if (sbytes)
        bulk_load(smem + lay.slots, p.states + ((size_t)bh * p.P + seg - 1) * (size_t)M * DP, sbytes, bar + F_SETUP);
    }
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmQ);
  }
  if (warp == 0) tmem_alloc(tslot, 512);
  // the ones operand; zero features beyond M in phi_k (the state MMA reads 128)
  for (int idx = tid; idx < kTile * (D == 64 ? 64 : 16); idx += kThreads) {
    const int r = D == 64 ? idx >> 6 : idx >> 4, x = D == 64 ? idx & 63 : idx & 15;
    *reinterpret_cast<__nv_bfloat16 *>(smem + lay.ones + (D == 64 ? sw128_offset(r, x, kTile) : n16_offset(r, x))) =
        __float2bfloat16_rn(x == 0 ? 1.f : 0.f);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t s_w = sbase + lay.w, s_phk = sbase + lay.phk, s_phq = sbase + lay.phq;
  const uint32_t s_rb = sbase + lay.rb, s_ones = sbase + lay.ones;
  float *ss = reinterpret_cast<float *>(smem + lay.ss);
  float *den = reinterpret_cast<float *>(smem + lay.den);
  auto slot_addr = [&](int n) { return sbase + lay.slots + (uint32_t)(n % kS) * LY::kTileBytes; };
  auto slot_par = [&](int n) { return (uint32_t)((n / kS) & 1); };
  const int q4 = warp & 3, row = 32 * q4 + lane;
  const uint32_t lane_base = 32u * q4;

  // bf16 copy of R' columns [c, c + 16) of feature f and, for the chunk that
  // starts at column d, S
  auto put_rb = [&](int f, int c, const float *v) {
    if (f >= M) return;
#pragma unroll
    for (int i = 0; i < 16; i += 8)
      if (c + i + 8 <= D) st_bf16x8(s_rb + sw128_offset(f, c + i, M), v + i);
    if (c == D) ss[f] = v[0];
  };

  // incoming state -> TMEM master R' and its bf16 copies; num' columns d ..
  // d+15 start at zero (the tail warps, which own those copies)
  if (warp >= 12) {
    const bool in = seg > 0;
    if ((FAVOR || in) && !mbar_wait(bar + F_SETUP, 0, p.status, abort_flag)) {
      // nothing usable arrived: the tiles below are skipped by the abort flag
    }
    const float *stage = reinterpret_cast<const float *>(smem + lay.slots);
    for (int k = 0; k < nb * NCH; ++k) {
      const int b = k / NCH, c = (k - b * NCH) * 16, f = 128 * b + row;
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = (in && f < M && c + i <= D) ? stage[f * DP + c + i] : 0.f;
      tmem_st16(tmem_addr(tbase, lane_base, lay.t_r + b * NC + c), v);
      put_rb(f, c, v);
    }
    float z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0.f;
    tmem_st16(tmem_addr(tbase, lane_base, lay.t_num + D), z);
    tmem_st_wait();
  }
  if (M < 128) {
    for (int idx = tid; idx < kTile * 128; idx += kThreads) {
      const int r = idx >> 7, x = idx & 127;
      if (x >= M) *reinterpret_cast<__nv_bfloat16 *>(smem + lay.phk + sw128_offset(r, x, kTile)) = __float2bfloat16_rn(0.f);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  bool ok = true;
  auto wait = [&](int b, uint32_t par) {
    if (ok) ok = mbar_wait(bar + b, par, p.status, abort_flag);
    return ok;
  };
  auto arrive = [&](int b) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar + b);
  };
  if (warp >= 12) arrive(F_RBFULL);  // phase 0: R(t0 - 1) is in place

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int n = 0;
      for (int t = t0; t < t1 && ok; ++t) {
        const CUtensorMap *maps[3] = {&tmK, &tmQ, &tmV};
        for (int r = 0; r < 3 && ok; ++r, ++n) {
          const int s = n % kS, u = n / kS;
          if (u > 0 && !wait(F_EMPTY + s, (u - 1) & 1)) break;
          mbar_arrive_expect_tx(bar + F_FULL + s, LY::kTileBytes);
          for (int c = 0; c < D; c += 64)
            tma_load_3d(smem + lay.slots + s * LY::kTileBytes + c * kTile * 2, maps[r], bar + F_FULL + s, c,
                        t * kTile, bh);
        }
      }
      for (int m = max(0, n - kS); m < n; ++m) mbar_drain(bar + F_FULL + m % kS, slot_par(m));
      if (FAVOR || seg > 0) mbar_drain(bar + F_SETUP, 0);
    }
  } else if (warp < 4) {
    // ---------------------------------------------------------------- MMA issuers
    if (lane == 0 && (FAVOR || warp == 3)) {
      constexpr uint32_t NV = D == 64 ? D + 16 : D;  // [V, 1] in one MMA when d = 64
      // Base descriptors, computed once.  The start address is the low field
      // (16-byte units) and no operand crosses 256 KB, so a K step, a slot or
      // a feature offset is an add to the descriptor.
      constexpr uint64_t kSlotStep = LY::kTileBytes >> 4;
      const uint64_t d_x0 = desc_kmajor(slot_addr(0), kTile, 0, 0);  // slot 0, K-major
      // K-major step s of a tile of `rows` rows
      auto ks = [](int s, uint32_t rows) { return (uint64_t)((s >> 2) * rows * 8u + (s & 3) * 2u); };
      auto commit = [&](int b) { mma_commit(bar + b); };
      if (warp < 3) {
        // feature jobs of one side, in order: job j = features [64 (j % JT), +64) of tile j / JT
        const int side = warp - 1;
        const uint32_t id_f = make_idesc(128, 64, false, false);
        const uint64_t d_w0 = desc_kmajor(s_w, M, 0, 0);
        const uint32_t t_d = tbase + (side ? lay.t_fq : lay.t_fk);
        const int b_full = side ? F_QJFULL : F_KJFULL, b_empty = side ? F_QJEMPTY : F_KJEMPTY;
        for (int j = 0; j < ntl * JT && ok; ++j) {
          const int i = j / JTd, n = 3 * i + side;
          if (j > 0 && !wait(b_empty, (j - 1) & 1)) break;
          if (j % JTd == 0 && !wait(F_FULL + n % kS, slot_par(n))) break;
          tc_fence_after();
          const uint64_t dx = d_x0 + (uint64_t)(n % kS) * kSlotStep;
          const uint64_t dw = d_w0 + (uint64_t)((j % JTd) * 512);  // 64 rows = 8 atoms of 1024 B
#pragma unroll
          for (int s = 0; s < D / 16; ++s) mma_bf16(t_d, dx + ks(s, kTile), dw + ks(s, M), id_f, s > 0);
          commit(b_full);
          if (j % JTd == JT - 1) commit(F_EMPTY + n % kS);
        }
      } else {
        const uint32_t id_a = make_idesc(128, 128, false, false);
        const uint32_t id_n = make_idesc(128, D, false, true);
        const uint32_t id_nv = make_idesc(128, NV, false, true);
        const uint32_t id_s = make_idesc(128, 16, false, true);
        const uint32_t id_r = make_idesc(128, NV, true, true);
        const uint32_t id_r1 = make_idesc(128, 16, true, true);
        const uint64_t d_v0 = D == 64 ? make_desc(slot_addr(0), s_ones - slot_addr(0), 1024u, kSwizzle128)
                                      : desc_mnmajor(slot_addr(0), kTile, 0, 0);  // [V, 1] (or V), slot 0
        const uint64_t d_phk_k = desc_kmajor(s_phk, kTile, 0, 0), d_phk_mn = desc_mnmajor(s_phk, kTile, 0, 0);
        const uint64_t d_phq_k = desc_kmajor(s_phq, kTile, 0, 0);
        const uint64_t d_rb = desc_mnmajor(s_rb, M, 0, 0);
        const uint64_t d_ones = desc_n16(s_ones, 0);
        // [V, 1] of load n: the slot moves the start address up and the ones block's LBO down
        auto slot_v = [&](int n) {
          const uint64_t q = (uint64_t)(n % kS) * kSlotStep;
          return D == 64 ? d_v0 + q - (q << 16) : d_v0 + q;
        };
        auto test = [&](int b, uint32_t par) { return mbar_test(bar + b, par); };
        // R'_h += phi_k,h^T [V, 1], in place
        auto issue_r = [&](int i, int h) {
          const uint64_t dv = slot_v(3 * i + 2);
          const uint32_t t_r = tbase + lay.t_r + h * NC;
#pragma unroll
          for (int s = 0; s < kTile / 16; ++s) {
            const uint64_t a = d_phk_mn + (uint64_t)(s * 128);
            mma_bf16(t_r, a, dv + (uint64_t)(s * 128), id_r, 1);
            if (D != 64) mma_bf16(t_r + D, a, d_ones + (uint64_t)(s * 32), id_r1, 1);
          }
        };
        // A += phi_q,h phi_k,h^T and num += phi_q,h R_h^T
        auto issue_an = [&](int h) {
          const uint64_t dr = d_rb + (uint64_t)(h * 8 * 128);
          const uint32_t t_a = tbase + lay.t_a, t_n = tbase + lay.t_num;
#pragma unroll
          for (int s = 0; s < FB / 16; ++s) {
            const uint32_t acc = (h > 0 || s > 0) ? 1u : 0u;
            const uint64_t aq = d_phq_k + ks(s, kTile);
            mma_bf16(t_a, aq, d_phk_k + ks(s, kTile), id_a, acc);
            mma_bf16(t_n, aq, dr + (uint64_t)(s * 128), id_n, acc);
          }
        };
        // num' += tril(A) [V, 1], the masked A as bf16 pairs in TMEM
        auto issue_av = [&](int i) {
          const uint64_t dv = slot_v(3 * i + 2);
          const uint32_t t_n = tbase + lay.t_num, t_a = tbase + lay.t_a;
#pragma unroll
          for (int s = 0; s < kTile / 16; ++s) {
            mma_bf16_ta(t_n, t_a + 8 * s, dv + (uint64_t)(s * 128), D == 64 ? id_nv : id_n, 1);
            if (D != 64) mma_bf16_ta(t_n + D, t_a + 8 * s, d_ones + (uint64_t)(s * 32), id_s, 1);
          }
        };
        const int NB = ntl * nb;
        int nr = 0, na = 0, nav = 0;
        // prerequisites of the next R, A/num and AV found complete (each
        // barrier phase is tested until it passes, then not again)
        int r_got = 0, a_got = 0;
        uint32_t idle = 0;
        uint64_t idle_since = 0;
        while (nr < NB || na < NB || nav < ntl) {
          bool did = false;
          if (nav < ntl && test(F_ATFULL, nav & 1)) {
            tc_fence_after();
            issue_av(nav);
            commit(F_NUMFULL);
            commit(F_EMPTY + (3 * nav + 2) % kS);
            ++nav;
            did = true;
          }
          if (!did && nr < NB) {
            const int i = nr / nb, h = nr % nb;
            if (r_got == 0 && test(F_PHK, nr & 1)) r_got = h > 0 ? 3 : 1;
            if (r_got == 1 && test(F_FULL + (3 * i + 2) % kS, slot_par(3 * i + 2))) r_got = 2;
            if (r_got == 2 && test(F_RBFULL, i & 1)) r_got = 3;
            if (r_got == 3) {
              tc_fence_after();
              issue_r(i, h);
              ++nr;
              r_got = 0;
              if (na > i * nb + h) {
                commit(F_KFREE);
                if (h == nb - 1) commit(F_AFULL);
              }
              did = true;
            }
          }
          if (!did && na < NB) {
            const int i = na / nb, h = na % nb;
            if (a_got == 0 && test(F_PHQ, na & 1)) a_got = 1;
            if (a_got == 1 && test(F_PHK, na & 1)) a_got = 2;
            if (a_got == 2 && test(F_RBFULL, i & 1)) a_got = (h > 0 || i == 0) ? 5 : 3;
            // A restarts where tril(A(t-1)) [V, 1] reads its operand: after
            // that MMA in this thread's (in-order) stream
            if (a_got == 3 && nav >= i) a_got = 4;
            if (a_got == 4 && test(F_NUMEMPTY, (i - 1) & 1)) a_got = 5;
            if (a_got == 5) {
              tc_fence_after();
              issue_an(h);
              ++na;
              a_got = 0;
              if (!FAVOR && h == 0) {
                // elu+1 features are formed by the epilogue alone: the MMA's share of the K and Q slots
                mbar_arrive(bar + F_EMPTY + (3 * i) % kS);
                mbar_arrive(bar + F_EMPTY + (3 * i + 1) % kS);
              }
              if (nr > i * nb + h) {
                commit(F_KFREE);
                if (h == nb - 1) commit(F_AFULL);
              }
              commit(F_QFREE);
              did = true;
            }
          }
          if (did) {
            idle = 0;
            continue;
          }
          // nothing ready: yield the scheduler to the epilogue warps sharing it
          __nanosleep(32);
          if (idle++ == 0) {
            idle_since = global_ns();
          } else if ((idle & 63u) == 0) {
            if (*abort_flag) break;
            if (global_ns() - idle_since > 1000000000ull) {
              atomicCAS(p.status, 0, 5);
              *abort_flag = 1;
              break;
            }
          }
        }
      }
      commit(F_DONE + (warp - 1));
      mbar_drain(bar + F_DONE + (warp - 1), 0);
    }
  } else if (warp < 12) {
    // ---------------------------------------------------------------- phi_k (4-7), phi_q (8-11)
    const int side = warp >= 8 ? 1 : 0;
    const uint32_t s_out = side ? s_phq : s_phk;
    const int b_jfull = side ? F_QJFULL : F_KJFULL, b_jempty = side ? F_QJEMPTY : F_KJEMPTY;
    const int b_free = side ? F_QFREE : F_KFREE, b_stored = side ? F_PHQ : F_PHK;
    const uint32_t t_f = tbase + (side ? lay.t_fq : lay.t_fk);
    int jobs = 0;
    for (int i = 0; i < ntl && ok; ++i) {
      const int t = t0 + i;
      const bool dead = row >= min(kTile, p.L - t * kTile);  // padding rows past L: features forced to zero
      const int n = 3 * i + side, s = n % kS;
      const uint32_t s_x = slot_addr(n);
      if (!wait(F_FULL + s, slot_par(n))) break;
      float cr = 0.f;  // exp2 offset of the row
      if (FAVOR) {
        cr = favor_row_const(tile_row_sqnorm(s_x, row, D), M);
        arrive(F_EMPTY + s);
      }
      // phi_q . S(t-1) needs S(t-1), written with the bf16 copy of R(t-1)
      if (side && !wait(F_RBFULL, i & 1)) break;
      float dp[4] = {0.f, 0.f, 0.f, 0.f};
      for (int h = 0; h < nb && ok; ++h) {
        const uint32_t c = (uint32_t)(i * nb + h);
        for (int half = 0; half < FB / 64; ++half) {
          float v[64];
          if (FAVOR) {
            if (!wait(b_jfull, jobs & 1)) break;
            tc_fence_after();
            tmem_ld32x2(tmem_addr(t_f, lane_base, 0), tmem_addr(t_f, lane_base, 32), v, v + 32);
            tc_fence_before();
            arrive(b_jempty);
            ++jobs;
#pragma unroll
            for (int x = 0; x < 64; ++x) v[x] = dead ? 0.f : favor_feature(v[x], cr);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              ld_bf16x8(s_x + sw128_offset(row, 128 * h + 64 * half + 8 * j, kTile), v + 8 * j);
#pragma unroll
              for (int x = 0; x < 8; ++x) v[8 * j + x] = dead ? 0.f : elu1_feature(v[8 * j + x]);
            }
          }
          if (side) {
            const float *sh = ss + 128 * h + 64 * half;
#pragma unroll
            for (int x = 0; x < 64; ++x) dp[x & 3] = fmaf(v[x], sh[x], dp[x & 3]);
          }
          if (half == 0 && c > 0 && !wait(b_free, (c - 1) & 1)) break;
#pragma unroll
          for (int j = 0; j < 8; ++j) st_bf16x8(s_out + sw128_offset(row, 64 * half + 8 * j, kTile), v + 8 * j);
        }
        if (!ok) break;
        fence_async_smem();
        arrive(b_stored);
      }
      if (!ok) break;
      if (!FAVOR) arrive(F_EMPTY + s);
      if (side) {
        den[(i & 1) * kTile + row] = (dp[0] + dp[1]) + (dp[2] + dp[3]);
        arrive(F_DEN + (i & 1));
      }
    }
  } else {
    // ---------------------------------------------------------------- tail (12-15)
    for (int i = 0; i < ntl && ok; ++i) {
      const int t = t0 + i;
      if (!wait(F_AFULL, i & 1)) break;
      tc_fence_after();
      // masked A (diagonal kept) -> bf16 pairs in place over A's first 64
      // columns: the A operand of tril(A) [V, 1], read from TMEM
      {
        uint32_t pk[64];
#pragma unroll
        for (int c0 = 0; c0 < kTile; c0 += 32) {
          float v[32];
          tmem_ld32(tmem_addr(tbase, lane_base, lay.t_a + c0), v);
#pragma unroll
          for (int x = 0; x < 32; x += 2)
            pk[(c0 + x) >> 1] = pack_bf16(c0 + x > row ? 0.f : v[x], c0 + x + 1 > row ? 0.f : v[x + 1]);
        }
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          float f[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) f[x] = __uint_as_float(pk[c + x]);
          tmem_st16(tmem_addr(tbase, lane_base, lay.t_a + c), f);
        }
        // num' columns d .. d+15 restart at zero (read for Y(t-1) by these warps)
        float z[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) z[x] = 0.f;
        tmem_st16(tmem_addr(tbase, lane_base, lay.t_num + D), z);
        tmem_st_wait();
        tc_fence_before();
      }
      arrive(F_ATFULL);
      // bf16 copies of R(t) and S(t) for tile t + 1
      if (i + 1 < ntl) {
        for (int k = 0; k < nb * NCH; ++k) {
          const int b = k / NCH, c = (k - b * NCH) * 16;
          float v[16];
          tmem_ld16(tmem_addr(tbase, lane_base, lay.t_r + b * NC + c), v);
          put_rb(128 * b + row, c, v);
        }
        fence_async_smem();
        tc_fence_before();
        arrive(F_RBFULL);
      }
      // Y = num / (den + rowsum A)
      if (!wait(F_NUMFULL, i & 1)) break;
      tc_fence_after();
      const bool live = row < min(kTile, p.L - t * kTile);
      __nv_bfloat16 *yrow = p.y + ((size_t)bh * p.L + (size_t)t * kTile + row) * D;
      auto store_y = [&](int c0, const float *v, float inv) {
        uint4 *dst = reinterpret_cast<uint4 *>(yrow + c0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          dst[k] = make_uint4(pack_bf16(v[8 * k] * inv, v[8 * k + 1] * inv), pack_bf16(v[8 * k + 2] * inv, v[8 * k + 3] * inv),
                              pack_bf16(v[8 * k + 4] * inv, v[8 * k + 5] * inv), pack_bf16(v[8 * k + 6] * inv, v[8 * k + 7] * inv));
      };
      const float rowsum_a = tmem_ld1(tmem_addr(tbase, lane_base, lay.t_num + D));
      if constexpr (D == 64) {
        float v[64];
        tmem_ld32x2(tmem_addr(tbase, lane_base, lay.t_num), tmem_addr(tbase, lane_base, lay.t_num + 32), v, v + 32);
        tc_fence_before();
        arrive(F_NUMEMPTY);
        if (!wait(F_DEN + (i & 1), (i >> 1) & 1)) break;
        if (live) {
          const float inv = 1.0f / (rowsum_a + den[(i & 1) * kTile + row]);
          store_y(0, v, inv);
          store_y(32, v + 32, inv);
        }
      } else {
        if (!wait(F_DEN + (i & 1), (i >> 1) & 1)) break;
        const float inv = 1.0f / (rowsum_a + den[(i & 1) * kTile + row]);
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float v[32];
          tmem_ld32(tmem_addr(tbase, lane_base, lay.t_num + c0), v);
          if (live) store_y(c0, v, inv);
        }
        tc_fence_before();
        arrive(F_NUMEMPTY);
      }
      arrive(F_EMPTY + (3 * i + 2) % kS);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

}  // namespace fw

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
  if constexpr (MODE == MODE_FWD) {
    const int smem = (int)fw::FwdLayout<D, FAVOR, M>().total + 1024;
    auto kern = fw::tc_fwd_ws_kernel<D, FAVOR, M>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(nseg, pl.BH), fw::kThreads, smem, st>>>(mq, mk, mv, p);
  } else {
    const Layout<D, FAVOR, MODE> lay(M);
    const int smem = (int)lay.total + 1024;
    auto kern = tc_fwd_kernel<D, FAVOR, MODE, M>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(nseg, pl.BH), kThreads, smem, st>>>(mq, mk, mv, mz ? mz[0] : mk, mz ? mz[1] : mk, mz ? mz[2] : mk, p);
  }
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
  if (d == 64 && favor) {
    if (M == 64) return tcf::fw::FwdLayout<64, true, 64>().total + 1024;
    if (M == 128) return tcf::fw::FwdLayout<64, true, 128>().total + 1024;
    return tcf::fw::FwdLayout<64, true, 256>().total + 1024;
  }
  if (d == 64) return tcf::fw::FwdLayout<64, false, 64>().total + 1024;
  return tcf::fw::FwdLayout<128, false, 128>().total + 1024;
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
