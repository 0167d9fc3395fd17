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
enum { MODE_STATE = 0, MODE_FWD = 1 };

struct Params {
  int L, M, nt, P, tps;
  int H, wstride;  // heads; bf16 elements between per-head W^T images (0: one shared W)
  int zero_grads;  // state pass of a two-CTA backward: zero these outputs tile by tile (1 dQ, 2 dK, 4 dV)
  __nv_bfloat16 *y;
  const __nv_bfloat16 *wimg;  // W^T shared-memory image (FAVOR+)
  float *states;     // fp32 [BH][P][M][D + 1]: high parts of the segment states
  float *states_lo;  // same layout: low parts
  const float *state_in;  // carried state of earlier rows, fp32 [BH][M][D + 1], or NULL
  int *status;
};

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
  // debug builds: a segment outside the plan records SLIM_ERR_BOUNDS and the CTA does nothing
  if (!SLIM_DCHECK(p.status, seg < p.P && seg * p.tps < p.nt)) return;
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
    // segment 0 starts from the carried state of earlier rows, if any
    const uint32_t sbytes = (seg > 0 || p.state_in) ? (uint32_t)(M * DP * 4) : 0u;
    if (wbytes + sbytes > 0) {
      mbar_arrive_expect_tx(bar + F_SETUP, wbytes + sbytes);
      if (wbytes) bulk_load(smem + lay.w, p.wimg + (size_t)(bh % p.H) * p.wstride, wbytes, bar + F_SETUP);
      if (sbytes)
        bulk_load(smem + lay.slots,
                  seg > 0 ? p.states + ((size_t)bh * p.P + seg - 1) * (size_t)M * DP
                          : p.state_in + (size_t)bh * M * DP,
                  sbytes, bar + F_SETUP);
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
  // Load n = 3 i + r is K (r = 0), Q (1) or V (2) of tile i.  Every slot holds
  // one kind only (K in 0, Q in 1, V in 2 and, with four slots, 3 for odd
  // tiles), so each consumer waits on every phase of the slots it reads.  A
  // slot that rotated through the kinds would make a consumer wait on a phase
  // whose predecessor (another kind's load, never waited on by it) may still
  // be in flight, and a parity wait then passes on that predecessor's
  // predecessor: the consumer reads the slot before its load lands.
  auto slot_idx = [&](int n) {
    const int i = n / 3, r = n - 3 * i;
    return r < 2 ? r : (kS == 4 ? 2 + (i & 1) : 2);
  };
  auto slot_use = [&](int n) {  // loads into this slot before load n
    const int i = n / 3, r = n - 3 * i;
    return (r == 2 && kS == 4) ? i >> 1 : i;
  };
  auto slot_addr = [&](int n) { return sbase + lay.slots + (uint32_t)slot_idx(n) * LY::kTileBytes; };
  auto slot_par = [&](int n) { return (uint32_t)(slot_use(n) & 1); };
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
    const bool in = seg > 0 || p.state_in != nullptr;
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
          const int s = slot_idx(n), u = slot_use(n);
          if (u > 0 && !wait(F_EMPTY + s, (u - 1) & 1)) break;
          mbar_arrive_expect_tx(bar + F_FULL + s, LY::kTileBytes);
          for (int c = 0; c < D; c += 64)
            tma_load_3d(smem + lay.slots + s * LY::kTileBytes + c * kTile * 2, maps[r], bar + F_FULL + s, c,
                        t * kTile, bh);
        }
      }
      // the last load of every slot (the last tile's K, Q, V and, with four
      // slots, the V before it)
      for (int m = max(0, n - kS); m < n; ++m) mbar_drain(bar + F_FULL + slot_idx(m), slot_par(m));
      if (FAVOR || seg > 0 || p.state_in) mbar_drain(bar + F_SETUP, 0);
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
          if (j % JTd == 0 && !wait(F_FULL + slot_idx(n), slot_par(n))) break;
          tc_fence_after();
          const uint64_t dx = d_x0 + (uint64_t)slot_idx(n) * kSlotStep;
          const uint64_t dw = d_w0 + (uint64_t)((j % JTd) * 512);  // 64 rows = 8 atoms of 1024 B
#pragma unroll
          for (int s = 0; s < D / 16; ++s) mma_bf16(t_d, dx + ks(s, kTile), dw + ks(s, M), id_f, s > 0);
          commit(b_full);
          if (j % JTd == JT - 1) commit(F_EMPTY + slot_idx(n));
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
          const uint64_t q = (uint64_t)slot_idx(n) * kSlotStep;
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
            commit(F_EMPTY + slot_idx(3 * nav + 2));
            ++nav;
            did = true;
          }
          if (!did && nr < NB) {
            const int i = nr / nb, h = nr % nb;
            if (r_got == 0 && test(F_PHK, nr & 1)) r_got = h > 0 ? 3 : 1;
            if (r_got == 1 && test(F_FULL + slot_idx(3 * i + 2), slot_par(3 * i + 2))) r_got = 2;
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
                mbar_arrive(bar + F_EMPTY + slot_idx(3 * i));
                mbar_arrive(bar + F_EMPTY + slot_idx(3 * i + 1));
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
      const int n = 3 * i + side, s = slot_idx(n);
      const uint32_t s_x = slot_addr(n);
      if (!wait(F_FULL + s, slot_par(n))) break;
      float cr = 0.f;  // exp2 offset of the row
      if (FAVOR) {
        // padding rows: F = 0 (zero-filled tile) and 2^-inf = 0, no select
        cr = dead ? -INFINITY : favor_row_const(tile_row_sqnorm(s_x, row, D), M);
        arrive(F_EMPTY + s);
      }
      // phi_q . S(t-1) needs S(t-1), written with the bf16 copy of R(t-1)
      // once the previous tile's last MMAs are done: the first block's
      // features are formed and stored without it, and its share of the dot
      // product is taken from the stored bf16 values once S(t-1) is in; later
      // blocks (after the wait) use their fp32 values.
      // dp[x & 3] sums of phi_q . S(t-1), as two packed pairs: (0, 1), (2, 3)
      float2 dp[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
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
            for (int x = 0; x < 64; x += 2) favor_feature2(v[x], v[x + 1], cr);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              ld_bf16x8(s_x + sw128_offset(row, 128 * h + 64 * half + 8 * j, kTile), v + 8 * j);
#pragma unroll
              for (int x = 0; x < 8; ++x) v[8 * j + x] = dead ? 0.f : elu1_feature(v[8 * j + x]);
            }
          }
          if (side && h > 0) {
            const float2 *sh = reinterpret_cast<const float2 *>(ss + 128 * h + 64 * half);
#pragma unroll
            for (int x = 0; x < 64; x += 2)
              dp[(x >> 1) & 1] = __ffma2_rn(make_float2(v[x], v[x + 1]), sh[x >> 1], dp[(x >> 1) & 1]);
          }
          if (half == 0 && c > 0 && !wait(b_free, (c - 1) & 1)) break;
#pragma unroll
          for (int j = 0; j < 8; ++j) st_bf16x8(s_out + sw128_offset(row, 64 * half + 8 * j, kTile), v + 8 * j);
        }
        if (!ok) break;
        if (side && h == 0) {
          // the first block's phi_q . S(t-1), from this row's stored bf16
          // features, before the MMAs are told the block is in (S(t) then
          // replaces S(t-1) only after this tile's last MMAs)
          if (!wait(F_RBFULL, i & 1)) break;
#pragma unroll 4
          for (int x0 = 0; x0 < FB; x0 += 8) {
            float f[8];
            ld_bf16x8(s_out + sw128_offset(row, x0, kTile), f);
            const float2 *sh = reinterpret_cast<const float2 *>(ss + x0);
#pragma unroll
            for (int x = 0; x < 8; x += 2)
              dp[(x >> 1) & 1] = __ffma2_rn(make_float2(f[x], f[x + 1]), sh[x >> 1], dp[(x >> 1) & 1]);
          }
        }
        fence_async_smem();
        arrive(b_stored);
      }
      if (!ok) break;
      if (!FAVOR) arrive(F_EMPTY + s);
      if (side) {
        den[(i & 1) * kTile + row] = (dp[0].x + dp[0].y) + (dp[1].x + dp[1].y);
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
        for (int c0 = 0; c0 < kTile; c0 += 64) {
          // two 32-column loads under one wait
          float v[64];
          tmem_ld32x2(tmem_addr(tbase, lane_base, lay.t_a + c0), tmem_addr(tbase, lane_base, lay.t_a + c0 + 32), v,
                      v + 32);
#pragma unroll
          for (int x = 0; x < 64; x += 2)
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
        const float2 inv2 = make_float2(inv, inv);
        auto y2 = [&](int x) {
          const float2 r = __fmul2_rn(make_float2(v[x], v[x + 1]), inv2);
          return pack_bf16(r.x, r.y);
        };
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(y2(8 * k), y2(8 * k + 2), y2(8 * k + 4), y2(8 * k + 6));
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
      arrive(F_EMPTY + slot_idx(3 * i + 2));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

}  // namespace fw

// ============================================================================
// Segment-state pass (the K side alone): writes each segment's total R' (the
// rows eq. (3) adds) for the segment scan.  Each tile's increment
// dR'_h = phi_k,h^T [V, 1] is an MMA that restarts at zero, and the tail
// warps add it into an fp32 master in TMEM, as a double-float (low part in
// shared memory) for the normaliser column S.  The backward recovers the
// first tiles' small states by subtracting increments from this total, so
// rounding in the total shows up there: accumulating in place on the tensor
// pipe cost dQ of the first tiles of a long segment a factor of two hundred,
// and plain fp32 still a factor of 2.6 through S, whose positive terms make
// its rounding errors add up; the signed R columns' errors do not.
//   warp 0       TMA producer (K, V ring; zero tiles of the outputs a
//                two-CTA backward accumulates into);
//   warp 1       feature MMAs F = K W, 64 features per job, two TMEM buffers;
//   warp 2       increment MMAs;
//   warps 4-11   phi_k: two threads per row, 32 columns of each job each,
//                into two phi_k buffers used in turn;
//   warps 12-15  master += increment, then the segment total.
namespace sw {

constexpr int kWarps = 16;
constexpr int kThreads = 32 * kWarps;

enum {
  S_FULL = 0,      // [4] slot loaded
  S_EMPTY = 4,     // [4] slot free: MMA commit + 8 consumer arrivals
  S_FFULL = 8,     // [2] feature job in TMEM buffer b
  S_FEMPTY = 10,   // [2] ... read out (8 warps)
  S_PHK = 12,      // [2] phi_k block stored in buffer b (8 warps)
  S_PHFREE = 14,   // [2] increment MMAs reading phi_k buffer b done
  S_AFULL = 16,    // the tile's increment complete
  S_INCFREE = 17,  // increment added into the master (4 warps)
  S_SETUP = 18,    // W image
  S_DONE = 19,     // [2] MMA drain of each issuing thread
  S_COUNT = 21
};

template <int D, bool FAVOR, int M>
struct StateLayout {
  static constexpr int kSlots = D == 128 ? 3 : 4;
  static constexpr uint32_t kTileBytes = kTile * D * 2;
  static constexpr int NC = D + 16;  // TMEM columns of one R' block
  uint32_t w, slots, phk, ones, zero, lo, nrm, bars, total;
  __host__ __device__ StateLayout() {
    uint32_t o = 0;
    w = o; o += FAVOR ? (uint32_t)M * 128u : 0u;  // W^T as [M][64] bf16
    slots = o; o += kSlots * kTileBytes;            // then, at the end, the [M][D + 1] outputs
    phk = o; o += 2u * kTile * 128 * 2;             // two phi_k blocks
    ones = o; o += D == 64 ? 16384u : 4096u;
    zero = o; o += kTile * 64 * 2;                  // zero box of [128][64] (two-CTA backward)
    lo = o; o += (uint32_t)M * 4u;                  // low parts of S
    nrm = o; o += 2u * 2u * kTile * 4u;             // [tile parity][half of d][row] partial |k|^2
    bars = o; o += 8 * S_COUNT + 16;
    total = o;
  }
};

template <int D, bool FAVOR, int M>
__global__ void __launch_bounds__(kThreads, 1)
    tc_state_ws_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmDK,
                       const __grid_constant__ CUtensorMap tmDV, Params p) {
  using LY = StateLayout<D, FAVOR, M>;
  constexpr int NC = LY::NC, kS = LY::kSlots, DP = D + 1;
  constexpr int nb = (M + 127) / 128, FB = M < 128 ? M : 128, NCH = NC / 16;
  constexpr int JT = FAVOR ? M / 64 : 0, JTd = JT > 0 ? JT : 1;  // feature jobs per tile
  static_assert(LY::kSlots * LY::kTileBytes + 2 * kTile * 128 * 2 >= (uint32_t)M * DP * 4, "output staging fits");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const LY lay;
  const uint32_t sbase = smem_u32(smem);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + lay.bars);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + S_COUNT);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(bar + S_COUNT) + 1;
  // TMEM: feature buffers 2 x 64 | increment nb x NC | master nb x NC
  const uint32_t t_f = 0, t_inc = FAVOR ? 128u : 0u, t_m = t_inc + nb * NC;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seg = blockIdx.x, bh = blockIdx.y;
  // debug builds: a segment outside the plan records SLIM_ERR_BOUNDS and the CTA does nothing
  if (!SLIM_DCHECK(p.status, seg < p.P && seg * p.tps < p.nt)) return;
  const int t0 = seg * p.tps, t1 = min(t0 + p.tps, p.nt), ntl = max(t1 - t0, 0);

  if (tid == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(bar + S_FULL + s, 1);
      mbar_init(bar + S_EMPTY + s, 9);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar + S_FFULL + b, 1);
      mbar_init(bar + S_FEMPTY + b, 8);
      mbar_init(bar + S_PHK + b, 8);
      mbar_init(bar + S_PHFREE + b, 1);
      mbar_init(bar + S_DONE + b, 1);
    }
    mbar_init(bar + S_AFULL, 1);
    mbar_init(bar + S_INCFREE, 4);
    mbar_init(bar + S_SETUP, 1);
    *abort_flag = 0;
    fence_barrier_init();
    if (FAVOR) {
      mbar_arrive_expect_tx(bar + S_SETUP, (uint32_t)M * 128u);
      bulk_load(smem + lay.w, p.wimg + (size_t)(bh % p.H) * p.wstride, (uint32_t)M * 128u, bar + S_SETUP);
    }
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
  }
  if (warp == 0) tmem_alloc(tslot, 512);
  for (int idx = tid; idx < kTile * 64 * 2 / 16; idx += kThreads)
    reinterpret_cast<uint4 *>(smem + lay.zero)[idx] = make_uint4(0u, 0u, 0u, 0u);
  for (int idx = tid; idx < M; idx += kThreads) reinterpret_cast<float *>(smem + lay.lo)[idx] = 0.f;
  for (int idx = tid; idx < kTile * (D == 64 ? 64 : 16); idx += kThreads) {
    const int r = D == 64 ? idx >> 6 : idx >> 4, x = D == 64 ? idx & 63 : idx & 15;
    *reinterpret_cast<__nv_bfloat16 *>(smem + lay.ones + (D == 64 ? sw128_offset(r, x, kTile) : n16_offset(r, x))) =
        __float2bfloat16_rn(x == 0 ? 1.f : 0.f);
  }
  if (M < 128) {
    // features beyond M stay zero: the increment MMA reads 128
    for (int idx = tid; idx < 2 * kTile * 128; idx += kThreads) {
      const int b = idx >> 14, r = (idx >> 7) & 127, x = idx & 127;
      if (x >= M)
        *reinterpret_cast<__nv_bfloat16 *>(smem + lay.phk + b * kTile * 256 + sw128_offset(r, x, kTile)) =
            __float2bfloat16_rn(0.f);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const int q4 = warp & 3, row = 32 * q4 + lane;
  const uint32_t lane_base = 32u * q4;
  if (warp >= 12) {
    // the master starts at zero
    float z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0.f;
    for (int k = 0; k < nb * NCH; ++k) tmem_st16(tmem_addr(tbase, lane_base, t_m + (k / NCH) * NC + (k % NCH) * 16), z);
    tmem_st_wait();
  }
  if (FAVOR && warp == 1 && lane == 0) mbar_wait(bar + S_SETUP, 0, p.status, abort_flag);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t s_w = sbase + lay.w, s_phk = sbase + lay.phk, s_ones = sbase + lay.ones;
  // Load n = 2 i + r is K (r = 0) or V (1) of tile i.  Every slot holds one
  // kind only, so each consumer waits on every phase of its slots (see the
  // forward): with four slots K takes 0 and 2, V 1 and 3, by tile parity;
  // with three, K takes 0 and V takes 1 and 2 by tile parity.
  auto slot_idx = [&](int n) {
    const int i = n >> 1, r = n & 1;
    return kS == 4 ? n & 3 : (r == 0 ? 0 : 1 + (i & 1));
  };
  auto slot_use = [&](int n) {  // loads into this slot before load n
    const int i = n >> 1, r = n & 1;
    return kS == 4 ? n >> 2 : (r == 0 ? i : i >> 1);
  };
  auto slot_addr = [&](int n) { return sbase + lay.slots + (uint32_t)slot_idx(n) * LY::kTileBytes; };
  auto slot_par = [&](int n) { return (uint32_t)(slot_use(n) & 1); };
  bool ok = true;
  auto wait = [&](int b, uint32_t par) {
    if (ok) ok = mbar_wait(bar + b, par, p.status, abort_flag);
    return ok;
  };
  auto arrive = [&](int b) {
    __syncwarp();
    if (lane == 0) mbar_arrive(bar + b);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int n = 0;
      for (int t = t0; t < t1 && ok; ++t) {
        for (int r = 0; r < 2 && ok; ++r, ++n) {
          const int s = slot_idx(n), u = slot_use(n);
          if (u > 0 && !wait(S_EMPTY + s, (u - 1) & 1)) break;
          mbar_arrive_expect_tx(bar + S_FULL + s, LY::kTileBytes);
          for (int c = 0; c < D; c += 64)
            tma_load_3d(smem + lay.slots + s * LY::kTileBytes + c * kTile * 2, r ? &tmV : &tmK, bar + S_FULL + s, c,
                        t * kTile, bh);
        }
        if (p.zero_grads) {
          // the two-CTA backward adds its per-CTA partials into these
          for (int c = 0; c < D; c += 64) {
            if (p.zero_grads & 1) tma_store_3d(&tmDQ, smem + lay.zero, c, t * kTile, bh);
            if (p.zero_grads & 2) tma_store_3d(&tmDK, smem + lay.zero, c, t * kTile, bh);
            if (p.zero_grads & 4) tma_store_3d(&tmDV, smem + lay.zero, c, t * kTile, bh);
          }
          tma_store_commit();
        }
      }
      if (p.zero_grads) tma_store_wait_all();
      // the last load of every slot
      for (int m = max(0, n - kS); m < n; ++m) mbar_drain(bar + S_FULL + slot_idx(m), slot_par(m));
      if (FAVOR) mbar_drain(bar + S_SETUP, 0);
    }
  } else if (warp == 1 || warp == 2) {
    // ---------------------------------------------------------------- MMA issuers
    if (lane == 0 && (FAVOR || warp == 2)) {
      if (warp == 1) {
        // feature jobs: job j = features [64 (j % JT), +64) of tile j / JT into buffer j & 1
        const uint32_t id_f = make_idesc(128, 64, false, false);
        const uint64_t d_w0 = desc_kmajor(s_w, M, 0, 0);
        for (int j = 0; j < ntl * JT && ok; ++j) {
          const int i = j / JTd, n = 2 * i, b = j & 1, u = j >> 1;
          if (u > 0 && !wait(S_FEMPTY + b, (u - 1) & 1)) break;
          if (j % JTd == 0 && !wait(S_FULL + slot_idx(n), slot_par(n))) break;
          tc_fence_after();
          const uint64_t dx = desc_kmajor(slot_addr(n), kTile, 0, 0);
          const uint64_t dw = d_w0 + (uint64_t)((j % JTd) * 512);  // 64 rows = 8 atoms of 1024 B
#pragma unroll
          for (int s = 0; s < D / 16; ++s)
            mma_bf16(tbase + t_f + 64 * b, dx + (uint64_t)((s & 3) * 2), dw + (uint64_t)((s & 3) * 2), id_f, s > 0);
          mma_commit(bar + S_FFULL + b);
          if (j % JTd == JT - 1) mma_commit(bar + S_EMPTY + slot_idx(n));
        }
      } else {
        constexpr uint32_t NV = D == 64 ? D + 16 : D;  // [V, 1] in one MMA when d = 64
        const uint32_t id_r = make_idesc(128, NV, true, true);
        const uint32_t id_r1 = make_idesc(128, 16, true, true);
        for (int i = 0; i < ntl && ok; ++i) {
          const int nV = 2 * i + 1;
          const uint32_t s_v = slot_addr(nV);
          const uint64_t dv = D == 64 ? make_desc(s_v, s_ones - s_v, 1024u, kSwizzle128) : desc_mnmajor(s_v, kTile, 0, 0);
          for (int h = 0; h < nb && ok; ++h) {
            const int c = i * nb + h, b = c & 1;
            if (!wait(S_PHK + b, (c >> 1) & 1)) break;
            if (h == 0) {
              if (!FAVOR) mbar_arrive(bar + S_EMPTY + slot_idx(2 * i));  // the MMA's share of the K slot
              if (!wait(S_FULL + slot_idx(nV), slot_par(nV))) break;
              if (i > 0 && !wait(S_INCFREE, (i - 1) & 1)) break;  // the last increment is added
            }
            tc_fence_after();
            const uint32_t t_r = tbase + t_inc + h * NC;
            const uint64_t da = desc_mnmajor(s_phk + b * kTile * 256, kTile, 0, 0);
#pragma unroll
            for (int s = 0; s < kTile / 16; ++s) {
              const uint64_t a = da + (uint64_t)(s * 128);
              mma_bf16(t_r, a, dv + (uint64_t)(s * 128), id_r, s > 0);
              if (D != 64) mma_bf16(t_r + D, a, desc_n16(s_ones, s), id_r1, s > 0);
            }
            mma_commit(bar + S_PHFREE + b);
          }
          if (!ok) break;
          mma_commit(bar + S_AFULL);
          mma_commit(bar + S_EMPTY + slot_idx(nV));
        }
      }
      mma_commit(bar + S_DONE + (warp - 1));
      mbar_drain(bar + S_DONE + (warp - 1), 0);
    }
  } else if (warp >= 4 && warp < 12) {
    // ---------------------------------------------------------------- phi_k
    const int part = (warp - 4) >> 2;  // columns [32 part, +32) of every 64-feature job
    int jobs = 0;
    for (int i = 0; i < ntl && ok; ++i) {
      const int t = t0 + i, n = 2 * i;
      const bool dead = row >= min(kTile, p.L - t * kTile);  // padding rows past L: features forced to zero
      const uint32_t s_k = slot_addr(n);
      if (!wait(S_FULL + slot_idx(n), slot_par(n))) break;
      float ck = 0.f;
      if (FAVOR) {
        // |k|^2 of the row: each of its two threads sums half of d
        float *nr = reinterpret_cast<float *>(smem + lay.nrm) + (i & 1) * 2 * kTile;
        nr[part * kTile + row] = tile_row_sqnorm_part(s_k, row, 32 * part, 32);
        named_barrier_sync(1, 256);
        // padding rows: F = 0 (zero-filled tile) and 2^-inf = 0, no select
        ck = dead ? -INFINITY : favor_row_const(nr[row] + nr[kTile + row], M);
      }
      for (int h = 0; h < nb && ok; ++h) {
        const int c = i * nb + h, b = c & 1;
        const uint32_t s_out = s_phk + b * kTile * 256;
        for (int half = 0; half < FB / 64; ++half) {
          float v[32];
          const int f0 = 64 * half + 32 * part;  // feature offset within the block
          if (FAVOR) {
            const int fb = jobs & 1;
            if (!wait(S_FFULL + fb, (jobs >> 1) & 1)) break;
            tc_fence_after();
            tmem_ld32(tmem_addr(tbase, lane_base, t_f + 64 * fb + 32 * part), v);
            tc_fence_before();
            arrive(S_FEMPTY + fb);
            ++jobs;
#pragma unroll
            for (int x = 0; x < 32; ++x) v[x] = favor_feature(v[x], ck);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              ld_bf16x8(s_k + sw128_offset(row, 128 * h + f0 + 8 * j, kTile), v + 8 * j);
#pragma unroll
              for (int x = 0; x < 8; ++x) v[8 * j + x] = dead ? 0.f : elu1_feature(v[8 * j + x]);
            }
          }
          // the buffer's last block has been read by its increment MMAs
          if (half == 0 && c >= 2 && !wait(S_PHFREE + b, ((c >> 1) - 1) & 1)) break;
#pragma unroll
          for (int j = 0; j < 4; ++j) st_bf16x8(s_out + sw128_offset(row, f0 + 8 * j, kTile), v + 8 * j);
        }
        if (!ok) break;
        fence_async_smem();
        arrive(S_PHK + b);
      }
      if (!ok) break;
      arrive(S_EMPTY + slot_idx(n));
    }
  } else if (warp >= 12) {
    // ---------------------------------------------------------------- master += increment
    float *lo = reinterpret_cast<float *>(smem + lay.lo);
    for (int i = 0; i < ntl && ok; ++i) {
      if (!wait(S_AFULL, i & 1)) break;
      tc_fence_after();
      // per block: the R columns in 32-column steps, then the chunk holding S
      for (int b = 0; b < nb; ++b) {
        const int f = 128 * b + row;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          float x[32], m[32];
          tmem_ld32x2(tmem_addr(tbase, lane_base, t_inc + b * NC + c), tmem_addr(tbase, lane_base, t_m + b * NC + c), x, m);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 s2 = __fadd2_rn(make_float2(m[e], m[e + 1]), make_float2(x[e], x[e + 1]));
            m[e] = s2.x;
            m[e + 1] = s2.y;
          }
          tmem_st16(tmem_addr(tbase, lane_base, t_m + b * NC + c), m);
          tmem_st16(tmem_addr(tbase, lane_base, t_m + b * NC + c + 16), m + 16);
        }
        float x[16], m[16];
        tmem_ld16x2(tmem_addr(tbase, lane_base, t_inc + b * NC + D), tmem_addr(tbase, lane_base, t_m + b * NC + D), x, m);
        const float ms = m[0], xs = x[0];
#pragma unroll
        for (int e = 0; e < 16; ++e) m[e] += x[e];
        if (f < M) {  // S is column 0 of the chunk at d: double-float
          float hs = ms, l = lo[f];
          df_add(hs, l, xs);
          lo[f] = l;
          m[0] = hs;
        }
        tmem_st16(tmem_addr(tbase, lane_base, t_m + b * NC + D), m);
      }
      // the increment's loads are complete (each load waits): its columns
      // are free for the next MMA.  The master's stores are waited for after
      // the release; only this thread rereads those columns, next tile
      tc_fence_before();
      arrive(S_INCFREE);
      tmem_st_wait();
      __syncwarp();
      if (lane == 0) mbar_arrive_n(bar + S_EMPTY + slot_idx(2 * i + 1), 2);  // V(t): 4 warps x 2
    }
  }

  // segment total of R' -> fp32 [M][D + 1] in the idle load slots (and phi_k
  // buffers), one coalesced bulk store each for the high and the low parts
  float *stage = reinterpret_cast<float *>(smem + lay.slots);
  const bool out = ok && !*abort_flag;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp >= 12 && out) {
    for (int k = 0; k < nb * NCH; ++k) {
      const int b = k / NCH, c = (k - b * NCH) * 16, f = 128 * b + row;
      float v[16];
      tmem_ld16(tmem_addr(tbase, lane_base, t_m + b * NC + c), v);
      if (f < M) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c + i <= D) stage[f * DP + c + i] = v[i];
      }
    }
  }
  fence_async_smem();
  __syncthreads();
  const size_t off = ((size_t)bh * p.P + seg) * (size_t)M * DP;
  if (tid == 0 && !*abort_flag) {
    bulk_store(p.states + off, sbase + lay.slots, (uint32_t)(M * DP * 4));
    tma_store_commit();
    tma_store_wait_read();
  }
  __syncthreads();
  if (!*abort_flag) {
    const float *lo = reinterpret_cast<const float *>(smem + lay.lo);
    for (int idx = tid; idx < M * DP; idx += kThreads) stage[idx] = (idx % DP == D) ? lo[idx / DP] : 0.f;
  }
  fence_async_smem();
  __syncthreads();
  if (tid == 0 && !*abort_flag) {
    bulk_store(p.states_lo + off, sbase + lay.slots, (uint32_t)(M * DP * 4));
    tma_store_commit();
    tma_store_wait_read();
  }
  if (warp == 0) tmem_dealloc(tbase, 512);
}

}  // namespace sw

template <int D, bool FAVOR, int MODE, int M>
cudaError_t launch_m(const Plan &pl, const Args &a, const CUtensorMap &mq, const CUtensorMap &mk,
                     const CUtensorMap &mv, const CUtensorMap *mz, int zero_mask, int nseg, const float *state_in,
                     cudaStream_t st) {
  Params p{};
  p.state_in = state_in;
  p.L = pl.L; p.M = pl.M; p.nt = pl.tc_tiles; p.P = pl.P; p.tps = pl.cps;
  p.H = pl.H; p.wstride = pl.wh > 1 ? pl.M * 64 : 0;
  p.zero_grads = mz != nullptr ? zero_mask : 0;
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
    const int smem = (int)sw::StateLayout<D, FAVOR, M>().total + 1024;
    auto kern = sw::tc_state_ws_kernel<D, FAVOR, M>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(nseg, pl.BH), sw::kThreads, smem, st>>>(mk, mv, mz ? mz[0] : mk, mz ? mz[1] : mk, mz ? mz[2] : mk, p);
  }
  return cudaGetLastError();
}

// M is a compile-time constant of the kernel: FAVOR+ with 64, 128 or 256
// features, elu+1 with M = d.
template <int D, bool FAVOR, int MODE>
cudaError_t launch(const Plan &pl, const Args &a, const CUtensorMap &mq, const CUtensorMap &mk,
                   const CUtensorMap &mv, const CUtensorMap *mz, int zero_mask, int nseg, const float *state_in,
                   cudaStream_t st) {
  if constexpr (!FAVOR) {
    return pl.M == D ? launch_m<D, FAVOR, MODE, D>(pl, a, mq, mk, mv, mz, zero_mask, nseg, state_in, st)
                     : cudaErrorInvalidValue;
  } else {
    if (pl.M == 64) return launch_m<D, FAVOR, MODE, 64>(pl, a, mq, mk, mv, mz, zero_mask, nseg, state_in, st);
    if (pl.M == 128) return launch_m<D, FAVOR, MODE, 128>(pl, a, mq, mk, mv, mz, zero_mask, nseg, state_in, st);
    if (pl.M == 256) return launch_m<D, FAVOR, MODE, 256>(pl, a, mq, mk, mv, mz, zero_mask, nseg, state_in, st);
    return cudaErrorInvalidValue;
  }
}

// W (fp32 [64][M], one per blockIdx.y) -> the bf16 [M][64] swizzled image
// of W^T that the kernels copy into shared memory as the K-major B operand of
// F = X W.
__global__ void prep_w_kernel(const float *__restrict__ w, __nv_bfloat16 *__restrict__ img, int M) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= M * 64) return;
  w += (size_t)blockIdx.y * M * 64;
  img += (size_t)blockIdx.y * M * 64;
  const int i = idx / M, m = idx - i * M;
  img[sw128_offset(m, i, M) / 2] = __float2bfloat16_rn(w[idx]);
}

cudaError_t prep_w(const Plan &pl, const Args &a, cudaStream_t st) {
  if (!pl.favor) return cudaSuccess;
  ProfScope ps("prep_w", st);
  const int n = pl.M * 64;
  prep_w_kernel<<<dim3((n + 255) / 256, pl.wh), 256, 0, st>>>(
      a.w, reinterpret_cast<__nv_bfloat16 *>(a.ws + pl.wimg_off), pl.M);
  return cudaGetLastError();
}

// Totals of R' over the first nseg segments, then their inclusive scan:
// states[s] = R' at the end of segment s, counting from `init` (the carried
// state of earlier rows, features-major, or NULL).  `exact`: the scan keeps
// the high and low parts (double-float), as the backward's reversal needs;
// the forward reads only the high parts of its incoming state, for which a
// plain fp32 scan of the high parts (a relative error of about 2^-24 per
// segment added) is enough and moves half the bytes.
template <int D, bool FAVOR>
cudaError_t segment_states(const Plan &pl, const Args &a, const CUtensorMap &mq,
                           const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap *mz, int zero_mask, int nseg,
                           bool exact, const float *init, cudaStream_t st) {
  cudaError_t e;
  {
    ProfScope ps("tc_segment_state", st);
    e = launch<D, FAVOR, MODE_STATE>(pl, a, mq, mk, mv, mz, zero_mask, nseg, nullptr, st);
    if (e != cudaSuccess) return e;
  }
  if (nseg > 1 || (nseg > 0 && init)) {
    ProfScope ps("scan_states", st);
    e = exact ? scan_states_df(pl, a.ws + pl.states_off, a.ws + pl.states_lo_off, nseg, 1, init, st)
              : scan_states_f32(pl, a.ws + pl.states_off, nseg, init, st);
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
  // carried state of earlier rows -> features-major, read by segment 0 and
  // the scan
  const float *init = nullptr;
  if (a.state_in) {
    float *fm = a.ws + pl.carry_off;
    e = emajor_to_fm(pl, a.state_in, fm, st);
    if (e != cudaSuccess) return e;
    init = fm;
  }
  // every segment's total when the final state is wanted, or when the
  // backward is to read the end states (kept exactly as double-float pairs
  // then), else all but the last
  const bool all = a.state_out != nullptr || a.keep_states;
  const int nseg = all ? pl.P : pl.P - 1;
  if (nseg > 0) {
    e = segment_states<D, FAVOR>(pl, a, mq, mk, mv, nullptr, 0, nseg, all, init, st);
    if (e != cudaSuccess) return e;
  }
  {
    ProfScope ps("tc_forward", st);
    e = launch<D, FAVOR, MODE_FWD>(pl, a, mq, mk, mv, nullptr, 0, pl.P, init, st);
    if (e != cudaSuccess) return e;
  }
  if (a.state_out)
    e = fm_to_emajor(pl, a.ws + pl.states_off, pl.P, pl.P - 1, a.ws + pl.states_lo_off, pl.P, pl.P - 1, a.state_out,
                     st);
  return e;
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

// The tensor path works on 128-row tiles whatever the slice size C: the
// slice recurrence is exact for any C (section 3.4), so C only changes the
// order of the roundings, and every supported C takes this path.
bool tc_forward_supported(int d, int M, int chunk, bool favor) {
  (void)chunk;
  if (d == 64) return favor ? (M == 64 || M == 128 || M == 256) : M == 64;
  if (d == 128) return !favor && M == 128;
  return false;
}

cudaError_t tc_segment_states(const Plan &p, const Args &a, int nseg, int zero_grads, const float *init,
                              cudaStream_t st) {
  CUtensorMap mk, mv, mz[3];
  const int d = p.d;
  cudaError_t e = tcf::prep_w(p, a, st);
  if (e != cudaSuccess) return e;
  if (!make_map_bf16_3d(&mk, a.k, p.BH, p.L, d, tcf::kTile) || !make_map_bf16_3d(&mv, a.v, p.BH, p.L, d, tcf::kTile))
    return cudaErrorInvalidValue;
  // dummies (never stored to) for the outputs left alone
  mz[0] = mz[1] = mz[2] = mk;
  void *const outs[3] = {a.dq, a.dk, a.dv};
  for (int o = 0; o < 3; ++o)
    if ((zero_grads >> o & 1) && !make_map_bf16_3d(&mz[o], outs[o], p.BH, p.L, d, tcf::kTile))
      return cudaErrorInvalidValue;
  const CUtensorMap *z = zero_grads ? mz : nullptr;
  if (d == 64 && p.favor) return tcf::segment_states<64, true>(p, a, mk, mk, mv, z, zero_grads, nseg, true, init, st);
  if (d == 64) return tcf::segment_states<64, false>(p, a, mk, mk, mv, z, zero_grads, nseg, true, init, st);
  if (d == 128 && !p.favor)
    return tcf::segment_states<128, false>(p, a, mk, mk, mv, z, zero_grads, nseg, true, init, st);
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
