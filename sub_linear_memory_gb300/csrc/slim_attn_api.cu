// slim_attn_api.cu -- the C ABI declared in include/slim_attn.h: argument
// validation, the segment plan, workspace layout and kernel dispatch.
#include <cuda_runtime.h>

#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "kernels.h"

namespace slim {

// Device status word: SLIM_OK, or the first device-side error recorded.
__device__ int g_device_status = 0;

namespace {

std::mutex g_mu;
void *g_ws = nullptr;
size_t g_ws_bytes = 0;
int g_opt_segments = 0;
int g_opt_path = 0;
int g_opt_w_per_head = 0;
int g_opt_reuse_states = 0;

// What the last forward with SLIM_OPT_REUSE_STATES left in the registered
// workspace: its inputs, shape and workspace, and the workspace generation
// (bumped by every call that writes the registered workspace's states).
struct StateTag {
  bool valid = false;
  const void *k = nullptr, *v = nullptr;
  const float *w = nullptr;
  int B = 0, H = 0, L = 0, d = 0, M = 0, chunk = 0, wh = 0, P = 0;
  const void *ws = nullptr;
  unsigned long long gen = 0;
};
StateTag g_tag;
unsigned long long g_ws_gen = 0;

// ---- per-kernel profiling ----
std::mutex g_prof_mu;
std::atomic<int> g_prof_on{0};
struct PendingEvent {
  const char *name;
  cudaEvent_t start, stop;
};
std::vector<PendingEvent> g_pending;
std::vector<cudaEvent_t> g_event_pool;
struct ProfTotal {
  long long launches = 0;
  double ms = 0.0;
};
std::vector<std::pair<std::string, ProfTotal>> g_prof_totals;

cudaEvent_t take_event() {
  cudaEvent_t e = nullptr;
  if (!g_event_pool.empty()) {
    e = g_event_pool.back();
    g_event_pool.pop_back();
  } else if (cudaEventCreate(&e) != cudaSuccess) {
    e = nullptr;
  }
  return e;
}

void fold_pending() {
  for (auto &pe : g_pending) {
    float ms = 0.f;
    if (cudaEventSynchronize(pe.stop) == cudaSuccess &&
        cudaEventElapsedTime(&ms, pe.start, pe.stop) == cudaSuccess) {
      auto it = g_prof_totals.begin();
      for (; it != g_prof_totals.end(); ++it)
        if (it->first == pe.name) break;
      if (it == g_prof_totals.end()) {
        g_prof_totals.emplace_back(pe.name, ProfTotal{});
        it = g_prof_totals.end() - 1;
      }
      it->second.launches += 1;
      it->second.ms += ms;
    }
    g_event_pool.push_back(pe.start);
    g_event_pool.push_back(pe.stop);
  }
  g_pending.clear();
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// The status a call returns once its work is enqueued.  Debug builds
// (-DSLIM_DEBUG) wait for the work and report device-side errors (a failed
// bounds check, a timed-out wait) from the call that caused them.
slim_status finish(cudaError_t err, cudaStream_t st) {
  if (err != cudaSuccess) return SLIM_ERR_CUDA;
#ifdef SLIM_DEBUG
  return slim_attn_sync_status((slim_stream_t)st);
#else
  (void)st;
  return SLIM_OK;
#endif
}

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

slim_status check_shape(int B, int H, int L, int d, int M, int chunk, bool favor) {
  if (B < 0 || H < 0 || L < 0 || d <= 0 || M <= 0 || chunk <= 0) return SLIM_ERR_INVALID_ARG;
  if (!favor && M != d) return SLIM_ERR_INVALID_ARG;
  if (!(d == 16 || d == 32 || d == 64 || d == 128)) return SLIM_ERR_UNSUPPORTED;
  if (M % 16 != 0 || M > 256) return SLIM_ERR_UNSUPPORTED;
  if (!pow2(chunk) || chunk < 16 || chunk > 256) return SLIM_ERR_UNSUPPORTED;
  if ((long long)B * H > (1LL << 30)) return SLIM_ERR_UNSUPPORTED;
  return SLIM_OK;
}

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 148;
  return sms;
}

// Segments per (b, h), never more than the work units (chunks, or 128-row
// tiles on the tensor path) and with no empty segment.  The CUDA-core path
// covers every SM once.  The tensor path runs one CTA per SM (cta_per_seg
// CTAs per segment), so it picks the count with the shortest makespan,
// waves x units per segment, preferring fewer segments on ties, and caps it
// at 8 waves' worth so the boundary states stay a bounded workspace.
// tail_w: work outside the main kernel that covers the rows of segments
// 0 .. P-2, in main-kernel tile times per tile and SM (the backward's
// correction of dK, dV by the later segments' reverse state).
// fwd_model: the tensor-path forward, whose segments each cost about two
// tiles' time more than their tiles (prologue, state and W loads, pipeline
// fill and drain), and whose segment-state pass runs segments 0 .. P-2 at
// about 0.4 of a forward tile per tile, with the same overhead.  Measured on
// the GB300: forward l4k 0.114 / 0.127 / 0.163 / 0.248 ms at P = 4 / 8 / 16 /
// 32 (the model's order and ratios within 5%), l32k best at P = 19.
// Makespan, in main-kernel tile times, of the tensor path cut into `segs`
// segments of `cps` units (the model choose_segments minimises).
double plan_span(int segs, int cps, int units, int bh, int cta_per_seg, double tail_w, bool fwd_model, int sms) {
  const long long waves = ((long long)segs * bh * cta_per_seg + sms - 1) / sms;
  if (fwd_model) {
    constexpr double kSegOverhead = 2.0, kStateTile = 0.4;
    const long long waves_s = ((long long)(segs - 1) * bh + sms - 1) / sms;
    return (double)waves * (cps + kSegOverhead) + kStateTile * (double)waves_s * (cps + kSegOverhead);
  }
  return (double)(waves * cps) + tail_w * (double)(segs - 1) / segs * (double)units * bh / sms;
}

void choose_segments(Plan &p, int requested, int units, int tensor_path, int cta_per_seg, double tail_w,
                     bool fwd_model = false) {
  const int sms = device_sms();
  const int bh = std::max(p.BH, 1);
  int P;
  if (requested > 0) {
    P = requested;
  } else if (!tensor_path) {
    P = (sms + bh - 1) / bh;
  } else {
    const int cap = std::max(1, 8 * ((sms + bh * cta_per_seg - 1) / (bh * cta_per_seg)));
    double best = -1.0;
    P = 1;
    for (int cand = 1; cand <= std::min(units, cap); ++cand) {
      const int cps = (units + cand - 1) / cand;
      const int segs = (units + cps - 1) / cps;
      const double span = plan_span(segs, cps, units, bh, cta_per_seg, tail_w, fwd_model, sms);
      if (best < 0.0 || span < best - 1e-9) {
        best = span;
        P = segs;
      }
    }
  }
  P = std::max(1, std::min(P, units));
  p.cps = (units + P - 1) / P;
  p.P = (units + p.cps - 1) / p.cps;
}

Plan make_plan(int B, int H, int L, int d, int M, int chunk, bool favor, bool bwd, bool want_dw,
               int path = 1) {
  Plan p{};
  p.B = B; p.H = H; p.L = L; p.d = d; p.M = M; p.C = chunk;
  p.BH = B * H;
  p.nchunks = (L + chunk - 1) / chunk;
  p.tc_tiles = (L + 127) / 128;
  p.favor = favor ? 1 : 0;
  p.wh = (favor && g_opt_w_per_head) ? H : 1;
  p.dp = d + 1;
  p.path = path;
  // the backward of 256 random features, and of elu+1 at d = 128, runs each
  // segment on a two-CTA cluster
  const int cta_per_seg = (path == 2 && bwd && (M > 128 || d == 128)) ? 2 : 1;
  // the tensor backward's correction pass: measured about a third of a
  // backward tile's time per tile and SM (l32k: 4.5 us against 13.2 us)
  const double tail_w = (path == 2 && bwd) ? 0.35 : 0.0;
  choose_segments(p, g_opt_segments, path == 2 ? p.tc_tiles : p.nchunks, path == 2, cta_per_seg, tail_w,
                  path == 2 && !bwd);
  // SLIM_OPT_REUSE_STATES: a tensor backward at d = 64 takes the forward's
  // segments when its own model puts them within 10% of its best, so that it
  // can read the forward's states (the state pass it skips is about a tenth of
  // its time; l32k measured 2.026 ms per step that way against 2.061 with
  // its own 7 segments and the forward's 9)
  if (path == 2 && bwd && d == 64 && g_opt_reuse_states && g_opt_segments == 0) {
    Plan f = p;
    choose_segments(f, 0, p.tc_tiles, 1, 1, 0.0, true);
    if (f.P != p.P) {
      const int sms = device_sms(), bh = std::max(p.BH, 1);
      const double own = plan_span(p.P, p.cps, p.tc_tiles, bh, cta_per_seg, tail_w, false, sms);
      const double theirs = plan_span(f.P, f.cps, p.tc_tiles, bh, cta_per_seg, tail_w, false, sms);
      if (theirs <= 1.1 * own) {
        p.P = f.P;
        p.cps = f.cps;
      }
    }
  }
  // master states: fp64 on the CUDA-core path; double-float (hi, lo) fp32
  // pairs on the tensor path, whose reverse states are plain fp32
  const size_t state = (path == 2 ? 1 : 2) * (size_t)p.BH * p.P * p.dp * p.M;
  size_t off = 0;
  p.states_off = off; off += align_floats(state);
  p.states_lo_off = off; if (path == 2) off += align_floats(state);
  // the W image next: at the same offset in a forward's and a backward's
  // layout of one shape and segment plan, so a backward on the forward's
  // states (SLIM_OPT_REUSE_STATES) reads its image too
  p.wimg_off = off; if (path == 2 && favor) off += align_floats((size_t)std::max(p.wh, 1) * M * 32);
  p.gstates_off = off; if (bwd) off += align_floats(state);
  p.scratch_stride = path == 2 ? 0 : align_floats(generic_scratch_floats(p, bwd));
  p.scratch_off = off; off += p.scratch_stride * p.BH * p.P;
  p.dwpart_off = off; if (bwd && want_dw) off += align_floats((size_t)p.BH * p.P * d * M);
  // bf16 G_end images [M][d] and fp32 G_S [M] per (head, segment)
  p.gimg_off = off; if (path == 2 && bwd) off += align_floats((size_t)p.BH * p.P * M * (d / 2 + 1));
  // carried states turned features-major: R'_0 and G (tensor path)
  p.carry_off = off; if (path == 2) off += align_floats((size_t)2 * p.BH * M * p.dp);
  p.total_floats = off;
  return p;
}

// Carried boundary states (fp32 e-major [B][H][d + 1][M] each, NULL = zero in
// / not wanted out): state_in, state_out (forward) and state_in, g_in, g_out
// (backward).
struct Carry {
  const float *state_in = nullptr;
  float *state_out = nullptr;
  const float *g_in = nullptr;
  float *g_out = nullptr;
  // a workspace for this call instead of the registered one (internal callers)
  float *ws = nullptr;
  size_t ws_bytes = 0;
  bool any() const { return state_in || state_out || g_in || g_out; }
};

// An NVTX range around one entry point (visible in Nsight timelines; free
// when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

template <typename T>
slim_status run(bool bwd, const void *q, const void *k, const void *v, const float *w,
                const void *dy, void *y, void *dq, void *dk, void *dv, float *dw, int B, int H,
                int L, int d, int M, int chunk, cudaStream_t stream, const Carry &c = Carry()) {
  NvtxRange range(bwd ? (sizeof(T) == 2 ? "slim_attn_bwd" : "slim_attn_bwd_f32")
                      : (sizeof(T) == 2 ? "slim_attn_fwd" : "slim_attn_fwd_f32"));
  const bool favor = w != nullptr;
  slim_status st = check_shape(B, H, L, d, M, chunk, favor);
  if (st != SLIM_OK) return st;
  if (!favor && dw) return SLIM_ERR_INVALID_ARG;
  if ((long long)B * H * L == 0) {
    const size_t dw_mats = g_opt_w_per_head ? (size_t)std::max(H, 0) : 1;
    if (dw && dw_mats && cudaMemsetAsync(dw, 0, sizeof(float) * dw_mats * d * M, stream) != cudaSuccess)
      return SLIM_ERR_CUDA;
    // no rows: the final state is the incoming one, and the gradient w.r.t. the
    // incoming state is the one arriving at the final state
    const size_t sbytes = sizeof(float) * (size_t)B * H * (d + 1) * M;
    const std::pair<float *, const float *> pass[2] = {{c.state_out, c.state_in}, {c.g_out, c.g_in}};
    for (const auto &pr : pass) {
      if (!pr.first || sbytes == 0) continue;
      const cudaError_t e = pr.second ? cudaMemcpyAsync(pr.first, pr.second, sbytes, cudaMemcpyDefault, stream)
                                      : cudaMemsetAsync(pr.first, 0, sbytes, stream);
      if (e != cudaSuccess) return SLIM_ERR_CUDA;
    }
    return SLIM_OK;
  }
  if (!q || !k || !v) return SLIM_ERR_INVALID_ARG;
  if (!bwd && !y) return SLIM_ERR_INVALID_ARG;
  if (bwd && (!dy || !dq || !dk || !dv)) return SLIM_ERR_INVALID_ARG;
  const bool io_ok = sizeof(T) == 2 && g_opt_path != 1 && aligned16(q) && aligned16(k) && aligned16(v);
  // the two-CTA elu+1 backward at d = 128 takes no carried state: such calls
  // run on the CUDA-core kernels
  const bool tc_bwd = tc_backward_supported(d, M, chunk, favor) &&
                      !(c.any() && tc_backward_elu128_supported(d, M, chunk, favor));
  const bool tc = io_ok && (bwd ? (tc_bwd && aligned16(dy) && aligned16(dq) && aligned16(dk) && aligned16(dv))
                                : (tc_forward_supported(d, M, chunk, favor) && aligned16(y)));
  Plan p = make_plan(B, H, L, d, M, chunk, favor, bwd, dw != nullptr, tc ? 2 : 1);
  Args a{};
  a.q = q; a.k = k; a.v = v; a.dy = dy; a.y = y; a.dq = dq; a.dk = dk; a.dv = dv;
  a.w = w; a.dw = dw;
  a.state_in = c.state_in;
  a.state_out = bwd ? nullptr : c.state_out;
  a.g_in = bwd ? c.g_in : nullptr;
  a.g_out = bwd ? c.g_out : nullptr;
  if (cudaGetSymbolAddress((void **)&a.status, g_device_status) != cudaSuccess) return SLIM_ERR_CUDA;
  // SLIM_OPT_REUSE_STATES: a forward on the registered workspace whose
  // segments are the ones the backward would choose tags the end states it
  // leaves there; a backward takes them when the tag matches its k, v, w,
  // shape, segments and workspace and no call has written the workspace since
  bool reuse = tc && d == 64 && !c.any() && !c.ws;
  if (reuse && !bwd) {
    const Plan pb = make_plan(B, H, L, d, M, chunk, favor, true, false, 2);
    reuse = pb.P == p.P && pb.cps == p.cps;
  }
  bool tag_it = false;
  if (c.ws) {
    if (c.ws_bytes < p.total_floats * sizeof(float)) return SLIM_ERR_WORKSPACE;
    a.ws = c.ws;
  } else {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ws || g_ws_bytes < p.total_floats * sizeof(float)) return SLIM_ERR_WORKSPACE;
    a.ws = static_cast<float *>(g_ws);
    const StateTag &t = g_tag;
    if (reuse && g_opt_reuse_states && bwd && t.valid && t.gen == g_ws_gen && t.ws == g_ws && t.k == k &&
        t.v == v && t.w == w && t.B == B && t.H == H && t.L == L && t.d == d && t.M == M && t.chunk == chunk &&
        t.wh == p.wh && t.P == p.P) {
      a.reuse_states = 1;  // reads the tagged states, writes none
    } else {
      ++g_ws_gen;
      g_tag.valid = false;
      if (reuse && g_opt_reuse_states && !bwd) {
        a.keep_states = 1;
        tag_it = true;
      }
    }
  }
  cudaError_t err = tc ? (bwd ? tc_backward(p, a, stream) : tc_forward(p, a, stream))
                      : (bwd ? generic_backward<T>(p, a, stream) : generic_forward<T>(p, a, stream));
  if (tag_it && err == cudaSuccess) {
    std::lock_guard<std::mutex> lk(g_mu);
    StateTag t;
    t.valid = true;
    t.k = k; t.v = v; t.w = w;
    t.B = B; t.H = H; t.L = L; t.d = d; t.M = M; t.chunk = chunk; t.wh = p.wh; t.P = p.P;
    t.ws = g_ws;
    t.gen = g_ws_gen;
    g_tag = t;
  }
  return finish(err, stream);
}

// State after all L rows of k, v (serving prefill), into the caller's fp32
// [B][H][d + 1][M] e-major buffer.
template <typename T>
slim_status run_state(const void *k, const void *v, const float *w, float *state, int B, int H, int L, int d,
                      int M, int chunk, cudaStream_t stream, float *ws_override = nullptr, size_t ws_bytes = 0) {
  NvtxRange range("slim_attn_state");
  const bool favor = w != nullptr;
  slim_status st = check_shape(B, H, L, d, M, chunk, favor);
  if (st != SLIM_OK) return st;
  if ((long long)B * H == 0) return SLIM_OK;
  if (!state) return SLIM_ERR_INVALID_ARG;
  if (L == 0) {
    const size_t bytes = sizeof(float) * (size_t)B * H * (d + 1) * M;
    return cudaMemsetAsync(state, 0, bytes, stream) == cudaSuccess ? SLIM_OK : SLIM_ERR_CUDA;
  }
  if (!k || !v) return SLIM_ERR_INVALID_ARG;
  const bool tc = sizeof(T) == 2 && g_opt_path != 1 && aligned16(k) && aligned16(v) &&
                  tc_forward_supported(d, M, chunk, favor);
  Plan p = make_plan(B, H, L, d, M, chunk, favor, false, false, tc ? 2 : 1);
  Args a{};
  a.k = k; a.v = v; a.w = w;
  if (cudaGetSymbolAddress((void **)&a.status, g_device_status) != cudaSuccess) return SLIM_ERR_CUDA;
  if (ws_override) {
    if (ws_bytes < p.total_floats * sizeof(float)) return SLIM_ERR_WORKSPACE;
    a.ws = ws_override;
  } else {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ws || g_ws_bytes < p.total_floats * sizeof(float)) return SLIM_ERR_WORKSPACE;
    a.ws = static_cast<float *>(g_ws);
    ++g_ws_gen;
    g_tag.valid = false;
  }
  cudaError_t err = tc ? tc_prefill_state(p, a, state, stream) : generic_prefill_state<T>(p, a, state, stream);
  return finish(err, stream);
}

// One new row per head against the carried state.
template <typename T>
slim_status run_decode(const void *q, const void *k, const void *v, const float *w, float *state, void *y, int B,
                       int H, int d, int M, cudaStream_t stream) {
  NvtxRange range("slim_attn_decode");
  const bool favor = w != nullptr;
  slim_status st = check_shape(B, H, 1, d, M, 64, favor);
  if (st != SLIM_OK) return st;
  if ((long long)B * H == 0) return SLIM_OK;
  if (!q || !k || !v || !state || !y) return SLIM_ERR_INVALID_ARG;
  const cudaError_t err = decode_step<T>(q, k, v, w, state, y, B * H, d, M, favor && g_opt_w_per_head ? H : 1, stream);
  return finish(err, stream);
}

}  // namespace

// The fp32 attention calls of the language-model driver (lm.cu), each on a
// workspace of its own.
slim_status attn_fwd_f32_ws(const float *q, const float *k, const float *v, const float *w, float *y,
                            const float *state_in, float *state_out, int B, int H, int L, int d, int M, int chunk,
                            float *ws, size_t ws_bytes, cudaStream_t st) {
  Carry c;
  c.state_in = state_in;
  c.state_out = state_out;
  c.ws = ws;
  c.ws_bytes = ws_bytes;
  return run<float>(false, q, k, v, w, nullptr, y, nullptr, nullptr, nullptr, nullptr, B, H, L, d, M, chunk, st, c);
}

slim_status attn_bwd_f32_ws(const float *q, const float *k, const float *v, const float *w, const float *dy,
                            float *dq, float *dk, float *dv, const float *state_in, const float *g_in, float *g_out,
                            int B, int H, int L, int d, int M, int chunk, float *ws, size_t ws_bytes,
                            cudaStream_t st) {
  Carry c;
  c.state_in = state_in;
  c.g_in = g_in;
  c.g_out = g_out;
  c.ws = ws;
  c.ws_bytes = ws_bytes;
  return run<float>(true, q, k, v, w, dy, nullptr, dq, dk, dv, nullptr, B, H, L, d, M, chunk, st, c);
}

slim_status attn_state_f32_ws(const float *k, const float *v, const float *w, float *state, int B, int H, int L,
                              int d, int M, int chunk, float *ws, size_t ws_bytes, cudaStream_t st) {
  return run_state<float>(k, v, w, state, B, H, L, d, M, chunk, st, ws, ws_bytes);
}

// Accessors for entry points that live in other translation units.
slim_status shape_status(int B, int H, int L, int d, int M, int chunk, bool favor) {
  return check_shape(B, H, L, d, M, chunk, favor);
}

Plan plan_for(int B, int H, int L, int d, int M, int chunk, bool favor, bool bwd, bool want_dw) {
  return make_plan(B, H, L, d, M, chunk, favor, bwd, want_dw);
}

int opt_w_per_head() {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_opt_w_per_head;
}

int *device_status_ptr() {
  int *ptr = nullptr;
  if (cudaGetSymbolAddress((void **)&ptr, g_device_status) != cudaSuccess) return nullptr;
  return ptr;
}

ProfScope::ProfScope(const char *name, cudaStream_t stream)
    : name_(name), stream_(stream), start_(nullptr) {
  if (!g_prof_on.load()) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t e = take_event();
  if (e && cudaEventRecord(e, stream) == cudaSuccess) start_ = e;
}

ProfScope::~ProfScope() {
  if (!start_) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t e = take_event();
  if (e && cudaEventRecord(e, stream_) == cudaSuccess) {
    g_pending.push_back(PendingEvent{name_, static_cast<cudaEvent_t>(start_), e});
  } else {
    g_event_pool.push_back(static_cast<cudaEvent_t>(start_));
    if (e) g_event_pool.push_back(e);
  }
}

}  // namespace slim

using slim::Carry;
using slim::run;
using slim::run_decode;
using slim::run_state;

extern "C" {

slim_status slim_attn_fwd(const void *q, const void *k, const void *v, const float *w, void *y,
                          int B, int H, int L, int d, int M, int chunk, slim_stream_t stream) {
  return run<__nv_bfloat16>(false, q, k, v, w, nullptr, y, nullptr, nullptr, nullptr, nullptr, B,
                            H, L, d, M, chunk, (cudaStream_t)stream);
}

slim_status slim_attn_bwd(const void *q, const void *k, const void *v, const float *w,
                          const void *dy, void *dq, void *dk, void *dv, float *dw, int B, int H,
                          int L, int d, int M, int chunk, slim_stream_t stream) {
  return run<__nv_bfloat16>(true, q, k, v, w, dy, nullptr, dq, dk, dv, dw, B, H, L, d, M, chunk,
                            (cudaStream_t)stream);
}

slim_status slim_attn_fwd_f32(const float *q, const float *k, const float *v, const float *w,
                              float *y, int B, int H, int L, int d, int M, int chunk,
                              slim_stream_t stream) {
  return run<float>(false, q, k, v, w, nullptr, y, nullptr, nullptr, nullptr, nullptr, B, H, L,
                    d, M, chunk, (cudaStream_t)stream);
}

slim_status slim_attn_bwd_f32(const float *q, const float *k, const float *v, const float *w,
                              const float *dy, float *dq, float *dk, float *dv, float *dw, int B,
                              int H, int L, int d, int M, int chunk, slim_stream_t stream) {
  return run<float>(true, q, k, v, w, dy, nullptr, dq, dk, dv, dw, B, H, L, d, M, chunk,
                    (cudaStream_t)stream);
}

slim_status slim_attn_fwd_carry(const void *q, const void *k, const void *v, const float *w, void *y,
                                const float *state_in, float *state_out, int B, int H, int L, int d, int M,
                                int chunk, slim_stream_t stream) {
  Carry c;
  c.state_in = state_in;
  c.state_out = state_out;
  return run<__nv_bfloat16>(false, q, k, v, w, nullptr, y, nullptr, nullptr, nullptr, nullptr, B, H, L, d, M,
                            chunk, (cudaStream_t)stream, c);
}

slim_status slim_attn_bwd_carry(const void *q, const void *k, const void *v, const float *w, const void *dy,
                                void *dq, void *dk, void *dv, float *dw, const float *state_in, const float *g_in,
                                float *g_out, int B, int H, int L, int d, int M, int chunk, slim_stream_t stream) {
  Carry c;
  c.state_in = state_in;
  c.g_in = g_in;
  c.g_out = g_out;
  return run<__nv_bfloat16>(true, q, k, v, w, dy, nullptr, dq, dk, dv, dw, B, H, L, d, M, chunk,
                            (cudaStream_t)stream, c);
}

slim_status slim_attn_fwd_carry_f32(const float *q, const float *k, const float *v, const float *w, float *y,
                                    const float *state_in, float *state_out, int B, int H, int L, int d, int M,
                                    int chunk, slim_stream_t stream) {
  Carry c;
  c.state_in = state_in;
  c.state_out = state_out;
  return run<float>(false, q, k, v, w, nullptr, y, nullptr, nullptr, nullptr, nullptr, B, H, L, d, M, chunk,
                    (cudaStream_t)stream, c);
}

slim_status slim_attn_bwd_carry_f32(const float *q, const float *k, const float *v, const float *w,
                                    const float *dy, float *dq, float *dk, float *dv, float *dw,
                                    const float *state_in, const float *g_in, float *g_out, int B, int H, int L,
                                    int d, int M, int chunk, slim_stream_t stream) {
  Carry c;
  c.state_in = state_in;
  c.g_in = g_in;
  c.g_out = g_out;
  return run<float>(true, q, k, v, w, dy, nullptr, dq, dk, dv, dw, B, H, L, d, M, chunk, (cudaStream_t)stream, c);
}

slim_status slim_attn_state(const void *k, const void *v, const float *w, float *state, int B, int H, int L,
                            int d, int M, int chunk, slim_stream_t stream) {
  return run_state<__nv_bfloat16>(k, v, w, state, B, H, L, d, M, chunk, (cudaStream_t)stream);
}

slim_status slim_attn_state_f32(const float *k, const float *v, const float *w, float *state, int B, int H,
                                int L, int d, int M, int chunk, slim_stream_t stream) {
  return run_state<float>(k, v, w, state, B, H, L, d, M, chunk, (cudaStream_t)stream);
}

slim_status slim_attn_decode(const void *q, const void *k, const void *v, const float *w, float *state, void *y,
                             int B, int H, int d, int M, slim_stream_t stream) {
  return run_decode<__nv_bfloat16>(q, k, v, w, state, y, B, H, d, M, (cudaStream_t)stream);
}

slim_status slim_attn_decode_f32(const float *q, const float *k, const float *v, const float *w, float *state,
                                 float *y, int B, int H, int d, int M, slim_stream_t stream) {
  return run_decode<float>(q, k, v, w, state, y, B, H, d, M, (cudaStream_t)stream);
}

size_t slim_attn_workspace_bytes(int B, int H, int L, int d, int M, int chunk, int is_bwd) {
  // the plan does not depend on the feature map: check the shape as FAVOR+
  // (which accepts every M that elu+1 does)
  if (slim::check_shape(B, H, L, d, M, chunk, true) != SLIM_OK) return 0;
  if ((long long)B * H * L == 0) return 0;
  size_t floats = 0;
  for (int path = 1; path <= 2; ++path) {
    slim::Plan p = slim::make_plan(B, H, L, d, M, chunk, true, is_bwd != 0, is_bwd != 0, path);
    floats = std::max(floats, p.total_floats);
  }
  return floats * sizeof(float);
}

slim_status slim_attn_set_workspace(void *ptr, size_t bytes) {
  if ((ptr == nullptr) != (bytes == 0)) return SLIM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ptr) % 256 != 0) return SLIM_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(slim::g_mu);
  if (ptr != slim::g_ws || bytes != slim::g_ws_bytes) {
    slim::g_tag.valid = false;
    ++slim::g_ws_gen;
  }
  slim::g_ws = ptr;
  slim::g_ws_bytes = bytes;
  return SLIM_OK;
}

slim_status slim_attn_set_option(int option, int value) {
  std::lock_guard<std::mutex> lk(slim::g_mu);
  switch (option) {
    case SLIM_OPT_SEGMENTS:
      if (value < 0) return SLIM_ERR_INVALID_ARG;
      slim::g_opt_segments = value;
      return SLIM_OK;
    case SLIM_OPT_PROFILE:
      slim::g_prof_on.store(value ? 1 : 0);
      return SLIM_OK;
    case SLIM_OPT_PATH:
      if (value < 0 || value > 2) return SLIM_ERR_INVALID_ARG;
      slim::g_opt_path = value;
      return SLIM_OK;
    case SLIM_OPT_W_PER_HEAD:
      if (value < 0 || value > 1) return SLIM_ERR_INVALID_ARG;
      slim::g_opt_w_per_head = value;
      return SLIM_OK;
    case SLIM_OPT_REUSE_STATES:
      if (value < 0 || value > 1) return SLIM_ERR_INVALID_ARG;
      slim::g_opt_reuse_states = value;
      slim::g_tag.valid = false;
      return SLIM_OK;
    default:
      return SLIM_ERR_INVALID_ARG;
  }
}

int slim_attn_segments(int B, int H, int L, int d, int M, int chunk) {
  if (slim::check_shape(B, H, L, d, M, chunk, true) != SLIM_OK) return 0;
  if ((long long)B * H * L == 0) return 0;
  // the bf16 forward's plan: the tensor path where either feature map has it
  const bool tc = slim::tc_forward_supported(d, M, chunk, true) || slim::tc_forward_supported(d, M, chunk, false);
  return slim::make_plan(B, H, L, d, M, chunk, true, false, false, tc ? 2 : 1).P;
}

int slim_attn_profile_count(void) {
  std::lock_guard<std::mutex> lk(slim::g_prof_mu);
  slim::fold_pending();
  return (int)slim::g_prof_totals.size();
}

slim_status slim_attn_profile_get(int i, const char **name, long long *launches, double *total_ms) {
  std::lock_guard<std::mutex> lk(slim::g_prof_mu);
  slim::fold_pending();
  if (i < 0 || i >= (int)slim::g_prof_totals.size()) return SLIM_ERR_INVALID_ARG;
  const auto &e = slim::g_prof_totals[i];
  if (name) *name = e.first.c_str();
  if (launches) *launches = e.second.launches;
  if (total_ms) *total_ms = e.second.ms;
  return SLIM_OK;
}

void slim_attn_profile_reset(void) {
  std::lock_guard<std::mutex> lk(slim::g_prof_mu);
  slim::fold_pending();
  slim::g_prof_totals.clear();
}

slim_status slim_attn_sync_status(slim_stream_t stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SLIM_ERR_CUDA;
  int host = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&host, slim::g_device_status, sizeof(int)) != cudaSuccess) return SLIM_ERR_CUDA;
  if (host != 0 && cudaMemcpyToSymbol(slim::g_device_status, &zero, sizeof(int)) != cudaSuccess)
    return SLIM_ERR_CUDA;
  return (slim_status)host;
}

const char *slim_status_string(slim_status status) {
  switch (status) {
    case SLIM_OK: return "SLIM_OK";
    case SLIM_ERR_INVALID_ARG: return "SLIM_ERR_INVALID_ARG: invalid argument";
    case SLIM_ERR_UNSUPPORTED: return "SLIM_ERR_UNSUPPORTED: shape or alignment not supported";
    case SLIM_ERR_WORKSPACE: return "SLIM_ERR_WORKSPACE: workspace missing or too small";
    case SLIM_ERR_CUDA: return "SLIM_ERR_CUDA: CUDA runtime error";
    case SLIM_ERR_TIMEOUT: return "SLIM_ERR_TIMEOUT: device-side wait gave up";
    case SLIM_ERR_BOUNDS: return "SLIM_ERR_BOUNDS: a debug-build bounds check failed";
    default: return "unknown slim_status";
  }
}

}  // extern "C"
