// api.cu -- the extern "C" entry points: validation, workspace layout, call order.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace invmoe {

namespace {
thread_local char g_last_error[512] = "";

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t route_ws(int T, int E) {
  const size_t NC = (static_cast<size_t>(T) + kDispatchChunk - 1) / kDispatchChunk;
  return align_up(NC * static_cast<size_t>(E) * sizeof(int32_t), 256);
}
size_t replay_ws(int T, int E, int k) {
  return route_ws(T, E) + align_up(static_cast<size_t>(T) * k * sizeof(int32_t), 256);
}
size_t ffn_ws(int T, int F_shared) { return align_up(static_cast<size_t>(T) * F_shared * 2, 256); }
size_t head_part_bytes(int T, int V) {
  const size_t NCH = (static_cast<size_t>(V) + kLseChunk - 1) / kLseChunk;
  return align_up(static_cast<size_t>(T) * NCH * sizeof(float2), 256);
}
size_t head_ws(int T, int V) { return head_part_bytes(T, V) + align_up(static_cast<size_t>(T) * 4, 256); }
// A head call on fewer than kHeadPadRows tokens reads its hidden rows from a copy in the workspace
// padded to kHeadPadRows rows (the GEMM's tensor map then spans 64 rows): measured faster on the
// GLM-scale head (V = 151552: 1 token 474-503 -> 307 us, 8 tokens 440 -> 309 us; 64 tokens take
// 308 us either way).  The rows past the batch are never stored; every row's bits are the same.
// (The same copy for the grouped expert GEMMs' token rows changed nothing and was not kept.)
constexpr int kHeadPadRows = 64;
size_t head_pad_bytes(int T, int H) {
  return T > 0 && T < kHeadPadRows ? align_up(static_cast<size_t>(kHeadPadRows) * H * 2, 256) : 0;
}

// Backward scratch, in this order after the status block (each part 256-byte aligned):
//   dh [T*k, F] fp32 | dgu [T*k, 2F] bf16 | h [T*k, F] bf16 |
//   dh_s [T, Fs] fp32 | dgu_s [T, 2Fs] bf16 | h_s [T, Fs] bf16 | dlog [T, E] bf16
struct BwdLayout {
  size_t dh, dgu, h, dh_s, dgu_s, h_s, dlog, end;
};
BwdLayout bwd_layout(int T, int E, int k, int F, int Fs) {
  BwdLayout L;
  const size_t S = static_cast<size_t>(T) * (k > 0 ? k : 0);
  size_t o = 0;
  L.dh = o;    o += align_up(S * F * 4, 256);
  L.dgu = o;   o += align_up(S * 2 * F * 2, 256);
  L.h = o;     o += align_up(S * F * 2, 256);
  L.dh_s = o;  o += align_up(static_cast<size_t>(T) * Fs * 4, 256);
  L.dgu_s = o; o += align_up(static_cast<size_t>(T) * 2 * Fs * 2, 256);
  L.h_s = o;   o += align_up(static_cast<size_t>(T) * Fs * 2, 256);
  L.dlog = o;  o += align_up(static_cast<size_t>(T) * (E > 0 ? E : 0) * 2, 256);
  L.end = o;
  return L;
}

unsigned int* status_word(void* ws) { return static_cast<unsigned int*>(ws); }
uint8_t* scratch(void* ws) { return static_cast<uint8_t*>(ws) + kStatusBytes; }
}  // namespace

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int check_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return INVMOE_OK;
  return set_error(INVMOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

namespace {
std::atomic<bool> g_pdl_on{true};
std::atomic<int> g_expert_engine{2};
std::atomic<int> g_shared_overlap{2};

// A stream of the library's own per device, and two events, on which moe_layer_forward runs
// the shared expert beside the routing and the routed experts.  Created on first use, never
// while the caller's stream is being captured into a graph; kept for the life of the process.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool ready = false;
};
std::mutex g_side_mu;
SideStream g_side[64];

// With g_side_mu held: this device's side stream, or null when there is none to use.
SideStream* side_stream_locked(cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) {
    cudaGetLastError();
    return nullptr;
  }
  SideStream& ss = g_side[dev];
  if (ss.ready) return &ss;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return nullptr;
  }
  if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    ss.s = nullptr;
    return nullptr;
  }
  if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    if (ss.fork) cudaEventDestroy(ss.fork);
    cudaStreamDestroy(ss.s);
    ss = SideStream{};
    return nullptr;
  }
  ss.ready = true;
  return &ss;
}
}  // namespace

bool pdl_enabled() { return g_pdl_on.load(std::memory_order_relaxed); }
int expert_engine() { return g_expert_engine.load(std::memory_order_relaxed); }

int device_sm_count(int* out) {
  static std::atomic<int> cache[64] = {};
  int dev = 0;
  int rc = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) {
      *out = c;
      return INVMOE_OK;
    }
  }
  int n = 0;
  rc = check_cuda(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute");
  if (rc) return rc;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  *out = n;
  return INVMOE_OK;
}

namespace {
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
std::atomic<bool> g_prof_on{false};
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t take_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}
}  // namespace

ProfScope::ProfScope(const char* name, cudaStream_t st) : idx_(-1), st_(st) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  ProfRec r{name, take_event(), take_event()};
  if (!r.a || !r.b) {
    // keep whichever event was obtained for later use
    if (r.a) g_prof_pool.push_back(r.a);
    if (r.b) g_prof_pool.push_back(r.b);
    return;
  }
  cudaEventRecord(r.a, st);
  g_prof_recs.push_back(r);
  idx_ = static_cast<long>(g_prof_recs.size()) - 1;
}

ProfScope::~ProfScope() {
  if (idx_ < 0) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (idx_ < static_cast<long>(g_prof_recs.size())) cudaEventRecord(g_prof_recs[idx_].b, st_);
}

// The shared expert: dense SwiGLU over all T tokens on the CTA-pair engine; the
// bf16 hidden activation [T, F_shared] lives in `hs` (workspace scratch).
// Router GEMM tiles: at most 64 tokens take the small-M kernel (one 64-expert tile per CTA, four
// K blocks per copy); otherwise 128 columns wide, or 64 when that still fits the whole GEMM in one
// wave of the SMs.  Neither the tile width nor the kernel changes a bit of a logit (the same M = 64
// MMA steps in the same K order for a tile of at most 64 tokens).
GemmVariant router_variant(int T, int E) {
  if (T <= 64) return GV_F32_SMALL64;
  if (E <= 64) return GV_F32_BN64_MT1;
  int sms = 0;
  if (device_sm_count(&sms) != INVMOE_OK) return GV_F32_BN128_MT1;
  const long long units64 = ((static_cast<long long>(T) + 127) / 128) * ((E + 63) / 64);
  return units64 <= sms ? GV_F32_BN64_MT1 : GV_F32_BN128_MT1;
}

int shared_expert_run(const void* x, const void* ws13, const void* ws2, int T, int H, int F_shared, float* y_shared,
                      void* hs, unsigned int* status, cudaStream_t st, int* sched) {
  // at most 64 tokens (decode): the small-M kernel, one 32-column tile of h (64 of y) per CTA and four K
  // blocks per copy; the same MMA steps, K order and SwiGLU expression as the CTA-pair engine
  const bool small = T <= 64 && F_shared % 32 == 0;
  GemmCall s1{};
  s1.name = "shared_gemm1_swiglu";
  s1.variant = small ? GV_SWIGLU_SMALL64 : GV_PAIR_SWIGLU;
  s1.A = x; s1.a_rows = T; s1.B = ws13; s1.b_rows = 2LL * F_shared; s1.K = H;
  s1.N = F_shared; s1.M = T; s1.G = 0; s1.b_group_rows = 0; s1.b_up_rows = F_shared;
  s1.out = hs; s1.ldo = F_shared; s1.status = status; s1.sched = sched;
  int rc = gemm_run(s1, st);
  if (rc) return rc;
  GemmCall s2{};
  s2.name = "shared_gemm2";
  s2.variant = small ? GV_F32_SMALL64 : GV_PAIR_F32;
  s2.A = hs; s2.a_rows = T; s2.B = ws2; s2.b_rows = H; s2.K = F_shared;
  s2.N = H; s2.M = T; s2.G = 0;
  s2.out = y_shared; s2.ldo = H; s2.status = status; s2.sched = sched;
  return gemm_run(s2, st);
}

}  // namespace invmoe

using namespace invmoe;

#define REQUIRE(cond, code, ...)             \
  do {                                       \
    if (!(cond)) return set_error(code, __VA_ARGS__); \
  } while (0)

#define REQUIRE_PTR(p) REQUIRE((p) != nullptr, INVMOE_ERR_INVALID_ARG, "%s is NULL", #p)
#define REQUIRE_ALIGNED(p) REQUIRE(aligned16(p), INVMOE_ERR_MISALIGNED, "%s is not 16-byte aligned", #p)

extern "C" {

int invmoe_version(void) { return 110; }

const char* invmoe_last_error(void) { return g_last_error; }

size_t invmoe_plan_len(int T, int E, int k) {
  if (T < 0 || E <= 0 || k <= 0) return 0;
  return static_cast<size_t>(2) * E + 1 + static_cast<size_t>(2) * T * k;
}

size_t invmoe_workspace_size(int T, int H, int E, int k, int F, int F_shared, int V) {
  (void)H; (void)F;
  if (T < 0) return 0;
  size_t need = 0;
  if (E > 0 && k > 0) need = replay_ws(T, E, k) > need ? replay_ws(T, E, k) : need;
  if (F_shared > 0) {
    // moe_layer_forward keeps the routing scratch and the shared expert's h apart (they run at once)
    const size_t w = ffn_ws(T, F_shared) + (E > 0 ? route_ws(T, E) : 0);
    need = w > need ? w : need;
  }
  if (V > 0) {
    const size_t w = head_ws(T, V) + (H > 0 ? head_pad_bytes(T, H) : 0);
    need = w > need ? w : need;
  }
  return kStatusBytes + need;
}

size_t invmoe_backward_workspace_size(int T, int H, int E, int k, int F, int F_shared) {
  (void)H;
  if (T < 0 || E < 0 || k < 0 || F < 0 || F_shared < 0) return 0;
  return kStatusBytes + bwd_layout(T, E, k, F, F_shared).end;
}

int invmoe_check(void* workspace, void* stream) {
  REQUIRE_PTR(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  int rc = check_cuda(cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st), "cudaMemcpyAsync");
  if (rc) return rc;
  if ((rc = check_cuda(cudaStreamSynchronize(st), "cudaStreamSynchronize"))) return rc;
  if (v != 0) {
    if ((rc = check_cuda(cudaMemsetAsync(workspace, 0, sizeof(v), st), "cudaMemsetAsync"))) return rc;
    if ((rc = check_cuda(cudaStreamSynchronize(st), "cudaStreamSynchronize"))) return rc;
    if (v & kStatusTimeout)
      return set_error(INVMOE_ERR_DEVICE_TIMEOUT, "a kernel's bounded wait ran out (status 0x%x)", v);
    if (v & kStatusBadCounts)
      return set_error(INVMOE_ERR_INVALID_ARG,
                       "expert-parallel regroup: the received row counts do not add up to R (status 0x%x)", v);
    return set_error(INVMOE_ERR_INVALID_ARG,
                     "router replay: an expert index was out of range or repeated within a token (status 0x%x)", v);
  }
  return INVMOE_OK;
}

int moe_route_topk(const void* x, const void* w_router, int T, int H, int E, int k, float* logits,
                   int32_t* topk_idx, float* topk_w, int32_t* plan, void* xp, void* workspace, size_t ws_bytes,
                   void* stream) {
  REQUIRE(T >= 0 && H > 0 && E > 0 && k > 0, INVMOE_ERR_INVALID_ARG, "need T >= 0, H, E, k > 0");
  REQUIRE(E <= 1024, INVMOE_ERR_UNSUPPORTED_SHAPE, "E=%d > 1024", E);
  REQUIRE(k <= E && k <= 32, INVMOE_ERR_INVALID_ARG, "need k <= min(E, 32) (k=%d, E=%d)", k, E);
  REQUIRE(H % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 64", H);
  REQUIRE_PTR(plan); REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= kStatusBytes + route_ws(T, E), INVMOE_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    return check_cuda(cudaMemsetAsync(plan, 0, (2 * static_cast<size_t>(E) + 1) * sizeof(int32_t), st),
                      "cudaMemsetAsync");
  }
  REQUIRE_PTR(x); REQUIRE_PTR(w_router); REQUIRE_PTR(logits); REQUIRE_PTR(topk_idx); REQUIRE_PTR(topk_w);
  REQUIRE_PTR(xp);
  REQUIRE_ALIGNED(x); REQUIRE_ALIGNED(w_router); REQUIRE_ALIGNED(logits); REQUIRE_ALIGNED(xp);
  REQUIRE_ALIGNED(workspace);

  GemmCall g{};
  g.name = "router_gemm";
  g.variant = router_variant(T, E);
  g.A = x; g.a_rows = T; g.B = w_router; g.b_rows = E; g.K = H; g.N = E; g.M = T; g.G = 0;
  g.out = logits; g.ldo = E; g.status = status_word(workspace);
  // the fp32 epilogue stores 4 columns at a time; E % 4 != 0 would need a scalar tail
  REQUIRE(E % 4 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "E=%d is not a multiple of 4", E);
  int rc = gemm_run(g, st);
  if (rc) return rc;
  return route_launch(logits, T, E, k, H, x, topk_idx, topk_w, plan, xp,
                      reinterpret_cast<int32_t*>(scratch(workspace)), st);
}

int moe_route_replay(const void* x, const void* w_router, const int32_t* topk_idx, int T, int H, int E, int k,
                     float* logits, float* topk_w, int32_t* plan, void* xp, void* workspace, size_t ws_bytes,
                     void* stream) {
  REQUIRE(T >= 0 && H > 0 && E > 0 && k > 0, INVMOE_ERR_INVALID_ARG, "need T >= 0, H, E, k > 0");
  REQUIRE(E <= 1024, INVMOE_ERR_UNSUPPORTED_SHAPE, "E=%d > 1024", E);
  REQUIRE(k <= E && k <= 32, INVMOE_ERR_INVALID_ARG, "need k <= min(E, 32) (k=%d, E=%d)", k, E);
  REQUIRE(H % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 64", H);
  REQUIRE(E % 4 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "E=%d is not a multiple of 4", E);
  REQUIRE_PTR(plan); REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= kStatusBytes + replay_ws(T, E, k), INVMOE_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    return check_cuda(cudaMemsetAsync(plan, 0, (2 * static_cast<size_t>(E) + 1) * sizeof(int32_t), st),
                      "cudaMemsetAsync");
  }
  REQUIRE_PTR(x); REQUIRE_PTR(w_router); REQUIRE_PTR(topk_idx); REQUIRE_PTR(logits); REQUIRE_PTR(topk_w);
  REQUIRE_PTR(xp);
  REQUIRE_ALIGNED(x); REQUIRE_ALIGNED(w_router); REQUIRE_ALIGNED(logits); REQUIRE_ALIGNED(xp);
  REQUIRE_ALIGNED(workspace);
  GemmCall g{};
  g.name = "router_gemm";
  g.variant = router_variant(T, E);
  g.A = x; g.a_rows = T; g.B = w_router; g.b_rows = E; g.K = H; g.N = E; g.M = T; g.G = 0;
  g.out = logits; g.ldo = E; g.status = status_word(workspace);
  int rc = gemm_run(g, st);
  if (rc) return rc;
  int32_t* counts = reinterpret_cast<int32_t*>(scratch(workspace));
  int32_t* idx_safe = reinterpret_cast<int32_t*>(scratch(workspace) + route_ws(T, E));
  return replay_launch(logits, topk_idx, T, E, k, H, x, idx_safe, topk_w, plan, xp, counts,
                       status_word(workspace), st);
}

int moe_grouped_ffn(const void* xp, const int32_t* plan, const void* w13, const void* w2, int T, int H, int E,
                    int k, int F, void* h, float* y, const void* x_shared, const void* ws13, const void* ws2,
                    int F_shared, float* y_shared, void* workspace, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0 && H > 0 && E > 0 && k > 0 && F > 0 && F_shared >= 0, INVMOE_ERR_INVALID_ARG, "bad sizes");
  REQUIRE(E <= 1024 && k <= E, INVMOE_ERR_INVALID_ARG, "need k <= E <= 1024");
  REQUIRE(H % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 64", H);
  REQUIRE(F % 128 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "F=%d is not a multiple of 128", F);
  REQUIRE(F_shared % 128 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "F_shared=%d is not a multiple of 128", F_shared);
  REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= kStatusBytes + (F_shared > 0 ? ffn_ws(T, F_shared) : 0), INVMOE_ERR_WORKSPACE_TOO_SMALL,
          "workspace too small");
  if (T == 0) return INVMOE_OK;
  REQUIRE_PTR(xp); REQUIRE_PTR(plan); REQUIRE_PTR(w13); REQUIRE_PTR(w2); REQUIRE_PTR(h); REQUIRE_PTR(y);
  REQUIRE_ALIGNED(xp); REQUIRE_ALIGNED(w13); REQUIRE_ALIGNED(w2); REQUIRE_ALIGNED(h); REQUIRE_ALIGNED(y);
  REQUIRE_ALIGNED(plan); REQUIRE_ALIGNED(workspace);
  if (F_shared > 0) {
    REQUIRE_PTR(x_shared); REQUIRE_PTR(ws13); REQUIRE_PTR(ws2); REQUIRE_PTR(y_shared);
    REQUIRE_ALIGNED(x_shared); REQUIRE_ALIGNED(ws13); REQUIRE_ALIGNED(ws2); REQUIRE_ALIGNED(y_shared);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long S = static_cast<long long>(T) * k;
  const int32_t* counts = plan;
  const int32_t* offsets = plan + E;
  unsigned int* status = status_word(workspace);

  // Engines (same bits either way): tokens on the MMA's M side in row tiles, or on its N side.
  // Measured on GB300 (same process, best of two; gate/up and down GEMM, token columns in the unit
  // size the batch takes vs row tiles), by token slots per expert on average:
  //   GLM-scale layer (H = 6144, F = 2048):   16: 1873 / 971 vs 1983 / 978 us;  32: 1902 / 990 vs
  //     2006 / 998;  64: 1976 / 1021 vs 1990 / 1029;  128: 2157 / 1192 vs 2113 / 1118;
  //     192: 2249 / 1291 vs 2267 / 1249;  256: 2595 / 1522 vs 2969 / 1610 (the row tiles stream an
  //     expert's weights again for its last few rows beyond 256);
  //   Qwen-like layer (H = 2048, F = 768, Zipf-skewed):  16: 138 / 85 vs 146 / 72;  32: 141 / 87 vs
  //     149 / 76;  64: 151 / 99 vs 158 / 80;  128: 170 / 113 vs 173 / 93;  256: 208 / 153 vs 225 / 131;
  //   one GLM-scale token 79 / 48 vs 113 / 57 us; tiny layer (H = 256) 15 / 14 vs 20 / 12 us.
  // So the gate/up GEMM always runs in token columns, and the down projection (whose fp32 epilogue
  // weighs more) in token columns for one wide decode token and, with a reduction of at least 32 K
  // blocks (F >= 2048), up to 64 slots per expert and from 256.
  const int eng = expert_engine();
  const bool tok1 = eng != 0;
  const bool tok2 = H % 256 == 0 &&
                    (eng == 1 || (eng == 2 && ((S <= 8 && H > 1024) ||
                                               (F >= 2048 && (S <= 64LL * E || S >= 256LL * E)))));
  GemmCall g1{};
  g1.name = "expert_gemm1_swiglu";
  g1.variant = tok1 ? GV_TOK_SWIGLU : GV_SWIGLU_BN256_MT2;
  g1.A = xp; g1.a_rows = S; g1.B = w13; g1.b_rows = static_cast<long long>(E) * 2 * F; g1.K = H;
  g1.N = F; g1.G = E; g1.counts = counts; g1.offsets = offsets; g1.b_group_rows = 2 * F; g1.b_up_rows = F;
  g1.out = h; g1.ldo = F; g1.status = status;
  int rc = gemm_run(g1, st);
  if (rc) return rc;

  GemmCall g2{};
  g2.name = "expert_gemm2";
  g2.variant = tok2 ? GV_TOK_F32 : GV_F32_BN256_MT2;
  g2.A = h; g2.a_rows = S; g2.B = w2; g2.b_rows = static_cast<long long>(E) * H; g2.K = F;
  g2.N = H; g2.G = E; g2.counts = counts; g2.offsets = offsets; g2.b_group_rows = H;
  g2.out = y; g2.ldo = H; g2.status = status;
  if ((rc = gemm_run(g2, st))) return rc;

  if (F_shared > 0)
    return shared_expert_run(x_shared, ws13, ws2, T, H, F_shared, y_shared, scratch(workspace), status, st);
  return INVMOE_OK;
}

int moe_layer_forward(const void* x, const void* w_router, const void* w13, const void* w2, const void* ws13,
                      const void* ws2, int T, int H, int E, int k, int F, int F_shared, float* logits,
                      int32_t* topk_idx, float* topk_w, int32_t* plan, void* xp, void* h, float* y, float* y_shared,
                      float* out, void* out_bf16, void* workspace, size_t ws_bytes, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The shared expert depends on x alone: with a large enough workspace it runs on the library's
  // side stream (its h after the routing scratch, its own unit counter) while the routing and the
  // routed experts run on `stream`; the combine waits for both.  Same kernels, same bits.
  const int mode = g_shared_overlap.load(std::memory_order_relaxed);
  const bool overlap = F_shared > 0 && T > 0 && E > 0 && (mode == 1 || (mode == 2 && T <= kSharedOverlapMaxT)) &&
                       workspace != nullptr && ws_bytes >= kStatusBytes + route_ws(T, E) + ffn_ws(T, F_shared);
  if (!overlap) {
    int rc = moe_route_topk(x, w_router, T, H, E, k, logits, topk_idx, topk_w, plan, xp, workspace, ws_bytes, stream);
    if (rc) return rc;
    rc = moe_grouped_ffn(xp, plan, w13, w2, T, H, E, k, F, h, y, x, ws13, ws2, F_shared, y_shared, workspace,
                         ws_bytes, stream);
    if (rc) return rc;
    return moe_combine(y, topk_w, plan, F_shared > 0 ? y_shared : nullptr, T, H, E, k, out, out_bf16, stream);
  }
  // everything the shared expert needs is checked before the fork, so no early return leaves it open
  REQUIRE(H > 0 && H % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 64", H);
  REQUIRE(F_shared % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "F_shared=%d is not a multiple of 64", F_shared);
  REQUIRE_PTR(x); REQUIRE_PTR(ws13); REQUIRE_PTR(ws2); REQUIRE_PTR(y_shared);
  REQUIRE_ALIGNED(x); REQUIRE_ALIGNED(ws13); REQUIRE_ALIGNED(ws2); REQUIRE_ALIGNED(y_shared);
  REQUIRE_ALIGNED(workspace);
  std::lock_guard<std::mutex> lock(g_side_mu);
  SideStream* ss = side_stream_locked(st);
  if (!ss) {
    int rc = moe_route_topk(x, w_router, T, H, E, k, logits, topk_idx, topk_w, plan, xp, workspace, ws_bytes, stream);
    if (rc) return rc;
    rc = moe_grouped_ffn(xp, plan, w13, w2, T, H, E, k, F, h, y, x, ws13, ws2, F_shared, y_shared, workspace,
                         ws_bytes, stream);
    if (rc) return rc;
    return moe_combine(y, topk_w, plan, y_shared, T, H, E, k, out, out_bf16, stream);
  }
  int rc = check_cuda(cudaEventRecord(ss->fork, st), "cudaEventRecord (fork)");
  if (rc) return rc;
  if ((rc = check_cuda(cudaStreamWaitEvent(ss->s, ss->fork, 0), "cudaStreamWaitEvent (fork)"))) return rc;
  unsigned int* status = status_word(workspace);
  int* side_sched = reinterpret_cast<int*>(reinterpret_cast<char*>(status) + 128);
  const int rc_side = shared_expert_run(x, ws13, ws2, T, H, F_shared, y_shared, scratch(workspace) + route_ws(T, E),
                                        status, ss->s, side_sched);
  rc = moe_route_topk(x, w_router, T, H, E, k, logits, topk_idx, topk_w, plan, xp, workspace, ws_bytes, stream);
  if (!rc)
    rc = moe_grouped_ffn(xp, plan, w13, w2, T, H, E, k, F, h, y, nullptr, nullptr, nullptr, 0, nullptr, workspace,
                         ws_bytes, stream);
  // the join is made whatever failed, so that `stream` (and a graph being captured) stays whole
  int rc_join = check_cuda(cudaEventRecord(ss->join, ss->s), "cudaEventRecord (join)");
  if (!rc_join) rc_join = check_cuda(cudaStreamWaitEvent(st, ss->join, 0), "cudaStreamWaitEvent (join)");
  if (rc_side) return rc_side;
  if (rc) return rc;
  if (rc_join) return rc_join;
  return moe_combine(y, topk_w, plan, y_shared, T, H, E, k, out, out_bf16, stream);
}

int moe_combine(const float* y, const float* topk_w, const int32_t* plan, const float* y_shared, int T, int H, int E,
                int k, float* out, void* out_bf16, void* stream) {
  REQUIRE(T >= 0 && H > 0 && E > 0 && k > 0 && k <= E, INVMOE_ERR_INVALID_ARG, "bad sizes");
  REQUIRE(H % 4 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 4", H);
  if (T == 0) return INVMOE_OK;
  REQUIRE_PTR(y); REQUIRE_PTR(topk_w); REQUIRE_PTR(plan); REQUIRE_PTR(out);
  REQUIRE_ALIGNED(y); REQUIRE_ALIGNED(out);
  if (y_shared) REQUIRE_ALIGNED(y_shared);
  if (out_bf16) REQUIRE(((uintptr_t)out_bf16 & 7u) == 0, INVMOE_ERR_MISALIGNED, "out_bf16 is not 8-byte aligned");
  const int32_t* slot_row = plan + 2 * E + 1 + static_cast<long long>(T) * k;
  return combine_launch(y, topk_w, slot_row, y_shared, T, H, k, out, out_bf16, static_cast<cudaStream_t>(stream));
}

int lm_logprob_kl(const void* hidden, const void* w_vocab, const int32_t* target, const float* rollout_logp, int T,
                  int H, int V, float beta, float* logits, float* logp, float* lse, float* k3, uint8_t* mask,
                  void* workspace, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0 && H > 0 && V > 0, INVMOE_ERR_INVALID_ARG, "bad sizes");
  REQUIRE(beta >= 1.0f, INVMOE_ERR_INVALID_ARG, "beta must be >= 1");
  REQUIRE(H % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 64", H);
  REQUIRE(V % 4 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "V=%d is not a multiple of 4", V);
  REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= kStatusBytes + head_ws(T, V), INVMOE_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  if (T == 0) return INVMOE_OK;
  REQUIRE_PTR(hidden); REQUIRE_PTR(w_vocab); REQUIRE_PTR(target); REQUIRE_PTR(logp);
  REQUIRE_ALIGNED(hidden); REQUIRE_ALIGNED(w_vocab); REQUIRE_ALIGNED(workspace);
  if (logits) REQUIRE_ALIGNED(logits);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float2* part = reinterpret_cast<float2*>(scratch(workspace));
  float* tgt_logit = reinterpret_cast<float*>(scratch(workspace) + head_part_bytes(T, V));
  const void* A = hidden;
  long long a_rows = T;
  if (head_pad_bytes(T, H) > 0 && ws_bytes >= kStatusBytes + head_ws(T, V) + head_pad_bytes(T, H)) {
    void* pad = scratch(workspace) + head_ws(T, V);
    int rc = check_cuda(cudaMemcpyAsync(pad, hidden, static_cast<size_t>(T) * H * 2, cudaMemcpyDeviceToDevice, st),
                        "cudaMemcpyAsync (head rows)");
    if (rc) return rc;
    A = pad;
    a_rows = kHeadPadRows;
  }
  GemmCall g{};
  g.name = "lm_head_gemm_lse";
  g.variant = GV_PAIR_LSE;
  g.A = A; g.a_rows = a_rows; g.B = w_vocab; g.b_rows = V; g.K = H; g.N = V; g.M = T; g.G = 0;
  // column-block-major in bands of 16 row chunks (4096 tokens, 50 MB of hidden
  // states at H = 6144): the band stays in L2 while every vocabulary tile streams past
  g.n_major = 1; g.m_group = 16; g.out = logits; g.ldo = V; g.status = status_word(workspace);
  g.part = part; g.target = target; g.tgt_logit = tgt_logit;
  int rc = gemm_run(g, st);
  if (rc) return rc;
  const int NCH = (V + kLseChunk - 1) / kLseChunk;
  return lse_merge_launch(part, NCH, NCH, 0, tgt_logit, 0, target, rollout_logp, T, V, beta, logp, lse, k3, mask,
                          st);
}

int lm_logprob_partials(const void* hidden, const void* w_vocab_shard, const int32_t* target, int T, int H, int V,
                        int v0, int v1, float* logits, float* partials, long long ld_part, float* tgt_logit,
                        void* workspace, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0 && H > 0 && V > 0, INVMOE_ERR_INVALID_ARG, "bad sizes");
  REQUIRE(H % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 64", H);
  REQUIRE(V % 4 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "V=%d is not a multiple of 4", V);
  REQUIRE(0 <= v0 && v0 < v1 && v1 <= V, INVMOE_ERR_INVALID_ARG, "need 0 <= v0 < v1 <= V (v0=%d, v1=%d, V=%d)", v0,
          v1, V);
  REQUIRE(v0 % kLseChunk == 0 && (v1 == V || v1 % kLseChunk == 0), INVMOE_ERR_INVALID_ARG,
          "a vocabulary shard must start and end on a %d-column chunk boundary (v0=%d, v1=%d)", kLseChunk, v0, v1);
  const int nch_shard = (v1 - v0 + kLseChunk - 1) / kLseChunk;
  REQUIRE(ld_part >= nch_shard, INVMOE_ERR_INVALID_ARG, "ld_part=%lld < the shard's %d chunks", ld_part, nch_shard);
  REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= kStatusBytes, INVMOE_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  if (T == 0) return INVMOE_OK;
  REQUIRE_PTR(hidden); REQUIRE_PTR(w_vocab_shard); REQUIRE_PTR(target); REQUIRE_PTR(partials);
  REQUIRE_PTR(tgt_logit);
  REQUIRE_ALIGNED(hidden); REQUIRE_ALIGNED(w_vocab_shard); REQUIRE_ALIGNED(workspace);
  REQUIRE((reinterpret_cast<uintptr_t>(partials) & 7u) == 0, INVMOE_ERR_MISALIGNED, "partials is not 8-byte aligned");
  if (logits) REQUIRE_ALIGNED(logits);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  GemmCall g{};
  g.name = "lm_head_gemm_lse";
  g.variant = GV_PAIR_LSE;
  g.A = hidden; g.a_rows = T; g.B = w_vocab_shard; g.b_rows = v1 - v0; g.K = H; g.N = v1 - v0; g.M = T; g.G = 0;
  // the unsharded call's order: column-block-major in bands of 16 row chunks
  g.n_major = 1; g.m_group = 16; g.out = logits ? logits + v0 : nullptr; g.ldo = V;
  g.status = status_word(workspace);
  g.part = reinterpret_cast<float2*>(partials); g.part_ld = ld_part; g.target_col0 = v0;
  g.target = target; g.tgt_logit = tgt_logit;
  return gemm_run(g, st);
}

int lm_logprob_merge(const float* partials, long long ld_part, int shard_chunks, long long shard_stride,
                     const float* tgt_logit, long long tgt_stride, const int32_t* target, const float* rollout_logp,
                     int T, int V, float beta, float* logp, float* lse, float* k3, uint8_t* mask, void* stream) {
  REQUIRE(T >= 0 && V > 0, INVMOE_ERR_INVALID_ARG, "bad sizes");
  REQUIRE(beta >= 1.0f, INVMOE_ERR_INVALID_ARG, "beta must be >= 1");
  REQUIRE(shard_chunks >= 1 && ld_part >= 1 && shard_stride >= 0 && tgt_stride >= 0, INVMOE_ERR_INVALID_ARG,
          "need shard_chunks >= 1, ld_part >= 1, shard_stride >= 0, tgt_stride >= 0");
  const int NCH = (V + kLseChunk - 1) / kLseChunk;
  REQUIRE(ld_part >= (shard_chunks < NCH ? shard_chunks : NCH), INVMOE_ERR_INVALID_ARG,
          "ld_part=%lld is shorter than a shard's row of chunks", ld_part);
  REQUIRE(shard_chunks >= NCH || shard_stride >= static_cast<long long>(T) * ld_part, INVMOE_ERR_INVALID_ARG,
          "shard_stride=%lld overlaps the previous shard's rows", shard_stride);
  REQUIRE(shard_chunks >= NCH || tgt_stride >= T, INVMOE_ERR_INVALID_ARG,
          "tgt_stride=%lld overlaps the previous shard's target logits", tgt_stride);
  if (T == 0) return INVMOE_OK;
  REQUIRE_PTR(partials); REQUIRE_PTR(tgt_logit); REQUIRE_PTR(target); REQUIRE_PTR(logp);
  REQUIRE((reinterpret_cast<uintptr_t>(partials) & 7u) == 0, INVMOE_ERR_MISALIGNED, "partials is not 8-byte aligned");
  return lse_merge_launch(reinterpret_cast<const float2*>(partials), ld_part, shard_chunks, shard_stride, tgt_logit,
                          tgt_stride, target, rollout_logp, T, V, beta, logp, lse, k3, mask,
                          static_cast<cudaStream_t>(stream));
}

int moe_shared_expert(const void* x, const void* ws13, const void* ws2, int T, int H, int F_shared, float* y_shared,
                      void* workspace, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0 && H > 0 && F_shared > 0, INVMOE_ERR_INVALID_ARG, "bad sizes");
  REQUIRE(H % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 64", H);
  REQUIRE(F_shared % 128 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "F_shared=%d is not a multiple of 128", F_shared);
  REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= kStatusBytes + ffn_ws(T, F_shared), INVMOE_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  if (T == 0) return INVMOE_OK;
  REQUIRE_PTR(x); REQUIRE_PTR(ws13); REQUIRE_PTR(ws2); REQUIRE_PTR(y_shared);
  REQUIRE_ALIGNED(x); REQUIRE_ALIGNED(ws13); REQUIRE_ALIGNED(ws2); REQUIRE_ALIGNED(y_shared);
  REQUIRE_ALIGNED(workspace);
  return shared_expert_run(x, ws13, ws2, T, H, F_shared, y_shared, scratch(workspace), status_word(workspace),
                           static_cast<cudaStream_t>(stream));
}

int moe_ep_regroup(const void* recv_xp, const int32_t* recv_counts, int n_src, int E_local, int R, int H,
                   void* xp_local, int32_t* plan_local, int32_t* row_src, void* workspace, size_t ws_bytes,
                   void* stream) {
  REQUIRE(n_src >= 1 && E_local >= 1 && R >= 0 && H > 0, INVMOE_ERR_INVALID_ARG, "bad sizes");
  REQUIRE(E_local <= 1024, INVMOE_ERR_UNSUPPORTED_SHAPE, "E_local=%d > 1024", E_local);
  REQUIRE(static_cast<long long>(n_src) * E_local <= 65535, INVMOE_ERR_UNSUPPORTED_SHAPE,
          "n_src * E_local = %lld > 65535", static_cast<long long>(n_src) * E_local);
  REQUIRE(H % 8 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 8", H);
  REQUIRE_PTR(recv_counts); REQUIRE_PTR(plan_local); REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= kStatusBytes, INVMOE_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  if (R > 0) {
    REQUIRE_PTR(recv_xp); REQUIRE_PTR(xp_local); REQUIRE_PTR(row_src);
    REQUIRE_ALIGNED(recv_xp); REQUIRE_ALIGNED(xp_local);
  }
  return ep_regroup_launch(recv_xp, recv_counts, n_src, E_local, R, H, xp_local, plan_local, row_src,
                           status_word(workspace), static_cast<cudaStream_t>(stream));
}

int moe_ep_ungroup(const float* y_local, const int32_t* row_src, int R, int H, float* y_send, void* stream) {
  REQUIRE(R >= 0 && H > 0, INVMOE_ERR_INVALID_ARG, "bad sizes");
  REQUIRE(H % 4 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 4", H);
  if (R == 0) return INVMOE_OK;
  REQUIRE_PTR(y_local); REQUIRE_PTR(row_src); REQUIRE_PTR(y_send);
  REQUIRE_ALIGNED(y_local); REQUIRE_ALIGNED(y_send);
  return ep_ungroup_launch(y_local, row_src, R, H, y_send, static_cast<cudaStream_t>(stream));
}

int lm_head_backward(const void* hidden, const void* w_vocab, const int32_t* target, const float* lse,
                     const float* grad_logp, int T, int H, int V, void* dlogits, float* d_hidden, float* d_wvocab,
                     void* workspace, size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0 && H > 0 && V > 0, INVMOE_ERR_INVALID_ARG, "bad sizes");
  REQUIRE(H % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 64", H);
  REQUIRE(V % 8 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "V=%d is not a multiple of 8", V);
  REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= kStatusBytes, INVMOE_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  if (T == 0) {
    // no token: d_wvocab is a sum over nothing
    if (d_wvocab != nullptr)
      return check_cuda(cudaMemsetAsync(d_wvocab, 0, static_cast<size_t>(V) * H * sizeof(float),
                                        static_cast<cudaStream_t>(stream)),
                        "cudaMemsetAsync");
    return INVMOE_OK;
  }
  REQUIRE_PTR(hidden); REQUIRE_PTR(w_vocab); REQUIRE_PTR(target); REQUIRE_PTR(lse); REQUIRE_PTR(grad_logp);
  REQUIRE_PTR(dlogits);
  REQUIRE_ALIGNED(hidden); REQUIRE_ALIGNED(w_vocab); REQUIRE_ALIGNED(workspace); REQUIRE_ALIGNED(dlogits);
  if (d_hidden) REQUIRE_ALIGNED(d_hidden);
  if (d_wvocab) REQUIRE_ALIGNED(d_wvocab);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // dz: the forward's vocabulary projection (same engine, tile and order) with the gradient epilogue
  GemmCall g{};
  g.name = "lm_head_dlogits";
  g.variant = GV_PAIR_DLOGITS;
  g.A = hidden; g.a_rows = T; g.B = w_vocab; g.b_rows = V; g.K = H; g.N = V; g.M = T; g.G = 0;
  g.n_major = 1; g.m_group = 16; g.out = dlogits; g.ldo = V; g.status = status_word(workspace);
  g.target = target; g.row_lse = lse; g.row_scale = grad_logp;
  int rc = gemm_run(g, st);
  if (rc) return rc;
  if (d_hidden) {
    // d_hidden = dz [T, V] (K-major) x w_vocab [V, H] (MN-major); a row chunk's
    // column blocks are consecutive units, so they stream the same dz rows together
    GemmCall b{};
    b.name = "lm_head_dhidden";
    b.variant = GV_PAIR_F32_BMN;
    b.A = dlogits; b.a_rows = T; b.B = w_vocab; b.b_rows = H; b.K = V; b.N = H; b.M = T; b.G = 0;
    b.out = d_hidden; b.ldo = H; b.status = status_word(workspace);
    if ((rc = gemm_run(b, st))) return rc;
  }
  if (d_wvocab) {
    // d_wvocab = dz^T: dz [T, V] read MN-major as a [V x T] operand, hidden [T, H] MN-major
    GemmCall w{};
    w.name = "lm_head_dwvocab";
    w.variant = GV_PAIR_F32_AMN_BMN;
    w.A = dlogits; w.a_rows = V; w.B = hidden; w.b_rows = H; w.K = T; w.N = H; w.M = V; w.G = 0;
    w.out = d_wvocab; w.ldo = H; w.status = status_word(workspace);
    if ((rc = gemm_run(w, st))) return rc;
  }
  return INVMOE_OK;
}

int moe_combine_backward(const float* dout, const float* y, const float* topk_w, const int32_t* plan, int T, int H,
                         int E, int k, void* dy, float* dgate, void* dout_bf16, void* stream) {
  REQUIRE(T >= 0 && H > 0 && E > 0 && k > 0 && k <= E && k <= 32, INVMOE_ERR_INVALID_ARG, "bad sizes");
  REQUIRE(H % 4 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 4", H);
  if (T == 0) return INVMOE_OK;
  REQUIRE_PTR(dout); REQUIRE_PTR(y); REQUIRE_PTR(topk_w); REQUIRE_PTR(plan); REQUIRE_PTR(dy); REQUIRE_PTR(dgate);
  REQUIRE_ALIGNED(dout); REQUIRE_ALIGNED(y);
  REQUIRE(((uintptr_t)dy & 7u) == 0, INVMOE_ERR_MISALIGNED, "dy is not 8-byte aligned");
  if (dout_bf16) REQUIRE(((uintptr_t)dout_bf16 & 7u) == 0, INVMOE_ERR_MISALIGNED, "dout_bf16 is not 8-byte aligned");
  const int32_t* slot_row = plan + 2 * E + 1 + static_cast<long long>(T) * k;
  return combine_bwd_launch(dout, y, topk_w, slot_row, T, H, k, dy, dgate, dout_bf16,
                            static_cast<cudaStream_t>(stream));
}

int moe_grouped_ffn_backward(const void* xp, const int32_t* plan, const void* w13, const void* w2, const void* dy,
                             int T, int H, int E, int k, int F, float* dxp, float* dw13, float* dw2,
                             const void* x_shared, const void* ws13, const void* ws2, const void* dout_bf16,
                             int F_shared, float* dx_shared, float* dws13, float* dws2, void* workspace,
                             size_t ws_bytes, void* stream) {
  REQUIRE(T >= 0 && H > 0 && E > 0 && k > 0 && k <= E && F > 0 && F_shared >= 0, INVMOE_ERR_INVALID_ARG,
          "bad sizes");
  REQUIRE(E <= 1024, INVMOE_ERR_UNSUPPORTED_SHAPE, "E=%d > 1024", E);
  REQUIRE(H % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 64", H);
  REQUIRE(F % 128 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "F=%d is not a multiple of 128", F);
  REQUIRE(F_shared % 128 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "F_shared=%d is not a multiple of 128", F_shared);
  REQUIRE_PTR(workspace);
  const BwdLayout L = bwd_layout(T, E, k, F, F_shared);
  REQUIRE(ws_bytes >= kStatusBytes + L.end, INVMOE_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  REQUIRE_ALIGNED(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    // no token: the weight gradients are sums over nothing
    int rc = INVMOE_OK;
    if (dw13) rc = check_cuda(cudaMemsetAsync(dw13, 0, static_cast<size_t>(E) * 2 * F * H * 4, st), "memset");
    if (!rc && dw2) rc = check_cuda(cudaMemsetAsync(dw2, 0, static_cast<size_t>(E) * H * F * 4, st), "memset");
    if (!rc && F_shared && dws13)
      rc = check_cuda(cudaMemsetAsync(dws13, 0, static_cast<size_t>(2) * F_shared * H * 4, st), "memset");
    if (!rc && F_shared && dws2)
      rc = check_cuda(cudaMemsetAsync(dws2, 0, static_cast<size_t>(H) * F_shared * 4, st), "memset");
    return rc;
  }
  REQUIRE_PTR(xp); REQUIRE_PTR(plan); REQUIRE_PTR(w13); REQUIRE_PTR(w2); REQUIRE_PTR(dy); REQUIRE_PTR(dxp);
  REQUIRE_ALIGNED(xp); REQUIRE_ALIGNED(w13); REQUIRE_ALIGNED(w2); REQUIRE_ALIGNED(dy); REQUIRE_ALIGNED(dxp);
  if (dw13) REQUIRE_ALIGNED(dw13);
  if (dw2) REQUIRE_ALIGNED(dw2);
  if (F_shared) {
    REQUIRE_PTR(x_shared); REQUIRE_PTR(ws13); REQUIRE_PTR(ws2); REQUIRE_PTR(dout_bf16); REQUIRE_PTR(dx_shared);
    REQUIRE_ALIGNED(x_shared); REQUIRE_ALIGNED(ws13); REQUIRE_ALIGNED(ws2); REQUIRE_ALIGNED(dout_bf16);
    REQUIRE_ALIGNED(dx_shared);
    if (dws13) REQUIRE_ALIGNED(dws13);
    if (dws2) REQUIRE_ALIGNED(dws2);
  }
  uint8_t* sc = scratch(workspace);
  float* dh = reinterpret_cast<float*>(sc + L.dh);
  void* dgu = sc + L.dgu;
  void* h = sc + L.h;
  const long long S = static_cast<long long>(T) * k;
  const int* counts = plan;
  const int* offsets = plan + E;
  unsigned int* status = status_word(workspace);
  int rc;
  // dh = dy W2_e (group e's W2 is the stored rows [e*H, (e+1)*H) of w2 viewed as [E*H, F])
  {
    GemmCall g{};
    g.name = "expert_dh";
    g.variant = GV_F32_BN256_MT2_BMN;
    g.A = dy; g.a_rows = S; g.B = w2; g.b_rows = F; g.b_outer = static_cast<long long>(E) * H;
    g.K = H; g.N = F; g.G = E; g.counts = counts; g.offsets = offsets; g.b_group_rows = H;
    g.out = dh; g.ldo = F; g.status = status;
    if ((rc = gemm_run(g, st))) return rc;
  }
  // gate/up recomputed from xp (the forward's tile and K order), SwiGLU backward in the epilogue
  {
    GemmCall g{};
    g.name = "expert_swiglu_bwd";
    g.variant = GV_PAIR_SWIGLU_BWD;
    g.A = xp; g.a_rows = S; g.B = w13; g.b_rows = static_cast<long long>(E) * 2 * F;
    g.K = H; g.N = F; g.G = E; g.counts = counts; g.offsets = offsets; g.b_group_rows = 2 * F; g.b_up_rows = F;
    g.out = dgu; g.ldo = 2 * F; g.out2 = h; g.ldo2 = F; g.aux = dh; g.ld_aux = F; g.status = status;
    if ((rc = gemm_run(g, st))) return rc;
  }
  // dxp = [dg, du] W13_e
  {
    GemmCall g{};
    g.name = "expert_dx";
    g.variant = GV_F32_BN256_MT2_BMN;
    g.A = dgu; g.a_rows = S; g.B = w13; g.b_rows = H; g.b_outer = static_cast<long long>(E) * 2 * F;
    g.K = 2 * F; g.N = H; g.G = E; g.counts = counts; g.offsets = offsets; g.b_group_rows = 2 * F;
    g.out = dxp; g.ldo = H; g.status = status;
    if ((rc = gemm_run(g, st))) return rc;
  }
  // weight gradients over each expert's own rows
  if (dw2) {
    GemmCall g{};
    g.name = "expert_dw2";
    g.variant = GV_F32_BN256_MT1_KGROUP;
    g.kgroup = 1;
    g.A = dy; g.a_rows = H; g.a_outer = S; g.B = h; g.b_rows = F; g.b_outer = S;
    g.K = 1; g.M = H; g.N = F; g.G = E; g.counts = counts; g.offsets = offsets;
    g.out = dw2; g.ldo = F; g.status = status;
    if ((rc = gemm_run(g, st))) return rc;
  }
  if (dw13) {
    GemmCall g{};
    g.name = "expert_dw13";
    g.variant = GV_F32_BN256_MT1_KGROUP;
    g.kgroup = 1;
    g.A = dgu; g.a_rows = 2 * F; g.a_outer = S; g.B = xp; g.b_rows = H; g.b_outer = S;
    g.K = 1; g.M = 2 * F; g.N = H; g.G = E; g.counts = counts; g.offsets = offsets;
    g.out = dw13; g.ldo = H; g.status = status;
    if ((rc = gemm_run(g, st))) return rc;
  }
  if (F_shared) {
    float* dh_s = reinterpret_cast<float*>(sc + L.dh_s);
    void* dgu_s = sc + L.dgu_s;
    void* h_s = sc + L.h_s;
    GemmCall a{};
    a.name = "shared_dh";
    a.variant = GV_PAIR_F32_BMN;
    a.A = dout_bf16; a.a_rows = T; a.B = ws2; a.b_rows = F_shared; a.K = H; a.N = F_shared; a.M = T;
    a.out = dh_s; a.ldo = F_shared; a.status = status;
    if ((rc = gemm_run(a, st))) return rc;
    GemmCall b{};
    b.name = "shared_swiglu_bwd";
    b.variant = GV_PAIR_SWIGLU_BWD;
    b.A = x_shared; b.a_rows = T; b.B = ws13; b.b_rows = 2 * F_shared; b.b_up_rows = F_shared;
    b.K = H; b.N = F_shared; b.M = T;
    b.out = dgu_s; b.ldo = 2 * F_shared; b.out2 = h_s; b.ldo2 = F_shared; b.aux = dh_s; b.ld_aux = F_shared;
    b.status = status;
    if ((rc = gemm_run(b, st))) return rc;
    GemmCall c{};
    c.name = "shared_dx";
    c.variant = GV_PAIR_F32_BMN;
    c.A = dgu_s; c.a_rows = T; c.B = ws13; c.b_rows = H; c.K = 2 * F_shared; c.N = H; c.M = T;
    c.out = dx_shared; c.ldo = H; c.status = status;
    if ((rc = gemm_run(c, st))) return rc;
    if (dws2) {
      GemmCall d{};
      d.name = "shared_dw2";
      d.variant = GV_PAIR_F32_AMN_BMN;
      d.A = dout_bf16; d.a_rows = H; d.B = h_s; d.b_rows = F_shared; d.K = T; d.N = F_shared; d.M = H;
      d.out = dws2; d.ldo = F_shared; d.status = status;
      if ((rc = gemm_run(d, st))) return rc;
    }
    if (dws13) {
      GemmCall e{};
      e.name = "shared_dw13";
      e.variant = GV_PAIR_F32_AMN_BMN;
      e.A = dgu_s; e.a_rows = 2 * F_shared; e.B = x_shared; e.b_rows = H; e.K = T; e.N = H; e.M = 2 * F_shared;
      e.out = dws13; e.ldo = H; e.status = status;
      if ((rc = gemm_run(e, st))) return rc;
    }
  }
  return INVMOE_OK;
}

int moe_route_backward(const void* x, const void* w_router, const int32_t* topk_idx, const float* topk_w,
                       const float* dgate, const float* dxp, const int32_t* plan, const float* dx_shared, int T,
                       int H, int E, int k, float* dx, float* dw_router, void* workspace, size_t ws_bytes,
                       void* stream) {
  REQUIRE(T >= 0 && H > 0 && E > 0 && k > 0 && k <= E && k <= 32, INVMOE_ERR_INVALID_ARG, "bad sizes");
  REQUIRE(H % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "H=%d is not a multiple of 64", H);
  REQUIRE(E % 8 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "E=%d is not a multiple of 8", E);
  REQUIRE_PTR(workspace);
  const BwdLayout L = bwd_layout(T, E, k, 0, 0);
  REQUIRE(ws_bytes >= kStatusBytes + L.end, INVMOE_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  REQUIRE_ALIGNED(workspace);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (dw_router)
      return check_cuda(cudaMemsetAsync(dw_router, 0, static_cast<size_t>(E) * H * 4, st), "memset");
    return INVMOE_OK;
  }
  REQUIRE_PTR(x); REQUIRE_PTR(w_router); REQUIRE_PTR(topk_idx); REQUIRE_PTR(topk_w); REQUIRE_PTR(dgate);
  REQUIRE_PTR(dxp); REQUIRE_PTR(plan); REQUIRE_PTR(dx);
  REQUIRE_ALIGNED(x); REQUIRE_ALIGNED(w_router); REQUIRE_ALIGNED(dxp); REQUIRE_ALIGNED(dx);
  if (dx_shared) REQUIRE_ALIGNED(dx_shared);
  if (dw_router) REQUIRE_ALIGNED(dw_router);
  void* dlog = scratch(workspace) + L.dlog;
  unsigned int* status = status_word(workspace);
  int rc = router_bwd_launch(topk_idx, topk_w, dgate, T, E, k, dlog, st);
  if (rc) return rc;
  // router part of dx: dlog [T, E] (K = E) times w_router [E, H] read MN-major
  GemmCall a{};
  a.name = "router_dx";
  a.variant = GV_PAIR_F32_BMN;
  a.A = dlog; a.a_rows = T; a.B = w_router; a.b_rows = H; a.K = E; a.N = H; a.M = T;
  a.out = dx; a.ldo = H; a.status = status;
  if ((rc = gemm_run(a, st))) return rc;
  if (dw_router) {
    GemmCall b{};
    b.name = "router_dw";
    b.variant = GV_PAIR_F32_AMN_BMN;
    b.A = dlog; b.a_rows = E; b.B = x; b.b_rows = H; b.K = T; b.N = H; b.M = E;
    b.out = dw_router; b.ldo = H; b.status = status;
    if ((rc = gemm_run(b, st))) return rc;
  }
  const int32_t* slot_row = plan + 2 * E + 1 + static_cast<long long>(T) * k;
  return unpermute_sum_launch(dxp, slot_row, dx_shared, T, H, k, dx, st);
}

int rl_token_loss(const float* logp_train, const float* logp_old, const float* logp_rollout, const float* advantage,
                  int T, float beta, float eps_low, float eps_high, uint8_t* icepop_mask, float* dis_weight,
                  float* loss, float* loss_mean, float* grad_logp, void* stream) {
  REQUIRE(T >= 0, INVMOE_ERR_INVALID_ARG, "T must be >= 0");
  REQUIRE(beta >= 1.0f, INVMOE_ERR_INVALID_ARG, "beta must be >= 1");
  REQUIRE(eps_low >= 0.0f && eps_low < 1.0f && eps_high >= 0.0f, INVMOE_ERR_INVALID_ARG,
          "need 0 <= eps_low < 1 and eps_high >= 0");
  if (T == 0) return INVMOE_OK;
  REQUIRE_PTR(logp_train); REQUIRE_PTR(logp_rollout); REQUIRE_PTR(advantage); REQUIRE_PTR(loss);
  return rl_loss_launch(logp_train, logp_old, logp_rollout, advantage, T, beta, eps_low, eps_high, icepop_mask,
                        dis_weight, loss, loss_mean, grad_logp, static_cast<cudaStream_t>(stream));
}

int invmoe_gemm_bf16(const void* a, const void* b, int M, int N, int K, float* d, int variant, void* workspace,
                     size_t ws_bytes, void* stream) {
  REQUIRE(M >= 0 && N > 0 && K > 0, INVMOE_ERR_INVALID_ARG, "bad sizes");
  const int n_major = (variant >> 8) & 1;
  variant &= 0xff;
  REQUIRE(variant >= 0 && variant <= 6, INVMOE_ERR_INVALID_ARG, "variant must be 0..6 (+256 for n-major)");
  if (variant <= 4) {
    REQUIRE(K % 64 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of 64", K);
    REQUIRE(N % 4 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "N=%d is not a multiple of 4", N);
  } else {
    REQUIRE(N % 8 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "N=%d is not a multiple of 8", N);
    if (variant == 5) REQUIRE(K % 8 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of 8", K);
    if (variant == 6) REQUIRE(M % 8 == 0, INVMOE_ERR_UNSUPPORTED_SHAPE, "M=%d is not a multiple of 8", M);
  }
  REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= kStatusBytes, INVMOE_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  if (M == 0) return INVMOE_OK;
  REQUIRE_PTR(a); REQUIRE_PTR(b); REQUIRE_PTR(d);
  REQUIRE_ALIGNED(a); REQUIRE_ALIGNED(b); REQUIRE_ALIGNED(d);
  GemmCall g{};
  g.name = "gemm_bf16";
  g.variant = variant == 4 ? GV_PAIR_F32 : variant == 5 ? GV_PAIR_F32_BMN : variant == 6 ? GV_PAIR_F32_AMN_BMN
                                                                                 : static_cast<GemmVariant>(variant);
  g.A = a; g.a_rows = M; g.B = b; g.b_rows = N; g.K = K; g.N = N; g.M = M; g.G = 0;
  g.n_major = n_major;
  g.out = d; g.ldo = N; g.status = status_word(workspace);
  return gemm_run(g, static_cast<cudaStream_t>(stream));
}

int invmoe_expert_engine(int which) {
  REQUIRE(which >= 0 && which <= 2, INVMOE_ERR_INVALID_ARG,
          "engine must be 0 (row tiles), 1 (token columns) or 2 (automatic)");
  g_expert_engine.store(which);
  return INVMOE_OK;
}

int invmoe_shared_overlap(int mode) {
  if (mode < 0 || mode > 2) return set_error(INVMOE_ERR_INVALID_ARG, "mode must be 0, 1 or 2");
  g_shared_overlap.store(mode);
  return INVMOE_OK;
}

int invmoe_pdl_enable(int on) {
  g_pdl_on.store(on != 0);
  return INVMOE_OK;
}

int invmoe_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on.store(on != 0);
  return INVMOE_OK;
}

int invmoe_profile_collect(char* names, float* total_ms, int* launches, int max_entries) {
  REQUIRE_PTR(names); REQUIRE_PTR(total_ms); REQUIRE_PTR(launches);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  int n = 0;
  int rc = INVMOE_OK;
  for (const ProfRec& r : g_prof_recs) {
    float ms = 0.f;
    if (!rc) rc = check_cuda(cudaEventSynchronize(r.b), "cudaEventSynchronize");
    if (!rc) rc = check_cuda(cudaEventElapsedTime(&ms, r.a, r.b), "cudaEventElapsedTime");
    int slot = -1;
    for (int i = 0; i < n; ++i)
      if (strncmp(names + 48 * i, r.name, 47) == 0) { slot = i; break; }
    if (slot < 0 && n < max_entries) {
      slot = n++;
      strncpy(names + 48 * slot, r.name, 47);
      names[48 * slot + 47] = 0;
      total_ms[slot] = 0.f;
      launches[slot] = 0;
    }
    if (slot >= 0) {
      total_ms[slot] += ms;
      launches[slot] += 1;
    }
    g_prof_pool.push_back(r.a);
    g_prof_pool.push_back(r.b);
  }
  g_prof_recs.clear();
  return rc ? rc : n;
}

int invmoe_debug_timeout_probe(void* workspace, size_t ws_bytes, int timeout_us, void* stream) {
  REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= kStatusBytes, INVMOE_ERR_WORKSPACE_TOO_SMALL, "workspace too small");
  REQUIRE(timeout_us >= 1 && timeout_us <= 2000000, INVMOE_ERR_INVALID_ARG, "timeout_us must be 1..2000000");
  return timeout_probe_launch(status_word(workspace), static_cast<unsigned long long>(timeout_us) * 1000ull,
                              static_cast<cudaStream_t>(stream));
}

}  // extern "C"
