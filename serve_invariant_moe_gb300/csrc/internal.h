// internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/invmoe.h"

namespace invmoe {

// Wait limit for every bounded device wait (1 s).
constexpr unsigned long long kTimeoutNs = 1000000000ull;

// Fixed chunk sizes (part of the numerical definition; never derived from T).
constexpr int kDispatchChunk = 64;   // tokens per dispatch-count chunk
constexpr int kSharedOverlapMaxT = 1024;   // moe_layer_forward's automatic choice: the shared expert
                                           // runs on the side stream for batches up to this size
constexpr int kLseChunk = 256;       // vocabulary columns per log-sum-exp partial

// Workspace: [0, 256) status block, then per-call scratch.
constexpr size_t kStatusBytes = 256;

int set_error(int code, const char* fmt, ...);

// Brackets one kernel launch with CUDA events while profiling is enabled.
class ProfScope {
 public:
  ProfScope(const char* name, cudaStream_t st);
  ~ProfScope();
 private:
  long idx_;
  cudaStream_t st_;
};
int check_cuda(cudaError_t e, const char* what);
int device_sm_count(int* out);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Whether kernels are launched with programmatic dependent launch (on unless switched off
// with invmoe_pdl_enable(0)).
bool pdl_enabled();

// Launch `kernel` on `st`; with programmatic dependent launch on, it may be scheduled while
// the previous kernel on the stream is finishing (every kernel launched this way calls
// pdl_wait() before touching global memory).  Extra attributes (a cluster shape) may be given.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             const cudaLaunchAttribute* extra, int n_extra, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[4];
  int n = 0;
  for (int i = 0; i < n_extra && n < 3; ++i) attr[n++] = extra[i];
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          Args... args) {
  return launch_kernel_ex(kernel, grid, block, smem, st, nullptr, 0, args...);
}

// ---------------------------------------------------------------- GEMM engine
enum GemmVariant : int {
  GV_F32_BN256_MT1 = 0,   // dense fp32-out, 4-stage ring, double-buffered TMEM (LM head)
  GV_F32_BN256_MT2 = 1,   // grouped/dense fp32-out, 2 row tiles per unit (expert down projection)
  GV_F32_BN128_MT1 = 2,
  GV_F32_BN64_MT1 = 3,
  GV_SWIGLU_BN256_MT2 = 4, // grouped/dense gate+up with SwiGLU epilogue -> bf16
  GV_PAIR_F32 = 6,         // CTA-pair 256 x 256 tile, fp32 out
  GV_PAIR_LSE = 7,         // CTA-pair tile, log-sum-exp epilogue
  GV_PAIR_SWIGLU = 8,      // CTA-pair tile, SwiGLU epilogue
  GV_PAIR_DLOGITS = 9,     // CTA-pair tile, bf16 g * (onehot - softmax) epilogue (head backward)
  GV_PAIR_F32_BMN = 10,    // CTA-pair tile, fp32 out, B MN-major ([K, N]), any K % 8 == 0
  GV_PAIR_F32_AMN_BMN = 11, // CTA-pair tile, fp32 out, A ([K, M]) and B ([K, N]) MN-major, any K
  GV_F32_BN256_MT2_BMN = 12, // grouped fp32-out, B MN-major: group g's B = stored rows [g*b_group_rows, +K)
  GV_SWIGLU_BWD_BN256_MT2 = 13, // grouped gate+up recompute with the SwiGLU backward epilogue
  GV_F32_BN256_MT1_KGROUP = 14, // K-grouped weight gradients: D_g = A_g^T B_g, A and B MN-major
  GV_PAIR_SWIGLU_BWD = 15, // CTA-pair gate+up recompute with the SwiGLU backward epilogue
  GV_TOK_SWIGLU = 16,      // grouped gate+up, tokens on the MMA's N side (CTA pair), SwiGLU -> bf16
  GV_TOK_F32 = 17,         // grouped, tokens on the MMA's N side (CTA pair), fp32 out
  GV_F32_SMALL64 = 18,     // dense fp32-out, at most 64 rows of A, one 64-column tile per CTA, 4 K blocks per copy
  GV_SWIGLU_SMALL64 = 19   // dense gate+up with SwiGLU -> bf16, at most 64 rows of A, 32 columns of h per CTA
};

// Which engine runs the forward grouped expert GEMMs: 0 = tokens on the MMA's M side in row
// tiles (tc_gemm.cuh), 1 = tokens on the N side (tc_gemm_tok.cuh), 2 = chosen per call (default).
int expert_engine();

struct GemmCall {
  const char* name;    // kernel label for the profiler
  GemmVariant variant;
  const void* A;       // [a_rows, K] bf16 (MN-major variants: [K, a_rows])
  long long a_rows;
  const void* B;       // [b_rows, K] bf16 (MN-major variants: [K, b_rows])
  long long b_rows;
  int K;
  int N;               // valid output columns
  int M;               // dense rows (ignored when G > 0)
  int G;               // groups (0 = dense)
  const int* counts;
  const int* offsets;
  int b_group_rows;
  int b_up_rows;
  int n_major;
  void* out;
  long long ldo;
  unsigned int* status;
  int* sched;            // unit counter and done count (two ints, zero between launches); null = the
                         // status block's first pair (byte 64); launches that may run at the same
                         // time need different pairs
  float2* part;          // GV_PAIR_LSE only: partials of the first column block of `row` 0
  long long part_ld;     // GV_PAIR_LSE: row stride of part in pairs (0 = ceil(N / 256))
  int target_col0;       // GV_PAIR_LSE: vocabulary column of B's first row (a shard's v0)
  const int* target;     // GV_PAIR_LSE / GV_PAIR_DLOGITS
  float* tgt_logit;      // GV_PAIR_LSE only
  int m_group;           // dense column-block-major order: row chunks per band (0 = all)
  const float* row_lse;  // GV_PAIR_DLOGITS only
  const float* row_scale;
  const float* aux;      // SwiGLU backward: dh [rows, N] fp32, row stride ld_aux
  long long ld_aux;
  void* out2;            // SwiGLU backward: recomputed h (bf16, nullable), row stride ldo2
  long long ldo2;
  int kgroup;            // K-grouped mode (GV_F32_BN256_MT1_KGROUP)
  long long a_outer;     // MN-major A in the single-CTA engine: stored rows
  long long b_outer;     // MN-major B in the single-CTA engine: stored rows
};

int gemm_run(const GemmCall& c, cudaStream_t st);

// ---------------------------------------------------------------- routing
int route_launch(const float* logits, int T, int E, int k, int H, const void* x, int32_t* topk_idx,
                 float* topk_w, int32_t* plan, void* xp, int32_t* chunk_counts, cudaStream_t st);

int dispatch_launch(const int32_t* topk_idx, int T, int E, int k, int H, const void* x, int32_t* plan, void* xp,
                    int32_t* chunk_counts, cudaStream_t st);
int permute_launch(const void* x, const int32_t* slot_row, int T, int k, int H, void* xp, cudaStream_t st);
int replay_launch(const float* logits, const int32_t* idx_in, int T, int E, int k, int H, const void* x,
                  int32_t* idx_safe, float* topk_w, int32_t* plan, void* xp, int32_t* chunk_counts,
                  unsigned int* status, cudaStream_t st);

// ---------------------------------------------------------------- combine / head
int combine_launch(const float* y, const float* topk_w, const int32_t* slot_row, const float* y_shared,
                   int T, int H, int k, float* out, void* out_bf16, cudaStream_t st);
// Partials of chunk c of token t at partials[(c / shard_chunks) * shard_stride + t * ld_part + c % shard_chunks];
// the target logit of token t at tgt_logit[(target[t] / 256 / shard_chunks) * tgt_stride + t].
int lse_merge_launch(const float2* partials, long long ld_part, int shard_chunks, long long shard_stride,
                     const float* tgt_logit, long long tgt_stride, const int32_t* target, const float* rollout_logp,
                     int T, int V, float beta, float* logp, float* lse, float* k3, uint8_t* mask, cudaStream_t st);
int rl_loss_launch(const float* lt, const float* lo, const float* lr, const float* adv, int T, float beta,
                   float el, float eh, uint8_t* mask, float* dis, float* loss, float* loss_mean, float* grad,
                   cudaStream_t st);
int timeout_probe_launch(unsigned int* status, unsigned long long limit_ns, cudaStream_t st);

int shared_expert_run(const void* x, const void* ws13, const void* ws2, int T, int H, int F_shared, float* y_shared,
                      void* hs, unsigned int* status, cudaStream_t st, int* sched = nullptr);

// ---------------------------------------------------------------- expert parallelism
int ep_regroup_launch(const void* recv_xp, const int32_t* recv_counts, int n_src, int E_local, int R, int H,
                      void* xp_local, int32_t* plan_local, int32_t* row_src, unsigned int* status, cudaStream_t st);
int ep_ungroup_launch(const float* y_local, const int32_t* row_src, int R, int H, float* y_send, cudaStream_t st);

// ---------------------------------------------------------------- backward
int combine_bwd_launch(const float* dout, const float* y, const float* topk_w, const int32_t* slot_row, int T,
                       int H, int k, void* dy, float* dgate, void* dout_bf16, cudaStream_t st);
int router_bwd_launch(const int32_t* topk_idx, const float* topk_w, const float* dgate, int T, int E, int k,
                      void* dlog, cudaStream_t st);
int unpermute_sum_launch(const float* dxp, const int32_t* slot_row, const float* dx_shared, int T, int H, int k,
                         float* dx, cudaStream_t st);

}  // namespace invmoe
