// combine_head.cu -- fp32 fixed-order combine; chunked two-pass log-sum-exp,
// token logprob, k3 and the IcePop mask; the bounded-wait probe.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace invmoe {

namespace {

// out[t, :] = ((w0*y0 + w1*y1) + ...) + y_shared, fp32, slots in rank order,
// every product and sum rounded on its own ("Reinforcement Learning: Why
// Numerical Alignment and MoE Routing Matter So Much", section
// "混合专家模型更难对齐": the precision and order of the weighted expert sum
// must be pinned).  One thread per 4 columns, 16-byte loads and stores.
__global__ void combine_kernel(const float4* __restrict__ y, const float* __restrict__ w,
                               const int32_t* __restrict__ slot_row, const float4* __restrict__ y_shared, int T,
                               int H4, int k, float4* __restrict__ out, uint2* __restrict__ out_bf16) {
  pdl_wait();
  pdl_trigger();
  const long long total = static_cast<long long>(T) * H4;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = i / H4;
    const int c = static_cast<int>(i - t * H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const float wj = w[t * k + j];
      const float4 v = y[static_cast<long long>(slot_row[t * k + j]) * H4 + c];
      const float4 pr = make_float4(__fmul_rn(wj, v.x), __fmul_rn(wj, v.y), __fmul_rn(wj, v.z), __fmul_rn(wj, v.w));
      if (j == 0) {
        acc = pr;
      } else {
        acc = make_float4(__fadd_rn(acc.x, pr.x), __fadd_rn(acc.y, pr.y), __fadd_rn(acc.z, pr.z),
                          __fadd_rn(acc.w, pr.w));
      }
    }
    if (y_shared != nullptr) {
      const float4 s = y_shared[i];
      acc = make_float4(__fadd_rn(acc.x, s.x), __fadd_rn(acc.y, s.y), __fadd_rn(acc.z, s.z), __fadd_rn(acc.w, s.w));
    }
    out[i] = acc;
    if (out_bf16 != nullptr) {
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      out_bf16[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
    }
  }
}

// Pass 2 of the chunked log-sum-exp ("GLM Post-Training Beyond SFT", section
// "动作与概率契约": logsumexp needs comparison tests; the chunking fixes its
// order).  Pass 1 runs in the vocabulary-projection epilogue: for the 256-column
// chunk c of row t it gives m_c = max z and s_c = sum of exp(z - m_c).
// Two partials combine as
//   (M, S) + (m, s) = (max(M, m), S*exp(M - max) + s*exp(m - max))
// with the factor for the larger maximum being exactly 1 (so one exp per step);
// the operation is commutative bit for bit.  Fixed order: one warp per token;
// lane l folds chunks [l*P, (l+1)*P), P = ceil(NCH / 32), in ascending order;
// the 32 lane results are then folded by a xor butterfly over lane distances
// 16, 8, 4, 2, 1.  The order depends only on V, never on the batch.
// Then lse = M + log S, logp = z[target] - lse and, with rollout logprobs
// ("GLM Post-Training Beyond SFT", section "IcePop 为什么有两层 ratio"),
// d = logp - rollout, k3 = expm1(d) - d, rho = exp(d), mask = 1/beta <= rho <= beta.
__device__ __forceinline__ void lse_fold(float& M, float& S, float m, float s) {
  if (m == -INFINITY) return;
  if (M == -INFINITY) {
    M = m;
    S = s;
  } else if (m > M) {
    S = __fadd_rn(__fmul_rn(S, expf(M - m)), s);
    M = m;
  } else {
    S = __fadd_rn(S, __fmul_rn(s, expf(m - M)));
  }
}

constexpr int kMergeWarps = 4;
constexpr int kMergeBatch = 4;   // partials a lane loads before folding them

// The partials of chunk c of token t sit at
//   part[(c / shard_chunks) * shard_stride + t * ld_part + c % shard_chunks]
// and the target logit of token t at tgt_logit[(shard of its target) * tgt_stride + t],
// which covers one [T, NCH] array (shard_chunks = NCH) and the [shards][T][P]
// arrays that gathering vocabulary shards of P chunks each produces; the fold
// order above is the same for every layout.
__global__ void lse_merge_kernel(const float2* __restrict__ part, long long ld_part, int shard_chunks,
                                 long long shard_stride, const float* __restrict__ tgt_logit, long long tgt_stride,
                                 const int32_t* __restrict__ target, const float* __restrict__ rollout, int T, int V,
                                 int NCH, float beta, float* __restrict__ logp, float* __restrict__ lse,
                                 float* __restrict__ k3, uint8_t* __restrict__ mask) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const int P = (NCH + 31) / 32;
  int c = lane * P;
  const int c1 = min(NCH, (lane + 1) * P);
  float M = -INFINITY, S = 0.0f;
  if (c < c1) {
    int sh = c / shard_chunks;
    int j = c - sh * shard_chunks;
    const float2* base = part + sh * shard_stride + static_cast<long long>(t) * ld_part;
    // the lane's partials in batches of kMergeBatch: a batch's loads are all issued before its
    // first fold (the folds keep their ascending order)
    for (; c < c1; c += kMergeBatch) {
      float2 v[kMergeBatch];
#pragma unroll
      for (int i = 0; i < kMergeBatch; ++i) {
        if (c + i < c1) {
          v[i] = base[j];
          if (++j == shard_chunks) {
            j = 0;
            base += shard_stride;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kMergeBatch; ++i)
        if (c + i < c1) lse_fold(M, S, v[i].x, v[i].y);
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    const float m = __shfl_xor_sync(0xffffffffu, M, d);
    const float s = __shfl_xor_sync(0xffffffffu, S, d);
    lse_fold(M, S, m, s);
  }
  if (lane != 0) return;
  const float l = __fadd_rn(M, logf(S));
  const int tg = target[t];
  // the target logit comes from the shard that owns the target's chunk
  const float lp = (tg >= 0 && tg < V)
                       ? __fsub_rn(tgt_logit[(tg / kLseChunk / shard_chunks) * tgt_stride + t], l)
                       : __uint_as_float(0x7fc00000u);
  logp[t] = lp;
  if (lse != nullptr) lse[t] = l;
  if (rollout != nullptr) {
    const float d = __fsub_rn(lp, rollout[t]);
    if (k3 != nullptr) k3[t] = __fsub_rn(expm1f(d), d);
    if (mask != nullptr) {
      const float rho = expf(d);
      const float lo = __fdiv_rn(1.0f, beta);
      mask[t] = (lo <= rho && rho <= beta) ? 1 : 0;
    }
  }
}

// Per-token policy-loss terms ("GLM Post-Training Beyond SFT", sections "GRPO
// 在优化什么", "IcePop 为什么有两层 ratio", "Direct Double-Sided Importance
// Sampling"), fp32:
//   rho = exp(lt - lr)            mismatch ratio train / rollout
//   r   = exp(lt - lo)            PPO ratio train / old train (lo = lr when absent)
//   m   = 1/beta <= rho <= beta   IcePop trust mask
//   loss = m ? -min(r*A, clip(r, 1-el, 1+eh)*A) : 0
//   dis  = (1-el < rho < 1+eh) ? rho : 0
__global__ void rl_token_kernel(const float* __restrict__ lt, const float* __restrict__ lo,
                                const float* __restrict__ lr, const float* __restrict__ adv, int T, float beta,
                                float el, float eh, uint8_t* __restrict__ mask, float* __restrict__ dis,
                                float* __restrict__ loss, float* __restrict__ grad) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const float rho = expf(__fsub_rn(lt[t], lr[t]));
  const float r = expf(__fsub_rn(lt[t], lo != nullptr ? lo[t] : lr[t]));
  const float lo_clip = __fsub_rn(1.0f, el), hi_clip = __fadd_rn(1.0f, eh);
  const bool m = (__fdiv_rn(1.0f, beta) <= rho) && (rho <= beta);
  const float a = adv[t];
  const float obj = fminf(__fmul_rn(r, a), __fmul_rn(fminf(fmaxf(r, lo_clip), hi_clip), a));
  loss[t] = m ? -obj : 0.0f;
  if (mask != nullptr) mask[t] = m ? 1 : 0;
  if (dis != nullptr) dis[t] = (lo_clip < rho && rho < hi_clip) ? rho : 0.0f;
  if (grad != nullptr) {
    // d mean / d logp_train with the mask held fixed: -(r A) / T where the unclipped term is the minimum
    const float ra = __fmul_rn(r, a);
    const bool unclipped = ra <= __fmul_rn(fminf(fmaxf(r, lo_clip), hi_clip), a);
    grad[t] = (m && unclipped) ? -__fdiv_rn(ra, static_cast<float>(T)) : 0.0f;
  }
}

// Mean of loss[0..T) in a fixed order: thread i of one 1024-thread block adds
// loss[i], loss[i + 1024], ... in ascending order; the 1024 partial sums are
// folded by a xor butterfly inside each warp (16, 8, 4, 2, 1) and then across
// the 32 warp sums the same way; the total is divided by T.
__global__ void fixed_order_mean_kernel(const float* __restrict__ v, int T, float* __restrict__ out) {
  __shared__ float warp_sum[32];
  float s = 0.0f;
  for (int i = threadIdx.x; i < T; i += 1024) s = __fadd_rn(s, v[i]);
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, d));
  if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    float w = warp_sum[threadIdx.x];
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) w = __fadd_rn(w, __shfl_xor_sync(0xffffffffu, w, d));
    if (threadIdx.x == 0) *out = __fdiv_rn(w, static_cast<float>(T));
  }
}

// Waits on an mbarrier that nothing completes, with a short limit; records the
// timeout in the status word and returns.
__global__ void timeout_probe_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtl w{&abort_flag, status, limit_ns};
    mbar_wait(&bar, 0, w);
    // release the barrier so the shared word is left in a completed state
    mbar_arrive(&bar);
  }
}

}  // namespace

int combine_launch(const float* y, const float* topk_w, const int32_t* slot_row, const float* y_shared, int T,
                   int H, int k, float* out, void* out_bf16, cudaStream_t st) {
  int sms = 0, rc;
  if ((rc = device_sm_count(&sms))) return rc;
  const int H4 = H / 4;
  const long long total = static_cast<long long>(T) * H4;
  long long blocks = (total + 255) / 256;
  if (blocks > static_cast<long long>(sms) * 16) blocks = static_cast<long long>(sms) * 16;
  if (blocks == 0) return INVMOE_OK;
  ProfScope prof("combine", st);
  return check_cuda(launch_kernel(combine_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                                  reinterpret_cast<const float4*>(y), topk_w, slot_row,
                                  reinterpret_cast<const float4*>(y_shared), T, H4, k, reinterpret_cast<float4*>(out),
                                  reinterpret_cast<uint2*>(out_bf16)),
                    "combine_kernel");
}

int lse_merge_launch(const float2* partials, long long ld_part, int shard_chunks, long long shard_stride,
                     const float* tgt_logit, long long tgt_stride, const int32_t* target, const float* rollout_logp,
                     int T, int V, float beta, float* logp, float* lse, float* k3, uint8_t* mask, cudaStream_t st) {
  const int NCH = (V + kLseChunk - 1) / kLseChunk;
  if (T == 0) return INVMOE_OK;
  ProfScope prof("lse_merge", st);
  return check_cuda(launch_kernel(lse_merge_kernel, dim3((T + kMergeWarps - 1) / kMergeWarps), dim3(32 * kMergeWarps),
                                  0, st, partials, ld_part, shard_chunks, shard_stride, tgt_logit, tgt_stride, target,
                                  rollout_logp, T, V, NCH, beta, logp, lse, k3, mask),
                    "lse_merge_kernel");
}

int rl_loss_launch(const float* lt, const float* lo, const float* lr, const float* adv, int T, float beta,
                   float el, float eh, uint8_t* mask, float* dis, float* loss, float* loss_mean, float* grad,
                   cudaStream_t st) {
  int rc;
  {
    ProfScope prof("rl_token_loss", st);
    rl_token_kernel<<<(T + 255) / 256, 256, 0, st>>>(lt, lo, lr, adv, T, beta, el, eh, mask, dis, loss, grad);
    if ((rc = check_cuda(cudaGetLastError(), "rl_token_kernel"))) return rc;
  }
  if (loss_mean == nullptr) return INVMOE_OK;
  ProfScope prof("fixed_order_mean", st);
  fixed_order_mean_kernel<<<1, 1024, 0, st>>>(loss, T, loss_mean);
  return check_cuda(cudaGetLastError(), "fixed_order_mean_kernel");
}

int timeout_probe_launch(unsigned int* status, unsigned long long limit_ns, cudaStream_t st) {
  timeout_probe_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return check_cuda(cudaGetLastError(), "timeout_probe_kernel");
}

}  // namespace invmoe
