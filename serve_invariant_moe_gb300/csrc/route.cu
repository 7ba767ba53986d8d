// route.cu -- top-k with lowest-index ties, gates, deterministic dispatch, permute.
//
// Sources: "位级一致：前沿训练的差异化关键", section "为什么比特级一致是一个复杂的问题"
// (a router near-tie flips which expert fires; fix: a deterministic tie
// decision); "GLM Post-Training Beyond SFT", section "迁移到 NPU 时" (a top-k must
// fix ties, boundary ties, sort order, NaN handling and the index dtype).
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace invmoe {

namespace {

constexpr unsigned kFull = 0xffffffffu;

// Total order key: larger = ranks earlier.  NaN -> 0 (below every number,
// including -inf); -0.0 and +0.0 map to the same key (a tie).
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 0u;
  uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  if (key == 0u) return __uint_as_float(0x7fc00000u);
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// One warp per token.  Lane l holds experts l, l+32, ... (EPL of them).  Each of
// the k rounds takes the warp-wide maximum of the order keys still in play
// (redux.sync max), then the lowest expert index holding that key (redux.sync
// min): a larger logit wins, an exact tie goes to the lower expert index, and a
// NaN (key 0) is taken only after every number, lowest index first.  The gate
// softmax is taken over the k selected logits in rank order, in fp32.  Lane j < k
// returns the j-th ranked expert and its gate.  Both routing kernels below call
// this one function, so they take the same decisions and compute the same gate bits.
template <int EPL>
__device__ __forceinline__ void topk_token(const float* __restrict__ row, int E, int k, int lane, int& out_e,
                                           float& out_w) {
  uint32_t key[EPL];
  uint32_t live = 0u;   // bit i: expert i*32 + lane exists and has not been taken yet
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = i * 32 + lane;
    key[i] = (e < E) ? order_key(row[e]) : 0u;
    if (e < E) live |= 1u << i;
  }
  int my_e = 0;
  float my_v = 0.0f;
  for (int j = 0; j < k; ++j) {
    uint32_t best = 0u;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (((live >> i) & 1u) && key[i] > best) best = key[i];
    const uint32_t gbest = __reduce_max_sync(kFull, best);
    uint32_t cand = 0xffffffffu;
#pragma unroll
    for (int i = EPL - 1; i >= 0; --i)
      if (((live >> i) & 1u) && key[i] == gbest) cand = static_cast<uint32_t>(i * 32 + lane);
    const int e = static_cast<int>(__reduce_min_sync(kFull, cand));
    if ((e & 31) == lane) live &= ~(1u << (e >> 5));
    if (lane == j) {
      my_e = e;
      my_v = key_value(gbest);
    }
  }
  // gates: w_j = exp(v_j - v_0) / sum_{i<k} exp(v_i - v_0), the sum in rank order
  const float v0 = __shfl_sync(kFull, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - v0) : 0.0f;
  float s = 0.0f;
  for (int j = 0; j < k; ++j) s = __fadd_rn(s, __shfl_sync(kFull, ex, j));
  out_e = my_e;
  out_w = __fdiv_rn(ex, s);
}

// Blocks of kTopkThreads; up to E = 256 at most 32 registers a thread, so that a whole batch of
// 8192 tokens (one warp each) is resident at once (64 warps per SM on 152 SMs) instead of a
// second wave of a few blocks.
constexpr int kTopkThreads = 256;
template <int EPL>
__global__ void __launch_bounds__(kTopkThreads, EPL <= 8 ? 8 : 1)
    topk_gate_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ idx,
                     float* __restrict__ w) {
  pdl_wait();
  pdl_trigger();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int e;
  float wt;
  topk_token<EPL>(logits + static_cast<long long>(t) * E, E, k, lane, e, wt);
  if (lane < k) {
    idx[static_cast<long long>(t) * k + lane] = e;
    w[static_cast<long long>(t) * k + lane] = wt;
  }
}

// Routing of a small batch in one block of 1024 threads: the top-k and gates of
// every token, the dispatch plan and (when the copy is small) the permute, in one
// launch instead of five.  The plan is the same stable counting sort as the
// multi-kernel path (within an expert, rows in ascending (token, slot) order):
// warp w counts and then places the (token, slot) pairs of the w-th contiguous
// range of the batch, so every position is the same integer whichever path
// computes it.
constexpr int kSmallThreads = 1024;
constexpr int kSmallMaxTokens = 256;
constexpr int kSmallMaxPairs = 4096;
constexpr long long kSmallPermuteBytes = 512 * 1024;

// Shared memory of route_small_kernel: the plan's scratch (ints), then, when they fit, the
// logits [T, E] and the rows of x [T, H] staged with one round trip each at the start.
constexpr size_t kSmallSmemMax = 227 * 1024;
size_t route_small_plan_smem(int T, int E, int k) {
  return align_up((2 * static_cast<size_t>(T) * k + 32 * static_cast<size_t>(E) + E + 1 + 32) * sizeof(int), 16);
}

template <int EPL>
__global__ void __launch_bounds__(kSmallThreads, 1)
    route_small_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ idx,
                       float* __restrict__ w, int32_t* __restrict__ plan, const uint4* __restrict__ x,
                       int vec_per_row, uint4* __restrict__ xp, int do_permute, int stage_logits, int stage_x) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) int sm[];
  const int S = T * k;
  int* s_idx = sm;                 // [S] expert of each pair
  int* s_pos = s_idx + S;          // [S] permuted row of each pair
  int* hist = s_pos + S;           // [32][E] per-warp counts, then per-warp running positions
  int* s_off = hist + 32 * E;      // [E + 1] segment starts
  int* warp_tot = s_off + E + 1;   // [32]
  uint8_t* extra = reinterpret_cast<uint8_t*>(sm) + ((2 * S + 32 * E + E + 1 + 32) * sizeof(int) + 15) / 16 * 16;
  float* s_logits = reinterpret_cast<float*>(extra);                                    // [T, E] if staged
  uint4* s_x = reinterpret_cast<uint4*>(extra + (stage_logits ? ((T * E * 4 + 15) / 16) * 16 : 0));  // [T, H]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int32_t* counts = plan;
  int32_t* offsets = plan + E;
  int32_t* row_token = plan + 2 * E + 1;
  int32_t* slot_row = row_token + S;
  // the loads that do not depend on the routing are all issued first
  if (stage_x)
    for (int i = tid; i < T * vec_per_row; i += kSmallThreads) s_x[i] = __ldg(x + i);
  if (stage_logits) {
    for (int i = tid; i < T * E; i += kSmallThreads) s_logits[i] = __ldg(logits + i);
    __syncthreads();
  }
  const float* lrow0 = stage_logits ? s_logits : logits;
  // top-k and gates: warp w takes tokens w, w + 32, ...
  for (int t = warp; t < T; t += 32) {
    int e;
    float wt;
    topk_token<EPL>(lrow0 + static_cast<long long>(t) * E, E, k, lane, e, wt);
    if (lane < k) {
      idx[t * k + lane] = e;
      w[t * k + lane] = wt;
      s_idx[t * k + lane] = e;
    }
  }
  for (int i = tid; i < 32 * E; i += kSmallThreads) hist[i] = 0;
  __syncthreads();
  // per-warp counts over contiguous ranges of pairs
  const int per = (S + 31) / 32;
  const int p0 = min(S, warp * per), p1 = min(S, p0 + per);
  for (int p = p0 + lane; p < p1; p += 32) atomicAdd(&hist[warp * E + s_idx[p]], 1);
  __syncthreads();
  // per expert: exclusive scan over warps (in place) and the expert total
  int run = 0;
  if (tid < E) {
    for (int v = 0; v < 32; ++v) {
      const int c = hist[v * E + tid];
      hist[v * E + tid] = run;
      run += c;
    }
    counts[tid] = run;
  }
  // exclusive scan of the totals over experts (E <= 1024: one per thread)
  int incl = run;
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int t = warp_tot[lane];
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(kFull, t, d);
      if (lane >= d) t += v;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  const int excl = incl - run + (warp > 0 ? warp_tot[warp - 1] : 0);
  if (tid < E) {
    offsets[tid] = excl;
    s_off[tid] = excl;
  }
  if (tid == E - 1) offsets[E] = excl + run;
  __syncthreads();
  // placement: each warp walks its range 32 pairs at a time in ascending order
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int pb = p0; pb < p1; pb += 32) {
    const int p = pb + lane;
    const int e = (p < p1) ? s_idx[p] : -1;
    const unsigned m = __match_any_sync(kFull, e);
    const int rank = __popc(m & lt_mask);
    if (e >= 0) {
      const int pos = s_off[e] + hist[warp * E + e] + rank;
      row_token[pos] = p / k;
      slot_row[p] = pos;
      s_pos[p] = pos;
    }
    __syncwarp();
    if (e >= 0 && rank == 0) hist[warp * E + e] += __popc(m);
    __syncwarp();
  }
  if (!do_permute) return;
  __syncthreads();
  // permute: xp[slot_row[t, j]] = x[t] in 16-byte vectors, one vector of one token per thread and
  // step over the whole block (one warp per token left most of the block idle for a decode batch:
  // 4.0-4.4 us for one token of H = 6144)
  const int nvec = T * vec_per_row;
  for (int i = tid; i < nvec; i += kSmallThreads) {
    const int t = i / vec_per_row;
    const int c = i - t * vec_per_row;
    const uint4 v = stage_x ? s_x[i] : __ldg(x + i);
    for (int j = 0; j < k; ++j) xp[static_cast<long long>(s_pos[t * k + j]) * vec_per_row + c] = v;
  }
}

// Router replay ("Reinforcement Learning: Why Numerical Alignment and MoE Routing
// Matter So Much", section "MoE 路由会放大这种不匹配": router replay records the
// rollout's expert choices and reuses them in training; the same page notes that
// the outputs' computation and combine must still match).  One warp per token:
// the k given experts are checked (in range, distinct); gates are the softmax of
// their logits, w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max) with the sum in
// slot order -- for experts given in descending-logit order this is exactly the
// arithmetic of topk_gate_kernel.  A token with an invalid list gets experts
// 0..k-1 and NaN gates, and the status word records kStatusBadIndex.
__global__ void replay_gate_kernel(const float* __restrict__ logits, const int32_t* __restrict__ idx_in, int T,
                                   int E, int k, int32_t* __restrict__ idx_out, float* __restrict__ w,
                                   unsigned int* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  int e = lane < k ? idx_in[static_cast<long long>(t) * k + lane] : -1;
  const unsigned m = __match_any_sync(kFull, e);
  const bool bad_lane = lane < k && (e < 0 || e >= E || __popc(m) > 1);
  const bool bad = __any_sync(kFull, bad_lane);
  if (bad) {
    if (lane == 0) atomicOr(status, kStatusBadIndex);
    if (lane < k) {
      idx_out[static_cast<long long>(t) * k + lane] = lane;
      w[static_cast<long long>(t) * k + lane] = __uint_as_float(0x7fc00000u);
    }
    return;
  }
  const float v = lane < k ? logits[static_cast<long long>(t) * E + e] : -INFINITY;
  float vmax = v;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, d));
  const float ex = (lane < k) ? expf(v - vmax) : 0.0f;
  float s = 0.0f;
  for (int j = 0; j < k; ++j) s = __fadd_rn(s, __shfl_sync(kFull, ex, j));
  if (lane < k) {
    idx_out[static_cast<long long>(t) * k + lane] = e;
    w[static_cast<long long>(t) * k + lane] = __fdiv_rn(ex, s);
  }
}

// Per chunk of kDispatchChunk tokens: how many of its (token, slot) pairs go to each expert.
__global__ void dispatch_count_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                      int32_t* __restrict__ chunk_counts) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int hist[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int c = blockIdx.x;
  const long long p0 = static_cast<long long>(c) * kDispatchChunk * k;
  const long long p1 = min(static_cast<long long>(T), static_cast<long long>(c + 1) * kDispatchChunk) * k;
  for (long long p = p0 + threadIdx.x; p < p1; p += blockDim.x) atomicAdd(&hist[idx[p]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[static_cast<long long>(c) * E + e] = hist[e];
}

// One block of 1024 threads: per expert an exclusive scan over chunks (in place),
// the expert totals, and an exclusive scan over experts for the segment offsets.
// When every thread's share fits in registers, Q = 1024 / E threads (at most 4)
// share an expert's chunks: thread (q, e) loads its whole range [q*per, +per) at
// once, the Q range totals meet in shared memory, and each thread writes its
// range's exclusive counts from the total of the ranges before it.  Integer sums,
// so the plan is the same whichever way it is computed.
constexpr int kScanRegs = 32;
__global__ void __launch_bounds__(1024, 1)
    dispatch_scan_kernel(int32_t* __restrict__ chunk_counts, int NC, int E, int32_t* __restrict__ counts,
                         int32_t* __restrict__ offsets) {
  pdl_wait();
  pdl_trigger();
  __shared__ int warp_tot[32];
  __shared__ int part[1024];
  const int e = threadIdx.x;
  const int Q = E <= 256 ? 4 : (E <= 512 ? 2 : 1);
  const int per = (NC + Q - 1) / Q;
  int run = 0;
  if (per <= kScanRegs) {
    const int q = e / E, ee = e - q * E;
    const int c0 = q * per;
    const int n = q < Q ? max(0, min(per, NC - c0)) : 0;
    int32_t* col = chunk_counts + static_cast<long long>(c0) * E + ee;
    int v[kScanRegs];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < kScanRegs; ++i)
      if (i < n) v[i] = col[static_cast<long long>(i) * E];
#pragma unroll
    for (int i = 0; i < kScanRegs; ++i)
      if (i < n) sum += v[i];
    part[e] = sum;
    __syncthreads();
    if (q < Q) {
      int base = 0;
      for (int qq = 0; qq < q; ++qq) base += part[qq * E + ee];
#pragma unroll
      for (int i = 0; i < kScanRegs; ++i) {
        if (i < n) {
          col[static_cast<long long>(i) * E] = base;
          base += v[i];
        }
      }
    }
    if (e < E) {
      for (int qq = 0; qq < Q; ++qq) run += part[qq * E + e];
      counts[e] = run;
    }
  } else if (e < E) {
    // eight chunks' counts are loaded before any of them is overwritten, so the loads of a
    // batch are in flight together instead of one dependent round trip per chunk
    int c = 0;
    for (; c + 8 <= NC; c += 8) {
      int v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = chunk_counts[static_cast<long long>(c + i) * E + e];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        chunk_counts[static_cast<long long>(c + i) * E + e] = run;
        run += v[i];
      }
    }
    for (; c < NC; ++c) {
      const long long i = static_cast<long long>(c) * E + e;
      const int v = chunk_counts[i];
      chunk_counts[i] = run;
      run += v;
    }
    counts[e] = run;
  }
  // block exclusive scan of run over e (blockDim.x = 1024)
  const int lane = e & 31, wid = e >> 5;
  int incl = run;
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(kFull, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int t = warp_tot[lane];
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(kFull, t, d);
      if (lane >= d) t += v;
    }
    warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const int excl = incl - run + (wid > 0 ? warp_tot[wid - 1] : 0);
  if (e < E) offsets[e] = excl;
  if (e == E - 1) offsets[E] = excl + run;
}

// One warp per chunk: walk the chunk's pairs p = t*k + j in ascending order, 32 at
// a time.  Lanes holding the same expert are ranked by lane (match_any), and a
// per-expert running position in shared memory carries the rank across batches, so
// each expert's rows come out in ascending token order (a token never picks the
// same expert twice).  The chunk's expert indices and each expert's first position
// for the chunk (segment offset + the chunk's exclusive count) are staged in shared
// memory first, with all their loads in flight together, so the walk itself makes
// no dependent global round trip.
__global__ void dispatch_scatter_kernel(const int32_t* __restrict__ idx, int T, int E, int k,
                                        const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets,
                                        int32_t* __restrict__ row_token, int32_t* __restrict__ slot_row) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int sm_scatter[];
  int* run = sm_scatter;            // [E] next position of each expert's rows from this chunk
  int* s_e = sm_scatter + E;        // [kDispatchChunk * k] the chunk's expert indices
  const int lane = threadIdx.x;
  const int c = blockIdx.x;
  const long long p0 = static_cast<long long>(c) * kDispatchChunk * k;
  const long long p1 = min(static_cast<long long>(T), static_cast<long long>(c + 1) * kDispatchChunk) * k;
  const int np = static_cast<int>(p1 - p0);
  for (int e = lane; e < E; e += 32) run[e] = offsets[e] + chunk_base[static_cast<long long>(c) * E + e];
  for (int i = lane; i < np; i += 32) s_e[i] = idx[p0 + i];
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int ib = 0; ib < np; ib += 32) {
    const int i = ib + lane;
    const int e = (i < np) ? s_e[i] : -1;
    const unsigned m = __match_any_sync(kFull, e);
    const int rank = __popc(m & lt_mask);
    if (e >= 0) {
      const int pos = run[e] + rank;
      const long long p = p0 + i;
      row_token[pos] = static_cast<int32_t>(p / k);
      slot_row[p] = pos;
    }
    __syncwarp();
    if (e >= 0 && rank == 0) run[e] += __popc(m);
    __syncwarp();
  }
}

// The permute, token-major: xp[slot_row[t, j], :] = x[t, :] for j < k, in
// 16-byte vectors.  One warp per token (tokens strided over the grid's warps):
// each X row is read once and written to its k Xp rows, so X is not re-read
// from DRAM once the Xp writes have pushed it out of L2.  Lane j (< k) holds
// slot j's row index; each lane keeps four vectors in flight.
constexpr int kPermuteThreads = 256;
__global__ void __launch_bounds__(kPermuteThreads) permute_rows_kernel(const uint4* __restrict__ x,
                                                                      const int32_t* __restrict__ slot_row,
                                                                      long long T, int k, int vec_per_row,
                                                                      int seg_vec, int nseg,
                                                                      uint4* __restrict__ xp) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long nwarps = static_cast<long long>(gridDim.x) * (kPermuteThreads / 32);
  // a warp copies segment `seg` (vectors [seg * seg_vec, +seg_vec) of the row) of token t to its
  // k rows of xp; one segment per token for large batches, 2 KB segments for small ones
  for (long long item = blockIdx.x * static_cast<long long>(kPermuteThreads / 32) + (threadIdx.x >> 5);
       item < T * nseg; item += nwarps) {
    const long long t = item / nseg;
    const int seg = static_cast<int>(item - t * nseg);
    const int c_end = min(vec_per_row, (seg + 1) * seg_vec);
    const int my_row = lane < k ? __ldg(slot_row + t * k + lane) : 0;
    const uint4* src = x + t * vec_per_row;
    // every loop bound below is warp-uniform, so the shuffles always see all 32 lanes
    int c0 = seg * seg_vec;
    for (; c0 + 128 <= c_end; c0 += 128) {
      const int c = c0 + lane;
      const uint4 v0 = __ldg(src + c), v1 = __ldg(src + c + 32), v2 = __ldg(src + c + 64), v3 = __ldg(src + c + 96);
      for (int j = 0; j < k; ++j) {
        uint4* dst = xp + static_cast<long long>(__shfl_sync(0xffffffffu, my_row, j)) * vec_per_row;
        dst[c] = v0;
        dst[c + 32] = v1;
        dst[c + 64] = v2;
        dst[c + 96] = v3;
      }
    }
    // tail: the segment's last (c_end - c0) < 128 vectors; lanes past its end only skip their store
    for (; c0 < c_end; c0 += 32) {
      const int cc = c0 + lane;
      const uint4 v = cc < c_end ? __ldg(src + cc) : make_uint4(0u, 0u, 0u, 0u);
      for (int j = 0; j < k; ++j) {
        const long long row = __shfl_sync(0xffffffffu, my_row, j);
        if (cc < c_end) xp[row * vec_per_row + cc] = v;
      }
    }
  }
}

}  // namespace

namespace {

template <int EPL>
int route_small_launch_epl(const float* logits, int T, int E, int k, int H, const void* x, int32_t* topk_idx,
                           float* topk_w, int32_t* plan, void* xp, bool do_permute, cudaStream_t st) {
  // stage the logits and the rows of x in shared memory when they fit
  size_t smem = route_small_plan_smem(T, E, k);
  const size_t lbytes = align_up(static_cast<size_t>(T) * E * 4, 16);
  const size_t xbytes = static_cast<size_t>(T) * H * 2;
  const bool stage_logits = smem + lbytes <= kSmallSmemMax && lbytes <= 64 * 1024;
  if (stage_logits) smem += lbytes;
  const bool stage_x = do_permute && smem + xbytes <= kSmallSmemMax && xbytes <= 64 * 1024;
  if (stage_x) smem += xbytes;
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  int rc = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit == 0 || !(attr_set.load(std::memory_order_acquire) & bit)) {
    // the largest shared-memory request of this kernel (E = 1024, 4096 pairs) is 164 KB
    rc = check_cuda(cudaFuncSetAttribute(route_small_kernel<EPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmallSmemMax)),
                    "cudaFuncSetAttribute");
    if (rc) return rc;
    if (bit) attr_set.fetch_or(bit, std::memory_order_release);
  }
  ProfScope prof("route_small", st);
  return check_cuda(launch_kernel(route_small_kernel<EPL>, dim3(1), dim3(kSmallThreads), smem, st, logits, T, E, k,
                                  topk_idx, topk_w, plan, static_cast<const uint4*>(x), H / 8,
                                  static_cast<uint4*>(xp), do_permute ? 1 : 0, stage_logits ? 1 : 0,
                                  stage_x ? 1 : 0),
                    "route_small_kernel");
}

}  // namespace

int route_launch(const float* logits, int T, int E, int k, int H, const void* x, int32_t* topk_idx,
                 float* topk_w, int32_t* plan, void* xp, int32_t* chunk_counts, cudaStream_t st) {
  int rc;
  if (T <= kSmallMaxTokens && static_cast<long long>(T) * k <= kSmallMaxPairs) {
    // small batch: one block routes it (same decisions, same plan), and copies the rows too when
    // they are few; otherwise the grid-wide permute follows
    const bool fused_permute = static_cast<long long>(T) * k * H * 2 <= kSmallPermuteBytes;
    const int epl = (E + 31) / 32;
    if (epl <= 1) rc = route_small_launch_epl<1>(logits, T, E, k, H, x, topk_idx, topk_w, plan, xp, fused_permute, st);
    else if (epl <= 2) rc = route_small_launch_epl<2>(logits, T, E, k, H, x, topk_idx, topk_w, plan, xp, fused_permute, st);
    else if (epl <= 4) rc = route_small_launch_epl<4>(logits, T, E, k, H, x, topk_idx, topk_w, plan, xp, fused_permute, st);
    else if (epl <= 8) rc = route_small_launch_epl<8>(logits, T, E, k, H, x, topk_idx, topk_w, plan, xp, fused_permute, st);
    else if (epl <= 16) rc = route_small_launch_epl<16>(logits, T, E, k, H, x, topk_idx, topk_w, plan, xp, fused_permute, st);
    else rc = route_small_launch_epl<32>(logits, T, E, k, H, x, topk_idx, topk_w, plan, xp, fused_permute, st);
    if (rc || fused_permute) return rc;
    return permute_launch(x, plan + 2 * E + 1 + static_cast<long long>(T) * k, T, k, H, xp, st);
  }
  // top-k + gates
  {
    const int threads = kTopkThreads;
    const long long blocks = (static_cast<long long>(T) * 32 + threads - 1) / threads;
    const int epl = (E + 31) / 32;
    ProfScope prof("topk_gate", st);
    const dim3 g(static_cast<unsigned>(blocks)), b(threads);
    cudaError_t e;
    if (epl <= 1) e = launch_kernel(topk_gate_kernel<1>, g, b, 0, st, logits, T, E, k, topk_idx, topk_w);
    else if (epl <= 2) e = launch_kernel(topk_gate_kernel<2>, g, b, 0, st, logits, T, E, k, topk_idx, topk_w);
    else if (epl <= 4) e = launch_kernel(topk_gate_kernel<4>, g, b, 0, st, logits, T, E, k, topk_idx, topk_w);
    else if (epl <= 8) e = launch_kernel(topk_gate_kernel<8>, g, b, 0, st, logits, T, E, k, topk_idx, topk_w);
    else if (epl <= 16) e = launch_kernel(topk_gate_kernel<16>, g, b, 0, st, logits, T, E, k, topk_idx, topk_w);
    else e = launch_kernel(topk_gate_kernel<32>, g, b, 0, st, logits, T, E, k, topk_idx, topk_w);
    if ((rc = check_cuda(e, "topk_gate_kernel"))) return rc;
  }
  return dispatch_launch(topk_idx, T, E, k, H, x, plan, xp, chunk_counts, st);
}

int replay_launch(const float* logits, const int32_t* idx_in, int T, int E, int k, int H, const void* x,
                  int32_t* idx_safe, float* topk_w, int32_t* plan, void* xp, int32_t* chunk_counts,
                  unsigned int* status, cudaStream_t st) {
  int rc;
  {
    const int threads = 256;
    const long long blocks = (static_cast<long long>(T) * 32 + threads - 1) / threads;
    ProfScope prof("replay_gate", st);
    rc = check_cuda(launch_kernel(replay_gate_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, st,
                                  logits, idx_in, T, E, k, idx_safe, topk_w, status),
                    "replay_gate_kernel");
    if (rc) return rc;
  }
  return dispatch_launch(idx_safe, T, E, k, H, x, plan, xp, chunk_counts, st);
}

int dispatch_launch(const int32_t* topk_idx, int T, int E, int k, int H, const void* x, int32_t* plan, void* xp,
                    int32_t* chunk_counts, cudaStream_t st) {
  int rc;
  int32_t* counts = plan;
  int32_t* offsets = plan + E;
  const long long S = static_cast<long long>(T) * k;
  int32_t* row_token = plan + 2 * E + 1;
  int32_t* slot_row = row_token + S;
  // dispatch plan
  const int NC = (T + kDispatchChunk - 1) / kDispatchChunk;
  {
    ProfScope prof("dispatch_count", st);
    rc = check_cuda(launch_kernel(dispatch_count_kernel, dim3(NC), dim3(256), E * sizeof(int), st, topk_idx, T, E,
                                  k, chunk_counts),
                    "dispatch_count_kernel");
  }
  if (rc) return rc;
  {
    ProfScope prof("dispatch_scan", st);
    rc = check_cuda(launch_kernel(dispatch_scan_kernel, dim3(1), dim3(1024), 0, st, chunk_counts, NC, E, counts,
                                  offsets),
                    "dispatch_scan_kernel");
  }
  if (rc) return rc;
  {
    ProfScope prof("dispatch_scatter", st);
    rc = check_cuda(launch_kernel(dispatch_scatter_kernel, dim3(NC), dim3(32),
                                  (static_cast<size_t>(E) + static_cast<size_t>(kDispatchChunk) * k) * sizeof(int), st,
                                  topk_idx, T, E,
                                  k, static_cast<const int32_t*>(chunk_counts), static_cast<const int32_t*>(offsets),
                                  row_token, slot_row),
                    "dispatch_scatter_kernel");
  }
  if (rc) return rc;
  return permute_launch(x, slot_row, T, k, H, xp, st);
}

int permute_launch(const void* x, const int32_t* slot_row, int T, int k, int H, void* xp, cudaStream_t st) {
  int rc;
  const int vec_per_row = H / 8;
  int sms = 0;
  if ((rc = device_sm_count(&sms))) return rc;
  // a warp per token; with fewer tokens than about four per SM, a warp per 2 KB segment of a
  // token's row (128 vectors), so that small batches are not copied by a handful of warps
  const int seg_vec = static_cast<long long>(T) < 4LL * sms ? 128 : (vec_per_row > 0 ? vec_per_row : 1);
  const int nseg = vec_per_row > 0 ? (vec_per_row + seg_vec - 1) / seg_vec : 1;
  const long long items = static_cast<long long>(T) * nseg;
  // at most 8 resident blocks of 256 threads per SM
  long long blocks = (items + kPermuteThreads / 32 - 1) / (kPermuteThreads / 32);
  const long long cap = static_cast<long long>(sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks > 0 && vec_per_row > 0) {
    ProfScope prof("permute_rows", st);
    rc = check_cuda(launch_kernel(permute_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kPermuteThreads), 0,
                                  st, static_cast<const uint4*>(x), slot_row, static_cast<long long>(T), k, vec_per_row,
                                  seg_vec, nseg, static_cast<uint4*>(xp)),
                    "permute_rows_kernel");
    if (rc) return rc;
  }
  return INVMOE_OK;
}

}  // namespace invmoe
