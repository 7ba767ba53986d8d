// expert_parallel.cu -- regrouping of the rows an expert-parallel rank receives.
//
// With the experts split over ranks (rank r owns experts [e0_r, e1_r)), every
// rank routes its own tokens with the full router and sends each owner the rows
// of its permuted activations xp that belong to the owner's experts.  Because
// xp is sorted by expert, those rows are one contiguous slice per owner; an
// all-to-all delivers them source-major: the rows from source 0 (expert by
// expert), then from source 1, and so on.  The owner needs them expert-major
// to run its grouped GEMMs, and must later send each output row back to the
// position it came from.  Rows are only moved here, never combined: an expert
// output row depends on its own input row alone (one fixed tile, K ascending),
// so it has the same bits on whichever rank and at whichever row position it
// is computed -- the cross-GPU path adds no reduction whose order could change
// ("位级一致：前沿训练的差异化关键", section "为什么比特级一致是一个复杂的问题":
// a cross-device reduction whose algorithm changes with size breaks agreement).
#include <cuda_runtime.h>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace invmoe {

namespace {

constexpr int kPlanThreads = 256;

// Block-wide sum of one long long per thread (integer: exact in any order).
__device__ long long block_sum(long long v, long long* red) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  long long t = 0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kPlanThreads / 32; ++i) t += red[i];
  __syncthreads();
  if (threadIdx.x == 0) red[0] = t;
  __syncthreads();
  const long long out = red[0];
  __syncthreads();
  return out;
}

// Blocks b < n_src * E_local: block b is (source s, local expert e), b = s * E_local + e,
// the source-major order in which the rows arrived.  Its rows start at
//   src = sum of counts[f] over f < b                       (received order)
//   dst = (rows of experts < e from every source) + (rows of expert e from sources < s)
// and row_src[dst + j] = src + j for j < counts[b].  The last block writes the local
// plan (counts per local expert, exclusive offsets) and checks that the counts add up
// to R.  Writes outside [0, R) are skipped, so counts that do not add up cannot make
// a later kernel read or write out of bounds (the status word records the mismatch).
__global__ void __launch_bounds__(kPlanThreads) ep_plan_kernel(const int32_t* __restrict__ cnt, int n_src, int E_local,
                                                               int R, int32_t* __restrict__ plan_local,
                                                               int32_t* __restrict__ row_src,
                                                               unsigned int* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  __shared__ long long red[kPlanThreads / 32];
  const int nflat = n_src * E_local;
  const int b = blockIdx.x;
  if (b < nflat) {
    const int s = b / E_local, e = b - s * E_local;
    long long src = 0, dst = 0;
    for (int f = threadIdx.x; f < nflat; f += kPlanThreads) {
      const long long c = cnt[f];
      const int fs = f / E_local, fe = f - fs * E_local;
      if (f < b) src += c;
      if (fe < e || (fe == e && fs < s)) dst += c;
    }
    src = block_sum(src, red);
    dst = block_sum(dst, red);
    const int n = cnt[b];
    for (int j = threadIdx.x; j < n; j += kPlanThreads) {
      const long long d = dst + j, r = src + j;
      if (d >= 0 && d < R && r >= 0 && r < R) row_src[d] = static_cast<int32_t>(r);
    }
    return;
  }
  // local plan: counts[E_local] | offsets[E_local + 1]
  __shared__ int tot[1024];
  for (int e = threadIdx.x; e < E_local; e += kPlanThreads) {
    long long t = 0;
    for (int s = 0; s < n_src; ++s) t += cnt[s * E_local + e];
    tot[e] = static_cast<int>(t);
    plan_local[e] = static_cast<int32_t>(t);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    long long run = 0;
    bool bad = false;
    for (int e = 0; e < E_local; ++e) {
      plan_local[E_local + e] = static_cast<int32_t>(run);
      bad |= tot[e] < 0;
      run += tot[e];
    }
    plan_local[2 * E_local] = static_cast<int32_t>(run);
    if (bad || run != R) atomicOr(status, kStatusBadCounts);
  }
}

// xp_local[i, :] = recv[row_src[i], :], 16-byte vectors, one warp per row.
__global__ void ep_gather_kernel(const uint4* __restrict__ recv, const int32_t* __restrict__ row_src, int R,
                                 int vec_per_row, uint4* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long nw = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5); i < R; i += nw) {
    const int r = __ldg(row_src + i);
    if (r < 0 || r >= R) continue;    // counts that did not add up (recorded in the status word)
    const uint4* src = recv + static_cast<long long>(r) * vec_per_row;
    uint4* dst = out + i * vec_per_row;
    for (int c = lane; c < vec_per_row; c += 32) dst[c] = __ldg(src + c);
  }
}

// y_send[row_src[i], :] = y_local[i, :], fp32 rows in 16-byte vectors, one warp per row.
__global__ void ep_scatter_kernel(const float4* __restrict__ y_local, const int32_t* __restrict__ row_src, int R,
                                  int vec_per_row, float4* __restrict__ y_send) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const long long nw = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5); i < R; i += nw) {
    const int r = __ldg(row_src + i);
    if (r < 0 || r >= R) continue;
    const float4* src = y_local + i * vec_per_row;
    float4* dst = y_send + static_cast<long long>(r) * vec_per_row;
    for (int c = lane; c < vec_per_row; c += 32) dst[c] = __ldg(src + c);
  }
}

int row_grid(long long rows) {
  int sms = 0;
  if (device_sm_count(&sms)) return 0;
  long long blocks = (rows + 7) / 8;            // 8 warps per block, a warp per row
  const long long cap = static_cast<long long>(sms) * 8;
  return static_cast<int>(blocks < cap ? blocks : cap);
}

}  // namespace

int ep_regroup_launch(const void* recv_xp, const int32_t* recv_counts, int n_src, int E_local, int R, int H,
                      void* xp_local, int32_t* plan_local, int32_t* row_src, unsigned int* status, cudaStream_t st) {
  int rc;
  {
    ProfScope prof("ep_plan", st);
    rc = check_cuda(launch_kernel(ep_plan_kernel, dim3(n_src * E_local + 1), dim3(kPlanThreads), 0, st, recv_counts,
                                  n_src, E_local, R, plan_local, row_src, status),
                    "ep_plan_kernel");
    if (rc) return rc;
  }
  if (R == 0) return INVMOE_OK;
  const int blocks = row_grid(R);
  if (blocks <= 0) return set_error(INVMOE_ERR_CUDA, "could not size the regroup grid");
  ProfScope prof("ep_gather_rows", st);
  return check_cuda(launch_kernel(ep_gather_kernel, dim3(blocks), dim3(256), 0, st,
                                  static_cast<const uint4*>(recv_xp), static_cast<const int32_t*>(row_src), R, H / 8,
                                  static_cast<uint4*>(xp_local)),
                    "ep_gather_kernel");
}

int ep_ungroup_launch(const float* y_local, const int32_t* row_src, int R, int H, float* y_send, cudaStream_t st) {
  const int blocks = row_grid(R);
  if (blocks <= 0) return set_error(INVMOE_ERR_CUDA, "could not size the ungroup grid");
  ProfScope prof("ep_scatter_rows", st);
  return check_cuda(launch_kernel(ep_scatter_kernel, dim3(blocks), dim3(256), 0, st,
                                  reinterpret_cast<const float4*>(y_local), row_src, R, H / 4,
                                  reinterpret_cast<float4*>(y_send)),
                    "ep_scatter_kernel");
}

}  // namespace invmoe
