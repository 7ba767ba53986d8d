// backward.cu -- the MoE layer's backward outside the GEMM engine: the combine
// backward, the router's softmax backward and the fixed-order un-permute sum.
//
// The trainer's side of the same definition ("位级一致：前沿训练的差异化关键",
// section "端到端零 KLD": the trainer follows the same bit-exact standard as the
// serving path): every sum here runs in an order fixed by the shapes alone, and
// no value is accumulated through atomics, so repeated calls give identical bits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace invmoe {

namespace {

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// One block per token, warp j = slot j (blockDim = 32 * k):
//   dy[slot_row[t, j], :] = bf16(w[t, j] * dout[t, :])
//   dgate[t, j] = sum_h dout[t, h] * y[slot_row[t, j], h]: lane l adds, in
//   ascending order, the elements 4*(l + 32 i) .. +3 of the row (i ascending),
//   then the 32 lane sums fold by a xor butterfly (16, 8, 4, 2, 1).
// Warp 0 also writes dout_bf16[t, :] = bf16(dout[t, :]) when requested.
__global__ void combine_bwd_kernel(const float* __restrict__ dout, const float* __restrict__ y,
                                   const float* __restrict__ topk_w, const int32_t* __restrict__ slot_row, int H,
                                   int k, __nv_bfloat16* __restrict__ dy, float* __restrict__ dgate,
                                   __nv_bfloat16* __restrict__ dout_bf16) {
  const int t = blockIdx.x;
  const int j = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long r = slot_row[static_cast<long long>(t) * k + j];
  const float w = topk_w[static_cast<long long>(t) * k + j];
  const float4* d4 = reinterpret_cast<const float4*>(dout + static_cast<long long>(t) * H);
  const float4* y4 = reinterpret_cast<const float4*>(y + r * H);
  uint2* dy2 = reinterpret_cast<uint2*>(dy + r * H);
  uint2* db2 = dout_bf16 != nullptr ? reinterpret_cast<uint2*>(dout_bf16 + static_cast<long long>(t) * H) : nullptr;
  float acc = 0.0f;
  for (int i = lane; i < H / 4; i += 32) {
    const float4 d = __ldg(d4 + i);
    const float4 v = __ldg(y4 + i);
    acc = __fadd_rn(acc, __fmul_rn(d.x, v.x));
    acc = __fadd_rn(acc, __fmul_rn(d.y, v.y));
    acc = __fadd_rn(acc, __fmul_rn(d.z, v.z));
    acc = __fadd_rn(acc, __fmul_rn(d.w, v.w));
    dy2[i] = make_uint2(pack2(__fmul_rn(w, d.x), __fmul_rn(w, d.y)), pack2(__fmul_rn(w, d.z), __fmul_rn(w, d.w)));
    if (j == 0 && db2 != nullptr) db2[i] = make_uint2(pack2(d.x, d.y), pack2(d.z, d.w));
  }
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, s));
  if (lane == 0) dgate[static_cast<long long>(t) * k + j] = acc;
}

// One warp per token: the gates are w = softmax(s) over the k selected logits, so
//   S = sum_i w_i dgate_i (i ascending),  ds_j = w_j (dgate_j - S),
// and the router-logit gradient row is ds_j at column idx_j, 0 elsewhere (bf16).
__global__ void router_bwd_kernel(const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
                                  const float* __restrict__ dgate, int T, int E, int k,
                                  __nv_bfloat16* __restrict__ dlog) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const long long base = static_cast<long long>(t) * k;
  const float w = lane < k ? topk_w[base + lane] : 0.0f;
  const float dg = lane < k ? dgate[base + lane] : 0.0f;
  const int e_sel = lane < k ? topk_idx[base + lane] : -1;
  const float prod = __fmul_rn(w, dg);
  float S = 0.0f;
  for (int i = 0; i < k; ++i) S = __fadd_rn(S, __shfl_sync(0xffffffffu, prod, i));
  const float ds = __fmul_rn(w, __fsub_rn(dg, S));
  __nv_bfloat16* row = dlog + static_cast<long long>(t) * E;
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    float v = 0.0f;
    for (int i = 0; i < k; ++i) {
      const int ei = __shfl_sync(0xffffffffu, e_sel, i);
      const float di = __shfl_sync(0xffffffffu, ds, i);
      if (ei == e) v = di;
    }
    if (e < E) row[e] = __float2bfloat16_rn(v);
  }
}

// dx[t, :] = ((sum_j dxp[slot_row[t, j], :]) + dx_shared[t, :]) + dx[t, :], the
// slots in rank order, each sum rounded separately; dx holds the router part.
__global__ void unpermute_sum_kernel(const float* __restrict__ dxp, const int32_t* __restrict__ slot_row,
                                     const float* __restrict__ dx_shared, int T, int H, int k, float* __restrict__ dx) {
  const long long n4 = static_cast<long long>(T) * (H / 4);
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = i / (H / 4);
    const long long c = i - t * (H / 4);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const long long r = slot_row[t * k + j];
      const float4 v = __ldg(reinterpret_cast<const float4*>(dxp + r * H) + c);
      s.x = __fadd_rn(s.x, v.x); s.y = __fadd_rn(s.y, v.y); s.z = __fadd_rn(s.z, v.z); s.w = __fadd_rn(s.w, v.w);
    }
    if (dx_shared != nullptr) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(dx_shared + t * H) + c);
      s.x = __fadd_rn(s.x, v.x); s.y = __fadd_rn(s.y, v.y); s.z = __fadd_rn(s.z, v.z); s.w = __fadd_rn(s.w, v.w);
    }
    float4* o = reinterpret_cast<float4*>(dx + t * H) + c;
    const float4 v = *o;
    s.x = __fadd_rn(s.x, v.x); s.y = __fadd_rn(s.y, v.y); s.z = __fadd_rn(s.z, v.z); s.w = __fadd_rn(s.w, v.w);
    *o = s;
  }
}

}  // namespace

int combine_bwd_launch(const float* dout, const float* y, const float* topk_w, const int32_t* slot_row, int T,
                       int H, int k, void* dy, float* dgate, void* dout_bf16, cudaStream_t st) {
  ProfScope prof("combine_bwd", st);
  combine_bwd_kernel<<<T, 32 * k, 0, st>>>(dout, y, topk_w, slot_row, H, k, static_cast<__nv_bfloat16*>(dy), dgate,
                                           static_cast<__nv_bfloat16*>(dout_bf16));
  return check_cuda(cudaGetLastError(), "combine_bwd_kernel");
}

int router_bwd_launch(const int32_t* topk_idx, const float* topk_w, const float* dgate, int T, int E, int k,
                      void* dlog, cudaStream_t st) {
  ProfScope prof("router_bwd", st);
  router_bwd_kernel<<<(T + 7) / 8, 256, 0, st>>>(topk_idx, topk_w, dgate, T, E, k,
                                                 static_cast<__nv_bfloat16*>(dlog));
  return check_cuda(cudaGetLastError(), "router_bwd_kernel");
}

int unpermute_sum_launch(const float* dxp, const int32_t* slot_row, const float* dx_shared, int T, int H, int k,
                         float* dx, cudaStream_t st) {
  int sms = 0;
  int rc = device_sm_count(&sms);
  if (rc) return rc;
  const long long n4 = static_cast<long long>(T) * (H / 4);
  long long blocks = (n4 + 255) / 256;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  ProfScope prof("unpermute_sum", st);
  unpermute_sum_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(dxp, slot_row, dx_shared, T, H, k, dx);
  return check_cuda(cudaGetLastError(), "unpermute_sum_kernel");
}

}  // namespace invmoe
