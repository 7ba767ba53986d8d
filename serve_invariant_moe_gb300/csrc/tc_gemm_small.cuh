// tc_gemm_small.cuh -- dense fp32-out GEMM for at most 64 rows of A (sm_103a): the router GEMM of a
// decode-sized batch.
//
// D[m, n] = sum_k A[m, k] * B[n, k] for m < M <= 64, one 64-column block of B per CTA (no unit
// queue: one tile per CTA).  The arithmetic of every element is that of the engines in
// tc_gemm.cuh: bf16 products, K ascending in 64-wide blocks of four K = 16 MMA steps, fp32
// accumulation in TMEM (an M = 64 MMA there too for a tile of at most 64 rows), no split of K.
// So a logit computed here has the bits the row-tile engine gives it in any other batch.
//
// What differs is the load pipeline.  A K loop of a decode-sized tile moves few bytes per K block,
// and its time goes to issuing copies and recycling ring stages, not to bytes or MMAs (one thread
// issues a tile copy every ~55-65 ns, a ring stage round trip adds ~120 ns more, while a dependent
// chain of M = 64..128, N <= 64 MMAs runs at ~29 ns per MMA).  Here a ring stage holds kSmallKsub
// consecutive K blocks of both operands, each operand loaded by ONE rank-3 TMA copy (64 elements x
// 64 rows x kSmallKsub blocks of 64 columns of K): two copies per stage feed 4 * kSmallKsub MMAs.
//   * A: the M <= 64 rows of X, as (64, rows, K / 64), in 64-row copies (16-row ones for M <= 16,
//     see SmallShape); rows past M are zero-filled by the copy.
//   * B: 64 rows of W starting at row 64 * blockIdx.x, as (64, rows, K / 64).
//   Each 64-row x 128-byte slice of a box lands 8 KB apart in shared memory with the 128-byte
//   swizzle of a 2-D box, which is the operand layout of one K block.
//   * A last stage past K holds zero-filled blocks; their MMAs are not issued.
// EPI_F32 writes D (fp32) for 64 columns per CTA.  EPI_SWIGLU computes h = silu(g) * u (the
// expression of the other engines, bf16 round to nearest) for 32 columns of h per CTA: B is the gate
// rows [32c, 32c + 32) and the matching up rows N + 32c.. in one rank-4 copy (64, 32 rows, gate/up,
// K blocks), which lands per K block as 32 gate rows then 32 up rows, so one N = 64 MMA gives the
// CTA's gate columns in accumulator columns [0, 32) and its up columns in [32, 64).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"
#include "tc_gemm.cuh"

namespace invmoe {

constexpr int kSmallKsub = 4;                              // K blocks per ring stage
constexpr int kSmallThreads = 64 + 128;                    // producer warp, MMA warp, 4 epilogue warps

// ABOX: rows of A per copy, 64 or (for at most 16 rows) 16.  A stage holds A's kSmallKsub slices of
// ABOX rows x 128 B, then B's of 64 rows x 128 B.  With 16-row slices (2 KB apart) the M = 64 MMA of
// slice j also reads the next 48 rows' worth of bytes (other slices, or B): they only feed
// accumulator rows 16..63, which are never stored; the smaller stage leaves room for 5 of them.
template <int ABOX>
struct SmallShape {
  static_assert(ABOX == 64 || ABOX == 16, "A rows per copy");
  static constexpr int A_SLICE = ABOX * 128;
  static constexpr int B_SLICE = 64 * 128;
  static constexpr int STAGE_BYTES = kSmallKsub * (A_SLICE + B_SLICE);   // 64 KB or 40 KB
  static constexpr int STAGES = ABOX == 64 ? 3 : 5;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 8 * (2 * STAGES + 1) + 16;
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// TMA load of rank 4 into this CTA's shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// TMA load of rank 3 into this CTA's shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

template <int EPI, int ABOX>
__global__ void __launch_bounds__(kSmallThreads, 1)
    tc_gemm_small_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         int M, int N, int K, void* __restrict__ out, long long ldo, unsigned int* status,
                         unsigned long long timeout_ns) {
  static_assert(EPI == EPI_F32 || EPI == EPI_SWIGLU, "epilogue");
  using S = SmallShape<ABOX>;
  constexpr int kSmallStages = S::STAGES;
  constexpr int kSmallStageBytes = S::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(ring + kSmallStages * kSmallStageBytes);
  uint64_t* empty_bar = full_bar + kSmallStages;
  uint64_t* acc_bar = empty_bar + kSmallStages;
  uint32_t* misc = reinterpret_cast<uint32_t*>(acc_bar + 1);
  uint32_t* tmem_slot = misc;
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSmallStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(acc_bar, 1);
    *s_abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // everything above touches only shared memory, TMEM and the kernel parameters
  pdl_wait();
  pdl_trigger();

  const uint32_t tmem_base = *tmem_slot;
  const int num_kb = K / kBK;
  const int num_st = (num_kb + kSmallKsub - 1) / kSmallKsub;
  // first output column of this CTA: 64 per CTA (fp32 D), 32 per CTA (h)
  const int n0 = static_cast<int>(blockIdx.x) * (EPI == EPI_SWIGLU ? 32 : 64);
  WaitCtl wc{s_abort, status, timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int filled_phase[kSmallStages];
#pragma unroll
      for (int s = 0; s < kSmallStages; ++s) filled_phase[s] = -1;
      for (int ks = 0; ks < num_st; ++ks) {
        if (!mbar_wait(&empty_bar[stage], phase ^ 1u, wc)) break;
        uint8_t* st = ring + stage * kSmallStageBytes;
        // a box counts its full size, zero-filled rows and blocks included
        mbar_arrive_expect_tx(&full_bar[stage], kSmallStageBytes);
        tma_load_3d(st, &tmA, &full_bar[stage], 0, 0, ks * kSmallKsub);
        if (EPI == EPI_SWIGLU)
          tma_load_4d(st + kSmallKsub * S::A_SLICE, &tmB, &full_bar[stage], 0, n0, 0, ks * kSmallKsub);
        else
          tma_load_3d(st + kSmallKsub * S::A_SLICE, &tmB, &full_bar[stage], 0, n0, ks * kSmallKsub);
        filled_phase[stage] = static_cast<int>(phase);
        if (++stage == kSmallStages) { stage = 0; phase ^= 1u; }
      }
      // every copy this thread issued lands before the CTA can exit
      WaitCtl drain{nullptr, status, timeout_ns};
      for (int s = 0; s < kSmallStages; ++s)
        if (filled_phase[s] >= 0) mbar_wait(&full_bar[s], static_cast<uint32_t>(filled_phase[s]), drain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(64, 64);
      const uint64_t adesc0 = sdesc_k_sw128(smem_u32(ring));
      const uint64_t bdesc0 = sdesc_k_sw128(smem_u32(ring + kSmallKsub * S::A_SLICE));
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int ks = 0; ks < num_st; ++ks) {
        if (!mbar_wait(&full_bar[stage], phase, wc)) { ok = false; break; }
        tc_fence_after();
        const int nsub = min(kSmallKsub, num_kb - ks * kSmallKsub);
        for (int j = 0; j < nsub; ++j) {
          const int kb = ks * kSmallKsub + j;     // K blocks ascending, one accumulation chain
          const uint64_t sa = static_cast<uint64_t>((stage * kSmallStageBytes + j * S::A_SLICE) >> 4);
          const uint64_t sb = static_cast<uint64_t>((stage * kSmallStageBytes + j * S::B_SLICE) >> 4);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16(tmem_base, adesc0 + sa + 2u * kk, bdesc0 + sb + 2u * kk, IDESC, (kb | kk) != 0 ? 1u : 0u);
        }
        umma_commit(&empty_bar[stage]);
        if (++stage == kSmallStages) { stage = 0; phase ^= 1u; }
      }
      // the accumulator is complete (or, after a timeout, every issued MMA has finished; the
      // abort flag is up before the epilogue can see the commit)
      if (!ok) *s_abort = 1;
      umma_commit(acc_bar);
      // every MMA issued here has finished before the CTA releases TMEM
      WaitCtl drain{nullptr, status, timeout_ns};
      mbar_wait(acc_bar, 0, drain);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // M = 64 accumulator: row 16q + L in lane L (< 16) of TMEM lane quadrant q
    const int q = warp & 3;
    const bool okw = mbar_wait(acc_bar, 0, wc);
    // one decision per warp, so that the .sync.aligned TMEM loads below never run diverged
    if (__all_sync(0xffffffffu, okw && !*s_abort)) {
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      uint32_t v0[32], v1[32];
      tmem_ld32(tbase, v0);
      tmem_ld32(tbase + 32, v1);
      tmem_ld_wait();
      tmem_reg_fence(v0);
      tmem_reg_fence(v1);
      const int row = q * 16 + lane;
      if (lane < 16 && row < M) {
        if (EPI == EPI_SWIGLU) {
          // h[row, n0 + j] = silu(g_j) * u_j, g in accumulator columns [0, 32), u in [32, 64)
          uint32_t packed[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float h0 = __fmul_rn(silu_f32(__uint_as_float(v0[2 * j])), __uint_as_float(v1[2 * j]));
            const float h1 = __fmul_rn(silu_f32(__uint_as_float(v0[2 * j + 1])), __uint_as_float(v1[2 * j + 1]));
            packed[j] = pack_bf16x2(h0, h1);
          }
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + static_cast<long long>(row) * ldo + n0;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4*>(o + 8 * c) =
                make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
        } else {
          float* o = static_cast<float*>(out) + static_cast<long long>(row) * ldo + n0;
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            if (n0 + c < N)
              *reinterpret_cast<uint4*>(o + c) = make_uint4(v0[c], v0[c + 1], v0[c + 2], v0[c + 3]);
            if (n0 + 32 + c < N)
              *reinterpret_cast<uint4*>(o + 32 + c) = make_uint4(v1[c], v1[c + 1], v1[c + 2], v1[c + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 64);
  }
}

}  // namespace invmoe
