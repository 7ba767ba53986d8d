// tc_gemm2.cuh -- the CTA-pair (cta_group::2) tcgen05 GEMM engine (sm_103a).
//
// Same contract as tc_gemm.cuh -- one fixed tile per call site, K ascending in
// 64-wide blocks of four K=16 MMAs, fp32 accumulation in TMEM, no split-K, rows
// past a group's end computed but never stored -- with a 256 x 256 tile computed
// by a pair of CTAs on two SMs (a cluster of 2):
//   * CTA r of the pair loads A rows [row0 + 128r, +128) and B rows
//     [b_row + 128r, +128) (for SwiGLU: CTA 0 the 128 gate rows, CTA 1 the 128 up
//     rows of the column block) into its own shared memory: 32 KB per stage;
//   * the even CTA issues tcgen05.mma.cta_group::2 with M = 256, N = 256: the
//     hardware reads A from each CTA for that CTA's 128 rows and B from both;
//     each CTA's TMEM receives its own 128 rows x 256 fp32 columns;
//   * commits are multicast to both CTAs (ring slot free, accumulator ready);
//     the odd CTA's TMA completions and epilogue releases are counted on the
//     even CTA's barriers.
// Per SM this halves the weight bytes per MMA compared with a 128 x 256 tile and
// keeps two 256-column accumulators per CTA, so the epilogue of one tile
// overlaps the main loop of the next.  The pairing changes only which SM holds
// which row; every element's reduction is the same K-ascending chain.
//
// Operand majorness (A_MN / B_MN): a K-major operand is stored [rows, K] and
// arrives as one 128-row x 64-K box per stage; an MN-major operand is stored
// [K, rows] (its row index contiguous, as Wv is for dHs = dZ Wv, and as dZ and
// Hs are for dWv = dZ^T Hs) and arrives as two 64-row x 64-K boxes.  Only the
// shared-memory layout and the descriptors change; the MMAs, their K order and
// the accumulation are the same.  A reduction length K that is not a multiple
// of 64 is padded by the tensor map's zero fill (0 * 0 adds nothing).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"
#include "tc_gemm.cuh"

namespace invmoe {

template <int EPI, int STAGES>
struct PairShape {
  static constexpr int BN = 256;                 // pair tile: 256 rows x 256 columns
  static constexpr int TILE_BYTES = kBM * kBK * 2;   // 16 KB: 128 rows x 64 bf16
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES; // own A rows + own B half
  static constexpr int ACC_COLS = 256;
  static constexpr int ACC_STAGES = 2;
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int THREADS = 64 + EPI_THREADS;
  static constexpr int QDEPTH = 4;              // scheduled-unit queue depth
  static constexpr int MAX_GROUPS = 1024;
  static constexpr int BAR_BYTES = 8 * (2 * STAGES + 2 * ACC_STAGES + 1 + 2 * QDEPTH);
  static constexpr int MISC_BYTES = 16 + 4 * QDEPTH;
  static constexpr int OSTAGE_BYTES = EPI_WARPS * kOutStageBytes;   // epilogue store staging
  static constexpr int SMEM_BYTES =
      1024 + STAGES * STAGE_BYTES + OSTAGE_BYTES + BAR_BYTES + MISC_BYTES + 4 * (MAX_GROUPS + 1);
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ uint32_t dlogit_bf16x2(float z0, float z1, bool t0, bool t1, float lse, float g) {
  // d = g * (onehot - p), p = exp(z - lse); the target column takes 1 - p
  const float p0 = expf(z0 - lse), p1 = expf(z1 - lse);
  const float d0 = __fmul_rn(g, t0 ? __fsub_rn(1.0f, p0) : -p0);
  const float d1 = __fmul_rn(g, t1 ? __fsub_rn(1.0f, p1) : -p1);
  return pack_bf16x2(d0, d1);
}

template <int EPI, int STAGES, bool A_MN = false, bool B_MN = false>
__global__ void __launch_bounds__(PairShape<EPI, STAGES>::THREADS, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmO, const GemmParams p) {
  using S = PairShape<EPI, STAGES>;
  constexpr int BN = S::BN;
  static_assert(!(B_MN && EPI == EPI_SWIGLU), "SwiGLU reads gate/up row blocks of a K-major B");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* ostage = smem + STAGES * S::STAGE_BYTES;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * S::STAGE_BYTES + S::OSTAGE_BYTES);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* accf_bar = empty_bar + STAGES;
  uint64_t* acce_bar = accf_bar + S::ACC_STAGES;
  uint64_t* final_bar = acce_bar + S::ACC_STAGES;
  uint64_t* qfull_bar = final_bar + 1;
  uint64_t* qempty_bar = qfull_bar + S::QDEPTH;
  uint32_t* misc = reinterpret_cast<uint32_t*>(qempty_bar + S::QDEPTH);
  uint32_t* tmem_slot = misc;
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + 1);
  int* s_total = reinterpret_cast<int*>(misc + 2);
  volatile int* s_queue = reinterpret_cast<volatile int*>(misc + 4);    // [QDEPTH]
  int* s_prefix = reinterpret_cast<int*>(misc + 4 + S::QDEPTH);         // [G+1]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();          // 0 = leader (issues the MMAs), 1 = follower
  const uint32_t peer = rank ^ 1u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < S::ACC_STAGES; ++a) {
      mbar_init(&accf_bar[a], 1);
      mbar_init(&acce_bar[a], 2 * S::EPI_THREADS);
    }
    mbar_init(final_bar, 1);
    for (int qq = 0; qq < S::QDEPTH; ++qq) {
      mbar_init(&qfull_bar[qq], 1);
      // consumers of a queue slot: per CTA its epilogue threads, plus the
      // leader's MMA thread and the follower's producer thread
      mbar_init(&qempty_bar[qq], 2 + 2 * S::EPI_THREADS);
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, S::TMEM_COLS);
  // everything above touches only shared memory, TMEM and the kernel parameters; the
  // previous kernel on the stream (which wrote this kernel's inputs) is waited for here
  pdl_wait();
  pdl_trigger();

  constexpr int CH = 2 * kBM;   // rows per pair unit
  if (warp == 2) {
    if (p.G > 0) {
      const int per = (p.G + 31) / 32;
      const int g0 = lane * per;
      int local = 0;
      for (int i = 0; i < per; ++i) {
        const int g = g0 + i;
        if (g < p.G) local += (__ldg(p.counts + g) + CH - 1) / CH;
      }
      int incl = local;
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      int run = incl - local;
      for (int i = 0; i < per; ++i) {
        const int g = g0 + i;
        if (g < p.G) {
          s_prefix[g] = run;
          run += (__ldg(p.counts + g) + CH - 1) / CH;
        }
      }
      if (lane == 31) {
        s_prefix[p.G] = incl;
        *s_total = incl;
      }
    } else if (lane == 0) {
      *s_total = (p.M + CH - 1) / CH;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();     // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int total_chunks = *s_total;
  const int total_units = total_chunks * p.n_blocks;
  const int num_kb = (p.K + kBK - 1) / kBK;
  WaitCtl wc{s_abort, p.status, p.timeout_ns};
  const uint32_t peer_abort = mapa_shared(smem_u32(const_cast<int*>(s_abort)), peer);
  const uint32_t qempty_leader0 = mapa_shared(smem_u32(&qempty_bar[0]), 0);
  // Units are handed out dynamically by the leader's producer: it takes the next
  // index from a global counter and publishes it into both CTAs' queues.  Every
  // consumer releases a slot on the leader's qempty barrier.

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int filled_phase[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) filled_phase[s] = -1;
      bool ok = true;
      int qi = 0;
      uint32_t qphase = 0;
      const uint32_t q_peer0 = mapa_shared(smem_u32(const_cast<int*>(s_queue)), peer);
      const uint32_t qfull_peer0 = mapa_shared(smem_u32(&qfull_bar[0]), peer);
      // the leader's first unit is its pair index (no counter round trip on the way in); later
      // ones come from the counter, offset past those
      bool first = true;
      while (ok) {
        int u;
        if (rank == 0) {
          const int pairs = static_cast<int>(gridDim.x) / 2;
          u = first ? static_cast<int>(blockIdx.x) / 2 : pairs + atomicAdd(p.sched, 1);
          first = false;
          if (u >= total_units) u = -1;
          if (!mbar_wait<true>(&qempty_bar[qi], qphase ^ 1u, wc)) { ok = false; break; }
          s_queue[qi] = u;
          mbar_arrive(&qfull_bar[qi]);
          st_shared_remote_u32(q_peer0 + 4u * qi, static_cast<uint32_t>(u));
          mbar_arrive_remote(qfull_peer0 + 8u * qi);
        } else {
          if (!mbar_wait<true>(&qfull_bar[qi], qphase, wc)) { ok = false; break; }
          u = s_queue[qi];
          mbar_arrive_remote(qempty_leader0 + 8u * qi);
        }
        if (++qi == S::QDEPTH) { qi = 0; qphase ^= 1u; }
        if (u < 0) break;
        const Unit U = decode_unit<2, EPI, BN>(u, p, s_prefix, total_chunks);
        const int a_row = U.row0 + static_cast<int>(rank) * kBM;
        const int b_row = (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD) ? U.b_row + static_cast<int>(rank) * p.b_up_rows
                                                                        : U.b_row + static_cast<int>(rank) * kBM;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, wc)) { ok = false; break; }
          uint8_t* st = ring + stage * S::STAGE_BYTES;
          const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], 2 * S::STAGE_BYTES);
          if (A_MN) {
            tma_load_2d_pair(st, &tmA, fb, a_row, kb * kBK);
            tma_load_2d_pair(st + kMnBoxBytes, &tmA, fb, a_row + 64, kb * kBK);
          } else {
            tma_load_2d_pair(st, &tmA, fb, kb * kBK, a_row);
          }
          if (B_MN) {
            tma_load_2d_pair(st + S::TILE_BYTES, &tmB, fb, b_row, kb * kBK);
            tma_load_2d_pair(st + S::TILE_BYTES + kMnBoxBytes, &tmB, fb, b_row + 64, kb * kBK);
          } else {
            tma_load_2d_pair(st + S::TILE_BYTES, &tmB, fb, kb * kBK, b_row);
          }
          filled_phase[stage] = static_cast<int>(phase);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) st_shared_remote_u32(peer_abort, 1u);
      // this CTA takes no more units (the follower's last one came from the leader after the
      // leader's last counter access): once every CTA is past this point the counter is reset
      sched_release(p.sched);
      // The leader's full barrier counts both CTAs' copies; it may only drain its own.
      if (rank == 0) {
        WaitCtl drain{nullptr, p.status, p.timeout_ns};
        for (int s = 0; s < STAGES; ++s)
          if (filled_phase[s] >= 0) mbar_wait(&full_bar[s], static_cast<uint32_t>(filled_phase[s]), drain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t IDESC = idesc_bf16_f32(2 * kBM, BN, A_MN, B_MN);
      // per K = 16 step: +32 B inside a K-major swizzle row, +2048 B (16 rows) MN-major; encoded >> 4
      constexpr uint64_t A_STEP = A_MN ? 128u : 2u;
      constexpr uint64_t B_STEP = B_MN ? 128u : 2u;
      // stage-0 descriptors; stage s adds s * STAGE_BYTES to the start address (encoded >> 4;
      // shared addresses stay below 256 KB, so the 14-bit field never carries)
      const uint64_t adesc0 = A_MN ? sdesc_mn_sw128(smem_u32(ring)) : sdesc_k_sw128(smem_u32(ring));
      const uint64_t bdesc0 = B_MN ? sdesc_mn_sw128(smem_u32(ring + S::TILE_BYTES))
                                   : sdesc_k_sw128(smem_u32(ring + S::TILE_BYTES));
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      int qi = 0;
      uint32_t qphase = 0;
      while (ok) {
        if (!mbar_wait(&qfull_bar[qi], qphase, wc)) { ok = false; break; }
        const int u = s_queue[qi];
        mbar_arrive(&qempty_bar[qi]);
        if (++qi == S::QDEPTH) { qi = 0; qphase ^= 1u; }
        if (u < 0) break;
        if (!mbar_wait<true>(&acce_bar[acc], acc_phase ^ 1u, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * S::ACC_COLS);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, wc)) { ok = false; break; }
          tc_fence_after();
          const uint64_t so = static_cast<uint64_t>((stage * S::STAGE_BYTES) >> 4);
          const uint64_t adesc = adesc0 + so;
          const uint64_t bdesc = bdesc0 + so;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16_pair(d0, adesc + A_STEP * kk, bdesc + B_STEP * kk, IDESC, (kb | kk) != 0 ? 1u : 0u);
          umma_commit_pair(&empty_bar[stage], 0x3);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair(&accf_bar[acc], 0x3);
        if (++acc == S::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok) st_shared_remote_u32(peer_abort, 1u);
      umma_commit_pair(final_bar, 0x1);
      WaitCtl drain{nullptr, p.status, p.timeout_ns};
      mbar_wait(final_bar, 0, drain);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int ew = warp - 2;
    const int q = warp & 3;
    const int half = ew >> 2;
    const int r_in_tile = q * 32 + lane;
    const uint32_t acce_leader0 = mapa_shared(smem_u32(&acce_bar[0]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    int qi = 0;
    uint32_t qphase = 0;
    while (true) {
      const bool okq = mbar_wait<true>(&qfull_bar[qi], qphase, wc);
      if (!__all_sync(0xffffffffu, okq)) break;
      const int u = s_queue[qi];
      mbar_arrive_remote(qempty_leader0 + 8u * qi);
      if (++qi == S::QDEPTH) { qi = 0; qphase ^= 1u; }
      if (u < 0) break;
      const Unit U = decode_unit<2, EPI, BN>(u, p, s_prefix, total_chunks);
      const bool ok = mbar_wait(&accf_bar[acc], acc_phase, wc);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int row_local = static_cast<int>(rank) * kBM + r_in_tile;
      const bool valid = row_local < U.rows;
      const long long row = static_cast<long long>(U.row0) + row_local;
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * S::ACC_COLS);
      if (EPI == EPI_LSE) {
        if (half == 0) {
          const int n0 = U.nb * BN;
          float* orow = p.out != nullptr ? static_cast<float*>(p.out) + row * p.ldo + n0 : nullptr;
          const int tg = valid ? __ldg(p.target + row) - p.col0 - n0 : -1;
          float mx[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
          float tv = 0.0f;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tbase + c * 32, v);
            tmem_ld_wait();
            tmem_reg_fence(v);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float z = __uint_as_float(v[j]);
              if (n0 + c * 32 + j < p.N) mx[j & 7] = fmaxf(mx[j & 7], z);
              if (tg == c * 32 + j) tv = z;
            }
            if (valid && orow != nullptr) {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (n0 + c * 32 + j * 4 < p.N)
                  *reinterpret_cast<float4*>(orow + c * 32 + j * 4) =
                      make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                  __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
            }
          }
          const float m = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
          float a8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) a8[i] = 0.0f;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld32(tbase + c * 32, v);
            tmem_ld_wait();
            tmem_reg_fence(v);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n0 + c * 32 + j < p.N) a8[j & 7] = __fadd_rn(a8[j & 7], expf(__uint_as_float(v[j]) - m));
          }
          const float sum = __fadd_rn(__fadd_rn(__fadd_rn(a8[0], a8[1]), __fadd_rn(a8[2], a8[3])),
                                      __fadd_rn(__fadd_rn(a8[4], a8[5]), __fadd_rn(a8[6], a8[7])));
          if (valid) {
            p.part[row * p.nch + U.nb] = make_float2(m, sum);
            if (tg >= 0 && tg < BN && n0 + tg < p.N) p.tgt_logit[row] = tv;
          }
        }
      } else if (EPI == EPI_DLOGITS) {
        // one bf16 gradient row segment per thread; N is a multiple of 8, so each
        // 8-column group is either wholly inside the matrix or wholly past it
        const int n0 = U.nb * BN;
        const float lse = valid ? __ldg(p.row_lse + row) : 0.0f;
        const float g = valid ? __ldg(p.row_scale + row) : 0.0f;
        const int tg = valid ? __ldg(p.target + row) - n0 : -1;
        const int rows_valid = U.rows - (static_cast<int>(rank) * kBM + q * 32);
        uint8_t* obase = rows_valid > 0
                             ? reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(p.out) +
                                                          (static_cast<long long>(U.row0) + rank * kBM + q * 32) *
                                                              p.ldo + n0)
                             : nullptr;
        uint8_t* stg = ostage + ew * kOutStageBytes;
#pragma unroll 1
        for (int c = half; c < BN / 32; c += 2) {
          uint32_t v[32];
          tmem_ld32(tbase + c * 32, v);
          tmem_ld_wait();
          tmem_reg_fence(v);
          if (rows_valid > 0) {
            uint32_t packed[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              packed[j] = dlogit_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]),
                                        tg == c * 32 + 2 * j, tg == c * 32 + 2 * j + 1, lse, g);
            stage_store_rows64(stg, packed, obase + c * 64, p.ldo * 2, rows_valid, (p.N - (n0 + c * 32)) * 2);
          }
        }
      } else if (EPI == EPI_F32 && p.out_map && U.rows - (static_cast<int>(rank) * kBM + q * 32) >= 32) {
        // a whole 32-row slab of one group: each 32-row x 16-column piece leaves the warp's
        // staging buffer (64-byte swizzle layout) as one bulk tensor store through the
        // [1][rows][N] map, which clips columns past N
        const int n0 = U.nb * BN;
        const int m0 = U.row0 + static_cast<int>(rank) * kBM + q * 32;
        uint8_t* stg = ostage + ew * kOutStageBytes;
#pragma unroll 1
        for (int c = half; c < BN / 32; c += 2) {
          uint32_t v[32];
          tmem_ld32(tbase + c * 32, v);
          tmem_ld_wait();
          tmem_reg_fence(v);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = n0 + c * 32 + 16 * h;
            if (col >= p.N) break;
            if (lane == 0) bulk_wait_group_read0();    // the previous piece has left the buffer
            __syncwarp();
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
              *reinterpret_cast<uint4*>(stg + lane * 64 + ((qq ^ ((lane >> 1) & 3)) << 4)) =
                  make_uint4(v[16 * h + 4 * qq], v[16 * h + 4 * qq + 1], v[16 * h + 4 * qq + 2],
                             v[16 * h + 4 * qq + 3]);
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmO, stg, col, m0, 0);
              bulk_commit_group();
            }
          }
        }
      } else if (EPI == EPI_F32) {
        const int n0 = U.nb * BN;
        const int rows_valid = U.rows - (static_cast<int>(rank) * kBM + q * 32);
        uint8_t* obase = rows_valid > 0 ? reinterpret_cast<uint8_t*>(static_cast<float*>(p.out) +
                                              (static_cast<long long>(U.row0) + rank * kBM + q * 32) * p.ldo + n0)
                                        : nullptr;
        uint8_t* stg = ostage + ew * kOutStageBytes;
        if (p.out_map) {
          if (lane == 0) bulk_wait_group_read0();    // a bulk store may still read the buffer
          __syncwarp();
        }
#pragma unroll 1
        for (int c = half; c < BN / 32; c += 2) {
          uint32_t v[32];
          tmem_ld32(tbase + c * 32, v);
          tmem_ld_wait();
          tmem_reg_fence(v);
          if (rows_valid > 0) {
            const int bytes_valid = (p.N - (n0 + c * 32)) * 4;
            stage_store_rows64(stg, *reinterpret_cast<uint32_t(*)[16]>(&v[0]), obase + c * 128, p.ldo * 4,
                               rows_valid, bytes_valid);
            stage_store_rows64(stg, *reinterpret_cast<uint32_t(*)[16]>(&v[16]), obase + c * 128 + 64, p.ldo * 4,
                               rows_valid, bytes_valid - 64);
          }
        }
      } else if (EPI == EPI_SWIGLU_BWD) {
        constexpr int HALF = BN / 2;
        const int n0 = U.nb * HALF;
        const int rows_valid = U.rows - (static_cast<int>(rank) * kBM + q * 32);
        const long long r0 = static_cast<long long>(U.row0) + rank * kBM + q * 32;
        uint8_t* stg = ostage + ew * kOutStageBytes;
#pragma unroll 1
        for (int c = half; c < HALF / 32; c += 2) {
          uint32_t gv[32], uv[32];
          tmem_ld32(tbase + c * 32, gv);
          tmem_ld32(tbase + HALF + c * 32, uv);
          tmem_ld_wait();
          tmem_reg_fence(gv);
          tmem_reg_fence(uv);
          if (rows_valid > 0) {
            const int col = n0 + c * 32;
            __nv_bfloat16* dgu = static_cast<__nv_bfloat16*>(p.out) + r0 * p.ldo;
            swiglu_bwd_chunk(stg, gv, uv, reinterpret_cast<const uint8_t*>(p.aux + r0 * p.ld_aux + col), p.ld_aux * 4,
                             reinterpret_cast<uint8_t*>(dgu + col), reinterpret_cast<uint8_t*>(dgu + p.N + col),
                             p.ldo * 2,
                             p.out2 != nullptr ? reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(p.out2) +
                                                                            r0 * p.ldo2 + col)
                                               : nullptr,
                             p.ldo2 * 2, rows_valid, p.N - col);
          }
        }
      } else {
        constexpr int HALF = BN / 2;
        const int n0 = U.nb * HALF;
        const int rows_valid = U.rows - (static_cast<int>(rank) * kBM + q * 32);
        uint8_t* obase = rows_valid > 0
                             ? reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(p.out) +
                                                          (static_cast<long long>(U.row0) + rank * kBM + q * 32) *
                                                              p.ldo + n0)
                             : nullptr;
        uint8_t* stg = ostage + ew * kOutStageBytes;
#pragma unroll 1
        for (int c = half; c < HALF / 32; c += 2) {
          uint32_t gv[32], uv[32];
          tmem_ld32(tbase + c * 32, gv);
          tmem_ld32(tbase + HALF + c * 32, uv);
          tmem_ld_wait();
          tmem_reg_fence(gv);
          tmem_reg_fence(uv);
          if (rows_valid > 0) {
            uint32_t packed[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float h0 = __fmul_rn(silu_f32(__uint_as_float(gv[2 * j])), __uint_as_float(uv[2 * j]));
              const float h1 = __fmul_rn(silu_f32(__uint_as_float(gv[2 * j + 1])), __uint_as_float(uv[2 * j + 1]));
              packed[j] = pack_bf16x2(h0, h1);
            }
            stage_store_rows64(stg, packed, obase + c * 64, p.ldo * 2, rows_valid, (p.N - (n0 + c * 32)) * 2);
          }
        }
      }
      tc_fence_before();
      // release the accumulator on the leader (counts both CTAs' epilogue threads)
      mbar_arrive_remote(acce_leader0 + static_cast<uint32_t>(acc * 8));
      if (++acc == S::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
    }
    // the bulk stores this warp issued complete before the CTA exits
    if (EPI == EPI_F32 && lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();     // no remote arrive or multicast commit can still target this CTA
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, S::TMEM_COLS);
  }
}

}  // namespace invmoe
