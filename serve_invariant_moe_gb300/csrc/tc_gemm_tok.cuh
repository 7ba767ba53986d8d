// tc_gemm_tok.cuh -- grouped expert GEMMs with the tokens on the MMA's N side (sm_103a).
//
// The expert GEMMs of the layer multiply each expert's token rows by that
// expert's weights.  The row-tile engines (tc_gemm.cuh, tc_gemm2.cuh) put the
// tokens on the MMA's M side, in tiles of 128 (or 64) rows: an expert with 269
// tokens then runs as a 256-row unit and a 13-row unit, and the 13-row unit
// streams the whole weight tile again for 5 % of the work.  This engine puts the
// weights on the M side and the tokens on the N side, where the MMA takes any
// multiple of 16 up to 256 (and a second MMA extends it to kTokChunk columns):
//   D^T[w, t] = sum_k W[w, k] * X[t, k]       (W: an expert's weight rows, X: its tokens)
// on a CTA pair (cta_group::2, M = 256 weight rows, 128 per CTA).  One unit is
// (expert, token chunk of at most kTokChunk tokens, weight block); an expert
// with up to kTokChunk tokens is one chunk, so its weights stream exactly once.
//
// Per-element arithmetic is that of the row-tile engines: the same bf16
// products, K ascending in 64-wide blocks of four K = 16 steps, fp32
// accumulation in TMEM, no split-K (swapping the operands' roles, the tile
// position and the N of the MMA change no bit of an element; the tests compare
// this engine's outputs with the row-tile engines' bit for bit).
//
//   * CTA r loads its 128 weight rows of the block and its half of the token
//     rows, each as one TMA box per stage (at this size the producer thread's
//     copy issue, not the bytes, sets the pace; rows past the chunk are read
//     from L2 and never stored).  A chunk of at most 256 tokens is one MMA of
//     N1 columns, CTA r holding tokens [r*N1/2, (r+1)*N1/2) in a 32-, 64- or
//     128-row box.  A longer chunk adds a second MMA of N2 columns, and CTA 0
//     holds tokens [0, 128 + N2/2), CTA 1 the next 128 + N2/2, each in one
//     160-row box whose rows [0, 128) feed MMA 1 and rows [128, 128 + N2/2)
//     MMA 2; the epilogue maps the columns back to tokens (MMA 1 column j >= 128
//     is token j + N2/2, MMA 2 column j is token 128 + j below N2/2, else
//     256 + j).  SwiGLU: the CTA's h columns are [f0, f0 + 64),
//     f0 = 128 * block + 64 * r, and its weight rows arrive as 4 groups of 16
//     gate rows and the matching 16 up rows: tile rows 32i + [0, 16) are the
//     gate rows of h columns f0 + 16i + [0, 16), tile rows 32i + [16, 32) the
//     up rows, so the warp on TMEM lanes 32i holds both halves of its 16 SwiGLU
//     pairs and exchanges them with one shuffle.
//   * Prefill-sized units of at most 256 experts run a 6-stage ring (216 KB of operands
//     in flight per CTA; the GEMM is paced per SM by the bytes it keeps in flight), with
//     smaller epilogue staging tiles (the fp32 store then leaves in passes of 8 tokens).
//   * Smaller batches run the same kernel with smaller units (an expert with
//     more tokens takes several): at most 1024 token slots or 16 per expert
//     (decode), units of at most 64 tokens, a 32-row token tile per CTA, 20 KB
//     per K block and a ring of 5 stages of two K blocks each; at most 64 slots
//     per expert, units of at most 128 tokens, a 64-row tile, 24 KB per K block
//     (SwiGLU: 4 stages of two K blocks; fp32: 8 stages of one).
//   * TMEM: lane = weight row, one column per token.  Consecutive units of a CTA
//     alternate between two placements: slot 0 puts MMA 1 at column 0 and MMA 2
//     at column 256 (columns [0, 320)), slot 1 puts MMA 1 at column 256 and
//     MMA 2 at column 192 (columns [192, 512)).  Two consecutive units share
//     only columns [192, 320): the epilogue drains its chunks there first and
//     releases them, and the next unit's MMAs run while it drains the rest;
//     when neither unit has a second MMA they share no column at all and the
//     next unit's MMAs do not wait.
//   * Epilogues read 32 token columns per tcgen05.ld (two loads per wait),
//     release a phase's columns (one arrive per warp) as soon as its last loads
//     complete, and store through a per-warp staging tile: SwiGLU forms
//     h = silu(g) * u in fp32 -> bf16 and stores 32-byte row segments of h; the
//     fp32 epilogue stores 128-byte row segments of Y.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"
#include "tc_gemm.cuh"

namespace invmoe {

// TMA load of rank 5 into this CTA's shared memory, completion counted on an
// mbarrier that may live in the peer CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_5d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster_addr, int c0,
                                                 int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

// Arrive on an mbarrier of the pair (possibly the peer CTA's) with CTA-scope release: for an
// epilogue warp that frees TMEM columns.  The arrive follows tcgen05.wait::ld, so the columns' loads
// are complete; it hands over no global or shared data, and a cluster-scope release would first wait
// for the warp's earlier global stores to become visible cluster-wide (same-box A/B: fp32 down
// projection in token columns 153 -> 141 us on the Qwen-like layer, GLM-scale -1 %).
__device__ __forceinline__ void mbar_arrive_remote_cta(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

constexpr int kTokChunk = 320;     // most tokens (TMEM columns) of one unit
constexpr int kTokBoxRows = 32;    // token rows per TMA box: 32, 64 or 128 (a CTA's share of one MMA) ...
constexpr int kTokMidRows = 64;
constexpr int kTokBigRows = 128;
constexpr int kTokTwoRows = 160;   // ... or 160 (its share of both MMAs of a chunk of more than 256 tokens)

// CHUNK: most tokens of one unit.  kTokChunk for prefill-sized batches; 64 for batches of at most
// 1024 token slots or 16 per expert (decode) and 128 for at most 64 per expert, where a CTA's
// token tile is one 32- or 64-row box and the stages are small enough for a deeper ring.
template <int EPI, int STAGES, int CHUNK = kTokChunk>
struct TokShape {
  static_assert(CHUNK == kTokChunk || CHUNK == 64 || CHUNK == 128, "unit size");
  static constexpr int A_BYTES = kBM * kBK * 2;                   // 16 KB: 128 weight rows x 64 K
  // token rows per CTA: MMA 1 (half of up to 256) + MMA 2 (half of up to 64), or half of the unit
  static constexpr int B_ROWS = CHUNK == kTokChunk ? 128 + 32 : CHUNK / 2;
  static constexpr int B_BYTES = B_ROWS * kBK * 2;                // 20 KB (4 or 8 KB)
  // 64-wide K blocks per ring stage: two for the 64-token units and the 128-token SwiGLU units
  // (measured faster there; one stage then holds both blocks' weights and tokens, one after the other)
  static constexpr int KSUB = (CHUNK == 64 || (CHUNK == 128 && EPI == EPI_SWIGLU)) ? 2 : 1;
  static constexpr int SUB_BYTES = A_BYTES + B_BYTES;             // 36 KB (20 or 24 KB; 1 KB multiples)
  static constexpr int STAGE_BYTES = KSUB * SUB_BYTES;
  static constexpr int TMEM_COLS = 512;
  static constexpr int EPI_WARPS = 8;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int THREADS = 64 + EPI_THREADS;
  static constexpr int QDEPTH = 4;
  // a sixth 36 KB stage for the 320-token units fits once the chunk table holds at most 256 experts
  // and each epilogue warp's staging tile is the 1,056 bytes the SwiGLU store uses
  // (SwiGLU), or 1 KB for the fp32 store in passes of 8 tokens (16 otherwise)
  static constexpr bool DEEP = CHUNK == kTokChunk && STAGES >= 6;
  static constexpr int MAX_GROUPS = DEEP ? 256 : 1024;
  static constexpr int OST_WARP = DEEP ? (EPI == EPI_SWIGLU ? 1088 : 1024) : 2048;   // a warp's staging tile
  static constexpr int OSTAGE_BYTES = EPI_WARPS * OST_WARP;
  static constexpr int BAR_BYTES = 8 * (2 * STAGES + 6 + 1 + 2 * QDEPTH);
  static constexpr int MISC_BYTES = 16 + 4 * QDEPTH;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + OSTAGE_BYTES + BAR_BYTES + MISC_BYTES +
                                    4 * (MAX_GROUPS + 1);
  static_assert(STAGE_BYTES % 1024 == 0, "stage alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
  static_assert(EPI == EPI_SWIGLU || EPI == EPI_F32, "epilogue");
};

struct TokUnit {
  int g;      // group (expert)
  int wb;     // weight block
  int tok0;   // first token row of the chunk (row of X and of the output)
  int nv;     // tokens in the chunk (1 .. CHUNK)
};

// Chunks of group g: ceil(n / CHUNK), near-equal sizes (the kernel's prefix holds the counts).  Units are ordered
// group by group, chunk-major inside a group, so consecutive units share the
// chunk's token rows in L2.
__device__ __forceinline__ TokUnit decode_tok_unit(int u, const GemmParams& p, const int* s_prefix) {
  const int NB = p.n_blocks;
  int lo = 0, hi = p.G;  // NB*s_prefix[lo] <= u < NB*s_prefix[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (NB * s_prefix[mid] <= u) lo = mid; else hi = mid;
  }
  TokUnit U;
  U.g = lo;
  const int nch = s_prefix[lo + 1] - s_prefix[lo];
  const int local = u - NB * s_prefix[lo];
  const int c = local / NB;
  U.wb = local - c * NB;
  const int n = __ldg(p.counts + lo);
  const int s0 = static_cast<int>(static_cast<long long>(n) * c / nch);
  const int s1 = static_cast<int>(static_cast<long long>(n) * (c + 1) / nch);
  U.tok0 = __ldg(p.offsets + lo) + s0;
  U.nv = s1 - s0;
  return U;
}

// TMEM placement of a unit in column slot `slot` (0 or 1; consecutive units of a
// CTA alternate): MMA 1 (tokens [0, 256)) and MMA 2 (tokens [256, kTokChunk)).
__device__ __forceinline__ uint32_t tok_col1(int slot) { return slot ? 256u : 0u; }
__device__ __forceinline__ uint32_t tok_col2(int slot) { return slot ? 192u : 256u; }
// TMEM column of the 32-token chunk c (tokens [32c, 32c + 32) of the unit)
__device__ __forceinline__ uint32_t tok_chunk_col(int slot, int c) {
  return c < 8 ? tok_col1(slot) + 32u * c : tok_col2(slot) + 32u * (c - 8);
}
// The epilogue drains a unit's nchunk chunks in two phases: phase 0 the chunks
// whose columns lie in [192, 320) (the only columns the next unit, in the other
// slot, may write), phase 1 the rest.  Length of a phase and its k-th chunk:
__device__ __forceinline__ int tok_phase_len(int slot, int ph, int nchunk) {
  if (slot == 0) return ph == 0 ? max(0, nchunk - 6) : min(nchunk, 6);
  return ph == 0 ? min(nchunk, 2) + max(0, nchunk - 8) : max(0, min(nchunk, 8) - 2);
}
__device__ __forceinline__ int tok_phase_chunk(int slot, int ph, int nchunk, int k) {
  if (slot == 0) return ph == 0 ? 6 + k : k;
  if (ph == 1) return 2 + k;
  const int a = min(nchunk, 2);
  return k < a ? k : 8 + (k - a);
}

template <int EPI, int STAGES, int CHUNK>
__global__ void __launch_bounds__(TokShape<EPI, STAGES, CHUNK>::THREADS, 1)
    tc_gemm_tok_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmXm, const __grid_constant__ CUtensorMap tmXb,
                       const __grid_constant__ CUtensorMap tmXt, const GemmParams p) {
  using S = TokShape<EPI, STAGES, CHUNK>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* ostage = smem + STAGES * S::STAGE_BYTES;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(ostage + S::OSTAGE_BYTES);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* accf_bar = empty_bar + STAGES;           // [2] per column slot: the unit's MMAs are done
  uint64_t* accmid_bar = accf_bar + 2;               // [2] columns [192, 320) of the slot drained
  uint64_t* accall_bar = accmid_bar + 2;             // [2] every column of the slot drained
  uint64_t* final_bar = accall_bar + 2;
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
    for (int x = 0; x < 2; ++x) {
      mbar_init(&accf_bar[x], 1);
      mbar_init(&accmid_bar[x], 2 * S::EPI_WARPS);    // one arrive per epilogue warp of each CTA
      mbar_init(&accall_bar[x], 2 * S::EPI_WARPS);
    }
    mbar_init(final_bar, 1);
    for (int qq = 0; qq < S::QDEPTH; ++qq) {
      mbar_init(&qfull_bar[qq], 1);
      // consumers of a queue slot: per CTA its epilogue warps, plus the
      // leader's MMA thread and the follower's producer thread
      mbar_init(&qempty_bar[qq], 2 + 2 * S::EPI_WARPS);
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    if (CHUNK >= 128) tma_prefetch_desc(&tmXm);
    if (CHUNK == kTokChunk) {
      tma_prefetch_desc(&tmXb);
      tma_prefetch_desc(&tmXt);
    }
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, S::TMEM_COLS);
  // everything above touches only shared memory, TMEM and the kernel parameters; the
  // previous kernel on the stream (which wrote this kernel's inputs) is waited for here
  pdl_wait();
  pdl_trigger();

  // chunk prefix over groups (warp 2; G <= 1024): s_prefix[g] = sum_{g'<g} ceil(counts[g'] / CHUNK)
  if (warp == 2) {
    const int per = (p.G + 31) / 32;
    const int g0 = lane * per;
    int local = 0;
    for (int i = 0; i < per; ++i) {
      const int g = g0 + i;
      if (g < p.G) local += (__ldg(p.counts + g) + CHUNK - 1) / CHUNK;
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
        run += (__ldg(p.counts + g) + CHUNK - 1) / CHUNK;
      }
    }
    if (lane == 31) {
      s_prefix[p.G] = incl;
      *s_total = incl;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();     // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int total_units = *s_total * p.n_blocks;
  const int num_kb = (p.K + kBK - 1) / kBK;                      // 64-wide K blocks
  const int num_st = (num_kb + S::KSUB - 1) / S::KSUB;             // ring stages per unit
  WaitCtl wc{s_abort, p.status, p.timeout_ns};
  const uint32_t peer_abort = mapa_shared(smem_u32(const_cast<int*>(s_abort)), peer);
  const uint32_t qempty_leader0 = mapa_shared(smem_u32(&qempty_bar[0]), 0);

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
      // the leader's first unit is its pair index; later ones come from the counter, offset past those
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
        const TokUnit U = decode_tok_unit(u, p, s_prefix);
        const int nmma = (U.nv + 15) & ~15;
        const int n1 = nmma < 256 ? nmma : 256;
        const int r1 = n1 / 2, r2 = (nmma - n1) / 2;
        // this CTA's token rows, one box: its share of MMA 1 alone in the smallest box that
        // holds it, or its shares of both MMAs in one 160-row box (CTA 0 tokens [0, 128 + r2),
        // CTA 1 the next 128 + r2)
        int box_rows = kTokBoxRows;
        const CUtensorMap* tmT = &tmX;
        if (CHUNK == kTokChunk) {
          if (r2 > 0) { box_rows = kTokTwoRows; tmT = &tmXt; }
          else if (r1 > kTokMidRows) { box_rows = kTokBigRows; tmT = &tmXb; }
          else if (r1 > kTokBoxRows) { box_rows = kTokMidRows; tmT = &tmXm; }
        } else if (CHUNK == 128 && r1 > kTokBoxRows) {
          box_rows = kTokMidRows;
          tmT = &tmXm;
        }
        const uint32_t bytes = S::A_BYTES + box_rows * (kBK * 2);
        // this CTA's weight rows: SwiGLU h columns [f0, f0 + 64), f0 = 128 wb + 64r (gate rows f0.., up
        // rows F + f0..); fp32 rows [256 wb + 128r, +128)
        const int f0 = U.wb * 128 + 64 * static_cast<int>(rank);
        const int wrow = U.g * p.b_group_rows + U.wb * 256 + 128 * static_cast<int>(rank);
        const int t1 = U.tok0 + static_cast<int>(rank) * (r1 + r2);
        for (int ks = 0; ks < num_st; ++ks) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, wc)) { ok = false; break; }
          uint8_t* st = ring + stage * S::STAGE_BYTES;
          const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
          const int nsub = min(S::KSUB, num_kb - ks * S::KSUB);    // K blocks in this stage
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], 2 * nsub * bytes);
          for (int j = 0; j < nsub; ++j) {
            uint8_t* sj = st + j * S::SUB_BYTES;
            const int kx = (ks * S::KSUB + j) * kBK;
            if (EPI == EPI_SWIGLU) {
              // one box of 4 row groups x (16 gate rows, the matching 16 up rows): tile rows
              // 32i + [0, 16) are gate rows f0 + 16i + [0, 16), 32i + [16, 32) the up rows
              tma_load_5d_pair(sj, &tmW, fb, kx, 0, 0, f0 / 16, U.g);
            } else {
              tma_load_2d_pair(sj, &tmW, fb, kx, wrow);
            }
            tma_load_2d_pair(sj + S::A_BYTES, tmT, fb, kx, t1);
          }
          filled_phase[stage] = static_cast<int>(phase);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) st_shared_remote_u32(peer_abort, 1u);
      // this CTA takes no more units: once every CTA is past this point the counter is reset
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
      const uint64_t adesc0 = sdesc_k_sw128(smem_u32(ring));
      const uint64_t bdesc0 = sdesc_k_sw128(smem_u32(ring + S::A_BYTES));
      constexpr uint64_t B2_OFF = (128 * kBK * 2) >> 4;      // MMA 2's token rows start at row 128
      int stage = 0;
      uint32_t phase = 0;
      uint32_t nunit = 0;        // units this pair has run: column slot nunit & 1
      int prev_n2 = 0;           // width of the previous unit's second MMA (0: none)
      bool ok = true;
      int qi = 0;
      uint32_t qphase = 0;
      while (ok) {
        if (!mbar_wait(&qfull_bar[qi], qphase, wc)) { ok = false; break; }
        const int u = s_queue[qi];
        mbar_arrive(&qempty_bar[qi]);
        if (++qi == S::QDEPTH) { qi = 0; qphase ^= 1u; }
        if (u < 0) break;
        const TokUnit U = decode_tok_unit(u, p, s_prefix);
        const int nmma = (U.nv + 15) & ~15;
        const int n1 = nmma < 256 ? nmma : 256;
        const int n2 = nmma - n1;
        const uint32_t idesc1 = idesc_bf16_f32(2 * kBM, n1);
        const uint32_t idesc2 = idesc_bf16_f32(2 * kBM, n2 > 0 ? n2 : 16);
        const int slot = static_cast<int>(nunit & 1u);
        // the slot's previous unit fully drained; the previous unit (other slot) drained its
        // columns in [192, 320), the only ones the two slots share.  When neither unit has a
        // second MMA, the previous one's columns (all its chunks, read in either phase) and this
        // one's are disjoint ([0, 256) and [256, 512)), and the MMAs start at once.
        if (!mbar_wait<true>(&accall_bar[slot], ((nunit >> 1) & 1u) ^ 1u, wc)) { ok = false; break; }
        if (nunit > 0 && (n2 > 0 || prev_n2 > 0) &&
            !mbar_wait<true>(&accmid_bar[slot ^ 1], ((nunit - 1) >> 1) & 1u, wc)) {
          ok = false;
          break;
        }
        prev_n2 = n2;
        tc_fence_after();
        const uint32_t d1 = tmem_base + tok_col1(slot);
        const uint32_t d2 = tmem_base + tok_col2(slot);
        for (int ks = 0; ks < num_st; ++ks) {
          if (!mbar_wait(&full_bar[stage], phase, wc)) { ok = false; break; }
          tc_fence_after();
          const int nsub = min(S::KSUB, num_kb - ks * S::KSUB);
          for (int j = 0; j < nsub; ++j) {
            const int kb = ks * S::KSUB + j;         // K blocks in ascending order, as one chain
            const uint64_t so = static_cast<uint64_t>((stage * S::STAGE_BYTES + j * S::SUB_BYTES) >> 4);
            const uint64_t adesc = adesc0 + so;
            const uint64_t bdesc = bdesc0 + so;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_bf16_pair(d1, adesc + 2u * kk, bdesc + 2u * kk, idesc1, (kb | kk) != 0 ? 1u : 0u);
            if (n2 > 0) {
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk)
                umma_bf16_pair(d2, adesc + 2u * kk, bdesc + B2_OFF + 2u * kk, idesc2, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit_pair(&empty_bar[stage], 0x3);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair(&accf_bar[slot], 0x3);
        ++nunit;
      }
      if (!ok) st_shared_remote_u32(peer_abort, 1u);
      umma_commit_pair(final_bar, 0x1);
      WaitCtl drain{nullptr, p.status, p.timeout_ns};
      mbar_wait(final_bar, 0, drain);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int ew = warp - 2;
    const int q = warp & 3;                 // TMEM lane quadrant this warp may access
    const int half = ew >> 2;               // every other chunk of each phase, starting at `half`
    const uint32_t accmid_leader0 = mapa_shared(smem_u32(accmid_bar), 0);
    const uint32_t accall_leader0 = mapa_shared(smem_u32(accall_bar), 0);
    uint8_t* stg = ostage + ew * S::OST_WARP;
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    uint32_t nunit = 0;
    int qi = 0;
    uint32_t qphase = 0;
    while (true) {
      const bool okq = mbar_wait<true>(&qfull_bar[qi], qphase, wc);
      if (!__all_sync(0xffffffffu, okq)) break;
      const int u = s_queue[qi];
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(qempty_leader0 + 8u * qi);
      if (++qi == S::QDEPTH) { qi = 0; qphase ^= 1u; }
      if (u < 0) break;
      const TokUnit U = decode_tok_unit(u, p, s_prefix);
      const int slot = static_cast<int>(nunit & 1u);
      const bool ok = mbar_wait(&accf_bar[slot], (nunit >> 1) & 1u, wc);
      if (!__all_sync(0xffffffffu, ok)) break;
      ++nunit;
      tc_fence_after();
      const int nchunk = (U.nv + 31) / 32;
      // half of the second MMA's width (0: none); the token of row r of chunk c (columns
      // 32c + r of MMA 1 for c < 8, 32(c - 8) + r of MMA 2 after; the loader's split above)
      const int h2 = max(0, ((U.nv + 15) & ~15) - 256) / 2;
      auto tok_of = [&](int c, int r) -> int {
        const int j = 32 * (c & 7) + r;
        if (h2 == 0) return 32 * c + r;
        if (c < 8) return j < 128 ? j : j + h2;
        return j < h2 ? 128 + j : 256 + j;
      };

      // one 32-token chunk c held in v (this thread's lane, 32 consecutive columns)
      auto store_chunk = [&](int c, const uint32_t (&v)[32]) {
        if (EPI == EPI_SWIGLU) {
          // lanes 0-15 hold gate rows, lanes 16-31 the matching up rows of h columns
          // [fq, fq + 16): a lane computes h for its column and 16 of the 32 tokens
          // (lanes 0-15 tokens 0-15, lanes 16-31 tokens 16-31) after one exchange
          const int fq = U.wb * 128 + 64 * static_cast<int>(rank) + 16 * q;
          const bool upper = lane >= 16;
          const int tb = upper ? 16 : 0;
          __nv_bfloat16* hs = reinterpret_cast<__nv_bfloat16*>(stg);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const uint32_t send = upper ? v[j] : v[16 + j];
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 16);
            const float g = __uint_as_float(upper ? recv : v[j]);
            const float uu = __uint_as_float(upper ? v[16 + j] : recv);
            // staging row r (token) at byte 32r, rows 16-31 one row further on (no bank conflict)
            hs[(tb + j) * 16 + tb + (lane & 15)] = __float2bfloat16_rn(__fmul_rn(silu_f32(g), uu));
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int m = lane + 32 * i;
            const int r = m >> 1;
            const uint4 w = *reinterpret_cast<const uint4*>(stg + r * 32 + (r >= 16 ? 32 : 0) + (m & 1) * 16);
            const int t = tok_of(c, r);
            if (t < U.nv)
              *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                        static_cast<long long>(U.tok0 + t) * p.ldo + fq + (m & 1) * 8) = w;
          }
          __syncwarp();
        } else {
          // fp32 Y[token, h0 + lane] for the warp's 32 rows of this CTA's 128 weight rows
          const int h0 = U.wb * 256 + 128 * static_cast<int>(rank) + 32 * q;
          float* ys = reinterpret_cast<float*>(stg);
          constexpr int TPP = S::OST_WARP / 128;    // tokens per staging pass (128 B of Y per token)
#pragma unroll
          for (int hh = 0; hh < 32 / TPP; ++hh) {
#pragma unroll
            for (int j = 0; j < TPP; ++j) ys[j * 32 + lane] = __uint_as_float(v[TPP * hh + j]);
            __syncwarp();
            const int ch = lane & 7;
#pragma unroll
            for (int i = 0; i < TPP / 4; ++i) {
              const int r = 4 * i + (lane >> 3);
              const uint4 w = *reinterpret_cast<const uint4*>(stg + r * 128 + ch * 16);
              const int t = tok_of(c, TPP * hh + r);
              if (t < U.nv)
                *reinterpret_cast<uint4*>(static_cast<float*>(p.out) +
                                          static_cast<long long>(U.tok0 + t) * p.ldo + h0 + ch * 4) = w;
            }
            __syncwarp();
          }
        }
      };

      // A warp releases a phase's columns (one arrive per warp on the leader: phase 0 lets the
      // next unit, in the other slot, write columns [192, 320); phase 1 frees the slot) as soon
      // as its last TMEM loads of the phase have completed, before it forms and stores them.
      const uint32_t rel0 = accmid_leader0 + 8u * slot;
      const uint32_t rel1 = accall_leader0 + 8u * slot;
      auto release = [&](uint32_t bar) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_cta(bar);
      };
#pragma unroll 1
      for (int ph = 0; ph < 2; ++ph) {
        const int len = tok_phase_len(slot, ph, nchunk);
        const uint32_t rel = ph == 0 ? rel0 : rel1;
        if (half >= len) release(rel);
        // two chunks per TMEM round trip: k and k + 2 (the second load repeats the first
        // when k + 2 is past the phase, and is not stored)
#pragma unroll 1
        for (int k = half; k < len; k += 4) {
          const int ca = tok_phase_chunk(slot, ph, nchunk, k);
          const bool two = k + 2 < len;
          const int cb = two ? tok_phase_chunk(slot, ph, nchunk, k + 2) : ca;
          uint32_t va[32], vb[32];
          tmem_ld32(tbase + tok_chunk_col(slot, ca), va);
          tmem_ld32(tbase + tok_chunk_col(slot, cb), vb);
          tmem_ld_wait();
          tmem_reg_fence(va);
          tmem_reg_fence(vb);
          if (k + 4 >= len) release(rel);
          store_chunk(ca, va);
          if (two) store_chunk(cb, vb);
        }
      }
    }
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
