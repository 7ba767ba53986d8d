// tc_gemm.cuh -- the fixed-tile tcgen05 GEMM engine (sm_103a).
//
//   D[r, n] = sum_k A[r, k] * B[n, k]      A, B bf16, D accumulated in fp32 TMEM
//
// Operands are K-major ([rows, K]) unless a template flag makes one MN-major
// ([K, rows]; see tc_gemm2.cuh for the layout).
//
// Batch invariance ("位级一致：前沿训练的差异化关键", section
// "为什么比特级一致是一个复杂的问题": one fixed kernel choice for the expert
// matmuls whatever the per-expert token count; DeepGEMM dropped split-K because
// it breaks invariance):
//   * one tile shape per call site (BM = 128 rows, BN columns, BK = 64), chosen
//     from the model shape only, never from T or from a group's row count;
//   * every output element is produced by exactly one CTA that walks K from 0
//     upward in 64-wide blocks, each block as four K=16 MMAs in ascending order,
//     accumulating in TMEM; no split-K, no stream-K;
//   * which CTA handles which tile (the persistent schedule) varies freely: it
//     never changes the order of any element's reduction;
//   * rows of a tile that belong to another group, or lie past the end of A,
//     are loaded (TMA fills out-of-range rows with zeros) and multiplied, but
//     never stored: an MMA row depends only on its own A row;
//   * a tile with at most 64 valid rows is issued as an M = 64 MMA: its rows get
//     the same products in the same order (bit-identical to the M = 128 tile).
//
// Grouped mode: groups g = 0..G-1 own the A rows [offsets[g], offsets[g]+counts[g])
// and the B rows [g*b_group_rows, (g+1)*b_group_rows).  A group's rows are cut
// into chunks of MT*128 rows; a work unit is (chunk, column block).  Each unit
// streams its B tile once per K block and multiplies it against up to MT row
// tiles, so an expert with at most MT*128 tokens reads its weights once.
//
// K-grouped mode (weight gradients, dW_g = A_g^T B_g): group g owns the rows
// [offsets[g], offsets[g]+counts[g]) of two MN-major operands A [rows, M] and
// B [rows, N]; the reduction runs over the group's rows only.  The block of 64
// rows that crosses the group's end issues its K = 16 steps only up to the one
// holding the group's last row (the steps after it would add exact zeros), and
// that step's rows past the end are zeroed in shared memory before its MMAs, so
// the next group's rows are never multiplied in.  A group with no rows gets an
// all-zero block.  Output rows g*M .. g*M+M-1, written by bulk tensor stores
// through a [G][M][N] map that clips rows past M and columns past N.
//
// Warp roles (320 threads, one CTA per SM, persistent over units):
//   warp 0      scheduler + TMA producer (one lane): takes a unit index from a
//               global counter, publishes it to the other roles through a small
//               shared queue, and loads the A row tiles + B tile of each K block
//               into a STAGES-deep shared-memory ring (128-byte swizzle)
//   warp 1      TMEM owner + MMA issuer (one lane; the whole warp in K-grouped
//               mode, to zero the rows past a group's end): tcgen05.mma
//               kind::f16, commit frees a ring slot / publishes an accumulator
//   warps 2..9  epilogue (two warps per TMEM lane quadrant): tcgen05.ld 32 lanes
//               x 32 columns at a time, convert, stage through shared memory and
//               store (fp32 rows, SwiGLU -> bf16 h, or the SwiGLU backward)
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace invmoe {

constexpr int kBM = 128;
constexpr int kBK = 64;

enum Epilogue : int { EPI_F32 = 0, EPI_SWIGLU = 1, EPI_LSE = 2, EPI_DLOGITS = 3, EPI_SWIGLU_BWD = 4 };

struct GemmParams {
  int K;                  // reduction length (multiple of 64)
  int N;                  // valid output columns (F32: of D; SwiGLU: of h)
  int n_blocks;           // column blocks per row chunk
  int M;                  // dense mode: rows of A and D
  int G;                  // groups (0 = dense)
  const int* counts;      // [G] rows per group (device)
  const int* offsets;     // [G+1] first A row per group (device)
  int b_group_rows;       // B rows per group
  int b_up_rows;          // SwiGLU: offset of the up-projection rows inside a group
  int n_major;            // 1: consecutive units walk row chunks of one column block
  void* out;              // D (fp32) or h (bf16)
  long long ldo;          // output row stride, elements
  unsigned int* status;   // status word (bit 0: a bounded wait ran out)
  int* sched;             // unit counter for the dynamic schedule (zero before launch)
  unsigned long long timeout_ns;
  // EPI_LSE only: per (row, column block) log-sum-exp partials and the target logit
  float2* part;           // (max, sum exp(z - max)) of column block nb of `row` at part[row * nch + nb]
  int nch;                // row stride of part in pairs (ceil(N / 256) unless the caller sets one)
  int col0;               // column index of B's first row in the whole vocabulary (vocabulary shards)
  const int* target;      // [rows] target column of each row (in the whole vocabulary)
  float* tgt_logit;       // [rows] z[row, target[row]] (written by the block holding it)
  int m_group;            // dense column-block-major order: row chunks per band (>= 1)
  // EPI_DLOGITS only (target as above): out = bf16 g[row] * (onehot - exp(z - lse[row]))
  const float* row_lse;   // [rows] log-sum-exp of each row of Z
  const float* row_scale; // [rows] upstream gradient g of each row's logprob
  // EPI_SWIGLU_BWD only: out = [dg | du] bf16 (ldo = 2N), out2 = h bf16 (ldo2, nullable),
  // aux = dh fp32 (ld_aux); N = columns of h
  const float* aux;
  long long ld_aux;
  void* out2;
  long long ldo2;
  int kgroup;             // 1: K-grouped mode (weight gradients); M = output rows per group
  int out_map;            // fp32 D: 1 if the output store map was built (bulk tensor stores)
};

// Epilogue stores.  After tcgen05.ld.32x32b each lane of a warp holds one row
// of the tile (lane = row), so a direct store from registers writes 32 rows x
// 16 bytes per instruction.  Instead each warp writes a 32-row x 64-byte
// segment into its own 2 KB of shared memory and stores it back out with four
// lanes per row: 8 rows x 64 contiguous bytes per instruction.  The 16-byte
// chunk q of row r sits at r*64 + (q ^ ((r >> 1) & 3))*16, so both the
// row-wise writes and the chunk-wise reads are free of bank conflicts.
constexpr int kOutStageBytes = 32 * 64;

// The reverse of stage_store_rows64: the warp reads a 32-row x 64-byte segment
// with four lanes per row (rows past rows_valid and bytes past bytes_valid read
// as zero) and each lane gets its own row's 16 words.
__device__ __forceinline__ void stage_load_rows64(uint8_t* stage, const uint8_t* in_row0, long long ld_bytes,
                                                  int rows_valid, int bytes_valid, uint32_t (&v)[16]) {
  const int lane = threadIdx.x & 31;
  const int q = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2);
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (r < rows_valid && q * 16 < bytes_valid) w = __ldg(reinterpret_cast<const uint4*>(in_row0 + r * ld_bytes + q * 16));
    *reinterpret_cast<uint4*>(stage + r * 64 + ((q ^ ((r >> 1) & 3)) << 4)) = w;
  }
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 w = *reinterpret_cast<const uint4*>(stage + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4));
    v[4 * c] = w.x; v[4 * c + 1] = w.y; v[4 * c + 2] = w.z; v[4 * c + 3] = w.w;
  }
  __syncwarp();
}

__device__ __forceinline__ void stage_store_rows64(uint8_t* stage, const uint32_t (&v)[16], uint8_t* out_row0,
                                                   long long ld_bytes, int rows_valid, int bytes_valid) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(stage + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)) =
        make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  __syncwarp();
  const int q = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2);
    const uint4 w = *reinterpret_cast<const uint4*>(stage + r * 64 + ((q ^ ((r >> 1) & 3)) << 4));
    if (r < rows_valid && q * 16 < bytes_valid)
      *reinterpret_cast<uint4*>(out_row0 + r * ld_bytes + q * 16) = w;
  }
  __syncwarp();
}

template <int BN, int MT, int EPI, int STAGES>
struct GemmShape {
  static constexpr int A_BYTES = kBM * kBK * 2;                 // 16 KB per 128-row tile
  static constexpr int B_BYTES = BN * kBK * 2;
  static constexpr int STAGE_BYTES = MT * A_BYTES + B_BYTES;    // one ring stage: A row tiles + B tile
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int ACC_COLS = MT * BN;                      // fp32 TMEM columns per accumulator
  static constexpr int ACC_STAGES = (2 * ACC_COLS <= 512) ? 2 : 1;
  static constexpr int TMEM_NEED = ACC_STAGES * ACC_COLS;
  static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128
                                   : TMEM_NEED <= 256 ? 256 : 512;
  static constexpr int EPI_WARPS = 8;                           // two warps per TMEM lane quadrant
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int THREADS = 64 + EPI_THREADS;
  static constexpr int QDEPTH = 4;                              // scheduled-unit queue depth
  static constexpr int MAX_GROUPS = 1024;
  static constexpr int BAR_BYTES = 8 * (2 * STAGES + 2 * ACC_STAGES + 1 + 2 * QDEPTH);
  static constexpr int MISC_BYTES = 16 + 4 * QDEPTH;
  static constexpr int OSTAGE_BYTES = EPI_WARPS * kOutStageBytes;   // epilogue store staging
  static constexpr int SMEM_BYTES = 1024 /* alignment slack */ + RING_BYTES + OSTAGE_BYTES + BAR_BYTES +
                                    MISC_BYTES + 4 * (MAX_GROUPS + 1);
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert(EPI != EPI_LSE && EPI != EPI_DLOGITS, "the LSE and dlogits epilogues run on the CTA-pair engine");
  static_assert(TMEM_NEED <= 512, "TMEM");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct Unit {
  int row0;    // first D row of the chunk (and first A row, except in K-grouped mode)
  int rows;    // valid rows in the chunk (1 .. MT*128)
  int b_row;   // first B row of the column block (gate rows for SwiGLU), K-major B
  int nb;      // column block
  int g;       // group
  int a_m0;    // K-grouped: first M index of the chunk (A is MN-major)
  int k0;      // K-grouped: first K row of the group
  int kcount;  // K-grouped: K rows of the group
};

// Unit order.  Grouped: group by group; inside a group column-block-major, so
// all row chunks of one (group, column block) are consecutive units and share
// the weight tile while it is in L2.  Dense: row-chunk-major, or column-block-
// major when n_major (consecutive units then share a weight tile).
template <int MT, int EPI, int BN>
__device__ __forceinline__ Unit decode_unit(int u, const GemmParams& p, const int* s_prefix, int total_chunks) {
  constexpr int CH = MT * kBM;
  Unit U;
  int g = 0, nb;
  U.a_m0 = 0;
  U.k0 = 0;
  U.kcount = p.K;
  if (p.kgroup) {
    // group-major, then M chunk, then column block
    const int mch = (p.M + CH - 1) / CH;
    g = u / (mch * p.n_blocks);
    const int local = u - g * mch * p.n_blocks;
    const int c = local / p.n_blocks;
    nb = local - c * p.n_blocks;
    U.a_m0 = c * CH;
    U.row0 = g * p.M + c * CH;
    U.rows = min(CH, p.M - c * CH);
    U.k0 = __ldg(p.offsets + g);
    U.kcount = __ldg(p.counts + g);
  } else if (p.G > 0) {
    const int NB = p.n_blocks;
    int lo = 0, hi = p.G;  // NB*s_prefix[lo] <= u < NB*s_prefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (NB * s_prefix[mid] <= u) lo = mid; else hi = mid;
    }
    g = lo;
    const int nch = s_prefix[g + 1] - s_prefix[g];
    const int local = u - NB * s_prefix[g];
    nb = local / nch;
    const int c = local - nb * nch;
    U.row0 = __ldg(p.offsets + g) + c * CH;
    U.rows = min(CH, __ldg(p.counts + g) - c * CH);
  } else {
    int chunk;
    if (p.n_major) {
      // bands of m_group row chunks; inside a band column-block-major, so the
      // band's A rows stay in L2 while every B tile streams past them once
      const int gm = min(max(p.m_group, 1), total_chunks);
      const int band = u / (gm * p.n_blocks);
      const int c0 = band * gm;
      const int gsize = min(gm, total_chunks - c0);
      const int local = u - band * gm * p.n_blocks;
      nb = local / gsize;
      chunk = c0 + (local - nb * gsize);
    } else {
      chunk = u / p.n_blocks;
      nb = u - chunk * p.n_blocks;
    }
    U.row0 = chunk * CH;
    U.rows = min(CH, p.M - U.row0);
  }
  constexpr int NB_ROWS = (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD) ? BN / 2 : BN;
  U.b_row = g * p.b_group_rows + nb * NB_ROWS;
  U.nb = nb;
  U.g = g;
  return U;
}

__device__ __forceinline__ float silu_f32(float g) {
  // silu(g) = g / (1 + exp(-g)), IEEE division
  return g / (1.0f + expf(-g));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// SwiGLU backward for one 32-column chunk of a warp's 32 rows (lane = row):
//   s = 1 / (1 + exp(-g)),  silu = g / (1 + exp(-g)) (the forward's own expression),
//   h = silu * u (bit-identical to the forward's h),
//   dg = (dh * u) * (s * (1 + g * (1 - s))),  du = dh * silu,
// every operation rounded separately in fp32; dg, du and h are stored as bf16.
// dh (fp32, 128 B per row) is read through the warp's staging buffer.
__device__ __forceinline__ void swiglu_bwd_chunk(uint8_t* stg, const uint32_t (&gv)[32], const uint32_t (&uv)[32],
                                                 const uint8_t* dh_row0, long long ld_dh_bytes, uint8_t* dg_row0,
                                                 uint8_t* du_row0, long long ld_dgu_bytes, uint8_t* h_row0,
                                                 long long ld_h_bytes, int rows_valid, int cols_valid) {
  uint32_t d0[16], d1[16];
  stage_load_rows64(stg, dh_row0, ld_dh_bytes, rows_valid, cols_valid * 4, d0);
  stage_load_rows64(stg, dh_row0 + 64, ld_dh_bytes, rows_valid, cols_valid * 4 - 64, d1);
  uint32_t pg[16], pu[16], ph[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float dgv[2], duv[2], hv[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = 2 * j + e;
      const float g = __uint_as_float(gv[col]);
      const float u = __uint_as_float(uv[col]);
      const float d = __uint_as_float(col < 16 ? d0[col & 15] : d1[col & 15]);
      const float si = silu_f32(g);
      const float sg = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-g)));
      const float ds = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, sg))));
      dgv[e] = __fmul_rn(__fmul_rn(d, u), ds);
      duv[e] = __fmul_rn(d, si);
      hv[e] = __fmul_rn(si, u);
    }
    pg[j] = pack_bf16x2(dgv[0], dgv[1]);
    pu[j] = pack_bf16x2(duv[0], duv[1]);
    ph[j] = pack_bf16x2(hv[0], hv[1]);
  }
  stage_store_rows64(stg, pg, dg_row0, ld_dgu_bytes, rows_valid, cols_valid * 2);
  stage_store_rows64(stg, pu, du_row0, ld_dgu_bytes, rows_valid, cols_valid * 2);
  if (h_row0 != nullptr) stage_store_rows64(stg, ph, h_row0, ld_h_bytes, rows_valid, cols_valid * 2);
}

// Zero K rows [rem, end) of `nbox` consecutive MN-major boxes (64 K rows x 128 B
// each) at `base`: the rows of a K-grouped block's last K = 16 step that lie past
// its group's last row (end - rem < 16; whole rows, so the swizzle does not
// matter).  All 32 lanes of the calling warp take part.
__device__ __forceinline__ void zero_k_tail(uint8_t* base, int nbox, int rem, int end) {
  const int lane = threadIdx.x & 31;
  const int per_box = (end - rem) * 8;          // 16-byte chunks per box
  uint8_t* p0 = base + rem * 128;
  for (int b = 0; b < nbox; ++b)
    for (int c = lane; c < per_box; c += 32)
      *reinterpret_cast<uint4*>(p0 + b * kMnBoxBytes + c * 16) = make_uint4(0u, 0u, 0u, 0u);
}

// Work units are handed out dynamically: the producer thread takes the next
// unit index from a global counter and publishes it through a small shared
// queue to the MMA thread and the epilogue warps.  Which CTA computes which
// tile therefore varies from run to run; the arithmetic of every tile does not.
// A_MN / B_MN: operand stored MN-major (see tc_gemm2.cuh).  In this engine an
// MN-major A occurs only in K-grouped mode (KG); an MN-major B with M-grouped
// rows takes group g's B from the stored rows [g*b_group_rows, +K).
template <int BN, int MT, int EPI, int STAGES, bool A_MN = false, bool B_MN = false, bool KG = false>
__global__ void __launch_bounds__(GemmShape<BN, MT, EPI, STAGES>::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmO, const GemmParams p) {
  using S = GemmShape<BN, MT, EPI, STAGES>;
  static_assert(A_MN == KG, "an MN-major A only in K-grouped mode, and K-grouped mode needs it");
  static_assert(!KG || B_MN, "K-grouped mode reads both operands MN-major");
  static_assert(!B_MN || (EPI == EPI_F32 && BN >= 64), "MN-major B: fp32 epilogue");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* ostage = smem + S::RING_BYTES;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + S::RING_BYTES + S::OSTAGE_BYTES);
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

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < S::ACC_STAGES; ++a) {
      mbar_init(&accf_bar[a], 1);
      mbar_init(&acce_bar[a], S::EPI_THREADS);
    }
    mbar_init(final_bar, 1);
    for (int q = 0; q < S::QDEPTH; ++q) {
      mbar_init(&qfull_bar[q], 1);
      mbar_init(&qempty_bar[q], 1 + S::EPI_THREADS);   // consumers: MMA thread + epilogue threads
    }
    *s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, S::TMEM_COLS);
  // everything above touches only shared memory, TMEM and the kernel parameters; the
  // previous kernel on the stream (which wrote this kernel's inputs) is waited for here
  pdl_wait();
  pdl_trigger();

  // Row-chunk prefix over groups (warp 2; G <= 1024): s_prefix[g] = sum_{g'<g} ceil(counts[g'] / (MT*128)).
  constexpr int CH = MT * kBM;
  if (warp == 2) {
    if (KG) {
      if (lane == 0) *s_total = p.G * ((p.M + CH - 1) / CH);
    } else if (p.G > 0) {
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
  tc_fence_after();

  const uint32_t tmem_base = *tmem_slot;
  const int total_chunks = *s_total;
  const int total_units = total_chunks * p.n_blocks;
  WaitCtl wc{s_abort, p.status, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer + scheduler
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int qi = 0;
      uint32_t qphase = 0;
      int filled_phase[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) filled_phase[s] = -1;
      // the unit index is taken only when its loads are about to be issued: units
      // with neighbouring indices (the row chunks of one expert's column block,
      // which share the weight tile) then start close together and share it in L2
      // the first unit of every CTA is its block index (no counter round trip on the way in);
      // later ones come from the counter, offset past those
      bool first = true;
      while (true) {
        int u = first ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(p.sched, 1);
        first = false;
        if (u >= total_units) u = -1;
        if (!mbar_wait(&qempty_bar[qi], qphase ^ 1u, wc)) break;
        s_queue[qi] = u;
        mbar_arrive(&qfull_bar[qi]);
        if (++qi == S::QDEPTH) { qi = 0; qphase ^= 1u; }
        if (u < 0) break;
        const Unit U = decode_unit<MT, EPI, BN>(u, p, s_prefix, total_chunks);
        const int ntile = (U.rows + kBM - 1) / kBM;
        const uint32_t bytes = ntile * S::A_BYTES + S::B_BYTES;
        const int num_kb = (U.kcount + kBK - 1) / kBK;
        // MN-major B: the K row the group's B starts at
        const int b_k0 = KG ? U.k0 : U.g * p.b_group_rows;
        bool ok = true;
        // B row blocks of 128 this unit streams (SwiGLU: gate block, up block)
        constexpr int NBB = BN >= 128 ? BN / 128 : 1;
        int brow[NBB];
        if (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD) {
          brow[0] = U.b_row;
          brow[NBB - 1] = U.b_row + p.b_up_rows;
        } else {
#pragma unroll
          for (int i = 0; i < NBB; ++i) brow[i] = U.b_row + i * 128;
        }
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, wc)) { ok = false; break; }
          uint8_t* st = ring + stage * S::STAGE_BYTES;
          mbar_arrive_expect_tx(&full_bar[stage], bytes);
          for (int t = 0; t < ntile; ++t) {
            if (A_MN) {
              tma_load_2d(st + t * S::A_BYTES, &tmA, &full_bar[stage], U.a_m0 + t * kBM, U.k0 + kb * kBK);
              tma_load_2d(st + t * S::A_BYTES + kMnBoxBytes, &tmA, &full_bar[stage], U.a_m0 + t * kBM + 64,
                          U.k0 + kb * kBK);
            } else {
              tma_load_2d(st + t * S::A_BYTES, &tmA, &full_bar[stage], kb * kBK, U.row0 + t * kBM);
            }
          }
          if (B_MN) {
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(st + MT * S::A_BYTES + i * kMnBoxBytes, &tmB, &full_bar[stage], U.nb * BN + i * 64,
                          b_k0 + kb * kBK);
          } else if (BN >= 128) {
#pragma unroll
            for (int i = 0; i < NBB; ++i)
              tma_load_2d(st + MT * S::A_BYTES + i * (kBM * kBK * 2), &tmB, &full_bar[stage], kb * kBK,
                               brow[i]);
          } else {
            tma_load_2d(st + MT * S::A_BYTES, &tmB, &full_bar[stage], kb * kBK, U.b_row);
          }
          filled_phase[stage] = static_cast<int>(phase);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      // this CTA takes no more units: once every CTA is past this point the counter is reset
      sched_release(p.sched);
      // Let every copy this thread issued land before the CTA can exit.
      WaitCtl drain{nullptr, p.status, p.timeout_ns};
      for (int s = 0; s < STAGES; ++s)
        if (filled_phase[s] >= 0) mbar_wait(&full_bar[s], static_cast<uint32_t>(filled_phase[s]), drain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Lane 0 issues; in K-grouped mode the whole warp follows the ring so that
    // it can zero the rows past a group's end before the block's MMAs.
    if (KG || lane == 0) {
      const bool leader = lane == 0;
      constexpr uint32_t IDESC = idesc_bf16_f32(kBM, BN, A_MN, B_MN);
      // a tile with at most 64 valid rows runs as an M = 64 MMA (same per-row products and order)
      constexpr uint32_t IDESC64 = idesc_bf16_f32(64, BN, A_MN, B_MN);
      // per K = 16 step: +32 B inside a K-major swizzle row, +2048 B (16 rows) MN-major; encoded >> 4
      constexpr uint64_t A_STEP = A_MN ? 128u : 2u;
      constexpr uint64_t B_STEP = B_MN ? 128u : 2u;
      // stage-0 descriptors; stage s, row tile t add s * STAGE_BYTES + t * A_BYTES to the start
      // address (encoded >> 4; shared addresses stay below 256 KB, so the 14-bit field never carries)
      const uint64_t adesc0 = A_MN ? sdesc_mn_sw128(smem_u32(ring)) : sdesc_k_sw128(smem_u32(ring));
      const uint64_t bdesc0 = B_MN ? sdesc_mn_sw128(smem_u32(ring + MT * S::A_BYTES))
                                   : sdesc_k_sw128(smem_u32(ring + MT * S::A_BYTES));
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int qi = 0;
      uint32_t qphase = 0;
      while (true) {
        bool okw = mbar_wait(&qfull_bar[qi], qphase, wc);
        if (KG) okw = __all_sync(0xffffffffu, okw);
        if (!okw) break;
        const int u = s_queue[qi];
        if (KG) __syncwarp();
        if (leader) mbar_arrive(&qempty_bar[qi]);
        if (++qi == S::QDEPTH) { qi = 0; qphase ^= 1u; }
        if (u < 0) break;
        const Unit U = decode_unit<MT, EPI, BN>(u, p, s_prefix, total_chunks);
        const int ntile = (U.rows + kBM - 1) / kBM;
        const int num_kb = (U.kcount + kBK - 1) / kBK;
        okw = mbar_wait(&acce_bar[acc], acc_phase ^ 1u, wc);
        if (KG) okw = __all_sync(0xffffffffu, okw);
        if (!okw) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * S::ACC_COLS);
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          okw = mbar_wait(&full_bar[stage], phase, wc);
          if (KG) okw = __all_sync(0xffffffffu, okw);
          if (!okw) { ok = false; break; }
          tc_fence_after();
          uint8_t* st = ring + stage * S::STAGE_BYTES;
          // K = 16 steps this block issues: a K-grouped group's last block stops at the
          // step holding its last row (the skipped steps would add exact zeros)
          int nkk = kBK / 16;
          if (KG) {
            const int rem = U.kcount - kb * kBK;
            if (rem < kBK) {
              nkk = (rem + 15) >> 4;
              // rows of that step past the group's end belong to the next group (or are
              // the zero fill): clear them in both operands
              if (rem & 15) {
                zero_k_tail(st, ntile * 2, rem, nkk * 16);
                zero_k_tail(st + MT * S::A_BYTES, BN / 64, rem, nkk * 16);
                fence_proxy_async_shared();
              }
            }
            __syncwarp();
          }
          if (leader) {
            const uint64_t so = static_cast<uint64_t>((stage * S::STAGE_BYTES) >> 4);
            const uint64_t bdesc = bdesc0 + so;
            for (int t = 0; t < ntile; ++t) {
              const uint64_t adesc = adesc0 + so + static_cast<uint64_t>((t * S::A_BYTES) >> 4);
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk)
                if (kk < nkk)
                  umma_bf16(d0 + static_cast<uint32_t>(t * BN), adesc + A_STEP * kk, bdesc + B_STEP * kk,
                            U.rows - t * kBM <= 64 ? IDESC64 : IDESC, (kb | kk) != 0 ? 1u : 0u);
            }
            umma_commit(&empty_bar[stage]);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        // (a K-grouped unit whose group has no rows issues no MMA: its epilogue writes zeros)
        if (leader) umma_commit(&accf_bar[acc]);
        if (++acc == S::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
      }
      // Every MMA this thread issued must finish before TMEM is released.
      if (leader) {
        umma_commit(final_bar);
        WaitCtl drain{nullptr, p.status, p.timeout_ns};
        mbar_wait(final_bar, 0, drain);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;                 // 0 .. EPI_WARPS-1
    const int q = warp & 3;                  // TMEM lane quadrant this warp may access
    constexpr int NPART = S::EPI_WARPS / 4;  // warps sharing one lane quadrant
    const int half = ew >> 2;                // which of them this warp is (column chunks c = half mod NPART)
    int acc = 0;
    uint32_t acc_phase = 0;
    int qi = 0;
    uint32_t qphase = 0;
    while (true) {
      const bool okq = mbar_wait(&qfull_bar[qi], qphase, wc);
      if (!__all_sync(0xffffffffu, okq)) break;
      const int u = s_queue[qi];
      mbar_arrive(&qempty_bar[qi]);
      if (++qi == S::QDEPTH) { qi = 0; qphase ^= 1u; }
      if (u < 0) break;
      const Unit U = decode_unit<MT, EPI, BN>(u, p, s_prefix, total_chunks);
      const int ntile = (U.rows + kBM - 1) / kBM;
      // every lane waits; the warp proceeds only if all lanes saw the phase
      // complete, so the .sync.aligned TMEM loads below never run diverged
      const bool ok = mbar_wait(&accf_bar[acc], acc_phase, wc);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      for (int t = 0; t < ntile; ++t) {
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>(acc * S::ACC_COLS + t * BN);
        // The warp's rows in this tile: lane L of quadrant q holds tile row q*32 + L for
        // an M = 128 accumulator, and row q*16 + L (lanes 0..15) for an M = 64 one.
        const int tile_rows = U.rows - t * kBM;
        const bool m64 = tile_rows <= 64;
        const int wrow = m64 ? q * 16 : q * 32;
        const int rows_valid = m64 ? max(0, min(16, tile_rows - q * 16)) : tile_rows - q * 32;
        // fp32 D through bulk tensor stores: each 32-row x 16-column piece goes out through the
        // warp's staging buffer (already in the 64-byte swizzle layout) as one store.  The map is
        // [G][M][N] in K-grouped mode (rows past the group's M and columns past N are clipped) and
        // [1][rows][N] otherwise, where only whole 32-row slabs of one group take this path (a
        // slab that ends inside the tile would reach the next group's rows).
        if (EPI == EPI_F32 && p.out_map && !m64 && (KG ? rows_valid > 0 : rows_valid >= 32)) {
          const int n0 = U.nb * BN;
          const int m0 = KG ? U.a_m0 + t * kBM + wrow : U.row0 + t * kBM + wrow;
          const int z0 = KG ? U.g : 0;
          uint8_t* stg = ostage + ew * kOutStageBytes;
#pragma unroll 1
          for (int c = half; c < BN / 32; c += NPART) {
            uint32_t v[32];
            tmem_ld32(tbase + c * 32, v);
            tmem_ld_wait();
            tmem_reg_fence(v);
            if (KG && U.kcount == 0) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0u;       // a group with no rows: the sum over nothing
            }
            {
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
                  tma_store_3d(&tmO, stg, col, m0, z0);
                  bulk_commit_group();
                }
              }
            }
          }
        } else if (EPI == EPI_F32) {
          // the warp's 32 rows start at tile row q*32; lane L stores row r of them
          const int n0 = U.nb * BN;
          uint8_t* obase = rows_valid > 0 ? reinterpret_cast<uint8_t*>(static_cast<float*>(p.out) +
                                                (static_cast<long long>(U.row0) + t * kBM + wrow) * p.ldo + n0)
                                          : nullptr;
          uint8_t* stg = ostage + ew * kOutStageBytes;
          if (p.out_map) {
            if (lane == 0) bulk_wait_group_read0();   // a bulk store may still read the buffer
            __syncwarp();
          }
#pragma unroll 1
          for (int c = half; c < BN / 32; c += NPART) {
            uint32_t v[32];
            tmem_ld32(tbase + c * 32, v);
            tmem_ld_wait();
            tmem_reg_fence(v);
            if (KG && U.kcount == 0) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0u;       // a group with no rows: the sum over nothing
            }
            if (rows_valid > 0) {
              const int bytes_valid = (p.N - (n0 + c * 32)) * 4;
              stage_store_rows64(stg, *reinterpret_cast<uint32_t(*)[16]>(&v[0]), obase + c * 128, p.ldo * 4,
                                 rows_valid, bytes_valid);
              stage_store_rows64(stg, *reinterpret_cast<uint32_t(*)[16]>(&v[16]), obase + c * 128 + 64, p.ldo * 4,
                                 rows_valid, bytes_valid - 64);
            }
          }
        } else if (EPI == EPI_SWIGLU_BWD) {
          // recomputed gate/up columns [n0, n0+HALF) of h: dg -> out[:, n0..], du -> out[:, N+n0..], h -> out2
          constexpr int HALF = BN / 2;
          const int n0 = U.nb * HALF;
          const long long r0 = static_cast<long long>(U.row0) + t * kBM + wrow;
          uint8_t* stg = ostage + ew * kOutStageBytes;
#pragma unroll 1
          for (int c = half; c < HALF / 32; c += NPART) {
            uint32_t gv[32], uv[32];
            tmem_ld32(tbase + c * 32, gv);
            tmem_ld32(tbase + HALF + c * 32, uv);
            tmem_ld_wait();
            tmem_reg_fence(gv);
            tmem_reg_fence(uv);
            if (rows_valid > 0) {
              const int col = n0 + c * 32;
              __nv_bfloat16* dgu = static_cast<__nv_bfloat16*>(p.out) + r0 * p.ldo;
              swiglu_bwd_chunk(stg, gv, uv, reinterpret_cast<const uint8_t*>(p.aux + r0 * p.ld_aux + col),
                               p.ld_aux * 4, reinterpret_cast<uint8_t*>(dgu + col),
                               reinterpret_cast<uint8_t*>(dgu + p.N + col), p.ldo * 2,
                               p.out2 != nullptr ? reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(p.out2) +
                                                                              r0 * p.ldo2 + col)
                                                 : nullptr,
                               p.ldo2 * 2, rows_valid, p.N - col);
            }
          }
        } else {
          constexpr int HALF = BN / 2;
          const int n0 = U.nb * HALF;
          uint8_t* obase = rows_valid > 0
                               ? reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(p.out) +
                                                            (static_cast<long long>(U.row0) + t * kBM + wrow) * p.ldo +
                                                            n0)
                               : nullptr;
          uint8_t* stg = ostage + ew * kOutStageBytes;
#pragma unroll 1
          for (int c = half; c < HALF / 32; c += NPART) {
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
                const float h1 =
                    __fmul_rn(silu_f32(__uint_as_float(gv[2 * j + 1])), __uint_as_float(uv[2 * j + 1]));
                packed[j] = pack_bf16x2(h0, h1);
              }
              stage_store_rows64(stg, packed, obase + c * 64, p.ldo * 2, rows_valid, (p.N - (n0 + c * 32)) * 2);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acce_bar[acc]);
      if (++acc == S::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
    }
    // the bulk stores this warp issued complete before the CTA exits
    if (EPI == EPI_F32 && lane == 0) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

}  // namespace invmoe
