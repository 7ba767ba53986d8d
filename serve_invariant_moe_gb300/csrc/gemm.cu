// gemm.cu -- host side of the tcgen05 GEMM engine: tensor maps, launch shapes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "internal.h"
#include "tc_gemm.cuh"
#include "tc_gemm2.cuh"
#include "tc_gemm_tok.cuh"
#include "tc_gemm_small.cuh"

namespace invmoe {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// Row-major bf16 [rows, inner] matrix; box = 64 elements (128 B, one swizzle row) x box_rows.
int make_tmap(CUtensorMap* m, const void* base, long long inner, long long rows, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(INVMOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(INVMOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return INVMOE_OK;
}

// Row-major bf16 [rows, inner] matrix as a rank-3 tensor (64 elements, rows, inner / 64 blocks):
// one box = 64 elements x box_rows rows x kblocks consecutive 64-column blocks of the row.
int make_tmap_kblocks(CUtensorMap* m, const void* base, long long inner, long long rows, int box_rows, int kblocks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(INVMOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (inner % kBK != 0) return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "K=%lld is not a multiple of 64", inner);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kBK), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(inner / kBK)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 2, static_cast<cuuint64_t>(kBK) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(box_rows),
                       static_cast<cuuint32_t>(kblocks)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(INVMOE_ERR_CUDA, "cuTensorMapEncodeTiled (K blocks) failed (%d)", (int)r);
  return INVMOE_OK;
}

// SwiGLU weights [E][2F][K] bf16 as a rank-5 tensor (K, 16 rows, gate/up, F/16 row
// groups, E) whose box (64, 16, 2, 4, 1) holds 4 groups of 16 gate rows each
// followed by the matching 16 up rows.
int make_tmap_gate_up(CUtensorMap* m, const void* base, long long K, long long F, long long E) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(INVMOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (F % 64 != 0) return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "F=%lld is not a multiple of 64", F);
  const cuuint64_t row = static_cast<cuuint64_t>(K) * 2;
  cuuint64_t dims[5] = {static_cast<cuuint64_t>(K), 16, 2, static_cast<cuuint64_t>(F / 16),
                        static_cast<cuuint64_t>(E)};
  cuuint64_t strides[4] = {row, row * F, row * 16, row * 2 * F};
  cuuint32_t box[5] = {static_cast<cuuint32_t>(kBK), 16, 2, 4, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(INVMOE_ERR_CUDA, "cuTensorMapEncodeTiled (gate/up) failed (%d)", (int)r);
  return INVMOE_OK;
}

// K-grouped fp32 output of G groups, each [M rows, N columns] with row stride
// ldo floats, group g starting at row g*M: a [G][M][N] map whose box (16
// columns = 64 B, 32 rows) matches the epilogue's 64-byte-swizzled staging.
int make_tmap_out_grouped_f32(CUtensorMap* m, void* base, long long N, long long M, long long G, long long ldo) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(INVMOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (ldo % 4 != 0 || (reinterpret_cast<uintptr_t>(base) & 15) != 0)
    return set_error(INVMOE_ERR_INVALID_ARG, "K-grouped output needs a 16-byte aligned base and ldo %% 4 == 0");
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(G)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldo) * 4, static_cast<cuuint64_t>(ldo) * 4 * M};
  cuuint32_t box[3] = {16, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(INVMOE_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (%d)", (int)r);
  return INVMOE_OK;
}

// Raise a kernel's dynamic shared-memory limit once per device (devices 0..63
// are remembered in `done`; a higher device index sets it on every call).
int set_smem_attr(const void* kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  int rc = check_cuda(cudaGetDevice(&dev), "cudaGetDevice");
  if (rc) return rc;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return INVMOE_OK;
  rc = check_cuda(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
                  "cudaFuncSetAttribute");
  if (rc) return rc;
  if (bit != 0) done.fetch_or(bit, std::memory_order_release);
  return INVMOE_OK;
}

GemmParams make_params(const GemmCall& c, int nb_cols) {
  GemmParams p{};
  p.K = c.K;
  p.N = c.N;
  p.n_blocks = (c.N + nb_cols - 1) / nb_cols;
  p.M = c.M;
  p.G = c.G;
  p.counts = c.counts;
  p.offsets = c.offsets;
  p.b_group_rows = c.b_group_rows;
  p.b_up_rows = c.b_up_rows;
  p.n_major = c.n_major;
  p.out = c.out;
  p.ldo = c.ldo;
  p.status = c.status;
  // the dynamic-schedule counter lives in the workspace's status block, after the status word
  p.sched = c.sched ? c.sched : reinterpret_cast<int*>(reinterpret_cast<char*>(c.status) + 64);
  p.timeout_ns = kTimeoutNs;
  p.part = c.part;
  p.nch = c.part_ld > 0 ? static_cast<int>(c.part_ld) : (c.N + 255) / 256;
  p.col0 = c.target_col0;
  p.target = c.target;
  p.tgt_logit = c.tgt_logit;
  p.m_group = c.m_group > 0 ? c.m_group : (1 << 30);
  p.row_lse = c.row_lse;
  p.row_scale = c.row_scale;
  p.aux = c.aux;
  p.ld_aux = c.ld_aux;
  p.out2 = c.out2;
  p.ldo2 = c.ldo2;
  p.kgroup = c.kgroup;
  return p;
}

// Single-CTA engine.  K-major operands as [rows, K]; an MN-major operand is
// stored [outer rows, inner] with the M or N index inner (a_rows / b_rows =
// inner extent, a_outer / b_outer = stored rows).
template <int BN, int MT, int EPI, int STAGES, bool A_MN = false, bool B_MN = false, bool KG = false>
int launch(const GemmCall& c, cudaStream_t st) {
  using S = GemmShape<BN, MT, EPI, STAGES>;
  if (KG != (c.kgroup != 0)) return set_error(INVMOE_ERR_INVALID_ARG, "K-grouped flag does not match the variant");
  if (c.G > S::MAX_GROUPS) return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "more than %d groups", S::MAX_GROUPS);
  CUtensorMap ta, tb;
  int rc = A_MN ? make_tmap(&ta, c.A, c.a_rows, c.a_outer, 64) : make_tmap(&ta, c.A, c.K, c.a_rows, kBM);
  if (rc) return rc;
  rc = B_MN ? make_tmap(&tb, c.B, c.b_rows, c.b_outer, 64)
            : make_tmap(&tb, c.B, c.K, c.b_rows, BN >= 128 ? 128 : BN);
  if (rc) return rc;
  // fp32 D: a store map for the bulk-store epilogue ([G][M][N] in K-grouped mode, [1][rows][N]
  // otherwise); without one (unaligned output) the epilogue keeps its plain stores
  CUtensorMap to = ta;
  bool out_map = false;
  if (EPI == EPI_F32 && c.N > 0) {
    const long long rows = KG ? c.M : (c.G > 0 ? c.a_rows : c.M);
    const long long groups = KG ? c.G : 1;
    if (rows > 0 && groups > 0 && c.ldo % 4 == 0 && (reinterpret_cast<uintptr_t>(c.out) & 15) == 0) {
      if ((rc = make_tmap_out_grouped_f32(&to, c.out, c.N, rows, groups, c.ldo))) return rc;
      out_map = true;
    }
  }

  static std::atomic<uint64_t> attr_set{0};
  if ((rc = set_smem_attr(reinterpret_cast<const void*>(tc_gemm_kernel<BN, MT, EPI, STAGES, A_MN, B_MN, KG>),
                          S::SMEM_BYTES, attr_set)))
    return rc;
  int sms = 0;
  if ((rc = device_sm_count(&sms))) return rc;

  GemmParams p = make_params(c, (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD) ? BN / 2 : BN);
  p.out_map = out_map ? 1 : 0;

  constexpr long long CH = static_cast<long long>(MT) * kBM;
  long long max_chunks = KG ? static_cast<long long>(c.G) * ((c.M + CH - 1) / CH)
                            : (c.G > 0) ? (c.a_rows + CH - 1) / CH + c.G : (c.M + CH - 1) / CH;
  long long max_units = max_chunks * p.n_blocks;
  if (max_units <= 0) return INVMOE_OK;
  const int grid = static_cast<int>(max_units < sms ? max_units : sms);
  // the unit counter (p.sched) is zero here: the workspace starts zero-filled and every
  // launch's last CTA resets it (sched_release)
  ProfScope prof(c.name ? c.name : "tc_gemm", st);
  return check_cuda(launch_kernel(tc_gemm_kernel<BN, MT, EPI, STAGES, A_MN, B_MN, KG>, dim3(grid), dim3(S::THREADS),
                                  S::SMEM_BYTES, st, ta, tb, to, p),
                    "tc_gemm_kernel launch");
}


// CTA-pair engine: clusters of 2, grid = 2 x min(units, SMs / 2).  A K-major
// operand is [rows, K] (box 64 K x 128 rows); an MN-major one is [K, rows]
// (box 64 rows x 64 K, two per 128-row half tile).
template <int EPI, int STAGES, bool A_MN = false, bool B_MN = false>
int launch_pair(const GemmCall& c, cudaStream_t st) {
  using S = PairShape<EPI, STAGES>;
  if (c.G > S::MAX_GROUPS) return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "more than %d groups", S::MAX_GROUPS);
  CUtensorMap ta, tb;
  int rc = A_MN ? make_tmap(&ta, c.A, c.a_rows, c.K, 64) : make_tmap(&ta, c.A, c.K, c.a_rows, kBM);
  if (rc) return rc;
  rc = B_MN ? make_tmap(&tb, c.B, c.b_rows, c.K, 64) : make_tmap(&tb, c.B, c.K, c.b_rows, kBM);
  if (rc) return rc;
  static std::atomic<uint64_t> attr_set{0};
  if ((rc = set_smem_attr(reinterpret_cast<const void*>(tc_gemm_pair_kernel<EPI, STAGES, A_MN, B_MN>),
                          S::SMEM_BYTES, attr_set)))
    return rc;
  int sms = 0;
  if ((rc = device_sm_count(&sms))) return rc;
  GemmParams p = make_params(c, (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_BWD) ? 128 : 256);
  // fp32 D: a [1][rows][N] store map for the bulk-store epilogue (none for an unaligned output)
  CUtensorMap to = ta;
  if (EPI == EPI_F32 && c.N > 0) {
    const long long rows = c.G > 0 ? c.a_rows : c.M;
    if (rows > 0 && c.ldo % 4 == 0 && (reinterpret_cast<uintptr_t>(c.out) & 15) == 0) {
      if ((rc = make_tmap_out_grouped_f32(&to, c.out, c.N, rows, 1, c.ldo))) return rc;
      p.out_map = 1;
    }
  }
  constexpr long long CH = 2LL * kBM;
  long long max_chunks = (c.G > 0) ? (c.a_rows + CH - 1) / CH + c.G : (c.M + CH - 1) / CH;
  long long max_units = max_chunks * p.n_blocks;
  if (max_units <= 0) return INVMOE_OK;
  const long long pairs = max_units < sms / 2 ? max_units : sms / 2;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the unit counter (p.sched) is zero here: the workspace starts zero-filled and every
  // launch's last CTA resets it (sched_release)
  ProfScope prof(c.name ? c.name : "tc_gemm_pair", st);
  return check_cuda(launch_kernel_ex(tc_gemm_pair_kernel<EPI, STAGES, A_MN, B_MN>,
                                     dim3(static_cast<unsigned>(2 * pairs)), dim3(S::THREADS), S::SMEM_BYTES, st, attr,
                                     1, ta, tb, to, p),
                    "tc_gemm_pair_kernel launch");
}

// Token-column engine (grouped only): clusters of 2, grid = 2 x min(units, SMs / 2).
// Weights [G * b_group_rows, K] in 64-row boxes, tokens [rows, K] in 32-, 64-, 128- or 160-row boxes.
template <int EPI, int STAGES, int CHUNK>
int launch_tok(const GemmCall& c, cudaStream_t st) {
  using S = TokShape<EPI, STAGES, CHUNK>;
  if (c.G <= 0) return set_error(INVMOE_ERR_INVALID_ARG, "the token-column engine is grouped only");
  if (c.G > S::MAX_GROUPS) return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "more than %d groups", S::MAX_GROUPS);
  const int wb_cols = EPI == EPI_SWIGLU ? 128 : 256;
  if (c.N % wb_cols != 0)
    return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "N=%d is not a multiple of %d", c.N, wb_cols);
  CUtensorMap tw, tx, txm, txb, txt;
  int rc = EPI == EPI_SWIGLU ? make_tmap_gate_up(&tw, c.B, c.K, c.b_up_rows, c.b_rows / c.b_group_rows)
                             : make_tmap(&tw, c.B, c.K, c.b_rows, 128);
  if (rc) return rc;
  if ((rc = make_tmap(&tx, c.A, c.K, c.a_rows, kTokBoxRows))) return rc;
  txm = txb = txt = tx;         // the 64-token form loads 32-row boxes only, the 128-token form 32 or 64
  if (CHUNK >= 128 && (rc = make_tmap(&txm, c.A, c.K, c.a_rows, kTokMidRows))) return rc;
  if (CHUNK == kTokChunk) {
    if ((rc = make_tmap(&txb, c.A, c.K, c.a_rows, kTokBigRows))) return rc;
    if ((rc = make_tmap(&txt, c.A, c.K, c.a_rows, kTokTwoRows))) return rc;
  }
  static std::atomic<uint64_t> attr_set{0};
  if ((rc = set_smem_attr(reinterpret_cast<const void*>(tc_gemm_tok_kernel<EPI, STAGES, CHUNK>), S::SMEM_BYTES, attr_set)))
    return rc;
  int sms = 0;
  if ((rc = device_sm_count(&sms))) return rc;
  GemmParams p = make_params(c, wb_cols);
  const long long max_chunks = (c.a_rows + CHUNK - 1) / CHUNK + c.G;
  const long long max_units = max_chunks * p.n_blocks;
  if (max_units <= 0) return INVMOE_OK;
  const long long pairs = max_units < sms / 2 ? max_units : sms / 2;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the unit counter (p.sched) is zero here: the workspace starts zero-filled and every
  // launch's last producer resets it (sched_release)
  ProfScope prof(c.name ? c.name : "tc_gemm_tok", st);
  return check_cuda(launch_kernel_ex(tc_gemm_tok_kernel<EPI, STAGES, CHUNK>, dim3(static_cast<unsigned>(2 * pairs)),
                                     dim3(S::THREADS), S::SMEM_BYTES, st, attr, 1, tw, tx, txm, txb, txt, p),
                    "tc_gemm_tok_kernel launch");
}

// SwiGLU weights [2F, K] (gate rows, then up rows) for the small-M kernel: a rank-4 tensor (64 elements,
// F rows, gate/up, K blocks) whose box (64, 32, 2, kblocks) holds, per K block, 32 gate rows followed by
// the matching 32 up rows.
int make_tmap_gate_up_small(CUtensorMap* m, const void* base, long long K, long long F, int kblocks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(INVMOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  if (K % kBK != 0) return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "K=%lld is not a multiple of 64", K);
  const cuuint64_t row = static_cast<cuuint64_t>(K) * 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(kBK), static_cast<cuuint64_t>(F), 2, static_cast<cuuint64_t>(K / kBK)};
  cuuint64_t strides[3] = {row, row * F, static_cast<cuuint64_t>(kBK) * 2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(kBK), 32, 2, static_cast<cuuint32_t>(kblocks)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(INVMOE_ERR_CUDA, "cuTensorMapEncodeTiled (small gate/up) failed (%d)", (int)r);
  return INVMOE_OK;
}

// At most 64 rows of A, dense: fp32 out in 64-column tiles, or SwiGLU h in 32-column tiles, one tile per
// CTA (tc_gemm_small.cuh).
template <int EPI, int ABOX>
int launch_small_rows(const GemmCall& c, cudaStream_t st) {
  using S = SmallShape<ABOX>;
  const bool swiglu = EPI == EPI_SWIGLU;
  const int cw = swiglu ? 32 : 64;
  const int eb = swiglu ? 2 : 4;     // output element bytes
  if (c.G != 0 || c.M > 64 || (swiglu ? c.N % 32 != 0 || c.b_up_rows != c.N : c.N % 4 != 0) ||
      (c.ldo * eb) % 16 != 0 || (reinterpret_cast<uintptr_t>(c.out) & 15) != 0)
    return set_error(INVMOE_ERR_INVALID_ARG, "the small-M GEMM takes a dense A of at most 64 rows and an aligned output");
  CUtensorMap ta, tb;
  int rc = make_tmap_kblocks(&ta, c.A, c.K, c.a_rows, ABOX, kSmallKsub);
  if (rc) return rc;
  rc = swiglu ? make_tmap_gate_up_small(&tb, c.B, c.K, c.N, kSmallKsub)
              : make_tmap_kblocks(&tb, c.B, c.K, c.b_rows, 64, kSmallKsub);
  if (rc) return rc;
  static std::atomic<uint64_t> attr_set{0};
  if ((rc = set_smem_attr(reinterpret_cast<const void*>(tc_gemm_small_kernel<EPI, ABOX>), S::SMEM_BYTES, attr_set)))
    return rc;
  const int grid = (c.N + cw - 1) / cw;
  ProfScope prof(c.name ? c.name : "tc_gemm_small", st);
  return check_cuda(launch_kernel(tc_gemm_small_kernel<EPI, ABOX>, dim3(grid), dim3(kSmallThreads), S::SMEM_BYTES, st,
                                  ta, tb, c.M, c.N, c.K, c.out, c.ldo, c.status, kTimeoutNs),
                    "tc_gemm_small_kernel launch");
}

// at most 16 rows of A: 16-row copies of A and a 5-stage ring; otherwise 64-row copies, 3 stages
template <int EPI>
int launch_small(const GemmCall& c, cudaStream_t st) {
  return c.M <= 16 ? launch_small_rows<EPI, 16>(c, st) : launch_small_rows<EPI, 64>(c, st);
}

}  // namespace

int gemm_run(const GemmCall& c, cudaStream_t st) {
  if (c.a_rows <= 0 || (c.G == 0 && c.M <= 0)) return INVMOE_OK;
  if (c.K <= 0) return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "K=%d", c.K);
  // the MN-major variants take any K (zero-filled tail); every other one needs K % 64 == 0
  const bool ragged_k_ok = c.variant == GV_PAIR_F32_BMN || c.variant == GV_PAIR_F32_AMN_BMN ||
                           c.variant == GV_F32_BN256_MT1_KGROUP;
  if (!ragged_k_ok && c.K % kBK != 0)
    return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of 64", c.K);
  if (c.variant == GV_PAIR_F32_BMN && c.K % 8 != 0)
    return set_error(INVMOE_ERR_UNSUPPORTED_SHAPE, "K=%d is not a multiple of 8 (row stride of A)", c.K);
  switch (c.variant) {
    case GV_F32_BN256_MT1: return launch<256, 1, EPI_F32, 4>(c, st);
    case GV_F32_BN256_MT2: return launch<256, 2, EPI_F32, 3>(c, st);
    case GV_F32_BN128_MT1: return launch<128, 1, EPI_F32, 6>(c, st);
    case GV_F32_BN64_MT1: return launch<64, 1, EPI_F32, 8>(c, st);
    case GV_SWIGLU_BN256_MT2: return launch<256, 2, EPI_SWIGLU, 3>(c, st);
    case GV_PAIR_F32: return launch_pair<EPI_F32, 6>(c, st);
    case GV_PAIR_LSE: return launch_pair<EPI_LSE, 6>(c, st);
    case GV_PAIR_SWIGLU: return launch_pair<EPI_SWIGLU, 6>(c, st);
    case GV_PAIR_DLOGITS: return launch_pair<EPI_DLOGITS, 6>(c, st);
    case GV_PAIR_F32_BMN: return launch_pair<EPI_F32, 6, false, true>(c, st);
    case GV_PAIR_F32_AMN_BMN: return launch_pair<EPI_F32, 6, true, true>(c, st);
    case GV_F32_BN256_MT2_BMN: return launch<256, 2, EPI_F32, 3, false, true, false>(c, st);
    case GV_SWIGLU_BWD_BN256_MT2: return launch<256, 2, EPI_SWIGLU_BWD, 3>(c, st);
    case GV_F32_BN256_MT1_KGROUP: return launch<256, 1, EPI_F32, 4, true, true, true>(c, st);
    case GV_PAIR_SWIGLU_BWD: return launch_pair<EPI_SWIGLU_BWD, 6>(c, st);
    // units by batch size (an expert with more tokens than a unit takes several): decode batches
    // (at most 1024 token slots, or at most 16 per expert on average) 64 tokens, a 32-row token
    // tile, 5 stages of two K blocks; at most 64 slots per expert 128 tokens, a 64-row tile,
    // 4 stages of two K blocks (SwiGLU) or 8 of one (fp32)
    case GV_TOK_SWIGLU:
      if (c.a_rows <= 1024 || c.a_rows <= 16LL * c.G) return launch_tok<EPI_SWIGLU, 5, 64>(c, st);
      if (c.a_rows <= 64LL * c.G) return launch_tok<EPI_SWIGLU, 4, 128>(c, st);
      // a 6-stage ring for at most 256 experts (its chunk table), else 5 stages
      return c.G <= 256 ? launch_tok<EPI_SWIGLU, 6, kTokChunk>(c, st) : launch_tok<EPI_SWIGLU, 5, kTokChunk>(c, st);
    case GV_F32_SMALL64: return launch_small<EPI_F32>(c, st);
    case GV_SWIGLU_SMALL64: return launch_small<EPI_SWIGLU>(c, st);
    case GV_TOK_F32:
      if (c.a_rows <= 1024 || c.a_rows <= 16LL * c.G) return launch_tok<EPI_F32, 5, 64>(c, st);
      if (c.a_rows <= 64LL * c.G) return launch_tok<EPI_F32, 8, 128>(c, st);
      return c.G <= 256 ? launch_tok<EPI_F32, 6, kTokChunk>(c, st) : launch_tok<EPI_F32, 5, kTokChunk>(c, st);
  }
  return set_error(INVMOE_ERR_INVALID_ARG, "unknown GEMM variant %d", (int)c.variant);
}

}  // namespace invmoe
