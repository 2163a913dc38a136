// gemm_epi.cu -- host side of the C ABI in include/gemm_epi.h.
//
// create = validate the descriptor and the epilogue program, derive the
// kernel flags (host only, no CUDA call).  run = check the device and the
// pointer pack, zero the reduction outputs and the workspace with
// cudaMemsetAsync, encode the TMA descriptors for this call's pointers and
// launch the persistent kernel on the caller's stream.  This follows the
// "build once, execute with a variant pack of pointers and a workspace" shape
// of the cuDNN Graph API tutorial (five-step build paragraph); nothing here
// allocates or synchronises, so a run can be captured in a CUDA graph (same
// page, CUDA graph paragraph).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "gemm_epi.h"
#include "programs.cuh"
#include "rmsnorm_bwd.cuh"
#include "unfused_kernel.cuh"

namespace {

thread_local std::string g_last_error;

gemm_epi_status fail(gemm_epi_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

gemm_epi_status cuda_fail(cudaError_t e, const char* what) {
  return fail(GEMM_EPI_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t WS_HEADER = 256;  // status words; row counters follow
constexpr int DEFAULT_GROUP_M = 16;
// Part of L2 that keeps a wave's operand panels until the next wave reads them
// (measured: a wave of the persistent walk reads ~16 A and ~5 B panels of
// 256 x K, and the DRAM reads of every benchmark shape follow from assuming
// that they stay when they fit in about 60 MB, and are read again otherwise).
constexpr double L2_KEEP_BYTES = 60e6;
constexpr uint32_t DEFAULT_TIMEOUT_MS = 2000;

struct DeviceState {
  bool ready = false;
  int cc_major = 0, cc_minor = 0, sms = 0;
  int pair_clusters = 0;  // CTA pairs of the 2-SM kernel that fit on the GPU at once
  int rb_blocks[2] = {0, 0};  // resident blocks per SM of the RMSNorm backward pass (without, with add)
  void* no_alloc_scratch = nullptr;  // device address of g_no_alloc_scratch
};

std::mutex g_mu;
DeviceState g_dev[128];

// Every table of static kernels (internal linkage: each copy of the library
// in a process keeps its own).
struct SpecTable {
  const ge::KernelSpec* specs;
  const int* n;
};
const SpecTable kSpecTables[] = {
    {ge::kSpecsForward, &ge::kNumSpecsForward}, {ge::kSpecsAux, &ge::kNumSpecsAux}, {ge::kSpecsFp8, &ge::kNumSpecsFp8},
    {ge::kSpecsCommon, &ge::kNumSpecsCommon}};
constexpr int kNumSpecTables = sizeof(kSpecTables) / sizeof(kSpecTables[0]);

// The interpreting kernels (any program); static ones come from the tables.
const void* const kDynamic1 = reinterpret_cast<const void*>(&ge::fused_gemm_epilogue_kernel<1, ge::DynamicProgram>);
const void* const kDynamic2 = reinterpret_cast<const void*>(&ge::fused_gemm_epilogue_kernel<2, ge::DynamicProgram>);

// Scratch of gemm_epi_run_no_alloc: the status words and row counters that
// gemm_epi_run keeps in the caller's workspace.  Every device that loads the
// library holds this array until the process exits.  On the host its name is
// only a stand-in; the kernel gets the address cudaGetSymbolAddress returns
// for the current device.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[GEMM_EPI_NO_ALLOC_SCRATCH_BYTES];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

gemm_epi_status device_state(DeviceState** out, int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 128) return fail(GEMM_EPI_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute");
    if (d.cc_major == 10 && d.cc_minor == 3) {
      // Every compiled kernel needs the large dynamic shared memory opt-in.
      e = cudaFuncSetAttribute(kDynamic1, cudaFuncAttributeMaxDynamicSharedMemorySize, ge::Smem<1>::BYTES);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kDynamic2, cudaFuncAttributeMaxDynamicSharedMemorySize, ge::Smem<2>::BYTES);
      for (int c = 0; c < 2 && e == cudaSuccess; ++c)
        e = cudaFuncSetAttribute(ge::kDynamicFp8[c], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 c == 0 ? ge::Smem<1>::BYTES : ge::Smem<2>::BYTES);
      for (int t = 0; t < kNumSpecTables && e == cudaSuccess; ++t) {
        const ge::KernelSpec* tab = kSpecTables[t].specs;
        const int n = *kSpecTables[t].n;
        for (int i = 0; i < n && e == cudaSuccess; ++i) {
          e = cudaFuncSetAttribute(tab[i].kernel_1sm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   ge::Smem<1>::BYTES);
          if (e == cudaSuccess)
            e = cudaFuncSetAttribute(tab[i].kernel_2sm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     ge::Smem<2>::BYTES);
        }
      }
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
      // How many CTA pairs the GPU holds at once (a persistent grid larger
      // than that would leave pairs waiting for others to finish).
      cudaLaunchConfig_t cfg;
      std::memset(&cfg, 0, sizeof cfg);
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = 2;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * d.sms, 1, 1);
      cfg.blockDim = dim3(ge::NUM_THREADS, 1, 1);
      cfg.dynamicSmemBytes = ge::Smem<2>::BYTES;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, kDynamic2, &cfg);
      if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters");
      d.pair_clusters = clusters;
      for (int add = 0; add < 2; ++add) {
        const void* k = add ? reinterpret_cast<const void*>(&ge::rmsnorm_bwd_kernel<true>)
                            : reinterpret_cast<const void*>(&ge::rmsnorm_bwd_kernel<false>);
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.rb_blocks[add], k, ge::RB_THREADS,
                                                          ge::rb_ring_bytes(add != 0));
        if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        d.rb_blocks[add] = std::max(1, d.rb_blocks[add]);
      }
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(GEMM_EPI_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
  }
  if (d.cc_major != 10 || d.cc_minor != 3)
    return fail(GEMM_EPI_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                d.cc_major, d.cc_minor);
  *out = &d;
  if (dev_out) *dev_out = dev;
  return GEMM_EPI_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D tiled map: x (contiguous), rows, batch.  `batch_bytes` == 0 means the
// operand is shared across the batch (a batch extent of 1).
gemm_epi_status make_map(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                         uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                         CUtensorMapSwizzle sw, CUtensorMapL2promotion l2, const char* what,
                         uint64_t batch = 1, uint64_t batch_bytes = 0) {
  if (batch_bytes == 0) {
    batch = 1;
    batch_bytes = row_bytes * (outer > 0 ? outer : 1);
  }
  cuuint64_t dims[3] = {inner, outer, batch};
  cuuint64_t strides[2] = {row_bytes, batch_bytes};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(GEMM_EPI_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, static_cast<int>(r));
  return GEMM_EPI_OK;
}

// 4-D map of an MN-major (K x N) bf16 operand: 64 columns, K rows, the
// 64-column blocks, batch.  A box of `blocks` blocks lands in shared memory as
// that many consecutive 64 x 64 boxes, the layout the 3-D map fills with one
// load per box.  Used only when N is a multiple of 64: a partial last block
// would read past column N inside its 64-column extent.
gemm_epi_status make_map_blocked(CUtensorMap* map, const void* base, uint64_t n, uint64_t k, uint64_t row_bytes,
                                 uint32_t blocks, const char* what, uint64_t batch, uint64_t batch_bytes) {
  if (batch_bytes == 0) {
    batch = 1;
    batch_bytes = row_bytes * (k > 0 ? k : 1);
  }
  cuuint64_t dims[4] = {64, k, n / 64, batch};
  cuuint64_t strides[3] = {row_bytes, 128, batch_bytes};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(ge::BLOCK_K), blocks, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(GEMM_EPI_ERR_CUDA, "cuTensorMapEncodeTiled(%s, blocked) failed with %d", what, static_cast<int>(r));
  return GEMM_EPI_OK;
}

// Ops that write an output buffer: each may appear once per program.
bool is_output_op(int c) {
  return c == GEMM_EPI_OP_AMAX || c == GEMM_EPI_OP_STORE_BF16 || c == GEMM_EPI_OP_STORE_E4M3 ||
         c == GEMM_EPI_OP_ROW_RMS_RSQRT || c == GEMM_EPI_OP_ROW_DOT || c == GEMM_EPI_OP_COL_SUM;
}

bool is_pre_pair_op(int c) {
  return c == GEMM_EPI_OP_SCALE_ALPHA || c == GEMM_EPI_OP_ADD_BIAS_COL || c == GEMM_EPI_OP_MUL_COL_SCALE ||
         c == GEMM_EPI_OP_MUL_ROW_SCALE ||
         c == GEMM_EPI_OP_ACT_GELU_TANH || c == GEMM_EPI_OP_ACT_RELU || c == GEMM_EPI_OP_ACT_SILU;
}

}  // namespace

struct gemm_epi_plan {
  gemm_epi_desc d;
  std::vector<gemm_epi_op> ops;
  int64_t n_out = 0;
  int pair_at = -1, pair_g = 1, pair_silu = 1;
  int expand_at = -1, expand_g = 1;  // DSWIGLU
  bool dual = false;  // GEMM_EPI_B_DUAL: B columns alternate with B2 in 128-column blocks
  bool in8 = false;   // 8-bit operands (kind::f8f6f4)
  int64_t batch = 1, row_blocks = 0;
  uint32_t flags = 0;
  bool uses_bias = false, uses_row_scale = false, uses_residual = false, uses_preact = false;
  bool uses_col_scale = false;
  float rms_eps = 0.0f;
  int rms_unrounded = 0;
  int64_t num_m_tiles = 0, num_n_tiles = 0;
  size_t ws_bytes = WS_HEADER;
  const ge::KernelSpec* spec = nullptr;  // compiled form of the program, or NULL
};

namespace {

gemm_epi_status validate(gemm_epi_plan& P) {
  const gemm_epi_desc& d = P.d;
  const int64_t LIM = 0x7FFFFFFF;
  if (d.M < 0 || d.N < 0 || d.K < 0 || d.M > LIM || d.N > LIM || d.K > LIM)
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "M, N, K must be in [0, 2^31)");
  const int b_base = d.b_layout & ~GEMM_EPI_B_DUAL;
  P.dual = (d.b_layout & GEMM_EPI_B_DUAL) != 0;
  if (b_base != GEMM_EPI_B_KN && b_base != GEMM_EPI_B_NK)
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "unknown b_layout %d", d.b_layout);
  if (P.dual && d.N % 256 != 0)
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "GEMM_EPI_B_DUAL needs N %% 256 == 0 (N=%lld)",
                static_cast<long long>(d.N));
  if (d.a_type < GEMM_EPI_TYPE_BF16 || d.a_type > GEMM_EPI_TYPE_E5M2 || d.b_type < GEMM_EPI_TYPE_BF16 ||
      d.b_type > GEMM_EPI_TYPE_E5M2)
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "unknown operand type (a_type %d, b_type %d)", d.a_type, d.b_type);
  P.in8 = d.a_type != GEMM_EPI_TYPE_BF16;
  if (P.in8 != (d.b_type != GEMM_EPI_TYPE_BF16))
    return fail(GEMM_EPI_ERR_UNSUPPORTED, "A and B must both be BF16 or both 8-bit");
  if (P.in8 && b_base != GEMM_EPI_B_NK)
    return fail(GEMM_EPI_ERR_UNSUPPORTED, "8-bit operands need B stored N x K (GEMM_EPI_B_NK)");
  if (d.n_ops < 0 || d.n_ops > GEMM_EPI_MAX_OPS)
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "n_ops must be in [0, %d]", GEMM_EPI_MAX_OPS);
  if (d.n_ops > 0 && !d.ops) return fail(GEMM_EPI_ERR_INVALID_VALUE, "ops is NULL");

  int seen[32] = {0};  // indexed by op code
  for (int i = 0; i < d.n_ops; ++i) {
    const gemm_epi_op& op = d.ops[i];
    if (op.code < GEMM_EPI_OP_SCALE_ALPHA || op.code > GEMM_EPI_OP_ROW_DOT)
      return fail(GEMM_EPI_ERR_INVALID_VALUE, "op %d: unknown code %d", i, op.code);
    if (is_output_op(op.code) && seen[op.code])
      return fail(GEMM_EPI_ERR_INVALID_VALUE, "op %d: output op %d appears twice", i, op.code);
    seen[op.code]++;
    switch (op.code) {
      case GEMM_EPI_OP_DSWIGLU: {
        if (P.pair_at >= 0 || P.expand_at >= 0)
          return fail(GEMM_EPI_ERR_INVALID_VALUE, "a program has at most one pair op");
        const int g = op.i0 == 0 ? 1 : op.i0;
        if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16)
          return fail(GEMM_EPI_ERR_INVALID_VALUE, "DSWIGLU group %d not in {1,2,4,8,16}", op.i0);
        if (P.dual) return fail(GEMM_EPI_ERR_UNSUPPORTED, "DSWIGLU with GEMM_EPI_B_DUAL");
        if (d.N % g != 0)
          return fail(GEMM_EPI_ERR_INVALID_VALUE, "DSWIGLU group %d needs N %% %d == 0", g, g);
        if (2 * d.N > 0x7FFFFFFF) return fail(GEMM_EPI_ERR_INVALID_VALUE, "DSWIGLU needs 2N < 2^31");
        for (int j = 0; j < i; ++j)
          if (!is_pre_pair_op(d.ops[j].code))
            return fail(GEMM_EPI_ERR_UNSUPPORTED, "op %d (code %d) before DSWIGLU is not supported", j,
                        d.ops[j].code);
        for (int j = i + 1; j < d.n_ops; ++j)
          if (d.ops[j].code == GEMM_EPI_OP_ADD_RESIDUAL || d.ops[j].code == GEMM_EPI_OP_MUL_GELU_TANH_GRAD)
            return fail(GEMM_EPI_ERR_UNSUPPORTED, "DSWIGLU reads preact; op %d would need a second "
                                                  "auxiliary tensor", j);
        P.expand_at = i;
        P.expand_g = g;
        P.uses_preact = true;
        break;
      }
      case GEMM_EPI_OP_PAIR_SWIGLU:
      case GEMM_EPI_OP_PAIR_MUL: {
        if (P.pair_at >= 0 || P.expand_at >= 0)
          return fail(GEMM_EPI_ERR_INVALID_VALUE, "a program has at most one pair op");
        int g = op.i0 == 0 ? 1 : op.i0;
        if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16 && g != 32 && g != 128)
          return fail(GEMM_EPI_ERR_INVALID_VALUE, "pair group %d not in {1,2,4,8,16,32,128}", op.i0);
        if (P.dual && g != 128)
          return fail(GEMM_EPI_ERR_INVALID_VALUE, "with GEMM_EPI_B_DUAL the pair group must be 128");
        if (d.N % (2 * g) != 0)
          return fail(GEMM_EPI_ERR_INVALID_VALUE, "PAIR_SWIGLU group %d needs N %% %d == 0 (N=%lld)", g,
                      2 * g, static_cast<long long>(d.N));
        for (int j = 0; j < i; ++j) {
          if (!is_pre_pair_op(d.ops[j].code))
            return fail(GEMM_EPI_ERR_UNSUPPORTED, "op %d (code %d) before a pair op is not supported", j,
                        d.ops[j].code);
          // Group 128 pairs columns 128 apart within a tile, so a column bias
          // before it would have to follow that layout; not offered.
          if (g == 128 && (d.ops[j].code == GEMM_EPI_OP_ADD_BIAS_COL || d.ops[j].code == GEMM_EPI_OP_MUL_COL_SCALE))
            return fail(GEMM_EPI_ERR_UNSUPPORTED, "a column vector before a pair op of group 128");
        }
        P.pair_at = i;
        P.pair_g = g;
        P.pair_silu = op.code == GEMM_EPI_OP_PAIR_SWIGLU ? 1 : 0;
        break;
      }
      case GEMM_EPI_OP_ROW_RMS_RSQRT:
        if (!(op.f0 >= 0.0f) || !std::isfinite(op.f0))
          return fail(GEMM_EPI_ERR_INVALID_VALUE, "ROW_RMS_RSQRT eps must be finite and >= 0");
        if (op.i0 != 0 && op.i0 != 1) return fail(GEMM_EPI_ERR_INVALID_VALUE, "ROW_RMS_RSQRT mode must be 0 or 1");
        P.rms_eps = op.f0;
        P.rms_unrounded = op.i0;
        P.flags |= ge::F_ROW | ge::F_RSQRT;
        break;
      case GEMM_EPI_OP_ROW_DOT:
        P.flags |= ge::F_ROW;
        P.uses_residual = true;
        break;
      case GEMM_EPI_OP_MUL_COL_SCALE: P.uses_col_scale = true; break;
      case GEMM_EPI_OP_ADD_BIAS_COL: P.uses_bias = true; break;
      case GEMM_EPI_OP_MUL_ROW_SCALE: P.uses_row_scale = true; break;
      case GEMM_EPI_OP_ADD_RESIDUAL: P.uses_residual = true; break;
      case GEMM_EPI_OP_MUL_GELU_TANH_GRAD: P.uses_preact = true; break;
      case GEMM_EPI_OP_AMAX: P.flags |= ge::F_AMAX; break;
      case GEMM_EPI_OP_STORE_BF16: P.flags |= ge::F_STORE; break;
      case GEMM_EPI_OP_STORE_E4M3: P.flags |= ge::F_E8; break;
      case GEMM_EPI_OP_COL_SUM: P.flags |= ge::F_COL; break;
      default: break;
    }
  }
  if (P.uses_residual && P.uses_preact)
    return fail(GEMM_EPI_ERR_UNSUPPORTED, "ops reading residual and ops reading preact in one program need two "
                                          "auxiliary tensors; this library reads one");
  if (P.uses_residual || P.uses_preact) P.flags |= ge::F_AUX;
  if (d.K == 0) P.flags |= ge::F_ZERO_ACC;
  P.n_out = P.pair_at >= 0 ? d.N / 2 : P.expand_at >= 0 ? 2 * d.N : d.N;
  if (seen[GEMM_EPI_OP_ROW_DOT] && seen[GEMM_EPI_OP_ROW_RMS_RSQRT])
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "ROW_DOT and ROW_RMS_RSQRT both write row_out");
  if ((P.flags & ge::F_RSQRT) && P.n_out == 0 && d.M > 0)
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "ROW_RMS_RSQRT over zero columns is undefined");

  // Strides: bounds first, then the 16-byte TMA rule.
  const bool kn = b_base == GEMM_EPI_B_KN;
  const int64_t b_cols = P.dual ? d.N / 2 : d.N;  // columns of each B operand
  // Operand elements per 16-byte group: 8 bf16 or 16 FP8.
  const int64_t op_group = P.in8 ? 16 : 8;
  if (d.K % op_group)  // the K tail of a TMA box is clipped in 16-byte groups
    return fail(GEMM_EPI_ERR_MISALIGNED, "K must be a multiple of %lld (got %lld)",
                static_cast<long long>(op_group), static_cast<long long>(d.K));
  if (d.K > 0) {  // A and B are not read when K == 0
    if (d.lda < d.K) return fail(GEMM_EPI_ERR_INVALID_VALUE, "lda < K");
    if (d.ldb < (kn ? b_cols : d.K) || d.ldb <= 0) return fail(GEMM_EPI_ERR_INVALID_VALUE, "ldb too small");
    if (d.lda % op_group || d.ldb % op_group)
      return fail(GEMM_EPI_ERR_MISALIGNED, "lda and ldb must be multiples of %lld", static_cast<long long>(op_group));
  }
  if ((P.flags & ge::F_STORE) && (d.ldc < P.n_out || d.ldc <= 0))
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "ldc < output columns");
  if ((P.flags & ge::F_E8) && (d.ldc8 < P.n_out || d.ldc8 <= 0))
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "ldc8 < output columns");
  if ((P.flags & ge::F_AUX) && (d.ld_aux < P.n_out || d.ld_aux <= 0))
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "ld_aux < output columns");
  if ((P.flags & ge::F_STORE) && d.ldc % 8) return fail(GEMM_EPI_ERR_MISALIGNED, "ldc must be a multiple of 8");
  if ((P.flags & ge::F_E8) && d.ldc8 % 16) return fail(GEMM_EPI_ERR_MISALIGNED, "ldc8 must be a multiple of 16");
  if ((P.flags & ge::F_AUX) && d.ld_aux % 8) return fail(GEMM_EPI_ERR_MISALIGNED, "ld_aux must be a multiple of 8");
  if (d.lda > (int64_t(1) << 38) || d.ldb > (int64_t(1) << 38) || d.ldc > (int64_t(1) << 38) ||
      d.ldc8 > (int64_t(1) << 39) || d.ld_aux > (int64_t(1) << 38))
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "row stride beyond the TMA limit");

  P.num_m_tiles = (d.M + ge::BLOCK_M - 1) / ge::BLOCK_M;
  P.num_n_tiles = (d.N + ge::BLOCK_N - 1) / ge::BLOCK_N;
  // Batch: 0 or 1 is a single problem; strides in elements (bytes for C8).
  P.batch = d.batch <= 1 ? 1 : d.batch;
  if (d.batch < 0 || P.batch > 65535) return fail(GEMM_EPI_ERR_INVALID_VALUE, "batch must be in [0, 65535]");
  if (P.batch > 1) {
    const int64_t b_rows = kn ? d.K : b_cols;
    auto bad_stride = [&](int64_t st, int64_t need, int64_t mult, bool may_share) {
      if (st == 0) return !may_share;
      return st < need || st % mult != 0;
    };
    if (d.K > 0 && (bad_stride(d.batch_stride_a, d.M * d.lda, op_group, true) ||
                    bad_stride(d.batch_stride_b, b_rows * d.ldb, op_group, true)))
      return fail(GEMM_EPI_ERR_INVALID_VALUE, "A / B batch strides must be 0 (shared) or span a whole "
                                              "operand, in multiples of 16 bytes");
    if ((P.flags & ge::F_STORE) && bad_stride(d.batch_stride_c, d.M * d.ldc, 8, false))
      return fail(GEMM_EPI_ERR_INVALID_VALUE, "batch_stride_c must span M x ldc, a multiple of 8");
    if ((P.flags & ge::F_E8) && bad_stride(d.batch_stride_c8, d.M * d.ldc8, 16, false))
      return fail(GEMM_EPI_ERR_INVALID_VALUE, "batch_stride_c8 must span M x ldc8, a multiple of 16");
    if ((P.flags & ge::F_AUX) && bad_stride(d.batch_stride_aux, d.M * d.ld_aux, 8, false))
      return fail(GEMM_EPI_ERR_INVALID_VALUE, "batch_stride_aux must span M x ld_aux, a multiple of 8");
  }
  if (P.num_m_tiles * P.num_n_tiles * P.batch > LIM) return fail(GEMM_EPI_ERR_INVALID_VALUE, "too many tiles");
  // One row counter per 128-row block, counted in whole 256-row tiles so
  // both main-loop shapes fit.
  const size_t row_blocks = static_cast<size_t>((d.M + 2 * ge::BLOCK_M - 1) / (2 * ge::BLOCK_M)) * 2;
  P.row_blocks = static_cast<int64_t>(row_blocks);
  P.ws_bytes = WS_HEADER + ((row_blocks * P.batch * 4 + 255) / 256) * 256;

  // A compiled kernel whose op list (and pair group) is exactly this one.
  P.spec = nullptr;
  for (int t = 0; t < kNumSpecTables && !P.spec; ++t) {
    const ge::KernelSpec* tab = kSpecTables[t].specs;
    const int n = *kSpecTables[t].n;
    for (int i = 0; i < n && !P.spec; ++i) {
      if (tab[i].n_ops != d.n_ops || tab[i].in8 != (P.in8 ? 1 : 0)) continue;
      bool same = true;
      for (int j = 0; j < d.n_ops && same; ++j) {
        const int c = d.ops[j].code;
        const bool pair = c == GEMM_EPI_OP_PAIR_SWIGLU || c == GEMM_EPI_OP_PAIR_MUL;
        const int enc = c | (pair ? P.pair_g << 8 : c == GEMM_EPI_OP_DSWIGLU ? P.expand_g << 8 : 0);
        same = enc == tab[i].ops[j];
      }
      if (same) P.spec = &tab[i];
    }
  }
  return GEMM_EPI_OK;
}

struct Launch {
  CUtensorMap ta, tb, tb2, tc, tc8;
  ge::KernelParams kp;
  int grid;
  int cg;              // CTAs per tile: 1 (128 x 256) or 2 (a CTA pair, 256 x 256)
  const void* kernel;  // static kernel of the plan's program, or the interpreting one
};

// 2-SM tiles unless the problem has a single 128-row block (then half of
// every pair would idle) or a test forces one shape.
int choose_cta_group(const gemm_epi_plan& P, const gemm_epi_args& a, const DeviceState& dev) {
  if (a.debug_flags & GEMM_EPI_DEBUG_FORCE_1SM) return 1;
  if (dev.pair_clusters <= 0) return 1;
  if (a.debug_flags & GEMM_EPI_DEBUG_FORCE_2SM) return 2;
  return P.d.M > ge::BLOCK_M ? 2 : 1;
}

// Fills the kernel parameters and tensor maps of one fused launch.  `c`/`ldc`
// may differ from the plan's (the unfused baseline stores the bare
// accumulator into its scratch buffer with a store-only program).
gemm_epi_status prepare(const gemm_epi_plan& P, const gemm_epi_args& a, const DeviceState& dev, Launch& L) {
  const gemm_epi_desc& d = P.d;
  std::memset(&L, 0, sizeof L);
  L.cg = choose_cta_group(P, a, dev);
  if (P.spec && !(a.debug_flags & GEMM_EPI_DEBUG_FORCE_INTERPRETER))
    L.kernel = L.cg == 2 ? P.spec->kernel_2sm : P.spec->kernel_1sm;
  else if (P.in8)
    L.kernel = ge::kDynamicFp8[L.cg == 2 ? 1 : 0];
  else
    L.kernel = L.cg == 2 ? kDynamic2 : kDynamic1;
  const int tile_m = ge::BLOCK_M * L.cg;
  ge::KernelParams& k = L.kp;
  k.M = static_cast<int32_t>(d.M);
  k.N = static_cast<int32_t>(d.N);
  k.K = static_cast<int32_t>(d.K);
  k.n_out = static_cast<int32_t>(P.n_out);
  k.n_al = static_cast<int32_t>(P.n_out / 8 * 8);
  k.n_al8 = static_cast<int32_t>(P.n_out / 16 * 16);
  k.num_m_tiles = static_cast<int32_t>((d.M + tile_m - 1) / tile_m);
  k.num_n_tiles = static_cast<int32_t>(P.num_n_tiles);
  k.num_tiles = k.num_m_tiles * k.num_n_tiles * static_cast<int32_t>(P.batch);
  k.a_batched = P.batch > 1 && d.batch_stride_a != 0;
  k.b_batched = P.batch > 1 && d.batch_stride_b != 0;
  k.row_blocks = static_cast<int32_t>(P.row_blocks);
  k.bs_c = P.batch > 1 ? d.batch_stride_c : 0;
  k.bs_c8 = P.batch > 1 ? d.batch_stride_c8 : 0;
  k.bs_aux = P.batch > 1 ? d.batch_stride_aux : 0;
  // A K block is one 128-byte swizzle row of each operand: 64 bf16 or 128
  // 8-bit elements.
  const int k_step = P.in8 ? 2 * ge::BLOCK_K : ge::BLOCK_K;
  k.num_k_blocks = static_cast<int32_t>((d.K + k_step - 1) / k_step);
  // Groups of 16 M tiles walked along N: a wave of 76 tile pairs then reads
  // ~16 A and ~5 B panels (256 x K each), which stay in L2 for the next wave
  // while K is small.  When they cannot stay (large K), every wave reads its
  // panels again, and groups of 8 make the wave's block of tiles squarer:
  // ~12 A + 10 B panels, 10-15% fewer DRAM bytes at the same time.
  const double panel_bytes = static_cast<double>(ge::BLOCK_N) * static_cast<double>(d.K) * (P.in8 ? 1.0 : 2.0);
  k.group_m = 21.0 * panel_bytes > L2_KEEP_BYTES ? DEFAULT_GROUP_M / 2 : DEFAULT_GROUP_M;
  k.b_kn = (d.b_layout & ~GEMM_EPI_B_DUAL) == GEMM_EPI_B_KN ? 1 : 0;
  k.dual = P.dual ? 1 : 0;
  // Instruction descriptor: D fp32 (bits 4-5), A and B formats (bits 7-9,
  // 10-12: bf16 = 1 for kind::f16; e4m3 = 0, e5m2 = 1 for kind::f8f6f4),
  // A K-major, B K- or MN-major (bit 16), N >> 3 (bits 17-22), M >> 4
  // (bits 24-28) with M = 128 per CTA of the group.
  auto fmt = [](int32_t t) -> uint32_t { return t == GEMM_EPI_TYPE_E4M3 ? 0u : 1u; };  // bf16 or e5m2: 1
  k.idesc = (1u << 4) | (fmt(d.a_type) << 7) | (fmt(d.b_type) << 10) | (k.b_kn ? (1u << 16) : 0u) |
            (static_cast<uint32_t>(ge::BLOCK_N >> 3) << 17) | (static_cast<uint32_t>(tile_m >> 4) << 24);
  k.flags = P.flags;
  if (a.a_scale_inv || a.b_scale_inv) k.flags |= ge::F_DEQ;
  k.a_scale_inv = a.a_scale_inv;
  k.b_scale_inv = a.b_scale_inv;
  k.n_ops = static_cast<int32_t>(P.ops.size());
  k.pair_at = P.pair_at;
  k.pair_g = P.pair_g;
  k.pair_silu = P.pair_silu;
  k.expand_at = P.expand_at;
  k.expand_g = P.expand_g;
  k.alpha = a.alpha;
  k.fp8_scale = a.fp8_scale;
  k.rms_eps = P.rms_eps;
  k.rms_unrounded = P.rms_unrounded;
  k.bias = a.bias;
  k.col_scale = a.col_scale;
  k.row_scale = a.row_scale;
  k.amax = a.amax;
  k.row_out = a.row_out;
  k.col_out = a.col_out;
  k.c = static_cast<uint16_t*>(a.C);
  k.c8 = static_cast<uint8_t*>(a.C8);
  k.ldc = d.ldc;
  k.ldc8 = d.ldc8;
  k.aux = static_cast<const uint16_t*>(P.uses_residual ? a.residual : a.preact);
  k.ld_aux = d.ld_aux;
  k.status = static_cast<uint32_t*>(a.workspace);
  k.row_counter = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.workspace) + WS_HEADER);
  k.timeout_ns = static_cast<uint64_t>(a.timeout_ms ? a.timeout_ms : DEFAULT_TIMEOUT_MS) * 1000000ull;
  k.debug_flags = a.debug_flags;
  for (size_t i = 0; i < P.ops.size(); ++i) {
    k.ops[i].code = P.ops[i].code;
    k.ops[i].i0 = P.ops[i].i0;
    k.ops[i].f0 = P.ops[i].f0;
  }
  if (L.cg == 2)
    L.grid = 2 * static_cast<int>(std::min<int64_t>(k.num_tiles, dev.pair_clusters));
  else
    L.grid = static_cast<int>(std::min<int64_t>(k.num_tiles, dev.sms));

  gemm_epi_status s;
  if (d.K > 0) {
    const CUtensorMapDataType op_dt = P.in8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int64_t esz = P.in8 ? 1 : 2;  // bytes per operand element
    s = make_map(&L.ta, op_dt, a.A, d.K, d.M, d.lda * esz, k_step, ge::BLOCK_M, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, "A", P.batch, k.a_batched ? d.batch_stride_a * esz : 0);
    if (s) return s;
    // Each B operand: N (or N/2 with B2) columns; K-major boxes hold the
    // rows one CTA stages from one operand.
    const int64_t b_cols = P.dual ? d.N / 2 : d.N;
    const uint32_t nk_rows = (P.dual || L.cg == 2) ? ge::BLOCK_N / 2 : ge::BLOCK_N;
    // One load per K block and operand fetches the 64-column boxes this CTA
    // stages from it: 2 (a CTA pair, or B and B2 apart) or 4.
    k.b_blk = (k.b_kn && b_cols % 64 == 0) ? 1 : 0;
    const uint32_t blk_boxes = (P.dual || L.cg == 2) ? 2u : 4u;
    for (int which = 0; which < (P.dual ? 2 : 1); ++which) {
      CUtensorMap* map = which == 0 ? &L.tb : &L.tb2;
      const void* base = which == 0 ? a.B : a.B2;
      if (k.b_blk)
        s = make_map_blocked(map, base, b_cols, d.K, d.ldb * 2, blk_boxes, which ? "B2" : "B", P.batch,
                             k.b_batched ? d.batch_stride_b * 2 : 0);
      else if (k.b_kn)
        s = make_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, b_cols, d.K, d.ldb * 2, 64, ge::BLOCK_K,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, which ? "B2" : "B", P.batch,
                     k.b_batched ? d.batch_stride_b * 2 : 0);
      else
        s = make_map(map, op_dt, base, d.K, b_cols, d.ldb * esz, k_step, nk_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, which ? "B2" : "B", P.batch,
                     k.b_batched ? d.batch_stride_b * esz : 0);
      if (s) return s;
    }
  }
  if ((P.flags & ge::F_STORE) && k.n_al > 0) {
    s = make_map(&L.tc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.C, k.n_al, d.M, d.ldc * 2, ge::CHUNK, 32,
                 CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, "C", P.batch, k.bs_c * 2);
    if (s) return s;
  }
  if ((P.flags & ge::F_E8) && k.n_al8 > 0) {
    s = make_map(&L.tc8, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.C8, k.n_al8, d.M, d.ldc8, ge::CHUNK, 32,
                 CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE, "C8", P.batch, k.bs_c8);
    if (s) return s;
  }
  return GEMM_EPI_OK;
}

gemm_epi_status check_args(const gemm_epi_plan& P, const gemm_epi_args& a) {
  const gemm_epi_desc& d = P.d;
  const bool work = d.M > 0 && P.n_out > 0;
  auto need = [&](const void* ptr, const char* name) -> gemm_epi_status {
    if (!ptr) return fail(GEMM_EPI_ERR_INVALID_VALUE, "%s is NULL but the program uses it", name);
    if (!aligned16(ptr)) return fail(GEMM_EPI_ERR_MISALIGNED, "%s is not 16-byte aligned", name);
    return GEMM_EPI_OK;
  };
  gemm_epi_status s;
  if (work && d.K > 0) {
    if ((s = need(a.A, "A")) || (s = need(a.B, "B"))) return s;
    if (P.dual && (s = need(a.B2, "B2"))) return s;
  }
  if (work) {
    if ((P.flags & ge::F_STORE) && (s = need(a.C, "C"))) return s;
    if ((P.flags & ge::F_E8) && (s = need(a.C8, "C8"))) return s;
    if (P.uses_bias && (s = need(a.bias, "bias"))) return s;
    if (P.uses_col_scale && (s = need(a.col_scale, "col_scale"))) return s;
    if (P.uses_row_scale && (s = need(a.row_scale, "row_scale"))) return s;
    if (P.uses_residual && (s = need(a.residual, "residual"))) return s;
    if (P.uses_preact && (s = need(a.preact, "preact"))) return s;
  }
  if ((P.flags & ge::F_AMAX) && (s = need(a.amax, "amax"))) return s;
  for (const float* sc : {a.a_scale_inv, a.b_scale_inv})
    if (sc && (reinterpret_cast<uintptr_t>(sc) & 3u))
      return fail(GEMM_EPI_ERR_MISALIGNED, "a_scale_inv / b_scale_inv must be 4-byte aligned");
  if ((P.flags & ge::F_ROW) && d.M > 0 && (s = need(a.row_out, "row_out"))) return s;
  if ((P.flags & ge::F_COL) && P.n_out > 0 && (s = need(a.col_out, "col_out"))) return s;
  if (!a.workspace || !aligned16(a.workspace) || a.workspace_bytes < P.ws_bytes)
    return fail(GEMM_EPI_ERR_WORKSPACE, "workspace must be 16-byte aligned and hold %zu bytes (got %zu)",
                P.ws_bytes, a.workspace ? a.workspace_bytes : static_cast<size_t>(0));
  return GEMM_EPI_OK;
}

// Zeroes what the kernels accumulate into: status words and row counters,
// amax, row sums, column sums.
gemm_epi_status clear_outputs(const gemm_epi_plan& P, const gemm_epi_args& a, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(a.workspace, 0, P.ws_bytes, st);
  if (e == cudaSuccess && (P.flags & ge::F_AMAX)) e = cudaMemsetAsync(a.amax, 0, sizeof(float), st);
  if (e == cudaSuccess && (P.flags & ge::F_ROW) && P.d.M > 0)
    e = cudaMemsetAsync(a.row_out, 0, sizeof(float) * P.d.M * P.batch, st);
  if (e == cudaSuccess && (P.flags & ge::F_COL) && P.n_out > 0)
    e = cudaMemsetAsync(a.col_out, 0, sizeof(float) * P.n_out * P.batch, st);
  return e == cudaSuccess ? GEMM_EPI_OK : cuda_fail(e, "cudaMemsetAsync");
}

gemm_epi_status launch_fused(const Launch& L, cudaStream_t st) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3(L.grid, 1, 1);
  cfg.blockDim = dim3(ge::NUM_THREADS, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr;  // lives until the launch below
  std::memset(&attr, 0, sizeof attr);
  if (L.cg == 2) {
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    cfg.dynamicSmemBytes = ge::Smem<2>::BYTES;
  } else {
    cfg.dynamicSmemBytes = ge::Smem<1>::BYTES;
  }
  void* params[] = {const_cast<CUtensorMap*>(&L.ta), const_cast<CUtensorMap*>(&L.tb),
                    const_cast<CUtensorMap*>(&L.tb2),
                    const_cast<CUtensorMap*>(&L.tc), const_cast<CUtensorMap*>(&L.tc8),
                    const_cast<ge::KernelParams*>(&L.kp)};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, L.kernel, params);
  return e == cudaSuccess ? GEMM_EPI_OK : cuda_fail(e, "launch of the fused kernel");
}

}  // namespace

extern "C" {

gemm_epi_status gemm_epi_create(gemm_epi_handle* out, const gemm_epi_desc* desc) {
  g_last_error.clear();
  if (!out || !desc) return fail(GEMM_EPI_ERR_INVALID_VALUE, "out and desc must not be NULL");
  gemm_epi_plan* P = new (std::nothrow) gemm_epi_plan();
  if (!P) return fail(GEMM_EPI_ERR_INVALID_VALUE, "out of host memory");
  P->d = *desc;
  if (desc->n_ops > 0 && desc->ops && desc->n_ops <= GEMM_EPI_MAX_OPS)
    P->ops.assign(desc->ops, desc->ops + desc->n_ops);
  P->d.ops = P->ops.data();
  gemm_epi_status s = validate(*P);
  if (s != GEMM_EPI_OK) {
    delete P;
    return s;
  }
  *out = P;
  return GEMM_EPI_OK;
}

gemm_epi_status gemm_epi_destroy(gemm_epi_handle h) {
  delete h;
  return GEMM_EPI_OK;
}

size_t gemm_epi_workspace_size(gemm_epi_handle h) { return h ? h->ws_bytes : 0; }

int64_t gemm_epi_out_cols(gemm_epi_handle h) { return h ? h->n_out : -1; }

gemm_epi_status gemm_epi_run(gemm_epi_handle h, const gemm_epi_args* args, void* stream) {
  g_last_error.clear();
  if (!h || !args) return fail(GEMM_EPI_ERR_INVALID_VALUE, "handle and args must not be NULL");
  gemm_epi_status s = check_args(*h, *args);  // host-only checks first
  if (s) return s;
  DeviceState* dev = nullptr;
  if ((s = device_state(&dev, nullptr))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = clear_outputs(*h, *args, st))) return s;
  if (h->d.M == 0 || h->n_out == 0) return GEMM_EPI_OK;
  Launch L;
  if ((s = prepare(*h, *args, *dev, L))) return s;
  return launch_fused(L, st);
}

gemm_epi_status gemm_epi_run_unfused(gemm_epi_handle h, const gemm_epi_args* args, void* scratch,
                                     int64_t ld_scratch, void* stream) {
  g_last_error.clear();
  if (!h || !args) return fail(GEMM_EPI_ERR_INVALID_VALUE, "handle and args must not be NULL");
  if (h->pair_at >= 0 && h->pair_g > 8)
    return fail(GEMM_EPI_ERR_UNSUPPORTED, "the separate pass handles pair groups up to 8");
  if (h->batch > 1) return fail(GEMM_EPI_ERR_UNSUPPORTED, "the separate pass runs single problems");
  if (h->expand_at >= 0 && h->expand_g > 4)
    return fail(GEMM_EPI_ERR_UNSUPPORTED, "the separate pass handles DSWIGLU groups up to 4");
  DeviceState* dev = nullptr;
  gemm_epi_status s = device_state(&dev, nullptr);
  if (s) return s;
  if ((s = check_args(*h, *args))) return s;
  const gemm_epi_desc& d = h->d;
  if (d.M > 0 && d.N > 0) {
    if (!scratch) return fail(GEMM_EPI_ERR_INVALID_VALUE, "scratch is NULL");
    if (!aligned16(scratch)) return fail(GEMM_EPI_ERR_MISALIGNED, "scratch is not 16-byte aligned");
    if (ld_scratch < d.N) return fail(GEMM_EPI_ERR_INVALID_VALUE, "ld_scratch < N");
    if (ld_scratch % 8) return fail(GEMM_EPI_ERR_MISALIGNED, "ld_scratch must be a multiple of 8");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = clear_outputs(*h, *args, st))) return s;
  if (d.M == 0 || h->n_out == 0) return GEMM_EPI_OK;

  // 1) bare GEMM: the same kernel with a store-only program into scratch.
  gemm_epi_plan bare;
  bare.d = d;
  bare.d.ldc = ld_scratch;
  bare.ops.push_back(gemm_epi_op{GEMM_EPI_OP_STORE_BF16, 0, 0.0f});
  bare.d.ops = bare.ops.data();
  bare.d.n_ops = 1;
  if ((s = validate(bare))) return s;
  gemm_epi_args ba = *args;
  ba.C = scratch;
  Launch L;
  if ((s = prepare(bare, ba, *dev, L))) return s;
  if ((s = launch_fused(L, st))) return s;

  // 2) the epilogue as a separate memory-bound pass over scratch.
  ge::UnfusedParams u;
  std::memset(&u, 0, sizeof u);
  u.M = static_cast<int32_t>(d.M);
  u.N = static_cast<int32_t>(d.N);
  u.n_out = static_cast<int32_t>(h->n_out);
  u.pair_at = h->pair_at;
  u.pair_g = h->pair_g;
  u.pair_silu = h->pair_silu;
  u.expand_at = h->expand_at;
  u.expand_g = h->expand_g;
  u.n_ops = static_cast<int32_t>(h->ops.size());
  u.flags = h->flags;
  u.alpha = args->alpha;
  u.fp8_scale = args->fp8_scale;
  u.rms_eps = h->rms_eps;
  u.rms_unrounded = h->rms_unrounded;
  u.acc = static_cast<const uint16_t*>(scratch);
  u.ld_acc = ld_scratch;
  u.aux = static_cast<const uint16_t*>(h->uses_residual ? args->residual : args->preact);
  u.ld_aux = d.ld_aux;
  u.bias = args->bias;
  u.col_scale = args->col_scale;
  u.row_scale = args->row_scale;
  u.c = static_cast<uint16_t*>(args->C);
  u.ldc = d.ldc;
  u.c8 = static_cast<uint8_t*>(args->C8);
  u.ldc8 = d.ldc8;
  u.amax = args->amax;
  u.row_out = args->row_out;
  u.col_out = args->col_out;
  for (size_t i = 0; i < h->ops.size(); ++i) {
    u.ops[i].code = h->ops[i].code;
    u.ops[i].i0 = h->ops[i].i0;
    u.ops[i].f0 = h->ops[i].f0;
  }
  dim3 grid(static_cast<unsigned>((h->n_out + ge::UF_COLS - 1) / ge::UF_COLS),
            static_cast<unsigned>((d.M + ge::UF_ROWS - 1) / ge::UF_ROWS));
  if (grid.y > 65535u) return fail(GEMM_EPI_ERR_UNSUPPORTED, "separate pass: M too large for its grid");
  // The program's compiled separate pass, else the interpreting one.
  const void* uk = (h->spec && h->spec->kernel_unfused && !(args->debug_flags & GEMM_EPI_DEBUG_FORCE_INTERPRETER))
                       ? h->spec->kernel_unfused
                       : reinterpret_cast<const void*>(&ge::unfused_epilogue_kernel<ge::DynamicProgram>);
  void* uargs[] = {&u};
  cudaError_t e = cudaLaunchKernel(uk, grid, dim3(ge::UF_THREADS), uargs, 0, st);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch of the separate epilogue pass");
  if ((h->flags & ge::F_ROW) && (h->flags & ge::F_RSQRT)) {
    const int threads = 256;
    ge::row_rms_finalize_kernel<<<static_cast<unsigned>((d.M + threads - 1) / threads), threads, 0, st>>>(
        args->row_out, static_cast<int>(d.M), 1.0f / static_cast<float>(h->n_out), h->rms_eps);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch of the row finalize kernel");
  }
  return GEMM_EPI_OK;
}

// Same launch as gemm_epi_run with the workspace replaced by the static
// scratch above.  The first call on a device looks up the scratch's address
// on that device (no allocation), so make it before any stream capture.
// Calls share the scratch and clear it on their stream before the kernel:
// calls whose kernels overlap on the GPU race on it.
gemm_epi_status gemm_epi_run_no_alloc(gemm_epi_handle h, const gemm_epi_args* args, void* stream) {
  g_last_error.clear();
  if (!h || !args) return fail(GEMM_EPI_ERR_INVALID_VALUE, "handle and args must not be NULL");
  DeviceState* dev = nullptr;
  int dev_id = 0;
  gemm_epi_status s = device_state(&dev, &dev_id);
  if (s) return s;
  if (h->ws_bytes > GEMM_EPI_NO_ALLOC_SCRATCH_BYTES) {
    // One 4-byte counter per 128-row block, M rounded up to 256 rows, per batch.
    const int64_t counters = static_cast<int64_t>((GEMM_EPI_NO_ALLOC_SCRATCH_BYTES - WS_HEADER) / 4);
    const int64_t max_m = counters / (2 * h->batch) * 2 * ge::BLOCK_M;
    return fail(GEMM_EPI_ERR_WORKSPACE,
                "this plan needs %zu bytes of scratch; the built-in scratch of gemm_epi_run_no_alloc "
                "holds %d: %lld row-block counters, ceil(M/256)*2*batch of them, so with batch %lld "
                "M is limited to %lld rows",
                h->ws_bytes, GEMM_EPI_NO_ALLOC_SCRATCH_BYTES, static_cast<long long>(counters),
                static_cast<long long>(h->batch), static_cast<long long>(max_m));
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!dev->no_alloc_scratch) {
      cudaError_t e = cudaGetSymbolAddress(&dev->no_alloc_scratch, g_no_alloc_scratch);
      if (e != cudaSuccess) {
        dev->no_alloc_scratch = nullptr;
        return cuda_fail(e, "cudaGetSymbolAddress of the built-in scratch");
      }
    }
    scratch = dev->no_alloc_scratch;
  }
  gemm_epi_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = GEMM_EPI_NO_ALLOC_SCRATCH_BYTES;
  if ((s = check_args(*h, a))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = clear_outputs(*h, a, st))) return s;
  if (h->d.M == 0 || h->n_out == 0) return GEMM_EPI_OK;
  Launch L;
  if ((s = prepare(*h, a, *dev, L))) return s;
  return launch_fused(L, st);
}

gemm_epi_status gemm_epi_rmsnorm_backward(const gemm_epi_rmsnorm_bwd_args* a, void* stream) {
  g_last_error.clear();
  if (!a) return fail(GEMM_EPI_ERR_INVALID_VALUE, "args must not be NULL");
  if (a->M < 0 || a->N < 0 || a->M > 0x7FFFFFFF || a->N > 0x7FFFFFFF)
    return fail(GEMM_EPI_ERR_INVALID_VALUE, "M, N must be in [0, 2^31)");
  gemm_epi_status s;
  if (a->dw && (reinterpret_cast<uintptr_t>(a->dw) & 3u))
    return fail(GEMM_EPI_ERR_MISALIGNED, "dw must be 4-byte aligned");
  const bool work = a->M > 0 && a->N > 0 && (a->dx || a->dw);
  auto tensor = [&](const void* ptr, int64_t ld, const char* name) -> gemm_epi_status {
    if (!ptr) return fail(GEMM_EPI_ERR_INVALID_VALUE, "%s is NULL", name);
    if (ld < a->N) return fail(GEMM_EPI_ERR_INVALID_VALUE, "row stride of %s < N", name);
    if (!aligned16(ptr) || ld % 8) return fail(GEMM_EPI_ERR_MISALIGNED, "%s: 16-byte base and stride needed", name);
    return GEMM_EPI_OK;
  };
  auto vec = [&](const float* ptr, const char* name) -> gemm_epi_status {
    if (!ptr) return fail(GEMM_EPI_ERR_INVALID_VALUE, "%s is NULL", name);
    if (reinterpret_cast<uintptr_t>(ptr) & 3u) return fail(GEMM_EPI_ERR_MISALIGNED, "%s must be 4-byte aligned", name);
    return GEMM_EPI_OK;
  };
  if (work) {
    if ((s = tensor(a->dy, a->ld_dy, "dy")) || (s = tensor(a->x, a->ld_x, "x")) || (s = vec(a->s, "s"))) return s;
    if (a->dx && ((s = tensor(a->dx, a->ld_dx, "dx")) || (s = vec(a->r, "r")))) return s;
    if (a->dx && a->add && (s = tensor(a->add, a->ld_add, "add"))) return s;
    if (a->w && (s = vec(a->w, "w"))) return s;
  }
  DeviceState* dev = nullptr;
  if ((s = device_state(&dev, nullptr))) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (a->dw && a->N > 0) {
    cudaError_t e = cudaMemsetAsync(a->dw, 0, sizeof(float) * a->N, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync of dw");
  }
  if (!work) return GEMM_EPI_OK;
  ge::RmsBwdParams p;
  p.M = static_cast<int32_t>(a->M);
  p.N = static_cast<int32_t>(a->N);
  p.dy = static_cast<const uint16_t*>(a->dy);
  p.ld_dy = a->ld_dy;
  p.x = static_cast<const uint16_t*>(a->x);
  p.ld_x = a->ld_x;
  p.add = a->dx ? static_cast<const uint16_t*>(a->add) : nullptr;
  p.ld_add = a->ld_add;
  p.w = a->w;
  p.s = a->s;
  p.r = a->r;
  p.dx = static_cast<uint16_t*>(a->dx);
  p.ld_dx = a->ld_dx;
  p.dw = a->dw;
  // One wave of resident blocks, striding over the rows.
  const bool add = p.add != nullptr;
  const int64_t col_blocks = (a->N + ge::RB_COLS - 1) / ge::RB_COLS;
  const int64_t want = std::max<int64_t>(1, static_cast<int64_t>(dev->rb_blocks[add]) * dev->sms / col_blocks);
  const int64_t row_blocks = std::min<int64_t>(want, (a->M + ge::RB_TY - 1) / ge::RB_TY);
  const dim3 grid(static_cast<unsigned>(col_blocks), static_cast<unsigned>(std::min<int64_t>(row_blocks, 65535)));
  const dim3 block(ge::RB_TX, ge::RB_TY);
  if (add)
    ge::rmsnorm_bwd_kernel<true><<<grid, block, ge::rb_ring_bytes(true), st>>>(p);
  else
    ge::rmsnorm_bwd_kernel<false><<<grid, block, ge::rb_ring_bytes(false), st>>>(p);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GEMM_EPI_OK : cuda_fail(e, "launch of the RMSNorm backward kernel");
}

gemm_epi_status gemm_epi_query_status(gemm_epi_handle h, const void* workspace, void* stream) {
  g_last_error.clear();
  if (!h || !workspace) return fail(GEMM_EPI_ERR_INVALID_VALUE, "handle and workspace must not be NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t words[4] = {0, 0, 0, 0};
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  e = cudaMemcpy(words, workspace, sizeof words, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy of the status words");
  if (words[0] & 1u)
    return fail(GEMM_EPI_ERR_TIMEOUT, "in-kernel wait ran out (site %u, block %u)%s", words[1], words[2],
                (words[0] & 2u) ? "; waiting for its operand loads to land also ran out" : "");
  return GEMM_EPI_OK;
}

const char* gemm_epi_status_string(gemm_epi_status s) {
  switch (s) {
    case GEMM_EPI_OK: return "ok";
    case GEMM_EPI_ERR_INVALID_VALUE: return "invalid value";
    case GEMM_EPI_ERR_MISALIGNED: return "misaligned pointer or stride";
    case GEMM_EPI_ERR_UNSUPPORTED: return "unsupported program";
    case GEMM_EPI_ERR_ARCH: return "unsupported device architecture";
    case GEMM_EPI_ERR_CUDA: return "CUDA error";
    case GEMM_EPI_ERR_TIMEOUT: return "in-kernel wait timed out";
    case GEMM_EPI_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char* gemm_epi_last_error(void) { return g_last_error.c_str(); }

int gemm_epi_version(void) { return GEMM_EPI_VERSION; }

}  // extern "C"
