// unfused_kernel.cuh -- the separate-pass epilogue used as the unfused
// baseline: it reads a stored bf16 accumulator back from global memory and
// applies the same op program as the fused kernel.  This is the "write the
// intermediate, launch another kernel, read it back" pattern whose extra
// traffic the pages measure against (Superoptimizer, section 9 "RMSNorm":
// the second kernel re-reads what the first wrote; cuDNN Graph API tutorial:
// the baddbmm -> activation -> amax chain).
//
// Layout of the work: a 256-thread block covers 32 rows x 256 output columns;
// warp w takes rows w, w+8, w+16, w+24 of the block, lane l takes 8
// consecutive output columns (16-byte loads and stores, coalesced per warp).
//
// Like the fused kernel, the pass comes in two forms: compiled for one
// static program (the op dispatch, pair and expansion groups fold at compile
// time), and interpreting the op list of any other program.
#pragma once

#include "fused_kernel.cuh"

namespace ge {

constexpr int UF_ROWS = 32;
constexpr int UF_COLS = 256;
constexpr int UF_THREADS = 256;

struct UnfusedParams {
  int32_t M, N, n_out;
  int32_t pair_at, pair_g, n_ops;
  int32_t pair_silu;  // 1: SwiGLU pair, 0: plain product
  int32_t expand_at, expand_g;  // DSWIGLU (groups up to 4), or -1
  uint32_t flags;
  float alpha, fp8_scale, rms_eps;
  int32_t rms_unrounded;
  const uint16_t* acc;  // M x N bf16, row stride ld_acc
  int64_t ld_acc;
  const uint16_t* aux;  // residual or preact, row stride ld_aux
  int64_t ld_aux;
  const float* bias;
  const float* col_scale;
  const float* row_scale;
  uint16_t* c;
  int64_t ldc;
  uint8_t* c8;
  int64_t ldc8;
  float* amax;
  float* row_out;  // accumulates sums of squares; finalised by a second kernel
  float* col_out;
  EpiOpDev ops[GEMM_EPI_MAX_OPS];
};

__device__ __forceinline__ float bf16_bits_to_f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Point-wise op on 8 values whose columns are col0..col0+7 (< ncols checked).
// `code` is an int, or a std::integral_constant whose switch folds.
template <class CodeT>
__device__ __forceinline__ void uf_pointwise(CodeT code, float (&v)[8], const UnfusedParams& p, int col0, int ncols,
                                             float rs) {
  switch (static_cast<int>(code)) {
    case GEMM_EPI_OP_SCALE_ALPHA:
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] *= p.alpha;
      break;
    case GEMM_EPI_OP_ADD_BIAS_COL:
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (col0 + j < ncols) v[j] += __ldg(p.bias + col0 + j);
      break;
    case GEMM_EPI_OP_MUL_COL_SCALE:
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (col0 + j < ncols) v[j] *= __ldg(p.col_scale + col0 + j);
      break;
    case GEMM_EPI_OP_MUL_ROW_SCALE:
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] *= rs;
      break;
    case GEMM_EPI_OP_ACT_GELU_TANH:
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = gelu_tanh_f(v[j]);
      break;
    case GEMM_EPI_OP_ACT_RELU:
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = fmaxf(v[j], 0.0f);
      break;
    case GEMM_EPI_OP_ACT_SILU:
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = silu_f(v[j]);
      break;
    default:
      break;
  }
}

__device__ __forceinline__ void load8_bf16(const uint16_t* src, bool full, int valid, float (&v)[8]) {
  if (full) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(src));
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[2 * h] = __uint_as_float(ww[h] << 16);
      v[2 * h + 1] = __uint_as_float(ww[h] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = j < valid ? bf16_bits_to_f(src[j]) : 0.0f;
  }
}

// Runs f(std::integral_constant<int, code>) for the static program's ops
// [Begin, End), or f(code) for the interpreted ops [begin, end).
template <class Prog, int Begin, int End, class F>
__device__ __forceinline__ void uf_ops(const UnfusedParams& p, int begin, int end, F&& f) {
  if constexpr (Prog::is_static) {
    static_for<Begin, End>([&](auto I) { f(std::integral_constant<int, Prog::code_of(decltype(I)::value)>{}); });
  } else {
    for (int k = begin; k < end; ++k) f(p.ops[k].code);
  }
}

template <class Prog>
__global__ void __launch_bounds__(UF_THREADS)
    unfused_epilogue_kernel(const __grid_constant__ UnfusedParams p) {
  constexpr bool kStatic = Prog::is_static;
  // Positions of the pair / expanding op in a static program (0 if absent).
  constexpr int kPairAt = prog_pair_at<Prog>() < 0 ? 0 : prog_pair_at<Prog>();
  constexpr int kExpandAt = prog_expand_at<Prog>() < 0 ? 0 : prog_expand_at<Prog>();
  __shared__ float col_part[UF_THREADS / 32][UF_COLS];
  __shared__ uint32_t amax_part[UF_THREADS / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row_base = blockIdx.y * UF_ROWS;
  const int c0 = blockIdx.x * UF_COLS + lane * 8;  // first output column of this thread
  const int pair_at = kStatic ? prog_pair_at<Prog>() : p.pair_at;
  const int expand_at = kStatic ? prog_expand_at<Prog>() : p.expand_at;
  const bool paired = pair_at >= 0;
  const bool expand = expand_at >= 0;
  const int op_begin = paired ? pair_at + 1 : expand ? expand_at + 1 : 0;
  const int n_ops = kStatic ? prog_n<Prog>() : p.n_ops;
  const uint32_t flags = kStatic ? static_flags<Prog>() : p.flags;
  const int valid = min(8, p.n_out - c0);
  const bool full = valid == 8;

  uint32_t amax_bits = 0;
  float colacc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) colacc[j] = 0.0f;

  for (int i = 0; i < UF_ROWS / 8; ++i) {
    const int m = row_base + warp + 8 * i;
    if (m >= p.M || valid <= 0) continue;
    const float rs = p.row_scale ? __ldg(p.row_scale + m) : 0.0f;
    float v[8];
    float dh[4];  // DSWIGLU: the 4 accumulator columns c0/2.. of this thread's 8 outputs
    if (expand) {
      const int a0 = c0 / 2;
#pragma unroll
      for (int j = 0; j < 4; ++j) dh[j] = a0 + j < p.N ? bf16_bits_to_f(p.acc[m * p.ld_acc + a0 + j]) : 0.0f;
      uf_ops<Prog, 0, kExpandAt>(p, 0, expand_at, [&](auto code) {
        float h[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) h[j] = j < 4 ? dh[j] : 0.0f;
        uf_pointwise(code, h, p, a0, min(p.N, a0 + 4), rs);
#pragma unroll
        for (int j = 0; j < 4; ++j) dh[j] = h[j];
      });
    } else if (!paired) {
      load8_bf16(p.acc + m * p.ld_acc + c0, full, valid, v);
    } else {
      // 8 outputs need 16 accumulator columns starting at the pair block.
      float a[16];
      float lo[8], hi[8];
      const int a0 = 2 * c0;  // 8 outputs span 16 accumulator columns for any g <= 8
      const int avalid = min(16, p.N - a0);
      load8_bf16(p.acc + m * p.ld_acc + a0, avalid >= 8, max(0, min(8, avalid)), lo);
      load8_bf16(p.acc + m * p.ld_acc + a0 + 8, avalid >= 16, max(0, avalid - 8), hi);
      uf_ops<Prog, 0, kPairAt>(p, 0, pair_at, [&](auto code) {
        uf_pointwise(code, lo, p, a0, p.N, rs);
        uf_pointwise(code, hi, p, a0 + 8, p.N, rs);
      });
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        a[j] = lo[j];
        a[8 + j] = hi[j];
      }
      // Groups g <= 8 keep the pair inside these 16 columns (checked on the host).
      if constexpr (kStatic) {
        constexpr int g = prog_pair_g<Prog>();
        static_assert(g <= 8, "the separate pass handles pair groups up to 8");
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int gate = (j / g) * 2 * g + (j % g);
          v[j] = (prog_pair_silu<Prog>() ? silu_f(a[gate]) : a[gate]) * a[gate + g];
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int g = p.pair_g;
          const int gate = (j / g) * 2 * g + (j % g);
          float ga = 0.0f, ua = 0.0f;
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            if (q == gate) ga = a[q];
            if (q == gate + g) ua = a[q];
          }
          v[j] = (p.pair_silu ? silu_f(ga) : ga) * ua;
        }
      }
    }
    float x[8];
    if (flags & F_AUX) {
      load8_bf16(p.aux + m * p.ld_aux + c0, full, valid, x);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = 0.0f;
    }
    if (expand) {
      // Groups g <= 4 keep whole gate / up pairs inside these 8 outputs
      // (checked on the host).
      if constexpr (kStatic) {
        constexpr int g = prog_expand_g<Prog>();
        static_assert(g <= 4, "the separate pass handles DSWIGLU groups up to 4");
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int gate = (j / (2 * g)) * 2 * g + j % g;
          const int jl = (j / (2 * g)) * g + j % g;
          const float gt = x[gate], up = x[gate + g], d = dh[jl];
          const float sg = sigmoid_f(gt);
          v[j] = (j % (2 * g)) < g ? d * up * (sg * fmaf(gt, 1.0f - sg, 1.0f)) : d * (gt * sg);
        }
      } else {
        const int g = p.expand_g;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int gate = (j / (2 * g)) * 2 * g + j % g;
          const int jl = (j / (2 * g)) * g + j % g;
          float gt = 0.0f, up = 0.0f, d = 0.0f;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (q == gate) gt = x[q];
            if (q == gate + g) up = x[q];
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (q == jl) d = dh[q];
          const float sg = sigmoid_f(gt);
          v[j] = (j % (2 * g)) < g ? d * up * (sg * fmaf(gt, 1.0f - sg, 1.0f)) : d * (gt * sg);
        }
      }
    }
    float row_ss = 0.0f;
    auto run_op = [&](auto code) {
      switch (static_cast<int>(code)) {
        case GEMM_EPI_OP_ADD_RESIDUAL:
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] += x[j];
          break;
        case GEMM_EPI_OP_MUL_GELU_TANH_GRAD:
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] *= gelu_tanh_grad_f(x[j]);
          break;
        case GEMM_EPI_OP_AMAX:
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j < valid) amax_bits = max(amax_bits, __float_as_uint(fabsf(v[j])));
          break;
        case GEMM_EPI_OP_STORE_BF16: {
          uint16_t* dst = p.c + m * p.ldc + c0;
          if (full) {
            uint4 w;
            w.x = ptx::pack_bf16x2(v[0], v[1]);
            w.y = ptx::pack_bf16x2(v[2], v[3]);
            w.z = ptx::pack_bf16x2(v[4], v[5]);
            w.w = ptx::pack_bf16x2(v[6], v[7]);
            *reinterpret_cast<uint4*>(dst) = w;
          } else {
            for (int j = 0; j < valid; ++j) dst[j] = static_cast<uint16_t>(ptx::pack_bf16x2(v[j], 0.f));
          }
          break;
        }
        case GEMM_EPI_OP_STORE_E4M3: {
          uint8_t* dst = p.c8 + m * p.ldc8 + c0;
          uint32_t w[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t lo = ptx::pack_e4m3x2(v[4 * h] * p.fp8_scale, v[4 * h + 1] * p.fp8_scale);
            const uint32_t hi = ptx::pack_e4m3x2(v[4 * h + 2] * p.fp8_scale, v[4 * h + 3] * p.fp8_scale);
            w[h] = lo | (hi << 16);
          }
          if (full) {
            *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
          } else {
            for (int j = 0; j < valid; ++j) dst[j] = static_cast<uint8_t>(w[j / 4] >> (8 * (j % 4)));
          }
          break;
        }
        case GEMM_EPI_OP_ROW_DOT:
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j < valid) row_ss = fmaf(v[j], x[j], row_ss);
          break;
        case GEMM_EPI_OP_ROW_RMS_RSQRT:
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float u = p.rms_unrounded ? v[j] : bf16_round_f(v[j]);
            if (j < valid) row_ss = fmaf(u, u, row_ss);
          }
          break;
        case GEMM_EPI_OP_COL_SUM:
#pragma unroll
          for (int j = 0; j < 8; ++j) colacc[j] += v[j];
          break;
        default:
          uf_pointwise(code, v, p, c0, p.n_out, rs);
          break;
      }
    };
    uf_ops<Prog, prog_post_begin<Prog>(), prog_n<Prog>()>(p, op_begin, n_ops, run_op);
    if (flags & F_ROW) {
#pragma unroll
      for (int s = 16; s >= 1; s >>= 1) row_ss += __shfl_xor_sync(0xffffffffu, row_ss, s);
      if (lane == 0) atomicAdd(p.row_out + m, row_ss);
    }
  }

  if (flags & F_COL) {
#pragma unroll
    for (int j = 0; j < 8; ++j) col_part[warp][lane * 8 + j] = colacc[j];
    __syncthreads();
    const int col = blockIdx.x * UF_COLS + threadIdx.x;
    float s = 0.0f;
#pragma unroll
    for (int w = 0; w < UF_THREADS / 32; ++w) s += col_part[w][threadIdx.x];
    if (col < p.n_out) atomicAdd(p.col_out + col, s);
  }
  if (flags & F_AMAX) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, s));
    if (lane == 0) amax_part[warp] = amax_bits;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t b = 0;
      for (int w = 0; w < UF_THREADS / 32; ++w) b = max(b, amax_part[w]);
      if (b) atomicMax(reinterpret_cast<unsigned int*>(p.amax), b);
    }
  }
}

// The separate pass of a static program, or NULL where the pass does not
// cover the program (pair groups above 8, DSWIGLU groups above 4).
template <class Prog>
inline const void* unfused_kernel_for() {
  if constexpr (Prog::pair_at() >= 0 && Prog::pair_g() > 8) {
    return nullptr;
  } else if constexpr (Prog::expand_at() >= 0 && Prog::expand_g() > 4) {
    return nullptr;
  } else {
    return reinterpret_cast<const void*>(&unfused_epilogue_kernel<Prog>);
  }
}

// row_out[m] = 1 / sqrt(row_out[m] / n + eps) for the separate pass.
static __global__ void row_rms_finalize_kernel(float* row_out, int M, float inv_n, float eps) {
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m < M) row_out[m] = 1.0f / sqrtf(fmaf(row_out[m], inv_n, eps));
}

}  // namespace ge
