// rmsnorm_bwd.cuh -- the second pass of the RMSNorm backward.
//
// For y = x * S * w with S[m] = 1/sqrt(mean_n x^2 + eps) ("Lean4-TileLang
// Tensor Program Superoptimizer", section 3 "RMSNorm") and upstream gradient
// dy, the GEMM that produced dy already reduced r[m] = sum_n w dy x in its
// epilogue (ROW_DOT; CODA's reductions on the output tile).  Every element of
// dx needs its row's r, so the rest is one memory-bound pass:
//   dx[m,n] = S[m] w[n] dy[m,n] - x[m,n] S[m]^3 r[m] / N  (+ add[m,n])
//   dw[n]   = sum_m dy[m,n] x[m,n] S[m]
//
// Work layout: a block is 32 x 8 threads; thread (tx, ty) covers 8
// consecutive columns (16-byte loads and stores, a warp = 512 contiguous
// bytes of one row) and rows ty, ty + 8, ... of the block's row stride.  The
// dw partial sums stay in registers over the rows, are combined across ty in
// shared memory and leave with one atomic per column per block.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace ge {

constexpr int RB_TX = 32;
constexpr int RB_TY = 8;
constexpr int RB_COLS = RB_TX * 8;  // columns per block

struct RmsBwdParams {
  int32_t M, N;
  const uint16_t* dy;
  int64_t ld_dy;
  const uint16_t* x;
  int64_t ld_x;
  const uint16_t* add;
  int64_t ld_add;
  const float* w;
  const float* s;
  const float* r;
  uint16_t* dx;
  int64_t ld_dx;
  float* dw;
};

__device__ __forceinline__ void rb_load8(const uint16_t* src, bool full, int valid, float (&v)[8]) {
  if (full) {
    const uint4 q = __ldg(reinterpret_cast<const uint4*>(src));
    const uint32_t ww[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[2 * h] = __uint_as_float(ww[h] << 16);
      v[2 * h + 1] = __uint_as_float(ww[h] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = j < valid ? __uint_as_float(static_cast<uint32_t>(src[j]) << 16) : 0.0f;
  }
}

__global__ void __launch_bounds__(RB_TX* RB_TY) rmsnorm_bwd_kernel(const __grid_constant__ RmsBwdParams p) {
  __shared__ float part[RB_TY][RB_COLS];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int c0 = blockIdx.x * RB_COLS + tx * 8;
  const int valid = min(8, p.N - c0);
  const bool active = valid > 0;
  const bool full = valid == 8;
  float wv[8], dwa[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    wv[j] = (p.w != nullptr && active && j < valid) ? __ldg(p.w + c0 + j) : 1.0f;
    dwa[j] = 0.0f;
  }
  const float inv_n = 1.0f / static_cast<float>(p.N);
  if (active) {
    for (int m = blockIdx.y * RB_TY + ty; m < p.M; m += gridDim.y * RB_TY) {
      const float sm = __ldg(p.s + m);
      float dy[8], x[8];
      rb_load8(p.dy + static_cast<int64_t>(m) * p.ld_dy + c0, full, valid, dy);
      rb_load8(p.x + static_cast<int64_t>(m) * p.ld_x + c0, full, valid, x);
      if (p.dx) {
        const float c = sm * sm * sm * __ldg(p.r + m) * inv_n;
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = fmaf(sm * wv[j], dy[j], -x[j] * c);
        if (p.add) {
          float a[8];
          rb_load8(p.add + static_cast<int64_t>(m) * p.ld_add + c0, full, valid, a);
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] += a[j];
        }
        uint16_t* dst = p.dx + static_cast<int64_t>(m) * p.ld_dx + c0;
        if (full) {
          uint4 q;
          q.x = ptx::pack_bf16x2(v[0], v[1]);
          q.y = ptx::pack_bf16x2(v[2], v[3]);
          q.z = ptx::pack_bf16x2(v[4], v[5]);
          q.w = ptx::pack_bf16x2(v[6], v[7]);
          *reinterpret_cast<uint4*>(dst) = q;
        } else {
          for (int j = 0; j < valid; ++j) dst[j] = static_cast<uint16_t>(ptx::pack_bf16x2(v[j], 0.0f) & 0xFFFFu);
        }
      }
      if (p.dw) {
#pragma unroll
        for (int j = 0; j < 8; ++j) dwa[j] = fmaf(dy[j] * x[j], sm, dwa[j]);
      }
    }
  }
  if (p.dw) {
#pragma unroll
    for (int j = 0; j < 8; ++j) part[ty][tx * 8 + j] = dwa[j];
    __syncthreads();
    // Thread (tx, ty) sums column tx * 8 + ty over the 8 row groups.
    const int col = tx * 8 + ty;
    float t = 0.0f;
#pragma unroll
    for (int k = 0; k < RB_TY; ++k) t += part[k][col];
    const int n = blockIdx.x * RB_COLS + col;
    if (n < p.N) atomicAdd(p.dw + n, t);
  }
}

}  // namespace ge
