// rmsnorm_bwd.cuh -- the second pass of the RMSNorm backward.
//
// For y = x * S * w with S[m] = 1/sqrt(mean_n x^2 + eps) ("Lean4-TileLang
// Tensor Program Superoptimizer", section 9 "RMSNorm") and upstream gradient
// dy, the GEMM that produced dy already reduced r[m] = sum_n w dy x in its
// epilogue (ROW_DOT; CODA's reductions on the output tile).  Every element of
// dx needs its row's r, so the rest is one memory-bound pass:
//   dx[m,n] = S[m] w[n] dy[m,n] - x[m,n] S[m]^3 r[m] / N  (+ add[m,n])
//   dw[n]   = sum_m dy[m,n] x[m,n] S[m]
//
// Work layout: a block is 32 x 8 threads; thread (tx, ty) covers 8
// consecutive columns (16-byte accesses, a warp = 512 contiguous bytes of one
// row) and rows ty, ty + 8 * gridDim.y, ...  Each thread keeps RB_DEPTH of
// its rows in flight: per-thread asynchronous copies (cp.async) put the dy, x
// (and add) segments of its next rows into shared-memory slots only it
// reads, so the loop has no block barrier and holds no row in registers while
// it waits.  The dw partial sums stay in registers over the rows, are
// combined across ty in shared memory and leave with one atomic per column
// per block.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace ge {

constexpr int RB_TX = 32;
constexpr int RB_TY = 8;
constexpr int RB_THREADS = RB_TX * RB_TY;
constexpr int RB_COLS = RB_TX * 8;   // columns per block
constexpr int RB_DEPTH = 3;          // rows in flight per thread
constexpr int RB_MIN_BLOCKS = 4;     // resident blocks per SM the register budget allows

// Dynamic shared memory of the kernel: RB_DEPTH slots of one 16-byte segment
// per tensor per thread.
constexpr int rb_ring_bytes(bool add) { return RB_DEPTH * (add ? 3 : 2) * RB_THREADS * 16; }

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

__device__ __forceinline__ void rb_unpack(const uint4 q, float (&v)[8]) {
  const uint32_t ww[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    v[2 * h] = __uint_as_float(ww[h] << 16);
    v[2 * h + 1] = __uint_as_float(ww[h] & 0xFFFF0000u);
  }
}

// ADD: dx also adds a third tensor (the residual branch's gradient).
template <bool ADD>
__global__ void __launch_bounds__(RB_THREADS, RB_MIN_BLOCKS) rmsnorm_bwd_kernel(const __grid_constant__ RmsBwdParams p) {
  constexpr int T = ADD ? 3 : 2;  // tensors read per row
  extern __shared__ uint4 rb_ring[];   // [RB_DEPTH][T][RB_THREADS]
  __shared__ float part[RB_TY][RB_COLS];
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int tid = ty * RB_TX + tx;
  const int c0 = blockIdx.x * RB_COLS + tx * 8;
  const int valid = min(8, p.N - c0);  // columns of this thread (<= 0: none)
  float wv[8], dwa[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    wv[j] = (p.w != nullptr && j < valid) ? __ldg(p.w + c0 + j) : 1.0f;
    dwa[j] = 0.0f;
  }
  if (valid > 0) {
    const uint32_t src_bytes = 2u * static_cast<uint32_t>(valid);
    const uint32_t ring = ptx::smem_addr(rb_ring) + static_cast<uint32_t>(tid) * 16u;
    const int stride = gridDim.y * RB_TY;
    const int m0 = blockIdx.y * RB_TY + ty;
    const float inv_n = 1.0f / static_cast<float>(p.N);
    // Slot (d, t) of this thread: ring + (d * T + t) * RB_THREADS * 16.
    auto fetch = [&](int d, int m) {
      const uint32_t slot = ring + static_cast<uint32_t>(d * T) * (RB_THREADS * 16u);
      ptx::cp_async16(slot, p.dy + static_cast<int64_t>(m) * p.ld_dy + c0, src_bytes);
      ptx::cp_async16(slot + RB_THREADS * 16u, p.x + static_cast<int64_t>(m) * p.ld_x + c0, src_bytes);
      if constexpr (ADD)
        ptx::cp_async16(slot + 2u * RB_THREADS * 16u, p.add + static_cast<int64_t>(m) * p.ld_add + c0, src_bytes);
    };
    // One copy group per row slot, empty past the last row, so that
    // "at most RB_DEPTH - 1 groups pending" always means "this row landed".
#pragma unroll
    for (int d = 0; d < RB_DEPTH; ++d) {
      const int m = m0 + d * stride;
      if (m < p.M) fetch(d, m);
      ptx::cp_async_commit();
    }
    int d = 0;
    for (int m = m0; m < p.M; m += stride) {
      const float sm = __ldg(p.s + m);
      const float rm = p.dx ? __ldg(p.r + m) : 0.0f;
      ptx::cp_async_wait<RB_DEPTH - 1>();
      float dy[8], x[8];
      rb_unpack(rb_ring[(d * T + 0) * RB_THREADS + tid], dy);
      rb_unpack(rb_ring[(d * T + 1) * RB_THREADS + tid], x);
      if (p.dx) {
        const float c = sm * sm * sm * rm * inv_n;
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = fmaf(sm * wv[j], dy[j], -x[j] * c);
        if constexpr (ADD) {
          float a[8];
          rb_unpack(rb_ring[(d * T + 2) * RB_THREADS + tid], a);
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] += a[j];
        }
        uint16_t* dst = p.dx + static_cast<int64_t>(m) * p.ld_dx + c0;
        if (valid == 8) {
          uint4 q;
          q.x = ptx::pack_bf16x2(v[0], v[1]);
          q.y = ptx::pack_bf16x2(v[2], v[3]);
          q.z = ptx::pack_bf16x2(v[4], v[5]);
          q.w = ptx::pack_bf16x2(v[6], v[7]);
          *reinterpret_cast<uint4*>(dst) = q;
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j < valid) dst[j] = static_cast<uint16_t>(ptx::pack_bf16x2(v[j], 0.0f) & 0xFFFFu);
        }
      }
      if (p.dw) {
#pragma unroll
        for (int j = 0; j < 8; ++j) dwa[j] = fmaf(dy[j] * x[j], sm, dwa[j]);
      }
      // The slot's values are in registers: refill it with the row
      // RB_DEPTH ahead (or commit an empty group).
      const int mn = m + RB_DEPTH * stride;
      if (mn < p.M) fetch(d, mn);
      ptx::cp_async_commit();
      d = d + 1 == RB_DEPTH ? 0 : d + 1;
    }
    ptx::cp_async_wait<0>();
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
