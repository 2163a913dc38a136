// fused_kernel.cuh -- persistent tcgen05 GEMM with the epilogue program
// finished on chip.
//
// What it computes: acc = A @ B on 128 x 256 output tiles ("Lean4-TileLang
// Tensor Program Superoptimizer", section 8 "Matmul": tiles staged through
// shared memory, a pipelined K loop, swizzled tile order, tensor cores), then
// the epilogue primitives of include/gemm_epi.h on each tile while it is still
// on chip ("CODA: ... GEMM-Epilogue", "How CODA works"; the TileLang
// tutorial's fused bias + GELU epilogue; the cuDNN Graph API tutorial's
// alpha / bias / activation / AMAX epilogue).
//
// How, on sm_103a:
//   warp 0      TMA producer: A (K-major, 128x64 box) and B (K-major 256x64
//               box, or four MN-major 64x64 boxes) into a ring of 128B-swizzled
//               shared-memory slots, one K-block each.  A stage (two slots on
//               the CTA-pair loop, one on the single-CTA loop) shares one
//               full barrier (mbarrier transaction counts); each slot has its
//               own empty barrier.
//   warp 1      allocates 512 TMEM columns (two 128x256 fp32 accumulators),
//               then one lane issues tcgen05.mma (N=256, K=16) and commits
//               each slot back to the producer and each finished
//               accumulator to the epilogue.
// Two main-loop shapes share the code (template parameter CG):
//   CG = 1  one CTA per 128 x 256 tile, M = 128 MMAs, 4 slots of 48 KB.
//   CG = 2  a cluster of two CTAs per 256 x 256 tile: each CTA stages its
//           128 rows of A and its 128 columns of B (6 slots of 32 KB), the
//           even CTA issues tcgen05.mma.cta_group::2 (M = 256) for the pair
//           and multicasts its commits to both CTAs; each CTA's epilogue
//           drains the 128 x 256 accumulator in its own TMEM.  Each SM then
//           stages a third less operand data per FLOP than with CG = 1.
//   warps 2..5  epilogue: warp w drains TMEM lanes 32*(w%4).. with
//               tcgen05.ld (thread = row, register = column), runs the op
//               program in registers, stages bf16 / e4m3 results in swizzled
//               shared memory and writes them with TMA stores.  Residual and
//               pre-activation rows are read straight into registers one
//               chunk ahead.
// The accumulator is double-buffered, so a tile's epilogue overlaps the next
// tile's main loop.  Tiles are walked persistently (grid = number of SMs) in
// groups of `group_m` M-tiles so that neighbouring CTAs share A and B in L2.
//
// Every mbarrier wait is bounded: when one runs out the CTA records a status
// in the workspace, raises a shared abort flag that every other wait checks,
// waits (bounded) for its copies and MMAs in flight -- the operand loads of
// both CTAs of a pair included -- frees TMEM and exits.
#pragma once

#include <stdint.h>

#include <type_traits>
#include <utility>

#include "gemm_epi.h"
#include "ptx.cuh"

namespace ge {

constexpr int BLOCK_M = 128;
constexpr int BLOCK_N = 256;
constexpr int BLOCK_K = 64;  // 64 bf16 = 128 bytes = one swizzle row (128 FP8 elements)
constexpr int UMMA_K = 16;   // bf16 elements per MMA = 32 bytes of a row (32 FP8 elements)
constexpr int NUM_EPI_WARPS = 4;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int CHUNK = 32;     // output columns per epilogue step
constexpr int EPI_BUFS = 3;   // bf16 output staging buffers per epilogue warp
constexpr int E8_BUFS = 2;    // e4m3 staging buffers per epilogue warp
constexpr uint32_t TMEM_COLS = 2 * BLOCK_N;

constexpr uint32_t A_KB_BYTES = BLOCK_M * BLOCK_K * 2;  // one K-block of A
constexpr uint32_t B_MN_BOX_BYTES = 64 * BLOCK_K * 2;  // one 64-column MN-major box
constexpr uint32_t EPI_BUF_BYTES = 32 * CHUNK * 2;     // 32 rows x 64 bytes
constexpr uint32_t E8_BUF_BYTES = 32 * CHUNK;          // 32 rows x 32 bytes
constexpr uint64_t DRAIN_LIMIT_NS = 20000000ull;       // bound of the abort-path drains

// Shared-memory map of one CTA when CG CTAs share a tile.
template <int CG>
struct Smem {
  // The operand ring holds SLOTS K-blocks.  A stage is KB_PER_STAGE
  // consecutive slots under one full barrier: the CTA pair's MMA warp waits
  // once per eight MMAs.  Each slot has its own empty barrier and is
  // refilled as soon as its four MMAs are done, which keeps the loads as far
  // ahead as with one K-block per stage.  The single-CTA loop runs the
  // memory-bound small-M problems and waits per K-block.
  static constexpr int SLOTS = CG == 1 ? 4 : 6;
  static constexpr int KB_PER_STAGE = CG == 2 ? 2 : 1;
  static constexpr int STAGES = SLOTS / KB_PER_STAGE;
  static constexpr int B_COLS = BLOCK_N / CG;  // B columns (N) this CTA stages
  static constexpr uint32_t B_KB_BYTES = B_COLS * BLOCK_K * 2;  // one K-block of B
  static constexpr uint32_t A_STAGE_BYTES = KB_PER_STAGE * A_KB_BYTES;
  static constexpr uint32_t B_STAGE_BYTES = KB_PER_STAGE * B_KB_BYTES;
  static constexpr uint32_t OFF_A = 0;
  static constexpr uint32_t OFF_B = OFF_A + STAGES * A_STAGE_BYTES;
  static constexpr uint32_t OFF_EPI = OFF_B + STAGES * B_STAGE_BYTES;
  static constexpr uint32_t OFF_E8 = OFF_EPI + NUM_EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_E8 + NUM_EPI_WARPS * E8_BUFS * E8_BUF_BYTES;
  static constexpr uint32_t BAR_FULL = 0;
  static constexpr uint32_t BAR_EMPTY = BAR_FULL + STAGES;
  static constexpr uint32_t BAR_TFULL = BAR_EMPTY + SLOTS;
  static constexpr uint32_t BAR_TEMPTY = BAR_TFULL + 2;
  static constexpr uint32_t BAR_DRAIN = BAR_TEMPTY + 2;
  static constexpr uint32_t NUM_BARS = BAR_DRAIN + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16 + 1024;  // + room to align the base to 1 KB
  static_assert(BYTES <= 232448, "shared memory budget of one CTA exceeded");
  static_assert(OFF_B % 1024 == 0 && OFF_EPI % 1024 == 0 && OFF_E8 % 1024 == 0,
                "operand and staging buffers must stay 1 KB aligned");
};

// Program flags derived on the host.
enum : uint32_t {
  F_AUX = 1u << 0,    // residual or preact tile is read
  F_STORE = 1u << 1,  // bf16 C is written
  F_E8 = 1u << 2,     // e4m3 C8 is written
  F_AMAX = 1u << 3,
  F_ROW = 1u << 4,
  F_COL = 1u << 5,
  F_ZERO_ACC = 1u << 6,  // K == 0: the accumulator is zero, TMEM is not read
  F_DEQ = 1u << 7,       // the accumulator is multiplied by the operands' dequantisation factors
  F_RSQRT = 1u << 8,     // row sums become 1/sqrt(mean + eps) (ROW_RMS_RSQRT; ROW_DOT keeps the sum)
};

// Where a bounded wait ran out (second status word).
enum : uint32_t {
  W_PRODUCER_EMPTY = 1,
  W_MMA_FULL = 2,
  W_MMA_TMEM_EMPTY = 3,
  W_EPI_TMEM_FULL = 4,
  W_DRAIN = 6,
};

struct EpiOpDev {
  int32_t code;
  int32_t i0;
  float f0;
};

struct KernelParams {
  int32_t M, N, K, n_out;
  // Output widths the TMA stores cover: n_out rounded down to whole 16-byte
  // groups (8 bf16 / 16 e4m3 columns).  The tensor unit clips a box at the
  // tensor edge in 16-byte groups, so the few columns of a ragged last group
  // are written with plain stores instead.
  int32_t n_al, n_al8;
  int32_t num_m_tiles, num_n_tiles, num_tiles, num_k_blocks;
  int32_t group_m;
  int32_t b_kn;  // 1: B stored K x N (MN-major operand)
  // 1: the MN-major B map is 4-D (64 columns, K, 64-column blocks, batch),
  // so one load fetches all of a K block's 64-column boxes of one operand
  int32_t b_blk;
  int32_t dual;  // 1: accumulator columns alternate between B and B2 in 128-column blocks
  int32_t a_batched, b_batched;  // operand advances with the batch (else shared)
  int32_t row_blocks;            // row counters per batch
  const float* a_scale_inv;      // dequantisation factors (F_DEQ), NULL = 1
  const float* b_scale_inv;
  int64_t bs_c, bs_c8, bs_aux;   // batch strides for direct accesses (elements; bytes for C8)
  uint32_t idesc;
  uint32_t flags;
  int32_t n_ops;
  int32_t pair_at;  // index of PAIR_SWIGLU in ops, or -1
  int32_t pair_g;
  int32_t pair_silu;  // 1: SwiGLU pair, 0: plain product
  int32_t expand_at;  // index of DSWIGLU in ops, or -1
  int32_t expand_g;   // its group
  float alpha, fp8_scale, rms_eps;
  int32_t rms_unrounded;
  const float* bias;
  const float* col_scale;
  const float* row_scale;
  float* amax;
  float* row_out;
  float* col_out;
  uint16_t* c;   // bf16 output (plain stores of a ragged last 16-byte group)
  uint8_t* c8;   // e4m3 output (ragged-tail stores)
  int64_t ldc, ldc8;
  const uint16_t* aux;  // residual or pre-activation (direct loads)
  int64_t ld_aux;
  uint32_t* status;       // workspace: [0] error bits, [1] where, [2] block
  uint32_t* row_counter;  // workspace: one arrival counter per 128-row block
  uint64_t timeout_ns;
  uint32_t debug_flags;
  EpiOpDev ops[GEMM_EPI_MAX_OPS];
};

// ------------------------------------------------------------------ programs
//
// The epilogue program reaches the kernel in one of two forms:
//  - DynamicProgram: the op list is read from KernelParams and interpreted
//    per 32-column chunk (any program create() accepts);
//  - StaticProgram<ops...>: the op codes are template arguments, so every
//    dispatch folds away and the kernel holds only the code of its own ops.
//    Each entry is code | (pair group << 8).  Per-call values (alpha, bias,
//    eps, ...) still come from KernelParams.
// The library compiles static forms of the programs it is benchmarked on and
// falls back to the interpreter for the rest; both run the same op bodies.

struct DynamicProgram {
  static constexpr bool is_static = false;
};

template <int... Ops>
struct StaticProgram {
  static constexpr bool is_static = true;
  static constexpr int n = sizeof...(Ops);
  static constexpr int code_of(int i) {
    constexpr int c[] = {Ops..., 0};
    return c[i] & 0xFF;
  }
  static constexpr int arg_of(int i) {
    constexpr int c[] = {Ops..., 0};
    return c[i] >> 8;
  }
  static constexpr int pair_at() {
    for (int i = 0; i < n; ++i)
      if (code_of(i) == GEMM_EPI_OP_PAIR_SWIGLU || code_of(i) == GEMM_EPI_OP_PAIR_MUL) return i;
    return -1;
  }
  static constexpr int pair_g() {
    return pair_at() < 0 ? 1 : (arg_of(pair_at()) == 0 ? 1 : arg_of(pair_at()));
  }
  static constexpr int expand_at() {
    for (int i = 0; i < n; ++i)
      if (code_of(i) == GEMM_EPI_OP_DSWIGLU) return i;
    return -1;
  }
  static constexpr int expand_g() {
    return expand_at() < 0 ? 1 : (arg_of(expand_at()) == 0 ? 1 : arg_of(expand_at()));
  }
  static constexpr bool has(int code) {
    for (int i = 0; i < n; ++i)
      if (code_of(i) == code) return true;
    return false;
  }
};

template <int Begin, class F, int... Is>
__device__ __forceinline__ void static_for_impl(F&& f, std::integer_sequence<int, Is...>) {
  (f(std::integral_constant<int, Begin + Is>{}), ...);
}

// f(integral_constant<int, i>) for i in [Begin, End), unrolled at compile time.
template <int Begin, int End, class F>
__device__ __forceinline__ void static_for(F&& f) {
  if constexpr (End > Begin) static_for_impl<Begin>(f, std::make_integer_sequence<int, End - Begin>{});
}

template <class Prog>
__host__ __device__ constexpr int prog_pair_at() {
  if constexpr (Prog::is_static) return Prog::pair_at(); else return -1;
}
template <class Prog>
__host__ __device__ constexpr int prog_pair_g() {
  if constexpr (Prog::is_static) return Prog::pair_g(); else return 1;
}
template <class Prog>
__host__ __device__ constexpr int prog_expand_at() {
  if constexpr (Prog::is_static) return Prog::expand_at(); else return -1;
}
template <class Prog>
__host__ __device__ constexpr int prog_expand_g() {
  if constexpr (Prog::is_static) return Prog::expand_g(); else return 1;
}
// First op applied to output columns: after the pair or expanding op.
template <class Prog>
__host__ __device__ constexpr int prog_post_begin() {
  if constexpr (Prog::is_static) {
    return Prog::pair_at() >= 0 ? Prog::pair_at() + 1 : Prog::expand_at() >= 0 ? Prog::expand_at() + 1 : 0;
  } else {
    return 0;
  }
}
template <class Prog>
__host__ __device__ constexpr bool prog_pair_silu() {
  if constexpr (Prog::is_static) {
    return Prog::pair_at() >= 0 && Prog::code_of(Prog::pair_at()) == GEMM_EPI_OP_PAIR_SWIGLU;
  } else {
    return true;
  }
}
template <class Prog>
__host__ __device__ constexpr int prog_n() {
  if constexpr (Prog::is_static) return Prog::n; else return 0;
}

// Flags a static program implies (F_ZERO_ACC stays a per-call flag).
template <class Prog>
__host__ __device__ constexpr uint32_t static_flags() {
  if constexpr (!Prog::is_static) {
    return 0u;
  } else {
    uint32_t f = 0;
    if (Prog::has(GEMM_EPI_OP_ADD_RESIDUAL) || Prog::has(GEMM_EPI_OP_MUL_GELU_TANH_GRAD) ||
        Prog::has(GEMM_EPI_OP_DSWIGLU) || Prog::has(GEMM_EPI_OP_ROW_DOT))
      f |= F_AUX;
    if (Prog::has(GEMM_EPI_OP_STORE_BF16)) f |= F_STORE;
    if (Prog::has(GEMM_EPI_OP_STORE_E4M3)) f |= F_E8;
    if (Prog::has(GEMM_EPI_OP_AMAX)) f |= F_AMAX;
    if (Prog::has(GEMM_EPI_OP_ROW_RMS_RSQRT)) f |= F_ROW | F_RSQRT;
    if (Prog::has(GEMM_EPI_OP_ROW_DOT)) f |= F_ROW;
    if (Prog::has(GEMM_EPI_OP_COL_SUM)) f |= F_COL;
    return f;
  }
}

// ------------------------------------------------------------------ helpers

// Tile t of the persistent walk: batch b, then groups of group_m M-tiles
// walked along N.
__device__ __forceinline__ void tile_coords(const KernelParams& p, int t, int& b, int& mb, int& nb) {
  const int per_batch = p.num_m_tiles * p.num_n_tiles;
  b = t / per_batch;
  t -= b * per_batch;
  const int per_group = p.group_m * p.num_n_tiles;
  const int g = t / per_group;
  const int first_m = g * p.group_m;
  const int gsz = min(p.num_m_tiles - first_m, p.group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gsz;
  nb = r / gsz;
}

template <int CG>
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                       const KernelParams& p, uint32_t where) {
  const uint64_t t0 = ptx::globaltimer_ns();
#pragma unroll 1
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ptx::mbar_test(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > p.timeout_ns) {
      *abort_flag = 1u;
      if (CG == 2) {  // the peer CTA stops waiting on this one too
        const uint32_t mine = ptx::smem_addr(const_cast<uint32_t*>(abort_flag));
        ptx::st_shared_cluster_u32(ptx::mapa_shared(mine, ptx::cluster_ctarank() ^ 1u), 1u);
      }
      if (atomicOr(p.status, 1u) == 0u) {
        p.status[1] = where;
        p.status[2] = blockIdx.x;
      }
      __threadfence();
      return false;
    }
  }
}

// Bounded wait for the phase of parity `parity` of mbarrier `bar`.
template <int CG>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         const KernelParams& p, uint32_t where) {
  if (ptx::mbar_test(bar, parity)) return true;
  return wait_slow<CG>(bar, parity, abort_flag, p, where);
}

// Short bounded wait used while draining after an abort (no flag check);
// false when the limit ran out first.
static __device__ __noinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
#pragma unroll 1
  while (!ptx::mbar_test(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Test hooks (first CTA, first tile): loads the producer leaves out so that
// a bounded wait runs out.  A skipped load is neither counted nor, for the
// first K-block of a stage, armed.
__device__ __forceinline__ bool skip_load_hook(uint32_t flags, int ks, int kb) {
  return ((flags & GEMM_EPI_DEBUG_SKIP_FIRST_LOAD) && ks == 0) ||
         ((flags & GEMM_EPI_DEBUG_SKIP_SECOND_LOAD) && kb == 1);
}

// Operand loads issued into one ring slot: a 2-bit count per slot (mod 4).
__device__ __forceinline__ uint32_t count_load(uint32_t cnt, uint32_t slot) {
  const uint32_t sh = 2u * slot;
  return (cnt & ~(3u << sh)) | ((((cnt >> sh) & 3u) + 1u) & 3u) << sh;
}

// After an abort: waits (bounded) until every operand load issued into this
// CTA group's shared memory has landed, so that no copy writes into shared
// memory after the group exits.  Runs in the CTA that owns the full
// barriers (the even CTA of a pair), once every role of both CTAs is done.
// `own` and `peer` hold the per-slot load counts of this CTA and of the odd
// CTA, whose loads complete on this CTA's barriers.  This CTA arms a stage's
// full barrier, for every slot of the stage in both CTAs, when it loads the
// stage's first slot, so that slot's count a0 is the number of phases armed.
// A slot is reloaded only after the pair's MMAs used it, which needed both
// CTAs' previous loads, and each CTA fills a stage's slots in order; so every
// count of the stage is a0 - 1, a0 or (odd CTA only) a0 + 1:
//   none at a0 + 1  phase a0 is the last one armed: the slots never loaded
//                   for it are counted as arrived, then it is waited for;
//   some at a0 + 1  the odd CTA loaded into a phase this CTA never armed:
//                   it is armed now, every slot not loaded for it counted
//                   as arrived, and waited for.
// Records status bit 1 when a wait ran out and, in status word 3, the stages
// settled each way (bits 0-7 and 8-15).
template <int CG, int STAGES, int KPS>
__device__ __noinline__ void drain_operand_loads(uint32_t bar_full0, uint32_t own, uint32_t peer,
                                                 uint32_t slot_bytes, uint32_t* status) {
  bool late = false;
  uint32_t settled = 0;
  constexpr uint32_t SLOTS_PER_PHASE = CG * KPS;  // slot loads one phase expects
#pragma unroll 1
  for (uint32_t s = 0; s < STAGES; ++s) {
    const uint32_t bar = bar_full0 + 8u * s;
    const uint32_t a0 = (own >> (2u * s * KPS)) & 3u;
    uint32_t at_a0 = 0, ahead = 0;
    bool uneven = false;
    for (uint32_t h = 0; h < KPS; ++h) {
      const uint32_t sh = 2u * (s * KPS + h);
      if (((own >> sh) & 3u) == a0) ++at_a0;
      if (CG == 2) {
        const uint32_t d = (((peer >> sh) & 3u) - a0) & 3u;
        if (d == 0u)
          ++at_a0;
        else if (d == 1u)
          ++ahead;
        else if (d == 2u)
          uneven = true;  // not reachable when the producers keep in step
      }
    }
    if (uneven) {
      late = true;
      continue;
    }
    uint32_t phases = a0;  // phases armed once settled (mod 4)
    if (ahead) {
      ptx::mbar_arrive_expect_tx(bar, SLOTS_PER_PHASE * slot_bytes);
      ptx::mbar_complete_tx(bar, (SLOTS_PER_PHASE - ahead) * slot_bytes);
      settled |= 1u << (8u + s);
      phases = a0 + 1u;
    } else if (at_a0 < SLOTS_PER_PHASE) {
      ptx::mbar_complete_tx(bar, (SLOTS_PER_PHASE - at_a0) * slot_bytes);
      settled |= 1u << s;
    }
    // The last phase armed has parity (phases - 1) & 1; with no load at all
    // that names the phase before the first, which tests complete.
    if (!drain_wait(bar, (phases + 1u) & 1u, DRAIN_LIMIT_NS)) late = true;
  }
  if (late) atomicOr(status, 2u);
  if (settled) atomicOr(status + 3, settled);
}

// tcgen05 shared-memory descriptor for a 128B-swizzled operand tile.
// K-major: rows of 128 bytes along K, 8-row groups SBO = 1024 bytes apart.
// MN-major: 64-element (128 B) rows along MN, 8 K-rows per 1024-byte group
// (SBO), successive 64-element MN blocks LBO bytes apart.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// ------------------------------------------------------------------ math

constexpr float LOG2E = 1.4426950408889634f;
// 2 * sqrt(2/pi) and that times 0.044715: 2u = x * (GELU_K0 + GELU_K1 x^2)
constexpr float GELU_K0 = 1.5957691216057308f;
constexpr float GELU_K1 = 1.5957691216057308f * 0.044715f;

// 1 / (1 + e^-z) with e^-z = 2^(-z log2 e), the exp2 form the Superoptimizer
// page uses for SiLU (section 7).
__device__ __forceinline__ float sigmoid_f(float z) {
  return ptx::rcp_approx(1.0f + ptx::ex2_approx(-z * LOG2E));
}

// GELU, tanh approximation, as x * sigmoid(2u).
__device__ __forceinline__ float gelu_tanh_f(float x) {
  return x * sigmoid_f(x * fmaf(GELU_K1, x * x, GELU_K0));
}

// d/dx of x * sigmoid(2u) = s + x s (1 - s) (2u)'.
__device__ __forceinline__ float gelu_tanh_grad_f(float x) {
  const float x2 = x * x;
  const float s = sigmoid_f(x * fmaf(GELU_K1, x2, GELU_K0));
  return fmaf(x * s * (1.0f - s), fmaf(3.0f * GELU_K1, x2, GELU_K0), s);
}

__device__ __forceinline__ float silu_f(float x) { return x * sigmoid_f(x); }

// ---- pairs of values in sm_100's packed fp32 arithmetic (f32x2 add, mul,
// fma: two lanes per instruction, each rounded like its scalar form); the
// special-function steps (ex2, rcp) stay scalar.

__device__ __forceinline__ float2 splat2(float c) { return make_float2(c, c); }

// 1 / (1 + 2^zl) of two values: the sigmoid of z for zl = -z log2 e.
__device__ __forceinline__ float2 sigmoid_from_neg_log2_f2(float2 zl) {
  const float2 d = __fadd2_rn(make_float2(ptx::ex2_approx(zl.x), ptx::ex2_approx(zl.y)), splat2(1.0f));
  return make_float2(ptx::rcp_approx(d.x), ptx::rcp_approx(d.y));
}

// sigmoid(2u) of GELU-tanh, 2u = x (GELU_K0 + GELU_K1 x^2), from x and x^2.
__device__ __forceinline__ float2 gelu_sigmoid_f2(float2 x, float2 x2) {
  const float2 zl = __fmul2_rn(x, __ffma2_rn(x2, splat2(-GELU_K1 * LOG2E), splat2(-GELU_K0 * LOG2E)));
  return sigmoid_from_neg_log2_f2(zl);
}

__device__ __forceinline__ float2 gelu_tanh_f2(float2 x) {
  return __fmul2_rn(x, gelu_sigmoid_f2(x, __fmul2_rn(x, x)));
}

// s + x s (1 - s) (2u)' of two values (the derivative above).
__device__ __forceinline__ float2 gelu_tanh_grad_f2(float2 x) {
  const float2 x2 = __fmul2_rn(x, x);
  const float2 s = gelu_sigmoid_f2(x, x2);
  const float2 t = __fmul2_rn(__fmul2_rn(x, s), __ffma2_rn(s, splat2(-1.0f), splat2(1.0f)));
  return __ffma2_rn(t, __ffma2_rn(x2, splat2(3.0f * GELU_K1), splat2(GELU_K0)), s);
}

__device__ __forceinline__ float2 silu_f2(float2 x) {
  return __fmul2_rn(x, sigmoid_from_neg_log2_f2(__fmul2_rn(x, splat2(-LOG2E))));
}

// v[2i], v[2i+1] <- f(pair i, i) for every pair of an even-length array.
template <int NV, class F>
__device__ __forceinline__ void for_pairs(float (&v)[NV], F&& f) {
#pragma unroll
  for (int i = 0; i < NV / 2; ++i) {
    const float2 r = f(make_float2(v[2 * i], v[2 * i + 1]), i);
    v[2 * i] = r.x;
    v[2 * i + 1] = r.y;
  }
}

__device__ __forceinline__ float bf16_round_f(float x) {
  const uint32_t h = ptx::pack_bf16x2(x, 0.0f) & 0xFFFFu;
  return __uint_as_float(h << 16);
}

// Internal op of compiled programs: SCALE_ALPHA directly followed by
// ADD_BIAS_COL, as one fused multiply-add (not a public op code).
constexpr int OP_ALPHA_THEN_BIAS = 0x70;

// Element-wise ops that may run on accumulator columns (before the pair op)
// or on output columns.  Columns of v[j]: col0 + j; `ncols` bounds the bias.
// `code` is an int, or a std::integral_constant whose switch folds away.
template <int NV, class CodeT>
__device__ __forceinline__ void apply_pointwise(CodeT code, float (&v)[NV], const KernelParams& p,
                                                int col0, int ncols, float row_scale_m) {
  switch (static_cast<int>(code)) {
    case GEMM_EPI_OP_SCALE_ALPHA: {
      const float2 a = splat2(p.alpha);
      for_pairs(v, [&](float2 y, int) { return __fmul2_rn(y, a); });
      break;
    }
    case OP_ALPHA_THEN_BIAS:
      if (col0 + NV <= ncols) {
        const float2 a = splat2(p.alpha);
        const float4* b4 = reinterpret_cast<const float4*>(p.bias + col0);
        for_pairs(v, [&](float2 y, int i) {
          const float4 b = __ldg(b4 + i / 2);
          return __ffma2_rn(y, a, (i & 1) ? make_float2(b.z, b.w) : make_float2(b.x, b.y));
        });
      } else {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          v[j] *= p.alpha;
          if (col0 + j < ncols) v[j] += __ldg(p.bias + col0 + j);
        }
      }
      break;
    case GEMM_EPI_OP_ADD_BIAS_COL:
      if (col0 + NV <= ncols) {
        const float4* b4 = reinterpret_cast<const float4*>(p.bias + col0);
        for_pairs(v, [&](float2 y, int i) {
          const float4 b = __ldg(b4 + i / 2);  // one 16-byte load per two pairs
          return __fadd2_rn(y, (i & 1) ? make_float2(b.z, b.w) : make_float2(b.x, b.y));
        });
      } else {
#pragma unroll
        for (int j = 0; j < NV; ++j)
          if (col0 + j < ncols) v[j] += __ldg(p.bias + col0 + j);
      }
      break;
    case GEMM_EPI_OP_MUL_COL_SCALE:
      if (col0 + NV <= ncols) {
        const float4* c4 = reinterpret_cast<const float4*>(p.col_scale + col0);
        for_pairs(v, [&](float2 y, int i) {
          const float4 c = __ldg(c4 + i / 2);
          return __fmul2_rn(y, (i & 1) ? make_float2(c.z, c.w) : make_float2(c.x, c.y));
        });
      } else {
#pragma unroll
        for (int j = 0; j < NV; ++j)
          if (col0 + j < ncols) v[j] *= __ldg(p.col_scale + col0 + j);
      }
      break;
    case GEMM_EPI_OP_MUL_ROW_SCALE: {
      const float2 r = splat2(row_scale_m);
      for_pairs(v, [&](float2 y, int) { return __fmul2_rn(y, r); });
      break;
    }
    case GEMM_EPI_OP_ACT_GELU_TANH:
      for_pairs(v, [&](float2 y, int) { return gelu_tanh_f2(y); });
      break;
    case GEMM_EPI_OP_ACT_RELU:
#pragma unroll
      for (int j = 0; j < NV; ++j) v[j] = fmaxf(v[j], 0.0f);
      break;
    case GEMM_EPI_OP_ACT_SILU:
      for_pairs(v, [&](float2 y, int) { return silu_f2(y); });
      break;
    default:
      break;
  }
}

// out[j] = silu(a[gate(j)]) * a[up(j)] (SwiGLU) or a[gate(j)] * a[up(j)]
// (the RMSNorm-MLP's plain product), gate(j) = (j/G)*2G + j%G, up = gate + G.
template <int G, bool SILU>
__device__ __forceinline__ void pair_combine_g(const float (&a)[64], float (&out)[32]) {
#pragma unroll
  for (int j = 0; j < 32; j += 2) {  // outputs j and j + 1 as one packed pair
    const int g0 = (j / G) * 2 * G + (j % G), g1 = ((j + 1) / G) * 2 * G + ((j + 1) % G);
    const float2 gate = make_float2(a[g0], a[g1]), up = make_float2(a[g0 + G], a[g1 + G]);
    const float2 r = __fmul2_rn(SILU ? silu_f2(gate) : gate, up);
    out[j] = r.x;
    out[j + 1] = r.y;
  }
}

template <bool SILU>
__device__ __forceinline__ void pair_combine_s(const float (&a)[64], float (&out)[32], int g) {
  switch (g) {
    case 2: pair_combine_g<2, SILU>(a, out); break;
    case 4: pair_combine_g<4, SILU>(a, out); break;
    case 8: pair_combine_g<8, SILU>(a, out); break;
    case 16: pair_combine_g<16, SILU>(a, out); break;
    case 32:
    case 128: pair_combine_g<32, SILU>(a, out); break;  // 128: the halves were loaded as 32 | 32
    default: pair_combine_g<1, SILU>(a, out); break;
  }
}

__device__ __forceinline__ void pair_combine(const float (&a)[64], float (&out)[32], int g, bool silu) {
  if (silu)
    pair_combine_s<true>(a, out, g);
  else
    pair_combine_s<false>(a, out, g);
}

// The SwiGLU backward on one 32-column output chunk: dh holds the 16
// accumulator columns the chunk's pairs come from, x the forward gate / up
// pre-activations at the chunk's output columns.  For h = silu(gate) * up,
// output gate(j) = dh[j] * up * silu'(gate), output up(j) = dh[j] * silu(gate),
// silu'(g) = s (1 + g (1 - s)), s = sigmoid(g); gate(j) = (j/G)*2G + j%G.
template <int G>
__device__ __forceinline__ void dswiglu_expand_g(const float (&dh)[16], const float (&x)[32], float (&out)[32]) {
#pragma unroll
  for (int j = 0; j < 16; j += 2) {  // pairs j and j + 1 as one packed pair
    const int g0 = (j / G) * 2 * G + (j % G), g1 = ((j + 1) / G) * 2 * G + ((j + 1) % G);
    const float2 gt = make_float2(x[g0], x[g1]), up = make_float2(x[g0 + G], x[g1 + G]);
    const float2 d = make_float2(dh[j], dh[j + 1]);
    const float2 s = sigmoid_from_neg_log2_f2(__fmul2_rn(gt, splat2(-LOG2E)));
    // silu'(g) = s (1 + g (1 - s)); silu(g) = g s
    const float2 one_minus_s = __ffma2_rn(s, splat2(-1.0f), splat2(1.0f));
    const float2 dsilu = __fmul2_rn(s, __ffma2_rn(gt, one_minus_s, splat2(1.0f)));
    const float2 og = __fmul2_rn(__fmul2_rn(d, up), dsilu);
    const float2 ou = __fmul2_rn(d, __fmul2_rn(gt, s));
    out[g0] = og.x;
    out[g1] = og.y;
    out[g0 + G] = ou.x;
    out[g1 + G] = ou.y;
  }
}

__device__ __forceinline__ void dswiglu_expand(const float (&dh)[16], const float (&x)[32], float (&out)[32], int g) {
  switch (g) {
    case 2: dswiglu_expand_g<2>(dh, x, out); break;
    case 4: dswiglu_expand_g<4>(dh, x, out); break;
    case 8: dswiglu_expand_g<8>(dh, x, out); break;
    case 16: dswiglu_expand_g<16>(dh, x, out); break;
    default: dswiglu_expand_g<1>(dh, x, out); break;
  }
}

// This thread's 32 auxiliary bf16 values of row m, columns col0.. (zeros
// outside the tensor), straight from global memory.
__device__ __forceinline__ void load_aux_row(uint4 (&w)[4], const KernelParams& p, const uint16_t* aux,
                                             int m, bool row_ok, int col0) {
  if (row_ok && col0 + 32 <= p.n_out) {
    const uint4* src = reinterpret_cast<const uint4*>(aux + static_cast<int64_t>(m) * p.ld_aux + col0);
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = __ldg(src + q);
  } else {
    uint32_t h[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int n = col0 + 2 * j;
      const uint16_t* rowp = aux + static_cast<int64_t>(m) * p.ld_aux;
      const uint32_t lo = (row_ok && n < p.n_out) ? rowp[n] : 0u;
      const uint32_t hi = (row_ok && n + 1 < p.n_out) ? rowp[n + 1] : 0u;
      h[j] = lo | (hi << 16);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
  }
}

// Lane l returns the sum over the warp's 32 lanes of x[l] (x is consumed).
__device__ __forceinline__ float warp_transpose_sum(float (&x)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = upper ? x[i] : x[i + s];
      const float keep = upper ? x[i + s] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return x[0];
}

// Column sums of a 32-row x 32-column chunk held thread = row: the chunk goes
// back into its own TMEM columns (`taddr`: lane quad base, first column) and
// returns in the MMA-fragment layout, where each thread holds 4 rows of 8
// columns.  After 3 in-thread adds per column, a transpose-reduce over the 8
// lanes that share lane % 4 (7 shuffles, where thread = row takes 31) leaves
// lane l with the sum of column 8 (g / 2) + 2 (l % 4) + (g % 2), g = l / 4,
// which is returned in `col`.
// Rows with row_ok false (past M) count as zero; `all_rows` (warp-uniform)
// says that the warp has none, so the chunk goes to TMEM unmasked.
__device__ __forceinline__ float tmem_column_sums(const float (&s)[32], bool row_ok, bool all_rows, uint32_t taddr,
                                                  int lane, int& col) {
  uint32_t w[32];
  if (all_rows) {
#pragma unroll
    for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(s[j]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) w[j] = row_ok ? __float_as_uint(s[j]) : 0u;
  }
  ptx::tmem_st32_sync(taddr, w);
  uint32_t a[16], b[16];
  ptx::tmem_ld16x256_x4_pair_sync(taddr, taddr + (16u << 16), a, b);
  // p[2i + e]: this thread's 4 rows of column 8i + 2 (lane % 4) + e
  float p[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 lo = __fadd2_rn(make_float2(__uint_as_float(a[4 * i]), __uint_as_float(a[4 * i + 1])),
                                 make_float2(__uint_as_float(a[4 * i + 2]), __uint_as_float(a[4 * i + 3])));
    const float2 hi = __fadd2_rn(make_float2(__uint_as_float(b[4 * i]), __uint_as_float(b[4 * i + 1])),
                                 make_float2(__uint_as_float(b[4 * i + 2]), __uint_as_float(b[4 * i + 3])));
    const float2 t = __fadd2_rn(lo, hi);
    p[2 * i] = t.x;
    p[2 * i + 1] = t.y;
  }
  // transpose-reduce over lane bits 4, 3, 2 (value index bits 2, 1, 0)
#pragma unroll
  for (int s2 = 4, m = 16; s2 >= 1; s2 >>= 1, m >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < s2; ++i) {
      const float send = upper ? p[i] : p[i + s2];
      const float keep = upper ? p[i + s2] : p[i];
      p[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
  const int g = lane >> 2;
  col = 8 * (g >> 1) + 2 * (lane & 3) + (g & 1);
  return p[0];
}

// ------------------------------------------------------------------ kernel

// IN8 = 1: 8-bit operands (tcgen05 kind::f8f6f4); a K block is still one
// 128-byte swizzle row per operand, now 128 elements.  The operand width is a
// compile-time choice: a kernel issues MMAs of one kind only.
template <int CG, class Prog, int IN8 = 0>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fused_gemm_epilogue_kernel(const __grid_constant__ CUtensorMap tm_a,
                               const __grid_constant__ CUtensorMap tm_b,
                               const __grid_constant__ CUtensorMap tm_b2,
                               const __grid_constant__ CUtensorMap tm_c,
                               const __grid_constant__ CUtensorMap tm_c8,
                               const __grid_constant__ KernelParams p) {
  using L = Smem<CG>;
  constexpr int STAGES = L::STAGES;
  constexpr int KPS = L::KB_PER_STAGE;
  constexpr int TILE_M = BLOCK_M * CG;  // rows of one tile (the whole CTA group)
  constexpr int K_STEP = IN8 ? 2 * BLOCK_K : BLOCK_K;  // K elements per K-block
  constexpr uint32_t BAR_FULL = L::BAR_FULL, BAR_EMPTY = L::BAR_EMPTY, BAR_TFULL = L::BAR_TFULL,
                     BAR_TEMPTY = L::BAR_TEMPTY, BAR_DRAIN = L::BAR_DRAIN;
  extern __shared__ uint8_t smem_raw[];
  // Same offset in both CTAs of a pair: the pair MMA addresses the peer's
  // operands and accumulator by this CTA's offsets.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  const uint32_t bar0 = sbase + L::OFF_BAR;
  auto bar = [&](uint32_t i) { return bar0 + 8u * i; };
  // misc[0] TMEM base, misc[1] abort flag, misc[2] the odd CTA's per-slot
  // load counts (written there by the odd CTA of a pair).
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;
  uint32_t load_cnt = 0;  // producer lane: operand loads issued per ring slot (2 bits each)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = CG == 2 ? ptx::cluster_ctarank() : 0u;  // CTA within the pair
  const int group = blockIdx.x / CG;                             // tile-walker index
  const int num_groups = gridDim.x / CG;

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < STAGES; ++s) ptx::mbar_init(bar(BAR_FULL + s), 1);
    for (uint32_t s = 0; s < L::SLOTS; ++s) ptx::mbar_init(bar(BAR_EMPTY + s), 1);
    for (uint32_t b = 0; b < 2; ++b) {
      ptx::mbar_init(bar(BAR_TFULL + b), 1);
      ptx::mbar_init(bar(BAR_TEMPTY + b), NUM_EPI_WARPS * CG);  // every epilogue warp of the group
    }
    ptx::mbar_init(bar(BAR_DRAIN), 1);
    *abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    if (CG == 2) {
      ptx::tmem_alloc_cg2(sbase + L::OFF_MISC, TMEM_COLS);
      ptx::tmem_relinquish_cg2();
    } else {
      ptx::tmem_alloc(sbase + L::OFF_MISC, TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0 && p.num_k_blocks > 0) {
    ptx::tma_prefetch_desc(&tm_a);
    ptx::tma_prefetch_desc(&tm_b);
  }
  ptx::tc_fence_before_sync();
  if (CG == 2)
    ptx::cluster_sync();  // the peer's barriers are initialised before anyone signals them
  else
    __syncthreads();
  ptx::tc_fence_after_sync();
  const uint32_t tmem_base = misc[0];

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0 && p.num_k_blocks > 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      const int num_steps = (p.num_k_blocks + KPS - 1) / KPS;  // stages per tile
      for (int t = group; ok && t < p.num_tiles; t += num_groups) {
        int bt, mb, nb;
        tile_coords(p, t, bt, mb, nb);
        const int za = p.a_batched ? bt : 0, zb = p.b_batched ? bt : 0;
        const int a_row = mb * TILE_M + rank * BLOCK_M;
        // B columns of this tile.  With two weight operands, tile nb covers
        // columns [nb*128, nb*128+128) of B (accumulator columns 0..127) and
        // the same columns of B2 (accumulator columns 128..255).
        const int b_col = p.dual ? nb * (BLOCK_N / 2) : nb * BLOCK_N + rank * L::B_COLS;
        const CUtensorMap* tmb_own = (p.dual && rank == 1) ? &tm_b2 : &tm_b;  // 2-SM: one operand per CTA
        const bool hooks = (p.debug_flags & (GEMM_EPI_DEBUG_SKIP_FIRST_LOAD | GEMM_EPI_DEBUG_SKIP_SECOND_LOAD)) &&
                           blockIdx.x == 0 && t == group;
        for (int ks = 0; ok && ks < num_steps; ++ks) {
          const uint32_t fb = bar(BAR_FULL + stage);
#pragma unroll
          for (int h = 0; h < KPS; ++h) {
            const uint32_t slot = stage * KPS + h;
            if (!wait_bar<CG>(bar(BAR_EMPTY + slot), phase ^ 1u, abort_flag, p, W_PRODUCER_EMPTY)) {
              ok = false;
              break;
            }
            if (hooks && skip_load_hook(p.debug_flags, ks, ks * KPS + h)) continue;
            if (h == 0) {
              // The stage's full barrier expects all of its slots; with a
              // CTA pair both CTAs' halves complete on the even CTA's.
              if (CG == 1)
                ptx::mbar_arrive_expect_tx(fb, L::A_STAGE_BYTES + L::B_STAGE_BYTES);
              else if (rank == 0)
                ptx::mbar_arrive_expect_tx(fb, 2u * (L::A_STAGE_BYTES + L::B_STAGE_BYTES));
            }
            // A slot past the last K-block (odd count) loads the last one
            // again, so that every stage carries the same bytes; its MMAs
            // are not issued.
            const int kb = min(ks * KPS + h, p.num_k_blocks - 1);
            const uint32_t sa = sbase + L::OFF_A + stage * L::A_STAGE_BYTES + h * A_KB_BYTES;
            const uint32_t sb = sbase + L::OFF_B + stage * L::B_STAGE_BYTES + h * L::B_KB_BYTES;
            if (CG == 1) {
              ptx::tma_load_3d(sa, &tm_a, fb, kb * K_STEP, a_row, za);
              if (p.b_kn && p.b_blk) {
                // with B2, blocks 0-1 come from B and 2-3 from B2
                ptx::tma_load_4d(sb, &tm_b, fb, 0, kb * BLOCK_K, b_col / 64, zb);
                if (p.dual) ptx::tma_load_4d(sb + 2 * B_MN_BOX_BYTES, &tm_b2, fb, 0, kb * BLOCK_K, b_col / 64, zb);
              } else if (p.b_kn) {
#pragma unroll
                for (int j = 0; j < L::B_COLS / 64; ++j) {
                  // with B2, boxes 0-1 come from B and 2-3 from B2
                  const bool second = p.dual && j >= 2;
                  const int col = p.dual ? b_col + (j & 1) * 64 : b_col + j * 64;
                  ptx::tma_load_3d(sb + j * B_MN_BOX_BYTES, second ? &tm_b2 : &tm_b, fb, col, kb * BLOCK_K, zb);
                }
              } else if (p.dual) {
                // two 128-row K-major boxes, one per operand, stacked in the slot
                ptx::tma_load_3d(sb, &tm_b, fb, kb * K_STEP, b_col, zb);
                ptx::tma_load_3d(sb + (BLOCK_N / 2) * BLOCK_K * 2, &tm_b2, fb, kb * K_STEP, b_col, zb);
              } else {
                ptx::tma_load_3d(sb, &tm_b, fb, kb * K_STEP, b_col, zb);
              }
            } else {
              const uint32_t fb0 = ptx::mapa_shared(fb, 0);
              ptx::tma_load_3d_cg2(sa, &tm_a, fb0, kb * K_STEP, a_row, za);
              if (p.b_kn && p.b_blk) {
                ptx::tma_load_4d_cg2(sb, tmb_own, fb0, 0, kb * BLOCK_K, b_col / 64, zb);
              } else if (p.b_kn) {
#pragma unroll
                for (int j = 0; j < L::B_COLS / 64; ++j)
                  ptx::tma_load_3d_cg2(sb + j * B_MN_BOX_BYTES, tmb_own, fb0, b_col + j * 64, kb * BLOCK_K, zb);
              } else {
                ptx::tma_load_3d_cg2(sb, tmb_own, fb0, kb * K_STEP, b_col, zb);
              }
            }
            load_cnt = count_load(load_cnt, slot);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (CG == 2 && rank == 1) {
        // This CTA's loads complete on the even CTA's barriers: its counts go
        // there for the abort drain (read after the cluster barrier below).
        ptx::st_shared_cluster_u32(ptx::mapa_shared(sbase + L::OFF_MISC + 8u, 0), load_cnt);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && rank == 0) {  // the even CTA issues for the whole group
      uint32_t stage = 0, phase = 0;
      bool ok = true, any_mma = false;
      const int num_steps = (p.num_k_blocks + KPS - 1) / KPS;
      int local = 0;
      for (int t = group; ok && t < p.num_tiles; t += num_groups, ++local) {
        const uint32_t buf = local & 1, use = local >> 1;
        if (!wait_bar<CG>(bar(BAR_TEMPTY + buf), (use & 1u) ^ 1u, abort_flag, p, W_MMA_TMEM_EMPTY)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after_sync();
        if (p.num_k_blocks == 0) {
          if (CG == 1) {
            ptx::mbar_arrive(bar(BAR_TFULL + buf));
          } else {
            ptx::mbar_arrive_cluster(ptx::mapa_shared(bar(BAR_TFULL + buf), 0));
            ptx::mbar_arrive_cluster(ptx::mapa_shared(bar(BAR_TFULL + buf), 1));
          }
          continue;
        }
        const uint32_t d_tmem = tmem_base + buf * BLOCK_N;
        for (int ks = 0; ks < num_steps; ++ks) {
          // Everything the stage's MMAs need but its data is computed before
          // the wait: the time from a completed barrier to the first MMA is
          // on the tensor pipe's critical path.  The descriptors of the
          // stage's first K block step by 32 bytes per MMA (K-major) or by 16
          // rows of 128 bytes (MN-major B); the address field counts 16 bytes.
          const uint64_t a_d0 = smem_desc_sw128(sbase + L::OFF_A + stage * L::A_STAGE_BYTES, 16, 1024);
          const uint64_t b_d0 =
              smem_desc_sw128(sbase + L::OFF_B + stage * L::B_STAGE_BYTES, p.b_kn ? B_MN_BOX_BYTES : 16u, 1024);
          const uint32_t b_k = p.b_kn ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
          const int kb_left = p.num_k_blocks - ks * KPS;  // K blocks of the tile from this stage on
          const uint32_t empty0 = bar(BAR_EMPTY + stage * KPS);
          if (!wait_bar<CG>(bar(BAR_FULL + stage), phase, abort_flag, p, W_MMA_FULL)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after_sync();
#pragma unroll
          for (int h = 0; h < KPS; ++h) {
            if (h < kb_left) {
              // Each MMA consumes 32 bytes of every operand row: 16 bf16 or 32
              // FP8 elements, so both kinds step through a K block the same way.
#pragma unroll
              for (int k = 0; k < BLOCK_K / UMMA_K; ++k) {
                const uint64_t ad = a_d0 + ((h * A_KB_BYTES + k * (UMMA_K * 2)) >> 4);
                const uint64_t bd = b_d0 + ((h * L::B_KB_BYTES) >> 4) + k * b_k;
                const uint32_t acc = (ks | h | k) != 0 ? 1u : 0u;
                if constexpr (CG == 1) {
                  if constexpr (IN8)
                    ptx::mma_f8_ss(d_tmem, ad, bd, p.idesc, acc);
                  else
                    ptx::mma_f16_ss(d_tmem, ad, bd, p.idesc, acc);
                } else {
                  if constexpr (IN8)
                    ptx::mma_f8_ss_cg2(d_tmem, ad, bd, p.idesc, acc);
                  else
                    ptx::mma_f16_ss_cg2(d_tmem, ad, bd, p.idesc, acc);
                }
              }
            }
            // the slot is free once its MMAs are done
            if (CG == 1)
              ptx::mma_commit(empty0 + 8u * h);
            else
              ptx::mma_commit_cg2_multicast(empty0 + 8u * h, 0x3);
          }
          any_mma = true;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (CG == 1)
          ptx::mma_commit(bar(BAR_TFULL + buf));
        else
          ptx::mma_commit_cg2_multicast(bar(BAR_TFULL + buf), 0x3);
      }
      if (any_mma) {
        // Every MMA this thread issued is complete before TMEM is released.
        if (CG == 1)
          ptx::mma_commit(bar(BAR_DRAIN));
        else
          ptx::mma_commit_cg2(bar(BAR_DRAIN));
        drain_wait(bar(BAR_DRAIN), 0, DRAIN_LIMIT_NS);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int ew = warp - 2;    // staging-buffer owner index 0..3
    const int quad = warp & 3;  // TMEM lane quadrant this warp may read
    constexpr bool kStatic = Prog::is_static;
    const int pair_at = kStatic ? prog_pair_at<Prog>() : p.pair_at;
    const bool paired = pair_at >= 0;
    const bool pair_g128 = paired && (kStatic ? prog_pair_g<Prog>() == 128 : p.pair_g == 128);
    // DSWIGLU expands: each 32-column output chunk comes from 16 accumulator
    // columns, so a tile has 2 * BLOCK_N output columns.
    const int expand_at = kStatic ? prog_expand_at<Prog>() : p.expand_at;
    const bool expand = expand_at >= 0;
    const int chunks = paired ? BLOCK_N / 64 : expand ? 2 * BLOCK_N / CHUNK : BLOCK_N / CHUNK;
    const int tile_out_cols = paired ? BLOCK_N / 2 : expand ? 2 * BLOCK_N : BLOCK_N;
    // A static program fixes every flag but the K == 0 one at compile time.
    const uint32_t flags = kStatic ? (p.flags & (F_ZERO_ACC | F_DEQ)) | static_flags<Prog>() : p.flags;
    // Product of the dequantisation factors, in fp32 (1 without F_DEQ).
    const float deq = (flags & F_DEQ) ? (p.a_scale_inv ? __ldg(p.a_scale_inv) : 1.0f) *
                                            (p.b_scale_inv ? __ldg(p.b_scale_inv) : 1.0f)
                                      : 1.0f;
    const uint32_t epi0 = sbase + L::OFF_EPI + ew * EPI_BUFS * EPI_BUF_BYTES;
    const uint32_t e80 = sbase + L::OFF_E8 + ew * E8_BUFS * E8_BUF_BYTES;
    uint8_t* epi0_ptr = smem + L::OFF_EPI + ew * EPI_BUFS * EPI_BUF_BYTES;
    uint8_t* e80_ptr = smem + L::OFF_E8 + ew * E8_BUFS * E8_BUF_BYTES;
    const int op_begin = paired ? pair_at + 1 : expand ? expand_at + 1 : 0;

    float amax_f = 0.0f;  // max |y| so far; a NaN sticks (NaN wins, as in the integer maximum below)
    uint32_t gchunk = 0;                 // this warp's running chunk number
    bool ok = true;
    int local = 0;


    for (int t = group; ok && t < p.num_tiles; t += num_groups, ++local) {
      int bt, mb, nb;
      tile_coords(p, t, bt, mb, nb);
      const int64_t row_base = static_cast<int64_t>(bt) * p.M;  // this batch's rows in row_scale / row_out
      const uint16_t* aux_b = p.aux ? p.aux + bt * p.bs_aux : nullptr;
      uint16_t* c_b = p.c ? p.c + bt * p.bs_c : nullptr;
      uint8_t* c8_b = p.c8 ? p.c8 + bt * p.bs_c8 : nullptr;
      float* col_b = p.col_out ? p.col_out + static_cast<int64_t>(bt) * p.n_out : nullptr;
      const int blk = mb * CG + static_cast<int>(rank);  // this CTA's 128-row block
      const int m = blk * BLOCK_M + quad * 32 + lane;
      const bool row_ok = m < p.M;
      const int slab_row0 = blk * BLOCK_M + quad * 32;
      const bool slab_ok = slab_row0 < p.M;
      const int n0 = nb * tile_out_cols;       // first output column of the tile
      const int nacc0 = nb * BLOCK_N;          // first accumulator column
      const uint32_t buf = local & 1, use = local >> 1;
      const float rs_m = (p.row_scale != nullptr && row_ok) ? __ldg(p.row_scale + row_base + m) : 0.0f;

      // Residual / pre-activation rows are read straight into registers,
      // one chunk ahead of their use (each thread reads its own row).
      uint4 xa[4];
      if (flags & F_AUX) load_aux_row(xa, p, aux_b, m, row_ok, n0);

      // All lanes wait; the outcome is made warp-uniform so that no lane
      // leaves while the others enter a warp-synchronous step.
      if (!__all_sync(0xffffffffu,
                      wait_bar<CG>(bar(BAR_TFULL + buf), use & 1u, abort_flag, p, W_EPI_TMEM_FULL))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after_sync();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + buf * BLOCK_N;
      float row_ss = 0.0f;

      for (int c = 0; c < chunks; ++c) {
        const uint32_t g = gchunk + c;
        const uint32_t eb = g % EPI_BUFS;
        const int col0 = n0 + c * CHUNK;  // first output column of the chunk
        float v[32];

        // ---- accumulator -> registers (and the pair op)
        float dh[16];  // DSWIGLU: the chunk's 16 accumulator columns after the ops before it
        if (expand) {
          if (flags & F_ZERO_ACC) {
#pragma unroll
            for (int j = 0; j < 16; ++j) dh[j] = 0.0f;
          } else {
            uint32_t r[16];
            ptx::tmem_ld16_sync(t_row + c * 16, r);
#pragma unroll
            for (int j = 0; j < 16; ++j) dh[j] = __uint_as_float(r[j]);
            if (flags & F_DEQ) {
#pragma unroll
              for (int j = 0; j < 16; ++j) dh[j] *= deq;
            }
          }
          if constexpr (kStatic) {
            static_for<0, (prog_expand_at<Prog>() < 0 ? 0 : prog_expand_at<Prog>())>([&](auto I) {
              apply_pointwise<16>(std::integral_constant<int, Prog::code_of(decltype(I)::value)>{}, dh, p,
                                  nacc0 + c * 16, p.N, rs_m);
            });
          } else {
            for (int i = 0; i < expand_at; ++i) apply_pointwise<16>(p.ops[i].code, dh, p, nacc0 + c * 16, p.N, rs_m);
          }
        } else if (!paired) {
          if (flags & F_ZERO_ACC) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.0f;
          } else {
            uint32_t r[32];
            ptx::tmem_ld32_sync(t_row + c * 32, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
            if (flags & F_DEQ) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] *= deq;
            }
          }
        } else {
          float a[64];
          if (flags & F_ZERO_ACC) {
#pragma unroll
            for (int j = 0; j < 64; ++j) a[j] = 0.0f;
          } else {
            uint32_t r[64];
            // Groups up to 32 pair within 64 adjacent columns; group 128
            // pairs column j of the tile's first half with j of its second.
            if (pair_g128)
              ptx::tmem_ld64_sync(t_row + c * 32, t_row + BLOCK_N / 2 + c * 32, r);
            else
              ptx::tmem_ld64_sync(t_row + c * 64, t_row + c * 64 + 32, r);
#pragma unroll
            for (int j = 0; j < 64; ++j) a[j] = __uint_as_float(r[j]);
            if (flags & F_DEQ) {
#pragma unroll
              for (int j = 0; j < 64; ++j) a[j] *= deq;
            }
          }
          if constexpr (kStatic) {
            static_for<0, (prog_pair_at<Prog>() < 0 ? 0 : prog_pair_at<Prog>())>([&](auto I) {
              apply_pointwise<64>(std::integral_constant<int, Prog::code_of(decltype(I)::value)>{}, a, p,
                                  nacc0 + c * 64, p.N, rs_m);
            });
            pair_combine_g<(prog_pair_g<Prog>() == 128 ? 32 : prog_pair_g<Prog>()), prog_pair_silu<Prog>()>(a, v);
          } else {
            for (int i = 0; i < pair_at; ++i)
              apply_pointwise<64>(p.ops[i].code, a, p, nacc0 + c * 64, p.N, rs_m);
            pair_combine(a, v, p.pair_g, p.pair_silu != 0);
          }
        }
        // The accumulator buffer is free for the next tile's MMAs once the last
        // chunk is read -- or, when column sums pass through the chunk's TMEM
        // columns, once the last chunk's sums are done (below).
        // (Compiled programs without a pair or expanding op, whose output
        // chunk c sits in accumulator columns 32c..32c+31; the interpreter
        // keeps the shuffle form, which needs no extra registers.)
        const bool tmem_col_sums = kStatic && (flags & F_COL) && !expand && !paired;
        auto release_accumulator = [&]() {
          ptx::tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) {
            if (CG == 1)
              ptx::mbar_arrive(bar(BAR_TEMPTY + buf));
            else
              ptx::mbar_arrive_cluster(ptx::mapa_shared(bar(BAR_TEMPTY + buf), 0));
          }
        };
        if (c == chunks - 1 && !tmem_col_sums) release_accumulator();

        // ---- auxiliary tile (residual / pre-activation), this thread's row
        float x[32];
        if (flags & F_AUX) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t ww[4] = {xa[q].x, xa[q].y, xa[q].z, xa[q].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              x[8 * q + 2 * h] = __uint_as_float(ww[h] << 16);
              x[8 * q + 2 * h + 1] = __uint_as_float(ww[h] & 0xFFFF0000u);
            }
          }
          if (c + 1 < chunks) load_aux_row(xa, p, aux_b, m, row_ok, n0 + (c + 1) * CHUNK);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = 0.0f;
        }
        if (expand) {  // x holds the forward gate / up pairs of the chunk's output columns
          if constexpr (kStatic)
            dswiglu_expand_g<prog_expand_g<Prog>()>(dh, x, v);
          else
            dswiglu_expand(dh, x, v, p.expand_g);
        }

        // ---- the op program on output columns
        const bool full_cols = col0 + 32 <= p.n_out;
        // The chunk's bf16 bits once STORE_BF16 has packed them: a compiled
        // program's ROW_RMS_RSQRT squares these instead of rounding again.
        uint32_t pk[16];
        bool packed = false;
        // One body per op; `code` is an int (interpreted program) or an
        // integral_constant (static program), for which the switch folds.
        auto run_op = [&](auto code) {
          switch (static_cast<int>(code)) {
            case GEMM_EPI_OP_ADD_RESIDUAL:
              for_pairs(v, [&](float2 y, int i) { return __fadd2_rn(y, make_float2(x[2 * i], x[2 * i + 1])); });
              packed = false;
              break;
            case GEMM_EPI_OP_MUL_GELU_TANH_GRAD:
              for_pairs(v, [&](float2 y, int i) {
                return __fmul2_rn(y, gelu_tanh_grad_f2(make_float2(x[2 * i], x[2 * i + 1])));
              });
              packed = false;
              break;
            case GEMM_EPI_OP_AMAX:
              if (row_ok) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (full_cols || col0 + j < p.n_out)
                    amax_f = ptx::max_abs_nan(amax_f, v[j]);
              }
              break;
            case GEMM_EPI_OP_STORE_BF16: {
              uint8_t* rowp = epi0_ptr + eb * EPI_BUF_BYTES + lane * 64;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint4 w;
                w.x = ptx::pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
                w.y = ptx::pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
                w.z = ptx::pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
                w.w = ptx::pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
                *reinterpret_cast<uint4*>(rowp + ((q ^ ((lane >> 1) & 3)) << 4)) = w;
                if constexpr (kStatic) {
                  pk[4 * q] = w.x;
                  pk[4 * q + 1] = w.y;
                  pk[4 * q + 2] = w.z;
                  pk[4 * q + 3] = w.w;
                }
              }
              packed = kStatic;
              if (col0 + 32 > p.n_al && row_ok) {  // ragged last 16-byte group
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const int n = col0 + j;
                  if (n >= p.n_al && n < p.n_out)
                    c_b[static_cast<int64_t>(m) * p.ldc + n] =
                        static_cast<uint16_t>(ptx::pack_bf16x2(v[j], 0.0f) & 0xFFFFu);
                }
              }
              break;
            }
            case GEMM_EPI_OP_STORE_E4M3: {
              const float s = p.fp8_scale;
              uint8_t* rowp = e80_ptr + (g % E8_BUFS) * E8_BUF_BYTES + lane * 32;
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                uint32_t w[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const int j = 16 * q + 4 * h;
                  const uint32_t lo = ptx::pack_e4m3x2(v[j] * s, v[j + 1] * s);
                  const uint32_t hi = ptx::pack_e4m3x2(v[j + 2] * s, v[j + 3] * s);
                  w[h] = lo | (hi << 16);
                }
                *reinterpret_cast<uint4*>(rowp + ((q ^ ((lane >> 2) & 1)) << 4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
              }
              if (col0 + 32 > p.n_al8 && row_ok) {  // ragged last 16-byte group
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const int n = col0 + j;
                  if (n >= p.n_al8 && n < p.n_out)
                    c8_b[static_cast<int64_t>(m) * p.ldc8 + n] =
                        static_cast<uint8_t>(ptx::pack_e4m3x2(v[j] * s, 0.0f) & 0xFFu);
                }
              }
              break;
            }
            case GEMM_EPI_OP_ROW_DOT:
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (full_cols || col0 + j < p.n_out) row_ss = fmaf(v[j], x[j], row_ss);
              break;
            case GEMM_EPI_OP_ROW_RMS_RSQRT:
              if (packed && full_cols && !p.rms_unrounded) {
                float2 ss = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                  const float2 u = make_float2(__uint_as_float(pk[h] << 16), __uint_as_float(pk[h] & 0xFFFF0000u));
                  ss = __ffma2_rn(u, u, ss);
                }
                row_ss += ss.x + ss.y;
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const float u = p.rms_unrounded ? v[j] : bf16_round_f(v[j]);
                  if (full_cols || col0 + j < p.n_out) row_ss = fmaf(u, u, row_ss);
                }
              }
              break;
            case GEMM_EPI_OP_COL_SUM: {
              if (!tmem_col_sums) {
                float s[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) s[j] = row_ok ? v[j] : 0.0f;
                const float tot = warp_transpose_sum(s, lane);
                if (slab_ok && col0 + lane < p.n_out) atomicAdd(col_b + col0 + lane, tot);
              } else {
                // The chunk's own accumulator columns (already read) hold it.
                int cj;
                const float tot = tmem_column_sums(v, row_ok, slab_row0 + 32 <= p.M, t_row + c * 32, lane, cj);
                if (slab_ok && col0 + cj < p.n_out) atomicAdd(col_b + col0 + cj, tot);
              }
              break;
            }
            default:
              apply_pointwise<32>(code, v, p, col0, p.n_out, rs_m);
              packed = false;  // the values changed after any earlier store
              break;
          }
        };
        if constexpr (kStatic) {
          static_for<prog_post_begin<Prog>(), prog_n<Prog>()>([&](auto I) {
            constexpr int i = decltype(I)::value;
            constexpr int code = Prog::code_of(i);
            constexpr bool bias_next = i + 1 < prog_n<Prog>() && Prog::code_of(i + 1) == GEMM_EPI_OP_ADD_BIAS_COL;
            constexpr bool alpha_before = i > prog_post_begin<Prog>() && Prog::code_of(i - 1) == GEMM_EPI_OP_SCALE_ALPHA;
            if constexpr (code == GEMM_EPI_OP_SCALE_ALPHA && bias_next)
              run_op(std::integral_constant<int, OP_ALPHA_THEN_BIAS>{});
            else if constexpr (!(code == GEMM_EPI_OP_ADD_BIAS_COL && alpha_before))  // else folded in above
              run_op(std::integral_constant<int, code>{});
          });
        } else {
          for (int i = op_begin; i < p.n_ops; ++i) run_op(p.ops[i].code);
        }
        if (c == chunks - 1 && tmem_col_sums) release_accumulator();

        // ---- TMA stores of this chunk's staged outputs
        if (flags & (F_STORE | F_E8)) {
          ptx::fence_proxy_async_smem();  // generic smem writes before the async-proxy reads
          __syncwarp();
          if (lane == 0) {
            const bool st_c = slab_ok && (flags & F_STORE) && col0 < p.n_al;
            const bool st_8 = slab_ok && (flags & F_E8) && col0 < p.n_al8;
            if (st_c) ptx::tma_store_3d(&tm_c, epi0 + eb * EPI_BUF_BYTES, col0, slab_row0, bt);
            if (st_8) ptx::tma_store_3d(&tm_c8, e80 + (g % E8_BUFS) * E8_BUF_BYTES, col0, slab_row0, bt);
            // At most the group of this chunk stays in flight, so the next
            // chunk's buffers are free.  A chunk without stores commits no
            // group and waits for every earlier read instead: a chunk past
            // the output edge must not count as the group that frees a buffer.
            if (st_c || st_8) {
              ptx::bulk_commit_group();
              ptx::bulk_wait_group_read<1>();
            } else {
              ptx::bulk_wait_group_read<0>();
            }
          }
        }
        __syncwarp();
      }
      if (!ok) break;
      gchunk += chunks;

      // ---- row statistics: partial sums, then the last arriving warp of
      // this row block turns them into 1/sqrt(mean + eps).
      if ((flags & F_ROW) && !(flags & F_RSQRT)) {
        // ROW_DOT: the partial sums are the result.
        if (row_ok) atomicAdd(p.row_out + row_base + m, row_ss);
      } else if (flags & F_ROW) {
        if (row_ok) atomicAdd(p.row_out + row_base + m, row_ss);
        __threadfence();
        __syncwarp();
        uint32_t prev = 0;
        if (lane == 0) prev = atomicAdd(p.row_counter + static_cast<int64_t>(bt) * p.row_blocks + blk, 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == static_cast<uint32_t>(NUM_EPI_WARPS * p.num_n_tiles - 1)) {
          __threadfence();
          const float inv_n = 1.0f / static_cast<float>(p.n_out);
          for (int r = lane; r < BLOCK_M; r += 32) {
            const int mm = blk * BLOCK_M + r;
            if (mm < p.M) {
              const float ss = __ldcg(p.row_out + row_base + mm);
              p.row_out[row_base + mm] = 1.0f / sqrtf(fmaf(ss, inv_n, p.rms_eps));
            }
          }
        }
      }
    }

    // ---- teardown of the epilogue warp
    if (lane == 0) ptx::bulk_wait_group<0>();
    if (flags & F_AMAX) {
      // Non-negative floats order like their bit patterns, and NaN's bits
      // exceed infinity's: one integer maximum across the warp and the grid.
      uint32_t amax_bits = __float_as_uint(amax_f);
#pragma unroll
      for (int s = 16; s >= 1; s >>= 1) amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, s));
      if (lane == 0 && amax_bits != 0u) atomicMax(reinterpret_cast<unsigned int*>(p.amax), amax_bits);
    }
  }

  __syncwarp();  // role branches reconverge before the warp-aligned barrier
  ptx::tc_fence_before_sync();
  // Every role of the group has finished: any abort flag is set by now, and
  // the odd CTA's load counts are visible to the even CTA.
  if (CG == 2)
    ptx::cluster_sync();
  else
    __syncthreads();
  if (threadIdx.x == 0 && rank == 0 && *abort_flag && p.num_k_blocks > 0)
    drain_operand_loads<CG, STAGES, KPS>(bar(BAR_FULL), load_cnt, CG == 2 ? misc[2] : 0u,
                                         A_KB_BYTES + L::B_KB_BYTES, p.status);
  __syncwarp();
  if (CG == 2)
    ptx::cluster_sync();  // no CTA of the pair releases TMEM or smem the other still uses
  else
    __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after_sync();
    if (CG == 2)
      ptx::tmem_dealloc_cg2(tmem_base, TMEM_COLS);
    else
      ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace ge
