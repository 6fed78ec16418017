// attn_bwd_tc.cu — causal GQA flash-attention backward on tcgen05 / TMEM.
//
// The backward of the attention core of one rank's local heads ([Grasp-TP]
// §4; [Troverld] §I.O: the backward recomputes QKᵀ from the saved log-sum-
// exp; [hjcheng-TP] Attention 单卡backward: dP = dO·Vᵀ, dV = Pᵀ·dO, dS from
// the softmax backward, dQ = dS·K, dK = dSᵀ·Q).
//
//   pre-pass  D = rowsum(dO ∘ O) and LSE·log2e per (batch, head, position),
//             padded with zeros to a multiple of 128 positions.
//   dK, dV    CTA = 128 keys of one (batch, kv head); per q head of the GQA
//             group and block of 128 queries at or after the keys
//               Sᵀ = K·Qᵀ, then dPᵀ = V·dOᵀ      (M=128, N=128, K=128) → TMEM
//               Pᵀ = exp2(Sᵀ·c − LSE·log2e), dSᵀ = Pᵀ ⊙ (dPᵀ − D)
//               dV += Pᵀ·dO,  dK += dSᵀ·Q        (M=128, N=128, K=128) → TMEM
//             K and V sit in TMEM as the A operands; Sᵀ and dPᵀ of a block
//             take turns in one 128-column TMEM buffer, which leaves room
//             for both accumulators.  Each dSᵀ tile (fp16, 32 KB) also goes
//             out to global memory with one bulk copy, in the swizzled
//             layout the tensor cores read.
//   dQ        a persistent streaming GEMM over those tiles: per (batch, q
//             head, block of 128 queries) dQ = Σ_kb dS_kb·K_kb over the key
//             blocks at or before it (M=128, N=128, K=128 per tile; dSᵀ is
//             the M-major A operand, K the N-major B), two TMEM accumulators
//             so the epilogue of one block overlaps the next.
// Computing dQ from the stored dS instead of recomputing S and dP per query
// block moves 2·32 KB of HBM traffic per 128×128 block pair (the tile out,
// then back in) in place of two of the seven products of the backward; the
// dQ kernel is bound by reading the tiles.
// dK/dV: warp 0 TMA (+ one thread for the dSᵀ copies), warp 1 TMEM
// allocation + single-thread MMA issue, warps 2–9 elementwise (two threads
// per TMEM lane, half of the columns each).  The MMAs go in the order
// Sᵀ(i), dK(i−1), dPᵀ(i), dV(i): the score products of a block are issued as
// soon as the elementwise warps have copied the previous contents of X to
// registers, and dK(i−1) keeps the tensor cores busy while they copy Sᵀ(i)
// out, so the tensor cores work while the elementwise warps do.  The elementwise loops are unrolled but
// branch-free (masks come from padding and a fix-up of the causal diagonal
// on packed words): a per-block body that outgrows the instruction cache
// runs several times slower.  Q and dO stream through rings of their own,
// each tile freed by the last MMA that reads it.  A tcgen05.mma of M=128
// costs about the same for N=64 as for N=128, so the wider blocks do twice
// the work per instruction.  No atomics: reruns are bit-identical, and the
// GQA sums of dK, dV stay inside one CTA.
// Operands fp16, accumulation fp32; dQ, dK, dV are written in bf16.
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cstring>

#include "attention.h"
#include "common.cuh"
#include "gemm.h"
#include "profile.h"

namespace tp {
namespace {

constexpr int HD = 128;
constexpr int A128 = 128 * 128;   // one 64-column half of a 128-row tile
constexpr int THREADS = 320;
constexpr uint32_t TMEM_COLS = 512;
constexpr float LOG2E_F = 1.4426950408889634f;

__device__ __forceinline__ void bulk_load(void* dst, const void* src,
                                          uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Shared → global bulk copy (async proxy), tracked by this thread's bulk
// groups: commit, then wait until the source may be overwritten (read) or
// until the writes are done.
__device__ __forceinline__ void bulk_store(void* dst, const void* src,
                                           uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(dst), "r"(smem_u32(src)), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// K-major operand with K = 128 in two 64-column halves `atom` bytes apart.
__device__ __forceinline__ uint64_t dk128(uint32_t base, int kk, int atom) {
  return smem_desc_sw128(base + (kk >> 2) * atom + (kk & 3) * 32, 16, 1024);
}
// MN-major B: rows are K, N = 128 in two 64-wide halves `atom` bytes apart.
__device__ __forceinline__ uint64_t dmn(uint32_t base, int kk, int atom) {
  return smem_desc_sw128(base + kk * 2048, atom, 1024);
}

__device__ __forceinline__ void store_bf16_row64(__nv_bfloat16* dst,
                                                 const uint32_t (&a)[32],
                                                 const uint32_t (&b)[32],
                                                 float scale) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t* src = q < 4 ? a : b;
    const int o = (q & 3) * 8;
    uint4 u;
    u.x = pack_bf16x2(__uint_as_float(src[o + 0]) * scale,
                      __uint_as_float(src[o + 1]) * scale);
    u.y = pack_bf16x2(__uint_as_float(src[o + 2]) * scale,
                      __uint_as_float(src[o + 3]) * scale);
    u.z = pack_bf16x2(__uint_as_float(src[o + 4]) * scale,
                      __uint_as_float(src[o + 5]) * scale);
    u.w = pack_bf16x2(__uint_as_float(src[o + 6]) * scale,
                      __uint_as_float(src[o + 7]) * scale);
    reinterpret_cast<uint4*>(dst)[q] = u;
  }
}

// ---------------------------------------------------------------- pre-pass --
// D = Σ_d dO·O (dO fp16, O bf16) and L2 = LSE·log2e per (batch, head,
// padded position).  One warp takes eight consecutive positions of one
// (batch, head), half a warp per row and 16 bytes of each tensor per lane,
// and issues all eight rows' loads before it uses any, so that enough bytes
// are in flight to stream the two tensors.  Past the sequence end D = 0 and
// L2 = +∞, so that P = exp2(S·c − L2) of a padded query is exactly 0
// without a mask.
constexpr int PRE_ROWS = 8;
__global__ void __launch_bounds__(256)
    attn_bwd_prepass_kernel(const __nv_bfloat16* __restrict__ O,
                            const __half* __restrict__ dO,
                            const float* __restrict__ LSE,
                            float* __restrict__ Dp, float* __restrict__ L2p,
                            int b_, int nq, int s, int s_pad) {
  const int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int per = s_pad / PRE_ROWS;
  if (w >= (int64_t)b_ * nq * per) return;
  const int64_t bh = w / per;      // b·nq + head
  const int pos0 = (int)(w % per) * PRE_ROWS;
  const int head = (int)(bh % nq);
  const int64_t bb = bh / nq;
  const int half = lane >> 4, col = (lane & 15) * 8;
  uint4 uo[PRE_ROWS / 2], ud[PRE_ROWS / 2];
#pragma unroll
  for (int i = 0; i < PRE_ROWS / 2; ++i) {
    const int pos = pos0 + 2 * i + half;
    if (pos < s) {
      const int64_t off = ((bb * s + pos) * nq + head) * HD + col;
      uo[i] = __ldg(reinterpret_cast<const uint4*>(O + off));
      ud[i] = __ldg(reinterpret_cast<const uint4*>(dO + off));
    } else {
      uo[i] = make_uint4(0u, 0u, 0u, 0u);
      ud[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int i = 0; i < PRE_ROWS / 2; ++i) {
    const uint32_t ow[4] = {uo[i].x, uo[i].y, uo[i].z, uo[i].w};
    const uint32_t dw[4] = {ud[i].x, ud[i].y, ud[i].z, ud[i].w};
    float acc = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 o = unpack_bf16x2(ow[q]);
      const float2 d = unpack_f16x2(dw[q]);
      acc += o.x * d.x + o.y * d.y;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    const int pos = pos0 + 2 * i + half;
    if ((lane & 15) == 0) {
      Dp[bh * s_pad + pos] = acc;
      L2p[bh * s_pad + pos] =
          pos < s ? LSE[bh * s + pos] * LOG2E_F : __int_as_float(0x7f800000);
    }
  }
}

struct BwdTcArgs {
  CUtensorMap mq, mk, mv, mdo;
  const __half* q;       // [b, s, nq·d] as the tensor maps
  const __half* dout;
  const __half* k;       // [b, s, nkv·d]
  const __half* v;
  const float* Dp;
  const float* L2p;
  __nv_bfloat16* out0;   // dQ, or dK
  __nv_bfloat16* out1;   // dV
  uint8_t* ds;           // dSᵀ tiles, 32 KB each (see ds_tile)
  int hk0, hkn;          // this pass: (batch, kv head) pairs [hk0, hk0+hkn)
  int s, s_pad, nq, nkv, causal;
  float scale, scale_log2;
  unsigned* status;
};

// Index of the dSᵀ tile of (q head lh of this pass, query block qb, key
// block kb), lh = (pair − hk0)·group + head within the group: per head the
// query blocks in order, each with its key blocks in order (causal: kb ≤ qb
// only), so one query block's tiles are contiguous.
__device__ __forceinline__ int64_t ds_tile(const BwdTcArgs& a, int lh, int qb,
                                           int kb, int nblk) {
  const int64_t per_head =
      a.causal ? (int64_t)nblk * (nblk + 1) / 2 : (int64_t)nblk * nblk;
  const int64_t first =
      a.causal ? (int64_t)qb * (qb + 1) / 2 : (int64_t)qb * nblk;
  return (int64_t)lh * per_head + first + kb;
}

// Row r of a 128-row K-major swizzled half tile (128-byte rows): its eight
// 16-byte chunks from 32 packed words.
__device__ __forceinline__ void st_row8(uint8_t* tile, int r,
                                        const uint32_t (&pk)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<uint4*>(tile + r * 128 + ((q ^ (r & 7)) << 4)) =
        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}

// Causal mask of a diagonal block on 64 fp16 values in 32 packed words:
// keep elements [t, 64), zero the rest.  Applied to packed words so the
// unrolled hot loop stays branch-free.
__device__ __forceinline__ void keep_from(uint32_t (&w)[32], int t) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    w[j] &= (2 * j + 1 < t) ? 0u : (2 * j < t ? 0xffff0000u : 0xffffffffu);
}

// ----------------------------------------------------------------------- dQ --
namespace dq {
constexpr int NS = 3;                          // stages of (dSᵀ, K) tiles
constexpr int TILE = 2 * A128;                 // 128 × 128 fp16, 32 KB
constexpr int OFF_DS = 0;
constexpr int OFF_K = NS * TILE;
constexpr int OFF_BAR = 2 * NS * TILE;
constexpr int SMEM = OFF_BAR + 256 + 1024;
constexpr int NTHREADS = 192;                  // TMA, MMA, 4 epilogue warps
constexpr uint32_t NCOLS = 256;                // two 128-column accumulators
}  // namespace dq

__global__ void __launch_bounds__(dq::NTHREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ BwdTcArgs a) {
  using namespace dq;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* full = bar;              // [NS] dSᵀ and K tiles landed
  uint64_t* empty = full + NS;       // [NS] their MMAs done
  uint64_t* tfull = empty + NS;      // [2] accumulator complete
  uint64_t* tempty = tfull + 2;      // [2] accumulator read out
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work items in heavy-first order (query block rank slowest), dealt out
  // round-robin to the persistent CTAs
  const int nblk = (a.s + 127) / 128;
  const int group = a.nq / a.nkv;
  const int per = a.hkn * group;   // q heads of this pass
  const int items = nblk * per;
  auto decode = [&](int t, int& bb, int& jq, int& lh, int& qb, int& nkb) {
    const int rank = t / per;
    lh = t % per;
    const int pair = a.hk0 + lh / group;
    bb = pair / a.nkv;
    jq = (pair % a.nkv) * group + lh % group;
    qb = nblk - 1 - rank;
    nkb = a.causal ? qb + 1 : nblk;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, NCOLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------- TMA --
      tma_prefetch_desc(&a.mk);
      uint32_t st = 0, ph = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < items; t += gridDim.x) {
        int bb, jq, lh, qb, nkb;
        decode(t, bb, jq, lh, qb, nkb);
        const int kvh = jq / group;
        const uint8_t* src = a.ds + ds_tile(a, lh, qb, 0, nblk) * TILE;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[st], ph ^ 1, abort_flag, a.status, 31)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], 2 * TILE);
          armed |= 1u << st;
          armed_par = (armed_par & ~(1u << st)) | (ph << st);
          bulk_load(sm + OFF_DS + st * TILE, src + (int64_t)kb * TILE, TILE,
                    &full[st]);
          for (int hh = 0; hh < 2; ++hh)
            tma_load_3d(sm + OFF_K + st * TILE + hh * A128, &a.mk, &full[st],
                        kvh * HD + hh * 64, kb * 128, bb);
          if (++st == NS) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int i = 0; i < NS; ++i)
          if (armed & (1u << i))
            mbar_wait(&full[i], (armed_par >> i) & 1u, &no_abort, nullptr, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMA --
      // D[q][d] += Σ_key dSᵀ[key][q] · K[key][d]: both operands have the
      // key (the reduction) as their row, so A is M-major and B N-major
      constexpr uint32_t IDESC = idesc_f16_f32(128, 128, 1, 1);
      uint32_t st = 0, ph = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; ok && t < items; t += gridDim.x, ++it) {
        int bb, jq, lh, qb, nkb;
        decode(t, bb, jq, lh, qb, nkb);
        const int buf = it & 1;
        if (!mbar_wait(&tempty[buf], ((it >> 1) & 1) ^ 1, abort_flag,
                       a.status, 32)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * 128;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[st], ph, abort_flag, a.status, 33)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sdS = smem_u32(sm + OFF_DS + st * TILE);
          const uint32_t sK = smem_u32(sm + OFF_K + st * TILE);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_f16(d_tmem, dmn(sdS, kk, A128), dmn(sK, kk, A128), IDESC,
                       (kb > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[st]);
          if (++st == NS) {
            st = 0;
            ph ^= 1;
          }
        }
        if (ok) tc_commit(&tfull[buf]);
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        tc_commit(drain);
        mbar_wait(drain, 0, &no_abort, nullptr, 0);
      }
    }
  } else {
    // -------------------------------------------------------- epilogue --
    // thread: query row of the block (TMEM lane), all 128 columns of dQ
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < items; t += gridDim.x, ++it) {
      int bb, jq, lh, qb, nkb;
      decode(t, bb, jq, lh, qb, nkb);
      const int buf = it & 1;
      if (!mbar_wait_warp(&tfull[buf], (it >> 1) & 1, abort_flag, a.status,
                          38))
        break;
      tc_fence_after();
      const int qi = qb * 128 + row;
      const uint32_t lanes = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                             buf * 128;
      __nv_bfloat16* dst = a.out0 +
                           ((int64_t)bb * a.s + qi) * (int64_t)(a.nq * HD) +
                           jq * HD;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t o0[32], o1[32];
        tmem_ld32(lanes + hh * 64, o0);
        tmem_ld32(lanes + hh * 64 + 32, o1);
        tmem_ld_wait(o0);
        reg_fence32(o1);
        if (qi < a.s) store_bf16_row64(dst + hh * 64, o0, o1, a.scale);
      }
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, NCOLS);
}

// ------------------------------------------------------------------ dK, dV --
namespace dkv {
constexpr int NQ = 3, NO = 2;                  // Q ring and dO ring depths
constexpr int TILE = 2 * A128;                 // 128 rows × 128 d, 32 KB
constexpr int OFF_Q = 0;
constexpr int OFF_O = OFF_Q + NQ * TILE;
constexpr int OFF_P = OFF_O + NO * TILE;       // Pᵀ: 128 keys × 128 queries
constexpr int OFF_DS = OFF_P + TILE;           // dSᵀ
constexpr int OFF_QST = OFF_DS + TILE;         // NQ × 128 LSE·log2e
constexpr int OFF_OST = OFF_QST + NQ * 512;    // NO × 128 D
constexpr int OFF_BAR = OFF_OST + NO * 512;
// No alignment slack: the kernel checks that the dynamic shared memory
// starts on a 1024-byte boundary (as the 128-byte swizzle requires).
constexpr int SMEM = OFF_BAR + 256;
// K and V in TMEM as the A operands of Sᵀ and dPᵀ; Sᵀ and then dPᵀ of each
// block take turns in X; dV and dK accumulate in the last 256 columns.
constexpr uint32_t COL_K = 0, COL_V = 64, COL_X = 128, COL_DV = 256,
                   COL_DK = 384;
}  // namespace dkv

__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_dkdv_tc_kernel(const __grid_constant__ BwdTcArgs a) {
  using namespace dkv;
  extern __shared__ __align__(1024) uint8_t smem_aligned[];
  uint8_t* sm = smem_aligned;
  if (smem_u32(sm) & 1023u) {   // uniform across the CTA: nothing started yet
    if (threadIdx.x == 0) record_error(a.status, kDevTimeout, 99);
    return;
  }
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* q_full = bar;              // [NQ] Q tile + its LSE·log2e
  uint64_t* q_empty = q_full + NQ;     // [NQ]
  uint64_t* o_full = q_empty + NQ;     // [NO] dO tile + its D
  uint64_t* o_empty = o_full + NO;     // [NO]
  uint64_t* kv_full = o_empty + NO;    // K and V written to TMEM
  uint64_t* x_full = kv_full + 1;      // Sᵀ, then dPᵀ, in X
  uint64_t* x_free = x_full + 1;       // X copied to registers
  uint64_t* p_full = x_free + 1;       // Pᵀ written
  uint64_t* p_free = p_full + 1;       // dV += Pᵀ·dO done with it
  uint64_t* ds_full = p_free + 1;      // dSᵀ written
  uint64_t* ds_free = ds_full + 1;     // dK += dSᵀ·Q and its copy out done
  uint64_t* done = ds_free + 1;
  uint64_t* drain = done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 1-D grid, block rank slowest: the heaviest (first, under the causal
  // mask) key blocks of every kv head start first; in (kv head, key block)
  // order the last heads' heavy blocks would start late and set the tail
  const int nblk = (a.s + 127) / 128;
  const int per = a.hkn;              // (batch, kv head) pairs of this pass
  const int rank = blockIdx.x / per, rem = blockIdx.x % per;
  const int b = (a.hk0 + rem) / a.nkv, kvh = (a.hk0 + rem) % a.nkv;
  const int k0 = rank * 128;
  const int group = a.nq / a.nkv;
  const int nqb = (a.s + 127) / 128;
  const int qb_first = a.causal ? k0 / 128 : 0;
  const int per_head = nqb - qb_first;
  const int iters = per_head * group;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int i = 0; i < NO; ++i) {
      mbar_init(&o_full[i], 1);
      mbar_init(&o_empty[i], 1);
    }
    mbar_init(kv_full, 256);
    mbar_init(x_full, 1);
    mbar_init(x_free, 256);
    mbar_init(p_full, 256);
    mbar_init(p_free, 1);
    mbar_init(ds_full, 256);
    mbar_init(ds_free, 2);
    mbar_init(done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane < 2) {
      // lane 0: Q tiles and their LSE (freed after dK += dSᵀ·Q);
      // lane 1: dO tiles and their D (freed after dV += Pᵀ·dO)
      const bool is_q = lane == 0;
      const CUtensorMap* map = is_q ? &a.mq : &a.mdo;
      uint64_t* full = is_q ? q_full : o_full;
      uint64_t* empty = is_q ? q_empty : o_empty;
      uint8_t* ring = sm + (is_q ? OFF_Q : OFF_O);
      uint8_t* stats = sm + (is_q ? OFF_QST : OFF_OST);
      const float* src_stats = is_q ? a.L2p : a.Dp;
      const int depth = is_q ? NQ : NO;
      tma_prefetch_desc(map);
      uint32_t armed = 0, armed_par = 0;
      for (int it = 0; it < iters; ++it) {
        const int st = it % depth;
        const uint32_t ph = (it / depth) & 1;
        if (!mbar_wait(&empty[st], ph ^ 1, abort_flag, a.status, 41)) break;
        const int jq = kvh * group + it / per_head;
        const int qb = qb_first + it % per_head;
        mbar_arrive_expect_tx(&full[st], TILE + 512);
        armed |= 1u << st;
        armed_par = (armed_par & ~(1u << st)) | (ph << st);
        for (int hh = 0; hh < 2; ++hh)
          tma_load_3d(ring + st * TILE + hh * A128, map, &full[st],
                      jq * HD + hh * 64, qb * 128, b);
        const int64_t soff = ((int64_t)b * a.nq + jq) * a.s_pad + qb * 128;
        bulk_load(stats + st * 512, src_stats + soff, 512, &full[st]);
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int st = 0; st < depth; ++st)
          if (armed & (1u << st))
            mbar_wait(&full[st], (armed_par >> st) & 1u, &no_abort, nullptr, 0);
      }
    } else if (lane == 2) {
      // each dSᵀ tile out to global memory for the dQ kernel; the buffer is
      // released (second arrival on ds_free) once the copy has read it
      for (int it = 0; it < iters; ++it) {
        if (!mbar_wait(ds_full, it & 1, abort_flag, a.status, 54)) break;
        const int qb = qb_first + it % per_head;
        bulk_store(a.ds + ds_tile(a, rem * group + it / per_head, qb, rank,
                                  nblk) *
                              TILE,
                   sm + OFF_DS, TILE);
        bulk_wait_read();
        mbar_arrive(ds_free);
      }
      bulk_wait_all();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_f16_f32(128, 128, 0, 0);
      constexpr uint32_t IDESC_G = idesc_f16_f32(128, 128, 0, 1);
      bool ok = mbar_wait(kv_full, 0, abort_flag, a.status, 42);
      tc_fence_after();
      // dV += Pᵀ·dO of block i (releases Pᵀ and the dO tile)
      auto dv_mma = [&](int i) -> bool {
        if (!mbar_wait(p_full, i & 1, abort_flag, a.status, 43)) return false;
        tc_fence_after();
        const uint32_t sdO = smem_u32(sm + OFF_O + (i % NO) * TILE);
        const uint32_t sP = smem_u32(sm + OFF_P);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(tmem + COL_DV, dk128(sP, kk, A128), dmn(sdO, kk, A128),
                     IDESC_G, (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(p_free);
        tc_commit(&o_empty[i % NO]);
        return true;
      };
      // dK += dSᵀ·Q of block i (releases dSᵀ and the Q tile)
      auto dk_mma = [&](int i) -> bool {
        if (!mbar_wait(ds_full, i & 1, abort_flag, a.status, 52)) return false;
        tc_fence_after();
        const uint32_t sQ = smem_u32(sm + OFF_Q + (i % NQ) * TILE);
        const uint32_t sdS = smem_u32(sm + OFF_DS);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(tmem + COL_DK, dk128(sdS, kk, A128), dmn(sQ, kk, A128),
                     IDESC_G, (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(ds_free);
        tc_commit(&q_empty[i % NQ]);
        return true;
      };
      // per block: Sᵀ(it); dK of it−1 (its dSᵀ was written while Sᵀ(it)
      // ran), which keeps the tensor cores busy while the elementwise warps
      // copy Sᵀ(it) out of the shared X buffer; dPᵀ(it) into X once they
      // have; dV of it (Pᵀ(it) is written while dK(it−1) and dPᵀ(it) run)
      for (int it = 0; ok && it < iters; ++it) {
        ok = mbar_wait(&q_full[it % NQ], (it / NQ) & 1, abort_flag, a.status,
                       44) &&
             (it == 0 || mbar_wait(x_free, 1, abort_flag, a.status, 45));
        if (!ok) break;
        tc_fence_after();
        const uint32_t sQ = smem_u32(sm + OFF_Q + (it % NQ) * TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16_ts(tmem + COL_X, tmem + COL_K + kk * 8,
                        dk128(sQ, kk, A128), IDESC_S, kk > 0 ? 1u : 0u);
        tc_commit(x_full);
        if (it > 0 && !(ok = dk_mma(it - 1))) break;
        ok = mbar_wait(&o_full[it % NO], (it / NO) & 1, abort_flag, a.status,
                       49) &&
             mbar_wait(x_free, 0, abort_flag, a.status, 50);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sdO = smem_u32(sm + OFF_O + (it % NO) * TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16_ts(tmem + COL_X, tmem + COL_V + kk * 8,
                        dk128(sdO, kk, A128), IDESC_S, kk > 0 ? 1u : 0u);
        tc_commit(x_full);
        if (!(ok = dv_mma(it))) break;
      }
      if (ok && iters > 0) ok = dk_mma(iters - 1);
      if (ok) tc_commit(done);
      if (*abort_flag) {
        volatile int no_abort = 0;
        tc_commit(drain);
        mbar_wait(drain, 0, &no_abort, nullptr, 0);
      }
    }
  } else {
    // ------------------------------------------------------ elementwise --
    // thread: key row r (TMEM lane), queries [64·half, 64·half + 64) of
    // each block
    const int half = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int key = k0 + r;
    const uint32_t lanes = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c = a.scale_log2;
    const int64_t ldk = (int64_t)a.nkv * HD;
    const int64_t row = ((int64_t)b * a.s + key) * ldk + kvh * HD + half * 64;
    {
      // this thread's half row of K and of V into TMEM (zeros past the end)
      uint32_t kv[32];
      const __half* const srcs[2] = {a.k, a.v};
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint4* src = reinterpret_cast<const uint4*>(srcs[t] + row);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 u = key < a.s ? src[i] : make_uint4(0u, 0u, 0u, 0u);
          kv[4 * i] = u.x;
          kv[4 * i + 1] = u.y;
          kv[4 * i + 2] = u.z;
          kv[4 * i + 3] = u.w;
        }
        tmem_st32(lanes + (t == 0 ? COL_K : COL_V) + half * 32, kv);
      }
      tc_fence_before();
      mbar_arrive(kv_full);
    }
    bool ok = true;
    for (int it = 0; it < iters; ++it) {
      const int qb = qb_first + it % per_head;
      // queries past the end have L2 = +∞ (P = 0); keys past the end get
      // P = 0 (their dSᵀ rows go to the dQ kernel); the causal diagonal
      // block keeps queries ≥ the key
      const bool diag = a.causal && qb * 128 == k0;
      // Sᵀ → P, kept in fp16
      if (!mbar_wait_warp(x_full, 0, abort_flag, a.status, 46)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t x0[32], x1[32];
      tmem_ld32(lanes + COL_X + half * 64, x0);
      tmem_ld32(lanes + COL_X + half * 64 + 32, x1);
      tmem_ld_wait(x0);
      reg_fence32(x1);
      tc_fence_before();
      mbar_arrive(x_free);
      // LSE·log2e of this half's 64 queries: all loads issued before use
      const float4* lst = reinterpret_cast<const float4*>(
                              sm + OFF_QST + (it % NQ) * 512) +
                          half * 16;
      uint32_t pp[32];   // P in fp16 pairs (Pᵀ row of this key)
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        float lv[32];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4*>(&lv[4 * i]) = lst[ch * 8 + i];
        const uint32_t(&xs)[32] = ch == 0 ? x0 : x1;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(xs[i]), c, -lv[i]));
          const float p1 =
              ex2_approx(fmaf(__uint_as_float(xs[i + 1]), c, -lv[i + 1]));
          pp[ch * 16 + (i >> 1)] = pack_f16x2(p0, p1);
        }
      }
      if (diag) keep_from(pp, r - half * 64);
      const uint32_t kmask = key < a.s ? 0xffffffffu : 0u;
#pragma unroll
      for (int i = 0; i < 32; ++i) pp[i] &= kmask;
      // Pᵀ(it) out now: the tile is free once dV of it−1 has completed
      if (it >= 1 &&
          !mbar_wait_warp(p_free, (it - 1) & 1, abort_flag, a.status, 47)) {
        ok = false;
        break;
      }
      st_row8(sm + OFF_P + half * A128, r, pp);
      fence_proxy_async_smem();
      mbar_arrive(p_full);
      // dPᵀ → dS = P ⊙ (dP − D), P taken in its fp16 form
      if (!mbar_wait_warp(x_full, 1, abort_flag, a.status, 51)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_ld32(lanes + COL_X + half * 64, x0);
      tmem_ld32(lanes + COL_X + half * 64 + 32, x1);
      tmem_ld_wait(x0);
      reg_fence32(x1);
      tc_fence_before();
      mbar_arrive(x_free);
      const float4* dst = reinterpret_cast<const float4*>(
                              sm + OFF_OST + (it % NO) * 512) +
                          half * 16;
      uint32_t pd[32];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        float dv[16];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<float4*>(&dv[4 * i]) = dst[ch * 4 + i];
        const uint32_t(&xs)[32] = ch < 2 ? x0 : x1;
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const int e = (ch & 1) * 16 + i;   // index within xs
          const float2 pf = unpack_f16x2(pp[ch * 8 + (i >> 1)]);
          pd[ch * 8 + (i >> 1)] =
              pack_f16x2(pf.x * (__uint_as_float(xs[e]) - dv[i]),
                         pf.y * (__uint_as_float(xs[e + 1]) - dv[i + 1]));
        }
      }
      // dSᵀ(it) out: the tile is free once dK of it−1 has completed
      if (it >= 1 &&
          !mbar_wait_warp(ds_free, (it - 1) & 1, abort_flag, a.status, 53)) {
        ok = false;
        break;
      }
      st_row8(sm + OFF_DS + half * A128, r, pd);
      fence_proxy_async_smem();
      mbar_arrive(ds_full);
    }
    if (iters > 0 && __all_sync(0xffffffffu, ok) &&
        mbar_wait_warp(done, 0, abort_flag, a.status, 48)) {
      tc_fence_after();
      uint32_t o0[32], o1[32];
      tmem_ld32(lanes + COL_DK + half * 64, o0);
      tmem_ld32(lanes + COL_DK + half * 64 + 32, o1);
      tmem_ld_wait(o0);
      reg_fence32(o1);
      if (key < a.s) store_bf16_row64(a.out0 + row, o0, o1, a.scale);
      tmem_ld32(lanes + COL_DV + half * 64, o0);
      tmem_ld32(lanes + COL_DV + half * 64 + 32, o1);
      tmem_ld_wait(o0);
      reg_fence32(o1);
      if (key < a.s) store_bf16_row64(a.out1 + row, o0, o1, 1.0f);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

int64_t attn_stats_pad(int64_t s) { return (s + 127) / 128 * 128; }

namespace {
// dSᵀ tiles of one (batch, kv head) pair: its GQA group's q heads
int64_t ds_pair_bytes(const AttnShape& sh) {
  const int64_t nblk = (sh.s + 127) / 128;
  const int64_t per_head = sh.causal ? nblk * (nblk + 1) / 2 : nblk * nblk;
  return (int64_t)(sh.nq / sh.nkv) * per_head * (int64_t)dq::TILE;
}
// (batch, kv head) pairs per pass: as many as fit in the budget of tile
// bytes (at least one), so the scratch stays bounded for long sequences
constexpr int64_t kDsBudgetDefault = int64_t(8) << 30;
std::atomic<int64_t> g_ds_budget{kDsBudgetDefault};
}  // namespace

int64_t attn_ds_pairs_per_pass(const AttnShape& sh) {
  return std::max<int64_t>(
      1, std::min<int64_t>(sh.b * sh.nkv,
                           g_ds_budget.load() / ds_pair_bytes(sh)));
}

int64_t attn_set_ds_budget(int64_t bytes) {
  return g_ds_budget.exchange(bytes > 0 ? bytes : kDsBudgetDefault);
}

int64_t attn_ds_bytes(const AttnShape& sh) {
  return sh.ds_pairs * ds_pair_bytes(sh);
}

int flash_bwd(const AttnShape& sh, const void* Q, const void* K, const void* V,
              const void* O, const void* dO, const float* LSE, float* Dp,
              float* L2p, void* dS, void* dQ, void* dK, void* dV,
              unsigned* status, void* stream) {
  if (sh.d != HD || sh.ds_pairs < 1) return cudaErrorInvalidValue;
  static cudaError_t e1 = cudaFuncSetAttribute(
      attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      dq::SMEM);
  static cudaError_t e2 = cudaFuncSetAttribute(
      attn_bwd_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      dkv::SMEM);
  if (e1 != cudaSuccess) return e1;
  if (e2 != cudaSuccess) return e2;
  if (reinterpret_cast<uintptr_t>(dS) & 15u) return cudaErrorInvalidValue;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t s_pad = attn_stats_pad(sh.s);
  const double sd = (double)sh.s;
  const double pairs = sh.causal ? sd * (sd + 1.0) / 2.0 : sd * sd;
  const double core = 4.0 * sh.b * sh.nq * HD * pairs;
  const double io = 2.0 * sh.b * sh.s * HD;
  const double ds_bytes_all =
      (double)ds_pair_bytes(sh) * (double)(sh.b * sh.nkv);
  {
    const int64_t warps = sh.b * sh.nq * (s_pad / PRE_ROWS);
    ProfScope ps(stream, KF_ELEMENTWISE, 2.0 * sh.b * sh.s * sh.nq * HD,
                 2.0 * io * sh.nq);
    attn_bwd_prepass_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0,
                              s>>>(static_cast<const __nv_bfloat16*>(O),
                                   static_cast<const __half*>(dO), LSE, Dp,
                                   L2p, (int)sh.b, sh.nq, (int)sh.s,
                                   (int)s_pad);
  }
  BwdTcArgs a;
  memset(&a, 0, sizeof(a));
  // all four in 128-row boxes of 64 columns
  const uint64_t ldq = (uint64_t)sh.nq * HD * 2, ldk = (uint64_t)sh.nkv * HD * 2;
  const bool ok =
      encode_tmap_3d_f16(&a.mq, Q, (uint64_t)sh.nq * HD, sh.s, sh.b, ldq,
                         ldq * sh.s, 64, 128, 1) &&
      encode_tmap_3d_f16(&a.mdo, dO, (uint64_t)sh.nq * HD, sh.s, sh.b, ldq,
                         ldq * sh.s, 64, 128, 1) &&
      encode_tmap_3d_f16(&a.mk, K, (uint64_t)sh.nkv * HD, sh.s, sh.b, ldk,
                         ldk * sh.s, 64, 128, 1) &&
      encode_tmap_3d_f16(&a.mv, V, (uint64_t)sh.nkv * HD, sh.s, sh.b, ldk,
                         ldk * sh.s, 64, 128, 1);
  if (!ok) return cudaErrorInvalidValue;
  a.q = static_cast<const __half*>(Q);
  a.dout = static_cast<const __half*>(dO);
  a.k = static_cast<const __half*>(K);
  a.v = static_cast<const __half*>(V);
  a.Dp = Dp;
  a.L2p = L2p;
  a.ds = static_cast<uint8_t*>(dS);
  a.s = (int)sh.s;
  a.s_pad = (int)s_pad;
  a.nq = sh.nq;
  a.nkv = sh.nkv;
  a.causal = sh.causal;
  a.scale = sh.scale;
  a.scale_log2 = sh.scale * LOG2E_F;
  a.status = status;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  sms = std::max(sms, 1);
  const int64_t pairs_all = sh.b * sh.nkv;
  // the pairs the caller's dS region was carved for (never the budget,
  // which another thread may have changed since)
  const int64_t chunk = std::min<int64_t>(sh.ds_pairs, pairs_all);
  const int64_t nblk = (sh.s + 127) / 128;
  const int group = sh.nq / sh.nkv;
  int passes = 0;
  for (int64_t hk0 = 0; hk0 < pairs_all; hk0 += chunk, ++passes) {
    const int64_t hkn = std::min(chunk, pairs_all - hk0);
    const double frac = (double)hkn / (double)pairs_all;
    a.hk0 = (int)hk0;
    a.hkn = (int)hkn;
    a.out0 = static_cast<__nv_bfloat16*>(dK);
    a.out1 = static_cast<__nv_bfloat16*>(dV);
    {
      ProfScope ps(stream, KF_ATTN_BWD_DKDV, 1.5 * core * frac,
                   (io * (2.0 * sh.nq + 4.0 * sh.nkv) + ds_bytes_all) * frac);
      attn_bwd_dkdv_tc_kernel<<<(unsigned)(nblk * hkn), THREADS, dkv::SMEM,
                                s>>>(a);
    }
    a.out0 = static_cast<__nv_bfloat16*>(dQ);
    a.out1 = nullptr;
    {
      const int64_t items = nblk * hkn * group;
      ProfScope ps(stream, KF_ATTN_BWD_DQ, 0.5 * core * frac,
                   (ds_bytes_all + io * sh.nq) * frac);
      attn_bwd_dq_tc_kernel<<<(unsigned)std::min<int64_t>(items, sms),
                              dq::NTHREADS, dq::SMEM, s>>>(a);
    }
  }
  count_launch(1 + 2 * passes);
  return cudaGetLastError();
}

}  // namespace tp
