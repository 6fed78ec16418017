// attn_bwd_tc.cu — causal GQA flash-attention backward on tcgen05 / TMEM.
//
// The backward of the attention core of one rank's local heads ([Grasp-TP]
// §4; [Troverld] §I.O: the backward recomputes QKᵀ from the saved log-sum-
// exp; [hjcheng-TP] Attention 单卡backward: dP = dO·Vᵀ, dV = Pᵀ·dO, dS from
// the softmax backward, dQ = dS·K, dK = dSᵀ·Q).
//
//   pre-pass  D = rowsum(dO ∘ O) and LSE·log2e per (batch, head, position),
//             padded with zeros to a multiple of 128 positions.
//   dQ        CTA = 128 queries of one (batch, q head); per block of 128 keys
//               S = Q·Kᵀ, dP = dO·Vᵀ            (M=128, N=128, K=128) → TMEM
//               dS = P ⊙ (dP − D), P = exp2(S·c − LSE·log2e)   (elementwise)
//               dQ += dS·K                       (M=128, N=128, K=128) → TMEM
//             Q and dO sit in TMEM as the A operands of S and dP.
//   dK, dV    CTA = 128 keys of one (batch, kv head); per q head of the GQA
//             group and block of 128 queries at or after the keys
//               Sᵀ = K·Qᵀ, then dPᵀ = V·dOᵀ      (M=128, N=128, K=128) → TMEM
//               dV += Pᵀ·dO,  dK += dSᵀ·Q        (M=128, N=128, K=128) → TMEM
//             K and V sit in TMEM as the A operands; Sᵀ and dPᵀ of a block
//             take turns in one 128-column TMEM buffer, which leaves room
//             for both accumulators.
// Both: warp 0 TMA, warp 1 TMEM allocation + single-thread MMA issue, warps
// 2–9 elementwise (two threads per TMEM lane, half of the columns each).
// The score MMAs of the next block are issued as soon as the elementwise
// warps have copied the current scores to registers, ahead of the gradient
// MMAs, so the tensor cores work while the elementwise warps do.  The
// elementwise loops are unrolled but branch-free (masks come from padding
// and a fix-up of the causal diagonal on packed words): a per-block body
// that outgrows the instruction cache runs several times slower.  K and V
// (dQ) or Q and dO (dK, dV) stream through rings of their own, each tile
// freed by the last MMA that reads it.  A tcgen05.mma of M=128 costs about
// the same for N=64 as for N=128, so the wider blocks do twice the work per
// instruction.  No atomics: reruns are bit-identical, and the GQA sums of
// dK, dV stay inside one CTA.
// Operands fp16, accumulation fp32; dQ, dK, dV are written in bf16.
#include <cuda_fp16.h>

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
// One warp per (batch, head, padded position): D = Σ_d dO·O (dO fp16, O
// bf16) and L2 = LSE·log2e.  Past the sequence end D = 0 and L2 = +∞, so
// that P = exp2(S·c − L2) of a padded query is exactly 0 without a mask.
__global__ void __launch_bounds__(256)
    attn_bwd_prepass_kernel(const __nv_bfloat16* __restrict__ O,
                            const __half* __restrict__ dO,
                            const float* __restrict__ LSE,
                            float* __restrict__ Dp, float* __restrict__ L2p,
                            int b_, int nq, int s, int s_pad) {
  const int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= (int64_t)b_ * nq * s_pad) return;
  const int pos = (int)(w % s_pad);
  const int64_t bh = w / s_pad;   // b·nq + head
  const int head = (int)(bh % nq);
  const int64_t bb = bh / nq;
  float acc = 0.0f;
  if (pos < s) {
    const int64_t off = ((bb * s + pos) * nq + head) * HD + lane * 4;
    const uint2 uo = *reinterpret_cast<const uint2*>(O + off);
    const uint2 ud = *reinterpret_cast<const uint2*>(dO + off);
    const float2 o0 = unpack_bf16x2(uo.x), o1 = unpack_bf16x2(uo.y);
    const float2 d0 = unpack_f16x2(ud.x), d1 = unpack_f16x2(ud.y);
    acc = o0.x * d0.x + o0.y * d0.y + o1.x * d1.x + o1.y * d1.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) {
    Dp[w] = acc;
    L2p[w] = pos < s ? LSE[bh * s + pos] * LOG2E_F : __int_as_float(0x7f800000);
  }
}

// ----------------------------------------------------------------------- dQ --
namespace dq {
constexpr int NK = 3, NV = 2;                 // K ring and V ring depths
constexpr int TILE = 2 * A128;                // one 128-key tile, 32 KB
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + NK * TILE;
constexpr int OFF_DS = OFF_V + NV * TILE;     // 2 buffers of 32 KB
constexpr int OFF_BAR = OFF_DS + 2 * TILE;
constexpr int SMEM = OFF_BAR + 256 + 1024;
// Q and dO live in TMEM as the A operands of S and dP (fp16 pairs, 64
// columns each); S, dP (128 keys each) and the dQ accumulator fill the rest.
constexpr uint32_t COL_Q = 0, COL_DO = 64, COL_S = 128, COL_DP = 256,
                   COL_DQ = 384;
}  // namespace dq

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
  int s, s_pad, nq, nkv, causal;
  float scale, scale_log2;
  unsigned* status;
};

// Row r of a 128-row K-major swizzled half tile (128-byte rows): its eight
// 16-byte chunks from 32 packed words.
__device__ __forceinline__ void st_row8(uint8_t* tile, int r,
                                        const uint32_t (&pk)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<uint4*>(tile + r * 128 + ((q ^ (r & 7)) << 4)) =
        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}

// dS for 32 keys of one query row: P = exp2(S·c − L2), dS = P·(dP − D),
// packed in fp16 pairs (element 2j in the low half of word j).
__device__ __forceinline__ void ds_chunk(const uint32_t (&sv)[32],
                                         const uint32_t (&pv)[32], float c,
                                         float l2, float dd, uint32_t* pk) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float p0 = ex2_approx(fmaf(__uint_as_float(sv[i]), c, -l2));
    const float p1 = ex2_approx(fmaf(__uint_as_float(sv[i + 1]), c, -l2));
    pk[i >> 1] = pack_f16x2(p0 * (__uint_as_float(pv[i]) - dd),
                            p1 * (__uint_as_float(pv[i + 1]) - dd));
  }
}

// Causal masks of a diagonal block on 64 fp16 values in 32 packed words:
// keep elements [0, t] (keep_upto) or [t, 64) (keep_from), zero the rest.
// Applied to packed words so the unrolled hot loops stay branch-free.
__device__ __forceinline__ void keep_upto(uint32_t (&w)[32], int t) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    w[j] &= (2 * j > t) ? 0u : (2 * j + 1 > t ? 0x0000ffffu : 0xffffffffu);
}
__device__ __forceinline__ void keep_from(uint32_t (&w)[32], int t) {
#pragma unroll
  for (int j = 0; j < 32; ++j)
    w[j] &= (2 * j + 1 < t) ? 0u : (2 * j < t ? 0xffff0000u : 0xffffffffu);
}

__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ BwdTcArgs a) {
  using namespace dq;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* q_full = bar;              // Q and dO written to TMEM
  uint64_t* k_full = bar + 1;          // [NK]
  uint64_t* k_empty = k_full + NK;     // [NK]
  uint64_t* v_full = k_empty + NK;     // [NV]
  uint64_t* v_empty = v_full + NV;     // [NV]
  uint64_t* sdp_full = v_empty + NV;   // S and dP of the current block
  uint64_t* sdp_free = sdp_full + 1;   // S, dP copied to registers
  uint64_t* ds_full = sdp_free + 1;    // [2]
  uint64_t* ds_free = ds_full + 2;     // [2]
  uint64_t* dq_done = ds_free + 2;
  uint64_t* drain = dq_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 1-D grid, block rank slowest: the heaviest query blocks first
  const int nblk = (a.s + 127) / 128;
  const int per = gridDim.x / nblk;   // n_q · batch
  const int rank = blockIdx.x / per, rem = blockIdx.x % per;
  const int b = rem / a.nq, j = rem % a.nq;
  const int q0 = (nblk - 1 - rank) * 128;
  const int kvh = j / (a.nq / a.nkv);
  const int kv_end = a.causal ? min(a.s, q0 + 128) : a.s;
  const int nkb = (kv_end + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 256);
    for (int i = 0; i < NK; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(sdp_free, 256);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ds_full[i], 256);
      mbar_init(&ds_free[i], 1);
    }
    mbar_init(dq_done, 1);
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
      // lane 0: the K ring (K_j is freed after dQ += dS_j·K_j);
      // lane 1: the V ring (V_j is freed as soon as dP_j is done)
      const bool is_k = lane == 0;
      const CUtensorMap* map = is_k ? &a.mk : &a.mv;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* ring = sm + (is_k ? OFF_K : OFF_V);
      const int depth = is_k ? NK : NV;
      tma_prefetch_desc(map);
      uint32_t armed = 0, armed_par = 0;
      for (int jb = 0; jb < nkb; ++jb) {
        const int st = jb % depth;
        const uint32_t ph = (jb / depth) & 1;
        if (!mbar_wait(&empty[st], ph ^ 1, abort_flag, a.status, 31)) break;
        mbar_arrive_expect_tx(&full[st], TILE);
        armed |= 1u << st;
        armed_par = (armed_par & ~(1u << st)) | (ph << st);
        for (int hh = 0; hh < 2; ++hh)
          tma_load_3d(ring + st * TILE + hh * A128, map, &full[st],
                      kvh * HD + hh * 64, jb * 128, b);
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        for (int st = 0; st < depth; ++st)
          if (armed & (1u << st))
            mbar_wait(&full[st], (armed_par >> st) & 1u, &no_abort, nullptr, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_f16_f32(128, 128, 0, 0);
      constexpr uint32_t IDESC_Q = idesc_f16_f32(128, 128, 0, 1);
      bool ok = mbar_wait(q_full, 0, abort_flag, a.status, 32);
      tc_fence_after();
      auto sdp_mma = [&](int jb) -> bool {
        if (!mbar_wait(&k_full[jb % NK], (jb / NK) & 1, abort_flag, a.status,
                       34) ||
            !mbar_wait(&v_full[jb % NV], (jb / NV) & 1, abort_flag, a.status,
                       39))
          return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(sm + OFF_K + (jb % NK) * TILE);
        const uint32_t sV = smem_u32(sm + OFF_V + (jb % NV) * TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          tc_mma_f16_ts(tmem + COL_S, tmem + COL_Q + kk * 8,
                        dk128(sK, kk, A128), IDESC_S, kk > 0 ? 1u : 0u);
          tc_mma_f16_ts(tmem + COL_DP, tmem + COL_DO + kk * 8,
                        dk128(sV, kk, A128), IDESC_S, kk > 0 ? 1u : 0u);
        }
        tc_commit(sdp_full);
        tc_commit(&v_empty[jb % NV]);
        return true;
      };
      auto dq_mma = [&](int i) -> bool {
        const int bb = i & 1;
        if (!mbar_wait(&ds_full[bb], (i >> 1) & 1, abort_flag, a.status, 33))
          return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(sm + OFF_K + (i % NK) * TILE);
        const uint32_t sdS = smem_u32(sm + OFF_DS + bb * TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(tmem + COL_DQ, dk128(sdS, kk, A128), dmn(sK, kk, A128),
                     IDESC_Q, (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&ds_free[bb]);
        tc_commit(&k_empty[i % NK]);
        return true;
      };
      // S_{j+1}, dP_{j+1} go in as soon as S_j, dP_j are in registers, ahead
      // of dQ += dS_j·K_j, so the elementwise warps never wait on dQ.
      if (ok) ok = sdp_mma(0);
      for (int jb = 0; ok && jb < nkb; ++jb) {
        ok = mbar_wait(sdp_free, jb & 1, abort_flag, a.status, 35);
        if (ok && jb + 1 < nkb) ok = sdp_mma(jb + 1);
        if (ok) ok = dq_mma(jb);
      }
      if (ok) tc_commit(dq_done);
      if (*abort_flag) {
        volatile int no_abort = 0;
        tc_commit(drain);
        mbar_wait(drain, 0, &no_abort, nullptr, 0);
      }
    }
  } else {
    // ------------------------------------------------------ elementwise --
    // thread: query row r (TMEM lane), keys [64·half, 64·half + 64) of each
    // block
    const int half = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qi = q0 + r;
    const uint32_t lanes = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int64_t srow = ((int64_t)b * a.nq + j) * a.s_pad + qi;
    const float l2 = a.L2p[srow], dd = a.Dp[srow];
    const float c = a.scale_log2;
    {
      // this thread's half row of Q and of dO into TMEM (zeros past the end)
      const int64_t off =
          ((int64_t)b * a.s + qi) * (int64_t)(a.nq * HD) + j * HD + half * 64;
      uint32_t qv[32];
      const __half* const srcs[2] = {a.q, a.dout};
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint4* src = reinterpret_cast<const uint4*>(srcs[t] + off);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 u = qi < a.s ? src[i] : make_uint4(0u, 0u, 0u, 0u);
          qv[4 * i] = u.x;
          qv[4 * i + 1] = u.y;
          qv[4 * i + 2] = u.z;
          qv[4 * i + 3] = u.w;
        }
        tmem_st32(lanes + (t == 0 ? COL_Q : COL_DO) + half * 32, qv);
      }
      tc_fence_before();
      mbar_arrive(q_full);
    }
    bool ok = true;
    for (int jb = 0; jb < nkb; ++jb) {
      const int bb = jb & 1;
      if (!mbar_wait_warp(sdp_full, jb & 1, abort_flag, a.status, 36)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s0[32], s1[32], p0[32], p1[32];
      tmem_ld32(lanes + COL_S + half * 64, s0);
      tmem_ld32(lanes + COL_S + half * 64 + 32, s1);
      tmem_ld32(lanes + COL_DP + half * 64, p0);
      tmem_ld32(lanes + COL_DP + half * 64 + 32, p1);
      tmem_ld_wait(s0);
      reg_fence32(s1);
      reg_fence32(p0);
      reg_fence32(p1);
      tc_fence_before();
      mbar_arrive(sdp_free);
      // keys past the end need no mask: their K rows are zero, so they add
      // nothing to dS·K; on the causal diagonal keep keys ≤ the query
      uint32_t pk[32];
      ds_chunk(s0, p0, c, l2, dd, pk);
      ds_chunk(s1, p1, c, l2, dd, pk + 16);
      if (a.causal && jb * 128 == q0) keep_upto(pk, r - half * 64);
      // the dS buffer is free once dQ += dS_{j-2}·K_{j-2} has completed
      if (jb >= 2 && !mbar_wait_warp(&ds_free[bb], ((jb - 2) >> 1) & 1,
                                     abort_flag, a.status, 37)) {
        ok = false;
        break;
      }
      st_row8(sm + OFF_DS + bb * TILE + half * A128, r, pk);
      fence_proxy_async_smem();
      mbar_arrive(&ds_full[bb]);
    }
    if (__all_sync(0xffffffffu, ok) &&
        mbar_wait_warp(dq_done, 0, abort_flag, a.status, 38)) {
      tc_fence_after();
      uint32_t o0[32], o1[32];
      tmem_ld32(lanes + COL_DQ + half * 64, o0);
      tmem_ld32(lanes + COL_DQ + half * 64 + 32, o1);
      tmem_ld_wait(o0);
      reg_fence32(o1);
      if (qi < a.s)
        store_bf16_row64(a.out0 + ((int64_t)b * a.s + qi) * (int64_t)(a.nq * HD) +
                             j * HD + half * 64,
                         o0, o1, a.scale);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
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
  uint64_t* ds_free = ds_full + 1;     // dK += dSᵀ·Q done with it
  uint64_t* done = ds_free + 1;
  uint64_t* drain = done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 1-D grid, block rank slowest: the heaviest (first, under the causal
  // mask) key blocks of every kv head start first; in (kv head, key block)
  // order the last heads' heavy blocks would start late and set the tail
  const int nblk = (a.s + 127) / 128;
  const int per = gridDim.x / nblk;   // n_kv · batch
  const int rank = blockIdx.x / per, rem = blockIdx.x % per;
  const int b = rem / a.nkv, kvh = rem % a.nkv;
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
    mbar_init(ds_free, 1);
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
      // per block: Sᵀ(it); dPᵀ(it) as soon as Sᵀ(it) is in registers; dK of
      // it−1 (its dSᵀ was written while Sᵀ(it) ran); dV of it (Pᵀ(it) is
      // written while dPᵀ(it) and dK(it−1) run)
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
        if (it > 0 && !(ok = dk_mma(it - 1))) break;
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
      // queries past the end have L2 = +∞ (P = 0); keys past the end feed
      // only dK, dV rows that are never stored; the causal diagonal block
      // keeps queries ≥ the key
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

int flash_bwd(const AttnShape& sh, const void* Q, const void* K, const void* V,
              const void* O, const void* dO, const float* LSE, float* Dp,
              float* L2p, void* dQ, void* dK, void* dV, unsigned* status,
              void* stream) {
  if (sh.d != HD) return cudaErrorInvalidValue;
  static cudaError_t e1 = cudaFuncSetAttribute(
      attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      dq::SMEM);
  static cudaError_t e2 = cudaFuncSetAttribute(
      attn_bwd_dkdv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      dkv::SMEM);
  if (e1 != cudaSuccess) return e1;
  if (e2 != cudaSuccess) return e2;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t s_pad = attn_stats_pad(sh.s);
  const double sd = (double)sh.s;
  const double pairs = sh.causal ? sd * (sd + 1.0) / 2.0 : sd * sd;
  const double core = 4.0 * sh.b * sh.nq * HD * pairs;
  const double io = 2.0 * sh.b * sh.s * HD;
  {
    const int64_t warps = sh.b * sh.nq * s_pad;
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
  a.s = (int)sh.s;
  a.s_pad = (int)s_pad;
  a.nq = sh.nq;
  a.nkv = sh.nkv;
  a.causal = sh.causal;
  a.scale = sh.scale;
  a.scale_log2 = sh.scale * LOG2E_F;
  a.status = status;
  a.out0 = static_cast<__nv_bfloat16*>(dQ);
  {
    const unsigned grid = (unsigned)(((sh.s + 127) / 128) * sh.nq * sh.b);
    ProfScope ps(stream, KF_ATTN_BWD_DQ, 0.5 * core,
                 io * (3.0 * sh.nq + 2.0 * sh.nkv));
    attn_bwd_dq_tc_kernel<<<grid, THREADS, dq::SMEM, s>>>(a);
  }
  a.out0 = static_cast<__nv_bfloat16*>(dK);
  a.out1 = static_cast<__nv_bfloat16*>(dV);
  {
    const unsigned grid = (unsigned)(((sh.s + 127) / 128) * sh.nkv * sh.b);
    ProfScope ps(stream, KF_ATTN_BWD_DKDV, 1.5 * core,
                 io * (2.0 * sh.nq + 4.0 * sh.nkv));
    attn_bwd_dkdv_tc_kernel<<<grid, THREADS, dkv::SMEM, s>>>(a);
  }
  count_launch(3);
  return cudaGetLastError();
}

}  // namespace tp
