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
//             group and block of 64 queries at or after the keys
//               Sᵀ = K·Qᵀ, dPᵀ = V·dOᵀ          (M=128, N=64, K=128) → TMEM
//               dV += Pᵀ·dO,  dK += dSᵀ·Q        (M=128, N=128, K=64) → TMEM
// Both: warp 0 TMA, warp 1 TMEM allocation + single-thread MMA issue, warps
// 2–9 elementwise (two threads per TMEM lane, half of the columns each).
// The score MMAs of the next block are issued as soon as the elementwise
// warps have copied the current scores to registers, ahead of the gradient
// MMAs, so the tensor cores work while the elementwise warps do.  K and V
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
constexpr int A64 = 64 * 128;     // one 64-column half of a 64-row tile
constexpr int THREADS = 320;
constexpr uint32_t TMEM_COLS = 512;
constexpr float LN2 = 0.69314718055994531f;
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
// K-major operand with K = 64 (one 128-byte-wide half).
__device__ __forceinline__ uint64_t dk64(uint32_t base, int kk) {
  return smem_desc_sw128(base + kk * 32, 16, 1024);
}
// MN-major B: rows are K, N = 128 in two 64-wide halves `atom` bytes apart.
__device__ __forceinline__ uint64_t dmn(uint32_t base, int kk, int atom) {
  return smem_desc_sw128(base + kk * 2048, atom, 1024);
}

// Write 32 fp16 values (16 packed words) as four 16-byte chunks of row r of
// a K-major swizzled tile whose rows are 128 bytes (64 columns), starting at
// 8-column chunk `c0`.
__device__ __forceinline__ void st_row_chunks(uint8_t* tile, int r, int c0,
                                              const uint32_t (&pk)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(tile + r * 128 + (((c0 + q) ^ (r & 7)) << 4)) =
        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
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
// bf16) and L2 = LSE·log2e; zeros past the sequence end.
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
    L2p[w] = pos < s ? LSE[bh * s + pos] * LOG2E_F : 0.0f;
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

// dS for 32 keys of one query row: P = exp2(S·c − L2) (0 past the last key
// this row may see), dS = P·(dP − D), packed in fp16 pairs.
__device__ __forceinline__ void ds_chunk(const uint32_t (&sv)[32],
                                         const uint32_t (&pv)[32], float c,
                                         float l2, float dd, bool masked,
                                         int k0, int kmax, uint32_t* pk) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    float p0 = ex2_approx(fmaf(__uint_as_float(sv[i]), c, -l2));
    float p1 = ex2_approx(fmaf(__uint_as_float(sv[i + 1]), c, -l2));
    if (masked) {
      p0 = (k0 + i <= kmax) ? p0 : 0.0f;
      p1 = (k0 + i + 1 <= kmax) ? p1 : 0.0f;
    }
    pk[i >> 1] = pack_f16x2(p0 * (__uint_as_float(pv[i]) - dd),
                            p1 * (__uint_as_float(pv[i + 1]) - dd));
  }
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
  const int b = blockIdx.z, j = blockIdx.y;
  const int q0 = (gridDim.x - 1 - blockIdx.x) * 128;
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
    const int kmax = a.causal ? min(qi, a.s - 1) : a.s - 1;
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
      const int k0 = jb * 128 + half * 64;
      const bool masked =
          (jb * 128 + 128 > a.s) || (a.causal && jb * 128 + 127 > q0);
      uint32_t pk[32];
      ds_chunk(s0, p0, c, l2, dd, masked, k0, kmax, pk);
      ds_chunk(s1, p1, c, l2, dd, masked, k0 + 32, kmax, pk + 16);
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
constexpr int OFF_K = 0;
constexpr int OFF_V = 2 * A128;
constexpr int OFF_QS = 4 * A128;                 // NST stages
constexpr int STAGE = 4 * A64;                   // Q 16 KB, dO 16 KB
constexpr int NST = 4;
constexpr int OFF_P = OFF_QS + NST * STAGE;      // 16 KB
constexpr int OFF_DS = OFF_P + A128;             // 16 KB
constexpr int OFF_ST = OFF_DS + A128;            // NST × (64 L2, 64 D) fp32
constexpr int OFF_BAR = OFF_ST + NST * 512;
// No alignment slack: the kernel checks that the dynamic shared memory
// starts on a 1024-byte boundary (as the 128-byte swizzle requires).
constexpr int SMEM = OFF_BAR + 256;
constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 384;
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
  uint64_t* kv_full = bar;         // K and V
  uint64_t* qs_full = bar + 1;     // [NST] Q, dO, stats
  uint64_t* qs_empty = bar + 5;    // [NST]
  uint64_t* sdp_full = bar + 9;    // [2]
  uint64_t* sdp_free = bar + 11;   // [2] Sᵀ, dPᵀ copied to registers
  uint64_t* pds_full = bar + 13;   // Pᵀ and dSᵀ written
  uint64_t* pds_free = bar + 14;   // gradient MMAs done with them
  uint64_t* done = bar + 15;
  uint64_t* drain = bar + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int k0 = blockIdx.x * 128;
  const int group = a.nq / a.nkv;
  const int nqb = (a.s + 63) / 64;
  const int qb_first = a.causal ? k0 / 64 : 0;
  const int per_head = nqb - qb_first;
  const int iters = per_head * group;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int i = 0; i < NST; ++i) {
      mbar_init(&qs_full[i], 1);
      mbar_init(&qs_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sdp_full[i], 1);
      mbar_init(&sdp_free[i], 256);
    }
    mbar_init(pds_full, 256);
    mbar_init(pds_free, 1);
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
    if (lane == 0) {
      tma_prefetch_desc(&a.mq);
      tma_prefetch_desc(&a.mdo);
      tma_prefetch_desc(&a.mk);
      tma_prefetch_desc(&a.mv);
      uint32_t armed = 0, armed_par = 0;
      mbar_arrive_expect_tx(kv_full, 4 * A128);
      for (int hh = 0; hh < 2; ++hh) {
        tma_load_3d(sm + OFF_K + hh * A128, &a.mk, kv_full, kvh * HD + hh * 64,
                    k0, b);
        tma_load_3d(sm + OFF_V + hh * A128, &a.mv, kv_full, kvh * HD + hh * 64,
                    k0, b);
      }
      for (int it = 0; it < iters; ++it) {
        const int st = it % NST;
        const uint32_t ph = (it / NST) & 1;
        if (!mbar_wait(&qs_empty[st], ph ^ 1, abort_flag, a.status, 41)) break;
        const int jq = kvh * group + it / per_head;
        const int qb = qb_first + it % per_head;
        mbar_arrive_expect_tx(&qs_full[st], 4 * A64 + 512);
        armed |= 1u << st;
        armed_par = (armed_par & ~(1u << st)) | (ph << st);
        uint8_t* stg = sm + OFF_QS + st * STAGE;
        for (int hh = 0; hh < 2; ++hh) {
          tma_load_3d(stg + hh * A64, &a.mq, &qs_full[st], jq * HD + hh * 64,
                      qb * 64, b);
          tma_load_3d(stg + 2 * A64 + hh * A64, &a.mdo, &qs_full[st],
                      jq * HD + hh * 64, qb * 64, b);
        }
        const int64_t soff = ((int64_t)b * a.nq + jq) * a.s_pad + qb * 64;
        uint8_t* sst = sm + OFF_ST + st * 512;
        bulk_load(sst, a.L2p + soff, 256, &qs_full[st]);
        bulk_load(sst + 256, a.Dp + soff, 256, &qs_full[st]);
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        mbar_wait(kv_full, 0, &no_abort, nullptr, 0);
        for (int st = 0; st < NST; ++st)
          if (armed & (1u << st))
            mbar_wait(&qs_full[st], (armed_par >> st) & 1u, &no_abort, nullptr,
                      0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC_S = idesc_f16_f32(128, 64, 0, 0);
      constexpr uint32_t IDESC_G = idesc_f16_f32(128, 128, 0, 1);
      const uint32_t sK = smem_u32(sm + OFF_K), sV = smem_u32(sm + OFF_V);
      bool ok = mbar_wait(kv_full, 0, abort_flag, a.status, 42);
      // Sᵀ and dPᵀ run two iterations ahead of the gradient MMAs
      auto sdp_mma = [&](int it) -> bool {
        const int st = it % NST, bb = it & 1;
        if (!mbar_wait(&qs_full[st], (it / NST) & 1, abort_flag, a.status, 44))
          return false;
        tc_fence_after();
        const uint32_t stg = smem_u32(sm + OFF_QS + st * STAGE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {   // the two chains interleaved
          tc_mma_f16(tmem + COL_S + bb * 64, dk128(sK, kk, A128),
                     dk128(stg, kk, A64), IDESC_S, kk > 0 ? 1u : 0u);
          tc_mma_f16(tmem + COL_DP + bb * 64, dk128(sV, kk, A128),
                     dk128(stg + 2 * A64, kk, A64), IDESC_S, kk > 0 ? 1u : 0u);
        }
        tc_commit(&sdp_full[bb]);
        return true;
      };
      auto grads = [&](int i) -> bool {
        const int st = i % NST;
        if (!mbar_wait(pds_full, i & 1, abort_flag, a.status, 43)) return false;
        tc_fence_after();
        const uint32_t stg = smem_u32(sm + OFF_QS + st * STAGE);
        const uint32_t sP = smem_u32(sm + OFF_P);
        const uint32_t sdS = smem_u32(sm + OFF_DS);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {   // the two chains interleaved
          tc_mma_f16(tmem + COL_DV, dk64(sP, kk), dmn(stg + 2 * A64, kk, A64),
                     IDESC_G, (i > 0 || kk > 0) ? 1u : 0u);
          tc_mma_f16(tmem + COL_DK, dk64(sdS, kk), dmn(stg, kk, A64), IDESC_G,
                     (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(pds_free);
        tc_commit(&qs_empty[st]);
        return true;
      };
      if (ok) ok = sdp_mma(0);
      if (ok && iters > 1) ok = sdp_mma(1);
      for (int it = 0; ok && it < iters; ++it) {
        if (it + 2 < iters) {
          ok = mbar_wait(&sdp_free[it & 1], (it >> 1) & 1, abort_flag,
                         a.status, 45) &&
               sdp_mma(it + 2);
          if (!ok) break;
        }
        ok = grads(it);
      }
      if (ok) tc_commit(done);
      if (*abort_flag) {
        volatile int no_abort = 0;
        tc_commit(drain);
        mbar_wait(drain, 0, &no_abort, nullptr, 0);
      }
    }
  } else {
    // ------------------------------------------------------ elementwise --
    const int half = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int key = k0 + r;
    const uint32_t lanes = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float c = a.scale_log2;
    bool ok = true;
    for (int it = 0; it < iters; ++it) {
      const int st = it & 1;
      if (!mbar_wait_warp(&sdp_full[st], (it >> 1) & 1, abort_flag, a.status,
                          46)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[32], pv[32];
      tmem_ld32(lanes + COL_S + st * 64 + half * 32, sv);
      tmem_ld32(lanes + COL_DP + st * 64 + half * 32, pv);
      tmem_ld_wait(sv);
      reg_fence32(pv);
      tc_fence_before();
      mbar_arrive(&sdp_free[st]);
      const int qb = qb_first + it % per_head;
      const int qc0 = qb * 64 + half * 32;   // first query column of this half
      const float* stats =
          reinterpret_cast<const float*>(sm + OFF_ST + (it % NST) * 512);
      const bool masked = (qb * 64 + 64 > a.s) || (k0 + 128 > a.s) ||
                          (a.causal && qb * 64 < k0 + 127);
      uint32_t pp[16], pd[16];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(stats + half * 32 + i);
        const float4 d4 =
            *reinterpret_cast<const float4*>(stats + 64 + half * 32 + i);
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
        const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
        float p[4], ds[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          p[e] = ex2_approx(fmaf(__uint_as_float(sv[i + e]), c, -lv[e]));
          if (masked) {
            const int q = qc0 + i + e;
            const bool valid =
                q < a.s && key < a.s && (!a.causal || key <= q);
            p[e] = valid ? p[e] : 0.0f;
          }
          ds[e] = p[e] * (__uint_as_float(pv[i + e]) - dv[e]);
        }
        pp[i >> 1] = pack_f16x2(p[0], p[1]);
        pp[(i >> 1) + 1] = pack_f16x2(p[2], p[3]);
        pd[i >> 1] = pack_f16x2(ds[0], ds[1]);
        pd[(i >> 1) + 1] = pack_f16x2(ds[2], ds[3]);
      }
      // the P / dS tiles are free once the gradient MMAs of it−1 finished
      if (it >= 1 && !mbar_wait_warp(pds_free, (it - 1) & 1, abort_flag,
                                     a.status, 47)) {
        ok = false;
        break;
      }
      st_row_chunks(sm + OFF_P, r, half * 4, pp);
      st_row_chunks(sm + OFF_DS, r, half * 4, pd);
      fence_proxy_async_smem();
      mbar_arrive(pds_full);
    }
    if (iters > 0 && __all_sync(0xffffffffu, ok) &&
        mbar_wait_warp(done, 0, abort_flag, a.status, 48)) {
      tc_fence_after();
      const int64_t ldk = (int64_t)a.nkv * HD;
      const int64_t row = ((int64_t)b * a.s + key) * ldk + kvh * HD + half * 64;
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
  // Q and dO in 64-row boxes (the dK/dV kernel), K and V in 128-row boxes
  const uint64_t ldq = (uint64_t)sh.nq * HD * 2, ldk = (uint64_t)sh.nkv * HD * 2;
  const bool ok =
      encode_tmap_3d_f16(&a.mq, Q, (uint64_t)sh.nq * HD, sh.s, sh.b, ldq,
                         ldq * sh.s, 64, 64, 1) &&
      encode_tmap_3d_f16(&a.mdo, dO, (uint64_t)sh.nq * HD, sh.s, sh.b, ldq,
                         ldq * sh.s, 64, 64, 1) &&
      encode_tmap_3d_f16(&a.mk, K, (uint64_t)sh.nkv * HD, sh.s, sh.b, ldk,
                         ldk * sh.s, 64, 128, 1) &&
      encode_tmap_3d_f16(&a.mv, V, (uint64_t)sh.nkv * HD, sh.s, sh.b, ldk,
                         ldk * sh.s, 64, 128, 1);
  if (!ok) return cudaErrorInvalidValue;
  a.q = static_cast<const __half*>(Q);
  a.dout = static_cast<const __half*>(dO);
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
    dim3 grid((unsigned)((sh.s + 127) / 128), (unsigned)sh.nq, (unsigned)sh.b);
    ProfScope ps(stream, KF_ATTN_BWD_DQ, 0.5 * core,
                 io * (3.0 * sh.nq + 2.0 * sh.nkv));
    attn_bwd_dq_tc_kernel<<<grid, THREADS, dq::SMEM, s>>>(a);
  }
  a.out0 = static_cast<__nv_bfloat16*>(dK);
  a.out1 = static_cast<__nv_bfloat16*>(dV);
  {
    dim3 grid((unsigned)((sh.s + 127) / 128), (unsigned)sh.nkv,
              (unsigned)sh.b);
    ProfScope ps(stream, KF_ATTN_BWD_DKDV, 1.5 * core,
                 io * (2.0 * sh.nq + 4.0 * sh.nkv));
    attn_bwd_dkdv_tc_kernel<<<grid, THREADS, dkv::SMEM, s>>>(a);
  }
  count_launch(3);
  return cudaGetLastError();
}

}  // namespace tp
