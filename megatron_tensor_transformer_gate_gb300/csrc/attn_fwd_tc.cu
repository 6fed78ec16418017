// attn_fwd_tc.cu — causal GQA flash-attention forward on tcgen05 / TMEM.
//
// The attention core of one rank's local heads ([Grasp-TP] §4: softmax per
// head over the sequence; [Troverld] §I.O FlashAttention: row-blocked with an
// online softmax, O(S) statistics written for the backward pass).
//
// One CTA = 128 query rows of one (batch, q head); 192 threads:
//   warp 0     TMA: the Q tile once, then K_j and V_j (128 keys each) into
//              two independent 2-stage rings (fp16, 128-byte swizzle, two
//              64-column halves); lane 0 feeds K, lane 1 feeds V.
//   warp 1     allocates 512 TMEM columns and issues, per key block j,
//                S_j = Q·K_jᵀ   (M=128, N=128, K=128) into TMEM S[j mod 2]
//                O += P_j·V_j   (M=128, N=128, K=128) into TMEM O, with
//                               P_j read from TMEM P[j mod 2]
//              with the scores two blocks ahead (S_0, S_1, S_2, PV_0, S_3,
//              PV_1, …) so the tensor cores never wait for a softmax block.
//   warps 2–9  softmax, two threads per query row (same TMEM lane, one per
//              64-column half), reference
//              max m and sum l in fp32, P_j = exp2(S·scale·log2e − m) stored
//              as fp16 pairs into TMEM (double-buffered, so block j+1 is
//              written while O += P_j·V_j runs).
//              O accumulates in TMEM; when a block's max exceeds
//              m by more than 2^8 the softmax rescales O and l by
//              exp2(m − m_new) first.  The epilogue writes O / l (bf16) and
//              LSE = (m + log2 l)·ln 2.
// Operands are fp16 and accumulation fp32: the softmax amplifies score
// errors, and bf16 operands (8-bit mantissa) put the row-wise error of causal
// outputs above 3e-2 of the row rms, while fp16 (10-bit mantissa, same bytes)
// stays near the bf16 output-rounding floor.  Q, K, V (and dO) are written in
// fp16 by the projection GEMMs; O is written in bf16 for the bf16 out-
// projection GEMM.
#include <cuda_fp16.h>

#include <cstring>

#include "attention.h"
#include "common.cuh"
#include "gemm.h"
#include "profile.h"

namespace tp {
namespace {

constexpr int HD = 128;
constexpr int BLK = 128;                 // queries per CTA, keys per block
constexpr int ATOM = BLK * 128;          // one 64-column half: 128 rows × 128 B
constexpr int TILE = 2 * ATOM;           // 32 KB fp16 tile [128][128]
constexpr int THREADS = 320;   // TMA, MMA, 8 softmax warps
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE;      // 2 stages
constexpr int OFF_V = OFF_K + 2 * TILE;  // 2 stages
constexpr int OFF_BAR = OFF_V + 2 * TILE;
constexpr int OFF_RED = OFF_BAR + 256;   // row-max / row-sum exchange
constexpr int RED_SLOTS = 3;             // 2 for block parity, 1 for the end
constexpr int OFF_SEQ = OFF_RED + RED_SLOTS * 2 * 128 * 4;
constexpr int SMEM = OFF_SEQ + RED_SLOTS * 2 * 128 * 4 + 1024;
constexpr uint32_t TMEM_COLS = 512;
// TMEM: S[2] in columns 0-255, O in 256-383, P[2] (fp16 pairs, the A
// operand of O += P·V) in 384-511.
constexpr uint32_t COL_O = 256, COL_P = 384;
// The output accumulates in TMEM against a reference max m; it is rescaled
// only when a block's row max exceeds m by more than this (log2 units), which
// keeps the fp16 probabilities ≤ 2^8 and the fp32 accumulator far from
// overflow.
constexpr float RESCALE_LOG2 = 8.0f;

// Exchange of one float between the two threads that own a query row: write
// this thread's value with a sequence tag, then wait (bounded, abort-aware)
// until the partner's entry carries the same tag.  Returns false when it gave
// up.
__device__ __forceinline__ bool pair_exchange(float* val, int* seq, int self,
                                              int other, float mine, int tag,
                                              float* theirs,
                                              volatile int* abort_flag,
                                              unsigned* status) {
  val[self] = mine;
  __threadfence_block();
  reinterpret_cast<volatile int*>(seq)[self] = tag;
  volatile int* ps = reinterpret_cast<volatile int*>(seq) + other;
  if (*ps != tag) {
    const long long t0 = clock64();
    while (*ps != tag) {
      if (*abort_flag) return false;
      if (clock64() - t0 > kWaitTimeoutCycles) {
        record_error(status, kDevTimeout, 20);
        *abort_flag = 1;
        return false;
      }
    }
  }
  __threadfence_block();
  *theirs = reinterpret_cast<volatile float*>(val)[other];
  return true;
}

struct FwdTcArgs {
  CUtensorMap mq, mk, mv;
  __nv_bfloat16* O;
  float* LSE;
  int s, nq, nkv, causal;
  float scale_log2;
  unsigned* status;
};

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int kk) {
  // K-major tile of two 64-column halves: K step kk (16 columns)
  return smem_desc_sw128(base + (kk >> 2) * ATOM + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int kk) {
  // MN-major B (V: rows = keys = K, two 64-wide d halves ATOM apart)
  return smem_desc_sw128(base + kk * 2048, ATOM, 1024);
}

__global__ void __launch_bounds__(THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ FwdTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* k_full = bar + 1;     // [2]
  uint64_t* k_empty = bar + 3;    // [2]
  uint64_t* v_full = bar + 5;     // [2]
  uint64_t* v_empty = bar + 7;    // [2]
  uint64_t* s_full = bar + 9;     // [2]
  uint64_t* s_free = bar + 11;    // [2] scores copied to registers
  uint64_t* p_full = bar + 13;    // [2]
  uint64_t* pv_done = bar + 15;   // [2]
  uint64_t* drain = bar + 17;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 18);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 1-D grid, block rank slowest: the heaviest (last, under the causal
  // mask) query blocks of every head start first, which shortens the tail
  const int nblk = (a.s + BLK - 1) / BLK;
  const int per = gridDim.x / nblk;   // n_q · batch
  const int rank = blockIdx.x / per, rem = blockIdx.x % per;
  const int b = rem / a.nq, j = rem % a.nq;
  const int q0 = (nblk - 1 - rank) * BLK;
  const int kvh = j / (a.nq / a.nkv);
  const int kv_end = a.causal ? min(a.s, q0 + BLK) : a.s;
  const int nkb = (kv_end + BLK - 1) / BLK;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 256);
      mbar_init(&p_full[i], 256);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < RED_SLOTS * 2 * 128; i += THREADS)
    reinterpret_cast<int*>(sm + OFF_SEQ)[i] = 0;
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane < 2) {
      // ------------------------------------------------------------- TMA --
      // lane 0: Q, then the K ring; lane 1: the V ring.  K_j is released as
      // soon as S_j is done, V_j only after O += P_j·V_j, so the two rings
      // advance independently.
      const bool is_k = lane == 0;
      const CUtensorMap* map = is_k ? &a.mk : &a.mv;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* ring = sm + (is_k ? OFF_K : OFF_V);
      tma_prefetch_desc(map);
      uint32_t armed = 0, armed_par = 0;
      if (is_k) {
        tma_prefetch_desc(&a.mq);
        mbar_arrive_expect_tx(q_full, TILE);
        for (int hh = 0; hh < 2; ++hh)
          tma_load_3d(sm + OFF_Q + hh * ATOM, &a.mq, q_full, j * HD + hh * 64,
                      q0, b);
      }
      for (int jb = 0; jb < nkb; ++jb) {
        const int st = jb & 1;
        const uint32_t ph = (jb >> 1) & 1;
        if (!mbar_wait(&empty[st], ph ^ 1, abort_flag, a.status, 11)) break;
        mbar_arrive_expect_tx(&full[st], TILE);
        armed |= 1u << st;
        armed_par = (armed_par & ~(1u << st)) | (ph << st);
        for (int hh = 0; hh < 2; ++hh)
          tma_load_3d(ring + st * TILE + hh * ATOM, map, &full[st],
                      kvh * HD + hh * 64, jb * BLK, b);
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        if (is_k) mbar_wait(q_full, 0, &no_abort, nullptr, 0);
        for (int st = 0; st < 2; ++st)
          if (armed & (1u << st))
            mbar_wait(&full[st], (armed_par >> st) & 1u, &no_abort, nullptr, 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMA --
      // Score tiles run two blocks ahead of O += P·V: S_{j+2} is issued as
      // soon as the softmax has copied S_j to registers, so the tensor
      // cores never wait for the softmax to finish a block.
      constexpr uint32_t IDESC_S = idesc_f16_f32(128, 128, 0, 0);
      constexpr uint32_t IDESC_O = idesc_f16_f32(128, 128, 0, 1);
      const uint32_t sQ = smem_u32(sm + OFF_Q);
      bool ok = mbar_wait(q_full, 0, abort_flag, a.status, 12);
      auto s_mma = [&](int jb) -> bool {
        const int st = jb & 1;
        if (!mbar_wait(&k_full[st], (jb >> 1) & 1, abort_flag, a.status, 15))
          return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(sm + OFF_K + st * TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(tmem + st * 128, desc_kmajor(sQ, kk), desc_kmajor(sK, kk),
                     IDESC_S, kk > 0 ? 1u : 0u);
        tc_commit(&s_full[st]);
        tc_commit(&k_empty[st]);
        return true;
      };
      // O += P_i·V_i; the softmax rescaled O (if needed) before p_full[i]
      auto pv = [&](int i) -> bool {
        if (!mbar_wait(&p_full[i & 1], (i >> 1) & 1, abort_flag, a.status, 13) ||
            !mbar_wait(&v_full[i & 1], (i >> 1) & 1, abort_flag, a.status, 14))
          return false;
        tc_fence_after();
        const uint32_t sV = smem_u32(sm + OFF_V + (i & 1) * TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16_ts(tmem + COL_O, tmem + COL_P + (i & 1) * 64 + kk * 8,
                        desc_mnmajor(sV, kk), IDESC_O,
                        (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&pv_done[i & 1]);
        tc_commit(&v_empty[i & 1]);
        return true;
      };
      if (ok) ok = s_mma(0);
      if (ok && nkb > 1) ok = s_mma(1);
      for (int jb = 0; ok && jb < nkb; ++jb) {
        if (jb + 2 < nkb) {
          ok = mbar_wait(&s_free[jb & 1], (jb >> 1) & 1, abort_flag, a.status,
                         16) &&
               s_mma(jb + 2);
          if (!ok) break;
        }
        ok = pv(jb);
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        tc_commit(drain);
        mbar_wait(drain, 0, &no_abort, nullptr, 0);
      }
    }
  } else {
    // --------------------------------------------------------- softmax --
    // Two warps per row: `half` 0 owns key columns and output columns 0-63,
    // half 1 owns 64-127; the two threads of a row (same TMEM lane) exchange
    // the row max through shared memory each block, tagged with the block
    // index (slots alternate by block parity; slot 2 carries the final sums).
    const int sw = warp - 2;
    const int half = sw >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int qi = q0 + r;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* red = reinterpret_cast<float*>(sm + OFF_RED);  // [slot][half][row]
    int* seq = reinterpret_cast<int*>(sm + OFF_SEQ);
    const float c = a.scale_log2;
    const float thr = RESCALE_LOG2 / c;   // the rescale threshold in raw units
    float m_ref = -INFINITY, l_part = 0.0f;
    bool ok = true;
    for (int jb = 0; jb < nkb; ++jb) {
      const int st = jb & 1;
      if (!mbar_wait_warp(&s_full[st], (jb >> 1) & 1, abort_flag, a.status,
                          16)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[2][32];
      tmem_ld32(lane_base + st * 128 + half * 64, v[0]);
      tmem_ld32(lane_base + st * 128 + half * 64 + 32, v[1]);
      tmem_ld_wait(v[0]);
      reg_fence32(v[1]);
      tc_fence_before();
      mbar_arrive(&s_free[st]);   // S buffer st may take S_{j+2} now
      const int k0 = jb * BLK + half * 64;
      if ((jb + 1) * BLK > a.s || (a.causal && (jb + 1) * BLK - 1 > q0)) {
        // diagonal or ragged block: invalid keys become −inf (branch-free)
        const int kmax = a.causal ? min(qi, a.s - 1) : a.s - 1;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            v[cc][i] = (k0 + cc * 32 + i <= kmax) ? v[cc][i]
                                                  : __float_as_uint(-INFINITY);
      }
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        mx8[i] = fmaxf(__uint_as_float(v[0][i]), __uint_as_float(v[0][i + 8]));
#pragma unroll
      for (int i = 16; i < 64; ++i)
        mx8[i & 7] = fmaxf(mx8[i & 7], __uint_as_float(v[i >> 5][i & 31]));
      float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      float mx_other;
      const bool got = pair_exchange(red, seq, (st * 2 + half) * 128 + r,
                                     (st * 2 + (half ^ 1)) * 128 + r, mx,
                                     jb + 1, &mx_other, abort_flag, a.status);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, mx_other);
      if (jb == 0) {
        m_ref = mx;
      } else if (__any_sync(0xffffffffu, mx > m_ref + thr)) {
        // rescale this warp's half of the TMEM accumulator once
        // O += P_{j-1}·V_{j-1} has landed; the whole warp takes part (TMEM
        // access is warp-collective), rows that keep their reference scale
        // by 1.  Both warps of a pair see the same rows and decide alike.
        const int pj = jb - 1;
        if (!mbar_wait_warp(&pv_done[pj & 1], (pj >> 1) & 1, abort_flag,
                            a.status, 17)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float m_new = mx > m_ref + thr ? mx : m_ref;
        const float alpha = ex2_approx((m_ref - m_new) * c);
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t o[32];
          const uint32_t ta = lane_base + COL_O + half * 64 + cc * 32;
          tmem_ld32(ta, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(ta, o);
        }
        l_part *= alpha;
        m_ref = m_new;
      }
      // P buffer st is free once O += P_{j-2}·V_{j-2} has completed
      if (jb >= 2 && !mbar_wait_warp(&pv_done[st], ((jb - 2) >> 1) & 1,
                                     abort_flag, a.status, 18)) {
        ok = false;
        break;
      }
      // P = exp2(c·(s − m)) in fp16 pairs into this half's 32 columns of P[st]
      const float neg = -m_ref * c;
      float sum8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) sum8[i] = 0.0f;
      uint32_t pk[32];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(v[cc][i]), c, neg));
          const float p1 =
              ex2_approx(fmaf(__uint_as_float(v[cc][i + 1]), c, neg));
          sum8[i & 7] += p0;
          sum8[(i + 1) & 7] += p1;
          pk[cc * 16 + (i >> 1)] = pack_f16x2(p0, p1);
        }
      }
      tmem_st32(lane_base + COL_P + st * 64 + half * 32, pk);
      l_part += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
                ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      tc_fence_before();
      mbar_arrive(&p_full[st]);
    }
    // epilogue: the row sum is the two halves' partial sums; wait for the
    // last O += P·V, then O / l for this warp's 64 columns and the LSE
    float l_other = 0.0f;
    if (__all_sync(0xffffffffu, ok))
      ok = pair_exchange(red, seq, (4 + half) * 128 + r,
                         (4 + (half ^ 1)) * 128 + r, l_part, nkb + 1, &l_other,
                         abort_flag, a.status);
    const int last = nkb - 1;
    if (__all_sync(0xffffffffu, ok) &&
        mbar_wait_warp(&pv_done[last & 1], (last >> 1) & 1, abort_flag,
                       a.status, 19)) {
      tc_fence_after();
      const float l_run = l_part + l_other;
      const float inv = 1.0f / l_run;
      __nv_bfloat16* dst = a.O + ((int64_t)b * a.s + qi) * (int64_t)(a.nq * HD) +
                           j * HD + half * 64;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t o[32];
        tmem_ld32(lane_base + COL_O + half * 64 + cc * 32, o);
        tmem_ld_wait(o);
        if (qi < a.s) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 u;
            u.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv,
                              __uint_as_float(o[8 * q + 1]) * inv);
            u.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv,
                              __uint_as_float(o[8 * q + 3]) * inv);
            u.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv,
                              __uint_as_float(o[8 * q + 5]) * inv);
            u.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv,
                              __uint_as_float(o[8 * q + 7]) * inv);
            reinterpret_cast<uint4*>(dst)[cc * 4 + q] = u;
          }
        }
      }
      if (half == 0 && qi < a.s)
        a.LSE[((int64_t)b * a.nq + j) * a.s + qi] =
            (m_ref * c + log2f(l_run)) * 0.69314718055994531f;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

int flash_fwd(const AttnShape& sh, const void* Q, const void* K, const void* V,
              void* O, float* LSE, unsigned* status, void* stream) {
  if (sh.d != HD) return cudaErrorInvalidValue;
  static cudaError_t e = cudaFuncSetAttribute(
      attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  FwdTcArgs a;
  memset(&a, 0, sizeof(a));
  const uint64_t ldq = (uint64_t)sh.nq * HD * 2, ldk = (uint64_t)sh.nkv * HD * 2;
  // dims {columns, positions, batch}: rows past a sequence's end read as zero
  if (!encode_tmap_3d_f16(&a.mq, Q, (uint64_t)sh.nq * HD, sh.s, sh.b, ldq,
                          ldq * sh.s, 64, BLK, 1) ||
      !encode_tmap_3d_f16(&a.mk, K, (uint64_t)sh.nkv * HD, sh.s, sh.b, ldk,
                          ldk * sh.s, 64, BLK, 1) ||
      !encode_tmap_3d_f16(&a.mv, V, (uint64_t)sh.nkv * HD, sh.s, sh.b, ldk,
                          ldk * sh.s, 64, BLK, 1))
    return cudaErrorInvalidValue;
  a.O = static_cast<__nv_bfloat16*>(O);
  a.LSE = LSE;
  a.s = (int)sh.s;
  a.nq = sh.nq;
  a.nkv = sh.nkv;
  a.causal = sh.causal;
  a.scale_log2 = sh.scale * 1.4426950408889634f;
  a.status = status;
  const unsigned grid = (unsigned)(((sh.s + BLK - 1) / BLK) * sh.nq * sh.b);
  const double s = (double)sh.s;
  const double pairs = sh.causal ? s * (s + 1.0) / 2.0 : s * s;
  {
    ProfScope ps(stream, KF_ATTN_FWD, 4.0 * sh.b * sh.nq * HD * pairs,
                 2.0 * sh.b * sh.s * HD * (2.0 * sh.nq + 2.0 * sh.nkv));
    attn_fwd_tc_kernel<<<grid, THREADS, SMEM,
                         static_cast<cudaStream_t>(stream)>>>(a);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace tp
