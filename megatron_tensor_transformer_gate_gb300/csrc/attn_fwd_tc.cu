// attn_fwd_tc.cu — causal GQA flash-attention forward on tcgen05 / TMEM.
//
// The attention core of one rank's local heads ([Grasp-TP] §4: softmax per
// head over the sequence; [Troverld] §I.O FlashAttention: row-blocked with an
// online softmax, O(S) statistics written for the backward pass).
//
// One CTA = two query tiles of 128 rows that read the same keys and values:
// two q heads of one GQA group at the same query block when the group size is
// even, else two consecutive query blocks of one head.  320 threads:
//   warp 0     TMA: both Q tiles once, then K_0, K_1, V_0, K_2, V_1, … (the
//              order the MMAs use them) through one 3-slot ring (fp16,
//              128-byte swizzle, two 64-column halves per tile).
//   warp 1     allocates 512 TMEM columns (S of each tile, O of both) and
//              issues, per key block j,
//                S_t = Q_t·K_jᵀ     (M=128, N=128, K=128) into TMEM S[t],
//                                   for each tile t
//                Oᵀ += Vᵀ_j·Pᵀ      (M=128 features, N=256 queries of both
//                                   tiles, K=128 keys) into TMEM Oᵀ, P of
//                                   both tiles read from shared memory
//              S_t for block j+1 as soon as tile t's softmax has copied S_t
//              of block j to registers, so the scores of the next block are
//              computed while the softmax of this one runs.  The output is
//              accumulated transposed so that one N=256 instruction serves
//              both tiles: on this tensor core an M=128 instruction costs
//              nearly as much at N=128 as at N=256.
//   warps 2–9  softmax, one thread per query row (warps 2–5 tile 0, 6–9
//              tile 1): reference max m and sum l in fp32, P = exp2(S·scale·
//              log2e − m) stored as fp16 into the P buffer.  Oᵀ accumulates
//              in TMEM; when a block's max exceeds m by more than 2^12 the row
//              takes a new m, and its column of Oᵀ and l are scaled by
//              exp2(m − m_new) first (each thread holds one feature lane of
//              every column, so the factors pass through shared memory).  The
//              epilogue writes O / l (bf16) and LSE = (m + log2 l)·ln 2.
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
constexpr int BLK = 128;                 // queries per tile, keys per block
constexpr int ATOM = BLK * 128;          // one 64-column half: 128 rows × 128 B
constexpr int TILE = 2 * ATOM;           // 32 KB fp16 tile [128][128]
constexpr int NT = 2;                    // query tiles per CTA
constexpr int NSLOT = 3;                 // K/V ring slots
constexpr int THREADS = 64 + NT * 128;   // TMA warp, MMA warp, softmax rows
constexpr int OFF_Q = 0;                 // NT tiles
// P of both tiles as one 256-row K-major operand: half hh (keys 64·hh to
// 64·hh + 63) of tile t's row r at OFF_P + hh·2·ATOM + (128·t + r)·128.
constexpr int OFF_P = OFF_Q + NT * TILE;
constexpr int OFF_KV = OFF_P + NT * TILE;
constexpr int OFF_BAR = OFF_KV + NSLOT * TILE;
constexpr int OFF_COLF = OFF_BAR + 256;      // per-query factors, NT × 128 fp32
constexpr int SMEM = OFF_COLF + NT * BLK * 4 + 1024;   // + 1024-B alignment
constexpr uint32_t TMEM_COLS = 512;
// TMEM: S of tile t in columns [128·t, 128·t + 128); the output transposed,
// Oᵀ (lane = feature d, column = query), tile t's queries in columns
// [256 + 128·t, 384 + 128·t).
constexpr uint32_t COL_O = 256;
// The output accumulates in TMEM against a reference max m; it is rescaled
// only when a block's row max exceeds m by more than this (log2 units), which
// keeps the fp16 probabilities ≤ 2^12 (a factor 16 below the fp16 maximum)
// and the fp32 accumulator far from overflow.  A rescale makes the four warps
// of a tile wait for one another, and with scores of a few units of spread a
// 2^8 threshold let some row of a 128-row tile cross it in about a third of
// the key blocks, 2^12 in under 2 %.
constexpr float RESCALE_LOG2 = 12.0f;

struct FwdTcArgs {
  CUtensorMap mq, mk, mv;
  __nv_bfloat16* O;
  float* LSE;
  int s, nb, nq, nkv, causal, pair_heads;
  float scale_log2;
  unsigned* status;
};

// The CTA's two query tiles: batch, kv head, and per tile its q head, first
// query row and number of key blocks (0 for a tile past the sequence end).
// The 1-D grid has the block rank slowest, so the heaviest (last, under the
// causal mask) query blocks of every head start first.
struct Tiles {
  int b, kvh;
  int head[NT], q0[NT], nkb[NT];
};

__device__ __forceinline__ Tiles cta_tiles(const FwdTcArgs& a) {
  Tiles T;
  const int nblk = (a.s + BLK - 1) / BLK;
  if (a.pair_heads) {
    const int hp = a.nq / 2;
    const int per = a.nb * hp;
    const int rank = blockIdx.x / per, rem = blockIdx.x % per;
    T.b = rem / hp;
    for (int t = 0; t < NT; ++t) {
      T.head[t] = 2 * (rem % hp) + t;
      T.q0[t] = (nblk - 1 - rank) * BLK;
    }
  } else {
    const int npair = (nblk + 1) / 2;
    const int per = a.nb * a.nq;
    const int rank = blockIdx.x / per, rem = blockIdx.x % per;
    T.b = rem / a.nq;
    for (int t = 0; t < NT; ++t) {
      T.head[t] = rem % a.nq;
      T.q0[t] = (2 * (npair - 1 - rank) + t) * BLK;
    }
  }
  T.kvh = T.head[0] / (a.nq / a.nkv);
  for (int t = 0; t < NT; ++t) {
    const int kv_end = a.causal ? min(a.s, T.q0[t] + BLK) : a.s;
    T.nkb[t] = T.q0[t] < a.s ? (kv_end + BLK - 1) / BLK : 0;
  }
  return T;
}

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int kk) {
  // K-major tile of two 64-column halves: K step kk (16 columns)
  return smem_desc_sw128(base + (kk >> 2) * ATOM + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int kk) {
  // MN-major Vᵀ as A (rows = keys = K, M = d in two 64-wide halves ATOM apart)
  return smem_desc_sw128(base + kk * 2048, ATOM, 1024);
}
__device__ __forceinline__ uint64_t desc_p(uint32_t base, int kk) {
  // K-major P (rows = queries = N; its two key halves 2·ATOM apart)
  return smem_desc_sw128(base + (kk >> 2) * 2 * ATOM + (kk & 3) * 32, 16,
                         1024);
}

// Row r of a 128-row K-major swizzled half tile (128-byte rows): its eight
// 16-byte chunks from 32 packed words (the layout TMA writes with the 128-byte
// swizzle, which the MMA descriptors above read).
__device__ __forceinline__ void st_row(uint8_t* half_tile, int r,
                                       const uint32_t (&pk)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<uint4*>(half_tile + r * 128 + ((q ^ (r & 7)) << 4)) =
        make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}

// 16 TMEM lanes × 64 columns (eight 8-column units) into 32 registers: in
// unit u a thread holds lanes base + lane/4 (r[4u], r[4u+1]) and base + 8 +
// lane/4 (r[4u+2], r[4u+3]), columns 8u + 2·(lane % 4) and the next one.
__device__ __forceinline__ void tmem_ld16x256b_x8(uint32_t taddr,
                                                  uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Four 8×8 b16 matrices stored transposed: register j of a lane holds
// elements (lane/4, 2·(lane % 4)) and (lane/4, 2·(lane % 4) + 1) of matrix j;
// lane 8j + i gives the address of stored row i of matrix j, which receives
// column i (16 bytes).
__device__ __forceinline__ void stmatrix_x4_trans(const void* row, uint32_t a0,
                                                  uint32_t a1, uint32_t a2,
                                                  uint32_t a3) {
  asm volatile(
      "stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};"
      ::"r"(smem_u32(row)), "r"(a0), "r"(a1), "r"(a2), "r"(a3)
      : "memory");
}

__device__ __forceinline__ float max3f(float x, float y, float z) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(x), "f"(y), "f"(z));
  return r;
}

// 168 registers a thread: ten warps, three on some SM sub-partitions
// (16384 registers each)
__global__ void __maxnreg__(168)
    attn_fwd_tc_kernel(const __grid_constant__ FwdTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  uint64_t* q_full = bar + 0;
  uint64_t* kv_full = bar + 1;    // [NSLOT]
  uint64_t* kv_empty = bar + 4;   // [NSLOT]
  uint64_t* s_full = bar + 7;     // [NT] S_t written
  uint64_t* s_free = bar + 9;     // [NT] S_t copied to registers
  uint64_t* p_full = bar + 11;    // [NT] P_t written (and Oᵀ rescaled)
  uint64_t* pv_done = bar + 13;   // [NT] Oᵀ += Vᵀ·P_tᵀ done (P_t free)
  uint64_t* drain = bar + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* f_full = bar + 17;    // [NT] tile t's rescale flags written
  uint64_t* g_full = bar + 19;    // [NT] tile t's per-query factors written
  // [NT][2][4]: per tile and key-block parity, the last block at which a row
  // of warp quarter q took a new reference max (only ever increases, so it
  // needs no reset)
  volatile int* rescale_at = reinterpret_cast<volatile int*>(bar + 21);
  float* colf = reinterpret_cast<float*>(sm + OFF_COLF);   // [NT][BLK]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Tiles T = cta_tiles(a);
  const int nk = max(T.nkb[0], T.nkb[1]);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int t = 0; t < NT; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&s_free[t], 128);
      mbar_init(&p_full[t], 128);
      mbar_init(&pv_done[t], 1);
      mbar_init(&f_full[t], 128);
      mbar_init(&g_full[t], 128);
      for (int q = 0; q < 8; ++q) rescale_at[t * 8 + q] = 0;
    }
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
      // ------------------------------------------------------------- TMA --
      // The ring carries K_0, then K_{j+1} and V_j for each block j: a K
      // slot is released once both tiles' S MMAs have read it, a V slot once
      // the output product has.
      tma_prefetch_desc(&a.mq);
      tma_prefetch_desc(&a.mk);
      tma_prefetch_desc(&a.mv);
      const int ntiles = T.nkb[1] > 0 ? 2 : 1;
      mbar_arrive_expect_tx(q_full, ntiles * TILE);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t >= ntiles) continue;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          tma_load_3d(sm + OFF_Q + t * TILE + hh * ATOM, &a.mq, q_full,
                      T.head[t] * HD + hh * 64, T.q0[t], T.b);
      }
      uint32_t armed = 0, armed_par = 0;
      int e = 0;
      auto put = [&](const CUtensorMap* map, int jb) -> bool {
        const int st = e % NSLOT;
        const uint32_t ph = (e / NSLOT) & 1;
        if (!mbar_wait(&kv_empty[st], ph ^ 1, abort_flag, a.status, 11))
          return false;
        mbar_arrive_expect_tx(&kv_full[st], TILE);
        armed |= 1u << st;
        armed_par = (armed_par & ~(1u << st)) | (ph << st);
        for (int hh = 0; hh < 2; ++hh)
          tma_load_3d(sm + OFF_KV + st * TILE + hh * ATOM, map, &kv_full[st],
                      T.kvh * HD + hh * 64, jb * BLK, T.b);
        ++e;
        return true;
      };
      bool ok = put(&a.mk, 0);
      for (int jb = 0; ok && jb < nk; ++jb) {
        if (jb + 1 < nk) ok = put(&a.mk, jb + 1);
        if (ok) ok = put(&a.mv, jb);
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        mbar_wait(q_full, 0, &no_abort, nullptr, 0);
        for (int st = 0; st < NSLOT; ++st)
          if (armed & (1u << st))
            mbar_wait(&kv_full[st], (armed_par >> st) & 1u, &no_abort, nullptr,
                      0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------- MMA --
      constexpr uint32_t IDESC_S = idesc_f16_f32(128, 128, 0, 0);
      // Oᵀ += Vᵀ·Pᵀ: A = V read MN-major, B = P K-major; N = 256 covers
      // both tiles' queries in one instruction, N = 128 one tile
      constexpr uint32_t IDESC_O2 = idesc_f16_f32(128, 256, 1, 0);
      constexpr uint32_t IDESC_O1 = idesc_f16_f32(128, 128, 1, 0);
      bool ok = mbar_wait(q_full, 0, abort_flag, a.status, 12);
      int e = 0;
      uint32_t sKV = 0;
      auto take = [&]() -> bool {
        if (!mbar_wait(&kv_full[e % NSLOT], (e / NSLOT) & 1, abort_flag,
                       a.status, 13))
          return false;
        tc_fence_after();
        sKV = smem_u32(sm + OFF_KV + (e % NSLOT) * TILE);
        return true;
      };
      auto give = [&]() {
        tc_commit(&kv_empty[e % NSLOT]);
        ++e;
      };
      auto s_mma = [&](int t) {
        const uint32_t sQ = smem_u32(sm + OFF_Q + t * TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(tmem + t * 128, desc_kmajor(sQ, kk), desc_kmajor(sKV, kk),
                     IDESC_S, kk > 0 ? 1u : 0u);
        tc_commit(&s_full[t]);
      };
      if (ok && (ok = take())) {
#pragma unroll
        for (int t = 0; t < NT; ++t)
          if (T.nkb[t] > 0) s_mma(t);
        give();
      }
      for (int jb = 0; ok && jb < nk; ++jb) {
        if (jb + 1 < nk) {
          if (!(ok = take())) break;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (!ok || jb + 1 >= T.nkb[t]) continue;
            // S_t is free once tile t's softmax has copied block jb out
            if (!(ok = mbar_wait(&s_free[t], jb & 1, abort_flag, a.status, 14)))
              break;
            tc_fence_after();
            s_mma(t);
          }
          if (!ok) break;
          give();
        }
        if (!(ok = take())) break;
        // Oᵀ += Vᵀ_jb·Pᵀ over the tiles still reading keys at block jb; the
        // softmax rescaled Oᵀ (if needed) before signalling P_t
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (!ok || jb >= T.nkb[t]) continue;
          ok = mbar_wait(&p_full[t], jb & 1, abort_flag, a.status, 15);
        }
        if (!ok) break;
        tc_fence_after();
        {
          const bool both = jb < T.nkb[0] && jb < T.nkb[1];
          const int t0 = jb < T.nkb[0] ? 0 : 1;
          const uint32_t sP = smem_u32(sm + OFF_P + t0 * ATOM);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_f16(tmem + COL_O + t0 * 128, desc_mnmajor(sKV, kk),
                       desc_p(sP, kk), both ? IDESC_O2 : IDESC_O1,
                       (jb > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (jb < T.nkb[t]) tc_commit(&pv_done[t]);
        }
        give();
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        tc_commit(drain);
        mbar_wait(drain, 0, &no_abort, nullptr, 0);
      }
    }
  } else {
    // --------------------------------------------------------- softmax --
    // thread: query row r of tile t (TMEM lane r), all 128 key columns
    const int t = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int nkb = t ? T.nkb[1] : T.nkb[0];
    const int q0 = t ? T.q0[1] : T.q0[0];
    const int head = t ? T.head[1] : T.head[0];
    const int qi = q0 + r;
    const uint32_t lane_base =
        tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t s_col = lane_base + t * 128;
    const uint32_t o_col = lane_base + COL_O + t * 128;
    uint8_t* ptile = sm + OFF_P + t * ATOM;
    float* tcolf = colf + t * BLK;
    const float c = a.scale_log2;
    const float thr = RESCALE_LOG2 / c;   // the rescale threshold in raw units
    float m_ref = -INFINITY, l_run = 0.0f;
    int n_g = 0;   // completed phases of g_full[t]
    bool read_f = false;   // the last block's factors may still be read
    bool ok = true;
    for (int jb = 0; jb < nkb; ++jb) {
      if (!mbar_wait_warp(&s_full[t], jb & 1, abort_flag, a.status, 16)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t v[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(s_col + cc * 32, v[cc]);
      tmem_ld_wait(v[0]);
      reg_fence32(v[1]);
      reg_fence32(v[2]);
      reg_fence32(v[3]);
      tc_fence_before();
      mbar_arrive(&s_free[t]);   // S_t may take the next block's scores now
      if ((jb + 1) * BLK > a.s || (a.causal && (jb + 1) * BLK - 1 > q0)) {
        // diagonal or ragged block: invalid keys become −inf (branch-free)
        const int lim = (a.causal ? min(qi, a.s - 1) : a.s - 1) - jb * BLK;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            v[cc][i] = (cc * 32 + i <= lim) ? v[cc][i]
                                            : __float_as_uint(-INFINITY);
      }
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        mx8[i] = fmaxf(__uint_as_float(v[0][i]), __uint_as_float(v[0][i + 8]));
#pragma unroll
      for (int i = 16; i < 128; i += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mx8[k] = max3f(mx8[k], __uint_as_float(v[i >> 5][(i & 31) + k]),
                         __uint_as_float(v[i >> 5][(i & 31) + k + 8]));
      const float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]),
                             max3f(mx8[3], mx8[4], mx8[5]),
                             fmaxf(mx8[6], mx8[7]));
      // a new reference max when the block's max exceeds it by more than
      // the threshold; rows that keep theirs get the factor 1
      float alpha = 1.0f;
      bool new_ref = false;
      if (jb == 0) {
        m_ref = mx;
      } else if (mx > m_ref + thr) {
        alpha = ex2_approx((m_ref - mx) * c);
        m_ref = mx;
        new_ref = true;
      }
      // query r's factor scales column r of Oᵀ, which every warp of the tile
      // holds 32 feature lanes of; columns 32·q to 32·q + 31 are the rows of
      // warp quarter q, which flags them here (read after the exponentials)
      if (jb >= 1) {
        if (__any_sync(0xffffffffu, new_ref) && lane == 0)
          rescale_at[t * 8 + (jb & 1) * 4 + quarter] = jb;
        mbar_arrive(&f_full[t]);
      }
      // P = exp2(c·(s − m)) in fp16 pairs: keys 0–63 in pk[0], 64–127 in pk[1]
      const float neg = -m_ref * c;
      float sum8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) sum8[i] = 0.0f;
      uint32_t pk[2][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(v[cc][i]), c, neg));
          const float p1 =
              ex2_approx(fmaf(__uint_as_float(v[cc][i + 1]), c, neg));
          sum8[i & 7] += p0;
          sum8[(i + 1) & 7] += p1;
          pk[cc >> 1][(cc & 1) * 16 + (i >> 1)] = pack_f16x2(p0, p1);
        }
      }
      if (jb >= 1) {
        // the tile's flags of this block (complete by now: every warp set
        // them before its exponentials), read while Oᵀ += Vᵀ·Pᵀ of the
        // previous block may still run
        if (!mbar_wait_warp(&f_full[t], (jb - 1) & 1, abort_flag, a.status,
                            18)) {
          ok = false;
          break;
        }
        volatile int* flags = rescale_at + t * 8 + (jb & 1) * 4;
        const int f0 = flags[0], f1 = flags[1], f2 = flags[2], f3 = flags[3];
        const bool any = __any_sync(
            0xffffffffu, (f0 == jb) | (f1 == jb) | (f2 == jb) | (f3 == jb));
        // that product must have completed before Oᵀ is rescaled, the P
        // buffer overwritten or the factors rewritten (its start needed every
        // row of the tile past its reads of them)
        if (!mbar_wait_warp(&pv_done[t], (jb - 1) & 1, abort_flag, a.status,
                            17)) {
          ok = false;
          break;
        }
        read_f = any;
        if (any) {
          tcolf[r] = alpha;
          mbar_arrive(&g_full[t]);
          if (!mbar_wait_warp(&g_full[t], n_g & 1, abort_flag, a.status, 22)) {
            ok = false;
            break;
          }
          ++n_g;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            const int fc = cc == 0 ? f0 : cc == 1 ? f1 : cc == 2 ? f2 : f3;
            if (fc != jb) continue;
            uint32_t o[32];
            tmem_ld32(o_col + cc * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 f =
                  *reinterpret_cast<const float4*>(tcolf + cc * 32 + i);
              o[i] = __float_as_uint(__uint_as_float(o[i]) * f.x);
              o[i + 1] = __float_as_uint(__uint_as_float(o[i + 1]) * f.y);
              o[i + 2] = __float_as_uint(__uint_as_float(o[i + 2]) * f.z);
              o[i + 3] = __float_as_uint(__uint_as_float(o[i + 3]) * f.w);
            }
            tmem_st32(o_col + cc * 32, o);
          }
        }
      }
      st_row(ptile, r, pk[0]);
      st_row(ptile + 2 * ATOM, r, pk[1]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[t]);
      l_run = l_run * alpha +
              (((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) +
               ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7])));
    }
    // epilogue: wait for the last Oᵀ += Vᵀ·Pᵀ, then O / l and the LSE.  The
    // queries' 1 / l pass through shared memory (unless the last block
    // rescaled, nothing reads the factors any more and this exchange runs
    // while the last product completes); the scaled bf16 output goes,
    // transposed by stmatrix, into the tile's P rows (free now) as two
    // 64-feature halves of 128-byte rows in the 128-byte swizzle (conflict-
    // free), and each warp then stores 32 whole rows of 256 bytes.
    const int last = nkb - 1;
    if (nkb > 0 && __all_sync(0xffffffffu, ok)) {
      bool fine = true;
      if (read_f)
        fine = mbar_wait_warp(&pv_done[t], last & 1, abort_flag, a.status, 19);
      if (fine) {
        tcolf[r] = 1.0f / l_run;
        mbar_arrive(&f_full[t]);
        if (!read_f)
          fine = mbar_wait_warp(&pv_done[t], last & 1, abort_flag, a.status,
                                19);
      }
      fine = fine &&
             mbar_wait_warp(&f_full[t], last & 1, abort_flag, a.status, 20);
      if (fine) {
        // Oᵀ read in 8×8 blocks of (feature, query), scaled by the queries'
        // 1 / l and stored transposed: 8 query rows of 8 features each.
        // This lane addresses stored row i of matrix j: features f0 to f0 + 7
        // of query 8·(u + j/2) + i.
        tc_fence_after();
        const int j = lane >> 3, i = lane & 7;
        const int qp = 2 * (lane & 3);
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t x[2][32];
          const uint32_t ta = o_col + (static_cast<uint32_t>(hh * 16) << 16);
          tmem_ld16x256b_x8(ta, x[0]);
          tmem_ld16x256b_x8(ta + 64, x[1]);
          tmem_ld_wait(x[0]);
          reg_fence32(x[1]);
          const int f0 = quarter * 32 + hh * 16 + 8 * (j & 1);
          uint8_t* row = ptile + (f0 >> 6) * 2 * ATOM + (j >> 1) * 1024 +
                         i * 128 + ((((f0 & 63) >> 3) ^ i) << 4);
#pragma unroll
          for (int u = 0; u < 16; u += 2) {
            const uint32_t* xa = &x[u >> 3][(u & 7) * 4];
            const float2 c0 =
                *reinterpret_cast<const float2*>(tcolf + 8 * u + qp);
            const float2 c1 =
                *reinterpret_cast<const float2*>(tcolf + 8 * u + 8 + qp);
            stmatrix_x4_trans(
                row + u * 1024,
                pack_bf16x2(__uint_as_float(xa[0]) * c0.x,
                            __uint_as_float(xa[1]) * c0.y),
                pack_bf16x2(__uint_as_float(xa[2]) * c0.x,
                            __uint_as_float(xa[3]) * c0.y),
                pack_bf16x2(__uint_as_float(xa[4]) * c1.x,
                            __uint_as_float(xa[5]) * c1.y),
                pack_bf16x2(__uint_as_float(xa[6]) * c1.x,
                            __uint_as_float(xa[7]) * c1.y));
          }
        }
        mbar_arrive(&f_full[t]);
        fine = mbar_wait_warp(&f_full[t], (last + 1) & 1, abort_flag, a.status,
                              21);
      }
      if (fine) {
        // lanes 0–15 one row, 16–31 the next: 16 chunks of 16 bytes each
        const int ld = a.nq * HD;
        const int chunk = lane & 15;
        const uint8_t* src = ptile + (chunk >> 3) * 2 * ATOM;
#pragma unroll 4
        for (int k = 0; k < 16; ++k) {
          const int q = quarter * 32 + 2 * k + (lane >> 4);
          const uint4 u = *reinterpret_cast<const uint4*>(
              src + q * 128 + (((chunk & 7) ^ (q & 7)) << 4));
          if (q0 + q < a.s)
            reinterpret_cast<uint4*>(a.O + ((int64_t)T.b * a.s + q0 + q) * ld +
                                     head * HD)[chunk] = u;
        }
        if (qi < a.s)
          a.LSE[((int64_t)T.b * a.nq + head) * a.s + qi] =
              (m_ref * c + log2f(l_run)) * 0.69314718055994531f;
      }
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
  a.nb = (int)sh.b;
  a.nq = sh.nq;
  a.nkv = sh.nkv;
  a.causal = sh.causal;
  // two heads of a GQA group share a CTA when the group size is even
  a.pair_heads = (sh.nq / sh.nkv) % 2 == 0;
  a.scale_log2 = sh.scale * 1.4426950408889634f;
  a.status = status;
  const int64_t nblk = (sh.s + BLK - 1) / BLK;
  const unsigned grid =
      (unsigned)(a.pair_heads ? nblk * (sh.nq / 2) * sh.b
                              : (nblk + 1) / 2 * sh.nq * sh.b);
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
