// gemm_tc.cu — tcgen05 (5th-generation tensor core) GEMM of the TP block.
//
// One persistent kernel per GEMM launch over clusters of two CTAs (one CTA
// per SM): the pair computes a 256×256 output tile with tcgen05.mma of
// M=256 (cta_group::2), each CTA holding its 128 rows of A and half of the
// B tile, so every SM streams 32 KB per 64-deep K block instead of 48 KB
// and six stages fit in shared memory.  192 threads per CTA:
//   warp 0   TMA producer: one thread streams this CTA's A rows and B half
//            into a 6-stage ring (128-byte swizzle); the bytes of both CTAs
//            are counted on the leader's (rank 0) barrier.
//   warp 1   allocates 512 TMEM columns in both SMs (two 128×256 fp32
//            accumulators per SM); one thread of the leader issues the MMAs
//            and multicasts their completion to both CTAs.
//   warps 2–5 epilogue (both CTAs): tcgen05.ld of the finished accumulator
//            (one TMEM lane = one output row per thread), the fused
//            elementwise work of the launch, 16-byte stores.  Double-
//            buffered accumulators let the epilogue of tile i overlap the
//            main loop of tile i+1.
// The segment / part structure of the K loop is described in gemm.h; it is
// how the shard sum of a row-parallel projection (g) or of an input gradient
// (f) is taken in the accumulator ([Grasp-TP] §2–§3, [adu-TP] 算子 f 和 g).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "gemm.h"
#include "profile.h"

namespace tp {
namespace {

constexpr int BM = 128;                        // rows per CTA (256 per pair)
constexpr int BN = 256;                        // columns per tile
constexpr int BNH = BN / 2;                    // B rows held by each CTA
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;           // 16 KB
constexpr int B_BYTES = BNH * BK * 2;          // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int THREADS = 192;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;

struct TcPart {
  int kblocks;
  int nsub;
  int seg_z_stride;
  int seg_sub_stride;
};

struct TcParams {
  CUtensorMap ma[3];
  CUtensorMap mb[3];
  CUtensorMap mb2;
  TcPart part[3];
  int nparts;
  int M, N;            // N is the logical output width
  int m_tiles, n_tiles, nz, total_tiles, group_m;
  int f16;             // fp16 A and B (kind::f16 with the F16 formats)
  GemmEpilogue epi;
  unsigned* status;
};

__device__ __forceinline__ void decode_tile(const TcParams& p, int t, int& z,
                                            int& mt, int& nt) {
  const int per_z = p.m_tiles * p.n_tiles;
  z = t / per_z;
  const int r = t - z * per_z;
  const int gsz = p.group_m * p.n_tiles;
  const int g = r / gsz;
  const int first_m = g * p.group_m;
  const int gm = min(p.group_m, p.m_tiles - first_m);
  const int rr = r - g * gsz;
  mt = first_m + rr % gm;
  nt = rr / gm;
}

// ---------------------------------------------------------------- epilogue --
__device__ __forceinline__ void load32_bf16(const __nv_bfloat16* src,
                                            float* v, int valid) {
  if (valid >= 32) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = __ldg(s + q);
      float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y),
             c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
      v[8 * q + 0] = a.x; v[8 * q + 1] = a.y; v[8 * q + 2] = b.x;
      v[8 * q + 3] = b.y; v[8 * q + 4] = c.x; v[8 * q + 5] = c.y;
      v[8 * q + 6] = d.x; v[8 * q + 7] = d.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      v[i] = (i < valid) ? __bfloat162float(src[i]) : 0.0f;
  }
}

__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst,
                                             const float* v, int valid) {
  if (valid >= 32) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 u;
      u.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
      u.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
      u.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
      u.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
      d[q] = u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < valid) dst[i] = __float2bfloat16_rn(v[i]);
  }
}

__device__ __forceinline__ void store32_f16(__half* dst, const float* v,
                                            int valid, unsigned* status) {
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 32; ++i) bad |= (i < valid) && !(fabsf(v[i]) <= kF16Max);
  if (bad) record_error(status, kDevRange, 5);
  if (valid >= 32) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 u;
      u.x = pack_f16x2(v[8 * q + 0], v[8 * q + 1]);
      u.y = pack_f16x2(v[8 * q + 2], v[8 * q + 3]);
      u.z = pack_f16x2(v[8 * q + 4], v[8 * q + 5]);
      u.w = pack_f16x2(v[8 * q + 6], v[8 * q + 7]);
      d[q] = u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < valid) dst[i] = __float2half_rn(v[i]);
  }
}

template <int EPI>
__device__ __forceinline__ void epilogue_tile(const TcParams& p,
                                              uint32_t taddr, int z, int m,
                                              int n0, float dq) {
  const GemmEpilogue& e = p.epi;
  const bool row_ok = m < p.M;
  if constexpr (EPI == EPI_SWIGLU) {
    // accumulator columns [0,128): gate, [128,256): up, same hidden units
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t rg[32], ru[32];
      tmem_ld32(taddr + c * 32, rg);
      tmem_ld_wait(rg);
      tmem_ld32(taddr + 128 + c * 32, ru);
      tmem_ld_wait(ru);
      const int n = n0 + c * 32;
      if (row_ok && n < p.N) {
        const int valid = min(32, p.N - n);
        float g[32], u[32], a[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          g[i] = __uint_as_float(rg[i]) * dq;
          u[i] = __uint_as_float(ru[i]) * dq;
          a[i] = g[i] * sigmoid_f(g[i]) * u[i];
        }
        const int64_t off = (int64_t)m * e.ldo + n;
        store32_bf16(static_cast<__nv_bfloat16*>(e.out) + off, g, valid);
        store32_bf16(static_cast<__nv_bfloat16*>(e.out2) + off, u, valid);
        store32_bf16(static_cast<__nv_bfloat16*>(e.out3) +
                         (int64_t)m * e.ldo2 + n,
                     a, valid);
      }
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(taddr + c * 32, r);
      tmem_ld_wait(r);
      const int n = n0 + c * 32;
      if (!row_ok || n >= p.N) continue;
      const int valid = min(32, p.N - n);
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * dq;
      if constexpr (EPI == EPI_STORE) {
        if (e.bias != nullptr) {
          float b[32];
          load32_bf16(static_cast<const __nv_bfloat16*>(e.bias) + n, b, valid);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] += b[i];
        }
        if (e.dropout) {
          const uint64_t base = (uint64_t)m * (uint64_t)p.N + (uint64_t)n;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            v[i] = dropout_keep(e.seed, base + i, e.drop_thr)
                       ? v[i] * e.drop_scale
                       : 0.0f;
        }
        if (e.resid != nullptr) {
          float rr[32];
          load32_bf16(static_cast<const __nv_bfloat16*>(e.resid) +
                          (int64_t)m * e.ldr + n,
                      rr, valid);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] += rr[i];
        }
        void* dst = e.out;
        int64_t ld = e.ldo, col = n;
        if (e.split1 != 0 && n >= e.split1) {
          if (e.split2 != 0 && n >= e.split2) {
            dst = e.out3;
            ld = e.ldo3;
            col = n - e.split2;
          } else {
            dst = e.out2;
            ld = e.ldo2;
            col = n - e.split1;
          }
        }
        const int64_t off = (int64_t)z * e.out_z_stride + (int64_t)m * ld + col;
        if (e.out_f16)
          store32_f16(static_cast<__half*>(dst) + off, v, valid, p.status);
        else
          store32_bf16(static_cast<__nv_bfloat16*>(dst) + off, v, valid);
      } else if constexpr (EPI == EPI_GELU) {
        if (e.bias != nullptr) {
          float b[32];
          load32_bf16(static_cast<const __nv_bfloat16*>(e.bias) + n, b, valid);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] += b[i];
        }
        const int64_t off = (int64_t)m * e.ldo + n;
        store32_bf16(static_cast<__nv_bfloat16*>(e.out) + off, v, valid);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = gelu_f(v[i]);
        store32_bf16(static_cast<__nv_bfloat16*>(e.out2) +
                         (int64_t)m * e.ldo2 + n,
                     v, valid);
      } else if constexpr (EPI == EPI_DGELU) {
        float hv[32];
        load32_bf16(static_cast<const __nv_bfloat16*>(e.aux1) +
                        (int64_t)m * e.ld_aux + n,
                    hv, valid);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= gelu_grad_f(hv[i]);
        store32_bf16(static_cast<__nv_bfloat16*>(e.out) + (int64_t)m * e.ldo + n,
                     v, valid);
      } else if constexpr (EPI == EPI_DSWIGLU) {
        float g[32], u[32], dg[32];
        const int64_t aoff = (int64_t)m * e.ld_aux + n;
        load32_bf16(static_cast<const __nv_bfloat16*>(e.aux1) + aoff, g, valid);
        load32_bf16(static_cast<const __nv_bfloat16*>(e.aux2) + aoff, u, valid);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float s = sigmoid_f(g[i]);
          dg[i] = v[i] * u[i] * s * (1.0f + g[i] * (1.0f - s));
          v[i] = v[i] * g[i] * s;   // dU = dA · SiLU(G)
        }
        const int64_t off = (int64_t)m * e.ldo + n;
        store32_bf16(static_cast<__nv_bfloat16*>(e.out) + off, dg, valid);
        store32_bf16(static_cast<__nv_bfloat16*>(e.out2) + off, v, valid);
      }
    }
  }
}

// ------------------------------------------------------------------ kernel --
// F8 = 1: E4M3 operands; a K block is 128 elements (the same 128 bytes per
// row as 64 bf16 elements), one kind::f8f6f4 instruction per 32 of them.
template <int A_MN, int B_MN, int EPI, int F8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ TcParams p) {
  constexpr int BKE = F8 ? 2 * BK : BK;   // K elements per stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smB + STAGES * B_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank() & 1u;
  const bool leader = rank == 0;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  constexpr int BN_LOG = (EPI == EPI_SWIGLU) ? BN / 2 : BN;

  if (threadIdx.x == 0) {
    // full: the leader's counts both CTAs' bytes; empty, tfull: one arrival
    // from the leader's commits; tempty (leader's): both epilogues
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.nparts; ++i) {
      tma_prefetch_desc(&p.ma[i]);
      tma_prefetch_desc(&p.mb[i]);
    }
    if (EPI == EPI_SWIGLU) tma_prefetch_desc(&p.mb2);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // barriers of both CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------- TMA producer --
      const uint32_t full0 = cluster_addr(full, 0);   // the leader's full[0]
      uint32_t stage = 0, phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int t = cid; ok && t < p.total_tiles; t += ncl) {
        int z, mt, nt;
        decode_tile(p, t, z, mt, nt);
        const int m0 = mt * 2 * BM + (int)rank * BM, n0 = nt * BN_LOG;
        for (int pi = 0; ok && pi < p.nparts; ++pi) {
          const TcPart& pt = p.part[pi];
          for (int j = 0; ok && j < pt.nsub; ++j) {
            const int seg = z * pt.seg_z_stride + j * pt.seg_sub_stride;
            for (int kb = 0; kb < pt.kblocks; ++kb) {
              if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status,
                             1)) {
                ok = false;
                break;
              }
              if (leader) {
                mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
                armed |= 1u << stage;
                armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
              }
              const uint32_t fb = full0 + stage * 8;
              uint8_t* sa = smA + stage * A_BYTES;
              uint8_t* sb = smB + stage * B_BYTES;
              const int k0 = kb * BKE;
              if (A_MN) {
                tma_load_3d_pair(sa, &p.ma[pi], fb, m0, k0, seg);
                tma_load_3d_pair(sa + 8192, &p.ma[pi], fb, m0 + 64, k0, seg);
              } else {
                tma_load_3d_pair(sa, &p.ma[pi], fb, k0, seg, m0);
              }
              if (EPI == EPI_SWIGLU) {
                // rank 0: the gate rows, rank 1: the up rows of the same units
                tma_load_3d_pair(sb, leader ? &p.mb[pi] : &p.mb2, fb, k0, seg,
                                 n0);
              } else if (B_MN) {
                tma_load_3d_pair(sb, &p.mb[pi], fb, n0 + (int)rank * BNH, k0,
                                 seg);
                tma_load_3d_pair(sb + 8192, &p.mb[pi], fb,
                                 n0 + (int)rank * BNH + 64, k0, seg);
              } else {
                tma_load_3d_pair(sb, &p.mb[pi], fb, k0, seg,
                                 n0 + (int)rank * BNH);
              }
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
              }
            }
          }
        }
      }
      if (ok) {
        // the leader's last commits land on this CTA's empty barriers before
        // the CTA may exit
        for (int i = 0; i < STAGES; ++i) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status, 6))
            break;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (*abort_flag && leader) {
        // let every copy counted on this CTA's barriers land
        volatile int no_abort = 0;
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s))
            mbar_wait(&full[s], (armed_par >> s) & 1u, &no_abort, nullptr, 0);
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // -------------------------------------------------------- MMA issue --
      const uint32_t IDESC =
          F8 ? idesc_e4m3_f32(2 * BM, BN)
             : (p.f16 ? idesc_f16_f32(2 * BM, BN, A_MN, B_MN)
                      : idesc_bf16_f32(2 * BM, BN, A_MN, B_MN));
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = cid; ok && t < p.total_tiles; t += ncl, ++it) {
        const int buf = it & 1;
        const uint32_t aphase = (it >> 1) & 1;
        if (!mbar_wait(&tempty[buf], aphase ^ 1, abort_flag, p.status, 2)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        uint32_t acc = 0;
        for (int pi = 0; ok && pi < p.nparts; ++pi) {
          const TcPart& pt = p.part[pi];
          for (int j = 0; ok && j < pt.nsub; ++j) {
            for (int kb = 0; kb < pt.kblocks; ++kb) {
              if (!mbar_wait(&full[stage], phase, abort_flag, p.status, 3)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a0 = smem_u32(smA + stage * A_BYTES);
              const uint32_t b0 = smem_u32(smB + stage * B_BYTES);
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t ad =
                    A_MN ? smem_desc_sw128(a0 + kk * 2048, 8192, 1024)
                         : smem_desc_sw128(a0 + kk * 32, 16, 1024);
                const uint64_t bd =
                    B_MN ? smem_desc_sw128(b0 + kk * 2048, 8192, 1024)
                         : smem_desc_sw128(b0 + kk * 32, 16, 1024);
                if (F8)
                  tc_mma_f8_pair(d_tmem, ad, bd, IDESC, acc);
                else
                  tc_mma_f16_pair(d_tmem, ad, bd, IDESC, acc);
                acc = 1;
              }
              tc_commit_pair(&empty[stage], 3);
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1;
              }
            }
          }
        }
        if (ok) tc_commit_pair(&tfull[buf], 3);
      }
      if (*abort_flag) {
        volatile int no_abort = 0;
        tc_commit_pair(drain, 1);
        mbar_wait(drain, 0, &no_abort, nullptr, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int quarter = warp & 3;   // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;
    const uint32_t tempty0 = cluster_addr(tempty, 0);   // the leader's
    const float dq = (F8 && p.epi.scale_a != nullptr)
                         ? 1.0f / (*p.epi.scale_a * *p.epi.scale_b)
                         : 1.0f;
    int it = 0;
    for (int t = cid; t < p.total_tiles; t += ncl, ++it) {
      int z, mt, nt;
      decode_tile(p, t, z, mt, nt);
      const int buf = it & 1;
      const uint32_t aphase = (it >> 1) & 1;
      if (!mbar_wait_warp(&tfull[buf], aphase, abort_flag, p.status, 4)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * BN;
      epilogue_tile<EPI>(p, taddr, z, mt * 2 * BM + (int)rank * BM + row,
                         nt * BN_LOG, dq);
      tc_fence_before();
      mbar_arrive_cluster(tempty0 + buf * 8);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // neither CTA leaves while the pair still uses it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// ------------------------------------------------------------------- host --
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

bool encode_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1,
               uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0,
               uint32_t b1, uint32_t b2,
               CUtensorMapDataType ty = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, ty, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K-major operand (rows × K, row stride ld): dims {kseg, nseg, rows}.
// MN-major operand (K × rows, row stride ld): dims {rows, kseg, nseg}.
bool encode_operand(CUtensorMap* m, const GemmOperand& o, int64_t kseg,
                    int nseg, uint32_t box_rows, bool f8 = false,
                    bool f16 = false) {
  if (f8)   // E4M3, K-major: 128-element (128-byte) K boxes
    return !o.mn_major &&
           encode_3d(m, o.ptr, kseg, nseg, o.rows, kseg, o.ld, 2 * BK, 1,
                     box_rows, CU_TENSOR_MAP_DATA_TYPE_UINT8);
  const CUtensorMapDataType ty = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (o.mn_major)
    return encode_3d(m, o.ptr, o.rows, kseg, nseg, o.ld * 2,
                     (uint64_t)kseg * o.ld * 2, 64, BK, 1, ty);
  return encode_3d(m, o.ptr, kseg, nseg, o.rows, kseg * 2, o.ld * 2, BK, 1,
                   box_rows, ty);
}

// One CTA pair per two SMs: the grid is as many pairs as can be resident
// at once (clusters need both CTAs on SMs of one GPC), capped by the tiles.
template <int A_MN, int B_MN, int EPI, int F8 = 0>
int launch_inst(const TcParams& prm, cudaStream_t s, double flops,
                double bytes) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int clusters = 0;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_tc_kernel<A_MN, B_MN, EPI, F8>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    SMEM_BYTES);
    if (attr_err != cudaSuccess) return;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)(device_sm_count() & ~1));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    attr_err = cudaOccupancyMaxActiveClusters(
        &clusters, gemm_tc_kernel<A_MN, B_MN, EPI, F8>, &cfg);
    if (attr_err == cudaSuccess && clusters < 1) attr_err = cudaErrorInvalidConfiguration;
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int grid = 2 * std::min(prm.total_tiles, clusters);
  {
    ProfScope ps(s, F8 ? KF_GEMM_TC_FP8 : KF_GEMM_TC, flops, bytes);
    gemm_tc_kernel<A_MN, B_MN, EPI, F8><<<grid, THREADS, SMEM_BYTES, s>>>(prm);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace

bool encode_tmap_3d_f16(CUtensorMap* m, const void* base, uint64_t d0,
                        uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
                        uint32_t b0, uint32_t b1, uint32_t b2) {
  if (!get_encode()) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_gemm_tc(const GemmProblem& pr, void* stream, unsigned* status) {
  if (!get_encode()) return cudaErrorNotSupported;
  const GemmEpilogue& e = pr.epi;
  const int a_mn = pr.parts[0].a.mn_major, b_mn = pr.parts[0].b.mn_major;
  for (int i = 1; i < pr.nparts; ++i)
    if (pr.parts[i].a.mn_major != a_mn || pr.parts[i].b.mn_major != b_mn)
      return cudaErrorInvalidValue;
  if (e.kind == EPI_SWIGLU && (b_mn || a_mn || pr.nparts != 1))
    return cudaErrorInvalidValue;
  if ((e.split1 || e.split2) &&
      (e.kind != EPI_STORE || e.split1 % 32 || e.split2 % 32 ||
       (e.split2 && e.split2 < e.split1) || pr.nz != 1))
    return cudaErrorInvalidValue;
  const bool f8 = pr.dtype == 2;
  const bool f16 = !f8 && pr.f16 != 0;
  if (f8 && (a_mn || b_mn ||
             (e.kind != EPI_STORE && e.kind != EPI_GELU &&
              e.kind != EPI_SWIGLU)))
    return cudaErrorInvalidValue;
  const int bke = f8 ? 2 * BK : BK;   // K elements per stage

  TcParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.nparts = pr.nparts;
  for (int i = 0; i < pr.nparts; ++i) {
    const GemmPart& pt = pr.parts[i];
    if (!encode_operand(&prm.ma[i], pt.a, pt.kseg, pt.nseg, BM, f8, f16))
      return cudaErrorInvalidValue;
    const uint32_t brows = BNH;   // each CTA of the pair loads half of B
    if (!encode_operand(&prm.mb[i], pt.b, pt.kseg, pt.nseg, brows, f8, f16))
      return cudaErrorInvalidValue;
    if (e.kind == EPI_SWIGLU &&
        !encode_operand(&prm.mb2, pt.b2, pt.kseg, pt.nseg, brows, f8, f16))
      return cudaErrorInvalidValue;
    prm.part[i].kblocks = (int)((pt.kseg + bke - 1) / bke);
    prm.part[i].nsub = pt.nsub;
    prm.part[i].seg_z_stride = pt.seg_z_stride;
    prm.part[i].seg_sub_stride = pt.seg_sub_stride;
  }
  const int bn_log = (e.kind == EPI_SWIGLU) ? BN / 2 : BN;
  prm.M = (int)pr.M;
  prm.N = (int)pr.N;
  prm.m_tiles = (int)((pr.M + 2 * BM - 1) / (2 * BM));   // CTA-pair tiles
  prm.n_tiles = (int)((pr.N + bn_log - 1) / bn_log);
  prm.nz = pr.nz;
  prm.total_tiles = prm.m_tiles * prm.n_tiles * pr.nz;
  prm.group_m = 8;
  prm.f16 = f16 ? 1 : 0;
  prm.epi = e;
  prm.status = status;
  if (prm.total_tiles == 0) return cudaSuccess;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // algorithmic work of the launch: 2·M·N·K per batch, both B halves for
  // SwiGLU; bytes = operands read once + outputs written once
  double ktile = 0.0;
  for (int i = 0; i < pr.nparts; ++i)
    ktile += (double)pr.parts[i].kseg * pr.parts[i].nsub;
  const double ntot = (double)pr.N * (e.kind == EPI_SWIGLU ? 2.0 : 1.0);
  const double flops = 2.0 * (double)pr.M * ntot * ktile * pr.nz;
  const int outs = e.kind == EPI_SWIGLU ? 3
                   : (e.kind == EPI_GELU || e.kind == EPI_DSWIGLU) ? 2 : 1;
  const double bytes = (f8 ? 1.0 : 2.0) * ((double)pr.M + ntot) * ktile * pr.nz +
                       2.0 * (double)pr.M * pr.N * pr.nz * outs;

  if (f8) {
    switch (e.kind) {
      case EPI_STORE: return launch_inst<0, 0, EPI_STORE, 1>(prm, s, flops, bytes);
      case EPI_GELU: return launch_inst<0, 0, EPI_GELU, 1>(prm, s, flops, bytes);
      case EPI_SWIGLU: return launch_inst<0, 0, EPI_SWIGLU, 1>(prm, s, flops, bytes);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (e.kind) {
    case EPI_STORE:
      if (!a_mn && !b_mn) return launch_inst<0, 0, EPI_STORE>(prm, s, flops, bytes);
      if (!a_mn && b_mn) return launch_inst<0, 1, EPI_STORE>(prm, s, flops, bytes);
      if (a_mn && b_mn) return launch_inst<1, 1, EPI_STORE>(prm, s, flops, bytes);
      return launch_inst<1, 0, EPI_STORE>(prm, s, flops, bytes);
    case EPI_GELU:
      if (a_mn || b_mn) return cudaErrorInvalidValue;
      return launch_inst<0, 0, EPI_GELU>(prm, s, flops, bytes);
    case EPI_SWIGLU:
      return launch_inst<0, 0, EPI_SWIGLU>(prm, s, flops, bytes);
    case EPI_DGELU:
      if (a_mn || !b_mn) return cudaErrorInvalidValue;
      return launch_inst<0, 1, EPI_DGELU>(prm, s, flops, bytes);
    case EPI_DSWIGLU:
      if (a_mn || !b_mn) return cudaErrorInvalidValue;
      return launch_inst<0, 1, EPI_DSWIGLU>(prm, s, flops, bytes);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tp
