// gemm_simt.cu — fp32 GEMM on CUDA cores for the fp32 workloads.
//
// The same problem description as the tensor-core path (parts, shard
// segments, batches, fused epilogues; see gemm.h) evaluated with fp32 FMAs:
// the fp32 workloads need ~1e-4 relative accuracy, which tf32 tensor-core
// inputs (10-bit mantissa) cannot give.  64×64 output tile per 256-thread
// block, 4×4 outputs per thread, K staged through shared memory 16 at a time.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "gemm.h"
#include "profile.h"

namespace tp {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

struct SimtPart {
  const float* a;
  const float* b;
  const float* b2;
  int64_t lda, ldb;
  int a_mn, b_mn;
  int64_t kseg;
  int nsub, seg_z_stride, seg_sub_stride;
};

struct SimtParams {
  SimtPart part[3];
  int nparts;
  int64_t M, N;
  GemmEpilogue epi;
};

template <bool DUAL>
__device__ __forceinline__ void load_tile(float (*S)[TM + 1], const float* P,
                                          int64_t ld, int mn, int64_t r0,
                                          int64_t rows, int64_t kbase,
                                          int64_t k0, int64_t kseg) {
  for (int idx = threadIdx.x; idx < TM * TK; idx += blockDim.x) {
    int r, kk;
    if (mn) {
      r = idx % TM;
      kk = idx / TM;
    } else {
      r = idx / TK;
      kk = idx % TK;
    }
    const int64_t row = r0 + r, k = k0 + kk;
    float v = 0.0f;
    if (row < rows && k < kseg) {
      const int64_t kg = kbase + k;
      v = mn ? P[kg * ld + row] : P[row * ld + kg];
    }
    S[kk][r] = v;
  }
}

template <int EPI>
__global__ void __launch_bounds__(256)
    gemm_simt_kernel(const __grid_constant__ SimtParams p) {
  constexpr bool DUAL = (EPI == EPI_SWIGLU);
  __shared__ float As[TK][TM + 1];
  __shared__ float Bs[TK][TN + 1];
  __shared__ float B2s[DUAL ? TK : 1][TN + 1];
  const int z = blockIdx.z;
  const int64_t m0 = (int64_t)blockIdx.y * TM, n0 = (int64_t)blockIdx.x * TN;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {}, acc2[4][4] = {};
  for (int pi = 0; pi < p.nparts; ++pi) {
    const SimtPart& pt = p.part[pi];
    for (int j = 0; j < pt.nsub; ++j) {
      const int seg = z * pt.seg_z_stride + j * pt.seg_sub_stride;
      const int64_t kbase = (int64_t)seg * pt.kseg;
      for (int64_t k0 = 0; k0 < pt.kseg; k0 += TK) {
        load_tile<DUAL>(As, pt.a, pt.lda, pt.a_mn, m0, p.M, kbase, k0, pt.kseg);
        load_tile<DUAL>(Bs, pt.b, pt.ldb, pt.b_mn, n0, p.N, kbase, k0, pt.kseg);
        if (DUAL)
          load_tile<DUAL>(B2s, pt.b2, pt.ldb, pt.b_mn, n0, p.N, kbase, k0,
                          pt.kseg);
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < TK; ++kk) {
          float a[4], b[4], b2[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            b[jj] = Bs[kk][tx + 16 * jj];
            if (DUAL) b2[jj] = B2s[kk][tx + 16 * jj];
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              acc[i][jj] = fmaf(a[i], b[jj], acc[i][jj]);
              if (DUAL) acc2[i][jj] = fmaf(a[i], b2[jj], acc2[i][jj]);
            }
        }
        __syncthreads();
      }
    }
  }
  const GemmEpilogue& e = p.epi;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t m = m0 + ty + 16 * i;
    if (m >= p.M) continue;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int64_t n = n0 + tx + 16 * jj;
      if (n >= p.N) continue;
      float v = acc[i][jj];
      if constexpr (EPI == EPI_STORE) {
        if (e.bias) v += static_cast<const float*>(e.bias)[n];
        if (e.dropout)
          v = dropout_keep(e.seed, (uint64_t)m * p.N + n, e.drop_thr)
                  ? v * e.drop_scale
                  : 0.0f;
        if (e.resid) v += static_cast<const float*>(e.resid)[m * e.ldr + n];
        static_cast<float*>(e.out)[z * e.out_z_stride + m * e.ldo + n] = v;
      } else if constexpr (EPI == EPI_GELU) {
        if (e.bias) v += static_cast<const float*>(e.bias)[n];
        static_cast<float*>(e.out)[m * e.ldo + n] = v;
        static_cast<float*>(e.out2)[m * e.ldo2 + n] = gelu_f(v);
      } else if constexpr (EPI == EPI_SWIGLU) {
        const float g = v, u = acc2[i][jj];
        static_cast<float*>(e.out)[m * e.ldo + n] = g;
        static_cast<float*>(e.out2)[m * e.ldo + n] = u;
        static_cast<float*>(e.out3)[m * e.ldo2 + n] = g * sigmoid_f(g) * u;
      } else if constexpr (EPI == EPI_DGELU) {
        const float hv = static_cast<const float*>(e.aux1)[m * e.ld_aux + n];
        static_cast<float*>(e.out)[m * e.ldo + n] = v * gelu_grad_f(hv);
      } else if constexpr (EPI == EPI_DSWIGLU) {
        const float g = static_cast<const float*>(e.aux1)[m * e.ld_aux + n];
        const float u = static_cast<const float*>(e.aux2)[m * e.ld_aux + n];
        const float s = sigmoid_f(g);
        static_cast<float*>(e.out)[m * e.ldo + n] =
            v * u * s * (1.0f + g * (1.0f - s));
        static_cast<float*>(e.out2)[m * e.ldo + n] = v * g * s;
      }
    }
  }
}

}  // namespace

int launch_gemm_simt(const GemmProblem& pr, void* stream) {
  SimtParams p;
  memset(&p, 0, sizeof(p));
  p.nparts = pr.nparts;
  for (int i = 0; i < pr.nparts; ++i) {
    const GemmPart& s = pr.parts[i];
    SimtPart& d = p.part[i];
    d.a = static_cast<const float*>(s.a.ptr);
    d.b = static_cast<const float*>(s.b.ptr);
    d.b2 = static_cast<const float*>(s.b2.ptr);
    d.lda = s.a.ld;
    d.ldb = s.b.ld;
    d.a_mn = s.a.mn_major;
    d.b_mn = s.b.mn_major;
    d.kseg = s.kseg;
    d.nsub = s.nsub;
    d.seg_z_stride = s.seg_z_stride;
    d.seg_sub_stride = s.seg_sub_stride;
  }
  p.M = pr.M;
  p.N = pr.N;
  p.epi = pr.epi;
  dim3 grid((unsigned)((pr.N + TN - 1) / TN), (unsigned)((pr.M + TM - 1) / TM),
            (unsigned)pr.nz);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  double ktile = 0.0;
  for (int i = 0; i < pr.nparts; ++i)
    ktile += (double)pr.parts[i].kseg * pr.parts[i].nsub;
  const double ntot = (double)pr.N * (pr.epi.kind == EPI_SWIGLU ? 2.0 : 1.0);
  ProfScope ps(s, KF_GEMM_SIMT, 2.0 * (double)pr.M * ntot * ktile * pr.nz,
               4.0 * (((double)pr.M + ntot) * ktile + (double)pr.M * pr.N) *
                   pr.nz);
  switch (pr.epi.kind) {
    case EPI_STORE: gemm_simt_kernel<EPI_STORE><<<grid, 256, 0, s>>>(p); break;
    case EPI_GELU: gemm_simt_kernel<EPI_GELU><<<grid, 256, 0, s>>>(p); break;
    case EPI_SWIGLU: gemm_simt_kernel<EPI_SWIGLU><<<grid, 256, 0, s>>>(p); break;
    case EPI_DGELU: gemm_simt_kernel<EPI_DGELU><<<grid, 256, 0, s>>>(p); break;
    case EPI_DSWIGLU:
      gemm_simt_kernel<EPI_DSWIGLU><<<grid, 256, 0, s>>>(p);
      break;
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace tp
