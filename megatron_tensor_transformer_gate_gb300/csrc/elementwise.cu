// elementwise.cu — HBM-bound kernels of the TP block.
//
//  * reduce_partials: the materialised g / f reduction
//      out = resid + Dropout(Σ_{i=0}^{n−1} P_i + bias)
//    summed in fp32 in shard order and rounded once ([Grasp-TP] §3: the full
//    bias is added once, after the sum; [Troverld] §II.III: fused bias +
//    dropout + residual add and fused all-reduce + residual add).
//  * dropout_bwd: dZ = dOut ⊙ mask / (1 − p)  ([hjcheng-TP] 单卡backward).
//  * column sums (bias gradients) in two deterministic stages.
//  * RMSNorm forward / backward ([Troverld] §II.III fused norm).
// All loads and stores are 16-byte vectors; grids are a multiple of the SM
// count and grid-stride.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "elementwise.h"
#include "gemm.h"
#include "profile.h"

namespace tp {
namespace {

template <typename T>
struct Vec;  // 16-byte vector of T
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void from_raw(uint4 u, float* v) {
    v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
  }
  __device__ static void store_f32(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
  __device__ static void load(const float* p, float* v) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
  }
  __device__ static void store(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void from_raw(uint4 u, float* v) {
    float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y),
           c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    v[4] = c.x; v[5] = c.y; v[6] = d.x; v[7] = d.y;
  }
  __device__ static void store_f32(float* p, const float* v) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
  __device__ static void load(const __nv_bfloat16* p, float* v) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y),
           c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    v[4] = c.x; v[5] = c.y; v[6] = d.x; v[7] = d.y;
  }
  __device__ static void store(__nv_bfloat16* p, const float* v) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = u;
  }
};

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// v rounded to T and back (the value a T store would hold).
template <typename T>
__device__ __forceinline__ float round_to(float v) {
  return to_f<T>(from_f<T>(v));
}

// acc = Σ_{s<n} P[s·zstride] for one 16-byte vector, summed in fp32 in shard
// order.  The loads of the first AHEAD shards are issued together (AHEAD
// 16-byte requests in flight per thread instead of one), the rest one by one.
template <typename T, int AHEAD = 8>
__device__ __forceinline__ void sum_shards(const T* __restrict__ p, int n,
                                           int64_t zstride, float* acc) {
  constexpr int V = Vec<T>::N;
  uint4 raw[AHEAD];
#pragma unroll
  for (int s = 0; s < AHEAD; ++s)
    if (s < n)
      raw[s] = *reinterpret_cast<const uint4*>(p + (int64_t)s * zstride);
  Vec<T>::from_raw(raw[0], acc);
#pragma unroll
  for (int s = 1; s < AHEAD; ++s) {
    if (s < n) {
      float v[V];
      Vec<T>::from_raw(raw[s], v);
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] += v[q];
    }
  }
  for (int s = AHEAD; s < n; ++s) {
    float v[V];
    Vec<T>::load(p + (int64_t)s * zstride, v);
#pragma unroll
    for (int q = 0; q < V; ++q) acc[q] += v[q];
  }
}

// ------------------------------------------------------- reduce_partials --
template <typename T>
__global__ void __launch_bounds__(256)
    reduce_partials_kernel(const T* __restrict__ P, int n, int64_t count,
                           int64_t zstride, int64_t e0, int64_t h,
                           const T* __restrict__ bias,
                           const T* __restrict__ resid, T* __restrict__ out,
                           int dropout, uint32_t thr, float scale,
                           uint64_t seed) {
  constexpr int V = Vec<T>::N;
  const int64_t nvec = count / V;
  for (int64_t iv = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; iv < nvec;
       iv += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = iv * V;
    float acc[V], v[V];
    sum_shards<T>(P + i, n, zstride, acc);
    if (bias != nullptr) {
      Vec<T>::load(bias + (i % h), v);
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] += v[q];
    }
    if (dropout) {
#pragma unroll
      for (int q = 0; q < V; ++q)
        acc[q] = dropout_keep(seed, (uint64_t)(e0 + i + q), thr)
                     ? acc[q] * scale
                     : 0.0f;
    }
    if (resid != nullptr) {
      Vec<T>::load(resid + i, v);
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] += v[q];
    }
    Vec<T>::store(out + i, acc);
  }
}

// ----------------------------------------------------------- dropout_bwd --
template <typename T>
__global__ void __launch_bounds__(256)
    dropout_bwd_kernel(const T* __restrict__ dout, int64_t count,
                       T* __restrict__ dz, uint32_t thr, float scale,
                       uint64_t seed) {
  constexpr int V = Vec<T>::N;
  const int64_t nvec = count / V;
  for (int64_t iv = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; iv < nvec;
       iv += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = iv * V;
    float v[V];
    Vec<T>::load(dout + i, v);
#pragma unroll
    for (int q = 0; q < V; ++q)
      v[q] = dropout_keep(seed, (uint64_t)(i + q), thr) ? v[q] * scale : 0.0f;
    Vec<T>::store(dz + i, v);
  }
}

// --------------------------------------------------------------- colsum --
// Stage 1: block (cx, chunk) sums rows [chunk·rpc, (chunk+1)·rpc) of columns
// [cx·32·V, (cx+1)·32·V): 32 column groups of V × 8 row lanes; the 8 lane
// partials are combined in a fixed order.
template <typename T>
__global__ void __launch_bounds__(256)
    colsum_stage1(const T* __restrict__ X, int64_t rows, int64_t cols,
                  int64_t ld, int64_t rpc, float* __restrict__ partial) {
  constexpr int V = Vec<T>::N;
  __shared__ float red[8][32 * V + 1];
  const int cg = threadIdx.x & 31, rl = threadIdx.x >> 5;
  const int64_t c0 = (int64_t)blockIdx.x * 32 * V + cg * V;
  const int64_t r_begin = (int64_t)blockIdx.y * rpc;
  const int64_t r_end = min(rows, r_begin + rpc);
  float acc[V];
#pragma unroll
  for (int q = 0; q < V; ++q) acc[q] = 0.0f;
  if (c0 < cols) {
    for (int64_t r = r_begin + rl; r < r_end; r += 8) {
      float v[V];
      Vec<T>::load(X + r * ld + c0, v);
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] += v[q];
    }
  }
#pragma unroll
  for (int q = 0; q < V; ++q) red[rl][cg * V + q] = acc[q];
  __syncthreads();
  for (int c = threadIdx.x; c < 32 * V; c += blockDim.x) {
    float s = 0.0f;
#pragma unroll
    for (int l = 0; l < 8; ++l) s += red[l][c];
    const int64_t col = (int64_t)blockIdx.x * 32 * V + c;
    if (col < cols) partial[(int64_t)blockIdx.y * cols + col] = s;
  }
}

// Stage 2: out[c] = Σ_chunk partial[chunk][c] in chunk order.
// Stage 2: out[c] = Σ_k partial[k][c].  A block of 8 warps takes 32
// columns; warp w adds chunks w, w + 8, … for its lane's column, then warp 0
// adds the 8 warp sums in order (fixed order: reruns are bit-identical).
template <typename T>
__global__ void __launch_bounds__(256)
    colsum_stage2(const float* __restrict__ partial, int chunks, int64_t cols,
                  T* __restrict__ out) {
  __shared__ float red[8][33];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 32 + lane;
  float s = 0.0f;
  if (c < cols)
    for (int k = w; k < chunks; k += 8) s += partial[(int64_t)k * cols + c];
  red[w][lane] = s;
  __syncthreads();
  if (w == 0 && c < cols) {
    float t = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += red[i][lane];
    out[c] = from_f<T>(t);
  }
}

// -------------------------------------------------------------- RMSNorm --
// One block per row (grid-stride over rows); each thread owns columns
// {V·(tid + 256·j)}: the sum of squares in that order, then the row read
// again (from L2) and normalised.  y16 (optional) receives the same rows in
// fp16, the operand of fp16 projections; a value beyond the fp16 range
// records a range error.  Same bits as the norm half of reduce_norm_fwd.
template <typename T>
__global__ void __launch_bounds__(256)
    rmsnorm_fwd_kernel(const T* __restrict__ x, const T* __restrict__ gamma,
                       T* __restrict__ y, __half* __restrict__ y16,
                       float* __restrict__ rstd_out, int64_t rows, int64_t h,
                       float eps, unsigned* status) {
  constexpr int V = Vec<T>::N;
  __shared__ float red[8];
  bool bad = false;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const T* xr = x + r * h;
    float ss = 0.0f;
    for (int64_t c = (int64_t)threadIdx.x * V; c < h; c += 256 * V) {
      float v[V];
      Vec<T>::load(xr + c, v);
#pragma unroll
      for (int q = 0; q < V; ++q) ss += v[q] * v[q];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    const float rs = rsqrtf(tot / (float)h + eps);
    if (threadIdx.x == 0) rstd_out[r] = rs;
    for (int64_t c = (int64_t)threadIdx.x * V; c < h; c += 256 * V) {
      float v[V], g[V];
      Vec<T>::load(xr + c, v);
      Vec<T>::load(gamma + c, g);
#pragma unroll
      for (int q = 0; q < V; ++q) v[q] = v[q] * rs * g[q];
      Vec<T>::store(y + r * h + c, v);
      if (y16 != nullptr) {
        uint32_t u[V / 2];
#pragma unroll
        for (int q = 0; q < V; q += 2) {
          bad |= !(fabsf(v[q]) <= kF16Max) || !(fabsf(v[q + 1]) <= kF16Max);
          u[q / 2] = pack_f16x2(v[q], v[q + 1]);
        }
        __half* dst = y16 + r * h + c;
        if constexpr (V == 8)
          *reinterpret_cast<uint4*>(dst) = make_uint4(u[0], u[1], u[2], u[3]);
        else
          *reinterpret_cast<uint2*>(dst) = make_uint2(u[0], u[1]);
      }
    }
    __syncthreads();
  }
  if (bad) record_error(status, kDevRange, 30);
}

// ------------------------------------------------------- bf16 → fp16 copy --
// dst = fp16(src_0 | src_1 | src_2): up to three bf16 arrays of n_i elements
// (each a multiple of 8) converted into one contiguous fp16 array; a value
// beyond the fp16 range records a range error.  bf16 values of magnitude
// below 2^-14 become fp16 subnormals (below 2^-24: zero).
struct F16Segments {
  const __nv_bfloat16* src[3];
  int64_t end[3];   // cumulative 8-element vectors after segment i
};

__global__ void __launch_bounds__(256)
    convert_f16_kernel(const F16Segments sg, __half* __restrict__ dst,
                       unsigned* status) {
  bool bad = false;
  const int64_t nvec = sg.end[2];
  for (int64_t iv = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; iv < nvec;
       iv += (int64_t)gridDim.x * blockDim.x) {
    const int i = iv < sg.end[0] ? 0 : iv < sg.end[1] ? 1 : 2;
    const int64_t base = i == 0 ? 0 : sg.end[i - 1];
    float v[8];
    Vec<__nv_bfloat16>::load(sg.src[i] + (iv - base) * 8, v);
    uint32_t u[4];
#pragma unroll
    for (int q = 0; q < 8; q += 2) {
      bad |= !(fabsf(v[q]) <= kF16Max) || !(fabsf(v[q + 1]) <= kF16Max);
      u[q / 2] = pack_f16x2(v[q], v[q + 1]);
    }
    reinterpret_cast<uint4*>(dst)[iv] = make_uint4(u[0], u[1], u[2], u[3]);
  }
  if (bad) record_error(status, kDevRange, 31);
}

// One block of 512 threads per chunk of consecutive rows (about one chunk
// per SM); each thread owns the 16-byte column vectors {V·(tid + 512·j)},
// keeps its dγ partial sums in registers (γ comes from L1 each row), and
// loads the next row's dy, x and dres while it finishes the current one.
// Per row: dot = Σ dy·γ·x (block reduction through a double-buffered slot,
// one barrier),
//   dx = dres + rstd·dy·γ − x·rstd³·dot / h,   dγ_partial += dy·x·rstd.
// SUM (the f reduction fused in, Megatron-SP backward): dy is not read but
// formed per row as Σ_{i<n} P_i in fp32, in shard order, rounded once to T —
// the value the materialised reduce would have stored.
template <typename T, int NV, bool SUM>
__global__ void __launch_bounds__(512, 1)
    rmsnorm_bwd_kernel(const T* __restrict__ dy, int n, int64_t zstride,
                       const T* __restrict__ x, const T* __restrict__ gamma,
                       const float* __restrict__ rstd,
                       const T* __restrict__ dres, T* __restrict__ dx,
                       float* __restrict__ dg_partial, int64_t rows, int64_t h,
                       int64_t rpc) {
  constexpr int V = Vec<T>::N;
  __shared__ float red[2][16];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int64_t col[NV];
  bool on[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    col[j] = ((int64_t)threadIdx.x + 512 * j) * V;
    on[j] = col[j] < h;
  }
  float dgacc[NV * V];
#pragma unroll
  for (int q = 0; q < NV * V; ++q) dgacc[q] = 0.0f;
  const int64_t r_begin = (int64_t)blockIdx.x * rpc;
  const int64_t r_end = min(rows, r_begin + rpc);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const bool has_res = dres != nullptr;
  uint4 cd[NV], cx[NV], cr[NV];   // current row, raw 16-byte vectors
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const bool ld = on[j] && r_begin < r_end;
    cd[j] = (!SUM && ld)
                ? *reinterpret_cast<const uint4*>(dy + r_begin * h + col[j])
                : zero;
    cx[j] = ld ? *reinterpret_cast<const uint4*>(x + r_begin * h + col[j])
               : zero;
    cr[j] = (has_res && ld)
                ? *reinterpret_cast<const uint4*>(dres + r_begin * h + col[j])
                : zero;
  }
  for (int64_t r = r_begin; r < r_end; ++r) {
    uint4 nd[NV], nx[NV], nr[NV];
    const bool more = r + 1 < r_end;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      nd[j] = (!SUM && more && on[j])
                  ? *reinterpret_cast<const uint4*>(dy + (r + 1) * h + col[j])
                  : zero;
      nx[j] = (more && on[j])
                  ? *reinterpret_cast<const uint4*>(x + (r + 1) * h + col[j])
                  : zero;
      nr[j] = (has_res && more && on[j])
                  ? *reinterpret_cast<const uint4*>(dres + (r + 1) * h +
                                                    col[j])
                  : zero;
    }
    const float rs = rstd[r];
    float d[NV * V], xv[NV * V], g[NV * V];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if (on[j]) {
        Vec<T>::load(gamma + col[j], g + j * V);
      } else {
#pragma unroll
        for (int q = 0; q < V; ++q) g[j * V + q] = 0.0f;
      }
    }
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if constexpr (SUM) {
        float acc[V];
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = 0.0f;
        if (on[j]) sum_shards<T>(dy + r * h + col[j], n, zstride, acc);
#pragma unroll
        for (int q = 0; q < V; ++q) d[j * V + q] = round_to<T>(acc[q]);
      } else {
        Vec<T>::from_raw(cd[j], d + j * V);
      }
      Vec<T>::from_raw(cx[j], xv + j * V);
    }
    float dot = 0.0f;
#pragma unroll
    for (int i = 0; i < NV * V; ++i) {
      dot = fmaf(d[i] * g[i], xv[i], dot);
      dgacc[i] = fmaf(d[i] * xv[i], rs, dgacc[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0) red[r & 1][w] = dot;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) tot += red[r & 1][i];
    const float coef = rs * rs * rs * tot / (float)h;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if (!on[j]) continue;
      float o[V];
      Vec<T>::from_raw(cr[j], o);
#pragma unroll
      for (int q = 0; q < V; ++q)
        o[q] += rs * d[j * V + q] * g[j * V + q] - xv[j * V + q] * coef;
      Vec<T>::store(dx + r * h + col[j], o);
    }
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      cd[j] = nd[j];
      cx[j] = nx[j];
      cr[j] = nr[j];
    }
  }
#pragma unroll
  for (int j = 0; j < NV; ++j)
    if (on[j])
      Vec<T>::store_f32(dg_partial + (int64_t)blockIdx.x * h + col[j],
                        dgacc + j * V);
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global memory into this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src,
                                         uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// rmsnorm_bwd_kernel<T, NV, true> for rows whose n shard partials fit in
// shared memory: one thread copies the n partial rows of the next row into
// shared memory by bulk copies (the bytes in flight are the copy engine's,
// not registers) while the block finishes the current row.  Per row, as
// there: dy = Σ_{i<n} P_i in fp32 in shard order, rounded once to T, then the
// RMSNorm backward.  Waits are bounded (site 33); the block agrees on every
// outcome before it leaves the loop.
template <typename T, int NV>
__global__ void __launch_bounds__(512, 1)
    rmsnorm_bwd_bulk_kernel(const T* __restrict__ P, int n, int64_t zstride,
                            const T* __restrict__ x,
                            const T* __restrict__ gamma,
                            const float* __restrict__ rstd,
                            const T* __restrict__ dres, T* __restrict__ dx,
                            float* __restrict__ dg_partial, int64_t rows,
                            int64_t h, int64_t rpc, unsigned* status) {
  constexpr int V = Vec<T>::N;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  T* buf = reinterpret_cast<T*>(smem_raw);   // n partial rows of h
  uint64_t* full =
      reinterpret_cast<uint64_t*>(smem_raw + (size_t)n * h * sizeof(T));
  __shared__ float red[2][16];
  __shared__ int abort_flag;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int64_t col[NV];
  bool on[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    col[j] = ((int64_t)threadIdx.x + 512 * j) * V;
    on[j] = col[j] < h;
  }
  float dgacc[NV * V];
#pragma unroll
  for (int q = 0; q < NV * V; ++q) dgacc[q] = 0.0f;
  const int64_t r_begin = (int64_t)blockIdx.x * rpc;
  const int64_t r_end = min(rows, r_begin + rpc);
  const uint32_t row_bytes = (uint32_t)(h * (int64_t)sizeof(T));
  if (threadIdx.x == 0) {
    mbar_init(full, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // thread 0: the n partial rows of row r into buf
  auto issue = [&](int64_t r) {
    mbar_arrive_expect_tx(full, (uint32_t)n * row_bytes);
    for (int i = 0; i < n; ++i)
      bulk_g2s(buf + (int64_t)i * h, P + (int64_t)i * zstride + r * h,
               row_bytes, full);
  };
  if (threadIdx.x == 0 && r_begin < r_end) issue(r_begin);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const bool has_res = dres != nullptr;
  uint4 cx[NV], cr[NV];   // current row of x and dres, raw 16-byte vectors
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    const bool ld = on[j] && r_begin < r_end;
    cx[j] = ld ? *reinterpret_cast<const uint4*>(x + r_begin * h + col[j])
               : zero;
    cr[j] = (has_res && ld)
                ? *reinterpret_cast<const uint4*>(dres + r_begin * h + col[j])
                : zero;
  }
  int64_t r = r_begin;
  for (; r < r_end; ++r) {
    uint4 nx[NV], nr[NV];
    const bool more = r + 1 < r_end;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      nx[j] = (more && on[j])
                  ? *reinterpret_cast<const uint4*>(x + (r + 1) * h + col[j])
                  : zero;
      nr[j] = (has_res && more && on[j])
                  ? *reinterpret_cast<const uint4*>(dres + (r + 1) * h +
                                                    col[j])
                  : zero;
    }
    const bool got =
        mbar_wait(full, (uint32_t)((r - r_begin) & 1),
                  reinterpret_cast<volatile int*>(&abort_flag), status, 33);
    if (!__syncthreads_and(got)) break;
    float d[NV * V], xv[NV * V], g[NV * V];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      float acc[V];
#pragma unroll
      for (int q = 0; q < V; ++q) acc[q] = 0.0f;
      if (on[j]) {
        for (int i = 0; i < n; ++i) {
          float v[V];
          Vec<T>::load(buf + (int64_t)i * h + col[j], v);
#pragma unroll
          for (int q = 0; q < V; ++q) acc[q] += v[q];
        }
      }
#pragma unroll
      for (int q = 0; q < V; ++q) d[j * V + q] = round_to<T>(acc[q]);
    }
    __syncthreads();   // the partial rows are consumed
    if (threadIdx.x == 0 && more) issue(r + 1);
    const float rs = rstd[r];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if (on[j]) {
        Vec<T>::load(gamma + col[j], g + j * V);
      } else {
#pragma unroll
        for (int q = 0; q < V; ++q) g[j * V + q] = 0.0f;
      }
      Vec<T>::from_raw(cx[j], xv + j * V);
    }
    float dot = 0.0f;
#pragma unroll
    for (int i = 0; i < NV * V; ++i) {
      dot = fmaf(d[i] * g[i], xv[i], dot);
      dgacc[i] = fmaf(d[i] * xv[i], rs, dgacc[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0) red[r & 1][w] = dot;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) tot += red[r & 1][i];
    const float coef = rs * rs * rs * tot / (float)h;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if (!on[j]) continue;
      float o[V];
      Vec<T>::from_raw(cr[j], o);
#pragma unroll
      for (int q = 0; q < V; ++q)
        o[q] += rs * d[j * V + q] * g[j * V + q] - xv[j * V + q] * coef;
      Vec<T>::store(dx + r * h + col[j], o);
    }
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      cx[j] = nx[j];
      cr[j] = nr[j];
    }
  }
  if (r < r_end && threadIdx.x == 0) {
    // gave up: let the copies of row r land before the block exits
    volatile int no_abort = 0;
    mbar_wait(full, (uint32_t)((r - r_begin) & 1), &no_abort, nullptr, 0);
  }
#pragma unroll
  for (int j = 0; j < NV; ++j)
    if (on[j])
      Vec<T>::store_f32(dg_partial + (int64_t)blockIdx.x * h + col[j],
                        dgacc + j * V);
}

// rmsnorm_bwd_kernel<T, NV, false> with the rows staged in shared memory:
// one thread copies dy, x and dres (when given) of row r + 2 into one of two
// stages by bulk copies while the block computes row r from the other, so
// two rows of inputs are in flight per SM against one in the register form.
// The arithmetic is the register form's, in the same order, so the results
// are bit-identical to it.  Waits are bounded (site 34); the block agrees on
// every outcome before it leaves the loop.
template <typename T, int NV>
__global__ void __launch_bounds__(512, 1)
    rmsnorm_bwd_staged_kernel(const T* __restrict__ dy,
                              const T* __restrict__ x,
                              const T* __restrict__ gamma,
                              const float* __restrict__ rstd,
                              const T* __restrict__ dres, T* __restrict__ dx,
                              float* __restrict__ dg_partial, int64_t rows,
                              int64_t h, int64_t rpc, unsigned* status) {
  constexpr int V = Vec<T>::N;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int nin = dres != nullptr ? 3 : 2;   // rows a stage holds
  T* const stage0 = reinterpret_cast<T*>(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(
      smem_raw + (size_t)2 * nin * h * sizeof(T));   // [2]
  __shared__ float red[2][16];
  __shared__ int abort_flag;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int64_t col[NV];
  bool on[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    col[j] = ((int64_t)threadIdx.x + 512 * j) * V;
    on[j] = col[j] < h;
  }
  float dgacc[NV * V];
#pragma unroll
  for (int q = 0; q < NV * V; ++q) dgacc[q] = 0.0f;
  const int64_t r_begin = (int64_t)blockIdx.x * rpc;
  const int64_t r_end = min(rows, r_begin + rpc);
  const uint32_t row_bytes = (uint32_t)(h * (int64_t)sizeof(T));
  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // thread 0: dy, x (and dres) of row r into stage sg
  auto issue = [&](int64_t r, int sg) {
    T* st = stage0 + (int64_t)sg * nin * h;
    mbar_arrive_expect_tx(&full[sg], (uint32_t)nin * row_bytes);
    bulk_g2s(st, dy + r * h, row_bytes, &full[sg]);
    bulk_g2s(st + h, x + r * h, row_bytes, &full[sg]);
    if (nin == 3) bulk_g2s(st + 2 * h, dres + r * h, row_bytes, &full[sg]);
  };
  if (threadIdx.x == 0) {
    if (r_begin < r_end) issue(r_begin, 0);
    if (r_begin + 1 < r_end) issue(r_begin + 1, 1);
  }
  int64_t r = r_begin;
  for (; r < r_end; ++r) {
    const int64_t k = r - r_begin;
    const int sg = (int)(k & 1);
    const bool got =
        mbar_wait(&full[sg], (uint32_t)((k >> 1) & 1),
                  reinterpret_cast<volatile int*>(&abort_flag), status, 34);
    if (!__syncthreads_and(got)) break;
    const T* st = stage0 + (int64_t)sg * nin * h;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    float d[NV * V], xv[NV * V], g[NV * V];
    uint4 cr[NV];   // this row's dres, raw 16-byte vectors
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const uint4 cd =
          on[j] ? *reinterpret_cast<const uint4*>(st + col[j]) : zero;
      const uint4 cx =
          on[j] ? *reinterpret_cast<const uint4*>(st + h + col[j]) : zero;
      cr[j] = (on[j] && nin == 3)
                  ? *reinterpret_cast<const uint4*>(st + 2 * h + col[j])
                  : zero;
      Vec<T>::from_raw(cd, d + j * V);
      Vec<T>::from_raw(cx, xv + j * V);
    }
    __syncthreads();   // stage sg consumed
    if (threadIdx.x == 0 && r + 2 < r_end) issue(r + 2, sg);
    const float rs = rstd[r];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if (on[j]) {
        Vec<T>::load(gamma + col[j], g + j * V);
      } else {
#pragma unroll
        for (int q = 0; q < V; ++q) g[j * V + q] = 0.0f;
      }
    }
    float dot = 0.0f;
#pragma unroll
    for (int i = 0; i < NV * V; ++i) {
      dot = fmaf(d[i] * g[i], xv[i], dot);
      dgacc[i] = fmaf(d[i] * xv[i], rs, dgacc[i]);
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1)
      dot += __shfl_xor_sync(0xffffffffu, dot, o2);
    if (lane == 0) red[r & 1][w] = dot;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) tot += red[r & 1][i];
    const float coef = rs * rs * rs * tot / (float)h;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      if (!on[j]) continue;
      float o[V];
      Vec<T>::from_raw(cr[j], o);
#pragma unroll
      for (int q = 0; q < V; ++q)
        o[q] += rs * d[j * V + q] * g[j * V + q] - xv[j * V + q] * coef;
      Vec<T>::store(dx + r * h + col[j], o);
    }
  }
  if (r < r_end && threadIdx.x == 0) {
    // gave up: let the copies of rows r and r + 1 land before the block exits
    volatile int no_abort = 0;
    for (int64_t k = r - r_begin; k < min(r_end - r_begin, r - r_begin + 2);
         ++k)
      mbar_wait(&full[k & 1], (uint32_t)((k >> 1) & 1), &no_abort, nullptr, 0);
  }
#pragma unroll
  for (int j = 0; j < NV; ++j)
    if (on[j])
      Vec<T>::store_f32(dg_partial + (int64_t)blockIdx.x * h + col[j],
                        dgacc + j * V);
}

// The g reduction with the next block's RMSNorm fused in (Megatron-SP
// forward, [Troverld] §III.III: the reduce-scatter leaves each rank its rows
// of the block output, the token-wise ops of the next block run on them, and
// the all-gather hands the normalised rows to the next column-parallel
// GEMM — on one device the gathered buffer is the output itself).  One block
// of 256 threads per row, thread t owning the column vectors {V·(t + 256·j)}
// as the RMSNorm forward does:
//   out = resid + Dropout(Σ_{i<n} P_i + bias)   (the materialised reduce)
//   rstd = 1/√(mean(out²) + ε),  y = out·rstd·γ  (the RMSNorm forward, on the
//                                                 stored values of out)
// Both halves round and reduce exactly as the two separate kernels do.  y16
// (optional) receives the normalised rows also in fp16; a value beyond the
// fp16 range records a range error.  out may be NULL (not stored).
template <typename T, int NV, int AHEAD>
__global__ void __launch_bounds__(256)
    reduce_norm_fwd_kernel(const T* __restrict__ P, int n, int64_t zstride,
                           const T* __restrict__ bias,
                           const T* __restrict__ resid, T* __restrict__ out,
                           int dropout, uint32_t thr, float scale,
                           uint64_t seed, const T* __restrict__ gamma,
                           T* __restrict__ y, __half* __restrict__ y16,
                           float* __restrict__ rstd_out, int64_t rows,
                           int64_t h, float eps, unsigned* status) {
  constexpr int V = Vec<T>::N;
  __shared__ float red[8];
  bool bad = false;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    float row[NV * V];
    float ss = 0.0f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int64_t c = ((int64_t)threadIdx.x + 256 * j) * V;
      if (c >= h) break;
      const int64_t i0 = r * h + c;
      float acc[V], v[V];
      sum_shards<T, AHEAD>(P + i0, n, zstride, acc);
      if (bias != nullptr) {
        Vec<T>::load(bias + c, v);
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] += v[q];
      }
      if (dropout) {
#pragma unroll
        for (int q = 0; q < V; ++q)
          acc[q] = dropout_keep(seed, (uint64_t)(i0 + q), thr)
                       ? acc[q] * scale
                       : 0.0f;
      }
      if (resid != nullptr) {
        Vec<T>::load(resid + i0, v);
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] += v[q];
      }
      if (out != nullptr) Vec<T>::store(out + i0, acc);
#pragma unroll
      for (int q = 0; q < V; ++q) {
        row[j * V + q] = round_to<T>(acc[q]);
        ss += row[j * V + q] * row[j * V + q];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    const float rs = rsqrtf(tot / (float)h + eps);
    if (threadIdx.x == 0) rstd_out[r] = rs;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int64_t c = ((int64_t)threadIdx.x + 256 * j) * V;
      if (c >= h) break;
      float g[V], v[V];
      Vec<T>::load(gamma + c, g);
#pragma unroll
      for (int q = 0; q < V; ++q) v[q] = row[j * V + q] * rs * g[q];
      Vec<T>::store(y + r * h + c, v);
      if (y16 != nullptr) {
        uint32_t u[V / 2];
#pragma unroll
        for (int q = 0; q < V; q += 2) {
          bad |= !(fabsf(v[q]) <= kF16Max) || !(fabsf(v[q + 1]) <= kF16Max);
          u[q / 2] = pack_f16x2(v[q], v[q + 1]);
        }
        __half* dst = y16 + r * h + c;
        if constexpr (V == 8)
          *reinterpret_cast<uint4*>(dst) = make_uint4(u[0], u[1], u[2], u[3]);
        else
          *reinterpret_cast<uint2*>(dst) = make_uint2(u[0], u[1]);
      }
    }
    __syncthreads();
  }
  if (bad) record_error(status, kDevRange, 32);
}

int grid_for(int64_t work_items, int per_block) {
  const int64_t blocks = (work_items + per_block - 1) / per_block;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  return (int)std::max<int64_t>(1, std::min(blocks, cap));
}

}  // namespace

// ------------------------------------------------------------------- host --
template <typename T>
int reduce_partials(const void* P, int n, int64_t rows, int64_t h,
                    int64_t zstride, int64_t row0, const void* bias,
                    const void* resid, void* out, const DropoutSpec& d,
                    void* stream) {
  const int64_t count = rows * h;
  if (count == 0) return cudaSuccess;
  const int grid = grid_for(count / Vec<T>::N, 256);
  ProfScope ps(stream, KF_REDUCE, (double)n * count,
               (double)sizeof(T) * count *
                   (n + 1 + (resid != nullptr ? 1 : 0)));
  reduce_partials_kernel<T><<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const T*>(P), n, count, zstride, row0 * h, h,
      static_cast<const T*>(bias),
      static_cast<const T*>(resid), static_cast<T*>(out), d.enabled, d.thr,
      d.scale, d.seed);
  count_launch();
  return cudaGetLastError();
}

template <typename T>
int dropout_bwd(const void* dout, int64_t count, void* dz, const DropoutSpec& d,
                void* stream) {
  if (count == 0) return cudaSuccess;
  const int grid = grid_for(count / Vec<T>::N, 256);
  ProfScope ps(stream, KF_ELEMENTWISE, 0.0, 2.0 * sizeof(T) * count);
  dropout_bwd_kernel<T><<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const T*>(dout), count, static_cast<T*>(dz), d.thr, d.scale,
      d.seed);
  count_launch();
  return cudaGetLastError();
}

int colsum_chunks(int64_t rows) {
  return (int)std::max<int64_t>(1, std::min<int64_t>(64, (rows + 63) / 64));
}

size_t colsum_scratch_bytes(int64_t rows, int64_t cols) {
  return (size_t)colsum_chunks(rows) * (size_t)cols * sizeof(float);
}

template <typename T>
int colsum(const void* X, int64_t rows, int64_t cols, int64_t ld, void* out,
           float* scratch, void* stream) {
  if (cols == 0) return cudaSuccess;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int chunks = colsum_chunks(rows);
  const int64_t rpc = (rows + chunks - 1) / chunks;
  constexpr int V = Vec<T>::N;
  dim3 g1((unsigned)((cols + 32 * V - 1) / (32 * V)), (unsigned)chunks);
  ProfScope ps(stream, KF_ELEMENTWISE, (double)rows * cols,
               (double)sizeof(T) * rows * cols);
  colsum_stage1<T><<<g1, 256, 0, s>>>(static_cast<const T*>(X), rows, cols, ld,
                                      rpc, scratch);
  colsum_stage2<T><<<(unsigned)((cols + 31) / 32), 256, 0, s>>>(scratch, chunks, cols,
                                                       static_cast<T*>(out));
  count_launch(2);
  return cudaGetLastError();
}

template <typename T, int AHEAD>
int norm_rows(const void* P, int n, int64_t zstride, const void* bias,
              const void* resid, void* out, const DropoutSpec& d,
              const void* gamma, void* y, void* y16, float* rstd, int64_t rows,
              int64_t h, float eps, unsigned* status, int family,
              double bytes, void* stream) {
  if (rows == 0) return cudaSuccess;
  constexpr int V = Vec<T>::N;
  const int64_t sweeps = (h + 256 * V - 1) / (256 * V);
  if (sweeps > 8 || n < 1) return cudaErrorInvalidValue;
  const int grid = (int)std::min<int64_t>(rows, (int64_t)device_sm_count() * 8);
  ProfScope ps(stream, family, (double)(n + 3) * rows * h, bytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
#define TP_FWD(NVV)                                                           \
  reduce_norm_fwd_kernel<T, NVV, AHEAD><<<grid, 256, 0, s>>>(                 \
      static_cast<const T*>(P), n, zstride, static_cast<const T*>(bias),      \
      static_cast<const T*>(resid), static_cast<T*>(out), d.enabled, d.thr,   \
      d.scale, d.seed, static_cast<const T*>(gamma), static_cast<T*>(y),      \
      static_cast<__half*>(y16), rstd, rows, h, eps, status)
  if (sweeps <= 1) TP_FWD(1);
  else if (sweeps <= 2) TP_FWD(2);
  else if (sweeps <= 4) TP_FWD(4);
  else TP_FWD(8);
#undef TP_FWD
  count_launch();
  return cudaGetLastError();
}

template <typename T>
int rmsnorm_fwd(const void* x, const void* gamma, void* y, float* rstd,
                int64_t rows, int64_t h, float eps, void* stream, void* y16,
                unsigned* status) {
  if (rows == 0) return cudaSuccess;
  const int grid = (int)std::min<int64_t>(rows, (int64_t)device_sm_count() * 8);
  ProfScope ps(stream, KF_NORM, 4.0 * rows * h,
               (2.0 * sizeof(T) + (y16 != nullptr ? 2.0 : 0.0)) * rows * h);
  rmsnorm_fwd_kernel<T><<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const T*>(x), static_cast<const T*>(gamma),
      static_cast<T*>(y), static_cast<__half*>(y16), rstd, rows, h, eps,
      status);
  count_launch();
  return cudaGetLastError();
}

int convert_f16(const void* const* srcs, const int64_t* ns, int nseg,
                void* dst, unsigned* status, void* stream) {
  if (nseg < 1 || nseg > 3) return cudaErrorInvalidValue;
  F16Segments sg;
  int64_t tot = 0;
  for (int i = 0; i < 3; ++i) {
    const int64_t n = i < nseg ? ns[i] : 0;
    if (n % 8) return cudaErrorInvalidValue;
    sg.src[i] = i < nseg ? static_cast<const __nv_bfloat16*>(srcs[i]) : nullptr;
    tot += n / 8;
    sg.end[i] = tot;
  }
  if (tot == 0) return cudaSuccess;
  const int grid = grid_for(tot, 256);
  ProfScope ps(stream, KF_ELEMENTWISE, 0.0, 32.0 * tot);
  convert_f16_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      sg, static_cast<__half*>(dst), status);
  count_launch();
  return cudaGetLastError();
}

// A fixed chunk count keeps the scratch size independent of the device.
int rmsnorm_bwd_chunks(int64_t rows) {
  return (int)std::max<int64_t>(1, std::min<int64_t>(rows, 256));
}

size_t rmsnorm_bwd_scratch(int64_t rows, int64_t h) {
  return (size_t)rmsnorm_bwd_chunks(rows) * (size_t)h * sizeof(float);
}

// The RMSNorm backward; with n > 1 dy is the sum of n partials (zstride
// elements apart) formed in the kernel.
// The bulk-copy form of the summed backward (n partial rows in shared
// memory) up to this many bytes of partials per row.
constexpr int64_t kBulkRowBytes = 200 * 1024;

template <typename T, int NV>
int launch_rmsnorm_bwd_bulk(int chunks, size_t smem, cudaStream_t s,
                            const T* P, int n, int64_t zstride, const T* x,
                            const T* gamma, const float* rstd, const T* dres,
                            T* dx, float* scratch, int64_t rows, int64_t h,
                            int64_t rpc, unsigned* status) {
  static cudaError_t attr = cudaFuncSetAttribute(
      rmsnorm_bwd_bulk_kernel<T, NV>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kBulkRowBytes + 64));
  if (attr != cudaSuccess) return attr;
  rmsnorm_bwd_bulk_kernel<T, NV><<<chunks, 512, smem, s>>>(
      P, n, zstride, x, gamma, rstd, dres, dx, scratch, rows, h, rpc, status);
  return cudaSuccess;
}

// The staged form of the plain backward: two stages of dy, x and dres rows
// in shared memory, up to this many bytes.
constexpr int64_t kStagedBytes = 200 * 1024;

template <typename T, int NV>
int launch_rmsnorm_bwd_staged(int chunks, size_t smem, cudaStream_t s,
                              const T* dy, const T* x, const T* gamma,
                              const float* rstd, const T* dres, T* dx,
                              float* scratch, int64_t rows, int64_t h,
                              int64_t rpc, unsigned* status) {
  static cudaError_t attr = cudaFuncSetAttribute(
      rmsnorm_bwd_staged_kernel<T, NV>,
      cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kStagedBytes + 64));
  if (attr != cudaSuccess) return attr;
  rmsnorm_bwd_staged_kernel<T, NV><<<chunks, 512, smem, s>>>(
      dy, x, gamma, rstd, dres, dx, scratch, rows, h, rpc, status);
  return cudaSuccess;
}

template <typename T>
int rmsnorm_bwd_sum(const void* dy, int n, int64_t zstride, const void* x,
                    const void* gamma, const float* rstd, const void* dres,
                    void* dx, void* dgamma, float* scratch, int64_t rows,
                    int64_t h, void* stream, unsigned* status) {
  if (rows == 0) return cudaSuccess;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // at most one chunk per SM (the scratch holds rmsnorm_bwd_chunks rows)
  const int chunks = (int)std::min<int64_t>(rmsnorm_bwd_chunks(rows),
                                            device_sm_count());
  const int64_t rpc = (rows + chunks - 1) / chunks;
  constexpr int V = Vec<T>::N;
  // 16-byte vectors per thread: 512 threads × V columns per sweep
  const int64_t sweeps = (h + 512 * V - 1) / (512 * V);
  if (sweeps > 4 || n < 1) return cudaErrorInvalidValue;
  const int kind = n > 1 ? KF_REDUCE : KF_NORM;
  ProfScope ps(stream, kind, 8.0 * rows * h + (n - 1.0) * rows * h,
               (double)sizeof(T) * rows * h * (n + (dres != nullptr ? 3 : 2)));
  const T* dyp = static_cast<const T*>(dy);
  const T* xp = static_cast<const T*>(x);
  const T* gp = static_cast<const T*>(gamma);
  const T* rp = static_cast<const T*>(dres);
  T* dxp = static_cast<T*>(dx);
#define TP_BWD(NVV, SUMV)                                                     \
  rmsnorm_bwd_kernel<T, NVV, SUMV><<<chunks, 512, 0, s>>>(                    \
      dyp, n, zstride, xp, gp, rstd, rp, dxp, scratch, rows, h, rpc)
  const int64_t part_bytes = (int64_t)n * h * (int64_t)sizeof(T);
  const int64_t staged_bytes =
      2 * (dres != nullptr ? 3 : 2) * h * (int64_t)sizeof(T) + 16;
  if (n == 1 && staged_bytes <= kStagedBytes) {
    int err;
    if (sweeps <= 1)
      err = launch_rmsnorm_bwd_staged<T, 1>(chunks, (size_t)staged_bytes, s,
                                            dyp, xp, gp, rstd, rp, dxp,
                                            scratch, rows, h, rpc, status);
    else if (sweeps <= 2)
      err = launch_rmsnorm_bwd_staged<T, 2>(chunks, (size_t)staged_bytes, s,
                                            dyp, xp, gp, rstd, rp, dxp,
                                            scratch, rows, h, rpc, status);
    else
      err = launch_rmsnorm_bwd_staged<T, 4>(chunks, (size_t)staged_bytes, s,
                                            dyp, xp, gp, rstd, rp, dxp,
                                            scratch, rows, h, rpc, status);
    if (err) return err;
  } else if (n > 1 && part_bytes <= kBulkRowBytes) {
    const size_t smem = (size_t)part_bytes + 16;
    int err;
    if (sweeps <= 1)
      err = launch_rmsnorm_bwd_bulk<T, 1>(chunks, smem, s, dyp, n, zstride, xp,
                                          gp, rstd, rp, dxp, scratch, rows, h,
                                          rpc, status);
    else if (sweeps <= 2)
      err = launch_rmsnorm_bwd_bulk<T, 2>(chunks, smem, s, dyp, n, zstride, xp,
                                          gp, rstd, rp, dxp, scratch, rows, h,
                                          rpc, status);
    else
      err = launch_rmsnorm_bwd_bulk<T, 4>(chunks, smem, s, dyp, n, zstride, xp,
                                          gp, rstd, rp, dxp, scratch, rows, h,
                                          rpc, status);
    if (err) return err;
  } else if (n == 1) {
    if (sweeps <= 1) TP_BWD(1, false);
    else if (sweeps <= 2) TP_BWD(2, false);
    else TP_BWD(4, false);
  } else {
    if (sweeps <= 1) TP_BWD(1, true);
    else if (sweeps <= 2) TP_BWD(2, true);
    else TP_BWD(4, true);
  }
#undef TP_BWD
  colsum_stage2<T><<<(unsigned)((h + 31) / 32), 256, 0, s>>>(scratch, chunks, h,
                                                    static_cast<T*>(dgamma));
  count_launch(2);
  return cudaGetLastError();
}

template <typename T>
int rmsnorm_bwd(const void* dy, const void* x, const void* gamma,
                const float* rstd, const void* dres, void* dx, void* dgamma,
                float* scratch, int64_t rows, int64_t h, void* stream) {
  return rmsnorm_bwd_sum<T>(dy, 1, 0, x, gamma, rstd, dres, dx, dgamma,
                            scratch, rows, h, stream, nullptr);
}

template <typename T>
int reduce_norm_fwd(const void* P, int n, int64_t zstride, const void* bias,
                    const void* resid, void* out, const DropoutSpec& d,
                    const void* gamma, void* y, void* y16, float* rstd,
                    int64_t rows, int64_t h, float eps, unsigned* status,
                    void* stream) {
  const double bytes = (double)sizeof(T) * rows * h *
                           (n + 2 + (resid != nullptr ? 1 : 0)) +
                       (y16 != nullptr ? 2.0 * rows * h : 0.0);
  return norm_rows<T, 8>(P, n, zstride, bias, resid, out, d, gamma, y, y16,
                         rstd, rows, h, eps, status, KF_REDUCE, bytes, stream);
}

#define TP_INST(T)                                                            \
  template int reduce_partials<T>(const void*, int, int64_t, int64_t,         \
                                  int64_t, int64_t, const void*, const void*, \
                                  void*, const DropoutSpec&, void*);          \
  template int dropout_bwd<T>(const void*, int64_t, void*, const DropoutSpec&, \
                              void*);                                         \
  template int colsum<T>(const void*, int64_t, int64_t, int64_t, void*,       \
                         float*, void*);                                      \
  template int rmsnorm_fwd<T>(const void*, const void*, void*, float*,        \
                              int64_t, int64_t, float, void*, void*,          \
                              unsigned*);                                     \
  template int rmsnorm_bwd<T>(const void*, const void*, const void*,          \
                              const float*, const void*, void*, void*,        \
                              float*, int64_t, int64_t, void*);               \
  template int rmsnorm_bwd_sum<T>(const void*, int, int64_t, const void*,     \
                                  const void*, const float*, const void*,     \
                                  void*, void*, float*, int64_t, int64_t,     \
                                  void*, unsigned*);                          \
  template int reduce_norm_fwd<T>(const void*, int, int64_t, const void*,     \
                                  const void*, void*, const DropoutSpec&,     \
                                  const void*, void*, void*, float*, int64_t, \
                                  int64_t, float, unsigned*, void*);
TP_INST(float)
TP_INST(__nv_bfloat16)
#undef TP_INST

// ------------------------------------------- RMSNorm backward, no allocation --
// Callers that cannot allocate device memory (see tp_rmsnorm_bwd_noalloc) get
// the dγ partial sums in this fixed array instead of a caller scratch buffer:
// one fp32 row of h partial sums per row chunk, at most 256 chunks × 8192
// columns = 8 MiB, held by every GPU that loads the library until the process
// exits.  Every chunk row that a call uses is fully written by that call
// before it is read, so nothing has to be cleared between calls; calls that
// overlap on the GPU share the array and race.
static __device__ __align__(256) float
    g_norm_scratch[256 * kNoallocNormMaxH];

namespace {
std::mutex g_norm_mu;
float* g_norm_ptr[64];
}  // namespace

// Device address of g_norm_scratch for the current device.  The host-side
// name of a __device__ array is only a stand-in for it, so the address is
// looked up once per device (with that device current) and cached.
int norm_scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_norm_mu);
  if (g_norm_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_norm_scratch);
    if (e != cudaSuccess) return e;
    g_norm_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_norm_ptr[dev];
  return cudaSuccess;
}

template <typename T>
int rmsnorm_bwd_noalloc(const void* dy, const void* x, const void* gamma,
                        const float* rstd, const void* dres, void* dx,
                        void* dgamma, int64_t rows, int64_t h, void* stream) {
  if (h > kNoallocNormMaxH ||
      rmsnorm_bwd_scratch(rows, h) > sizeof(g_norm_scratch))
    return cudaErrorInvalidValue;
  float* scratch = nullptr;
  const int e = norm_scratch_address(&scratch);
  if (e != cudaSuccess) return e;
  return rmsnorm_bwd<T>(dy, x, gamma, rstd, dres, dx, dgamma, scratch, rows, h,
                        stream);
}

template int rmsnorm_bwd_noalloc<float>(const void*, const void*, const void*,
                                        const float*, const void*, void*,
                                        void*, int64_t, int64_t, void*);
template int rmsnorm_bwd_noalloc<__nv_bfloat16>(const void*, const void*,
                                                const void*, const float*,
                                                const void*, void*, void*,
                                                int64_t, int64_t, void*);

// ------------------------------------------------------- bounded waits --
// One thread waits on an mbarrier that nothing completes, through the same
// bounded wait every kernel of the library uses: the wait gives up after
// kWaitTimeoutCycles, records kDevTimeout (site 90) in the status word and
// the kernel returns, leaving the context usable.
__global__ void wait_timeout_selftest_kernel(unsigned* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    mbar_wait(&bar, 0, reinterpret_cast<volatile int*>(&abort_flag), status,
              90);
}

int selftest_wait_timeout(unsigned* status, void* stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace tp
