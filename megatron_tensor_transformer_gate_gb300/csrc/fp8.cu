// fp8.cu — per-tensor scaled E4M3 quantization of bf16 tensors.
//
// The quantize step of the FP8 fused kernel ([Troverld] §II.III: quantize +
// compute + dequantize):
//   amax  = max |x| over the tensor (exact: bf16 values, float max),
//   scale = 448 / amax in fp32 (round to nearest; 1 when amax = 0),
//   q     = E4M3 code of fp32(x·scale), round to nearest even, values beyond
//           ±448 saturated (cvt ... satfinite),
// so that q / scale approximates x and a GEMM of two quantized operands is
// dequantized by 1 / (scale_a·scale_b).  Two kernels: a grid-wide max (one
// atomicMax of the float's bits per block: non-negative floats order like
// their bit patterns) and the conversion, which also writes the scale.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "elementwise.h"
#include "gemm.h"
#include "profile.h"

namespace tp {
namespace {

constexpr float kE4M3Max = 448.0f;

__global__ void __launch_bounds__(256)
    amax_kernel(const uint4* __restrict__ x, int64_t nvec,
                unsigned* __restrict__ amax_bits) {
  __shared__ float red[8];
  float m = 0.0f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 u = x[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = unpack_bf16x2(w[k]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) b = fmaxf(b, red[i]);
    atomicMax(amax_bits, __float_as_uint(b));
  }
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo =
      __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi =
      __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

__global__ void __launch_bounds__(256)
    quantize_kernel(const uint4* __restrict__ x, int64_t nvec,
                    uint2* __restrict__ q,
                    const unsigned* __restrict__ amax_bits,
                    float* __restrict__ scale_out) {
  const float amax = __uint_as_float(*amax_bits);
  const float scale = amax == 0.0f ? 1.0f : __fdiv_rn(kE4M3Max, amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = scale;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 u = x[i];
    const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y),
                 c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
    uint2 o;
    o.x = e4m3x4(__fmul_rn(a.x, scale), __fmul_rn(a.y, scale),
                 __fmul_rn(b.x, scale), __fmul_rn(b.y, scale));
    o.y = e4m3x4(__fmul_rn(c.x, scale), __fmul_rn(c.y, scale),
                 __fmul_rn(d.x, scale), __fmul_rn(d.y, scale));
    q[i] = o;
  }
}

}  // namespace

int quantize_fp8(const void* x, int64_t n, void* q, float* scale,
                 unsigned* amax_work, void* stream) {
  if (n % 8) return cudaErrorInvalidValue;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int err = cudaMemsetAsync(amax_work, 0, sizeof(unsigned), s);
  if (err) return err;
  const int64_t nvec = n / 8;
  const int grid = (int)std::max<int64_t>(
      1, std::min<int64_t>((nvec + 255) / 256, (int64_t)device_sm_count() * 8));
  {
    ProfScope ps(stream, KF_QUANT, 0.0, 2.0 * n);
    amax_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4*>(x), nvec,
                                     amax_work);
  }
  {
    ProfScope ps(stream, KF_QUANT, 0.0, 3.0 * n);
    quantize_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4*>(x), nvec,
                                         static_cast<uint2*>(q), amax_work,
                                         scale);
  }
  count_launch(2);
  return cudaGetLastError();
}

}  // namespace tp
