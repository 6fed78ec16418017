// elementwise.h — host launchers of the HBM-bound kernels (elementwise.cu).
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace tp {

struct DropoutSpec {
  int enabled = 0;
  uint32_t thr = 0;       // keep iff the top 24 bits of the draw ≥ thr
  float scale = 1.0f;     // 1 / (1 − p)
  uint64_t seed = 0;
};

// out = resid + Dropout(Σ_{i<n} P[i] + bias) over rows [rows, h]; partial i
// starts zstride elements after partial i−1; row0 is the first row's index
// in the whole [T, h] tensor (the dropout draw of element (t, j) is t·h + j).
template <typename T>
int reduce_partials(const void* P, int n, int64_t rows, int64_t h,
                    int64_t zstride, int64_t row0, const void* bias,
                    const void* resid, void* out, const DropoutSpec& d,
                    void* stream);
// dz = dout ⊙ mask · scale over `count` elements of a [*, h] tensor.
template <typename T>
int dropout_bwd(const void* dout, int64_t count, void* dz,
                const DropoutSpec& d, void* stream);
// out[c] = Σ_r X[r, c] (deterministic two-stage; scratch from
// colsum_scratch_bytes).
size_t colsum_scratch_bytes(int64_t rows, int64_t cols);
template <typename T>
int colsum(const void* X, int64_t rows, int64_t cols, int64_t ld, void* out,
           float* scratch, void* stream);
// y16 (optional): the normalised rows also in fp16 (range errors recorded in
// status).
template <typename T>
int rmsnorm_fwd(const void* x, const void* gamma, void* y, float* rstd,
                int64_t rows, int64_t h, float eps, void* stream,
                void* y16 = nullptr, unsigned* status = nullptr);
// dst = fp16 of nseg (1 to 3) bf16 arrays srcs[i] of ns[i] values (each a
// multiple of 8, 16-byte aligned), one after another in one launch; a value
// beyond the fp16 range records a range error in status.
int convert_f16(const void* const* srcs, const int64_t* ns, int nseg,
                void* dst, unsigned* status, void* stream);
size_t rmsnorm_bwd_scratch(int64_t rows, int64_t h);
template <typename T>
int rmsnorm_bwd(const void* dy, const void* x, const void* gamma,
                const float* rstd, const void* dres, void* dx, void* dgamma,
                float* scratch, int64_t rows, int64_t h, void* stream);
// Megatron-SP fusions (the reduce-scatter and the token-wise op after it):
// rmsnorm_bwd_sum takes dy as the sum of n partials zstride elements apart
// (rounded once to T, as the materialised reduce stores it), then runs the
// RMSNorm backward (n = 1: plain dy, same as rmsnorm_bwd);
// reduce_norm_fwd writes out = resid + Dropout(Σ P_i + bias) and the RMSNorm
// of those stored rows (y, optional fp16 copy y16, rstd) in one pass.  Both
// give the same bits as the separate kernels.
// (status: the device status word a bounded wait of the n > 1 form records
// a time-out in.)
template <typename T>
int rmsnorm_bwd_sum(const void* dy, int n, int64_t zstride, const void* x,
                    const void* gamma, const float* rstd, const void* dres,
                    void* dx, void* dgamma, float* scratch, int64_t rows,
                    int64_t h, void* stream, unsigned* status = nullptr);
template <typename T>
int reduce_norm_fwd(const void* P, int n, int64_t zstride, const void* bias,
                    const void* resid, void* out, const DropoutSpec& d,
                    const void* gamma, void* y, void* y16, float* rstd,
                    int64_t rows, int64_t h, float eps, unsigned* status,
                    void* stream);

// The RMSNorm backward with its dγ partial sums in a fixed device array
// (no caller scratch); h ≤ kNoallocNormMaxH.
constexpr int64_t kNoallocNormMaxH = 8192;
template <typename T>
int rmsnorm_bwd_noalloc(const void* dy, const void* x, const void* gamma,
                        const float* rstd, const void* dres, void* dx,
                        void* dgamma, int64_t rows, int64_t h, void* stream);

// Per-tensor scaled E4M3 codes of n bf16 values (n a multiple of 8): writes
// q (n bytes) and the scale (one device float); amax_work is one device word
// of scratch.  fp8.cu.
// A kernel whose one wait runs out (the failure path of the bounded waits).
int selftest_wait_timeout(unsigned* status, void* stream);
int quantize_fp8(const void* x, int64_t n, void* q, float* scale,
                 unsigned* amax_work, void* stream);

}  // namespace tp
