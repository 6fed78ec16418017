// gemm.h — host-side description of one GEMM launch of the TP block.
//
// Every projection of the block is   C[m, n] = Σ_parts Σ_segments Σ_k
// A_p[m, k]·B_p[n, k]   followed by a fused epilogue.  The segment structure
// is how the n logical shards appear in a launch:
//  * column-parallel projections (W1, gate/up, Wq/Wk/Wv): one segment; the
//    shards are disjoint column ranges of the same output, so one tile grid
//    over all columns is exactly the union of the n per-rank GEMMs;
//  * row-parallel projections and the input gradients (W2, Wo, dX): the
//    reduction axis K is cut into the n shard segments.  In FUSED mode one
//    tile accumulates all segments in order 0..n−1 (the g / f sum happens in
//    the accumulator); in MATERIALISED mode batch z = shard z consumes only
//    its own segments and writes a partial that a reduce kernel sums.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace tp {

enum EpiKind : int {
  EPI_STORE = 0,    // C (+ bias[n]) → dropout → (+ resid[m, n]) → out
  EPI_GELU = 1,     // H = C (+ bias) → out;  A = GeLU(H) → out2
  EPI_SWIGLU = 2,   // G = C_gate, U = C_up → out, out2;  A = SiLU(G)·U → out3
  EPI_DGELU = 3,    // dH = C ⊙ GeLU'(aux1) → out
  EPI_DSWIGLU = 4,  // dG = C ⊙ aux2 ⊙ SiLU'(aux1) → out; dU = C ⊙ SiLU(aux1) → out2
};

struct GemmOperand {
  const void* ptr = nullptr;
  int64_t ld = 0;     // elements between rows of the stored matrix
  int mn_major = 0;   // 0: (r, k) at ptr[r·ld + k];  1: (r, k) at ptr[k·ld + r]
  int64_t rows = 0;   // extent along M (for A) or N (for B)
};

struct GemmPart {
  GemmOperand a, b;
  GemmOperand b2;        // EPI_SWIGLU: the up-projection rows (b = gate rows)
  int64_t kseg = 0;      // K extent of one segment
  int nseg = 1;          // segments along the operands' K axis
  int seg_z_stride = 0;  // batch z starts at segment z·seg_z_stride
  int nsub = 1;          // segments consumed per tile
  int seg_sub_stride = 1;
};

struct GemmEpilogue {
  EpiKind kind = EPI_STORE;
  void* out = nullptr;
  int64_t ldo = 0;
  int64_t out_z_stride = 0;  // elements between batch outputs
  void* out2 = nullptr;
  void* out3 = nullptr;
  int64_t ldo2 = 0;          // for out2 and out3
  const void* bias = nullptr;
  const void* resid = nullptr;
  int64_t ldr = 0;
  const void* aux1 = nullptr;
  const void* aux2 = nullptr;
  int64_t ld_aux = 0;
  int dropout = 0;
  uint32_t drop_thr = 0;
  float drop_scale = 1.0f;
  uint64_t seed = 0;
  // EPI_STORE only: write fp16 instead of bf16 (the attention-core operands);
  // a value beyond the fp16 range records a range error in the status word
  int out_f16 = 0;
  // EPI_STORE only: output columns [split1, split2) go to out2 (row stride
  // ldo2) and [split2, N) to out3 (row stride ldo3), each from its own column
  // 0 — one launch writing several tensors (0 = no split; multiples of 32)
  int64_t split1 = 0, split2 = 0, ldo3 = 0;
  // FP8 operands (GemmProblem::dtype 2): device pointers to the per-tensor
  // quantization scales of A and B; the accumulator is multiplied by
  // 1 / (scale_a·scale_b) before the rest of the epilogue
  const float* scale_a = nullptr;
  const float* scale_b = nullptr;
};

struct GemmProblem {
  // tp_dtype: 0 fp32 (CUDA cores), 1 bf16 (tensor cores), 2 E4M3 operands
  // (tensor cores, K-major only, bf16 outputs, scales in the epilogue)
  int dtype = 1;
  // dtype 1 only: the operands are fp16 instead of bf16 (same layouts)
  int f16 = 0;
  int64_t M = 0, N = 0;
  int nparts = 1;
  GemmPart parts[3];
  int nz = 1;
  GemmEpilogue epi;
};

// Launchers (return a cudaError_t value; 0 = success).
int launch_gemm_tc(const GemmProblem& p, void* stream, unsigned* status);
int launch_gemm_simt(const GemmProblem& p, void* stream);

// 3-D fp16 tensor map with 128-byte swizzle (dims d0 innermost; strides in
// bytes for d1, d2); false if the driver entry point or the encode fails.
bool encode_tmap_3d_f16(CUtensorMap* m, const void* base, uint64_t d0,
                        uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
                        uint32_t b0, uint32_t b1, uint32_t b2);

// Number of SMs of the current device.
int device_sm_count();
// Host counter of launched kernels (tp_launch_count).
void count_launch(int n = 1);

}  // namespace tp
