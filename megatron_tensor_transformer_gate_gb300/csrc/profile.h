// profile.h — optional per-kernel-family timing with CUDA events.
//
// While enabled (tp_profile_enable), every kernel launch of the library is
// bracketed by two CUDA events recorded on its own launch stream, tagged with
// the launch's kernel family and its algorithmic FLOPs and bytes.  The event
// pool is created by tp_profile_enable; compute calls only record into it.
#pragma once

#include <stdint.h>

namespace tp {

enum KernelFamily : int {
  KF_GEMM_TC = 0,
  KF_GEMM_SIMT = 1,
  KF_ATTN_FWD = 2,
  KF_ATTN_BWD_DKDV = 3,
  KF_ATTN_BWD_DQ = 4,
  KF_REDUCE = 5,
  KF_ELEMENTWISE = 6,
  KF_NORM = 7,
  KF_GEMM_TC_FP8 = 8,
  KF_QUANT = 9,
  KF_COUNT = 10
};

// RAII bracket around one kernel launch.
struct ProfScope {
  ProfScope(void* stream, int family, double flops, double bytes);
  ~ProfScope();
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;
  int slot;
  void* stream;
};

}  // namespace tp
