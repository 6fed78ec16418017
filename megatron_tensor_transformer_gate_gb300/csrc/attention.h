// attention.h — launchers of the flash-attention kernels (attention.cu).
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace tp {

// Causal (or full) GQA attention on per-head views of row-major Q [T, nq·d],
// K/V [T, nkv·d], O [T, nq·d]; token t = batch·s + position; LSE [b, nq, s].
struct AttnShape {
  int64_t b, s;
  int nq, nkv, d;
  int causal;
  float scale;  // 1/√d
  // Backward only: (batch, kv head) pairs whose dS tiles are held at once,
  // fixed when the caller's scratch is carved (attn_ds_pairs_per_pass) so
  // that the tile region and the passes of flash_bwd agree.
  int64_t ds_pairs = 0;
};

// Forward on tcgen05 (attn_fwd_tc.cu); Q, K, V fp16, O bf16.
int flash_fwd(const AttnShape& sh, const void* Q, const void* K, const void* V,
              void* O, float* LSE, unsigned* status, void* stream);
// Backward on tcgen05 (attn_bwd_tc.cu): dQ, dK, dV (bf16, GQA groups summed).
// Dp and L2p are fp32 scratch of b·nq·attn_stats_pad(s) elements each
// (D = rowsum(dO∘O) and LSE·log2e, zero-padded); dO is fp16.  dS is
// attn_ds_bytes(sh) bytes of scratch (16-byte aligned) for the fp16 score
// gradient tiles that the dK/dV kernel writes and the dQ kernel reads; the
// backward runs in passes of sh.ds_pairs (batch, kv head) pairs.
int64_t attn_stats_pad(int64_t s);
// Pairs per pass under the current budget (read once; at least one).
int64_t attn_ds_pairs_per_pass(const AttnShape& sh);
// Bytes of dS tiles for sh.ds_pairs pairs.
int64_t attn_ds_bytes(const AttnShape& sh);
// Bound on the dS tile bytes per pass (0 = the default 8 GiB); returns the
// previous bound.
int64_t attn_set_ds_budget(int64_t bytes);
int flash_bwd(const AttnShape& sh, const void* Q, const void* K, const void* V,
              const void* O, const void* dO, const float* LSE, float* Dp,
              float* L2p, void* dS, void* dQ, void* dK, void* dV,
              unsigned* status, void* stream);

}  // namespace tp
