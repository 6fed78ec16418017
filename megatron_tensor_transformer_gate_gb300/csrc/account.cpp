// account.cpp — host-only communication-volume and FLOP accountant.
//
// What a real TP group of degree n would send, per microbatch:
//  * one reduction in forward (g after the row-parallel projection) and one
//    in backward (f on the input gradient) per MLP or attention block; four
//    per layer ([Grasp-TP] §5 list; [adu-TP] 张量并行的通信开销);
//  * each reduction's logical payload P = T·h·δ bytes ([Grasp-TP] §5,
//    δ from [Troverld] §O.I: FP32 4, BF16 2; FP8 1 for the FP8 buffers of
//    [Grasp-TP] §6);
//  * a ring all-reduce moves 2(n−1)·P/n per rank ([Grasp-TP] §5), returned
//    as an exact reduced fraction; [Troverld] §II.II counts 2·P.
// Megatron-SP ([Troverld] §III.III): each all-reduce position splits into a
// reduce-scatter and an all-gather of (n−1)·P/n per rank each.
// Saved activations ([hjcheng-TP] MLP / Attention 激活值): see tp.h.
// FLOPs ([hjcheng-TP] 单卡forward / 单卡backward): each GEMM of m×k by k×n is
// 2·m·n·k; backward is twice forward.  GeLU MLP 4·T·h·f, SwiGLU 6·T·h·f;
// attention 2·T·h·(n_q+2·n_kv)·d + 2·T·n_q·d·h + 4·b·n_q·d·C with
// C = s(s+1)/2 causal, s² full.
#include <stdint.h>

#include "../../include/tp.h"

namespace {

uint64_t gcd_u64(uint64_t a, uint64_t b) {
  while (b != 0) {
    const uint64_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

}  // namespace

extern "C" tp_status tp_comm_bytes(int32_t scope, int64_t T, int64_t h,
                                   int32_t n, int32_t dtype,
                                   tp_comm_report* out) {
  if (out == nullptr) return TP_ERR_NULL;
  if (T < 0 || h < 0 || n < 1) return TP_ERR_SHAPE;
  uint64_t delta;
  switch (dtype) {
    case TP_F32: delta = 4; break;
    case TP_BF16: delta = 2; break;
    case TP_FP8: delta = 1; break;
    default: return TP_ERR_DTYPE;
  }
  uint64_t fwd, bwd;
  switch (scope) {
    case TP_SCOPE_MLP:
    case TP_SCOPE_ATTN: fwd = 1; bwd = 1; break;
    case TP_SCOPE_LAYER: fwd = 2; bwd = 2; break;
    default: return TP_ERR_DTYPE;
  }
  const uint64_t P = (uint64_t)T * (uint64_t)h * delta;
  uint64_t num = 2ull * (uint64_t)(n - 1) * P;
  uint64_t den = (uint64_t)n;
  const uint64_t g = num == 0 ? den : gcd_u64(num, den);
  num /= g;
  den /= g;
  const uint64_t count = fwd + bwd;
  out->reductions_fwd = fwd;
  out->reductions_bwd = bwd;
  out->payload_bytes = P;
  out->ring_bytes_num = num;
  out->ring_bytes_den = den;
  out->page2_bytes = 2 * P;
  out->total_payload = count * P;
  out->total_ring_num = count * num;
  out->total_page2 = count * 2 * P;
  // Megatron-SP: a reduce-scatter and an all-gather at each all-reduce
  // position, (n−1)·P/n per rank each, as their own reduced fraction
  uint64_t hn = (uint64_t)(n - 1) * P, hd = (uint64_t)n;
  const uint64_t g2 = hn == 0 ? hd : gcd_u64(hn, hd);
  hn /= g2;
  hd /= g2;
  out->sp_rs_bytes_num = hn;
  out->sp_ag_bytes_num = hn;
  out->sp_bytes_den = hd;
  out->sp_reduce_scatters = count;
  out->sp_all_gathers = count;
  out->sp_total_num = count * 2 * hn;
  return TP_OK;
}

extern "C" tp_status tp_act_memory(const tp_act_desc* d, tp_act_report* out) {
  if (d == nullptr || out == nullptr) return TP_ERR_NULL;
  if (d->b < 0 || d->s < 0 || d->h < 0 || d->h_ffn < 0 || d->n_q < 0 ||
      d->n_kv < 0 || d->d < 0 || d->n < 1)
    return TP_ERR_SHAPE;
  if (d->n_q % d->n || d->n_kv % d->n || d->h_ffn % d->n) return TP_ERR_SHAPE;
  uint64_t delta;
  switch (d->dtype) {
    case TP_F32: delta = 4; break;
    case TP_BF16: delta = 2; break;
    case TP_FP8: delta = 1; break;
    default: return TP_ERR_DTYPE;
  }
  if (d->act != TP_GELU && d->act != TP_SWIGLU) return TP_ERR_DTYPE;
  const uint64_t n = (uint64_t)d->n, b = (uint64_t)d->b, s = (uint64_t)d->s;
  const uint64_t h = (uint64_t)d->h, f = (uint64_t)d->h_ffn;
  const uint64_t T = b * s, dd = (uint64_t)d->d;
  const uint64_t q = (uint64_t)d->n_q / n, k = (uint64_t)d->n_kv / n;
  // token-wise region: s/n positions per rank (rounded up) under SP
  const uint64_t Ttok = d->seq_parallel ? b * ((s + n - 1) / n) : T;
  tp_act_report r{};
  r.mlp_x = T * h;
  r.mlp_hidden = (d->act == TP_GELU ? 1 : 2) * T * (f / n);
  r.mlp_act = T * (f / n);
  r.mlp_mask = d->dropout ? Ttok * h : 0;
  r.attn_x = T * h;
  r.attn_q = T * q * dd;
  r.attn_kv = 2 * T * k * dd;
  r.attn_scores = b * q * s * s;
  r.attn_lse = b * q * s;
  r.attn_o = T * q * dd;
  r.norm_x = Ttok * h;
  r.norm_rstd = Ttok;
  const uint64_t attn_mask = d->dropout ? Ttok * h : 0;
  r.mlp_bytes = (r.mlp_x + r.mlp_hidden + r.mlp_act) * delta + r.mlp_mask;
  const uint64_t attn_common =
      (r.attn_x + r.attn_q + r.attn_kv + r.attn_o) * delta + attn_mask;
  r.attn_bytes_pages = attn_common + r.attn_scores * delta;
  r.attn_bytes_flash = attn_common + r.attn_lse * 4;
  r.layer_bytes_flash = 2 * (r.norm_x * delta + r.norm_rstd * 4) +
                        r.attn_bytes_flash + r.mlp_bytes;
  *out = r;
  return TP_OK;
}

extern "C" tp_status tp_mlp_flops(const tp_mlp_desc* d, uint64_t* fwd,
                                  uint64_t* bwd) {
  if (d == nullptr || fwd == nullptr || bwd == nullptr) return TP_ERR_NULL;
  if (d->T < 0 || d->h < 0 || d->h_ffn < 0) return TP_ERR_SHAPE;
  uint64_t gemms;
  switch (d->act) {
    case TP_GELU: gemms = 2; break;
    case TP_SWIGLU: gemms = 3; break;
    default: return TP_ERR_DTYPE;
  }
  const uint64_t one = 2ull * (uint64_t)d->T * (uint64_t)d->h * (uint64_t)d->h_ffn;
  *fwd = gemms * one;
  *bwd = 2 * gemms * one;
  return TP_OK;
}

extern "C" tp_status tp_attn_flops(const tp_attn_desc* d, uint64_t* fwd,
                                   uint64_t* bwd) {
  if (d == nullptr || fwd == nullptr || bwd == nullptr) return TP_ERR_NULL;
  if (d->b < 0 || d->s < 0 || d->h < 0 || d->n_q < 0 || d->n_kv < 0 ||
      d->d < 0)
    return TP_ERR_SHAPE;
  const uint64_t T = (uint64_t)d->b * (uint64_t)d->s;
  const uint64_t h = (uint64_t)d->h, dd = (uint64_t)d->d;
  const uint64_t nq = (uint64_t)d->n_q, nkv = (uint64_t)d->n_kv;
  const uint64_t s = (uint64_t)d->s;
  const uint64_t proj = 2 * T * h * (nq + 2 * nkv) * dd + 2 * T * nq * dd * h;
  const uint64_t pairs = d->causal ? s * (s + 1) / 2 : s * s;
  const uint64_t core = 4 * (uint64_t)d->b * nq * dd * pairs;
  *fwd = proj + core;
  *bwd = 2 * (proj + core);
  return TP_OK;
}
