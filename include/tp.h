/*
 * tp.h — C ABI of the GB300 tensor-parallel Transformer-block library.
 *
 * A Megatron tensor-parallel (TP) group of degree n is simulated as n logical
 * shards on ONE GPU.  The g all-reduce (after the row-parallel projection, in
 * forward) and the f all-reduce (on the input gradient, in backward) become an
 * on-device sum over the n shard partials, either accumulated in the GEMM's
 * tensor-memory accumulator in shard order ("fused") or written out as n
 * partial tensors and summed by a reduce kernel ("materialised").
 *
 * Pages cited (short name -> page title):
 *   [Grasp-TP]   Grasp lesson 11, "张量并行线性层分片与前反向通信量计算"
 *   [Troverld]   cnblogs post "ラブパラ" (survey of parallelisms)
 *   [hjcheng-TP] hjcheng0602 blog post "TP"
 *   [adu-TP]     "Tensor Parallelism张量并行（一）" (Megatron-LM paper notes)
 *
 * Conventions for every call:
 *  - All tensors are dense, row-major, on the device unless stated.  Token
 *    t = batch·s + position; activations are [T, h] with T = b·s.
 *  - Weights are stored [out_features, in_features] (the Linear.weight
 *    storage noted in [Grasp-TP] §1) and are passed UNSHARDED: shard i of a
 *    column-parallel weight is its row block i, shard i of a row-parallel
 *    weight is its column block i.  The library never copies weights.
 *  - Element type is the descriptor's dtype for every tensor argument except
 *    the fp32 statistics named as `float*`.  TP_BF16 computes with fp32
 *    accumulation; TP_F32 computes in fp32 throughout.
 *  - Inner dimensions (h, h_ffn/n, n_q·d, n_kv·d) must be multiples of 8 and
 *    all device pointers 16-byte aligned; otherwise TP_ERR_SHAPE / TP_ERR_ARG.
 *  - Ownership: the caller allocates every buffer.  The library allocates no
 *    device or host memory on any compute path.  `ws` (saved activations,
 *    written by a forward call and read by the matching backward call) must
 *    stay alive and unmodified between the two.  Gradients are overwritten,
 *    never accumulated into.
 *  - Asynchrony: compute calls only enqueue work on `stream` (a cudaStream_t;
 *    NULL = the legacy default stream) and never synchronise.  A sequence of
 *    calls can therefore be captured into a CUDA graph and replayed (the
 *    overlapped mode forks a library-owned stream from `stream` and joins it
 *    back inside the call, which the capture follows); make the first call
 *    of each kind before capturing (it sets kernel attributes once), and
 *    leave event timing (tp_profile_enable) off while capturing.
 *  - Errors: argument, shape and workspace errors are returned before any
 *    launch, with nothing enqueued.  A failed launch returns TP_ERR_CUDA.
 *    Device-side waits are bounded; one that runs out records a device status
 *    word that tp_device_status() returns as TP_ERR_DEVICE_TIMEOUT (or
 *    TP_ERR_RANGE for an fp16 overflow).  No C++ exception crosses this
 *    boundary.
 */
#ifndef TP_H_
#define TP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TP_OK = 0,
  TP_ERR_NULL = 1,            /* a required pointer is NULL */
  TP_ERR_SHAPE = 2,           /* n∤h_ffn, n∤n_q, n∤n_kv, n_kv∤n_q, bad sizes */
  TP_ERR_DTYPE = 3,           /* unknown dtype / activation / mode */
  TP_ERR_WORKSPACE = 4,       /* ws or scratch smaller than the *_bytes query */
  TP_ERR_UNSUPPORTED = 5,     /* valid but not implemented (e.g. d != 128) */
  TP_ERR_CUDA = 6,            /* a CUDA runtime/driver call failed */
  TP_ERR_DEVICE_TIMEOUT = 7,  /* a bounded device wait ran out */
  TP_ERR_ARG = 8,             /* misaligned pointer or other bad argument */
  TP_ERR_RANGE = 9            /* an fp16 attention operand overflowed */
} tp_status;

/* TP_FP8 (E4M3, δ = 1): an FP8 payload in the accountants; for the MLP it
 * selects forward GEMMs on per-tensor scaled E4M3 operands (bf16 storage). */
typedef enum { TP_F32 = 0, TP_BF16 = 1, TP_FP8 = 2 } tp_dtype;  /* δ = 4, 2, 1 */
typedef enum { TP_GELU = 0, TP_SWIGLU = 1 } tp_act;
/* TP_REDUCE_OVERLAP: materialised partials, summed band by band (row bands
 * of the GEMM, up to 4) on a second stream while the GEMM computes the next
 * band ([Troverld] §II.II tile-wise overlap of the reduction with the GEMM);
 * the result equals TP_REDUCE_MATERIALISED bit for bit.  The library creates
 * that stream (one per device) and orders it against the caller's stream
 * with events; the call returns with all work ordered on `stream`. */
/* TP_REDUCE_SP: Megatron sequence parallelism ([Troverld] §III.III).  Each
 * all-reduce becomes a reduce-scatter to the ranks' T/n token rows, the
 * token-wise ops run on those rows, and an all-gather hands the whole
 * activation to the next column-parallel GEMM; on one device the gathered
 * buffer is the reduced one.  A block call computes what
 * TP_REDUCE_MATERIALISED computes (its token-wise ops — bias, dropout,
 * residual — already run inside the reduce).  In a layer call the next
 * block's RMSNorm joins the reduction: forward, one pass sums the attention
 * partials, adds the residual, writes x1 and the second RMSNorm's output;
 * backward, each f reduction is summed inside the RMSNorm backward kernel.
 * Results equal TP_REDUCE_MATERIALISED bit for bit, with one [T, h] write
 * and read fewer per fused reduction. */
typedef enum { TP_REDUCE_FUSED = 0, TP_REDUCE_MATERIALISED = 1,
               TP_REDUCE_OVERLAP = 2, TP_REDUCE_SP = 3 } tp_reduce_mode;
typedef enum { TP_SCOPE_MLP = 0, TP_SCOPE_ATTN = 1, TP_SCOPE_LAYER = 2 } tp_scope;

typedef void* tp_stream; /* cudaStream_t */

/* ------------------------------------------------------------------ MLP --
 * The Megatron MLP ([Grasp-TP] §3; [hjcheng-TP] MLP, TP forward/backward;
 * [adu-TP] 张量并行应用于 MLP 和 Attention):
 *   GeLU:   H_i = X·W1_iᵀ (+ b1_i),  A_i = GeLU(H_i) = H_i·Φ(H_i)
 *   SwiGLU: G_i = X·Wg_iᵀ, U_i = X·Wu_iᵀ, A_i = SiLU(G_i) ⊙ U_i
 *   Z^i = A_i·W2_iᵀ,  Z = Σ_{i=0}^{n-1} Z^i  (g),
 *   Out = R + mask ⊙ (Z + b2) / (1 − p)   (b2 once, after the sum: [Grasp-TP] §3)
 * W1 is [h_ffn, h] (GeLU) or [2·h_ffn, h] with gate rows [0, h_ffn) and up
 * rows [h_ffn, 2·h_ffn) (SwiGLU); W2 is [h, h_ffn].  Rank i holds W1 rows
 * (and, for SwiGLU, gate and up rows) [i·h_ffn/n, (i+1)·h_ffn/n) and the same
 * columns of W2.
 * Dropout (p > 0) keeps element (t, j) of the [T, h] output when the top 24
 * bits of draw e = t·h + j of the splitmix64 stream seeded with `seed` are
 * ≥ round(p·2^24); the mask is regenerated, not stored, in backward.
 */
typedef struct {
  int64_t T;          /* tokens b·s (≥ 1) */
  int64_t h;          /* hidden size */
  int64_t h_ffn;      /* MLP intermediate size f */
  int32_t n;          /* TP degree: number of logical shards (n | h_ffn) */
  int32_t dtype;      /* tp_dtype (TP_FP8: see below) */
  int32_t act;        /* tp_act */
  int32_t mode;       /* tp_reduce_mode for the g and f reductions */
  float dropout_p;    /* in [0, 1) */
  uint64_t seed;      /* dropout stream seed */
} tp_mlp_desc;
/* dtype TP_FP8: tensors are stored in bf16 as for TP_BF16, and the two
 * forward GEMMs run the FP8 fused kernel (tp_quantize_fp8 of X, W1, A, W2;
 * E4M3 GEMMs dequantized in the epilogue, whose bias, activation, dropout
 * and residual steps are unchanged); the backward is the bf16 backward on
 * the saved bf16 activations.  Needs h and h_ffn/n multiples of 16. */

/* Bytes of `ws` for tp_mlp_fwd/tp_mlp_bwd: saved activations (H and A for
 * GeLU; G, U and A for SwiGLU; each [T, h_ffn] in dtype) followed by the
 * forward scratch (n partial [T, h] tensors in materialised mode; for
 * TP_FP8 also the E4M3 copies of X [T, h], W1, A [T, h_ffn] and W2 and 16
 * bytes of scales).  Every region starts at the next 256-byte boundary, in
 * the order listed. */
size_t tp_mlp_workspace_bytes(const tp_mlp_desc* d);
/* Bytes of `scratch` for tp_mlp_bwd: dZ [T, h] (when p > 0), the
 * activation-input gradient ([T, h_ffn] or [T, 2·h_ffn]), partial input
 * gradients (materialised mode) and fp32 column-sum partials. */
size_t tp_mlp_bwd_scratch_bytes(const tp_mlp_desc* d);

/* Forward.  b1, b2, R may be NULL (absent).  Out: [T, h]. */
tp_status tp_mlp_fwd(const tp_mlp_desc* d, const void* X, const void* W1,
                     const void* b1, const void* W2, const void* b2,
                     const void* R, void* Out, void* ws, size_t ws_bytes,
                     tp_stream stream);

/* Backward ([hjcheng-TP] 单卡backward / TP backward; f of [adu-TP]):
 *   dZ = dOut ⊙ mask/(1−p);  db2 = Σ_t dZ;  dW2 = dZᵀ·A;  dA = dZ·W2;
 *   dH = dA ⊙ GeLU'(H)  (SwiGLU: dG = dA ⊙ U ⊙ SiLU'(G), dU = dA ⊙ SiLU(G));
 *   db1 = Σ_t dH;  dW1 = dHᵀ·X;  dX = Σ_i dH_i·W1_i (f)  + dres.
 * `ws` is the buffer the forward call filled.  db1, db2 and dres may be NULL
 * (not computed / not added); dres is the gradient of a residual whose
 * source is X itself (e.g. R = X), added once after the f sum. */
tp_status tp_mlp_bwd(const tp_mlp_desc* d, const void* dOut, const void* X,
                     const void* W1, const void* W2, const void* ws,
                     const void* dres, void* dX, void* dW1, void* db1,
                     void* dW2, void* db2, void* scratch,
                     size_t scratch_bytes, tp_stream stream);

/* ------------------------------------------------------------ attention --
 * Head-sharded causal GQA attention ([Grasp-TP] §4; [Troverld] §I.III;
 * [hjcheng-TP] Attention):
 *   Q = X·Wqᵀ [T, n_q·d], K = X·Wkᵀ, V = X·Wvᵀ [T, n_kv·d]
 *   O_j = softmax(mask(Q_j K_kvᵀ/√d)) V_kv per batch element and q head j,
 *         kv = ⌊j·n_kv/n_q⌋, causal mask key ≤ query within one sequence
 *   Z^i = O_i·Wo_iᵀ, Z = Σ_i Z^i (g), Out = R + Z + bo (bo once)
 * Wq [n_q·d, h], Wk/Wv [n_kv·d, h], Wo [h, n_q·d].  Rank i holds q heads
 * [i·n_q/n, (i+1)·n_q/n) and kv heads [i·n_kv/n, (i+1)·n_kv/n); n must divide
 * n_q and n_kv ([Grasp-TP] §4 GQA note) else TP_ERR_SHAPE.  d must be 128
 * (else TP_ERR_UNSUPPORTED). */
typedef struct {
  int64_t b, s, h;
  int32_t n_q, n_kv, d, n;
  int32_t dtype;      /* TP_BF16 or TP_FP8 (TP_F32 -> TP_ERR_UNSUPPORTED) */
  int32_t causal;     /* 1 = causal mask, 0 = full */
  int32_t mode;       /* tp_reduce_mode */
} tp_attn_desc;
/* dtype TP_FP8: storage and backward as for TP_BF16; the Q, K, V and output
 * projections of the forward run on E4M3 operands (tp_quantize_fp8 of X,
 * Wq, Wk, Wv, then of O and Wo; dequantized in the epilogue).  Needs h a
 * multiple of 16.  ws then also holds the E4M3 copies of X, Wq, Wk, Wv, O,
 * Wo and their six scales (and six amax words) after the regions below. */

/* ws: Q [T, n_q·d], K, V [T, n_kv·d] (fp16), O [T, n_q·d] (bf16) and LSE
 * [b, n_q, s] fp32 saved for backward, then the forward scratch (n partial
 * [T, h] tensors in materialised mode); each region starts at the next
 * 256-byte boundary, in this order.
 * The attention core multiplies fp16 operands with fp32 accumulation (Q, K,
 * V, dO in fp16; the probabilities and their gradients rounded to fp16):
 * |Q|, |K|, |V|, |dO| must stay below 65504, else tp_device_status reports
 * TP_ERR_RANGE. */
size_t tp_attn_workspace_bytes(const tp_attn_desc* d);
/* scratch: dO (fp16), dQ, dK, dV (bf16), D = rowsum(dO∘O) and LSE·log2e
 * (fp32, [b, n_q, s rounded up to 128]), the score gradient dS in fp16
 * 128×128 tiles (b·n_q·B(B+1)/2 tiles causal, b·n_q·B² full, B = ⌈s/128⌉;
 * 32 KB each), partials and column-sum partials. */
size_t tp_attn_bwd_scratch_bytes(const tp_attn_desc* d);
/* Upper bound, in bytes, on the dS tiles held at once: the backward runs in
 * passes over (batch, kv head) pairs, as many per pass as fit (at least
 * one), so the scratch stays bounded for long sequences.  bytes = 0 restores
 * the default (8 GiB).  Returns the previous bound.  Host only; it changes
 * what tp_attn_bwd_scratch_bytes returns, so query the scratch size after
 * setting it.  Results do not depend on it (each pair's work is the same). */
size_t tp_attn_set_ds_budget(size_t bytes);

tp_status tp_attn_fwd(const tp_attn_desc* d, const void* X, const void* Wq,
                      const void* Wk, const void* Wv, const void* Wo,
                      const void* bo, const void* R, void* Out, void* ws,
                      size_t ws_bytes, tp_stream stream);

/* dWo = dOutᵀ·O; dO = dOut·Wo; flash backward → dQ, dK, dV (GQA groups
 * summed); dWq = dQᵀ·X, dWk, dWv likewise; dX = Σ_i (dQ_i Wq_i + dK_i Wk_i
 * + dV_i Wv_i) (f) + dres; dbo = Σ_t dOut.  dbo and dres may be NULL. */
tp_status tp_attn_bwd(const tp_attn_desc* d, const void* dOut, const void* X,
                      const void* Wq, const void* Wk, const void* Wv,
                      const void* Wo, const void* ws, const void* dres,
                      void* dX, void* dWq, void* dWk, void* dWv, void* dWo,
                      void* dbo, void* scratch, size_t scratch_bytes,
                      tp_stream stream);

/* -------------------------------------------------------------- RMSNorm --
 * Token-wise RMSNorm on the replicated activation ([Troverld] §II.III fused
 * norm; pre-norm reading of §III.III):  rstd_t = 1/sqrt(mean_j x_tj² + ε),
 * y = x·rstd·γ.  rstd [T] fp32 is written for the backward call. */
tp_status tp_rmsnorm_fwd(int64_t T, int64_t h, float eps, int32_t dtype,
                         const void* x, const void* gamma, void* y,
                         float* rstd, tp_stream stream);
size_t tp_rmsnorm_bwd_scratch_bytes(int64_t T, int64_t h);
/* dx = rstd·(dy⊙γ) − x·rstd³·Σ_j(dy⊙γ⊙x)_j/h + dres;  dγ = Σ_t dy⊙x·rstd.
 * dres may be NULL.  dgamma is reduced deterministically through scratch. */
tp_status tp_rmsnorm_bwd(int64_t T, int64_t h, float eps, int32_t dtype,
                         const void* dy, const void* x, const void* gamma,
                         const float* rstd, const void* dres, void* dx,
                         void* dgamma, void* scratch, size_t scratch_bytes,
                         tp_stream stream);

/* The same RMSNorm backward for callers that cannot allocate device memory:
 * code that runs under another framework's memory pool, a real-time loop
 * where cudaMalloc (which can synchronise the device and stall) is not
 * allowed after start-up, or an embedding that hands the library only its
 * input and output tensors.  There is no counterpart on the pages; this is a
 * service of the library.  The dγ partial sums go to a fixed 8 MiB device
 * array inside the library instead of a caller scratch buffer, so h must be
 * at most TP_RMSNORM_NOALLOC_MAX_H (TP_ERR_WORKSPACE otherwise).  The first
 * call on each device looks up that array's device address (no allocation);
 * make it before capturing a stream.  All calls share the array: calls that
 * overlap on the GPU (other streams, other threads) race and must be
 * serialised by the caller.  Results equal tp_rmsnorm_bwd's. */
#define TP_RMSNORM_NOALLOC_MAX_H 8192
tp_status tp_rmsnorm_bwd_noalloc(int64_t T, int64_t h, float eps,
                                 int32_t dtype, const void* dy, const void* x,
                                 const void* gamma, const float* rstd,
                                 const void* dres, void* dx, void* dgamma,
                                 tp_stream stream);

/* ---------------------------------------------------------------- layer --
 * The pre-norm layer of the C5 workload as one call per direction
 * ([Troverld] §III.III layer with the norm before each block; [Grasp-TP]
 * §3–§4 blocks):  x1 = x + Attn(RMSNorm₁(x)),  out = x1 + MLP(RMSNorm₂(x1)),
 * causal GQA attention without bias, SwiGLU MLP without bias or dropout,
 * four reductions (g after each row-parallel projection, f on each block's
 * input gradient) taken as the desc's mode says.  Composes tp_rmsnorm_*,
 * tp_attn_* and tp_mlp_* in this order on one stream; every tensor is bf16
 * [T, h] (weights as for the blocks, γ₁ and γ₂ [h]).  dtype TP_FP8 runs both
 * blocks' forward projections on E4M3 operands (see the blocks). */
typedef struct {
  int64_t b, s, h, h_ffn;
  int32_t n_q, n_kv, d, n;
  int32_t dtype;      /* TP_BF16 or TP_FP8 */
  int32_t mode;       /* tp_reduce_mode */
  float eps;          /* RMSNorm ε (> 0) */
} tp_layer_desc;
/* ws: saved for backward — RMSNorm₁ output, x1, RMSNorm₂ output (bf16
 * [T, h]), rstd₁, rstd₂ (fp32 [T]), then the attention block's ws and the
 * MLP block's ws (tp_attn_workspace_bytes, tp_mlp_workspace_bytes of the
 * blocks' descs); for TP_BF16 then the forward's fp16 operands of the Q, K,
 * V projections (one launch): the RMSNorm₁ output [T, h] and [Wq; Wk; Wv]
 * stacked.  Each region on the next 256-byte boundary.
 * Precision (TP_BF16): the Q, K, V projections multiply fp16 copies of the
 * RMSNorm₁ output and of Wq, Wk, Wv (fp32 accumulation).  The softmax
 * multiplies the relative error of its input's rounding by the score scale
 * (a few units at the layer workload), and fp16 carries 3 more mantissa bits
 * than bf16; a norm output is bounded by √h·max|γ|, so fp16's range holds it
 * for |γ| ≤ 65504/√h.  A weight beyond ±65504 reports TP_ERR_RANGE through
 * tp_device_status; weights below 2^-14 in magnitude lose precision
 * (fp16 subnormals). */
size_t tp_layer_workspace_bytes(const tp_layer_desc* d);
/* scratch: the two block gradients' [T, h] hand-overs (bf16), the RMSNorm
 * scratch, then the larger of the attention and MLP backward scratches
 * (the blocks run one after the other and share it). */
size_t tp_layer_bwd_scratch_bytes(const tp_layer_desc* d);
tp_status tp_layer_fwd(const tp_layer_desc* d, const void* x, const void* g1,
                       const void* Wq, const void* Wk, const void* Wv,
                       const void* Wo, const void* g2, const void* W1,
                       const void* W2, void* out, void* ws, size_t ws_bytes,
                       tp_stream stream);
/* Gradients of ⟨dout, out⟩ with respect to x and every weight (overwritten);
 * ws must hold what tp_layer_fwd saved for the same inputs. */
tp_status tp_layer_bwd(const tp_layer_desc* d, const void* dout, const void* x,
                       const void* g1, const void* Wq, const void* Wk,
                       const void* Wv, const void* Wo, const void* g2,
                       const void* W1, const void* W2, const void* ws,
                       void* dx, void* dg1, void* dWq, void* dWk, void* dWv,
                       void* dWo, void* dg2, void* dW1, void* dW2,
                       void* scratch, size_t scratch_bytes, tp_stream stream);

/* ----------------------------------------------------------- accounting --
 * Host-only, exact integer figures; no GPU needed.
 * Communication ([Grasp-TP] §5; [Troverld] §II.II; [adu-TP] 通信开销): each
 * reduction carries payload P = T·h·δ bytes; a ring all-reduce moves
 * 2(n−1)·P/n per rank (kept as the reduced fraction num/den); [Troverld]'s
 * figure drops (n−1)/n: 2·P.  MLP and attention: 1 reduction forward + 1
 * backward; a layer: 2 + 2. */
typedef struct {
  uint64_t reductions_fwd, reductions_bwd;
  uint64_t payload_bytes;               /* T·h·δ */
  uint64_t ring_bytes_num, ring_bytes_den; /* 2(n−1)·P / n, reduced */
  uint64_t page2_bytes;                 /* 2·P */
  uint64_t total_payload;               /* (fwd+bwd)·P */
  uint64_t total_ring_num;              /* (fwd+bwd)·ring, over ring_bytes_den */
  uint64_t total_page2;                 /* (fwd+bwd)·2·P */
  /* Megatron-SP ([Troverld] §III.III): each all-reduce position becomes a
   * reduce-scatter to (b, s/n, H) at a block's end and an all-gather back to
   * (b, s, H) at the next block's start (in backward the conjugates).  Per
   * rank in a ring each moves (n−1)·P/n, kept as the reduced fraction
   * num/sp_bytes_den; rs + ag equals the ring all-reduce.  Counts per
   * microbatch, forward + backward. */
  uint64_t sp_rs_bytes_num, sp_ag_bytes_num, sp_bytes_den;
  uint64_t sp_reduce_scatters, sp_all_gathers;
  uint64_t sp_total_num;                /* over sp_bytes_den */
} tp_comm_report;

tp_status tp_comm_bytes(int32_t scope, int64_t T, int64_t h, int32_t n,
                        int32_t dtype, tp_comm_report* out);

/* Saved activations per rank ([hjcheng-TP] MLP and Attention: the tensors
 * each block keeps for its backward, single card and TP; TP divides the
 * column- / head-sharded ones by n, the block input stays whole).
 *
 * Element counts per rank (T = b·s, f = h_ffn, q = n_q/n, k = n_kv/n):
 *   MLP:   x T·h; hidden H (GeLU) T·f/n or G and U (SwiGLU) 2·T·f/n;
 *          activation A T·f/n; dropout mask T·h (if dropout)
 *   attention: x T·h; Q T·q·d; K and V T·k·d each; the page's score matrix
 *          S b·q·s² (unfused) or the log-sum-exp b·q·s (flash); AV T·q·d
 *   layer (pre-norm, flash): both blocks plus each RMSNorm's input T·h and
 *          rstd T, and the dropout masks after the two reductions.
 * Megatron-SP ([Troverld] §III.III): the token-wise region (norm input and
 * rstd, dropout masks) holds s/n positions per rank, rounded up; the block
 * inputs stay whole.
 * Bytes: activations δ (2 bf16 / 4 fp32), masks 1 byte, S δ, LSE and rstd
 * 4.  The flash attention figure is what this library's attention
 * workspace holds (Q, K, V in fp16 as δ = 2, O, LSE) plus x. */
typedef struct {
  int64_t b, s, h, h_ffn;
  int32_t n_q, n_kv, d, n;
  int32_t dtype;          /* TP_F32 | TP_BF16 */
  int32_t act;            /* TP_GELU | TP_SWIGLU */
  int32_t dropout;        /* 1: a mask after each block's reduction */
  int32_t seq_parallel;   /* 1: Megatron-SP token-wise region */
} tp_act_desc;
typedef struct {
  uint64_t mlp_x, mlp_hidden, mlp_act, mlp_mask;                  /* elements */
  uint64_t attn_x, attn_q, attn_kv, attn_scores, attn_lse, attn_o; /* elements */
  uint64_t norm_x, norm_rstd;                                      /* per norm */
  uint64_t mlp_bytes;          /* MLP block */
  uint64_t attn_bytes_pages;   /* attention with the score matrix S */
  uint64_t attn_bytes_flash;   /* attention with LSE instead of S */
  uint64_t layer_bytes_flash;  /* pre-norm layer: norms + flash attn + MLP */
} tp_act_report;

/* TP_ERR_NULL, TP_ERR_SHAPE (negative sizes, n < 1, n∤n_q, n∤n_kv, n∤h_ffn),
 * TP_ERR_DTYPE (dtype / act). */
tp_status tp_act_memory(const tp_act_desc* d, tp_act_report* out);

/* Algorithmic FLOPs ([hjcheng-TP] 单卡forward/backward tables): GeLU MLP
 * 4·T·h·f forward, SwiGLU 6·T·h·f; attention projections
 * 2·T·h·(n_q+2·n_kv)·d + 2·T·n_q·d·h plus 4·b·n_q·d·C with C = s(s+1)/2
 * (causal) or s² (full); backward = 2 × forward. */
tp_status tp_mlp_flops(const tp_mlp_desc* d, uint64_t* fwd, uint64_t* bwd);
tp_status tp_attn_flops(const tp_attn_desc* d, uint64_t* fwd, uint64_t* bwd);

/* ------------------------------------------------------- GEMM building block
 * C[M, N] = Σ_k A[m, k]·B[n, k] on the tensor cores (bf16 in, fp32
 * accumulate, bf16 out) or on CUDA cores (fp32).  a_mn_major = 0: A is
 * [M, K] row-major (lda ≥ K); 1: A is stored [K, M] (lda ≥ M).  Likewise B
 * ([N, K] or [K, N]).  C is [M, N] with ldc.  The building block of every
 * projection above, exported for tests. */
tp_status tp_gemm(int32_t dtype, int64_t M, int64_t N, int64_t K,
                  const void* A, int64_t lda, int32_t a_mn_major,
                  const void* B, int64_t ldb, int32_t b_mn_major, void* C,
                  int64_t ldc, tp_stream stream);


/* ------------------------------------------------------------------ FP8 --
 * The quantize and compute steps of the FP8 fused kernel ([Troverld]
 * §II.III: quantize + compute + dequantize), per-tensor scaled E4M3:
 *   amax = max |x|, scale = 448 / amax in fp32 (1 when amax = 0),
 *   q = E4M3 code of fp32(x·scale), round to nearest even, saturating at ±448.
 * tp_quantize_fp8: x is n bf16 values (16-byte aligned, n a multiple of 8);
 * writes q (n bytes, 16-byte aligned) and *scale_out (one device float);
 * amax_work is one device word of scratch.  All pointers device memory
 * owned by the caller.  TP_ERR_NULL, TP_ERR_ARG (alignment), TP_ERR_SHAPE.
 * tp_gemm_fp8: C[M, N] (bf16, row-major, ldc) =
 *   Σ_k qa[m, k]·qb[n, k] / (scale_a·scale_b) on the tensor cores
 * (kind::f8f6f4, fp32 accumulate); qa [M, K] and qb [N, K] row-major E4M3
 * codes (lda, ldb ≥ K, multiples of 16 bytes); scale_a, scale_b device
 * floats as written by tp_quantize_fp8.  TP_ERR_SHAPE / TP_ERR_ARG on bad
 * sizes or alignment, before any launch. */
tp_status tp_quantize_fp8(int64_t n, const void* x, void* q, float* scale_out,
                          void* amax_work, tp_stream stream);
tp_status tp_gemm_fp8(int64_t M, int64_t N, int64_t K, const void* qa,
                      int64_t lda, const float* scale_a, const void* qb,
                      int64_t ldb, const float* scale_b, void* C, int64_t ldc,
                      tp_stream stream);

/* ------------------------------------------------------------ profiling --
 * Per-kernel-family device time for roofline reporting.  While enabled,
 * every kernel the library launches is bracketed by two CUDA events recorded
 * on that kernel's launch stream, tagged with its family and its algorithmic
 * FLOPs and bytes.  tp_profile_enable(max_launches) creates the event pool
 * (host-side CUDA event objects; no device buffers); 0 disables it and
 * destroys the pool.  Launches beyond max_launches are not recorded.
 * tp_profile_read synchronises the recorded events and returns, for one
 * family, the number of recorded launches, their summed duration and their
 * summed algorithmic FLOPs and bytes.  Families: 0 tcgen05 GEMM, 1 fp32
 * GEMM, 2 attention forward, 3 attention backward dK/dV, 4 attention
 * backward dQ, 5 shard-partial reduce, 6 other elementwise, 7 RMSNorm,
 * 8 tcgen05 GEMM on E4M3 operands, 9 FP8 amax / quantize. */
typedef struct {
  uint64_t launches;
  double ms;
  double flops;
  double bytes;
} tp_profile_entry;

tp_status tp_profile_enable(int32_t max_launches);
tp_status tp_profile_reset(void);
tp_status tp_profile_read(int32_t family, tp_profile_entry* out);

/* ----------------------------------------------------------------- status */
/* Synchronises `stream`, returns and clears the device status word
 * (TP_OK, TP_ERR_DEVICE_TIMEOUT or TP_ERR_RANGE), or TP_ERR_CUDA if the
 * stream failed. */
tp_status tp_device_status(tp_stream stream);
const char* tp_status_string(tp_status s);
/* Failure-path self-test: enqueues one kernel whose single wait (on an
 * mbarrier that nothing completes) runs through the same bounded wait as
 * every kernel of this library.  After about two seconds at the maximum SM
 * clock the wait gives up, the kernel records the timeout and returns; the
 * next tp_device_status on the stream then returns TP_ERR_DEVICE_TIMEOUT
 * (and clears the word), and the context stays usable.  Returns TP_OK once
 * the kernel is enqueued. */
tp_status tp_selftest_wait_timeout(tp_stream stream);
/* The CUDA runtime error code behind the latest TP_ERR_CUDA (0 if none
 * yet) and, when name is not NULL, its name (a static string). */
int32_t tp_last_cuda_error(const char** name);
/* Number of kernels this library has launched since load (host counter). */
uint64_t tp_launch_count(void);
/* SM count of the current device (0 if none); cached per device. */
int32_t tp_num_sms(void);

#ifdef __cplusplus
}
#endif

#endif /* TP_H_ */
